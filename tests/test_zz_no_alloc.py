"""ssb_reconstruct_noalloc: the reconstruction for callers that cannot allocate
device memory (for example plugin code inside an application that owns the
device allocator, or an acquisition loop that must not allocate once running).

It must give the same result as ssb_reconstruct with a caller workspace, on
two calls in a row (the second call reuses the library's fixed scratch array
left over from the first, with a different problem size), and it must reject
problems whose scratch need exceeds that array.  Called through the C ABI
with ctypes.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TOL = 1e-4


def _np(t):
    x = t.cpu().numpy()
    return x.astype(np.complex128) if np.iscomplexobj(x) else x.astype(np.float64)


def _rel(a, b):
    a, b = _np(a), _np(b)
    return float(np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-30))


@pytest.fixture(scope="module")
def ssb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge
    ge.build()
    import electron_microscopy_gb300 as m
    m.load()
    return m


def _problem(ssb, name):
    from synth import forward as F
    d = F.make_numpy_dataset(name)
    geom, ab = d["geom"], d["ab"]
    bf = ssb.bf_indices(geom, ab)
    fr = d["frames"]
    frames = torch.from_numpy(fr.view(np.int16) if fr.dtype == np.uint16 else fr).cuda()
    bfd = torch.from_numpy(bf).cuda()
    G = ssb.build_G(frames, geom, bfd)
    return geom, ab, bfd, G


def _call_noalloc(ssb, G, geom, bfd, ab):
    lib = ssb.load()
    g = ssb.to_geometry(geom)
    a = ssb.to_aberr(ab)
    n, h = g.n, g.n // 2 + 1
    O = torch.full((n, h), float("nan"), dtype=torch.complex64, device=G.device)
    N = torch.full((n, h), -1, dtype=torch.int32, device=G.device)
    ph = torch.full((n, n), float("nan"), dtype=torch.float32, device=G.device)
    stream = ctypes.c_void_p(int(torch.cuda.current_stream().cuda_stream))
    rc = lib.ssb_reconstruct_noalloc(ctypes.c_void_p(G.data_ptr()), ctypes.byref(g),
                                     ctypes.c_void_p(bfd.data_ptr()), int(bfd.numel()), ctypes.byref(a),
                                     ctypes.c_void_p(O.data_ptr()), ctypes.c_void_p(N.data_ptr()),
                                     ctypes.c_void_p(ph.data_ptr()), stream)
    assert rc == ssb.SSB_OK, lib.ssb_last_error().decode()
    torch.cuda.synchronize()
    return O, N, ph


def test_noalloc_matches_workspace_entry_point_twice(ssb):
    # first call: the small workload; second call: the tiny one (another size,
    # so the scratch array holds the previous call's contents)
    for name in ("small", "tiny"):
        geom, ab, bfd, G = _problem(ssb, name)
        O_ref, N_ref, ph_ref = ssb.reconstruct(G, geom, bfd, ab)
        torch.cuda.synchronize()
        O, N, ph = _call_noalloc(ssb, G, geom, bfd, ab)
        assert torch.equal(N, N_ref)
        assert _rel(O, O_ref) <= TOL
        assert _rel(ph, ph_ref) <= TOL
        assert bool(torch.isfinite(ph).all())


def test_noalloc_rejects_oversized_problems(ssb):
    from synth import configs as C
    lib = ssb.load()
    g = C.Geometry(n=1024, det_y=192, det_x=192, scan_step_A=0.373, det_pitch_invA=0.028,
                   wavelength_A=0.019687, semiangle_rad=0.03, det_center_y=96, det_center_x=96)
    need = ssb.workspace_bytes(g, 9354, ssb.OP_RECON)
    assert need > ssb.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    a = ssb.Aberr()
    rc = lib.ssb_reconstruct_noalloc(fake, ctypes.byref(ssb.to_geometry(g)), fake, 9354, ctypes.byref(a),
                                     fake, fake, fake, None)
    assert rc == ssb.SSB_UNSUPPORTED
    assert "16 MiB" in lib.ssb_last_error().decode()


def test_noalloc_checks_arguments_before_the_size_limit(ssb):
    """A NULL output or an n_bf beyond the detector is an invalid argument, as
    for ssb_reconstruct, even on a problem too large for the fixed array."""
    from synth import configs as C
    lib = ssb.load()
    a = ssb.Aberr()
    fake = ctypes.c_void_p(1 << 20)
    big = C.Geometry(n=1024, det_y=192, det_x=192, scan_step_A=0.373, det_pitch_invA=0.028,
                     wavelength_A=0.019687, semiangle_rad=0.03, det_center_y=96, det_center_x=96)
    small = C.Geometry(n=64, det_y=8, det_x=8, scan_step_A=0.373, det_pitch_invA=0.4,
                       wavelength_A=0.019687, semiangle_rad=0.03, det_center_y=4, det_center_x=4)
    for g, n_bf, O in ((big, 9354, None), (small, 10, None), (small, 65, fake), (big, 192 * 192 + 1, fake)):
        rc = lib.ssb_reconstruct_noalloc(fake, ctypes.byref(ssb.to_geometry(g)), fake, n_bf, ctypes.byref(a),
                                         O, fake, fake, None)
        assert rc == ssb.SSB_INVALID_ARG, (g.n, n_bf, lib.ssb_last_error().decode())
