"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, computes the host-side index sets bit for bit like the
oracle, and rejects bad arguments with status codes before launching."""
import ctypes
import os
import re

import numpy as np
import pytest

import electron_microscopy_gb300 as ssb
from oracle import ssb_oracle as O
from synth import configs as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ssb.LIB_PATH):
        import __graft_entry__ as ge
        ge.build()
    return ssb.load()


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
            names |= set(re.findall(r"\b(ssb_[A-Za-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_names():
    assert set(_declared_functions()) == set(ssb.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", ssb.LIB_PATH], capture_output=True, text=True).stdout
    syms = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for fn in _declared_functions():
        assert fn in syms, fn
        assert hasattr(lib, fn)


@pytest.mark.parametrize("name", ["tiny", "small", "full", "large"])
@pytest.mark.parametrize("tilt", [(0.0, 0.0), (5.92e-3, -0.07e-3), (-3.3e-3, 7.1e-3)])
def test_bf_indices_match_oracle(lib, name, tilt):
    g = C.geometry(C.WORKLOADS[name])
    ab = C.Aberrations(tilt_x_rad=tilt[0], tilt_y_rad=tilt[1])
    got = ssb.bf_indices(g, ab)
    ref = O.bf_indices(g, *tilt)
    assert np.array_equal(got, ref)


def test_bf_indices_on_exact_edge(lib):
    # a geometry whose disk edge falls exactly on pixel centres
    g = C.Geometry(n=8, det_y=11, det_x=11, scan_step_A=1.0, det_pitch_invA=0.5,
                   wavelength_A=0.02, semiangle_rad=0.05, det_center_y=5.0, det_center_x=5.0)
    got = ssb.bf_indices(g, C.Aberrations())
    ref = O.bf_indices(g)
    assert np.array_equal(got, ref)
    assert len(ref) == 81  # radius 2.5 1/A = 5 px: the 4 axis pixels at distance 5 are in


@pytest.mark.parametrize("n", [8, 32, 128, 512, 1024])
def test_band_indices_match_oracle(lib, n):
    g = C.Geometry(n=n, det_y=8, det_x=8, scan_step_A=0.373, det_pitch_invA=0.1,
                   wavelength_A=0.019687, semiangle_rad=0.03, det_center_y=4, det_center_x=4)
    for lo, hi in [(0.2, 0.9), (0.0, 0.5), (0.0, 10.0), (1.0, 1.0)]:
        got = ssb.band_indices(g, lo, hi)
        ref = O.band_indices(g, lo, hi)
        assert np.array_equal(got, ref)


def test_band_count_printed_on_pages(lib):
    g = C.geometry(C.WORKLOADS["full"])
    assert len(ssb.band_indices(g, 0.2, 0.9)) == 44247


def test_workspace_bytes(lib):
    g = C.geometry(C.WORKLOADS["full"])
    assert ssb.workspace_bytes(g, 9354, ssb.OP_BUILD) > 0
    r = ssb.workspace_bytes(g, 9354, ssb.OP_RECON)
    assert r >= 512 * 257 * (8 + 4)
    s1 = ssb.workspace_bytes(g, 9354, ssb.OP_SCORE, 1, 44247)
    s8 = ssb.workspace_bytes(g, 9354, ssb.OP_SCORE, 8, 44247)
    assert 0 < s1 < s8
    assert ssb.workspace_bytes(g, 9354, ssb.OP_SCORE, 9, 44247) == 0
    assert ssb.workspace_bytes(g, 0, ssb.OP_RECON) == 0
    assert ssb.workspace_bytes(g, 10, 7) == 0
    m = ssb.workspace_bytes(g, 9354, ssb.OP_MOMENTS)
    # one chunk of 32 corrected half planes plus 8 float64 (sum, square) images
    assert m >= 32 * 512 * 257 * 8 + 8 * 512 * 512 * 16
    assert ssb.workspace_bytes(g, 0, ssb.OP_MOMENTS) == 0
    bad = C.Geometry(**{**g.__dict__, "n": 100})
    assert ssb.workspace_bytes(bad, 10, ssb.OP_RECON) == 0


def _g(**kw):
    g = C.geometry(C.WORKLOADS["tiny"])
    return ssb.to_geometry(C.Geometry(**{**g.__dict__, **kw}))


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its host checks


def _err(lib):
    return lib.ssb_last_error().decode()


def test_error_codes_build(lib):
    g = _g()
    big = 1 << 30
    rc = lib.ssb_build_G(None, 0, ctypes.byref(g), FAKE, 10, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG and "NULL" in _err(lib)
    rc = lib.ssb_build_G(FAKE, 7, ctypes.byref(g), FAKE, 10, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    for n in (100, 4, 2048, 0, -8):
        rc = lib.ssb_build_G(FAKE, 0, ctypes.byref(_g(n=n)), FAKE, 10, FAKE, FAKE, big, None)
        assert rc == ssb.SSB_UNSUPPORTED, n
    rc = lib.ssb_build_G(FAKE, 0, ctypes.byref(_g(det_x=0)), FAKE, 10, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    rc = lib.ssb_build_G(FAKE, 0, ctypes.byref(g), FAKE, 0, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    rc = lib.ssb_build_G(FAKE, 0, ctypes.byref(g), FAKE, 24 * 24 + 1, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    rc = lib.ssb_build_G(FAKE, 0, ctypes.byref(g), FAKE, 10, FAKE, FAKE, 16, None)
    assert rc == ssb.SSB_WORKSPACE_TOO_SMALL and "needs" in _err(lib)
    rc = lib.ssb_build_G(FAKE, 0, ctypes.byref(g), FAKE, 10, FAKE, ctypes.c_void_p((1 << 20) + 8), big, None)
    assert rc == ssb.SSB_INVALID_ARG and "aligned" in _err(lib)
    rc = lib.ssb_build_G(FAKE, 0, ctypes.byref(_g(wavelength_A=0.0)), FAKE, 10, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    rc = lib.ssb_build_G(FAKE, 0, None, FAKE, 10, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG


def test_error_codes_reconstruct_and_score(lib):
    g = _g()
    a = ssb.Aberr()
    big = 1 << 30
    rc = lib.ssb_reconstruct(FAKE, ctypes.byref(g), FAKE, 10, None, FAKE, FAKE, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    rc = lib.ssb_reconstruct(FAKE, ctypes.byref(g), FAKE, 10, ctypes.byref(a), FAKE, FAKE, FAKE, FAKE, 100, None)
    assert rc == ssb.SSB_WORKSPACE_TOO_SMALL
    nan = ssb.Aberr(C10=float("nan"))
    rc = lib.ssb_reconstruct(FAKE, ctypes.byref(g), FAKE, 10, ctypes.byref(nan), FAKE, FAKE, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    sets = (ssb.Aberr * 9)()
    for B in (0, 9):
        rc = lib.ssb_score_batch(FAKE, ctypes.byref(g), FAKE, 10, sets, B, FAKE, 5, FAKE, FAKE, FAKE, FAKE, big, None)
        assert rc == ssb.SSB_UNSUPPORTED, B
    rc = lib.ssb_score_batch(FAKE, ctypes.byref(g), FAKE, 10, sets, 2, FAKE, 0, FAKE, FAKE, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    rc = lib.ssb_score_batch(FAKE, ctypes.byref(g), FAKE, 10, sets, 2, FAKE, 32 * 17 + 1, FAKE, FAKE, FAKE, FAKE,
                             big, None)
    assert rc == ssb.SSB_INVALID_ARG
    rc = lib.ssb_score_batch(FAKE, ctypes.byref(g), FAKE, 10, sets, 2, None, 5, FAKE, FAKE, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    rc = lib.ssb_score_batch(FAKE, ctypes.byref(g), FAKE, 10, sets, 2, FAKE, 5, FAKE, FAKE, FAKE, FAKE, 64, None)
    assert rc == ssb.SSB_WORKSPACE_TOO_SMALL


def test_peak_probes_reject_bad_arguments(lib):
    before = lib.ssb_launch_count()
    assert lib.ssb_peak_sincos(None, 4, 4, None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_peak_fma(FAKE, 0, 4, None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_peak_fma(FAKE, 4, 0, None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_launch_count() == before


def test_no_launches_from_failed_checks(lib):
    before = lib.ssb_launch_count()
    g = _g(n=100)
    lib.ssb_build_G(FAKE, 0, ctypes.byref(g), FAKE, 10, FAKE, FAKE, 1 << 30, None)
    assert lib.ssb_launch_count() == before


def test_build_G_host_bytes(lib):
    """Workspace of the host-input build: the BF bounding box of every frame
    (rows padded to a multiple of 16 bytes), the remapped index list and the
    build workspace of the cropped detector."""
    g = C.geometry(C.WORKLOADS["full"])
    bf = O.bf_indices(g)
    rows, cols = bf // g.det_x, bf % g.det_x
    r0, r1, c0, c1 = int(rows.min()), int(rows.max()), int(cols.min()), int(cols.max())
    pitch = (c1 - (c0 & ~1) + 1 + 7) // 8 * 8
    crop = C.Geometry(**{**g.__dict__, "det_y": r1 - r0 + 1, "det_x": pitch})
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    want = (a256(g.n * g.n * (r1 - r0 + 1) * pitch * 2) + a256(len(bf) * 4)
            + ssb.workspace_bytes(crop, len(bf), ssb.OP_BUILD))
    assert ssb.build_G_host_bytes(g, bf, ssb.SSB_U16) == want
    # the full workload's disk spans rows and columns 42..150 of 192: 32 % of the frame bytes cross the link
    assert (r0, r1, c0, c1) == (42, 150, 42, 150)
    assert ssb.build_G_host_bytes(g, bf, ssb.SSB_F32) > want
    assert ssb.build_G_host_bytes(g, np.array([-1], np.int32), ssb.SSB_U16) == 0
    assert ssb.build_G_host_bytes(g, np.array([g.det_y * g.det_x], np.int32), ssb.SSB_U16) == 0
    assert ssb.build_G_host_bytes(g, bf, 7) == 0


def test_error_codes_build_host(lib):
    g = _g()
    big = 1 << 40
    bf = np.array([5, 30, 100], np.int32)
    bfp = bf.ctypes.data_as(ctypes.c_void_p)
    before = lib.ssb_launch_count()
    rc = lib.ssb_build_G_host(None, 0, ctypes.byref(g), bfp, FAKE, 3, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG and "NULL" in _err(lib)
    rc = lib.ssb_build_G_host(FAKE, 0, ctypes.byref(g), None, FAKE, 3, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    bad = np.array([5, 24 * 24], np.int32)
    rc = lib.ssb_build_G_host(FAKE, 0, ctypes.byref(g), bad.ctypes.data_as(ctypes.c_void_p), FAKE, 2, FAKE, FAKE,
                              big, None)
    assert rc == ssb.SSB_INVALID_ARG and "outside the detector" in _err(lib)
    rc = lib.ssb_build_G_host(FAKE, 0, ctypes.byref(g), bfp, FAKE, 3, FAKE, FAKE, 64, None)
    assert rc == ssb.SSB_WORKSPACE_TOO_SMALL
    rc = lib.ssb_build_G_host(FAKE, 0, ctypes.byref(_g(n=100)), bfp, FAKE, 3, FAKE, FAKE, big, None)
    assert rc == ssb.SSB_UNSUPPORTED
    assert lib.ssb_launch_count() == before


def test_error_codes_compact_storage(lib):
    """The compact-storage entry points and the G descriptor are checked on
    the host and rejected before anything is launched."""
    g = _g()  # n = 32
    before = lib.ssb_launch_count()
    S = ssb.GStoreC
    big = 1 << 30
    # ssb_compact_G16
    assert lib.ssb_compact_G16(None, ctypes.byref(g), 10, 1, FAKE, FAKE, None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_compact_G16(FAKE, ctypes.byref(g), 0, 1, FAKE, FAKE, None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_compact_G16(FAKE, ctypes.byref(g), 10, 1, FAKE, None, None) == ssb.SSB_INVALID_ARG
    for rows in (0, 2, 16, 64):
        assert lib.ssb_compact_G16(FAKE, ctypes.byref(g), 10, rows, FAKE, FAKE, None) == ssb.SSB_UNSUPPORTED, rows
    # ssb_compact_band
    src = S(FAKE.value, ssb.G_C64, 0, 0, 0)
    assert lib.ssb_compact_band(None, ctypes.byref(g), 10, FAKE, 5, FAKE, None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_compact_band(ctypes.byref(src), ctypes.byref(g), 10, FAKE, 0, FAKE, None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_compact_band(ctypes.byref(src), ctypes.byref(g), 10, FAKE, 32 * 17 + 1, FAKE,
                                None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_compact_band(ctypes.byref(src), ctypes.byref(g), 0, FAKE, 5, FAKE, None) == ssb.SSB_INVALID_ARG
    bad = S(FAKE.value, 7, 0, 0, 0)
    assert lib.ssb_compact_band(ctypes.byref(bad), ctypes.byref(g), 10, FAKE, 5, FAKE, None) == ssb.SSB_INVALID_ARG
    banded = S(FAKE.value, ssb.G_C64, 0, 0, 1)
    assert lib.ssb_compact_band(ctypes.byref(banded), ctypes.byref(g), 10, FAKE, 5, FAKE,
                                None) == ssb.SSB_INVALID_ARG
    # descriptors the reductions reject
    a = ssb.Aberr()
    sets = (ssb.Aberr * 2)()
    no_scale = S(FAKE.value, ssb.G_SN16, 0, 1, 0)
    odd_rows = S(FAKE.value, ssb.G_SN16, FAKE.value, 4, 0)
    for store, code in ((bad, ssb.SSB_INVALID_ARG), (no_scale, ssb.SSB_INVALID_ARG),
                        (odd_rows, ssb.SSB_UNSUPPORTED)):
        rc = lib.ssb_reconstruct_g(ctypes.byref(store), ctypes.byref(g), FAKE, 10, ctypes.byref(a), FAKE, FAKE,
                                   FAKE, FAKE, big, None)
        assert rc == code
        rc = lib.ssb_score_batch_g(ctypes.byref(store), ctypes.byref(g), FAKE, 10, sets, 2, FAKE, 5, FAKE, FAKE,
                                   FAKE, FAKE, big, None)
        assert rc == code
    rc = lib.ssb_reconstruct_g(ctypes.byref(banded), ctypes.byref(g), FAKE, 10, ctypes.byref(a), FAKE, FAKE, FAKE,
                               FAKE, big, None)
    assert rc == ssb.SSB_INVALID_ARG
    assert lib.ssb_reconstruct_g(None, ctypes.byref(g), FAKE, 10, ctypes.byref(a), FAKE, FAKE, FAKE, FAKE, big,
                                 None) == ssb.SSB_INVALID_ARG
    assert lib.ssb_launch_count() == before


def test_error_codes_phase_moments(lib):
    g = _g()
    a = ssb.Aberr()
    S = ssb.GStoreC
    big = 1 << 30
    before = lib.ssb_launch_count()
    ok = S(FAKE.value, ssb.G_C64, 0, 0, 0)
    banded = S(FAKE.value, ssb.G_C64, 0, 0, 1)
    nan = ssb.Aberr(C30=float("inf"))
    cases = [
        ((None, ctypes.byref(g), FAKE, 10, ctypes.byref(a), FAKE, FAKE, FAKE, big, None), ssb.SSB_INVALID_ARG),
        ((ctypes.byref(banded), ctypes.byref(g), FAKE, 10, ctypes.byref(a), FAKE, FAKE, FAKE, big, None),
         ssb.SSB_INVALID_ARG),
        ((ctypes.byref(ok), ctypes.byref(g), FAKE, 10, ctypes.byref(a), None, FAKE, FAKE, big, None),
         ssb.SSB_INVALID_ARG),
        ((ctypes.byref(ok), ctypes.byref(g), FAKE, 0, ctypes.byref(a), FAKE, FAKE, FAKE, big, None),
         ssb.SSB_INVALID_ARG),
        ((ctypes.byref(ok), ctypes.byref(g), FAKE, 10, ctypes.byref(nan), FAKE, FAKE, FAKE, big, None),
         ssb.SSB_INVALID_ARG),
        ((ctypes.byref(ok), ctypes.byref(g), FAKE, 10, ctypes.byref(a), FAKE, FAKE, FAKE, 1000, None),
         ssb.SSB_WORKSPACE_TOO_SMALL),
        ((ctypes.byref(ok), ctypes.byref(_g(n=12)), FAKE, 10, ctypes.byref(a), FAKE, FAKE, FAKE, big, None),
         ssb.SSB_UNSUPPORTED),
    ]
    for args, code in cases:
        assert lib.ssb_phase_moments(*args) == code, _err(lib)
    assert lib.ssb_launch_count() == before
