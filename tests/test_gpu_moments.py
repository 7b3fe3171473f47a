"""GPU parity of the per-BF phase moments (the exact mean(angle) path)
through the C ABI, against the oracle on the same seeded inputs: the mean and
the population variance over BF pixels of atan2(b_k, a_k) within the float32
tolerance (relative L2 <= 1e-4), from a complex64 or a herm16 G."""
import numpy as np
import pytest

from oracle import ssb_oracle as O
from synth import configs as C

pytestmark = pytest.mark.gpu

TOL = 1e-4

torch = pytest.importorskip("torch")


def rel(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    den = np.linalg.norm(b.ravel())
    return float(np.linalg.norm((a - b).ravel()) / (den if den > 0 else 1.0))


@pytest.fixture(scope="module")
def ssb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge
    ge.build()
    import electron_microscopy_gb300 as m
    return m


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _frames_dev(frames):
    if frames.dtype == np.uint16:
        return _dev(frames.view(np.int16))
    return _dev(frames)


def _check(ssb, frames, geom, ab, tol=TOL):
    bf = O.bf_indices(geom, ab.tilt_x_rad, ab.tilt_y_rad)
    bfd = _dev(bf)
    G = ssb.build_G(_frames_dev(frames), geom, bfd)
    mean, var = ssb.phase_moments(G, geom, bfd, ab)
    torch.cuda.synchronize()
    Gor = O.build_G(frames, bf)
    mref, vref = O.phase_moments(Gor, geom, ab, bf)
    assert np.all(np.isfinite(mean.cpu().numpy())) and var.min().item() >= 0
    assert rel(mean.cpu().numpy(), mref) < tol
    assert rel(var.cpu().numpy(), vref) < tol
    return G, bf, mean, var, Gor


def test_tiny_workload(ssb, tiny_dataset):
    d = tiny_dataset
    _check(ssb, d["frames"], d["geom"], d["ab"])


def test_small_workload(ssb, small_dataset):
    d = small_dataset
    _check(ssb, d["frames"], d["geom"], d["ab"])


AB = C.Aberrations(C10=-60.0, C12a=12.0, C12b=-20.0, C21a=15.0, C21b=-9.0, C23a=20.0, C23b=5.0,
                   C30=3e3, C32a=-1e3, C32b=500.0, C34a=800.0, C34b=-600.0, tilt_x_rad=2e-3, tilt_y_rad=-1e-3)


@pytest.mark.parametrize("n,det,dk", [(8, 6, 0.6), (64, 14, 0.25), (256, 10, 0.4)])
def test_random_counts_sizes(ssb, n, det, dk):
    """Sizes from the smallest scan to several chunks of 32 BF pixels with a
    ragged last chunk (the det 14 case), uint16 counts."""
    rng = np.random.default_rng(300 + n)
    g = C.Geometry(n=n, det_y=det, det_x=det, scan_step_A=C.SCAN_STEP_A, det_pitch_invA=dk,
                   wavelength_A=C.WAVELENGTH_300KV_A, semiangle_rad=C.SEMIANGLE_RAD,
                   det_center_y=det // 2, det_center_x=det // 2)
    frames = rng.poisson(6.0, size=(n, n, det, det)).astype(np.uint16)
    _check(ssb, frames, g, AB)


@pytest.mark.parametrize("per_row", [False, True])
def test_herm16_store(ssb, small_dataset, per_row):
    d = small_dataset
    g, ab = d["geom"], d["ab"]
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    bfd = _dev(bf)
    G = ssb.build_G(_frames_dev(d["frames"]), g, bfd)
    rows = 1 if per_row else g.n
    mean, var = ssb.phase_moments(ssb.compact_G16(G, g, rows), g, bfd, ab)
    torch.cuda.synchronize()
    Gor = O.build_G(d["frames"], bf)
    codes, sc = O.herm16_pack(Gor.astype(np.complex64), rows)
    mref, vref = O.phase_moments(O.herm16_unpack(codes, sc, rows), g, ab, bf)
    assert rel(mean.cpu().numpy(), mref) < TOL
    assert rel(var.cpu().numpy(), vref) < TOL


def test_one_pixel_and_determinism(ssb, small_dataset):
    d = small_dataset
    g, ab = d["geom"], d["ab"]
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    bfd = _dev(bf)
    G = ssb.build_G(_frames_dev(d["frames"]), g, bfd)
    a = ssb.phase_moments(G, g, bfd, ab)
    b = ssb.phase_moments(G, g, bfd, ab)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    k = len(bf) // 3
    mean, var = ssb.phase_moments(G[k:k + 1].contiguous(), g, bfd[k:k + 1].contiguous(), ab)
    (ak, bk), = list(O.per_bf_images(O.build_G(d["frames"], bf[k:k + 1]), g, ab, bf[k:k + 1]))
    ref = np.arctan2(bk, ak)
    assert rel(mean.cpu().numpy(), ref) < TOL
    assert var.max().item() <= 1e-6 * float(np.max(ref * ref))
