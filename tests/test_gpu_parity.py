"""GPU parity: the CUDA library (called through its C ABI) against the CPU
oracle on the same seeded inputs.

Bars: bit-exact for integer work (trotter counts N, BF and band index sets);
relative L2 <= 1e-4 for the float32 paths (G, O, phase, score), the tolerance
stated for the hot path's float32 results.
"""
import numpy as np
import pytest

from oracle import ssb_oracle as O
from synth import configs as C
from synth import forward as F

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


def _run_all(ssb, frames, geom, ab, bf):
    fd = _frames_dev(frames)
    bfd = _dev(bf)
    G = ssb.build_G(fd, geom, bfd)
    Od, Nd, ph = ssb.reconstruct(G, geom, bfd, ab)
    torch.cuda.synchronize()
    return G.cpu().numpy(), Od.cpu().numpy(), Nd.cpu().numpy(), ph.cpu().numpy()


def _check_against_oracle(ssb, frames, geom, ab, tol=TOL):
    bf = O.bf_indices(geom, ab.tilt_x_rad, ab.tilt_y_rad)
    assert np.array_equal(ssb.bf_indices(geom, ab), bf)
    G, Od, Nd, ph = _run_all(ssb, frames, geom, ab, bf)
    ref = O.reconstruct(frames, geom, ab, bf_idx=bf)
    n, h = geom.n, geom.n // 2 + 1
    assert G.shape == (len(bf), n, h)
    assert rel(G, ref["G"]) < tol
    assert np.array_equal(Nd.ravel(), ref["N"])
    assert rel(Od.ravel(), ref["O"]) < tol
    assert rel(ph, ref["phase"]) < tol
    return G, Od, Nd, ph, ref


# ----------------------------------------------------------------------------
# the seeded workloads
# ----------------------------------------------------------------------------

def test_tiny_workload(ssb, tiny_dataset):
    d = tiny_dataset
    _, _, _, ph, ref = _check_against_oracle(ssb, d["frames"], d["geom"], d["ab"])
    # the recovered phase tracks the ground truth like the oracle's does
    r = np.corrcoef(ph.ravel(), d["truth"].ravel())[0, 1]
    assert r > 0.95


def test_small_workload(ssb, small_dataset):
    d = small_dataset
    _check_against_oracle(ssb, d["frames"], d["geom"], d["ab"])


# ----------------------------------------------------------------------------
# sizes, ragged tails and edge cases on random counts
# ----------------------------------------------------------------------------

def _geom(n, det, dk, step=C.SCAN_STEP_A):
    return C.Geometry(n=n, det_y=det, det_x=det, scan_step_A=step, det_pitch_invA=dk,
                      wavelength_A=C.WAVELENGTH_300KV_A, semiangle_rad=C.SEMIANGLE_RAD,
                      det_center_y=det // 2, det_center_x=det // 2)


AB = C.Aberrations(C10=-60.0, C12a=12.0, C12b=-20.0, C21a=15.0, C21b=-9.0, C23a=20.0, C23b=5.0,
                   C30=4e3, C32a=-3e3, C32b=2e3, C34a=1e3, C34b=-2.5e3, tilt_x_rad=2e-3, tilt_y_rad=-1e-3)


@pytest.mark.parametrize("n,det,dk", [(8, 6, 0.6), (16, 10, 0.35), (64, 14, 0.25), (256, 10, 0.4)])
def test_random_counts_sizes(ssb, n, det, dk):
    rng = np.random.default_rng(n)
    frames = rng.poisson(3.0, size=(n, n, det, det)).astype(np.uint16)
    _check_against_oracle(ssb, frames, _geom(n, det, dk), AB)


def test_float32_frames_ragged(ssb):
    # n_bf = 45: one full 32-pixel group plus a ragged tail
    rng = np.random.default_rng(7)
    n, det = 32, 9
    frames = rng.uniform(0, 10, size=(n, n, det, det)).astype(np.float32)
    g = _geom(n, det, 0.45)
    bf = O.bf_indices(g, AB.tilt_x_rad, AB.tilt_y_rad)
    assert len(bf) % 32 != 0
    _check_against_oracle(ssb, frames, g, AB)


def test_single_bf_pixel(ssb):
    rng = np.random.default_rng(8)
    n = 32
    g = C.Geometry(n=n, det_y=3, det_x=3, scan_step_A=C.SCAN_STEP_A, det_pitch_invA=2.0,
                   wavelength_A=C.WAVELENGTH_300KV_A, semiangle_rad=C.SEMIANGLE_RAD,
                   det_center_y=1, det_center_x=1)
    bf = O.bf_indices(g)
    assert len(bf) == 1
    frames = rng.poisson(5.0, size=(n, n, 3, 3)).astype(np.uint16)
    _check_against_oracle(ssb, frames, g, C.Aberrations(C10=30.0))


def test_full_scan_size_small_detector(ssb):
    """n = 512 (the full workload's FFT and image launch geometry) with a
    12 x 12 detector so the oracle finishes in seconds."""
    rng = np.random.default_rng(9)
    n, det = 512, 12
    frames = rng.poisson(3.0, size=(n, n, det, det)).astype(np.uint16)
    g = _geom(n, det, 0.33)
    _check_against_oracle(ssb, frames, g, AB)


@pytest.mark.parametrize("det,dk", [(16, 0.2), (24, 0.13)])
def test_full_scan_size_aligned_detectors(ssb, det, dk):
    """n = 512 with detector rows a multiple of 16 bytes: the build reads
    8-pixel pieces of each frame in one 16-byte load."""
    rng = np.random.default_rng(40 + det)
    n = 512
    frames = rng.poisson(3.0, size=(n, n, det, det)).astype(np.uint16)
    _check_against_oracle(ssb, frames, _geom(n, det, dk), AB)


def test_full_scan_size_any_index_order(ssb):
    """n = 512: a BF list in random order with a repeated index and isolated
    pixels builds, entry by entry, the oracle's planes."""
    rng = np.random.default_rng(44)
    n, det = 512, 16
    frames = rng.poisson(3.0, size=(n, n, det, det)).astype(np.uint16)
    g = _geom(n, det, 0.2)
    bf = O.bf_indices(g, AB.tilt_x_rad, AB.tilt_y_rad)
    lst = np.concatenate([rng.permutation(bf)[:40], bf[:3], [bf[5], 0, det * det - 1]]).astype(np.int32)
    G = ssb.build_G(_frames_dev(frames), g, _dev(lst))
    torch.cuda.synchronize()
    assert rel(G.cpu().numpy(), O.build_G(frames, lst)) < TOL


def test_full_scan_size_float32_frames(ssb):
    """n = 512 with float32 frames (the general two-pass kernels at this size)."""
    rng = np.random.default_rng(11)
    n, det = 512, 8
    frames = rng.uniform(0, 6, size=(n, n, det, det)).astype(np.float32)
    g = _geom(n, det, 0.45)
    _check_against_oracle(ssb, frames, g, AB)


@pytest.mark.parametrize("dtype", [np.uint16, np.float32])
def test_max_scan_size_1024(ssb, dtype):
    """n = 1024: the 32 x 32 column kernel for both frame types and, for uint16
    frames, the 16-pixel row kernel; 31 BF pixels = one full pixel group plus
    a ragged one."""
    rng = np.random.default_rng(10)
    n, det = 1024, 6
    frames = rng.poisson(3.0, size=(n, n, det, det)).astype(dtype)
    g = _geom(n, det, 0.45)
    ab = AB.replace(tilt_x_rad=0.0, tilt_y_rad=0.0)
    assert 16 < len(O.bf_indices(g)) < 32
    _check_against_oracle(ssb, frames, g, ab)


def test_zero_frames_give_zero_G_and_flat_phase(ssb):
    n, det = 16, 8
    frames = np.zeros((n, n, det, det), dtype=np.uint16)
    frames[..., :, :] = 4
    g = _geom(n, det, 0.4)
    bf = O.bf_indices(g)
    G, Od, Nd, ph = _run_all(ssb, frames, g, C.Aberrations(), bf)
    assert np.allclose(G[:, 0, 0], 4.0 * n * n)
    G2 = G.copy()
    G2[:, 0, 0] = 0
    assert np.abs(G2).max() < 1e-3
    assert np.abs(ph).max() < 1e-6


# ----------------------------------------------------------------------------
# batched scoring
# ----------------------------------------------------------------------------

@pytest.fixture(scope="module")
def small_G(ssb, small_dataset):
    d = small_dataset
    bf = O.bf_indices(d["geom"], d["ab"].tilt_x_rad, d["ab"].tilt_y_rad)
    G = ssb.build_G(_frames_dev(d["frames"]), d["geom"], _dev(bf))
    return d, bf, G


def test_score_batch_matches_oracle(ssb, small_G):
    d, bf, G = small_G
    g = d["geom"]
    band = O.band_indices(g, 0.2, 0.9)
    sets = C.perturbed_sets(d["ab"], 8, seed=4)
    Ob, Nb, sc = ssb.score_batch(G, g, _dev(bf), sets, _dev(band))
    torch.cuda.synchronize()
    Gor = O.build_G(d["frames"], bf)
    for s, ab in enumerate(sets):
        Oref, Nref = O.reduce(Gor, g, ab, bf, entries=band)
        assert np.array_equal(Nb[s].cpu().numpy(), Nref)
        assert rel(Ob[s].cpu().numpy(), Oref) < TOL
        assert abs(sc[s].item() - O.score(Oref, Nref)) <= TOL * abs(O.score(Oref, Nref))


def test_score_batch_B_invariance(ssb, small_G):
    """Set s of an 8-set pass equals the single-set pass bit for bit."""
    d, bf, G = small_G
    g = d["geom"]
    band = _dev(O.band_indices(g, 0.2, 0.9))
    bfd = _dev(bf)
    sets = C.perturbed_sets(d["ab"], 8, seed=11)
    O8, N8, s8 = ssb.score_batch(G, g, bfd, sets, band)
    for B in (2, 4, 5):
        OB, NB, sB = ssb.score_batch(G, g, bfd, sets[:B], band)
        assert torch.equal(OB, O8[:B]) and torch.equal(NB, N8[:B]) and torch.equal(sB, s8[:B])
    for s in range(8):
        O1, N1, s1 = ssb.score_batch(G, g, bfd, [sets[s]], band)
        assert torch.equal(O1[0], O8[s]) and torch.equal(N1[0], N8[s]) and torch.equal(s1[0], s8[s])


def test_score_of_matched_set_is_highest(ssb, tiny_dataset):
    """Noiseless data: the simulated set outscores sets with defocus steps."""
    d = tiny_dataset
    g = d["geom"]
    bf = O.bf_indices(g)
    G = ssb.build_G(_frames_dev(d["frames"]), g, _dev(bf))
    band = _dev(O.band_indices(g, 0.2, 0.9))
    sets = [d["ab"].replace(C10=d["ab"].C10 + dz) for dz in (-40.0, -20.0, 0.0, 20.0, 40.0)]
    _, _, sc = ssb.score_batch(G, g, _dev(bf), sets, band)
    assert int(torch.argmax(sc)) == 2


def test_reconstruct_both_dispatch_paths(ssb, small_G):
    """G rows 16-byte aligned: the reconstruction streams them through
    shared memory (TMA kernel); G shifted by one complex entry (8 bytes): the
    per-thread-load kernel.  Both match the oracle (N bit for bit, O and the
    phase within 1e-4) and each other."""
    d, bf, G = small_G
    bfd = _dev(bf)
    buf = torch.empty(G.numel() + 1, dtype=G.dtype, device=G.device)
    Gs = buf[1:].view(G.shape)
    Gs.copy_(G)
    assert G.data_ptr() % 16 == 0 and Gs.data_ptr() % 16 == 8
    a = ssb.reconstruct(G, d["geom"], bfd, d["ab"])
    b = ssb.reconstruct(Gs, d["geom"], bfd, d["ab"])
    torch.cuda.synchronize()
    ref = O.reconstruct(d["frames"], d["geom"], d["ab"], bf_idx=bf)
    for Od, Nd, ph in (a, b):
        assert np.array_equal(Nd.cpu().numpy().ravel(), ref["N"])
        assert rel(Od.cpu().numpy().ravel(), ref["O"]) < TOL
        assert rel(ph.cpu().numpy(), ref["phase"]) < TOL
    assert torch.equal(a[1], b[1])
    assert rel(a[0].cpu().numpy(), b[0].cpu().numpy()) < 1e-5


def test_reconstruct_is_deterministic(ssb, small_G):
    d, bf, G = small_G
    bfd = _dev(bf)
    a = ssb.reconstruct(G, d["geom"], bfd, d["ab"])
    b = ssb.reconstruct(G, d["geom"], bfd, d["ab"])
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_build_G_host_on_two_streams(ssb, small_dataset):
    """Host-input builds issued on two streams in turn, one stream reusing its
    workspace while its previous build may still be reading it: the copies
    queue on the library's copy stream, yet every build sees its own frames
    (each G bit for bit the device-input build of the same frames)."""
    d = small_dataset
    g, ab = d["geom"], d["ab"]
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    bfd = _dev(bf)
    f1 = d["frames"]
    f2 = np.ascontiguousarray(f1[::-1, ::-1])  # another scan: frames in reverse scan order
    ref = [ssb.build_G(_frames_dev(f), g, bfd) for f in (f1, f2)]
    hosts = [torch.from_numpy(f.view(np.int16)).pin_memory() for f in (f1, f2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ws = [ssb.Workspace(ssb.build_G_host_bytes(g, bf, ssb.SSB_U16), bfd.device) for _ in range(2)]
    order = [(0, 0), (1, 1), (0, 1), (1, 0), (0, 0), (1, 1)]  # (stream and workspace, frames)
    out = []
    for lane, fi in order:
        G = torch.empty_like(ref[0])
        ssb.build_G_host(hosts[fi], g, bf, bfd, G=G, ws=ws[lane], stream=streams[lane])
        out.append((G, fi))
    torch.cuda.synchronize()
    for G, fi in out:
        assert torch.equal(G, ref[fi])


@pytest.mark.parametrize("case", ["tiny", "small", "n512", "whole"])
def test_build_G_host_equals_device_build(ssb, case, tiny_dataset, small_dataset):
    """The host-input build copies only the bright-field bounding box of each
    frame (3D copy; "whole": every pixel is bright field, the 2D path); G is
    bit for bit the device-input build's, and matches the oracle."""
    if case == "n512":
        rng = np.random.default_rng(21)
        frames = rng.poisson(3.0, size=(512, 512, 12, 12)).astype(np.uint16)
        g, ab = _geom(512, 12, 0.33), AB
    elif case == "whole":
        rng = np.random.default_rng(22)
        frames = rng.poisson(4.0, size=(64, 64, 6, 6)).astype(np.uint16)
        g, ab = _geom(64, 6, 0.05), C.Aberrations()
    else:
        d = tiny_dataset if case == "tiny" else small_dataset
        frames, g, ab = d["frames"], d["geom"], d["ab"]
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    rows, cols = bf // g.det_x, bf % g.det_x
    if case == "whole":
        assert len(bf) == g.det_y * g.det_x
    else:  # the copy really skips rows and columns
        assert rows.max() - rows.min() + 1 < g.det_y and cols.max() - cols.min() + 1 < g.det_x
    bfd = _dev(bf)
    Gd = ssb.build_G(_frames_dev(frames), g, bfd)
    host = torch.from_numpy(np.ascontiguousarray(frames.view(np.int16) if frames.dtype == np.uint16
                                                 else frames)).pin_memory()
    Gh = ssb.build_G_host(host, g, bf, bfd)
    torch.cuda.synchronize()
    assert torch.equal(Gh, Gd)
    if case != "n512":
        assert rel(Gh.cpu().numpy(), O.build_G(frames, bf)) < TOL


# ----------------------------------------------------------------------------
# batched scoring with a different probe tilt per set: the reduction then
# takes each set's own aperture tests (its aperture bit at k, its trotter
# classes at k -/+ q) instead of sharing one set of tests across the batch
# ----------------------------------------------------------------------------

# tilt offsets (mrad) added to the base tilt, set by set; the third moves the
# disk by several detector pixels on both workloads below
TILT_STEPS_MRAD = [(0.0, 0.0), (1.5, -0.5), (9.0, -6.0), (-2.0, 1.0), (0.4, 2.5), (-3.5, -3.0),
                   (2.0, 2.0), (-0.8, 0.3)]


def _tilted_sets(base, B, seed):
    sets = C.perturbed_sets(base, B, seed=seed)
    return [s.replace(tilt_x_rad=base.tilt_x_rad + dx * 1e-3, tilt_y_rad=base.tilt_y_rad + dy * 1e-3)
            for s, (dx, dy) in zip(sets, TILT_STEPS_MRAD)]


def _per_set_tilt_case(case, small_dataset):
    if case == "small":
        d = small_dataset
        return d["frames"], d["geom"], d["ab"]
    rng = np.random.default_rng(31)
    n, det = 512, 20
    frames = rng.poisson(3.0, size=(n, n, det, det)).astype(np.uint16)
    return frames, _geom(n, det, 0.2), AB


@pytest.mark.parametrize("case", ["small", "n512"])
@pytest.mark.parametrize("B", [3, 8])
def test_score_batch_per_set_tilts_match_oracle(ssb, case, B, small_dataset):
    """Sets with distinct tilts: N bit-exact, O within 1e-4 and the score within
    1e-4, set by set, against the oracle's reduction."""
    frames, g, base = _per_set_tilt_case(case, small_dataset)
    bf = O.bf_indices(g, base.tilt_x_rad, base.tilt_y_rad)
    sets = _tilted_sets(base, B, seed=40 + B)
    # the sets really differ in tilt, by several pixels for one of them
    shift = max(C.tilt_shift_px(g, s.replace(tilt_x_rad=s.tilt_x_rad - base.tilt_x_rad,
                                             tilt_y_rad=s.tilt_y_rad - base.tilt_y_rad)) for s in sets)
    assert len({(s.tilt_x_rad, s.tilt_y_rad) for s in sets}) == B and shift > 1.5
    band = O.band_indices(g, 0.2, 0.9)
    G = ssb.build_G(_frames_dev(frames), g, _dev(bf))
    Ob, Nb, sc = ssb.score_batch(G, g, _dev(bf), sets, _dev(band))
    torch.cuda.synchronize()
    Gor = O.build_G(frames, bf)
    for s, ab in enumerate(sets):
        Oref, Nref = O.reduce(Gor, g, ab, bf, entries=band)
        assert np.array_equal(Nb[s].cpu().numpy(), Nref), f"set {s}: trotter counts differ"
        assert rel(Ob[s].cpu().numpy(), Oref) < TOL, f"set {s}"
        ref = O.score(Oref, Nref)
        assert abs(sc[s].item() - ref) <= TOL * abs(ref), f"set {s}"
    # a tilted set changes which pixels are trotter pixels
    assert not torch.equal(Nb[0], Nb[2])


@pytest.mark.parametrize("case", ["small", "n512"])
def test_score_batch_per_set_tilts_B_invariance(ssb, case, small_dataset):
    """Per-set tilts: set s of the 8-set pass equals the same set in a shorter
    pass and in a single-set pass, bit for bit."""
    frames, g, base = _per_set_tilt_case(case, small_dataset)
    bf = O.bf_indices(g, base.tilt_x_rad, base.tilt_y_rad)
    bfd = _dev(bf)
    band = _dev(O.band_indices(g, 0.2, 0.9))
    G = ssb.build_G(_frames_dev(frames), g, bfd)
    sets = _tilted_sets(base, 8, seed=53)
    O8, N8, s8 = ssb.score_batch(G, g, bfd, sets, band)
    for B in (2, 3, 5):
        OB, NB, sB = ssb.score_batch(G, g, bfd, sets[:B], band)
        assert torch.equal(OB, O8[:B]) and torch.equal(NB, N8[:B]) and torch.equal(sB, s8[:B])
    for s in range(8):
        O1, N1, s1 = ssb.score_batch(G, g, bfd, [sets[s]], band)
        assert torch.equal(O1[0], O8[s]) and torch.equal(N1[0], N8[s]) and torch.equal(s1[0], s8[s])


# ----------------------------------------------------------------------------
# a reconstruction split over shards of the BF pixels, through the library
# ----------------------------------------------------------------------------

def test_sharded_reconstruction_through_the_library(ssb, small_G):
    """ssb_reconstruct_sums on each shard, the shards' sums added on the
    device, ssb_phase_from_sums: N bit-exact and O, phase within 1e-4 of the
    whole reconstruction and of the oracle; one shard holding every pixel
    reproduces ssb_reconstruct bit for bit."""
    d, bf, G = small_G
    g, ab = d["geom"], d["ab"]
    bfd = _dev(bf)
    O_ref, N_ref, ph_ref = ssb.reconstruct(G, g, bfd, ab)
    O1, N1, s1 = ssb.reconstruct_sums(G, g, bfd, ab)
    ph1 = ssb.phase_from_sums(O1, N1, s1, len(bf), g)
    torch.cuda.synchronize()
    assert torch.equal(O1, O_ref) and torch.equal(N1, N_ref) and torch.equal(ph1, ph_ref)
    assert abs(s1.item() - float(G[:, 0, 0].real.double().sum())) <= 1e-9 * abs(s1.item())
    # two shards, split away from the reduction's 64-pixel chunks
    h = len(bf) * 3 // 7
    parts = [ssb.reconstruct_sums(G[a:b], g, bfd[a:b], ab) for a, b in ((0, h), (h, len(bf)))]
    O2 = parts[0][0] + parts[1][0]
    N2 = parts[0][1] + parts[1][1]
    s2 = parts[0][2] + parts[1][2]
    ph2 = ssb.phase_from_sums(O2, N2, s2, len(bf), g)
    torch.cuda.synchronize()
    assert torch.equal(N2, N_ref)
    assert rel(O2.cpu().numpy(), O_ref.cpu().numpy()) < TOL
    assert rel(ph2.cpu().numpy(), ph_ref.cpu().numpy()) < TOL
    ref = O.reconstruct(d["frames"], g, ab, bf_idx=bf)
    assert rel(ph2.cpu().numpy(), ref["phase"]) < TOL
