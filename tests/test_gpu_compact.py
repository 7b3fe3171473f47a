"""GPU parity of the compact G storage: herm16 (snorm16 codes with per-BF or
per-q-row float32 scales) and the band-compacted copy, through the C ABI.

Bars: the packer and the band copy are integer/byte work and must match the
oracle bit for bit on the same seeded float32 input; reductions over a stored
G match the oracle's reduction over its own dequantised G within the float32
tolerance (relative L2 <= 1e-4), with the trotter counts exact; a
band-compacted copy scores bit for bit like the half plane it came from.
"""
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


def _seeded_G(seed, nbf, n):
    """complex64 half planes with magnitudes over 12 decades, a DC-like peak,
    one empty pixel, one empty q row and entries exactly at +/- the scale."""
    rng = np.random.default_rng(seed)
    h = n // 2 + 1
    mag = 10.0 ** rng.uniform(-6, 6, size=(nbf, n, h))
    G = (mag * np.exp(1j * rng.uniform(-np.pi, np.pi, size=(nbf, n, h)))).astype(np.complex64)
    G[:, 0, 0] = (10.0 ** rng.uniform(6, 7, size=nbf)).astype(np.float32)
    if nbf > 2:
        G[1] = 0
        G[2, n // 2] = 0
        G[2, 1, :] = 0
        G[2, 1, 0] = 3.0
        G[2, 1, 1] = -3.0
        G[2, 1, 2] = 3.0j
    return G


def _codes(G16):
    """int32 words -> int16 (re, im) pairs."""
    w = G16.cpu().numpy()
    return w.view(np.int16).reshape(w.shape + (2,))


@pytest.mark.parametrize("n,nbf", [(8, 3), (64, 37), (512, 19)])
@pytest.mark.parametrize("per_row", [False, True])
def test_compact_G16_bitexact(ssb, n, nbf, per_row):
    G = _seeded_G(100 + n, nbf, n)
    g = C.Geometry(n=n, det_y=8, det_x=8, scan_step_A=C.SCAN_STEP_A, det_pitch_invA=0.2,
                   wavelength_A=C.WAVELENGTH_300KV_A, semiangle_rad=C.SEMIANGLE_RAD, det_center_y=4, det_center_x=4)
    rows = 1 if per_row else n
    st = ssb.compact_G16(_dev(G), g, rows)
    torch.cuda.synchronize()
    codes, sc = O.herm16_pack(G, rows)
    assert st.scale.shape == sc.shape
    assert np.array_equal(st.scale.cpu().numpy().view(np.uint32), sc.view(np.uint32))
    assert np.array_equal(_codes(st.G), codes)


@pytest.mark.parametrize("fmt", ["c64", "sn16"])
def test_compact_band_bitexact(ssb, fmt):
    n, nbf = 128, 45  # 45: a ragged last group of 16 BF pixels
    G = _seeded_G(7, nbf, n)
    g = C.Geometry(n=n, det_y=8, det_x=8, scan_step_A=C.SCAN_STEP_A, det_pitch_invA=0.2,
                   wavelength_A=C.WAVELENGTH_300KV_A, semiangle_rad=C.SEMIANGLE_RAD, det_center_y=4, det_center_x=4)
    band = O.band_indices(g, 0.2, 0.9)
    assert 0 < len(band) and len(band) % 256
    if fmt == "c64":
        src, want = ssb.GStore(_dev(G)), O.band_compact(G, band)
    else:
        codes, sc = O.herm16_pack(G, 1)
        words = codes.view(np.int32).reshape(codes.shape[:3])
        src = ssb.GStore(_dev(words), ssb.G_SN16, _dev(sc), 1)
        want = O.band_compact(words, band)
    dst = ssb.compact_band(src, g, _dev(band))
    torch.cuda.synchronize()
    assert dst.band_compact and dst.G.shape == (nbf, len(band))
    assert np.array_equal(dst.G.cpu().numpy(), want)


@pytest.fixture(scope="module")
def small(ssb, small_dataset):
    d = small_dataset
    g, ab = d["geom"], d["ab"]
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    G = ssb.build_G(_frames_dev(d["frames"]), g, _dev(bf))
    Gor = O.build_G(d["frames"], bf)
    band = O.band_indices(g, 0.2, 0.9)
    return d, bf, G, Gor, band


@pytest.mark.parametrize("per_row", [False, True])
def test_reconstruct_herm16_matches_oracle(ssb, small, per_row):
    """CUDA build -> herm16 -> reconstruction against the oracle's G rounded
    to float32 -> herm16 -> dequantised -> reduction -> phase."""
    d, bf, G, Gor, _ = small
    g, ab = d["geom"], d["ab"]
    n = g.n
    rows = 1 if per_row else n
    st = ssb.compact_G16(G, g, rows)
    Od, Nd, ph = ssb.reconstruct_g(st, g, _dev(bf), ab)
    torch.cuda.synchronize()
    # the encoding's closed-form bound, CUDA codes against the CUDA G:
    # half a code step plus the float32 roundings, per component
    Gc = G.cpu().numpy()
    cc = _codes(st.G).astype(np.float64)
    s_full = np.repeat(st.scale.cpu().numpy().T.astype(np.float64), rows, axis=1)[:, :, None]
    bound = s_full * ((0.5 + 2.0 ** -10) / 32767 + 2.0 ** -22)
    assert np.all(np.abs(np.maximum(cc[..., 0] / 32767, -1) * s_full - Gc.real) <= bound)
    assert np.all(np.abs(np.maximum(cc[..., 1] / 32767, -1) * s_full - Gc.imag) <= bound)
    codes, sc = O.herm16_pack(Gor.astype(np.complex64), rows)
    assert rel(st.scale.cpu().numpy(), sc) < 1e-5
    Gq = O.herm16_unpack(codes, sc, rows)
    Oref, Nref = O.reduce(Gq, g, ab, bf)
    phref = O.phase_image(Oref, Nref, O.g0_mean(Gq), n)
    assert np.array_equal(Nd.cpu().numpy().ravel(), Nref)
    assert rel(Od.cpu().numpy().ravel(), Oref) < TOL
    assert rel(ph.cpu().numpy(), phref) < TOL


def test_reconstruct_g_c64_is_reconstruct(ssb, small):
    d, bf, G, _, _ = small
    bfd = _dev(bf)
    a = ssb.reconstruct(G, d["geom"], bfd, d["ab"])
    b = ssb.reconstruct_g(ssb.GStore(G), d["geom"], bfd, d["ab"])
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("B", [1, 8])
def test_band_copy_scores_like_half_plane(ssb, small, B):
    """complex64 band copy: bit for bit the half-plane pass (same arithmetic,
    other addresses); herm16 band copy: bit for bit the herm16 half plane."""
    d, bf, G, _, band = small
    g = d["geom"]
    bfd, bd = _dev(bf), _dev(band)
    sets = C.perturbed_sets(d["ab"], 8, seed=4)[:B]
    ref = ssb.score_batch(G, g, bfd, sets, bd)
    got = ssb.score_batch_g(ssb.compact_band(G, g, bd), g, bfd, sets, bd)
    for x, y in zip(ref, got):
        assert torch.equal(x, y)
    h16 = ssb.compact_G16(G, g, 1)
    ref16 = ssb.score_batch_g(h16, g, bfd, sets, bd)
    got16 = ssb.score_batch_g(ssb.compact_band(h16, g, bd), g, bfd, sets, bd)
    for x, y in zip(ref16, got16):
        assert torch.equal(x, y)


@pytest.mark.parametrize("per_row", [False, True])
def test_score_herm16_band_matches_oracle(ssb, small, per_row):
    d, bf, G, Gor, band = small
    g = d["geom"]
    rows = 1 if per_row else g.n
    sets = C.perturbed_sets(d["ab"], 8, seed=4)
    st = ssb.compact_band(ssb.compact_G16(G, g, rows), g, _dev(band))
    Ob, Nb, scb = ssb.score_batch_g(st, g, _dev(bf), sets, _dev(band))
    torch.cuda.synchronize()
    codes, sc = O.herm16_pack(Gor.astype(np.complex64), rows)
    Gq = O.herm16_unpack(codes, sc, rows)
    for s, ab in enumerate(sets):
        Oref, Nref = O.reduce(Gq, g, ab, bf, entries=band)
        assert np.array_equal(Nb[s].cpu().numpy(), Nref)
        assert rel(Ob[s].cpu().numpy(), Oref) < TOL
        ref = O.score(Oref, Nref)
        assert abs(scb[s].item() - ref) <= TOL * abs(ref)
