"""GPU parity of the depth-spread ("thick") fit: ssb_score_batch_depth called
through the C ABI against the oracle's reduce_depth on the same seeded data.

Bars: N bit-exact; O within relative L2 1e-4 and the score within 1e-4 per
set; depth 0 gives the depth-0 scoring bit for bit; a set's result does not
depend on the batch it runs in (bit for bit)."""
import numpy as np
import pytest

from oracle import ssb_oracle as O
from synth import configs as C

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TOL = 1e-4
DEPTHS = [136.0, 0.0, 400.0, 40.0, 250.0, 136.0, 800.0, 10.0]


def rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


@pytest.fixture(scope="module")
def ssb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as ge
    ge.build()
    import electron_microscopy_gb300 as m
    return m


@pytest.fixture(scope="module")
def small(ssb, small_dataset):
    d = small_dataset
    g, ab = d["geom"], d["ab"]
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    fr = d["frames"]
    G = ssb.build_G(torch.from_numpy(fr.view(np.int16)).cuda(), g, torch.from_numpy(bf).cuda())
    band = O.band_indices(g, 0.2, 0.9)
    return d, bf, G, band, O.build_G(fr, bf)


@pytest.mark.parametrize("B", [2, 8])
def test_shared_depth_matches_oracle_and_single_sets(ssb, small, B):
    """Every set at the same spread (136 A, the pages' fit depth): the factor is
    taken once per (q, k) for all sets.  Each set matches the oracle and equals
    the same set scored alone, bit for bit."""
    d, bf, G, band, Gor = small
    g = d["geom"]
    bfd, bd = torch.from_numpy(bf).cuda(), torch.from_numpy(band).cuda()
    sets = C.perturbed_sets(d["ab"], B, seed=90 + B)
    Ob, Nb, sc = ssb.score_batch_depth(G, g, bfd, sets, [136.0] * B, bd)
    torch.cuda.synchronize()
    for s, ab in enumerate(sets):
        Oref, Nref = O.reduce_depth(Gor, g, ab, bf, 136.0, entries=band)
        assert np.array_equal(Nb[s].cpu().numpy(), Nref), s
        assert rel(Ob[s].cpu().numpy(), Oref) < TOL, s
        O1, N1, s1 = ssb.score_batch_depth(G, g, bfd, [ab], [136.0], bd)
        assert torch.equal(O1[0], Ob[s]) and torch.equal(N1[0], Nb[s]) and torch.equal(s1[0], sc[s]), s


@pytest.mark.parametrize("B", [1, 3, 8])
def test_depth_scores_match_oracle(ssb, small, B):
    d, bf, G, band, Gor = small
    g = d["geom"]
    sets = C.perturbed_sets(d["ab"], B, seed=70 + B)
    depths = DEPTHS[:B]
    Ob, Nb, sc = ssb.score_batch_depth(G, g, torch.from_numpy(bf).cuda(), sets, depths,
                                       torch.from_numpy(band).cuda())
    torch.cuda.synchronize()
    for s, (ab, t) in enumerate(zip(sets, depths)):
        Oref, Nref = O.reduce_depth(Gor, g, ab, bf, t, entries=band)
        assert np.array_equal(Nb[s].cpu().numpy(), Nref), s
        assert rel(Ob[s].cpu().numpy(), Oref) < TOL, (s, t)
        ref = O.score(Oref, Nref)
        assert abs(sc[s].item() - ref) <= TOL * abs(ref), (s, t)


def test_depth_zero_is_the_plain_scoring_bit_for_bit(ssb, small):
    d, bf, G, band, _ = small
    g = d["geom"]
    sets = C.perturbed_sets(d["ab"], 8, seed=81)
    bfd, bd = torch.from_numpy(bf).cuda(), torch.from_numpy(band).cuda()
    O0, N0, s0 = ssb.score_batch(G, g, bfd, sets, bd)
    Od, Nd, sd = ssb.score_batch_depth(G, g, bfd, sets, [0.0] * 8, bd)
    # one set with a spread sends the batch through the depth kernel; the
    # sets with t = 0 still give the plain results bit for bit
    dep = [0.0] * 7 + [300.0]
    Om, Nm, sm = ssb.score_batch_depth(G, g, bfd, sets, dep, bd)
    torch.cuda.synchronize()
    assert torch.equal(O0, Od) and torch.equal(N0, Nd) and torch.equal(s0, sd)
    assert torch.equal(O0[:7], Om[:7]) and torch.equal(N0, Nm) and torch.equal(s0[:7], sm[:7])
    assert not torch.equal(O0[7], Om[7])


def test_depth_B_invariance(ssb, small):
    d, bf, G, band, _ = small
    g = d["geom"]
    sets = C.perturbed_sets(d["ab"], 8, seed=82)
    bfd, bd = torch.from_numpy(bf).cuda(), torch.from_numpy(band).cuda()
    O8, N8, s8 = ssb.score_batch_depth(G, g, bfd, sets, DEPTHS, bd)
    for B in (2, 5):
        OB, NB, sB = ssb.score_batch_depth(G, g, bfd, sets[:B], DEPTHS[:B], bd)
        assert torch.equal(OB, O8[:B]) and torch.equal(NB, N8[:B]) and torch.equal(sB, s8[:B])
    for s in range(8):
        O1, N1, s1 = ssb.score_batch_depth(G, g, bfd, [sets[s]], [DEPTHS[s]], bd)
        assert torch.equal(O1[0], O8[s]) and torch.equal(s1[0], s8[s])


def test_depth_with_per_set_tilts(ssb, small):
    """Sets with different tilts (each set's own aperture tests and D)."""
    d, bf, G, band, Gor = small
    g = d["geom"]
    base = d["ab"]
    sets = [s.replace(tilt_x_rad=base.tilt_x_rad + dx * 1e-3, tilt_y_rad=base.tilt_y_rad + dy * 1e-3)
            for s, (dx, dy) in zip(C.perturbed_sets(base, 4, seed=83),
                                   [(0.0, 0.0), (3.0, -2.0), (-1.5, 1.0), (6.0, 4.0)])]
    depths = [136.0, 300.0, 0.0, 60.0]
    Ob, Nb, sc = ssb.score_batch_depth(G, g, torch.from_numpy(bf).cuda(), sets, depths,
                                       torch.from_numpy(band).cuda())
    torch.cuda.synchronize()
    for s, (ab, t) in enumerate(zip(sets, depths)):
        Oref, Nref = O.reduce_depth(Gor, g, ab, bf, t, entries=band)
        assert np.array_equal(Nb[s].cpu().numpy(), Nref), s
        assert rel(Ob[s].cpu().numpy(), Oref) < TOL, (s, t)


def test_depth_on_herm16_band_copy(ssb, small):
    """The fit's storage: a herm16 band copy (one scale per q row), scored with
    depth against the oracle's reduction over the decoded G."""
    d, bf, G, band, Gor = small
    g = d["geom"]
    bd = torch.from_numpy(band).cuda()
    h16 = ssb.compact_G16(G, g, 1)
    bandG = ssb.compact_band(h16, g, bd)
    sets = C.perturbed_sets(d["ab"], 4, seed=84)
    depths = [136.0, 0.0, 500.0, 20.0]
    Ob, Nb, sc = ssb.score_batch_depth(bandG, g, torch.from_numpy(bf).cuda(), sets, depths, bd)
    torch.cuda.synchronize()
    codes, scl = O.herm16_pack(G.cpu().numpy(), 1)
    Gq = O.herm16_unpack(codes, scl, 1)
    for s, (ab, t) in enumerate(zip(sets, depths)):
        Oref, Nref = O.reduce_depth(Gq, g, ab, bf, t, entries=band)
        assert np.array_equal(Nb[s].cpu().numpy(), Nref), s
        assert rel(Ob[s].cpu().numpy(), Oref) < TOL, (s, t)


def test_depth_rejects_bad_spreads(ssb, small):
    d, bf, G, band, _ = small
    bd = torch.from_numpy(band).cuda()
    for bad in ([-1.0], [float("nan")], [float("inf")]):
        with pytest.raises(ssb.SSBError) as ei:
            ssb.score_batch_depth(G, d["geom"], torch.from_numpy(bf).cuda(), [d["ab"]], bad, bd)
        assert ei.value.code == ssb.SSB_INVALID_ARG
