"""Pins of the CPU oracle against things other than itself.

Each test fixes a part of the oracle by an independent route: a brute-force
DFT, exact integer sums, a symmetry the mathematics guarantees, a closed-form
weak-phase object, textbook special cases of the aberration function, values
the pages print, or brute force over tiny inputs.  A plausible slip anywhere
in the oracle (a dropped term, a wrong sign or index, a transposed operand)
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import ssb_oracle as O
from synth import configs as C
from synth import forward as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _geom(n=32, det=24, dk=0.19, step=C.SCAN_STEP_A):
    return C.Geometry(n=n, det_y=det, det_x=det, scan_step_A=step, det_pitch_invA=dk,
                      wavelength_A=C.WAVELENGTH_300KV_A, semiangle_rad=C.SEMIANGLE_RAD,
                      det_center_y=det // 2, det_center_x=det // 2)


# ----------------------------------------------------------------------------
# G(q, k)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n", [8, 32])
def test_G_matches_bruteforce_dft(n):
    """G against a direct O(n^4) DFT written as explicit sums (1e-12)."""
    rng = np.random.default_rng(10 + n)
    det = 6
    frames = rng.uniform(0, 20, size=(n, n, det, det))
    bf = np.array([0, 7, 8, 14, 21, 35])  # 6 arbitrary detector pixels
    G = O.build_G(frames, bf)
    assert G.shape == (len(bf), n, n // 2 + 1)
    ry, rx = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    for b, pix in enumerate(bf):
        x = frames[:, :, pix // det, pix % det]
        ref = np.zeros((n, n // 2 + 1), dtype=np.complex128)
        for row in range(n):
            fy = row if row < n // 2 else row - n
            for fx in range(n // 2 + 1):
                ang = -2.0 * math.pi * (fy * ry + fx * rx) / n
                ref[row, fx] = np.sum(x * (np.cos(ang) + 1j * np.sin(ang)))
        err = np.abs(G[b] - ref).max() / np.abs(ref).max()
        assert err < 1e-12


def test_G_dc_is_exact_integer_sum():
    """G(0, k) = sum_r I(r, k) exactly for uint16 counts."""
    rng = np.random.default_rng(3)
    n, det = 64, 16
    frames = rng.integers(0, 60000, size=(n, n, det, det)).astype(np.uint16)
    bf = np.arange(0, det * det, 5)
    G = O.build_G(frames, bf)
    exact = frames.reshape(n * n, det * det)[:, bf].astype(np.int64).sum(axis=0)
    assert np.array_equal(G[:, 0, 0].real, exact.astype(np.float64))
    assert np.all(G[:, 0, 0].imag == 0)


def test_G_hermitian_half_plane():
    """Full fft2 of real traces is Hermitian; the half plane is its left part."""
    rng = np.random.default_rng(4)
    n, det = 32, 8
    frames = rng.uniform(0, 5, size=(n, n, det, det))
    bf = np.arange(det * det)[::3]
    G = O.build_G(frames, bf)
    x = O.bf_traces(frames, bf)
    full = np.fft.fft2(x, axes=(-2, -1))
    neg = np.roll(np.flip(full, axis=(-2, -1)), shift=1, axis=(-2, -1))  # full(-q)
    scale = np.abs(full).max()
    assert np.abs(neg - np.conj(full)).max() < 1e-12 * scale
    assert np.abs(full[:, :, : n // 2 + 1] - G).max() < 1e-12 * scale
    # the trace layout is (scan_y, scan_x): axis 0 of a plane is y
    assert np.array_equal(x[1], frames[:, :, bf[1] // det, bf[1] % det])


# ----------------------------------------------------------------------------
# aberration function
# ----------------------------------------------------------------------------

def _ab(**kw):
    return C.Aberrations(**kw)


LAM = C.WAVELENGTH_300KV_A


def test_chi_textbook_defocus_and_spherical():
    """Pure C10: chi = pi lambda C10 |v|^2; pure C30: chi = pi/2 C30 lambda^3 |v|^4."""
    rng = np.random.default_rng(0)
    vx, vy = rng.normal(0, 1.0, 50), rng.normal(0, 1.0, 50)
    k2 = vx * vx + vy * vy
    np.testing.assert_allclose(O.chi(vx, vy, _ab(C10=123.0), LAM),
                               math.pi * LAM * 123.0 * k2, rtol=1e-13)
    np.testing.assert_allclose(O.chi(vx, vy, _ab(C30=-7.5e3), LAM),
                               0.5 * math.pi * (-7.5e3) * LAM ** 3 * k2 * k2, rtol=1e-13)


def test_chi_axis_values():
    """At phi = 0, pi/2 and pi/4 every a/b term reduces to a known sign."""
    names = C.ABERRATION_NAMES
    rng = np.random.default_rng(1)
    vals = dict(zip(names, rng.uniform(-100, 100, len(names))))
    ab = _ab(**vals)
    v = 1.3
    t = LAM * v
    pre = 2 * math.pi / LAM
    x_axis = pre * (t ** 2 / 2 * (vals["C10"] + vals["C12a"])
                    + t ** 3 / 3 * (vals["C21a"] + vals["C23a"])
                    + t ** 4 / 4 * (vals["C30"] + vals["C32a"] + vals["C34a"]))
    y_axis = pre * (t ** 2 / 2 * (vals["C10"] - vals["C12a"])
                    + t ** 3 / 3 * (vals["C21b"] - vals["C23b"])
                    + t ** 4 / 4 * (vals["C30"] - vals["C32a"] + vals["C34a"]))
    r = math.sqrt(0.5)
    diag = pre * (t ** 2 / 2 * (vals["C10"] + vals["C12b"])
                  + t ** 3 / 3 * (r * vals["C21a"] + r * vals["C21b"] - r * vals["C23a"] + r * vals["C23b"])
                  + t ** 4 / 4 * (vals["C30"] + vals["C32b"] - vals["C34a"]))
    assert O.chi(v, 0.0, ab, LAM) == pytest.approx(x_axis, rel=1e-12)
    assert O.chi(0.0, v, ab, LAM) == pytest.approx(y_axis, rel=1e-12)
    assert O.chi(v * r, v * r, ab, LAM) == pytest.approx(diag, rel=1e-12)


@pytest.mark.parametrize("name,fold", [("C12a", 2), ("C12b", 2), ("C23a", 3), ("C23b", 3),
                                       ("C34a", 4), ("C34b", 4), ("C21a", 1), ("C32b", 2)])
def test_chi_rotational_order(name, fold):
    """An m-fold term is invariant under rotation by 2 pi / m and (m > 1) changes
    sign under rotation by pi / m."""
    ab = _ab(**{name: 37.0})
    rng = np.random.default_rng(2)
    vx, vy = rng.normal(0, 1, 20), rng.normal(0, 1, 20)

    def rot(a):
        return vx * math.cos(a) - vy * math.sin(a), vx * math.sin(a) + vy * math.cos(a)

    base = O.chi(vx, vy, ab, LAM)
    np.testing.assert_allclose(O.chi(*rot(2 * math.pi / fold), ab, LAM), base, rtol=1e-10, atol=1e-14)
    if fold > 1:
        np.testing.assert_allclose(O.chi(*rot(math.pi / fold), ab, LAM), -base, rtol=1e-10, atol=1e-14)


def test_chi_matches_independent_complex_power_form():
    """The generator's complex-power evaluation of the same polynomial agrees."""
    rng = np.random.default_rng(5)
    vals = {k: float(v) for k, v in zip(C.ABERRATION_NAMES, rng.uniform(-5e3, 5e3, 12))}
    ab = _ab(**vals)
    vx, vy = rng.normal(0, 1.5, 100), rng.normal(0, 1.5, 100)
    np.testing.assert_allclose(O.chi(vx, vy, ab, LAM), F.probe_phase(vx, vy, ab, LAM), rtol=1e-11)


# ----------------------------------------------------------------------------
# trotter sets and weights
# ----------------------------------------------------------------------------

def _aperture_scalar(px, py, tx, ty, r2):
    f = np.float32
    dx = f(f(px) - f(tx))
    dy = f(f(py) - f(ty))
    return f(f(dx * dx) + f(dy * dy)) <= f(r2)


def test_trotters_bruteforce():
    """Double loop over (q, k) with scalar float32 ops matches the vectorised sets."""
    g = C.geometry(C.WORKLOADS["tiny"])
    ab = _ab(C10=10.0, tilt_x_rad=2e-3, tilt_y_rad=-1e-3)
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    qx_col, qy_row = O.q_coords(g)
    entries = np.arange(0, g.n * (g.n // 2 + 1), 7)
    h = g.n // 2 + 1
    qx, qy = qx_col[entries % h], qy_row[entries // h]
    tm, tp = O.trotters(g, ab, bf, qx, qy)
    tx, ty = np.float32(ab.tilt_x_rad / g.wavelength_A), np.float32(ab.tilt_y_rad / g.wavelength_A)
    r = g.semiangle_rad / g.wavelength_A
    r2 = np.float32(r * r)
    for a, (x, y) in enumerate(zip(qx, qy)):
        for b, pix in enumerate(bf):
            i, j = divmod(int(pix), g.det_x)
            kx = np.float32((j - g.det_center_x) * g.det_pitch_invA)
            ky = np.float32((i - g.det_center_y) * g.det_pitch_invA)
            qxf, qyf = np.float32(x), np.float32(y)
            aa = _aperture_scalar(kx, ky, tx, ty, r2)
            m = _aperture_scalar(np.float32(kx - qxf), np.float32(ky - qyf), tx, ty, r2)
            p = _aperture_scalar(np.float32(kx + qxf), np.float32(ky + qyf), tx, ty, r2)
            assert tm[a, b] == (aa and m and not p)
            assert tp[a, b] == (aa and p and not m)


def test_bf_set_bruteforce():
    g = C.geometry(C.WORKLOADS["small"])
    ab = C.aberrations(C.WORKLOADS["small"])
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    ref = []
    r = g.semiangle_rad / g.wavelength_A
    for i in range(g.det_y):
        for j in range(g.det_x):
            ex = (j - g.det_center_x) * g.det_pitch_invA - ab.tilt_x_rad / g.wavelength_A
            ey = (i - g.det_center_y) * g.det_pitch_invA - ab.tilt_y_rad / g.wavelength_A
            if ex * ex + ey * ey <= r * r:
                ref.append(i * g.det_x + j)
    assert np.array_equal(bf, np.array(ref, dtype=np.int32))


def test_zero_aberration_weights_are_plus_minus_one_and_O_antihermitian():
    """No aberrations: w = +1 on T-, -1 on T+ (plain SSB difference of the two
    sidebands), and O(-q) = -conj O(q) on a full-plane evaluation."""
    d = F.make_numpy_dataset("tiny")
    g, frames = d["geom"], d["frames"]
    ab = _ab()
    bf = O.bf_indices(g)
    n = g.n
    dq = 1.0 / (n * g.scan_step_A)
    rng = np.random.default_rng(6)
    fys = rng.integers(-n // 2 + 1, n // 2, 12)
    fxs = rng.integers(1, n // 2, 12)
    qx, qy = fxs * dq, fys * dq
    tm, tp = O.trotters(g, ab, bf, qx, qy)
    w = O.weights(g, ab, bf, qx, qy, tm, tp)
    assert np.all(w[tm] == 1.0) and np.all(w[tp] == -1.0)
    assert np.all(w[~(tm | tp)] == 0.0)
    full = np.fft.fft2(O.bf_traces(frames, bf), axes=(-2, -1))    # (N_bf, n, n)
    for sgn_case in range(len(qx)):
        vals = []
        for s in (1, -1):
            fy, fx = s * fys[sgn_case], s * fxs[sgn_case]
            tm1, tp1 = O.trotters(g, ab, bf, [fx * dq], [fy * dq])
            w1 = O.weights(g, ab, bf, [fx * dq], [fy * dq], tm1, tp1)[0]
            vals.append(np.sum(full[:, fy % n, fx % n] * w1))
        assert abs(vals[1] + np.conj(vals[0])) <= 1e-9 * max(1.0, abs(vals[0]))


# ----------------------------------------------------------------------------
# closed-form weak-phase object: fixes the signs of w and T+/-
# ----------------------------------------------------------------------------

def _linear_intensity_single_cosine(g, ab, bf, eps, fy0, fx0):
    """I = |A(k)|^2 + eps Re[i A~*(k) (A~(k-q0) e^{2pi i q0.r} + A~(k+q0) e^{-2pi i q0.r})],
    A~(k) = A(k - k_t) exp(-i chi(k - k_t)), for phi(r) = eps cos(2 pi q0.r)."""
    n = g.n
    lam = g.wavelength_A
    dq = 1.0 / (n * g.scan_step_A)
    q0x, q0y = fx0 * dq, fy0 * dq
    ktx, kty = ab.tilt_x_rad / lam, ab.tilt_y_rad / lam
    kmax2 = (g.semiangle_rad / lam) ** 2

    def atilde(kx, ky):
        vx, vy = kx - ktx, ky - kty
        a = (vx * vx + vy * vy) <= kmax2
        return np.where(a, np.exp(-1j * F.probe_phase(vx, vy, ab, lam)), 0.0)

    i = np.arange(g.det_y)[:, None]
    j = np.arange(g.det_x)[None, :]
    kx = (j - g.det_center_x) * g.det_pitch_invA + 0 * i
    ky = (i - g.det_center_y) * g.det_pitch_invA + 0 * j
    a0 = atilde(kx, ky)
    am = atilde(kx - q0x, ky - q0y)
    ap = atilde(kx + q0x, ky + q0y)
    ry, rx = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    ph = np.exp(2j * math.pi * (fy0 * ry + fx0 * rx) / n)[:, :, None, None]
    inten = (np.abs(a0) ** 2)[None, None] + eps * np.real(
        1j * np.conj(a0)[None, None] * (am[None, None] * ph + ap[None, None] * np.conj(ph)))
    return inten, (kx, ky, q0x, q0y, kmax2, ktx, kty)


@pytest.mark.parametrize("fy0,fx0", [(-3, 5), (4, 0), (2, 9)])
def test_single_cosine_object_closed_form(fy0, fx0):
    """G vanishes off {0, +-q0}; O(q0) = N(q0) * i eps/2 * n^2 exactly."""
    g = _geom(n=32, det=28, dk=0.17)
    ab = _ab(C10=-80.0, C12a=20.0, C12b=-15.0, C21a=30.0, C23b=-25.0, C30=5e3,
             C32a=-2e3, C34b=3e3, tilt_x_rad=3e-3, tilt_y_rad=-1.5e-3)
    eps = 1e-3
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    inten, (kx, ky, q0x, q0y, kmax2, ktx, kty) = _linear_intensity_single_cosine(g, ab, bf, eps, fy0, fx0)
    # precondition: no aperture test lies within 1e-5 of its edge, so the float64
    # generator and the float32 trotter contract classify every pixel alike
    for sx, sy in ((0, 0), (-q0x, -q0y), (q0x, q0y)):
        d2 = (kx + sx - ktx) ** 2 + (ky + sy - kty) ** 2
        assert np.min(np.abs(d2 - kmax2)) > 1e-5 * kmax2
    G = O.build_G(inten, bf)
    n, h = g.n, g.n // 2 + 1
    scale = np.abs(G).max()
    mask = np.ones((n, h), dtype=bool)
    mask[0, 0] = False
    mask[fy0 % n, fx0] = False
    if fx0 == 0:
        mask[(-fy0) % n, 0] = False
    assert np.abs(G[:, mask]).max() < 1e-12 * scale
    e = np.array([(fy0 % n) * h + fx0])
    Oq, Nq = O.reduce(G, g, ab, bf, entries=e)
    assert Nq[0] > 0
    expect = Nq[0] * 1j * eps / 2 * n * n
    assert abs(Oq[0] - expect) < 1e-10 * abs(expect)
    # a mismatched set dephases the terms: |O| drops (triangle inequality)
    O2, N2 = O.reduce(G, g, ab.replace(C10=ab.C10 + 40.0), bf, entries=e)
    assert N2[0] == Nq[0] and abs(O2[0]) < abs(Oq[0]) * (1 - 1e-6)
    # and the score of the matched set is the larger one
    assert O.score(Oq, Nq) > O.score(O2, N2)


def _trotter_count_scalar(g, ab, bf, fy, fx):
    """|T-(q)| + |T+(q)| by a loop over BF pixels with scalar float32 aperture
    tests (independent of the oracle's vectorised trotters)."""
    dq = 1.0 / (g.n * g.scan_step_A)
    tx, ty = np.float32(ab.tilt_x_rad / g.wavelength_A), np.float32(ab.tilt_y_rad / g.wavelength_A)
    r = g.semiangle_rad / g.wavelength_A
    r2 = np.float32(r * r)
    qxf, qyf = np.float32(fx * dq), np.float32(fy * dq)
    cnt = 0
    for pix in bf:
        i, j = divmod(int(pix), g.det_x)
        kx = np.float32((j - g.det_center_x) * g.det_pitch_invA)
        ky = np.float32((i - g.det_center_y) * g.det_pitch_invA)
        a = _aperture_scalar(kx, ky, tx, ty, r2)
        m = _aperture_scalar(np.float32(kx - qxf), np.float32(ky - qyf), tx, ty, r2)
        p = _aperture_scalar(np.float32(kx + qxf), np.float32(ky + qyf), tx, ty, r2)
        cnt += int(a and (m != p))
    return cnt


@pytest.mark.parametrize("fy0,fx0", [(-3, 5), (4, 0), (2, 9)])
def test_score_single_cosine_closed_form(fy0, fx0):
    """Score over the 0.2-0.9 1/A band of the single-cosine object, in closed
    form: O vanishes on the band except at the stored copies of +-q0, where
    O = N(q) i eps/2 n^2, so score = (eps/2 n^2)^2 sum_{q0 copies} N(q)^2 /
    sum_band N(q), with every N counted by the scalar brute force.  A wrong
    denominator (band length, BF count) or a dropped square fails it."""
    g = _geom(n=32, det=28, dk=0.17)
    ab = _ab(C10=-80.0, C12a=20.0, C12b=-15.0, C21a=30.0, C23b=-25.0, C30=5e3,
             C32a=-2e3, C34b=3e3, tilt_x_rad=3e-3, tilt_y_rad=-1.5e-3)
    eps = 1e-3
    n, h = g.n, g.n // 2 + 1
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    inten, _ = _linear_intensity_single_cosine(g, ab, bf, eps, fy0, fx0)
    G = O.build_G(inten, bf)
    band = O.band_indices(g, 0.2, 0.9)
    rows, cols = band // h, band % h
    fys = np.where(rows < n // 2, rows, rows - n)
    # the stored copies of q0: (fy0, fx0), and (-fy0, 0) as well on the fx = 0 column
    copies = {(fy0, fx0)} | ({(-fy0, 0)} if fx0 == 0 else set())
    assert all(any(fy == c[0] and fx == c[1] for fy, fx in zip(fys, cols)) for c in copies)
    Nb = np.array([_trotter_count_scalar(g, ab, bf, fy, fx) for fy, fx in zip(fys, cols)])
    num = (eps / 2 * n * n) ** 2 * sum(
        int(Nb[np.flatnonzero((fys == c[0]) & (cols == c[1]))[0]]) ** 2 for c in copies)
    expect = num / float(Nb.sum())
    Ob, Nq = O.reduce(G, g, ab, bf, entries=band)
    assert np.array_equal(Nq, Nb)
    assert abs(O.score(Ob, Nq) - expect) <= 1e-10 * expect
    # the band length differs from the trotter count, so a denominator mix-up shows
    assert len(band) != Nb.sum()


def test_phase_image_single_cosine_closed_form():
    """From O = N i (eps/2) n^2 at one q0 and a = 1, the image is
    atan2(eps cos(2 pi q0.r), 1) exactly (C2R normalisation, -i, DC)."""
    n = 16
    h = n // 2 + 1
    eps = 0.05
    for fy0, fx0 in ((3, 2), (5, 0), (-2, 7)):
        Oh = np.zeros((n, h), dtype=np.complex128)
        Nh = np.zeros((n, h), dtype=np.int64)
        Nh[:] = 3
        Oh[fy0 % n, fx0] = 3 * 1j * eps / 2 * n * n
        if fx0 == 0:
            Oh[(-fy0) % n, 0] = 3 * 1j * eps / 2 * n * n
        ph = O.phase_image(Oh, Nh, n * n, n)
        ry, rx = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
        ref = np.arctan2(eps * np.cos(2 * math.pi * (fy0 * ry + fx0 * rx) / n), 1.0)
        assert np.abs(ph - ref).max() < 1e-14


def test_phase_image_drops_nyquist_and_dc():
    n = 8
    h = n // 2 + 1
    Oh = np.zeros((n, h), dtype=np.complex128)
    Nh = np.ones((n, h), dtype=np.int64)
    Oh[n // 2, 1] = 5.0
    Oh[1, n // 2] = 7.0
    Oh[0, 0] = 11.0
    ph = O.phase_image(Oh, Nh, 2.0 * n * n, n)
    assert np.all(ph == 0.0)


# ----------------------------------------------------------------------------
# end to end on the full non-linear forward model
# ----------------------------------------------------------------------------

def test_pearson_recovery_tiny(tiny_dataset):
    """Noiseless, matched aberrations: Pearson r(phase, truth) > 0.95.  The
    plain BF-mean normalisation (object fast path) is reported, and is lower."""
    d = tiny_dataset
    r = O.reconstruct(d["frames"], d["geom"], d["ab"])
    rt = np.corrcoef(r["phase"].ravel(), d["truth"].ravel())[0, 1]
    rb = O.reconstruct(d["frames"], d["geom"], d["ab"], norm="bf_mean")
    rbm = np.corrcoef(rb["phase"].ravel(), d["truth"].ravel())[0, 1]
    assert rt > 0.95
    assert rbm < rt


def test_pearson_recovery_small_noisy(small_dataset):
    """Small workload (random aberrations + tilt, Poisson 5 counts): the matched
    reconstruction still tracks the truth clearly."""
    d = small_dataset
    r = O.reconstruct(d["frames"], d["geom"], d["ab"])
    rt = np.corrcoef(r["phase"].ravel(), d["truth"].ravel())[0, 1]
    assert rt > 0.6


# ----------------------------------------------------------------------------
# values printed on the pages
# ----------------------------------------------------------------------------

def test_golden_band_count_and_sizes():
    with open(os.path.join(GOLDEN, "pages_values.json")) as fh:
        gold = json.load(fh)
    b = gold["band_count"]
    g = _geom(n=b["n"], step=b["scan_step_A"])
    band = O.band_indices(g, b["qmin"], b["qmax"])
    assert len(band) == b["count"]
    # the bytes of G one pass reads over that band
    pb = gold["band_pass_bytes"]
    assert round(b["count"] * pb["n_bf"] * 8 / 1e9, 1) == pb["GB"]
    for row in gold["g_memory"]:
        got = {"exact": C.g_bytes, "nxn": C.full_plane_bytes,
               "herm16": C.herm16_bytes}[row["mode"]](row["n_bf"], row["n"])
        assert round(got / row["unit"], row["digits"]) == row["value"], row


def test_band_membership_integer_rule():
    g = C.geometry(C.WORKLOADS["small"])
    band = O.band_indices(g)
    n, h = g.n, g.n // 2 + 1
    dq = 1.0 / (n * g.scan_step_A)
    fy, fx = O.scan_freq_index(n)
    q = np.hypot(fy[band // h] * dq, fx[band % h] * dq)
    assert q.min() >= 0.2 - 1e-12 and q.max() <= 0.9 + 1e-12
    allq = np.hypot(fy[:, None] * dq, fx[None, :] * dq).ravel()
    inside = np.flatnonzero((allq > 0.2 + 1e-9) & (allq < 0.9 - 1e-9))
    assert set(inside).issubset(set(band))


# ----------------------------------------------------------------------------
# per-BF phase moments (the exact mean(angle) path)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("fy0,fx0", [(-3, 5), (4, 0)])
def test_phase_moments_single_cosine_closed_form(fy0, fx0):
    """Linear intensities of phi = eps cos(2 pi q0.r): S_k(q0) = i eps/2 n^2
    on every trotter pixel of q0 and 0 on the others, a_k = 1, so phase_k =
    atan(eps cos) on a fraction f = N(q0) / N_bf of the pixels and 0 on the
    rest: mean = f atan(eps cos), variance = f (1 - f) atan(eps cos)^2."""
    g = _geom(n=32, det=28, dk=0.17)
    ab = _ab(C10=-80.0, C12a=20.0, C12b=-15.0, C21a=30.0, C23b=-25.0, C30=5e3,
             C32a=-2e3, C34b=3e3, tilt_x_rad=3e-3, tilt_y_rad=-1.5e-3)
    eps = 0.05
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    inten, _ = _linear_intensity_single_cosine(g, ab, bf, eps, fy0, fx0)
    G = O.build_G(inten, bf)
    n, h = g.n, g.n // 2 + 1
    _, Nq = O.reduce(G, g, ab, bf, entries=np.array([(fy0 % n) * h + fx0]))
    f = Nq[0] / len(bf)
    assert 0 < f < 1
    mean, var = O.phase_moments(G, g, ab, bf)
    ry, rx = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    t = np.arctan(eps * np.cos(2 * math.pi * (fy0 * ry + fx0 * rx) / n))
    assert np.abs(mean - f * t).max() < 1e-12
    assert np.abs(var - f * (1 - f) * t * t).max() < 1e-12


def test_per_bf_image_matches_bruteforce_inverse_dft():
    """b_k against an explicit inverse DFT over the full plane, the other half
    filled by S(-q) = -conj S(q) (anti-Hermitian corrected spectrum)."""
    rng = np.random.default_rng(21)
    n, det = 8, 10
    g = _geom(n=n, det=det, dk=0.45)
    ab = _ab(C10=-30.0, C12a=8.0, C21b=20.0, C30=4e3, tilt_x_rad=2e-3)
    frames = rng.uniform(0, 30, size=(n, n, det, det))
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)[:6]
    G = O.build_G(frames, bf)
    S = O.corrected_planes(G, g, ab, bf)
    h = n // 2 + 1
    ry, rx = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    for k, (a, b) in enumerate(O.per_bf_images(G, g, ab, bf)):
        assert a == G[k, 0, 0].real / (n * n)
        ref = np.zeros((n, n))
        for fy in range(-n // 2, n // 2):
            for fx in range(-n // 2, n // 2):
                if fy == -n // 2 or fx == -n // 2 or (fy == 0 and fx == 0):
                    continue  # Nyquist row and column, DC: zeroed
                if fx >= 0:
                    s = S[k, fy % n, fx]
                else:
                    s = -np.conj(S[k, (-fy) % n, -fx])
                ref += np.real(-1j * s * np.exp(2j * math.pi * (fy * ry + fx * rx) / n))
        ref /= n * n
        assert np.abs(b - ref).max() < 1e-12 * max(1.0, np.abs(ref).max())


def test_per_bf_mean_of_objects_is_the_fast_path():
    """The pages' identity mean_k ifft2(corrected_k) = ifft2(mean_k corrected_k):
    atan2(mean b_k, mean a_k) equals the single image with the BF-mean
    normalisation (O / N_bf), an independent route through the reduction."""
    rng = np.random.default_rng(22)
    n, det = 16, 14
    g = _geom(n=n, det=det, dk=0.3)
    ab = _ab(C10=-50.0, C12b=10.0, C23a=15.0, C30=2e3, tilt_y_rad=1e-3)
    frames = rng.uniform(0, 30, size=(n, n, det, det))
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    G = O.build_G(frames, bf)
    sa, sb = 0.0, np.zeros((n, n))
    for a, b in O.per_bf_images(G, g, ab, bf):
        sa += a
        sb += b
    Oq, Nq = O.reduce(G, g, ab, bf)
    fast = O.phase_image(Oq, Nq, O.g0_mean(G), n, norm="bf_mean", n_bf=len(bf))
    assert np.abs(np.arctan2(sb / len(bf), sa / len(bf)) - fast).max() < 1e-12


def test_phase_moments_of_one_pixel():
    rng = np.random.default_rng(23)
    n, det = 16, 12
    g = _geom(n=n, det=det, dk=0.3)
    ab = _ab(C10=-20.0, C30=1e3)
    frames = rng.uniform(0, 30, size=(n, n, det, det))
    bf = O.bf_indices(g)[5:6]
    G = O.build_G(frames, bf)
    mean, var = O.phase_moments(G, g, ab, bf)
    (a, b), = list(O.per_bf_images(G, g, ab, bf))
    assert np.array_equal(mean, np.arctan2(b, a))
    assert var.max() < 1e-15
