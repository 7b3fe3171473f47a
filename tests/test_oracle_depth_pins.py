"""Pins of the oracle's depth-spread fit weights (reduce_depth) against things
other than its own sinc formula: the depth-0 weights, Gauss-Legendre
quadrature of the forward model's chi over the defocus spread, and a
single-cosine weak-phase object whose linearised intensity is averaged over
the spread by quadrature (not by the formula under test)."""
import math

import numpy as np
import pytest

from oracle import ssb_oracle as O
from synth import configs as C
from synth import forward as F

from tests.test_oracle_pins import _geom, _linear_intensity_single_cosine  # noqa: F401

AB = C.Aberrations(C10=-80.0, C12a=20.0, C12b=-15.0, C21a=30.0, C23b=-25.0, C30=5e3,
                   C32a=-2e3, C34b=3e3, tilt_x_rad=3e-3, tilt_y_rad=-1.5e-3)


def _gauss_z(t, m=48):
    """Gauss-Legendre nodes and weights of the mean over z in [-t/2, t/2]."""
    x, w = np.polynomial.legendre.leggauss(m)
    return 0.5 * t * x, 0.5 * w


def _trotter_setup(g, ab, entries):
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    h = g.n // 2 + 1
    qx_col, qy_row = O.q_coords(g)
    qx, qy = qx_col[entries % h], qy_row[entries // h]
    tm, tp = O.trotters(g, ab, bf, qx, qy)
    return bf, qx, qy, tm, tp


def test_depth_zero_is_the_depth0_reduction():
    g = _geom(n=32, det=28, dk=0.17)
    rng = np.random.default_rng(3)
    bf = O.bf_indices(g, AB.tilt_x_rad, AB.tilt_y_rad)
    G = rng.normal(size=(len(bf), 32, 17)) + 1j * rng.normal(size=(len(bf), 32, 17))
    e = np.arange(0, 32 * 17, 5)
    O0, N0 = O.reduce(G, g, AB, bf, entries=e)
    Od, Nd = O.reduce_depth(G, g, AB, bf, 0.0, entries=e)
    assert np.array_equal(O0, Od) and np.array_equal(N0, Nd)


@pytest.mark.parametrize("t", [136.0, 400.0])
def test_factor_is_the_quadrature_mean_over_the_spread(t):
    """sinc factor = mean over z of exp(i [chi_z(k) - chi_z(k -/+ q)] - i [same at
    z = 0]) with chi_z the forward model's chi at defocus C10 + z (1e-10)."""
    g = _geom(n=32, det=28, dk=0.17)
    e = np.array([3, 40, 77, 150, 201, 333, 400, 499])
    bf, qx, qy, tm, tp = _trotter_setup(g, AB, e)
    f = O.depth_factor(g, AB, bf, qx, qy, tm, tp, t)
    lam = g.wavelength_A
    ktx, kty = AB.tilt_x_rad / lam, AB.tilt_y_rad / lam
    kx, ky = O.det_k(g, bf // g.det_x, bf % g.det_x)
    zs, ws = _gauss_z(t)
    for a in range(len(e)):
        for b in np.flatnonzero(tm[a] | tp[a])[:40]:
            s = -1.0 if tm[a, b] else 1.0
            vk = (kx[b] - ktx, ky[b] - kty)
            vo = (kx[b] + s * qx[a] - ktx, ky[b] + s * qy[a] - kty)
            d0 = F.probe_phase(*vk, AB, lam) - F.probe_phase(*vo, AB, lam)
            mean = 0j
            for z, w in zip(zs, ws):
                abz = AB.replace(C10=AB.C10 + z)
                dz = F.probe_phase(*vk, abz, lam) - F.probe_phase(*vo, abz, lam)
                mean += w * np.exp(1j * (dz - d0))
            assert abs(mean - f[a, b]) < 1e-10, (a, b, mean, f[a, b])
    assert np.all(f[~(tm | tp)] == 1.0)


@pytest.mark.parametrize("fy0,fx0", [(-3, 5), (2, 9)])
def test_single_cosine_object_over_a_defocus_spread(fy0, fx0):
    """Data: the linearised single-cosine intensity averaged over the defocus
    spread by quadrature (48 slices).  Then O(q0) = i eps/2 n^2 sum_k |m_k|^2
    with m_k the quadrature mean transfer factor of trotter pixel k (1e-9)."""
    t = 136.0
    g = _geom(n=32, det=28, dk=0.17)
    eps = 1e-3
    n, h = g.n, g.n // 2 + 1
    bf = O.bf_indices(g, AB.tilt_x_rad, AB.tilt_y_rad)
    zs, ws = _gauss_z(t)
    inten = 0.0
    for z, w in zip(zs, ws):
        Iz, _ = _linear_intensity_single_cosine(g, AB.replace(C10=AB.C10 + z), bf, eps, fy0, fx0)
        inten = inten + w * Iz
    G = O.build_G(inten, bf)
    e = np.array([(fy0 % n) * h + fx0])
    Od, Nd = O.reduce_depth(G, g, AB, bf, t, entries=e)
    # expected from the quadrature alone: the transfer factor m_k of each
    # trotter pixel, mean over z of exp(i pi lambda z D) computed numerically
    _, qx, qy, tm, tp = _trotter_setup(g, AB, e)
    lam = g.wavelength_A
    ktx, kty = AB.tilt_x_rad / lam, AB.tilt_y_rad / lam
    kx, ky = O.det_k(g, bf // g.det_x, bf % g.det_x)
    tot = 0.0
    for b in np.flatnonzero(tm[0] | tp[0]):
        s = -1.0 if tm[0, b] else 1.0
        vk = (kx[b] - ktx, ky[b] - kty)
        vo = (kx[b] + s * qx[0] - ktx, ky[b] + s * qy[0] - kty)
        d0 = F.probe_phase(*vk, AB, lam) - F.probe_phase(*vo, AB, lam)
        m = sum(w * np.exp(1j * (F.probe_phase(*vk, AB.replace(C10=AB.C10 + z), lam)
                                 - F.probe_phase(*vo, AB.replace(C10=AB.C10 + z), lam) - d0))
                for z, w in zip(zs, ws))
        tot += abs(m) ** 2
    expect = 1j * eps / 2 * n * n * tot
    assert Nd[0] == int((tm[0] | tp[0]).sum()) > 0
    assert abs(Od[0] - expect) < 1e-9 * abs(expect)
    # the spread really attenuates: weaker than the depth-0 closed form
    assert abs(Od[0]) < 0.999 * Nd[0] * eps / 2 * n * n


def test_score_with_depth_single_cosine():
    """score = sum_band |O|^2 / sum_band N with the depth weights: off q0 the
    data carry no signal, so the score is |O(q0)|^2 / sum_band N."""
    t = 136.0
    g = _geom(n=32, det=28, dk=0.17)
    eps = 1e-3
    n, h = g.n, g.n // 2 + 1
    fy0, fx0 = -3, 5
    bf = O.bf_indices(g, AB.tilt_x_rad, AB.tilt_y_rad)
    inten, _ = _linear_intensity_single_cosine(g, AB, bf, eps, fy0, fx0)
    G = O.build_G(inten, bf)
    band = O.band_indices(g, 0.2, 0.9)
    Ob, Nb = O.reduce_depth(G, g, AB, bf, t, entries=band)
    i0 = int(np.flatnonzero(band == (fy0 % n) * h + fx0)[0])
    mask = np.ones(len(band), bool)
    mask[i0] = False
    assert np.abs(Ob[mask]).max() < 1e-9 * abs(Ob[i0])
    assert abs(O.score(Ob, Nb) - abs(Ob[i0]) ** 2 / Nb.sum()) < 1e-12 * O.score(Ob, Nb)
