"""Pins of the oracle's compact G storage (herm16 and the band-compacted copy).

herm16 follows "Historical WebGPU G(q,k) memory experiment", section
"Implementation" (scaleMax, then pack2x16snorm(clamp(v / scale)); readers
multiply unpack2x16snorm by the scale), with the per-q-row block scales of the
section "Scan-size sweep" as the second block shape.  The pins are
hand-derived codes, the closed-form rounding bound of the encoding, the
saturation of each block's largest entry, the relation between the two block
shapes, the page's printed storage sizes and the page's phase-error scale.
"""
import json
import os

import numpy as np
import pytest

from oracle import ssb_oracle as O
from synth import configs as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pack_one(v, scale):
    """Code of the real part of one entry in a 1-row, 1-pixel plane whose
    largest modulus is `scale` (the plane holds `scale` at another entry)."""
    G = np.zeros((1, 8, 5), dtype=np.complex64)
    G[0, 0, 0] = scale
    G[0, 0, 1] = v
    codes, sc = O.herm16_pack(G, 8)
    assert sc[0, 0] == np.float32(scale)
    return int(codes[0, 0, 1, 0])


@pytest.mark.parametrize("v,scale,code", [
    (4.0, 4.0, 32767),      # e = 1
    (-4.0, 4.0, -32767),    # e = -1: the code -32768 is never written
    (0.0, 4.0, 0),
    (1.0, 4.0, 8192),       # 32767 / 4 = 8191.75, + 0.5 -> floor 8192
    (-1.0, 4.0, -8192),     # -8191.75 + 0.5 = -8191.25 -> floor -8192
    (2.0, 4.0, 16384),      # 16383.5 + 0.5 = 16384 exactly
    (-2.0, 4.0, -16383),    # -16383.5 + 0.5 = -16383: halves round up
    (0.5, 1024.0, 16),      # 32767 / 2048 = 15.9995..., + 0.5 -> 16
    (-0.5, 1024.0, -16),    # -15.9995 + 0.5 = -15.4995 -> -16
])
def test_snorm16_hand_values(v, scale, code):
    """Codes worked out by hand from floor(0.5 + 32767 e), e = v / scale."""
    assert _pack_one(v, scale) == code


def test_unpack_of_most_negative_code_is_minus_one():
    codes = np.zeros((1, 2, 2, 2), dtype=np.int16)
    codes[0, 0, 0, 0] = -32768
    codes[0, 0, 0, 1] = -32767
    g = O.herm16_unpack(codes, np.array([[2.0]], dtype=np.float32), 2)
    assert g[0, 0, 0] == -2.0 - 2.0j


def _wide_range_G(rng, nbf=5, n=16):
    """Magnitudes spread log-uniformly over 12 decades, a DC-like peak per pixel."""
    h = n // 2 + 1
    mag = 10.0 ** rng.uniform(-6, 6, size=(nbf, n, h))
    ph = rng.uniform(-np.pi, np.pi, size=(nbf, n, h))
    G = mag * np.exp(1j * ph)
    G[:, 0, 0] = 10.0 ** rng.uniform(6, 7, size=nbf)
    return G.astype(np.complex64)


@pytest.mark.parametrize("per_row", [False, True])
def test_herm16_rounding_bound(per_row):
    """|unpack(code) scale - v| <= scale ((0.5 + 2^-10) / 32767 + 2^-22) for every
    component: half a code step plus the float32 roundings of v / scale,
    32767 e and 0.5 + 32767 e.  A wrong multiplier (32768), truncation instead
    of rounding, or a missing scale breaks it."""
    rng = np.random.default_rng(5)
    G = _wide_range_G(rng)
    nbf, n, h = G.shape
    rows = 1 if per_row else n
    codes, sc = O.herm16_pack(G, rows)
    back = O.herm16_unpack(codes, sc, rows)
    s_full = np.repeat(sc.T.astype(np.float64), rows, axis=1)[:, :, None]
    bound = s_full * ((0.5 + 2.0 ** -10) / 32767 + 2.0 ** -22)
    G64 = G.astype(np.complex128)
    assert np.all(np.abs(back.real - G64.real) <= bound)
    assert np.all(np.abs(back.imag - G64.imag) <= bound)
    # and the bound is nearly reached: the codes really are 16-bit
    worst = (np.abs(back.real - G64.real) / s_full).max()
    assert worst > 0.4 / 32767


@pytest.mark.parametrize("per_row", [False, True])
def test_herm16_block_maximum_saturates(per_row):
    """In every block the entry of largest modulus has a code modulus of
    32767 (to rounding); no code exceeds 32767 in magnitude."""
    rng = np.random.default_rng(6)
    G = _wide_range_G(rng)
    nbf, n, h = G.shape
    rows = 1 if per_row else n
    codes, sc = O.herm16_pack(G, rows)
    assert np.abs(codes.astype(np.int32)).max() <= 32767
    cm = np.hypot(codes[..., 0].astype(np.float64), codes[..., 1].astype(np.float64))
    cm = cm.reshape(nbf, n // rows, rows * h)
    gm = np.abs(G.astype(np.complex128)).reshape(nbf, n // rows, rows * h)
    at_max = np.take_along_axis(cm, gm.argmax(axis=2)[..., None], axis=2)[..., 0]
    assert np.all(np.abs(at_max - 32767) <= 1.0)
    # the scale is the largest modulus (float32 sqrt of the float32 |G|^2)
    assert np.allclose(sc.T, gm.max(axis=2), rtol=2e-7, atol=0)


def test_per_bf_scale_is_max_of_per_row_scales():
    rng = np.random.default_rng(7)
    G = _wide_range_G(rng)
    n = G.shape[1]
    _, s_bf = O.herm16_pack(G, n)
    _, s_row = O.herm16_pack(G, 1)
    assert s_bf.shape == (1, G.shape[0]) and s_row.shape == (n, G.shape[0])
    assert np.array_equal(s_bf[0], s_row.max(axis=0))


def test_empty_block_stores_zero():
    G = np.zeros((2, 8, 5), dtype=np.complex64)
    G[1, 3, 2] = 1.0 - 2.0j
    codes, sc = O.herm16_pack(G, 1)
    assert sc[:, 0].max() == 0 and np.count_nonzero(codes[0]) == 0
    assert sc[3, 1] == np.float32(np.sqrt(np.float32(5.0)))
    assert np.count_nonzero(codes[1]) == 2


def test_herm16_storage_matches_page_table():
    """Stored bytes against the page's memory planning table (4 bytes per
    half-plane entry + 4 per BF pixel), and the arrays the packer returns."""
    gold = json.load(open(os.path.join(GOLDEN, "pages_values.json")))
    for row in gold["g_memory"]:
        if row["mode"] != "herm16":
            continue
        got = O.herm16_bytes(row["n_bf"], row["n"], row["n"])
        assert round(got / row["unit"], row["digits"]) == row["value"], row
        assert got == C.herm16_bytes(row["n_bf"], row["n"])
    G = np.ones((3, 16, 9), dtype=np.complex64)
    for rows in (16, 1):
        codes, sc = O.herm16_pack(G, rows)
        assert codes.nbytes + sc.nbytes == O.herm16_bytes(3, 16, rows)


def test_band_compact_is_the_band_columns():
    rng = np.random.default_rng(8)
    G = (rng.standard_normal((4, 8, 5)) + 1j * rng.standard_normal((4, 8, 5))).astype(np.complex64)
    band = np.array([39, 0, 7, 12, 5], dtype=np.int32)
    Gb = O.band_compact(G, band)
    assert Gb.shape == (4, 5)
    for i, e in enumerate(band):
        assert np.array_equal(Gb[:, i], G[:, e // 5, e % 5])
    codes, _ = O.herm16_pack(G, 8)
    assert np.array_equal(O.band_compact(codes, band)[:, 2], codes[:, 1, 2])


@pytest.mark.slow
def test_herm16_phase_error_scale(small_dataset):
    """Phase through herm16 against the exact half plane on the 128^2 scan.
    The page reports, with one scale per BF pixel, a worst-case error of
    0.07 % of the phase span at a 128^2 scan up to 0.16 % at 512^2
    ("Historical WebGPU G(q,k) memory experiment", sections "Scan-size sweep"
    and "Raw numbers") and expects per-q-row scales to pull it down.  This
    noisier synthetic scan (5 counts per BF pixel) gives 0.12 % per pixel
    scale and 0.01 % per q row: the bounds are 2e-3 and 1e-3 of the span, and
    the per-q-row error at least 5x below the per-pixel one."""
    ds = small_dataset
    g, ab = ds["geom"], ds["ab"]
    a = O._ab(ab)
    bf = O.bf_indices(g, a[12], a[13])
    G = O.build_G(ds["frames"], bf)
    n = G.shape[1]
    O0, N0 = O.reduce(G, g, ab, bf)
    ph0 = O.phase_image(O0, N0, O.g0_mean(G), n)
    span = ph0.max() - ph0.min()
    errs = {}
    for rows in (n, 1):
        codes, sc = O.herm16_pack(G.astype(np.complex64), rows)
        Gq = O.herm16_unpack(codes, sc, rows)
        Oq, Nq = O.reduce(Gq, g, ab, bf)
        assert np.array_equal(Nq, N0)
        ph = O.phase_image(Oq, Nq, O.g0_mean(Gq), n)
        errs[rows] = np.abs(ph - ph0).max() / span
    assert errs[n] < 2e-3
    assert errs[1] < 1e-3
    assert errs[1] * 5 < errs[n]
