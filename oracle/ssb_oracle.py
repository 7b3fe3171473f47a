"""CPU float64 oracle for SSB direct ptychography (TEST INFRASTRUCTURE).

This module is the slow, obviously-correct statement of what the CUDA library
computes.  Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import it; the product path never does.  It shares no code
with the CUDA library (no kernels, headers, tables or helpers).

Sources (quantem.gpu pages):
* "Historical WebGPU G(q,k) memory experiment", sections "Why herm is exactly
  lossless" and "Implementation": G(q,k) is the scan-space FFT of each
  bright-field pixel's real intensity trace, stored as the Hermitian half plane
  (n, n/2+1).
* same page, "Object-redraw fast path": the object estimate is the inverse 2D
  FFT of the aberration-corrected G summed over bright-field pixels, and the
  phase image is its angle (angle of the mean object).
* "Tilt-corrected SSB on CUDA", sections "Changes" / "Where the time went": per
  (k, q, set) the kernel evaluates chi, the aperture (trotter) tests and a
  sincos; alpha^2 (1, cos 2phi, sin 2phi) = lambda^2 (|v|^2, dx^2-dy^2, 2dxdy);
  and "Open": the corrected spectrum of a real image is anti-Hermitian except
  at DC, so the image comes from a half-plane complex-to-real transform.
* "Where the 9 s of regularized preparation goes", "Setup": 512^2 scan, 192^2
  detector, 300 kV, 30 mrad, G_qk (N_bf, 512, 257) complex64.

The pages never write the SSB sums out; the readings taken here (marked
READING) are the plainest ones consistent with them and with the weak-phase
forward model I = |FFT[P(x-r) e^{i phi}]|^2, P = IFFT[A e^{-i chi}]:

* READING geometry: k of detector pixel (i, j) is ((j - cx) Dk, (i - cy) Dk);
  scan frequency of half-plane entry (row, col) is (f_x, f_y) dq with
  f_x = col in [0, n/2], f_y = fftfreq index of row, dq = 1/(n Delta);
  detector rotation 0.
* READING aperture: A(v) = 1 if |v|^2 <= (alpha/lambda)^2 (hard edge), centred
  on the tilt k_t = tilt/lambda; chi is also evaluated at v = k - k_t.
* READING trotters: with a = A(k), m = A(k - q), p = A(k + q):
  T- = a & m & !p, T+ = a & p & !m; double- and no-overlap pixels are dropped.
  The three aperture tests are a fixed float32 operation sequence (below) so
  that integer outcomes agree bit for bit with the GPU.
* READING weights (first order in phi): on T-, w = exp(-i (chi(k) - chi(k-q)));
  on T+, w = -exp(+i (chi(k) - chi(k+q))).  O(q) = sum G(q,k) w, N(q) = |T-|+|T+|.
* READING image: S(q) = O(q)/N(q) (0 where N = 0), zero on the Nyquist row
  f_y = -n/2 and column f_x = n/2, b = irfft2(-i S with S(0) = 0),
  a = mean_k G(0,k) / n^2, phase = atan2(b, a).
* READING score: over half-plane entries with 0.2 <= |q| <= 0.9 1/A (decided in
  integers against float64 bounds), score = sum |O|^2 / sum N.
"""
from __future__ import annotations

import math

import numpy as np

TWO_PI = 2.0 * math.pi


# ----------------------------------------------------------------------------
# geometry helpers
# ----------------------------------------------------------------------------

def _g(geom):
    """Accept either a configs.Geometry or a plain tuple in ssb_geometry order."""
    if hasattr(geom, "astuple"):
        return geom.astuple()
    return tuple(geom)


def _ab(ab):
    if hasattr(ab, "astuple"):
        return ab.astuple()
    return tuple(ab)


def det_k(geom, i, j):
    """Detector pixel (i, j) -> (k_x, k_y) in 1/A (float64).  Rotation 0."""
    n, dy, dxn, step, dk, lam, alpha, cy, cx = _g(geom)
    kx = (np.asarray(j, dtype=np.float64) - cx) * dk
    ky = (np.asarray(i, dtype=np.float64) - cy) * dk
    return kx, ky


def bf_indices(geom, tilt_x_rad=0.0, tilt_y_rad=0.0):
    """Bright-field set: detector pixels inside the tilted aperture disk.

    ((j - cx) Dk - t_x/lambda)^2 + ((i - cy) Dk - t_y/lambda)^2 <= (alpha/lambda)^2,
    float64, row-major detector index, ascending (WebGPU G(q,k) page,
    "Gotchas recorded": only aperture-active pixels carry G).
    """
    n, det_y, det_x, step, dk, lam, alpha, cy, cx = _g(geom)
    i, j = np.meshgrid(np.arange(det_y), np.arange(det_x), indexing="ij")
    ex = (j - cx) * dk - tilt_x_rad / lam
    ey = (i - cy) * dk - tilt_y_rad / lam
    r = alpha / lam
    inside = (ex * ex + ey * ey) <= r * r
    return np.flatnonzero(inside.ravel()).astype(np.int32)


def scan_freq_index(n):
    """(f_y per half-plane row, f_x per half-plane column) as integers."""
    fy = np.fft.fftfreq(n, d=1.0 / n).round().astype(np.int64)
    fx = np.arange(n // 2 + 1, dtype=np.int64)
    return fy, fx


def band_indices(geom, qmin=0.2, qmax=0.9):
    """Half-plane entries (row*(n/2+1)+col) with qmin <= |q| <= qmax.

    Decided in integers: f_y^2 + f_x^2 against (qmin/dq)^2 and (qmax/dq)^2
    computed in float64.  The tilt-speed page's fit band 0.2..0.9 1/A holds
    44,247 entries at 512^2 and 0.373 A ("Setup").
    """
    n, _, _, step, *_ = _g(geom)
    dq = 1.0 / (n * step)
    lo = (qmin / dq) * (qmin / dq)
    hi = (qmax / dq) * (qmax / dq)
    fy, fx = scan_freq_index(n)
    r2 = (fy[:, None] ** 2 + fx[None, :] ** 2).astype(np.float64)
    sel = (r2 >= lo) & (r2 <= hi)
    return np.flatnonzero(sel.ravel()).astype(np.int32)


# ----------------------------------------------------------------------------
# a2-a4: G(q, k)
# ----------------------------------------------------------------------------

def bf_traces(frames, bf_idx):
    """x_k(r) = float64(frames[r_y, r_x, i_k, j_k]) as (N_bf, n, n)."""
    f = np.asarray(frames)
    n = f.shape[0]
    flat = f.reshape(n * n, -1)
    x = flat[:, np.asarray(bf_idx)].astype(np.float64)
    return np.ascontiguousarray(x.T.reshape(len(bf_idx), n, n))


def build_G(frames, bf_idx):
    """G(q, k) = sum_r x_k(r) exp(-2 pi i q.r), Hermitian half plane.

    WebGPU G(q,k) page, "Why herm is exactly lossless": intensities are real,
    so G(-q,k) = conj G(q,k) and the (n, n/2+1) half plane holds everything.
    Library step: numpy's rfft2 over the two scan axes, float64.
    Output complex128 (N_bf, n, n/2+1), layout [k][q_y row][q_x].
    """
    x = bf_traces(frames, bf_idx)
    return np.fft.rfft2(x, axes=(-2, -1))


# ----------------------------------------------------------------------------
# a5: aberration function
# ----------------------------------------------------------------------------

def chi(vx, vy, ab, lam):
    """Aberration phase chi(v) in radians, polar Krivanek form (float64).

    omega = lambda |v|, phi = atan2(v_y, v_x):
    chi = 2pi/lambda [ omega^2/2 (C10 + C12a cos2phi + C12b sin2phi)
                     + omega^3/3 (C21a cos phi + C21b sin phi + C23a cos3phi + C23b sin3phi)
                     + omega^4/4 (C30 + C32a cos2phi + C32b sin2phi + C34a cos4phi + C34b sin4phi) ]
    (tilt-speed page, "Changes": alpha^2 (1, cos 2 phi, sin 2 phi) structure.)
    """
    (C10, C12a, C12b, C21a, C21b, C23a, C23b, C30, C32a, C32b, C34a, C34b,
     _tx, _ty) = _ab(ab)
    vx = np.asarray(vx, dtype=np.float64)
    vy = np.asarray(vy, dtype=np.float64)
    om = lam * np.hypot(vx, vy)
    ph = np.arctan2(vy, vx)
    c1, s1 = np.cos(ph), np.sin(ph)
    c2, s2 = np.cos(2 * ph), np.sin(2 * ph)
    c3, s3 = np.cos(3 * ph), np.sin(3 * ph)
    c4, s4 = np.cos(4 * ph), np.sin(4 * ph)
    val = (om ** 2 / 2.0 * (C10 + C12a * c2 + C12b * s2)
           + om ** 3 / 3.0 * (C21a * c1 + C21b * s1 + C23a * c3 + C23b * s3)
           + om ** 4 / 4.0 * (C30 + C32a * c2 + C32b * s2 + C34a * c4 + C34b * s4))
    return (TWO_PI / lam) * val


# ----------------------------------------------------------------------------
# a6: trotter classification (fp32 contract) and weights
# ----------------------------------------------------------------------------

def k_coords_f32(geom, bf_idx):
    """float32(k) of each BF pixel: the float64 (j - cx) * Dk rounded once."""
    _, _, det_x, *_ = _g(geom)
    idx = np.asarray(bf_idx, dtype=np.int64)
    kx, ky = det_k(geom, idx // det_x, idx % det_x)
    return kx.astype(np.float32), ky.astype(np.float32)


def q_coords(geom):
    """float64 q_x per column (n/2+1) and q_y per row (n) of the half plane."""
    n, _, _, step, *_ = _g(geom)
    dq = 1.0 / (n * step)
    fy, fx = scan_freq_index(n)
    return fx.astype(np.float64) * dq, fy.astype(np.float64) * dq


def aperture_f32(px, py, tx, ty, r2):
    """Aperture test, float32 contract.

    d2 = (px - tx)*(px - tx) + (py - ty)*(py - ty) <= r2, every operation a
    separate IEEE float32 round-to-nearest operation in exactly this order (no
    fused multiply-add).  px, py, tx, ty, r2 are float32.
    """
    f = np.float32
    dx = (np.asarray(px, f) - f(tx)).astype(f)
    dy = (np.asarray(py, f) - f(ty)).astype(f)
    xx = (dx * dx).astype(f)
    yy = (dy * dy).astype(f)
    d2 = (xx + yy).astype(f)
    return d2 <= f(r2)


def set_constants(geom, ab):
    """float32 tilt centre k_t and float32 (alpha/lambda)^2 of one set."""
    _, _, _, _, _, lam, alpha, *_ = _g(geom)
    a = _ab(ab)
    tx = np.float32(a[12] / lam)
    ty = np.float32(a[13] / lam)
    r = alpha / lam
    r2 = np.float32(r * r)
    return tx, ty, r2


def trotters(geom, ab, bf_idx, qx, qy):
    """Boolean (Nq, N_bf) masks T-, T+ for q = (qx[i], qy[i]) (float64 inputs).

    kappa = float32(k) -/+ float32(q) (one float32 op), then aperture_f32.
    """
    kx, ky = k_coords_f32(geom, bf_idx)
    tx, ty, r2 = set_constants(geom, ab)
    qxf = np.asarray(qx, dtype=np.float64).astype(np.float32)[:, None]
    qyf = np.asarray(qy, dtype=np.float64).astype(np.float32)[:, None]
    a = aperture_f32(kx, ky, tx, ty, r2)[None, :]
    m = aperture_f32((kx[None, :] - qxf).astype(np.float32),
                     (ky[None, :] - qyf).astype(np.float32), tx, ty, r2)
    p = aperture_f32((kx[None, :] + qxf).astype(np.float32),
                     (ky[None, :] + qyf).astype(np.float32), tx, ty, r2)
    tminus = a & m & ~p
    tplus = a & p & ~m
    return tminus, tplus


def weights(geom, ab, bf_idx, qx, qy, tminus, tplus):
    """Complex128 weights w(q,k) on T- / T+ (zero elsewhere), float64 chi.

    Derivation (weak phase, first order): G(q != 0, k) = i Phi(q) n^2
    [A~*(k) A~(k-q) - A~(k) A~*(k+q)], A~ = A exp(-i chi); on T- the first
    bracket term survives and w cancels its phase, on T+ the second survives
    with a minus sign.  Hence G w = i Phi(q) n^2 on every trotter pixel.
    """
    _, _, _, _, _, lam, *_ = _g(geom)
    a = _ab(ab)
    ktx, kty = a[12] / lam, a[13] / lam
    idx = np.asarray(bf_idx, dtype=np.int64)
    _, _, det_x, *_ = _g(geom)
    kx, ky = det_k(geom, idx // det_x, idx % det_x)
    kx = kx[None, :]
    ky = ky[None, :]
    qx = np.asarray(qx, dtype=np.float64)[:, None]
    qy = np.asarray(qy, dtype=np.float64)[:, None]
    chi_k = chi(kx - ktx, ky - kty, ab, lam)
    w = np.zeros(np.broadcast_shapes(tminus.shape), dtype=np.complex128)
    chi_m = chi(kx - qx - ktx, ky - qy - kty, ab, lam)
    chi_p = chi(kx + qx - ktx, ky + qy - kty, ab, lam)
    w = np.where(tminus, np.exp(-1j * (chi_k - chi_m)), w)
    w = np.where(tplus, -np.exp(1j * (chi_k - chi_p)), w)
    return w


def reduce(G, geom, ab, bf_idx, entries=None, chunk=512):
    """O(q) = sum_k G(q,k) w(q,k) and N(q) = |T-(q)| + |T+(q)|.

    G: (N_bf, n, n/2+1) complex; entries: half-plane flat indices
    (row*(n/2+1)+col) or None for all.  Returns (O complex128, N int64) over
    `entries` in order.
    """
    n = G.shape[1]
    h = n // 2 + 1
    if entries is None:
        entries = np.arange(n * h, dtype=np.int64)
    entries = np.asarray(entries, dtype=np.int64)
    qx_col, qy_row = q_coords(geom)
    Gf = G.reshape(G.shape[0], n * h)
    O = np.zeros(len(entries), dtype=np.complex128)
    N = np.zeros(len(entries), dtype=np.int64)
    for s in range(0, len(entries), chunk):
        e = entries[s:s + chunk]
        qx = qx_col[e % h]
        qy = qy_row[e // h]
        tm, tp = trotters(geom, ab, bf_idx, qx, qy)
        w = weights(geom, ab, bf_idx, qx, qy, tm, tp)
        g = Gf[:, e].T                                      # (chunk, N_bf)
        O[s:s + chunk] = (g * w).sum(axis=1)
        N[s:s + chunk] = (tm | tp).sum(axis=1)
    return O, N


# ----------------------------------------------------------------------------
# a7-a8: spectrum assembly, complex-to-real inverse, phase
# ----------------------------------------------------------------------------

def phase_image(O_half, N_half, G0_mean, n, norm="trotter", n_bf=None):
    """Phase image from the half-plane O, N and a = mean_k G(0,k).

    norm="trotter": S = O/N (0 where N = 0).  norm="bf_mean": S = O/N_bf, the
    plain mean over bright-field pixels of the WebGPU page's object fast path.
    Nyquist row/column zeroed, DC removed, b = irfft2(-i S) (numpy semantics),
    a = G0_mean / n^2, phase = atan2(b, a).  Returns float64 (n, n).
    """
    h = n // 2 + 1
    O = np.asarray(O_half, dtype=np.complex128).reshape(n, h)
    N = np.asarray(N_half).reshape(n, h)
    if norm == "trotter":
        S = np.where(N > 0, O / np.maximum(N, 1), 0.0)
    elif norm == "bf_mean":
        S = O / float(n_bf)
    else:
        raise ValueError(norm)
    S = S.copy()
    S[n // 2, :] = 0.0
    S[:, n // 2] = 0.0
    S[0, 0] = 0.0
    b = np.fft.irfft2(-1j * S, s=(n, n))
    a = float(np.real(G0_mean)) / (n * n)
    return np.arctan2(b, a)


def g0_mean(G):
    return np.mean(G[:, 0, 0])


# ----------------------------------------------------------------------------
# a9: score
# ----------------------------------------------------------------------------

def score(O_band, N_band):
    """sum_q |O(q)|^2 / sum_q N(q) over the band (0 if the band is empty)."""
    den = float(np.sum(N_band))
    if den == 0:
        return 0.0
    return float(np.sum(np.abs(O_band) ** 2) / den)


# ----------------------------------------------------------------------------
# end to end
# ----------------------------------------------------------------------------

def reconstruct(frames, geom, ab, bf_idx=None, norm="trotter"):
    """G build + reduction over the half plane + phase image (float64)."""
    if bf_idx is None:
        a = _ab(ab)
        bf_idx = bf_indices(geom, a[12], a[13])
    G = build_G(frames, bf_idx)
    O, N = reduce(G, geom, ab, bf_idx)
    n = G.shape[1]
    ph = phase_image(O, N, g0_mean(G), n, norm=norm, n_bf=len(bf_idx))
    return {"G": G, "O": O, "N": N, "phase": ph, "bf_idx": bf_idx}


def score_sets(G, geom, sets, bf_idx, band):
    """Per set: O over the band, N over the band and the score."""
    out = []
    for ab in sets:
        O, N = reduce(G, geom, ab, bf_idx, entries=band)
        out.append((O, N, score(O, N)))
    return out


# ----------------------------------------------------------------------------
# depth-spread ("thick") fit: the weights averaged over a defocus spread
# ----------------------------------------------------------------------------
# Source: "Tilt-corrected SSB on CUDA: fit and preview speed", sections
# "Changes" (the fit kernel at depth 136 A and at depth 0; per (k, q, set) term
# two sincos and two sin at depth, the transcendental pipe busiest) and
# "Results" (a depth spread is one of the fitted parameters); "Where the 9 s of
# regularized preparation goes", list item 2 ("chi, sinc and phase factor" of
# a transfer term, evaluated only inside the lens).  The pages never write
# the depth model out.
# READING depth model: the probe's defocus is spread uniformly over a slab of
# thickness t centred on the set's C10 (z in [-t/2, t/2], defocus C10 + z);
# defocus enters chi(v) as pi lambda C10 |v|^2 (radians), so the transfer of a
# trotter pixel, averaged over the slab, is its depth-0 value times the real
# factor avg_z exp(i pi lambda z D) = sinc(pi lambda t D / 2), sinc(x) =
# sin(x)/x, with D = |v_k|^2 - |v_{k-q}|^2 on T- and |v_k|^2 - |v_{k+q}|^2 on T+
# (v = k - k_t).
# READING weight: the fit weights each trotter term by the depth-0 weight
# times that factor (the matched filter of the averaged transfer); N(q) still
# counts trotter pixels, and the score is sum |O|^2 / sum N as at depth 0.
# t = 0 gives the depth-0 weights exactly.

def depth_factor(geom, ab, bf_idx, qx, qy, tminus, tplus, depth_A):
    """Real (Nq, N_bf) factor sinc(pi lambda t D / 2) on T-/T+ (1 elsewhere),
    float64; depth_A = t (Angstrom, >= 0)."""
    _, _, det_x, _, _, lam, *_ = _g(geom)
    a = _ab(ab)
    ktx, kty = a[12] / lam, a[13] / lam
    idx = np.asarray(bf_idx, dtype=np.int64)
    kx, ky = det_k(geom, idx // det_x, idx % det_x)
    vkx, vky = (kx - ktx)[None, :], (ky - kty)[None, :]
    qx = np.asarray(qx, dtype=np.float64)[:, None]
    qy = np.asarray(qy, dtype=np.float64)[:, None]
    vk2 = vkx * vkx + vky * vky
    dm = vk2 - ((vkx - qx) ** 2 + (vky - qy) ** 2)
    dp = vk2 - ((vkx + qx) ** 2 + (vky + qy) ** 2)
    d = np.where(tminus, dm, np.where(tplus, dp, 0.0))
    x = math.pi * lam * float(depth_A) * d / 2.0
    return np.sinc(x / math.pi)  # numpy's sinc is sin(pi u)/(pi u)


def reduce_depth(G, geom, ab, bf_idx, depth_A, entries=None, chunk=512):
    """reduce() with the depth-spread weights w * sinc(pi lambda t D / 2)."""
    n = G.shape[1]
    h = n // 2 + 1
    if entries is None:
        entries = np.arange(n * h, dtype=np.int64)
    entries = np.asarray(entries, dtype=np.int64)
    qx_col, qy_row = q_coords(geom)
    Gf = G.reshape(G.shape[0], n * h)
    O = np.zeros(len(entries), dtype=np.complex128)
    N = np.zeros(len(entries), dtype=np.int64)
    for s in range(0, len(entries), chunk):
        e = entries[s:s + chunk]
        qx = qx_col[e % h]
        qy = qy_row[e // h]
        tm, tp = trotters(geom, ab, bf_idx, qx, qy)
        w = weights(geom, ab, bf_idx, qx, qy, tm, tp) * depth_factor(geom, ab, bf_idx, qx, qy, tm, tp, depth_A)
        g = Gf[:, e].T
        O[s:s + chunk] = (g * w).sum(axis=1)
        N[s:s + chunk] = (tm | tp).sum(axis=1)
    return O, N


# ----------------------------------------------------------------------------
# compact G storage: herm16 (snorm16 codes + float32 block scales) and the
# band-compacted copy
# ----------------------------------------------------------------------------
# Sources: "Historical WebGPU G(q,k) memory experiment", section
# "Implementation": a post-pass over the built half plane first takes the
# per-BF-pixel maximum of |G| (scaleMax), then stores each component as
# pack2x16snorm(clamp(v / scale)); a reader multiplies unpack2x16snorm(word) by
# the pixel's scale.  Section "Memory planning table": active_BF * N * (N/2+1)
# * 4 bytes plus 4 bytes per BF pixel.  Section "Scan-size sweep", conclusions,
# and "Lessons learned" item 3: per-q-row block scales (n scales per BF pixel)
# as the follow-up that bounds the dynamic range inside each block.
#
# READING pack2x16snorm (the WGSL built-in the page names): component e is
# stored as the 16-bit two's complement integer floor(0.5 + 32767 * clamp(e,
# -1, 1)), component 0 (real) in bits 0-15 and component 1 (imaginary) in bits
# 16-31; unpack2x16snorm gives max(c / 32767, -1).
# READING precision: the pages fix none; scale, quotient and code are taken in
# float32 (the kernel's precision), each operation rounded once, so the integer
# codes are decided in the same precision on both sides.
# READING |G|: the complex modulus, sqrt(re^2 + im^2).  max |G| = sqrt(max
# re^2 + im^2) since a correctly rounded sqrt is monotone.
# READING empty block: a block whose max |G| is 0 stores scale 0 and codes 0.
# READING block shapes: rows_per_scale = n (one scale per BF pixel, the page's
# preview) or 1 (one scale per q row of the half plane, the follow-up).
# Scales are laid out [n / rows_per_scale][N_bf].

SNORM16_MAX = 32767


def herm16_scales(G32, rows_per_scale):
    """max |G| per (row block, BF pixel) in float32: array (n/rows, N_bf)."""
    G32 = np.asarray(G32, dtype=np.complex64)
    nbf, n, h = G32.shape
    if rows_per_scale not in (1, n):
        raise ValueError("rows_per_scale must be 1 or n")
    x = G32.real.astype(np.float32)
    y = G32.imag.astype(np.float32)
    m2 = x * x + y * y                                   # float32, one rounding per op
    blocks = n // rows_per_scale
    m2 = m2.reshape(nbf, blocks, rows_per_scale * h).max(axis=2)
    return np.sqrt(m2).T.copy()                          # (blocks, N_bf) float32


def _snorm16(v, s):
    """floor(0.5 + 32767 clamp(v / s, -1, 1)) in float32; 0 where s == 0."""
    v = np.asarray(v, dtype=np.float32)
    s = np.asarray(s, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.where(s > 0, v / np.where(s > 0, s, np.float32(1)), np.float32(0)).astype(np.float32)
    e = np.minimum(np.float32(1), np.maximum(np.float32(-1), e))
    c = np.floor(np.float32(0.5) + np.float32(SNORM16_MAX) * e)
    return c.astype(np.int16)


def herm16_pack(G32, rows_per_scale):
    """(codes int16 (N_bf, n, n/2+1, 2) [re, im], scales float32 (n/rows, N_bf))."""
    G32 = np.asarray(G32, dtype=np.complex64)
    nbf, n, h = G32.shape
    sc = herm16_scales(G32, rows_per_scale)
    # scale of entry (k, row, col): block row // rows_per_scale
    s_full = np.repeat(sc.T, rows_per_scale, axis=1)[:, :, None]      # (N_bf, n, 1)
    codes = np.empty((nbf, n, h, 2), dtype=np.int16)
    codes[..., 0] = _snorm16(G32.real, s_full)
    codes[..., 1] = _snorm16(G32.imag, s_full)
    return codes, sc


def herm16_unpack(codes, scales, rows_per_scale):
    """complex128 G~ = max(c / 32767, -1) * scale, per component."""
    codes = np.asarray(codes)
    nbf, n, h, _ = codes.shape
    s_full = np.repeat(np.asarray(scales, dtype=np.float64).T, rows_per_scale, axis=1)[:, :, None]
    u = np.maximum(codes.astype(np.float64) / SNORM16_MAX, -1.0)
    return (u[..., 0] + 1j * u[..., 1]) * s_full


def herm16_bytes(nbf, n, rows_per_scale):
    """Stored bytes: 4 per half-plane entry plus 4 per scale."""
    return nbf * n * (n // 2 + 1) * 4 + (n // rows_per_scale) * nbf * 4


def band_compact(G, band):
    """The band entries of every BF pixel's half plane, in band order:
    (N_bf, n, n/2+1, ...) -> (N_bf, nq, ...).  No page describes this copy;
    the scoring passes of a fit ("Tilt-corrected SSB on CUDA", section "Where
    the time went": 78 passes) read only these entries."""
    G = np.asarray(G)
    nbf, n, h = G.shape[:3]
    return G.reshape((nbf, n * h) + G.shape[3:])[:, np.asarray(band, dtype=np.int64)]


# ----------------------------------------------------------------------------
# per-BF phase moments: the exact mean(angle) path
# ----------------------------------------------------------------------------
# Sources: "Historical WebGPU G(q,k) memory experiment", section "Object-redraw
# fast path": the exact per-BF path takes, for every BF pixel, the inverse FFT
# of its aberration-corrected plane and the angle of that object, and averages
# the angles (mean(angle(object))); the loss needs the per-BF phases because it
# uses the variance of mean(angle).  "Tilt-corrected SSB on CUDA", sections
# "Changes" (Loss path: the corrected plane is written from the stored half
# plane, the angles are reduced to moments as they are read) and "Open" (the
# corrected spectrum of a real image is anti-Hermitian except at DC, so a
# half-plane complex-to-real transform gives the image).
#
# READING corrected plane: S_k(q) = G(q,k) w(q,k) on the trotter pixels of BF
# pixel k (the terms the reduction sums), 0 elsewhere; zeroed at DC and on the
# Nyquist row and column as in the single image.
# READING object of one BF pixel: a_k + i b_k with a_k = Re G(0,k) / n^2 and
# b_k = irfft2(-i S_k) (numpy semantics), the per-pixel form of the image's
# a + i b; its angle is atan2(b_k, a_k).
# READING moments: per scan pixel, the mean over the N_bf BF pixels of the
# angle and its population variance (divided by N_bf).  The pages give no
# scalar loss formula, so the moments are the output.


def corrected_planes(G, geom, ab, bf_idx, chunk=512):
    """S_k(q) = G(q,k) w(q,k) on T-(q) | T+(q) of pixel k, 0 elsewhere:
    complex128 (N_bf, n, n/2+1)."""
    nbf, n, h = G.shape
    qx_col, qy_row = q_coords(geom)
    Gf = np.asarray(G).reshape(nbf, n * h)
    S = np.zeros((nbf, n * h), dtype=np.complex128)
    for s in range(0, n * h, chunk):
        e = np.arange(s, min(s + chunk, n * h))
        qx = qx_col[e % h]
        qy = qy_row[e // h]
        tm, tp = trotters(geom, ab, bf_idx, qx, qy)
        w = weights(geom, ab, bf_idx, qx, qy, tm, tp)          # (chunk, N_bf), 0 off the trotters
        S[:, e] = Gf[:, e] * w.T
    return S.reshape(nbf, n, h)


def per_bf_images(G, geom, ab, bf_idx):
    """(a_k, b_k) of every BF pixel in order: a_k = Re G(0,k) / n^2 (float),
    b_k = irfft2(-i S_k) (float64 (n, n)) with S_k zeroed at DC and on the
    Nyquist row and column."""
    nbf, n, h = G.shape
    S = corrected_planes(G, geom, ab, bf_idx)
    for k in range(nbf):
        Sk = S[k].copy()
        Sk[n // 2, :] = 0.0
        Sk[:, n // 2] = 0.0
        Sk[0, 0] = 0.0
        yield float(np.real(G[k, 0, 0])) / (n * n), np.fft.irfft2(-1j * Sk, s=(n, n))


def phase_moments(G, geom, ab, bf_idx):
    """Per scan pixel: mean over BF pixels of atan2(b_k, a_k) and its
    population variance.  Returns (mean, var), float64 (n, n)."""
    nbf, n, _ = G.shape
    s1 = np.zeros((n, n))
    s2 = np.zeros((n, n))
    for a, b in per_bf_images(G, geom, ab, bf_idx):
        ph = np.arctan2(b, a)
        s1 += ph
        s2 += ph * ph
    mean = s1 / nbf
    var = np.maximum(s2 / nbf - mean * mean, 0.0)
    return mean, var
