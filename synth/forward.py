"""Seeded single-slice 4D-STEM forward model (input generator).

Simulates I(r, k) = |FFT[P(x - r) exp(i phi(x))](k)|^2 for a probe
P = IFFT[A(k - k_t) exp(-i chi(k - k_t))] scanned over a periodic weak-phase
object, then crops the central det x det detector and (optionally) draws
Poisson counts.  This is the data model the SSB workloads are quoted on; the
reconstruction itself (G build, trotter reduction, phase image) lives in the
oracle and in the CUDA library, not here.

Conventions shared with everything downstream (they are conventions of the
data, not of the method):

* object pixel size dx = scan step / 4; scan position (ry, rx) sits on object
  pixel (4 ry, 4 rx); the probe window is N_w x N_w object pixels centred on
  the scan position, periodic wrap;
* detector pixel (i, j) <-> k = ((j - det/2) Dk, (i - det/2) Dk) with
  Dk = 1/(N_w dx), i.e. the central det x det crop of the fftshifted window
  spectrum;
* frames are laid out (scan_y, scan_x, det_y, det_x).

The probe phase here is evaluated from complex powers of omega = lambda (v_x +
i v_y) (theta^m cos(n phi) = Re(omega^n) |omega|^(m-n)); it is a data
generator's own evaluation, independent of the oracle's and the kernels'.
"""
from __future__ import annotations

import math

import numpy as np

from . import configs as C


# ----------------------------------------------------------------------------
# object
# ----------------------------------------------------------------------------

def _splat_gaussians(npix: int, dx: float, centers: np.ndarray, sigma: float,
                     amp: float) -> np.ndarray:
    """Periodic sum of Gaussians amp * exp(-|x - c|^2 / (2 sigma^2))."""
    phi = np.zeros((npix, npix), dtype=np.float64)
    rad = int(math.ceil(5.0 * sigma / dx))
    rad = min(rad, (npix - 1) // 2)
    offs = np.arange(-rad, rad + 1)
    for cy, cx in centers:
        py, px = cy / dx, cx / dx
        iy0, ix0 = int(round(py)), int(round(px))
        ys = iy0 + offs
        xs = ix0 + offs
        gy = np.exp(-((ys - py) * dx) ** 2 / (2 * sigma * sigma))
        gx = np.exp(-((xs - px) * dx) ** 2 / (2 * sigma * sigma))
        phi[np.ix_(ys % npix, xs % npix)] += amp * np.outer(gy, gx)
    return phi


def object_phase(w: C.Workload, rng: np.random.Generator) -> np.ndarray:
    """Weak-phase object phi (radians) on the 4x oversampled periodic grid."""
    npix = w.n * C.OVERSAMPLE
    dx = C.SCAN_STEP_A / C.OVERSAMPLE
    box = npix * dx
    if w.object_kind == "gaussians":
        centers = rng.uniform(0.0, box, size=(w.n_atoms, 2))
    elif w.object_kind == "hex":
        a = w.lattice_A
        origin = rng.uniform(0.0, a, size=2)
        rows = int(math.ceil(box / (a * math.sqrt(3) / 2))) + 2
        cols = int(math.ceil(box / a)) + 2
        jj, ii = np.meshgrid(np.arange(-1, rows), np.arange(-1, cols), indexing="ij")
        ys = origin[0] + jj * a * math.sqrt(3) / 2
        xs = origin[1] + ii * a + (jj % 2) * a / 2
        keep = (ys >= 0) & (ys < box) & (xs >= 0) & (xs < box)
        centers = np.stack([ys[keep], xs[keep]], axis=1)
        present = rng.random(len(centers)) >= w.vacancy
        centers = centers[present]
    else:
        raise ValueError(w.object_kind)
    return _splat_gaussians(npix, dx, centers, w.atom_sigma_A, w.atom_phase)


def truth_at_scan(phi: np.ndarray, n: int) -> np.ndarray:
    """Ground-truth phase sampled at the n x n scan positions."""
    return phi[::C.OVERSAMPLE, ::C.OVERSAMPLE][:n, :n].copy()


# ----------------------------------------------------------------------------
# probe
# ----------------------------------------------------------------------------

def probe_phase(vx, vy, ab: C.Aberrations, lam: float):
    """Probe aberration phase (radians) at detector-plane offset v = k - k_t."""
    om = lam * (np.asarray(vx) + 1j * np.asarray(vy))
    t2 = (om * np.conj(om)).real
    om2 = om * om
    om3 = om2 * om
    om4 = om2 * om2

    def re(c_a, c_b, z):
        return ((c_a - 1j * c_b) * z).real

    val = (0.5 * (ab.C10 * t2 + re(ab.C12a, ab.C12b, om2))
           + (1.0 / 3.0) * (re(ab.C21a, ab.C21b, om) * t2 + re(ab.C23a, ab.C23b, om3))
           + 0.25 * (ab.C30 * t2 * t2 + re(ab.C32a, ab.C32b, om2) * t2
                     + re(ab.C34a, ab.C34b, om4)))
    return (2.0 * math.pi / lam) * val


def probe_window_spectrum(geom: C.Geometry, ab: C.Aberrations, n_w: int, dx: float):
    """A(k - k_t) exp(-i chi(k - k_t)) on the N_w x N_w window frequency grid
    (unshifted FFT order)."""
    f = np.fft.fftfreq(n_w, d=dx)
    ky, kx = np.meshgrid(f, f, indexing="ij")
    lam = geom.wavelength_A
    vx = kx - ab.tilt_x_rad / lam
    vy = ky - ab.tilt_y_rad / lam
    kmax = geom.semiangle_rad / lam
    aperture = (vx * vx + vy * vy) <= kmax * kmax
    return np.where(aperture, np.exp(-1j * probe_phase(vx, vy, ab, lam)), 0.0)


def probe_centered(geom: C.Geometry, ab: C.Aberrations, n_w: int, dx: float):
    """Real-space probe with its origin moved to window pixel N_w/2."""
    p = np.fft.ifft2(probe_window_spectrum(geom, ab, n_w, dx))
    return np.fft.fftshift(p)


def detector_crop_index(n_w: int, det: int) -> np.ndarray:
    """Unshifted window-spectrum indices of detector pixels 0..det-1."""
    return (np.arange(det) - det // 2) % n_w


# ----------------------------------------------------------------------------
# simulation
# ----------------------------------------------------------------------------

def simulate_numpy(phi: np.ndarray, geom: C.Geometry, ab: C.Aberrations,
                   n_w: int, dx: float) -> np.ndarray:
    """Noiseless intensities, float64 (n, n, det_y, det_x)."""
    n = geom.n
    npix = phi.shape[0]
    pc = probe_centered(geom, ab, n_w, dx)
    obj = np.exp(1j * phi)
    cy = detector_crop_index(n_w, geom.det_y)
    cx = detector_crop_index(n_w, geom.det_x)
    out = np.empty((n, n, geom.det_y, geom.det_x), dtype=np.float64)
    win = np.arange(n_w) - n_w // 2
    for ry in range(n):
        rows = (C.OVERSAMPLE * ry + win) % npix
        strip = obj[rows]                                   # (n_w, npix)
        cols = (C.OVERSAMPLE * np.arange(n)[:, None] + win[None, :]) % npix
        windows = strip[:, cols].transpose(1, 0, 2)         # (n, n_w, n_w)
        psi = np.fft.fft2(windows * pc[None], axes=(-2, -1))
        psi = psi[:, cy][:, :, cx]
        out[ry] = (psi * np.conj(psi)).real
    return out


def poisson_counts(intensity: np.ndarray, dose: float, rng: np.random.Generator) -> np.ndarray:
    """Poisson counts at mean `dose` x intensity, stored as uint16."""
    counts = rng.poisson(intensity * dose)
    return np.minimum(counts, 65535).astype(np.uint16)


def make_numpy_dataset(name: str):
    """Frames, geometry, aberrations and truth for the CPU-sized workloads.

    Returns dict(frames, geom, ab, phi, truth, n_w, dx).  RNG draw order for a
    workload seed: aberrations (in ``configs.aberrations``, own generator),
    then object atoms, then Poisson noise.
    """
    w = C.WORKLOADS[name]
    geom = C.geometry(w)
    ab = C.aberrations(w)
    n_w, dx = C.probe_window(w)
    rng = np.random.default_rng(w.seed + 100)
    phi = object_phase(w, rng)
    inten = simulate_numpy(phi, geom, ab, n_w, dx)
    if w.dtype == "f32":
        frames = inten.astype(np.float32)
    else:
        frames = poisson_counts(inten, w.dose, rng)
    return {"frames": frames, "geom": geom, "ab": ab, "phi": phi,
            "truth": truth_at_scan(phi, w.n), "n_w": n_w, "dx": dx, "workload": w}


def make_torch_dataset(name: str, device="cuda", rows_per_batch: int = 1):
    """GPU-generated frames for the full-size workloads (torch, off the timed
    path).  Returns dict(frames=int16 tensor on `device` holding the uint16
    counts bit for bit, geom, ab, phi, truth, n_w, dx, workload, max_count,
    mean_bf_count)."""
    import torch

    w = C.WORKLOADS[name]
    geom = C.geometry(w)
    ab = C.aberrations(w)
    n_w, dx = C.probe_window(w)
    rng = np.random.default_rng(w.seed + 100)
    phi = object_phase(w, rng)
    n = geom.n
    npix = phi.shape[0]
    dev = torch.device(device)
    obj = torch.exp(1j * torch.from_numpy(phi).to(dev, torch.float64)).to(torch.complex64)
    pc = torch.from_numpy(probe_centered(geom, ab, n_w, dx)).to(dev, torch.complex64)
    win = torch.arange(n_w, device=dev) - n_w // 2
    ext_cols = (torch.arange(npix + n_w, device=dev) - n_w // 2) % npix
    cy = torch.from_numpy(detector_crop_index(n_w, geom.det_y)).to(dev)
    cx = torch.from_numpy(detector_crop_index(n_w, geom.det_x)).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    frames = torch.empty((n, n, geom.det_y, geom.det_x), dtype=torch.int16, device=dev)
    max_count = 0
    total = 0.0
    for ry0 in range(0, n, rows_per_batch):
        ry1 = min(n, ry0 + rows_per_batch)
        for ry in range(ry0, ry1):
            rows = (C.OVERSAMPLE * ry + win) % npix
            strip = obj.index_select(0, rows)[:, ext_cols]            # (n_w, npix + n_w)
            windows = strip.unfold(1, n_w, C.OVERSAMPLE)[:, :n]       # (n_w, n, n_w)
            windows = windows.permute(1, 0, 2)                        # (n, n_w, n_w)
            psi = torch.fft.fft2(windows * pc, dim=(-2, -1))
            psi = psi.index_select(1, cy).index_select(2, cx)
            inten = psi.real * psi.real + psi.imag * psi.imag
            counts = torch.poisson(inten * w.dose, generator=gen)
            counts = counts.clamp_(max=65535).to(torch.int32)
            frames[ry] = counts.to(torch.int16)
            max_count = max(max_count, int(counts.max().item()))
    return {"frames": frames, "geom": geom, "ab": ab, "phi": phi,
            "truth": truth_at_scan(phi, n), "n_w": n_w, "dx": dx, "workload": w,
            "max_count": max_count}
