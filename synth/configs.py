"""Seeded synthetic workloads for SSB direct ptychography.

This module holds configuration only: scan/detector geometry, the seeded
aberration draws and the per-workload recipe.  It contains none of the
reconstruction arithmetic; both the CPU oracle and the CUDA path receive the
numbers produced here as plain inputs.

Workloads (scan n x n at 0.373 A, 300 kV, 30 mrad):

* ``tiny``  32^2 scan, 24^2 float32 detector, 6 Gaussian atoms, C10=-50 A,
  C30=1e4 A, noiseless (the small worked case the oracle finishes in seconds).
* ``small`` 128^2 scan, 64^2 uint16 detector, 120 atoms, random aberrations,
  tilt (5.92, -0.07) mrad, Poisson at a mean of 5 counts per BF pixel.
* ``full``  512^2 scan, 192^2 uint16 detector, hexagonal crystal a=3.16 A with
  2 % vacancies, random aberrations + tilt, Poisson at a mean of 3 counts.
* ``batch`` B aberration sets perturbed from the ``full`` draw, scored over
  the band 0.2 <= |q| <= 0.9 1/A.
* ``large`` as ``full`` on a 1024^2 scan.
* ``mid``   512^2 scan with the 64^2 detector of ``small`` (profiling case).
* ``middet`` 256^2 scan, 128^2 detector at the ``full`` sampling (~9.3k BF
  pixels; profiling case for the reductions).
* ``midlarge`` 1024^2 scan, 32^2 detector (~250 BF pixels; profiling case for
  the two-pass n = 1024 build).

The sources for these numbers are the MoS2 / crystal scans of the quantem.gpu
SSB reports (2026-10-24 regularized preparation, "Setup"; 2026-10-20 tilt
speed, "Setup"), where a 512^2 scan with a 192^2 detector at 300 kV, 30 mrad
and 0.373 A step carries ~9.3k bright-field pixels and max ~17 counts.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Relativistic electron wavelength at 300 kV, as printed for these workloads.
WAVELENGTH_300KV_A = 0.019687
SEMIANGLE_RAD = 30e-3
SCAN_STEP_A = 0.373
OVERSAMPLE = 4  # object pixels per scan step

ABERRATION_NAMES = ("C10", "C12a", "C12b", "C21a", "C21b", "C23a", "C23b",
                    "C30", "C32a", "C32b", "C34a", "C34b")

# Uniform draw ranges (Angstrom) for random aberrations.
ABERRATION_RANGES = {
    "C10": (-200.0, 200.0),
    "C12a": (-50.0, 50.0), "C12b": (-50.0, 50.0),
    "C21a": (-50.0, 50.0), "C21b": (-50.0, 50.0),
    "C23a": (-50.0, 50.0), "C23b": (-50.0, 50.0),
    "C30": (-1e4, 1e4),
    "C32a": (-1e4, 1e4), "C32b": (-1e4, 1e4),
    "C34a": (-1e4, 1e4), "C34b": (-1e4, 1e4),
}


@dataclasses.dataclass(frozen=True)
class Geometry:
    """Scan + detector geometry (mirrors ``ssb_geometry`` in include/ssb.h)."""
    n: int                 # scan is n x n positions
    det_y: int
    det_x: int
    scan_step_A: float     # Delta, scan step in Angstrom
    det_pitch_invA: float  # Delta_k, detector pixel pitch in 1/Angstrom
    wavelength_A: float    # lambda
    semiangle_rad: float   # alpha
    det_center_y: float    # detector pixel index of k_y = 0
    det_center_x: float    # detector pixel index of k_x = 0

    def astuple(self):
        return dataclasses.astuple(self)


@dataclasses.dataclass(frozen=True)
class Aberrations:
    """One aberration set (mirrors ``ssb_aberr``): Krivanek a/b coefficients in
    Angstrom and the probe tilt in radians."""
    C10: float = 0.0
    C12a: float = 0.0
    C12b: float = 0.0
    C21a: float = 0.0
    C21b: float = 0.0
    C23a: float = 0.0
    C23b: float = 0.0
    C30: float = 0.0
    C32a: float = 0.0
    C32b: float = 0.0
    C34a: float = 0.0
    C34b: float = 0.0
    tilt_x_rad: float = 0.0
    tilt_y_rad: float = 0.0

    def astuple(self):
        return dataclasses.astuple(self)

    def replace(self, **kw):
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    n: int                 # scan size
    det: int               # square detector size
    det_mrad_per_px: float  # stated detector sampling (mrad per pixel)
    dtype: str             # "f32" or "u16"
    dose: float | None     # mean counts per BF pixel (None: noiseless)
    object_kind: str       # "gaussians" or "hex"
    n_atoms: int = 0
    lattice_A: float = 3.16
    vacancy: float = 0.02
    atom_phase: float = 0.1
    atom_sigma_A: float = 0.4


WORKLOADS = {
    # tiny / small state the aperture radius (8 / 18 px at 30 mrad); full and
    # large state 0.551 mrad per pixel directly.
    "tiny": Workload("tiny", 0, 32, 24, 30.0 / 8.0, "f32", None, "gaussians", n_atoms=6),
    "small": Workload("small", 1, 128, 64, 30.0 / 18.0, "u16", 5.0, "gaussians", n_atoms=120),
    "full": Workload("full", 2, 512, 192, 0.551, "u16", 3.0, "hex"),
    "large": Workload("large", 3, 1024, 192, 0.551, "u16", 3.0, "hex"),
    # profiling case: the full scan size with the small detector (2.1 GB of
    # frames, ~1k BF pixels) so that many-pass counter captures stay small
    "mid": Workload("mid", 5, 512, 64, 30.0 / 18.0, "u16", 3.0, "hex"),
    # profiling case for the reductions: the full workload's detector sampling
    # and aperture (~9.3k BF pixels, rows of ~86 pixels; the 109-pixel BF disc
    # fits a 128^2 detector) on a 256^2 scan: 2.1 GB of frames, 2.5 GB of G
    "middet": Workload("middet", 6, 256, 128, 0.551, "u16", 3.0, "hex"),
    # profiling case for the two-pass n = 1024 build: the large scan with a
    # 32^2 detector (BF radius ~9 px, ~250 BF pixels): 2.1 GB of frames, 1 GB of G
    "midlarge": Workload("midlarge", 7, 1024, 32, 30.0 / 9.0, "u16", 3.0, "hex"),
}


def probe_window(w: Workload) -> tuple[int, float]:
    """Forward-model probe window N_w (object pixels) and object pixel size dx.

    The object grid is 4x oversampled (dx = step/4).  The stated detector
    sampling gives a target pitch Dk_t = (mrad per px)/lambda; the window is the
    even integer nearest 1/(Dk_t dx), so the detector pitch actually simulated
    is 1/(N_w dx).
    """
    dx = SCAN_STEP_A / OVERSAMPLE
    dk_target = (w.det_mrad_per_px * 1e-3) / WAVELENGTH_300KV_A
    raw = 1.0 / (dk_target * dx)
    n_w = int(2 * round(raw / 2.0))
    return n_w, dx


def geometry(w: Workload) -> Geometry:
    n_w, dx = probe_window(w)
    dk = 1.0 / (n_w * dx)
    return Geometry(n=w.n, det_y=w.det, det_x=w.det, scan_step_A=SCAN_STEP_A,
                    det_pitch_invA=dk, wavelength_A=WAVELENGTH_300KV_A,
                    semiangle_rad=SEMIANGLE_RAD,
                    det_center_y=float(w.det // 2), det_center_x=float(w.det // 2))


def draw_aberrations(rng: np.random.Generator) -> dict:
    """Uniform draw of the 12 coefficients over ABERRATION_RANGES, fixed order."""
    out = {}
    for name in ABERRATION_NAMES:
        lo, hi = ABERRATION_RANGES[name]
        out[name] = float(rng.uniform(lo, hi))
    return out


SMALL_TILT = (5.92e-3, -0.07e-3)   # (tilt_x, tilt_y) rad


def aberrations(w: Workload) -> Aberrations:
    """The aberration set a workload's data is simulated with (and that the
    matched reconstruction uses)."""
    if w.name == "tiny":
        return Aberrations(C10=-50.0, C30=1e4)
    rng = np.random.default_rng(w.seed)
    coeffs = draw_aberrations(rng)
    return Aberrations(**coeffs, tilt_x_rad=SMALL_TILT[0], tilt_y_rad=SMALL_TILT[1])


def perturbed_sets(base: Aberrations, count: int, seed: int = 4) -> list[Aberrations]:
    """Aberration sets for batched scoring: base + N(0, sd) per coefficient,
    sd = 20 A for C10 and 10 % of the range width for the others.  The tilt
    is not perturbed (no range is given for it)."""
    rng = np.random.default_rng(seed)
    sets = []
    for _ in range(count):
        kw = {}
        for name in ABERRATION_NAMES:
            lo, hi = ABERRATION_RANGES[name]
            sd = 20.0 if name == "C10" else 0.1 * (hi - lo)
            kw[name] = getattr(base, name) + float(rng.normal(0.0, sd))
        sets.append(base.replace(**kw))
    return sets


BAND_INVA = (0.2, 0.9)


def g_bytes(n_bf: int, n: int) -> int:
    """Bytes of the complex64 Hermitian half-plane G(q,k)."""
    return n_bf * n * (n // 2 + 1) * 8


def full_plane_bytes(n_bf: int, n: int) -> int:
    return n_bf * n * n * 8


def herm16_bytes(n_bf: int, n: int) -> int:
    return n_bf * n * (n // 2 + 1) * 4 + n_bf * 4


def nominal_bf_radius_px(g: Geometry) -> float:
    return (g.semiangle_rad / g.wavelength_A) / g.det_pitch_invA


def describe(w: Workload) -> dict:
    g = geometry(w)
    n_w, dx = probe_window(w)
    return {"workload": w.name, "scan": f"{w.n}x{w.n}", "detector": f"{w.det}x{w.det}",
            "dtype": w.dtype, "probe_window": n_w, "dx_A": dx,
            "det_pitch_mrad": g.det_pitch_invA * g.wavelength_A * 1e3,
            "bf_radius_px": nominal_bf_radius_px(g)}


def tilt_shift_px(g: Geometry, ab: Aberrations) -> float:
    return math.hypot(ab.tilt_x_rad, ab.tilt_y_rad) / g.wavelength_A / g.det_pitch_invA
