"""GB300 single-sideband (SSB) direct ptychography: Python binding of libssb.

The functions here only marshal arguments (torch tensors -> device pointers,
dataclasses -> C structs, the current CUDA stream) and call the C ABI declared
in ``include/ssb.h``; every step of the computation runs in the library's
CUDA kernels.  There is no fallback: if ``libssb.so`` is missing or a GPU call
fails, these functions raise.

Typical use::

    import electron_microscopy_gb300 as ssb
    bf = ssb.bf_indices(geom, base_set)                  # numpy int32 (host)
    G = ssb.build_G(frames, geom, bf_dev)                # frames: cuda tensor
    O, N, phase = ssb.reconstruct(G, geom, bf_dev, base_set)
    O_b, N_b, score = ssb.score_batch(G, geom, bf_dev, sets, band_dev)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssb.so")

SSB_OK, SSB_INVALID_ARG, SSB_UNSUPPORTED, SSB_WORKSPACE_TOO_SMALL, SSB_CUDA_ERROR = range(5)
SSB_U16, SSB_F32 = 0, 1
OP_BUILD, OP_RECON, OP_SCORE, OP_MOMENTS, OP_PHASE = 0, 1, 2, 3, 4
MAX_SETS = 8

STATUS_NAMES = {0: "SSB_OK", 1: "SSB_INVALID_ARG", 2: "SSB_UNSUPPORTED",
                3: "SSB_WORKSPACE_TOO_SMALL", 4: "SSB_CUDA_ERROR"}

EXPORTED = ("ssb_bf_indices", "ssb_band_indices", "ssb_workspace_bytes", "ssb_build_G",
            "ssb_reconstruct", "ssb_score_batch", "ssb_last_error", "ssb_launch_count",
            "ssb_reconstruct_noalloc", "ssb_build_G_host", "ssb_build_G_host_bytes",
            "ssb_compact_G16", "ssb_compact_band", "ssb_reconstruct_g", "ssb_score_batch_g",
            "ssb_phase_moments", "ssb_reconstruct_sums", "ssb_phase_from_sums", "ssb_peak_sincos",
            "ssb_peak_fma", "ssb_score_batch_depth")

G_C64, G_SN16 = 0, 1

NOALLOC_SCRATCH_BYTES = 16 << 20


class Geometry(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int), ("det_y", ctypes.c_int), ("det_x", ctypes.c_int),
                ("scan_step_A", ctypes.c_double), ("det_pitch_invA", ctypes.c_double),
                ("wavelength_A", ctypes.c_double), ("semiangle_rad", ctypes.c_double),
                ("det_center_y", ctypes.c_double), ("det_center_x", ctypes.c_double)]


ABERR_FIELDS = ("C10", "C12a", "C12b", "C21a", "C21b", "C23a", "C23b", "C30", "C32a", "C32b",
                "C34a", "C34b", "tilt_x_rad", "tilt_y_rad")


class Aberr(ctypes.Structure):
    _fields_ = [(f, ctypes.c_double) for f in ABERR_FIELDS]


class GStoreC(ctypes.Structure):
    """ssb_gstore: a stored G as the reductions read it."""
    _fields_ = [("G", ctypes.c_void_p), ("fmt", ctypes.c_int), ("scale", ctypes.c_void_p),
                ("rows_per_scale", ctypes.c_int), ("band_compact", ctypes.c_int)]


class GStore:
    """Device tensors of a stored G: complex64 [n_bf, n, n/2+1] (fmt G_C64) or
    herm16 words int32 [n_bf, n, n/2+1] with float32 scales
    [n / rows_per_scale, n_bf] (fmt G_SN16); band_compact: the last two axes
    are one band axis [n_bf, nq] (made by compact_band)."""

    def __init__(self, G, fmt=G_C64, scale=None, rows_per_scale=0, band_compact=False):
        self.G, self.fmt, self.scale = G, fmt, scale
        self.rows_per_scale, self.band_compact = rows_per_scale, bool(band_compact)

    def c(self) -> GStoreC:
        return GStoreC(int(self.G.data_ptr()), self.fmt,
                       int(self.scale.data_ptr()) if self.scale is not None else 0,
                       self.rows_per_scale, 1 if self.band_compact else 0)


class SSBError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_lib = None


def load(path: str | None = None):
    """Load libssb.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build() "
                           "or python -m electron_microscopy_gb300._build")
    lib = ctypes.CDLL(p)
    c_int, c_size, c_vp, c_d = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_double
    G_p, A_p = ctypes.POINTER(Geometry), ctypes.POINTER(Aberr)
    i32p, ip = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int)
    lib.ssb_bf_indices.argtypes = [G_p, A_p, i32p, ip]
    lib.ssb_band_indices.argtypes = [G_p, c_d, c_d, i32p, ip]
    lib.ssb_workspace_bytes.argtypes = [G_p, c_int, c_int, c_int, c_int]
    lib.ssb_workspace_bytes.restype = c_size
    lib.ssb_build_G.argtypes = [c_vp, c_int, G_p, c_vp, c_int, c_vp, c_vp, c_size, c_vp]
    lib.ssb_build_G_host.argtypes = [c_vp, c_int, G_p, c_vp, c_vp, c_int, c_vp, c_vp, c_size, c_vp]
    lib.ssb_build_G_host_bytes.argtypes = [G_p, c_int, c_vp, c_int]
    lib.ssb_build_G_host_bytes.restype = c_size
    lib.ssb_reconstruct.argtypes = [c_vp, G_p, c_vp, c_int, A_p, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]
    lib.ssb_score_batch.argtypes = [c_vp, G_p, c_vp, c_int, A_p, c_int, c_vp, c_int, c_vp, c_vp, c_vp,
                                    c_vp, c_size, c_vp]
    lib.ssb_reconstruct_noalloc.argtypes = [c_vp, G_p, c_vp, c_int, A_p, c_vp, c_vp, c_vp, c_vp]
    S_p = ctypes.POINTER(GStoreC)
    lib.ssb_compact_G16.argtypes = [c_vp, G_p, c_int, c_int, c_vp, c_vp, c_vp]
    lib.ssb_compact_band.argtypes = [S_p, G_p, c_int, c_vp, c_int, c_vp, c_vp]
    lib.ssb_reconstruct_g.argtypes = [S_p, G_p, c_vp, c_int, A_p, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]
    lib.ssb_score_batch_g.argtypes = [S_p, G_p, c_vp, c_int, A_p, c_int, c_vp, c_int, c_vp, c_vp, c_vp,
                                      c_vp, c_size, c_vp]
    lib.ssb_phase_moments.argtypes = [S_p, G_p, c_vp, c_int, A_p, c_vp, c_vp, c_vp, c_size, c_vp]
    lib.ssb_reconstruct_sums.argtypes = [c_vp, G_p, c_vp, c_int, A_p, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]
    lib.ssb_phase_from_sums.argtypes = [c_vp, c_vp, c_vp, c_int, G_p, c_vp, c_vp, c_size, c_vp]
    lib.ssb_score_batch_depth.argtypes = [S_p, G_p, c_vp, c_int, A_p, ctypes.POINTER(c_d), c_int, c_vp, c_int,
                                          c_vp, c_vp, c_vp, c_vp, c_size, c_vp]
    lib.ssb_peak_sincos.argtypes = [c_vp, c_int, c_int, c_vp]
    lib.ssb_peak_fma.argtypes = [c_vp, c_int, c_int, c_vp]
    lib.ssb_last_error.restype = ctypes.c_char_p
    lib.ssb_launch_count.restype = ctypes.c_longlong
    for fn in ("ssb_bf_indices", "ssb_band_indices", "ssb_build_G", "ssb_build_G_host", "ssb_reconstruct",
               "ssb_score_batch", "ssb_reconstruct_noalloc", "ssb_compact_G16", "ssb_compact_band",
               "ssb_reconstruct_g", "ssb_score_batch_g", "ssb_phase_moments", "ssb_reconstruct_sums",
               "ssb_phase_from_sums", "ssb_peak_sincos", "ssb_peak_fma", "ssb_score_batch_depth"):
        getattr(lib, fn).restype = c_int
    _lib = lib
    return lib


def _check(fn, code):
    if code != SSB_OK:
        raise SSBError(fn, code, load().ssb_last_error().decode())


def to_geometry(g) -> Geometry:
    if isinstance(g, Geometry):
        return g
    return Geometry(*g.astuple())


def to_aberr(a) -> Aberr:
    if isinstance(a, Aberr):
        return a
    return Aberr(*a.astuple())


def _ptr(t):
    return ctypes.c_void_p(int(t.data_ptr())) if t is not None else ctypes.c_void_p(0)


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(int(s.cuda_stream))


# ----------------------------------------------------------------------------
# host-only entry points
# ----------------------------------------------------------------------------

def bf_indices(geom, base) -> np.ndarray:
    lib = load()
    g, a = to_geometry(geom), to_aberr(base)
    cnt = ctypes.c_int(0)
    _check("ssb_bf_indices", lib.ssb_bf_indices(ctypes.byref(g), ctypes.byref(a), None, ctypes.byref(cnt)))
    out = np.zeros(max(cnt.value, 1), dtype=np.int32)
    _check("ssb_bf_indices", lib.ssb_bf_indices(ctypes.byref(g), ctypes.byref(a),
                                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                                ctypes.byref(cnt)))
    return out[:cnt.value]


def band_indices(geom, qmin=0.2, qmax=0.9) -> np.ndarray:
    lib = load()
    g = to_geometry(geom)
    cnt = ctypes.c_int(0)
    _check("ssb_band_indices", lib.ssb_band_indices(ctypes.byref(g), qmin, qmax, None, ctypes.byref(cnt)))
    out = np.zeros(max(cnt.value, 1), dtype=np.int32)
    _check("ssb_band_indices", lib.ssb_band_indices(ctypes.byref(g), qmin, qmax,
                                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                                    ctypes.byref(cnt)))
    return out[:cnt.value]


def workspace_bytes(geom, n_bf, op, B=1, nq=1) -> int:
    return int(load().ssb_workspace_bytes(ctypes.byref(to_geometry(geom)), int(n_bf), int(op), int(B), int(nq)))


def launch_count() -> int:
    return int(load().ssb_launch_count())


# ----------------------------------------------------------------------------
# device entry points (torch tensors on the current CUDA device)
# ----------------------------------------------------------------------------

def _workspace(nbytes, device):
    import torch
    # 256 extra bytes so the pointer can be rounded up to a 256-byte boundary
    raw = torch.empty(int(nbytes) + 256, dtype=torch.uint8, device=device)
    off = (-int(raw.data_ptr())) % 256
    return raw, raw[off:off + int(nbytes)]


class Workspace:
    """A reusable device workspace (caller-owned scratch for the library)."""

    def __init__(self, nbytes, device="cuda"):
        self._raw, self.view = _workspace(max(int(nbytes), 256), device)
        self.nbytes = int(nbytes)

    def ptr(self):
        return _ptr(self.view)


def _dtype_code(frames):
    import torch
    if frames.dtype == torch.float32:
        return SSB_F32
    if frames.dtype in (torch.int16, torch.uint16 if hasattr(torch, "uint16") else torch.int16):
        return SSB_U16
    raise TypeError(f"frames must be float32 or 16-bit counts, got {frames.dtype}")


def build_G(frames, geom, bf_idx_dev, G=None, ws=None, stream=None):
    """G(q,k) half plane (complex64 [n_bf, n, n/2+1]) from device frames."""
    import torch
    lib = load()
    g = to_geometry(geom)
    n_bf = int(bf_idx_dev.numel())
    if not frames.is_cuda or not bf_idx_dev.is_cuda:
        raise ValueError("frames and bf_idx must be CUDA tensors")
    if not frames.is_contiguous():
        raise ValueError("frames must be contiguous")
    if G is None:
        G = torch.empty((n_bf, g.n, g.n // 2 + 1), dtype=torch.complex64, device=frames.device)
    need = workspace_bytes(g, n_bf, OP_BUILD)
    if ws is None:
        ws = Workspace(need, frames.device)
    _check("ssb_build_G", lib.ssb_build_G(_ptr(frames), _dtype_code(frames), ctypes.byref(g),
                                          _ptr(bf_idx_dev), n_bf, _ptr(G), ws.ptr(),
                                          ws.nbytes, _stream(stream)))
    return G


def build_G_host_bytes(geom, bf_idx_host, dtype) -> int:
    """Workspace bytes of build_G_host for this host index list (numpy int32)."""
    bf = np.ascontiguousarray(bf_idx_host, dtype=np.int32)
    return int(load().ssb_build_G_host_bytes(ctypes.byref(to_geometry(geom)), int(dtype),
                                             bf.ctypes.data_as(ctypes.c_void_p), int(bf.size)))


def build_G_host(frames_host, geom, bf_idx_host, bf_idx_dev, G=None, ws=None, stream=None):
    """G(q,k) from frames in host memory (a CPU tensor, pinned for full copy
    speed): only the bounding box of the bright-field pixels on the detector is copied.
    bf_idx_host (numpy int32) and bf_idx_dev hold the same indices.  The copy
    is asynchronous on `stream`: keep frames_host alive and unchanged until
    the stream has passed it."""
    import torch
    lib = load()
    g = to_geometry(geom)
    bf = np.ascontiguousarray(bf_idx_host, dtype=np.int32)
    n_bf = int(bf.size)
    if frames_host.is_cuda or not frames_host.is_contiguous():
        raise ValueError("frames_host must be a contiguous CPU tensor")
    if not bf_idx_dev.is_cuda or int(bf_idx_dev.numel()) != n_bf:
        raise ValueError("bf_idx_dev must be a CUDA tensor with the host list's length")
    dev = bf_idx_dev.device
    if G is None:
        G = torch.empty((n_bf, g.n, g.n // 2 + 1), dtype=torch.complex64, device=dev)
    dt = _dtype_code(frames_host)
    need = build_G_host_bytes(g, bf, dt)
    if ws is None:
        ws = Workspace(need, dev)
    _check("ssb_build_G_host", lib.ssb_build_G_host(
        ctypes.c_void_p(int(frames_host.data_ptr())), dt, ctypes.byref(g), bf.ctypes.data_as(ctypes.c_void_p),
        _ptr(bf_idx_dev), n_bf, _ptr(G), ws.ptr(), ws.nbytes, _stream(stream)))
    return G


def reconstruct(G, geom, bf_idx_dev, aberr, O=None, N=None, phase=None, ws=None, stream=None):
    """One reconstruction: returns (O complex64 [n, n/2+1], N int32 [n, n/2+1],
    phase float32 [n, n])."""
    import torch
    lib = load()
    g = to_geometry(geom)
    a = to_aberr(aberr)
    n_bf = int(bf_idx_dev.numel())
    n, h = g.n, g.n // 2 + 1
    dev = G.device
    O = torch.empty((n, h), dtype=torch.complex64, device=dev) if O is None else O
    N = torch.empty((n, h), dtype=torch.int32, device=dev) if N is None else N
    phase = torch.empty((n, n), dtype=torch.float32, device=dev) if phase is None else phase
    if ws is None:
        ws = Workspace(workspace_bytes(g, n_bf, OP_RECON), dev)
    _check("ssb_reconstruct", lib.ssb_reconstruct(_ptr(G), ctypes.byref(g), _ptr(bf_idx_dev), n_bf,
                                                  ctypes.byref(a), _ptr(O), _ptr(N), _ptr(phase),
                                                  ws.ptr(), ws.nbytes, _stream(stream)))
    return O, N, phase


def reconstruct_sums(G, geom, bf_idx_dev, aberr, O=None, N=None, g0_sum=None, ws=None, stream=None):
    """One shard of a reconstruction: the raw sums (O complex64 [n, n/2+1],
    N int32 [n, n/2+1]) over this shard's BF pixels and sum_k Re G(0,k)
    (float64 [1]).  Add the shards' results, then call phase_from_sums."""
    import torch
    lib = load()
    g = to_geometry(geom)
    a = to_aberr(aberr)
    n_bf = int(bf_idx_dev.numel())
    n, h = g.n, g.n // 2 + 1
    dev = G.device
    O = torch.empty((n, h), dtype=torch.complex64, device=dev) if O is None else O
    N = torch.empty((n, h), dtype=torch.int32, device=dev) if N is None else N
    g0_sum = torch.empty((1,), dtype=torch.float64, device=dev) if g0_sum is None else g0_sum
    if ws is None:
        ws = Workspace(workspace_bytes(g, n_bf, OP_RECON), dev)
    _check("ssb_reconstruct_sums", lib.ssb_reconstruct_sums(
        _ptr(G), ctypes.byref(g), _ptr(bf_idx_dev), n_bf, ctypes.byref(a), _ptr(O), _ptr(N), _ptr(g0_sum),
        ws.ptr(), ws.nbytes, _stream(stream)))
    return O, N, g0_sum


def phase_from_sums(O, N, g0_sum, n_bf_total, geom, phase=None, ws=None, stream=None):
    """Phase image (float32 [n, n]) from summed shard results."""
    import torch
    lib = load()
    g = to_geometry(geom)
    dev = O.device
    phase = torch.empty((g.n, g.n), dtype=torch.float32, device=dev) if phase is None else phase
    if ws is None:
        ws = Workspace(workspace_bytes(g, 1, OP_PHASE), dev)
    _check("ssb_phase_from_sums", lib.ssb_phase_from_sums(
        _ptr(O), _ptr(N), _ptr(g0_sum), int(n_bf_total), ctypes.byref(g), _ptr(phase), ws.ptr(), ws.nbytes,
        _stream(stream)))
    return phase


def peak_rates(device=None, iters=(4096, 32768), stream=None):
    """Measured rates on the current device: transcendental results per second
    (one __sincosf = 2) and float32 flops per second (FMA = 2), from the
    library's probe kernels timed with CUDA events on `stream`."""
    import torch
    lib = load()
    dev = torch.device("cuda") if device is None else device
    props = torch.cuda.get_device_properties(dev)
    blocks = props.multi_processor_count * 8
    out = torch.zeros(1, dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream(dev) if stream is None else stream
    res = {}
    for (name, fn), it in zip((("sincos_per_s", lib.ssb_peak_sincos), ("fma_flops_per_s", lib.ssb_peak_fma)),
                              iters):
        for _ in range(2):  # warm-up
            _check(fn.__name__, fn(_ptr(out), blocks, it, _stream(st)))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        _check(fn.__name__, fn(_ptr(out), blocks, it, _stream(st)))
        e1.record(st)
        e1.synchronize()
        res[name] = 2.0 * 8 * 256 * blocks * it / (e0.elapsed_time(e1) * 1e-3)
    res["blocks"], res["iters"] = blocks, list(iters)
    return res


def score_batch(G, geom, bf_idx_dev, sets, band_dev, O=None, N=None, score=None, ws=None, stream=None):
    """Batched scoring of B <= 8 sets over a band list: returns
    (O complex64 [B, nq], N int32 [B, nq], score float64 [B])."""
    import torch
    lib = load()
    g = to_geometry(geom)
    B = len(sets)
    arr = (Aberr * max(B, 1))(*[to_aberr(s) for s in sets])
    n_bf = int(bf_idx_dev.numel())
    nq = int(band_dev.numel())
    dev = G.device
    O = torch.empty((B, nq), dtype=torch.complex64, device=dev) if O is None else O
    N = torch.empty((B, nq), dtype=torch.int32, device=dev) if N is None else N
    score = torch.empty((B,), dtype=torch.float64, device=dev) if score is None else score
    if ws is None:
        need = workspace_bytes(g, n_bf, OP_SCORE, B, nq)
        if need == 0:
            raise SSBError("ssb_workspace_bytes", SSB_INVALID_ARG, f"invalid sizes (B={B}, nq={nq})")
        ws = Workspace(need, dev)
    _check("ssb_score_batch", lib.ssb_score_batch(_ptr(G), ctypes.byref(g), _ptr(bf_idx_dev), n_bf, arr, B,
                                                  _ptr(band_dev), nq, _ptr(O), _ptr(N), _ptr(score),
                                                  ws.ptr(), ws.nbytes, _stream(stream)))
    return O, N, score


def reconstruct_noalloc(G, geom, bf_idx_dev, aberr, O=None, N=None, phase=None, stream=None):
    """ssb_reconstruct_noalloc: the reconstruction with the library's fixed
    scratch array instead of a workspace (for callers that cannot allocate
    device memory; the output tensors are created here only if not given)."""
    import torch
    lib = load()
    g = to_geometry(geom)
    a = to_aberr(aberr)
    n_bf = int(bf_idx_dev.numel())
    n, h = g.n, g.n // 2 + 1
    dev = G.device
    O = torch.empty((n, h), dtype=torch.complex64, device=dev) if O is None else O
    N = torch.empty((n, h), dtype=torch.int32, device=dev) if N is None else N
    phase = torch.empty((n, n), dtype=torch.float32, device=dev) if phase is None else phase
    _check("ssb_reconstruct_noalloc", lib.ssb_reconstruct_noalloc(
        _ptr(G), ctypes.byref(g), _ptr(bf_idx_dev), n_bf, ctypes.byref(a), _ptr(O), _ptr(N), _ptr(phase),
        _stream(stream)))
    return O, N, phase


# ----------------------------------------------------------------------------
# compact storage of G
# ----------------------------------------------------------------------------

def compact_G16(G, geom, rows_per_scale, G16=None, scale=None, stream=None) -> GStore:
    """herm16 of a complex64 G [n_bf, n, n/2+1]: int32 words (real code in the
    low 16 bits) and float32 scales [n / rows_per_scale, n_bf]; rows_per_scale
    is n (one scale per BF pixel) or 1 (one per q row)."""
    import torch
    lib = load()
    g = to_geometry(geom)
    n_bf = int(G.shape[0])
    dev = G.device
    G16 = torch.empty(G.shape, dtype=torch.int32, device=dev) if G16 is None else G16
    nblk = g.n // rows_per_scale if rows_per_scale in (1, g.n) else 1
    scale = torch.empty((nblk, n_bf), dtype=torch.float32, device=dev) if scale is None else scale
    _check("ssb_compact_G16", lib.ssb_compact_G16(_ptr(G), ctypes.byref(g), n_bf, rows_per_scale, _ptr(G16),
                                                  _ptr(scale), _stream(stream)))
    return GStore(G16, G_SN16, scale, rows_per_scale)


def compact_band(src, geom, band_dev, dst=None, stream=None) -> GStore:
    """Band-compacted copy [n_bf, nq] of a half-plane G (a GStore or a complex64
    tensor); a herm16 copy keeps the source's scales."""
    import torch
    lib = load()
    if not isinstance(src, GStore):
        src = GStore(src)
    g = to_geometry(geom)
    n_bf = int(src.G.shape[0])
    nq = int(band_dev.numel())
    if dst is None:
        dst = torch.empty((n_bf, nq), dtype=src.G.dtype, device=src.G.device)
    sc = src.c()
    _check("ssb_compact_band", lib.ssb_compact_band(ctypes.byref(sc), ctypes.byref(g), n_bf, _ptr(band_dev), nq,
                                                    _ptr(dst), _stream(stream)))
    return GStore(dst, src.fmt, src.scale, src.rows_per_scale, band_compact=True)


def reconstruct_g(store, geom, bf_idx_dev, aberr, O=None, N=None, phase=None, ws=None, stream=None):
    """reconstruct() from a GStore (half plane, either format)."""
    import torch
    lib = load()
    g = to_geometry(geom)
    a = to_aberr(aberr)
    n_bf = int(bf_idx_dev.numel())
    n, h = g.n, g.n // 2 + 1
    dev = store.G.device
    O = torch.empty((n, h), dtype=torch.complex64, device=dev) if O is None else O
    N = torch.empty((n, h), dtype=torch.int32, device=dev) if N is None else N
    phase = torch.empty((n, n), dtype=torch.float32, device=dev) if phase is None else phase
    if ws is None:
        ws = Workspace(workspace_bytes(g, n_bf, OP_RECON), dev)
    sc = store.c()
    _check("ssb_reconstruct_g", lib.ssb_reconstruct_g(ctypes.byref(sc), ctypes.byref(g), _ptr(bf_idx_dev), n_bf,
                                                      ctypes.byref(a), _ptr(O), _ptr(N), _ptr(phase),
                                                      ws.ptr(), ws.nbytes, _stream(stream)))
    return O, N, phase


def score_batch_g(store, geom, bf_idx_dev, sets, band_dev, O=None, N=None, score=None, ws=None, stream=None):
    """score_batch() from a GStore (half plane or band copy, either format)."""
    import torch
    lib = load()
    g = to_geometry(geom)
    B = len(sets)
    arr = (Aberr * max(B, 1))(*[to_aberr(s) for s in sets])
    n_bf = int(bf_idx_dev.numel())
    nq = int(band_dev.numel())
    dev = store.G.device
    O = torch.empty((B, nq), dtype=torch.complex64, device=dev) if O is None else O
    N = torch.empty((B, nq), dtype=torch.int32, device=dev) if N is None else N
    score = torch.empty((B,), dtype=torch.float64, device=dev) if score is None else score
    if ws is None:
        need = workspace_bytes(g, n_bf, OP_SCORE, B, nq)
        if need == 0:
            raise SSBError("ssb_workspace_bytes", SSB_INVALID_ARG, f"invalid sizes (B={B}, nq={nq})")
        ws = Workspace(need, dev)
    sc = store.c()
    _check("ssb_score_batch_g", lib.ssb_score_batch_g(ctypes.byref(sc), ctypes.byref(g), _ptr(bf_idx_dev), n_bf,
                                                      arr, B, _ptr(band_dev), nq, _ptr(O), _ptr(N), _ptr(score),
                                                      ws.ptr(), ws.nbytes, _stream(stream)))
    return O, N, score


def score_batch_depth(store, geom, bf_idx_dev, sets, depth_A, band_dev, O=None, N=None, score=None, ws=None,
                      stream=None):
    """score_batch_g() with a defocus spread per set (depth_A: B thicknesses in
    Angstrom, each >= 0): every trotter term is weighted by the depth-0 weight
    times sinc(pi lambda t D / 2).  `store` may be a GStore or a complex64
    half-plane tensor."""
    import torch
    lib = load()
    if not isinstance(store, GStore):
        store = GStore(store)
    g = to_geometry(geom)
    B = len(sets)
    if len(depth_A) != B:
        raise ValueError("depth_A needs one value per set")
    arr = (Aberr * max(B, 1))(*[to_aberr(s) for s in sets])
    dep = (ctypes.c_double * max(B, 1))(*[float(t) for t in depth_A])
    n_bf = int(bf_idx_dev.numel())
    nq = int(band_dev.numel())
    dev = store.G.device
    O = torch.empty((B, nq), dtype=torch.complex64, device=dev) if O is None else O
    N = torch.empty((B, nq), dtype=torch.int32, device=dev) if N is None else N
    score = torch.empty((B,), dtype=torch.float64, device=dev) if score is None else score
    if ws is None:
        need = workspace_bytes(g, n_bf, OP_SCORE, B, nq)
        if need == 0:
            raise SSBError("ssb_workspace_bytes", SSB_INVALID_ARG, f"invalid sizes (B={B}, nq={nq})")
        ws = Workspace(need, dev)
    sc = store.c()
    _check("ssb_score_batch_depth", lib.ssb_score_batch_depth(
        ctypes.byref(sc), ctypes.byref(g), _ptr(bf_idx_dev), n_bf, arr, dep, B, _ptr(band_dev), nq, _ptr(O),
        _ptr(N), _ptr(score), ws.ptr(), ws.nbytes, _stream(stream)))
    return O, N, score


def phase_moments(store, geom, bf_idx_dev, aberr, mean=None, var=None, ws=None, stream=None):
    """Per-BF phase moments: (mean, var) float32 [n, n] over BF pixels of
    atan2(b_k, a_k); store: a GStore or a complex64 half-plane G."""
    import torch
    lib = load()
    if not isinstance(store, GStore):
        store = GStore(store)
    g = to_geometry(geom)
    a = to_aberr(aberr)
    n_bf = int(bf_idx_dev.numel())
    dev = store.G.device
    mean = torch.empty((g.n, g.n), dtype=torch.float32, device=dev) if mean is None else mean
    var = torch.empty((g.n, g.n), dtype=torch.float32, device=dev) if var is None else var
    if ws is None:
        ws = Workspace(workspace_bytes(g, n_bf, OP_MOMENTS), dev)
    sc = store.c()
    _check("ssb_phase_moments", lib.ssb_phase_moments(ctypes.byref(sc), ctypes.byref(g), _ptr(bf_idx_dev), n_bf,
                                                      ctypes.byref(a), _ptr(mean), _ptr(var), ws.ptr(), ws.nbytes,
                                                      _stream(stream)))
    return mean, var
