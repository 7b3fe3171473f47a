// api.cu -- the C ABI declared in include/ssb.h: argument checks, host-side
// index sets, workspace layout and the launch sequence of each operation.
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.cuh"

namespace ssb {

static thread_local char g_err[512] = "";
static std::atomic<long long> g_launches{0};

void count_launch(int k) { g_launches.fetch_add(k, std::memory_order_relaxed); }

static int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
static int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

static int cuda_fail(cudaError_t e, const char* where) {
    return fail(SSB_CUDA_ERROR, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

int set_last_error(int code, const char* msg, cudaError_t err) {
    if (err != cudaSuccess) return fail(code, "%s: %s (%s)", msg, cudaGetErrorName(err), cudaGetErrorString(err));
    return fail(code, "%s", msg);
}

// IEEE double product with its own rounding, whatever the host compiler's
// contraction settings (the BF predicate must match a plain float64 reading).
static double mul_rn(double a, double b) {
    volatile double r = a * b;
    return r;
}

static bool is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

static int check_geom(const ssb_geometry* g) {
    if (!g) return fail(SSB_INVALID_ARG, "geometry is NULL");
    if (g->det_y < 1 || g->det_x < 1) return fail(SSB_INVALID_ARG, "detector size must be >= 1");
    if ((long long)g->det_y * g->det_x > (1LL << 30))
        return fail(SSB_INVALID_ARG, "detector too large");
    if (!(g->scan_step_A > 0) || !(g->det_pitch_invA > 0) || !(g->wavelength_A > 0) ||
        !(g->semiangle_rad > 0))
        return fail(SSB_INVALID_ARG, "scan step, detector pitch, wavelength and semi-angle must be > 0");
    if (!std::isfinite(g->det_center_x) || !std::isfinite(g->det_center_y))
        return fail(SSB_INVALID_ARG, "detector centre must be finite");
    if (!is_pow2(g->n) || g->n < SSB_MIN_N || g->n > SSB_MAX_N)
        return fail(SSB_UNSUPPORTED, "scan size n=%d must be a power of two in [%d, %d]", g->n, SSB_MIN_N,
                    SSB_MAX_N);
    return SSB_OK;
}

static int check_set(const ssb_aberr* a) {
    const double* v = &a->C10;
    for (int i = 0; i < 14; ++i)
        if (!std::isfinite(v[i])) return fail(SSB_INVALID_ARG, "aberration value %d is not finite", i);
    return SSB_OK;
}

// float32 constants of one aberration set (chi in turns, see internal.cuh)
static SetParams set_params(const ssb_geometry* g, const ssb_aberr* a) {
    const double lam = g->wavelength_A, l2 = lam * lam, l3 = l2 * lam;
    SetParams p;
    p.tx = (float)(a->tilt_x_rad / lam);
    p.ty = (float)(a->tilt_y_rad / lam);
    p.c[0] = (float)(lam * a->C10 / 2.0);
    p.c[1] = (float)(lam * a->C12a / 2.0);
    p.c[2] = (float)(lam * a->C12b);
    p.c[3] = (float)(l2 * a->C21a / 3.0);
    p.c[4] = (float)(l2 * a->C21b / 3.0);
    p.c[5] = (float)(l2 * a->C23a / 3.0);
    p.c[6] = (float)(l2 * a->C23b / 3.0);
    p.c[7] = (float)(l3 * a->C30 / 4.0);
    p.c[8] = (float)(l3 * a->C32a / 4.0);
    p.c[9] = (float)(l3 * a->C32b / 2.0);
    p.c[10] = (float)(l3 * a->C34a / 4.0);
    p.c[11] = (float)(l3 * a->C34b);
    // the quartic-in-vx regrouping, combined in double and rounded once
    const double d[12] = {lam * a->C10 / 2.0,  lam * a->C12a / 2.0, lam * a->C12b,       l2 * a->C21a / 3.0,
                          l2 * a->C21b / 3.0,  l2 * a->C23a / 3.0,  l2 * a->C23b / 3.0,  l3 * a->C30 / 4.0,
                          l3 * a->C32a / 4.0,  l3 * a->C32b / 2.0,  l3 * a->C34a / 4.0,  l3 * a->C34b};
    p.h[0] = (float)(d[7] + d[8] + d[10]);
    p.h[1] = (float)(d[3] + d[5]);
    p.h[2] = (float)(d[9] + d[11]);
    p.h[3] = (float)(d[0] + d[1]);
    p.h[4] = (float)(d[4] + 3.0 * d[6]);
    p.h[5] = (float)(2.0 * d[7] - 6.0 * d[10]);
    p.h[6] = (float)d[2];
    p.h[7] = (float)(d[3] - 3.0 * d[5]);
    p.h[8] = (float)(d[9] - d[11]);
    p.h[9] = (float)(d[0] - d[1]);
    p.h[10] = (float)(d[4] - d[6]);
    p.h[11] = (float)(d[7] - d[8] + d[10]);
    return p;
}

static float aperture_r2(const ssb_geometry* g) {
    const double r = g->semiangle_rad / g->wavelength_A;
    return (float)mul_rn(r, r);
}

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Number of k-splits of the reduction.  The grid is (nq / 256) x splits CTAs
// of equal length; a wave is 152 SMs x 4 resident CTAs, and a partly filled
// last wave takes about as long as a full one, so the count is the smallest
// one (from two waves up) whose CTAs fill at least 97 % of their waves, else
// the best filling one; at most 64 splits and about 16 k per split.  Depends
// only on (nq, n_bf), so that the summation order is the same for every B.
static int red_splits(int nq, int n_bf) {
    const long bx = (nq + 255) / 256, wave = 152 * 4;
    int max_s = (n_bf + 15) / 16;
    if (max_s > 64) max_s = 64;
    if (max_s < 1) max_s = 1;
    int lo = (int)((2 * wave + bx - 1) / bx);
    if (lo > max_s) lo = max_s;
    if (lo < 1) lo = 1;
    auto fill = [&](int s) {
        const long ctas = bx * s, waves = (ctas + wave - 1) / wave;
        return (double)ctas / (double)(waves * wave);
    };
    int best = lo;
    for (int s = lo; s <= max_s; ++s) {
        if (fill(s) >= 0.97) return s;
        if (fill(s) > fill(best)) best = s;
    }
    return best;
}

struct WsLayout {
    size_t tw, xbuf, ktab, chik, kxcol, status, Opart, Npart, dcpart, Y, total;
};

static WsLayout layout(const ssb_geometry* g, int n_bf, int op, int B, int nq) {
    WsLayout L{};
    const int n = g->n, H = n / 2 + 1;
    size_t off = 0;
    L.tw = off;
    off += align256((size_t)n * sizeof(float2));
    if (op == SSB_OP_BUILD) {
        if (n == 512) {  // chunk buffers of the cluster build
            L.xbuf = off;
            off += align256(plane512_chunk_bytes());
        }
        L.total = off;
        return L;
    }
    if (op == SSB_OP_PHASE) {  // the complex-to-real intermediate
        L.Y = off;
        off += align256((size_t)n * H * sizeof(float2));
        L.total = off;
        return L;
    }
    if (op == SSB_OP_MOMENTS) {
        L.ktab = off;
        off += align256((size_t)n_bf * sizeof(float4));
        L.chik = off;
        off += align256((size_t)n_bf * kChiStride * sizeof(float));
        L.Y = off;
        off += align256(moments_chunk_bytes(n));
        L.Opart = off;  // the moment partial sums
        off += align256(moments_part_bytes(n));
        L.total = off;
        return L;
    }
    if (op == SSB_OP_RECON) {
        B = 1;
        nq = n * H;
    }
    const int ns = red_splits(nq, n_bf);
    L.ktab = off;
    off += align256((size_t)n_bf * sizeof(float4));
    L.chik = off;
    off += align256((size_t)n_bf * kChiStride * sizeof(float));
    L.kxcol = off;
    off += align256((size_t)g->det_x * sizeof(float));
    L.status = off;
    off += align256(sizeof(int));
    L.Opart = off;
    off += align256((size_t)ns * B * nq * sizeof(float2));
    L.Npart = off;
    off += align256((size_t)ns * B * nq * sizeof(int));
    L.dcpart = off;
    off += align256((size_t)((n_bf + 255) / 256) * sizeof(double));
    if (op == SSB_OP_RECON) {
        L.Y = off;
        off += align256((size_t)n * H * sizeof(float2));
    }
    L.total = off;
    return L;
}

template <typename T>
static T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

static int check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (!ws) return fail(SSB_INVALID_ARG, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(SSB_INVALID_ARG, "workspace must be 256-byte aligned");
    if (ws_bytes < need)
        return fail(SSB_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes, need);
    return SSB_OK;
}

// shared by reconstruct and score: k tables, reduction, finalize
// the reductions' view of a stored G (checked); nq: band length of a
// band-compacted copy
static int gview_of(const ssb_gstore* s, const ssb_geometry* g, int nq, GView* v) {
    if (!s || !s->G) return fail(SSB_INVALID_ARG, "G store or its G pointer is NULL");
    if (s->fmt != SSB_G_C64 && s->fmt != SSB_G_SN16) return fail(SSB_INVALID_ARG, "unknown G format %d", s->fmt);
    if (s->fmt == SSB_G_SN16) {
        if (!s->scale) return fail(SSB_INVALID_ARG, "a herm16 G needs its scale array");
        if (s->rows_per_scale != 1 && s->rows_per_scale != g->n)
            return fail(SSB_UNSUPPORTED, "rows_per_scale=%d must be 1 or n=%d", s->rows_per_scale, g->n);
    }
    v->G = s->G;
    v->fmt = s->fmt;
    v->band = s->band_compact ? 1 : 0;
    v->stride = s->band_compact ? (size_t)nq : (size_t)g->n * (g->n / 2 + 1);
    v->scale = s->fmt == SSB_G_SN16 ? s->scale : nullptr;
    v->srows = s->fmt == SSB_G_SN16 ? s->rows_per_scale : g->n;
    return SSB_OK;
}

static int run_reduction(const GView& gv, const ssb_geometry* g, const int32_t* bf_idx, int n_bf,
                         const SetBatch& sb, const int32_t* qlist, int nq, float2* O, int32_t* N,
                         void* ws, const WsLayout& Lw, int want_dc, cudaStream_t st, int depth = 0) {
    cudaError_t e;
    float4* ktab = at<float4>(ws, Lw.ktab);
    float* chik = at<float>(ws, Lw.chik);
    float* kxcol = at<float>(ws, Lw.kxcol);
    if ((e = launch_prep(bf_idx, n_bf, g->det_x, g->det_center_y, g->det_center_x, g->det_pitch_invA, sb,
                         ktab, chik, kxcol, at<int>(ws, Lw.status), gv, want_dc ? at<double>(ws, Lw.dcpart) : nullptr,
                         st)) != cudaSuccess)
        return cuda_fail(e, "prep");
    RedLaunch P{};
    P.g = gv;
    P.n = g->n;
    P.n_bf = n_bf;
    P.nq = nq;
    P.nsplit = red_splits(nq, n_bf);
    P.kps = (n_bf + P.nsplit - 1) / P.nsplit;
    P.dq = 1.0 / ((double)g->n * g->scan_step_A);
    P.qlist = qlist;
    P.ktab = ktab;
    P.chik = chik;
    P.kxcol = kxcol;
    P.status = at<int>(ws, Lw.status);
    P.ncol = g->det_x;
    P.inv_dk = (float)(1.0 / g->det_pitch_invA);
    P.ccol = (float)g->det_center_x;
    P.shared_tilt = 1;
    P.depth = depth;
    for (int s = 1; s < sb.B; ++s)
        if (sb.s[s].tx != sb.s[0].tx || sb.s[s].ty != sb.s[0].ty) P.shared_tilt = 0;
    P.Opart = at<float2>(ws, Lw.Opart);
    P.Npart = at<int>(ws, Lw.Npart);
    if ((e = launch_reduce(P, sb, st)) != cudaSuccess) return cuda_fail(e, "reduce");
    if ((e = launch_finalize(P.Opart, P.Npart, P.nsplit, sb.B, nq, P.status, O, N, st)) != cudaSuccess)
        return cuda_fail(e, "finalize");
    return SSB_OK;
}

}  // namespace ssb

using namespace ssb;

extern "C" {

const char* ssb_last_error(void) { return g_err; }

long long ssb_launch_count(void) { return g_launches.load(); }

int ssb_bf_indices(const ssb_geometry* geom, const ssb_aberr* base, int32_t* out, int* n_bf) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    if (!base || !n_bf) return fail(SSB_INVALID_ARG, "base set and n_bf must not be NULL");
    if ((rc = check_set(base)) != SSB_OK) return rc;
    const double lam = geom->wavelength_A, dk = geom->det_pitch_invA;
    const double r = geom->semiangle_rad / lam;
    const double r2 = mul_rn(r, r);
    const double tkx = base->tilt_x_rad / lam, tky = base->tilt_y_rad / lam;
    int count = 0;
    for (int i = 0; i < geom->det_y; ++i) {
        const double ey = mul_rn((double)i - geom->det_center_y, dk) - tky;
        for (int j = 0; j < geom->det_x; ++j) {
            const double ex = mul_rn((double)j - geom->det_center_x, dk) - tkx;
            if (mul_rn(ex, ex) + mul_rn(ey, ey) <= r2) {
                if (out) out[count] = i * geom->det_x + j;
                ++count;
            }
        }
    }
    *n_bf = count;
    g_err[0] = 0;
    return SSB_OK;
}

int ssb_band_indices(const ssb_geometry* geom, double qmin, double qmax, int32_t* out, int* nq) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    if (!nq) return fail(SSB_INVALID_ARG, "nq must not be NULL");
    if (!(qmin >= 0) || !(qmax >= qmin)) return fail(SSB_INVALID_ARG, "need 0 <= qmin <= qmax");
    const int n = geom->n, H = n / 2 + 1;
    const double dq = 1.0 / ((double)n * geom->scan_step_A);
    const double lo = mul_rn(qmin / dq, qmin / dq);
    const double hi = mul_rn(qmax / dq, qmax / dq);
    int count = 0;
    for (int row = 0; row < n; ++row) {
        const long long fy = row < n / 2 ? row : row - n;
        for (int col = 0; col < H; ++col) {
            const double r2 = (double)(fy * fy + (long long)col * col);
            if (r2 >= lo && r2 <= hi) {
                if (out) out[count] = row * H + col;
                ++count;
            }
        }
    }
    *nq = count;
    g_err[0] = 0;
    return SSB_OK;
}

size_t ssb_workspace_bytes(const ssb_geometry* geom, int n_bf, int op, int B, int nq) {
    if (check_geom(geom) != SSB_OK) return 0;
    if (n_bf < 1) return 0;
    if (op == SSB_OP_SCORE && (B < 1 || B > SSB_MAX_SETS || nq < 1)) return 0;
    if (op != SSB_OP_BUILD && op != SSB_OP_RECON && op != SSB_OP_SCORE && op != SSB_OP_MOMENTS &&
        op != SSB_OP_PHASE)
        return 0;
    return layout(geom, n_bf, op, B, nq).total;
}

int ssb_build_G(const void* frames, int dtype, const ssb_geometry* geom, const int32_t* bf_idx_dev,
                int n_bf, void* G_dev, void* ws, size_t ws_bytes, void* stream) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    if (!frames || !bf_idx_dev || !G_dev) return fail(SSB_INVALID_ARG, "frames, bf_idx and G must not be NULL");
    if (dtype != SSB_U16 && dtype != SSB_F32) return fail(SSB_INVALID_ARG, "dtype must be SSB_U16 or SSB_F32");
    if (n_bf < 1 || (long long)n_bf > (long long)geom->det_y * geom->det_x)
        return fail(SSB_INVALID_ARG, "n_bf=%d out of range", n_bf);
    const WsLayout Lw = layout(geom, n_bf, SSB_OP_BUILD, 1, 1);
    if ((rc = check_ws(ws, ws_bytes, Lw.total)) != SSB_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float2* tw = at<float2>(ws, Lw.tw);
    cudaError_t e;
    if ((e = launch_twiddles(tw, geom->n, st)) != cudaSuccess) return cuda_fail(e, "twiddles");
    if (geom->n == 512 && dtype == SSB_U16 && plane512_cluster_size() > 0)
        e = launch_build512(static_cast<const uint16_t*>(frames), geom->det_y * geom->det_x, bf_idx_dev, n_bf,
                            static_cast<float2*>(G_dev), tw, at<void>(ws, Lw.xbuf), st);
    else
        e = launch_build(frames, dtype, geom->n, geom->det_y * geom->det_x, bf_idx_dev, n_bf,
                         static_cast<float2*>(G_dev), tw, st);
    if (e != cudaSuccess) return cuda_fail(e, "build");
    g_err[0] = 0;
    return SSB_OK;
}

// ssb_build_G_host: the bounding box of the bright-field pixels on the
// detector (rows r0.., columns c0..), staged in the workspace ahead of the
// build workspace
struct HostLayout {
    int r0 = 0, rows = 0, c0 = 0, cols = 0, pitch = 0;
    size_t crop = 0, idx = 0, build = 0, total = 0;
};

static int host_layout(const ssb_geometry* geom, int dtype, const int32_t* bf_host, int n_bf, HostLayout* H) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    if (dtype != SSB_U16 && dtype != SSB_F32) return fail(SSB_INVALID_ARG, "dtype must be SSB_U16 or SSB_F32");
    if (!bf_host) return fail(SSB_INVALID_ARG, "bf_idx_host must not be NULL");
    const long long det_pix = (long long)geom->det_y * geom->det_x;
    if (n_bf < 1 || n_bf > det_pix) return fail(SSB_INVALID_ARG, "n_bf=%d out of range", n_bf);
    int rlo = geom->det_y, rhi = -1, clo = geom->det_x, chi = -1;
    for (int i = 0; i < n_bf; ++i) {
        const int v = bf_host[i];
        if (v < 0 || v >= det_pix) return fail(SSB_INVALID_ARG, "bf_idx_host[%d]=%d outside the detector", i, v);
        const int r = v / geom->det_x, c = v - r * geom->det_x;
        rlo = r < rlo ? r : rlo;
        rhi = r > rhi ? r : rhi;
        clo = c < clo ? c : clo;
        chi = c > chi ? c : chi;
    }
    // the box starts on an even column (kept so that any build that pairs
    // the two pixels of a 4-byte detector word sees the same words)
    if (chi - clo + 1 < geom->det_x) clo &= ~1;
    ssb_geometry crop = *geom;
    crop.det_y = rhi - rlo + 1;
    const size_t es = dtype == SSB_U16 ? 2 : 4;
    H->r0 = rlo;
    H->rows = crop.det_y;
    H->c0 = clo;
    H->cols = chi - clo + 1;
    // staged rows are padded to a multiple of 16 bytes (whole detector rows
    // are copied unpadded), so the build can read them in 16-byte pieces
    H->pitch = H->cols == geom->det_x ? geom->det_x : (int)(((size_t)H->cols * es + 15) / 16 * 16 / es);
    crop.det_x = H->pitch;
    H->crop = 0;
    H->idx = align256((size_t)geom->n * geom->n * crop.det_y * crop.det_x * es);
    H->build = H->idx + align256((size_t)n_bf * sizeof(int32_t));
    H->total = H->build + layout(&crop, n_bf, SSB_OP_BUILD, 1, 1).total;
    return SSB_OK;
}

// One library-internal stream per device carries the host-to-device copies of
// every ssb_build_G_host call, forked from and joined to the caller's stream
// with events.  Successive calls' copies queue behind one another whatever
// stream they come from, so a pipeline of calls on two caller streams keeps
// the host link busy while the previous scan is built, instead of copying on
// both streams at once and then computing on both.  The record/wait pairs are
// issued under the device's mutex, so one event of each kind suffices.
struct HostCopyStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex mu;
    bool ready = false;
};

static cudaError_t host_copy_stream(HostCopyStream** out) {
    static HostCopyStream per_dev[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    HostCopyStream& h = per_dev[dev];
    std::lock_guard<std::mutex> lock(h.mu);
    if (!h.ready) {
        if ((e = cudaStreamCreateWithFlags(&h.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&h.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&h.join, cudaEventDisableTiming)) != cudaSuccess) return e;
        h.ready = true;
    }
    *out = &h;
    return cudaSuccess;
}

size_t ssb_build_G_host_bytes(const ssb_geometry* geom, int dtype, const int32_t* bf_idx_host, int n_bf) {
    HostLayout H;
    if (host_layout(geom, dtype, bf_idx_host, n_bf, &H) != SSB_OK) return 0;
    return H.total;
}

int ssb_build_G_host(const void* frames_host, int dtype, const ssb_geometry* geom, const int32_t* bf_idx_host,
                     const int32_t* bf_idx_dev, int n_bf, void* G_dev, void* ws, size_t ws_bytes, void* stream) {
    int rc;
    HostLayout H;
    if ((rc = host_layout(geom, dtype, bf_idx_host, n_bf, &H)) != SSB_OK) return rc;
    if (!frames_host || !bf_idx_dev || !G_dev) return fail(SSB_INVALID_ARG, "frames, bf_idx and G must not be NULL");
    if ((rc = check_ws(ws, ws_bytes, H.total)) != SSB_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t es = dtype == SSB_U16 ? 2 : 4;
    const size_t row_bytes = (size_t)geom->det_x * es;
    cudaError_t e;
    HostCopyStream* hc = nullptr;
    if ((e = host_copy_stream(&hc)) != cudaSuccess) return cuda_fail(e, "host copy stream");
    std::lock_guard<std::mutex> lock(hc->mu);
    // the copy starts once the caller's earlier work (which may still read the
    // staging area) is done, and after the previous call's copy
    if ((e = cudaEventRecord(hc->fork, st)) != cudaSuccess || (e = cudaStreamWaitEvent(hc->s, hc->fork, 0)) != cudaSuccess)
        return cuda_fail(e, "host copy fork");
    if (H.cols == geom->det_x) {
        // whole detector rows: one pitched 2D copy, one row of r1 - r0 + 1 detector rows per frame
        e = cudaMemcpy2DAsync(at<char>(ws, H.crop), (size_t)H.rows * row_bytes,
                              static_cast<const char*>(frames_host) + (size_t)H.r0 * row_bytes,
                              (size_t)geom->det_y * row_bytes, (size_t)H.rows * row_bytes, (size_t)geom->n * geom->n,
                              cudaMemcpyHostToDevice, hc->s);
    } else {
        // the bounding box: a 3D copy (columns x rows x frames); measured on GB300 at ~170 GB/s
        // against ~210 GB/s for whole rows, a net gain once the box is narrower than ~80 % of a row
        cudaMemcpy3DParms p = {};
        p.srcPtr = make_cudaPitchedPtr(const_cast<void*>(frames_host), row_bytes, row_bytes, (size_t)geom->det_y);
        p.srcPos = make_cudaPos((size_t)H.c0 * es, (size_t)H.r0, 0);
        p.dstPtr = make_cudaPitchedPtr(at<char>(ws, H.crop), (size_t)H.pitch * es, (size_t)H.cols * es,
                                       (size_t)H.rows);
        p.dstPos = make_cudaPos(0, 0, 0);
        p.extent = make_cudaExtent((size_t)H.cols * es, (size_t)H.rows, (size_t)geom->n * geom->n);
        p.kind = cudaMemcpyHostToDevice;
        e = cudaMemcpy3DAsync(&p, hc->s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy of the bright-field box");
    if ((e = cudaEventRecord(hc->join, hc->s)) != cudaSuccess || (e = cudaStreamWaitEvent(st, hc->join, 0)) != cudaSuccess)
        return cuda_fail(e, "host copy join");
    int32_t* idx = at<int32_t>(ws, H.idx);
    if ((e = launch_crop_idx(bf_idx_dev, n_bf, geom->det_x, H.r0, H.c0, H.pitch, idx, st)) != cudaSuccess)
        return cuda_fail(e, "index remap");
    ssb_geometry crop = *geom;
    crop.det_y = H.rows;
    crop.det_x = H.pitch;
    return ssb_build_G(at<char>(ws, H.crop), dtype, &crop, idx, n_bf, G_dev, at<char>(ws, H.build),
                       ws_bytes - H.build, stream);
}

static ssb_gstore c64_store(const void* G_dev) {
    ssb_gstore s{};
    s.G = G_dev;
    s.fmt = SSB_G_C64;
    return s;
}

// every argument check of a reconstruction except the workspace's
static int check_recon_args(const ssb_gstore* store, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                            const ssb_aberr* set, const void* O_dev, const int32_t* N_dev, const float* phase_dev,
                            GView* gv) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    if ((rc = gview_of(store, geom, 0, gv)) != SSB_OK) return rc;
    if (gv->band) return fail(SSB_INVALID_ARG, "a reconstruction needs the half plane, not a band-compacted G");
    if (!bf_idx_dev || !set || !O_dev || !N_dev || !phase_dev)
        return fail(SSB_INVALID_ARG, "G, bf_idx, set, O, N and phase must not be NULL");
    if (n_bf < 1 || (long long)n_bf > (long long)geom->det_y * geom->det_x)
        return fail(SSB_INVALID_ARG, "n_bf=%d out of range", n_bf);
    return check_set(set);
}

}  // extern "C"

namespace ssb {
int check_reconstruct_args(const void* G_dev, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                           const ssb_aberr* set, const void* O_dev, const int32_t* N_dev, const float* phase_dev) {
    const ssb_gstore s = c64_store(G_dev);
    GView gv{};
    return check_recon_args(&s, geom, bf_idx_dev, n_bf, set, O_dev, N_dev, phase_dev, &gv);
}
}  // namespace ssb

extern "C" {

static int reconstruct_impl(const ssb_gstore* store, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                            const ssb_aberr* set, void* O_dev, int32_t* N_dev, float* phase_dev, void* ws,
                            size_t ws_bytes, void* stream) {
    int rc;
    GView gv{};
    if ((rc = check_recon_args(store, geom, bf_idx_dev, n_bf, set, O_dev, N_dev, phase_dev, &gv)) != SSB_OK)
        return rc;
    const WsLayout Lw = layout(geom, n_bf, SSB_OP_RECON, 1, 0);
    if ((rc = check_ws(ws, ws_bytes, Lw.total)) != SSB_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SetBatch sb{};
    sb.B = 1;
    sb.r2 = aperture_r2(geom);
    sb.s[0] = set_params(geom, set);
    const int n = geom->n, nq = n * (n / 2 + 1);
    float2* tw = at<float2>(ws, Lw.tw);
    cudaError_t e;
    if ((e = launch_twiddles(tw, n, st)) != cudaSuccess) return cuda_fail(e, "twiddles");
    if ((rc = run_reduction(gv, geom, bf_idx_dev, n_bf, sb, nullptr, nq, static_cast<float2*>(O_dev), N_dev,
                            ws, Lw, 1, st)) != SSB_OK)
        return rc;
    if ((e = launch_phase(static_cast<const float2*>(O_dev), N_dev, at<double>(ws, Lw.dcpart),
                          (n_bf + 255) / 256, n_bf, n, at<float2>(ws, Lw.Y), tw, phase_dev, st)) != cudaSuccess)
        return cuda_fail(e, "phase");
    g_err[0] = 0;
    return SSB_OK;
}

int ssb_reconstruct_sums(const void* G_dev, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                         const ssb_aberr* set, void* O_dev, int32_t* N_dev, double* g0_sum_dev, void* ws,
                         size_t ws_bytes, void* stream) {
    int rc;
    GView gv{};
    const ssb_gstore store = c64_store(G_dev);
    if (!g0_sum_dev) return fail(SSB_INVALID_ARG, "g0_sum must not be NULL");
    // the image is not formed here: any non-null pointer stands in for it
    if ((rc = check_recon_args(&store, geom, bf_idx_dev, n_bf, set, O_dev, N_dev,
                               reinterpret_cast<const float*>(g0_sum_dev), &gv)) != SSB_OK)
        return rc;
    const WsLayout Lw = layout(geom, n_bf, SSB_OP_RECON, 1, 0);
    if ((rc = check_ws(ws, ws_bytes, Lw.total)) != SSB_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SetBatch sb{};
    sb.B = 1;
    sb.r2 = aperture_r2(geom);
    sb.s[0] = set_params(geom, set);
    const int n = geom->n, nq = n * (n / 2 + 1);
    if ((rc = run_reduction(gv, geom, bf_idx_dev, n_bf, sb, nullptr, nq, static_cast<float2*>(O_dev), N_dev,
                            ws, Lw, 1, st)) != SSB_OK)
        return rc;
    cudaError_t e;
    if ((e = launch_dc_total(at<double>(ws, Lw.dcpart), (n_bf + 255) / 256, g0_sum_dev, st)) != cudaSuccess)
        return cuda_fail(e, "G(0,k) sum");
    g_err[0] = 0;
    return SSB_OK;
}

int ssb_phase_from_sums(const void* O_dev, const int32_t* N_dev, const double* g0_sum_dev, int n_bf_total,
                        const ssb_geometry* geom, float* phase_dev, void* ws, size_t ws_bytes, void* stream) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    if (!O_dev || !N_dev || !g0_sum_dev || !phase_dev)
        return fail(SSB_INVALID_ARG, "O, N, g0_sum and phase must not be NULL");
    if (n_bf_total < 1) return fail(SSB_INVALID_ARG, "n_bf_total=%d must be >= 1", n_bf_total);
    const WsLayout Lw = layout(geom, 1, SSB_OP_PHASE, 1, 0);
    if ((rc = check_ws(ws, ws_bytes, Lw.total)) != SSB_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float2* tw = at<float2>(ws, Lw.tw);
    cudaError_t e;
    if ((e = launch_twiddles(tw, geom->n, st)) != cudaSuccess) return cuda_fail(e, "twiddles");
    if ((e = launch_phase(static_cast<const float2*>(O_dev), N_dev, g0_sum_dev, 1, n_bf_total, geom->n,
                          at<float2>(ws, Lw.Y), tw, phase_dev, st)) != cudaSuccess)
        return cuda_fail(e, "phase");
    g_err[0] = 0;
    return SSB_OK;
}

static int score_impl(const ssb_gstore* store, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                      const ssb_aberr* sets, int B, const int32_t* band_dev, int nq, void* O_dev,
                      int32_t* N_dev, double* score_dev, void* ws, size_t ws_bytes, void* stream,
                      const double* depth_A = nullptr) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    GView gv{};
    if ((rc = gview_of(store, geom, nq, &gv)) != SSB_OK) return rc;
    if (!bf_idx_dev || !sets || !band_dev || !O_dev || !N_dev || !score_dev)
        return fail(SSB_INVALID_ARG, "G, bf_idx, sets, band, O, N and score must not be NULL");
    if (B < 1 || B > SSB_MAX_SETS) return fail(SSB_UNSUPPORTED, "B=%d not in [1, %d]", B, SSB_MAX_SETS);
    if (n_bf < 1 || (long long)n_bf > (long long)geom->det_y * geom->det_x)
        return fail(SSB_INVALID_ARG, "n_bf=%d out of range", n_bf);
    if (nq < 1 || (long long)nq > (long long)geom->n * (geom->n / 2 + 1))
        return fail(SSB_INVALID_ARG, "nq=%d out of range", nq);
    for (int s = 0; s < B; ++s)
        if ((rc = check_set(&sets[s])) != SSB_OK) return rc;
    if (depth_A)
        for (int s = 0; s < B; ++s)
            if (!std::isfinite(depth_A[s]) || depth_A[s] < 0.0)
                return fail(SSB_INVALID_ARG, "depth_A[%d] must be finite and >= 0", s);
    const WsLayout Lw = layout(geom, n_bf, SSB_OP_SCORE, B, nq);
    if ((rc = check_ws(ws, ws_bytes, Lw.total)) != SSB_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SetBatch sb{};
    sb.B = B;
    sb.r2 = aperture_r2(geom);
    for (int s = 0; s < B; ++s) sb.s[s] = set_params(geom, &sets[s]);
    // the batched kernels compute a compile-time number of sets (2, 4 or 8);
    // the slots past B hold copies of set 0, whose sums are never written
    for (int s = B; s < SSB_MAX_SETS; ++s) sb.s[s] = sb.s[0];
    int depth = 0;
    for (int s = 0; depth_A && s < B; ++s) {
        sb.depth_a[s] = (float)(M_PI * geom->wavelength_A * depth_A[s] / 2.0);
        if (depth_A[s] > 0.0) depth = 1;
    }
    sb.depth_shared = 1;
    for (int s = 1; s < B; ++s)
        if (sb.depth_a[s] != sb.depth_a[0]) sb.depth_shared = 0;
    if ((rc = run_reduction(gv, geom, bf_idx_dev, n_bf, sb, band_dev, nq, static_cast<float2*>(O_dev), N_dev,
                            ws, Lw, 0, st, depth)) != SSB_OK)
        return rc;
    cudaError_t e;
    if ((e = launch_score(static_cast<const float2*>(O_dev), N_dev, B, nq, score_dev, st)) != cudaSuccess)
        return cuda_fail(e, "score");
    g_err[0] = 0;
    return SSB_OK;
}

int ssb_reconstruct(const void* G_dev, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                    const ssb_aberr* set, void* O_dev, int32_t* N_dev, float* phase_dev, void* ws,
                    size_t ws_bytes, void* stream) {
    const ssb_gstore s = c64_store(G_dev);
    return reconstruct_impl(&s, geom, bf_idx_dev, n_bf, set, O_dev, N_dev, phase_dev, ws, ws_bytes, stream);
}

int ssb_reconstruct_g(const ssb_gstore* G, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                      const ssb_aberr* set, void* O_dev, int32_t* N_dev, float* phase_dev, void* ws,
                      size_t ws_bytes, void* stream) {
    return reconstruct_impl(G, geom, bf_idx_dev, n_bf, set, O_dev, N_dev, phase_dev, ws, ws_bytes, stream);
}

int ssb_score_batch(const void* G_dev, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                    const ssb_aberr* sets, int B, const int32_t* band_dev, int nq, void* O_dev,
                    int32_t* N_dev, double* score_dev, void* ws, size_t ws_bytes, void* stream) {
    const ssb_gstore s = c64_store(G_dev);
    return score_impl(&s, geom, bf_idx_dev, n_bf, sets, B, band_dev, nq, O_dev, N_dev, score_dev, ws, ws_bytes,
                      stream);
}

int ssb_score_batch_g(const ssb_gstore* G, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                      const ssb_aberr* sets, int B, const int32_t* band_dev, int nq, void* O_dev,
                      int32_t* N_dev, double* score_dev, void* ws, size_t ws_bytes, void* stream) {
    return score_impl(G, geom, bf_idx_dev, n_bf, sets, B, band_dev, nq, O_dev, N_dev, score_dev, ws, ws_bytes,
                      stream);
}

int ssb_score_batch_depth(const ssb_gstore* G, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                          const ssb_aberr* sets, const double* depth_A, int B, const int32_t* band_dev, int nq,
                          void* O_dev, int32_t* N_dev, double* score_dev, void* ws, size_t ws_bytes, void* stream) {
    if (!depth_A) return fail(SSB_INVALID_ARG, "depth_A must not be NULL");
    return score_impl(G, geom, bf_idx_dev, n_bf, sets, B, band_dev, nq, O_dev, N_dev, score_dev, ws, ws_bytes,
                      stream, depth_A);
}

int ssb_phase_moments(const ssb_gstore* store, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                      const ssb_aberr* set, float* mean_dev, float* var_dev, void* ws, size_t ws_bytes,
                      void* stream) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    GView gv{};
    if ((rc = gview_of(store, geom, 0, &gv)) != SSB_OK) return rc;
    if (gv.band) return fail(SSB_INVALID_ARG, "the phase moments need the half plane, not a band-compacted G");
    if (!bf_idx_dev || !set || !mean_dev || !var_dev)
        return fail(SSB_INVALID_ARG, "G, bf_idx, set, mean and var must not be NULL");
    if (n_bf < 1 || (long long)n_bf > (long long)geom->det_y * geom->det_x)
        return fail(SSB_INVALID_ARG, "n_bf=%d out of range", n_bf);
    if ((rc = check_set(set)) != SSB_OK) return rc;
    const WsLayout Lw = layout(geom, n_bf, SSB_OP_MOMENTS, 1, 0);
    if ((rc = check_ws(ws, ws_bytes, Lw.total)) != SSB_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SetBatch sb{};
    sb.B = 1;
    sb.r2 = aperture_r2(geom);
    sb.s[0] = set_params(geom, set);
    float2* tw = at<float2>(ws, Lw.tw);
    float4* ktab = at<float4>(ws, Lw.ktab);
    cudaError_t e;
    if ((e = launch_twiddles(tw, geom->n, st)) != cudaSuccess) return cuda_fail(e, "twiddles");
    if ((e = launch_prep(bf_idx_dev, n_bf, geom->det_x, geom->det_center_y, geom->det_center_x, geom->det_pitch_invA,
                         sb, ktab, at<float>(ws, Lw.chik), nullptr, nullptr, gv, nullptr, st)) != cudaSuccess)
        return cuda_fail(e, "prep");
    if ((e = launch_moments(gv, geom->n, n_bf, ktab, sb, 1.0 / ((double)geom->n * geom->scan_step_A), tw,
                            at<void>(ws, Lw.Y), at<void>(ws, Lw.Opart), mean_dev, var_dev, st)) != cudaSuccess)
        return cuda_fail(e, "moments");
    g_err[0] = 0;
    return SSB_OK;
}

int ssb_compact_G16(const void* G_dev, const ssb_geometry* geom, int n_bf, int rows_per_scale, void* G16_dev,
                    float* scale_dev, void* stream) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    if (!G_dev || !G16_dev || !scale_dev) return fail(SSB_INVALID_ARG, "G, G16 and scale must not be NULL");
    if (n_bf < 1) return fail(SSB_INVALID_ARG, "n_bf=%d must be >= 1", n_bf);
    if (rows_per_scale != 1 && rows_per_scale != geom->n)
        return fail(SSB_UNSUPPORTED, "rows_per_scale=%d must be 1 or n=%d", rows_per_scale, geom->n);
    cudaError_t e = launch_compact_g16(static_cast<const float2*>(G_dev), geom->n, n_bf, rows_per_scale,
                                       static_cast<uint32_t*>(G16_dev), scale_dev, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "compact_G16");
    g_err[0] = 0;
    return SSB_OK;
}

int ssb_compact_band(const ssb_gstore* src, const ssb_geometry* geom, int n_bf, const int32_t* band_dev, int nq,
                     void* dst_dev, void* stream) {
    int rc;
    if ((rc = check_geom(geom)) != SSB_OK) return rc;
    if (!src || !src->G || !band_dev || !dst_dev) return fail(SSB_INVALID_ARG, "G, band and dst must not be NULL");
    if (src->fmt != SSB_G_C64 && src->fmt != SSB_G_SN16) return fail(SSB_INVALID_ARG, "unknown G format %d", src->fmt);
    if (src->band_compact) return fail(SSB_INVALID_ARG, "the source must be a half-plane G");
    if (n_bf < 1) return fail(SSB_INVALID_ARG, "n_bf=%d must be >= 1", n_bf);
    if (nq < 1 || (long long)nq > (long long)geom->n * (geom->n / 2 + 1))
        return fail(SSB_INVALID_ARG, "nq=%d out of range", nq);
    cudaError_t e = launch_compact_band(src->G, src->fmt, (size_t)geom->n * (geom->n / 2 + 1), n_bf, band_dev, nq,
                                        dst_dev, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "compact_band");
    g_err[0] = 0;
    return SSB_OK;
}

}  // extern "C"
