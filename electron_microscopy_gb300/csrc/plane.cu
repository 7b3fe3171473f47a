// plane.cu -- G(q,k) build for the n = 512 scan: gather + one-pass 2D R2C on a
// thread-block cluster.
//
// What is computed is the same as build.cu (G(q,k) = sum_r x_k(r)
// exp(-2 pi i (f_y r_y + f_x r_x)/n), half plane [k][q_y][q_x]; quantem.gpu
// "Historical WebGPU G(q,k) memory experiment", sections "Why herm is exactly
// lossless" and "Implementation"); how differs:
//
//  1. ssb_gather: for a chunk of up to 64 bright-field pixels, reads the frames
//     once (each warp load takes 32 neighbouring detector pixels of one frame,
//     16-32 loads in flight per thread, streaming cache hint) and writes the
//     transposed traces X[pixel][r] (uint16, or float for float frames) into a
//     chunk buffer that stays in L2 for the next kernel.
//  2. ssb_plane512: one cluster of 8 CTAs per bright-field pixel (persistent:
//     as many clusters as fit, each looping over planes).  CTA j owns scan
//     rows r_y = j + 8 m (m < 64), staged from the chunk buffer into shared
//     memory by 16-byte asynchronous copies issued by every thread:
//       a. real-to-complex FFT of each of its 64 rows along r_x: a 256-point
//          complex FFT of the packed even/odd samples (16 threads per row,
//          two radix-16 passes, one shared-memory transpose) and the split
//          step, into a 64 x 257 slab in shared memory;
//       b. for each of the 257 columns, the 64-point DFT over its own rows,
//          times exp(-2 pi i j k_lo / 512) (8 threads per column, radix 8 x 8);
//       c. the 64 x 257 results go to one of two L2-resident exchange slots
//          of the cluster; cluster barrier; then the last radix-8 stage across
//          the 8 CTAs: CTA j reads the 8 CTAs' entries (k_lo, q_x) for k_lo in
//          [8j, 8j+8) from L2 and writes G[k][k_lo + 64 k_hi][q_x] straight
//          to HBM, once.  (Reading the slabs through distributed shared
//          memory instead measured ~34 GB/s per SM, 3x slower than L2.)
//     Phase c of a plane runs during the row phase of the cluster's next
//     plane (an L2 -> HBM stream under shared-memory arithmetic); the two
//     exchange slots alternate so that one cluster barrier per plane orders
//     both.  The chunk buffer lines a CTA consumed are dropped from L2
//     without being written back (discard.global.L2): they are dead.
// The HBM traffic of a build is therefore the frames read once plus G
// written once; the n x (n/2+1) intermediate stays on chip (shared memory
// and L2).
#include <mutex>

#include "internal.cuh"

namespace ssb {

constexpr int kGatherThreads = 256;
constexpr int kGatherFrames = 64;  // scan positions per gather CTA

template <typename T>
__host__ __device__ constexpr int gather_pixels() { return sizeof(T) == 2 ? 64 : 32; }

// ---------------------------------------------------------------------------
// gather: frames (npos, det_pix) -> X[p][r] for p < kc, r in this CTA's block
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kGatherThreads)
ssb_gather(const T* __restrict__ frames, int det_pix, const int32_t* __restrict__ bf_idx, int k0, int kc,
           int npos, T* __restrict__ X) {
    constexpr int KC = gather_pixels<T>();
    constexpr int FS = kGatherThreads / KC;          // frame slots per pass
    constexpr int NL = kGatherFrames / FS;           // loads per thread
    constexpr int PAD = sizeof(T) == 2 ? 2 : 1;      // odd word stride between rows
    constexpr int RS = kGatherFrames + PAD;
    __shared__ __align__(16) T s[KC * RS];
    const int tid = threadIdx.x;
    const int p = tid % KC, fs = tid / KC;
    const int f0 = blockIdx.x * kGatherFrames;
    if (p < kc) {
        const T* src = frames + (size_t)(f0 + fs) * det_pix + bf_idx[k0 + p];
        T v[NL];
#pragma unroll
        for (int i = 0; i < NL; ++i) v[i] = __ldcs(src + (size_t)(FS * i) * det_pix);
#pragma unroll
        for (int i = 0; i < NL; ++i) s[p * RS + fs + FS * i] = v[i];
    }
    __syncthreads();
    // write rows of kGatherFrames elements as 16-byte vectors
    constexpr int VE = 16 / (int)sizeof(T);
    constexpr int VPR = kGatherFrames / VE;
    for (int idx = tid; idx < kc * VPR; idx += kGatherThreads) {
        const int row = idx / VPR, col = idx - row * VPR;
        const T* r = s + row * RS + col * VE;
        uint4 pk;
        if constexpr (sizeof(T) == 2) {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(r);  // 4-byte aligned: RS even
            pk = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            pk = make_uint4(__float_as_uint(r[0]), __float_as_uint(r[1]), __float_as_uint(r[2]),
                            __float_as_uint(r[3]));
        }
        *reinterpret_cast<uint4*>(X + (size_t)row * npos + f0 + col * VE) = pk;
    }
}

// ---------------------------------------------------------------------------
// cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cluster barrier without release semantics: for the end of a phase whose
// only cross-CTA accesses were reads that have already completed
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// 16-byte asynchronous global -> shared copies (L2 only), and the wait for
// all of this thread's outstanding ones
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void discard_l2_line(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// ---------------------------------------------------------------------------
// one bright-field pixel's 512 x 512 real-to-complex FFT on a C-CTA cluster;
// persistent: cluster c handles chunk planes c, c + nclusters, ...
//   C = 8:  64 scan rows per CTA, 512 threads, ~137 KB shared: 1 CTA per SM
//   C = 16: 32 scan rows per CTA, 256 threads, ~106 KB shared: 2 CTAs per SM
//           (kept as a template form; see plane_cluster_size)
// ---------------------------------------------------------------------------
constexpr int kPlaneN = 512;
constexpr int kPlaneH = kPlaneN / 2 + 1;
constexpr int kPlanePS = 258;   // slab row stride (float2)
constexpr int kStageRS = 544;   // staged uint16 row stride: 16 words mod 32 (disjoint banks for the two
                                // half-warps reading adjacent rows), 16-byte aligned
constexpr int kXchRS = 264;     // exchange row stride (float2), 32-byte aligned rows
constexpr int kMaxClusters = 24;
// cross-CTA exchange through L2: per cluster slot, [rank][k_lo][kXchRS] float2,
// rank x k_lo = 512 rows whatever the cluster size
constexpr size_t kXchSlot = (size_t)kPlaneN * kXchRS * sizeof(float2);

template <int C>
struct PlaneCfg {
    static constexpr int M = kPlaneN / C;                  // scan rows per CTA (local column DFT length)
    static constexpr int T = M / 8;                        // column threads: DFT8 over n2, then DFT_T over t
    static constexpr int THREADS = 64 * T;                 // 64 columns per pass
    static constexpr int MINB = C == 8 ? 1 : 2;
    // shared memory: split-step twiddles W512^k (k <= 256), row twiddles
    // W256^(t k2) as [k2][t], column twiddles W_M^(t k2) as [k2][t], cross
    // twiddles W512^(j k_lo), the M x PS slab, the staged rows
    static constexpr int TW_SPLIT = 0, TW_ROW = 260, TW_COL = TW_ROW + 256, TW_X = TW_COL + 8 * T,
                         TW_TOTAL = TW_X + M;
    static constexpr size_t SLAB = (size_t)M * kPlanePS * sizeof(float2);
    static constexpr size_t SMEM = (size_t)TW_TOTAL * sizeof(float2) + SLAB + (size_t)M * kStageRS * 2;
    static_assert(THREADS == 16 * (M / 2), "two row iterations of THREADS/16 rows");
    static_assert(M != 64 || (size_t)2 * 64 * 64 * sizeof(float2) <= (size_t)M * kStageRS * 2,
                  "two column-transpose buffers fit the staging area");
};

// stage the M rows r_y = j + C m of plane Xk (1 KB each) into shared memory:
// every thread issues its share of the 16-byte copies (consecutive threads,
// consecutive 16 bytes of a row).  Bulk copies of whole rows were measured
// slower here: the copy engine took ~30 ns per 1 KB row.
template <int C>
__device__ __forceinline__ void stage_rows(const uint16_t* Xk, uint32_t stage, uint32_t j, int tid) {
    constexpr int M = PlaneCfg<C>::M, NT = PlaneCfg<C>::THREADS;
    constexpr int CPR = kPlaneN * (int)sizeof(uint16_t) / 16;  // copies per row
#pragma unroll
    for (int i = tid; i < M * CPR; i += NT) {
        const int m = i / CPR, c = i - m * CPR;
        cp_async16(stage + (uint32_t)(m * kStageRS * 2 + 16 * c), Xk + (size_t)(j + C * m) * kPlaneN + 8 * c);
    }
}

template <int C>
__global__ void __launch_bounds__(PlaneCfg<C>::THREADS, PlaneCfg<C>::MINB)
ssb_plane512(const uint16_t* __restrict__ X, int k0, int kc, float2* __restrict__ G, const float2* __restrict__ twg,
             float2* __restrict__ xch) {
    using Cfg = PlaneCfg<C>;
    constexpr int N = kPlaneN, H = kPlaneH, PS = kPlanePS, M = Cfg::M, T = Cfg::T, NT = Cfg::THREADS;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float2* tws = reinterpret_cast<float2*>(smem_raw);
    float2* slab = tws + Cfg::TW_TOTAL;  // [M][PS]
    const uint32_t* stg = reinterpret_cast<const uint32_t*>(smem_raw + Cfg::TW_TOTAL * sizeof(float2) + Cfg::SLAB);
    float2* scratch = reinterpret_cast<float2*>(smem_raw + Cfg::TW_TOTAL * sizeof(float2) + Cfg::SLAB);
    const uint32_t stage = smem_addr(stg);
    const int tid = threadIdx.x;
    const uint32_t j = cluster_rank();
    const int ncl = gridDim.x / C;
    int kk = blockIdx.x / C;
    if (kk < kc) stage_rows<C>(X + (size_t)kk * N * N, stage, j, tid);

    for (int i = tid; i < Cfg::TW_TOTAL; i += NT) {
        float2 w = make_float2(1.f, 0.f);
        if (i < Cfg::TW_ROW) {
            if (i <= N / 2) w = twg[i];
        } else if (i < Cfg::TW_COL) {
            const int k2 = (i - Cfg::TW_ROW) >> 4, t = (i - Cfg::TW_ROW) & 15;
            w = twg[2 * t * k2];  // W256^(t k2)
        } else if (i < Cfg::TW_X) {
            const int k2 = (i - Cfg::TW_COL) / T, t = (i - Cfg::TW_COL) % T;
            w = twg[(N / M) * t * k2];  // W_M^(t k2)
        } else {
            w = twg[j * (i - Cfg::TW_X)];  // W512^(j k_lo)
        }
        tws[i] = w;
    }
    __syncthreads();  // twiddles in place
    // two exchange slots per cluster: the column phase of plane i writes slot
    // i & 1 while the radix-C phase of plane i - 1 still reads the other
    constexpr size_t kSlotF = kXchSlot / sizeof(float2);
    float2* xbase = xch + (size_t)(2 * (blockIdx.x / C)) * kSlotF;
    // ---- c. radix-C across the cluster, straight to G: pair p = (k_lo, q_x)
    //         of a plane whose exchange rows are complete ----
    constexpr int KL = M / C;        // k_lo values per CTA
    constexpr int P = KL * H;        // pairs per CTA
    constexpr int QF = P / NT;       // rounds every thread takes
    constexpr int PT = P - QF * NT;  // threads taking one more
    static_assert(QF >= 2, "two rounds before the row phase");
    auto c_load = [&](const float2* xs, int p, float2 (&v)[C]) {
        const int kl = KL * (int)j + p / H, c = p % H;
        const float2* src = xs + (size_t)kl * kXchRS + c;
#pragma unroll
        for (int r = 0; r < C; ++r) v[r] = __ldcg(src + (size_t)r * M * kXchRS);
    };
    auto c_store = [&](float2* Gk, int p, float2 (&v)[C]) {
        const int kl = KL * (int)j + p / H, c = p % H;
        Dft<C>::run(v);
#pragma unroll
        for (int kh = 0; kh < C; ++kh) __stcs(Gk + (size_t)(kl + M * kh) * H + c, v[kh]);
    };

    // Software pipeline over the planes of this cluster: iteration i runs the
    // radix-C phase of plane i - 1 (an L2 -> HBM stream) inside the row phase
    // of plane i (shared-memory arithmetic), so that one hides the other, and
    // the next plane's staging copies fly while the first rounds of it run.
    int prev = -1;       // plane whose radix-C phase is pending
    uint32_t slot = 0;   // exchange slot the next column phase writes
#pragma unroll 1
    for (; kk < kc; kk += ncl) {
        const float2* xprev = xbase + (size_t)(slot ^ 1u) * kSlotF;
        float2* Gprev = G + (size_t)(k0 + (prev >= 0 ? prev : 0)) * N * H;
        if (prev >= 0) {
            float2 ca[C], cb[C];
            c_load(xprev, tid, ca);
            c_load(xprev, tid + NT, cb);
            c_store(Gprev, tid, ca);
            c_store(Gprev, tid + NT, cb);
        }
        // the staged rows have landed; their global copies are dead: drop them
        // from L2 without write-back (thread i takes 128-byte line i)
        cp_async_wait_all();
        discard_l2_line(reinterpret_cast<const char*>(X + (size_t)kk * N * N + (size_t)(j + C * (tid >> 3)) * N) +
                        128 * (tid & 7));
        __syncthreads();
        // ---- a. row R2C: 16 threads per row, NT/16 rows at a time; rounds
        //         2 and 3 of the pending radix-C phase ride along ----
        {
            const int t = tid & 15, hw = tid >> 4;
            const int lane = tid & 31;
            const int src_lane = (lane & 16) | ((16 - t) & 15);
#pragma unroll 1
            for (int it = 0; it < 2; ++it) {
                const int q = 2 + it;
                const bool cq = prev >= 0 && q < QF;
                float2 cv[C];
                if (cq) c_load(xprev, tid + q * NT, cv);
                const int m = it * (NT / 16) + hw;
                const uint32_t* row = stg + m * (kStageRS / 2);
                float2 v[16];
#pragma unroll
                for (int n2 = 0; n2 < 16; ++n2) v[n2] = half_pair(row[t + 16 * n2]);
                Dft<16>::run(v);
#pragma unroll
                for (int k2 = 1; k2 < 16; ++k2) v[k2] = cmul(v[k2], tws[Cfg::TW_ROW + 16 * k2 + t]);
                float2* s = slab + m * PS;
#pragma unroll
                for (int k2 = 0; k2 < 16; ++k2) s[k2 * 16 + (t ^ k2)] = v[k2];
                __syncwarp();
#pragma unroll
                for (int n1 = 0; n1 < 16; ++n1) v[n1] = s[t * 16 + (n1 ^ t)];
                __syncwarp();
                Dft<16>::run(v);  // v[k1] = Z[t + 16 k1] (Z of the halved samples)
                // split step: X[k] = a - i W^k b, a = Z[k] + conj Z[L-k], b = Z[k] - conj Z[L-k]
#pragma unroll
                for (int k1 = 0; k1 < 16; ++k1) {
                    float2 pr;
                    pr.x = __shfl_sync(0xffffffffu, v[15 - k1].x, src_lane);
                    pr.y = __shfl_sync(0xffffffffu, v[15 - k1].y, src_lane);
                    if (t == 0) pr = v[(16 - k1) & 15];
                    const float2 z = v[k1];
                    const float ax = z.x + pr.x, ay = z.y - pr.y;
                    const float bx = z.x - pr.x, by = z.y + pr.y;
                    const float2 w = tws[Cfg::TW_SPLIT + t + 16 * k1];
                    s[t + 16 * k1] = make_float2(ax + w.x * by + w.y * bx, ay - w.x * bx + w.y * by);
                }
                if (t == 0) s[N / 2] = make_float2(2.0f * (v[0].x - v[0].y), 0.0f);
                if (cq) c_store(Gprev, tid + q * NT, cv);
            }
            // the remaining rounds of the pending radix-C phase
#pragma unroll 1
            for (int q = 4; prev >= 0 && q < QF; ++q) {
                float2 cv[C];
                c_load(xprev, tid + q * NT, cv);
                c_store(Gprev, tid + q * NT, cv);
            }
            if (prev >= 0 && tid < PT) {
                float2 cv[C];
                c_load(xprev, tid + QF * NT, cv);
                c_store(Gprev, tid + QF * NT, cv);
            }
        }
        __syncthreads();
        // ---- b. local M-point column DFTs (DFT8 over rows t + T n2, twiddle,
        //         DFT_T over t), times W512^(j k_lo), to the L2 exchange ----
        {
            float2* xout = xbase + (size_t)slot * kSlotF + (size_t)j * M * kXchRS;
            const int t = tid >> 6, cl = tid & 63;
            float2 wc[8], wx[8];
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) wc[k2] = tws[Cfg::TW_COL + k2 * T + t];  // W_M^(t k2)
#pragma unroll
            for (int i = 0; i < 8 / T; ++i)
#pragma unroll
                for (int k1 = 0; k1 < T; ++k1) wx[i * T + k1] = tws[Cfg::TW_X + (t + T * i) + 8 * k1];
            auto col = [&](int c, int tt, const float2* wcv, const float2* wxv, auto sync) {
                float2 v[8];
#pragma unroll
                for (int n2 = 0; n2 < 8; ++n2) v[n2] = slab[(tt + T * n2) * PS + c];
                Dft<8>::run(v);
#pragma unroll
                for (int k2 = 1; k2 < 8; ++k2) v[k2] = cmul(v[k2], wcv[k2]);
                sync();
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) slab[(k2 * T + tt) * PS + c] = v[k2];
                sync();
#pragma unroll
                for (int i = 0; i < 8 / T; ++i) {
                    const int k2 = tt + T * i;
                    float2 u[T];
#pragma unroll
                    for (int n1 = 0; n1 < T; ++n1) u[n1] = slab[(k2 * T + n1) * PS + c];
                    Dft<T>::run(u);  // u[k1] = Y[k2 + 8 k1]
#pragma unroll
                    for (int k1 = 0; k1 < T; ++k1) xout[(k2 + 8 * k1) * kXchRS + c] = cmul(u[k1], wxv[i * T + k1]);
                }
            };
            // columns 0..n/2-1, 64 per batch: the transpose between the two
            // radix-8 stages goes through one of two [64][64] buffers in the
            // staging area (idle until the next plane's copies), so one block
            // barrier per batch suffices: buffer b is rewritten two batches on,
            // after the next batch's barrier
            static_assert(T == 8, "batched column transpose written for 64-row slabs");
#pragma unroll 1
            for (int i = 0; i < N / 2 / 64; ++i) {
                const int c = cl + 64 * i;
                float2* buf = scratch + (size_t)(i & 1) * 64 * 64;
                float2 v[8];
#pragma unroll
                for (int n2 = 0; n2 < 8; ++n2) v[n2] = slab[(t + 8 * n2) * PS + c];
                Dft<8>::run(v);
#pragma unroll
                for (int k2 = 1; k2 < 8; ++k2) v[k2] = cmul(v[k2], wc[k2]);
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) buf[(k2 * 8 + t) * 64 + cl] = v[k2];
                __syncthreads();
#pragma unroll
                for (int n1 = 0; n1 < 8; ++n1) v[n1] = buf[(t * 8 + n1) * 64 + cl];
                Dft<8>::run(v);  // v[k1] = Y[t + 8 k1]
#pragma unroll
                for (int k1 = 0; k1 < 8; ++k1) xout[(t + 8 * k1) * kXchRS + c] = cmul(v[k1], wx[k1]);
            }
            // column q_x = n/2: lanes 0..T-1 of warp 0, t = lane, in place
            if (tid < T) {
                float2 wc2[8], wx2[8];
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) wc2[k2] = tws[Cfg::TW_COL + k2 * T + tid];
#pragma unroll
                for (int i = 0; i < 8 / T; ++i)
#pragma unroll
                    for (int k1 = 0; k1 < T; ++k1) wx2[i * T + k1] = tws[Cfg::TW_X + (tid + T * i) + 8 * k1];
                col(N / 2, tid, wc2, wx2, [] { __syncwarp((1u << T) - 1u); });
            }
        }
        __syncthreads();
        // exchange rows of this plane written and visible to the cluster; every
        // read of the other slot (the previous plane's) has completed, so the
        // next column phase may overwrite it
        cluster_sync();
        // the staging buffer has been free since the row phase: fetch the next
        // plane now (issued earlier it competed with the column phase's
        // exchange stores for the SM's path to L2)
        if (kk + ncl < kc) stage_rows<C>(X + (size_t)(kk + ncl) * N * N, stage, j, tid);
        prev = kk;
        slot ^= 1u;
    }
    // the last plane's radix-C phase
    if (prev >= 0) {
        const float2* xprev = xbase + (size_t)(slot ^ 1u) * kSlotF;
        float2* Gprev = G + (size_t)(k0 + prev) * N * H;
        // nothing else is live here: every round's loads go out at once
        float2 cv4[QF][C];
#pragma unroll
        for (int q = 0; q < QF; ++q) c_load(xprev, tid + q * NT, cv4[q]);
#pragma unroll
        for (int q = 0; q < QF; ++q) c_store(Gprev, tid + q * NT, cv4[q]);
        if (tid < PT) {
            float2 cv[C];
            c_load(xprev, tid + QF * NT, cv);
            c_store(Gprev, tid + QF * NT, cv);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// co-resident clusters of ssb_plane512<C> on this device (cached per device)
template <int C>
static int plane_clusters() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] != 0) return cached[dev] > 0 ? cached[dev] : 0;
    using Cfg = PlaneCfg<C>;
    int ncl = 0;
    if (cudaFuncSetAttribute(ssb_plane512<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::SMEM) ==
            cudaSuccess &&
        (C <= 8 || cudaFuncSetAttribute(ssb_plane512<C>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                       cudaSuccess)) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(C, 1, 1);
        cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&ncl, ssb_plane512<C>, &cfg) != cudaSuccess) ncl = 0;
    }
    cudaGetLastError();  // clear a refused attribute or query
    cached[dev] = ncl > 0 ? ncl : -1;
    return ncl;
}

// The cluster size used: 8 (portable). 16-CTA clusters (2 CTAs per SM) were
// measured on GB300: 14 co-resident clusters (112 SMs) against 15 8-CTA
// clusters (120 SMs), and the same plane throughput (9.32 vs 9.42 ms for all
// planes of the 512^2 x 9354 workload), so the portable form is kept.
static int plane_cluster_size() { return plane_clusters<8>() > 0 ? 8 : 0; }

int plane512_cluster_size() { return plane_cluster_size(); }

// two gather buffers of 64 planes, two exchange slots per cluster
size_t plane512_chunk_bytes() {
    return (size_t)2 * 64 * kPlaneN * kPlaneN * sizeof(uint16_t) + (size_t)2 * kMaxClusters * kXchSlot;
}

// Two internal streams per device (gather, plane) and the events that order
// them, created on first use; the launch sequence of one build holds the
// device's mutex so that concurrent builds cannot interleave their events.
struct BuildStreams {
    cudaStream_t sg = nullptr, sp = nullptr;
    cudaEvent_t fork = nullptr, g_done[2] = {}, p_done[2] = {};
    std::mutex mu;
    bool ready = false;
};

static cudaError_t get_streams(BuildStreams** out) {
    static BuildStreams per_dev[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    BuildStreams& b = per_dev[dev];
    {
        std::lock_guard<std::mutex> lock(b.mu);
        if (!b.ready) {
            int lo = 0, hi = 0;
            if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
            if ((e = cudaStreamCreateWithPriority(&b.sg, cudaStreamNonBlocking, lo)) != cudaSuccess) return e;
            if ((e = cudaStreamCreateWithPriority(&b.sp, cudaStreamNonBlocking, hi)) != cudaSuccess) return e;
            if ((e = cudaEventCreateWithFlags(&b.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
            for (int i = 0; i < 2; ++i) {
                if ((e = cudaEventCreateWithFlags(&b.g_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
                if ((e = cudaEventCreateWithFlags(&b.p_done[i], cudaEventDisableTiming)) != cudaSuccess) return e;
            }
            b.ready = true;
        }
    }
    *out = &b;
    return cudaSuccess;
}

template <int C>
static cudaError_t build512_c(const uint16_t* frames, int det_pix, const int32_t* bf_idx, int n_bf, float2* G,
                              const float2* tw, void* xbuf, cudaStream_t st) {
    using Cfg = PlaneCfg<C>;
    constexpr int KCMAX = gather_pixels<uint16_t>();
    const int npos = kPlaneN * kPlaneN;
    cudaError_t e;
    int ncl = plane_clusters<C>();
    if (ncl < 1) return cudaErrorLaunchOutOfResources;
    if (ncl > kMaxClusters) ncl = kMaxClusters;
    BuildStreams* bs = nullptr;
    if ((e = get_streams(&bs)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(bs->mu);
    // planes per chunk: a multiple of the co-resident clusters, at most KCMAX
    const int KC = ncl >= KCMAX ? KCMAX : ncl * (KCMAX / ncl);
    uint16_t* xb[2] = {static_cast<uint16_t*>(xbuf), static_cast<uint16_t*>(xbuf) + (size_t)KCMAX * npos};
    float2* xch = reinterpret_cast<float2*>(static_cast<uint16_t*>(xbuf) + (size_t)2 * KCMAX * npos);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // fork from the caller's stream
    if ((e = cudaEventRecord(bs->fork, st)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(bs->sg, bs->fork, 0)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(bs->sp, bs->fork, 0)) != cudaSuccess) return e;
    int c = 0;
    for (int k0 = 0; k0 < n_bf; ++c, k0 += KC) {
        const int kc = n_bf - k0 < KC ? n_bf - k0 : KC;
        const int b = c & 1;
        uint16_t* Xc = xb[b];
        // gather(c) may overwrite buffer b once plane(c - 2) has read it
        if (c >= 2 && (e = cudaStreamWaitEvent(bs->sg, bs->p_done[b], 0)) != cudaSuccess) return e;
        ssb_gather<uint16_t><<<npos / kGatherFrames, kGatherThreads, 0, bs->sg>>>(frames, det_pix, bf_idx, k0, kc,
                                                                                 npos, Xc);
        count_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = cudaEventRecord(bs->g_done[b], bs->sg)) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(bs->sp, bs->g_done[b], 0)) != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        const int grid_cl = kc < ncl ? kc : ncl;
        cfg.gridDim = dim3(grid_cl * C, 1, 1);
        cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
        cfg.dynamicSmemBytes = Cfg::SMEM;
        cfg.stream = bs->sp;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, ssb_plane512<C>, (const uint16_t*)Xc, k0, kc, G, tw, xch)) !=
            cudaSuccess)
            return e;
        count_launch();
        if ((e = cudaEventRecord(bs->p_done[b], bs->sp)) != cudaSuccess) return e;
    }
    // join: the caller's stream waits for the last plane (which follows every
    // gather through the event chain)
    if ((e = cudaStreamWaitEvent(st, bs->p_done[(c - 1) & 1], 0)) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_build512(const uint16_t* frames, int det_pix, const int32_t* bf_idx, int n_bf, float2* G,
                            const float2* tw, void* xbuf, cudaStream_t st) {
    if (plane_cluster_size() == 8) return build512_c<8>(frames, det_pix, bf_idx, n_bf, G, tw, xbuf, st);
    return cudaErrorLaunchOutOfResources;
}

}  // namespace ssb
