// reduce_kernel.cuh -- the fused trotter-masked reduction (ssb_reduce) as a
// template shared by reduce.cu (depth-0 weights) and reduce_depth.cu (weights
// averaged over a defocus spread); see reduce.cu for what it computes.
#pragma once

#include <type_traits>

#include "internal.cuh"

namespace ssb {

// ---------------------------------------------------------------------------
// fused reduction
// ---------------------------------------------------------------------------
constexpr int kRedThreads = 256;
constexpr int kKChunk = 256;  // k pixels whose tables a block stages at a time
// k steps whose G loads are issued together: the single-set pass streams G
// and is bound by load latency, so it keeps more loads in flight
template <int MAXB>
__host__ __device__ constexpr int red_unroll() { return MAXB == 1 ? 8 : 4; }

// Row tables of the batched forms: per warp, up to kRowSlots distinct scan
// rows (q_y) among its 32 lanes (neighbouring entries: normally 1 or 2), per
// trotter side and set one float4 (a3, a2, a1, a0); the set index is padded
// to MAXB + 1 so that the (slot, side) groups of one load fall on distinct
// banks.  A warp whose lanes span more rows evaluates the row form per term.
constexpr int kRowSlots = 4;
template <int MAXB>
__host__ __device__ constexpr int row_tab_stride() { return MAXB + 1; }
template <int MAXB>
constexpr size_t red_smem_bytes() {
    return MAXB > 1 ? (size_t)(kRedThreads / 32) * kRowSlots * 2 * row_tab_stride<MAXB>() * sizeof(float4) : 0;
}

// resident CTAs per SM the register budget is sized for (the per-set tilt
// form of the batched pass keeps its per-set aperture state: 2)
template <int MAXB, bool SHARED>
__host__ __device__ constexpr int red_min_blocks() { return (MAXB == 1 || SHARED) ? 4 : 2; }

// The aperture test at k -/+ q on one detector row.  Along a row (k_y
// fixed) the float32 test d2 = (dx*dx + dy*dy) <= r2, dx = (k_x -/+ q_x) - t_x,
// holds on a contiguous run of columns: dx is a rounded monotone function of
// k_x, dx*dx is rounded monotone on either side of dx = 0, and the sum is
// rounded monotone in it.  row_run returns the k_x of the run's first and
// last column (+inf, -inf: no column), so that for a pixel of the row the
// test equals lo <= k_x <= hi exactly.  The run is located by testing
// columns: the smallest d2 on the grid is at one of the columns next to the
// centre k_x = t_x +/- q_x, so the run is empty unless one of those passes;
// its ends are walked from estimates given by the circle's half-width.
struct RowRun {
    float lo, hi;
};
__device__ __forceinline__ RowRun row_run(const float* __restrict__ kxcol, int ncol, float inv_dk, float ccol,
                                          float ky, float qx, float qy, bool minus, float tx, float ty, float r2) {
    const RowRun none{__int_as_float(0x7f800000), __int_as_float(0xff800000)};
    const float dy = __fsub_rn(minus ? __fsub_rn(ky, qy) : __fadd_rn(ky, qy), ty);
    const float yy = __fmul_rn(dy, dy);
    if (!(yy <= r2)) return none;  // d2 >= yy at every column
    auto pass = [&](int j) {
        const float kx = __ldg(kxcol + j);
        const float dx = __fsub_rn(minus ? __fsub_rn(kx, qx) : __fadd_rn(kx, qx), tx);
        return __fadd_rn(__fmul_rn(dx, dx), yy) <= r2;
    };
    // fractional column of the centre, and the circle's half-width in columns
    const float cc = fmaf(minus ? (tx + qx) : (tx - qx), inv_dk, ccol);
    const float hw = sqrtf(r2 - yy) * inv_dk;
    const float top = (float)(ncol - 1);
    const int j0 = (int)rintf(fminf(fmaxf(cc, 0.0f), top));
    int js;
    if (pass(j0))
        js = j0;
    else if (j0 > 0 && pass(j0 - 1))
        js = j0 - 1;
    else if (j0 < ncol - 1 && pass(j0 + 1))
        js = j0 + 1;
    else
        return none;
    // first column: from the estimate, walk to the run's edge (the walks stay
    // within [0, js] and [js, ncol - 1]: js passes)
    int a = min((int)ceilf(fminf(fmaxf(cc - hw, 0.0f), top)), js);
    if (pass(a)) {
        while (a > 0 && pass(a - 1)) --a;
    } else {
        while (!pass(a)) ++a;
    }
    int b = max((int)floorf(fminf(fmaxf(cc + hw, 0.0f), top)), js);
    if (pass(b)) {
        while (b < ncol - 1 && pass(b + 1)) ++b;
    } else {
        while (!pass(b)) --b;
    }
    return RowRun{__ldg(kxcol + a), __ldg(kxcol + b)};
}

// DEPTH: each set's terms are also weighted by the defocus-spread factor
// sinc(a_s D), a_s = pi lambda t_s / 2, D = |v_k|^2 - |v_{k-/+q}|^2 (the
// squared distances the aperture tests already form, so the factor is a
// function of the same float32 values as the masks)
template <int MAXB, bool SHARED, int FMT, bool DEPTH>
__global__ void __launch_bounds__(kRedThreads, red_min_blocks<MAXB, SHARED>())
ssb_reduce(RedLaunch P, SetBatch sb) {
    const int qi = blockIdx.x * kRedThreads + threadIdx.x;
    const int split = blockIdx.y;
    const int kb = split * P.kps;
    const int ke = min(P.n_bf, kb + P.kps);
    const int H = P.n / 2 + 1;
    const bool valid = qi < P.nq;
    const int e = valid ? (P.qlist ? P.qlist[qi] : qi) : 0;
    const int row = e / H, col = e - row * H;
    const int fy = row < P.n / 2 ? row : row - P.n;
    const float qx = __double2float_rn(__dmul_rn((double)col, P.dq));
    const float qy = __double2float_rn(__dmul_rn((double)fy, P.dq));

    float2 acc[MAXB];
    int cnt[MAXB];
#pragma unroll
    for (int s = 0; s < MAXB; ++s) {
        acc[s] = make_float2(0.f, 0.f);
        cnt[s] = 0;
    }
    // this lane's G entry of pixel k sits at k * gstride + gi: the half-plane
    // entry, or the band position in a band-compacted copy; herm16 scales of
    // the lane's q row (one scale per pixel: block 0)
    const size_t gstride = P.g.stride;
    const size_t gi = valid ? (P.g.band ? (size_t)qi : (size_t)e) : 0;
    const float2* gp = static_cast<const float2*>(P.g.G) + gi;
    const uint32_t* gw = static_cast<const uint32_t*>(P.g.G) + gi;
    const float* gsc = P.g.scale + (FMT == kGSN16 && P.g.srows == 1 ? (size_t)row * P.n_bf : 0);

    // chi(k -/+ q) along the current detector row: per trotter side and set,
    // the coefficients of chi as a quartic in vx (vy is fixed along a row at
    // this q); rebuilt when the k walk enters a new row.  One set: registers;
    // more: the warp's shared-memory table, indexed by the lane's row slot.
    extern __shared__ float4 rowtab[];
    float4 row_m = make_float4(0.f, 0.f, 0.f, 0.f), row_p = row_m;
    // one set: the columns of the current row where the aperture test at
    // k - q (run_m) and at k + q (run_p) holds
    RowRun run_m{0.0f, 0.0f}, run_p{0.0f, 0.0f};
    const int lane = threadIdx.x & 31;
    float4* wtab = rowtab + (size_t)(threadIdx.x >> 5) * kRowSlots * 2 * row_tab_stride<MAXB>();
    int slot = 0, nslots = 1;
    int lead = 0;  // lanes 0..2*kRowSlots-1: the leading lane of row slot lane/2
    if constexpr (MAXB > 1) {
        const int prev_row = __shfl_up_sync(0xffffffffu, row, 1);
        const unsigned starts = __ballot_sync(0xffffffffu, lane == 0 || row != prev_row);
        slot = __popc(starts & ((2u << lane) - 1u)) - 1;
        nslots = __popc(starts);
        unsigned b = starts;
        for (int i = 0; i < (lane >> 1) && b; ++i) b &= b - 1u;
        lead = b ? __ffs(b) - 1 : 0;
    }
    const bool row_table = nslots <= kRowSlots;  // warp-uniform
    auto new_row = [&](float ky) {
        if constexpr (MAXB == 1) {
            row_m = chi_row(sb.s[0].h, __fsub_rn(__fsub_rn(ky, qy), sb.s[0].ty));
            row_p = chi_row(sb.s[0].h, __fsub_rn(__fadd_rn(ky, qy), sb.s[0].ty));
        } else {
            // lane 2 i + side fills slot i, trotter side `side` (0: k - q, 1: k + q)
            const float qs = __shfl_sync(0xffffffffu, qy, lead);
            __syncwarp();
            if (row_table && lane < 2 * nslots) {
                const float kq = (lane & 1) ? __fadd_rn(ky, qs) : __fsub_rn(ky, qs);
                float4* e = wtab + (size_t)lane * row_tab_stride<MAXB>();
#pragma unroll
                for (int s = 0; s < MAXB; ++s)
                    e[s] = chi_row(sb.s[s].h, __fsub_rn(kq, sb.s[s].ty));
            }
            __syncwarp();
        }
    };
    // chi(k -/+ q) of set s at vx = x, vy = y on trotter side m (true: k - q);
    // TAB: the warp's row table is in use (else the row form per term)
    auto chi_v = [&](auto tab, int s, bool m, float x, float y) -> float {
        if constexpr (MAXB == 1) {
            return chi_horner(sb.s[0].h[0], m ? row_m : row_p, x);
        } else if constexpr (decltype(tab)::value) {
            return chi_horner(sb.s[s].h[0], wtab[(size_t)(2 * slot + (m ? 0 : 1)) * row_tab_stride<MAXB>() + s], x);
        } else {
            return chi_horner(sb.s[s].h[0], chi_row(sb.s[s].h, y), x);
        }
    };

    // a k step's G: complex64 as loaded, or (herm16 word, scale bits),
    // dequantised only inside the branches that accumulate a term
    using GIn = std::conditional_t<FMT == kGC64, float2, uint2>;
    auto gval = [&](const GIn& gi) -> float2 {
        if constexpr (FMT == kGC64)
            return gi;
        else
            return sn16_unpack(gi.x, __fmul_rn(__uint_as_float(gi.y), kInv32767));
    };
    // the defocus-spread weight of set s for squared distances d2k (at k) and
    // d2o (at k -/+ q): gs times sinc(a_s (d2k - d2o)); without DEPTH, gs
    auto depth_w = [&](int s, float2 gs, float d2k, float d2o) -> float2 {
        if constexpr (DEPTH) {
            const float f = depth_sinc(sb.depth_a[s], __fsub_rn(d2k, d2o));
            return make_float2(__fmul_rn(gs.x, f), __fmul_rn(gs.y, f));
        } else {
            return gs;
        }
    };
    // the row state at a pixel that starts a detector row, or the split's
    // first pixel (uniform: every lane walks the same k): one set, the
    // aperture runs and the row polynomials; more sets, the row table
    constexpr bool RUNS = SHARED && MAXB == 1;
    auto row_enter = [&](float ky) {
        if constexpr (RUNS) {
            run_m = row_run(P.kxcol, P.ncol, P.inv_dk, P.ccol, ky, qx, qy, true, sb.s[0].tx, sb.s[0].ty, sb.r2);
            run_p = row_run(P.kxcol, P.ncol, P.inv_dk, P.ccol, ky, qx, qy, false, sb.s[0].tx, sb.s[0].ty, sb.r2);
        }
        new_row(ky);
    };
    auto step = [&](const GIn& g, float4 kd, const float* chk, auto tab) {
        const uint32_t am = __float_as_uint(kd.z);
        if constexpr (RUNS) {
            // one set: the aperture tests are comparisons with the row's
            // runs; the result is committed only on a single-overlap pixel
            const bool m = kd.x >= run_m.lo && kd.x <= run_m.hi;
            const bool p = kd.x >= run_p.lo && kd.x <= run_p.hi;
            const bool act = (am & 1u) && (m != p);
            // warp-uniform skip: lanes of a warp hold neighbouring q, so whole
            // warps often have no trotter pixel at this k
            if (__any_sync(0xffffffffu, act)) {
                // inactive lanes add an exact zero: gs = 0 * G, and every
                // later term is finite.  The side's offset: k_x - (-q_x) is
                // the same float as k_x + q_x
                const float qsx = m ? qx : -qx;
                const float sg = act ? (m ? 1.0f : -1.0f) : 0.0f;
                const float2 gv = gval(g);
                const float x = __fsub_rn(__fsub_rn(kd.x, qsx), sb.s[0].tx);
                float d2k = 0.0f, d2o = 0.0f;
                if constexpr (DEPTH) {
                    d2k = d2_f32(kd.x, kd.y, sb.s[0].tx, sb.s[0].ty);
                    d2o = d2_f32(__fsub_rn(kd.x, qsx), __fsub_rn(kd.y, m ? qy : -qy), sb.s[0].tx, sb.s[0].ty);
                }
                accumulate(acc[0], depth_w(0, make_float2(__fmul_rn(sg, gv.x), __fmul_rn(sg, gv.y)), d2k, d2o),
                           kd.w, chi_v(tab, 0, m, x, 0.f), m ? kTwoPi : -kTwoPi);
                cnt[0] += act ? 1 : 0;
            }
            return;
        }
        const float mx = __fsub_rn(kd.x, qx), my = __fsub_rn(kd.y, qy);
        const float px = __fadd_rn(kd.x, qx), py = __fadd_rn(kd.y, qy);
        if constexpr (SHARED) {
            // one tilt for all sets: the aperture tests are common, only the
            // row polynomial, the phase and the accumulation run per set
            if (am & 1u) {
                float mvx, mvy, pvx, pvy, d2m, d2p;
                const bool m = aperture_f32(mx, my, sb.s[0].tx, sb.s[0].ty, sb.r2, &mvx, &mvy, &d2m);
                const bool p = aperture_f32(px, py, sb.s[0].tx, sb.s[0].ty, sb.r2, &pvx, &pvy, &d2p);
                if (m != p) {
                    const float x = m ? mvx : pvx, y = m ? mvy : pvy;
                    const float2 gs = side_sign(gval(g), m);
                    const float tw = m ? kTwoPi : -kTwoPi;
                    const float d2k = DEPTH ? d2_f32(kd.x, kd.y, sb.s[0].tx, sb.s[0].ty) : 0.0f;
                    const float d2o = m ? d2m : d2p;
                    cnt[0] += 1;
                    float ck[MAXB];
                    const float4* cp = reinterpret_cast<const float4*>(chk);
#pragma unroll
                    for (int v4 = 0; v4 < (MAXB + 3) / 4; ++v4) {
                        const float4 c4 = cp[v4];
                        ck[4 * v4] = c4.x;
                        if (4 * v4 + 1 < MAXB) ck[4 * v4 + 1] = c4.y;
                        if (4 * v4 + 2 < MAXB) ck[4 * v4 + 2] = c4.z;
                        if (4 * v4 + 3 < MAXB) ck[4 * v4 + 3] = c4.w;
                    }
                    // every set's term runs unconditionally (sets past B
                    // are copies of set 0, their sums never written), so the
                    // sets' dependent chains can interleave.  With one tilt
                    // the spread factor depends on the set only through its
                    // depth: when all sets share it, it is taken once
                    if (DEPTH && sb.depth_shared) {
                        const float2 g1 = depth_w(0, gs, d2k, d2o);
#pragma unroll
                        for (int s = 0; s < MAXB; ++s)
                            accumulate(acc[s], g1, ck[s], chi_v(tab, s, m, x, y), tw);
                    } else {
#pragma unroll
                        for (int s = 0; s < MAXB; ++s)
                            accumulate(acc[s], depth_w(s, gs, d2k, d2o), ck[s], chi_v(tab, s, m, x, y), tw);
                    }
                }
            }
        } else {
            // sets with their own tilts: every set's two aperture tests first;
            // then, if any lane has a single-overlap pixel in any set, every
            // set's term, an inactive one with zero weight, so that the sets'
            // dependent chains can interleave (sets past B have no aperture
            // bits and never contribute)
            uint32_t mbits = 0u, pbits = 0u;
#pragma unroll
            for (int s = 0; s < MAXB; ++s) {
                float vx, vy;
                mbits |= (aperture_f32(mx, my, sb.s[s].tx, sb.s[s].ty, sb.r2, &vx, &vy) ? 1u : 0u) << s;
                pbits |= (aperture_f32(px, py, sb.s[s].tx, sb.s[s].ty, sb.r2, &vx, &vy) ? 1u : 0u) << s;
            }
            const uint32_t actb = am & (mbits ^ pbits);
            if (__any_sync(0xffffffffu, actb != 0u)) {
                const float2 gv = gval(g);
#pragma unroll
                for (int s = 0; s < MAXB; ++s) {
                    const bool m = (mbits >> s) & 1u, act = (actb >> s) & 1u;
                    // the side's (v_x, v_y) as the aperture test formed them
                    const float x = __fsub_rn(m ? mx : px, sb.s[s].tx), y = __fsub_rn(m ? my : py, sb.s[s].ty);
                    const float2 gs = act ? side_sign(gv, m) : make_float2(0.f, 0.f);
                    const float d2k = DEPTH ? d2_f32(kd.x, kd.y, sb.s[s].tx, sb.s[s].ty) : 0.0f;
                    const float d2o = DEPTH ? __fadd_rn(__fmul_rn(x, x), __fmul_rn(y, y)) : 0.0f;
                    accumulate(acc[s], depth_w(s, gs, d2k, d2o), chk[s], chi_v(tab, s, m, x, y),
                               m ? kTwoPi : -kTwoPi);
                    cnt[s] += act ? 1 : 0;
                }
            }
        }
    };
    // the k tables of a chunk of kKChunk pixels are staged in shared memory by
    // the whole block (every thread walks the same k), so a step reads them
    // as short broadcasts and the registers go to G loads in flight
    __shared__ float4 s_ktab[kKChunk];
    __shared__ float4 s_chik[MAXB > 1 ? kKChunk * kChiStride / 4 : 1];
    // A chunk is walked in row segments: the row state is rebuilt once at a
    // segment's start (a pixel marked kRowStart, or the split's first pixel),
    // and within a segment the k steps run in batches of U with no row check.
    auto walk = [&](auto tab, int kc0, int kcn) {
        constexpr int U = red_unroll<MAXB>();
        constexpr bool ROWS = decltype(tab)::value;
        [[maybe_unused]] const float2* gk = gp + (size_t)kc0 * gstride;
        [[maybe_unused]] const uint32_t* wk = gw + (size_t)kc0 * gstride;
        [[maybe_unused]] const float* sk = gsc + kc0;
        int i = 0;
#pragma unroll 1
        while (i < kcn) {
            int e = kcn;  // end of this segment
            if constexpr (ROWS) {
                if (i > 0 || kc0 == kb || (__float_as_uint(s_ktab[0].z) & kRowStart)) row_enter(s_ktab[i].y);
                // the next row start within the chunk (uniform search)
#pragma unroll 1
                for (int j0 = i + 1; j0 < kcn; j0 += 32) {
                    const int j = j0 + lane;
                    const unsigned bal =
                        __ballot_sync(0xffffffffu, j < kcn && (__float_as_uint(s_ktab[j].z) & kRowStart));
                    if (bal) {
                        e = j0 + __ffs(bal) - 1;
                        break;
                    }
                }
            }
#pragma unroll 1
            for (; i + U <= e; i += U) {
                GIn g[U];
                if constexpr (FMT == kGC64) {
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        g[u] = valid ? __ldcs(gk + (size_t)(i + u) * gstride) : make_float2(0.f, 0.f);
                } else {
#pragma unroll
                    for (int u = 0; u < U; ++u) g[u].x = valid ? __ldcs(wk + (size_t)(i + u) * gstride) : 0u;
#pragma unroll
                    for (int u = 0; u < U; ++u) g[u].y = __float_as_uint(__ldg(sk + i + u));
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
                    step(g[u], s_ktab[i + u], reinterpret_cast<const float*>(s_chik) + (i + u) * kChiStride, tab);
            }
#pragma unroll 1
            for (; i < e; ++i) {
                GIn g;
                if constexpr (FMT == kGC64)
                    g = valid ? __ldcs(gk + (size_t)i * gstride) : make_float2(0.f, 0.f);
                else
                    g = make_uint2(valid ? __ldcs(wk + (size_t)i * gstride) : 0u, __float_as_uint(__ldg(sk + i)));
                step(g, s_ktab[i], reinterpret_cast<const float*>(s_chik) + i * kChiStride, tab);
            }
        }
    };
#pragma unroll 1
    for (int kc0 = kb; kc0 < ke; kc0 += kKChunk) {
        const int kcn = min(kKChunk, ke - kc0);
        __syncthreads();  // every read of the previous chunk's tables is done
        for (int i = threadIdx.x; i < kcn; i += kRedThreads) s_ktab[i] = __ldg(P.ktab + kc0 + i);
        if constexpr (MAXB > 1) {
            const float4* src = reinterpret_cast<const float4*>(P.chik) + (size_t)kc0 * (kChiStride / 4);
            for (int i = threadIdx.x; i < kcn * (kChiStride / 4); i += kRedThreads) s_chik[i] = __ldg(src + i);
        }
        __syncthreads();
        if (MAXB == 1 || row_table)
            walk(std::true_type{}, kc0, kcn);
        else
            walk(std::false_type{}, kc0, kcn);
    }
    if (valid) {
#pragma unroll
        for (int s = 0; s < MAXB; ++s) {
            if (s < sb.B) {
                const size_t o = ((size_t)split * sb.B + s) * P.nq + qi;
                P.Opart[o] = acc[s];
                P.Npart[o] = SHARED ? cnt[0] : cnt[s];
            }
        }
    }
}



template <int MAXB, bool SHARED, int FMT, bool DEPTH>
static void launch_reduce_bsf(const RedLaunch& P, const SetBatch& sb, dim3 grid, cudaStream_t st) {
    constexpr size_t smem = red_smem_bytes<MAXB>();
    if (smem > 48 * 1024)  // set on every call: the attribute belongs to the current device's context
        cudaFuncSetAttribute(ssb_reduce<MAXB, SHARED, FMT, DEPTH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    ssb_reduce<MAXB, SHARED, FMT, DEPTH><<<grid, kRedThreads, smem, st>>>(P, sb);
}

template <int MAXB, int FMT, bool DEPTH>
static void launch_reduce_bf(const RedLaunch& P, const SetBatch& sb, dim3 grid, cudaStream_t st) {
    if (P.shared_tilt)
        launch_reduce_bsf<MAXB, true, FMT, DEPTH>(P, sb, grid, st);
    else
        launch_reduce_bsf<MAXB, false, FMT, DEPTH>(P, sb, grid, st);
}

template <int FMT, bool DEPTH>
static void launch_reduce_f(const RedLaunch& P, const SetBatch& sb, dim3 grid, cudaStream_t st) {
    if (sb.B == 1)
        launch_reduce_bf<1, FMT, DEPTH>(P, sb, grid, st);
    else if (sb.B == 2)
        launch_reduce_bf<2, FMT, DEPTH>(P, sb, grid, st);
    else if (sb.B <= 4)
        launch_reduce_bf<4, FMT, DEPTH>(P, sb, grid, st);
    else
        launch_reduce_bf<8, FMT, DEPTH>(P, sb, grid, st);
}

template <bool DEPTH>
static cudaError_t launch_reduce_t(const RedLaunch& P, const SetBatch& sb, cudaStream_t st) {
    dim3 grid((P.nq + kRedThreads - 1) / kRedThreads, P.nsplit);
    if (P.g.fmt == kGSN16)
        launch_reduce_f<kGSN16, DEPTH>(P, sb, grid, st);
    else
        launch_reduce_f<kGC64, DEPTH>(P, sb, grid, st);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ssb
