// reduce.cu -- trotter-masked, aberration-weighted reduction over bright-field
// pixels, spectrum assembly + complex-to-real inverse + atan2, and the band score.
//
// Per (q, k, set) term (quantem.gpu "Tilt-corrected SSB on CUDA", sections
// "Where the time went" and "Changes"): three aperture tests decide the
// trotter class; a single-overlap pixel adds G(q,k) w to O(q) and 1 to N(q),
// with w = exp(-i(chi(k) - chi(k-q))) on T- and -exp(+i(chi(k) - chi(k+q))) on
// T+.  Per-set accumulators live in registers (the set loop is unrolled to a
// compile-time maximum with a uniform b < B guard); chi(k) and the aperture at
// k are computed once per call into k-only tables.
//
// chi(k -/+ q) is a quartic in v_x along a detector row (v_y is fixed there
// for a given q and trotter side): its coefficients are rebuilt once per row
// and each term costs 4 FMAs per set.  When all sets share one tilt (the
// batched-scoring case) the three aperture tests are computed once per (q, k)
// and only the row polynomial, the phase and the accumulation run per set.
//
// Thread <-> q layout: consecutive lanes own consecutive half-plane entries,
// so each k step reads G[k][q..q+31] as one coalesced 256-byte segment and the
// sum over k needs no cross-thread reduction.  The k range is split across
// grid.y; partial sums are added in a fixed order by the finalize kernel, so
// results are deterministic and independent of the number of sets B.
#include <type_traits>

#include "internal.cuh"

namespace ssb {

// ---------------------------------------------------------------------------
// k-only tables: float32 k, aperture bit per set, chi_s(k) in turns
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
ssb_prep(const int32_t* __restrict__ bf_idx, int n_bf, int det_x, double cy, double cx, double dk, SetBatch sb,
         float4* __restrict__ ktab, float* __restrict__ chik, GView g, double* __restrict__ dcpart) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (dcpart) {
        // sum_k Re G(0, k) for the image offset a: per-block partial in
        // float64, added in a fixed order by the image kernel (entry 0 of a
        // half plane is q = 0, in the scale block of row 0)
        __shared__ double red[256];
        float g0 = 0.f;
        if (k < n_bf) {
            if (g.fmt == kGSN16)
                g0 = sn16_unpack(static_cast<const uint32_t*>(g.G)[(size_t)k * g.stride],
                                 __fmul_rn(g.scale[k], kInv32767)).x;
            else
                g0 = static_cast<const float2*>(g.G)[(size_t)k * g.stride].x;
        }
        red[threadIdx.x] = (double)g0;
        __syncthreads();
        for (int w = 128; w > 0; w >>= 1) {
            if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
            __syncthreads();
        }
        if (threadIdx.x == 0) dcpart[blockIdx.x] = red[0];
    }
    if (k >= n_bf) return;
    const int idx = bf_idx[k];
    const int i = idx / det_x, j = idx - i * det_x;
    const float kx = __double2float_rn(__dmul_rn(__dsub_rn((double)j, cx), dk));
    const float ky = __double2float_rn(__dmul_rn(__dsub_rn((double)i, cy), dk));
    uint32_t bits = 0;
    float chi0 = 0.f;
    for (int s = 0; s < kChiStride; ++s) {
        float c = 0.f;
        if (s < sb.B) {
            float vx, vy;
            const bool a = aperture_f32(kx, ky, sb.s[s].tx, sb.s[s].ty, sb.r2, &vx, &vy);
            bits |= (a ? 1u : 0u) << s;
            c = a ? chi_turns(sb.s[s].c, vx, vy) : 0.f;
        }
        if (s == 0) chi0 = c;
        chik[(size_t)k * kChiStride + s] = c;
    }
    ktab[k] = make_float4(kx, ky, __uint_as_float(bits), chi0);
}

cudaError_t launch_prep(const int32_t* bf_idx, int n_bf, int det_x, double cy, double cx, double dk,
                        const SetBatch& sb, float4* ktab, float* chik, const GView& g,
                        double* dcpart, cudaStream_t st) {
    ssb_prep<<<(n_bf + 255) / 256, 256, 0, st>>>(bf_idx, n_bf, det_x, cy, cx, dk, sb, ktab, chik, g, dcpart);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// fused reduction
// ---------------------------------------------------------------------------
constexpr int kRedThreads = 256;
constexpr int kKChunk = 64;  // k pixels whose tables a block stages at a time
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

template <int MAXB, bool SHARED, int FMT>
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
    float cur_ky = __int_as_float(0x7fc00000);  // NaN: no row yet
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
                    if (s < sb.B) e[s] = chi_row(sb.s[s].h, __fsub_rn(kq, sb.s[s].ty));
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
    auto step = [&](const GIn& g, float4 kd, const float* chk, auto tab) {
        if (decltype(tab)::value && kd.y != cur_ky) {  // uniform: every lane walks the same k
            new_row(kd.y);
            cur_ky = kd.y;
        }
        const uint32_t am = __float_as_uint(kd.z);
        const float mx = __fsub_rn(kd.x, qx), my = __fsub_rn(kd.y, qy);
        const float px = __fadd_rn(kd.x, qx), py = __fadd_rn(kd.y, qy);
        if constexpr (SHARED && MAXB == 1) {
            // one set: no branch, so the unrolled k steps can overlap; the
            // result is committed only on a single-overlap pixel
            float mvx, mvy, pvx, pvy;
            const bool m = aperture_f32(mx, my, sb.s[0].tx, sb.s[0].ty, sb.r2, &mvx, &mvy);
            const bool p = aperture_f32(px, py, sb.s[0].tx, sb.s[0].ty, sb.r2, &pvx, &pvy);
            const bool act = (am & 1u) && (m != p);
            // warp-uniform skip: lanes of a warp hold neighbouring q, so whole
            // warps often have no trotter pixel at this k
            if (__any_sync(0xffffffffu, act)) {
                // inactive lanes add an exact zero: gs = 0 * G, and every
                // later term is finite
                const float sg = act ? (m ? 1.0f : -1.0f) : 0.0f;
                const float2 gv = gval(g);
                accumulate(acc[0], make_float2(__fmul_rn(sg, gv.x), __fmul_rn(sg, gv.y)), kd.w,
                           chi_v(tab, 0, m, m ? mvx : pvx, 0.f), m ? kTwoPi : -kTwoPi);
                cnt[0] += act ? 1 : 0;
            }
        } else if constexpr (SHARED) {
            // one tilt for all sets: the aperture tests are common, only the
            // row polynomial, the phase and the accumulation run per set
            if (am & 1u) {
                float mvx, mvy, pvx, pvy;
                const bool m = aperture_f32(mx, my, sb.s[0].tx, sb.s[0].ty, sb.r2, &mvx, &mvy);
                const bool p = aperture_f32(px, py, sb.s[0].tx, sb.s[0].ty, sb.r2, &pvx, &pvy);
                if (m != p) {
                    const float x = m ? mvx : pvx, y = m ? mvy : pvy;
                    const float2 gs = side_sign(gval(g), m);
                    const float tw = m ? kTwoPi : -kTwoPi;
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
#pragma unroll
                    for (int s = 0; s < MAXB; ++s)
                        if (s < sb.B) accumulate(acc[s], gs, ck[s], chi_v(tab, s, m, x, y), tw);
                }
            }
        } else {
#pragma unroll
            for (int s = 0; s < MAXB; ++s) {
                if (s < sb.B && ((am >> s) & 1u)) {
                    float mvx, mvy, pvx, pvy;
                    const bool m = aperture_f32(mx, my, sb.s[s].tx, sb.s[s].ty, sb.r2, &mvx, &mvy);
                    const bool p = aperture_f32(px, py, sb.s[s].tx, sb.s[s].ty, sb.r2, &pvx, &pvy);
                    if (m != p) {
                        const float cq = chi_v(tab, s, m, m ? mvx : pvx, m ? mvy : pvy);
                        accumulate(acc[s], side_sign(gval(g), m), chk[s], cq,
                                   m ? kTwoPi : -kTwoPi);
                        cnt[s] += 1;
                    }
                }
            }
        }
    };

    // the k tables of a chunk of kKChunk pixels are staged in shared memory by
    // the whole block (every thread walks the same k), so a step reads them
    // as short broadcasts and the registers go to G loads in flight
    __shared__ float4 s_ktab[kKChunk];
    __shared__ float4 s_chik[MAXB > 1 ? kKChunk * kChiStride / 4 : 1];
    auto walk = [&](auto tab, int kc0, int kcn) {
        constexpr int U = red_unroll<MAXB>();
        [[maybe_unused]] const float2* gk = gp + (size_t)kc0 * gstride;
        [[maybe_unused]] const uint32_t* wk = gw + (size_t)kc0 * gstride;
        [[maybe_unused]] const float* sk = gsc + kc0;
        int i = 0;
#pragma unroll 1
        for (; i + U <= kcn; i += U) {
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
        for (; i < kcn; ++i) {
            GIn g;
            if constexpr (FMT == kGC64)
                g = valid ? __ldcs(gk + (size_t)i * gstride) : make_float2(0.f, 0.f);
            else
                g = make_uint2(valid ? __ldcs(wk + (size_t)i * gstride) : 0u, __float_as_uint(__ldg(sk + i)));
            step(g, s_ktab[i], reinterpret_cast<const float*>(s_chik) + i * kChiStride, tab);
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

template <int MAXB, bool SHARED, int FMT>
static void launch_reduce_bsf(const RedLaunch& P, const SetBatch& sb, dim3 grid, cudaStream_t st) {
    constexpr size_t smem = red_smem_bytes<MAXB>();
    if (smem > 48 * 1024) {
        static bool opted = false;  // idempotent attribute; a racing second set is harmless
        if (!opted) {
            cudaFuncSetAttribute(ssb_reduce<MAXB, SHARED, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
            opted = true;
        }
    }
    ssb_reduce<MAXB, SHARED, FMT><<<grid, kRedThreads, smem, st>>>(P, sb);
}

template <int MAXB, int FMT>
static void launch_reduce_bf(const RedLaunch& P, const SetBatch& sb, dim3 grid, cudaStream_t st) {
    if (P.shared_tilt)
        launch_reduce_bsf<MAXB, true, FMT>(P, sb, grid, st);
    else
        launch_reduce_bsf<MAXB, false, FMT>(P, sb, grid, st);
}

template <int FMT>
static void launch_reduce_f(const RedLaunch& P, const SetBatch& sb, dim3 grid, cudaStream_t st) {
    if (sb.B == 1)
        launch_reduce_bf<1, FMT>(P, sb, grid, st);
    else if (sb.B == 2)
        launch_reduce_bf<2, FMT>(P, sb, grid, st);
    else if (sb.B <= 4)
        launch_reduce_bf<4, FMT>(P, sb, grid, st);
    else
        launch_reduce_bf<8, FMT>(P, sb, grid, st);
}

cudaError_t launch_reduce(const RedLaunch& P, const SetBatch& sb, cudaStream_t st) {
    dim3 grid((P.nq + kRedThreads - 1) / kRedThreads, P.nsplit);
    if (P.g.fmt == kGSN16)
        launch_reduce_f<kGSN16>(P, sb, grid, st);
    else
        launch_reduce_f<kGC64>(P, sb, grid, st);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// partial sums -> O, N (fixed order over splits)
// ---------------------------------------------------------------------------
__global__ void ssb_finalize(const float2* __restrict__ Opart, const int* __restrict__ Npart,
                                int nsplit, int B, int nq, float2* __restrict__ O,
                                int32_t* __restrict__ N) {
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)B * nq;
    if (t >= total) return;
    float2 a = Opart[t];
    int c = Npart[t];
    for (int sp = 1; sp < nsplit; ++sp) {
        const float2 v = Opart[(size_t)sp * total + t];
        a.x = __fadd_rn(a.x, v.x);
        a.y = __fadd_rn(a.y, v.y);
        c += Npart[(size_t)sp * total + t];
    }
    O[t] = a;
    N[t] = c;
}

cudaError_t launch_finalize(const float2* Opart, const int* Npart, int nsplit, int B, int nq,
                            float2* O, int32_t* N, cudaStream_t st) {
    const size_t total = (size_t)B * nq;
    ssb_finalize<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(Opart, Npart, nsplit, B, nq, O, N);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// phase image: S = O/N, Nyquist row/column and DC zeroed, B = -i S,
// y = inverse C2C along q_y (unnormalised), b = C2R along q_x (numpy irfft
// semantics), b /= n^2, phase = atan2(b, a), a = mean_k G(0,k) / n^2
// ---------------------------------------------------------------------------
constexpr int kPhaseThreads = 256;

template <int N>
__global__ void __launch_bounds__(kPhaseThreads)
ssb_c2r_cols(const float2* __restrict__ O, const int32_t* __restrict__ Nn, float2* __restrict__ Y,
                const float2* __restrict__ twg) {
    constexpr int H = N / 2 + 1;
    constexpr int CW = (N / 2 >= 16) ? 16 : N / 2;
    constexpr int NG = (N / 2) / CW;
    constexpr int CS = N + 1;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float2* tw = reinterpret_cast<float2*>(smem_raw);
    float2* cols = tw + N;
    const int g = blockIdx.x;
    const int c0 = g * CW;
    const int nc = CW + ((g == NG - 1) ? 1 : 0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = kPhaseThreads / 32;
    for (int m = threadIdx.x; m < N; m += kPhaseThreads) tw[m] = twg[m];
    for (int idx = threadIdx.x; idx < N * nc; idx += kPhaseThreads) {
        const int row = idx / nc, c = idx - row * nc;
        const int col = c0 + c;
        const int e = row * H + col;
        float2 b = make_float2(0.f, 0.f);
        const int cnt = Nn[e];
        if (cnt > 0 && row != N / 2 && col != N / 2 && e != 0) {
            const float2 o = O[e];
            const float sx = __fdiv_rn(o.x, (float)cnt), sy = __fdiv_rn(o.y, (float)cnt);
            b = make_float2(sy, -sx);  // -i S
        }
        cols[c * CS + row] = cconj(b);  // inverse via conj(FFT(conj(.)))
    }
    __syncthreads();
    for (int c = warp; c < nc; c += NW) fft_warp<N, 1>(cols + c * CS, tw, lane);
    __syncthreads();
    for (int idx = threadIdx.x; idx < N * nc; idx += kPhaseThreads) {
        const int row = idx / nc, c = idx - row * nc;
        Y[(size_t)row * H + c0 + c] = cconj(cols[c * CS + row]);
    }
}

template <int N>
__global__ void __launch_bounds__(kPhaseThreads)
ssb_c2r_rows(const float2* __restrict__ Y, const double* __restrict__ dcpart, int ndc, int n_bf,
                const float2* __restrict__ twg, float* __restrict__ phase) {
    constexpr int L = N / 2;
    constexpr int H = N / 2 + 1;
    constexpr int RPB = kPhaseThreads / 32;  // rows per block, one warp each
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float2* tw = reinterpret_cast<float2*>(smem_raw);
    float2* zs = tw + N;  // RPB rows of L points
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int m = threadIdx.x; m < N; m += kPhaseThreads) tw[m] = twg[m];
    double dc = 0.0;
    for (int sp = 0; sp < ndc; ++sp) dc += dcpart[sp];
    const float a = (float)(dc / (double)n_bf / ((double)N * (double)N));
    __syncthreads();
    const int row = blockIdx.x * RPB + warp;
    if (row >= N) return;
    const float2* y = Y + (size_t)row * H;
    float2* z = zs + warp * L;
    // Z[k] = E[k] + i O[k], E = X[k] + conj X[L-k], O = (X[k] - conj X[L-k]) W^-k,
    // with the imaginary parts of X[0] and X[L] dropped
    for (int k = lane; k < L; k += 32) {
        float2 xk = y[k];
        float2 xl = y[L - k];
        if (k == 0) {
            xk.y = 0.f;
            xl.y = 0.f;
        }
        const float2 xc = cconj(xl);
        const float2 e = cadd(xk, xc);
        const float2 o = cmul(csub(xk, xc), cconj(tw[k]));
        const float2 zz = cadd(e, cmul_pi(o));
        z[k] = cconj(zz);  // inverse via conj trick
    }
    __syncwarp();
    fft_warp<L, 2>(z, tw, lane);
    const float inv = 1.0f / ((float)N * (float)N);
    float* out = phase + (size_t)row * N;
    for (int m = lane; m < L; m += 32) {
        const float2 v = cconj(z[m]);
        out[2 * m] = atan2f(v.x * inv, a);
        out[2 * m + 1] = atan2f(v.y * inv, a);
    }
}

template <int N>
static cudaError_t phase_n(const float2* O, const int32_t* Nn, const double* dcpart, int nsplit,
                           int n_bf, float2* Y, const float2* tw, float* phase, cudaStream_t st) {
    constexpr int CW = (N / 2 >= 16) ? 16 : N / 2;
    constexpr int NG = (N / 2) / CW;
    const size_t cs = (size_t)N * sizeof(float2) + (size_t)(CW + 1) * (N + 1) * sizeof(float2);
    const size_t rs = (size_t)N * sizeof(float2) + (size_t)(kPhaseThreads / 32) * (N / 2) * sizeof(float2);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ssb_c2r_cols<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)cs)) != cudaSuccess)
        return e;
    ssb_c2r_cols<N><<<NG, kPhaseThreads, cs, st>>>(O, Nn, Y, tw);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    constexpr int RPB = kPhaseThreads / 32;
    ssb_c2r_rows<N><<<(N + RPB - 1) / RPB, kPhaseThreads, rs, st>>>(Y, dcpart, nsplit, n_bf, tw, phase);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_phase(const float2* O, const int32_t* Nn, const double* dcpart, int nsplit, int n_bf,
                         int n, float2* Y, const float2* tw, float* phase, cudaStream_t st) {
    switch (n) {
        case 8: return phase_n<8>(O, Nn, dcpart, nsplit, n_bf, Y, tw, phase, st);
        case 16: return phase_n<16>(O, Nn, dcpart, nsplit, n_bf, Y, tw, phase, st);
        case 32: return phase_n<32>(O, Nn, dcpart, nsplit, n_bf, Y, tw, phase, st);
        case 64: return phase_n<64>(O, Nn, dcpart, nsplit, n_bf, Y, tw, phase, st);
        case 128: return phase_n<128>(O, Nn, dcpart, nsplit, n_bf, Y, tw, phase, st);
        case 256: return phase_n<256>(O, Nn, dcpart, nsplit, n_bf, Y, tw, phase, st);
        case 512: return phase_n<512>(O, Nn, dcpart, nsplit, n_bf, Y, tw, phase, st);
        case 1024: return phase_n<1024>(O, Nn, dcpart, nsplit, n_bf, Y, tw, phase, st);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// sum_k Re G(0,k) from the per-256-pixel partials, in the order the image
// kernel adds them (so one shard holding every pixel reproduces its offset)
// ---------------------------------------------------------------------------
__global__ void ssb_dc_total(const double* __restrict__ part, int nparts, double* __restrict__ total) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    double dc = 0.0;
    for (int sp = 0; sp < nparts; ++sp) dc += part[sp];
    total[0] = dc;
}

cudaError_t launch_dc_total(const double* part, int nparts, double* total, cudaStream_t st) {
    ssb_dc_total<<<1, 32, 0, st>>>(part, nparts, total);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// score_s = sum_q |O_s(q)|^2 / sum_q N_s(q), one block per set, float64 sums
// ---------------------------------------------------------------------------
__global__ void ssb_score(const float2* __restrict__ O, const int32_t* __restrict__ Nn, int nq,
                             double* __restrict__ score) {
    __shared__ double s_num[256];
    __shared__ long long s_den[256];
    const int s = blockIdx.x;
    double num = 0.0;
    long long den = 0;
    for (int q = threadIdx.x; q < nq; q += 256) {
        const float2 o = O[(size_t)s * nq + q];
        num += (double)o.x * (double)o.x + (double)o.y * (double)o.y;
        den += Nn[(size_t)s * nq + q];
    }
    s_num[threadIdx.x] = num;
    s_den[threadIdx.x] = den;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) {
            s_num[threadIdx.x] += s_num[threadIdx.x + w];
            s_den[threadIdx.x] += s_den[threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) score[s] = s_den[0] > 0 ? s_num[0] / (double)s_den[0] : 0.0;
}

cudaError_t launch_score(const float2* O, const int32_t* Nn, int B, int nq, double* score,
                         cudaStream_t st) {
    ssb_score<<<B, 256, 0, st>>>(O, Nn, nq, score);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ssb
