// moments.cu -- per-BF phase moments: the exact mean(angle) path.
//
// For every bright-field pixel k the aberration-corrected plane
// S_k(q) = G(q,k) w(q,k) (its trotter pixels, 0 elsewhere) is brought back to
// real space as the image b_k = irfft2(-i S_k), and the per-pixel angle
// atan2(b_k, a_k), a_k = Re G(0,k) / n^2, is reduced to its mean and
// population variance over k.  Source: quantem.gpu "Historical WebGPU G(q,k)
// memory experiment", section "Object-redraw fast path" (mean(angle(object))
// over BF pixels, the variance for the loss); "Tilt-corrected SSB on CUDA",
// sections "Changes" (Loss path: the corrected plane is written straight from
// the stored half plane and the angles are reduced as they are read) and "Open"
// (the corrected spectrum of a real image is anti-Hermitian except at DC, so a
// half-plane complex-to-real transform gives the image).
//
// Chunks of kMomChunk BF pixels stay in L2 through three kernels:
//   1. ssb_correct: per (q, k) the same trotter tests, chi(k -/+ q) and term
//      arithmetic as the one-set reduction, written as -i S_k(q) instead of
//      summed (0 off the trotters, at DC and on the Nyquist row and column);
//   2. ssb_inv_cols: the inverse C2C along q_y of every column of every plane
//      of the chunk, in place;
//   3. ssb_inv_rows_moments: the C2R along q_x of each row, atan2 and the sums
//      of the angle and its square (float32 in shared memory over the block's
//      planes of the chunk).  Block (row group, plane group p) owns the same
//      pixels of partial sum p in every chunk and adds its planes in order,
//      so the sums are deterministic; ssb_moments_final adds the kMomGroups
//      float64 partial sums in a fixed order.
#include "internal.cuh"

namespace ssb {

constexpr int kMomThreads = 256;

// one k of a stored G at half-plane entry e of row `row` (herm16: dequantised);
// STREAM: read once, evict first, so G passing through does not push the
// chunk and the partial sums out of L2
template <bool STREAM = false>
__device__ __forceinline__ float2 g_entry(const GView& g, int n_bf, int k, size_t e, int row) {
    if (g.fmt == kGSN16) {
        const uint32_t* p = static_cast<const uint32_t*>(g.G) + (size_t)k * g.stride + e;
        const uint32_t w = STREAM ? __ldcs(p) : *p;
        const float s = g.scale[(size_t)(g.srows == 1 ? row : 0) * n_bf + k];
        return sn16_unpack(w, __fmul_rn(s, kInv32767));
    }
    const float2* p = static_cast<const float2*>(g.G) + (size_t)k * g.stride + e;
    return STREAM ? __ldcs(p) : *p;
}

// 1. Y[kk][e] = -i S_{k0+kk}(q_e): thread e of block row y walks BF pixels
// kk = y, y + kMomKSplit, ... of the chunk (q and its row decoded once), the
// G loads of kMomUnroll pixels issued together
constexpr int kMomKSplit = 4;
constexpr int kMomUnroll = 4;

__global__ void __launch_bounds__(kMomThreads)
ssb_correct(GView g, int n_bf, const float4* __restrict__ ktab, SetBatch sb, int n, double dq, int k0, int kc,
            float2* __restrict__ Y) {
    const int H = n / 2 + 1;
    const int nH = n * H;
    const int e = blockIdx.x * kMomThreads + threadIdx.x;
    if (e >= nH) return;
    const int row = e / H, col = e - row * H;
    const int fy = row < n / 2 ? row : row - n;
    const bool live = e != 0 && row != n / 2 && col != n / 2;
    const float qx = __double2float_rn(__dmul_rn((double)col, dq));
    const float qy = __double2float_rn(__dmul_rn((double)fy, dq));
    const SetParams& sp = sb.s[0];
    for (int kb = blockIdx.y; kb < kc; kb += kMomKSplit * kMomUnroll) {
        float2 gv[kMomUnroll];
#pragma unroll
        for (int u = 0; u < kMomUnroll; ++u) {
            const int kk = kb + u * kMomKSplit;
            gv[u] = kk < kc ? g_entry<true>(g, n_bf, k0 + kk, (size_t)e, row) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kMomUnroll; ++u) {
            const int kk = kb + u * kMomKSplit;
            if (kk >= kc) break;
            float2 out = make_float2(0.f, 0.f);
            const float4 kd = ktab[k0 + kk];
            if (live && (__float_as_uint(kd.z) & 1u)) {
                float mvx, mvy, pvx, pvy;
                const bool m =
                    aperture_f32(__fsub_rn(kd.x, qx), __fsub_rn(kd.y, qy), sp.tx, sp.ty, sb.r2, &mvx, &mvy);
                const bool p =
                    aperture_f32(__fadd_rn(kd.x, qx), __fadd_rn(kd.y, qy), sp.tx, sp.ty, sb.r2, &pvx, &pvy);
                if (m != p) {
                    const float chiq = chi_horner(sp.h[0], chi_row(sp.h, m ? mvy : pvy), m ? mvx : pvx);
                    float2 acc = make_float2(0.f, 0.f);
                    accumulate(acc, side_sign(gv[u], m), kd.w, chiq, m ? kTwoPi : -kTwoPi);
                    out = cmul_mi(acc);
                }
            }
            Y[(size_t)kk * nH + e] = out;
        }
    }
}

// 2. inverse C2C along q_y, in place: item (plane, column group of CW), a
// grid of resident blocks walking the chunk's items
template <int N>
__host__ __device__ constexpr int inv_cols_width() { return (N / 2 >= 8) ? 8 : N / 2; }

template <int N>
__global__ void __launch_bounds__(kMomThreads)
ssb_inv_cols(float2* __restrict__ Y, const float2* __restrict__ twg, int items) {
    constexpr int H = N / 2 + 1;
    constexpr int CW = inv_cols_width<N>();
    constexpr int NG = (N / 2) / CW;
    // column stride N + 4 and rows stored swizzled: the transposes and the
    // FFT passes hit each bank pair at most twice per warp
    constexpr int CS = N + 4;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float2* tw = reinterpret_cast<float2*>(smem_raw);
    float2* cols = tw + N;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = kMomThreads / 32;
    for (int m = threadIdx.x; m < N; m += kMomThreads) tw[m] = twg[m];
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        __syncthreads();  // the previous item's columns are written back
        const int grp = it % NG;
        float2* y = Y + (size_t)(it / NG) * N * H;
        const int c0 = grp * CW;
        const int nc = CW + ((grp == NG - 1) ? 1 : 0);
        // CW columns per group (compile-time index split), plus column N/2
        // in the last group; inverse via conj(FFT(conj(.)))
        if constexpr ((N * CW) % kMomThreads == 0) {
            // every load of the item in flight at once, then into shared memory
            constexpr int LPT = N * CW / kMomThreads;
            float2 v[LPT];
#pragma unroll
            for (int i = 0; i < LPT; ++i) {
                const int idx = threadIdx.x + i * kMomThreads;
                v[i] = y[(size_t)(idx / CW) * H + c0 + idx % CW];
            }
#pragma unroll
            for (int i = 0; i < LPT; ++i) {
                const int idx = threadIdx.x + i * kMomThreads;
                cols[(idx % CW) * CS + swz(idx / CW)] = cconj(v[i]);
            }
        } else {
            for (int idx = threadIdx.x; idx < N * CW; idx += kMomThreads) {
                const int row = idx / CW, c = idx % CW;
                cols[c * CS + swz(row)] = cconj(y[(size_t)row * H + c0 + c]);
            }
        }
        if (nc > CW)
            for (int row = threadIdx.x; row < N; row += kMomThreads)
                cols[CW * CS + swz(row)] = cconj(y[(size_t)row * H + N / 2]);
        __syncthreads();
        for (int c = warp; c < nc; c += NW) fft_warp<N, 1, true>(cols + c * CS, tw, lane);
        __syncthreads();
        for (int idx = threadIdx.x; idx < N * CW; idx += kMomThreads) {
            const int row = idx / CW, c = idx % CW;
            y[(size_t)row * H + c0 + c] = cconj(cols[c * CS + swz(row)]);
        }
        if (nc > CW)
            for (int row = threadIdx.x; row < N; row += kMomThreads)
                y[(size_t)row * H + N / 2] = cconj(cols[CW * CS + swz(row)]);
    }
}

// 3. C2R along q_x (numpy irfft semantics), atan2, moment sums: block
// (8 rows, plane group p) walks planes [p * per, (p + 1) * per) of the chunk
constexpr int kMomGroups = 8;   // 8 float64 (sum, square) images: 33.5 MB at n = 512
constexpr int kMomChunk = 64;   // 64 corrected half planes: 67 MB; both stay in L2

template <int N>
__global__ void __launch_bounds__(kMomThreads)
ssb_inv_rows_moments(const float2* __restrict__ Y, int kc, GView g, int n_bf, int k0,
                     const float2* __restrict__ twg, double2* __restrict__ part) {
    constexpr int L = N / 2;
    constexpr int H = N / 2 + 1;
    constexpr int RPB = kMomThreads / 32;
    constexpr int PER = (L + 31) / 32;  // outputs pairs per lane
    // shared memory: twiddles, one row of L points per warp, and per warp
    // the running (sum, sum of squares) of its row's N outputs
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float2* tw = reinterpret_cast<float2*>(smem_raw);
    float2* zs = tw + N;
    float2* acc = zs + RPB * L;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int m = threadIdx.x; m < N; m += kMomThreads) tw[m] = twg[m];
    __syncthreads();
    const int row = blockIdx.x * RPB + warp;
    if (row >= N) return;
    const int per = (kc + kMomGroups - 1) / kMomGroups;
    const int p0 = blockIdx.y * per, p1 = min(kc, p0 + per);
    float2* s12 = acc + (size_t)warp * N;
    for (int m = lane; m < N; m += 32) s12[m] = make_float2(0.f, 0.f);
    float2* z = zs + warp * L;
    const float inv = 1.0f / ((float)N * (float)N);
    for (int kk = p0; kk < p1; ++kk) {
        const float2* y = Y + (size_t)kk * N * H + (size_t)row * H;
        const float a = __fmul_rn(g_entry(g, n_bf, k0 + kk, 0, 0).x, inv);
        // Z[k] = E[k] + i O[k], E = X[k] + conj X[L-k], O = (X[k] - conj X[L-k]) W^-k,
        // the imaginary parts of X[0] and X[L] dropped
        for (int k = lane; k < L; k += 32) {
            float2 xk = y[k];
            float2 xl = y[L - k];
            if (k == 0) {
                xk.y = 0.f;
                xl.y = 0.f;
            }
            const float2 xc = cconj(xl);
            const float2 ev = cadd(xk, xc);
            const float2 od = cmul(csub(xk, xc), cconj(tw[k]));
            z[swz(k)] = cconj(cadd(ev, cmul_pi(od)));  // inverse via conj trick
        }
        __syncwarp();
        fft_warp<L, 2, true>(z, tw, lane);
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int m = lane + 32 * j;
            if (m < L) {
                const float2 v = cconj(z[swz(m)]);
                const float t0 = atan2f(v.x * inv, a), t1 = atan2f(v.y * inv, a);
                // (sum, square) of outputs 2m and 2m + 1 as one 16-byte access
                float4 u = reinterpret_cast<float4*>(s12)[m];
                u.x += t0;
                u.y = __fmaf_rn(t0, t0, u.y);
                u.z += t1;
                u.w = __fmaf_rn(t1, t1, u.w);
                reinterpret_cast<float4*>(s12)[m] = u;
            }
        }
        __syncwarp();
    }
    double2* out = part + (size_t)blockIdx.y * N * N + (size_t)row * N;
    for (int m = lane; m < N; m += 32) {
        double2 v = out[m];
        const float2 u = s12[m];
        v.x += (double)u.x;
        v.y += (double)u.y;
        out[m] = v;
    }
}

__global__ void ssb_moments_final(const double2* __restrict__ part, int npix, int n_bf, float* __restrict__ mean,
                                  float* __restrict__ var) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= npix) return;
    double a = 0.0, b = 0.0;
    for (int p = 0; p < kMomGroups; ++p) {
        const double2 v = part[(size_t)p * npix + i];
        a += v.x;
        b += v.y;
    }
    const double mu = a / n_bf;
    const double s = b / n_bf - mu * mu;
    mean[i] = (float)mu;
    var[i] = (float)(s > 0.0 ? s : 0.0);
}

template <int N>
static cudaError_t moments_n(const GView& g, int n_bf, const float4* ktab, const SetBatch& sb, double dq,
                             const float2* tw, float2* Y, double2* part, float* mean, float* var, cudaStream_t st) {
    constexpr int H = N / 2 + 1;
    constexpr int CW = inv_cols_width<N>();
    constexpr int NG = (N / 2) / CW;
    constexpr int RPB = kMomThreads / 32;
    const size_t cs = (size_t)N * sizeof(float2) + (size_t)(CW + 1) * (N + 4) * sizeof(float2);
    const size_t rs = (size_t)N * sizeof(float2) + (size_t)RPB * (N / 2) * sizeof(float2) +
                      (size_t)RPB * N * sizeof(float2);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ssb_inv_cols<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cs)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(ssb_inv_rows_moments<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rs)) !=
        cudaSuccess)
        return e;
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ssb_inv_cols<N>, kMomThreads, cs);
    const int col_grid = sms * (per_sm > 0 ? per_sm : 1);
    if ((e = cudaMemsetAsync(part, 0, (size_t)kMomGroups * N * N * sizeof(double2), st)) != cudaSuccess) return e;
    for (int k0 = 0; k0 < n_bf; k0 += kMomChunk) {
        const int kc = min(kMomChunk, n_bf - k0);
        ssb_correct<<<dim3((N * H + kMomThreads - 1) / kMomThreads, kMomKSplit), kMomThreads, 0, st>>>(
            g, n_bf, ktab, sb, N, dq, k0, kc, Y);
        const int items = NG * kc;
        ssb_inv_cols<N><<<items < col_grid ? items : col_grid, kMomThreads, cs, st>>>(Y, tw, items);
        ssb_inv_rows_moments<N><<<dim3((N + RPB - 1) / RPB, kMomGroups), kMomThreads, rs, st>>>(Y, kc, g, n_bf, k0,
                                                                                              tw, part);
        count_launch(3);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    ssb_moments_final<<<(N * N + 255) / 256, 256, 0, st>>>(part, N * N, n_bf, mean, var);
    count_launch();
    return cudaGetLastError();
}

size_t moments_chunk_bytes(int n) { return (size_t)kMomChunk * n * (n / 2 + 1) * sizeof(float2); }
size_t moments_part_bytes(int n) { return (size_t)kMomGroups * n * n * sizeof(double2); }

cudaError_t launch_moments(const GView& g, int n, int n_bf, const float4* ktab, const SetBatch& sb, double dq,
                           const float2* tw, void* Y, void* part, float* mean, float* var, cudaStream_t st) {
    float2* y = static_cast<float2*>(Y);
    double2* pt = static_cast<double2*>(part);
    switch (n) {
        case 8: return moments_n<8>(g, n_bf, ktab, sb, dq, tw, y, pt, mean, var, st);
        case 16: return moments_n<16>(g, n_bf, ktab, sb, dq, tw, y, pt, mean, var, st);
        case 32: return moments_n<32>(g, n_bf, ktab, sb, dq, tw, y, pt, mean, var, st);
        case 64: return moments_n<64>(g, n_bf, ktab, sb, dq, tw, y, pt, mean, var, st);
        case 128: return moments_n<128>(g, n_bf, ktab, sb, dq, tw, y, pt, mean, var, st);
        case 256: return moments_n<256>(g, n_bf, ktab, sb, dq, tw, y, pt, mean, var, st);
        case 512: return moments_n<512>(g, n_bf, ktab, sb, dq, tw, y, pt, mean, var, st);
        case 1024: return moments_n<1024>(g, n_bf, ktab, sb, dq, tw, y, pt, mean, var, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssb
