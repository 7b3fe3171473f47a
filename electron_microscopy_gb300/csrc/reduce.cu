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
#include "reduce_kernel.cuh"

namespace ssb {

// ---------------------------------------------------------------------------
// k-only tables: float32 k, aperture bit per set, chi_s(k) in turns
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
ssb_prep(const int32_t* __restrict__ bf_idx, int n_bf, int det_x, double cy, double cx, double dk, SetBatch sb,
         float4* __restrict__ ktab, float* __restrict__ chik, float* __restrict__ kxcol, int* __restrict__ status,
         GView g, double* __restrict__ dcpart) {
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (status && k == 0) *status = 0;
    // k_x of every detector column, by the same expression as a BF pixel's
    if (kxcol && blockIdx.x == 0)
        for (int j = threadIdx.x; j < det_x; j += blockDim.x)
            kxcol[j] = __double2float_rn(__dmul_rn(__dsub_rn((double)j, cx), dk));
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
    // the first pixel of a detector row in list order (a different row
    // from the previous list entry) carries kRowStart
    if (k == 0 || bf_idx[k - 1] / det_x != i) bits |= kRowStart;
    ktab[k] = make_float4(kx, ky, __uint_as_float(bits), chi0);
}

cudaError_t launch_prep(const int32_t* bf_idx, int n_bf, int det_x, double cy, double cx, double dk,
                        const SetBatch& sb, float4* ktab, float* chik, float* kxcol, int* status,
                        const GView& g, double* dcpart, cudaStream_t st) {
    ssb_prep<<<(n_bf + 255) / 256, 256, 0, st>>>(bf_idx, n_bf, det_x, cy, cx, dk, sb, ktab, chik, kxcol, status, g,
                                                 dcpart);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_reduce(const RedLaunch& P, const SetBatch& sb, cudaStream_t st) {
    if (P.depth) return launch_reduce_depth(P, sb, st);
    if (recon_tma_applies(P, sb)) return launch_recon_tma(P, sb, st);
    return launch_reduce_t<false>(P, sb, st);
}

// ---------------------------------------------------------------------------
// partial sums -> O, N (fixed order over splits)
// ---------------------------------------------------------------------------
__global__ void ssb_finalize(const float2* __restrict__ Opart, const int* __restrict__ Npart,
                                int nsplit, int B, int nq, const int* __restrict__ status,
                                float2* __restrict__ O, int32_t* __restrict__ N) {
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t total = (size_t)B * nq;
    if (t >= total) return;
    if (status && *status) {  // a reduction wait ran out: no valid sums
        O[t] = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
        N[t] = -1;
        return;
    }
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
                            const int* status, float2* O, int32_t* N, cudaStream_t st) {
    const size_t total = (size_t)B * nq;
    ssb_finalize<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(Opart, Npart, nsplit, B, nq, status, O, N);
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
