// build.cu -- G(q,k) build: bright-field gather + 2D real-to-complex FFT over the scan.
//
// G(q,k) = sum_r x_k(r) exp(-2 pi i (f_y r_y + f_x r_x)/n), stored as the
// Hermitian half plane [k][q_y row][q_x], q_x in [0, n/2] (quantem.gpu
// "Historical WebGPU G(q,k) memory experiment", sections "Why herm is exactly
// lossless" and "Implementation").
//
// Every size except n = 512 with uint16 frames (plane.cu) builds G in two
// passes over it: a row pass (gather + real-to-complex FFT along r_x of the
// packed even/odd samples, plus the split step, written as G's rows) and a
// column pass (complex FFT along r_y, in place).
//  - general n: row pass one CTA per (scan row r_y, 32 BF pixels), gathering
//    the 32 pixels from the n frames of that scan row, transposing them through
//    shared memory and running a warp-level Stockham FFT; column pass one CTA
//    per (BF pixel, 16 q_x columns), Stockham in shared memory.  The host walks
//    the BF pixels in chunks and issues row(c) and column(c-1) back to back so
//    that a chunk's rows are still in L2 when the column pass reads them.
//  - n = 1024: the column pass is ssb_col1024 (32 x 32 in registers, 8 columns
//    per CTA); with uint16 frames the row pass is ssb_row1024 (16 pixels per
//    CTA, 32 x 16 in registers), one launch over all BF pixels.
// The host-input build (ssb_build_G_host) first remaps the indices into the
// copied detector box (ssb_crop_idx).
#include <type_traits>

#include "internal.cuh"

namespace ssb {

// ---------------------------------------------------------------------------
// twiddle table W[m] = exp(-2 pi i m / n), m < n, from double precision
// ---------------------------------------------------------------------------
__global__ void ssb_twiddles(float2* tw, int n) {
    int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m < n) {
        double s, c;
        sincospi(-2.0 * (double)m / (double)n, &s, &c);
        tw[m] = make_float2((float)c, (float)s);
    }
}

cudaError_t launch_twiddles(float2* tw, int n, cudaStream_t st) {
    ssb_twiddles<<<(n + 255) / 256, 256, 0, st>>>(tw, n);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// bright-field indices into a detector crop (the host-input build)
// ---------------------------------------------------------------------------
__global__ void ssb_crop_idx(const int32_t* __restrict__ in, int n, int det_x, int r0, int c0, int cols,
                             int32_t* __restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const int v = in[i], r = v / det_x;
        out[i] = (r - r0) * cols + (v - r * det_x - c0);
    }
}

cudaError_t launch_crop_idx(const int32_t* in, int n, int det_x, int r0, int c0, int cols, int32_t* out,
                            cudaStream_t st) {
    ssb_crop_idx<<<(n + 255) / 256, 256, 0, st>>>(in, n, det_x, r0, c0, cols, out);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// row pass
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 256;
constexpr int kRowPix = 32;  // BF pixels per CTA (one per lane in the gather)

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<uint16_t>(uint16_t v) { return (float)v; }
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }

template <int N>
__host__ __device__ constexpr int row_stride_floats() { return N + 2; }  // even (float2 aligned), breaks bank aliasing

template <int N>
constexpr size_t row_smem_bytes() {
    return (size_t)N * sizeof(float2) + (size_t)kRowPix * row_stride_floats<N>() * sizeof(float);
}

template <int N, typename T>
__global__ void __launch_bounds__(kRowThreads)
ssb_row_r2c(const T* __restrict__ frames, int det_pix, const int32_t* __restrict__ bf_idx,
               int k_begin, int k_end, float2* __restrict__ G, const float2* __restrict__ twg) {
    constexpr int L = N / 2;
    constexpr int H = N / 2 + 1;
    constexpr int RS = row_stride_floats<N>();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float2* tw = reinterpret_cast<float2*>(smem_raw);
    float* rows = reinterpret_cast<float*>(smem_raw + (size_t)N * sizeof(float2));

    const int ry = blockIdx.x;
    const int kb = k_begin + blockIdx.y * kRowPix;
    const int nk = min(kRowPix, k_end - kb);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = kRowThreads / 32;

    for (int m = threadIdx.x; m < N; m += kRowThreads) tw[m] = twg[m];

    // gather + transpose: lane <-> BF pixel, warp <-> scan column r_x
    const int pix = (lane < nk) ? bf_idx[kb + lane] : 0;
    const T* base = frames + (size_t)ry * N * (size_t)det_pix + pix;
    if (lane < nk) {
#pragma unroll 4
        for (int rx = warp; rx < N; rx += NW) rows[lane * RS + rx] = to_f<T>(base[(size_t)rx * det_pix]);
    }
    __syncthreads();

    // per BF pixel: complex FFT of z[m] = x[2m] + i x[2m+1] (L points), then split
    for (int p = warp; p < nk; p += NW) {
        float2* z = reinterpret_cast<float2*>(rows + p * RS);
        fft_warp<L, 2>(z, tw, lane);
        float2* out = G + ((size_t)(kb + p) * N + ry) * H;
        for (int k = lane; k <= L; k += 32) {
            const float2 zk = z[k & (L - 1)];
            const float2 zc = cconj(z[(L - k) & (L - 1)]);
            const float2 e = make_float2(0.5f * (zk.x + zc.x), 0.5f * (zk.y + zc.y));
            // o = -i/2 (zk - zc)
            const float2 o = cmul_mi(make_float2(0.5f * (zk.x - zc.x), 0.5f * (zk.y - zc.y)));
            out[k] = cadd(e, cmul(tw[k], o));
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// column pass (in place on G)
// ---------------------------------------------------------------------------
constexpr int kColThreads = 256;

template <int N>
__host__ __device__ constexpr int col_width() { return (N / 2 >= 16) ? 16 : N / 2; }

template <int N>
constexpr size_t col_smem_bytes() {
    return (size_t)N * sizeof(float2) + (size_t)(col_width<N>() + 1) * (N + 1) * sizeof(float2);
}

template <int N>
__global__ void __launch_bounds__(kColThreads)
ssb_col_c2c(float2* __restrict__ G, int k_begin, const float2* __restrict__ twg) {
    constexpr int H = N / 2 + 1;
    constexpr int CW = col_width<N>();
    constexpr int NG = (N / 2) / CW;
    constexpr int CS = N + 1;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float2* tw = reinterpret_cast<float2*>(smem_raw);
    float2* cols = tw + N;

    const int g = blockIdx.x;
    const int k = k_begin + blockIdx.y;
    const int c0 = g * CW;
    const int nc = CW + ((g == NG - 1) ? 1 : 0);  // the last group also takes q_x = n/2
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = kColThreads / 32;

    for (int m = threadIdx.x; m < N; m += kColThreads) tw[m] = twg[m];
    float2* P = G + (size_t)k * N * H + c0;
    for (int idx = threadIdx.x; idx < N * nc; idx += kColThreads) {
        const int ry = idx / nc, c = idx - ry * nc;
        cols[c * CS + ry] = P[(size_t)ry * H + c];
    }
    __syncthreads();
    for (int c = warp; c < nc; c += NW) fft_warp<N, 1>(cols + c * CS, tw, lane);
    __syncthreads();
    for (int idx = threadIdx.x; idx < N * nc; idx += kColThreads) {
        const int ry = idx / nc, c = idx - ry * nc;
        P[(size_t)ry * H + c] = cols[c * CS + ry];
    }
}

// ---------------------------------------------------------------------------
// column pass for n = 1024 (in place on G): 1024 = 32 x 32 in registers.
// CTA = 8 columns of one plane, 32 threads per column; thread t first takes
// rows t + 32 r2 (r2 < 32): DFT32 over r2 -> A[t][k2], times W1024^(t k2),
// transposed through shared memory; then thread k2 takes A[r1][k2] (r1 < 32):
// DFT32 over r1 -> X[k2 + 32 k1].  A warp covers 8 columns x 4 rows, so every
// global access is four 64-byte row segments; the shared layout
// [column][k2][t] with strides 1060 and 33 (float2) puts both the stores and
// the loads of a warp on distinct bank pairs.
// ---------------------------------------------------------------------------
constexpr int kC1024Cols = 8;
constexpr int kC1024Threads = 256;
constexpr int kC1024RS = 33;    // k2 stride (float2)
constexpr int kC1024CS = 1060;  // column stride (float2): 8 words mod 32
constexpr size_t kC1024Smem = (size_t)kC1024Cols * kC1024CS * sizeof(float2);

__global__ void __launch_bounds__(kC1024Threads, 2)
ssb_col1024(float2* __restrict__ G, int k_begin, const float2* __restrict__ tw) {
    constexpr int N = 1024, H = N / 2 + 1;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float2* S = reinterpret_cast<float2*>(smem_raw);
    const int tid = threadIdx.x;
    const int c = tid & 7;                           // column within the group
    const int t = ((tid >> 3) & 3) + 4 * (tid >> 5);  // 0..31
    const int col = blockIdx.x * kC1024Cols + c;
    const bool has = col < H;
    float2* P = G + (size_t)(k_begin + blockIdx.y) * N * H + (has ? col : 0);
    float2* Sc = S + c * kC1024CS;
    float2 v[32];
#pragma unroll
    for (int r2 = 0; r2 < 32; ++r2) v[r2] = has ? P[(size_t)(t + 32 * r2) * H] : make_float2(0.f, 0.f);
    Dft<32>::run(v);  // v[k2] = A[t][k2]
#pragma unroll
    for (int k2 = 0; k2 < 32; ++k2) {
        const float2 w = k2 == 0 ? make_float2(1.f, 0.f) : __ldg(tw + ((t * k2) & (N - 1)));
        Sc[k2 * kC1024RS + t] = k2 == 0 ? v[k2] : cmul(v[k2], w);
    }
    __syncthreads();
#pragma unroll
    for (int r1 = 0; r1 < 32; ++r1) v[r1] = Sc[t * kC1024RS + r1];  // A[r1][k2 = t]
    Dft<32>::run(v);  // v[k1] = X[t + 32 k1]
    if (has) {
#pragma unroll
        for (int k1 = 0; k1 < 32; ++k1) P[(size_t)(t + 32 * k1) * H] = v[k1];
    }
}

// ---------------------------------------------------------------------------
// row pass for n = 1024, uint16 frames: gather + real-to-complex FFT.
// CTA = one scan row r_y x 16 bright-field pixels; the grid runs pixel groups
// fastest, so neighbouring groups of a scan row read the same frame lines
// while they are in L2.
//  gather: the 16 pixels of the row's 1024 frames into a uint16 stage
//          [pixel][word m] (word m holds samples 2m, 2m+1), the word index
//          XOR-swizzled by the pixel so that the gather's stores (16 pixels x
//          2 words per warp) and the FFT's loads (2 pixel rows p, p + 8 per
//          warp) both fall on 32 distinct banks;
//  FFT:    16 threads per pixel; the 512-point complex FFT of the halved
//          packed pairs z[m] = (x[2m] + i x[2m+1]) / 2 as 32 x 16: thread t
//          takes z[t + 16 n] (n < 32), DFT32 over n -> A[t][k2], times
//          W512^(t k2), through a padded buffer; thread t then takes
//          k2 in {t, t + 16}: DFT16 over t' -> Z[k2 + 32 k1];
//  split:  X[k] = a - i W1024^k b with a = Z[k] + conj Z[512 - k],
//          b = Z[k] - conj Z[512 - k] (the halving supplies the 1/2),
//          X[512] = 2 (Re Z[0] - Im Z[0]); written straight to G[k][r_y][q_x].
// ---------------------------------------------------------------------------
constexpr int kR1024Pix = 16;
constexpr int kR1024Threads = 16 * kR1024Pix;
constexpr int kR1024Words = 512;  // stage words per pixel
constexpr int kR1024TS = 33;      // transpose stride per t (float2)
constexpr int kR1024ZS = 16 * kR1024TS;
constexpr size_t kR1024Smem =
    (size_t)kR1024Pix * kR1024Words * sizeof(uint32_t) + (size_t)kR1024Pix * kR1024ZS * sizeof(float2);

__device__ __forceinline__ int r1024_word(int p, int m) {
    return p * kR1024Words + (m ^ ((p & 7) | (((p >> 3) & 1) << 4)));
}

__global__ void __launch_bounds__(kR1024Threads, 2)
ssb_row1024(const uint16_t* __restrict__ frames, int det_pix, const int32_t* __restrict__ bf_idx, int n_bf,
            float2* __restrict__ G, const float2* __restrict__ tw) {
    constexpr int N = 1024, H = N / 2 + 1;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint32_t* stage = reinterpret_cast<uint32_t*>(smem_raw);
    float2* zb = reinterpret_cast<float2*>(smem_raw + (size_t)kR1024Pix * kR1024Words * sizeof(uint32_t));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k0 = blockIdx.x * kR1024Pix;
    const int ry = blockIdx.y;
    {
        const int p = lane & 15, mb = lane >> 4;
        const int pix = k0 + p < n_bf ? bf_idx[k0 + p] : 0;
        const uint16_t* src = frames + (size_t)ry * N * det_pix + pix;
        // all of a thread's 64 loads in flight (registers are idle here)
        uint32_t wv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int m = warp + 8 * mb + 16 * j;
            const uint32_t lo = __ldcs(src + (size_t)(2 * m) * det_pix);
            const uint32_t hi = __ldcs(src + (size_t)(2 * m + 1) * det_pix);
            wv[j] = lo | (hi << 16);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int m = warp + 8 * mb + 16 * j;
            stage[r1024_word(p, m)] = wv[j];
        }
    }
    __syncthreads();
    const int t = lane & 15, p = warp + 8 * (lane >> 4);
    float2* zp = zb + p * kR1024ZS;
    {
        float2 v[32];
#pragma unroll
        for (int n = 0; n < 32; ++n) v[n] = half_pair(stage[r1024_word(p, t + 16 * n)]);
        Dft<32>::run(v);  // v[k2] = A[t][k2]
#pragma unroll
        for (int k2 = 0; k2 < 32; ++k2)
            zp[t * kR1024TS + k2] = k2 == 0 ? v[0] : cmul(v[k2], __ldg(tw + ((2 * t * k2) & (N - 1))));
    }
    __syncwarp();  // a pixel's 16 threads are one half of a warp
    {
        float2 a[16], b[16];
#pragma unroll
        for (int t2 = 0; t2 < 16; ++t2) {
            a[t2] = zp[t2 * kR1024TS + t];
            b[t2] = zp[t2 * kR1024TS + t + 16];
        }
        Dft<16>::run(a);  // a[k1] = Z[t + 32 k1]
        Dft<16>::run(b);  // b[k1] = Z[t + 16 + 32 k1]
        __syncwarp();
#pragma unroll
        for (int k1 = 0; k1 < 16; ++k1) {
            zp[t + 32 * k1] = a[k1];
            zp[t + 16 + 32 * k1] = b[k1];
        }
    }
    __syncwarp();
    const int kp = k0 + p;
    if (kp < n_bf) {
        float2* out = G + ((size_t)kp * N + ry) * H;
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
            const int k = t + 16 * j;
            const float2 z = zp[k], pr = zp[(512 - k) & 511];
            const float ax = z.x + pr.x, ay = z.y - pr.y;
            const float bx = z.x - pr.x, by = z.y + pr.y;
            const float2 w = __ldg(tw + k);
            out[k] = make_float2(ax + w.x * by + w.y * bx, ay - w.x * bx + w.y * by);
        }
        if (t == 0) out[512] = make_float2(2.0f * (zp[0].x - zp[0].y), 0.0f);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// column pass of one chunk of planes: the 32 x 32 register kernel at n = 1024,
// the shared-memory Stockham kernel otherwise
template <int N>
static void launch_col(float2* G, int k_begin, int count, const float2* tw, size_t cs, cudaStream_t st) {
    if constexpr (N == 1024) {
        ssb_col1024<<<dim3((N / 2 + 1 + kC1024Cols - 1) / kC1024Cols, count), kC1024Threads, kC1024Smem, st>>>(
            G, k_begin, tw);
    } else {
        constexpr int NG = (N / 2) / col_width<N>();
        ssb_col_c2c<N><<<dim3(NG, count), kColThreads, cs, st>>>(G, k_begin, tw);
    }
}

template <int N, typename T>
static cudaError_t build_n(const T* frames, int det_pix, const int32_t* bf_idx, int n_bf,
                           float2* G, const float2* tw, cudaStream_t st) {
    const size_t rs = row_smem_bytes<N>(), cs = col_smem_bytes<N>();
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ssb_row_r2c<N, T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)rs)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(ssb_col_c2c<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)cs)) != cudaSuccess)
        return e;
    if constexpr (N == 1024) {
        if ((e = cudaFuncSetAttribute(ssb_col1024, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kC1024Smem)) != cudaSuccess)
            return e;
    }
    // chunk of BF pixels whose intermediate rows (chunk * n * (n/2+1) * 8 B)
    // stay well inside L2
    const size_t plane = (size_t)N * (N / 2 + 1) * sizeof(float2);
    int chunk = (int)((48u << 20) / plane);
    chunk = chunk < kRowPix ? kRowPix : (chunk / kRowPix) * kRowPix;
    int prev_b = -1, prev_e = -1;
    for (int kb = 0; kb < n_bf || prev_b >= 0; kb += chunk) {
        if (kb < n_bf) {
            const int ke = kb + chunk < n_bf ? kb + chunk : n_bf;
            dim3 grid(N, (ke - kb + kRowPix - 1) / kRowPix);
            ssb_row_r2c<N, T><<<grid, kRowThreads, rs, st>>>(frames, det_pix, bf_idx, kb, ke, G, tw);
            count_launch();
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            if (prev_b >= 0) {
                launch_col<N>(G, prev_b, prev_e - prev_b, tw, cs, st);
                count_launch();
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
            }
            prev_b = kb;
            prev_e = ke;
        } else {
            launch_col<N>(G, prev_b, prev_e - prev_b, tw, cs, st);
            count_launch();
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
            prev_b = -1;
        }
    }
    return cudaSuccess;
}

// n = 1024, uint16 frames: one row pass over every BF pixel (G written once
// as the row spectra), then the column pass in place, in launches of at most
// 65535 planes
static cudaError_t build_1024_u16(const uint16_t* frames, int det_pix, const int32_t* bf_idx, int n_bf, float2* G,
                                  const float2* tw, cudaStream_t st) {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ssb_row1024, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kR1024Smem)) !=
        cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(ssb_col1024, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kC1024Smem)) !=
        cudaSuccess)
        return e;
    ssb_row1024<<<dim3((n_bf + kR1024Pix - 1) / kR1024Pix, 1024), kR1024Threads, kR1024Smem, st>>>(
        frames, det_pix, bf_idx, n_bf, G, tw);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    for (int kb = 0; kb < n_bf; kb += 65535) {
        const int cnt = n_bf - kb < 65535 ? n_bf - kb : 65535;
        ssb_col1024<<<dim3((1024 / 2 + 1 + kC1024Cols - 1) / kC1024Cols, cnt), kC1024Threads, kC1024Smem, st>>>(
            G, kb, tw);
        count_launch();
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename T>
static cudaError_t build_t(const T* frames, int n, int det_pix, const int32_t* bf_idx, int n_bf,
                           float2* G, const float2* tw, cudaStream_t st) {
    switch (n) {
        case 8: return build_n<8, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
        case 16: return build_n<16, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
        case 32: return build_n<32, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
        case 64: return build_n<64, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
        case 128: return build_n<128, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
        case 256: return build_n<256, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
        case 512: return build_n<512, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
        case 1024:
            if constexpr (std::is_same<T, uint16_t>::value)
                return build_1024_u16(frames, det_pix, bf_idx, n_bf, G, tw, st);
            else
                return build_n<1024, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_build(const void* frames, int dtype, int n, int det_pix, const int32_t* bf_idx,
                         int n_bf, float2* G, const float2* tw, cudaStream_t st) {
    if (dtype == SSB_U16)
        return build_t<uint16_t>(static_cast<const uint16_t*>(frames), n, det_pix, bf_idx, n_bf, G, tw, st);
    return build_t<float>(static_cast<const float*>(frames), n, det_pix, bf_idx, n_bf, G, tw, st);
}

}  // namespace ssb
