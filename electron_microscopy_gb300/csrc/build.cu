// build.cu -- G(q,k) build: bright-field gather + 2D real-to-complex FFT over the scan.
//
// G(q,k) = sum_r x_k(r) exp(-2 pi i (f_y r_y + f_x r_x)/n), stored as the
// Hermitian half plane [k][q_y row][q_x], q_x in [0, n/2] (quantem.gpu
// "Historical WebGPU G(q,k) memory experiment", sections "Why herm is exactly
// lossless" and "Implementation").
//
// Two passes per chunk of bright-field pixels:
//   row pass    one CTA per (scan row r_y, 32 BF pixels): gathers the 32
//               pixels from the n frames of that scan row (each warp load
//               reads 32 neighbouring detector pixels of one frame), transposes
//               them through shared memory, runs the real-to-complex FFT along
//               r_x (n/2-point complex FFT of the packed even/odd samples plus
//               the split step) and writes the n/2+1 outputs into G's row r_y;
//   column pass one CTA per (BF pixel, group of 16 q_x columns): loads the
//               columns, runs the complex FFT along r_y and writes them back in
//               place.
// The host walks the BF pixels in chunks and issues row(c) and column(c-1)
// back to back so that a chunk's intermediate rows are still in L2 when the
// column pass reads them.
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
        case 1024: return build_n<1024, T>(frames, det_pix, bf_idx, n_bf, G, tw, st);
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
