// compact.cu -- compact storage of G: herm16 and the band-compacted copy.
//
// herm16 (quantem.gpu "Historical WebGPU G(q,k) memory experiment", sections
// "Implementation" and "Scan-size sweep"): a post-pass over the built half
// plane takes the largest |G| of each block (scaleMax), then stores each
// component as floor(0.5 + 32767 clamp(v / scale, -1, 1)) in 16 bits, real part
// in the low half of a 32-bit word.  Blocks are a whole BF pixel's half plane
// (one scale per pixel, the page's preview) or one q row of it (n scales per
// pixel, the page's follow-up).  Every step is a separately rounded float32
// operation, so the codes are a function of G alone.
//
//  * one scale per q row: one warp per (k, row) reads the row's n/2+1 entries,
//    takes the warp maximum of re^2 + im^2, and packs the row from L1 (the
//    row, <= 4 KB, was just read): G read from HBM once.
//  * one scale per pixel: one CTA per pixel reduces the plane's maximum, then
//    an elementwise pass packs; G is read twice (a plane does not stay in L2
//    across the ~1,200 CTAs in flight).
//
// Band-compacted copy: dst[k][i] = G[k][band[i]], a gather whose reads follow
// the band's runs along q_x and whose writes are coalesced.
#include "internal.cuh"

namespace ssb {

constexpr int kCompactThreads = 256;

__device__ __forceinline__ float mod2(float2 v) { return __fadd_rn(__fmul_rn(v.x, v.x), __fmul_rn(v.y, v.y)); }

// 16-bit two's complement code of v at block scale sc (0 for an empty block)
__device__ __forceinline__ uint32_t snorm16(float v, float sc) {
    if (!(sc > 0.f)) return 0u;
    const float e = fminf(1.f, fmaxf(-1.f, __fdiv_rn(v, sc)));
    const int c = (int)floorf(__fadd_rn(0.5f, __fmul_rn(32767.f, e)));
    return (uint32_t)c & 0xffffu;
}

__device__ __forceinline__ uint32_t sn16_pack(float2 v, float sc) {
    return snorm16(v.x, sc) | (snorm16(v.y, sc) << 16);
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

// one scale per q row: warp w of the grid takes row r = k n + row
__global__ void __launch_bounds__(kCompactThreads)
ssb_g16_rows(const float2* __restrict__ G, int n, int H, int n_bf, uint32_t* __restrict__ G16,
             float* __restrict__ scale) {
    const long long r = (long long)blockIdx.x * (kCompactThreads / 32) + (threadIdx.x >> 5);
    if (r >= (long long)n_bf * n) return;  // warp-uniform
    const int lane = threadIdx.x & 31;
    const float2* src = G + r * H;
    float m = 0.f;
    for (int c = lane; c < H; c += 32) m = fmaxf(m, mod2(__ldg(src + c)));
    const float sc = __fsqrt_rn(warp_max(m));
    const int k = (int)(r / n), row = (int)(r - (long long)k * n);
    if (lane == 0) scale[(size_t)row * n_bf + k] = sc;
    uint32_t* dst = G16 + r * H;
    for (int c = lane; c < H; c += 32) dst[c] = sn16_pack(__ldg(src + c), sc);
}

// one scale per pixel, pass 1: CTA k reduces the plane's largest |G|
__global__ void __launch_bounds__(kCompactThreads)
ssb_g16_plane_max(const float2* __restrict__ G, size_t plane, float* __restrict__ scale) {
    __shared__ float red[kCompactThreads / 32];
    const int k = blockIdx.x;
    const float2* src = G + (size_t)k * plane;
    float m = 0.f;
#pragma unroll 4
    for (size_t c = threadIdx.x; c < plane; c += kCompactThreads) m = fmaxf(m, mod2(__ldcs(src + c)));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < kCompactThreads / 32 ? red[threadIdx.x] : 0.f;
        m = warp_max(m);
        if (threadIdx.x == 0) scale[k] = __fsqrt_rn(m);
    }
}

// one scale per pixel, pass 2: elementwise pack; grid (plane chunks, pixels)
__global__ void __launch_bounds__(kCompactThreads)
ssb_g16_plane_pack(const float2* __restrict__ G, size_t plane, int n_bf, const float* __restrict__ scale,
                   uint32_t* __restrict__ G16) {
    const size_t step = (size_t)gridDim.x * kCompactThreads;
    for (int k = blockIdx.y; k < n_bf; k += gridDim.y) {
        const float sc = __ldg(scale + k);
        const float2* src = G + (size_t)k * plane;
        uint32_t* dst = G16 + (size_t)k * plane;
        for (size_t c = (size_t)blockIdx.x * kCompactThreads + threadIdx.x; c < plane; c += step)
            dst[c] = sn16_pack(__ldcs(src + c), sc);
    }
}

cudaError_t launch_compact_g16(const float2* G, int n, int n_bf, int srows, uint32_t* G16, float* scale,
                               cudaStream_t st) {
    const int H = n / 2 + 1;
    const size_t plane = (size_t)n * H;
    if (srows == 1) {
        const long long rows = (long long)n_bf * n;
        const long long wpb = kCompactThreads / 32;
        ssb_g16_rows<<<(unsigned)((rows + wpb - 1) / wpb), kCompactThreads, 0, st>>>(G, n, H, n_bf, G16, scale);
        count_launch();
        return cudaGetLastError();
    }
    ssb_g16_plane_max<<<n_bf, kCompactThreads, 0, st>>>(G, plane, scale);
    count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t chunks = (plane + kCompactThreads - 1) / kCompactThreads;
    const dim3 grid((unsigned)((chunks + 3) / 4), (unsigned)(n_bf < 65535 ? n_bf : 65535));
    ssb_g16_plane_pack<<<grid, kCompactThreads, 0, st>>>(G, plane, n_bf, scale, G16);
    count_launch();
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// band-compacted copy: block (x, y) copies band positions [256 x, 256 x + 256)
// of BF pixels [kBandK y, kBandK y + kBandK)
// ---------------------------------------------------------------------------
constexpr int kBandK = 16;

template <typename T>
__global__ void __launch_bounds__(kCompactThreads)
ssb_band_gather(const T* __restrict__ G, size_t plane, int n_bf, const int32_t* __restrict__ band, int nq,
                T* __restrict__ dst) {
    const int i = blockIdx.x * kCompactThreads + threadIdx.x;
    if (i >= nq) return;
    const size_t e = (size_t)__ldg(band + i);
    const int k0 = blockIdx.y * kBandK;
    const int kn = min(kBandK, n_bf - k0);
    if (kn == kBandK) {
        T v[kBandK];
#pragma unroll
        for (int u = 0; u < kBandK; ++u) v[u] = __ldcs(G + (size_t)(k0 + u) * plane + e);
#pragma unroll
        for (int u = 0; u < kBandK; ++u) dst[(size_t)(k0 + u) * nq + i] = v[u];
    } else {
        for (int u = 0; u < kn; ++u) dst[(size_t)(k0 + u) * nq + i] = __ldcs(G + (size_t)(k0 + u) * plane + e);
    }
}

cudaError_t launch_compact_band(const void* G, int fmt, size_t plane, int n_bf, const int32_t* band, int nq,
                                void* dst, cudaStream_t st) {
    const size_t esz = fmt == kGSN16 ? sizeof(uint32_t) : sizeof(float2);
    const int kmax = 65535 * kBandK;  // BF pixels per launch (grid.y limit)
    for (int kb = 0; kb < n_bf; kb += kmax) {
        const int nk = min(kmax, n_bf - kb);
        const dim3 grid((unsigned)((nq + kCompactThreads - 1) / kCompactThreads), (unsigned)((nk + kBandK - 1) / kBandK));
        const char* src = static_cast<const char*>(G) + (size_t)kb * plane * esz;
        char* out = static_cast<char*>(dst) + (size_t)kb * nq * esz;
        if (fmt == kGSN16)
            ssb_band_gather<uint32_t><<<grid, kCompactThreads, 0, st>>>(reinterpret_cast<const uint32_t*>(src), plane,
                                                                         nk, band, nq, reinterpret_cast<uint32_t*>(out));
        else
            ssb_band_gather<float2><<<grid, kCompactThreads, 0, st>>>(reinterpret_cast<const float2*>(src), plane, nk,
                                                                       band, nq, reinterpret_cast<float2*>(out));
        count_launch();
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ssb
