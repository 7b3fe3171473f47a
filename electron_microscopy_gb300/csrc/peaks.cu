// peaks.cu -- throughput probes (include/ssb_peaks.h): the transcendental
// (sin/cos) and float32 multiply-add rates the scoring and build rooflines
// are measured against.
#include "../../include/ssb_peaks.h"
#include "internal.cuh"

namespace ssb {

constexpr int kPeakThreads = 256;

__global__ void __launch_bounds__(kPeakThreads) ssb_peak_sincos_k(float* out, int iters, float a) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 1e-3f * (float)(threadIdx.x + 37 * i);
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float s, c;
            __sincosf(x[i], &s, &c);
            x[i] = __fmaf_rn(s, a, c);
        }
    }
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += x[i];
    if (t == 12345.678f) out[0] = t;
}

__global__ void __launch_bounds__(kPeakThreads) ssb_peak_fma_k(float* out, int iters, float a) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 1e-3f * (float)(threadIdx.x + 37 * i);
    const float b = 1.0f - a;
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __fmaf_rn(x[i], b, a);
    }
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += x[i];
    if (t == 12345.678f) out[0] = t;
}

template <typename K>
static int run_probe(K kernel, float* out, int blocks, int iters, void* stream) {
    if (!out || blocks < 1 || iters < 1) return set_last_error(SSB_INVALID_ARG, "out must not be NULL; blocks, iters >= 1",
                                                               cudaSuccess);
    kernel<<<blocks, kPeakThreads, 0, static_cast<cudaStream_t>(stream)>>>(out, iters, 1e-3f);
    count_launch();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return set_last_error(SSB_CUDA_ERROR, "peak probe launch", e);
    return SSB_OK;
}

}  // namespace ssb

extern "C" int ssb_peak_sincos(float* out_dev, int blocks, int iters, void* stream) {
    return ssb::run_probe(ssb::ssb_peak_sincos_k, out_dev, blocks, iters, stream);
}

extern "C" int ssb_peak_fma(float* out_dev, int blocks, int iters, void* stream) {
    return ssb::run_probe(ssb::ssb_peak_fma_k, out_dev, blocks, iters, stream);
}
