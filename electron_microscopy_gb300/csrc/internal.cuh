// internal.cuh -- device building blocks shared by the SSB kernels (not part of the C ABI).
//
// * Complex helpers on float2.
// * A warp-level in-place Stockham FFT (radix 8/4/2) on a shared-memory row:
//   each pass reads every point of the row into registers, applies the
//   twiddles and a radix-R butterfly, and writes the autosorted output back
//   (the Stockham formulation of Govindaraju et al., "High Performance
//   Discrete Fourier Transforms on Graphics Processors", SC 2008).  Twiddles
//   come from a per-call table W[m] = exp(-2 pi i m / n), m < n, rounded once
//   from double precision.
// * The aberration polynomial chi/(2 pi) in Cartesian form and the float32
//   aperture test whose operation order is part of the library contract.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssb.h"

namespace ssb {

// ---------------------------------------------------------------------------
// complex helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
__device__ __forceinline__ float2 cconj(float2 a) { return make_float2(a.x, -a.y); }
// multiply by -i
__device__ __forceinline__ float2 cmul_mi(float2 a) { return make_float2(a.y, -a.x); }
// multiply by +i
__device__ __forceinline__ float2 cmul_pi(float2 a) { return make_float2(-a.y, a.x); }

// ---------------------------------------------------------------------------
// radix-R forward DFT in registers, X[k] = sum_m v[m] exp(-2 pi i m k / R)
// ---------------------------------------------------------------------------
template <int R> struct Dft;

template <> struct Dft<2> {
    static __device__ __forceinline__ void run(float2* v) {
        float2 a = v[0], b = v[1];
        v[0] = cadd(a, b);
        v[1] = csub(a, b);
    }
};

template <> struct Dft<4> {
    static __device__ __forceinline__ void run(float2* v) {
        float2 t0 = cadd(v[0], v[2]), t1 = csub(v[0], v[2]);
        float2 t2 = cadd(v[1], v[3]), t3 = cmul_mi(csub(v[1], v[3]));
        v[0] = cadd(t0, t2);
        v[2] = csub(t0, t2);
        v[1] = cadd(t1, t3);
        v[3] = csub(t1, t3);
    }
};

template <> struct Dft<8> {
    // split into a radix-2 stage (m, m+4), twiddles W8^m on the difference
    // half, then two radix-4 DFTs giving the even and odd outputs.
    static __device__ __forceinline__ void run(float2* v) {
        const float h = 0.70710678118654752f;  // 1/sqrt(2)
        float2 a[4], b[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            a[m] = cadd(v[m], v[m + 4]);
            b[m] = csub(v[m], v[m + 4]);
        }
        // b1 *= (1 - i)/sqrt2 ; b2 *= -i ; b3 *= (-1 - i)/sqrt2
        b[1] = make_float2(h * (b[1].x + b[1].y), h * (b[1].y - b[1].x));
        b[2] = cmul_mi(b[2]);
        b[3] = make_float2(h * (b[3].y - b[3].x), -h * (b[3].x + b[3].y));
        Dft<4>::run(a);
        Dft<4>::run(b);
        v[0] = a[0]; v[2] = a[1]; v[4] = a[2]; v[6] = a[3];
        v[1] = b[0]; v[3] = b[1]; v[5] = b[2]; v[7] = b[3];
    }
};

// multiply by W16^M = exp(-2 pi i M / 16), trivial factors written out
template <int M>
__device__ __forceinline__ float2 w16(float2 a) {
    constexpr float c1 = 0.92387953251128676f;  // cos(pi/8)
    constexpr float s1 = 0.38268343236508977f;  // sin(pi/8)
    constexpr float h = 0.70710678118654752f;
    if constexpr (M == 0) {
        return a;
    } else if constexpr (M == 1) {  // (c1, -s1)
        return make_float2(c1 * a.x + s1 * a.y, c1 * a.y - s1 * a.x);
    } else if constexpr (M == 2) {  // (h, -h)
        return make_float2(h * (a.x + a.y), h * (a.y - a.x));
    } else if constexpr (M == 3) {  // (s1, -c1)
        return make_float2(s1 * a.x + c1 * a.y, s1 * a.y - c1 * a.x);
    } else if constexpr (M == 4) {  // -i
        return cmul_mi(a);
    } else if constexpr (M == 6) {  // (-h, -h)
        return make_float2(h * (a.y - a.x), -h * (a.x + a.y));
    } else {                        // M == 9: (-c1, s1)
        static_assert(M == 9, "only the factors of a 4x4 split are needed");
        return make_float2(-c1 * a.x - s1 * a.y, s1 * a.x - c1 * a.y);
    }
}

template <> struct Dft<16> {
    // 16 = 4 x 4: radix-4 over n2 for each n1 (input index n1 + 4 n2), twiddle
    // W16^(n1 k2), radix-4 over n1; output index k2 + 4 k1.
    static __device__ __forceinline__ void run(float2* v) {
        float2 a0[4] = {v[0], v[4], v[8], v[12]};
        float2 a1[4] = {v[1], v[5], v[9], v[13]};
        float2 a2[4] = {v[2], v[6], v[10], v[14]};
        float2 a3[4] = {v[3], v[7], v[11], v[15]};
        Dft<4>::run(a0);
        Dft<4>::run(a1);
        Dft<4>::run(a2);
        Dft<4>::run(a3);
        float2 b0[4] = {a0[0], a1[0], a2[0], a3[0]};
        float2 b1[4] = {a0[1], w16<1>(a1[1]), w16<2>(a2[1]), w16<3>(a3[1])};
        float2 b2[4] = {a0[2], w16<2>(a1[2]), w16<4>(a2[2]), w16<6>(a3[2])};
        float2 b3[4] = {a0[3], w16<3>(a1[3]), w16<6>(a2[3]), w16<9>(a3[3])};
        Dft<4>::run(b0);
        Dft<4>::run(b1);
        Dft<4>::run(b2);
        Dft<4>::run(b3);
#pragma unroll
        for (int k1 = 0; k1 < 4; ++k1) {
            v[0 + 4 * k1] = b0[k1];
            v[1 + 4 * k1] = b1[k1];
            v[2 + 4 * k1] = b2[k1];
            v[3 + 4 * k1] = b3[k1];
        }
    }
};

// packed even/odd samples z = (x[2w], x[2w+1]) / 2 from one 32-bit word of
// two uint16 counts: 2^23 + u is exact in float, (2^23 + u)/2 - 2^22 = u/2
__device__ __forceinline__ float2 half_pair(uint32_t u) {
    const float lo = __fmaf_rn(__uint_as_float(0x4B000000u | (u & 0xFFFFu)), 0.5f, -4194304.0f);
    const float hi = __fmaf_rn(__uint_as_float(0x4B000000u | (u >> 16)), 0.5f, -4194304.0f);
    return make_float2(lo, hi);
}

// cos and sin of 2 pi k / 32, k < 16 (the mathematical values, rounded to
// float): W32^k = kCos32[k] - i kSin32[k]
__device__ constexpr float kCos32[16] = {1.0f, 0.98078528040323043f, 0.92387953251128674f, 0.83146961230254524f,
                                         0.70710678118654752f, 0.55557023301960218f, 0.38268343236508977f,
                                         0.19509032201612826f, 0.0f, -0.19509032201612826f, -0.38268343236508977f,
                                         -0.55557023301960218f, -0.70710678118654752f, -0.83146961230254524f,
                                         -0.92387953251128674f, -0.98078528040323043f};
__device__ constexpr float kSin32[16] = {0.0f, 0.19509032201612826f, 0.38268343236508977f, 0.55557023301960218f,
                                         0.70710678118654752f, 0.83146961230254524f, 0.92387953251128674f,
                                         0.98078528040323043f, 1.0f, 0.98078528040323043f, 0.92387953251128674f,
                                         0.83146961230254524f, 0.70710678118654752f, 0.55557023301960218f,
                                         0.38268343236508977f, 0.19509032201612826f};

template <> struct Dft<32> {
    // 32 = 2 x 16: DFT16 of the even and of the odd samples, then
    // X[k] = A[k] + W32^k B[k], X[k + 16] = A[k] - W32^k B[k]; natural order
    static __device__ __forceinline__ void run(float2* v) {
        float2 a[16], b[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            a[i] = v[2 * i];
            b[i] = v[2 * i + 1];
        }
        Dft<16>::run(a);
        Dft<16>::run(b);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float2 t = cmul(b[k], make_float2(kCos32[k], -kSin32[k]));
            v[k] = cadd(a[k], t);
            v[k + 16] = csub(a[k], t);
        }
    }
};

// ---------------------------------------------------------------------------
// warp-level in-place Stockham pass over a row of L points in shared memory.
// NS: span of the sub-transforms already done; TWS: stride into the
// length-n twiddle table (n / L).
// ---------------------------------------------------------------------------
// SWZ: the buffer holds point i at swz(i) = i ^ ((i >> 4) & 15), a bijection
// within each 16-point block that makes both the stride-R writes of a pass
// and the unit-stride reads of the next hit every bank pair at most twice
// per warp (8-byte points)
__device__ __forceinline__ int swz(int i) { return i ^ ((i >> 4) & 15); }

template <int L, int R, int NS, int TWS, bool SWZ = false>
__device__ __forceinline__ void stockham_pass(float2* buf, const float2* tw, int lane) {
    constexpr int NB = L / R;
    constexpr int PER = (NB + 31) / 32;
    float2 v[PER][R];
#pragma unroll
    for (int t = 0; t < PER; ++t) {
        const int j = lane + 32 * t;
        if (NB >= 32 || j < NB) {
#pragma unroll
            for (int r = 0; r < R; ++r) v[t][r] = buf[SWZ ? swz(j + r * NB) : j + r * NB];
        }
    }
    __syncwarp();
#pragma unroll
    for (int t = 0; t < PER; ++t) {
        const int j = lane + 32 * t;
        if (NB >= 32 || j < NB) {
            const int k = j & (NS - 1);
            if (NS > 1) {
#pragma unroll
                for (int r = 1; r < R; ++r)
                    v[t][r] = cmul(v[t][r], tw[(k * r * (L / (NS * R))) * TWS]);
            }
            Dft<R>::run(v[t]);
            const int base = (j - k) * R + k;
#pragma unroll
            for (int r = 0; r < R; ++r) buf[SWZ ? swz(base + r * NS) : base + r * NS] = v[t][r];
        }
    }
    __syncwarp();
}

template <int L, int NS, int TWS, bool SWZ>
__device__ __forceinline__ void fft_passes(float2* buf, const float2* tw, int lane) {
    if constexpr (NS < L) {
        constexpr int REM = L / NS;
        constexpr int R = (REM >= 8) ? 8 : REM;
        stockham_pass<L, R, NS, TWS, SWZ>(buf, tw, lane);
        fft_passes<L, NS * R, TWS, SWZ>(buf, tw, lane);
    }
}

// Forward complex FFT (exp(-2 pi i ...)) of length L, in place, by one warp.
// SWZ: input and output are in the swizzled order swz(i) (see stockham_pass).
template <int L, int TWS, bool SWZ = false>
__device__ __forceinline__ void fft_warp(float2* buf, const float2* tw, int lane) {
    fft_passes<L, 1, TWS, SWZ>(buf, tw, lane);
}

// ---------------------------------------------------------------------------
// aberration sets
// ---------------------------------------------------------------------------
// chi/(2 pi) in turns as a polynomial of v = (vx, vy) (1/Angstrom):
//   xx = vx^2, yy = vy^2, s = xx + yy, u = xx - yy, p = vx vy
//   deg2 = c0 s + c1 u + c2 p
//   deg3 = s (c3 vx + c4 vy) + c5 vx (xx - 3 yy) + c6 vy (3 xx - yy)
//   deg4 = s (c7 s + c8 u + c9 p) + c10 (u^2 - 4 p^2) + c11 u p
// with c0 = lam C10/2, c1 = lam C12a/2, c2 = lam C12b, c3 = lam^2 C21a/3,
// c4 = lam^2 C21b/3, c5 = lam^2 C23a/3, c6 = lam^2 C23b/3, c7 = lam^3 C30/4,
// c8 = lam^3 C32a/4, c9 = lam^3 C32b/2, c10 = lam^3 C34a/4, c11 = lam^3 C34b.
// (theta^m cos(n phi), theta^m sin(n phi) written through Re/Im of
// (vx + i vy)^n; the division-free Cartesian form the tilt-speed page uses.)
struct SetParams {
    float tx, ty;   // float32(k_t)
    float c[12];
    // chi/(2 pi) regrouped as a quartic in vx for a fixed vy (see chi_row):
    // h[0] = c7 + c8 + c10 (the vx^4 coefficient), then the vy-polynomials
    // of the vx^3..vx^0 coefficients: h1 + h2 y; h3 + h4 y + h5 y^2;
    // y (h6 + h7 y + h8 y^2); y^2 (h9 + h10 y + h11 y^2)
    float h[12];
};

struct SetBatch {
    SetParams s[SSB_MAX_SETS];
    float depth_a[SSB_MAX_SETS];  // pi lambda t / 2 per set (depth-spread fit; 0: none)
    int depth_shared;             // every set has the same depth_a
    float r2;       // float32((alpha/lambda)^2)
    int B;
};

// chi/(2 pi) = sum_i c[i] m_i(v) over 12 monomials of v = (vx, vy):
//   m = (s, u, p, s vx, s vy, vx (xx - 3 yy), vy (3 xx - yy), s^2, s u, s p,
//        u^2 - 4 p^2, u p),  xx = vx^2, yy = vy^2, s = xx + yy, u = xx - yy, p = vx vy.
// Every operation is explicitly rounded and the dot product runs in a fixed
// order, so chi(k) is bit-identical wherever it is evaluated.  The reduction
// evaluates chi(k -/+ q) through the row form (chi_row, chi_horner below),
// also in a fixed order, so a set's result does not depend on the batch it
// runs in.
__device__ __forceinline__ void chi_monomials(float vx, float vy, float* m) {
    const float xx = __fmul_rn(vx, vx), yy = __fmul_rn(vy, vy);
    const float s = __fadd_rn(xx, yy), u = __fsub_rn(xx, yy), p = __fmul_rn(vx, vy);
    m[0] = s;
    m[1] = u;
    m[2] = p;
    m[3] = __fmul_rn(s, vx);
    m[4] = __fmul_rn(s, vy);
    m[5] = __fmul_rn(vx, __fmaf_rn(-3.0f, yy, xx));
    m[6] = __fmul_rn(vy, __fmaf_rn(3.0f, xx, -yy));
    m[7] = __fmul_rn(s, s);
    m[8] = __fmul_rn(s, u);
    m[9] = __fmul_rn(s, p);
    m[10] = __fmaf_rn(u, u, __fmul_rn(-4.0f, __fmul_rn(p, p)));
    m[11] = __fmul_rn(u, p);
}

__device__ __forceinline__ float chi_dot(const float* c, const float* m) {
    float a = __fmul_rn(c[0], m[0]);
#pragma unroll
    for (int i = 1; i < 12; ++i) a = __fmaf_rn(c[i], m[i], a);
    return a;
}

__device__ __forceinline__ float chi_turns(const float* c, float vx, float vy) {
    float m[12];
    chi_monomials(vx, vy, m);
    return chi_dot(c, m);
}

// Coefficients (a3, a2, a1, a0) of chi(vx, vy)/(2 pi) = (((h0 vx + a3) vx + a2)
// vx + a1) vx + a0 for one vy: a detector row at one scan frequency has one
// vy per trotter side, so the reduction evaluates chi(k -/+ q) along the row
// with 4 FMAs per set instead of the 12-monomial dot product.  Fixed
// operation order: the values do not depend on where or for which batch this
// runs.
__device__ __forceinline__ float4 chi_row(const float* h, float y) {
    const float yy = __fmul_rn(y, y);
    const float a3 = __fmaf_rn(h[2], y, h[1]);
    const float a2 = __fmaf_rn(h[5], yy, __fmaf_rn(h[4], y, h[3]));
    const float a1 = __fmul_rn(__fmaf_rn(h[8], yy, __fmaf_rn(h[7], y, h[6])), y);
    const float a0 = __fmul_rn(__fmaf_rn(h[11], yy, __fmaf_rn(h[10], y, h[9])), yy);
    return make_float4(a3, a2, a1, a0);
}

__device__ __forceinline__ float chi_horner(float h0, float4 a, float x) {
    return __fmaf_rn(__fmaf_rn(__fmaf_rn(__fmaf_rn(h0, x, a.x), x, a.y), x, a.z), x, a.w);
}

// Squared distance from the tilt centre, float32 contract: dx = px - tx;
// dy = py - ty; d2 = dx*dx + dy*dy, each operation rounded separately.
__device__ __forceinline__ float d2_f32(float px, float py, float tx, float ty) {
    const float dx = __fsub_rn(px, tx), dy = __fsub_rn(py, ty);
    return __fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy));
}

// Aperture test, float32 contract: inside iff d2_f32(...) <= r2; also
// returns dx, dy (and d2 in the second form).
__device__ __forceinline__ bool aperture_f32(float px, float py, float tx, float ty, float r2,
                                             float* dxo, float* dyo, float* d2o) {
    const float dx = __fsub_rn(px, tx), dy = __fsub_rn(py, ty);
    const float d2 = __fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy));
    *dxo = dx;
    *dyo = dy;
    *d2o = d2;
    return d2 <= r2;
}
__device__ __forceinline__ bool aperture_f32(float px, float py, float tx, float ty, float r2,
                                             float* dxo, float* dyo) {
    float d2;
    return aperture_f32(px, py, tx, ty, r2, dxo, dyo, &d2);
}

// sinc(a D) = sin(a D) / (a D), 1 near 0, from the fast sine: the depth-spread
// factor of a trotter term (a = pi lambda t / 2, D a difference of squared
// distances in 1/A^2)
__device__ __forceinline__ float depth_sinc(float a, float D) {
    const float x = __fmul_rn(a, D);
    return fabsf(x) < 1e-4f ? 1.0f : __fdividef(__sinf(x), x);
}

// w(q,k) G(q,k) added to acc: d = chi(k) - chi(k -/+ q) in turns, reduced to
// [-1/2, 1/2] exactly.  T-: w = exp(-2 pi i d); T+: w = -exp(+2 pi i d), which
// is the T- form with G and the angle negated: the caller passes
// gs = +/-G and tw = +/-2 pi once per (q, k), and every set adds
// gs exp(-i tw r) with four FMAs.
__device__ __forceinline__ void accumulate(float2& acc, float2 gs, float chik, float chiq, float tw) {
    const float d = __fsub_rn(chik, chiq);
    const float r = __fsub_rn(d, rintf(d));
    float sn, cs;
    __sincosf(__fmul_rn(tw, r), &sn, &cs);  // |argument| <= pi
    acc.x = __fmaf_rn(gs.y, sn, __fmaf_rn(gs.x, cs, acc.x));
    acc.y = __fmaf_rn(-gs.x, sn, __fmaf_rn(gs.y, cs, acc.y));
}

__device__ __forceinline__ float2 side_sign(float2 g, bool minus) {
    return minus ? g : make_float2(-g.x, -g.y);
}
constexpr float kTwoPi = 6.28318530717958648f;

// ---------------------------------------------------------------------------
// host-side launchers (defined in build.cu / reduce.cu); return cudaError_t
// ---------------------------------------------------------------------------
cudaError_t launch_twiddles(float2* tw, int n, cudaStream_t st);
cudaError_t launch_build(const void* frames, int dtype, int n, int det_pix,
                         const int32_t* bf_idx, int n_bf, float2* G, const float2* tw,
                         cudaStream_t st);
// bright-field indices into a detector crop: in[i] = r det_x + c ->
// out[i] = (r - r0) cols + (c - c0)
cudaError_t launch_crop_idx(const int32_t* in, int n, int det_x, int r0, int c0, int cols, int32_t* out,
                            cudaStream_t st);
// n = 512, uint16 frames: gather + cluster FFT (plane.cu); xbuf holds
// plane512_chunk_bytes(); plane512_cluster_size() is 0 when the cluster kernel
// cannot be scheduled on the current device
size_t plane512_chunk_bytes();
int plane512_cluster_size();
cudaError_t launch_build512(const uint16_t* frames, int det_pix, const int32_t* bf_idx, int n_bf,
                            float2* G, const float2* tw, void* xbuf, cudaStream_t st);

// k-only table per bright-field pixel: (float32 kx, float32 ky, aperture
// bits of the sets as float bits, chi_0(k) in turns); chi_s(k) of every set
// in chik[k * kChiStride + s]
constexpr int kChiStride = 8;
// ktab[k].z bits: bit s the aperture test of set s at k; kRowStart marks a
// pixel whose detector row differs from the previous list entry's
constexpr uint32_t kRowStart = 0x80000000u;

// a stored G as the reductions read it: complex64 entries, or herm16 words
// (two int16 codes, real in the low half) with float32 scales
// [n / srows][n_bf]; entry (k, i) sits at k * stride + i, i the half-plane
// entry or, for a band-compacted copy, the band position
enum GFormat { kGC64 = 0, kGSN16 = 1 };
struct GView {
    const void* G;
    int fmt;
    size_t stride;          // entries between consecutive BF pixels
    int band;               // 1: indexed by band position, not half-plane entry
    const float* scale;     // kGSN16
    int srows;              // kGSN16: q rows per scale block (1 or n)
};

// one herm16 word to complex64: max(code, -32767) * s, s = scale * (1/32767)
__device__ __forceinline__ float2 sn16_unpack(uint32_t w, float s) {
    const int re = max((int)(int16_t)(w & 0xffffu), -32767);
    const int im = max((int)(int16_t)(w >> 16), -32767);
    return make_float2(__fmul_rn((float)re, s), __fmul_rn((float)im, s));
}
constexpr float kInv32767 = 1.0f / 32767.0f;

struct RedLaunch {
    GView g;
    int n, n_bf, nq, nsplit, kps;
    double dq;
    const int32_t* qlist;   // null: identity over the half plane
    float4* ktab;           // [n_bf]
    float* chik;            // [n_bf][kChiStride]
    const float* kxcol;     // [ncol]: float32 k_x of each detector column, as in ktab
    int ncol;
    float inv_dk, ccol;     // 1 / detector pitch, column of k_x = 0 (starting points only)
    float2* Opart;          // [nsplit][B][nq]
    int* Npart;             // [nsplit][B][nq]
    int* status;            // nonzero after a kernel wait ran out (zeroed by the prep kernel)
    int shared_tilt;        // every set has the same float32 tilt centre
    int depth;              // weights include the depth-spread factor (SetBatch::depth_a)
};

// dcpart (may be null): per-256-pixel-block sums of Re G(0,k) in float64
// (G must then be a half plane: entry 0 is q = 0)
cudaError_t launch_prep(const int32_t* bf_idx, int n_bf, int det_x, double cy, double cx, double dk,
                        const SetBatch& sb, float4* ktab, float* chik, float* kxcol, int* status, const GView& g,
                        double* dcpart, cudaStream_t st);
cudaError_t launch_reduce(const RedLaunch& L, const SetBatch& sb, cudaStream_t st);
// the single-set pass over the whole half plane with TMA-streamed G rows
// (recon_tma.cu), where the layout allows it (complex64 half plane, 16-byte
// aligned rows)
bool recon_tma_applies(const RedLaunch& P, const SetBatch& sb);
cudaError_t launch_recon_tma(const RedLaunch& P, const SetBatch& sb, cudaStream_t st);
cudaError_t launch_reduce_depth(const RedLaunch& L, const SetBatch& sb, cudaStream_t st);  // reduce_depth.cu
cudaError_t launch_finalize(const float2* Opart, const int* Npart, int nsplit, int B, int nq,
                            const int* status, float2* O, int32_t* N, cudaStream_t st);
cudaError_t launch_phase(const float2* O, const int32_t* N, const double* dcpart, int nsplit,
                         int n_bf, int n, float2* Y, const float2* tw, float* phase,
                         cudaStream_t st);
// total[0] = sum of part[0..nparts) in that order (float64)
cudaError_t launch_dc_total(const double* part, int nparts, double* total, cudaStream_t st);
cudaError_t launch_score(const float2* O, const int32_t* N, int B, int nq, double* score,
                         cudaStream_t st);
// per-BF phase moments (moments.cu): Y holds moments_chunk_bytes(n), part
// moments_part_bytes(n)
size_t moments_chunk_bytes(int n);
size_t moments_part_bytes(int n);
cudaError_t launch_moments(const GView& g, int n, int n_bf, const float4* ktab, const SetBatch& sb, double dq,
                           const float2* tw, void* Y, void* part, float* mean, float* var, cudaStream_t st);
// compact storage (compact.cu)
cudaError_t launch_compact_g16(const float2* G, int n, int n_bf, int srows, uint32_t* G16, float* scale,
                               cudaStream_t st);
cudaError_t launch_compact_band(const void* G, int fmt, size_t plane, int n_bf, const int32_t* band, int nq,
                                void* dst, cudaStream_t st);

// the argument checks of ssb_reconstruct on a complex64 G, without the
// workspace's (api.cu): SSB_OK or the status ssb_reconstruct would return,
// with the message set
int check_reconstruct_args(const void* G_dev, const ssb_geometry* geom, const int32_t* bf_idx_dev, int n_bf,
                           const ssb_aberr* set, const void* O_dev, const int32_t* N_dev, const float* phase_dev);

// launch bookkeeping (api.cu)
void count_launch(int k = 1);

// record `msg` (plus the CUDA error text when err != cudaSuccess) as this
// thread's last error and return `code` (api.cu)
int set_last_error(int code, const char* msg, cudaError_t err);

}  // namespace ssb
