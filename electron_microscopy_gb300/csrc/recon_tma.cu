// recon_tma.cu -- the single-set trotter-masked reduction over the whole
// half plane (the reconstruction's pass), with the G rows streamed into
// shared memory by bulk asynchronous copies (TMA) instead of per-thread loads.
//
// The terms, their order and the trotter classification are those of
// ssb_reduce<1, shared tilt, complex64> (reduce.cu, reduce_kernel.cuh): a
// block owns 256 consecutive half-plane entries q, grid.y splits the
// bright-field list, and each block walks its split's pixels k in list
// order.  Two things differ.  The float32 evaluation of a term is leaner:
// chi(k -/+ q) comes from a per-row quartic in k_x, and the T+ sign is
// folded into the phase (see step below).  And G(q, k) reaches the threads
// through shared memory:
//
//  * the split's pixels are taken in groups of kTmaPix; a group's G row
//    segments (256 entries, 2 KB each) and its k-table entries are copied
//    into one stage of a kTmaStages-deep shared-memory ring by one thread,
//    with an mbarrier counting the bytes (cp.async.bulk ... complete_tx);
//  * threads wait on the stage's barrier and read G from shared memory, so
//    no registers hold loads in flight and the copies of the next stages
//    proceed while the block computes;
//  * the last warp to finish a stage refills it with the group kTmaStages
//    ahead (a shared-memory counter; nobody blocks on the refill).
//
// Every wait is bounded in time.  A wait that runs out (which only a fault
// elsewhere could cause) sets the status word, the block stops, waits (again
// bounded) for its own copies still in flight, and the finalize kernel then
// writes NaN into O and -1 into N.
#include "reduce_kernel.cuh"

namespace ssb {

constexpr int kTmaPix = 8;      // pixels per stage
constexpr int kTmaStages = 3;   // stages in the ring
constexpr int kTmaThreads = 256;
constexpr int kTmaWarps = kTmaThreads / 32;

struct TmaRing {
    float2 g[kTmaStages][kTmaPix][kTmaThreads];
    float4 k[kTmaStages][kTmaPix];
    unsigned long long full[kTmaStages];
    int drained[kTmaStages];  // warps done with the stage's current group
    int issued[kTmaStages];   // groups issued into the stage so far
    int fail;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// a few KB of copies complete in microseconds; 2 s (or 2^26 polls) means
// something else has failed
constexpr uint64_t kWaitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (uint32_t it = 0; it < (1u << 26); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_ns() - t0 > kWaitNs) return false;
    }
    return false;
}
__device__ __forceinline__ bool mbar_wait(const unsigned long long* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    return mbar_try_wait(a, parity) || mbar_wait_slow(a, parity);
}
// global -> shared bulk copy (16-byte aligned addresses, size a multiple of
// 16), completing `bytes` transactions on the barrier
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, unsigned long long* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// coefficients (a3, a2, a1, a0) of P(y - s) for the quartic
// P(x) = h0 x^4 + a3 x^3 + a2 x^2 + a1 x + a0 (Taylor shift by repeated
// synthetic division; the leading coefficient stays h0)
__device__ __forceinline__ float4 shift_quartic(float h0, float4 a, float s) {
    const float ns = -s;
    float b1 = a.x, b2 = a.y, b3 = a.z, b4 = a.w;
    b1 = __fmaf_rn(ns, h0, b1);
    b2 = __fmaf_rn(ns, b1, b2);
    b3 = __fmaf_rn(ns, b2, b3);
    b4 = __fmaf_rn(ns, b3, b4);
    b1 = __fmaf_rn(ns, h0, b1);
    b2 = __fmaf_rn(ns, b1, b2);
    b3 = __fmaf_rn(ns, b2, b3);
    b1 = __fmaf_rn(ns, h0, b1);
    b2 = __fmaf_rn(ns, b1, b2);
    b1 = __fmaf_rn(ns, h0, b1);
    return make_float4(b1, b2, b3, b4);
}

__global__ void __launch_bounds__(kTmaThreads, 4) ssb_recon_tma(RedLaunch P, SetBatch sb) {
    extern __shared__ __align__(128) unsigned char tma_smem[];
    TmaRing& R = *reinterpret_cast<TmaRing*>(tma_smem);
    const int tid = threadIdx.x, lane = tid & 31;
    const int q0 = blockIdx.x * kTmaThreads;
    const int nqb = min(kTmaThreads, P.nq - q0);  // entries of this block (even)
    const int qi = q0 + tid;
    const bool valid = tid < nqb;
    const int H = P.n / 2 + 1;
    const int e = valid ? qi : 0;
    const int row = e / H, col = e - row * H;
    const int fy = row < P.n / 2 ? row : row - P.n;
    const float qx = __double2float_rn(__dmul_rn((double)col, P.dq));
    const float qy = __double2float_rn(__dmul_rn((double)fy, P.dq));
    const int split = blockIdx.y;
    const int kb = split * P.kps;
    const int ke = min(P.n_bf, kb + P.kps);
    const int nk = max(ke - kb, 0);
    const int ng = (nk + kTmaPix - 1) / kTmaPix;
    const float2* G = static_cast<const float2*>(P.g.G);
    const size_t gstride = P.g.stride;
    const uint32_t gbytes = (uint32_t)nqb * (uint32_t)sizeof(float2);

    // one thread: group grp's G row segments and k-table entries into its stage
    auto issue = [&](int grp) {
        const int s = grp % kTmaStages;
        const int k0 = kb + grp * kTmaPix, cnt = min(kTmaPix, ke - k0);
        mbar_expect_tx(&R.full[s], (uint32_t)cnt * (gbytes + (uint32_t)sizeof(float4)));
        for (int u = 0; u < cnt; ++u) bulk_g2s(&R.g[s][u][0], G + (size_t)(k0 + u) * gstride + q0, gbytes, &R.full[s]);
        bulk_g2s(&R.k[s][0], P.ktab + k0, (uint32_t)cnt * (uint32_t)sizeof(float4), &R.full[s]);
        R.issued[s] += 1;
    };
    if (tid == 0) {
        for (int s = 0; s < kTmaStages; ++s) {
            mbar_init(&R.full[s], 1);
            R.drained[s] = 0;
            R.issued[s] = 0;
        }
        R.fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0)
        for (int grp = 0; grp < min(kTmaStages, ng); ++grp) issue(grp);

    float2 acc = make_float2(0.f, 0.f);
    int cnt = 0;
    float4 row_m = make_float4(0.f, 0.f, 0.f, 0.f), row_p = row_m;
    RowRun run_m{0.0f, 0.0f}, run_p{0.0f, 0.0f};
    // the row state at a pixel that starts a detector row (or the split's
    // first pixel): the aperture runs at k -/+ q, and chi(k -/+ q) along the
    // row as a quartic in k_x itself (the quartic in v_x = k_x - s, shifted
    // by s = t_x +/- q_x), so that a step evaluates it at k_x directly
    auto row_enter = [&](float ky) {
        run_m = row_run(P.kxcol, P.ncol, P.inv_dk, P.ccol, ky, qx, qy, true, sb.s[0].tx, sb.s[0].ty, sb.r2);
        run_p = row_run(P.kxcol, P.ncol, P.inv_dk, P.ccol, ky, qx, qy, false, sb.s[0].tx, sb.s[0].ty, sb.r2);
        row_m = shift_quartic(sb.s[0].h[0], chi_row(sb.s[0].h, __fsub_rn(__fsub_rn(ky, qy), sb.s[0].ty)),
                              __fadd_rn(qx, sb.s[0].tx));
        row_p = shift_quartic(sb.s[0].h[0], chi_row(sb.s[0].h, __fsub_rn(__fadd_rn(ky, qy), sb.s[0].ty)),
                              __fsub_rn(sb.s[0].tx, qx));
    };
    // one pixel: the aperture tests are comparisons with the row's runs.  A
    // single-overlap pixel adds G exp(-2 pi i r), r the phase in turns
    // reduced to [-1/2, 1/2]: on T-, of d = chi(k) - chi(k - q); on T+, of
    // -d - 1/2 (d = chi(k) - chi(k + q)), since -exp(2 pi i d) equals
    // exp(-2 pi i (-d - 1/2)).  Every lane evaluates every pixel's term and
    // only active lanes accumulate: with no branch between them, the pixels'
    // dependent chains can interleave.
    auto step = [&](const float2* gsrc, float4 kd) {
        const uint32_t am = __float_as_uint(kd.z);
        const bool m = kd.x >= run_m.lo && kd.x <= run_m.hi;
        const bool p = kd.x >= run_p.lo && kd.x <= run_p.hi;
        const bool act = (am & 1u) && (m != p);
        const float2 gv = *gsrc;
        const float d = __fsub_rn(kd.w, chi_horner(sb.s[0].h[0], m ? row_m : row_p, kd.x));
        const float ds = m ? d : __fsub_rn(-0.5f, d);
        const float r = __fsub_rn(ds, rintf(ds));
        float sn, cs;
        __sincosf(__fmul_rn(kTwoPi, r), &sn, &cs);  // |argument| <= pi
        if (act) {
            acc.x = __fmaf_rn(gv.y, sn, __fmaf_rn(gv.x, cs, acc.x));
            acc.y = __fmaf_rn(-gv.x, sn, __fmaf_rn(gv.y, cs, acc.y));
            cnt += 1;
        }
    };

#pragma unroll 1
    for (int grp = 0; grp < ng; ++grp) {
        const int s = grp % kTmaStages;
        // the warp leaves together if any lane's wait ran out
        if (!__all_sync(0xffffffffu, mbar_wait(&R.full[s], (uint32_t)(grp / kTmaStages) & 1u))) {
            if (lane == 0) {
                atomicOr(P.status, 1);
                R.fail = 1;
            }
            break;
        }
        const int np = min(kTmaPix, ke - (kb + grp * kTmaPix));
        const float2* gs = &R.g[s][0][tid];
        float4 kd[kTmaPix];
        uint32_t f = grp == 0 ? kRowStart : 0u;
#pragma unroll
        for (int u = 0; u < kTmaPix; ++u) {
            kd[u] = R.k[s][u];
            f |= __float_as_uint(kd[u].z);
        }
        if (np == kTmaPix && !(f & kRowStart)) {
            // a whole group within one detector row: straight-line steps
#pragma unroll
            for (int u = 0; u < kTmaPix; ++u) step(gs + u * kTmaThreads, kd[u]);
        } else {
#pragma unroll 1
            for (int u = 0; u < np; ++u) {
                const float4 kdu = R.k[s][u];
                if ((__float_as_uint(kdu.z) & kRowStart) || (grp == 0 && u == 0)) row_enter(kdu.y);
                step(gs + u * kTmaThreads, kdu);
            }
        }
        // this warp is done with the stage; the last warp refills it (its
        // reads, and the other warps', ordered before the async copies)
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&R.drained[s], 1) == kTmaWarps - 1) {
                R.drained[s] = 0;
                __threadfence_block();
                if (grp + kTmaStages < ng) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(grp + kTmaStages);
                }
            }
        }
    }
    __syncthreads();
    if (R.fail) {
        // no copy may outlive the block: wait (bounded) for each stage's
        // last issued group
        if (tid == 0)
            for (int s = 0; s < kTmaStages; ++s)
                if (R.issued[s] > 0) (void)mbar_wait(&R.full[s], (uint32_t)(R.issued[s] - 1) & 1u);
        return;
    }
    if (valid) {
        const size_t o = (size_t)split * P.nq + qi;
        P.Opart[o] = acc;
        P.Npart[o] = cnt;
    }
}

bool recon_tma_applies(const RedLaunch& P, const SetBatch& sb) {
    return sb.B == 1 && P.shared_tilt && !P.depth && P.g.fmt == kGC64 && !P.g.band && !P.qlist && P.status &&
           P.kxcol && (P.nq % 2) == 0 && (P.g.stride % 2) == 0 && ((uintptr_t)P.g.G % 16) == 0 &&
           ((uintptr_t)P.ktab % 16) == 0;
}

cudaError_t launch_recon_tma(const RedLaunch& P, const SetBatch& sb, cudaStream_t st) {
    const size_t smem = sizeof(TmaRing);
    // set on every call: the attribute belongs to the current device's context
    const cudaError_t e = cudaFuncSetAttribute(ssb_recon_tma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((P.nq + kTmaThreads - 1) / kTmaThreads, P.nsplit);
    ssb_recon_tma<<<grid, kTmaThreads, smem, st>>>(P, sb);
    count_launch();
    return cudaGetLastError();
}

}  // namespace ssb
