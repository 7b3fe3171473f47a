// noalloc.cu -- ssb_reconstruct_noalloc: a reconstruction that allocates nothing.
//
// Some callers cannot call cudaMalloc: plugin code running inside a host
// application that owns the device allocator, or acquisition loops that must
// not allocate once they have started.  This entry point runs the same kernels
// as ssb_reconstruct, with the scratch memory they need (twiddles, k tables,
// per-split partial sums, the complex-to-real intermediate) taken from a
// file-scope device array instead of a caller workspace.
//
// * The array is kNoallocScratchBytes (16 MiB); every GPU that loads the
//   library holds it until the process exits.  Arguments are checked first,
//   exactly as ssb_reconstruct checks them (same status codes); then calls
//   whose scratch need (ssb_workspace_bytes(..., SSB_OP_RECON, ...)) exceeds
//   the array are rejected with SSB_UNSUPPORTED before anything is launched.
//   16 MiB covers every n <= 512 (the full 512^2 workload needs ~12 MiB, and
//   13.3 MiB with a whole 192 x 192 detector bright) but
//   not n = 1024.
// * Host code cannot use the array's name as a device address, so every call
//   asks the runtime for the address on the current device with
//   cudaGetSymbolAddress (a host-side lookup) and passes that pointer on.
//   Nothing is cached, so a call made after a device reset sees the address of
//   the array in the new context.  The first call on a device may load the
//   library's device code there; make it before any stream capture.
// * Every call shares the one array and it keeps the last call's contents.
//   Nothing in it needs to start at zero: each kernel writes its part of the
//   scratch before any kernel reads it.  Calls that overlap on the GPU (two
//   streams, or two host threads) race on the array; serialise them.
#include "internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = SSB_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch array on the current device.  Returns SSB_OK
// or an error code with the message already set.
static int scratch_for_current_device(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
        return ssb::set_last_error(SSB_CUDA_ERROR, "cudaGetSymbolAddress of the scratch array failed", e);
    *out = p;
    return SSB_OK;
}

}  // namespace

extern "C" int ssb_reconstruct_noalloc(const void* G_dev, const ssb_geometry* geom, const int32_t* bf_idx_dev,
                                       int n_bf, const ssb_aberr* set, void* O_dev, int32_t* N_dev,
                                       float* phase_dev, void* stream) {
    int rc = ssb::check_reconstruct_args(G_dev, geom, bf_idx_dev, n_bf, set, O_dev, N_dev, phase_dev);
    if (rc != SSB_OK) return rc;
    const size_t need = ssb_workspace_bytes(geom, n_bf, SSB_OP_RECON, 1, 1);
    if (need > kNoallocScratchBytes)
        return ssb::set_last_error(SSB_UNSUPPORTED,
                                   "scratch need exceeds the library's fixed 16 MiB array "
                                   "(use ssb_reconstruct with a caller workspace)",
                                   cudaSuccess);
    void* ws = nullptr;
    if ((rc = scratch_for_current_device(&ws)) != SSB_OK) return rc;
    return ssb_reconstruct(G_dev, geom, bf_idx_dev, n_bf, set, O_dev, N_dev, phase_dev, ws, kNoallocScratchBytes,
                           stream);
}
