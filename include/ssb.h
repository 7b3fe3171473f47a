/*
 * ssb.h -- C ABI of the GB300 single-sideband (SSB) direct-ptychography library.
 *
 * The library computes, on one GPU, the data-parallel hot path of
 * aberration-corrected SSB ptychography from 4D-STEM frames:
 *
 *   1. G(q,k): gather the bright-field (BF) detector pixels from raw
 *      (scan_y, scan_x, det_y, det_x) frames and take the 2D real-to-complex
 *      FFT over the two scan axes for every BF pixel, stored as the Hermitian
 *      half plane (n, n/2+1).  Source: quantem.gpu "Historical WebGPU G(q,k)
 *      memory experiment", sections "Why herm is exactly lossless" and
 *      "Implementation" (G is the scan-space FFT of real intensity traces, so
 *      G(-q,k) = conj G(q,k) and the half plane is lossless).
 *   2. Per scan frequency q, the trotter-masked, aberration-phase-weighted sum
 *      over BF pixels k, for one or B <= 8 aberration sets per pass.  Source:
 *      quantem.gpu "Tilt-corrected SSB on CUDA: fit and preview speed",
 *      sections "Where the time went" and "Changes" (per (k, q, set): chi,
 *      aperture tests, sincos; per-set accumulators unrolled to a compile-time
 *      maximum).
 *   3. The object estimate: the corrected half-plane spectrum is summed over k,
 *      normalised, and brought back to real space by one complex-to-real
 *      inverse FFT plus atan2.  Source: "Historical WebGPU G(q,k) memory
 *      experiment", section "Object-redraw fast path" (mean over BF in Fourier
 *      space, then one inverse 2D FFT and one atan2); "Tilt-corrected SSB on
 *      CUDA", section "Open" (the corrected spectrum is anti-Hermitian except
 *      at DC, so a half-plane complex-to-real transform suffices).
 *
 * Conventions (the plainest reading of the pages; all fixed here):
 *   - Detector pixel (i, j) has k = ((j - det_center_x) Dk, (i - det_center_y) Dk),
 *     Dk = det_pitch_invA, detector rotation 0.
 *   - Half-plane entry (row, col), row in [0, n), col in [0, n/2], is the scan
 *     frequency q = (f_x, f_y) dq with f_x = col, f_y = row for row < n/2 and
 *     row - n otherwise, dq = 1 / (n scan_step_A).
 *   - Aperture of a set: A(v) = 1 iff |v - k_t|^2 <= (alpha/lambda)^2, with
 *     k_t = (tilt_x, tilt_y)/lambda.  Evaluated as the float32 sequence
 *     dx = px - tx; dy = py - ty; d2 = dx*dx + dy*dy; d2 <= r2, every step a
 *     separately rounded IEEE float32 operation (no fused multiply-add), with
 *     px, py = float32(k) -/+ float32(q), tx, ty = float32(k_t) and
 *     r2 = float32((alpha/lambda)^2).  Integer outcomes (trotter membership,
 *     N(q)) are therefore reproducible bit for bit.
 *   - Trotters: a = A(k), m = A(k - q), p = A(k + q); T- = a & m & !p,
 *     T+ = a & p & !m.  On T- the weight is exp(-i (chi(k) - chi(k - q))), on
 *     T+ it is -exp(+i (chi(k) - chi(k + q))); chi is the Krivanek aberration
 *     function of v - k_t (12 a/b coefficients through 4th order, Angstrom).
 *     O(q) = sum_k G(q,k) w(q,k), N(q) = |T-(q)| + |T+(q)|.
 *   - Phase image: S(q) = O(q)/N(q) (0 where N = 0), zeroed on the Nyquist row
 *     f_y = -n/2 and column f_x = n/2 and at DC; b = irfft2(-i S) with numpy
 *     semantics (1/n^2 normalisation, imaginary parts of self-conjugate bins
 *     dropped); a = mean_k G(0,k) / n^2; phase = atan2(b, a).
 *   - Score of a set over a band list: sum_q |O(q)|^2 / sum_q N(q).
 *
 * Ownership and asynchrony: every device buffer is owned by the caller.  The
 * library never allocates or frees memory; kernels that need scratch space use
 * the caller's workspace, sized by ssb_workspace_bytes().  Device calls are
 * asynchronous on the given stream (a cudaStream_t passed as void*; NULL is the
 * legacy default stream) and never synchronise the host.
 *
 * Errors: every entry point returns an ssb_status.  Argument checks happen on
 * the host before anything is launched; on SSB_CUDA_ERROR the launch error
 * text is available from ssb_last_error() (thread-local).  Checks cover null
 * pointers, sizes and workspace size; the contents of device buffers
 * (bf_idx_dev, band_dev) are the caller's responsibility: every index must be
 * in range (detector indices < det_y*det_x, band entries < n*(n/2+1)).
 */
#ifndef SSB_H
#define SSB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Scan and detector geometry.  The scan is n x n (n a power of two, 8..1024). */
typedef struct ssb_geometry {
    int n;
    int det_y, det_x;
    double scan_step_A;      /* Delta: scan step (Angstrom)                   */
    double det_pitch_invA;   /* Dk: detector pixel pitch (1/Angstrom)         */
    double wavelength_A;     /* lambda (Angstrom)                             */
    double semiangle_rad;    /* alpha: probe-forming aperture semi-angle      */
    double det_center_y;     /* detector pixel coordinate of k_y = 0          */
    double det_center_x;     /* detector pixel coordinate of k_x = 0          */
} ssb_geometry;

/* One aberration set: Krivanek a/b coefficients (Angstrom) and probe tilt. */
typedef struct ssb_aberr {
    double C10, C12a, C12b, C21a, C21b, C23a, C23b, C30, C32a, C32b, C34a, C34b;
    double tilt_x_rad, tilt_y_rad;
} ssb_aberr;

typedef enum ssb_dtype { SSB_U16 = 0, SSB_F32 = 1 } ssb_dtype;

typedef enum ssb_status {
    SSB_OK = 0,
    SSB_INVALID_ARG = 1,          /* null pointer, non-positive size, bad dtype/op     */
    SSB_UNSUPPORTED = 2,          /* n not a power of two in [8, 1024], B not in 1..8  */
    SSB_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < ssb_workspace_bytes(...)               */
    SSB_CUDA_ERROR = 4            /* a launch failed; see ssb_last_error()             */
} ssb_status;

typedef enum ssb_op {
    SSB_OP_BUILD = 0, SSB_OP_RECON = 1, SSB_OP_SCORE = 2, SSB_OP_MOMENTS = 3, SSB_OP_PHASE = 4
} ssb_op;

#define SSB_MAX_SETS 8
#define SSB_MIN_N 8
#define SSB_MAX_N 1024

/*
 * Bright-field pixel set (host only, no GPU).  Pixels (i, j) with
 *   ((j - cx) Dk - tx/lambda)^2 + ((i - cy) Dk - ty/lambda)^2 <= (alpha/lambda)^2
 * evaluated in float64 in exactly that order (no fused multiply-add), tilt from
 * `base`.  Output: row-major detector indices i*det_x + j, ascending.
 * `out` (host, may be NULL) must hold det_y*det_x entries; *n_bf receives the
 * count.  Source: "Historical WebGPU G(q,k) memory experiment", section
 * "Gotchas recorded" (only aperture-active BF pixels carry G).
 */
int ssb_bf_indices(const ssb_geometry* geom, const ssb_aberr* base,
                   int32_t* out, int* n_bf);

/*
 * Band list (host only).  Half-plane entries row*(n/2+1)+col with
 * (qmin/dq)^2 <= f_y^2 + f_x^2 <= (qmax/dq)^2, bounds in float64, ascending.
 * `out` (host, may be NULL) must hold n*(n/2+1) entries; *nq receives the
 * count.  Source: "Tilt-corrected SSB on CUDA", section "Setup" (fit band
 * 0.2 to 0.9 1/A, 44,247 frequencies on a 512^2 scan).
 */
int ssb_band_indices(const ssb_geometry* geom, double qmin, double qmax,
                     int32_t* out, int* nq);

/*
 * Bytes of device workspace an operation needs (0 on invalid arguments).
 * op = SSB_OP_BUILD, SSB_OP_RECON (ssb_reconstruct and ssb_reconstruct_sums;
 * B ignored, nq ignored), SSB_OP_SCORE (B sets over nq band entries),
 * SSB_OP_MOMENTS (B, nq ignored) or SSB_OP_PHASE (ssb_phase_from_sums; n_bf,
 * B, nq ignored but n_bf must be >= 1).  The workspace must be 256-byte
 * aligned.
 */
size_t ssb_workspace_bytes(const ssb_geometry* geom, int n_bf, int op, int B, int nq);

/*
 * G(q,k) build.  frames: device, (n, n, det_y, det_x) uint16 or float32,
 * contiguous.  bf_idx_dev: device int32[n_bf] detector indices.  G_dev:
 * device complex64 [n_bf][n][n/2+1] (q_x fastest), fully overwritten.
 * G(q,k) = sum_r x_k(r) exp(-2 pi i (f_y r_y + f_x r_x)/n), float32 arithmetic.
 * Source: "Historical WebGPU G(q,k) memory experiment", sections
 * "Implementation" and "Memory planning table" (layout and size
 * n_bf * n * (n/2+1) * 8 bytes).
 * For n = 512 and uint16 frames the work runs on two library-internal
 * streams per device (created on the first such call, kept for the process):
 * they wait on an event recorded on `stream` and `stream` waits on their
 * last event, so ordering against the caller's stream is as for a single
 * launch.  Concurrent builds on one device are serialised on the host while
 * their launches are issued.
 */
int ssb_build_G(const void* frames, int dtype, const ssb_geometry* geom,
                const int32_t* bf_idx_dev, int n_bf, void* G_dev,
                void* ws, size_t ws_bytes, void* stream);

/*
 * G(q,k) build from frames in HOST memory (page-locked for full copy speed).
 * Only bright-field pixels carry G ("Historical WebGPU G(q,k) memory
 * experiment", sections "Implementation" and "Gotchas recorded"), so only
 * their bounding box on the detector crosses the host link: rows r0..r1 and
 * columns c0..c1 are the extremes of bf_idx_host (c0 rounded down to an
 * even column unless the box spans the detector's width), and one pitched
 * copy moves that box of every frame into the workspace (a 2D copy of whole
 * rows when the box spans the detector's width, else a 3D copy).  The copy
 * runs on a library-internal stream of the device (created on the first
 * call, kept for the process) that carries the copies of every
 * ssb_build_G_host call in call order: it waits on an event recorded on
 * `stream`, and `stream` waits on its completion, so ordering against the
 * caller's stream is as for a copy on `stream`, while the copy of the next
 * call (from another stream) can start as soon as this one ends.  The build
 * then runs on `stream` as ssb_build_G on the box; G_dev is bit-identical to
 * what ssb_build_G gives on device frames.
 * frames_host: (n, n, det_y, det_x) uint16 or float32, contiguous; it must
 * stay valid and unmodified until the copy has completed (any later work on
 * `stream` completing implies it).
 * bf_idx_host, bf_idx_dev: the same n_bf detector indices, host and device
 * copies.  The workspace must hold ssb_build_G_host_bytes() bytes.
 * Errors as ssb_build_G, plus SSB_INVALID_ARG for a host index outside the
 * detector.
 */
int ssb_build_G_host(const void* frames_host, int dtype, const ssb_geometry* geom,
                     const int32_t* bf_idx_host, const int32_t* bf_idx_dev, int n_bf,
                     void* G_dev, void* ws, size_t ws_bytes, void* stream);

/*
 * Workspace bytes ssb_build_G_host needs for this index list (host): the
 * staged bright-field box of every frame, the remapped index list and the
 * build workspace.  0 on invalid arguments.
 */
size_t ssb_build_G_host_bytes(const ssb_geometry* geom, int dtype, const int32_t* bf_idx_host, int n_bf);

/*
 * One reconstruction at one aberration set (set: host pointer).
 * Writes O_dev (complex64 [n][n/2+1]), N_dev (int32 [n][n/2+1]) and phase_dev
 * (float32 [n][n], row = scan_y).  Source: "Historical WebGPU G(q,k) memory
 * experiment", section "Object-redraw fast path"; "Tilt-corrected SSB on
 * CUDA", sections "Changes" and "Open".
 * When G_dev is 16-byte aligned (and n is even) the pass streams G's rows
 * through shared memory with bulk asynchronous copies whose barrier waits are
 * bounded in time; a wait that runs out (possible only after a fault
 * elsewhere on the device) cannot be reported by the asynchronous call, so it
 * leaves NaN in O_dev and phase_dev and -1 in N_dev instead.  Any other G_dev
 * alignment runs the same sums with per-thread loads.
 */
int ssb_reconstruct(const void* G_dev, const ssb_geometry* geom,
                    const int32_t* bf_idx_dev, int n_bf, const ssb_aberr* set,
                    void* O_dev, int32_t* N_dev, float* phase_dev,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * A reconstruction split over shards of the BF pixels (one shard per GPU, or
 * any partition of the BF list).  Every quantity the image needs is a sum over
 * BF pixels ("Tilt-corrected SSB on CUDA", section "Where the time went": the
 * reduction is a sum over k; "Historical WebGPU G(q,k) memory experiment",
 * section "Implementation": G is built per BF pixel), so each shard reduces
 * its own pixels and the shards' results are added (an all-reduce across
 * GPUs) before one call forms the image.
 *
 * ssb_reconstruct_sums: for the n_bf pixels given (G_dev holds their half
 * planes, [n_bf][n][n/2+1]; bf_idx_dev their detector indices), writes the
 * raw sums O_dev (complex64 [n][n/2+1]) and N_dev (int32 [n][n/2+1]) exactly
 * as ssb_reconstruct does, and g0_sum_dev[0] (float64) = sum_k Re G(0,k) over
 * these pixels.  Workspace: ssb_workspace_bytes(..., SSB_OP_RECON, ...).
 * Errors as ssb_reconstruct (g0_sum_dev must not be NULL).
 *
 * ssb_phase_from_sums: phase_dev (float32 [n][n]) from the shards' summed O,
 * N and G(0,k) sum, with n_bf_total the number of BF pixels over all shards
 * (a = g0_sum / n_bf_total / n^2, the rest as ssb_reconstruct).  Workspace:
 * ssb_workspace_bytes(geom, 1, SSB_OP_PHASE, 1, 1).  With one shard holding
 * every pixel, the two calls give ssb_reconstruct's O, N and phase bit for
 * bit.  Errors: SSB_INVALID_ARG for a NULL pointer or n_bf_total < 1.
 */
int ssb_reconstruct_sums(const void* G_dev, const ssb_geometry* geom,
                         const int32_t* bf_idx_dev, int n_bf, const ssb_aberr* set,
                         void* O_dev, int32_t* N_dev, double* g0_sum_dev,
                         void* ws, size_t ws_bytes, void* stream);

int ssb_phase_from_sums(const void* O_dev, const int32_t* N_dev, const double* g0_sum_dev,
                        int n_bf_total, const ssb_geometry* geom, float* phase_dev,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * Batched scoring of B aberration sets (sets: host array of B) over a band
 * list (band_dev: device int32[nq] half-plane entries).  Writes O_dev
 * (complex64 [B][nq]), N_dev (int32 [B][nq]) and score_dev (float64 [B]).
 * Set s of a B-set call equals the corresponding single-set call bit for bit.
 * Source: "Tilt-corrected SSB on CUDA", sections "Where the time went" and
 * "Changes" (eight sets per pass, per-set loops unrolled to a compile-time
 * maximum with a uniform b < B guard).
 */
int ssb_score_batch(const void* G_dev, const ssb_geometry* geom,
                    const int32_t* bf_idx_dev, int n_bf, const ssb_aberr* sets, int B,
                    const int32_t* band_dev, int nq,
                    void* O_dev, int32_t* N_dev, double* score_dev,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * Compact storage of G.
 *
 * herm16 (source: "Historical WebGPU G(q,k) memory experiment", sections
 * "Implementation", "Memory planning table" and "Scan-size sweep"): each
 * half-plane entry is one 32-bit word holding two 16-bit two's complement
 * codes, the real part in bits 0-15 and the imaginary part in bits 16-31,
 *   code = floor(0.5 + 32767 * clamp(v / scale, -1, 1)),
 * every operation a separately rounded float32 operation, with scale the
 * largest |G| (float32 sqrt of the float32 re*re + im*im) over a block of the
 * pixel's half plane: the whole plane (rows_per_scale = n, the page's preview
 * form, 4 bytes per BF pixel) or one q row (rows_per_scale = 1, the page's
 * follow-up, n scales per BF pixel).  A block whose largest |G| is 0 has scale
 * 0 and codes 0.  Scales are float32 [n / rows_per_scale][n_bf] (block-major).
 * A reader takes max(code, -32767) * (scale * (1/32767)) in float32.
 *
 * Band-compacted copy (no page describes it; the scoring passes of a fit read
 * only the band, 78 passes per fit in "Tilt-corrected SSB on CUDA", section
 * "Where the time went"): entry i of row k is the half-plane entry band[i] of
 * BF pixel k, [n_bf][nq], in either element format.  herm16 scales are not
 * copied: the band entry's q row still selects the scale.
 */
typedef enum ssb_gfmt { SSB_G_C64 = 0, SSB_G_SN16 = 1 } ssb_gfmt;

/* A stored G as the reductions read it (every pointer device memory). */
typedef struct ssb_gstore {
    const void* G;          /* complex64 (SSB_G_C64) or herm16 words (SSB_G_SN16)        */
    int fmt;                /* ssb_gfmt                                                   */
    const float* scale;     /* SSB_G_SN16: [n / rows_per_scale][n_bf]; else ignored       */
    int rows_per_scale;     /* SSB_G_SN16: 1 or n; else ignored                           */
    int band_compact;       /* 0: [n_bf][n][n/2+1] half planes; 1: [n_bf][nq] band copy   */
} ssb_gstore;

/*
 * herm16 from a complex64 G (G_dev: [n_bf][n][n/2+1]).  Writes G16_dev (uint32
 * [n_bf][n][n/2+1]) and scale_dev (float32 [n / rows_per_scale][n_bf]); the
 * outputs must not overlap G_dev.  Deterministic: the codes and scales are a
 * function of G alone (bit for bit).  Errors: SSB_INVALID_ARG for a null
 * pointer or n_bf < 1, SSB_UNSUPPORTED for rows_per_scale not in {1, n}.
 */
int ssb_compact_G16(const void* G_dev, const ssb_geometry* geom, int n_bf, int rows_per_scale,
                    void* G16_dev, float* scale_dev, void* stream);

/*
 * Band-compacted copy of a half-plane G (src->band_compact must be 0; only
 * src->G and src->fmt are read): dst_dev[k][i] = G[k][band[i]], 8-byte entries
 * for SSB_G_C64, 4-byte words for SSB_G_SN16.  band_dev: device int32[nq] of
 * half-plane entries (as ssb_band_indices writes them).  Bit-exact copy;
 * dst_dev must not overlap the source.
 * Errors: SSB_INVALID_ARG for a null pointer, n_bf < 1, nq out of
 * [1, n*(n/2+1)], an unknown format or a band-compacted source.
 */
int ssb_compact_band(const ssb_gstore* src, const ssb_geometry* geom, int n_bf, const int32_t* band_dev,
                     int nq, void* dst_dev, void* stream);

/*
 * ssb_reconstruct from any stored G (G: host pointer to the descriptor; the
 * half plane is needed, so G->band_compact must be 0).  With SSB_G_C64 this is
 * ssb_reconstruct bit for bit.  Errors as ssb_reconstruct, plus
 * SSB_INVALID_ARG for a band-compacted G, a missing scale array or an unknown
 * format, SSB_UNSUPPORTED for rows_per_scale not in {1, n}.
 */
int ssb_reconstruct_g(const ssb_gstore* G, const ssb_geometry* geom,
                      const int32_t* bf_idx_dev, int n_bf, const ssb_aberr* set,
                      void* O_dev, int32_t* N_dev, float* phase_dev,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * ssb_score_batch from any stored G.  A band-compacted G must come from the
 * same band_dev and nq.  Every (G format, layout) gives, per set, the same
 * arithmetic in the same order as ssb_score_batch on the G it stores, so a
 * band-compacted complex64 copy scores bit for bit like the half plane.
 * Errors as ssb_score_batch, plus those of ssb_reconstruct_g for the
 * descriptor.
 */
int ssb_score_batch_g(const ssb_gstore* G, const ssb_geometry* geom,
                      const int32_t* bf_idx_dev, int n_bf, const ssb_aberr* sets, int B,
                      const int32_t* band_dev, int nq,
                      void* O_dev, int32_t* N_dev, double* score_dev,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * Batched scoring with a depth (defocus) spread per set: ssb_score_batch_g
 * with each trotter term's weight multiplied by the real factor
 * sinc(pi lambda t_s D / 2), sinc(x) = sin(x)/x, where t_s = depth_A[s] is set
 * s's spread (Angstrom; the defocus runs uniformly over C10 +/- t_s/2) and D =
 * |v_k|^2 - |v_{k-q}|^2 on T-, |v_k|^2 - |v_{k+q}|^2 on T+ (v = k - k_t, the
 * squared distances of the float32 aperture tests).  That factor is the mean
 * of exp(i pi lambda z D) over the spread, so the weight is the depth-0 weight
 * times the transfer's own attenuation.  N counts trotter pixels and the score
 * is sum |O|^2 / sum N as in ssb_score_batch.  t_s = 0 gives ssb_score_batch_g
 * bit for bit; set s does not depend on B (bit for bit).  Source:
 * "Tilt-corrected SSB on CUDA", sections "Changes" (the fit kernel at depth
 * 136 A: two sincos and two sin per term) and "Results" (the depth spread is a
 * fitted parameter); "Where the 9 s of regularized preparation goes", list
 * item 2 (chi, sinc and phase factor of a transfer term).  The pages do not
 * write the depth model out; this is the plainest reading.
 * depth_A: host array of B values, each finite and >= 0.  Errors as
 * ssb_score_batch_g, plus SSB_INVALID_ARG for a NULL, negative or non-finite
 * depth.
 */
int ssb_score_batch_depth(const ssb_gstore* G, const ssb_geometry* geom,
                          const int32_t* bf_idx_dev, int n_bf, const ssb_aberr* sets,
                          const double* depth_A, int B, const int32_t* band_dev, int nq,
                          void* O_dev, int32_t* N_dev, double* score_dev,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * Per-BF phase moments at one aberration set (set: host pointer): for every BF
 * pixel k, the corrected plane S_k(q) = G(q,k) w(q,k) on the trotter pixels
 * of k (0 elsewhere, and at DC and on the Nyquist row and column), its image
 * b_k = irfft2(-i S_k) (numpy semantics) and the angle atan2(b_k, a_k) with
 * a_k = Re G(0,k) / n^2; writes the mean over the n_bf pixels (mean_dev) and
 * the population variance (var_dev), float32 [n][n] each, row = scan_y.  The
 * sums are deterministic (fixed order; float32 within groups of at most 4 BF
 * pixels, float64 across them).  G: host pointer to the descriptor; the half
 * plane is needed (G->band_compact must be 0).  Source: "Historical WebGPU
 * G(q,k) memory experiment", section "Object-redraw fast path" (the exact
 * per-BF path, mean(angle(object)), and the variance the loss uses);
 * "Tilt-corrected SSB on CUDA", sections "Changes" (Loss path) and "Open".
 * Errors as ssb_reconstruct_g.
 */
int ssb_phase_moments(const ssb_gstore* G, const ssb_geometry* geom,
                      const int32_t* bf_idx_dev, int n_bf, const ssb_aberr* set,
                      float* mean_dev, float* var_dev,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * ssb_reconstruct for callers that cannot allocate device memory.
 *
 * No page describes this call; it has no counterpart in the method.  It exists
 * for callers that are not allowed to call cudaMalloc or any allocating
 * routine: plugin code running inside a host application that owns the device
 * allocator, or acquisition loops that must not allocate once started.  It
 * computes exactly what ssb_reconstruct computes (same kernels, same outputs,
 * same argument meaning, layout and status codes), but its scratch memory is a
 * fixed array of SSB_NOALLOC_SCRATCH_BYTES inside the library (held by every
 * GPU that loads the library until the process exits) instead of a caller
 * workspace.  It calls no allocating routine.
 *   - The arguments are checked first, as ssb_reconstruct checks them (same
 *     status codes).  Then calls whose scratch need,
 *     ssb_workspace_bytes(geom, n_bf, SSB_OP_RECON, 1, 1), exceeds
 *     SSB_NOALLOC_SCRATCH_BYTES return SSB_UNSUPPORTED before launching
 *     anything (every n <= 512 fits; n = 1024 does not).
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress, a host-side lookup; nothing is cached, so calls
 *     after a device reset use the new context's array).  The first call on a
 *     device may load the library's device code there: make it before any
 *     stream capture.
 *   - All calls share the one array, which keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls that overlap on the GPU
 *     (different streams or host threads) race on it: serialise them.
 */
#define SSB_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

int ssb_reconstruct_noalloc(const void* G_dev, const ssb_geometry* geom,
                            const int32_t* bf_idx_dev, int n_bf, const ssb_aberr* set,
                            void* O_dev, int32_t* N_dev, float* phase_dev, void* stream);

/* Text of the last error on this host thread ("" if none). */
const char* ssb_last_error(void);

/* Number of kernels this library has launched in this process. */
long long ssb_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SSB_H */
