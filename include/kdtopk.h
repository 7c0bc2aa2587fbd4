/*
 * kdtopk.h - C ABI of the fused, chunked top-K KL distillation loss over the
 * LM head, for NVIDIA B300 (sm_103a).
 *
 * Method: "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and
 * a Fused Chunked KL Loss" (arXiv 2608.03796).  The student is trained
 * against an offline cache of the teacher's top-K ids and probabilities
 * (aimodeling.com, "The Hidden Memory Bottleneck in LLM Distillation",
 * section "First cut"); the loss is fused with the output projection and
 * computed in sequence chunks, recomputing each chunk's logits in the backward
 * pass, so the [T,V] logit tensor never exists (same article, "Second cut";
 * thorstenmeyerai.com, "Making Knowledge Distillation Cheap Enough to Run at
 * Scale", pipeline steps "Train in chunks" and "Recompute backward").
 *
 * Definitions.  H[T,d] student hidden states, W[V,d] LM-head weights,
 * idx[T,K] teacher top-K ids, p[T,K] their probabilities (M_t = sum_k p_tk,
 * at most 1 in intended use), z = H W^T:
 *
 *   lse_t = log sum_j exp(z_tj)
 *   L     = sum_t sum_k p_tk (log p_tk - (z_{t,idx_tk} - lse_t)),  0 log 0 = 0
 *   G_t   = M_t softmax(z_t) - sum_k p_tk e_{idx_tk}     (legiblepapers.com
 *           summary, FAQ Q5: dense M-times-softmax term minus the sparse
 *           teacher correction at the top-K positions)
 *   dH    = dloss * G W,    dW = dloss * G^T H
 *
 * Conventions shared by every call below.
 *   - Pointers: all tensor pointers are DEVICE pointers owned by the caller
 *     and 16-byte aligned.  The library allocates no device memory; it uses
 *     the caller's workspace (see kd_topk_kl_workspace_size).
 *   - Layouts: row-major, no padding.  H [T,d] bf16, W [V,d] bf16,
 *     idx [T,K] int32, p [T,K] fp32, lse [T] fp32, dH [T,d] fp32,
 *     dW [V,d] fp32.  bf16 is passed as `const void*` (IEEE bfloat16 bits).
 *   - Sizes: T >= 1, d >= 8 with d % 8 == 0 (TMA row strides are multiples
 *     of 16 bytes), 1 <= K <= min(V, 1024), V >= 1, chunk >= 1.  T, V and chunk
 *     need not be multiples of any tile size.
 *   - Ids: duplicates within a row are allowed (each occurrence counts); p may
 *     hold zeros (padding).  A row with an id outside [0, V) contributes
 *     nothing (its loss, G row, dH row are 0) and the call reports
 *     KD_ERR_BAD_INDEX through kd_topk_kl_device_status.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *     default stream).  Every call is asynchronous on it: host-detectable
 *     errors are returned before anything is launched; device-detected errors
 *     (bad ids, a timed-out internal wait) are recorded in the workspace and
 *     read back by kd_topk_kl_device_status.
 *   - Concurrency: calls that share a workspace must be ordered on one
 *     stream.  Apart from the optional profiler (kd_profile_*), the library
 *     keeps no mutable global state.
 *   - CUDA graphs: forward, backward and both fused steps only launch kernels
 *     and set the workspace's status word on `stream`, so they can be
 *     captured and replayed (inputs, outputs and workspace at fixed
 *     addresses); read the status with kd_topk_kl_device_status outside the
 *     captured region.
 */
#ifndef KDTOPK_H
#define KDTOPK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KD_API __attribute__((visibility("default")))
#else
#define KD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kd_status {
  KD_OK = 0,
  KD_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, K > V ...      */
  KD_ERR_UNSUPPORTED = 2,  /* d % 8 != 0, misaligned pointer, K > 1024, no sm_103a GPU */
  KD_ERR_WORKSPACE = 3,    /* ws_bytes smaller than kd_topk_kl_workspace_size */
  KD_ERR_BAD_INDEX = 4,    /* device: an id outside [0, V) (row zeroed)       */
  KD_ERR_TIMEOUT = 5,      /* device: an internal pipeline wait ran out        */
  KD_ERR_CUDA = 6          /* a CUDA runtime/driver call failed                */
} kd_status;

/* Which calls a workspace must serve (bit mask). */
#define KD_WS_FORWARD 1
#define KD_WS_BACKWARD 2
#define KD_WS_FUSED 3

/*
 * Bytes of device workspace the calls selected by `what` need for this
 * problem.  The size depends on chunk, d, V and K (and on the current
 * device's SM count, which sets the split of the dH reduction), and only
 * through ceil(T / chunk) on T: the chunk working set (a [chunk,V] bf16
 * gradient operand and [chunk, V/256] softmax partials) is reused chunk after
 * chunk, so memory grows linearly in T only through the caller's own inputs
 * and outputs.  With KD_WS_FUSED and an even number of chunks per dW group
 * (below) the partials hold two chunks' rows, so that the step without the
 * recompute can run two chunks' forward GEMMs as one launch.  Returns 0 for
 * invalid sizes.
 * When chunk is a multiple of 128 the backward keeps G for a group of
 * consecutive chunks (up to 4096 rows, at most 4 chunks; environment variable
 * KD_DW_GROUP_ROWS, read once per process, changes the row target, 0 turns it
 * off) and runs one dW GEMM per group; the workspace size includes it.
 * Chunks of 256 rows or more run their GEMMs on two-CTA clusters (256-row
 * tiles; the chunk's rows are padded to a multiple of 256 in the workspace);
 * environment variable KD_PAIR=0 (read once per process) selects one CTA per
 * 128-row tile instead.
 */
KD_API size_t kd_topk_kl_workspace_size(int64_t T, int d, int V, int K, int chunk, int what);

/*
 * Forward: loss[0] = L (fp32 on the device; accumulated in fp64 over rows in
 * a fixed order), lse[T] = lse_t (saved for the backward), and, if
 * loss_rows != NULL, loss_rows[T] = L_t.  The logits of each chunk live only
 * in tensor memory: the projection, the softmax normaliser and the top-K
 * gather are fused (aimodeling.com "Second cut": output projection,
 * normalization and sparse teacher terms processed in sequence chunks).
 */
KD_API kd_status kd_topk_kl_forward(const void* H, const void* W, const int32_t* idx, const float* p,
                             int64_t T, int d, int V, int K, int chunk,
                             float* loss, float* lse, float* loss_rows,
                             void* workspace, size_t ws_bytes, void* stream);

/*
 * Backward: recomputes each chunk's logits (the pages' "recompute backward"
 * step), forms G in bf16 from lse (as written by the forward), then
 * dH = dloss * G W (overwritten) and dW = dloss * G^T H, accumulated in fp32
 * over chunks; dW is overwritten unless accumulate_dW != 0, in which case the
 * result is added to dW's contents.
 */
KD_API kd_status kd_topk_kl_backward(const void* H, const void* W, const int32_t* idx, const float* p,
                              const float* lse, int64_t T, int d, int V, int K, int chunk,
                              float dloss, float* dH, float* dW, int accumulate_dW,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * Forward and backward in one pass over the chunks: per chunk the logits are
 * computed once for the normaliser and once more for G.  Outputs as above
 * (loss_rows may be NULL).  The loop is pipelined by one chunk: chunk c's G
 * GEMM and chunk c+1's forward GEMM run as one launch over both chunks' rows,
 * sharing every W tile (results are those of separate launches, bit for bit;
 * environment variable KD_MERGE_LOGITS=0, read once per process, keeps them
 * apart).
 */
KD_API kd_status kd_topk_kl_fused_step(const void* H, const void* W, const int32_t* idx, const float* p,
                                int64_t T, int d, int V, int K, int chunk,
                                float dloss, float* loss, float* lse, float* loss_rows,
                                float* dH, float* dW, int accumulate_dW,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * The same forward and backward in one pass over the chunks, without the
 * backward's second logits GEMM: the forward GEMM's epilogue also writes the
 * chunk's exponentials e_tj = exp(z_tj - m_t,tile) (rounded to bf16, one
 * [chunk, V] buffer that the workspace already holds for G), and once lse_t is
 * known an elementwise pass forms G_tj = M_t e_tj exp(m_t,tile - lse_t) -
 * (p at the ids) in place, rounded to bf16 once.  Three chunk GEMMs instead of
 * four (6 T V d instead of 8 T V d flops); the logits still never exist for
 * more than one chunk (or one dW group of chunks), so the workspace is the
 * fused step's, flat in T.  This trades the recompute the paper's fused loss
 * performs (thorstenmeyerai.com pipeline step "Recompute backward") for one
 * extra bf16 rounding of G (relative 2^-9).  Arguments, outputs, ownership and
 * errors as kd_topk_kl_fused_step; workspace size: KD_WS_FUSED.
 */
KD_API kd_status kd_topk_kl_fused_step_norecompute(const void* H, const void* W, const int32_t* idx,
                                            const float* p, int64_t T, int d, int V, int K, int chunk,
                                            float dloss, float* loss, float* lse, float* loss_rows,
                                            float* dH, float* dW, int accumulate_dW,
                                            void* workspace, size_t ws_bytes, void* stream);

/*
 * kd_topk_kl_forward for callers that cannot allocate device memory (the
 * paper has no counterpart; this is a convenience of this library).  Same
 * inputs, outputs and results as kd_topk_kl_forward, but the workspace is a
 * scratch array owned by the library: KD_NOALLOC_SCRATCH_BYTES (32 MiB) of
 * device memory that every GPU which loads the library holds until the
 * process exits.  The call allocates nothing and calls no allocating routine.
 *   - Sizes whose forward workspace (kd_topk_kl_workspace_size with
 *     KD_WS_FORWARD) exceeds KD_NOALLOC_SCRATCH_BYTES are rejected with
 *     KD_ERR_WORKSPACE before anything is launched (for example chunk 2048
 *     fits both a 128,256- and a 201,088-word vocabulary; chunk 4096 with a
 *     201,088-word vocabulary does not).
 *   - The call waits for `stream` (below), so it cannot be captured into a
 *     CUDA graph: kd_topk_kl_forward with a caller workspace is the form to
 *     capture.
 *   - The first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with that device current.  The address is kept
 *     for the life of the process: cudaDeviceReset unloads the array with the
 *     library's device code, so do not use this entry point across a reset.
 *   - Every call on a device shares the one array and finds the previous
 *     call's contents in it; each call re-initialises what it needs.  Calls
 *     that could overlap on the GPU (other streams, other host threads) race
 *     on the array: order them on one stream.
 *   - Unlike kd_topk_kl_forward it waits for `stream` before returning and
 *     returns the device-side status (KD_OK, KD_ERR_BAD_INDEX, ...), since
 *     the caller has no workspace to query.
 */
#define KD_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
KD_API kd_status kd_topk_kl_forward_noalloc(const void* H, const void* W, const int32_t* idx, const float* p,
                                            int64_t T, int d, int V, int K, int chunk,
                                            float* loss, float* lse, float* loss_rows, void* stream);

/*
 * Teacher-cache builder: the offline step that turns teacher logits into the
 * top-K cache this loss consumes (thorstenmeyerai.com pipeline, "Infer once"
 * and "Select top-K"; aimodeling.com "First cut": the top-100 probabilities
 * of every token are cached).  For each row t of logits[T, V] (row-major,
 * device memory; bf16 if logits_bf16 != 0, else fp32; 2- or 4-byte aligned):
 *   idx[t, 0..K)  the ids of the K largest logits, largest first, equal
 *                 logits ordered by ascending id (int32, device, [T, K]);
 *   p[t, k]       exp(z_t,idx - lse_t), the teacher's softmax probability
 *                 (fp32, device, [T, K]); the row mass sum_k p <= 1;
 *   lse[t]        log sum_j exp(z_tj) (fp32, device, [T]; may be NULL).
 * Temperature 1; -0 and +0 are equal logits; -inf logits carry no
 * probability; NaN logits are not supported (their rank and the row's p and
 * lse are unspecified).  1 <= K <= min(V, 1024) (KD_ERR_INVALID_ARG /
 * KD_ERR_UNSUPPORTED otherwise).  Rows whose length in bytes is a multiple
 * of 32 (with a 32-byte aligned base) are read with 32-byte loads, those
 * whose length is a multiple of 16 (16-byte aligned base) with 16-byte loads,
 * others element by element; the results are the same either way.  Allocates nothing, waits on nothing (no device-side
 * errors are possible); asynchronous on `stream`.
 */
KD_API kd_status kd_topk_cache_build(const void* logits, int logits_bf16, int64_t T, int V, int K,
                                     int32_t* idx, float* p, float* lse, void* stream);

/*
 * dst[i] = bf16(scale * src[i]) (round to nearest even) for i < n: the fp32
 * gradients dH / dW as bf16 parameter gradients, scaled by an incoming loss
 * gradient (the paper has no counterpart; a convenience for autograd
 * wrappers).  src: device fp32, 16-byte aligned; dst: device bf16, 8-byte
 * aligned; they must not overlap.  Asynchronous on `stream`.
 */
KD_API kd_status kd_grad_to_bf16(const float* src, void* dst, int64_t n, float scale, void* stream);

/*
 * Waits for `stream`, then returns and clears the device-side status the
 * last call on this workspace recorded (KD_OK, KD_ERR_BAD_INDEX or
 * KD_ERR_TIMEOUT), or KD_ERR_CUDA if the wait itself failed.
 */
KD_API kd_status kd_topk_kl_device_status(void* workspace, void* stream);

/* Human-readable name of a status code (static storage). */
KD_API const char* kd_status_string(kd_status s);

/*
 * Plain tensor-core GEMM used by the loss, exposed for testing:
 * D[M,N] (fp32, row stride ldd elements) = A B^T with bf16 A and B.
 * a_mn == 0: A is stored [M,K] row-major (row stride lda); a_mn == 1: A is
 * stored [K,M] row-major.  Likewise b_mn for B ([N,K] or [K,N], stride ldb).
 * Strides are in elements and must give 16-byte-aligned rows.  cta_pair != 0
 * runs the two-CTA-cluster form (256-row tiles, cta_group::2 MMAs) that the
 * loss uses for chunks of 256 rows or more.  `workspace` (>= 256 bytes) holds
 * the status word read by kd_topk_kl_device_status.
 */
KD_API kd_status kd_gemm_bf16(const void* A, const void* B, float* D, int M, int N, int K,
                       int lda, int ldb, int ldd, int a_mn, int b_mn, int cta_pair,
                       void* workspace, size_t ws_bytes, void* stream);

/*
 * Test hook for failure detection: runs the GEMM pipeline with its loads
 * withheld, so the first internal wait runs out after `wait_limit_ms`; the
 * kernel then winds down (frees tensor memory, returns) and records
 * KD_ERR_TIMEOUT in the workspace (>= 256 bytes), which this call returns
 * after synchronising `stream`.  cta_pair != 0 runs it on one two-CTA
 * cluster (both CTAs wind down).  No fault, trap or hang is involved; the
 * context stays usable.
 */
KD_API kd_status kd_debug_wait_timeout(int wait_limit_ms, int cta_pair, void* workspace, size_t ws_bytes,
                                      void* stream);

/*
 * Optional per-kernel timing (CUDA events recorded on the launching stream
 * around each kernel launch).  Not thread-safe; meant for benchmarks.
 * kd_profile_read synchronises, fills per-kind totals and launch counts for
 * up to `n` kinds and returns the number of kinds (KD_PROF_KINDS).
 */
#define KD_PROF_KINDS 10
enum { KD_K_PREP = 0, KD_K_LOGITS_FWD = 1, KD_K_COMBINE = 2, KD_K_LOGITS_G = 3,
       KD_K_GEMM_DH = 4, KD_K_DH_REDUCE = 5, KD_K_GEMM_DW = 6, KD_K_OTHER = 7,
       KD_K_G_FROM_E = 8, KD_K_LOGITS_GF = 9 };
KD_API kd_status kd_profile_enable(int on);
KD_API int kd_profile_read(double* ms_total, int64_t* launches, int n, int reset);
KD_API const char* kd_profile_kind_name(int kind);

#ifdef __cplusplus
}
#endif

#endif /* KDTOPK_H */
