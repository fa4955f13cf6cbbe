/*
 * fa.h -- C ABI of the GB300 (sm_103a) tiled exact attention library.
 *
 * The operation is exact softmax attention for training, computed the way the
 * FlashAttention method does it:
 *
 *   forward  ("What Ordinary Autograd Saves: Tiling the Forward Pass Is Only
 *            Half the Algorithm", section "The implementation under test"):
 *            an online-softmax pass over key/value tiles that never forms the
 *            Tq x Tk score matrix and returns O and the per-row logsumexp L.
 *   backward ("What Ordinary Autograd Saves", section "Why this is
 *            FlashAttention's second idea"; "Backward Pass Implementation",
 *            section "The Recomputation Strategy"): keeps only O and L from the
 *            forward and rebuilds every score/probability tile on chip from Q,
 *            K and L, with D = rowsum(dO * O), dS = P * (dP - D),
 *            dV += P^T dO, dK += dS^T Q * scale, dQ += dS K * scale.
 *
 * Tensors (all row-major, contiguous, device memory, 16-byte aligned):
 *   Q, dQ   bf16 [B, Hq,  Tq, d]
 *   K, dK   bf16 [B, Hkv, Tk, d]
 *   V, dV   bf16 [B, Hkv, Tk, dv]
 *   O, dO   bf16 [B, Hq,  Tq, dv]
 *   L       fp32 [B, Hq,  Tq]   natural-log logsumexp of the scaled scores
 * Query head h reads key/value head h / (Hq / Hkv) (grouped-query attention in
 * the repeat_interleave order of "The Autograd Memory Trap", section "The GQA
 * Expansion Question"); Hq must be a multiple of Hkv.
 *
 * Masking: key j is visible to query i iff j < Tk and, when causal, also
 * j <= i + (Tk - Tq) (bottom-right alignment, the same as top-left when
 * Tq == Tk).  A causal sliding window of W >= 1 keys (the local-attention
 * layers of "The Autograd Memory Trap", section "Assumptions and
 * Uncertainties", item 3, which attend to a bounded number of keys) further
 * requires j > i + (Tk - Tq) - W: each row sees at most its last W keys.
 * A query row that sees no key gets O = 0, L = -inf, dQ = 0 and contributes
 * nothing to dK, dV.
 *
 * Supported: d and dv each in {64, 128} (dv may differ from d).  Any B, Hq, Hkv, Tq, Tk >= 0 (ragged tails
 * are handled; a zero-sized problem is a no-op; Tk == 0 yields O = 0 and
 * L = -inf), up to size limits: Tq <= 65535 * 256, B * Hkv * ceil(Tk / 128)
 * < 2^31, B * Hq < 2^31 (beyond them FA_ERR_UNSUPPORTED).
 *
 * Ownership and execution: the caller allocates and frees every buffer,
 * including the backward workspace.  The library never allocates or frees
 * device memory and never synchronises the stream (fa_last_device_status
 * excepted); all work is enqueued on `stream` (a cudaStream_t, NULL for the
 * legacy default stream).  Inputs are read-only; outputs are fully overwritten.
 *
 * Errors: a bad argument returns FA_ERR_INVALID_ARG and an unsupported shape
 * FA_ERR_UNSUPPORTED, before anything is enqueued.  A CUDA launch or
 * tensor-map error returns FA_ERR_CUDA.  Every on-chip wait of the kernels is
 * bounded in time; if one gives up, the kernel stops, leaves its outputs
 * undefined and records FA_ERR_TIMEOUT in a device status word that
 * fa_last_device_status reports.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_CUDA = 3,
  FA_ERR_TIMEOUT = 4,
  FA_ERR_SCRATCH_TOO_SMALL = 5
} fa_status;

typedef struct {
  int B, Hq, Hkv, Tq, Tk, d, dv;
  int causal; /* 0 or 1 */
  float scale; /* multiplies Q K^T; <= 0 selects 1/sqrt(d) */
  int window;  /* causal sliding window in keys; 0 = none; > 0 needs causal == 1 */
} fa_dims;

/* Forward pass: O = softmax(scale * Q K^T + mask) V, L = logsumexp rows.
 * Only O and L need to be kept for the backward pass. */
FA_API fa_status fa_forward(const fa_dims* dims, const void* Q, const void* K, const void* V, void* O, float* L,
                     void* stream);

/* Size in bytes of the scratch buffer for fa_backward's fastest schedule:
 * an fp32 dQ accumulator [B, Hq, ceil(Tq/128)*128, d] plus two fp32 row
 * vectors (D and log2-scaled L) of B*Hq*ceil(Tq/128)*128 entries, plus
 * alignment; without a causal mask also room for the partial dK / dV of up
 * to min(B*Hkv*ceil(Tk/128), 128) key tiles whose work may be split in two
 * (fp32, 2 x 128 x (d + dv) each) and a 4-byte counter per such tile.
 * Returns 0 for invalid dims. */
FA_API size_t fa_backward_workspace_bytes(const fa_dims* dims);

/* The least workspace fa_backward accepts: the dQ accumulator and the two
 * row vectors alone.  With less than fa_backward_workspace_bytes(dims) the
 * backward runs every key tile as one work item (same results, a slower
 * last round without a causal mask).  Equal to fa_backward_workspace_bytes
 * with a causal mask.  Returns 0 for invalid dims. */
FA_API size_t fa_backward_workspace_min_bytes(const fa_dims* dims);

/* Backward pass from O, L of fa_forward (same dims) and the upstream gradient
 * dO.  Writes dQ, dK, dV.  `workspace` must hold at least
 * fa_backward_workspace_min_bytes(dims) bytes (fa_backward_workspace_bytes
 * for the fastest schedule), 256-byte aligned; its contents on entry are
 * ignored. */
FA_API fa_status fa_backward(const fa_dims* dims, const void* Q, const void* K, const void* V, const void* O,
                      const void* dO, const float* L, void* dQ, void* dK, void* dV, void* workspace,
                      size_t workspace_bytes, void* stream);

/* The backward in separately launchable stages, for callers that interleave
 * other work or time the stages: bit 0 = preprocess (D = rowsum(dO * O), L in
 * log2 units, zero the dQ accumulator and the split-tile counters in
 * `workspace`), bit 1 = the main
 * recompute kernel (dK, dV, dQ accumulation), bit 2 = dQ cast.  Stages must run
 * in order on the same workspace; fa_backward is fa_backward_stages(..., 7). */
enum { FA_BWD_PRE = 1, FA_BWD_MAIN = 2, FA_BWD_CAST = 4, FA_BWD_ALL = 7 };
FA_API fa_status fa_backward_stages(const fa_dims* dims, const void* Q, const void* K, const void* V, const void* O,
                                    const void* dO, const float* L, void* dQ, void* dK, void* dV, void* workspace,
                                    size_t workspace_bytes, int stages, void* stream);

/* Backward pass for callers that cannot allocate device memory, such as code
 * running inside a host framework that passes it only its inputs and outputs
 * and owns every other byte of device memory, or a latency-critical loop that
 * must not call cudaMalloc.  Same arguments and results as fa_backward, but
 * no workspace: the scratch comes from a fixed array of
 * FA_NOALLOC_SCRATCH_BYTES that the library keeps in device memory on every
 * GPU that loads it, for the life of the process.  This entry point has no
 * counterpart on the pages; it is an interface convenience.
 *  - A problem whose fa_backward_workspace_min_bytes exceeds
 *    FA_NOALLOC_SCRATCH_BYTES is rejected with FA_ERR_SCRATCH_TOO_SMALL
 *    before anything is enqueued (use fa_backward for it); one that fits
 *    the minimum but not fa_backward_workspace_bytes runs unsplit.
 *  - Nothing is allocated or freed.  The first call on each device looks up
 *    the array's device address with that device current and keeps it for
 *    the life of the process; make that first call before any stream capture
 *    on the device.  Resetting the device (cudaDeviceReset) after that first
 *    call is not supported: the kept address would point into the destroyed
 *    context.  (The device status word behind fa_last_device_status is kept
 *    the same way.)
 *  - All calls on a device share the array.  Calls that may overlap on the
 *    GPU race on it; the caller must order them (e.g. one stream).  Stale
 *    contents from an earlier call are harmless: every part of the scratch the
 *    backward reads is rewritten (the dQ accumulator is zeroed) first. */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)
FA_API fa_status fa_backward_noalloc(const fa_dims* dims, const void* Q, const void* K, const void* V,
                                     const void* O, const void* dO, const float* L, void* dQ, void* dK, void* dV,
                                     void* stream);

/* Static description of a status code. */
FA_API const char* fa_status_string(fa_status s);

/* Synchronises `stream`, then reports (and clears) the device status word:
 * FA_ERR_TIMEOUT if a kernel gave up waiting since the last call, FA_ERR_CUDA
 * if the stream holds an asynchronous CUDA error, FA_OK otherwise. */
FA_API fa_status fa_last_device_status(void* stream);

/* Number of kernel launches the last fa_forward / fa_backward call on this
 * host thread enqueued (for launch accounting). */
FA_API int fa_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
