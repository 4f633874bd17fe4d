/*
 * afd_ffn.h -- C ABI of libafd_ffn.so: the FFN-server side of
 * Attention-FFN Disaggregation (AFD) on one GB300 (sm_103a).
 *
 * One aggregated decode batch of hidden states, gathered from M
 * attention-instance buffers, runs through one MoE layer:
 *   router (logits, top-k, softmax over the selected) -> per-expert
 *   histogram / exclusive prefix sum / stable expert-contiguous order ->
 *   pack (optionally e4m3 quantisation) -> grouped gate/up GEMM + SwiGLU ->
 *   grouped down GEMM x routing weight -> weighted combine back into the M
 *   output buffers.  (A bf16 batch of at most 8 tokens skips the pack: its
 *   gate/up GEMM reads the token rows from the source buffers.)
 *
 * Sources for the operation:
 *   - "大模型推理的内存与计算解耦：AFD 架构解析与性能验证" (FastAFD blog),
 *     section 2 benefit one (several attention instances feed one FFN server,
 *     e.g. 4 x 128 -> 512 tokens) and section 3 (the FFN service is a daemon:
 *     receive activations -> gate routing + expert compute -> return;
 *     batch shape travels as control-plane metadata, tensors as data plane).
 *   - "MoE 大规模分布式推理工程实战", section 4.1 (router: linear gate,
 *     optional bias on the logits, top-k on logits, softmax over the top-k),
 *     section 2.2 (per-destination counts, prefix-sum offsets, pack kernel)
 *     and section 1.1 (dispatch / combine of k copies per token).
 *   - "MoE系统与AFD架构概述", section 2.1 (6*B*H*I FLOPs per expert layer),
 *     section 3.3 (pre-sorting routing results, FP8 activations, fused
 *     expert kernels) and section 1 (three-buffer overlap, 3BO).
 *
 * Conventions (all entry points):
 *   - Return 0 on success, a negative AFD_E* code on failure; nothing throws.
 *     afd_ffn_last_error() gives a one-line description of the last failure
 *     on a handle.
 *   - Pointers named *_dev are device pointers (cudaMalloc'd or torch
 *     tensors on the same device); pointers named *_host are host memory.
 *     All matrices are dense row-major.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Asynchronous calls only enqueue work: they never synchronise
 *     the host, and their device-side failures show up in afd_ffn_check().
 *   - The caller owns every buffer it passes in; the library owns its copies
 *     of the weights and its workspaces, freed by afd_ffn_destroy().
 *   - One handle runs one forward at a time: calls on one handle must not
 *     overlap on the GPU.  afd_ffn_forward_pipelined (micro-batches) and
 *     afd_ffn_forward_host_async (a stream of batches) order their own
 *     concurrency on library streams.
 */
#ifndef AFD_FFN_H_
#define AFD_FFN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AFD_MAX_SOURCES 64 /* attention-instance buffers per forward */
#define AFD_MAX_MICRO 4    /* micro-batches of afd_ffn_forward_pipelined */

/* status codes */
#define AFD_OK 0
#define AFD_EINVAL -1      /* bad argument (null, size, alignment, config) */
#define AFD_ECUDA -2       /* a CUDA runtime/driver call failed */
#define AFD_ECAPACITY -3   /* batch larger than max_tokens / max_sources */
#define AFD_EUNSUPPORTED -4 /* configuration not supported by this build */
#define AFD_EDEVICE -5     /* afd_ffn_check: the device error word was set */

typedef enum {
  AFD_FP32 = 0,     /* fp32 activations, weights, output (fp32 SIMT path) */
  AFD_BF16 = 1,     /* bf16 activations, weights, output; fp32 accumulate */
  AFD_FP8_E4M3 = 2, /* bf16 activations in/out; e4m3 weights (fp32 scale per
                       128x128 block); activations quantised to e4m3 per
                       token per 128 channels inside the layer */
} afd_dtype;

/* Layer shape and capacity.
 *   H hidden size; I expert intermediate size; E routed experts; k top-k
 *   (1 <= k <= E <= 256); n_shared 0 or 1 always-on shared expert of the
 *   same shape, added with weight 1; max_sources bound on M per forward
 *   (<= AFD_MAX_SOURCES); max_tokens bound on T = sum of src_counts.
 *   bf16/fp8 need H % 256 == 0 and I % 128 == 0; fp32 needs H % 8 == 0. */
typedef struct {
  int H, I, E, k, n_shared, max_sources, max_tokens;
  afd_dtype dtype;
} afd_ffn_config;

/* Weights (device pointers, row-major; read once by afd_ffn_create, which
 * copies and re-lays them out -- the caller may free them afterwards).
 *   w_router   [H, E]  fp32 for AFD_FP32, bf16 otherwise
 *   router_bias [E] fp32, added to the logits before selection, or NULL
 *   w_gate, w_up [E, H, I]; w_down [E, I, H]   (fp32 / bf16 / e4m3 codes)
 *   s_gate, s_up [E, H/128, I/128]; s_down [E, I/128, H/128]  fp32 block
 *              scales, AFD_FP8_E4M3 only (weight = e4m3 value * scale)
 *   sh_*       shared expert, [H, I], [H, I], [I, H] (+ scales), when
 *              n_shared == 1; NULL otherwise */
typedef struct {
  const void* w_router;
  const float* router_bias;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const float* s_gate;
  const float* s_up;
  const float* s_down;
  const void* sh_gate;
  const void* sh_up;
  const void* sh_down;
  const float* sh_s_gate;
  const float* sh_s_up;
  const float* sh_s_down;
} afd_ffn_weights;

typedef struct afd_ffn* afd_ffn_t;

/* Create a layer on the current CUDA device.  Validates the config, copies
 * the weights into kernel layout (K-major for the tensor-core GEMMs) and
 * sizes one workspace for max_tokens.  Synchronous.  On failure *out is
 * NULL and the return code says why (use afd_ffn_create_error() for text). */
int afd_ffn_create(const afd_ffn_config* cfg, const afd_ffn_weights* w, afd_ffn_t* out);

/* Text of the last afd_ffn_create failure in this thread. */
const char* afd_ffn_create_error(void);

/* One forward over M source buffers (the FFN daemon's loop body in the
 * FastAFD blog, section 3).
 *   src_ptrs_dev[m]  device pointer to [src_counts_host[m], H] activations
 *                    (fp32 for AFD_FP32, bf16 otherwise), 16-byte aligned
 *   src_counts_host  host array of M row counts (>= 0; 0 allowed); this is
 *                    the control-plane batch metadata; tokens are numbered
 *                    in (m, row) order, T = sum of the counts <= max_tokens
 *   out_ptrs_dev[m]  device pointer to [src_counts_host[m], H] outputs
 *                    (fp32 for AFD_FP32, bf16 otherwise), 16-byte aligned;
 *                    must not alias the sources
 * Enqueues the whole layer on `stream`; T == 0 enqueues nothing. */
int afd_ffn_forward(afd_ffn_t h, void* stream, const void* const* src_ptrs_dev,
                    const int* src_counts_host, int M, void* const* out_ptrs_dev);

/* Same layer with the batch split into n_micro (1..AFD_MAX_MICRO) contiguous
 * token ranges (sizes differ by at most one, earlier ones larger), each run on
 * its own library stream and workspace; the ranges fork from and join back
 * to `stream` with events.  This is the one-GPU stand-in for the three-buffer
 * overlap ("MoE系统与AFD架构概述", section 1 and section 2.3).  Outputs are
 * identical to afd_ffn_forward. */
int afd_ffn_forward_pipelined(afd_ffn_t h, void* stream, int n_micro, const void* const* src_ptrs_dev,
                              const int* src_counts_host, int M, void* const* out_ptrs_dev);

/* End-to-end call with HOST buffers: copies each source to the device
 * (one cudaMemcpyAsync per buffer), runs afd_ffn_forward (n_micro == 1) or
 * afd_ffn_forward_pipelined (n_micro in [2, AFD_MAX_MICRO]), copies each
 * output back, and synchronises `stream` before returning.  Pinned host
 * memory makes the copies asynchronous DMA; pageable memory works but is
 * slower.  The staging buffers are part of the handle's workspace.  n_micro
 * outside [1, AFD_MAX_MICRO] returns AFD_EINVAL. */
int afd_ffn_forward_host(afd_ffn_t h, void* stream, int n_micro, const void* const* src_ptrs_host,
                         const int* src_counts_host, int M, void* const* out_ptrs_host);

/* HOST buffers for a stream of batches, asynchronous: the FFN daemon's loop
 * with each batch's transfers hidden under another batch's compute (the dual
 * batch overlap of the FastAFD blog, section 4).  Enqueues the host->device
 * copy of the sources, the layer (as afd_ffn_forward_host with the same
 * n_micro) and the device->host copy of the outputs on library streams
 * (copy-in, copy-out, and one compute stream per slot) and returns without
 * waiting.  Consecutive calls alternate between two device staging slots;
 * events order them on the device, so the sources of call i+1 cross the host
 * link while call i computes and call i-1's outputs return.  Single-pass calls
 * (n_micro == 1) also alternate between two compute streams and workspaces, so
 * one call's first kernels may run while the previous call's last ones finish;
 * a micro-batched call waits for the previous call.  Each call's outputs are
 * those of afd_ffn_forward_host on the same batch.  Host buffers
 * must stay valid until afd_ffn_host_wait returns, and be pinned for the
 * copies to be asynchronous.  While calls are in flight, issue no other
 * forward on this handle.  Argument errors return at once (nothing is
 * enqueued); the staging slots (2 x 2 x max_tokens x H activations) are
 * allocated on first use, and so is a second workspace. */
int afd_ffn_forward_host_async(afd_ffn_t h, int n_micro, const void* const* src_ptrs_host,
                               const int* src_counts_host, int M, void* const* out_ptrs_host);

/* Blocks until every afd_ffn_forward_host_async call so far has its outputs
 * in host memory.  Returns AFD_OK, or the first error met since the last
 * wait. */
int afd_ffn_host_wait(afd_ffn_t h);

/* Copy the routing of the last forward (for a micro-batched forward, that of
 * its first micro-batch) into caller device
 * buffers, each may be NULL to skip:
 *   topk_idx [T*k] int32, topk_w [T*k] fp32 (slot order: descending logit,
 *   ties to the lower expert id), counts [E] int32, offsets [E+1] int32
 *   (exclusive prefix sum, offsets[E] = T*k), perm_token [T*k] int32 (token of
 *   each packed row; rows of an expert in ascending token order), pos [T*k]
 *   int32 (packed row of each (token, slot)), logits [T*E] fp32.
 * Logits: for AFD_FP32 every entry is the canonical fp32 dot product (plus
 * bias).  For AFD_BF16 and AFD_FP8_E4M3 the router first estimates all
 * logits on the tensor cores, then recomputes in the canonical order every
 * expert whose estimate could reach the k-th largest once the estimate's
 * error bound is taken into account; those entries (always including the k
 * selected ones) hold the canonical value and the rest hold the estimate.
 * The selection and the weights are therefore those of the canonical logits.
 * Enqueued on `stream`; T is the token count of that forward. */
int afd_ffn_debug_routing(afd_ffn_t h, void* stream, int* topk_idx, float* topk_w, int* counts, int* offsets,
                          int* perm_token, int* pos, float* logits);

/* Copy the expert-GEMM operands of the last forward (for a micro-batched
 * forward, those of its first micro-batch) into caller device buffers, for
 * tests that check the packing and the fp8 quantisation code for code.  Each
 * pointer may be NULL to skip it.  R = T*(k + n_shared) packed rows: the
 * routed rows in expert-contiguous order (offsets / perm_token of
 * afd_ffn_debug_routing), then, with a shared expert, one row per token in
 * token order.
 *   P       [R, H] packed token rows: fp32 (AFD_FP32), bf16 (AFD_BF16) or
 *           e4m3 codes (AFD_FP8_E4M3, one byte each)
 *   P_scale [H/128, R] fp32 (AFD_FP8_E4M3 only): the scale of each row's
 *           128-channel block; code * scale is the packed value
 *   Hmid    [R, I] SwiGLU output, the down GEMM's operand: fp32, bf16 or
 *           e4m3 codes as P
 *   H_scale [I/128, R] fp32 (AFD_FP8_E4M3 only), as P_scale
 * The quantisation follows "MoE系统与AFD架构概述", section 3.3 (FP8
 * activations) with the per-token-per-128-channel rule of the fp8 layer:
 * scale = amax/448, code = e4m3(x / scale), nearest even, saturating; an
 * all-zero block has scale 1 and zero codes.  Scales are rejected (AFD_EINVAL)
 * for layers other than AFD_FP8_E4M3.  A bf16 forward of at most 8 tokens
 * writes no P (its gate/up GEMM reads the token rows from the sources), so P
 * is then rejected (AFD_EINVAL) too.  Enqueued on `stream`. */
int afd_ffn_debug_operands(afd_ffn_t h, void* stream, void* P, float* P_scale, void* Hmid, float* H_scale);

/* Synchronise `stream`, then read and clear the device error word of every
 * workspace.  Returns 0, or AFD_EDEVICE with the word's bits in
 * afd_ffn_last_error(): 1 = a kernel's bounded wait ran out (the kernel
 * abandoned its work and returned), 2 = a routing value out of range. */
int afd_ffn_check(afd_ffn_t h, void* stream);

/* Fault-path hook for tests: makes one of the device-side checks fire without
 * faulting or hanging the GPU, so that afd_ffn_check() can be seen to report it.
 *   AFD_INJECT_TIMEOUT: one block waits on a barrier that nothing arrives on,
 *     through the bounded wait every kernel uses, and gives up after `arg` SM
 *     clock cycles (clamped to [1e3, 4e9]), setting bit 1 of the error word.
 *   AFD_INJECT_RANGE: runs the routing-table kernels on a one-token batch whose
 *     first expert id is E (out of range); their range check skips it and sets
 *     bit 2.  This overwrites the routing afd_ffn_debug_routing() returns.
 * Enqueued on `stream` (AFD_INJECT_RANGE first synchronises it once, for its
 * host-side token).  The handle stays usable once afd_ffn_check() has read
 * and cleared the word.  Any other kind returns AFD_EINVAL. */
#define AFD_INJECT_TIMEOUT 1
#define AFD_INJECT_RANGE 2
int afd_ffn_debug_inject(afd_ffn_t h, void* stream, int kind, long long arg);

/* Last error text of the handle ("" if none). */
const char* afd_ffn_last_error(afd_ffn_t h);

/* Per-kernel timing (benchmark aid).  afd_ffn_profile_begin() makes every
 * following forward record CUDA events on its stream around each of its
 * AFD_NUM_KERNELS kernels (router, routing tables, pack, gate/up GEMM, down
 * GEMM, combine; a forward without a pack launch records ~0 for it).
 * afd_ffn_profile_end() synchronises the device, writes the
 * summed milliseconds per kernel over the recorded forwards into
 * ms_per_kernel[AFD_NUM_KERNELS] and their number into *n_forwards, and turns
 * recording off.  Recording adds one event per kernel launch. */
#define AFD_NUM_KERNELS 6
int afd_ffn_profile_begin(afd_ffn_t h);
int afd_ffn_profile_end(afd_ffn_t h, double* ms_per_kernel, int* n_forwards);

/* Number of kernel launches one afd_ffn_forward of T > 0 tokens enqueues
 * (it depends on T: for bf16/fp8 layers small batches route in one launch and
 * larger ones in two; the routing tables take one launch up to 2048 tokens and
 * two above; a bf16 layer packs no rows for at most 8 tokens).
 * Returns AFD_EINVAL for a NULL handle or T < 1. */
int afd_ffn_launches_per_forward(afd_ffn_t h, int T);

/* Bytes of device memory the handle holds (weights + workspaces). */
size_t afd_ffn_device_bytes(afd_ffn_t h);

/* Router top-k with no device allocation (the pages have no counterpart:
 * this serves callers that cannot allocate).  A caller that has handed all
 * of its device memory to its own pool (e.g. an attention-side server that
 * reserves HBM for its KV cache) cannot cudaMalloc, and one inside a
 * latency-critical decode loop must not make an allocation call, which can
 * block or synchronise the device.  This computes exactly the routing of
 * afd_ffn_forward (same top-k slots and weights, both from the canonical
 * fp32 logits, which this call computes for every expert)
 * without a handle and without allocating.
 *   src_ptrs_dev[m], src_counts_host[m], M  as afd_ffn_forward (16-byte
 *                    aligned rows of H activations, fp32 for AFD_FP32, bf16
 *                    for AFD_BF16 and AFD_FP8_E4M3)
 *   w_router_dev     [H, E] router weights in the same dtype, row-major,
 *                    16-byte aligned; router_bias_dev [E] fp32 or NULL
 *   topk_idx_dev     [T, k] int32 output; topk_w_dev [T, k] fp32 output
 * Limits: T <= 4096 tokens, E <= 256 with E % 8 == 0, k <= 16, H % 8 == 0,
 * M <= AFD_MAX_SOURCES.  Sizes beyond a limit return AFD_ECAPACITY; bad
 * pointers or shapes return AFD_EINVAL; a failed CUDA call AFD_ECUDA.
 * Scratch: one file-scope device array of 4 MiB + 1 KiB (logits and
 * completion tickets), held by every GPU that loads the library until the
 * process exits.  The first call on a device (with it current) looks up the
 * array's address with cudaGetSymbolAddress and keeps it for the life of the
 * process; make that first call before any stream capture begins.  After
 * cudaDeviceReset (or anything else that destroys the device's primary
 * context) that address is stale: restart the process before calling again.  All calls share the array: calls whose work
 * overlaps on the GPU race and must be serialised by the caller.  Each call
 * clears the tickets with cudaMemsetAsync on `stream`, then launches one
 * kernel; nothing is allocated or freed. */
int afd_ffn_router_noalloc(void* stream, const void* const* src_ptrs_dev, const int* src_counts_host, int M,
                           int H, int E, int k, afd_dtype dtype, const void* w_router_dev,
                           const float* router_bias_dev, int* topk_idx_dev, float* topk_w_dev);

/* Free everything the handle owns.  Synchronises the device first.
 * NULL is a no-op. */
void afd_ffn_destroy(afd_ffn_t h);

#ifdef __cplusplus
}
#endif
#endif /* AFD_FFN_H_ */
