/*
 * flce.h - C ABI of libflce, a fused linear cross-entropy (FLCE) for one NVIDIA GB300 (sm_103a).
 *
 * The operation. "Fused linear + cross-entropy" (KernelIndex operation page), summary and
 * "Semantics" table: x float[tokens, hidden], weight float[vocab, hidden], target int64[tokens],
 * loss float[1]; the LM-head projection z = x . weight^T is scored by cross-entropy against the
 * integer targets without ever materialising the tokens x vocab logits. "[example]
 * fused_linear_cross_entropy kernel" (Helion PR #1268), description: the forward computes the
 * per-token log-sum-exp (kept for the backward) and the target logits; the backward recomputes
 * the logits to form grad_input and grad_weight. "feat(FLCE): add helion version of fused linear
 * cross entropy" (Liger-Kernel PR #928), failing-test list: reductions 'sum' and 'mean'.
 *
 *   lse[t]  = ln sum_v exp(z[t, v])                     z = x . weight^T
 *   loss    = sum_t (lse[t] - z[t, target[t]])          (SUM),  divided by T for MEAN
 *   dz      = (softmax(z) - onehot(target)) * g         g = grad_loss (SUM) or grad_loss / T (MEAN)
 *   grad_x  = dz . weight                               grad_weight = dz^T . x
 *
 * Layout. Every matrix is row-major with its last index contiguous: x[T][H], weight[V][H],
 * grad_x[T][H], grad_weight[V][H]. target is int64[T]; lse is float32[T]; loss and grad_loss are
 * float32[1]. All pointers except those documented as host pointers are DEVICE pointers on the
 * current CUDA device. Matrix rows must start on 16-byte boundaries: H * element size must be a
 * multiple of 16 bytes and every base pointer 16-byte aligned, else FLCE_ERR_UNSUPPORTED.
 *
 * Types. FLCE_DTYPE_BF16: x, weight, grad_x, grad_weight are bfloat16; products are summed in
 * fp32 on the tensor cores and the softmax is evaluated in fp32. FLCE_DTYPE_F32: those four are
 * float32 and every contraction runs as three TF32 tensor-core products (hi*hi + hi*lo + lo*hi)
 * with fp32 accumulation. lse, loss and grad_loss are float32 in both cases.
 *
 * Ownership. The caller owns every buffer, including the workspace and the device status word;
 * the library allocates no device memory. Inputs are never written (KernelIndex "Semantics": inputs
 * are neither modified nor aliased): an output that overlaps an input or another output is rejected with
 * FLCE_ERR_ALIAS.
 *
 * Asynchrony. Both compute calls only enqueue work on `stream` (a cudaStream_t; NULL means the
 * legacy default stream) and return. Results are valid once the stream has been synchronised.
 * A call that fails validation (FLCE_ERR_ARG, _UNSUPPORTED, _WORKSPACE, _ALIAS) has enqueued
 * nothing; after FLCE_ERR_CUDA part of the work may have been enqueued and the outputs are
 * undefined.
 *
 * Errors. Host-detectable problems are returned as negative codes (see FLCE_ERR_*). Problems only
 * the device can see are OR-ed into the device int *status as FLCE_STATUS_* bits and never trap:
 * a target outside [0, V) makes the loss NaN; a pipeline wait that exceeds its time limit makes
 * the kernel stop early and leaves its outputs undefined. The caller zeroes *status before the
 * first call and reads it after synchronising.
 *
 * Determinism. Results are bitwise identical from run to run on the same device for the same
 * inputs: there are no floating-point atomics and every reduction has a fixed order.
 */
#ifndef FLCE_H
#define FLCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define FLCE_OK 0
#define FLCE_ERR_ARG (-1)         /* null pointer, T/H/V <= 0 or too large, unknown enum value   */
#define FLCE_ERR_UNSUPPORTED (-2) /* misaligned pointer or row stride, or not an sm_103 device   */
#define FLCE_ERR_WORKSPACE (-3)   /* workspace pointer null or smaller than the size query says  */
#define FLCE_ERR_ALIAS (-4)       /* an output overlaps an input or another output               */
#define FLCE_ERR_CUDA (-5)        /* a CUDA runtime/driver call failed (launch, tensor map, ...)  */

/* Device status bits (OR-ed into *status by the kernels). */
#define FLCE_STATUS_TARGET_RANGE 1 /* some target[t] outside [0, V): the loss is NaN             */
#define FLCE_STATUS_TIMEOUT 2      /* a pipeline wait ran out of time; outputs are undefined      */

/* Element type of x, weight, grad_x and grad_weight. */
#define FLCE_DTYPE_BF16 0
#define FLCE_DTYPE_F32 1

/* Reduction over tokens ("sum" and "mean", Liger-Kernel PR #928 failing-test list). NONE is an
 * extension the pages do not list: the per-token losses l[t] = lse[t] - z[t, target[t]] that
 * SUM and MEAN aggregate. With NONE, `loss` is float32[T] in flce_forward and `grad_loss` is
 * float32[T] (one upstream gradient per token) in flce_backward. */
#define FLCE_REDUCTION_SUM 0
#define FLCE_REDUCTION_MEAN 1
#define FLCE_REDUCTION_NONE 2

/* Bytes of device workspace flce_forward needs for this problem; 0 for invalid arguments.
 * Holds per-(vocab tile, token) partial log-sum-exp terms, the target logits and per-block loss
 * sums (plus the TF32 hi/lo operand copies for FLCE_DTYPE_F32). Pure host arithmetic. */
size_t flce_forward_workspace_size(int64_t T, int64_t H, int64_t V, int dtype);

/* Bytes of device workspace flce_backward needs; 0 for invalid arguments. Holds one bounded
 * vocab slab of dz (T x Vc, never the full T x V logits) and, for bf16, the fp32 grad_x
 * accumulator (T x H). Pure host arithmetic. */
size_t flce_backward_workspace_size(int64_t T, int64_t H, int64_t V, int dtype);

/* Vocab slab width Vc the backward uses for this problem (a multiple of 256), 0 if invalid. */
int64_t flce_backward_slab_width(int64_t T, int64_t H, int64_t V, int dtype);

/* Process-wide override of the backward vocab slab width: vc = 0 restores the automatic choice
 * (a dz slab of at most 1 GiB), otherwise vc must be a positive multiple of 256. Affects the
 * size query and the backward alike, so set it before querying the workspace size. A tuning and
 * testing knob: it trades workspace memory against the number of slab passes. Returns FLCE_OK
 * or FLCE_ERR_ARG. */
int flce_set_backward_slab_width(int64_t vc);

/*
 * Forward ("[example] fused_linear_cross_entropy kernel", Helion PR #1268, description of the
 * forward pass): computes loss[0] and the per-token log-sum-exp lse[T] that flce_backward needs.
 *   x [T][H], weight [V][H]  (dtype), target [T] int64   - inputs, device, read only
 *   loss [1] float32 ([T] for FLCE_REDUCTION_NONE), lse [T] float32 - outputs, device
 *   workspace: device, >= flce_forward_workspace_size() bytes, 256-byte aligned, scratch only
 *   status: device int, OR-ed with FLCE_STATUS_* bits
 *   stream: cudaStream_t to enqueue on
 * Returns FLCE_OK or a negative FLCE_ERR_* code.
 */
int flce_forward(const void* x, const void* weight, const int64_t* target,
                 int64_t T, int64_t H, int64_t V, int dtype, int reduction,
                 float* loss, float* lse,
                 void* workspace, size_t workspace_bytes, int* status, void* stream);

/*
 * Backward ("[example] fused_linear_cross_entropy kernel", Helion PR #1268, description of the
 * backward pass; the atomic grad_weight accumulation there is replaced by a deterministic
 * vocab-slab schedule): recomputes the logits slab by slab, forms dz in registers and writes
 *   grad_x [T][H] = dz . weight   and   grad_weight [V][H] = dz^T . x     (dtype, device)
 * x, weight, target, lse: as passed to / produced by flce_forward (device, read only)
 * grad_loss [1] float32 ([T] for FLCE_REDUCTION_NONE): device, the upstream gradient of loss
 * workspace: device, >= flce_backward_workspace_size() bytes, 256-byte aligned, scratch only
 * Returns FLCE_OK or a negative FLCE_ERR_* code.
 */
int flce_backward(const void* x, const void* weight, const int64_t* target, const float* lse,
                  int64_t T, int64_t H, int64_t V, int dtype, int reduction,
                  const float* grad_loss, void* grad_x, void* grad_weight,
                  void* workspace, size_t workspace_bytes, int* status, void* stream);

/*
 * Forward and backward in one call, when the upstream gradient is known before the forward (the
 * usual case for a training loss: grad_loss = 1). The Liger-Kernel approach discussed in "[example]
 * fused_linear_cross_entropy kernel" (Helion PR #1268) computes the gradients inside the forward
 * over token chunks; "feat(FLCE): add helion version of fused linear cross entropy"
 * (Liger-Kernel PR #928) reports its chunk-materialised backward as sound. Here the logits of a
 * chunk of tokens (at most half of all tokens and at most FLCE_TUNE_CHUNK_BYTES of bf16, 1.5 GiB
 * by default) are computed once and turned into dz in place, so the call does 6 T H V FLOPs
 * instead of the 8 T H V of flce_forward + flce_backward, at the price of the chunk buffer in
 * the workspace. grad_weight is summed over the chunks in its own output: the first chunk writes
 * it and each later chunk adds its part in fp32 and rounds the sum back to bf16, so for n chunks
 * it is rounded n times (a relative error of at most about n 2^-9 of the largest partial sums,
 * against 2^-9 for flce_backward, whose grad_weight is rounded once).
 *   Arguments as for flce_forward and flce_backward together: grad_loss (device, [1] or [T] for
 *   FLCE_REDUCTION_NONE) is read by the call; loss, lse, grad_x and grad_weight are written.
 *   bf16 with T >= 512 uses the chunked schedule; otherwise the call runs flce_forward followed
 *   by flce_backward in the same workspace (same results as calling them).
 * Returns FLCE_OK or a negative FLCE_ERR_* code.
 */
size_t flce_forward_backward_workspace_size(int64_t T, int64_t H, int64_t V, int dtype);
/* Tokens per chunk of the single-call schedule (T itself when it does not apply), 0 if invalid. */
int64_t flce_forward_backward_chunk_tokens(int64_t T, int64_t H, int64_t V, int dtype);
int flce_forward_backward(const void* x, const void* weight, const int64_t* target, int64_t T,
                          int64_t H, int64_t V, int dtype, int reduction, const float* grad_loss,
                          float* loss, float* lse, void* grad_x, void* grad_weight,
                          void* workspace, size_t workspace_bytes, int* status, void* stream);

/* Size of the device array behind flce_forward_static_scratch (64 MiB). */
#define FLCE_STATIC_SCRATCH_BYTES (64ull << 20)

/*
 * Forward without a workspace, for callers that cannot allocate device memory. (The pages
 * have no counterpart: this is an interface addition of this library.) Some callers have no
 * device allocator to hand the library a workspace from, e.g. a plain C or foreign-language
 * host program without a CUDA memory pool, or a service whose device-memory budget is fixed at
 * start-up and which may not call cudaMalloc while it runs (cudaMalloc can also synchronise the
 * device). This call computes exactly what flce_forward computes, with the same arguments minus
 * the workspace, and allocates nothing: its scratch is one file-scope device array of
 * FLCE_STATIC_SCRATCH_BYTES, part of the library's device code.
 *   - The array is reserved in a CUDA context when the library's module holding it is loaded
 *     there; with CUDA's default lazy module loading that is this call's first use in the
 *     context, and the reservation lasts until the context is destroyed or the process exits.
 *     A caller with a fixed budget should make one small call at start-up, so that this
 *     reservation (which fails with FLCE_ERR_CUDA when the device is out of memory) happens then.
 *   - Returns FLCE_ERR_WORKSPACE, enqueuing nothing, when the problem's forward scratch
 *     (flce_forward_workspace_size) exceeds FLCE_STATIC_SCRATCH_BYTES. bf16 problems up to
 *     about T = 16700 tokens fit at V = 128256. fp32 problems also hold TF32 hi/lo copies of x
 *     and weight there, 8 (T + V) H bytes plus the per-tile partials, so only small fp32
 *     problems fit (T = 1269, H = 1000, V = 10000 needs about 90 MB and is rejected).
 *   - All calls in a context share the array and it keeps the last call's contents; nothing in
 *     it has to start at zero. Calls whose GPU work overlaps (e.g. on unordered streams) race.
 *   - The array's device address is looked up (cudaGetSymbolAddress) with the caller's context
 *     current, once per CUDA context, and cached under that context's unique id, so a context
 *     created by the caller or a device's primary context created again after a reset gets its
 *     own lookup. Make the first call in each context before any stream capture.
 */
int flce_forward_static_scratch(const void* x, const void* weight, const int64_t* target,
                                int64_t T, int64_t H, int64_t V, int dtype, int reduction,
                                float* loss, float* lse, int* status, void* stream);

/* Per-launch timing of the contraction kernels, for benchmarks. While enabled (on != 0), each
 * tensor-core kernel launch is bracketed by two CUDA events recorded on its launch stream (the
 * library creates the events; it allocates no device memory). flce_timing_read() waits for the
 * recorded events and returns, per kernel role, the number of launches and their summed
 * duration in milliseconds since the previous read, then forgets them. Roles (arrays of
 * FLCE_TIMING_ROLES): 0 forward projection + online log-sum-exp, 1 backward dz, 2 backward
 * grad_weight alone and 3 backward grad_x alone (fp32 path), 4 backward grad_weight and grad_x
 * of one vocab slab in a single launch (bf16 path).
 * Process-wide and not thread-safe. Returns FLCE_OK, FLCE_ERR_ARG or FLCE_ERR_CUDA. */
#define FLCE_TIMING_ROLES 5
int flce_timing_enable(int on);
int flce_timing_read(int64_t counts[FLCE_TIMING_ROLES], double ms[FLCE_TIMING_ROLES]);

/* Process-wide tuning of the contraction kernels; results do not depend on these, only speed.
 *   FLCE_TUNE_RASTER_ROWS  rows of a contraction's M dimension per raster group: tiles sweep
 *                          the N dimension inside a group, so the group's A rows stay in L2
 *                          while the B operand streams past. Multiple of 256; default 2048.
 *   FLCE_TUNE_SM_PAIRS     which contractions run on pairs of SMs (tcgen05 cta_group::2,
 *                          one MMA stream per pair) instead of single-SM 128 x 256 tiles, for
 *                          bf16 and fp32 (3xTF32, 256 x 256 pair tiles) inputs alike: a bit
 *                          mask of FLCE_ROLE_FORWARD, FLCE_ROLE_DZ and FLCE_ROLE_GRADS; -1 (the default)
 *                          picks a measured mask when every SM of the current device can be
 *                          given a partner at once and 0 otherwise (how many pairs fit depends
 *                          on how a chip's SMs are grouped, not only on their number).
 *   FLCE_TUNE_WIDE_TILES   which of the roles on SM pairs use wide tiles: each CTA stages 256
 *                          rows of the A operand and issues two MMAs per K step (512 x 256 pair
 *                          tiles), which needs 25% less shared-memory fill per FLOP than the
 *                          128-row CTA tiles but leaves no TMEM for overlapping a tile's
 *                          epilogue with the next tile. A bit mask of FLCE_ROLE_*; -1 (the
 *                          default) picks a measured mask. Roles not on SM pairs ignore it.
 *   FLCE_TUNE_RASTER_VOCAB vocabulary rows per raster group of the forward projection and
 *                          the backward's dz contraction (whose N dimension is the vocabulary):
 *                          tiles sweep the token rows inside a group, so the group's weight rows
 *                          stay in L2 while x streams past. Multiple of 256; default 4096; 0
 *                          rasters them over token rows instead (FLCE_TUNE_RASTER_ROWS).
 *   FLCE_TUNE_SPLIT_EPILOGUE which roles on wide pair tiles drain each finished 128-row block
 *                          with two epilogue warps of 128 columns each (16 epilogue warps per
 *                          CTA) instead of one of 256: the single accumulator of a wide tile is
 *                          released sooner, at the price of fewer registers per thread. A bit mask
 *                          of FLCE_ROLE_FORWARD (forward projection and single-call chunk
 *                          logits) and FLCE_ROLE_DZ; FLCE_ROLE_GRADS is ignored. -1 restores
 *                          the default, 0 (measured no faster on GB300).
 *   FLCE_TUNE_ORDERED_DRAIN which roles on wide pair tiles (with one epilogue warp per row
 *                          block) drain a finished tile's two 128-row halves one after the
 *                          other, all epilogue warps on the first half and then on the second,
 *                          and hand each half's accumulator columns back as soon as it is read:
 *                          the next tile's MMAs on the first half then overlap the drain of the
 *                          second. A bit mask of FLCE_ROLE_*; -1 restores the default,
 *                          FLCE_ROLE_FORWARD | FLCE_ROLE_DZ (the roles with K = H).
 *   FLCE_TUNE_CHUNK_BYTES  bytes of bf16 chunk logits the single call (flce_forward_backward)
 *                          may hold at once: it takes as few token chunks of (nearly) equal size
 *                          as this budget and the half-of-all-tokens limit allow. Fewer chunks
 *                          mean fewer passes over grad_weight, more chunks less memory. 0
 *                          restores the default, 1.5 GiB. Affects the size query and the call
 *                          alike, so set it before querying the workspace size.
 * Read at each launch. Returns FLCE_OK or FLCE_ERR_ARG. */
#define FLCE_TUNE_RASTER_ROWS 1
#define FLCE_TUNE_SM_PAIRS 2
#define FLCE_TUNE_WIDE_TILES 3
#define FLCE_TUNE_RASTER_VOCAB 4
#define FLCE_TUNE_SPLIT_EPILOGUE 5
#define FLCE_TUNE_CHUNK_BYTES 6
#define FLCE_TUNE_ORDERED_DRAIN 7
#define FLCE_ROLE_FORWARD 1
#define FLCE_ROLE_DZ 2
#define FLCE_ROLE_GRADS 4
int flce_set_tuning(int key, int64_t value);

/* The value a tuning key takes on the current device (automatic choices resolved), in *value.
 * Returns FLCE_OK, FLCE_ERR_ARG or FLCE_ERR_CUDA. */
int flce_get_tuning(int key, int64_t* value);

/* Testing aid for the failure path; never needed in normal use. The next bf16 or fp32
 * contraction launch withholds, in its first CTA (or first CTA pair) only, the signal that its
 * first accumulator tile is ready: that CTA's (that pair's) epilogue wait then runs out of time
 * (about 2 s) and the launch ends early with FLCE_STATUS_TIMEOUT OR-ed into the status word and
 * undefined outputs, instead of hanging. One-shot: later launches are unaffected and the device
 * stays usable. Returns FLCE_OK. */
int flce_test_withhold_signal(void);

/* Static, human-readable name of a return code. Never NULL. */
const char* flce_strerror(int code);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int flce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H */
