/*
 * lema.h -- C ABI of liblema.so: the fused optimizer step of selective full
 * fine-tuning on one GB300 (sm_103a).
 *
 * The method (page "LEMA: Layer-wise Efficient Memory Abstraction"):
 *   - section "Selective Full Fine-Tuning": real weights are trained, the
 *     optimizer states and the gradient accumulators are kept in fp32, AdamW runs
 *     layer by layer, and checkpoints store the fp32 difference between the
 *     updated and the original weights;
 *   - section "Quick Start": the optimizer is torch.optim.AdamW (decoupled weight
 *     decay, bias-corrected first and second moments, eps outside the square root);
 *   - sections "Features" and "TensorStore: Unified Streaming Core": optimizer
 *     states and accumulators either stay in VRAM or live in (pinned) RAM and are
 *     streamed through a slot pool, each stream with its own residency policy.
 *
 * Conventions for every entry point:
 *   - Pointers are plain addresses.  "device" = CUDA device memory of the current
 *     device; "pinned host" = page-locked host memory (cudaHostAlloc or
 *     cudaHostRegister, e.g. torch's pin_memory()).  bf16 values are passed as
 *     uint16_t bit patterns; fp32 as float.  Every array is a contiguous 1-D view
 *     of a tensor with n elements.
 *   - Every base address must be 16-byte aligned (LEMA_ERR_ALIGN otherwise); n may
 *     be any value >= 0 (ragged lengths are handled inside the kernels).
 *   - Ownership: the caller owns every buffer it passes and must keep it alive and
 *     untouched until the enqueued work completes.  The library owns only its
 *     per-device descriptor ring and cached chunk maps and, inside a lema_pool,
 *     the slot memory, streams and events.
 *   - Streams: `cuda_stream` is a cudaStream_t (NULL = the legacy default stream).
 *     Calls enqueue work and return; they do not synchronize the host.
 *     lema_accum_grad and lema_adamw_step launch their kernels with programmatic
 *     dependent launch: the kernel's blocks may be scheduled while the kernel
 *     before it on the stream finishes, and wait for it to complete (its memory
 *     visible) before they touch any buffer, so stream order holds as for a plain
 *     launch; back-to-back small calls lose less time between kernels.
 *   - Errors: every call returns a lema_status.  Arguments are validated before
 *     anything is enqueued; on a validation failure nothing is launched or copied.
 *     lema_last_error() gives a message for the calling thread's last failure.
 *     No call aborts, throws or traps.
 */
#ifndef LEMA_H
#define LEMA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lema_status {
    LEMA_OK = 0,
    LEMA_ERR_ARG = -1,     /* bad argument (null pointer, negative size, domain, overlap) */
    LEMA_ERR_ALIGN = -2,   /* a base address is not 16-byte aligned                     */
    LEMA_ERR_CUDA = -3,    /* a CUDA call failed; the CUDA message is kept              */
    LEMA_ERR_OOM = -4,     /* device or host allocation failed                          */
    LEMA_ERR_TIMEOUT = -5, /* a bounded host wait ran out before the work completed     */
    LEMA_ERR_STATE = -6,   /* object in the wrong state (e.g. pool used on another GPU) */
    LEMA_ERR_IO = -7       /* a file read or write failed or came up short              */
} lema_status;

/* One trainable tensor of n elements for the optimizer step.
 *   master      fp32, read (and written when master_out is NULL): master weights
 *   m, v        fp32, read (and written when m_out/v_out are NULL): AdamW moments
 *   acc         fp32, read: sum of the K micro-batch grads of this step; an in-place
 *               step then resets it to +0.0, an out-of-place step leaves it untouched
 *   delta       fp32, written: master' - (fp32)orig, the cumulative change since the
 *               original weight (section "Selective Full Fine-Tuning", checkpoints)
 *   orig_bf16   bf16, read: the original weight
 *   w_bf16      bf16, written: round-to-nearest-even of master' (the working weight)
 *   master_out, m_out, v_out
 *               NULL (all three) = update in place; otherwise (all three non-NULL)
 *               separate outputs, and every input is left unchanged.
 *   grad_bf16   optional (NULL = none), bf16, read: the last micro-batch's grad,
 *               folded into the step.  The step then uses acc + (fp32)grad_bf16 --
 *               the same single fp32 add lema_accum_grad performs -- as the sum of
 *               the K grads, without writing it back; acc holds the sum of the
 *               first K-1 micro-steps, or acc may be NULL when K == 1.
 *   flags       LEMA_STEP_KEEP_ACC: an in-place step leaves acc as it is instead
 *               of resetting it to +0.0 (for callers whose next step starts with a
 *               LEMA_GRAD_FIRST accumulate, which never reads the old contents).
 * In lema_adamw_step every pointer is device memory.  In lema_stream_layers with
 * LEMA_STREAMED the same fields are pinned-host addresses (see there); grad_bf16
 * and flags are ignored there (the pool folds the last grad in itself). */
typedef struct lema_tensor {
    float* master;
    float* m;
    float* v;
    float* acc;
    float* delta;
    const uint16_t* orig_bf16;
    uint16_t* w_bf16;
    float* master_out;
    float* m_out;
    float* v_out;
    const uint16_t* grad_bf16;
    int64_t n;
    int32_t flags;
    int32_t reserved;            /* must be 0 */
} lema_tensor;

enum { LEMA_STEP_KEEP_ACC = 1 };

/* One micro-batch gradient to accumulate: acc[i] = acc[i] + (fp32)grad_bf16[i].
 * flags LEMA_GRAD_FIRST: the first micro-step of a step, acc[i] = +0.0 + (fp32)g[i]
 * (the same value as adding to a reset accumulator) without reading acc. */
typedef struct lema_grad {
    float* acc;                  /* device, fp32, n elements, written (and read)  */
    const uint16_t* grad_bf16;   /* device, bf16, n elements, read                */
    int64_t n;
    int32_t flags;
    int32_t reserved;            /* must be 0 */
} lema_grad;

enum { LEMA_GRAD_FIRST = 1 };

/* Gradient accumulation for `count` tensors in one multi-tensor launch (descriptor
 * tables as in lema_adamw_step).
 * Section "Selective Full Fine-Tuning": gradient accumulation is fp32.
 * Each element: acc = acc + (fp32)g, one fp32 add rounded to nearest even.
 * count == 0 is a no-op.  Tensors with n == 0 may have NULL pointers.
 * The accumulators of different entries must not overlap.
 * Returns LEMA_OK, LEMA_ERR_ARG, LEMA_ERR_ALIGN or LEMA_ERR_CUDA. */
int lema_accum_grad(const lema_grad* grads, int32_t count, void* cuda_stream);

/* One bias-corrected AdamW step with decoupled weight decay for `count` tensors in
 * one multi-tensor launch.
 * Sections "Selective Full Fine-Tuning" (fp32 master/m/v, per-layer AdamW, fp32
 * delta) and "Quick Start" (torch.optim.AdamW).
 *
 * step        1-based step counter t, shared by every tensor of the call (>= 1)
 * lr, beta1, beta2, eps, weight_decay
 *             fp64 hyperparameters: 0 <= beta < 1, eps > 0, lr >= 0, wd >= 0 and
 *             lr*wd < 1
 * accum_steps K >= 1: acc holds the sum of K micro-batch grads; the step uses acc/K
 *
 * Per call, on the host in fp64, rounded once to fp32: decay = 1 - lr*wd,
 * beta1, 1-beta1, beta2, 1-beta2, step_size = lr/(1-beta1^t), sqrt(1-beta2^t), eps
 * (beta^t is the product of t factors of beta taken one at a time).
 * Per element, each operation an IEEE fp32 operation rounded to nearest even, no
 * fused multiply-add, subnormals kept:
 *   g = acc/K;  w = master*decay;  m = beta1*m + (1-beta1)*g;
 *   v = beta2*v + (1-beta2)*(g*g);  den = sqrt(v)/sqrt(1-beta2^t) + eps;
 *   w = w - step_size*(m/den);  delta = w - orig;  w_bf16 = bf16_rne(w)
 * (a NaN weight gives the bf16 pattern 0x7FC0).
 *
 * With grad_bf16 set, g = (acc + grad)/K with that one extra fp32 add first.
 *
 * Outputs (master/m/v when in place, delta, w_bf16, acc when it is reset) must not
 * overlap any other buffer of the call, except that an in-place field is the same
 * buffer as its input.  A call of at most 64 tensors passes its descriptor table to
 * the kernel as a launch parameter; a larger one stages it through the library's
 * per-device ring buffer (a small copy kernel on `cuda_stream` before the step).
 * The chunk map of a list of sizes is built and uploaded once, on the first call
 * that uses it, and kept.  The ring and the chunk maps are allocated on first use.
 * Returns LEMA_OK, LEMA_ERR_ARG, LEMA_ERR_ALIGN, LEMA_ERR_OOM or LEMA_ERR_CUDA. */
int lema_adamw_step(const lema_tensor* tensors, int32_t count, int64_t step,
                    double lr, double beta1, double beta2, double eps,
                    double weight_decay, int32_t accum_steps, void* cuda_stream);

/* ------------------------------------------------------------------------------
 * 8-bit optimizer states (section "Quantization": opt_state_bits = 8 and
 * grad_acc_bits = 8 keep the Adam moments and the gradient accumulators as 8-bit
 * integers, expanded to full precision only within each layer's AdamW update).  The pages do not
 * fix the format; this library's:
 *   - blocks of 256 consecutive elements of a tensor (the last one ragged), one
 *     fp32 scale per block, n_blocks = ceil(n / 256);
 *   - m and the accumulator: int8 codes in [-127, 127]; scale = absmax / 127;
 *     code = rint(x * (127 / absmax)) (nearest even; all 0 when the scale is 0);
 *     value = code * scale;
 *   - v is stored as its square root r: uint8 codes; scale = rmax / 255;
 *     code = min(ceil(r * (255 / rmax)), 255), rounded up so that the stored second
 *     moment does not understate the true one; v = (code * scale)^2;
 *   - a block whose largest magnitude is below 2^-100 is stored as zero (scale 0).
 * Master weights, delta and the bf16 weights stay as in lema_tensor.  States must
 * be finite (a NaN has no 8-bit code).
 * ---------------------------------------------------------------------------- */

/* One trainable tensor with 8-bit states (all device memory, 16-byte aligned).
 *   m_q, m_scale      int8 codes (n) and fp32 block scales (n_blocks), read + written
 *   r_q, r_scale      uint8 codes of sqrt(v) and their scales, read + written
 *   acc_q, acc_scale  the accumulated grads (int8 + scales), read; reset to zero
 *                     codes and scales by an in-place step unless LEMA_STEP_KEEP_ACC;
 *                     may both be NULL when grad_bf16 is set and K == 1
 *   grad_bf16         optional last micro-batch grad, folded in as in lema_tensor
 *   master_out, m_q_out, m_scale_out, r_q_out, r_scale_out
 *                     all NULL (in place) or all set (out of place, inputs untouched)
 */
typedef struct lema_tensor_q8 {
    float* master;
    int8_t* m_q;
    float* m_scale;
    uint8_t* r_q;
    float* r_scale;
    int8_t* acc_q;
    float* acc_scale;
    float* delta;
    const uint16_t* orig_bf16;
    uint16_t* w_bf16;
    const uint16_t* grad_bf16;
    float* master_out;
    int8_t* m_q_out;
    float* m_scale_out;
    uint8_t* r_q_out;
    float* r_scale_out;
    int64_t n;
    int32_t flags;               /* LEMA_STEP_KEEP_ACC */
    int32_t reserved;            /* must be 0 */
} lema_tensor_q8;

/* One micro-batch gradient into an 8-bit accumulator: per block, decode, add the
 * fp32 grads, encode again (LEMA_GRAD_FIRST: start from +0 without reading). */
typedef struct lema_grad_q8 {
    int8_t* acc_q;
    float* acc_scale;
    const uint16_t* grad_bf16;
    int64_t n;
    int32_t flags;               /* LEMA_GRAD_FIRST */
    int32_t reserved;            /* must be 0 */
} lema_grad_q8;

/* Gradient accumulation into 8-bit accumulators, one multi-tensor launch.
 * Returns LEMA_OK, LEMA_ERR_ARG, LEMA_ERR_ALIGN or LEMA_ERR_CUDA. */
int lema_accum_grad_q8(const lema_grad_q8* grads, int32_t count, void* cuda_stream);

/* The AdamW step of lema_adamw_step on 8-bit states: per element, decode m, v
 * (from its root) and the accumulated grads, run the same fp32 update (same
 * operation order), write master, delta and w_bf16; per block, encode m and
 * sqrt(v) again.  Same hyperparameter rules and errors as lema_adamw_step.
 *
 * The kernel stages its inputs through shared memory and waits for those copies
 * with a bounded wait (about a second).  If a wait runs out, the kernel stops early
 * and the groups it had not finished keep their old outputs.  That is reported the
 * way CUDA reports errors of asynchronous work: the next lema_adamw_step_q8 call on
 * the same device that starts after the kernel has finished returns
 * LEMA_ERR_TIMEOUT and launches nothing (a call after that runs normally), and
 * lema_kernel_wait_timeouts counts the event.  Expected never to happen. */
int lema_adamw_step_q8(const lema_tensor_q8* tensors, int32_t count, int64_t step,
                       double lr, double beta1, double beta2, double eps,
                       double weight_decay, int32_t accum_steps, void* cuda_stream);

/* ------------------------------------------------------------------------------
 * Serving from a checkpoint (section "Selective Full Fine-Tuning", its paragraph on
 * checkpoints and serving: a servable model is the base model plus the saved fp32
 * delta).
 * ---------------------------------------------------------------------------- */

/* One tensor to merge (device memory, 16-byte aligned, n elements):
 * merged_bf16[i] = bf16_rne((fp32)base_bf16[i] + delta[i]), one fp32 add.
 * merged_bf16 may be base_bf16 (in place); otherwise they must not overlap. */
typedef struct lema_merge {
    const uint16_t* base_bf16;
    const float* delta;
    uint16_t* merged_bf16;
    int64_t n;
} lema_merge;

/* Merge saved deltas into base weights, one multi-tensor launch.
 * Returns LEMA_OK, LEMA_ERR_ARG, LEMA_ERR_ALIGN or LEMA_ERR_CUDA. */
int lema_merge_delta(const lema_merge* items, int32_t count, void* cuda_stream);

/* lema_adamw_step without any allocation.  The paper has no counterpart to this
 * entry point; it exists for callers that cannot let a library allocate: a
 * framework that hands all free HBM to its own caching allocator at start-up (a
 * library cudaMalloc then fails or fragments that pool), or a loop whose streams
 * must keep overlapping (cudaMalloc and cudaFree can synchronize the device).
 *
 * Same arguments, checks, arithmetic and results as lema_adamw_step.  The
 * descriptor table and chunk map live in a fixed file-scope device array (about
 * 1.1 MiB, held by every GPU that loads the library until the process exits), so
 * one call takes at most 1024 tensors and 536,870,912 elements (65536 chunks of
 * 8192); beyond that it returns LEMA_ERR_ARG with a message and launches nothing.
 * It calls no cudaMalloc, cudaFree or other allocating routine, on the device or
 * the host heap.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any stream
 * capture.  Each call rewrites the part of the array it uses (nothing has to start
 * at zero) and the array keeps the last call's contents.  Calls share the array:
 * two calls whose work overlaps on the GPU (different streams with no ordering
 * between them) race; calls on one stream are ordered.  The table is staged from a
 * static host buffer and copied on cuda_stream, so a call may wait for work already
 * on that stream before it returns.
 * Returns LEMA_OK, LEMA_ERR_ARG, LEMA_ERR_ALIGN, LEMA_ERR_STATE or LEMA_ERR_CUDA. */
int lema_adamw_step_noalloc(const lema_tensor* tensors, int32_t count, int64_t step,
                            double lr, double beta1, double beta2, double eps,
                            double weight_decay, int32_t accum_steps, void* cuda_stream);

/* ------------------------------------------------------------------------------
 * Streamed residency: a slot pool in VRAM through which layers whose fp32 states
 * live in pinned host RAM pass one at a time (sections "Features": pinned RAM to
 * VRAM with asynchronous prefetch, module pool; "TensorStore: Unified Streaming
 * Core": slot-pool address space, residency per stream).
 * ---------------------------------------------------------------------------- */

typedef struct lema_pool lema_pool;

typedef struct lema_adamw_hparams {
    double lr, beta1, beta2, eps, weight_decay;
    int32_t accum_steps;                /* K */
} lema_adamw_hparams;

/* One streaming unit (a decoder layer, the embedding, the LM head, ...).
 *   tensors  host array of `count` lema_tensor
 *   grads    host array of `count` pointers to this micro-step's bf16 grads, each
 *            either memory of the pool's device or pinned host memory (then copied
 *            to the slot)
 *   flags    LEMA_UNIT_PACKED: the unit's host states are laid out like a slot.  For
 *            every state field (master, m, v, acc, delta, orig_bf16, w_bf16, and the
 *            *_out fields when set), tensor j's pointer is the first non-empty
 *            tensor's pointer plus o_j - o_first elements, o_j = sum over i < j of
 *            n_i rounded up to a multiple of 64,
 *            and the gaps between tensors belong to the caller's same allocation
 *            (tensors with n == 0 are skipped: they carry no data).  Accumulators
 *            kept in device memory (below) are exempt from the rule.
 *            The pool then moves each field of the unit with one copy (gaps
 *            included) instead of one per tensor.  Checked: a unit flagged packed
 *            whose pointers do not follow the rule is rejected (LEMA_ERR_ARG). */
typedef struct lema_layer {
    const lema_tensor* tensors;
    const uint16_t* const* grads;
    int32_t count;
    int32_t flags;
} lema_layer;

enum { LEMA_UNIT_PACKED = 1 };

enum { LEMA_RESIDENT = 0, LEMA_STREAMED = 1 };

/* Create a pool of n_slots (>= 2) VRAM slots on the current device, each able to
 * hold one unit of up to slot_params elements (each tensor of a unit is padded to a
 * multiple of 64 elements).  A slot holds an input half (fp32 master, m, v, acc;
 * bf16 orig and grad) and an output half (fp32 master', m', v', delta; bf16 w): 38
 * bytes per element.  The pool owns three streams (host-to-device, compute,
 * device-to-host) and its events.  Returns LEMA_OK, LEMA_ERR_ARG, LEMA_ERR_OOM or
 * LEMA_ERR_CUDA; *out is NULL on failure. */
int lema_pool_create(int32_t n_slots, int64_t slot_params, lema_pool** out);

/* Micro-step `micro_step` (k, 1-based, 1 <= k <= K) of optimizer step `step` for
 * n_layers units.
 *
 * LEMA_STREAMED: every lema_tensor field is pinned host memory, updated in place
 * (or written to the *_out fields).  For each unit L, on the pool's streams:
 *   host-to-device: unit L's inputs into a free slot (acc when k >= 2; pinned-host
 *                   grads; master, m, v and orig when k == K);
 *   compute:        acc' = acc + g (from +0.0 when k == 1); when k == K also the
 *                   AdamW step above, out of place from the slot's input half into
 *                   its output half;
 *   device-to-host: acc' to the host acc (k < K), or master', m', v', delta and
 *                   w_bf16 to the host (k == K).  The host acc is staging for the
 *                   partial sums: after k == K it still holds the sum of micro-steps
 *                   1..K-1 (never written when K == 1), and the next step's k == 1
 *                   starts again from +0.0 without reading it.
 * Accumulator residency (page "LEMA: Layer-wise Efficient Memory Abstraction",
 * section "TensorStore: Unified Streaming Core": weights, optimizer states and
 * gradient accumulators each with a residency policy of their own): a unit's acc
 * may instead be memory of the pool's device (16-byte aligned, all of the unit's
 * non-empty tensors alike; a unit mixing the two is rejected with LEMA_ERR_ARG).  It then
 * stays in HBM: the compute stage reads and updates it in place (k < K) or reads it
 * (k == K), and no acc copy crosses the host link, which leaves master, m, v, orig
 * in and master', m', v', delta, w_bf16 out at k == K, and nothing but host grads
 * at k < K.  A unit whose grads are device memory as well moves nothing at k < K
 * and takes no slot: its accumulate runs on the compute stream in call order, and
 * the copies of the next calls (the states the step at k == K loads) need not wait
 * for it.  Its contents follow the same rule as the host acc (after k == K the sum
 * of micro-steps 1..K-1).  It is written on the pool's compute stream: order the
 * caller's own accesses with lema_pool_wait_stream or lema_pool_sync.
 * With two or more slots the three stages of consecutive units overlap: while unit
 * L is computed, unit L+1 is copied in and unit L-1 copied out; a packed unit also
 * moves in slices (lema_pool_slices), so its own three stages overlap too.  Results
 * are identical, bit for bit, to lema_accum_grad + lema_adamw_step on the same
 * values.
 *
 * LEMA_RESIDENT: every field is device memory and `pool` may be NULL; the call is
 * lema_accum_grad (and, when k == K, an in-place lema_adamw_step) on cuda_stream.
 *
 * cuda_stream: the pool's streams wait for work already enqueued on it (e.g. the
 * backward pass that produced the grads) before they start.  Completion is not
 * joined back; use lema_pool_sync or lema_pool_wait_stream.
 * Every unit must fit a slot (LEMA_ERR_ARG otherwise, nothing enqueued).  On a CUDA
 * failure part of the call may have run: the host states of that call are then
 * unspecified, the pool stays usable.
 * Returns LEMA_OK, LEMA_ERR_ARG, LEMA_ERR_ALIGN, LEMA_ERR_STATE or LEMA_ERR_CUDA. */
int lema_stream_layers(lema_pool* pool, const lema_layer* layers, int32_t n_layers,
                       int32_t residency, int32_t micro_step,
                       const lema_adamw_hparams* hparams, int64_t step,
                       void* cuda_stream);

/* One streaming unit with 8-bit states: as lema_layer, with lema_tensor_q8
 * descriptors whose fields are pinned host memory.  LEMA_UNIT_PACKED: the rule of
 * lema_layer with tensors at 1024-element offsets (o_j = sum over i < j of n_i
 * rounded up to a multiple of 1024) and each block-scale field at o_j / 256. */
typedef struct lema_layer_q8 {
    const lema_tensor_q8* tensors;
    const uint16_t* const* grads;
    int32_t count;
    int32_t flags;
} lema_layer_q8;

/* lema_stream_layers (LEMA_STREAMED) for 8-bit states, through the same pool.
 * Micro-steps k < K move the 8-bit accumulator (codes + scales) in and out; k == K
 * moves master, m and sqrt(v) codes + scales and orig in, runs the 8-bit step with
 * the last grad folded in, and moves master, the codes + scales, delta and w_bf16
 * out (the host accumulator keeps micro-steps 1..K-1, as in lema_stream_layers).
 * As there, a unit's accumulators (acc_q and acc_scale of all its non-empty
 * tensors) may be device memory instead: they then stay in HBM and are updated in
 * place, and no accumulator copy crosses the host link.
 * Results equal lema_accum_grad_q8 + lema_adamw_step_q8 (last grad folded in) on
 * the same values, bit for bit.  Each unit must fit a slot with its tensors at
 * 1024-element offsets.  Errors as lema_stream_layers. */
int lema_stream_layers_q8(lema_pool* pool, const lema_layer_q8* layers, int32_t n_layers,
                          int32_t micro_step, const lema_adamw_hparams* hparams,
                          int64_t step, void* cuda_stream);

/* ----------------------------------------------------------------- disk tier --
 *
 * Page "LEMA: Layer-wise Efficient Memory Abstraction", section "Features" (three
 * tiers, disk, page-locked host memory and GPU memory, filled ahead of use; the
 * fp32 optimizer state kept in host memory like the weights, a memory-mapped file
 * standing in when host memory runs short) and section "Selective Full
 * Fine-Tuning" (host memory holds the optimizer state and the accumulated grads,
 * a file can back them).  Reading taken here: the optimizer
 * states (master, m, v), the original and working weights and the delta live in
 * one file; the gradient accumulators stay in pinned RAM (or device memory, as
 * lema_stream_layers allows), since every micro-step rewrites them.  The step's last micro-step streams each unit file -> pinned
 * staging buffer -> VRAM slot -> staging -> file; three staging buffers rotate so
 * that the read of unit L+2, the GPU work of unit L and the write-back of unit L-1
 * run at once.  File IO runs on the library's own threads (pread/pwrite, O_DIRECT
 * when asked); the GPU side is lema_stream_layers' pool.
 *
 * File layout.  Unit u of P_u elements (its tensors at the slot offsets of
 * lema_layer: o_j = sum over i < j of n_i rounded up to a multiple of 64, and
 * P_u = the packed size of the unit) occupies one block at byte offset
 * unit_offset[u]; with Q_u = P_u rounded up to a multiple of 2048 elements, the
 * block holds six fields at these byte offsets (every field starts on a 4096-byte
 * boundary, as O_DIRECT wants):
 *     master fp32 at 0, m fp32 at 4 Q_u, v fp32 at 8 Q_u, delta fp32 at 12 Q_u,
 *     orig bf16 at 16 Q_u, w bf16 at 18 Q_u           (block size 20 Q_u bytes)
 * and tensor j's elements start o_j elements into each field.  Blocks follow each
 * other in unit order from offset 0.  The caller writes the initial state (master
 * = widened orig, m = v = delta = 0, w = orig) before the first step.
 *
 * 8-bit layout (LEMA_DISK_Q8; the states of lema_tensor_q8).  Tensors at the
 * 1024-element offsets of lema_layer_q8 (P_u = the unit's packed size on those
 * offsets); Q_u = P_u rounded up to a multiple of 4096 elements and
 * S_u = 4 Q_u / 256 bytes (one fp32 scale per 256 elements) rounded up to a
 * multiple of 4096.  The block holds eight fields at these byte offsets:
 *     master fp32 at 0, m codes int8 at 4 Q_u, sqrt(v) codes uint8 at 5 Q_u,
 *     orig bf16 at 6 Q_u, delta fp32 at 8 Q_u, w bf16 at 12 Q_u,
 *     m scales fp32 at 14 Q_u, sqrt(v) scales fp32 at 14 Q_u + S_u
 *                                                      (block size 14 Q_u + 2 S_u)
 * with tensor j's codes and values o_j elements, and its scales o_j / 256 floats,
 * into each field.  The initial state: master = widened orig, all codes 0, all
 * scales +0.0, delta = 0, w = orig.  The step moves 20 bytes per element through
 * the file (reads master, the codes, orig, the scales; writes all but orig),
 * against 32 for fp32 states. */
typedef struct lema_disk lema_disk;

enum {
    LEMA_DISK_DIRECT = 1,   /* open the file with O_DIRECT (page cache bypassed) */
    LEMA_DISK_Q8 = 2        /* the file holds 8-bit states (the 8-bit layout above) */
};

/* The file layout for n_units units of unit_params[u] = P_u elements:
 * unit_offset[u] (n_units + 1 entries; the last is the file size) and padded[u] =
 * Q_u.  Pure host computation.  LEMA_ERR_ARG on a negative size. */
int lema_disk_layout(const int64_t* unit_params, int32_t n_units, int64_t* unit_offset,
                     int64_t* padded);

/* The same for the 8-bit layout (padded[u] = its Q_u). */
int lema_disk_layout_q8(const int64_t* unit_params, int32_t n_units, int64_t* unit_offset,
                        int64_t* padded);

/* Open an existing state file of that layout for reading and writing (its size
 * must be at least the layout's; flags LEMA_DISK_Q8 selects the 8-bit layout).
 * n_io_threads file-IO threads (1..64).  The pinned staging buffers (3 x the
 * largest block) are allocated at the first step that needs them.  LEMA_ERR_ARG, LEMA_ERR_IO (open failed, file too small) or
 * LEMA_ERR_OOM. */
int lema_disk_open(const char* path, const int64_t* unit_params, int32_t n_units,
                   int32_t flags, int32_t n_io_threads, lema_disk** out);

/* Wait, at most timeout_ms, for every read and write-back the disk has queued.
 * Returns LEMA_OK, LEMA_ERR_TIMEOUT (still pending; call again), or the first
 * error a queued operation met (LEMA_ERR_IO, or LEMA_ERR_TIMEOUT when a
 * write-back gave up waiting for the GPU copy it follows). */
int lema_disk_sync(lema_disk* disk, int32_t timeout_ms);

/* Waits for all queued IO (without a time limit), then closes the file and frees
 * the staging buffers and threads.  NULL is a no-op. */
int lema_disk_close(lema_disk* disk);

/* lema_stream_layers (LEMA_STREAMED) with the states of unit L in the disk's unit L
 * (L < the disk's n_units; each layer's packed size must equal its P_L).  In the
 * layers only n, acc (pinned host, at the slot offsets when the layer is flagged
 * LEMA_UNIT_PACKED; or device memory, as in lema_stream_layers) and the grads are read; the other pointers of each tensor
 * must be NULL.  Micro-steps k < K touch no file (the accumulator streams as in
 * lema_stream_layers).  At k == K the call blocks on the host until the last
 * unit's read has finished and its GPU work is enqueued, and queues every unit's
 * write-back; lema_disk_sync waits for those.  Results (file contents, host
 * accumulator) equal lema_stream_layers' on the same values, bit for bit.  Errors
 * as lema_stream_layers, plus LEMA_ERR_IO / LEMA_ERR_TIMEOUT from the file side. */
int lema_stream_layers_disk(lema_pool* pool, lema_disk* disk, const lema_layer* layers,
                            int32_t n_layers, int32_t micro_step,
                            const lema_adamw_hparams* hparams, int64_t step, void* cuda_stream);

/* lema_stream_layers_disk for a disk opened with LEMA_DISK_Q8: lema_stream_layers_q8
 * with the states of unit L in the disk's unit L.  In the layers only n, acc_q and
 * acc_scale (pinned host or device memory) and the grads are read; the other pointers must be NULL.
 * Results equal lema_stream_layers_q8's on the same values, bit for bit.  Errors as
 * lema_stream_layers_disk (LEMA_ERR_ARG when the disk's kind and the call differ). */
int lema_stream_layers_disk_q8(lema_pool* pool, lema_disk* disk, const lema_layer_q8* layers,
                               int32_t n_layers, int32_t micro_step,
                               const lema_adamw_hparams* hparams, int64_t step,
                               void* cuda_stream);

/* Disk bandwidth probe with the disk tier's own IO threads: writes `bytes` to a
 * new file at `path` (untimed: allocates its blocks), then times an overwrite of
 * it, a read back (checking the data), and a read of the first half while the
 * second half is overwritten, each the best of two runs; the file is removed.
 * Results in GB/s.  No CUDA. */
int lema_disk_probe(const char* path, int64_t bytes, int32_t flags, int32_t n_io_threads,
                    double* write_gbs, double* read_gbs, double* mixed_gbs);

/* Wait on the host, at most timeout_ms milliseconds (polling, never blocking in a
 * driver call), for all work the pool has enqueued.  Returns LEMA_OK, or
 * LEMA_ERR_TIMEOUT if work is still pending (the pool stays usable), or
 * LEMA_ERR_CUDA if that work failed.  Once the work is done it also returns
 * LEMA_ERR_TIMEOUT (with a message that says so) when an 8-bit step kernel of this
 * pool gave up waiting for its staged inputs since the last report: the outputs of
 * that call are then incomplete.  An lema_stream_layers_q8 call that finds such a
 * report pending returns it instead of enqueueing anything. */
int lema_pool_sync(lema_pool* pool, int32_t timeout_ms);

/* Make cuda_stream wait (on the device) for all work the pool has enqueued. */
int lema_pool_wait_stream(lema_pool* pool, void* cuda_stream);

/* Wait for the pool's work (without a time limit) and free its slots, streams and
 * events.  NULL is a no-op. */
int lema_pool_destroy(lema_pool* pool);

/* How the pool splits a unit laid out packed (LEMA_UNIT_PACKED): into at most
 * max_slices (1..8) slices of whole 8192-element chunks, each at least
 * min_slice_params elements (rounded up to whole chunks).  Each slice's
 * host-to-device copies, kernel and device-to-host copies run as soon as the same
 * slice of the stage before is done, so a unit's computation starts once its first
 * slice has arrived and its results start leaving before it is all computed; the
 * results are the same, bit for bit, for any slicing.  Units that are not packed
 * move whole.  Default: 1 (whole units; minimum slice 8,388,608 elements when
 * raised).  Applies to calls made after it.  Returns LEMA_OK or LEMA_ERR_ARG. */
int lema_pool_slices(lema_pool* pool, int32_t max_slices, int64_t min_slice_params);

/* With `on` != 0, lema_pool_slices applies only to the first unit of each streamed
 * call that goes through a slot; the other units move whole.  The first unit is the
 * one whose load no earlier copy of the call hides (the results of a call cannot go
 * back before it has arrived and been computed), while slicing the others makes the
 * two copy directions overlap more.  Off (0) by default.  Applies to calls made
 * after it.  Returns LEMA_OK or LEMA_ERR_ARG (pool is NULL). */
int lema_pool_slice_first_unit(lema_pool* pool, int32_t on);

/* Measurement mode of a pool: with `on` != 0, every later streamed call
 * (lema_stream_layers, lema_stream_layers_q8 and their disk forms) enqueues its
 * copies, events and stream ordering exactly as usual but launches no kernel, so
 * the host buffers receive whatever the slots held, not results.  Timing a step in
 * this mode against the same step with the kernels shows how much of the streamed
 * step the kernels add (nothing, when compute is fully hidden behind the copies).
 * Off (0) by default; never for training.  Waits for the pool's work first.
 * Returns LEMA_OK, LEMA_ERR_ARG or the error of that wait. */
int lema_pool_copies_only(lema_pool* pool, int32_t on);

/* Stage tracing of a pool (a timeline without an external profiler).  With
 * tracing on, each host-to-device, compute and device-to-host stage of every unit
 * records a timed CUDA event pair on its stream, after the stage's waits, so a
 * record spans exactly the stage's own work.  Timing events cost a little, so it is
 * off by default. */
typedef struct lema_trace_event {
    int32_t stage;       /* LEMA_STAGE_H2D, LEMA_STAGE_COMPUTE or LEMA_STAGE_D2H     */
    int32_t unit;        /* index of the unit within its call                        */
    int32_t call;        /* index of the lema_stream_layers call since tracing began */
    int32_t reserved;
    double start_ms;     /* relative to the earliest recorded stage start           */
    double end_ms;
} lema_trace_event;

enum { LEMA_STAGE_H2D = 0, LEMA_STAGE_COMPUTE = 1, LEMA_STAGE_D2H = 2 };

/* Waits for the pool's work, drops any earlier trace, and records at most
 * max_events stages from now on (0 turns tracing off). */
int lema_pool_trace(lema_pool* pool, int32_t max_events);

/* Waits for the pool's work and copies up to `max` records into `out`;
 * *n_out = the number recorded. */
int lema_pool_trace_read(lema_pool* pool, lema_trace_event* out, int32_t max, int32_t* n_out);

/* *count = the number of bounded waits inside kernels that ran out on the current
 * device since the library was loaded (the 8-bit step stages its inputs through
 * shared memory and waits for those copies at most about a second; a CTA whose wait
 * runs out stops and is counted here).  Expected 0.  Reads a device counter
 * (synchronous). */
int lema_kernel_wait_timeouts(int64_t* count);

/* Message for the calling thread's last failed call ("" if none). */
const char* lema_last_error(void);

/* Name of a status code. */
const char* lema_status_string(int status);

/* ------------------------------------------------------------------------------
 * Test hooks.  For the library's own failure-handling tests only: they make a
 * failure happen on purpose.  A program that trains or serves never calls them.
 * ---------------------------------------------------------------------------- */

/* The `nth_copy`-th host<->device copy the pool enqueues from now on (1 = the next
 * one) fails with LEMA_ERR_CUDA without calling CUDA; 0 disarms it.  The fault is
 * made on the host; nothing faults on the GPU. */
void lema_test_fail_copy(int64_t nth_copy);

/* Sets how long the 8-bit step kernel waits for its staged inputs on the current
 * device before it gives up (limit_ns < 0 restores the default of about a second;
 * 0 gives up at the first poll that finds the copies still in flight), so that a
 * test can make that bounded wait run out.  The kernel still lets every copy it
 * issued land (with its own, fixed bound) before it stops.  Synchronous (a copy to
 * the device).  Returns LEMA_OK or LEMA_ERR_CUDA. */
int lema_test_kernel_wait_limit(int64_t limit_ns);

/* The 8-bit step divides sqrt(v) by the per-call constant c = sqrt(1 - beta2^t)
 * with a reciprocal and two fused multiply-adds (Markstein's method) instead of a
 * division; this runs that operation on the GPU for every x >= 0 (all 2^31 bit
 * patterns, inf and NaN included) against the IEEE division, for each of `count`
 * host divisors in (2^-27, 1].  mismatches[i] counts the differing results where
 * the step uses the method (x = 0, 2^-100 <= x <= 2^64, inf, NaN; expected 0),
 * outside[i] those for the x it never meets (subnormal or tiny, and finite x above
 * 2^64, where the quotient may overflow).  Synchronous; allocates a
 * small device buffer.  Returns LEMA_OK, LEMA_ERR_ARG or LEMA_ERR_CUDA. */
int lema_test_divide_by_constant(const float* divisors, int32_t count, int64_t* mismatches,
                                 int64_t* outside);

#ifdef __cplusplus
}
#endif

#endif /* LEMA_H */
