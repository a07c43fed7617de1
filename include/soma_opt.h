/*
 * soma_opt.h -- C ABI of the fused "normalize -> global-norm clip -> AdamW"
 * optimizer step for GB300 (sm_103a).
 *
 * What one step computes (SomaSpeed page, "Robot learning, at a different
 * pace", its two optimizer paragraphs: the first lists what a step does to
 * each gradient, the second how the work is batched over the tensor list):
 *
 *   over a list of tensors, with d = grad_divisor (or the tensor's group
 *   divisor, see soma_opt_set_group_divisor),
 *     norm = sqrt( sum over trainable, owned tensors of sum_i (g_i / d)^2 )
 *     c    = min(1, max_norm / (norm + 1e-6))
 *   then, for every element of every trainable tensor (owned or not),
 *     g' = g * c / d
 *     p  = p * (1 - lr * wd)
 *     m  = b1 * m + (1 - b1) * g'
 *     v  = b2 * v + (1 - b2) * g'^2
 *     p  = p - (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps),   bc_k = 1 - b_k^t
 *   with lr, b1, b2, eps, wd and the step count t of the tensor's group.
 *
 * The coefficient is that of torch.nn.utils.clip_grad_norm_ with the L2 norm,
 * which the veRL write-up calls before optimizer.step() ("veRL Training
 * Process", 4.2 PPO Update; max_norm 1.0 in "PPO Update Summary").  The
 * update is torch.optim.AdamW (decoupled decay, bias correction, eps outside
 * the square root).  Gradients may be bf16 on fp32 weights and moments; they
 * are widened to fp32 for the update (RLinf, "Adding New Models with
 * FSDP+HuggingFace", "Retaining Low-Precision Gradients").  Gradient buffers
 * are only read; frozen tensors are neither read nor written.
 *
 * Ownership of memory: every tensor buffer and the stream belong to the
 * caller; the library never frees them.  The library owns its handle and the
 * device memory behind it (tensor/chunk tables, per-chunk partial sums, the
 * norm/coefficient result) and frees it in soma_opt_destroy.
 *
 * Errors: every call returns a status; nothing aborts or exits.  All
 * argument checks run before any state change or launch, so a call that
 * returns an error other than SOMA_ERR_CUDA has changed nothing.
 * soma_opt_last_error() gives the detail text of the last failure.
 *
 * Threads: a handle may be used by one thread at a time.  Distinct handles
 * are independent.
 *
 * Streams are passed as `void*` holding a cudaStream_t (NULL = the legacy
 * default stream).
 */
#ifndef SOMA_OPT_H
#define SOMA_OPT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
typedef int32_t soma_status_t;
#define SOMA_OK               0
#define SOMA_ERR_INVALID_ARG  1  /* null pointer, negative size, bad flag, non-finite or out-of-range value */
#define SOMA_ERR_BAD_GROUP    2  /* group id not returned by soma_opt_add_group */
#define SOMA_ERR_DTYPE        3  /* unknown gradient dtype code */
#define SOMA_ERR_ALIGNMENT    4  /* buffer not aligned to its element size */
#define SOMA_ERR_OOM          5  /* device or pinned host allocation failed */
#define SOMA_ERR_CUDA         6  /* a CUDA runtime call failed (detail in soma_opt_last_error) */
#define SOMA_ERR_STATE        7  /* null or destroyed handle */
#define SOMA_ERR_LIMIT        8  /* a fixed limit: SOMA_MAX_GROUPS, or the no-alloc scratch size */

/* ---- gradient dtypes --------------------------------------------------- */
#define SOMA_DTYPE_F32   0  /* IEEE binary32 */
#define SOMA_DTYPE_BF16  1  /* bfloat16: the upper 16 bits of a binary32 */
#define SOMA_DTYPE_F16   2  /* IEEE binary16 */

#define SOMA_MAX_GROUPS  64
#define SOMA_ABI_VERSION 5

typedef struct soma_opt soma_opt;
typedef soma_opt *soma_opt_t;

/* One entry of the tensor list (56 bytes, no implicit padding).
 * All buffers are contiguous 1-D views of `numel` elements in device memory
 * (torch's Tensor.data_ptr() of a contiguous tensor).
 *   param       fp32 weights, updated in place; 4-byte aligned.  With
 *               param_lowp set these are the fp32 master weights.
 *   grad        gradient in grad_dtype; NEVER written; aligned to its element size.
 *   exp_avg     fp32 first moment m, updated in place (zeros before step 1).
 *   exp_avg_sq  fp32 second moment v, updated in place (zeros before step 1).
 *   param_lowp  optional (NULL = none): the model's bf16 or fp16 copy of the
 *               weights, overwritten in the same pass with the updated fp32
 *               weights rounded to nearest even (RLinf's FP32MasterAdamW:
 *               bf16/fp16 parameters with an fp32 master copy); 2-byte aligned.
 *   numel       >= 0.  An empty entry (0) is never read or written; its
 *               pointers may be NULL, with or without a copy dtype.
 *   group       id from soma_opt_add_group; ignored when frozen.
 *   grad_dtype  SOMA_DTYPE_F32, _BF16 or _F16; ignored when frozen.
 *   trainable   0 = frozen: never read, never written, not in the norm; its
 *               pointers may be NULL.  1 = trainable.
 *   owned       1 = this rank owns the tensor (shard): it enters the norm.
 *               0 = replicated copy: updated with the same c, not in the norm.
 *   lowp_dtype  SOMA_DTYPE_BF16 or _F16 when param_lowp is set, else 0.
 * Buffers of different entries, and the buffers of one entry, must not
 * overlap. */
typedef struct {
    float *param;
    const void *grad;
    float *exp_avg;
    float *exp_avg_sq;
    void *param_lowp;
    int64_t numel;
    int32_t group;
    uint8_t grad_dtype;
    uint8_t trainable;
    uint8_t owned;
    uint8_t lowp_dtype;
} soma_tensor_t;

/* Create a handle bound to CUDA device `device`.  Makes no CUDA call: device
 * memory is allocated on the first step.  *out is set to NULL on failure.
 * The handle stands for the optimizer object of the unfused step that the
 * veRL write-up runs after clip_grad_norm_ ("veRL Training Process", 4.2 PPO
 * Update): it holds the group settings and step counts, while the weights
 * and moments it updates stay in the caller's buffers (see "Ownership of
 * memory" above). */
soma_status_t soma_opt_create(soma_opt_t *out, int32_t device);

/* Add a parameter group with torch.optim.AdamW's hyperparameters
 * (lr >= 0, 0 <= beta1, beta2 < 1, eps > 0, weight_decay >= 0, all finite).
 * Its step count starts at 0.  Writes the new id (0, 1, ...) to *group_id.
 * Groups exist because the fused step must keep each parameter group's
 * configured behaviour (SomaSpeed page, second optimizer paragraph), as
 * RLinf's FP32MasterAdamW keeps the groups and settings of the optimizer it
 * replaces (RLinf page, "Retaining Low-Precision Gradients"). */
soma_status_t soma_opt_add_group(soma_opt_t opt, double lr, double beta1, double beta2,
                                 double eps, double weight_decay, int32_t *group_id);

/* Change a group's lr; applies to the next step.  This is how a
 * learning-rate schedule reaches the fused step, whose schedules keep their
 * configured behaviour (SomaSpeed page, second optimizer paragraph). */
soma_status_t soma_opt_set_lr(soma_opt_t opt, int32_t group, double lr);

/* Read or replace all hyperparameters of a group (same ranges as add_group):
 * the group settings that the fused step preserves (SomaSpeed page, second
 * optimizer paragraph; RLinf page, "Retaining Low-Precision Gradients"). */
soma_status_t soma_opt_get_group(soma_opt_t opt, int32_t group, double *lr, double *beta1,
                                 double *beta2, double *eps, double *weight_decay);
soma_status_t soma_opt_set_group(soma_opt_t opt, int32_t group, double lr, double beta1,
                                 double beta2, double eps, double weight_decay);

/* A group's own effective-batch divisor: its gradients are normalized by it
 * (in the norm and in the update) instead of the step's grad_divisor, e.g.
 * for parameters accumulated over a different number of micro-batches.
 * divisor > 0 and finite, or 0 to use the step's divisor (the default).
 * The normalization is the first thing the SomaSpeed page's step does to a
 * gradient (its first optimizer paragraph); the veRL write-up divides the
 * loss by the number of accumulated micro-batches (4.2 PPO Update), and
 * groups accumulated over different counts divide by different numbers. */
soma_status_t soma_opt_set_group_divisor(soma_opt_t opt, int32_t group, double divisor);
soma_status_t soma_opt_get_group_divisor(soma_opt_t opt, int32_t group, double *divisor);

/* Step count of a group (checkpoint and resume).  set: t >= 0.  AdamW's
 * bias corrections depend on it, so a resumed run must restore it to keep
 * the group's configured behaviour (SomaSpeed page, second optimizer
 * paragraph); the veRL write-up saves checkpoints every 20 training steps
 * ("Complete Training Loop", step 7, Checkpoint Saving). */
soma_status_t soma_opt_get_group_step(soma_opt_t opt, int32_t group, int64_t *t);
soma_status_t soma_opt_set_group_step(soma_opt_t opt, int32_t group, int64_t t);

/* One optimizer step over `list[0..n)` (n >= 0; list may be NULL when n == 0),
 * with effective-batch divisor grad_divisor > 0 and max_norm > 0, both
 * finite.  Each group with at least one trainable entry in the list advances
 * its step count by one.  Enqueues two kernels on `stream` and returns without
 * waiting for them: the owned square-sum (which also derives norm and c on
 * the device) and the fused update.  A list small enough for the
 * single-launch step (soma_opt_set_single_launch) runs as one kernel instead,
 * one thread-block cluster, with the same results bit for bit, unless kernel
 * timing is on.  No device-to-host synchronisation happens, except that a
 * list the handle has not prepared yet waits for the previous step's kernels
 * before its device tables are written (see the prepared-list cache below).  The group constants are fixed when the step is
 * enqueued, so a capturing `stream` gets SOMA_ERR_STATE: capture
 * soma_opt_step_graph instead. */
soma_status_t soma_opt_step(soma_opt_t opt, const soma_tensor_t *list, int64_t n,
                            double grad_divisor, double max_norm, void *stream);

/* ---- graph-capturable step -------------------------------------------------
 * The SomaSpeed page replays repeated learner work with CUDA graphs to cut
 * launch overhead (its paragraph on replaying repeated learner work).  This
 * variant of soma_opt_step can be captured in a CUDA graph and replayed: it
 * enqueues only the two kernels, which read each group's hyperparameters and
 * step count from a table in device memory and advance the step counts there
 * (one extra CTA of the square-sum kernel does it while the others stream).
 * A list small enough for the single-launch step runs as that one kernel here
 * too, its CTAs deriving the group constants themselves.
 * grad_divisor, max_norm and the group divisors become part of a captured
 * graph.
 *
 * Rules: soma_opt_push_groups must have run once; the first call with a list
 * must happen outside capture (it builds and uploads the tables); from then
 * on the handle keeps that list and its launch plan for its lifetime (other
 * lists and soma_opt_set_tuning fail with SOMA_ERR_STATE; use another handle),
 * so a captured graph never sees its tables move.  The host copy of the step
 * counts is not advanced; soma_opt_pull_groups refreshes it.  To mix the two
 * kinds of step on one handle, call soma_opt_pull_groups before a regular step
 * that follows graph steps, and soma_opt_push_groups before graph steps that
 * follow regular ones. */
soma_status_t soma_opt_step_graph(soma_opt_t opt, const soma_tensor_t *list, int64_t n,
                                  double grad_divisor, double max_norm, void *stream);

/* Device table entry of one group (64 bytes); soma_opt_device_groups returns
 * SOMA_MAX_GROUPS of them, indexed by group id. */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
    int64_t reserved[2];
} soma_device_group_t;

/* Copy the host-side hyperparameters of every group to the device table,
 * and the host step count of each group whose count is newer than the
 * device's (the first push, soma_opt_set_group_step, or regular steps since
 * the last push); step counts that only graph steps advanced are kept.
 * Enqueued on `stream` from library-owned pinned memory; not capturable; it
 * waits only if its previous copy is still queued.  Call it after
 * add/set_group/set_lr/set_group_step changes that graph steps should see. */
soma_status_t soma_opt_push_groups(soma_opt_t opt, void *stream);

/* Copy the device step counts back to the host copy, so that
 * soma_opt_get_group_step reports graph steps (waits on `stream`; not
 * capturable). */
soma_status_t soma_opt_pull_groups(soma_opt_t opt, void *stream);

/* Device address of the group table (library-owned, valid until destroy).
 * A caller may write lr or other fields there between or inside graph
 * replays, e.g. from its own learning-rate schedule kernel. */
soma_status_t soma_opt_device_groups(soma_opt_t opt, soma_device_group_t **table);

/* ---- multi-rank step (shard groups) -----------------------------------------
 * With FSDP/HSDP each rank owns some shards; the SomaSpeed page takes one
 * global clipping decision in which every shard counts once (its second
 * optimizer paragraph, on batching the work over the tensor list).  The only data
 * the ranks exchange is one double per rank:
 *
 *   1. soma_opt_sumsq: this rank's sum over its trainable, owned entries of
 *      (g/d)^2, written by the square-sum kernel to sumsq_out (device memory);
 *   2. the caller gathers the ranks' values into one device array, rank r at
 *      index r (e.g. an all-gather over the shard group);
 *   3. soma_opt_step_from_sumsq: adds rank_sumsq[0..nranks) in index order,
 *      so every rank derives the same norm and c bit for bit, then runs the
 *      fused update on this rank's list.  Group step counts advance as in
 *      soma_opt_step; soma_opt_get_norm reports the global norm.
 *
 * Both calls are asynchronous on `stream`; a replicated tensor must be owned
 * by exactly one rank of the group.  Like soma_opt_step, both return
 * SOMA_ERR_STATE on a capturing stream. */
#define SOMA_MAX_RANKS 65536
soma_status_t soma_opt_sumsq(soma_opt_t opt, const soma_tensor_t *list, int64_t n, double grad_divisor,
                             double *sumsq_out, void *stream);
soma_status_t soma_opt_step_from_sumsq(soma_opt_t opt, const soma_tensor_t *list, int64_t n,
                                       double grad_divisor, double max_norm,
                                       const double *rank_sumsq, int32_t nranks, void *stream);

/* Norm and clip coefficient of the last step (fp64): the total norm that
 * torch.nn.utils.clip_grad_norm_ returns in the unfused step of the veRL
 * write-up ("veRL Training Process", 4.2 PPO Update), read here from device
 * memory after the fused step.  Also the number of steps
 * since the previous soma_opt_get_norm on this handle whose norm was not
 * finite (so at least 1 if the last step's was not; a loop that reads the norm
 * only every few steps still learns of a non-finite one in between).  Any
 * output pointer may be NULL.  Waits for the last step on `stream`: the only
 * call besides soma_opt_read_timing that blocks. */
soma_status_t soma_opt_get_norm(soma_opt_t opt, double *norm, double *clip_coef,
                                int32_t *nonfinite, void *stream);

/* Kernel timing: when enabled, each step records CUDA events around its two
 * kernels on the step's stream (a timed step always runs as the two kernels,
 * also for a list that would otherwise take the single-launch step).
 * read_timing waits for them and returns the summed kernel times (ms) and the
 * number of steps since the last read. */
soma_status_t soma_opt_set_timing(soma_opt_t opt, int32_t enable);
soma_status_t soma_opt_read_timing(soma_opt_t opt, double *norm_ms, double *update_ms,
                                   int64_t *steps);

/* Launch plan of the last step: chunk and segment counts, grid and block
 * sizes of the square-sum and update kernels, the kernels the last step
 * launched, and single_launch_ctas: the CTAs of its one cluster when it ran
 * as the single-launch step, else 0.  Any pointer may be NULL. */
typedef struct {
    int64_t norm_chunks, norm_segments, update_chunks, update_segments;
    int32_t norm_grid, norm_block, update_grid, update_block;
    int64_t trainable_numel, owned_numel;
    int32_t launches_per_step;
    int32_t single_launch_ctas;
} soma_plan_t;
soma_status_t soma_opt_get_plan(soma_opt_t opt, soma_plan_t *plan);

/* Segment table of the last step's list, for tests and debugging.  A table
 * cuts the list's tensors into segments (a contiguous element range of one
 * tensor) and groups them into chunks of about the same size; one CTA
 * processes one chunk.  The update table covers every trainable element, the
 * norm table the trainable, owned ones (the work that the SomaSpeed page
 * batches across tensors, its second optimizer paragraph).
 *   grad   address of the segment's first gradient element, so that
 *          (grad - tensor's grad) / element size is its offset in the tensor
 *   chunk  index of the chunk that holds the segment (chunks in table order)
 *   len    elements; head: elements before the 8-element vector body;
 *   nvec   vectors in the body; group: the entry's group
 * which: 0 = update table, 1 = norm table.  Writes the table's segment
 * count to *count and its first min(cap, count) segments to out (out may be
 * NULL when cap is 0).  Waits for the handle's last step; SOMA_ERR_STATE
 * before the first step. */
typedef struct {
    const void *grad;
    int64_t chunk;
    int32_t len, head, nvec, group;
} soma_segment_t;
soma_status_t soma_opt_get_segments(soma_opt_t opt, int32_t which, soma_segment_t *out, int64_t cap,
                                    int64_t *count);

/* Prepared-list cache.  A handle keeps the device tables of the last
 * SOMA_PLAN_CACHE distinct lists it stepped (lists compared entry by entry,
 * bytewise), so that steps alternating between a few lists, such as two
 * gradient buffers used in turn, find their tables ready: no validation, no
 * host table build, no upload and no wait.  A new list replaces the least
 * recently used one.  soma_opt_set_tuning drops them all.  The caller must
 * not free or reuse a buffer that a prepared list names while a step on that
 * list may still be in flight; the cache holds pointers only and never
 * dereferences them on the host.
 * builds: table builds so far; reuses: steps that found their list
 * prepared; entries: lists held now.  Any pointer may be NULL. */
#define SOMA_PLAN_CACHE 4
soma_status_t soma_opt_get_cache_stats(soma_opt_t opt, int64_t *builds, int64_t *reuses,
                                       int32_t *entries);

/* Tuning knobs for benchmarks: elements per update chunk and per norm chunk
 * (rounded to a multiple of 64; 0 = automatic) and, per kernel, resident CTAs
 * per SM for a persistent grid (0 = one CTA per chunk).  Automatic sizes:
 *   update chunks of 12 Ki elements, or 8 Ki when at least half of the
 *   trainable elements have fp32 gradients; a list that one wave of the
 *   update kernel's resident CTAs (two per SM) holds in such chunks is cut
 *   into one wave's worth instead, one that two waves hold into two waves'
 *   worth, never below 1 Ki;
 *   norm chunks of 320 Ki with a shrinking tail for lists whose owned
 *   tensors average at least 320 Ki elements; for other lists 112 Ki, or one
 *   wave of the square-sum kernel's resident CTAs (three per SM) for a list
 *   that one wave holds in such chunks, never below 1 Ki.
 * Results do not depend on the grid, only on the chunk sizes.  Takes effect
 * at the next list (re)build. */
soma_status_t soma_opt_set_tuning(soma_opt_t opt, int32_t update_chunk, int32_t norm_chunk,
                                  int32_t update_ctas_per_sm, int32_t norm_ctas_per_sm);

/* Single-launch step for small lists.  For a list of at most max_elements
 * trainable elements, a regular or graph-capturable step is one kernel: one
 * thread-block cluster (16 CTAs where the device can run such a cluster, else
 * 8, 4 or 2) whose CTAs square-sum their share of the norm chunks, meet at
 * the hardware cluster barrier, each add all chunk sums in the fixed order of
 * the two-kernel path (so each derives the same c), and update their share of
 * the list.  The chain of two dependent kernels costs more than the work of
 * such a list.  Such lists are cut into about one chunk per CTA in both
 * tables (unless soma_opt_set_tuning fixed the chunk sizes), and the
 * two-kernel path (timed steps, the multi-rank step) uses the same tables, so
 * every path gives the same bits.  max_elements: -1 = automatic (4096 per CTA
 * of the cluster, one 8-element vector per thread: 65536 with 16 CTAs; larger
 * lists ran faster as two kernels on GB300), 0 = never.  Drops the prepared
 * lists like soma_opt_set_tuning, and like it fails with SOMA_ERR_STATE on a
 * handle that ran a graph-capturable step. */
soma_status_t soma_opt_set_single_launch(soma_opt_t opt, int64_t max_elements);

/* Text of a status code (static storage). */
const char *soma_status_string(soma_status_t status);

/* Detail of the last failure on `opt` (or, for opt == NULL, of the calling
 * thread's last failed soma_opt_create).  Valid until the next call on it. */
const char *soma_opt_last_error(soma_opt_t opt);

/* SOMA_ABI_VERSION of the loaded library. */
int32_t soma_abi_version(void);

/* Wait for the handle's outstanding work, free its device and host memory
 * and the handle.  NULL is ignored.  Only what the library allocated is freed
 * ("Ownership of memory" above): the caller's weights, gradients and moments,
 * the state of the unfused AdamW this step replaces (veRL write-up, 4.2 PPO
 * Update), are left as they are. */
void soma_opt_destroy(soma_opt_t opt);

/* ---- norm without allocation ---------------------------------------------
 * No counterpart on the pages: this entry point exists for callers that may
 * not allocate device memory -- an application whose own allocator owns the
 * device heap (where an extra cudaMalloc fails or fragments its pool), or a
 * latency-critical loop where cudaMalloc/cudaFree, which can synchronise the
 * device, are not allowed.
 *
 * Computes, on `stream`, the norm and clip coefficient that the first kernel
 * of soma_opt_step computes (norm over trainable, owned entries of `list`,
 * c = min(1, max_norm / (norm + 1e-6))) and writes them as two doubles
 * {norm, c} to `out` (device memory, 8-byte aligned, caller-owned).  Its
 * chunks are larger than the step's, so its partial sums are added in a
 * different grouping: the two norms agree within 1e-5 relative, not bit for
 * bit.  It updates nothing and needs no handle; only the entries' grad,
 * grad_dtype, numel, trainable and owned fields are read.
 *
 * Scratch: a fixed array of SOMA_NOALLOC_SCRATCH_BYTES (4 MiB) in the
 * library's device image.  The CUDA runtime loads that image lazily, so the
 * array takes its 4 MiB of device memory on the first call on each device and
 * keeps it until the process exits: make that first call while 4 MiB are
 * still free, before the caller's own allocator reserves the device heap.  No
 * cudaMalloc, cudaFree or other allocating call is made.  A list whose tables
 * and partial sums do not fit returns SOMA_ERR_LIMIT before anything is
 * enqueued.  Each owned entry takes at least one 64-byte segment, and a list
 * is cut into at most about 32 768 chunks of at least 32 Ki elements, so at
 * least 26 000 owned entries fit whatever their sizes (about 65 000 when they
 * are small enough to share chunks).
 *
 * Asynchrony: the call enqueues its work on `stream` and returns without
 * waiting for the GPU.  The tables travel to the array in the arguments of
 * small copy kernels (one launch per 30,400 bytes of table; a launch copies
 * its arguments when it is enqueued), then the square-sum kernel and a
 * device-to-device copy of {norm, c} to `out` follow, so `out` is valid once
 * `stream` reaches that point.  The first call on a device, with that device
 * made current, also looks up the array's device address and keeps it; make
 * that first call before any stream capture.  Every call shares the array
 * and overwrites what the previous call left there (it clears the result
 * block each time).  Calls on one stream are ordered; calls that overlap on
 * the GPU -- on unordered streams, or from several host threads -- race on
 * the array: order them.  Returns SOMA_ERR_INVALID_ARG, SOMA_ERR_DTYPE,
 * SOMA_ERR_ALIGNMENT, SOMA_ERR_LIMIT or SOMA_ERR_CUDA (no detail text). */
#define SOMA_NOALLOC_SCRATCH_BYTES (4u << 20)
soma_status_t soma_clip_norm_noalloc(int32_t device, const soma_tensor_t *list, int64_t n,
                                     double grad_divisor, double max_norm, double *out,
                                     void *stream);

#ifdef __cplusplus
}
#endif
#endif /* SOMA_OPT_H */
