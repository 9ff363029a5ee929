/*
 * psgd.h -- C ABI of the GB300-native PowerSGD communication-hook step.
 *
 * A data-parallel job of W workers is either simulated inside one GPU by W
 * replica gradient buckets resident in the same HBM -- the "allreduce" of the
 * pages is then a mean over those W buckets, folded into the kernels that read
 * them (psgd_step) -- or spread over W processes with one replica each, the
 * pages' two exchanges left to the caller's collective on library-owned
 * buffers (psgd_dp_*).  Every step of the method runs in CUDA kernels of this
 * library; the host side only plans, allocates (at create time) and enqueues.
 *
 * Sources (web pages; the operations are restated here, not copied):
 *   [DDP]  "DDP Communication Hooks" (PyTorch 1.11 documentation):
 *          "PowerSGD State" (PowerSGDState and its items 1-4),
 *          "PowerSGD Hooks" (powerSGD_hook steps 1-3.7, the vanilla-allreduce
 *          note, the error-feedback memory warning),
 *          "Default Communication Hooks" (allreduce_hook: the mean).
 *   [DDP2] "DDP Communication Hooks" (spec-zone.ru translation of a later
 *          version): "PowerSGD State" item 5, batch_tensors_with_same_shape.
 *   [AMP]  "Automatic Mixed Precision package - torch.cuda.amp",
 *          GradScaler: unscale, inf/NaN check, skipped step.
 *
 * Conventions for every call:
 *   - Return value: PSGD_OK (0) or a positive informational code on success,
 *     a negative PSGD_E* code on failure; psgd_last_error() then holds a
 *     message (thread-local, valid until the next failing call on the thread).
 *   - "device pointer" = CUDA global memory on the state's device; "host
 *     pointer" = ordinary (pageable or pinned) CPU memory.  The caller owns
 *     every pointer it passes; the library never frees or retains them past
 *     the call (psgd_step: past the enqueued work).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  psgd_step enqueues only and never synchronises.
 *   - Host threads: calls on one state (or one group) must not overlap in
 *     time; different states may be driven from different threads at once
 *     (the library's process-wide launch settings are atomic or locked).
 *   - Elements of a bucket are in bucket order: tensor 0 first, each tensor
 *     row-major in its own shape, with no padding between tensors.
 */
#ifndef PSGD_H
#define PSGD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct psgd_state psgd_state; /* opaque, library-owned */

/* Type of the replica gradient buckets.  F16 / BF16: 16-bit gradients, as
 * produced by GradScaler-scaled half-precision training or by the pages'
 * fp16/bf16 compress wrappers ("Default Communication Hooks":
 * fp16_compress_wrapper / bf16_compress_wrapper cast the bucket to 16 bits);
 * the library computes in fp32 and returns fp32 (the cast back). */
typedef enum { PSGD_F32 = 0, PSGD_F16 = 1, PSGD_BF16 = 2 } psgd_dtype;

#define PSGD_OK 0
#define PSGD_SKIPPED_NONFINITE 1 /* [AMP] inf/NaN seen: step skipped, state kept   */
#define PSGD_EINVAL (-1)         /* bad argument                                   */
#define PSGD_ENOMEM (-2)         /* device or host allocation failed               */
#define PSGD_ECUDA (-3)          /* a CUDA call failed                             */
#define PSGD_ETIMEOUT (-4)       /* a bounded device-side wait gave up             */

#define PSGD_MAX_RANK 32  /* largest matrix_approximation_rank ([DDP] item 1 names up to 32) */
#define PSGD_MAX_WORLD 64 /* largest number of simulated replicas W              */

/*
 * psgd_plan -- host-only planner query (no GPU needed).
 *
 * [DDP] powerSGD_hook step 1: views the flat bucket as per-parameter tensors
 * and splits them into a compressed group and an uncompressed group (every
 * tensor of fewer than 2 dimensions is uncompressed).  A tensor of >= 2 dims
 * is viewed as (shape[0], prod(shape[1:])) and compressed iff
 *   (rows + cols) * matrix_approximation_rank * min_compression_rate < rows * cols
 * ([DDP] "PowerSGD State" item 3; strict, evaluated in double precision).
 *
 *   dims, ndims, n_tensors : shapes, concatenated: tensor t has ndims[t]
 *                            entries of dims starting after the previous ones.
 *   compressed[n_tensors]  : out, 1 if the tensor is compressed.
 *   ranks[n_tensors]       : out, min(rank, rows, cols) if compressed, else 0.
 *   rows[n_tensors], cols[n_tensors] : out, the 2-D view (0,0 for < 2 dims).
 *   Any of the out arrays may be NULL.
 * Errors: PSGD_EINVAL for a negative dimension, n_tensors < 0 or rank outside
 * [1, PSGD_MAX_RANK].
 */
int psgd_plan(const int64_t* dims, const int32_t* ndims, int32_t n_tensors,
              int32_t matrix_approximation_rank, double min_compression_rate,
              int32_t* compressed, int32_t* ranks, int64_t* rows, int64_t* cols);

/*
 * psgd_state_create -- [DDP] PowerSGDState(...) for one bucket layout.
 *
 * Hyper-parameters keep the pages' names and meaning ([DDP] items 1-4,
 * [DDP2] item 5).  world_size = W simulated replicas.  grad_dtype is the type
 * of the replica buckets passed to psgd_step (F16 / BF16: 16-bit buckets).
 * Allocates on `device` everything a step needs: the per-replica error
 * feedback store, P/Q memory and all scratch; psgd_step allocates nothing.
 * The error store is kept twice (the current and the next step) so that a
 * skipped step ([AMP]) leaves the state bit-identical.
 * random_seed seeds the counter-based generator (Philox4x32-10) that draws
 * the initial standard-normal Q when none was injected with psgd_set_q.
 * Errors: PSGD_EINVAL (rank outside [1,32], world_size outside [1,64],
 * negative dims, start_powerSGD_iter < 0, min_compression_rate < 0 or NaN,
 * epsilon < 0, device ordinal 64 or above), PSGD_ENOMEM, PSGD_ECUDA (no such
 * device).  *out is NULL on failure.  Every creator takes the same device
 * rule; states on several devices may live in one process.
 */
int psgd_state_create(const int64_t* dims, const int32_t* ndims, int32_t n_tensors,
                      int32_t world_size, int32_t matrix_approximation_rank,
                      int64_t start_powerSGD_iter, double min_compression_rate,
                      int32_t use_error_feedback, int32_t warm_start,
                      float orthogonalization_epsilon, uint64_t random_seed,
                      int32_t batch_tensors_with_same_shape, psgd_dtype grad_dtype,
                      int32_t device, psgd_state** out);

/*
 * psgd_state_create_batched -- the state of [DDP] batched_powerSGD_hook
 * ("PowerSGD Hooks", batched_powerSGD_hook steps 1-9): the whole flat bucket
 * of `numel` elements is viewed as ONE square matrix of side
 * ceil(sqrt(numel)), zero beyond the bucket, compressed by one PowerSGD step
 * per psgd_step call, and the result truncated to `numel` elements.  There
 * is no compression-rate gate.  Error feedback covers the padded square
 * (psgd_error_numel = side * side; tensor 0 of psgd_tensor_info is the
 * square).  Other arguments as psgd_state_create; psgd_step and the other
 * calls work unchanged on the returned state.  Rows are read with 16-byte
 * vector accesses when side is a multiple of 4, element by element
 * otherwise.
 * Errors: PSGD_EINVAL (numel < 1, rank outside [1, 32], ...), PSGD_ENOMEM,
 * PSGD_ECUDA.
 */
int psgd_state_create_batched(int64_t numel, int32_t world_size, int32_t matrix_approximation_rank,
                              int64_t start_powerSGD_iter, int32_t use_error_feedback,
                              int32_t warm_start, float orthogonalization_epsilon,
                              uint64_t random_seed, psgd_dtype grad_dtype, int32_t device,
                              psgd_state** out);

/* Frees every device and host allocation of the state.  NULL is a no-op. */
void psgd_state_destroy(psgd_state* s);

/*
 * psgd_step -- one call of [DDP] powerSGD_hook on the W replicas.
 *
 *   grads[W] : host array of W device pointers; grads[w] is replica w's flat
 *              bucket of N elements of grad_dtype.  Read only.
 *   out      : device pointer, N floats: the bucket every replica receives
 *              (the hook's in-place update).  May alias grads[0] when
 *              grad_dtype is F32; must not overlap any other grads[w].
 *   inv_loss_scale : [AMP] unscale factor 1/scale multiplied into every
 *              gradient element (1.0f when no scaler is used).
 *   stream   : cudaStream_t; all work is enqueued on it, nothing waits.
 *
 * Semantics: while the call count is below start_powerSGD_iter, out is the
 * replica mean of every element ([DDP] vanilla-allreduce note).  Afterwards
 * the uncompressed tensors get their replica mean ([DDP] step 2) and each
 * compressed tensor M gets P Q^T with P = orth(mean_w M_w Q) and
 * Q = mean_w M_w^T P, M_w = replica w's gradient plus its error-feedback
 * residual, which then becomes M_w - P Q^T ([DDP] steps 3.1-3.7).  If any
 * unscaled gradient element is inf or NaN the step is skipped: state is left
 * as it was, `out` is unspecified, psgd_step_status reports
 * PSGD_SKIPPED_NONFINITE.  The call counter advances either way.
 * Errors (synchronous): PSGD_EINVAL (NULL pointers, overlap), PSGD_ECUDA.
 */
int psgd_step(psgd_state* s, const void* const* grads, float* out, float inv_loss_scale,
              void* stream);

/*
 * psgd_step_host -- psgd_step on HOST buffers: copies the W host buckets to
 * the device (one cudaMemcpyAsync per replica), runs the step and copies
 * `out` back to host memory.  Two device staging sets are allocated on the
 * first call (so the first call may return PSGD_ENOMEM) and alternated call
 * by call: the uploads run on an internal stream and wait only for the
 * download that last used the same set, the step runs on `stream` after the
 * uploads, and the download runs on a second internal stream after the step.
 * `stream` then waits for the download, so host_out is valid once `stream`
 * is synchronised, and consecutive calls overlap the next upload with the
 * current step and download.  Pinned host memory makes the copies
 * asynchronous; the host buffers must stay untouched until `stream` is
 * synchronised.
 *   host_grads[W] : host pointers, N elements of grad_dtype each.
 *   host_out      : host pointer, N floats.
 */
int psgd_step_host(psgd_state* s, const void* const* host_grads, float* host_out,
                   float inv_loss_scale, void* stream);

/*
 * psgd_set_graph -- enable (1) or disable (0) CUDA-graph replay of the steady
 * compressed step.  Once a state is past start_powerSGD_iter, has made its
 * first compressed step and warm-starts Q, every step enqueues the same
 * launches, and what is left to decide (skip on inf/NaN, the double-buffer
 * half, warm or fresh Q after a skipped first step) is decided on the device.
 * With graphs enabled, psgd_step captures that sequence once (on a private
 * stream, executing nothing) for its grads/out pointers and inv_loss_scale,
 * and afterwards enqueues it on `stream` with one cudaGraphLaunch while they
 * stay the same; other pointers or another scale capture again.  Results are
 * bit-identical to the launch-by-launch path.  Not used while profiling is on.
 * For callers that step with the same buffers every iteration and want the
 * host's launch cost out of the way (many small buckets).  Default: off.
 */
int psgd_set_graph(psgd_state* s, int32_t enable);

/* Graph captures and replays so far (either pointer may be NULL). */
int psgd_graph_stats(const psgd_state* s, int64_t* captures, int64_t* replays);

/*
 * psgd_step_status -- synchronises `stream` and returns the outcome of the
 * last step enqueued: PSGD_OK, PSGD_SKIPPED_NONFINITE, PSGD_ETIMEOUT (a
 * bounded wait inside a tensor-core kernel or at a grid barrier of the
 * cooperative Gram-Schmidt stage gave up; the step was not committed and the
 * state is as before it -- the call rebuilds the tensor-core operand images
 * of the committed factors, on `stream`, before returning), or PSGD_ECUDA.
 */
int psgd_step_status(psgd_state* s, void* stream);

/*
 * psgd_get_stats -- [DDP] "PowerSGD State": compression statistics.
 *   numel_before : elements of the bucket (N).
 *   numel_after  : elements exchanged per compressed step:
 *                  sum over compressed tensors of (rows + cols) * rank, plus
 *                  the uncompressed elements.
 *   iter         : psgd_step calls so far.
 * Any pointer may be NULL.
 */
int psgd_get_stats(const psgd_state* s, int64_t* numel_before, int64_t* numel_after,
                   int64_t* iter);

/*
 * psgd_tensor_info -- the planner's view of tensor `tensor`:
 * compressed flag, rows, cols, effective rank, first element in the bucket,
 * and first element in the packed error layout of psgd_get_error (-1 for an
 * uncompressed tensor).  Any out pointer may be NULL.
 */
int psgd_tensor_info(const psgd_state* s, int32_t tensor, int32_t* compressed,
                     int64_t* rows, int64_t* cols, int32_t* rank,
                     int64_t* bucket_offset, int64_t* packed_offset);

/* Elements of one replica's packed error buffer (psgd_get_error/set_error). */
int64_t psgd_error_numel(const psgd_state* s);

/*
 * psgd_set_q -- install Q for compressed tensor `tensor` from host memory,
 * cols x rank floats, row-major (rank = the tensor's effective rank).
 *   is_draw = 1 : the values are a standard-normal draw ([DDP] step 3.1: Q
 *                 is initialised from a standard normal distribution and
 *                 orthogonalised); it replaces the library's own draw the
 *                 next time the tensor needs a fresh Q (its first compressed
 *                 step, or every step when warm_start is 0) and is
 *                 orthogonalised there.
 *   is_draw = 0 : the values become the warm-start Q used as is by the next
 *                 compressed step (checkpoint restore).
 * Synchronous (blocks until the copy is done).  PSGD_EINVAL if the tensor is
 * not compressed.
 */
int psgd_set_q(psgd_state* s, int32_t tensor, const float* host_in, int32_t is_draw);

/* psgd_get_q -- the warm-start Q after the last committed step (cols x rank,
 * host memory; zeros before the first compressed step).  Synchronous. */
int psgd_get_q(psgd_state* s, int32_t tensor, float* host_out);

/* psgd_get_p -- the orthogonalised P of the last committed compressed step
 * (rows x rank, host memory; zeros before it).  Synchronous. */
int psgd_get_p(psgd_state* s, int32_t tensor, float* host_out);

/*
 * psgd_get_error / psgd_set_error -- replica `replica`'s error-feedback
 * residual ([DDP] "PowerSGD Hooks" warning: the extra memory that error
 * feedback needs), packed: compressed tensors in bucket order, each
 * row-major, at psgd_tensor_info's packed_offset; psgd_error_numel floats.
 * dev_out / dev_in are device pointers; the work is enqueued on `stream`.
 * PSGD_EINVAL when error feedback is off.
 */
int psgd_get_error(psgd_state* s, int32_t replica, float* dev_out, void* stream);
int psgd_set_error(psgd_state* s, int32_t replica, const float* dev_in, void* stream);

/* Bytes of device memory the state holds (error store, P/Q, scratch). */
size_t psgd_workspace_bytes(const psgd_state* s);

/*
 * psgd_set_error_store_halves -- keep the error-feedback store once (1) or
 * twice (2, the default).  The pages put error feedback's memory at the size
 * of the model's gradients ([DDP] "PowerSGD Hooks", the warning on error
 * feedback): one half is that, W x (compressed elements) floats per state.
 * With one half, pass 1 writes each step's M_w over the residual it has just
 * read, so the results are the same bits; but a step that meets an inf/NaN
 * has by then overwritten the store with that step's M_w, so its skip leaves
 * the factors as they were and the error feedback changed (reset it with
 * psgd_set_error, or keep two halves when gradients can be non-finite, as
 * with a GradScaler).  Must precede the first psgd_step (reallocates the
 * store, zeroed).  Errors: PSGD_EINVAL (NULL state, halves not 1 or 2, a step
 * already taken, a data-parallel state), PSGD_ENOMEM, PSGD_ECUDA.  A state
 * without error feedback has no store: the call then only returns PSGD_OK.
 */
int psgd_set_error_store_halves(psgd_state* s, int32_t halves);

/*
 * Kernel timing for measurement.  psgd_profile(s, 1) makes later psgd_step
 * calls record a CUDA event pair around every kernel they launch (on the
 * step's stream); 0 stops it.  psgd_profile_read synchronises the device,
 * then returns for kernel kind `kind` (0 .. psgd_profile_kinds()-1) its name,
 * the number of launches and the summed device time since the last read, and
 * the algorithmic bytes one launch must move (the roofline numerator); it
 * then clears that kind's record.  With launches and total_ms both NULL it
 * returns the name and bytes only and leaves the record.
 */
int psgd_profile(psgd_state* s, int32_t enable);
/*
 * psgd_profile_select -- as psgd_profile, for the kinds whose bit is set in
 * kind_mask only (bit k: kind k; 0 stops): a timed region that needs one
 * kernel's duration then carries two events per step, not two per kernel.
 * Returns PSGD_EINVAL for a NULL state.
 */
int psgd_profile_select(psgd_state* s, uint32_t kind_mask);
int32_t psgd_profile_kinds(void);
int psgd_profile_read(psgd_state* s, int32_t kind, const char** name, int64_t* launches,
                      double* total_ms, double* bytes_per_launch);

/*
 * psgd_project_q_static -- Q = M^T P for one matrix, allocating nothing.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot call cudaMalloc -- a job that reserved nearly all device memory up
 * front, code whose device memory must come from a framework's own
 * allocator, or latency-sensitive code that cannot afford cudaMalloc's
 * implicit synchronisation.  It computes what pass 2 of psgd_step computes
 * for one replica (Q(j, k) = sum_i M(i, j) P(i, k)), summing per block of
 * 512 rows in row order and then over the blocks in block order, with those
 * partial sums kept in a file-scope __device__ array of 2 Mi floats (8 MiB)
 * that every GPU loading this library holds until the process exits.
 *
 *   dev_m  : device pointer, rows x cols floats, row-major.
 *   dev_p  : device pointer, rows x rank floats, row-major.
 *   dev_q  : device pointer, cols x rank floats, row-major (output).
 *   rank   : 1 .. 32.
 *   stream : cudaStream_t; the work is enqueued on it.
 * Runs on the calling thread's current CUDA device; the first call on a
 * device looks up the array's device address (make that first call before
 * any stream capture).  Sizes with ceil(rows / 512) * next_pow2(rank) * cols
 * above 2 Mi return PSGD_EINVAL.  Every call overwrites the whole part of the
 * array it uses, so nothing carries over between calls, but calls that
 * overlap on the GPU (other streams, other threads) race on the array.
 * Errors: PSGD_EINVAL (NULL pointer, sizes), PSGD_ECUDA.
 */
int psgd_project_q_static(const float* dev_m, const float* dev_p, float* dev_q, int64_t rows,
                          int64_t cols, int32_t rank, void* stream);

/*
 * Bucket groups -- overlap across buckets.
 *
 * [DDP] "What Does a Communication Hook Operate On?": DDP splits the
 * gradients into buckets so that communication overlaps computation and calls
 * the hook once per bucket as it becomes ready; the PowerSGD state keeps its
 * error-feedback residuals and warm-start Qs per bucket.  A group holds one
 * psgd_state per bucket, all with the same hyper-parameters, and steps each
 * bucket on one of n_streams internal CUDA streams, so that one bucket's
 * latency-bound launches (Gram-Schmidt stage, reductions) run beside another
 * bucket's streaming passes.  The buckets' compressed tensors are numbered
 * across the group in bucket order for the Q draws, so a group draws the
 * same Qs as one state over the concatenated buckets.
 */
typedef struct psgd_group psgd_group; /* opaque, library-owned */

#define PSGD_MAX_GROUP_STREAMS 16

/*
 * psgd_group_create -- n_buckets buckets; bucket b holds tensors_per_bucket[b]
 * tensors, and dims/ndims list every tensor of every bucket in bucket order,
 * as psgd_state_create takes them for one bucket.  The other arguments are
 * psgd_state_create's and apply to every bucket; n_streams in [1, 16].
 * More than 8 streams overlap fully only when the process starts CUDA with
 * as many hardware work queues (CUDA_DEVICE_MAX_CONNECTIONS >= n_streams;
 * CUDA's default is 8) or replays the steps as graphs (psgd_set_graph).
 * Allocates every bucket's state and the streams on `device`.
 * Errors: PSGD_EINVAL, PSGD_ENOMEM, PSGD_ECUDA (nothing is left allocated).
 */
int psgd_group_create(int32_t n_buckets, const int32_t* tensors_per_bucket, const int64_t* dims,
                      const int32_t* ndims, int32_t world_size, int32_t matrix_approximation_rank,
                      int64_t start_powerSGD_iter, double min_compression_rate,
                      int32_t use_error_feedback, int32_t warm_start,
                      float orthogonalization_epsilon, uint64_t random_seed,
                      int32_t batch_tensors_with_same_shape, psgd_dtype grad_dtype,
                      int32_t n_streams, int32_t device, psgd_group** out);

/* Synchronises the group's streams and frees everything.  NULL is a no-op. */
void psgd_group_destroy(psgd_group* g);

/*
 * psgd_group_step -- psgd_step of bucket `bucket` (grads/out/inv_loss_scale
 * as there, sized for that bucket), enqueued on internal stream
 * bucket mod n_streams after the work enqueued so far on `stream`.  Returns
 * once enqueued; grads and out must stay valid until psgd_group_wait's
 * stream has reached the step.  Each bucket is stepped once per training
 * iteration, in any order.
 * Errors: psgd_step's, and PSGD_EINVAL for a bucket index out of range.
 */
int psgd_group_step(psgd_group* g, int32_t bucket, const void* const* grads, float* out,
                    float inv_loss_scale, void* stream);

/* Makes `stream` wait for every bucket step enqueued so far.  Enqueues only. */
int psgd_group_wait(psgd_group* g, void* stream);

/*
 * psgd_group_status -- psgd_group_wait, then synchronises `stream`:
 * PSGD_SKIPPED_NONFINITE if the last step of any bucket was skipped ([AMP]
 * inf/NaN; each bucket skips on its own inputs), else PSGD_OK.
 */
int psgd_group_status(psgd_group* g, void* stream);

/* Bucket b's state, owned by the group (introspection, Q and error views,
 * checkpointing); do not destroy it. */
int psgd_group_bucket(psgd_group* g, int32_t bucket, psgd_state** out);

/* Number of buckets (0 for NULL). */
int32_t psgd_group_size(const psgd_group* g);

/*
 * Data-parallel split of the step -- one replica per process.
 *
 * [DDP] "PowerSGD Hooks", powerSGD_hook: each worker computes its own
 * P = M_w Q and Q = M_w^T P, and the hook allreduces the uncompressed batch
 * (step 2), the Ps (step 3.3) and the Qs (step 3.6) across the workers;
 * "Default Communication Hooks", allreduce_hook: the result is the mean.
 * When each process (typically one per GPU) holds ONE replica, the linearity
 * fold that psgd_step uses for its W simulated replicas no longer applies,
 * and the step is split at its two exchanges:
 *
 *   psgd_dp_begin    pass 1 on the local replica: M = g * s + e, the local
 *                    P = M Q, the local uncompressed values and a skip flag,
 *                    all packed into one exchange buffer;
 *   (caller)         SUM-allreduce that buffer across the W processes;
 *   psgd_dp_project  P = sum / W, orthogonalise P, local Q = M^T P into a
 *                    second exchange buffer;
 *   (caller)         SUM-allreduce that buffer;
 *   psgd_dp_finish   Q = sum / W, out = P Q^T, uncompressed out = sum / W,
 *                    residual kept (factored), commit.
 *
 * The exchange buffers are library-owned device memory at fixed addresses
 * (psgd_dp_begin / psgd_dp_project return them with their float counts), so
 * the caller's collective (NCCL on device memory, or a host exchange through
 * a copy) reads and writes them in place; a SUM reduction with any
 * association order is expected.  The library itself makes no collective
 * call and reads no peer memory.  Every process must call the three stages
 * in order, step after step, with the same bucket layout and
 * hyper-parameters (random_seed included: the initial Q is drawn the same
 * on every process).  A non-finite input on any process raises that
 * process's flag in the exchanged buffer, so after the sum every process
 * skips the same step ([AMP]) and keeps its state bit-identical.  Before
 * start_powerSGD_iter the exchange buffer of psgd_dp_begin is `out` itself,
 * holding this replica's unscaled gradient (psgd_dp_project then returns
 * count 0), and psgd_dp_finish divides it by W; a non-finite sum skips.
 */

/*
 * psgd_dp_create -- the state of ONE process of a W-process data-parallel job
 * (W = world_size in [1, 64]).  Arguments as psgd_state_create; the state
 * holds this process's error-feedback residual (one replica) and the shared
 * factors.  psgd_step on it returns PSGD_EINVAL (use the three stages);
 * psgd_step_status, psgd_get_stats, psgd_tensor_info, psgd_set_q, psgd_get_q,
 * psgd_get_p, psgd_get_error / psgd_set_error (replica 0 = this process's),
 * psgd_workspace_bytes, psgd_profile* and psgd_state_destroy work as for any
 * state.  Errors: as psgd_state_create.
 */
int psgd_dp_create(const int64_t* dims, const int32_t* ndims, int32_t n_tensors, int32_t world_size,
                   int32_t matrix_approximation_rank, int64_t start_powerSGD_iter,
                   double min_compression_rate, int32_t use_error_feedback, int32_t warm_start,
                   float orthogonalization_epsilon, uint64_t random_seed,
                   int32_t batch_tensors_with_same_shape, psgd_dtype grad_dtype, int32_t device,
                   psgd_state** out);

/*
 * psgd_dp_begin -- first stage of one hook call on this process's replica.
 *   grad  : device pointer, this replica's flat bucket (N elements of
 *           grad_dtype); read here and, without error feedback, again by
 *           psgd_dp_project's kernels: keep it valid and unchanged until
 *           that call's work has run on `stream`.
 *   out   : device pointer, N floats, the bucket the hook returns (written
 *           by psgd_dp_finish; before start_powerSGD_iter also the exchange
 *           buffer).  Must not overlap grad unless grad == out (F32).
 *   inv_loss_scale, stream : as psgd_step.
 *   exchange, count : out; the device buffer (`count` floats) to
 *           SUM-allreduce across the W processes before psgd_dp_project.
 * Enqueues only.  Errors: PSGD_EINVAL (NULL pointers, stage out of order,
 * not a data-parallel state), PSGD_ECUDA.
 */
int psgd_dp_begin(psgd_state* s, const void* grad, float* out, float inv_loss_scale, void* stream,
                  float** exchange, int64_t* count);

/*
 * psgd_dp_project -- second stage, after the caller's SUM-allreduce of the
 * first exchange buffer: P = sum / W, Gram-Schmidt, local Q = M^T P.
 * exchange, count : out; the device buffer to SUM-allreduce before
 * psgd_dp_finish (count 0: nothing to exchange, as before
 * start_powerSGD_iter).  Enqueues only.  Errors: PSGD_EINVAL (stage out of
 * order), PSGD_ECUDA.
 */
int psgd_dp_project(psgd_state* s, void* stream, float** exchange, int64_t* count);

/*
 * psgd_dp_finish -- last stage, after the caller's SUM-allreduce of the
 * second exchange buffer (if any): Q = sum / W (the next warm-start Q),
 * out = P Q^T for the compressed tensors and the replica mean for the rest,
 * then the commit (or the skip).  psgd_step_status reports the outcome, the
 * same on every process.  Enqueues only.  Errors: PSGD_EINVAL (stage out of
 * order), PSGD_ECUDA.
 */
int psgd_dp_finish(psgd_state* s, void* stream);

/*
 * psgd_build_id -- "psgd-source-hash:" followed by the SHA-256 (32 hex
 * digits) of the sources, header, flags and compiler version this library
 * was built from, so that a caller can check that the loaded binary matches
 * its sources.  The string is static.
 */
const char* psgd_build_id(void);

/* Message of the last failing call on this thread ("" if none). */
const char* psgd_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PSGD_H */
