/*
 * vpce.h -- vocab-parallel cross-entropy on one GB300 (sm_103a).
 *
 * The operation ("Distributed Training III: Model Parallelism", CMU 11-868
 * Lecture 16 notes, §5.5 "Embedding and output layer"; "LLM Internals" §7.3
 * "Model and tensor parallelism", §7.3.4): the LM-head logits z[s, V] are split
 * along the vocabulary into t shards.  Each shard reduces, per row, its
 * maximum, its sum of exponentials and -- if the row's target column falls in
 * the shard's [vocab_start, vocab_end) -- the target logit.  The partials
 * combine into logsumexp(z_r) and the loss CE_r = logsumexp(z_r) - z_r[y_r]
 * without ever gathering the full rows.  Here all t shards live on one GPU and
 * the combine runs on the device, in a fixed order.
 *
 * The backward (not given by the pages; the standard derivative of the reduced
 * loss) overwrites the shards in place with
 *     dlogits_rk = g * (softmax(z_r)_k - [k == y_r]) / n_valid    (mean)
 *     dlogits_rk = g * (softmax(z_r)_k - [k == y_r])              (sum)
 *     dlogits_rk = g_r * (softmax(z_r)_k - [k == y_r])            (none)
 * and with zeros on rows whose target is ignore_index.  'none' is the
 * per-row mode of torch.nn.functional.cross_entropy, the routine the CMU notes
 * check the sharded loss against: one loss per row, and one upstream gradient
 * g_r per row (the *_rows entry points take them as a device vector).
 *
 * Conventions for every entry point
 * ---------------------------------
 * - All calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL
 *   is the legacy default stream), except vpce_read_error_flag, which
 *   synchronises the stream.  The current CUDA device must be the one that
 *   owns every device pointer, and it must be a compute-capability 10.3 GPU.
 * - The caller owns every buffer.  The library allocates nothing and keeps no
 *   per-call state; the only thing carried from forward to backward is the
 *   caller's workspace.
 * - Host-detectable argument errors return a non-OK status and launch
 *   nothing.  A launch failure returns VPCE_ERR_CUDA.
 * - Logits layout: shard i is a row-major [s, w_i] array of `dtype` elements
 *   at device address shards[i], w_i = vocab_start[i+1] - vocab_start[i], with
 *   a row stride of `ld` elements (ld = 0: each shard is dense, stride w_i).
 *   A shard may be a column block of one big [s, V] tensor (shards[i] =
 *   base + vocab_start[i], ld = V).  Shard pointers need only element
 *   alignment; rows that are not 16-byte aligned take a scalar path for their
 *   ragged head and tail elements.
 * - Targets: int64[s] on the device, replicated view of the whole batch.  A
 *   target equal to ignore_index drops its row; any other target outside
 *   [0, V) is not trapped: the row's loss, lse and gradient become NaN and the
 *   workspace error flag gets bit 0 (read it with vpce_read_error_flag).
 */
#ifndef VPCE_H
#define VPCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime's opaque stream handle). */
typedef struct CUstream_st* vpce_stream_t;

typedef enum {
  VPCE_OK = 0,
  VPCE_ERR_INVALID_ARG = 1,       /* null pointer, bad t/s/ld/vocab_start/reduction */
  VPCE_ERR_ALIGNMENT = 2,         /* a pointer not aligned to its element / 256 B workspace */
  VPCE_ERR_DTYPE = 3,             /* dtype is not VPCE_FP32 or VPCE_BF16 */
  VPCE_ERR_WORKSPACE = 4,         /* workspace_bytes < vpce_workspace_bytes(t, s) */
  VPCE_ERR_CUDA = 5,              /* a CUDA runtime call or a launch failed */
  VPCE_ERR_UNSUPPORTED_DEVICE = 6 /* current device is not compute capability 10.3 */
} vpce_status;

typedef enum { VPCE_FP32 = 0, VPCE_BF16 = 1 } vpce_dtype;

/* Reduction of the per-row losses, as torch.nn.functional.cross_entropy. */
typedef enum { VPCE_MEAN = 0, VPCE_SUM = 1, VPCE_NONE = 2 } vpce_reduction;

#define VPCE_MAX_SHARDS 64

/* Error-flag bits written to the workspace by the device. */
#define VPCE_FLAG_BAD_TARGET 1    /* some target is neither ignore_index nor in [0, V) */
#define VPCE_FLAG_WAIT_TIMEOUT 2  /* a pipeline wait gave up (never expected) */

/*
 * Bytes of device workspace vpce_forward / vpce_backward need for t shards
 * and s rows (t in [1, VPCE_MAX_SHARDS], s >= 0).  Returns 0 for arguments out
 * of range.  The workspace holds the per-(shard, row) partials (8 B each), the
 * per-row target logit and logsumexp (4 B each), the batch count n_valid, the
 * error flag and the combine's per-block sums.  Caller allocated, 256-byte
 * aligned, no initialisation needed.
 */
size_t vpce_workspace_bytes(int t, int64_t s);

/*
 * Forward: loss of the vocab-sharded logits.  Implements the pages' sharded
 * cross-entropy ("Distributed Training III: Model Parallelism", CMU 11-868
 * Lecture 16 notes, §5.5 "Embedding and output layer": each card reduces its
 * block to a maximum, a sum of exponentials and, where it holds the target,
 * the target logit; the blocks combine to logsumexp minus the target logit;
 * "LLM Internals" §7.3.4: the same three quantities for the [8192, 128256]
 * head split 16032 columns per card), with the t shards on one GPU and the
 * combine on the device.  A wait that gave up (VPCE_FLAG_WAIT_TIMEOUT) makes
 * every valid row's loss and the reduced loss NaN.
 *   shards       host array of t device pointers (read only here).
 *   dtype        element type of every shard.
 *   t            number of shards, 1..VPCE_MAX_SHARDS.
 *   s            rows (tokens), >= 0.  s = 0 gives loss NaN (mean) or 0 (sum).
 *   vocab_start  host array of t+1 offsets: vocab_start[0] = 0, strictly
 *                increasing, V = vocab_start[t] < 2^31.  Shard i holds global
 *                columns [vocab_start[i], vocab_start[i+1]); widths may differ
 *                (a V not divisible by t needs no padding).
 *   ld           row stride in elements shared by all shards, >= every
 *                width; 0 means each shard is dense.
 *   targets      device int64[s].
 *   ignore_index target value that drops a row (torch default -100).
 *   reduction    VPCE_MEAN: sum of valid-row losses / n_valid (NaN when
 *                n_valid = 0); VPCE_SUM: the plain sum; VPCE_NONE: the
 *                per-row losses are the result (row_loss_out required).
 *   loss_out     device float, receives the reduced loss.  With VPCE_NONE
 *                it may be NULL; when given it receives the plain sum.
 *   row_loss_out device float[s] or NULL (required for VPCE_NONE when s > 0); receives
 *                CE_r for valid rows, 0 for ignored rows, NaN for
 *                out-of-range targets.
 *   workspace    device buffer of workspace_bytes >= vpce_workspace_bytes.
 * Results are bitwise reproducible for fixed inputs and t: the shards fold
 * in ascending index order and the batch sum runs in a fixed order (a
 * compensated fp32 pair per lane, about 48 bits, added across warps in
 * fp64).
 */
vpce_status vpce_forward(const void* const* shards, vpce_dtype dtype, int t, int64_t s,
                         const int64_t* vocab_start, int64_t ld,
                         const int64_t* targets, int64_t ignore_index,
                         vpce_reduction reduction, float* loss_out, float* row_loss_out,
                         void* workspace, size_t workspace_bytes, vpce_stream_t stream);

/*
 * Backward: overwrite the shards in place with dlogits (same dtype; bf16 is
 * rounded to nearest-even from the fp32 value).  Not on the pages, which
 * give no backward: the standard derivative of the reduced cross-entropy,
 * g * (softmax - onehot) / n_valid for 'mean', computed shard by shard from
 * the forward's logsumexp (the combine of the CMU notes' §5.5 and "LLM
 * Internals" §7.3.4 is what makes softmax available per shard).  Every argument describing the
 * logits and targets must equal the preceding vpce_forward's, the shards must
 * still hold that call's logits, and `workspace` must be that call's,
 * unmodified (it carries logsumexp, n_valid and the reduction).
 * grad_output is the upstream gradient g of the reduced loss (1.0 normally);
 * after a VPCE_NONE forward it is applied to every row, as VPCE_SUM.
 * vocab_start[0] may be > 0 when the shards are one process's part of the
 * vocabulary and the workspace comes from vpce_combine_partials.
 * Padding columns (ld > w_i) are neither read nor written.
 */
vpce_status vpce_backward(void* const* shards, vpce_dtype dtype, int t, int64_t s,
                          const int64_t* vocab_start, int64_t ld,
                          const int64_t* targets, int64_t ignore_index,
                          float grad_output, const void* workspace, size_t workspace_bytes,
                          vpce_stream_t stream);

/*
 * Backward of the per-row losses (reduction 'none'): as vpce_backward, but
 * with one upstream gradient per row, dlogits_rk = grad_rows[r] *
 * (softmax(z_r)_k - [k == y_r]), whatever reduction the forward used.
 *   grad_rows  device float[s] (4-byte aligned), read only; entry r is
 *              d(outer loss)/d(CE_r).  Ignored rows get zeros whatever their
 *              entry; any other entry is used as given (0 gives zeros, a
 *              negative value flips the sign, NaN gives NaN).
 */
vpce_status vpce_backward_rows(void* const* shards, vpce_dtype dtype, int t, int64_t s,
                               const int64_t* vocab_start, int64_t ld,
                               const int64_t* targets, int64_t ignore_index,
                               const float* grad_rows, const void* workspace, size_t workspace_bytes,
                               vpce_stream_t stream);

/*
 * The two halves of vpce_forward, for shards spread over several processes
 * (one GPU each), with the exchange in between done by the caller -- the
 * pages' multi-card method ("Distributed Training III: Model Parallelism",
 * CMU 11-868 Lecture 16 notes, §5.5; "LLM Internals" §7.3.4): each card
 * reduces its columns to per-row partials, the cards exchange them, and every
 * card combines them.
 *
 * vpce_partials: this process's shards (vocab_start: t+1 global column
 * offsets, vocab_start[0] >= 0, the shards' part of the vocabulary) reduced
 * per (shard, row) to part_out[i * s + r] = (max, sum exp(z - max)) (device
 * float2 [t][s]) and tgt_out[r] = the target logit when this process holds
 * the target's column, else 0 (device float [s], cleared here).  workspace
 * as vpce_forward's (vpce_workspace_bytes(t, s)); other arguments as
 * vpce_forward.
 *
 * vpce_combine_partials: n_part partials [n_part][s] (all processes' part_out
 * gathered, in a fixed order) and tgt [s] (the sum over processes of tgt_out,
 * exact since one term per row is non-zero) combined into logsumexp, the row
 * losses and the reduced loss with vpce_forward's per-row arithmetic (folded
 * in index order; the batch sum in fp64 over fixed blocks).  V is the whole vocabulary (the bad-target
 * check).  The workspace is laid out for t_local shards so that
 * vpce_backward on this process's t_local shards (with their global
 * vocab_start) reads its logsumexp and n_valid; its header is cleared here.
 */
vpce_status vpce_partials(const void* const* shards, vpce_dtype dtype, int t, int64_t s,
                          const int64_t* vocab_start, int64_t ld, const int64_t* targets,
                          int64_t ignore_index, float* part_out, float* tgt_out,
                          void* workspace, size_t workspace_bytes, vpce_stream_t stream);
vpce_status vpce_combine_partials(const float* part, int n_part, const float* tgt, int64_t s, int64_t V,
                                  const int64_t* targets, int64_t ignore_index, vpce_reduction reduction,
                                  float* loss_out, float* row_loss_out, int t_local,
                                  void* workspace, size_t workspace_bytes, vpce_stream_t stream);

/*
 * One process's partials folded to one (max, sum exp) pair per row before
 * the exchange, so that each process sends the pages' three scalars per
 * token -- maximum, sum of exponentials and (through the target all-reduce)
 * the target logit -- whatever number of shards it holds ("Distributed
 * Training III: Model Parallelism", CMU 11-868 Lecture 16 notes, §5.5: 12
 * bytes per token instead of the logits).  part: device float2 [t][s] as
 * vpce_partials writes it; out: device float2 [s] (8-byte aligned, may not
 * overlap part), out[r] = (M, S) with M = max_i part[i][r].max and
 * S = sum over i ascending of part[i][r].sum * exp(part[i][r].max - M), the
 * combine's arithmetic.  Folded pairs of all processes, gathered in process
 * order, go to vpce_combine_partials as n_part = (number of processes)
 * partials.  Errors: t outside 1..VPCE_MAX_SHARDS or s < 0
 * (VPCE_ERR_INVALID_ARG), misaligned pointers (VPCE_ERR_ALIGNMENT).
 */
vpce_status vpce_fold_partials(const float* part, int t, int64_t s, float* out, vpce_stream_t stream);

/*
 * Forward and backward in one call: the loss (as vpce_forward) and the shards
 * overwritten in place with dlogits for upstream gradient grad_output (as
 * vpce_backward), for the common case where the loss is the last op and g is
 * known before the forward runs (1.0, or a loss scale).  Each row's backward
 * follows its forward while the row is still in L2 (a CTA's stats warps
 * stream a row in, its grad warps re-read it from L2 about a row later), so
 * the logits cross HBM about once in each direction instead of three passes.  Arguments
 * as vpce_forward plus grad_output; the workspace afterwards holds logsumexp
 * and n_valid like a forward's.  Rows that are not 16-byte aligned (shard
 * pointer, row stride or width in bytes) run the two-call path instead, with
 * the same results.  The batch loss is summed in a fixed order (compensated
 * fp32 pairs, fp64 across warps), so results are bitwise reproducible; they
 * agree with the two-call path within rounding.
 */
vpce_status vpce_forward_backward(void* const* shards, vpce_dtype dtype, int t, int64_t s,
                                  const int64_t* vocab_start, int64_t ld,
                                  const int64_t* targets, int64_t ignore_index,
                                  vpce_reduction reduction, float grad_output,
                                  float* loss_out, float* row_loss_out,
                                  void* workspace, size_t workspace_bytes, vpce_stream_t stream);

/*
 * vpce_forward_backward with one upstream gradient per row (known before the
 * call, e.g. per-token loss weights): the loss as vpce_forward with
 * `reduction`, and dlogits as vpce_backward_rows with grad_rows (device
 * float[s], 4-byte aligned).  Same single pass over HBM and same fallback.
 */
vpce_status vpce_forward_backward_rows(void* const* shards, vpce_dtype dtype, int t, int64_t s,
                                       const int64_t* vocab_start, int64_t ld,
                                       const int64_t* targets, int64_t ignore_index,
                                       vpce_reduction reduction, const float* grad_rows,
                                       float* loss_out, float* row_loss_out,
                                       void* workspace, size_t workspace_bytes, vpce_stream_t stream);

/*
 * How vpce_forward_backward would run the given problem on the current
 * device (no launch): *kernel = 0 two-call path (a shard's width in bytes is
 * not a multiple of 16; misaligned pointers or strides also take it),
 * 1 fused streaming kernel on a persistent grid of *grid CTAs, one per SM.
 * *cluster is 1, or 2 when rows are longer than 224 KB: a pair of CTAs then
 * shares each row, so that the rows kept live between the two passes still
 * fit in L2 with room for the statistics pass to run ahead.
 */
vpce_status vpce_fused_plan(vpce_dtype dtype, int t, const int64_t* vocab_start, int64_t s,
                            int* kernel, int* cluster, int* grid);

/*
 * Forward without a workspace argument, for callers that cannot allocate
 * device memory where they need the loss: a plugin inside a framework whose
 * pooling allocator already owns the GPU's memory (a raw cudaMalloc would fail
 * or fragment that pool), a path that cannot afford cudaMalloc's implicit
 * device synchronisation, or a deployment that forbids device allocation
 * after start-up.  The pages have no counterpart: this is a packaging
 * variant of vpce_forward, with identical arguments and results except that
 * the scratch is a file-scope device array of VPCE_STATIC_SCRATCH_BYTES held
 * by every GPU that loads this library until the process exits.  The caller
 * still passes the logits, targets and outputs.
 *   - Calls the library makes: no cudaMalloc, cudaFree or other allocating
 *     routine; the first call on each device looks the array's address up
 *     (cudaGetSymbolAddress, with that device current), so make that first
 *     call before any stream capture.
 *   - Limit: returns VPCE_ERR_WORKSPACE, launching nothing, when
 *     vpce_workspace_bytes(t, s) > VPCE_STATIC_SCRATCH_BYTES (8 MiB covers,
 *     e.g., t = 16 at s = 32768, t = 8 at s = 65536 and t = 64 at s = 8192;
 *     roughly 8 * t * s + 12 * s bytes are needed).
 *   - Every call on a device shares the one array and the next call overwrites
 *     it (each call clears what must start at zero), so calls that may
 *     overlap on the GPU -- on different streams, or from different threads --
 *     race: serialise them on one stream.  The workspace stays inside the
 *     library, so no vpce_backward can follow this forward, and its error
 *     flag cannot be read: a bad target gives that row, and a wait that gave
 *     up gives every row, a NaN loss, so a NaN loss_out is the signal.
 *   - The array's address is cached per device after the first call, so a
 *     device reset (cudaDeviceReset) after that call is not supported.
 */
#define VPCE_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)
vpce_status vpce_forward_static(const void* const* shards, vpce_dtype dtype, int t, int64_t s,
                                const int64_t* vocab_start, int64_t ld,
                                const int64_t* targets, int64_t ignore_index,
                                vpce_reduction reduction, float* loss_out, float* row_loss_out,
                                vpce_stream_t stream);

/*
 * LM-head GEMM fused with the forward loss: the logits of shard i are
 * z_i = X W_i^T, computed tile by tile on the tensor cores (bf16 in, fp32
 * accumulate) and reduced in the tile's epilogue to the per-row maximum, sum
 * of exponentials and target logit, so the [s, V] logits are never written
 * ("Distributed Training III: Model Parallelism", CMU 11-868 Lecture 16
 * notes, §5.5: do not assemble the big tensor, move the later computation to
 * the data; "LLM Internals" §7.3.4: the LM head [128256, 8192] split by
 * vocabulary, 16032 rows per card at t = 8).  The combine and the batch sum
 * are vpce_forward's, so loss_out, row_loss_out, the reduction and the
 * workspace's logsumexp / n_valid / error flag mean the same.
 *   hidden         device bf16 [s, h], row stride ld_hidden elements (0 = h);
 *                  16-byte aligned base, ld_hidden * 2 a multiple of 16.
 *   weight_shards  host array of t device pointers; shard i is bf16
 *                  [w_i, h] (one row per vocabulary entry, K contiguous),
 *                  row stride ld_weight elements (0 = h); 16-byte aligned,
 *                  ld_weight * 2 a multiple of 16.
 *   t              1..32 shards; vocab_start as vpce_forward (t+1 offsets).
 *   h              hidden size, a positive multiple of 64.
 *   workspace      vpce_lmhead_workspace_bytes(s) bytes, 256-byte aligned.
 * Other arguments and errors as vpce_forward.  The backward is
 * vpce_lmhead_backward.
 */
#define VPCE_LMHEAD_MAX_GROUPS 256
size_t vpce_lmhead_workspace_bytes(int64_t s);
vpce_status vpce_lmhead_forward(const void* hidden, int64_t ld_hidden,
                                const void* const* weight_shards, int64_t ld_weight,
                                int t, int64_t s, int64_t h, const int64_t* vocab_start,
                                const int64_t* targets, int64_t ignore_index,
                                vpce_reduction reduction, float* loss_out, float* row_loss_out,
                                void* workspace, size_t workspace_bytes, vpce_stream_t stream);

/*
 * Backward of vpce_lmhead_forward (the pages give none; the standard
 * derivative): with dZ = (softmax(z) - onehot) * g / n_valid ('mean'; g for
 * 'sum'; g_r = grad_rows[r] when grad_rows is given),
 *     grad_hidden         = dZ W              bf16 [s, h], overwritten
 *     grad_weight_shards[i] += dZ_i^T X       fp32 [w_i, h], accumulated
 * The logits are formed again tile by tile on the tensor cores (the forward
 * kept none) and written as bf16 dZ for one chunk of rows at a time into
 * `workspace`; two more tensor-core kernels then form the products (bf16 in,
 * fp32 accumulate): dX with the contraction over all t shards in one
 * accumulator, rounded once to bf16; dW_i added into grad_weight_shards[i]
 * by tile reductions, one add per element per chunk, so the result is the
 * same on every run.  Every argument describing X, the head, the targets and
 * fwd_workspace must be the preceding vpce_lmhead_forward's, unmodified
 * (it carries logsumexp, n_valid and the reduction).
 *   grad_output / grad_rows  as vpce_backward / vpce_backward_rows (grad_rows
 *                   device float[s] or NULL).
 *   grad_hidden     device bf16 [s, h], row stride ld_grad_hidden (0 = h).
 *   grad_weight_shards  host array of t device float pointers, [w_i, h],
 *                   row stride ld_grad_weight (0 = h), 16-byte aligned,
 *                   ld_grad_weight a multiple of 4.
 *   workspace       256-byte aligned; vpce_lmhead_backward_workspace_bytes(V, h)
 *                   bytes give 8192-row chunks (the chunk's bf16 dZ, each
 *                   shard's columns padded to a multiple of 8).  A smaller
 *                   workspace gives smaller chunks, in steps of 128 rows;
 *                   less than 128 rows' worth returns VPCE_ERR_WORKSPACE.
 * Calls launch kernels only (no allocation, no host synchronisation).
 */
size_t vpce_lmhead_backward_workspace_bytes(int64_t V, int64_t h);
vpce_status vpce_lmhead_backward(const void* hidden, int64_t ld_hidden,
                                 const void* const* weight_shards, int64_t ld_weight,
                                 int t, int64_t s, int64_t h, const int64_t* vocab_start,
                                 const int64_t* targets, int64_t ignore_index,
                                 float grad_output, const float* grad_rows,
                                 const void* fwd_workspace, size_t fwd_workspace_bytes,
                                 void* grad_hidden, int64_t ld_grad_hidden,
                                 float* const* grad_weight_shards, int64_t ld_grad_weight,
                                 void* workspace, size_t workspace_bytes, vpce_stream_t stream);

/*
 * vpce_lmhead_forward followed by vpce_lmhead_backward in one call, for a
 * training step whose upstream gradient is known up front (grad_output, or
 * grad_rows per row): loss, dX and dW without forming any logits twice.
 * Per row chunk, the tensor-core kernel writes the loss statistics and keeps
 * the chunk's fp32 logits in the workspace (a chunk is the unit the CMU notes
 * (§5.5) keep resident instead of the whole [s, V] tensor).  A row kernel
 * then forms each row's logsumexp, loss and bf16 dZ from them, and the
 * tensor-core kernels of vpce_lmhead_backward compute dX = dZ W and
 * dW += dZ^T X.
 *   loss_out, row_loss_out, reduction   as vpce_lmhead_forward (the mean
 *                  divides by the batch's n_valid; the loss sum runs over
 *                  fixed 256-row blocks in compensated fp32 pairs, fp64
 *                  across warps).
 *   grad_output, grad_rows, grad_hidden, grad_weight_shards, their strides
 *                  as vpce_lmhead_backward.  VPCE_NONE requires grad_rows.
 *   workspace      256-byte aligned.  With
 *                  vpce_lmhead_forward_backward_workspace_bytes(s, V, h)
 *                  bytes, chunks are min(8192, s rounded up to 128) rows.
 *                  Each chunk holds [R, V] fp32 logits and [R, V] bf16 dZ,
 *                  4.2 GB and 2.1 GB at R = 8192, V = 128256 (rows padded
 *                  per shard).  A smaller workspace gives chunks smaller
 *                  by steps of 128 rows; less than 128 rows' worth returns
 *                  VPCE_ERR_WORKSPACE.  The workspace starts with the loss
 *                  header: vpce_read_error_flag works on it.
 * Other arguments and errors as vpce_lmhead_forward and vpce_lmhead_backward.
 * The results equal those two calls' up to the column grouping of the
 * logsumexp (the same arithmetic on a different split of the columns).
 */
size_t vpce_lmhead_forward_backward_workspace_bytes(int64_t s, int64_t V, int64_t h);
vpce_status vpce_lmhead_forward_backward(const void* hidden, int64_t ld_hidden,
                                         const void* const* weight_shards, int64_t ld_weight,
                                         int t, int64_t s, int64_t h, const int64_t* vocab_start,
                                         const int64_t* targets, int64_t ignore_index,
                                         vpce_reduction reduction, float grad_output,
                                         const float* grad_rows, float* loss_out, float* row_loss_out,
                                         void* grad_hidden, int64_t ld_grad_hidden,
                                         float* const* grad_weight_shards, int64_t ld_grad_weight,
                                         void* workspace, size_t workspace_bytes, vpce_stream_t stream);

/*
 * Vocabulary-parallel input embedding ("Distributed Training III: Model
 * Parallelism", CMU 11-868 Lecture 16 notes, §5.5; "LLM Internals" §7.3.4):
 * the table [V, h] is split by vocabulary into t shards; card i looks up only
 * the ids in its range and writes zeros elsewhere, and an all-reduce sums the
 * cards.  On one GPU the sum has one non-zero term per row, so
 *     out[r] = table_shard_i[ids[r] - vocab_start[i]]  for the shard i holding ids[r],
 *     out[r] = 0                                          for an id outside [0, V).
 *   table_shards  host array of t device pointers, shard i [w_i, h] of dtype,
 *                 row stride ld_table elements (0 = h); element-aligned.
 *   ids           device int64[s].
 *   out           device [s, h] of dtype, row stride ld_out (0 = h).
 *   flag_out      device int or NULL: set to 0, then bit 0
 *                 (VPCE_FLAG_BAD_TARGET) if some id is outside [0, V).
 * Rows whose source and destination are 16-byte aligned (and h * element
 * size a multiple of 16) are copied in 16-byte vectors; others by element.
 */
vpce_status vpce_embedding_forward(const void* const* table_shards, vpce_dtype dtype, int t,
                                   const int64_t* vocab_start, int64_t h, int64_t ld_table,
                                   const int64_t* ids, int64_t s, void* out, int64_t ld_out,
                                   int* flag_out, vpce_stream_t stream);

/*
 * Backward of vpce_embedding_forward (not on the pages; the adjoint of the
 * lookup): adds each output-gradient row into the fp32 gradient-table row of
 * its id, accumulating into what grad_shards already hold:
 *     grad_shard_i[j] += sum over r with ids[r] = vocab_start[i] + j of grad_out[r].
 * Ids outside [0, V) contribute nothing.  Deterministic: the rows of an id
 * with at most 64 rows in a chunk are summed in ascending row order (fp32);
 * an id with more is summed as eight contiguous slices of its rows, each in
 * ascending order, then the slices in order; the sum is then added once.
 * Batches longer than 16384 rows run in 16384-row chunks in order.
 *   grad_out      device [s, h] of grad_dtype, row stride ld_grad (0 = h);
 *                 16-byte aligned, ld_grad * element size a multiple of 16.
 *   grad_shards   host array of t device float pointers, shard i [w_i, h],
 *                 row stride ld_grad_table (0 = h); 16-byte aligned,
 *                 ld_grad_table a multiple of 4.
 *   h             a positive multiple of 4.
 *   workspace     vpce_embedding_backward_workspace_bytes() bytes, 256-byte
 *                 aligned, caller owned.  It starts with the same header as
 *                 the loss workspace: vpce_read_error_flag on it returns
 *                 VPCE_FLAG_WAIT_TIMEOUT if a bounded wait of the kernels gave
 *                 up (the gradient is then incomplete), else 0.
 */
size_t vpce_embedding_backward_workspace_bytes(void);
vpce_status vpce_embedding_backward(const void* grad_out, vpce_dtype grad_dtype, int64_t ld_grad,
                                    const int64_t* ids, int64_t s, float* const* grad_shards, int t,
                                    const int64_t* vocab_start, int64_t h, int64_t ld_grad_table,
                                    void* workspace, size_t workspace_bytes, vpce_stream_t stream);

/*
 * Synchronise `stream`, then copy the workspace error flag to *flag (bit 0:
 * bad target seen by the last forward; bit 1: a device wait timed out, in
 * which case the forward's loss is NaN).
 */
vpce_status vpce_read_error_flag(const void* workspace, int* flag, vpce_stream_t stream);

/* Static, human-readable name of a status code. */
const char* vpce_status_string(vpce_status status);

#ifdef __cplusplus
}
#endif

#endif /* VPCE_H */
