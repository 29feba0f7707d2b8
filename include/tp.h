/*
 * tp.h -- C ABI of the GB300 tensor-parallel sharded projection library (libtp.so).
 *
 * The method (diffusers documentation, "Tensor parallelism" page): every
 * weight matrix of a transformer block is split across tp_degree ranks,
 * either "colwise" (output features, weight dim 0: each rank computes a slice
 * of the output) or "rowwise" (input features, weight dim 1: each rank
 * computes a partial sum).  Fused projections are split block by block.  The
 * slices are joined at the layer boundary: concatenation (AllGather) for
 * colwise, summation (AllReduce) for rowwise.
 *
 * This library runs all tp_degree logical ranks on ONE GPU.  Every rank's
 * shard lives in its own buffer, every rank's GEMM runs inside one kernel
 * launch, and the joins happen in device memory inside the kernels.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Layout: every matrix is row-major and dense unless a leading dimension is
 *   given.  Weights use the nn.Linear layout [out_features, in_features];
 *   activations are [tokens, features].  Elements are bf16 (raw 16-bit
 *   patterns) unless stated; fp32 where stated.
 * - Ownership: the caller allocates and owns every buffer (inputs, outputs and
 *   workspace).  The library allocates no memory and keeps no pointer after a
 *   call returns.
 * - Asynchrony: kernels are enqueued on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream) and the call returns without waiting.  Buffers
 *   must stay valid until the stream reaches that point.
 * - Validation: every argument is checked on the host before anything is
 *   copied or launched; a rejected call has no effect on device memory.  The
 *   plan checks follow the page's §Constraints and verification ("check both
 *   before loading or sharding any weight").
 * - Errors: a call returns a tp_status; TP_OK means the work was enqueued.
 *   tp_last_error() gives a message for the calling thread's last failure.
 *   Nothing falls back silently to another path (§Limitations: unsupported
 *   options raise instead of quietly doing something else).
 * - Device: the current CUDA device of the calling thread.  Requires sm_103a
 *   (GB300) for the GEMM entry points.
 */
#ifndef TP_H_
#define TP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

typedef struct CUstream_st* tp_stream_t; /* same type as cudaStream_t */

typedef enum {
  TP_OK = 0,
  TP_ERR_INVALID_ARG = 1,         /* null pointer, negative size, rank outside [0, tp_degree), ... */
  TP_ERR_HEADS_NOT_DIVISIBLE = 2, /* tp_degree does not divide the attention-head count */
  TP_ERR_SPLIT_NOT_DIVISIBLE = 3, /* a packed block is not divisible by tp_degree on its own */
  TP_ERR_SPLIT_SUM = 4,           /* packed block sizes do not add up to the sharded dimension */
  TP_ERR_NOT_WHOLE_HEADS = 5,     /* a rank's part of a head-structured block is not whole heads */
  TP_ERR_ALIGNMENT = 6,           /* a pointer or row stride the kernels need 16-byte aligned is not */
  TP_ERR_NOT_PINNED = 7,          /* a host source pointer is pageable (not page-locked) memory */
  TP_ERR_WORKSPACE = 8,           /* workspace missing or smaller than tp_rowwise_workspace_bytes() */
  TP_ERR_CUDA = 9,                /* a CUDA runtime call failed (message in tp_last_error) */
  TP_ERR_TIMEOUT = 10,            /* a kernel gave up waiting on an internal barrier (tp_device_status) */
  TP_ERR_UNSUPPORTED = 11,        /* valid plan outside what this build implements (e.g. tp_degree > 16) */
  TP_ERR_IO = 12,                 /* a file could not be opened or read (tp_safetensors.h) */
  TP_ERR_FORMAT = 13,             /* a file is not a well-formed safetensors file (tp_safetensors.h) */
  TP_ERR_NOT_FOUND = 14           /* no tensor of that name in the file (tp_safetensors.h) */
} tp_status;

typedef enum { TP_COLWISE = 0, TP_ROWWISE = 1 } tp_style;
typedef enum { TP_GATHER = 0, TP_REDUCE = 1 } tp_combine_mode;
typedef enum { TP_ACT_NONE = 0, TP_ACT_GELU_TANH = 1, TP_ACT_SWIGLU = 2 } tp_act;
/* Flag OR'd into tp_linear_colwise's act argument: chunked fp32 accumulation (see there). */
#define TP_ACCUM_CHUNKED 0x100
typedef enum {
  TP_REDUCE_NONE = 0,      /* write every rank's fp32 partial; join later with tp_combine(TP_REDUCE) */
  TP_REDUCE_WORKSPACE = 1, /* fp32 partials to a workspace, summed in the GEMM epilogue by the ranks */
  TP_REDUCE_ACCUM = 2      /* each tile's ranks accumulate in turn into one fp32 on-chip accumulator */
} tp_reduce_mode;

#define TP_MAX_DEGREE 16 /* largest tp_degree the GEMM entry points accept */
#define TP_MAX_SPLITS 16 /* largest number of packed blocks in one weight */

/* ------------------------------------------------------------------------ */
/* Plan                                                                      */
/* ------------------------------------------------------------------------ */

/*
 * tp_validate -- check a sharding plan for one weight [rows, cols].
 *
 * "Tensor parallelism" page: §Load a sharded model (tp_degree must divide the
 * number of attention heads), §Fused projections (packed blocks, absolute
 * sizes as stored in _tp_packed_col_blocks / _tp_packed_row_blocks) and
 * §Constraints and verification (every packed block divisible by tp_degree
 * on its own).  Checks, in order:
 *   1. TP_ERR_INVALID_ARG: tp_degree >= 1, rows/cols/num_heads/head_dim >= 0,
 *      style valid, 0 <= n_splits <= TP_MAX_SPLITS, fused_splits non-NULL when
 *      n_splits > 0, every split > 0.
 *   2. TP_ERR_HEADS_NOT_DIVISIBLE: num_heads > 0 and num_heads % tp_degree != 0.
 *   3. TP_ERR_SPLIT_SUM: the splits do not add up to the sharded dimension
 *      (rows for TP_COLWISE, cols for TP_ROWWISE).
 *   4. TP_ERR_SPLIT_NOT_DIVISIBLE: some split % tp_degree != 0.
 *   5. TP_ERR_NOT_WHOLE_HEADS: head_dim > 0 and some (split / tp_degree) %
 *      head_dim != 0 (the sharded dimension is made of heads of head_dim).
 * fused_splits: host array of n_splits absolute block sizes along the sharded
 * dimension, in packed order; NULL/0 means one block (a plain split).
 * Pure host function; touches no device.
 */
TP_API tp_status tp_validate(int64_t rows, int64_t cols, tp_style style, int tp_degree, int64_t num_heads,
                      int64_t head_dim, const int64_t* fused_splits, int n_splits);

/*
 * tp_shard_shape -- shape of every rank's dense shard after tp_validate's
 * checks 1, 3 and 4: [rows / tp_degree, cols] for TP_COLWISE, [rows, cols /
 * tp_degree] for TP_ROWWISE.  out_rows/out_cols: host pointers, written on
 * TP_OK only.  Pure host function.
 */
TP_API tp_status tp_shard_shape(int64_t rows, int64_t cols, tp_style style, int tp_degree,
                         const int64_t* fused_splits, int n_splits, int64_t* out_rows, int64_t* out_cols);

/* ------------------------------------------------------------------------ */
/* Shard extraction                                                          */
/* ------------------------------------------------------------------------ */

/*
 * tp_plan_shard -- copy rank `rank`'s slice of a bf16 weight into a dense
 * device buffer.
 *
 * "Tensor parallelism" page, §Load a sharded model: each rank reads only its
 * own slice of every weight and places it directly on its device, so no
 * full-size weight is ever staged there; §Limitations: enable_parallelism()
 * shards a model already in memory.  Both are this call: `weight` may be
 * page-locked host memory (the slice is read over the CPU-GPU link straight
 * into `dev_out` by the copy engines, one transfer per packed block -- a
 * column window of every row for TP_ROWWISE -- so no SM is taken from kernels
 * running beside the load; nothing else reaches the device) or device memory
 * (a device-to-device copy kernel).  Pageable host memory is rejected with
 * TP_ERR_NOT_PINNED.
 *
 * Slice definition (§Colwise and rowwise, §Fused projections): with packed
 * blocks of sizes s_0..s_{n-1} at offsets o_b along the sharded dimension,
 * block b contributes [o_b + rank*s_b/p, o_b + (rank+1)*s_b/p) and the parts
 * are concatenated in block order.  TP_COLWISE slices rows, TP_ROWWISE slices
 * columns.  A fused QKV weight with splits {H,H,H} thus gives rank r the rows
 * [Q_r; K_r; V_r] of whole heads; a gate/up weight with {F,F} gives
 * [gate_r; up_r].
 *
 * weight:  bf16 [rows, cols] row-major (host page-locked or device).
 * dev_out: device buffer of tp_shard_shape() elements, dense row-major.
 * num_heads/head_dim: as in tp_validate (0 to skip those checks).
 * The copy is bit-exact (any 16-bit pattern, NaN payloads included).
 * Errors: everything tp_validate returns, TP_ERR_INVALID_ARG for NULL
 * pointers with a non-empty shard or a dev_out that is not device memory,
 * TP_ERR_NOT_PINNED, TP_ERR_CUDA.
 */
TP_API tp_status tp_plan_shard(const void* weight, int64_t rows, int64_t cols, tp_style style, int tp_degree, int rank,
                        const int64_t* fused_splits, int n_splits, int64_t num_heads, int64_t head_dim,
                        void* dev_out, tp_stream_t stream);

/*
 * tp_plan_shard_ranks -- tp_plan_shard for ranks [rank_begin, rank_begin +
 * rank_count) in one launch: dev_outs is a host array of rank_count device
 * buffers, dev_outs[i] receiving rank (rank_begin + i)'s shard.  Same slice
 * definition, checks, sources and errors as tp_plan_shard; the range must lie
 * in [0, tp_degree).  rank_count == 0 validates the plan and copies nothing.
 * This is how one process that plays every rank loads all their shards.
 */
TP_API tp_status tp_plan_shard_ranks(const void* weight, int64_t rows, int64_t cols, tp_style style, int tp_degree,
                                     int rank_begin, int rank_count, const int64_t* fused_splits, int n_splits,
                                     int64_t num_heads, int64_t head_dim, void* const* dev_outs, tp_stream_t stream);

/*
 * tp_plan_shard_many -- several extractions (e.g. every weight of a block) in
 * as few launches as possible: every request is a tp_plan_shard_ranks call,
 * with the same slice definition, checks and errors.  All requests are
 * checked before anything is copied; a refused request leaves every output
 * untouched and the error message names the request's index.  Requests from
 * device memory share one copy-kernel launch (more only beyond 64 copy
 * segments: one per packed block per rank); requests from page-locked host
 * memory are one copy-engine transfer per segment.  1 <= n_requests <= TP_MAX_SHARD_REQUESTS (0 is a no-op);
 * `requests` and the arrays it points to are read during the call only.
 */
#define TP_MAX_SHARD_REQUESTS 64
typedef struct {
  const void* weight;           /* bf16 [rows, cols] row-major: page-locked host or device memory */
  int64_t rows, cols;
  tp_style style;
  int tp_degree;
  int rank_begin, rank_count;   /* ranks [rank_begin, rank_begin + rank_count) */
  const int64_t* fused_splits;  /* NULL, or n_splits absolute packed block sizes */
  int n_splits;
  int64_t num_heads, head_dim;  /* as in tp_validate (0 skips the check) */
  void* const* dev_outs;        /* host array of rank_count device buffers */
} tp_shard_request;
TP_API tp_status tp_plan_shard_many(const tp_shard_request* requests, int n_requests, tp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Sharded projections                                                       */
/* ------------------------------------------------------------------------ */

/*
 * tp_linear_colwise -- every rank's colwise projection in one launch:
 *     Y_r = act(X . W_r^T + b_r)      for r = 0 .. tp_degree-1
 *
 * "Tensor parallelism" page, §Colwise and rowwise: the input X is replicated
 * and each rank computes its slice of the output features; the output stays
 * sharded for the rowwise projection that follows.
 *
 * x:           device bf16 [T, K] (shared by every rank).
 * w_shards:    host array of tp_degree device pointers, each bf16 [N_r, K]
 *              (the dense shards tp_plan_shard writes).
 * bias_shards: NULL, or host array of tp_degree device pointers (each NULL or
 *              bf16 [N_r], sharded like the weight's rows).
 * act:         TP_ACT_NONE / TP_ACT_GELU_TANH (0.5x(1+tanh(sqrt(2/pi)(x+0.044715x^3))))
 *              / TP_ACT_SWIGLU (the shard is [gate_r; up_r], N_r even, and
 *              Y_r = silu(gate) * up has N_r/2 columns).  The activation is
 *              applied to the fp32 accumulator before rounding to bf16.
 * y_shards:    host array of tp_degree device pointers, each bf16 [T, N_out]
 *              with row stride ldy elements (N_out = N_r, or N_r/2 for SwiGLU).
 *              ldy = 0 means N_out (dense).  Passing y_shards[r] = Y + r*N_out
 *              with ldy = tp_degree*N_out writes the gathered (AllGather)
 *              output [T, tp_degree*N_out] directly.
 * Accumulation is fp32; outputs are rounded to nearest-even bf16.
 * act | TP_ACCUM_CHUNKED (TP_ACT_NONE only; TP_ERR_UNSUPPORTED otherwise):
 *              the tensor core adds each step of 16 products into its fp32
 *              accumulator without rounding to nearest, so a long K sum drifts:
 *              over K = 6144 about 0.35 % of the bf16 outputs round to the
 *              other neighbour of the exact value (0.02 % for a sum rounded to
 *              nearest at every step).  With this flag the products are summed
 *              on the tensor core in chunks of K = 1024, each from zero, and
 *              the chunks are added in fp32 with round-to-nearest by the
 *              epilogue, which brings it to about 0.07 %.  Use it where the
 *              output feeds a step that amplifies one-ulp differences -- the
 *              Q, K and V of attention, whose softmax turns a rounding flip in
 *              a key into a change of every query's weights.  It costs about
 *              9 % of the projection's time (8 epilogue warps keep the running
 *              sums in registers; the accumulator is handed to them once per
 *              chunk instead of once per tile).
 * Alignment (TP_ERR_ALIGNMENT): K % 8 == 0, N_out % 8 == 0, ldy % 8 == 0 and
 * every pointer 16-byte aligned.  tp_degree <= TP_MAX_DEGREE.
 * T == 0 or N_r == 0 enqueues nothing and returns TP_OK.
 */
TP_API tp_status tp_linear_colwise(const void* x, const void* const* w_shards, const void* const* bias_shards, tp_act act,
                            int tp_degree, int64_t T, int64_t K, int64_t N_r, void* const* y_shards, int64_t ldy,
                            tp_stream_t stream);

/*
 * tp_linear_rowwise -- every rank's rowwise projection and the sum of the
 * partials in one launch:
 *     P_r = X_r . W_r^T ,  Z = sum_r P_r (+ bias, once)
 *
 * "Tensor parallelism" page, §Colwise and rowwise: each rank computes a
 * partial sum from its slice of the input features, and one AllReduce at the
 * block boundary (after the colwise -> rowwise pair) rebuilds the result.
 * The partials are summed in rank order, in fp32.
 *
 * x_shards: host array of tp_degree device pointers, each bf16 [T, K_r]
 *           (rank r's slice of the input features, e.g. the colwise output).
 * w_shards: host array of tp_degree device pointers, each bf16 [N, K_r].
 * bias:     NULL or device bf16 [N]; added once, after the sum.
 * mode:
 *   TP_REDUCE_ACCUM: for each output tile, rank 0's, then rank 1's, ...
 *     products accumulate into one fp32 tensor-memory accumulator; out is
 *     bf16 [T, N].  No workspace (ws_bytes may be 0).
 *   TP_REDUCE_WORKSPACE: each rank's fp32 partial tile goes to `workspace`
 *     and is counted on a per-tile atomic counter; when all tp_degree partials
 *     of a tile are in (a bounded wait; the launch is cooperative so the ranks'
 *     CTAs are resident together), each rank sums its 1/tp_degree share of the
 *     tile's rows in rank order and writes bf16 [T, N] to out.  Needs
 *     ws_bytes >= tp_rowwise_workspace_bytes(...).  The counters are cleared on
 *     `stream` by the call itself.
 *   TP_REDUCE_NONE: out is fp32 [tp_degree][T][N], rank r's partial (the bias,
 *     if any, is added to rank 0's partial only); join with tp_combine.
 * Alignment (TP_ERR_ALIGNMENT): K_r % 8 == 0, N % 8 == 0, pointers 16-byte
 * aligned.  tp_degree <= TP_MAX_DEGREE.  T == 0 or N == 0 enqueues nothing.
 * Calls that share a workspace must not overlap on the GPU.
 */
TP_API tp_status tp_linear_rowwise(const void* const* x_shards, const void* const* w_shards, const void* bias, int tp_degree,
                            int64_t T, int64_t K_r, int64_t N, tp_reduce_mode mode, void* workspace, size_t ws_bytes,
                            void* out, tp_stream_t stream);

/*
 * tp_linear_rowwise_split_input -- the "rowwise_split_input" style: a rowwise
 * projection whose input is replicated on every rank, each rank computing its
 * partial from its own slice of that input.
 *
 * "Tensor parallelism" page, §Colwise and rowwise table: "rowwise_split_input"
 * shards the input features (weight dim 1) and each rank computes a partial
 * result from its slice of the replicated input and its weights; the sum
 * gives every rank all output features (for a standalone projection reading a
 * replicated activation, e.g. an AdaLN modulation projection).
 *     Z = sum_r X[:, r*K/p : (r+1)*K/p] . W_r^T (+ bias, once)
 *
 * x: device bf16 [T, K] with row stride ldx elements (0 = K); rank r reads
 *    columns [r*K/p, (r+1)*K/p) in place (no copy).
 * w_shards: host array of tp_degree device pointers, each bf16 [N, K/p] (the
 *    plain rowwise shards).  bias, mode, workspace, out: as tp_linear_rowwise.
 * Errors: TP_ERR_SPLIT_NOT_DIVISIBLE if tp_degree does not divide K; the
 * alignment rules of tp_linear_rowwise with K/p and ldx multiples of 8.
 */
TP_API tp_status tp_linear_rowwise_split_input(const void* x, int64_t ldx, const void* const* w_shards,
                                               const void* bias, int tp_degree, int64_t T, int64_t K, int64_t N,
                                               tp_reduce_mode mode, void* workspace, size_t ws_bytes, void* out,
                                               tp_stream_t stream);

/* Bytes of device workspace tp_linear_rowwise needs for `mode` (0 unless TP_REDUCE_WORKSPACE). */
TP_API size_t tp_rowwise_workspace_bytes(int tp_degree, int64_t T, int64_t N, tp_reduce_mode mode);

/* Size of the library's built-in scratch array used by tp_linear_rowwise_noalloc (64 MiB per GPU). */
#define TP_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * tp_linear_rowwise_noalloc -- tp_linear_rowwise in TP_REDUCE_WORKSPACE mode,
 * for callers that cannot allocate device memory.  The pages have no
 * counterpart of this call; it exists for the host program, not the method.
 *
 * Who needs it: code that runs where allocating is not allowed or not
 * possible -- for instance a plug-in called by a framework that owns all
 * device memory and hands out none, or a process whose memory was claimed up
 * front by a pool so that a new cudaMalloc would fail (cudaMalloc can also
 * stall the whole device, which latency-bound callers must avoid).  Such a
 * caller still passes its inputs and output; the fp32 partials and tile
 * counters live in one fixed array compiled into this library
 * (TP_NOALLOC_SCRATCH_BYTES of device memory, held by every GPU that loads the
 * library until the process exits).
 *
 * Arguments, layout, result and numerics are those of tp_linear_rowwise with
 * mode TP_REDUCE_WORKSPACE: x_shards/w_shards are host arrays of tp_degree
 * device pointers (bf16 [T, K_r] and [N, K_r]), bias is NULL or bf16 [N]
 * (added once), out is bf16 [T, N].
 * Limits: the call is refused with TP_ERR_WORKSPACE, before any device work,
 * when tp_rowwise_workspace_bytes(tp_degree, T, N, TP_REDUCE_WORKSPACE)
 * exceeds TP_NOALLOC_SCRATCH_BYTES (roughly tp_degree * T * N <= 16M).
 * When the memory is claimed: the array belongs to the library's GEMM
 * module, and the CUDA driver claims its device memory when it loads that
 * module on a device -- with lazy module loading (the default) at the first
 * call on that device that launches one of the library's GEMMs or looks the
 * array up (this call).  A caller whose memory pool will claim the device's
 * free memory should make one call of this entry point on each device (any
 * small problem, e.g. T = 1) before the pool does; from then on no call
 * claims memory.
 * The first call on a device (and the first in a new CUDA context, e.g.
 * after cudaDeviceReset) looks up the array's device address with that
 * device current; make that first call before any stream capture.  No
 * allocation happens in this call or the ones it makes.
 * Every call uses the same array and it keeps the last call's contents; the
 * call clears the tile counters itself.  Calls whose kernels overlap on the
 * GPU (other streams, other threads) race on the array: serialise them.
 */
TP_API tp_status tp_linear_rowwise_noalloc(const void* const* x_shards, const void* const* w_shards, const void* bias,
                                           int tp_degree, int64_t T, int64_t K_r, int64_t N, void* out,
                                           tp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Attention over a rank's local heads                                       */
/* ------------------------------------------------------------------------ */

/*
 * tp_attention_heads -- attention of one rank over its local heads:
 *     O_h = softmax(Q_h K_h^T / sqrt(head_dim)) V_h     for h < n_heads
 *
 * "Tensor parallelism" page, §Colwise and rowwise: the colwise Q, K and V
 * projections give each rank a subset of heads (tp_degree divides the head
 * count), so the rank attends over them alone and its output feeds its
 * rowwise out-projection directly.  No mask, no positional embedding; head h
 * occupies columns [h*head_dim, (h+1)*head_dim) of each of Q, K and V.
 *
 * qkv:  device bf16 [T, 3*n_heads*head_dim] with row stride ld_qkv elements
 *       (0 = dense): Q, then K, then V -- the rank's colwise QKV output.
 * out:  device bf16 [T, n_heads*head_dim] with row stride ldo (0 = dense).
 * workspace: device buffer of tp_attention_workspace_bytes(T, n_heads,
 *       head_dim) bytes, owned by the caller; none (NULL, 0) at head_dim 64 and
 *       128, where the fused kernel reads Q, K and V in place; for other head
 *       sizes V^T (each group of 8 keys twice) and the fp32 scores of up to
 *       16 heads at a time.
 * Scores and softmax are fp32; the probabilities enter the P.V product (fp32
 * accumulation) as two bf16 terms, P_hi (P truncated to bf16 in the fused
 * kernel of head_dim 64 and 128, rounded elsewhere) and P_lo = bf16(P - P_hi), which
 * carry P to about 2^-16 relative (one bf16 term would carry 2^-9, an error
 * that the block's later bf16 roundings amplify); O is rounded to bf16.
 * Alignment (TP_ERR_ALIGNMENT): T, head_dim, ld_qkv, ldo multiples of 8, pointers
 * 16-byte aligned.  T == 0 enqueues nothing.  TP_ERR_WORKSPACE if too small.
 */
TP_API tp_status tp_attention_heads(const void* qkv, int64_t ld_qkv, int64_t T, int n_heads, int head_dim,
                                    void* workspace, size_t ws_bytes, void* out, int64_t ldo, tp_stream_t stream);

/* Bytes of device workspace tp_attention_heads needs (0 at head_dim 64 and 128). */
TP_API size_t tp_attention_workspace_bytes(int64_t T, int n_heads, int head_dim);

/*
 * tp_attention_heads_ranks -- tp_attention_heads for n_ranks ranks in one
 * call: qkv[r] and out[r] (host arrays of n_ranks device pointers) are rank
 * r's QKV output and attention output, every rank with the same T, n_heads,
 * head_dim, ld_qkv and ldo.  With head_dim 64 or 128 one kernel launch covers every
 * rank's heads, so a small per-rank head count still fills the GPU, and no
 * workspace is needed; other head sizes run the ranks one after another
 * through the same workspace.  Same arithmetic, checks and errors as
 * tp_attention_heads; 1 <= n_ranks <= TP_MAX_DEGREE (TP_ERR_UNSUPPORTED above).
 * workspace: tp_attention_ranks_workspace_bytes(n_ranks, T, n_heads, head_dim).
 */
TP_API tp_status tp_attention_heads_ranks(int n_ranks, const void* const* qkv, int64_t ld_qkv, int64_t T, int n_heads,
                                          int head_dim, void* workspace, size_t ws_bytes, void* const* out,
                                          int64_t ldo, tp_stream_t stream);

/* Bytes of device workspace tp_attention_heads_ranks needs (0 at head_dim 64 and 128, and for an empty or
 * invalid call). */
TP_API size_t tp_attention_ranks_workspace_bytes(int n_ranks, int64_t T, int n_heads, int head_dim);

/* ------------------------------------------------------------------------ */
/* Join                                                                      */
/* ------------------------------------------------------------------------ */

/*
 * tp_combine -- join per-rank results in device memory (the page's opening
 * paragraph: "an AllReduce or AllGather at the layer boundary").
 *   TP_GATHER: partials[r] is bf16 [T, N_each]; out is bf16 [T, tp_degree*N_each]
 *              with columns [r*N_each, (r+1)*N_each) taken from rank r.  Bit-exact.
 *   TP_REDUCE: partials[r] is fp32 [T, N_each]; out is bf16 [T, N_each] =
 *              round_nearest_even(sum_r partials[r]), summed in rank order in fp32.
 * partials: host array of tp_degree device pointers.  out: device buffer.
 * Any alignment is accepted (16-byte aligned rows take the vector path).
 */
TP_API tp_status tp_combine(tp_combine_mode mode, const void* const* partials, int tp_degree, int64_t T, int64_t N_each,
                     void* out, tp_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                               */
/* ------------------------------------------------------------------------ */

/* Message for the calling thread's last failed call ("" if none).  Valid until the thread's next call. */
TP_API const char* tp_last_error(void);

/* Name of a status code ("TP_OK", "TP_ERR_ALIGNMENT", ...). */
TP_API const char* tp_status_name(tp_status status);

/*
 * tp_device_status -- synchronise `stream`, then report whether any kernel of
 * this library on the current device gave up on an internal wait (every wait
 * is bounded; a kernel that gives up records it and exits cleanly).  Returns
 * TP_ERR_TIMEOUT and clears the record if so, TP_ERR_CUDA if the stream
 * reported an error, TP_OK otherwise.
 */
TP_API tp_status tp_device_status(tp_stream_t stream);

/*
 * tp_set_tile_wait_limit_ns -- how long a CTA of a TP_REDUCE_WORKSPACE call
 * waits for the other ranks' partials of its output tile (the one wait of the
 * library on other CTAs) before it gives up: it then records TP_ERR_TIMEOUT
 * for tp_device_status, skips its share of the tile's sums, drains its copies
 * and MMAs and exits.  The output of such a call is not valid.  0 restores
 * the default of 2 s.  The value is read when a call enqueues its kernel, so
 * it applies to calls made after this one (and a captured CUDA graph keeps the
 * value of its capture).  Process-wide; the waits of a CTA on its own copies
 * and MMAs keep a fixed bound of 2 s.  Exists so that the give-up path can be
 * exercised: a budget far below the time the ranks of a tile take to arrive
 * makes the wait run out without any fault.
 */
TP_API void tp_set_tile_wait_limit_ns(uint64_t ns);

/* The current tile-wait bound in nanoseconds (see tp_set_tile_wait_limit_ns). */
TP_API uint64_t tp_tile_wait_limit_ns(void);

/* Library ABI version (major * 100 + minor). */
TP_API int tp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TP_H_ */
