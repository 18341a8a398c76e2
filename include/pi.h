/*
 * pi.h — C ABI of the activation-sparse decode FFN library (libpi.so).
 *
 * The library implements the online part of the method described on the
 * page "PowerInfer: Quick Massive Language Mannequin Serving with a
 * Client-grade GPU": a predictor scores every FFN neuron, the neurons
 * predicted inactive are skipped ("Online Section"), and neuron-aware
 * operators compute only the rows of the up projection and the column
 * vectors of the down projection that belong to activated neurons, directly
 * on the stored matrices ("Neuron Conscious Operator").  Neurons are stored
 * hot-first (most frequently active first, "Offline Section"), so the
 * hot block is a contiguous prefix; neuron indices are positions in the
 * stored matrices ("Neuron Placement and Administration").  Everything runs
 * on one GPU; there is no CPU executor and no CPU fallback.
 *
 * Conventions for every call
 * --------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library never allocates, frees or copies to the host on these calls.
 *  - Calls are asynchronous on the caller's stream (NULL = legacy default
 *    stream); they never synchronise the host.  Counts stay on the device,
 *    so a sequence of calls can be captured in a CUDA graph.
 *  - Layouts are row-major with one row per neuron:
 *      A   [n][r]      predictor factor   (dtype)
 *      Bm  [r][d]      predictor factor   (dtype)
 *      b1  [n]         fp32 bias of the predictor and of the up projection
 *                      (gated: of the gate)
 *      W1  [n][d]      up projection, or gated [n][2][d]: per neuron the
 *                      gate row followed by the up row        (dtype)
 *      W2  [n][d]      down projection, one row per neuron   (dtype)
 *      (or both in one per-neuron record: see pi_layout)
 *      b2  [d]         fp32 output bias, may be NULL (= 0)
 *      x   [batch][d]  fp32 activations;  y [batch][d] fp32 outputs
 *  - Alignment: every pointer passed must be 16-byte aligned.
 *  - Sizes: d % 8 == 0 and 8 <= d <= 8192; r % 8 == 0 and 8 <= r <= 256;
 *    1 <= n <= 1 << 24; 1 <= batch <= 32 (sparse / fused paths: see each
 *    call).
 *  - Workspace: `ws` is caller-owned device scratch of at least
 *    pi_workspace_size(desc, batch) bytes.  It must be zero-filled before
 *    its first use; afterwards the library leaves it ready for the next
 *    call.  One workspace serves one stream at a time (calls that overlap
 *    on the GPU must use different workspaces).  After PI_ERR_TIMEOUT it
 *    must be zero-filled again.
 *  - Errors come on two channels.  Host-detected errors (NULL pointer, bad
 *    size or dtype, misalignment, small workspace, grid that cannot be
 *    co-resident, failed launch) are returned before or at launch; nothing
 *    has been launched when the status is not PI_OK, except for PI_ERR_CUDA
 *    raised by the launch itself.  Device-detected errors (capacity
 *    exceeded, an index out of range, a bounded wait that ran out) are
 *    written to *dev_status
 *    (an int32 in device memory the caller zeroes; the first error wins)
 *    and can be read after the caller synchronises its stream.
 */
#ifndef PI_H
#define PI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* pi_stream;

typedef enum {
  PI_OK = 0,
  PI_ERR_NULL = 1,       /* a required pointer is NULL                         */
  PI_ERR_SHAPE = 2,      /* a size or the batch is outside the supported range */
  PI_ERR_DTYPE = 3,      /* dtype is not PI_F16 / PI_BF16                      */
  PI_ERR_ALIGN = 4,      /* a pointer is not 16-byte aligned                   */
  PI_ERR_WORKSPACE = 5,  /* ws_bytes < pi_workspace_size(desc, batch)          */
  PI_ERR_CAPACITY = 6,   /* device: more active neurons than the list holds    */
  PI_ERR_LAUNCH = 7,     /* the persistent grid cannot be co-resident          */
  PI_ERR_TIMEOUT = 8,    /* device: a bounded grid-wide wait ran out           */
  PI_ERR_CUDA = 9,       /* a CUDA runtime call failed                         */
  PI_ERR_INDEX = 10,     /* device: an active-list entry is outside [0, n)     */
  PI_ERR_RANGE = 11,     /* device: a predictor partial sum exceeds the range
                            of the fixed-point exchange (|value| >= 2^23)      */
  PI_ERR_CAPTURE = 12    /* a call's one-time setup was asked for while its
                            stream was being captured into a CUDA graph        */
} pi_status;

typedef enum { PI_F16 = 0, PI_BF16 = 1 } pi_dtype;

/* Storage of the FFN weights.
 *  PI_LAYOUT_SPLIT : W1 [n][d] (gated [n][2][d]) and W2 [n][d], two matrices.
 *  PI_LAYOUT_PACKED: one record per neuron, W1 [n][m d] with m = 2 (plain:
 *                    up row, down row) or m = 3 (gated: gate, up, down rows);
 *                    W2 must be NULL.  The same bytes, so the same results;
 *                    a neuron's rows then arrive in one bulk copy.  Build it
 *                    with pi_pack_weights.                                   */
typedef enum { PI_LAYOUT_SPLIT = 0, PI_LAYOUT_PACKED = 1 } pi_layout;

/* Shape of one FFN layer. */
typedef struct {
  int32_t d;           /* model (hidden) dimension                              */
  int32_t n;           /* FFN neurons                                           */
  int32_t r;           /* predictor rank                                        */
  int32_t dtype;       /* pi_dtype of A, Bm, W1, W2                             */
  int32_t gated;       /* 0: h = ReLU(W1 x + b1); 1: h = ReLU(Wg x + b1)(Wu x)  */
  int32_t hot_prefix;  /* neurons [0, hot_prefix) form the hot block: their
                          rows are fetched towards the chip before the mask is
                          known (0 = off).  Never changes results.             */
  int32_t layout;      /* pi_layout of W1 / W2                                  */
} pi_ffn_desc;

/* Device pointers of one layer's weights (layouts above). */
typedef struct {
  const void* A;
  const void* Bm;
  const float* b1;
  const void* W1;  /* PI_LAYOUT_PACKED: the per-neuron records */
  const void* W2;  /* PI_LAYOUT_PACKED: NULL                   */
  const float* b2; /* may be NULL */
} pi_layer_weights;

/* Bytes of workspace the calls below need for this shape and batch.
 * Returns 0 for an invalid descriptor or batch.  Host-only; no CUDA call. */
size_t pi_workspace_size(const pi_ffn_desc* desc, int32_t batch);

/* Predictor ("Adaptive Sparsity Predictors": the engine predicts which
 * neurons will activate before computing the FFN; the predictor lives in
 * GPU memory).  For each token t < batch:
 *     u      = Bm x[t]                    (fp32 accumulate, kept fp32)
 *     logits[t][i] = A_i . u + b1_i       (fp32)
 * logits is [batch][n] fp32.  batch <= 32. */
pi_status pi_predict(const pi_ffn_desc* desc, const void* A, const void* Bm,
                     const float* b1, const float* x, int32_t batch,
                     float* logits, void* ws, size_t ws_bytes,
                     pi_stream stream);

/* Compaction of the predicted mask into the active-neuron list ("Online
 * Section": non-activated neurons are skipped; the list plays the part of
 * the GPU-side neuron table).  For each token t:
 *     idx[t][0 .. cnt[t]) = ascending { i : logits[t][i] > 0 }   (strict)
 * idx is [batch][cap] int32, cnt is [batch] int32.  If cnt[t] > cap only the
 * first cap entries are written, cnt[t] still holds the full count, and
 * PI_ERR_CAPACITY is written to *dev_status.
 * If union_idx is not NULL (batched decode) also:
 *     union_idx[0 .. *union_cnt) = ascending { i : some token active }
 *     tok_mask[k] bit t set iff token t is active at neuron union_idx[k]
 * (capacity n for both; batch <= 32).  dev_status may be NULL only when no
 * capacity error can occur (cap >= n).  ws: with a workspace of
 * pi_workspace_size bytes (any descriptor with this n) the compaction runs
 * over the whole grid, using the workspace's last region for its counts;
 * with ws == NULL (or too small) it runs one block per token and one for
 * the union (slower for large batches; same results). */
pi_status pi_compact(const float* logits, int32_t n, int32_t batch,
                     int32_t* idx, int32_t* cnt, int32_t cap,
                     int32_t* union_idx, int32_t* union_cnt,
                     uint32_t* tok_mask, int32_t* dev_status, void* ws,
                     size_t ws_bytes, pi_stream stream);

/* Neuron-aware sparse FFN ("Neuron Conscious Operator": only the activated
 * neurons' row vectors of W1 and column vectors of W2 are touched, with no
 * conversion to a dense or sparse format).  batch == 1:
 *     h_k = ReLU(W1[idx[k]] . x + b1[idx[k]])
 *           (gated: ReLU(Wg[idx[k]] . x + b1[idx[k]]) * (Wu[idx[k]] . x))
 *     y   = b2 + sum_{k < cnt[0]} h_k W2[idx[k]]
 * with fp32 accumulation and a fixed-order (deterministic) split reduction.
 * idx / cnt are device arrays (e.g. from pi_compact); cnt[0] must be <= cap
 * (else PI_ERR_CAPACITY on *dev_status and nothing is computed).  An entry
 * outside [0, n) is not read: it contributes nothing and PI_ERR_INDEX is
 * written to *dev_status.
 * batch > 1: the union form; union_idx / union_cnt / tok_mask as written by
 * pi_compact, and token t uses exactly the union neurons whose mask bit t is
 * set, so y[t] equals the batch-1 result for token t (idx, cnt and cap are
 * then unused; dev_status, if not NULL, receives PI_ERR_TIMEOUT should a
 * bounded wait of the tensor-core phase run out).  The union's rows are
 * read once and contracted with all tokens on the tensor cores (16-bit
 * operands with a high/low split of x and h, fp32 accumulation; the
 * environment variable PI_BATCH_TC=1 selects a tcgen05 up projection with
 * its accumulator in tensor memory); needs d % 128 == 0. */
pi_status pi_sparse_ffn(const pi_ffn_desc* desc, const pi_layer_weights* w,
                        const float* x, int32_t batch, const int32_t* idx,
                        const int32_t* cnt, int32_t cap,
                        const int32_t* union_idx, const int32_t* union_cnt,
                        const uint32_t* tok_mask, float* y,
                        int32_t* dev_status, void* ws, size_t ws_bytes,
                        pi_stream stream);

/* Dense FFN over all n neurons, the comparison point of the sparse path.
 * No passage of the method's pages defines it: this call is the baseline
 * that the sparse calls are measured against (every row read, no
 * predictor):
 *     y[t] = b2 + sum_i ReLU(W1_i . x[t] + b1_i) W2_i   (gated as above).
 * batch <= 32.  batch > 1 with d % 128 == 0 reads every row once for all
 * tokens on the tensor cores: tcgen05 MMAs with accumulators in tensor
 * memory and operands staged by TMA where n % 64 == 0 and a block of the
 * 1-per-SM grid holds at most 256 rows (PI_BATCH_LEGACY=1 in the environment
 * keeps the mma.sync phases instead), the mma.sync phases of the batched
 * sparse path over all n neurons otherwise; batch 1, or d % 128 != 0: one
 * persistent CUDA-core launch per token. */
pi_status pi_dense_ffn(const pi_ffn_desc* desc, const pi_layer_weights* w,
                       const float* x, int32_t batch, float* y, void* ws,
                       size_t ws_bytes, pi_stream stream);

/* One decode step of one layer: predictor, compaction and sparse FFN
 * ("Online Section" end to end).  batch == 1 runs as one persistent launch
 * whose grid-wide waits are bounded (PI_ERR_TIMEOUT on *dev_status if one
 * runs out).  batch > 1 (with d % 128 == 0) runs the batched predictor,
 * the per-token compaction and their union, and the batched sparse FFN on
 * the tensor cores; otherwise one batch-1 step per token.
 *     y[t] = (residual ? residual[t] : 0) + FFN_sparse(x[t])
 * residual may be NULL; pass residual = x for a residual stack.  idx_out
 * ([batch][n]) and cnt_out ([batch]) may be NULL; when given they receive
 * each token's ascending active list and count (for batch 1 and for
 * batches that run token by token these two need only 4-byte alignment;
 * the batched union path needs 16).  dev_status must not be NULL. */
pi_status pi_layer_decode(const pi_ffn_desc* desc, const pi_layer_weights* w,
                          const float* x, int32_t batch, float* y,
                          const float* residual, int32_t* idx_out,
                          int32_t* cnt_out, int32_t* dev_status, void* ws,
                          size_t ws_bytes, pi_stream stream);

/* Batch-1 decode through a sequence of J layer steps in one persistent
 * launch: the same per-layer computation as pi_layer_decode ("Online
 * Section", "Neuron Conscious Operator"), with each step's weights that do
 * not depend on its input (hot rows, predictor rows) fetched while the
 * previous step finishes; a step's input is read only after the previous
 * step is complete.
 *   descs / layers: host arrays of R (1 <= R <= 128) layers with one shape
 *     (d, n, dtype, gated, layout equal); hot_prefix and the predictor rank
 *     r may differ per layer (each layer's predictor sized by that layer's
 *     skewness and sparsity: "PowerInfer: Quick Massive Language Mannequin
 *     Serving with a Client-grade GPU", section "Adaptive Sparsity
 *     Predictors"); step j uses layer j % R.
 *   chain = 1: a residual stack, x_0 = x [d], x_{j+1} = x_j + FFN_j(x_j),
 *     y[j] = x_{j+1};  chain = 0: independent steps, x [J][d] (one input
 *     per step), y[j] = FFN_j(x[j]).  y: [J][d] fp32.
 *   cnt_out: NULL or [J], active neurons of each step; mask_out: NULL or
 *     [J][n] bytes, 1 where the neuron was predicted active.
 *   ws: pi_workspace_size(desc, 1) bytes for a desc of the table with the
 *   largest r (the size grows with r).  Needs d / 8 <= 8 x the
 *   number of SMs.  Device-side errors go to *dev_status as in
 *   pi_layer_decode.  The paper has no counterpart: it decodes one layer
 *   call at a time. */
pi_status pi_decode_layers(const pi_ffn_desc* descs, const pi_layer_weights* layers,
                           int32_t R, int32_t J, const float* x, int32_t chain,
                           float* y, int32_t* cnt_out, uint8_t* mask_out,
                           int32_t* dev_status, void* ws, size_t ws_bytes,
                           pi_stream stream);

/* pi_layer_decode for batch 1 without a caller-provided workspace.  The
 * paper has no counterpart to this call; it exists for callers that cannot
 * allocate device memory: for example a plugin inside a host framework that
 * owns all device memory and hands plugins no allocator, or a latency-bound
 * loop that must not call cudaMalloc (it can synchronise the device).
 * Inputs and outputs are the caller's, as in pi_layer_decode with batch = 1
 * and ws = NULL.  The scratch is a fixed array of PI_STATIC_SCRATCH_BYTES in
 * the library's device image, held by every GPU that loads the library until
 * the process exits.  A shape needs
 *     ru(256) + ru(32 r) + ru(4 P) + ru(n) + ru(4 P d)   bytes,
 * ru() rounding up to a multiple of 256 and P the GPU's SM count (at most
 * 512); shapes that need more are rejected with PI_ERR_WORKSPACE before
 * anything is launched (before any CUDA call when even P = 1 would not fit).
 * The call allocates and frees nothing; each call clears the array's barrier
 * block with one cudaMemsetAsync on `stream` before its launch.  The first
 * call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture: made while `stream` is being captured it
 * returns PI_ERR_CAPTURE and launches nothing.  All calls share the one
 * array: calls that overlap on the GPU (other streams, other threads) race
 * and corrupt each other's results; issue them in one stream order. */
#define PI_STATIC_SCRATCH_BYTES (8u << 20)
pi_status pi_layer_decode_static(const pi_ffn_desc* desc, const pi_layer_weights* w,
                                 const float* x, float* y, const float* residual,
                                 int32_t* idx_out, int32_t* cnt_out, int32_t* dev_status,
                                 pi_stream stream);

/* Offline profiling and neuron placement ("Offline Section": a profiler
 * records how often each neuron activates over sample inputs, and the
 * neurons are placed so that the hot ones come first; "Neuron Placement and
 * Administration": a neuron table maps each placed position to the neuron's
 * original one).  Run before decoding, on the caller's stream:
 *   pi_profile_counts: counts[i] += #{t < batch : logits[t][i] > 0} for
 *     logits [batch][n] fp32 (e.g. from pi_predict over sample tokens);
 *     counts [n] uint32 accumulate across calls (zero them first).
 *     n <= 2^24, batch <= 32.
 *   pi_hot_order: perm[k] = the original neuron placed at position k: more
 *     activations first, equal counts in ascending index.  perm [n] int32
 *     is the neuron table.  n <= 2^22 (each entry is ranked against every
 *     count: O(n^2) work, a fraction of a millisecond at n = 28 672).
 *   pi_permute_neurons: dst row k = src row perm[k] for A, b1, W1 (gated:
 *     gate|up rows; packed: whole records) and W2 (split layout); dst holds
 *     buffers of the same sizes, distinct from src (PI_ERR_SHAPE otherwise);
 *     dst->Bm and dst->b2 are not written (Bm is not per neuron; they may
 *     be src's).  perm must be a permutation of [0, n): an entry outside
 *     [0, n) is not followed, its row is left unwritten and PI_ERR_INDEX is
 *     written to *dev_status.  Decoding the placed layer gives the same y;
 *     its active list maps to original neurons through perm. */
pi_status pi_profile_counts(const float* logits, int32_t n, int32_t batch,
                            uint32_t* counts, pi_stream stream);
pi_status pi_hot_order(const uint32_t* counts, int32_t n, int32_t* perm,
                       pi_stream stream);
pi_status pi_permute_neurons(const pi_ffn_desc* desc, const pi_layer_weights* src,
                             const int32_t* perm, const pi_layer_weights* dst,
                             int32_t* dev_status, pi_stream stream);

/* Offline step: builds the PI_LAYOUT_PACKED records of a layer from its
 * split matrices (desc->layout is ignored).  W1 [n][d] (gated [n][2][d]) and
 * W2 [n][d] are read, packed [n][m d] is written (m = 2, or 3 if gated); the
 * buffers must not overlap.  Like the neuron reordering it accompanies
 * ("Offline Section": neurons are laid out by their profiled activation
 * before serving), it runs once per layer, not per token. */
pi_status pi_pack_weights(const pi_ffn_desc* desc, const void* W1, const void* W2,
                          void* packed, pi_stream stream);

/* ---------------------------------------------------------------- dispatch plan
 * Density / batch-aware choice of the decode path ("Efficient,
 * VRAM-Constrained xLM Inference on Clients", section "Methodology, A.
 * Pipelined Sharding": per tier of tokens per step, a time estimator built
 * on bytes moved and measured rates picks the cheapest plan).  Host only: no
 * GPU work, no allocation.
 *
 * Paths:
 *   PI_PATH_FUSED     batch 1: pi_layer_decode (one persistent launch);
 *   PI_PATH_PER_TOKEN batch > 1 as `batch` batch-1 fused decodes;
 *   PI_PATH_UNION     batch 2..32: pi_layer_decode's union of the tokens'
 *                     active rows on the tensor cores (needs d % 128 == 0);
 *   PI_PATH_DENSE     pi_dense_ffn: every row, no predictor.  It computes the
 *                     plain dense FFN, not the predicted-sparse result, so a
 *                     plan offers it only when allow_dense != 0.
 * The first three give the same result (each token's own predicted set).
 *
 * Expected rows: with p_i = P(neuron i active for a token) -- p_active[i]
 * (host array of n values, e.g. pi_profile_counts / profiled tokens), or
 * `density` for every neuron when p_active is NULL -- a token's active rows
 * are sum_i p_i and a batch's union sum_i (1 - (1 - p_i)^batch) (tokens
 * independent).  Bytes per step: predictor P = n r e + r d e + 4 n, a row
 * R = m d e (e = 2, m = 2 plain / 3 gated): FUSED P + active R; PER_TOKEN
 * batch x (P + active R); UNION P + union R; DENSE n R.
 * Time = fixed_us + bytes / (gbs x 1e3) in microseconds, with the path's
 * constants of the batch's tier (PER_TOKEN: batch x FUSED's tier-0 time). */
typedef enum {
  PI_PATH_FUSED = 0,
  PI_PATH_PER_TOKEN = 1,
  PI_PATH_UNION = 2,
  PI_PATH_DENSE = 3
} pi_path;

#define PI_PATHS 4
#define PI_COST_TIERS 4

/* Measured cost of each path per batch tier.  tier_max_batch ascending: a
 * batch uses the first tier whose max is >= batch (the last tier above). */
typedef struct {
  int32_t tier_max_batch[PI_COST_TIERS];
  double fixed_us[PI_PATHS][PI_COST_TIERS];
  double gbs[PI_PATHS][PI_COST_TIERS];  /* GB/s, > 0 */
} pi_cost_model;

typedef struct {
  pi_path path;                /* the available path of least estimated time */
  double est_us[PI_PATHS];     /* estimate per path; -1 when not available */
  double bytes[PI_PATHS];      /* weight bytes per step behind each estimate; -1 n/a */
  double active_rows;          /* expected active neurons per token */
  double union_rows;           /* expected union of the batch's active neurons */
} pi_plan;

/* The built-in model: fitted on one GB300 (measured copy peak 6.78 TB/s) to
 * the density x batch sweep of the OPT-13B-shaped layer (d 5120, n 20480,
 * r 192, fp16; within 5.8 % of every measured point, the faster path picked
 * at all 20 points).  Other shapes move the fixed costs (grid-wide waits,
 * launches) by some microseconds. */
void pi_default_cost_model(pi_cost_model* out);

/* Fills *out for one layer shape and batch (1..32).  model NULL: the
 * built-in one.  Errors: PI_ERR_NULL (desc or out), PI_ERR_SHAPE (bad desc,
 * batch outside 1..32, density outside [0, 1] without p_active, a model
 * rate <= 0 or tiers not ascending). */
pi_status pi_plan_dispatch(const pi_ffn_desc* desc, int32_t batch, const float* p_active,
                           float density, int32_t allow_dense, const pi_cost_model* model,
                           pi_plan* out);

/* Runs one decode step through `path` (a pi_path, e.g. pi_plan.path):
 *   PI_PATH_FUSED      batch == 1: pi_layer_decode;
 *   PI_PATH_PER_TOKEN  one batch-1 pi_layer_decode per token;
 *   PI_PATH_UNION      batch 2..32, d % 128 == 0: pi_layer_decode's union
 *                      path (the tokens' active rows read once, tensor cores);
 *   PI_PATH_DENSE      pi_dense_ffn (+ residual): the plain dense FFN, not
 *                      the predicted-sparse result; idx_out / cnt_out are not
 *                      written.
 * Arguments as in pi_layer_decode (ws of pi_workspace_size(desc, batch)
 * bytes or more).  The first three paths give the same result: each token
 * uses its own predicted set ("PowerInfer: Quick Massive Language Mannequin
 * Serving with a Client-grade GPU", "Online Section").  PI_ERR_SHAPE for a
 * path the batch or shape does not allow. */
pi_status pi_decode_planned(const pi_ffn_desc* desc, const pi_layer_weights* w, int32_t path,
                            const float* x, int32_t batch, float* y, const float* residual,
                            int32_t* idx_out, int32_t* cnt_out, int32_t* dev_status, void* ws,
                            size_t ws_bytes, pi_stream stream);

/* A decoder: one layer, its activation profile and fixed buffers, executing
 * the dispatch plan with one captured CUDA graph per batch size (the tiers of
 * "Efficient, VRAM-Constrained xLM Inference on Clients", "Methodology, A.
 * Pipelined Sharding": a plan per number of tokens per step, chosen by the
 * time estimator).
 *   pi_decoder_create: desc / w as in pi_layer_decode; p_active, density,
 *     allow_dense, model as in pi_plan_dispatch (p_active is copied); x
 *     [32][d] and y [32][d] fp32, residual NULL or [32][d], dev_status and ws
 *     (pi_workspace_size(desc, 32) bytes, zero-filled) are device buffers
 *     the decoder reads and writes on every run; they must outlive it.
 *     Creates a non-blocking stream for its captures (current device).
 *   pi_decoder_run: decodes tokens x[0 .. batch) into y[0 .. batch) through
 *     the path planned for this batch.  The first run of a batch size runs
 *     the calls directly on `stream`, then captures them into a graph; later
 *     runs of that size launch the graph on `stream`.  If `stream` is being
 *     captured by the caller, the calls are recorded into the caller's graph
 *     and no graph of the decoder's is made.  Runs of one decoder must not
 *     overlap on the GPU (they share ws).  PI_ERR_SHAPE on another device.
 *   pi_decoder_plan: the plan used for a batch size.
 *   pi_decoder_destroy: releases the graphs and the stream (after the
 *     caller's last run has completed). */
typedef struct pi_decoder pi_decoder;
pi_status pi_decoder_create(const pi_ffn_desc* desc, const pi_layer_weights* w,
                            const float* p_active, float density, int32_t allow_dense,
                            const pi_cost_model* model, const float* x, float* y,
                            const float* residual, int32_t* dev_status, void* ws, size_t ws_bytes,
                            pi_decoder** out);
pi_status pi_decoder_run(pi_decoder* dec, int32_t batch, pi_stream stream);
pi_status pi_decoder_plan(pi_decoder* dec, int32_t batch, pi_plan* out);
void pi_decoder_destroy(pi_decoder* dec);

/* Neuron-sharded decode across G ranks (one GPU each).  Neurons are
 * independent until the down projection adds their column vectors ("PowerInfer:
 * Quick Massive Language Mannequin Serving with a Client-grade GPU", "Neuron
 * Conscious Operator"), so rank g of G can hold the neurons i = g, g + G,
 * g + 2G, ... of the hot-first order (its neuron table: local row k is
 * neuron g + k G, "Neuron Placement and Administration") with a full copy
 * of Bm, and decode them with the ordinary calls into a partial output
 * (b2 on one rank only, no residual).  One exchange of the G partial
 * outputs (d floats per token, e.g. an all-gather over the ranks) and
 * pi_shard_reduce complete the layer.
 *   pi_shard_desc: the shard's descriptor (host only): n = the rank's neuron
 *     count, hot_prefix = its neurons below the layer's hot prefix (still a
 *     prefix of its rows); G in 1..1024, 0 <= g < min(G, n).
 *   pi_shard_layer: copies rows g, g + G, ... of A, b1, W1 (gated: gate|up;
 *     packed: whole records) and W2 (split layout) into dst, whose buffers
 *     hold the shard's rows (sizes from pi_shard_desc) and differ from src's;
 *     dst->Bm and dst->b2 are not written (pass src->Bm, and b2 on one rank).
 *     Asynchronous strided device-to-device copies on `stream`.
 *   pi_shard_reduce: y[t] = residual[t] (or 0) + sum over g = 0, 1, ..., G-1
 *     of parts[g][t], in that order (deterministic); parts [G][batch][d],
 *     residual NULL or [batch][d], y [batch][d] fp32; batch <= 32. */
pi_status pi_shard_desc(const pi_ffn_desc* desc, int32_t G, int32_t g, pi_ffn_desc* out);
pi_status pi_shard_layer(const pi_ffn_desc* desc, const pi_layer_weights* src, int32_t G,
                         int32_t g, const pi_layer_weights* dst, pi_stream stream);
pi_status pi_shard_reduce(const float* parts, int32_t G, int32_t batch, int32_t d,
                          const float* residual, float* y, pi_stream stream);

/* Static text of a status code. */
const char* pi_status_string(pi_status s);

/* Diagnostic of the failure path: runs the persistent grid's bounded wait
 * with one arrival that never comes, for limit_ns nanoseconds, so every
 * block gives up and PI_ERR_TIMEOUT lands in *dev_status.  ws must be a
 * zero-filled workspace of pi_workspace_size(desc, 1) bytes for some valid
 * desc; it must be zero-filled again afterwards.  Returns PI_OK when the
 * launch was issued. */
/* Diagnostic of the ring's failure path: pi_sparse_ffn for batch 1, except
 * that in every block the copy of the first listed neuron's rows is never
 * issued, so the compute warps' wait for it runs out after limit_ns
 * nanoseconds (1e3 .. 5e9).  The block then abandons its ring, lets every
 * copy it did issue land, and PI_ERR_TIMEOUT lands in *dev_status; y is not
 * meaningful.  Arguments as in pi_sparse_ffn (batch 1); ws must be zero-filled
 * again afterwards.  Returns PI_OK when the launch was issued. */
pi_status pi_selftest_ring_timeout(const pi_ffn_desc* desc, const pi_layer_weights* w,
                                   const float* x, const int32_t* idx, const int32_t* cnt,
                                   int32_t cap, float* y, int32_t* dev_status, void* ws,
                                   size_t ws_bytes, int64_t limit_ns, pi_stream stream);

pi_status pi_selftest_wait_timeout(int32_t* dev_status, void* ws,
                                   size_t ws_bytes, int64_t limit_ns,
                                   pi_stream stream);

#ifdef __cplusplus
}
#endif
#endif
