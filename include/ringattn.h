/*
 * ringattn.h -- C ABI of the GB300 (sm_103a) ring-attention library.
 *
 * The library runs the data-parallel hot path of ring attention on one GPU:
 * the sequence of N tokens is split into P virtual shards; shard r keeps its
 * queries resident while the K/V blocks travel around a ring, and step s pairs
 * Q_r with block j = (r - s) mod P under the step's causal mask.  Each block
 * contributes a per-row online-softmax state (m, l, O~) that is merged exactly.
 *
 * Sources (web pages, cited by title and section):
 *   [GRA]   "GPU Ring Attention" (aicassindra.com)
 *   [ZQ]    ring-attention explainer page (zenaique.com)
 *   [RA-CN] "Ring Attention：把超长序列沿设备环流动" (charlestar.github.io)
 *
 * Conventions for every call:
 *   - Every function returns a ring_status_t; RING_OK is 0, errors are < 0.
 *     No exception crosses the ABI.  ring_attn_last_error() gives a message
 *     for the calling thread's last failure.
 *   - Tensor pointers are DEVICE pointers to caller-owned memory, dense
 *     row-major, 16-byte aligned.  bf16 tensors are passed as const void*.
 *     The library never frees caller memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Launches are asynchronous on it; a device-side bounded wait
 *     that runs out sets an error word that ring_attn_check() reports as
 *     RING_ERR_TIMEOUT.
 *   - Shapes: B batch, H heads, N tokens, d head dim (64 or 128), P shards
 *     (N % P == 0), n = N / P.  "Natural order" tensors are [B][H][N][d]
 *     (or [B][H][N] for per-row scalars) indexed by global token position.
 *     "Shard-major" tensors of one shard are [B][H][n][d] (or [B][H][n])
 *     indexed by local row i.
 *   - Global position of local row i of shard r ([RA-CN] "位置编码必须使用全局位置";
 *     the striped map sends token t to shard t mod P):
 *       contiguous: pos(r, i) = r*n + i        striped: pos(r, i) = i*P + r
 *   - Scores are s = (q . k) / sqrt(d); lse is the natural log of the sum of
 *     exp(s) over the row's allowed keys; causal allows key pos <= query pos.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>

#if defined(__GNUC__)
#define RINGATTN_API __attribute__((visibility("default")))
#else
#define RINGATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ring_attn* ring_attn_t; /* opaque handle */

typedef enum {
  RING_OK = 0,
  RING_ERR_INVALID_ARG = -1, /* bad pointer, shape, index or alignment */
  RING_ERR_UNSUPPORTED = -2, /* valid request the library does not implement */
  RING_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
  RING_ERR_TIMEOUT = -4,     /* a device-side bounded wait ran out */
  RING_ERR_OOM = -5          /* host allocation failed */
} ring_status_t;

/* Token t of the sequence goes to shard:
 *   CONTIGUOUS  t / n, local row t mod n;
 *   STRIPED     t mod P, local row t / P;
 *   ZIGZAG      the sequence cut into 2P chunks of c = n/2 tokens, shard r
 *               holding chunk r (local rows 0..c-1) and chunk 2P-1-r (rows
 *               c..n-1), so every shard has one early and one late chunk
 *               ([GRA] "Striping the sequence to flatten the triangle");
 *               needs N divisible by 2P and c a multiple of 128. */
typedef enum { RING_LAYOUT_CONTIGUOUS = 0, RING_LAYOUT_STRIPED = 1, RING_LAYOUT_ZIGZAG = 2 } ring_layout_t;

/* Class of the (query shard r, K/V block j) pair under the mask
 * ([RA-CN] "Causal Attention 让环不再完全对称": skip a strictly-future block,
 * mask a block crossing the diagonal, run the rest unmasked).  PARTIAL (the
 * zigzag layout only): whole chunks of the block are allowed for whole
 * chunks of the shard's rows, and the rest is skipped (no diagonal); see
 * ring_attn_plan_mask. */
typedef enum {
  RING_BLOCK_SKIP = 0,
  RING_BLOCK_FULL = 1,
  RING_BLOCK_DIAG = 2,
  RING_BLOCK_PARTIAL = 3
} ring_block_class_t;

/* Per-row online-softmax state of one shard ([RA-CN] "局部 Softmax 为什么不能直接相加":
 * running max m, exp-sum l scaled by exp(-m), unnormalised value sum O~).
 * Device pointers, fp32, shard-major: m[B][H][n], l[B][H][n], o[B][H][n][d].
 * An empty row is (m = -inf, l = 0, O~ = 0).  m is a reference point: any
 * m with l and O~ scaled by exp(-m) describes the same state; m + ln(l) and
 * O~ / l are unique. */
typedef struct {
  float* m;
  float* l;
  float* o;
} ring_state_t;

/* Options for ring_attn_set_option. */
typedef enum {
  /* How ring_attn_fwd moves each K/V block to the next shard between steps
   * (every shard sends its block to shard r+1 through a double buffer).
   * 2 (default): the step kernel sends it: the CTAs store the key/value tiles
   *   they have loaded into slot r+1 of the other buffer (TMA stores from
   *   shared memory); only the slots of shards with no work at that step
   *   (skipped causal blocks) are copied on a side stream.
   * 1: device-to-device copies of the whole buffer on a side stream.
   * 0: no movement; every step reads its block straight from the packed
   *   buffer (for measuring the cost of the other two).
   * All three give bit-identical results. */
  RING_OPT_ROTATION = 0,
  /* 1: record CUDA events around every pack, copy and step kernel of
   * ring_attn_fwd so ring_attn_get_timing can report them, one set of
   * events per call (the handle keeps up to 64).  Default 0. */
  RING_OPT_TIMING = 1,
  /* Upper bound, in nanoseconds, of every device-side wait.  Default 2e9. */
  RING_OPT_WAIT_LIMIT_NS = 2,
  /* Test hook, default 0.  1: the step kernels issue no loads of V tiles,
   * so the first wait for a V tile runs out after RING_OPT_WAIT_LIMIT_NS;
   * the kernel then drains what it started, frees its tensor memory and
   * returns, and ring_attn_check reports RING_ERR_TIMEOUT.  The outputs of
   * such a call are undefined.  Exists to test the bounded-wait error path. */
  RING_OPT_DEBUG_DROP_V_LOADS = 3,
  /* Causal sliding window W (tokens; 0 = none, the default): a query sees
   * itself and the W-1 tokens before it ([RA-CN] "正确性测试应覆盖哪些边界"
   * lists sliding-window masks).  Applies to ring_attn_fwd, block_partial,
   * the planner queries, ring_attn_decode and ring_attn_bwd, in all three
   * layouts.  Rebuilds the plan; needs the causal mask (RING_ERR_UNSUPPORTED
   * otherwise, the handle keeping its previous window). */
  RING_OPT_WINDOW = 4,
  /* How ring_attn_bwd schedules the ring ([RA-CN] "Backward 需要让梯度也沿环传播"
   * has each block's dK/dV accumulators travel with it around the ring).
   * 0: one dK/dV and one dQ launch per ring step; the travelling
   *   accumulators pass between steps through the workspace buffers.
   * 1 (default): one launch of each kernel for the whole ring: a CTA owning a key
   *   tile of block j visits shards j, j+1, .. in step order, and a CTA
   *   owning a query tile of shard r visits blocks r, r-1, .., with the
   *   accumulators held in tensor memory from the first visit to the last
   *   (the accumulator buffers are not used).  The MMAs run in the same
   *   order on the same fp32 values as in mode 0, so the results are
   *   identical.  ring_attn_get_bwd_timing then reports both kernels' times
   *   in entry 0 and zeros in the others. */
  RING_OPT_BWD_LAP = 5,
  /* How ring_attn_fwd schedules the ring's steps.
   * 0 (default): one step kernel per ring step, the running state (m, l, O~)
   *   passing from step to step through the workspace, and the K/V blocks
   *   moved as RING_OPT_ROTATION says.
   * 1: one launch for the whole ring ("lap"): a CTA owning a pair of query
   *   tiles of shard r meets blocks r, r-1, .. in step order, the state held
   *   on chip from the first step to the last, and the blocks read in place
   *   (from k and v, or the packed buffer for zigzag; no rotation;
   *   RING_OPT_ROTATION is ignored).
   *   Same arithmetic per key tile; the result matches mode 0 within the
   *   parity tolerances, not bit for bit (mode 0 visits the key tiles of a
   *   block without a diagonal in a rotated order, and stores m between
   *   steps in natural-log units, so P is rounded against other running
   *   maxima).  Worth it where a step has little work per query tile
   *   (sliding windows, packed documents).
   *   ring_attn_get_timing then reports the launch in kernel_ms[0]. */
  RING_OPT_FWD_LAP = 6
} ring_option_t;

/* Create a handle for one problem shape.  Validates the shape and builds the
 * host plan (per step, per shard: block, class, diagonal offset, work
 * counts).  Touches no GPU; device resources are made on first use.
 * Errors: RING_ERR_INVALID_ARG for out == NULL or a non-positive size,
 * causal not 0/1, layout not a ring_layout_t, P > N;
 * RING_ERR_UNSUPPORTED for N % P != 0 or d not in {64, 128}. */
RINGATTN_API int ring_attn_create(ring_attn_t* out, int B, int H, long long N, int d, int P, int causal, int layout);

/* As ring_attn_create, with grouped-query (GQA) or multi-query (MQA, Hkv = 1)
 * attention: H query heads share Hkv K/V heads, query head h reading K/V
 * head h / (H / Hkv).  k and v (and the K/V blocks of ring_attn_block_partial)
 * are then [B][Hkv][.][d]; q, out, lse and the states keep H heads.  Only
 * the Hkv heads travel the ring, so the rotation buffers and the bytes sent
 * per step shrink by H / Hkv ([GRA] "What memory actually does as the ring
 * grows": KV per device; the shared K/V of grouped heads rotates once).
 * Errors as ring_attn_create, plus RING_ERR_INVALID_ARG when Hkv <= 0 or H is
 * not a multiple of Hkv.  ring_attn_create(..., H, ...) is Hkv = H. */
RINGATTN_API int ring_attn_create_gqa(ring_attn_t* out, int B, int H, int Hkv, long long N, int d, int P, int causal,
                                      int layout);

/* Release a handle (its events, side stream and plan memory).  Waits for no
 * stream; the caller must not destroy a handle with launches in flight.
 * NULL is accepted. */
RINGATTN_API int ring_attn_destroy(ring_attn_t h);

/* Message for the calling thread's last failed call ("" if none). */
RINGATTN_API const char* ring_attn_last_error(void);

/* Bytes of device workspace ring_attn_fwd needs: the two K/V rotation
 * buffers A and B, each [P][B][H][n][d] bf16 for K and for V ([RA-CN]
 * "双缓冲是重叠成立的基础": buffer A read by compute while B receives), plus
 * the running state (m, l, O~) between steps, fp32, stored per 128-row tile
 * of each shard (n rounded up to whole tiles).  256-byte aligned by the
 * caller. */
RINGATTN_API int ring_attn_workspace_size(ring_attn_t h, size_t* bytes);

/* ---------------------------------------------------------------- planner
 * Host-only queries of the plan (no GPU needed). */

/* Block held by shard r at ring step s, j = (r - s) mod P ([GRA] "One lap
 * around the ring"; [RA-CN] "环是怎样工作的"), its class and its diagonal
 * offset delta: within the block a (row i, column k) pair is allowed iff
 * k - i <= delta (contiguous delta = (r - j) n; striped delta = 0 if j <= r
 * else -1; non-causal FULL).  Any output pointer may be NULL. */
RINGATTN_API int ring_attn_plan_block(ring_attn_t h, int r, int step, int* j, int* cls, long long* delta);

/* The mask of local query row `row` of shard r at ring step s, in the
 * block's local key columns: key k is allowed iff k < key_limit and
 * k - row <= delta.  For CONTIGUOUS and STRIPED every row of a block has
 * key_limit = n (0 for a skipped block) and the block's delta.  ZIGZAG
 * (chunks of c = n/2; the rule follows from comparing global positions):
 *   j < r:  key_limit = c for every row (the block's early chunk), no diagonal;
 *   j = r:  key_limit = n, delta = 0;
 *   j > r:  rows of the early chunk none (key_limit 0), rows of the late
 *           chunk every key.
 * "No diagonal" is returned as delta = n.  The causal rule only: with a
 * window or segments ring_attn_plan_key_range gives a row's keys.  Any
 * output pointer may be NULL. */
RINGATTN_API int ring_attn_plan_mask(ring_attn_t h, int r, int step, long long row, long long* key_limit,
                                     long long* delta);

/* The keys local row `row` of shard r sees at ring step s, in the block's
 * local columns: first .. last inclusive (first > last: none).  Covers every
 * mask the handle applies (causal, layout, sliding window, segments).  Any
 * output pointer may be NULL. */
RINGATTN_API int ring_attn_plan_key_range(ring_attn_t h, int r, int step, long long row, long long* first,
                                          long long* last);

/* Per-shard totals over all P steps: allowed (q, k) pairs[P] and the
 * 128x128 MMA tiles the kernel computes[P] (any pointer may be NULL). */
RINGATTN_API int ring_attn_shard_work(ring_attn_t h, long long* pairs, long long* tiles);

/* Totals of one step over all shards: allowed pairs and computed tiles. */
RINGATTN_API int ring_attn_step_work(ring_attn_t h, int step, long long* pairs, long long* tiles);

/* ---------------------------------------------------------------- state */

/* Set a shard's state to empty: m = -inf, l = 0, O~ = 0 (the pages'
 * empty_online_softmax_state, [RA-CN] "环是怎样工作的"). */
RINGATTN_API int ring_attn_state_init(ring_attn_t h, ring_state_t s, void* stream);

/* Block partial of ring step `step` for shard r ([RA-CN] "环是怎样工作的":
 * block_attention(local_q, kv, mask_for(step)); "两层分块如何嵌套": the kernel
 * can emit a mergeable state or update the local running buffer).
 *   q_shard  shard r's queries, shard-major [B][H][n][d] bf16
 *   k_block, v_block  block j = (r - step) mod P, shard-major [B][H][n][d] bf16
 *   state    shard r's state (see ring_state_t)
 *   accumulate  0: overwrite `state` with this block's partial state
 *               1: merge this block into `state` (exact rescale merge)
 * The mask uses global positions of shard r's rows and block j's keys.  A
 * SKIP block leaves `state` unchanged (accumulate 1) or writes the empty
 * state (accumulate 0).  All pointers 16-byte aligned. */
RINGATTN_API int ring_attn_block_partial(ring_attn_t h, int r, int step, const void* q_shard, const void* k_block,
                            const void* v_block, ring_state_t state, int accumulate, void* stream);

/* a <- merge(a, b) over one shard's B*H*n rows ([GRA] "Why partial results
 * are allowed to merge"; [ZQ]: rescale by exp(old_max - new_max)):
 *   m = max(ma, mb); alpha = exp(ma - m), beta = exp(mb - m) (0 for an
 *   m = -inf side); l = alpha la + beta lb; O~ = alpha O~a + beta O~b.
 * a and b must not overlap. */
RINGATTN_API int ring_attn_merge(ring_attn_t h, ring_state_t a, ring_state_t b, void* stream);

/* Finalize shard r's state into natural-order outputs ([RA-CN] "环是怎样工作的":
 * local_output = finalize(state)): out[b][h][pos(r,i)][:] = O~ / l and
 * lse[b][h][pos(r,i)] = m + ln(l); an empty row gives out = 0, lse = -inf.
 *   out  [B][H][N][d] fp32, lse [B][H][N] fp32 (only shard r's rows written) */
RINGATTN_API int ring_attn_finalize(ring_attn_t h, int r, ring_state_t s, float* out, float* lse, void* stream);

/* Whole ring forward on one device ([RA-CN] "环是怎样工作的" forward loop;
 * "双缓冲是重叠成立的基础" double buffering):
 *   q, k, v   natural order [B][H][N][d] bf16
 *   out       natural order [B][H][N][d] fp32
 *   lse       natural order [B][H][N]   fp32
 *   workspace ring_attn_workspace_size() bytes, 256-byte aligned
 * K/V are packed shard-major into buffer A; step s runs one kernel over every
 * shard's block (r - s) mod P, reading slot r of the current buffer, and
 * moves every block to slot r+1 of the other buffer for step s+1 as set by
 * RING_OPT_ROTATION.  (The lap, RING_OPT_FWD_LAP, reads the blocks in place
 * from k and v instead, except in the zigzag layout.)  The running state stays in the workspace; the last step
 * writes the normalised output and lse.  Returns after enqueueing; `stream`
 * orders it with the caller's work. */
RINGATTN_API int ring_attn_fwd(ring_attn_t h, const void* q, const void* k, const void* v, float* out, float* lse,
                  void* workspace, void* stream);

/* ring_attn_fwd from HOST memory and back, with the copies overlapped with
 * the computation.  The heads are independent problems, so they run in
 * groups of whole K/V heads (with 8 or more K/V heads over all batches: one
 * K/V head in each of the first two and the last two groups, the rest in an
 * even number of near-equal groups; with fewer, one K/V head per group),
 * each group a ring_attn_fwd over its heads.  The inputs are copied in
 * group by group; each group computes as soon as its inputs are in, on one
 * of two lanes in turn (`stream` and a stream the handle owns), so two
 * groups share the SMs; each group's outputs are copied out as soon as it
 * is done.  The results equal ring_attn_fwd's over all heads.
 *   q, k, v   HOST pointers, natural order as in ring_attn_fwd (bf16);
 *             page-locked (cudaHostAlloc, or a pinned torch tensor) for the
 *             copies to be asynchronous and overlapped
 *   out, lse  HOST pointers, as in ring_attn_fwd (fp32)
 * The handle owns the device buffers (the inputs and outputs of all heads,
 * and a workspace for each group size on each lane), made on the first call
 * and kept until ring_attn_destroy, two copy streams and the second lane's
 * stream.  Asynchronous on `stream`: the copies start after the caller's
 * earlier work on it, and `stream` completes after the last output copy and
 * the second lane's last kernel, so the host may read out and lse after
 * synchronising it.  The host buffers must stay valid, and the inputs
 * unchanged, until then.  ring_attn_check covers the copy streams, the
 * second lane and the group handles.  Errors: RING_ERR_INVALID_ARG for NULL
 * pointers; RING_ERR_CUDA, RING_ERR_OOM. */
RINGATTN_API int ring_attn_fwd_host(ring_attn_t h, const void* q, const void* k, const void* v, float* out,
                                    float* lse, void* stream);

/* Ring backward on one device ([RA-CN] "Backward 需要让梯度也沿环传播": every
 * Q-K/V block interaction contributes a gradient; the owner of a query shard
 * accumulates its dQ from every K/V block, while the dK and dV of a
 * travelling block accumulate the contributions of each query owner it
 * passes and return to the block's owner; the probabilities are recomputed
 * from the forward's saved per-row logsumexp).  With P = exp(scale QK^T -
 * lse) over the allowed pairs, D = rowsum(dO * out), dS = P (dO V^T - D):
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 *   q         natural order [B][H][N][d] bf16 (the forward's input)
 *   k, v      natural order [B][Hkv][N][d] bf16 (Hkv = H unless the handle
 *             was made by ring_attn_create_gqa)
 *   out, lse  the forward's outputs: [B][H][N][d] and [B][H][N] fp32
 *   dout      the gradient of the loss with respect to out, [B][H][N][d] bf16
 *   dq        output, natural order [B][H][N][d] fp32
 *   dk, dv    outputs, natural order [B][Hkv][N][d] fp32; with grouped K/V
 *             heads a shared head's gradient sums the contributions of the
 *             H/Hkv query heads that read it
 *   workspace ring_attn_bwd_workspace_size() bytes, 256-byte aligned: the
 *             per-row lse and D, shard-major; with RING_OPT_BWD_LAP 0 and
 *             P > 1 also two buffers of the travelling dK/dV accumulators,
 *             fp32 [P][B][Hkv][n][d] each.  The size depends on that option:
 *             query it after setting the option.
 * The ring: at step s every shard r meets block j = (r - s) mod P.  Two
 * kernels cover it: one per 128-key tile of a block (dK and dV) and one per
 * 128-row query tile of a shard (dQ).  RING_OPT_BWD_LAP 1 (default): one
 * launch of each, every CTA making its tile's visits in step order with the
 * accumulators in tensor memory.  RING_OPT_BWD_LAP 0: two launches per step,
 * the dK/dV accumulators entering from slot r of one buffer and leaving to
 * slot r + 1 of the other, dQ kept in dq between steps.
 * K/V blocks are read in place through strided views of k and v.  Layouts
 * CONTIGUOUS, STRIPED and ZIGZAG, causal or not, with or without
 * RING_OPT_WINDOW and segments.
 * Pointers 16-byte aligned.  Asynchronous on `stream`. */
RINGATTN_API int ring_attn_bwd_workspace_size(ring_attn_t h, size_t* bytes);
RINGATTN_API int ring_attn_bwd(ring_attn_t h, const void* q, const void* k, const void* v, const float* out,
                               const float* lse, const void* dout, float* dq, float* dk, float* dv,
                               void* workspace, void* stream);

/* Timings of the last ring_attn_bwd with RING_OPT_TIMING on, in ms: the
 * dK/dV kernel and the dQ kernel of every step (arrays of P entries, NULL to
 * skip) and the preprocessing kernel (lse * log2(e) and D).  Synchronises
 * on the recorded events. */
RINGATTN_API int ring_attn_get_bwd_timing(ring_attn_t h, float* dkdv_ms, float* dq_ms, float* prep_ms);

/* Split-K/V decode and short-query prefill ([RA-CN]: the query is sent to
 * every K/V shard, each shard computes a local online-softmax state, and the
 * states are merged exactly; [GRA] "Why partial results are allowed to
 * merge").  Lq new queries sit at global positions N-Lq .. N-1 of the
 * sequence the handle describes, and their K/V are already part of the
 * cache, so under the causal mask query i sees the cached keys at positions
 * <= N-Lq+i (all N keys for Lq = 1).  The cache is read in place in natural
 * order; its keys are cut into ksplit contiguous pieces (the ring's shards
 * are one partition of them; on one GPU the pieces are sized for the SMs),
 * and one launch computes a local state per piece and query tile pair: the
 * smallest ksplit that fills at least 90 % of the SMs in whole waves, at
 * least 4 key tiles a piece (at Lq = 1 on 16 heads and 152 SMs: 9 pieces
 * of about 114 key tiles, one wave).  A second launch merges the ksplit
 * states of each row and finalizes.  The result does not depend on the
 * handle's layout or P.
 *   q         [B][H][Lq][d] bf16
 *   k, v      the cache, natural order [B][Hkv][N][d] bf16
 *   out       [B][H][Lq][d] fp32,  lse [B][H][Lq] fp32
 *   workspace ring_attn_decode_workspace_size(h, Lq) bytes, 256-byte aligned
 *             (it depends on the current device's SM count)
 * Windows and documents apply (RING_OPT_WINDOW, ring_attn_set_segments);
 * 1 <= Lq <= N.  Asynchronous on `stream`. */
RINGATTN_API int ring_attn_decode_workspace_size(ring_attn_t h, long long Lq, size_t* bytes);
RINGATTN_API int ring_attn_decode(ring_attn_t h, const void* q, const void* k, const void* v, long long Lq, float* out,
                                  float* lse, void* workspace, void* stream);

/* Sequence packing ([RA-CN] "正确性测试应覆盖哪些边界": several documents packed
 * into one sequence must not attend to each other; the same list names
 * sliding-window/segment masks and the tail padding with a valid-length
 * mask).  bounds: host array of num_segments + 1 natural positions,
 * 0 = b_0 < b_1 < .. < b_num_segments = N; document s is [b_s, b_{s+1}).
 * A pair (query, key) is then allowed only inside one document, on top of
 * the causal mask and the window.  A valid length L < N is the list
 * {0, L, N}: the padding forms its own document, so no real token sees it.
 * num_segments = 0 (bounds may be NULL) removes the segments.  Rebuilds the
 * plan (the work counts follow the segments); the device copy of the table
 * (two ints per position, owned by the handle) is made by the next compute
 * call.  Applies to ring_attn_fwd, block_partial, decode and bwd.
 * RING_ERR_INVALID_ARG for a list that does not rise strictly from 0 to N;
 * RING_ERR_UNSUPPORTED for N >= 2^31 (the handle keeps its previous
 * segments).  ring_attn_fwd_noalloc returns
 * RING_ERR_UNSUPPORTED while segments are set. */
RINGATTN_API int ring_attn_set_segments(ring_attn_t h, const long long* bounds, int num_segments);

/* Set an option (see ring_option_t). */
RINGATTN_API int ring_attn_set_option(ring_attn_t h, int option, long long value);

/* Timings of the ring_attn_fwd calls made with RING_OPT_TIMING on, in ms,
 * each the mean over the calls timed since the previous read of the timings
 * (this function or ring_attn_get_release_wait; the latest 64 calls when
 * there were more); each array has P entries (NULL to skip): step kernel
 * time, rotation copy time for the copy that feeds step s (0 for s = 0, and
 * 0 in calls where no copy fed step s), and the time the compute stream
 * waited for that copy (exposed copy time).  pack_ms: the packing kernel
 * (0 for a lap that reads the blocks in place).  Reading does not clear the
 * record; the next timed call starts a new one.  Synchronises on the
 * recorded events.  RING_ERR_INVALID_ARG when no timed call was recorded. */
RINGATTN_API int ring_attn_get_timing(ring_attn_t h, float* kernel_ms, float* copy_ms, float* wait_ms, float* pack_ms);

/* The other side of the overlap check of the timed ring_attn_fwd calls
 * ([RA-CN] "如何判断通信是否真的被覆盖": besides compute waiting for the
 * communication, record how long the communication waits for the buffer to
 * be released): release_wait_ms[s] (P entries, ms) is the time the side
 * stream spent, before the copy that feeds step s, waiting for step s - 2 to
 * release the buffer it fills (0 where no copy fed step s), the mean over the
 * same calls as ring_attn_get_timing.  Needs RING_OPT_TIMING; synchronises
 * on the recorded events. */
RINGATTN_API int ring_attn_get_release_wait(ring_attn_t h, float* release_wait_ms);

/* Synchronise `stream` and report any device-side error recorded by this
 * handle's kernels since the last check (RING_ERR_TIMEOUT for a wait that
 * ran out), clearing it. */
RINGATTN_API int ring_attn_check(ring_attn_t h, void* stream);

/* ring_attn_fwd for callers that cannot allocate device memory (the pages
 * have no counterpart: this is a packaging of ring_attn_fwd, not a step of
 * the method).  Callers such as a plug-in inside a host application that
 * owns all device memory through its own pool, or code on a latency-critical
 * path where cudaMalloc/cudaFree may synchronise the device, pass only
 * inputs and outputs; the scratch ring_attn_fwd takes as a workspace (the
 * packed K/V and the running l state) lives in a fixed 64 MiB __device__
 * array inside the library, which every GPU that loads the library holds
 * until the process exits.
 *   q, k, v, out, lse  as for ring_attn_fwd (device, 16-byte aligned)
 *   status  optional device int (NULL to skip): receives the device-side
 *           error flags of this call (0 = ok, nonzero = a bounded wait ran
 *           out), written on `stream` at the end of the call
 * Errors: RING_ERR_UNSUPPORTED when the problem's scratch
 * (4*B*Hkv*N*d bytes of packed K and V, Hkv the K/V heads, plus
 * 4*B*H*N bytes of l and alignment) exceeds the array; otherwise
 * as ring_attn_fwd.  Every step reads its block straight from the packed
 * buffer (no rotation copies); the result equals ring_attn_fwd's.
 * The call allocates nothing.  Its first call on a device, with that device
 * current, does a one-time set-up (device check, kernel attributes, the
 * array's device address via cudaGetSymbolAddress); make that first call
 * before any stream capture.  All calls share the array and it keeps the
 * last call's contents: calls that overlap on the GPU race on it, so
 * serialise them. */
RINGATTN_API int ring_attn_fwd_noalloc(ring_attn_t h, const void* q, const void* k, const void* v, float* out,
                                       float* lse, int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
