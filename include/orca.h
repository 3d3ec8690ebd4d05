/*
 * orca.h - C ABI of liborca: one selectively batched Transformer iteration
 * (Orca-style iteration-level scheduling + selective batching) on one GPU.
 *
 * Passages this interface follows (page title, section):
 *   - "连续批处理完全拆解：Orca 的迭代级调度与选择性批处理" (Orca walk-through):
 *       Algorithm 1 "ORCA scheduling algorithm" (Select, max_bs, n_slots,
 *       max_tokens reservation, break on overflow); Figure 5 (flatten the
 *       batch to [sum L_i, H], Split before attention, per-request attention
 *       against the Attention K/V manager, Merge after it).
 *   - CS349D Lecture 2 "批处理与调度", section 4.3 (reservation rule) and
 *       section 5.1 (try_admit / free memory-manager interface).
 *   - "Orca: The beginning of Morden LLM serving." notes, section "Scheduling
 *       Algorithm" (select_batch sketch).
 *
 * Conventions for every call:
 *   - Return 0 (ORCA_OK) or a negative ORCA_E* code.  No exception, abort or
 *     exit crosses this boundary.  orca_last_error() gives a message.
 *   - Device pointers are owned by the caller (the library never frees or
 *     allocates device memory; it allocates only pinned host staging buffers
 *     and CUDA events).  Host pointers are borrowed for the duration of a call,
 *     except orca_request.tokens, which must stay valid while the request is
 *     in a pool passed to orca_select_batch / orca_iteration.
 *   - An engine is not thread-safe; one host thread drives one engine.
 *   - Streams are passed as a cudaStream_t cast to void* (NULL = legacy
 *     default stream).
 */
#ifndef ORCA_H_
#define ORCA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- codes */
#define ORCA_OK 0
#define ORCA_EINVAL (-1)          /* bad argument, shape or state            */
#define ORCA_ENOSLOTS (-2)        /* reservation exceeds n_slots or no hole  */
#define ORCA_EBATCH (-3)          /* n_batch > max_bs or sum L_i > max_rows  */
#define ORCA_EUNKNOWN_REQ (-4)    /* release of an id that never reserved    */
#define ORCA_EDOUBLE_RELEASE (-5) /* release of an id already released       */
#define ORCA_EDEVICE (-6)         /* a kernel raised its device status word  */
#define ORCA_ECUDA (-7)           /* a CUDA runtime call failed              */
#define ORCA_ESTATE (-8)          /* engine has no device side (host-only)   */

#define ORCA_DTYPE_F32 0
#define ORCA_DTYPE_BF16 1

/* request states (Algorithm 1) */
#define ORCA_INITIATION 0
#define ORCA_INCREMENT 1
#define ORCA_RUNNING 2
#define ORCA_FINISHED 3

/* orca_iteration flags */
#define ORCA_ITER_TEACHER_FORCE 1 /* read every input token from req.tokens;
                                     never write generated tokens into it   */
#define ORCA_ITER_EAGER 2         /* launch the kernels one by one instead of
                                     replaying the engine's CUDA graph      */
#define ORCA_ITER_SELFTEST_TIMEOUT 4 /* test hook: after the forward, one CTA
                                     waits on a barrier that nothing
                                     completes; its bounded wait (about 2 s)
                                     expires and sets the iteration's status
                                     word, so the wait returns ORCA_EDEVICE
                                     (the failure path, without a fault)    */

/* ---------------------------------------------------------------- types */
typedef struct orca_engine orca_engine;

#define ORCA_RESERVE_MAX 0
#define ORCA_RESERVE_POW2 1
#define ORCA_RESERVE_ORACLE 2
#define ORCA_RESERVE_PAGED 3
#define ORCA_KV_BLOCK 32

/* Model shape and scheduler parameters.
 *   GPT decoder: n_layers blocks of hidden size `hidden`, n_heads heads
 *   (head_dim = hidden / n_heads), MLP width `ffn`, vocabulary `vocab`,
 *   learned positions 0..max_pos-1.
 *   dtype: ORCA_DTYPE_F32 (all fp32) or ORCA_DTYPE_BF16 (matrices,
 *   embeddings, K/V slots and stored activations bf16; residual stream,
 *   LayerNorm statistics, accumulation and logits fp32).
 *   max_bs, n_slots: Algorithm 1 parameters.  n_slots < 2^31.
 *   max_rows: capacity for sum L_i of one iteration.
 *   reserve_policy: K/V slots a request reserves at first schedule (CS349D
 *   Lecture 2, section 6.1): ORCA_RESERVE_MAX max_tokens (Orca's rule);
 *   ORCA_RESERVE_POW2 its true final length n_prompt + out_len rounded up to
 *   a power of two (a rough length prediction); ORCA_RESERVE_ORACLE the true
 *   final length; both capped at max_tokens.  ORCA_RESERVE_PAGED reserves
 *   nothing: slots come in blocks of ORCA_KV_BLOCK as a request grows
 *   (n_slots must be a multiple of ORCA_KV_BLOCK); see orca_select_batch.
 *   bf16 requires hidden % 64 == 0 and ffn % 64 == 0; every dtype requires
 *   head_dim in {16, 32, 64, 128}. */
typedef struct {
  int32_t n_layers, hidden, n_heads, ffn, vocab, max_pos;
  int32_t dtype;
  int32_t max_bs;
  int64_t n_slots;
  int32_t max_rows;
  int32_t reserve_policy;
} orca_config;

/* One request of the pool (host memory, owned by the caller).
 *   arrival, req_id: Select sorts by (arrival, req_id) ascending.
 *   state: ORCA_INITIATION until first scheduled; Select sets RUNNING,
 *   orca_iteration sets INCREMENT or FINISHED.
 *   n_prompt: prompt tokens; out_len: tokens to generate (no EOS);
 *   max_tokens: the request's length limit, prompt included (>= n_prompt).
 *   n_cached: tokens whose K/V are stored; n_generated: tokens produced.
 *   n_sched: rows of this request in the selected batch, set by the Select
 *   calls (0 = the default: the rest of the prompt while n_cached <
 *   n_prompt, else one row); orca_iteration resets it to 0.
 *   n_reserved: K/V slots reserved at first schedule (0 before; set by
 *   Select); slot_base: first reserved slot (-1 before reservation).
 *   tokens: host int32 buffer of capacity n_prompt + out_len holding the
 *   prompt followed by the generated (or teacher-forced) tokens.
 * Callers initialise n_sched = n_reserved = 0 and slot_base = -1.
 * A request finishes when n_generated == out_len or
 * n_prompt + n_generated >= max_tokens; its slots are then released. */
typedef struct {
  int64_t req_id;
  int64_t arrival;
  int32_t state;
  int32_t n_prompt;
  int32_t max_tokens;
  int32_t out_len;
  int32_t n_cached;
  int32_t n_generated;
  int32_t n_sched;
  int32_t n_reserved;
  int64_t slot_base;
  int32_t *tokens;
} orca_request;

/* Per-kernel-class timing gathered when profiling is enabled. */
typedef struct {
  int64_t launches;
  double total_ms;     /* sum of CUDA-event durations of the launches      */
  double flops;        /* algorithmic FLOPs of those launches              */
  double bytes;        /* algorithmic HBM bytes of those launches          */
} orca_kernel_stats;

#define ORCA_K_EMBED 0
#define ORCA_K_LAYERNORM 1
#define ORCA_K_GEMM_QKV 2
#define ORCA_K_ATTENTION 3
#define ORCA_K_GEMM_O 4
#define ORCA_K_GEMM_FC1 5
#define ORCA_K_GEMM_FC2 6
#define ORCA_K_LM_HEAD 7
#define ORCA_K_ARGMAX 8
#define ORCA_K_COUNT 9

/* ---------------------------------------------------------------- sizing */
/* Bytes of the K/V slot pool: n_layers * 2 * n_slots * hidden * elem.
 * Layout (row-major): [n_layers][2 (K,V)][n_heads][n_slots][head_dim];
 * slot s of a request holds the K/V of its token at position s - slot_base. */
int orca_kv_pool_bytes(const orca_config *cfg, size_t *bytes);

/* Bytes of device workspace orca_engine_create needs (activations, the
 * device batch descriptor, attention scratch, logits; in bf16 also the
 * row statistics and per-layer vectors of the LayerNorms folded into the
 * Linears after them). */
int orca_workspace_bytes(const orca_config *cfg, size_t *bytes);

/* Number of weight pointers orca_engine_create expects: 4 + 12 * n_layers.
 * Order: tok_emb [vocab, hidden], pos_emb [max_pos, hidden], lnf_g [hidden],
 * lnf_b [hidden], then per layer: ln1_g, ln1_b, w_qkv [3H, H], b_qkv [3H],
 * w_o [H, H], b_o [H], ln2_g, ln2_b, w_fc1 [ffn, H], b_fc1 [ffn],
 * w_fc2 [H, ffn], b_fc2 [H].  Matrices are [out, in] row-major; y = W x + b.
 * Matrices and embeddings are in cfg.dtype; LayerNorm parameters and biases
 * are fp32.  Every pointer must be 16-byte aligned. */
int orca_weight_count(const orca_config *cfg, int32_t *count);

/* ---------------------------------------------------------------- engine */
/* Create an engine.  weights: n_weights device pointers (see
 * orca_weight_count); kv_pool: device memory of kv_bytes >=
 * orca_kv_pool_bytes; workspace: device memory of ws_bytes >=
 * orca_workspace_bytes, 256-byte aligned.  All three stay owned by the
 * caller and must outlive the engine.  Passing weights = kv_pool =
 * workspace = NULL creates a host-only engine (scheduler and slot pool
 * only; orca_iteration then returns ORCA_ESTATE) that makes no CUDA call.
 * The current CUDA device at creation is the engine's device.  A bf16
 * engine reads the weights once here (after a device synchronisation) to
 * derive the vectors of its folded LayerNorms: the weights must not change
 * while the engine lives. */
int orca_engine_create(const orca_config *cfg, const void *const *weights, int32_t n_weights,
                       void *kv_pool, size_t kv_bytes, void *workspace, size_t ws_bytes,
                       orca_engine **out);
int orca_engine_destroy(orca_engine *eng);

/* ---------------------------------------------------------------- K/V slots */
/* Reserve n_tokens contiguous slots for req_id (Algorithm 1: max_tokens per
 * request, kept until the request finishes).  First fit at the lowest free
 * base.  ORCA_ENOSLOTS if n_rsrv + n_tokens > n_slots or no contiguous hole
 * is large enough; ORCA_EINVAL if n_tokens <= 0 or req_id already holds a
 * reservation. */
int orca_kv_reserve(orca_engine *eng, int64_t req_id, int32_t n_tokens, int64_t *slot_base);
/* Release req_id's slots.  ORCA_EDOUBLE_RELEASE if already released,
 * ORCA_EUNKNOWN_REQ if it never reserved. */
int orca_kv_release(orca_engine *eng, int64_t req_id);
/* n_rsrv: reserved slots; n_free_blocks: holes in the free list;
 * frag_blocks: reservations that passed the count rule but found no hole. */
int orca_kv_stats(const orca_engine *eng, int64_t *n_rsrv, int64_t *n_free_blocks,
                  int64_t *frag_blocks);

/* K/V memory use over a pool (CS349D Lecture 2, section 6.1: reserved is
 * not the same as used): *reserved = slots currently reserved by the
 * engine; *stored = sum of n_cached over the pool's requests that hold a
 * reservation (not INITIATION, not FINISHED), the slots that hold K/V. */
int orca_kv_usage(const orca_engine *eng, const orca_request *pool, int32_t n_pool, int64_t *reserved,
                  int64_t *stored);

/* ---------------------------------------------------------------- scheduling */
/* Algorithm 1 Select over pool[0..n_pool): skip RUNNING and FINISHED
 * requests, sort the rest by (arrival, req_id), take at most max_bs; an
 * INITIATION request first reserves slots by reserve_policy (slot_base and
 * n_reserved are set),
 * and a failed reservation ends the selection (no skipping).  Selected
 * requests become RUNNING.  batch_idx (capacity max_bs) receives pool
 * indices in batch order; *n_batch their count (0 is valid). */
int orca_select_batch(orca_engine *eng, orca_request *pool, int32_t n_pool, int32_t *batch_idx,
                      int32_t *n_batch);
/* With ORCA_RESERVE_PAGED (CS349D Lecture 2, sections 5.1 and 6.1: blocks
 * handed out on demand, preemption of the latest arrival when memory runs
 * short) the same walk over the candidates grows each one's block table to
 * cover the rows it runs this iteration (lowest free blocks first).  When
 * the pool is short, the latest-arrived requests holding blocks that are not
 * in the batch (and not RUNNING) are preempted: their blocks are freed and
 * they return to INITIATION with n_cached = 0, to recompute their prompt and
 * generated tokens when selected again.  If it still does not fit, a request
 * that holds no blocks ends the selection (as a failed reservation does),
 * and one that does is itself preempted and ends it.  n_reserved = slots
 * held; slot_base stays -1. */

/* Select with chunked prefill under a per-iteration token budget (CS349D
 * Lecture 2, Exercise 9: prompts cut into chunks, SeqWork(n_new = chunk,
 * n_past = tokens already processed), a cap on the tokens of one
 * iteration; static-to-continuous article, chunked prefill: decode first).
 * First Algorithm 1 Select exactly as orca_select_batch (FCFS, max_bs,
 * reservation, break); then, over the selected requests, every decoding
 * request (n_cached >= n_prompt) takes one row while the budget lasts, in
 * batch order, and then every prompting request takes
 * min(n_prompt - n_cached, chunk, budget left) rows, in batch order.
 * Requests left with no row are dropped from batch_idx and become
 * INCREMENT (a reservation made for them is kept); the rest are RUNNING
 * with n_sched set.  token_budget >= 1 and chunk >= 1 (INT32_MAX for no
 * limit: then the result equals orca_select_batch). */
int orca_select_batch_budget(orca_engine *eng, orca_request *pool, int32_t n_pool, int32_t token_budget,
                             int32_t chunk, int32_t *batch_idx, int32_t *n_batch);

/* Run one selectively batched iteration for pool[batch_idx[0..n_batch)]
 * (all RUNNING) on `stream`, then wait for it.  Request i contributes
 * L_i = n_sched rows when n_sched > 0, else n_prompt - n_cached rows when
 * n_cached < n_prompt (prefill) and one row otherwise (decode); n_sched
 * may not exceed that default.  Its rows carry tokens[n_cached + j] at
 * positions n_cached + j.  Rows are flattened in batch order (Figure 5).
 * next_tokens (host, capacity n_batch) receives each request's greedy
 * token (argmax of the last row's logits, lowest index on ties; -1 for a
 * request whose prompt is not complete after this iteration).
 * logits_dev, if not NULL, receives fp32 [n_batch, vocab] logits.
 * Afterwards each request is INCREMENT (or FINISHED, slots released) with
 * n_cached += L_i and n_sched = 0; once its prompt is complete it also
 * gets n_generated += 1 and, unless ORCA_ITER_TEACHER_FORCE, the token is
 * appended to tokens[] (a prompt chunk that leaves part of the prompt
 * unprocessed generates nothing).  On error no request is modified.
 * bf16 engines replay a CUDA graph of the whole forward (captured on first
 * use for each GEMM tile-shape choice and logits pointer, on an internal
 * stream; every kernel reads the iteration's sizes from the device
 * descriptor) unless ORCA_ITER_EAGER is set or profiling is enabled. */
int orca_iteration(orca_engine *eng, orca_request *pool, const int32_t *batch_idx, int32_t n_batch,
                   int32_t flags, int32_t *next_tokens, float *logits_dev, void *stream);

/* orca_iteration in two halves, so that up to two iterations are in flight
 * (Algorithm 1 with n_workers = 2: the scheduler selects and enqueues the
 * next batch, from the requests not RUNNING, while the previous one runs;
 * Orca walk-through, Algorithm 1 and pipelined workers).
 * orca_iteration_submit validates the batch, stages its descriptor and
 * enqueues the forward and the result copy on `stream`, without waiting;
 * the requests stay RUNNING.  Iterations in flight together share one
 * stream, run in submission order, never share a request, and use distinct
 * logits_dev buffers (or NULL).  ORCA_ESTATE
 * when two are already in flight.  `pool` must stay valid until the wait.
 * orca_iteration_wait waits for the oldest iteration in flight and applies
 * its updates as orca_iteration does; *n_batch and batch_idx (capacity
 * max_bs; either may be NULL) receive its batch, next_tokens (capacity
 * max_bs, may be NULL) its tokens.  ORCA_ESTATE when none is in flight.
 * orca_iteration itself is submit + wait and needs none in flight. */
int orca_iteration_submit(orca_engine *eng, orca_request *pool, const int32_t *batch_idx, int32_t n_batch,
                          int32_t flags, float *logits_dev, void *stream);
int orca_iteration_wait(orca_engine *eng, int32_t *n_batch, int32_t *batch_idx, int32_t *next_tokens);

/* Host copy of the last iteration's ragged descriptor: row_off[n_batch+1],
 * per-row position row_pos[n_rows] and K/V slot row_slot[n_rows], and
 * last_row[n_batch].  Any output may be NULL. */
int orca_last_descriptor(const orca_engine *eng, int32_t *n_batch, int32_t *n_rows,
                         int32_t *row_off, int32_t *row_pos, int32_t *row_slot,
                         int32_t *last_row, int32_t capacity);

/* Bytes the last orca_iteration copied host->device (ragged descriptor:
 * request, row and attention work records) and device->host (status word
 * and greedy tokens), and its attention work-item count. */
int orca_last_transfer(const orca_engine *eng, int64_t *h2d_bytes, int64_t *d2h_bytes, int32_t *n_work);

/* Number of kernels the last orca_iteration launched on the device (the
 * kernel nodes of its CUDA graph when it replayed one, else the kernels it
 * enqueued eagerly).  Host call; ORCA_EINVAL on a NULL argument. */
int orca_last_launches(const orca_engine *eng, int32_t *n_kernels);

/* ---------------------------------------------------------------- kernels */
/* Greedy choice over forced logits: out_dev[r] = argmax_c logits_dev[r, c]
 * (lowest index among equal maxima; NaN never wins).  Device pointers;
 * enqueued on `stream`, not synchronised. */
int orca_argmax_rows(const float *logits_dev, int32_t n_rows, int32_t vocab, int32_t *out_dev,
                     void *stream);

/* Self-test of the kernels' failure path.  Every wait inside the library's
 * kernels is bounded (about 2 s); on expiry the kernel ORs 1 into its device
 * status word and returns, so the CUDA context stays usable.  This call
 * enqueues one CTA on `stream` that waits on a barrier nothing completes:
 * after the bound it ORs 1 into *status_dev (a device int32) and ends.
 * Returns ORCA_ECUDA if the launch fails, else ORCA_OK (not synchronised). */
int orca_selftest_wait_timeout(int32_t *status_dev, void *stream);

/* The token-wise Linear of Figure 5 on its own - the kernel orca_iteration
 * runs for the QKV, Attn-Out and MLP Linears and the LM head - exposed for
 * tests and benchmarks:  out[m, n] = f(sum_k A[m, k] W[n, k] + bias[n]),
 *   A [M, K], W [N, K] row-major in `dtype` (device pointers),
 *   bias [N] fp32 device pointer or NULL,
 *   mode ORCA_LINEAR_STORE: out[M, N] in dtype;  ORCA_LINEAR_GELU: out[M, N]
 *   = gelu_tanh(.) in dtype;  ORCA_LINEAR_RESID: out[M, N] fp32 += (.);
 *   ORCA_LINEAR_F32OUT: out[M, N] fp32 (out may be NULL when argmax_keys_dev
 *   is given).
 * bf16 runs on tcgen05 tensor cores and needs K % 64 == 0 and 16-byte
 * aligned A and W; fp32 runs CUDA-core FMA.  The bf16 kernel starts reading
 * W and bias before the work enqueued ahead of it on `stream` has finished
 * (programmatic dependent launch; A and out wait for it), so W and bias must
 * not be written by the library call enqueued just before it on the same
 * stream.
 * scratch / scratch_bytes: optional 256-byte aligned device scratch; with
 *   enough of it (counters, then fp32 partial tiles) a bf16 product with few
 *   output tiles is split along K over more SMs; NULL disables that.
 * argmax_keys_dev: optional device uint64 [M] (bf16, F32OUT only), zeroed by
 *   the call, receiving each row's greedy choice packed as key = (ordered
 *   value bits << 32) | (0xFFFFFFFF - column); key 0 means no column.
 * status_dev: device int32 that kernels OR error bits into (1 wait timeout,
 * 2 bad index, 4 unsupported shape).  Enqueued on `stream`, not synchronised. */
#define ORCA_LINEAR_STORE 0
#define ORCA_LINEAR_GELU 1
#define ORCA_LINEAR_RESID 2
#define ORCA_LINEAR_F32OUT 3
int orca_linear(int32_t dtype, int32_t mode, const void *A, const void *W, const float *bias, void *out,
                int32_t M, int32_t N, int32_t K, void *scratch, size_t scratch_bytes, void *argmax_keys_dev,
                int32_t *status_dev, void *stream);

/* How a bf16 token-wise Linear (orca_linear, and every Linear of an
 * iteration) is planned on a GPU of n_sms SMs, computed on the host by the
 * planner the launches use; no device is touched.  The pages have no
 * counterpart: this is a view of the library's own GEMM planning (which
 * kernel, which tiles, whether tiles are shared out along K) for tests and
 * tools.  with_scratch: the launch has the split scratch the engine gives
 * every Linear (orca_linear: a scratch buffer of at least 3 KB + n_sms / 2 x
 * 512 KB, about 40 MB on 152 SMs).
 * M, N, K > 0, K % 64 == 0, 2 <= n_sms <= 4096, out != NULL, else
 * ORCA_EINVAL. */
typedef struct {
  int32_t kernel;  /* 0 persistent single-CTA tiles, 1 cluster split-K, 2 CTA pairs */
  int32_t tile_m, tile_n; /* output tile: 128 x tile_n, or 256 x 256 for CTA pairs */
  int32_t tiles;   /* output tiles */
  int32_t k_split; /* CTA pairs: 0 whole tiles, 1 equal k-ranges per tile, 2 stream ranges */
  int32_t ranges;  /* k-ranges per tile (cluster S; pairs kind 1: S), or the pairs the
                      stream is cut among (kind 2); else 1 */
  int32_t workers; /* CTAs (kernels 0, 1) or CTA pairs (kernel 2) that take work */
  int32_t code;    /* the plan's small integer (below 64; engine CUDA-graph keys) */
} orca_gemm_plan_info;
int orca_gemm_plan_query(int32_t M, int32_t N, int32_t K, int32_t n_sms, int32_t with_scratch,
                         orca_gemm_plan_info *out);

/* The work of CTA pair `pair` of n_pairs in the CTA-pair GEMM of an M x N x K
 * product, in the order the pair runs it (with_split: tiles may be shared out
 * along K, as with the engine's scratch).  Writes up to max_seg rows of 9
 * int32 into seg (caller-owned): {tile, row tile, column tile, first k-block,
 * end k-block, pairs sharing the tile, this pair's place among them in k
 * order, the shared tile's counter pair (-1 when whole), this piece's partial
 * slot (-1 when whole)}, and returns the number of segments (which may exceed
 * max_seg), or ORCA_EINVAL for M, N, K <= 0, K % 64 != 0, n_pairs <= 0, pair
 * outside [0, n_pairs), max_seg < 0, or seg == NULL with max_seg > 0.  The
 * pages have no counterpart (as orca_gemm_plan_query). */
int orca_gemm_pair_segments(int32_t M, int32_t N, int32_t K, int32_t n_pairs, int32_t with_split, int32_t pair,
                            int32_t *seg, int32_t max_seg);

/* Ragged attention of one layer on its own (Figure 5: each request's
 * queries against its own K/V slots, rows split and merged in place).
 * Batch on the host: request i owns rows row_off[i] .. row_off[i+1]-1
 * (row_off[0] = 0, strictly increasing), whose positions are ctx[i] + j;
 * row j reads keys 0 .. ctx[i] + j of slots slot_base[i] + key.  q and out
 * are [row_off[n_batch], n_heads * head_dim] device arrays; k_layer and
 * v_layer one layer of the K/V pool, [n_heads][n_slots][head_dim], already
 * holding every key the rows read (their own included).  dtype is the
 * element type of q, K/V and out.  workspace: device scratch of at least
 * orca_attention_workspace_bytes(n_batch, rows, ...) bytes, 256-byte
 * aligned, owned by the caller.  The host arrays are read before return;
 * the call synchronises the stream before staging them (pageable copy) and
 * enqueues the kernel without waiting for it. */
int orca_attention_workspace_bytes(int32_t n_batch, int32_t n_rows, int32_t n_heads, int32_t head_dim,
                                   size_t *bytes);
int orca_attention(int32_t dtype, int32_t n_heads, int32_t head_dim, int64_t n_slots, const void *q,
                   const void *k_layer, const void *v_layer, void *out, int32_t n_batch,
                   const int32_t *row_off, const int32_t *ctx, const int64_t *slot_base, void *workspace,
                   size_t ws_bytes, int32_t *status_dev, void *stream);

/* orca_attention without a workspace, for callers that cannot allocate
 * device memory.  The Orca pages have no counterpart to this call: it
 * exists for callers such as a host runtime that owns every device
 * allocation itself, or code running under a fixed memory budget, which must
 * not call cudaMalloc (or anything that allocates device memory) where they
 * run attention.  Arguments are those of orca_attention minus workspace and
 * ws_bytes; the caller still owns q, the K/V slots and out.  The scratch
 * (request and work records, key-split partials, counters) is one 8 MiB
 * array compiled into the library, held on every device that loads it until
 * the process exits.  A batch whose scratch need (what
 * orca_attention_workspace_bytes reports) exceeds 8 MiB returns ORCA_EBATCH
 * before any launch.  The need grows with the number of requests (key-split
 * partials are sized for 16 splits of every request and head), so the cap is
 * 25 requests at 40 heads of 128, 31 at 32 heads of 128 and 164 at 12 heads
 * of 64, whatever their rows.
 * Set-up: the first call on a device (per CUDA context), with that device
 * current, looks up the array's device address and keeps it.  With lazy
 * module loading that lookup may make the driver load the library's device
 * code and reserve the array then, so make the first call early, where the
 * caller may still allocate, and before any stream capture.  If the device's
 * context is replaced (cudaDeviceReset), the next call repeats the set-up.
 * All calls share the array and it keeps the last call's contents; each call
 * clears the counters it uses, and calls that overlap on the GPU (unordered
 * streams) race on it.  Apart from that first-call set-up nothing is
 * allocated: no cudaMalloc, cudaFree or allocating library routine is
 * called. */
int orca_attention_noalloc(int32_t dtype, int32_t n_heads, int32_t head_dim, int64_t n_slots, const void *q,
                           const void *k_layer, const void *v_layer, void *out, int32_t n_batch,
                           const int32_t *row_off, const int32_t *ctx, const int64_t *slot_base,
                           int32_t *status_dev, void *stream);

/* ---------------------------------------------------------------- profiling */
/* Per-kernel-class timing of the iterations that follow; resets the
 * statistics orca_profile_read returns.  No iteration may be in flight.
 *   0: off.
 *   1: CUDA events around every launch; the forward then runs eagerly (no
 *      CUDA graph) and waits for each kernel before the next starts.
 *   2 (bf16 models): launch stamps on the path that runs anyway - every
 *      kernel of the (graph-replayed) forward raises its end time
 *      (%globaltimer) in device memory, and the stamps come back with the
 *      tokens.  A launch's share is its end minus the previous launch's end
 *      (the two attention launches of a layer count as one), so the shares
 *      of an iteration add up to its time on the device.
 * Each launch adds its algorithmic FLOPs and bytes to its class. */
int orca_profile_enable(orca_engine *eng, int32_t enable);
int orca_profile_read(const orca_engine *eng, int32_t kernel_class, orca_kernel_stats *out);

/* Copy the last error message (NUL-terminated, truncated to n). */
int orca_last_error(const orca_engine *eng, char *buf, size_t n);

#ifdef __cplusplus
}
#endif
#endif /* ORCA_H_ */
