// Internal declarations shared by the host engine and the CUDA kernels.
//
// Device batch descriptor of one selectively batched iteration (Orca
// walk-through, Figure 5): the new tokens of all requests flattened into
// rows 0..n_rows-1 in batch order.  "Split" and "Merge" around attention
// are this index math; no activation is copied.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <utility>

namespace orca {

// Paged K/V: a request's slots are blocks of kKvBlock consecutive slots
// (key k of the request lives in block table[k / kKvBlock] at offset
// k % kKvBlock).  A multiple of the decode chunk and of 8 (TMA swizzle atom).
constexpr int kKvBlock = 32;

// One request of the batch.
struct ReqInfo {
  int32_t row_off;    // first row of this request
  int32_t n_new;      // L_i: rows this iteration
  int32_t ctx;        // c_i: tokens cached before this iteration
  int32_t slot_base;  // first K/V slot of a contiguous reservation
  int32_t block_off;  // paged K/V: first entry of the request's block table, else -1
  int32_t n_blocks;   // paged K/V: entries of that table
};

// One row (token) of the flattened [sum L_i, H] tensor.
struct RowInfo {
  int32_t tok;   // token id
  int32_t pos;   // position c_i + j
  int32_t req;   // batch index i
  int32_t slot;  // K/V slot: slot_base + pos
};

// Work item of the ragged attention launch (grid.x = work items, grid.y = heads).
//   kind 0 (query tile): rows a .. a+b-1 of one request, b <= kQTile, all keys
//                        up to each row's causal limit.
//   kind 1 (key split):  one row a, keys [b*split, min((b+1)*split, pos+1)).
struct AttnWork {
  int32_t kind;
  int32_t req;
  int32_t a;
  int32_t b;
};

constexpr int kQTile = 16;
constexpr int kMaxSplits = 16;  // key splits per decode row, at most

// Per-iteration sizes on the device, read by every kernel of a replayed
// CUDA graph (the host writes them with the request records).
struct DevHeader {
  int32_t n_rows;     // sum L_i
  int32_t n_batch;    // B
  int32_t n_work;     // attention work items of the CUDA-core kernel
  int32_t split;      // keys per decode split
  int32_t n_work_tc;  // attention work items of the tensor-core prefill kernel
  int32_t pad[3];
};

// Prompts of at least this many rows (bf16, head_dim 64 or 128) take the
// tensor-core prefill path, in 128-row query tiles.
constexpr int kTcMinRows = 32;
constexpr int kTcRows = 128;

// Device status word bits (set by kernels, read by the host after the sync).
enum : int32_t {
  kStatusWaitTimeout = 1,   // an mbarrier wait gave up
  kStatusBadIndex = 2,      // a bounds check failed (access skipped)
  kStatusBadShape = 4,      // a launch got an unsupported shape
  kStatusRange = 8,         // a value outside the range a fixed-point sum holds
};

// Row statistics of a LayerNorm input, summed across the CTAs that hold the
// row's columns.  Each CTA's partial sums go in as integers in units of
// kLnStatUnit: integer addition does not depend on the order the atomics
// land in, so the sums (and every result after them) repeat bit for bit from
// run to run.  A partial of magnitude kLnStatMax or more raises kStatusRange
// (2^53 units per partial, at most 2^10 partials: no overflow of 63 bits).
struct LnStats {
  unsigned long long sum;    // sum of x, two's complement
  unsigned long long sumsq;  // sum of x^2
};
constexpr float kLnStatScale = 16777216.0f;  // 1 / kLnStatUnit = 2^24
constexpr float kLnStatMax = 536870912.0f;   // 2^29

// GEMM epilogue: C[m, n] = sum_k A[m, k] W[n, k] + bias[n], then one of:
enum EpiMode : int32_t {
  kEpiQKV = 0,     // n < H -> q[m, n]; H <= n < 2H -> K slot; 2H <= n -> V slot
  kEpiResid = 1,   // x[m, n] += C (fp32 residual stream)
  kEpiGelu = 2,    // u[m, n] = gelu_tanh(C)
  kEpiLogits = 3,  // logits[m, n] = C (fp32)
  kEpiStore = 4,   // out[m, n] = C in the activation dtype
};

struct EpiParams {
  int32_t mode;
  int32_t ldo;            // leading dimension of `out` (elements)
  const float *bias;      // [N] fp32 or nullptr
  void *out;              // q (QKV), x (Resid), u (Gelu), logits (Logits)
  void *k_layer;          // QKV: K slots of this layer [n_heads][n_slots][head_dim]
  void *v_layer;          // QKV: V slots
  const RowInfo *rows;    // QKV: row -> slot
  int32_t hidden, head_dim;
  int64_t n_slots;
  int32_t *status;        // device status word
  unsigned long long *argmax_keys;  // Logits mode: per-row packed (value, index) max, or nullptr
  // LayerNorm folded into the Linear that consumes it (tcgen05 GEMM only).
  // The A operand then holds bf16(gamma * x) of the un-normalised rows x, and
  // LN(x) W + b = rstd * (A W - mean * c) + d with c = sum_k gamma_k W[n, k]
  // and d = b + sum_k beta_k W[n, k] (d is passed as `bias`).
  const LnStats *ln_in;   // [rows] statistics of x over ln_width columns, or nullptr (no fold)
  const float *ln_c;      // [N] c of the fold
  int32_t ln_width;       // LayerNorm width (hidden)
  // Residual mode: the residual rows also feed the next LayerNorm.  The
  // epilogue writes bf16(ln_gamma * x) to ln_xb and adds each row's partial
  // sums of x and x^2 into ln_out (zeroed beforehand).
  const float *ln_gamma;  // [N] gamma of the next LayerNorm, or nullptr
  void *ln_xb;            // bf16 [rows, ldo]
  LnStats *ln_out;        // [rows]
  // Rows of a statistics buffer this launch clears for a later residual
  // epilogue (by the thread that stores the row's column 0), or nullptr.
  LnStats *ln_zero;
  unsigned long long *stamp;  // launch-end stamp (stamp_end), or nullptr
};

// Greedy-choice key of (value, column): larger value first, then lower
// column; NaN never wins.  0 is below every key.
__host__ __device__ __forceinline__ unsigned long long argmax_key(float v, int col) {
  unsigned int u;
#ifdef __CUDA_ARCH__
  u = __float_as_uint(v);
#else
  memcpy(&u, &v, 4);
#endif
  const unsigned int ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned int)col);
}
__host__ __device__ __forceinline__ int argmax_key_col(unsigned long long key) {
  return key == 0ull ? -1 : (int)(0xFFFFFFFFu - (unsigned int)(key & 0xFFFFFFFFull));
}

// Scratch of the split-K tcgen05 GEMM: fp32 partial tiles and one arrival
// counter per output tile (zero between launches).
struct GemmScratch {
  float *partials;
  size_t partial_bytes;
  int32_t *counters;
  int32_t n_counters;
};

struct AttnArgs {
  const void *q;          // [n_rows, H]
  const void *k_layer;    // [n_heads][n_slots][D]
  const void *v_layer;
  void *out;              // [n_rows, H]
  const ReqInfo *reqs;
  const RowInfo *rows;
  const AttnWork *work;
  float *part;            // key-split partials [max_bs * kMaxSplits][n_heads][D + 2]
  int32_t *counters;      // [max_bs][n_heads] split arrivals, zero between launches
  int32_t *ticket;        // [2]: next work item, CTAs done; zero between launches
  int32_t *status;
  int32_t hidden, n_heads, n_rows, split, n_work;
  int64_t n_slots;
  float scale_log2;       // log2(e) / sqrt(D)
  const DevHeader *hdr;   // when set, n_rows / n_work / split come from it
  const int32_t *blocks;  // paged K/V block tables (ReqInfo::block_off >= 0)
  unsigned long long *stamp;  // launch-end stamp (stamp_end), or nullptr
};

// Arguments of the tensor-core prefill attention (work items: kind 2,
// req, a = first row, b = rows, at most kTcRows).
struct TcAttnArgs {
  void *out;              // [n_rows, H] bf16
  const ReqInfo *reqs;
  const AttnWork *work;   // query tiles grouped by request, kind = (group start << 10) | group size
  int32_t *ticket;        // [2], zero between launches
  int32_t *status;
  int32_t hidden, n_heads, n_work;
  const int32_t *n_work_dev;  // when set, the item count comes from it
  const int32_t *blocks;      // paged K/V block tables (ReqInfo::block_off >= 0)
  int64_t n_slots;
  float scale_log2;
  unsigned long long *stamp;  // launch-end stamp (stamp_end), or nullptr
};

// ---- launch wrappers (defined in the .cu files); all return cudaError_t.
// Row counts: `n_rows` on the host, or *n_rows_dev when given (then n_rows
// is only the capacity the fixed grid is sized for).
// ln_g / ln_b / ln_out (optional, together): the first block's LayerNorm of
// each embedded row, written to ln_out in the model dtype.
// stamp_start / stamp (optional): the iteration's start (CTA 0, once the
// kernel may read its inputs) and this launch's end (stamp_end).
cudaError_t launch_embed(int dtype, const RowInfo *rows, int n_rows, const int32_t *n_rows_dev,
                         const void *tok_emb, const void *pos_emb, float *x, int H,
                         int vocab, int max_pos, int32_t *status, const float *ln_g, const float *ln_b,
                         void *ln_out, unsigned long long *stamp_start, unsigned long long *stamp, cudaStream_t st);
// c[n] = sum_k gamma_k W[n, k] and d[n] = bias[n] + sum_k beta_k W[n, k]
// for a bf16 weight W [N, K] (row n = output column n): the vectors of a
// LayerNorm folded into the Linear W.  bias may be nullptr.
cudaError_t launch_ln_fold_vectors(const void *W, const float *gamma, const float *beta, const float *bias, int N,
                                   int K, float *c, float *d, cudaStream_t st);
// zero_keys (optional): per-row argmax keys set to 0 (final LayerNorm, ahead
// of the LM head's fused greedy choice).
cudaError_t launch_layernorm(int dtype, const float *x, const float *g, const float *b, void *out,
                             int n_rows, const int32_t *n_rows_dev, int H, const ReqInfo *gather_last_row,
                             unsigned long long *zero_keys, unsigned long long *stamp, cudaStream_t st);
// One CTA that waits on an mbarrier nothing completes: the bounded wait
// expires and raises kStatusWaitTimeout in *status (the failure path of
// every kernel's waits, exercised without a fault).
cudaError_t launch_wait_selftest(int32_t *status, cudaStream_t st);
// Greedy choice per row: column index to `out`, or its packed argmax_key to `keys` when given.
cudaError_t launch_argmax(const float *logits, int n_rows, int vocab, int32_t *out, unsigned long long *keys,
                          cudaStream_t st);
cudaError_t launch_gemm_simt_f32(const float *A, const float *W, int M, int N, int K,
                                 const EpiParams &epi, cudaStream_t st);
// TMA maps of one weight matrix [N, K] with 128-, 64- and 32-row boxes
// (the GEMM picks its output-tile width per product).
// TMA maps of one bf16 operand [rows, cols] (cols a multiple of 64) for the
// tcgen05 GEMM, viewed in three dimensions {64, rows, cols / 64} with the
// 64-column blocks as the outer dimension (strides: a row, 128 bytes), so one
// box {64, box rows, ks} brings ks k-blocks of 64 columns, each a 128-byte-
// swizzled K-major sub-tile of `box rows` rows.  m[b][k]: box rows 32 / 64 /
// 128 (b = 0, 1, 2) and ks = 1 / 2 / 4 (k = 0, 1, 2).
struct OperandMaps {
  CUtensorMap m[3][3];
  const CUtensorMap *get(int box_rows, int ks) const {
    const int b = box_rows == 32 ? 0 : box_rows == 64 ? 1 : 2;
    const int k = ks == 1 ? 0 : ks == 2 ? 1 : 2;
    return &m[b][k];
  }
};

// C = A W^T on tcgen05.  M rows (or *M_dev when M_dev is given: the grid is
// then sized for max_M rows and idle CTAs exit).  Split-K is used when the
// output has few tiles and `scratch` is large enough.
// How one Linear runs (persistent kernel with tile width bn, or the cluster
// split-K kernel with S CTAs per output tile, kbs k-blocks each, A boxes of
// a_box rows); gemm_plan_code is a small integer unique per plan.
struct GemmPlan {
  bool pair = false;   // CTA-pair kernel (256 x 256 tiles, cta_group::2)
  bool split = false;  // ... with its tiles shared out along K
  bool cluster = false;
  int bn = 128, S = 1, kbs = 0, a_box = 128, ks = 1;
};
// split_scratch: the launch will have scratch enough for the CTA-pair
// kernel's split tiles (the engine's always has).
GemmPlan gemm_plan(int M, int N, int K, bool split_scratch);
// The plan as a small integer (CUDA-graph keys), for launches with scratch.
int gemm_plan_code(int M, int N, int K);
cudaError_t launch_gemm_tc_bf16(const OperandMaps &A, const OperandMaps &W, int M, const int32_t *M_dev, int N,
                                int K, const EpiParams &epi, const GemmScratch &scratch, int32_t *status,
                                cudaStream_t st);
int gemm_sm_count();
// Output-tile width (128 or 256) the tcgen05 GEMM uses for an M x N product.
int gemm_tile_n(int M, int N, int K);
// Per-device one-time set-up of the GEMM kernels (shared-memory limits);
// call before any stream capture.
cudaError_t gemm_prepare();
// Same for the attention kernels.
cudaError_t attention_prepare();
cudaError_t attention_tc_prepare();
bool attention_tc_supported(int dtype, int head_dim);
// tmQ: q buffer [rows, H] (box 64 x 128); tmK / tmV: one layer's K / V slots
// viewed as [n_heads * n_slots, D] (box 64 x 128); tmKb / tmVb: the same
// views with box 64 x kKvBlock (paged block tables).
cudaError_t launch_attention_tc(int head_dim, const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                                const CUtensorMap *tmKb, const CUtensorMap *tmVb, const TcAttnArgs &a, int n_work,
                                cudaStream_t st);
// Persistent over (work item, head) pairs; n_work is the host count, or
// the capacity when args.hdr is set.  early = false: an ordinary launch, which
// starts only once everything before it on `st` has completed (instead of a
// programmatic dependent launch that may start while the previous kernel
// runs).
cudaError_t launch_attention(int dtype, int head_dim, const AttnArgs &args, int n_work, cudaStream_t st,
                             bool early = true);

// GEMM tile shape of the tcgen05 kernel (used by the host to build TMA maps).
constexpr int kTcBM = 128;
constexpr int kTcBN = 128;
constexpr int kTcBK = 64;

// ---- programmatic dependent launch (PDL)
// Every kernel of the iteration is launched with programmatic stream
// serialisation: it calls pdl_trigger() on entry so the next kernel may
// start launching, and pdl_wait() before it touches anything an earlier
// kernel wrote (work before that point may only read weights, the descriptor
// header copied before the forward, or set up shared / tensor memory).
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Launch-end stamp: thread 0 of every CTA, once the CTA's work is done, raises
// *stamp to the current %globaltimer (ns), so that after the launch *stamp is
// the time its last CTA finished.  The engine zeroes the stamps of an
// iteration before its first launch and reads them after the last.
__device__ __forceinline__ void stamp_end(unsigned long long *stamp) {
  if (stamp != nullptr && threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    atomicMax(stamp, t);
  }
}
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

// early = true: programmatic dependent launch (the kernel may start while
// the previous one on `st` runs; its pdl_wait() then waits for it).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_if(bool early, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
  return launch_pdl_if(true, kernel, grid, block, smem, st, std::forward<Args>(args)...);
}

}  // namespace orca
