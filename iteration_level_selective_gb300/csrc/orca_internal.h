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

namespace orca {

// One request of the batch.
struct ReqInfo {
  int32_t row_off;    // first row of this request
  int32_t n_new;      // L_i: rows this iteration
  int32_t ctx;        // c_i: tokens cached before this iteration
  int32_t slot_base;  // first K/V slot of the request's reservation
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

// Device status word bits (set by kernels, read by the host after the sync).
enum : int32_t {
  kStatusWaitTimeout = 1,   // an mbarrier wait gave up
  kStatusBadIndex = 2,      // a bounds check failed (access skipped)
  kStatusBadShape = 4,      // a launch got an unsupported shape
};

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
};

struct AttnArgs {
  const void *q;          // [n_rows, H]
  const void *k_layer;    // [n_heads][n_slots][D]
  const void *v_layer;
  void *out;              // [n_rows, H]
  const ReqInfo *reqs;
  const RowInfo *rows;
  const AttnWork *work;
  float *part;            // key-split partials [n_work][n_heads][D + 2]
  int32_t *counters;      // [max_bs][n_heads], zero between launches
  int32_t *status;
  int32_t hidden, n_heads, n_rows, split;
  int64_t n_slots;
  float scale_log2;       // log2(e) / sqrt(D)
};

// ---- launch wrappers (defined in the .cu files); all return cudaError_t.
cudaError_t launch_embed(int dtype, const RowInfo *rows, int n_rows,
                         const void *tok_emb, const void *pos_emb, float *x, int H,
                         int vocab, int max_pos, int32_t *status, cudaStream_t st);
cudaError_t launch_layernorm(int dtype, const float *x, const float *g, const float *b, void *out,
                             int n_rows, int H, const ReqInfo *gather_last_row, cudaStream_t st);
cudaError_t launch_argmax(const float *logits, int n_rows, int vocab, int32_t *out, cudaStream_t st);
cudaError_t launch_gemm_simt_f32(const float *A, const float *W, int M, int N, int K,
                                 const EpiParams &epi, cudaStream_t st);
cudaError_t launch_gemm_tc_bf16(const CUtensorMap *tmA, const CUtensorMap *tmW, int M, int N, int K,
                                const EpiParams &epi, int32_t *status, cudaStream_t st);
cudaError_t launch_attention(int dtype, int head_dim, const AttnArgs &args, int n_work, cudaStream_t st);

// GEMM tile shape of the tcgen05 kernel (used by the host to build TMA maps).
constexpr int kTcBM = 128;
constexpr int kTcBN = 128;
constexpr int kTcBK = 64;

}  // namespace orca
