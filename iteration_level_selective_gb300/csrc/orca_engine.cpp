// Host side of liborca: Algorithm 1 scheduling, the K/V slot pool, the
// ragged batch descriptor, and the launch sequence of one selectively
// batched iteration.  Declarations and contracts: include/orca.h.
//
// Passages followed (page title, section):
//   Orca walk-through "连续批处理完全拆解", Algorithm 1 (Select with max_bs and
//   max_tokens reservation, break on overflow; main loop state updates and
//   release of finished requests) and Figure 5 (flatten to [sum L_i, H],
//   per-request attention, Merge);
//   CS349D Lecture 2, section 4.3 (reservation of max_tokens slots at the
//   first schedule, kept until the request finishes) and section 5.1
//   (prefill rows and decode rows of running requests in one step).
#include "../../include/orca.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <set>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "orca_internal.h"

using namespace orca;

namespace {

constexpr int kMinSplit = 256;   // keys per decode split, at least
// split-K GEMM: counters (one per split tile of the single-CTA kernel, two
// per CTA of the CTA-pair kernel) and fp32 partial tiles of 128 x 256 - up to
// one per SM for the single-CTA kernel, two per SM for the CTA-pair kernel
constexpr int kGemmMaxSms = 192;
constexpr int kGemmCounters = 4 * kGemmMaxSms;
constexpr size_t kGemmPartialBytes = (size_t)2 * kGemmMaxSms * 128 * 256 * 4;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct SlotPool {
  int64_t n_slots = 0;
  int64_t n_rsrv = 0;
  int64_t frag_blocks = 0;
  std::map<int64_t, int64_t> free_;                                   // base -> length
  std::unordered_map<int64_t, std::pair<int64_t, int64_t>> owned;     // id -> (base, n)
  std::unordered_set<int64_t> released;

  void init(int64_t n) {
    n_slots = n;
    free_.clear();
    if (n > 0) free_[0] = n;
  }
  int reserve(int64_t id, int64_t n, int64_t *base) {
    if (n <= 0 || owned.count(id)) return ORCA_EINVAL;
    if (n_rsrv + n > n_slots) return ORCA_ENOSLOTS;
    for (auto it = free_.begin(); it != free_.end(); ++it) {
      if (it->second >= n) {
        const int64_t b = it->first, len = it->second;
        free_.erase(it);
        if (len > n) free_[b + n] = len - n;
        owned[id] = {b, n};
        released.erase(id);
        n_rsrv += n;
        *base = b;
        return ORCA_OK;
      }
    }
    ++frag_blocks;
    return ORCA_ENOSLOTS;
  }
  int release(int64_t id) {
    auto it = owned.find(id);
    if (it == owned.end()) return released.count(id) ? ORCA_EDOUBLE_RELEASE : ORCA_EUNKNOWN_REQ;
    int64_t b = it->second.first, n = it->second.second;
    owned.erase(it);
    released.insert(id);
    n_rsrv -= n;
    auto nx = free_.lower_bound(b);
    if (nx != free_.end() && nx->first == b + n) {  // merge with the next hole
      n += nx->second;
      free_.erase(nx);
    }
    auto pv = free_.lower_bound(b);
    if (pv != free_.begin()) {
      --pv;
      if (pv->first + pv->second == b) {  // merge with the previous hole
        pv->second += n;
        return ORCA_OK;
      }
    }
    free_[b] = n;
    return ORCA_OK;
  }
};

// Paged K/V (CS349D Lecture 2, sections 5.1 and 6.1: memory handed out in
// blocks as requests grow, nothing reserved ahead): the pool's slots are
// n_slots / kKvBlock blocks; a request holds a table of blocks in position
// order; the lowest free block is handed out first.
struct BlockPool {
  int32_t n_blocks = 0;
  std::set<int32_t> free_;
  std::unordered_map<int64_t, std::vector<int32_t>> table;
  std::unordered_set<int64_t> released;

  void init(int32_t n) {
    n_blocks = n;
    free_.clear();
    for (int32_t b = 0; b < n; ++b) free_.insert(b);
  }
  int32_t held(int64_t id) const {
    auto it = table.find(id);
    return it == table.end() ? 0 : (int32_t)it->second.size();
  }
  int64_t used_slots() const { return (int64_t)(n_blocks - (int32_t)free_.size()) * kKvBlock; }
  // Grow the request's table to `total` blocks; false (nothing taken) if the pool is short.
  bool grow(int64_t id, int32_t total) {
    const int32_t need = total - held(id);
    if (need <= 0) return true;
    if ((int32_t)free_.size() < need) return false;
    auto &t = table[id];
    for (int32_t k = 0; k < need; ++k) {
      t.push_back(*free_.begin());
      free_.erase(free_.begin());
    }
    released.erase(id);
    return true;
  }
  int release(int64_t id) {
    auto it = table.find(id);
    if (it == table.end()) return released.count(id) ? ORCA_EDOUBLE_RELEASE : ORCA_EUNKNOWN_REQ;
    for (int32_t b : it->second) free_.insert(b);
    table.erase(it);
    released.insert(id);
    return ORCA_OK;
  }
};

int32_t max_attn_work(int32_t n_batch, int32_t n_rows);
int32_t max_tc_work(int32_t n_batch, int32_t n_rows);
int order_tc_work(AttnWork *w, int32_t n, const ReqInfo *req);

// Iterations one engine keeps in flight at once (Algorithm 1 with up to
// two scheduled batches): each has its own descriptor and result buffers;
// the activations are shared because the batches run in stream order.
constexpr int kMaxInflight = 2;

struct Layout {  // byte offsets into the device workspace
  size_t x, h, q, u, hf, logits, part, counters, gemm_cnt, gemm_part, total;
  // LayerNorms folded into the Linears after them (bf16): the scaled rows
  // bf16(gamma * x), two row-statistics buffers and per layer the vectors
  // c, d of QKV (3H each) and of FC1 (F each)
  size_t xb, ln_a, ln_b, fold;
  size_t out[kMaxInflight], req[kMaxInflight], row[kMaxInflight], work[kMaxInflight], work_tc[kMaxInflight];
  size_t blocks[kMaxInflight];  // paged K/V: the batch's block tables
  int max_work;
};

int elem_bytes(int dtype) { return dtype == ORCA_DTYPE_BF16 ? 2 : 4; }

// Block-table entries one batch may need (paged K/V): each request's
// positions stay below max_pos.
size_t max_table_entries(const orca_config *c) {
  return c->reserve_policy == ORCA_RESERVE_PAGED ? (size_t)c->max_bs * ((c->max_pos + kKvBlock - 1) / kKvBlock) : 1;
}

int check_config(const orca_config *c, std::string *why) {
  if (!c) { *why = "config is NULL"; return ORCA_EINVAL; }
  if (c->n_layers <= 0 || c->hidden <= 0 || c->n_heads <= 0 || c->ffn <= 0 || c->vocab <= 0 ||
      c->max_pos <= 0 || c->max_bs <= 0 || c->max_rows <= 0 || c->n_slots <= 0) {
    *why = "all sizes must be positive";
    return ORCA_EINVAL;
  }
  if (c->dtype != ORCA_DTYPE_F32 && c->dtype != ORCA_DTYPE_BF16) { *why = "unknown dtype"; return ORCA_EINVAL; }
  if (c->hidden % c->n_heads) { *why = "hidden must be a multiple of n_heads"; return ORCA_EINVAL; }
  const int d = c->hidden / c->n_heads;
  if (d != 16 && d != 32 && d != 64 && d != 128) { *why = "head_dim must be 16, 32, 64 or 128"; return ORCA_EINVAL; }
  if (c->hidden % 4 || c->ffn % 4) { *why = "hidden and ffn must be multiples of 4"; return ORCA_EINVAL; }
  if (c->dtype == ORCA_DTYPE_BF16 && (c->hidden % 64 || c->ffn % 64)) {
    *why = "bf16 needs hidden and ffn multiples of 64";
    return ORCA_EINVAL;
  }
  if (c->n_slots >= (int64_t)INT32_MAX) { *why = "n_slots must be < 2^31"; return ORCA_EINVAL; }
  if (c->max_rows < c->max_bs) { *why = "max_rows must be >= max_bs"; return ORCA_EINVAL; }
  if (c->reserve_policy < ORCA_RESERVE_MAX || c->reserve_policy > ORCA_RESERVE_PAGED) {
    *why = "unknown reserve_policy";
    return ORCA_EINVAL;
  }
  if (c->reserve_policy == ORCA_RESERVE_PAGED && c->n_slots % kKvBlock) {
    *why = "paged K/V needs n_slots to be a multiple of ORCA_KV_BLOCK";
    return ORCA_EINVAL;
  }
  return ORCA_OK;
}

// Launch stamps of one iteration: the start, then one end per launch (the
// two attention launches of a layer share one).
size_t stamp_capacity(const orca_config *c) { return 4 + 8 * (size_t)c->n_layers; }

Layout make_layout(const orca_config *c) {
  Layout L{};
  const size_t e = elem_bytes(c->dtype);
  const size_t H = c->hidden, F = c->ffn, R = c->max_rows, B = c->max_bs, V = c->vocab;
  const int d = c->hidden / c->n_heads;
  L.max_work = max_attn_work(c->max_bs, c->max_rows);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
  L.x = take(R * H * 4);
  L.h = take(R * H * e);
  L.q = take(R * H * e);
  L.u = take(R * F * e);
  L.hf = take(B * H * e);
  L.logits = take(B * V * 4);
  for (int k = 0; k < kMaxInflight; ++k) {
    // [0] status word, [1..B] packed argmax keys, then the launch stamps
    L.out[k] = take((B + 1 + stamp_capacity(c)) * 8);
    L.req[k] = take(sizeof(DevHeader) + B * sizeof(ReqInfo));  // header, then request records
    L.row[k] = take(R * sizeof(RowInfo));
    L.work[k] = take((size_t)L.max_work * sizeof(AttnWork));
    L.work_tc[k] = take((size_t)max_tc_work(c->max_bs, c->max_rows) * sizeof(AttnWork));
    L.blocks[k] = take((size_t)max_table_entries(c) * 4);
  }
  L.part = take((size_t)B * kMaxSplits * c->n_heads * (d + 2) * 4);
  L.counters = take((B * c->n_heads + 4) * 4);  // split arrivals, then two work tickets
  L.gemm_cnt = take(kGemmCounters * 4);
  L.gemm_part = take(kGemmPartialBytes);
  const bool fold = c->dtype == ORCA_DTYPE_BF16;
  L.xb = take(fold ? R * H * 2 : 0);
  L.ln_a = take(fold ? R * sizeof(LnStats) : 0);
  L.ln_b = take(fold ? R * sizeof(LnStats) : 0);
  L.fold = take(fold ? (size_t)c->n_layers * 2 * (3 * H + F) * 4 : 0);
  L.total = o;
  return L;
}

// Fold vectors of layer l: 0 = c of QKV, 1 = d of QKV, 2 = c of FC1, 3 = d of FC1.
float *fold_vec(char *ws, const Layout &L, const orca_config &c, int l, int which) {
  const size_t H = c.hidden, F = c.ffn;
  const size_t within = which == 0 ? 0 : which == 1 ? 3 * H : which == 2 ? 6 * H : 6 * H + F;
  const size_t at = (size_t)l * 2 * (3 * H + F) + within;
  return reinterpret_cast<float *>(ws + L.fold) + at;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Keys per decode split.  Rows are split only when the batch's (row, head)
// pairs cannot fill the persistent attention grid: the split then aims at
// about one item per CTA (sum_keys * n_heads / grid), at least kMinSplit
// keys, and at most kMaxSplits splits for the longest row (max_keys).
int attn_split(int max_keys, double sum_keys, int n_heads) {
  const double grid = 8.0 * gemm_sm_count();
  int split = (int)std::min<double>(std::max(1.0, sum_keys * n_heads / grid), 1 << 30);
  split = (split + 63) / 64 * 64;
  split = std::max(split, kMinSplit);
  split = std::max(split, (max_keys + kMaxSplits - 1) / kMaxSplits);
  return split;
}

// Work items of request i (rows row .. row+L-1 at positions ctx .. ctx+L-1):
// query tiles of up to kQTile rows for a multi-row request, key splits for
// a single-row one.  Returns the new item count.
int32_t append_attn_work(AttnWork *w, int32_t n, int32_t i, int32_t row, int32_t L, int32_t ctx, int split) {
  if (L == 1) {
    const int ns = (ctx + 1 + split - 1) / split;
    for (int s = 0; s < ns; ++s) w[n++] = {1, i, row, s};
  } else {
    for (int t = 0; t < L; t += kQTile) w[n++] = {0, i, row + t, std::min(kQTile, L - t)};
  }
  return n;
}

// Order work items longest first (query tiles: rows x keys; key splits:
// keys) so the attention CTAs, which take items from a ticket, finish
// together.
void order_attn_work(AttnWork *w, int32_t n, const ReqInfo *req, int split) {
  auto cost = [&](const AttnWork &x) -> int64_t {
    const ReqInfo &r = req[x.req];
    if (x.kind != 1) return (int64_t)x.b * (r.ctx + (x.a - r.row_off) + x.b);
    const int n_keys = r.ctx + 1;
    return std::min<int64_t>(split, n_keys - (int64_t)x.b * split);
  };
  std::stable_sort(w, w + n, [&](const AttnWork &x, const AttnWork &y) { return cost(x) > cost(y); });
}

// Work items of the tensor-core prefill kernel (kind 2): request i's rows in
// query tiles of up to kTcRows.
int32_t append_tc_work(AttnWork *w, int32_t n, int32_t i, int32_t row, int32_t L) {
  for (int t = 0; t < L; t += kTcRows) w[n++] = {2, i, row + t, std::min(kTcRows, L - t)};
  return n;
}

// Tensor-core items grouped by request (groups with the most work first,
// within a group the query tiles with the most keys first).  Each item's kind
// records its group as (first index << 10) | size: the kernel walks a group's
// tiles head by head, so the CTAs working at one time share K/V in L2.
int order_tc_work(AttnWork *w, int32_t n, const ReqInfo *req) {
  auto cost = [&](const AttnWork &x) -> int64_t {
    const ReqInfo &r = req[x.req];
    return (int64_t)x.b * (r.ctx + (x.a - r.row_off) + x.b);
  };
  int32_t max_req = 0;
  for (int32_t k = 0; k < n; ++k) max_req = std::max(max_req, w[k].req);
  std::vector<int64_t> group_cost(max_req + 1, 0);  // indexed by request
  for (int32_t k = 0; k < n; ++k) group_cost[w[k].req] += cost(w[k]);
  std::stable_sort(w, w + n, [&](const AttnWork &x, const AttnWork &y) {
    if (x.req != y.req) {
      if (group_cost[x.req] != group_cost[y.req]) return group_cost[x.req] > group_cost[y.req];
      return x.req < y.req;
    }
    return cost(x) > cost(y);
  });
  for (int32_t k = 0; k < n;) {
    int32_t e = k;
    while (e < n && w[e].req == w[k].req) ++e;
    if (e - k > 1023 || k >= (1 << 21)) return ORCA_EBATCH;
    for (int32_t j = k; j < e; ++j) w[j].kind = (k << 10) | (e - k);
    k = e;
  }
  return ORCA_OK;
}

int32_t max_tc_work(int32_t n_batch, int32_t n_rows) { return n_rows / kTcMinRows + n_batch; }

int32_t max_attn_work(int32_t n_batch, int32_t n_rows) {
  return (n_rows + kQTile - 1) / kQTile + n_batch + kMaxSplits * n_batch;
}

}  // namespace

struct orca_engine {
  orca_config cfg{};
  bool host_only = true;
  int device = 0;
  int head_dim = 0;
  std::string err;
  SlotPool slots;
  bool paged = false;  // ORCA_RESERVE_PAGED: K/V in blocks handed out on demand
  BlockPool blocks;
  Layout lay{};
  // device side (caller-owned memory)
  std::vector<const void *> w;
  char *kv = nullptr;
  char *ws = nullptr;
  struct Unit { int cls; double flops, bytes; };  // one launch (stamp slot) of the forward
  // one in-flight iteration: pinned host staging and what its wait needs
  struct IterSlot {
    DevHeader *h_hdr = nullptr;  // pinned: header followed by the request records
    ReqInfo *h_req = nullptr;
    RowInfo *h_row = nullptr;
    AttnWork *h_work = nullptr;
    AttnWork *h_work_tc = nullptr;
    unsigned long long *h_out = nullptr;  // [0] status word, [1..] packed argmax keys
    int32_t *h_blocks = nullptr;          // paged K/V: the batch's block tables
    cudaEvent_t done = nullptr;           // recorded after the result copy
    orca_request *pool = nullptr;
    float *logits = nullptr;
    cudaStream_t st = nullptr;
    int32_t flags = 0, n_batch = 0;
    std::vector<int32_t> idx, L;
    std::vector<Unit> units;  // stamps: the launches of this iteration, in stamp order
  };
  IterSlot slot[kMaxInflight];
  int q_head = 0, q_len = 0;  // submitted iterations, oldest first
  // tensor maps (bf16)
  OperandMaps tm_h{}, tm_u{}, tm_hf{}, tm_xb{};  // GEMM activation operands
  CUtensorMap tm_q{};
  std::vector<CUtensorMap> tm_k;      // per layer: K slots as [n_heads * n_slots, head_dim]
  std::vector<CUtensorMap> tm_v;      // per layer: V slots, same view
  std::vector<CUtensorMap> tm_kb, tm_vb;  // per layer: the same views in kKvBlock-row boxes (paged)
  bool attn_tc = false;               // prompts take the tensor-core prefill kernel
  OperandMaps tm_emb{};
  std::vector<OperandMaps> tm_layer;  // 4 per layer: qkv, o, fc1, fc2
  // last descriptor (host copy)
  int32_t last_B = 0, last_N = 0, last_work = 0, last_launches = 0;
  int32_t n_launch = 0;               // kernels enqueued by the current eager forward
  int64_t last_h2d = 0, last_d2h = 0;
  std::vector<int32_t> last_row_off, last_row_pos, last_row_slot, last_last_row;
  // profiling: prof = CUDA-event pairs around eager launches; stamps = every
  // launch of the (graph-replayed) forward raises its end stamp, read back
  // with the tokens.  A dry enqueue (nothing launched) lists the launches'
  // classes and algorithmic work in stamp order.
  bool prof = false;
  bool stamps = false;
  bool dry = false;
  std::vector<Unit> dry_units;
  orca_kernel_stats stats[ORCA_K_COUNT]{};
  struct Pending { int slot, cls; cudaEvent_t a, b; double flops, bytes; };
  std::vector<cudaEvent_t> ev_all, ev_free;  // every event created; those not recorded for a pending launch
  std::vector<Pending> pending;
  int cur_slot = 0;                          // in-flight slot of the iteration being enqueued
  // CUDA graphs of the forward, keyed by GEMM tile choices and logits pointer
  cudaStream_t cap_stream = nullptr;
  // layers with prompt rows on the tensor cores: the decode-attention launch
  // runs on side_stream, forked after the QKV Linear and joined before Attn-Out
  cudaStream_t side_stream = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  struct Graph {
    cudaGraphExec_t exec;
    int32_t n_kernels;  // kernel nodes in the captured forward
  };
  std::map<std::pair<uint64_t, uintptr_t>, Graph> graphs;
};

namespace {

int fail(orca_engine *e, int code, const char *fmt, ...) {
  if (e) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    e->err = buf;
  }
  return code;
}

#define CUDA_TRY(eng, call)                                                                 \
  do {                                                                                      \
    cudaError_t _e = (call);                                                                \
    if (_e != cudaSuccess)                                                                  \
      return fail(eng, ORCA_ECUDA, "%s failed: %s", #call, cudaGetErrorString(_e));         \
  } while (0)

// A kernel launch of the forward: checked, and counted for orca_last_launches.
#define LAUNCH(eng, call)               \
  do {                                  \
    if (!(eng)->dry) CUDA_TRY(eng, call); \
    ++(eng)->n_launch;                  \
  } while (0)

template <typename T> T *ws_ptr(orca_engine *e, size_t off) { return reinterpret_cast<T *>(e->ws + off); }

PFN_cuTensorMapEncodeTiled_v12000 encoder(orca_engine *e) {
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    cudaError_t r = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (r != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
      fail(e, ORCA_ECUDA, "cuTensorMapEncodeTiled is not available");
      return nullptr;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// Row-major bf16 [rows, cols] in boxes of 64 columns x box_rows rows (SW128).
int make_tmap(orca_engine *e, CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols,
              uint32_t box_rows) {
  auto enc = encoder(e);
  if (!enc) return ORCA_ECUDA;
  if (reinterpret_cast<uintptr_t>(base) & 15) return fail(e, ORCA_EINVAL, "TMA base must be 16-byte aligned");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcBK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(e, ORCA_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ORCA_OK;
}

// GEMM operand views: the same row-major bf16 [rows, cols] seen as
// {64 columns, rows, cols / 64 k-blocks}, so that one box of
// {64, box_rows, ks} brings ks consecutive K-major SW128 sub-tiles.  Box
// heights 32 / 64 / 128 by ks 1 / 2 / 4; a ks above cols / 64 is never
// chosen and left unencoded.
int make_operand_maps(orca_engine *e, OperandMaps *m, const void *base, uint64_t rows, uint64_t cols) {
  auto enc = encoder(e);
  if (!enc) return ORCA_ECUDA;
  if (reinterpret_cast<uintptr_t>(base) & 15) return fail(e, ORCA_EINVAL, "TMA base must be 16-byte aligned");
  if (cols % kTcBK) return fail(e, ORCA_EINVAL, "GEMM operand width %llu is no multiple of 64", (unsigned long long)cols);
  *m = OperandMaps{};
  const uint32_t heights[3] = {32, 64, 128};
  const uint32_t kss[3] = {1, 2, 4};
  for (int b = 0; b < 3; ++b)
    for (int k = 0; k < 3; ++k) {
      if (kss[k] > cols / kTcBK) continue;
      cuuint64_t dims[3] = {(cuuint64_t)kTcBK, rows, cols / kTcBK};
      cuuint64_t strides[2] = {cols * 2, (cuuint64_t)kTcBK * 2};
      cuuint32_t box[3] = {(cuuint32_t)kTcBK, heights[b], kss[k]};
      cuuint32_t es[3] = {1, 1, 1};
      CUresult r = enc(&m->m[b][k], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                       es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(e, ORCA_ECUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
    }
  return ORCA_OK;
}

// Weight pointer index helpers (order documented in orca.h).
enum { W_TOK = 0, W_POS = 1, W_LNF_G = 2, W_LNF_B = 3 };
enum { L_LN1_G = 0, L_LN1_B, L_WQKV, L_BQKV, L_WO, L_BO, L_LN2_G, L_LN2_B, L_W1, L_B1, L_W2, L_B2, L_COUNT };
inline const void *lw(const orca_engine *e, int layer, int which) { return e->w[4 + layer * L_COUNT + which]; }

// ---- profiling helpers
cudaEvent_t prof_event(orca_engine *e) {
  if (e->ev_free.empty()) {
    cudaEvent_t ev;
    if (cudaEventCreate(&ev) != cudaSuccess) return nullptr;
    e->ev_all.push_back(ev);
    return ev;
  }
  cudaEvent_t ev = e->ev_free.back();
  e->ev_free.pop_back();
  return ev;
}
void prof_begin(orca_engine *e, cudaStream_t st, cudaEvent_t *a) {
  *a = nullptr;
  if (!e->prof || e->dry) return;
  *a = prof_event(e);
  if (*a) cudaEventRecord(*a, st);
}
void prof_end(orca_engine *e, cudaStream_t st, cudaEvent_t a, int cls, double flops, double bytes) {
  if (e->dry) {
    e->dry_units.push_back({cls, flops, bytes});
    return;
  }
  if (!e->prof || !a) return;
  cudaEvent_t b = prof_event(e);
  if (!b) {
    e->ev_free.push_back(a);
    return;
  }
  cudaEventRecord(b, st);
  e->pending.push_back({e->cur_slot, cls, a, b, flops, bytes});
}
// Add the launches of in-flight slot k (now complete) to the statistics.
void prof_collect(orca_engine *e, int k) {
  std::vector<orca_engine::Pending> keep;
  for (auto &p : e->pending) {
    if (p.slot != k) {
      keep.push_back(p);
      continue;
    }
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      auto &s = e->stats[p.cls];
      s.launches += 1;
      s.total_ms += ms;
      s.flops += p.flops;
      s.bytes += p.bytes;
    }
    e->ev_free.push_back(p.a);
    e->ev_free.push_back(p.b);
  }
  e->pending.swap(keep);
}


// Per-iteration sizes and algorithmic attention work of one iteration.
struct FwdSizes {
  int32_t N, B, n_work, split, n_work_tc;
  double attn_pairs, attn_kv_tokens;
};

// Enqueue the forward of one iteration on `st`: embedding, the layers
// (LN1, QKV + K/V Split, ragged attention, Attn-Out + residual, LN2, FC1 +
// GeLU, FC2 + residual), final LN on the last rows, LM head + greedy choice.
// In bf16 the LayerNorms inside the layers launch nothing of their own: the
// first runs in the embedding kernel, the others are folded into QKV / FC1.
// Two row-statistics buffers alternate; each is cleared by a Linear that runs
// after its last reader and before its next writer in stream order (QKV
// clears ln_a, which Attn-Out fills and FC1 reads; FC1 clears ln_b, which
// FC2 fills and the next QKV reads).
// graph = true: every kernel reads its sizes from the device header and
// grids are fixed (the sequence is being captured into a CUDA graph);
// otherwise sizes are passed by value.  Profiling events only when eager.
int enqueue_forward(orca_engine *e, cudaStream_t st, const FwdSizes &z, float *logits, bool graph, int k) {
  const orca_config &c = e->cfg;
  const int H = c.hidden, F = c.ffn, V = c.vocab, nh = c.n_heads, D = e->head_dim;
  const bool bf16 = c.dtype == ORCA_DTYPE_BF16;
  const size_t eb = elem_bytes(c.dtype);
  const Layout &Ly = e->lay;
  DevHeader *d_hdr = ws_ptr<DevHeader>(e, Ly.req[k]);
  ReqInfo *d_req = reinterpret_cast<ReqInfo *>(d_hdr + 1);
  RowInfo *d_row = ws_ptr<RowInfo>(e, Ly.row[k]);
  AttnWork *d_work = ws_ptr<AttnWork>(e, Ly.work[k]);
  unsigned long long *d_out = ws_ptr<unsigned long long>(e, Ly.out[k]);
  int32_t *status = reinterpret_cast<int32_t *>(d_out);
  unsigned long long *d_keys = d_out + 1;
  GemmScratch scr{ws_ptr<float>(e, Ly.gemm_part), kGemmPartialBytes, ws_ptr<int32_t>(e, Ly.gemm_cnt),
                  4 * std::min(kGemmMaxSms, gemm_sm_count())};
  float *x = ws_ptr<float>(e, Ly.x);
  void *h = e->ws + Ly.h;
  void *q = e->ws + Ly.q;
  void *u = e->ws + Ly.u;
  void *hf = e->ws + Ly.hf;
  const int N = z.N, B = z.B;
  // graph mode: capacities for grid sizing, device pointers for the sizes
  const int32_t *N_dev = graph ? &d_hdr->n_rows : nullptr;
  const int32_t *B_dev = graph ? &d_hdr->n_batch : nullptr;
  const int N_grid = graph ? c.max_rows : N;
  const int B_grid = graph ? c.max_bs : B;

  // bf16: each LayerNorm inside the layers is folded into the Linear after it
  // (the residual epilogue before it writes bf16(gamma * x) and the row sums);
  // the first one runs in the embedding kernel
  const bool fold = bf16;
  void *xb = e->ws + Ly.xb;
  LnStats *ln_a = ws_ptr<LnStats>(e, Ly.ln_a);  // LN2 of each layer
  LnStats *ln_b = ws_ptr<LnStats>(e, Ly.ln_b);  // LN1 of layers 1 ..

  // launch stamps (stamps mode): [0] the start, then launch j's end at 1 + j
  unsigned long long *stamps = e->stamps ? d_out + 1 + c.max_bs : nullptr;
  int su = 0;  // launches (stamp slots) so far
  auto stamp = [&]() { return stamps != nullptr ? stamps + 1 + su : nullptr; };
  if (stamps != nullptr && !e->dry)
    CUDA_TRY(e, cudaMemsetAsync(stamps, 0, stamp_capacity(&c) * sizeof(unsigned long long), st));

  cudaEvent_t ev;
  prof_begin(e, st, &ev);
  LAUNCH(e, launch_embed(c.dtype, d_row, N_grid, N_dev, e->w[W_TOK], e->w[W_POS], x, H, V, c.max_pos, status,
                         fold ? (const float *)lw(e, 0, L_LN1_G) : nullptr,
                         fold ? (const float *)lw(e, 0, L_LN1_B) : nullptr, fold ? h : nullptr, stamps, stamp(), st));
  prof_end(e, st, ev, ORCA_K_EMBED, 0.0, (double)N * H * (2 * eb + 4 + (fold ? eb : 0)));
  ++su;

  const size_t layer_kv = (size_t)2 * nh * c.n_slots * D * eb;
  const double attn_flops = 4.0 * D * z.attn_pairs * nh;
  const double attn_bytes = z.attn_kv_tokens * 2 * H * eb + 2.0 * N * H * eb;
  auto gemm_bytes = [&](double M, double Nn, double K, double out_b) { return (M * K + Nn * K) * eb + M * Nn * out_b; };

  for (int l = 0; l < c.n_layers; ++l) {
    char *kl = e->kv + (size_t)l * layer_kv;
    char *vl = kl + layer_kv / 2;
    const bool fold_in = fold && l > 0;  // LN1 folded into QKV (layer 0: the embedding kernel's LN)
    if (!fold) {  // h = LN1(x)
      prof_begin(e, st, &ev);
      LAUNCH(e, launch_layernorm(c.dtype, x, (const float *)lw(e, l, L_LN1_G), (const float *)lw(e, l, L_LN1_B), h,
                                   N_grid, N_dev, H, nullptr, nullptr, stamp(), st));
      prof_end(e, st, ev, ORCA_K_LAYERNORM, 0.0, (double)N * H * (4 + eb));
      ++su;
    }
    // QKV Linear; K/V scattered to the requests' slots (Split)
    EpiParams ep{};
    ep.mode = kEpiQKV;
    ep.ldo = H;
    ep.bias = fold_in ? fold_vec(e->ws, Ly, c, l, 1) : (const float *)lw(e, l, L_BQKV);
    if (fold_in) {
      ep.ln_in = ln_b;
      ep.ln_c = fold_vec(e->ws, Ly, c, l, 0);
      ep.ln_width = H;
    }
    if (fold) ep.ln_zero = ln_a;  // for this layer's Attn-Out epilogue
    ep.out = q;
    ep.k_layer = kl;
    ep.v_layer = vl;
    ep.rows = d_row;
    ep.hidden = H;
    ep.head_dim = D;
    ep.n_slots = c.n_slots;
    ep.status = status;
    ep.stamp = stamp();
    prof_begin(e, st, &ev);
    if (bf16)
      LAUNCH(e, launch_gemm_tc_bf16(fold_in ? e->tm_xb : e->tm_h, e->tm_layer[4 * l + 0], N, N_dev, 3 * H, H, ep,
                                    scr, status, st));
    else
      LAUNCH(e, launch_gemm_simt_f32((const float *)h, (const float *)lw(e, l, L_WQKV), N, 3 * H, H, ep, st));
    prof_end(e, st, ev, ORCA_K_GEMM_QKV, 2.0 * N * 3 * H * H, gemm_bytes(N, 3.0 * H, H, eb));
    ++su;
    // ragged attention -> h (rows in place: Merge)
    AttnArgs aa{};
    aa.q = q;
    aa.k_layer = kl;
    aa.v_layer = vl;
    aa.out = h;
    aa.reqs = d_req;
    aa.rows = d_row;
    aa.work = d_work;
    aa.part = ws_ptr<float>(e, Ly.part);
    aa.counters = ws_ptr<int32_t>(e, Ly.counters);
    aa.ticket = aa.counters + (size_t)c.max_bs * nh;
    aa.status = status;
    aa.hidden = H;
    aa.n_heads = nh;
    aa.n_rows = N;
    aa.split = z.split;
    aa.n_work = z.n_work;
    aa.n_slots = c.n_slots;
    aa.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    aa.hdr = graph ? d_hdr : nullptr;
    aa.blocks = ws_ptr<int32_t>(e, Ly.blocks[k]);
    aa.stamp = stamp();  // both attention launches of the layer: one stamp
    prof_begin(e, st, &ev);
    // With prompt rows on the tensor cores and 64-dim heads the two attention
    // launches run side by side: the prompt launch follows the QKV Linear as a
    // dependent launch (its CTAs take their SMs first), and the decode launch
    // goes to the side stream as an ordinary launch after the QKV Linear has
    // completed, so it no longer waits for the prompt launch to finish; the
    // streams join before Attn-Out.  With 128-dim heads a decode CTA does not
    // fit on an SM beside a prompt CTA, so the two would only race for the
    // SMs: there the decode launch follows the prompt launch on the same
    // stream as a dependent launch (streaming its older keys while the prompt
    // launch drains).  Measured on GB300: side by side 1.5% faster on the
    // GPT-2-small trace, one after the other 1.6 ms (2%) less attention per
    // prefill-heavy 13B iteration.
    const bool overlap = e->attn_tc && z.n_work_tc > 0 && D < 128;
    if (overlap && !e->dry) {
      CUDA_TRY(e, cudaEventRecord(e->ev_fork, st));
      CUDA_TRY(e, cudaStreamWaitEvent(e->side_stream, e->ev_fork, 0));
    }
    if (e->attn_tc && z.n_work_tc > 0) {  // prompts: tensor-core tiles; then decodes and short prompts
      TcAttnArgs ta{};
      ta.out = h;
      ta.reqs = d_req;
      ta.work = ws_ptr<AttnWork>(e, Ly.work_tc[k]);
      ta.ticket = aa.ticket + 2;
      ta.status = status;
      ta.hidden = H;
      ta.n_heads = nh;
      ta.n_work = z.n_work_tc;
      ta.n_work_dev = graph ? &d_hdr->n_work_tc : nullptr;
      ta.blocks = aa.blocks;
      ta.n_slots = c.n_slots;
      ta.scale_log2 = aa.scale_log2;
      ta.stamp = aa.stamp;
      if (!e->dry)
        CUDA_TRY(e, launch_attention_tc(D, &e->tm_q, &e->tm_k[l], &e->tm_v[l], &e->tm_kb[l], &e->tm_vb[l], ta,
                                        z.n_work_tc, st));
      ++e->n_launch;
    }
    LAUNCH(e, launch_attention(c.dtype, D, aa, graph ? Ly.max_work : z.n_work, overlap ? e->side_stream : st,
                               !overlap));
    if (overlap && !e->dry) {
      CUDA_TRY(e, cudaEventRecord(e->ev_join, e->side_stream));
      CUDA_TRY(e, cudaStreamWaitEvent(st, e->ev_join, 0));
    }
    prof_end(e, st, ev, ORCA_K_ATTENTION, attn_flops, attn_bytes);
    ++su;
    // x += a Wo + bo
    EpiParams eo{};
    eo.mode = kEpiResid;
    eo.ldo = H;
    eo.bias = (const float *)lw(e, l, L_BO);
    eo.out = x;
    eo.status = status;
    eo.stamp = stamp();
    if (fold) {  // the residual feeds LN2: bf16(gamma2 * x) and the row sums
      eo.ln_gamma = (const float *)lw(e, l, L_LN2_G);
      eo.ln_xb = xb;
      eo.ln_out = ln_a;
    }
    prof_begin(e, st, &ev);
    if (bf16)
      LAUNCH(e, launch_gemm_tc_bf16(e->tm_h, e->tm_layer[4 * l + 1], N, N_dev, H, H, eo, scr, status,
                                    st));
    else
      LAUNCH(e, launch_gemm_simt_f32((const float *)h, (const float *)lw(e, l, L_WO), N, H, H, eo, st));
    prof_end(e, st, ev, ORCA_K_GEMM_O, 2.0 * N * H * H, gemm_bytes(N, H, H, fold ? 8 + eb : 8));
    ++su;
    if (!fold) {  // h = LN2(x)
      prof_begin(e, st, &ev);
      LAUNCH(e, launch_layernorm(c.dtype, x, (const float *)lw(e, l, L_LN2_G), (const float *)lw(e, l, L_LN2_B), h,
                                   N_grid, N_dev, H, nullptr, nullptr, stamp(), st));
      prof_end(e, st, ev, ORCA_K_LAYERNORM, 0.0, (double)N * H * (4 + eb));
      ++su;
    }
    // u = GeLU(LN2(x) W1 + b1)
    EpiParams e1{};
    e1.mode = kEpiGelu;
    e1.ldo = F;
    e1.bias = fold ? fold_vec(e->ws, Ly, c, l, 3) : (const float *)lw(e, l, L_B1);
    e1.out = u;
    e1.status = status;
    e1.stamp = stamp();
    if (fold) {
      e1.ln_in = ln_a;
      e1.ln_c = fold_vec(e->ws, Ly, c, l, 2);
      e1.ln_width = H;
      e1.ln_zero = ln_b;  // for this layer's FC2 epilogue
    }
    prof_begin(e, st, &ev);
    if (bf16)
      LAUNCH(e, launch_gemm_tc_bf16(fold ? e->tm_xb : e->tm_h, e->tm_layer[4 * l + 2], N, N_dev, F, H, e1, scr,
                                    status, st));
    else
      LAUNCH(e, launch_gemm_simt_f32((const float *)h, (const float *)lw(e, l, L_W1), N, F, H, e1, st));
    prof_end(e, st, ev, ORCA_K_GEMM_FC1, 2.0 * N * F * H, gemm_bytes(N, F, H, eb));
    ++su;
    // x += u W2 + b2
    EpiParams e2{};
    e2.mode = kEpiResid;
    e2.ldo = H;
    e2.bias = (const float *)lw(e, l, L_B2);
    e2.out = x;
    e2.status = status;
    e2.stamp = stamp();
    const bool feeds_ln1 = fold && l + 1 < c.n_layers;  // the next layer's LN1 (the last feeds the final LN)
    if (feeds_ln1) {
      e2.ln_gamma = (const float *)lw(e, l + 1, L_LN1_G);
      e2.ln_xb = xb;
      e2.ln_out = ln_b;
    }
    prof_begin(e, st, &ev);
    if (bf16)
      LAUNCH(e, launch_gemm_tc_bf16(e->tm_u, e->tm_layer[4 * l + 3], N, N_dev, H, F, e2, scr, status,
                                    st));
    else
      LAUNCH(e, launch_gemm_simt_f32((const float *)u, (const float *)lw(e, l, L_W2), N, H, F, e2, st));
    prof_end(e, st, ev, ORCA_K_GEMM_FC2, 2.0 * N * H * F, gemm_bytes(N, H, F, feeds_ln1 ? 8 + eb : 8));
    ++su;
  }
  // final LayerNorm on each request's last row, LM head (tied), greedy choice
  prof_begin(e, st, &ev);
  // (also zeroes the argmax keys the LM head's epilogue max-reduces into)
  LAUNCH(e, launch_layernorm(c.dtype, x, (const float *)e->w[W_LNF_G], (const float *)e->w[W_LNF_B], hf, B_grid,
                               B_dev, H, d_req, d_keys, stamp(), st));
  prof_end(e, st, ev, ORCA_K_LAYERNORM, 0.0, (double)B * H * (4 + eb));
  ++su;
  EpiParams el{};
  el.mode = kEpiLogits;
  el.ldo = V;
  el.bias = nullptr;
  el.out = logits;
  el.status = status;
  el.argmax_keys = bf16 ? d_keys : nullptr;
  el.stamp = stamp();
  prof_begin(e, st, &ev);
  if (bf16)
    LAUNCH(e, launch_gemm_tc_bf16(e->tm_hf, e->tm_emb, B, B_dev, V, H, el, scr, status, st));
  else
    LAUNCH(e, launch_gemm_simt_f32((const float *)hf, (const float *)e->w[W_TOK], B, V, H, el, st));
  prof_end(e, st, ev, ORCA_K_LM_HEAD, 2.0 * B * V * H, gemm_bytes(B, V, H, logits ? 4 : 0));
  ++su;
  if (!bf16) {
    prof_begin(e, st, &ev);
    LAUNCH(e, launch_argmax(logits, B, V, nullptr, d_keys, st));
    prof_end(e, st, ev, ORCA_K_ARGMAX, 0.0, (double)B * V * 4);
  }
  return ORCA_OK;
}

}  // namespace

// ======================================================================= API

extern "C" {

int orca_kv_pool_bytes(const orca_config *cfg, size_t *bytes) {
  std::string why;
  int rc = check_config(cfg, &why);
  if (rc) return rc;
  if (!bytes) return ORCA_EINVAL;
  *bytes = (size_t)cfg->n_layers * 2 * (size_t)cfg->n_slots * cfg->hidden * elem_bytes(cfg->dtype);
  return ORCA_OK;
}

int orca_workspace_bytes(const orca_config *cfg, size_t *bytes) {
  std::string why;
  int rc = check_config(cfg, &why);
  if (rc) return rc;
  if (!bytes) return ORCA_EINVAL;
  *bytes = make_layout(cfg).total;
  return ORCA_OK;
}

int orca_weight_count(const orca_config *cfg, int32_t *count) {
  std::string why;
  int rc = check_config(cfg, &why);
  if (rc) return rc;
  if (!count) return ORCA_EINVAL;
  *count = 4 + L_COUNT * cfg->n_layers;
  return ORCA_OK;
}

int orca_engine_create(const orca_config *cfg, const void *const *weights, int32_t n_weights, void *kv_pool,
                       size_t kv_bytes, void *workspace, size_t ws_bytes, orca_engine **out) {
  if (!out) return ORCA_EINVAL;
  *out = nullptr;
  std::string why;
  int rc = check_config(cfg, &why);
  if (rc) return rc;
  orca_engine *e = new (std::nothrow) orca_engine();
  if (!e) return ORCA_EINVAL;
  e->cfg = *cfg;
  e->head_dim = cfg->hidden / cfg->n_heads;
  e->slots.init(cfg->n_slots);
  e->paged = cfg->reserve_policy == ORCA_RESERVE_PAGED;
  if (e->paged) e->blocks.init((int32_t)(cfg->n_slots / kKvBlock));
  e->lay = make_layout(cfg);
  const bool any = weights || kv_pool || workspace;
  if (!any) {  // host-only engine: scheduler and slot pool, no CUDA call
    e->host_only = true;
    *out = e;
    return ORCA_OK;
  }
  e->host_only = false;
  size_t need_kv = 0;
  orca_kv_pool_bytes(cfg, &need_kv);
  const int nw = 4 + L_COUNT * cfg->n_layers;
  if (!weights || n_weights != nw || !kv_pool || kv_bytes < need_kv || !workspace || ws_bytes < e->lay.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) || (reinterpret_cast<uintptr_t>(kv_pool) & 15)) {
    delete e;
    return ORCA_EINVAL;
  }
  for (int i = 0; i < nw; ++i) {
    if (!weights[i] || (reinterpret_cast<uintptr_t>(weights[i]) & 15)) {
      delete e;
      return ORCA_EINVAL;
    }
    e->w.push_back(weights[i]);
  }
  e->kv = static_cast<char *>(kv_pool);
  e->ws = static_cast<char *>(workspace);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { delete e; return ORCA_ECUDA; }
  e->device = dev;
  const auto &L = e->lay;
  bool ok = cudaStreamCreateWithFlags(&e->cap_stream, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&e->side_stream, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&e->ev_fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&e->ev_join, cudaEventDisableTiming) == cudaSuccess;
  for (int k = 0; k < kMaxInflight && ok; ++k) {
    orca_engine::IterSlot &S = e->slot[k];
    ok = cudaHostAlloc(&S.h_hdr, sizeof(DevHeader) + sizeof(ReqInfo) * cfg->max_bs, cudaHostAllocDefault) ==
             cudaSuccess &&
         cudaHostAlloc(&S.h_row, sizeof(RowInfo) * cfg->max_rows, cudaHostAllocDefault) == cudaSuccess &&
         cudaHostAlloc(&S.h_work, sizeof(AttnWork) * L.max_work, cudaHostAllocDefault) == cudaSuccess &&
         cudaHostAlloc(&S.h_work_tc, sizeof(AttnWork) * max_tc_work(cfg->max_bs, cfg->max_rows),
                       cudaHostAllocDefault) == cudaSuccess &&
         cudaHostAlloc(&S.h_out, sizeof(unsigned long long) * (cfg->max_bs + 1 + stamp_capacity(cfg)),
                       cudaHostAllocDefault) ==
             cudaSuccess &&
         cudaHostAlloc(&S.h_blocks, max_table_entries(cfg) * 4, cudaHostAllocDefault) == cudaSuccess &&
         cudaEventCreateWithFlags(&S.done, cudaEventDisableTiming) == cudaSuccess &&
         cudaMemset(e->ws + L.out[k], 0, 8) == cudaSuccess;
    if (ok) S.h_req = reinterpret_cast<ReqInfo *>(S.h_hdr + 1);
  }
  ok = ok && cudaMemset(e->ws + L.counters, 0, ((size_t)cfg->max_bs * cfg->n_heads + 4) * 4) == cudaSuccess &&
       cudaMemset(e->ws + L.gemm_cnt, 0, kGemmCounters * 4) == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess;
  if (ok)
    ok = gemm_prepare() == cudaSuccess && attention_prepare() == cudaSuccess && attention_tc_prepare() == cudaSuccess;
  if (!ok) {
    orca_engine_destroy(e);
    return ORCA_ECUDA;
  }
  if (cfg->dtype == ORCA_DTYPE_BF16) {
    const uint64_t H = cfg->hidden, F = cfg->ffn;
    e->tm_layer.resize(4 * cfg->n_layers);
    rc = make_operand_maps(e, &e->tm_h, e->ws + L.h, cfg->max_rows, H);
    if (!rc) rc = make_operand_maps(e, &e->tm_u, e->ws + L.u, cfg->max_rows, F);
    if (!rc) rc = make_operand_maps(e, &e->tm_hf, e->ws + L.hf, cfg->max_bs, H);
    if (!rc) rc = make_operand_maps(e, &e->tm_emb, e->w[W_TOK], cfg->vocab, H);
    e->attn_tc = attention_tc_supported(cfg->dtype, e->head_dim);
    if (!rc && e->attn_tc) {
      rc = make_tmap(e, &e->tm_q, e->ws + L.q, cfg->max_rows, H, kTcBM);
      const size_t layer_kv = (size_t)2 * cfg->n_heads * cfg->n_slots * e->head_dim * 2;
      e->tm_k.resize(cfg->n_layers);
      e->tm_v.resize(cfg->n_layers);
      e->tm_kb.resize(cfg->n_layers);
      e->tm_vb.resize(cfg->n_layers);
      const uint64_t kv_rows = (uint64_t)cfg->n_heads * cfg->n_slots;
      for (int l = 0; l < cfg->n_layers && !rc; ++l) {
        char *kl = e->kv + (size_t)l * layer_kv, *vl = kl + layer_kv / 2;
        rc = make_tmap(e, &e->tm_k[l], kl, kv_rows, e->head_dim, kTcBM);
        if (!rc) rc = make_tmap(e, &e->tm_v[l], vl, kv_rows, e->head_dim, kTcBM);
        if (!rc) rc = make_tmap(e, &e->tm_kb[l], kl, kv_rows, e->head_dim, kKvBlock);
        if (!rc) rc = make_tmap(e, &e->tm_vb[l], vl, kv_rows, e->head_dim, kKvBlock);
      }
    }
    for (int l = 0; l < cfg->n_layers && !rc; ++l) {
      rc = make_operand_maps(e, &e->tm_layer[4 * l + 0], lw(e, l, L_WQKV), 3 * H, H);
      if (!rc) rc = make_operand_maps(e, &e->tm_layer[4 * l + 1], lw(e, l, L_WO), H, H);
      if (!rc) rc = make_operand_maps(e, &e->tm_layer[4 * l + 2], lw(e, l, L_W1), F, H);
      if (!rc) rc = make_operand_maps(e, &e->tm_layer[4 * l + 3], lw(e, l, L_W2), H, F);
    }
    if (!rc) rc = make_operand_maps(e, &e->tm_xb, e->ws + L.xb, cfg->max_rows, H);
    // c and d of every folded LayerNorm, from the weights as they are now (the
    // caller keeps them unchanged for the engine's lifetime)
    if (!rc) {
      bool okf = cudaDeviceSynchronize() == cudaSuccess;
      for (int l = 0; l < cfg->n_layers && okf; ++l)
        okf = launch_ln_fold_vectors(lw(e, l, L_WQKV), (const float *)lw(e, l, L_LN1_G),
                                     (const float *)lw(e, l, L_LN1_B), (const float *)lw(e, l, L_BQKV), 3 * H, H,
                                     fold_vec(e->ws, L, *cfg, l, 0), fold_vec(e->ws, L, *cfg, l, 1),
                                     0) == cudaSuccess &&
              launch_ln_fold_vectors(lw(e, l, L_W1), (const float *)lw(e, l, L_LN2_G),
                                     (const float *)lw(e, l, L_LN2_B), (const float *)lw(e, l, L_B1), F, H,
                                     fold_vec(e->ws, L, *cfg, l, 2), fold_vec(e->ws, L, *cfg, l, 3),
                                     0) == cudaSuccess;
      if (!okf || cudaDeviceSynchronize() != cudaSuccess) rc = ORCA_ECUDA;
    }
    if (rc) {
      orca_engine_destroy(e);
      return rc;
    }
  }
  *out = e;
  return ORCA_OK;
}

int orca_engine_destroy(orca_engine *e) {
  if (!e) return ORCA_EINVAL;
  if (!e->host_only) {
    for (auto &g : e->graphs) cudaGraphExecDestroy(g.second.exec);
    if (e->cap_stream) cudaStreamDestroy(e->cap_stream);
    if (e->side_stream) {
      cudaStreamSynchronize(e->side_stream);
      cudaStreamDestroy(e->side_stream);
    }
    if (e->ev_fork) cudaEventDestroy(e->ev_fork);
    if (e->ev_join) cudaEventDestroy(e->ev_join);
    for (auto &S : e->slot) {
      if (S.done) cudaEventSynchronize(S.done);
      cudaFreeHost(S.h_hdr);
      cudaFreeHost(S.h_row);
      cudaFreeHost(S.h_work);
      cudaFreeHost(S.h_work_tc);
      cudaFreeHost(S.h_out);
      cudaFreeHost(S.h_blocks);
      if (S.done) cudaEventDestroy(S.done);
    }
    for (auto ev : e->ev_all) cudaEventDestroy(ev);
  }
  delete e;
  return ORCA_OK;
}

int orca_kv_reserve(orca_engine *e, int64_t req_id, int32_t n_tokens, int64_t *slot_base) {
  if (!e || !slot_base) return ORCA_EINVAL;
  if (e->paged) return fail(e, ORCA_ESTATE, "paged K/V hands out blocks on demand; nothing to reserve");
  int rc = e->slots.reserve(req_id, n_tokens, slot_base);
  if (rc == ORCA_ENOSLOTS) return fail(e, rc, "cannot reserve %d slots (n_rsrv %lld of %lld)", n_tokens,
                                       (long long)e->slots.n_rsrv, (long long)e->slots.n_slots);
  if (rc) return fail(e, rc, "invalid reservation for request %lld", (long long)req_id);
  return ORCA_OK;
}

int orca_kv_release(orca_engine *e, int64_t req_id) {
  if (!e) return ORCA_EINVAL;
  int rc = e->paged ? e->blocks.release(req_id) : e->slots.release(req_id);
  if (rc) return fail(e, rc, "release of request %lld: %s", (long long)req_id,
                      rc == ORCA_EDOUBLE_RELEASE ? "already released" : "unknown request");
  return ORCA_OK;
}

int orca_kv_stats(const orca_engine *e, int64_t *n_rsrv, int64_t *n_free_blocks, int64_t *frag_blocks) {
  if (!e) return ORCA_EINVAL;
  if (n_rsrv) *n_rsrv = e->paged ? e->blocks.used_slots() : e->slots.n_rsrv;
  if (n_free_blocks) *n_free_blocks = e->paged ? (int64_t)e->blocks.free_.size() : (int64_t)e->slots.free_.size();
  if (frag_blocks) *frag_blocks = e->paged ? 0 : e->slots.frag_blocks;
  return ORCA_OK;
}

namespace {

// Rows a selected request contributes when nothing narrower was scheduled:
// its known tokens (prompt + generated) not yet in the K/V slots - the rest
// of the prompt, one decode row, or everything after a preemption.
int32_t known_len(const orca_request &r) { return r.n_prompt + r.n_generated; }
int32_t default_rows(const orca_request &r) { return std::max(1, known_len(r) - r.n_cached); }
// A request that runs one decode row (its prompt and all but the last
// generated token are in the slots).
bool decoding(const orca_request &r) { return r.n_generated > 0 && r.n_cached == known_len(r) - 1; }

// Slots a request reserves at first schedule (CS349D Lecture 2, section
// 6.1): max_tokens (Orca), or its true final length n_prompt + out_len
// rounded up to a power of two, or that length itself; never above
// max_tokens, the most a request can hold.
int32_t reserve_size(int policy, const orca_request &r) {
  const int64_t len = std::min<int64_t>((int64_t)r.n_prompt + r.out_len, r.max_tokens);
  if (policy == ORCA_RESERVE_ORACLE) return (int32_t)len;
  if (policy == ORCA_RESERVE_POW2) {
    int64_t p = 1;
    while (p < len) p <<= 1;
    return (int32_t)std::min<int64_t>(p, r.max_tokens);
  }
  return r.max_tokens;
}

// Algorithm 1 Select (Orca walk-through, Algorithm 1): candidates are the
// non-RUNNING, unfinished requests in (arrival, req_id) order; at most max_bs;
// an INITIATION request first reserves max_tokens slots and a failed
// reservation ends the selection.  Fills batch_idx; states are not changed.
void preempt(orca_engine *e, orca_request &v) {
  e->blocks.release(v.req_id);
  v.n_cached = 0;
  v.n_reserved = 0;
  v.n_sched = 0;
  v.state = ORCA_INITIATION;
}

int select_fcfs(orca_engine *e, orca_request *pool, int32_t n_pool, int32_t *batch_idx, int32_t *nb_out,
                int64_t chunk_cap) {
  *nb_out = 0;
  std::vector<int32_t> cand;
  cand.reserve(n_pool);
  for (int32_t i = 0; i < n_pool; ++i) {
    const int s = pool[i].state;
    if (s == ORCA_INITIATION || s == ORCA_INCREMENT) cand.push_back(i);
    else if (s != ORCA_RUNNING && s != ORCA_FINISHED)
      return fail(e, ORCA_EINVAL, "request %lld has unknown state %d", (long long)pool[i].req_id, s);
  }
  std::stable_sort(cand.begin(), cand.end(), [&](int32_t a, int32_t b) {
    if (pool[a].arrival != pool[b].arrival) return pool[a].arrival < pool[b].arrival;
    return pool[a].req_id < pool[b].req_id;
  });
  int32_t nb = 0;
  std::vector<char> in_batch(e->paged ? n_pool : 0, 0);
  for (int32_t idx : cand) {
    if (nb == e->cfg.max_bs) break;
    orca_request &r = pool[idx];
    if (r.state == ORCA_INITIATION &&
        (r.max_tokens < r.n_prompt || r.n_prompt <= 0 || r.out_len <= 0 || r.n_generated < 0))
      return fail(e, ORCA_EINVAL, "request %lld: need 0 < n_prompt <= max_tokens and out_len > 0",
                  (long long)r.req_id);
    if (e->paged) {
      const int64_t rows = std::min<int64_t>(default_rows(r), chunk_cap);
      const int32_t total = (int32_t)((r.n_cached + rows + kKvBlock - 1) / kKvBlock);
      while ((int32_t)e->blocks.free_.size() < total - e->blocks.held(r.req_id)) {
        int32_t v = -1;  // the latest arrival that holds blocks and is neither batched nor running
        for (int32_t i = 0; i < n_pool; ++i) {
          const orca_request &q = pool[i];
          if (i == idx || in_batch[i] || q.state != ORCA_INCREMENT || e->blocks.held(q.req_id) == 0) continue;
          if (v < 0 || q.arrival > pool[v].arrival || (q.arrival == pool[v].arrival && q.req_id > pool[v].req_id))
            v = i;
        }
        if (v < 0) break;
        preempt(e, pool[v]);
      }
      if (!e->blocks.grow(r.req_id, total)) {
        if (e->blocks.held(r.req_id) > 0) preempt(e, r);  // cannot grow even alone: recompute later
        break;                                            // as a failed reservation: stop selecting
      }
      r.n_reserved = e->blocks.held(r.req_id) * kKvBlock;
      r.slot_base = -1;
      r.state = ORCA_INCREMENT;
      in_batch[idx] = 1;
      batch_idx[nb++] = idx;
      continue;
    }
    if (r.state == ORCA_INITIATION) {
      int64_t base = -1;
      const int32_t want = reserve_size(e->cfg.reserve_policy, r);
      const int rc = e->slots.reserve(r.req_id, want, &base);
      if (rc == ORCA_ENOSLOTS) break;  // Algorithm 1: stop selecting, never skip
      if (rc) return fail(e, rc, "request %lld already holds a reservation", (long long)r.req_id);
      r.slot_base = base;
      r.n_reserved = want;
      r.state = ORCA_INCREMENT;  // admitted: holds its slots from now on
    }
    batch_idx[nb++] = idx;
  }
  *nb_out = nb;
  return ORCA_OK;
}

}  // namespace

int orca_kv_usage(const orca_engine *e, const orca_request *pool, int32_t n_pool, int64_t *reserved,
                  int64_t *stored) {
  if (!e || n_pool < 0 || (n_pool > 0 && !pool)) return ORCA_EINVAL;
  int64_t st = 0;
  for (int32_t i = 0; i < n_pool; ++i) {
    const orca_request &r = pool[i];
    if (r.state != ORCA_INITIATION && r.state != ORCA_FINISHED && (r.slot_base >= 0 || r.n_reserved > 0))
      st += r.n_cached;
  }
  if (reserved) *reserved = e->paged ? e->blocks.used_slots() : e->slots.n_rsrv;
  if (stored) *stored = st;
  return ORCA_OK;
}

int orca_select_batch(orca_engine *e, orca_request *pool, int32_t n_pool, int32_t *batch_idx, int32_t *n_batch) {
  if (!e || !n_batch || (n_pool > 0 && (!pool || !batch_idx)) || n_pool < 0) return ORCA_EINVAL;
  *n_batch = 0;
  int32_t nb = 0;
  const int rc = select_fcfs(e, pool, n_pool, batch_idx, &nb, INT32_MAX);
  if (rc) return rc;
  for (int32_t i = 0; i < nb; ++i) {
    orca_request &r = pool[batch_idx[i]];
    r.n_sched = default_rows(r);
    r.state = ORCA_RUNNING;
  }
  *n_batch = nb;
  return ORCA_OK;
}

int orca_select_batch_budget(orca_engine *e, orca_request *pool, int32_t n_pool, int32_t token_budget,
                             int32_t chunk, int32_t *batch_idx, int32_t *n_batch) {
  if (!e || !n_batch || (n_pool > 0 && (!pool || !batch_idx)) || n_pool < 0) return ORCA_EINVAL;
  *n_batch = 0;
  if (token_budget < 1 || chunk < 1) return fail(e, ORCA_EINVAL, "token_budget and chunk must be >= 1");
  int32_t nb = 0;
  const int rc = select_fcfs(e, pool, n_pool, batch_idx, &nb, chunk);
  if (rc) return rc;
  int64_t left = token_budget;
  std::vector<int32_t> rows(nb, 0);
  for (int32_t i = 0; i < nb; ++i) {  // decodes first: one row each
    const orca_request &r = pool[batch_idx[i]];
    if (decoding(r) && left >= 1) {
      rows[i] = 1;
      left -= 1;
    }
  }
  for (int32_t i = 0; i < nb; ++i) {  // then prompt chunks (and recomputations), in batch order
    const orca_request &r = pool[batch_idx[i]];
    if (!decoding(r)) {
      const int64_t n = std::min<int64_t>(std::min<int64_t>(default_rows(r), chunk), left);
      rows[i] = (int32_t)n;
      left -= n;
    }
  }
  int32_t out = 0;
  for (int32_t i = 0; i < nb; ++i) {
    orca_request &r = pool[batch_idx[i]];
    if (rows[i] == 0) continue;  // admitted or waiting, but no row this iteration (state stays INCREMENT)
    r.n_sched = rows[i];
    r.state = ORCA_RUNNING;
    batch_idx[out++] = batch_idx[i];
  }
  *n_batch = out;
  return ORCA_OK;
}

int orca_iteration_submit(orca_engine *e, orca_request *pool, const int32_t *batch_idx, int32_t n_batch,
                          int32_t flags, float *logits_dev, void *stream) {
  if (!e) return ORCA_EINVAL;
  if (e->host_only) return fail(e, ORCA_ESTATE, "host-only engine has no device side");
  const orca_config &c = e->cfg;
  if (n_batch <= 0) return fail(e, ORCA_EINVAL, "empty batch");
  if (n_batch > c.max_bs) return fail(e, ORCA_EBATCH, "n_batch %d > max_bs %d", n_batch, c.max_bs);
  if (!pool || !batch_idx) return fail(e, ORCA_EINVAL, "NULL argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (e->q_len == kMaxInflight) return fail(e, ORCA_ESTATE, "%d iterations already in flight", kMaxInflight);
  if (e->q_len > 0 && e->slot[e->q_head].st != st)
    return fail(e, ORCA_EINVAL, "iterations in flight together must use one stream");
  for (int j = 0; j < e->q_len && logits_dev; ++j)
    if (e->slot[(e->q_head + j) % kMaxInflight].logits == logits_dev)
      return fail(e, ORCA_EINVAL, "iterations in flight together need distinct logits buffers");
  const int k = (e->q_head + e->q_len) % kMaxInflight;
  orca_engine::IterSlot &S = e->slot[k];
  e->cur_slot = k;
  const int H = c.hidden, F = c.ffn, V = c.vocab, nh = c.n_heads;
  const bool bf16 = c.dtype == ORCA_DTYPE_BF16;

  // ---- ragged descriptor (host): rows in batch order, Figure 5
  std::vector<int32_t> L(n_batch);
  int32_t N = 0, max_keys = 0;
  double sum_keys = 0.0;
  for (int32_t i = 0; i < n_batch; ++i) {
    const orca_request &r = pool[batch_idx[i]];
    if (r.state != ORCA_RUNNING) return fail(e, ORCA_EINVAL, "request %lld is not RUNNING", (long long)r.req_id);
    if (!r.tokens || (!e->paged && r.slot_base < 0))
      return fail(e, ORCA_EINVAL, "request %lld has no tokens or slots", (long long)r.req_id);
    if (r.n_cached < 0) return fail(e, ORCA_EINVAL, "request %lld: negative n_cached", (long long)r.req_id);
    const int32_t dflt = default_rows(r);
    if (r.n_sched < 0 || r.n_sched > dflt)
      return fail(e, ORCA_EINVAL, "request %lld: n_sched %d outside 0..%d", (long long)r.req_id, r.n_sched, dflt);
    L[i] = r.n_sched > 0 ? r.n_sched : dflt;
    // slots the request holds
    const int64_t cap = e->paged ? (int64_t)e->blocks.held(r.req_id) * kKvBlock
                                 : (r.n_reserved > 0 ? r.n_reserved : r.max_tokens);
    const int64_t end = (int64_t)r.n_cached + L[i];
    if (end > cap || end > r.max_tokens || end > c.max_pos || end > (int64_t)r.n_prompt + r.out_len)
      return fail(e, ORCA_EINVAL, "request %lld: position %lld beyond its slots, max_pos or its buffer",
                  (long long)r.req_id, (long long)end);
    if (!e->paged && r.slot_base + cap > c.n_slots)
      return fail(e, ORCA_EINVAL, "request %lld: slots beyond n_slots", (long long)r.req_id);
    for (int j = 0; j < e->q_len; ++j) {  // a request is in at most one batch in flight
      const orca_engine::IterSlot &O = e->slot[(e->q_head + j) % kMaxInflight];
      for (int32_t x : O.idx)
        if (O.pool == pool && x == batch_idx[i])
          return fail(e, ORCA_EINVAL, "request %lld is already in an iteration in flight", (long long)r.req_id);
    }
    N += L[i];
    if (N > c.max_rows) return fail(e, ORCA_EBATCH, "sum L_i > max_rows %d", c.max_rows);
    if (L[i] == 1) {
      max_keys = std::max<int32_t>(max_keys, r.n_cached + 1);
      sum_keys += r.n_cached + 1;
    }
  }
  const int split = attn_split(max_keys, sum_keys, nh);
  int32_t n_work = 0, n_work_tc = 0;
  int32_t row = 0, n_entries = 0;
  for (int32_t i = 0; i < n_batch; ++i) {
    const orca_request &r = pool[batch_idx[i]];
    const std::vector<int32_t> *table = nullptr;
    if (e->paged) {  // the request's block table, for the kernels and the row slots
      table = &e->blocks.table.at(r.req_id);
      S.h_req[i] = {row, L[i], r.n_cached, -1, n_entries, (int32_t)table->size()};
      std::copy(table->begin(), table->end(), S.h_blocks + n_entries);
      n_entries += (int32_t)table->size();
    } else {
      S.h_req[i] = {row, L[i], r.n_cached, (int32_t)r.slot_base, -1, 0};
    }
    for (int32_t j = 0; j < L[i]; ++j) {
      const int32_t pos = r.n_cached + j;
      const int32_t tok = r.tokens[pos];
      if (tok < 0 || tok >= V) return fail(e, ORCA_EINVAL, "token id %d out of range", tok);
      const int32_t slot = table ? (*table)[pos / kKvBlock] * kKvBlock + pos % kKvBlock : (int32_t)(r.slot_base + pos);
      S.h_row[row + j] = {tok, pos, i, slot};
    }
    if (e->attn_tc && L[i] >= kTcMinRows)
      n_work_tc = append_tc_work(S.h_work_tc, n_work_tc, i, row, L[i]);
    else
      n_work = append_attn_work(S.h_work, n_work, i, row, L[i], r.n_cached, split);
    row += L[i];
  }
  order_attn_work(S.h_work, n_work, S.h_req, split);
  if (order_tc_work(S.h_work_tc, n_work_tc, S.h_req))
    return fail(e, ORCA_EBATCH, "a prompt has more than 1023 query tiles");
  // host copy for orca_last_descriptor / orca_last_transfer
  e->last_B = n_batch;
  e->last_N = N;
  e->last_work = n_work;
  e->last_h2d = (int64_t)sizeof(DevHeader) + (int64_t)sizeof(ReqInfo) * n_batch + (int64_t)sizeof(RowInfo) * N +
                (int64_t)sizeof(AttnWork) * (n_work + n_work_tc) + (int64_t)sizeof(int32_t) * n_entries;
  e->last_row_off.assign(n_batch + 1, 0);
  e->last_last_row.resize(n_batch);
  for (int32_t i = 0; i < n_batch; ++i) {
    e->last_row_off[i + 1] = e->last_row_off[i] + L[i];
    e->last_last_row[i] = e->last_row_off[i + 1] - 1;
  }
  e->last_row_pos.resize(N);
  e->last_row_slot.resize(N);
  for (int32_t r = 0; r < N; ++r) {
    e->last_row_pos[r] = S.h_row[r].pos;
    e->last_row_slot[r] = S.h_row[r].slot;
  }

  // ---- device work, all on `st`
  CUDA_TRY(e, cudaSetDevice(e->device));
  const Layout &Ly = e->lay;
  DevHeader *d_hdr = ws_ptr<DevHeader>(e, Ly.req[k]);
  RowInfo *d_row = ws_ptr<RowInfo>(e, Ly.row[k]);
  AttnWork *d_work = ws_ptr<AttnWork>(e, Ly.work[k]);
  unsigned long long *d_out = ws_ptr<unsigned long long>(e, Ly.out[k]);
  *S.h_hdr = DevHeader{N, n_batch, n_work, split, n_work_tc, {0, 0, 0}};
  CUDA_TRY(e, cudaMemcpyAsync(d_hdr, S.h_hdr, sizeof(DevHeader) + sizeof(ReqInfo) * n_batch, cudaMemcpyHostToDevice, st));
  CUDA_TRY(e, cudaMemcpyAsync(d_row, S.h_row, sizeof(RowInfo) * N, cudaMemcpyHostToDevice, st));
  if (n_work > 0)
    CUDA_TRY(e, cudaMemcpyAsync(d_work, S.h_work, sizeof(AttnWork) * n_work, cudaMemcpyHostToDevice, st));
  if (n_work_tc > 0)
    CUDA_TRY(e, cudaMemcpyAsync(ws_ptr<AttnWork>(e, Ly.work_tc[k]), S.h_work_tc, sizeof(AttnWork) * n_work_tc,
                                cudaMemcpyHostToDevice, st));
  if (n_entries > 0)
    CUDA_TRY(e, cudaMemcpyAsync(ws_ptr<int32_t>(e, Ly.blocks[k]), S.h_blocks, sizeof(int32_t) * n_entries,
                                cudaMemcpyHostToDevice, st));

  FwdSizes z{N, n_batch, n_work, split, n_work_tc, 0.0, 0.0};
  for (int32_t i = 0; i < n_batch; ++i) {  // attention algorithmic work: pairs and unique K/V tokens
    const double cc = pool[batch_idx[i]].n_cached, l = L[i];
    z.attn_pairs += l * cc + l * (l + 1) / 2;
    z.attn_kv_tokens += cc + l;
  }
  // bf16: the LM head's epilogue takes the greedy choice itself and writes
  // logits only when the caller asks for them; fp32: logits, then argmax.
  float *logits = logits_dev ? logits_dev : (bf16 ? nullptr : ws_ptr<float>(e, Ly.logits));
  const bool use_graph = bf16 && !e->prof && !(flags & ORCA_ITER_EAGER);
  S.units.clear();
  if (e->stamps) {  // the launches' classes and algorithmic work, in stamp order (nothing is launched)
    e->dry = true;
    e->dry_units.clear();
    const int rc = enqueue_forward(e, st, z, logits, use_graph, k);
    e->dry = false;
    if (rc) return rc;
    S.units = e->dry_units;
  }
  if (use_graph) {
    // graphs differ in their GEMM plans, in whether the tensor-core prompt
    // attention runs at all, and in the in-flight slot they read
    const uint64_t key = (uint64_t)gemm_plan_code(N, 3 * H, H) | ((uint64_t)gemm_plan_code(N, H, H) << 6) |
                         ((uint64_t)gemm_plan_code(N, F, H) << 12) | ((uint64_t)gemm_plan_code(N, H, F) << 18) |
                         ((uint64_t)gemm_plan_code(n_batch, V, H) << 24) | ((uint64_t)(n_work_tc > 0) << 30) |
                         ((uint64_t)k << 31) | ((uint64_t)e->stamps << 32);
    const auto gk = std::make_pair(key, reinterpret_cast<uintptr_t>(logits));
    auto it = e->graphs.find(gk);
    if (it == e->graphs.end()) {
      CUDA_TRY(e, cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeThreadLocal));
      const int rc = enqueue_forward(e, e->cap_stream, z, logits, true, k);
      cudaGraph_t g = nullptr;
      const cudaError_t ce = cudaStreamEndCapture(e->cap_stream, &g);
      if (rc) {
        if (g) cudaGraphDestroy(g);
        return rc;
      }
      if (ce != cudaSuccess) return fail(e, ORCA_ECUDA, "graph capture failed: %s", cudaGetErrorString(ce));
      int32_t n_kernels = 0;
      size_t n_nodes = 0;
      if (cudaGraphGetNodes(g, nullptr, &n_nodes) == cudaSuccess && n_nodes > 0) {
        std::vector<cudaGraphNode_t> nodes(n_nodes);
        if (cudaGraphGetNodes(g, nodes.data(), &n_nodes) == cudaSuccess)
          for (size_t q = 0; q < n_nodes; ++q) {
            cudaGraphNodeType t;
            if (cudaGraphNodeGetType(nodes[q], &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++n_kernels;
          }
      }
      cudaGraphExec_t ex = nullptr;
      const cudaError_t ie = cudaGraphInstantiate(&ex, g, 0);
      cudaGraphDestroy(g);
      if (ie != cudaSuccess) return fail(e, ORCA_ECUDA, "graph instantiate failed: %s", cudaGetErrorString(ie));
      it = e->graphs.emplace(gk, orca_engine::Graph{ex, n_kernels}).first;
    }
    CUDA_TRY(e, cudaGraphLaunch(it->second.exec, st));
    e->last_launches = it->second.n_kernels;
  } else {
    e->n_launch = 0;
    const int rc = enqueue_forward(e, st, z, logits, false, k);
    if (rc) return rc;
    e->last_launches = e->n_launch;
  }
  if (flags & ORCA_ITER_SELFTEST_TIMEOUT)  // test hook: a bounded wait expires on the status word
    CUDA_TRY(e, launch_wait_selftest(reinterpret_cast<int32_t *>(d_out), st));
  // the status word and the tokens (with stamps: up to the last stamp, in one copy)
  const size_t out_words = e->stamps ? (size_t)e->cfg.max_bs + 2 + S.units.size() : (size_t)n_batch + 1;
  CUDA_TRY(e, cudaMemcpyAsync(S.h_out, d_out, sizeof(unsigned long long) * out_words, cudaMemcpyDeviceToHost, st));
  e->last_d2h = (int64_t)(sizeof(unsigned long long) * out_words);
  CUDA_TRY(e, cudaEventRecord(S.done, st));
  S.pool = pool;
  S.logits = logits_dev;
  S.st = st;
  S.flags = flags;
  S.n_batch = n_batch;
  S.idx.assign(batch_idx, batch_idx + n_batch);
  S.L = std::move(L);
  ++e->q_len;
  return ORCA_OK;
}

int orca_iteration_wait(orca_engine *e, int32_t *n_batch, int32_t *batch_idx, int32_t *next_tokens) {
  if (!e) return ORCA_EINVAL;
  if (e->q_len == 0) return fail(e, ORCA_ESTATE, "no iteration in flight");
  const int k = e->q_head;
  orca_engine::IterSlot &S = e->slot[k];
  const int V = e->cfg.vocab;
  // the oldest iteration leaves the queue whatever its outcome
  e->q_head = (e->q_head + 1) % kMaxInflight;
  --e->q_len;
  if (n_batch) *n_batch = S.n_batch;
  if (batch_idx) std::copy(S.idx.begin(), S.idx.end(), batch_idx);
  CUDA_TRY(e, cudaEventSynchronize(S.done));
  if (e->prof) prof_collect(e, k);
  if (e->stamps && !S.units.empty()) {  // each launch's share: its end minus the previous end
    const unsigned long long *ts = S.h_out + 1 + e->cfg.max_bs;
    unsigned long long prev = ts[0];
    for (size_t j = 0; j < S.units.size(); ++j) {
      const unsigned long long t = ts[1 + j];
      const double ms = (prev != 0 && t > prev) ? (double)(t - prev) * 1e-6 : 0.0;
      if (t > prev) prev = t;
      orca_kernel_stats &ks = e->stats[S.units[j].cls];
      ks.launches += 1;
      ks.total_ms += ms;
      ks.flops += S.units[j].flops;
      ks.bytes += S.units[j].bytes;
    }
  }
  const int32_t dev_status = (int32_t)(S.h_out[0] & 0xFFFFFFFFull);
  if (dev_status != 0) {
    int32_t *status = ws_ptr<int32_t>(e, e->lay.out[k]);
    cudaMemsetAsync(status, 0, 4, S.st);
    cudaStreamSynchronize(S.st);
    return fail(e, ORCA_EDEVICE, "device status word 0x%x (1 wait timeout, 2 bad index, 4 bad shape, 8 out of range)",
                dev_status);
  }
  for (int32_t i = 0; i < S.n_batch; ++i) {
    const int32_t tok = argmax_key_col(S.h_out[1 + i]);
    if (tok < 0 || tok >= V) return fail(e, ORCA_EDEVICE, "argmax produced no token (NaN logits?)");
  }
  // ---- Algorithm 1 main loop: returned requests become INCREMENT; finished ones release their slots
  for (int32_t i = 0; i < S.n_batch; ++i) {
    orca_request &r = S.pool[S.idx[i]];
    const int32_t tok = argmax_key_col(S.h_out[1 + i]);
    r.state = ORCA_INCREMENT;
    r.n_sched = 0;
    r.n_cached += S.L[i];
    if (r.n_cached < known_len(r)) {  // a chunk: known tokens remain unprocessed, nothing generated
      if (next_tokens) next_tokens[i] = -1;
      continue;
    }
    if (next_tokens) next_tokens[i] = tok;
    r.n_generated += 1;
    if (!(S.flags & ORCA_ITER_TEACHER_FORCE)) r.tokens[r.n_prompt + r.n_generated - 1] = tok;
    if (r.n_generated >= r.out_len || r.n_prompt + r.n_generated >= r.max_tokens) {
      r.state = ORCA_FINISHED;
      if (e->paged)
        e->blocks.release(r.req_id);
      else
        e->slots.release(r.req_id);
    }
  }
  return ORCA_OK;
}

int orca_iteration(orca_engine *e, orca_request *pool, const int32_t *batch_idx, int32_t n_batch, int32_t flags,
                   int32_t *next_tokens, float *logits_dev, void *stream) {
  if (!e) return ORCA_EINVAL;
  if (!next_tokens) return fail(e, ORCA_EINVAL, "NULL argument");
  if (e->q_len > 0) return fail(e, ORCA_ESTATE, "iterations in flight: use orca_iteration_wait");
  const int rc = orca_iteration_submit(e, pool, batch_idx, n_batch, flags, logits_dev, stream);
  if (rc) return rc;
  return orca_iteration_wait(e, nullptr, nullptr, next_tokens);
}

int orca_last_descriptor(const orca_engine *e, int32_t *n_batch, int32_t *n_rows, int32_t *row_off, int32_t *row_pos,
                         int32_t *row_slot, int32_t *last_row, int32_t capacity) {
  if (!e) return ORCA_EINVAL;
  if (n_batch) *n_batch = e->last_B;
  if (n_rows) *n_rows = e->last_N;
  if (capacity < e->last_N + 1 && (row_off || row_pos || row_slot || last_row)) return ORCA_EINVAL;
  if (row_off) std::copy(e->last_row_off.begin(), e->last_row_off.end(), row_off);
  if (row_pos) std::copy(e->last_row_pos.begin(), e->last_row_pos.end(), row_pos);
  if (row_slot) std::copy(e->last_row_slot.begin(), e->last_row_slot.end(), row_slot);
  if (last_row) std::copy(e->last_last_row.begin(), e->last_last_row.end(), last_row);
  return ORCA_OK;
}

int orca_last_launches(const orca_engine *e, int32_t *n_kernels) {
  if (!e || !n_kernels) return ORCA_EINVAL;
  *n_kernels = e->last_launches;
  return ORCA_OK;
}

int orca_last_transfer(const orca_engine *e, int64_t *h2d_bytes, int64_t *d2h_bytes, int32_t *n_work) {
  if (!e) return ORCA_EINVAL;
  if (h2d_bytes) *h2d_bytes = e->last_h2d;
  if (d2h_bytes) *d2h_bytes = e->last_d2h;
  if (n_work) *n_work = e->last_work;
  return ORCA_OK;
}

// Workspace of orca_attention: request records | CUDA-core work items |
// tensor-core work items | split partials | counters (split arrivals, then
// two work tickets).
struct AttnWsLayout {
  size_t req, work, work_tc, part, cnt, total;
};

AttnWsLayout attn_ws_layout(int32_t n_batch, int32_t n_rows, int32_t n_heads, int32_t head_dim) {
  AttnWsLayout L{};
  size_t o = 0;
  auto take = [&](size_t b) { size_t at = o; o = align_up(o + b, 256); return at; };
  L.req = take(sizeof(ReqInfo) * n_batch);
  L.work = take(sizeof(AttnWork) * (size_t)max_attn_work(n_batch, n_rows));
  L.work_tc = take(sizeof(AttnWork) * (size_t)max_tc_work(n_batch, n_rows));
  L.part = take((size_t)n_batch * kMaxSplits * n_heads * (head_dim + 2) * 4);
  L.cnt = take(((size_t)n_batch * n_heads + 4) * 4);
  L.total = o;
  return L;
}

int orca_attention_workspace_bytes(int32_t n_batch, int32_t n_rows, int32_t n_heads, int32_t head_dim,
                                   size_t *bytes) {
  if (!bytes || n_batch <= 0 || n_rows < n_batch || n_heads <= 0 || head_dim <= 0) return ORCA_EINVAL;
  *bytes = attn_ws_layout(n_batch, n_rows, n_heads, head_dim).total;
  return ORCA_OK;
}

int orca_attention(int32_t dtype, int32_t n_heads, int32_t head_dim, int64_t n_slots, const void *q,
                   const void *k_layer, const void *v_layer, void *out, int32_t n_batch, const int32_t *row_off,
                   const int32_t *ctx, const int64_t *slot_base, void *workspace, size_t ws_bytes,
                   int32_t *status_dev, void *stream) {
  if ((dtype != ORCA_DTYPE_F32 && dtype != ORCA_DTYPE_BF16) || n_heads <= 0 || n_batch <= 0 || !row_off || !ctx ||
      !slot_base || !q || !k_layer || !v_layer || !out || !workspace || !status_dev || n_slots <= 0 ||
      n_slots >= INT32_MAX)
    return ORCA_EINVAL;
  if (head_dim != 16 && head_dim != 32 && head_dim != 64 && head_dim != 128) return ORCA_EINVAL;
  const int32_t N = row_off[n_batch];
  if (row_off[0] != 0 || N <= 0) return ORCA_EINVAL;
  size_t need = 0;
  if (orca_attention_workspace_bytes(n_batch, N, n_heads, head_dim, &need) || ws_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return ORCA_EINVAL;
  const AttnWsLayout Lw = attn_ws_layout(n_batch, N, n_heads, head_dim);
  std::vector<ReqInfo> req(n_batch);
  std::vector<AttnWork> work(max_attn_work(n_batch, N)), work_tc(max_tc_work(n_batch, N));
  int max_keys = 0;
  double sum_keys = 0.0;
  for (int32_t i = 0; i < n_batch; ++i) {
    const int32_t L = row_off[i + 1] - row_off[i];
    if (L <= 0 || ctx[i] < 0 || slot_base[i] < 0 || slot_base[i] + ctx[i] + L > n_slots) return ORCA_EINVAL;
    req[i] = {row_off[i], L, ctx[i], (int32_t)slot_base[i], -1, 0};
    if (L == 1) {
      max_keys = std::max(max_keys, ctx[i] + 1);
      sum_keys += ctx[i] + 1;
    }
  }
  const int split = attn_split(max_keys, sum_keys, n_heads);
  const bool tc = attention_tc_supported(dtype, head_dim);
  int32_t n_work = 0, n_work_tc = 0;
  for (int32_t i = 0; i < n_batch; ++i) {
    if (tc && req[i].n_new >= kTcMinRows)
      n_work_tc = append_tc_work(work_tc.data(), n_work_tc, i, req[i].row_off, req[i].n_new);
    else
      n_work = append_attn_work(work.data(), n_work, i, req[i].row_off, req[i].n_new, req[i].ctx, split);
  }
  order_attn_work(work.data(), n_work, req.data(), split);
  if (order_tc_work(work_tc.data(), n_work_tc, req.data())) return ORCA_EBATCH;
  char *ws = static_cast<char *>(workspace);
  ReqInfo *d_req = reinterpret_cast<ReqInfo *>(ws + Lw.req);
  AttnWork *d_work = reinterpret_cast<AttnWork *>(ws + Lw.work);
  AttnWork *d_work_tc = reinterpret_cast<AttnWork *>(ws + Lw.work_tc);
  float *d_part = reinterpret_cast<float *>(ws + Lw.part);
  int32_t *d_cnt = reinterpret_cast<int32_t *>(ws + Lw.cnt);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(d_cnt, 0, ((size_t)n_batch * n_heads + 4) * 4, st) != cudaSuccess ||
      cudaMemcpyAsync(d_req, req.data(), sizeof(ReqInfo) * n_batch, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return ORCA_ECUDA;
  if (n_work > 0 &&
      cudaMemcpyAsync(d_work, work.data(), sizeof(AttnWork) * n_work, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return ORCA_ECUDA;
  if (n_work_tc > 0 &&
      cudaMemcpyAsync(d_work_tc, work_tc.data(), sizeof(AttnWork) * n_work_tc, cudaMemcpyHostToDevice, st) !=
          cudaSuccess)
    return ORCA_ECUDA;
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  if (n_work_tc > 0) {
    CUtensorMap tq, tk, tv;
    if (make_tmap(nullptr, &tq, q, N, (uint64_t)n_heads * head_dim, kTcBM) ||
        make_tmap(nullptr, &tk, k_layer, (uint64_t)n_heads * n_slots, head_dim, kTcBM) ||
        make_tmap(nullptr, &tv, v_layer, (uint64_t)n_heads * n_slots, head_dim, kTcBM))
      return ORCA_EINVAL;
    TcAttnArgs ta{};
    ta.out = out;
    ta.reqs = d_req;
    ta.work = d_work_tc;
    ta.ticket = d_cnt + (size_t)n_batch * n_heads + 2;
    ta.status = status_dev;
    ta.hidden = n_heads * head_dim;
    ta.n_heads = n_heads;
    ta.n_work = n_work_tc;
    ta.n_work_dev = nullptr;
    ta.n_slots = n_slots;
    ta.scale_log2 = scale_log2;
    if (launch_attention_tc(head_dim, &tq, &tk, &tv, &tk, &tv, ta, n_work_tc, st) != cudaSuccess) return ORCA_ECUDA;
  }
  AttnArgs aa{};
  aa.q = q;
  aa.k_layer = k_layer;
  aa.v_layer = v_layer;
  aa.out = out;
  aa.reqs = d_req;
  aa.rows = nullptr;
  aa.work = d_work;
  aa.part = d_part;
  aa.counters = d_cnt;
  aa.ticket = d_cnt + (size_t)n_batch * n_heads;
  aa.status = status_dev;
  aa.hidden = n_heads * head_dim;
  aa.n_heads = n_heads;
  aa.n_rows = N;
  aa.split = split;
  aa.n_work = n_work;
  aa.n_slots = n_slots;
  aa.scale_log2 = scale_log2;
  return launch_attention(dtype, head_dim, aa, n_work, st) == cudaSuccess ? ORCA_OK : ORCA_ECUDA;
}

int orca_argmax_rows(const float *logits_dev, int32_t n_rows, int32_t vocab, int32_t *out_dev, void *stream) {
  if (n_rows < 0 || vocab <= 0 || (n_rows > 0 && (!logits_dev || !out_dev))) return ORCA_EINVAL;
  return launch_argmax(logits_dev, n_rows, vocab, out_dev, nullptr, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ORCA_OK
             : ORCA_ECUDA;
}

int orca_selftest_wait_timeout(int32_t *status_dev, void *stream) {
  if (!status_dev) return ORCA_EINVAL;
  return launch_wait_selftest(status_dev, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ORCA_OK : ORCA_ECUDA;
}

int orca_linear(int32_t dtype, int32_t mode, const void *A, const void *W, const float *bias, void *out, int32_t M,
                int32_t N, int32_t K, void *scratch, size_t scratch_bytes, void *argmax_keys_dev, int32_t *status_dev,
                void *stream) {
  if (M < 0 || N <= 0 || K <= 0 || (M > 0 && (!A || !W || !status_dev))) return ORCA_EINVAL;
  if (dtype != ORCA_DTYPE_F32 && dtype != ORCA_DTYPE_BF16) return ORCA_EINVAL;
  if (M == 0) return ORCA_OK;
  EpiParams ep{};
  switch (mode) {
    case ORCA_LINEAR_STORE: ep.mode = kEpiStore; break;
    case ORCA_LINEAR_GELU: ep.mode = kEpiGelu; break;
    case ORCA_LINEAR_RESID: ep.mode = kEpiResid; break;
    case ORCA_LINEAR_F32OUT: ep.mode = kEpiLogits; break;
    default: return ORCA_EINVAL;
  }
  if (!out && !(mode == ORCA_LINEAR_F32OUT && argmax_keys_dev)) return ORCA_EINVAL;
  if (argmax_keys_dev && (mode != ORCA_LINEAR_F32OUT || dtype != ORCA_DTYPE_BF16)) return ORCA_EINVAL;
  ep.ldo = N;
  ep.bias = bias;
  ep.out = out;
  ep.status = status_dev;
  ep.argmax_keys = static_cast<unsigned long long *>(argmax_keys_dev);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == ORCA_DTYPE_F32) {
    if (mode == ORCA_LINEAR_STORE) ep.mode = kEpiLogits;  // fp32 store
    return launch_gemm_simt_f32(static_cast<const float *>(A), static_cast<const float *>(W), M, N, K, ep, st) ==
                   cudaSuccess
               ? ORCA_OK
               : ORCA_ECUDA;
  }
  if (K % kTcBK) return ORCA_EINVAL;
  GemmScratch scr{nullptr, 0, nullptr, 0};
  const size_t cnt_bytes = align_up(kGemmCounters * 4, 256);
  if (scratch && scratch_bytes > cnt_bytes && !(reinterpret_cast<uintptr_t>(scratch) & 255)) {
    scr.counters = static_cast<int32_t *>(scratch);
    scr.n_counters = 4 * std::min(kGemmMaxSms, gemm_sm_count());
    scr.partials = reinterpret_cast<float *>(static_cast<char *>(scratch) + cnt_bytes);
    scr.partial_bytes = scratch_bytes - cnt_bytes;
    if (cudaMemsetAsync(scratch, 0, kGemmCounters * 4, st) != cudaSuccess) return ORCA_ECUDA;
  }
  if (argmax_keys_dev && cudaMemsetAsync(argmax_keys_dev, 0, (size_t)M * 8, st) != cudaSuccess) return ORCA_ECUDA;
  OperandMaps ta, tw;
  if (make_operand_maps(nullptr, &ta, A, M, K) || make_operand_maps(nullptr, &tw, W, N, K)) return ORCA_EINVAL;
  return launch_gemm_tc_bf16(ta, tw, M, nullptr, N, K, ep, scr, status_dev, st) == cudaSuccess ? ORCA_OK : ORCA_ECUDA;
}

int orca_profile_enable(orca_engine *e, int32_t enable) {
  if (!e || enable < 0 || enable > 2) return ORCA_EINVAL;
  if (e->host_only && enable) return ORCA_ESTATE;
  if (e->q_len > 0) return fail(e, ORCA_ESTATE, "iterations in flight");
  if (enable == 2 && e->cfg.dtype != ORCA_DTYPE_BF16) return fail(e, ORCA_EINVAL, "launch stamps need a bf16 model");
  e->prof = enable == 1;
  e->stamps = enable == 2;
  for (auto &s : e->stats) s = orca_kernel_stats{};
  for (auto &p : e->pending) {  // launches still in flight are not counted
    e->ev_free.push_back(p.a);
    e->ev_free.push_back(p.b);
  }
  e->pending.clear();
  return ORCA_OK;
}

int orca_profile_read(const orca_engine *e, int32_t cls, orca_kernel_stats *out) {
  if (!e || !out || cls < 0 || cls >= ORCA_K_COUNT) return ORCA_EINVAL;
  *out = e->stats[cls];
  return ORCA_OK;
}

int orca_last_error(const orca_engine *e, char *buf, size_t n) {
  if (!e || !buf || n == 0) return ORCA_EINVAL;
  snprintf(buf, n, "%s", e->err.c_str());
  return ORCA_OK;
}

}  // extern "C"
