// Ragged attention: every request attends only to its own K/V slots.
//
// Selective batching splits the flattened rows by request before attention
// and merges them back afterwards (Orca walk-through, Figure 5: Split,
// per-request Attention against the Attention K/V manager, Merge).  Here the
// split and the merge are index math: one launch covers all requests, each
// CTA takes one work item of one head and writes its rows of the [sum L_i, H]
// output in place.  Orca stitches the thread blocks of different requests
// into one kernel (CS349D Lecture 2, section 4.2); this launch does the same
// for two kinds of work:
//
//   kind 0, query tile : up to 16 rows of one request (a prefill), causal,
//                        K/V tiles of 32 keys staged in shared memory, online
//                        softmax per row;
//   kind 1, key split  : one row (a decode) over a range of at most `split`
//                        keys, streamed from HBM with 16-byte loads, a group
//                        of lanes per key; when a row has several splits the
//                        partial (max, sum, acc) of each goes to scratch and
//                        the last CTA to finish (atomic counter, no waiting)
//                        merges them and resets the counter.
//
// Row r of request i sits at position c_i + (r - row_off_i) and reads keys
// 0 .. that position (its own K/V was written by the QKV epilogue).  Scores
// are scaled by log2(e)/sqrt(d) so the softmax uses exp2.
#include <cuda_bf16.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "orca_internal.h"

namespace orca {
namespace {

template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4 v, float *o) {
    o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y); o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static void load(const float *p, float *o) {
    unpack(__ldg(reinterpret_cast<const uint4 *>(p)), o);
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4 v, float *o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
  __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float *o) {
    unpack(__ldg(reinterpret_cast<const uint4 *>(p)), o);
  }
};

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kThreads = 128;
constexpr int kKeyTile = 32;

template <int D>
struct TileSmem {
  float q[kQTile][D];
  float k[kKeyTile][D + 1];
  float v[kKeyTile][D];
};
// Key-split streaming: K and V chunks of chunk_keys<D>() keys flow through a
// ring_stages<D>()-stage shared-memory ring, filled by 1-D bulk copies issued
// by thread 0 (one per K/V block of the chunk: the keys of a request and head
// are contiguous in the slot pool, or one run per block of a paged table).
// One block per chunk; four stages for 64-dim heads: on GPT-2-small decode,
// larger chunks or an 8-stage ring (fewer waits per key, more bytes in flight
// per CTA) measured slower, as the bigger ring halves the CTAs resident per SM
// and the batch's items then need two waves.
template <int D>
__host__ __device__ constexpr int chunk_keys() {
  return kKvBlock;
}
// 128-dim heads take three stages (50 KB of shared memory): four CTAs fit on
// an SM, against three of four stages, and the 13B decode-only attention
// measured 16% faster so (more items in flight per SM for the same bytes).
template <int D>
__host__ __device__ constexpr int ring_stages() {
  return D == 128 ? 3 : 4;
}
constexpr int kRingMax = 4;

template <typename T, int D>
struct SplitSmem {
  static constexpr int CHUNK = chunk_keys<D>() * D * (int)sizeof(T);  // bytes of one K (or V) chunk
  alignas(128) unsigned char k[ring_stages<D>()][CHUNK];
  alignas(128) unsigned char v[ring_stages<D>()][CHUNK];
  float m[kThreads / 32];
  float l[kThreads / 32];
  float acc[kThreads / 32][D];
  int last;
};

// Ring barriers and flags (static shared memory, set up once per CTA).
struct Ring {
  uint64_t full[kRingMax];   // one arrival (with the copy bytes) per fill
  uint64_t empty[kRingMax];  // one arrival per warp per chunk consumed
  int abort;
};

// First slot of keys k0 .. k0 + kKvBlock - 1 of a request (k0 a multiple of
// kKvBlock), in the per-head [n_slots] view: consecutive slots of a
// contiguous reservation, or one block of a paged table.  -1 for a block
// outside the request's table or the pool.
__device__ __forceinline__ int64_t key_run_slot(const int32_t *blocks, int64_t n_slots, int slot_base, int block_off,
                                                int n_blocks, int k0) {
  if (block_off < 0) return (int64_t)slot_base + k0;
  const int bi = k0 / kKvBlock;
  if (bi >= n_blocks) return -1;
  const int64_t blk = blocks[block_off + bi];
  if (blk < 0 || (blk + 1) * kKvBlock > n_slots) return -1;
  return blk * kKvBlock;
}

// The request may read keys 0 .. n_keys-1 (contiguous: inside its
// reservation and the pool; paged: inside its block table).
__device__ __forceinline__ bool keys_in_range(const AttnArgs &a, const ReqInfo &rq, int n_keys) {
  if (rq.block_off < 0) return rq.slot_base >= 0 && (int64_t)rq.slot_base + n_keys <= a.n_slots;
  return (int64_t)rq.n_blocks * kKvBlock >= n_keys;
}

static_assert(kKeyTile == kKvBlock, "key tiles are one K/V block");
static_assert(chunk_keys<64>() % kKvBlock == 0 && chunk_keys<128>() % kKvBlock == 0,
              "decode chunks are whole K/V blocks");

// kind 0: rows r0 .. r0+cnt-1 of one request, keys 0 .. last row's position.
template <typename T, int D>
__device__ __forceinline__ void query_tile(const AttnArgs &a, const AttnWork &w, int head, TileSmem<D> &sm) {
  const ReqInfo rq = a.reqs[w.req];
  const int r0 = w.a, cnt = w.b;
  const int pos0 = rq.ctx + (r0 - rq.row_off);
  const int kv_len = pos0 + cnt;
  bool bad = !keys_in_range(a, rq, kv_len) || cnt > kQTile || r0 + cnt > a.n_rows;
  for (int t0 = 0; t0 < kv_len && !bad && rq.block_off >= 0; t0 += kKeyTile)  // every block of a paged table
    bad = key_run_slot(a.blocks, a.n_slots, rq.slot_base, rq.block_off, rq.n_blocks, t0) < 0;
  if (bad) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBadIndex);
    return;
  }
  // contiguous: keys from the reservation's first slot; paged: one block per key tile
  const int32_t *table = rq.block_off >= 0 ? a.blocks + rq.block_off : nullptr;
  const int64_t first = table ? 0 : rq.slot_base;
  const T *Kl = static_cast<const T *>(a.k_layer) + ((int64_t)head * a.n_slots + first) * D;
  const T *Vl = static_cast<const T *>(a.v_layer) + ((int64_t)head * a.n_slots + first) * D;
  const T *Q = static_cast<const T *>(a.q);
  for (int e = threadIdx.x; e < kQTile * D; e += kThreads) {
    const int i = e / D, d = e - i * D;
    sm.q[i][d] = i < cnt ? to_f(Q[(int64_t)(r0 + i) * a.hidden + head * D + d]) * a.scale_log2 : 0.f;
  }
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int NDL = (D + 31) / 32;
  constexpr int RPW = kQTile / (kThreads / 32);  // rows per warp
  float m_run[RPW], l_run[RPW], acc[RPW][NDL];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int j = 0; j < NDL; ++j) acc[i][j] = 0.f;
  }
  constexpr int VN = Vec16<T>::N;
  for (int t0 = 0; t0 < kv_len; t0 += kKeyTile) {
    __syncthreads();
    // the tile's keys are one run of slots (checked above)
    const int64_t s0 = table ? (int64_t)table[t0 / kKvBlock] * kKvBlock : t0;
    const T *Kp = Kl + s0 * D;
    const T *Vp = Vl + s0 * D;
    for (int e = threadIdx.x; e < kKeyTile * (D / VN); e += kThreads) {
      const int kk = e / (D / VN), c = (e - kk * (D / VN)) * VN;
      float kv[VN], vv[VN];
      if (t0 + kk < kv_len) {
        Vec16<T>::load(Kp + (int64_t)kk * D + c, kv);
        Vec16<T>::load(Vp + (int64_t)kk * D + c, vv);
      } else {
#pragma unroll
        for (int j = 0; j < VN; ++j) kv[j] = vv[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < VN; ++j) {
        sm.k[kk][c + j] = kv[j];
        sm.v[kk][c + j] = vv[j];
      }
    }
    __syncthreads();
    const int key = t0 + lane;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int li = wid * RPW + i;
      if (li >= cnt) continue;  // warp-uniform
      const int pos = pos0 + li;
      if (t0 > pos) continue;   // warp-uniform: whole tile is in this row's future
      float s = -INFINITY;
      if (key <= pos) {
        float dot = 0.f;
#pragma unroll 16
        for (int d = 0; d < D; ++d) dot = fmaf(sm.q[li][d], sm.k[lane][d], dot);
        s = dot;
      }
      const float mn = fmaxf(m_run[i], warp_max(s));
      const float p = key <= pos ? exp2f(s - mn) : 0.f;
      const float corr = exp2f(m_run[i] - mn);
      l_run[i] = l_run[i] * corr + warp_sum(p);
      float sum[NDL];
#pragma unroll
      for (int j = 0; j < NDL; ++j) sum[j] = 0.f;
#pragma unroll 8
      for (int kk = 0; kk < kKeyTile; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
        for (int j = 0; j < NDL; ++j) {
          const int dim = lane + 32 * j;
          if (dim < D) sum[j] = fmaf(pk, sm.v[kk][dim], sum[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < NDL; ++j) acc[i][j] = acc[i][j] * corr + sum[j];
      m_run[i] = mn;
    }
  }
  T *O = static_cast<T *>(a.out);
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int li = wid * RPW + i;
    if (li >= cnt) continue;
    const float inv = 1.f / l_run[i];
#pragma unroll
    for (int j = 0; j < NDL; ++j) {
      const int dim = lane + 32 * j;
      if (dim < D) O[(int64_t)(r0 + li) * a.hidden + head * D + dim] = from_f<T>(acc[i][j] * inv);
    }
  }
}

// Merge (m2, l2, acc2) into (m, l, acc); states with m = -inf are empty.
template <int VN>
__device__ __forceinline__ void merge_state(float &m, float &l, float *acc, float m2, float l2, const float *acc2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  const float c1 = exp2f(m - mn), c2 = exp2f(m2 - mn);
  l = l * c1 + l2 * c2;
#pragma unroll
  for (int j = 0; j < VN; ++j) acc[j] = acc[j] * c1 + acc2[j] * c2;
  m = mn;
}

// kind 1: one row over keys [split_idx * split, min(+split, pos + 1)).
// `g` counts the ring chunks this CTA has consumed (identical in every thread).
// `waited`: whether this CTA has waited for the kernels it depends on (the
// QKV Linear); until then only keys below the row's own position - written
// by earlier iterations - are read.
template <typename T, int D>
__device__ __forceinline__ void key_split(const AttnArgs &a, const AttnWork &w, int w_idx, int head,
                                          SplitSmem<T, D> &sm, Ring &rg, uint32_t &g, bool &waited) {
  constexpr int VN = Vec16<T>::N;
  constexpr int LPK = D / VN;          // lanes per key (16 bytes each)
  constexpr int KPW = 32 / LPK;        // keys per warp step
  constexpr int NW = kThreads / 32;
  const ReqInfo rq = a.reqs[w.req];
  const int r = w.a;
  const int pos = rq.ctx + (r - rq.row_off);
  const int n_keys = pos + 1;
  const int n_splits = (n_keys + a.split - 1) / a.split;
  const int kb = w.b * a.split;
  const int ke = min(kb + a.split, n_keys);
  bool bad = !keys_in_range(a, rq, n_keys) || r >= a.n_rows || kb >= n_keys || w.b >= kMaxSplits || kb % kKvBlock;
  for (int k0 = kb; k0 < ke && !bad && rq.block_off >= 0; k0 += kKvBlock)  // every block of a paged table
    bad = key_run_slot(a.blocks, a.n_slots, rq.slot_base, rq.block_off, rq.n_blocks, k0) < 0;
  if (bad) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusBadIndex);
    return;
  }
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane % LPK, grp = lane / LPK;
  // contiguous slots: keys from the reservation's first slot; paged: one
  // block of kKvBlock slots per chunk (blocks checked above)
  const bool paged = rq.block_off >= 0;
  const int32_t *table = paged ? a.blocks + rq.block_off : nullptr;
  const T *Kbase = static_cast<const T *>(a.k_layer) + ((int64_t)head * a.n_slots + (paged ? 0 : rq.slot_base)) * D;
  const T *Vbase = static_cast<const T *>(a.v_layer) + ((int64_t)head * a.n_slots + (paged ? 0 : rq.slot_base)) * D;
  constexpr int CK = chunk_keys<D>();
  constexpr int kRing = ring_stages<D>();
  const int n_chunks = (ke - kb + CK - 1) / CK;
  auto issue = [&](int c) {  // thread 0: fill the ring stage of chunk c
    const uint32_t idx = g + (uint32_t)c;
    const int st = (int)(idx % kRing);
    if (!mbar_wait(&rg.empty[st], ((idx / kRing) & 1u) ^ 1u, &rg.abort, a.status) || rg.abort) return;
    const int k0 = kb + c * CK;
    const int nk = min(CK, ke - k0);
    mbar_expect_tx(&rg.full[st], 2u * (uint32_t)(nk * D * (int)sizeof(T)));
    if (!paged) {
      const uint32_t bytes = (uint32_t)(nk * D * (int)sizeof(T));
      bulk_load(sm.k[st], Kbase + (int64_t)k0 * D, bytes, &rg.full[st]);
      bulk_load(sm.v[st], Vbase + (int64_t)k0 * D, bytes, &rg.full[st]);
    } else {
      for (int b0 = 0; b0 < nk; b0 += kKvBlock) {  // one run per block of the table
        const int64_t off = (int64_t)table[(k0 + b0) / kKvBlock] * kKvBlock;
        const uint32_t bytes = (uint32_t)(min(kKvBlock, nk - b0) * D * (int)sizeof(T));
        bulk_load(sm.k[st] + b0 * D * (int)sizeof(T), Kbase + off * D, bytes, &rg.full[st]);
        bulk_load(sm.v[st] + b0 * D * (int)sizeof(T), Vbase + off * D, bytes, &rg.full[st]);
      }
    }
  };
  const int n_first = min(kRing - 1, n_chunks);
  // chunks wholly below the row's position hold keys of earlier iterations:
  // they are requested before waiting for the QKV Linear (which writes the
  // row's own key and q)
  const int n_old = waited ? n_first : min(n_first, max(0, (pos - kb) / CK));
  if (threadIdx.x == 0)
    for (int c = 0; c < n_old; ++c) issue(c);
  if (!waited) {
    pdl_wait();
    waited = true;
  }
  if (threadIdx.x == 0)
    for (int c = n_old; c < n_first; ++c) issue(c);

  float q[VN];
  Vec16<T>::load(static_cast<const T *>(a.q) + (int64_t)r * a.hidden + head * D + sub * VN, q);
#pragma unroll
  for (int j = 0; j < VN; ++j) q[j] *= a.scale_log2;

  float m = -INFINITY, l = 0.f, acc[VN];
#pragma unroll
  for (int j = 0; j < VN; ++j) acc[j] = 0.f;
  for (int c = 0; c < n_chunks; ++c) {
    if (threadIdx.x == 0 && c + kRing - 1 < n_chunks) issue(c + kRing - 1);
    const uint32_t idx = g + (uint32_t)c;
    const int st = (int)(idx % kRing);
    const bool ok = mbar_wait(&rg.full[st], (idx / kRing) & 1u, &rg.abort, a.status);
    const int nk = min(CK, ke - (kb + c * CK));
    const T *ks = reinterpret_cast<const T *>(sm.k[st]);
    const T *vs = reinterpret_cast<const T *>(sm.v[st]);
    // warp `wid` takes key groups wid, wid + NW, ... of the chunk (KPW keys
    // each); warp-uniform trip count so every lane joins the shuffles
#pragma unroll
    for (int j = wid * KPW; j < CK; j += NW * KPW) {
      const int kk = j + grp;
      const bool valid = ok && kk < nk;
      float kv[VN], vv[VN];
      if (valid) {
        Vec16<T>::unpack(*reinterpret_cast<const uint4 *>(ks + kk * D + sub * VN), kv);
        Vec16<T>::unpack(*reinterpret_cast<const uint4 *>(vs + kk * D + sub * VN), vv);
      } else {
#pragma unroll
        for (int t = 0; t < VN; ++t) kv[t] = vv[t] = 0.f;
      }
      float sc = 0.f;
#pragma unroll
      for (int t = 0; t < VN; ++t) sc = fmaf(q[t], kv[t], sc);
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
      if (valid) {
        if (sc > m) {  // rescale only when the running max grows
          const float corr = exp2f(m - sc);
          l *= corr;
#pragma unroll
          for (int t = 0; t < VN; ++t) acc[t] *= corr;
          m = sc;
        }
        const float p = exp2f(sc - m);
        l += p;
#pragma unroll
        for (int t = 0; t < VN; ++t) acc[t] = fmaf(p, vv[t], acc[t]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rg.empty[st]);  // this warp is done reading the stage
  }
  g += (uint32_t)n_chunks;
  // merge the KPW key groups of the warp
#pragma unroll
  for (int o = LPK; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    float acc2[VN];
#pragma unroll
    for (int j = 0; j < VN; ++j) acc2[j] = __shfl_xor_sync(0xffffffffu, acc[j], o);
    merge_state<VN>(m, l, acc, m2, l2, acc2);
  }
  if (grp == 0) {
#pragma unroll
    for (int j = 0; j < VN; ++j) sm.acc[wid][sub * VN + j] = acc[j];
    if (sub == 0) {
      sm.m[wid] = m;
      sm.l[wid] = l;
    }
  }
  __syncthreads();
  // merge the warps: thread `dim` owns one output dimension
  const int dim = threadIdx.x;
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < NW; ++i) M = fmaxf(M, sm.m[i]);
  float L = 0.f, A = 0.f;
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const float c = sm.m[i] == -INFINITY ? 0.f : exp2f(sm.m[i] - M);
    L += sm.l[i] * c;
    if (dim < D) A += sm.acc[i][dim] * c;
  }
  T *O = static_cast<T *>(a.out) + (int64_t)r * a.hidden + head * D;
  if (n_splits == 1) {
    if (dim < D) O[dim] = from_f<T>(A / L);
    return;
  }
  // partial slot of (request, split): independent of the work-list order
  float *part = a.part + ((int64_t)(w.req * kMaxSplits + w.b) * a.n_heads + head) * (D + 2);
  if (dim < D) part[dim] = A;
  if (dim == 0) {
    part[D] = M;
    part[D + 1] = L;
  }
  __syncthreads();  // the CTA's partial is written ...
  if (threadIdx.x == 0) {
    __threadfence();  // ... and visible GPU-wide before it is counted
    const int prev = atomicAdd(a.counters + (int64_t)w.req * a.n_heads + head, 1);
    sm.last = prev == n_splits - 1;
    if (sm.last) __threadfence();  // the other splits' partials, counted before, are read below
  }
  __syncthreads();
  if (!sm.last) return;
  const int64_t s0 = (int64_t)w.req * kMaxSplits;  // the row's split partials
  if (dim < D) {
    // online merge of the splits' (max, sum, value) in split order, this
    // CTA's own state taken from registers at its index: the result does not
    // depend on which CTA finished last (the loads are independent of one
    // another, so they overlap)
    float Mx = -INFINITY, Lx = 0.f, Ax = 0.f;
#pragma unroll 4
    for (int j = 0; j < n_splits; ++j) {
      float mj = M, lj = L, aj = A;
      if (j != w.b) {
        const float *pj = a.part + ((s0 + j) * a.n_heads + head) * (D + 2);
        mj = __ldcg(pj + D);
        lj = __ldcg(pj + D + 1);
        aj = __ldcg(pj + dim);
      }
      const float mn = fmaxf(Mx, mj);
      if (mn == -INFINITY) continue;
      const float c1 = exp2f(Mx - mn), c2 = exp2f(mj - mn);
      Lx = Lx * c1 + lj * c2;
      Ax = Ax * c1 + aj * c2;
      Mx = mn;
    }
    O[dim] = from_f<T>(Ax / Lx);
  }
  if (threadIdx.x == 0) a.counters[(int64_t)w.req * a.n_heads + head] = 0;
}

// Persistent: CTA i takes (work item, head) pair i of the list (the host
// orders it longest first); when the pairs outnumber the CTAs, each CTA then
// takes further pairs from an atomic ticket until none is left, and the
// last CTA to finish resets the ticket for the next launch.
template <typename T, int D>
constexpr int attn_smem_bytes() {
  return (int)(sizeof(TileSmem<D>) > sizeof(SplitSmem<T, D>) ? sizeof(TileSmem<D>) : sizeof(SplitSmem<T, D>));
}

// CTAs per SM that shared memory allows (at most 8, i.e. at least 64
// registers a thread): the register budget is sized to keep that many
// resident, so registers never lower the occupancy.
template <typename T, int D>
constexpr int attn_min_ctas() {
  const int by_smem = (227 * 1024) / (attn_smem_bytes<T, D>() + 1024);
  return by_smem < 1 ? 1 : (by_smem > 8 ? 8 : by_smem);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, (attn_min_ctas<T, D>())) attention_kernel(AttnArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ Ring rg;
  __shared__ int s_item;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingMax; ++i) {
      mbar_init(&rg.full[i], 1);
      mbar_init(&rg.empty[i], kThreads / 32);
    }
    rg.abort = 0;
    mbar_fence_init();
  }
  uint32_t g = 0;  // ring chunks consumed
  pdl_trigger();
  if (a.hdr != nullptr) {  // written before the forward, not by an earlier kernel
    a.n_rows = a.hdr->n_rows;
    a.n_work = a.hdr->n_work;
    a.split = a.hdr->split;
  }
  // q and this step's K/V rows come from the QKV Linear: every item waits for
  // it (griddepcontrol.wait) before reading them; the work list, request
  // records and older K/V slots are read before
  bool waited = false;
  const int total = a.n_work * a.n_heads;
  // CTA i takes item i first; only when there are more items than CTAs do
  // the rest go out by ticket (so a small batch costs no atomics at all)
  const bool ticketed = total > (int)gridDim.x;
  int item = blockIdx.x;
  __syncthreads();  // the ring barriers are initialised
  while (item < total) {
    const int w_idx = item / a.n_heads;
    const int head = item - w_idx * a.n_heads;
    const AttnWork w = a.work[w_idx];
    if (w.kind == 0) {
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      query_tile<T, D>(a, w, head, *reinterpret_cast<TileSmem<D> *>(smem_raw));
    } else {
      key_split<T, D>(a, w, w_idx, head, *reinterpret_cast<SplitSmem<T, D> *>(smem_raw), rg, g, waited);
    }
    if (!ticketed) break;
    __syncthreads();  // the item's shared-memory reads are done
    if (threadIdx.x == 0) s_item = (int)gridDim.x + atomicAdd(a.ticket, 1);
    __syncthreads();
    item = s_item;
  }
  if (rg.abort) drain_after_abort();
  if (ticketed && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.ticket + 1, 1) == (int)gridDim.x - 1) {  // every CTA has left the loop
      a.ticket[0] = 0;
      a.ticket[1] = 0;
    }
  }
  __syncthreads();
  stamp_end(a.stamp);
}

// CTAs that fit on the GPU at once (one wave) for this instantiation; the
// first call on a device also raises the kernel's shared-memory limit.
template <typename T, int D>
int resident_ctas() {
  static int cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cache[dev]) return cache[dev];
  cudaFuncSetAttribute(attention_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, attn_smem_bytes<T, D>());
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attention_kernel<T, D>, kThreads, attn_smem_bytes<T, D>());
  const int n = (per_sm > 0 ? per_sm : 1) * gemm_sm_count();
  if (dev < 64) cache[dev] = n;
  return n;
}

template <typename T, int D>
cudaError_t launch_d(const AttnArgs &a, int n_work, cudaStream_t st, bool early) {
  const long long total = (long long)n_work * a.n_heads;
  const int cap = resident_ctas<T, D>();
  const dim3 grid(a.hdr != nullptr ? cap : (int)(total < cap ? total : cap));
  return launch_pdl_if(early, attention_kernel<T, D>, grid, kThreads, attn_smem_bytes<T, D>(), st, a);
}

template <typename T>
cudaError_t launch_t(int head_dim, const AttnArgs &a, int n_work, cudaStream_t st, bool early) {
  switch (head_dim) {
    case 16: return launch_d<T, 16>(a, n_work, st, early);
    case 32: return launch_d<T, 32>(a, n_work, st, early);
    case 64: return launch_d<T, 64>(a, n_work, st, early);
    case 128: return launch_d<T, 128>(a, n_work, st, early);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attention(int dtype, int head_dim, const AttnArgs &a, int n_work, cudaStream_t st, bool early) {
  if (n_work <= 0) return cudaSuccess;
  return dtype == 1 ? launch_t<__nv_bfloat16>(head_dim, a, n_work, st, early)
                    : launch_t<float>(head_dim, a, n_work, st, early);
}

// One-time per-device set-up of the attention kernels (shared-memory limits,
// occupancy); call before any stream capture.
cudaError_t attention_prepare() {
  resident_ctas<float, 16>();
  resident_ctas<float, 32>();
  resident_ctas<float, 64>();
  resident_ctas<float, 128>();
  resident_ctas<__nv_bfloat16, 16>();
  resident_ctas<__nv_bfloat16, 32>();
  resident_ctas<__nv_bfloat16, 64>();
  resident_ctas<__nv_bfloat16, 128>();
  return cudaGetLastError();
}

}  // namespace orca
