// Prefill attention on the tensor cores (tcgen05 + TMEM), bf16 heads of 64 or 128.
//
// The per-request attention of Figure 5 (Orca walk-through) for the rows of
// a prompt is a dense, causal contraction: S = Q K^T over the request's own
// keys, softmax, O = P V.  One work item is up to 128 query rows of one
// request and one head; persistent CTAs take items from an atomic ticket.
//
// Per item (two passes over the key tiles of 128 keys up to the last row's
// position, so the output accumulator never needs rescaling):
//   pass 1  S = Q K^T on tcgen05 into TMEM; each thread (one query row =
//           one TMEM lane) reads its row of S and keeps the running max of
//           the keys it may see (key position <= its own position);
//   pass 2  S again; p = exp2((s - max) * log2(e)/sqrt(d)) in fp32, the row
//           sum in registers, P rounded to bf16 into shared memory (K-major,
//           128-byte swizzle); O += P V on tcgen05 with V transposed by the
//           threads into a K-major tile (keys past the causal range are
//           zero, so stale slot contents never reach O);
//   end     O / sum -> bf16 rows of the output.
// Q and K tiles arrive by TMA (tensor maps over the q buffer and the
// layer's K slots).  Rows beyond the item's rows and keys beyond a row's
// position are masked by selection.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "orca_internal.h"

namespace orca {
namespace {

constexpr int kRows = 128;  // query rows per item = TMEM lanes
constexpr int kKeys = 128;  // keys per tile
constexpr int kThreadsTc = 128;

template <int D>
struct TcCfg {
  static constexpr int KB = D / 64;              // 64-element K-blocks of the head dim
  static constexpr int Q_BYTES = KB * kRows * 128;
  static constexpr int K_BYTES = KB * kKeys * 128;
  static constexpr int VT_BYTES = 2 * D * 128;   // D rows x 128 keys (two 64-key K-blocks)
  static constexpr int P_BYTES = 2 * kRows * 128;
  static constexpr int SMEM = Q_BYTES + K_BYTES + VT_BYTES + P_BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = 256;     // S: [0, 128), O: [128, 128 + D)
  static constexpr uint32_t IDESC_S =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kKeys >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
  static constexpr uint32_t IDESC_O =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
};

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of element (row, k) in a K-major, 128-byte-swizzled operand
// tile of `rows` rows (64-element K-blocks stacked, 8-row atoms of 1024 B).
__device__ __forceinline__ uint32_t sw128_offset(int row, int k, int rows) {
  const int kb = k >> 6, kk = k & 63;
  return (uint32_t)(kb * rows * 128 + row * 128 + ((((kk >> 3) ^ (row & 7)) << 4) | ((kk & 7) << 1)));
}

struct TcShared {
  uint64_t kbar, sbar, obar;
  uint32_t tmem;
  int item;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kThreadsTc, 1)
    prefill_attention_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                                TcAttnArgs a) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ TcShared sh;
  pdl_trigger();
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *sQ = smem_raw + pad;
  uint8_t *sK = sQ + C::Q_BYTES;
  uint8_t *sVt = sK + C::K_BYTES;
  uint8_t *sP = sVt + C::VT_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = warp * 32 + lane;  // query row of this thread = TMEM lane
  if (threadIdx.x == 0) {
    mbar_init(&sh.kbar, 1);
    mbar_init(&sh.sbar, 1);
    mbar_init(&sh.obar, 1);
    sh.abort = 0;
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  const int n_work = a.n_work_dev ? *a.n_work_dev : a.n_work;  // header written before the forward
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;
  const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tmem + t_lane, tO = tmem + t_lane + 128;
  volatile int *abort_flag = &sh.abort;
  uint32_t kph = 0, sph = 0, oph = 0;  // phases of the three barriers
  const __nv_bfloat16 *Vl = static_cast<const __nv_bfloat16 *>(a.v_layer);
  pdl_wait();  // q and the K/V slots come from the QKV Linear

  while (true) {
    __syncthreads();
    if (threadIdx.x == 0) sh.item = atomicAdd(a.ticket, 1);
    __syncthreads();
    const int item = sh.item;
    if (item >= n_work * a.n_heads) break;
    const int w_idx = item / a.n_heads, head = item - w_idx * a.n_heads;
    const AttnWork w = a.work[w_idx];
    const ReqInfo rq = a.reqs[w.req];
    const int r0 = w.a, nq = w.b;
    const int p0 = rq.ctx + (r0 - rq.row_off);
    const int kv_len = p0 + nq;                 // keys 0 .. p0 + nq - 1
    const bool bad = rq.slot_base < 0 || (int64_t)rq.slot_base + kv_len > a.n_slots || nq > kRows || nq <= 0;
    if (bad) {
      if (threadIdx.x == 0) atomicOr(a.status, kStatusBadIndex);
      continue;
    }
    const int my_pos = row < nq ? p0 + row : -1;  // -1: no key is visible to this row
    const int n_tiles = (kv_len + kKeys - 1) / kKeys;
    const int64_t krow0 = (int64_t)head * a.n_slots + rq.slot_base;  // K / V row of key 0
    // ---- Q tile (TMA) with the first K tile
    auto load_k = [&](int t, bool with_q) {
      if (threadIdx.x != 0 || *abort_flag) return;
      mbar_expect_tx(&sh.kbar, C::K_BYTES + (with_q ? C::Q_BYTES : 0));
      for (int kb = 0; kb < C::KB; ++kb) {
        if (with_q) tma_load_2d(sQ + kb * kRows * 128, &tmQ, head * D + kb * 64, r0, &sh.kbar);
        tma_load_2d(sK + kb * kKeys * 128, &tmK, kb * 64, (int)(krow0 + (int64_t)t * kKeys), &sh.kbar);
      }
    };
    auto mma_s = [&]() {  // S = Q K^T
      if (threadIdx.x != 0) return;
      tc_fence_after();
      for (int kb = 0; kb < C::KB; ++kb)
        for (int k = 0; k < 4; ++k)
          tc_mma(tmem, sw128_desc(smem_u32(sQ + kb * kRows * 128) + k * 32),
                 sw128_desc(smem_u32(sK + kb * kKeys * 128) + k * 32), C::IDESC_S, (kb | k) ? 1u : 0u);
      tc_commit(&sh.sbar);
    };
    // ---- pass 1: row max of the visible scores (raw dot products)
    float mx = -INFINITY;
    for (int t = 0; t < n_tiles; ++t) {
      load_k(t, t == 0);
      mbar_wait(&sh.kbar, kph, abort_flag, a.status);
      kph ^= 1u;
      mma_s();
      mbar_wait(&sh.sbar, sph, abort_flag, a.status);
      sph ^= 1u;
      tc_fence_after();
      for (int c = 0; c < kKeys; c += 32) {
        float v[32];
        tmem_ld32(tS + (uint32_t)c, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = t * kKeys + c + i;
          if (key <= my_pos) mx = fmaxf(mx, v[i]);
        }
      }
      tc_fence_before();
      __syncthreads();  // S and the K tile are free again
    }
    // ---- pass 2: P = exp2((S - max) * scale), O += P V
    float sum = 0.f;
    for (int t = 0; t < n_tiles; ++t) {
      load_k(t, false);
      // V tile transposed into sVt (K-major: row = head dim, 128 keys per row);
      // keys beyond kv_len are written as zero
      for (int e = threadIdx.x; e < (kKeys / 2) * (D / 8); e += kThreadsTc) {
        const int kp = e % (kKeys / 2), dc = e / (kKeys / 2);
        const int key = t * kKeys + 2 * kp;
        uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
        if (key < kv_len) v0 = __ldg(reinterpret_cast<const uint4 *>(Vl + (krow0 + key) * D + dc * 8));
        if (key + 1 < kv_len) v1 = __ldg(reinterpret_cast<const uint4 *>(Vl + (krow0 + key + 1) * D + dc * 8));
        const uint16_t *h0 = reinterpret_cast<const uint16_t *>(&v0);
        const uint16_t *h1 = reinterpret_cast<const uint16_t *>(&v1);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t pk = (uint32_t)h0[j] | ((uint32_t)h1[j] << 16);
          *reinterpret_cast<uint32_t *>(sVt + sw128_offset(dc * 8 + j, 2 * kp, D)) = pk;
        }
      }
      mbar_wait(&sh.kbar, kph, abort_flag, a.status);
      kph ^= 1u;
      mma_s();
      mbar_wait(&sh.sbar, sph, abort_flag, a.status);
      sph ^= 1u;
      tc_fence_after();
      for (int c = 0; c < kKeys; c += 32) {
        float v[32];
        tmem_ld32(tS + (uint32_t)c, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int key = t * kKeys + c + i;
          const float pa = key <= my_pos ? exp2f((v[i] - mx) * a.scale_log2) : 0.f;
          const float pb = key + 1 <= my_pos ? exp2f((v[i + 1] - mx) * a.scale_log2) : 0.f;
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(pa, pb);
          sum += __low2float(b2) + __high2float(b2);  // the sum of the P that reaches the MMA
          pk[i / 2] = *reinterpret_cast<const uint32_t *>(&b2);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *reinterpret_cast<uint4 *>(sP + sw128_offset(row, c + q4 * 8, kRows)) =
              make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
      }
      tc_fence_before();
      fence_proxy_async();  // P and V^T (generic stores) become visible to the tensor core
      __syncthreads();
      if (threadIdx.x == 0) {
        tc_fence_after();
        for (int kb = 0; kb < 2; ++kb)
          for (int k = 0; k < 4; ++k)
            tc_mma(tmem + 128, sw128_desc(smem_u32(sP + kb * kRows * 128) + k * 32),
                   sw128_desc(smem_u32(sVt + kb * D * 128) + k * 32), C::IDESC_O, (t | kb | k) ? 1u : 0u);
        tc_commit(&sh.obar);
      }
      mbar_wait(&sh.obar, oph, abort_flag, a.status);  // P, V^T, S free for the next tile
      oph ^= 1u;
    }
    // ---- O / sum -> output rows
    tc_fence_after();
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.out) + (int64_t)(r0 + row) * a.hidden + head * D;
    for (int c = 0; c < D; c += 32) {
      float v[32];
      tmem_ld32(tO + (uint32_t)c, v);
      if (row < nq && !*abort_flag) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t pk[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[q4 * 8 + 2 * j] * inv, v[q4 * 8 + 2 * j + 1] * inv);
            pk[j] = *reinterpret_cast<const uint32_t *>(&b2);
          }
          *reinterpret_cast<uint4 *>(orow + c + q4 * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    tc_fence_before();
  }
  // teardown: the last CTA out resets the ticket; free tensor memory
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.ticket + 1, 1) == (int)gridDim.x - 1) {
      a.ticket[0] = 0;
      a.ticket[1] = 0;
    }
  }
  if (*abort_flag && threadIdx.x == 0) drain_after_abort();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
  }
}

template <int D>
cudaError_t set_limit(int dev) {
  static uint64_t mask = 0;
  if (dev >= 64 || !(mask & (1ull << dev))) {
    cudaError_t e = cudaFuncSetAttribute(prefill_attention_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) mask |= 1ull << dev;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t attention_tc_prepare() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = set_limit<64>(dev);
  if (e == cudaSuccess) e = set_limit<128>(dev);
  return e;
}

bool attention_tc_supported(int dtype, int head_dim) { return dtype == 1 && (head_dim == 64 || head_dim == 128); }

cudaError_t launch_attention_tc(int head_dim, const CUtensorMap *tmQ, const CUtensorMap *tmK, const TcAttnArgs &a,
                                int n_work, cudaStream_t st) {
  if (n_work <= 0 && a.n_work_dev == nullptr) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int sm = gemm_sm_count();
  const long long total = (long long)n_work * a.n_heads;
  const int grid = a.n_work_dev != nullptr ? sm : (int)(total < sm ? total : sm);
  if (head_dim == 64) {
    e = set_limit<64>(dev);
    if (e != cudaSuccess) return e;
    return launch_pdl(prefill_attention_tc_kernel<64>, grid, kThreadsTc, TcCfg<64>::SMEM, st, *tmQ, *tmK, a);
  }
  if (head_dim == 128) {
    e = set_limit<128>(dev);
    if (e != cudaSuccess) return e;
    return launch_pdl(prefill_attention_tc_kernel<128>, grid, kThreadsTc, TcCfg<128>::SMEM, st, *tmQ, *tmK, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace orca
