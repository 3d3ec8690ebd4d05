// bf16 token-wise Linear on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Selective batching runs every non-attention Linear once over the whole
// flattened [sum L_i, H] tensor, so each weight tile is read once per
// iteration for all requests (Orca walk-through, "为什么注意力"不批量"的损失很小":
// batching pays off through parameter reuse).  This kernel computes
//   C[m, n] = sum_k A[m, k] * W[n, k]     A: [M, K] bf16, W: [N, K] bf16
// with fp32 accumulation in tensor memory, then the fused epilogue.
//
// Persistent CTAs (one per SM) walk a list of work units; a unit is one
// 128 x BN output tile, or one K-range of it when the output has too few
// tiles to fill the GPU (split-K, used for decode-sized M).  Tiles are
// visited in groups of 8 M-tiles so the CTAs running at the same time share
// their W tiles and A rows in L2.  Six warps:
//   warp 0      one lane issues TMA loads of 128x64 A and BNx64 W tiles
//               (128-byte swizzle) into a shared-memory ring;
//   warp 1      allocates 2*BN TMEM columns (two accumulators); one lane
//               issues tcgen05.mma (kind::f16, M=128, N=BN, K=16), releases
//               each ring stage with tcgen05.commit and hands a finished
//               accumulator to the epilogue;
//   warps 2..5  tcgen05.ld the accumulator (one TMEM lane quarter each),
//               free it for the next tile at once, and run the epilogue:
//               bias, then QKV scatter to K/V slots, GeLU, residual add,
//               logits store and/or a fused greedy argmax.  A split unit
//               stores an fp32 partial; the last unit of a tile to arrive
//               (atomic counter, no waiting) sums the partials and runs the
//               epilogue.
// Every mbarrier wait is bounded (about 2 s of %globaltimer).  On expiry the
// CTA sets kStatusWaitTimeout and an abort flag that ends every other wait at
// once; the roles then skip their work but keep their barrier sequence, and
// the tensor memory is still freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "epilogue.cuh"
#include "orca_internal.h"

namespace orca {
namespace {

constexpr int BM = kTcBM, BK = kTcBK;
constexpr int kStageBudget = 200 * 1024;
constexpr int kGroupM = 8;

template <int BN>
struct Cfg {
  // W tiles arrive as boxes of min(BN, 128) rows: one box for BN <= 128
  // (tensor map with that box height), two 128-row boxes for BN = 256.
  static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 256, "BN must be 32, 64, 128 or 256");
  static constexpr int BOX = BN < kTcBM ? BN : kTcBM;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (kStageBudget / STAGE) > 12 ? 12 : (kStageBudget / STAGE);
  static constexpr int SMEM = STAGES * STAGE + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  // Instruction descriptor, kind::f16: D fp32 (bit 4), A bf16 (bits 7-9),
  // B bf16 (bits 10-12), both K-major, N>>3 at bits 17-22, M>>4 at bits 24-28.
  static constexpr uint32_t IDESC =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
};

// Work decomposition, computed identically on the host (grid size) and by
// every thread of the kernel.
struct Sched {
  int nM, nN, KB, S, kbs, tiles, units;
  __host__ __device__ void init(int M, int N, int K, int BN, int sm, const GemmScratch &scr) {
    nM = (M + BM - 1) / BM;
    nN = (N + BN - 1) / BN;
    KB = K / BK;
    tiles = nM * nN;
    S = 1;
    kbs = KB;
    // The last unit of a tile reads all S partials through one SM, so split
    // only long K (>= 16 k-blocks) and at most 4 ways.
    if (scr.partials != nullptr && tiles > 0 && tiles * 2 <= sm && KB >= 16 && tiles <= scr.n_counters) {
      int s = sm / tiles;
      if (s > KB / 8) s = KB / 8;
      if (s > 4) s = 4;
      if (s > 1) {
        const int k = (KB + s - 1) / s;
        const int S2 = (KB + k - 1) / k;
        if ((size_t)tiles * S2 * BM * BN * sizeof(float) <= scr.partial_bytes) {
          S = S2;
          kbs = k;
        }
      }
    }
    units = tiles * S;
  }
  __device__ __forceinline__ void unit(int u, int &m, int &n, int &kb0, int &kb1, int &tile, int &split) const {
    split = u % S;
    tile = u / S;
    const int group = tile / (kGroupM * nN);
    const int first_m = group * kGroupM;
    const int gm = min(kGroupM, nM - first_m);
    const int r = tile - group * kGroupM * nN;
    m = first_m + r % gm;
    n = r / gm;
    kb0 = split * kbs;
    kb1 = min(KB, kb0 + kbs);
  }
};

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), descriptor version 1 (bit 46), layout 2 = SW128.
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

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane; the
// wait is in the same asm statement so no register is read before it lands.
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

__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Bias + epilogue store (+ fused argmax candidate) of one 32-column run of
// this thread's row.  Every lane of the warp calls it (the bias of the 32
// columns is one coalesced load, broadcast by shuffles); `active` masks rows
// beyond M.
__device__ __forceinline__ void finish_run(const EpiParams &epi, int row, int col, float *v, int cnt, bool active,
                                           unsigned long long &best) {
  if (epi.bias != nullptr) {
    const int lane = threadIdx.x & 31;
    const float bl = col + lane < col + cnt ? __ldg(epi.bias + col + lane) : 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] += __shfl_sync(0xffffffffu, bl, i);
  }
  if (!active) return;
  epi_store<__nv_bfloat16, 32>(epi, row, col, v, cnt);
  if (epi.argmax_keys != nullptr) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < cnt && v[i] == v[i]) {
        const unsigned long long k = argmax_key(v[i], col + i);
        best = k > best ? k : best;
      }
  }
}

template <int BN>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, int M_arg,
                        const int32_t *M_dev, int N, int K, int sm, EpiParams epi, GemmScratch scr,
                        int32_t *status) {
  using C = Cfg<BN>;
  constexpr int ST = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *sA = smem_raw + pad;
  uint8_t *sB = sA + ST * C::A_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + ST * C::B_BYTES);
  uint64_t *empty = full + ST;
  uint64_t *tfull = empty + ST;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *last_flag = abort_flag + 1;

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // M_dev is the descriptor header, written before the forward (not by an earlier kernel)
  const int M = M_dev != nullptr ? *M_dev : M_arg;
  Sched sc;
  sc.init(M, N, K, BN, sm, scr);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 4);
    mbar_init(&tempty[1], 4);
    *abort_flag = 0;
    *last_flag = 0;
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      // The weights do not depend on earlier kernels: the first stages' W
      // tiles are requested before waiting for them, so their latency
      // overlaps the previous kernel's tail.
      int pre = 0;
      if ((int)blockIdx.x < sc.units) {
        int m, n, kb0, kb1, tile, split;
        sc.unit(blockIdx.x, m, n, kb0, kb1, tile, split);
        pre = min(ST, kb1 - kb0);
        for (int j = 0; j < pre; ++j) {  // ring round 0: the stages are free
          mbar_expect_tx(&full[j], C::STAGE);
#pragma unroll
          for (int h = 0; h < BN / C::BOX; ++h)
            tma_load_2d(sB + j * C::B_BYTES + h * (C::BOX * BK * 2), &tmW, (kb0 + j) * BK, n * BN + h * C::BOX,
                        &full[j]);
        }
      }
      pdl_wait();  // A (activations) comes from earlier kernels
      int it = 0;
      for (int u = blockIdx.x; u < sc.units; u += gridDim.x) {
        int m, n, kb0, kb1, tile, split;
        sc.unit(u, m, n, kb0, kb1, tile, split);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % ST;
          if (it < pre) {  // W already requested
            tma_load_2d(sA + s * C::A_BYTES, &tmA, kb * BK, m * BM, &full[s]);
            continue;
          }
          const uint32_t ph = (uint32_t)(it / ST) & 1u;
          // once the CTA has aborted no further copy is issued
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, status) || *abort_flag) continue;
          mbar_expect_tx(&full[s], C::STAGE);
          tma_load_2d(sA + s * C::A_BYTES, &tmA, kb * BK, m * BM, &full[s]);
#pragma unroll
          for (int h = 0; h < BN / C::BOX; ++h)
            tma_load_2d(sB + s * C::B_BYTES + h * (C::BOX * BK * 2), &tmW, kb * BK, n * BN + h * C::BOX, &full[s]);
        }
      }
      if (*abort_flag) drain_after_abort();  // copies issued before the abort land first
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int it = 0, i = 0;
      for (int u = blockIdx.x; u < sc.units; u += gridDim.x, ++i) {
        int m, n, kb0, kb1, tile, split;
        sc.unit(u, m, n, kb0, kb1, tile, split);
        const int acc = i & 1;
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
        mbar_wait(&tempty[acc], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag, status);
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % ST;
          const uint32_t ph = (uint32_t)(it / ST) & 1u;
          if (mbar_wait(&full[s], ph, abort_flag, status)) {
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * C::A_BYTES);
            const uint32_t b0 = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc_mma(d_tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), C::IDESC,
                     (kb > kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        tc_commit(&tfull[acc]);
      }
    }
  } else {  // epilogue warps 2..5: TMEM lane quarter = warp % 4
    pdl_wait();  // the epilogue reads / writes buffers of earlier kernels (x, K/V slots)
    const int q = warp & 3;
    int i = 0;
    for (int u = blockIdx.x; u < sc.units; u += gridDim.x, ++i) {
      int m, n, kb0, kb1, tile, split;
      sc.unit(u, m, n, kb0, kb1, tile, split);
      const int acc = i & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], (uint32_t)(i >> 1) & 1u, abort_flag, status));
      tc_fence_after();
      const int row = m * BM + q * 32 + lane;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      unsigned long long best = 0ull;
      if (sc.S == 1) {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          if (ok) tmem_ld32(tbase + (uint32_t)c, v);
          if (c + 32 == BN) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          const int col = n * BN + c;
          if (ok && col < N) finish_run(epi, row, col, v, min(32, N - col), row < M, best);
        }
      } else {
        float *part = scr.partials + ((size_t)(tile * sc.S + split) * BM + q * 32 + lane) * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          if (ok) tmem_ld32(tbase + (uint32_t)c, v);
          if (c + 32 == BN) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          if (ok && row < M) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4 *>(part + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
        }
        __threadfence();
        epi_barrier();
        if (threadIdx.x == 64) *last_flag = atomicAdd(scr.counters + tile, 1) == sc.S - 1;
        epi_barrier();
        if (*last_flag) {
          __threadfence();
          if (threadIdx.x == 64) scr.counters[tile] = 0;
          if (ok) {
            const float *p0 = scr.partials + ((size_t)tile * sc.S * BM + q * 32 + lane) * BN;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
              const int col = n * BN + c;
              if (col >= N) break;
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
#pragma unroll 1
              for (int s = 0; s < sc.S && row < M; ++s) {
                const float4 *ps = reinterpret_cast<const float4 *>(p0 + (size_t)s * BM * BN + c);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float4 t = __ldcg(ps + j);
                  v[4 * j] += t.x;
                  v[4 * j + 1] += t.y;
                  v[4 * j + 2] += t.z;
                  v[4 * j + 3] += t.w;
                }
              }
              finish_run(epi, row, col, v, min(32, N - col), row < M, best);
            }
          }
        }
      }
      if (epi.argmax_keys != nullptr && best != 0ull) atomicMax(epi.argmax_keys + row, best);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int BN>
cudaError_t set_smem_limit(int dev) {
  static uint64_t attr_mask = 0;  // one bit per device ordinal
  if (dev >= 64 || !(attr_mask & (1ull << dev))) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_bf16_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<BN>::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_mask |= 1ull << dev;
  }
  return cudaSuccess;
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap *tmA, const CUtensorMap *tmW, int M, const int32_t *M_dev, int N, int K,
                      const EpiParams &epi, const GemmScratch &scr, int32_t *status, cudaStream_t st, int sm,
                      int dev) {
  cudaError_t e = set_smem_limit<BN>(dev);
  if (e != cudaSuccess) return e;
  Sched sc;
  sc.init(M, N, K, BN, sm, scr);
  const int grid = M_dev != nullptr ? sm : (sc.units < sm ? sc.units : sm);
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(gemm_tc_bf16_kernel<BN>, grid, 192, Cfg<BN>::SMEM, st, *tmA, *tmW, M, M_dev, N, K, sm, epi, scr,
                    status);
}

}  // namespace

int gemm_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cache[dev] = n;
  return n;
}

// Output-tile width: 256 when those tiles fill the GPU, else the widest of
// 128 / 64 / 32 whose tiles occupy at least half the SMs (narrower tiles
// spread a small-M product's weight stream over more SMs).
int gemm_tile_n(int M, int N) {
  const long long nM = (M + BM - 1) / BM;
  const int sm = gemm_sm_count();
  if (nM * ((N + 255) / 256) >= sm) return 256;
  if (nM * ((N + 127) / 128) * 2 >= sm) return 128;
  if (nM * ((N + 63) / 64) * 2 >= sm) return 64;
  return 32;
}

cudaError_t gemm_prepare() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = set_smem_limit<32>(dev);
  if (e == cudaSuccess) e = set_smem_limit<64>(dev);
  if (e == cudaSuccess) e = set_smem_limit<128>(dev);
  if (e == cudaSuccess) e = set_smem_limit<256>(dev);
  gemm_sm_count();
  return e;
}

// M selects the tile width; with M_dev the kernel reads the row count from
// the device (the tile width chosen from M must then stay valid for it).
cudaError_t launch_gemm_tc_bf16(const CUtensorMap *tmA, const WeightMaps &W, int M, const int32_t *M_dev, int N,
                                int K, const EpiParams &epi, const GemmScratch &scr, int32_t *status,
                                cudaStream_t st) {
  if (M <= 0 && M_dev == nullptr) return cudaSuccess;
  if (K % BK != 0 || K <= 0) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int sm = gemm_sm_count();
  switch (gemm_tile_n(M, N)) {
    case 256: return launch_bn<256>(tmA, &W.box128, M, M_dev, N, K, epi, scr, status, st, sm, dev);
    case 128: return launch_bn<128>(tmA, &W.box128, M, M_dev, N, K, epi, scr, status, st, sm, dev);
    case 64: return launch_bn<64>(tmA, &W.box64, M, M_dev, N, K, epi, scr, status, st, sm, dev);
    default: return launch_bn<32>(tmA, &W.box32, M, M_dev, N, K, epi, scr, status, st, sm, dev);
  }
}

}  // namespace orca
