// bf16 token-wise Linear on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Selective batching runs every non-attention Linear once over the whole
// flattened [sum L_i, H] tensor, so each weight tile is read once per
// iteration for all requests (Orca walk-through, "为什么注意力"不批量"的损失很小":
// batching pays off through parameter reuse).  This kernel computes
//   C[m, n] = sum_k A[m, k] * W[n, k]     A: [M, K] bf16, W: [N, K] bf16
// with fp32 accumulation in tensor memory, then the fused epilogue.
//
// Structure (one 128 x 128 output tile per CTA, 6 warps):
//   warp 0      one lane issues TMA loads of 128x64 A and W tiles (128-byte
//               swizzle) into a 4-stage shared-memory ring;
//   warp 1      allocates 128 TMEM columns; one lane issues tcgen05.mma
//               (kind::f16, M=128, N=128, K=16) and commits each stage back to
//               the producer and the finished tile to the epilogue;
//   warps 2..5  tcgen05.ld the accumulator (one TMEM lane quarter each) and
//               run the epilogue.
// Every mbarrier wait is bounded (about 2 s of %globaltimer); on expiry the
// kernel sets kStatusWaitTimeout, skips the remaining work and still frees
// its tensor memory.  Ragged M and N are handled by TMA zero fill on load
// and masked epilogue stores.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "epilogue.cuh"
#include "orca_internal.h"

namespace orca {
namespace {

constexpr int BM = kTcBM, BN = kTcBN, BK = kTcBK, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int SMEM_BYTES = STAGES * (A_BYTES + B_BYTES) + 1024 + 256;
constexpr uint32_t TMEM_COLS = BN;

// Instruction descriptor, kind::f16: D fp32 (bit 4), A bf16 (bits 7-9),
// B bf16 (bits 10-12), both K-major, N>>3 at bits 17-22, M>>4 at bits 24-28.
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                           ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete; false after ~2 s.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(addr, parity)) return true;
    if (global_ns() - t0 > 2000000000ull) return false;
  }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

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

__device__ __forceinline__ void tc_mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accum)
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

__global__ void __launch_bounds__(192, 1)
    gemm_tc_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, int M,
                        int N, int K, EpiParams epi, int32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *sA = smem_raw + pad;
  uint8_t *sB = sA + STAGES * A_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + STAGES * B_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *done = empty + STAGES;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int KB = K / BK;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u)) {
          atomicOr(status, kStatusWaitTimeout);
          break;
        }
        mbar_expect_tx(&full[s], A_BYTES + B_BYTES);
        tma_load_2d(sA + s * A_BYTES, &tmA, kb * BK, m0, &full[s]);
        tma_load_2d(sB + s * B_BYTES, &tmW, kb * BK, n0, &full[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (uint32_t)(kb / STAGES) & 1u;
        if (!mbar_wait(&full[s], ph)) {
          atomicOr(status, kStatusWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * A_BYTES);
        const uint32_t b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc_mma(tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), (kb > 0 || k > 0) ? 1u : 0u);
        tc_commit(&empty[s]);
      }
      tc_commit(done);
    }
  } else {
    // warp-uniform decision: tcgen05.ld below is .sync.aligned
    const bool ok = __all_sync(0xffffffffu, mbar_wait(done, 0));
    if (!ok && lane == 0) atomicOr(status, kStatusWaitTimeout);
    tc_fence_after();
    const int quarter = warp & 3;
    const int row = m0 + quarter * 32 + lane;
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, v);
        const int col = n0 + c;
        if (row < M && col < N) epi_apply<__nv_bfloat16, 32>(epi, row, col, v, min(32, N - col));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_gemm_tc_bf16(const CUtensorMap *tmA, const CUtensorMap *tmW, int M, int N, int K,
                                const EpiParams &epi, int32_t *status, cudaStream_t st) {
  if (M <= 0) return cudaSuccess;
  if (K % BK != 0 || K <= 0) return cudaErrorInvalidValue;
  static uint64_t attr_set_mask = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_set_mask & (1ull << dev))) {
    e = cudaFuncSetAttribute(gemm_tc_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set_mask |= 1ull << dev;
  }
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  gemm_tc_bf16_kernel<<<grid, 192, SMEM_BYTES, st>>>(*tmA, *tmW, M, N, K, epi, status);
  return cudaGetLastError();
}

}  // namespace orca
