// bf16 token-wise Linear on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Selective batching runs every non-attention Linear once over the whole
// flattened [sum L_i, H] tensor, so each weight tile is read once per
// iteration for all requests (Orca walk-through, "为什么注意力"不批量"的损失很小":
// batching pays off through parameter reuse).  This kernel computes
//   C[m, n] = sum_k A[m, k] * W[n, k]     A: [M, K] bf16, W: [N, K] bf16
// with fp32 accumulation in tensor memory, then the fused epilogue.
//
// Three kernels; gemm_plan picks one per Linear.  The persistent one: CTAs
// (one per SM) walk a list of work
// units; a unit is one 128 x BN output tile, or one K-range of it when the
// output has too few tiles to fill the GPU and each tile's weight block is
// large (split-K).  Tiles are visited in groups of 8 M-tiles so the CTAs
// running at the same time share their W tiles and A rows in L2.  Six warps:
//   warp 0      one lane issues TMA loads into a shared-memory ring, one A
//               box and one W box per stage, each of KS k-blocks of 64
//               columns (128-byte swizzle);
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
// The cluster split-K kernel (further down) serves one 128-row tile with a
// long K: the K-ranges of an output tile go to the CTAs of one cluster, which
// exchange their fp32 partials through distributed shared memory.  The
// CTA-pair kernel (further down) computes 256 x 256 tiles on the two SMs of a
// cluster (cta_group::2); for a large weight stream at a few hundred rows
// its tiles are shared out along K over every pair, the last pair of a tile
// summing the pieces in k order.
// Every mbarrier wait is bounded (about 2 s of %globaltimer).  On expiry the
// CTA sets kStatusWaitTimeout and an abort flag that ends every other wait at
// once; the roles then skip their work but keep their barrier sequence, and
// the tensor memory is still freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "epilogue.cuh"
#include "orca.h"
#include "orca_internal.h"

namespace orca {
namespace {

constexpr int BM = kTcBM, BK = kTcBK;
constexpr int kStageBudget = 200 * 1024;
constexpr int kGroupM = 8;

template <int BN, int KS = 1>
struct Cfg {
  // A stage holds KS k-blocks of 64 columns, each a K-major SW128 sub-tile:
  // A as one box {64, a_box rows, KS} (sub-tiles a_box * 128 bytes apart),
  // W as boxes of min(BN, 128) rows - one box {64, BN, KS} for BN <= 128,
  // two 128-row boxes for BN = 256 (KS = 1).  The ring takes as many stages
  // of this size as fit in the budget (up to 12): with 64-row A boxes twice
  // as many A sub-tiles fit.
  static_assert(BN == 32 || BN == 64 || BN == 128 || BN == 256, "BN must be 32, 64, 128 or 256");
  static_assert(KS == 1 || KS == 2 || KS == 4, "KS must be 1, 2 or 4");
  static_assert(BN <= 128 || KS == 1, "256-wide tiles take one k-block per stage");
  static constexpr int BOX = BN < kTcBM ? BN : kTcBM;
  static constexpr int B_BYTES = KS * BN * BK * 2;
  static constexpr int MAX_STAGES = 12;
  static constexpr int SMEM = kStageBudget + 1024 + 256;  // the most a launch asks for
  // stage bytes of the A part for boxes of a_box rows
  __host__ __device__ static constexpr int a_stage(int a_box) { return KS * a_box * BK * 2; }
  __host__ __device__ static constexpr int stages(int a_box) {
    return kStageBudget / (a_stage(a_box) + B_BYTES) > MAX_STAGES ? MAX_STAGES
                                                                   : kStageBudget / (a_stage(a_box) + B_BYTES);
  }
  // dynamic shared memory of a launch: the ring, then its barriers
  __host__ __device__ static constexpr int smem(int a_box) {
    return stages(a_box) * (a_stage(a_box) + B_BYTES) + 1024 + 256;
  }
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
  // KB counts stages' worth of k-blocks (K / (64 * KS)).
  __host__ __device__ void init(int M, int N, int K, int BN, int KSb, int sm, const GemmScratch &scr) {
    nM = (M + BM - 1) / BM;
    nN = (N + BN - 1) / BN;
    KB = K / (BK * KSb);
    tiles = nM * nN;
    S = 1;
    kbs = KB;
    // The last unit of a tile reads all S partials through one SM, so split
    // only long K (>= 16 k-blocks of 64), at most 4 ways, and only tiles
    // whose weight block is at least 1 MB (a weight stream that one SM would
    // take microseconds to bring in; smaller ones - the MLP of GPT-2-small
    // at a few hundred rows - measured slower split than whole).
    if (scr.partials != nullptr && tiles > 0 && tiles * 2 <= sm && KB * KSb >= 16 && tiles <= scr.n_counters &&
        (long long)BN * K * 2 >= (1ll << 20)) {
      int s = sm / tiles;
      if (s > KB * KSb / 8) s = KB * KSb / 8;
      if (s > KB) s = KB;
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
// Bias of column col + lane (0 past the run or without bias).
__device__ __forceinline__ float run_bias(const EpiParams &epi, int col, int cnt) {
  const int lane = threadIdx.x & 31;
  return epi.bias != nullptr && lane < cnt ? __ldg(epi.bias + col + lane) : 0.f;
}

// LayerNorm folded into this Linear: v = rstd * (v - mean * c), with the
// row's mean and rstd from its fixed-point sums (biased variance, eps 1e-5,
// as the LayerNorm kernel).  Every lane calls it (c is shuffled).
__device__ __forceinline__ void fold_ln(const EpiParams &epi, int row, int col, float *v, int cnt, bool active) {
  const int lane = threadIdx.x & 31;
  const float cl = lane < cnt ? __ldg(epi.ln_c + col + lane) : 0.f;
  float mean = 0.f, rstd = 0.f;
  if (active) {
    const LnStats st = epi.ln_in[row];
    const float inv = 1.f / ((float)epi.ln_width * kLnStatScale);
    mean = (float)(long long)st.sum * inv;
    const float ex2 = (float)(long long)st.sumsq * inv;
    rstd = rsqrtf(fmaxf(ex2 - mean * mean, 0.f) + 1e-5f);
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = rstd * (v[i] - mean * __shfl_sync(0xffffffffu, cl, i));
}

// Residual rows that feed the next LayerNorm: x += v, then bf16(gamma * x)
// to ln_xb and the run's sums of x and x^2 into the row's statistics.  On
// return v holds the new x and g gamma * x.
__device__ __forceinline__ void resid_ln_run(const EpiParams &epi, int row, int col, float *v, float *g, int cnt) {
  float *xp = static_cast<float *>(epi.out) + (int64_t)row * epi.ldo + col;
  if ((reinterpret_cast<uintptr_t>(xp) & 15) == 0) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      if (i + 4 <= cnt) {
        float4 o = *reinterpret_cast<float4 *>(xp + i);
        o.x += v[i]; o.y += v[i + 1]; o.z += v[i + 2]; o.w += v[i + 3];
        *reinterpret_cast<float4 *>(xp + i) = o;
        v[i] = o.x; v[i + 1] = o.y; v[i + 2] = o.z; v[i + 3] = o.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (i + j < cnt) {
            v[i + j] += xp[i + j];
            xp[i + j] = v[i + j];
          }
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < cnt) {
        v[i] += xp[i];
        xp[i] = v[i];
      }
  }
  float s = 0.f, ss = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < cnt) {
      s += v[i];
      ss += v[i] * v[i];
      g[i] *= v[i];
    }
  store_run<__nv_bfloat16, 32>(static_cast<__nv_bfloat16 *>(epi.ln_xb) + (int64_t)row * epi.ldo + col, g, cnt);
  if (!(fabsf(s) < kLnStatMax && ss < kLnStatMax)) {  // also NaN
    atomicOr(epi.status, kStatusRange);
    return;
  }
  atomicAdd(&epi.ln_out[row].sum, (unsigned long long)__float2ll_rn(s * kLnStatScale));
  atomicAdd(&epi.ln_out[row].sumsq, (unsigned long long)__float2ll_rn(ss * kLnStatScale));
}

// bl: this lane's bias value of the run (run_bias), loaded ahead.
__device__ __forceinline__ void finish_run(const EpiParams &epi, int row, int col, float *v, int cnt, bool active,
                                           unsigned long long &best, float bl) {
  if (epi.ln_in != nullptr) fold_ln(epi, row, col, v, cnt, active);
  if (epi.bias != nullptr) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] += __shfl_sync(0xffffffffu, bl, i);
  }
  if (epi.ln_gamma != nullptr) {  // residual mode feeding the next LayerNorm
    const int lane = threadIdx.x & 31;
    const float gl = lane < cnt ? __ldg(epi.ln_gamma + col + lane) : 0.f;
    float g[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) g[i] = __shfl_sync(0xffffffffu, gl, i);
    if (active) resid_ln_run(epi, row, col, v, g, cnt);
    return;
  }
  if (!active) return;
  if (epi.ln_zero != nullptr && col == 0) epi.ln_zero[row] = LnStats{0ull, 0ull};
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

template <int BN, int KS>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, int M_arg,
                        const int32_t *M_dev, int N, int K, int sm, int a_box, EpiParams epi, GemmScratch scr,
                        int32_t *status) {
  using C = Cfg<BN, KS>;
  const int ST = C::stages(a_box);
  const int A_ST = C::a_stage(a_box);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *sA = smem_raw + pad;
  uint8_t *sB = sA + ST * A_ST;
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + ST * C::B_BYTES);
  uint64_t *empty = full + C::MAX_STAGES;
  uint64_t *tfull = empty + C::MAX_STAGES;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // M_dev is the descriptor header, written before the forward (not by an earlier kernel)
  const int M = M_dev != nullptr ? *M_dev : M_arg;
  Sched sc;
  sc.init(M, N, K, BN, KS, sm, scr);
  // bytes of one stage: the A box (a_box rows; 64 for products of <= 64 rows,
  // whose MMA rows 64..127 read the next 8 KB of shared memory - still inside
  // the stage area - and are never stored) + W
  const uint32_t stage_tx = (uint32_t)A_ST + C::B_BYTES;
  const uint32_t a_sub = (uint32_t)a_box * BK * 2;  // bytes between A sub-tiles of a stage

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
  // The next kernel may start only once this CTA holds its tensor memory: a
  // dependent CTA that allocated first and then waited for this kernel could
  // otherwise leave it without columns.
  pdl_trigger();

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
          mbar_expect_tx(&full[j], stage_tx);
#pragma unroll
          for (int h = 0; h < BN / C::BOX; ++h)
            tma_load_3d(sB + j * C::B_BYTES + h * (C::BOX * BK * 2), &tmW, 0, n * BN + h * C::BOX, (kb0 + j) * KS,
                        &full[j]);
        }
      }
      pdl_wait();  // A (activations) comes from earlier kernels
      // ring position (stage s, its phase parity ph) of copy number it
      int it = 0, s = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < sc.units; u += gridDim.x) {
        int m, n, kb0, kb1, tile, split;
        sc.unit(u, m, n, kb0, kb1, tile, split);
        for (int kb = kb0; kb < kb1; ++kb, ++it, s = s + 1 == ST ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
          if (it < pre) {  // W already requested
            tma_load_3d(sA + s * A_ST, &tmA, 0, m * BM, kb * KS, &full[s]);
            continue;
          }
          // once the CTA has aborted no further copy is issued
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, status) || *abort_flag) continue;
          mbar_expect_tx(&full[s], stage_tx);
          tma_load_3d(sA + s * A_ST, &tmA, 0, m * BM, kb * KS, &full[s]);
#pragma unroll
          for (int h = 0; h < BN / C::BOX; ++h)
            tma_load_3d(sB + s * C::B_BYTES + h * (C::BOX * BK * 2), &tmW, 0, n * BN + h * C::BOX, kb * KS,
                        &full[s]);
        }
      }
      if (*abort_flag) drain_after_abort();  // copies issued before the abort land first
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      int i = 0, s = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < sc.units; u += gridDim.x, ++i) {
        int m, n, kb0, kb1, tile, split;
        sc.unit(u, m, n, kb0, kb1, tile, split);
        const int acc = i & 1;
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
        mbar_wait(&tempty[acc], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag, status);
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb, s = s + 1 == ST ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
          if (mbar_wait(&full[s], ph, abort_flag, status)) {
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * A_ST);
            const uint32_t b0 = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
            for (int j = 0; j < KS; ++j)
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                tc_mma(d_tmem, sw128_desc(a0 + j * a_sub + k * 32), sw128_desc(b0 + j * (BN * BK * 2) + k * 32),
                       C::IDESC, (kb > kb0 || j > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(&empty[s]);
        }
        tc_commit(&tfull[acc]);
      }
    }
  } else {  // epilogue warps 2..5: TMEM lane quarter = warp % 4
    const int q = warp & 3;
    int i = 0;
    for (int u = blockIdx.x; u < sc.units; u += gridDim.x, ++i) {
      int m, n, kb0, kb1, tile, split;
      sc.unit(u, m, n, kb0, kb1, tile, split);
      const int acc = i & 1;
      // the bias of the first run (a weight, like W) is loaded while the tile
      // is computed; each run then loads the next run's
      float bl_next = n * BN < N ? run_bias(epi, n * BN, min(32, N - n * BN)) : 0.f;
      if (i == 0) pdl_wait();  // the epilogue reads / writes buffers of earlier kernels (x, K/V slots)
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
          const float bl = bl_next;
          if (c + 32 < BN && col + 32 < N) bl_next = run_bias(epi, col + 32, min(32, N - col - 32));
          if (ok && col < N) finish_run(epi, row, col, v, min(32, N - col), row < M, best, bl);
        }
      } else {
        // partial tiles are column-major [BN columns][BM rows]: the 32 lanes of a
        // warp (32 consecutive rows) store and load 128 contiguous bytes
        float *part = scr.partials + (size_t)(tile * sc.S + split) * BM * BN + q * 32 + lane;
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
            for (int j = 0; j < 32; ++j) __stcg(part + (size_t)(c + j) * BM, v[j]);
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
            const float *p0 = scr.partials + (size_t)tile * sc.S * BM * BN + q * 32 + lane;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
              const int col = n * BN + c;
              if (col >= N) break;
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
              // the splits in order, two at a time: all 64 loads in flight together
#pragma unroll 1
              for (int s = 0; s < sc.S && row < M; s += 2) {
                const float *ps = p0 + (size_t)s * BM * BN + (size_t)c * BM;
                float t0[32], t1[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) t0[j] = __ldcg(ps + (size_t)j * BM);
                const bool two = s + 1 < sc.S;
                if (two) {
#pragma unroll
                  for (int j = 0; j < 32; ++j) t1[j] = __ldcg(ps + (size_t)BM * BN + (size_t)j * BM);
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += t0[j];
                if (two) {
#pragma unroll
                  for (int j = 0; j < 32; ++j) v[j] += t1[j];
                }
              }
              finish_run(epi, row, col, v, min(32, N - col), row < M, best, run_bias(epi, col, min(32, N - col)));
            }
          }
        }
      }
      if (epi.argmax_keys != nullptr && best != 0ull) atomicMax(epi.argmax_keys + row, best);
    }
  }
  tc_fence_before();
  __syncthreads();
  stamp_end(epi.stamp);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Small-M products (one 128-row output tile in M): split-K over a thread-block
// cluster.  With few rows the cost of a Linear is moving its operands into
// the SMs and issuing its MMAs (one tcgen05.mma of N <= 64 columns takes
// about as long as one of 128), so the work is cut along K instead of into
// narrow tiles.  Each output tile of BN columns is one cluster of S CTAs; CTA
// r multiplies the r-th K-range (every k-block of it loaded at once onto one
// barrier, so there is no ring to recycle).  Column group g (BN / S columns)
// of the tile belongs to rank g: every rank writes its fp32 partial tile to
// its own shared memory grouped by owner, sends group g to rank g with one
// bulk copy over distributed shared memory (completing on rank g's receive
// barrier), and each rank then sums the S partials of its own group and runs
// the epilogue on them.  The CTAs of a cluster are resident together, so its
// two cluster barriers (all CTAs running; all copies landed before any CTA
// leaves) always complete; every other wait is bounded.  With at most 64 rows
// the A tile is loaded as a 64-row box (the MMA's rows 64..127 read the 8 KB
// after it and are never stored).
template <int BN>
struct CCfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr uint32_t TMEM_COLS = BN;
  // stage area for kbs k-blocks with A boxes of a_box rows (+ 8 KB read by the
  // MMA past 64-row boxes)
  __host__ __device__ static constexpr int stage_bytes(int kbs, int a_box) {
    return kbs * (a_box * BK * 2 + B_BYTES) + (a_box < BM ? 8192 : 0);
  }
  // this rank's partial tile, [owner g][row][BN / S] floats, written once the
  // MMAs are done (over the stage area); then the S received partials of the
  // owned group, [source rank][row][BN / S]
  static constexpr int TILE_BYTES = BM * BN * 4;
  __host__ __device__ static constexpr int work_bytes(int kbs, int a_box) {
    return stage_bytes(kbs, a_box) > TILE_BYTES ? stage_bytes(kbs, a_box) : TILE_BYTES;
  }
  __host__ __device__ static constexpr int smem(int kbs, int a_box) {
    return work_bytes(kbs, a_box) + TILE_BYTES + 1024 + 64;
  }
};
constexpr int kClusterSmemMax = 227 * 1024;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to
// another CTA's (dst and bar are shared::cluster addresses from mapa),
// completing on that CTA's barrier.
__device__ __forceinline__ void bulk_copy_to_rank(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "r"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_cta() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// k-blocks [kb0, kb0 + nk) of one operand (rows from y) into consecutive
// sub-tiles `sub` bytes apart, in boxes of 4, 2 and 1 k-blocks (t4 / t2 /
// t1), all completing on one barrier.  A box of ks k-blocks exists whenever
// ks <= K / 64, which nk never exceeds.
__device__ __forceinline__ void load_kblocks(uint8_t *dst, const CUtensorMap *t1, const CUtensorMap *t2,
                                             const CUtensorMap *t4, int y, int kb0, int nk, uint32_t sub,
                                             uint64_t *bar) {
  int j = 0;
  for (; j + 4 <= nk; j += 4) tma_load_3d(dst + j * sub, t4, 0, y, kb0 + j, bar);
  if (j + 2 <= nk) {
    tma_load_3d(dst + j * sub, t2, 0, y, kb0 + j, bar);
    j += 2;
  }
  if (j < nk) tma_load_3d(dst + j * sub, t1, 0, y, kb0 + j, bar);
}

// grid = nN * S CTAs in clusters of S (S in {2, 4, 8}); a_box = rows of one A
// box (64 or 128); rank r takes k-blocks [r * KB / S, (r + 1) * KB / S), at
// most kbs.  Shared memory: the work area (A sub-tiles a_box * 128 bytes
// apart, then W sub-tiles of BN * 128 bytes; later the partial tile), the
// receive area, then the barriers.  In both tile areas the 16-byte chunks of
// a row are XOR-swizzled by the row (spreading a warp's stores over the
// banks).  tmA1/2/4, tmW1/2/4: boxes of 1, 2 and 4 k-blocks.
template <int BN>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_cluster_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmA2,
                           const __grid_constant__ CUtensorMap tmA4, const __grid_constant__ CUtensorMap tmW1,
                           const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmW4,
                           int M_arg, const int32_t *M_dev, int N, int K, int S, int kbs, int a_box, EpiParams epi,
                           int32_t *status) {
  using C = CCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *body = smem_raw + pad;
  const uint32_t a_sub = (uint32_t)a_box * BK * 2;
  uint8_t *sW = body + kbs * a_sub + (a_box < BM ? 8192 : 0);
  float *part = reinterpret_cast<float *>(body);  // over the stage area once the MMAs are done
  float *recv = reinterpret_cast<float *>(body + C::work_bytes(kbs, a_box));
  uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(recv) + C::TILE_BYTES);
  uint64_t *done = full + 1;
  uint64_t *recv_bar = done + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(recv_bar + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = M_dev != nullptr ? *M_dev : M_arg;  // M_dev: the descriptor header, written before the forward
  const int rank = (int)cluster_rank();
  const int n = blockIdx.x / S;  // output tile = cluster
  const int KB = K / BK;
  const int kb0 = rank * KB / S, kb1 = (rank + 1) * KB / S, nkb = kb1 - kb0;
  const int cw = BN / S;            // columns of the group this rank owns
  const int swz = cw / 4 - 1;       // chunk swizzle mask (cw / 4 is a power of two)
  const bool shape_ok = nkb <= kbs && M <= BM && BN % (4 * S) == 0;

  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    mbar_init(done, 1);
    mbar_init(recv_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();  // only once this CTA holds its tensor memory (as in the persistent kernel)
  // first cluster phase: this CTA runs (its receive area may be written once
  // every CTA of the cluster has arrived here)
  cluster_arrive_relaxed();

  if (warp == 0) {
    if (lane == 0 && shape_ok && nkb > 0) {  // TMA producer: every k-block of this rank at once
      mbar_expect_tx(full, (uint32_t)nkb * (a_sub + C::B_BYTES));
      // weights do not depend on earlier kernels
      if (BN <= 128) {
        load_kblocks(sW, &tmW1, &tmW2, &tmW4, n * BN, kb0, nkb, C::B_BYTES, full);
      } else {
        for (int j = 0; j < nkb; ++j)
#pragma unroll
          for (int h = 0; h < BN / Cfg<BN>::BOX; ++h)
            tma_load_3d(sW + j * C::B_BYTES + h * (Cfg<BN>::BOX * BK * 2), &tmW1, 0, n * BN + h * Cfg<BN>::BOX,
                        kb0 + j, full);
      }
      pdl_wait();  // A (activations) comes from earlier kernels
      load_kblocks(body, &tmA1, &tmA2, &tmA4, 0, kb0, nkb, a_sub, full);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      if (shape_ok && nkb > 0) {
        if (mbar_wait(full, 0, abort_flag, status)) {
          tc_fence_after();
          const uint32_t a0 = smem_u32(body), b0 = smem_u32(sW);
          for (int j = 0; j < nkb; ++j)
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc_mma(tmem, sw128_desc(a0 + j * a_sub + k * 32), sw128_desc(b0 + j * C::B_BYTES + k * 32),
                     Cfg<BN>::IDESC, (j > 0 || k > 0) ? 1u : 0u);
        } else {
          drain_after_abort();  // copies issued before the abort land first
        }
      }
      tc_commit(done);  // also when there was nothing to multiply: the partial is then zero
    }
  }
  __syncwarp();
  const int q = warp & 3;  // TMEM lane quarter of an epilogue warp (rows q * 32 ...)
  const int row = q * 32 + lane;
  float bl_next = 0.f;
  if (warp >= 2) {
    // the bias of the owned group's first run (a weight, like W) is loaded
    // during the MMAs; each run then loads the next run's
    const int col = n * BN + rank * cw;
    bl_next = col < N ? run_bias(epi, col, min(min(32, cw), N - col)) : 0.f;
    pdl_wait();
  }
  const bool ok = warp >= 2 && __all_sync(0xffffffffu, warp >= 2 ? mbar_wait(done, 0, abort_flag, status) : true) &&
                  nkb > 0 && shape_ok;
  cluster_wait_acquire();  // every CTA of the cluster runs (its barriers are initialised)
  const int rows = M < BM ? (M > 0 ? M : 0) : BM;  // rows sent and summed
  if (warp >= 2) {
    tc_fence_after();
    // partial tile (zeros without MMAs) into the work area, grouped by owner;
    // the whole warp loads (tcgen05.ld is warp-collective), rows past M are
    // not stored
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float v[32];
      if (ok) {
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      if (row < rows) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const int col = c + i, g = col / cw, ch = (col - g * cw) >> 2;
          *reinterpret_cast<float4 *>(part + (size_t)(g * BM + row) * cw + ((ch ^ (row & swz)) << 2)) =
              make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
      }
    }
    tc_fence_before();
    fence_proxy_async_cta();  // the bulk copies read what these threads wrote
    epi_barrier();
    if (warp == 2) {  // lane g sends group g (the S copies are issued side by side)
      const uint32_t grp = (uint32_t)(rows * cw * 4);  // bytes of one group
      if (lane == 0) mbar_expect_tx(recv_bar, (uint32_t)S * grp);
      if (grp > 0 && lane < S) {
        const uint32_t slot = smem_u32(recv) + (uint32_t)(rank * BM * cw * 4);
        bulk_copy_to_rank(map_to_rank(slot, (uint32_t)lane), smem_u32(part + (size_t)lane * BM * cw), grp,
                          map_to_rank(smem_u32(recv_bar), (uint32_t)lane));
      }
    }
    // every lane: finish_run shuffles the bias across the warp; rows past M store nothing
    const bool got = __all_sync(0xffffffffu, mbar_wait(recv_bar, 0, abort_flag, status));
    const bool alive = got && __all_sync(0xffffffffu, *abort_flag == 0);
    unsigned long long best = 0ull;
    const float *mine = recv + (size_t)row * cw;
#pragma unroll 1
    for (int r0 = 0; r0 < cw; r0 += 32) {
      const int cnt = min(32, cw - r0);
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
      if (alive && row < rows) {
#pragma unroll 1
        for (int j = 0; j < S; ++j) {
          const float *src = mine + (size_t)j * BM * cw;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (4 * i < cnt) {
              const int ch = (r0 >> 2) + i;
              const float4 t = *reinterpret_cast<const float4 *>(src + ((ch ^ (row & swz)) << 2));
              v[4 * i] += t.x;
              v[4 * i + 1] += t.y;
              v[4 * i + 2] += t.z;
              v[4 * i + 3] += t.w;
            }
          }
        }
      }
      const int col = n * BN + rank * cw + r0;
      const float bl = bl_next;
      if (r0 + 32 < cw && col + 32 < N) bl_next = run_bias(epi, col + 32, min(min(32, cw - r0 - 32), N - col - 32));
      if (col < N && alive) finish_run(epi, row, col, v, min(cnt, N - col), row < M, best, bl);
    }
    if (epi.argmax_keys != nullptr && best != 0ull) atomicMax(epi.argmax_keys + row, best);
    if (!got) drain_after_abort();  // copies still on their way land before the CTA leaves
  }
  if (threadIdx.x == 0 && !shape_ok) atomicOr(status, kStatusBadShape);
  // second phase: every CTA has received its copies, so no copy still reads
  // the shared memory of a CTA that leaves
  __syncwarp();
  cluster_arrive_release();
  cluster_wait_acquire();
  tc_fence_before();
  __syncthreads();
  stamp_end(epi.stamp);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Large-M products: one 256 x 256 output tile per CTA pair (tcgen05 with
// cta_group::2).  The two CTAs of a cluster of 2 share one MMA of M = 256,
// N = 256: each holds 128 rows of the A tile and 128 rows (output columns) of
// the W tile in its own shared memory, at the same offsets, and 128 rows x
// 256 columns of the accumulator in its own tensor memory.  Per k-block an SM
// then takes in 32 KB (A and W halves) for the same 128 x 256 x 64 MMA work
// that costs a single CTA 48 KB; with the operand stream the bound of the
// single-CTA kernel at large M (about 70% tensor-pipe activity, the ring's
// bytes in flight over the L2 latency), this is what feeds the tensor core.
// Roles, in both CTAs unless stated:
//   warp 0      one lane loads its CTA's A and W halves of each stage; the
//               copies complete on the leader CTA's (rank 0) full barrier,
//               whose expected bytes the leader sets for both;
//   warp 1      allocates 512 TMEM columns (cta_group::2, both CTAs); in the
//               leader one lane issues the MMAs and commits each stage's
//               release and each finished accumulator to both CTAs' barriers
//               (multicast);
//   warps 2..5  read their CTA's accumulator rows and run the epilogue, then
//               tell the leader that the accumulator is free (its tempty
//               barrier counts the 8 epilogue warps of the pair).
// Two cluster barriers: barriers initialised before any copy or arrive
// crosses CTAs; every MMA and epilogue done before either CTA frees its
// tensor memory or leaves.  Every other wait is bounded.
constexpr int kPairBN = 256;                             // output columns of a pair tile
constexpr int kPairBM = 2 * BM;                          // output rows of a pair tile
constexpr int kPairHalf = BM * BK * 2;                   // one operand half of a stage: 16 KB
constexpr int kPairStage = 2 * kPairHalf;                // A half + W half
constexpr int kPairStages = 7;
constexpr int kPairSmem = kPairStages * kPairStage + 1024 + 512;
// 16 KB slots of the ring that the last pair of a shared tile loads the other
// pieces into (one 32-column run of one piece each), once its ring is idle
constexpr int kPairRedSlots = kPairStages * kPairStage / (BM * 32 * 4);
constexpr int kPairGroupM = 16;  // pair tiles per row group (4096 rows; measured best of 4, 8, 16)
// Pair tiles shared out along K (PairSched): weight streams of at least
// 128 MB only, ranges of at least 8 k-blocks, and reading back one other
// pair's piece (a 128 KB fp32 partial per CTA, through L2) counted as 16
// k-blocks of MMA time.
constexpr double kPairSplitMinBytes = 128.0 * (1 << 20);
constexpr int kPairMinRange = 8;
constexpr int kPairPieceKb = 16;
// kind::f16, D fp32, A/B bf16 K-major, N = 256, M = 256 (the pair's rows)
constexpr uint32_t kPairIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kPairBN >> 3) << 17) |
                                ((uint32_t)(kPairBM >> 4) << 24);

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// Arrive on `bar` (same offset) in both CTAs of the pair once the MMAs issued
// so far are complete.
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
// 3-D tiled load into this CTA's shared memory, completing on a barrier that
// may be in the peer CTA (bar: shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *tm, int x, int y, int z,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for a barrier that the peer CTA also arrives on (cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                  int32_t *status) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait_cluster(addr, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(addr, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > 2000000000ull) {
      *abort_flag = 1;
      atomicOr(status, kStatusWaitTimeout);
      return false;
    }
  }
}

// One stretch of work of a pair: k-blocks [kb0, kb1) of output tile `tile`
// (row tile m, column tile n).  pieces = how many pairs share the tile (1: the
// pair computes it whole), mine = which of them this pair is in k order.
struct PairSeg {
  int m, n, tile, kb0, kb1, pieces, mine, first;
};

// Pair tiles in groups of kPairGroupM row tiles, so the pairs running at the
// same time share their W tiles in L2.  P pairs run.  A large weight stream
// at a few hundred rows leaves most pairs idle in its last wave (the 13B FC1
// at 200 rows: 80 tiles on 76 pairs, two waves; the FC2: 20 tiles of 320
// k-blocks on 76 pairs), so its tiles are shared out along K in one of two
// ways:
//   kind 1 (split): S pairs per tile, pair p = tile * S + s taking the s-th
//     of S equal k-ranges (tiles * S <= P);
//   kind 2 (stream): the W = tiles * KB k-blocks in tile-major order cut into
//     P equal ranges, pair p taking [p W / P, (p + 1) W / P), so a tile is
//     shared by the pairs whose ranges meet it (a range's first and last
//     tiles may be shared, those in between are whole).
// The cost of either, in k-blocks of one pair's MMA time: its longest range
// plus kPairPieceKb for each other piece the last pair of a tile reads back;
// taken when it beats whole tiles by 15%.  A pair keeps a shared piece in
// slot `unit` (split) or 2p / 2p + 1 (stream: its first / last tile); the
// last pair to finish a tile sums its pieces in k order, so the result does
// not depend on which pair finishes last.  Computed identically on the host
// and by every thread of the kernel.
struct PairSched {
  int nM, nN, KB, tiles, P, kind, S, kbs, W;
  __host__ __device__ void init(int M, int N, int K, int pairs, bool can_split) {
    nM = (M + kPairBM - 1) / kPairBM;
    nN = (N + kPairBN - 1) / kPairBN;
    KB = K / BK;
    tiles = nM * nN;
    P = pairs;
    kind = 0;
    S = 1;
    kbs = KB;
    W = 0;
    if (!can_split || P <= 0 || tiles <= 0 || M <= BM || 2.0 * N * K < kPairSplitMinBytes) return;
    long long best = (long long)((tiles + P - 1) / P) * KB * 85 / 100;
    if (tiles * 2 <= P) {
      int s = min(P / tiles, KB / kPairMinRange);
      if (s >= 2) {
        const int k = (KB + s - 1) / s;
        s = (KB + k - 1) / k;  // no empty range
        const long long cost = k + (long long)(s - 1) * kPairPieceKb;
        if (cost < best) {
          best = cost;
          kind = 1;
          S = s;
          kbs = k;
        }
      }
    }
    // a stream range walks the row tiles of a column of W one after another,
    // so W comes from HBM once per row tile: only for one row tile, or when
    // whole tiles would leave at least 45% of the pairs idle
    const long long w = (long long)tiles * KB, least = w / P;
    const bool stream_ok = nM == 1 || (long long)tiles * 100 <= (long long)((tiles + P - 1) / P) * P * 55;
    if (stream_ok && least >= kPairMinRange) {
      const long long pieces = (KB + least - 1) / least + 1;  // the most a tile can have
      const long long cost = (w + P - 1) / P + (pieces - 1) * kPairPieceKb;
      if (cost < best) {
        kind = 2;
        S = 1;
        kbs = KB;
        W = (int)w;
      }
    }
  }
  __host__ __device__ bool split() const { return kind != 0; }
  // pairs that take work (the grid when split)
  __host__ __device__ int busy() const { return kind == 1 ? tiles * S : kind == 2 ? P : min(tiles, P); }
  __host__ __device__ __forceinline__ long long start(int p) const { return (long long)p * W / P; }
  // the pair whose stream range holds k-block x (no range is empty: every one
  // has at least kPairMinRange k-blocks)
  __host__ __device__ __forceinline__ int owner(long long x) const { return (int)(((x + 1) * P + W - 1) / W) - 1; }
  __host__ __device__ __forceinline__ void unit(int u, int &m, int &n) const {
    const int group = u / (kPairGroupM * nN);
    const int first_m = group * kPairGroupM;
    const int gm = kPairGroupM < nM - first_m ? kPairGroupM : nM - first_m;
    const int r = u - group * kPairGroupM * nN;
    m = first_m + r % gm;
    n = r / gm;
  }
  // segment j of pair p; false past its last
  __host__ __device__ __forceinline__ bool segment(int p, int j, PairSeg &g) const {
    g.pieces = 1;
    g.mine = 0;
    g.first = p;
    g.kb0 = 0;
    g.kb1 = KB;
    if (kind == 0) {
      g.tile = p + j * P;
      if (g.tile >= tiles) return false;
    } else if (kind == 1) {
      if (j > 0 || p >= tiles * S) return false;
      g.tile = p / S;
      g.mine = p - g.tile * S;
      g.pieces = S;
      g.first = g.tile * S;
      g.kb0 = g.mine * kbs;
      g.kb1 = g.kb0 + kbs < KB ? g.kb0 + kbs : KB;
    } else {
      const long long b = start(p), e = start(p + 1);
      const int t0 = (int)(b / KB);
      const int t = t0 + j;
      if ((long long)t * KB >= e) return false;
      g.tile = t;
      g.kb0 = j == 0 ? (int)(b - (long long)t0 * KB) : 0;
      g.kb1 = (int)(e - (long long)t * KB < KB ? e - (long long)t * KB : KB);
      g.first = owner((long long)t * KB);
      g.pieces = owner((long long)(t + 1) * KB - 1) - g.first + 1;
      g.mine = p - g.first;
    }
    unit(g.tile, g.m, g.n);
    return true;
  }
  // partial slot of piece i (k order) of a shared tile
  __host__ __device__ __forceinline__ int piece_slot(const PairSeg &g, int i) const {
    if (kind == 1) return g.first + i;
    const int q = g.first + i;
    return 2 * q + (start(q) / KB == g.tile ? 0 : 1);
  }
  // arrival counters of a shared tile: [0, 2P) arrivals, [2P, 4P) pieces stored
  __host__ __device__ __forceinline__ int counter(const PairSeg &g, uint32_t rank) const {
    return 2 * (kind == 1 ? g.tile : g.first) + (int)rank;
  }
};

// A split needs four counters per pair (arrivals and pieces stored, per
// rank) and four partial tiles of 128 x 256 floats per pair (two slots, two
// ranks).
__host__ __device__ __forceinline__ bool pair_split_ok(const GemmScratch &scr, int pairs) {
  return scr.partials != nullptr && scr.counters != nullptr && 4 * pairs <= scr.n_counters &&
         (size_t)4 * pairs * BM * kPairBN * sizeof(float) <= scr.partial_bytes;
}

// grid = 2 x pairs, clusters of 2; tmA / tmW: 3-D views with boxes of 128
// rows x 1 k-block.  kSplit: tiles may be shared out along K (PairSched);
// scr: their partials (slot s of CTA rank r at (2 s + r) * 128 * 256 floats,
// column-major) and arrival counters.  Without kSplit the kernel carries none
// of that code (the large products, whole tiles only).
template <bool kSplit>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, int M_arg,
                        const int32_t *M_dev, int N, int K, EpiParams epi, GemmScratch scr, int32_t *status) {
  constexpr int ST = kPairStages;
  extern __shared__ uint8_t smem_raw[];
  // the same offsets in both CTAs (same kernel, same static shared memory)
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *sA = smem_raw + pad;
  uint8_t *sB = sA + ST * kPairHalf;
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + ST * kPairHalf);
  uint64_t *empty = full + ST;
  uint64_t *tfull = empty + ST;
  uint64_t *tempty = tfull + 2;
  uint64_t *red = tempty + 2;  // kPairRedSlots
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(red + kPairRedSlots);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M = M_dev != nullptr ? *M_dev : M_arg;  // M_dev: the descriptor header, written before the forward
  const uint32_t rank = cluster_rank();             // 0: leader (issues the MMAs), 1: peer
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  PairSched sc;
  sc.init(M, N, K, npairs, kSplit && pair_split_ok(scr, npairs));

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 8);
    mbar_init(&tempty[1], 8);
    if (kSplit)
      for (int r = 0; r < kPairRedSlots; ++r) mbar_init(&red[r], 1);
    *abort_flag = 0;
    *last_flag = 0;
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 2 * kPairBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();  // only once this CTA holds its tensor memory (as in the persistent kernel)
  // both CTAs' barriers are initialised before any copy or arrive crosses over
  cluster_arrive_release();
  cluster_wait_acquire();

  PairSeg g;
  if (warp == 0) {
    if (lane == 0) {  // TMA producer (both CTAs): this CTA's halves, on the leader's full barriers
      const uint32_t full0 = map_to_rank(smem_u32(full), 0);
      const int row_half = (int)rank * BM, col_half = (int)rank * BM;
      int pre = 0;
      if (sc.segment(pair, 0, g)) {  // weights first: they do not depend on earlier kernels
        pre = min(ST, g.kb1 - g.kb0);
        for (int j = 0; j < pre; ++j) {
          if (rank == 0) mbar_expect_tx(&full[j], 2u * kPairStage);
          tma_load_3d_pair(sB + j * kPairHalf, &tmW, 0, g.n * kPairBN + col_half, g.kb0 + j, full0 + 8u * j);
        }
      }
      pdl_wait();  // A (activations) comes from earlier kernels
      int it = 0, s = 0;
      uint32_t ph = 0;
      for (int j = 0; sc.segment(pair, j, g); ++j) {
        for (int kb = g.kb0; kb < g.kb1; ++kb, ++it, s = s + 1 == ST ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
          const uint32_t bar = full0 + 8u * (uint32_t)s;
          if (it < pre) {  // W already requested
            tma_load_3d_pair(sA + s * kPairHalf, &tmA, 0, g.m * kPairBM + row_half, kb, bar);
            continue;
          }
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, status) || *abort_flag) continue;
          if (rank == 0) mbar_expect_tx(&full[s], 2u * kPairStage);
          tma_load_3d_pair(sA + s * kPairHalf, &tmA, 0, g.m * kPairBM + row_half, kb, bar);
          tma_load_3d_pair(sB + s * kPairHalf, &tmW, 0, g.n * kPairBN + col_half, kb, bar);
        }
      }
      if (*abort_flag) drain_after_abort();  // copies issued before the abort land first
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // MMA issuer (leader)
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; sc.segment(pair, i, g); ++i) {
        const int acc = i & 1;
        const uint32_t d_tmem = tmem + (uint32_t)(acc * kPairBN);
        mbar_wait_cluster(&tempty[acc], ((uint32_t)(i >> 1) & 1u) ^ 1u, abort_flag, status);
        tc_fence_after();
        for (int kb = g.kb0; kb < g.kb1; ++kb, s = s + 1 == ST ? 0 : s + 1, ph ^= s == 0 ? 1u : 0u) {
          if (mbar_wait(&full[s], ph, abort_flag, status)) {
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * kPairHalf);
            const uint32_t b0 = smem_u32(sB + s * kPairHalf);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc_mma_pair(d_tmem, sw128_desc(a0 + k * 32), sw128_desc(b0 + k * 32), kPairIdesc,
                          (kb > g.kb0 || k > 0) ? 1u : 0u);
          }
          tc_commit_pair(&empty[s]);
        }
        tc_commit_pair(&tfull[acc]);
      }
    }
  } else {  // epilogue warps 2..5 (both CTAs): TMEM lane quarter = warp % 4
    const int q = warp & 3;
    const uint32_t tempty0 = map_to_rank(smem_u32(tempty), 0);
    for (int i = 0; sc.segment(pair, i, g); ++i) {
      const int acc = i & 1;
      float bl_next = g.n * kPairBN < N ? run_bias(epi, g.n * kPairBN, min(32, N - g.n * kPairBN)) : 0.f;
      if (i == 0) pdl_wait();  // the epilogue reads / writes buffers of earlier kernels (x, K/V slots)
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], (uint32_t)(i >> 1) & 1u, abort_flag, status));
      tc_fence_after();
      const int row = g.m * kPairBM + (int)rank * BM + q * 32 + lane;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kPairBN);
      unsigned long long best = 0ull;
      if (g.pieces == 1) {
#pragma unroll 1
        for (int c = 0; c < kPairBN; c += 32) {
          float v[32];
          if (ok) tmem_ld32(tbase + (uint32_t)c, v);
          if (c + 32 == kPairBN) {  // the accumulator is read: free it for the leader's next tile
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
          }
          const int col = g.n * kPairBN + c;
          const float bl = bl_next;
          if (c + 32 < kPairBN && col + 32 < N) bl_next = run_bias(epi, col + 32, min(32, N - col - 32));
          if (ok && col < N) finish_run(epi, row, col, v, min(32, N - col), row < M, best, bl);
        }
      } else if constexpr (kSplit) {
        // a tile shared by g.pieces pairs.  Each counts itself in once its
        // accumulator is ready; all but the last to do so store their piece
        // (column-major: a warp's 32 rows are 128 contiguous bytes) and count
        // it stored; the last waits for those stores - their pairs are
        // already running, nothing they do waits - and sums the pieces in
        // k order, its own straight from tensor memory.
        int32_t *arrived = scr.counters + sc.counter(g, rank);
        int32_t *stored = arrived + 2 * sc.P;
        epi_barrier();
        if (threadIdx.x == 64) *last_flag = atomicAdd(arrived, 1) == g.pieces - 1;
        epi_barrier();
        const bool last = *last_flag != 0;
        if (!last) {
          float *part = scr.partials + (size_t)(2 * sc.piece_slot(g, g.mine) + (int)rank) * BM * kPairBN + q * 32 + lane;
#pragma unroll 1
          for (int c = 0; c < kPairBN; c += 32) {
            float v[32];
            if (ok) tmem_ld32(tbase + (uint32_t)c, v);
            if (ok && row < M) {
#pragma unroll
              for (int j = 0; j < 32; ++j) __stcg(part + (size_t)(c + j) * BM, v[j]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
          __threadfence();
          epi_barrier();
          if (threadIdx.x == 64) atomicAdd(stored, 1);
        } else {
          if (threadIdx.x == 64) {
            bool got = true;
            const uint64_t t0 = global_ns();
            while (*reinterpret_cast<volatile int32_t *>(stored) < g.pieces - 1) {
              if (*abort_flag || global_ns() - t0 > 2000000000ull) {
                *abort_flag = 1;
                atomicOr(status, kStatusWaitTimeout);
                got = false;
                break;
              }
            }
            *last_flag = got ? 1 : 2;
          }
          epi_barrier();
          const bool all_in = *last_flag == 1;  // the same in every epilogue warp
          const bool sum_ok = ok && all_in;
          __threadfence();  // the stored pieces, counted before, are read below
          if (threadIdx.x == 64) {
            *arrived = 0;
            *stored = 0;
            // the pieces were written by ordinary stores and are read below by
            // bulk copies (the async proxy)
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
          PairSeg nx;
          const int others = g.pieces - 1;
          if (all_in && others <= kPairRedSlots && !sc.segment(pair, i + 1, nx)) {
            // this pair's last segment: its MMAs are done, so the ring is idle.
            // The other pieces come in by bulk copies, R >= 1 runs of 32 columns
            // at a time (one 16 KB slot per run and piece), all in flight together
            const int R = min(kPairBN / 32, kPairRedSlots / others);
            for (int c0 = 0, round = 0; c0 < kPairBN / 32; c0 += R, ++round) {
              const int nc = min(R, kPairBN / 32 - c0);
              if (round > 0) {
                epi_barrier();  // the previous round's slots are read
                if (threadIdx.x == 64) fence_proxy_async_cta();
              }
              if (threadIdx.x == 64) {
                for (int cc = 0; cc < nc; ++cc)
                  for (int o = 0; o < others; ++o) {
                    const int pc = o < g.mine ? o : o + 1;
                    const int slot = cc * others + o;
                    mbar_expect_tx(&red[slot], BM * 32 * 4);
                    bulk_load(sA + (size_t)slot * (BM * 32 * 4),
                              scr.partials + (size_t)(2 * sc.piece_slot(g, pc) + (int)rank) * BM * kPairBN +
                                  (size_t)(c0 + cc) * 32 * BM,
                              BM * 32 * 4, &red[slot]);
                  }
              }
#pragma unroll 1
              for (int cc = 0; cc < nc; ++cc) {
                const int c = (c0 + cc) * 32;
                const int col = g.n * kPairBN + c;
                bool in = true;
                for (int o = 0; o < others; ++o) in = mbar_wait(&red[cc * others + o], (uint32_t)round & 1u, abort_flag, status) && in;
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
#pragma unroll 1
                for (int pc = 0; pc < g.pieces; ++pc) {
                  float t[32];
                  if (pc == g.mine) {
                    if (ok) tmem_ld32(tbase + (uint32_t)c, t);
                    else {
#pragma unroll
                      for (int j = 0; j < 32; ++j) t[j] = 0.f;
                    }
                  } else {
                    const float *src = reinterpret_cast<const float *>(
                                           sA + (size_t)(cc * others + (pc < g.mine ? pc : pc - 1)) * (BM * 32 * 4)) +
                                       q * 32 + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) t[j] = src[j * BM];
                  }
#pragma unroll
                  for (int j = 0; j < 32; ++j) v[j] += t[j];
                }
                if (sum_ok && in && col < N)
                  finish_run(epi, row, col, v, min(32, N - col), row < M, best, run_bias(epi, col, min(32, N - col)));
              }
            }
          } else {
#pragma unroll 1
          for (int c = 0; c < kPairBN; c += 32) {
            const int col = g.n * kPairBN + c;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
            // the pieces in k order, two at a time (up to 64 loads in flight)
#pragma unroll 1
            for (int pc = 0; pc < g.pieces; pc += 2) {
              const bool two = pc + 1 < g.pieces;
              float t0[32], t1[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) t0[j] = t1[j] = 0.f;
              if (pc == g.mine) {
                if (ok) tmem_ld32(tbase + (uint32_t)c, t0);
              } else if (sum_ok && row < M) {
                const float *src = scr.partials + (size_t)(2 * sc.piece_slot(g, pc) + (int)rank) * BM * kPairBN +
                                   (size_t)c * BM + q * 32 + lane;
#pragma unroll
                for (int j = 0; j < 32; ++j) t0[j] = __ldcg(src + (size_t)j * BM);
              }
              if (two) {
                if (pc + 1 == g.mine) {
                  if (ok) tmem_ld32(tbase + (uint32_t)c, t1);
                } else if (sum_ok && row < M) {
                  const float *src = scr.partials + (size_t)(2 * sc.piece_slot(g, pc + 1) + (int)rank) * BM * kPairBN +
                                     (size_t)c * BM + q * 32 + lane;
#pragma unroll
                  for (int j = 0; j < 32; ++j) t1[j] = __ldcg(src + (size_t)j * BM);
                }
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] += t0[j];
              if (two) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += t1[j];
              }
            }
            if (sum_ok && col < N)
              finish_run(epi, row, col, v, min(32, N - col), row < M, best, run_bias(epi, col, min(32, N - col)));
          }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
        }
      }
      if (epi.argmax_keys != nullptr && best != 0ull) atomicMax(epi.argmax_keys + row, best);
    }
  }
  // every MMA of the pair is complete (each epilogue saw its last commit) and
  // every epilogue is done before either CTA frees its tensor memory or leaves
  tc_fence_before();
  __syncthreads();
  cluster_arrive_release();
  cluster_wait_acquire();
  stamp_end(epi.stamp);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 2 * kPairBN);
  }
}

template <int BN, int KS>
cudaError_t set_smem_limit(int dev) {
  static uint64_t attr_mask = 0;  // one bit per device ordinal
  if (dev >= 64 || !(attr_mask & (1ull << dev))) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_bf16_kernel<BN, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<BN, KS>::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_mask |= 1ull << dev;
  }
  return cudaSuccess;
}

template <int BN>
cudaError_t set_cluster_smem_limit(int dev) {
  static uint64_t attr_mask = 0;
  if (dev >= 64 || !(attr_mask & (1ull << dev))) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_cluster_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kClusterSmemMax);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_mask |= 1ull << dev;
  }
  return cudaSuccess;
}

template <int BN>
cudaError_t launch_cluster(const OperandMaps &A, const OperandMaps &W, int M, const int32_t *M_dev, int N, int K,
                           int S, int kbs, int a_box, const EpiParams &epi, int32_t *status, cudaStream_t st, int dev) {
  cudaError_t e = set_cluster_smem_limit<BN>(dev);
  if (e != cudaSuccess) return e;
  const int smem = CCfg<BN>::smem(kbs, a_box);
  if (smem > kClusterSmemMax || BN % (4 * S) != 0) return cudaErrorInvalidValue;
  const int nN = (N + BN - 1) / BN;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(nN * S);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = smem;  // only what this launch uses
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const int wb = BN < 128 ? BN : 128;
  return cudaLaunchKernelEx(&cfg, gemm_tc_cluster_kernel<BN>, *A.get(a_box, 1), *A.get(a_box, 2), *A.get(a_box, 4),
                            *W.get(wb, 1), *W.get(wb, 2), *W.get(wb, 4), M, M_dev, N, K, S, kbs, a_box, epi, status);
}

template <int BN, int KS>
cudaError_t launch_bn(const CUtensorMap *tmA, const CUtensorMap *tmW, int M, const int32_t *M_dev, int N, int K,
                      int a_box, const EpiParams &epi, const GemmScratch &scr, int32_t *status, cudaStream_t st,
                      int sm, int dev) {
  cudaError_t e = set_smem_limit<BN, KS>(dev);
  if (e != cudaSuccess) return e;
  Sched sc;
  sc.init(M, N, K, BN, KS, sm, scr);
  const int grid = M_dev != nullptr ? sm : (sc.units < sm ? sc.units : sm);
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(gemm_tc_bf16_kernel<BN, KS>, grid, 192, Cfg<BN, KS>::smem(a_box), st, *tmA, *tmW, M, M_dev, N, K,
                    sm, a_box, epi, scr, status);
}

cudaError_t set_pair_smem_limit(int dev) {
  static uint64_t attr_mask = 0;
  if (dev >= 64 || !(attr_mask & (1ull << dev))) {
    cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tc_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_mask |= 1ull << dev;
  }
  return cudaSuccess;
}

// Persistent pairs: at most one pair per two SMs; every pair when the tiles
// are split (with M_dev the grid is fixed, the device decides the work: a
// grid of fewer pairs than tiles would decide the same on the device).
// split: the plan shares tiles out along K at this M (the kernel that can).
cudaError_t launch_pair(const CUtensorMap *tmA, const CUtensorMap *tmW, int M, const int32_t *M_dev, int N, int K,
                        const EpiParams &epi, const GemmScratch &scr, bool split, int32_t *status, cudaStream_t st,
                        int sm, int dev) {
  cudaError_t e = set_pair_smem_limit(dev);
  if (e != cudaSuccess) return e;
  PairSched sc;
  sc.init(M, N, K, sm / 2, split && pair_split_ok(scr, sm / 2));
  const int pairs = M_dev != nullptr || sc.split() ? sm / 2 : sc.busy();
  if (pairs <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = kPairSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, split ? gemm_tc_pair_kernel<true> : gemm_tc_pair_kernel<false>, *tmA, *tmW, M,
                            M_dev, N, K, epi, scr, status);
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

// Below this many rows a large weight stream may take 256-wide single-CTA
// tiles split along K (gemm_tile_n).
constexpr int kPairMinRows = 512;
// Weight streams at least this large, at a few hundred rows, take 256-wide
// tiles split along K.  Measured on GB300 at 200-256 rows: the 13B FC2 (210 MB)
// 17% faster than on 128-wide unsplit tiles, the Attn-Out (52 MB) 25% slower
// (its reduction of 3 partial tiles costs more than its shorter K saves).
constexpr double kSplitMinWeightBytes = 128.0 * (1 << 20);

// Output-tile width of the persistent kernel: 256 when those tiles fill the
// GPU, else the widest of 128 / 64 / 32 whose tiles occupy at least half the
// SMs (narrower tiles spread a small-M product's weight stream over more SMs).
static int gemm_tile_n_sm(int M, int N, int K, int sm) {
  const long long nM = (M + BM - 1) / BM;
  if (nM * ((N + 255) / 256) >= sm) return 256;
  // a large weight stream (tens of MB) at a few hundred rows: 256-wide tiles
  // few enough to be split along K over the SMs (persistent split-K)
  if (M > BM && M < kPairMinRows && 2.0 * N * K >= kSplitMinWeightBytes && nM * ((N + 255) / 256) * 2 <= sm)
    return 256;
  if (nM * ((N + 127) / 128) * 2 >= sm) return 128;
  if (nM * ((N + 63) / 64) * 2 >= sm) return 64;
  return 32;
}
int gemm_tile_n(int M, int N, int K) { return gemm_tile_n_sm(M, N, K, gemm_sm_count()); }

namespace {

int bn_code(int bn) { return bn == 256 ? 3 : bn == 128 ? 2 : bn == 64 ? 1 : 0; }

// k-blocks per stage of the persistent kernel: one TMA box then carries
// KS * 64 columns, so narrow tiles (whose per-box issue cost would dominate)
// take 4, 128-wide tiles 2, 256-wide tiles 1; fewer when K is no multiple.
int gemm_ks(int bn, int K) {
  int ks = bn == 256 ? 1 : bn == 128 ? 2 : 4;
  while (ks > 1 && K % (BK * ks) != 0) ks /= 2;
  return ks;
}
int cluster_smem(int bn, int kbs, int a_box) {
  return bn == 256   ? CCfg<256>::smem(kbs, a_box)
         : bn == 128 ? CCfg<128>::smem(kbs, a_box)
         : bn == 64  ? CCfg<64>::smem(kbs, a_box)
                     : CCfg<32>::smem(kbs, a_box);
}

// Issue time of one tcgen05.mma (M = 128, K = 16) by its N, in microseconds:
// measured on GB300 at about 50 cycles for N <= 64, 65 for 128 and 127 for
// 256 (where it is bound by the tensor core's throughput), at 1.9 GHz.
double mma_us(int bn) { return (bn <= 64 ? 50.0 : bn == 128 ? 65.0 : 127.0) / 1900.0; }
// Operand bytes one SM takes in: a few TMA boxes in flight land at about
// 115 GB/s, the first about 0.45 us after it is issued.
double load_us(double bytes) { return 0.45 + bytes / 115e3; }

}  // namespace

// How one Linear runs.  Rows of one 128-row tile (M <= 128) and a long K
// (at least 32 k-blocks): the cluster split-K kernel, whose exchange of
// partial tiles costs a few microseconds but which splits the many MMAs of a
// long K over S SMs; its tile width and S are the ones with the least
// estimated load and MMA-issue time per wave.  Otherwise the persistent
// kernel with gemm_tile_n's width.  (Measured on GB300 for M <= 128: with
// K = 768 the persistent kernel was faster for every N of GPT-2 small, with
// K = 3072 the cluster kernel by 30-40%.)
constexpr int kClusterMinKb = 32;
// Products of more than one row tile take the CTA-pair kernel when its tiles
// are shared out along K (PairSched), else the kernel with the lower estimate
// of its whole waves: waves x K-blocks x the time of one k-block of a tile,
// for a pair's 256 x 256 tile 1, for the single CTA's 128 x bn tile
// kSingleKb x (its operand bytes per k-block, A 16 KB + W bn x 128 B) / 48 KB
// - at bn = 256 the single CTA reaches 71% tensor-pipe activity against the
// pair's 84% (both operand-bound).  Measured on GB300 over the 13B Linears at
// 200-3000 rows (all 52 shapes) this picks the faster of the two every time:
// e.g. the Attn-Out at 512-768 rows 15-19% and the FC2 36% faster on pairs (one
// wave of 60 pair tiles against two of single-CTA tiles), the FC1 at 300-384
// and the QKV at 600 rows 10% faster on single CTAs (2 waves against 3).
constexpr double kSingleKb = 1.18;
static double single_waves_cost(int M, int N, int K, int sm) {
  const int bn = gemm_tile_n_sm(M, N, K, sm);
  const long long tiles = (long long)((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  const long long waves = (tiles + sm - 1) / sm;
  return (double)waves * (K / BK) * kSingleKb * (16.0 + bn / 8.0) / 48.0;
}
// The plan for a GPU of `sm` SMs (gemm_plan: this device's).
static GemmPlan gemm_plan_sm(int M, int N, int K, bool split_scratch, int sm) {
  GemmPlan p{};
  const long long pair_tiles = (long long)((M + 2 * BM - 1) / (2 * BM)) * ((N + 255) / 256);
  if (M > BM && K % BK == 0 && sm >= 2) {
    PairSched ps;
    ps.init(M, N, K, sm / 2, split_scratch);
    const long long pair_waves = (pair_tiles + sm / 2 - 1) / (sm / 2);
    p.split = ps.split();
    p.pair = p.split || (double)pair_waves * (K / BK) < single_waves_cost(M, N, K, sm);
  }
  if (p.pair) {
    p.bn = kPairBN;
    return p;
  }
  p.bn = gemm_tile_n_sm(M, N, K, sm);
  p.ks = gemm_ks(p.bn, K);
  const int KB = K / BK;
  if (M > BM || M <= 0) return p;
  const int a_box = M <= 64 ? 64 : 128;  // products of <= 64 rows load 64-row A boxes
  p.a_box = a_box;
  if (KB < kClusterMinKb) return p;
  double best = 1e30;
  for (int bn : {64, 128}) {
    const int nN = (N + bn - 1) / bn;
    for (int S : {4, 8}) {
      const int kbs = (KB + S - 1) / S;
      // one wave at most: with more waves the per-wave estimate below no longer
      // holds (measured: 64 x 15360 x 5120 took 4x its estimate)
      if (bn % (4 * S) != 0 || cluster_smem(bn, kbs, a_box) > kClusterSmemMax || nN * S > sm) continue;
      const long long waves = ((long long)nN * S + sm - 1) / sm;
      const double t = (double)waves * (load_us((double)kbs * (a_box + bn) * 128.0) + kbs * 4 * mma_us(bn));
      if (t < best) {
        best = t;
        p.cluster = true;
        p.bn = bn;
        p.S = S;
        p.kbs = kbs;
        p.a_box = a_box;
        p.ks = 1;
      }
    }
  }
  if (!p.cluster) {
    p.bn = gemm_tile_n_sm(M, N, K, sm);
    p.ks = gemm_ks(p.bn, K);
  }
  return p;
}
GemmPlan gemm_plan(int M, int N, int K, bool split_scratch) {
  return gemm_plan_sm(M, N, K, split_scratch, gemm_sm_count());
}

// A small integer naming the plan, below 64: callers pack one per Linear
// into 6 bits of their CUDA-graph keys (persistent 0..7, cluster 8..39,
// CTA pair 40, CTA pair with tiles shared out along K 41).
static int plan_code_of(const GemmPlan &p) {
  if (p.pair) return p.split ? 41 : 40;
  if (!p.cluster) return bn_code(p.bn) * 2 + (p.a_box == 64 ? 1 : 0);
  return 8 + bn_code(p.bn) * 8 + (p.S == 2 ? 0 : p.S == 4 ? 1 : 2) * 2 + (p.a_box == 64 ? 1 : 0);
}
int gemm_plan_code(int M, int N, int K) { return plan_code_of(gemm_plan(M, N, K, true)); }

cudaError_t gemm_prepare() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = set_smem_limit<32, 1>(dev);
  if (e == cudaSuccess) e = set_smem_limit<32, 2>(dev);
  if (e == cudaSuccess) e = set_smem_limit<32, 4>(dev);
  if (e == cudaSuccess) e = set_smem_limit<64, 1>(dev);
  if (e == cudaSuccess) e = set_smem_limit<64, 2>(dev);
  if (e == cudaSuccess) e = set_smem_limit<64, 4>(dev);
  if (e == cudaSuccess) e = set_smem_limit<128, 1>(dev);
  if (e == cudaSuccess) e = set_smem_limit<128, 2>(dev);
  if (e == cudaSuccess) e = set_smem_limit<256, 1>(dev);
  if (e == cudaSuccess) e = set_cluster_smem_limit<32>(dev);
  if (e == cudaSuccess) e = set_cluster_smem_limit<64>(dev);
  if (e == cudaSuccess) e = set_cluster_smem_limit<128>(dev);
  if (e == cudaSuccess) e = set_cluster_smem_limit<256>(dev);
  if (e == cudaSuccess) e = set_pair_smem_limit(dev);
  gemm_sm_count();
  return e;
}

// M selects the plan; with M_dev the kernel reads the row count from the
// device (the plan chosen from M must then stay valid for it: callers key
// their CUDA graphs on gemm_plan_code).  A and W come as 3-D views
// {64 columns, rows, K / 64} with boxes of 32 / 64 / 128 rows by 1 / 2 / 4
// k-blocks; the plan picks the ones it loads.
cudaError_t launch_gemm_tc_bf16(const OperandMaps &A, const OperandMaps &W, int M, const int32_t *M_dev, int N, int K,
                                const EpiParams &epi, const GemmScratch &scr, int32_t *status, cudaStream_t st) {
  if (M <= 0 && M_dev == nullptr) return cudaSuccess;
  if (K % BK != 0 || K <= 0) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int sm = gemm_sm_count();
  const GemmPlan p = gemm_plan(M, N, K, pair_split_ok(scr, sm / 2));
  if (p.pair) return launch_pair(A.get(BM, 1), W.get(BM, 1), M, M_dev, N, K, epi, scr, p.split, status, st, sm, dev);
  if (p.cluster) {
    switch (p.bn) {
      case 256: return launch_cluster<256>(A, W, M, M_dev, N, K, p.S, p.kbs, p.a_box, epi, status, st, dev);
      case 128: return launch_cluster<128>(A, W, M, M_dev, N, K, p.S, p.kbs, p.a_box, epi, status, st, dev);
      case 64: return launch_cluster<64>(A, W, M, M_dev, N, K, p.S, p.kbs, p.a_box, epi, status, st, dev);
      default: return launch_cluster<32>(A, W, M, M_dev, N, K, p.S, p.kbs, p.a_box, epi, status, st, dev);
    }
  }
  const int ks = p.ks;
  const CUtensorMap *a = A.get(p.a_box, ks);
#define ORCA_GEMM_CASE(BN_, KS_)                                                                          \
  if (p.bn == BN_ && ks == KS_)                                                                           \
    return launch_bn<BN_, KS_>(a, W.get(BN_ < 128 ? BN_ : 128, KS_), M, M_dev, N, K, p.a_box, epi, scr, status, st, \
                               sm, dev);
  ORCA_GEMM_CASE(256, 1)
  ORCA_GEMM_CASE(128, 2)
  ORCA_GEMM_CASE(128, 1)
  ORCA_GEMM_CASE(64, 4)
  ORCA_GEMM_CASE(64, 2)
  ORCA_GEMM_CASE(64, 1)
  ORCA_GEMM_CASE(32, 4)
  ORCA_GEMM_CASE(32, 2)
  ORCA_GEMM_CASE(32, 1)
#undef ORCA_GEMM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace orca

// Host-side views of the planning above (orca.h): no device is touched.
extern "C" int orca_gemm_plan_query(int32_t M, int32_t N, int32_t K, int32_t n_sms, int32_t with_scratch,
                                    orca_gemm_plan_info *out) {
  using namespace orca;
  if (out == nullptr || M <= 0 || N <= 0 || K <= 0 || K % BK != 0 || n_sms < 2 || n_sms > 4096) return ORCA_EINVAL;
  const GemmPlan p = gemm_plan_sm(M, N, K, with_scratch != 0, n_sms);
  orca_gemm_plan_info r{};
  r.code = plan_code_of(p);
  if (p.pair) {
    PairSched sc;
    sc.init(M, N, K, n_sms / 2, with_scratch != 0);
    r.kernel = 2;
    r.tile_m = kPairBM;
    r.tile_n = kPairBN;
    r.tiles = sc.tiles;
    r.k_split = sc.kind;
    r.ranges = sc.kind == 1 ? sc.S : sc.kind == 2 ? sc.P : 1;
    r.workers = sc.busy();
  } else if (p.cluster) {
    r.kernel = 1;
    r.tile_m = BM;
    r.tile_n = p.bn;
    r.tiles = (N + p.bn - 1) / p.bn;
    r.ranges = p.S;
    r.workers = r.tiles * p.S;
  } else {
    r.kernel = 0;
    r.tile_m = BM;
    r.tile_n = p.bn;
    r.tiles = ((M + BM - 1) / BM) * ((N + p.bn - 1) / p.bn);
    r.ranges = 1;
    r.workers = r.tiles < n_sms ? r.tiles : n_sms;
  }
  *out = r;
  return ORCA_OK;
}

extern "C" int orca_gemm_pair_segments(int32_t M, int32_t N, int32_t K, int32_t n_pairs, int32_t with_split,
                                       int32_t pair, int32_t *seg, int32_t max_seg) {
  using namespace orca;
  if (M <= 0 || N <= 0 || K <= 0 || K % BK != 0 || n_pairs <= 0 || pair < 0 || pair >= n_pairs || max_seg < 0 ||
      (max_seg > 0 && seg == nullptr))
    return ORCA_EINVAL;
  PairSched sc;
  sc.init(M, N, K, n_pairs, with_split != 0);
  PairSeg g;
  int n = 0;
  for (int j = 0; sc.segment(pair, j, g); ++j, ++n) {
    if (n >= max_seg) continue;  // counted, not written
    int32_t *r = seg + 9 * n;
    r[0] = g.tile;
    r[1] = g.m;
    r[2] = g.n;
    r[3] = g.kb0;
    r[4] = g.kb1;
    r[5] = g.pieces;
    r[6] = g.mine;
    r[7] = g.pieces > 1 ? sc.counter(g, 0u) / 2 : -1;
    r[8] = g.pieces > 1 ? sc.piece_slot(g, g.mine) : -1;
  }
  return n;
}
