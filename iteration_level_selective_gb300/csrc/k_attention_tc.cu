// Prefill attention on the tensor cores (tcgen05 + TMEM), bf16 heads of 64 or 128.
//
// The per-request attention of Figure 5 (Orca walk-through) for the rows of
// a prompt is a dense, causal contraction: S = Q K^T over the request's own
// keys, softmax, O = P V.  One work item is up to 128 query rows of one
// request and one head; persistent CTA i takes item i, and further items from
// an atomic ticket when the items outnumber the CTAs.
//
// One pass over the key tiles (128 keys each) with an online softmax, the
// roles of a CTA running as a pipeline:
//   warp 0     claims items and loads Q, then K and V tiles by TMA into two
//              rings of stages, K one tile ahead of V: a K stage is free
//              once S of its tile is done, a V stage once P V is;
//   warp 1     issues the MMAs: S = Q K^T into one of two TMEM buffers, and
//              O += P V into a TMEM accumulator (V is the B operand as it
//              lies in the K/V pool, head dim contiguous: MN-major);
//   warps 2-9  softmax in two groups of four warps: warp w and warp w + 4
//              share one TMEM lane quarter, so each query row (one TMEM lane)
//              has two threads, one per half of the tile's 128 keys.  They
//              read their half of the row of S, mask the keys past the row's
//              position and swap their half-row maxima through shared memory
//              (a named barrier per lane quarter), so both keep the same
//              running max m; each keeps the sum l of its half and writes its
//              half of P = exp2((S - m) * log2(e)/sqrt(d)) as bf16 into
//              tensor memory, in one of two P buffers, from where the P V
//              MMA reads it as its A operand.  O is
//              rescaled, half of its columns by each, only when m grows by
//              more than a factor 2^8 (until then P may exceed 1, which fp32
//              and bf16 hold as well); at the end the two sums are added and
//              each thread writes its half of the row of O / l.
// While the softmax warps work on tile t the tensor core computes S of tile
// t+1 and P V of tile t-1; with two P buffers the softmax of tile t waits only
// for P V of tile t-2 (and, when O must be rescaled, of tile t-1).  Keys beyond the item's causal range are masked by
// selection; their V rows are zeroed in shared memory before P V, so stale
// slot contents never reach O.  Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "orca_internal.h"

namespace orca {
namespace {

constexpr int kRows = 128;       // query rows per item = TMEM lanes
constexpr int kKeys = 128;       // keys per tile
constexpr int kThreadsTc = 320;  // warp 0 loads, warp 1 issues MMAs, warps 2-9 softmax
constexpr int kSoftmaxThreads = 256;
constexpr int kHalf = kKeys / 2;  // keys of a tile per softmax thread
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct TcCfg {
  static constexpr int KB = D / 64;                // 64-element blocks of the head dim
  // K and V rings, freed apart: a K stage once S of its tile is done, a V
  // stage once P V is (measured on the 13B prompts: 0.79 -> 0.66 ms a layer
  // against one ring of K/V pairs freed by P V; a third K stage gained nothing)
  static constexpr int NSK = D == 128 ? 2 : 4;
  static constexpr int NSV = D == 128 ? 2 : 4;
  static constexpr int Q_BYTES = KB * kRows * 128;
  static constexpr int K_BYTES = KB * kKeys * 128;  // K-major: key rows of 128 B per block
  static constexpr int V_BYTES = KB * kKeys * 128;  // same bytes, read as an MN-major operand
  static constexpr int SMEM = Q_BYTES + NSK * K_BYTES + NSV * V_BYTES + 1024;
  // S0 [0,128), S1 [128,256), O [256, 256+D), P0 [384,448), P1 [448,512):
  // P as bf16 pairs, 64 columns per 128-key tile
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 256;
  static constexpr uint32_t P_COL = 384;
  // kind::f16: D fp32 (bit 4), A bf16 (bits 7-9), B bf16 (bits 10-12),
  // B MN-major (bit 16) for P V, N >> 3 (bits 17-22), M >> 4 (bits 24-28)
  static constexpr uint32_t IDESC_S =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kKeys >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
  static constexpr uint32_t IDESC_O = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                      ((uint32_t)(D >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
};

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptors, 128-byte swizzle (layout 2), version 1.
// K-major: 8-row groups 1024 B apart (SBO), leading offset unused.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// MN-major: rows of 64 MN-elements (128 B) along K; 8-row groups along K are
// `sbo` apart, 64-element column blocks along MN are `lbo` apart.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
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

// D (+)= A B with A (M x K) in tensor memory: lane = row, K packed two bf16
// to a column.
__device__ __forceinline__ void tc_mma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive TMEM columns of this thread's lane (warp-collective).
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

// 64 consecutive TMEM columns of this thread's lane (warp-collective).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float *v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63"
      "}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barrier of the two softmax warps that share a TMEM lane quarter.
__device__ __forceinline__ void pair_barrier(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }


__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Hardware base-2 exponential (PTX ex2.approx; ftz).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One claimed work item, decoded by the loader for the other roles.
struct TcItem {
  int head, r0, nq, p0;  // query rows r0 .. r0+nq-1 at positions p0 ..
  int kv_len, n_tiles;   // keys 0 .. kv_len-1; n_tiles < 0 ends the CTA
  int block_off;         // paged K/V: the request's block table, else -1
  long long krow0;       // contiguous: row of key 0 in the [n_heads * n_slots, D] view;
                         // paged: row of the head's slot 0
};

template <int NSK, int NSV>
struct TcShared {
  uint64_t q_full, q_empty;
  uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], o_done[2];  // per P buffer: P written; P V with it done
  uint64_t it_full[2], it_empty[2];
  TcItem it[2];
  float half_max[2][2][kRows];  // [tile parity][key half][row]: the softmax halves' maxima
  float half_sum[2][kRows];     // [key half][row]: each half's sum at the end of an item
  uint32_t tmem;
  int abort;
};

// All lanes of the warp wait; the warp continues only if every lane saw the
// phase (so the warp-collective TMEM accesses that follow stay converged).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
  const bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kThreadsTc, 1)
    prefill_attention_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKb,
                                const __grid_constant__ CUtensorMap tmVb, TcAttnArgs a) {
  using C = TcCfg<D>;
  constexpr int NSK = C::NSK, NSV = C::NSV;
  extern __shared__ uint8_t smem_raw[];
  __shared__ TcShared<NSK, NSV> sh;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *sQ = smem_raw + pad;
  uint8_t *sK = sQ + C::Q_BYTES;        // NSK stages of K
  uint8_t *sV = sK + NSK * C::K_BYTES;  // NSV stages of V
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.s_empty[b], kSoftmaxThreads);
      mbar_init(&sh.it_full[b], 1);
      mbar_init(&sh.it_empty[b], 1 + 8);  // the MMA warp and the eight softmax warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.p_full[b], kSoftmaxThreads);
      mbar_init(&sh.o_done[b], 1);
    }
    sh.abort = 0;
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmKb)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmVb)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;
  volatile int *abort_flag = &sh.abort;
  // The next kernel may start only once this CTA holds its tensor memory: a
  // dependent CTA that allocated first and then waited for this kernel could
  // otherwise leave it without columns.
  pdl_trigger();
  pdl_wait();  // q and the K/V slots come from the QKV Linear; the output rows are its input
  const int n_work = a.n_work_dev ? *a.n_work_dev : a.n_work;  // descriptor header, written before the forward
  const int total = n_work * a.n_heads;
  // CTA i takes item i first; only when there are more items than CTAs do
  // the rest go out by ticket (so a small batch costs no atomics at all)
  const bool ticketed = total > (int)gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      uint32_t n_item = 0, g = 0;  // items enqueued, K/V tiles loaded
      bool first = true;
      while (!*abort_flag) {
        const int t = first ? (int)blockIdx.x : ticketed ? (int)gridDim.x + atomicAdd(a.ticket, 1) : total;
        first = false;
        TcItem it{};
        it.n_tiles = -1;
        if (t < total) {
          // ticket -> (request group, head, query tile): a group is one
          // request's query tiles (work[G .. G+T-1]); its tickets run over
          // the heads, the tiles of one head consecutive (shared K/V in L2)
          const int g0 = a.work[t / a.n_heads].kind;
          const int G = g0 >> 10, T = g0 & 1023;
          const int local = t - G * a.n_heads;
          const int head = T > 0 ? local / T : a.n_heads;
          const int wi = T > 0 ? G + local % T : 0;
          const AttnWork w = a.work[wi < n_work ? wi : 0];
          const ReqInfo rq = a.reqs[w.req];
          it.head = head;
          it.r0 = w.a;
          it.nq = w.b;
          it.p0 = rq.ctx + (w.a - rq.row_off);
          it.kv_len = it.p0 + w.b;
          it.block_off = rq.block_off;
          it.krow0 = (long long)head * a.n_slots + (rq.block_off < 0 ? rq.slot_base : 0);
          it.n_tiles = (it.kv_len + kKeys - 1) / kKeys;
          const bool keys_ok = rq.block_off < 0
                                   ? rq.slot_base >= 0 && (int64_t)rq.slot_base + it.kv_len <= a.n_slots
                                   : (int64_t)rq.n_blocks * kKvBlock >= it.kv_len;
          if (T <= 0 || wi >= n_work || local < 0 || head >= a.n_heads || !keys_ok || w.b > kRows || w.b <= 0 ||
              it.p0 < 0) {
            atomicOr(a.status, kStatusBadIndex);
            continue;
          }
        }
        const uint32_t slot = n_item & 1;
        if (n_item >= 2 && !mbar_wait(&sh.it_empty[slot], ((n_item - 2) >> 1) & 1, abort_flag, a.status)) break;
        sh.it[slot] = it;
        mbar_arrive(&sh.it_full[slot]);
        ++n_item;
        if (it.n_tiles < 0) break;
        // Q of this item once the previous item's S products are done
        if (n_item >= 2 && !mbar_wait(&sh.q_empty, (n_item - 2) & 1, abort_flag, a.status)) break;
        mbar_expect_tx(&sh.q_full, C::Q_BYTES);
        for (int kb = 0; kb < C::KB; ++kb)
          tma_load_2d(sQ + kb * kRows * 128, &tmQ, it.head * D + kb * 64, it.r0, &sh.q_full);
        // K of tile t goes in as soon as S of the tile NSK earlier has used
        // its stage; V of tile t - 1 after it, once P V of the tile NSV earlier
        // has used its stage (V is needed only after a tile's softmax), so a
        // late P V never holds back the next S products
        auto runs = [&](int tile, int *rows) {  // paged: the tile's block runs (past the keys: none)
          int n_runs = 0;
          for (int j = 0; j < kKeys / kKvBlock; ++j) {
            const int k0 = tile * kKeys + j * kKvBlock;
            if (k0 >= it.kv_len) break;
            const int blk = a.blocks[it.block_off + k0 / kKvBlock];
            const long long run =
                (blk >= 0 && (long long)(blk + 1) * kKvBlock <= a.n_slots) ? it.krow0 + (long long)blk * kKvBlock : -1;
            if (run < 0) {
              atomicOr(a.status, kStatusBadIndex);
              break;
            }
            rows[n_runs++] = (int)run;
          }
          return n_runs;
        };
        auto load = [&](int tile, uint32_t gt, bool is_v) {
          const uint32_t ns = is_v ? NSV : NSK, s = gt % ns, use = gt / ns;
          if (use >= 1 && !mbar_wait(is_v ? &sh.v_empty[s] : &sh.k_empty[s], (use - 1) & 1, abort_flag, a.status))
            return false;
          uint8_t *dst = (is_v ? sV + s * C::V_BYTES : sK + s * C::K_BYTES);
          uint64_t *bar = is_v ? &sh.v_full[s] : &sh.k_full[s];
          if (it.block_off < 0) {  // contiguous slots: one 128-row box per 64-column block
            const int krow = (int)(it.krow0 + (long long)tile * kKeys);
            mbar_expect_tx(bar, C::K_BYTES);
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(dst + kb * kKeys * 128, is_v ? &tmV : &tmK, kb * 64, krow, bar);
            return true;
          }
          // paged: the tile's keys in blocks of kKvBlock slots; blocks past the
          // item's keys are not loaded (their rows are masked, and zeroed in V,
          // before use)
          int rows[kKeys / kKvBlock];
          const int n_runs = runs(tile, rows);
          mbar_expect_tx(bar, n_runs * C::KB * kKvBlock * 128);
          for (int j = 0; j < n_runs; ++j)
            for (int kb = 0; kb < C::KB; ++kb)
              tma_load_2d(dst + kb * kKeys * 128 + j * kKvBlock * 128, is_v ? &tmVb : &tmKb, kb * 64, rows[j], bar);
          return true;
        };
        bool ok = true;
        for (int tile = 0; tile <= it.n_tiles && ok; ++tile) {
          if (tile < it.n_tiles) ok = load(tile, g + tile, false);
          if (ok && tile >= 1) ok = load(tile - 1, g + tile - 1, true);
        }
        g += it.n_tiles;
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t n_item = 0, g = 0;
    const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV);
    while (true) {
      const uint32_t slot = n_item & 1;
      if (!warp_wait(&sh.it_full[slot], (n_item >> 1) & 1, abort_flag, a.status)) break;
      const TcItem it = sh.it[slot];
      if (it.n_tiles < 0) break;
      if (!warp_wait(&sh.q_full, n_item & 1, abort_flag, a.status)) break;
      bool ok = true;
      for (int tile = 0; tile <= it.n_tiles; ++tile) {
        if (tile < it.n_tiles) {  // S(tile) = Q K^T into buffer (g + tile) & 1
          const uint32_t gt = g + tile, s = gt % NSK, b = gt & 1, use_b = gt >> 1;
          if ((use_b >= 1 && !warp_wait(&sh.s_empty[b], (use_b - 1) & 1, abort_flag, a.status)) ||
              !warp_wait(&sh.k_full[s], (gt / NSK) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            tc_fence_after();
            for (int kb = 0; kb < C::KB; ++kb)
              for (int k = 0; k < 4; ++k)
                tc_mma(tmem + b * 128, sw128_desc(qa + kb * kRows * 128 + k * 32),
                       sw128_desc(ka + s * C::K_BYTES + kb * kKeys * 128 + k * 32), C::IDESC_S,
                       (kb | k) ? 1u : 0u);
            tc_commit(&sh.s_full[b]);
            tc_commit(&sh.k_empty[s]);
            if (tile == it.n_tiles - 1) tc_commit(&sh.q_empty);
          }
          __syncwarp();
        }
        if (tile >= 1) {  // O += P(tile-1) V(tile-1)
          const int tp = tile - 1;
          const uint32_t gp = g + tp, s = gp % NSV, pb = gp & 1;
          if (!warp_wait(&sh.p_full[pb], (gp >> 1) & 1, abort_flag, a.status) ||
              !warp_wait(&sh.v_full[s], (gp / NSV) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          const int valid = it.kv_len - tp * kKeys;  // V rows holding keys of this item
          if (valid < kKeys) {
            uint8_t *vt = sV + s * C::V_BYTES;
            const int n_chunks = (kKeys - valid) * C::KB * 8;
            for (int c = lane; c < n_chunks; c += 32) {
              const int r = valid + c / (C::KB * 8), rem = c % (C::KB * 8);
              *reinterpret_cast<uint4 *>(vt + (rem >> 3) * kKeys * 128 + r * 128 + (rem & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
          }
          __syncwarp();
          if (lane == 0) {
            tc_fence_after();
            for (int kk = 0; kk < kKeys / 16; ++kk)  // 16 keys = 8 columns of the P buffer
              tc_mma_ts(tmem + C::O_COL, tmem + C::P_COL + pb * 64 + kk * 8,
                        sw128_mn_desc(va + s * C::V_BYTES + kk * 2048, kKeys * 128, 1024), C::IDESC_O,
                        (tp | kk) ? 1u : 0u);
            tc_commit(&sh.v_empty[s]);
            tc_commit(&sh.o_done[pb]);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      g += it.n_tiles;
      if (lane == 0) mbar_arrive(&sh.it_empty[slot]);
      ++n_item;
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;         // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // keys [half * 64, half * 64 + 64) of every tile
    const int row = quad * 32 + lane;  // query row of this thread
    const int bar_id = 1 + quad;       // the two warps of this lane quarter
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    constexpr int DH = D / 2;          // output columns of this thread's half
    uint32_t n_item = 0, g = 0;
    // P V of global tile j has completed once phase j >> 1 of o_done[j & 1] has
    auto pv_done = [&](uint32_t j) {
      return warp_wait(&sh.o_done[j & 1], (j >> 1) & 1, abort_flag, a.status);
    };
    while (true) {
      const uint32_t slot = n_item & 1;
      if (!warp_wait(&sh.it_full[slot], (n_item >> 1) & 1, abort_flag, a.status)) break;
      const TcItem it = sh.it[slot];
      if (it.n_tiles < 0) break;
      const int my_pos = row < it.nq ? it.p0 + row : -1;  // -1: no key is visible to this row
      float m = -INFINITY, l = 0.f;  // l: the sum over this thread's half of the keys
      bool ok = true;
      for (int tile = 0; tile < it.n_tiles; ++tile) {
        const uint32_t gt = g + tile, b = gt & 1;
        if (!warp_wait(&sh.s_full[b], (gt >> 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float v[kHalf];
        tmem_ld64(tl + b * 128 + half * kHalf, v);
        tc_fence_before();
        mbar_arrive(&sh.s_empty[b]);
        const int k0 = tile * kKeys + half * kHalf;
        if (k0 + kHalf - 1 > my_pos) {
#pragma unroll
          for (int i = 0; i < kHalf; ++i)
            if (k0 + i > my_pos) v[i] = -INFINITY;
        }
        float mx[8];  // eight independent chains, then a tree
#pragma unroll
        for (int j = 0; j < 8; ++j) mx[j] = v[j];
#pragma unroll
        for (int i = 8; i < kHalf; ++i) mx[i & 7] = fmaxf(mx[i & 7], v[i]);
        const float hmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        // both threads of the row take the maximum of the two halves, so they
        // keep the same running max and rescale decision
        sh.half_max[b][half][row] = hmax;
        pair_barrier(bar_id);
        const float tmax = fmaxf(hmax, sh.half_max[b][half ^ 1][row]);
        const float m_new = fmaxf(m, tmax);
        const bool need = (m_new - m) * a.scale_log2 > kRescaleLog2;  // false while both are -inf
        float alpha = 1.f;
        if (need) {
          alpha = m == -INFINITY ? 0.f : ex2((m - m_new) * a.scale_log2);
          l *= alpha;
          m = m_new;
        }
        const float ms = m == -INFINITY ? 0.f : m * a.scale_log2;
        uint32_t pk[kHalf / 2];
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kHalf; i += 2) {
          const float p0 = ex2(fmaf(v[i], a.scale_log2, -ms));
          const float p1 = ex2(fmaf(v[i + 1], a.scale_log2, -ms));
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
          ls[(i >> 1) & 7] += __low2float(b2) + __high2float(b2);  // the P that reaches the MMA
          pk[i / 2] = *reinterpret_cast<const uint32_t *>(&b2);
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        // P buffer gt & 1 is free once P V of tile gt - 2 is done; O may be
        // rescaled only once P V of the previous tile (the last to add to it) is
        if ((gt >= 2 && !pv_done(gt - 2)) || (tile > 0 && __any_sync(0xffffffffu, need) && !pv_done(gt - 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (tile > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = half * DH; c < half * DH + DH; c += 32) {
            float o[32];
            tmem_ld32(tl + C::O_COL + c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tl + C::O_COL + c, o);
          }
        }
        // this half's 64 keys: 32 columns of bf16 pairs in P buffer gt & 1
        tmem_st32(tl + C::P_COL + (gt & 1) * 64 + half * 32, reinterpret_cast<const float *>(pk));
        tc_fence_before();
        mbar_arrive(&sh.p_full[gt & 1]);
      }
      if (!ok) break;
      // ---- O / l -> output rows (l = the two halves' sums)
      if (!pv_done(g + it.n_tiles - 1)) break;
      tc_fence_after();
      sh.half_sum[half][row] = l;
      pair_barrier(bar_id);
      const float lt = l + sh.half_sum[half ^ 1][row];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(a.out) + (int64_t)(it.r0 + row) * a.hidden + it.head * D;
#pragma unroll 1
      for (int c = half * DH; c < half * DH + DH; c += 32) {
        float o[32];
        tmem_ld32(tl + C::O_COL + c, o);
        if (row < it.nq) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t pk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[q4 * 8 + 2 * j] * inv, o[q4 * 8 + 2 * j + 1] * inv);
              pk[j] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            *reinterpret_cast<uint4 *>(orow + c + q4 * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
      }
      tc_fence_before();
      if (lane == 0) mbar_arrive(&sh.it_empty[slot]);
      g += it.n_tiles;
      ++n_item;
    }
  }

  // teardown: the last CTA out resets the ticket (when it was used); free tensor memory
  __syncthreads();
  if (threadIdx.x == 0) {
    if (ticketed) {
      __threadfence();
      if (atomicAdd(a.ticket + 1, 1) == (int)gridDim.x - 1) {
        a.ticket[0] = 0;
        a.ticket[1] = 0;
      }
    }
    if (*abort_flag) drain_after_abort();
  }
  __syncthreads();
  stamp_end(a.stamp);
  if (warp == 1) {
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

cudaError_t launch_attention_tc(int head_dim, const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                                const CUtensorMap *tmKb, const CUtensorMap *tmVb, const TcAttnArgs &a, int n_work,
                                cudaStream_t st) {
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
    return launch_pdl(prefill_attention_tc_kernel<64>, grid, kThreadsTc, TcCfg<64>::SMEM, st, *tmQ, *tmK, *tmV, *tmKb,
                      *tmVb, a);
  }
  if (head_dim == 128) {
    e = set_limit<128>(dev);
    if (e != cudaSuccess) return e;
    return launch_pdl(prefill_attention_tc_kernel<128>, grid, kThreadsTc, TcCfg<128>::SMEM, st, *tmQ, *tmK, *tmV,
                      *tmKb, *tmVb, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace orca
