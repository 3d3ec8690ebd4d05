// Token-wise, HBM-bound kernels of one selectively batched iteration:
// embedding gather (with the first LayerNorm), LayerNorm, greedy argmax; and
// the one-time vectors of a LayerNorm folded into the Linear after it.
//
// These operate on every row of the flattened [sum L_i, H] tensor without
// knowing which request a row belongs to (Orca walk-through, section on
// non-attention operators and Figure 5).  Rows are independent, so one warp
// (LayerNorm) or one CTA (embedding, argmax) per row, 16-byte accesses.
#include <cuda_bf16.h>
#include <stdint.h>

#include <climits>

#include "orca_internal.h"

namespace orca {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 4 consecutive elements as float.
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
  uint2 u = *reinterpret_cast<const uint2 *>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&u.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162 *>(&u.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = u;
}

// LayerNorm of one row by one warp: (x - mean) / sqrt(var + eps) * g + b,
// statistics in fp32, biased variance.  NV4 > 0: the row (NV4 float4 per
// lane) stays in registers, one read of x; NV4 == 0: three passes.
template <typename T, int NV4>
__device__ __forceinline__ void layernorm_row(const float *__restrict__ x, const float *__restrict__ g,
                                              const float *__restrict__ b, T *__restrict__ out, int row, int src,
                                              int H, int lane) {
  const float *xr = x + (int64_t)src * H;
  T *orow = out + (int64_t)row * H;
  if constexpr (NV4 > 0) {
    float4 v[NV4];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NV4; ++i) {
      v[i] = load4(xr + lane * 4 + i * 128);
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
    const float mean = warp_sum(s) / (float)H;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < NV4; ++i) {
      const float a = v[i].x - mean, bb = v[i].y - mean, cc = v[i].z - mean, d = v[i].w - mean;
      q += (a * a + bb * bb) + (cc * cc + d * d);
    }
    const float rstd = rsqrtf(warp_sum(q) / (float)H + 1e-5f);
#pragma unroll
    for (int i = 0; i < NV4; ++i) {
      const int c = lane * 4 + i * 128;
      const float4 gg = load4(g + c), bv = load4(b + c);
      store4(orow + c, make_float4((v[i].x - mean) * rstd * gg.x + bv.x, (v[i].y - mean) * rstd * gg.y + bv.y,
                                   (v[i].z - mean) * rstd * gg.z + bv.z, (v[i].w - mean) * rstd * gg.w + bv.w));
    }
  } else {
    float s = 0.f;
    for (int c = lane * 4; c < H; c += 128) {
      float4 v = load4(xr + c);
      s += (v.x + v.y) + (v.z + v.w);
    }
    const float mean = warp_sum(s) / (float)H;
    float q = 0.f;
    for (int c = lane * 4; c < H; c += 128) {
      float4 v = load4(xr + c);
      float a = v.x - mean, bb = v.y - mean, cc = v.z - mean, d = v.w - mean;
      q += (a * a + bb * bb) + (cc * cc + d * d);
    }
    const float rstd = rsqrtf(warp_sum(q) / (float)H + 1e-5f);
    for (int c = lane * 4; c < H; c += 128) {
      float4 v = load4(xr + c), gg = load4(g + c), bv = load4(b + c);
      store4(orow + c, make_float4((v.x - mean) * rstd * gg.x + bv.x, (v.y - mean) * rstd * gg.y + bv.y,
                                   (v.z - mean) * rstd * gg.z + bv.z, (v.w - mean) * rstd * gg.w + bv.w));
    }
  }
}

// x[r] = tok_emb[tok_r] + pos_emb[pos_r]  (fp32 residual stream), one CTA
// per row.  With ln_out, warp 0 then takes the row's LayerNorm (the first
// block's LN1) from the x just written, so that no separate launch reads x.
template <typename T>
__global__ void embed_kernel(const RowInfo *__restrict__ rows, int n_rows_arg, const int32_t *n_rows_dev,
                             const T *__restrict__ tok_emb, const T *__restrict__ pos_emb, float *__restrict__ x,
                             int H, int vocab, int max_pos, int32_t *status, const float *__restrict__ ln_g,
                             const float *__restrict__ ln_b, T *__restrict__ ln_out,
                             unsigned long long *stamp_start, unsigned long long *stamp) {
  pdl_trigger();
  const int n_rows = n_rows_dev ? *n_rows_dev : n_rows_arg;
  pdl_wait();
  if (stamp_start != nullptr && blockIdx.x == 0 && threadIdx.x == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    *stamp_start = t;
  }
  for (int r = blockIdx.x; r < n_rows; r += gridDim.x) {
    const RowInfo ri = rows[r];
    if (ri.tok < 0 || ri.tok >= vocab || ri.pos < 0 || ri.pos >= max_pos) {
      if (threadIdx.x == 0) atomicOr(status, kStatusBadIndex);
      continue;
    }
    const T *te = tok_emb + (int64_t)ri.tok * H;
    const T *pe = pos_emb + (int64_t)ri.pos * H;
    float *xr = x + (int64_t)r * H;
    for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
      float4 a = load4(te + c), b = load4(pe + c);
      store4(xr + c, make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w));
    }
    if (ln_out != nullptr) {
      __syncthreads();  // the row of x is written
      if (threadIdx.x < 32) layernorm_row<T, 0>(x, ln_g, ln_b, ln_out, r, r, H, threadIdx.x);
    }
  }
  __syncthreads();
  stamp_end(stamp);
}

// out[i] = LayerNorm(x[src_i]), one warp per output row, rows grid-strided;
// src_i = i, or the last row of request i when `gather` is given (final
// LayerNorm on the rows whose logits are sampled).
template <typename T, int NV4>
__global__ void layernorm_kernel(const float *__restrict__ x, const float *__restrict__ g,
                                 const float *__restrict__ b, T *__restrict__ out, int n_rows_arg,
                                 const int32_t *n_rows_dev, int H, const ReqInfo *__restrict__ gather,
                                 unsigned long long *zero_keys, unsigned long long *stamp) {
  pdl_trigger();
  const int n_rows = n_rows_dev ? *n_rows_dev : n_rows_arg;
  const int lane = threadIdx.x & 31;
  const int wpc = blockDim.x / 32;
  pdl_wait();
  for (int row = blockIdx.x * wpc + threadIdx.x / 32; row < n_rows; row += gridDim.x * wpc) {
    layernorm_row<T, NV4>(x, g, b, out, row, gather ? gather[row].row_off + gather[row].n_new - 1 : row, H, lane);
    if (zero_keys != nullptr && lane == 0) zero_keys[row] = 0ull;
  }
  __syncthreads();
  stamp_end(stamp);
}

// (value, index) order of the greedy choice: larger value wins, equal values
// go to the lower index, NaN never wins.  idx < 0 means "nothing yet".
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  if (i < 0) return false;
  if (bi < 0) return v == v;  // anything but NaN beats nothing
  return v > bv || (v == bv && i < bi);
}

__global__ void argmax_kernel(const float *__restrict__ logits, int V, int32_t *__restrict__ out,
                              unsigned long long *__restrict__ keys) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  const float *lr = logits + (int64_t)r * V;
  float bv = -INFINITY;
  int bi = -1;
  for (int c = threadIdx.x; c < V; c += blockDim.x) {
    const float v = lr[c];
    if (better(v, c, bv, bi)) { bv = v; bi = c; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  __shared__ float sv[32];
  __shared__ int si[32];
  const int w = threadIdx.x / 32, lane = threadIdx.x & 31;
  if (lane == 0) { sv[w] = bv; si[w] = bi; }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x / 32;
    bv = lane < nw ? sv[lane] : -INFINITY;
    bi = lane < nw ? si[lane] : -1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) {
      if (keys != nullptr)
        keys[r] = bi < 0 ? 0ull : argmax_key(bv, bi);
      else
        out[r] = bi;
    }
  }
}

// c[n] = sum_k gamma_k W[n, k], d[n] = bias[n] + sum_k beta_k W[n, k]: one
// warp per output column n, fp32 sums over the bf16 row W[n, :].
__global__ void ln_fold_vectors_kernel(const __nv_bfloat16 *__restrict__ W, const float *__restrict__ gamma,
                                       const float *__restrict__ beta, const float *__restrict__ bias, int N, int K,
                                       float *__restrict__ c, float *__restrict__ d) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (n >= N) return;
  const __nv_bfloat16 *wr = W + (int64_t)n * K;
  float sc = 0.f, sd = 0.f;
  for (int k = lane; k < K; k += 32) {
    const float w = __bfloat162float(wr[k]);
    sc += gamma[k] * w;
    sd += beta[k] * w;
  }
  sc = warp_sum(sc);
  sd = warp_sum(sd);
  if (lane == 0) {
    c[n] = sc;
    d[n] = (bias != nullptr ? bias[n] : 0.f) + sd;
  }
}

}  // namespace

cudaError_t launch_embed(int dtype, const RowInfo *rows, int n_rows, const int32_t *n_rows_dev, const void *tok_emb,
                         const void *pos_emb, float *x, int H, int vocab, int max_pos, int32_t *status,
                         const float *ln_g, const float *ln_b, void *ln_out, unsigned long long *stamp_start,
                         unsigned long long *stamp, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  const int threads = H >= 512 ? 128 : 32;
  const int grid = n_rows < 1184 ? n_rows : 1184;
  if ((ln_out != nullptr) != (ln_g != nullptr && ln_b != nullptr)) return cudaErrorInvalidValue;
  if (dtype == 1)
    return launch_pdl(embed_kernel<__nv_bfloat16>, grid, threads, 0, st, rows, n_rows, n_rows_dev,
                      static_cast<const __nv_bfloat16 *>(tok_emb), static_cast<const __nv_bfloat16 *>(pos_emb), x, H,
                      vocab, max_pos, status, ln_g, ln_b, static_cast<__nv_bfloat16 *>(ln_out), stamp_start, stamp);
  return launch_pdl(embed_kernel<float>, grid, threads, 0, st, rows, n_rows, n_rows_dev,
                    static_cast<const float *>(tok_emb), static_cast<const float *>(pos_emb), x, H, vocab, max_pos,
                    status, ln_g, ln_b, static_cast<float *>(ln_out), stamp_start, stamp);
}

cudaError_t launch_ln_fold_vectors(const void *W, const float *gamma, const float *beta, const float *bias, int N,
                                   int K, float *c, float *d, cudaStream_t st) {
  if (N <= 0 || K <= 0) return cudaErrorInvalidValue;
  const int warps = 8;
  ln_fold_vectors_kernel<<<(N + warps - 1) / warps, 32 * warps, 0, st>>>(
      static_cast<const __nv_bfloat16 *>(W), gamma, beta, bias, N, K, c, d);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t layernorm_t(const float *x, const float *g, const float *b, T *out, int n_rows,
                               const int32_t *n_rows_dev, int H, const ReqInfo *gather, unsigned long long *zk,
                               unsigned long long *stamp, cudaStream_t st) {
  const int rows_per_cta = 8;
  int grid = (n_rows + rows_per_cta - 1) / rows_per_cta;
  if (grid > 1184) grid = 1184;
  const dim3 block(32 * rows_per_cta);
  switch (H) {
    case 768: return launch_pdl(layernorm_kernel<T, 6>, grid, block, 0, st, x, g, b, out, n_rows, n_rows_dev, H, gather, zk,
                                  stamp);
    case 1024: return launch_pdl(layernorm_kernel<T, 8>, grid, block, 0, st, x, g, b, out, n_rows, n_rows_dev, H, gather, zk,
                                  stamp);
    case 2048: return launch_pdl(layernorm_kernel<T, 16>, grid, block, 0, st, x, g, b, out, n_rows, n_rows_dev, H, gather, zk,
                                  stamp);
    default: return launch_pdl(layernorm_kernel<T, 0>, grid, block, 0, st, x, g, b, out, n_rows, n_rows_dev, H, gather, zk,
                                  stamp);
  }
}

cudaError_t launch_layernorm(int dtype, const float *x, const float *g, const float *b, void *out, int n_rows,
                             const int32_t *n_rows_dev, int H, const ReqInfo *gather, unsigned long long *zero_keys,
                             unsigned long long *stamp, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  if (dtype == 1)
    return layernorm_t(x, g, b, static_cast<__nv_bfloat16 *>(out), n_rows, n_rows_dev, H, gather, zero_keys, stamp,
                       st);
  return layernorm_t(x, g, b, static_cast<float *>(out), n_rows, n_rows_dev, H, gather, zero_keys, stamp, st);
}

cudaError_t launch_argmax(const float *logits, int n_rows, int vocab, int32_t *out, unsigned long long *keys,
                          cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  return launch_pdl(argmax_kernel, n_rows, 512, 0, st, logits, vocab, out, keys);
}

}  // namespace orca
