// Token-wise, HBM-bound kernels of one selectively batched iteration:
// embedding gather, LayerNorm, greedy argmax.
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

// x[r] = tok_emb[tok_r] + pos_emb[pos_r]  (fp32 residual stream)
template <typename T>
__global__ void embed_kernel(const RowInfo *__restrict__ rows, const T *__restrict__ tok_emb,
                             const T *__restrict__ pos_emb, float *__restrict__ x, int H, int vocab,
                             int max_pos, int32_t *status) {
  const int r = blockIdx.x;
  const RowInfo ri = rows[r];
  if (ri.tok < 0 || ri.tok >= vocab || ri.pos < 0 || ri.pos >= max_pos) {
    if (threadIdx.x == 0) atomicOr(status, kStatusBadIndex);
    return;
  }
  const T *te = tok_emb + (int64_t)ri.tok * H;
  const T *pe = pos_emb + (int64_t)ri.pos * H;
  float *xr = x + (int64_t)r * H;
  for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
    float4 a = load4(te + c), b = load4(pe + c);
    store4(xr + c, make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w));
  }
}

// out[i] = LayerNorm(x[src_i]) * g + b, one warp per output row; src_i = i,
// or the last row of request i when `gather` is given (final LayerNorm on
// the rows whose logits are sampled).  Statistics in fp32, biased variance.
template <typename T>
__global__ void layernorm_kernel(const float *__restrict__ x, const float *__restrict__ g,
                                 const float *__restrict__ b, T *__restrict__ out, int n_rows, int H,
                                 const ReqInfo *__restrict__ gather) {
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  const int src = gather ? gather[row].row_off + gather[row].n_new - 1 : row;
  const float *xr = x + (int64_t)src * H;
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
  T *orow = out + (int64_t)row * H;
  for (int c = lane * 4; c < H; c += 128) {
    float4 v = load4(xr + c), gg = load4(g + c), bv = load4(b + c);
    store4(orow + c, make_float4((v.x - mean) * rstd * gg.x + bv.x, (v.y - mean) * rstd * gg.y + bv.y,
                                 (v.z - mean) * rstd * gg.z + bv.z, (v.w - mean) * rstd * gg.w + bv.w));
  }
}

// (value, index) order of the greedy choice: larger value wins, equal values
// go to the lower index, NaN never wins.  idx < 0 means "nothing yet".
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  if (i < 0) return false;
  if (bi < 0) return v == v;  // anything but NaN beats nothing
  return v > bv || (v == bv && i < bi);
}

__global__ void argmax_kernel(const float *__restrict__ logits, int V, int32_t *__restrict__ out) {
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
    if (lane == 0) out[r] = bi;
  }
}

}  // namespace

cudaError_t launch_embed(int dtype, const RowInfo *rows, int n_rows, const void *tok_emb,
                         const void *pos_emb, float *x, int H, int vocab, int max_pos, int32_t *status,
                         cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  const int threads = H >= 512 ? 128 : 32;
  if (dtype == 1)
    embed_kernel<__nv_bfloat16><<<n_rows, threads, 0, st>>>(
        rows, static_cast<const __nv_bfloat16 *>(tok_emb), static_cast<const __nv_bfloat16 *>(pos_emb), x, H,
        vocab, max_pos, status);
  else
    embed_kernel<float><<<n_rows, threads, 0, st>>>(rows, static_cast<const float *>(tok_emb),
                                                     static_cast<const float *>(pos_emb), x, H, vocab,
                                                     max_pos, status);
  return cudaGetLastError();
}

cudaError_t launch_layernorm(int dtype, const float *x, const float *g, const float *b, void *out, int n_rows,
                             int H, const ReqInfo *gather, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  const int rows_per_cta = 4;
  const int grid = (n_rows + rows_per_cta - 1) / rows_per_cta;
  if (dtype == 1)
    layernorm_kernel<__nv_bfloat16><<<grid, 32 * rows_per_cta, 0, st>>>(
        x, g, b, static_cast<__nv_bfloat16 *>(out), n_rows, H, gather);
  else
    layernorm_kernel<float><<<grid, 32 * rows_per_cta, 0, st>>>(x, g, b, static_cast<float *>(out), n_rows,
                                                                 H, gather);
  return cudaGetLastError();
}

cudaError_t launch_argmax(const float *logits, int n_rows, int vocab, int32_t *out, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  argmax_kernel<<<n_rows, 512, 0, st>>>(logits, vocab, out);
  return cudaGetLastError();
}

}  // namespace orca
