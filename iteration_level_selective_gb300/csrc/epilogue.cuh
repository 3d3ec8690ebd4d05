// GEMM epilogues shared by the SIMT (fp32) and tcgen05 (bf16) GEMMs.
//
// The token-wise Linears of the block (Orca walk-through, Figure 5: QKV
// Linear, Attn Out Linear, the MLP Linears, with GeLU and the residual Add
// fused) all end here: bias add, then the mode's store.  The QKV epilogue
// is the "Split" of Figure 5 for K and V: each row's K/V go straight to the
// request's reserved slot (slot_base + position) of the layer's K/V pool.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "orca_internal.h"

namespace orca {

__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float k0 = 0.7978845608028654f;  // sqrt(2 / pi)
  return 0.5f * x * (1.0f + tanhf(k0 * (x + 0.044715f * x * x * x)));
}

template <typename T> __device__ __forceinline__ T cvt_out(float v);
template <> __device__ __forceinline__ float cvt_out<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Store cnt <= CNT consecutive values: 16-byte stores for every whole 16-byte
// group of the run when dst is 16-byte aligned, element stores for the rest.
template <typename T, int CNT>
__device__ __forceinline__ void store_run(T *dst, const float *v, int cnt) {
  constexpr int PER = 16 / sizeof(T);
  if constexpr ((CNT * sizeof(T)) % 16 == 0) {
    if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < CNT; i += PER) {  // predicated, fully unrolled: v stays in registers
        if (i + PER <= cnt) {
          uint4 pk;
          T *pt = reinterpret_cast<T *>(&pk);
#pragma unroll
          for (int j = 0; j < PER; ++j) pt[j] = cvt_out<T>(v[i + j]);
          *reinterpret_cast<uint4 *>(dst + i) = pk;
        } else {
#pragma unroll
          for (int j = 0; j < PER; ++j)
            if (i + j < cnt) dst[i + j] = cvt_out<T>(v[i + j]);
        }
      }
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < CNT; ++i)
    if (i < cnt) dst[i] = cvt_out<T>(v[i]);
}

// Columns n0 .. n0+cnt-1 of row m; v holds accumulators with the bias
// already added.  CNT must divide head_dim (a run never crosses a head) and
// hidden.
template <typename T, int CNT>
__device__ __forceinline__ void epi_store(const EpiParams &e, int m, int n0, float *v, int cnt) {
  switch (e.mode) {
    case kEpiQKV: {
      const int H = e.hidden;
      const int section = n0 / H;
      const int nn = n0 - section * H;
      T *dst;
      if (section == 0) {
        dst = static_cast<T *>(e.out) + (int64_t)m * e.ldo + nn;
      } else {
        const int slot = e.rows[m].slot;
        if (slot < 0 || slot >= e.n_slots) {
          atomicOr(e.status, kStatusBadIndex);
          return;
        }
        const int head = nn / e.head_dim;
        const int dim = nn - head * e.head_dim;
        T *base = static_cast<T *>(section == 1 ? e.k_layer : e.v_layer);
        dst = base + ((int64_t)head * e.n_slots + slot) * e.head_dim + dim;
      }
      store_run<T, CNT>(dst, v, cnt);
      break;
    }
    case kEpiResid: {
      float *xp = static_cast<float *>(e.out) + (int64_t)m * e.ldo + n0;
      if ((CNT % 4) == 0 && (reinterpret_cast<uintptr_t>(xp) & 15) == 0) {
#pragma unroll
        for (int i = 0; i < CNT; i += 4) {
          if (i + 4 <= cnt) {
            float4 o = *reinterpret_cast<float4 *>(xp + i);
            o.x += v[i]; o.y += v[i + 1]; o.z += v[i + 2]; o.w += v[i + 3];
            *reinterpret_cast<float4 *>(xp + i) = o;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (i + j < cnt) xp[i + j] += v[i + j];
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < CNT; ++i)
          if (i < cnt) xp[i] += v[i];
      }
      break;
    }
    case kEpiGelu: {
#pragma unroll
      for (int i = 0; i < CNT; ++i) v[i] = gelu_tanh_f(v[i]);
      store_run<T, CNT>(static_cast<T *>(e.out) + (int64_t)m * e.ldo + n0, v, cnt);
      break;
    }
    case kEpiStore: {
      store_run<T, CNT>(static_cast<T *>(e.out) + (int64_t)m * e.ldo + n0, v, cnt);
      break;
    }
    default: {  // kEpiLogits (out may be nullptr when only the fused argmax is wanted)
      if (e.out != nullptr) store_run<float, CNT>(static_cast<float *>(e.out) + (int64_t)m * e.ldo + n0, v, cnt);
      break;
    }
  }
}

// Bias (per column) then the epilogue store.
template <typename T, int CNT>
__device__ __forceinline__ void epi_apply(const EpiParams &e, int m, int n0, float *v, int cnt) {
  if (e.bias != nullptr) {
#pragma unroll
    for (int i = 0; i < CNT; ++i)
      if (i < cnt) v[i] += __ldg(e.bias + n0 + i);
  }
  epi_store<T, CNT>(e, m, n0, v, cnt);
}

}  // namespace orca
