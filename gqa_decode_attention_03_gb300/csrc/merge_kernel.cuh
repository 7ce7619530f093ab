// merge_kernel.cuh -- log-sum-exp merge of split-KV partials.
//
// One CTA of D threads per (head h, row t); thread d owns output dim d.  Over the first n_valid[t]
// chunks c (layout part[t][c][h][acc(D) | m | l], natural-log m):
//   M = max_c m_c,  e_c = exp(m_c - M),  L = sum_c l_c e_c,  out[d] = sum_c acc_c[d] e_c / L
// as in qsa2.metal's qsa_merge2 (regolith) and FORWARD_MSL's attn_combine (there in exp2 units).
// A row without valid chunks, or with L == 0, gets zeros.
#pragma once

#include "common.cuh"

namespace gqa {

__device__ __forceinline__ float block_allreduce(float v, bool is_max, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  __syncthreads();  // red may still be read by a previous call
  if (lane == 0) red[w] = v;
  __syncthreads();
  v = red[0];
  for (int i = 1; i < nw; ++i) v = is_max ? fmaxf(v, red[i]) : v + red[i];
  return v;
}

template <int D>
__global__ void __launch_bounds__(D) merge_kernel(const float* __restrict__ part,
                                                  const int32_t* __restrict__ n_valid, int n_split,
                                                  int n_heads, float* __restrict__ out) {
  constexpr int EB = 256;  // chunk weights staged per round
  __shared__ float red[32];
  __shared__ float e_s[EB];
  const int h = blockIdx.x, t = blockIdx.y, d = threadIdx.x;
  int nv = __ldg(n_valid + t);
  nv = nv < 0 ? 0 : (nv > n_split ? n_split : nv);
  float* o = out + ((size_t)t * n_heads + h) * D;
  if (nv == 0) {
    o[d] = 0.f;
    return;
  }
  const size_t stride = (size_t)n_heads * (D + 2);
  const float* base = part + ((size_t)t * n_split * n_heads + h) * (D + 2);

  float m = -INFINITY;
  for (int c = d; c < nv; c += D) m = fmaxf(m, __ldg(base + c * stride + D));
  const float M = block_allreduce(m, true, red);
  if (M == -INFINITY) {
    o[d] = 0.f;
    return;
  }
  float l = 0.f;
  for (int c = d; c < nv; c += D) {
    const float mc = __ldg(base + c * stride + D);
    if (mc != -INFINITY) l = fmaf(__ldg(base + c * stride + D + 1), __expf(mc - M), l);
  }
  const float L = block_allreduce(l, false, red);

  float a = 0.f;
  for (int c0 = 0; c0 < nv; c0 += EB) {
    const int n = min(EB, nv - c0);
    __syncthreads();
    for (int i = d; i < n; i += D) {
      const float mc = __ldg(base + (c0 + i) * stride + D);
      e_s[i] = mc == -INFINITY ? 0.f : __expf(mc - M);
    }
    __syncthreads();
    const float* pc = base + (size_t)c0 * stride + d;
#pragma unroll 4
    for (int i = 0; i < n; ++i) a = fmaf(__ldg(pc + i * stride), e_s[i], a);
  }
  o[d] = L > 0.f ? a / L : 0.f;
}

}  // namespace gqa
