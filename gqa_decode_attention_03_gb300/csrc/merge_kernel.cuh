// merge_kernel.cuh -- log-sum-exp merge of split-KV partials.
//
// One warp per (row t, head h), four warps per CTA.  Over the first n_valid[t] chunks c (layout
// part[t][c][h][acc(D) | m | l], natural-log m):
//   M = max_c m_c,  e_c = exp(m_c - M),  L = sum_c l_c e_c,  out[d] = sum_c acc_c[d] e_c / L
// as in qsa2.metal's qsa_merge2 (regolith) and FORWARD_MSL's attn_combine (there in exp2 units).
// Lane c holds chunk c's (m, l) and weight and broadcasts the weight by shuffle, and a lane owns
// D/32 output dims, so a (row, head)'s loads go out in one round per 32 chunks.  A row without
// valid chunks, or with L == 0, gets zeros.
#pragma once

#include "common.cuh"

namespace gqa {

template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const float* __restrict__ part,
                                                    const int32_t* __restrict__ n_valid,
                                                    int n_split, int n_heads,
                                                    float* __restrict__ out) {
  constexpr int DPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 4 + warp, t = blockIdx.y;
  if (h >= n_heads) return;
  int nv = __ldg(n_valid + t);
  nv = nv < 0 ? 0 : (nv > n_split ? n_split : nv);
  const size_t rec = (size_t)n_heads * (D + 2);  // floats between consecutive chunks
  const float* base = part + ((size_t)t * n_split * n_heads + h) * (D + 2);
  float M = -INFINITY;
  for (int c = lane; c < nv; c += 32) M = fmaxf(M, __ldg(base + c * rec + D));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float a[DPL];
#pragma unroll
  for (int k = 0; k < DPL; ++k) a[k] = 0.f;
  float L = 0.f;
  if (M != -INFINITY) {
    for (int c0 = 0; c0 < nv; c0 += 32) {
      float e = 0.f;
      if (c0 + lane < nv) {
        const float m = __ldg(base + (c0 + lane) * rec + D);
        e = m == -INFINITY ? 0.f : __expf(m - M);
        L = fmaf(__ldg(base + (c0 + lane) * rec + D + 1), e, L);
      }
      const int nb = min(32, nv - c0);
#pragma unroll 8
      for (int j = 0; j < nb; ++j) {
        const float ej = __shfl_sync(0xffffffffu, e, j);
        const float* ac = base + (c0 + j) * rec + lane * DPL;
#pragma unroll
        for (int k = 0; k < DPL; k += 2) {
          const float2 v = __ldg(reinterpret_cast<const float2*>(ac + k));
          a[k] = fmaf(ej, v.x, a[k]);
          a[k + 1] = fmaf(ej, v.y, a[k + 1]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float* op = out + ((size_t)t * n_heads + h) * D + lane * DPL;
#pragma unroll
  for (int k = 0; k < DPL; k += 2)
    *reinterpret_cast<float2*>(op + k) = make_float2(a[k] * inv, a[k + 1] * inv);
}

}  // namespace gqa
