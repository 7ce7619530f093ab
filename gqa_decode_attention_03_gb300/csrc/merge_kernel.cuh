// merge_kernel.cuh -- log-sum-exp merge of split-KV partials.
//
// One CTA of D / 2 threads per (row t, head h); thread i owns output dims 2i and 2i + 1.  Over
// the first n_valid[t] chunks c (layout
// part[t][c][h][acc(D) | m | l], natural-log m):
//   M = max_c m_c,  e_c = exp(m_c - M),  L = sum_c l_c e_c,  out[d] = sum_c acc_c[d] e_c / L
// as in qsa2.metal's qsa_merge2 (regolith) and FORWARD_MSL's attn_combine (there in exp2 units).
// With a gate, the merged row is multiplied by 1 / (1 + exp(-gate)) on the way out -- the
// sigmoid output gate both pages apply after their merge.
// Every thread reads the chunks' (m, l) itself (the same few lines for all threads of the CTA,
// served by L1), so all its loads are independent and go out together.  A row without valid
// chunks, or with L == 0, gets zeros.
#pragma once

#include "common.cuh"

namespace gqa {

template <int D>
__global__ void __launch_bounds__(D / 2) merge_kernel(const float* __restrict__ part,
                                                      const int32_t* __restrict__ n_valid,
                                                      int n_split, int n_heads,
                                                      const float* __restrict__ gate,
                                                      long long gate_stride,
                                                      float* __restrict__ out) {
  const int h = blockIdx.x, t = blockIdx.y, d = 2 * threadIdx.x;
  int nv = __ldg(n_valid + t);
  nv = nv < 0 ? 0 : (nv > n_split ? n_split : nv);
  const size_t rec = (size_t)n_heads * (D + 2);  // floats between consecutive chunks
  const float* base = part + ((size_t)t * n_split * n_heads + h) * (D + 2);
  float M = -INFINITY;
#pragma unroll 8
  for (int c = 0; c < nv; ++c) M = fmaxf(M, __ldg(base + c * rec + D));  // loads overlap
  float2 a = make_float2(0.f, 0.f);
  float L = 0.f;
  if (M != -INFINITY) {
#pragma unroll 8
    for (int c = 0; c < nv; ++c) {
      const float m = __ldg(base + c * rec + D);
      const float e = m == -INFINITY ? 0.f : __expf(m - M);
      L = fmaf(__ldg(base + c * rec + D + 1), e, L);
      const float2 v = __ldg(reinterpret_cast<const float2*>(base + c * rec + d));
      a.x = fmaf(e, v.x, a.x);
      a.y = fmaf(e, v.y, a.y);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float2 y = make_float2(a.x * inv, a.y * inv);
  if (gate) {  // sigmoid output gate (qsa_merge2, attn_combine)
    const float2 gv =
        __ldg(reinterpret_cast<const float2*>(gate + ((size_t)t * n_heads + h) * gate_stride + d));
    y.x *= 1.f / (1.f + __expf(-gv.x));
    y.y *= 1.f / (1.f + __expf(-gv.y));
  }
  *reinterpret_cast<float2*>(out + ((size_t)t * n_heads + h) * D + d) = y;
}

}  // namespace gqa
