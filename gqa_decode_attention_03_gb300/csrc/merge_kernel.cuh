// merge_kernel.cuh -- log-sum-exp merge of split-KV partials.
//
// One warp per (row t, head h), four per CTA.  Over the first n_valid[t] chunks c (layout
// part[t][c][h][acc(D) | m | l], natural-log m):
//   M = max_c m_c,  e_c = exp(m_c - M),  L = sum_c l_c e_c,  out[d] = sum_c acc_c[d] e_c / L
// as in qsa2.metal's qsa_merge2 (regolith) and FORWARD_MSL's attn_combine (there in exp2 units).
// With a gate, the merged row is multiplied by 1 / (1 + exp(-gate)) on the way out -- the
// sigmoid output gate both pages apply after their merge.  With `signs` (TurboQuant partials,
// accumulated in the rotated basis) the merged row is rotated back first (rotate_back).
// Lanes take the chunks 32 at a time: lane c reads (m_c, l_c), a warp max gives the batch's
// maximum, and each lane then folds every chunk of the batch into its own D/32 output dims with
// the chunk's weight broadcast by shuffle; the accumulator loads do not depend on the weights,
// so a batch's loads go out together.  More than 32 chunks are folded batch by batch with the
// running maximum rescaling what came before.  A row without valid chunks, or with L == 0, gets
// zeros.
#pragma once

#include "common.cuh"

namespace gqa {

constexpr int kMergeWarps = 4;

// A lane's D/32 consecutive accumulator values of one partial.  Records are D + 2 floats long,
// so they are 8-byte but not 16-byte aligned: float2 loads.
template <int DPL>
__device__ __forceinline__ void merge_load(const float* p, float (&v)[DPL]) {
#pragma unroll
  for (int k = 0; k < DPL; k += 2) {
    const float2 x = __ldg(reinterpret_cast<const float2*>(p + k));
    v[k] = x.x;
    v[k + 1] = x.y;
  }
}

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps)
    merge_kernel(const float* __restrict__ part, const int32_t* __restrict__ n_valid, int n_split,
                 int n_tok, int n_heads, const float* __restrict__ gate, long long gate_stride,
                 const float* __restrict__ signs, float* __restrict__ out) {
  constexpr int DPL = D / 32;  // output dims per lane
  // launched as a programmatic dependent of the partials' kernel: wait for that grid's
  // completion and memory (a no-op after an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long pair = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (pair >= (long long)n_tok * n_heads) return;
  const int t = static_cast<int>(pair / n_heads), h = static_cast<int>(pair % n_heads);
  int nv = __ldg(n_valid + t);
  nv = nv < 0 ? 0 : (nv > n_split ? n_split : nv);
  const size_t rec = (size_t)n_heads * (D + 2);  // floats between consecutive chunks
  const float* base = part + ((size_t)t * n_split * n_heads + h) * (D + 2);
  float a[DPL];
#pragma unroll
  for (int k = 0; k < DPL; ++k) a[k] = 0.f;
  float M = -INFINITY, L = 0.f;  // L: this lane's share of the sum, reduced at the end
  for (int c0 = 0; c0 < nv; c0 += 32) {
    const int nb = min(32, nv - c0);
    float m = -INFINITY, l = 0.f;
    if (lane < nb) {
      m = __ldg(base + (c0 + lane) * rec + D);
      l = __ldg(base + (c0 + lane) * rec + D + 1);
    }
    float mb = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const float M_new = fmaxf(M, mb);
    if (M_new == -INFINITY) continue;  // every chunk so far empty
    const float corr = M == -INFINITY ? 0.f : __expf(M - M_new);
    M = M_new;
    L *= corr;
#pragma unroll
    for (int k = 0; k < DPL; ++k) a[k] *= corr;
    const float e = m == -INFINITY ? 0.f : __expf(m - M);
    L = fmaf(l, e, L);
    const float* ac = base + c0 * rec + lane * DPL;
#pragma unroll 8
    for (int j = 0; j < nb; ++j) {
      float v[DPL];
      merge_load<DPL>(ac + j * rec, v);
      const float ej = __shfl_sync(0xffffffffu, e, j);
#pragma unroll
      for (int k = 0; k < DPL; ++k) a[k] = fmaf(ej, v[k], a[k]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int k = 0; k < DPL; ++k) a[k] *= inv;
  if (signs) rotate_back<D>(a, signs, lane);  // warp-uniform
  float* orow = out + ((size_t)t * n_heads + h) * D + lane * DPL;
  const float* grow = gate ? gate + ((size_t)t * n_heads + h) * gate_stride + lane * DPL : nullptr;
#pragma unroll
  for (int k = 0; k < DPL; ++k) {
    float y = a[k];
    if (grow) y *= 1.f / (1.f + __expf(-__ldg(grow + k)));  // sigmoid output gate
    orow[k] = y;
  }
}

}  // namespace gqa
