// tq_common.cuh -- pieces shared by the two TurboQuant decode kernels (tq_decode.cu, tq_mma.cu).
//
// flash_attention_tq.metal (cera 0.4.0 sources).  Keys are never reconstructed: a key's score
// is a PolarQuant term, its 2-bit centroid indices dotted with the rotated query, plus a QJL
// correction from its sign bits and residual norm:
//   x_j = (norm_j sum_d q_rot[d] c[kidx_j(d)] + norm_j rn_j qjl_scale sum_d q_jl[d] s_j(d)) scale
// and values are accumulated in the rotated basis, vnorm_j c[vidx_j(d)], so the inverse
// rotation -- 1/sqrt(D), a Walsh-Hadamard transform, the sign flip -- runs once on the merged
// row.  Packed format and layout as on the page: 16 two-bit indices per uint32, index k in bits
// 2k..2k+1; 32 sign bits per uint32; f16 norm pairs; every region head-major, each (sequence,
// KV head) holding its cache_cap positions contiguously.
//
// Both kernels run one CTA of kTqWarps warps per (KV chunk, KV head x head split, query row):
// a group of more than kTqMaxGroup query heads is served by head_split CTAs of at most
// kTqMaxGroup heads each (each decoding the same K/V).  Each warp keeps its own online-softmax
// state for every head of the CTA; at the end the warps' states meet in shared memory (`mg`, [warp][head][D + 2]: rotated accumulator, running max in log2
// units, running sum) and tq_finish combines them, then either normalises, rotates back and
// writes the row, or writes the chunk's rotated partial for the last CTA's merge.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime_api.h>

#include "partial_kernel.cuh"

namespace gqa {

constexpr int kTqWarps = 4;
constexpr int kTqMaxGroup = 8;

struct TqParams {
  PartialParams base;          // q unused; out, part, counters, n_valid, lengths, sizes
  const float* q_rot;          // [T][H][D]
  const float* q_jl;           // [T][H][D]
  const uint32_t* k_polar;     // [n_seq][Hk][cap][D/16]
  const uint32_t* k_jl;        // [n_seq][Hk][cap][D/32]
  const uint32_t* k_norms;     // [n_seq][Hk][cap]
  const uint32_t* v_polar;     // [n_seq][Hk][cap][D/16]
  const uint32_t* v_norms;     // [n_seq][Hk][cap]
  const float* signs;          // [D]
  float c0, c1, c2, c3;        // centroids
  float qjl_scale;
};

// The query heads one CTA serves: KV head g, heads head0 .. head0 + G - 1 of its group, and the
// column of the (row, column) arrival counters its chunks share.
struct TqCta {
  int g, head0, G, col;
};
__device__ __forceinline__ TqCta tq_cta(const PartialParams& p) {
  TqCta a;
  a.g = blockIdx.y / p.head_split;
  a.G = p.group / p.head_split;
  a.head0 = a.g * p.group + (blockIdx.y % p.head_split) * a.G;
  a.col = blockIdx.y;
  return a;
}

__device__ __forceinline__ float half_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// Inverse rotation of a merged rotated row held D/32 consecutive dims per lane (common.cuh's
// rotate_back), as the epilogue of merge_if_last.
template <int D>
struct TqRotateBack {
  const float* signs;
  __device__ __forceinline__ void operator()(float (&a)[D / 32], int /*head*/, int lane) const {
    rotate_back<D>(a, signs, lane);
  }
};

// Row t's length and sequence (out-of-range values flagged and clamped), the chunk's [c0, c1),
// and the row's bookkeeping (n_valid; zeros for an empty context, as the page writes for
// seq_len == 0).  False when this CTA has no positions.
__device__ __forceinline__ bool tq_row_setup(const PartialParams& p, int t, int c, const TqCta& a,
                                             int D, int& L, int& s, int& c0, int& c1) {
  L = __ldg(p.kv_len + t);
  int errbits = 0;
  const int lmax = static_cast<int>(p.cache_cap < p.max_kv_len ? p.cache_cap : p.max_kv_len);
  if (L < 0 || L > lmax) {
    errbits |= GQA_ERR_KVLEN_RANGE;
    L = L < 0 ? 0 : lmax;
  }
  s = p.seq_of ? __ldg(p.seq_of + t) : t;
  if (s < 0 || s >= p.n_seq) {
    errbits |= GQA_ERR_SEQ_RANGE;
    L = 0;
  }
  c0 = c * p.chunk;
  c1 = min(c0 + p.chunk, L);
  if (c == 0 && a.col == 0 && threadIdx.x == 0) {
    if (errbits) flag_error(p.err, errbits);
    if (p.merge) p.n_valid[t] = (L + p.chunk - 1) / p.chunk;
  }
  if (c0 >= L) {
    if (c == 0)
      for (int i = threadIdx.x; i < a.G * D; i += blockDim.x)
        p.out[((size_t)t * p.n_heads + a.head0 + i / D) * D + i % D] = 0.f;
    return false;
  }
  return true;
}

// Combines the warps' states in mg (written, then a __syncthreads, by the caller) and writes
// the row (normalised and rotated back) or this chunk's rotated partial; with a split, the
// last CTA of the (row, KV head) then merges the partials and rotates the merged rows.
template <int D>
__device__ __forceinline__ void tq_finish(const TqParams& tp, const float* mg, int t,
                                          const TqCta& cta, int c, int L) {
  const int G = cta.G;
  constexpr int DPL = D / 32;
  const PartialParams& p = tp.base;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TqRotateBack<D> rot{tp.signs};
  for (int h = warp; h < G; h += kTqWarps) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTqWarps; ++w) M = fmaxf(M, mg[(w * kTqMaxGroup + h) * (D + 2) + D]);
    float a[DPL], Ls = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) a[k] = 0.f;
#pragma unroll
    for (int w = 0; w < kTqWarps; ++w) {
      const float* r = mg + (w * kTqMaxGroup + h) * (D + 2);
      const float e = r[D] == -INFINITY ? 0.f : fast_exp2(r[D] - M);
      Ls = fmaf(r[D + 1], e, Ls);
#pragma unroll
      for (int k = 0; k < DPL; ++k) a[k] = fmaf(r[lane * DPL + k], e, a[k]);
    }
    const int head = cta.head0 + h;
    if (p.merge) {
      float* pr = p.part + (((size_t)t * p.n_split + c) * p.n_heads + head) * (D + 2);
#pragma unroll
      for (int k = 0; k < DPL; ++k) pr[lane * DPL + k] = a[k];
      if (lane == 0) {
        pr[D] = M == -INFINITY ? -INFINITY : M * kLn2;  // natural-log units
        pr[D + 1] = Ls;
      }
    } else {
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
      for (int k = 0; k < DPL; ++k) a[k] *= inv;
      rot(a, head, lane);
      float* o = p.out + ((size_t)t * p.n_heads + head) * D + lane * DPL;
#pragma unroll
      for (int k = 0; k < DPL; ++k) o[k] = gated(p, t, head, lane * DPL + k, a[k]);
    }
  }
  if (p.merge)
    merge_if_last<D>(p, t, cta.head0, G, (size_t)t * gridDim.y + cta.col,
                     (L + p.chunk - 1) / p.chunk, kTqWarps, rot);
}

// Launchers (tq_decode.cu: CUDA cores; tq_mma.cu: tensor cores, nb = ceil(G / 4) n-blocks).
cudaError_t launch_tq_fma(int head_dim, dim3 grid, const TqParams& tp, cudaStream_t stream);
cudaError_t launch_tq_mma(int head_dim, int nb, dim3 grid, const TqParams& tp,
                          cudaStream_t stream);
// tq_rows.cu: rows sharing a sequence (grid.z = group slots), head_dim 64 or 128
cudaError_t launch_tq_rows(int head_dim, dim3 grid, const TqParams& tp, cudaStream_t stream);

}  // namespace gqa
