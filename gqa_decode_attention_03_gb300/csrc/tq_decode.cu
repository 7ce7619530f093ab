// tq_decode.cu -- TurboQuant decode on the CUDA cores, and the attn_decode_tq entry point.
//
// flash_attention_tq.metal (cera 0.4.0 sources); the score and accumulator definitions are in
// tq_common.cuh.  This kernel gives each lane one cache position for q.k (its 2-bit fields and
// sign bits decoded once, dotted with every head's rotated query, broadcast from shared memory)
// and D/32 dims of the rotated accumulator for p.v.  It is the plain form of the path, kept
// beside the tensor-core kernel (tq_mma.cu, the default) as a cross-check: GQA_TQ_KERNEL=fma
// selects it.
#include <cuda_fp16.h>
#include <cuda_runtime_api.h>

#include <cmath>
#include <cstdlib>
#include <cstring>

#include "dispatch.h"
#include "tq_common.cuh"

namespace gqa {

void set_last_error(const char* msg);

__device__ __forceinline__ float tq_centroid(uint32_t idx, float c0, float c1, float c2, float c3) {
  return (idx & 2u) ? ((idx & 1u) ? c3 : c2) : ((idx & 1u) ? c1 : c0);
}

template <int D>
__global__ void __launch_bounds__(32 * kTqWarps) tq_decode_kernel(const TqParams tp) {
  constexpr int DPL = D / 32, PW = D / 16, JW = D / 32;
  const PartialParams& p = tp.base;
  __shared__ __align__(16) float qr[kTqMaxGroup][D];
  __shared__ __align__(16) float qj[kTqMaxGroup][D];
  __shared__ float qjsum[kTqMaxGroup];
  __shared__ uint32_t vbuf[kTqWarps][32][PW];
  __shared__ float mg[kTqWarps * kTqMaxGroup * (D + 2)];
  const int c = blockIdx.x, t = blockIdx.z;
  const TqCta cta = tq_cta(p);
  const int g = cta.g, G = cta.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int L, s, c0, c1;
  if (!tq_row_setup(p, t, c, cta, D, L, s, c0, c1)) return;

  // the CTA's rotated and JL queries, and the per-head sum of q_jl
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const size_t qi = ((size_t)t * p.n_heads + cta.head0) * D + i;
    qr[i / D][i % D] = __ldg(tp.q_rot + qi);
    qj[i / D][i % D] = __ldg(tp.q_jl + qi);
  }
  __syncthreads();
  for (int h = warp; h < G; h += kTqWarps) {
    float x = 0.f;
    for (int d = lane; d < D; d += 32) x += qj[h][d];
    x = warp_sum(x);
    if (lane == 0) qjsum[h] = x;
  }
  __syncthreads();

  const float kx = p.scale_log2;  // scores in log2 units
  float m_run[kTqMaxGroup], l_run[kTqMaxGroup], acc[kTqMaxGroup][DPL];
#pragma unroll
  for (int h = 0; h < kTqMaxGroup; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[h][k] = 0.f;
  }

  for (int base = c0 + warp * 32; base < c1; base += kTqWarps * 32) {
    const int pos = base + lane;
    const bool valid = pos < c1;
    const int nvb = min(32, c1 - base);  // valid positions of the block, a prefix
    const size_t row = ((size_t)s * p.n_kv_heads + g) * p.cache_cap + (valid ? pos : c0);
    float x[kTqMaxGroup];
    float vn = 0.f;
    {
      uint32_t kp[PW], kj[JW], vp[PW];
      if constexpr (PW >= 4) {  // a row's polar words: 16-byte loads (8 bytes at D = 32)
#pragma unroll
        for (int w = 0; w < PW; w += 4) {
          const uint4 u = __ldg(reinterpret_cast<const uint4*>(tp.k_polar + row * PW + w));
          kp[w] = u.x; kp[w + 1] = u.y; kp[w + 2] = u.z; kp[w + 3] = u.w;
          const uint4 v4 = __ldg(reinterpret_cast<const uint4*>(tp.v_polar + row * PW + w));
          vp[w] = v4.x; vp[w + 1] = v4.y; vp[w + 2] = v4.z; vp[w + 3] = v4.w;
        }
      } else {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(tp.k_polar + row * PW));
        kp[0] = u.x; kp[1] = u.y;
        const uint2 v2 = __ldg(reinterpret_cast<const uint2*>(tp.v_polar + row * PW));
        vp[0] = v2.x; vp[1] = v2.y;
      }
      if constexpr (JW >= 2) {  // sign words: 8-byte loads (4 bytes at D = 32)
#pragma unroll
        for (int w = 0; w < JW; w += 2) {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(tp.k_jl + row * JW + w));
          kj[w] = u.x; kj[w + 1] = u.y;
        }
      } else {
        kj[0] = __ldg(tp.k_jl + row);
      }
      const uint32_t kn = __ldg(tp.k_norms + row);
      vn = half_lo(__ldg(tp.v_norms + row));
#pragma unroll
      for (int w = 0; w < PW; ++w) vbuf[warp][lane][w] = vp[w];
      float polar[kTqMaxGroup], pos_sum[kTqMaxGroup];
#pragma unroll
      for (int h = 0; h < kTqMaxGroup; ++h) polar[h] = pos_sum[h] = 0.f;
#pragma unroll
      for (int w = 0; w < PW; ++w) {
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
          float cv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            cv[e] = tq_centroid((kp[w] >> (2 * (k4 + e))) & 3u, tp.c0, tp.c1, tp.c2, tp.c3);
#pragma unroll
          for (int h = 0; h < kTqMaxGroup; ++h) {
            if (h >= G) break;
            const float4 q4 = *reinterpret_cast<const float4*>(&qr[h][w * 16 + k4]);
            polar[h] = fmaf(q4.x, cv[0], fmaf(q4.y, cv[1], fmaf(q4.z, cv[2], fmaf(q4.w, cv[3], polar[h]))));
          }
        }
      }
#pragma unroll
      for (int w = 0; w < JW; ++w) {
#pragma unroll
        for (int k4 = 0; k4 < 32; k4 += 4) {
          float b[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) b[e] = static_cast<float>((kj[w] >> (k4 + e)) & 1u);
#pragma unroll
          for (int h = 0; h < kTqMaxGroup; ++h) {
            if (h >= G) break;
            const float4 q4 = *reinterpret_cast<const float4*>(&qj[h][w * 32 + k4]);
            pos_sum[h] = fmaf(q4.x, b[0], fmaf(q4.y, b[1], fmaf(q4.z, b[2], fmaf(q4.w, b[3], pos_sum[h]))));
          }
        }
      }
      const float norm = half_lo(kn), rn = half_hi(kn);
#pragma unroll
      for (int h = 0; h < kTqMaxGroup; ++h) {
        const float signed_sum = 2.f * pos_sum[h] - qjsum[h < G ? h : 0];
        const float sc = (norm * polar[h] + norm * rn * tp.qjl_scale * signed_sum) * kx;
        x[h] = (valid && h < G) ? sc : -INFINITY;  // masked by selection: no NaN gets through
      }
    }
    __syncwarp();
    // online softmax per head over the block (every block holds at least one valid position)
    float pr[kTqMaxGroup];
#pragma unroll
    for (int h = 0; h < kTqMaxGroup; ++h) {
      if (h >= G) break;
      const float m_new = fmaxf(m_run[h], warp_max(x[h]));
      const float corr = fast_exp2(m_run[h] - m_new);  // first block: exp2(-inf) = 0
      pr[h] = fast_exp2(x[h] - m_new);
      l_run[h] = fmaf(l_run[h], corr, warp_sum(pr[h]));
      m_run[h] = m_new;
#pragma unroll
      for (int k = 0; k < DPL; ++k) acc[h][k] *= corr;
    }
    // p.v in the rotated basis: this lane's dims lane*DPL .. + DPL-1
    const int vw = (lane * DPL) / 16, vsh = 2 * ((lane * DPL) % 16);
    for (int j = 0; j < nvb; ++j) {
      const uint32_t word = vbuf[warp][j][vw] >> vsh;
      const float vnj = __shfl_sync(0xffffffffu, vn, j);
      float cv[DPL];
#pragma unroll
      for (int k = 0; k < DPL; ++k)
        cv[k] = vnj * tq_centroid((word >> (2 * k)) & 3u, tp.c0, tp.c1, tp.c2, tp.c3);
#pragma unroll
      for (int h = 0; h < kTqMaxGroup; ++h) {
        if (h >= G) break;
        const float ph = __shfl_sync(0xffffffffu, pr[h], j);
#pragma unroll
        for (int k = 0; k < DPL; ++k) acc[h][k] = fmaf(ph, cv[k], acc[h][k]);
      }
    }
    __syncwarp();
  }

  // ---- the warps' states to shared memory; tq_finish combines them
#pragma unroll
  for (int h = 0; h < kTqMaxGroup; ++h) {
    if (h >= G) break;
    float* r = mg + (warp * kTqMaxGroup + h) * (D + 2);
#pragma unroll
    for (int k = 0; k < DPL; ++k) r[lane * DPL + k] = acc[h][k];
    if (lane == 0) {
      r[D] = m_run[h];
      r[D + 1] = l_run[h];
    }
  }
  __syncthreads();
  tq_finish<D>(tp, mg, t, cta, c, L);
}

cudaError_t launch_tq_fma(int head_dim, dim3 grid, const TqParams& tp, cudaStream_t stream) {
  if (head_dim == 32)
    tq_decode_kernel<32><<<grid, 32 * kTqWarps, 0, stream>>>(tp);
  else if (head_dim == 64)
    tq_decode_kernel<64><<<grid, 32 * kTqWarps, 0, stream>>>(tp);
  else
    tq_decode_kernel<128><<<grid, 32 * kTqWarps, 0, stream>>>(tp);
  return cudaGetLastError();
}

}  // namespace gqa

// ------------------------------------------------------------------------------ C ABI

static gqa_status tq_fail(gqa_status st, const char* msg) {
  gqa::set_last_error(msg);
  return st;
}

static bool tq_aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

static gqa_status tq_entry(const float* q_rot, const float* q_jl, const uint32_t* k_polar,
                           const uint32_t* k_jl, const uint32_t* k_norms, const uint32_t* v_polar,
                           const uint32_t* v_norms, const float* centroids, const float* signs,
                           float qjl_scale, float scale, float* out, const int32_t* kv_len,
                           const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                           int n_kv_heads, int head_dim, int64_t cache_cap, int max_kv_len,
                           void* ws, size_t ws_bytes, int32_t* err_word, cudaStream_t stream,
                           const float* gate, int64_t gate_stride) {
  if (gate && (gate_stride < head_dim || (reinterpret_cast<uintptr_t>(gate) & 3)))
    return tq_fail(GQA_EINVAL, "attn_decode_tq: gate 4-byte aligned, gate_stride >= head_dim");
  if (head_dim != 32 && head_dim != 64 && head_dim != 128)
    return tq_fail(GQA_EINVAL, "attn_decode_tq: head_dim must be 32, 64 or 128");
  if (n_kv_heads <= 0 || n_heads % n_kv_heads)
    return tq_fail(GQA_EINVAL, "attn_decode_tq: n_heads must be a positive multiple of n_kv_heads");
  if (n_heads / n_kv_heads > 16)
    return tq_fail(GQA_EUNSUPPORTED, "attn_decode_tq: group size above 16");
  if (n_tok < 0 || n_tok > 65535) return tq_fail(GQA_EINVAL, "attn_decode_tq: n_tok outside [0, 65535]");
  if (n_tok == 0) return GQA_OK;
  if (!q_rot || !q_jl || !k_polar || !k_jl || !k_norms || !v_polar || !v_norms || !centroids ||
      !signs || !out || !kv_len)
    return tq_fail(GQA_EINVAL, "attn_decode_tq: a required pointer is NULL");
  if (!tq_aligned16(k_polar) || !tq_aligned16(v_polar) || !tq_aligned16(k_jl) ||
      !tq_aligned16(k_norms) || !tq_aligned16(v_norms) || (reinterpret_cast<uintptr_t>(out) & 7))
    return tq_fail(GQA_EINVAL, "attn_decode_tq: packed caches 16-byte, out 8-byte aligned");
  if (n_seq <= 0 || cache_cap <= 0 || max_kv_len < 0)
    return tq_fail(GQA_EINVAL, "attn_decode_tq: n_seq, cache_cap > 0, max_kv_len >= 0");
  if (!seq_of && n_seq < n_tok) return tq_fail(GQA_EINVAL, "seq_of NULL needs n_seq >= n_tok");
  if (!std::isfinite(scale) || !std::isfinite(qjl_scale))
    return tq_fail(GQA_EINVAL, "attn_decode_tq: scale and qjl_scale must be finite");
  const int max_len = (int)(max_kv_len < cache_cap ? max_kv_len : cache_cap);
  gqa_plan plan;
  gqa_status st = attn_decode_plan(n_tok, n_seq, n_heads, n_kv_heads, head_dim, max_len, -1,
                                   GQA_KIND_TQ, 0, &plan);
  if (st != GQA_OK) return st;
  if (plan.merge && (!ws || ws_bytes < plan.ws_bytes || !tq_aligned16(ws)))
    return tq_fail(GQA_EWORKSPACE, "attn_decode_tq: workspace too small or misaligned");

  gqa::TqParams tp{};
  gqa::PartialParams& p = tp.base;
  p.out = out;
  p.kv_len = kv_len;
  p.seq_of = seq_of;
  p.err = err_word;
  p.n_tok = n_tok;
  p.n_seq = n_seq;
  p.n_heads = n_heads;
  p.n_kv_heads = n_kv_heads;
  p.group = n_heads / n_kv_heads;
  p.head_split = plan.grid_y / n_kv_heads;  // CTAs per KV head, kTqMaxGroup heads each at most
  p.cache_cap = cache_cap;
  p.max_kv_len = max_len;
  p.budget = INT32_MAX;
  p.chunk = plan.chunk;
  p.n_split = plan.n_split;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.merge = plan.merge;
  p.gate = gate;
  p.gate_stride = gate ? gate_stride : 0;
  {  // the tensor-core kernel goes out as a programmatic dependent; GQA_PDL=0 launches it plainly
    const char* pd = std::getenv("GQA_PDL");
    p.pdl = !(pd && std::strcmp(pd, "0") == 0);
  }
  if (plan.merge) {
    const size_t cnt = ((size_t)n_tok * plan.grid_y * sizeof(uint32_t) + 255) / 256 * 256;
    const size_t part = (size_t)n_tok * plan.n_split * n_heads * (head_dim + 2) * sizeof(float);
    p.counters = static_cast<unsigned int*>(ws);
    p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + cnt);
    p.n_valid =
        reinterpret_cast<int32_t*>(static_cast<char*>(ws) + cnt + (part + 255) / 256 * 256);
  }
  tp.q_rot = q_rot;
  tp.q_jl = q_jl;
  tp.k_polar = k_polar;
  tp.k_jl = k_jl;
  tp.k_norms = k_norms;
  tp.v_polar = v_polar;
  tp.v_norms = v_norms;
  tp.signs = signs;
  tp.c0 = centroids[0];
  tp.c1 = centroids[1];
  tp.c2 = centroids[2];
  tp.c3 = centroids[3];
  tp.qjl_scale = qjl_scale;
  const dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
  const char* kern = std::getenv("GQA_TQ_KERNEL");  // "fma": the CUDA-core kernel
  const int G = n_heads / n_kv_heads;
  // head_dim 32 runs on the CUDA cores: a 32-dim polar row is 8 bytes, below the tensor-core
  // kernel's 16-byte staging pieces
  const int nb = G / p.head_split <= 4 ? 1 : 2;  // n-blocks of 4 heads per CTA
  if (plan.row_group > 1 && plan.merge) {
    // rows sharing a sequence: their chunk CTAs merge the group's partials themselves when the
    // whole grid fits one CTA per SM (a cooperative launch); otherwise merge_kernel follows
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
      const long long ctas = (long long)plan.grid_x * plan.grid_y * plan.grid_z;
      tp.base.fused_merge = ctas <= sms ? 1 : 0;
    }
    (void)cudaGetLastError();
    // polls of the fused merge's wait before it gives up; GQA_MERGE_SPIN (tests) sets fewer
    const char* spin = std::getenv("GQA_MERGE_SPIN");
    tp.base.merge_spin = spin ? (unsigned)std::strtoul(spin, nullptr, 10) : gqa::kSpinLimit;
  }
  if (plan.row_group > 1) {  // rows sharing a sequence: one decoded tile for up to 64 pairs
    cudaError_t el = gqa::launch_tq_rows(head_dim, grid, tp, stream);
    if (el == cudaErrorCooperativeLaunchTooLarge && tp.base.fused_merge) {  // not all resident
      (void)cudaGetLastError();
      tp.base.fused_merge = 0;
      (void)gqa::launch_tq_rows(head_dim, grid, tp, stream);
    }
  }
  else if (head_dim == 32 || (kern && std::strcmp(kern, "fma") == 0))
    (void)gqa::launch_tq_fma(head_dim, grid, tp, stream);
  else
    (void)gqa::launch_tq_mma(head_dim, nb, grid, tp, stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return tq_fail(GQA_ECUDA, cudaGetErrorString(e));
  if (plan.row_group > 1 && plan.merge && !tp.base.fused_merge) {  // merged, rotated back
    e = gqa::launch_merge(head_dim, p.part, p.n_valid, plan.n_split, n_tok, n_heads, out, stream,
                          gate, gate ? gate_stride : 0, /*after_partials=*/true, signs);
    if (e != cudaSuccess) return tq_fail(GQA_ECUDA, cudaGetErrorString(e));
  }
  return GQA_OK;
}

extern "C" gqa_status attn_decode_tq(const float* q_rot, const float* q_jl,
                                     const uint32_t* k_polar, const uint32_t* k_jl,
                                     const uint32_t* k_norms, const uint32_t* v_polar,
                                     const uint32_t* v_norms, const float* centroids,
                                     const float* signs, float qjl_scale, float scale, float* out,
                                     const int32_t* kv_len, const int32_t* seq_of, int n_tok,
                                     int n_seq, int n_heads, int n_kv_heads, int head_dim,
                                     int64_t cache_cap, int max_kv_len, void* ws, size_t ws_bytes,
                                     int32_t* err_word, cudaStream_t stream) {
  return tq_entry(q_rot, q_jl, k_polar, k_jl, k_norms, v_polar, v_norms, centroids, signs,
                  qjl_scale, scale, out, kv_len, seq_of, n_tok, n_seq, n_heads, n_kv_heads,
                  head_dim, cache_cap, max_kv_len, ws, ws_bytes, err_word, stream, nullptr, 0);
}

extern "C" gqa_status attn_decode_tq_gated(
    const float* q_rot, const float* q_jl, const uint32_t* k_polar, const uint32_t* k_jl,
    const uint32_t* k_norms, const uint32_t* v_polar, const uint32_t* v_norms,
    const float* centroids, const float* signs, float qjl_scale, float scale, float* out,
    const int32_t* kv_len, const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
    int n_kv_heads, int head_dim, int64_t cache_cap, int max_kv_len, const float* gate,
    int64_t gate_stride, void* ws, size_t ws_bytes, int32_t* err_word, cudaStream_t stream) {
  if (!gate) return tq_fail(GQA_EINVAL, "attn_decode_tq_gated: gate is NULL");
  return tq_entry(q_rot, q_jl, k_polar, k_jl, k_norms, v_polar, v_norms, centroids, signs,
                  qjl_scale, scale, out, kv_len, seq_of, n_tok, n_seq, n_heads, n_kv_heads,
                  head_dim, cache_cap, max_kv_len, ws, ws_bytes, err_word, stream, gate,
                  gate_stride);
}
