// append_q8.cu -- quantise-on-append into the int8 cache (FORWARD_MSL, kv_append_q8).
//
// New K and V rows arrive in fp32; each group of GS dims (64, or the page's 32-element blocks)
// of a (position, KV head) row becomes GS int8 codes and one f16 scale in the cache layout the
// int8 decode reads ([n_seq][cap][Hk][D] int8, [n_seq][cap][Hk][D/GS] f16; with n_seq = 1 and
// GS = 32 this is FORWARD_MSL's pair of planes, quants [max_t][row] and scales [max_t][row/32]):
//   d = amax|x| / 127,  q = rint(x / d) clamped to [-127, 127] (0 when d = 0),  scale = f16(d).
// One warp per group, GS/32 elements per lane; K and V groups share one launch.  All arithmetic
// is IEEE fp32 (division rounded to nearest, rint to even), so the codes are a fixed function of
// the inputs.
#include <cuda_fp16.h>
#include <cuda_runtime_api.h>

#include "common.cuh"
#include "gqa_decode.h"

namespace gqa {

void set_last_error(const char* msg);  // host.cu: the text gqa_last_error() returns

template <int GS>
__global__ void __launch_bounds__(256)
    append_q8_kernel(const float* __restrict__ k_new, const float* __restrict__ v_new,
                     int n_new, int hk, int d, int8_t* __restrict__ kq, int8_t* __restrict__ vq,
                     __half* __restrict__ ksc, __half* __restrict__ vsc, long long row0) {
  constexpr int EPL = GS / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const int gpr = d / GS;                                     // groups per (position, head)
  const long long groups = (long long)n_new * hk * gpr;       // per side
  const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= 2 * groups) return;
  const bool is_v = gw >= groups;
  const long long gi = is_v ? gw - groups : gw;  // group index within [n_new][hk][d/GS]
  const float* src = (is_v ? v_new : k_new) + gi * GS + EPL * lane;
  float x[EPL];
  if constexpr (EPL == 2) {
    const float2 v2 = *reinterpret_cast<const float2*>(src);
    x[0] = v2.x;
    x[1] = v2.y;
  } else {
    x[0] = *src;
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float dq = amax / 127.0f;
  signed char c[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const float qv = dq > 0.f ? fminf(fmaxf(rintf(x[e] / dq), -127.f), 127.f) : 0.f;
    c[e] = static_cast<signed char>(static_cast<int>(qv));
  }
  // destination: cache row (row0 + position) x hk + head, group within the row
  const long long per_row = (long long)hk * gpr;
  const long long pos = gi / per_row, rem = gi % per_row;
  const long long head = rem / gpr, grp = rem % gpr;
  const long long crow = (row0 + pos) * hk + head;
  int8_t* dst = (is_v ? vq : kq) + crow * d + grp * GS + EPL * lane;
  if constexpr (EPL == 2) {
    char2 c2;
    c2.x = c[0];
    c2.y = c[1];
    *reinterpret_cast<char2*>(dst) = c2;
  } else {
    *dst = c[0];
  }
  if (lane == 0) (is_v ? vsc : ksc)[crow * gpr + grp] = __float2half_rn(dq);
}

}  // namespace gqa

extern "C" gqa_status kv_append_q8_sg(const float* k_new, const float* v_new, int n_new,
                                      int n_kv_heads, int head_dim, int scale_group, int8_t* kq,
                                      int8_t* vq, uint16_t* ksc, uint16_t* vsc, int n_seq,
                                      int64_t cache_cap, int seq, int t0, cudaStream_t stream) {
  if (scale_group != 32 && scale_group != 64) {
    gqa::set_last_error("kv_append_q8: scale_group must be 32 or 64");
    return GQA_EINVAL;
  }
  if (n_new < 0 || n_kv_heads <= 0 || (head_dim != 64 && head_dim != 128 && head_dim != 256)) {
    gqa::set_last_error("kv_append_q8: n_new >= 0, n_kv_heads >= 1, head_dim in {64, 128, 256}");
    return GQA_EINVAL;
  }
  if (n_new == 0) return GQA_OK;
  if (!k_new || !v_new || !kq || !vq || !ksc || !vsc) {
    gqa::set_last_error("kv_append_q8: a required pointer is NULL");
    return GQA_EINVAL;
  }
  if (((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 7) ||
      ((reinterpret_cast<uintptr_t>(kq) | reinterpret_cast<uintptr_t>(vq) |
        reinterpret_cast<uintptr_t>(ksc) | reinterpret_cast<uintptr_t>(vsc)) & 1)) {
    gqa::set_last_error("kv_append_q8: k_new, v_new 8-byte and the cache 2-byte aligned");
    return GQA_EINVAL;
  }
  if (seq < 0 || seq >= n_seq || t0 < 0 || (int64_t)t0 + n_new > cache_cap) {
    gqa::set_last_error("kv_append_q8: seq outside [0, n_seq) or positions past cache_cap");
    return GQA_EINVAL;
  }
  const long long groups = 2LL * n_new * n_kv_heads * (head_dim / scale_group);
  const long long blocks = (groups + 7) / 8;  // 8 warps per block
  if (blocks > 0x7fffffffLL) {
    gqa::set_last_error("kv_append_q8: too many rows for one launch");
    return GQA_EUNSUPPORTED;
  }
  if (scale_group == 64)
    gqa::append_q8_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(
        k_new, v_new, n_new, n_kv_heads, head_dim, kq, vq, reinterpret_cast<__half*>(ksc),
        reinterpret_cast<__half*>(vsc), (long long)seq * cache_cap + t0);
  else
    gqa::append_q8_kernel<32><<<(unsigned)blocks, 256, 0, stream>>>(
        k_new, v_new, n_new, n_kv_heads, head_dim, kq, vq, reinterpret_cast<__half*>(ksc),
        reinterpret_cast<__half*>(vsc), (long long)seq * cache_cap + t0);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    gqa::set_last_error(cudaGetErrorString(e));
    return GQA_ECUDA;
  }
  return GQA_OK;
}

extern "C" gqa_status kv_append_q8(const float* k_new, const float* v_new, int n_new,
                                   int n_kv_heads, int head_dim, int8_t* kq, int8_t* vq,
                                   uint16_t* ksc, uint16_t* vsc, int n_seq, int64_t cache_cap,
                                   int seq, int t0, cudaStream_t stream) {
  return kv_append_q8_sg(k_new, v_new, n_new, n_kv_heads, head_dim, 64, kq, vq, ksc, vsc, n_seq,
                         cache_cap, seq, t0, stream);
}
