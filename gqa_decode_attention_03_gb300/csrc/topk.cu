// topk.cu -- block top-k selection of the int8 path's selected-cell id list.
//
// qsa2.metal (regolith), qsa_topk2: a row's n_kv cells come in blocks of 4 (the last block holds
// n_kv % 4 cells), every cell carries its block's score, and the row keeps the `budget` cells
// with the largest scores, emitted in ascending order; equal scores go to the lower cell.  Rows
// with n_kv <= budget keep every cell.  Scores are compared through an order-preserving fp32 ->
// uint32 key.
//
// One CTA of 1024 threads per row.  The row's block keys are staged in shared memory once when
// the longest row fits kTopkSmemBlocks blocks; otherwise every pass reads them from global
// memory (L2 after the first).  The
// threshold key is found digit by digit, 8 bits per pass
// over 4 passes: a 256-bin shared histogram counts the cells (4 per block, fewer for the tail)
// whose key agrees with the digits fixed so far; a block-wide scan of the bins from the top
// finds the digit at which the running count reaches the number of cells still needed.  The
// emit pass then gives each thread a contiguous range of blocks: blocks above the threshold
// give all their cells, blocks at the threshold give cells in ascending order until the budget
// is met (exclusive scans over the threads place every cell).  Integer work only: the result is
// a deterministic function of the keys.
#include <cuda_runtime_api.h>

#include "common.cuh"
#include "gqa_decode.h"

namespace gqa {

constexpr int kTopkThreads = 1024;
constexpr int kTopkSmemBlocks = 49152;  // 192 KB of staged keys: n_kv up to 196607 cells

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u >> 31) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum of v over the CTA's threads (in thread order); *total gets the sum.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* wsum,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();  // wsum may still be read by the previous scan
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t z = lane < nw ? wsum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    if (lane < nw) wsum[lane] = z;  // inclusive warp totals
  }
  __syncthreads();
  *total = wsum[nw - 1];
  return (x - v) + (warp > 0 ? wsum[warp - 1] : 0u);
}

__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float* __restrict__ scores, long long stride,
                const int32_t* __restrict__ kv_len, int budget, int max_kv_len,
                int smem_blocks, int32_t* __restrict__ ids, int32_t* err) {
  extern __shared__ uint32_t s_key[];  // smem_blocks keys: the row's block keys, when they fit
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[32];
  __shared__ uint32_t s_digit, s_need;
  const int t = blockIdx.x, tid = threadIdx.x;
  int n_kv = __ldg(kv_len + t);
  if (n_kv < 0 || n_kv > max_kv_len) {
    if (tid == 0) flag_error(err, GQA_ERR_KVLEN_RANGE);
    n_kv = n_kv < 0 ? 0 : max_kv_len;
  }
  int32_t* out = ids + (size_t)t * budget;
  if (n_kv <= budget) {  // every cell, then -1 padding
    for (int c = tid; c < budget; c += kTopkThreads) out[c] = c < n_kv ? c : -1;
    return;
  }
  const float* row = scores + (size_t)t * stride;
  const int nfull = n_kv >> 2, nb = nfull + 1, tail = n_kv & 3;
  const bool staged = nb <= smem_blocks;
  if (staged) {
    for (int b = tid; b < nb; b += kTopkThreads) s_key[b] = order_key(__ldg(row + b));
    __syncthreads();
  }
  auto key = [&](int b) { return staged ? s_key[b] : order_key(__ldg(row + b)); };

  uint32_t prefix = 0, pmask = 0, need = (uint32_t)budget;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) hist[tid] = 0u;
    __syncthreads();
    for (int b = tid; b < nb; b += kTopkThreads) {
      const uint32_t k = key(b);
      const uint32_t w = b < nfull ? 4u : (uint32_t)tail;
      if (w && (k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], w);
    }
    __syncthreads();
    // thread i < 256 holds bin 255 - i: the scan gives the cells in strictly higher bins
    const uint32_t cnt = tid < 256 ? hist[255 - tid] : 0u;
    uint32_t total;
    const uint32_t above = block_exclusive_scan(cnt, wsum, &total);
    if (tid < 256 && above < need && above + cnt >= need) {
      s_digit = 255u - tid;
      s_need = need - above;
    }
    __syncthreads();
    prefix |= s_digit << shift;
    pmask |= 255u << shift;
    need = s_need;
  }
  const uint32_t T = prefix;  // the threshold key; `need` cells at T are still wanted

  // emit: thread tid owns blocks [b0, b1), ascending with tid
  const int per = (nb + kTopkThreads - 1) / kTopkThreads;
  const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
  uint32_t gt = 0, eq = 0;
  for (int b = b0; b < b1; ++b) {
    const uint32_t k = key(b);
    const uint32_t w = b < nfull ? 4u : (uint32_t)tail;
    if (k > T) gt += w;
    else if (k == T) eq += w;
  }
  uint32_t total;
  const uint32_t eq_before = block_exclusive_scan(eq, wsum, &total);
  const uint32_t eq_take = eq_before >= need ? 0u : min(eq, need - eq_before);
  uint32_t off = block_exclusive_scan(gt + eq_take, wsum, &total);
  uint32_t left = eq_take;
  for (int b = b0; b < b1; ++b) {
    const uint32_t k = key(b);
    const uint32_t w = b < nfull ? 4u : (uint32_t)tail;
    uint32_t take = 0;
    if (k > T) {
      take = w;
    } else if (k == T) {
      take = min(w, left);
      left -= take;
    }
    for (uint32_t c = 0; c < take; ++c) out[off + c] = 4 * b + (int)c;
    off += take;
  }
}

}  // namespace gqa

namespace gqa {
void set_last_error(const char* msg);          // host.cu: the text gqa_last_error() returns
cudaError_t ensure_smem(const void* fn, int bytes);  // launch_util.cu: the opt-in, once
}

static gqa_status topk_fail(gqa_status s, const char* msg) {
  gqa::set_last_error(msg);
  return s;
}

extern "C" gqa_status attn_select_topk(const float* block_scores, int64_t score_stride,
                                       const int32_t* kv_len, int n_tok, int max_kv_len,
                                       int budget, int32_t* ids, int32_t* err_word,
                                       cudaStream_t stream) {
  if (n_tok < 0 || budget <= 0 || max_kv_len < 0)
    return topk_fail(GQA_EINVAL, "attn_select_topk: needs n_tok >= 0, budget >= 1, max_kv_len >= 0");
  if (n_tok == 0) return GQA_OK;
  if (!block_scores || !kv_len || !ids)
    return topk_fail(GQA_EINVAL, "attn_select_topk: a required pointer is NULL");
  if (score_stride < (int64_t)max_kv_len / 4 + 1)
    return topk_fail(GQA_EINVAL, "attn_select_topk: score_stride < max_kv_len / 4 + 1");
  // the staged keys: room for the longest row's blocks if they fit, else none (a row stages
  // only when its own block count fits the room launched)
  const int nb_max = max_kv_len / 4 + 1;
  const int smem_blocks = nb_max <= gqa::kTopkSmemBlocks ? nb_max : 0;
  if (smem_blocks > 0) {  // the opt-in past 48 KB (static + dynamic), once, at the largest size
    const cudaError_t e = gqa::ensure_smem(reinterpret_cast<const void*>(gqa::topk_kernel),
                                           gqa::kTopkSmemBlocks * sizeof(uint32_t));
    if (e != cudaSuccess) return topk_fail(GQA_ECUDA, cudaGetErrorString(e));
  }
  gqa::topk_kernel<<<n_tok, gqa::kTopkThreads, (size_t)smem_blocks * sizeof(uint32_t), stream>>>(
      block_scores, (long long)score_stride, kv_len, budget, max_kv_len, smem_blocks, ids,
      err_word);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return topk_fail(GQA_ECUDA, cudaGetErrorString(e));
  return GQA_OK;
}
