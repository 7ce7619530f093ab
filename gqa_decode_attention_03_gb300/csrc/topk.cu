// topk.cu -- the selected-cell id list of the int8 path: block top-k selection.
//
// What is selected (qsa2.metal, regolith, qsa_topk2): row t's n = kv_len[t] cells come in blocks
// of 4 (block b holds cells 4b .. 4b + 3; the last block holds n % 4 cells when that is not 0)
// and every cell carries its block's score.  The row keeps the `budget` cells with the largest
// scores, equal scores going to the lower cell, and lists them in ascending order.  A row with
// n <= budget keeps every cell.  Scores are ranked through the order-preserving map of fp32 bit
// patterns to uint32 (the page's `okey`, which it leaves undefined).
//
// How it is found here -- one CTA of kSelThreads threads per row:
//   1. The threshold.  Let ge(c) be the number of cells whose key is >= c.  The threshold T is
//      the largest key value with ge(T) >= budget, i.e. the key of the budget-th cell in
//      descending order.  It is found by a binary search on the 32-bit key value, one bit per
//      step from the most significant: each step counts ge(candidate) over the row with one
//      CTA-wide sum (a warp reduction, one barrier).  One more count gives ge(T + 1), the cells
//      strictly above T; the remaining need = budget - ge(T + 1) cells come from blocks whose
//      key equals T, lowest cells first.
//   2. The list.  Blocks are visited in ascending order, kSelThreads of them per round (block
//      r * kSelThreads + tid in round r).  A CTA-wide exclusive scan of the cells at key T gives
//      each block the number of such cells before it, hence how many of its own it takes; a
//      second scan of the taken cells gives each block its place in the output.  Both running
//      totals carry over to the next round.
// The row's block keys are staged in shared memory when its block count fits the room the
// launch reserved; otherwise each step reads them from global memory (L2 after the first).
// Integer work only: the list is a deterministic function of the keys.
#include <cuda_runtime_api.h>

#include "common.cuh"
#include "gqa_decode.h"

namespace gqa {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelStageBlocks = 53248;  // 208 KB of staged keys: rows of up to 212,991 cells

// fp32 bit pattern -> uint32 whose unsigned order is the float order (-0 below +0; NaNs at the
// ends): negative values have every bit flipped, the others get the sign bit set.
__device__ __forceinline__ uint32_t monotone_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u ^ 0x80000000u);
}

// The CTA-wide sum of v, returned to every thread.  One barrier; `slot` (kSelWarps words) must
// not be the slot of the previous CTA-wide call (callers alternate two).
__device__ __forceinline__ uint32_t cta_sum(uint32_t v, uint32_t* slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  if (lane == 0) slot[warp] = v;
  __syncthreads();
  return __reduce_add_sync(0xffffffffu, lane < kSelWarps ? slot[lane] : 0u);
}

// The exclusive prefix sum of v over the threads in thread order; *total gets the CTA's sum.
// One barrier; slots as for cta_sum.
__device__ __forceinline__ uint32_t cta_exclusive(uint32_t v, uint32_t* slot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;  // inclusive prefix within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) slot[warp] = inc;
  __syncthreads();
  const uint32_t wt = lane < kSelWarps ? slot[lane] : 0u;
  *total = __reduce_add_sync(0xffffffffu, wt);
  const uint32_t before = __reduce_add_sync(0xffffffffu, lane < warp ? wt : 0u);
  return before + inc - v;
}

__global__ void __launch_bounds__(kSelThreads)
    select_cells_kernel(const float* __restrict__ scores, long long stride,
                        const int32_t* __restrict__ kv_len, int budget, int max_kv_len,
                        int stage_cap, int32_t* __restrict__ ids, int32_t* err) {
  extern __shared__ uint32_t staged[];
  __shared__ uint32_t slots[2][kSelWarps];
  const int t = blockIdx.x, tid = threadIdx.x;
  int n = __ldg(kv_len + t);
  if (n < 0 || n > max_kv_len) {
    if (tid == 0) flag_error(err, GQA_ERR_KVLEN_RANGE);
    n = n < 0 ? 0 : max_kv_len;
  }
  int32_t* out = ids + (size_t)t * budget;
  if (n <= budget) {  // every cell, then -1
    for (int i = tid; i < budget; i += kSelThreads) out[i] = i < n ? i : -1;
    return;
  }
  const int nb = (n + 3) >> 2;  // blocks; the last one may hold fewer than 4 cells
  const float* row = scores + (size_t)t * stride;
  const bool stage = nb <= stage_cap;
  if (stage) {
    for (int b = tid; b < nb; b += kSelThreads) staged[b] = monotone_key(__ldg(row + b));
    __syncthreads();
  }
  auto key = [&](int b) { return stage ? staged[b] : monotone_key(__ldg(row + b)); };
  auto cells = [&](int b) { return static_cast<uint32_t>(min(4, n - 4 * b)); };
  int sn = 0;  // alternates the reduction slots
  auto count_ge = [&](uint32_t c) {
    uint32_t m = 0;
    for (int b = tid; b < nb; b += kSelThreads)
      if (key(b) >= c) m += cells(b);
    return cta_sum(m, slots[sn++ & 1]);
  };

  // ---- 1. the threshold key: the largest T with ge(T) >= budget (ge(0) = n > budget)
  const uint32_t want = static_cast<uint32_t>(budget);
  uint32_t T = 0;
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t c = T | (1u << bit);
    if (count_ge(c) >= want) T = c;
  }
  const uint32_t above = T == 0xffffffffu ? 0u : count_ge(T + 1u);
  const uint32_t need = want - above;  // cells taken from blocks at the threshold, >= 1

  // ---- 2. the list, ascending: rounds of kSelThreads blocks, running totals carried over
  uint32_t eq_seen = 0, placed = 0;
  for (int r0 = 0; r0 < nb && placed < want; r0 += kSelThreads) {
    const int b = r0 + tid;
    const bool real = b < nb;
    const uint32_t k = real ? key(b) : 0u;
    const uint32_t w = real ? cells(b) : 0u;
    uint32_t round_eq, round_taken;
    const uint32_t eq_before = eq_seen + cta_exclusive(k == T ? w : 0u, slots[sn++ & 1], &round_eq);
    uint32_t take = 0;
    if (real && k > T) take = w;
    if (real && k == T && need > eq_before) take = min(w, need - eq_before);
    const uint32_t at = placed + cta_exclusive(take, slots[sn++ & 1], &round_taken);
    for (uint32_t i = 0; i < take; ++i) out[at + i] = 4 * b + static_cast<int>(i);
    eq_seen += round_eq;
    placed += round_taken;
  }
}

}  // namespace gqa

namespace gqa {
void set_last_error(const char* msg);               // host.cu: the text gqa_last_error() returns
cudaError_t ensure_smem(const void* fn, int bytes);  // launch_util.cu: the opt-in, once
}

static gqa_status select_fail(gqa_status s, const char* msg) {
  gqa::set_last_error(msg);
  return s;
}

extern "C" gqa_status attn_select_topk(const float* block_scores, int64_t score_stride,
                                       const int32_t* kv_len, int n_tok, int max_kv_len,
                                       int budget, int32_t* ids, int32_t* err_word,
                                       cudaStream_t stream) {
  if (n_tok < 0 || budget <= 0 || max_kv_len < 0)
    return select_fail(GQA_EINVAL,
                       "attn_select_topk: needs n_tok >= 0, budget >= 1, max_kv_len >= 0");
  if (n_tok == 0) return GQA_OK;
  if (!block_scores || !kv_len || !ids)
    return select_fail(GQA_EINVAL, "attn_select_topk: a required pointer is NULL");
  if (score_stride < (int64_t)max_kv_len / 4 + 1)
    return select_fail(GQA_EINVAL, "attn_select_topk: score_stride < max_kv_len / 4 + 1");
  // room for the longest row's keys when they fit the staging limit, else none: a row is staged
  // only when its own block count fits the room launched
  const int nb_max = max_kv_len / 4 + 1;
  const int stage_cap = nb_max <= gqa::kSelStageBlocks ? nb_max : 0;
  if (stage_cap > 0) {  // the opt-in past 48 KB, once, at the largest size
    const cudaError_t e = gqa::ensure_smem(reinterpret_cast<const void*>(gqa::select_cells_kernel),
                                           gqa::kSelStageBlocks * (int)sizeof(uint32_t));
    if (e != cudaSuccess) return select_fail(GQA_ECUDA, cudaGetErrorString(e));
  }
  gqa::select_cells_kernel<<<n_tok, gqa::kSelThreads, (size_t)stage_cap * sizeof(uint32_t),
                             stream>>>(block_scores, (long long)score_stride, kv_len, budget,
                                       max_kv_len, stage_cap, ids, err_word);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return select_fail(GQA_ECUDA, cudaGetErrorString(e));
  return GQA_OK;
}
