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
//      descending order.  It is built eight bits at a time from the most significant.  At the
//      step for bits sh .. sh + 7, a block whose key agrees with T above them adds its cells to
//      bin `digit` of its warp's 257-bin histogram (shared atomics), a block whose higher bits
//      already exceed T's to bin 256; the others count for nothing.  The warps' bins are summed
//      and a CTA scan turns them into suffix sums, ge(T + j 2^sh) for every candidate digit j;
//      the digit is the one whose suffix still holds budget cells while the next one's does
//      not.  After the last step the next suffix is ge(T + 1), the cells strictly above T; the
//      remaining need = budget - ge(T + 1) cells come from blocks whose key equals T, lowest
//      cells first.  When a step leaves at most kSelFinishCells cells in the chosen digit's bin
//      (at most 32 blocks: scores spread over a range end there after two steps), those blocks
//      are gathered and one warp ranks them directly: T is the key of the candidate whose
//      cells above it fall short of the need while its own reach it, the same T and ge(T + 1)
//      the remaining steps would find.
//   2. The list.  Blocks are visited in ascending order in rounds of 4 kSelThreads blocks,
//      four consecutive blocks a thread.  Exclusive scans (within the thread, then over the
//      CTA) of the cells at key T give each block the number of such cells before it, hence how
//      many of its own it takes; a second pair of scans of the taken cells gives each block its
//      place in the output.  Both running totals carry over to the next round.
// The row's block keys are staged in shared memory when its block count fits the room the
// launch reserved; otherwise each step reads them from global memory (L2 after the first).
// Integer work only: the list is a deterministic function of the keys.
#include <cuda_runtime_api.h>

#include "common.cuh"
#include "gqa_decode.h"

namespace gqa {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelStageBlocks = 46080;  // 180 KB of staged keys: rows of up to 184,319 cells
constexpr int kSelBins = 257;           // digits 0..255 of a step, and "above every candidate"
constexpr int kSelSpecBlocks = 4096;    // block scores read before the row length is known
constexpr uint32_t kSelFinishCells = 124;  // candidates ranked by one warp: <= 32 blocks

// fp32 bit pattern -> uint32 whose unsigned order is the float order (-0 below +0; NaNs at the
// ends): negative values have every bit flipped, the others get the sign bit set.
__device__ __forceinline__ uint32_t monotone_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u ^ 0x80000000u);
}

// The exclusive prefix sum of v over the threads in thread order; *total gets the CTA's sum.
// One barrier; `slot` (kSelWarps words or more) must not be the slot of the previous
// CTA-wide call (callers alternate two).
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
  __shared__ uint32_t hist[2][kSelWarps][kSelBins];  // per-warp digit histograms, two steps
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // a decode launched after this kernel as a programmatic dependent may be scheduled now: its
  // CTAs set up beside this one and wait for this grid's completion before reading ids
  asm volatile("griddepcontrol.launch_dependents;");
  int n = __ldg(kv_len + t);
  // the row's first kSelSpecBlocks block scores are read beside its length, not after it (the
  // row holds stride >= stage_cap of them: in bounds whatever the length)
  const float* row = scores + (size_t)t * stride;
  const int spec = min(stage_cap, kSelSpecBlocks);
  float pre[kSelSpecBlocks / kSelThreads];
#pragma unroll
  for (int i = 0; i < kSelSpecBlocks / kSelThreads; ++i) {
    const int b = tid + i * kSelThreads;
    pre[i] = b < spec ? __ldg(row + b) : 0.f;
  }
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
  const bool stage = nb <= stage_cap;
  for (int i = lane; i < kSelBins; i += 32) hist[0][warp][i] = hist[1][warp][i] = 0u;
  if (stage) {
#pragma unroll
    for (int i = 0; i < kSelSpecBlocks / kSelThreads; ++i) {
      const int b = tid + i * kSelThreads;
      if (b < min(nb, spec)) staged[b] = monotone_key(pre[i]);
    }
    for (int b = spec + tid; b < nb; b += kSelThreads) staged[b] = monotone_key(__ldg(row + b));
  }
  __syncthreads();
  auto key = [&](int b) { return stage ? staged[b] : monotone_key(__ldg(row + b)); };
  auto cells = [&](int b) { return static_cast<uint32_t>(min(4, n - 4 * b)); };
  int sn = 0;  // alternates the reduction slots

  // ---- 1. the threshold key, eight bits a step (ge(T) >= budget holds throughout: ge(0) = n)
  __shared__ uint32_t pick[3];  // the step's digit, the cells above T + 2^sh, the digit's cells
  __shared__ uint32_t cand_key[32], cand_cells[32], cand_n;  // the direct finish's candidates
  const uint32_t want = static_cast<uint32_t>(budget);
  uint32_t T = 0, above = 0;
  for (int step = 0, sh = 24; sh >= 0; ++step, sh -= 8) {
    // Bin of a block: its key's digit at sh (0 .. 255) when the key agrees with T above bit
    // sh + 8, bin 256 when its higher bits already exceed T's (above every candidate), no bin
    // when they fall short.  Cells go into the warp's own histogram by shared atomics.
    uint32_t(*h)[kSelBins] = hist[step & 1];
    const uint32_t hiT = sh == 24 ? 0u : T >> (sh + 8);
    for (int b = tid; b < nb; b += kSelThreads) {
      const uint32_t k = key(b);
      const uint32_t hk = sh == 24 ? 0u : k >> (sh + 8);
      if (hk >= hiT) atomicAdd(&h[warp][hk > hiT ? 256u : (k >> sh) & 255u], cells(b));
    }
    __syncthreads();
    // thread i (< 257) gathers bin i over the warps; suf_i = cells in bins >= i, i.e.
    // ge(T + i 2^sh) for the digits i = 1 .. 255, and the cells above every candidate for 256
    uint32_t bin = 0;
    if (tid < kSelBins)
      for (int w = 0; w < kSelWarps; ++w) bin += h[w][tid];
    uint32_t total;
    const uint32_t before = cta_exclusive(bin, slots[sn++ & 1], &total);
    const uint32_t suf = total - before;
    // the digit: the one i in 0 .. 255 with suf_i >= budget > suf_(i+1) = suf_i - bin_i
    // (suf_0 >= budget, and suf does not grow with i)
    if (tid < 256 && suf >= want && suf - bin < want) {
      pick[0] = tid;
      pick[1] = suf - bin;
      pick[2] = bin;
    }
    if (tid == 0) cand_n = 0u;
    __syncthreads();
    T |= pick[0] << sh;
    above = pick[1];  // cells at or above T + 2^sh
    // the other histogram was last read in the previous step, before two barriers: clear it
    // (this warp's own rows) for the next step
    for (int i = lane; i < kSelBins; i += 32) hist[(step + 1) & 1][warp][i] = 0u;
    __syncwarp();
    if (sh > 0 && pick[2] <= kSelFinishCells) {  // the same for every thread
      // ---- the direct finish: the blocks of the chosen digit's bin (keys agreeing with T
      //      from bit sh up), then warp 0 ranks them
      for (int b = tid; b < nb; b += kSelThreads) {
        const uint32_t k = key(b);
        if ((k >> sh) == (T >> sh)) {
          const uint32_t at = atomicAdd(&cand_n, 1u);
          cand_key[at] = k;
          cand_cells[at] = cells(b);
        }
      }
      __syncthreads();
      if (warp == 0) {
        const uint32_t nc = cand_n, need_c = want - above;  // 1 <= need_c <= the bin's cells
        const uint32_t kl = lane < nc ? cand_key[lane] : 0u;
        const uint32_t wl = lane < nc ? cand_cells[lane] : 0u;
        uint32_t gt = 0, eq = 0;  // cells of the candidates above / at this lane's key
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
          const uint32_t kj = __shfl_sync(0xffffffffu, kl, j);
          const uint32_t wj = __shfl_sync(0xffffffffu, wl, j);
          gt += kj > kl ? wj : 0u;
          eq += kj == kl ? wj : 0u;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, lane < nc && gt < need_c && need_c <= gt + eq);
        if (lane == (hit ? __ffs(hit) - 1 : 0)) {
          pick[0] = kl;
          pick[1] = above + gt;
        }
      }
      __syncthreads();
      T = pick[0];
      above = pick[1];  // cells above T
      break;
    }
  }
  const uint32_t need = want - above;  // cells taken from blocks at the threshold, >= 1

  // ---- 2. the list, ascending: rounds of 4 kSelThreads blocks, 4 consecutive blocks a
  //      thread, running totals carried over
  constexpr int BPT = 4;
  uint32_t eq_seen = 0, placed = 0;
  for (int r0 = 0; r0 < nb && placed < want; r0 += BPT * kSelThreads) {
    const int b0 = r0 + BPT * tid;
    uint32_t k[BPT], w[BPT], eq_own = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      const bool real = b0 + i < nb;
      k[i] = real ? key(b0 + i) : 0u;
      w[i] = real ? cells(b0 + i) : 0u;
      eq_own += k[i] == T ? w[i] : 0u;
    }
    uint32_t round_eq, round_taken;
    uint32_t eq_before = eq_seen + cta_exclusive(eq_own, slots[sn++ & 1], &round_eq);
    uint32_t take[BPT], take_own = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      take[i] = k[i] > T ? w[i] : 0u;
      if (k[i] == T) {
        take[i] = need > eq_before ? min(w[i], need - eq_before) : 0u;
        eq_before += w[i];
      }
      take_own += take[i];
    }
    uint32_t at = placed + cta_exclusive(take_own, slots[sn++ & 1], &round_taken);
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      for (uint32_t c = 0; c < take[i]; ++c) out[at + c] = 4 * (b0 + i) + static_cast<int>(c);
      at += take[i];
    }
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
