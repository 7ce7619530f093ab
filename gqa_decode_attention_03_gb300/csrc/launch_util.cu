// launch_util.cu -- merge-kernel launcher and the per-function shared-memory attribute cache.
#include <mutex>
#include <set>
#include <utility>

#include "dispatch.h"
#include "merge_kernel.cuh"

namespace gqa {

cudaError_t ensure_smem(const void* fn, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({fn, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({fn, dev});
  return e;
}

cudaError_t launch_merge(int head_dim, const float* part, const int32_t* n_valid, int n_split,
                         int n_tok, int n_heads, float* out, cudaStream_t s, const float* gate,
                         long long gate_stride) {
  // one warp per (row, head), kMergeWarps per CTA
  const long long pairs = (long long)n_tok * n_heads;
  const unsigned grid = static_cast<unsigned>((pairs + kMergeWarps - 1) / kMergeWarps);
  const int threads = 32 * kMergeWarps;
  if (head_dim == 64)
    merge_kernel<64><<<grid, threads, 0, s>>>(part, n_valid, n_split, n_tok, n_heads, gate,
                                              gate_stride, out);
  else if (head_dim == 128)
    merge_kernel<128><<<grid, threads, 0, s>>>(part, n_valid, n_split, n_tok, n_heads, gate,
                                               gate_stride, out);
  else
    merge_kernel<256><<<grid, threads, 0, s>>>(part, n_valid, n_split, n_tok, n_heads, gate,
                                               gate_stride, out);
  return cudaGetLastError();
}

}  // namespace gqa
