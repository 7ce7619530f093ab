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
  const dim3 grid(n_heads, n_tok);  // one CTA of head_dim / 2 threads per (head, row)
  if (head_dim == 64)
    merge_kernel<64><<<grid, 32, 0, s>>>(part, n_valid, n_split, n_heads, gate, gate_stride, out);
  else if (head_dim == 128)
    merge_kernel<128><<<grid, 64, 0, s>>>(part, n_valid, n_split, n_heads, gate, gate_stride,
                                          out);
  else
    merge_kernel<256><<<grid, 128, 0, s>>>(part, n_valid, n_split, n_heads, gate, gate_stride,
                                           out);
  return cudaGetLastError();
}

}  // namespace gqa
