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
                         long long gate_stride, bool after_partials, const float* signs) {
  // one warp per (row, head), kMergeWarps per CTA
  const long long pairs = (long long)n_tok * n_heads;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>((pairs + kMergeWarps - 1) / kMergeWarps));
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.stream = s;
  // Right after the kernel that writes the partials, as a programmatic dependent launch: the
  // merge CTAs are scheduled while that kernel drains and wait (griddepcontrol.wait) for its
  // completion and memory, so no launch gap separates the two.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_partials ? 1 : 0;
  if (head_dim == 64)
    return cudaLaunchKernelEx(&cfg, merge_kernel<64>, part, n_valid, n_split, n_tok, n_heads,
                              gate, gate_stride, signs, out);
  if (head_dim == 128)
    return cudaLaunchKernelEx(&cfg, merge_kernel<128>, part, n_valid, n_split, n_tok, n_heads,
                              gate, gate_stride, signs, out);
  return cudaLaunchKernelEx(&cfg, merge_kernel<256>, part, n_valid, n_split, n_tok, n_heads, gate,
                            gate_stride, signs, out);
}

}  // namespace gqa
