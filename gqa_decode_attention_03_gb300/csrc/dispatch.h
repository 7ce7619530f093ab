// dispatch.h -- host-side entry points into the kernel instantiations.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "gqa_decode.h"
#include "partial_kernel.cuh"
#include "rows_mma.cuh"
#include "rows_umma.cuh"
#include "streamk_mma.cuh"

namespace gqa {

struct Variant {
  int gw;   // CUDA-core kernel: query heads per consumer warp (1, 2 or 4)
  int nps;  // CUDA-core kernel: row slices of a stage (consumer warps per head group)
  int mma;  // 1: the tensor-core kernel (f16 caches only)
};

Variant pick_variant(int heads_per_cta);
int head_split_for(int kind, int group);
int stage_rows(int kind, int head_dim);
bool use_streamk(int kind, int n_tok);  // f16 on the tensor cores with few enough rows
int row_group_for(int kind, int n_tok, int n_seq, int group, int head_dim);
bool rows_on_umma();  // grouped rows on the tcgen05 kernel (default) or the mma.sync one
bool q8_on_mma();     // int8 caches on the tensor-core kernel (default) or the CUDA-core one
bool q8_cluster_merge();  // int8 tensor-core kernel: split rows merge inside a cluster

// Defined in the inst_*.cu files, one per (cache kind, head_dim).
cudaError_t launch_partial_f16_d64(Variant v, const CUtensorMap&, const CUtensorMap&,
                                   const PartialParams&, dim3, int, cudaStream_t);
cudaError_t launch_partial_f16_d128(Variant v, const CUtensorMap&, const CUtensorMap&,
                                    const PartialParams&, dim3, int, cudaStream_t);
cudaError_t launch_partial_f16_d256(Variant v, const CUtensorMap&, const CUtensorMap&,
                                    const PartialParams&, dim3, int, cudaStream_t);
cudaError_t launch_partial_q8_d64(Variant v, const CUtensorMap&, const CUtensorMap&,
                                  const PartialParams&, dim3, int, cudaStream_t);
cudaError_t launch_partial_q8_d128(Variant v, const CUtensorMap&, const CUtensorMap&,
                                   const PartialParams&, dim3, int, cudaStream_t);
cudaError_t launch_partial_q8_d256(Variant v, const CUtensorMap&, const CUtensorMap&,
                                   const PartialParams&, dim3, int, cudaStream_t);

inline cudaError_t launch_partial(int kind, int head_dim, Variant v, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const PartialParams& p, dim3 grid,
                                  int threads, cudaStream_t s) {
  if (kind == GQA_KIND_F16) {
    if (head_dim == 64) return launch_partial_f16_d64(v, tk, tv, p, grid, threads, s);
    if (head_dim == 128) return launch_partial_f16_d128(v, tk, tv, p, grid, threads, s);
    return launch_partial_f16_d256(v, tk, tv, p, grid, threads, s);
  }
  if (head_dim == 64) return launch_partial_q8_d64(v, tk, tv, p, grid, threads, s);
  if (head_dim == 128) return launch_partial_q8_d128(v, tk, tv, p, grid, threads, s);
  return launch_partial_q8_d256(v, tk, tv, p, grid, threads, s);
}

cudaError_t launch_streamk_f16_d64(const CUtensorMap&, const CUtensorMap&, const PartialParams&,
                                   dim3, cudaStream_t);
cudaError_t launch_streamk_f16_d128(const CUtensorMap&, const CUtensorMap&, const PartialParams&,
                                    dim3, cudaStream_t);
cudaError_t launch_streamk_f16_d256(const CUtensorMap&, const CUtensorMap&, const PartialParams&,
                                    dim3, cudaStream_t);

inline cudaError_t launch_streamk_f16(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                                      const PartialParams& p, dim3 grid, cudaStream_t s) {
  if (head_dim == 64) return launch_streamk_f16_d64(tk, tv, p, grid, s);
  if (head_dim == 128) return launch_streamk_f16_d128(tk, tv, p, grid, s);
  return launch_streamk_f16_d256(tk, tv, p, grid, s);
}

// tq: the q tensor map of the tcgen05 row kernel ([n_tok][n_heads][D] fp32, box D x G x rows
// of a group); the mma.sync row kernel reads q directly
cudaError_t launch_rows_f16_d64(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                               const PartialParams&, dim3, cudaStream_t);
cudaError_t launch_rows_f16_d128(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                const PartialParams&, dim3, cudaStream_t);

inline cudaError_t launch_rows_f16(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const CUtensorMap& tq, const PartialParams& p, dim3 grid,
                                   cudaStream_t s) {
  return head_dim == 64 ? launch_rows_f16_d64(tk, tv, tq, p, grid, s)
                        : launch_rows_f16_d128(tk, tv, tq, p, grid, s);
}

cudaError_t launch_merge(int head_dim, const float* part, const int32_t* n_valid, int n_split,
                         int n_tok, int n_heads, float* out, cudaStream_t s,
                         const float* gate = nullptr, long long gate_stride = 0,
                         bool after_partials = false, const float* signs = nullptr);

// ensure_smem (raises a function's dynamic shared-memory limit) is declared in
// partial_kernel.cuh.

}  // namespace gqa
