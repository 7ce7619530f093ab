// inst_f16_d64.cu -- kernel instantiations for f16 caches, head_dim 64: the stream-K
// tensor-core kernel (default), the chunked-grid tensor-core kernel (more than 8192 rows, or
// GQA_F16_SPLIT=chunked) and the CUDA-core kernel (GQA_F16_KERNEL=fma; comparison and parity
// cross-check).
#include "dispatch.h"
#include "rows_mma.cuh"
#include "rows_umma.cuh"
#include "streamk_mma.cuh"

namespace gqa {

template <Kind K, int D, int GW, int NPS>
static cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const PartialParams& p,
                              dim3 grid, int threads, cudaStream_t s) {
  using C = Cfg<K, D, GW, NPS>;
  const void* fn = reinterpret_cast<const void*>(&partial_kernel<K, D, GW, NPS>);
  cudaError_t e = ensure_smem(fn, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (threads > C::MAX_THREADS) return cudaErrorInvalidConfiguration;
  partial_kernel<K, D, GW, NPS><<<grid, threads, C::SMEM_BYTES, s>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int NHG>
static cudaError_t launch_sk(const CUtensorMap& tk, const CUtensorMap& tv, const PartialParams& p,
                             dim3 grid, cudaStream_t s) {
  using C = MmaCfg<64, NHG>;
  const void* fn = reinterpret_cast<const void*>(&streamk_mma_kernel<64, NHG>);
  // the stage ring, barriers and the [slices][group][D + 2] slice-merge area
  const int smem = C::SMEM_BYTES + C::NPS * p.group * (64 + 2) * 4;
  cudaError_t e = ensure_smem(fn, C::SMEM_BYTES + C::NPS * 16 * (64 + 2) * 4);
  if (e != cudaSuccess) return e;
  streamk_mma_kernel<64, NHG><<<grid, C::MAX_THREADS, smem, s>>>(tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_streamk_f16_d64(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const PartialParams& p, dim3 grid, cudaStream_t s) {
  return p.group <= 8 ? launch_sk<1>(tk, tv, p, grid, s) : launch_sk<2>(tk, tv, p, grid, s);
}

cudaError_t launch_rows_f16_d64(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                                const PartialParams& p, dim3 grid, cudaStream_t s) {
  if (rows_on_umma()) {
    using U = UmmaRowsCfg<64>;
    const void* fu = reinterpret_cast<const void*>(&umma_rows_kernel<64>);
    cudaError_t e = ensure_smem(fu, U::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // with the fused merge the chunk CTAs of a group wait for one another: a cooperative launch
    // guarantees they are all resident
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(U::THREADS);
    cfg.dynamicSmemBytes = U::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.fused_merge ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, umma_rows_kernel<64>, tk, tv, tq, p);
  }
  using C = RowsCfg<64>;
  const void* fn = reinterpret_cast<const void*>(&partial_mma_rows_kernel<64>);
  cudaError_t e = ensure_smem(fn, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  partial_mma_rows_kernel<64><<<grid, C::MAX_THREADS, C::SMEM_BYTES, s>>>(tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_partial_f16_d64(Variant v, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const PartialParams& p, dim3 grid, int threads,
                                    cudaStream_t s) {
  constexpr Kind K = Kind::F16;
  if (v.mma) return p.group <= 8 ? launch_mma_f16<64, 1>(tk, tv, p, grid, s)
                                 : launch_mma_f16<64, 2>(tk, tv, p, grid, s);
  if (v.nps == 4) {
    if (v.gw == 1) return launch_one<K, 64, 1, 4>(tk, tv, p, grid, threads, s);
    if (v.gw == 2) return launch_one<K, 64, 2, 4>(tk, tv, p, grid, threads, s);
    return launch_one<K, 64, 4, 4>(tk, tv, p, grid, threads, s);
  }
  return launch_one<K, 64, 4, 2>(tk, tv, p, grid, threads, s);
}

}  // namespace gqa
