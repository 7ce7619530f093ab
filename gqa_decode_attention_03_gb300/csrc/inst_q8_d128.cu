// inst_q8_d128.cu -- partial-kernel instantiations for int8 caches with f16 scales (cp.async gather), head_dim 128.
#include "dispatch.h"
#include "partial_mma_q8.cuh"

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

cudaError_t launch_partial_q8_d128(Variant v, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const PartialParams& p, dim3 grid, int threads,
                                    cudaStream_t s) {
  constexpr Kind K = Kind::Q8;
  if (v.mma)
    return p.group / p.head_split <= 8 ? launch_mma_q8<128, 1>(p, grid, s)
                                       : launch_mma_q8<128, 2>(p, grid, s);
  if (v.nps == 8) return launch_one<K, 128, 4, 8>(tk, tv, p, grid, threads, s);
  if (v.nps == 4) {
    if (v.gw == 1) return launch_one<K, 128, 1, 4>(tk, tv, p, grid, threads, s);
    if (v.gw == 2) return launch_one<K, 128, 2, 4>(tk, tv, p, grid, threads, s);
    return launch_one<K, 128, 4, 4>(tk, tv, p, grid, threads, s);
  }
  return launch_one<K, 128, 4, 2>(tk, tv, p, grid, threads, s);
}

}  // namespace gqa
