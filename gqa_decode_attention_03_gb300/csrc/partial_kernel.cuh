// partial_kernel.cuh -- split-KV decode-attention partial kernel (f16 and int8+scale caches).
//
// One CTA per (KV chunk c, KV head g, query row t).  The CTA stages its chunk of K/V rows through
// a ring of shared-memory stages once and every query head of g's group reads them there: the
// "load K/V once per KV head, reuse across the group" structure of attention_gqa.metal (cera
// 0.5.4), with the tiled online softmax of flash_attention.metal (cera 0.2.0, the tile loop with
// its running max / running sum / correction and the guard for the first tile) and the chunked
// partials of qsa2.metal (regolith, qsa_attn2: unnormalised accumulator, chunk max, chunk sum).
//
// Warp roles.
//   * one producer warp: f16 caches arrive by TMA (3-D tensor map over [seq*cap][Hk][D], 128-byte
//     swizzle, one box per 64 dims); int8 caches (dense or through a selected-cell id list) are
//     gathered row by row with 16-byte cp.async, the f16 scales with 8/4-byte cp.async.  Stage
//     completion is tracked by mbarriers (transaction bytes for TMA, cp.async arrivals for the
//     gather); consumers release a stage through a second mbarrier.
//   * nhg * NPS consumer warps: warp w serves head group w % nhg (GW heads each) on the row
//     slice w / nhg of every stage.  Each warp keeps its own running max / sum / accumulator in
//     registers (scores in log2 units: q is pre-scaled by scale * log2 e), so no CTA-wide barrier
//     sits in the tile loop.  At the end the slices are merged by log-sum-exp in shared memory.
//
// q.k: LPP lanes share a row, each holding CPL 16-byte chunks of it and the matching q slice in
// registers; the GW partial dots are reduce-scattered across the LPP lanes (log2 LPP shuffle
// levels, halving the values held at each level).  p.v: a lane owns D/32 consecutive dims for
// all GW heads; p comes from a per-warp shared buffer (broadcast reads).
#pragma once

#include <atomic>

#include "common.cuh"

namespace gqa {

enum class Kind { F16 = 0, Q8 = 1 };

struct PartialParams {
  const float* q;          // [T][H][D]
  const void* kc;          // int8 caches (gather path); f16 caches come through tensor maps
  const void* vc;
  const __half* ksc;       // [n_seq][cap][Hk][D >> sc_shift] (int8 only)
  const __half* vsc;
  int sc_shift;            // int8: log2 of the dims sharing a scale (6: 64 dims, 5: 32 dims)
  const int32_t* ids;      // [T][budget] or null
  const int32_t* kv_len;   // [T]
  const int32_t* seq_of;   // [T] or null
  float* out;              // [T][H][D]          (merge == 0)
  float* part;             // [T][S][H][D+2]     (merge == 1)
  int32_t* n_valid;        // [T] chunks holding data, written when merge == 1
  unsigned int* counters;  // [T][Hk] chunk arrivals (zero before and after every call)
  int32_t* err;            // device error word or null
  int n_tok, n_seq, n_heads, n_kv_heads, group;
  int head_split;          // CUDA-core kernel: CTAs per KV head, each serving group/head_split
                           // query heads (grid.y = n_kv_heads * head_split); 1 elsewhere
  long long cache_cap;
  int max_kv_len;
  int budget;              // ids != null: width cap; otherwise unused
  int chunk;               // rows (positions or selected cells) per chunk; multiple of TP
  int n_split;             // chunks per row in the grid (grid.x)
  float scale_log2;        // scale * log2(e)
  int merge;
  int fused_merge;         // row kernels (tcgen05 f16, TurboQuant): the chunk CTAs of a group
                           // merge its partials themselves (cooperative launch; counters
                           // [groups][n_kv_heads], [groups][grid.y] for TurboQuant)
  unsigned int merge_spin; // polls of the fused merge's wait for the group's other chunk CTAs
                           // before it gives up (kSpinLimit unless a test asks for fewer)
  const float* gate;       // sigmoid output gate or null: element (t, h, d) at
  long long gate_stride;   //   gate[(t * n_heads + h) * gate_stride + d]
  int pdl;                 // f16 tensor-core kernel launched as a programmatic dependent
  int rows_fixed;          // tcgen05 row kernel, one sequence: group k is rows [k R, k R + R),
                           // found without a scan of seq_of, a row valid iff its seq_of is 0
                           // (host-set when n_seq == 1)
  int cluster;             // tensor-core per-row kernels: > 1 when the row's chunk CTAs form
                           // one thread-block cluster (dims (n_split, 1, 1)) and merge through
                           // distributed shared memory instead of the arrival counters (the
                           // host sets 1 where the f16 kernel may, the launcher the size)
};

// The sigmoid output gate that both pages apply to the merged row (qsa2.metal, qsa_merge2;
// FORWARD_MSL, attn_combine): y / (1 + exp(-gate)) for output element (t, h, d); y itself when
// the call has no gate.  Applied wherever a kernel writes an output row, after any epilogue.
__device__ __forceinline__ float gated(const PartialParams& p, int t, int h, int d, float y) {
  if (!p.gate) return y;
  const float g = __ldg(p.gate + ((size_t)t * p.n_heads + h) * p.gate_stride + d);
  return y * (1.f / (1.f + __expf(-g)));
}

__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int align_up(int a, int b) { return (a + b - 1) / b * b; }

template <Kind K, int D, int GW, int NPS>
struct Cfg {
  static constexpr int ESZ = (K == Kind::F16) ? 2 : 1;     // bytes per cache element
  static constexpr int RB = D * ESZ;                       // bytes per cache row
  static constexpr int CPR = RB / 16;                      // 16-byte chunks per row
  static constexpr int DPC = 16 / ESZ;                     // dims per chunk
  static constexpr int NBOX = (RB + 127) / 128;            // 128-byte boxes per row
  static constexpr int CPL_MAX = cmax(1, 64 / (DPC * GW)); // q registers per lane <= 64
  static constexpr int LPP = cmax(cmin(8, CPR), CPR / CPL_MAX);  // lanes per row in q.k
  static constexpr int CPL = CPR / LPP;                    // chunks per lane
  static constexpr int RPP = 32 / LPP;                     // rows per warp pass
  static constexpr int TP = (K == Kind::F16) ? (D == 64 ? 128 : D == 128 ? 64 : 32)
                                             : (D == 256 ? 64 : 128);  // rows per stage
  static constexpr int TPW = TP / NPS;                     // rows per warp per stage
  static constexpr int NP = TPW / RPP;                     // q.k passes per warp per stage
  static constexpr int NST = 3;                            // pipeline stages
  static constexpr int DPL = D / 32;                       // p.v dims per lane
  static constexpr int NSC = D / 32;                       // staged f16 scales per int8 row
                                                           // (room for 32-dim groups)
  static constexpr int BOX_BYTES = TP * 128;
  static constexpr int KV_BYTES = 2 * NBOX * BOX_BYTES;    // K and V tiles of one stage
  static constexpr int SC_BYTES = (K == Kind::Q8) ? align_up(2 * TP * NSC * 2, 16) : 0;
  static constexpr int OK_BYTES = (K == Kind::Q8) ? align_up(TP * 4, 16) : 0;
  static constexpr int STAGE_BYTES = align_up(KV_BYTES + SC_BYTES + OK_BYTES, 1024);
  static constexpr int MAX_WARPS = (NPS == 4) ? 4 : 8;     // consumer warps at most
  static constexpr int PS_BYTES = MAX_WARPS * TPW * GW * 4;
  static constexpr int MERGE_BYTES = MAX_WARPS * GW * (D + 2) * 4;
  static constexpr int SMEM_BYTES =
      1024 /*alignment slack*/ + NST * STAGE_BYTES + PS_BYTES + 2 * NST * 8;
  static constexpr int MAX_THREADS = 32 * (MAX_WARPS + 1);
  static constexpr int MIN_BLOCKS = (NPS == 4) ? 2 : 1;
  static_assert(GW <= LPP, "reduce-scatter needs at least GW lanes per row");
  static_assert(TPW % RPP == 0, "rows per warp must fill whole passes");
  static_assert(MERGE_BYTES <= NST * STAGE_BYTES, "merge area aliases the stages");
  static_assert(CPR % LPP == 0, "chunks must split evenly over the lanes of a row");
};

// 8 f16 (one 16-byte chunk) -> 8 floats
__device__ __forceinline__ void cvt_chunk(const uint4& u, float (&f)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 x = __half22float2(h[i]);
    f[2 * i] = x.x;
    f[2 * i + 1] = x.y;
  }
}

// 16 int8 (one 16-byte chunk) -> 16 floats
__device__ __forceinline__ void cvt_chunk(const uint4& u, float (&f)[16]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int b = 0; b < 4; ++b) f[4 * i + b] = static_cast<float>(static_cast<int8_t>(w[i] >> (8 * b)));
  }
}

// D/32 consecutive cache elements of one row (the p.v slice of a lane) -> floats.
template <Kind K, int N>
__device__ __forceinline__ void load_pv(const uint8_t* src, float (&f)[N]) {
  if constexpr (K == Kind::F16) {
    if constexpr (N == 2) {
      const float2 x = __half22float2(*reinterpret_cast<const __half2*>(src));
      f[0] = x.x;
      f[1] = x.y;
    } else if constexpr (N == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(src);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      static_assert(N == 8, "f16 p.v slice is 2, 4 or 8 dims");
      cvt_chunk(*reinterpret_cast<const uint4*>(src), f);
    }
  } else {
    if constexpr (N == 2) {
      const uint16_t u = *reinterpret_cast<const uint16_t*>(src);
      f[0] = static_cast<float>(static_cast<int8_t>(u & 0xff));
      f[1] = static_cast<float>(static_cast<int8_t>(u >> 8));
    } else if constexpr (N == 4) {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(src);
#pragma unroll
      for (int b = 0; b < 4; ++b) f[b] = static_cast<float>(static_cast<int8_t>(u >> (8 * b)));
    } else {
      static_assert(N == 8, "int8 p.v slice is 2, 4 or 8 dims");
      const uint2 u = *reinterpret_cast<const uint2*>(src);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        f[b] = static_cast<float>(static_cast<int8_t>(u.x >> (8 * b)));
        f[4 + b] = static_cast<float>(static_cast<int8_t>(u.y >> (8 * b)));
      }
    }
  }
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Sums GW values over the LPP lanes of a row group (aligned, xor-addressed) and leaves lane li
// holding the total of value li / (LPP / GW) in v[0].  At each shuffle level a lane keeps one half
// of its values and trades the other half with its partner, so the level count is log2(LPP) and
// the shuffle count GW - 1 + log2(LPP / GW).
template <int GW, int LPP>
__device__ __forceinline__ void reduce_scatter(float (&v)[GW], int lane) {
#pragma unroll
  for (int l = 0; l < ilog2(LPP); ++l) {
    const int mask = LPP >> (l + 1);
    const int n = (GW >> l) > 1 ? (GW >> l) : 1;
    if (n > 1) {
      const int half = n / 2;
      const bool up = (lane & mask) != 0;
#pragma unroll
      for (int k = 0; k < half; ++k) {
        const float send = up ? v[k] : v[k + half];
        const float keep = up ? v[k + half] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
    }
  }
}

// ------------------------------------------------------------------------------ fused merge

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Called by every consumer thread after this CTA wrote its chunk's partial records.  The CTA
// takes a ticket on its counter (one per row, KV head and CTA head group); the CTA holding the
// last of the nv tickets merges the nv chunks of heads head0 .. head0 + nheads - 1 by
// log-sum-exp (qsa2.metal, qsa_merge2) and writes out.  atomicInc wraps the counter back to 0
// on the last ticket, so every call leaves it at zero.  Nobody waits for anybody: the CTAs that
// are not last simply finish.  One warp per head; lane c holds chunk c's (m, l) and weight and
// broadcasts the weight by shuffle, so a head's loads go out in one round.
struct NoEpilogue {  // merge_if_last writes the merged rows as they are
  template <int N>
  __device__ __forceinline__ void operator()(float (&)[N], int /*head*/, int /*lane*/) const {}
};

template <int D, class Epi = NoEpilogue>
__device__ __forceinline__ void merge_if_last(const PartialParams& p, int t, int head0,
                                              int nheads, size_t counter, int nv, int ncw,
                                              const Epi& epi = Epi()) {
  __shared__ int s_last;
  __threadfence();  // this thread's partial stores, visible device-wide before the ticket
  named_bar_sync(1, ncw * 32);
  if (threadIdx.x == 0)
    s_last = atomicInc(p.counters + counter, (unsigned)(nv - 1)) == (unsigned)(nv - 1);
  named_bar_sync(1, ncw * 32);
  if (!s_last) return;
  __threadfence();
  constexpr int DPL = D / 32;  // output dims per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rec = (size_t)p.n_heads * (D + 2);  // floats between consecutive chunks
  for (int h = warp; h < nheads; h += ncw) {
    const int head = head0 + h;
    const float* base = p.part + ((size_t)t * p.n_split * p.n_heads + head) * (D + 2);
    float* o = p.out + ((size_t)t * p.n_heads + head) * D + lane * DPL;
    float M = -INFINITY;
    for (int cc = lane; cc < nv; cc += 32) M = fmaxf(M, __ldcg(base + cc * rec + D));
    M = warp_max(M);
    float a[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) a[k] = 0.f;
    float Ls = 0.f;
    if (M != -INFINITY) {
      for (int c0 = 0; c0 < nv; c0 += 32) {
        float e = 0.f;
        if (c0 + lane < nv) {
          const float m = __ldcg(base + (c0 + lane) * rec + D);
          e = m == -INFINITY ? 0.f : __expf(m - M);
          Ls = fmaf(__ldcg(base + (c0 + lane) * rec + D + 1), e, Ls);
        }
        const int nb = min(32, nv - c0);
#pragma unroll 8
        for (int j = 0; j < nb; ++j) {
          const float ej = __shfl_sync(0xffffffffu, e, j);
          const float* ac = base + (c0 + j) * rec + lane * DPL;
          if constexpr (DPL == 1) {  // D = 32: one dim a lane, 4-byte loads
            a[0] = fmaf(ej, __ldcg(ac), a[0]);
          } else {
#pragma unroll
            for (int k = 0; k < DPL; k += 2) {
              const float2 v = __ldcg(reinterpret_cast<const float2*>(ac + k));
              a[k] = fmaf(ej, v.x, a[k]);
              a[k + 1] = fmaf(ej, v.y, a[k + 1]);
            }
          }
        }
      }
      Ls = warp_sum(Ls);
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
    for (int k = 0; k < DPL; ++k) a[k] *= inv;
    epi(a, head, lane);  // e.g. the inverse rotation of a rotated-space accumulator
#pragma unroll
    for (int k = 0; k < DPL; ++k) a[k] = gated(p, t, head, lane * DPL + k, a[k]);
    if constexpr (DPL == 1) {
      o[0] = a[0];
    } else {
#pragma unroll
      for (int k = 0; k < DPL; k += 2) *reinterpret_cast<float2*>(o + k) = make_float2(a[k], a[k + 1]);
    }
  }
}

// The row's chunk CTAs, one thread-block cluster (chunk c = cluster rank c), each holding its
// partial [head][D + 2] (acc | m in log2 units | l) at `cp` in its shared memory, merge by
// log-sum-exp through distributed shared memory: after a cluster barrier, the CTAs of chunks
// 0 .. nchunks-1 share the (head, dim) outputs, reading every chunk's partial, and write the
// (gated) output; a second barrier keeps every CTA resident until all reads are done.  Every
// thread of every CTA of the cluster must take both barriers (CTAs whose chunk is empty and
// producer warps call cluster_sync twice instead).
template <int D, int MAXC>
__device__ __forceinline__ void cluster_merge(const PartialParams& p, int t, int head0, int nheads,
                                              int c, int nchunks, const uint8_t* cp, int ncw) {
  cluster_sync();  // every chunk's partial is in place
  const uint32_t cpa = smem_addr(cp);
  for (int idx = c * ncw * 32 + threadIdx.x; idx < nheads * D; idx += nchunks * ncw * 32) {
    const int h2 = idx / D, d = idx % D;
    const uint32_t rec = cpa + static_cast<uint32_t>(h2 * (D + 2)) * 4u;
    float mr[MAXC], ar[MAXC], lr[MAXC];
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < MAXC; ++r) {
      mr[r] = -INFINITY;
      ar[r] = lr[r] = 0.f;
      if (r < nchunks) {
        mr[r] = ld_cluster_f32(cluster_map(rec + D * 4u, r));
        lr[r] = ld_cluster_f32(cluster_map(rec + (D + 1) * 4u, r));
        ar[r] = ld_cluster_f32(cluster_map(rec + d * 4u, r));
      }
      M = fmaxf(M, mr[r]);
    }
    float A = 0.f, Ls = 0.f;
#pragma unroll
    for (int r = 0; r < MAXC; ++r) {
      const float e = mr[r] == -INFINITY ? 0.f : fast_exp2(mr[r] - M);
      A = fmaf(ar[r], e, A);
      Ls = fmaf(lr[r], e, Ls);
    }
    const int head = head0 + h2;
    p.out[((size_t)t * p.n_heads + head) * D + d] = gated(p, t, head, d, Ls > 0.f ? A / Ls : 0.f);
  }
  cluster_sync();  // no CTA leaves while another still reads its shared memory
}

// Host: raises the function's dynamic shared-memory limit once per (function, device)
// (launch_util.cu).
cudaError_t ensure_smem(const void* fn, int bytes);

// Host: whether clusters of n CTAs of this launch configuration fit the GPU at all (asked once
// per cluster size and kernel instantiation), and the launch attributes for a cluster of n
// (n > 1) and a programmatic dependent launch; returns how many were written to at[0..1].
template <int MAXC>
bool cluster_fits(const void* fn, const cudaLaunchConfig_t& cfg0, unsigned n) {
  static std::atomic<int> fits[MAXC + 1];  // 0 unknown, 1 yes, 2 no
  if (n < 2 || n > static_cast<unsigned>(MAXC)) return false;
  if (fits[n].load() == 0) {
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = n;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = cfg0;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int k = 0;
    const bool ok = cudaOccupancyMaxActiveClusters(&k, fn, &cfg) == cudaSuccess && k > 0;
    if (!ok) (void)cudaGetLastError();
    fits[n].store(ok ? 1 : 2);
  }
  return fits[n].load() == 1;
}

inline int cluster_attrs(cudaLaunchAttribute* at, int cluster, int pdl) {
  int n = 0;
  if (cluster > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  return n;
}

// ------------------------------------------------------------------------------ producers

// f16: lane 0 streams the chunk's K/V tiles by TMA into the stage ring.
template <class C>
__device__ __forceinline__ void produce_tma(const CUtensorMap* tmK, const CUtensorMap* tmV,
                                            uint8_t* stages, uint64_t* full, uint64_t* empty,
                                            int ntiles, int g, int z0, int32_t* err) {
  tma_prefetch_desc(tmK);
  tma_prefetch_desc(tmV);
  int issued = 0;
  bool ok = true;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::NST;
    if (i >= C::NST && !mbar_wait(&empty[st], ((i / C::NST) - 1) & 1)) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(&full[st], C::KV_BYTES);
    uint8_t* sk = stages + st * C::STAGE_BYTES;
    uint8_t* sv = sk + C::NBOX * C::BOX_BYTES;
    const int z = z0 + i * C::TP;
#pragma unroll
    for (int b = 0; b < C::NBOX; ++b) {
      tma_load_3d(sk + b * C::BOX_BYTES, tmK, b * 64, g, z, &full[st]);
      tma_load_3d(sv + b * C::BOX_BYTES, tmV, b * 64, g, z, &full[st]);
    }
    issued = i + 1;
  }
  if (!ok) flag_error(err, GQA_ERR_TIMEOUT);
  // the last load issued into each stage must land before the CTA may exit
  for (int st = 0; st < C::NST && st < issued; ++st) {
    const int last = st + ((issued - 1 - st) / C::NST) * C::NST;
    if (!mbar_wait(&full[st], (last / C::NST) & 1)) flag_error(err, GQA_ERR_TIMEOUT);
  }
}

// int8: the 32 lanes gather the chunk's rows (through the id list when there is one) with
// cp.async; a row whose id lies outside [0, L) is flagged, masked, and filled from cell 0 so
// the staged bytes stay finite.  The ids of tile i + 1 are loaded before tile i's copies are
// issued (a lane's rows of a tile at once), so their latency overlaps the copies instead of
// preceding each row's.
template <class C, int D, int NPW = 1>
__device__ __forceinline__ void produce_gather(const PartialParams& p, uint8_t* stages,
                                               uint64_t* full, uint64_t* empty, int ntiles,
                                               int t, int g, int s, int L, int c0, int c1,
                                               int lane, const int* first = nullptr,
                                               int pw = 0) {
  const uint8_t* kq = static_cast<const uint8_t*>(p.kc);
  const uint8_t* vq = static_cast<const uint8_t*>(p.vc);
  // rows of a tile per lane: producer warp pw of NPW takes rows lane + 32 (pw + NPW k)
  constexpr int RPL = C::TP / 32 / NPW;
  static_assert(C::TP % (32 * NPW) == 0, "whole rows per lane");
  static_assert(C::TP % 32 == 0, "whole rows per lane");
  auto fetch = [&](int i, int (&cell)[RPL]) {  // the visited-list entries of tile i
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int j = c0 + i * C::TP + lane + 32 * (pw + NPW * k);
      cell[k] = j < c1 ? (p.ids ? __ldg(p.ids + (size_t)t * p.budget + j) : j) : 0;
    }
  };
  int cur[RPL], nxt[RPL];
  if (first) {  // tile 0's entries, fetched by the caller (any value where j >= c1)
#pragma unroll
    for (int k = 0; k < RPL; ++k) cur[k] = first[k];
  } else {
    fetch(0, cur);
  }
  int issued = 0;
  bool ok = true;
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::NST;
    if (i + 1 < ntiles) fetch(i + 1, nxt);
    if (i >= C::NST) {
      const bool w = __all_sync(0xffffffffu, mbar_wait(&empty[st], ((i / C::NST) - 1) & 1));
      if (!w) {
        ok = false;
        break;
      }
    }
    uint8_t* sk = stages + st * C::STAGE_BYTES;
    uint8_t* sv = sk + C::NBOX * C::BOX_BYTES;
    __half* skc = reinterpret_cast<__half*>(sk + C::KV_BYTES);
    __half* svc = skc + C::TP * C::NSC;
    int* rowok = reinterpret_cast<int*>(sk + C::KV_BYTES + C::SC_BYTES);
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int r = lane + 32 * (pw + NPW * k);
      const int j = c0 + i * C::TP + r;  // index into the visited list
      int okr = 0;
      if (j < c1) {
        int cell = cur[k];
        okr = (cell >= 0 && cell < L);
        if (!okr) {
          flag_error(p.err, GQA_ERR_ID_RANGE);
          cell = 0;
        }
        const size_t row = ((size_t)s * p.cache_cap + cell) * p.n_kv_heads + g;
        const uint8_t* gk = kq + row * D;
        const uint8_t* gv = vq + row * D;
#pragma unroll
        for (int ch = 0; ch < C::CPR; ++ch) {
          cp_async_16(sk + swz_off(r, ch, C::TP), gk + ch * 16);
          cp_async_16(sv + swz_off(r, ch, C::TP), gv + ch * 16);
        }
        const int nsc = D >> p.sc_shift;  // scales of this row: 2 .. 8
        const __half* gks = p.ksc + row * nsc;
        const __half* gvs = p.vsc + row * nsc;
        if (nsc == 8) {
          cp_async_16(skc + r * C::NSC, gks);
          cp_async_16(svc + r * C::NSC, gvs);
        } else if (nsc == 4) {
          cp_async_8(skc + r * C::NSC, gks);
          cp_async_8(svc + r * C::NSC, gvs);
        } else if (nsc == 2) {
          cp_async_4(skc + r * C::NSC, gks);
          cp_async_4(svc + r * C::NSC, gvs);
        } else {
          skc[r * C::NSC] = gks[0];
          svc[r * C::NSC] = gvs[0];
        }
      }
      rowok[r] = okr;
    }
    mbar_arrive(&full[st]);            // releases rowok and the plain scale stores
    cp_async_arrive_noinc(&full[st]);  // fires once this lane's copies have landed
    issued = i + 1;
#pragma unroll
    for (int k = 0; k < RPL; ++k) cur[k] = nxt[k];
  }
  if (!ok && lane == 0) flag_error(p.err, GQA_ERR_TIMEOUT);
  for (int st = 0; st < C::NST && st < issued; ++st) {
    const int last = st + ((issued - 1 - st) / C::NST) * C::NST;
    if (!mbar_wait(&full[st], (last / C::NST) & 1)) flag_error(p.err, GQA_ERR_TIMEOUT);
  }
}

// ------------------------------------------------------------------------------ the kernel

template <Kind K, int D, int GW, int NPS>
__global__ void __launch_bounds__(Cfg<K, D, GW, NPS>::MAX_THREADS, Cfg<K, D, GW, NPS>::MIN_BLOCKS)
    partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const PartialParams p) {
  using C = Cfg<K, D, GW, NPS>;
  extern __shared__ uint8_t smem_raw[];
  const int c = blockIdx.x, t = blockIdx.z;
  const int g = blockIdx.y / p.head_split;        // KV head
  const int G = p.group / p.head_split;           // query heads served by this CTA
  const int head0 = g * p.group + (blockIdx.y % p.head_split) * G;  // its first query head
  const int nhg = (G + GW - 1) / GW;
  const int ncw = nhg * NPS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the row's visited list (uniform over the CTA)
  int L = __ldg(p.kv_len + t);
  int errbits = 0;
  const int lmax = static_cast<int>(p.cache_cap < p.max_kv_len ? p.cache_cap : p.max_kv_len);
  if (L < 0 || L > lmax) {
    errbits |= GQA_ERR_KVLEN_RANGE;
    L = L < 0 ? 0 : lmax;
  }
  const int s = p.seq_of ? __ldg(p.seq_of + t) : t;
  if (s < 0 || s >= p.n_seq) {
    errbits |= GQA_ERR_SEQ_RANGE;
    L = 0;
  }
  const int nsel = p.ids ? min(L, p.budget) : L;  // qsa2.metal: width = min(n_kv, budget)
  const int c0 = c * p.chunk;
  const int c1 = min(c0 + p.chunk, nsel);
  if (c == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    if (errbits) flag_error(p.err, errbits);
    if (p.merge) p.n_valid[t] = (nsel + p.chunk - 1) / p.chunk;
  }
  if (c0 >= nsel) {
    // empty context: zeros (flash_attention.metal's seq_len == 0 guard), written by chunk 0
    // whether or not the row is split, since no CTA of the row merges anything
    if (c == 0)
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        p.out[((size_t)t * p.n_heads + head0 + i / D) * D + i % D] = 0.f;
    return;
  }
  const int ntiles = (c1 - c0 + C::TP - 1) / C::TP;

  // ---- shared memory: [stages][p buffers][barriers], stage base 1024-byte aligned
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  float* psbuf = reinterpret_cast<float*>(stages + C::NST * C::STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::NST * C::STAGE_BYTES + C::PS_BYTES);
  uint64_t* empty = full + C::NST;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], K == Kind::F16 ? 1 : 64);
      mbar_init(&empty[i], ncw);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == ncw) {  // ---- producer warp
    if constexpr (K == Kind::F16) {
      if (lane == 0)
        produce_tma<C>(&tmK, &tmV, stages, full, empty, ntiles, g,
                       s * static_cast<int>(p.cache_cap) + c0, p.err);
    } else {
      produce_gather<C, D>(p, stages, full, empty, ntiles, t, g, s, L, c0, c1, lane);
    }
    return;
  }

  // ---- consumer warps
  const int hg = warp % nhg, slice = warp / nhg;
  const int lrow = lane / C::LPP, li = lane % C::LPP;
  constexpr int DUP = C::LPP / GW;  // lanes of a row holding the same head after the scatter
  const int hsel = li / DUP;

  float qr[C::CPL][C::DPC][GW];  // this lane's q slice, pre-scaled by scale * log2(e)
#pragma unroll
  for (int h = 0; h < GW; ++h) {
    const int hh = hg * GW + h;
    const float* qh = p.q + ((size_t)t * p.n_heads + head0 + (hh < G ? hh : 0)) * D;
#pragma unroll
    for (int k = 0; k < C::CPL; ++k) {
      const int d0 = (li + k * C::LPP) * C::DPC;
#pragma unroll
      for (int e = 0; e < C::DPC; e += 4) {
        float4 x = __ldg(reinterpret_cast<const float4*>(qh + d0 + e));
        const float f = hh < G ? p.scale_log2 : 0.f;
        qr[k][e][h] = x.x * f;
        qr[k][e + 1][h] = x.y * f;
        qr[k][e + 2][h] = x.z * f;
        qr[k][e + 3][h] = x.w * f;
      }
    }
  }

  float m_run = -INFINITY, l_run = 0.f;
  float acc[C::DPL][GW];
#pragma unroll
  for (int d = 0; d < C::DPL; ++d)
#pragma unroll
    for (int h = 0; h < GW; ++h) acc[d][h] = 0.f;
  float* ps = psbuf + warp * C::TPW * GW;
  const int rbase = slice * C::TPW;
  const int pv_byte = lane * C::DPL * C::ESZ;  // this lane's p.v slice within a row
  const int pv_ch = pv_byte / 16, pv_off = pv_byte % 16;
  bool ok = true;

  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::NST;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (i / C::NST) & 1));
    if (!ok) break;
    const uint8_t* sk = stages + st * C::STAGE_BYTES;
    const uint8_t* sv = sk + C::NBOX * C::BOX_BYTES;
    const __half* skc = reinterpret_cast<const __half*>(sk + C::KV_BYTES);
    const __half* svc = skc + C::TP * C::NSC;
    const int* rowok = reinterpret_cast<const int*>(sk + C::KV_BYTES + C::SC_BYTES);
    const int nvw = min(max(c1 - (c0 + i * C::TP + rbase), 0), C::TPW);  // valid rows, a prefix
    if (nvw > 0) {
      // -- scores x * log2(e) for head hsel of the rows of this pass
      float sc[C::NP];
#pragma unroll
      for (int pp = 0; pp < C::NP; ++pp) {
        const int r = rbase + pp * C::RPP + lrow;
        float v[C::CPL][GW];
#pragma unroll
        for (int k = 0; k < C::CPL; ++k) {
          const int ch = li + k * C::LPP;
          const uint4 u = *reinterpret_cast<const uint4*>(sk + swz_off(r, ch, C::TP));
          float kf[C::DPC];
          cvt_chunk(u, kf);
#pragma unroll
          for (int h = 0; h < GW; ++h) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < C::DPC; ++e) a = fmaf(qr[k][e][h], kf[e], a);
            v[k][h] = a;
          }
          if constexpr (K == Kind::Q8) {  // qsa_attn3's factoring: scale the group's partial dot
            const float ks = __half2float(skc[r * C::NSC + ((ch * C::DPC) >> p.sc_shift)]);
#pragma unroll
            for (int h = 0; h < GW; ++h) v[k][h] *= ks;
          }
        }
        float tot[GW];
#pragma unroll
        for (int h = 0; h < GW; ++h) {
          tot[h] = v[0][h];
#pragma unroll
          for (int k = 1; k < C::CPL; ++k) tot[h] += v[k][h];
        }
        reduce_scatter<GW, C::LPP>(tot, lane);
        bool valid = (pp * C::RPP + lrow) < nvw;
        if constexpr (K == Kind::Q8) valid = valid && rowok[r] != 0;
        sc[pp] = valid ? tot[0] : -INFINITY;
      }
      // -- online softmax for head hsel over this slice (flash_attention.metal's tile step)
      float mt = sc[0];
#pragma unroll
      for (int pp = 1; pp < C::NP; ++pp) mt = fmaxf(mt, sc[pp]);
#pragma unroll
      for (int mask = C::LPP; mask < 32; mask <<= 1)
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, mask));
      const float m_new = fmaxf(m_run, mt);
      // every row masked so far (only possible with skipped ids): keep the state empty rather
      // than form -inf - -inf; otherwise the first tile gives corr = exp2(-inf) = 0
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float corr = fast_exp2(m_run - m_use);
      float lsum = 0.f;
#pragma unroll
      for (int pp = 0; pp < C::NP; ++pp) {
        sc[pp] = fast_exp2(sc[pp] - m_use);
        lsum += sc[pp];
      }
#pragma unroll
      for (int mask = C::LPP; mask < 32; mask <<= 1)
        lsum += __shfl_xor_sync(0xffffffffu, lsum, mask);
      l_run = fmaf(l_run, corr, lsum);
      m_run = m_new;
      if (li % DUP == 0) {
#pragma unroll
        for (int pp = 0; pp < C::NP; ++pp) ps[(pp * C::RPP + lrow) * GW + hsel] = sc[pp];
      }
      float cr[GW];
#pragma unroll
      for (int h = 0; h < GW; ++h) cr[h] = __shfl_sync(0xffffffffu, corr, h * DUP);
      __syncwarp();
#pragma unroll
      for (int d = 0; d < C::DPL; ++d)
#pragma unroll
        for (int h = 0; h < GW; ++h) acc[d][h] *= cr[h];
      // -- p.v over the valid rows of the slice
#pragma unroll 2
      for (int j = 0; j < nvw; ++j) {
        const int r = rbase + j;
        float vf[C::DPL];
        load_pv<K, C::DPL>(sv + swz_off(r, pv_ch, C::TP) + pv_off, vf);
        float pj[GW];
        if constexpr (GW == 4) {
          const float4 x = *reinterpret_cast<const float4*>(ps + j * 4);
          pj[0] = x.x; pj[1] = x.y; pj[2] = x.z; pj[3] = x.w;
        } else {
#pragma unroll
          for (int h = 0; h < GW; ++h) pj[h] = ps[j * GW + h];
        }
        if constexpr (K == Kind::Q8) {
          const float vs = __half2float(svc[r * C::NSC + (pv_byte >> p.sc_shift)]);
#pragma unroll
          for (int h = 0; h < GW; ++h) pj[h] *= vs;
        }
#pragma unroll
        for (int d = 0; d < C::DPL; ++d)
#pragma unroll
          for (int h = 0; h < GW; ++h) acc[d][h] = fmaf(pj[h], vf[d], acc[d][h]);
      }
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (!ok && lane == 0) flag_error(p.err, GQA_ERR_TIMEOUT);

  // ---- merge the row slices of each head group (log-sum-exp, qsa_merge2's rule) and write
  named_bar_sync(1, ncw * 32);  // every consumer is past its last stage: reuse them
  float* mg = reinterpret_cast<float*>(stages);  // [ncw][GW][D + 2]
  float* mw = mg + warp * GW * (D + 2);
#pragma unroll
  for (int d = 0; d < C::DPL; ++d)
#pragma unroll
    for (int h = 0; h < GW; ++h) mw[h * (D + 2) + lane * C::DPL + d] = acc[d][h];
  if (lrow == 0 && li % DUP == 0) {
    mw[hsel * (D + 2) + D] = m_run;
    mw[hsel * (D + 2) + D + 1] = l_run;
  }
  named_bar_sync(1, ncw * 32);
  for (int idx = threadIdx.x; idx < nhg * GW * D; idx += ncw * 32) {
    const int d = idx % D, h = (idx / D) % GW, hg2 = idx / (GW * D);
    const int hh = hg2 * GW + h;
    if (hh >= G) continue;
    float M = -INFINITY;
#pragma unroll
    for (int q2 = 0; q2 < NPS; ++q2) M = fmaxf(M, mg[((q2 * nhg + hg2) * GW + h) * (D + 2) + D]);
    float A = 0.f, Ls = 0.f;
#pragma unroll
    for (int q2 = 0; q2 < NPS; ++q2) {
      const float* rr = mg + ((q2 * nhg + hg2) * GW + h) * (D + 2);
      const float e = rr[D] == -INFINITY ? 0.f : fast_exp2(rr[D] - M);
      A = fmaf(rr[d], e, A);
      Ls = fmaf(rr[D + 1], e, Ls);
    }
    const int head = head0 + hh;
    if (p.merge) {
      float* pr = p.part + (((size_t)t * p.n_split + c) * p.n_heads + head) * (D + 2);
      pr[d] = A;
      if (d == 0) {
        pr[D] = M == -INFINITY ? -INFINITY : M * kLn2;  // natural-log units
        pr[D + 1] = Ls;
      }
    } else {
      p.out[((size_t)t * p.n_heads + head) * D + d] = gated(p, t, head, d, Ls > 0.f ? A / Ls : 0.f);
    }
  }
  if (p.merge)
    merge_if_last<D>(p, t, head0, G, (size_t)t * gridDim.y + blockIdx.y,
                     (nsel + p.chunk - 1) / p.chunk, ncw);
}

}  // namespace gqa
