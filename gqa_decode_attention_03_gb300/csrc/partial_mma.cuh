// partial_mma.cuh -- split-KV decode-attention partial kernel for f16 caches on the tensor cores.
//
// Same CTA structure, TMA producer, stage ring, partial format, end-of-chunk merge and fused
// last-CTA merge as partial_kernel (see partial_kernel.cuh), but q.k^T and p.v run as
// mma.sync m16n8k16 with f32 accumulation instead of fp32 FMA: the CUDA-core kernel is
// issue-bound (about 64 warp instructions per position and KV head), this one needs about 14.
//
// Exactness.  K and V are f16 already, so they enter the MMA unchanged.  q (fp32, pre-scaled by
// scale * log2 e) and p (fp32 probabilities) are each split into an f16 "hi" part and an f16 "lo"
// remainder; products of f16 values are exact in fp32, so the split carries about 22 mantissa
// bits of q and p through the contraction.
//
// Fragment layout (per warp, 16 cache positions per block).  The A operand's 16 rows are the
// warp's up-to-8 query heads twice: rows 0-7 hold the hi parts, rows 8-15 the lo parts, so a
// thread's accumulator registers c0/c1 (row gid) and c2/c3 (row gid + 8) hold the two halves of
// the same head and recombine without a shuffle.
//   S = Q . K^T    A = Q (16 x 16 dims), B = K^T read by ldmatrix from the swizzled K tile,
//                  C = scores for 8 positions; two n-tiles per block.
//   O += P . V     A = P, built in registers from the score accumulators (hi rows 0-7, lo rows
//                  8-15), B = V read by ldmatrix.trans, C = O for 8 dims per n-tile.
// The online softmax (flash_attention.metal's running max / sum / correction) rescales lazily:
// the running max only moves when a block's max exceeds it by more than 2^8, so p <= 256 and
// most blocks skip the rescale of O.  Rows past the chunk end are masked by selection: their
// scores become -inf and their V fragment halves are zeroed in registers, so cache garbage past
// a sequence's length never reaches the output.
#pragma once

#include "partial_kernel.cuh"

namespace gqa {

template <int D, int NHG>
struct MmaCfg {
  static constexpr int NBOX = D / 64;                         // 128-byte boxes per f16 row
  static constexpr int TP = D == 64 ? 128 : (D == 128 ? 64 : 32);
  static constexpr int NPS = D == 256 ? 2 : 4;                // row slices per stage
  static constexpr int TPW = TP / NPS;                        // rows per warp per stage
  static constexpr int NB16 = TPW / 16;                       // 16-row blocks per warp per stage
  static constexpr int DSPLIT = D == 256 ? 2 : 1;             // warps sharing one O (by dims)
  static constexpr int DW = D / DSPLIT;                       // O dims per warp
  static constexpr int NT = DW / 8;                           // O n-tiles per warp
  static constexpr int KS = D / 16;                           // k-steps of q.k
  static constexpr int NST = 3;
  static constexpr int BOX_BYTES = TP * 128;
  static constexpr int KV_BYTES = 2 * NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = KV_BYTES;
  static constexpr int NCW = NHG * DSPLIT * NPS;              // consumer warps
  static constexpr int MAX_THREADS = 32 * (NCW + 1);
  static constexpr int MIN_BLOCKS = NHG == 1 ? 2 : 1;
  static constexpr int MERGE_BYTES = NPS * NHG * 8 * (D + 2) * 4;
  static constexpr int SMEM_BYTES = 1024 + NST * STAGE_BYTES + 2 * NST * 8;
  static constexpr float RESCALE_LOG2 = 8.f;                  // lazy-rescale threshold
  // a cluster-merged row: this CTA's partial [head][D + 2] (acc | m | l), beside the merge area
  static constexpr int CP_OFF = align_up(MERGE_BYTES, 16);
  static constexpr int CP_BYTES = NHG * 8 * (D + 2) * 4;
  static constexpr int MAX_CLUSTER = 8;
  static_assert(TPW % 16 == 0, "whole 16-row blocks per warp");
  static_assert(MERGE_BYTES <= NST * STAGE_BYTES, "merge area aliases the stages");
  static_assert(CP_OFF + CP_BYTES <= NST * STAGE_BYTES, "cluster partial inside the stages");
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// Not volatile: the MMA has no side effect beyond its outputs, so the compiler may schedule
// independent work (softmax math of another block) around it.
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// (a, b) -> f16x2 hi = round(a, b) and lo = round((a, b) - hi); low half holds a.
__device__ __forceinline__ void split_hi_lo(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  hi = h2_bits(h);
  lo = h2_bits(__floats2half2_rn(a - hf.x, b - hf.y));
}

template <int D, int NHG>
__global__ void __launch_bounds__(MmaCfg<D, NHG>::MAX_THREADS, MmaCfg<D, NHG>::MIN_BLOCKS)
    partial_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const PartialParams p) {
  using C = MmaCfg<D, NHG>;
  extern __shared__ uint8_t smem_raw[];
  const int c = blockIdx.x, g = blockIdx.y;
  const int t = blockIdx.z;
  // the row's chunk CTAs merge inside their cluster (only when the launch made one of them)
  const bool clus = p.cluster > 1 && cluster_nctarank() == static_cast<uint32_t>(p.cluster);
  if (p.pdl) {
    // launched as a programmatic dependent of the previous kernel on the stream: wait for its
    // completion and memory before touching global memory, and let the next such launch be
    // scheduled as soon as this grid's CTAs start retiring
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
  }
  const int G = p.group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- the row's visited positions (uniform over the CTA)
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
  // the row's chunks: ceil(L / chunk) of them, of p.chunk positions each (the last one shorter)
  const int nchunks = (L + p.chunk - 1) / p.chunk;
  const int c0 = c * p.chunk;
  const int c1 = min(c0 + p.chunk, L);
  if (c == 0 && g == 0 && threadIdx.x == 0) {
    if (errbits) flag_error(p.err, errbits);
    if (p.merge) p.n_valid[t] = nchunks;
  }
  if (c0 >= L) {
    if (c == 0)  // empty context: zeros (flash_attention.metal, seq_len == 0), split or not
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        p.out[((size_t)t * p.n_heads + g * G + i / D) * D + i % D] = 0.f;
    if (clus) {  // the cluster's two barriers count every thread of every CTA
      cluster_sync();
      cluster_sync();
    }
    return;
  }
  const int ntiles = (c1 - c0 + C::TP - 1) / C::TP;

  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::NST * C::STAGE_BYTES);
  uint64_t* empty = full + C::NST;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C::NCW);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == C::NCW) {  // ---- producer warp
    if (lane == 0)
      produce_tma<C>(&tmK, &tmV, stages, full, empty, ntiles, g,
                     s * static_cast<int>(p.cache_cap) + c0, p.err);
    __syncwarp();
    if (clus) {
      cluster_sync();
      cluster_sync();
    }
    return;
  }

  // ---- consumer warps: w = (slice * NHG + hg) * DSPLIT + dh
  const int gid = lane >> 2, tig = lane & 3;
  const int dh = warp % C::DSPLIT;
  const int hg = (warp / C::DSPLIT) % NHG;
  const int slice = warp / (C::DSPLIT * NHG);
  const int hh = hg * 8 + gid;  // this thread's head within the group (rows gid and gid + 8)
  const bool hv = hh < G;

  uint32_t qa[C::KS][4];  // A fragments of q: hi in rows 0-7, lo in rows 8-15
  {
    const float* qrow = p.q + ((size_t)t * p.n_heads + g * G + (hv ? hh : 0)) * D;
    const float f = hv ? p.scale_log2 : 0.f;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const int d0 = ks * 16 + 2 * tig;
      const float2 x0 = __ldg(reinterpret_cast<const float2*>(qrow + d0));
      const float2 x1 = __ldg(reinterpret_cast<const float2*>(qrow + d0 + 8));
      split_hi_lo(x0.x * f, x0.y * f, qa[ks][0], qa[ks][1]);
      split_hi_lo(x1.x * f, x1.y * f, qa[ks][2], qa[ks][3]);
    }
  }

  float o[C::NT][4];
#pragma unroll
  for (int n = 0; n < C::NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // head hh; l_run over this thread's positions
  // ldmatrix lane roles: matrix mi = lane / 8, row rr = lane % 8 of it
  const int mi = lane >> 3, rr = lane & 7;
  bool ok = true;

  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::NST;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (i / C::NST) & 1));
    if (!ok) break;
    const uint32_t sk = smem_addr(stages + st * C::STAGE_BYTES);
    const uint32_t sv = sk + C::NBOX * C::BOX_BYTES;
#pragma unroll
    for (int b = 0; b < C::NB16; ++b) {
      const int r0 = slice * C::TPW + b * 16;
      const int nv = min(max(c1 - (c0 + i * C::TP + r0), 0), 16);  // valid rows, a prefix
      if (nv == 0) continue;
      // -- S = Q . K^T for 16 positions (two n-tiles of 8)
      // four independent accumulator chains (n-tile x k-step parity), summed after
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < C::KS; ks += 2) {
        uint32_t kb[4], kc[4];
        ldsm_x4(kb, sk + swz_off(r0 + (mi >> 1) * 8 + rr, ks * 2 + (mi & 1), C::TP));
        ldsm_x4(kc, sk + swz_off(r0 + (mi >> 1) * 8 + rr, ks * 2 + 2 + (mi & 1), C::TP));
        mma_f16(sc[0], qa[ks], kb[0], kb[1]);
        mma_f16(sc[1], qa[ks], kb[2], kb[3]);
        mma_f16(sd[0], qa[ks + 1], kc[0], kc[1]);
        mma_f16(sd[1], qa[ks + 1], kc[2], kc[3]);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
      // -- scores of head hh at positions nt*8 + 2*tig + j (hi row + lo row)
      float x[2][2];
      float mt = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float v = sc[nt][j] + sc[nt][2 + j];
          x[nt][j] = (nt * 8 + 2 * tig + j) < nv ? v : -INFINITY;
          mt = fmaxf(mt, x[nt][j]);
        }
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      // -- lazy online-softmax update (first block: m_run = -inf, corr = exp2(-inf) = 0)
      const bool grow = mt > m_run + C::RESCALE_LOG2;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? mt : m_run;
        const float corr = fast_exp2(m_run - m_new);
        m_run = m_new;
        l_run *= corr;
#pragma unroll
        for (int n = 0; n < C::NT; ++n) {
          o[n][0] *= corr;
          o[n][1] *= corr;
          o[n][2] *= corr;
          o[n][3] *= corr;
        }
      }
      float pr[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          pr[nt][j] = fast_exp2(x[nt][j] - m_run);
          l_run += pr[nt][j];
        }
      uint32_t pa[4];  // A fragments of P: hi rows 0-7, lo rows 8-15
      split_hi_lo(pr[0][0], pr[0][1], pa[0], pa[1]);
      split_hi_lo(pr[1][0], pr[1][1], pa[2], pa[3]);
      // -- O += P . V over this warp's dims
      const bool tail = nv < 16;
      const uint32_t mk0 = ((2 * tig < nv) ? 0x0000ffffu : 0u) | ((2 * tig + 1 < nv) ? 0xffff0000u : 0u);
      const uint32_t mk1 = ((2 * tig + 8 < nv) ? 0x0000ffffu : 0u) |
                           ((2 * tig + 9 < nv) ? 0xffff0000u : 0u);
#pragma unroll
      for (int np = 0; np < C::NT / 2; ++np) {
        uint32_t vb[4];
        const int chunk = (dh * C::DW + np * 16) / 8 + (mi >> 1);
        ldsm_x4_t(vb, sv + swz_off(r0 + (mi & 1) * 8 + rr, chunk, C::TP));
        if (tail) {  // rows past the chunk end: zero their V halves (they may hold NaN)
          vb[0] &= mk0;
          vb[1] &= mk1;
          vb[2] &= mk0;
          vb[3] &= mk1;
        }
        mma_f16(o[2 * np], pa, vb[0], vb[1]);
        mma_f16(o[2 * np + 1], pa, vb[2], vb[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (!ok && lane == 0) flag_error(p.err, GQA_ERR_TIMEOUT);

  // ---- per-thread l covers its own positions: sum the quad
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

  // ---- merge the row slices (log-sum-exp) and write
  named_bar_sync(1, C::NCW * 32);
  float* mg = reinterpret_cast<float*>(stages);  // [NPS][NHG][8][D + 2]
  float* mrow = mg + ((slice * NHG + hg) * 8 + gid) * (D + 2);
#pragma unroll
  for (int n = 0; n < C::NT; ++n) {
    const int d = dh * C::DW + n * 8 + 2 * tig;
    mrow[d] = o[n][0] + o[n][2];
    mrow[d + 1] = o[n][1] + o[n][3];
  }
  if (tig == 0 && dh == 0) {
    mrow[D] = m_run;
    mrow[D + 1] = l_run;
  }
  named_bar_sync(1, C::NCW * 32);
  for (int idx = threadIdx.x; idx < NHG * 8 * D; idx += C::NCW * 32) {
    const int d = idx % D, h8 = (idx / D) % 8, hg2 = idx / (8 * D);
    const int h2 = hg2 * 8 + h8;
    if (h2 >= G) continue;
    float M = -INFINITY;
#pragma unroll
    for (int q2 = 0; q2 < C::NPS; ++q2) M = fmaxf(M, mg[((q2 * NHG + hg2) * 8 + h8) * (D + 2) + D]);
    float A = 0.f, Ls = 0.f;
#pragma unroll
    for (int q2 = 0; q2 < C::NPS; ++q2) {
      const float* rr2 = mg + ((q2 * NHG + hg2) * 8 + h8) * (D + 2);
      const float e = rr2[D] == -INFINITY ? 0.f : fast_exp2(rr2[D] - M);
      A = fmaf(rr2[d], e, A);
      Ls = fmaf(rr2[D + 1], e, Ls);
    }
    const int head = g * G + h2;
    if (clus) {  // log2 units, as the cluster merge below takes them
      float* cp = reinterpret_cast<float*>(stages + C::CP_OFF) + h2 * (D + 2);
      cp[d] = A;
      if (d == 0) {
        cp[D] = M;
        cp[D + 1] = Ls;
      }
    } else if (p.merge) {
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
  if (clus) {
    cluster_merge<D, C::MAX_CLUSTER>(p, t, g * G, G, c, nchunks, stages + C::CP_OFF, C::NCW);
    return;
  }
  if (p.merge)
    merge_if_last<D>(p, t, g * G, G, (size_t)t * p.n_kv_heads + g, nchunks,
                     C::NCW);
}

// Launches the kernel, as a programmatic dependent when p.pdl.  When the host allows it
// (p.cluster != 0: a split grid that fits the GPU) and a row's chunks fit one cluster (2 .. 8),
// the chunk CTAs of a row go out as one thread-block cluster and merge in distributed shared
// memory instead of through the workspace.
template <int D, int NHG>
cudaError_t launch_mma_f16(const CUtensorMap& tk, const CUtensorMap& tv, PartialParams p,
                           dim3 grid, cudaStream_t s) {
  using C = MmaCfg<D, NHG>;
  auto kern = &partial_mma_kernel<D, NHG>;
  const void* fn = reinterpret_cast<const void*>(kern);
  cudaError_t e = ensure_smem(fn, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::MAX_THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  const bool want = p.cluster != 0 && p.merge && grid.x > 1 &&
                    grid.x <= static_cast<unsigned>(C::MAX_CLUSTER);
  p.cluster = want && cluster_fits<C::MAX_CLUSTER>(fn, cfg, grid.x) ? static_cast<int>(grid.x) : 0;
  cfg.attrs = at;
  cfg.numAttrs = cluster_attrs(at, p.cluster, p.pdl);
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace gqa
