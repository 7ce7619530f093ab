// partial_mma_q8.cuh -- split-KV decode-attention partial kernel for int8 caches on the tensor
// cores (dense, or through a selected-cell id list).
//
// The CTA structure, the gather producer and the staged layout are those of the CUDA-core int8
// kernel (partial_kernel.cuh: rows gathered by cp.async into 128-byte swizzled boxes, the rows'
// f16 scales and flags beside them); the contractions are those of the f16 tensor-core kernel
// (partial_mma.cuh: mma.sync m16n8k16, q and the weights as f16 hi + lo rows), with two
// int8-specific steps:
//
//   * Exact f16 of an int8.  |v| <= 127, so v is an f16 integer.  Four code bytes x (v + 128,
//     one xor) are spread into the low bytes of f16 words whose high byte is 0x64 (a byte
//     permute): 0x64xx is 1024 + x; one f16x2 subtraction of 1152 leaves v.
//   * Scales (qsa2.metal, qsa_attn2 / qsa_attn3: one f16 scale per 64 -- or 32 -- dims of a
//     row).  q.k: the k-steps of every 32 dims accumulate into a fresh accumulator, which is
//     multiplied by each position's scale of the group holding them and added to the scores,
//     as qsa_attn3 factors the scale out of a group's partial dot.  p.v: a position's V scale of a group is
//     folded into its weight, so the weights fed to the MMAs of a group's output dims are
//     p_j * vscale_j,g (hi + lo parts).
//
// Fragment layout.  For q.k (A = q: up to 8 heads as hi rows 0-7 and lo rows 8-15; B = K^T) the
// k index is permuted within every 16-dim step: a thread's B registers (k 2t, 2t+1 and 2t+8,
// 2t+9 of position g) are dims 4t .. 4t+3, one 32-bit shared load, and q's A fragments are laid
// out the same way.  For p.v (A = the weights, B = V with k = positions, n = dims) the four
// n-tiles of a 32-dim block take dims 4n + t (n-tile t, column n): a thread's 32-bit load of a
// position's bytes 4n .. 4n+3 serves all four n-tiles.
#pragma once

#include "partial_mma.cuh"

namespace gqa {

template <int D, int NHG>
struct MmaQ8Cfg {
  // the staged layout of produce_gather (partial_kernel.cuh)
  static constexpr int RB = D, CPR = RB / 16, NBOX = (RB + 127) / 128;
  static constexpr int TP = D == 256 ? 64 : 128;  // rows per stage
  static constexpr int NST = 3;
  static constexpr int NSC = D / 32;              // staged scale slots per row (32-dim groups)
  static constexpr int BOX_BYTES = TP * 128;
  static constexpr int KV_BYTES = 2 * NBOX * BOX_BYTES;
  static constexpr int SC_BYTES = align_up(2 * TP * NSC * 2, 16);
  static constexpr int OK_BYTES = align_up(TP * 4, 16);
  static constexpr int STAGE_BYTES = align_up(KV_BYTES + SC_BYTES + OK_BYTES, 1024);
  // consumers: at most 8 warps (with ~200 registers a thread, 9 warps fill the register file)
  static constexpr int DSPLIT = D == 256 ? 2 : 1;  // warps sharing a head group's output dims
  static constexpr int NPS = NHG * DSPLIT > 2 ? 2 : 4;  // row slices of a stage
  static constexpr int TPW = TP / NPS;             // rows per warp per stage
  static constexpr int NB16 = TPW / 16;
  static constexpr int DW = D / DSPLIT;
  static constexpr int NJ = DW / 32;               // 32-dim blocks of p.v per warp
  static constexpr int KS = D / 16;
  static constexpr int NCW = NPS * NHG * DSPLIT;
  // gather warps: two share a tile's rows (GB300, 1024 selected cells: a 64-row tile's copies
  // go out in ~1.3 us either way -- the SM's bytes in flight bound them -- and two warps take
  // ~0.2 us off the first)
  static constexpr int NPW = 2;
  static constexpr int MAX_THREADS = 32 * (NCW + NPW);
  static constexpr int MERGE_BYTES = NPS * NHG * 8 * (D + 2) * 4;
  // at D = 256 q's A fragments live in shared memory ([head group][k-step][lane] x 16 bytes),
  // not in 64 registers a thread
  static constexpr bool QSMEM = D == 256;
  static constexpr int QF_OFF = align_up(NST * STAGE_BYTES + 2 * NST * 8, 16);
  static constexpr int QF_BYTES = QSMEM ? NHG * KS * 32 * 16 : 0;
  // D = 256: the two warps of a pair (same rows and heads, output dims split) each contract
  // half of q.k and swap their partial scores: [pair][buffer][dh][lane] x float4
  static constexpr int NPAIR = NPS * NHG;
  static constexpr int GPW = KS / 4 / DSPLIT;  // 64-dim q.k groups per warp
  static constexpr int XC_OFF = QF_OFF + QF_BYTES;
  static constexpr int XC_BYTES = DSPLIT > 1 ? NPAIR * 2 * DSPLIT * 32 * 16 : 0;
  static constexpr int SMEM_BYTES = 1024 + XC_OFF + XC_BYTES;
  // a cluster-merged row: this CTA's partial [head][D + 2] (acc | m | l), beside the merge area
  static constexpr int CP_OFF = align_up(MERGE_BYTES, 16);
  static constexpr int CP_BYTES = NHG * 8 * (D + 2) * 4;
  static constexpr int MAX_CLUSTER = 8;
  static constexpr float RESCALE_LOG2 = 8.f;
  static_assert(CP_OFF + CP_BYTES <= NST * STAGE_BYTES, "cluster partial inside the stages");
  static_assert(TPW % 16 == 0, "whole 16-row blocks per warp");
  static_assert(DSPLIT <= 2 && 2 + NPAIR <= 16, "one named barrier per warp pair");
  static_assert(MERGE_BYTES <= NST * STAGE_BYTES, "merge area aliases the stages");
};

// Four int8 codes (v + 128 as bytes of x) -> the f16x2 pairs (v0, v1) and (v2, v3), exact.
__device__ __forceinline__ void i8x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const uint32_t a = __byte_perm(x, 0x64646464u, 0x4140);  // (1024 + x0, 1024 + x1)
  const uint32_t b = __byte_perm(x, 0x64646464u, 0x4342);  // (1024 + x2, 1024 + x3)
  lo = h2_bits(__hsub2(*reinterpret_cast<const __half2*>(&a), off));
  hi = h2_bits(__hsub2(*reinterpret_cast<const __half2*>(&b), off));
}

// Bytes t of (x, y) -> the f16x2 (x.t - 128, y.t - 128), exact: codes stored as v + 128.
__device__ __forceinline__ uint32_t i8_pair_to_f16(uint32_t xy, int sel) {
  const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const uint32_t a = __byte_perm(xy, 0x64646464u, sel);
  return h2_bits(__hsub2(*reinterpret_cast<const __half2*>(&a), off));
}

template <int D, int NHG>
__global__ void __launch_bounds__(MmaQ8Cfg<D, NHG>::MAX_THREADS, 1)
    partial_mma_q8_kernel(const PartialParams p) {
  using C = MmaQ8Cfg<D, NHG>;
  extern __shared__ uint8_t smem_raw[];
  const int c = blockIdx.x, t = blockIdx.z;
  const int g = blockIdx.y / p.head_split;        // KV head
  const int G = p.group / p.head_split;           // query heads served by this CTA (<= 8 NHG)
  const int head0 = g * p.group + (blockIdx.y % p.head_split) * G;  // its first query head
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the row's chunk CTAs merge inside their cluster (only when the launch made one of them)
  const bool clus = p.cluster > 1 && cluster_nctarank() == static_cast<uint32_t>(p.cluster);
  if (p.pdl) {
    // launched as a programmatic dependent of the previous kernel on the stream (e.g. the
    // top-k selection that writes ids): wait for its completion and memory before touching
    // global memory; the next such launch may be scheduled from here on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
  }

  // ---- the first tile's visited-list entries, loaded by the producer warp beside the row's
  //      length rather than after it (any chunk's entries lie below min(chunk end, budget))
  constexpr int RPL = C::TP / 32 / C::NPW;
  int first[RPL];
  const int pw = warp - C::NCW;  // gather warp index (consumers: negative)
  const bool pre = pw >= 0 && p.ids != nullptr;
  if (pre) {
    const int j0 = c * p.chunk, lim = min(j0 + p.chunk, p.budget);
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int j = j0 + lane + 32 * (pw + C::NPW * k);
      first[k] = j < lim ? __ldg(p.ids + (size_t)t * p.budget + j) : 0;
    }
  }

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
  const int nchunks = (nsel + p.chunk - 1) / p.chunk;
  const int c0 = c * p.chunk;
  const int c1 = min(c0 + p.chunk, nsel);
  if (c == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    if (errbits) flag_error(p.err, errbits);
    if (p.merge) p.n_valid[t] = nchunks;
  }
  if (c0 >= nsel) {
    if (c == 0)  // empty context: zeros (flash_attention.metal, seq_len == 0), split or not
      for (int i = threadIdx.x; i < G * D; i += blockDim.x)
        p.out[((size_t)t * p.n_heads + head0 + i / D) * D + i % D] = 0.f;
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
      mbar_init(&full[i], 64 * C::NPW);  // per gather lane: an arrival and a cp.async one
      mbar_init(&empty[i], C::NCW);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (pw >= 0) {  // ---- gather warps
    produce_gather<C, D, C::NPW>(p, stages, full, empty, ntiles, t, g, s, L, c0, c1, lane,
                                 pre ? first : nullptr, pw);
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
  const int sh = p.sc_shift;    // dims per scale: 1 << sh (64 or 32)

  // A fragments of q: hi in rows 0-7, lo in rows 8-15, permuted k; in registers, or (D = 256)
  // built once per head group into shared memory and read back per k-step
  uint32_t qa[C::QSMEM ? 1 : C::KS][4];
  uint4* qf = reinterpret_cast<uint4*>(stages + C::QF_OFF) + hg * C::KS * 32 + lane;
  if (!C::QSMEM || (slice == 0 && dh == 0)) {
    const float* qrow = p.q + ((size_t)t * p.n_heads + head0 + (hv ? hh : 0)) * D;
    const float f = hv ? p.scale_log2 : 0.f;
#pragma unroll
    for (int ks = 0; ks < C::KS; ++ks) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(qrow + ks * 16 + 4 * tig));
      uint32_t a[4];
      split_hi_lo(x.x * f, x.y * f, a[0], a[1]);
      split_hi_lo(x.z * f, x.w * f, a[2], a[3]);
      if constexpr (C::QSMEM) {
        qf[ks * 32] = make_uint4(a[0], a[1], a[2], a[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) qa[ks][e] = a[e];
      }
    }
  }
  if constexpr (C::QSMEM) named_bar_sync(1, C::NCW * 32);  // the fragments are written

  float o[C::NJ * 4][4];
#pragma unroll
  for (int n = 0; n < C::NJ * 4; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // head hh; l_run over this thread's positions
  bool ok = true;
  float4* xc = reinterpret_cast<float4*>(stages + C::XC_OFF) +
               (slice * NHG + hg) * 2 * C::DSPLIT * 32 + lane;

  for (int i = 0; i < ntiles; ++i) {
    const int st = i % C::NST;
    // after a timeout the warp runs on without waiting, so that both warps of a pair keep
    // meeting at their barrier; the error word marks the result
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (i / C::NST) & 1));
    const uint8_t* sk = stages + st * C::STAGE_BYTES;
    const uint8_t* sv = sk + C::NBOX * C::BOX_BYTES;
    const __half* skc = reinterpret_cast<const __half*>(sk + C::KV_BYTES);
    const __half* svc = skc + C::TP * C::NSC;
    const int* rowok = reinterpret_cast<const int*>(sk + C::KV_BYTES + C::SC_BYTES);
#pragma unroll
    for (int b = 0; b < C::NB16; ++b) {
      const int r0 = slice * C::TPW + b * 16;
      const int nv = min(max(c1 - (c0 + i * C::TP + r0), 0), 16);  // valid rows, a prefix
      if (nv == 0) continue;  // the same for both warps of a pair
      // -- partial scores of positions r0 + 8 nt + 2 tig + j over this warp's 64-dim groups:
      //    per 32 dims a fresh accumulator, times the positions' K scale of the group holding
      //    those dims (a 64-dim scale group's two halves take the same scale)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int gq = 0; gq < C::GPW; ++gq) {
        const int gb = (dh * C::GPW + gq) * 4;  // first k-step of the group
        float acc[2][2][4];  // [32-dim half][n-tile][c]
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) acc[u][nt][0] = acc[u][nt][1] = acc[u][nt][2] = acc[u][nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int ks = gb + kk, u = kk / 2;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(
                sk + swz_off(r0 + nt * 8 + gid, ks, C::TP) + 4 * tig);
            uint32_t b0, b1;
            i8x4_to_f16(w ^ 0x80808080u, b0, b1);
            if constexpr (C::QSMEM) {
              const uint4 a4 = qf[ks * 32];
              const uint32_t a[4] = {a4.x, a4.y, a4.z, a4.w};
              mma_f16(acc[u][nt], a, b0, b1);
            } else {
              mma_f16(acc[u][nt], qa[ks], b0, b1);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int ra = r0 + nt * 8 + 2 * tig;
          if (sh == 6) {  // one scale for the 64 dims
            const int slot = gb >> 2;
            const float s0 = __half2float(skc[ra * C::NSC + slot]);
            const float s1 = __half2float(skc[(ra + 1) * C::NSC + slot]);
            sc[nt][0] = fmaf(acc[0][nt][0] + acc[1][nt][0], s0, sc[nt][0]);
            sc[nt][1] = fmaf(acc[0][nt][1] + acc[1][nt][1], s1, sc[nt][1]);
            sc[nt][2] = fmaf(acc[0][nt][2] + acc[1][nt][2], s0, sc[nt][2]);
            sc[nt][3] = fmaf(acc[0][nt][3] + acc[1][nt][3], s1, sc[nt][3]);
          } else {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int slot = (gb >> 1) + u;  // 32-dim groups
              const float s0 = __half2float(skc[ra * C::NSC + slot]);
              const float s1 = __half2float(skc[(ra + 1) * C::NSC + slot]);
              sc[nt][0] = fmaf(acc[u][nt][0], s0, sc[nt][0]);
              sc[nt][1] = fmaf(acc[u][nt][1], s1, sc[nt][1]);
              sc[nt][2] = fmaf(acc[u][nt][2], s0, sc[nt][2]);
              sc[nt][3] = fmaf(acc[u][nt][3], s1, sc[nt][3]);
            }
          }
        }
      }
      // -- head hh's scores: hi row + lo row, plus the partner warp's half of the dims
      float xs[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) xs[nt][j] = sc[nt][j] + sc[nt][2 + j];
      if constexpr (C::DSPLIT > 1) {
        const int buf = (i * C::NB16 + b) & 1;  // two buffers: a write never meets a late read
        xc[(buf * C::DSPLIT + dh) * 32] = make_float4(xs[0][0], xs[0][1], xs[1][0], xs[1][1]);
        named_bar_sync(2 + slice * NHG + hg, 64);
        const float4 y = xc[(buf * C::DSPLIT + (dh ^ 1)) * 32];
        // the same order of addition in both warps: identical scores, identical weights
        const bool first = dh == 0;
        xs[0][0] = first ? xs[0][0] + y.x : y.x + xs[0][0];
        xs[0][1] = first ? xs[0][1] + y.y : y.y + xs[0][1];
        xs[1][0] = first ? xs[1][0] + y.z : y.z + xs[1][0];
        xs[1][1] = first ? xs[1][1] + y.w : y.w + xs[1][1];
      }
      // -- rows past the chunk or with a bad id: -inf
      float x[2][2];
      float mt = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int rr = nt * 8 + 2 * tig + j;
          const bool valid = rr < nv && rowok[r0 + rr] != 0;
          x[nt][j] = valid ? xs[nt][j] : -INFINITY;
          mt = fmaxf(mt, x[nt][j]);
        }
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      // -- lazy online-softmax update; a head with no valid position yet keeps an empty state
      const bool grow = mt > m_run + C::RESCALE_LOG2;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? mt : m_run;
        const float corr = m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_new);
        m_run = m_new;
        l_run *= corr;
#pragma unroll
        for (int n = 0; n < C::NJ * 4; ++n) {
          o[n][0] *= corr;
          o[n][1] *= corr;
          o[n][2] *= corr;
          o[n][3] *= corr;
        }
      }
      const float mu = m_run == -INFINITY ? 0.f : m_run;
      float pr[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          pr[nt][j] = fast_exp2(x[nt][j] - mu);  // 0 for masked rows
          l_run += pr[nt][j];
        }
      // -- O += P_g . V over this warp's dims, 32-dim block by block; P_g = p * vscale_g,
      //    formed again only where the scale group changes
      const int ra = r0 + 2 * tig;  // this thread's weight rows: ra, ra + 1, ra + 8, ra + 9
      uint32_t pa[4];
      int pslot = -1;
#pragma unroll
      for (int j = 0; j < C::NJ; ++j) {
        const int d0 = dh * C::DW + 32 * j;  // the block's first dim
        const int slot = d0 >> sh;
        if (slot != pslot) {
          pslot = slot;
          const float v0 = __half2float(svc[ra * C::NSC + slot]);
          const float v1 = __half2float(svc[(ra + 1) * C::NSC + slot]);
          const float v8 = __half2float(svc[(ra + 8) * C::NSC + slot]);
          const float v9 = __half2float(svc[(ra + 9) * C::NSC + slot]);
          // masked rows have weight 0; their scale may be anything (selected away)
          split_hi_lo(pr[0][0] > 0.f ? pr[0][0] * v0 : 0.f, pr[0][1] > 0.f ? pr[0][1] * v1 : 0.f,
                      pa[0], pa[1]);
          split_hi_lo(pr[1][0] > 0.f ? pr[1][0] * v8 : 0.f, pr[1][1] > 0.f ? pr[1][1] * v9 : 0.f,
                      pa[2], pa[3]);
        }
        // V bytes 4 gid .. 4 gid + 3 of the block at rows ra, ra + 1, ra + 8, ra + 9
        const int ch = (d0 >> 4) + (gid >> 2), bo = 4 * (gid & 3);
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(sv + swz_off(ra, ch, C::TP) + bo);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(sv + swz_off(ra + 1, ch, C::TP) + bo);
        const uint32_t wc = *reinterpret_cast<const uint32_t*>(sv + swz_off(ra + 8, ch, C::TP) + bo);
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(sv + swz_off(ra + 9, ch, C::TP) + bo);
        // byte t of two rows side by side: (ra.t, ra1.t, ...) for t = 0, 1 and 2, 3
        const uint32_t ab01 = __byte_perm(wa, wb, 0x5140) ^ 0x80808080u;
        const uint32_t ab23 = __byte_perm(wa, wb, 0x7362) ^ 0x80808080u;
        const uint32_t cd01 = __byte_perm(wc, wd, 0x5140) ^ 0x80808080u;
        const uint32_t cd23 = __byte_perm(wc, wd, 0x7362) ^ 0x80808080u;
        // rows past the chunk end hold whatever was staged (finite codes): their weights are 0
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          const uint32_t xab = tt < 2 ? ab01 : ab23, xcd = tt < 2 ? cd01 : cd23;
          const int sel = (tt & 1) ? 0x4342 : 0x4140;
          mma_f16(o[j * 4 + tt], pa, i8_pair_to_f16(xab, sel), i8_pair_to_f16(xcd, sel));
        }
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
  for (int j = 0; j < C::NJ; ++j)
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      // n-tile (j, tt), column n = 2 tig (+1): dim d0 + 4 n + tt
      const int d = dh * C::DW + 32 * j + 8 * tig + tt;
      mrow[d] = o[j * 4 + tt][0] + o[j * 4 + tt][2];
      mrow[d + 4] = o[j * 4 + tt][1] + o[j * 4 + tt][3];
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
    const int head = head0 + h2;
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
    cluster_merge<D, C::MAX_CLUSTER>(p, t, head0, G, c, nchunks, stages + C::CP_OFF, C::NCW);
    return;
  }
  if (p.merge)
    merge_if_last<D>(p, t, head0, G, (size_t)t * gridDim.y + blockIdx.y, nchunks, C::NCW);
}

// Launches the kernel, as a programmatic dependent when p.pdl.  A split row whose chunks fit one
// cluster (2 .. 8 CTAs) goes out as clusters of its chunk CTAs, which merge in distributed
// shared memory (no partial records, no arrival counters), unless GQA_Q8_CLUSTER=0 or the GPU
// cannot hold such a cluster.
template <int D, int NHG>
cudaError_t launch_mma_q8(PartialParams p, dim3 grid, cudaStream_t s) {
  using C = MmaQ8Cfg<D, NHG>;
  auto kern = &partial_mma_q8_kernel<D, NHG>;
  const void* fn = reinterpret_cast<const void*>(kern);
  cudaError_t e = ensure_smem(fn, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::MAX_THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  const bool want = p.merge && grid.x > 1 && grid.x <= static_cast<unsigned>(C::MAX_CLUSTER) &&
                    q8_cluster_merge();
  p.cluster = want && cluster_fits<C::MAX_CLUSTER>(fn, cfg, grid.x) ? static_cast<int>(grid.x) : 0;
  cfg.attrs = at;
  cfg.numAttrs = cluster_attrs(at, p.cluster, p.pdl);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace gqa
