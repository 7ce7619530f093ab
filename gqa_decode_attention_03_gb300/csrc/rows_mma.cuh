// rows_mma.cuh -- f16 decode attention for rows that share a sequence (row grouping).
//
// Several query rows often read the same cache: the rows of a causal prefill chunk (row r at
// position p attends to [0, p], flash_attention_tq.metal's per-query window), or decode rows of
// one sequence.  Served one CTA per row, each row re-reads the sequence's K/V.  Here one CTA
// serves a run of up to R consecutive rows with the same seq_of[] value: it stages every K/V
// tile of its chunk once (TMA, three-stage mbarrier ring, as in partial_mma.cuh) and all rows'
// heads read it there -- attention_gqa.metal's "load K/V once, reuse across the group",
// extended from the heads of a group to the rows of a sequence.
//
// Warps.  The A operand of a consumer warp's m16n8k16 MMAs holds 8 (row, head) pairs: rows
// 0-7 the f16 hi parts of q, rows 8-15 the lo parts (so 8 / G query rows per warp), and the warp
// walks every position of every stage.  Each thread owns one (row, head) pair: its row's own
// length masks its scores (positions at or past L_row become -inf), its online softmax is its
// own, and at the end it writes its own output or chunk partial.  V fragment halves of
// positions past the group's longest row are zeroed in registers, as cache garbage may sit
// there.  Split rows are merged afterwards by merge_kernel (one CTA per row and head): a
// group's rows bring many partials at once, too many for one last CTA to merge quickly.
//
// Rows.  The grid stays (chunks, KV heads, rows); the CTA of row t works only if t leads a
// group: groups of consecutive rows with equal seq_of[] start at every multiple of R and
// wherever seq_of[] changes.  Every other CTA exits at once.  A row keeps its own chunk count
// ceil(L / chunk) (n_valid), so a row shorter than the group's longest simply has no partials
// for the chunks past its end.
#pragma once

#include "partial_mma.cuh"

namespace gqa {

template <int D>
struct RowsCfg {
  static constexpr int NBOX = D / 64;
  static constexpr int TP = D == 64 ? 128 : 64;  // positions per stage
  static constexpr int NB16 = TP / 16;            // 16-position blocks per stage
  static constexpr int NT = D / 8;                // O n-tiles per warp
  static constexpr int KS = D / 16;               // q.k k-steps
  static constexpr int NST = 3;
  static constexpr int BOX_BYTES = TP * 128;
  static constexpr int KV_BYTES = 2 * NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = KV_BYTES;
  static constexpr int NCW = 8;                   // consumer warps: 64 (row, head) pairs
  static constexpr int MAX_THREADS = 32 * (NCW + 1);
  static constexpr int SMEM_BYTES = 1024 + NST * STAGE_BYTES + 2 * NST * 8;
  static constexpr float RESCALE_LOG2 = 8.f;
  static_assert(D == 64 || D == 128, "row grouping serves head_dim 64 and 128");
};

__device__ __forceinline__ int rows_seq(const PartialParams& p, int t) {
  return p.seq_of ? __ldg(p.seq_of + t) : t;
}

template <int D>
__global__ void __launch_bounds__(RowsCfg<D>::MAX_THREADS, 1)
    partial_mma_rows_kernel(const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const PartialParams p) {
  using C = RowsCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_len[64];  // clamped length of each row of the group
  const int c = blockIdx.x, g = blockIdx.y, t0 = blockIdx.z;
  const int G = p.group;             // 1, 2, 4 or 8
  const int rpw = 8 / G;             // rows per warp
  const int R = rpw * C::NCW;        // rows per group at most
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- is row t0 a group leader?  Groups start at every multiple of R and wherever seq_of
  //      changes, and run on while seq_of stays the same (uniform over the CTA).
  const int s = rows_seq(p, t0);
  if (t0 % R != 0 && rows_seq(p, t0 - 1) == s) return;
  int nr = 1;  // rows of this group
  while ((t0 + nr) % R != 0 && t0 + nr < p.n_tok && rows_seq(p, t0 + nr) == s) ++nr;

  // ---- the rows' lengths (clamped and flagged like the per-row kernels)
  const int lmax = static_cast<int>(p.cache_cap < p.max_kv_len ? p.cache_cap : p.max_kv_len);
  const bool seq_ok = s >= 0 && s < p.n_seq;
  if (threadIdx.x < nr) {
    int L = __ldg(p.kv_len + t0 + threadIdx.x);
    int err = 0;
    if (L < 0 || L > lmax) {
      err |= GQA_ERR_KVLEN_RANGE;
      L = L < 0 ? 0 : lmax;
    }
    if (!seq_ok) {
      err |= GQA_ERR_SEQ_RANGE;
      L = 0;
    }
    if (err && c == 0 && g == 0) flag_error(p.err, err);
    if (c == 0 && g == 0 && p.merge) p.n_valid[t0 + threadIdx.x] = (L + p.chunk - 1) / p.chunk;
    s_len[threadIdx.x] = L;
  }
  __syncthreads();
  int Lmax = 0;
  for (int j = 0; j < nr; ++j) Lmax = max(Lmax, s_len[j]);
  const int c0 = c * p.chunk;
  // empty rows: zeros, written by chunk 0 (flash_attention.metal, seq_len == 0)
  if (c == 0)
    for (int j = 0; j < nr; ++j)
      if (s_len[j] == 0)
        for (int i = threadIdx.x; i < G * D; i += blockDim.x)
          p.out[((size_t)(t0 + j) * p.n_heads + g * G + i / D) * D + i % D] = 0.f;
  if (c0 >= Lmax) return;
  const int c1 = min(c0 + p.chunk, Lmax);
  const int ntiles = (c1 - c0 + C::TP - 1) / C::TP;
  const int nw = (nr * G + 7) / 8;  // consumer warps with rows

  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::NST * C::STAGE_BYTES);
  uint64_t* empty = full + C::NST;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], nw);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == C::NCW) {  // ---- producer warp
    if (lane == 0)
      produce_tma<C>(&tmK, &tmV, stages, full, empty, ntiles, g,
                     s * static_cast<int>(p.cache_cap) + c0, p.err);
    return;
  }
  if (warp >= nw) return;  // no rows for this warp

  // ---- consumer warp: pairs (row j, head h) with j = warp * rpw + gid / G, h = gid % G
  const int gid = lane >> 2, tig = lane & 3;
  const int j = warp * rpw + gid / G, h = gid % G;
  const bool rv = j < nr;                  // this thread's pair is a real row
  const int t = t0 + (rv ? j : 0);
  const int Lr = rv ? s_len[j] : 0;        // this row's length
  const int head = g * G + h;

  uint32_t qa[C::KS][4];
  {
    const float* qrow = p.q + ((size_t)t * p.n_heads + head) * D;
    const float f = rv ? p.scale_log2 : 0.f;
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
  float m_run = -INFINITY, l_run = 0.f;
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
      const int r0 = b * 16;
      const int base = c0 + i * C::TP + r0;             // cache position of the block's row 0
      const int nv = min(max(c1 - base, 0), 16);         // rows holding data for some row
      if (nv == 0) continue;
      const int nrow = min(max(Lr - base, 0), 16);       // rows inside this thread's window
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
      float x[2][2];
      float mt = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const float v = sc[nt][jj] + sc[nt][2 + jj];
          x[nt][jj] = (nt * 8 + 2 * tig + jj) < nrow ? v : -INFINITY;
          mt = fmaxf(mt, x[nt][jj]);
        }
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      // a pair whose row ends before this block keeps mt = -inf: nothing to add
      const bool grow = mt != -INFINITY && mt > m_run + C::RESCALE_LOG2;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? mt : m_run;
        const float corr = grow ? fast_exp2(m_run - m_new) : 1.f;
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
        for (int jj = 0; jj < 2; ++jj) {
          pr[nt][jj] = m_run == -INFINITY ? 0.f : fast_exp2(x[nt][jj] - m_run);
          l_run += pr[nt][jj];
        }
      uint32_t pa[4];
      split_hi_lo(pr[0][0], pr[0][1], pa[0], pa[1]);
      split_hi_lo(pr[1][0], pr[1][1], pa[2], pa[3]);
      const bool tail = nv < 16;
      const uint32_t mk0 =
          ((2 * tig < nv) ? 0x0000ffffu : 0u) | ((2 * tig + 1 < nv) ? 0xffff0000u : 0u);
      const uint32_t mk1 =
          ((2 * tig + 8 < nv) ? 0x0000ffffu : 0u) | ((2 * tig + 9 < nv) ? 0xffff0000u : 0u);
#pragma unroll
      for (int np = 0; np < C::NT / 2; ++np) {
        uint32_t vb[4];
        ldsm_x4_t(vb, sv + swz_off(r0 + (mi & 1) * 8 + rr, np * 2 + (mi >> 1), C::TP));
        if (tail) {
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

  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

  // ---- this thread's (row, head): output, or the chunk's partial plus the row's ticket
  const bool has = rv && c0 < Lr;  // the chunk holds positions of this row
  if (!p.merge) {
    if (has) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      float* orow = p.out + ((size_t)t * p.n_heads + head) * D;
#pragma unroll
      for (int n = 0; n < C::NT; ++n) {
        const int d = n * 8 + 2 * tig;
        *reinterpret_cast<float2*>(orow + d) =
            make_float2((o[n][0] + o[n][2]) * inv, (o[n][1] + o[n][3]) * inv);
      }
    }
    return;
  }
  if (has) {
    float* pr = p.part + (((size_t)t * p.n_split + c) * p.n_heads + head) * (D + 2);
#pragma unroll
    for (int n = 0; n < C::NT; ++n) {
      const int d = n * 8 + 2 * tig;
      *reinterpret_cast<float2*>(pr + d) = make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
    }
    if (tig == 0) {
      pr[D] = m_run == -INFINITY ? -INFINITY : m_run * kLn2;  // natural-log units
      pr[D + 1] = l_run;
    }
  }
}

}  // namespace gqa
