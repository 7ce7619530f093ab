// rows_mma.cuh -- f16 decode attention for rows that share a sequence (row grouping).
//
// Several query rows often read the same cache: the rows of a causal prefill chunk (row r at
// position p attends to [0, p], flash_attention_tq.metal's per-query window), or decode rows of
// one sequence.  Served one CTA per row, each row re-reads the sequence's K/V.  Here one CTA
// serves a run of up to R consecutive rows with the same seq_of[] value: it stages every K/V
// tile of its chunk once (TMA, two-stage mbarrier ring, as in partial_mma.cuh) and all rows'
// heads read it there -- attention_gqa.metal's "load K/V once, reuse across the group",
// extended from the heads of a group to the rows of a sequence.
//
// Warps.  The A operand of a consumer warp's m16n8k16 MMAs holds 16 (row, head) pairs, q in
// f16 with the scale folded in (16 / G query rows per pair set); the softmax weights go back
// into the p.v MMAs as f16 straight from the score fragments.  (The per-row decode kernels
// carry q and the weights as f16 hi + lo pairs; this kernel is compute-bound, and single f16
// keeps its error near 3e-5, inside the f16 path's 2e-3, for half the MMAs.)  Two pair sets
// per CTA, and two warps per set, each taking half of every stage's 16-position blocks with its
// own online softmax; at the end of a chunk the second half hands its (m, l, acc) to the first
// through shared memory, which combines them.  Each thread owns two pairs (fragment rows gid
// and gid + 8): a pair's row length masks its scores (positions at or past L_row become -inf).
// V fragment halves of positions past the group's longest row are zeroed in registers, as
// cache garbage may sit there.  Split rows are merged afterwards by merge_kernel (one warp per
// row and head): a group's rows bring many partials at once, too many for one last CTA to
// merge quickly.  (Merging inside a thread-block cluster of the chunks measured slower on
// GB300: clusters of 16 CTAs could not all be resident at once.)
//
// Rows.  Groups of consecutive rows with equal seq_of[] start at every multiple of R and
// wherever seq_of[] changes.  The grid is (chunks, KV heads, slots): slot z serves groups
// z, z + slots, ..., found on the device by a warp-wide ballot over seq_of[], with the TMA ring
// running on from one group to the next.  The host sizes the slots from the row and sequence
// counts, so that no CTA is launched only to exit.  A row keeps its own chunk count
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
  static constexpr int NST = 2;
  static constexpr int BOX_BYTES = TP * 128;
  static constexpr int KV_BYTES = 2 * NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = KV_BYTES;
  static constexpr int NPSET = 2;                 // pair sets: 16 (row, head) pairs each
  static constexpr int NHALF = 2;                 // warps per pair set, each on half of a stage
  static constexpr int NCW = NPSET * NHALF;       // consumer warps
  static constexpr int NBH = NB16 / NHALF;        // 16-position blocks per warp and stage
  static constexpr int XF = 2 * (2 * NT + 2);     // floats a thread hands to its partner warp
  static constexpr int X_BYTES = NPSET * 32 * XF * 4;
  static constexpr int MAX_THREADS = 32 * (NCW + 1);
  static constexpr int SMEM_BYTES = 1024 + NST * STAGE_BYTES + X_BYTES + 2 * NST * 8;
  static constexpr float RESCALE_LOG2 = 8.f;
  static_assert(D == 64 || D == 128, "row grouping serves head_dim 64 and 128");
  static_assert(NB16 % NHALF == 0, "whole blocks per half");
};

__device__ __forceinline__ int rows_seq(const PartialParams& p, int t) {
  return p.seq_of ? __ldg(p.seq_of + t) : t;
}

// Group leaders: a group starts at every multiple of R and wherever seq_of[] changes.
__device__ __forceinline__ bool rows_is_leader(const PartialParams& p, int t, int R) {
  return t % R == 0 || rows_seq(p, t - 1) != rows_seq(p, t);
}

// Warp-cooperative search for the k-th group leader, scanning rows forward 32 at a time from a
// cursor (scan_t, scan_cnt = leaders before scan_t) that only moves forward; -1 past the last.
// Every lane of the warp calls it with the same arguments and gets the same answer.
__device__ __forceinline__ int rows_find_leader(const PartialParams& p, int R, int k, int& scan_t,
                                                int& scan_cnt, int lane) {
  if (p.rows_fixed) return k * R < p.n_tok ? k * R : -1;  // one sequence: groups of R rows
  while (scan_t < p.n_tok) {
    const int t = scan_t + lane;
    const unsigned m = __ballot_sync(0xffffffffu, t < p.n_tok && rows_is_leader(p, t, R));
    const int n = __popc(m);
    if (scan_cnt + n > k) {
      unsigned mm = m;
      for (int i = 0; i < k - scan_cnt; ++i) mm &= mm - 1;  // drop the earlier leaders
      return scan_t + __ffs(mm) - 1;
    }
    scan_cnt += n;
    scan_t += 32;
  }
  return -1;
}

// One group: its leader row, row count, sequence and longest (clamped) length.  Warp-wide.
struct RowGroup {
  int t0, nr, s, lmax;
};

// Row t's length L (kv_len[t] as read), clamped to the cache and zero for a bad sequence.
__device__ __forceinline__ int rows_len_of(const PartialParams& p, int L, bool seq_ok, int* err) {
  const int lmax = static_cast<int>(p.cache_cap < p.max_kv_len ? p.cache_cap : p.max_kv_len);
  if (L < 0 || L > lmax) {
    *err |= GQA_ERR_KVLEN_RANGE;
    L = L < 0 ? 0 : lmax;
  }
  if (!seq_ok) {
    *err |= GQA_ERR_SEQ_RANGE;
    L = 0;
  }
  return L;
}

__device__ __forceinline__ int rows_len(const PartialParams& p, int t, bool seq_ok, int* err) {
  return rows_len_of(p, __ldg(p.kv_len + t), seq_ok, err);
}

// Whether row t's sequence is valid: its group's verdict (a group's rows share one sequence),
// or with fixed groups (one sequence) its own seq_of entry, which must be that sequence, 0.
__device__ __forceinline__ bool rows_row_ok(const PartialParams& p, int t, bool group_ok) {
  return p.rows_fixed ? rows_seq(p, t) == 0 : group_ok;
}

// len0: kv_len[lane] for rows 0..31 when the caller loaded them beside the leader search (so
// that a group among the first 32 rows costs no second round trip); used when have_len0.
__device__ __forceinline__ RowGroup rows_group(const PartialParams& p, int t0, int R, int lane,
                                               int len0 = 0, bool have_len0 = false) {
  RowGroup gr;
  gr.t0 = t0;
  gr.s = p.rows_fixed ? 0 : rows_seq(p, t0);
  // rows t0 + 1 + i belong to the group while seq_of stays and no multiple of R is crossed;
  // checked 32 rows at a time (R can reach 64); with fixed groups, the next R rows
  gr.nr = p.rows_fixed ? min(R, p.n_tok - t0) : 1;
  for (int base = 0; !p.rows_fixed && base < R - 1; base += 32) {
    const int i = base + lane, t = t0 + 1 + i;
    const bool same = i < R - 1 && t < p.n_tok && t % R != 0 && rows_seq(p, t) == gr.s;
    const unsigned run = __ballot_sync(0xffffffffu, same);
    const int lead = __ffs(~run) - 1;  // leading rows of this window inside the group (-1: 32)
    gr.nr += lead < 0 ? 32 : lead;
    if (lead >= 0) break;
  }
  const bool seq_ok = gr.s >= 0 && gr.s < p.n_seq;
  int err = 0;
  int L = 0;
  const int lw = __shfl_sync(0xffffffffu, len0, (t0 + lane) & 31);  // row t0 + lane's, if < 32
  for (int jj = lane; jj < gr.nr; jj += 32) {
    const int t = t0 + jj;
    const bool ok = rows_row_ok(p, t, seq_ok);
    L = max(L, have_len0 && t < 32 ? rows_len_of(p, lw, ok, &err) : rows_len(p, t, ok, &err));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L = max(L, __shfl_xor_sync(0xffffffffu, L, o));
  gr.lmax = L;
  return gr;
}

// Two CTAs per SM: 168 registers a thread, so that three warps fit one SM sub-partition's
// 16K registers (200 registers measured 20 % slower: one CTA per SM)
template <int D>
__global__ void __launch_bounds__(RowsCfg<D>::MAX_THREADS, 2)
    partial_mma_rows_kernel(const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const PartialParams p) {
  using C = RowsCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int c = blockIdx.x, g = blockIdx.y, slot = blockIdx.z, nslots = gridDim.z;
  const int G = p.group;             // 1, 2, 4 or 8
  const int rpw = 16 / G;            // rows per warp
  const int R = rpw * C::NPSET;      // rows per group at most
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = c * p.chunk;

  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  float* xbuf = reinterpret_cast<float*>(stages + C::NST * C::STAGE_BYTES);  // [pset][XF][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::NST * C::STAGE_BYTES + C::X_BYTES);
  uint64_t* empty = full + C::NST;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C::NCW);
    }
    mbar_init_fence();
  }
  __syncthreads();

  // Every warp walks the same groups (k = slot, slot + nslots, ...) in the same order, so the
  // producer's tiles and the consumers' waits line up across groups.
  int scan_t = 0, scan_cnt = 0;

  if (warp == C::NCW) {  // ---- producer warp: lane 0 issues, the warp walks the groups
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    int it = 0;
    bool ok = true;
    for (int k = slot; ok; k += nslots) {
      const int t0 = rows_find_leader(p, R, k, scan_t, scan_cnt, lane);
      if (t0 < 0) break;
      const RowGroup gr = rows_group(p, t0, R, lane);
      const int c1 = min(c0 + p.chunk, gr.lmax);  // nothing to issue when c1 <= c0
      const int zb = gr.s * static_cast<int>(p.cache_cap) + c0;
      for (int pos = c0; pos < c1; pos += C::TP, ++it) {
        const int st = it % C::NST;
        if (it >= C::NST &&
            !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((it / C::NST) - 1) & 1))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[st], C::KV_BYTES);
          uint8_t* sk = stages + st * C::STAGE_BYTES;
          uint8_t* sv = sk + C::NBOX * C::BOX_BYTES;
#pragma unroll
          for (int bx = 0; bx < C::NBOX; ++bx) {
            tma_load_3d(sk + bx * C::BOX_BYTES, &tmK, bx * 64, g, zb + pos - c0, &full[st]);
            tma_load_3d(sv + bx * C::BOX_BYTES, &tmV, bx * 64, g, zb + pos - c0, &full[st]);
          }
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      if (!ok) flag_error(p.err, GQA_ERR_TIMEOUT);
      for (int st = 0; st < C::NST && st < it; ++st) {  // the last load of each stage lands
        const int last = st + ((it - 1 - st) / C::NST) * C::NST;
        if (!mbar_wait(&full[st], (last / C::NST) & 1)) flag_error(p.err, GQA_ERR_TIMEOUT);
      }
    }
    return;
  }

  // ---- consumer warps: pair set ps = warp % 4 holds 16 (row, head) pairs, pair i = A row i
  //      with row j = ps * rpw + i / G and head h = i % G; half hf = warp / 4 takes blocks
  //      [hf * NBH, (hf + 1) * NBH) of every stage.  Thread (gid, tig) owns pairs gid, gid + 8.
  const int ps = warp % C::NPSET, hf = warp / C::NPSET;
  const int gid = lane >> 2, tig = lane & 3;
  const int mi = lane >> 3, rr = lane & 7;
  int it = 0;
  bool ok = true;

  // Every consumer warp walks every group, also after a failed wait (then computing nothing),
  // so that the CTA's named barriers stay in step.
  for (int k = slot;; k += nslots) {
    const int t0 = rows_find_leader(p, R, k, scan_t, scan_cnt, lane);
    if (t0 < 0) break;
    const RowGroup gr = rows_group(p, t0, R, lane);
    const bool seq_ok = gr.s >= 0 && gr.s < p.n_seq;
    if (c == 0 && warp == 0) {  // per-row bookkeeping: flags, chunk counts, empty rows
      for (int jb = 0; jb < gr.nr; jb += 32) {
        int err = 0;
        const int L = jb + lane < gr.nr ? rows_len(p, t0 + jb + lane, seq_ok, &err) : 0;
        if (jb + lane < gr.nr) {
          if (err && g == 0) flag_error(p.err, err);
          if (g == 0 && p.merge) p.n_valid[t0 + jb + lane] = (L + p.chunk - 1) / p.chunk;
        }
        for (int jj = 0; jj < 32 && jb + jj < gr.nr; ++jj) {
          if (__shfl_sync(0xffffffffu, L, jj) != 0) continue;  // empty row: zeros
          for (int i = lane; i < G * D; i += 32)
            p.out[((size_t)(t0 + jb + jj) * p.n_heads + g * G + i / D) * D + i % D] = 0.f;
        }
      }
    }
    if (c0 < gr.lmax) {  // the same for every consumer warp
      const int c1 = min(c0 + p.chunk, gr.lmax);
      bool rv[2];
      int tr[2], Lr[2], hd[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = gid + 8 * u;
        const int j = ps * rpw + i / G;
        rv[u] = j < gr.nr;  // this pair is a real row
        tr[u] = t0 + (rv[u] ? j : 0);
        int dummy = 0;
        Lr[u] = rv[u] ? rows_len(p, tr[u], seq_ok, &dummy) : 0;  // the row's own length
        hd[u] = g * G + i % G;
      }
      const bool active = ps * rpw < gr.nr;  // the pair set has rows in this group

      // q in f16 with scale * log2(e) folded in: rows gid and gid + 8 of the A fragments
      uint32_t qa[C::KS][4];
      {
        const float* q0 = p.q + ((size_t)tr[0] * p.n_heads + hd[0]) * D;
        const float* q1 = p.q + ((size_t)tr[1] * p.n_heads + hd[1]) * D;
        const float f0 = rv[0] ? p.scale_log2 : 0.f, f1 = rv[1] ? p.scale_log2 : 0.f;
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          const int d0 = ks * 16 + 2 * tig;
          const float2 x0 = __ldg(reinterpret_cast<const float2*>(q0 + d0));
          const float2 x1 = __ldg(reinterpret_cast<const float2*>(q0 + d0 + 8));
          const float2 y0 = __ldg(reinterpret_cast<const float2*>(q1 + d0));
          const float2 y1 = __ldg(reinterpret_cast<const float2*>(q1 + d0 + 8));
          qa[ks][0] = h2_bits(__floats2half2_rn(x0.x * f0, x0.y * f0));
          qa[ks][1] = h2_bits(__floats2half2_rn(y0.x * f1, y0.y * f1));
          qa[ks][2] = h2_bits(__floats2half2_rn(x1.x * f0, x1.y * f0));
          qa[ks][3] = h2_bits(__floats2half2_rn(y1.x * f1, y1.y * f1));
        }
      }
      float o[C::NT][4];
#pragma unroll
      for (int n = 0; n < C::NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

      for (int pos0 = c0; ok && pos0 < c1; pos0 += C::TP, ++it) {
        const int st = it % C::NST;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (it / C::NST) & 1));
        if (!ok) break;
        if (active) {
          const uint32_t sk = smem_addr(stages + st * C::STAGE_BYTES);
          const uint32_t sv = sk + C::NBOX * C::BOX_BYTES;
          // q.k^T for this warp's blocks of the stage first (independent MMA chains), then the
          // softmax and p.v of each block
          float sc[C::NBH][2][4];
#pragma unroll
          for (int bb = 0; bb < C::NBH; ++bb) {
            const int r0 = (hf * C::NBH + bb) * 16;
            float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) sc[bb][nt][e] = 0.f;
            if (pos0 + r0 >= c1) continue;  // block past the chunk end
#pragma unroll
            for (int ks = 0; ks < C::KS; ks += 2) {
              uint32_t kb[4], kc[4];
              ldsm_x4(kb, sk + swz_off(r0 + (mi >> 1) * 8 + rr, ks * 2 + (mi & 1), C::TP));
              ldsm_x4(kc, sk + swz_off(r0 + (mi >> 1) * 8 + rr, ks * 2 + 2 + (mi & 1), C::TP));
              mma_f16(sc[bb][0], qa[ks], kb[0], kb[1]);
              mma_f16(sc[bb][1], qa[ks], kb[2], kb[3]);
              mma_f16(sd[0], qa[ks + 1], kc[0], kc[1]);
              mma_f16(sd[1], qa[ks + 1], kc[2], kc[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) sc[bb][nt][e] += sd[nt][e];
          }
#pragma unroll
          for (int bb = 0; bb < C::NBH; ++bb) {
            const int r0 = (hf * C::NBH + bb) * 16;
            const int base = pos0 + r0;  // cache position of the block's row 0
            const int nv = min(max(c1 - base, 0), 16);  // rows holding data for some row
            if (nv == 0) continue;
            float x[2][2][2], mt[2];
            bool grow[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int nrow = min(max(Lr[u] - base, 0), 16);  // rows inside the pair's window
              mt[u] = -INFINITY;
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                  x[u][nt][jj] = (nt * 8 + 2 * tig + jj) < nrow ? sc[bb][nt][2 * u + jj] : -INFINITY;
                  mt[u] = fmaxf(mt[u], x[u][nt][jj]);
                }
              mt[u] = fmaxf(mt[u], __shfl_xor_sync(0xffffffffu, mt[u], 1));
              mt[u] = fmaxf(mt[u], __shfl_xor_sync(0xffffffffu, mt[u], 2));
              // a pair whose row ends before this block keeps mt = -inf: nothing to add
              grow[u] = mt[u] != -INFINITY && mt[u] > m_run[u] + C::RESCALE_LOG2;
            }
            if (__any_sync(0xffffffffu, grow[0] || grow[1])) {
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const float m_new = grow[u] ? mt[u] : m_run[u];
                const float corr = grow[u] ? fast_exp2(m_run[u] - m_new) : 1.f;
                m_run[u] = m_new;
                l_run[u] *= corr;
#pragma unroll
                for (int n = 0; n < C::NT; ++n) {
                  o[n][2 * u] *= corr;
                  o[n][2 * u + 1] *= corr;
                }
              }
            }
            float pr[2][2][2];
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                  pr[u][nt][jj] = m_run[u] == -INFINITY ? 0.f : fast_exp2(x[u][nt][jj] - m_run[u]);
                  l_run[u] += pr[u][nt][jj];
                }
            // the weights straight from the score fragments: A rows gid / gid + 8, k = positions
            uint32_t pa[4];
            pa[0] = h2_bits(__floats2half2_rn(pr[0][0][0], pr[0][0][1]));
            pa[1] = h2_bits(__floats2half2_rn(pr[1][0][0], pr[1][0][1]));
            pa[2] = h2_bits(__floats2half2_rn(pr[0][1][0], pr[0][1][1]));
            pa[3] = h2_bits(__floats2half2_rn(pr[1][1][0], pr[1][1][1]));
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
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }

      // ---- the second half's states join the first's: half 1 hands its (m, l, o) over in
      //      shared memory, thread by thread; half 0 combines them
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        l_run[u] += __shfl_xor_sync(0xffffffffu, l_run[u], 1);
        l_run[u] += __shfl_xor_sync(0xffffffffu, l_run[u], 2);
      }
      float* xb = xbuf + ps * C::XF * 32 + lane;  // element f at xb[f * 32]
      if (hf == 1) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          xb[(u * (2 * C::NT + 2)) * 32] = m_run[u];
          xb[(u * (2 * C::NT + 2) + 1) * 32] = l_run[u];
#pragma unroll
          for (int n = 0; n < C::NT; ++n) {
            xb[(u * (2 * C::NT + 2) + 2 + 2 * n) * 32] = o[n][2 * u];
            xb[(u * (2 * C::NT + 2) + 3 + 2 * n) * 32] = o[n][2 * u + 1];
          }
        }
      }
      named_bar_sync(1, 32 * C::NCW);
      if (hf == 0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float m1 = xb[(u * (2 * C::NT + 2)) * 32];
          const float l1 = xb[(u * (2 * C::NT + 2) + 1) * 32];
          const float M = fmaxf(m_run[u], m1);
          const float e0 = m_run[u] == -INFINITY ? 0.f : fast_exp2(m_run[u] - M);
          const float e1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
          l_run[u] = l_run[u] * e0 + l1 * e1;
          m_run[u] = M;
#pragma unroll
          for (int n = 0; n < C::NT; ++n) {
            o[n][2 * u] = o[n][2 * u] * e0 + xb[(u * (2 * C::NT + 2) + 2 + 2 * n) * 32] * e1;
            o[n][2 * u + 1] = o[n][2 * u + 1] * e0 + xb[(u * (2 * C::NT + 2) + 3 + 2 * n) * 32] * e1;
          }
        }
      }
      named_bar_sync(1, 32 * C::NCW);  // half 1 may refill its slots for the next group

      // ---- each of this thread's pairs (half 0): the output, or the chunk's partial (merged
      //      afterwards by merge_kernel)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (!ok || !active || hf != 0) break;
        if (!rv[u] || c0 >= Lr[u]) continue;
        const float l = l_run[u];
        if (!p.merge) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          float* orow = p.out + ((size_t)tr[u] * p.n_heads + hd[u]) * D;
#pragma unroll
          for (int n = 0; n < C::NT; ++n) {
            const int d = n * 8 + 2 * tig;
            *reinterpret_cast<float2*>(orow + d) =
                make_float2(gated(p, tr[u], hd[u], d, o[n][2 * u] * inv),
                            gated(p, tr[u], hd[u], d + 1, o[n][2 * u + 1] * inv));
          }
        } else {
          float* prt = p.part + (((size_t)tr[u] * p.n_split + c) * p.n_heads + hd[u]) * (D + 2);
#pragma unroll
          for (int n = 0; n < C::NT; ++n)
            *reinterpret_cast<float2*>(prt + n * 8 + 2 * tig) =
                make_float2(o[n][2 * u], o[n][2 * u + 1]);
          if (tig == 0) {
            prt[D] = m_run[u] == -INFINITY ? -INFINITY : m_run[u] * kLn2;  // natural-log units
            prt[D + 1] = l;
          }
        }
      }
    }  // this chunk's work on the group
  }
  if (!ok && lane == 0) flag_error(p.err, GQA_ERR_TIMEOUT);
  // this CTA's partials are written: the merge kernel launched after this one may be scheduled
  // (it waits for this grid's completion and memory before reading anything)
  asm volatile("griddepcontrol.launch_dependents;");
}

}  // namespace gqa
