// rows_umma.cuh -- row-grouped f16 decode attention on the fifth-generation tensor cores.
//
// The rows of a causal prefill chunk (flash_attention_tq.metal's per-query window: row r at
// position p attends to [0, p]) or the decode rows of one sequence read the same K/V.  One CTA
// serves a group of up to 64 / G such rows for one KV head and one chunk of positions, so every
// K/V tile is read from HBM once for all of the group's (row, head) pairs (attention_gqa.metal's
// "load K/V once, reuse across the group", widened from the heads of a group to the rows of a
// sequence).  The group's 64 pairs are the rows of the MMAs.
//
// Per 64-position tile, flash-attention style:
//   S  = Q . K^T    M = 128, N = 64 positions, K = D: Q (scale * log2 e folded in) as an f16 hi
//                   part in row 32 (p / 16) + p % 16 for pair p and its f16 lo remainder 16 rows
//                   below (about 22 bits of the fp32 q), the K tile K-major in shared memory; S
//                   in TMEM, row r in lane r, so a pair's hi and lo rows sit in the lanes of one
//                   softmax warp.  (An M = 64 MMA costs what an M = 128 one does: one MMA per
//                   k-step carries both parts.)
//   softmax         two threads per pair: thread (warp w, lane l) owns pair 16 w + l % 16 and
//                   the tile's positions [32 h, 32 h + 32), h = l / 16.  Each reads its own
//                   lane's 64 columns (two tcgen05.ld 32x32b) and swaps 32 of them with its
//                   partner (lane l xor 16), so that it holds hi + lo for its half.
//                   It masks positions at or past its row's length; the two halves' maxima meet
//                   by one shuffle, so both keep the same running max, and each keeps its own
//                   part of the running sum.  The max moves lazily (only when a tile's max
//                   exceeds it by more than 2^8, so p <= 256); when it moves, each thread
//                   rescales its half of the pair's O row in TMEM (ld, scale, st) after the
//                   previous tile's P.V has completed.
//   O += P . V      M = 64 pairs: P (f16, written by the softmax threads into shared memory,
//                   K-major) times the V tile read MN-major (N = D contiguous), accumulated in
//                   TMEM (row i in lane 32 (i / 16) + i % 16).
// Three S buffers in TMEM and three P buffers in shared memory let the tensor cores run up to two
// tiles' S ahead of the softmax.  K/V tiles stream through a four-stage TMA ring;
// the group's fp32 q arrives first, by bulk copies from the producer into a staging area, and is
// converted there.  V rows past the group's longest row are zeroed in shared memory before the
// P.V MMA (P is zero there, but cache garbage could be NaN).  At the end of the chunk the O rows
// go through shared memory so that the records (or outputs) are written row by row, coalesced.
//
// Warps: 0-3 softmax and epilogue, 4 TMA producer, 5 S issuer (one lane) and TMEM owner, 6 P.V
// issuer (one lane).  S(i) goes once K/V tile i has landed and the softmax has read S(i - 3)
// (three S buffers); P.V(i) once P(i) is written.  Barriers: full/empty per stage (TMA <-> MMA),
// q_land (q staged), q_full (softmax wrote the group's Q), s_full per S buffer (S issuer ->
// softmax), p_full per P buffer (softmax -> both issuers), pv_done per P buffer (P.V issuer ->
// softmax: P buffer free again, O final for a rescale or the epilogue), x_free (softmax ->
// producer: the staging area is free for the next group's q).  Every wait is bounded.  A wait
// that runs out flags GQA_ERR_TIMEOUT; the producer and the issuers then stop, while the softmax
// warps stop waiting but walk on to the end (their named barriers and the merge counters stay in
// step).  Before TMEM is freed each issuer waits for all of its MMAs to complete.
//
// MMA cost (measured on GB300, one thread issuing back to back): M64 N64 K16 ~56 cycles, M64
// N128 K16 ~70, M128 N256 K16 ~133 (the dense peak).  M = 64 half-fills the tensor core: P.V
// leaves that half empty, S fills it with q's lo rows.
//
// Groups, slots, the per-row bookkeeping (n_valid, empty rows) and the partial format are those
// of the mma.sync row kernel (rows_mma.cuh).  Split rows are merged inside this kernel when the
// whole grid fits one CTA per SM: the host then launches it cooperatively, so that a group's
// chunk CTAs are resident together and can wait for one another (rows_fused_merge below).  A
// larger grid is followed by merge_kernel instead, as a programmatic dependent launch.
#pragma once

#include "rows_mma.cuh"
#include "umma.cuh"

namespace gqa {

template <int D>
struct UmmaRowsCfg {
  static constexpr int M = 64;                     // MMA rows: (row, head) pairs per group
  static constexpr int NP = M;
  static constexpr int TP = 64;                    // positions per tile (one TMA box high)
  static constexpr int CPT = TP / 2;               // score columns per softmax thread and tile
  static constexpr int NBOX = D / 64;              // 128-byte boxes across D
  static constexpr int BOX_BYTES = TP * 128;       // one box: TP rows x 128 bytes
  static constexpr int KV_BYTES = NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;  // K boxes, then V boxes
  static constexpr int NST = 4;
  // S = Q.K^T runs at M = 128: pair p's q as f16 hi in row 32 (p / 16) + p % 16 and its f16 lo
  // remainder 16 rows below, so that both land in the TMEM lanes of one softmax warp.  An
  // M = 64 MMA costs as much as an M = 128 one: the lo rows ride along for free.
  static constexpr int MS = 128;
  static constexpr int Q_BOX = MS * 128;           // Q: [box][128 rows][128 bytes]
  static constexpr int Q_BYTES = NBOX * Q_BOX;
  static constexpr int P_BYTES = M * TP * 2;       // P: [64 pairs][64 positions] f16
  static constexpr int NPB = 3;                    // S buffers (TMEM) and P buffers (smem)
  static constexpr int S_COL = 0, O_COL = NPB * TP;
  static constexpr int TMEM_COLS = NPB * TP + D <= 256 ? 256 : 512;
  static constexpr int KS_S = D / 16;              // k steps of S = Q.K^T
  static constexpr int KS_O = TP / 16;             // k steps of O += P.V
  static constexpr int NSW = 4, PRODUCER = 4, ISSUER = 5, PV_ISSUER = 6;
  static constexpr int THREADS = 224;
  static constexpr int NBAR = 2 * NST + 4 + 3 * NPB + 1;
  // staging of the group's fp32 q, then the epilogue's exchange: records [NP][D + 2] + flags
  static constexpr int X_BYTES = cmax(NP * D * 4, NP * (D + 2) * 4 + NP * 4);
  static constexpr int BAR_OFF = NST * STAGE_BYTES + Q_BYTES + NPB * P_BYTES;
  static constexpr int X_OFF = align_up(BAR_OFF + NBAR * 8 + 8, 128);  // bulk copies, float4
  static constexpr int SMEM_BYTES = 1024 + X_OFF + X_BYTES;
  static constexpr float RESCALE_LOG2 = 8.f;
  static_assert(D == 64 || D == 128, "row grouping serves head_dim 64 and 128");
  static_assert(P_BYTES == M * 128, "P rows are one 128-byte box row");
  static_assert(CPT == 32, "one 32-column TMEM load per thread and tile");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(STAGE_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0 && P_BYTES % 1024 == 0,
                "swizzled tiles start on 1024-byte atoms");
  static_assert(BAR_OFF % 8 == 0 && X_OFF % 16 == 0, "barrier and staging alignment");
};

// The fused merge of one group (run by the 128 softmax threads of every chunk CTA of the group,
// all resident under a cooperative launch).  Every CTA's records are stored and fenced before it
// counts itself in; once all gridDim.x chunk CTAs are in, CTA c merges the group's pairs
// c, c + gridDim.x, ... (warp w of it takes every fourth of those), reading the records past L1,
// with merge_kernel's arithmetic.
//
// The counter protocol survives a wait that runs out.  Every chunk CTA counts in exactly twice
// per group, whatever happens: once after its records are stored, and once more after its wait
// (seen all in, or given up after p.merge_spin polls).  The counter therefore reaches 2 nctas
// in every call, and the CTA whose second count-in takes it there resets it to zero: no later
// call on the same workspace can find it part-way.  A CTA whose wait ran out flags
// GQA_ERR_TIMEOUT and skips its share of the merge; that call's output is not to be used.
template <int D>
__device__ void rows_fused_merge(const PartialParams& p, const RowGroup& gr, int k, int g, int c,
                                 bool seq_ok, int* merge_ok) {
  constexpr int DPL = D / 32;
  constexpr int NSW = UmmaRowsCfg<D>::NSW;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = p.group;
  const unsigned int nctas = gridDim.x;
  unsigned int* cnt = p.counters + (size_t)k * p.n_kv_heads + g;
  __threadfence();  // this thread's record stores, device-wide
  named_bar_sync(1, 32 * NSW);
  if (threadIdx.x == 0) {
    atomicAdd(cnt, 1u);
    int ok = 0;
    for (uint32_t i = 0; i < p.merge_spin; ++i) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
      if (v >= nctas) {
        ok = 1;
        break;
      }
    }
    // the second count-in, taken by every CTA whether or not its wait succeeded; the last one
    // resets the counter for the next call (its latency overlaps this CTA's merge)
    if (atomicAdd(cnt, 1u) == 2 * nctas - 1) atomicExch(cnt, 0u);
    if (!ok) flag_error(p.err, GQA_ERR_TIMEOUT);
    *merge_ok = ok;
  }
  named_bar_sync(1, 32 * NSW);
  const bool ok = *merge_ok != 0;
  if (ok) {
    const size_t rec = (size_t)p.n_heads * (D + 2);
    for (int q = c + warp * (int)nctas; q < gr.nr * G; q += NSW * (int)nctas) {
      const int t = gr.t0 + q / G, h = g * G + q % G;
      int dummy = 0;
      const int L = rows_len(p, t, rows_row_ok(p, t, seq_ok), &dummy);
      if (L == 0) continue;  // zeroed by the bookkeeping
      const int nv = min((L + p.chunk - 1) / p.chunk, p.n_split);
      const float* base = p.part + ((size_t)t * p.n_split * p.n_heads + h) * (D + 2);
      float a[DPL];
#pragma unroll
      for (int e = 0; e < DPL; ++e) a[e] = 0.f;
      float M = -INFINITY, Ls = 0.f;
      // batches of up to MB chunks: every load of a batch (lane c's (m, l), each lane's D / 32
      // dims of every chunk) is issued before any is used, so a batch costs one L2 round trip
      constexpr int MB = 24;
      for (int cb = 0; cb < nv; cb += MB) {
        const int nb = min(MB, nv - cb);
        float m = -INFINITY, l = 0.f;
        if (lane < nb) {
          m = __ldcg(base + (cb + lane) * rec + D);
          l = __ldcg(base + (cb + lane) * rec + D + 1);
        }
        const float* ac = base + cb * rec + lane * DPL;
        float2 v[MB][DPL / 2];
#pragma unroll
        for (int j = 0; j < MB; ++j)
#pragma unroll
          for (int e = 0; e < DPL / 2; ++e)
            v[j][e] = j < nb ? __ldcg(reinterpret_cast<const float2*>(ac + j * rec) + e)
                             : make_float2(0.f, 0.f);
        float mb = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
        const float M_new = fmaxf(M, mb);
        if (M_new == -INFINITY) continue;
        const float corr = M == -INFINITY ? 0.f : __expf(M - M_new);
        M = M_new;
        Ls *= corr;
#pragma unroll
        for (int e = 0; e < DPL; ++e) a[e] *= corr;
        const float w = m == -INFINITY ? 0.f : __expf(m - M);
        Ls = fmaf(l, w, Ls);
#pragma unroll
        for (int j = 0; j < MB; ++j) {
          const float wj = __shfl_sync(0xffffffffu, w, j);  // 0 past nb (lanes >= nb: w = 0)
#pragma unroll
          for (int e = 0; e < DPL / 2; ++e) {
            a[2 * e] = fmaf(wj, v[j][e].x, a[2 * e]);
            a[2 * e + 1] = fmaf(wj, v[j][e].y, a[2 * e + 1]);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      float* orow = p.out + ((size_t)t * p.n_heads + h) * D + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; e += 2)
        *reinterpret_cast<float2*>(orow + e) =
            make_float2(gated(p, t, h, lane * DPL + e, a[e] * inv),
                        gated(p, t, h, lane * DPL + e + 1, a[e + 1] * inv));
    }
  }
  // (merge_ok is written again only after the next named barrier, which every thread reaches
  // after its read above)
}

template <int D>
__global__ void __launch_bounds__(UmmaRowsCfg<D>::THREADS, 1)
    umma_rows_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const PartialParams p) {
  using C = UmmaRowsCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const int c = blockIdx.x, g = blockIdx.y, slot = blockIdx.z, nslots = gridDim.z;
  const int G = p.group;    // 1, 2, 4 or 8
  const int R = C::NP / G;  // rows per group at most
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = c * p.chunk;

  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  uint8_t* sQ = stages + C::NST * C::STAGE_BYTES;
  uint8_t* sP = sQ + C::Q_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sP + C::NPB * C::P_BYTES);
  uint64_t* empty = full + C::NST;
  uint64_t* q_full = empty + C::NST;
  uint64_t* s_full = q_full + 1;
  uint64_t* p_full = s_full + C::NPB;
  uint64_t* pv_done = p_full + C::NPB;
  uint64_t* drain = pv_done + C::NPB;  // [2]: one per issuing thread
  uint64_t* q_land = drain + 2;
  uint64_t* x_free = q_land + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(x_free + 1);
  int* merge_ok = reinterpret_cast<int*>(tmem_holder + 1);
  uint8_t* sX = stages + C::X_OFF;  // 128-byte aligned

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(q_full, 32 * C::NSW);
    for (int i = 0; i < C::NPB; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 32 * C::NSW);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(q_land, 1);
    mbar_init(x_free, 32 * C::NSW);
    mbar_init_fence();
  }
  // Every warp walks the same groups (k = slot, slot + nslots, ...) in the same order.  The first
  // group is looked up while thread 0 sets up the barriers and the issuer warp allocates TMEM.
  int scan_t = 0, scan_cnt = 0;
  // rows 0..31's lengths, loaded beside the leader search's reads of seq_of
  const int len0 = lane < p.n_tok ? __ldg(p.kv_len + lane) : 0;
  const int t0_first = rows_find_leader(p, R, slot, scan_t, scan_cnt, lane);
  RowGroup gr_first{};
  if (t0_first >= 0) gr_first = rows_group(p, t0_first, R, lane, len0, true);
  auto group = [&](int k, RowGroup& gr) {  // the k-th group's leader (-1 past the last)
    if (k == slot) {
      gr = gr_first;
      return t0_first;
    }
    const int t0 = rows_find_leader(p, R, k, scan_t, scan_cnt, lane);
    if (t0 >= 0) gr = rows_group(p, t0, R, lane);
    return t0;
  };
  if (warp == C::ISSUER) tmem_alloc(tmem_holder, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;
  bool ok = true;

  if (warp == C::PRODUCER) {  // ---- TMA producer: lane 0 issues, the warp walks the groups
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmQ);
    }
    int it = 0, gn = 0;
    for (int k = slot; ok; k += nslots) {
      RowGroup gr;
      const int t0 = group(k, gr);
      if (t0 < 0) break;
      const int c1 = min(c0 + p.chunk, gr.lmax);
      if (c1 <= c0) continue;
      // the group's fp32 q first (one TMA box: its rows' G heads, rows past the group read
      // too and ignored), into the staging area once the previous group's epilogue is done
      // with it (16 bulk copies, one per row, took ~1.1 us to issue)
      if (gn > 0) ok = __all_sync(0xffffffffu, mbar_wait(x_free, (gn - 1) & 1));
      if (!ok) break;
      ++gn;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_land, C::NP * D * 4);
        tma_load_3d(sX, &tmQ, 0, g * G, t0, q_land);
      }
      const int zb = gr.s * static_cast<int>(p.cache_cap);
      for (int pos = c0; pos < c1; pos += C::TP, ++it) {
        const int st = it % C::NST;
        if (it >= C::NST &&
            !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((it / C::NST) - 1) & 1))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
          uint8_t* sk = stages + st * C::STAGE_BYTES;
          uint8_t* sv = sk + C::KV_BYTES;
#pragma unroll
          for (int bx = 0; bx < C::NBOX; ++bx) {
            tma_load_3d(sk + bx * C::BOX_BYTES, &tmK, bx * 64, g, zb + pos, &full[st]);
            tma_load_3d(sv + bx * C::BOX_BYTES, &tmV, bx * 64, g, zb + pos, &full[st]);
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
  } else if (warp == C::ISSUER || warp == C::PV_ISSUER) {
    // ---- MMA issuers, lane 0 of each: warp ISSUER issues S = Q . K^T, warp PV_ISSUER
    //      O += P . V (two issuing threads keep both MMA streams going; MMAs of one shape issued
    //      back to back also run faster than alternating ones)
    const bool is_s = warp == C::ISSUER;
    constexpr uint32_t kIdS = umma_idesc_f16(C::MS, C::TP, false);
    constexpr uint32_t kIdO = umma_idesc_f16(C::M, D, true);
    const uint32_t q_addr = smem_addr(sQ), p_addr = smem_addr(sP);
    int it = 0, qn = 0;
    for (int k = slot; ok; k += nslots) {
      RowGroup gr;
      const int t0 = group(k, gr);
      if (t0 < 0) break;
      const int c1 = min(c0 + p.chunk, gr.lmax);
      if (c1 <= c0) continue;
      const int ntile = (c1 - c0 + C::TP - 1) / C::TP;
      ok = __all_sync(0xffffffffu, mbar_wait(q_full, qn & 1));
      ++qn;
      if (!ok) break;
      if (lane == 0) {
        for (int j = 0; j < ntile && ok; ++j) {
          const int i = it + j;
          if (is_s) {
            // S(i) once tile i has landed and the softmax has read S(i - NPB) (its P is out)
            const int st = i % C::NST;
            ok = mbar_wait(&full[st], (i / C::NST) & 1) &&
                 (j < C::NPB ||
                  mbar_wait(&p_full[(i - C::NPB) % C::NPB], ((i - C::NPB) / C::NPB) & 1));
            if (!ok) break;
            tc_fence_after();
            const uint32_t sk = smem_addr(stages + st * C::STAGE_BYTES);
#pragma unroll
            for (int kk = 0; kk < C::KS_S; ++kk) {
              const uint32_t ko = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
              const uint32_t qo = (kk >> 2) * C::Q_BOX + (kk & 3) * 32;
              // q's hi and lo rows (f16 parts, about 22 bits) against the f16 K tile
              umma_f16(tbase + C::S_COL + (i % C::NPB) * C::TP,
                       umma_desc_sw128(q_addr + qo, 16, 1024),
                       umma_desc_sw128(sk + ko, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[i % C::NPB]);
          } else {
            // P.V(i) once P(i) is written (after S(i) completed); its completion frees the
            // stage (K was read by S(i) before) and P buffer i % NPB
            ok = mbar_wait(&p_full[i % C::NPB], (i / C::NPB) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint32_t sv = smem_addr(stages + (i % C::NST) * C::STAGE_BYTES + C::KV_BYTES);
            const uint32_t pa = p_addr + (i % C::NPB) * C::P_BYTES;
#pragma unroll
            for (int kk = 0; kk < C::KS_O; ++kk)
              umma_f16(tbase + C::O_COL, umma_desc_sw128(pa + kk * 32, 16, 1024),
                       umma_desc_sw128(sv + kk * 2048, C::BOX_BYTES, 1024), kIdO,
                       (j == 0 && kk == 0) ? 0u : 1u);
            umma_commit(&empty[i % C::NST]);
            umma_commit(&pv_done[i % C::NPB]);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      it += ntile;
    }
    if (!ok && lane == 0) flag_error(p.err, GQA_ERR_TIMEOUT);
    // every MMA this thread issued has completed before TMEM is freed
    if (lane == 0) {
      umma_commit(&drain[is_s ? 0 : 1]);
      if (!mbar_wait(&drain[is_s ? 0 : 1], 0)) flag_error(p.err, GQA_ERR_TIMEOUT);
    }
    __syncwarp();
  } else {  // ---- softmax warpgroup: two threads per pair (position halves of each tile)
    const int h = lane >> 4;                 // tile positions [32 h, 32 h + 32)
    const int i = warp * 16 + (lane & 15);   // pair = MMA row
    const int jr = i / G;
    const uint32_t t_q = tbase + (static_cast<uint32_t>(warp * 32) << 16);  // lane quadrant
    float* xo = reinterpret_cast<float*>(sX);  // exchange: records [NP][D + 2], then flags
    int* xw = reinterpret_cast<int*>(xo + C::NP * (D + 2));
    // A completed phase is seen at once by a test; a pending one is waited for (bounded).
    // After a wait has run out (ok false) no wait is tried again, but every softmax warp still
    // walks every group and tile to the end -- computing garbage, flagged GQA_ERR_TIMEOUT --
    // so that the four warps reach the same named barriers and every chunk CTA counts in on
    // every group's merge counter.  ok is warp-uniform.
    auto wait = [&ok](uint64_t* bar, uint32_t parity) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_test(bar, parity) || mbar_wait(bar, parity));
      return ok;
    };
    int it = 0, qn = 0;
    for (int k = slot;; k += nslots) {
      RowGroup gr;
      const int t0 = group(k, gr);
      if (t0 < 0) break;
      const bool seq_ok = gr.s >= 0 && gr.s < p.n_seq;
      const int c1 = min(c0 + p.chunk, gr.lmax);
      if (c == 0 && warp == 0) {  // per-row bookkeeping: flags, chunk counts, empty rows
        for (int jb = 0; jb < gr.nr; jb += 32) {
          int err = 0;
          const int tr = t0 + jb + lane;
          const int L = jb + lane < gr.nr ? rows_len(p, tr, rows_row_ok(p, tr, seq_ok), &err) : 0;
          if (jb + lane < gr.nr) {
            if (err && g == 0) flag_error(p.err, err);
            if (g == 0 && p.merge) p.n_valid[t0 + jb + lane] = (L + p.chunk - 1) / p.chunk;
          }
          for (int jj = 0; jj < 32 && jb + jj < gr.nr; ++jj) {
            if (__shfl_sync(0xffffffffu, L, jj) != 0) continue;  // empty row: zeros
            for (int e = lane; e < G * D; e += 32)
              p.out[((size_t)(t0 + jb + jj) * p.n_heads + g * G + e / D) * D + e % D] = 0.f;
          }
        }
      }
      if (c1 <= c0) {  // the same decision as the producer's and the issuer's
        if (p.merge && p.fused_merge) rows_fused_merge<D>(p, gr, k, g, c, seq_ok, merge_ok);
        continue;
      }
      const int ntile = (c1 - c0 + C::TP - 1) / C::TP;
      const bool rv = jr < gr.nr;  // this pair is a real row
      const int t = t0 + (rv ? jr : 0);
      int dummy = 0;
      const int Lp = rv ? rows_len(p, t, rows_row_ok(p, t, seq_ok), &dummy) : 0;
      // chunk positions [0, lim0) are the pair's, counted from this thread's half of a tile
      const int lim0 = min(Lp, c0 + p.chunk) - c0 - C::CPT * h;

      // ---- Q: the staged fp32 q [pair][D] to f16 with scale * log2(e), 128-byte swizzled:
      //      thread r takes float4 pieces r, r + 128, ... (all loads first).  Pad pairs get
      //      zeros (their staging is not loaded).  No P is written before S(0), which waits for
      //      every thread's q_full arrival.
      wait(q_land, qn & 1);
      {
        constexpr int NQ = C::NP * D / 4 / (32 * C::NSW);  // float4 pieces per thread
        const float4* qs = reinterpret_cast<const float4*>(sX);
        float4 v[NQ];
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
          const int f = threadIdx.x + u * 32 * C::NSW, qr = f / (D / 4);
          v[u] = qr / G < gr.nr ? qs[f] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float sc = p.scale_log2;
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
          const int f = threadIdx.x + u * 32 * C::NSW, qr = f / (D / 4), c4 = f % (D / 4);
          const int ch = c4 >> 1;  // 16-byte chunk of the f16 row
          uint2 hv, lv;  // the f16 hi part and the f16 lo remainder of q * scale * log2(e)
          split_hi_lo(v[u].x * sc, v[u].y * sc, hv.x, lv.x);
          split_hi_lo(v[u].z * sc, v[u].w * sc, hv.y, lv.y);
          const int rh = 32 * (qr >> 4) + (qr & 15);  // the hi row; the lo row is rh + 16
          uint8_t* dst = sQ + (ch >> 3) * C::Q_BOX + rh * 128 + (((ch & 7) ^ (rh & 7)) << 4) +
                         (c4 & 1) * 8;
          *reinterpret_cast<uint2*>(dst) = hv;
          *reinterpret_cast<uint2*>(dst + 16 * 128) = lv;
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(q_full);
      ++qn;

      float m_run = -INFINITY, l_run = 0.f;  // m_run: the pair's (both halves'); l_run: this half's
      for (int j = 0; j < ntile; ++j) {
        const int it_j = it + j, b = it_j % C::NPB;
        wait(&s_full[b], (it_j / C::NPB) & 1);
        tc_fence_after();
        // lane l < 16 of this warp's quadrant holds q_hi.K of pair i, lane l + 16 its q_lo.K:
        // each thread reads its lane's 64 columns, and the two swap halves so that this
        // thread keeps the hi + lo sum of its 32 columns [32 h, 32 h + 32)
        uint32_t sr[32], s0[32], s1[32];
        tmem_ld32(t_q + C::S_COL + b * C::TP, s0);
        tmem_ld32(t_q + C::S_COL + b * C::TP + 32, s1);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float y = __uint_as_float(__shfl_xor_sync(0xffffffffu, h ? s0[e] : s1[e], 16));
          sr[e] = __float_as_uint(__uint_as_float(h ? s1[e] : s0[e]) + y);
        }
        const int lim = lim0 - j * C::TP;  // columns [0, lim) of this thread's 32
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < 32; ++e)
          mq[e & 3] = fmaxf(mq[e & 3], e < lim ? __uint_as_float(sr[e]) : -INFINITY);
        float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));  // the pair's other half
        const bool grow = mt > m_run + C::RESCALE_LOG2;  // false while mt = -inf
        const bool resc = grow && m_run != -INFINITY;     // O holds weight: rescale it
        if (__any_sync(0xffffffffu, resc)) {
          // O must be final for tile it_j - 1 (this warp's lanes rescale their rows together)
          wait(&pv_done[(it_j - 1) % C::NPB], ((it_j - 1) / C::NPB) & 1);
          tc_fence_after();
          const float corr = resc ? ex2_approx(m_run - mt) : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < D / 64; ++cc) {  // this half's D / 2 columns, 32 at a time
            uint32_t o[32];
            tmem_ld16x2<D / 2>(t_q + C::O_COL + cc * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st16x2<D / 2>(t_q + C::O_COL + cc * 32, o);
          }
          tmem_st_wait();
          if (resc) l_run *= corr;
        }
        if (grow) m_run = mt;
        // P buffer b is free once P.V(it_j - NPB) has completed (earlier groups' all have)
        if (j >= C::NPB) {
          wait(&pv_done[b], ((it_j - C::NPB) / C::NPB) & 1);
        }
        const float mu = m_run == -INFINITY ? 0.f : m_run;  // lim <= 0 there: all weights 0
        float lq[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t ph[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float w0 = e < lim ? ex2_approx(__uint_as_float(sr[e]) - mu) : 0.f;
          const float w1 = e + 1 < lim ? ex2_approx(__uint_as_float(sr[e + 1]) - mu) : 0.f;
          lq[(e >> 1) & 3] += w0 + w1;
          ph[e >> 1] = h2_bits(__floats2half2_rn(w0, w1));
        }
        l_run += (lq[0] + lq[1]) + (lq[2] + lq[3]);
        // P row i, this half's 4 chunks of 8 positions
        uint8_t* prow = sP + b * C::P_BYTES + i * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(prow + (((4 * h + q) ^ (i & 7)) << 4)) =
              make_uint4(ph[4 * q], ph[4 * q + 1], ph[4 * q + 2], ph[4 * q + 3]);
        // V rows past the group's longest row may hold cache garbage: zero them (P is 0 there)
        const int nv = gr.lmax - (c0 + j * C::TP);
        if (nv < C::TP) {
          const int st = it_j % C::NST;
          wait(&full[st], (it_j / C::NST) & 1);
          uint8_t* sv = stages + st * C::STAGE_BYTES + C::KV_BYTES;
          const int n16 = (C::TP - nv) * 8;  // 16-byte pieces per box
          for (int e = threadIdx.x; e < C::NBOX * n16; e += 32 * C::NSW) {
            const int bx = e / n16, vr = nv + (e % n16) / 8, ch = e % 8;
            *reinterpret_cast<uint4*>(sv + bx * C::BOX_BYTES + vr * 128 + ch * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[b]);
      }

      // ---- epilogue: O final after the last tile's P.V; each thread moves its half of the
      //      pair's O row into the exchange area, then the warpgroup writes the records (or
      //      outputs) row by row, coalesced
      const int last = it + ntile - 1;
      wait(&pv_done[last % C::NPB], (last / C::NPB) & 1);
      it += ntile;
      tc_fence_after();
      const float l = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
      const float f = p.merge ? 1.f : (l > 0.f ? 1.f / l : 0.f);
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t o[32];
        tmem_ld16x2<D / 2>(t_q + C::O_COL + cc * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          xo[i * (D + 2) + h * (D / 2) + cc * 32 + e] = __uint_as_float(o[e]) * f;
      }
      if (h == 0) {
        xo[i * (D + 2) + D] = m_run == -INFINITY ? -INFINITY : m_run * kLn2;  // natural log
        xo[i * (D + 2) + D + 1] = l;
        xw[i] = rv && c0 < Lp;  // the pair has positions in this chunk
      }
      named_bar_sync(1, 32 * C::NSW);
      // the records (merge) or output rows, coalesced: a row's G heads are contiguous in both
      // (G (D + 2) floats of records, G D floats of output), copied as float2
      if (p.merge) {
        const int per_row = G * (D + 2) / 2;  // float2 pieces of a row's records
        for (int row = warp; row < gr.nr; row += C::NSW) {
          if (!xw[row * G]) continue;
          const float2* src = reinterpret_cast<const float2*>(xo) + row * per_row;
          float2* dst = reinterpret_cast<float2*>(
              p.part + (((size_t)(t0 + row) * p.n_split + c) * p.n_heads + g * G) * (D + 2));
#pragma unroll 4
          for (int e = lane; e < per_row; e += 32) dst[e] = src[e];
        }
      } else {
        for (int q = warp; q < gr.nr * G; q += C::NSW) {
          if (!xw[q]) continue;
          const float2* src = reinterpret_cast<const float2*>(xo + q * (D + 2));
          const int tq = t0 + q / G, hq = g * G + q % G;
          float2* dst = reinterpret_cast<float2*>(p.out + ((size_t)tq * p.n_heads + hq) * D);
#pragma unroll
          for (int e = lane; e < D / 2; e += 32) {
            const float2 y = src[e];
            dst[e] = make_float2(gated(p, tq, hq, 2 * e, y.x), gated(p, tq, hq, 2 * e + 1, y.y));
          }
        }
      }
      tc_fence_before();  // these TMEM reads precede the next group's MMAs (after q_full)
      named_bar_sync(1, 32 * C::NSW);  // the exchange area is read before the next q lands
      fence_async_smem();               // (generic reads before the next bulk copy's writes)
      mbar_arrive(x_free);
      if (p.merge && p.fused_merge) rows_fused_merge<D>(p, gr, k, g, c, seq_ok, merge_ok);
    }
    if (!ok && lane == 0) flag_error(p.err, GQA_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::ISSUER) {
    tc_fence_after();
    tmem_free(tbase, C::TMEM_COLS);
  }
  // this CTA's partials are written: the merge kernel launched after this one may be scheduled
  asm volatile("griddepcontrol.launch_dependents;");
}

}  // namespace gqa
