// tq_rows.cu -- TurboQuant decode for rows that share a sequence (a chunked-prefill step), on
// the tensor cores.
//
// flash_attention_tq.metal (cera 0.4.0 sources) serves a chunked-prefill step with the same
// kernel as decode, one threadgroup per (query head, row), each with its own causal window
// (row r at position p sees [0, p]); every row re-decodes the same compressed K/V.  Here one
// CTA serves a group of up to 64 / G rows of one sequence for one KV head and one chunk of
// positions: the group's (row, head) pairs -- up to 64 -- share every decoded tile.
//
// Per stage of 32 positions:
//   1. The packed rows arrive in a four-stage ring: polar words (and, at D = 128, the sign
//      words) by bulk copy issued by one thread, norms (and D = 64 sign words) by per-lane
//      cp.async, all counted on the stage's mbarrier.
//   2. The whole CTA decodes the stage once into shared memory as f16 planes, [position][slot]
//      with the 128-byte swizzle: the K centroids in hi and lo parts (c = hi + lo to about 22
//      bits), the QJL signs as +-1, the V centroids in hi and lo parts.  A polar word's 16
//      fields go to slots in the order 0 4 8 12 1 5 9 13 2 6 10 14 3 7 11 15 (what one shift,
//      one mask and two byte permutes produce); a sign word's 32 bits in the order 0 16 1 17 ..
//      15 31; the queries are laid out in the same orders, so the contractions are unchanged.
//   3. Each of the 8 warps contracts the decoded planes with its own 8 pairs: q.k as
//      mma.sync m16n8k16 with A = the K planes (ldmatrix), B = q_rot / q_jl in hi and lo parts;
//      the online softmax per pair with the pair's causal length masking positions; p.v with
//      A = the V planes (ldmatrix.trans), B = the weights in hi and lo parts.
// Decoding stage k + 1 overlaps the contractions of stage k (two decoded buffers, one CTA
// barrier per stage).  At the end of the chunk each warp holds its pairs' complete states: it
// normalises, rotates back and writes them, or writes rotated partials.  When the whole grid
// fits one CTA per SM (a cooperative launch) the group's chunk CTAs then merge those partials
// themselves: they meet on a counter in the workspace, and CTA c merges, rotates back and
// writes the group's pairs c NW + w, ... (tq_rows_fused_merge); otherwise merge_kernel,
// launched next as a programmatic dependent, does it, one warp per (row, head).  (A merge by
// each row's last chunk CTA left the rows' merges queued behind one another in whichever CTA
// finished last.)
#include <cuda_runtime_api.h>

#include "rows_mma.cuh"
#include "tq_frag.cuh"

namespace gqa {

cudaError_t ensure_smem(const void* fn, int bytes);  // launch_util.cu: the opt-in, once

template <int D>
struct TqRowsCfg {
  static constexpr int PW = D / 16, JW = D / 32;
  static constexpr int TPOS = 32;  // positions per stage
  static constexpr int NW = 8;     // warps; warp w serves pairs 8 w .. 8 w + 7
  static constexpr int NP = 8 * NW;
  static constexpr int NB = 2;     // n-blocks of 4 pairs per warp
  static constexpr int S = 4;      // packed stages in flight
  // packed stage, in words
  static constexpr int oKp = 0, oVp = TPOS * PW, oKj = 2 * TPOS * PW;
  static constexpr int oKn = oKj + TPOS * JW, oVn = oKn + TPOS, SW = oVn + TPOS;
  // decoded stage, in bytes: five planes of [TPOS][D] f16 in 128-byte swizzled boxes of 64 slots
  static constexpr int PLANE = TPOS * D * 2;
  static constexpr int dKh = 0, dKl = PLANE, dSg = 2 * PLANE, dVh = 3 * PLANE, dVl = 4 * PLANE;
  static constexpr int DEC = 5 * PLANE;
  static constexpr int RING_BYTES = S * SW * 4;
  static constexpr int DEC_OFF = align_up(RING_BYTES, 1024);
  static constexpr int MG_BYTES = NW * 8 * (D + 2) * 4;  // the warps' states, after the chunk
  static constexpr int Q_BYTES = 2 * NP * D * 4;         // the group's queries, at its start
  static constexpr int BAR_OFF = DEC_OFF + cmax(cmax(2 * DEC, MG_BYTES), Q_BYTES);
  static constexpr int SMEM = 1024 + BAR_OFF + S * 8;
  static_assert(oVp % 4 == 0 && oKj % 4 == 0 && oKn % 4 == 0 && SW % 4 == 0,
                "packed parts on 16-byte boundaries");
  static_assert(PLANE % 1024 == 0 && DEC_OFF % 1024 == 0, "swizzled planes on 1024-byte atoms");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// Dim of slot s of a 16-slot polar block, and of slot s of a 32-slot sign block.
__host__ __device__ constexpr int polar_dim(int s) { return 4 * (s % 4) + s / 4; }
__host__ __device__ constexpr int sign_dim(int s) { return s / 2 + 16 * (s % 2); }

// The fused merge of one group, run by every thread of every chunk CTA of the group (all
// resident under a cooperative launch), with the counter protocol of the tcgen05 row kernel's
// fused merge: each CTA stores and fences its partials and counts itself in on the group's
// counter, thread 0 waits (at most p.merge_spin polls) until all gridDim.x chunk CTAs are in,
// counts in a second time whatever happened (the CTA whose second count-in takes the counter
// to 2 gridDim.x resets it), and then warp w of CTA c merges the group's pairs c NW + w,
// c NW + w + gridDim.x NW, ... with merge_kernel's arithmetic, rotates them back and writes
// them.  A wait that runs out flags GQA_ERR_TIMEOUT and skips this CTA's share of the merge.
template <int D>
__device__ void tq_rows_fused_merge(const TqParams& tp, const RowGroup& gr, int k, int c,
                                    int Gc, int head0, bool seq_ok) {
  constexpr int DPL = D / 32, NW = TqRowsCfg<D>::NW;
  const PartialParams& p = tp.base;
  __shared__ int merge_ok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned int nctas = gridDim.x;
  unsigned int* cnt = p.counters + (size_t)k * gridDim.y + blockIdx.y;
  __threadfence();  // this thread's partial stores, device-wide
  __syncthreads();
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
    if (atomicAdd(cnt, 1u) == 2 * nctas - 1) atomicExch(cnt, 0u);
    if (!ok) flag_error(p.err, GQA_ERR_TIMEOUT);
    merge_ok = ok;
  }
  __syncthreads();
  if (merge_ok) {
    const size_t rec = (size_t)p.n_heads * (D + 2);  // floats between consecutive chunks
    const TqRotateBack<D> rot{tp.signs};
    for (int q = c * NW + warp; q < gr.nr * Gc; q += static_cast<int>(nctas) * NW) {
      const int t = gr.t0 + q / Gc, head = head0 + q % Gc;
      int dummy = 0;
      const int L = rows_len(p, t, seq_ok, &dummy);
      if (L == 0) continue;  // zeroed by the bookkeeping
      const int nv = min((L + p.chunk - 1) / p.chunk, p.n_split);
      const float* base = p.part + ((size_t)t * p.n_split * p.n_heads + head) * (D + 2);
      float a[DPL];
#pragma unroll
      for (int e = 0; e < DPL; ++e) a[e] = 0.f;
      float M = -INFINITY, Ls = 0.f;  // Ls: this lane's share of the sum
      for (int cb = 0; cb < nv; cb += 32) {
        const int nb = min(32, nv - cb);
        float m = -INFINITY, l = 0.f;
        if (lane < nb) {
          m = __ldcg(base + (cb + lane) * rec + D);
          l = __ldcg(base + (cb + lane) * rec + D + 1);
        }
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
        const float* ac = base + cb * rec + lane * DPL;
#pragma unroll 4
        for (int j = 0; j < nb; ++j) {
          const float wj = __shfl_sync(0xffffffffu, w, j);
#pragma unroll
          for (int e = 0; e < DPL; e += 2) {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(ac + j * rec + e));
            a[e] = fmaf(wj, v.x, a[e]);
            a[e + 1] = fmaf(wj, v.y, a[e + 1]);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) a[e] *= inv;
      rot(a, head, lane);
      float* o = p.out + ((size_t)t * p.n_heads + head) * D + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[e] = gated(p, t, head, lane * DPL + e, a[e]);
    }
  }
  __syncthreads();  // merge_ok is read before a later group's merge writes it
}

template <int D>
__global__ void __launch_bounds__(32 * TqRowsCfg<D>::NW, 1) tq_rows_kernel(const TqParams tp) {
  using C = TqRowsCfg<D>;
  constexpr int PW = C::PW, JW = C::JW, TPOS = C::TPOS, NB = C::NB, S = C::S;
  const PartialParams& p = tp.base;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* base = smem_raw + pad;
  uint32_t* ring = reinterpret_cast<uint32_t*>(base);
  uint8_t* dec = base + C::DEC_OFF;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::BAR_OFF);
  const int c = blockIdx.x, slot = blockIdx.z, nslots = gridDim.z;
  const TqCta cta = tq_cta(p);
  const int g = cta.g, Gc = cta.G;
  const int R = C::NP / Gc;  // rows per group at most
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int fr = lane >> 2, fq = lane & 3;
  const int c0 = c * p.chunk;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&full[i], 33);  // warp 0: one expect_tx, 32 cp.async
    mbar_init_fence();
  }
  __syncthreads();

  // centroid tables (hi and lo planes, scaled by a power of two), as in tq_mma.cu
  const float sc = pow2_scale(fmaxf(fmaxf(fabsf(tp.c0), fabsf(tp.c1)), fmaxf(fabsf(tp.c2), fabsf(tp.c3))));
  uint32_t th01, th23, tl01, tl23;
  split_hi_lo(tp.c0 * sc, tp.c1 * sc, th01, tl01);
  split_hi_lo(tp.c2 * sc, tp.c3 * sc, th23, tl23);
  const int part = fr & 1;
  const int mi = lane >> 3, rr = lane & 7;  // ldmatrix roles

  int scan_t = 0, scan_cnt = 0;
  long long gs = 0;  // stages issued so far over all groups: ring slot gs % S, phase gs / S
  bool ok = true;
  for (int k = slot;; k += nslots) {
    const int t0 = rows_find_leader(p, R, k, scan_t, scan_cnt, lane);
    if (t0 < 0) break;
    const RowGroup gr = rows_group(p, t0, R, lane);
    const bool seq_ok = gr.s >= 0 && gr.s < p.n_seq;
    if (c == 0 && warp == 0) {  // per-row bookkeeping: flags, chunk counts, empty rows
      for (int jb = 0; jb < gr.nr; jb += 32) {
        int err = 0;
        const int L = jb + lane < gr.nr ? rows_len(p, t0 + jb + lane, seq_ok, &err) : 0;
        if (jb + lane < gr.nr && cta.col == 0) {
          if (err) flag_error(p.err, err);
          if (p.merge) p.n_valid[t0 + jb + lane] = (L + p.chunk - 1) / p.chunk;
        }
        for (int jj = 0; jj < 32 && jb + jj < gr.nr; ++jj) {
          if (__shfl_sync(0xffffffffu, L, jj) != 0) continue;  // empty row: zeros
          for (int e = lane; e < Gc * D; e += 32)
            p.out[((size_t)(t0 + jb + jj) * p.n_heads + cta.head0 + e / D) * D + e % D] = 0.f;
        }
      }
    }
    const int c1 = min(c0 + p.chunk, gr.lmax);
    if (c1 <= c0) {  // the same for every warp
      if (p.merge && p.fused_merge) tq_rows_fused_merge<D>(tp, gr, k, c, Gc, cta.head0, seq_ok);
      continue;
    }
    const int nst = (c1 - c0 + TPOS - 1) / TPOS;
    const size_t hrow0 = ((size_t)(seq_ok ? gr.s : 0) * p.n_kv_heads + g) * p.cache_cap;

    // ---- this warp's pairs: B columns (pair 8 w + 4 nb + fr / 2) and C state (8 w + 4 nb + fq)
    const int np = gr.nr * Gc;  // real pairs of the group
    int Lq[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int q = 8 * warp + 4 * nb + fq;
      int dummy = 0;
      Lq[nb] = q < np ? rows_len(p, t0 + q / Gc, seq_ok, &dummy) : 0;
    }
    uint32_t qb[PW][NB][2], qjb[2 * JW][NB][2];
    float sp, sj;
    {
      // the group's queries, staged by coalesced loads into the (not yet used) decoded buffers:
      // q_rot [pair][D] then q_jl [pair][D]
      float* qs = reinterpret_cast<float*>(dec);
      float* qjs = qs + C::NP * D;
      for (int i = tid; i < np * (D / 4); i += 32 * C::NW) {
        const int q = i / (D / 4), d4 = i % (D / 4);
        const size_t qi = ((size_t)(t0 + q / Gc) * p.n_heads + cta.head0 + q % Gc) * D + 4 * d4;
        reinterpret_cast<float4*>(qs)[i] = __ldg(reinterpret_cast<const float4*>(tp.q_rot + qi));
        reinterpret_cast<float4*>(qjs)[i] = __ldg(reinterpret_cast<const float4*>(tp.q_jl + qi));
      }
      __syncthreads();
      const int nq = min(8, max(np - 8 * warp, 0));  // the warp's real pairs
      float amr = 0.f, amj = 0.f;  // their max |q|, for the power-of-two scales
      for (int i = lane; i < nq * D; i += 32) {
        amr = fmaxf(amr, fabsf(qs[8 * warp * D + i]));
        amj = fmaxf(amj, fabsf(qjs[8 * warp * D + i]));
      }
      const float sr = pow2_scale(warp_max(amr)), sjq = pow2_scale(warp_max(amj));
      sp = p.scale_log2 / (sr * sc);
      sj = p.scale_log2 * tp.qjl_scale / sjq;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int q = 8 * warp + 4 * nb + (fr >> 1);
        const bool hv = q < np;
        const float* qrot = qs + (hv ? q : 0) * D;
        const float* qjl = qjs + (hv ? q : 0) * D;
#pragma unroll
        for (int kb = 0; kb < PW; ++kb) {
          const int d = 16 * kb;
          qb[kb][nb][0] = hv ? f16_part(qrot[d + polar_dim(2 * fq)] * sr,
                                        qrot[d + polar_dim(2 * fq + 1)] * sr, part) : 0u;
          qb[kb][nb][1] = hv ? f16_part(qrot[d + polar_dim(2 * fq + 8)] * sr,
                                        qrot[d + polar_dim(2 * fq + 9)] * sr, part) : 0u;
        }
#pragma unroll
        for (int ks = 0; ks < 2 * JW; ++ks) {
          const int d = 32 * (ks / 2), s0 = 16 * (ks % 2);
          qjb[ks][nb][0] = hv ? f16_part(qjl[d + sign_dim(s0 + 2 * fq)] * sjq,
                                         qjl[d + sign_dim(s0 + 2 * fq + 1)] * sjq, part) : 0u;
          qjb[ks][nb][1] = hv ? f16_part(qjl[d + sign_dim(s0 + 2 * fq + 8)] * sjq,
                                         qjl[d + sign_dim(s0 + 2 * fq + 9)] * sjq, part) : 0u;
        }
      }
      __syncthreads();  // the staging area is read before the first stage decodes into it
    }
    const bool active = 8 * warp < np;  // the warp has real pairs (warp-uniform)

    // ---- the packed ring: warp 0 issues stage i of this group into ring slot (gs0 + i) % S
    const long long gs0 = gs;
    auto issue = [&](int i) {
      const long long gi = gs0 + i;
      uint32_t* st = ring + (gi % S) * C::SW;
      uint64_t* bar = &full[gi % S];
      const int p0 = c0 + TPOS * i;
      const int n = min(TPOS, c1 - p0);
      const size_t row = hrow0 + p0;
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        constexpr bool kBulkJ = JW == 4;
        mbar_arrive_expect_tx(bar, n * (2 * PW + (kBulkJ ? JW : 0)) * 4);
        bulk_load(st + C::oKp, tp.k_polar + row * PW, n * PW * 4, bar);
        bulk_load(st + C::oVp, tp.v_polar + row * PW, n * PW * 4, bar);
        if (kBulkJ) bulk_load(st + C::oKj, tp.k_jl + row * JW, n * JW * 4, bar);
      }
      const size_t r = row + (lane < n ? lane : 0);  // a valid row for every lane
      cp_async_4(st + C::oKn + lane, tp.k_norms + r);
      cp_async_4(st + C::oVn + lane, tp.v_norms + r);
      if constexpr (JW == 2) cp_async_8(st + C::oKj + 2 * lane, tp.k_jl + r * 2);
      cp_async_arrive_noinc(bar);
    };
    auto wait_stage = [&](int i) {
      const long long gi = gs0 + i;
      return mbar_wait(&full[gi % S], (uint32_t)((gi / S) & 1));
    };
    // decode packed stage i into decoded buffer i & 1 (all threads)
    auto decode = [&](int i) {
      const uint32_t* st = ring + ((gs0 + i) % S) * C::SW;
      uint8_t* db = dec + (i & 1) * C::DEC;
      for (int it = tid; it < TPOS * PW; it += 32 * C::NW) {  // (position, polar word)
        const int kb = it / TPOS, pos = it % TPOS;
        const uint32_t wk = st[C::oKp + pos * PW + kb], wv = st[C::oVp + pos * PW + kb];
        uint32_t kh[8], kl[8], vh[8], vl[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t s0, s1;
          field_sel((wk >> (2 * j)) & 0x03030303u, s0, s1);
          kh[2 * j] = prmt(th01, th23, s0);
          kh[2 * j + 1] = prmt(th01, th23, s1);
          kl[2 * j] = prmt(tl01, tl23, s0);
          kl[2 * j + 1] = prmt(tl01, tl23, s1);
          field_sel((wv >> (2 * j)) & 0x03030303u, s0, s1);
          vh[2 * j] = prmt(th01, th23, s0);
          vh[2 * j + 1] = prmt(th01, th23, s1);
          vl[2 * j] = prmt(tl01, tl23, s0);
          vl[2 * j + 1] = prmt(tl01, tl23, s1);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // slots 8 h .. 8 h + 7: chunk 2 kb + h
          const uint32_t off = swz_off(pos, 2 * kb + h, TPOS);
          *reinterpret_cast<uint4*>(db + C::dKh + off) = make_uint4(kh[4 * h], kh[4 * h + 1], kh[4 * h + 2], kh[4 * h + 3]);
          *reinterpret_cast<uint4*>(db + C::dKl + off) = make_uint4(kl[4 * h], kl[4 * h + 1], kl[4 * h + 2], kl[4 * h + 3]);
          *reinterpret_cast<uint4*>(db + C::dVh + off) = make_uint4(vh[4 * h], vh[4 * h + 1], vh[4 * h + 2], vh[4 * h + 3]);
          *reinterpret_cast<uint4*>(db + C::dVl + off) = make_uint4(vl[4 * h], vl[4 * h + 1], vl[4 * h + 2], vl[4 * h + 3]);
        }
      }
      for (int it = tid; it < TPOS * JW; it += 32 * C::NW) {  // (position, sign word)
        const int w = it / TPOS, pos = it % TPOS;
        const uint32_t z = st[C::oKj + pos * JW + w];
        uint32_t sg[16];
#pragma unroll
        for (int b = 0; b < 16; ++b) sg[b] = ((z * (1u << (15 - b))) & 0x80008000u) ^ 0xBC00BC00u;
#pragma unroll
        for (int h = 0; h < 4; ++h)  // slots 8 h .. 8 h + 7 of the word's 32: chunk 4 w + h
          *reinterpret_cast<uint4*>(db + C::dSg + swz_off(pos, 4 * w + h, TPOS)) =
              make_uint4(sg[4 * h], sg[4 * h + 1], sg[4 * h + 2], sg[4 * h + 3]);
      }
    };

    float acc[PW][NB][4], m_run[NB], l_run[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      m_run[nb] = -INFINITY;
      l_run[nb] = 0.f;
#pragma unroll
      for (int mb = 0; mb < PW; ++mb) acc[mb][nb][0] = acc[mb][nb][1] = acc[mb][nb][2] = acc[mb][nb][3] = 0.f;
    }

    if (warp == 0)
      for (int i = 0; i < S && i < nst; ++i) issue(i);
    ok = __all_sync(0xffffffffu, wait_stage(0)) && ok;
    decode(0);
    __syncthreads();

    for (int i = 0; i < nst; ++i) {
      if (i + 1 < nst) {
        ok = __all_sync(0xffffffffu, wait_stage(i + 1)) && ok;
        decode(i + 1);
      }
      const uint32_t* st = ring + ((gs0 + i) % S) * C::SW;
      const uint32_t db = smem_addr(dec + (i & 1) * C::DEC);
      const int pb0 = c0 + TPOS * i;        // the stage's first position
      const int nv = min(TPOS, c1 - pb0);    // positions of the chunk in it
      const int nm = nv > 16 ? 2 : 1;
      if (active) {
        float x[2][NB][2];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          if (m >= nm) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) x[m][nb][0] = x[m][nb][1] = -INFINITY;
            continue;
          }
          float pol[NB][4], pol2[NB][4], jl[NB][4], jl2[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) pol[nb][e] = pol2[nb][e] = jl[nb][e] = jl2[nb][e] = 0.f;
          const int ar = 16 * m + (mi & 1) * 8 + rr;  // this lane's ldmatrix row (position)
#pragma unroll
          for (int kb = 0; kb < PW; ++kb) {
            uint32_t ah[4], al[4];
            const uint32_t off = swz_off(ar, 2 * kb + (mi >> 1), TPOS);
            ldsm_x4(ah, db + C::dKh + off);
            ldsm_x4(al, db + C::dKl + off);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              mma_f16(pol[nb], ah, qb[kb][nb][0], qb[kb][nb][1]);
              mma_f16(pol2[nb], al, qb[kb][nb][0], qb[kb][nb][1]);
            }
          }
#pragma unroll
          for (int ks = 0; ks < 2 * JW; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, db + C::dSg + swz_off(ar, 2 * ks + (mi >> 1), TPOS));
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              if (ks & 1) mma_f16(jl2[nb], a, qjb[ks][nb][0], qjb[ks][nb][1]);
              else mma_f16(jl[nb], a, qjb[ks][nb][0], qjb[ks][nb][1]);
            }
          }
          const int r0 = 16 * m + fr, r1 = r0 + 8;
          const uint32_t kn0 = st[C::oKn + r0], kn1 = st[C::oKn + r1];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const float P0 = (pol[nb][0] + pol2[nb][0]) + (pol[nb][1] + pol2[nb][1]);
            const float P1 = (pol[nb][2] + pol2[nb][2]) + (pol[nb][3] + pol2[nb][3]);
            const float J0 = (jl[nb][0] + jl2[nb][0]) + (jl[nb][1] + jl2[nb][1]);
            const float J1 = (jl[nb][2] + jl2[nb][2]) + (jl[nb][3] + jl2[nb][3]);
            // positions at or past the pair's own length are selected away, never multiplied
            x[m][nb][0] = pb0 + r0 < Lq[nb] ? half_lo(kn0) * fmaf(half_hi(kn0) * sj, J0, P0 * sp) : -INFINITY;
            x[m][nb][1] = pb0 + r1 < Lq[nb] ? half_lo(kn1) * fmaf(half_hi(kn1) * sj, J1, P1 * sp) : -INFINITY;
          }
        }

        // online softmax per pair over the stage; the p.v weights of both m-blocks
        uint32_t pbw[2][NB][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          float mx = fmaxf(fmaxf(x[0][nb][0], x[0][nb][1]), fmaxf(x[1][nb][0], x[1][nb][1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[nb], mx);
          // a pair with no position yet keeps an empty state instead of forming -inf - -inf
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          const float corr = fast_exp2(m_run[nb] - m_use);
          float pr[2][2];
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            pr[m][0] = fast_exp2(x[m][nb][0] - m_use);
            pr[m][1] = fast_exp2(x[m][nb][1] - m_use);
          }
          l_run[nb] = fmaf(l_run[nb], corr, (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
          if (__any_sync(0xffffffffu, m_new > m_run[nb])) {
#pragma unroll
            for (int mb = 0; mb < PW; ++mb)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[mb][nb][e] *= corr;
          }
          m_run[nb] = m_new;
          const bool hv = 8 * warp + 4 * nb + (fr >> 1) < np;
          const int la = 8 * fq + (fr >> 1), lb = la + 4;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const float vn0 = half_lo(st[C::oVn + 16 * m + fr]);
            const float vn1 = half_lo(st[C::oVn + 16 * m + fr + 8]);
            const float v0 = pr[m][0] > 0.f ? pr[m][0] * vn0 : 0.f;
            const float v1 = pr[m][1] > 0.f ? pr[m][1] * vn1 : 0.f;
            const float e0 = __shfl_sync(0xffffffffu, v0, la), e1 = __shfl_sync(0xffffffffu, v0, lb);
            const float e2 = __shfl_sync(0xffffffffu, v1, la), e3 = __shfl_sync(0xffffffffu, v1, lb);
            pbw[m][nb][0] = hv ? f16_part(e0, e1, part) : 0u;
            pbw[m][nb][1] = hv ? f16_part(e2, e3, part) : 0u;
          }
        }

        // p.v: A = the V planes transposed (rows = slots of a 16-dim block, k = positions)
#pragma unroll
        for (int mb = 0; mb < PW; ++mb) {
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            if (m >= nm) continue;
            uint32_t ah[4], al[4];
            const uint32_t off = swz_off(16 * m + (mi >> 1) * 8 + rr, 2 * mb + (mi & 1), TPOS);
            ldsm_x4_t(ah, db + C::dVh + off);
            ldsm_x4_t(al, db + C::dVl + off);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              mma_f16(acc[mb][nb], ah, pbw[m][nb][0], pbw[m][nb][1]);
              mma_f16(acc[mb][nb], al, pbw[m][nb][0], pbw[m][nb][1]);
            }
          }
        }
      }
      __syncthreads();  // decoded buffer i is free, buffer i + 1 is visible, ring slot i is free
      if (warp == 0 && i + S < nst) issue(i + S);
    }
    gs = gs0 + nst;

    // ---- the warps' pair states into shared memory (the decoded buffers are no longer read)
    float* mg = reinterpret_cast<float*>(dec);  // [NW][8][D + 2]
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float l = l_run[nb];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      float* r = mg + (warp * 8 + 4 * nb + fq) * (D + 2);
      const float sv = 1.f / sc;
#pragma unroll
      for (int mb = 0; mb < PW; ++mb) {
        r[16 * mb + polar_dim(fr)] = (acc[mb][nb][0] + acc[mb][nb][1]) * sv;
        r[16 * mb + polar_dim(fr + 8)] = (acc[mb][nb][2] + acc[mb][nb][3]) * sv;
      }
      if (fr == 0) {
        r[D] = m_run[nb];
        r[D + 1] = l;
      }
    }
    __syncwarp();
    // each warp finishes its own pairs: the output row (normalised, rotated back, gated) or the
    // chunk's rotated partial
    {
      constexpr int DPL = D / 32;
      const TqRotateBack<D> rot{tp.signs};
      for (int j = 0; j < 8; ++j) {
        const int q = 8 * warp + j;
        if (q >= np) break;
        const int t = t0 + q / Gc, head = cta.head0 + q % Gc;
        int dummy = 0;
        if (c0 >= rows_len(p, t, seq_ok, &dummy)) continue;  // no position of this row here
        const float* r = mg + (warp * 8 + j) * (D + 2);
        float a[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) a[e] = r[lane * DPL + e];
        const float M = r[D], Ls = r[D + 1];
        if (p.merge) {
          float* pr = p.part + (((size_t)t * p.n_split + c) * p.n_heads + head) * (D + 2);
#pragma unroll
          for (int e = 0; e < DPL; ++e) pr[lane * DPL + e] = a[e];
          if (lane == 0) {
            pr[D] = M == -INFINITY ? -INFINITY : M * kLn2;  // natural-log units
            pr[D + 1] = Ls;
          }
        } else {
          const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
          for (int e = 0; e < DPL; ++e) a[e] *= inv;
          rot(a, head, lane);
          float* o = p.out + ((size_t)t * p.n_heads + head) * D + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[e] = gated(p, t, head, lane * DPL + e, a[e]);
        }
      }
    }
    __syncthreads();  // the state area is read before the next group decodes into it
    if (p.merge && p.fused_merge) tq_rows_fused_merge<D>(tp, gr, k, c, Gc, cta.head0, seq_ok);
  }
  if (!ok && lane == 0) flag_error(p.err, GQA_ERR_TIMEOUT);
  // this CTA's partials are written: the merge kernel launched after this one may be scheduled
  asm volatile("griddepcontrol.launch_dependents;");
}

template <int D>
static cudaError_t launch_rows(dim3 grid, const TqParams& tp, cudaStream_t stream) {
  using C = TqRowsCfg<D>;
  const void* fn = reinterpret_cast<const void*>(&tq_rows_kernel<D>);
  cudaError_t e = ensure_smem(fn, C::SMEM);
  if (e != cudaSuccess) return e;
  // with the fused merge the chunk CTAs of a group wait for one another: a cooperative launch
  // guarantees they are all resident
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(32 * C::NW);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = tp.base.fused_merge ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tq_rows_kernel<D>, tp);
}

cudaError_t launch_tq_rows(int head_dim, dim3 grid, const TqParams& tp, cudaStream_t stream) {
  return head_dim == 64 ? launch_rows<64>(grid, tp, stream) : launch_rows<128>(grid, tp, stream);
}

}  // namespace gqa
