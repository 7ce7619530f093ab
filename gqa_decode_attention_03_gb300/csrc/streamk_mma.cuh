// streamk_mma.cuh -- f16 decode attention with a stream-K work split over a persistent grid.
//
// The work of a step is the concatenation, row by row and KV head by KV head, of every
// (row t, KV head g) "segment" of n_t visited positions: W = n_kv_heads * sum_t n_t positions.
// CTA i of P takes exactly the positions [i W / P, (i + 1) W / P) of that stream, so every CTA
// reads the same number of K/V bytes whatever the mix of sequence lengths (a batch with lengths
// spread over 1K..32K has no long-row tail).  A segment cut by CTA boundaries becomes a few
// "pieces".  At the end of a piece the CTA merges its warps' row slices in shared memory; a
// segment that lies inside one share is written out at once, otherwise the CTA writes one
// partial record per piece (the chunk partials of qsa2.metal's qsa_attn2, here in log2 units)
// and takes a ticket on the segment's counter, and the CTA holding the last ticket merges the
// segment's records by log-sum-exp (qsa_merge2) and writes the output.  Tickets use atomicInc
// with the segment's piece count as the wrap limit, so the counters are zero again after every
// call.  Nothing ever waits on another CTA.
//
// Inside a piece the math is the tensor-core kernel's (partial_mma.cuh): TMA producer warp,
// three-stage mbarrier ring that runs on across piece boundaries, mma.sync m16n8k16 for q.k^T
// and p.v with f16 hi/lo splits of q and p, lazy online-softmax rescale.
#pragma once

#include "partial_mma.cuh"

namespace gqa {

constexpr int kStreamKMaxRows = 8192;  // rows whose prefix fits in the stage ring at set-up

// Visited length of row t after the kernel-side clamps (f16 caches: dense rows).
__device__ __forceinline__ int sk_row_len(const PartialParams& p, int t, int* errbits) {
  int L = __ldg(p.kv_len + t);
  const int lmax = static_cast<int>(p.cache_cap < p.max_kv_len ? p.cache_cap : p.max_kv_len);
  if (L < 0 || L > lmax) {
    *errbits |= GQA_ERR_KVLEN_RANGE;
    L = L < 0 ? 0 : lmax;
  }
  const int s = p.seq_of ? __ldg(p.seq_of + t) : t;
  if (s < 0 || s >= p.n_seq) {
    *errbits |= GQA_ERR_SEQ_RANGE;
    L = 0;
  }
  return L;
}

// Position of the stream -> the CTA whose share holds it: largest i with floor(i W / P) <= w.
__device__ __forceinline__ int sk_cta_of(long long w, long long W, int P) {
  const long long i = ((w + 1) * P + W - 1) / W - 1;
  return static_cast<int>(i < P - 1 ? i : P - 1);
}

// A forward walk over the stream from a CTA's first position.
struct SkWalk {
  int t, g, a;  // row, KV head, offset inside the segment
  int n;        // visited length of row t
  long long w;  // stream position of (t, g, a)
};

__device__ __forceinline__ void sk_next_row(const PartialParams& p, SkWalk& it) {
  int dummy = 0;
  do {
    ++it.t;
    it.n = it.t < p.n_tok ? sk_row_len(p, it.t, &dummy) : 1;
  } while (it.t < p.n_tok && it.n == 0);
  it.g = 0;
  it.a = 0;
}

// Takes the next piece [a, b) of segment (t, g) that lies before w_end; advances the walk.
__device__ __forceinline__ int sk_take(const PartialParams& p, SkWalk& it, long long w_end,
                                       int& t, int& g, int& a, int& b, int& n,
                                       long long& seg_start) {
  t = it.t;
  g = it.g;
  a = it.a;
  n = it.n;
  const long long left = w_end - it.w;
  const int take = static_cast<int>(left < (long long)(it.n - it.a) ? left : (it.n - it.a));
  b = a + take;
  seg_start = it.w - it.a;
  it.w += take;
  it.a += take;
  if (it.a == it.n) {
    it.a = 0;
    if (++it.g == p.n_kv_heads) sk_next_row(p, it);
  }
  return take;
}

// The CTA that finished segment (t, g) last merges its pieces' records (record id
// piece = cta + seg for the CTAs i_first..i_last, consecutive in memory) by log-sum-exp in log2
// units (qsa2.metal, qsa_merge2) and writes out.  One warp per head: lane c holds piece c's
// (m, l) and its weight, which reach the other lanes by shuffle, so the record loads of a head
// go out in one round.
template <int D>
__device__ __forceinline__ void sk_merge_segment(const PartialParams& p, int t, int g, int seg,
                                                 int i_first, int i_last, int warp, int nwarps,
                                                 int lane) {
  constexpr int DPL = D / 32;
  const int G = p.group;
  const int nrec = i_last - i_first + 1;
  const size_t rec_f = (size_t)G * (D + 2);
  const float* first = p.part + (size_t)(i_first + seg) * rec_f;
  for (int h = warp; h < G; h += nwarps) {
    const float* hrow = first + (size_t)h * (D + 2);
    float M = -INFINITY;
    for (int r = lane; r < nrec; r += 32) M = fmaxf(M, __ldcg(hrow + r * rec_f + D));
    M = warp_max(M);
    float a[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) a[k] = 0.f;
    float Ls = 0.f;
    if (M != -INFINITY) {
      for (int r0 = 0; r0 < nrec; r0 += 32) {
        const int r = r0 + lane;
        float e = 0.f;
        if (r < nrec) {
          const float m = __ldcg(hrow + r * rec_f + D);
          e = m == -INFINITY ? 0.f : fast_exp2(m - M);
          Ls = fmaf(__ldcg(hrow + r * rec_f + D + 1), e, Ls);
        }
        const int nb = min(32, nrec - r0);
#pragma unroll 8
        for (int j = 0; j < nb; ++j) {
          const float ej = __shfl_sync(0xffffffffu, e, j);
          const float* rp = hrow + (size_t)(r0 + j) * rec_f + lane * DPL;
#pragma unroll
          for (int k = 0; k < DPL; k += 2) {
            const float2 v = __ldcg(reinterpret_cast<const float2*>(rp + k));
            a[k] = fmaf(ej, v.x, a[k]);
            a[k + 1] = fmaf(ej, v.y, a[k + 1]);
          }
        }
      }
      Ls = warp_sum(Ls);
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    float* o = p.out + ((size_t)t * p.n_heads + g * G + h) * D + lane * DPL;
#pragma unroll
    for (int k = 0; k < DPL; k += 2)
      *reinterpret_cast<float2*>(o + k) =
          make_float2(gated(p, t, g * G + h, lane * DPL + k, a[k] * inv),
                      gated(p, t, g * G + h, lane * DPL + k + 1, a[k + 1] * inv));
  }
}

template <int D, int NHG>
__global__ void __launch_bounds__(MmaCfg<D, NHG>::MAX_THREADS, MmaCfg<D, NHG>::MIN_BLOCKS)
    streamk_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const PartialParams p) {
  using C = MmaCfg<D, NHG>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ long long s_w0, s_W;
  __shared__ int s_t0, s_g0, s_a0, s_n0, s_last;
  const int cta = blockIdx.x;
  int P = gridDim.x;  // shares: min(grid, W) after the set-up, so that none is empty
  const int G = p.group, Hk = p.n_kv_heads, T = p.n_tok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  uint8_t* stages = smem_raw + pad;
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::NST * C::STAGE_BYTES);
  uint64_t* empty = full + C::NST;
  float* ms = reinterpret_cast<float*>(empty + C::NST);  // [NPS][G][D + 2] slice merge area

  // ---- set-up: per-row visited lengths and their prefix, in the (not yet used) stage ring
  {
    long long* pre = reinterpret_cast<long long*>(stages);  // [T + 1]
    int errs = 0;
    const int nthr = blockDim.x;
    const int per = (T + nthr - 1) / nthr;
    const int r0 = threadIdx.x * per, r1 = min(T, r0 + per);
    long long run = 0;
    for (int t = r0; t < r1; ++t) {
      const int n = sk_row_len(p, t, &errs);
      pre[t] = n;  // lengths first, turned into prefix sums below
      run += n;
      if (n == 0 && t % P == cta)  // empty context: zeros (flash_attention.metal)
        for (int i = 0; i < p.n_heads * D; ++i) p.out[(size_t)t * p.n_heads * D + i] = 0.f;
    }
    if (cta == 0 && errs) flag_error(p.err, errs);
    // exclusive scan of the per-thread sums (one warp scans the warp totals)
    __shared__ long long s_wsum[32];
    long long x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      long long z = lane < (nthr >> 5) ? s_wsum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      if (lane < (nthr >> 5)) s_wsum[lane] = z;  // inclusive warp totals
    }
    __syncthreads();
    long long base = (x - run) + (warp > 0 ? s_wsum[warp - 1] : 0);  // exclusive prefix
    for (int t = r0; t < r1; ++t) {
      const long long n = pre[t];
      pre[t] = base;
      base += n;
    }
    if (threadIdx.x == nthr - 1) pre[T] = base;
    __syncthreads();
    if (threadIdx.x == 0) {
      const long long W = (long long)Hk * pre[T];
      const int Pe = (long long)P < W ? P : static_cast<int>(W);
      const long long w0 = cta < Pe ? W * cta / Pe : W;
      s_W = W;
      s_w0 = w0;
      if (w0 < W) {
        int lo = 0, hi = T - 1;  // largest t with Hk * pre[t] <= w0
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if ((long long)Hk * pre[mid] <= w0) lo = mid; else hi = mid - 1;
        }
        const int n = static_cast<int>(pre[lo + 1] - pre[lo]);
        const long long off = w0 - (long long)Hk * pre[lo];
        s_t0 = lo;
        s_n0 = n;
        s_g0 = static_cast<int>(off / n);
        s_a0 = static_cast<int>(off % n);
      }
    }
    __syncthreads();
  }
  const long long W = s_W, w0 = s_w0;
  if ((long long)P > W) P = static_cast<int>(W);
  if (cta >= P) return;  // more CTAs than positions: this one has no share
  const long long w1 = W * (cta + 1) / P;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C::NCW);
    }
    mbar_init_fence();
  }
  __syncthreads();  // also: nobody reads the set-up prefix any more

  SkWalk walk{s_t0, s_g0, s_a0, s_n0, w0};

  if (warp == C::NCW) {  // ---- producer warp: lane 0 streams every tile of every piece
    if (lane != 0) return;
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    int it = 0;
    bool ok = true;
    while (ok && walk.w < w1) {
      int t, g, a, b, n;
      long long ss;
      sk_take(p, walk, w1, t, g, a, b, n, ss);
      const int seq = p.seq_of ? __ldg(p.seq_of + t) : t;
      const int z0 = seq * static_cast<int>(p.cache_cap) + a;
      for (int k = 0; k < b - a; k += C::TP, ++it) {
        const int st = it % C::NST;
        if (it >= C::NST && !mbar_wait(&empty[st], ((it / C::NST) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], C::KV_BYTES);
        uint8_t* sk = stages + st * C::STAGE_BYTES;
        uint8_t* sv = sk + C::NBOX * C::BOX_BYTES;
#pragma unroll
        for (int bx = 0; bx < C::NBOX; ++bx) {
          tma_load_3d(sk + bx * C::BOX_BYTES, &tmK, bx * 64, g, z0 + k, &full[st]);
          tma_load_3d(sv + bx * C::BOX_BYTES, &tmV, bx * 64, g, z0 + k, &full[st]);
        }
      }
    }
    if (!ok) flag_error(p.err, GQA_ERR_TIMEOUT);
    for (int st = 0; st < C::NST && st < it; ++st) {  // the last load of each stage lands first
      const int last = st + ((it - 1 - st) / C::NST) * C::NST;
      if (!mbar_wait(&full[st], (last / C::NST) & 1)) flag_error(p.err, GQA_ERR_TIMEOUT);
    }
    return;
  }

  // ---- consumer warps: w = (slice * NHG + hg) * DSPLIT + dh
  const int gid = lane >> 2, tig = lane & 3;
  const int dh = warp % C::DSPLIT;
  const int hg = (warp / C::DSPLIT) % NHG;
  const int slice = warp / (C::DSPLIT * NHG);
  const int hh = hg * 8 + gid;
  const bool hv = hh < G;
  const int mi = lane >> 3, rr = lane & 7;
  int it = 0;
  bool ok = true;

  while (walk.w < w1) {
    int t, g, a, b, n_row;
    long long seg_start;
    sk_take(p, walk, w1, t, g, a, b, n_row, seg_start);
    const int seg = t * Hk + g;

    uint32_t qa[C::KS][4];
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
    float m_run = -INFINITY, l_run = 0.f;

    for (int k = 0; ok && k < b - a; k += C::TP, ++it) {
      const int st = it % C::NST;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (it / C::NST) & 1));
      if (!ok) break;
      const uint32_t sk = smem_addr(stages + st * C::STAGE_BYTES);
      const uint32_t sv = sk + C::NBOX * C::BOX_BYTES;
#pragma unroll
      for (int bb = 0; bb < C::NB16; ++bb) {
        const int r0 = slice * C::TPW + bb * 16;
        const int nv = min(max(b - a - k - r0, 0), 16);
        if (nv == 0) continue;
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
          for (int j = 0; j < 2; ++j) {
            const float v = sc[nt][j] + sc[nt][2 + j];
            x[nt][j] = (nt * 8 + 2 * tig + j) < nv ? v : -INFINITY;
            mt = fmaxf(mt, x[nt][j]);
          }
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
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
          const int chunk = (dh * C::DW + np * 16) / 8 + (mi >> 1);
          ldsm_x4_t(vb, sv + swz_off(r0 + (mi & 1) * 8 + rr, chunk, C::TP));
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
    if (!ok) break;

    // -- merge the CTA's row slices of this piece in shared memory (all consumer warps finish
    //    a piece together: they share its stages)
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (hv) {
      float* row = ms + ((size_t)slice * G + hh) * (D + 2);
#pragma unroll
      for (int n = 0; n < C::NT; ++n) {
        const int d = dh * C::DW + n * 8 + 2 * tig;
        row[d] = o[n][0] + o[n][2];
        row[d + 1] = o[n][1] + o[n][3];
      }
      if (tig == 0 && dh == 0) {
        row[D] = m_run;
        row[D + 1] = l_run;
      }
    }
    named_bar_sync(1, C::NCW * 32);
    const int i_first = sk_cta_of(seg_start, W, P);
    const int i_last = sk_cta_of(seg_start + n_row - 1, W, P);
    const bool whole = i_first == i_last;  // the segment lies inside this CTA's share
    float* rec = p.part + (size_t)(cta + seg) * G * (D + 2);
    for (int idx = threadIdx.x; idx < G * D; idx += C::NCW * 32) {
      const int h = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int sl = 0; sl < C::NPS; ++sl) M = fmaxf(M, ms[((size_t)sl * G + h) * (D + 2) + D]);
      float A = 0.f, Ls = 0.f;
#pragma unroll
      for (int sl = 0; sl < C::NPS; ++sl) {
        const float* r = ms + ((size_t)sl * G + h) * (D + 2);
        const float e = r[D] == -INFINITY ? 0.f : fast_exp2(r[D] - M);
        A = fmaf(r[d], e, A);
        Ls = fmaf(r[D + 1], e, Ls);
      }
      if (whole) {
        p.out[((size_t)t * p.n_heads + g * G + h) * D + d] =
            gated(p, t, g * G + h, d, Ls > 0.f ? A / Ls : 0.f);
      } else {
        rec[(size_t)h * (D + 2) + d] = A;
        if (d == 0) {
          rec[(size_t)h * (D + 2) + D] = M;
          rec[(size_t)h * (D + 2) + D + 1] = Ls;
        }
      }
    }
    if (!whole) __threadfence();  // this thread's record stores, before the CTA's ticket
    named_bar_sync(1, C::NCW * 32);  // records written; ms free for the next piece
    if (!whole) {
      // ticket: the CTA that brings the segment's last piece merges all of them
      if (threadIdx.x == 0)
        s_last = atomicInc(p.counters + seg, (unsigned)(i_last - i_first)) ==
                 (unsigned)(i_last - i_first);
      named_bar_sync(1, C::NCW * 32);
      if (s_last) {
        __threadfence();
        sk_merge_segment<D>(p, t, g, seg, i_first, i_last, warp, C::NCW, lane);
      }
    }
  }
  if (!ok && lane == 0) flag_error(p.err, GQA_ERR_TIMEOUT);
}

}  // namespace gqa
