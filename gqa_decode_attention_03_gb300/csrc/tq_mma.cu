// tq_mma.cu -- TurboQuant decode on the tensor cores (mma.sync m16n8k16, f16 in, f32 out).
//
// flash_attention_tq.metal (cera 0.4.0 sources); the score and accumulator definitions are in
// tq_common.cuh.  The page decodes every 2-bit field into a float and multiplies on the scalar
// units.  Here both contractions of a 16-position tile run on the tensor cores, with the
// decoded values built directly as f16 fragments:
//
//   q.k  C[pos][head, part] = sum_d A[pos][d] B[d][head, part]: A holds the decoded centroids
//        c[kidx(d)] (PolarQuant term) or the signs +-1 of the QJL bits (QJL term), B the
//        rotated (JL-projected) query split into f16 hi and lo parts, one column each.
//   p.v  C[d][head, part] = sum_pos A[d][pos] B[pos][head, part]: A holds c[vidx(d)], B the
//        weights p * vnorm split into hi and lo parts.
//
// Centroids are split the same way (hi and lo f16 planes, one MMA each), so products carry
// about 22 significant bits and sums are fp32, as on the scalar path.  Power-of-two scales keep
// the f16 parts clear of overflow and of the subnormal range; they are exact and undone in fp32.
//
// Decoding a 2-bit field into an f16 costs a byte permute: a word's four 2-bit fields picked
// into four bytes (shift, and) become a prmt selector (times 0x22, plus 0x10101010: nibbles
// 2k and 2k + 1 for field value k) that gathers two f16 centroids from the 8-byte table
// {c0, c1, c2, c3}.  The k index of the fragments is permuted so that a thread's four fields
// sit at bit offsets 2i, 2i + 8, 2i + 16, 2i + 24 of one word; B is permuted the same way.  A
// sign bit becomes +-1 by moving it to an f16 sign position: ((w << s) & 0x80008000) ^ 0xBC00BC00.
//
// Each warp streams its own tiles (positions base + 16 * (warp + 4 k)) through a 4-stage
// cp.async ring in shared memory and keeps its own online-softmax state per head; the states
// meet in tq_finish.  Fragment roles (m16n8k16): lane = 4 fr + fq; A rows fr and fr + 8,
// k pairs 2 fq and 2 fq + 8; B column fr; C rows fr and fr + 8, columns 2 fq and 2 fq + 1.  B
// columns are (head, part) pairs: column n is head 4 nb + n / 2, part n % 2 (hi, lo), so a
// thread's C columns are one head's hi and lo parts and its softmax state is that head's.
#include <cuda_fp16.h>
#include <cuda_runtime_api.h>

#include "tq_frag.cuh"

namespace gqa {

constexpr int kTqStages = 4;


__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int D>
struct TqMmaLayout {
  static constexpr int PW = D / 16, JW = D / 32;
  static constexpr int KPS = PW == 8 ? 12 : PW;  // polar row stride in words (bank spread)
  static constexpr int oKp = 0, oKj = oKp + 16 * KPS, oKn = oKj + 16 * JW;
  static constexpr int oVp = oKn + 16, oVn = oVp + 16 * KPS, SW = oVn + 16;  // stage words
  static_assert(SW % 4 == 0 && oKj % 4 == 0 && oVp % 4 == 0, "16-byte aligned stage parts");
  static constexpr int kStageRing = kTqWarps * kTqStages * SW;
  static constexpr int kMg = kTqWarps * kTqMaxGroup * (D + 2);
  static constexpr int kBuf = kStageRing > kMg ? kStageRing : kMg;
};

// Three CTAs per SM at one n-block (up to 170 registers): 5 % faster on GB300 than four CTAs
// at 128 registers, which spill
template <int D, int NB>
__global__ void __launch_bounds__(32 * kTqWarps, NB == 1 ? 3 : 2)
    tq_mma_kernel(const TqParams tp) {
  using Lay = TqMmaLayout<D>;
  constexpr int PW = Lay::PW, JW = Lay::JW, KPS = Lay::KPS, S = kTqStages;
  const PartialParams& p = tp.base;
  __shared__ __align__(16) uint32_t sbuf[Lay::kBuf];  // stage ring, then the warps' states
  __shared__ __align__(16) float qr[kTqMaxGroup][D];
  __shared__ __align__(16) float qj[kTqMaxGroup][D];
  const int c = blockIdx.x, t = blockIdx.z;
  const TqCta cta = tq_cta(p);
  const int g = cta.g, G = cta.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int fr = lane >> 2, fq = lane & 3;

  int L, s, c0, c1;
  if (!tq_row_setup(p, t, c, cta, D, L, s, c0, c1)) return;

  // The first tiles' loads go out before the query setup, so their latency hides behind it.
  // per-thread constants of the decode: sign-bit multipliers (1 << (15 - bit)) of the QJL
  // fragments, and the byte gather / shift of the p.v fields
  uint32_t jmul[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    jmul[j][0] = 1u << (15 - (8 * j + fq));
    jmul[j][1] = 1u << (11 - (8 * j + fq));
  }
  const uint32_t vb = static_cast<uint32_t>(fr >> 2);
  const uint32_t vsel = vb | ((4u + vb) << 4) | ((2u + vb) << 8) | ((6u + vb) << 12);
  const int vsh = 2 * (fr & 3);

  // ---- this warp's tiles through its cp.async ring
  uint32_t* ring = sbuf + warp * S * Lay::SW;
  const int ntiles = (c1 - c0 + 15) / 16;
  const int my_n = ntiles > warp ? (ntiles - warp + kTqWarps - 1) / kTqWarps : 0;
  // the (sequence, KV head)'s positions are contiguous (head-major): a tile's polar rows, sign
  // words and norms are each one contiguous run, copied by consecutive lanes in 16-byte pieces
  const size_t hrow0 = ((size_t)s * p.n_kv_heads + g) * p.cache_cap;
  const bool norms16 = (p.cache_cap & 3) == 0;  // 16-byte pieces of 4 norms stay in the head
  auto issue = [&](int k) {
    uint32_t* st = ring + (k % S) * Lay::SW;
    const int tb = c0 + 16 * (warp + kTqWarps * k);
    constexpr int CPP = PW / 4;  // 16-byte pieces of a polar row
    if (lane < 16 * CPP) {
      const int pp = lane / CPP, ch = lane % CPP;
      const int pos = min(tb + pp, c1 - 1);  // past the chunk: any valid row, masked later
      const size_t row = hrow0 + pos;
      cp_async_16(st + Lay::oKp + pp * KPS + 4 * ch, tp.k_polar + row * PW + 4 * ch);
      cp_async_16(st + Lay::oVp + pp * KPS + 4 * ch, tp.v_polar + row * PW + 4 * ch);
    }
    if (lane < 16) {
      const size_t row = hrow0 + min(tb + lane, c1 - 1);
      if constexpr (JW == 4)
        cp_async_16(st + Lay::oKj + lane * 4, tp.k_jl + row * 4);
      else
        cp_async_8(st + Lay::oKj + lane * 2, tp.k_jl + row * 2);
    }
    if (norms16) {
      if (lane >= 16 && lane < 24) {  // 4 pieces of K norms, 4 of V norms
        const int q = lane & 3;
        int p4 = tb + 4 * q;
        if (p4 >= c1) p4 = (c1 - 1) & ~3;  // a piece wholly past the chunk: a valid one
        if (lane < 20)
          cp_async_16(st + Lay::oKn + 4 * q, tp.k_norms + hrow0 + p4);
        else
          cp_async_16(st + Lay::oVn + 4 * q, tp.v_norms + hrow0 + p4);
      }
    } else {
      const int pp = lane & 15;
      const size_t row = hrow0 + min(tb + pp, c1 - 1);
      if (lane < 16)
        cp_async_4(st + Lay::oVn + pp, tp.v_norms + row);
      else
        cp_async_4(st + Lay::oKn + pp, tp.k_norms + row);
    }
  };
#pragma unroll
  for (int k = 0; k < S - 1; ++k) {
    if (k < my_n) issue(k);
    cp_async_commit();
  }

  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const size_t qi = ((size_t)t * p.n_heads + cta.head0) * D + i;
    qr[i / D][i % D] = __ldg(tp.q_rot + qi);
    qj[i / D][i % D] = __ldg(tp.q_jl + qi);
  }
  __syncthreads();

  // ---- scales and f16 fragments of the queries (B operands of q.k) and of the centroids
  float amr = 0.f, amj = 0.f;
  for (int i = lane; i < G * D; i += 32) {
    amr = fmaxf(amr, fabsf(qr[i / D][i % D]));
    amj = fmaxf(amj, fabsf(qj[i / D][i % D]));
  }
  amr = warp_max(amr);
  amj = warp_max(amj);
  const float sr = pow2_scale(amr), sjq = pow2_scale(amj);
  const float sc = pow2_scale(fmaxf(fmaxf(fabsf(tp.c0), fabsf(tp.c1)), fmaxf(fabsf(tp.c2), fabsf(tp.c3))));
  uint32_t th01, th23, tl01, tl23;  // centroid tables: hi and lo planes, f16 {c0, c1 | c2, c3}
  {
    uint32_t h, l;
    split_hi_lo(tp.c0 * sc, tp.c1 * sc, h, l);
    th01 = h;
    tl01 = l;
    split_hi_lo(tp.c2 * sc, tp.c3 * sc, h, l);
    th23 = h;
    tl23 = l;
  }
  const int part = fr & 1;
  uint32_t qb[PW][NB][2], qjb[JW][2][NB][2];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int hd = 4 * nb + (fr >> 1);
    const bool hv = hd < G;
    const int hr = hv ? hd : 0;
#pragma unroll
    for (int kb = 0; kb < PW; ++kb) {
      const float* q = &qr[hr][16 * kb + fq];
      qb[kb][nb][0] = hv ? f16_part(q[0] * sr, q[4] * sr, part) : 0u;
      qb[kb][nb][1] = hv ? f16_part(q[8] * sr, q[12] * sr, part) : 0u;
    }
#pragma unroll
    for (int w = 0; w < JW; ++w)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float* q = &qj[hr][32 * w + 8 * j + fq];
        qjb[w][j][nb][0] = hv ? f16_part(q[0] * sjq, q[16] * sjq, part) : 0u;
        qjb[w][j][nb][1] = hv ? f16_part(q[4] * sjq, q[20] * sjq, part) : 0u;
      }
  }
  // x = norm (polar sp + rn signed sj), in log2 units
  const float sp = p.scale_log2 / (sr * sc), sj = p.scale_log2 * tp.qjl_scale / sjq;

  float acc[PW][NB][4], m_run[NB], l_run[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    m_run[nb] = -INFINITY;
    l_run[nb] = 0.f;
#pragma unroll
    for (int mb = 0; mb < PW; ++mb) acc[mb][nb][0] = acc[mb][nb][1] = acc[mb][nb][2] = acc[mb][nb][3] = 0.f;
  }

  for (int k = 0; k < my_n; ++k) {
    __syncwarp();  // every lane is done with the stage the next issue overwrites
    if (k + S - 1 < my_n) issue(k + S - 1);
    cp_async_commit();
    cp_async_wait<S - 1>();
    __syncwarp();
    const uint32_t* st = ring + (k % S) * Lay::SW;
    const int nv = c1 - (c0 + 16 * (warp + kTqWarps * k));  // valid positions (>= 1)

    // q.k: PolarQuant term (hi and lo centroid planes) and QJL term, 16 positions x heads
    float pol[NB][4], pol2[NB][4], jl[NB][4], jl2[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) pol[nb][e] = pol2[nb][e] = jl[nb][e] = jl2[nb][e] = 0.f;
#pragma unroll
    for (int kb = 0; kb < PW; ++kb) {
      const uint32_t w0 = st[Lay::oKp + fr * KPS + kb], w1 = st[Lay::oKp + (fr + 8) * KPS + kb];
      uint32_t s0, s0h, s1, s1h;
      field_sel((w0 >> (2 * fq)) & 0x03030303u, s0, s0h);
      field_sel((w1 >> (2 * fq)) & 0x03030303u, s1, s1h);
      const uint32_t ah[4] = {prmt(th01, th23, s0), prmt(th01, th23, s1),
                              prmt(th01, th23, s0h), prmt(th01, th23, s1h)};
      const uint32_t al[4] = {prmt(tl01, tl23, s0), prmt(tl01, tl23, s1),
                              prmt(tl01, tl23, s0h), prmt(tl01, tl23, s1h)};
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {  // two accumulators: shorter MMA dependency chains
        mma_f16(pol[nb], ah, qb[kb][nb][0], qb[kb][nb][1]);
        mma_f16(pol2[nb], al, qb[kb][nb][0], qb[kb][nb][1]);
      }
    }
#pragma unroll
    for (int w = 0; w < JW; ++w) {
      const uint32_t z0 = st[Lay::oKj + fr * JW + w], z1 = st[Lay::oKj + (fr + 8) * JW + w];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        // bit -> f16 sign bit 15 (and bit + 16 -> 31): a left shift, as a multiply
        const uint32_t m0 = jmul[j][0], m1 = jmul[j][1];
        const uint32_t a[4] = {((z0 * m0) & 0x80008000u) ^ 0xBC00BC00u,
                               ((z1 * m0) & 0x80008000u) ^ 0xBC00BC00u,
                               ((z0 * m1) & 0x80008000u) ^ 0xBC00BC00u,
                               ((z1 * m1) & 0x80008000u) ^ 0xBC00BC00u};
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          if (j == 0) mma_f16(jl[nb], a, qjb[w][j][nb][0], qjb[w][j][nb][1]);
          else mma_f16(jl2[nb], a, qjb[w][j][nb][0], qjb[w][j][nb][1]);
        }
      }
    }

    // scores of positions fr and fr + 8 for head 4 nb + fq; online softmax; p.v weights
    const uint32_t kn0 = st[Lay::oKn + fr], kn1 = st[Lay::oKn + fr + 8];
    const float vn0 = half_lo(st[Lay::oVn + fr]), vn1 = half_lo(st[Lay::oVn + fr + 8]);
    uint32_t pb[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const float P0 = (pol[nb][0] + pol2[nb][0]) + (pol[nb][1] + pol2[nb][1]);
      const float P1 = (pol[nb][2] + pol2[nb][2]) + (pol[nb][3] + pol2[nb][3]);
      const float J0 = (jl[nb][0] + jl2[nb][0]) + (jl[nb][1] + jl2[nb][1]);
      const float J1 = (jl[nb][2] + jl2[nb][2]) + (jl[nb][3] + jl2[nb][3]);
      const float x0 = fr < nv ? half_lo(kn0) * fmaf(half_hi(kn0) * sj, J0, P0 * sp) : -INFINITY;
      const float x1 = fr + 8 < nv ? half_lo(kn1) * fmaf(half_hi(kn1) * sj, J1, P1 * sp) : -INFINITY;
      float mx = fmaxf(x0, x1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run[nb], mx);
      const float corr = fast_exp2(m_run[nb] - m_new);  // first tile: exp2(-inf) = 0
      const float p0 = fast_exp2(x0 - m_new), p1 = fast_exp2(x1 - m_new);
      l_run[nb] = fmaf(l_run[nb], corr, p0 + p1);
      if (__any_sync(0xffffffffu, m_new > m_run[nb])) {
#pragma unroll
        for (int mb = 0; mb < PW; ++mb)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mb][nb][e] *= corr;
      }
      m_run[nb] = m_new;
      // B of p.v: column fr = (head 4 nb + fr / 2, part fr % 2) at positions 2 fq, 2 fq + 1,
      // 2 fq + 8, 2 fq + 9, held by lanes 4 (2 fq) + fr / 2 and 4 (2 fq + 1) + fr / 2
      // norms past the chunk may be anything (NaN past a sequence's length): select, never
      // multiply by a zero weight
      const float v0 = fr < nv ? p0 * vn0 : 0.f, v1 = fr + 8 < nv ? p1 * vn1 : 0.f;
      const int la = 8 * fq + (fr >> 1), lb = la + 4;
      const float e0 = __shfl_sync(0xffffffffu, v0, la), e1 = __shfl_sync(0xffffffffu, v0, lb);
      const float e2 = __shfl_sync(0xffffffffu, v1, la), e3 = __shfl_sync(0xffffffffu, v1, lb);
      const bool hv = 4 * nb + (fr >> 1) < G;
      pb[nb][0] = hv ? f16_part(e0, e1, part) : 0u;
      pb[nb][1] = hv ? f16_part(e2, e3, part) : 0u;
    }

    // p.v: rows = dims fr, fr + 8 of each 16-dim polar word, k = the tile's positions
#pragma unroll
    for (int mb = 0; mb < PW; ++mb) {
      const uint32_t wa = st[Lay::oVp + (2 * fq) * KPS + mb];
      const uint32_t wb = st[Lay::oVp + (2 * fq + 1) * KPS + mb];
      const uint32_t wc = st[Lay::oVp + (2 * fq + 8) * KPS + mb];
      const uint32_t wd = st[Lay::oVp + (2 * fq + 9) * KPS + mb];
      // bytes (wa.b[fr/4], wb.b[fr/4], wa.b[2 + fr/4], wb.b[2 + fr/4]) hold the fields of dims
      // fr and fr + 8 at bit 2 (fr % 4) of each byte
      uint32_t sa, sah, sc2, sch;
      field_sel((__byte_perm(wa, wb, vsel) >> vsh) & 0x03030303u, sa, sah);
      field_sel((__byte_perm(wc, wd, vsel) >> vsh) & 0x03030303u, sc2, sch);
      const uint32_t ah[4] = {prmt(th01, th23, sa), prmt(th01, th23, sah),
                              prmt(th01, th23, sc2), prmt(th01, th23, sch)};
      const uint32_t al[4] = {prmt(tl01, tl23, sa), prmt(tl01, tl23, sah),
                              prmt(tl01, tl23, sc2), prmt(tl01, tl23, sch)};
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        mma_f16(acc[mb][nb], ah, pb[nb][0], pb[nb][1]);
        mma_f16(acc[mb][nb], al, pb[nb][0], pb[nb][1]);
      }
    }
  }
  cp_async_wait<0>();

  // ---- this warp's state per head into shared memory (the ring is no longer read)
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    float l = l_run[nb];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    l_run[nb] = l;
  }
  __syncthreads();
  float* mg = reinterpret_cast<float*>(sbuf);
  const float sv = 1.f / sc;
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int hd = 4 * nb + fq;
    if (hd < G) {
      float* r = mg + (warp * kTqMaxGroup + hd) * (D + 2);
#pragma unroll
      for (int mb = 0; mb < PW; ++mb) {
        r[16 * mb + fr] = (acc[mb][nb][0] + acc[mb][nb][1]) * sv;
        r[16 * mb + fr + 8] = (acc[mb][nb][2] + acc[mb][nb][3]) * sv;
      }
      if (fr == 0) {
        r[D] = m_run[nb];
        r[D + 1] = l_run[nb];
      }
    }
  }
  __syncthreads();
  tq_finish<D>(tp, mg, t, cta, c, L);
}

cudaError_t launch_tq_mma(int head_dim, int nb, dim3 grid, const TqParams& tp,
                          cudaStream_t stream) {
  const int threads = 32 * kTqWarps;
  if (head_dim == 64) {
    if (nb == 1) tq_mma_kernel<64, 1><<<grid, threads, 0, stream>>>(tp);
    else tq_mma_kernel<64, 2><<<grid, threads, 0, stream>>>(tp);
  } else {
    if (nb == 1) tq_mma_kernel<128, 1><<<grid, threads, 0, stream>>>(tp);
    else tq_mma_kernel<128, 2><<<grid, threads, 0, stream>>>(tp);
  }
  return cudaGetLastError();
}

}  // namespace gqa
