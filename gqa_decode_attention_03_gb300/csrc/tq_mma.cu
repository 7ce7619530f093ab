// tq_mma.cu -- TurboQuant decode on the tensor cores (mma.sync m16n8k16, f16 in, f32 out).
//
// flash_attention_tq.metal (cera 0.4.0 sources); the score and accumulator definitions are in
// tq_common.cuh.  The page decodes every 2-bit field into a float and multiplies on the scalar
// units.  Here both contractions of a 16-position tile run on the tensor cores, with the
// decoded values built directly as f16 fragments:
//
//   q.k  C[pos][head, part] = sum_d A[pos][d] B[d][head, part]: A holds bit planes of the keys'
//        2-bit centroid indices (PolarQuant term) or their QJL sign bits, B the rotated
//        (JL-projected) query split into f16 hi and lo parts, one column each.
//   p.v  C[d][head, part] = sum_pos A[d][pos] B[pos][head, part]: A holds bit planes of the
//        values' indices, B the weights p * vnorm times a plane coefficient, split into hi / lo.
//
// No centroid is ever decoded.  Over the two bits (b0, b1) of an index the centroid is exactly
//   c[idx] = c0 + (c1 - c0) b0 + (c2 - c0) b1 + (c3 - c2 - c1 + c0) b0 b1,
// so sum_d q[d] c[idx(d)] = c0 sum_d q[d] + the planes' sums (the last plane drops out for any
// centroid set symmetric about zero, and the kernel is instantiated without it then), and a
// sign sum is 2 sum_{bit set} q_jl - sum_d q_jl.  A plane bit enters the MMA as the f16 whose
// only set bit is the field's own bit, masked in place: bit k of a half-word is the f16
// 2^(k - 24) for k <= 10 (subnormal below 10), 2^-11 at bit 12 and 2 at bit 14 -- one exact
// power of two per k, folded into the other operand (or undone per output row) in fp32.  One
// AND then makes a fragment register (two elements), where a centroid lookup took two byte
// permutes (hi and lo planes) and a selector.  The per-head sums of q_rot and q_jl are taken
// once per CTA; products carry about 22 significant bits of q and of the weights, sums are
// fp32, as on the scalar path.  Power-of-two scales keep the f16 parts clear of overflow.
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

constexpr int kTqStages = 5;


// A 16-byte cp.async under a per-thread predicate, as one predicated instruction (no branch).
__device__ __forceinline__ void cp_async_16_if(void* dst, const void* src, bool on) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p cp.async.cg.shared.global [%0], [%1], 16;\n}"
      ::"r"(smem_addr(dst)), "l"(src), "r"((int)on)
      : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The 8x8 16-bit matrix held across the warp in mma fragment order (lane 4 r + c: row r, columns
// 2 c, 2 c + 1), transposed in registers.
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
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

// Each warp takes its tiles two at a time: both tiles' q.k, one softmax step over their 32
// positions, both tiles' p.v -- two independent instruction streams in every phase, where a
// single tile left the warp waiting on each MMA's and mask's latency (3 warps per scheduler).
// The q.k B fragments (the same for every warp) live in shared memory, over the staged queries,
// which frees the registers the second tile needs: three CTAs per SM at one n-block.
template <int D, int NB, bool B01>
__global__ void __launch_bounds__(32 * kTqWarps, NB == 1 ? 4 : 2)
    tq_mma_kernel(const TqParams tp) {
  using Lay = TqMmaLayout<D>;
  constexpr int PW = Lay::PW, JW = Lay::JW, KPS = Lay::KPS, S = kTqStages;
  const PartialParams& p = tp.base;
  __shared__ __align__(16) uint32_t sbuf[Lay::kBuf];  // stage ring, then the warps' states
  // the group's staged queries [q_rot | q_jl][head][D], then the q.k B fragments [slot][lane]
  __shared__ __align__(16) float qs[2][kTqMaxGroup][D];
  static_assert((PW + 2 * JW) * NB * 32 * 8 <= (int)sizeof(qs), "B fragments fit the staging");
  float(&qr)[kTqMaxGroup][D] = qs[0];
  float(&qj)[kTqMaxGroup][D] = qs[1];
  const uint2* fqb = reinterpret_cast<const uint2*>(&qs[0][0][0]);  // [kb][nb][lane]
  const uint2* fjb = fqb + PW * NB * 32;                              // [w][j][nb][lane]
  // launched as a programmatic dependent of the previous kernel on the stream (a no-op
  // otherwise): nothing in global memory is touched before that kernel has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int c = blockIdx.x, t = blockIdx.z;
  const TqCta cta = tq_cta(p);
  const int g = cta.g, G = cta.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int fr = lane >> 2, fq = lane & 3;

  int L, s, c0, c1;
  if (!tq_row_setup(p, t, c, cta, D, L, s, c0, c1)) return;

  // The first tiles' loads go out before the query setup, so their latency hides behind it.
  // ---- this warp's tiles (chunk tiles warp, warp + 4, ...) through its cp.async ring
  uint32_t* ring = sbuf + warp * S * Lay::SW;
  const int ntiles = (c1 - c0 + 15) / 16;
  const int my_n = ntiles > warp ? (ntiles - warp + kTqWarps - 1) / kTqWarps : 0;
  // the (sequence, KV head)'s positions are contiguous (head-major): a tile's polar rows, sign
  // words and norms are each one contiguous run, copied by consecutive lanes in 16-byte pieces
  const size_t hrow0 = ((size_t)s * p.n_kv_heads + g) * p.cache_cap;
  const bool norms16 = (p.cache_cap & 3) == 0;  // 16-byte pieces of 4 norms stay in the head
  // A tile wholly inside the chunk (and 4-position norm pieces inside the head) goes out
  // branch-free: every lane's copies are fixed pieces at a fixed offset from the tile's first
  // position, one 16-byte copy each (a predicated one for lanes with none of a kind).
  // D = 128: lane = 2 row + half for the polar rows (K and V); lanes 0-15 a sign row, 16-19 and
  // 20-23 four K / V norms.  D = 64: lanes 0-15 a K polar row, 16-31 a V one; lanes 0-7 two
  // sign rows, 8-11 and 12-15 four K / V norms.
  const size_t pos0 = hrow0 + c0 + 16 * warp;  // the warp's first tile, first position
  const uint32_t* fa;
  const uint32_t* fb;
  const uint32_t* fc;
  int da, db, dc;
  bool hc;
  if constexpr (PW == 8) {
    const int pp = lane >> 1, ch = lane & 1;
    fa = tp.k_polar + (pos0 + pp) * PW + 4 * ch;
    da = Lay::oKp + pp * KPS + 4 * ch;
    fb = tp.v_polar + (pos0 + pp) * PW + 4 * ch;
    db = Lay::oVp + pp * KPS + 4 * ch;
    const int q = (lane - 16) & 3;
    fc = lane < 16 ? tp.k_jl + (pos0 + lane) * JW
                   : (lane < 20 ? tp.k_norms : tp.v_norms) + pos0 + 4 * q;
    dc = lane < 16 ? Lay::oKj + lane * JW : (lane < 20 ? Lay::oKn : Lay::oVn) + 4 * q;
    hc = lane < 24;
  } else {
    const int pp = lane & 15;
    fa = (lane < 16 ? tp.k_polar : tp.v_polar) + (pos0 + pp) * PW;
    da = (lane < 16 ? Lay::oKp : Lay::oVp) + pp * KPS;
    fb = fa;
    db = da;
    const int q = lane & 3;
    fc = lane < 8 ? tp.k_jl + (pos0 + 2 * lane) * JW
                  : (lane < 12 ? tp.k_norms : tp.v_norms) + pos0 + 4 * q;
    dc = lane < 8 ? Lay::oKj + 2 * lane * JW : (lane < 12 ? Lay::oKn : Lay::oVn) + 4 * q;
    hc = lane < 16;
  }
  // per tile the warp moves on by 16 x kTqWarps positions: the same number of words per
  // position for each piece of a kind (polar PW, signs JW, norms 1)
  constexpr size_t kStep = 16 * kTqWarps;
  const size_t ic = PW == 8 ? (lane < 16 ? kStep * JW : kStep) : (lane < 8 ? kStep * JW : kStep);
  auto issue = [&](int k) {
    uint32_t* st = ring + (k % S) * Lay::SW;
    const int tb = c0 + 16 * (warp + kTqWarps * k);
    if (norms16 && tb + 16 <= c1) {
      cp_async_16(st + da, fa + k * kStep * PW);
      if constexpr (PW == 8) cp_async_16(st + db, fb + k * kStep * PW);
      cp_async_16_if(st + dc, fc + k * ic, hc);
      return;
    }
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
  // S - 2 tiles ahead: each step consumes two stages and refills the two its predecessor freed
#pragma unroll
  for (int k = 0; k < S - 2; ++k) {
    if (k < my_n) issue(k);
    cp_async_commit();
  }

  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const size_t qi = ((size_t)t * p.n_heads + cta.head0) * D + i;
    qr[i / D][i % D] = __ldg(tp.q_rot + qi);
    qj[i / D][i % D] = __ldg(tp.q_jl + qi);
  }
  __syncthreads();

  // ---- scales, per-head sums and the f16 fragments of the queries (B operands of q.k)
  float amr = 0.f, amj = 0.f;
  for (int i = lane; i < G * D; i += 32) {
    amr = fmaxf(amr, fabsf(qr[i / D][i % D]));
    amj = fmaxf(amj, fabsf(qj[i / D][i % D]));
  }
  amr = warp_max(amr);
  amj = warp_max(amj);
  const float sr = pow2_scale(amr), sjq = pow2_scale(amj);
  const int part = fr & 1;
  float base[NB], cj[NB];  // per softmax head 4 nb + fq: c0 sum_d q_rot, qjl_scale sum_d q_jl
  {
    uint32_t qb[PW][NB][2], qjb[JW][2][NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int hd = 4 * nb + (fr >> 1);
      const bool hv = hd < G;
      const int hr = hv ? hd : 0;
#pragma unroll
      for (int kb = 0; kb < PW; ++kb) {  // dims fq, fq + 8 (bit 0 of a half), fq + 4, fq + 12 (bit 8)
        const float* q = &qr[hr][16 * kb + fq];
        qb[kb][nb][0] = hv ? f16_part(q[0] * sr, q[8] * sr, part) : 0u;
        qb[kb][nb][1] = hv ? f16_part(q[4] * (sr * 0x1p-8f), q[12] * (sr * 0x1p-8f), part) : 0u;
      }
#pragma unroll
      for (int w = 0; w < JW; ++w)
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // sign bits fq + 8 j (+16) at bit 8 j, fq + 8 j + 4 (+16) at 8 j + 4
          const float* q = &qj[hr][32 * w + 8 * j + fq];
          const float s0 = j ? sjq * 0x1p-8f : sjq, s1 = j ? sjq * 0x1p-13f : sjq * 0x1p-4f;
          qjb[w][j][nb][0] = hv ? f16_part(q[0] * s0, q[16] * s0, part) : 0u;
          qjb[w][j][nb][1] = hv ? f16_part(q[4] * s1, q[20] * s1, part) : 0u;
        }
      // the softmax head of this thread: 4 nb + fq; its sums over D dims, 8 lanes (fr) a share
      const int hs = 4 * nb + fq < G ? 4 * nb + fq : 0;
      float sq = 0.f, sj = 0.f;
#pragma unroll
      for (int e = 0; e < D / 8; ++e) {
        sq += qr[hs][fr * (D / 8) + e];
        sj += qj[hs][fr * (D / 8) + e];
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sj += __shfl_xor_sync(0xffffffffu, sj, o);
      }
      base[nb] = tp.c0 * sq * p.scale_log2;
      cj[nb] = tp.qjl_scale * sj * p.scale_log2;
    }
    __syncthreads();  // every warp is done with the staged queries
    if (warp == 0) {
      uint2* fq2 = reinterpret_cast<uint2*>(&qs[0][0][0]);
      uint2* fj2 = fq2 + PW * NB * 32;
#pragma unroll
      for (int kb = 0; kb < PW; ++kb)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
          fq2[(kb * NB + nb) * 32 + lane] = make_uint2(qb[kb][nb][0], qb[kb][nb][1]);
#pragma unroll
      for (int w = 0; w < JW; ++w)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            fj2[((w * 2 + j) * NB + nb) * 32 + lane] = make_uint2(qjb[w][j][nb][0], qjb[w][j][nb][1]);
    }
    __syncthreads();
  }
  // c[idx] = c0 + (c1 - c0) b0 + (c2 - c0) b1 + (c3 - c2 - c1 + c0) b0 b1 over the index bits.
  // Plane sums come out of the MMAs in units of sr 2^-24 (b1: twice that, read at bit 1), the
  // sign sum in units of sjq 2^-24; x = norm (base + sum_p kq_p P_p + rn (kj J - cj)), log2 units
  const float d1 = tp.c1 - tp.c0, d2 = tp.c2 - tp.c0, d3 = (tp.c3 - tp.c2) - (tp.c1 - tp.c0);
  const float kq0 = d1 * (0x1p24f / sr) * p.scale_log2, kq1 = d2 * (0x1p23f / sr) * p.scale_log2;
  const float kq2 = d3 * (0x1p24f / sr) * p.scale_log2;
  const float kj = 2.f * tp.qjl_scale * (0x1p24f / sjq) * p.scale_log2;
  // p.v weights times the plane coefficients, scaled by a power of two that keeps them <= 1 x w
  float cs;
  {
    int e;
    frexpf(fmaxf(fmaxf(fabsf(d1), fabsf(d2)), fmaxf(fabsf(d3), 0x1p-100f)), &e);
    cs = ldexpf(1.f, -e);
  }
  const float cw0 = d1 * cs, cw1 = d2 * cs, cw2 = d3 * cs;
  // p.v A operands.  Each value word is masked in the keys' layout (position rows fr, fr + 8;
  // fields fq, fq + 8 and fq + 4, fq + 12 of a 16-dim word at bits 2 fq and 8 + 2 fq of each
  // half), one AND a register, and every 8x8 block is transposed in registers (movmatrix): rows
  // become dims, columns positions.  Slot m of a word is dim (m % 8) / 2 + 4 (m / 8) + 8 (m % 2),
  // field j = (m % 8) / 2 + 4 (m / 8) at bit 2 j of its half: the f16 2^(2 j - 24) (2^-11 for
  // j = 6, 2 for j = 7).  This thread's accumulator rows are slots fr (dim dr0), fr + 8 (dr1).
  const uint32_t vm0 = 0x00010001u << (2 * fq), vm1 = 0x01000100u << (2 * fq);
  const int j0 = fr >> 1, j1 = j0 + 4;
  const int dr0 = j0 + 8 * (fr & 1), dr1 = j1 + 8 * (fr & 1);
  auto bitval = [](int j) { return j < 6 ? ldexpf(1.f, 2 * j - 24) : (j == 6 ? 0x1p-11f : 2.f); };
  const float vu0 = bitval(j0), vu1 = bitval(j1);

  float acc[PW][NB][4], m_run[NB], l_run[NB], w_run[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    m_run[nb] = -INFINITY;
    l_run[nb] = 0.f;
    w_run[nb] = 0.f;
#pragma unroll
    for (int mb = 0; mb < PW; ++mb) acc[mb][nb][0] = acc[mb][nb][1] = acc[mb][nb][2] = acc[mb][nb][3] = 0.f;
  }

  for (int k = 0; k < my_n; k += 2) {
    __syncwarp();  // every lane is done with the two stages the next issues overwrite
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (k + S - 2 + i < my_n) issue(k + S - 2 + i);
      cp_async_commit();
    }
    cp_async_wait<S - 2>();  // tiles k and k + 1 have landed
    __syncwarp();
    const uint32_t* st[2] = {ring + (k % S) * Lay::SW, ring + ((k + 1) % S) * Lay::SW};
    // valid positions of the two tiles (the second: <= 0 when this warp has no tile k + 1;
    // its stage then holds an earlier tile's words, whose scores and weights are selected away)
    const int nv0 = c1 - (c0 + 16 * (warp + kTqWarps * k));
    const int nv[2] = {nv0, nv0 - 16 * kTqWarps};

    // q.k: the index bit planes (exact 0 / power-of-two f16) against q, 16 positions x heads
    float pl0[2][NB][4], pl1[2][NB][4], pl2[2][NB][4], jl[2][NB][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) pl0[u][nb][e] = pl1[u][nb][e] = pl2[u][nb][e] = jl[u][nb][e] = 0.f;
#pragma unroll
    for (int kb = 0; kb < PW; ++kb) {
      uint2 b[NB];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) b[nb] = fqb[(kb * NB + nb) * 32 + lane];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        // fields fq, fq + 4, fq + 8, fq + 12 of each position's word at bits 0, 8, 16, 24
        const uint32_t u0 = st[u][Lay::oKp + fr * KPS + kb] >> (2 * fq);
        const uint32_t u1 = st[u][Lay::oKp + (fr + 8) * KPS + kb] >> (2 * fq);
        const uint32_t a0[4] = {u0 & 0x00010001u, u1 & 0x00010001u, u0 & 0x01000100u, u1 & 0x01000100u};
        const uint32_t a1[4] = {u0 & 0x00020002u, u1 & 0x00020002u, u0 & 0x02000200u, u1 & 0x02000200u};
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          mma_f16(pl0[u][nb], a0, b[nb].x, b[nb].y);
          mma_f16(pl1[u][nb], a1, b[nb].x, b[nb].y);
        }
        if constexpr (B01) {
          const uint32_t v0 = u0 >> 1, v1 = u1 >> 1;
          const uint32_t a2[4] = {u0 & v0 & 0x00010001u, u1 & v1 & 0x00010001u,
                                  u0 & v0 & 0x01000100u, u1 & v1 & 0x01000100u};
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_f16(pl2[u][nb], a2, b[nb].x, b[nb].y);
        }
      }
    }
#pragma unroll
    for (int w = 0; w < JW; ++w) {
      uint2 b0[NB], b1[NB];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        b0[nb] = fjb[((w * 2 + 0) * NB + nb) * 32 + lane];
        b1[nb] = fjb[((w * 2 + 1) * NB + nb) * 32 + lane];
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        // sign bits fq, fq + 4, fq + 8, fq + 12 of each half at bits 0, 4, 8, 12
        const uint32_t z0 = st[u][Lay::oKj + fr * JW + w] >> fq;
        const uint32_t z1 = st[u][Lay::oKj + (fr + 8) * JW + w] >> fq;
        const uint32_t a0[4] = {z0 & 0x00010001u, z1 & 0x00010001u, z0 & 0x00100010u, z1 & 0x00100010u};
        const uint32_t a1[4] = {z0 & 0x01000100u, z1 & 0x01000100u, z0 & 0x10001000u, z1 & 0x10001000u};
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          mma_f16(jl[u][nb], a0, b0[nb].x, b0[nb].y);
          mma_f16(jl[u][nb], a1, b1[nb].x, b1[nb].y);
        }
      }
    }

    // scores of positions fr and fr + 8 of both tiles for head 4 nb + fq; one online-softmax
    // step over the 32 positions; p.v weights
    uint32_t kn[2][2];
    float vn[2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      kn[u][0] = st[u][Lay::oKn + fr];
      kn[u][1] = st[u][Lay::oKn + fr + 8];
      vn[u][0] = half_lo(st[u][Lay::oVn + fr]);
      vn[u][1] = half_lo(st[u][Lay::oVn + fr + 8]);
    }
    uint32_t pb[2][NB][3][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float x[2][2];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float tt = fmaf(kq1, pl1[u][nb][2 * r] + pl1[u][nb][2 * r + 1],
                          fmaf(kq0, pl0[u][nb][2 * r] + pl0[u][nb][2 * r + 1], base[nb]));
          if constexpr (B01) tt = fmaf(kq2, pl2[u][nb][2 * r] + pl2[u][nb][2 * r + 1], tt);
          const float J = jl[u][nb][2 * r] + jl[u][nb][2 * r + 1];
          tt = fmaf(half_hi(kn[u][r]), fmaf(kj, J, -cj[nb]), tt);
          x[u][r] = fr + 8 * r < nv[u] ? half_lo(kn[u][r]) * tt : -INFINITY;
        }
      float mx = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run[nb], mx);
      const float corr = fast_exp2(m_run[nb] - m_new);  // first step: exp2(-inf) = 0
      float pr[2][2], v[2][2];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          pr[u][r] = fast_exp2(x[u][r] - m_new);
          // norms past the chunk may be anything (NaN past a sequence's length): select, never
          // multiply by a zero weight
          v[u][r] = fr + 8 * r < nv[u] ? pr[u][r] * vn[u][r] : 0.f;
        }
      l_run[nb] = fmaf(l_run[nb], corr, (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
      w_run[nb] = fmaf(w_run[nb], corr, (v[0][0] + v[0][1]) + (v[1][0] + v[1][1]));
      if (__any_sync(0xffffffffu, m_new > m_run[nb])) {
#pragma unroll
        for (int mb = 0; mb < PW; ++mb)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mb][nb][e] *= corr;
      }
      m_run[nb] = m_new;
      // B of p.v: column fr = (head 4 nb + fr / 2, part fr % 2) at positions 2 fq, 2 fq + 1,
      // 2 fq + 8, 2 fq + 9, held by lanes 4 (2 fq) + fr / 2 and 4 (2 fq + 1) + fr / 2; one
      // B per index plane (the weights times its coefficient)
      const int la = 8 * fq + (fr >> 1), lb = la + 4;
      const bool hv = 4 * nb + (fr >> 1) < G;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float e0 = __shfl_sync(0xffffffffu, v[u][0], la), e1 = __shfl_sync(0xffffffffu, v[u][0], lb);
        const float e2 = __shfl_sync(0xffffffffu, v[u][1], la), e3 = __shfl_sync(0xffffffffu, v[u][1], lb);
        pb[u][nb][0][0] = hv ? f16_part(cw0 * e0, cw0 * e1, part) : 0u;
        pb[u][nb][0][1] = hv ? f16_part(cw0 * e2, cw0 * e3, part) : 0u;
        pb[u][nb][1][0] = hv ? f16_part(cw1 * e0, cw1 * e1, part) : 0u;
        pb[u][nb][1][1] = hv ? f16_part(cw1 * e2, cw1 * e3, part) : 0u;
        if constexpr (B01) {
          pb[u][nb][2][0] = hv ? f16_part(cw2 * e0, cw2 * e1, part) : 0u;
          pb[u][nb][2][1] = hv ? f16_part(cw2 * e2, cw2 * e3, part) : 0u;
        }
      }
    }

    // p.v: rows = the 16 dims of a polar word (slot order above), k = a tile's positions
#pragma unroll
    for (int mb = 0; mb < PW; ++mb) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t w0 = st[u][Lay::oVp + fr * KPS + mb];
        const uint32_t w8 = st[u][Lay::oVp + (fr + 8) * KPS + mb];
        const uint32_t h0 = w0 >> 1, h8 = w8 >> 1;  // b1 at b0's bit
        const uint32_t a0[4] = {movm_t(w0 & vm0), movm_t(w0 & vm1), movm_t(w8 & vm0),
                                movm_t(w8 & vm1)};
        const uint32_t a1[4] = {movm_t(h0 & vm0), movm_t(h0 & vm1), movm_t(h8 & vm0),
                                movm_t(h8 & vm1)};
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          mma_f16(acc[mb][nb], a0, pb[u][nb][0][0], pb[u][nb][0][1]);
          mma_f16(acc[mb][nb], a1, pb[u][nb][1][0], pb[u][nb][1][1]);
        }
        if constexpr (B01) {
          const uint32_t a2[4] = {movm_t(w0 & h0 & vm0), movm_t(w0 & h0 & vm1),
                                  movm_t(w8 & h8 & vm0), movm_t(w8 & h8 & vm1)};
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_f16(acc[mb][nb], a2, pb[u][nb][2][0], pb[u][nb][2][1]);
        }
      }
    }
  }
  cp_async_wait<0>();

  // ---- this warp's state per head into shared memory (the ring is no longer read)
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    float l = l_run[nb], wsum = w_run[nb];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, o);
      wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    }
    l_run[nb] = l;
    w_run[nb] = wsum;
  }
  __syncthreads();
  float* mg = reinterpret_cast<float*>(sbuf);
  // the planes' bit values and the coefficients' scale, undone per row
  const float sv0 = 1.f / (vu0 * cs), sv1 = 1.f / (vu1 * cs);
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int hd = 4 * nb + fq;
    if (hd < G) {
      float* r = mg + (warp * kTqMaxGroup + hd) * (D + 2);
      const float cw = tp.c0 * w_run[nb];  // the c0 term of every dim
#pragma unroll
      for (int mb = 0; mb < PW; ++mb) {
        r[16 * mb + dr0] = fmaf(acc[mb][nb][0] + acc[mb][nb][1], sv0, cw);
        r[16 * mb + dr1] = fmaf(acc[mb][nb][2] + acc[mb][nb][3], sv1, cw);
      }
      if (fr == 0) {
        r[D] = m_run[nb];
        r[D + 1] = l_run[nb];
      }
    }
  }
  __syncthreads();
  tq_finish<D>(tp, mg, t, cta, c, L);
  // the next kernel on the stream may be scheduled once every CTA is here (not earlier: this
  // grid runs in several waves, whose slots a waiting dependent would take)
  asm volatile("griddepcontrol.launch_dependents;");
}

cudaError_t launch_tq_mma(int head_dim, int nb, dim3 grid, const TqParams& tp,
                          cudaStream_t stream) {
  const int threads = 32 * kTqWarps;
  // the b0 b1 plane only when the centroids need it (c3 - c2 - c1 + c0 = 0 for any centroid set
  // symmetric about zero, such as the Lloyd-Max points of a symmetric distribution)
  const bool b01 = (tp.c3 - tp.c2) - (tp.c1 - tp.c0) != 0.f;
  // a programmatic dependent of whatever precedes it on the stream: the launch overlaps that
  // kernel's tail (the kernel waits for it before touching global memory)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = tp.base.pdl ? 1 : 0;
#define GQA_TQ_LAUNCH(DD, NBB)                                                          \
  do {                                                                                  \
    if (b01) return cudaLaunchKernelEx(&cfg, tq_mma_kernel<DD, NBB, true>, tp);         \
    return cudaLaunchKernelEx(&cfg, tq_mma_kernel<DD, NBB, false>, tp);                 \
  } while (0)
  if (head_dim == 64) {
    if (nb == 1) GQA_TQ_LAUNCH(64, 1);
    GQA_TQ_LAUNCH(64, 2);
  }
  if (nb == 1) GQA_TQ_LAUNCH(128, 1);
  GQA_TQ_LAUNCH(128, 2);
#undef GQA_TQ_LAUNCH
}

}  // namespace gqa
