// host.cu -- the C ABI of libgqadecode.so: argument checks, the split planner, TMA descriptors,
// and kernel dispatch.  Nothing here allocates device memory or synchronises; every launch goes
// to the caller's stream.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <string>
#include <utility>

#include "dispatch.h"

namespace {

thread_local std::string g_last_error;

gqa_status fail(gqa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

gqa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GQA_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device, cached per device id.
int current_sm_count(gqa_status* st) {
  static std::mutex mu;
  static int cache[128] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *st = cuda_fail(e, "cudaGetDevice");
    return -1;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (dev >= 0 && dev < 128 && cache[dev] > 0) return cache[dev];
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    *st = cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
    return -1;
  }
  if (dev >= 0 && dev < 128) cache[dev] = n;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int env_int(const char* name) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : 0;
}

// Chunked split: enough chunks for about one wave of CTAs (two per SM) at the longest row, but
// no chunk longer than kMaxChunk positions.  Measured on GB300 (f16, D = 128): a CTA streams at
// most ~51 GB/s (three 32 KB stages in flight), so chunks far above 8192 positions leave a
// long tail, while short chunks multiply the fixed cost of a CTA (pipeline fill, partial
// write, merge ticket); 4096..8192-position chunks gave 98-108 % of the measured copy
// bandwidth on both the mixed-length and the uniform batch.
constexpr int kCtasPerSm = 2;
constexpr long long kMaxChunk = 8192;
// f16 rows longer than kMaxChunk are cut into chunks of at most kLongRowChunk: with ragged
// lengths the finer pieces even out the wave's tail, with uniform ones they add merge work
// (GB300, 16 rows, D = 128, one box, chunk 8192 -> 4096: lengths U[1024, 32768] 141.6 -> 140.3
// us, 4 such rows 72.2 -> 70.6; 16 x 32768 302.9 -> 305.5)
constexpr long long kLongRowChunk = 4096;
// The tcgen05 row kernel holds ~194 KB of shared memory: one CTA per SM.
constexpr int kUmmaRowsCtasPerSm = 1;
// Rows whose whole visited list is at most this many bytes of K/V (and scales) are not split:
// one CTA streams them in a few microseconds, less than a split's merge step costs.
constexpr long long kMinSplitBytes = 128 << 10;
// TurboQuant caches: 88 bytes per position and KV head at D = 128 against ~8 KB of decode and
// tensor work, so the split is sized by compute: more, shorter chunks (8 CTAs per SM, at most
// 1792 positions) and a split from 32 KB of packed row up.  (GB300, 16 rows U[1024, 32768],
// D = 128, bit-plane kernel, one box: chunks of 1024, 1280, 1536, 1792, 2048 positions gave
// 113.1, 110.2, 110.0, 108.2, 113.8 us.)
constexpr int kTqCtasPerSm = 8;
constexpr long long kTqMaxChunk = 1792;
constexpr long long kTqMinSplitBytes = 32 << 10;
// The TurboQuant row kernel: 8 warps and ~94 KB of shared memory, one CTA per SM.
constexpr int kTqRowsCtasPerSm = 1;

// Shapes that do not depend on the device.
gqa_status check_shape(int n_tok, int n_heads, int n_kv_heads, int head_dim, int max_kv_len,
                       int kind) {
  if (kind != GQA_KIND_F16 && kind != GQA_KIND_Q8 && kind != GQA_KIND_TQ)
    return fail(GQA_EINVAL, "kind must be 0, 1 or 2");
  if (n_tok < 0 || n_tok > 65535) return fail(GQA_EINVAL, "n_tok %d outside [0, 65535]", n_tok);
  if (n_heads <= 0 || n_kv_heads <= 0 || n_kv_heads > 65535)
    return fail(GQA_EINVAL, "n_heads %d / n_kv_heads %d", n_heads, n_kv_heads);
  if (n_heads % n_kv_heads)
    return fail(GQA_EINVAL, "n_heads %d is not a multiple of n_kv_heads %d", n_heads, n_kv_heads);
  if (head_dim != 64 && head_dim != 128 && head_dim != 256 &&
      !(kind == GQA_KIND_TQ && head_dim == 32))
    return fail(GQA_EINVAL, "head_dim %d not in {64, 128, 256} (TurboQuant: 32, 64, 128)",
                head_dim);
  if (max_kv_len < 0) return fail(GQA_EINVAL, "max_kv_len %d < 0", max_kv_len);
  if (n_heads / n_kv_heads > 16)
    return fail(GQA_EUNSUPPORTED, "group size %d > 16", n_heads / n_kv_heads);
  return GQA_OK;
}

}  // namespace

namespace gqa {

void set_last_error(const char* msg) { g_last_error = msg; }

// CUDA-core kernel: heads per warp for the query heads one CTA serves (at most 4 after the
// head split), four row slices per stage.
Variant pick_variant(int heads_per_cta) {
  if (heads_per_cta <= 4) return Variant{heads_per_cta <= 1 ? 1 : (heads_per_cta <= 2 ? 2 : 4), 4, 0};
  return Variant{4, 2, 0};
}

// The CUDA-core kernel (GQA_Q8_KERNEL=fma for int8 caches, GQA_F16_KERNEL=fma for f16) splits
// a KV head's query heads over head_split CTAs of at most four heads each -- the smallest
// divisor of the group size that gets there -- so a wide group (12 heads) spreads over three
// times as many CTAs.  The int8 tensor-core kernel takes up to eight heads a CTA (more CTAs on
// a grid smaller than the GPU: attn_decode_plan); the f16 tensor-core kernels the whole group.
// int8 caches run on the tensor-core kernel (partial_mma_q8.cuh) unless GQA_Q8_KERNEL=fma asks
// for the CUDA-core one (comparison and parity cross-check).
bool q8_on_mma() {
  const char* k = std::getenv("GQA_Q8_KERNEL");
  return !(k && std::strcmp(k, "fma") == 0);
}

// A split row of at most 8 chunks on the int8 tensor-core kernel merges inside a thread-block
// cluster of its chunk CTAs unless GQA_Q8_CLUSTER=0 asks for the last-CTA merge through the
// workspace (comparison and parity cross-check).
bool q8_cluster_merge() {
  const char* k = std::getenv("GQA_Q8_CLUSTER");
  return !(k && std::strcmp(k, "0") == 0);
}

int head_split_for(int kind, int group) {
  if (kind == GQA_KIND_TQ) {  // the TurboQuant kernels serve up to 8 heads of a group per CTA
    for (int hs = 1; hs <= group; ++hs)
      if (group % hs == 0 && group / hs <= 8) return hs;
    return group;
  }
  const char* k = std::getenv("GQA_F16_KERNEL");
  const bool fma = kind == GQA_KIND_Q8 ? !q8_on_mma() : (k && std::strcmp(k, "fma") == 0);
  if (!fma && kind != GQA_KIND_Q8) return 1;
  const int forced = env_int("GQA_HEAD_SPLIT");  // tuning sweeps: a divisor of the group size
  if (forced > 0 && group % forced == 0) return forced;
  // the int8 tensor-core kernel serves up to 8 heads a CTA by default (one warp per row slice
  // and output half: 16 heads a CTA measured 21.1 us against 16.4 on GB300, 1024 selected
  // cells), up to 16 when a head split of 1 is forced; the CUDA-core kernels up to 4
  const int per_cta = fma ? 4 : 8;
  for (int hs = 1; hs <= group; ++hs)
    if (group % hs == 0 && group / hs <= per_cta) return hs;
  return group;
}

// The stream-K split is opt-in (GQA_F16_SPLIT=streamk): on GB300 the chunked grid measured
// faster on both the mixed-length and the uniform batch (a fixed cost per piece end outweighs
// the perfect balance), so it stays the default.
bool use_streamk(int kind, int n_tok) {
  if (kind != GQA_KIND_F16 || n_tok > kStreamKMaxRows) return false;
  const char* k = std::getenv("GQA_F16_KERNEL");  // "fma": CUDA-core kernel, chunked grid
  if (k && std::strcmp(k, "fma") == 0) return false;
  const char* m = std::getenv("GQA_F16_SPLIT");
  return m && std::strcmp(m, "streamk") == 0;
}

// Grouped rows run on the tcgen05 kernel (rows_umma.cuh) unless GQA_F16_ROWS=mma asks for the
// mma.sync kernel (rows_mma.cuh; comparison and parity cross-check).
bool rows_on_umma() {
  const char* r = std::getenv("GQA_F16_ROWS");
  return !(r && std::strcmp(r, "mma") == 0);
}

// Rows sharing a sequence are grouped on the f16 tensor-core path when the caller's cache holds
// fewer sequences than there are rows: 64 / group size rows per CTA on the tcgen05 kernel (its
// 128 MMA rows hold each (row, head) pair twice, once per position half), 32 / group size on the
// mma.sync kernel.
int row_group_for(int kind, int n_tok, int n_seq, int group, int head_dim) {
  if (kind == GQA_KIND_TQ) {
    // TurboQuant rows sharing a sequence: the tensor-core row kernel (tq_rows.cu) serves up to
    // 64 (row, head) pairs per CTA from one decoded tile; head_dim 32 and the CUDA-core kernel
    // stay one CTA per row
    const char* k = std::getenv("GQA_TQ_KERNEL");
    const char* r = std::getenv("GQA_TQ_ROWS");  // "off": one CTA per row (tests, comparison)
    if (n_seq >= n_tok || head_dim == 32 || (k && std::strcmp(k, "fma") == 0) ||
        (r && std::strcmp(r, "off") == 0))
      return 1;
    return 64 / (group / head_split_for(kind, group));
  }
  if (kind != GQA_KIND_F16 || n_seq >= n_tok || use_streamk(kind, n_tok)) return 1;
  const char* k = std::getenv("GQA_F16_KERNEL");
  if (k && std::strcmp(k, "fma") == 0) return 1;
  const char* r = std::getenv("GQA_F16_ROWS");  // "off": one CTA per row (tests, comparison)
  if (r && std::strcmp(r, "off") == 0) return 1;
  if (head_dim == 256 || (group != 1 && group != 2 && group != 4 && group != 8)) return 1;
  return (rows_on_umma() ? 64 : 32) / group;
}

int stage_rows(int kind, int head_dim) {
  if (kind == GQA_KIND_TQ) return 128;  // 4 warps x 32 positions per pass
  if (kind == GQA_KIND_F16) return head_dim == 64 ? 128 : (head_dim == 128 ? 64 : 32);
  return head_dim == 256 ? 64 : 128;
}

}  // namespace gqa

extern "C" {

int gqa_abi_version(void) { return GQA_ABI_VERSION; }

const char* gqa_last_error(void) { return g_last_error.c_str(); }

const char* gqa_status_string(gqa_status s) {
  switch (s) {
    case GQA_OK: return "GQA_OK";
    case GQA_EINVAL: return "GQA_EINVAL";
    case GQA_EWORKSPACE: return "GQA_EWORKSPACE";
    case GQA_EUNSUPPORTED: return "GQA_EUNSUPPORTED";
    case GQA_ECUDA: return "GQA_ECUDA";
  }
  return "GQA_UNKNOWN";
}

gqa_status attn_decode_plan(int n_tok, int n_seq, int n_heads, int n_kv_heads, int head_dim,
                            int max_kv_len, int budget, int kind, int num_sms, gqa_plan* plan) {
  if (!plan) return fail(GQA_EINVAL, "plan is NULL");
  std::memset(plan, 0, sizeof *plan);
  gqa_status st = check_shape(n_tok, n_heads, n_kv_heads, head_dim, max_kv_len, kind);
  if (st != GQA_OK) return st;
  if (n_seq <= 0) return fail(GQA_EINVAL, "n_seq %d must be > 0", n_seq);
  plan->row_group = 1;
  if (kind == GQA_KIND_F16) budget = -1;
  if (budget == 0 || budget < -1) return fail(GQA_EINVAL, "budget %d (use -1 for dense)", budget);
  if (num_sms <= 0) {
    st = GQA_OK;
    num_sms = current_sm_count(&st);
    if (num_sms <= 0) return st != GQA_OK ? st : fail(GQA_ECUDA, "no SM count");
  }
  int tile = gqa::stage_rows(kind, head_dim);
  const long long nmax = budget > 0 ? std::min(max_kv_len, budget) : max_kv_len;
  if (gqa::use_streamk(kind, n_tok)) {
    // equal shares of the whole stream, at least 256 positions each, two CTAs per SM at most
    const long long wmax = (long long)n_tok * n_kv_heads * std::max(nmax, 1LL);
    int ctas = (int)std::min<long long>(2LL * num_sms, std::max(1LL, (wmax + 255) / 256));
    const int forced_ctas = env_int("GQA_FORCE_CTAS");  // tests: many small shares
    if (forced_ctas > 0) ctas = std::min(forced_ctas, 65535);
    const int group = n_heads / n_kv_heads;
    plan->chunk = 0;
    plan->n_split = ctas;
    plan->tile = tile;
    plan->grid_x = ctas;
    plan->grid_y = 1;
    plan->grid_z = 1;
    plan->merge = 1;
    plan->streamk = 1;
    const size_t cnt = ((size_t)n_tok * n_kv_heads * sizeof(uint32_t) + 255) / 256 * 256;
    plan->ws_bytes = cnt + ((size_t)ctas + (size_t)n_tok * n_kv_heads) * group *
                               (head_dim + 2) * sizeof(float);
    return GQA_OK;
  }
  const int group = n_heads / n_kv_heads;
  int hsplit = gqa::head_split_for(kind, group);
  const int rgroup = gqa::row_group_for(kind, n_tok, n_seq, group, head_dim);
  // CTAs that do work: one per row, or per group of rows sharing a sequence (at least one group
  // per sequence, and at least n_tok / rgroup groups)
  const long long groups =
      rgroup > 1 ? std::max<long long>((n_tok + rgroup - 1) / rgroup, std::min(n_seq, n_tok)) : n_tok;
  plan->row_group = rgroup;
  const bool tq = kind == GQA_KIND_TQ;
  const bool umma_rows = rgroup > 1 && !tq && gqa::rows_on_umma();
  if (umma_rows) tile = 64;  // the tcgen05 row kernel's tile, whatever head_dim
  const bool tq_rows = rgroup > 1 && tq;
  if (tq_rows) tile = 32;    // the TurboQuant row kernel's stage
  const int forced = env_int("GQA_FORCE_CHUNK");
  // the chunk length for a head split hs
  auto chunk_for = [&](int hs) {
    const long long units = groups * n_kv_heads * hs * std::max(nmax, 1LL);
    const long long slots =
        (long long)(tq_rows ? kTqRowsCtasPerSm
                    : tq    ? kTqCtasPerSm
                    : umma_rows ? kUmmaRowsCtasPerSm
                                : kCtasPerSm) *
        num_sms;
    long long chunk = (units + slots - 1) / slots;
    chunk = std::min(chunk, tq ? kTqMaxChunk : kMaxChunk);
    if (kind == GQA_KIND_F16 && rgroup == 1 && nmax > kMaxChunk) chunk = std::min(chunk, kLongRowChunk);
    // a split chunk spans at least two stages, so its pipeline has something to overlap
    // (GB300 sweeps: int8 gather 1024 cells 20 us at 2 stages a chunk against 23 us at 1; f16
    // D=64 4096 positions 14.7 against 16.1)
    chunk = std::max(chunk, 2LL * tile);
    const long long row_bytes =
        kind == GQA_KIND_F16   ? 4LL * head_dim
        : kind == GQA_KIND_Q8 ? 2LL * (head_dim + head_dim / 32)
                               : 4LL * (head_dim / 16 + head_dim / 32 + 1) + 4LL * (head_dim / 16 + 1);
    if (nmax * row_bytes <= (tq ? kTqMinSplitBytes : kMinSplitBytes)) chunk = std::max(nmax, 1LL);
    if (forced > 0) {
      chunk = forced;
    } else if (umma_rows) {
      // at most one CTA per SM in all, so that the chunk CTAs can merge their own partials (a
      // cooperative launch); when even one chunk per group and KV head is too many, the merge
      // kernel follows instead
      const long long per_split = (long long)n_kv_heads * hs * std::min<long long>(groups, n_tok);
      const long long cap = num_sms / std::max(per_split, 1LL);
      if (cap >= 1) chunk = std::max(chunk, (std::max(nmax, 1LL) + cap - 1) / cap);
    }
    chunk = (std::max(chunk, 1LL) + tile - 1) / tile * tile;
    const long long whole = (std::max(nmax, 1LL) + tile - 1) / tile * tile;
    return std::min(chunk, whole);
  };
  long long chunk = chunk_for(hsplit);
  if (kind == GQA_KIND_Q8 && gqa::q8_on_mma() && env_int("GQA_HEAD_SPLIT") <= 0) {
    // a grid smaller than the GPU is latency-bound: the int8 tensor-core kernel then serves
    // fewer heads per CTA (down to 4), as long as the grid still fits on the SMs -- a CTA's
    // tile time does not shrink with fewer heads, but 1.5-3x more CTAs share the positions'
    // merge and the per-CTA merge has fewer heads (GB300, 1024 selected cells, 12 heads per KV
    // head: 21.1 us at 12 heads a CTA, 16.4 at 6, 15.8 at 4)
    for (int hs = group; hs > hsplit; --hs) {
      if (group % hs != 0 || group / hs < 4) continue;
      const long long c = chunk_for(hs);
      const long long ns = std::max(1LL, (nmax + c - 1) / c);
      if (ns * n_kv_heads * hs * (long long)n_tok <= num_sms) {
        hsplit = hs;
        chunk = c;
        break;
      }
    }
  }
  {
    // a split grid that fits the GPU merges each row inside a thread-block cluster of its chunk
    // CTAs (the per-row tensor-core kernels): then up to 8 chunks a row, one stage each at the
    // least (GB300, D=64 GQA rows: 4096 positions 14.5 -> 12.6 us, 1024 positions 10.5 -> 9.5)
    const char* fk = std::getenv("GQA_F16_KERNEL");
    const char* fc = std::getenv("GQA_F16_CLUSTER");
    const bool f16_cl = kind == GQA_KIND_F16 && !(fk && std::strcmp(fk, "fma") == 0) &&
                        !(fc && std::strcmp(fc, "0") == 0);
    const bool q8_cl = kind == GQA_KIND_Q8 && gqa::q8_on_mma() && gqa::q8_cluster_merge();
    if ((f16_cl || q8_cl) && rgroup == 1 && forced <= 0 && chunk < nmax) {
      long long c8 = (nmax + 7) / 8;
      c8 = std::max((c8 + tile - 1) / tile * tile, (long long)tile);
      const long long ns8 = (nmax + c8 - 1) / c8;
      if (groups * n_kv_heads * hsplit * ns8 <= num_sms) chunk = c8;
    }
  }
  const long long n_split = std::max(1LL, (nmax + chunk - 1) / chunk);
  if (n_split > (1LL << 30)) return fail(GQA_EUNSUPPORTED, "too many chunks");
  plan->chunk = (int)chunk;
  plan->n_split = (int)n_split;
  plan->tile = tile;
  plan->grid_x = (int)n_split;
  plan->grid_y = n_kv_heads * hsplit;
  plan->grid_z = rgroup > 1 ? (int)std::min<long long>(groups, n_tok) : n_tok;  // group slots
  plan->merge = n_split > 1 ? 1 : 0;
  if (plan->merge) {
    const size_t cnt = ((size_t)n_tok * plan->grid_y * sizeof(uint32_t) + 255) / 256 * 256;
    const size_t part = (size_t)n_tok * n_split * n_heads * (head_dim + 2) * sizeof(float);
    plan->ws_bytes = cnt + (part + 255) / 256 * 256 + (size_t)n_tok * sizeof(int32_t);
  }
  return GQA_OK;
}

size_t attn_decode_workspace_bytes(int n_tok, int n_seq, int n_heads, int n_kv_heads,
                                   int head_dim, int max_kv_len, int budget, int kind) {
  gqa_plan plan;
  if (attn_decode_plan(n_tok, n_seq, n_heads, n_kv_heads, head_dim, max_kv_len, budget, kind, 0,
                       &plan) != GQA_OK)
    return 0;
  return plan.ws_bytes;
}

}  // extern "C"

namespace {

// Shared body of the two decode entry points.
gqa_status decode_common(int kind, const float* q, const void* kc, const void* vc,
                         const uint16_t* ksc, const uint16_t* vsc, const int32_t* ids, int budget,
                         float* out, const int32_t* kv_len, const int32_t* seq_of, int n_tok,
                         int n_seq, int n_heads, int n_kv_heads, int head_dim, int64_t cache_cap,
                         int max_kv_len, float scale, void* ws, size_t ws_bytes,
                         int32_t* err_word, cudaStream_t stream, int scale_group = 64,
                         const float* gate = nullptr, int64_t gate_stride = 0) {
  gqa_status st = check_shape(n_tok, n_heads, n_kv_heads, head_dim, max_kv_len, kind);
  if (st != GQA_OK) return st;
  if (n_tok == 0) return GQA_OK;
  if (gate && (gate_stride < head_dim || (reinterpret_cast<uintptr_t>(gate) & 3)))
    return fail(GQA_EINVAL, "gate must be 4-byte aligned with gate_stride >= head_dim");
  if (!q || !kc || !vc || !out || !kv_len) return fail(GQA_EINVAL, "a required pointer is NULL");
  if (kind == GQA_KIND_Q8 && (!ksc || !vsc)) return fail(GQA_EINVAL, "scale pointer is NULL");
  if (!aligned16(q) || !aligned16(out) || !aligned16(kc) || !aligned16(vc))
    return fail(GQA_EINVAL, "q, out and the caches must be 16-byte aligned");
  if (kind == GQA_KIND_Q8 && scale_group != 32 && scale_group != 64)
    return fail(GQA_EINVAL, "scale_group %d: 32 or 64 dims per scale", scale_group);
  if (kind == GQA_KIND_Q8) {  // a row's scales are copied in one piece of nsc * 2 bytes
    const int piece = std::min(16, 2 * (head_dim / scale_group));
    if (((reinterpret_cast<uintptr_t>(ksc) | reinterpret_cast<uintptr_t>(vsc)) & (piece - 1)) != 0)
      return fail(GQA_EINVAL, "scales must be %d-byte aligned", piece);
  }
  if (n_seq <= 0 || cache_cap <= 0) return fail(GQA_EINVAL, "n_seq and cache_cap must be > 0");
  if ((int64_t)n_seq * cache_cap > INT32_MAX)
    return fail(GQA_EUNSUPPORTED, "n_seq * cache_cap must stay below 2^31 rows");
  if (!seq_of && n_seq < n_tok) return fail(GQA_EINVAL, "seq_of NULL needs n_seq >= n_tok");
  if (!std::isfinite(scale)) return fail(GQA_EINVAL, "scale is not finite");
  if (ids && budget <= 0) return fail(GQA_EINVAL, "budget must be >= 1 with ids");
  const int max_len = (int)std::min<int64_t>(max_kv_len, cache_cap);

  gqa_plan plan;
  st = attn_decode_plan(n_tok, n_seq, n_heads, n_kv_heads, head_dim, max_len, ids ? budget : -1,
                        kind, 0, &plan);
  if (st != GQA_OK) return st;
  if (plan.merge && (!ws || ws_bytes < plan.ws_bytes || !aligned16(ws)))
    return fail(GQA_EWORKSPACE, "workspace needs %zu bytes (16-byte aligned), got %zu",
                plan.ws_bytes, ws ? ws_bytes : (size_t)0);

  gqa::PartialParams p{};
  p.q = q;
  p.kc = kc;
  p.vc = vc;
  p.ksc = reinterpret_cast<const __half*>(ksc);
  p.vsc = reinterpret_cast<const __half*>(vsc);
  p.sc_shift = scale_group == 32 ? 5 : 6;
  p.ids = ids;
  p.kv_len = kv_len;
  p.seq_of = seq_of;
  p.out = out;
  p.err = err_word;
  p.n_tok = n_tok;
  p.n_seq = n_seq;
  p.n_heads = n_heads;
  p.n_kv_heads = n_kv_heads;
  p.group = n_heads / n_kv_heads;
  p.head_split = 1;
  p.cache_cap = cache_cap;
  p.max_kv_len = max_len;
  p.budget = ids ? budget : INT32_MAX;
  p.chunk = plan.chunk;
  p.n_split = plan.n_split;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.merge = plan.merge;
  p.gate = gate;
  p.gate_stride = gate ? gate_stride : 0;
  // the per-row f16 tensor-core kernel goes out as a programmatic dependent of whatever precedes
  // it on the stream: its launch and rasterisation overlap that kernel's tail (GB300, back-to-back
  // steps: long context 143.2 -> 141.8 us, batched 296.8 -> 295.0); GQA_PDL=0 launches it plainly
  {
    const char* pd = std::getenv("GQA_PDL");
    p.pdl = !(pd && std::strcmp(pd, "0") == 0);
  }
  if (plan.streamk) {  // ws = [arrival counters][piece records]
    const size_t cnt = ((size_t)n_tok * n_kv_heads * sizeof(uint32_t) + 255) / 256 * 256;
    p.counters = static_cast<unsigned int*>(ws);
    p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + cnt);
  } else if (plan.merge) {  // ws = [arrival counters][partials][n_valid], 256-byte aligned
    const size_t cnt = ((size_t)n_tok * plan.grid_y * sizeof(uint32_t) + 255) / 256 * 256;
    const size_t part = (size_t)n_tok * plan.n_split * n_heads * (head_dim + 2) * sizeof(float);
    p.counters = static_cast<unsigned int*>(ws);
    p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + cnt);
    p.n_valid = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + cnt + (part + 255) / 256 * 256);
  }

  CUtensorMap tk, tv, tq;
  std::memset(&tk, 0, sizeof tk);
  std::memset(&tv, 0, sizeof tv);
  std::memset(&tq, 0, sizeof tq);
  if (kind == GQA_KIND_F16) {
    auto encode = tensor_map_encoder();
    if (!encode) return fail(GQA_ECUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_kv_heads,
                                (cuuint64_t)n_seq * (cuuint64_t)cache_cap};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2,
                                   (cuuint64_t)head_dim * 2 * (cuuint64_t)n_kv_heads};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)plan.tile};
    const cuuint32_t estr[3] = {1, 1, 1};
    for (int i = 0; i < 2; ++i) {
      CUresult r = encode(i ? &tv : &tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void*>(i ? vc : kc), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(GQA_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    if (plan.row_group > 1 && gqa::rows_on_umma()) {
      // the tcgen05 row kernel stages a group's fp32 q [rows][G heads][D] with one copy: box
      // D x G x 64 / G rows (rows past n_tok read as zeros)
      const int G = n_heads / n_kv_heads;
      const cuuint64_t qdims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_heads, (cuuint64_t)n_tok};
      const cuuint64_t qstr[2] = {(cuuint64_t)head_dim * 4,
                                  (cuuint64_t)head_dim * 4 * (cuuint64_t)n_heads};
      const cuuint32_t qbox[3] = {(cuuint32_t)head_dim, (cuuint32_t)G, (cuuint32_t)(64 / G)};
      CUresult r = encode(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(q), qdims,
                          qstr, qbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(GQA_ECUDA, "cuTensorMapEncodeTiled (q) failed (%d)", (int)r);
    }
  }

  p.head_split = plan.streamk ? 1 : plan.grid_y / n_kv_heads;
  gqa::Variant var = gqa::pick_variant(p.group / p.head_split);
  {
    // int8 grids smaller than the GPU (a few rows of selected cells) are latency-bound: eight
    // row slices per stage give each CTA twice the consumer warps (GB300, the 1024-of-8192
    // selected-cell workload: 17.0 us per step against 18.9 with four)
    st = GQA_OK;
    const long long ctas = (long long)plan.grid_x * plan.grid_y * plan.grid_z;
    if (kind == GQA_KIND_Q8 && !var.mma && var.gw == 4 && var.nps == 4 && !plan.streamk &&
        ctas < current_sm_count(&st))
      var.nps = 8;
  }
  const int nhg = (p.group / p.head_split + var.gw - 1) / var.gw;
  const int threads = 32 * (nhg * var.nps + 1);
  // f16 caches run on the tensor cores unless GQA_F16_KERNEL=fma asks for the CUDA-core kernel,
  // int8 caches unless GQA_Q8_KERNEL=fma does
  if (kind == GQA_KIND_F16) {
    const char* k = std::getenv("GQA_F16_KERNEL");
    var.mma = !(k && std::strcmp(k, "fma") == 0);
  } else if (kind == GQA_KIND_Q8) {
    var.mma = gqa::q8_on_mma() ? 1 : 0;
  }
  const dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
  // grouped rows on the tcgen05 kernel merge their own partials when the whole grid fits one
  // CTA per SM (a cooperative launch); otherwise merge_kernel follows
  // one sequence on the tcgen05 row kernel: its groups are fixed runs of rows, found without a
  // scan of seq_of (GB300, 16 rows of one 8192-position sequence: 18.47 us per step against 18.56)
  if (kind == GQA_KIND_F16 && plan.row_group > 1 && gqa::rows_on_umma() && n_seq == 1)
    p.rows_fixed = 1;
  if (plan.merge && !plan.streamk && plan.row_group > 1 && gqa::rows_on_umma()) {
    st = GQA_OK;
    const long long ctas = (long long)plan.grid_x * plan.grid_y * plan.grid_z;
    p.fused_merge = ctas <= current_sm_count(&st) ? 1 : 0;
  }
  // a split f16 grid that fits the GPU (latency-bound: a few short rows) may merge each row's
  // chunks inside a thread-block cluster (partial_mma.cuh); GQA_F16_CLUSTER=0 keeps the
  // last-CTA merge through the workspace
  if (kind == GQA_KIND_F16 && plan.merge && !plan.streamk && plan.row_group == 1 && var.mma) {
    st = GQA_OK;
    const long long ctas = (long long)plan.grid_x * plan.grid_y * plan.grid_z;
    const char* k = std::getenv("GQA_F16_CLUSTER");
    p.cluster = ctas <= current_sm_count(&st) && !(k && std::strcmp(k, "0") == 0) ? 1 : 0;
  }
  // polls of the fused merge's wait before it gives up; GQA_MERGE_SPIN (tests) sets fewer,
  // 0 making every such wait run out at once
  const char* spin = std::getenv("GQA_MERGE_SPIN");
  p.merge_spin = spin ? (unsigned)std::strtoul(spin, nullptr, 10) : gqa::kSpinLimit;
  cudaError_t e =
      plan.streamk        ? gqa::launch_streamk_f16(head_dim, tk, tv, p, grid, stream)
      : plan.row_group > 1 ? gqa::launch_rows_f16(head_dim, tk, tv, tq, p, grid, stream)
                           : gqa::launch_partial(kind, head_dim, var, tk, tv, p, grid, threads, stream);
  if (e == cudaErrorCooperativeLaunchTooLarge && p.fused_merge) {  // not all resident after all
    (void)cudaGetLastError();
    p.fused_merge = 0;
    e = gqa::launch_rows_f16(head_dim, tk, tv, tq, p, grid, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "partial kernel launch");
  if (plan.merge && !plan.streamk && plan.row_group > 1 && !p.fused_merge) {
    // grouped rows: their partials are merged by merge_kernel, one warp per (row, head)
    e = gqa::launch_merge(head_dim, p.part, p.n_valid, plan.n_split, n_tok, n_heads, out, stream,
                          p.gate, p.gate_stride, /*after_partials=*/true);
    if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  }
  return GQA_OK;  // otherwise split rows were merged inside the kernel by their last CTA
}

}  // namespace

extern "C" {

gqa_status attn_decode_f16(const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                           float* out, const int32_t* kv_len, const int32_t* seq_of, int n_tok,
                           int n_seq, int n_heads, int n_kv_heads, int head_dim,
                           int64_t cache_cap, int max_kv_len, float scale, void* ws,
                           size_t ws_bytes, int32_t* err_word, cudaStream_t stream) {
  return decode_common(GQA_KIND_F16, q, k_cache, v_cache, nullptr, nullptr, nullptr, -1, out,
                       kv_len, seq_of, n_tok, n_seq, n_heads, n_kv_heads, head_dim, cache_cap,
                       max_kv_len, scale, ws, ws_bytes, err_word, stream);
}

gqa_status attn_decode_q8_sel(const float* q, const int8_t* kq, const int8_t* vq,
                              const uint16_t* ksc, const uint16_t* vsc, const int32_t* ids,
                              int budget, float* out, const int32_t* kv_len,
                              const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                              int n_kv_heads, int head_dim, int64_t cache_cap, int max_kv_len,
                              float scale, void* ws, size_t ws_bytes, int32_t* err_word,
                              cudaStream_t stream) {
  return decode_common(GQA_KIND_Q8, q, kq, vq, ksc, vsc, ids, budget, out, kv_len, seq_of, n_tok,
                       n_seq, n_heads, n_kv_heads, head_dim, cache_cap, max_kv_len, scale, ws,
                       ws_bytes, err_word, stream);
}

gqa_status attn_decode_q8_sel_sg(const float* q, const int8_t* kq, const int8_t* vq,
                                 const uint16_t* ksc, const uint16_t* vsc, int scale_group,
                                 const int32_t* ids, int budget, float* out,
                                 const int32_t* kv_len, const int32_t* seq_of, int n_tok,
                                 int n_seq, int n_heads, int n_kv_heads, int head_dim,
                                 int64_t cache_cap, int max_kv_len, float scale, void* ws,
                                 size_t ws_bytes, int32_t* err_word, cudaStream_t stream) {
  return decode_common(GQA_KIND_Q8, q, kq, vq, ksc, vsc, ids, budget, out, kv_len, seq_of, n_tok,
                       n_seq, n_heads, n_kv_heads, head_dim, cache_cap, max_kv_len, scale, ws,
                       ws_bytes, err_word, stream, scale_group);
}

gqa_status attn_decode_f16_gated(const float* q, const uint16_t* k_cache,
                                 const uint16_t* v_cache, float* out, const int32_t* kv_len,
                                 const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                                 int n_kv_heads, int head_dim, int64_t cache_cap, int max_kv_len,
                                 float scale, const float* gate, int64_t gate_stride, void* ws,
                                 size_t ws_bytes, int32_t* err_word, cudaStream_t stream) {
  if (!gate) return fail(GQA_EINVAL, "attn_decode_f16_gated: gate is NULL");
  return decode_common(GQA_KIND_F16, q, k_cache, v_cache, nullptr, nullptr, nullptr, -1, out,
                       kv_len, seq_of, n_tok, n_seq, n_heads, n_kv_heads, head_dim, cache_cap,
                       max_kv_len, scale, ws, ws_bytes, err_word, stream, 64, gate, gate_stride);
}

gqa_status attn_decode_q8_sel_gated(const float* q, const int8_t* kq, const int8_t* vq,
                                    const uint16_t* ksc, const uint16_t* vsc, int scale_group,
                                    const int32_t* ids, int budget, float* out,
                                    const int32_t* kv_len, const int32_t* seq_of, int n_tok,
                                    int n_seq, int n_heads, int n_kv_heads, int head_dim,
                                    int64_t cache_cap, int max_kv_len, float scale,
                                    const float* gate, int64_t gate_stride, void* ws,
                                    size_t ws_bytes, int32_t* err_word, cudaStream_t stream) {
  if (!gate) return fail(GQA_EINVAL, "attn_decode_q8_sel_gated: gate is NULL");
  return decode_common(GQA_KIND_Q8, q, kq, vq, ksc, vsc, ids, budget, out, kv_len, seq_of, n_tok,
                       n_seq, n_heads, n_kv_heads, head_dim, cache_cap, max_kv_len, scale, ws,
                       ws_bytes, err_word, stream, scale_group, gate, gate_stride);
}

gqa_status attn_merge_gated(const float* part, const int32_t* n_valid, int n_split, int n_tok,
                            int n_heads, int head_dim, const float* gate, int64_t gate_stride,
                            float* out, cudaStream_t stream) {
  if (!gate) return fail(GQA_EINVAL, "attn_merge_gated: gate is NULL");
  if (gate_stride < head_dim || (gate_stride & 1) || (reinterpret_cast<uintptr_t>(gate) & 7))
    return fail(GQA_EINVAL, "attn_merge_gated: gate 8-byte aligned, gate_stride even and >= head_dim");
  if (n_tok < 0 || n_tok > 65535 || n_heads <= 0 || n_heads > 65535 || n_split <= 0)
    return fail(GQA_EINVAL, "bad sizes n_tok %d n_heads %d n_split %d", n_tok, n_heads, n_split);
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(GQA_EINVAL, "head_dim %d not in {64, 128, 256}", head_dim);
  if (n_tok == 0) return GQA_OK;
  if (!part || !n_valid || !out) return fail(GQA_EINVAL, "a required pointer is NULL");
  if (!aligned16(part) || !aligned16(out)) return fail(GQA_EINVAL, "part/out not 16-byte aligned");
  cudaError_t e = gqa::launch_merge(head_dim, part, n_valid, n_split, n_tok, n_heads, out, stream,
                                    gate, gate_stride);
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  return GQA_OK;
}

gqa_status attn_merge(const float* part, const int32_t* n_valid, int n_split, int n_tok,
                      int n_heads, int head_dim, float* out, cudaStream_t stream) {
  if (n_tok < 0 || n_tok > 65535 || n_heads <= 0 || n_heads > 65535 || n_split <= 0)
    return fail(GQA_EINVAL, "bad sizes n_tok %d n_heads %d n_split %d", n_tok, n_heads, n_split);
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(GQA_EINVAL, "head_dim %d not in {64, 128, 256}", head_dim);
  if (n_tok == 0) return GQA_OK;
  if (!part || !n_valid || !out) return fail(GQA_EINVAL, "a required pointer is NULL");
  if (!aligned16(part) || !aligned16(out)) return fail(GQA_EINVAL, "part/out not 16-byte aligned");
  cudaError_t e = gqa::launch_merge(head_dim, part, n_valid, n_split, n_tok, n_heads, out, stream);
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  return GQA_OK;
}

}  // extern "C"
