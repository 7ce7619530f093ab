// noalloc.cu -- attn_decode_f16_noalloc: the f16 decode call with its scratch in a static device
// array, for callers that cannot allocate device memory themselves.
//
// Some hosts own every byte of device memory and give a plug-in no allocator: an inference
// server that carves a fixed arena at start-up and forbids cudaMalloc afterwards, or a foreign
// runtime that calls this library through its C ABI with only input and output buffers in hand.
// Such a caller cannot provide the `ws` buffer that attn_decode_f16 needs once a row is split
// into several KV chunks.  This entry point supplies that buffer from a file-scope __device__
// array instead, so it allocates nothing at all.
//
// The array's name in host code is only a host-side stand-in, never a device address.  The real
// address is looked up once per device with cudaGetSymbolAddress, on the first call made while
// that device is current, and cached.
#include <cuda_runtime_api.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "gqa_decode.h"

namespace gqa {
void set_last_error(const char* msg);  // host.cu: the text gqa_last_error() returns
}

namespace {

// Scratch shared by every call on a device; held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GQA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_addr[128] = {nullptr};  // device address of g_noalloc_scratch, per device id

}  // namespace

extern "C" {

gqa_status attn_decode_f16_noalloc(const float* q, const uint16_t* k_cache,
                                   const uint16_t* v_cache, float* out, const int32_t* kv_len,
                                   const int32_t* seq_of, int n_tok, int n_seq, int n_heads,
                                   int n_kv_heads, int head_dim, int64_t cache_cap,
                                   int max_kv_len, float scale, int32_t* err_word,
                                   cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    gqa::set_last_error((std::string("cudaGetDevice: ") + cudaGetErrorString(e)).c_str());
    return GQA_ECUDA;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
      e = cudaGetSymbolAddress(&g_addr[dev], g_noalloc_scratch);
      if (e != cudaSuccess) {
        g_addr[dev] = nullptr;
        gqa::set_last_error(
            (std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e)).c_str());
        return GQA_ECUDA;
      }
    }
    scratch = g_addr[dev];
  }
  // The same plan attn_decode_f16 will use; reject what does not fit before anything launches.
  const int64_t len = max_kv_len < cache_cap ? max_kv_len : cache_cap;
  const size_t need = attn_decode_workspace_bytes(n_tok, n_seq, n_heads, n_kv_heads, head_dim,
                                                  len < 0 ? -1 : (int)len, -1, GQA_KIND_F16);
  if (need > (size_t)GQA_NOALLOC_SCRATCH_BYTES) {
    char buf[256];
    snprintf(buf, sizeof buf,
             "these sizes need %zu bytes of scratch; the static scratch holds %d bytes",
             need, GQA_NOALLOC_SCRATCH_BYTES);
    gqa::set_last_error(buf);
    return GQA_EWORKSPACE;
  }
  return attn_decode_f16(q, k_cache, v_cache, out, kv_len, seq_of, n_tok, n_seq, n_heads,
                         n_kv_heads, head_dim, cache_cap, max_kv_len, scale, scratch,
                         GQA_NOALLOC_SCRATCH_BYTES, err_word, stream);
}

}  // extern "C"
