// astr_decode_attention_noalloc: paged decode whose split-K scratch is a fixed array inside
// this library instead of buffers the caller allocates.
//
// Some callers cannot call cudaMalloc: plugin hosts that hand a library only the tensors of
// one call, embedded runtimes that reserve all device memory at start-up and forbid later
// allocations, and serving loops that must never block on the allocator. For them this
// entry point keeps the log-sum-exp partials of split-K decode
// in `g_split_scratch`, a static device array of kScratchBytes (8 MiB) that every GPU loading
// the library holds until the process exits. The call itself allocates nothing: it fills in
// the partial-buffer fields of a private copy of the caller's astr_kv_cache and hands it to
// astr_decode_attention unchanged.
#include <stdio.h>

#include <mutex>

#include "astr_internal.cuh"
#include "launch.h"

namespace astr {
namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;
constexpr size_t kScratchFloats = kScratchBytes / sizeof(float);

// Shared by every call on a device and never cleared: each call writes every partial entry
// it later reads, so nothing has to start at zero. Calls whose work overlaps on the GPU
// (issued to different streams) race on it.
static __device__ __align__(256) float g_split_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device. The host-side name g_split_scratch
// is only a stand-in, so the address is looked up once per device, with that device current.
cudaError_t scratch_on_current_device(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace astr

using namespace astr;

extern "C" {

astr_status astr_decode_attention_noalloc(const astr_kv_cache *kv, int32_t layer_id,
                                          const void *q, int32_t n_heads, astr_stream stream) {
  char msg[320];
  if (!kv) {
    set_last_error_message("kv is NULL");
    return ASTR_ERR_INVALID;
  }
  astr_kv_cache k2 = *kv;
  k2.decode_o_part = nullptr;
  k2.decode_ml_part = nullptr;
  k2.max_splits = 0;
  if (kv->batch > 0 && kv->n_kv_heads > 0 && n_heads > 0 && kv->head_dim > 0) {
    // splits per (request, head) that fit: o_part [B, H, S, D] and ml_part [B, H, S, 2]
    const int64_t per_split = (int64_t)kv->batch * n_heads * (kv->head_dim + 2);
    const int64_t cap = (int64_t)(kScratchFloats / (size_t)per_split);
    if (kv->split_chunk > 0 && kv->max_len > kv->split_chunk) {
      const int64_t need = (kv->max_len + (int64_t)kv->split_chunk - 1) / kv->split_chunk;
      if (need > cap) {
        snprintf(msg, sizeof msg,
                 "split_chunk %d needs %lld splits of %lld bytes; the built-in split-K scratch "
                 "holds %zu bytes (%lld splits): raise split_chunk or use astr_decode_attention",
                 kv->split_chunk, (long long)need, (long long)(per_split * 4), kScratchBytes,
                 (long long)cap);
        set_last_error_message(msg);
        return ASTR_ERR_INVALID;
      }
    }
    if (cap >= 2) {
      float *base = nullptr;
      cudaError_t e = scratch_on_current_device(&base);
      if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "looking up the split-K scratch: %s", cudaGetErrorString(e));
        set_last_error_message(msg);
        return ASTR_ERR_CUDA;
      }
      const int32_t S = cap > 1 << 20 ? 1 << 20 : (int32_t)cap;
      k2.max_splits = S;
      k2.decode_o_part = base;
      k2.decode_ml_part = base + (int64_t)kv->batch * n_heads * S * kv->head_dim;
    }
  }
  return astr_decode_attention(&k2, layer_id, q, n_heads, stream);
}

}  // extern "C"
