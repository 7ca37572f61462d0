// extern "C" entry points of libastr.so: host-side validation, split planning, launches,
// checked mode and the per-device error word. The operations themselves are defined in
// include/astr.h with the passages of the AstrAI pages they follow.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <string>
#include <vector>

#include "astr_internal.cuh"
#include "launch.h"

namespace astr {

__device__ uint32_t g_error_word = 0;

namespace {

// device address of g_error_word on the current device (looked up once per device)
uint32_t *error_word() {
  static std::atomic<uint32_t *> cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  uint32_t *w = cache[dev].load(std::memory_order_acquire);
  if (!w) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    w = static_cast<uint32_t *>(p);
    cache[dev].store(w, std::memory_order_release);
  }
  return w;
}

thread_local std::string t_last_error;
std::atomic<int> g_checked{0};
std::atomic<int64_t> g_wait_ns{1000000000LL};

astr_status fail(astr_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
astr_status fail(astr_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

astr_status ok() {
  t_last_error.clear();
  return ASTR_OK;
}

astr_status cuda_fail(cudaError_t e, const char *what) {
  return fail(ASTR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

astr_status check_cache(const astr_kv_cache *kv, int32_t layer_id, int32_t n_heads) {
  if (!kv) return fail(ASTR_ERR_INVALID, "kv is NULL");
  if (!kv->k_buffer || !kv->v_buffer) return fail(ASTR_ERR_INVALID, "k_buffer / v_buffer is NULL");
  if (!aligned16(kv->k_buffer) || !aligned16(kv->v_buffer))
    return fail(ASTR_ERR_INVALID, "k_buffer / v_buffer must be 16-byte aligned");
  if (kv->dtype != ASTR_F32 && kv->dtype != ASTR_BF16)
    return fail(ASTR_ERR_UNSUPPORTED, "dtype %d is not ASTR_F32 or ASTR_BF16", kv->dtype);
  if (kv->head_dim != 64 && kv->head_dim != 128)
    return fail(ASTR_ERR_UNSUPPORTED, "head_dim %d is not 64 or 128", kv->head_dim);
  if (kv->n_kv_heads < 1) return fail(ASTR_ERR_INVALID, "n_kv_heads %d < 1", kv->n_kv_heads);
  if (n_heads < 1 || n_heads % kv->n_kv_heads != 0)
    return fail(ASTR_ERR_INVALID, "n_heads %d is not a positive multiple of n_kv_heads %d", n_heads,
                kv->n_kv_heads);
  if (kv->n_layers < 1 || layer_id < 0 || layer_id >= kv->n_layers)
    return fail(ASTR_ERR_INVALID, "layer_id %d outside [0, %d)", layer_id, kv->n_layers);
  if (kv->size < 1) return fail(ASTR_ERR_INVALID, "size %lld < 1", (long long)kv->size);
  return ASTR_OK;
}

astr_status check_table(const astr_kv_cache *kv) {
  if (!kv->req_to_token || !kv->req_pool_indices)
    return fail(ASTR_ERR_INVALID, "req_to_token / req_pool_indices is NULL");
  if (kv->num_reqs < 1 || kv->max_ctx_len < 1)
    return fail(ASTR_ERR_INVALID, "req_to_token shape [%d, %d] is empty", kv->num_reqs, kv->max_ctx_len);
  return ASTR_OK;
}

// after the launches of one entry point: checked mode synchronises and reads the error word
astr_status finish(cudaStream_t s) {
  if (!g_checked.load()) return ok();
  uint32_t flags = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&flags, g_error_word, sizeof flags, 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "checked mode: reading the device error word");
  if (flags) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "checked mode: clearing the device error word");
    if (flags & ASTR_DEVERR_TIMEOUT)
      return fail(ASTR_ERR_TIMEOUT, "a kernel wait ran out of time (error word 0x%x)", flags);
    return fail(ASTR_ERR_INDEX, "a kernel met an out-of-range index (error word 0x%x)", flags);
  }
  return ok();
}

bool use_tc_decode(const astr_kv_cache *kv, int n_heads) {
  return tc_decode_supported(kv->dtype, kv->head_dim, n_heads / kv->n_kv_heads);
}

int decode_chunk(const astr_kv_cache *kv, int n_heads) {
  const int max_len = kv->max_len;
  if (kv->split_chunk > 0) return kv->split_chunk;
  if (!kv->decode_o_part || !kv->decode_ml_part || kv->max_splits <= 1) return max_len;
  const bool tc = use_tc_decode(kv, n_heads);
  const int tile = tc ? tc_decode_tile_tokens() : simt_tile_tokens(n_heads / kv->n_kv_heads);
  // The persistent tensor-core kernel claims each split's requests longest first, so whole
  // requests balance the SMs once there are six (per KV head) per SM: then nothing is split and
  // nothing merged (measured on GB300, 256 requests x 4 KV heads: 331.5 us unsplit against
  // 347 us in 3072-token chunks).
  if (tc && kv->batch <= tc_decode_ranked_batch_max() &&
      (int64_t)kv->batch * kv->n_kv_heads >= 6 * (int64_t)num_sms())
    return max_len;
  // Otherwise, taking the mean length as half of max_len, aim for about four work items per SM
  // for the tensor-core kernel (measured on GB300) or four waves of three resident blocks per
  // SM for the CUDA-core kernel; keep the chunk within [lo, 4096] tokens and never need more
  // splits than the scratch holds.
  const int64_t est_tokens = (int64_t)kv->batch * max_len / 2;
  const int64_t target_blocks = (int64_t)num_sms() * (tc ? 4 : 12);
  int64_t c = est_tokens * kv->n_kv_heads / (target_blocks > 0 ? target_blocks : 1);
  const int64_t lo = tc ? 512 : 256;
  if (c < lo) c = lo;
  if (c > 4096) c = 4096;
  const int64_t min_c = (max_len + kv->max_splits - 1) / kv->max_splits;
  if (c < min_c) c = min_c;
  c = (c + tile - 1) / tile * tile;
  if (c >= max_len) c = max_len;
  return (int)c;
}

}  // namespace

// ------------------------------------------------------------------------------------------
// checked-mode metadata validation
// ------------------------------------------------------------------------------------------
namespace {
__global__ void validate_kernel(const astr_kv_cache kv, int what, uint32_t *err) {
  const int tid = threadIdx.x;
  if (what == VALIDATE_DECODE) {
    for (int b = tid; b < kv.batch; b += blockDim.x) {
      const int L = kv.seq_lens[b];
      if (L < 1 || L > kv.max_len || L > kv.max_ctx_len) raise_error(err, ASTR_DEVERR_LEN);
      const int r = kv.req_pool_indices[b];
      if (r < 0 || r >= kv.num_reqs) raise_error(err, ASTR_DEVERR_ROW);
      if (kv.kv_indptr && kv.kv_indptr[b + 1] - kv.kv_indptr[b] != L) raise_error(err, ASTR_DEVERR_META);
    }
    if (tid == 0 && kv.kv_indptr && kv.kv_indptr[0] != 0) raise_error(err, ASTR_DEVERR_META);
    return;
  }
  // prefill: indptr sanity, every tile inside its request, non-empty entries = sum
  // ceil(Q/rows), and no two tiles naming the same (request, index)
  __shared__ long long total, real;
  if (tid == 0) total = real = 0;
  __syncthreads();
  long long mine = 0;
  for (int b = tid; b < kv.batch; b += blockDim.x) {
    const int Q = kv.qo_indptr[b + 1] - kv.qo_indptr[b];
    const int K = kv.kv_indptr[b + 1] - kv.kv_indptr[b];
    if (Q < 0 || K < Q || K > kv.max_ctx_len) raise_error(err, ASTR_DEVERR_LEN);
    const int r = kv.req_pool_indices[b];
    if (r < 0 || r >= kv.num_reqs) raise_error(err, ASTR_DEVERR_ROW);
    if (Q > 0) mine += (Q + kv.q_tile_rows - 1) / kv.q_tile_rows;
  }
  atomicAdd(reinterpret_cast<unsigned long long *>(&total), (unsigned long long)mine);
  __syncthreads();
  if (tid == 0 && (kv.qo_indptr[0] != 0 || kv.kv_indptr[0] != 0)) raise_error(err, ASTR_DEVERR_META);
  long long mine_real = 0;
  for (int t = tid; t < kv.num_q_tiles; t += blockDim.x) {
    const int b = kv.q_tile_to_batch[t], i = kv.q_tile_to_index[t];
    if (b == -1) continue;  // an empty entry
    ++mine_real;
    if (b < 0 || b >= kv.batch) {
      raise_error(err, ASTR_DEVERR_META);
      continue;
    }
    const int Q = kv.qo_indptr[b + 1] - kv.qo_indptr[b];
    if (i < 0 || (long long)i * kv.q_tile_rows >= Q) raise_error(err, ASTR_DEVERR_META);
    for (int u = t + 1; u < kv.num_q_tiles; ++u)
      if (kv.q_tile_to_batch[u] == b && kv.q_tile_to_index[u] == i) raise_error(err, ASTR_DEVERR_META);
  }
  atomicAdd(reinterpret_cast<unsigned long long *>(&real), (unsigned long long)mine_real);
  __syncthreads();
  if (tid == 0 && real != total) raise_error(err, ASTR_DEVERR_META);
}
}  // namespace

namespace {
__global__ void selftest_wait_kernel(uint64_t ns, uint32_t *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, ns, err);  // nothing arrives: the wait must run out
}
}  // namespace

void set_last_error_message(const char *msg) { t_last_error = msg ? msg : ""; }

cudaError_t launch_validate(const astr_kv_cache &kv, int what, uint32_t *err, cudaStream_t stream) {
  validate_kernel<<<1, 1024, 0, stream>>>(kv, what, err);
  return cudaGetLastError();
}

}  // namespace astr

namespace astr {
namespace {
astr_status decode_impl(const astr_kv_cache *kv, int32_t layer_id, const void *q, int32_t n_heads,
                        astr_stream stream, const DecodeRope *rope);
}  // namespace
}  // namespace astr

namespace astr {
namespace {
astr_status rope_apply_impl(const void *q, void *q_out, const void *k, void *k_out,
                            int64_t n_tokens, int32_t n_heads, int32_t n_kv_heads,
                            int32_t head_dim, int32_t dtype, const float *freqs_cis,
                            int32_t freqs_max_len, const int32_t *position_ids, bool inverse,
                            astr_stream stream, const char *name) {
  if (n_tokens < 0 || n_heads < 0 || n_kv_heads < 0)
    return fail(ASTR_ERR_INVALID, "%s: n_tokens %lld, n_heads %d, n_kv_heads %d", name,
                (long long)n_tokens, n_heads, n_kv_heads);
  if (dtype != ASTR_F32 && dtype != ASTR_BF16) return fail(ASTR_ERR_INVALID, "%s: dtype %d", name, dtype);
  if (head_dim != 64 && head_dim != 128)
    return fail(ASTR_ERR_UNSUPPORTED, "%s: head_dim %d (64 or 128)", name, head_dim);
  if (n_tokens == 0 || n_heads + n_kv_heads == 0) return ok();
  if (!freqs_cis || !position_ids || (n_heads > 0 && (!q || !q_out)) ||
      (n_kv_heads > 0 && (!k || !k_out)))
    return fail(ASTR_ERR_INVALID, "%s: a NULL tensor", name);
  if ((n_heads > 0 && (!aligned16(q) || !aligned16(q_out))) ||
      (n_kv_heads > 0 && (!aligned16(k) || !aligned16(k_out))) || !aligned16(freqs_cis))
    return fail(ASTR_ERR_INVALID, "%s: tensors and freqs_cis must be 16-byte aligned", name);
  if (freqs_max_len < 1) return fail(ASTR_ERR_INVALID, "%s: freqs_max_len %d < 1", name, freqs_max_len);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t *err = error_word();
  if (!err) return fail(ASTR_ERR_CUDA, "no CUDA device / error word unavailable");
  cudaError_t e = launch_rope_apply(q, q_out, k, k_out, n_tokens, n_heads, n_kv_heads, head_dim,
                                    dtype, freqs_cis, freqs_max_len, position_ids, inverse, s,
                                    num_sms(), err);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return finish(s);
}
}  // namespace
}  // namespace astr

using namespace astr;

extern "C" {

int32_t astr_version(void) { return 100; }

int32_t astr_kv_cache_bytes(void) { return (int32_t)sizeof(astr_kv_cache); }

const char *astr_last_error(void) { return t_last_error.c_str(); }

astr_status astr_set_checked(int32_t on) {
  g_checked.store(on ? 1 : 0);
  return ok();
}

astr_status astr_set_wait_timeout_ns(int64_t ns) {
  g_wait_ns.store(ns < 1 ? 1 : ns);
  return ok();
}

astr_status astr_device_error(astr_stream stream, uint32_t *flags) {
  if (!flags) return fail(ASTR_ERR_INVALID, "flags is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  const uint32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_error_word, sizeof v, 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  *flags = v;
  return ok();
}

astr_status astr_selftest_wait_timeout(astr_stream stream, int64_t ns) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t *err = error_word();
  if (!err) return fail(ASTR_ERR_CUDA, "no CUDA device / error word unavailable");
  selftest_wait_kernel<<<1, 32, 0, s>>>((uint64_t)(ns < 1 ? 1 : ns), err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  uint32_t flags = 0;
  const uint32_t zero = 0;
  e = cudaMemcpyFromSymbolAsync(&flags, g_error_word, sizeof flags, 0, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "self-test synchronisation");
  if (flags & ASTR_DEVERR_TIMEOUT) return fail(ASTR_ERR_TIMEOUT, "the bounded wait ran out (expected)");
  return ok();
}

astr_status astr_rope_kv_write(const astr_kv_cache *kv, int32_t layer_id, const void *q,
                               void *q_out, const void *k, const void *v, int32_t n_heads,
                               const float *freqs_cis, int32_t freqs_max_len,
                               const int32_t *position_ids, astr_stream stream) {
  astr_status st = check_cache(kv, layer_id, n_heads);
  if (st != ASTR_OK) return st;
  if (kv->n_tokens < 0) return fail(ASTR_ERR_INVALID, "n_tokens %lld < 0", (long long)kv->n_tokens);
  if (kv->n_tokens == 0) return ok();
  if (!q || !q_out || !k || !v || !freqs_cis || !position_ids || !kv->out_cache_loc)
    return fail(ASTR_ERR_INVALID, "q, q_out, k, v, freqs_cis, position_ids and out_cache_loc must be non-NULL");
  if (!aligned16(q) || !aligned16(q_out) || !aligned16(k) || !aligned16(v) || !aligned16(freqs_cis))
    return fail(ASTR_ERR_INVALID, "q, q_out, k, v and freqs_cis must be 16-byte aligned");
  if (freqs_max_len < 1) return fail(ASTR_ERR_INVALID, "freqs_max_len %d < 1", freqs_max_len);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t *err = error_word();
  if (!err) return fail(ASTR_ERR_CUDA, "no CUDA device / error word unavailable");
  cudaError_t e = launch_rope_kv_write(*kv, layer_id, q, q_out, k, v, n_heads, freqs_cis,
                                       freqs_max_len, position_ids, s, num_sms(), err);
  if (e != cudaSuccess) return cuda_fail(e, "astr_rope_kv_write launch");
  return finish(s);
}


astr_status astr_rope_apply(const void *q, void *q_out, const void *k, void *k_out,
                            int64_t n_tokens, int32_t n_heads, int32_t n_kv_heads,
                            int32_t head_dim, int32_t dtype, const float *freqs_cis,
                            int32_t freqs_max_len, const int32_t *position_ids,
                            astr_stream stream) {
  return astr::rope_apply_impl(q, q_out, k, k_out, n_tokens, n_heads, n_kv_heads, head_dim, dtype,
                               freqs_cis, freqs_max_len, position_ids, false, stream,
                               "astr_rope_apply");
}

astr_status astr_rope_backward(const void *grad_q_out, void *grad_q, const void *grad_k_out,
                               void *grad_k, int64_t n_tokens, int32_t n_heads,
                               int32_t n_kv_heads, int32_t head_dim, int32_t dtype,
                               const float *freqs_cis, int32_t freqs_max_len,
                               const int32_t *position_ids, astr_stream stream) {
  return astr::rope_apply_impl(grad_q_out, grad_q, grad_k_out, grad_k, n_tokens, n_heads,
                               n_kv_heads, head_dim, dtype, freqs_cis, freqs_max_len,
                               position_ids, true, stream, "astr_rope_backward");
}

astr_status astr_decode_plan(const astr_kv_cache *kv, int32_t n_heads, int32_t *split_chunk,
                             int32_t *n_splits) {
  if (!kv || !split_chunk || !n_splits) return fail(ASTR_ERR_INVALID, "NULL argument");
  if (kv->n_kv_heads < 1 || n_heads < 1 || n_heads % kv->n_kv_heads)
    return fail(ASTR_ERR_INVALID, "n_heads %d / n_kv_heads %d", n_heads, kv->n_kv_heads);
  if (kv->max_len < 1) return fail(ASTR_ERR_INVALID, "max_len %d < 1", kv->max_len);
  const int c = decode_chunk(kv, n_heads);
  *split_chunk = c;
  *n_splits = (kv->max_len + c - 1) / c;
  return ok();
}

astr_status astr_prefill_tiles(const int32_t *q_lens, const int32_t *kv_lens, int32_t batch,
                               int32_t q_tile_rows, int32_t *qo_indptr, int32_t *kv_indptr,
                               int32_t *q_tile_to_batch, int32_t *q_tile_to_index,
                               int32_t max_tiles, int32_t *num_tiles) {
  if (!num_tiles || !qo_indptr || !kv_indptr || (batch > 0 && (!q_lens || !kv_lens)))
    return fail(ASTR_ERR_INVALID, "NULL argument");
  if (batch < 0 || q_tile_rows < 1 || max_tiles < 0)
    return fail(ASTR_ERR_INVALID, "batch %d, q_tile_rows %d, max_tiles %d", batch, q_tile_rows, max_tiles);
  int64_t qsum = 0, ksum = 0, tiles = 0;
  for (int32_t b = 0; b < batch; ++b) {
    if (q_lens[b] < 0 || kv_lens[b] < q_lens[b])
      return fail(ASTR_ERR_INVALID, "request %d: q_len %d, kv_len %d (need 0 <= q_len <= kv_len)", b,
                  q_lens[b], kv_lens[b]);
    qsum += q_lens[b];
    ksum += kv_lens[b];
    tiles += (q_lens[b] + q_tile_rows - 1) / q_tile_rows;
  }
  if (qsum >= (int64_t(1) << 31) || ksum >= (int64_t(1) << 31))
    return fail(ASTR_ERR_INVALID, "the int32 indptrs cannot hold %lld q rows / %lld keys",
                (long long)qsum, (long long)ksum);
  *num_tiles = (int32_t)tiles;
  if (tiles > max_tiles)
    return fail(ASTR_ERR_INVALID, "%lld tiles do not fit max_tiles %d", (long long)tiles, max_tiles);
  if (tiles > 0 && (!q_tile_to_batch || !q_tile_to_index)) return fail(ASTR_ERR_INVALID, "NULL tile maps");
  qo_indptr[0] = kv_indptr[0] = 0;
  std::vector<int32_t> tb, ti;
  std::vector<int64_t> cost;
  tb.reserve(tiles), ti.reserve(tiles), cost.reserve(tiles);
  for (int32_t b = 0; b < batch; ++b) {
    qo_indptr[b + 1] = qo_indptr[b] + q_lens[b];
    kv_indptr[b + 1] = kv_indptr[b] + kv_lens[b];
    const int64_t prefix = (int64_t)kv_lens[b] - q_lens[b];
    for (int32_t t = 0; t * (int64_t)q_tile_rows < q_lens[b]; ++t) {
      const int64_t last_row = std::min<int64_t>(q_lens[b], (int64_t)(t + 1) * q_tile_rows);
      tb.push_back(b);
      ti.push_back(t);
      cost.push_back((prefix + last_row + 127) / 128);  // 128-key tiles the Q tile visits
    }
  }
  std::vector<int32_t> order(tb.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int32_t)i;
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return cost[x] < cost[y]; });
  for (size_t i = 0; i < order.size(); ++i) {
    q_tile_to_batch[i] = tb[order[i]];
    q_tile_to_index[i] = ti[order[i]];
  }
  return ok();
}

astr_status astr_bind_tasks(const int32_t *q_lens, const int32_t *kv_lens, int32_t batch,
                            int32_t q_tile_rows, int32_t *qo_indptr, int32_t *kv_indptr,
                            int32_t *q_tile_to_batch, int32_t *q_tile_to_index, int32_t max_tiles,
                            astr_stream stream) {
  if (!kv_indptr || (batch > 0 && !kv_lens) || (q_lens && !qo_indptr))
    return fail(ASTR_ERR_INVALID, "NULL argument");
  if (max_tiles > 0 && (!q_tile_to_batch || !q_tile_to_index)) return fail(ASTR_ERR_INVALID, "NULL tile maps");
  if (batch < 0 || q_tile_rows < 1 || max_tiles < 0)
    return fail(ASTR_ERR_INVALID, "batch %d, q_tile_rows %d, max_tiles %d", batch, q_tile_rows, max_tiles);
  if (batch > bind_tasks_max_batch())
    return fail(ASTR_ERR_UNSUPPORTED, "batch %d above the %d requests the device planner holds", batch,
                bind_tasks_max_batch());
  uint32_t *err = error_word();
  if (!err) return fail(ASTR_ERR_CUDA, "no CUDA device / error word unavailable");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_bind_tasks(q_lens, kv_lens, batch, q_tile_rows, qo_indptr, kv_indptr,
                                    q_tile_to_batch, q_tile_to_index, max_tiles, num_sms(), err, s);
  if (e != cudaSuccess) return cuda_fail(e, "bind_tasks launch");
  return finish(s);
}

astr_status astr_decode_attention(const astr_kv_cache *kv, int32_t layer_id, const void *q,
                                  int32_t n_heads, astr_stream stream) {
  return decode_impl(kv, layer_id, q, n_heads, stream, nullptr);
}

astr_status astr_decode_attention_rope(const astr_kv_cache *kv, int32_t layer_id, const void *q,
                                       const void *k_new, const void *v_new, int32_t n_heads,
                                       const float *freqs_cis, int32_t freqs_max_len,
                                       const int32_t *position_ids, astr_stream stream) {
  astr_status st = check_cache(kv, layer_id, n_heads);
  if (st != ASTR_OK) return st;
  if (!use_tc_decode(kv, n_heads))
    return fail(ASTR_ERR_UNSUPPORTED,
                "decode with RoPE folded in serves bf16, head_dim 128 and group sizes 1/2/4/8/16; "
                "use astr_rope_kv_write + astr_decode_attention");
  if (kv->batch > 0) {
    if (!k_new || !v_new || !freqs_cis || !position_ids || !kv->out_cache_loc)
      return fail(ASTR_ERR_INVALID, "k_new, v_new, freqs_cis, position_ids and out_cache_loc must be non-NULL");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(freqs_cis))
      return fail(ASTR_ERR_INVALID, "k_new, v_new and freqs_cis must be 16-byte aligned");
    if (freqs_max_len < 1) return fail(ASTR_ERR_INVALID, "freqs_max_len %d < 1", freqs_max_len);
  }
  DecodeRope r;
  r.k_new = k_new;
  r.v_new = v_new;
  r.freqs = freqs_cis;
  r.freqs_max_len = freqs_max_len;
  r.position_ids = position_ids;
  return decode_impl(kv, layer_id, q, n_heads, stream, &r);
}

}  // extern "C"

namespace astr {
namespace {
astr_status decode_impl(const astr_kv_cache *kv, int32_t layer_id, const void *q, int32_t n_heads,
                        astr_stream stream, const DecodeRope *rope) {
  astr_status st = check_cache(kv, layer_id, n_heads);
  if (st != ASTR_OK) return st;
  if (kv->batch < 0) return fail(ASTR_ERR_INVALID, "batch %d < 0", kv->batch);
  if (kv->batch == 0) return ok();
  if ((st = check_table(kv)) != ASTR_OK) return st;
  if (!q || !kv->seq_lens || !kv->decode_out)
    return fail(ASTR_ERR_INVALID, "q, seq_lens and decode_out must be non-NULL");
  if (!aligned16(q)) return fail(ASTR_ERR_INVALID, "q must be 16-byte aligned");
  const int G = n_heads / kv->n_kv_heads;
  if (!simt_attn_supported(kv->dtype, kv->head_dim, G) && !use_tc_decode(kv, n_heads))
    return fail(ASTR_ERR_UNSUPPORTED, "decode: group size %d (n_heads / n_kv_heads) not served", G);
  if (kv->max_len < 1 || kv->max_len > kv->max_ctx_len)
    return fail(ASTR_ERR_INVALID, "max_len %d outside [1, max_ctx_len %d]", kv->max_len, kv->max_ctx_len);
  if (kv->split_chunk < 0) return fail(ASTR_ERR_INVALID, "split_chunk %d < 0", kv->split_chunk);
  SimtAttnPlan plan;
  plan.mode = 0;
  plan.chunk = decode_chunk(kv, n_heads);
  plan.n_splits = (kv->max_len + plan.chunk - 1) / plan.chunk;
  plan.wait_ns = (uint64_t)g_wait_ns.load();
  if (plan.n_splits > 1) {
    if (!kv->decode_o_part || !kv->decode_ml_part)
      return fail(ASTR_ERR_INVALID, "decode_o_part / decode_ml_part are NULL but %d splits are needed",
                  plan.n_splits);
    if (plan.n_splits > kv->max_splits)
      return fail(ASTR_ERR_INVALID, "max_len %d / split_chunk %d needs %d splits > max_splits %d",
                  kv->max_len, plan.chunk, plan.n_splits, kv->max_splits);
  }
  plan.err = error_word();
  if (!plan.err) return fail(ASTR_ERR_CUDA, "no CUDA device / error word unavailable");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (g_checked.load() && (e = launch_validate(*kv, VALIDATE_DECODE, plan.err, s)) != cudaSuccess)
    return cuda_fail(e, "checked-mode validation launch");
  if (use_tc_decode(kv, n_heads))
    e = launch_tc_decode(*kv, layer_id, q, n_heads, plan, s, rope);
  else
    e = launch_simt_attention(*kv, layer_id, q, kv->decode_out, n_heads, plan, s);
  if (e != cudaSuccess) return cuda_fail(e, "astr_decode_attention launch");
  return finish(s);
}
}  // namespace
}  // namespace astr

extern "C" {

astr_status astr_prefill_attention(const astr_kv_cache *kv, int32_t layer_id, const void *q,
                                   void *out, int32_t n_heads, astr_stream stream) {
  astr_status st = check_cache(kv, layer_id, n_heads);
  if (st != ASTR_OK) return st;
  if (kv->batch < 0 || kv->num_q_tiles < 0) return fail(ASTR_ERR_INVALID, "negative batch / num_q_tiles");
  if (kv->batch == 0 || kv->num_q_tiles == 0) return ok();
  if ((st = check_table(kv)) != ASTR_OK) return st;
  if (!q || !out || !kv->qo_indptr || !kv->kv_indptr || !kv->q_tile_to_batch || !kv->q_tile_to_index)
    return fail(ASTR_ERR_INVALID, "q, out, qo_indptr, kv_indptr and the q-tile maps must be non-NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(ASTR_ERR_INVALID, "q and out must be 16-byte aligned");
  if (kv->q_tile_rows != 128) return fail(ASTR_ERR_UNSUPPORTED, "q_tile_rows %d is not 128", kv->q_tile_rows);
  const int G = n_heads / kv->n_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t *err = error_word();
  if (!err) return fail(ASTR_ERR_CUDA, "no CUDA device / error word unavailable");
  cudaError_t e;
  if (g_checked.load() && (e = launch_validate(*kv, VALIDATE_PREFILL, err, s)) != cudaSuccess)
    return cuda_fail(e, "checked-mode validation launch");
  const uint64_t wait_ns = (uint64_t)g_wait_ns.load();
  if (kv->dtype == ASTR_BF16 && tc_prefill_supported(kv->dtype, kv->head_dim, G, kv->q_tile_rows)) {
    if (!tc_prefill_fits(*kv))
      return fail(ASTR_ERR_INVALID, "bf16 prefill needs n_tokens = the number of packed q rows (got %lld) "
                  "and n_layers * size < 2^31", (long long)kv->n_tokens);
    e = launch_tc_prefill(*kv, layer_id, q, out, n_heads, wait_ns, err, s);
  } else {
    if (!simt_attn_supported(kv->dtype, kv->head_dim, G))
      return fail(ASTR_ERR_UNSUPPORTED, "prefill: group size %d not in {1,2,4,8}", G);
    SimtAttnPlan plan;
    plan.mode = 1;
    plan.chunk = 0;
    plan.n_splits = 1;
    plan.wait_ns = wait_ns;
    plan.err = err;
    e = launch_simt_attention(*kv, layer_id, q, out, n_heads, plan, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "astr_prefill_attention launch");
  return finish(s);
}

}  // extern "C"
