// Internal launchers behind the C ABI (host side). Each returns the launch's cudaError_t.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/astr.h"

namespace astr {

cudaError_t launch_rope_kv_write(const astr_kv_cache &kv, int32_t layer_id, const void *q,
                                 void *q_out, const void *k, const void *v, int32_t n_heads,
                                 const float *freqs, int32_t freqs_max_len,
                                 const int32_t *position_ids, cudaStream_t stream, int num_sms,
                                 uint32_t *err);

// RoPE with no cache write (training path): the rotation, or its transpose with `inverse`
cudaError_t launch_rope_apply(const void *q, void *q_out, const void *k, void *k_out,
                              int64_t n_tokens, int32_t n_heads, int32_t n_kv_heads,
                              int32_t head_dim, int32_t dtype, const float *freqs,
                              int32_t freqs_max_len, const int32_t *position_ids, bool inverse,
                              cudaStream_t stream, int num_sms, uint32_t *err);

// Chunked attention on the CUDA cores: decode (mode 0, one query per request, split into
// `chunk`-token pieces) or f32 prefill rows (mode 1, one query per packed row, unsplit).
struct SimtAttnPlan {
  int mode;        // 0 decode, 1 prefill rows
  int chunk;       // decode: tokens per split
  int n_splits;    // decode: ceil(max_len / chunk)
  uint64_t wait_ns;
  uint32_t *err;   // device error word
};

bool simt_attn_supported(int dtype, int head_dim, int group);
cudaError_t launch_simt_attention(const astr_kv_cache &kv, int32_t layer_id, const void *q,
                                  void *out, int32_t n_heads, const SimtAttnPlan &plan,
                                  cudaStream_t stream);
int simt_tile_tokens(int group);

// log-sum-exp merge of the decode split-K partials into decode_out
cudaError_t launch_split_merge(const astr_kv_cache &kv, int32_t n_heads, const SimtAttnPlan &plan,
                               cudaStream_t stream);

// tcgen05 bf16 decode (head_dim 128)
bool tc_decode_supported(int dtype, int head_dim, int group);
int tc_decode_tile_tokens();
int tc_decode_ranked_batch_max();  // batches up to this size claim their requests longest first
// RoPE and the new token's cache write folded into the decode (astr_decode_attention_rope)
struct DecodeRope {
  const void *k_new;
  const void *v_new;
  const float *freqs;
  int32_t freqs_max_len;
  const int32_t *position_ids;
};
cudaError_t launch_tc_decode(const astr_kv_cache &kv, int32_t layer_id, const void *q,
                             int32_t n_heads, const SimtAttnPlan &plan, cudaStream_t stream,
                             const DecodeRope *rope = nullptr);

// tcgen05 bf16 prefill.
bool tc_prefill_supported(int dtype, int head_dim, int group, int q_tile_rows);
bool tc_prefill_fits(const astr_kv_cache &kv);  // n_tokens set, row coordinates within int32
cudaError_t launch_tc_prefill(const astr_kv_cache &kv, int32_t layer_id, const void *q,
                              void *out, int32_t n_heads, uint64_t wait_ns, uint32_t *err,
                              cudaStream_t stream);

// the persistent, pipelined form of the bf16 prefill (query groups of an even size); it is
// launched when there are more (Q tile, head pair) items than SMs
bool tc_prefill_pipe_supported(int group);
cudaError_t launch_tc_prefill_pipe(const astr_kv_cache &kv, int32_t layer_id, const void *q, void *out,
                                   int32_t n_heads, uint64_t wait_ns, uint32_t *err, cudaStream_t stream);

// per-step metadata on the device (astr_bind_tasks); batch <= bind_tasks_max_batch()
int bind_tasks_max_batch();
cudaError_t launch_bind_tasks(const int32_t *q_lens, const int32_t *kv_lens, int32_t batch,
                              int32_t q_tile_rows, int32_t *qo_indptr, int32_t *kv_indptr,
                              int32_t *q_tile_to_batch, int32_t *q_tile_to_index,
                              int32_t max_tiles, int num_sms, uint32_t *err, cudaStream_t stream);

// a pair of work counters on the current device for one launch of a persistent kernel
// ([0]: claims, [1]: blocks done; the launch's last block zeroes both), and its SM count
cudaError_t sched_slot(unsigned **out, int *sms);
// the current device's SM count (looked up once per device)
cudaError_t device_sm_count(int *sms);

// sets the message astr_last_error() returns on this thread
void set_last_error_message(const char *msg);

// checked mode: device-side validation of the index metadata
cudaError_t launch_validate(const astr_kv_cache &kv, int what, uint32_t *err, cudaStream_t stream);
enum { VALIDATE_DECODE = 1, VALIDATE_PREFILL = 2 };

}  // namespace astr
