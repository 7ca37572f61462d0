/*
 * astr.h -- C ABI of libastr.so, the GB300 (sm_103a) paged KV-cache attention path.
 *
 * The path: RoPE applied to Q/K from a precomputed f32 [cos, sin] table and written into the
 * KV cache at out_cache_loc (rotation before the write), then GQA softmax(q.k/sqrt(d)).v over
 * a paged k_buffer / v_buffer, for decode (split-K partials merged by log-sum-exp) and for
 * varlen causal prefill (including prefill resumed after a cached prefix).
 *
 * Sources: the AstrAI documentation -- internals page ("Autoregression & Causal Masking",
 * "Rotary Position Embedding (RoPE)", "KV Cache Mathematics", "Cache Architecture",
 * "Attention Backend") and inference guide ("KV Cache", "KVCache System", "Attention
 * Backend", "Rotary Embedding Backend").
 *
 * Conventions shared by every entry point:
 *  - Every pointer inside astr_kv_cache and every tensor argument is a DEVICE pointer owned by
 *    the caller. The library allocates nothing and frees nothing; it writes only the outputs
 *    named at each call (and, for decode, the caller's split-K scratch).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t / CUstream handle; NULL is
 *    the legacy default stream). No call synchronises the host unless checked mode is on.
 *  - CUDA graphs: with checked mode off, every enqueuing call can be stream-captured. Make one
 *    eager call of each entry point on a device before capturing it there (first calls look up
 *    device symbols and raise kernel attributes). A captured call keeps the plan it derived
 *    from its host arguments (batch, max_len, n_tokens, num_q_tiles, split_chunk, the pointers)
 *    and, for the persistent decode, its work counter; between replays the caller may change
 *    the contents of the device arrays within those bounds (e.g. seq_lens up to max_len).
 *  - Layouts are row-major and packed: q/k/v rows are [token, head, head_dim] (the pages'
 *    blhd layout with batch and sequence flattened), the cache is
 *    [n_layers, size, n_kv_heads, head_dim], index arrays are int32.
 *  - Element types: ASTR_F32 or ASTR_BF16 for q, k, v, the cache and the outputs; freqs_cis
 *    is always f32. head_dim is 64 or 128. n_heads must be a multiple of n_kv_heads (GQA:
 *    query head h reads KV head h / (n_heads / n_kv_heads)).
 *  - The softmax scale is always 1/sqrt(head_dim) (internals page, "Attention Backend").
 *  - Errors: arguments are validated on the host before any launch; a failure returns
 *    ASTR_ERR_INVALID / ASTR_ERR_UNSUPPORTED, enqueues nothing and sets astr_last_error().
 *    Kernels bounds-check every gathered slot, position and page-table row; an out-of-range
 *    index skips that access and raises a bit in a per-device error word instead of faulting.
 *    Every wait inside a kernel is bounded in time; a wait that runs out raises
 *    ASTR_DEVERR_TIMEOUT. astr_device_error() reads and clears the word. Nothing ever falls
 *    back to another implementation.
 */
#ifndef ASTR_H_
#define ASTR_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *astr_stream; /* cudaStream_t */

typedef enum { ASTR_F32 = 0, ASTR_BF16 = 1 } astr_dtype;

typedef enum {
  ASTR_OK = 0,
  ASTR_ERR_INVALID = 1,     /* bad argument: null pointer, inconsistent sizes */
  ASTR_ERR_UNSUPPORTED = 2, /* valid but not implemented: head_dim, dtype, group size */
  ASTR_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  ASTR_ERR_INDEX = 4,       /* checked mode: a kernel met an out-of-range index */
  ASTR_ERR_TIMEOUT = 5,     /* checked mode: a kernel wait ran out of time */
  ASTR_ERR_NO_SPACE = 6     /* page pool: not enough free or evictable pages */
} astr_status;

/* bits of the per-device error word */
#define ASTR_DEVERR_SLOT 0x1u     /* a slot outside [0, size) */
#define ASTR_DEVERR_POS 0x2u      /* a position outside [0, freqs_max_len) */
#define ASTR_DEVERR_ROW 0x4u      /* a req_pool_indices entry outside [0, num_reqs) */
#define ASTR_DEVERR_LEN 0x8u      /* a length < 1 or beyond max_ctx_len / max_len (bind_tasks:
                                     a q_len < 0, kv_len < q_len or a sum beyond int32) */
#define ASTR_DEVERR_TIMEOUT 0x10u /* a bounded wait ran out */
#define ASTR_DEVERR_META 0x20u    /* checked mode: indptr / tile map inconsistent;
                                     bind_tasks: the tiles do not fit max_tiles */

/*
 * The pages' KVCache dataclass (inference guide, "KVCache System": a plain data record
 * without methods), as plain device pointers and host sizes. Fields a call does not use may be
 * NULL / 0.
 */
typedef struct astr_kv_cache {
  /* KVStorage: flat token-level buffers [n_layers, size, n_kv_heads, head_dim] of `dtype` */
  void *k_buffer;
  void *v_buffer;
  int32_t n_layers;
  int32_t n_kv_heads;
  int64_t size;
  int32_t head_dim;
  int32_t dtype; /* astr_dtype */
  /* ReqToTokenPool: [num_reqs, max_ctx_len] -> physical slot, shared across layers */
  const int32_t *req_to_token;
  int32_t num_reqs;
  int32_t max_ctx_len;
  /* the batch of this forward */
  const int32_t *req_pool_indices; /* [batch] row of req_to_token per request */
  const int32_t *seq_lens;         /* [batch] decode: cached positions incl. the new token */
  int32_t batch;
  int32_t max_len;                 /* host int: max(seq_lens) (decode grid sizing, no sync) */
  const int32_t *out_cache_loc;    /* [n_tokens] write slots of this forward */
  int64_t n_tokens;                /* new tokens of this forward (prefill: packed q rows) */
  const int32_t *kv_indptr;        /* [batch+1] prefix sum of kv lengths */
  const int32_t *qo_indptr;        /* [batch+1] prefix sum of q lengths (prefill) */
  const int32_t *q_tile_to_batch;  /* [num_q_tiles] prefill: tile -> request */
  const int32_t *q_tile_to_index;  /* [num_q_tiles] prefill: tile -> request-local tile index */
  int32_t num_q_tiles;
  int32_t q_tile_rows;             /* rows per Q tile; 128 */
  /* decode split-K scratch (caller-owned, f32): see astr_decode_attention */
  float *decode_o_part;            /* [batch, n_heads, max_splits, head_dim] */
  float *decode_ml_part;           /* [batch, n_heads, max_splits, 2] = (m, l) */
  int32_t max_splits;
  int32_t split_chunk;             /* tokens per split; 0 = chosen by the library */
  void *decode_out;                /* [batch, n_heads, head_dim] of `dtype` */
} astr_kv_cache;

/*
 * Fused RoPE + KV cache write (internals page, "Rotary Position Embedding (RoPE)" and "KV
 * Cache Mathematics": RoPE is applied before the cache write; inference guide, "KVCache
 * System": k_buffer[layer_id, out_cache_loc] = k; "Rotary Embedding Backend": freqs_cis
 * [max_len, dim/2, 2] f32, view_as_complex pairing of adjacent elements).
 *
 * For every token t < kv->n_tokens with p = position_ids[t], s = kv->out_cache_loc[t] and
 * (c_i, s_i) = freqs_cis[p, i]:
 *   q_out[t, h, 2i], q_out[t, h, 2i+1] = rotation of (q[t,h,2i], q[t,h,2i+1]) by (c_i, s_i)
 *   k_buffer[layer_id, s, g, :]         = the same rotation of k[t, g, :]
 *   v_buffer[layer_id, s, g, :]         = v[t, g, :]
 * The rotation is a' = RN(RN(a c) - RN(b s)), b' = RN(RN(a s) + RN(b c)) in f32 with no fused
 * multiply-add, then rounded to the element type (bf16: nearest, ties to even), so results
 * are bit-reproducible. q: [n_tokens, n_heads, head_dim]; q_out may equal q (in place);
 * k, v: [n_tokens, n_kv_heads, head_dim]. Slots in out_cache_loc must be distinct (the
 * allocator hands out unique slots); duplicates give an unspecified one of the rows. A token
 * whose position or slot is out of range is skipped (ASTR_DEVERR_POS / _SLOT).
 */
astr_status astr_rope_kv_write(const astr_kv_cache *kv, int32_t layer_id, const void *q,
                               void *q_out, const void *k, const void *v, int32_t n_heads,
                               const float *freqs_cis, int32_t freqs_max_len,
                               const int32_t *position_ids, astr_stream stream);

/*
 * Paged GQA decode attention (internals page, "KV Cache Mathematics":
 * o_n = sum_j softmax(q_n k_j / sqrt(d_k)) v_j; inference guide, "Attention Backend": the
 * req_to_token table serves as the page table; "KVCache System": decode_o_part /
 * decode_ml_part split-K partials merged into decode_out).
 *
 * For request b < kv->batch with L = seq_lens[b] (1 <= L <= max_len <= max_ctx_len) and row
 * r = req_pool_indices[b]:
 *   decode_out[b, h, :] = sum_{j<L} softmax_j(q[b,h,:] . K_j / sqrt(d)) V_j,
 *   K_j = k_buffer[layer_id, req_to_token[r, j], h / G, :] (V likewise).
 * The query is the request's newest token (position L-1), whose K/V must already be written.
 * q: [batch, n_heads, head_dim]. The positions of each request are cut into chunks of C
 * tokens (C = split_chunk, or chosen by the library when 0; astr_decode_plan reports it).
 * A request with more than one chunk writes, per chunk s, the normalised partial output to
 * decode_o_part[b, h, s, :] and (m_s, l_s) to decode_ml_part[b, h, s, :] -- m_s a reference
 * score (q.k/sqrt(d) units, natural exponent) and l_s = sum_j exp(score_j - m_s) over the
 * chunk -- and a second kernel merges them by log-sum-exp. Requires
 * ceil(max_len / C) <= max_splits; the scratch may be NULL only when every request fits in
 * one chunk (C >= max_len). kv_indptr is not read (checked mode verifies it equals the prefix
 * sum of seq_lens).
 * With split_chunk 0 the library may also leave every request in one chunk (C = max_len,
 * nothing merged) when the batch alone balances the GPU.
 * The bf16 head_dim-128 kernel is persistent: one block per SM takes (request, chunk, KV
 * head) items from a work counter in device memory that belongs to the library, chunk by
 * chunk and, for batches up to 1024, each chunk's requests longest first (the order moves work
 * between SMs and changes no result). Each call uses the next of 32 such counters on the
 * current device (its last block resets it), so calls overlapping on different streams stay
 * independent unless 32 of them run at once.
 */
astr_status astr_decode_attention(const astr_kv_cache *kv, int32_t layer_id, const void *q,
                                  int32_t n_heads, astr_stream stream);

/*
 * RoPE on the training path, with no cache write (internals page, "Rotary Position Embedding
 * (RoPE)": training applies the rotation as a complex multiply that autograd differentiates;
 * inference guide, "Rotary Embedding Backend": the torch complex path serves training).
 *
 * astr_rope_apply, for every token t < n_tokens with p = position_ids[t], (c_i, s_i) =
 * freqs_cis[p, i] and every pair i:
 *   q_out[t, h, 2i..2i+1] = rotation of q[t, h, 2i..2i+1] by (c_i, s_i)      (h < n_heads)
 *   k_out[t, g, 2i..2i+1] = the same rotation of k[t, g, 2i..2i+1]            (g < n_kv_heads)
 * in the arithmetic of astr_rope_kv_write, whose q_out it reproduces bit for bit.
 * astr_rope_backward applies the transposed rotation R^T (the complex multiply by the conjugate
 * c_i - i s_i, i.e. by -theta) to grad_q_out and grad_k_out, giving grad_q and grad_k: the
 * rotation is linear, so this is its exact backward pass. Its arithmetic is the forward's with
 * s_i negated: a' = RN(RN(a c) + RN(b s)), b' = RN(RN(b c) - RN(a s)).
 *
 * All tensors are DEVICE memory owned by the caller, row-major [n_tokens, heads, head_dim] of
 * `dtype` (ASTR_F32 or ASTR_BF16), 16-byte aligned; an output may equal its input (in place).
 * head_dim is 64 or 128 (otherwise ASTR_ERR_UNSUPPORTED). n_kv_heads may be 0 (k and k_out
 * unused, may be NULL), as may n_heads. freqs_cis is f32 [freqs_max_len, head_dim/2, 2]. A
 * token whose position is outside [0, freqs_max_len) is skipped and raises ASTR_DEVERR_POS.
 */
astr_status astr_rope_apply(const void *q, void *q_out, const void *k, void *k_out,
                            int64_t n_tokens, int32_t n_heads, int32_t n_kv_heads,
                            int32_t head_dim, int32_t dtype, const float *freqs_cis,
                            int32_t freqs_max_len, const int32_t *position_ids,
                            astr_stream stream);
astr_status astr_rope_backward(const void *grad_q_out, void *grad_q, const void *grad_k_out,
                               void *grad_k, int64_t n_tokens, int32_t n_heads,
                               int32_t n_kv_heads, int32_t head_dim, int32_t dtype,
                               const float *freqs_cis, int32_t freqs_max_len,
                               const int32_t *position_ids, astr_stream stream);

/*
 * Decode that allocates nothing. The pages have no counterpart: it exists for callers that
 * cannot call cudaMalloc to provide split-K scratch -- plugin hosts that hand a library only
 * the tensors of one call, embedded runtimes that reserve all device memory at start-up and
 * forbid later allocations, serving loops that must never block on the allocator.
 * Computes exactly what astr_decode_attention computes and writes kv->decode_out, but keeps
 * the split-K partials in an 8 MiB array compiled into this library (one per GPU that loads
 * it, held until the process exits); kv->decode_o_part, decode_ml_part and max_splits are
 * ignored. The number of splits is limited to what fits, 8 MiB / (batch * n_heads *
 * (head_dim + 2) * 4 bytes): with split_chunk = 0 the library picks a chunk that fits, an
 * explicit split_chunk needing more splits is rejected with ASTR_ERR_INVALID. The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress); make that first
 * call before any stream capture. Every call shares the array and it keeps the last call's
 * contents; no entry has to start at zero because each call writes every entry it reads.
 * Calls whose work overlaps on the GPU (several streams) race on the array. The looked-up
 * address is kept for the life of the process: after a device reset (cudaDeviceReset, or a
 * reset of the primary context) it is stale, so do not call this entry point again after one.
 */
astr_status astr_decode_attention_noalloc(const astr_kv_cache *kv, int32_t layer_id,
                                          const void *q, int32_t n_heads, astr_stream stream);

/*
 * Decode with RoPE and the new token's cache write folded in, in one launch (plus the split-K
 * merge): the decode path of the inference guide's "Attention Backend" writes the new token's
 * K/V while calling the paged decode op; "Rotary Position Embedding (RoPE)" (internals page)
 * rotates q and k before the cache write.
 *
 * For request b: q[b] ([batch, n_heads, head_dim], not rotated yet) is rotated by the
 * (cos, sin) row freqs_cis[position_ids[b]]; k_new[b] ([batch, n_kv_heads, head_dim]) is
 * rotated the same way and written, with v_new[b] unchanged, into slot kv->out_cache_loc[b]
 * of layer `layer_id`; then decode_out[b] is computed exactly as astr_decode_attention does,
 * with the rotated query. Rounding is that of astr_rope_kv_write, so the cache bytes are the
 * same as a rotate + write call would leave. out_cache_loc[b] must be the slot of the
 * request's newest position, req_to_token[req_pool_indices[b], seq_lens[b] - 1]. q is read
 * only (the rotated query is not written back). A position or slot out of range raises
 * ASTR_DEVERR_POS / _SLOT in the error word and that token is neither rotated nor written.
 * Serves bf16 with head_dim 128 (the tensor-core decode) and returns ASTR_ERR_UNSUPPORTED
 * otherwise. The pages name no such single call: their RoPE runs as a separate step.
 */
astr_status astr_decode_attention_rope(const astr_kv_cache *kv, int32_t layer_id, const void *q,
                                       const void *k_new, const void *v_new, int32_t n_heads,
                                       const float *freqs_cis, int32_t freqs_max_len,
                                       const int32_t *position_ids, astr_stream stream);

/*
 * The per-step metadata of a prefill batch, on the HOST (inference guide, "KVCache System":
 * qo_indptr, kv_indptr and the q_tile_to_batch / q_tile_to_index maps, computed once per step
 * and shared by every layer; internals page, "Attention Backend").
 *
 * From q_lens[b] (new rows) and kv_lens[b] (keys, cached prefix included; q_len <= kv_len)
 * for b < batch, writes qo_indptr[0..batch] and kv_indptr[0..batch] (prefix sums) and one
 * entry per q_tile_rows-row Q tile to q_tile_to_batch / q_tile_to_index, listed by the number
 * of 128-key tiles the Q tile visits under the causal mask, cheapest first (ties in request
 * order): the order in which the bf16 prefill balances best (it starts from the end of the
 * list). *num_tiles receives the tile count. All pointers are host memory owned by the
 * caller; the indptrs (batch + 1 entries each) are required even for batch 0, q_lens and
 * kv_lens may be NULL only when batch is 0, and the maps (room for max_tiles entries) only
 * when there are no tiles. Returns ASTR_ERR_INVALID for bad lengths
 * or too small a max_tiles (*num_tiles still holds the count needed). Enqueues nothing.
 */
astr_status astr_prefill_tiles(const int32_t *q_lens, const int32_t *kv_lens, int32_t batch,
                               int32_t q_tile_rows, int32_t *qo_indptr, int32_t *kv_indptr,
                               int32_t *q_tile_to_batch, int32_t *q_tile_to_index,
                               int32_t max_tiles, int32_t *num_tiles);

/*
 * The same per-step metadata computed on the DEVICE, enqueued on `stream` (inference guide,
 * "KVCache System": bind_tasks() builds the KVCache of a step, its kv_indptr, qo_indptr and
 * Q-tile maps computed once per step and shared by every layer). For steps captured in a
 * CUDA graph whose lengths change between replays: the host writes only q_lens / kv_lens.
 *
 * q_lens, kv_lens: device int32 [batch]; q_lens may be NULL (a decode batch: only kv_indptr,
 * the prefix sum of kv_lens = seq_lens, is written, and qo_indptr may be NULL too). Writes
 * qo_indptr and kv_indptr [batch + 1] and all max_tiles entries of q_tile_to_batch /
 * q_tile_to_index: the n real tiles in astr_prefill_tiles' order at entries max_tiles - n ..
 * max_tiles - 1, and -1 in both maps at entries 0 .. max_tiles - n - 1. astr_prefill_attention
 * skips -1 entries, so it runs on these maps with num_q_tiles = max_tiles, a capacity fixed at
 * capture. All pointers are device memory owned by the caller. Host-side argument errors
 * return ASTR_ERR_INVALID (batch above 16383: ASTR_ERR_UNSUPPORTED, the requests held in
 * shared memory). Device-side: a q_len < 0 or a kv_len < q_len raises ASTR_DEVERR_LEN, more than
 * max_tiles tiles raises ASTR_DEVERR_META; in both cases every map entry becomes -1 (the
 * prefill then writes nothing). One launch; each tile's position costs O(batch).
 */
astr_status astr_bind_tasks(const int32_t *q_lens, const int32_t *kv_lens, int32_t batch,
                            int32_t q_tile_rows, int32_t *qo_indptr, int32_t *kv_indptr,
                            int32_t *q_tile_to_batch, int32_t *q_tile_to_index, int32_t max_tiles,
                            astr_stream stream);

/*
 * The split plan astr_decode_attention would use for `kv`: chunk length and the number of
 * splits ceil(max_len / chunk). Host-only; enqueues nothing.
 */
astr_status astr_decode_plan(const astr_kv_cache *kv, int32_t n_heads, int32_t *split_chunk,
                             int32_t *n_splits);

/*
 * Varlen causal prefill over the paged pool (inference guide, "Attention Backend": a
 * ragged-batch prefill that reads K/V straight from the flat pool through req_to_token,
 * addressing each request through qo_indptr and kv_indptr; "KVCache System": q_tile_to_batch
 * / q_tile_to_index, and prefill resumed right after a cached prefix; internals page,
 * "Autoregression & Causal Masking").
 *
 * Request b owns packed rows qo_indptr[b] .. qo_indptr[b+1]-1 of q and out
 * ([sum q, n_heads, head_dim]) and keys 0..K_b-1, K_b = kv_indptr[b+1] - kv_indptr[b] >= Q_b.
 * Row i of request b sits at absolute position P_b + i, P_b = K_b - Q_b (the cached prefix),
 * and attends keys j <= P_b + i:
 *   out[t, h, :] = sum_{j <= P_b+i} softmax_j(q[t,h,:] . K_j / sqrt(d)) V_j.
 * The new tokens' K/V (positions P_b..K_b-1) must already be in the cache; kv->n_tokens is
 * the number of rows q and out hold: qo_indptr[batch], or more (a CUDA graph passes its
 * capacity; rows past qo_indptr[batch] are never written, though a partial last tile may load
 * and discard some of them). n_layers * size must stay below 2^31 for the bf16 path, whose row
 * coordinates are 32-bit. Tile t covers request q_tile_to_batch[t], rows
 * [q_tile_rows * q_tile_to_index[t], +q_tile_rows) clipped to Q_b; together the tiles must
 * cover every row exactly once. An entry with q_tile_to_batch[t] == -1 is empty and skipped
 * (astr_bind_tasks pads with these); any other out-of-range entry raises ASTR_DEVERR_META.
 * Rows are written only by their tile. bf16 runs on the tcgen05 tensor cores (bf16 operands,
 * f32 accumulation); f32 runs on the CUDA cores in f32 (no TF32).
 * Tile order changes no result. The bf16 kernel starts its blocks from the END of the tile
 * list, so listing tiles in request order runs each request's longest (last) tiles first, and
 * listing them by the number of 128-key tiles they visit, cheapest first, schedules the
 * costliest first across the whole batch.
 */
astr_status astr_prefill_attention(const astr_kv_cache *kv, int32_t layer_id, const void *q,
                                   void *out, int32_t n_heads, astr_stream stream);

/*
 * Paged-pool bookkeeping on the HOST (inference guide, "KVCache System": PagePool over a
 * bitmask page allocator with ref-counts and LRU eviction, and RadixCache, exact page-aligned
 * prefix matching; internals page, "Cache Architecture"). Enqueues no GPU work; every call
 * takes the pool's mutex.
 *
 * Page p owns the token slots [p * page_size, (p + 1) * page_size) of the flat KV buffers, so a
 * request whose pages are pg[0..] has slot pg[j / page_size] * page_size + j % page_size at
 * position j of its req_to_token row. A page is free, referenced (held by requests: ref > 0) or
 * cached without a reference. The radix cache holds complete pages only, as edges from a parent
 * prefix labelled by the page's exact token tuple: a page is shared only under the same parent
 * prefix, and the hash each entry keeps (astr_pool_page_info) never decides a match. With
 * page_size 1 there is no prefix sharing: match finds nothing and record keeps nothing.
 *
 * astr_pool_match: the longest run of complete pages of tokens[0..n_tokens) cached along one
 *   path from the root, at most max_pages; writes them to pages[0..*n_matched) and takes a
 *   reference on each (they cannot be evicted until released). A request resumes prefill after
 *   *n_matched * page_size tokens; to keep at least one row to compute, pass n_tokens = prompt
 *   length - 1.
 * astr_pool_alloc: n fresh pages (ref 1), the lowest free page numbers first. When too few are
 *   free, unreferenced cached leaves are evicted least recently used first (match and record
 *   count as uses), a parent becoming a leaf in turn. ASTR_ERR_NO_SPACE if that is not enough
 *   (pages evicted on the way stay evicted; nothing is allocated).
 * astr_pool_record: enter the complete pages of tokens[0..n_materialized) -- the tokens whose
 *   K/V are in the cache: on completion the prompt plus the generated tokens except the last
 *   sampled one -- with the request's pages[0..n_pages) (pages[i] holds tokens i * page_size..).
 *   Where the path already has an edge with the same tuple, the cached page is kept and the
 *   request's own copy stays private (freed when released). The partial last page is never
 *   entered. The caller must hold a reference on every page it passes; a page already cached on
 *   another path, or passed twice, is rejected (ASTR_ERR_INVALID, nothing changed).
 * astr_pool_release: drop one reference per entry of pages[0..n) (repeats drop several). A page
 *   left with no reference is freed if it is not cached, or becomes evictable once it is a
 *   cached leaf. Releasing a reference not held is ASTR_ERR_INVALID and changes nothing.
 * astr_pool_stats / astr_pool_page_info: counts (free, cached, evictable) and one page's
 *   reference count, whether it is cached and its entry's hash (0 when not cached).
 * astr_pool_slots: the req_to_token row entries of positions 0..n_tokens-1 for a request
 *   holding pages[0..n_pages): slots[j] = pages[j / page_size] * page_size + j % page_size.
 *   ASTR_ERR_INVALID (nothing written past the failing entry) when the pages cannot hold
 *   n_tokens or a page number is outside the pool. Reads no pool state beyond its size.
 */
typedef struct astr_page_pool astr_page_pool;
astr_status astr_pool_create(int32_t n_pages, int32_t page_size, astr_page_pool **pool);
astr_status astr_pool_destroy(astr_page_pool *pool);
astr_status astr_pool_match(astr_page_pool *pool, const int32_t *tokens, int64_t n_tokens,
                            int32_t max_pages, int32_t *pages, int32_t *n_matched);
astr_status astr_pool_alloc(astr_page_pool *pool, int32_t n, int32_t *pages);
astr_status astr_pool_record(astr_page_pool *pool, const int32_t *tokens, int64_t n_materialized,
                             const int32_t *pages, int32_t n_pages);
astr_status astr_pool_release(astr_page_pool *pool, const int32_t *pages, int32_t n);
astr_status astr_pool_stats(astr_page_pool *pool, int32_t *free_pages, int32_t *cached_pages,
                            int32_t *evictable_pages);
astr_status astr_pool_page_info(astr_page_pool *pool, int32_t page, int32_t *refs,
                                int32_t *cached, uint64_t *hash);
astr_status astr_pool_slots(astr_page_pool *pool, const int32_t *pages, int32_t n_pages,
                            int64_t n_tokens, int32_t *slots);

/* Message of the last failing call on this host thread ("" if none). */
const char *astr_last_error(void);

/*
 * Checked mode (process-wide, off by default): every entry point also validates the index
 * metadata on the device, synchronises `stream` after its kernels and returns ASTR_ERR_INDEX
 * or ASTR_ERR_TIMEOUT when the device error word is set (then clears it).
 */
astr_status astr_set_checked(int32_t on);

/*
 * Upper bound, in nanoseconds, on any single wait inside a kernel (default 1e9). A wait that
 * runs out abandons the rest of that block's work, raises ASTR_DEVERR_TIMEOUT and returns
 * after its in-flight copies land. Values below 1 are clamped to 1.
 */
astr_status astr_set_wait_timeout_ns(int64_t ns);

/*
 * Synchronise `stream`, then read and clear the current device's error word (ASTR_DEVERR_*
 * bits) into *flags.
 */
astr_status astr_device_error(astr_stream stream, uint32_t *flags);

/*
 * Self-test of the bounded-wait path: launches one block that waits on an mbarrier no thread
 * ever arrives at, with the wait limited to `ns` nanoseconds, then synchronises `stream`.
 * Returns ASTR_ERR_TIMEOUT (and clears the error word) when the wait ran out as it must; any
 * other status means the mechanism is broken. The GPU context stays usable afterwards.
 */
astr_status astr_selftest_wait_timeout(astr_stream stream, int64_t ns);

/* ABI version of this header (major * 100 + minor). */
int32_t astr_version(void);

/* sizeof(astr_kv_cache) as compiled into the library (lets bindings check their mirror). */
int32_t astr_kv_cache_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* ASTR_H_ */
