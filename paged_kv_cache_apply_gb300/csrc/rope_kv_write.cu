// Fused RoPE + KV cache write.
//
// AstrAI internals, "Rotary Position Embedding (RoPE)": freqs_cis [max_len, dim/2, 2] f32
// [cos, sin] pairs indexed by position_ids; RoPE is applied before the KV cache write.
// AstrAI inference guide, "KVCache System": k_buffer[layer_id, out_cache_loc] = k;
// "Rotary Embedding Backend": the complex product pairs adjacent elements (x[2i], x[2i+1]).
//
// One thread handles one 8-element chunk (4 rotation pairs) of one head row of one token:
// a 16-byte (bf16) or 32-byte (f32) load of the row chunk plus a 32-byte load of the four
// (cos, sin) pairs, the rotation in f32 with separately rounded products and sums, and one
// coalesced store -- to q_out for query heads, to the cache row out_cache_loc[t] for key
// heads (rotated) and value heads (copied). Every 1 KB cache row is written by contiguous
// threads, so the scatter stays fully coalesced.
#include "astr_internal.cuh"
#include "launch.h"

namespace astr {

namespace {

struct RopeArgs {
  const void *q;
  void *q_out;
  const void *k;
  const void *v;
  void *k_layer;  // k_buffer + layer_id * size * Hk * D
  void *v_layer;
  const float *freqs;
  const int32_t *pos;
  const int32_t *loc;
  int64_t n_tokens;
  int64_t size;
  int32_t freqs_max_len;
  int32_t H, Hk, D;
  uint32_t *err;
};

template <typename T>
struct Chunk;

template <>
struct Chunk<float> {
  struct Raw {
    float4 a, b;
  };
  static __device__ __forceinline__ Raw load_raw(const void *base, int64_t off) {
    const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + off);
    return Raw{__ldg(p), __ldg(p + 1)};
  }
  static __device__ __forceinline__ void unpack(const Raw &w, float (&x)[8]) {
    x[0] = w.a.x; x[1] = w.a.y; x[2] = w.a.z; x[3] = w.a.w;
    x[4] = w.b.x; x[5] = w.b.y; x[6] = w.b.z; x[7] = w.b.w;
  }
  static __device__ __forceinline__ void store_raw(void *base, int64_t off, const Raw &w) {
    float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(base) + off);
    p[0] = w.a;
    p[1] = w.b;
  }
  static __device__ __forceinline__ void load(const void *base, int64_t off, float (&x)[8]) {
    const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(base) + off);
    float4 a = __ldg(p), b = __ldg(p + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
  static __device__ __forceinline__ void store(void *base, int64_t off, const float (&y)[8]) {
    float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(base) + off);
    p[0] = make_float4(y[0], y[1], y[2], y[3]);
    p[1] = make_float4(y[4], y[5], y[6], y[7]);
  }
  static __device__ __forceinline__ void copy(const void *src, int64_t so, void *dst, int64_t dof) {
    const float4 *s = reinterpret_cast<const float4 *>(static_cast<const float *>(src) + so);
    float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(dst) + dof);
    d[0] = __ldg(s);
    d[1] = __ldg(s + 1);
  }
};

template <>
struct Chunk<bf16_t> {
  using Raw = uint4;
  static __device__ __forceinline__ Raw load_raw(const void *base, int64_t off) {
    return __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + off));
  }
  static __device__ __forceinline__ void unpack(const Raw &w, float (&x)[8]) {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  }
  static __device__ __forceinline__ void store_raw(void *base, int64_t off, const Raw &w) {
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + off) = w;
  }
  static __device__ __forceinline__ void load(const void *base, int64_t off, float (&x)[8]) {
    uint4 w = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + off));
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  }
  static __device__ __forceinline__ void store(void *base, int64_t off, const float (&y)[8]) {
    uint4 w;
    w.x = pack_bf16x2_rn(y[0], y[1]);
    w.y = pack_bf16x2_rn(y[2], y[3]);
    w.z = pack_bf16x2_rn(y[4], y[5]);
    w.w = pack_bf16x2_rn(y[6], y[7]);
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(base) + off) = w;
  }
  static __device__ __forceinline__ void copy(const void *src, int64_t so, void *dst, int64_t dof) {
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(dst) + dof) =
        __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src) + so));
  }
};

// Idx is the integer type of the chunk index: 32-bit whenever the launch's chunks fit, since a
// 64-bit division is emulated in many instructions and the kernel is otherwise a few loads
template <typename T, typename Idx>
__global__ void __launch_bounds__(256) rope_kv_write_kernel(const RopeArgs a) {
  const int chunk_shift = a.D == 128 ? 4 : 3;  // log2 of the 8-element chunks per row
  const int rows = a.H + 2 * a.Hk;
  const Idx per_token = (Idx)rows << chunk_shift;
  const Idx total = (Idx)a.n_tokens * per_token;
  for (Idx id = (Idx)blockIdx.x * blockDim.x + threadIdx.x; id < total;
       id += (Idx)gridDim.x * blockDim.x) {
    const Idx tq = id / per_token;
    const int c = (int)(id - tq * per_token);
    const int64_t t = (int64_t)tq;  // element offsets below can exceed 32 bits
    const int row = c >> chunk_shift;
    const int e0 = (c - (row << chunk_shift)) << 3;
    const int32_t p = __ldg(a.pos + t);
    const int32_t s = __ldg(a.loc + t);
    const bool pos_ok = p >= 0 && p < a.freqs_max_len;
    const bool slot_ok = s >= 0 && (int64_t)s < a.size;
    if (!(pos_ok && slot_ok)) {
      if (c == 0) raise_error(a.err, (pos_ok ? 0u : ASTR_DEVERR_POS) | (slot_ok ? 0u : ASTR_DEVERR_SLOT));
      continue;
    }
    if (row >= a.H + a.Hk) {  // value head: copied unchanged
      const int g = row - a.H - a.Hk;
      Chunk<T>::copy(a.v, (t * a.Hk + g) * a.D + e0, a.v_layer, ((int64_t)s * a.Hk + g) * a.D + e0);
      continue;
    }
    float cs[8];
    {
      const float4 *f =
          reinterpret_cast<const float4 *>(a.freqs + (int64_t)p * a.D + 2 * (e0 >> 1));
      float4 f0 = __ldg(f), f1 = __ldg(f + 1);
      cs[0] = f0.x; cs[1] = f0.y; cs[2] = f0.z; cs[3] = f0.w;
      cs[4] = f1.x; cs[5] = f1.y; cs[6] = f1.z; cs[7] = f1.w;
    }
    float x[8], y[8];
    if (row < a.H) {
      const int64_t off = (t * a.H + row) * a.D + e0;
      Chunk<T>::load(a.q, off, x);
      rotate4(x, cs, y);
      Chunk<T>::store(a.q_out, off, y);
    } else {
      const int g = row - a.H;
      Chunk<T>::load(a.k, (t * a.Hk + g) * a.D + e0, x);
      rotate4(x, cs, y);
      Chunk<T>::store(a.k_layer, ((int64_t)s * a.Hk + g) * a.D + e0, y);
    }
  }
}

// The same work with one block per token: the block's threads take the token's chunks (a
// stride loop when there are more chunks than threads), so the position and slot are read once
// per block and no chunk index is divided to find its token.
template <typename T>
__global__ void __launch_bounds__(512) rope_kv_write_token_kernel(const RopeArgs a) {
  const int64_t t = blockIdx.x;
  const int chunk_shift = a.D == 128 ? 4 : 3;
  const int per_token = (a.H + 2 * a.Hk) << chunk_shift;
  const int32_t p = __ldg(a.pos + t);
  const int32_t s = __ldg(a.loc + t);
  const bool pos_ok = p >= 0 && p < a.freqs_max_len;
  const bool slot_ok = s >= 0 && (int64_t)s < a.size;
  if (!(pos_ok && slot_ok)) {
    if (threadIdx.x == 0) raise_error(a.err, (pos_ok ? 0u : ASTR_DEVERR_POS) | (slot_ok ? 0u : ASTR_DEVERR_SLOT));
    return;
  }
  for (int c = threadIdx.x; c < per_token; c += blockDim.x) {
    const int row = c >> chunk_shift;
    const int e0 = (c - (row << chunk_shift)) << 3;
    if (row >= a.H + a.Hk) {  // value head: copied unchanged
      const int g = row - a.H - a.Hk;
      Chunk<T>::copy(a.v, (t * a.Hk + g) * a.D + e0, a.v_layer, ((int64_t)s * a.Hk + g) * a.D + e0);
      continue;
    }
    float cs[8];
    {
      const float4 *f =
          reinterpret_cast<const float4 *>(a.freqs + (int64_t)p * a.D + 2 * (e0 >> 1));
      float4 f0 = __ldg(f), f1 = __ldg(f + 1);
      cs[0] = f0.x; cs[1] = f0.y; cs[2] = f0.z; cs[3] = f0.w;
      cs[4] = f1.x; cs[5] = f1.y; cs[6] = f1.z; cs[7] = f1.w;
    }
    float x[8], y[8];
    if (row < a.H) {
      const int64_t off = (t * a.H + row) * a.D + e0;
      Chunk<T>::load(a.q, off, x);
      rotate4(x, cs, y);
      Chunk<T>::store(a.q_out, off, y);
    } else {
      const int g = row - a.H;
      Chunk<T>::load(a.k, (t * a.Hk + g) * a.D + e0, x);
      rotate4(x, cs, y);
      Chunk<T>::store(a.k_layer, ((int64_t)s * a.Hk + g) * a.D + e0, y);
    }
  }
}

// One block of kTokThreads threads per token; thread i takes the token's chunks i, i + kTokThreads,
// ... (NC of them). A thread issues all its row loads before it reads the position and the slot,
// so they are in flight together with those two loads; only the (cos, sin) loads wait for the
// position and only the stores for the slot. Small blocks let every token of a step be resident
// at once, which keeps enough bytes in flight on every SM.
constexpr int kTokThreads = 128;

template <typename T, int NC>
__global__ void __launch_bounds__(kTokThreads) rope_kv_write_token_nc_kernel(const RopeArgs a) {
  const int64_t t = blockIdx.x;
  const int chunk_shift = a.D == 128 ? 4 : 3;
  const int per_token = (a.H + 2 * a.Hk) << chunk_shift;
  const int32_t p = __ldg(a.pos + t);
  const int32_t s = __ldg(a.loc + t);
  typename Chunk<T>::Raw raw[NC];
#pragma unroll
  for (int k = 0; k < NC; ++k) {
    const int c = threadIdx.x + k * kTokThreads;
    if (c < per_token) {
      const int row = c >> chunk_shift;
      const int e0 = (c - (row << chunk_shift)) << 3;
      if (row < a.H)
        raw[k] = Chunk<T>::load_raw(a.q, (t * a.H + row) * a.D + e0);
      else if (row < a.H + a.Hk)
        raw[k] = Chunk<T>::load_raw(a.k, (t * a.Hk + (row - a.H)) * a.D + e0);
      else
        raw[k] = Chunk<T>::load_raw(a.v, (t * a.Hk + (row - a.H - a.Hk)) * a.D + e0);
    }
  }
  const bool pos_ok = p >= 0 && p < a.freqs_max_len;
  const bool slot_ok = s >= 0 && (int64_t)s < a.size;
  if (!(pos_ok && slot_ok)) {
    if (threadIdx.x == 0) raise_error(a.err, (pos_ok ? 0u : ASTR_DEVERR_POS) | (slot_ok ? 0u : ASTR_DEVERR_SLOT));
    return;
  }
#pragma unroll
  for (int k = 0; k < NC; ++k) {
    const int c = threadIdx.x + k * kTokThreads;
    if (c < per_token) {
      const int row = c >> chunk_shift;
      const int e0 = (c - (row << chunk_shift)) << 3;
      if (row >= a.H + a.Hk) {  // value head: copied unchanged
        Chunk<T>::store_raw(a.v_layer, ((int64_t)s * a.Hk + (row - a.H - a.Hk)) * a.D + e0, raw[k]);
        continue;
      }
      float cs[8];
      {
        const float4 *f = reinterpret_cast<const float4 *>(a.freqs + (int64_t)p * a.D + 2 * (e0 >> 1));
        float4 f0 = __ldg(f), f1 = __ldg(f + 1);
        cs[0] = f0.x; cs[1] = f0.y; cs[2] = f0.z; cs[3] = f0.w;
        cs[4] = f1.x; cs[5] = f1.y; cs[6] = f1.z; cs[7] = f1.w;
      }
      float x[8], y[8];
      Chunk<T>::unpack(raw[k], x);
      rotate4(x, cs, y);
      if (row < a.H)
        Chunk<T>::store(a.q_out, (t * a.H + row) * a.D + e0, y);
      else
        Chunk<T>::store(a.k_layer, ((int64_t)s * a.Hk + (row - a.H)) * a.D + e0, y);
    }
  }
}

template <typename T>
cudaError_t launch_token_nc(const RopeArgs &a, int nc, unsigned blocks, cudaStream_t stream) {
  switch (nc) {
    case 1: rope_kv_write_token_nc_kernel<T, 1><<<blocks, kTokThreads, 0, stream>>>(a); break;
    case 2: rope_kv_write_token_nc_kernel<T, 2><<<blocks, kTokThreads, 0, stream>>>(a); break;
    case 3: rope_kv_write_token_nc_kernel<T, 3><<<blocks, kTokThreads, 0, stream>>>(a); break;
    case 4: rope_kv_write_token_nc_kernel<T, 4><<<blocks, kTokThreads, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// RoPE with no cache write (the training path): q_out = R q and k_out = R k, or with Inverse
// the transposed rotation R^T (the complex multiply by the conjugate entry: s negated), which
// maps the gradients of the rotated tensors to those of their inputs. One thread per 8-element
// chunk as above; rows 0..H-1 of a token are query heads, H..H+Hk-1 key heads.
struct RopeApplyArgs {
  const void *q;
  void *q_out;
  const void *k;
  void *k_out;
  const float *freqs;
  const int32_t *pos;
  int64_t n_tokens;
  int32_t freqs_max_len;
  int32_t H, Hk, D;
  uint32_t *err;
};

template <typename T, typename Idx, bool Inverse>
__global__ void __launch_bounds__(256) rope_apply_kernel(const RopeApplyArgs a) {
  const int chunk_shift = a.D == 128 ? 4 : 3;
  const Idx per_token = (Idx)(a.H + a.Hk) << chunk_shift;
  const Idx total = (Idx)a.n_tokens * per_token;
  for (Idx id = (Idx)blockIdx.x * blockDim.x + threadIdx.x; id < total;
       id += (Idx)gridDim.x * blockDim.x) {
    const Idx tq = id / per_token;
    const int c = (int)(id - tq * per_token);
    const int64_t t = (int64_t)tq;
    const int row = c >> chunk_shift;
    const int e0 = (c - (row << chunk_shift)) << 3;
    const int32_t p = __ldg(a.pos + t);
    if (p < 0 || p >= a.freqs_max_len) {
      if (c == 0) raise_error(a.err, ASTR_DEVERR_POS);
      continue;
    }
    float cs[8];
    {
      const float4 *f =
          reinterpret_cast<const float4 *>(a.freqs + (int64_t)p * a.D + 2 * (e0 >> 1));
      float4 f0 = __ldg(f), f1 = __ldg(f + 1);
      cs[0] = f0.x; cs[1] = f0.y; cs[2] = f0.z; cs[3] = f0.w;
      cs[4] = f1.x; cs[5] = f1.y; cs[6] = f1.z; cs[7] = f1.w;
    }
    if (Inverse) cs[1] = -cs[1], cs[3] = -cs[3], cs[5] = -cs[5], cs[7] = -cs[7];
    float x[8], y[8];
    if (row < a.H) {
      const int64_t off = (t * a.H + row) * a.D + e0;
      Chunk<T>::load(a.q, off, x);
      rotate4(x, cs, y);
      Chunk<T>::store(a.q_out, off, y);
    } else {
      const int64_t off = (t * a.Hk + (row - a.H)) * a.D + e0;
      Chunk<T>::load(a.k, off, x);
      rotate4(x, cs, y);
      Chunk<T>::store(a.k_out, off, y);
    }
  }
}

template <bool Inverse>
void launch_apply(const RopeApplyArgs &a, int dtype, int64_t blocks, bool narrow, cudaStream_t s) {
  if (dtype == ASTR_BF16) {
    if (narrow) rope_apply_kernel<bf16_t, uint32_t, Inverse><<<(unsigned)blocks, 256, 0, s>>>(a);
    else rope_apply_kernel<bf16_t, int64_t, Inverse><<<(unsigned)blocks, 256, 0, s>>>(a);
  } else {
    if (narrow) rope_apply_kernel<float, uint32_t, Inverse><<<(unsigned)blocks, 256, 0, s>>>(a);
    else rope_apply_kernel<float, int64_t, Inverse><<<(unsigned)blocks, 256, 0, s>>>(a);
  }
}

}  // namespace

cudaError_t launch_rope_apply(const void *q, void *q_out, const void *k, void *k_out,
                              int64_t n_tokens, int32_t n_heads, int32_t n_kv_heads,
                              int32_t head_dim, int32_t dtype, const float *freqs,
                              int32_t freqs_max_len, const int32_t *position_ids, bool inverse,
                              cudaStream_t stream, int num_sms, uint32_t *err) {
  RopeApplyArgs a;
  a.q = q;
  a.q_out = q_out;
  a.k = k;
  a.k_out = k_out;
  a.freqs = freqs;
  a.pos = position_ids;
  a.n_tokens = n_tokens;
  a.freqs_max_len = freqs_max_len;
  a.H = n_heads;
  a.Hk = n_kv_heads;
  a.D = head_dim;
  a.err = err;
  const int64_t total = n_tokens * (int64_t)(n_heads + n_kv_heads) * (head_dim / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 32;
  if (blocks > cap) blocks = cap;
  const bool narrow = total + blocks * 256 < (int64_t(1) << 32);
  if (inverse) launch_apply<true>(a, dtype, blocks, narrow, stream);
  else launch_apply<false>(a, dtype, blocks, narrow, stream);
  return cudaGetLastError();
}

cudaError_t launch_rope_kv_write(const astr_kv_cache &kv, int32_t layer_id, const void *q,
                                 void *q_out, const void *k, const void *v, int32_t n_heads,
                                 const float *freqs, int32_t freqs_max_len,
                                 const int32_t *position_ids, cudaStream_t stream,
                                 int num_sms, uint32_t *err) {
  RopeArgs a;
  const size_t esz = kv.dtype == ASTR_BF16 ? 2 : 4;
  const int64_t layer_elems = (int64_t)layer_id * kv.size * kv.n_kv_heads * kv.head_dim;
  a.q = q;
  a.q_out = q_out;
  a.k = k;
  a.v = v;
  a.k_layer = static_cast<char *>(kv.k_buffer) + layer_elems * esz;
  a.v_layer = static_cast<char *>(kv.v_buffer) + layer_elems * esz;
  a.freqs = freqs;
  a.pos = position_ids;
  a.loc = kv.out_cache_loc;
  a.n_tokens = kv.n_tokens;
  a.size = kv.size;
  a.freqs_max_len = freqs_max_len;
  a.H = n_heads;
  a.Hk = kv.n_kv_heads;
  a.D = kv.head_dim;
  a.err = err;
  const int64_t total = kv.n_tokens * (int64_t)(n_heads + 2 * kv.n_kv_heads) * (kv.head_dim / 8);
  if (total == 0) return cudaSuccess;
  if (kv.n_tokens <= INT32_MAX) {  // a block per token
    const int64_t per_token = (int64_t)(n_heads + 2 * kv.n_kv_heads) * (kv.head_dim / 8);
    const int nc = (int)((per_token + kTokThreads - 1) / kTokThreads);
    if (nc <= 4) {
      if (kv.dtype == ASTR_BF16) return launch_token_nc<bf16_t>(a, nc, (unsigned)kv.n_tokens, stream);
      return launch_token_nc<float>(a, nc, (unsigned)kv.n_tokens, stream);
    }
    const int threads = per_token >= 512 ? 512 : (int)((per_token + 31) / 32 * 32);
    if (kv.dtype == ASTR_BF16)
      rope_kv_write_token_kernel<bf16_t><<<(unsigned)kv.n_tokens, threads, 0, stream>>>(a);
    else
      rope_kv_write_token_kernel<float><<<(unsigned)kv.n_tokens, threads, 0, stream>>>(a);
    return cudaGetLastError();
  }
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 32;
  if (blocks > cap) blocks = cap;
  // the loop's last index reaches total + grid threads, which must not wrap around either
  const bool narrow = total + blocks * 256 < (int64_t(1) << 32);
  if (kv.dtype == ASTR_BF16) {
    if (narrow) rope_kv_write_kernel<bf16_t, uint32_t><<<(unsigned)blocks, 256, 0, stream>>>(a);
    else rope_kv_write_kernel<bf16_t, int64_t><<<(unsigned)blocks, 256, 0, stream>>>(a);
  } else {
    if (narrow) rope_kv_write_kernel<float, uint32_t><<<(unsigned)blocks, 256, 0, stream>>>(a);
    else rope_kv_write_kernel<float, int64_t><<<(unsigned)blocks, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace astr
