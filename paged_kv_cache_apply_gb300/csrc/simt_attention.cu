// Paged GQA attention on the CUDA cores: split-K decode and the f32 prefill rows.
//
// AstrAI internals, "KV Cache Mathematics": o_n = sum_j softmax(q_n k_j / sqrt(d_k)) v_j.
// AstrAI inference guide, "Attention Backend": req_to_token is the page table (one slot per
// token); "KVCache System": decode_o_part / decode_ml_part hold split-K partials that a
// log-sum-exp merge folds into decode_out.
//
// One thread block handles one (query, KV head, chunk of positions). Decode is bound by HBM
// (2 KB of K+V per token for 4 KV heads of 128 bf16 values), so the block is organised
// around keeping bytes in flight:
//  * warp 4 is the producer: per tile of NT tokens it reads the tokens' slots from the page
//    table and issues one 1-D bulk copy (TMA) per token for the K row slice and one for the
//    V row slice of this KV head into a ring of NSTAGE shared-memory stages, completing on
//    the stage's mbarrier;
//  * warps 0-3 are consumers: each LPR-lane group owns one head_dim slice per lane (16 bytes)
//    and a private online-softmax state for the G query heads that share this KV head.
//    For a batch of NB tokens every lane forms G*NB partial dot products; a reduce-scatter
//    over the group's lanes leaves lane l with the full score of one (head, token) pair.
//    The register <-> pair assignment is permuted by the lane index (register r of lane l
//    holds pair r ^ l), so each butterfly level keeps the lower half of the registers and
//    ships the upper half: LPR-1 shuffles and adds, no selects. The softmax reference max is
//    only raised when a score exceeds it by 2^8 (lazy rescaling), so the accumulators are
//    rescaled only a handful of times per chunk.
//  * at the end the groups' (m, l, acc) states are merged through shared memory; a
//    single-chunk request writes decode_out directly, otherwise the normalised partial and
//    (m, l) go to decode_o_part / decode_ml_part for the merge kernel.
// Every wait is bounded in time; a bad slot or length raises a bit in the device error word
// and is replaced by a safe value instead of faulting.
#include <math.h>

#include "astr_internal.cuh"
#include "launch.h"

namespace astr {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kLazyRescale = 8.0f;  // log2 units

struct AttnArgs {
  const void *q;
  const void *k_layer;
  const void *v_layer;
  const int32_t *r2t;
  const int32_t *rpi;
  const int32_t *seq_lens;
  const int32_t *qo_indptr;
  const int32_t *kv_indptr;
  const int32_t *tile_b;
  const int32_t *tile_i;
  float *o_part;
  float *ml_part;
  void *out;
  int64_t size;
  uint64_t wait_ns;
  uint32_t *err;
  int32_t num_reqs, max_ctx;
  int32_t H, Hk, B;
  int32_t chunk, n_splits, max_splits, max_len;
  int32_t mode;
  int32_t tile_rows;
  float scale_log2;
};

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVec = 4;
  // 16 bytes -> kVec/2 float2
  static __device__ __forceinline__ void unpack(const uint4 &w, float2 (&x)[2]) {
    x[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
    x[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
  static __device__ __forceinline__ void store_out(void *base, int64_t off, float v) {
    static_cast<float *>(base)[off] = v;
  }
};
template <>
struct Elem<bf16_t> {
  static constexpr int kVec = 8;
  static __device__ __forceinline__ void unpack(const uint4 &w, float2 (&x)[4]) {
    x[0] = make_float2(bf16_lo(w.x), bf16_hi(w.x));
    x[1] = make_float2(bf16_lo(w.y), bf16_hi(w.y));
    x[2] = make_float2(bf16_lo(w.z), bf16_hi(w.z));
    x[3] = make_float2(bf16_lo(w.w), bf16_hi(w.w));
  }
  static __device__ __forceinline__ void store_out(void *base, int64_t off, float v) {
    static_cast<uint16_t *>(base)[off] = f32_to_bf16_rn(v);
  }
};

template <typename T, int D, int G>
struct Cfg {
  static constexpr int kVec = Elem<T>::kVec;     // elements per lane (16 bytes)
  static constexpr int kV2 = kVec / 2;            // float2 per lane
  static constexpr int LPR = D / kVec;            // lanes covering one head_dim row
  static_assert(G <= LPR, "group larger than the lanes of a row");
  static constexpr int NB = LPR / G;              // tokens per group batch
  static constexpr int GPW = 32 / LPR;            // lane groups per warp
  static constexpr int NG = kConsumerWarps * GPW; // lane groups per block
  static constexpr int ROWB = D * (int)sizeof(T); // bytes of one token's K (or V) head slice
  // tokens per tile: one batch for every group (128 / G), capped at 48 KB a stage; with the
  // cap some groups see no tokens (wide f32 rows at small G only)
  static constexpr int NT_FULL = NG * NB;
  static constexpr int NT_CAP = (49152 / (2 * ROWB)) / NB * NB;
  static constexpr int NT = NT_FULL <= NT_CAP ? NT_FULL : (NT_CAP < NB ? NB : NT_CAP);
  static constexpr int STAGE_BYTES = 2 * NT * ROWB;
  static constexpr int NSTAGE =
      (65536 / STAGE_BYTES) < 2 ? 2 : ((65536 / STAGE_BYTES) > 8 ? 8 : (65536 / STAGE_BYTES));
  static constexpr int MERGE_BYTES = NG * G * (D + 2) * 4;
  static constexpr int RING_BYTES = NSTAGE * STAGE_BYTES;
  static constexpr int DATA_BYTES = RING_BYTES > MERGE_BYTES ? RING_BYTES : MERGE_BYTES;
  static constexpr int SMEM_BYTES = DATA_BYTES + 2 * NSTAGE * 8 + 16 + 128;
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kThreads) simt_attention_kernel(const AttnArgs a) {
  using C = Cfg<T, D, G>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  unsigned char *ring = smem;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::DATA_BYTES);
  uint64_t *empty = full + C::NSTAGE;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::NSTAGE);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which (query, KV head, chunk) -----------------------------------------------------
  const int g = blockIdx.x % a.Hk;
  int64_t qidx;  // row of q / out
  int b, split = 0;
  int64_t j0, j1;
  if (a.mode == 0) {
    const int64_t w = blockIdx.x / a.Hk;
    split = (int)(w % a.n_splits);
    b = (int)(w / a.n_splits);
    qidx = b;
    const int L = __ldg(a.seq_lens + b);
    if (L < 1 || L > a.max_len || L > a.max_ctx) {
      if (split == 0 && g == 0 && threadIdx.x == 0) raise_error(a.err, ASTR_DEVERR_LEN);
      return;
    }
    j0 = (int64_t)split * a.chunk;
    if (j0 >= L) return;
    j1 = j0 + a.chunk < L ? j0 + a.chunk : L;
  } else {
    const int64_t w = blockIdx.x / a.Hk;
    const int tile = (int)(w / a.tile_rows);
    b = __ldg(a.tile_b + tile);
    if (b == -1) return;  // an empty entry of the tile list
    if (b < 0 || b >= a.B) {
      if (g == 0 && threadIdx.x == 0) raise_error(a.err, ASTR_DEVERR_META);
      return;
    }
    const int64_t i = (int64_t)__ldg(a.tile_i + tile) * a.tile_rows + (w % a.tile_rows);
    const int64_t Qb = (int64_t)__ldg(a.qo_indptr + b + 1) - __ldg(a.qo_indptr + b);
    const int64_t Kb = (int64_t)__ldg(a.kv_indptr + b + 1) - __ldg(a.kv_indptr + b);
    if (i >= Qb) return;
    if (Kb < Qb || Kb > a.max_ctx) {
      if (g == 0 && threadIdx.x == 0) raise_error(a.err, ASTR_DEVERR_LEN);
      return;
    }
    qidx = __ldg(a.qo_indptr + b) + i;
    j0 = 0;
    j1 = Kb - Qb + i + 1;
  }
  const int r = __ldg(a.rpi + b);
  if (r < 0 || r >= a.num_reqs) {
    if (g == 0 && threadIdx.x == 0) raise_error(a.err, ASTR_DEVERR_ROW);
    return;
  }
  const int32_t *row = a.r2t + (int64_t)r * a.max_ctx;
  const int ntiles = (int)((j1 - j0 + C::NT - 1) / C::NT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // per-group merge results are written here after the loop
  float *merge_acc = reinterpret_cast<float *>(smem);
  float *merge_ml = merge_acc + C::NG * G * D;

  if (warp == kConsumerWarps) {
    // ================================ producer ===========================================
    const T *kl = static_cast<const T *>(a.k_layer);
    const T *vl = static_cast<const T *>(a.v_layer);
    int issued = 0;
    for (int it = 0; it < ntiles; ++it) {
      const int st = it % C::NSTAGE;
      if (it >= C::NSTAGE) {
        if (!mbar_wait(&empty[st], ((it / C::NSTAGE) - 1) & 1, a.wait_ns, a.err)) *abort_flag = 1;
      }
      if (*abort_flag) break;
      const int64_t tok0 = j0 + (int64_t)it * C::NT;
      const int n = (int)((j1 - tok0) < C::NT ? (j1 - tok0) : C::NT);
      if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)(n * 2 * C::ROWB));
      __syncwarp();
      unsigned char *kst = ring + st * C::STAGE_BYTES;
      unsigned char *vst = kst + C::NT * C::ROWB;
      for (int i = lane; i < n; i += 32) {
        int64_t slot = __ldg(row + tok0 + i);
        if (slot < 0 || slot >= a.size) {
          raise_error(a.err, ASTR_DEVERR_SLOT);
          slot = 0;
        }
        const int64_t off = (slot * a.Hk + g) * D;
        bulk_g2s(kst + i * C::ROWB, kl + off, C::ROWB, &full[st]);
        bulk_g2s(vst + i * C::ROWB, vl + off, C::ROWB, &full[st]);
      }
      issued = it + 1;
    }
    __syncthreads();  // join the consumers
    if (*abort_flag) {
      // a consumer gave up: the copies already issued must land before the block (and its
      // shared memory) goes away; the last NSTAGE tiles cover one phase of every stage
      for (int it = issued - C::NSTAGE < 0 ? 0 : issued - C::NSTAGE; it < issued; ++it)
        mbar_wait(&full[it % C::NSTAGE], (it / C::NSTAGE) & 1, kDrainLimitNs, a.err);
    }
    return;
  }

  // ================================== consumers ============================================
  const int grp = lane / C::LPR;           // lane group within the warp
  const int l = lane % C::LPR;             // lane within the group: head_dim slice index
  const int lh = l / C::NB, lt = l % C::NB;
  const int gi = warp * C::GPW + grp;      // group index within the block
  const int gbase = grp * C::LPR;          // first lane of my group

  float2 q2[G][C::kV2];
#pragma unroll
  for (int rh = 0; rh < G; ++rh) {
    const int head = g * G + (rh ^ lh);
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(static_cast<const T *>(a.q) +
                                                          (qidx * a.H + head) * D) + l);
    Elem<T>::unpack(w, q2[rh]);
  }
  float2 acc[G][C::kV2];
  float m[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
#pragma unroll
    for (int e = 0; e < C::kV2; ++e) acc[h][e] = make_float2(0.f, 0.f);
  }
  float l_lane = 0.f;

  for (int it = 0; it < ntiles; ++it) {
    const int st = it % C::NSTAGE;
    if (*abort_flag) break;
    if (!mbar_wait(&full[st], (it / C::NSTAGE) & 1, a.wait_ns, a.err)) {
      *abort_flag = 1;
      break;
    }
    const int64_t tok0 = j0 + (int64_t)it * C::NT;
    const int n = (int)((j1 - tok0) < C::NT ? (j1 - tok0) : C::NT);
    const unsigned char *kst = ring + st * C::STAGE_BYTES;
    const unsigned char *vst = kst + C::NT * C::ROWB;
    const int tb = gi * C::NB;  // my group's first token in the tile

    // ---- scores: partial dot products, then a reduce-scatter over the group's lanes ----
    float part[C::LPR];
#pragma unroll
    for (int rt = 0; rt < C::NB; ++rt) {
      const int tok = tb + (rt ^ lt);
      float2 k2[C::kV2];
      if (tok < n) {
        const uint4 w = *reinterpret_cast<const uint4 *>(kst + tok * C::ROWB + l * 16);
        Elem<T>::unpack(w, k2);
      } else {
#pragma unroll
        for (int e = 0; e < C::kV2; ++e) k2[e] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int rh = 0; rh < G; ++rh) {
        float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < C::kV2; ++e) d2 = ffma2(q2[rh][e], k2[e], d2);
        part[rh * C::NB + rt] = d2.x + d2.y;
      }
    }
#pragma unroll
    for (int msk = C::LPR / 2; msk >= 1; msk >>= 1) {
#pragma unroll
      for (int i = 0; i < msk; ++i) part[i] += __shfl_xor_sync(0xffffffffu, part[i + msk], msk);
    }
    const bool valid = (tb + lt) < n;
    const float s = valid ? part[0] * a.scale_log2 : -INFINITY;

    // ---- online softmax with lazy rescaling ----
    float bmax = s;
#pragma unroll
    for (int msk = C::NB / 2; msk >= 1; msk >>= 1)
      bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, msk));
    float m_own = m[0];
#pragma unroll
    for (int h = 1; h < G; ++h)
      if (h == lh) m_own = m[h];
    const float m_new_own = (bmax > m_own + kLazyRescale) ? bmax : m_own;
    if (__any_sync(0xffffffffu, m_new_own != m_own)) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mn = __shfl_sync(0xffffffffu, m_new_own, gbase + h * C::NB);
        if (mn != m[h]) {
          const float alpha = ex2_approx(m[h] - mn);  // m[h] = -inf gives 0
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < C::kV2; ++e) acc[h][e] = ffma2(acc[h][e], a2, make_float2(0.f, 0.f));
          if (h == lh) l_lane *= alpha;
          m[h] = mn;
        }
      }
    }
    const float p = valid ? ex2_approx(s - m_new_own) : 0.f;
    l_lane += p;

    // ---- P.V ----
#pragma unroll
    for (int t = 0; t < C::NB; ++t) {
      float pt[G];
#pragma unroll
      for (int h = 0; h < G; ++h) pt[h] = __shfl_sync(0xffffffffu, p, gbase + h * C::NB + t);
      if (tb + t < n) {
        const uint4 w = *reinterpret_cast<const uint4 *>(vst + (tb + t) * C::ROWB + l * 16);
        float2 v2[C::kV2];
        Elem<T>::unpack(w, v2);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float2 p2 = make_float2(pt[h], pt[h]);
#pragma unroll
          for (int e = 0; e < C::kV2; ++e) acc[h][e] = ffma2(p2, v2[e], acc[h][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---- fold this group's state: l per head, then publish (m, l, acc) ----
#pragma unroll
  for (int msk = C::NB / 2; msk >= 1; msk >>= 1) l_lane += __shfl_xor_sync(0xffffffffu, l_lane, msk);
  float lsum[G];
#pragma unroll
  for (int h = 0; h < G; ++h) lsum[h] = __shfl_sync(0xffffffffu, l_lane, gbase + h * C::NB);

  __syncthreads();  // join the producer: without an abort every copy has landed and been read
  if (*abort_flag) return;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float *dst = merge_acc + ((int64_t)gi * G + h) * D + l * C::kVec;
#pragma unroll
    for (int e = 0; e < C::kV2; ++e) {
      dst[2 * e] = acc[h][e].x;
      dst[2 * e + 1] = acc[h][e].y;
    }
    if (l == 0) {
      merge_ml[(gi * G + h) * 2] = m[h];
      merge_ml[(gi * G + h) * 2 + 1] = lsum[h];
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32));

  // ---- merge the groups and write the chunk's result ----
  const bool single = a.mode == 1 || a.n_splits == 1 ||
                      (a.mode == 0 && (int64_t)__ldg(a.seq_lens + b) <= a.chunk);
  for (int o = threadIdx.x; o < G * D; o += kConsumerWarps * 32) {
    const int h = o / D, e = o % D;
    float M = -INFINITY;
    for (int q = 0; q < C::NG; ++q) M = fmaxf(M, merge_ml[(q * G + h) * 2]);
    float num = 0.f, den = 0.f;
    for (int q = 0; q < C::NG; ++q) {
      const float mq = merge_ml[(q * G + h) * 2];
      if (mq == -INFINITY) continue;
      const float w = ex2_approx(mq - M);
      num += w * merge_acc[((int64_t)q * G + h) * D + e];
      den += w * merge_ml[(q * G + h) * 2 + 1];
    }
    const int head = g * G + h;
    if (single) {
      Elem<T>::store_out(a.out, (qidx * a.H + head) * D + e, num / den);
    } else {
      const int64_t pidx = ((int64_t)b * a.H + head) * a.max_splits + split;
      a.o_part[pidx * D + e] = num / den;
      if (e == 0) {
        a.ml_part[pidx * 2] = M * 0.69314718055994531f;  // back to natural-exponent units
        a.ml_part[pidx * 2 + 1] = den;
      }
    }
  }
}

// Log-sum-exp merge of the split-K partials: one warp per (request, head). The maximum and the
// weights are taken with the lanes spread over the splits; the weighted partials are then
// summed split by split, eight splits' loads in flight at a time (a warp that waited on each
// split's loads in turn spent most of a many-split merge on memory latency).
template <typename T, int D>
__global__ void __launch_bounds__(256) split_merge_kernel(const AttnArgs a) {
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)a.B * a.H) return;
  const int b = (int)(wid / a.H), h = (int)(wid % a.H);
  const int L = __ldg(a.seq_lens + b);
  if (L < 1 || L > a.max_len) return;
  const int n = (L + a.chunk - 1) / a.chunk;
  if (n <= 1) return;  // written directly by the attention kernel
  const int64_t base = ((int64_t)b * a.H + h) * a.max_splits;
  const float2 *ml = reinterpret_cast<const float2 *>(a.ml_part) + base;  // (m, l) per split
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, ml[s].x);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int PER = D / 32;
  float o[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) o[e] = 0.f;
  float den_part = 0.f;
  for (int s0 = 0; s0 < n; s0 += 32) {
    float w_mine = 0.f;  // the weight of split s0 + lane
    if (s0 + lane < n) {
      const float2 v = ml[s0 + lane];
      w_mine = v.y * ex2_approx((v.x - M) * 1.4426950408889634f);
    }
    den_part += w_mine;
    const int cnt = n - s0 < 32 ? n - s0 : 32;
#pragma unroll 8
    for (int j = 0; j < cnt; ++j) {
      const float w = __shfl_sync(0xffffffffu, w_mine, j);
      const float *op = a.o_part + (base + s0 + j) * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[e] += w * op[e];
    }
  }
  float den = den_part;
#pragma unroll
  for (int o2 = 16; o2 >= 1; o2 >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o2);
  const float inv = 1.f / den;
#pragma unroll
  for (int e = 0; e < PER; ++e) Elem<T>::store_out(a.out, ((int64_t)b * a.H + h) * D + lane * PER + e, o[e] * inv);
}

template <typename T, int D, int G>
cudaError_t run(const AttnArgs &a, int64_t grid, cudaStream_t stream) {
  using C = Cfg<T, D, G>;
  auto kern = simt_attention_kernel<T, D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (grid > 0) kern<<<(unsigned)grid, kThreads, C::SMEM_BYTES, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.mode == 0 && a.n_splits > 1) {
    const int64_t warps = (int64_t)a.B * a.H;
    split_merge_kernel<T, D><<<(unsigned)((warps * 32 + 255) / 256), 256, 0, stream>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

AttnArgs merge_args(const astr_kv_cache &kv, int32_t n_heads, const SimtAttnPlan &plan) {
  AttnArgs a = {};
  a.seq_lens = kv.seq_lens;
  a.o_part = kv.decode_o_part;
  a.ml_part = kv.decode_ml_part;
  a.out = kv.decode_out;
  a.H = n_heads;
  a.B = kv.batch;
  a.chunk = plan.chunk;
  a.n_splits = plan.n_splits;
  a.max_splits = kv.max_splits;
  a.max_len = kv.max_len;
  return a;
}

template <typename T, int D>
cudaError_t dispatch_g(int G, const AttnArgs &a, int64_t grid, cudaStream_t s) {
  switch (G) {
    case 1: return run<T, D, 1>(a, grid, s);
    case 2: return run<T, D, 2>(a, grid, s);
    case 4: return run<T, D, 4>(a, grid, s);
    case 8: return run<T, D, 8>(a, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_split_merge(const astr_kv_cache &kv, int32_t n_heads, const SimtAttnPlan &plan,
                               cudaStream_t stream) {
  const AttnArgs a = merge_args(kv, n_heads, plan);
  const int64_t warps = (int64_t)kv.batch * n_heads;
  const unsigned grid = (unsigned)((warps * 32 + 255) / 256);
  if (kv.dtype == ASTR_BF16) {
    if (kv.head_dim == 128) split_merge_kernel<bf16_t, 128><<<grid, 256, 0, stream>>>(a);
    else split_merge_kernel<bf16_t, 64><<<grid, 256, 0, stream>>>(a);
  } else {
    if (kv.head_dim == 128) split_merge_kernel<float, 128><<<grid, 256, 0, stream>>>(a);
    else split_merge_kernel<float, 64><<<grid, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

bool simt_attn_supported(int dtype, int head_dim, int group) {
  return (dtype == ASTR_F32 || dtype == ASTR_BF16) && (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8);
}

int simt_tile_tokens(int group) { return 128 / group; }

cudaError_t launch_simt_attention(const astr_kv_cache &kv, int32_t layer_id, const void *q,
                                  void *out, int32_t n_heads, const SimtAttnPlan &plan,
                                  cudaStream_t stream) {
  AttnArgs a;
  const size_t esz = kv.dtype == ASTR_BF16 ? 2 : 4;
  const int64_t layer_elems = (int64_t)layer_id * kv.size * kv.n_kv_heads * kv.head_dim;
  a.q = q;
  a.k_layer = static_cast<const char *>(kv.k_buffer) + layer_elems * esz;
  a.v_layer = static_cast<const char *>(kv.v_buffer) + layer_elems * esz;
  a.r2t = kv.req_to_token;
  a.rpi = kv.req_pool_indices;
  a.seq_lens = kv.seq_lens;
  a.qo_indptr = kv.qo_indptr;
  a.kv_indptr = kv.kv_indptr;
  a.tile_b = kv.q_tile_to_batch;
  a.tile_i = kv.q_tile_to_index;
  a.tile_rows = kv.q_tile_rows;
  a.o_part = kv.decode_o_part;
  a.ml_part = kv.decode_ml_part;
  a.out = out;
  a.size = kv.size;
  a.wait_ns = plan.wait_ns;
  a.err = plan.err;
  a.num_reqs = kv.num_reqs;
  a.max_ctx = kv.max_ctx_len;
  a.H = n_heads;
  a.Hk = kv.n_kv_heads;
  a.B = kv.batch;
  a.chunk = plan.chunk;
  a.n_splits = plan.n_splits;
  a.max_splits = kv.max_splits;
  a.max_len = kv.max_len;
  a.mode = plan.mode;
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kv.head_dim));
  int64_t grid;
  if (plan.mode == 0) {
    grid = (int64_t)kv.batch * plan.n_splits * kv.n_kv_heads;
  } else {
    grid = (int64_t)kv.num_q_tiles * kv.q_tile_rows * kv.n_kv_heads;
  }
  const int G = n_heads / kv.n_kv_heads;
  if (kv.dtype == ASTR_BF16) {
    if (kv.head_dim == 128) return dispatch_g<bf16_t, 128>(G, a, grid, stream);
    return dispatch_g<bf16_t, 64>(G, a, grid, stream);
  }
  if (kv.head_dim == 128) return dispatch_g<float, 128>(G, a, grid, stream);
  return dispatch_g<float, 64>(G, a, grid, stream);
}

}  // namespace astr
