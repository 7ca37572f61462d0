// Paged GQA decode attention on the tcgen05 tensor cores (bf16, head_dim 128).
//
// AstrAI internals, "KV Cache Mathematics": o_n = sum_j softmax(q_n k_j / sqrt(d_k)) v_j.
// AstrAI inference guide, "Attention Backend" (req_to_token as the page table) and "KVCache
// System" (decode_o_part / decode_ml_part split-K partials, merged by log-sum-exp).
//
// Decode reads 512 bytes of K+V per token and KV head and does 4*G multiply-adds per byte,
// so the kernel is built around the copy pipeline and keeps the arithmetic off the CUDA
// cores. A work item is (request, chunk, KV head g) with the G query heads of the group. The
// kernel is persistent: one block per SM claims items from a counter until none are left, and
// its copy pipeline streams from one item into the next without draining, so a block's
// start-up (3.5 us before its first tile) is paid once per SM instead of once per item:
//  * warp 9 claims items (split-major: every request's first chunk before any second one, and
//    within a split the requests longest first, so the run ends on the shortest chunks),
//    publishes each through a two-slot ring in shared memory, and
//    stages the item's query rows in one of two Q buffers;
//  * warps 4-7 stream 128-token tiles of the item's KV-head slices of K and V into a 3-stage
//    ring in the 128-byte-swizzled operand layout, 32 tokens per warp: when those are two
//    whole pages (two runs of 16 consecutive slots) they come as four TMA boxes of 16 rows
//    (one per 64-element half of K and of V), otherwise as 16-byte cp.async copies (eight
//    lanes per token row, four whole rows per instruction; the lanes take their rows' slots
//    from shared memory) with positions past the chunk zero-filled.
//    Which path a warp takes is uniform across it, so the copy loop stays straight-line code;
//  * warp 8 allocates 64 TMEM columns -- two S buffers and two O^T buffers of 16 columns --
//    and issues, per tile, S^T = K Q^T (M = 128 tokens on the TMEM lanes, N = 16 query rows
//    of which G are the group, K = 128) and, one tile behind, O^T += V^T P^T (M = 128 =
//    head_dim, N = 16, K = 128 tokens) with V read as an MN-major operand and P^T from shared
//    memory (MN-major too, 32-byte swizzled); consecutive items accumulate into alternate O^T
//    buffers;
//  * warps 0-3 (one TMEM lane each) read a token's G scores, take the tile max per head
//    across the 128 lanes (a butterfly of warp shuffles that splits the G values across
//    lanes, then one named barrier), keep the softmax reference
//    max lazily (raised only when a score exceeds it by 2^8, then O^T is rescaled in TMEM),
//    write P^T in bf16 and, after an item's last tile, normalise O^T and store the output or
//    the chunk's partial and (m, l).
// Tile and item counters run on across items, and every barrier phase follows them.
// Every wait is bounded; a bad slot is zero-filled and flagged; on a timeout the block stops,
// waits for its own copies and MMAs, frees TMEM and returns.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "astr_internal.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace astr {

namespace {

constexpr int kTok = 128;                 // tokens per tile (M of S^T)
constexpr int kD = 128;                   // head_dim
constexpr int kNPad = 16;                 // query rows per MMA (N)
constexpr int kStages = 3;
constexpr int kTileBytes = kTok * kD * 2; // 32 KB: K (or V) of one tile
constexpr int kBlockBytes = kTok * 128;   // 16 KB: one 64-element half of a tile
constexpr int kThreads = 320;             // 4 softmax + 4 loader + MMA + scheduler warps
constexpr int kSchedSlots = 32;           // work counters, used in turn by successive launches
constexpr float kLazyRescale = 8.0f;

// shared-memory map (offsets from a 1 KB aligned base)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffQ = kOffV + kStages * kTileBytes;  // 2 buffers x (16 rows x 128: 2 blocks of 2 KB)
constexpr int kOffP = kOffQ + 2 * 4096;               // 2 buffers x (16 rows x 128 tokens)
constexpr int kOffRed = kOffP + 2 * 4096;             // [2][4 warps][16] f32 tile maxima
constexpr int kOffLsum = kOffRed + 2 * 4 * 16 * 4;    // [4 warps][16] f32
constexpr int kOffBar = kOffLsum + 4 * 16 * 4;
constexpr int kOffRing = kOffBar + 32 * 8;            // 2 published work items, 64 bytes each
constexpr int kOffMisc = kOffRing + 2 * 64;
constexpr int kSortMax = 1024;                        // batches up to this size claim longest first
constexpr int kBuckets = 1024;                        // seq_len ranks by 128-token tile count
constexpr int kOffOrder = kOffMisc + 64;              // [kSortMax] requests by seq_len, [kBuckets] counts
constexpr int kOffSlots = kOffOrder + (kSortMax + kBuckets) * 4;  // [4 loader warps][2][32] slots
constexpr int kSmemBytes = kOffSlots + 4 * 2 * 32 * 4 + 1024;  // + alignment slack

constexpr uint32_t kIdescQK = tc::idesc_bf16(128, kNPad, false, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, kNPad, true, true);

struct DecArgs {
  const void *q;
  const void *k_layer;
  const void *v_layer;
  const int32_t *r2t;
  const int32_t *rpi;
  const int32_t *seq_lens;
  float *o_part;
  float *ml_part;
  void *out;
  int64_t size;
  uint64_t wait_ns;
  uint32_t *err;
  int32_t num_reqs, max_ctx;
  int32_t H, Hk, B;
  int32_t chunk, n_splits, max_splits, max_len;
  int32_t layer_row0;  // first row of this layer in the [n_layers * size, Hk * D] tensor maps
  int32_t use_tma;     // page runs by TMA (the maps' row coordinates fit in 32 bits)
  float scale_log2;
  int64_t n_items;     // batch * n_splits * Hk work items
  unsigned *sched;     // [0]: items claimed past the first one of each block, [1]: blocks done
  // RoPE and the new token's cache write folded in (astr_decode_attention_rope); fused = 0
  // for plain decode
  const void *k_new;   // [B, Hk, D]: the new token's key, rotated here
  const void *v_new;   // [B, Hk, D]: its value
  const float *freqs;  // [freqs_max_len, D / 2, 2] (cos, sin)
  const int32_t *pos;  // [B] position of the new token
  const int32_t *loc;  // [B] its cache slot
  int32_t freqs_max_len;
  int32_t fused;
};

// One work item, (request b, chunk `split`, KV head g), as the scheduler warp hands it to the
// other roles (ntiles = 0 ends the sequence).
struct DecItem {
  int64_t j0, j1;      // positions [j0, j1) of the request
  const int32_t *row;  // its page-table row
  int32_t b, g, split, L, ntiles;
};
static_assert(sizeof(DecItem) <= 64, "ring slot");

// mbar_wait for a thread nothing waits on closely: it sleeps between polls instead of
// taking issue slots from the warps it shares a scheduler with
__device__ __forceinline__ bool sleepy_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                            uint32_t *err) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      raise_error(err, ASTR_DEVERR_TIMEOUT);
      return false;
    }
    __nanosleep(500);
  }
  return true;
}

__device__ __forceinline__ bool bar_any(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int G>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&x)[G]) {
  if constexpr (G <= 4) {
    uint32_t r[4];
    tc::tmem_ld4(taddr, r);
    tc::tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < G; ++h) x[h] = __uint_as_float(r[h]);
  } else if constexpr (G == 8) {
    uint32_t r[8];
    tc::tmem_ld8(taddr, r);
    tc::tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < G; ++h) x[h] = __uint_as_float(r[h]);
  } else {
    uint32_t r[16];
    tc::tmem_ld16(taddr, r);
    tc::tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < G; ++h) x[h] = __uint_as_float(r[h]);
  }
}

template <int G>
__device__ __forceinline__ void st_cols(uint32_t taddr, const float (&x)[G]) {
  if constexpr (G <= 4) {
    uint32_t r[4] = {0, 0, 0, 0};
#pragma unroll
    for (int h = 0; h < G; ++h) r[h] = __float_as_uint(x[h]);
    tc::tmem_st4(taddr, r);
  } else if constexpr (G == 8) {
    uint32_t r[8];
#pragma unroll
    for (int h = 0; h < G; ++h) r[h] = __float_as_uint(x[h]);
    tc::tmem_st8(taddr, r);
  } else {
    uint32_t r[16];
#pragma unroll
    for (int h = 0; h < G; ++h) r[h] = __float_as_uint(x[h]);
    tc::tmem_st16(taddr, r);
  }
  tc::tmem_st_wait();
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const DecArgs a, const __grid_constant__ CUtensorMap k16,
                     const __grid_constant__ CUtensorMap v16) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *full = bars;                 // [kStages] loaders -> MMA (128 + 4 arrivals, TMA bytes)
  uint64_t *empty = bars + kStages;      // [kStages] MMA -> loaders (commit)
  uint64_t *s_full = bars + 2 * kStages; // [2] MMA -> softmax (commit), per tile
  uint64_t *p_full = s_full + 2;         // [2] softmax -> MMA (128 arrivals), per tile
  uint64_t *pv_done = p_full + 2;        // [2] MMA -> softmax (commit), per tile
  uint64_t *q_full = pv_done + 2;        // [2] scheduler -> MMA, per item
  uint64_t *q_empty = q_full + 2;        // [2] MMA commit after an item's last S, per item
  uint64_t *o_free = q_empty + 2;        // [2] softmax (128 arrivals) read O, per item
  uint64_t *item_full = o_free + 2;      // [2] scheduler published an item
  uint64_t *item_empty = item_full + 2;  // [2] loaders (4), MMA (1), softmax (128) took it
  uint64_t *drain = item_empty + 2;      // MMA -> itself (commit)
  DecItem *ring = reinterpret_cast<DecItem *>(smem + kOffRing);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
  float *red = reinterpret_cast<float *>(smem + kOffRed);
  float *lsum_s = reinterpret_cast<float *>(smem + kOffLsum);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- set-up --------------------------------------------------------------------------------
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 128 + 4);  // every loader lane's cp.async + one expect-tx per warp
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&o_free[i], 128);
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], 4 + 1 + 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tc::tmem_alloc(tmem_slot, 64);
    tc::tmem_relinquish();
  }
  if (warp < 4) {  // zero both Q and both P buffers (rows past the group stay zero)
    uint4 *z = reinterpret_cast<uint4 *>(smem + kOffQ);
    for (int i = tid; i < (8192 + 8192) / 16; i += 128) z[i] = make_uint4(0, 0, 0, 0);
  }
  // Requests ranked by seq_len in 128-token tiles, most tiles first (ties by index): the claims
  // walk the ranks within each split, so every split's long chunks go first and the run ends on
  // the shortest ones. A stable counting sort: a histogram of tile counts, a descending exclusive
  // scan over it, and a placement in index order. It must be deterministic: every block ranks
  // for itself, and the claim counter they share only means the same request to all of them if
  // their ranks agree.
  int32_t *order = reinterpret_cast<int32_t *>(smem + kOffOrder);
  const bool ranked = a.B <= kSortMax;
  if (ranked) {
    int32_t *cnt = order + kSortMax;  // [kBuckets]: counts, then the next free rank of each
    __shared__ int32_t warp_sums[kThreads / 32];
    auto bucket = [](int32_t L) {
      const int32_t t = L > 0 ? (L + 127) >> 7 : 0;
      return t < kBuckets ? t : kBuckets - 1;
    };
    for (int k = tid; k < kBuckets; k += kThreads) cnt[k] = 0;
    __syncthreads();
    for (int b = tid; b < a.B; b += kThreads) atomicAdd(&cnt[bucket(__ldg(a.seq_lens + b))], 1);
    __syncthreads();
    // thread i holds buckets kBuckets-1-4i .. kBuckets-4-4i (descending); scan their sums
    constexpr int kPer = (kBuckets + kThreads - 1) / kThreads;
    int local[kPer], sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int rv = tid * kPer + j;
      local[j] = rv < kBuckets ? cnt[kBuckets - 1 - rv] : 0;
      sum += local[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += warp_sums[w];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int rv = tid * kPer + j;
      if (rv < kBuckets) cnt[kBuckets - 1 - rv] = run;  // first rank of that bucket
      run += local[j];
    }
    __syncthreads();
    if (warp == 0) {  // 32 requests at a time, in index order; lanes sharing a count take turns
      for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        const bool live = b < a.B;
        const int k = live ? bucket(__ldg(a.seq_lens + b)) : -1 - lane;  // unique for dead lanes
        const unsigned same = __match_any_sync(0xffffffffu, k);
        const int before = __popc(same & ((1u << lane) - 1u));
        const int base = live ? cnt[k] : 0;
        __syncwarp();
        if (live) {
          order[base + before] = b;
          if (before == 0) cnt[k] = base + __popc(same);
        }
        __syncwarp();
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem, tO0 = tmem + 32;  // S: 2 x 16 columns; O^T: 2 x 16 columns

  // publication n of the ring: every reader waits, copies and arrives once
  auto take = [&](uint32_t n, DecItem &w) -> bool {
    if (!mbar_wait(&item_full[n & 1], (n >> 1) & 1, a.wait_ns, a.err)) return false;
    w = ring[n & 1];
    mbar_arrive(&item_empty[n & 1]);
    return true;
  };

  if (warp < 4) {
    // ============================ softmax / epilogue ===========================================
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t it = 0;  // tiles passed, over all items
    bool aborted = false;
    for (uint32_t n = 0; !aborted; ++n) {
      DecItem w;
      if (!take(n, w)) {
        aborted = true;
        break;
      }
      if (w.ntiles == 0) break;
      const uint32_t tO = tO0 + (n & 1) * 16;
      float m[G], l[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      for (int j = 0; j < w.ntiles; ++j, ++it) {
        const int sb = it & 1;
        const int64_t tok0 = w.j0 + (int64_t)j * kTok;
        const int nv = (int)((w.j1 - tok0) < kTok ? (w.j1 - tok0) : kTok);
        bool ok = true;
        if (it >= 2) ok = mbar_wait(&pv_done[sb], ((it - 2) >> 1) & 1, a.wait_ns, a.err);
        ok = ok && mbar_wait(&s_full[sb], (it >> 1) & 1, a.wait_ns, a.err);
        float x[G];
#pragma unroll
        for (int h = 0; h < G; ++h) x[h] = -INFINITY;
        if (ok) {
          tc::fence_after_sync();
          float s[G];
          ld_cols<G>(tS0 + lane_base + sb * 16, s);
          const bool valid = tid < nv;
#pragma unroll
          for (int h = 0; h < G; ++h) x[h] = valid ? s[h] * a.scale_log2 : -INFINITY;
          // The warp's G maxima in (G - 1) + 5 - log2(G) shuffles instead of 5 G: while a lane
          // holds w > 1 values, the exchange across lane bit m halves them (a lane with the bit
          // set keeps the upper half and sends the lower one), and single values then finish
          // the remaining lane bits. The lanes whose low log2(32 / G) bits are zero end with one
          // head's maximum each (head hsel). Measured on GB300 against five shuffles per head
          // (G = 4): one-token pages 75.8 against 76.4 us, the mixed batch 328.1 against 329.2.
          float v[G];
#pragma unroll
          for (int h = 0; h < G; ++h) v[h] = x[h];
          int hsel = 0;
#pragma unroll
          for (int w = G, m = 16; w > 1; w >>= 1, m >>= 1) {
            const bool up = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < w / 2; ++i) {
              const float send = up ? v[i] : v[i + w / 2];
              const float keep = up ? v[i + w / 2] : v[i];
              v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, m));
            }
            if (up) hsel += w / 2;
          }
#pragma unroll
          for (int m = 16 / G; m >= 1; m >>= 1) v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], m));
          if ((lane & (32 / G - 1)) == 0) red[(sb * 4 + warp) * 16 + hsel] = v[0];
        }
        if (bar_any(1, 128, !ok)) {
          aborted = true;
          break;
        }
        float mnew[G];
        bool changed = false;
        float M[G];
        // the four warps' maxima, read as 16-byte vectors where G allows (measured on GB300 with the
        // row sums' butterfly below: one-token pages 75.8 against 76.8 us)
        if constexpr (G % 4 == 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int h4 = 0; h4 < G; h4 += 4) {
              const float4 r4 = *reinterpret_cast<const float4 *>(red + (sb * 4 + q) * 16 + h4);
              M[h4 + 0] = q == 0 ? r4.x : fmaxf(M[h4 + 0], r4.x);
              M[h4 + 1] = q == 0 ? r4.y : fmaxf(M[h4 + 1], r4.y);
              M[h4 + 2] = q == 0 ? r4.z : fmaxf(M[h4 + 2], r4.z);
              M[h4 + 3] = q == 0 ? r4.w : fmaxf(M[h4 + 3], r4.w);
            }
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            M[h] = red[(sb * 4 + 0) * 16 + h];
#pragma unroll
            for (int q = 1; q < 4; ++q) M[h] = fmaxf(M[h], red[(sb * 4 + q) * 16 + h]);
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          mnew[h] = (M[h] > m[h] + kLazyRescale) ? M[h] : m[h];
          changed |= mnew[h] != m[h];
        }
        if (changed) {  // the same decision in every thread
          float alpha[G];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            alpha[h] = ex2_approx(m[h] - mnew[h]);  // 0 while m is still -inf
            l[h] *= alpha[h];
            m[h] = mnew[h];
          }
          if (j > 0) {  // O^T holds this item's earlier tiles: rescale once PV(it-1) has landed
            const bool ok2 = mbar_wait(&pv_done[(it - 1) & 1], ((it - 1) >> 1) & 1, a.wait_ns, a.err);
            if (bar_any(1, 128, !ok2)) {
              aborted = true;
              break;
            }
            tc::fence_after_sync();
            float o[G];
            ld_cols<G>(tO + lane_base, o);
#pragma unroll
            for (int h = 0; h < G; ++h) o[h] *= alpha[h];
            st_cols<G>(tO + lane_base, o);
          }
        }
        // P^T for this tile, MN-major with 32-byte swizzling: token `tid`'s 16 query rows are one
        // 32-byte line whose two 16-byte halves swap when bit 2 of the token is set; the G
        // values of this thread go out in one store per half (measured on GB300 against the
        // K-major layout, G two-byte stores per thread: one-token pages 75.3 against 75.7 us,
        // long decode 161.0 against 163.1, the mixed batch 327.2 against 328.7)
        unsigned char *pb = smem + kOffP + sb * 4096 + tid * 32;
        const uint32_t swz = (uint32_t)((tid >> 2) & 1) << 4;
        float p[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          p[h] = (tid < nv) ? ex2_approx(x[h] - m[h]) : 0.f;
          l[h] += p[h];
        }
        if constexpr (G == 1) {
          *reinterpret_cast<uint16_t *>(pb + swz) = f32_to_bf16_rn(p[0]);
        } else if constexpr (G == 2) {
          *reinterpret_cast<uint32_t *>(pb + swz) = pack_bf16x2_rn(p[0], p[1]);
        } else if constexpr (G == 4) {
          *reinterpret_cast<uint2 *>(pb + swz) = make_uint2(pack_bf16x2_rn(p[0], p[1]), pack_bf16x2_rn(p[2], p[3]));
        } else {
#pragma unroll
          for (int c = 0; c < G / 8; ++c)
            *reinterpret_cast<uint4 *>(pb + (((uint32_t)c << 4) ^ swz)) =
                make_uint4(pack_bf16x2_rn(p[8 * c], p[8 * c + 1]), pack_bf16x2_rn(p[8 * c + 2], p[8 * c + 3]),
                           pack_bf16x2_rn(p[8 * c + 4], p[8 * c + 5]), pack_bf16x2_rn(p[8 * c + 6], p[8 * c + 7]));
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        mbar_arrive(&p_full[sb]);
      }
      if (aborted) break;
      // epilogue: the commit after the item's last P.V covers all of its MMAs
      const uint32_t last = it - 1;
      const bool ok = mbar_wait(&pv_done[last & 1], (last >> 1) & 1, a.wait_ns, a.err);
      if (bar_any(1, 128, !ok)) {
        aborted = true;
        break;
      }
      tc::fence_after_sync();
      {  // l over the 128 token lanes: the value-splitting butterfly of the tile maxima, with sums
        float v[G];
#pragma unroll
        for (int h = 0; h < G; ++h) v[h] = l[h];
        int hsel = 0;
#pragma unroll
        for (int w = G, m = 16; w > 1; w >>= 1, m >>= 1) {
          const bool up = (lane & m) != 0;
#pragma unroll
          for (int i = 0; i < w / 2; ++i) {
            const float send = up ? v[i] : v[i + w / 2];
            const float keep = up ? v[i + w / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
          }
          if (up) hsel += w / 2;
        }
#pragma unroll
        for (int m = 16 / G; m >= 1; m >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
        if ((lane & (32 / G - 1)) == 0) lsum_s[warp * 16 + hsel] = v[0];
      }
      bar_sync(1, 128);
      float o[G];
      ld_cols<G>(tO + lane_base, o);  // lane = head_dim index `tid`
      tc::fence_before_sync();
      mbar_arrive(&o_free[n & 1]);  // the next item but one may accumulate into these columns
      const bool single = a.n_splits == 1 || w.L <= a.chunk;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float Lh = lsum_s[h] + lsum_s[16 + h] + lsum_s[32 + h] + lsum_s[48 + h];
        const float val = o[h] / Lh;
        const int head = w.g * G + h;
        if (single) {
          static_cast<uint16_t *>(a.out)[((int64_t)w.b * a.H + head) * kD + tid] = f32_to_bf16_rn(val);
        } else {
          const int64_t pidx = ((int64_t)w.b * a.H + head) * a.max_splits + w.split;
          a.o_part[pidx * kD + tid] = val;
          if (tid == 0) {
            a.ml_part[pidx * 2] = m[h] * 0.69314718055994531f;
            a.ml_part[pidx * 2 + 1] = Lh;
          }
        }
      }
      bar_sync(1, 128);  // lsum_s is rewritten by the next item's epilogue
    }
    if (aborted) *abort_flag = 1;
  } else if (warp < 8) {
    // ================================ loaders =================================================
    const int lw = warp - 4;
    const int64_t rowb = (int64_t)a.Hk * kD * 2;  // bytes between consecutive slots
    const int q4 = lane >> 3, c8 = lane & 7;
    uint32_t it = 0;      // tiles issued, over all items
    bool stop = false;
    for (uint32_t n = 0; !stop; ++n) {
      // every lane reads the slot; lane 0 releases it once the whole warp has
      int got = 1;
      if (lane == 0) got = mbar_wait(&item_full[n & 1], (n >> 1) & 1, a.wait_ns, a.err) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        stop = true;
        break;
      }
      mbar_wait(&item_full[n & 1], (n >> 1) & 1, a.wait_ns, a.err);  // completed: acquires at once
      const DecItem w = ring[n & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[n & 1]);
      if (w.ntiles == 0) break;
      const char *kg = static_cast<const char *>(a.k_layer) + (int64_t)w.g * kD * 2;
      const char *vg = static_cast<const char *>(a.v_layer) + (int64_t)w.g * kD * 2;
      // slots of this lane's token in the next two tiles, each read two tiles before its copies
      int64_t nxt = -1, nxt2 = -1;
      {
        const int64_t t0 = w.j0 + lw * 32 + lane;
        if (t0 < w.j1) nxt = __ldg(w.row + t0);
        if (w.ntiles > 1 && t0 + kTok < w.j1) nxt2 = __ldg(w.row + t0 + kTok);
      }
      // whether this warp's 32 tokens of a tile are two runs of consecutive slots (whole pages)
      auto runs = [&](int64_t s) {
        const int64_t s_first = __shfl_sync(0xffffffffu, s, lane & 16);
        return __all_sync(0xffffffffu, a.use_tma && s >= 0 && s == s_first + (lane & 15));
      };
      for (int j = 0; j < w.ntiles; ++j, ++it) {
        const int st = it % kStages;
        const int64_t tok0 = w.j0 + (int64_t)j * kTok;
        int64_t my = nxt;  // slot of token tok0 + lw*32 + lane (or -1 past the chunk)
        nxt = nxt2;
        {
          const int64_t tn = tok0 + 2 * kTok + lw * 32 + lane;
          nxt2 = (j + 2 < w.ntiles && tn < w.j1) ? (int64_t)__ldg(w.row + tn) : -1;
        }
        if (my >= a.size || (my < 0 && tok0 + lw * 32 + lane < w.j1)) {
          raise_error(a.err, ASTR_DEVERR_SLOT);
          my = -1;
        }
        // when both 16-token halves of this warp's 32 tokens are page runs, they come as TMA
        // boxes, one per 64-element half of K and of V; otherwise all 32 tokens take the 16-byte
        // cp.async path
        const bool boxes = runs(my);
        // Warm L2 with the next tile's rows of this lane's token while this tile waits for its
        // stage: a plain prefetch holds no register, shared memory or TMA slot, so the boxes of
        // the next tile find their rows on chip (measured on GB300, 256 requests on 16-token
        // pages: +2.6 %). Only after a tile that came as boxes: where every lane issues 16-byte
        // copies, the extra requests slow the gather (one-token pages: -5 %).
        if (boxes && nxt >= 0 && nxt < a.size) {
          const char *kr = kg + nxt * rowb, *vr = vg + nxt * rowb;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(kr) : "memory");
          asm volatile("prefetch.global.L2 [%0];" ::"l"(vr) : "memory");
          asm volatile("prefetch.global.L2 [%0];" ::"l"(kr + 128) : "memory");
          asm volatile("prefetch.global.L2 [%0];" ::"l"(vr + 128) : "memory");
        }
        int ok = 1;
        if (lane == 0) {
          if (it >= kStages) ok = mbar_wait(&empty[st], ((it / kStages) - 1) & 1, a.wait_ns, a.err);
          if (*abort_flag) ok = 0;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
        const uint32_t kst = sbase + kOffK + st * kTileBytes;
        const uint32_t vst = sbase + kOffV + st * kTileBytes;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], boxes ? 4u * 4096u : 0u);
        __syncwarp();  // the bytes are expected before any box can land
        if (boxes) {
          if ((lane & 15) == 0) {
            const int t0 = lw * 32 + (lane & 16);  // first token of the run within the tile
            const int y = a.layer_row0 + (int)my;
            for (int hf = 0; hf < 2; ++hf) {
              tc::tma_load_2d(kst + hf * kBlockBytes + t0 * 128, &k16, w.g * kD + hf * 64, y, &full[st]);
              tc::tma_load_2d(vst + hf * kBlockBytes + t0 * 128, &v16, w.g * kD + hf * 64, y, &full[st]);
            }
          }
        } else {
          // Eight lanes per token row, two 16-byte chunks each (c8 and c8 + 8, one in each
          // 64-element half): four whole rows per copy instruction. Lanes 8q .. 8q + 7 copy the
          // rows of tokens 8q .. 8q + 7 of the warp's 32, whose slots (checked above to lie in
          // [0, size) or be -1) they read back from shared memory as two 16-byte vectors; the
          // buffer alternates by tile, so one warp barrier orders each tile's writes and reads.
          // Measured on GB300 (one-token pages): 76.1 us, against 77.4 with the slots gathered
          // by eight shuffles, 79.7 with one chunk of 16 rows per lane (16 shuffles) and 85.1
          // with four lanes per row.
          int32_t *sx = reinterpret_cast<int32_t *>(smem + kOffSlots) + lw * 64 + (it & 1) * 32;
          sx[lane] = (int32_t)my;
          __syncwarp();
          const int4 s0 = *reinterpret_cast<const int4 *>(sx + q4 * 8);
          const int4 s1 = *reinterpret_cast<const int4 *>(sx + q4 * 8 + 4);
          const int32_t sl[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int t = lw * 32 + q4 * 8 + jj;  // token within the tile
            const uint32_t off = tc::sw128_chunk_offset(t, c8, kBlockBytes);
            const bool v = sl[jj] >= 0;
            const int64_t go = v ? (int64_t)sl[jj] * rowb + c8 * 16 : 0;
            tc::cp_async16(kst + off, kg + go, v ? 16u : 0u);
            tc::cp_async16(kst + off + kBlockBytes, kg + go + 128, v ? 16u : 0u);
            tc::cp_async16(vst + off, vg + go, v ? 16u : 0u);
            tc::cp_async16(vst + off + kBlockBytes, vg + go + 128, v ? 16u : 0u);
          }
        }
        tc::cp_async_arrive_noinc(&full[st]);
      }
    }
    tc::cp_async_wait_all();
    if (stop && lane == 0) {
      // stopped early: boxes still in flight land before the block can go away
      for (uint32_t u = it > kStages ? it - kStages : 0; u < it; ++u)
        mbar_wait(&full[u % kStages], (u / kStages) & 1, kDrainLimitNs, a.err);
    }
  } else if (warp == 9) {
    // ============ scheduler: claims items, publishes them, stages their query rows ============
    // Work positions are split-major (every request's first chunk before any second one) and,
    // within a split, follow the requests' seq_len ranks, so the long chunks go first and the
    // run ends on the short ones. Block c starts at position c; each further position comes
    // from the counter once the other roles have taken the block's previous item.
    const int64_t per_split = (int64_t)a.B * a.Hk;
    auto claim = [&]() -> int64_t {
      unsigned got = 0;
      if (lane == 0) got = atomicAdd(&a.sched[0], 1u);
      return (int64_t)gridDim.x + __shfl_sync(0xffffffffu, got, 0);
    };
    uint32_t n = 0;
    bool ok = true;
    int64_t pos = blockIdx.x;
    while (ok) {
      DecItem w;
      w.ntiles = 0;
      while (pos < a.n_items) {
        w.split = (int)(pos / per_split);
        const int rest = (int)(pos % per_split);
        w.b = ranked ? order[rest / a.Hk] : rest / a.Hk;
        w.g = rest % a.Hk;
        w.L = __ldg(a.seq_lens + w.b);
        bool good = true;
        if (w.L < 1 || w.L > a.max_len || w.L > a.max_ctx) {
          if (w.split == 0 && w.g == 0 && lane == 0) raise_error(a.err, ASTR_DEVERR_LEN);
          good = false;
        }
        w.j0 = (int64_t)w.split * a.chunk;
        if (good && w.j0 >= w.L) good = false;  // this request has no such chunk
        const int r = good ? __ldg(a.rpi + w.b) : 0;
        if (good && (r < 0 || r >= a.num_reqs)) {
          if (w.split == 0 && w.g == 0 && lane == 0) raise_error(a.err, ASTR_DEVERR_ROW);
          good = false;
        }
        if (good) {
          w.j1 = w.j0 + a.chunk < w.L ? w.j0 + a.chunk : w.L;
          w.row = a.r2t + (int64_t)r * a.max_ctx;
          w.ntiles = (int)((w.j1 - w.j0 + kTok - 1) / kTok);
          break;
        }
        pos = claim();
      }
      // with RoPE folded in: the query position and, for the chunk that ends at the newest
      // position, that token's rotated key and its value written into its cache slot before the
      // item is published, so the loaders' copies of that tile read them
      bool qrot = false;
      const float *cs_row = nullptr;
      if (a.fused && w.ntiles > 0) {
        const int p = __ldg(a.pos + w.b);
        const int32_t sl = __ldg(a.loc + w.b);
        const bool pos_ok = p >= 0 && p < a.freqs_max_len;
        const bool slot_ok = sl >= 0 && (int64_t)sl < a.size;
        if (!(pos_ok && slot_ok) && lane == 0)
          raise_error(a.err, (pos_ok ? 0u : ASTR_DEVERR_POS) | (slot_ok ? 0u : ASTR_DEVERR_SLOT));
        qrot = pos_ok;
        cs_row = a.freqs + (int64_t)p * kD;
        if (pos_ok && slot_ok && w.j1 == w.L && lane < 16) {
          const int e0 = lane * 8;
          float cs[8], x[8], y[8];
          const float4 f0 = __ldg(reinterpret_cast<const float4 *>(cs_row + e0));
          const float4 f1 = __ldg(reinterpret_cast<const float4 *>(cs_row + e0) + 1);
          cs[0] = f0.x; cs[1] = f0.y; cs[2] = f0.z; cs[3] = f0.w;
          cs[4] = f1.x; cs[5] = f1.y; cs[6] = f1.z; cs[7] = f1.w;
          const int64_t src = ((int64_t)w.b * a.Hk + w.g) * kD + e0;
          const int64_t dst = ((int64_t)sl * a.Hk + w.g) * kD + e0;
          const uint4 kr = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.k_new) + src));
          x[0] = bf16_lo(kr.x); x[1] = bf16_hi(kr.x); x[2] = bf16_lo(kr.y); x[3] = bf16_hi(kr.y);
          x[4] = bf16_lo(kr.z); x[5] = bf16_hi(kr.z); x[6] = bf16_lo(kr.w); x[7] = bf16_hi(kr.w);
          rotate4(x, cs, y);
          uint4 ko;
          ko.x = pack_bf16x2_rn(y[0], y[1]);
          ko.y = pack_bf16x2_rn(y[2], y[3]);
          ko.z = pack_bf16x2_rn(y[4], y[5]);
          ko.w = pack_bf16x2_rn(y[6], y[7]);
          *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(const_cast<void *>(a.k_layer)) + dst) = ko;
          *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(const_cast<void *>(a.v_layer)) + dst) =
              __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.v_new) + src));
          // the loaders may read the row by TMA (async proxy) or cp.async
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence_block();
        }
        __syncwarp();
      }
      // publish into slot n & 1 once every reader has taken publication n - 2
      int fine = 1;
      if (lane == 0) {
        if (n >= 2) fine = sleepy_wait(&item_empty[n & 1], ((n >> 1) - 1) & 1, a.wait_ns, a.err);
        if (fine) {
          ring[n & 1] = w;
          mbar_arrive(&item_full[n & 1]);
        }
      }
      if (!(ok = __shfl_sync(0xffffffffu, fine, 0) != 0) || w.ntiles == 0) break;
      // the item's query rows into Q buffer n & 1 once item n - 2's last S has read it
      int qok = 1;
      if (lane == 0 && n >= 2) qok = sleepy_wait(&q_empty[n & 1], ((n >> 1) - 1) & 1, a.wait_ns, a.err);
      if (!(ok = __shfl_sync(0xffffffffu, qok, 0) != 0)) break;
      {
        const uint16_t *qh = static_cast<const uint16_t *>(a.q) + ((int64_t)w.b * a.H + w.g * G) * kD;
        unsigned char *qs = smem + kOffQ + (n & 1) * 4096;
        for (int k = lane; k < G * 16; k += 32) {
          const int h = k >> 4, cc = k & 15;
          uint4 v = __ldg(reinterpret_cast<const uint4 *>(qh + h * kD) + cc);
          if (qrot) {  // RoPE on the query, rounded as the separate rotate + write call does
            float cs[8], x[8], y[8];
            const float4 f0 = __ldg(reinterpret_cast<const float4 *>(cs_row + cc * 8));
            const float4 f1 = __ldg(reinterpret_cast<const float4 *>(cs_row + cc * 8) + 1);
            cs[0] = f0.x; cs[1] = f0.y; cs[2] = f0.z; cs[3] = f0.w;
            cs[4] = f1.x; cs[5] = f1.y; cs[6] = f1.z; cs[7] = f1.w;
            x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
            x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
            rotate4(x, cs, y);
            v.x = pack_bf16x2_rn(y[0], y[1]);
            v.y = pack_bf16x2_rn(y[2], y[3]);
            v.z = pack_bf16x2_rn(y[4], y[5]);
            v.w = pack_bf16x2_rn(y[6], y[7]);
          }
          *reinterpret_cast<uint4 *>(qs + tc::sw128_chunk_offset(h, cc, 2048)) = v;
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[n & 1]);
      }
      // claim the next item once this one is taken, so a block holds at most one in reserve
      int taken = 1;
      if (lane == 0) taken = sleepy_wait(&item_empty[n & 1], (n >> 1) & 1, a.wait_ns, a.err);
      if (!(ok = __shfl_sync(0xffffffffu, taken, 0) != 0)) break;
      ++n;
      pos = claim();
    }
    if (!ok) *abort_flag = 1;
  } else {
    // ============ MMA issuer: warp 8, converged; one elected lane issues each MMA ============
    // Descriptors are built once per buffer and stepped by constants (16-byte units): an MMA
    // loop run by one lane with two descriptors built per MMA measured about 120 cycles an
    // issue, most of a tile's time on one-token pages.
    {
      auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        const bool got = !*abort_flag && mbar_wait(bar, parity, a.wait_ns, a.err);
        return __all_sync(0xffffffffu, got);
      };
      const uint64_t k_desc = tc::desc_sw128(sbase + kOffK, 16, 1024);           // K stage 0 (A of S^T)
      const uint64_t q_desc = tc::desc_sw128(sbase + kOffQ, 16, 1024);           // Q buffer 0 (B of S^T)
      const uint64_t v_desc = tc::desc_sw128(sbase + kOffV, kBlockBytes, 1024);  // V stage 0, MN-major
      // P^T buffer 0 (B, MN-major, 32-byte swizzling: 8-token groups of 256 bytes)
      const uint64_t p_desc = (tc::desc_sw128(sbase + kOffP, 256, 256) & ~((uint64_t)7 << 61)) | ((uint64_t)6 << 61);
      constexpr uint64_t kStageStep = kTileBytes >> 4, kBufStep = 4096 >> 4;
      // O^T += V^T P^T for tile i (P^T from buffer i & 1) into O buffer ob; `first` starts it
      auto pv = [&](uint32_t i, int ob, bool first) -> bool {
        const int sb = i & 1, st = i % kStages;
        if (!wait(&p_full[sb], (i >> 1) & 1)) return false;
        tc::fence_after_sync();
        tc::fence_proxy_async_smem();
        const uint64_t vd = v_desc + (uint64_t)st * kStageStep, pd = p_desc + (uint64_t)sb * kBufStep;
#pragma unroll
        for (int ks = 0; ks < kTok / 16; ++ks)
          tc::mma_ss_elect(tO0 + ob * 16, vd + (uint64_t)ks * (2048 >> 4),
                           pd + (uint64_t)ks * (512 >> 4), kIdescPV,
                           (!first || ks > 0) ? 1u : 0u);
        tc::mma_commit_elect(&empty[st]);
        tc::mma_commit_elect(&pv_done[sb]);
        return true;
      };
      bool ok = true;
      uint32_t it = 0;                 // tiles issued, over all items
      bool have_prev = false;          // a tile whose P.V is still to be issued
      int prev_ob = 0;
      bool prev_first = false;
      for (uint32_t n = 0; ok; ++n) {
        DecItem w;
        if (!wait(&item_full[n & 1], (n >> 1) & 1)) {
          ok = false;
          break;
        }
        w = ring[n & 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[n & 1]);
        if (w.ntiles == 0) break;
        const int qb = n & 1, ob = n & 1;
        if (!wait(&q_full[qb], (n >> 1) & 1)) {
          ok = false;
          break;
        }
        const uint64_t qd = q_desc + (uint64_t)qb * kBufStep;
        for (int j = 0; j < w.ntiles && ok; ++j, ++it) {
          const int st = it % kStages, sb = it & 1;
          if (!wait(&full[st], (it / kStages) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          tc::fence_proxy_async_smem();
          const uint64_t kd = k_desc + (uint64_t)st * kStageStep;
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks)
            tc::mma_ss_elect(tS0 + sb * 16, kd + (uint64_t)((ks >> 2) * (kBlockBytes >> 4) + (ks & 3) * 2),
                             qd + (uint64_t)((ks >> 2) * (2048 >> 4) + (ks & 3) * 2), kIdescQK, ks > 0 ? 1u : 0u);
          tc::mma_commit_elect(&s_full[sb]);
          if (j + 1 == w.ntiles) tc::mma_commit_elect(&q_empty[qb]);  // the item's last read of Q
          if (have_prev && !pv(it - 1, prev_ob, prev_first)) {
            ok = false;
            break;
          }
          // this tile's P.V goes in after the next tile's S; the first one of an item waits for
          // the epilogue of the item two back to have read the O buffer
          if (j == 0 && n >= 2 && !wait(&o_free[ob], ((n >> 1) - 1) & 1)) {
            ok = false;
            break;
          }
          have_prev = true;
          prev_ob = ob;
          prev_first = j == 0;
        }
        // the item's last P.V goes in now rather than after the next item's first S: its stage
        // frees sooner and the epilogue, which waits for it, overlaps the next item's loads
        if (ok && have_prev) {
          ok = pv(it - 1, prev_ob, prev_first);
          have_prev = false;
        }
      }
      if (ok && have_prev && !pv(it - 1, prev_ob, prev_first)) ok = false;
      if (!ok) *abort_flag = 1;
      tc::mma_commit_elect(drain);  // nothing may still be in flight when TMEM is freed
      mbar_wait(drain, 0, kDrainLimitNs, a.err);
      __syncwarp();
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 64);
  }
  if (tid == 0) {
    // the last block to finish resets the counters for the next launch that uses them (every
    // block has made its last claim before its __syncthreads above)
    __threadfence();
    if (atomicAdd(&a.sched[1], 1u) == gridDim.x - 1) {
      atomicExch(&a.sched[0], 0u);
      atomicExch(&a.sched[1], 0u);
    }
  }
}

template <int G>
cudaError_t run_g(const DecArgs &a, const CUtensorMap &k16, const CUtensorMap &v16, int64_t grid,
                  cudaStream_t s) {
  auto k = decode_tc_kernel<G>;
  static std::atomic<uint64_t> attr_devices{0};
  cudaError_t e = raise_smem_limit_once(reinterpret_cast<const void *>(k), kSmemBytes, attr_devices);
  if (e != cudaSuccess) return e;
  if (grid > 0) k<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(a, k16, v16);
  return cudaGetLastError();
}

}  // namespace

// Work counters: each launch takes the next of kSchedSlots pairs, so launches that overlap
// on different streams use different ones unless kSchedSlots of them run at once. A launch's
// last block puts its pair back to zero. The persistent decode and prefill kernels share them.
__device__ unsigned g_sched[2 * kSchedSlots];
constexpr int kMaxDevices = 64;
std::mutex g_sched_mutex;
unsigned *g_sched_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::atomic<unsigned> g_sched_next{0};

cudaError_t sched_slot(unsigned **out, int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(g_sched_mutex);
    if (!g_sched_ptr[dev]) {
      void *p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_sched)) != cudaSuccess) return e;
      if ((e = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
      g_sched_ptr[dev] = static_cast<unsigned *>(p);
    }
  }
  *out = g_sched_ptr[dev] + 2 * (g_sched_next.fetch_add(1) % kSchedSlots);
  *sms = g_sms[dev];
  return cudaSuccess;
}

cudaError_t device_sm_count(int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_sched_mutex);
  if (!g_sms[dev] && (e = cudaDeviceGetAttribute(&g_sms[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  *sms = g_sms[dev];
  return cudaSuccess;
}

bool tc_decode_supported(int dtype, int head_dim, int group) {
  return dtype == ASTR_BF16 && head_dim == kD &&
         (group == 1 || group == 2 || group == 4 || group == 8 || group == 16);
}

int tc_decode_tile_tokens() { return kTok; }
int tc_decode_ranked_batch_max() { return kSortMax; }

cudaError_t launch_tc_decode(const astr_kv_cache &kv, int32_t layer_id, const void *q,
                             int32_t n_heads, const SimtAttnPlan &plan, cudaStream_t stream,
                             const DecodeRope *rope) {
  DecArgs a;
  a.fused = rope != nullptr;
  a.k_new = rope ? rope->k_new : nullptr;
  a.v_new = rope ? rope->v_new : nullptr;
  a.freqs = rope ? rope->freqs : nullptr;
  a.pos = rope ? rope->position_ids : nullptr;
  a.loc = rope ? kv.out_cache_loc : nullptr;
  a.freqs_max_len = rope ? rope->freqs_max_len : 0;
  const int64_t layer_elems = (int64_t)layer_id * kv.size * kv.n_kv_heads * kv.head_dim;
  a.q = q;
  a.k_layer = static_cast<const char *>(kv.k_buffer) + layer_elems * 2;
  a.v_layer = static_cast<const char *>(kv.v_buffer) + layer_elems * 2;
  a.r2t = kv.req_to_token;
  a.rpi = kv.req_pool_indices;
  a.seq_lens = kv.seq_lens;
  a.o_part = kv.decode_o_part;
  a.ml_part = kv.decode_ml_part;
  a.out = kv.decode_out;
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
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kv.head_dim));
  // the pool as a [n_layers * size, Hk * D] tensor for 16-row boxes; TMA row coordinates are
  // 32-bit, so larger pools take the cp.async path only
  CUtensorMap k16, v16;
  memset(&k16, 0, sizeof k16);
  memset(&v16, 0, sizeof v16);
  const uint64_t rows = (uint64_t)kv.n_layers * kv.size;
  const uint64_t cols = (uint64_t)kv.n_kv_heads * kv.head_dim;
  a.use_tma = rows < (uint64_t(1) << 31) && encode_map_bf16_2d(&k16, kv.k_buffer, rows, cols, 64, 16) &&
              encode_map_bf16_2d(&v16, kv.v_buffer, rows, cols, 64, 16);
  a.layer_row0 = a.use_tma ? (int32_t)((int64_t)layer_id * kv.size) : 0;
  a.n_items = (int64_t)kv.batch * plan.n_splits * kv.n_kv_heads;
  int sms = 0;
  cudaError_t se = sched_slot(&a.sched, &sms);
  if (se != cudaSuccess) return se;
  // one block per SM: the blocks claim work items until none are left
  const int64_t grid = a.n_items < sms ? a.n_items : sms;
  const int G = n_heads / kv.n_kv_heads;
  cudaError_t e;
  switch (G) {
    case 1: e = run_g<1>(a, k16, v16, grid, stream); break;
    case 2: e = run_g<2>(a, k16, v16, grid, stream); break;
    case 4: e = run_g<4>(a, k16, v16, grid, stream); break;
    case 8: e = run_g<8>(a, k16, v16, grid, stream); break;
    case 16: e = run_g<16>(a, k16, v16, grid, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  if (plan.n_splits > 1) return launch_split_merge(kv, n_heads, plan, stream);
  return cudaSuccess;
}

}  // namespace astr
