// Varlen causal prefill on the tcgen05 tensor cores, persistent and pipelined (bf16, head_dim
// 128, query groups of an even size).
//
// AstrAI inference guide, "Attention Backend": a ragged-batch prefill reading K/V straight
// from the flat pool through req_to_token, each request addressed by qo_indptr / kv_indptr;
// "KVCache System": 128-row Q tiles named by q_tile_to_batch / q_tile_to_index, and prefill
// resumed right after a cached prefix. AstrAI internals, "Autoregression & Causal Masking":
// query position i attends to keys j <= i (positions are absolute: row i of a request with
// prefix P sits at P + i).
//
// A work item is one 128-row Q tile for a pair of query heads of one KV group, so every K/V
// tile staged feeds two heads. One block per SM claims items, most KV tiles first, from a
// counter until none are left. The roles:
//  * warps 8 and 10 (loaders; warp 8 also claims and publishes the items through a two-slot
//    ring) stream each item's two Q tiles and then its K and V tiles through a three-slot ring
//    in the order the tensor core takes them (K0, K1, V0, K2, V1, ..., V_last): one TMA box per
//    run of 16 keys with consecutive slots (a page), 16-byte cp.async copies for the other keys,
//    zero fill past the request. A warp issues TMA copies at a limited rate, so the boxes of a
//    tile are split between the two warps;
//  * warps 9 and 11 issue the MMAs of head 0 and head 1 (warp 9 also holds all 512 TMEM
//    columns, S0 | S1 | O0 | O1): S(j+1) = Q K_{j+1}^T as soon as the head's softmax has read
//    S(j) out of TMEM, so the next scores are computed while the current tile's softmax runs,
//    and O += P(j) V_j once P(j) is in shared memory. Each warp runs converged and one elected
//    lane issues, with descriptors built once per buffer;
//  * warps 0-3 and 4-7 are the softmax of head 0 and head 1, one thread per row: the row max
//    over all 128 scores of a tile, the reference max raised only when the row max exceeds it
//    by 2^8 (O is then rescaled in TMEM after the previous P.V has completed), exp2 of the
//    scaled scores written as bf16 P into shared memory in the 128-byte-swizzled K-major
//    layout, and after an item's last tile the epilogue: O normalised, TMEM released to the
//    next item at once, and whole tiles sent out as two TMA boxes staged in the P buffer. The
//    first thread of each head also hands the ring slots and the Q buffer back to the loaders
//    once it has seen both MMAs that read them complete.
// KV tiles beyond the diagonal of a Q tile are skipped; the mask applies only to tiles that
// cross the diagonal or the end of the request. Every barrier phase follows counters that run
// on across items. All waits are bounded (and suspend the waiting warp): a wait that runs out
// raises ASTR_DEVERR_TIMEOUT, and the block stops, lets its copies and MMAs land and returns.
#include <math.h>

#include <atomic>

#include "astr_internal.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace astr {

namespace {

constexpr int kRows = 128;              // Q tile rows (M)
constexpr int kKeys = 128;              // keys per KV tile (N of S, K of P.V)
constexpr int kD = 128;
constexpr int kTile = kRows * kD * 2;   // 32 KB: one Q, P, K or V tile
constexpr int kBlk = kRows * 128;       // 16 KB: one 64-element half
constexpr int kThreads = 384;           // 8 softmax warps, 2 loader warps, 2 MMA warps
constexpr int kLoaders = 2;             // warps 8 and 10
constexpr int kRing = 3;                // K/V ring slots
constexpr float kLazyRescale = 8.0f;

constexpr int kOffQ = 0;                          // Q_0, Q_1
constexpr int kOffP = kOffQ + 2 * kTile;          // P_0, P_1 (also the output staging)
constexpr int kOffKV = kOffP + 2 * kTile;         // K/V ring
constexpr int kOffBar = kOffKV + kRing * kTile;
constexpr int kNumBars = 32;
// barrier indices in the array at kOffBar (each 8 bytes)
constexpr int kBarItemFull = 0, kBarItemEmpty = 2, kBarQFull = 4, kBarQEmpty = 5, kBarKvFull = 6,
              kBarKvEmpty = 9, kBarSFull = 12, kBarSFree = 14, kBarPFull = 16, kBarPFree = 18,
              kBarOFree = 22, kBarStageFull = 24, kBarStageFree = 26, kBarDrain = 28;
constexpr int kOffItem = kOffBar + kNumBars * 8;  // two published items
constexpr int kOffMisc = kOffItem + 2 * 64;
constexpr int kSmemBytes = kOffMisc + 32 + 1024;  // + alignment slack

constexpr uint32_t kIdescQK = tc::idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, false, true);

struct PipeArgs {
  const int32_t *r2t;
  const int32_t *rpi;
  const int32_t *qo_indptr;
  const int32_t *kv_indptr;
  const int32_t *tile_b;
  const int32_t *tile_i;
  const void *k_layer;
  const void *v_layer;
  void *out;
  unsigned *sched;  // [0]: claims past each block's first item, [1]: blocks done
  int64_t size;
  int64_t n_rows;   // packed q rows
  int64_t n_items;  // num_tiles * head pairs
  uint64_t wait_ns;
  uint32_t *err;
  int32_t layer_row0;  // first row of this layer in the [n_layers * size, Hk * D] view
  int32_t num_reqs, max_ctx;
  int32_t H, Hk, B;
  int32_t num_tiles;
  int32_t tma_out;  // whole tiles leave through a TMA map of `out`
  float scale_log2;
};

// an item as the scheduler publishes it
struct PipeItem {
  int64_t q0;         // first packed row of the request
  int64_t r0;         // first request-local row of the tile
  int64_t Pb;         // cached prefix of the request
  int64_t Kb;         // kv length of the request
  int32_t rows_here;  // rows of the tile inside the request
  int32_t nkv;        // KV tiles to visit (0: no more items)
  int32_t h0;         // first query head of the pair
  int32_t rq;         // the request's row of req_to_token
  int32_t col0;       // the KV head's first column in the [rows, Hk * D] view
  int32_t pad;
};
static_assert(2 * sizeof(PipeItem) <= kOffMisc - kOffItem, "two published items");

__global__ void __launch_bounds__(kThreads, 1)
    prefill_pipe_kernel(const PipeArgs a, const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap k16, const __grid_constant__ CUtensorMap v16,
                        const __grid_constant__ CUtensorMap omap) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *item_full = bars + kBarItemFull;    // [2] scheduler -> all roles (1 arrival)
  uint64_t *item_empty = bars + kBarItemEmpty;  // [2] 8 softmax warps, loader warp 10, 2 MMA threads
  uint64_t *q_full = bars + kBarQFull;          // TMA (transaction bytes)
  uint64_t *q_empty = bars + kBarQEmpty;        // one arrival per head once the item's last S has completed
  uint64_t *kv_full = bars + kBarKvFull;        // [3] per loader warp: 32 lanes (cp.async) + one expect-tx
  uint64_t *kv_empty = bars + kBarKvEmpty;      // [3] one arrival per head once its MMAs on the tile completed
  uint64_t *s_full = bars + kBarSFull;          // [2] per head, MMA commit
  uint64_t *s_free = bars + kBarSFree;          // [2] per head, 128 arrivals (scores read out of TMEM)
  uint64_t *p_full = bars + kBarPFull;          // [2] per head, 128 arrivals (P in shared memory)
  uint64_t *p_free = bars + kBarPFree;          // [2] per head, MMA commit after P.V
  uint64_t *o_free = bars + kBarOFree;          // [2] per head, 128 arrivals (O read out of TMEM)
  uint64_t *stage_full = bars + kBarStageFull;  // [2] per head, 128 arrivals (output tile staged)
  uint64_t *stage_free = bars + kBarStageFree;  // [2] per head, 1 arrival (the TMA store has read it)
  uint64_t *drain = bars + kBarDrain;           // [2] per MMA thread
  PipeItem *items = reinterpret_cast<PipeItem *>(smem + kOffItem);
  // per ring slot: c + 1 when fill c of the slot holds rows written by cp.async (generic
  // proxy), which the tensor core may read only after a proxy fence
  volatile uint32_t *slot_generic = reinterpret_cast<volatile uint32_t *>(smem + kOffMisc + 16);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], 8 + (kLoaders - 1) + 2);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
      mbar_init(&p_full[i], 128);
      mbar_init(&p_free[i], 1);
      mbar_init(&o_free[i], 128);
      mbar_init(&stage_full[i], 128);
      mbar_init(&stage_free[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 2);  // one arrival per head
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&kv_full[i], 33 * kLoaders);
      mbar_init(&kv_empty[i], 2);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int i = 0; i < kRing; ++i) slot_generic[i] = 0;
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ===================== softmax and epilogue: head h, row r ==================================
    const int h = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + h * 128 + lane_base;
    const uint32_t tO = tmem + 256 + h * 128 + lane_base;
    const uint32_t poff = kOffP + h * kTile;
    // The softmax addresses its barriers and its P tile through 32-bit shared-window addresses:
    // one base register plus constants, which leaves more registers to the 128 scores of a row.
    const uint32_t sbar = sbase + kOffBar;
    auto bar = [&](int i) -> uint32_t { return sbar + 8u * (uint32_t)i; };
    // this row's 128-byte line of the P tile with the row's swizzle in the chunk bits; the tile is
    // 1024-byte aligned, so chunk c of the row is at (prow ^ (c % 8) * 16) + (c / 8) * kBlk
    const uint32_t prow = sbase + poff + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u +
                          ((uint32_t)(r & 7) << 4);
    uint32_t n = 0, T = 0, ns = 0;  // items, tiles, staged stores
    uint32_t cs = 0;                // K/V ring fills before the current item
    bool staged = false;            // a TMA store may still be reading the P buffer
    // a ring slot or the Q buffer is free once both heads' MMAs on it have completed: the
    // first thread of each head arrives when it sees that completion
    auto release = [&](uint32_t b) {
      if (r == 0) mbar_arrive(b);
    };
    bool aborted = false;
    // a wait whose outcome is the same for the whole warp (the TMEM loads and stores that
    // follow are warp-collective)
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
      const bool got = mbar_wait_sleep(b, parity, a.wait_ns, a.err);
      return __all_sync(0xffffffffu, got);
    };
    while (!aborted) {
      if (!wait_warp(bar(kBarItemFull + (n & 1)), (n >> 1) & 1)) {
        aborted = true;
        break;
      }
      const PipeItem it = items[n & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarItemEmpty + (n & 1)));
      if (it.nkv == 0) break;
      // keys [0, lim_row) are visible to this row; the tiles from j_mask on need masking (the
      // first tile that crosses the diagonal or the end of the request, and all after it)
      const int32_t lim_row = (int32_t)(it.Pb + it.r0 + r + 1 < it.Kb ? it.Pb + it.r0 + r + 1 : it.Kb);
      const int64_t j_diag = it.Pb + it.r0 >= kKeys - 1 ? (it.Pb + it.r0 - (kKeys - 1)) / kKeys + 1 : 0;
      const int64_t j_end = it.Kb >= kKeys ? (it.Kb - kKeys) / kKeys + 1 : 0;
      const int32_t j_mask = (int32_t)(j_diag < j_end ? j_diag : j_end);
      float m = -INFINITY, l = 0.f;
      // the ring carries K0, K1, V0, K2, V1, ..., V_{nkv-1}: K_j is fill cs + 2j - 1 (K_0: cs),
      // V_j is fill cs + 2j + 2 (the last V: cs + 2 nkv - 1)
      for (int j = 0; j < it.nkv; ++j, ++T) {
        if (!wait_warp(bar(kBarSFull + h), T & 1)) {
          aborted = true;
          break;
        }
        tc::fence_after_sync();
        release(bar(kBarKvEmpty + ((cs + (j == 0 ? 0 : 2 * j - 1))) % kRing));
        if (j + 1 == it.nkv) release(bar(kBarQEmpty));
        uint32_t sv[128];
        tc::tmem_ld128(tS, sv);
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        mbar_arrive(bar(kBarSFree + h));  // the tensor core may write the next S here now
        if (j >= j_mask) {
          const int32_t lim = lim_row - j * kKeys;
          const int nvalid = lim < 0 ? 0 : (lim > kKeys ? kKeys : lim);
#pragma unroll
          for (int k = 0; k < kKeys; ++k) sv[k] = k < nvalid ? sv[k] : 0xFF800000u;  // -inf
        }
        float mxa = -INFINITY, mxb = -INFINITY, mxc = -INFINITY, mxd = -INFINITY;
#pragma unroll
        for (int k = 0; k < kKeys; k += 8) {
          mxa = fmax3(mxa, __uint_as_float(sv[k]), __uint_as_float(sv[k + 1]));
          mxb = fmax3(mxb, __uint_as_float(sv[k + 2]), __uint_as_float(sv[k + 3]));
          mxc = fmax3(mxc, __uint_as_float(sv[k + 4]), __uint_as_float(sv[k + 5]));
          mxd = fmax3(mxd, __uint_as_float(sv[k + 6]), __uint_as_float(sv[k + 7]));
        }
        const float mx = fmax3(mxa, mxb, fmaxf(mxc, mxd)) * a.scale_log2;
        const float m_new = (mx > m + kLazyRescale) ? mx : m;
        const float alpha = ex2_approx(m - m_new);
        const bool rescale = j > 0 && __any_sync(0xffffffffu, m_new != m);
        l *= alpha;
        m = m_new;
        // the P buffer is free (and O settled) once the previous P.V has completed; for an
        // item's first tile, once the last output staged in the buffer has been read
        if (j > 0) {
          if (!wait_warp(bar(kBarPFree + h), (T - 1) & 1)) {
            aborted = true;
            break;
          }
          tc::fence_after_sync();
          release(bar(kBarKvEmpty + ((cs + 2 * j)) % kRing));  // V_{j-1}
        } else if (staged) {
          if (r == 0) {
            tc::bulk_wait_read_all();
            mbar_arrive(bar(kBarStageFree + h));
          }
          if (!wait_warp(bar(kBarStageFree + h), (ns - 1) & 1)) {
            aborted = true;
            break;
          }
          staged = false;
        }
        // P = exp2(score * scale - m) in bf16, 8 keys (one 16-byte chunk) at a time
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 nm2 = make_float2(-m, -m);
        float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          uint32_t pk[4];
#pragma unroll
          for (int k = 0; k < 8; k += 2) {
            const float2 x = ffma2(make_float2(__uint_as_float(sv[8 * c + k]), __uint_as_float(sv[8 * c + k + 1])),
                                   sc2, nm2);
            const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);  // ex2(-inf) = 0
            sum2[k >> 1] = fadd2(sum2[k >> 1], make_float2(p0, p1));
            pk[k >> 1] = pack_bf16x2_rn(p0, p1);
          }
          st_shared_v4((prow ^ (uint32_t)((c & 7) << 4)) + (uint32_t)(c >> 3) * kBlk, pk[0], pk[1], pk[2], pk[3]);
        }
        const float2 s01 = fadd2(sum2[0], sum2[1]), s23 = fadd2(sum2[2], sum2[3]);
        l += (s01.x + s01.y) + (s23.x + s23.y);
        if (rescale) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tc::tmem_ld32(tO + c * 32, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tc::tmem_st16(tO + c * 32, o);
            tc::tmem_st16(tO + c * 32 + 16, o + 16);
          }
          tc::tmem_st_wait();
        }
        tc::fence_proxy_async_smem();  // P is read by the tensor core (async proxy)
        tc::fence_before_sync();
        mbar_arrive(bar(kBarPFull + h));
      }
      if (aborted) break;
      // ---- epilogue: O / l to bf16; whole tiles through the P buffer as two TMA boxes, a tile
      // cut by the request's end row by row (a box would overwrite the next request's rows)
      // O is complete with the item's last P.V
      if (!wait_warp(bar(kBarPFree + h), (T - 1) & 1)) {
        aborted = true;
        break;
      }
      tc::fence_after_sync();
      release(bar(kBarKvEmpty + ((cs + 2 * it.nkv - 1)) % kRing));  // V_last
      cs += 2 * it.nkv;
      const bool by_tma = a.tma_out && it.rows_here == kRows;  // uniform over the head
      const float inv = 1.f / l;
      uint16_t *orow = static_cast<uint16_t *>(a.out) + ((it.q0 + it.r0 + r) * a.H + it.h0 + h) * kD;
      const bool write = r < it.rows_here;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tO + c * 32, o);
        tc::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          uint4 w;
          w.x = pack_bf16x2_rn(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv);
          w.y = pack_bf16x2_rn(__uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
          w.z = pack_bf16x2_rn(__uint_as_float(o[k + 4]) * inv, __uint_as_float(o[k + 5]) * inv);
          w.w = pack_bf16x2_rn(__uint_as_float(o[k + 6]) * inv, __uint_as_float(o[k + 7]) * inv);
          if (by_tma)
            *reinterpret_cast<uint4 *>(smem + poff + tc::sw128_chunk_offset(r, c * 4 + (k >> 3), kBlk)) = w;
          else if (write)
            *reinterpret_cast<uint4 *>(orow + c * 32 + k) = w;
        }
      }
      tc::fence_before_sync();
      mbar_arrive(bar(kBarOFree + h));  // the next item's first P.V may overwrite O
      if (by_tma) {
        tc::fence_proxy_async_smem();
        mbar_arrive(bar(kBarStageFull + h));
        if (r == 0) {
          if (mbar_wait_sleep(bar(kBarStageFull + h), ns & 1, a.wait_ns, a.err)) {
            tc::tma_store_2d(&omap, (it.h0 + h) * kD, (int)(it.q0 + it.r0), sbase + poff);
            tc::tma_store_2d(&omap, (it.h0 + h) * kD + 64, (int)(it.q0 + it.r0), sbase + poff + kBlk);
            tc::bulk_commit();
          } else {
            aborted = true;
          }
        }
        ++ns;
        staged = true;
        aborted = __any_sync(0xffffffffu, aborted);  // keep the warp together
      }
      ++n;
    }
    if (aborted) *abort_flag = 1;
    if (r == 0) tc::bulk_wait_read_all();  // the staging buffer stays put until it is read
  } else if (warp == 8 || warp == 10) {
    // ===================== scheduler and loaders (warps 8 and 10) ===============================
    // A warp issues TMA copies at a limited rate, so the K/V boxes of a tile are spread over
    // two warps on two SM sub-partitions; warp 8 also claims and publishes the items and loads
    // Q. Each warp copies the 16-key groups g of a tile with g % 2 == its index.
    const int lw = warp == 8 ? 0 : 1;
    const int pairs = a.H / 2;
    const int G = a.H / a.Hk;
    const int64_t rowb_kv = (int64_t)a.Hk * kD * 2;
    const bool mine = ((lane >> 2) % kLoaders) == lw;
    auto claim = [&]() -> int64_t {
      unsigned got = 0;
      if (lane == 0) got = atomicAdd(&a.sched[0], 1u);
      return (int64_t)gridDim.x + __shfl_sync(0xffffffffu, got, 0);
    };
    uint32_t n = 0, c = 0, nq = 0;  // items, K/V tiles issued, Q loads issued
    bool ok = true;
    int64_t pos = blockIdx.x;
    while (ok) {
      PipeItem w;
      w.nkv = 0;
      if (lw == 0) {
        // ---- the next item with work: Q tile `ti` of request b, heads h0, h0 + 1 ----
        while (pos < a.n_items) {
          const int tile = a.num_tiles - 1 - (int)(pos / pairs);  // later tiles carry more keys
          const int h0 = (int)(pos % pairs) * 2;
          const int b = __ldg(a.tile_b + tile);
          bool good = b != -1;  // -1: an empty entry of the tile list
          uint32_t bad = 0;
          if (good && (b < 0 || b >= a.B)) bad = ASTR_DEVERR_META;
          int64_t q0 = 0, Qb = 0, Kb = 0, r0 = 0;
          if (good && !bad) {
            const int ti = __ldg(a.tile_i + tile);
            q0 = __ldg(a.qo_indptr + b);
            Qb = (int64_t)__ldg(a.qo_indptr + b + 1) - q0;
            Kb = (int64_t)__ldg(a.kv_indptr + b + 1) - __ldg(a.kv_indptr + b);
            r0 = (int64_t)ti * kRows;
            if (ti < 0 || r0 >= Qb) bad = ASTR_DEVERR_META;
            else if (Kb - Qb < 0 || Kb > a.max_ctx || q0 + Qb > a.n_rows) bad = ASTR_DEVERR_LEN;
          }
          int rq = 0;
          if (good && !bad) {
            rq = __ldg(a.rpi + b);
            if (rq < 0 || rq >= a.num_reqs) bad = ASTR_DEVERR_ROW;
          }
          if (bad) {
            if (lane == 0 && h0 == 0) raise_error(a.err, bad);
            good = false;
          }
          if (good) {
            w.q0 = q0;
            w.r0 = r0;
            w.Pb = Kb - Qb;
            w.Kb = Kb;
            w.rows_here = (int32_t)((Qb - r0) < kRows ? (Qb - r0) : kRows);
            const int64_t key_end = (w.Pb + r0 + w.rows_here) < Kb ? (w.Pb + r0 + w.rows_here) : Kb;
            w.nkv = (int32_t)((key_end + kKeys - 1) / kKeys);
            w.h0 = h0;
            w.rq = rq;
            w.col0 = (h0 / G) * kD;  // this KV head's columns in the [rows, Hk * D] view
            break;
          }
          pos = claim();
        }
        // ---- publish it (nkv = 0 tells the other roles to stop) ----
        if (lane == 0) {
          if (n >= 2 && !mbar_wait_sleep(&item_empty[n & 1], ((n >> 1) - 1) & 1, a.wait_ns, a.err)) ok = false;
          if (ok) {
            items[n & 1] = w;
            mbar_arrive(&item_full[n & 1]);
          }
        }
      } else {
        ok = mbar_wait_sleep(&item_full[n & 1], (n >> 1) & 1, a.wait_ns, a.err);
        if (ok) w = items[n & 1];
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[n & 1]);
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || w.nkv == 0) break;
      const int32_t *row = a.r2t + (int64_t)w.rq * a.max_ctx;
      const int col0 = w.col0;
      const int64_t key_end = (w.Pb + w.r0 + w.rows_here) < w.Kb ? (w.Pb + w.r0 + w.rows_here) : w.Kb;
      int64_t next_pos = -1;
      // ---- Q tiles of both heads, once the previous item's last S has read the buffer ----
      if (lw == 0) {
        if (lane == 0) {
          if (n >= 1 && !mbar_wait_sleep(q_empty, (n - 1) & 1, a.wait_ns, a.err)) ok = false;
          if (ok && *abort_flag) ok = false;
          if (ok) {
            mbar_arrive_expect_tx(q_full, 2 * kTile);
            for (int qh = 0; qh < 2; ++qh)
              for (int hf = 0; hf < 2; ++hf)
                tc::tma_load_2d(sbase + kOffQ + qh * kTile + hf * kBlk, &qmap, (w.h0 + qh) * kD + hf * 64,
                                (int)(w.q0 + w.r0), q_full);
            ++nq;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      // ---- K and V tiles: slots of a tile are read one tile ahead of its copies ----
      int sl_next[4], slK[4] = {-1, -1, -1, -1}, slV[4];
      bool vdK[4] = {false, false, false, false}, vdV[4];
      unsigned balK = 0, balV = 0;
      auto fetch_slots = [&](int j, int (&sl)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t kk = (int64_t)j * kKeys + 4 * lane + i;
          sl[i] = kk < key_end ? __ldg(row + kk) : -1;
        }
      };
      // validity and page runs of tile j's keys (a set bit per lane whose four keys continue a
      // run of consecutive slots; a 16-key group whose four bits are set is one page)
      auto classify = [&](int j, const int (&sl)[4], bool (&vd)[4]) -> unsigned {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          vd[i] = (int64_t)j * kKeys + 4 * lane + i < key_end;
          if (vd[i] && (sl[i] < 0 || (int64_t)sl[i] >= a.size)) {
            if (lw == 0) raise_error(a.err, ASTR_DEVERR_SLOT);
            vd[i] = false;
          }
        }
        const bool run4 = vd[0] && vd[1] && vd[2] && vd[3] && sl[1] == sl[0] + 1 &&
                          sl[2] == sl[1] + 1 && sl[3] == sl[2] + 1;
        const int next0 = __shfl_down_sync(0xffffffffu, sl[0], 1);
        const bool link = ((lane & 3) == 3) || (next0 == sl[3] + 1);
        return __ballot_sync(0xffffffffu, run4 && link);
      };
      // this warp's share of one K (kvsel 0) or V (kvsel 1) tile into the next ring slot
      auto issue = [&](int kvsel, const int (&sl)[4], const bool (&vd)[4], unsigned bal) -> bool {
        const int st = (int)(c % kRing);
        const unsigned runs = bal & 0x11111111u & (bal >> 1) & (bal >> 2) & (bal >> 3);
        const unsigned my_runs = runs & (lw == 0 ? 0x01010101u : 0x10101010u);  // bit 4g: group g
        // this warp's groups that are not whole pages go by cp.async
        const unsigned my_groups = lw == 0 ? 0x01010101u : 0x10101010u;
        const bool generic = (my_groups & ~runs) != 0;
        int okl = 1;
        if (lane == 0) {
          if (c >= kRing) okl = mbar_wait_sleep(&kv_empty[st], ((c / kRing) - 1) & 1, a.wait_ns, a.err);
          if (*abort_flag) okl = 0;
          if (okl && generic) slot_generic[st] = c + 1;  // published by the arrival below
          if (okl) mbar_arrive_expect_tx(&kv_full[st], (uint32_t)__popc(my_runs) * 4096u);
        }
        okl = __shfl_sync(0xffffffffu, okl, 0);
        if (!okl) return false;
        const bool group_run = ((bal >> (lane & ~3)) & 0xFu) == 0xFu;
        const int first_slot = __shfl_sync(0xffffffffu, sl[0], lane & ~3);  // the page's first slot
        const uint32_t dst = sbase + kOffKV + st * kTile;
        if (mine) {
          if (group_run) {
            if ((lane & 3) < 2) {  // one box per 64-element half, from two lanes
              const int hf = lane & 1;
              const void *m16 = kvsel ? (const void *)&v16 : (const void *)&k16;
              tc::tma_load_2d(dst + hf * kBlk + (4 * (lane & ~3)) * 128, m16, col0 + hf * 64,
                              a.layer_row0 + first_slot, &kv_full[st]);
            }
          } else {
            const char *base = static_cast<const char *>(kvsel ? a.v_layer : a.k_layer) + (int64_t)col0 * 2;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int t = 4 * lane + i;
              const char *src = base + (vd[i] ? (int64_t)sl[i] * rowb_kv : 0);
#pragma unroll
              for (int cc = 0; cc < 16; ++cc)
                tc::cp_async16(dst + tc::sw128_chunk_offset(t, cc, kBlk), src + cc * 16, vd[i] ? 16u : 0u);
            }
          }
        }
        tc::cp_async_arrive_noinc(&kv_full[st]);
        ++c;
        return true;
      };
      fetch_slots(0, sl_next);
      for (int j = 0; j < w.nkv && ok; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          slV[i] = slK[i];
          vdV[i] = vdK[i];
          slK[i] = sl_next[i];
        }
        balV = balK;
        if (j + 1 < w.nkv) fetch_slots(j + 1, sl_next);
        // the next item is claimed during this item's last tile: a block holds no item in
        // reserve while it still has a long one to run, so the last items go to idle blocks
        if (j + 1 == w.nkv && lw == 0) next_pos = claim();
        balK = classify(j, slK, vdK);
        if (!issue(0, slK, vdK, balK)) ok = false;                 // K_j
        else if (j > 0 && !issue(1, slV, vdV, balV)) ok = false;   // V_{j-1}
      }
      if (ok && !issue(1, slK, vdK, balK)) ok = false;             // V_last
      if (!ok) break;
      ++n;
      pos = next_pos;
    }
    if (!ok) *abort_flag = 1;
    tc::cp_async_wait_all();
    if (!ok && lane == 0) {
      // stopped early: copies still in flight land before the block can go away
      for (uint32_t u = c > kRing ? c - kRing : 0; u < c; ++u)
        mbar_wait_sleep(&kv_full[u % kRing], (u / kRing) & 1, kDrainLimitNs, a.err);
      if (nq > 0) mbar_wait_sleep(q_full, (nq - 1) & 1, kDrainLimitNs, a.err);
    }
  } else {
    // ===================== MMA issuers: warp 9 (head 0) and warp 11 (head 1) =====================
    // Each head's MMAs come from a warp of their own, so neither head's chain waits behind
    // the other's: S(j+1) as soon as the softmax has read S(j), P(j).V_j once P(j) is written.
    // The whole warp runs the loop (converged); one elected lane issues each MMA and commit.
    const int hh = warp == 9 ? 0 : 1;
    {
      auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        bool got = !*abort_flag && mbar_wait_sleep(bar, parity, a.wait_ns, a.err);
        got = __all_sync(0xffffffffu, got);
        if (got) tc::fence_after_sync();
        return got;
      };
      // Shared-memory descriptors are built once per buffer; a K step of 16 elements adds a
      // constant to the start-address field (16-byte units). Building two descriptors per MMA
      // in one thread measured about 120 cycles an issue against the tensor core's 64.
      const uint64_t q_desc = tc::desc_sw128(sbase + kOffQ + hh * kTile, 16, 1024);
      const uint64_t p_desc = tc::desc_sw128(sbase + kOffP + hh * kTile, 16, 1024);
      const uint64_t k_desc = tc::desc_sw128(sbase + kOffKV, 16, 1024);     // K-major, slot 0
      const uint64_t v_desc = tc::desc_sw128(sbase + kOffKV, kBlk, 1024);   // MN-major, slot 0
      constexpr uint64_t kSlotStep = kTile >> 4;
      const uint32_t tS = tmem + hh * 128;
      const uint32_t tO = tmem + 256 + hh * 128;
      auto qk = [&](int st) {
        const uint64_t kd = k_desc + (uint64_t)st * kSlotStep;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint64_t off = (uint64_t)((ks >> 2) * (kBlk >> 4) + (ks & 3) * 2);  // 16-element step
          tc::mma_ss_elect(tS, q_desc + off, kd + off, kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit_elect(&s_full[hh]);
      };
      auto pv = [&](int st, bool acc) {
        const uint64_t vd = v_desc + (uint64_t)st * kSlotStep;
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks) {
          const uint64_t aoff = (uint64_t)((ks >> 2) * (kBlk >> 4) + (ks & 3) * 2);
          tc::mma_ss_elect(tO, p_desc + aoff, vd + (uint64_t)ks * (2048 >> 4), kIdescPV, (acc || ks > 0) ? 1u : 0u);
        }
        tc::mma_commit_elect(&p_free[hh]);
      };
      // the next K or V tile of the ring, once it has landed (rows that came by cp.async are
      // generic-proxy writes: fenced before the tensor core reads them)
      uint32_t n = 0, T = 0, c = 0;  // items, tiles, K/V ring tiles consumed
      auto next_kv = [&](int &st) -> bool {
        st = (int)(c % kRing);
        if (!wait(&kv_full[st], (c / kRing) & 1)) return false;
        if (slot_generic[st] == c + 1) tc::fence_proxy_async_smem();
        ++c;
        return true;
      };
      bool ok = true;
      while (ok) {
        if (!wait(&item_full[n & 1], (n >> 1) & 1)) {
          ok = false;
          break;
        }
        const int nkv = items[n & 1].nkv;
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[n & 1]);
        if (nkv == 0) break;
        int st = 0;
        // S(0): the S buffer is free once the softmax has read the previous item's last tile
        if (!wait(q_full, n & 1) || !next_kv(st) || (T >= 1 && !wait(&s_free[hh], (T - 1) & 1))) {
          ok = false;
          break;
        }
        qk(st);
        for (int j = 0; j < nkv; ++j) {
          if (j + 1 < nkv) {  // S(j+1) from K_{j+1}
            if (!next_kv(st) || !wait(&s_free[hh], (T + j) & 1)) {
              ok = false;
              break;
            }
            qk(st);
          }
          // O += P(j).V_j; an item's first P.V overwrites O once the last epilogue has read it
          if (!next_kv(st) || !wait(&p_full[hh], (T + j) & 1) ||
              (j == 0 && n >= 1 && !wait(&o_free[hh], (n - 1) & 1))) {
            ok = false;
            break;
          }
          pv(st, j > 0);
        }
        T += nkv;
        ++n;
      }
      if (!ok) *abort_flag = 1;
      tc::mma_commit_elect(&drain[hh]);  // nothing may still be in flight when TMEM is freed
      mbar_wait_sleep(&drain[hh], 0, kDrainLimitNs, a.err);
      __syncwarp();
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
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

}  // namespace

bool tc_prefill_pipe_supported(int group) { return group % 2 == 0; }

cudaError_t launch_tc_prefill_pipe(const astr_kv_cache &kv, int32_t layer_id, const void *q, void *out,
                                   int32_t n_heads, uint64_t wait_ns, uint32_t *err, cudaStream_t stream) {
  PipeArgs a;
  const int64_t layer_elems = (int64_t)layer_id * kv.size * kv.n_kv_heads * kv.head_dim;
  a.k_layer = static_cast<const char *>(kv.k_buffer) + layer_elems * 2;
  a.v_layer = static_cast<const char *>(kv.v_buffer) + layer_elems * 2;
  a.out = out;
  a.r2t = kv.req_to_token;
  a.rpi = kv.req_pool_indices;
  a.qo_indptr = kv.qo_indptr;
  a.kv_indptr = kv.kv_indptr;
  a.tile_b = kv.q_tile_to_batch;
  a.tile_i = kv.q_tile_to_index;
  a.size = kv.size;
  a.n_rows = kv.n_tokens;
  a.wait_ns = wait_ns;
  a.err = err;
  a.num_reqs = kv.num_reqs;
  a.max_ctx = kv.max_ctx_len;
  a.H = n_heads;
  a.Hk = kv.n_kv_heads;
  a.B = kv.batch;
  a.num_tiles = kv.num_q_tiles;
  a.n_items = (int64_t)kv.num_q_tiles * (n_heads / 2);
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kv.head_dim));
  a.layer_row0 = (int32_t)((int64_t)layer_id * kv.size);
  CUtensorMap qm, k16, v16, om;
  const uint64_t rows = (uint64_t)kv.n_layers * kv.size;
  const uint64_t cols = (uint64_t)kv.n_kv_heads * kv.head_dim;
  if (!encode_map_bf16_2d(&qm, q, (uint64_t)kv.n_tokens, (uint64_t)n_heads * kv.head_dim, 64, kRows) ||
      !encode_map_bf16_2d(&k16, kv.k_buffer, rows, cols, 64, 16) ||
      !encode_map_bf16_2d(&v16, kv.v_buffer, rows, cols, 64, 16))
    return cudaErrorInvalidValue;
  // `out` as a TMA store target: any 16-byte aligned base (its rows are H * D * 2 bytes)
  a.tma_out = (reinterpret_cast<uintptr_t>(out) & 15) == 0 &&
              encode_map_bf16_2d(&om, out, (uint64_t)kv.n_tokens, (uint64_t)n_heads * kv.head_dim, 64, kRows);
  if (!a.tma_out) om = qm;  // unused
  int sms = 0;
  cudaError_t e = sched_slot(&a.sched, &sms);
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> attr_devices{0};
  e = raise_smem_limit_once(reinterpret_cast<const void *>(prefill_pipe_kernel), kSmemBytes, attr_devices);
  if (e != cudaSuccess) return e;
  const int64_t grid = a.n_items < sms ? a.n_items : sms;
  if (grid <= 0) return cudaSuccess;
  prefill_pipe_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(a, qm, k16, v16, om);
  return cudaGetLastError();
}

}  // namespace astr
