// Varlen causal prefill on the tcgen05 tensor cores (bf16, head_dim 128).
//
// AstrAI inference guide, "Attention Backend": a ragged-batch prefill reading K/V straight
// from the flat pool through req_to_token, each request addressed by qo_indptr / kv_indptr;
// "KVCache System": 128-row Q tiles named by q_tile_to_batch / q_tile_to_index, and prefill
// resumed right after a cached prefix. AstrAI internals, "Autoregression & Causal Masking":
// query position i attends to keys j <= i (here positions are absolute: row i of a request
// with prefix P sits at P + i).
//
// One block computes a 128-row Q tile for NQ = 2 query heads of the same KV group (1 when
// the group has a single head), so every K/V tile it stages feeds two heads:
//  * warp 8 streams the two Q tiles once and then 128-key K and V tiles (two stages each,
//    released separately) into the 128-byte-swizzled layout: one TMA tensor copy of a 16-row
//    box per run of 16 keys whose slots are consecutive (a page; destinations 2 KB aligned),
//    16-byte cp.async copies for keys outside such runs, zero-filled past the request; the
//    page-table entries of a tile are read while the previous tile's copies are issued;
//  * warp 9 allocates all 512 TMEM columns -- S0 | S1 | O0 | O1, 128 each -- and issues the
//    MMAs (the whole warp runs converged, an elected lane issues, descriptors are built once
//    per buffer), S_h = Q_h K^T (M = N = K = 128) and O_h += P_h V (P_h read from TMEM where
//    the softmax wrote it over S_h, V an MN-major operand), head by head, so that the tensor
//    core works on one head while the other head's softmax runs;
//  * warps 0-3 and 4-7 are the softmax of head 0 and head 1, one thread per row holding all
//    128 scores of a tile in registers: the row max, the reference max raised only when the
//    row max exceeds it by 2^8 (the O row is then rescaled in TMEM; the commit that published
//    S also covers the previous P.V), exp2 of the scaled scores written as bf16 P over the
//    first 64 columns of S, and the epilogue that normalises O and sends a whole tile out as
//    two TMA boxes from the head's Q buffer (plain stores for a tile cut by the request's end).
// KV tiles beyond the diagonal of the tile are skipped; the mask is applied only to tiles
// that cross the diagonal or the end of the request. All waits are bounded.
#include <math.h>

#include "astr_internal.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tma_maps.h"

namespace astr {

namespace {

constexpr int kRows = 128;                 // Q tile rows (M)
constexpr int kKeys = 128;                 // keys per KV tile (N of S, K of P.V)
constexpr int kD = 128;
constexpr int kTile = kRows * kD * 2;      // 32 KB: one Q, K or V tile
constexpr int kBlk = kRows * 128;          // 16 KB: one 64-element half
constexpr int kThreads = 320;              // 8 softmax + 1 loader + 1 MMA warp
constexpr float kLazyRescale = 8.0f;

constexpr int kOffQ = 0;                   // 2 Q tiles
constexpr int kOffK = kOffQ + 2 * kTile;   // 2 K stages
constexpr int kOffV = kOffK + 2 * kTile;   // 2 V stages
constexpr int kOffBar = kOffV + 2 * kTile;
constexpr int kOffMisc = kOffBar + 32 * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;

constexpr uint32_t kIdescQK = tc::idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, false, true);

struct PreArgs {
  const void *q;
  void *out;
  const void *k_layer;
  const void *v_layer;
  const int32_t *r2t;
  const int32_t *rpi;
  const int32_t *qo_indptr;
  const int32_t *kv_indptr;
  const int32_t *tile_b;
  const int32_t *tile_i;
  int64_t size;
  int64_t n_rows;  // packed q rows
  int32_t layer_row0;  // first row of this layer in the [n_layers * size, Hk * D] view
  int32_t total_rows;  // n_layers * size: any row at or past it reads as zero
  uint64_t wait_ns;
  uint32_t *err;
  int32_t num_reqs, max_ctx;
  int32_t H, Hk, B;
  int32_t num_tiles;
  int32_t tma_out;  // whole tiles leave through a TMA map of `out`
  float scale_log2;
};

// the 128 threads of one head's softmax warps (barrier 1 for head 0, 2 for head 1)
__device__ __forceinline__ void head_bar_sync(int h) {
  if (h == 0)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    asm volatile("bar.sync 2, 128;" ::: "memory");
}

// O += P V with P (the A operand) read from TMEM, issued by the elected lane of a converged warp
__device__ __forceinline__ void mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int NQ>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PreArgs a, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap k16, const __grid_constant__ CUtensorMap v16,
                      const __grid_constant__ CUtensorMap omap) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *q_full = bars;           // TMA -> MMA (transaction bytes)
  uint64_t *k_full = bars + 1;       // [2] TMA -> MMA
  uint64_t *v_full = bars + 3;       // [2] TMA -> MMA
  uint64_t *k_empty = bars + 5;      // [2] MMA commit
  uint64_t *v_empty = bars + 7;      // [2] MMA commit
  uint64_t *s_full = bars + 9;       // [2] per head, MMA commit
  uint64_t *p_full = bars + 11;      // [2] per head, 128 arrivals
  uint64_t *o_done = bars + 13;      // [2] per head, MMA commit
  uint64_t *drain = bars + 15;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- work item: Q tile `ti` of request b, query heads h0 .. h0+NQ-1 ---------------------
  const int pairs = a.H / NQ;
  const int tile = a.num_tiles - 1 - (int)(blockIdx.x / pairs);  // later tiles carry more keys
  const int h0 = (int)(blockIdx.x % pairs) * NQ;
  const int G = a.H / a.Hk;
  const int g = h0 / G;
  // The item's metadata in two rounds of loads: the tile's entries, then the request's lengths
  // and page-table row together (read at a clamped index, checked afterwards), since each round
  // costs a memory latency before anything else can start.
  const int b = __ldg(a.tile_b + tile);
  const int ti = __ldg(a.tile_i + tile);
  const int bc = b < 0 ? 0 : (b >= a.B ? a.B - 1 : b);
  const int32_t qo_a = __ldg(a.qo_indptr + bc), qo_b = __ldg(a.qo_indptr + bc + 1);
  const int32_t kv_a = __ldg(a.kv_indptr + bc), kv_b = __ldg(a.kv_indptr + bc + 1);
  const int rq = __ldg(a.rpi + bc);
  if (b == -1) return;  // an empty entry of the tile list
  if (b < 0 || b >= a.B) {
    if (tid == 0) raise_error(a.err, ASTR_DEVERR_META);
    return;
  }
  const int64_t q0 = qo_a;
  const int64_t Qb = (int64_t)qo_b - q0;
  const int64_t Kb = (int64_t)kv_b - kv_a;
  const int64_t Pb = Kb - Qb;
  const int64_t r0 = (int64_t)ti * kRows;  // first request-local row of the tile
  if (ti < 0 || r0 >= Qb) {
    if (tid == 0) raise_error(a.err, ASTR_DEVERR_META);
    return;
  }
  if (Pb < 0 || Kb > a.max_ctx || q0 + Qb > a.n_rows) {
    if (tid == 0) raise_error(a.err, ASTR_DEVERR_LEN);
    return;
  }
  if (rq < 0 || rq >= a.num_reqs) {
    if (tid == 0) raise_error(a.err, ASTR_DEVERR_ROW);
    return;
  }
  const int32_t *row = a.r2t + (int64_t)rq * a.max_ctx;
  const int64_t rows_here = (Qb - r0) < kRows ? (Qb - r0) : kRows;
  const int64_t key_end = (Pb + r0 + rows_here) < Kb ? (Pb + r0 + rows_here) : Kb;  // keys needed
  const int nkv = (int)((key_end + kKeys - 1) / kKeys);

  // ---- set-up ---------------------------------------------------------------------------------
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {  // 32 loader lanes (cp.async) + one expect-tx arrival (TMA)
      mbar_init(&k_full[i], 33);
      mbar_init(&v_full[i], 33);
      mbar_init(&k_empty[i], 1);  // MMA commits
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drain, 1);
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
    // ============ softmax: head h = warp / 4, one thread per row, all 128 scores in registers
    const int h = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    if (h < NQ) {
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + h * 128 + lane_base;
      const uint32_t tO = tmem + 256 + h * 128 + lane_base;
      const int64_t pos = Pb + r0 + r;  // absolute position of this row
      const int64_t pos_min = Pb + r0;
      const int64_t lim_row = (pos + 1 < Kb ? pos + 1 : Kb);  // keys [0, lim_row) are visible
      float m = -INFINITY, l = 0.f;
      bool aborted = false;
      for (int j = 0; j < nkv; ++j) {
        if (!mbar_wait(&s_full[h], j & 1, a.wait_ns, a.err)) {
          aborted = true;
          break;
        }
        tc::fence_after_sync();
        uint32_t sv[128];
        tc::tmem_ld32(tS, sv);
        tc::tmem_ld32(tS + 32, sv + 32);
        tc::tmem_ld32(tS + 64, sv + 64);
        tc::tmem_ld32(tS + 96, sv + 96);
        tc::tmem_ld_wait();
        // only tiles crossing this tile's diagonal or the end of the request carry masked keys
        if ((int64_t)j * kKeys + kKeys - 1 > pos_min || (int64_t)j * kKeys + kKeys > Kb) {
          const int64_t lim = lim_row - (int64_t)j * kKeys;
          const int nvalid = lim < 0 ? 0 : (lim > kKeys ? kKeys : (int)lim);
#pragma unroll
          for (int k = 0; k < kKeys; ++k)
            if (k >= nvalid) sv[k] = 0xFF800000u;  // -inf
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
        // P = exp2(score * scale - m) in bf16 over the first 64 columns of S (the row's
        // scores are all in registers, so nothing still to be read is overwritten)
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 nm2 = make_float2(-m, -m);
        float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            const float2 x = ffma2(make_float2(__uint_as_float(sv[32 * c + k]), __uint_as_float(sv[32 * c + k + 1])),
                                   sc2, nm2);
            const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);  // ex2(-inf) = 0
            sum2[(k >> 1) & 3] = fadd2(sum2[(k >> 1) & 3], make_float2(p0, p1));
            pk[k >> 1] = pack_bf16x2_rn(p0, p1);
          }
          tc::tmem_st16(tS + c * 16, pk);
        }
        const float2 s01 = fadd2(sum2[0], sum2[1]), s23 = fadd2(sum2[2], sum2[3]);
        l += (s01.x + s01.y) + (s23.x + s23.y);
        if (rescale) {
          // the commit behind s_full also covers P.V of the previous tile: O is settled
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
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        mbar_arrive(&p_full[h]);
      }
      // A whole tile leaves through this head's Q buffer as two TMA boxes: the commit behind
      // o_done also covers the head's last S, the buffer's last reader. (One thread per row
      // storing its 256 bytes straight to global memory sends each warp store to 32 lines;
      // measured on GB300 the boxes take 1-1.5 % off the prefill.) A tile cut by the request's
      // end stores its own rows directly: a box would overwrite the next request's rows.
      const bool by_tma = a.tma_out && rows_here == kRows && nkv > 0;  // uniform over the head
      const uint32_t qoff = kOffQ + h * kTile;
      if (!aborted && nkv > 0) {
        if (!mbar_wait(&o_done[h], 0, a.wait_ns, a.err)) {
          aborted = true;
        } else {
          tc::fence_after_sync();
          const float inv = 1.f / l;
          uint16_t *orow = static_cast<uint16_t *>(a.out) + ((q0 + r0 + r) * a.H + h0 + h) * kD;
          const bool write = (int64_t)r < rows_here;
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
                *reinterpret_cast<uint4 *>(smem + qoff + tc::sw128_chunk_offset(r, c * 4 + (k >> 3), kBlk)) = w;
              else if (write)
                *reinterpret_cast<uint4 *>(orow + c * 32 + k) = w;
            }
          }
        }
      }
      if (aborted) *abort_flag = 1;
      if (by_tma) {
        // every thread of the head arrives, aborted or not, so the barrier cannot hang
        tc::fence_proxy_async_smem();
        head_bar_sync(h);
        if (r == 0 && !*abort_flag) {
          tc::tma_store_2d(&omap, (h0 + h) * kD, (int)(q0 + r0), sbase + qoff);
          tc::tma_store_2d(&omap, (h0 + h) * kD + 64, (int)(q0 + r0), sbase + qoff + kBlk);
          tc::bulk_commit();
          tc::bulk_wait_read_all();  // the buffer stays put until the engine has read it
        }
      }
    }
  } else if (warp == 8) {
    // ============================== TMA loader (one warp) ======================================
    const int col0 = g * kD;  // this KV head's columns in the [rows, Hk * D] view
    const int64_t rowb_kv = (int64_t)a.Hk * kD * 2;
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, NQ * kTile);
      for (int qh = 0; qh < NQ; ++qh)
        for (int hf = 0; hf < 2; ++hf)
          tc::tma_load_2d(sbase + kOffQ + qh * kTile + hf * kBlk, &qmap, (h0 + qh) * kD + hf * 64,
                          (int)(q0 + r0), q_full);
    }
    // keys k0 + 4 * lane + i of a tile: their slots are read one tile ahead of the copies
    auto fetch_slots = [&](int j, int (&sl)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t kk = (int64_t)j * kKeys + 4 * lane + i;
        sl[i] = kk < key_end ? __ldg(row + kk) : -1;
      }
    };
    int sl_next[4];
    fetch_slots(0, sl_next);
    for (int j = 0; j < nkv; ++j) {
      const int st = j & 1;
      int sl[4];
      bool vd[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sl[i] = sl_next[i];
        vd[i] = (int64_t)j * kKeys + 4 * lane + i < key_end;
        if (vd[i] && (sl[i] < 0 || (int64_t)sl[i] >= a.size)) {
          raise_error(a.err, ASTR_DEVERR_SLOT);
          vd[i] = false;
        }
      }
      if (j + 1 < nkv) fetch_slots(j + 1, sl_next);
      // whether each 16-key group is a run of consecutive slots (one page)
      const bool run4 = vd[0] && vd[1] && vd[2] && vd[3] && sl[1] == sl[0] + 1 &&
                        sl[2] == sl[1] + 1 && sl[3] == sl[2] + 1;
      const int next0 = __shfl_down_sync(0xffffffffu, sl[0], 1);
      const bool link = ((lane & 3) == 3) || (next0 == sl[3] + 1);
      const unsigned bal = __ballot_sync(0xffffffffu, run4 && link);
      const bool group_run = ((bal >> (lane & ~3)) & 0xFu) == 0xFu;
      for (int kvsel = 0; kvsel < 2; ++kvsel) {  // 0: K, 1: V
        uint64_t *fullb = kvsel ? &v_full[st] : &k_full[st];
        uint64_t *emptyb = kvsel ? &v_empty[st] : &k_empty[st];
        int ok = 1;
        if (lane == 0) {
          if (j >= 2) ok = mbar_wait(emptyb, ((j >> 1) - 1) & 1, a.wait_ns, a.err);
          if (*abort_flag) ok = 0;
          if (ok) mbar_arrive_expect_tx(fullb, (uint32_t)__popc(bal & 0x11111111u & (bal >> 1) & (bal >> 2) & (bal >> 3)) * 4096u);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        const uint32_t dst = sbase + (kvsel ? kOffV : kOffK) + st * kTile;
        if (group_run) {
          if ((lane & 3) == 0) {
            const void *m16 = kvsel ? (const void *)&v16 : (const void *)&k16;
            for (int hf = 0; hf < 2; ++hf)
              tc::tma_load_2d(dst + hf * kBlk + (4 * lane) * 128, m16, col0 + hf * 64,
                              a.layer_row0 + sl[0], fullb);
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
        tc::cp_async_arrive_noinc(fullb);
      }
      if (*abort_flag) break;
    }
  } else {
    // ===================== MMA issuer: warp 9, converged; one elected lane issues ==============
    // Each head's MMAs run as a block in a fixed order -- per KV tile, head 0's P.V and next S,
    // then head 1's -- so head 1's S lands one block after head 0's, and from then on one
    // head's softmax runs while the tensor core works for the other. Descriptors are built once
    // per buffer and stepped by constants (16-byte units); the whole warp runs the loop and an
    // elected lane issues, which keeps the issue at the tensor core's rate (a loop run by one
    // lane of a divergent branch with two descriptors built per MMA measured about 120 cycles an
    // issue against the tensor core's 64).
    {
      auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        bool got = !*abort_flag && mbar_wait_sleep(bar, parity, a.wait_ns, a.err);
        got = __all_sync(0xffffffffu, got);
        if (got) {
          tc::fence_after_sync();
          tc::fence_proxy_async_smem();  // rows that came by cp.async (generic proxy)
        }
        return got;
      };
      constexpr uint64_t kStep = kTile >> 4;
      const uint64_t q_desc = tc::desc_sw128(sbase + kOffQ, 16, 1024);     // head 0's Q
      const uint64_t k_desc = tc::desc_sw128(sbase + kOffK, 16, 1024);     // K stage 0
      const uint64_t v_desc = tc::desc_sw128(sbase + kOffV, kBlk, 1024);   // V stage 0, MN-major
      auto qk = [&](int hh, int j) {
        const uint64_t qd = q_desc + (uint64_t)hh * kStep;
        const uint64_t kd = k_desc + (uint64_t)(j & 1) * kStep;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint64_t off = (uint64_t)((ks >> 2) * (kBlk >> 4) + (ks & 3) * 2);  // 16-element step
          tc::mma_ss_elect(tmem + hh * 128, qd + off, kd + off, kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit_elect(&s_full[hh]);
      };
      bool ok = __all_sync(0xffffffffu, mbar_wait_sleep(q_full, 0, a.wait_ns, a.err));
      if (ok) {
        tc::fence_after_sync();
        ok = wait(&k_full[0], 0);
        if (ok) {
          for (int hh = 0; hh < NQ; ++hh) qk(hh, 0);
          tc::mma_commit_elect(&k_empty[0]);
        }
        for (int j = 0; j < nkv && ok; ++j) {
          if (!wait(&v_full[j & 1], (j >> 1) & 1)) {
            ok = false;
            break;
          }
          const uint64_t vd = v_desc + (uint64_t)(j & 1) * kStep;
          for (int hh = 0; hh < NQ && ok; ++hh) {
            if (!wait(&p_full[hh], j & 1)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int ks = 0; ks < kKeys / 16; ++ks)
              mma_ts_elect(tmem + 256 + hh * 128, tmem + hh * 128 + ks * 8, vd + (uint64_t)ks * (2048 >> 4),
                           kIdescPV, (j > 0 || ks > 0) ? 1u : 0u);
            if (j + 1 == nkv) {
              tc::mma_commit_elect(&o_done[hh]);
            } else {
              if (hh == 0 && !wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1)) {
                ok = false;
                break;
              }
              qk(hh, j + 1);  // overwrites S_hh: issued after the P.V that reads P_hh from it
            }
          }
          if (!ok) break;
          tc::mma_commit_elect(&v_empty[j & 1]);
          if (j + 1 < nkv) tc::mma_commit_elect(&k_empty[(j + 1) & 1]);
        }
      }
      if (!ok) *abort_flag = 1;
      tc::mma_commit_elect(drain);  // nothing may still be in flight when TMEM is freed
      mbar_wait_sleep(drain, 0, kDrainLimitNs, a.err);
      __syncwarp();
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

struct Maps {
  CUtensorMap q, k16, v16, o;
};

template <int NQ>
cudaError_t run_nq(const PreArgs &a, const Maps &m, int64_t grid, cudaStream_t s) {
  auto k = prefill_tc_kernel<NQ>;
  static std::atomic<uint64_t> attr_devices{0};
  cudaError_t e = raise_smem_limit_once(reinterpret_cast<const void *>(k), kSmemBytes, attr_devices);
  if (e != cudaSuccess) return e;
  if (grid <= 0) return cudaSuccess;
  k<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(a, m.q, m.k16, m.v16, m.o);
  return cudaGetLastError();
}

}  // namespace

bool tc_prefill_supported(int dtype, int head_dim, int group, int q_tile_rows) {
  return dtype == ASTR_BF16 && head_dim == kD && q_tile_rows == kRows && group >= 1;
}

bool tc_prefill_fits(const astr_kv_cache &kv) {
  // TMA row coordinates are 32-bit
  return (int64_t)kv.n_layers * kv.size < (int64_t(1) << 31) && kv.n_tokens >= 1 &&
         kv.n_tokens < (int64_t(1) << 31);
}

cudaError_t launch_tc_prefill(const astr_kv_cache &kv, int32_t layer_id, const void *q, void *out,
                              int32_t n_heads, uint64_t wait_ns, uint32_t *err,
                              cudaStream_t stream) {
  PreArgs a;
  const int64_t layer_elems = (int64_t)layer_id * kv.size * kv.n_kv_heads * kv.head_dim;
  a.q = q;
  a.out = out;
  a.k_layer = static_cast<const char *>(kv.k_buffer) + layer_elems * 2;
  a.v_layer = static_cast<const char *>(kv.v_buffer) + layer_elems * 2;
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
  a.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kv.head_dim));
  a.layer_row0 = (int32_t)((int64_t)layer_id * kv.size);
  a.total_rows = (int32_t)((int64_t)kv.n_layers * kv.size);
  Maps m;
  const uint64_t rows = (uint64_t)kv.n_layers * kv.size;
  const uint64_t cols = (uint64_t)kv.n_kv_heads * kv.head_dim;
  if (!encode_map_bf16_2d(&m.q, q, (uint64_t)kv.n_tokens, (uint64_t)n_heads * kv.head_dim, 64, kRows) ||
      !encode_map_bf16_2d(&m.k16, kv.k_buffer, rows, cols, 64, 16) ||
      !encode_map_bf16_2d(&m.v16, kv.v_buffer, rows, cols, 64, 16))
    return cudaErrorInvalidValue;
  // `out` as a TMA store target: any 16-byte aligned base (its rows are H * D * 2 bytes)
  a.tma_out = (reinterpret_cast<uintptr_t>(out) & 15) == 0 &&
              encode_map_bf16_2d(&m.o, out, (uint64_t)kv.n_tokens, (uint64_t)n_heads * kv.head_dim, 64, kRows);
  if (!a.tma_out) m.o = m.q;  // unused
  const int G = n_heads / kv.n_kv_heads;
  // More (Q tile, head pair) items than SMs: the persistent pipelined kernel, whose blocks run
  // item after item with the next item's loads and first scores overlapping the current
  // epilogue. Fewer: one block per item (measured faster for the 128 items of four 512-row
  // chunks: 16.8 against 18.3 us).
  if (tc_prefill_pipe_supported(G)) {
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    if ((int64_t)kv.num_q_tiles * (n_heads / 2) > sms)
      return launch_tc_prefill_pipe(kv, layer_id, q, out, n_heads, wait_ns, err, stream);
  }
  if (G % 2 == 0) return run_nq<2>(a, m, (int64_t)kv.num_q_tiles * (n_heads / 2), stream);
  return run_nq<1>(a, m, (int64_t)kv.num_q_tiles * n_heads, stream);
}

}  // namespace astr
