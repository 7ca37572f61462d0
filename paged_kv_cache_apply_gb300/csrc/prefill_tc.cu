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
//  * warps 8-11 stream the two Q tiles once and then 128-key K and V tiles (two stages each,
//    released separately) with 16-byte cp.async copies into the 128-byte-swizzled layout,
//    zero-filling keys past the request;
//  * warp 12 allocates all 512 TMEM columns -- S0 | S1 | O0 | O1, 128 each -- and issues the
//    MMAs head by head, S_h = Q_h K^T (M = N = K = 128) and O_h += P_h V (P_h read from TMEM
//    where the softmax wrote it over S_h, V an MN-major operand), interleaving the heads so
//    the tensor core works on one head while the other head's softmax runs;
//  * warps 0-3 and 4-7 are the softmax of head 0 and head 1, one row per thread: a pass for
//    the row max, the reference max raised only when the row max exceeds it by 2^8 (the O row
//    is then rescaled in TMEM; the commit that published S also covers the previous P.V),
//    a pass writing exp2 of the scaled scores as bf16 P, and the epilogue that normalises O.
// KV tiles beyond the diagonal of the tile are skipped; the mask is applied only to tiles
// that cross the diagonal or the end of the request. All waits are bounded.
#include <math.h>

#include "astr_internal.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace astr {

namespace {

constexpr int kRows = 128;                 // Q tile rows (M)
constexpr int kKeys = 128;                 // keys per KV tile (N of S, K of P.V)
constexpr int kD = 128;
constexpr int kTile = kRows * kD * 2;      // 32 KB: one Q, K or V tile
constexpr int kBlk = kRows * 128;          // 16 KB: one 64-element half
constexpr int kThreads = 416;              // 8 softmax + 4 loader + 1 MMA warps
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
  uint64_t wait_ns;
  uint32_t *err;
  int32_t num_reqs, max_ctx;
  int32_t H, Hk, B;
  int32_t num_tiles;
  float scale_log2;
};

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

template <int NQ>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const PreArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *q_full = bars;           // loaders -> MMA (128 arrivals)
  uint64_t *k_full = bars + 1;       // [2]
  uint64_t *v_full = bars + 3;       // [2]
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
  const int b = __ldg(a.tile_b + tile);
  if (b < 0 || b >= a.B) {
    if (tid == 0) raise_error(a.err, ASTR_DEVERR_META);
    return;
  }
  const int ti = __ldg(a.tile_i + tile);
  const int64_t q0 = __ldg(a.qo_indptr + b);
  const int64_t Qb = (int64_t)__ldg(a.qo_indptr + b + 1) - q0;
  const int64_t Kb = (int64_t)__ldg(a.kv_indptr + b + 1) - __ldg(a.kv_indptr + b);
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
  const int rq = __ldg(a.rpi + b);
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
    mbar_init(q_full, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 128);
      mbar_init(&v_full[i], 128);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 12) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < 8) {
    // ======================= softmax of head h = warp / 4, row = tid % 128 =======================
    const int h = warp >> 2;
    const int r = tid & 127;
    if (h < NQ) {
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + h * 128 + lane_base;
      const uint32_t tO = tmem + 256 + h * 128 + lane_base;
      const int64_t pos = Pb + r0 + r;  // absolute position of this row
      const int64_t pos_min = Pb + r0;
      float m = -INFINITY, l = 0.f;
      bool aborted = false;
      const int bar_id = 1 + h;
      for (int j = 0; j < nkv; ++j) {
        const bool ok = mbar_wait(&s_full[h], j & 1, a.wait_ns, a.err);
        if (bar_any(bar_id, 128, !ok)) {
          aborted = true;
          break;
        }
        tc::fence_after_sync();
        const int64_t k0 = (int64_t)j * kKeys;
        const bool masked = (k0 + kKeys - 1 > pos_min) || (k0 + kKeys > Kb);
        // pass 1: row max of the raw scores
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t s[32];
          tc::tmem_ld32(tS + c * 32, s);
          tc::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            float v = __uint_as_float(s[k]);
            if (masked) {
              const int64_t key = k0 + c * 32 + k;
              if (key > pos || key >= Kb) v = -INFINITY;
            }
            mx = fmaxf(mx, v);
          }
        }
        mx *= a.scale_log2;
        const float m_new = (mx > m + kLazyRescale) ? mx : m;
        const float alpha = ex2_approx(m - m_new);
        if (j > 0 && __any_sync(0xffffffffu, m_new != m)) {
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
          tc::tmem_st_wait();
        }
        l *= alpha;
        m = m_new;
        // pass 2: P = exp2(score * scale - m) in bf16, written over S (column pairs)
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t s[32];
          tc::tmem_ld32(tS + c * 32, s);
          tc::tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            float x0 = __uint_as_float(s[k]) * a.scale_log2 - m;
            float x1 = __uint_as_float(s[k + 1]) * a.scale_log2 - m;
            if (masked) {
              const int64_t key = k0 + c * 32 + k;
              if (key > pos || key >= Kb) x0 = -INFINITY;
              if (key + 1 > pos || key + 1 >= Kb) x1 = -INFINITY;
            }
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            sum += p0 + p1;
            pk[k >> 1] = pack_bf16x2_rn(p0, p1);
          }
          tc::tmem_st16(tS + c * 16, pk);
        }
        l += sum;
        tc::tmem_st_wait();
        tc::fence_before_sync();
        mbar_arrive(&p_full[h]);
      }
      if (!aborted && nkv > 0) {
        const bool ok = mbar_wait(&o_done[h], 0, a.wait_ns, a.err);
        if (bar_any(bar_id, 128, !ok)) {
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
            if (write) {
#pragma unroll
              for (int k = 0; k < 32; k += 8) {
                uint4 w;
                w.x = pack_bf16x2_rn(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv);
                w.y = pack_bf16x2_rn(__uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
                w.z = pack_bf16x2_rn(__uint_as_float(o[k + 4]) * inv, __uint_as_float(o[k + 5]) * inv);
                w.w = pack_bf16x2_rn(__uint_as_float(o[k + 6]) * inv, __uint_as_float(o[k + 7]) * inv);
                *reinterpret_cast<uint4 *>(orow + c * 32 + k) = w;
              }
            }
          }
        }
      }
      if (aborted) *abort_flag = 1;
    }
  } else if (warp < 12) {
    // ================================ loaders ==================================================
    const int lt = tid - 256;      // 0..127
    const int lw = lt >> 5;
    const int half = lane >> 4, c = lane & 15;
    const int64_t rowb_kv = (int64_t)a.Hk * kD * 2;
    const char *kg = static_cast<const char *>(a.k_layer) + (int64_t)g * kD * 2;
    const char *vg = static_cast<const char *>(a.v_layer) + (int64_t)g * kD * 2;
    // Q tiles: row t of head h0 + qh sits at q[(q0 + r0 + t) * H + h0 + qh]
    {
      const char *qb = static_cast<const char *>(a.q);
      for (int qh = 0; qh < NQ; ++qh) {
        const uint32_t qs = sbase + kOffQ + qh * kTile;
        // 128 rows x 16 chunks = 2048 copies over 128 threads: 16 each, two rows per warp pass
#pragma unroll 4
        for (int j = 0; j < 16; ++j) {
          const int t = j * 8 + lw * 2 + half;  // row within the tile
          const bool v = (int64_t)t < rows_here;
          const char *src = v ? qb + (((q0 + r0 + t) * a.H + h0 + qh) * kD) * 2 + c * 16 : qb;
          tc::cp_async16(qs + tc::sw128_chunk_offset(t, c, kBlk), src, v ? 16u : 0u);
        }
      }
      tc::cp_async_arrive_noinc(q_full);
    }
    // K / V tiles
    int64_t nxt = -1;
    if (nkv > 0 && lw * 32 + lane < key_end) nxt = __ldg(row + lw * 32 + lane);
    for (int j = 0; j < nkv; ++j) {
      const int st = j & 1;
      const int64_t k0 = (int64_t)j * kKeys;
      int64_t my = nxt;  // slot of key k0 + lw*32 + lane
      {
        const int64_t kn = k0 + kKeys + lw * 32 + lane;
        nxt = (j + 1 < nkv && kn < key_end) ? (int64_t)__ldg(row + kn) : -1;
      }
      const bool in_range = k0 + lw * 32 + lane < key_end;
      if (my >= a.size || (my < 0 && in_range)) {
        raise_error(a.err, ASTR_DEVERR_SLOT);
        my = -1;
      }
      // K
      int ok = 1;
      if (lane == 0) {
        if (j >= 2) ok = mbar_wait(&k_empty[st], ((j >> 1) - 1) & 1, a.wait_ns, a.err);
        if (*abort_flag) ok = 0;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      const uint32_t kst = sbase + kOffK + st * kTile;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int tl = i * 2 + half;
        const int t = lw * 32 + tl;
        const int64_t s = __shfl_sync(0xffffffffu, my, tl);
        const bool v = s >= 0;
        tc::cp_async16(kst + tc::sw128_chunk_offset(t, c, kBlk), kg + (v ? s * rowb_kv + c * 16 : 0),
                       v ? 16u : 0u);
      }
      tc::cp_async_arrive_noinc(&k_full[st]);
      // V
      ok = 1;
      if (lane == 0) {
        if (j >= 2) ok = mbar_wait(&v_empty[st], ((j >> 1) - 1) & 1, a.wait_ns, a.err);
        if (*abort_flag) ok = 0;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      const uint32_t vst = sbase + kOffV + st * kTile;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int tl = i * 2 + half;
        const int t = lw * 32 + tl;
        const int64_t s = __shfl_sync(0xffffffffu, my, tl);
        const bool v = s >= 0;
        tc::cp_async16(vst + tc::sw128_chunk_offset(t, c, kBlk), vg + (v ? s * rowb_kv + c * 16 : 0),
                       v ? 16u : 0u);
      }
      tc::cp_async_arrive_noinc(&v_full[st]);
    }
    tc::cp_async_wait_all();
  } else {
    // ============================== MMA issuer (one lane) =====================================
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, a.wait_ns, a.err);
      auto qk = [&](int hh, int j) {
        const uint32_t qaddr = sbase + kOffQ + hh * kTile;
        const uint32_t kaddr = sbase + kOffK + (j & 1) * kTile;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          const uint64_t ad = tc::desc_sw128(qaddr + (ks >> 2) * kBlk + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = tc::desc_sw128(kaddr + (ks >> 2) * kBlk + (ks & 3) * 32, 16, 1024);
          tc::mma_ss(tmem + hh * 128, ad, bd, kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc::mma_commit(&s_full[hh]);
      };
      auto pv = [&](int hh, int j) {
        const uint32_t vaddr = sbase + kOffV + (j & 1) * kTile;
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks) {
          const uint64_t bd = tc::desc_sw128(vaddr + ks * 2048, kBlk, 1024);
          tc::mma_ts(tmem + 256 + hh * 128, tmem + hh * 128 + ks * 8, bd, kIdescPV,
                     (j > 0 || ks > 0) ? 1u : 0u);
        }
      };
      auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
        if (*abort_flag || !mbar_wait(bar, parity, a.wait_ns, a.err)) return false;
        tc::fence_after_sync();
        tc::fence_proxy_async_smem();
        return true;
      };
      if (ok) {
        tc::fence_after_sync();
        tc::fence_proxy_async_smem();
        ok = nkv == 0 || wait(&k_full[0], 0);
        if (ok && nkv > 0) {
          for (int hh = 0; hh < NQ; ++hh) qk(hh, 0);
          tc::mma_commit(&k_empty[0]);
        }
        for (int j = 0; j < nkv && ok; ++j) {
          const bool more = j + 1 < nkv;
          for (int hh = 0; hh < NQ && ok; ++hh) {
            if (!wait(&p_full[hh], j & 1)) { ok = false; break; }
            if (hh == 0 && !wait(&v_full[j & 1], (j >> 1) & 1)) { ok = false; break; }
            pv(hh, j);
            if (!more) tc::mma_commit(&o_done[hh]);
            if (hh == NQ - 1) tc::mma_commit(&v_empty[j & 1]);
            if (more) {
              if (hh == 0 && !wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1)) { ok = false; break; }
              qk(hh, j + 1);
              if (hh == NQ - 1) tc::mma_commit(&k_empty[(j + 1) & 1]);
            }
          }
        }
      }
      if (!ok) *abort_flag = 1;
      tc::mma_commit(drain);
      mbar_wait(drain, 0, kDrainLimitNs, a.err);
    }
    __syncwarp();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 12) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int NQ>
cudaError_t run_nq(const PreArgs &a, int64_t grid, cudaStream_t s) {
  auto k = prefill_tc_kernel<NQ>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (grid > 0) k<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool tc_prefill_supported(int dtype, int head_dim, int group, int q_tile_rows) {
  return dtype == ASTR_BF16 && head_dim == kD && q_tile_rows == kRows && group >= 1;
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
  const int G = n_heads / kv.n_kv_heads;
  if (G % 2 == 0) return run_nq<2>(a, (int64_t)kv.num_q_tiles * (n_heads / 2), stream);
  return run_nq<1>(a, (int64_t)kv.num_q_tiles * n_heads, stream);
}

}  // namespace astr
