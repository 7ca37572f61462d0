// Per-step batch metadata computed on the device: the prefix sums qo_indptr / kv_indptr and
// the Q-tile maps q_tile_to_batch / q_tile_to_index (inference guide, "KVCache System": the
// KVCache dataclass that bind_tasks() returns carries kv_indptr, qo_indptr and the tile maps,
// computed once per step and shared by every layer).
//
// The order of the tiles is the host planner's: by cost -- the number of 128-key tiles a Q
// tile visits under the causal mask -- cheapest first, ties in request order, which is what a
// stable sort by cost of the tiles enumerated request by request gives. Here each thread puts
// one tile straight at its position in that order,
//   rank(b, t) = #{tiles with cost < c} + #{tiles of requests b' < b with cost c}
//              + #{tiles t' < t of request b with cost c},        c = cost(b, t),
// counted request by request. The costs of one request's tiles do not decrease with the tile
// index, so the count of its tiles below a cost has a closed form: a rank costs O(batch)
// integer arithmetic, which the 32 lanes of a warp share, with no sort and no atomics.
//
// Every block rebuilds the per-request table (q_len, prefix, running tile count) in shared
// memory from q_lens / kv_lens, so the whole computation is a single launch.
#include <cuda_runtime.h>
#include <stdint.h>

#include "astr_internal.cuh"
#include "launch.h"

namespace astr {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// Tiles of one request (Q new rows after a prefix of P keys, n = ceil(Q / R) tiles of R rows)
// whose cost ceil((P + min(Q, (t+1) R)) / 128) is below c:
//   cost(t) < c  <=>  min(Q, (t+1) R) <= X,  X = 128 (c - 1) - P.
// If Q <= X every tile qualifies; otherwise exactly the t with (t+1) R <= X, of which there are
// floor(X / R) (fewer than n, since X < Q). In that branch R <= X < Q < 2^31, so the division
// is a 32-bit one (a shift when R is a power of two, r_shift >= 0).
__device__ __forceinline__ int tiles_below(int Q, int P, int n, int R, int r_shift, int c) {
  const long long X = 128LL * (c - 1) - P;
  if (Q <= X) return n;
  if (X < R) return 0;
  return r_shift >= 0 ? (int)((unsigned)X >> r_shift) : (int)((unsigned)X / (unsigned)R);
}

// inclusive scan of v across the block; `sh` holds kWarps partial sums; all threads call it
__device__ __forceinline__ int64_t block_inclusive_scan(int64_t v, int64_t *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) sh[warp] = v;
  __syncthreads();
  int64_t before = 0;
  for (int w = 0; w < warp; ++w) before += sh[w];
  __syncthreads();
  return v + before;
}

__global__ void __launch_bounds__(kThreads)
bind_tasks_kernel(const int32_t *__restrict__ q_lens, const int32_t *__restrict__ kv_lens,
                  int B, int R, int32_t *__restrict__ qo_indptr, int32_t *__restrict__ kv_indptr,
                  int32_t *__restrict__ tile_b, int32_t *__restrict__ tile_i, int max_tiles,
                  uint32_t *err) {
  extern __shared__ int2 table[];
  int2 *sQP = table;                                  // [B]   (new rows, cached prefix) of b
  int32_t *sT = reinterpret_cast<int32_t *>(table + B);  // [B+1] tiles of requests before b
  __shared__ int64_t part[3][kWarps];
  const int tid = threadIdx.x;

  // ---- per-request table and the three prefix sums (segment per thread, then block scans) ----
  const int seg = (B + kThreads - 1) / kThreads;
  const int lo = min(B, tid * seg), hi = min(B, lo + seg);
  int64_t sq = 0, sk = 0, st = 0;
  bool bad = false;
  for (int b = lo; b < hi; ++b) {
    const int q = q_lens ? q_lens[b] : 0, k = kv_lens[b];
    const bool ok = q >= 0 && k >= q;
    bad |= !ok;
    const int2 qp = ok ? make_int2(q, k - q) : make_int2(0, 0);  // a bad request counts as
    sQP[b] = qp;                                                  // empty (the maps become -1)
    sq += qp.x;
    sk += qp.x + qp.y;
    st += (qp.x + R - 1) / R;
  }
  const int64_t iq = block_inclusive_scan(sq, part[0]);
  const int64_t ik = block_inclusive_scan(sk, part[1]);
  const int64_t it = block_inclusive_scan(st, part[2]);
  int64_t rq = iq - sq, rk = ik - sk, rt = it - st;  // exclusive prefixes of this segment
  for (int b = lo; b < hi; ++b) {
    if (blockIdx.x == 0) {
      if (qo_indptr) qo_indptr[b] = (int32_t)rq;
      kv_indptr[b] = (int32_t)rk;
    }
    const int2 qp = sQP[b];
    sT[b] = (int32_t)rt;
    rq += qp.x;
    rk += qp.x + qp.y;
    rt += (qp.x + R - 1) / R;
  }
  // the block totals sit in the last thread's inclusive sums
  __shared__ int64_t totals[3];
  if (tid == kThreads - 1) totals[0] = iq, totals[1] = ik, totals[2] = it;
  bad = __syncthreads_or(bad) != 0;
  const int64_t n_real = totals[2];
  if (tid == 0) {
    sT[B] = (int32_t)(n_real < INT32_MAX ? n_real : INT32_MAX);
    if (blockIdx.x == 0) {
      if (qo_indptr) qo_indptr[B] = (int32_t)(totals[0] < INT32_MAX ? totals[0] : INT32_MAX);
      kv_indptr[B] = (int32_t)(totals[1] < INT32_MAX ? totals[1] : INT32_MAX);
    }
  }
  const bool overflow = totals[0] > INT32_MAX || totals[1] > INT32_MAX;
  __syncthreads();
  const bool fail = bad || overflow || n_real > max_tiles;
  if (fail && blockIdx.x == 0 && tid == 0)
    raise_error(err, bad || overflow ? ASTR_DEVERR_LEN : ASTR_DEVERR_META);

  // ---- one tile per warp: its request by binary search, then its rank by counting over the
  // requests, split across the lanes ----------------------------------------------------------
  const int lane = tid & 31;
  const int r_shift = (R & (R - 1)) == 0 ? __ffs(R) - 1 : -1;
  const int64_t pad = fail ? 0 : max_tiles - n_real;
  for (int64_t e = (int64_t)blockIdx.x * kWarps + (tid >> 5); e < max_tiles;
       e += (int64_t)gridDim.x * kWarps) {
    if (fail || e >= n_real) {  // the empty entries go first, so the walk from the end meets
      const int64_t at = fail ? e : e - n_real;  // real tiles first
      if (lane == 0) tile_b[at] = -1, tile_i[at] = -1;
      continue;
    }
    int l = 0, h = B - 1;  // the last request whose first tile is at or before e
    while (l < h) {
      const int m = (l + h + 1) >> 1;
      if (sT[m] <= e) l = m; else h = m - 1;
    }
    const int b = l;
    const int t = (int)(e - sT[b]);
    const int Qb = sQP[b].x, Pb = sQP[b].y;
    const int last_row = (int64_t)(t + 1) * R < Qb ? (t + 1) * R : Qb;
    const int c = (int)(((int64_t)Pb + last_row + 127) / 128);
    unsigned part_rank = 0;
    for (int u = lane; u < B; u += 32) {
      const int2 qp = sQP[u];
      const int nu = r_shift >= 0 ? (int)(((unsigned)qp.x + R - 1) >> r_shift) : sT[u + 1] - sT[u];
      const int below = tiles_below(qp.x, qp.y, nu, R, r_shift, c);
      part_rank += below;
      if (u < b) part_rank += tiles_below(qp.x, qp.y, nu, R, r_shift, c + 1) - below;
    }
    // + own earlier tiles of the same cost
    const int64_t rank = (int64_t)__reduce_add_sync(0xffffffffu, part_rank) + t -
                         tiles_below(Qb, Pb, sT[b + 1] - sT[b], R, r_shift, c);
    if (lane != 0) continue;
    if (rank < 0 || rank >= n_real) {  // cannot happen; flag it rather than store outside
      raise_error(err, ASTR_DEVERR_META);
      continue;
    }
    tile_b[pad + rank] = b;
    tile_i[pad + rank] = t;
  }
}

// the per-request table: 3 * batch + 1 int32 in dynamic shared memory, up to 192 KB
constexpr int kMaxBatch = 16383;
constexpr int kMaxTableBytes = (3 * kMaxBatch + 1) * 4;
size_t table_bytes(int batch) { return (size_t)(3 * batch + 1) * sizeof(int32_t); }

}  // namespace

int bind_tasks_max_batch() { return kMaxBatch; }

cudaError_t launch_bind_tasks(const int32_t *q_lens, const int32_t *kv_lens, int32_t batch,
                              int32_t q_tile_rows, int32_t *qo_indptr, int32_t *kv_indptr,
                              int32_t *q_tile_to_batch, int32_t *q_tile_to_index,
                              int32_t max_tiles, int num_sms, uint32_t *err, cudaStream_t stream) {
  if (batch < 0 || batch > kMaxBatch) return cudaErrorInvalidValue;
  static std::atomic<uint64_t> attr_devices{0};
  cudaError_t e = raise_smem_limit_once(reinterpret_cast<const void *>(bind_tasks_kernel),
                                        kMaxTableBytes, attr_devices);
  if (e != cudaSuccess) return e;
  const size_t smem = table_bytes(batch);
  // a warp per tile, and no more blocks than are resident at once: each block rebuilds the table
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bind_tasks_kernel, kThreads, smem);
  if (e != cudaSuccess) return e;
  int64_t blocks = ((int64_t)max_tiles + kWarps - 1) / kWarps;
  const int64_t resident = (int64_t)num_sms * (per_sm < 1 ? 1 : per_sm);
  if (blocks > resident) blocks = resident;
  if (blocks < 1) blocks = 1;
  bind_tasks_kernel<<<(unsigned)blocks, kThreads, smem, stream>>>(
      q_lens, kv_lens, batch, q_tile_rows, qo_indptr, kv_indptr, q_tile_to_batch, q_tile_to_index,
      max_tiles, err);
  return cudaGetLastError();
}

}  // namespace astr
