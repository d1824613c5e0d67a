// score_decode.cuh -- paged block scorer on CUDA cores (decode rows).
//
// Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen sparse
// attention (QSA)", score equation:
//   s[t][b] = (1/sqrt(128)) * sum_{h<4} ReLU(<q[t][h], kbar[b]>)
// for the visible compressed blocks b < row_len[t]/4; decode uses the paged
// form of the scorer (keys found through the page table at full_slot/4).
//
// Design: for a few query rows per request the work is a stream of 256-byte
// keys (4 FLOP per byte per row), so the kernel is built for HBM bandwidth.
// Persistent CTAs walk tiles of 64 consecutive blocks of one request.  One
// thread feeds a 6-stage shared-memory ring with bulk asynchronous copies
// (the TMA engine, one copy per page run -- 4 KB for 64-token pages), so up
// to five tiles per CTA are in flight without holding registers.  Each
// half-warp takes one key per step from shared memory (16 lanes x 16 B,
// conflict-free); every lane keeps its 8 dims of the 4 query heads in
// registers, the 4 partial dot products are reduced across the 16 lanes with
// a reduce-scatter (5 shuffles), ReLU and the head sum follow (2 shuffles),
// and the tile's scores are staged in shared memory and written as coalesced
// rows.  Keys cross HBM once per request; all rows of the request reuse the
// staged tile.
#pragma once
#include "common.cuh"

namespace qsa {

struct ScoreArgs {
  const __nv_bfloat16* q;       // [n_rows][4][128]
  const __nv_bfloat16* pool;    // [pool_rows][128]
  int64_t pool_rows;
  int32_t n_req;
  const int32_t* req_row_start; // [n_req+1]
  int32_t n_rows;
  const int32_t* row_len;       // [n_rows]
  int32_t max_len;
  const int32_t* page_table;    // [n_req][ld_pt]
  int64_t ld_pt;
  int32_t page_size;
  float* scores;                // [n_rows][ld_scores]
  int64_t ld_scores;
  int64_t n_fill;
  int32_t trigger_dependents;   // let a dependent grid launch early (PDL)
  int32_t tiles_per_req;        // ceil(max(max_len/4, n_fill) / kScoreTile)
};

constexpr int kScoreThreads = 256;
constexpr int kScoreTile = 64;                              // blocks per tile
constexpr int kScoreStages = 6;                             // ring depth
constexpr int kScoreHalfWarps = kScoreThreads / 16;         // 16
constexpr int kScoreKeysPerHW = kScoreTile / kScoreHalfWarps;  // 4
constexpr int kScoreRowGroup = 8;                           // rows staged per pass

struct ScoreTileInfo {
  int r, b0, nb_req, row0, row1;
};

struct ScoreShared {
  __nv_bfloat16 keys[kScoreStages][kScoreTile][kDim];   // 96 KB ring
  uint64_t full[kScoreStages];
  ScoreTileInfo info[kScoreStages];
  float s_tile[kScoreRowGroup][kScoreTile];
  int s_nb[kScoreRowGroup];
  int abort_flag;
};
constexpr size_t kScoreSmem = sizeof(ScoreShared);

// Sum 4 values over the 16 lanes of a half-warp; lane l ends with the total
// of value index l >> 2 (all 4 lanes of a quad hold the same total).
__device__ __forceinline__ float reduce_scatter4_x16(float a0, float a1, float a2, float a3,
                                                     int lane16) {
  const bool up8 = lane16 & 8;
  float b0 = (up8 ? a2 : a0) + __shfl_xor_sync(0xffffffffu, up8 ? a0 : a2, 8);
  float b1 = (up8 ? a3 : a1) + __shfl_xor_sync(0xffffffffu, up8 ? a1 : a3, 8);
  const bool up4 = lane16 & 4;
  float c = (up4 ? b1 : b0) + __shfl_xor_sync(0xffffffffu, up4 ? b0 : b1, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

// Producer side (one thread): fill stage `stage` with tile slot `slot`.
__device__ __forceinline__ void score_issue_tile(const ScoreArgs& a, ScoreShared& sh, int stage,
                                                 int slot) {
  ScoreTileInfo inf;
  inf.r = slot / a.tiles_per_req;
  inf.b0 = (slot - inf.r * a.tiles_per_req) * kScoreTile;
  inf.row0 = __ldg(a.req_row_start + inf.r);
  inf.row1 = __ldg(a.req_row_start + inf.r + 1);
  if (inf.row0 < 0 || inf.row1 < inf.row0 || inf.row1 > a.n_rows) {
    raise_fault(kFaultGrouping);
    inf.row0 = inf.row1 = 0;
  }
  int nb = 0;
  for (int t = inf.row0; t < inf.row1; ++t) {
    int L = __ldg(a.row_len + t);
    if (L < 0 || L > a.max_len) { raise_fault(kFaultGrouping); L = 0; }
    nb = max(nb, L / kBlock);
  }
  inf.nb_req = nb;
  sh.info[stage] = inf;
  // Copy the tile's keys page run by page run.
  const int kpp = a.page_size / kBlock;  // keys per page
  const int end = min(nb, inf.b0 + kScoreTile);
  uint32_t bytes = 0;
  for (int pass = 0; pass < 2; ++pass) {
    // pass 0 counts the bytes (announced first), pass 1 issues the copies
    for (int b = inf.b0; b < end;) {
      const int page_idx = b / kpp;
      const int in_page = b - page_idx * kpp;
      const int n = min(kpp - in_page, end - b);
      bool ok = page_idx < a.ld_pt;
      int64_t row = 0;
      if (ok) {
        const int64_t page = __ldg(a.page_table + (int64_t)inf.r * a.ld_pt + page_idx);
        row = page * kpp + in_page;
        ok = page >= 0 && row + n <= a.pool_rows;
      }
      if (ok) {
        if (pass == 0) bytes += (uint32_t)n * (kDim * 2);
        else bulk_copy_g2s(&sh.keys[stage][b - inf.b0][0], a.pool + row * kDim,
                           (uint32_t)n * (kDim * 2), &sh.full[stage]);
      } else if (pass == 0) {
        raise_fault(page_idx < a.ld_pt ? kFaultPool : kFaultIndex);
      }
      b += n;
    }
    if (pass == 0) mbar_arrive_expect_tx(&sh.full[stage], bytes);
  }
}

__global__ void __launch_bounds__(kScoreThreads, 2)
score_decode_kernel(ScoreArgs a) {
  extern __shared__ __align__(128) unsigned char score_smem_raw[];
  ScoreShared& sh = *reinterpret_cast<ScoreShared*>(score_smem_raw);

  if (a.trigger_dependents) pdl_launch_dependents();

  const int n_slots = a.n_req * a.tiles_per_req;
  const int lane16 = threadIdx.x & 15;
  const int hw = threadIdx.x >> 4;
  // this CTA's slots: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int n_mine = blockIdx.x < n_slots ? (n_slots - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kScoreStages; ++s) mbar_init(&sh.full[s], 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int n = 0; n < kScoreStages - 1 && n < n_mine; ++n)
      score_issue_tile(a, sh, n, blockIdx.x + n * gridDim.x);

  for (int n = 0; n < n_mine; ++n) {
    const int stage = n % kScoreStages;
    if (threadIdx.x == 0 && n + kScoreStages - 1 < n_mine)
      score_issue_tile(a, sh, (n + kScoreStages - 1) % kScoreStages,
                       blockIdx.x + (n + kScoreStages - 1) * gridDim.x);
    if (!mbar_wait_bounded(&sh.full[stage], (uint32_t)(n / kScoreStages) & 1u)) {
      sh.abort_flag = 1;
      raise_fault(kFaultWait);
    }
    // B0: the tile's info (written by thread 0 before it issued the copies)
    // and the abort flag are now visible to every thread; it also orders the
    // previous tile's write-out before this tile's use of s_tile / s_nb.
    __syncthreads();
    if (sh.abort_flag) return;  // a copy never arrived: leave together
    const ScoreTileInfo inf = sh.info[stage];
    const bool any_key = inf.b0 < inf.nb_req;

    for (int g0 = inf.row0; g0 < inf.row1; g0 += kScoreRowGroup) {
      if (g0 != inf.row0) __syncthreads();  // previous group's write-out done
      const int g1 = min(inf.row1, g0 + kScoreRowGroup);
      if (threadIdx.x < g1 - g0) {
        const int L = __ldg(a.row_len + g0 + threadIdx.x);
        sh.s_nb[threadIdx.x] = (L < 0 || L > a.max_len) ? 0 : L / kBlock;
      }
      if (any_key) {
        for (int t = g0; t < g1; ++t) {
          float qv[kHeads][8];
          const __nv_bfloat16* qrow = a.q + (int64_t)t * (kHeads * kDim);
#pragma unroll
          for (int h = 0; h < kHeads; ++h) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(qrow + h * kDim + 8 * lane16));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = bf16x2_to_float2(w[e]);
              qv[h][2 * e] = f.x;
              qv[h][2 * e + 1] = f.y;
            }
          }
#pragma unroll
          for (int j = 0; j < kScoreKeysPerHW; ++j) {
            const int kk = hw + kScoreHalfWarps * j;
            const uint4 kv = *reinterpret_cast<const uint4*>(&sh.keys[stage][kk][8 * lane16]);
            const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
            float kf[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = bf16x2_to_float2(w[e]);
              kf[2 * e] = f.x;
              kf[2 * e + 1] = f.y;
            }
            float d[kHeads];
#pragma unroll
            for (int h = 0; h < kHeads; ++h) {
              float acc = 0.f;
#pragma unroll
              for (int e = 0; e < 8; ++e) acc = fmaf(qv[h][e], kf[e], acc);
              d[h] = acc;
            }
            // lane quad l>>2 holds the full dot product of head l>>2
            float sc = reduce_scatter4_x16(d[0], d[1], d[2], d[3], lane16);
            sc = fmaxf(sc, 0.f);
            sc += __shfl_xor_sync(0xffffffffu, sc, 4);
            sc += __shfl_xor_sync(0xffffffffu, sc, 8);
            if (lane16 == 0) sh.s_tile[t - g0][kk] = sc * kScoreScale;
          }
        }
      }
      __syncthreads();  // B1: the group's scores are staged
      // Coalesced write-out: visible blocks get their score, [nb_t, n_fill) -inf.
      for (int idx = threadIdx.x; idx < (g1 - g0) * kScoreTile; idx += kScoreThreads) {
        const int tr = idx / kScoreTile;
        const int kk = idx % kScoreTile;
        const int64_t b = inf.b0 + kk;
        float* dst = a.scores + (int64_t)(g0 + tr) * a.ld_scores + b;
        if (b < sh.s_nb[tr]) *dst = sh.s_tile[tr][kk];
        else if (b < a.n_fill) *dst = -__int_as_float(0x7f800000);
      }
    }
  }
}

}  // namespace qsa
