// score_decode.cuh -- paged block scorer on CUDA cores (decode rows).
//
// Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen sparse
// attention (QSA)", score equation:
//   s[t][b] = (1/sqrt(128)) * sum_{h<4} ReLU(<q[t][h], kbar[b]>)
// for the visible compressed blocks b < row_len[t]/4; decode uses the paged
// form of the scorer (keys found through the page table at full_slot/4).
//
// Design: with a few query rows per request the work is a stream of 256-byte
// keys (4 FLOP per byte per row), so the kernel is built for HBM bandwidth.
// Measured on this GPU, plain 16-byte vector loads with many keys in flight
// stream scattered 4 KB pages faster than bulk-copy rings (each bulk copy
// carries a fixed cost of ~90 ns), so:
//  - Work items are tiles of 64 consecutive blocks of one request.  Every
//    CTA computes the per-request tile counts, prefix-sums them, and takes a
//    balanced contiguous range of tiles (consecutive tiles mostly share a
//    request).  CTAs are persistent: two per SM.
//  - A half-warp (16 lanes x 16 B) owns one key per step and 4 keys per
//    tile; the next tile's 4 keys are loaded into registers while the
//    current tile is computed, so loads stay in flight continuously.
//  - The query rows of the current request are staged in shared memory
//    (re-staged only when the request changes); each lane keeps its 8 dims
//    of the 4 heads of one row in registers while it walks its keys.
//  - The 4 partial dot products are reduced over the 16 lanes with a
//    reduce-scatter (5 shuffles); ReLU, the head sum (2 shuffles) and the
//    1/sqrt(128) scale follow in registers; one lane stores the FP32 score.
#pragma once
#include <cstddef>

#include "common.cuh"

namespace qsa {

struct ScoreArgs {
  const __nv_bfloat16* q;       // [n_rows][4][128]
  const __nv_bfloat16* pool;    // [pool_rows][128]
  int64_t pool_rows;
  int32_t n_req;                // requests in this launch (<= kScoreMaxReq)
  const int32_t* req_row_start; // [n_req+1] (absolute row indices)
  int32_t n_rows;
  const int32_t* row_len;       // [n_rows]
  int32_t max_len;
  const int32_t* page_table;    // [n_req][ld_pt] (row 0 = first request of the launch)
  int64_t ld_pt;
  int32_t page_size;
  float* scores;                // [n_rows][ld_scores]
  int64_t ld_scores;
  int64_t n_fill;
  int32_t trigger_dependents;   // let a dependent grid launch early (PDL)
  const int32_t* new_pos;       // see TcArgs::new_pos (TMA scorers only; others wait in full)
  // FP8 keys (mma.sync scorer only): nullptr, or the e4m3 codes [pool_rows][128]
  // and one FP32 scale per pool row; `pool` is then unused
  const uint8_t* pool8;
  const float* key_scales;
  // nullptr, or a gate per row and head [n_rows][4] (FP32) multiplying the
  // head's rectified dot product before the head sum (DSA-style head gates)
  const float* head_gates;
};

// Gate of (row, head): 1 without gates (then the products below are exact).
__device__ __forceinline__ float head_gate(const float* gates, int64_t row, int head) {
  return gates != nullptr ? __ldg(gates + row * kHeads + head) : 1.f;
}

constexpr int kScoreThreads = 256;
constexpr int kScoreHalfWarps = kScoreThreads / 16;            // 16
constexpr int kScoreKeysPerHW = 4;
constexpr int kScoreTile = kScoreHalfWarps * kScoreKeysPerHW;  // 64 blocks per tile
constexpr int kScoreRowGroup = 8;                              // q rows staged at once
constexpr int kScoreMaxReq = 4096;                             // requests per launch

struct ScoreShared {
  // read and written as 16-byte vectors: first member, 16-byte aligned
  alignas(16) __nv_bfloat16 q[kScoreRowGroup][kHeads][kDim];
  int tile_start[kScoreMaxReq + 1];
  int warp_sum[kScoreThreads / 32];
};
static_assert(offsetof(ScoreShared, q) % 16 == 0, "q stage must be 16-byte aligned");
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

// Visible blocks of request r: the longest of its rows, / 4.
__device__ __forceinline__ int request_blocks(const ScoreArgs& a, int r) {
  const int row0 = __ldg(a.req_row_start + r), row1 = __ldg(a.req_row_start + r + 1);
  if (row0 < 0 || row1 < row0 || row1 > a.n_rows) {
    raise_fault(kFaultGrouping);
    return 0;
  }
  int nb = 0;
  for (int t = row0; t < row1; ++t) {
    int L = __ldg(a.row_len + t);
    if (L < 0 || L > a.max_len) { raise_fault(kFaultGrouping); L = 0; }
    nb = max(nb, L / kBlock);
  }
  return nb;
}

// This half-warp's 8 keys of tile (r, tile j): lane16 loads bytes
// [16*lane16, 16*lane16 + 16) of each key row; keys outside the request's
// visible blocks are zero (and never stored).
__device__ __forceinline__ void load_tile_keys(const ScoreArgs& a, int r, int j, int nb_req, int hw,
                                               int lane16, uint4 (&kv)[kScoreKeysPerHW]) {
  const int kpp = a.page_size / kBlock;  // keys per page
  const int32_t* pt_row = a.page_table + (int64_t)r * a.ld_pt;
#pragma unroll
  for (int u = 0; u < kScoreKeysPerHW; ++u) {
    const int b = j * kScoreTile + hw + kScoreHalfWarps * u;
    kv[u] = make_uint4(0u, 0u, 0u, 0u);
    if (b < nb_req) {
      const int page_idx = b / kpp;
      if (page_idx < a.ld_pt) {
        const int64_t page = __ldg(pt_row + page_idx);
        const int64_t row = page * kpp + (b - page_idx * kpp);
        if (page >= 0 && row < a.pool_rows) kv[u] = ld_stream_16(a.pool + row * kDim + 8 * lane16);
        else if (lane16 == 0) raise_fault(kFaultPool);
      } else if (lane16 == 0) {
        raise_fault(kFaultIndex);
      }
    }
  }
}

__global__ void __launch_bounds__(kScoreThreads, 2)
score_decode_kernel(ScoreArgs a) {
  extern __shared__ __align__(128) unsigned char score_smem_raw[];
  ScoreShared& sh = *reinterpret_cast<ScoreShared*>(score_smem_raw);
  // Launched with programmatic serialisation: nothing is read before the
  // previous grid on the stream has finished, and the dependent selection
  // may only start once that holds here.
  pdl_wait_primary();
  if (a.trigger_dependents) pdl_launch_dependents();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lane16 = threadIdx.x & 15;
  const int hw = threadIdx.x >> 4;
  const int64_t cols_fill = a.n_fill;

  // ---- per-request tile counts and their prefix sum ---------------------
  // Tiles of request r cover max(visible blocks, n_fill) columns.  Counts are
  // computed one request per thread, then scanned in place in contiguous
  // chunks of kPer entries per thread.
  for (int r = threadIdx.x; r < a.n_req; r += kScoreThreads) {
    const int64_t nbr = request_blocks(a, r);
    const int64_t cols = nbr > cols_fill ? nbr : cols_fill;
    sh.tile_start[r] = (int)((cols + kScoreTile - 1) / kScoreTile);
  }
  __syncthreads();
  constexpr int kPer = (kScoreMaxReq + kScoreThreads - 1) / kScoreThreads;  // 16
  int local = 0;
  for (int i = 0; i < kPer; ++i) {
    const int r = threadIdx.x * kPer + i;
    if (r < a.n_req) local += sh.tile_start[r];
  }
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.warp_sum[warp] = incl;
  __syncthreads();
  int wbase = 0, total = 0;
  for (int w = 0; w < kScoreThreads / 32; ++w) {
    const int v = sh.warp_sum[w];
    if (w < warp) wbase += v;
    total += v;
  }
  int run = wbase + incl - local;
  for (int i = 0; i < kPer; ++i) {
    const int r = threadIdx.x * kPer + i;
    if (r < a.n_req) {
      const int c = sh.tile_start[r];
      sh.tile_start[r] = run;
      run += c;
    }
  }
  if (threadIdx.x == 0) sh.tile_start[a.n_req] = total;
  __syncthreads();

  // ---- this CTA's contiguous range of tiles -----------------------------
  const int t_lo = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_hi = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  if (t_lo >= t_hi) return;

  // request of a tile index: advance a cursor (ranges are ascending)
  int cur_r = 0;
  {
    int lo = 0, hi = a.n_req - 1;  // last r with tile_start[r] <= t_lo
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sh.tile_start[mid] <= t_lo) lo = mid; else hi = mid - 1;
    }
    cur_r = lo;
  }
  int next_r = cur_r;
  auto advance = [&](int tile, int& rr) {
    while (rr + 1 < a.n_req && sh.tile_start[rr + 1] <= tile) ++rr;
  };

  uint4 kcur[kScoreKeysPerHW], knext[kScoreKeysPerHW];
  int nb_next = request_blocks(a, next_r);
  load_tile_keys(a, next_r, t_lo - sh.tile_start[next_r], nb_next, hw, lane16, knext);
  int staged_r = -1, staged_g0 = -1;

  for (int tile = t_lo; tile < t_hi; ++tile) {
    // rotate the prefetched keys in, start loading the next tile's keys
    const int r = next_r;
    const int j = tile - sh.tile_start[r];
#pragma unroll
    for (int u = 0; u < kScoreKeysPerHW; ++u) kcur[u] = knext[u];
    if (tile + 1 < t_hi) {
      advance(tile + 1, next_r);
      if (next_r != r) nb_next = request_blocks(a, next_r);
      load_tile_keys(a, next_r, tile + 1 - sh.tile_start[next_r], nb_next, hw, lane16, knext);
    }
    cur_r = r;

    const int row0 = __ldg(a.req_row_start + r), row1 = __ldg(a.req_row_start + r + 1);
    const int b_base = j * kScoreTile;
    for (int g0 = row0; g0 < row1; g0 += kScoreRowGroup) {
      const int g1 = min(row1, g0 + kScoreRowGroup);
      if (staged_r != r || staged_g0 != g0) {
        // stage the group's query rows (16-byte pieces)
        __syncthreads();
        const int pieces = (g1 - g0) * (kHeads * kDim / 8);
        const uint4* src = reinterpret_cast<const uint4*>(a.q + (int64_t)g0 * kHeads * kDim);
        uint4* dst = reinterpret_cast<uint4*>(&sh.q[0][0][0]);
        for (int i = threadIdx.x; i < pieces; i += kScoreThreads) dst[i] = __ldg(src + i);
        __syncthreads();
        staged_r = r;
        staged_g0 = g0;
      }
      for (int t = g0; t < g1; ++t) {
        const int L = __ldg(a.row_len + t);
        const int nb_t = (L < 0 || L > a.max_len) ? 0 : L / kBlock;
        float* srow = a.scores + (int64_t)t * a.ld_scores;
        if (b_base < nb_t) {
          float qv[kHeads][8];
#pragma unroll
          for (int h = 0; h < kHeads; ++h) {
            const uint4 v = *reinterpret_cast<const uint4*>(&sh.q[t - g0][h][8 * lane16]);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = bf16x2_to_float2(w[e]);
              qv[h][2 * e] = f.x;
              qv[h][2 * e + 1] = f.y;
            }
          }
#pragma unroll
          for (int u = 0; u < kScoreKeysPerHW; ++u) {
            const int b = b_base + hw + kScoreHalfWarps * u;
            const uint32_t w[4] = {kcur[u].x, kcur[u].y, kcur[u].z, kcur[u].w};
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
            sc = fmaxf(sc, 0.f) * head_gate(a.head_gates, t, lane16 >> 2);
            sc += __shfl_xor_sync(0xffffffffu, sc, 4);
            sc += __shfl_xor_sync(0xffffffffu, sc, 8);
            if (lane16 == 0 && b < nb_t) srow[b] = sc * kScoreScale;
          }
        }
        // columns [nb_t, n_fill) of this tile get -inf
        const int64_t f_lo = nb_t > b_base ? nb_t : b_base;
        const int64_t f_hi = cols_fill < b_base + kScoreTile ? cols_fill : (int64_t)(b_base + kScoreTile);
        for (int64_t b = f_lo + threadIdx.x; b < f_hi; b += kScoreThreads) srow[b] = -__int_as_float(0x7f800000);
      }
    }
  }
  (void)cur_r;
}

}  // namespace qsa
