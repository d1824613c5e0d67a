// score_decode.cuh -- paged block scorer on CUDA cores (decode rows).
//
// Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen sparse
// attention (QSA)", score equation:
//   s[t][b] = (1/sqrt(128)) * sum_{h<4} ReLU(<q[t][h], kbar[b]>)
// for the visible compressed blocks b < row_len[t]/4; decode uses the paged
// form of the scorer (keys found through the page table at full_slot/4).
//
// Design: the work is a stream of 256-byte keys, so the kernel is built for
// HBM bandwidth.  A CTA owns one request and a tile of 128 consecutive blocks;
// a half-warp (16 lanes x 16 B) loads one key with one coalesced 16-byte
// vector per lane, 8 keys per half-warp in flight.  Each lane keeps its 8 dims
// of the 4 query heads in registers; the 4 partial dot products are reduced
// across the 16 lanes with a reduce-scatter (5 shuffles), ReLU and the head
// sum follow in registers (2 shuffles), and the scores of a tile are staged in
// shared memory and written as coalesced rows.  Keys are read from HBM once
// per request; the rows of a request reuse them from registers.
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
};

constexpr int kScoreThreads = 256;
constexpr int kScoreTile = 128;                            // blocks per CTA
constexpr int kScoreHalfWarps = kScoreThreads / 16;         // 16
constexpr int kScoreKeysPerHW = kScoreTile / kScoreHalfWarps;  // 8
constexpr int kScoreMaxRowsSmem = 8;                        // rows staged per pass

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

__global__ void __launch_bounds__(kScoreThreads)
score_decode_kernel(ScoreArgs a) {
  __shared__ float s_tile[kScoreMaxRowsSmem][kScoreTile];
  __shared__ int s_nb[kScoreMaxRowsSmem];
  __shared__ int s_nb_req;

  if (a.trigger_dependents) pdl_launch_dependents();

  const int r = blockIdx.y;
  const int64_t b0 = (int64_t)blockIdx.x * kScoreTile;
  const int row0 = __ldg(a.req_row_start + r);
  const int row1 = __ldg(a.req_row_start + r + 1);
  const int nb_cap = a.max_len / kBlock;
  if (row0 < 0 || row1 < row0 || row1 > a.n_rows) {
    if (threadIdx.x == 0) raise_fault(kFaultGrouping);
    return;
  }

  // Visible blocks of the request (the longest of its rows).
  if (threadIdx.x == 0) s_nb_req = 0;
  __syncthreads();
  for (int t = row0 + threadIdx.x; t < row1; t += kScoreThreads) {
    int L = __ldg(a.row_len + t);
    if (L < 0 || L > a.max_len) { raise_fault(kFaultGrouping); L = 0; }
    atomicMax(&s_nb_req, L / kBlock);
  }
  __syncthreads();
  const int nb_req = min(s_nb_req, nb_cap);
  const bool any_key = b0 < nb_req;
  if (!any_key && b0 >= a.n_fill) return;

  const int lane16 = threadIdx.x & 15;
  const int hw = threadIdx.x >> 4;

  // Load this half-warp's keys (zero for blocks outside the request).
  uint4 key[kScoreKeysPerHW];
  const int rows_per_page = a.page_size / kBlock;
#pragma unroll
  for (int j = 0; j < kScoreKeysPerHW; ++j) {
    const int64_t b = b0 + hw + kScoreHalfWarps * j;
    key[j] = make_uint4(0u, 0u, 0u, 0u);
    if (b < nb_req) {
      const int64_t page_idx = b / rows_per_page;
      if (page_idx < a.ld_pt) {
        const int64_t page = __ldg(a.page_table + (int64_t)r * a.ld_pt + page_idx);
        const int64_t row = page * rows_per_page + (b - page_idx * rows_per_page);
        if (page >= 0 && row < a.pool_rows) {
          key[j] = ld_stream_16(a.pool + row * kDim + 8 * lane16);
        } else if (lane16 == 0) {
          raise_fault(kFaultPool);
        }
      } else if (lane16 == 0) {
        raise_fault(kFaultIndex);
      }
    }
  }

  for (int g0 = row0; g0 < row1; g0 += kScoreMaxRowsSmem) {
    const int g1 = min(row1, g0 + kScoreMaxRowsSmem);
    if (threadIdx.x < g1 - g0) {
      int L = __ldg(a.row_len + g0 + threadIdx.x);
      s_nb[threadIdx.x] = (L < 0 || L > a.max_len) ? 0 : L / kBlock;
    }
    if (any_key) {
      for (int t = g0; t < g1; ++t) {
        // This lane's 8 dims of the 4 heads of row t.
        float qv[kHeads][8];
        const __nv_bfloat16* qrow = a.q + (int64_t)t * (kHeads * kDim);
#pragma unroll
        for (int h = 0; h < kHeads; ++h) {
          uint4 v = __ldg(reinterpret_cast<const uint4*>(qrow + h * kDim + 8 * lane16));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 f = bf16x2_to_float2(w[e]);
            qv[h][2 * e] = f.x;
            qv[h][2 * e + 1] = f.y;
          }
        }
#pragma unroll
        for (int j = 0; j < kScoreKeysPerHW; ++j) {
          const uint32_t w[4] = {key[j].x, key[j].y, key[j].z, key[j].w};
          float kf[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 f = bf16x2_to_float2(w[e]);
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
          // Lane quad l>>2 holds the full dot product of head l>>2.
          float s = reduce_scatter4_x16(d[0], d[1], d[2], d[3], lane16);
          s = fmaxf(s, 0.f);
          s += __shfl_xor_sync(0xffffffffu, s, 4);
          s += __shfl_xor_sync(0xffffffffu, s, 8);
          if (lane16 == 0) s_tile[t - g0][hw + kScoreHalfWarps * j] = s * kScoreScale;
        }
      }
    }
    __syncthreads();
    // Coalesced write-out: valid blocks get their score, [nb_t, n_fill) -inf.
    for (int idx = threadIdx.x; idx < (g1 - g0) * kScoreTile; idx += kScoreThreads) {
      const int tr = idx / kScoreTile;
      const int64_t b = b0 + (idx % kScoreTile);
      float* dst = a.scores + (int64_t)(g0 + tr) * a.ld_scores + b;
      if (b < s_nb[tr]) *dst = s_tile[tr][idx % kScoreTile];
      else if (b < a.n_fill) *dst = -__int_as_float(0x7f800000);
    }
    __syncthreads();
  }
}

}  // namespace qsa
