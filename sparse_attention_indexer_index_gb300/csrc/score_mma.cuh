// score_mma.cuh -- decode block scorer on the warp-level tensor-core path
// (mma.sync m16n8k16, BF16 in, FP32 accumulate), keys streamed with plain
// 16-byte loads.
//
// Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen sparse
// attention (QSA)", score equation:
//   s[t][b] = (1/sqrt(128)) * sum_{h<4} ReLU(<q[t][h], kbar[b]>)
// for the visible compressed blocks b < row_len[t]/4 of each decode row; the
// keys are found through the page table at full_slot/4.
//
// Why this shape: decode scoring is a stream of 256-byte keys with a few
// query rows per request.  Measured on this GPU, 16-byte loads issued by
// many warps stream scattered 4 KB pages at ~6.5 TB/s, while TMA and
// bulk-copy rings stop near 5.5 TB/s; the arithmetic (4 heads x rows x 128
// MACs per key) fits easily on mma.sync (~0.47 MMAs per clock per SM
// measured, a decode row needs < 0.05), so no shared-memory staging of the
// keys is needed at all:
//  - A tile is 16 consecutive blocks of one request (one MMA M): one 4 KB run
//    of pool rows when a page holds a multiple of 16 compressed keys, two
//    2 KB runs when it holds 8 (32-token pages).
//  - Lane (g, t) of a warp loads the 16-byte chunks 4c + t (c < 4) of key rows
//    g and g + 8 straight into A fragments.  The MMA's K index is a
//    permutation of the head dimension: step (c, h) pairs logical columns
//    {2t, 2t+1} / {2t+8, 2t+9} with dims 8(4c+t) + 4h + {0,1} / {2,3}; the
//    query columns (B) use the same permutation, so each B fragment is one
//    16-byte chunk of a query head.  A warp instruction reads 8 rows x 64
//    contiguous bytes.
//  - N = 8 columns = 2 rows x 4 heads per n-tile; up to 4 n-tiles (8 rows).
//    The B fragments of the current request sit in the warp's own slot of
//    shared memory (re-staged only when the request changes).
//  - Epilogue in registers: ReLU, the optional head gates, the 4-head sum
//    (one shuffle), the scale.
//  - Every CTA builds the list of tiles of all requests (prefix over the
//    requests' visible blocks); each warp takes a balanced contiguous range.
//    The loads are plain 16-byte loads from 24 warps per SM.  (Measured: a
//    4 KB bulk prefetch into L2 a few tiles ahead made the 32-request batch
//    slower, 35.5 against 31.5 us.)
//  - Page-table entries of the next 32 tiles are fetched one tile per lane.
//
// FP8 keys (kFp8): the pool holds e4m3 codes (128 bytes per key) and one
// FP32 scale per key.  Lane (g, t) loads the 16-byte chunks 4c + t (c < 2)
// of rows g and g + 8 (16 dims each); the codes become FP16 in registers
// (exact) and the MMA runs on FP16 with the query held in FP16: step (c, j)
// pairs logical columns {2t, 2t+1} / {2t+8, 2t+9} with dims
// 16(4c+t) + 4j + {0,1} / {2,3}.  The accumulator times the key's scale is
// the dot product with the dequantised key.  For one-row requests a tile
// holds 32 FP8 keys (rows g, g + 8, g + 16, g + 24: 4 KB, as a BF16 tile),
// so the per-tile work (page rows, request lookup, epilogue set-up) is spread
// over as many bytes as with BF16 keys.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "score_decode.cuh"

namespace qsa {

constexpr int kSmWarps = 8;
constexpr int kSmThreads = 32 * kSmWarps;
constexpr int kSmTile = 16;        // keys per tile (MMA M); FP8 tiles of one-row requests hold 32 (two MMA M)
// Keys per tile: 4 KB of BF16 keys; FP8 keys of one-row requests take 32
// (4 KB of codes; with more rows the second accumulator set would spill).
template <int NT, bool kFp8>
__host__ __device__ constexpr int sm_tile() { return kFp8 && NT == 1 ? 32 : 16; }
constexpr int kSmMaxRows = 8;      // rows per request: 4 n-tiles of 2 rows x 4 heads
constexpr int kSmMaxReq = 4096;    // requests per launch (tile prefix in shared memory)
constexpr int kSmMinCtas = 2;      // CTAs per SM the register budget is sized for

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e4m3 codes (low byte first) -> two FP16 values packed low first.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// A tile's key fragments of one lane: BF16 keys use a[0..3] / b[0..3]
// (chunks of rows g / g + 8), FP8 keys a[0..1] / b[0..1] and the two rows'
// scales.
struct SmFrag {
  uint4 a[4], b[4];
  float sa, sb, sc, sd;
};

// Dynamic shared memory of one CTA: the tile prefix, then per warp a slot of
// NT x 4 x 32 B fragments (16 bytes each).
__host__ __device__ constexpr size_t sm_smem_bytes(int n_req, int nt) {
  return (((size_t)(n_req + 1) * 4 + 15) & ~(size_t)15) + (size_t)kSmWarps * nt * 4 * 32 * 16;
}

template <int NT, bool kFp8>
__global__ void __launch_bounds__(kSmThreads, kSmMinCtas) score_mma_kernel(ScoreArgs a) {
  extern __shared__ __align__(16) unsigned char sm_raw[];
  int* g_pre = reinterpret_cast<int*>(sm_raw);  // [n_req + 1]: tiles before request r
  uint4* bslot_all = reinterpret_cast<uint4*>(sm_raw + ((((size_t)a.n_req + 1) * 4 + 15) & ~(size_t)15));
  __shared__ int s_wsum[kSmWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint4* bslot = bslot_all + (size_t)warp * NT * 4 * 32;  // [nt][c][lane]
  constexpr int kTile = sm_tile<NT, kFp8>();
  constexpr int kRuns = kTile / 8;        // 8-key runs of pool rows per tile

  // Without new_pos nothing is read before the previous grid completes.
  // With it (the key path of the same step runs before): the metadata, the
  // queries and keys the key path does not write are read at once; a warp
  // waits before its first tile that reaches block new_pos[r] / 4.
  const bool relaxed = a.new_pos != nullptr;
  if (!relaxed) pdl_wait_primary();
  if (a.trigger_dependents) pdl_launch_dependents();

  // One request (a verify step, a lone decode row): the tile list follows
  // from max_len alone and the request's metadata is loaded here, beside the
  // page-table entries below, so that the keys are one memory round trip
  // away instead of four (metadata, row lengths, page table, new_pos).
  // Tiles past the request's blocks load nothing.  A row list that does not
  // start at row 0 reads its lengths again after the start is known.
  const bool single = a.n_req == 1;
  int pf_rs0 = 0, pf_rs1 = 0, pf_np = 0, pf_len = 0;
  if (single) {
    pf_rs0 = __ldg(a.req_row_start);
    pf_rs1 = __ldg(a.req_row_start + 1);
    if (relaxed) pf_np = __ldg(a.new_pos);
    if (lane < min(a.n_rows, 2 * NT)) pf_len = __ldg(a.row_len + lane);
  }

  // ---- tile list: ceil(nb_r / 16) tiles per request, prefix in shared memory
  if (single) {
    if (threadIdx.x == 0) {
      g_pre[0] = 0;
      g_pre[1] = (a.max_len / kBlock + kTile - 1) / kTile;
    }
    __syncthreads();
  } else {
    const int per = (a.n_req + kSmThreads - 1) / kSmThreads;
    const int r_lo = min(a.n_req, (int)threadIdx.x * per), r_hi = min(a.n_req, r_lo + per);
    int local = 0;
    for (int r = r_lo; r < r_hi; ++r) {
      local += (request_blocks(a, r) + kTile - 1) / kTile;
      g_pre[r + 1] = local;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int before = incl - local;
    for (int w = 0; w < warp; ++w) before += s_wsum[w];
    for (int r = r_lo; r < r_hi; ++r) g_pre[r + 1] += before;
    if (threadIdx.x == 0) g_pre[0] = 0;
    __syncthreads();
  }
  const int64_t T = g_pre[a.n_req];
  const int64_t W = (int64_t)gridDim.x * kSmWarps;
  const int64_t gw = (int64_t)blockIdx.x * kSmWarps + warp;
  const int i0 = (int)(T * gw / W), i1 = (int)(T * (gw + 1) / W);
  // With new_pos, thread 0 of CTA 0 waits for the previous grid before it
  // leaves, so that this grid still completes after it.
  const bool anchor = relaxed && blockIdx.x == 0 && threadIdx.x == 0;
  if (i0 >= i1) {
    if (anchor) pdl_wait_primary();
    return;
  }

  const int kpp = a.page_size / kBlock;  // compressed keys per page (a multiple of 8 here)
  // Request of tile i: last r with g_pre[r] <= i (binary search).
  auto request_of = [&](int i) {
    int lo = 0, hi = a.n_req - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (g_pre[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // Pool rows of tile i's 8-key runs (a run never straddles a page: pages
  // hold a multiple of 8 keys); -1 if a page is out of range or the run lies
  // past the request's blocks (its last tile only: no page-table entry is
  // read there).  One request: the tile list may reach past the request's
  // blocks, so an out-of-range entry gives kRunBadIndex / kRunBadPool and
  // faults at the load only if the run's first block is below the length.
  constexpr int kRunBadIndex = -2, kRunBadPool = -3;
  auto run_row = [&](int r, int b) -> int {
    const int page_idx = b / kpp;
    if (page_idx >= a.ld_pt) {
      if (single) return kRunBadIndex;
      raise_fault(kFaultIndex);
      return -1;
    }
    const int64_t page = __ldg(a.page_table + (int64_t)r * a.ld_pt + page_idx);
    const int64_t row = page * kpp + (int64_t)(b - page_idx * kpp);
    if (page < 0 || row >= a.pool_rows) {
      if (single) return kRunBadPool;
      raise_fault(kFaultPool);
      return -1;
    }
    return (int)row;
  };
  auto tile_rows = [&](int i, int (&rr)[kRuns]) {
#pragma unroll
    for (int q = 0; q < kRuns; ++q) rr[q] = -1;
    if (i >= i1) return;
    const int r = request_of(i);
    const int b = (i - g_pre[r]) * kTile;
    const int nbv = !single && i == g_pre[r + 1] - 1 ? request_blocks(a, r) : INT_MAX;
#pragma unroll
    for (int q = 0; q < kRuns; ++q) {
      const int bq = b + 8 * q;
      if (bq >= nbv) break;
      rr[q] = (q > 0 && bq % kpp != 0) ? (rr[q - 1] >= 0 ? rr[q - 1] + 8 : -1) : run_row(r, bq);
    }
  };
  int base = i0;
  int pr_cur[kRuns], pr_nxt[kRuns];
  tile_rows(i0 + lane, pr_cur);
  tile_rows(i0 + 32 + lane, pr_nxt);
  auto rows_of = [&](int i, int (&rr)[kRuns]) {  // warp-uniform i in [base, base + 64)
    const int d = i - base;
#pragma unroll
    for (int q = 0; q < kRuns; ++q) rr[q] = __shfl_sync(0xffffffffu, d < 32 ? pr_cur[q] : pr_nxt[q], d & 31);
  };
  // ---- load side: the tile's request, its longest row, the PDL wait -------
  int r_ld = -1, nb_ld = 0, fn_ld = INT_MAX;
  bool waited = !relaxed;
  auto load_tile = [&](int i, SmFrag& f) {
    if (i - base >= 32) {  // next batch of pool rows
      base += 32;
#pragma unroll
      for (int q = 0; q < kRuns; ++q) pr_cur[q] = pr_nxt[q];
      tile_rows(base + 32 + lane, pr_nxt);
    }
    if (r_ld < 0 || i >= g_pre[r_ld + 1]) {
      if (r_ld < 0) r_ld = request_of(i);
      while (i >= g_pre[r_ld + 1]) ++r_ld;  // g_pre is non-decreasing: empty requests are skipped
      int L;
      if (single) {  // the loads issued at the start
        const int nrl = min(pf_rs1 - pf_rs0, 2 * NT);
        L = lane < nrl ? (pf_rs0 == 0 ? pf_len : __ldg(a.row_len + pf_rs0 + lane)) : 0;
        fn_ld = relaxed ? max(0, pf_np) / kBlock : INT_MAX;
      } else {
        const int t0l = __ldg(a.req_row_start + r_ld);
        const int nrl = min(__ldg(a.req_row_start + r_ld + 1) - t0l, 2 * NT);
        L = lane < nrl ? __ldg(a.row_len + t0l + lane) : 0;
        fn_ld = relaxed ? max(0, __ldg(a.new_pos + r_ld)) / kBlock : INT_MAX;
      }
      if (L < 0 || L > a.max_len) L = 0;
      nb_ld = __reduce_max_sync(0xffffffffu, (unsigned)(L / kBlock));
    }
    const int j = i - g_pre[r_ld];
    const int vis = min(kTile, nb_ld - j * kTile);
    if (!waited && vis > 0 && kTile * (j + 1) > fn_ld) {  // this tile may hold keys the key path writes
      pdl_wait_primary();
      waited = true;
    }
    int pr[kRuns];
    rows_of(i, pr);
    if (single) {  // deferred page faults: only runs below the request's length
#pragma unroll
      for (int q = 0; q < kRuns; ++q)
        if (pr[q] <= kRunBadIndex && 8 * q < vis && lane == 0) raise_fault(pr[q] == kRunBadIndex ? kFaultIndex : kFaultPool);
    }
    // key row g of each run (rows past the request's blocks: zero)
    bool v[kRuns];
    bool bad = false;
#pragma unroll
    for (int q = 0; q < kRuns; ++q) {
      v[q] = pr[q] >= 0 && g + 8 * q < vis;
      if (v[q] && pr[q] + g >= a.pool_rows) {
        bad = true;
        v[q] = false;
      }
    }
    if (bad) raise_fault(kFaultPool);
    const int pra = pr[0], prb = pr[1];
    const bool va = v[0], vb = v[1];
    if (kFp8) {
      // runs 0/1 (rows g, g + 8) in a/b[0..1], runs 2/3 (rows g + 16, g + 24)
      // in a/b[2..3]: chunks 4c + t (c < 2) of each row, 16 dims each
#pragma unroll
      for (int h = 0; h < kRuns / 2; ++h) {
        const int q0 = 2 * h, q1 = 2 * h + 1;
        const uint8_t* ra = a.pool8 + ((int64_t)max(pr[q0], 0) + g) * kDim + 16 * t;
        const uint8_t* rb = a.pool8 + ((int64_t)max(pr[q1], 0) + g) * kDim + 16 * t;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          f.a[2 * h + c] = v[q0] ? ld_stream_16(ra + 64 * c) : make_uint4(0u, 0u, 0u, 0u);
          f.b[2 * h + c] = v[q1] ? ld_stream_16(rb + 64 * c) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      f.sa = v[0] ? __ldg(a.key_scales + max(pr[0], 0) + g) : 0.f;
      f.sb = v[1] ? __ldg(a.key_scales + max(pr[1], 0) + g) : 0.f;
      if constexpr (kRuns == 4) {
        f.sc = v[2] ? __ldg(a.key_scales + max(pr[2], 0) + g) : 0.f;
        f.sd = v[3] ? __ldg(a.key_scales + max(pr[3], 0) + g) : 0.f;
      }
    } else {
      const __nv_bfloat16* ra = a.pool + ((int64_t)max(pra, 0) + g) * kDim + 8 * t;
      const __nv_bfloat16* rb = a.pool + ((int64_t)max(prb, 0) + g) * kDim + 8 * t;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        f.a[c] = va ? ld_stream_16(ra + 32 * c) : make_uint4(0u, 0u, 0u, 0u);
        f.b[c] = vb ? ld_stream_16(rb + 32 * c) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };

  // ---- compute side: query fragments of the tile's request, row lengths ---
  int r = -1, t0 = 0, nrows = 0;
  int nbr[NT];
  float gate_a[NT], gate_b[NT];  // gates of this lane's two heads (columns 2t, 2t+1) of row 2nt + t/2
  auto compute_tile = [&](int i, const SmFrag& f) {
    if (r < 0 || i >= g_pre[r + 1]) {
      if (r < 0) r = request_of(i);
      while (i >= g_pre[r + 1]) ++r;
      t0 = __ldg(a.req_row_start + r);
      nrows = min(__ldg(a.req_row_start + r + 1) - t0, 2 * NT);
      if (__ldg(a.req_row_start + r + 1) - t0 > 2 * NT && lane == 0) raise_fault(kFaultGrouping);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int rl = 2 * nt + (t >> 1);
        int nb = 0;
        gate_a[nt] = gate_b[nt] = 1.f;
        if (rl < nrows) {
          const int L = __ldg(a.row_len + t0 + rl);
          nb = (L >= 0 && L <= a.max_len) ? L / kBlock : 0;
          gate_a[nt] = head_gate(a.head_gates, t0 + rl, 2 * (t & 1));
          gate_b[nt] = head_gate(a.head_gates, t0 + rl, 2 * (t & 1) + 1);
        }
        nbr[nt] = nb;
      }
      __syncwarp();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int rl = 2 * nt + (g >> 2), head = g & 3;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          // BF16: chunk 4c + t of the head (8 dims); FP8 path: dims
          // 16(4(c/2) + t) + 8(c%2) .. +7 as FP16
          const int d0 = kFp8 ? 16 * (4 * (c >> 1) + t) + 8 * (c & 1) : 8 * (4 * c + t);
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (rl < nrows)
            v = __ldg(reinterpret_cast<const uint4*>(a.q + ((int64_t)(t0 + rl) * kHeads + head) * kDim + d0));
          if (kFp8) {  // BF16 -> FP16, nearest (exact for |q| in [2^-14, 65504) and BF16's 8 bits)
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 p = bf16x2_to_float2(w[e]);
              const __half2 h = __floats2half2_rn(p.x, p.y);
              w[e] = *reinterpret_cast<const uint32_t*>(&h);
            }
            v = make_uint4(w[0], w[1], w[2], w[3]);
          }
          bslot[(nt * 4 + c) * 32 + lane] = v;
        }
      }
      __syncwarp();
    }
    const int j = i - g_pre[r];
    // One MMA M block of 16 keys at a time (FP8 tiles hold two: keys g, g + 8
    // of fragments a/b[0..1], then g + 16, g + 24 of a/b[2..3]), each
    // followed by its epilogue: ReLU, head sum (lanes t and t^1 hold the two
    // head pairs), scale.
#pragma unroll
    for (int h = 0; h < kRuns / 2; ++h) {
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      if (kFp8) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 fa = f.a[2 * h + c], fb = f.b[2 * h + c];
          const uint32_t wa[4] = {fa.x, fa.y, fa.z, fa.w};
          const uint32_t wb[4] = {fb.x, fb.y, fb.z, fb.w};
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {  // dims 16(4c+t) + 4jj + {0,1} / {2,3}
            const uint32_t a0 = e4m3x2_to_f16x2(wa[jj]), a2 = e4m3x2_to_f16x2(wa[jj] >> 16);
            const uint32_t a1 = e4m3x2_to_f16x2(wb[jj]), a3 = e4m3x2_to_f16x2(wb[jj] >> 16);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 bq = bslot[(nt * 4 + 2 * c + (jj >> 1)) * 32 + lane];
              if (jj & 1) mma_f16_16816(acc[nt], a0, a1, a2, a3, bq.z, bq.w);
              else mma_f16_16816(acc[nt], a0, a1, a2, a3, bq.x, bq.y);
            }
          }
        }
        const float s_lo = h == 0 ? f.sa : f.sc, s_hi = h == 0 ? f.sb : f.sd;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {  // dequantise: each key row by its own scale
          acc[nt][0] *= s_lo;
          acc[nt][1] *= s_lo;
          acc[nt][2] *= s_hi;
          acc[nt][3] *= s_hi;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 bq = bslot[(nt * 4 + c) * 32 + lane];
            mma_bf16_16816(acc[nt], f.a[c].x, f.b[c].x, f.a[c].y, f.b[c].y, bq.x, bq.y);
            mma_bf16_16816(acc[nt], f.a[c].z, f.b[c].z, f.a[c].w, f.b[c].w, bq.z, bq.w);
          }
        }
      }
      const int b = j * kTile + 16 * h + g;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // gated heads (gates 1 without head gates: then exactly the plain sums)
        float v0 = fmaf(gate_b[nt], fmaxf(acc[nt][1], 0.f), gate_a[nt] * fmaxf(acc[nt][0], 0.f));
        float v1 = fmaf(gate_b[nt], fmaxf(acc[nt][3], 0.f), gate_a[nt] * fmaxf(acc[nt][2], 0.f));
        v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        const int rl = 2 * nt + (t >> 1);
        if ((t & 1) == 0 && rl < nrows) {
          float* dst = a.scores + (int64_t)(t0 + rl) * a.ld_scores + b;
          if (b < nbr[nt]) dst[0] = v0 * kScoreScale;
          if (b + 8 < nbr[nt]) dst[8] = v1 * kScoreScale;
        }
      }
    }
  };

  // ---- the warp's tiles: the next tile's fragments load while this one is
  // computed (2 tiles in flight per warp; measured: 2 at 2 CTAs per SM beats
  // 1 at 3, and 3 FP8 tiles in flight gained nothing) ------------------------
  SmFrag cur;
  load_tile(i0, cur);
  for (int i = i0; i < i1; ++i) {
    SmFrag nxt;
    if (i + 1 < i1) load_tile(i + 1, nxt);
    compute_tile(i, cur);
    cur = nxt;
  }
  if (anchor && !waited) pdl_wait_primary();
}

}  // namespace qsa
