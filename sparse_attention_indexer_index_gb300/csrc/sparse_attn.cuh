// sparse_attn.cuh -- the attention the selection feeds: softmax attention
// of each query head over the original K/V rows at the selected slots.
//
// Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen sparse
// attention (QSA)": the compressed keys only index; the final softmax and
// value aggregation use the original, uncompressed K/V (sparse GQA over at
// most 2051 positions per query).  vllm-sparse-mla-blackwell, "Design notes
// worth knowing": causality belongs to the indexer, the only mask is
// index >= 0, and a token whose whole selection is masked must not come out
// as NaN (here: output 0, log-sum-exp -inf).
//
// Shapes: q [rows][H_q][D] BF16; caches k, v [n_slots][H_kv][D] BF16 (a
// physical KV slot holds all KV heads); query head h reads KV head
// h / G, G = H_q / H_kv.  out [rows][H_q][D] FP32, lse [rows][H_q] FP32.
//
// Design (GB300).  The work is a gather: per (row, KV head) about 2K rows of
// K and V (2 x D x 2 B each) against G query heads, 2 G D multiply-adds per
// 4 D bytes, so HBM-bound once the arithmetic issues few instructions.
// Flash-decoding split: one 128-thread CTA per (row, KV head, chunk of the
// row's entries).
//  1. Logits on the tensor cores (mma.sync m16n8k16, BF16 products exact,
//     FP32 accumulation): a warp takes 16 slots at a time as the rows of A,
//     loaded straight from global memory into the A fragments (the head
//     dimension permuted alike for q and k so that every load is a 16-byte
//     piece and the 4 lanes of a row read 64 contiguous bytes); the query
//     heads are the 8 columns of B, held in registers.  The CUDA-core form
//     (a butterfly reduce-scatter of per-lane partial dot products) issued
//     about 80 instructions per slot here; this one issues a few.
//  2. Per head: chunk maximum m and weights exp(logit - m), sum l.
//  3. Values: each warp accumulates sum_j w_hj v_j for its slots (weights
//     broadcast from shared memory; packed fma.rn.f32x2), the 4 warps' sums
//     are added in shared memory.
// Every warp requests into L2 the K rows of its next tile ahead of its
// loads (further look-ahead, and any for the V rows, measured slower: the
// loads in flight already cover the latency).  One chunk: the CTA
// normalises and writes out and lse; several: it writes (m, l, unnormalised
// sum) and a second kernel merges the chunks of every (row, head).
#pragma once
#include "common.cuh"

namespace qsa {

constexpr int kSaThreads = 128;
constexpr int kSaWarps = kSaThreads / 32;
constexpr int kSaMaxChunk = 256;   // entries of a row per CTA
constexpr int kSaMinChunk = 64;

struct SaArgs {
  const uint16_t* q;        // [rows][h_q][D]
  const uint16_t* k;        // [n_slots][h_kv][D]
  const uint16_t* v;
  int64_t n_slots;
  int32_t n_rows, h_q, h_kv;
  const int32_t* slots;     // [rows][ld_slots]
  int64_t ld_slots;
  int32_t n_idx;            // entries of a row read
  int32_t chunk;            // entries per CTA (multiple of 32, <= kSaMaxChunk)
  int32_t n_split;          // chunks per row
  float scale;
  float* out;               // [rows][h_q][D]
  float* lse;               // [rows][h_q] or nullptr
  float* part;              // n_split > 1: [rows][h_q][n_split][D + 2] (m, l, sum)
};

// E consecutive BF16 (E = 4 or 8) at p (aligned to 2E bytes) -> FP32.
template <int E>
__device__ __forceinline__ void sa_load_row(const uint16_t* p, float (&x)[E]) {
  if constexpr (E == 8) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
}

// E consecutive BF16 at p as E/2 FP32 pairs.
template <int E>
__device__ __forceinline__ void sa_load_row2(const uint16_t* p, float2 (&x)[E / 2]) {
  float f[E];
  sa_load_row<E>(p, f);
#pragma unroll
  for (int i = 0; i < E / 2; ++i) x[i] = make_float2(f[2 * i], f[2 * i + 1]);
}

// Two FP32 fused multiply-adds in one instruction (each rounded as fmaf).
__device__ __forceinline__ float2 sa_fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<const float2*>(&d);
}

// Butterfly reduce-scatter of 32 per-lane partial sums: afterwards x[0] of
// lane l is the warp-wide sum of value l.
__device__ __forceinline__ float sa_reduce_scatter32(float (&x)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 16, half = 16; m >= 1; m >>= 1, half >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? x[i] : x[i + half];
      const float keep = up ? x[i + half] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  return x[0];
}

// D += A B on the tensor cores: A 16 x 16 BF16 (row-major fragment a0..a3),
// B 16 x 8 BF16 (column fragment b0, b1), D 16 x 8 FP32.
__device__ __forceinline__ void sa_mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared memory of one CTA (D, G fixed by the template).
template <int G, int D>
struct SaSmem {
  int32_t slot[kSaMaxChunk];           // the chunk's slots (-1: skip)
  float logit[G][kSaMaxChunk];         // scale * <q_h, k_j>, -inf when skipped
  float w[kSaMaxChunk][G];             // weights by slot (broadcast reads)
  float m[G], l[G];
  float red[kSaWarps][G][D];           // per-warp value sums
};

template <int G, int D>
__global__ void __launch_bounds__(kSaThreads, 4)
sparse_attn_kernel(SaArgs a) {
  constexpr int E = D / 32;   // elements of a row per lane
  constexpr int P = 32 / G;   // slots per warp step
  static_assert(G * P == 32 && G * E <= 64, "unsupported group size / head dim");
  extern __shared__ __align__(16) unsigned char sa_smem_raw[];
  SaSmem<G, D>& sm = *reinterpret_cast<SaSmem<G, D>*>(sa_smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, g = blockIdx.y, t = blockIdx.z;
  const int j0 = split * a.chunk;
  const int n = max(0, min(a.chunk, a.n_idx - j0));  // entries of this chunk

  // the chunk's slots; bad ones are skipped and flagged
  for (int j = tid; j < n; j += kSaThreads) {
    int32_t s = __ldg(a.slots + (int64_t)t * a.ld_slots + j0 + j);
    if (s >= 0 && (int64_t)s >= a.n_slots) {
      raise_fault(kFaultIndex);
      s = -1;
    }
    sm.slot[j] = s;
  }
  __syncthreads();

  // ---- 1. logits on the tensor cores ---------------------------------------------
  // mma.sync m16n8k16 (BF16 in, FP32 accumulate): a warp takes 16 slots at a
  // time (rows of A), the heads are the 8 columns of B (two n-tiles for 16).
  // The head dimension is permuted the same way for q and k -- a dot
  // product does not depend on the order of its terms -- so that the A words
  // of lane (gq, tq) are 16-byte pieces of its two K rows and the 4 lanes of
  // a row read 64 contiguous bytes per load: element d = 32 (s >> 1) + 8 tq
  // + 4 (s & 1) + c plays column 2tq + (c & 1) + 8 (c >> 1) of k-step s.
  constexpr int KS = D / 16;          // k-steps
  constexpr int NT = (G + 7) / 8;     // n-tiles of 8 heads
  constexpr int QW = D / 32;          // 16-byte words of a lane (one per 32 elements)
  constexpr int kLines = D * 2 / 128; // 128-byte lines of a row
  constexpr int kAhead = 1;           // tiles of K rows requested into L2 ahead
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t bq[NT][KS][2];  // B fragments: head nt*8 + gq
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = nt * 8 + gq;
    uint4 u[QW];
#pragma unroll
    for (int i = 0; i < QW; ++i)
      u[i] = h < G ? __ldg(reinterpret_cast<const uint4*>(a.q + ((int64_t)t * a.h_q + (int64_t)g * G + h) * D) +
                           tq + 4 * i)
                   : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      bq[nt][s][0] = (s & 1) ? u[s >> 1].z : u[s >> 1].x;
      bq[nt][s][1] = (s & 1) ? u[s >> 1].w : u[s >> 1].y;
    }
  }
  // the K rows of the tile at jj into L2 (16 rows x kLines lines)
  auto prefetch_tile = [&](int jj) {
#pragma unroll
    for (int u = 0; u < (16 * kLines + 31) / 32; ++u) {
      const int idx = lane + 32 * u;
      const int r = jj + idx / kLines;
      if (idx < 16 * kLines && r < n) {
        const int s = sm.slot[r];
        if (s >= 0)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(a.k + ((int64_t)s * a.h_kv + g) * D + (idx % kLines) * 64));
      }
    }
  };
  // the first K tiles
  for (int d = 0; d < kAhead; ++d) prefetch_tile(warp * 16 + d * kSaWarps * 16);
  const float ninf = -__int_as_float(0x7f800000);
  for (int j = warp * 16; j < n; j += kSaWarps * 16) {
    prefetch_tile(j + kAhead * kSaWarps * 16);
    const int r0 = j + gq, r1 = j + gq + 8;
    const int s0 = r0 < n ? sm.slot[r0] : -1, s1 = r1 < n ? sm.slot[r1] : -1;
    uint4 ka[QW], kb[QW];
    const uint4* pa = reinterpret_cast<const uint4*>(a.k + ((int64_t)max(s0, 0) * a.h_kv + g) * D) + tq;
    const uint4* pb = reinterpret_cast<const uint4*>(a.k + ((int64_t)max(s1, 0) * a.h_kv + g) * D) + tq;
#pragma unroll
    for (int i = 0; i < QW; ++i) {
      ka[i] = s0 >= 0 ? __ldg(pa + 4 * i) : make_uint4(0u, 0u, 0u, 0u);
      kb[i] = s1 >= 0 ? __ldg(pb + 4 * i) : make_uint4(0u, 0u, 0u, 0u);
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const uint4& x = ka[s >> 1];
      const uint4& y = kb[s >> 1];
      const uint32_t a0 = (s & 1) ? x.z : x.x, a2 = (s & 1) ? x.w : x.y;
      const uint32_t a1 = (s & 1) ? y.z : y.x, a3 = (s & 1) ? y.w : y.y;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sa_mma_bf16(acc[nt], a0, a1, a2, a3, bq[nt][s][0], bq[nt][s][1]);
    }
    // acc[nt]: (slot r0, heads 2tq, 2tq+1), then (slot r1, same heads)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int h = nt * 8 + 2 * tq + c;
        if (h < G) {
          if (r0 < n) sm.logit[h][r0] = s0 >= 0 ? a.scale * acc[nt][c] : ninf;
          if (r1 < n) sm.logit[h][r1] = s1 >= 0 ? a.scale * acc[nt][2 + c] : ninf;
        }
      }
  }
  __syncthreads();

  // ---- 2. per head: maximum, weights, sum ---------------------------------------
  for (int h = warp; h < G; h += kSaWarps) {
    float mx = -__int_as_float(0x7f800000);
    for (int j = lane; j < n; j += 32) mx = fmaxf(mx, sm.logit[h][j]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int j = lane; j < n; j += 32) {
      const float lg = sm.logit[h][j];
      const float wgt = lg == -__int_as_float(0x7f800000) ? 0.f : expf(lg - mx);
      sm.w[j][h] = wgt;
      sum += wgt;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) {
      sm.m[h] = mx;
      sm.l[h] = sum;
    }
  }
  __syncthreads();

  // ---- 3. weighted value sums ---------------------------------------------------
  float2 acc[G][E / 2];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < E / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);
  constexpr int U = 4;  // value rows in flight per warp
  for (int j = warp * U; j < n; j += kSaWarps * U) {
    float2 vv[U][E / 2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int s = j + u < n ? sm.slot[j + u] : -1;  // the same for the whole warp
      if (s >= 0) {
        sa_load_row2<E>(a.v + ((int64_t)s * a.h_kv + g) * D + lane * E, vv[u]);
      } else {
#pragma unroll
        for (int e = 0; e < E / 2; ++e) vv[u][e] = make_float2(0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (j + u >= n) break;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float wgt = sm.w[j + u][h];
        const float2 w2 = make_float2(wgt, wgt);
#pragma unroll
        for (int e = 0; e < E / 2; ++e) acc[h][e] = sa_fma2(w2, vv[u][e], acc[h][e]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < E / 2; ++e)
      *reinterpret_cast<float2*>(&sm.red[warp][h][lane * E + 2 * e]) = acc[h][e];
  __syncthreads();

  // ---- 4. the chunk's result ------------------------------------------------------
  for (int idx = tid; idx < G * D; idx += kSaThreads) {
    const int h = idx / D, e = idx % D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kSaWarps; ++w) o += sm.red[w][h][e];
    const int64_t hq = (int64_t)t * a.h_q + (int64_t)g * G + h;
    if (a.n_split == 1) {
      const float l = sm.l[h];
      a.out[hq * D + e] = l > 0.f ? o / l : 0.f;
      if (e == 0 && a.lse != nullptr) a.lse[hq] = l > 0.f ? sm.m[h] + logf(l) : -__int_as_float(0x7f800000);
    } else {
      float* pp = a.part + (hq * a.n_split + split) * (D + 2);
      pp[2 + e] = o;
      if (e == 0) {
        pp[0] = sm.m[h];
        pp[1] = sm.l[h];
      }
    }
  }
}

// Merge of the chunks of every (row, query head): m = max m_s,
// l = sum l_s e^(m_s - m), out = sum o_s e^(m_s - m) / l; l = 0 -> 0, -inf.
template <int D>
__global__ void __launch_bounds__(D)
sparse_attn_merge_kernel(SaArgs a) {
  pdl_wait_primary();
  const int64_t hq = blockIdx.x;  // row * h_q + head
  const int e = threadIdx.x;
  const float* pp = a.part + hq * a.n_split * (D + 2);
  float m = -__int_as_float(0x7f800000);
  for (int s = 0; s < a.n_split; ++s) m = fmaxf(m, pp[s * (D + 2)]);
  float l = 0.f, o = 0.f;
  if (m != -__int_as_float(0x7f800000)) {
    for (int s = 0; s < a.n_split; ++s) {
      const float ms = pp[s * (D + 2)];
      if (ms == -__int_as_float(0x7f800000)) continue;
      const float c = expf(ms - m);
      l += pp[s * (D + 2) + 1] * c;
      o += pp[s * (D + 2) + 2 + e] * c;
    }
  }
  a.out[hq * D + e] = l > 0.f ? o / l : 0.f;
  if (e == 0 && a.lse != nullptr) a.lse[hq] = l > 0.f ? m + logf(l) : -__int_as_float(0x7f800000);
}

}  // namespace qsa
