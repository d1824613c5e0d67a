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
// K and V (2 x D x 2 B each) against G query heads, 2 G D FMAs per 4 D bytes,
// so HBM-bound at the FP32 CUDA-core rate; no tensor cores.  Flash-decoding
// split: one 128-thread CTA per (row, KV head, chunk of the row's entries).
//  1. Logits: a warp takes 32 / G slots at a time, each lane D / 32
//     consecutive elements of every K row (one 8- or 16-byte load) and of
//     the G query rows (registers); the G x (32 / G) partial dot products are
//     summed by a butterfly reduce-scatter (31 shuffles for 32 sums), after
//     which lane l holds the logit of (head l / P, slot l % P).
//  2. Per head: chunk maximum m and weights exp(logit - m), sum l.
//  3. Values: each warp accumulates sum_j w_hj v_j for its slots (weights
//     broadcast from shared memory; packed fma.rn.f32x2), the 4 warps' sums
//     are added in shared memory.  Every warp requests the K (then V) rows
//     of its next 4 steps into L2 ahead of its loads.  One chunk: the CTA normalises and writes out and lse;
//     several: it writes (m, l, unnormalised sum) and a second kernel merges
//     the chunks of every (row, head).
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
  // this lane's part of the G query rows
  float2 qv[G][E / 2];
#pragma unroll
  for (int h = 0; h < G; ++h)
    sa_load_row2<E>(a.q + ((int64_t)t * a.h_q + (int64_t)g * G + h) * D + lane * E, qv[h]);
  __syncthreads();

  // ---- 1. logits ----------------------------------------------------------------
  constexpr int kLines = D * 2 / 128;  // 128-byte lines of a row
  constexpr int kAhead = 4;            // warp steps of rows requested into L2 ahead
  // the K rows of this warp's step `jj` into L2 (P rows x kLines lines)
  auto prefetch_rows = [&](const uint16_t* base, int jj, int rows) {
    if (lane < rows * kLines) {
      const int s = jj + lane / kLines < n ? sm.slot[jj + lane / kLines] : -1;
      if (s >= 0)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(base + ((int64_t)s * a.h_kv + g) * D + (lane % kLines) * 64));
    }
  };
  for (int d = 0; d < kAhead; ++d) prefetch_rows(a.k, warp * P + d * kSaWarps * P, P);
  for (int d = 0; d < kAhead; ++d) prefetch_rows(a.v, warp * 4 + d * kSaWarps * 4, 4);
  for (int j = warp * P; j < n; j += kSaWarps * P) {
    prefetch_rows(a.k, j + kAhead * kSaWarps * P, P);
    float2 kv[P][E / 2];
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const int s = j + i < n ? sm.slot[j + i] : -1;
      if (s >= 0) {
        sa_load_row2<E>(a.k + ((int64_t)s * a.h_kv + g) * D + lane * E, kv[i]);
      } else {
#pragma unroll
        for (int e = 0; e < E / 2; ++e) kv[i][e] = make_float2(0.f, 0.f);
      }
    }
    float x[32];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < P; ++i) {
        float2 acc = make_float2(0.f, 0.f);  // even and odd elements
#pragma unroll
        for (int e = 0; e < E / 2; ++e) acc = sa_fma2(qv[h][e], kv[i][e], acc);
        x[h * P + i] = acc.x + acc.y;
      }
    const float dot = sa_reduce_scatter32(x);
    const int h = lane / P, i = lane % P;
    if (j + i < n) sm.logit[h][j + i] = sm.slot[j + i] >= 0 ? a.scale * dot : -__int_as_float(0x7f800000);
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
    prefetch_rows(a.v, j + kAhead * kSaWarps * U, U);
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
