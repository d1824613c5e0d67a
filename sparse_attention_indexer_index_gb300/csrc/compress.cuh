// compress.cuh -- compressed index keys of the QSA indexer.
//
// Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen sparse
// attention (QSA)": each block of 4 raw index keys becomes one key -- the FP32
// average of the four, normalised, then rotated by the position encoding of
// the block's first token -- kept as BF16 in a paged cache addressed
// page-aligned at full_slot/4.
//
// Readings: "normalised" is the L2 norm (a zero mean stays zero); for text
// positions the multi-section RoPE reduces to plain RoPE over all 128 dims
// with rotate-half pairs (i, i+64) and angle p * base^(-2i/128).
//
// Work split: 8 lanes per block; lane j owns dims [8j, 8j+8) and
// [64+8j, 64+8j+8), i.e. exactly the rotation pairs it needs, so every load
// and store is one 16-byte vector and only the norm needs shuffles.
//
// Angle: p * base^(-2i/128) grows to ~1.3e5 rad at 131k tokens, so it is
// reduced exactly: t_i = base^(-2i/128) / (2 pi) is held as a 64-bit binary
// fraction of a turn, p * t_i mod 1 is a wrapping 64-bit integer product, and
// the top 32 bits give the angle in units of pi for sincospif.  Error
// < 3e-7 rad for p < 2^31.  The 64 fractions depend only on the RoPE base;
// the launching host code derives them once per base in FP64 and passes them
// as a kernel parameter (FP64 arithmetic is slow on this GPU: one pow per
// thread cost ~8 us of latency).
#pragma once
#include <cuda_fp8.h>

#include "common.cuh"

namespace qsa {

struct CompressArgs {
  const __nv_bfloat16* raw;   // [n_blocks*4][128]
  const int32_t* block_req;   // [n_blocks]
  const int32_t* block_id;    // [n_blocks]
  int64_t n_blocks;
  int32_t n_req;
  const int32_t* page_table;  // [n_req][ld_pt] or nullptr
  int64_t ld_pt;
  int32_t page_size;
  double rope_base;
  __nv_bfloat16* pool;        // [pool_rows][128]
  int64_t pool_rows;
};

// Rotation frequency i as a 64-bit fraction of a turn: base^(-2i/128)/(2 pi).
struct RopeTurns {
  uint64_t frac[kDim / 2];
};

constexpr int kCompressThreads = 256;
constexpr int kCompressLanes = 8;  // lanes per block

__device__ __forceinline__ void accumulate_bf16x8(float (&acc)[8], uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float2 f = bf16x2_to_float2(w[e]);
    acc[2 * e] = acc[2 * e] + f.x;
    acc[2 * e + 1] = acc[2 * e + 1] + f.y;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// sin and cos of the RoPE angle pos * t, with t a 64-bit fraction of a turn:
// pos * t mod 1 as a wrapping integer product, its top 32 bits (signed, half a
// turn either way) as the angle in units of pi.
__device__ __forceinline__ void rope_sincos(uint32_t pos, uint64_t turn_frac, float& s, float& c) {
  const uint64_t ph = (uint64_t)pos * turn_frac;               // turns mod 1, wraps
  const int32_t top = (int32_t)(ph >> 32);                     // signed: [-1/2, 1/2) turn
  const float y = (float)top * 4.656612873077392578125e-10f;   // * 2^-31: units of pi
  sincospif(y, &s, &c);
}

// One block compressed by the 8 lanes of a group: lane8 holds dims
// [8 lane8, +8) and [64 + 8 lane8, +8) of the 4 raw keys (vlo, vhi) and
// writes the same dims of the compressed key at dst.  The 8 lanes of a
// group always reach this together.
__device__ __forceinline__ void compress_block_8(const uint4 (&vlo)[kBlock], const uint4 (&vhi)[kBlock],
                                                 uint32_t pos, const uint64_t (&turn_frac)[8],
                                                 __nv_bfloat16* dst, int lane8) {
  // FP32 block mean, summed in token order: ((k0 + k1) + k2) + k3, * 0.25.
  float lo[8], hi[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 fx = bf16x2_to_float2((&vlo[0].x)[e]), fy = bf16x2_to_float2((&vhi[0].x)[e]);
    lo[2 * e] = fx.x; lo[2 * e + 1] = fx.y;
    hi[2 * e] = fy.x; hi[2 * e + 1] = fy.y;
  }
#pragma unroll
  for (int k = 1; k < kBlock; ++k) {
    accumulate_bf16x8(lo, vlo[k]);
    accumulate_bf16x8(hi, vhi[k]);
  }
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    lo[e] *= 0.25f;
    hi[e] *= 0.25f;
    ss = fmaf(lo[e], lo[e], ss);
    ss = fmaf(hi[e], hi[e], ss);
  }
  // The 8 lanes of a block always take the same path, so the shuffles name
  // only their own group.
  const unsigned group = 0xffu << (threadIdx.x & 24);
  ss += __shfl_xor_sync(group, ss, 1);
  ss += __shfl_xor_sync(group, ss, 2);
  ss += __shfl_xor_sync(group, ss, 4);
  const float inv_norm = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;

  uint32_t out_lo[4], out_hi[4];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float r_lo[2], r_hi[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float s, c;
      rope_sincos(pos, turn_frac[e + h], s, c);
      const float u = lo[e + h] * inv_norm, v = hi[e + h] * inv_norm;
      r_lo[h] = u * c - v * s;
      r_hi[h] = v * c + u * s;
    }
    out_lo[e / 2] = pack_bf16x2(r_lo[0], r_lo[1]);
    out_hi[e / 2] = pack_bf16x2(r_hi[0], r_hi[1]);
  }
  *reinterpret_cast<uint4*>(dst + 8 * lane8) = make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
  *reinterpret_cast<uint4*>(dst + 64 + 8 * lane8) =
      make_uint4(out_hi[0], out_hi[1], out_hi[2], out_hi[3]);
}

__global__ void __launch_bounds__(kCompressThreads)
compress_keys_kernel(CompressArgs a, const __grid_constant__ RopeTurns turns) {
  // A dependent grid (launched with programmatic serialisation) may start
  // its own set-up now; it waits for this grid before reading the pool.
  pdl_launch_dependents();
  const int lane8 = threadIdx.x & (kCompressLanes - 1);
  uint64_t turn_frac[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) turn_frac[e] = turns.frac[kCompressLanes * lane8 + e];

  const int64_t groups_per_cta = kCompressThreads / kCompressLanes;
  const int64_t stride = (int64_t)gridDim.x * groups_per_cta;
  for (int64_t blk = (int64_t)blockIdx.x * groups_per_cta + threadIdx.x / kCompressLanes;
       blk < a.n_blocks; blk += stride) {
    // Everything indexed by blk is loaded up front, so only the page-table
    // entry waits on another load.
    const int64_t b = a.block_id[blk];
    const int r = a.page_table != nullptr ? a.block_req[blk] : 0;
    const __nv_bfloat16* src = a.raw + blk * (kBlock * kDim);
    uint4 vlo[kBlock], vhi[kBlock];
#pragma unroll
    for (int k = 0; k < kBlock; ++k) {
      vlo[k] = ld_stream_16(src + k * kDim + 8 * lane8);
      vhi[k] = ld_stream_16(src + k * kDim + 64 + 8 * lane8);
    }
    // Destination pool row: slot of the block's first token, divided by 4
    // (positions are int32, so the page arithmetic is 32-bit).
    const uint32_t pos = (uint32_t)(kBlock * b);
    int64_t row = blk;
    bool ok = b >= 0 && b <= INT32_MAX / kBlock;
    if (a.page_table != nullptr && ok) {
      const uint32_t ps = (uint32_t)a.page_size;
      const uint32_t page_idx = pos / ps;
      ok = r >= 0 && r < a.n_req && (int64_t)page_idx < a.ld_pt;
      if (ok) {
        const int64_t page = a.page_table[(int64_t)r * a.ld_pt + page_idx];
        row = page * (int64_t)(ps / kBlock) + (int64_t)((pos - page_idx * ps) / kBlock);
        ok = page >= 0;
      }
    }
    if (!ok) {
      if (lane8 == 0) raise_fault(kFaultIndex);
      continue;
    }
    if (row < 0 || row >= a.pool_rows) {
      if (lane8 == 0) raise_fault(kFaultPool);
      continue;
    }

    compress_block_8(vlo, vhi, pos, turn_frac, a.pool + row * kDim, lane8);
  }
}

// Key path of a decode step: request r appends raw keys at positions
// first_pos[r] + i into its 4-slot ring (slot p mod 4) and compresses every
// block those positions complete -- the raw keys of this call where
// present, the ring's (earlier calls) otherwise -- into the pool at
// slot(4b)/4.  Same source as compress_keys_kernel for the arithmetic.
// One 64-thread CTA per request: 8 groups of 8 lanes compress the completed
// blocks (reading the ring as it was), then, after a barrier, the ring takes
// the last 4 appended keys.
struct AppendArgs {
  const __nv_bfloat16* keys;      // [n_tok][128]
  const int32_t* req_tok_start;   // [n_req+1]
  const int32_t* req_first_pos;   // [n_req]
  int32_t n_req;
  __nv_bfloat16* ring;            // [n_req][4][128]
  const int32_t* page_table;      // [n_req][ld_pt]
  int64_t ld_pt;
  int32_t page_size;
  __nv_bfloat16* pool;            // [pool_rows][128]
  int64_t pool_rows;
};

constexpr int kAppendThreads = 64;

__global__ void __launch_bounds__(kAppendThreads)
append_keys_kernel(AppendArgs a, const __grid_constant__ RopeTurns turns) {
  pdl_launch_dependents();
  const int r = blockIdx.x;
  const int lane8 = threadIdx.x & (kCompressLanes - 1), grp = threadIdx.x / kCompressLanes;
  const int start = __ldg(a.req_tok_start + r), end = __ldg(a.req_tok_start + r + 1);
  const int p0 = __ldg(a.req_first_pos + r);
  const int n = end - start;
  if (n <= 0) return;
  if (start < 0 || p0 < 0 || (int64_t)p0 + n > (int64_t)INT32_MAX) {
    if (threadIdx.x == 0) raise_fault(kFaultGrouping);
    return;
  }
  uint64_t turn_frac[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) turn_frac[e] = turns.frac[kCompressLanes * lane8 + e];
  __nv_bfloat16* ring = a.ring + (int64_t)r * kBlock * kDim;
  const __nv_bfloat16* keys = a.keys + (int64_t)start * kDim;

  // blocks b with 4b+3 in [p0, p0+n-1]
  const int b_first = p0 / kBlock;
  const int b_last = (p0 + n - kBlock) >= 0 ? (p0 + n - kBlock) / kBlock : -1;
  for (int b = b_first + grp; b <= b_last; b += kAppendThreads / kCompressLanes) {
    uint4 vlo[kBlock], vhi[kBlock];
#pragma unroll
    for (int c = 0; c < kBlock; ++c) {
      const int q = kBlock * b + c;
      const __nv_bfloat16* src = q >= p0 ? keys + (int64_t)(q - p0) * kDim : ring + c * kDim;
      vlo[c] = *reinterpret_cast<const uint4*>(src + 8 * lane8);
      vhi[c] = *reinterpret_cast<const uint4*>(src + 64 + 8 * lane8);
    }
    const uint32_t pos = (uint32_t)(kBlock * b);
    const uint32_t ps = (uint32_t)a.page_size;
    const uint32_t page_idx = pos / ps;
    int64_t row = -1;
    if ((int64_t)page_idx < a.ld_pt) {
      const int64_t page = a.page_table[(int64_t)r * a.ld_pt + page_idx];
      if (page >= 0) row = page * (int64_t)(ps / kBlock) + (int64_t)((pos - page_idx * ps) / kBlock);
    }
    if (row < 0) {
      if (lane8 == 0) raise_fault(kFaultIndex);
      continue;
    }
    if (row >= a.pool_rows) {
      if (lane8 == 0) raise_fault(kFaultPool);
      continue;
    }
    compress_block_8(vlo, vhi, pos, turn_frac, a.pool + row * kDim, lane8);
  }
  __syncthreads();  // every read of the ring is done
  // the ring keeps the key of every appended position, the last 4 win
  const int i0 = n > kBlock ? n - kBlock : 0;
  for (int x = threadIdx.x; x < (n - i0) * (kDim / 8); x += kAppendThreads) {
    const int i = i0 + x / (kDim / 8), part = x % (kDim / 8);
    const int slot = (p0 + i) % kBlock;
    *reinterpret_cast<uint4*>(ring + slot * kDim + 8 * part) =
        *reinterpret_cast<const uint4*>(keys + (int64_t)i * kDim + 8 * part);
  }
}

}  // namespace qsa

namespace qsa {

// ---------------------------------------------------------------------------
// Prologue tails (SGLang GLM-5.2 blog, section "Indexer Prologue Fusion": the
// query path applies RoPE and FP8 quantisation, the key path FP8 quantisation
// before the paged index-cache store).
// ---------------------------------------------------------------------------

// Query RoPE: the 4 heads of row t rotated at position pos[t] (the newest
// token the row sees), rotate-half pairs (i, i+64), the angle reduced exactly
// as in the key path; one BF16 rounding.  8 lanes per (row, head): lane j owns
// dims [8j, 8j+8) and their partners [64+8j, ...).
struct RopeQArgs {
  const __nv_bfloat16* q;   // [n_rows][4][128]
  const int32_t* pos;       // [n_rows]
  int32_t n_rows;
  __nv_bfloat16* out;       // [n_rows][4][128] (may be q)
};
constexpr int kRopeQThreads = 256;

__global__ void __launch_bounds__(kRopeQThreads)
rope_queries_kernel(RopeQArgs a, const __grid_constant__ RopeTurns turns) {
  pdl_launch_dependents();  // the scorer may start its set-up; it waits for the queries
  const int lane8 = threadIdx.x & (kCompressLanes - 1);
  const int64_t unit = (int64_t)blockIdx.x * (kRopeQThreads / kCompressLanes) + threadIdx.x / kCompressLanes;
  if (unit >= (int64_t)a.n_rows * kHeads) return;
  const int p = __ldg(a.pos + unit / kHeads);
  if (p < 0) {
    if (lane8 == 0) raise_fault(kFaultGrouping);
    return;
  }
  const __nv_bfloat16* src = a.q + unit * kDim;
  const uint4 lo4 = ld_stream_16(src + 8 * lane8), hi4 = ld_stream_16(src + 64 + 8 * lane8);
  const uint32_t lo[4] = {lo4.x, lo4.y, lo4.z, lo4.w}, hi[4] = {hi4.x, hi4.y, hi4.z, hi4.w};
  uint32_t out_lo[4], out_hi[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 u = bf16x2_to_float2(lo[e]), v = bf16x2_to_float2(hi[e]);
    float s0, c0, s1, c1;
    rope_sincos((uint32_t)p, turns.frac[8 * lane8 + 2 * e], s0, c0);
    rope_sincos((uint32_t)p, turns.frac[8 * lane8 + 2 * e + 1], s1, c1);
    out_lo[e] = pack_bf16x2(u.x * c0 - v.x * s0, u.y * c1 - v.y * s1);
    out_hi[e] = pack_bf16x2(v.x * c0 + u.x * s0, v.y * c1 + u.y * s1);
  }
  __nv_bfloat16* dst = a.out + unit * kDim;
  *reinterpret_cast<uint4*>(dst + 8 * lane8) = make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
  *reinterpret_cast<uint4*>(dst + 64 + 8 * lane8) = make_uint4(out_hi[0], out_hi[1], out_hi[2], out_hi[3]);
}

// FP8 compressed keys: per key, scale = max_d |k_d| / 448 (FP32 division)
// and code_d = e4m3(k_d / scale) (FP32 division, nearest e4m3 value, ties to
// even, saturating); a zero key gets scale 0 and zero codes.  8 lanes per key,
// 16 dims each.
struct QuantArgs {
  const __nv_bfloat16* keys;  // [n][128]
  int64_t n;
  uint8_t* codes;             // [n][128]
  float* scales;              // [n]
};
constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads) quantize_keys_fp8_kernel(QuantArgs a) {
  pdl_launch_dependents();
  const int lane8 = threadIdx.x & (kCompressLanes - 1);
  const int64_t key = (int64_t)blockIdx.x * (kQuantThreads / kCompressLanes) + threadIdx.x / kCompressLanes;
  const bool live = key < a.n;
  const __nv_bfloat16* src = a.keys + (live ? key : 0) * kDim + 16 * lane8;
  const uint4 w0 = live ? ld_stream_16(src) : make_uint4(0u, 0u, 0u, 0u);
  const uint4 w1 = live ? ld_stream_16(src + 8) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float x[16];
  float mx = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float2 f = bf16x2_to_float2(w[e]);
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
    mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  // the 8 lanes of a key always reach this together
  const unsigned group = 0xffu << (threadIdx.x & 24);
  mx = fmaxf(mx, __shfl_xor_sync(group, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(group, mx, 2));
  mx = fmaxf(mx, __shfl_xor_sync(group, mx, 4));
  if (!live) return;
  const float scale = mx / 448.0f;
  uint32_t out[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint32_t word = 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t code =
          scale > 0.f ? (uint32_t)__nv_cvt_float_to_fp8(x[4 * e + b] / scale, __NV_SATFINITE, __NV_E4M3) : 0u;
      word |= (code & 0xffu) << (8 * b);
    }
    out[e] = word;
  }
  *reinterpret_cast<uint4*>(a.codes + key * kDim + 16 * lane8) = make_uint4(out[0], out[1], out[2], out[3]);
  if (lane8 == 0) a.scales[key] = scale;
}

}  // namespace qsa
