// select_resident.cuh -- exact top-k of score rows that fit in shared memory
// (up to 32768 entries: every decode row of a context up to 128K tokens).
//
// Same contract as select_kernel (SGLang GLM-5.2 blog, "Kernel Optimization /
// TopK-V2": a selection, exact ties, runtime k, page-table transform fused;
// Qwen3.8-Flash-Next write-up, "Qwen sparse attention (QSA)": 512 blocks ->
// 4 positions each, then the 0-3 pending tokens; -1 marks an empty entry).
// Readings: ties go to the lower index; -0 == +0; NaN ranks below -inf; the
// result is in ascending index order with -1 only as tail padding.
//
// Design: one 1024-thread CTA per row.  A row is small (tens of KB), so the
// cost is the SM's instruction issue and the CTA barriers, not bytes; every
// pass over the whole row costs about a microsecond, and shared-memory
// atomics over the whole row serialise on the few hot bins that score
// distributions have.  So the whole row is touched by as few simple passes
// as possible, and the exact work runs on a short candidate list:
//  0. The row is read once with 16-byte loads (thread t owns entries
//     4(t + 1024 j) .. +3) and kept in shared memory as order-preserving u32
//     keys (larger float -> larger key).
//  1. Estimate: 1024 evenly spaced keys are counted into a histogram of the
//     top 11 bits and then of the next 11 bits inside the chosen bin; the
//     22-bit prefix where the sample reaches rank ~1.5k*1024/n + 8 is a
//     threshold t_s that about 1.5k entries of the row are expected to reach.
//  2. One pass appends every entry with key >= t_s to a candidate list
//     (per-thread counts, warp scans, one shared counter per warp).
//  3. If the list holds at least k entries (it then holds all of the top k),
//     exact radix passes over the list (11, 11, 10 bits; a pass is skipped
//     when its bin is taken whole) find the k-th key T and how many keys equal
//     to T to take (`need`, the first ones by index).  Winners set their bit
//     in a bitmap of the row (keys equal to T in a second one, of which the
//     first `need` by index are added with one prefix scan); one more prefix
//     scan over the bitmap words lists the selected indices in ascending
//     order.
//  4. If the list is short or overflows (a misleading sample, massive ties),
//     the same exact radix passes and an ordered emission run over the whole
//     row instead.
//  5. The outputs (indices and slots; for QSA the 4 positions of every block,
//     then the pending tokens, then -1) are written by consecutive threads to
//     consecutive entries, with page-table lookups from a staged copy of the
//     row's page-table entries.
#pragma once
#include "select.cuh"

namespace qsa {

constexpr int kRsThreads = 1024;
constexpr int kRsWarps = kRsThreads / 32;
constexpr int kRsChunk = 4 * kRsThreads;  // entries per chunk: one 16-byte load per thread
constexpr int kRsMaxChunks = 8;
constexpr int kRsMaxRow = kRsChunk * kRsMaxChunks;  // 32768 (= 32 bits x 1024 bitmap words)
constexpr int kRsSampleMin = 2048;                  // shorter rows: every entry is a candidate

struct RsFixed {
  uint32_t h1[2048];       // top 11 key bits
  uint32_t h2[2048];       // bits 20..10
  uint32_t h3[1024];       // bits 9..0
  uint32_t bm_gt[1024];    // bit i of word w: entry 32w + i is above the threshold
  uint32_t bm_eq[1024];    // ... equal to it
  uint32_t wsum[kRsWarps];
  uint32_t wsum2[kRsWarps];
  uint32_t wcnt[kRsMaxChunks][kRsWarps];
  int info[4];
  int list_n;
};
constexpr int kRsFixedBytes = (int)((sizeof(RsFixed) + 127) & ~size_t(127));
constexpr int kRsZeroWords = 2048 + 2048 + 1024 + 1024 + 1024;  // h1 .. bm_eq
static_assert(offsetof(RsFixed, bm_eq) == (kRsZeroWords - 1024) * 4, "zeroed arrays must be contiguous");

__device__ __forceinline__ uint32_t rs_warp_incl_scan(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive prefix of x over the CTA's threads in thread order, and the
// total.  One barrier; `buf` (32 words) must not be rewritten before the
// next barrier.
__device__ __forceinline__ uint32_t rs_block_excl_scan(uint32_t x, uint32_t* buf, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = rs_warp_incl_scan(x);
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  const uint32_t v = buf[lane];
  const uint32_t vincl = rs_warp_incl_scan(v);
  total = __shfl_sync(0xffffffffu, vincl, 31);
  return __shfl_sync(0xffffffffu, vincl - v, warp) + incl - x;
}

// The bin (counted from the top) that holds the k_rem-th largest key among
// `nbins` bins (2048 or 1024); returns (bin, keys in higher bins, keys in the
// bin).  Requires k_rem <= the histogram's total.  Two CTA barriers.
__device__ __forceinline__ int3 rs_find_bin(RsFixed& fx, const uint32_t* hist, int nbins, int k_rem) {
  const int per = nbins / kRsThreads;  // 2 or 1
  const int top = nbins - 1 - per * (int)threadIdx.x;  // this thread's bins: top, top-1
  const uint32_t c0 = hist[top];
  const uint32_t c1 = per == 2 ? hist[top - 1] : 0u;
  const uint32_t s = c0 + c1;
  uint32_t total;
  const uint32_t above = rs_block_excl_scan(s, fx.wsum, total);
  const uint32_t kr = (uint32_t)k_rem;
  if (above < kr && kr <= above + c0) {
    fx.info[0] = top;
    fx.info[1] = (int)above;
    fx.info[2] = (int)c0;
  } else if (per == 2 && above + c0 < kr && kr <= above + s) {
    fx.info[0] = top - 1;
    fx.info[1] = (int)(above + c0);
    fx.info[2] = (int)c1;
  }
  __syncthreads();
  return make_int3(fx.info[0], fx.info[1], fx.info[2]);
}

// Physical slot of token position p (the page-table map of the pages'
// problem statement); staged entries first, then global memory.
__device__ __forceinline__ int32_t rs_slot(const SelectArgs& a, const int32_t* pt_s, int pt_n,
                                           const int32_t* pt_row, int32_t p) {
  const uint32_t ps = (uint32_t)a.page_size;
  const uint32_t page_idx = (uint32_t)p / ps;
  const int32_t off = (int32_t)((uint32_t)p - page_idx * ps);
  int32_t page;
  if ((int)page_idx < pt_n) {
    page = pt_s[page_idx];
  } else if ((int64_t)page_idx < a.ld_pt) {
    page = __ldg(pt_row + page_idx);
  } else {
    raise_fault(kFaultIndex);
    return -1;
  }
  return page * a.page_size + off;
}

template <int kMode>
__global__ void __launch_bounds__(kRsThreads, 1)
select_resident_kernel(SelectArgs a) {
  extern __shared__ __align__(128) unsigned char rs_smem_raw[];
  RsFixed& fx = *reinterpret_cast<RsFixed*>(rs_smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(rs_smem_raw + a.off_row);    // [whole chunks]
  uint32_t* lkey = reinterpret_cast<uint32_t*>(rs_smem_raw + a.off_lkey);   // [list_cap]
  int32_t* lidx = reinterpret_cast<int32_t*>(rs_smem_raw + a.off_list);     // [list_cap]
  int32_t* pt_s = reinterpret_cast<int32_t*>(rs_smem_raw + a.off_pt);       // [pt_cap]
  int32_t* sel_s = reinterpret_cast<int32_t*>(rs_smem_raw + a.off_sel);     // [k]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- row metadata and page-table entries: not produced by the previous
  // grid, so read before waiting on it -----------------------------------
  int t;
  if (!sel_unit_row(a, blockIdx.x, t)) return;
  int n, L = 0;
  const int32_t* pt_row = nullptr;
  if (kMode == kModeTopk) {
    n = a.n_valid ? __ldg(a.n_valid + t) : a.n_max;
    if (a.out_slots != nullptr)
      pt_row = a.page_table + (int64_t)(a.row_req ? __ldg(a.row_req + t) : t) * a.ld_pt;
  } else {
    const int req = row_request(a.req_row_start, a.n_req, t);
    L = __ldg(a.row_len + t);
    n = L / kBlock;
    pt_row = a.page_table + (int64_t)req * a.ld_pt;
  }
  if (n < 0 || n > a.n_max || L < 0) {  // bad length: emit an empty row
    if (tid == 0) raise_fault(kFaultGrouping);
    n = 0;
    L = 0;
  }
  int pt_n = 0;
  if (pt_row != nullptr) {
    const int64_t last = kMode == kModeQsa ? (int64_t)L : (int64_t)n;  // positions < last
    int64_t np = last > 0 ? (last - 1) / a.page_size + 1 : 0;
    if (np > a.pt_cap) np = a.pt_cap;
    if (np > a.ld_pt) np = a.ld_pt;
    pt_n = (int)np;
    for (int i = tid; i < pt_n; i += kRsThreads) pt_s[i] = __ldg(pt_row + i);
  }
  uint32_t* hz = fx.h1;  // h1 .. bm_eq are contiguous
  for (int i = tid; i < kRsZeroWords; i += kRsThreads) hz[i] = 0u;
  if (tid < 4) fx.info[tid] = 0;
  if (tid == 0) fx.list_n = 0;
  __syncthreads();
  if (a.wait_primary) pdl_wait_primary();

  const float* row = a.scores + (int64_t)t * a.ld;
  const int k = a.k;
  const int m = n < k ? n : k;  // entries selected
  const int nch = (n + kRsChunk - 1) / kRsChunk;

  if (n > k) {
    // ---- 0. load the row as keys -----------------------------------------
    {
      float4 v[kRsMaxChunks];
#pragma unroll
      for (int j = 0; j < kRsMaxChunks; ++j) {
        const int i = 4 * (tid + kRsThreads * j);
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < nch) {
          if (a.vec_ok && i + 3 < n) {
            v[j] = __ldg(reinterpret_cast<const float4*>(row + i));
          } else {
            if (i < n) v[j].x = __ldg(row + i);
            if (i + 1 < n) v[j].y = __ldg(row + i + 1);
            if (i + 2 < n) v[j].z = __ldg(row + i + 2);
            if (i + 3 < n) v[j].w = __ldg(row + i + 3);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kRsMaxChunks; ++j) {
        if (j < nch) {
          const int i = 4 * (tid + kRsThreads * j);
          uint4 kk;
          kk.x = i < n ? order_key(v[j].x) : 0u;
          kk.y = i + 1 < n ? order_key(v[j].y) : 0u;
          kk.z = i + 2 < n ? order_key(v[j].z) : 0u;
          kk.w = i + 3 < n ? order_key(v[j].w) : 0u;
          *reinterpret_cast<uint4*>(keys + i) = kk;
        }
      }
    }
    __syncthreads();

    // ---- 1. threshold estimate from 1024 evenly spaced keys -------------
    uint32_t t_s = 0u;  // candidates: key >= t_s (0: every entry)
    if (n >= kRsSampleMin) {
      const uint32_t sk = keys[(int)(((int64_t)tid * n) >> 10)];
      atomicAdd(&fx.h1[sk >> 21], 1u);
      __syncthreads();
      const int target = min(kRsThreads, (int)((3LL * k * kRsThreads + 2LL * n - 1) / (2LL * n)) + 8);
      const int3 f1 = rs_find_bin(fx, fx.h1, 2048, target);
      if ((sk >> 21) == (uint32_t)f1.x) atomicAdd(&fx.h2[(sk >> 10) & 2047u], 1u);
      __syncthreads();
      const int3 f2 = rs_find_bin(fx, fx.h2, 2048, target - f1.y);
      t_s = ((uint32_t)f1.x << 21) | ((uint32_t)f2.x << 10);
      // h1 and h2 were last read before the barrier that ended find_bin;
      // clear them for the exact passes (read after the next barrier).
      for (int i = tid; i < 4096; i += kRsThreads) hz[i] = 0u;
    }

    // ---- 2. candidate list: every entry with key >= t_s -----------------
    const int cap = a.list_cap;
    {
      uint32_t c = 0u;
#pragma unroll
      for (int j = 0; j < kRsMaxChunks; ++j) {
        if (j < nch) {
          const int i = 4 * (tid + kRsThreads * j);
          const uint4 kk = *reinterpret_cast<const uint4*>(keys + i);
          c += (i < n && kk.x >= t_s) + (i + 1 < n && kk.y >= t_s) + (i + 2 < n && kk.z >= t_s) +
               (i + 3 < n && kk.w >= t_s);
        }
      }
      const uint32_t inc = rs_warp_incl_scan(c);
      uint32_t wbase = 0u;
      if (lane == 31) wbase = atomicAdd(reinterpret_cast<unsigned*>(&fx.list_n), inc);
      uint32_t o = __shfl_sync(0xffffffffu, wbase, 31) + inc - c;
      if (c > 0u) {
#pragma unroll
        for (int j = 0; j < kRsMaxChunks; ++j) {
          if (j < nch) {
            const int i = 4 * (tid + kRsThreads * j);
            const uint4 kk = *reinterpret_cast<const uint4*>(keys + i);
            const uint32_t kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (i + e < n && kv[e] >= t_s) {
                if (o < (uint32_t)cap) {
                  lkey[o] = kv[e];
                  lidx[o] = i + e;
                }
                ++o;
              }
            }
          }
        }
      }
    }
    __syncthreads();
    const int m_list = fx.list_n;

    if (m_list >= k && m_list <= cap) {
      // ---- 3. exact threshold among the candidates --------------------
      for (int i = tid; i < m_list; i += kRsThreads) atomicAdd(&fx.h1[lkey[i] >> 21], 1u);
      __syncthreads();
      int3 fb = rs_find_bin(fx, fx.h1, 2048, k);
      uint32_t prefix = (uint32_t)fb.x;
      int shift = 21;
      int k_rem = k - fb.y;
      if (fb.z != k_rem) {
        for (int i = tid; i < m_list; i += kRsThreads) {
          const uint32_t key = lkey[i];
          if ((key >> 21) == prefix) atomicAdd(&fx.h2[(key >> 10) & 2047u], 1u);
        }
        __syncthreads();
        fb = rs_find_bin(fx, fx.h2, 2048, k_rem);
        prefix = (prefix << 11) | (uint32_t)fb.x;
        shift = 10;
        k_rem -= fb.y;
        if (fb.z != k_rem) {
          for (int i = tid; i < m_list; i += kRsThreads) {
            const uint32_t key = lkey[i];
            if ((key >> 10) == prefix) atomicAdd(&fx.h3[key & 1023u], 1u);
          }
          __syncthreads();
          fb = rs_find_bin(fx, fx.h3, 1024, k_rem);
          prefix = (prefix << 10) | (uint32_t)fb.x;
          shift = 0;
          k_rem -= fb.y;
        }
      }
      const uint32_t need = (uint32_t)k_rem;  // equal keys to take, first by index
      const uint32_t n_eq = (uint32_t)fb.z;   // keys equal to the threshold prefix
      for (int i = tid; i < m_list; i += kRsThreads) {
        const uint32_t hb = lkey[i] >> shift;
        const int idx = lidx[i];
        if (hb > prefix) atomicOr(&fx.bm_gt[idx >> 5], 1u << (idx & 31));
        else if (hb == prefix) atomicOr(&fx.bm_eq[idx >> 5], 1u << (idx & 31));
      }
      __syncthreads();
      // bitmap word tid covers entries 32 tid .. 32 tid + 31 (n <= 32768)
      uint32_t w = fx.bm_gt[tid];
      const uint32_t weq = fx.bm_eq[tid];
      if (need == n_eq) {
        w |= weq;
      } else {  // ties at the threshold: the first `need` by index
        uint32_t tot;
        const uint32_t before = rs_block_excl_scan(__popc(weq), fx.wsum2, tot);
        uint32_t take = before >= need ? 0u : need - before;
        uint32_t rest = weq;
        while (take > 0u && rest != 0u) {
          w |= rest & (0u - rest);  // lowest remaining bit
          rest &= rest - 1u;
          --take;
        }
      }
      uint32_t tot;
      uint32_t pos = rs_block_excl_scan(__popc(w), fx.wsum, tot);
      while (w != 0u) {
        const int b = __ffs(w) - 1;
        if (pos < (uint32_t)k) sel_s[pos] = 32 * tid + b;
        ++pos;
        w &= w - 1u;
      }
      __syncthreads();
    } else {
      // ---- 4. exact passes and ordered emission over the whole row -------
      // (h1..h3 are zero here: the sample's counts were cleared above)
#pragma unroll
      for (int j = 0; j < kRsMaxChunks; ++j) {
        if (j < nch) {
          const int i = 4 * (tid + kRsThreads * j);
          const uint4 kk = *reinterpret_cast<const uint4*>(keys + i);
          if (i < n) atomicAdd(&fx.h1[kk.x >> 21], 1u);
          if (i + 1 < n) atomicAdd(&fx.h1[kk.y >> 21], 1u);
          if (i + 2 < n) atomicAdd(&fx.h1[kk.z >> 21], 1u);
          if (i + 3 < n) atomicAdd(&fx.h1[kk.w >> 21], 1u);
        }
      }
      __syncthreads();
      int3 fb = rs_find_bin(fx, fx.h1, 2048, k);
      uint32_t prefix = (uint32_t)fb.x;
      int shift = 21;
      int k_rem = k - fb.y;
      if (fb.z != k_rem) {
#pragma unroll
        for (int j = 0; j < kRsMaxChunks; ++j) {
          if (j < nch) {
            const int i = 4 * (tid + kRsThreads * j);
            const uint4 kk = *reinterpret_cast<const uint4*>(keys + i);
            if (i < n && (kk.x >> 21) == prefix) atomicAdd(&fx.h2[(kk.x >> 10) & 2047u], 1u);
            if (i + 1 < n && (kk.y >> 21) == prefix) atomicAdd(&fx.h2[(kk.y >> 10) & 2047u], 1u);
            if (i + 2 < n && (kk.z >> 21) == prefix) atomicAdd(&fx.h2[(kk.z >> 10) & 2047u], 1u);
            if (i + 3 < n && (kk.w >> 21) == prefix) atomicAdd(&fx.h2[(kk.w >> 10) & 2047u], 1u);
          }
        }
        __syncthreads();
        fb = rs_find_bin(fx, fx.h2, 2048, k_rem);
        prefix = (prefix << 11) | (uint32_t)fb.x;
        shift = 10;
        k_rem -= fb.y;
        if (fb.z != k_rem) {
#pragma unroll
          for (int j = 0; j < kRsMaxChunks; ++j) {
            if (j < nch) {
              const int i = 4 * (tid + kRsThreads * j);
              const uint4 kk = *reinterpret_cast<const uint4*>(keys + i);
              if (i < n && (kk.x >> 10) == prefix) atomicAdd(&fx.h3[kk.x & 1023u], 1u);
              if (i + 1 < n && (kk.y >> 10) == prefix) atomicAdd(&fx.h3[kk.y & 1023u], 1u);
              if (i + 2 < n && (kk.z >> 10) == prefix) atomicAdd(&fx.h3[kk.z & 1023u], 1u);
              if (i + 3 < n && (kk.w >> 10) == prefix) atomicAdd(&fx.h3[kk.w & 1023u], 1u);
            }
          }
          __syncthreads();
          fb = rs_find_bin(fx, fx.h3, 1024, k_rem);
          prefix = (prefix << 10) | (uint32_t)fb.x;
          shift = 0;
          k_rem -= fb.y;
        }
      }
      const uint32_t need = (uint32_t)k_rem;
      // Output position of a selected entry: entries above the threshold
      // before it + min(equal entries before it, need).  Packed counts per 4
      // entries: above (low 16 bits), equal (high 16 bits); a row has at
      // most 32768 entries, so neither field overflows.
      auto classify = [&](const uint4& kk, int i, uint32_t (&gt)[4], uint32_t (&eq)[4]) {
        const uint32_t kv[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t hb = kv[e] >> shift;
          const bool in = i + e < n;
          gt[e] = (in && hb > prefix) ? 1u : 0u;
          eq[e] = (in && hb == prefix) ? 1u : 0u;
        }
      };
      uint32_t pk[kRsMaxChunks];
#pragma unroll
      for (int j = 0; j < kRsMaxChunks; ++j) {
        pk[j] = 0u;
        if (j < nch) {
          const int i = 4 * (tid + kRsThreads * j);
          uint32_t gt[4], eq[4];
          classify(*reinterpret_cast<const uint4*>(keys + i), i, gt, eq);
          const uint32_t c = (gt[0] + gt[1] + gt[2] + gt[3]) | ((eq[0] + eq[1] + eq[2] + eq[3]) << 16);
          const uint32_t inc = rs_warp_incl_scan(c);
          pk[j] = inc - c;
          if (lane == 31) fx.wcnt[j][warp] = inc;
        }
      }
      __syncthreads();
      uint32_t run = 0u;
#pragma unroll
      for (int j = 0; j < kRsMaxChunks; ++j) {
        if (j < nch) {
          const uint32_t v = fx.wcnt[j][lane];
          const uint32_t inc = rs_warp_incl_scan(v);
          const uint32_t base = run + __shfl_sync(0xffffffffu, inc - v, warp) + pk[j];
          run += __shfl_sync(0xffffffffu, inc, 31);
          const int i = 4 * (tid + kRsThreads * j);
          uint32_t gt[4], eq[4];
          classify(*reinterpret_cast<const uint4*>(keys + i), i, gt, eq);
          uint32_t gb = base & 0xffffu, qb = base >> 16;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t pos = gb + (qb < need ? qb : need);
            if ((gt[e] || (eq[e] && qb < need)) && pos < (uint32_t)k) sel_s[pos] = i + e;
            gb += gt[e];
            qb += eq[e];
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- 5. outputs, consecutive threads on consecutive entries -----------
  // sel(j) = j-th selected index (ascending); when n <= k every index is.
  auto sel = [&](int j) { return n > k ? sel_s[j] : j; };
  if (kMode == kModeTopk) {
    int32_t* oi = a.out_idx + (int64_t)t * k;
    int32_t* os = a.out_slots ? a.out_slots + (int64_t)t * k : nullptr;
    for (int j = tid; j < k; j += kRsThreads) {
      const int32_t idx = j < m ? sel(j) : -1;
      oi[j] = idx;
      if (os != nullptr) os[j] = idx < 0 ? -1 : rs_slot(a, pt_s, pt_n, pt_row, idx);
    }
  } else {
    if (a.out_idx != nullptr) {
      int32_t* oi = a.out_idx + (int64_t)t * k;
      for (int j = tid; j < k; j += kRsThreads) oi[j] = j < m ? sel(j) : -1;
    }
    const int width = kBlock * k + (kBlock - 1);
    const int pend = L - kBlock * n;  // tokens of the incomplete block
    int32_t* xs = a.out_xslots + (int64_t)t * width;
    int32_t* xp = a.out_pos ? a.out_pos + (int64_t)t * width : nullptr;
    for (int j = tid; j < width; j += kRsThreads) {
      int32_t p = -1;
      if (j < kBlock * m) p = kBlock * sel(j >> 2) + (j & (kBlock - 1));
      else if (j - kBlock * m < pend) p = kBlock * n + (j - kBlock * m);
      xs[j] = p < 0 ? -1 : rs_slot(a, pt_s, pt_n, pt_row, p);
      if (xp != nullptr) xp[j] = p;
    }
  }
}

}  // namespace qsa
