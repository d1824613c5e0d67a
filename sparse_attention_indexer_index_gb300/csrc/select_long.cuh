// select_long.cuh -- exact top-k of long score rows (more than 32768
// entries, up to the 1M-token rows of long-context DSA), each row spread
// over a cluster of 2-16 CTAs that stream it.
//
// Same contract as select_kernel (SGLang GLM-5.2 blog, "Kernel Optimization /
// TopK-V2": a selection, not a sort; exactly k entries, exact ties, runtime k
// up to 2048; the page-table transform in the same kernel; for long rows a
// cluster of CTAs builds local radix histograms and reduces them across the
// cluster to find the threshold bin.  Qwen3.8-Flash-Next write-up, "Qwen
// sparse attention (QSA)": blocks -> 4 positions each, then the 0-3 pending
// tokens; -1 marks an empty entry).  Readings: ties go to the lower index;
// -0 == +0; NaN ranks below -inf; ascending index order.
//
// Design.  Keys are order-preserving u32 images of the scores.  CTA c of the
// cluster owns the slice [c S, c S + S) of the row; warp w of it a contiguous
// segment of the slice, walked 128 entries at a time (4 consecutive per
// lane).  Each warp brings the first part of its segment into its own
// shared-memory region with one bulk asynchronous copy (TMA engine) and reads
// the rest with 16-byte loads.
//  1. Sampled bound (no communication): every CTA reads the same 2048
//     entries (16 runs of 128 spread over the row) and takes the edge of the
//     top-12-bit bin below which the r-th largest sample lies, r about twice
//     the expected number of samples above the k-th entry.
//  2. One pass over the slice: each warp lists its entries at or above the
//     bound (key, index) in its own region of a candidate list, with ballot
//     counts; usually a few k entries of the whole row.
//  3. Radix levels of 12, 12 and 8 bits over the lists: each CTA counts the
//     digit of the keys in the current boundary bin, adds its non-zero bins
//     into the leader's histogram with distributed-shared-memory reductions,
//     and the leader finds the bin of the k_rem-th entry and sends it to
//     every CTA (two cluster barriers per level), until a bin is taken whole
//     or the key is complete: the k-th key's prefix P at bit `shift` and the
//     count `need` of entries in that bin to take, the first ones by index.
//  4. Ranks: each CTA marks its winners above P and its entries in P's bin
//     in two bitmaps of its slice; the CTAs exchange their counts (one
//     cluster barrier); prefix counts of the bitmap words give the entries of
//     P's bin that are taken (the first `need` of the row) and every
//     winner's ascending output position.  Each CTA places its winners'
//     indices in that order in shared memory and writes their outputs (with
//     the slot translation or the QSA expansion) from there, every thread
//     taking every 512-th output; all CTAs at once.
// Fallbacks, all exact: a CTA whose warp lists overflow counts and marks by
// walking its whole slice; a sampled bound with fewer than k entries above
// it (retry flag from the leader), or slices longer than the bitmaps, take
// the whole-slice path: radix levels over the slices, then per-warp counts
// and an ordered emission pass.  Every wait is a CTA or cluster barrier or a
// time-bounded mbarrier wait; there is no global scratch.
#pragma once
#include <type_traits>

#include "select_cluster.cuh"

namespace qsa {

constexpr int kSlThreads = 512;
constexpr int kSlWarps = kSlThreads / 32;
constexpr int kSlMaxCluster = 16;
constexpr int kSlBins = 4096;   // 12-bit digits; the last level uses 256 of them
constexpr int kSlUnroll = 4;    // 128-entry chunks per warp in flight from global memory
constexpr int kSlSamples = 2048;  // evenly spaced entries behind the first histogram's bound
// Candidate entries per CTA (kSlCandCap / kSlWarps per warp).  Rows of 80,000
// on clusters of 2 leave about 170 entries per warp above the sampled bound,
// up to 300 in the tail of ReLU-sum rows (2 % of rows passed 256, the
// previous capacity, and took the whole-slice path).
constexpr int kSlCandCap = 6144;
constexpr int kSlBitmapWords = kSlBins / 2;  // slices of up to 65536 entries for the list path

struct SlFixed {
  uint32_t hloc[kSlBins];       // this CTA's histogram of the current level; then two bitmaps
  uint32_t hred[2][kSlBins];    // leader: the cluster's histograms (levels 0 and 2 share [0]); then scans
  uint32_t cand_key[kSlCandCap];  // candidates (keys at or above the sampled bound), per warp
  uint32_t cand_idx[kSlCandCap];
  uint32_t wsum[kSlWarps];
  uint32_t wg[kSlWarps];        // per-warp entries above / in the boundary bin
  uint32_t wq[kSlWarps];
  int info[4];
  int binfo[4];                 // from the leader: bin, above, count, flags
  uint32_t cgt[kSlMaxCluster];  // every CTA's entries above / in the boundary bin
  uint32_t ceq[kSlMaxCluster];
  uint32_t n_emit;              // winners of this CTA listed for the output step (whole-slice path)
  uint32_t cnt2[2];             // this CTA's entries above / in the boundary bin
  int ovf;                      // a warp's candidate region overflowed
  uint64_t bar[kSlWarps];       // each warp's bulk copy of its staged entries
};
constexpr int kSlFixedBytes = (int)((sizeof(SlFixed) + 127) & ~size_t(127));

__device__ __forceinline__ void red_dsmem_add_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t sl_warp_incl_scan(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive prefix of x over the CTA in thread order and the total; one
// barrier before and after the shared totals are used.
__device__ __forceinline__ uint32_t sl_block_excl_scan(SlFixed& fx, uint32_t x, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = sl_warp_incl_scan(x);
  if (lane == 31) fx.wsum[warp] = incl;
  __syncthreads();
  uint32_t before = 0u, tot = 0u;
#pragma unroll
  for (int w = 0; w < kSlWarps; ++w) {
    const uint32_t v = fx.wsum[w];
    before += w < warp ? v : 0u;
    tot += v;
  }
  total = tot;
  __syncthreads();
  return before + incl - x;
}

// The bin (of kSlBins, counted from the top) of the local histogram `hist`
// that holds the k_rem-th largest entry: (bin, entries in higher bins,
// entries in the bin, histogram total).  Without such a bin (k_rem > total)
// the first three are 0.
__device__ __forceinline__ int4 sl_find_bin(SlFixed& fx, const uint32_t* hist, int k_rem) {
  const int top = kSlBins - 1 - 8 * (int)threadIdx.x;  // bins top .. top-7
  uint32_t c[8];
  uint32_t s = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = hist[top - j];
    s += c[j];
  }
  if (threadIdx.x < 3) fx.info[threadIdx.x] = 0;
  uint32_t tot;
  uint32_t above = sl_block_excl_scan(fx, s, tot);  // its barriers order the clear above
  const uint32_t kr = (uint32_t)k_rem;
  if (above < kr && kr <= above + s) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (above < kr && kr <= above + c[j]) {
        fx.info[0] = top - j;
        fx.info[1] = (int)above;
        fx.info[2] = (int)c[j];
      }
      above += c[j];
    }
  }
  __syncthreads();
  const int4 r = make_int4(fx.info[0], fx.info[1], fx.info[2], (int)tot);
  __syncthreads();  // info may be rewritten by the next call
  return r;
}

// "order_key(x) >= K" as one float compare, for every x including NaN (key
// 0) and -0 (the key of +0); K up to 2^32 (never true).  NaN compares false
// with everything, so K in (0, key(-inf)] becomes x >= -inf, K = 2^32 becomes
// x >= NaN, and only K = 0 (NaN included) needs the `all` flag.
struct SlBound {
  float f;
  bool all;
  __device__ __forceinline__ bool ge(float x) const { return (x >= f) | all; }
};
__device__ __forceinline__ SlBound sl_bound(uint64_t K) {
  SlBound b;
  b.all = K == 0ull;
  if (K >= (1ull << 32)) {
    b.f = __uint_as_float(0x7fffffffu);  // NaN: never
  } else if (K <= 0x007fffffull) {       // at or below the key of -inf
    b.f = __uint_as_float(0xff800000u);  // -inf: every non-NaN
  } else {
    const uint32_t k = (uint32_t)K;
    b.f = __uint_as_float(k >= 0x80000000u ? (k & 0x7fffffffu) : ~k);
  }
  return b;
}

__device__ __forceinline__ float4 sl_load4(const float* __restrict__ row, int i, int end, bool vec) {
  const float nan = __uint_as_float(0x7fffffffu);
  float4 v = make_float4(nan, nan, nan, nan);
  if (vec && i + 3 < end) {
    v = __ldg(reinterpret_cast<const float4*>(row + i));
  } else {
    if (i < end) v.x = __ldg(row + i);
    if (i + 1 < end) v.y = __ldg(row + i + 1);
    if (i + 2 < end) v.z = __ldg(row + i + 2);
    if (i + 3 < end) v.w = __ldg(row + i + 3);
  }
  return v;
}

// Positions are below 2^31 (row lengths are int32), so 32-bit arithmetic.
__device__ __forceinline__ int32_t sl_slot(const SelectArgs& a, const int32_t* pt_row, uint32_t pos) {
  const uint32_t ps = (uint32_t)a.page_size;
  // a shift for page sizes that are powers of two (the usual case)
  const uint32_t page_idx = (ps & (ps - 1u)) == 0u ? pos >> (31 - __clz((int)ps)) : pos / ps;
  if ((int64_t)page_idx >= a.ld_pt) {
    raise_fault(kFaultIndex);
    return -1;
  }
  return __ldg(pt_row + page_idx) * a.page_size + (int32_t)(pos - page_idx * ps);
}

template <int kMode>
__global__ void __launch_bounds__(kSlThreads, 1)
select_long_kernel(SelectArgs a) {
  extern __shared__ __align__(128) unsigned char sl_smem_raw[];
  SlFixed& fx = *reinterpret_cast<SlFixed*>(sl_smem_raw);
  float* stage = reinterpret_cast<float*>(sl_smem_raw + kSlFixedBytes);  // [a.list_cap] slice entries
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const uint32_t C = cluster_nctarank();
  // the row of this cluster (every CTA of a cluster gets the same answer, so
  // a cluster without a row leaves before its first cluster barrier)
  int t;
  if (!sel_unit_row(a, (int)(blockIdx.x / C), t)) return;

  for (int i = tid; i < kSlBins; i += kSlThreads) fx.hloc[i] = 0u;
  if (rank == 0)
    for (int i = tid; i < 2 * kSlBins; i += kSlThreads) (&fx.hred[0][0])[i] = 0u;
  if (tid == 0) {
    fx.n_emit = 0u;
    fx.cnt2[0] = fx.cnt2[1] = 0u;
    fx.ovf = 0;
  }
  if (tid < kSlWarps) mbar_init(&fx.bar[tid], 1);
  fence_mbar_init();
  __syncthreads();
  // The leader's zeroed histograms are visible to every CTA after this
  // arrive (release) and the matching wait (acquire) before the first
  // remote access.
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  // ---- row metadata --------------------------------------------------------
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
    if (tid == 0 && rank == 0) raise_fault(kFaultGrouping);
    n = 0;
    L = 0;
  }
  if (a.wait_primary) pdl_wait_primary();
  const float* row = a.scores + (int64_t)t * a.ld;
  const int k = a.k;
  const int m_sel = n < k ? n : k;

  auto emit = [&](uint32_t idx, int pos) {
    if (kMode == kModeTopk) {
      a.out_idx[(int64_t)t * k + pos] = (int32_t)idx;
      if (a.out_slots != nullptr) a.out_slots[(int64_t)t * k + pos] = sl_slot(a, pt_row, idx);
    } else {
      if (a.out_idx != nullptr) a.out_idx[(int64_t)t * k + pos] = (int32_t)idx;
      const int64_t width = (int64_t)kBlock * k + (kBlock - 1);
      const uint32_t p0 = kBlock * idx;  // 4 positions in one page
      const int32_t base = sl_slot(a, pt_row, p0);
      int32_t* xs = a.out_xslots + (int64_t)t * width + kBlock * pos;
#pragma unroll
      for (int c = 0; c < kBlock; ++c) xs[c] = base < 0 ? -1 : base + c;
      if (a.out_pos != nullptr) {
        int32_t* xp = a.out_pos + (int64_t)t * width + kBlock * pos;
#pragma unroll
        for (int c = 0; c < kBlock; ++c) xp[c] = (int32_t)p0 + c;
      }
    }
  };

  // ---- the tail after m_sel entries (leader) ---------------------------------
  if (rank == 0) {
    if (kMode == kModeTopk) {
      for (int j = m_sel + tid; j < k; j += kSlThreads) {
        a.out_idx[(int64_t)t * k + j] = -1;
        if (a.out_slots != nullptr) a.out_slots[(int64_t)t * k + j] = -1;
      }
    } else {
      if (a.out_idx != nullptr)
        for (int j = m_sel + tid; j < k; j += kSlThreads) a.out_idx[(int64_t)t * k + j] = -1;
      const int width = kBlock * k + (kBlock - 1);
      const int pend = L - kBlock * n;
      for (int j = kBlock * m_sel + tid; j < width; j += kSlThreads) {
        const int i = j - kBlock * m_sel;
        int32_t pos = -1, slot = -1;
        if (i < pend) {
          pos = kBlock * n + i;
          slot = sl_slot(a, pt_row, (uint32_t)pos);
        }
        a.out_xslots[(int64_t)t * width + j] = slot;
        if (a.out_pos != nullptr) a.out_pos[(int64_t)t * width + j] = pos;
      }
    }
  }

  if (n <= k) {  // every entry is selected, in order
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (rank != 0) return;
    for (int j = tid; j < m_sel; j += kSlThreads) emit(j, j);
    return;
  }

  // ---- slice and warp segments ------------------------------------------------
  // Warp w owns [w0, w1) of the slice; its first `st_n` entries (whole
  // 128-entry chunks) are brought into its own region of shared memory by
  // one bulk copy, the rest is read from global memory (L2 after the first
  // pass) in every pass.
  const int S = (((n + (int)C - 1) / (int)C) + 3) & ~3;
  const int s0 = min(n, (int)rank * S);
  const int s1 = min(n, s0 + S);
  const int seg = ((((s1 - s0) + kSlWarps - 1) / kSlWarps) + 127) & ~127;
  const int w0 = min(s1, s0 + warp * seg);
  const int w1 = min(s1, w0 + seg);
  const bool vec = a.vec_ok != 0;
  const int st_cap = (a.list_cap / kSlWarps) & ~127;  // staged entries per warp
  const int st_n = vec ? min(st_cap, (w1 - w0) & ~127) : 0;
  float* wstage = stage + warp * st_cap;
  if (lane == 0 && st_n > 0) {
    mbar_arrive_expect_tx(&fx.bar[warp], (uint32_t)st_n * 4u);
    bulk_copy_g2s(wstage, row + w0, (uint32_t)st_n * 4u, &fx.bar[warp]);
  }
  bool staged_ready = st_n == 0;
  // the page-table entries this CTA's winners will need, pulled into L2 now
  if (pt_row != nullptr && s1 > s0) {
    const int64_t p_lo = (int64_t)(kMode == kModeQsa ? kBlock : 1) * s0 / a.page_size;
    const int64_t p_hi = min(a.ld_pt - 1, ((int64_t)(kMode == kModeQsa ? kBlock : 1) * s1 - 1) / a.page_size);
    const char* b0 = reinterpret_cast<const char*>(pt_row + p_lo);
    const char* b1 = reinterpret_cast<const char*>(pt_row + p_hi);
    for (const char* q = b0 + 128 * tid; q <= b1; q += 128 * kSlThreads)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(q));
  }

  // f(i, v, full) on every chunk of this warp's segment (lane: entries
  // i..i+3, v; full: a compile-time flag, true when the whole chunk lies
  // before w1; otherwise f masks the entries at or past w1).  Staged chunks
  // first (index order) or last (any-order passes, which then start on the
  // global part while the bulk copy lands).
  auto walk = [&](bool staged_last, auto&& f) {
    for (int ph = 0; ph < 2; ++ph) {
      if ((ph == 0) != staged_last) {
        if (st_n > 0 && !staged_ready) {
          if (!mbar_wait_bounded(&fx.bar[warp], 0) && lane == 0) raise_fault(kFaultWait);
          staged_ready = true;
        }
#pragma unroll 2
        for (int c = 4 * lane; c < st_n; c += 128)
          f(w0 + c, *reinterpret_cast<const float4*>(wstage + c), std::true_type{});
      } else {
        for (int c0 = w0 + st_n; c0 < w1; c0 += 128 * kSlUnroll) {
          float4 v[kSlUnroll];
#pragma unroll
          for (int u = 0; u < kSlUnroll; ++u) v[u] = sl_load4(row, c0 + 128 * u + 4 * lane, w1, vec);
#pragma unroll
          for (int u = 0; u < kSlUnroll; ++u) f(c0 + 128 * u + 4 * lane, v[u], std::false_type{});
        }
      }
    }
  };

  // ---- sampled lower bound (the same in every CTA, no communication) ----------
  // 2048 entries in 16 runs of 128 spread evenly over the row (one 16-byte
  // load per thread).  The bound is the edge of the top-12-bit bin holding
  // the r-th largest of them, r about twice the expected number of samples
  // above the k-th entry: usually a few k entries of the row lie above it.
  // If fewer than k do, everything is redone over every entry.
  uint64_t k_low = 0ull;
  {
    const int64_t r = 2 * (((int64_t)kSlSamples * k + n - 1) / n) + 8;
    if (r < kSlSamples) {
      const int run = tid >> 5;  // kSlSamples / 128 == kSlWarps runs
      const int p = (int)((((int64_t)run * n) / kSlWarps) & ~int64_t(3)) + 4 * lane;  // n >= 2048 * 16
      const float4 v = sl_load4(row, p, n, vec);
      atomicAdd(&fx.hloc[order_key(v.x) >> 20], 1u);
      atomicAdd(&fx.hloc[order_key(v.y) >> 20], 1u);
      atomicAdd(&fx.hloc[order_key(v.z) >> 20], 1u);
      atomicAdd(&fx.hloc[order_key(v.w) >> 20], 1u);
      __syncthreads();
      const int4 f = sl_find_bin(fx, fx.hloc, (int)r);
      k_low = (uint64_t)f.x << 20;
      for (int b = tid; b < kSlBins; b += kSlThreads) fx.hloc[b] = 0u;
      __syncthreads();
    }
  }
  const SlBound low = sl_bound(k_low);

  // ---- pass 1: from HBM; each warp lists its entries at or above the bound -------
  // (key, index) in its own region of the candidate list, in any order, with
  // ballot counts (no atomics).  A warp whose region fills up marks the CTA,
  // which then works on its whole slice instead of its list.
  constexpr int kCw = kSlCandCap / kSlWarps;
  uint32_t* ckey = fx.cand_key + warp * kCw;
  uint32_t* cidx = fx.cand_idx + warp * kCw;
  uint32_t wn = 0u;  // this warp's listed entries (the same in every lane)
  walk(true, [&](int i, float4 v, auto full) {
    const float xv[4] = {v.x, v.y, v.z, v.w};
    bool c[4], any = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      c[e] = low.ge(xv[e]);
      if constexpr (!decltype(full)::value) c[e] &= i + e < w1;
      any |= c[e];
    }
    if (__ballot_sync(0xffffffffu, any) == 0u) return;
    uint32_t tot = 0u, before = 0u;
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t m = __ballot_sync(0xffffffffu, c[e]);
      tot += __popc(m);
      before += __popc(m & lt);
    }
    if (wn + tot > (uint32_t)kCw) {
      wn = kCw + 1;  // overflowed (stays so)
      return;
    }
    uint32_t o = wn + before;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (c[e]) {
        ckey[o] = order_key(xv[e]);
        cidx[o] = (uint32_t)(i + e);
        ++o;
      }
    }
    wn += tot;
  });
  if (lane == 0 && wn > (uint32_t)kCw) fx.ovf = 1;
  __syncthreads();
  const bool ovf = fx.ovf != 0;

  // ---- radix levels --------------------------------------------------------------
  // Level 0 counts the top 12 bits of the keys at or above the sampled bound
  // (all keys if the bound left fewer than k above it); levels 1 and 2 the
  // next 12 and 8 bits of the keys in the boundary bin, until a bin is taken
  // whole or the key is complete.  Each level: one histogram pass (over the
  // warps' lists, or the whole slice), every CTA adding its bins into the
  // leader's histogram of the level; the leader finds the bin of the
  // k_rem-th entry and sends it to every CTA with a retry flag (its
  // histogram held fewer than k_rem entries; it was cleared).
  uint32_t prefix = 0u;  // the k-th key's bits above `shift`
  int shift = 32, k_rem = k, lv = 0;
  bool use_list = S <= 32 * kSlBitmapWords;  // the bitmaps below cover the slice
  SlBound lo = low, hi = sl_bound(1ull << 32);
  bool first = true;
  for (;;) {
    const int nb = lv < 2 ? 12 : 8;
    const int nshift = shift - nb;
    const uint32_t mask = (1u << nb) - 1u;
    if (use_list && !ovf) {
      for (int j = lane; j < (int)wn; j += 32) {
        const uint32_t key = ckey[j];
        if (lv == 0 || (key >> shift) == prefix) atomicAdd(&fx.hloc[(key >> nshift) & mask], 1u);
      }
    } else {
      walk(true, [&](int i, float4 v, auto full) {
        // most lanes hold no entry at or above `lo`: one compare for all 4
        // (fmaxf skips NaN, which never passes unless lo takes everything)
        if (!lo.all && !(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)) >= lo.f)) return;
        const float xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          bool in = lo.ge(xv[e]) & !hi.ge(xv[e]);
          if constexpr (!decltype(full)::value) in &= i + e < w1;
          if (in) atomicAdd(&fx.hloc[(order_key(xv[e]) >> nshift) & mask], 1u);
        }
      });
    }
    __syncthreads();
    if (first) {  // the leader's cleared histograms are visible from here on
      asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
      first = false;
    }
    uint32_t* hl = &fx.hred[lv & 1][0];  // level 2 reuses level 0's histogram
    const uint32_t hr = map_shared_rank(hl, 0);
    for (int b = tid; b < kSlBins; b += kSlThreads) {
      const uint32_t c = fx.hloc[b];
      if (c != 0u) {
        fx.hloc[b] = 0u;
        red_dsmem_add_u32(hr + 4u * (uint32_t)b, c);
      }
    }
    cluster_sync();  // every CTA's bins are in the leader's histogram
    if (rank == 0) {
      const int4 f = sl_find_bin(fx, hl, k_rem);
      const int retry = f.w < k_rem ? 1 : 0;
      if (lv == 0)  // cleared for a retry or for level 2
        for (int b = tid; b < kSlBins; b += kSlThreads) hl[b] = 0u;
      if (tid < (int)C) {
        const uint32_t dst = map_shared_rank(&fx.binfo[0], (uint32_t)tid);
        st_dsmem_u32(dst, (uint32_t)f.x);
        st_dsmem_u32(dst + 4u, (uint32_t)f.y);
        st_dsmem_u32(dst + 8u, (uint32_t)f.z);
        st_dsmem_u32(dst + 12u, (uint32_t)retry);
      }
    }
    cluster_sync();  // every CTA has the leader's bin
    const int bin = fx.binfo[0], above = fx.binfo[1], cnt = fx.binfo[2], retry = fx.binfo[3];
    if (retry) {  // the sampled bound misled: every key, over the whole slice
      lo = sl_bound(0ull);
      use_list = false;
      continue;
    }
    prefix = shift == 32 ? (uint32_t)bin : ((prefix << nb) | (uint32_t)bin);
    shift = nshift;
    k_rem -= above;
    if (cnt == k_rem || lv == 2) break;
    ++lv;
    lo = sl_bound((uint64_t)prefix << shift);
    hi = sl_bound((uint64_t)(prefix + 1) << shift);
  }
  const uint32_t need = (uint32_t)k_rem;  // entries of the boundary bin to take, first by index
  lo = sl_bound((uint64_t)prefix << shift);
  hi = sl_bound((uint64_t)(prefix + 1) << shift);

  if (use_list) {
    // ---- ranks from bitmaps of the slice ------------------------------------------
    // Above the k-th key's bin (at `shift`): winners.  In it: winners while
    // fewer than `need` such entries come before them in the row.  Output
    // position = winners before it in the row.
    uint32_t* bm_eq = fx.hloc;                     // slice entries in the bin
    uint32_t* bm_win = fx.hloc + kSlBitmapWords;   // slice entries selected
    uint32_t* pre_eq = &fx.hred[0][0];             // per-word prefix counts
    uint32_t* pre_win = &fx.hred[0][0] + kSlBitmapWords;
    for (int b = tid; b < 2 * kSlBitmapWords; b += kSlThreads) fx.hloc[b] = 0u;
    __syncthreads();
    uint32_t cg = 0u, cq = 0u;
    auto mark = [&](uint32_t key, uint32_t idx) {
      const uint32_t hb = key >> shift;
      const uint32_t li = idx - (uint32_t)s0;
      if (hb > prefix) {
        atomicOr(&bm_win[li >> 5], 1u << (li & 31));
        ++cg;
      } else if (hb == prefix) {
        atomicOr(&bm_eq[li >> 5], 1u << (li & 31));
        ++cq;
      }
    };
    if (!ovf) {
      for (int j = lane; j < (int)wn; j += 32) mark(ckey[j], cidx[j]);
    } else {
      walk(true, [&](int i, float4 v, auto full) {
        if (!lo.all && !(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)) >= lo.f)) return;
        const float xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          bool in = lo.ge(xv[e]);
          if constexpr (!decltype(full)::value) in &= i + e < w1;
          if (in) mark(order_key(xv[e]), (uint32_t)(i + e));
        }
      });
    }
    cg = __reduce_add_sync(0xffffffffu, cg);
    cq = __reduce_add_sync(0xffffffffu, cq);
    if (lane == 0) {
      atomicAdd(&fx.cnt2[0], cg);
      atomicAdd(&fx.cnt2[1], cq);
    }
    __syncthreads();
    if (tid < (int)C) {
      st_dsmem_u32(map_shared_rank(&fx.cgt[rank], (uint32_t)tid), fx.cnt2[0]);
      st_dsmem_u32(map_shared_rank(&fx.ceq[rank], (uint32_t)tid), fx.cnt2[1]);
    }
    // prefix counts of set bits per bitmap word (4 words per thread)
    auto word_scan = [&](const uint32_t* bm, uint32_t* pre) {
      uint32_t c4[4], sum = 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        c4[u] = __popc(bm[4 * tid + u]);
        sum += c4[u];
      }
      uint32_t tot;
      uint32_t x = sl_block_excl_scan(fx, sum, tot);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        pre[4 * tid + u] = x;
        x += c4[u];
      }
      return tot;
    };
    static_assert(kSlBitmapWords == 4 * kSlThreads, "four bitmap words per thread");
    word_scan(bm_eq, pre_eq);
    cluster_sync();  // last remote access of the kernel
    uint32_t G = 0u, E = 0u;  // winners / bin entries of the CTAs before this one
    for (uint32_t r = 0; r < rank; ++r) {
      const uint32_t take = E >= need ? 0u : min(need - E, fx.ceq[r]);
      G += fx.cgt[r] + take;
      E += fx.ceq[r];
    }
    const uint32_t take = E >= need ? 0u : min(need - E, fx.cnt2[1]);  // this CTA's bin entries taken
    // the first `take` bin entries of the slice become winners
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int w = 4 * tid + u;
      uint32_t bits = bm_eq[w];
      uint32_t r = pre_eq[w];
      while (bits != 0u && r < take) {
        const uint32_t b = bits & (0u - bits);
        atomicOr(&bm_win[w], b);
        bits ^= b;
        ++r;
      }
    }
    __syncthreads();
    const uint32_t n_win = min(word_scan(bm_win, pre_win), (uint32_t)kSlCandCap);  // this CTA's winners
    __syncthreads();
    // The CTA's winners in output order into shared memory (the lists are no
    // longer read), then their outputs G.. from there, each thread taking
    // every kSlThreads-th one: coalesced stores, and the page-table loads of a
    // thread's outputs independent of one another.
    uint32_t* sel = fx.cand_idx;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int w = 4 * tid + u;
      uint32_t bits = bm_win[w];
      uint32_t pos = pre_win[w];
      while (bits != 0u) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1u;
        if (pos < n_win) sel[pos] = (uint32_t)(s0 + 32 * w + b);
        ++pos;
      }
    }
    __syncthreads();
    const uint32_t n_out = min(n_win, (uint32_t)k - min(G, (uint32_t)k));  // never past k (cannot happen)
    if (kMode == kModeTopk) {
#pragma unroll 4
      for (uint32_t j = tid; j < n_out; j += kSlThreads) {
        const uint32_t idx = sel[j];
        a.out_idx[(int64_t)t * k + G + j] = (int32_t)idx;
        if (a.out_slots != nullptr) a.out_slots[(int64_t)t * k + G + j] = sl_slot(a, pt_row, idx);
      }
    } else {
      if (a.out_idx != nullptr)
        for (uint32_t j = tid; j < n_out; j += kSlThreads) a.out_idx[(int64_t)t * k + G + j] = (int32_t)sel[j];
      const int64_t width = (int64_t)kBlock * k + (kBlock - 1);
      int32_t* xs = a.out_xslots + (int64_t)t * width + (int64_t)kBlock * G;
      int32_t* xp = a.out_pos != nullptr ? a.out_pos + (int64_t)t * width + (int64_t)kBlock * G : nullptr;
#pragma unroll 4
      for (uint32_t j = tid; j < kBlock * n_out; j += kSlThreads) {  // token j % 4 of winner j / 4 (one page)
        const uint32_t p0 = kBlock * sel[j / kBlock];
        const int32_t base = sl_slot(a, pt_row, p0);
        const int c = (int)(j & (kBlock - 1));
        xs[j] = base < 0 ? -1 : base + c;
        if (xp != nullptr) xp[j] = (int32_t)p0 + c;
      }
    }
    return;
  }

  // ---- counts above / in the boundary bin, per warp, then per CTA ----------------
  uint32_t g = 0u, q = 0u;
  walk(false, [&](int i, float4 v, auto) {
    const float xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool ok = i + e < w1;
      const bool gt = ok & hi.ge(xv[e]);
      g += gt;
      q += ok & !gt & lo.ge(xv[e]);
    }
  });
  const uint32_t wg = __reduce_add_sync(0xffffffffu, g), wq = __reduce_add_sync(0xffffffffu, q);
  if (lane == 0) {
    fx.wg[warp] = wg;
    fx.wq[warp] = wq;
  }
  __syncthreads();
  uint32_t bg = 0u, bq = 0u, cg = 0u, cq = 0u;  // before this warp in the CTA; CTA totals
#pragma unroll
  for (int w = 0; w < kSlWarps; ++w) {
    const uint32_t x = fx.wg[w], y = fx.wq[w];
    if (w < warp) {
      bg += x;
      bq += y;
    }
    cg += x;
    cq += y;
  }
  if (tid < (int)C) {
    st_dsmem_u32(map_shared_rank(&fx.cgt[rank], (uint32_t)tid), cg);
    st_dsmem_u32(map_shared_rank(&fx.ceq[rank], (uint32_t)tid), cq);
  }
  cluster_sync();  // last remote access of the kernel
  uint32_t G = bg, E = bq;
  for (uint32_t r = 0; r < rank; ++r) {
    G += fx.cgt[r];
    E += fx.ceq[r];
  }

  // ---- emission: ascending positions, every CTA at once ---------------------------
  // Winners are listed (index, output position) in this CTA's shared memory
  // (the level histogram is free now; a CTA has at most k winners), then
  // written out by all threads, so the page-table lookups are independent.
  uint32_t* e_idx = fx.hloc;
  uint32_t* e_pos = fx.hloc + kMaxK;
  walk(false, [&](int i, float4 v, auto) {
    const float xv[4] = {v.x, v.y, v.z, v.w};
    uint32_t fl = 0u, pk = 0u;  // per entry: bit 2e above, bit 2e+1 in the boundary bin
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool ok = i + e < w1;
      const bool gt = ok & hi.ge(xv[e]);
      const bool eq = ok & !gt & lo.ge(xv[e]);
      fl |= (gt ? 1u : 0u) << (2 * e);
      fl |= (eq ? 1u : 0u) << (2 * e + 1);
      pk += gt ? 1u : (eq ? 0x10000u : 0u);
    }
    if (__ballot_sync(0xffffffffu, pk != 0u) != 0u) {
      const uint32_t incl = sl_warp_incl_scan(pk);
      const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
      uint32_t lg = G + ((incl - pk) & 0xffffu), lq = E + ((incl - pk) >> 16);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool gt = (fl >> (2 * e)) & 1u, eq = (fl >> (2 * e + 1)) & 1u;
        if (gt || (eq && lq < need)) {
          const uint32_t slot = atomicAdd(&fx.n_emit, 1u);
          e_idx[slot] = (uint32_t)(i + e);
          e_pos[slot] = lg + (lq < need ? lq : need);
        }
        lg += gt;
        lq += eq;
      }
      G += total & 0xffffu;
      E += total >> 16;
    }
  });
  __syncthreads();
  const int ne = (int)fx.n_emit;
  for (int j = tid; j < ne; j += kSlThreads) emit(e_idx[j], (int)e_pos[j]);
}

}  // namespace qsa
