// select_rows.cuh -- exact top-k of many rows of up to 32768 entries: one
// small CTA per row, four per SM, so that launches with more rows than SMs
// (a batch of verify steps, a prefill chunk of thousands of rows) run in few
// waves and the rows stream at HBM rate instead of one row per SM.
//
// Same contract as select_kernel (SGLang GLM-5.2 blog, "Kernel Optimization /
// TopK-V2": a selection, not a sort; exactly k entries, exact ties, runtime k
// up to 2048; the page-table transform in the same kernel.  Qwen3.8-Flash-Next
// write-up, "Qwen sparse attention (QSA)": blocks -> 4 positions each, then
// the 0-3 pending tokens; -1 marks an empty entry).  Readings: ties go to the
// lower index; -0 == +0; NaN ranks below -inf; ascending index order.
//
// Design (the single-CTA form of select_long_kernel's list path).  256
// threads; warp w owns a contiguous segment of the row, walked 128 entries
// at a time (4 consecutive per lane) with 16-byte loads, 4 in flight.  The
// outputs read the page table through L2 (shared memory is kept to 54 KB so
// that four CTAs fit an SM: the rows are latency-bound, and a fourth CTA
// per SM took a 4096-row prefill chunk from 274 to 244 us).
//  1. Sampled bound: 1024 entries in 32 runs of 32 (one 16-byte load per
//     thread); the edge of the top-12-bit bin below which the r-th largest
//     sample lies, r about twice the expected number of samples above the
//     k-th entry.
//  2. One pass over the row: each warp lists its entries at or above the
//     bound (float bits, index) in its own region of a shared-memory list, with
//     ballot counts.  A warp whose region fills up makes the CTA walk the
//     whole row in the steps below instead of the list.
//  3. Radix levels of 12, 12 and 8 bits over the list (or the row) in a
//     shared-memory histogram, until a bin is taken whole or the key is
//     complete.  Fewer than k entries above the bound (the sample misled):
//     level 0 again over every entry of the row.
//  4. Two bitmaps of the row (entries above the k-th key's bin, entries in
//     it) and prefix counts of their words give the first `need` entries of
//     the bin and every winner's ascending output position; the winners'
//     indices are placed in that order in shared memory and the outputs are
//     written from there by all threads, each taking every 256-th output.
// Every wait is a CTA barrier; no global scratch.
#pragma once
#include <type_traits>

#include "select_long.cuh"

namespace qsa {

constexpr int kSrThreads = 256;
constexpr int kSrWarps = kSrThreads / 32;
constexpr int kSrMaxRow = 32768;
constexpr int kSrBins = 4096;
constexpr int kSrCandCap = 3840;                 // list entries per CTA (per warp: / kSrWarps)
constexpr int kSrWords = kSrMaxRow / 32;         // bitmap words
constexpr int kSrUnroll = 4;

struct SrSmem {
  uint32_t hist[kSrBins];
  uint32_t cand_val[kSrCandCap];  // the candidates' float bits (keys are made when read)
  uint32_t cand_idx[kSrCandCap];
  uint32_t bm_eq[kSrWords];
  uint32_t bm_win[kSrWords];
  uint32_t wsum[kSrWarps];
  int info[4];
  int ovf;
};

__device__ __forceinline__ uint32_t sr_block_excl_scan(SrSmem& sm, uint32_t x, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = sl_warp_incl_scan(x);
  if (lane == 31) sm.wsum[warp] = incl;
  __syncthreads();
  uint32_t before = 0u, tot = 0u;
#pragma unroll
  for (int w = 0; w < kSrWarps; ++w) {
    const uint32_t v = sm.wsum[w];
    before += w < warp ? v : 0u;
    tot += v;
  }
  total = tot;
  __syncthreads();
  return before + incl - x;
}

// (bin, entries in higher bins, entries in the bin, total) of the k_rem-th
// largest entry of sm.hist; the first three are 0 when k_rem > total.
__device__ __forceinline__ int4 sr_find_bin(SrSmem& sm, int k_rem) {
  constexpr int kPer = kSrBins / kSrThreads;  // 16
  const int top = kSrBins - 1 - kPer * (int)threadIdx.x;
  uint32_t c[kPer];
  uint32_t s = 0u;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    c[j] = sm.hist[top - j];
    s += c[j];
  }
  if (threadIdx.x < 3) sm.info[threadIdx.x] = 0;
  uint32_t tot;
  uint32_t above = sr_block_excl_scan(sm, s, tot);
  const uint32_t kr = (uint32_t)k_rem;
  if (above < kr && kr <= above + s) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (above < kr && kr <= above + c[j]) {
        sm.info[0] = top - j;
        sm.info[1] = (int)above;
        sm.info[2] = (int)c[j];
      }
      above += c[j];
    }
  }
  __syncthreads();
  const int4 r = make_int4(sm.info[0], sm.info[1], sm.info[2], (int)tot);
  __syncthreads();
  return r;
}

// four CTAs per SM: at most 56 KB of shared memory and 64 registers each
static_assert(sizeof(SrSmem) + 1024 <= 228 * 1024 / 4, "four CTAs per SM");
static_assert(2 * kSrWords <= kSrBins, "the word prefix counts reuse the histogram");

template <int kMode>
__global__ void __launch_bounds__(kSrThreads, 4)
select_rows_kernel(SelectArgs a) {
  extern __shared__ __align__(16) unsigned char sr_smem_raw[];
  SrSmem& sm = *reinterpret_cast<SrSmem*>(sr_smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int t;
  if (!sel_unit_row(a, blockIdx.x, t)) return;

  // ---- row metadata (not produced by the previous grid) ---------------------------
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
  if (n < 0 || n > a.n_max || n > kSrMaxRow || L < 0) {  // bad length: emit an empty row
    if (tid == 0) raise_fault(kFaultGrouping);
    n = 0;
    L = 0;
  }
  for (int i = tid; i < kSrBins; i += kSrThreads) sm.hist[i] = 0u;
  if (tid == 0) sm.ovf = 0;
  if (a.wait_primary) pdl_wait_primary();
  const float* row = a.scores + (int64_t)t * a.ld;
  const int k = a.k;
  const int m_sel = n < k ? n : k;
  const bool vec = a.vec_ok != 0;

  auto slot = [&](uint32_t pos) -> int32_t { return sl_slot(a, pt_row, pos); };
  auto emit = [&](uint32_t idx, int pos) {
    if (kMode == kModeTopk) {
      a.out_idx[(int64_t)t * k + pos] = (int32_t)idx;
      if (a.out_slots != nullptr) a.out_slots[(int64_t)t * k + pos] = slot(idx);
    } else {
      if (a.out_idx != nullptr) a.out_idx[(int64_t)t * k + pos] = (int32_t)idx;
      const int64_t width = (int64_t)kBlock * k + (kBlock - 1);
      const uint32_t p0 = kBlock * idx;  // 4 positions in one page
      const int32_t base = slot(p0);
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

  __syncthreads();
  // ---- the tail after m_sel entries ----------------------------------------------
  if (kMode == kModeTopk) {
    for (int j = m_sel + tid; j < k; j += kSrThreads) {
      a.out_idx[(int64_t)t * k + j] = -1;
      if (a.out_slots != nullptr) a.out_slots[(int64_t)t * k + j] = -1;
    }
  } else {
    if (a.out_idx != nullptr)
      for (int j = m_sel + tid; j < k; j += kSrThreads) a.out_idx[(int64_t)t * k + j] = -1;
    const int width = kBlock * k + (kBlock - 1);
    const int pend = L - kBlock * n;
    for (int j = kBlock * m_sel + tid; j < width; j += kSrThreads) {
      const int i = j - kBlock * m_sel;
      int32_t pos = -1, sl = -1;
      if (i < pend) {
        pos = kBlock * n + i;
        sl = slot((uint32_t)pos);
      }
      a.out_xslots[(int64_t)t * width + j] = sl;
      if (a.out_pos != nullptr) a.out_pos[(int64_t)t * width + j] = pos;
    }
  }
  if (n <= k) {  // every entry is selected, in order
    for (int j = tid; j < m_sel; j += kSrThreads) emit(j, j);
    return;
  }

  // ---- warp segments and the row walk ---------------------------------------------
  const int seg = (((n + kSrWarps - 1) / kSrWarps) + 127) & ~127;
  const int w0 = min(n, warp * seg);
  const int w1 = min(n, w0 + seg);
  // f(i, v, full) on every 128-entry chunk of this warp's segment (lane:
  // entries i..i+3; full: the chunk lies before w1, else f masks entries
  // from w1 on, which read as NaN)
  auto walk = [&](auto&& f) {
    for (int c0 = w0; c0 < w1; c0 += 128 * kSrUnroll) {
      float4 v[kSrUnroll];
      if (vec && c0 + 128 * kSrUnroll <= w1) {
#pragma unroll
        for (int u = 0; u < kSrUnroll; ++u)
          v[u] = __ldg(reinterpret_cast<const float4*>(row + c0 + 128 * u + 4 * lane));
#pragma unroll
        for (int u = 0; u < kSrUnroll; ++u) f(c0 + 128 * u + 4 * lane, v[u], std::true_type{});
      } else {
#pragma unroll
        for (int u = 0; u < kSrUnroll; ++u) v[u] = sl_load4(row, c0 + 128 * u + 4 * lane, w1, vec);
#pragma unroll
        for (int u = 0; u < kSrUnroll; ++u) f(c0 + 128 * u + 4 * lane, v[u], std::false_type{});
      }
    }
  };

  // f2(i, va, vb, full) on every pair of 128-entry chunks (lane: entries
  // i..i+3 and i+128..i+131; the list pass takes 8 entries per lane per
  // round of ballots)
  auto walk2 = [&](auto&& f2) {
    static_assert(kSrUnroll % 2 == 0, "chunks go in pairs");
    for (int c0 = w0; c0 < w1; c0 += 128 * kSrUnroll) {
      float4 v[kSrUnroll];
      if (vec && c0 + 128 * kSrUnroll <= w1) {
#pragma unroll
        for (int u = 0; u < kSrUnroll; ++u)
          v[u] = __ldg(reinterpret_cast<const float4*>(row + c0 + 128 * u + 4 * lane));
#pragma unroll
        for (int u = 0; u < kSrUnroll; u += 2) f2(c0 + 128 * u + 4 * lane, v[u], v[u + 1], std::true_type{});
      } else {
#pragma unroll
        for (int u = 0; u < kSrUnroll; ++u) v[u] = sl_load4(row, c0 + 128 * u + 4 * lane, w1, vec);
#pragma unroll
        for (int u = 0; u < kSrUnroll; u += 2) f2(c0 + 128 * u + 4 * lane, v[u], v[u + 1], std::false_type{});
      }
    }
  };

  // ---- 1. sampled bound -------------------------------------------------------------
  // The r-th largest of 1024 sampled keys, r = mu + 3.5 sqrt(mu) + 2 with mu
  // = 1024 k / n the expected number of samples among the row's k largest:
  // below the k-th largest entry unless the sample is off by 3.5 standard
  // deviations (then the exact passes run over the row).
  uint64_t k_low = 0ull;
  {
    const float mu = 1024.0f * (float)k / (float)n;
    const int64_t r = (int64_t)ceilf(mu + 3.5f * sqrtf(mu) + 2.0f);
    if (r < 1024) {
      const int run = tid >> 3;  // 32 runs of 32
      const int p = (int)((((int64_t)run * n) / 32) & ~int64_t(3)) + 4 * (tid & 7);
      const float4 v = sl_load4(row, p, n, vec);
      const bool ok0 = p < n, ok1 = p + 1 < n, ok2 = p + 2 < n, ok3 = p + 3 < n;
      __syncthreads();  // the histogram is cleared
      if (ok0) atomicAdd(&sm.hist[order_key(v.x) >> 20], 1u);
      if (ok1) atomicAdd(&sm.hist[order_key(v.y) >> 20], 1u);
      if (ok2) atomicAdd(&sm.hist[order_key(v.z) >> 20], 1u);
      if (ok3) atomicAdd(&sm.hist[order_key(v.w) >> 20], 1u);
      __syncthreads();
      const int4 f = sr_find_bin(sm, (int)r);
      k_low = (uint64_t)f.x << 20;
      for (int b = tid; b < kSrBins; b += kSrThreads) sm.hist[b] = 0u;
    }
  }
  __syncthreads();
  const SlBound low = sl_bound(k_low);

  // ---- 2. one pass: each warp lists its entries at or above the bound ----------------
  constexpr int kCw = kSrCandCap / kSrWarps;
  uint32_t* cval = sm.cand_val + warp * kCw;
  uint32_t* cidx = sm.cand_idx + warp * kCw;
  uint32_t wn = 0u;  // the same in every lane of the warp
  // Candidates are a few per cent of the row: a lane's (up to 8 per round)
  // are written in a loop over its mask (mostly no iteration), placed by
  // four ballots of the lanes' counts.
  const uint32_t lt = (1u << lane) - 1u;
  walk2([&](int i, float4 va, float4 vb, auto full) {
    const float xv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
    uint32_t cm = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      bool ce = low.ge(xv[e]);
      if (!decltype(full)::value) ce = ce & ((e < 4 ? i + e : i + 124 + e) < w1);
      cm |= (uint32_t)ce << e;
    }
    if (__ballot_sync(0xffffffffu, cm != 0u) == 0u) return;
    const uint32_t c = __popc(cm);
    const uint32_t b0 = __ballot_sync(0xffffffffu, c & 1u), b1 = __ballot_sync(0xffffffffu, c & 2u),
                   b2 = __ballot_sync(0xffffffffu, c & 4u), b3 = __ballot_sync(0xffffffffu, c & 8u);
    const uint32_t tot = __popc(b0) + 2u * __popc(b1) + 4u * __popc(b2) + 8u * __popc(b3);
    if (wn + tot > (uint32_t)kCw) {
      wn = kCw + 1;  // overflowed (stays so)
      return;
    }
    uint32_t o = wn + __popc(b0 & lt) + 2u * __popc(b1 & lt) + 4u * __popc(b2 & lt) + 8u * __popc(b3 & lt);
    while (cm != 0u) {
      const int e = __ffs(cm) - 1;
      cm &= cm - 1u;
      const float4& h = e < 4 ? va : vb;
      const int q = e & 3;
      const float x = q == 0 ? h.x : (q == 1 ? h.y : (q == 2 ? h.z : h.w));
      cval[o] = __float_as_uint(x);
      cidx[o] = (uint32_t)(e < 4 ? i + e : i + 124 + e);
      ++o;
    }
    wn += tot;
  });
  if (lane == 0 && wn > (uint32_t)kCw) sm.ovf = 1;
  __syncthreads();
  bool use_list = sm.ovf == 0;

  // ---- 3. radix levels ------------------------------------------------------------------
  uint32_t prefix = 0u;  // the k-th key's bits above `shift`
  int shift = 32, k_rem = k, lv = 0;
  SlBound lo = low, hi = sl_bound(1ull << 32);
  for (;;) {
    const int nb = lv < 2 ? 12 : 8;
    const int nshift = shift - nb;
    const uint32_t mask = (1u << nb) - 1u;
    if (use_list) {
      for (int j = lane; j < (int)wn; j += 32) {
        const uint32_t key = order_key(__uint_as_float(cval[j]));
        if (lv == 0 || (key >> shift) == prefix) atomicAdd(&sm.hist[(key >> nshift) & mask], 1u);
      }
    } else {
      walk([&](int i, float4 v, auto) {
        if (!lo.all && !(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)) >= lo.f)) return;
        const float xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool in = lo.ge(xv[e]) & !hi.ge(xv[e]) & (i + e < w1);
          if (in) atomicAdd(&sm.hist[(order_key(xv[e]) >> nshift) & mask], 1u);
        }
      });
    }
    __syncthreads();
    const int4 f = sr_find_bin(sm, k_rem);  // its barriers order the clear below
    for (int b = tid; b < kSrBins; b += kSrThreads) sm.hist[b] = 0u;
    if (lv == 0 && f.w < k_rem) {  // the sampled bound misled: every entry of the row
      lo = sl_bound(0ull);
      use_list = false;
      __syncthreads();
      continue;
    }
    prefix = shift == 32 ? (uint32_t)f.x : ((prefix << nb) | (uint32_t)f.x);
    shift = nshift;
    k_rem -= f.y;
    __syncthreads();
    if (f.z == k_rem || lv == 2) break;
    ++lv;
    lo = sl_bound((uint64_t)prefix << shift);
    hi = sl_bound((uint64_t)(prefix + 1) << shift);
  }
  const uint32_t need = (uint32_t)k_rem;  // entries of the boundary bin to take, first by index
  lo = sl_bound((uint64_t)prefix << shift);

  // ---- 4. ranks from bitmaps of the row, outputs ----------------------------------------
  for (int b = tid; b < kSrWords; b += kSrThreads) {
    sm.bm_eq[b] = 0u;
    sm.bm_win[b] = 0u;
  }
  __syncthreads();
  auto mark = [&](uint32_t key, uint32_t idx) {
    const uint32_t hb = key >> shift;
    if (hb > prefix) atomicOr(&sm.bm_win[idx >> 5], 1u << (idx & 31));
    else if (hb == prefix) atomicOr(&sm.bm_eq[idx >> 5], 1u << (idx & 31));
  };
  if (use_list) {
    for (int j = lane; j < (int)wn; j += 32) mark(order_key(__uint_as_float(cval[j])), cidx[j]);
  } else {
    walk([&](int i, float4 v, auto) {
      if (!lo.all && !(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)) >= lo.f)) return;
      const float xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (lo.ge(xv[e]) & (i + e < w1)) mark(order_key(xv[e]), (uint32_t)(i + e));
    });
  }
  __syncthreads();
  // prefix counts of set bits per word (kSrWords / kSrThreads words per thread)
  constexpr int kWpt = kSrWords / kSrThreads;
  auto word_scan = [&](const uint32_t* bm, uint32_t* pre) {
    uint32_t c[kWpt], sum = 0u;
#pragma unroll
    for (int u = 0; u < kWpt; ++u) {
      c[u] = __popc(bm[kWpt * tid + u]);
      sum += c[u];
    }
    uint32_t tot;
    uint32_t x = sr_block_excl_scan(sm, sum, tot);
#pragma unroll
    for (int u = 0; u < kWpt; ++u) {
      pre[kWpt * tid + u] = x;
      x += c[u];
    }
  };
  uint32_t* pre_eq = sm.hist;  // the histogram is free from here on
  uint32_t* pre_win = sm.hist + kSrWords;
  word_scan(sm.bm_eq, pre_eq);
  __syncthreads();
  // the first `need` entries of the bin become winners
#pragma unroll
  for (int u = 0; u < kWpt; ++u) {
    const int w = kWpt * tid + u;
    uint32_t bits = sm.bm_eq[w];
    uint32_t r = pre_eq[w];
    while (bits != 0u && r < need) {
      const uint32_t b = bits & (0u - bits);
      atomicOr(&sm.bm_win[w], b);
      bits ^= b;
      ++r;
    }
  }
  __syncthreads();
  word_scan(sm.bm_win, pre_win);
  __syncthreads();
  // the winners' indices in output order into shared memory (the lists are
  // no longer read), then the outputs from there, each thread taking every
  // kSrThreads-th one: coalesced stores, and the page-table loads of a
  // thread's outputs independent of one another (writing a word's winners
  // from its thread chained one L2 load per winner)
  uint32_t* sel = sm.cand_idx;
#pragma unroll
  for (int u = 0; u < kWpt; ++u) {
    const int w = kWpt * tid + u;
    uint32_t bits = sm.bm_win[w];
    uint32_t pos = pre_win[w];
    while (bits != 0u) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      if (pos < (uint32_t)k) sel[pos] = (uint32_t)(32 * w + b);
      ++pos;
    }
  }
  __syncthreads();
  if (kMode == kModeTopk) {
#pragma unroll 4
    for (int j = tid; j < k; j += kSrThreads) {
      const uint32_t idx = sel[j];
      a.out_idx[(int64_t)t * k + j] = (int32_t)idx;
      if (a.out_slots != nullptr) a.out_slots[(int64_t)t * k + j] = slot(idx);
    }
  } else {
    if (a.out_idx != nullptr)
      for (int j = tid; j < k; j += kSrThreads) a.out_idx[(int64_t)t * k + j] = (int32_t)sel[j];
    const int64_t width = (int64_t)kBlock * k + (kBlock - 1);
    int32_t* xs = a.out_xslots + (int64_t)t * width;
    int32_t* xp = a.out_pos != nullptr ? a.out_pos + (int64_t)t * width : nullptr;
#pragma unroll 4
    for (int j = tid; j < kBlock * k; j += kSrThreads) {  // token j % 4 of winner j / 4 (one page)
      const uint32_t p0 = kBlock * sel[j / kBlock];
      const int32_t base = slot(p0);
      const int c = j & (kBlock - 1);
      xs[j] = base < 0 ? -1 : base + c;
      if (xp != nullptr) xp[j] = (int32_t)p0 + c;
    }
  }
}

}  // namespace qsa
