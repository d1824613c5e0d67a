// select_fast.cuh -- low-latency exact top-k of one score row per CTA (rows
// of up to 32768 entries, k <= 1024), fused with the page-table transform
// (token mode) or the QSA expansion to positions and slots.
//
// SGLang GLM-5.2 blog (aihot.virxact.com), section "Kernel Optimization /
// TopK-V2": top-k as a selection with an exact tie-break and the page-table
// transform in the same kernel.  Qwen3.8-Flash-Next day-0 write-up
// (theainews.cc), section "Qwen sparse attention (QSA)": keep the best 512
// blocks, each standing for its 4 token positions, then the 0-3 pending
// tokens.  Readings as in select.cuh: ties to the lower index, -0 == +0, NaN
// below -inf, ascending output, -1 only as tail padding.
//
// The row is loaded once into registers (8 float4 per thread, index
// 4 * (thread + 1024 j) + c); two passes over them (thread maxima, then the
// candidates) and every later step works on a short list in shared memory:
//  1. Lower bound without sorting the row: every thread's maximum, then per
//     full warp (32 lanes holding entries, F such warps) the ceil(k/F)-th
//     largest of its lane maxima (one 32-lane bitonic sort in registers);
//     v = the smallest of those.  Each full warp has ceil(k/F) lanes whose
//     maxima are >= v, so at least k entries are >= v: only those are
//     candidates (about 2k for a row of 20K-32K).
//  2. A count, a warp scan and a write pass list the candidates of each warp
//     in shared memory and add them to a 2048-bin histogram of
//     (key - v) >> s, s chosen so the candidates' key range fits; a block
//     scan from the top finds the bin holding the k-th largest key.  Every
//     later step reads only the lists.  (A warp with more than 128
//     candidates -- heavy ties -- sends the row to the same steps over every
//     entry, read again from L2.)
//  3. The boundary bin, when it holds at most 64 entries (the usual case),
//     is resolved exactly by one warp (rank by counting); otherwise further
//     radix passes on the next bits (two histograms alternate, so no extra
//     barrier clears them).
//  4. Ordered emission through a bitmap of the row (one bit per entry, one
//     32-bit word per thread): entries above T set their bit; entries equal
//     to T too when all of them are taken, otherwise they go to a second
//     bitmap whose first `need` set bits (a block scan of its words'
//     popcounts) are added.  A block scan of the words' popcounts then gives
//     each thread the output position of its first set bit; it places the
//     indices of its set bits in that order in shared memory, and the
//     outputs (indices, or the 4 positions and slots of each block) are
//     written from there, every thread taking every 1024-th output.
// With 32 warps on the SM every per-entry instruction costs 8 issue slots per
// scheduler, so each step is a short loop body over the 32 entries held in
// registers, and the emission code is a single loop (not one copy per
// register).  Barriers: about 10 per row; nothing is staged in global memory.
#pragma once

#include "select.cuh"

namespace qsa {

constexpr int kSfThreads = 1024;   // == kSelThreads: emit_tail strides by it
constexpr int kSfWarps = kSfThreads / 32;
constexpr int kSfRuns = 8;         // float4 per thread
constexpr int kSfMaxRow = 4 * kSfThreads * kSfRuns;  // 32768 entries
constexpr int kSfMaxK = 1024;      // ceil(k / 32) lane maxima per warp
constexpr int kSfBins = 2048;
constexpr int kSfList = 64;        // boundary entries resolved by one warp
constexpr int kSfPtCap = 2560;     // page-table entries staged in shared memory (131K tokens at 64)
static_assert(kSfThreads == kSelThreads, "emit_tail walks rows with kSelThreads strides");

constexpr int kSfReqStage = 1024;  // request starts staged for the row -> request search

constexpr int kSfWarpCap = 128;   // candidates listed per warp (more: the register path)

struct SfShared {
  uint32_t hist[2][kSfBins];
  uint32_t lkey[kSfWarps * kSfWarpCap];  // candidate keys, per-warp lists
  uint16_t lidx[kSfWarps * kSfWarpCap];  // their row indices (< 32768)
  uint32_t wcnt[kSfWarps];
  uint32_t bm[kSfMaxRow / 32];  // selected entries
  uint32_t tm[kSfMaxRow / 32];  // entries equal to T (when only some are taken)
  uint32_t list[kSfList];
  uint32_t wv[kSfWarps];        // per-warp lower bound
  uint32_t wmax[kSfWarps];      // per-warp maximum
  uint32_t wsum[kSfWarps];      // block-scan partials
  int info[8];                  // bin, above, count, T, need, list length
  int32_t pt[kSfPtCap];
  int32_t rrs[kSfReqStage + 1];
};

// Exclusive block scan of one value per thread (two barriers); `total`
// receives the sum over the CTA.
__device__ __forceinline__ uint32_t sf_block_excl_scan(SfShared& sh, uint32_t x, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  const uint32_t w = sh.wsum[lane];
  const uint32_t before = __reduce_add_sync(0xffffffffu, lane < warp ? w : 0u);
  total = __reduce_add_sync(0xffffffffu, w);
  __syncthreads();  // wsum may be rewritten by the next caller
  return before + incl - x;
}

__device__ __forceinline__ uint32_t warp_incl_scan_u32(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Bins of `h` listed from the top (bin 2047 first, 2 per thread): the bin
// holding the k_rem-th largest key -> info[0] = bin, info[1] = keys above it,
// info[2] = its count.  Two barriers; every thread takes part.
__device__ __forceinline__ void sf_find_bin(SfShared& sh, const uint32_t* h, int k_rem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b_hi = kSfBins - 1 - 2 * (int)threadIdx.x;
  const uint32_t c_hi = h[b_hi], c_lo = h[b_hi - 1];
  const uint32_t sum = c_hi + c_lo;
  const uint32_t incl = warp_incl_scan_u32(sum);
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  const uint32_t before = __reduce_add_sync(0xffffffffu, lane < warp ? sh.wsum[lane] : 0u);
  const int above = (int)(before + incl - sum);
  if (above < k_rem && k_rem <= above + (int)c_hi) {
    sh.info[0] = b_hi;
    sh.info[1] = above;
    sh.info[2] = (int)c_hi;
  } else if (above + (int)c_hi < k_rem && k_rem <= above + (int)sum) {
    sh.info[0] = b_hi - 1;
    sh.info[1] = above + (int)c_hi;
    sh.info[2] = (int)c_lo;
  }
  __syncthreads();
}

// Outputs of a row from its winners' indices in output order (sel[0, m)):
// the same values as emit_one for each of them followed by emit_tail(m), each
// thread writing every kSfThreads-th output (coalesced stores).
template <int kMode>
__device__ __forceinline__ void sf_emit_sorted(const SelectArgs& a, const SelRow& r, const uint32_t* sel, int m) {
  const int t = r.t, k = a.k;
  if (kMode == kModeTopk) {
    for (int j = threadIdx.x; j < k; j += kSfThreads) {
      const int idx = j < m ? (int)sel[j] : -1;
      a.out_idx[(int64_t)t * k + j] = idx;
      if (a.out_slots != nullptr) a.out_slots[(int64_t)t * k + j] = idx < 0 ? -1 : slot_lookup(a, r, idx);
    }
  } else {
    if (a.out_idx != nullptr)
      for (int j = threadIdx.x; j < k; j += kSfThreads) a.out_idx[(int64_t)t * k + j] = j < m ? (int32_t)sel[j] : -1;
    const int width = kBlock * k + (kBlock - 1);
    const int nb = r.L / kBlock, pend = r.L - kBlock * nb;
    int32_t* xs = a.out_xslots + (int64_t)t * width;
    int32_t* xp = a.out_pos != nullptr ? a.out_pos + (int64_t)t * width : nullptr;
    for (int j = threadIdx.x; j < width; j += kSfThreads) {
      int32_t pos = -1, slot = -1;
      if (j < kBlock * m) {  // token c of the winner j / 4 (its block's 4 tokens share a page)
        const int c = j & (kBlock - 1);
        const int32_t p0 = kBlock * (int32_t)sel[j / kBlock];
        const int32_t base = slot_lookup(a, r, p0);
        slot = base < 0 ? -1 : base + c;
        pos = p0 + c;
      } else {
        const int i = j - kBlock * m;
        if (i < pend) {
          pos = kBlock * nb + i;
          slot = slot_lookup(a, r, pos);
        }
      }
      xs[j] = slot;
      if (xp != nullptr) xp[j] = pos;
    }
  }
}

template <int kMode>
__global__ void __launch_bounds__(kSfThreads, 1) select_fast_kernel(SelectArgs a) {
  extern __shared__ __align__(16) unsigned char sf_raw[];  // sizeof(SfShared) bytes
  SfShared& sh = *reinterpret_cast<SfShared*>(sf_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  SelRow r;
  if (!sel_unit_row(a, blockIdx.x, r.t)) return;
  r.L = 0;
  r.pt_row = nullptr;
  r.pt_s = sh.pt;
  r.pt_n = 0;
  // ---- row metadata and page-table entries (not produced by the scorer) --
  if (kMode == kModeTopk) {
    r.n = a.n_valid ? __ldg(a.n_valid + r.t) : a.n_max;
    if (a.out_slots != nullptr)
      r.pt_row = a.page_table + (int64_t)(a.row_req ? __ldg(a.row_req + r.t) : r.t) * a.ld_pt;
  } else {
    int req;
    if (a.n_req <= kSfReqStage) {  // the request starts in shared memory, then a search there
      for (int i = threadIdx.x; i <= a.n_req; i += kSfThreads) sh.rrs[i] = __ldg(a.req_row_start + i);
      __syncthreads();
      int lo = 0, hi = a.n_req - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sh.rrs[mid] <= r.t) lo = mid; else hi = mid - 1;
      }
      req = lo;
    } else {
      req = row_request(a.req_row_start, a.n_req, r.t);
    }
    r.L = __ldg(a.row_len + r.t);
    r.n = r.L / kBlock;
    r.pt_row = a.page_table + (int64_t)req * a.ld_pt;
  }
  if (r.n < 0 || r.n > a.n_max || r.n > kSfMaxRow) {  // bad length: an empty row
    if (threadIdx.x == 0) raise_fault(kFaultGrouping);
    r.n = 0;
    r.L = 0;
  }
  if (r.pt_row != nullptr) {
    const int64_t last = kMode == kModeQsa ? (int64_t)r.L : (int64_t)r.n;  // positions < last
    int64_t np = last > 0 ? (last - 1) / a.page_size + 1 : 0;
    if (np > kSfPtCap) np = kSfPtCap;
    if (np > a.ld_pt) np = a.ld_pt;
    r.pt_n = (int)np;
    for (int i = threadIdx.x; i < r.pt_n; i += kSfThreads) sh.pt[i] = __ldg(r.pt_row + i);
  }
  for (int i = threadIdx.x; i < 2 * kSfBins; i += kSfThreads) (&sh.hist[0][0])[i] = 0u;
  sh.bm[threadIdx.x] = 0u;
  sh.tm[threadIdx.x] = 0u;
  // info: bin (-1 = none), above, count, T, need, boundary list length, ties
  if (threadIdx.x < 8) sh.info[threadIdx.x] = threadIdx.x == 0 ? -1 : (threadIdx.x == 3 ? -1 : 0);

  if (a.wait_primary) pdl_wait_primary();
  const int n = r.n;
  const float* row = a.scores + (int64_t)r.t * a.ld;

  if (n <= a.k) {  // everything is selected: entry i goes to output position i
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kSfThreads) emit_one<kMode>(a, r, i, i);
    emit_tail<kMode>(a, r, n);
    return;
  }

  // ---- load: 32 floats per thread; entries past the row read as NaN (never
  // a candidate on the list path).  Rows of more than 4096 entries: index
  // 4 * (thread + 1024 j) + c (float4 loads); shorter rows: thread + 1024 c,
  // so every thread holds an entry when n >= 1024 (a tighter bound below).
  const bool small = n <= 4 * kSfThreads;
  auto index_of = [&](int j, int c) {
    return small ? (int)threadIdx.x + kSfThreads * c : 4 * ((int)threadIdx.x + kSfThreads * j) + c;
  };
  const float qnan = __int_as_float(0x7fffffff);
  float xs[kSfRuns][4];
#pragma unroll
  for (int j = 0; j < kSfRuns; ++j) {
    const int i = 4 * ((int)threadIdx.x + kSfThreads * j);
    if (small) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = (int)threadIdx.x + kSfThreads * c;
        xs[j][c] = (j == 0 && e < n) ? __ldcg(row + e) : qnan;
      }
    } else if (a.vec_ok && i + 3 < n) {
      const float4 q4 = __ldcg(reinterpret_cast<const float4*>(row + i));
      xs[j][0] = q4.x;
      xs[j][1] = q4.y;
      xs[j][2] = q4.z;
      xs[j][3] = q4.w;
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) xs[j][c] = i + c < n ? __ldcg(row + i + c) : qnan;
    }
  }

  // ---- 1. lower bound v (as key + 1; 0 = no entry) from the lane maxima ----
  uint32_t v, M;
  {
    float mf = xs[0][0];
#pragma unroll
    for (int j = 0; j < kSfRuns; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) mf = fmaxf(mf, xs[j][c]);  // NaN only if every entry is NaN
    const bool has = small ? (int)threadIdx.x < n : 4 * (int)threadIdx.x < n;
    uint32_t x = has ? order_key(mf) + 1u : 0u;
    // ascending bitonic sort of the 32 lane maxima
#pragma unroll
    for (int kb = 2; kb <= 32; kb <<= 1) {
#pragma unroll
      for (int jb = kb >> 1; jb > 0; jb >>= 1) {
        const uint32_t y = __shfl_xor_sync(0xffffffffu, x, jb);
        const bool lower = (lane & jb) == 0, asc = (lane & kb) == 0;
        x = (lower == asc) ? min(x, y) : max(x, y);
      }
    }
    // threads holding entries; full warps among them
    const int full = min(kSfThreads, small ? n : (n + 3) / 4) / 32;
    const int kw = full > 0 ? (a.k + full - 1) / full : 33;
    const uint32_t vw = (kw > 32) ? 0u : (warp < full ? __shfl_sync(0xffffffffu, x, 32 - kw) : 0xffffffffu);
    const uint32_t mw = __shfl_sync(0xffffffffu, x, 31);
    if (lane == 0) {
      sh.wv[warp] = vw;
      sh.wmax[warp] = mw;
    }
    __syncthreads();  // also publishes the page-table stage, the cleared histograms and info
    v = sh.wv[lane];
    M = sh.wmax[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
      M = max(M, __shfl_xor_sync(0xffffffffu, M, o));
    }
    v = max(v, 1u);
  }
  // Candidates are the entries whose key + 1 is >= v.  With v above NaN's
  // level that is x >= vf for the float vf of key v - 1 (NaN compares false,
  // -0 >= +0); otherwise every entry of the row is a candidate.
  const bool every = v <= 1u;
  float vf;
  {
    const uint32_t kv = v - 1u;  // keys below that of -inf are NaN patterns: threshold -inf
    vf = kv <= 0x007fffffu ? -__int_as_float(0x7f800000)
                           : __uint_as_float((kv & 0x80000000u) ? (kv & 0x7fffffffu) : ~kv);
  }

  // ---- 2. candidates into per-warp lists (count, warp scan, write), and
  // their first histogram: bins of (key - v) >> sbin0, sbin0 chosen so that
  // the candidates' range M - v fits 2048 bins ------------------------------
  const uint32_t R0 = M - v;
  const int sbin0 = R0 < (uint32_t)kSfBins ? 0 : (32 - __clz(R0) - 11);
  uint32_t* lkey = sh.lkey + warp * kSfWarpCap;
  uint16_t* lidx = sh.lidx + warp * kSfWarpCap;
  {
    // bit 4j + c: entry (j, c) is a candidate (independent compares, no
    // branches); set bits are then walked, each candidate's score read again
    // from L2 (registers cannot be indexed by a runtime bit number)
    uint32_t cm = 0u;
    if (!every) {
      // one compare per run of 4 (its maximum; NaN never passes), the 4
      // compares only for the few runs that hold a candidate
#pragma unroll
      for (int j = 0; j < kSfRuns; ++j) {
        if (fmaxf(fmaxf(xs[j][0], xs[j][1]), fmaxf(xs[j][2], xs[j][3])) >= vf) {
#pragma unroll
          for (int c = 0; c < 4; ++c) cm |= (xs[j][c] >= vf ? 1u : 0u) << (4 * j + c);
        }
      }
    }
    const int cnt = __popc(cm);
    int off = (int)warp_incl_scan_u32((uint32_t)cnt) - cnt;
    const int wtot = __shfl_sync(0xffffffffu, off + cnt, 31);
    const bool fits = wtot <= kSfWarpCap;
    // two candidates per step, their loads issued together
    while (cm != 0u) {
      const int b0 = __ffs(cm) - 1;
      cm &= cm - 1u;
      const bool two = cm != 0u;
      const int b1 = two ? __ffs(cm) - 1 : b0;
      cm &= cm - 1u;
      const int i0 = index_of(b0 >> 2, b0 & 3), i1 = index_of(b1 >> 2, b1 & 3);
      const float f0 = __ldcg(row + i0), f1 = __ldcg(row + i1);
      const uint32_t x0 = order_key(f0) + 1u;
      atomicAdd(&sh.hist[0][(x0 - v) >> sbin0], 1u);
      if (fits) {
        lkey[off] = x0;
        lidx[off] = (uint16_t)i0;
      }
      ++off;
      if (two) {
        const uint32_t x1 = order_key(f1) + 1u;
        atomicAdd(&sh.hist[0][(x1 - v) >> sbin0], 1u);
        if (fits) {
          lkey[off] = x1;
          lidx[off] = (uint16_t)i1;
        }
        ++off;
      }
    }
    if (lane == 0) sh.wcnt[warp] = every ? 0xffffffffu : (uint32_t)wtot;
  }
  __syncthreads();
  const int my_cnt = (int)sh.wcnt[warp];
  const bool overflow = __any_sync(0xffffffffu, sh.wcnt[lane] > (uint32_t)kSfWarpCap);

  // Steps 3-4 over the candidates: the lists, or (a list overflowed: heavy
  // ties, or no bound) every register entry.  over(f) calls f(key + 1, index)
  // on each.
  auto core = [&](auto over) {
    // ---- 3. radix passes ----------------------------------------------------
    // Pass 1 bins every candidate by (key - v) >> sbin, sbin chosen so that
    // the range M - v fits 2048 bins; each later pass bins the keys of the
    // boundary range [lo, lo + 2^span) by their next (up to 11) bits.  When
    // the boundary range holds at most kSfList keys one warp ranks them.
    uint32_t lo = v;
    int sbin = sbin0;
    int span = 32;  // pass 1: no upper limit
    int k_rem = a.k;
    uint32_t T = 0xffffffffu;
    int need = 0;
    bool all_ties = true;  // every entry equal to T is taken
    for (int pass = 0;; ++pass) {
      uint32_t* h = sh.hist[pass & 1];
      if (pass > 0 || every) {  // pass 1's histogram was built with the lists
        over([&](uint32_t x, int) {
          if (x >= lo && (span >= 32 || ((x - lo) >> span) == 0u)) atomicAdd(&h[(x - lo) >> sbin], 1u);
        });
        __syncthreads();
      }
      sf_find_bin(sh, h, k_rem);
      const int bin = sh.info[0];
      // h is read; clear it for the pass after next (this pass's and the
      // next pass's barriers order the clearing before that pass's atomics)
      h[2 * threadIdx.x] = 0u;
      h[2 * threadIdx.x + 1] = 0u;
      if (bin < 0) {  // cannot happen: at least k keys are >= v
        if (threadIdx.x == 0) raise_fault(kFaultGrouping);
        break;
      }
      k_rem -= sh.info[1];
      const int cnt = sh.info[2];
      lo += (uint32_t)bin << sbin;
      span = sbin;
      if (cnt == k_rem) {  // the whole bin is taken: the winners are the keys >= lo
        T = lo;
        need = k_rem;
        all_ties = true;
        break;
      }
      if (span == 0) {  // the bin is one key
        T = lo;
        need = k_rem;
        all_ties = cnt == k_rem;
        break;
      }
      if (cnt <= kSfList) {
        // gather the boundary range's keys (list counter reset at the start);
        // one warp ranks them by shuffles
        over([&](uint32_t x, int) {
          if (x >= lo && ((x - lo) >> span) == 0u) {
            const int p = atomicAdd(&sh.info[5], 1);
            if (p < kSfList) sh.list[p] = x;
          }
        });
        __syncthreads();
        if (warp == 0) {
          // two keys per lane (0 = none, below every key of the range)
          const int m = min(sh.info[5], kSfList);
          const uint32_t x0 = lane < m ? sh.list[lane] : 0u, x1 = lane + 32 < m ? sh.list[lane + 32] : 0u;
          int gt0 = 0, ge0 = 0, gt1 = 0, ge1 = 0;
#pragma unroll 8
          for (int q = 0; q < 32; ++q) {
            const uint32_t y0 = __shfl_sync(0xffffffffu, x0, q), y1 = __shfl_sync(0xffffffffu, x1, q);
            gt0 += (y0 > x0) + (y1 > x0);
            ge0 += (y0 >= x0) + (y1 >= x0);
            gt1 += (y0 > x1) + (y1 > x1);
            ge1 += (y0 >= x1) + (y1 >= x1);
          }
          // x is the k_rem-th largest of the range; ge - gt keys equal it
          if (lane < m && gt0 < k_rem && k_rem <= ge0) {
            sh.info[3] = (int)x0;
            sh.info[4] = k_rem - gt0;
            sh.info[6] = ge0 - gt0;
          }
          if (lane + 32 < m && gt1 < k_rem && k_rem <= ge1) {
            sh.info[3] = (int)x1;
            sh.info[4] = k_rem - gt1;
            sh.info[6] = ge1 - gt1;
          }
        }
        __syncthreads();
        T = (uint32_t)sh.info[3];
        need = sh.info[4];
        all_ties = sh.info[6] == need;
        break;
      }
      sbin = span > 11 ? span - 11 : 0;
    }

    // ---- 4. selected entries into the bitmap ---------------------------------
    // Entries equal to T (all of them are candidates, T >= v) are all taken
    // when their count is `need` (the usual case: the boundary key is
    // unique); otherwise the first `need` in index order, by a scan of the
    // tie words.
    over([&](uint32_t x, int i) {
      if (x > T || (x == T && all_ties)) atomicOr(&sh.bm[i >> 5], 1u << (i & 31));
      else if (x == T) atomicOr(&sh.tm[i >> 5], 1u << (i & 31));
    });
    __syncthreads();
    if (!all_ties) {
      const uint32_t w = sh.tm[threadIdx.x];
      uint32_t total;
      int before = (int)sf_block_excl_scan(sh, (uint32_t)__popc(w), total);
      uint32_t take = 0u, rest = w;
      while (rest != 0u && before < need) {
        const uint32_t bit = rest & (0u - rest);
        take |= bit;
        rest ^= bit;
        ++before;
      }
      if (take) sh.bm[threadIdx.x] |= take;
      __syncthreads();
    }
  };
  if (!overflow) {
    core([&](auto f) {
      for (int e = lane; e < my_cnt; e += 32) f(lkey[e], (int)lidx[e]);
    });
  } else {
    // rare (a warp listed more than kSfWarpCap candidates: heavy ties): the
    // entries are read again from L2 on every pass
    core([&](auto f) {
      for (int j = 0; j < (small ? 1 : kSfRuns); ++j)
        for (int c = 0; c < 4; ++c) {
          const int i = index_of(j, c);
          if (i < n) {
            const uint32_t x = order_key(__ldcg(row + i)) + 1u;
            if (x >= v) f(x, i);
          }
        }
    });
  }
  // ---- 5. ordered emission: a scan of the bitmap words' popcounts gives each
  // winner its output position; the winners' indices go to shared memory in
  // output order (the lists are no longer read), then every thread writes an
  // even, contiguous share of the outputs (a word holds 0 to about 6 winners,
  // so writing them from the word's thread left most threads idle)
  {
    uint32_t w = sh.bm[threadIdx.x];
    uint32_t total;
    int pos = (int)sf_block_excl_scan(sh, (uint32_t)__popc(w), total);
    if (total != (uint32_t)a.k && threadIdx.x == 0) raise_fault(kFaultGrouping);  // cannot happen
    uint32_t* sel = sh.lkey;
    while (w != 0u) {
      const int b = __ffs(w) - 1;
      w &= w - 1u;
      if (pos < a.k) sel[pos] = 32u * threadIdx.x + (uint32_t)b;
      ++pos;
    }
    __syncthreads();
    sf_emit_sorted<kMode>(a, r, sel, min((int)total, a.k));
  }
}

}  // namespace qsa
