// select.cuh -- exact top-k selection of FP32 score rows, fused with the
// page-table transform (token top-k) or with the QSA block expansion.
//
// SGLang GLM-5.2 blog (aihot.virxact.com), section "Kernel Optimization /
// TopK-V2", Figures 2-4: top-k is treated as a selection, not a sort; exactly
// k entries come back (runtime k up to 2048), ties are broken exactly, and the
// selected logical positions are turned into physical KV-cache slots in the
// same kernel.  Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section
// "Qwen sparse attention (QSA)": the best 512 blocks are kept and stand for
// their 4 token positions each, followed by the 0-3 pending tokens of the
// incomplete block.  vllm-sparse-mla-blackwell, "Design notes worth knowing":
// -1 marks an empty entry.
//
// Readings: ties go to the lower index; -0 == +0; NaN ranks below -inf; the
// result is returned in ascending index order with -1 only as tail padding.
//
// Design (GB300): one row is owned by a thread-block cluster of CS CTAs
// (CS = 1, 2, 4, 8).  Each CTA pulls its contiguous slice of the row into
// shared memory ONCE with a bulk asynchronous copy (TMA engine), converts it
// in place to order-preserving u32 keys and builds a histogram of the top 11
// key bits.  Cluster histograms are summed in two levels over distributed
// shared memory: CTA c adds everyone's counts for its 1/CS share of the bins
// with 16-byte remote loads, then every CTA reads the CS share totals and the
// one share that holds the k-th key -- a few hundred remote transactions per
// CTA and pass.  Two more passes (11 and 10 bits) over the on-chip keys refine
// the bin to the exact k-th key, stopping early when a bin holds exactly the
// remaining count.  Emission walks the slice in index order; warp ballots and
// warp/CTA/cluster prefix counts of keys above and equal to the threshold put
// every selected index straight at its ascending output position, equal keys
// at the boundary lowest-index first.  The page-table entries of the slice
// are staged in shared memory before the kernel waits for its input.  No
// sort, no global scratch; every wait is a hardware cluster barrier or a
// time-bounded mbarrier wait.
#pragma once
#include "common.cuh"

namespace qsa {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kHistBins = 2048;
constexpr int kMaxClusterSel = 8;    // largest cluster used for one row
constexpr int kSelPtCap = 2048;      // page-table entries staged per CTA

enum SelectMode { kModeTopk = 0, kModeQsa = 1 };

struct SelectArgs {
  const float* scores;          // [n_rows][ld]
  int64_t ld;
  int32_t n_rows;
  int32_t k;
  int32_t n_max;                // host bound of a row's candidates
  int32_t seg;                  // candidates per CTA slice (multiple of 4)
  int32_t vec_ok;               // rows are 16-byte aligned
  int32_t wait_primary;         // wait for the producing grid (PDL)
  // token top-k mode
  const int32_t* n_valid;       // [n_rows] or nullptr (all rows n_max)
  const int32_t* row_req;       // [n_rows] or nullptr (row t -> table row t)
  int32_t* out_idx;             // [n_rows][k]
  int32_t* out_slots;           // [n_rows][k] or nullptr
  // QSA mode: candidates of row t = row_len[t] / 4 blocks
  int32_t n_req;
  const int32_t* req_row_start; // [n_req+1]
  const int32_t* row_len;       // [n_rows]
  int32_t* out_pos;             // [n_rows][4k+3] or nullptr
  int32_t* out_xslots;          // [n_rows][4k+3]
  // paging
  const int32_t* page_table;    // [.][ld_pt] or nullptr
  int64_t ld_pt;
  int32_t page_size;
};

// Exclusive block-wide scan of two counters at once (kSelThreads threads).
__device__ __forceinline__ int2 block_scan2(int a, int b, int2* s_warp, int2& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = a, y = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int xa = __shfl_up_sync(0xffffffffu, x, o);
    const int ya = __shfl_up_sync(0xffffffffu, y, o);
    if (lane >= o) { x += xa; y += ya; }
  }
  if (lane == 31) s_warp[w] = make_int2(x, y);
  __syncthreads();
  if (w == 0) {
    int2 v = lane < kSelWarps ? s_warp[lane] : make_int2(0, 0);
    int ix = v.x, iy = v.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xa = __shfl_up_sync(0xffffffffu, ix, o);
      const int ya = __shfl_up_sync(0xffffffffu, iy, o);
      if (lane >= o) { ix += xa; iy += ya; }
    }
    if (lane < kSelWarps) s_warp[lane] = make_int2(ix - v.x, iy - v.y);
    if (lane == kSelWarps - 1) s_warp[kSelWarps] = make_int2(ix, iy);
  }
  __syncthreads();
  const int2 base = s_warp[w];
  total = s_warp[kSelWarps];
  __syncthreads();
  return make_int2(base.x + x - a, base.y + y - b);
}

struct SelShared {
  uint32_t hist[2][kHistBins];           // local histograms, double-buffered
  uint32_t stage[kHistBins];             // remote share rows being summed
  uint32_t red[2][kHistBins / 2];        // this CTA's reduced share (CS >= 2)
  uint32_t share_tot[2];                 // total of this CTA's share
  int32_t pt[kSelPtCap];                 // page-table entries of the slice
  int2 warp_scan[kSelWarps + 1];
  int2 cta_counts;                       // (above, equal) counts, read by peers
  int bin_info[4];                       // found bin, count above it, its count, owner
  uint64_t load_bar;                     // completion of the slice's bulk copy
};
// The row slice (u32 keys) follows the fixed part, 128-byte aligned.
constexpr size_t kSelKeysOffset = (sizeof(SelShared) + 127) & ~size_t(127);

__device__ __forceinline__ int32_t slot_lookup(const SelectArgs& a, const SelShared& sh,
                                               const int32_t* pt_row, int pt0, int pt_n,
                                               int64_t pos) {
  const int64_t page_idx = pos / a.page_size;
  const int32_t off = (int32_t)(pos - page_idx * a.page_size);
  if (page_idx >= pt0 && page_idx < pt0 + pt_n) return sh.pt[page_idx - pt0] * a.page_size + off;
  if (page_idx < a.ld_pt) return __ldg(pt_row + page_idx) * a.page_size + off;
  raise_fault(kFaultIndex);
  return -1;
}

template <int kMode>
__device__ __forceinline__ void emit_one(const SelectArgs& a, const SelShared& sh, int t,
                                         const int32_t* pt_row, int pt0, int pt_n, int64_t idx,
                                         int pos) {
  if (kMode == kModeTopk) {
    a.out_idx[(int64_t)t * a.k + pos] = (int32_t)idx;
    if (a.out_slots != nullptr)
      a.out_slots[(int64_t)t * a.k + pos] = slot_lookup(a, sh, pt_row, pt0, pt_n, idx);
  } else {
    if (a.out_idx != nullptr) a.out_idx[(int64_t)t * a.k + pos] = (int32_t)idx;
    const int64_t width = (int64_t)kBlock * a.k + (kBlock - 1);
    const int64_t p0 = kBlock * idx;  // first token of block idx (same page as p0+3)
    const int32_t base = slot_lookup(a, sh, pt_row, pt0, pt_n, p0);
    // Rows are 4k+3 entries wide, so these stores are not 16-byte aligned.
    int32_t* xs = a.out_xslots + (int64_t)t * width + kBlock * pos;
#pragma unroll
    for (int c = 0; c < kBlock; ++c) xs[c] = base < 0 ? -1 : base + c;
    if (a.out_pos != nullptr) {
      int32_t* xp = a.out_pos + (int64_t)t * width + kBlock * pos;
#pragma unroll
      for (int c = 0; c < kBlock; ++c) xp[c] = (int32_t)p0 + c;
    }
  }
}

// Tail of a row once m = min(k, n) entries are emitted: -1 padding (token
// mode) or pending tokens then -1 (QSA mode).  Run by one CTA of the cluster.
template <int kMode>
__device__ __forceinline__ void emit_tail(const SelectArgs& a, int t, const int32_t* pt_row, int m,
                                          int L) {
  if (kMode == kModeTopk) {
    for (int j = m + threadIdx.x; j < a.k; j += kSelThreads) {
      a.out_idx[(int64_t)t * a.k + j] = -1;
      if (a.out_slots != nullptr) a.out_slots[(int64_t)t * a.k + j] = -1;
    }
  } else {
    if (a.out_idx != nullptr)
      for (int j = m + threadIdx.x; j < a.k; j += kSelThreads) a.out_idx[(int64_t)t * a.k + j] = -1;
    const int width = kBlock * a.k + (kBlock - 1);
    const int nb = L / kBlock;
    const int pend = L - kBlock * nb;
    for (int j = kBlock * m + threadIdx.x; j < width; j += kSelThreads) {
      const int i = j - kBlock * m;
      int32_t pos = -1, slot = -1;
      if (i < pend) {
        pos = kBlock * nb + i;
        const int page_idx = pos / a.page_size;
        if (page_idx < a.ld_pt) {
          slot = __ldg(pt_row + page_idx) * a.page_size + (pos - page_idx * a.page_size);
        } else {
          raise_fault(kFaultIndex);
        }
      }
      a.out_xslots[(int64_t)t * width + j] = slot;
      if (a.out_pos != nullptr) a.out_pos[(int64_t)t * width + j] = pos;
    }
  }
}

// Among `nb` counts listed in DESCENDING bin order (read through get(d)),
// with `above_base` keys above the first, find the one holding the k_rem-th
// key: sh.bin_info = (its descending index, keys above it, its count).
template <typename Get>
__device__ __forceinline__ void find_bin(SelShared& sh, int nb, int above_base, int k_rem,
                                         Get get) {
  const int per = (nb + kSelThreads - 1) / kSelThreads;  // <= 4
  uint32_t c[4];
  int sum = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int d = threadIdx.x * per + j;
    c[j] = (j < per && d < nb) ? get(d) : 0u;
    sum += (int)c[j];
  }
  int2 tot;
  int above = above_base + block_scan2(sum, 0, sh.warp_scan, tot).x;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j < per && above < k_rem && k_rem <= above + (int)c[j]) {
      sh.bin_info[0] = threadIdx.x * per + j;
      sh.bin_info[1] = above;
      sh.bin_info[2] = (int)c[j];
    }
    above += (int)c[j];
  }
  __syncthreads();
}

__device__ __forceinline__ uint4 ld_dsmem_v4(uint32_t cluster_addr) {
  uint4 x;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
               : "r"(cluster_addr));
  return x;
}

template <int kMode>
__global__ void __launch_bounds__(kSelThreads)
select_kernel(SelectArgs a) {
  extern __shared__ __align__(128) unsigned char sel_smem_raw[];
  SelShared& sh = *reinterpret_cast<SelShared*>(sel_smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel_smem_raw + kSelKeysOffset);

  const uint32_t cs = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int t = blockIdx.x / cs;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // ---- row metadata and the slice's page-table entries: inputs that do
  // not come from the producing grid, so they are read before waiting ------
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
  if (n < 0 || n > a.n_max) {  // bad length: emit an empty row
    if (threadIdx.x == 0 && rank == 0) raise_fault(kFaultGrouping);
    n = 0;
    L = 0;
  }
  const int lo = (int)rank * a.seg;
  const int hi = min(n, lo + a.seg);
  const int len = max(0, hi - lo);
  // pages covering the positions of candidates [lo, hi) (QSA: 4 tokens each)
  const int64_t scale = kMode == kModeQsa ? kBlock : 1;
  int pt0 = 0, pt_n = 0;
  if (pt_row != nullptr && len > 0) {
    pt0 = (int)((scale * lo) / a.page_size);
    const int pt1 = (int)((scale * hi - 1) / a.page_size) + 1;
    int64_t np = min(pt1 - pt0, kSelPtCap);
    if (np > a.ld_pt - pt0) np = a.ld_pt - pt0;
    pt_n = np > 0 ? (int)np : 0;
    for (int i = threadIdx.x; i < pt_n; i += kSelThreads) sh.pt[i] = __ldg(pt_row + pt0 + i);
  }
  if (threadIdx.x == 0) {
    mbar_init(&sh.load_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (a.wait_primary) pdl_wait_primary();
  const float* row = a.scores + (int64_t)t * a.ld;

  if (n <= a.k) {
    // Everything is selected: index i goes to output position i.
    for (int i = lo + threadIdx.x; i < hi; i += kSelThreads)
      emit_one<kMode>(a, sh, t, pt_row, pt0, pt_n, i, i);
    if (rank == 0) emit_tail<kMode>(a, t, pt_row, n, L);
    return;  // no shared memory was shared, so CTAs may leave independently
  }

  // ---- load the slice once, convert in place, first histogram ----------
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) sh.hist[0][i] = 0;
  const int len_vec = a.vec_ok ? (len & ~3) : 0;  // bulk-copied part
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&sh.load_bar, (uint32_t)len_vec * 4u);
    for (int off = 0; off < len_vec; off += 8192)  // 32 KB pieces
      bulk_copy_g2s(keys + off, row + lo + off, (uint32_t)min(8192, len_vec - off) * 4u, &sh.load_bar);
  }
  for (int i = len_vec + threadIdx.x; i < len; i += kSelThreads) keys[i] = __float_as_uint(row[lo + i]);
  // A copy that never lands latches the fault and the row is garbage, but the
  // CTA keeps to the cluster's barrier sequence (leaving early could strand
  // its peers at a cluster barrier).
  if (!mbar_wait_bounded(&sh.load_bar, 0) && threadIdx.x == 0) raise_fault(kFaultWait);
  __syncthreads();
  const int len4 = (len + 3) & ~3;
  for (int i = 4 * threadIdx.x; i < len4; i += 4 * kSelThreads) {
    const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
    const uint4 kq = make_uint4(order_key(__uint_as_float(v.x)), order_key(__uint_as_float(v.y)),
                                order_key(__uint_as_float(v.z)), order_key(__uint_as_float(v.w)));
    *reinterpret_cast<uint4*>(keys + i) = kq;
    atomicAdd(&sh.hist[0][kq.x >> 21], 1u);
    if (i + 1 < len) atomicAdd(&sh.hist[0][kq.y >> 21], 1u);
    if (i + 2 < len) atomicAdd(&sh.hist[0][kq.z >> 21], 1u);
    if (i + 3 < len) atomicAdd(&sh.hist[0][kq.w >> 21], 1u);
  }

  // ---- radix refinement: 11 + 11 + 10 bits -------------------------------
  uint32_t prefix = 0;
  int shift = 32;
  int k_rem = a.k;
  for (int pass = 0; pass < 3; ++pass) {
    const int bits = pass < 2 ? 11 : 10;
    const int nbins = 1 << bits;
    const int nshift = shift - bits;
    uint32_t* hist = sh.hist[pass & 1];
    if (pass > 0) {
      for (int i = threadIdx.x; i < nbins; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      const uint32_t mask = (uint32_t)nbins - 1u;
      for (int i = 4 * threadIdx.x; i < len4; i += 4 * kSelThreads) {
        const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
        const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i + e < len && (kk[e] >> shift) == prefix) atomicAdd(&hist[(kk[e] >> nshift) & mask], 1u);
      }
    }
    int bin;
    if (cs == 1) {
      __syncthreads();
      find_bin(sh, nbins, 0, k_rem, [&](int d) { return hist[nbins - 1 - d]; });
      bin = nbins - 1 - sh.bin_info[0];
    } else {
      // Level 1: CTA `rank` sums every CTA's counts for its share of the
      // bins -- descending positions [rank*S, rank*S + S), i.e. bins
      // [nbins - (rank+1)*S, nbins - rank*S) -- with 16-byte remote loads.
      const int S = nbins / (int)cs;
      const int q4 = S / 4;
      const int share_lo = nbins - ((int)rank + 1) * S;
      uint32_t* red = sh.red[pass & 1];
      cluster_sync();  // every local histogram of this pass is final
      for (int i = threadIdx.x; i < q4 * (int)cs; i += kSelThreads) {
        const int p = i / q4, v = i - p * q4;
        const uint4 x = ld_dsmem_v4(map_shared_rank(&hist[share_lo + 4 * v], (uint32_t)p));
        *reinterpret_cast<uint4*>(&sh.stage[p * S + 4 * v]) = x;
      }
      __syncthreads();
      int part = 0;
      for (int b = threadIdx.x; b < S; b += kSelThreads) {
        uint32_t v = 0;
        for (int p = 0; p < (int)cs; ++p) v += sh.stage[p * S + b];
        red[b] = v;
        part += (int)v;
      }
      int2 tot;
      block_scan2(part, 0, sh.warp_scan, tot);
      if (threadIdx.x == 0) sh.share_tot[pass & 1] = (uint32_t)tot.x;
      cluster_sync();  // every share is reduced
      // Level 2: the share holding the k_rem-th key (shares in descending
      // order belong to ranks 0, 1, ...), then the bin inside it.
      if (warp == 0) {
        uint32_t st = 0;
        if (lane < (int)cs) st = ld_dsmem_u32(map_shared_rank(&sh.share_tot[pass & 1], (uint32_t)lane));
        int incl = (int)st;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int excl = incl - (int)st;
        if (lane < (int)cs && excl < k_rem && k_rem <= incl) {
          sh.bin_info[3] = lane;
          sh.bin_info[1] = excl;
        }
      }
      __syncthreads();
      const int owner = sh.bin_info[3];
      const int above_share = sh.bin_info[1];
      for (int v = threadIdx.x; v < q4; v += kSelThreads)
        *reinterpret_cast<uint4*>(&sh.stage[4 * v]) = ld_dsmem_v4(map_shared_rank(&red[4 * v], (uint32_t)owner));
      __syncthreads();
      const int owner_lo = nbins - (owner + 1) * S;
      find_bin(sh, S, above_share, k_rem, [&](int d) { return sh.stage[S - 1 - d]; });
      bin = owner_lo + (S - 1 - sh.bin_info[0]);
    }
    k_rem -= sh.bin_info[1];
    const int bin_count = sh.bin_info[2];
    prefix = pass == 0 ? (uint32_t)bin : ((prefix << bits) | (uint32_t)bin);
    shift = nshift;
    __syncthreads();
    if (bin_count == k_rem) break;  // the whole bin is selected
  }
  const int need = k_rem;  // keys equal to the threshold prefix to take

  // ---- emission in ascending index order --------------------------------
  // Each warp owns a contiguous piece of the slice, walked in chunks of 128
  // (4 consecutive keys per lane).
  const int piece = (((len + kSelWarps - 1) / kSelWarps) + 127) & ~127;
  const int w_lo = min(len, warp * piece);
  const int w_hi = min(len, w_lo + piece);
  int gt = 0, eq = 0;
  for (int i = w_lo + 4 * lane; i < w_hi; i += 128) {
    const uint4 v = *reinterpret_cast<const uint4*>(keys + i);
    const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (i + e < w_hi) {
        const uint32_t hb = kk[e] >> shift;
        gt += hb > prefix;
        eq += hb == prefix;
      }
    }
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  // Warp bases inside the CTA (only lane 0's counts enter the scan).
  int2 cta_tot;
  int2 wbase = block_scan2(lane == 0 ? gt : 0, lane == 0 ? eq : 0, sh.warp_scan, cta_tot);
  wbase.x = __shfl_sync(0xffffffffu, wbase.x, 0);
  wbase.y = __shfl_sync(0xffffffffu, wbase.y, 0);
  // CTA bases inside the cluster.
  int cta_gt = 0, cta_eq = 0;
  if (cs > 1) {
    if (threadIdx.x == 0) sh.cta_counts = cta_tot;
    cluster_sync();
    if (warp == 0) {
      int cx = 0, cy = 0;
      if (lane < (int)rank) {
        const uint32_t addr = map_shared_rank(&sh.cta_counts, (uint32_t)lane);
        cx = (int)ld_dsmem_u32(addr);
        cy = (int)ld_dsmem_u32(addr + 4);
      }
      cx = __reduce_add_sync(0xffffffffu, cx);
      cy = __reduce_add_sync(0xffffffffu, cy);
      if (lane == 0) {
        sh.bin_info[0] = cx;
        sh.bin_info[1] = cy;
      }
    }
    __syncthreads();
    cta_gt = sh.bin_info[0];
    cta_eq = sh.bin_info[1];
  }
  const unsigned lt_mask = (1u << lane) - 1u;
  int run_gt = cta_gt + wbase.x;  // keys above the threshold before this chunk
  int run_eq = cta_eq + wbase.y;  // keys equal to it before this chunk
  for (int c0 = w_lo; c0 < w_hi; c0 += 128) {
    const int i0 = c0 + 4 * lane;
    uint4 kq = make_uint4(0u, 0u, 0u, 0u);
    if (i0 < w_hi) kq = *reinterpret_cast<const uint4*>(keys + i0);
    const uint32_t kk[4] = {kq.x, kq.y, kq.z, kq.w};
    bool f_gt[4], f_eq[4];
    unsigned b_gt[4], b_eq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t hb = kk[e] >> shift;
      const bool in = i0 + e < w_hi;
      f_gt[e] = in && hb > prefix;
      f_eq[e] = in && hb == prefix;
      b_gt[e] = __ballot_sync(0xffffffffu, f_gt[e]);
      b_eq[e] = __ballot_sync(0xffffffffu, f_eq[e]);
    }
    if ((b_gt[0] | b_gt[1] | b_gt[2] | b_gt[3] | b_eq[0] | b_eq[1] | b_eq[2] | b_eq[3]) == 0u)
      continue;  // nothing selected in this chunk (warp-uniform)
    int eq_rank = run_eq;  // keys equal to the threshold before this lane's first key
    int n_gt = 0, n_eq = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      eq_rank += __popc(b_eq[e] & lt_mask);
      n_gt += __popc(b_gt[e]);
      n_eq += __popc(b_eq[e]);
    }
    bool sel[4];
    unsigned b_sel[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sel[e] = f_gt[e] || (f_eq[e] && eq_rank < need);
      eq_rank += f_eq[e];
      b_sel[e] = __ballot_sync(0xffffffffu, sel[e]);
    }
    int out = run_gt + min(run_eq, need);
#pragma unroll
    for (int e = 0; e < 4; ++e) out += __popc(b_sel[e] & lt_mask);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (sel[e]) emit_one<kMode>(a, sh, t, pt_row, pt0, pt_n, (int64_t)lo + i0 + e, out++);
    run_gt += n_gt;
    run_eq += n_eq;
  }
  if (rank == 0) emit_tail<kMode>(a, t, pt_row, a.k, L);
  if (cs > 1) cluster_sync();  // peers may still read this CTA's shared memory
}

}  // namespace qsa
