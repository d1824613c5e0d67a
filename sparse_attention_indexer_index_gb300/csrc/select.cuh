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
// (CS = 1, 2, 4, 8, 16).  Each CTA reads its contiguous slice of the row from
// global memory ONCE, converts it to order-preserving u32 keys in shared
// memory and builds a histogram of the top 11 key bits.  The CTAs add their
// histograms over distributed shared memory, every CTA finds the same
// threshold bin, and two more passes (11 and 10 bits) over the on-chip keys
// refine it to the exact k-th key, stopping early when the bin holds exactly
// the remaining count.  Emission walks the slice in index order: counts of
// keys above / equal to the threshold are prefix-summed over warps, CTAs
// and the cluster, so every selected index lands directly at its ascending
// output position and equal keys at the boundary are taken lowest-index
// first.  No sort, no global scratch, no spin-waits (cluster barriers only).
#pragma once
#include "common.cuh"

namespace qsa {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kHistBins = 2048;

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

// Warp exclusive scan of one counter; also returns the warp total.
__device__ __forceinline__ int warp_excl_scan(int v, int& total) {
  const int lane = threadIdx.x & 31;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

struct SelShared {
  uint32_t hist[2][kHistBins];  // double-buffered (peers read the other one)
  int2 warp_scan[kSelWarps + 1];
  int2 cta_counts;              // this CTA's (above, equal) counts, read by peers
  int bin_info[4];              // found bin, count above it, its count
};

template <int kMode>
__device__ __forceinline__ void emit_one(const SelectArgs& a, int t, int req, int64_t idx, int pos) {
  if (kMode == kModeTopk) {
    a.out_idx[(int64_t)t * a.k + pos] = (int32_t)idx;
    if (a.out_slots != nullptr) {
      const int tr = a.row_req ? __ldg(a.row_req + t) : t;
      const int64_t page_idx = idx / a.page_size;
      int32_t slot = -1;
      if (page_idx < a.ld_pt && tr >= 0) {
        slot = __ldg(a.page_table + (int64_t)tr * a.ld_pt + page_idx) * a.page_size +
               (int32_t)(idx - page_idx * a.page_size);
      } else {
        raise_fault(kFaultIndex);
      }
      a.out_slots[(int64_t)t * a.k + pos] = slot;
    }
  } else {
    if (a.out_idx != nullptr) a.out_idx[(int64_t)t * a.k + pos] = (int32_t)idx;
    const int64_t width = (int64_t)kBlock * a.k + (kBlock - 1);
    const int64_t p0 = kBlock * idx;  // first token of block idx
    const int64_t page_idx = p0 / a.page_size;
    int32_t base = -1;
    if (page_idx < a.ld_pt) {
      base = __ldg(a.page_table + (int64_t)req * a.ld_pt + page_idx) * a.page_size +
             (int32_t)(p0 - page_idx * a.page_size);
    } else {
      raise_fault(kFaultIndex);
    }
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
__device__ __forceinline__ void emit_tail(const SelectArgs& a, int t, int req, int m, int L) {
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
          slot = __ldg(a.page_table + (int64_t)req * a.ld_pt + page_idx) * a.page_size +
                 (pos - page_idx * a.page_size);
        } else {
          raise_fault(kFaultIndex);
        }
      }
      a.out_xslots[(int64_t)t * width + j] = slot;
      if (a.out_pos != nullptr) a.out_pos[(int64_t)t * width + j] = pos;
    }
  }
}

template <int kMode>
__global__ void __launch_bounds__(kSelThreads)
select_kernel(SelectArgs a) {
  extern __shared__ __align__(16) unsigned char sel_smem_raw[];
  SelShared& sh = *reinterpret_cast<SelShared*>(sel_smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(sel_smem_raw + sizeof(SelShared));

  const uint32_t cs = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int t = blockIdx.x / cs;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  if (a.wait_primary) pdl_wait_primary();

  // Candidates of this row.
  int n, req = 0, L = 0;
  if (kMode == kModeTopk) {
    n = a.n_valid ? __ldg(a.n_valid + t) : a.n_max;
  } else {
    req = row_request(a.req_row_start, a.n_req, t);
    L = __ldg(a.row_len + t);
    n = L / kBlock;
  }
  if (n < 0 || n > a.n_max) {  // bad length: emit an empty row
    if (threadIdx.x == 0 && rank == 0) raise_fault(kFaultGrouping);
    n = 0;
    L = 0;
  }
  const int lo = (int)rank * a.seg;
  const int hi = min(n, lo + a.seg);
  const int len = max(0, hi - lo);
  const float* row = a.scores + (int64_t)t * a.ld;

  if (n <= a.k) {
    // Everything is selected: index i goes to output position i.
    for (int i = lo + threadIdx.x; i < hi; i += kSelThreads) emit_one<kMode>(a, t, req, i, i);
    if (rank == 0) emit_tail<kMode>(a, t, req, n, L);
    return;  // no shared memory was shared, so CTAs may leave independently
  }

  // ---- load the slice once, build the first histogram (top 11 bits) -----
  for (int i = threadIdx.x; i < kHistBins; i += kSelThreads) sh.hist[0][i] = 0;
  __syncthreads();
  if (a.vec_ok) {
    const int len4 = (len + 3) & ~3;
    for (int i = 4 * threadIdx.x; i < len4; i += 4 * kSelThreads) {
      float4 v;
      if (i + 3 < len) {
        v = __ldg(reinterpret_cast<const float4*>(row + lo + i));
      } else {
        v.x = row[lo + i];
        v.y = i + 1 < len ? row[lo + i + 1] : 0.f;
        v.z = i + 2 < len ? row[lo + i + 2] : 0.f;
        v.w = i + 3 < len ? row[lo + i + 3] : 0.f;
      }
      uint4 kq = make_uint4(order_key(v.x), order_key(v.y), order_key(v.z), order_key(v.w));
      *reinterpret_cast<uint4*>(keys + i) = kq;
      atomicAdd(&sh.hist[0][kq.x >> 21], 1u);
      if (i + 1 < len) atomicAdd(&sh.hist[0][kq.y >> 21], 1u);
      if (i + 2 < len) atomicAdd(&sh.hist[0][kq.z >> 21], 1u);
      if (i + 3 < len) atomicAdd(&sh.hist[0][kq.w >> 21], 1u);
    }
  } else {
    for (int i = threadIdx.x; i < len; i += kSelThreads) {
      const uint32_t kq = order_key(row[lo + i]);
      keys[i] = kq;
      atomicAdd(&sh.hist[0][kq >> 21], 1u);
    }
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
      for (int i = threadIdx.x; i < len; i += kSelThreads) {
        const uint32_t kq = keys[i];
        if ((kq >> shift) == prefix) atomicAdd(&hist[(kq >> nshift) & mask], 1u);
      }
    }
    // Sum the cluster's histograms; thread tid owns descending bins
    // [tid*per, tid*per + per) counted from the top.
    if (cs > 1) cluster_sync(); else __syncthreads();
    const int per = nbins / kSelThreads;  // 4 or 2
    uint32_t c[4] = {0u, 0u, 0u, 0u};
    int sum = 0;
    for (int j = 0; j < per; ++j) {
      const int bin = nbins - 1 - (threadIdx.x * per + j);
      uint32_t v = hist[bin];
      for (uint32_t p = 1; p < cs; ++p) v += ld_dsmem_u32(map_shared_rank(&hist[bin], (rank + p) % cs));
      c[j] = v;
      sum += (int)v;
    }
    int2 tot;
    const int above0 = block_scan2(sum, 0, sh.warp_scan, tot).x;
    int above = above0;
    for (int j = 0; j < per; ++j) {
      if (above < k_rem && k_rem <= above + (int)c[j]) {
        sh.bin_info[0] = nbins - 1 - (threadIdx.x * per + j);
        sh.bin_info[1] = above;
        sh.bin_info[2] = (int)c[j];
      }
      above += (int)c[j];
    }
    __syncthreads();
    const uint32_t bin = (uint32_t)sh.bin_info[0];
    k_rem -= sh.bin_info[1];
    const int bin_count = sh.bin_info[2];
    prefix = pass == 0 ? bin : ((prefix << bits) | bin);
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
  for (int i = w_lo + lane; i < w_hi; i += 32) {
    const uint32_t hb = keys[i] >> shift;
    gt += hb > prefix;
    eq += hb == prefix;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
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
    for (uint32_t p = 0; p < rank; ++p) {
      const uint32_t addr = map_shared_rank(&sh.cta_counts, p);
      cta_gt += (int)ld_dsmem_u32(addr);
      cta_eq += (int)ld_dsmem_u32(addr + 4);
    }
  }
  int run_gt = cta_gt + wbase.x;  // keys above the threshold before this point
  int run_eq = cta_eq + wbase.y;  // keys equal to it before this point
  for (int c0 = w_lo; c0 < w_hi; c0 += 128) {
    const int i0 = c0 + 4 * lane;
    uint4 kq = make_uint4(0u, 0u, 0u, 0u);
    if (i0 < w_hi) kq = *reinterpret_cast<const uint4*>(keys + i0);
    const uint32_t kk[4] = {kq.x, kq.y, kq.z, kq.w};
    int f_gt = 0, f_eq = 0;  // bit masks over this lane's 4 keys
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (i0 + e < w_hi) {
        const uint32_t hb = kk[e] >> shift;
        f_gt |= (hb > prefix) << e;
        f_eq |= (hb == prefix) << e;
      }
    }
    int eq_tot;
    const int eq_before = run_eq + warp_excl_scan(__popc(f_eq), eq_tot);
    // Equal keys of this lane with rank < need are taken.
    int take = 0, r = eq_before;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if ((f_eq >> e) & 1) {
        if (r < need) take |= 1 << e;
        ++r;
      }
    }
    const int sel = f_gt | take;
    int sel_tot;
    int out = run_gt + min(run_eq, need) + warp_excl_scan(__popc(sel), sel_tot);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if ((sel >> e) & 1) emit_one<kMode>(a, t, req, (int64_t)lo + i0 + e, out++);
    }
    int gt_tot;
    warp_excl_scan(__popc(f_gt), gt_tot);
    run_gt += gt_tot;
    run_eq += eq_tot;
  }
  if (rank == 0) emit_tail<kMode>(a, t, req, a.k, L);
  if (cs > 1) cluster_sync();  // peers may still read this CTA's shared memory
}

}  // namespace qsa
