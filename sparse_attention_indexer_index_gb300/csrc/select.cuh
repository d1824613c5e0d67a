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
// Design (GB300): one 1024-thread CTA per row; every step synchronises with
// CTA barriers only, and as few as possible (a 1024-thread barrier plus its
// scan costs about half a microsecond).  Scores become order-preserving u32
// keys (larger float -> larger key).
//  1. Histogram of the top 11 key bits over the whole row (four copies to
//     spread atomic contention); a two-barrier scan finds the bin B0 holding
//     the k-th largest key.
//  2. Order-preserving compaction of every entry whose top bits are >= B0 --
//     the sure winners plus the boundary bin, typically k plus a few percent
//     of the row -- into a shared-memory list: each warp owns a contiguous
//     segment, counts, and after one barrier writes its matches with ballot
//     prefix counts.
//  3. Two radix passes (11 and 10 bits) over the boundary entries of the list
//     give the exact k-th key T (early exit when a bin holds exactly the
//     remaining count).
//  4. Emission over the list, segmented the same way: above T, or equal to T
//     among the first `need` equal ones, goes straight to its ascending
//     output position, with the slot translation (or the QSA expansion to 4
//     positions and slots) in the same step.
// A row of up to 32K scores is pulled once into shared memory by bulk
// asynchronous copies (TMA engine; one barrier per 16 KB piece, so the
// conversion overlaps the transfer).  A longer row streams through a 4-stage
// ring for step 1 and again for step 2.  If the list would overflow (heavy
// ties), steps 3-4 run over the whole row instead.  No sort, no global
// scratch, no cluster; every wait is a CTA barrier or a time-bounded mbarrier
// wait.
#pragma once
#include <cstddef>

#include "common.cuh"

namespace qsa {

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kHistBins = 2048;
constexpr int kHistCopies = 4;
constexpr int kSelPiece = 4096;          // elements per bulk piece (16 KB)
constexpr int kSelRing = 4;              // ring stages for streamed rows
constexpr int kSelResidentCap = 32768;   // longest row kept in shared memory
constexpr int kSelMaxBars = 8;           // >= kSelResidentCap / kSelPiece and kSelRing
constexpr int kSelSampleMin = 4096;      // shorter rows take the exact histogram directly

enum SelectMode { kModeTopk = 0, kModeQsa = 1 };

struct SelectArgs {
  const float* scores;          // [n_rows][ld]
  int64_t ld;
  int32_t n_rows;
  int32_t k;
  int32_t n_max;                // host bound of a row's candidates
  int32_t vec_ok;               // rows are 16-byte aligned
  int32_t wait_primary;         // wait for the producing grid (PDL)
  int32_t resident;             // 1: rows fit in shared memory (n_max <= kSelResidentCap); 2: select_resident_kernel
  int32_t list_cap;             // entries of the candidate list
  int32_t pt_cap;               // page-table entries staged in shared memory
  int32_t off_pt, off_list, off_lkey, off_row, off_sel;  // dynamic shared memory layout (bytes)
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
  // Row plan (rows split by length class on the device by plan_rows_kernel):
  // nullptr, or plan[0] = long rows, plan[1] = CTAs per long row, plan[2] =
  // short rows, then the long and the short row lists.  Unit u of a planned
  // launch (a CTA, or a cluster) serves row_list[u] for u < plan[count_at];
  // a launch standing for one cluster size (plan_c != 0) works only when the
  // plan chose that size.
  const int32_t* plan;
  const int32_t* row_list;
  int32_t count_at;
  int32_t plan_c;
};

// The row served by unit u (CTA or cluster) of this launch; false: none.
// A planned launch first waits for the planning grid (the previous one on the
// stream), then reads the plan.
__device__ __forceinline__ bool sel_unit_row(const SelectArgs& a, int u, int& t) {
  if (a.plan == nullptr) {
    t = u;
    return true;
  }
  pdl_wait_primary();
  if (a.plan_c != 0 && __ldcg(a.plan + 1) != a.plan_c) return false;
  if (u >= __ldcg(a.plan + a.count_at)) return false;
  t = __ldcg(a.row_list + u);
  return t >= 0 && t < a.n_rows;
}

// ---------------------------------------------------------------------------
// Row plan (SGLang GLM-5.2 blog, "Kernel Optimization / TopK-V2": a planning
// kernel reads the batch's sequence lengths and builds the work lists, so
// that long rows get a cluster of CTAs and short ones a single CTA).  One
// 1024-thread CTA: rows with more than `cut` candidates go to the long list,
// the others to the short list, both in row order; the long list's CTAs per
// row is the largest C allowed by c_mask (schedulable sizes among 16 and 2)
// with n_long * C <= SMs, else 1.
// ---------------------------------------------------------------------------
struct PlanArgs {
  const int32_t* n_valid;  // token mode: candidates per row (nullptr: n_max)
  const int32_t* row_len;  // QSA mode: visible tokens per row (candidates row_len / 4)
  int32_t n_rows;
  int32_t n_max;
  int32_t cut;
  int32_t c_mask;          // bit e set: the plan may pick clusters of 2^e CTAs (e = 1..4)
  int32_t sm_count;
  int32_t* plan;           // [4 + 2 * n_rows]
};

__global__ void __launch_bounds__(1024) plan_rows_kernel(PlanArgs p) {
  __shared__ int s_cnt[2][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the plan may still be read by the previous call's selection
  pdl_wait_primary();
  int n_long = 0, n_short = 0;
  for (int base = 0; base < p.n_rows; base += 1024) {
    const int t = base + tid;
    int n = 0;
    if (t < p.n_rows) n = p.row_len ? __ldg(p.row_len + t) / kBlock : (p.n_valid ? __ldg(p.n_valid + t) : p.n_max);
    const bool is_long = t < p.n_rows && n > p.cut, is_short = t < p.n_rows && !is_long;
    const unsigned bl = __ballot_sync(0xffffffffu, is_long), bs = __ballot_sync(0xffffffffu, is_short);
    if (lane == 0) {
      s_cnt[0][warp] = __popc(bl);
      s_cnt[1][warp] = __popc(bs);
    }
    __syncthreads();
    int ol = 0, os = 0, tl = 0, ts = 0;
    for (int w = 0; w < 32; ++w) {
      if (w < warp) {
        ol += s_cnt[0][w];
        os += s_cnt[1][w];
      }
      tl += s_cnt[0][w];
      ts += s_cnt[1][w];
    }
    const unsigned lt = (1u << lane) - 1u;
    if (is_long) p.plan[4 + n_long + ol + __popc(bl & lt)] = t;
    if (is_short) p.plan[4 + p.n_rows + n_short + os + __popc(bs & lt)] = t;
    n_long += tl;
    n_short += ts;
    __syncthreads();  // s_cnt is rewritten by the next chunk
  }
  if (tid == 0) {
    int c = 16;
    while (c > 1 && !((int64_t)n_long * c <= p.sm_count && (p.c_mask >> (31 - __clz(c)) & 1))) c >>= 1;
    p.plan[0] = n_long;
    p.plan[1] = c;
    p.plan[2] = n_short;
    p.plan[3] = 0;
  }
}

struct SelFixed {
  uint32_t hist[kHistCopies][kHistBins];
  int warp_tot[2][kSelWarps];   // per-warp counts (two counters)
  int info[8];
  uint64_t bar[kSelMaxBars];
};
constexpr int kSelFixedBytes = (int)((sizeof(SelFixed) + 127) & ~size_t(127));
static_assert(offsetof(SelFixed, bar) % 8 == 0, "mbarriers must be 8-byte aligned");

// Per-row context.
struct SelRow {
  int t, n, L;
  const float* row;
  const int32_t* pt_row;
  int pt_n;
  const int32_t* pt_s;  // staged page-table entries [0, pt_n)
};

__device__ __forceinline__ int32_t slot_lookup(const SelectArgs& a, const SelRow& r, int64_t pos) {
  // positions are below a row length (int32): 32-bit division, a shift and a
  // mask for page sizes that are powers of two (the usual case)
  const int32_t ps = a.page_size;
  int32_t page_idx, off;
  if ((ps & (ps - 1)) == 0) {
    page_idx = (int32_t)pos >> (31 - __clz(ps));
    off = (int32_t)pos & (ps - 1);
  } else {
    page_idx = (int32_t)pos / ps;
    off = (int32_t)pos - page_idx * ps;
  }
  if (page_idx < r.pt_n) return r.pt_s[page_idx] * a.page_size + off;
  if (page_idx < a.ld_pt) return __ldg(r.pt_row + page_idx) * a.page_size + off;
  raise_fault(kFaultIndex);
  return -1;
}

template <int kMode>
__device__ __forceinline__ void emit_one(const SelectArgs& a, const SelRow& r, int64_t idx, int pos) {
  const int t = r.t;
  if (kMode == kModeTopk) {
    a.out_idx[(int64_t)t * a.k + pos] = (int32_t)idx;
    if (a.out_slots != nullptr) a.out_slots[(int64_t)t * a.k + pos] = slot_lookup(a, r, idx);
  } else {
    if (a.out_idx != nullptr) a.out_idx[(int64_t)t * a.k + pos] = (int32_t)idx;
    const int64_t width = (int64_t)kBlock * a.k + (kBlock - 1);
    const int64_t p0 = kBlock * idx;  // first token of block idx (same page as p0+3)
    const int32_t base = slot_lookup(a, r, p0);
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
// mode) or pending tokens then -1 (QSA mode).
template <int kMode>
__device__ __forceinline__ void emit_tail(const SelectArgs& a, const SelRow& r, int m) {
  const int t = r.t;
  if (kMode == kModeTopk) {
    for (int j = m + threadIdx.x; j < a.k; j += kSelThreads) {
      a.out_idx[(int64_t)t * a.k + j] = -1;
      if (a.out_slots != nullptr) a.out_slots[(int64_t)t * a.k + j] = -1;
    }
  } else {
    if (a.out_idx != nullptr)
      for (int j = m + threadIdx.x; j < a.k; j += kSelThreads) a.out_idx[(int64_t)t * a.k + j] = -1;
    const int width = kBlock * a.k + (kBlock - 1);
    const int nb = r.L / kBlock;
    const int pend = r.L - kBlock * nb;
    for (int j = kBlock * m + threadIdx.x; j < width; j += kSelThreads) {
      const int i = j - kBlock * m;
      int32_t pos = -1, slot = -1;
      if (i < pend) {
        pos = kBlock * nb + i;
        slot = slot_lookup(a, r, pos);
      }
      a.out_xslots[(int64_t)t * width + j] = slot;
      if (a.out_pos != nullptr) a.out_pos[(int64_t)t * width + j] = pos;
    }
  }
}

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Publish per-warp totals (two counters) and return this warp's exclusive
// prefixes over the CTA; one barrier.  `tot` receives the CTA totals.
__device__ __forceinline__ int2 warp_bases(SelFixed& fx, int buf, int g, int q, int2& tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    fx.warp_tot[0][warp] = g;
    fx.warp_tot[1][warp] = q;
  }
  (void)buf;
  __syncthreads();
  const int vg = fx.warp_tot[0][lane], vq = fx.warp_tot[1][lane];
  const int ig = warp_incl_scan(vg), iq = warp_incl_scan(vq);
  tot.x = __shfl_sync(0xffffffffu, ig, 31);
  tot.y = __shfl_sync(0xffffffffu, iq, 31);
  const int2 base = make_int2(__shfl_sync(0xffffffffu, ig - vg, warp), __shfl_sync(0xffffffffu, iq - vq, warp));
  __syncthreads();  // warp_tot may be rewritten by the next caller
  return base;
}

// Among `nb` bins (nb = 2048 or 1024) of the histogram copies 0..ncopies-1,
// listed from the top bin down, with `above_base` keys above the first, find
// the bin holding the k_rem-th key: info[0..2] = (bin, keys above it, count).
__device__ __forceinline__ void find_bin(SelFixed& fx, int nb, int ncopies, int above_base, int k_rem) {
  const int per = nb / kSelThreads;  // 2 or 1
  uint32_t c[2] = {0u, 0u};
  int sum = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (j < per) {
      const int bin = nb - 1 - (threadIdx.x * per + j);
      uint32_t v = 0;
      for (int cp = 0; cp < ncopies; ++cp) v += fx.hist[cp][bin];
      c[j] = v;
      sum += (int)v;
    }
  }
  const int lane = threadIdx.x & 31;
  const int incl = warp_incl_scan(sum);
  int2 tot;
  const int2 wb = warp_bases(fx, 0, __shfl_sync(0xffffffffu, incl, 31), 0, tot);
  int above = above_base + wb.x + incl - sum;
  (void)lane;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    if (j < per && above < k_rem && k_rem <= above + (int)c[j]) {
      fx.info[0] = nb - 1 - (threadIdx.x * per + j);
      fx.info[1] = above;
      fx.info[2] = (int)c[j];
    }
    above += (int)c[j];
  }
  __syncthreads();
}

// Ordered compaction / emission over a segment-per-warp layout.  The items
// are [0, cnt); warp w owns [w*seg, (w+1)*seg) (seg a multiple of 128) and
// walks it 128 at a time, 4 consecutive items per lane.
__device__ __forceinline__ int warp_segment(int cnt) {
  return (((cnt + kSelWarps - 1) / kSelWarps) + 127) & ~127;
}

// Streams a long row through the ring: f(keys accessor for the piece, base,
// count) on every piece in order.  The piece's bulk part is read from shared
// memory as uint4; the (< 4) tail and rows that are not 16-byte aligned are
// read from global memory.
struct RowStream {
  int n;
  const float* row;
  int vec_ok;
  uint64_t* bar;
  float* ring;   // kSelRing * kSelPiece floats
  int seq;

  __device__ __forceinline__ void issue(int piece) {
    const int s = (seq + piece) % kSelRing;
    const int base = piece * kSelPiece;
    const int cnt = min(kSelPiece, n - base);
    const int bulk = vec_ok ? (cnt & ~3) : 0;
    mbar_arrive_expect_tx(&bar[s], (uint32_t)bulk * 4u);
    if (bulk > 0) bulk_copy_g2s(ring + (size_t)s * kSelPiece, row + base, (uint32_t)bulk * 4u, &bar[s]);
  }

  // f(const float* piece_smem, int bulk, const float* piece_global, int base, int cnt)
  template <typename F>
  __device__ __forceinline__ void walk(F f) {
    const int np = (n + kSelPiece - 1) / kSelPiece;
    if (threadIdx.x == 0)
      for (int p = 0; p < min(np, kSelRing); ++p) issue(p);
    for (int p = 0; p < np; ++p) {
      const int s = (seq + p) % kSelRing;
      const uint32_t parity = (uint32_t)((seq + p) / kSelRing) & 1u;
      if (!mbar_wait_bounded(&bar[s], parity) && threadIdx.x == 0) raise_fault(kFaultWait);
      const int base = p * kSelPiece;
      const int cnt = min(kSelPiece, n - base);
      f(ring + (size_t)s * kSelPiece, vec_ok ? (cnt & ~3) : 0, row + base, base, cnt);
      __syncthreads();  // the stage is free again
      if (threadIdx.x == 0 && p + kSelRing < np) issue(p + kSelRing);
    }
    seq += np;
  }
};

// Four keys of items [i, i+4) of a piece: from shared memory (bulk part, as
// floats to convert or as keys) or from global memory.
__device__ __forceinline__ void load4_keys(const float* sm, int bulk, const float* gl, int i, int cnt,
                                           bool already_keys, uint32_t (&kk)[4]) {
  if (i + 3 < bulk) {
    const uint4 v = *reinterpret_cast<const uint4*>(sm + i);
    if (already_keys) {
      kk[0] = v.x; kk[1] = v.y; kk[2] = v.z; kk[3] = v.w;
    } else {
      kk[0] = order_key(__uint_as_float(v.x));
      kk[1] = order_key(__uint_as_float(v.y));
      kk[2] = order_key(__uint_as_float(v.z));
      kk[3] = order_key(__uint_as_float(v.w));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t x = 0u;
      if (i + e < cnt) {
        if (i + e < bulk) x = already_keys ? __float_as_uint(sm[i + e]) : order_key(sm[i + e]);
        else x = order_key(__ldg(gl + i + e));
      }
      kk[e] = x;
    }
  }
}

template <int kMode>
__global__ void __launch_bounds__(kSelThreads, 1)
select_kernel(SelectArgs a) {
  extern __shared__ __align__(128) unsigned char sel_smem_raw[];
  SelFixed& fx = *reinterpret_cast<SelFixed*>(sel_smem_raw);
  int32_t* pt_s = reinterpret_cast<int32_t*>(sel_smem_raw + a.off_pt);
  int32_t* list_idx = reinterpret_cast<int32_t*>(sel_smem_raw + a.off_list);
  uint32_t* list_key = reinterpret_cast<uint32_t*>(sel_smem_raw + a.off_lkey);
  float* row_area = reinterpret_cast<float*>(sel_smem_raw + a.off_row);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;

  SelRow r;
  if (!sel_unit_row(a, blockIdx.x, r.t)) return;
  r.L = 0;
  r.pt_row = nullptr;
  r.pt_s = pt_s;
  r.pt_n = 0;
  // ---- row metadata and the row's page-table entries: inputs that do not
  // come from the producing grid, so they are read before waiting ---------
  if (kMode == kModeTopk) {
    r.n = a.n_valid ? __ldg(a.n_valid + r.t) : a.n_max;
    if (a.out_slots != nullptr)
      r.pt_row = a.page_table + (int64_t)(a.row_req ? __ldg(a.row_req + r.t) : r.t) * a.ld_pt;
  } else {
    const int req = row_request(a.req_row_start, a.n_req, r.t);
    r.L = __ldg(a.row_len + r.t);
    r.n = r.L / kBlock;
    r.pt_row = a.page_table + (int64_t)req * a.ld_pt;
  }
  if (r.n < 0 || r.n > a.n_max) {  // bad length: emit an empty row
    if (threadIdx.x == 0) raise_fault(kFaultGrouping);
    r.n = 0;
    r.L = 0;
  }
  if (r.pt_row != nullptr) {
    const int64_t last = kMode == kModeQsa ? (int64_t)r.L : (int64_t)r.n;  // positions < last
    int64_t np = last > 0 ? (last - 1) / a.page_size + 1 : 0;
    if (np > a.pt_cap) np = a.pt_cap;
    if (np > a.ld_pt) np = a.ld_pt;
    r.pt_n = (int)np;
    for (int i = threadIdx.x; i < r.pt_n; i += kSelThreads) pt_s[i] = __ldg(r.pt_row + i);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSelMaxBars; ++i) mbar_init(&fx.bar[i], 1);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < kHistCopies * kHistBins; i += kSelThreads) (&fx.hist[0][0])[i] = 0;
  __syncthreads();

  if (a.wait_primary) pdl_wait_primary();
  r.row = a.scores + (int64_t)r.t * a.ld;
  const int n = r.n;

  if (n <= a.k) {
    // Everything is selected: index i goes to output position i.
    for (int i = threadIdx.x; i < n; i += kSelThreads) emit_one<kMode>(a, r, i, i);
    emit_tail<kMode>(a, r, n);
    return;
  }

  // ---- 0. load: resident rows are pulled into shared memory as keys -----
  uint32_t* hcopy = fx.hist[warp & (kHistCopies - 1)];
  RowStream rs{n, r.row, a.vec_ok, fx.bar, row_area, 0};
  if (a.resident) {
    // Bulk-load the whole row (one barrier per 16 KB piece), convert in place.
    const int np = (n + kSelPiece - 1) / kSelPiece;
    if (threadIdx.x == 0) {
      for (int p = 0; p < np; ++p) {
        const int base = p * kSelPiece;
        const int bulk = a.vec_ok ? (min(kSelPiece, n - base) & ~3) : 0;
        mbar_arrive_expect_tx(&fx.bar[p], (uint32_t)bulk * 4u);
        if (bulk > 0) bulk_copy_g2s(row_area + base, r.row + base, (uint32_t)bulk * 4u, &fx.bar[p]);
      }
    }
    for (int p = 0; p < np; ++p) {
      const int base = p * kSelPiece;
      const int cnt = min(kSelPiece, n - base);
      const int bulk = a.vec_ok ? (cnt & ~3) : 0;
      if (!mbar_wait_bounded(&fx.bar[p], 0) && threadIdx.x == 0) raise_fault(kFaultWait);
      const int i = 4 * threadIdx.x;  // kSelPiece == 4 * kSelThreads
      if (i < cnt) {
        uint32_t kk[4];
        load4_keys(row_area + base, bulk, r.row + base, i, cnt, false, kk);
        uint32_t* dst = reinterpret_cast<uint32_t*>(row_area + base);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i + e < cnt) dst[i + e] = kk[e];
      }
    }
    __syncthreads();
  }

  // ---- 2. ordered compaction of the entries whose top 11 bits are >= b0
  // into the list: each warp owns a segment of the piece, counts, and after
  // one barrier writes its matches at ballot-prefix positions.  Writing
  // stops (overflow) once the list would exceed its capacity.
  bool overflow = false;
  auto compact = [&](const float* sm, int bulk, const float* gl, int base, int cnt, bool keys_in_sm,
                     uint32_t b0, int& run) {
    const int seg = warp_segment(cnt);
    const int w_lo = min(cnt, warp * seg), w_hi = min(cnt, w_lo + seg);
    int c = 0;
    for (int c0 = w_lo; c0 < w_hi; c0 += 128) {
      uint32_t kk[4];
      load4_keys(sm, bulk, gl, c0 + 4 * lane, w_hi, keys_in_sm, kk);
#pragma unroll
      for (int e = 0; e < 4; ++e) c += (c0 + 4 * lane + e < w_hi) && (kk[e] >> 21) >= b0;
    }
    c = __reduce_add_sync(0xffffffffu, c);
    int2 tot;
    int pos = run + warp_bases(fx, 0, c, 0, tot).x;
    if (run + tot.x > a.list_cap) {  // uniform: totals are the CTA's
      overflow = true;
      run += tot.x;
      return;
    }
    for (int c0 = w_lo; c0 < w_hi; c0 += 128) {
      const int i = c0 + 4 * lane;
      uint32_t kk[4];
      load4_keys(sm, bulk, gl, i, w_hi, keys_in_sm, kk);
      bool f[4];
      unsigned bf[4];
      int before = 0, all = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        f[e] = (i + e < w_hi) && (kk[e] >> 21) >= b0;
        bf[e] = __ballot_sync(0xffffffffu, f[e]);
        before += __popc(bf[e] & lt_mask);
        all += __popc(bf[e]);
      }
      int o = pos + before;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (f[e]) {
          list_idx[o] = base + i + e;
          list_key[o] = kk[e];
          ++o;
        }
      }
      pos += all;
    }
    run += tot.x;
  };
  auto compact_row = [&](uint32_t b0) {
    int run = 0;
    overflow = false;
    if (a.resident) {
      compact(row_area, n, r.row, 0, n, true, b0, run);
    } else {
      rs.walk([&](const float* sm, int bulk, const float* gl, int base, int cnt) {
        if (!overflow) compact(sm, bulk, gl, base, cnt, false, b0, run);
      });
    }
    __syncthreads();
    return run;
  };

  // ---- 1. a lower bound b0 for the top bits of the k-th key -------------
  // Sample 1024 keys at even strides; take the bin of the sample's r-th
  // largest key, r set so that about 1.5k + 8n/1024 keys of the row are
  // expected at or above it.  The estimate only steers the work: if the
  // list ends up with fewer than k entries (b0 too high) or overflows, the
  // exact histogram of the whole row decides b0 instead.
  uint32_t prefix = 0;
  int shift = 32;
  int k_rem = a.k;
  int m_list = 0;
  bool use_list = false;
  int first_pass = 0;
  if (n >= kSelSampleMin) {
    {
      const int64_t i = (int64_t)threadIdx.x * n / kSelThreads;
      const uint32_t kq = a.resident ? reinterpret_cast<const uint32_t*>(row_area)[i]
                                     : order_key(__ldg(r.row + i));
      atomicAdd(&fx.hist[0][kq >> 21], 1u);
    }
    __syncthreads();
    const int target = min(kSelThreads, (int)((3LL * a.k * kSelThreads + 2LL * n - 1) / (2LL * n)) + 8);
    find_bin(fx, kHistBins, 1, 0, target);
    const uint32_t b_s = (uint32_t)fx.info[0];
    m_list = compact_row(b_s);
    use_list = !overflow && m_list >= a.k;
  }
  if (!use_list) {
    // exact: histogram of the top 11 bits over the whole row
    for (int i = threadIdx.x; i < kHistCopies * kHistBins; i += kSelThreads) (&fx.hist[0][0])[i] = 0;
    __syncthreads();
    if (a.resident) {
      const uint32_t* keys = reinterpret_cast<const uint32_t*>(row_area);
      for (int i = 4 * threadIdx.x; i < n; i += 4 * kSelThreads) {
        uint32_t kk[4];
        load4_keys(row_area, n, r.row, i, n, true, kk);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (i + e < n) atomicAdd(&hcopy[kk[e] >> 21], 1u);
      }
      (void)keys;
    } else {
      rs.walk([&](const float* sm, int bulk, const float* gl, int base, int cnt) {
        const int i = 4 * threadIdx.x;
        if (i < cnt) {
          uint32_t kk[4];
          load4_keys(sm, bulk, gl, i, cnt, false, kk);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (i + e < cnt) atomicAdd(&hcopy[kk[e] >> 21], 1u);
        }
      });
    }
    __syncthreads();
    find_bin(fx, kHistBins, kHistCopies, 0, a.k);
    const uint32_t b0 = (uint32_t)fx.info[0];
    const int above0 = fx.info[1];
    const int cnt0 = fx.info[2];
    prefix = b0;
    shift = 21;
    k_rem = a.k - above0;
    first_pass = 1;
    if (above0 + cnt0 <= a.list_cap) {
      m_list = compact_row(b0);
      use_list = true;
    }
    if (cnt0 == k_rem) first_pass = 3;  // the whole bin is selected
  }

  // ---- 3. exact threshold: radix passes (11, 11, 10 bits) ---------------
  {
    for (int pass = first_pass; pass < 3; ++pass) {
      const int bits = pass < 2 ? 11 : 10;
      const int nbins = 1 << bits;
      const int nshift = shift - bits;
      const uint32_t mask = (uint32_t)nbins - 1u;
      for (int i = threadIdx.x; i < nbins; i += kSelThreads) fx.hist[0][i] = 0;
      __syncthreads();
      auto add = [&](uint32_t kq) {
        if (shift == 32 || (kq >> shift) == prefix) atomicAdd(&fx.hist[0][(kq >> nshift) & mask], 1u);
      };
      if (use_list) {
        for (int i = threadIdx.x; i < m_list; i += kSelThreads) add(list_key[i]);
      } else if (a.resident) {
        const uint32_t* keys = reinterpret_cast<const uint32_t*>(row_area);
        for (int i = threadIdx.x; i < n; i += kSelThreads) add(keys[i]);
      } else {
        rs.walk([&](const float* sm, int bulk, const float* gl, int base, int cnt) {
          const int i = 4 * threadIdx.x;
          if (i < cnt) {
            uint32_t kk[4];
            load4_keys(sm, bulk, gl, i, cnt, false, kk);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (i + e < cnt) add(kk[e]);
          }
        });
      }
      __syncthreads();
      find_bin(fx, nbins, 1, 0, k_rem);
      const uint32_t bin = (uint32_t)fx.info[0];
      k_rem -= fx.info[1];
      const int bin_count = fx.info[2];
      prefix = shift == 32 ? bin : ((prefix << bits) | bin);
      shift = nshift;
      if (bin_count == k_rem) break;  // the whole bin is selected
    }
  }
  const int need = k_rem;  // keys equal to the threshold prefix to take

  // ---- 4. emission in ascending index order -----------------------------
  int run_gt = 0, run_eq = 0;  // above / equal keys before the current piece
  // items [0, cnt) of a piece whose keys come from key4(i, kk) and whose
  // indices are index(i)
  auto emit_piece = [&](auto key4, auto index, int cnt) {
    const int seg = warp_segment(cnt);
    const int w_lo = min(cnt, warp * seg), w_hi = min(cnt, w_lo + seg);
    int g = 0, q = 0;
    for (int c0 = w_lo; c0 < w_hi; c0 += 128) {
      uint32_t kk[4];
      key4(c0 + 4 * lane, w_hi, kk);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = c0 + 4 * lane + e < w_hi;
        const uint32_t hb = kk[e] >> shift;
        g += in && hb > prefix;
        q += in && hb == prefix;
      }
    }
    g = __reduce_add_sync(0xffffffffu, g);
    q = __reduce_add_sync(0xffffffffu, q);
    int2 tot;
    const int2 wb = warp_bases(fx, 0, g, q, tot);
    int gt_b = run_gt + wb.x, eq_b = run_eq + wb.y;
    for (int c0 = w_lo; c0 < w_hi; c0 += 128) {
      const int i = c0 + 4 * lane;
      uint32_t kk[4];
      key4(i, w_hi, kk);
      bool fg[4], fq[4];
      unsigned bg[4], bq[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool in = i + e < w_hi;
        const uint32_t hb = kk[e] >> shift;
        fg[e] = in && hb > prefix;
        fq[e] = in && hb == prefix;
        bg[e] = __ballot_sync(0xffffffffu, fg[e]);
        bq[e] = __ballot_sync(0xffffffffu, fq[e]);
      }
      int gb = gt_b, qb = eq_b, ng = 0, nq = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        gb += __popc(bg[e] & lt_mask);
        qb += __popc(bq[e] & lt_mask);
        ng += __popc(bg[e]);
        nq += __popc(bq[e]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (fg[e] || (fq[e] && qb < need)) emit_one<kMode>(a, r, index(i + e), gb + min(qb, need));
        gb += fg[e];
        qb += fq[e];
      }
      gt_b += ng;
      eq_b += nq;
    }
    run_gt += tot.x;
    run_eq += tot.y;
  };
  if (use_list) {
    emit_piece([&](int i, int hi, uint32_t(&kk)[4]) {
                 if (i + 3 < hi) {
                   const uint4 v = *reinterpret_cast<const uint4*>(list_key + i);
                   kk[0] = v.x; kk[1] = v.y; kk[2] = v.z; kk[3] = v.w;
                 } else {
#pragma unroll
                   for (int e = 0; e < 4; ++e) kk[e] = i + e < hi ? list_key[i + e] : 0u;
                 }
               },
               [&](int i) { return (int64_t)list_idx[i]; }, m_list);
  } else if (a.resident) {
    const uint32_t* keys = reinterpret_cast<const uint32_t*>(row_area);
    emit_piece([&](int i, int hi, uint32_t(&kk)[4]) {
                 load4_keys(row_area, n, r.row, i, hi, true, kk);
               },
               [&](int i) { return (int64_t)i; }, n);
    (void)keys;
  } else {
    rs.walk([&](const float* sm, int bulk, const float* gl, int base, int cnt) {
      emit_piece([&](int i, int hi, uint32_t(&kk)[4]) { load4_keys(sm, bulk, gl, i, hi, false, kk); },
                 [&](int i) { return (int64_t)base + i; }, cnt);
    });
  }
  emit_tail<kMode>(a, r, a.k);
}

}  // namespace qsa
