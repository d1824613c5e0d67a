// select_cluster.cuh -- exact top-k of one score row spread over a cluster
// of 8 CTAs, for launches with few rows (decode), where one SM per row would
// leave most of the GPU idle and its instruction issue would bound the row.
//
// Same contract as select_kernel (SGLang GLM-5.2 blog, "Kernel Optimization /
// TopK-V2": a selection, exact ties, runtime k, page-table transform fused;
// Qwen3.8-Flash-Next write-up, "Qwen sparse attention (QSA)": 512 blocks ->
// 4 positions each, then the 0-3 pending tokens; -1 marks an empty entry).
// Readings: ties go to the lower index; -0 == +0; NaN ranks below -inf; the
// result is in ascending index order with -1 only as tail padding.
//
// Design.  Keys are order-preserving u32 images of the scores (larger float
// -> larger key; NaN -> 0).  CTA c of the cluster owns the slice
// [c S, c S + S) of the row (S = n / 8 rounded up to 4), thread t of it a
// contiguous run of the slice in registers, so thread order and CTA rank
// order are index order.
//  1. Every CTA counts the same 1024 evenly spaced keys of the row into a
//     histogram of the top 11 bits, then of the next 11 bits inside the
//     chosen bin: all CTAs get the same 22-bit threshold t_s, which about
//     1.5k entries of the row reach (no communication).
//  2. Each CTA counts its candidates (key >= t_s, a float compare against the
//     float image of t_s) and writes the count and its largest key into the
//     leader CTA's shared memory; after a cluster barrier every CTA knows its
//     offset and writes its candidates (key, index) straight into the
//     leader's list, in index order; after a second cluster barrier the
//     other CTAs are done.
//  3. Leader: if the list holds at least k entries (it then holds all of the
//     top k), radix passes over the candidates' offsets key - t_s (2048 bins
//     sized by the largest candidate, then 11 bits at a time while the
//     boundary bin is not taken whole) give the k-th key T and the count
//     `need` of keys equal to T to take (the first ones by index); one packed
//     block scan over the ordered list gives every winner its output
//     position.  If the sample misled (short list or overflow), the leader
//     runs exact radix passes and an ordered emission over the whole row.
//  4. The leader writes the outputs (indices and slots; for QSA the 4
//     positions of every block, one page lookup per block, then the pending
//     tokens, then -1) with consecutive threads on consecutive entries.
#pragma once
#include "select.cuh"

namespace qsa {

constexpr int kScThreads = 256;
constexpr int kScWarps = kScThreads / 32;
constexpr int kScMaxCluster = 8;
constexpr int kScSampleMin = 2048;  // shorter rows: every entry is a candidate

struct ScFixed {
  uint32_t h1[2048];
  uint32_t h2[2048];
  uint32_t h3[2048];
  uint32_t wsum[kScWarps];
  int info[8];
  int cnt[kScMaxCluster];        // leader: candidates of each CTA (written by that CTA)
  uint32_t cmax[kScMaxCluster];  // leader: largest candidate key of each CTA
  uint32_t bmax;                 // this CTA's largest candidate key
};
constexpr int kScFixedBytes = (int)((sizeof(ScFixed) + 127) & ~size_t(127));
static_assert(offsetof(ScFixed, h3) == 2 * 2048 * 4, "histograms must be contiguous");

__device__ __forceinline__ void st_dsmem_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t sc_warp_incl_scan(uint32_t x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}
// Exclusive prefix of x over the CTA in thread order, and the total.  One
// barrier; the next call must come after another barrier.
__device__ __forceinline__ uint32_t sc_block_excl_scan(uint32_t x, uint32_t* wsum, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = sc_warp_incl_scan(x);
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t before = 0u, tot = 0u;
#pragma unroll
  for (int w = 0; w < kScWarps; ++w) {
    const uint32_t v = wsum[w];
    before += w < warp ? v : 0u;
    tot += v;
  }
  total = tot;
  return before + incl - x;
}
// The bin (counted from the top of 2048) that holds the k_rem-th largest
// entry: (bin, entries in higher bins, entries in the bin).  Requires k_rem
// <= the histogram's total.  Two barriers.
__device__ __forceinline__ int3 sc_find_bin(ScFixed& fx, const uint32_t* hist, int k_rem) {
  const int top = 2047 - 8 * (int)threadIdx.x;  // bins top .. top-7
  uint32_t c[8];
  uint32_t s = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = hist[top - j];
    s += c[j];
  }
  uint32_t tot;
  uint32_t above = sc_block_excl_scan(s, fx.wsum, tot);
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
  return make_int3(fx.info[0], fx.info[1], fx.info[2]);
}

__device__ __forceinline__ int32_t sc_slot(const SelectArgs& a, const int32_t* pt_s, int pt_n,
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

// kJ: 16-byte loads per thread for the largest slice (slice <= 1024 kJ).
template <int kMode, int kJ>
__global__ void __launch_bounds__(kScThreads, 1)
select_cluster_kernel(SelectArgs a) {
  extern __shared__ __align__(128) unsigned char sc_smem_raw[];
  ScFixed& fx = *reinterpret_cast<ScFixed*>(sc_smem_raw);
  uint32_t* lkey = reinterpret_cast<uint32_t*>(sc_smem_raw + a.off_lkey);  // [list_cap]
  int32_t* lidx = reinterpret_cast<int32_t*>(sc_smem_raw + a.off_list);    // [list_cap]
  int32_t* pt_s = reinterpret_cast<int32_t*>(sc_smem_raw + a.off_pt);      // [pt_cap]
  int32_t* sel_s = reinterpret_cast<int32_t*>(sc_smem_raw + a.off_sel);    // [k]
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t C = cluster_nctarank();
  // Every CTA of the cluster has started before any shared memory of another
  // is touched: arrive now, wait just before the first remote access.
  cluster_arrive_relaxed();

  // ---- row metadata (not produced by the previous grid) -----------------
  const int t = (int)(blockIdx.x / C);
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
  int pt_n = 0;
  if (rank == 0 && pt_row != nullptr) {  // the leader writes the outputs
    const int64_t last = kMode == kModeQsa ? (int64_t)L : (int64_t)n;  // positions < last
    int64_t np = last > 0 ? (last - 1) / a.page_size + 1 : 0;
    if (np > a.pt_cap) np = a.pt_cap;
    if (np > a.ld_pt) np = a.ld_pt;
    pt_n = (int)np;
    for (int i0 = tid; i0 < pt_n; i0 += 4 * kScThreads) {  // four loads in flight per thread
      int32_t pv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kScThreads;
        pv[u] = i < pt_n ? __ldg(pt_row + i) : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kScThreads;
        if (i < pt_n) pt_s[i] = pv[u];
      }
    }
  }
  uint32_t* hz = fx.h1;  // h1 .. h3 are contiguous
  for (int i = tid; i < 3 * 2048; i += kScThreads) hz[i] = 0u;
  if (tid < 8) fx.info[tid] = 0;
  if (tid == 0) fx.bmax = 0u;
  __syncthreads();
  if (a.wait_primary) pdl_wait_primary();

  const float* row = a.scores + (int64_t)t * a.ld;
  const int k = a.k;
  const int m_sel = n < k ? n : k;  // entries selected

  if (n > k) {
    // The sample keys are needed first: their loads go out before the slice's.
    uint32_t sk[4];
    if (n >= kScSampleMin) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int p = (int)(((int64_t)(tid + kScThreads * u) * n) >> 10);
        sk[u] = order_key(__ldg(row + p));
      }
    }
    // ---- this CTA's slice, thread t's contiguous run in registers --------
    const int S = (((n + (int)C - 1) / (int)C) + 3) & ~3;
    const int s0 = (int)rank * S;
    const int s1 = min(n, s0 + S);
    const int J = (S + 4 * kScThreads - 1) / (4 * kScThreads);  // <= kJ
    const int i0 = s0 + 4 * J * tid;
    float4 v[kJ];
    const float nan = __uint_as_float(0x7fffffffu);  // padding: never a candidate
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      const int i = i0 + 4 * j;
      v[j] = make_float4(nan, nan, nan, nan);
      if (j < J) {
        if (a.vec_ok && i + 3 < s1) {
          v[j] = __ldg(reinterpret_cast<const float4*>(row + i));
        } else {
          if (i < s1) v[j].x = __ldg(row + i);
          if (i + 1 < s1) v[j].y = __ldg(row + i + 1);
          if (i + 2 < s1) v[j].z = __ldg(row + i + 2);
          if (i + 3 < s1) v[j].w = __ldg(row + i + 3);
        }
      }
    }

    // ---- 1. threshold estimate (identical in every CTA) -----------------
    uint32_t t_s = 0u;
    if (n >= kScSampleMin) {
#pragma unroll
      for (int u = 0; u < 4; ++u) atomicAdd(&fx.h1[sk[u] >> 21], 1u);
      __syncthreads();
      const int target = min(1024, (int)((3LL * k * 1024 + 2LL * n - 1) / (2LL * n)) + 8);
      const int3 f1 = sc_find_bin(fx, fx.h1, target);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if ((sk[u] >> 21) == (uint32_t)f1.x) atomicAdd(&fx.h2[(sk[u] >> 10) & 2047u], 1u);
      __syncthreads();
      const int3 f2 = sc_find_bin(fx, fx.h2, target - f1.y);
      t_s = ((uint32_t)f1.x << 21) | ((uint32_t)f2.x << 10);
      // h1, h2 were last read before find_bin's final barrier: clear them
      // for the leader's exact passes (read after the next barriers).
      for (int i = tid; i < 2 * 2048; i += kScThreads) hz[i] = 0u;
    }

    // ---- 2. candidates into the leader's list --------------------------
    // key(v) >= t_s as a float compare: t_s = 0 takes everything, t_s at or
    // below key(-inf) every non-NaN entry, otherwise v >= the float image
    // of t_s (exact for every non-NaN v).
    const int cmode = t_s == 0u ? 0 : (t_s <= 0x007fffffu ? 1 : 2);
    const float t_f = __uint_as_float(t_s >= 0x80000000u ? (t_s & 0x7fffffffu) : ~t_s);
    auto is_cand = [&](float x) { return cmode == 0 ? true : (cmode == 1 ? x == x : x >= t_f); };
    // The largest key of the slice (padding is NaN, key 0) is the largest
    // candidate key whenever the slice has a candidate; the leader takes the
    // maximum over the CTAs, which some candidate reaches.
    uint32_t c = 0u;
    float vmax = nan;
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      vmax = fmaxf(fmaxf(vmax, fmaxf(v[j].x, v[j].y)), fmaxf(v[j].z, v[j].w));  // NaN-ignoring
      if (j < J) {
        const int i = i0 + 4 * j;
        c += (i < s1 && is_cand(v[j].x)) + (i + 1 < s1 && is_cand(v[j].y)) + (i + 2 < s1 && is_cand(v[j].z)) +
             (i + 3 < s1 && is_cand(v[j].w));
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(vmax));
    if (lane == 0 && kmax > 0u) atomicMax(&fx.bmax, kmax);  // visible after the scan's barrier
    uint32_t ctot;
    uint32_t o = sc_block_excl_scan(c, fx.wsum, ctot);
    cluster_wait();  // every CTA has started
    if (tid == 0) {
      st_dsmem_u32(map_shared_rank(&fx.cnt[rank], 0), ctot);
      st_dsmem_u32(map_shared_rank(&fx.cmax[rank], 0), fx.bmax);
    }
    cluster_sync();
    // every warp reads the C counts lane-parallel and scans them
    const uint32_t cr = (uint32_t)lane < C ? ld_dsmem_u32(map_shared_rank(&fx.cnt[lane], 0)) : 0u;
    const uint32_t cincl = sc_warp_incl_scan(cr);
    const uint32_t base = __shfl_sync(0xffffffffu, cincl - cr, (int)rank);
    const uint32_t m = __shfl_sync(0xffffffffu, cincl, 31);
    const int cap = a.list_cap;
    const bool fast = m >= (uint32_t)k && m <= (uint32_t)cap;  // the same in every CTA
    if (fast) {
      const uint32_t lk0 = map_shared_rank(lkey, 0), li0 = map_shared_rank(lidx, 0);
      o += base;
      if (c > 0u) {
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
          if (j < J) {
            const int i = i0 + 4 * j;
            const float xv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (i + e < s1 && is_cand(xv[e])) {
                const uint32_t key = order_key(xv[e]);
                st_dsmem_u32(lk0 + 4u * o, key);
                st_dsmem_u32(li0 + 4u * o, (uint32_t)(i + e));
                ++o;
              }
            }
          }
        }
      }
    }
    cluster_sync();  // the list is complete; the leader's shared memory is no longer touched remotely
    if (rank != 0) return;

    if (fast) {
      // ---- 3. leader: exact k-th key among the candidates -----------------
      const int ml = (int)m;
      uint32_t cm = 0u;
      for (uint32_t r = 0; r < C; ++r) cm = cm > fx.cmax[r] ? cm : fx.cmax[r];
      const uint32_t rel_max = cm - t_s;
      int shift = 0;  // first pass: 2048 bins of 2^shift offsets each
      while ((rel_max >> shift) >= 2048u) ++shift;
      for (int i = tid; i < ml; i += kScThreads) atomicAdd(&fx.h1[(lkey[i] - t_s) >> shift], 1u);
      __syncthreads();
      int3 fb = sc_find_bin(fx, fx.h1, k);
      uint32_t prefix = (uint32_t)fb.x;
      int k_rem = k - fb.y;
      uint32_t* hnext = fx.h2;
      while (fb.z != k_rem && shift > 0) {  // at most two more passes (11 + 10 bits)
        const int nb = shift < 11 ? shift : 11;
        const int nshift = shift - nb;
        const uint32_t mask = (1u << nb) - 1u;
        for (int i = tid; i < ml; i += kScThreads) {
          const uint32_t rel = lkey[i] - t_s;
          if ((rel >> shift) == prefix) atomicAdd(&hnext[(rel >> nshift) & mask], 1u);
        }
        __syncthreads();
        fb = sc_find_bin(fx, hnext, k_rem);
        prefix = (prefix << nb) | (uint32_t)fb.x;
        shift = nshift;
        k_rem -= fb.y;
        hnext = fx.h3;
      }
      const uint32_t need = (uint32_t)k_rem;  // equal entries to take, first by index
      // emission over the ordered list: above before + min(equal before, need)
      const int q = (ml + kScThreads - 1) / kScThreads;
      const int l0 = min(ml, q * tid), l1 = min(ml, l0 + q);
      uint32_t pk = 0u;  // above (low 16 bits), equal (high 16 bits); ml <= list_cap < 65536
      for (int i = l0; i < l1; ++i) {
        const uint32_t hb = (lkey[i] - t_s) >> shift;
        pk += hb > prefix ? 1u : (hb == prefix ? 0x10000u : 0u);
      }
      uint32_t tot;
      const uint32_t bs = sc_block_excl_scan(pk, fx.wsum, tot);
      uint32_t gb = bs & 0xffffu, qb = bs >> 16;
      for (int i = l0; i < l1; ++i) {
        const uint32_t hb = (lkey[i] - t_s) >> shift;
        const bool gt = hb > prefix, eq = hb == prefix;
        const uint32_t pos = gb + (qb < need ? qb : need);
        if ((gt || (eq && qb < need)) && pos < (uint32_t)k) sel_s[pos] = lidx[i];
        gb += gt;
        qb += eq;
      }
      __syncthreads();
    } else {
      // ---- leader, exact over the whole row (the sample misled) -----------
      // Radix passes of 11, 11 and 10 bits over the row read from global
      // memory (h1..h3 are zero here), then an ordered emission.
      uint32_t prefix = 0u;
      int shift = 32, k_rem = k;
      for (int pass = 0; pass < 3; ++pass) {
        uint32_t* hist = pass == 0 ? fx.h1 : (pass == 1 ? fx.h2 : fx.h3);
        const int nb = pass < 2 ? 11 : 10;
        const int nshift = shift - nb;
        const uint32_t mask = (1u << nb) - 1u;
        for (int i = tid; i < n; i += kScThreads) {
          const uint32_t key = order_key(__ldg(row + i));
          if (shift == 32 || (key >> shift) == prefix) atomicAdd(&hist[(key >> nshift) & mask], 1u);
        }
        __syncthreads();
        const int3 fb = sc_find_bin(fx, hist, k_rem);
        prefix = shift == 32 ? (uint32_t)fb.x : ((prefix << nb) | (uint32_t)fb.x);
        shift = nshift;
        k_rem -= fb.y;
        if (fb.z == k_rem) break;
      }
      const uint32_t need = (uint32_t)k_rem;
      const int q = (n + kScThreads - 1) / kScThreads;
      const int l0 = min(n, q * tid), l1 = min(n, l0 + q);
      uint32_t pk = 0u;  // above (low 16 bits), equal (high 16 bits); n <= 32768
      for (int i = l0; i < l1; ++i) {
        const uint32_t hb = order_key(__ldg(row + i)) >> shift;
        pk += hb > prefix ? 1u : (hb == prefix ? 0x10000u : 0u);
      }
      uint32_t tot;
      const uint32_t bs = sc_block_excl_scan(pk, fx.wsum, tot);
      uint32_t gb = bs & 0xffffu, qb = bs >> 16;
      for (int i = l0; i < l1; ++i) {
        const uint32_t hb = order_key(__ldg(row + i)) >> shift;
        const bool gt = hb > prefix, eq = hb == prefix;
        const uint32_t pos = gb + (qb < need ? qb : need);
        if ((gt || (eq && qb < need)) && pos < (uint32_t)k) sel_s[pos] = i;
        gb += gt;
        qb += eq;
      }
      __syncthreads();
    }
  } else {
    cluster_wait();  // matches the arrive above; nothing remote follows
    if (rank != 0) return;
  }

  // ---- 4. outputs (leader) ------------------------------------------------
  auto sel = [&](int j) { return n > k ? sel_s[j] : j; };
  if (kMode == kModeTopk) {
    int32_t* oi = a.out_idx + (int64_t)t * k;
    int32_t* os = a.out_slots ? a.out_slots + (int64_t)t * k : nullptr;
    for (int j = tid; j < k; j += kScThreads) {
      const int32_t idx = j < m_sel ? sel(j) : -1;
      oi[j] = idx;
      if (os != nullptr) os[j] = idx < 0 ? -1 : sc_slot(a, pt_s, pt_n, pt_row, idx);
    }
  } else {
    int32_t* oi = a.out_idx != nullptr ? a.out_idx + (int64_t)t * k : nullptr;
    const int width = kBlock * k + (kBlock - 1);
    const int pend = L - kBlock * n;  // tokens of the incomplete block
    int32_t* xs = a.out_xslots + (int64_t)t * width;
    int32_t* xp = a.out_pos ? a.out_pos + (int64_t)t * width : nullptr;
    // Selected blocks: lane l of a warp owns block base + l and looks up its
    // page once (a page holds whole blocks, so the block's 4 slots are
    // consecutive); the warp then writes its 128 consecutive entries with
    // consecutive lanes, each taking the block's slot from its owner lane.
    for (int base = 32 * (tid >> 5); base < m_sel; base += kScThreads) {
      const int b = base + lane;
      int32_t blk = 0, s0 = 0;
      bool ok = false;
      if (b < m_sel) {
        blk = sel(b);
        s0 = sc_slot(a, pt_s, pt_n, pt_row, kBlock * blk);
        ok = s0 != -1;  // -1 only for a page index past the table (fault raised)
        if (oi != nullptr) oi[b] = blk;
      }
      const int nw = min(32, m_sel - base);
#pragma unroll
      for (int r = 0; r < kBlock; ++r) {
        const int e = lane + 32 * r;  // entry of the warp's 4 x 32
        const int src = e >> 2;
        const int32_t sv = __shfl_sync(0xffffffffu, s0, src);
        const int32_t bv = __shfl_sync(0xffffffffu, blk, src);
        const bool okv = __shfl_sync(0xffffffffu, (int)ok, src) != 0;
        if (src < nw) {
          const int j = kBlock * base + e;
          xs[j] = okv ? sv + (e & (kBlock - 1)) : -1;
          if (xp != nullptr) xp[j] = kBlock * bv + (e & (kBlock - 1));
        }
      }
    }
    // then the pending tokens and the -1 padding
    for (int j = kBlock * m_sel + tid; j < width; j += kScThreads) {
      const int32_t p = j - kBlock * m_sel < pend ? kBlock * n + (j - kBlock * m_sel) : -1;
      xs[j] = p < 0 ? -1 : sc_slot(a, pt_s, pt_n, pt_row, p);
      if (xp != nullptr) xp[j] = p;
    }
    if (oi != nullptr)
      for (int j = m_sel + tid; j < k; j += kScThreads) oi[j] = -1;
  }
}

}  // namespace qsa
