// expand.cuh -- selected blocks -> token positions + pending tokens -> KV
// slots.
//
// Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen sparse
// attention (QSA)": every kept block stands for its 4 token positions, and the
// 0-3 tokens of the still-incomplete block are appended, so attention sees at
// most 4k+3 positions.  SGLang GLM-5.2 blog, section "TopK-V2", Figure 2:
// logical positions are translated into physical KV-cache slots.
// vllm-sparse-mla-blackwell, "Design notes worth knowing": -1 marks an empty
// entry (consumers mask on index >= 0).
//
// One CTA per row: a block-wide scan compacts the non-negative block ids (so
// a -1 in the middle of the input is skipped), each kept block writes its 4
// positions and slots, and the tail holds the pending tokens then -1.
#pragma once
#include "common.cuh"

namespace qsa {

constexpr int kExpThreads = 256;

struct ExpandArgs {
  const int32_t* sel;            // [n_rows][k]
  int32_t k;
  int32_t n_req;
  const int32_t* req_row_start;  // [n_req+1]
  int32_t n_rows;
  const int32_t* row_len;        // [n_rows]
  const int32_t* page_table;     // [n_req][ld_pt]
  int64_t ld_pt;
  int32_t page_size;
  int32_t* out_pos;              // [n_rows][4k+3] or nullptr
  int32_t* out_slots;            // [n_rows][4k+3]
};

__device__ __forceinline__ int32_t slot_of(const int32_t* __restrict__ pt_row, int64_t ld_pt,
                                           int32_t page_size, int32_t pos) {
  const int32_t page_idx = pos / page_size;
  if (page_idx >= ld_pt) {
    raise_fault(kFaultIndex);
    return -1;
  }
  return __ldg(pt_row + page_idx) * page_size + (pos - page_idx * page_size);
}

__global__ void __launch_bounds__(kExpThreads)
expand_kernel(ExpandArgs a) {
  __shared__ int s_warp[kExpThreads / 32 + 1];
  const int t = blockIdx.x;
  const int req = row_request(a.req_row_start, a.n_req, t);
  const int L = max(0, __ldg(a.row_len + t));
  const int nb = L / kBlock;
  const int32_t* pt_row = a.page_table + (int64_t)req * a.ld_pt;
  const int width = kBlock * a.k + (kBlock - 1);
  const int per = (a.k + kExpThreads - 1) / kExpThreads;  // <= 8
  const int j0 = threadIdx.x * per;

  int cnt = 0;
  for (int j = j0; j < min(a.k, j0 + per); ++j) cnt += __ldg(a.sel + (int64_t)t * a.k + j) >= 0;
  // Block exclusive scan of cnt.
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < kExpThreads / 32; ++i) { const int v = s_warp[i]; s_warp[i] = run; run += v; }
    s_warp[kExpThreads / 32] = run;
  }
  __syncthreads();
  int out = s_warp[w] + x - cnt;
  const int m = s_warp[kExpThreads / 32];

  for (int j = j0; j < min(a.k, j0 + per); ++j) {
    const int b = __ldg(a.sel + (int64_t)t * a.k + j);
    if (b < 0) continue;
    int32_t base = -1;
    if (b < nb) base = slot_of(pt_row, a.ld_pt, a.page_size, kBlock * b);
    else raise_fault(kFaultIndex);
#pragma unroll
    for (int c = 0; c < kBlock; ++c) {
      a.out_slots[(int64_t)t * width + kBlock * out + c] = base < 0 ? -1 : base + c;
      if (a.out_pos != nullptr) a.out_pos[(int64_t)t * width + kBlock * out + c] = kBlock * b + c;
    }
    ++out;
  }
  const int pend = L - kBlock * nb;
  for (int j = kBlock * m + threadIdx.x; j < width; j += kExpThreads) {
    const int i = j - kBlock * m;
    int32_t pos = -1, slot = -1;
    if (i < pend) {
      pos = kBlock * nb + i;
      slot = slot_of(pt_row, a.ld_pt, a.page_size, pos);
    }
    a.out_slots[(int64_t)t * width + j] = slot;
    if (a.out_pos != nullptr) a.out_pos[(int64_t)t * width + j] = pos;
  }
}

// IndexShare reuse (Qwen3.8-Flash-Next day-0 write-up, section "IndexShare
// MTP: reusing the QSA selection across draft steps"): a draft row runs no
// scorer and no top-k; it reads the selection kept at its request's
// draft-extend row (cap_len tokens seen there) and every position from that
// row's first pending token, 4*floor(cap_len/4), up to its own position.
// Captured positions at or past the row's own length are cut (a row earlier
// than the capture sees only its past).  Row width 4k + 3 + n_extra.
//
// One CTA per row, as expand_kernel: a block-wide scan of the per-block
// position counts (4, fewer for a block cut by the row's length) places each
// block; the tail follows.  A captured block that was not complete at the
// capture is skipped (kFaultIndex), a tail that does not fit is cut at the
// width (kFaultCapacity), a request whose captured row is out of range gets
// a row of -1 (kFaultIndex).
struct ShareArgs {
  const int32_t* cap_sel;        // [n_cap][k]
  const int32_t* cap_len;        // [n_cap]
  int32_t n_cap;
  const int32_t* cap_row;        // [n_req]
  int32_t k;
  int32_t n_extra;
  int32_t n_req;
  const int32_t* req_row_start;  // [n_req+1]
  int32_t n_rows;
  const int32_t* row_len;        // [n_rows]
  const int32_t* page_table;     // [n_req][ld_pt]
  int64_t ld_pt;
  int32_t page_size;
  int32_t* out_pos;              // [n_rows][4k+3+n_extra] or nullptr
  int32_t* out_slots;            // [n_rows][4k+3+n_extra]
};

__global__ void __launch_bounds__(kExpThreads)
indexshare_kernel(ShareArgs a) {
  __shared__ int s_warp[kExpThreads / 32 + 1];
  const int t = blockIdx.x;
  const int req = row_request(a.req_row_start, a.n_req, t);
  const int64_t width = (int64_t)kBlock * a.k + (kBlock - 1) + a.n_extra;
  int32_t* o_slots = a.out_slots + (int64_t)t * width;
  int32_t* o_pos = a.out_pos != nullptr ? a.out_pos + (int64_t)t * width : nullptr;
  const int c = __ldg(a.cap_row + req);
  if (c < 0 || c >= a.n_cap) {
    if (threadIdx.x == 0) raise_fault(kFaultIndex);
    for (int64_t j = threadIdx.x; j < width; j += kExpThreads) {
      o_slots[j] = -1;
      if (o_pos != nullptr) o_pos[j] = -1;
    }
    return;
  }
  const int L = max(0, __ldg(a.row_len + t));
  const int nb0 = max(0, __ldg(a.cap_len + c)) / kBlock;
  const int32_t* sel = a.cap_sel + (int64_t)c * a.k;
  const int32_t* pt_row = a.page_table + (int64_t)req * a.ld_pt;
  constexpr int kPer = kMaxK / kExpThreads;
  const int per = (a.k + kExpThreads - 1) / kExpThreads;  // <= kPer
  const int j0 = threadIdx.x * per;

  // positions each captured block contributes (4, fewer when the row's
  // length cuts it, none for -1 or a block incomplete at the capture), and
  // the block's page-table entry, fetched before the scan so that its
  // latency overlaps the scan
  int nb_[kPer], b_[kPer];
  int32_t base_[kPer];
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = j0 + i;
    b_[i] = (i < per && j < a.k) ? __ldg(sel + j) : -1;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int b = b_[i];
    nb_[i] = 0;
    base_[i] = -1;
    if (b < 0) continue;
    if (b >= nb0) {
      raise_fault(kFaultIndex);
      continue;
    }
    nb_[i] = min(kBlock, max(0, L - kBlock * b));
    if (nb_[i] > 0) base_[i] = slot_of(pt_row, a.ld_pt, a.page_size, kBlock * b);  // 4b..4b+3 share a page
    cnt += nb_[i];
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < kExpThreads / 32; ++i) { const int v = s_warp[i]; s_warp[i] = run; run += v; }
    s_warp[kExpThreads / 32] = run;
  }
  __syncthreads();
  int out = s_warp[w] + x - cnt;
  const int m = s_warp[kExpThreads / 32];  // <= 4k < width

#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int n = nb_[i];
    for (int c = 0; c < n; ++c) {
      o_slots[out + c] = base_[i] < 0 ? -1 : base_[i] + c;
      if (o_pos != nullptr) o_pos[out + c] = kBlock * b_[i] + c;
    }
    out += n;
  }
  // the capture's pending tokens and every token drafted since
  const int start = kBlock * nb0;
  const int64_t n_tail = max(0, L - start);
  if (threadIdx.x == 0 && m + n_tail > width) raise_fault(kFaultCapacity);
  for (int64_t j = m + threadIdx.x; j < width; j += kExpThreads) {
    const int64_t i = j - m;
    int32_t pos = -1, slot = -1;
    if (i < n_tail) {
      pos = start + (int32_t)i;
      slot = slot_of(pt_row, a.ld_pt, a.page_size, pos);
    }
    o_slots[j] = slot;
    if (o_pos != nullptr) o_pos[j] = pos;
  }
}

}  // namespace qsa
