// score_tc.cuh -- block scorer on the 5th-generation tensor cores (tcgen05).
//
// Qwen3.8-Flash-Next day-0 write-up (theainews.cc), section "Qwen sparse
// attention (QSA)": prefill scores many query rows against the compressed
// keys with a custom kernel; the score equation is
//   s[t][b] = (1/sqrt(128)) * sum_{h<4} ReLU(<q[t][h], kbar[b]>).
// With several query rows per request the 4 head dot products of every row
// against every key form a dense contraction, so they run on the tensor
// cores:
//   D[key][c] = sum_k K[key][k] * Q[c][k],   c = 4*row + head,
// with M = 128 keys per tile (TMEM lanes), N = 4 * rows per tile (rounded up
// to a multiple of 16, zero-padded), K = 128 in 8 steps of 16 (BF16 inputs,
// FP32 accumulation in TMEM).  Both operands are K-major in shared memory
// with the 128-byte swizzle.  score_tc_kernel (pages of a multiple of 32
// tokens) takes the keys as TMA boxes, one 4 KB box per run of pool rows
// through a 4-D tensor map, so the engine writes them straight into the
// swizzled layout; score_tc_cpasync_kernel (smaller pages, whose compressed
// rows do not form whole 8-row atoms) fills the tile with 16-byte cp.async
// pieces, every 256-byte key row fetched on its own.  One thread issues the
// MMAs and commits them to an mbarrier; the epilogue reads TMEM (each warp
// its 32 lanes = 32 keys), applies ReLU, sums the 4 head columns of each
// row, scales, and stores the FP32 scores (coalesced: consecutive keys of one
// row).  A CTA keeps its query rows resident and walks a group of key tiles
// through a ring of up to 8 key buffers, and the accumulator is
// double-buffered in TMEM, so tile k's MMA overlaps tile k-1's epilogue.
//
// Every wait is bounded (a timeout latches kFaultWait and the CTA frees its
// tensor memory before leaving).
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace qsa {

constexpr int kTcThreads = 1024;          // 32 warps: all issue key copies; TMEM lane quarter = warp % 4
constexpr int kTcM = 128;                 // keys per tile
constexpr int kTcHalf = kTcM * 128;       // bytes of one K-half of the key tile (128 rows x 128 B)
constexpr int kTcMaxStages = 8;           // key-ring stages (32 KB each), sized to the shared memory left
constexpr int kTcPtStage = 4096;          // page-table entries staged in shared memory per CTA

struct TcArgs {
  const __nv_bfloat16* q;       // [n_rows][4][128]
  const __nv_bfloat16* pool;    // [pool_rows][128]
  int64_t pool_rows;
  int32_t n_req;
  const int32_t* req_row_start; // [n_req+1]
  int32_t n_rows;
  const int32_t* row_len;       // [n_rows]
  int32_t max_len;
  const int32_t* page_table;    // [n_req][ld_pt]
  int64_t ld_pt;
  int32_t page_size;
  float* scores;                // [n_rows][ld_scores]
  int64_t ld_scores;
  int32_t rows_per_tile;        // RT <= 64
  int32_t n_cols;               // N = round16(4 * RT)
  int32_t tmem_cols;            // power of two >= max(32, N)
  int32_t tiles_per_cta;        // key tiles walked by one CTA
  int32_t stages;               // key-ring stages (3..kTcMaxStages)
  int32_t trigger_dependents;
  int32_t box_rows;             // TMA kernel: pool rows per tensor-map box (8..128, divides page_size/4)
  int32_t pt_cap;               // TMA kernel: page-table entries staged in shared memory
  int32_t box4d;                // TMA kernel: 4-D view, one box per run covers both K-halves
  // TMA kernels: nullptr, or per request the first position the previous
  // grid (the key path of the same step) may have written: only CTAs whose
  // blocks reach block new_pos[r]/4 wait for that grid (and CTA 0, so that
  // this grid still completes after it); the rest read the pool at once.
  const int32_t* new_pos;
  const float* head_gates;      // nullptr, or [n_rows][4] gates (see ScoreArgs)
};

// Score of one (row, key) from its 4 head accumulators: the rectified dot
// products summed and scaled; gated: each multiplied by its head's gate
// first (with unit gates the same sums: 1 * x and fma(1, x, y) round like x
// and x + y).
__device__ __forceinline__ float tc_head_sum(const uint32_t* v) {
  float sc = fmaxf(__uint_as_float(v[0]), 0.f);
  sc += fmaxf(__uint_as_float(v[1]), 0.f);
  sc += fmaxf(__uint_as_float(v[2]), 0.f);
  sc += fmaxf(__uint_as_float(v[3]), 0.f);
  return sc * kScoreScale;
}
__device__ __forceinline__ float tc_head_sum_gated(const uint32_t* v, const float* gates, int64_t row) {
  const float4 g = __ldg(reinterpret_cast<const float4*>(gates) + row);
  const float r0 = fmaxf(__uint_as_float(v[0]), 0.f), r1 = fmaxf(__uint_as_float(v[1]), 0.f);
  const float r2 = fmaxf(__uint_as_float(v[2]), 0.f), r3 = fmaxf(__uint_as_float(v[3]), 0.f);
  return fmaf(g.w, r3, fmaf(g.z, r2, fmaf(g.y, r1, g.x * r0))) * kScoreScale;
}

// ---------------------------------------------------------------------------
// PTX wrappers (tcgen05, cp.async).
// ---------------------------------------------------------------------------
// No memory clobber: the copies are ordered by cp.async.wait_group, the proxy
// fence and the CTA barrier that follow them, and without it the compiler may
// hoist the address loads of later copies above earlier ones.
__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// wait_group takes an immediate: dispatch a runtime count (0..6).
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    default: cp_async_wait<6>(); break;
  }
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// K-major, 128-byte swizzle shared-memory matrix descriptor: start address,
// stride between 8-row atoms (1024 B when the atoms of one K-half are packed,
// 2048 B when the two K-halves of each 8 rows alternate), descriptor
// version 1, layout 2.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr, uint32_t sbo_bytes = 1024) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);        // start address
  d |= (uint64_t)1 << 16;                               // leading byte offset (unused, 16 B)
  d |= (uint64_t)(sbo_bytes >> 4) << 32;                // stride byte offset: between 8-row atoms
  d |= (uint64_t)1 << 46;                               // descriptor version
  d |= (uint64_t)2 << 61;                               // 128-byte swizzle
  return d;
}
// kind::f16 instruction descriptor: D = F32, A = B = BF16, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
        "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
        "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
        "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
        "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk c (0..15 along the 256-byte key row) of row r
// in a [2 K-halves][rows][128 B] region with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_offset(int r, int c, int rows) {
  const int kh = c >> 3, cc = c & 7;
  return (uint32_t)(kh * rows * 128 + r * 128 + ((cc ^ (r & 7)) << 4));
}

// Load key tile `kt` of request r (blocks [kt*128, kt*128 + 128) clipped to
// nb) into the swizzled A buffer; rows past nb or on bad pages are zero.
// Thread t copies 16-byte chunk t % 16 of rows t/16 + 32j (j < 4): its
// page-table entries are looked up first, then its copies are issued.
// (cp.async throughput grows with the number of issuing warps, hence 16.)
// Page-table entries [pt0, pt0 + pt_n) of the CTA's key range are staged in
// shared memory (pt_s); others are read from global memory.
__device__ __forceinline__ void tc_load_keys(const TcArgs& a, int r, int kt, int nb, unsigned char* buf,
                                             const int32_t* pt_s, int pt0, int pt_n) {
  constexpr int kRowStep = kTcThreads / 16;
  constexpr int kRowsPerThread = kTcM / kRowStep;
  const int kpp = a.page_size / kBlock;
  const int32_t* pt_row = a.page_table + (int64_t)r * a.ld_pt;
  const int c = threadIdx.x & 15, r0 = threadIdx.x >> 4;
  int64_t prow[kRowsPerThread];
#pragma unroll
  for (int j = 0; j < kRowsPerThread; ++j) {
    const int b = kt * kTcM + r0 + kRowStep * j;
    prow[j] = -1;
    if (b < nb) {
      const int page_idx = b / kpp;
      if (page_idx < a.ld_pt) {
        const int64_t page = (page_idx >= pt0 && page_idx < pt0 + pt_n) ? pt_s[page_idx - pt0]
                                                                          : __ldg(pt_row + page_idx);
        const int64_t pr = page * kpp + (b - page_idx * kpp);
        if (page >= 0 && pr < a.pool_rows) prow[j] = pr;
        else if (c == 0) raise_fault(kFaultPool);
      } else if (c == 0) {
        raise_fault(kFaultIndex);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kRowsPerThread; ++j) {
    const bool ok = prow[j] >= 0;
    cp_async_16(buf + sw128_offset(r0 + kRowStep * j, c, kTcM), ok ? a.pool + prow[j] * kDim + c * 8 : a.pool,
                ok ? 16u : 0u);
  }
}

__global__ void __launch_bounds__(kTcThreads)
score_tc_cpasync_kernel(TcArgs a) {
  extern __shared__ __align__(16) unsigned char tc_smem_raw[];
  // layout from the first 1024-byte boundary (the swizzle atoms need it):
  // [A stages x 32 KB][B: 2 x N x 128 B][2 mbarriers][TMEM address][fail flag][row lengths][page table]
  unsigned char* base = tc_smem_raw + ((1024u - (smem_u32(tc_smem_raw) & 1023u)) & 1023u);
  const int S = a.stages;
  auto abuf = [&](int stage) { return base + (size_t)stage * 2 * kTcHalf; };
  unsigned char* bbuf = base + (size_t)S * 2 * kTcHalf;
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(bbuf + 2 * a.n_cols * 128);  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_bar + 2);
  int* s_fail = reinterpret_cast<int*>(tmem_slot + 1);
  int* s_nb = s_fail + 1;               // [rows_per_tile]
  int32_t* pt_s = s_nb + a.rows_per_tile;  // [kTcPtStage]

  // Launched with programmatic serialisation: nothing is read before the
  // previous grid on the stream has finished, and the dependent selection
  // may only start once that holds here.
  pdl_wait_primary();
  if (a.trigger_dependents) pdl_launch_dependents();

  const int r = blockIdx.z;
  const int row0 = __ldg(a.req_row_start + r), row1 = __ldg(a.req_row_start + r + 1);
  if (row0 < 0 || row1 < row0 || row1 > a.n_rows) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_fault(kFaultGrouping);
    return;
  }
  if (row1 - row0 > (int)gridDim.y * a.rows_per_tile) {  // more rows than max_rows_per_req promised
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_fault(kFaultGrouping);
  }
  const int t0 = row0 + blockIdx.y * a.rows_per_tile;
  const int t1 = min(row1, t0 + a.rows_per_tile);
  if (t0 >= t1) return;
  // visible blocks of each row of the tile; the tile's key range ends at their max
  if (threadIdx.x < t1 - t0) {
    int L = __ldg(a.row_len + t0 + threadIdx.x);
    if (L < 0 || L > a.max_len) { raise_fault(kFaultGrouping); L = 0; }
    s_nb[threadIdx.x] = L / kBlock;
  }
  __syncthreads();
  int nb_tile = 0;
  for (int i = 0; i < t1 - t0; ++i) nb_tile = max(nb_tile, s_nb[i]);
  const int n_kt = (nb_tile + kTcM - 1) / kTcM;
  const int kt0 = blockIdx.x * a.tiles_per_cta;
  const int kt1 = min(n_kt, kt0 + a.tiles_per_cta);
  if (kt0 >= kt1) return;

  // ---- page-table entries of this CTA's key range, staged once ------------
  const int kpp = a.page_size / kBlock;
  const int pt0 = (kt0 * kTcM) / kpp;
  int pt_n = min((kt1 * kTcM - 1) / kpp + 1 - pt0, kTcPtStage);
  if (pt_n > a.ld_pt - pt0) pt_n = (int)(a.ld_pt - pt0);
  if (pt_n < 0) pt_n = 0;
  {
    const int32_t* pt_row = a.page_table + (int64_t)r * a.ld_pt;
    for (int i = threadIdx.x; i < pt_n; i += kTcThreads) pt_s[i] = __ldg(pt_row + pt0 + i);
  }
  __syncthreads();

  // ---- query rows -> B (zero rows beyond 4 * (t1 - t0)) and the first key tile
  const int valid_cols = 4 * (t1 - t0);
  for (int i = threadIdx.x; i < a.n_cols * 16; i += kTcThreads) {
    const int col = i >> 4, c = i & 15;
    const bool ok = col < valid_cols;
    const __nv_bfloat16* src = ok ? a.q + ((int64_t)t0 * kHeads + col) * kDim + c * 8 : a.q;
    cp_async_16(bbuf + sw128_offset(col, c, a.n_cols), src, ok ? 16u : 0u);
  }
  tc_load_keys(a, r, kt0, nb_tile, abuf(0), pt_s, pt0, pt_n);
  cp_async_commit();  // group 0: B and the first key tile
  for (int i = 1; i < S - 2; ++i) {  // groups 1..S-3: the next key tiles (or empty)
    if (kt0 + i < kt1) tc_load_keys(a, r, kt0 + i, nb_tile, abuf(i), pt_s, pt0, pt_n);
    cp_async_commit();
  }

  // ---- tensor memory for the accumulator ----------------------------------
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    mbar_init(&mma_bar[0], 1);
    mbar_init(&mma_bar[1], 1);
    *s_fail = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t idesc = umma_idesc_bf16(kTcM, a.n_cols);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Epilogue of tile kt (accumulator `acc`): warp w reads TMEM lane quarter
  // w % 4 (keys 32(w%4) .. +31) and the column chunks 32 * (w / 4 + 8m).
  auto epilogue = [&](int kt, int acc) {
    const int quarter = warp & 3;
    const int b = kt * kTcM + quarter * 32 + lane;
    const uint32_t acc_col = (uint32_t)(acc * a.n_cols);
    for (int c0 = 32 * (warp >> 2); c0 < a.n_cols; c0 += 32 * (kTcThreads / 128)) {
      uint32_t v[32];
      tmem_ld_32cols(tmem + ((uint32_t)(quarter * 32) << 16) + acc_col + (uint32_t)c0, v);
      if (a.head_gates == nullptr) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int tr = c0 / 4 + j;  // row within the tile
          if (tr < t1 - t0 && b < s_nb[tr]) a.scores[(int64_t)(t0 + tr) * a.ld_scores + b] = tc_head_sum(v + 4 * j);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int tr = c0 / 4 + j;
          if (tr < t1 - t0 && b < s_nb[tr])
            a.scores[(int64_t)(t0 + tr) * a.ld_scores + b] = tc_head_sum_gated(v + 4 * j, a.head_gates, t0 + tr);
        }
      }
    }
  };
  // Warps that read TMEM in the epilogue; only they wait on the MMA barrier
  // (the CTA barrier that follows orders everyone else after them, and a
  // thousand spinning threads would steal issue slots from the copies).
  const bool epi_warp = 32 * (warp >> 2) < a.n_cols;
  // Wait for the MMA of local tile i (accumulator i & 1, its (i >> 1)-th use).
  auto wait_mma = [&](int i) {
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&mma_bar[i & 1], (uint32_t)(i >> 1) & 1u));
    if (!ok && lane == 0) {
      *s_fail = 1;
      raise_fault(kFaultWait);
    }
    tc_fence_after();
    return ok;
  };

  const int n_local = kt1 - kt0;
  for (int i = 0; i < n_local; ++i) {
    const int kt = kt0 + i;
    // Refill the stage of tile i-2 (its MMA completed: waited in iteration
    // i-1) with tile i+S-2.
    if (i + S - 2 < n_local) tc_load_keys(a, r, kt + S - 2, nb_tile, abuf((i + S - 2) % S), pt_s, pt0, pt_n);
    cp_async_commit();
    cp_async_wait_dyn(S - 2);  // tile i (and everything older) has landed
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t a_base = smem_u32(abuf(i % S));
      const uint32_t b_base = smem_u32(bbuf);
      const uint32_t d = tmem + (uint32_t)((i & 1) * a.n_cols);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint32_t koff = (uint32_t)(st >> 2);          // K-half index
        const uint32_t within = (uint32_t)((st & 3) * 32);  // bytes along the 128-byte row
        const uint64_t ad = umma_desc_sw128(a_base + koff * kTcHalf + within);
        const uint64_t bd = umma_desc_sw128(b_base + koff * (uint32_t)(a.n_cols * 128) + within);
        umma_bf16(d, ad, bd, idesc, st > 0 ? 1u : 0u);
      }
      umma_commit(&mma_bar[i & 1]);
    }
    // meanwhile: the epilogue of the previous tile
    if (i > 0 && epi_warp && wait_mma(i - 1)) epilogue(kt - 1, (i - 1) & 1);
    tc_fence_before();
    __syncthreads();  // the previous accumulator and stage are free again
    if (*s_fail) break;  // uniform: read after the barrier
  }
  if (!*s_fail && n_local > 0 && epi_warp && wait_mma(n_local - 1)) epilogue(kt1 - 1, (n_local - 1) & 1);
  tc_fence_before();
  __syncthreads();
  cp_async_wait<0>();
  __syncthreads();
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// TMA-fed, warp-specialised variant (pages of a multiple of 32 tokens, so
// that a page's compressed keys form whole 8-row swizzle atoms).
//
// A page of P tokens holds P/4 consecutive pool rows, so the key tile of 128
// blocks is 128*4/P contiguous runs of pool rows.  Each run is one
// tensor-map box of 64 BF16 x box_rows per K-half, which the TMA engine
// writes straight into the 128-byte-swizzled K-major layout the MMA reads
// (the box's destination is 1024-byte aligned, so its swizzle phase is the
// tile's).  Roles:
//   warp 0      producer: looks up the pages of a tile (one lane per run)
//               and issues its boxes on the stage's `full` barrier;
//   warp 1      MMA issuer (one lane) and TMEM owner: waits `full`, issues
//               the 8 K-steps into one of two TMEM accumulators, commits to
//               the stage's `empty` barrier and the accumulator's `acc_full`;
//   warps 2..    epilogue (8, or 16 for wide prefill tiles): two or four
//               warps per TMEM lane quarter split the column chunks, read the
//               accumulator, apply ReLU / head sum / scale, store coalesced
//               scores, and release `acc_empty`.
// Every wait is bounded; a timeout latches kFaultWait and sets a shared
// abort flag that ends the other roles' waits too, and the CTA drains its
// outstanding copies and MMAs (again bounded) before freeing tensor memory.
// ---------------------------------------------------------------------------
constexpr int kTmWarps = 10;
constexpr int kTmThreads = 32 * kTmWarps;
constexpr int kTmEpiWarps = 8;

struct TmCtl {
  int abort;
  int issued;     // tiles whose copies were issued
  int consumed;   // tiles whose copies the MMA issuer saw land
  int mma_done;   // tiles whose MMAs were committed
  uint32_t tmem;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int g, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(0), "r"(g), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool tm_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_timer_ns() - t0 > 200000000ull) {
      *abort = 1;
      raise_fault(kFaultWait);
      return false;
    }
  }
  return true;
}

// kEpi: epilogue warps, 8 or 16 (4 per TMEM lane quarter, each taking a
// quarter of the column chunks; wide tiles -- prefill, N = 256 -- need 16 to
// keep up with the MMA).
template <int kEpi>
__global__ void __launch_bounds__(32 * (2 + kEpi), 1)
score_tc_kernel(TcArgs a, const __grid_constant__ CUtensorMap pool_map) {
  constexpr int kThreads = 32 * (2 + kEpi);
  extern __shared__ __align__(16) unsigned char tm_smem_raw[];
  // [A stages x 32 KB][B: 2 x N x 128 B][barriers][control][row lengths][page table]
  unsigned char* base = tm_smem_raw + ((1024u - (smem_u32(tm_smem_raw) & 1023u)) & 1023u);
  const int S = a.stages;
  const int N = a.n_cols;
  auto abuf = [&](int stage) { return base + (size_t)stage * 2 * kTcHalf; };
  unsigned char* bbuf = base + (size_t)S * 2 * kTcHalf;
  uint64_t* full = reinterpret_cast<uint64_t*>(bbuf + 2 * N * 128);  // [S]
  uint64_t* empty = full + S;                                         // [S]
  uint64_t* acc_full = empty + S;                                     // [2]
  uint64_t* acc_empty = acc_full + 2;                                 // [2]
  TmCtl* ctl = reinterpret_cast<TmCtl*>(acc_empty + 2);
  int* s_nb = reinterpret_cast<int*>(ctl + 1);  // [rows_per_tile]
  int32_t* pt_s = s_nb + a.rows_per_tile;       // [pt_cap]
  volatile int* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Launched with programmatic serialisation: nothing is read before the
  // previous grid on the stream has finished (with new_pos: nothing that
  // grid writes), and the dependent selection may only start once that
  // holds here.
  const bool relaxed = a.new_pos != nullptr;
  // relaxed: CTA 0 waits before it leaves, so that this grid completes after
  // the previous one; the producer waits before its first tile that reaches
  // a block the previous grid may write
  const bool cta0 = (blockIdx.x | blockIdx.y | blockIdx.z) == 0;
  auto leave = [&]() {
    if (relaxed && cta0) pdl_wait_primary();
  };
  if (!relaxed) pdl_wait_primary();
  if (a.trigger_dependents) pdl_launch_dependents();
  if (threadIdx.x == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&pool_map)) : "memory");

  const int r = blockIdx.z;
  // Page-table entries of this CTA's key range (at most tiles_per_cta tiles
  // from kt0, a range fixed by the CTA index): their loads go out next to
  // the row metadata's, one entry per thread, and land in shared memory
  // once the metadata is known.
  const int kpp = a.page_size / kBlock;
  const int kt0 = blockIdx.x * a.tiles_per_cta;
  const int pt0 = (kt0 * kTcM) / kpp;
  int pt_n = min(((kt0 + a.tiles_per_cta) * kTcM - 1) / kpp + 1 - pt0, a.pt_cap);
  if (pt_n > a.ld_pt - pt0) pt_n = (int)(a.ld_pt - pt0);
  if (pt_n < 0) pt_n = 0;
  const int32_t* pt_row = a.page_table + (int64_t)r * a.ld_pt;
  const int32_t pt_first = (int)threadIdx.x < pt_n ? __ldg(pt_row + pt0 + threadIdx.x) : 0;
  const int row0 = __ldg(a.req_row_start + r), row1 = __ldg(a.req_row_start + r + 1);
  if (row0 < 0 || row1 < row0 || row1 > a.n_rows) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_fault(kFaultGrouping);
    leave();
    return;
  }
  if (row1 - row0 > (int)gridDim.y * a.rows_per_tile) {  // more rows than max_rows_per_req promised
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_fault(kFaultGrouping);
  }
  const int t0 = row0 + blockIdx.y * a.rows_per_tile;
  const int t1 = min(row1, t0 + a.rows_per_tile);
  if (t0 >= t1) {
    leave();
    return;
  }
  const int nrows = t1 - t0;
  if (threadIdx.x < nrows) {
    int L = __ldg(a.row_len + t0 + threadIdx.x);
    if (L < 0 || L > a.max_len) { raise_fault(kFaultGrouping); L = 0; }
    s_nb[threadIdx.x] = L / kBlock;
  }
  __syncthreads();
  int nb_tile = 0, nb_min = INT_MAX;  // most and fewest visible blocks of the tile's rows
  for (int i = 0; i < nrows; ++i) {
    nb_tile = max(nb_tile, s_nb[i]);
    nb_min = min(nb_min, s_nb[i]);
  }
  const int n_kt = (nb_tile + kTcM - 1) / kTcM;
  const int kt1 = min(n_kt, kt0 + a.tiles_per_cta);
  if (kt0 >= kt1) {
    leave();
    return;
  }
  const int n_local = kt1 - kt0;
  const int first_new = relaxed ? max(0, __ldg(a.new_pos + r)) / kBlock : 0;

  // ---- page-table entries of this CTA's key range, staged once ------------
  if ((int)threadIdx.x < pt_n) pt_s[threadIdx.x] = pt_first;
  for (int i = threadIdx.x + kThreads; i < pt_n; i += kThreads) pt_s[i] = __ldg(pt_row + pt0 + i);

  // ---- query rows -> B (zero columns beyond 4 * nrows) ---------------------
  const int valid_cols = 4 * nrows;
  for (int i = threadIdx.x; i < N * 16; i += kThreads) {
    const int col = i >> 4, c = i & 15;
    const bool ok = col < valid_cols;
    const __nv_bfloat16* src = ok ? a.q + ((int64_t)t0 * kHeads + col) * kDim + c * 8 : a.q;
    cp_async_16(bbuf + sw128_offset(col, c, N), src, ok ? 16u : 0u);
  }
  cp_async_commit();

  // ---- barriers and tensor memory -------------------------------------------
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpi);
    }
    ctl->abort = 0;
    ctl->issued = 0;
    ctl->consumed = 0;
    ctl->mma_done = 0;
    fence_mbar_init();
  }
  cp_async_wait<0>();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;

  if (warp == 0) {
    // ---- producer: one lane per run of box_rows pool rows ------------------
    const int R = a.box_rows;
    const int runs = kTcM / R;
    bool waited = !relaxed;
    int i = 0;
    for (; i < n_local; ++i) {
      const int st = i % S;
      if (i >= S) {
        const bool ok = lane == 0 ? tm_wait(&empty[st], (uint32_t)((i / S) - 1) & 1u, abort) : true;
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      }
      if (!waited && (int64_t)(kt0 + i + 1) * kTcM > first_new) {  // this tile may hold new keys
        pdl_wait_primary();
        waited = true;
      }
      const int b = (kt0 + i) * kTcM + lane * R;  // first block of this lane's run
      bool valid = false;
      int prow = 0;
      if (lane < runs && b < nb_tile) {
        const int page_idx = b / kpp;
        if (page_idx < a.ld_pt) {
          const int64_t page = (page_idx >= pt0 && page_idx < pt0 + pt_n) ? pt_s[page_idx - pt0]
                                                                            : __ldg(pt_row + page_idx);
          const int64_t pr = page * kpp + (b - page_idx * kpp);
          if (page >= 0 && pr < a.pool_rows) {
            valid = true;
            prow = (int)pr;
            // visible rows of the run past the pool's end read as zero
            if (pr + min(R, nb_tile - b) > a.pool_rows) raise_fault(kFaultPool);
          } else {
            raise_fault(kFaultPool);
          }
        } else {
          raise_fault(kFaultIndex);
        }
      }
      const unsigned vm = __ballot_sync(0xffffffffu, valid);
      if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)__popc(vm) * 2u * (uint32_t)R * 128u);
      __syncwarp();
      if (valid) {
        if (a.box4d) {  // [run][8-row group][K-half][8 rows][128 B]
          tma_load_4d(abuf(st) + lane * R * 256, &pool_map, prow >> 3, &full[st]);
        } else {        // [K-half][128 rows][128 B]
          unsigned char* dst = abuf(st) + lane * R * 128;
          tma_load_2d(dst, &pool_map, 0, prow, &full[st]);
          tma_load_2d(dst + kTcHalf, &pool_map, 64, prow, &full[st]);
        }
      }
    }
    if (lane == 0) ctl->issued = i;
  } else if (warp == 1) {
    // ---- MMA issuer ---------------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kTcM, N);
      const uint32_t b_base = smem_u32(bbuf);
      const uint32_t a_half = a.box4d ? 1024u : (uint32_t)kTcHalf;  // offset of K-half 1
      const uint32_t a_sbo = a.box4d ? 2048u : 1024u;
      int i = 0;
      for (; i < n_local; ++i) {
        const int st = i % S, acc = i & 1;
        if (!tm_wait(&full[st], (uint32_t)(i / S) & 1u, abort)) break;
        ctl->consumed = i + 1;
        if (i >= 2 && !tm_wait(&acc_empty[acc], (uint32_t)((i >> 1) - 1) & 1u, abort)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(abuf(st));
        const uint32_t d = tmem + (uint32_t)(acc * N);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t koff = (uint32_t)(k >> 2);          // K-half index
          const uint32_t within = (uint32_t)((k & 3) * 32);  // bytes along the 128-byte row
          const uint64_t ad = umma_desc_sw128(a_base + koff * a_half + within, a_sbo);
          const uint64_t bd = umma_desc_sw128(b_base + koff * (uint32_t)(N * 128) + within);
          umma_bf16(d, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        umma_commit(&empty[st]);
        umma_commit(&acc_full[acc]);
        ctl->mma_done = i + 1;
      }
    }
  } else {
    // ---- epilogue: warp w reads TMEM lane quarter w % 4 (keys 32(w%4) ..
    // +31) and the column chunks of its half ---------------------------------
    const int quarter = warp & 3;
    const int cgroup = (warp - 2) >> 2;  // 0 .. kEpi/4 - 1
    for (int i = 0; i < n_local; ++i) {
      const int acc = i & 1;
      const bool ok = __all_sync(0xffffffffu, tm_wait(&acc_full[acc], (uint32_t)(i >> 1) & 1u, abort));
      if (!ok) break;
      tc_fence_after();
      const int b = (kt0 + i) * kTcM + quarter * 32 + lane;
      // every row of the tile sees every key of this key tile: no per-row test
      const bool all_vis = (kt0 + i + 1) * kTcM <= nb_min;
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * N);
      for (int c0 = 32 * cgroup; c0 < N; c0 += 32 * (kEpi / 4)) {
        uint32_t v[32];
        int ncols = 32;
        if (N - c0 >= 32) {
          tmem_ld_32cols(taddr + (uint32_t)c0, v);
        } else {
          uint32_t w16[16];
          tmem_ld_16cols(taddr + (uint32_t)c0, w16);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = w16[e];
          ncols = 16;
        }
        float* dst = a.scores + (int64_t)(t0 + c0 / 4) * a.ld_scores + b;
        if (a.head_gates == nullptr) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int tr = c0 / 4 + j;  // row within the tile
            if (4 * j < ncols && tr < nrows && (all_vis || b < s_nb[tr]))
              dst[(int64_t)j * a.ld_scores] = tc_head_sum(v + 4 * j);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int tr = c0 / 4 + j;
            if (4 * j < ncols && tr < nrows && (all_vis || b < s_nb[tr]))
              dst[(int64_t)j * a.ld_scores] = tc_head_sum_gated(v + 4 * j, a.head_gates, t0 + tr);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort) {
    // Drain before the shared and tensor memory are released: copies issued
    // but never seen landing, and the last committed MMAs.
    for (int j = ctl->consumed; j < ctl->issued; ++j) {
      const uint64_t t_start = global_timer_ns();
      while (!mbar_try_wait(&full[j % S], (uint32_t)(j / S) & 1u) && global_timer_ns() - t_start < 20000000ull) {
      }
    }
    for (int j = max(0, ctl->mma_done - 2); j < ctl->mma_done; ++j) {
      const uint64_t t_start = global_timer_ns();
      while (!mbar_try_wait(&acc_full[j & 1], (uint32_t)(j >> 1) & 1u) &&
             global_timer_ns() - t_start < 20000000ull) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) leave();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                 : "memory");
  }
}

// -inf into scores[t][b] for row_len[t]/4 <= b < n_fill (one CTA per row).
__global__ void fill_neginf_kernel(const int32_t* row_len, int32_t max_len, float* scores, int64_t ld,
                                   int64_t n_fill) {
  const int t = blockIdx.x;
  int L = __ldg(row_len + t);
  if (L < 0 || L > max_len) L = 0;
  for (int64_t b = L / kBlock + threadIdx.x; b < n_fill; b += blockDim.x)
    scores[(int64_t)t * ld + b] = -__int_as_float(0x7f800000);
}

}  // namespace qsa
