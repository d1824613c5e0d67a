// qsa_api.cu -- the extern "C" entry points of libqsa.so: host-side argument
// checks, launch shapes, and launches on the caller's stream.  Declarations
// and the contract of every call are in include/qsa.h.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/qsa.h"
#include "common.cuh"
#include "compress.cuh"
#include "expand.cuh"
#include "score_decode.cuh"
#include "score_mma.cuh"
#include "score_tc.cuh"
#include "select.cuh"
#include "select_resident.cuh"
#include "select_cluster.cuh"
#include "select_long.cuh"
#include "select_rows.cuh"
#include "select_fast.cuh"
#include "sparse_attn.cuh"

using namespace qsa;

namespace {

constexpr int kMaxDevices = 64;
// Tensor-core scorer limits: rows per tile (N = 4 rows <= 256 columns) and
// the largest shared-memory request (occupancy may be limited with it).
constexpr int kTcMaxRowsPerTile = 64;
constexpr int kTcMinRows = 2;  // requests with this many rows or more use the tensor cores
constexpr int kTcMaxSmem = 227 * 1024;
// Shared-memory plan of the selection kernel: candidate list and staged
// page-table entries per CTA, and the largest dynamic size it may use.
constexpr int kSelListCap = 6144;
constexpr int kSelPtStage = 2048;
constexpr int kSelMaxSmem = kSelFixedBytes + kSelPtStage * 4 + kSelListCap * 8 +
                            kSelResidentCap * 4;
// Rows of up to kRsMaxRow entries take the shared-memory-resident kernel;
// its candidate list gets what the row, page table and output leave of
// kRsMaxSmem (at least 2 * kMaxK entries, at most kRsListMax).
constexpr int kRsMaxSmem = 227 * 1024;
constexpr int kRsListMax = 8192;
// Few rows: one cluster of C CTAs per row (select_cluster_kernel), with a
// candidate list of kScListCap entries in the leader.
constexpr int kScListCap = 8192;
constexpr int kScSmem = kScFixedBytes + 2 * kScListCap * 4 + kSelPtStage * 4 + kMaxK * 4;

// Long rows (more than kRsMaxRow entries) with few rows: one cluster of
// 2..16 CTAs per row (select_long_kernel), each CTA keeping as much of its
// slice in shared memory as kSlSmem leaves.
constexpr int kSlSmem = 227 * 1024;

// Sparse attention instances: (query heads per KV head, head dim).
template <int G, int D>
bool set_attn_smem_one() {
  return cudaFuncSetAttribute(sparse_attn_kernel<G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sizeof(SaSmem<G, D>)) == cudaSuccess;
}
bool set_attn_smem() {
  return set_attn_smem_one<1, 128>() && set_attn_smem_one<2, 128>() && set_attn_smem_one<4, 128>() &&
         set_attn_smem_one<8, 128>() && set_attn_smem_one<16, 128>() && set_attn_smem_one<1, 256>() &&
         set_attn_smem_one<2, 256>() && set_attn_smem_one<4, 256>() && set_attn_smem_one<8, 256>();
}

template <bool kFp8>
bool set_mma_smem() {
  return cudaFuncSetAttribute(score_mma_kernel<1, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sm_smem_bytes(kSmMaxReq, 1)) == cudaSuccess &&
         cudaFuncSetAttribute(score_mma_kernel<2, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sm_smem_bytes(kSmMaxReq, 2)) == cudaSuccess &&
         cudaFuncSetAttribute(score_mma_kernel<3, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sm_smem_bytes(kSmMaxReq, 3)) == cudaSuccess &&
         cudaFuncSetAttribute(score_mma_kernel<4, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sm_smem_bytes(kSmMaxReq, 4)) == cudaSuccess;
}

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int sl_clusters[5] = {0, 0, 0, 0, 0};  // co-resident clusters of 1, 2, 4, 8, 16 long-row CTAs
  cudaStream_t side = nullptr;           // the planned selection's short class runs here, beside the long one
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device one-time set-up: SM count and the shared-memory opt-in of the
// selection kernels.
qsa_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return QSA_ERR_CUDA;
    if (d.side == nullptr && cudaStreamCreateWithFlags(&d.side, cudaStreamNonBlocking) != cudaSuccess)
      return QSA_ERR_CUDA;
    const int smem = kSelMaxSmem;
    if (cudaFuncSetAttribute(select_kernel<kModeTopk>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(select_kernel<kModeQsa>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess ||
        cudaFuncSetAttribute(select_resident_kernel<kModeTopk>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kRsMaxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(select_resident_kernel<kModeQsa>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kRsMaxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(select_cluster_kernel<kModeTopk, 4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kScSmem) != cudaSuccess ||
        cudaFuncSetAttribute(select_cluster_kernel<kModeQsa, 4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kScSmem) != cudaSuccess ||
        cudaFuncSetAttribute(score_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kScoreSmem) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_cpasync_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTcMaxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_cpasync_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTcMaxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTcMaxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_kernel<8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(score_tc_kernel<16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return QSA_ERR_CUDA;
    for (int m = 0; m < 2; ++m) {
      void (*kern)(SelectArgs) = m == 0 ? select_long_kernel<kModeTopk> : select_long_kernel<kModeQsa>;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSlSmem) != cudaSuccess)
        return QSA_ERR_CUDA;
      // clusters of 16 are beyond the portable size; without the opt-in the
      // 16-CTA plan is simply never taken
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        cudaGetLastError();
    }
    if (!set_attn_smem()) return QSA_ERR_CUDA;
    if (cudaFuncSetAttribute(select_fast_kernel<kModeTopk>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SfShared)) != cudaSuccess ||
        cudaFuncSetAttribute(select_fast_kernel<kModeQsa>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SfShared)) != cudaSuccess)
      return QSA_ERR_CUDA;
    if (!set_mma_smem<false>() || !set_mma_smem<true>()) return QSA_ERR_CUDA;
    if (cudaFuncSetAttribute(select_rows_kernel<kModeTopk>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SrSmem)) != cudaSuccess ||
        cudaFuncSetAttribute(select_rows_kernel<kModeQsa>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(SrSmem)) != cudaSuccess)
      return QSA_ERR_CUDA;
    for (int e = 1; e <= 4; ++e) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1u << e, 1, 1);
      cfg.blockDim = dim3(kSlThreads, 1, 1);
      cfg.dynamicSmemBytes = kSlSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 1u << e;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, select_long_kernel<kModeTopk>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        nc = 0;
      }
      d.sl_clusters[e] = nc;
    }
    d.ready = true;
  }
  *out = &d;
  return QSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// RoPE turn fractions for one base, cached (the last few bases used).
// frac[i] = round(2^64 * base^(-2i/128) / (2 pi)).
std::mutex g_rope_mu;
struct RopeCacheEntry {
  double base = 0.0;
  RopeTurns turns;
};
RopeCacheEntry g_rope_cache[4];
int g_rope_next = 0;

RopeTurns rope_turns(double base) {
  std::lock_guard<std::mutex> lk(g_rope_mu);
  for (const RopeCacheEntry& e : g_rope_cache)
    if (e.base == base) return e.turns;
  RopeCacheEntry& e = g_rope_cache[g_rope_next];
  g_rope_next = (g_rope_next + 1) % 4;
  e.base = base;
  for (int i = 0; i < kDim / 2; ++i) {
    const double turns = std::pow(base, -2.0 * (double)i / (double)kDim) * 0.15915494309189533577;
    e.turns.frac[i] = (uint64_t)std::llround(std::ldexp(turns, 62)) << 2;  // turns < 1/4
  }
  return e.turns;
}

// Launch with programmatic stream serialisation: the grid may become
// resident before the previous kernel on the stream finishes; every kernel
// launched this way executes griddepcontrol.wait before reading its inputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

qsa_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}

// Shared-memory layout of one selection CTA for rows of up to n_max
// candidates: resident rows (<= kSelResidentCap) live in shared memory, longer
// rows stream through the bulk-copy ring.
void plan_select(SelectArgs& a) {
  a.pt_cap = kSelPtStage;
  if (a.n_max <= kRsMaxRow) {
    // resident kernel: [fixed][keys, whole chunks of 4096][page table]
    // [selected][candidate keys][candidate indices]
    a.resident = 2;
    int off = kRsFixedBytes;
    a.off_row = off;
    off += ((a.n_max + kRsChunk - 1) / kRsChunk) * kRsChunk * 4;
    a.off_pt = off;
    off += a.pt_cap * 4;
    a.off_sel = off;
    off += ((a.k + 3) & ~3) * 4;
    int cap = ((kRsMaxSmem - off) / 8) & ~3;
    if (cap > kRsListMax) cap = kRsListMax;
    a.list_cap = cap;
    a.off_lkey = off;
    off += cap * 4;
    a.off_list = off;
    return;
  }
  a.resident = a.n_max <= kSelResidentCap;
  a.list_cap = kSelListCap;
  int off = kSelFixedBytes;
  a.off_pt = off;
  off += a.pt_cap * 4;
  a.off_list = off;
  off += a.list_cap * 4;
  a.off_lkey = off;
  off += a.list_cap * 4;
  a.off_row = off;
}

size_t select_smem_bytes(const SelectArgs& a) {
  if (a.resident == 2) return (size_t)a.off_list + (size_t)a.list_cap * 4;
  const size_t row = a.resident ? (size_t)((a.n_max + 3) & ~3) * 4 : (size_t)kSelRing * kSelPiece * 4;
  return (size_t)a.off_row + row;
}

// Cluster selection for launches with few rows: 8 CTAs per row when
// rows * 8 <= SMs.  Returns QSA_ERR_UNSUPPORTED when the single-CTA kernels
// should run instead.
template <int kMode>
qsa_status launch_select_cluster(const SelectArgs& args, bool pdl, int sm_count, cudaStream_t stream) {
  if (args.n_max > kRsMaxRow) return QSA_ERR_UNSUPPORTED;
  // one cluster of 8 CTAs per row when the rows leave that many SMs; with
  // more rows the single-CTA kernels keep the GPU busy as well
  const int C = 8;
  if ((int64_t)args.n_rows * C > sm_count) return QSA_ERR_UNSUPPORTED;
  SelectArgs a = args;
  int off = kScFixedBytes;
  a.list_cap = kScListCap;
  a.off_lkey = off;
  off += kScListCap * 4;
  a.off_list = off;
  off += kScListCap * 4;
  a.off_pt = off;
  a.pt_cap = kSelPtStage;
  off += kSelPtStage * 4;
  a.off_sel = off;
  off += ((a.k + 3) & ~3) * 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.n_rows * C), 1, 1);
  cfg.blockDim = dim3(kScThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)off;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = (unsigned)C;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e;
  e = cudaLaunchKernelEx(&cfg, select_cluster_kernel<kMode, 4>, a);  // slices of <= 4096 = 1024 x 4
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  return QSA_OK;
}

// Long rows on clusters of C CTAs (one cluster per row, `clusters` of them).
template <int kMode>
qsa_status launch_select_long_c(const SelectArgs& args, int C, int64_t clusters, bool pdl, cudaStream_t stream) {
  SelectArgs a = args;
  const int64_t S = (((int64_t)a.n_max + C - 1) / C + 3) & ~int64_t(3);
  const int64_t cap = ((kSlSmem - kSlFixedBytes) / 4) & ~3;
  a.list_cap = (int32_t)std::min(S, cap);  // slice entries kept in shared memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * C), 1, 1);
  cfg.blockDim = dim3(kSlThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)kSlFixedBytes + (size_t)a.list_cap * 4;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = (unsigned)C;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, select_long_kernel<kMode>, a) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  return QSA_OK;
}

// Long rows: a cluster of C CTAs per row, C the largest of 16, 8, 4, 2 with
// rows * C <= SMs (and such clusters schedulable).  QSA_ERR_UNSUPPORTED: one
// CTA per row (select_kernel) instead.
template <int kMode>
qsa_status launch_select_long(const SelectArgs& args, bool pdl, cudaStream_t stream) {
  if (args.n_max <= kRsMaxRow) return QSA_ERR_UNSUPPORTED;
  DeviceInfo* d = nullptr;
  if (qsa_status st = device_info(&d)) return st;
  int e = 4;
  while (e >= 1 && ((int64_t)args.n_rows << e > d->sm_count || d->sl_clusters[e] < 1)) --e;
  if (e < 1) return QSA_ERR_UNSUPPORTED;
  return launch_select_long_c<kMode>(args, 1 << e, args.n_rows, pdl, stream);
}

// More than two rows per SM, rows of up to kSrMaxRow entries: one 256-thread
// CTA per row, four per SM (select_rows_kernel).  Measured: a prefill chunk
// of 4096 rows 396 -> 274 us (three per SM) -> 244 us (four); a batch of 192 verify rows still runs the step
// faster on the 1024-thread kernel (72.3 against 74.5 us).
template <int kMode>
qsa_status launch_select_rows(const SelectArgs& a, bool pdl, cudaStream_t stream, int sm_count) {
  if (a.n_max > kSrMaxRow || sm_count <= 0 || a.n_rows <= 2 * sm_count) return QSA_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_rows, 1, 1);
  cfg.blockDim = dim3(kSrThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(SrSmem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, select_rows_kernel<kMode>, a) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  return QSA_OK;
}

// Rows of up to kSfMaxRow entries with k <= kSfMaxK: one 1024-thread CTA per
// row holding the row in registers (select_fast_kernel).
template <int kMode>
qsa_status launch_select_fast(const SelectArgs& a, bool pdl, cudaStream_t stream) {
  if (a.n_max > kSfMaxRow || a.k > kSfMaxK) return QSA_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_rows, 1, 1);
  cfg.blockDim = dim3(kSfThreads, 1, 1);
  cfg.dynamicSmemBytes = sizeof(SfShared);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, select_fast_kernel<kMode>, a) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  return QSA_OK;
}

// Bytes of the device row plan for n_rows rows (plan_rows_kernel).
size_t plan_bytes(int32_t n_rows) { return (((size_t)4 + 2 * (size_t)n_rows) * 4 + 255) & ~(size_t)255; }

// Whether a launch of these rows takes the device plan: some rows may be long
// (more than kRsMaxRow candidates) and there are too many rows to give each a
// cluster, so the host bound alone would send every row, short or long, to
// one streaming CTA.
bool wants_plan(int32_t n_rows, int32_t n_max, int sm_count) {
  return n_max > kRsMaxRow && (int64_t)n_rows * 2 > sm_count;
}

template <int kMode>
qsa_status launch_select(const SelectArgs& a, bool pdl, cudaStream_t stream, int sm_count = 0);

// Rows split by length class on the device (plan_rows_kernel, one CTA): the
// long rows (more than kRsMaxRow candidates) on clusters sized from their
// count, the short ones one CTA each.  The cluster size is a launch
// attribute, so the long class is launched once per size the plan can pick
// (16 or 2 CTAs per row, and the one-CTA streaming kernel); the launches the
// plan did not pick wait for it and exit.  The long launches follow the plan
// on the caller's stream (each waits for its predecessor, the plan for the
// previous grid: the scorer in the fused call); the short class runs on a
// side stream from the plan's completion, beside them, and the caller's
// stream waits for it before the call returns.
template <int kMode>
qsa_status launch_select_planned(const SelectArgs& args, int32_t* plan, bool pdl, cudaStream_t stream,
                                 DeviceInfo* d) {
  const int sm = d->sm_count;
  PlanArgs p{};
  p.n_valid = kMode == kModeTopk ? args.n_valid : nullptr;
  p.row_len = kMode == kModeQsa ? args.row_len : nullptr;
  p.n_rows = args.n_rows;
  p.n_max = args.n_max;
  p.cut = kRsMaxRow;
  // Sizes the plan may pick: 16 (a few long rows, e.g. one of 1M) and 2
  // (many); every size is one more launch, and each launch the plan does not
  // pick still costs a dependent-launch hop, so the sizes are few.
  for (int e : {1, 4})
    if (d->sl_clusters[e] >= 1) p.c_mask |= 1 << e;
  p.sm_count = sm;
  p.plan = plan;
  if (pdl) {
    if (launch_pdl(plan_rows_kernel, dim3(1), dim3(1024), 0, stream, p) != cudaSuccess) {
      cudaGetLastError();
      return QSA_ERR_CUDA;
    }
  } else {
    plan_rows_kernel<<<1, 1024, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return QSA_ERR_CUDA;
  }
  // short class: rows of at most kRsMaxRow candidates, one CTA each, on the
  // side stream once the plan is complete, so that it runs beside the long
  // class instead of after it; the caller's stream waits for both at the end
  cudaEvent_t planned = nullptr, short_done = nullptr;
  if (cudaEventCreateWithFlags(&planned, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&short_done, cudaEventDisableTiming) != cudaSuccess) {
    if (planned) cudaEventDestroy(planned);
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  struct EventGuard {  // destruction is deferred by CUDA until the events complete
    cudaEvent_t a, b;
    ~EventGuard() {
      cudaEventDestroy(a);
      cudaEventDestroy(b);
    }
  } guard{planned, short_done};
  SelectArgs S = args;
  S.plan = plan;
  S.row_list = plan + 4 + args.n_rows;
  S.count_at = 2;
  S.plan_c = 0;
  S.wait_primary = 0;  // stream order: the plan (and what it waited for) is complete
  S.n_max = kRsMaxRow;
  plan_select(S);
  if (cudaEventRecord(planned, stream) != cudaSuccess || cudaStreamWaitEvent(d->side, planned, 0) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  if (qsa_status st = launch_select<kMode>(S, false, d->side, sm)) return st;
  if (cudaEventRecord(short_done, d->side) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  // long class: the sizes the plan can pick for 1 <= n_long <= n_rows
  SelectArgs L = args;
  L.plan = plan;
  L.row_list = plan + 4;
  L.count_at = 0;
  L.wait_primary = 1;
  int64_t prev_hi = 0;  // rows a larger schedulable size takes
  for (int e = 4; e >= 1; --e) {
    if (!(p.c_mask >> e & 1)) continue;
    const int c = 1 << e;
    const int64_t hi = sm / c;  // the plan picks c for prev_hi < n_long <= hi
    if (prev_hi < args.n_rows && prev_hi < hi) {
      L.plan_c = c;
      if (qsa_status st = launch_select_long_c<kMode>(L, c, std::min<int64_t>(args.n_rows, hi), true, stream))
        return st;
    }
    prev_hi = std::max(prev_hi, hi);
  }
  if (prev_hi < args.n_rows) {  // one streaming CTA per long row
    L.plan_c = 1;
    plan_select(L);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)args.n_rows, 1, 1);
    cfg.blockDim = dim3(kSelThreads, 1, 1);
    cfg.dynamicSmemBytes = select_smem_bytes(L);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, select_kernel<kMode>, L) != cudaSuccess) {
      cudaGetLastError();
      return QSA_ERR_CUDA;
    }
  }
  if (cudaStreamWaitEvent(stream, short_done, 0) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  return QSA_OK;
}

template <int kMode>
qsa_status launch_select(const SelectArgs& a, bool pdl, cudaStream_t stream, int sm_count) {
  if (a.n_rows == 0) return QSA_OK;
  {
    const qsa_status st = launch_select_long<kMode>(a, pdl, stream);
    if (st != QSA_ERR_UNSUPPORTED) return st;
  }
  {
    const qsa_status st = launch_select_rows<kMode>(a, pdl, stream, sm_count);
    if (st != QSA_ERR_UNSUPPORTED) return st;
  }
  {
    const qsa_status st = launch_select_fast<kMode>(a, pdl, stream);
    if (st != QSA_ERR_UNSUPPORTED) return st;
  }
  if (sm_count > 0) {
    const qsa_status st = launch_select_cluster<kMode>(a, pdl, sm_count, stream);
    if (st != QSA_ERR_UNSUPPORTED) return st;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_rows, 1, 1);
  cfg.blockDim = dim3(kSelThreads, 1, 1);
  cfg.dynamicSmemBytes = select_smem_bytes(a);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const cudaError_t e = a.resident == 2 ? cudaLaunchKernelEx(&cfg, select_resident_kernel<kMode>, a)
                                         : cudaLaunchKernelEx(&cfg, select_kernel<kMode>, a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  return QSA_OK;
}

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point
// (the library does not link libcuda directly).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The compressed-key pool for the TMA scorer, with the 128-byte swizzle.
// 4-D view (pool_rows a multiple of 8): [row / 8][K-half][row % 8][64 BF16],
// one box of box_rows / 8 groups covers a run of box_rows keys, both
// K-halves, landing as [group][K-half][8 rows][128 B].  2-D view otherwise:
// [pool_rows][128 BF16], one box of 64 x box_rows per K-half.
bool encode_pool_map(CUtensorMap* m, const void* pool, int64_t pool_rows, int box_rows, bool four_d) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  if (four_d) {
    const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(pool_rows / 8)};
    const cuuint64_t strides[3] = {(cuuint64_t)kDim * 2, 128, (cuuint64_t)kDim * 2 * 8};
    const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(box_rows / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)pool_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA scorer (pages whose compressed rows form whole 8-row swizzle atoms).
// Returns QSA_ERR_UNSUPPORTED when the layout does not allow it, so that the
// caller takes the cp.async kernel.
qsa_status launch_scores_tma(TcArgs t, int64_t n_kt, int64_t row_tiles, int32_t n_req, int sm_count,
                             cudaStream_t stream) {
  const int kpp = t.page_size / kBlock;
  int R = 0;
  for (int c = kTcM; c >= 8; c >>= 1)
    if (kpp % c == 0) {
      R = c;
      break;
    }
  if (R == 0 || t.pool_rows <= 0 || t.pool_rows > INT32_MAX) return QSA_ERR_UNSUPPORTED;
  CUtensorMap map;
  t.box4d = t.pool_rows % 8 == 0 ? 1 : 0;
  if (!encode_pool_map(&map, t.pool, t.pool_rows, R, t.box4d != 0)) {
    t.box4d = 0;
    if (!encode_pool_map(&map, t.pool, t.pool_rows, R, false)) return QSA_ERR_UNSUPPORTED;
  }
  t.box_rows = R;
  int cols = 32;
  while (cols < 2 * t.n_cols) cols *= 2;  // two accumulators
  t.tmem_cols = cols;
  // One CTA per SM with the whole key ring, or two per SM with half of it
  // each when that leaves fewer key tiles on the busiest SM: 32 verify
  // requests split 4 ways fill only 128 SMs (40 tiles each), split 9 ways
  // they fill all of them (at most 36 tiles per SM).  Key tiles per CTA:
  // about one wave of CTAs in total.
  const int64_t units = row_tiles * n_req;
  int per_sm = 1;
  int64_t x_ctas = std::max<int64_t>(1, std::min<int64_t>(n_kt, sm_count / units));
  if (units <= sm_count && 2 * t.tmem_cols <= 512) {  // two CTAs' accumulators fit the SM's TMEM
    const int64_t t1 = (n_kt + x_ctas - 1) / x_ctas;
    const int64_t x2 = std::max<int64_t>(1, std::min<int64_t>(n_kt, 2 * sm_count / units));
    const int64_t t2 = (n_kt + x2 - 1) / x2;
    const int64_t busy2 = units * ((n_kt + t2 - 1) / t2) > sm_count ? 2 * t2 : t2;
    if (busy2 < t1) {
      per_sm = 2;
      x_ctas = x2;
    }
  }
  t.tiles_per_cta = (int32_t)((n_kt + x_ctas - 1) / x_ctas);
  t.pt_cap = (int32_t)std::min<int64_t>(kTcPtStage, (int64_t)t.tiles_per_cta * kTcM / kpp + 2);
  const size_t fixed = 1024 + 2 * (size_t)t.n_cols * 128 + (2 * kTcMaxStages + 4) * 8 + sizeof(TmCtl) +
                       4 * (size_t)t.rows_per_tile + 4 * (size_t)t.pt_cap;
  const size_t budget = per_sm == 1 ? (size_t)kTcMaxSmem : (size_t)kTcMaxSmem / 2 - 1024;
  t.stages = (int)std::min<size_t>(kTcMaxStages, (budget - fixed) / (2 * kTcHalf));
  if (t.stages < 2) return QSA_ERR_UNSUPPORTED;
  const size_t smem = fixed + (size_t)t.stages * 2 * kTcHalf;
  // wide tiles (prefill) get 16 epilogue warps, narrow ones 8
  const bool wide = t.n_cols >= 128;
  const int threads = wide ? 32 * (2 + 16) : 32 * (2 + 8);
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, wide ? score_tc_kernel<16> : score_tc_kernel<8>, threads,
                                                    smem) != cudaSuccess)
    return QSA_ERR_CUDA;
  if ((int64_t)occ * t.tmem_cols > 512) return QSA_ERR_UNSUPPORTED;
  dim3 grid((unsigned)((n_kt + t.tiles_per_cta - 1) / t.tiles_per_cta), (unsigned)row_tiles, (unsigned)n_req);
  if (launch_pdl(wide ? score_tc_kernel<16> : score_tc_kernel<8>, grid, dim3(threads), smem, stream, t, map) !=
      cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  return QSA_OK;
}

// Decode scorer on mma.sync (score_mma_kernel): requests of up to kSmMaxRows
// rows on pages holding a multiple of 8 compressed keys.  About one wave of
// CTAs (two per SM), at least one tile (16 BF16 or 32 FP8 keys) per warp.
template <int NT, bool kFp8>
qsa_status launch_scores_mma_nt(const ScoreArgs& s, int sm_count, cudaStream_t stream, int reserve) {
  const size_t smem = sm_smem_bytes(s.n_req, NT);
  // CTAs per SM, queried once (the query costs microseconds of host time on
  // every call otherwise): at the largest shared memory a launch can ask
  // for, so never more than fit for any request count (the register budget
  // caps it at kSmMinCtas anyway)
  static const int occ_max = [] {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, score_mma_kernel<NT, kFp8>, kSmThreads,
                                                      sm_smem_bytes(kSmMaxReq, NT)) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return o;
  }();
  if (occ_max <= 0) return QSA_ERR_CUDA;
  const int occ = occ_max;
  const int64_t nb_max = s.max_len / kBlock;
  const int64_t tiles_max = (int64_t)s.n_req * ((nb_max + sm_tile<NT, kFp8>() - 1) / sm_tile<NT, kFp8>());
  int64_t ctas =
      std::max<int64_t>(1, std::min<int64_t>((int64_t)std::max(occ, 1) * sm_count, (tiles_max + kSmWarps - 1) / kSmWarps));
  // A grid of about one CTA per SM leaves `reserve` SMs to the selection
  // launched after it, so that its CTAs become resident at once and read
  // their metadata and page-table entries while the scorer runs.
  if (reserve > 0 && ctas > sm_count - reserve && ctas <= sm_count + 2 * reserve)
    ctas = std::max<int64_t>(1, sm_count - reserve);
  if (launch_pdl(score_mma_kernel<NT, kFp8>, dim3((unsigned)ctas), dim3(kSmThreads), smem, stream, s) !=
      cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  return QSA_OK;
}

qsa_status launch_scores_mma(const ScoreArgs& s, int max_rows_per_req, int sm_count, cudaStream_t stream,
                             int reserve = 0) {
  const int64_t nb_max = s.max_len / kBlock;
  if (s.n_req == 0 || nb_max == 0 || max_rows_per_req <= 0) return QSA_OK;
  const int kpp = s.page_size / kBlock;
  if (kpp % 8 != 0 || max_rows_per_req > kSmMaxRows || s.n_req > kSmMaxReq || s.pool_rows <= 0 ||
      s.pool_rows > INT32_MAX || (int64_t)s.n_req * ((nb_max + kSmTile - 1) / kSmTile) > INT32_MAX)
    return QSA_ERR_UNSUPPORTED;
  qsa_status st;
  const bool fp8 = s.pool8 != nullptr;
  switch ((max_rows_per_req + 1) / 2) {
    case 1: st = fp8 ? launch_scores_mma_nt<1, true>(s, sm_count, stream, reserve) : launch_scores_mma_nt<1, false>(s, sm_count, stream, reserve); break;
    case 2: st = fp8 ? launch_scores_mma_nt<2, true>(s, sm_count, stream, reserve) : launch_scores_mma_nt<2, false>(s, sm_count, stream, reserve); break;
    case 3: st = fp8 ? launch_scores_mma_nt<3, true>(s, sm_count, stream, reserve) : launch_scores_mma_nt<3, false>(s, sm_count, stream, reserve); break;
    default: st = fp8 ? launch_scores_mma_nt<4, true>(s, sm_count, stream, reserve) : launch_scores_mma_nt<4, false>(s, sm_count, stream, reserve); break;
  }
  if (st == QSA_OK && s.n_fill > 0) {
    fill_neginf_kernel<<<(unsigned)s.n_rows, 256, 0, stream>>>(s.row_len, s.max_len, s.scores, s.ld_scores,
                                                              s.n_fill);
    return launch_status();
  }
  return st;
}

// Scorer dispatch: the mma.sync decode kernel for requests of up to 8 rows
// on pages of a multiple of 32 tokens, the per-request tensor-core kernel for
// requests with more rows (or several rows on smaller pages), the CUDA-core
// streaming kernel otherwise.
qsa_status launch_scores(ScoreArgs s, int sm_count, cudaStream_t stream);
qsa_status launch_scores_tc(const ScoreArgs& s, int max_rows_per_req, int sm_count, cudaStream_t stream);
qsa_status launch_scorer(const ScoreArgs& s, int max_rows_per_req, int sm_count, cudaStream_t stream,
                         int reserve = 0) {
  const qsa_status m = launch_scores_mma(s, max_rows_per_req, sm_count, stream, reserve);
  if (m != QSA_ERR_UNSUPPORTED || s.pool8 != nullptr) return m;  // FP8 keys: the mma.sync scorer only
  return max_rows_per_req >= kTcMinRows ? launch_scores_tc(s, max_rows_per_req, sm_count, stream)
                                        : launch_scores(s, sm_count, stream);
}

// Tensor-core scorer for requests with several rows: tiles of 128 keys x up
// to 64 rows (N = 4 * rows, multiple of 16), a group of key tiles per CTA
// when rows are plentiful (prefill), one otherwise (decode verify).  The
// dynamic shared memory is raised if needed so that the CTAs resident on an
// SM never ask for more than the 512 TMEM columns.
qsa_status launch_scores_tc(const ScoreArgs& s, int max_rows_per_req, int sm_count,
                            cudaStream_t stream) {
  const int64_t nb_max = s.max_len / kBlock;
  if (s.n_req == 0 || nb_max == 0 || max_rows_per_req <= 0) return QSA_OK;
  TcArgs t{};
  t.q = s.q;
  t.pool = s.pool;
  t.pool_rows = s.pool_rows;
  t.n_req = s.n_req;
  t.req_row_start = s.req_row_start;
  t.n_rows = s.n_rows;
  t.row_len = s.row_len;
  t.max_len = s.max_len;
  t.page_table = s.page_table;
  t.ld_pt = s.ld_pt;
  t.page_size = s.page_size;
  t.scores = s.scores;
  t.ld_scores = s.ld_scores;
  const int64_t n_kt = (nb_max + kTcM - 1) / kTcM;
  int rpt = std::min(kTcMaxRowsPerTile, max_rows_per_req);
  if (max_rows_per_req > kTcMaxRowsPerTile && sm_count > 0) {
    // Many rows (a prefill chunk): the tile height whose CTAs (row tiles x
    // key-range splits) fill one wave with the least work per CTA, i.e. key
    // tiles x (MMA columns + a fixed share per tile).  4096 rows on 152
    // SMs: 56-row tiles, 74 x 2 CTAs, instead of 64-row tiles on 128 SMs.
    int64_t best = INT64_MAX;
    for (int r = kTcMaxRowsPerTile; r >= 8; --r) {
      const int64_t rt = (max_rows_per_req + r - 1) / r;
      if (rt * s.n_req > sm_count) break;  // smaller r: more row tiles still
      const int64_t x = std::min<int64_t>(n_kt, sm_count / (rt * s.n_req));
      const int64_t cost = ((n_kt + x - 1) / x) * ((((int64_t)4 * r + 15) & ~15) + 32);
      if (cost < best) {
        best = cost;
        rpt = r;
      }
    }
  }
  t.rows_per_tile = rpt;
  t.n_cols = ((4 * t.rows_per_tile) + 15) & ~15;
  int cols = 32;
  while (cols < 2 * t.n_cols) cols *= 2;  // two accumulators
  t.tmem_cols = cols;
  t.trigger_dependents = s.trigger_dependents;
  t.new_pos = s.new_pos;
  t.head_gates = s.head_gates;
  const int64_t row_tiles = (max_rows_per_req + t.rows_per_tile - 1) / t.rows_per_tile;
  if (row_tiles > 65535) return QSA_ERR_UNSUPPORTED;
  qsa_status tma = launch_scores_tma(t, n_kt, row_tiles, s.n_req, sm_count, stream);
  if (tma == QSA_OK && s.n_fill > 0) {
    fill_neginf_kernel<<<(unsigned)s.n_rows, 256, 0, stream>>>(s.row_len, s.max_len, s.scores, s.ld_scores,
                                                              s.n_fill);
    return launch_status();
  }
  if (tma != QSA_ERR_UNSUPPORTED) return tma;
  // key-ring stages: as many 32 KB stages as fit beside B and the rest
  const size_t fixed = 1024 + 2 * (size_t)t.n_cols * 128 + 32 + 4 * (size_t)t.rows_per_tile +
                       4 * (size_t)kTcPtStage;
  t.stages = (int)std::min<size_t>(kTcMaxStages, ((size_t)kTcMaxSmem - fixed) / (2 * kTcHalf));
  if (t.stages < 3) return QSA_ERR_UNSUPPORTED;
  const size_t smem = fixed + (size_t)t.stages * 2 * kTcHalf;
  // resident CTAs per SM (shared memory bound; with the 4-stage ring this is
  // one) must never ask for more than the 512 TMEM columns
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, score_tc_cpasync_kernel, kTcThreads, smem) !=
      cudaSuccess)
    return QSA_ERR_CUDA;
  if ((int64_t)occ * t.tmem_cols > 512) return QSA_ERR_UNSUPPORTED;
  // Key tiles per CTA: about one wave of CTAs in total, consecutive tiles of
  // a CTA double-buffered (a lone CTA per tile pays its set-up every time).
  const int64_t wave = (int64_t)std::max(occ, 1) * sm_count;
  const int64_t x_ctas = std::max<int64_t>(1, std::min<int64_t>(n_kt, wave / (row_tiles * s.n_req)));
  t.tiles_per_cta = (int32_t)((n_kt + x_ctas - 1) / x_ctas);
  dim3 grid((unsigned)((n_kt + t.tiles_per_cta - 1) / t.tiles_per_cta), (unsigned)row_tiles,
            (unsigned)s.n_req);
  if (launch_pdl(score_tc_cpasync_kernel, grid, dim3(kTcThreads), smem, stream, t) != cudaSuccess) {
    cudaGetLastError();
    return QSA_ERR_CUDA;
  }
  if (s.n_fill > 0) {
    fill_neginf_kernel<<<(unsigned)s.n_rows, 256, 0, stream>>>(s.row_len, s.max_len, s.scores, s.ld_scores,
                                                              s.n_fill);
    return launch_status();
  }
  return QSA_OK;
}

qsa_status check_rows(int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                      const int32_t* row_len, int32_t max_len) {
  if (n_req < 0 || n_rows < 0 || max_len < 0) return QSA_ERR_INVALID_ARG;
  if (n_rows > 0 && (n_req < 1 || !req_row_start || !row_len)) return QSA_ERR_INVALID_ARG;
  if (n_req > 65535) return QSA_ERR_UNSUPPORTED;
  return QSA_OK;
}

qsa_status check_paging(const int32_t* page_table, int64_t ld_pt, int32_t page_size,
                        int32_t max_len) {
  if (!page_table || page_size <= 0 || ld_pt < 0) return QSA_ERR_INVALID_ARG;
  if (page_size % kBlock != 0) return QSA_ERR_UNSUPPORTED;
  if (max_len > 0 && (int64_t)(max_len - 1) / page_size >= ld_pt) return QSA_ERR_INVALID_ARG;
  return QSA_OK;
}

// Persistent scorer: two CTAs per SM walk balanced ranges of 128-block
// tiles.  Requests are handled in windows of at most kScoreMaxReq per launch.
qsa_status launch_scores(ScoreArgs s, int sm_count, cudaStream_t stream) {
  const int64_t nb_max = s.max_len / kBlock;
  const int64_t cols = std::max<int64_t>(nb_max, s.n_fill);
  if (s.n_req == 0 || cols == 0) return QSA_OK;
  const int32_t n_req = s.n_req;
  const int32_t* rrs = s.req_row_start;
  const int32_t* pt = s.page_table;
  const int32_t trigger = s.trigger_dependents;
  for (int32_t r0 = 0; r0 < n_req; r0 += kScoreMaxReq) {
    s.n_req = std::min<int32_t>(kScoreMaxReq, n_req - r0);
    // only the last launch may let the dependent selection start early
    s.trigger_dependents = trigger && (r0 + kScoreMaxReq >= n_req);
    s.req_row_start = rrs + r0;
    s.page_table = pt + (int64_t)r0 * s.ld_pt;
    const int64_t tiles = (int64_t)s.n_req * ((cols + kScoreTile - 1) / kScoreTile);
    if (tiles > INT32_MAX) return QSA_ERR_UNSUPPORTED;
    const int64_t grid = std::min<int64_t>(tiles, 2 * (int64_t)sm_count);
    if (launch_pdl(score_decode_kernel, dim3((unsigned)grid), dim3(kScoreThreads), kScoreSmem, stream, s) !=
        cudaSuccess) {
      cudaGetLastError();
      return QSA_ERR_CUDA;
    }
  }
  return QSA_OK;
}

template <int G, int D>
qsa_status launch_attn_gd(const SaArgs& a, cudaStream_t stream) {
  dim3 grid((unsigned)a.n_split, (unsigned)a.h_kv, (unsigned)a.n_rows);
  sparse_attn_kernel<G, D><<<grid, kSaThreads, sizeof(SaSmem<G, D>), stream>>>(a);
  if (cudaGetLastError() != cudaSuccess) return QSA_ERR_CUDA;
  if (a.n_split > 1) {
    if (launch_pdl(sparse_attn_merge_kernel<D>, dim3((unsigned)((int64_t)a.n_rows * a.h_q)), dim3(D), 0,
                   stream, a) != cudaSuccess) {
      cudaGetLastError();
      return QSA_ERR_CUDA;
    }
  }
  return QSA_OK;
}

qsa_status launch_attn(const SaArgs& a, int group, int d, cudaStream_t stream) {
  if (d == 128) {
    switch (group) {
      case 1: return launch_attn_gd<1, 128>(a, stream);
      case 2: return launch_attn_gd<2, 128>(a, stream);
      case 4: return launch_attn_gd<4, 128>(a, stream);
      case 8: return launch_attn_gd<8, 128>(a, stream);
      case 16: return launch_attn_gd<16, 128>(a, stream);
      default: return QSA_ERR_UNSUPPORTED;
    }
  }
  if (d == 256) {
    switch (group) {
      case 1: return launch_attn_gd<1, 256>(a, stream);
      case 2: return launch_attn_gd<2, 256>(a, stream);
      case 4: return launch_attn_gd<4, 256>(a, stream);
      case 8: return launch_attn_gd<8, 256>(a, stream);
      default: return QSA_ERR_UNSUPPORTED;
    }
  }
  return QSA_ERR_UNSUPPORTED;
}

bool attn_shape_ok(int32_t h_q, int32_t h_kv, int32_t d) {
  if (h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0) return false;
  const int group = h_q / h_kv;
  const bool pow2 = (group & (group - 1)) == 0;
  return pow2 && ((d == 128 && group <= 16) || (d == 256 && group <= 8));
}

}  // namespace

extern "C" {

const char* qsa_status_string(qsa_status s) {
  switch (s) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument";
    case QSA_ERR_UNSUPPORTED: return "unsupported size or layout";
    case QSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case QSA_ERR_CUDA: return "CUDA error";
    case QSA_ERR_DEVICE_FAULT: return "device-side check failed";
    default: return "unknown status";
  }
}

int qsa_version(void) { return 100; }

qsa_status qsa_device_status(void* stream, int clear, uint32_t* h_bits) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned bits = 0;
  if (cudaMemcpyFromSymbolAsync(&bits, g_fault_word, sizeof(bits), 0, cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return QSA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return QSA_ERR_CUDA;
  if (clear && bits) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbolAsync(g_fault_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return QSA_ERR_CUDA;
  }
  if (h_bits) *h_bits = bits;
  return bits ? QSA_ERR_DEVICE_FAULT : QSA_OK;
}

qsa_status qsa_compress_keys(const void* raw, const int32_t* block_req, const int32_t* block_id,
                             int64_t n_blocks, int32_t n_req, const int32_t* page_table,
                             int64_t ld_pt, int32_t page_size, double rope_base, void* pool,
                             int64_t pool_rows, void* stream) {
  if (n_blocks < 0 || pool_rows < 0) return QSA_ERR_INVALID_ARG;
  if (n_blocks == 0) return QSA_OK;
  if (!raw || !block_id || !pool || !aligned16(raw) || !aligned16(pool)) return QSA_ERR_INVALID_ARG;
  if (!(rope_base > 0.0)) return QSA_ERR_INVALID_ARG;
  if (page_table) {
    if (!block_req || n_req < 1 || ld_pt < 1 || page_size <= 0) return QSA_ERR_INVALID_ARG;
    if (page_size % kBlock != 0) return QSA_ERR_UNSUPPORTED;
  }
  DeviceInfo* d = nullptr;
  if (qsa_status st = device_info(&d)) return st;
  CompressArgs a{static_cast<const __nv_bfloat16*>(raw), block_req, block_id, n_blocks, n_req,
                 page_table, ld_pt, page_size, rope_base, static_cast<__nv_bfloat16*>(pool),
                 pool_rows};
  const int64_t per_cta = kCompressThreads / kCompressLanes;
  const int64_t grid = std::min<int64_t>((n_blocks + per_cta - 1) / per_cta, (int64_t)d->sm_count * 8);
  compress_keys_kernel<<<(unsigned)grid, kCompressThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      a, rope_turns(rope_base));
  return launch_status();
}

qsa_status qsa_append_keys(const void* new_keys, const int32_t* req_tok_start, const int32_t* req_first_pos,
                           int32_t n_req, void* ring, const int32_t* page_table, int64_t ld_pt,
                           int32_t page_size, double rope_base, void* pool, int64_t pool_rows, void* stream) {
  if (n_req < 0 || pool_rows < 0 || ld_pt < 0) return QSA_ERR_INVALID_ARG;
  if (n_req == 0) return QSA_OK;
  if (n_req > INT32_MAX / 2) return QSA_ERR_UNSUPPORTED;
  if (!req_tok_start || !req_first_pos || !ring || !page_table || !pool || page_size <= 0 ||
      !(rope_base > 0.0) || !std::isfinite(rope_base))
    return QSA_ERR_INVALID_ARG;
  if (page_size % kBlock != 0) return QSA_ERR_UNSUPPORTED;
  if (!aligned16(ring) || !aligned16(pool) || (new_keys && !aligned16(new_keys))) return QSA_ERR_INVALID_ARG;
  AppendArgs a{static_cast<const __nv_bfloat16*>(new_keys), req_tok_start, req_first_pos, n_req,
               static_cast<__nv_bfloat16*>(ring), page_table, ld_pt, page_size,
               static_cast<__nv_bfloat16*>(pool), pool_rows};
  const RopeTurns turns = rope_turns(rope_base);
  append_keys_kernel<<<(unsigned)n_req, kAppendThreads, 0, static_cast<cudaStream_t>(stream)>>>(a, turns);
  return launch_status();
}

qsa_status qsa_index_scores(const void* q, const void* pool, int64_t pool_rows, int32_t n_req,
                            const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                            int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table,
                            int64_t ld_pt, int32_t page_size, float* scores, int64_t ld_scores,
                            int64_t n_fill, void* stream) {
  return qsa_index_scores_gated(q, nullptr, pool, pool_rows, n_req, req_row_start, n_rows, row_len, max_len,
                                max_rows_per_req, page_table, ld_pt, page_size, scores, ld_scores, n_fill, stream);
}

qsa_status qsa_index_scores_gated(const void* q, const float* head_gates, const void* pool, int64_t pool_rows,
                                  int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                  const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
                                  const int32_t* page_table, int64_t ld_pt, int32_t page_size, float* scores,
                                  int64_t ld_scores, int64_t n_fill, void* stream) {
  if (qsa_status st = check_rows(n_req, req_row_start, n_rows, row_len, max_len)) return st;
  if (n_rows == 0) return QSA_OK;
  if (qsa_status st = check_paging(page_table, ld_pt, page_size, max_len)) return st;
  if (!q || !pool || !scores || pool_rows < 0 || n_fill < 0) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned4(scores)) return QSA_ERR_INVALID_ARG;
  if (head_gates && !aligned16(head_gates)) return QSA_ERR_INVALID_ARG;
  if (ld_scores < std::max<int64_t>(max_len / kBlock, n_fill)) return QSA_ERR_INVALID_ARG;
  DeviceInfo* d = nullptr;
  if (qsa_status st = device_info(&d)) return st;
  ScoreArgs s{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(pool),
              pool_rows, n_req, req_row_start, n_rows, row_len, max_len, page_table, ld_pt,
              page_size, scores, ld_scores, n_fill, 0};
  s.head_gates = head_gates;
  return launch_scorer(s, max_rows_per_req, d->sm_count, static_cast<cudaStream_t>(stream));
}

size_t topk_select_workspace_size(int32_t n_rows, int32_t n_max, int32_t k) {
  (void)k;
  // the device row plan when rows may exceed the single-CTA length
  return (n_rows > 0 && n_max > kRsMaxRow) ? plan_bytes(n_rows) : 0;
}

qsa_status topk_select(const float* scores, int64_t ld, const int32_t* n_valid, int32_t n_rows,
                       int32_t n_max, int32_t k, const int32_t* page_table, int64_t ld_pt,
                       const int32_t* row_req, int32_t page_size, int32_t* out_idx,
                       int32_t* out_slots, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_rows < 0 || n_max < 0 || ld < 0) return QSA_ERR_INVALID_ARG;
  if (k < 1 || k > kMaxK) return QSA_ERR_UNSUPPORTED;
  if (n_rows == 0) return QSA_OK;
  if (!out_idx || (n_max > 0 && !scores) || n_max > ld) return QSA_ERR_INVALID_ARG;
  if (out_slots && (!page_table || page_size <= 0 || ld_pt < 1)) return QSA_ERR_INVALID_ARG;
  if (scores && !aligned4(scores)) return QSA_ERR_INVALID_ARG;
  DeviceInfo* d = nullptr;
  if (qsa_status st = device_info(&d)) return st;
  SelectArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.n_rows = n_rows;
  a.k = k;
  a.n_max = n_max;
  plan_select(a);
  a.vec_ok = aligned16(scores) && (ld % 4 == 0);
  a.wait_primary = 0;
  a.n_valid = n_valid;
  a.row_req = row_req;
  a.out_idx = out_idx;
  a.out_slots = out_slots;
  a.page_table = page_table;
  a.ld_pt = ld_pt;
  a.page_size = page_size > 0 ? page_size : 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (workspace && aligned4(workspace) && workspace_bytes >= plan_bytes(n_rows) &&
      wants_plan(n_rows, n_max, d->sm_count))
    return launch_select_planned<kModeTopk>(a, static_cast<int32_t*>(workspace), false, st, d);
  return launch_select<kModeTopk>(a, false, st, d->sm_count);
}

qsa_status qsa_expand_slots(const int32_t* sel_blocks, int32_t k_blk, int32_t n_req,
                            const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                            const int32_t* page_table, int64_t ld_pt, int32_t page_size,
                            int32_t* out_pos, int32_t* out_slots, void* stream) {
  if (k_blk < 1 || k_blk > kMaxK) return QSA_ERR_UNSUPPORTED;
  if (qsa_status st = check_rows(n_req, req_row_start, n_rows, row_len, 0)) return st;
  if (n_rows == 0) return QSA_OK;
  if (!sel_blocks || !out_slots || !page_table || ld_pt < 1 || page_size <= 0)
    return QSA_ERR_INVALID_ARG;
  if (page_size % kBlock != 0) return QSA_ERR_UNSUPPORTED;
  ExpandArgs a{sel_blocks, k_blk, n_req, req_row_start, n_rows, row_len, page_table, ld_pt,
               page_size, out_pos, out_slots};
  expand_kernel<<<(unsigned)n_rows, kExpThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

qsa_status qsa_indexshare_slots(const int32_t* cap_blocks, const int32_t* cap_len, int32_t n_cap,
                               const int32_t* cap_row, int32_t k_blk, int32_t n_extra, int32_t n_req,
                               const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                               const int32_t* page_table, int64_t ld_pt, int32_t page_size,
                               int32_t* out_pos, int32_t* out_slots, void* stream) {
  if (k_blk < 1 || k_blk > kMaxK) return QSA_ERR_UNSUPPORTED;
  if (n_extra < 0 || n_cap < 0) return QSA_ERR_INVALID_ARG;
  if (n_extra > kMaxShareExtra) return QSA_ERR_UNSUPPORTED;
  if (qsa_status st = check_rows(n_req, req_row_start, n_rows, row_len, 0)) return st;
  if (n_rows == 0) return QSA_OK;
  if (!cap_row || !out_slots || !page_table || ld_pt < 1 || page_size <= 0) return QSA_ERR_INVALID_ARG;
  if (n_cap > 0 && (!cap_blocks || !cap_len)) return QSA_ERR_INVALID_ARG;
  if (page_size % kBlock != 0) return QSA_ERR_UNSUPPORTED;
  ShareArgs a{cap_blocks, cap_len, n_cap, cap_row, k_blk, n_extra, n_req, req_row_start, n_rows,
              row_len, page_table, ld_pt, page_size, out_pos, out_slots};
  indexshare_kernel<<<(unsigned)n_rows, kExpThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

size_t qsa_sparse_attn_workspace_size(int32_t n_rows, int32_t h_q, int32_t head_dim, int32_t n_idx) {
  if (n_rows <= 0 || h_q <= 0 || head_dim <= 0 || n_idx <= kSaMaxChunk) return 0;
  const int64_t n_split = ((int64_t)n_idx + kSaMinChunk - 1) / kSaMinChunk;
  return (size_t)((int64_t)n_rows * h_q * n_split * (head_dim + 2) * 4) + 256;
}

qsa_status qsa_sparse_attn(const void* q, const void* k_cache, const void* v_cache, int64_t n_slots,
                           int32_t n_rows, int32_t h_q, int32_t h_kv, int32_t head_dim,
                           const int32_t* slots, int64_t ld_slots, int32_t n_idx, float scale, float* out,
                           float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_rows < 0 || n_idx < 0 || n_slots < 0 || ld_slots < n_idx) return QSA_ERR_INVALID_ARG;
  if (!attn_shape_ok(h_q, h_kv, head_dim)) return QSA_ERR_UNSUPPORTED;
  if (n_rows == 0) return QSA_OK;
  if (n_rows > 65535 || h_kv > 65535) return QSA_ERR_UNSUPPORTED;
  if (!q || !out || (n_idx > 0 && (!k_cache || !v_cache || !slots))) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || (k_cache && !aligned16(k_cache)) || (v_cache && !aligned16(v_cache)) ||
      !aligned4(out) || (lse && !aligned4(lse)))
    return QSA_ERR_INVALID_ARG;
  const size_t ws_need = qsa_sparse_attn_workspace_size(n_rows, h_q, head_dim, n_idx);
  if (ws_need > 0 && (!workspace || workspace_bytes < ws_need)) return QSA_ERR_WORKSPACE_TOO_SMALL;
  if (ws_need > 0 && !aligned16(workspace)) return QSA_ERR_INVALID_ARG;
  DeviceInfo* d = nullptr;
  if (qsa_status st = device_info(&d)) return st;
  SaArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k_cache);
  a.v = static_cast<const uint16_t*>(v_cache);
  a.n_slots = n_slots;
  a.n_rows = n_rows;
  a.h_q = h_q;
  a.h_kv = h_kv;
  a.slots = slots;
  a.ld_slots = ld_slots;
  a.n_idx = n_idx;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  // entries per CTA: the largest of 256, 128, 64 that still gives two CTAs
  // per SM; rows of at most 256 entries take one CTA per (row, KV head)
  int chunk = kSaMaxChunk;
  const int64_t units = (int64_t)n_rows * h_kv;
  while (chunk > kSaMinChunk && units * (((int64_t)n_idx + chunk - 1) / chunk) < 2LL * d->sm_count) chunk >>= 1;
  if (n_idx <= kSaMaxChunk) chunk = kSaMaxChunk;
  a.chunk = chunk;
  a.n_split = (int32_t)std::max<int64_t>(1, ((int64_t)n_idx + chunk - 1) / chunk);
  if (a.n_split > 65535) return QSA_ERR_UNSUPPORTED;
  if (a.n_split > 1) a.part = static_cast<float*>(workspace);  // n_split <= the size query's split
  return launch_attn(a, h_q / h_kv, head_dim, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_select_blocks(const float* scores, int64_t ld_scores, int32_t n_req,
                             const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                             int32_t max_len, const int32_t* page_table, int64_t ld_pt,
                             int32_t page_size, int32_t k_blk, int32_t* out_blocks, int32_t* out_pos,
                             int32_t* out_slots, void* stream) {
  if (k_blk < 1 || k_blk > kMaxK) return QSA_ERR_UNSUPPORTED;
  if (qsa_status st = check_rows(n_req, req_row_start, n_rows, row_len, max_len)) return st;
  if (n_rows == 0) return QSA_OK;
  if (qsa_status st = check_paging(page_table, ld_pt, page_size, max_len)) return st;
  const int32_t nb_max = max_len / kBlock;
  if (!out_slots || (nb_max > 0 && !scores) || ld_scores < nb_max) return QSA_ERR_INVALID_ARG;
  if (scores && !aligned4(scores)) return QSA_ERR_INVALID_ARG;
  DeviceInfo* d = nullptr;
  if (qsa_status st = device_info(&d)) return st;
  SelectArgs a{};
  a.scores = scores;
  a.ld = ld_scores;
  a.n_rows = n_rows;
  a.k = k_blk;
  a.n_max = nb_max;
  plan_select(a);
  a.vec_ok = scores && aligned16(scores) && (ld_scores % 4 == 0);
  a.wait_primary = 0;
  a.n_req = n_req;
  a.req_row_start = req_row_start;
  a.row_len = row_len;
  a.out_idx = out_blocks;
  a.out_pos = out_pos;
  a.out_xslots = out_slots;
  a.page_table = page_table;
  a.ld_pt = ld_pt;
  a.page_size = page_size;
  return launch_select<kModeQsa>(a, false, static_cast<cudaStream_t>(stream), d->sm_count);
}

size_t qsa_indexer_select_workspace_size(int32_t n_rows, int32_t max_len, int32_t k_blk) {
  (void)k_blk;
  if (n_rows <= 0 || max_len <= 0) return 0;
  const int64_t ld = ((int64_t)(max_len / kBlock) + 3) & ~int64_t(3);
  // scores (256-byte aligned), then the device row plan when rows may be long
  const size_t scores = ((size_t)(n_rows * ld * (int64_t)sizeof(float)) + 255) & ~(size_t)255;
  return scores + 256 + (max_len / kBlock > kRsMaxRow ? plan_bytes(n_rows) : 0);
}

}  // extern "C"

namespace {
// The fused indexer call; new_pos: see TcArgs::new_pos (nullptr: the scorer
// waits for the previous grid in full).
qsa_status indexer_select_impl(const void* q, const void* pool, int64_t pool_rows, int32_t n_req,
                               const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                               int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table,
                               int64_t ld_pt, int32_t page_size, int32_t k_blk, int32_t* out_blocks,
                               int32_t* out_pos, int32_t* out_slots, float* scores_out,
                               int64_t ld_scores, void* workspace, size_t workspace_bytes,
                               void* stream, const int32_t* new_pos, const uint8_t* pool8 = nullptr,
                               const float* key_scales = nullptr, const float* head_gates = nullptr) {
  if (k_blk < 1 || k_blk > kMaxK) return QSA_ERR_UNSUPPORTED;
  if (qsa_status st = check_rows(n_req, req_row_start, n_rows, row_len, max_len)) return st;
  if (n_rows == 0) return QSA_OK;
  if (qsa_status st = check_paging(page_table, ld_pt, page_size, max_len)) return st;
  if (!q || !(pool || pool8) || !out_slots || pool_rows < 0) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || (pool && !aligned16(pool)) || (pool8 && (!aligned16(pool8) || !key_scales)))
    return QSA_ERR_INVALID_ARG;
  if (head_gates && !aligned16(head_gates)) return QSA_ERR_INVALID_ARG;
  const int32_t nb_max = max_len / kBlock;
  float* scores = scores_out;
  int64_t ld = ld_scores;
  int32_t* plan = nullptr;  // the device row plan, when the workspace holds one
  const uintptr_t ws_lo = (reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255);
  const uintptr_t ws_hi = reinterpret_cast<uintptr_t>(workspace) + workspace_bytes;
  if (scores_out) {
    if (ld_scores < nb_max || !aligned4(scores_out)) return QSA_ERR_INVALID_ARG;
    if (workspace && ws_lo + plan_bytes(n_rows) <= ws_hi) plan = reinterpret_cast<int32_t*>(ws_lo);
  } else {
    const size_t need = qsa_indexer_select_workspace_size(n_rows, max_len, k_blk);
    if (need > 0) {
      if (!workspace || workspace_bytes < need) return QSA_ERR_WORKSPACE_TOO_SMALL;
      scores = reinterpret_cast<float*>(ws_lo);
    }
    ld = (nb_max + 3) & ~3;
    const uintptr_t plan_at = (ws_lo + (uintptr_t)n_rows * (uintptr_t)ld * 4 + 255) & ~uintptr_t(255);
    if (workspace && plan_at + plan_bytes(n_rows) <= ws_hi) plan = reinterpret_cast<int32_t*>(plan_at);
  }
  DeviceInfo* d = nullptr;
  if (qsa_status st = device_info(&d)) return st;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  ScoreArgs s{static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(pool),
              pool_rows, n_req, req_row_start, n_rows, row_len, max_len, page_table, ld_pt,
              page_size, scores, ld, 0, 1, new_pos, pool8, key_scales, head_gates};
  // the register-resident selection (one 1024-thread CTA per row) follows
  const int reserve = (n_rows <= d->sm_count / 2 && nb_max <= kSfMaxRow && k_blk <= kSfMaxK) ? n_rows : 0;
  if (qsa_status e = launch_scorer(s, max_rows_per_req, d->sm_count, st, reserve))
    return e;

  SelectArgs a{};
  a.scores = scores;
  a.ld = ld;
  a.n_rows = n_rows;
  a.k = k_blk;
  a.n_max = nb_max;
  plan_select(a);
  a.vec_ok = scores && aligned16(scores) && (ld % 4 == 0);
  a.wait_primary = 1;
  a.n_req = n_req;
  a.req_row_start = req_row_start;
  a.row_len = row_len;
  a.out_idx = out_blocks;
  a.out_pos = out_pos;
  a.out_xslots = out_slots;
  a.page_table = page_table;
  a.ld_pt = ld_pt;
  a.page_size = page_size;
  if (plan && wants_plan(n_rows, nb_max, d->sm_count))
    return launch_select_planned<kModeQsa>(a, plan, nb_max > 0, st, d);
  return launch_select<kModeQsa>(a, nb_max > 0, st, d->sm_count);
}
}  // namespace

extern "C" {

qsa_status qsa_indexer_select(const void* q, const void* pool, int64_t pool_rows, int32_t n_req,
                              const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                              int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table,
                              int64_t ld_pt, int32_t page_size, int32_t k_blk, int32_t* out_blocks,
                              int32_t* out_pos, int32_t* out_slots, float* scores_out,
                              int64_t ld_scores, void* workspace, size_t workspace_bytes,
                              void* stream) {
  return indexer_select_impl(q, pool, pool_rows, n_req, req_row_start, n_rows, row_len, max_len,
                             max_rows_per_req, page_table, ld_pt, page_size, k_blk, out_blocks, out_pos,
                             out_slots, scores_out, ld_scores, workspace, workspace_bytes, stream, nullptr);
}

qsa_status qsa_decode_step(const void* new_keys, const int32_t* req_tok_start, const int32_t* req_first_pos,
                           void* ring, double rope_base, const void* q, void* pool, int64_t pool_rows,
                           int32_t n_req, const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                           int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table,
                           int64_t ld_pt, int32_t page_size, int32_t k_blk, int32_t* out_blocks,
                           int32_t* out_pos, int32_t* out_slots, float* scores_out, int64_t ld_scores,
                           void* workspace, size_t workspace_bytes, void* stream) {
  return qsa_decode_step_gated(new_keys, req_tok_start, req_first_pos, ring, rope_base, q, nullptr, pool, pool_rows,
                               n_req, req_row_start, n_rows, row_len, max_len, max_rows_per_req, page_table, ld_pt,
                               page_size, k_blk, out_blocks, out_pos, out_slots, scores_out, ld_scores, workspace,
                               workspace_bytes, stream);
}

qsa_status qsa_decode_step_gated(const void* new_keys, const int32_t* req_tok_start, const int32_t* req_first_pos,
                                 void* ring, double rope_base, const void* q, const float* head_gates, void* pool,
                                 int64_t pool_rows, int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                 const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
                                 const int32_t* page_table, int64_t ld_pt, int32_t page_size, int32_t k_blk,
                                 int32_t* out_blocks, int32_t* out_pos, int32_t* out_slots, float* scores_out,
                                 int64_t ld_scores, void* workspace, size_t workspace_bytes, void* stream) {
  if (k_blk < 1 || k_blk > kMaxK) return QSA_ERR_UNSUPPORTED;
  if (qsa_status st = check_rows(n_req, req_row_start, n_rows, row_len, max_len)) return st;
  if (n_rows > 0) {
    if (qsa_status st = check_paging(page_table, ld_pt, page_size, max_len)) return st;
    if (!q || !pool || !out_slots || pool_rows < 0 || !aligned16(q) || !aligned16(pool))
      return QSA_ERR_INVALID_ARG;
    if (!scores_out && workspace_bytes < qsa_indexer_select_workspace_size(n_rows, max_len, k_blk))
      return QSA_ERR_WORKSPACE_TOO_SMALL;
  }
  if (qsa_status st = qsa_append_keys(new_keys, req_tok_start, req_first_pos, n_req, ring, page_table, ld_pt,
                                      page_size, rope_base, pool, pool_rows, stream))
    return st;
  if (n_rows == 0) return QSA_OK;
  return indexer_select_impl(q, pool, pool_rows, n_req, req_row_start, n_rows, row_len, max_len,
                             max_rows_per_req, page_table, ld_pt, page_size, k_blk, out_blocks, out_pos,
                             out_slots, scores_out, ld_scores, workspace, workspace_bytes, stream,
                             req_first_pos, nullptr, nullptr, head_gates);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// qsa_indexer_select_noalloc: the fused path with its score scratch in a
// library-owned device array instead of a caller workspace, for callers that
// may not allocate device memory (pre-planned memory, plugins without an
// allocator).  See include/qsa.h for the contract.
// ---------------------------------------------------------------------------
namespace {

// The scratch array itself.  Host code must not take its address directly
// (on the host the name is only a stand-in for the device symbol); the
// device address is looked up once per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QSA_NOALLOC_SCRATCH_BYTES];

float* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device (set up on the
// first call per device, with that device current).
qsa_status noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return QSA_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return QSA_OK;
}

}  // namespace

extern "C" qsa_status qsa_indexer_select_noalloc(
    const void* q, const void* pool, int64_t pool_rows, int32_t n_req, const int32_t* req_row_start,
    int32_t n_rows, const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
    const int32_t* page_table, int64_t ld_pt, int32_t page_size, int32_t k_blk, int32_t* out_blocks,
    int32_t* out_pos, int32_t* out_slots, void* stream) {
  if (k_blk < 1 || k_blk > kMaxK) return QSA_ERR_UNSUPPORTED;
  if (qsa_status st = check_rows(n_req, req_row_start, n_rows, row_len, max_len)) return st;
  if (n_rows == 0) return QSA_OK;
  if (qsa_status st = check_paging(page_table, ld_pt, page_size, max_len)) return st;
  if (!q || !pool || !out_slots || pool_rows < 0) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool)) return QSA_ERR_INVALID_ARG;
  const int32_t nb_max = max_len / kBlock;
  const int64_t ld = (nb_max + 3) & ~3;
  if ((uint64_t)n_rows * (uint64_t)ld * sizeof(float) > (uint64_t)QSA_NOALLOC_SCRATCH_BYTES)
    return QSA_ERR_UNSUPPORTED;  // the scores do not fit in the fixed scratch array
  float* scores = nullptr;
  if (qsa_status st = noalloc_scratch(&scores)) return st;
  // the fused path with the scratch array as its score buffer
  return indexer_select_impl(q, pool, pool_rows, n_req, req_row_start, n_rows, row_len, max_len,
                             max_rows_per_req, page_table, ld_pt, page_size, k_blk, out_blocks, out_pos,
                             out_slots, scores, ld, nullptr, 0, stream, nullptr);
}

// ---------------------------------------------------------------------------
// Prologue tails: query RoPE, FP8 index keys and the indexer on them.
// ---------------------------------------------------------------------------
extern "C" {

qsa_status qsa_indexer_select_gated(const void* q, const float* head_gates, const void* pool, int64_t pool_rows,
                                    int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                    const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
                                    const int32_t* page_table, int64_t ld_pt, int32_t page_size, int32_t k_blk,
                                    int32_t* out_blocks, int32_t* out_pos, int32_t* out_slots, float* scores_out,
                                    int64_t ld_scores, void* workspace, size_t workspace_bytes, void* stream) {
  if (!pool) return QSA_ERR_INVALID_ARG;
  return indexer_select_impl(q, pool, pool_rows, n_req, req_row_start, n_rows, row_len, max_len, max_rows_per_req,
                             page_table, ld_pt, page_size, k_blk, out_blocks, out_pos, out_slots, scores_out,
                             ld_scores, workspace, workspace_bytes, stream, nullptr, nullptr, nullptr, head_gates);
}

qsa_status qsa_rope_queries(const void* q, const int32_t* pos, int32_t n_rows, double rope_base, void* q_out,
                            void* stream) {
  if (n_rows < 0) return QSA_ERR_INVALID_ARG;
  if (n_rows == 0) return QSA_OK;
  if (!q || !pos || !q_out || !aligned16(q) || !aligned16(q_out) || !(rope_base > 0.0) || !std::isfinite(rope_base))
    return QSA_ERR_INVALID_ARG;
  RopeQArgs a{static_cast<const __nv_bfloat16*>(q), pos, n_rows, static_cast<__nv_bfloat16*>(q_out)};
  const int64_t units = (int64_t)n_rows * kHeads;
  const int64_t per_cta = kRopeQThreads / kCompressLanes;
  rope_queries_kernel<<<(unsigned)((units + per_cta - 1) / per_cta), kRopeQThreads, 0,
                        static_cast<cudaStream_t>(stream)>>>(a, rope_turns(rope_base));
  return launch_status();
}

qsa_status qsa_quantize_keys_fp8(const void* keys, int64_t n_keys, uint8_t* codes, float* scales, void* stream) {
  if (n_keys < 0) return QSA_ERR_INVALID_ARG;
  if (n_keys == 0) return QSA_OK;
  if (!keys || !codes || !scales || !aligned16(keys) || !aligned16(codes) || !aligned4(scales))
    return QSA_ERR_INVALID_ARG;
  const int64_t per_cta = kQuantThreads / kCompressLanes;
  if ((n_keys + per_cta - 1) / per_cta > INT32_MAX) return QSA_ERR_UNSUPPORTED;
  QuantArgs a{static_cast<const __nv_bfloat16*>(keys), n_keys, codes, scales};
  quantize_keys_fp8_kernel<<<(unsigned)((n_keys + per_cta - 1) / per_cta), kQuantThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

qsa_status qsa_index_scores_fp8(const void* q, const uint8_t* codes, const float* scales, int64_t pool_rows,
                                int32_t n_req, const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                                int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table, int64_t ld_pt,
                                int32_t page_size, float* scores, int64_t ld_scores, int64_t n_fill, void* stream) {
  if (qsa_status st = check_rows(n_req, req_row_start, n_rows, row_len, max_len)) return st;
  if (n_rows == 0) return QSA_OK;
  if (qsa_status st = check_paging(page_table, ld_pt, page_size, max_len)) return st;
  if (!q || !codes || !scales || !scores || pool_rows < 0 || n_fill < 0) return QSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(codes) || !aligned4(scales) || !aligned4(scores)) return QSA_ERR_INVALID_ARG;
  if (ld_scores < std::max<int64_t>(max_len / kBlock, n_fill)) return QSA_ERR_INVALID_ARG;
  DeviceInfo* d = nullptr;
  if (qsa_status st = device_info(&d)) return st;
  ScoreArgs s{static_cast<const __nv_bfloat16*>(q), nullptr, pool_rows, n_req, req_row_start, n_rows, row_len,
              max_len, page_table, ld_pt, page_size, scores, ld_scores, n_fill, 0, nullptr, codes, scales};
  return launch_scorer(s, max_rows_per_req, d->sm_count, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_indexer_select_fp8(const void* q, const uint8_t* codes, const float* scales, int64_t pool_rows,
                                  int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                  const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
                                  const int32_t* page_table, int64_t ld_pt, int32_t page_size, int32_t k_blk,
                                  int32_t* out_blocks, int32_t* out_pos, int32_t* out_slots, float* scores_out,
                                  int64_t ld_scores, void* workspace, size_t workspace_bytes, void* stream) {
  if (!codes || !scales) return QSA_ERR_INVALID_ARG;
  return indexer_select_impl(q, nullptr, pool_rows, n_req, req_row_start, n_rows, row_len, max_len,
                             max_rows_per_req, page_table, ld_pt, page_size, k_blk, out_blocks, out_pos, out_slots,
                             scores_out, ld_scores, workspace, workspace_bytes, stream, nullptr, codes, scales);
}

}  // extern "C"
