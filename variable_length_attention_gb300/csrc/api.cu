// api.cu -- the C ABI of libjfa: argument validation, host planning, workspace
// layout and kernel launches.  The public contract is in include/jfa.h.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/jfa.h"
#include "block.h"
#include "bwd.h"
#include "host.h"
#include "plan.h"
#include "profile.h"
#include "rope.h"
#include "topk.h"

namespace jfa {

// ---------------------------------------------------------------- device info
int current_device(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return JFA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  DeviceInfo& d = cache[dev];
  if (d.device != dev) {
    DeviceInfo n;
    n.device = dev;
    if (cudaDeviceGetAttribute(&n.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return JFA_ERR_CUDA;
    d = n;
  }
  *out = d;
  return (d.cc_major == 10) ? JFA_OK : JFA_ERR_ARCH;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int make_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return JFA_ERR_CUDA;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? JFA_OK : JFA_ERR_INVALID_ARG;
}

int make_map_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                    uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return JFA_ERR_CUDA;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? JFA_OK : JFA_ERR_INVALID_ARG;
}

// ---------------------------------------------------------------- pinned staging
// Plans are built on the host every call.  They reach the device through a small
// ring of pinned host buffers so the copy never forces a host-device sync; each
// slot is reused only after the event recorded behind its previous copy has fired.
namespace {
struct Slot {
  void* host = nullptr;
  size_t cap = 0;
  cudaEvent_t done = nullptr;
  int device = -1;
};
constexpr int kSlots = 8;
std::mutex g_stage_mu;
Slot g_slots[kSlots];
int g_next_slot = 0;
}  // namespace

static int stage_to_device(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return JFA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_stage_mu);
  Slot& s = g_slots[g_next_slot];
  g_next_slot = (g_next_slot + 1) % kSlots;
  if (s.done != nullptr && cudaEventSynchronize(s.done) != cudaSuccess) return JFA_ERR_CUDA;
  if (s.done != nullptr && s.device != dev) {
    cudaEventDestroy(s.done);
    s.done = nullptr;
  }
  if (s.cap < bytes) {
    if (s.host) cudaFreeHost(s.host);
    s.host = nullptr;
    s.cap = 0;
    size_t cap = 1 << 16;
    while (cap < bytes) cap *= 2;
    if (cudaHostAlloc(&s.host, cap, cudaHostAllocPortable) != cudaSuccess) return JFA_ERR_CUDA;
    s.cap = cap;
  }
  if (s.done == nullptr) {
    if (cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming) != cudaSuccess) return JFA_ERR_CUDA;
    s.device = dev;
  }
  std::memcpy(s.host, src, bytes);
  if (cudaMemcpyAsync(dst, s.host, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) return JFA_ERR_CUDA;
  if (cudaEventRecord(s.done, stream) != cudaSuccess) return JFA_ERR_CUDA;
  return JFA_OK;
}

// ---------------------------------------------------------------- workspace layout
static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct FwdLayout {
  size_t err = 0, units = 0, cta = 0, empty = 0, qb = 0, total = 0;
};
// qb: the block-sparse forward's query-block prefix [batch+1] (topk only)
static FwdLayout fwd_layout(int n_units, int n_cta, int batch, bool topk = false) {
  FwdLayout l;
  l.err = 0;
  l.units = 256;
  l.cta = l.units + align256(static_cast<size_t>(n_units) * 16);
  l.empty = l.cta + align256(static_cast<size_t>(n_cta + 1) * 4);
  l.qb = l.empty + align256(static_cast<size_t>(batch) * 4);
  l.total = l.qb + (topk ? align256(static_cast<size_t>(batch + 1) * 4) : 0);
  return l;
}

// The first stage of the block-sparse forward (topk.cu): the blocks to average
// -- query blocks of 256 rows (b, h, m), in that order, then key blocks of 128
// keys (b, g, n) -- and, per query block, where its mean and its sequence's key
// means are.  Returns the number of query blocks.
static int topk_tasks(const int32_t* offs, int batch, int nq, int H, int Hkv, std::vector<int4>* mean_tasks,
                      std::vector<int4>* sel_tasks, int* nk_max) {
  mean_tasks->clear();
  sel_tasks->clear();
  *nk_max = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = offs[b + 1] - offs[b];
    if (L == 0) continue;
    const int rows = nq > 0 ? nq : L;
    for (int h = 0; h < H; ++h)
      for (int m = 0; m * kFwdRows < rows; ++m)
        mean_tasks->push_back(make_int4((nq > 0 ? 0 : offs[b]) + kFwdRows * m, std::min(kFwdRows, rows - kFwdRows * m),
                                        h, 0));
  }
  const int n_units = static_cast<int>(mean_tasks->size());
  std::vector<int> kb_first(batch + 1, 0);
  for (int b = 0; b < batch; ++b) {
    const int L = offs[b + 1] - offs[b];
    const int nblk = (L + kKvBlock - 1) / kKvBlock;
    kb_first[b] = static_cast<int>(mean_tasks->size()) - n_units;
    *nk_max = std::max(*nk_max, nblk);
    for (int g = 0; g < Hkv; ++g)
      for (int n = 0; n < nblk; ++n)
        mean_tasks->push_back(make_int4(offs[b] + kKvBlock * n, std::min(kKvBlock, L - kKvBlock * n), g, 1));
  }
  const int G = H / Hkv;
  for (int b = 0; b < batch; ++b) {
    const int L = offs[b + 1] - offs[b];
    if (L == 0) continue;
    const int rows = nq > 0 ? nq : L;
    const int nblk = (L + kKvBlock - 1) / kKvBlock;
    for (int h = 0; h < H; ++h)
      for (int m = 0; m * kFwdRows < rows; ++m)
        sel_tasks->push_back(make_int4(static_cast<int>(sel_tasks->size()), n_units + kb_first[b] + (h / G) * nblk,
                                       nblk, 0));
  }
  return n_units;
}

struct TopkLayout {
  size_t err = 0, mean_tasks = 0, sel_tasks = 0, means = 0, total = 0;
};
static TopkLayout topk_layout(int n_tasks, int n_units, int D) {
  TopkLayout l;
  l.mean_tasks = 256;
  l.sel_tasks = l.mean_tasks + align256(static_cast<size_t>(n_tasks) * 16);
  l.means = l.sel_tasks + align256(static_cast<size_t>(n_units) * 16);
  l.total = l.means + align256(static_cast<size_t>(n_tasks) * D * 4);
  return l;
}

struct BwdLayout {
  size_t err = 0, units = 0, cta = 0, lse2 = 0, di = 0, dq_acc = 0, total = 0;
};
static BwdLayout bwd_layout(int n_units, int n_cta, int q_rows, int o_rows, int H, int D) {
  BwdLayout l;
  l.units = 256;
  l.cta = l.units + align256(static_cast<size_t>(n_units) * 16);
  l.lse2 = l.cta + align256(static_cast<size_t>(n_cta + 1) * 4);
  l.di = l.lse2 + align256(static_cast<size_t>(H) * o_rows * 4);
  l.dq_acc = l.di + align256(static_cast<size_t>(H) * o_rows * 4);
  l.total = l.dq_acc + align256(static_cast<size_t>(q_rows) * H * D * 4);
  return l;
}

struct BlockLayout {
  size_t err = 0, bpb = 0, prog = 0, tab = 0, total = 0;
};
// tab_bytes: the rotary variants' packed (cos, sin) table, else 0
static BlockLayout block_layout(int batch, int n_prog, size_t tab_bytes = 0) {
  BlockLayout l;
  l.bpb = 256;
  l.prog = l.bpb + align256(static_cast<size_t>(batch + 1) * 4);
  l.tab = l.prog + align256(static_cast<size_t>(n_prog + 1) * 4);
  l.total = l.tab + align256(tab_bytes);
  return l;
}

// The longest sequence of a problem (the positions a rotary table must cover).
static int64_t longest(const int32_t* offsets_host, int batch) {
  int64_t m = 0;
  for (int b = 0; b < batch; ++b) m = std::max<int64_t>(m, static_cast<int64_t>(offsets_host[b + 1]) - offsets_host[b]);
  return m;
}

__global__ void fill_empty_broadcast_kernel(const int32_t* empty_seq, int n_empty, int nq, int H, int D,
                                            int o_rows, __nv_bfloat16* o, float* lse) {
  // one block row per (empty sequence, query row); threads over H*D
  const int r = blockIdx.x;
  if (r >= n_empty * nq) return;
  const int b = empty_seq[r / nq];
  const int row = b * nq + r % nq;
  for (int i = threadIdx.x; i < H * D; i += blockDim.x) o[static_cast<size_t>(row) * H * D + i] = __float2bfloat16(0.f);
  if (lse)
    for (int h = threadIdx.x; h < H; h += blockDim.x) lse[static_cast<size_t>(h) * o_rows + row] = -INFINITY;
}

struct Common {
  DeviceInfo dev;
  int q_rows = 0, kv_rows = 0, o_rows = 0;
};

static int validate_common(const void* q, const void* k, const void* v, const void* o, const int32_t* offsets_dev,
                           const int32_t* offsets_host, int batch, int max_len, int nq, int H, int Hkv, int D,
                           float scale, int causal, int broadcast_q, Common* c) {
  if (batch < 0 || H <= 0 || Hkv <= 0 || max_len < 0) return JFA_ERR_INVALID_ARG;
  if (offsets_host == nullptr || offsets_dev == nullptr) return JFA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
  if (H % Hkv != 0) return JFA_ERR_UNSUPPORTED;
  if (broadcast_q && causal) return JFA_ERR_UNSUPPORTED;
  if (broadcast_q && nq <= 0) return JFA_ERR_INVALID_ARG;
  const int st = check_offsets(offsets_host, batch, max_len);
  if (st != JFA_OK) return st;
  // row indices are 32-bit: the broadcast output's batch * nq rows must fit
  if (broadcast_q && static_cast<int64_t>(batch) * nq > INT32_MAX) return JFA_ERR_UNSUPPORTED;
  c->kv_rows = offsets_host[batch];
  c->q_rows = broadcast_q ? nq : c->kv_rows;
  c->o_rows = broadcast_q ? batch * nq : c->kv_rows;
  if (c->o_rows > 0 && (q == nullptr || o == nullptr)) return JFA_ERR_INVALID_ARG;
  if (c->kv_rows > 0 && (k == nullptr || v == nullptr)) return JFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return JFA_ERR_INVALID_ARG;
  return JFA_OK;  // the caller queries the device after its own argument checks
}

static int plan_ctas(const DeviceInfo& dev, int n_units) { return n_units < dev.num_sms ? n_units : dev.num_sms; }

static std::atomic<int> g_sched_mode{-1};

int sched_mode() {
  int m = g_sched_mode.load(std::memory_order_relaxed);
  if (m < 0) {
    const char* e = std::getenv("JFA_SCHED");
    m = (e != nullptr && std::strcmp(e, "static") == 0) ? 0 : (e != nullptr && std::strcmp(e, "clc") == 0 ? 1 : kDefaultSched);
    g_sched_mode.store(m, std::memory_order_relaxed);
  }
  return m;
}

static std::atomic<int> g_block_sched_mode{-1};

int block_sched_mode() {
  int m = g_block_sched_mode.load(std::memory_order_relaxed);
  if (m < 0) {
    const char* e = std::getenv("JFA_SCHED_BLOCK");
    m = (e != nullptr && std::strcmp(e, "static") == 0) ? 0
        : (e != nullptr && std::strcmp(e, "clc") == 0 ? 1 : kDefaultBlockSched);
    g_block_sched_mode.store(m, std::memory_order_relaxed);
  }
  return m;
}

static std::atomic<int> g_bwd_sched_mode{-1};

int bwd_sched_mode() {
  int m = g_bwd_sched_mode.load(std::memory_order_relaxed);
  if (m < 0) {
    const char* e = std::getenv("JFA_SCHED_BWD");
    m = (e != nullptr && std::strcmp(e, "static") == 0) ? 0
        : (e != nullptr && std::strcmp(e, "clc") == 0 ? 1 : kDefaultBwdSched);
    g_bwd_sched_mode.store(m, std::memory_order_relaxed);
  }
  return m;
}

// ---------------------------------------------------------------- helpers for noalloc.cu
// The same argument checks as jfa_fwd, then the device query; fills the row
// counts and the SM count.
int fwd_arg_checks(const void* q, const void* k, const void* v, const void* o, const int32_t* offsets_dev,
                   const int32_t* offsets_host, int batch, int max_len, int nq, int H, int Hkv, int D, float scale,
                   int causal, int broadcast_q, int* q_rows, int* kv_rows, int* o_rows, int* num_sms) {
  Common c;
  int st = validate_common(q, k, v, o, offsets_dev, offsets_host, batch, max_len, nq, H, Hkv, D, scale, causal,
                           broadcast_q, &c);
  if (st != JFA_OK) return st;
  st = current_device(&c.dev);
  if (st != JFA_OK) return st;
  *q_rows = c.q_rows;
  *kv_rows = c.kv_rows;
  *o_rows = c.o_rows;
  *num_sms = c.dev.num_sms;
  return JFA_OK;
}

// Zero output rows and -inf log-sum-exp for empty sequences in broadcast mode.
int launch_fill_empty(const int32_t* empty_dev, int n_empty, int nq, int H, int D, int o_rows, void* o, float* lse,
                      cudaStream_t stream) {
  if (n_empty == 0) return JFA_OK;
  fill_empty_broadcast_kernel<<<n_empty * nq, 256, 0, stream>>>(empty_dev, n_empty, nq, H, D, o_rows,
                                                                 static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError() == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

}  // namespace jfa

using namespace jfa;

extern "C" const char* jfa_status_string(int status) {
  switch (status) {
    case JFA_OK: return "ok";
    case JFA_ERR_INVALID_ARG: return "invalid argument";
    case JFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case JFA_ERR_BAD_OFFSETS: return "bad offsets";
    case JFA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case JFA_ERR_ARCH: return "device is not compute capability 10.x";
    case JFA_ERR_CUDA: return "CUDA error";
    case JFA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case JFA_ERR_TOO_LARGE: return "problem too large for the static scratch of jfa_fwd_noalloc";
    default: return "unknown status";
  }
}

extern "C" size_t jfa_workspace_size(int op, const int32_t* offsets_host, int batch, int nq_broadcast, int num_heads,
                                     int head_dim, int causal, int broadcast_q) {
  if (offsets_host == nullptr || batch < 0 || num_heads <= 0) return 0;
  if (check_offsets(offsets_host, batch, -1) != JFA_OK) return 0;
  DeviceInfo dev;
  if (current_device(&dev) != JFA_OK) return 0;
  const int nq = broadcast_q ? nq_broadcast : 0;
  if (broadcast_q && (nq <= 0 || static_cast<int64_t>(batch) * nq > INT32_MAX)) return 0;
  if (op == JFA_OP_FWD) {
    const int n = plan_fwd(offsets_host, batch, num_heads, nq, causal, 1, nullptr, nullptr);
    return fwd_layout(n, plan_ctas(dev, n), batch).total;
  }
  if (op == JFA_OP_BWD) {
    if (head_dim != 64 && head_dim != 128) return 0;
    // planned over all query heads: an upper bound when the call groups them
    // (grouped-query attention plans over the fewer K/V heads)
    const int n = plan_bwd(offsets_host, batch, num_heads, nq, causal, 1, nullptr, nullptr);
    const int q_rows = broadcast_q ? nq : offsets_host[batch];
    const int o_rows = broadcast_q ? batch * nq : offsets_host[batch];
    return bwd_layout(n, plan_ctas(dev, n), q_rows, o_rows, num_heads, head_dim).total;
  }
  if (op == JFA_OP_TOPK_SELECT) {
    if (head_dim != 64 && head_dim != 128) return 0;
    std::vector<int4> mt, stasks;
    int nk_max = 0;
    // key blocks counted for num_heads key/value heads: an upper bound under GQA
    const int n_units = topk_tasks(offsets_host, batch, nq, num_heads, num_heads, &mt, &stasks, &nk_max);
    return topk_layout(static_cast<int>(mt.size()), n_units, head_dim).total;
  }
  if (op == JFA_OP_FWD_TOPK) {
    const int n = plan_fwd_topk(offsets_host, batch, num_heads, nq, 1, 1, nullptr, nullptr);
    return fwd_layout(n, plan_ctas(dev, n), batch, true).total;
  }
  if (op == JFA_OP_BLOCK_FWD || op == JFA_OP_BLOCK_BWD || op == JFA_OP_BLOCK_FWD_ROPE ||
      op == JFA_OP_BLOCK_BWD_ROPE) {
    const int P = plan_block(offsets_host, batch, num_heads, dev.num_sms, nullptr, nullptr);
    const bool rope = op == JFA_OP_BLOCK_FWD_ROPE || op == JFA_OP_BLOCK_BWD_ROPE;
    const size_t tab = rope ? static_cast<size_t>(longest(offsets_host, batch)) * (head_dim / 2) * 4 : 0;
    return block_layout(batch, P, tab).total;
  }
  return 0;
}

// The key window of a call: causal is (-1, 0); a window needs self-attention
// and bounds of at least -1 (-1 leaves a side open).
static int window_of(int causal, int window_left, int window_right, int broadcast_q, int* left, int* right,
                     int* mask) {
  if (window_left < -1 || window_right < -1) return JFA_ERR_INVALID_ARG;
  *left = window_left;
  *right = causal ? (window_right < 0 ? 0 : std::min(window_right, 0)) : window_right;
  if (*left < 0 && *right < 0) {
    *mask = kMaskNone;
  } else if (*left < 0 && *right == 0) {
    *mask = kMaskCausal;
  } else {
    *mask = kMaskWindow;
  }
  if (broadcast_q && *mask != kMaskNone) return JFA_ERR_UNSUPPORTED;
  return JFA_OK;
}

static int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* offsets_dev,
                    const int32_t* offsets_host, int batch, int max_len, int nq_broadcast, int num_heads,
                    int num_kv_heads, int head_dim, float scale, int causal, int window_left, int window_right,
                    int broadcast_q, void* workspace, size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  Common c;
  const int nq = broadcast_q ? nq_broadcast : 0;
  int st = validate_common(q, k, v, o, offsets_dev, offsets_host, batch, max_len, nq, num_heads, num_kv_heads,
                           head_dim, scale, causal, broadcast_q, &c);
  if (st != JFA_OK) return st;
  int left = -1, right = -1, mask = kMaskNone;
  st = window_of(causal, window_left, window_right, broadcast_q, &left, &right, &mask);
  if (st != JFA_OK) return st;
  if (workspace == nullptr && workspace_bytes > 0) return JFA_ERR_INVALID_ARG;
  st = current_device(&c.dev);
  if (st != JFA_OK) return st;

  std::vector<int32_t> units, cta_start;
  const int n_probe = plan_fwd_window(offsets_host, batch, num_heads, nq, left, right, 1, nullptr, nullptr);
  const int n_cta = plan_ctas(c.dev, n_probe);
  const int clc = sched_mode();
  int n = 0;
  // Cluster Launch Control takes the units in plain cost order (the plan dealt to one CTA)
  if (n_cta > 0)
    n = plan_fwd_window(offsets_host, batch, num_heads, nq, left, right, clc ? 1 : n_cta, &units, &cta_start);
  std::vector<int32_t> empty;
  if (broadcast_q)
    for (int b = 0; b < batch; ++b)
      if (offsets_host[b + 1] == offsets_host[b]) empty.push_back(b);
  const FwdLayout lay = fwd_layout(n, n_cta, batch);
  if (workspace_bytes < lay.total || workspace == nullptr) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  if (!empty.empty()) {
    // one staging copy for the list of empty sequences, then a fill kernel
    st = stage_to_device(ws + lay.empty, empty.data(), empty.size() * 4, stream);
    if (st != JFA_OK) return st;
    const int blocks = static_cast<int>(empty.size()) * nq;
    ProfileScope prof(kKindFill, stream);
    fill_empty_broadcast_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const int32_t*>(ws + lay.empty),
                                                             static_cast<int>(empty.size()), nq, num_heads,
                                                             head_dim, c.o_rows, static_cast<__nv_bfloat16*>(o), lse);
    if (cudaGetLastError() != cudaSuccess) return JFA_ERR_CUDA;
  }
  if (n == 0) return cudaMemsetAsync(ws + lay.err, 0, sizeof(int), stream) == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
  // the cleared error word, the units and the CTA starts travel in one copy
  // (they are adjacent at the head of the workspace)
  std::vector<uint8_t> blob(lay.empty - lay.err, 0);
  units_for_device(&units, offsets_host);
  std::memcpy(blob.data() + (lay.units - lay.err), units.data(), units.size() * 4);
  std::memcpy(blob.data() + (lay.cta - lay.err), cta_start.data(), cta_start.size() * 4);
  st = stage_to_device(ws + lay.err, blob.data(), blob.size(), stream);
  if (st != JFA_OK) return st;

  FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.offsets_dev = offsets_dev;
  a.q_rows = c.q_rows;
  a.kv_rows = c.kv_rows;
  a.o_rows = c.o_rows;
  a.H = num_heads;
  a.Hkv = num_kv_heads;
  a.D = head_dim;
  a.nq = nq;
  a.scale = scale;
  a.causal = mask == kMaskCausal ? 1 : 0;
  a.mask = mask;
  a.win_left = left;
  a.win_right = right;
  a.topk_sel = nullptr;
  a.topk_qb = nullptr;
  a.topk = 0;
  a.units = reinterpret_cast<const int32_t*>(ws + lay.units);
  a.cta_start = reinterpret_cast<const int32_t*>(ws + lay.cta);
  a.n_cta = n_cta;
  a.n_units = n;
  a.use_clc = clc;
  a.err = reinterpret_cast<int*>(ws + lay.err);
  a.stream = stream;
  return launch_fwd(a);
}

extern "C" int jfa_topk_rows(const int32_t* offsets_host, int batch, int nq_broadcast, int num_heads,
                             int broadcast_q) {
  if (offsets_host == nullptr || batch < 0 || num_heads <= 0) return -JFA_ERR_INVALID_ARG;
  if (check_offsets(offsets_host, batch, -1) != JFA_OK) return -JFA_ERR_BAD_OFFSETS;
  if (broadcast_q && nq_broadcast <= 0) return -JFA_ERR_INVALID_ARG;
  int64_t n = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t L = static_cast<int64_t>(offsets_host[b + 1]) - offsets_host[b];
    if (L > 0) n += static_cast<int64_t>(num_heads) * (((broadcast_q ? nq_broadcast : L) + kFwdRows - 1) / kFwdRows);
  }
  return n > INT32_MAX ? -JFA_ERR_UNSUPPORTED : static_cast<int>(n);
}

extern "C" int jfa_topk_select(const void* q, const void* k, const int32_t* offsets_dev, const int32_t* offsets_host,
                               int batch, int max_len, int nq_broadcast, int num_heads, int num_kv_heads,
                               int head_dim, int topk, int broadcast_q, int32_t* selection, void* workspace,
                               size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  Common c;
  const int nq = broadcast_q ? nq_broadcast : 0;
  int st = validate_common(q, k, k, q, offsets_dev, offsets_host, batch, max_len, nq, num_heads, num_kv_heads,
                           head_dim, 1.0f, 0, broadcast_q, &c);
  if (st != JFA_OK) return st;
  if (topk < 1) return JFA_ERR_INVALID_ARG;
  std::vector<int4> mt, stasks;
  int nk_max = 0;
  const int n_units = topk_tasks(offsets_host, batch, nq, num_heads, num_kv_heads, &mt, &stasks, &nk_max);
  if (n_units > 0 && selection == nullptr) return JFA_ERR_INVALID_ARG;
  // the selection kernel keeps one score per key block of the longest sequence
  // in shared memory (48 KB: 12,288 blocks, 1,572,864 keys)
  if (static_cast<size_t>(nk_max) * sizeof(float) > 48 * 1024) return JFA_ERR_UNSUPPORTED;
  const TopkLayout lay = topk_layout(static_cast<int>(mt.size()), n_units, head_dim);
  if (workspace == nullptr || workspace_bytes < lay.total) return JFA_ERR_WORKSPACE_TOO_SMALL;
  st = current_device(&c.dev);
  if (st != JFA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // the cleared error word and both task lists in one copy
  std::vector<uint8_t> blob(lay.means - lay.err, 0);
  std::memcpy(blob.data() + lay.mean_tasks, mt.data(), mt.size() * 16);
  std::memcpy(blob.data() + lay.sel_tasks, stasks.data(), stasks.size() * 16);
  st = stage_to_device(ws, blob.data(), blob.size(), stream);
  if (st != JFA_OK) return st;
  TopkArgs a;
  a.q = q;
  a.k = k;
  a.H = num_heads;
  a.Hkv = num_kv_heads;
  a.D = head_dim;
  a.mean_tasks = reinterpret_cast<const int4*>(ws + lay.mean_tasks);
  a.n_tasks = static_cast<int>(mt.size());
  a.means = reinterpret_cast<float*>(ws + lay.means);
  a.sel_tasks = reinterpret_cast<const int4*>(ws + lay.sel_tasks);
  a.n_units = n_units;
  a.topk = topk;
  a.nk_max = nk_max;
  a.selection = selection;
  a.stream = stream;
  return launch_topk_select(a);
}

extern "C" int jfa_fwd_topk(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* selection,
                            int topk, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
                            int max_len, int nq_broadcast, int num_heads, int num_kv_heads, int head_dim,
                            float scale, int broadcast_q, void* workspace, size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  Common c;
  const int nq = broadcast_q ? nq_broadcast : 0;
  int st = validate_common(q, k, v, o, offsets_dev, offsets_host, batch, max_len, nq, num_heads, num_kv_heads,
                           head_dim, scale, 0, broadcast_q, &c);
  if (st != JFA_OK) return st;
  if (topk < 1) return JFA_ERR_INVALID_ARG;
  if (workspace == nullptr && workspace_bytes > 0) return JFA_ERR_INVALID_ARG;
  st = current_device(&c.dev);
  if (st != JFA_OK) return st;
  std::vector<int32_t> units, cta_start;
  const int n_probe = plan_fwd_topk(offsets_host, batch, num_heads, nq, topk, 1, nullptr, nullptr);
  if (n_probe > 0 && selection == nullptr) return JFA_ERR_INVALID_ARG;
  const int n_cta = plan_ctas(c.dev, n_probe);
  const int clc = sched_mode();
  int n = 0;
  if (n_cta > 0) n = plan_fwd_topk(offsets_host, batch, num_heads, nq, topk, clc ? 1 : n_cta, &units, &cta_start);
  std::vector<int32_t> empty, qb(batch + 1, 0);
  for (int b = 0; b < batch; ++b) {
    const int L = offsets_host[b + 1] - offsets_host[b];
    if (broadcast_q && L == 0) empty.push_back(b);
    qb[b + 1] = qb[b] + (L > 0 ? ((broadcast_q ? nq : L) + kFwdRows - 1) / kFwdRows : 0);
  }
  const FwdLayout lay = fwd_layout(n, n_cta, batch, true);
  if (workspace_bytes < lay.total || workspace == nullptr) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // the cleared error word, units, CTA starts, empty sequences and the
  // query-block prefix in one copy
  std::vector<uint8_t> blob(lay.total - lay.err, 0);
  units_for_device(&units, offsets_host);
  std::memcpy(blob.data() + (lay.units - lay.err), units.data(), units.size() * 4);
  std::memcpy(blob.data() + (lay.cta - lay.err), cta_start.data(), cta_start.size() * 4);
  std::memcpy(blob.data() + (lay.empty - lay.err), empty.data(), empty.size() * 4);
  std::memcpy(blob.data() + (lay.qb - lay.err), qb.data(), qb.size() * 4);
  st = stage_to_device(ws + lay.err, blob.data(), blob.size(), stream);
  if (st != JFA_OK) return st;
  if (!empty.empty()) {
    st = launch_fill_empty(reinterpret_cast<const int32_t*>(ws + lay.empty), static_cast<int>(empty.size()), nq,
                           num_heads, head_dim, c.o_rows, o, lse, stream);
    if (st != JFA_OK) return st;
  }
  if (n == 0) return JFA_OK;
  FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.offsets_dev = offsets_dev;
  a.q_rows = c.q_rows;
  a.kv_rows = c.kv_rows;
  a.o_rows = c.o_rows;
  a.H = num_heads;
  a.Hkv = num_kv_heads;
  a.D = head_dim;
  a.nq = nq;
  a.scale = scale;
  a.causal = 0;
  a.mask = kMaskTopK;
  a.win_left = a.win_right = -1;
  a.topk_sel = selection;
  a.topk_qb = reinterpret_cast<const int32_t*>(ws + lay.qb);
  a.topk = topk;
  a.units = reinterpret_cast<const int32_t*>(ws + lay.units);
  a.cta_start = reinterpret_cast<const int32_t*>(ws + lay.cta);
  a.n_cta = n_cta;
  a.n_units = n;
  a.use_clc = clc;
  a.err = reinterpret_cast<int*>(ws + lay.err);
  a.stream = stream;
  return launch_fwd(a);
}

extern "C" int jfa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* offsets_dev,
                       const int32_t* offsets_host, int batch, int max_len, int nq_broadcast, int num_heads,
                       int num_kv_heads, int head_dim, float scale, int causal, int broadcast_q, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return fwd_impl(q, k, v, o, lse, offsets_dev, offsets_host, batch, max_len, nq_broadcast, num_heads, num_kv_heads,
                  head_dim, scale, causal, -1, -1, broadcast_q, workspace, workspace_bytes, stream);
}

extern "C" int jfa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int32_t* offsets_dev, const int32_t* offsets_host, int batch, int max_len,
                              int num_heads, int num_kv_heads, int head_dim, float scale, int window_left,
                              int window_right, void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(q, k, v, o, lse, offsets_dev, offsets_host, batch, max_len, 0, num_heads, num_kv_heads, head_dim,
                  scale, 0, window_left, window_right, 0, workspace, workspace_bytes, stream);
}

static int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                    void* dq, void* dk, void* dv, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
                    int max_len, int nq_broadcast, int num_heads, int num_kv_heads, int head_dim, float scale,
                    int causal, int window_left, int window_right, int broadcast_q, void* workspace,
                    size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  Common c;
  const int nq = broadcast_q ? nq_broadcast : 0;
  int st = validate_common(q, k, v, o, offsets_dev, offsets_host, batch, max_len, nq, num_heads, num_kv_heads,
                           head_dim, scale, causal, broadcast_q, &c);
  if (st != JFA_OK) return st;
  int left = -1, right = -1, mask = kMaskNone;
  st = window_of(causal, window_left, window_right, broadcast_q, &left, &right, &mask);
  if (st != JFA_OK) return st;
  if (c.o_rows > 0 && (dout == nullptr || lse == nullptr || dq == nullptr)) return JFA_ERR_INVALID_ARG;
  if (c.kv_rows > 0 && (dk == nullptr || dv == nullptr)) return JFA_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv)) return JFA_ERR_INVALID_ARG;
  st = current_device(&c.dev);
  if (st != JFA_OK) return st;

  std::vector<int32_t> units, cta_start;
  // units run over the K/V heads; each loops over its group's query heads
  const int n_probe = plan_bwd_window(offsets_host, batch, num_kv_heads, nq, left, right, 1, nullptr, nullptr);
  const int n_cta = plan_ctas(c.dev, n_probe);
  const int clc = bwd_sched_mode();
  int n = 0;
  // Cluster Launch Control takes the units in plain cost order (the plan dealt to one CTA)
  if (n_cta > 0)
    n = plan_bwd_window(offsets_host, batch, num_kv_heads, nq, left, right, clc ? 1 : n_cta, &units, &cta_start);
  const BwdLayout lay = bwd_layout(n, n_cta, c.q_rows, c.o_rows, num_heads, head_dim);
  if (workspace == nullptr || workspace_bytes < lay.total) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.offsets_dev = offsets_dev;
  a.q_rows = c.q_rows;
  a.kv_rows = c.kv_rows;
  a.o_rows = c.o_rows;
  a.H = num_heads;
  a.Hkv = num_kv_heads;
  a.D = head_dim;
  a.nq = nq;
  a.scale = scale;
  a.causal = mask == kMaskCausal ? 1 : 0;
  a.mask = mask;
  a.win_left = left;
  a.win_right = right;
  a.units = reinterpret_cast<const int32_t*>(ws + lay.units);
  a.cta_start = reinterpret_cast<const int32_t*>(ws + lay.cta);
  a.n_cta = n_cta;
  a.n_units = n;
  a.use_clc = clc;
  a.lse2 = reinterpret_cast<float*>(ws + lay.lse2);
  a.di = reinterpret_cast<float*>(ws + lay.di);
  a.dq_acc = reinterpret_cast<float*>(ws + lay.dq_acc);
  a.err = reinterpret_cast<int*>(ws + lay.err);
  a.stream = stream;

  if (n > 0) {
    // the cleared error word, the units and the CTA starts in one copy, ahead of
    // the kernels so that they follow one another directly
    std::vector<uint8_t> blob(lay.lse2 - lay.err, 0);
    units_for_device(&units, offsets_host);
    std::memcpy(blob.data() + (lay.units - lay.err), units.data(), units.size() * 4);
    std::memcpy(blob.data() + (lay.cta - lay.err), cta_start.data(), cta_start.size() * 4);
    st = stage_to_device(ws + lay.err, blob.data(), blob.size(), stream);
  } else {
    st = cudaMemsetAsync(ws + lay.err, 0, sizeof(int), stream) == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
  }
  if (st != JFA_OK) return st;
  // the prepass also zeroes the dQ accumulator, so it runs even with no units
  // (broadcast-Q with every sequence empty still returns dQ = 0)
  st = launch_bwd_prep(a, c.dev.num_sms);
  if (st != JFA_OK) return st;
  if (n > 0) {
    st = launch_bwd_main(a);
    if (st != JFA_OK) return st;
  }
  return launch_dq_convert(a, c.dev.num_sms);
}

extern "C" int jfa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                       void* dq, void* dk, void* dv, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
                       int max_len, int nq_broadcast, int num_heads, int num_kv_heads, int head_dim, float scale,
                       int causal, int broadcast_q, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, offsets_dev, offsets_host, batch, max_len, nq_broadcast,
                  num_heads, num_kv_heads, head_dim, scale, causal, -1, -1, broadcast_q, workspace, workspace_bytes,
                  stream);
}

extern "C" int jfa_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, const int32_t* offsets_dev,
                              const int32_t* offsets_host, int batch, int max_len, int num_heads, int num_kv_heads,
                              int head_dim, float scale, int window_left, int window_right, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, offsets_dev, offsets_host, batch, max_len, 0, num_heads,
                  num_kv_heads, head_dim, scale, 0, window_left, window_right, 0, workspace, workspace_bytes, stream);
}

// Shared by the two block-diagonal entry points: checks, host plan, staging.
// With `tab` (the rotary variants) the workspace also holds the packed rotary
// table, whose address and row count come back in *tab and *tab_rows.
static int block_common(const void* q, const void* k, const void* v, const void* out0, const int32_t* offsets_dev,
                        const int32_t* offsets_host, int batch, int max_len, int num_heads, int head_dim, float scale,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream, BlockArgs* a,
                        uint32_t** tab = nullptr, int64_t* tab_rows = nullptr) {
  Common c;
  int st = validate_common(q, k, v, out0, offsets_dev, offsets_host, batch, max_len, 0, num_heads, num_heads,
                           head_dim, scale, 0, 0, &c);
  if (st != JFA_OK) return st;
  st = current_device(&c.dev);
  if (st != JFA_OK) return st;
  std::vector<int32_t> bpb, prog;
  const int P = plan_block(offsets_host, batch, num_heads, c.dev.num_sms, &bpb, &prog);
  const int64_t rows_tab = tab ? longest(offsets_host, batch) : 0;
  const BlockLayout lay = block_layout(batch, P, static_cast<size_t>(rows_tab) * (head_dim / 2) * 4);
  if (workspace == nullptr || workspace_bytes < lay.total) return JFA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (tab) {
    *tab = reinterpret_cast<uint32_t*>(ws + lay.tab);
    *tab_rows = rows_tab;
  }
  a->q = q;
  a->k = k;
  a->v = v;
  a->offsets_dev = offsets_dev;
  a->bpb = reinterpret_cast<const int32_t*>(ws + lay.bpb);
  a->prog_start = reinterpret_cast<const int32_t*>(ws + lay.prog);
  a->err = reinterpret_cast<int*>(ws + lay.err);
  a->rows = c.kv_rows;
  a->batch = batch;
  a->H = num_heads;
  a->D = head_dim;
  a->n_blocks = bpb[batch];
  a->n_prog = P;
  a->use_clc = block_sched_mode();
  a->chunk = kBlockChunk;
  a->n_tiles = static_cast<int>((static_cast<int64_t>(a->n_blocks) + 1) / 2 * num_heads);
  a->n_chunks = (a->n_tiles + kBlockChunk - 1) / kBlockChunk;
  a->scale = scale;
  a->stream = stream;
  if (P == 0) return cudaMemsetAsync(ws + lay.err, 0, sizeof(int), stream) == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
  // the cleared error word and both lists in one copy (the rotary table that
  // follows them is written by its own kernel)
  std::vector<uint8_t> blob(lay.tab - lay.err, 0);
  std::memcpy(blob.data() + (lay.bpb - lay.err), bpb.data(), bpb.size() * 4);
  std::memcpy(blob.data() + (lay.prog - lay.err), prog.data(), prog.size() * 4);
  return stage_to_device(ws + lay.err, blob.data(), blob.size(), stream);
}

extern "C" int block_attn_fwd(const void* q, const void* k, const void* v, void* o, const int32_t* offsets_dev,
                              const int32_t* offsets_host, int batch, int max_len, int num_heads, int head_dim,
                              float scale, void* workspace, size_t workspace_bytes, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  BlockArgs a{};
  int st = block_common(q, k, v, o, offsets_dev, offsets_host, batch, max_len, num_heads, head_dim, scale, workspace,
                        workspace_bytes, stream, &a);
  if (st != JFA_OK || a.n_prog == 0) return st;
  a.o = o;
  return launch_block_fwd(a);
}

// The rotary tables of the rotary block entry points: both given, 16-byte
// aligned, with a row for every position a sequence of max_len tokens has.
static int check_rope(const float* rope_cos, const float* rope_sin, int rope_rows, int max_len) {
  if (rope_cos == nullptr || rope_sin == nullptr || !aligned16(rope_cos) || !aligned16(rope_sin))
    return JFA_ERR_INVALID_ARG;
  if (rope_rows < max_len || rope_rows < 0) return JFA_ERR_INVALID_ARG;
  return JFA_OK;
}

extern "C" int block_attn_fwd_rope(const void* q, const void* k, const void* v, void* o, const float* rope_cos,
                                   const float* rope_sin, int rope_rows, const int32_t* offsets_dev,
                                   const int32_t* offsets_host, int batch, int max_len, int num_heads, int head_dim,
                                   float scale, void* workspace, size_t workspace_bytes, void* stream_) {
  int st = check_rope(rope_cos, rope_sin, rope_rows, max_len);
  if (st != JFA_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  BlockArgs a{};
  uint32_t* tab = nullptr;
  int64_t tab_rows = 0;
  st = block_common(q, k, v, o, offsets_dev, offsets_host, batch, max_len, num_heads, head_dim, scale, workspace,
                    workspace_bytes, stream, &a, &tab, &tab_rows);
  if (st != JFA_OK || a.n_prog == 0) return st;
  // the packed table, then the block forward, which rotates q and k tiles in
  // shared memory as they land
  st = launch_rope_pack(rope_cos, rope_sin, tab, tab_rows, head_dim / 2, stream);
  if (st != JFA_OK) return st;
  a.rope_tab = tab;
  a.o = o;
  return launch_block_fwd(a);
}

extern "C" int block_attn_bwd_rope(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                   void* dq, void* dk, void* dv, const float* rope_cos, const float* rope_sin,
                                   int rope_rows, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
                                   int max_len, int num_heads, int head_dim, float scale, void* workspace,
                                   size_t workspace_bytes, void* stream_) {
  (void)o;  // Di is formed inline as rowsum(P o dP); O itself is not read
  int st = check_rope(rope_cos, rope_sin, rope_rows, max_len);
  if (st != JFA_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (offsets_host != nullptr && batch >= 0 && offsets_host[batch] > 0 &&
      (dout == nullptr || dq == nullptr || dk == nullptr || dv == nullptr))
    return JFA_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv)) return JFA_ERR_INVALID_ARG;
  BlockArgs a{};
  uint32_t* tab = nullptr;
  int64_t tab_rows = 0;
  st = block_common(q, k, v, dq, offsets_dev, offsets_host, batch, max_len, num_heads, head_dim, scale, workspace,
                    workspace_bytes, stream, &a, &tab, &tab_rows);
  if (st != JFA_OK || a.n_prog == 0) return st;
  // the packed table, the block backward rotating q and k tiles as they land;
  // its dq and dk, with respect to the rotated rows, go back through the
  // transposed rotation in the kernel's epilogue
  st = launch_rope_pack(rope_cos, rope_sin, tab, tab_rows, head_dim / 2, stream);
  if (st != JFA_OK) return st;
  a.rope_tab = tab;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  return launch_block_bwd(a);
}

extern "C" int block_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, void* dq,
                              void* dk, void* dv, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
                              int max_len, int num_heads, int head_dim, float scale, void* workspace,
                              size_t workspace_bytes, void* stream_) {
  (void)o;  // Di is formed inline as rowsum(P o dP); O itself is not read
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (offsets_host != nullptr && batch >= 0 && offsets_host[batch] > 0 &&
      (dout == nullptr || dq == nullptr || dk == nullptr || dv == nullptr))
    return JFA_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv)) return JFA_ERR_INVALID_ARG;
  BlockArgs a{};
  int st = block_common(q, k, v, dq, offsets_dev, offsets_host, batch, max_len, num_heads, head_dim, scale,
                        workspace, workspace_bytes, stream, &a);
  if (st != JFA_OK || a.n_prog == 0) return st;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  return launch_block_bwd(a);
}

extern "C" int jfa_set_schedule(int mode) {
  if (mode != 0 && mode != 1) return JFA_ERR_INVALID_ARG;
  g_sched_mode.store(mode, std::memory_order_relaxed);
  return JFA_OK;
}

extern "C" int jfa_get_schedule(void) { return sched_mode(); }

extern "C" int jfa_set_bwd_schedule(int mode) {
  if (mode != 0 && mode != 1) return JFA_ERR_INVALID_ARG;
  g_bwd_sched_mode.store(mode, std::memory_order_relaxed);
  return JFA_OK;
}

extern "C" int jfa_get_bwd_schedule(void) { return bwd_sched_mode(); }

extern "C" int jfa_set_block_schedule(int mode) {
  if (mode != 0 && mode != 1) return JFA_ERR_INVALID_ARG;
  g_block_sched_mode.store(mode, std::memory_order_relaxed);
  return JFA_OK;
}

extern "C" int jfa_get_block_schedule(void) { return block_sched_mode(); }

extern "C" int jfa_device_status(const void* workspace, void* stream) {
  if (workspace == nullptr) return JFA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return JFA_ERR_CUDA;
  int err = 0;
  if (cudaMemcpy(&err, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return JFA_ERR_CUDA;
  return err == 0 ? JFA_OK : JFA_ERR_DEVICE_TIMEOUT;
}
