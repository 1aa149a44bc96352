// noalloc.cu -- jfa_fwd_noalloc: the jagged forward for callers that cannot
// give the library any device memory of its own.
//
// jfa_fwd needs a small caller-provided workspace (the host-built tile plan, an
// error word, the list of empty sequences).  Some callers cannot provide one:
// code running inside a host framework whose memory manager owns every device
// allocation and does not let extensions call cudaMalloc, or a tight serving
// loop that must never allocate (an allocation can synchronise the device or
// fail under memory pressure at the worst moment).  For them this entry point
// keeps its scratch in one file-scope device array of fixed size,
// kStaticScratchBytes (1 MiB), which every GPU that loads the library holds until
// the process exits.  Problems whose plan does not fit are rejected with
// JFA_ERR_TOO_LARGE.  Nothing here calls cudaMalloc, cudaFree, cudaHostAlloc or
// any other allocating routine; the plan reaches the device with a plain
// cudaMemcpyAsync from pageable host memory, so each call returns only after
// the work already queued on its stream has finished (the copy waits for it).
//
// A kernel that gives up a bounded wait records the failure in the array's
// error word; jfa_fwd_noalloc_status() reads it back, as jfa_device_status()
// does for a caller's workspace.
//
// All calls share the array and it keeps the last call's contents: the error
// word is cleared on every call, and calls that overlap on the GPU (different
// streams, no ordering between them) race on the plan.  The first call on a
// device looks up the array's device address (cudaGetSymbolAddress); make that
// first call before any stream capture.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/jfa.h"
#include "host.h"
#include "plan.h"

namespace jfa {

int fwd_arg_checks(const void* q, const void* k, const void* v, const void* o, const int32_t* offsets_dev,
                   const int32_t* offsets_host, int batch, int max_len, int nq, int H, int Hkv, int D, float scale,
                   int causal, int broadcast_q, int* q_rows, int* kv_rows, int* o_rows, int* num_sms);
int launch_fill_empty(const int32_t* empty_dev, int n_empty, int nq, int H, int D, int o_rows, void* o, float* lse,
                      cudaStream_t stream);
int launch_wait_forever(int* err, cudaStream_t stream);

namespace {

constexpr size_t kStaticScratchBytes = size_t(1) << 20;
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per device).
// In host code g_static_scratch names a host-side stand-in, never the device
// memory, so kernels must only ever receive this looked-up address.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return JFA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return JFA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return JFA_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace jfa

using namespace jfa;

extern "C" int jfa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                               const int32_t* offsets_dev, const int32_t* offsets_host, int batch, int max_len,
                               int nq_broadcast, int num_heads, int num_kv_heads, int head_dim, float scale,
                               int causal, int broadcast_q, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int nq = broadcast_q ? nq_broadcast : 0;
  int q_rows = 0, kv_rows = 0, o_rows = 0, num_sms = 0;
  int st = fwd_arg_checks(q, k, v, o, offsets_dev, offsets_host, batch, max_len, nq, num_heads, num_kv_heads,
                          head_dim, scale, causal, broadcast_q, &q_rows, &kv_rows, &o_rows, &num_sms);
  if (st != JFA_OK) return st;

  const int n_probe = plan_fwd(offsets_host, batch, num_heads, nq, causal, 1, nullptr, nullptr);
  const int n_cta = n_probe < num_sms ? n_probe : num_sms;
  // layout inside the static array: error word | units | CTA starts | empty sequences
  const size_t off_units = 256;
  const size_t off_cta = off_units + align256(static_cast<size_t>(n_probe) * 16);
  const size_t off_empty = off_cta + align256(static_cast<size_t>(n_cta + 1) * 4);
  const size_t total = off_empty + align256(static_cast<size_t>(batch) * 4);
  if (total > kStaticScratchBytes) return JFA_ERR_TOO_LARGE;

  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != JFA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  if (cudaMemsetAsync(ws, 0, sizeof(int), stream) != cudaSuccess) return JFA_ERR_CUDA;

  std::vector<int32_t> empty;
  if (broadcast_q)
    for (int b = 0; b < batch; ++b)
      if (offsets_host[b + 1] == offsets_host[b]) empty.push_back(b);
  if (!empty.empty()) {
    if (cudaMemcpyAsync(ws + off_empty, empty.data(), empty.size() * 4, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
      return JFA_ERR_CUDA;
    st = launch_fill_empty(reinterpret_cast<const int32_t*>(ws + off_empty), static_cast<int>(empty.size()), nq,
                           num_heads, head_dim, o_rows, o, lse, stream);
    if (st != JFA_OK) return st;
  }
  if (n_cta == 0) return JFA_OK;
  std::vector<int32_t> units, cta_start;
  plan_fwd(offsets_host, batch, num_heads, nq, causal, n_cta, &units, &cta_start);
  std::vector<uint8_t> blob(off_empty - off_units, 0);
  units_for_device(&units, offsets_host);
  std::memcpy(blob.data(), units.data(), units.size() * 4);
  std::memcpy(blob.data() + (off_cta - off_units), cta_start.data(), cta_start.size() * 4);
  // pageable source: the call returns only once the bytes have been taken, so the
  // vector may go out of scope right after
  if (cudaMemcpyAsync(ws + off_units, blob.data(), blob.size(), cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return JFA_ERR_CUDA;

  FwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.offsets_dev = offsets_dev;
  a.q_rows = q_rows;
  a.kv_rows = kv_rows;
  a.o_rows = o_rows;
  a.H = num_heads;
  a.Hkv = num_kv_heads;
  a.D = head_dim;
  a.nq = nq;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.mask = causal ? kMaskCausal : kMaskNone;
  a.win_left = -1;
  a.win_right = causal ? 0 : -1;
  a.topk_sel = nullptr;
  a.topk_qb = nullptr;
  a.topk = 0;
  a.units = reinterpret_cast<const int32_t*>(ws + off_units);
  a.cta_start = reinterpret_cast<const int32_t*>(ws + off_cta);
  a.n_cta = n_cta;
  a.n_units = static_cast<int>(units.size() / 4);
  a.use_clc = 0;  // always the static plan here
  a.err = reinterpret_cast<int*>(ws);
  a.stream = stream;
  return launch_fwd(a);
}

extern "C" size_t jfa_fwd_noalloc_capacity(void) { return kStaticScratchBytes; }

extern "C" int jfa_fwd_noalloc_status(void* stream_) {
  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != JFA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream_)) != cudaSuccess) return JFA_ERR_CUDA;
  int err = 0;  // the error word sits at offset 0 of the array
  if (cudaMemcpy(&err, scratch, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return JFA_ERR_CUDA;
  return err == 0 ? JFA_OK : JFA_ERR_DEVICE_TIMEOUT;
}

extern "C" int jfa_selftest_wait_timeout_noalloc(void* stream_) {
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != JFA_OK) return st;
  return launch_wait_forever(static_cast<int*>(scratch), static_cast<cudaStream_t>(stream_));
}
