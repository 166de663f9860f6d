// smqa_noalloc.cu -- forward and backward for callers that cannot allocate
// device memory: their scratch (the forward's exchange pool; the backward's
// fp32 dKV accumulator, Delta and exchange pool) lives in one file-scope
// static device array instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "sparse_mqa.h"
#include "smqa_internal.h"

namespace {

// The scratch buffer.  Every device that loads this library reserves it for
// the life of the process.  In host code `g_static_scratch` names a host-side
// stand-in, never the device buffer: its device address comes from
// cudaGetSymbolAddress, once per device, below.
static __device__ __align__(256) unsigned char g_static_scratch[SMQA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// The buffer's device address on the current device (looked up once per
// device, with that device current); nullptr after recording the error.
void* scratch_address() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    smqa::set_last_error("cudaGetDevice failed or device id out of range");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[160];
      std::snprintf(msg, sizeof msg, "cudaGetSymbolAddress(static scratch): %s",
                    cudaGetErrorString(e));
      smqa::set_last_error(msg);
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" smqa_status smqa_bwd_static_scratch(const void* q, const void* kv,
                                               const float* attn_sink, const void* o,
                                               const void* dout, const int32_t* topk_idxs,
                                               const float* lse, smqa_shape shape, float sm_scale,
                                               void* dq, void* dkv, float* dsink, unsigned flags,
                                               cudaStream_t stream) {
  // Size check first: a rejected call touches no CUDA state.
  const size_t need = smqa_bwd_workspace_bytes(shape, flags);
  if (need == 0) {
    smqa::set_last_error("unsupported shape (need 1<=H<=128, D in {64,512}, sizes < 2^31)");
    return SMQA_ERR_UNSUPPORTED;
  }
  if (need > static_cast<size_t>(SMQA_STATIC_SCRATCH_BYTES)) {
    char msg[160];
    std::snprintf(msg, sizeof msg,
                  "shape needs %zu bytes of backward scratch; the static buffer holds %zu",
                  need, static_cast<size_t>(SMQA_STATIC_SCRATCH_BYTES));
    smqa::set_last_error(msg);
    return SMQA_ERR_UNSUPPORTED;
  }
  void* scratch = scratch_address();
  if (!scratch) return SMQA_ERR_CUDA;
  // The ordinary backward on that buffer; its first kernel zeroes the fp32
  // accumulator region and overwrites Delta, so no state carries over from
  // the previous call.
  return smqa_bwd(q, kv, attn_sink, o, dout, topk_idxs, lse, shape, sm_scale, dq, dkv, dsink,
                  scratch, static_cast<size_t>(SMQA_STATIC_SCRATCH_BYTES), flags, stream);
}

extern "C" smqa_status smqa_fwd_static_scratch(const void* q, const void* kv,
                                               const float* attn_sink, const int32_t* topk_idxs,
                                               smqa_shape shape, float sm_scale, void* o,
                                               float* lse, unsigned flags, cudaStream_t stream) {
  // The forward's scratch (the exchange pool, D = 512 only) always fits:
  // the size check of smqa_fwd_workspace_bytes only rejects bad shapes.
  const size_t need = smqa_fwd_workspace_bytes(shape);
  if (need > static_cast<size_t>(SMQA_STATIC_SCRATCH_BYTES)) {
    smqa::set_last_error("forward scratch exceeds the static buffer");
    return SMQA_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  if (need != 0) {
    scratch = scratch_address();
    if (!scratch) return SMQA_ERR_CUDA;
  }
  return smqa_fwd(q, kv, attn_sink, topk_idxs, shape, sm_scale, o, lse, scratch,
                  need != 0 ? static_cast<size_t>(SMQA_STATIC_SCRATCH_BYTES) : 0, flags, stream);
}
