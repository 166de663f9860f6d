// smqa_api.cu -- the library's C ABI (include/sparse_mqa.h): host-side
// argument checks, TMA tensor-map encoding, kernel launches on the caller's
// stream and the device status word.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "sparse_mqa.h"
#include "smqa_internal.h"

namespace {

// Set by kernels whose bounded waits ran out (see smqa_ptx.cuh).
__device__ int g_smqa_status = 0;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
std::mutex g_mutex;
thread_local char g_last_error[256] = "no error";

void note_cuda(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", where, cudaGetErrorString(e));
}

smqa_status cuda_fail(cudaError_t e, const char* where) {
  note_cuda(e, where);
  return SMQA_ERR_CUDA;
}

// Device address of the status word on the current device.
int* status_ptr(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mutex);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_smqa_status);
    if (*err != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

uint64_t default_wait_limit_ns() {
  static uint64_t v = [] {
    const char* s = std::getenv("SMQA_WAIT_LIMIT_NS");
    if (s && *s) {
      const unsigned long long x = std::strtoull(s, nullptr, 10);
      if (x > 0) return static_cast<uint64_t>(x);
    }
    return static_cast<uint64_t>(4000000000ull);
  }();
  return v;
}

// A limit set through smqa_set_wait_limit_ns (0: none, use the default).
std::atomic<uint64_t> g_wait_limit_override{0};
// The CTA set through smqa_debug_stall (-1: none).
std::atomic<int> g_stall_cta{-1};

uint64_t wait_limit_ns() {
  const uint64_t o = g_wait_limit_override.load(std::memory_order_relaxed);
  return o != 0 ? o : default_wait_limit_ns();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// bf16 matrix [outer, inner] (row-major), boxes of box_inner x box_outer with
// the 128-byte swizzle that the tcgen05 K-major / MN-major operands expect.
bool encode_bf16_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                    uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) {
    std::snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_last_error, sizeof g_last_error, "cuTensorMapEncodeTiled failed (%d)",
                  static_cast<int>(r));
    return false;
  }
  return true;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

smqa_status check_shape(const smqa_shape& s) {
  if (s.B <= 0 || s.S <= 0 || s.S_kv <= 0 || s.H <= 0 || s.D <= 0 || s.topk <= 0) {
    std::snprintf(g_last_error, sizeof g_last_error, "non-positive size in shape");
    return SMQA_ERR_INVALID_ARG;
  }
  const int64_t lim = int64_t{1} << 31;
  if (s.H > 128 || (s.D != 64 && s.D != 512) ||
      static_cast<int64_t>(s.B) * s.S_kv * s.D >= lim ||
      static_cast<int64_t>(s.B) * s.S * s.H >= lim ||
      static_cast<int64_t>(s.B) * s.S >= (lim >> 1)) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "unsupported shape (need 1<=H<=128, D in {64,512}, sizes < 2^31)");
    return SMQA_ERR_UNSUPPORTED;
  }
  return SMQA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Exchange pool of the D = 512 forward and backward: slot flags, then the
// slots.
constexpr size_t kExchFlagBytes = 4096;
constexpr int kExchSlots = 96;
// The slot flags, then the backward's token counter, fit the flag block.
static_assert((kExchSlots + 1) * sizeof(int) <= kExchFlagBytes, "exchange flag block");

size_t exchange_bytes(const smqa_shape& s) {
  return s.D == 512 ? kExchFlagBytes + static_cast<size_t>(kExchSlots) * smqa::kBwdSlotBytes : 0;
}

size_t fwd_exchange_bytes(const smqa_shape& s) {
  return s.D == 512 ? kExchFlagBytes + static_cast<size_t>(kExchSlots) * smqa::kFwdSlotBytes : 0;
}

smqa_status bwd_main_impl(const void* q, const void* kv, const void* dout, const int32_t* idx,
                          const float* lse, const float* delta, const smqa_shape& s, float scale,
                          void* dq, float* acc, void* exch, cudaStream_t stream,
                          unsigned long long* acc_fixed = nullptr,
                          const int* fix_shift = nullptr) {
  cudaError_t e;
  int* st = status_ptr(&e);
  if (!st) return cuda_fail(e, "status word");
  if (exchange_bytes(s) != 0) {
    // Every slot free at launch (the kernel's pairs claim and release them),
    // and the token counter the pairs take their tokens from at zero.
    e = cudaMemsetAsync(exch, 0, (kExchSlots + 1) * sizeof(int), stream);
    if (e != cudaSuccess) return cuda_fail(e, "exchange flags clear");
  }
  CUtensorMap tq, tdo;
  const uint64_t T = static_cast<uint64_t>(s.B) * s.S;
  if (!encode_bf16_2d(&tq, q, s.D, T * s.H, 64, static_cast<uint32_t>(s.H)) ||
      !encode_bf16_2d(&tdo, dout, s.D, T * s.H, 64, static_cast<uint32_t>(s.H)))
    return SMQA_ERR_CUDA;
  smqa::BwdParams p{};
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.idx = idx;
  p.lse = lse;
  p.delta = delta;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dkv_acc = acc;
  p.dkv_fix = acc_fixed;
  p.fix_shift = fix_shift;
  p.det = acc_fixed != nullptr ? 1 : 0;
  p.S = s.S;
  p.S_kv = s.S_kv;
  p.H = s.H;
  p.D = s.D;
  p.topk = s.topk;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = st;
  p.limit_ns = wait_limit_ns();
  p.stall_cta = g_stall_cta.load(std::memory_order_relaxed);
  if (exchange_bytes(s) != 0) {
    p.slot_flags = static_cast<int*>(exch);
    p.exch = static_cast<uint8_t*>(exch) + kExchFlagBytes;
    p.nslots = kExchSlots;
    p.tok_counter = static_cast<int*>(exch) + kExchSlots;
  }
  e = smqa::launch_bwd_main(tq, tdo, p, static_cast<int>(T), stream);
  if (e != cudaSuccess) return cuda_fail(e, "bwd main launch");
  return SMQA_OK;
}

}  // namespace

namespace smqa {
void set_last_error(const char* msg) { std::snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

smqa_status validate_shape(const smqa_shape& s) { return check_shape(s); }

float effective_scale(float sm_scale, int D) {
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return 1.0f / std::sqrt(static_cast<float>(D));
  return sm_scale;
}

smqa_status bwd_main_launch(const void* q, const void* kv, const void* dout, const int32_t* idx,
                            const float* lse, const float* delta, const smqa_shape& s,
                            float scale, void* dq, float* acc, unsigned long long* acc_fixed,
                            const int* fix_shift, void* exch, cudaStream_t stream) {
  return bwd_main_impl(q, kv, dout, idx, lse, delta, s, scale, dq, acc, exch, stream, acc_fixed,
                       fix_shift);
}
}  // namespace smqa

using smqa::effective_scale;

extern "C" {

int smqa_abi_version(void) { return SMQA_ABI_VERSION; }

const char* smqa_status_string(smqa_status status) {
  switch (status) {
    case SMQA_OK: return "SMQA_OK";
    case SMQA_ERR_INVALID_ARG: return "SMQA_ERR_INVALID_ARG";
    case SMQA_ERR_UNSUPPORTED: return "SMQA_ERR_UNSUPPORTED";
    case SMQA_ERR_CUDA: return "SMQA_ERR_CUDA";
    case SMQA_ERR_DEVICE_TIMEOUT: return "SMQA_ERR_DEVICE_TIMEOUT";
  }
  return "SMQA_ERR_UNKNOWN";
}

const char* smqa_last_error(void) { return g_last_error; }

smqa_status smqa_fwd(const void* q, const void* kv, const float* attn_sink,
                     const int32_t* topk_idxs, smqa_shape shape, float sm_scale, void* o,
                     float* lse, void* workspace, size_t workspace_bytes, unsigned flags,
                     cudaStream_t stream) {
  const smqa_status sc = check_shape(shape);
  if (sc != SMQA_OK) return sc;
  const size_t need = fwd_exchange_bytes(shape);
  if (!q || !kv || !attn_sink || !topk_idxs || !o || !lse || (need != 0 && !workspace) ||
      (flags & ~SMQA_FLAG_REFERENCE_ROUNDING) || !aligned(q, 16) || !aligned(kv, 16) ||
      !aligned(o, 16) || !aligned(attn_sink, 4) || !aligned(topk_idxs, 4) || !aligned(lse, 4) ||
      !aligned(workspace, 256)) {
    std::snprintf(g_last_error, sizeof g_last_error, "null/misaligned pointer or bad flags");
    return SMQA_ERR_INVALID_ARG;
  }
  if (workspace_bytes < need) {
    std::snprintf(g_last_error, sizeof g_last_error, "workspace too small (%zu < %zu bytes)",
                  workspace_bytes, need);
    return SMQA_ERR_UNSUPPORTED;
  }
  cudaError_t e;
  int* st = status_ptr(&e);
  if (!st) return cuda_fail(e, "status word");
  CUtensorMap tq;
  const uint64_t T = static_cast<uint64_t>(shape.B) * shape.S;
  if (!encode_bf16_2d(&tq, q, shape.D, T * shape.H, 64, static_cast<uint32_t>(shape.H)))
    return SMQA_ERR_CUDA;
  if (need != 0) {
    // Every slot free at launch (the kernel's pairs claim and release them),
    // and the token counter the pairs take their tokens from at zero.
    e = cudaMemsetAsync(workspace, 0, (kExchSlots + 1) * sizeof(int), stream);
    if (e != cudaSuccess) return cuda_fail(e, "exchange flags clear");
  }
  const float scale = effective_scale(sm_scale, shape.D);
  smqa::FwdParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.idx = topk_idxs;
  p.sink = attn_sink;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.S = shape.S;
  p.S_kv = shape.S_kv;
  p.H = shape.H;
  p.D = shape.D;
  p.topk = shape.topk;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.ref_round = (flags & SMQA_FLAG_REFERENCE_ROUNDING) ? 1 : 0;
  p.status = st;
  p.limit_ns = wait_limit_ns();
  p.stall_cta = g_stall_cta.load(std::memory_order_relaxed);
  if (need != 0) {
    p.slot_flags = static_cast<int*>(workspace);
    p.exch = static_cast<uint8_t*>(workspace) + kExchFlagBytes;
    p.nslots = kExchSlots;
    p.tok_counter = static_cast<int*>(workspace) + kExchSlots;
  }
  e = smqa::launch_fwd(tq, p, static_cast<int>(T), stream);
  if (e != cudaSuccess) return cuda_fail(e, "fwd launch");
  return SMQA_OK;
}

size_t smqa_fwd_workspace_bytes(smqa_shape shape) {
  if (check_shape(shape) != SMQA_OK) return 0;
  return fwd_exchange_bytes(shape);
}

size_t smqa_bwd_workspace_bytes(smqa_shape shape, unsigned flags) {
  if (check_shape(shape) != SMQA_OK) return 0;
  size_t bytes = 0;
  const size_t elems = static_cast<size_t>(shape.B) * shape.S_kv * shape.D;
  if (flags & SMQA_FLAG_DETERMINISTIC_DKV)
    bytes += smqa::det_region_bytes(shape);  // fixed-point accumulator, statistics, row counts
  else if (!(flags & SMQA_FLAG_RETURN_DKV_FP32))
    bytes += round256(elems * sizeof(float));
  bytes += round256(static_cast<size_t>(shape.B) * shape.S * shape.H * sizeof(float));
  bytes += round256(exchange_bytes(shape));
  return bytes;
}

size_t smqa_bwd_exchange_bytes(smqa_shape shape) {
  if (check_shape(shape) != SMQA_OK) return 0;
  return exchange_bytes(shape);
}

smqa_status smqa_bwd_preprocess(const void* o, const void* dout, smqa_shape shape, float* delta,
                                float* dkv_accum, cudaStream_t stream) {
  const smqa_status sc = check_shape(shape);
  if (sc != SMQA_OK) return sc;
  if (!o || !dout || !delta || !dkv_accum || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(delta, 4) || !aligned(dkv_accum, 16)) {
    std::snprintf(g_last_error, sizeof g_last_error, "null or misaligned pointer");
    return SMQA_ERR_INVALID_ARG;
  }
  const int64_t rows = static_cast<int64_t>(shape.B) * shape.S * shape.H;
  const int64_t acc = static_cast<int64_t>(shape.B) * shape.S_kv * shape.D;
  const cudaError_t e = smqa::launch_bwd_preprocess(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta,
      dkv_accum, rows, shape.D, acc, stream);
  if (e != cudaSuccess) return cuda_fail(e, "bwd preprocess launch");
  return SMQA_OK;
}

smqa_status smqa_bwd_main(const void* q, const void* kv, const float* attn_sink, const void* dout,
                          const int32_t* topk_idxs, const float* lse, const float* delta,
                          smqa_shape shape, float sm_scale, void* dq, float* dkv_accum,
                          void* exchange, size_t exchange_bytes_given, cudaStream_t stream) {
  const smqa_status sc = check_shape(shape);
  if (sc != SMQA_OK) return sc;
  const size_t need = exchange_bytes(shape);
  if (!q || !kv || !attn_sink || !dout || !topk_idxs || !lse || !delta || !dq || !dkv_accum ||
      (need != 0 && !exchange) || !aligned(q, 16) || !aligned(kv, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(topk_idxs, 4) || !aligned(lse, 4) || !aligned(delta, 4) ||
      !aligned(dkv_accum, 16) || !aligned(exchange, 256)) {
    std::snprintf(g_last_error, sizeof g_last_error, "null or misaligned pointer");
    return SMQA_ERR_INVALID_ARG;
  }
  if (exchange_bytes_given < need) {
    std::snprintf(g_last_error, sizeof g_last_error, "exchange pool too small (%zu < %zu bytes)",
                  exchange_bytes_given, need);
    return SMQA_ERR_UNSUPPORTED;
  }
  return bwd_main_impl(q, kv, dout, topk_idxs, lse, delta, shape,
                       effective_scale(sm_scale, shape.D), dq, dkv_accum, exchange, stream);
}

smqa_status smqa_bwd_sink_grad(const float* attn_sink, const float* lse, const float* delta,
                               smqa_shape shape, float* dsink, cudaStream_t stream) {
  const smqa_status sc = check_shape(shape);
  if (sc != SMQA_OK) return sc;
  if (!attn_sink || !lse || !delta || !dsink || !aligned(attn_sink, 4) || !aligned(lse, 4) ||
      !aligned(delta, 4) || !aligned(dsink, 4)) {
    std::snprintf(g_last_error, sizeof g_last_error, "null or misaligned pointer");
    return SMQA_ERR_INVALID_ARG;
  }
  const cudaError_t e = smqa::launch_bwd_sink_grad(
      attn_sink, lse, delta, dsink, static_cast<int64_t>(shape.B) * shape.S, shape.H, stream);
  if (e != cudaSuccess) return cuda_fail(e, "bwd sink gradient launch");
  return SMQA_OK;
}

smqa_status smqa_bwd_postprocess(const float* dkv_accum, smqa_shape shape, void* dkv_bf16,
                                 cudaStream_t stream) {
  const smqa_status sc = check_shape(shape);
  if (sc != SMQA_OK) return sc;
  if (!dkv_accum || !dkv_bf16 || !aligned(dkv_accum, 16) || !aligned(dkv_bf16, 16)) {
    std::snprintf(g_last_error, sizeof g_last_error, "null or misaligned pointer");
    return SMQA_ERR_INVALID_ARG;
  }
  const int64_t n = static_cast<int64_t>(shape.B) * shape.S_kv * shape.D;
  const cudaError_t e =
      smqa::launch_bwd_postprocess(dkv_accum, static_cast<__nv_bfloat16*>(dkv_bf16), n, stream);
  if (e != cudaSuccess) return cuda_fail(e, "bwd postprocess launch");
  return SMQA_OK;
}

smqa_status smqa_bwd(const void* q, const void* kv, const float* attn_sink, const void* o,
                     const void* dout, const int32_t* topk_idxs, const float* lse,
                     smqa_shape shape, float sm_scale, void* dq, void* dkv, float* dsink,
                     void* workspace, size_t workspace_bytes, unsigned flags,
                     cudaStream_t stream) {
  const smqa_status sc = check_shape(shape);
  if (sc != SMQA_OK) return sc;
  if (!q || !kv || !attn_sink || !o || !dout || !topk_idxs || !lse || !dq || !dkv || !workspace ||
      (flags & ~(SMQA_FLAG_RETURN_DKV_FP32 | SMQA_FLAG_DETERMINISTIC_DKV)) || !aligned(q, 16) ||
      !aligned(kv, 16) || !aligned(o, 16) || !aligned(dout, 16) || !aligned(dq, 16) ||
      !aligned(dkv, 16) || !aligned(workspace, 16) || !aligned(attn_sink, 4) ||
      !aligned(topk_idxs, 4) || !aligned(lse, 4) || !aligned(dsink, 4)) {
    std::snprintf(g_last_error, sizeof g_last_error, "null/misaligned pointer or bad flags");
    return SMQA_ERR_INVALID_ARG;
  }
  if (workspace_bytes < smqa_bwd_workspace_bytes(shape, flags)) {
    std::snprintf(g_last_error, sizeof g_last_error, "workspace too small");
    return SMQA_ERR_UNSUPPORTED;
  }
  const bool fp32_out = (flags & SMQA_FLAG_RETURN_DKV_FP32) != 0;
  const bool det = (flags & SMQA_FLAG_DETERMINISTIC_DKV) != 0;
  const int64_t elems = static_cast<int64_t>(shape.B) * shape.S_kv * shape.D;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* acc = (fp32_out && !det) ? static_cast<float*>(dkv) : reinterpret_cast<float*>(ws);
  unsigned long long* acc_fixed = det ? reinterpret_cast<unsigned long long*>(ws) : nullptr;
  const size_t acc_bytes =
      det ? smqa::det_region_bytes(shape)
          : (fp32_out ? 0 : round256(static_cast<size_t>(elems) * sizeof(float)));
  float* delta = reinterpret_cast<float*>(ws + acc_bytes);
  void* exch = ws + acc_bytes +
               round256(static_cast<size_t>(shape.B) * shape.S * shape.H * sizeof(float));
  const float scale = effective_scale(sm_scale, shape.D);
  smqa_status r;
  uint32_t* stats = nullptr;
  if (det) {
    // Delta, and the whole fixed-point region zeroed (accumulator,
    // statistics and row counts); then the statistics and the binary point.
    stats = reinterpret_cast<uint32_t*>(ws + smqa::det_stats_offset(shape));
    uint32_t* counts = stats + smqa::kDetStatsBytes / sizeof(uint32_t);
    cudaError_t e = smqa::launch_bwd_preprocess(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta,
        acc, static_cast<int64_t>(shape.B) * shape.S * shape.H, shape.D,
        static_cast<int64_t>(acc_bytes / sizeof(float)), stream);
    if (e != cudaSuccess) return cuda_fail(e, "bwd preprocess launch");
    e = smqa::launch_bwd_det_stats(static_cast<const __nv_bfloat16*>(q),
                                   static_cast<const __nv_bfloat16*>(kv),
                                   static_cast<const __nv_bfloat16*>(dout), delta, topk_idxs,
                                   shape, stats, counts, stream);
    if (e != cudaSuccess) return cuda_fail(e, "bwd statistics launch");
    e = smqa::launch_bwd_det_scale(shape, scale, stats, counts, stream);
    if (e != cudaSuccess) return cuda_fail(e, "bwd scale launch");
  } else {
    r = smqa_bwd_preprocess(o, dout, shape, delta, acc, stream);
    if (r != SMQA_OK) return r;
  }
  if (dsink) {
    r = smqa_bwd_sink_grad(attn_sink, lse, delta, shape, dsink, stream);
    if (r != SMQA_OK) return r;
  }
  const int* shift = det ? reinterpret_cast<const int*>(stats + smqa::kDetShift) : nullptr;
  r = bwd_main_impl(q, kv, dout, topk_idxs, lse, delta, shape, scale, dq, acc, exch, stream,
                    acc_fixed, shift);
  if (r != SMQA_OK) return r;
  if (det) {
    const cudaError_t e =
        smqa::launch_bwd_post_fixed(acc_fixed, dkv, fp32_out ? 1 : 0, elems, shift, stream);
    if (e != cudaSuccess) return cuda_fail(e, "bwd postprocess launch");
    return SMQA_OK;
  }
  if (!fp32_out) return smqa_bwd_postprocess(acc, shape, dkv, stream);
  return SMQA_OK;
}

uint64_t smqa_set_wait_limit_ns(uint64_t ns) {
  const uint64_t before = wait_limit_ns();
  g_wait_limit_override.store(ns, std::memory_order_relaxed);
  return before;
}

}  // extern "C"

namespace {

// The indexer backward's argument checks and launch, for both layouts.
smqa_status indexer_impl(const void* q, const float* w, const void* k, const int32_t* idx,
                         const float* g, const smqa_shape& s, bool batched, void* dq,
                         cudaStream_t stream) {
  if (s.B <= 0 || s.S <= 0 || s.S_kv <= 0 || s.H <= 0 || s.D <= 0 || s.topk <= 0) {
    std::snprintf(g_last_error, sizeof g_last_error, "non-positive size in shape");
    return SMQA_ERR_INVALID_ARG;
  }
  const int64_t lim = int64_t{1} << 31;
  if (s.H > 128 || (s.D != 64 && s.D != 128) ||
      static_cast<int64_t>(s.B) * s.S_kv * s.D >= lim ||
      static_cast<int64_t>(s.B) * s.S * s.H * s.D >= lim ||
      static_cast<int64_t>(s.B) * s.S * s.topk >= lim) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "unsupported indexer shape (need 1<=H<=128, D in {64,128}, sizes < 2^31)");
    return SMQA_ERR_UNSUPPORTED;
  }
  if (!batched && s.B != 1) {
    std::snprintf(g_last_error, sizeof g_last_error,
                  "smqa_indexer_bwd takes one batch element (B = 1)");
    return SMQA_ERR_INVALID_ARG;
  }
  if (!q || !w || !k || !idx || !g || !dq || !aligned(q, 16) || !aligned(k, 16) ||
      !aligned(dq, 16) || !aligned(w, 4) || !aligned(idx, 4) || !aligned(g, 4)) {
    std::snprintf(g_last_error, sizeof g_last_error, "null or misaligned pointer");
    return SMQA_ERR_INVALID_ARG;
  }
  cudaError_t e;
  int* st = status_ptr(&e);
  if (!st) return cuda_fail(e, "status word");
  const uint64_t rows = static_cast<uint64_t>(s.B) * s.S * s.H;
  CUtensorMap tq, tdq;
  if (!encode_bf16_2d(&tq, q, s.D, rows, 64, static_cast<uint32_t>(s.H)) ||
      !encode_bf16_2d(&tdq, dq, s.D, rows, 64, static_cast<uint32_t>(s.H)))
    return SMQA_ERR_CUDA;
  smqa::IdxParams p{};
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.idx = idx;
  p.g = g;
  p.w = w;
  p.B = s.B;
  p.S = s.S;
  p.S_kv = s.S_kv;
  p.H = s.H;
  p.D = s.D;
  p.topk = s.topk;
  p.q_tok_rows = batched ? static_cast<int64_t>(s.B) * s.H : s.H;
  p.q_b_rows = batched ? s.H : 0;
  p.k_row_stride = batched ? static_cast<int64_t>(s.B) * s.D : s.D;
  p.k_b_stride = batched ? s.D : 0;
  p.status = st;
  p.limit_ns = wait_limit_ns();
  p.stall_cta = g_stall_cta.load(std::memory_order_relaxed);
  e = smqa::launch_indexer_bwd(tq, tdq, p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "indexer bwd launch");
  return SMQA_OK;
}

}  // namespace

extern "C" {

smqa_status smqa_indexer_bwd(const void* index_q, const float* weights, const void* index_k,
                             const int32_t* topk_indices, const float* grad_scores,
                             smqa_shape shape, void* dq, cudaStream_t stream) {
  return indexer_impl(index_q, weights, index_k, topk_indices, grad_scores, shape, false, dq,
                      stream);
}

smqa_status smqa_batched_indexer_bwd(const void* index_q, const float* weights,
                                     const void* index_k, const int32_t* topk_indices,
                                     const float* grad_scores, smqa_shape shape, void* dq,
                                     cudaStream_t stream) {
  return indexer_impl(index_q, weights, index_k, topk_indices, grad_scores, shape, true, dq,
                      stream);
}

void smqa_debug_stall(int cta) { g_stall_cta.store(cta < 0 ? -1 : cta, std::memory_order_relaxed); }

smqa_status smqa_device_status(int clear) {
  cudaError_t e;
  int* st = status_ptr(&e);
  if (!st) return cuda_fail(e, "status word");
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
  int v = 0;
  e = cudaMemcpy(&v, st, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (clear) {
    const int zero = 0;
    e = cudaMemcpy(st, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
  }
  return v ? SMQA_ERR_DEVICE_TIMEOUT : SMQA_OK;
}

}  // extern "C"
