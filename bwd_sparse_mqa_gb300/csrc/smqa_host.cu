// smqa_host.cu -- forward, and forward + backward, on HOST buffers.
//
// The entry points copy the inputs into a caller-provided device workspace,
// run the same kernels as smqa_fwd / smqa_bwd and copy the results back,
// token chunk by token chunk, on four streams: one for host->device copies,
// the caller's stream for the forward, one for the backward and one for
// device->host copies.  Events order each chunk's steps, so the copies of one
// chunk overlap the kernels of its neighbours and the forward of chunk c+1
// runs beside the backward of chunk c.  Every token's arithmetic is the one
// smqa_fwd / smqa_bwd perform: O, LSE, dQ and dsink are bit-identical to the
// device-buffer entry points, and dKV is too with SMQA_FLAG_DETERMINISTIC_DKV.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <vector>

#include "sparse_mqa.h"
#include "smqa_internal.h"

namespace {

constexpr int kMaxDevices = 64;
// Chunking: at most about this many chunks per call, none below
// kMinChunkTokens tokens except the last piece of a batch element's
// positions or a last group of whole batch elements (a chunk's kernels then
// still fill every SM).  More chunks shorten the copies before the first
// kernel and after the last one; on the H=128 D=512 topk=2048 S=8192
// workload 8, 16 and 24 chunks measured 20.8, 20.1 and 19.8 ms per forward
// + backward, 32 and 64 no better than 24.  Pieces of S are whole waves --
// multiples of the tokens one backward launch holds on the GPU at once, half
// the SM count for D = 512 (a CTA pair per token), the SM count for D = 64
// -- with the remainder last: a chunk of 4.5 waves leaves half the GPU idle
// for its last wave, and a short last chunk shortens the final copy of dq
// (with dout copied next to q: 19.96 -> 19.71 ms; 19.82 with the remainder
// first).
constexpr int64_t kTargetChunks = 24;
constexpr int64_t kMinChunkTokens = 256;
// The SM count assumed when no device is visible (a GB300).
constexpr int kDefaultSmCount = 152;

size_t r256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

smqa_status fail(smqa_status st, const char* msg) {
  smqa::set_last_error(msg);
  return st;
}

smqa_status cuda_fail(cudaError_t e, const char* where) {
  char msg[200];
  std::snprintf(msg, sizeof msg, "%s: %s", where, cudaGetErrorString(e));
  smqa::set_last_error(msg);
  return SMQA_ERR_CUDA;
}

// The SM count of the current device, or kDefaultSmCount when none answers.
int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return kDefaultSmCount;
  }
  return n;
}

// A run of tokens copied and computed together: batch elements
// [b0, b0 + nb) x positions [s0, s0 + ns).  nb > 1 only when ns = S, so a
// chunk's tokens are contiguous in every [B,S,...] tensor.
struct Chunk {
  int b0, nb, s0, ns;
};

std::vector<Chunk> plan_chunks(const smqa_shape& s, int sm_count) {
  const int64_t total = static_cast<int64_t>(s.B) * s.S;
  const int64_t wave = std::max(1, s.D == 512 ? sm_count / 2 : sm_count);
  int64_t t = std::max((total + kTargetChunks - 1) / kTargetChunks, kMinChunkTokens);
  std::vector<Chunk> out;
  if (s.S >= t) {
    // Pieces of t tokens rounded up to whole waves, the last piece of each S
    // the remainder; all of S in one piece when one such piece would not fit.
    t = std::min<int64_t>((t + wave - 1) / wave * wave, s.S);
    for (int b = 0; b < s.B; ++b)
      for (int64_t a = 0; a < s.S; a += t)
        out.push_back({b, 1, static_cast<int>(a), static_cast<int>(std::min<int64_t>(t, s.S - a))});
  } else {
    // Whole batch elements, k * S >= t tokens per chunk (the last chunk may
    // hold fewer elements).
    const int k = static_cast<int>((t + s.S - 1) / s.S);
    for (int b = 0; b < s.B; b += k) out.push_back({b, std::min(k, s.B - b), 0, s.S});
  }
  return out;
}

// Byte offsets of the device copies inside the workspace (each 256-byte
// aligned; a zero-sized region has no bytes).
struct Layout {
  size_t kv, sink, q, idx, o, lse, fexch;               // forward
  size_t dout, dq, delta, acc, dkv, dsink, bexch;       // backward
  size_t total;
};

Layout layout(const smqa_shape& s, unsigned flags, bool bwd) {
  const size_t tok = static_cast<size_t>(s.B) * s.S;
  const size_t rows = tok * s.H;
  const size_t kvel = static_cast<size_t>(s.B) * s.S_kv * s.D;
  const bool det = (flags & SMQA_FLAG_DETERMINISTIC_DKV) != 0;
  const bool f32 = (flags & SMQA_FLAG_RETURN_DKV_FP32) != 0;
  Layout L{};
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t at = off;
    off += r256(bytes);
    return at;
  };
  L.kv = take(kvel * 2);
  L.sink = take(static_cast<size_t>(s.H) * 4);
  L.q = take(rows * s.D * 2);
  L.idx = take(tok * s.topk * 4);
  L.o = take(rows * s.D * 2);
  L.lse = take(rows * 4);
  L.fexch = take(smqa_fwd_workspace_bytes(s));
  if (bwd) {
    L.dout = take(rows * s.D * 2);
    L.dq = take(rows * s.D * 2);
    L.delta = take(rows * 4);
    L.acc = take(det ? smqa::det_region_bytes(s) : kvel * 4);
    // Without the deterministic mode an fp32 result is the accumulator itself.
    L.dkv = (det || !f32) ? take(kvel * (f32 ? 4 : 2)) : L.acc;
    L.dsink = take(static_cast<size_t>(s.H) * 4);
    L.bexch = take(smqa_bwd_exchange_bytes(s));
  }
  L.total = off;
  return L;
}

// Streams and events the calls of one device share, created on first use
// and kept for the life of the process.  `m` is held while a call enqueues
// its work (the streams keep the calls' work in that order).
struct Side {
  std::mutex m;
  bool ready = false;
  cudaStream_t h2d = nullptr, bwd = nullptr, d2h = nullptr;
  std::vector<cudaEvent_t> ev;
};
Side g_side[kMaxDevices];

// Event slots: fixed ones, then four per chunk.
enum { kEvStart, kEvKv, kEvPost, kEvJoinH2d, kEvJoinBwd, kEvJoinD2h, kEvFixed };
size_t ev_in(size_t c) { return kEvFixed + 4 * c; }       // q, idx of chunk c on the device
size_t ev_do(size_t c) { return kEvFixed + 4 * c + 1; }   // dout of chunk c on the device
size_t ev_fwd(size_t c) { return kEvFixed + 4 * c + 2; }  // forward of chunk c done
size_t ev_bwd(size_t c) { return kEvFixed + 4 * c + 3; }  // backward of chunk c done

smqa_status side_prepare(Side& sd, size_t nev) {
  cudaError_t e;
  if (!sd.ready) {
    e = cudaStreamCreateWithFlags(&sd.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&sd.bwd, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&sd.d2h, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "side stream create");
    sd.ready = true;
  }
  while (sd.ev.size() < nev) {
    cudaEvent_t ev;
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "event create");
    sd.ev.push_back(ev);
  }
  return SMQA_OK;
}

// Host-side arguments of one call.
struct HostArgs {
  const void* q;
  const void* kv;
  const float* sink;
  const int32_t* idx;
  const void* dout;  // null: forward only
  smqa_shape s;
  float sm_scale;
  void* o;
  float* lse;
  void* dq;
  void* dkv;
  float* dsink;  // may be null
  unsigned flags;
};

// Checks that `p` is not device memory (host memory, page-locked or not).
bool is_host_pointer(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();  // older drivers: an unregistered host pointer is an error
    return true;
  }
  return a.type != cudaMemoryTypeDevice;
}

}  // namespace

namespace {

#define SMQA_TRY(call, where)                     \
  do {                                            \
    const cudaError_t e_ = (call);                \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

// Enqueues one call.  Streams are filled in the order host->device copies,
// forward, backward, device->host copies, so every cudaStreamWaitEvent is
// issued after the record it waits for (a wait binds to the latest record).
// On a failure the work enqueued so far stays queued.
smqa_status enqueue(const HostArgs& a, const Layout& L, uint8_t* ws,
                    const std::vector<Chunk>& ch, Side& sd, cudaStream_t st) {
  const smqa_shape& s = a.s;
  const bool bwd = a.dout != nullptr;
  const bool det = (a.flags & SMQA_FLAG_DETERMINISTIC_DKV) != 0;
  const bool f32 = (a.flags & SMQA_FLAG_RETURN_DKV_FP32) != 0;
  const size_t row_bytes = static_cast<size_t>(s.H) * s.D * 2;  // one token of q / o / dout / dq
  const size_t lse_bytes = static_cast<size_t>(s.H) * 4;        // one token of lse / delta
  const size_t idx_bytes = static_cast<size_t>(s.topk) * 4;     // one token of topk_idxs
  const size_t kv_per_b = static_cast<size_t>(s.S_kv) * s.D;    // kv elements per batch element
  const size_t kvel = static_cast<size_t>(s.B) * kv_per_b;
  const size_t n = ch.size();
  const float scale = smqa::effective_scale(a.sm_scale, s.D);
  auto tok0 = [&](size_t c) { return static_cast<size_t>(ch[c].b0) * s.S + ch[c].s0; };
  auto ntok = [&](size_t c) { return static_cast<size_t>(ch[c].nb) * ch[c].ns; };
  auto host = [](const void* p, size_t off) { return static_cast<const uint8_t*>(p) + off; };
  auto host_w = [](void* p, size_t off) { return static_cast<uint8_t*>(p) + off; };
  auto dev = [ws](size_t region, size_t off) { return ws + region + off; };
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;

  // ---- host -> device: kv and sink, then each chunk's q, idx and dout (the
  // backward is the longer stream: its first chunk starts as soon as the
  // forward of chunk 0 is done; dout one chunk later measured 0.5 % slower).
  SMQA_TRY(cudaMemcpyAsync(dev(L.kv, 0), a.kv, kvel * 2, h2d, sd.h2d), "kv copy");
  SMQA_TRY(cudaMemcpyAsync(dev(L.sink, 0), a.sink, lse_bytes, h2d, sd.h2d), "sink copy");
  SMQA_TRY(cudaEventRecord(sd.ev[kEvKv], sd.h2d), "event record");
  auto copy_dout = [&](size_t c) -> smqa_status {
    SMQA_TRY(cudaMemcpyAsync(dev(L.dout, tok0(c) * row_bytes), host(a.dout, tok0(c) * row_bytes),
                             ntok(c) * row_bytes, h2d, sd.h2d), "dout copy");
    SMQA_TRY(cudaEventRecord(sd.ev[ev_do(c)], sd.h2d), "event record");
    return SMQA_OK;
  };
  for (size_t c = 0; c < n; ++c) {
    SMQA_TRY(cudaMemcpyAsync(dev(L.q, tok0(c) * row_bytes), host(a.q, tok0(c) * row_bytes),
                             ntok(c) * row_bytes, h2d, sd.h2d), "q copy");
    SMQA_TRY(cudaMemcpyAsync(dev(L.idx, tok0(c) * idx_bytes), host(a.idx, tok0(c) * idx_bytes),
                             ntok(c) * idx_bytes, h2d, sd.h2d), "topk_idxs copy");
    SMQA_TRY(cudaEventRecord(sd.ev[ev_in(c)], sd.h2d), "event record");
    if (bwd) {
      const smqa_status r = copy_dout(c);
      if (r != SMQA_OK) return r;
    }
  }

  // ---- forward, chunk by chunk, on the caller's stream.
  SMQA_TRY(cudaStreamWaitEvent(st, sd.ev[kEvKv], 0), "stream wait");
  const size_t fexch_bytes = smqa_fwd_workspace_bytes(s);
  for (size_t c = 0; c < n; ++c) {
    const smqa_shape cs{ch[c].nb, ch[c].ns, s.S_kv, s.H, s.D, s.topk};
    SMQA_TRY(cudaStreamWaitEvent(st, sd.ev[ev_in(c)], 0), "stream wait");
    const smqa_status r = smqa_fwd(
        dev(L.q, tok0(c) * row_bytes), dev(L.kv, ch[c].b0 * kv_per_b * 2),
        reinterpret_cast<const float*>(dev(L.sink, 0)),
        reinterpret_cast<const int32_t*>(dev(L.idx, tok0(c) * idx_bytes)), cs, a.sm_scale,
        dev(L.o, tok0(c) * row_bytes), reinterpret_cast<float*>(dev(L.lse, tok0(c) * lse_bytes)),
        fexch_bytes ? dev(L.fexch, 0) : nullptr, fexch_bytes,
        a.flags & SMQA_FLAG_REFERENCE_ROUNDING, st);
    if (r != SMQA_OK) return r;
    SMQA_TRY(cudaEventRecord(sd.ev[ev_fwd(c)], st), "event record");
  }

  // ---- backward, chunk by chunk, on its own stream.
  if (bwd) {
    float* acc = reinterpret_cast<float*>(dev(L.acc, 0));
    unsigned long long* acc_fixed = det ? reinterpret_cast<unsigned long long*>(acc) : nullptr;
    float* delta = reinterpret_cast<float*>(dev(L.delta, 0));
    // The accumulator starts at zero (in the deterministic mode the whole
    // fixed-point region: accumulator, statistics and row counts).
    const size_t acc_bytes = det ? smqa::det_region_bytes(s) : kvel * 4;
    SMQA_TRY(smqa::launch_bwd_preprocess(nullptr, nullptr, nullptr, acc, 0, s.D,
                                         static_cast<int64_t>(acc_bytes / 4), sd.bwd),
             "accumulator clear");
    uint32_t* stats = det ? reinterpret_cast<uint32_t*>(dev(L.acc, smqa::det_stats_offset(s)))
                          : nullptr;
    const int* shift = det ? reinterpret_cast<const int*>(stats + smqa::kDetShift) : nullptr;
    auto delta_chunk = [&](size_t c) -> smqa_status {
      const size_t t0 = tok0(c);
      SMQA_TRY(cudaStreamWaitEvent(sd.bwd, sd.ev[ev_fwd(c)], 0), "stream wait");
      SMQA_TRY(cudaStreamWaitEvent(sd.bwd, sd.ev[ev_do(c)], 0), "stream wait");
      const auto* o = reinterpret_cast<const __nv_bfloat16*>(dev(L.o, t0 * row_bytes));
      const auto* g = reinterpret_cast<const __nv_bfloat16*>(dev(L.dout, t0 * row_bytes));
      SMQA_TRY(smqa::launch_bwd_preprocess(o, g, delta + t0 * s.H, nullptr,
                                           static_cast<int64_t>(ntok(c)) * s.H, s.D, 0, sd.bwd),
               "bwd preprocess launch");
      return SMQA_OK;
    };
    if (det) {
      // The binary point depends on the whole call's inputs: every chunk's
      // Delta first, then the statistics, then the main kernels.
      for (size_t c = 0; c < n; ++c) {
        const smqa_status r = delta_chunk(c);
        if (r != SMQA_OK) return r;
      }
      SMQA_TRY(smqa::launch_bwd_det_stats(
                   reinterpret_cast<const __nv_bfloat16*>(dev(L.q, 0)),
                   reinterpret_cast<const __nv_bfloat16*>(dev(L.kv, 0)),
                   reinterpret_cast<const __nv_bfloat16*>(dev(L.dout, 0)), delta,
                   reinterpret_cast<const int32_t*>(dev(L.idx, 0)), s, stats,
                   stats + smqa::kDetStatsBytes / 4, sd.bwd),
               "bwd statistics launch");
      SMQA_TRY(smqa::launch_bwd_det_scale(s, scale, stats, stats + smqa::kDetStatsBytes / 4,
                                          sd.bwd),
               "bwd scale launch");
    }
    for (size_t c = 0; c < n; ++c) {
      const smqa_shape cs{ch[c].nb, ch[c].ns, s.S_kv, s.H, s.D, s.topk};
      const size_t t0 = tok0(c);
      if (!det) {
        const smqa_status r = delta_chunk(c);
        if (r != SMQA_OK) return r;
      }
      const auto* g = reinterpret_cast<const __nv_bfloat16*>(dev(L.dout, t0 * row_bytes));
      const size_t kv_off = static_cast<size_t>(ch[c].b0) * kv_per_b;
      const smqa_status r = smqa::bwd_main_launch(
          dev(L.q, t0 * row_bytes), dev(L.kv, kv_off * 2), g,
          reinterpret_cast<const int32_t*>(dev(L.idx, t0 * idx_bytes)),
          reinterpret_cast<const float*>(dev(L.lse, t0 * lse_bytes)), delta + t0 * s.H, cs,
          scale, dev(L.dq, t0 * row_bytes),
          det ? reinterpret_cast<float*>(acc_fixed + kv_off) : acc + kv_off,
          det ? acc_fixed + kv_off : nullptr, shift, dev(L.bexch, 0), sd.bwd);
      if (r != SMQA_OK) return r;
      SMQA_TRY(cudaEventRecord(sd.ev[ev_bwd(c)], sd.bwd), "event record");
    }
    if (a.dsink)
      SMQA_TRY(smqa::launch_bwd_sink_grad(reinterpret_cast<const float*>(dev(L.sink, 0)),
                                          reinterpret_cast<const float*>(dev(L.lse, 0)), delta,
                                          reinterpret_cast<float*>(dev(L.dsink, 0)),
                                          static_cast<int64_t>(s.B) * s.S, s.H, sd.bwd),
               "bwd sink gradient launch");
    if (det)
      SMQA_TRY(smqa::launch_bwd_post_fixed(acc_fixed, dev(L.dkv, 0), f32 ? 1 : 0,
                                           static_cast<int64_t>(kvel), shift, sd.bwd),
               "bwd postprocess launch");
    else if (!f32)
      SMQA_TRY(smqa::launch_bwd_postprocess(acc, reinterpret_cast<__nv_bfloat16*>(dev(L.dkv, 0)),
                                            static_cast<int64_t>(kvel), sd.bwd),
               "bwd postprocess launch");
    SMQA_TRY(cudaEventRecord(sd.ev[kEvPost], sd.bwd), "event record");
  }

  // ---- device -> host: each chunk's o and lse after its forward, its dq
  // after its backward (one chunk later).
  auto copy_dq = [&](size_t c) -> smqa_status {
    SMQA_TRY(cudaStreamWaitEvent(sd.d2h, sd.ev[ev_bwd(c)], 0), "stream wait");
    SMQA_TRY(cudaMemcpyAsync(host_w(a.dq, tok0(c) * row_bytes), dev(L.dq, tok0(c) * row_bytes),
                             ntok(c) * row_bytes, d2h, sd.d2h), "dq copy");
    return SMQA_OK;
  };
  for (size_t c = 0; c < n; ++c) {
    SMQA_TRY(cudaStreamWaitEvent(sd.d2h, sd.ev[ev_fwd(c)], 0), "stream wait");
    SMQA_TRY(cudaMemcpyAsync(host_w(a.o, tok0(c) * row_bytes), dev(L.o, tok0(c) * row_bytes),
                             ntok(c) * row_bytes, d2h, sd.d2h), "o copy");
    SMQA_TRY(cudaMemcpyAsync(host_w(a.lse, tok0(c) * lse_bytes), dev(L.lse, tok0(c) * lse_bytes),
                             ntok(c) * lse_bytes, d2h, sd.d2h), "lse copy");
    if (bwd && c >= 1) {
      const smqa_status r = copy_dq(c - 1);
      if (r != SMQA_OK) return r;
    }
  }
  if (bwd) {
    const smqa_status r = copy_dq(n - 1);
    if (r != SMQA_OK) return r;
    SMQA_TRY(cudaStreamWaitEvent(sd.d2h, sd.ev[kEvPost], 0), "stream wait");
    SMQA_TRY(cudaMemcpyAsync(a.dkv, dev(L.dkv, 0), kvel * (f32 ? 4 : 2), d2h, sd.d2h), "dkv copy");
    if (a.dsink)
      SMQA_TRY(cudaMemcpyAsync(a.dsink, dev(L.dsink, 0), lse_bytes, d2h, sd.d2h), "dsink copy");
  }
  return SMQA_OK;
}

#undef SMQA_TRY

smqa_status run(const HostArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t st) {
  const bool bwd = a.dout != nullptr;
  // ---- checks that touch no CUDA state
  const smqa_status sc = smqa::validate_shape(a.s);
  if (sc != SMQA_OK) return sc;
  const unsigned allowed = bwd ? (SMQA_FLAG_REFERENCE_ROUNDING | SMQA_FLAG_RETURN_DKV_FP32 |
                                  SMQA_FLAG_DETERMINISTIC_DKV)
                               : SMQA_FLAG_REFERENCE_ROUNDING;
  if (!a.q || !a.kv || !a.sink || !a.idx || !a.o || !a.lse || !workspace ||
      (bwd && (!a.dq || !a.dkv)) || (a.flags & ~allowed) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(SMQA_ERR_INVALID_ARG, "null pointer, misaligned workspace or bad flags");
  const Layout L = layout(a.s, a.flags, bwd);
  if (workspace_bytes < L.total) {
    char msg[160];
    std::snprintf(msg, sizeof msg, "workspace too small (%zu < %zu bytes)", workspace_bytes,
                  L.total);
    return fail(SMQA_ERR_UNSUPPORTED, msg);
  }
  // ---- pointer kinds: the data on the host, the workspace on this device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(SMQA_ERR_UNSUPPORTED, "device id out of range");
  cudaPointerAttributes wa{};
  e = cudaPointerGetAttributes(&wa, workspace);
  if (e != cudaSuccess || wa.type != cudaMemoryTypeDevice || wa.device != dev) {
    (void)cudaGetLastError();
    return fail(SMQA_ERR_INVALID_ARG, "workspace is not device memory of the current device");
  }
  const void* host_ptrs[] = {a.q, a.kv, a.sink, a.idx, a.dout, a.o, a.lse, a.dq, a.dkv, a.dsink};
  for (const void* p : host_ptrs)
    if (p && !is_host_pointer(p))
      return fail(SMQA_ERR_INVALID_ARG, "a tensor argument is device memory (host buffers expected)");

  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  const std::vector<Chunk> ch = plan_chunks(a.s, sms);
  Side& sd = g_side[dev];
  std::lock_guard<std::mutex> lk(sd.m);
  smqa_status r = side_prepare(sd, kEvFixed + 4 * ch.size());
  if (r != SMQA_OK) return r;
  // Everything starts after the work already on the caller's stream ...
  e = cudaEventRecord(sd.ev[kEvStart], st);
  if (e != cudaSuccess) return cuda_fail(e, "event record");
  for (cudaStream_t x : {sd.h2d, sd.bwd, sd.d2h}) {
    e = cudaStreamWaitEvent(x, sd.ev[kEvStart], 0);
    if (e != cudaSuccess) return cuda_fail(e, "stream wait");
  }
  r = enqueue(a, L, static_cast<uint8_t*>(workspace), ch, sd, st);
  // ... and the caller's stream resumes after everything this call enqueued
  // (also after a failure part-way, so nothing of it outlives the call's
  // place in the caller's stream order).
  const int join_ev[3] = {kEvJoinH2d, kEvJoinBwd, kEvJoinD2h};
  const cudaStream_t join_st[3] = {sd.h2d, sd.bwd, sd.d2h};
  for (int i = 0; i < 3; ++i) {
    e = cudaEventRecord(sd.ev[join_ev[i]], join_st[i]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, sd.ev[join_ev[i]], 0);
    if (e != cudaSuccess && r == SMQA_OK) r = cuda_fail(e, "stream join");
  }
  return r;
}

}  // namespace

extern "C" {

int smqa_host_chunk_plan(smqa_shape shape, int32_t* out, int max_chunks) {
  if (smqa::validate_shape(shape) != SMQA_OK) return 0;
  const std::vector<Chunk> ch = plan_chunks(shape, current_sm_count());
  const int n = static_cast<int>(ch.size());
  for (int c = 0; out && c < n && c < max_chunks; ++c) {
    out[4 * c] = ch[c].b0;
    out[4 * c + 1] = ch[c].nb;
    out[4 * c + 2] = ch[c].s0;
    out[4 * c + 3] = ch[c].ns;
  }
  return n;
}

size_t smqa_fwd_host_workspace_bytes(smqa_shape shape) {
  if (smqa::validate_shape(shape) != SMQA_OK) return 0;
  return layout(shape, 0, false).total;
}

size_t smqa_fwd_bwd_host_workspace_bytes(smqa_shape shape, unsigned flags) {
  if (smqa::validate_shape(shape) != SMQA_OK) return 0;
  return layout(shape, flags, true).total;
}

smqa_status smqa_fwd_host(const void* q, const void* kv, const float* attn_sink,
                          const int32_t* topk_idxs, smqa_shape shape, float sm_scale, void* o,
                          float* lse, void* workspace, size_t workspace_bytes, unsigned flags,
                          cudaStream_t stream) {
  const HostArgs a{q, kv, attn_sink, topk_idxs, nullptr, shape, sm_scale, o, lse,
                   nullptr, nullptr, nullptr, flags};
  return run(a, workspace, workspace_bytes, stream);
}

smqa_status smqa_fwd_bwd_host(const void* q, const void* kv, const float* attn_sink,
                              const int32_t* topk_idxs, const void* dout, smqa_shape shape,
                              float sm_scale, void* o, float* lse, void* dq, void* dkv,
                              float* dsink, void* workspace, size_t workspace_bytes,
                              unsigned flags, cudaStream_t stream) {
  if (!dout) return fail(SMQA_ERR_INVALID_ARG, "dout is null");
  const HostArgs a{q, kv, attn_sink, topk_idxs, dout, shape, sm_scale, o, lse,
                   dq, dkv, dsink, flags};
  return run(a, workspace, workspace_bytes, stream);
}

}  // extern "C"
