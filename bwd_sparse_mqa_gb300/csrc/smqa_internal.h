// smqa_internal.h -- parameter blocks and launchers shared by the library's
// translation units (not part of the public C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sparse_mqa.h"

namespace smqa {

struct FwdParams {
  const __nv_bfloat16* q;   // [B,S,H,D]
  const __nv_bfloat16* kv;  // [B,S_kv,D]
  const int32_t* idx;    // [B,S,topk]
  const float* sink;     // [H]
  __nv_bfloat16* o;      // [B,S,H,D]
  float* lse;            // [B,S,H]
  int S, S_kv, H, D, topk;
  float scale;           // sm_scale
  float scale_log2;      // sm_scale * log2(e)
  int ref_round;         // 1: exp2 argument as (score * scale) * log2(e)
  int* status;           // device status word
  uint64_t limit_ns;     // bounded-wait limit
  int stall_cta;         // test hook: this CTA stalls after its first MMA (-1: none)
  // Persistent grid: `clusters` CTAs (pairs for D = 512) over `tokens`
  // tokens (set at launch).  With tok_counter (zero before the launch) a
  // pair takes its next token from it; without, cluster c takes tokens
  // c, c + clusters, ...
  int tokens, clusters;
  int* tok_counter;
  // D split across a CTA pair: the pairs trade their partial scores through
  // an L2-resident pool of nslots slots (kFwdSlotBytes each); slot_flags[s]
  // is 1 while a pair holds slot s (all zero before the launch).
  uint8_t* exch;
  int* slot_flags;
  int nslots;
};

struct BwdParams {
  const __nv_bfloat16* kv;  // [B,S_kv,D]
  const int32_t* idx;    // [B,S,topk]
  const float* lse;      // [B,S,H]  log2 LSE from the forward
  const float* delta;    // [B,S,H]  rowsum(O * dO)
  __nv_bfloat16* dq;     // [B,S,H,D]
  float* dkv_acc;        // [B,S_kv,D] fp32 accumulator (zeroed beforehand)
  // Deterministic mode (det != 0): the accumulator is dkv_fix instead, each
  // element a signed fixed-point integer with the per-call binary point
  // *fix_shift (value = integer * 2^-shift; zeroed beforehand).
  unsigned long long* dkv_fix;
  const int* fix_shift;
  int det;
  int S, S_kv, H, D, topk;
  float scale;           // sm_scale
  float scale_log2;      // sm_scale * log2(e)
  int* status;
  uint64_t limit_ns;
  int stall_cta;         // test hook: this CTA stalls after its first MMA (-1: none)
  // Persistent grid: `clusters` CTAs (pairs for D = 512) over `tokens`
  // tokens (set at launch).  With tok_counter (zero before the launch) a
  // pair takes its next token from it; without, cluster c takes tokens
  // c, c + clusters, ...
  int tokens, clusters;
  int* tok_counter;
  // D split across a CTA pair: the pairs trade their partial S / dP through
  // an L2-resident pool of nslots slots (kBwdSlotBytes each); slot_flags[s]
  // is 1 while a pair holds slot s (all zero before the launch).
  uint8_t* exch;
  int* slot_flags;
  int nslots;
};

// Lightning-indexer backward: dq[t,h] = w[t,h] sum_j g[t,j] [q.k_j > 0] k_j.
// Token (s, b) has its H rows of q, weights and dq at row
// s * q_tok_rows + b * q_b_rows ([S,H,D] per element: H, 0; the batched
// [S,B,H,D]: B*H, H); key row r of element b starts at element
// r * k_row_stride + b * k_b_stride; indices and grad_scores are [B,S,topk].
struct IdxParams {
  const __nv_bfloat16* k;
  const int32_t* idx;
  const float* g;
  const float* w;
  int B, S, S_kv, H, D, topk;
  int64_t q_tok_rows, q_b_rows;
  int64_t k_row_stride, k_b_stride;
  int* status;
  uint64_t limit_ns;
  int stall_cta;         // test hook: this CTA stalls after its first MMA (-1: none)
};

// One exchange slot of the forward: two receivers x six block buffers x
// 16.5 KB (the partial scores of 128 heads x 64 slots as int16 mantissas
// with one int32 power-of-two exponent per head).
constexpr size_t kFwdSlotBytes = 2 * 6 * (16384 + 512);
// One exchange slot of the backward: two receivers x two block parities x
// 33 KB (the partial S and dP of 128 heads x 64 slots as int16 mantissas
// with one packed pair of power-of-two exponents per head and 32-slot half).
constexpr size_t kBwdSlotBytes = 2 * 2 * (32768 + 1024);

// The deterministic mode's accumulator region: the fixed-point accumulator
// (8 bytes per element), a block of per-call statistics (kDet* words, 32-bit
// each) and a reference count per kv row ([B, S_kv] uint32).  The whole
// region is zeroed before use, as a multiple of 16 bytes.
constexpr size_t kDetStatsBytes = 256;
enum : int {
  kDetMaxAbsDout = 0,   // max |dO| (fp32 bits)
  kDetMaxDoutSq = 1,    // max over (token, head) rows of |dO row|^2 (fp32 bits)
  kDetMaxKvSq = 2,      // max over kv rows of |kv row|^2 (fp32 bits)
  kDetMaxAbsQ = 3,      // max |q| (fp32 bits)
  kDetMaxAbsDelta = 4,  // max |Delta| (fp32 bits)
  kDetMaxCount = 5,     // most slots naming one kv row
  kDetShift = 6,        // the binary point k: value = integer * 2^-k
  kDetTicket = 7,       // blocks of the scale kernel done
};
inline size_t det_region_bytes(const smqa_shape& s) {
  const size_t elems = static_cast<size_t>(s.B) * s.S_kv * s.D;
  const size_t rows = static_cast<size_t>(s.B) * s.S_kv;
  auto r256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  return r256(elems * 8) + kDetStatsBytes + r256(rows * 4);
}
inline size_t det_stats_offset(const smqa_shape& s) {
  const size_t elems = static_cast<size_t>(s.B) * s.S_kv * s.D;
  return (elems * 8 + 255) & ~static_cast<size_t>(255);
}

// Records `msg` as the text smqa_last_error() returns on this thread.
void set_last_error(const char* msg);

cudaError_t launch_fwd(const CUtensorMap& tm_q, const FwdParams& p, int tokens,
                       cudaStream_t stream);
cudaError_t launch_bwd_main(const CUtensorMap& tm_q, const CUtensorMap& tm_do,
                            const BwdParams& p, int tokens,
                            cudaStream_t stream);
cudaError_t launch_indexer_bwd(const CUtensorMap& tm_q, const CUtensorMap& tm_dq,
                               const IdxParams& p, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                  float* delta, float* dkv_acc, int64_t rows, int D,
                                  int64_t acc_elems, cudaStream_t stream);
cudaError_t launch_bwd_sink_grad(const float* sink, const float* lse, const float* delta,
                                float* dsink, int64_t tokens, int H, cudaStream_t stream);
cudaError_t launch_bwd_post_fixed(const unsigned long long* acc, void* out, int fp32_out,
                                 int64_t elems, const int* shift, cudaStream_t stream);
// Deterministic mode, before the main kernel: the statistics of the call's
// inputs (q, kv, dO, Delta, topk_idxs over all of `s`) into stats / counts
// (zeroed beforehand), then the binary point stats[kDetShift].
cudaError_t launch_bwd_det_stats(const __nv_bfloat16* q, const __nv_bfloat16* kv,
                                 const __nv_bfloat16* dout, const float* delta,
                                 const int32_t* idx, const smqa_shape& s, uint32_t* stats,
                                 uint32_t* counts, cudaStream_t stream);
cudaError_t launch_bwd_det_scale(const smqa_shape& s, float scale, uint32_t* stats,
                                 const uint32_t* counts, cudaStream_t stream);
cudaError_t launch_bwd_postprocess(const float* acc, __nv_bfloat16* out, int64_t elems,
                                   cudaStream_t stream);

// The backward's main kernel over the tokens of `s` (a whole call or a chunk
// of one): writes dq and adds every slot's dKV contribution into `acc`
// (fp32), or into `acc_fixed` (fixed point with the binary point *fix_shift)
// when that is non-null.
// `exch` is the exchange pool of smqa_bwd_exchange_bytes(s) bytes (D = 512).
// The caller has checked shapes and pointers.
smqa_status bwd_main_launch(const void* q, const void* kv, const void* dout, const int32_t* idx,
                            const float* lse, const float* delta, const smqa_shape& s,
                            float scale, void* dq, float* acc, unsigned long long* acc_fixed,
                            const int* fix_shift, void* exch, cudaStream_t stream);
// The entry points' shape check (records the reason on failure).
smqa_status validate_shape(const smqa_shape& s);
// sm_scale as the entry points interpret it (<= 0 or NaN selects D^-1/2).
float effective_scale(float sm_scale, int D);

}  // namespace smqa
