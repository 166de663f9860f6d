// smqa_bwd.cu -- backward of top-k sparse MQA with an attention sink on sm_103a.
//
// What it computes (DeepSeek-V4 kernel pages of NeMo AutoModel,
// tilelang_sparse_mla_bwd: `sparse_mqa_bwd_interface` and its `preprocess`,
// `bwd` and `postprocess` kernels).  With c = sm_scale, for token t, head h
// and valid slot j (row r = idx[t,j]):
//   P_j   = 2^(c log2(e) q.k_j - lse2[t,h])        (recomputed from the LSE)
//   dP_j  = dO[t,h] . kv[r]
//   dS_j  = P_j (dP_j - Delta[t,h]),   Delta = rowsum(O * dO)
//   dQ[t,h]  = c sum_j dS_j kv[r]
//   dKV[r]  += c dS_j q[t,h] + P_j dO[t,h]
//
// Three kernels, as on the page:
//   preprocess   Delta[t,h] in fp32 (one warp per row) and zeroing of the
//                fp32 dKV accumulator, fused into one launch;
//   main         persistent CTAs (a CTA pair for D = 512, each CTA owning
//                half of D) that take tokens one after another: per token,
//                S = Q.K^T and dP = dO.V^T on the tensor core over 64-slot
//                blocks, the pair's half-D partial sums traded in block
//                floating point through an L2-resident exchange slot (two
//                buffers per receiver, freed by a consumed-signal), P and dS
//                on CUDA cores, then dQ += dS.K accumulated in TMEM over all
//                blocks and dKV^T = Q^T.dS + dO^T.P per block, which a drain
//                warpgroup reads from TMEM and scatters with fp32
//                red.global.add into the accumulator; the next token's
//                gathers, scores and exchange start while the current one
//                finishes;
//   postprocess  fp32 accumulator -> bf16 (round to nearest even).
// dKV^T (lanes = head-dim rows, columns = slots) keeps M = 128 for the
// 64-slot blocks and lets each warp's 32 lanes add to 32 consecutive floats
// of a kv row.  A deterministic mode replaces the fp32 reductions by 64-bit
// fixed-point integer ones with a per-call binary point (below).
#include <cuda_runtime.h>

#include "smqa_internal.h"
#include "smqa_ptx.cuh"

namespace smqa {

// --------------------------------------------------------------------------
// preprocess: Delta = rowsum(O * dO) and dKV accumulator = 0
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    smqa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                        float* __restrict__ delta, float* __restrict__ acc, int64_t rows, int D,
                        int64_t acc_vec4) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = warp_id; r < rows; r += nwarps) {
    const uint4* po = reinterpret_cast<const uint4*>(o + r * D);
    const uint4* pd = reinterpret_cast<const uint4*>(dout + r * D);
    float s = 0.f;
    for (int v = lane; v < D / 8; v += 32) {
      const uint4 a = __ldg(po + v);
      const uint4 g = __ldg(pd + v);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 fa = __bfloat1622float2(a2[k]);
        const float2 fg = __bfloat1622float2(g2[k]);
        s = fmaf(fa.x, fg.x, s);
        s = fmaf(fa.y, fg.y, s);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) delta[r] = s;
  }
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  float4* a4 = reinterpret_cast<float4*>(acc);
  for (int64_t i = tid; i < acc_vec4; i += nthr) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// --------------------------------------------------------------------------
// postprocess: fp32 -> bf16
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    smqa_bwd_post_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ out,
                         int64_t vec8) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const float4* a4 = reinterpret_cast<const float4*>(acc);
  uint4* o4 = reinterpret_cast<uint4*>(out);
  for (int64_t i = tid; i < vec8; i += nthr) {
    const float4 x = __ldg(a4 + 2 * i);
    const float4 y = __ldg(a4 + 2 * i + 1);
    o4[i] = make_uint4(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w), pack_bf16x2(y.x, y.y),
                       pack_bf16x2(y.z, y.w));
  }
}

// --------------------------------------------------------------------------
// deterministic mode: statistics, binary point, postprocess
// --------------------------------------------------------------------------
// Every dKV contribution is added as a signed 64-bit fixed-point integer
// (value * 2^k rounded to nearest), and integer addition is associative, so
// the sum does not depend on the order of the atomics.  The binary point k
// is chosen per call from a bound on the contributions: one slot's
// contribution to dKV[r, d] (the sum over the H heads of the MMA) is
//   sum_h dS'_h q_h[d] + P_h dO_h[d],   dS'_h = P_h c (dP_h - Delta_h),
// with P_h <= 1, |dP_h| <= |dO_h| |kv_r| (Cauchy-Schwarz), so its magnitude
// is at most X = H (max|dO| + c (max|dO_h| max|kv_r| + max|Delta|) max|q|),
// and an element's sum is at most n X, n the most slots naming one kv row.
// k = 61 - ceil(log2(n X)) keeps every contribution and every sum below
// 2^61 (room for the fp32 roundings of the MMA and of the statistics); the
// resolution 2^-k is then at most n X 2^-60, relative to the bound, at any
// input scale.  All statistics are maxima or integer counts, so k itself is
// the same from run to run.
__device__ __forceinline__ void atomic_max_nonneg(uint32_t* w, float v) {
  // Non-negative floats order as their bit patterns.
  atomicMax(w, __float_as_uint(v));
}

__global__ void __launch_bounds__(256)
    smqa_bwd_det_stats_kernel(const __nv_bfloat16* __restrict__ q,
                              const __nv_bfloat16* __restrict__ kv,
                              const __nv_bfloat16* __restrict__ dout,
                              const float* __restrict__ delta, const int32_t* __restrict__ idx,
                              int64_t rows, int64_t kv_rows, int D, int S, int S_kv, int topk,
                              uint32_t* __restrict__ stats, uint32_t* __restrict__ counts) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  float m_do = 0.f, m_dosq = 0.f, m_kvsq = 0.f, m_q = 0.f, m_dl = 0.f;
  // Squared norm (warp-wide, in a fixed order) and largest magnitude of row r.
  auto row_stats = [&](const __nv_bfloat16* base, int64_t r, float& sq, float& mx) {
    const uint4* pr = reinterpret_cast<const uint4*>(base + r * D);
    float s = 0.f, m = 0.f;
    for (int v = lane; v < D / 8; v += 32) {
      const uint4 a = __ldg(pr + v);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(a2[k]);
        s = fmaf(f.x, f.x, s);
        s = fmaf(f.y, f.y, s);
        m = fmax3f(m, fabsf(f.x), fabsf(f.y));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    sq = s;
    mx = m;
  };
  for (int64_t r = warp_id; r < rows; r += nwarps) {
    float sq, mx;
    row_stats(dout, r, sq, mx);
    m_dosq = fmaxf(m_dosq, sq);
    m_do = fmaxf(m_do, mx);
    row_stats(q, r, sq, mx);
    m_q = fmaxf(m_q, mx);
  }
  for (int64_t r = warp_id; r < kv_rows; r += nwarps) {
    float sq, mx;
    row_stats(kv, r, sq, mx);
    m_kvsq = fmaxf(m_kvsq, sq);
  }
  for (int64_t i = tid; i < rows; i += nthr) m_dl = fmaxf(m_dl, fabsf(__ldg(delta + i)));
  // Reference counts: slot i of token t = i / topk names row idx[i] of batch
  // element t / S.
  const int64_t per_b = static_cast<int64_t>(S) * topk;
  const int64_t total = kv_rows / S_kv * per_b;
  for (int64_t i = tid; i < total; i += nthr) {
    const int r = __ldg(idx + i);
    if (static_cast<unsigned>(r) < static_cast<unsigned>(S_kv))
      atomicAdd(counts + (i / per_b) * S_kv + r, 1u);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    m_do = fmaxf(m_do, __shfl_xor_sync(0xffffffffu, m_do, off));
    m_dosq = fmaxf(m_dosq, __shfl_xor_sync(0xffffffffu, m_dosq, off));
    m_kvsq = fmaxf(m_kvsq, __shfl_xor_sync(0xffffffffu, m_kvsq, off));
    m_q = fmaxf(m_q, __shfl_xor_sync(0xffffffffu, m_q, off));
    m_dl = fmaxf(m_dl, __shfl_xor_sync(0xffffffffu, m_dl, off));
  }
  if (lane == 0) {
    atomic_max_nonneg(stats + kDetMaxAbsDout, m_do);
    atomic_max_nonneg(stats + kDetMaxDoutSq, m_dosq);
    atomic_max_nonneg(stats + kDetMaxKvSq, m_kvsq);
    atomic_max_nonneg(stats + kDetMaxAbsQ, m_q);
    atomic_max_nonneg(stats + kDetMaxAbsDelta, m_dl);
  }
}

// The most slots naming one kv row (block maxima, then atomicMax), and in
// the last block to finish the binary point k from the statistics.
__global__ void __launch_bounds__(256)
    smqa_bwd_det_scale_kernel(uint32_t* __restrict__ stats, const uint32_t* __restrict__ counts,
                              int64_t n, int H, float scale) {
  __shared__ uint32_t part[8];
  __shared__ bool last;
  uint32_t m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    m = max(m, __ldg(counts + i));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t bm = 0;
    for (int w = 0; w < 8; ++w) bm = max(bm, part[w]);
    atomicMax(stats + kDetMaxCount, bm);
    __threadfence();
    last = atomicAdd(stats + kDetTicket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  volatile uint32_t* vs = stats;
  const double a_do = __uint_as_float(vs[kDetMaxAbsDout]);
  const double n_do = sqrt(static_cast<double>(__uint_as_float(vs[kDetMaxDoutSq])));
  const double n_kv = sqrt(static_cast<double>(__uint_as_float(vs[kDetMaxKvSq])));
  const double a_q = __uint_as_float(vs[kDetMaxAbsQ]);
  const double a_dl = __uint_as_float(vs[kDetMaxAbsDelta]);
  const double cnt = static_cast<double>(vs[kDetMaxCount]);
  // X with a margin of 1 + 2^-8 for the fp32 roundings of the statistics.
  const double x = static_cast<double>(H) * (a_do + scale * (n_do * n_kv + a_dl) * a_q) *
                   (1.0 + 1.0 / 256.0);
  const double bound = cnt * x;
  int k;
  if (!(bound > 0.0)) {
    k = 100;  // every contribution is zero
  } else if (!(bound < 1e300)) {
    k = -100;  // non-finite inputs: the result is undefined
  } else {
    int e;
    frexp(bound, &e);  // bound <= 2^e
    k = min(max(61 - e, -100), 100);
  }
  vs[kDetShift] = static_cast<uint32_t>(k);
}

// Fixed point -> bf16 or fp32: value = integer * 2^-k.
__global__ void __launch_bounds__(256)
    smqa_bwd_post_fixed_kernel(const unsigned long long* __restrict__ acc, void* __restrict__ out,
                               int fp32_out, int64_t vec4, const int* __restrict__ shift) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const ulonglong2* a2 = reinterpret_cast<const ulonglong2*>(acc);
  const float inv = pow2f(-__ldg(shift));
  for (int64_t i = tid; i < vec4; i += nthr) {
    const ulonglong2 x = a2[2 * i], y = a2[2 * i + 1];
    const float v0 = __ll2float_rn(static_cast<long long>(x.x)) * inv;
    const float v1 = __ll2float_rn(static_cast<long long>(x.y)) * inv;
    const float v2 = __ll2float_rn(static_cast<long long>(y.x)) * inv;
    const float v3 = __ll2float_rn(static_cast<long long>(y.y)) * inv;
    if (fp32_out)
      reinterpret_cast<float4*>(out)[i] = make_float4(v0, v1, v2, v3);
    else
      reinterpret_cast<uint2*>(out)[i] = make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
  }
}

// --------------------------------------------------------------------------
// sink gradient: dsink[h] = -sum_t 2^(sink_h log2 e - lse2[t,h]) Delta[t,h]
// --------------------------------------------------------------------------
// The sink adds exp(sink_h) to row (t,h)'s denominator but no value, so
// dO[t,h]/dsink_h = -p_sink O[t,h] with p_sink = exp(sink_h)/Z, and the loss
// gradient is -p_sink (dO . O) = -p_sink Delta summed over tokens.  One CTA
// per head; thread i sums tokens i, i + 256, ... and the partial sums meet
// in a fixed order, so the result does not vary from run to run.
__global__ void __launch_bounds__(256)
    smqa_bwd_sink_kernel(const float* __restrict__ sink, const float* __restrict__ lse,
                         const float* __restrict__ delta, float* __restrict__ dsink, int64_t tokens,
                         int H) {
  __shared__ float part[8];
  const int h = blockIdx.x;
  const float s2 = __ldg(sink + h) * 1.4426950408889634f;
  float acc = 0.f;
  for (int64_t t = threadIdx.x; t < tokens; t += 256) {
    const int64_t r = t * H + h;
    acc = fmaf(exp2f(s2 - __ldg(lse + r)), __ldg(delta + r), acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += part[w];
    dsink[h] = -tot;
  }
}

// --------------------------------------------------------------------------
// main backward kernel
// --------------------------------------------------------------------------
template <int DC, int NC>
struct BwdLayout {
  static constexpr int kHPad = 128;
  static constexpr int kBI = 64;                 // slots per block (MMA N of S, dP, dKV^T)
  static constexpr int kChunks = DC / 64;
  static constexpr int kNE = DC >= 128 ? DC / 128 : 1;  // 128-row halves of dKV^T
  static constexpr int kStages = NC == 2 ? 2 : 4;
  static constexpr int kTokRing = 4;             // live-block counts published ahead
  static constexpr uint32_t kQChunkBytes = kHPad * 128;          // 16 KB
  static constexpr uint32_t kQBytes = kChunks * kQChunkBytes;
  static constexpr uint32_t kKvChunkBytes = kBI * 128;           // 8 KB
  static constexpr uint32_t kKvStageBytes = kChunks * kKvChunkBytes;
  static constexpr uint32_t kPBytes = kHPad * kBI * 2;           // 16 KB (128-byte rows)
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffDo = kOffQ + kQBytes;
  // For DC = 64 the 128-row M-major views of Q^T / dO^T read one chunk past
  // each tile (those rows are discarded); keep a full chunk mapped after dO.
  static constexpr uint32_t kOffKv = kOffDo + (kChunks >= 2 ? kQBytes : 2 * kQChunkBytes);
  static constexpr uint32_t kOffP = kOffKv + kStages * kKvStageBytes;
  static constexpr uint32_t kOffDs = kOffP + kPBytes;
  static constexpr uint32_t kOffCtrl = kOffDs + kPBytes;
  static constexpr int kBarKvFull = 0;
  static constexpr int kBarKvEmpty = kBarKvFull + kStages;
  // The P / dS groups alternate blocks (group = parity of the block's index
  // in the CTA's whole sequence), so the barriers between them and the MMA
  // issuer come one per parity: a group only ever waits on phases of its own
  // blocks.
  static constexpr int kBarSdpFull = kBarKvEmpty + kStages;  // [2]
  static constexpr int kBarSdpFree = kBarSdpFull + 2;        // [2]
  static constexpr int kBarPdsFull = kBarSdpFree + 2;        // [2]
  static constexpr int kBarPdsFree = kBarPdsFull + 2;        // [2]
  static constexpr int kBarDkvFull = kBarPdsFree + 2;
  static constexpr int kBarDkvFree = kBarDkvFull + 1;
  static constexpr int kBarRecvFull = kBarDkvFree + 1;  // [2], by block parity
  static constexpr int kBarSendOk = kBarRecvFull + 2;    // [2]
  static constexpr int kBarQdoFull = kBarSendOk + 2;     // one phase per token with blocks
  static constexpr int kBarQdoFree = kBarQdoFull + 1;    // its MMAs are done with Q and dO
  static constexpr int kBarDqDone = kBarQdoFree + 1;     // its dQ is complete in TMEM
  static constexpr int kBarDqFree = kBarDqDone + 1;      // ... and has been read out
  static constexpr int kBarTokFull = kBarDqFree + 1;     // [kTokRing]
  static constexpr int kBarTokEmpty = kBarTokFull + kTokRing;  // [kTokRing]
  // The pair's token sequence: rank 0 takes each token from the counter and
  // hands it to both CTAs (IdFull), rank 1 frees an entry again (IdEmpty,
  // on rank 0) once its readers are done with it.
  static constexpr int kBarIdFull = kBarTokEmpty + kTokRing;   // [kTokRing]
  static constexpr int kBarIdEmpty = kBarIdFull + kTokRing;    // [kTokRing]
  static constexpr int kBarDrain = kBarIdEmpty + kTokRing;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kOffTmemHolder = kOffCtrl + 8 * kNumBars;
  static constexpr uint32_t kOffAbort = kOffTmemHolder + 4;
  static constexpr uint32_t kOffSlot = kOffAbort + 4;
  static constexpr uint32_t kOffTokLast = kOffSlot + 4;           // int [kTokRing][2]
  static constexpr uint32_t kOffTokId = kOffTokLast + 8 * kTokRing;  // int [kTokRing], handed over
  static constexpr uint32_t kOffTokT = kOffTokId + 4 * kTokRing;     // int [kTokRing], published
  static constexpr uint32_t kCtrlBytes = 512;
  static_assert(kOffTokT + 4 * kTokRing - kOffCtrl <= kCtrlBytes, "control block overflow");
  static constexpr uint32_t kSmemBytes = kOffCtrl + kCtrlBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM: dQ, S, dP, dKV^T (one tile each).
  static constexpr uint32_t kTmemDq = 0;
  static constexpr uint32_t kTmemS = DC;
  static constexpr uint32_t kTmemDp = DC + kBI;
  static constexpr uint32_t kTmemDkv = DC + 2 * kBI;  // + e * kBI
  static constexpr uint32_t kTmemUsed = kTmemDkv + kNE * kBI;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  // warps 0-7: P / dS in two groups of four (group g = warp / 4 handles the
  // blocks of parity g; thread = head row 32 (warp % 4) + lane, all 64 slots
  // of a block; for D split across the pair they also send this CTA's
  // partial S / dP to the peer); 8-11: dKV drain (thread = head-dim row) and
  // each token's dQ read-out (thread = head row); 12-13: gather and each
  // token's live-block count; 14: TMEM owner + MMA issuer + Q / dO loads.
  static constexpr int kPdsThreads = 256;
  static constexpr int kGroupThreads = 128;
  static constexpr int kDrainWarp0 = 8;
  static constexpr int kProducerWarp0 = 12;
  static constexpr int kMmaWarp = 14;
  static constexpr int kThreads = 480;
  // Readers of a published live-block count: the MMA thread, the eight
  // P / dS warps and the four drain warps (one arrival each).
  static constexpr int kTokReaders = 1 + 8 + 4;
  // Exchange buffer of one receiver and block parity: 16 pieces of 16 bytes
  // per head (8 of S, 8 of dP, each the 16-bit block-floating-point fields
  // of 8 slots), piece-major, then per slot half and head one packed pair of
  // exponents.
  static constexpr uint32_t kXchgScaleOff = 16u * 16u * kHPad;
  static constexpr uint32_t kXchgBytes = kXchgScaleOff + 2u * 4u * kHPad;
  static_assert(2 * 2 * kXchgBytes == kBwdSlotBytes, "exchange slot size");
};

// This CTA's partial S (exp2 domain) and sm_scale dP of one head row over
// 32 slots of the block (one slot half), each in block floating point (one
// exponent per head, block and half, see bfp16_exponent): hs[w] / hp[w] hold
// the 16-bit fields of slots 2w, 2w+1; the returned word packs the two
// exponents (S in the low half, dP in the high half, each offset by 128).
// Both CTAs add the same two rounded values, so they agree bit for bit.
__device__ __forceinline__ uint32_t own_partials_bfp(uint32_t t_s, uint32_t t_dp,
                                                     float scale_log2, float scale,
                                                     uint32_t (&hs)[16], uint32_t (&hp)[16]) {
  float xs[32], xp[32];
  tmem_ld32x2(t_s, t_dp, xs, xp);
  const int es = bfp16_exponent(__fmul_rn(__fmul_rn(absmax_n<32>(xs), scale_log2), kExpMargin));
  const int ep = bfp16_exponent(__fmul_rn(__fmul_rn(absmax_n<32>(xp), scale), kExpMargin));
  const float fs = __fmul_rn(scale_log2, pow2f(14 - es));
  const float fp = __fmul_rn(scale, pow2f(14 - ep));
#pragma unroll
  for (int w = 0; w < 16; ++w) {
    const float2 rs = bfp16_round2(make_float2(xs[2 * w], xs[2 * w + 1]), fs);
    hs[w] = bfp16_pack(rs.x, rs.y);
    const float2 rp = bfp16_round2(make_float2(xp[2 * w], xp[2 * w + 1]), fp);
    hp[w] = bfp16_pack(rp.x, rp.y);
  }
  return static_cast<uint32_t>(es + 128) | (static_cast<uint32_t>(ep + 128) << 16);
}

// 2^(e - 14) for the exponent in the low (HI = false) or high half of a
// packed exponent word: the weight of one unit of that half's fields.
template <bool HI>
__device__ __forceinline__ float bfp16_unit(uint32_t exps) {
  const int e = static_cast<int>(HI ? (exps >> 16) : (exps & 0xffffu)) - 128;
  return pow2f(e - 14);
}

// Persistent: each CTA (pair) of the grid's p.clusters handles a sequence of
// tokens -- taken one at a time from p.tok_counter by the pair's rank 0 (so
// faster pairs take more), or c, c + p.clusters, ... without a counter -- as
// one sequence of 64-slot blocks (G counts them over the CTA's whole life),
// so that the next token's gathers, scores and exchange overlap the last
// blocks and the dQ read-out of the current one; only Q / dO (one buffer)
// wait for the previous token's gradient MMAs.  Every barrier phase follows
// G, or the token count k.  Ring entry k % kTokRing publishes token k's index
// (-1: no more tokens) and live-block count.
template <int DC, int NC, bool DET>
__global__ void __launch_bounds__(480, 1)
    smqa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using L = BwdLayout<DC, NC>;
  extern __shared__ uint8_t smem_raw[];
  uint32_t base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  base += pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cl = static_cast<int>(blockIdx.x) / NC;  // this CTA's (pair's) index
  const uint32_t rank = NC == 2 ? cluster_ctarank() : 0u;
  auto token_of = [&](int k) -> int { return cl + k * p.clusters; };  // k-th token of the CTA
  auto bar = [&](int i) -> uint32_t { return base + L::kOffCtrl + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + L::kOffTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  volatile int* slot_smem = reinterpret_cast<volatile int*>(smem + L::kOffSlot);
  volatile int* tok_last = reinterpret_cast<volatile int*>(smem + L::kOffTokLast);
  volatile int* tok_id = reinterpret_cast<volatile int*>(smem + L::kOffTokId);
  volatile int* tok_t = reinterpret_cast<volatile int*>(smem + L::kOffTokT);
  const WaitCtl ctl{abort_flag, p.status, p.limit_ns};
  // Live blocks of the token in ring entry e (after its full barrier).
  auto tok_blocks = [&](int e) -> int {
    const int last = max(tok_last[2 * e], tok_last[2 * e + 1]);
    return last < 0 ? 0 : last / L::kBI + 1;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarKvFull + s), 64);  // every gather thread arrives
      mbar_init(bar(L::kBarKvEmpty + s), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(bar(L::kBarSdpFull + g), 1);
      mbar_init(bar(L::kBarSdpFree + g), L::kGroupThreads);
      mbar_init(bar(L::kBarPdsFull + g), L::kGroupThreads);
      mbar_init(bar(L::kBarPdsFree + g), 1);
    }
    mbar_init(bar(L::kBarDkvFull), 1);
    mbar_init(bar(L::kBarDkvFree), 128);
    // Exchange buffer i serves the blocks of parity i: the four warps of the
    // peer's group i each signal it filled and, later, consumed.
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::kBarRecvFull + i), L::kGroupThreads / 32);
      mbar_init(bar(L::kBarSendOk + i), L::kGroupThreads / 32);
    }
    mbar_init(bar(L::kBarQdoFull), 1);
    mbar_init(bar(L::kBarQdoFree), 1);
    mbar_init(bar(L::kBarDqDone), 1);
    mbar_init(bar(L::kBarDqFree), 128);
    for (int e = 0; e < L::kTokRing; ++e) {
      mbar_init(bar(L::kBarTokFull + e), 2);  // one per gather warp
      mbar_init(bar(L::kBarTokEmpty + e), L::kTokReaders);
      mbar_init(bar(L::kBarIdFull + e), 1);
      mbar_init(bar(L::kBarIdEmpty + e), 1);
    }
    mbar_init(bar(L::kBarDrain), 1);
    *abort_flag = *reinterpret_cast<volatile int*>(p.status) != 0 ? 1 : 0;
    *slot_smem = -1;
    if (NC == 2 && rank == 0 && *abort_flag == 0) {
      // Claim an exchange slot for the pair (bounded; released at exit).
      const uint64_t t0 = globaltimer_ns();
      int got = -1;
      for (uint32_t it = 0; got < 0; ++it) {
        const int s = static_cast<int>((static_cast<uint32_t>(cl) + it) % static_cast<uint32_t>(p.nslots));
        if (atomicCAS(p.slot_flags + s, 0, 1) == 0) {
          got = s;
        } else if ((it % static_cast<uint32_t>(p.nslots)) == static_cast<uint32_t>(p.nslots) - 1u &&
                   globaltimer_ns() - t0 > p.limit_ns) {
          *abort_flag = 1;
          atomicOr(p.status, kStatusTimeout);
          break;
        }
      }
      *slot_smem = got;
    }
    fence_mbar_init();
  }
  if (warp == L::kMmaWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
    }
    tmem_alloc(base + L::kOffTmemHolder, L::kTmemCols);
  }
  // Heads beyond H are zero rows of the Q / dO operands (the TMA box covers
  // H rows, so later loads leave them zero).
  if (threadIdx.x < L::kHPad && static_cast<int>(threadIdx.x) >= p.H) {
    const uint32_t h = threadIdx.x;
#pragma unroll
    for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        st_shared_v4(base + L::kOffQ + c * L::kQChunkBytes + h * 128u + k * 16u, 0u, 0u, 0u, 0u);
        st_shared_v4(base + L::kOffDo + c * L::kQChunkBytes + h * 128u + k * 16u, 0u, 0u, 0u, 0u);
      }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if (NC == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // The pair's exchange slot (claimed by rank 0); without one, nothing runs.
  int slot = -1;
  if (NC == 2) {
    slot = rank == 0 ? *slot_smem : ld_shared_cluster_s32(mapa_shared(base + L::kOffSlot, 0u));
    if (slot < 0) *abort_flag = 1;
  }

  if (warp >= L::kProducerWarp0 && warp < L::kMmaWarp) {
    // ------------------------------------------------------------ gather
    // Per token: the index row's last valid slot (each warp scans half the
    // row) into ring entry k % kTokRing, then the token's live blocks.  Warp
    // pw copies slots [32 pw, 32 pw + 32) of each 64-slot block; one warp
    // instruction moves kRpi whole rows of this CTA's D slice (32 lanes x 16
    // bytes, coalesced) into the 128-byte-swizzled tile with cp.async.
    const int pw = warp - L::kProducerWarp0;
    constexpr int kCpr = DC / 8;
    constexpr int kRpi = 32 / kCpr;
    const int rsub = lane / kCpr;
    const int cc = lane % kCpr;
    const uint32_t lane_off = static_cast<uint32_t>(cc / 8) * L::kKvChunkBytes;
    const uint32_t c16 = static_cast<uint32_t>(cc % 8);
    bool ok = *abort_flag == 0;
    int G = 0;
    for (int k = 0; ok; ++k) {
      const int e = k % L::kTokRing;
      if (k >= L::kTokRing) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokEmpty + e),
                                               ((k / L::kTokRing) - 1) & 1, ctl));
        if (!ok) break;
      }
      int t;
      if (NC == 2 && p.tok_counter != nullptr) {
        // The pair's k-th token: rank 0 takes it from the counter and writes
        // it into both CTAs' entry e (the peer's only once the peer has
        // freed it); both read it after IdFull.
        if (pw == 0 && lane == 0) {
          if (rank == 1 && k >= L::kTokRing) {
            mbar_arrive_remote(mapa_shared(bar(L::kBarIdEmpty + e), 0u));
          } else if (rank == 0) {
            bool free_ok = true;
            if (k >= L::kTokRing)
              free_ok = mbar_wait<true>(bar(L::kBarIdEmpty + e), ((k / L::kTokRing) - 1) & 1, ctl);
            if (free_ok) {
              int nt = atomicAdd(p.tok_counter, 1);
              if (nt >= p.tokens) nt = -1;
              tok_id[e] = nt;
              st_shared_cluster_s32(mapa_shared(base + L::kOffTokId + 4u * e, 1u), nt);
              mbar_arrive_remote(mapa_shared(bar(L::kBarIdFull + e), 1u));
              mbar_arrive(bar(L::kBarIdFull + e));
            }
          }
        }
        // The whole warp again before anyone waits (lanes suspended in a wait
        // while lane 0 hands the token over slow the handover down).
        __syncwarp();
        ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarIdFull + e), (k / L::kTokRing) & 1, ctl));
        if (!ok) break;
        t = tok_id[e];
      } else {
        t = token_of(k) < p.tokens ? token_of(k) : -1;
      }
      if (t < 0) {
        // No more tokens: publish the end.
        if (lane == 0) {
          if (pw == 0) tok_t[e] = -1;
          tok_last[2 * e + pw] = -1;
          mbar_arrive(bar(L::kBarTokFull + e));
        }
        break;
      }
      const int32_t* idx_row = p.idx + static_cast<size_t>(t) * p.topk;
      // 16-byte loads issued eight at a time before any compare, so one
      // round of memory latency covers a 2048-slot row (the scalar scan it
      // replaces, eight dependent rounds, held up the token's first gathers
      // and cost 0.25 us per block).
      int last = -1;
      const int tid = 32 * pw + lane;
      if ((p.topk & 3) == 0 && (reinterpret_cast<uintptr_t>(idx_row) & 15u) == 0) {
        const int4* row4 = reinterpret_cast<const int4*>(idx_row);
        const unsigned skv = static_cast<unsigned>(p.S_kv);
#pragma unroll 8
        for (int q = tid; q < p.topk / 4; q += 64) {
          const int4 v = __ldg(row4 + q);
          if (static_cast<unsigned>(v.x) < skv) last = 4 * q;
          if (static_cast<unsigned>(v.y) < skv) last = 4 * q + 1;
          if (static_cast<unsigned>(v.z) < skv) last = 4 * q + 2;
          if (static_cast<unsigned>(v.w) < skv) last = 4 * q + 3;
        }
      } else {
#pragma unroll 8
        for (int j = tid; j < p.topk; j += 64)
          if (static_cast<unsigned>(__ldg(idx_row + j)) < static_cast<unsigned>(p.S_kv)) last = j;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
      if (lane == 0) {
        if (pw == 0) tok_t[e] = t;
        tok_last[2 * e + pw] = last;
        mbar_arrive(bar(L::kBarTokFull + e));
        // The token's Q / dO slices into L2: the MMA thread loads them once
        // the previous token's gradients are done, right at the token
        // boundary (12.54 -> 12.50 ms).
        if (k > 0) {
          for (int c = 2 * pw; c < 2 * pw + 2 && c < L::kChunks; ++c) {
            tma_prefetch_l2_2d(&tm_q, static_cast<int>(rank) * DC + c * 64, t * p.H);
            tma_prefetch_l2_2d(&tm_do, static_cast<int>(rank) * DC + c * 64, t * p.H);
          }
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokFull + e), (k / L::kTokRing) & 1, ctl));
      if (!ok) break;
      const int nblk = tok_blocks(e);
      const int b = t / p.S;
      const __nv_bfloat16* kv_col =
          p.kv + static_cast<size_t>(b) * p.S_kv * p.D + static_cast<size_t>(rank) * DC + cc * 8;
      auto load_idx = [&](int blk) -> int {
        const int j = blk * L::kBI + 32 * pw + lane;
        return j < p.topk ? __ldg(idx_row + j) : -1;
      };
      int r_next = nblk > 0 ? load_idx(0) : -1;
      for (int i = 0; i < nblk; ++i, ++G) {
        const int s = G % L::kStages;
        const int r = r_next;
        if (i + 1 < nblk) r_next = load_idx(i + 1);
        const int row = static_cast<unsigned>(r) < static_cast<unsigned>(p.S_kv) ? r : 0;
        if (G >= L::kStages) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarKvEmpty + s), ((G / L::kStages) - 1) & 1, ctl));
          if (!ok) break;
        } else if (*abort_flag) {
          ok = false;
          break;
        }
        const uint32_t stage = base + L::kOffKv + s * L::kKvStageBytes + lane_off;
#pragma unroll
        for (int kk = 0; kk < 32 / kRpi; ++kk) {
          const int rw = kk * kRpi + rsub;  // row within this warp's 32
          const int rr = __shfl_sync(0xffffffffu, row, rw);
          const uint32_t srow = static_cast<uint32_t>(32 * pw + rw);
          cp_async_16(stage + srow * 128u + ((c16 ^ (srow & 7u)) << 4),
                      kv_col + static_cast<size_t>(rr) * p.D);
        }
        // Arrives on the stage's full barrier once this thread's copies of
        // the block have landed; the MMA thread fences them into the async
        // proxy.
        cp_async_arrive_noinc(bar(L::kBarKvFull + s));
      }
    }
    // Let every copy this warp started land before the CTA can exit.
    cp_async_wait_all();
  } else if (warp == L::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_sdp = idesc_bf16_f32(128, L::kBI, false, false);
      constexpr uint32_t idesc_dq = idesc_bf16_f32(128, DC, false, true);
      constexpr uint32_t idesc_dkv = idesc_bf16_f32(128, L::kBI, true, true);
      // Descriptors are built once; per MMA only the start-address field
      // (bits 0-13, in 16-byte units) moves, by compile-time offsets.
      const uint64_t d_q = smem_desc(base + L::kOffQ, 16u, 1024u, kSwizzle128B);
      const uint64_t d_do = smem_desc(base + L::kOffDo, 16u, 1024u, kSwizzle128B);
      const uint64_t d_kv = smem_desc(base + L::kOffKv, 16u, 1024u, kSwizzle128B);
      const uint64_t d_kvmn = smem_desc(base + L::kOffKv, L::kKvChunkBytes, 1024u, kSwizzle128B);
      const uint64_t d_ds = smem_desc(base + L::kOffDs, 16u, 1024u, kSwizzle128B);
      const uint64_t d_qt = smem_desc(base + L::kOffQ, L::kQChunkBytes, 1024u, kSwizzle128B);
      const uint64_t d_dot = smem_desc(base + L::kOffDo, L::kQChunkBytes, 1024u, kSwizzle128B);
      const uint64_t d_dsmn = smem_desc(base + L::kOffDs, L::kPBytes, 1024u, kSwizzle128B);
      const uint64_t d_pmn = smem_desc(base + L::kOffP, L::kPBytes, 1024u, kSwizzle128B);
      // S and dP of block G (M = 128 heads, N = 64 slots, K = this CTA's D slice).
      auto issue_sdp = [&](int G) {
        const int s = G % L::kStages;
        const uint64_t dk = d_kv + ((static_cast<uint32_t>(s) * L::kKvStageBytes) >> 4);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t bd = dk + ((c * L::kKvChunkBytes + k * 32u) >> 4);
            const uint32_t acc = (c | k) != 0 ? 1u : 0u;
            mma_ss(tmem + L::kTmemS, d_q + ((c * L::kQChunkBytes + k * 32u) >> 4), bd,
                   idesc_sdp, acc);
            mma_ss(tmem + L::kTmemDp, d_do + ((c * L::kQChunkBytes + k * 32u) >> 4), bd,
                   idesc_sdp, acc);
          }
        }
        mma_commit(bar(L::kBarSdpFull + (G & 1)));
      };
      // Gradients of block G (block i of its token): dQ += dS'.K (M = 128
      // heads, N = DC, K = 64 slots; the token's first block overwrites);
      // dKV^T[e] = Q^T[e].dS' + dO^T[e].P (M = 128 dims, N = 64 slots, K =
      // 128 heads).
      auto issue_grad = [&](int G, int i) {
        const int sj = G % L::kStages;
        const uint64_t dkv = d_kvmn + ((static_cast<uint32_t>(sj) * L::kKvStageBytes) >> 4);
#pragma unroll
        for (int k = 0; k < L::kBI / 16; ++k)
          mma_ss(tmem + L::kTmemDq, d_ds + (k * 32u >> 4), dkv + (k * 2048u >> 4), idesc_dq,
                 (i > 0 || k > 0) ? 1u : 0u);
        // Only dQ reads the kv stage: the gather may refill it once these
        // MMAs are done, while the dKV^T MMAs still run.
        mma_commit(bar(L::kBarKvEmpty + sj));
#pragma unroll
        for (int e = 0; e < L::kNE; ++e) {
          const uint32_t d_tm = tmem + L::kTmemDkv + e * L::kBI;
#pragma unroll
          for (int k = 0; k < L::kHPad / 16; ++k)
            mma_ss(d_tm, d_qt + ((2 * e * L::kQChunkBytes + k * 2048u) >> 4),
                   d_dsmn + (k * 2048u >> 4), idesc_dkv, k > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < L::kHPad / 16; ++k)
            mma_ss(d_tm, d_dot + ((2 * e * L::kQChunkBytes + k * 2048u) >> 4),
                   d_pmn + (k * 2048u >> 4), idesc_dkv, 1u);
        }
        mma_commit(bar(L::kBarPdsFree + (G & 1)));
        mma_commit(bar(L::kBarDkvFull));
      };
      // Three cursors over the CTA's tokens: Q / dO loads (token lk; one per
      // token with blocks, into the single buffer once the previous such
      // token's MMAs have completed), S / dP (token sk, its block si,
      // sequence index sG) and gradients (gk, gi, gG).  Each caches its
      // token's live-block count (-1: not read yet) and touches the published
      // counts only at token boundaries, so an iteration stays short.  Event
      // loop (non-blocking tests): S / dP of the next block as soon as its kv
      // rows have landed, the previous S / dP tile has been read and its
      // token's Q / dO are in (first, so the other P / dS group gets its
      // tile early: 12.67 -> 12.55 ms); otherwise the gradients of the oldest
      // block once its P / dS are written and the drain has read the previous
      // dKV^T tile (and, for a token's first block, the previous token's dQ
      // has been read out); otherwise the next Q / dO load.
      auto tok_known = [&](int k) -> bool {
        return mbar_probe(bar(L::kBarTokFull + k % L::kTokRing), (k / L::kTokRing) & 1);
      };
      auto nblk_of = [&](int k) -> int { return tok_blocks(k % L::kTokRing); };
      int lk = 0, lnb = -1, la = 0, lt = -1;        // load cursor (token lt), loads issued
      bool l_end = false;                            // the load cursor met the end
      int sk = 0, si = 0, snb = -1, sG = 0, sa = 0;  // sa: load index of token sk
      int gk = 0, gi = 0, gnb = -1, gG = 0, ga = 0;  // ga: load index of token gk
      int qfree = 0;                                 // Q / dO releases committed
      bool ok = *abort_flag == 0;
      PollState ps = poll_start();
      uint32_t spins = 0;
      while (ok) {
        // ---- cursor bookkeeping (does work only at token boundaries).  The
        // next load's count is read only once the buffer is about to be free
        // (its previous token's last gradients issued), so that an iteration
        // in mid-token probes nothing but the events.
        if (lnb < 0 && !l_end && qfree >= la && tok_known(lk)) {
          lt = tok_t[lk % L::kTokRing];
          if (lt < 0) {
            l_end = true;
          } else {
            lnb = nblk_of(lk);
            if (lnb == 0) {  // nothing to load: on to the next token
              ++lk;
              lnb = -1;
              continue;
            }
          }
        }
        if (snb < 0 && sk < lk) snb = nblk_of(sk);  // published: the load cursor passed it
        if (snb >= 0 && si == snb) {                  // token sk done (or without blocks)
          if (snb > 0) ++sa;
          ++sk;
          si = 0;
          snb = -1;
          continue;
        }
        if (gnb < 0 && gk < lk) gnb = nblk_of(gk);
        if (gnb >= 0 && gi == gnb && gk < sk) {       // token gk done: release its count
          mbar_arrive(bar(L::kBarTokEmpty + gk % L::kTokRing));
          if (gnb > 0) ++ga;
          ++gk;
          gi = 0;
          gnb = -1;
          continue;
        }
        if (l_end && gk == lk) break;  // every token done
        // ---- events, within the current tokens: back to the bookkeeping
        // only at a token boundary or after a Q / dO load, so that a
        // mid-token iteration tests nothing but the events.
        const bool want_load = lnb > 0;
        const bool need_book = !want_load && lnb < 0 && !l_end && qfree >= la;
        for (;;) {
          if (si < snb &&
              mbar_probe(bar(L::kBarKvFull + sG % L::kStages), (sG / L::kStages) & 1) &&
              (sG == 0 || mbar_probe(bar(L::kBarSdpFree + ((sG - 1) & 1)), ((sG - 1) >> 1) & 1)) &&
              (si > 0 || mbar_probe(bar(L::kBarQdoFull), sa & 1))) {
            // The kv tile was written by cp.async (generic proxy): order it
            // before the tensor core's (async proxy) reads.
            fence_proxy_async_smem();
            tc_fence_after();
            issue_sdp(sG);
            ++si;
            ++sG;
            ps.t0 = globaltimer_ns();  // progress: the limit counts from the last issue
            if (static_cast<int>(blockIdx.x) == p.stall_cta && sG == 1) {  // test hook only
              ok = stall_until_limit(ctl);
              break;
            }
            if (si == snb) break;
          } else if (gG < sG && gi < gnb && mbar_probe(bar(L::kBarPdsFull + (gG & 1)), (gG >> 1) & 1) &&
                     (gG == 0 || mbar_probe(bar(L::kBarDkvFree), (gG - 1) & 1)) &&
                     (gi > 0 || ga == 0 || mbar_probe(bar(L::kBarDqFree), (ga - 1) & 1))) {
            tc_fence_after();
            issue_grad(gG, gi);
            ++gi;
            ++gG;
            ps.t0 = globaltimer_ns();
            if (gi == gnb) {
              // The token's last gradients: its dQ is complete once they
              // are, and Q / dO may take the next token.
              mma_commit(bar(L::kBarDqDone));
              mma_commit(bar(L::kBarQdoFree));
              ++qfree;
              break;
            }
          } else if (want_load && (la == 0 || mbar_probe(bar(L::kBarQdoFree), (la - 1) & 1))) {
            // Q and dO slices of token lt into the (free) buffer.
            const int t = lt;
            mbar_arrive_expect_tx(bar(L::kBarQdoFull),
                                  2u * static_cast<uint32_t>(p.H) * 128u * L::kChunks);
            for (int c = 0; c < L::kChunks; ++c) {
              const int x = static_cast<int>(rank) * DC + c * 64;
              tma_load_2d(base + L::kOffQ + c * L::kQChunkBytes, &tm_q, x, t * p.H, bar(L::kBarQdoFull));
              tma_load_2d(base + L::kOffDo + c * L::kQChunkBytes, &tm_do, x, t * p.H, bar(L::kBarQdoFull));
            }
            ++la;
            ++lk;
            lnb = -1;
            ps.t0 = globaltimer_ns();
            break;
          } else if (need_book && tok_known(lk)) {  // the next token is published
            break;
          } else if ((++spins & 63u) == 0u && !poll_check(ctl, ps)) {
            ok = false;
            break;
          }
        }
      }
      // No MMA may still be running when TMEM is released, and no Q / dO
      // load still landing when the CTA exits.
      mma_commit(bar(L::kBarDrain));
      mbar_wait_drain(bar(L::kBarDrain), 0);
      if (la > 0) mbar_wait_drain(bar(L::kBarQdoFull), (la - 1) & 1);
    }
    __syncwarp();
  } else if (warp >= L::kDrainWarp0) {
    // ------------------------------------------------------------ dKV drain
    // Thread = head-dim row of one lane quarter; per block 64 slots, read as
    // two 32-slot halves (both 128-row halves of the tile per TMEM trip).
    // After each token's blocks the same warps read its dQ out of TMEM
    // (thread = head row of the lane quarter) and store it, bf16.
    const int wq = warp - L::kDrainWarp0;  // TMEM lane quarter
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const bool active = (wq * 32) < DC;  // DC = 64: rows 64..127 are padding
    const size_t col0 = static_cast<size_t>(rank) * DC + wq * 32 + lane;
    // One contribution to element off of this lane's column: an fp32
    // reduction, or in the deterministic mode the value times 2^k (the
    // call's binary point) rounded to a 64-bit integer and added as an
    // integer, so the sum does not depend on the order of the additions.
    const float fix_scale = DET ? pow2f(__ldg(p.fix_shift)) : 0.f;
    auto add = [&](float* col, unsigned long long* colx, size_t off, float v) {
      if constexpr (DET) {
        const long long n = __float2ll_rn(v * fix_scale);
        asm volatile("red.global.add.u64 [%0], %1;" ::"l"(colx + off),
                     "l"(static_cast<unsigned long long>(n))
                     : "memory");
      } else {
        red_add_f32(col + off, v);
      }
    };
    const int h = wq * 32 + lane;  // head row of the dQ read-out
    // dQ rows start 32-byte aligned when the tensor does.
    const bool dq32 = (reinterpret_cast<uintptr_t>(p.dq) & 31u) == 0;
    bool ok = *abort_flag == 0;
    int G = 0, a = 0;
    for (int k = 0; ok; ++k) {
      const int e = k % L::kTokRing;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokFull + e), (k / L::kTokRing) & 1, ctl));
      if (!ok) break;
      const int t = tok_t[e];
      if (t < 0) break;
      const int nblk = tok_blocks(e);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kBarTokEmpty + e));
      const int b = t / p.S;
      const int32_t* idx_row = p.idx + static_cast<size_t>(t) * p.topk;
      float* col = p.dkv_acc + static_cast<size_t>(b) * p.S_kv * p.D + col0;
      unsigned long long* colx =
          DET ? p.dkv_fix + static_cast<size_t>(b) * p.S_kv * p.D + col0 : nullptr;
      // The index rows of the next block are loaded while this one is
      // drained, so their L2 latency stays off the way to DkvFree (12.66 ->
      // 12.36 ms).
      auto load_r = [&](int blk, int half) -> int {
        const int slot_j = blk * L::kBI + 32 * half + lane;
        return (blk < nblk && slot_j < p.topk) ? __ldg(idx_row + slot_j) : -1;
      };
      int rn0 = load_r(0, 0), rn1 = load_r(0, 1);
      for (int j = 0; j < nblk; ++j, ++G) {
        const int rc[2] = {rn0, rn1};
        rn0 = load_r(j + 1, 0);
        rn1 = load_r(j + 1, 1);
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDkvFull), G & 1, ctl));
        if (!ok) break;
        tc_fence_after();
        int row[2];
        uint32_t vm[2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int r = rc[half];
          const bool v = static_cast<unsigned>(r) < static_cast<unsigned>(p.S_kv);
          vm[half] = __ballot_sync(0xffffffffu, v);
          row[half] = v ? r : 0;
        }
        const uint32_t t0 = tmem + lane_base + L::kTmemDkv;
        if constexpr (L::kNE == 2) {
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float x[2][32];
            tmem_ld32x2(t0 + 32 * half, t0 + L::kBI + 32 * half, x[0], x[1]);
            if (half == 1) {  // the whole tile is in registers: let the MMAs reuse it
              tc_fence_before();
              mbar_arrive(bar(L::kBarDkvFree));
            }
            if (active) {
#pragma unroll
              for (int kk = 0; kk < 32; ++kk) {
                const int rk = __shfl_sync(0xffffffffu, row[half], kk);
                if ((vm[half] >> kk) & 1u) {
                  add(col, colx, static_cast<size_t>(rk) * p.D, x[0][kk]);
                  add(col, colx, static_cast<size_t>(rk) * p.D + 128, x[1][kk]);
                }
              }
            }
          }
        } else {
          float x[2][32];
          tmem_ld32x2(t0, t0 + 32, x[0], x[1]);
          tc_fence_before();
          mbar_arrive(bar(L::kBarDkvFree));
          if (active) {
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
              for (int kk = 0; kk < 32; ++kk) {
                const int rk = __shfl_sync(0xffffffffu, row[half], kk);
                if ((vm[half] >> kk) & 1u) add(col, colx, static_cast<size_t>(rk) * p.D, x[half][kk]);
              }
          }
        }
      }
      if (!ok) break;
      // dQ of the token, bf16, straight from TMEM to its rows (32-byte
      // stores, 16-byte ones when dq is not 32-byte aligned; 32 columns per
      // TMEM load -- 64 at a time cost 0.8 %, through the drain loop's
      // registers); a token without a valid slot gets zeros.
      if (nblk > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDqDone), a & 1, ctl));
        if (!ok) break;
        tc_fence_after();
      }
      __nv_bfloat16* qrow = p.dq + (static_cast<size_t>(t) * p.H + h) * p.D + static_cast<size_t>(rank) * DC;
#pragma unroll 1
      for (int c = 0; c < DC / 32; ++c) {
        float v[32];
        if (nblk > 0) {
          tmem_ld32(tmem + lane_base + L::kTmemDq + c * 32, v);
        } else {
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) v[kk] = 0.f;
        }
        if (h < p.H) {
          uint32_t w[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) w[u] = pack_bf16x2(v[2 * u], v[2 * u + 1]);
          if (dq32) {  // 32-byte stores: half the transactions of 16-byte ones
            st_global_v8(qrow + 32 * c, *reinterpret_cast<const uint32_t(*)[8]>(w));
            st_global_v8(qrow + 32 * c + 16, *reinterpret_cast<const uint32_t(*)[8]>(w + 8));
          } else {
            uint4* dst = reinterpret_cast<uint4*>(qrow + 32 * c);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              dst[kk] = make_uint4(w[4 * kk], w[4 * kk + 1], w[4 * kk + 2], w[4 * kk + 3]);
          }
        }
      }
      if (nblk > 0) {
        // dQ is in registers: the next token's first dQ MMA may overwrite it.
        tc_fence_before();
        mbar_arrive(bar(L::kBarDqFree));
        ++a;
      }
    }
  } else {
    // ------------------------------------------------------------ P / dS
    // Two groups of four warps alternate blocks (group g takes the blocks of
    // parity g in the CTA's sequence), so one block's latency chain -- read
    // the S / dP tile, round and send this CTA's partials, wait for the
    // peer's, decode, write P and dS' -- overlaps the next block's.  Thread
    // = head row h, all 64 slots of the block: the full S and dP of the row
    // (for D = 512 this CTA's partial plus the peer's, both in block
    // floating point), then
    //   P = 2^(S - lse2),  dS' = P (sm_scale dP - sm_scale Delta),
    // written bf16 for the gradient MMAs, 8 slots at a time.  The single
    // P / dS buffer is written only once the gradients of the previous block
    // (the other group's) have read it.
    const int h = (warp & 3) * 32 + lane;
    const int grp = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + L::kTmemS;
    const uint32_t t_dp = tmem + lane_base + L::kTmemDp;
    const uint32_t peer_full = NC == 2 ? mapa_shared(bar(L::kBarRecvFull + grp), rank ^ 1u) : 0u;
    const uint32_t peer_sendok = NC == 2 ? mapa_shared(bar(L::kBarSendOk + grp), rank ^ 1u) : 0u;
    // This group's receive buffer, and the peer's (which this group fills).
    const uint8_t* recv = NC == 2 ? p.exch + (static_cast<size_t>(slot) * 2 + rank) *
                                                 (2 * L::kXchgBytes) +
                                        grp * L::kXchgBytes
                                  : nullptr;
    uint8_t* send = NC == 2 ? p.exch + (static_cast<size_t>(slot) * 2 + (rank ^ 1u)) *
                                           (2 * L::kXchgBytes) +
                                  grp * L::kXchgBytes
                            : nullptr;
    const uint32_t row128 = static_cast<uint32_t>(h) * 128u;
    float lse2 = INFINITY, dlt_s = 0.f;
    // P and dS' of slots 8 ch .. 8 ch + 7 (ch = 0..7) from their scores zs
    // and scaled dP zp (slot validity: bit (8 ch + k) % 32 of msk).
    auto emit = [&](int ch, uint32_t msk, const float* zs, const float* zp) {
      uint32_t pp[4], pd[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 e = add2(make_float2(zs[2 * k], zs[2 * k + 1]), make_float2(-lse2, -lse2));
        const float2 g = add2(make_float2(zp[2 * k], zp[2 * k + 1]), make_float2(-dlt_s, -dlt_s));
        const int jj = (8 * ch + 2 * k) & 31;
        const float2 pv = make_float2(((msk >> jj) & 1u) ? fast_exp2(e.x) : 0.f,
                                      ((msk >> (jj + 1)) & 1u) ? fast_exp2(e.y) : 0.f);
        const float2 dv = mul2(pv, g);
        pp[k] = pack_bf16x2(pv.x, pv.y);
        pd[k] = pack_bf16x2(dv.x, dv.y);
      }
      const uint32_t off = row128 + ((static_cast<uint32_t>(ch) ^ static_cast<uint32_t>(h & 7)) << 4);
      st_shared_v4(base + L::kOffP + off, pp[0], pp[1], pp[2], pp[3]);
      st_shared_v4(base + L::kOffDs + off, pd[0], pd[1], pd[2], pd[3]);
    };
    bool ok = *abort_flag == 0;
    int G0 = 0;  // sequence index of the token's first block
    for (int k = 0; ok; ++k) {
      const int te = k % L::kTokRing;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokFull + te), (k / L::kTokRing) & 1, ctl));
      if (!ok) break;
      const int t = tok_t[te];
      if (t < 0) break;
      const int nblk = tok_blocks(te);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kBarTokEmpty + te));
      int i = ((G0 & 1) == grp) ? 0 : 1;  // this group's first block of the token
      if (i < nblk) {
        lse2 = h < p.H ? __ldg(p.lse + static_cast<size_t>(t) * p.H + h) : INFINITY;
        dlt_s = h < p.H ? __ldg(p.delta + static_cast<size_t>(t) * p.H + h) * p.scale : 0.f;
      }
      const int32_t* idx_row = p.idx + static_cast<size_t>(t) * p.topk;
      auto load_idx = [&](int blk, int half) -> int {
        const int j = blk * L::kBI + 32 * half + lane;
        return (blk < nblk && j < p.topk) ? __ldg(idx_row + j) : -1;
      };
      int r0 = load_idx(i, 0), r1 = load_idx(i, 1);
      for (; ok && i < nblk; i += 2) {
        const int G = G0 + i;
        const int n = G >> 1;  // this group's block count
        // Valid-slot masks of the block's two 32-slot halves (prefetched).
        const uint32_t m0 = __ballot_sync(0xffffffffu, static_cast<unsigned>(r0) < static_cast<unsigned>(p.S_kv));
        const uint32_t m1 = __ballot_sync(0xffffffffu, static_cast<unsigned>(r1) < static_cast<unsigned>(p.S_kv));
        r0 = load_idx(i + 2, 0);
        r1 = load_idx(i + 2, 1);
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSdpFull + grp), n & 1, ctl));
        if (!ok) break;
        tc_fence_after();
        if constexpr (NC == 2) {
          uint32_t hs[2][16], hp[2][16], own_exps[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            own_exps[hh] = own_partials_bfp(t_s + 32 * hh, t_dp + 32 * hh, p.scale_log2, p.scale,
                                            hs[hh], hp[hh]);
          tc_fence_before();
          mbar_arrive(bar(L::kBarSdpFree + grp));
          // Send: the peer has consumed this group's previous block from the
          // buffer.
          if (n >= 1) {
            ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarSendOk + grp), (n - 1) & 1, ctl));
            if (!ok) break;
          }
          {
            uint4* dst = reinterpret_cast<uint4*>(send) + h;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                dst[(4 * hh + c) * L::kHPad] = make_uint4(hs[hh][4 * c], hs[hh][4 * c + 1],
                                                          hs[hh][4 * c + 2], hs[hh][4 * c + 3]);
                dst[(8 + 4 * hh + c) * L::kHPad] = make_uint4(hp[hh][4 * c], hp[hh][4 * c + 1],
                                                              hp[hh][4 * c + 2], hp[hh][4 * c + 3]);
              }
            uint32_t* ex = reinterpret_cast<uint32_t*>(send + L::kXchgScaleOff);
            ex[h] = own_exps[0];
            ex[L::kHPad + h] = own_exps[1];
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(peer_full);
          }
          // The P / dS buffer was last read by the gradient MMAs of block G-1.
          if (G >= 1) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(L::kBarPdsFree + ((G - 1) & 1)), ((G - 1) >> 1) & 1, ctl));
            if (!ok) break;
          }
          ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarRecvFull + grp), n & 1, ctl));
          if (!ok) break;
          const uint4* src = reinterpret_cast<const uint4*>(recv) + h;
          const unsigned int* pex = reinterpret_cast<const unsigned int*>(recv + L::kXchgScaleOff);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t peer_exps = __ldcg(pex + hh * L::kHPad + h);
            const float us = bfp16_unit<false>(own_exps[hh]), up = bfp16_unit<true>(own_exps[hh]);
            const float vs = bfp16_unit<false>(peer_exps), vp = bfp16_unit<true>(peer_exps);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 ys = __ldcg(src + (4 * hh + c) * L::kHPad);
              const uint4 yp = __ldcg(src + (8 + 4 * hh + c) * L::kHPad);
              const uint32_t ysa[4] = {ys.x, ys.y, ys.z, ys.w};
              const uint32_t ypa[4] = {yp.x, yp.y, yp.z, yp.w};
              float zs[8], zp[8];
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                // Both decodings are exact; the sum is one rounding and
                // commutes, so the two CTAs get the same full S and dP.
                const float2 a =
                    add2(bfp16_unpack(hs[hh][4 * c + kk], us), bfp16_unpack(ysa[kk], vs));
                const float2 d =
                    add2(bfp16_unpack(hp[hh][4 * c + kk], up), bfp16_unpack(ypa[kk], vp));
                zs[2 * kk] = a.x;
                zs[2 * kk + 1] = a.y;
                zp[2 * kk] = d.x;
                zp[2 * kk + 1] = d.y;
              }
              emit(4 * hh + c, hh == 0 ? m0 : m1, zs, zp);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(L::kBarPdsFull + grp));
          // The exchange buffer may take the peer's next block of this
          // parity (a cluster-scope release: signalled after P / dS so the
          // gradients need not wait; the last one is never waited for).
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(peer_sendok);
        } else {
          // One CTA per token: the tile holds the full S and dP.  It is read
          // half by half right before the half is written, so it stays busy
          // until the P / dS buffer is free.
          if (G >= 1) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(L::kBarPdsFree + ((G - 1) & 1)), ((G - 1) >> 1) & 1, ctl));
            if (!ok) break;
          }
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            float xs[32], xp[32];
            tmem_ld32x2(t_s + 32 * hh, t_dp + 32 * hh, xs, xp);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              float zs[8], zp[8];
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                zs[kk] = xs[8 * c + kk] * p.scale_log2;
                zp[kk] = xp[8 * c + kk] * p.scale;
              }
              emit(4 * hh + c, hh == 0 ? m0 : m1, zs, zp);
            }
          }
          tc_fence_before();
          mbar_arrive(bar(L::kBarSdpFree + grp));
          fence_proxy_async_smem();
          mbar_arrive(bar(L::kBarPdsFull + grp));
        }
      }
      G0 += nblk;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (NC == 2) cluster_sync();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  // Release the pair's exchange slot once both CTAs are done with it.
  if (NC == 2 && rank == 0 && threadIdx.x == 0 && slot >= 0) {
    __threadfence();
    atomicExch(p.slot_flags + slot, 0);
  }
}

// Clusters (pairs, or single CTAs for D = 64) of one instantiation that fit
// on the device at once, per device (the persistent grid's size).
template <int DC, int NC, bool DET>
static int bwd_resident_clusters(cudaLaunchConfig_t cfg) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  int n = 0;
  auto kern = smqa_bwd_kernel<DC, NC, DET>;
  if (NC > 1) {
    cfg.gridDim = dim3(NC, 1, 1);
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  } else {
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, static_cast<int>(cfg.blockDim.x),
                                                      cfg.dynamicSmemBytes) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      n = per_sm * sms;
  }
  if (n <= 0) {
    (void)cudaGetLastError();
    return 0;
  }
  cached[dev] = n;
  return n;
}

template <int DC, int NC, bool DET>
static cudaError_t launch_bwd_impl(const CUtensorMap& tm_q, const CUtensorMap& tm_do,
                                   const BwdParams& p0, int tokens, cudaStream_t stream) {
  using L = BwdLayout<DC, NC>;
  auto kern = smqa_bwd_kernel<DC, NC, DET>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(L::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int resident = bwd_resident_clusters<DC, NC, DET>(cfg);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  BwdParams p = p0;
  p.tokens = tokens;
  p.clusters = tokens < resident ? tokens : resident;
  cfg.gridDim = dim3(static_cast<unsigned>(p.clusters) * NC, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, tm_q, tm_do, p);
}

cudaError_t launch_bwd_main(const CUtensorMap& tm_q, const CUtensorMap& tm_do,
                            const BwdParams& p, int tokens, cudaStream_t stream) {
  // The deterministic mode is a separate instantiation, so the default
  // kernel's reduction loop carries no branch for it.
  if (p.D == 512)
    return p.det ? launch_bwd_impl<256, 2, true>(tm_q, tm_do, p, tokens, stream)
                 : launch_bwd_impl<256, 2, false>(tm_q, tm_do, p, tokens, stream);
  if (p.D == 64)
    return p.det ? launch_bwd_impl<64, 1, true>(tm_q, tm_do, p, tokens, stream)
                 : launch_bwd_impl<64, 1, false>(tm_q, tm_do, p, tokens, stream);
  return cudaErrorInvalidValue;
}

static int grid_for(int64_t work, int per_block) {
  int64_t g = (work + per_block - 1) / per_block;
  if (g < 1) g = 1;
  if (g > 152 * 16) g = 152 * 16;
  return static_cast<int>(g);
}

cudaError_t launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* dout, float* delta,
                                  float* dkv_acc, int64_t rows, int D, int64_t acc_elems,
                                  cudaStream_t stream) {
  const int64_t acc_vec4 = acc_elems / 4;
  const int64_t work = rows * 32 > acc_vec4 ? rows * 32 : acc_vec4;
  smqa_bwd_pre_kernel<<<grid_for(work, 256), 256, 0, stream>>>(o, dout, delta, dkv_acc, rows, D,
                                                               acc_vec4);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post_fixed(const unsigned long long* acc, void* out, int fp32_out,
                                 int64_t elems, const int* shift, cudaStream_t stream) {
  const int64_t vec4 = elems / 4;
  smqa_bwd_post_fixed_kernel<<<grid_for(vec4, 256), 256, 0, stream>>>(acc, out, fp32_out, vec4,
                                                                      shift);
  return cudaGetLastError();
}

cudaError_t launch_bwd_det_stats(const __nv_bfloat16* q, const __nv_bfloat16* kv,
                                 const __nv_bfloat16* dout, const float* delta,
                                 const int32_t* idx, const smqa_shape& s, uint32_t* stats,
                                 uint32_t* counts, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(s.B) * s.S * s.H;
  const int64_t kv_rows = static_cast<int64_t>(s.B) * s.S_kv;
  const int64_t slots = static_cast<int64_t>(s.B) * s.S * s.topk;
  const int64_t work = rows * 32 > slots ? rows * 32 : slots;
  smqa_bwd_det_stats_kernel<<<grid_for(work, 256), 256, 0, stream>>>(
      q, kv, dout, delta, idx, rows, kv_rows, s.D, s.S, s.S_kv, s.topk, stats, counts);
  return cudaGetLastError();
}

cudaError_t launch_bwd_det_scale(const smqa_shape& s, float scale, uint32_t* stats,
                                 const uint32_t* counts, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(s.B) * s.S_kv;
  int g = static_cast<int>((n + 256 * 16 - 1) / (256 * 16));
  if (g < 1) g = 1;
  if (g > 152) g = 152;
  smqa_bwd_det_scale_kernel<<<g, 256, 0, stream>>>(stats, counts, n, s.H, scale);
  return cudaGetLastError();
}

cudaError_t launch_bwd_sink_grad(const float* sink, const float* lse, const float* delta,
                                float* dsink, int64_t tokens, int H, cudaStream_t stream) {
  smqa_bwd_sink_kernel<<<H, 256, 0, stream>>>(sink, lse, delta, dsink, tokens, H);
  return cudaGetLastError();
}

cudaError_t launch_bwd_postprocess(const float* acc, __nv_bfloat16* out, int64_t elems,
                                   cudaStream_t stream) {
  const int64_t vec8 = elems / 8;
  smqa_bwd_post_kernel<<<grid_for(vec8, 256), 256, 0, stream>>>(acc, out, vec8);
  return cudaGetLastError();
}

}  // namespace smqa
