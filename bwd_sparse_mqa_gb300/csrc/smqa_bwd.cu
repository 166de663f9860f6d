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
//   main         per token (a CTA pair for D = 512, each CTA owning half of
//                D): S = Q.K^T and dP = dO.V^T on the tensor core, partial
//                sums exchanged with the peer CTA through DSMEM, P and dS on
//                CUDA cores, then dQ += dS.K accumulated in TMEM over all
//                blocks and dKV^T = Q^T.dS + dO^T.P per block, which a drain
//                warpgroup reads from TMEM and scatters with fp32
//                red.global.add into the accumulator;
//   postprocess  fp32 accumulator -> bf16 (round to nearest even).
// dKV^T (lanes = head-dim rows, columns = slots) keeps M = 128 for 32-slot
// blocks and lets each warp's 32 lanes add to 32 consecutive floats of a row.
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
// main backward kernel
// --------------------------------------------------------------------------
template <int DC, int NC>
struct BwdLayout {
  static constexpr int kHPad = 128;
  static constexpr int kBI = 32;                 // slots per block
  static constexpr int kChunks = DC / 64;
  static constexpr int kNE = DC >= 128 ? DC / 128 : 1;  // 128-row halves of dKV^T
  static constexpr int kStages = NC == 2 ? 3 : 4;
  static constexpr uint32_t kQChunkBytes = kHPad * 128;          // 16 KB
  static constexpr uint32_t kQBytes = kChunks * kQChunkBytes;
  static constexpr uint32_t kKvChunkBytes = kBI * 128;           // 4 KB
  static constexpr uint32_t kKvStageBytes = kChunks * kKvChunkBytes;
  static constexpr uint32_t kPBytes = kHPad * kBI * 2;           // 8 KB (64-byte rows)
  // peer's partial S and dP, fp16 (see the exchange in the P / dS role)
  static constexpr uint32_t kRecvBytes = NC == 2 ? kHPad * 2 * kBI * 2 : 0;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffDo = kOffQ + kQBytes;
  // For DC = 64 the 128-row M-major views of Q^T / dO^T read one chunk past
  // each tile (those rows are discarded); keep a full chunk mapped after dO.
  static constexpr uint32_t kOffKv = kOffDo + (kChunks >= 2 ? kQBytes : 2 * kQChunkBytes);
  static constexpr uint32_t kOffP = kOffKv + kStages * kKvStageBytes;
  static constexpr uint32_t kOffDs = kOffP + kPBytes;
  static constexpr uint32_t kOffRecv = kOffDs + kPBytes;
  static constexpr uint32_t kOffCtrl = kOffRecv + kRecvBytes;
  static constexpr int kBarKvFull = 0;
  static constexpr int kBarKvEmpty = kBarKvFull + kStages;
  static constexpr int kBarSdpFull = kBarKvEmpty + kStages;
  static constexpr int kBarSdpFree = kBarSdpFull + 1;
  static constexpr int kBarPdsFull = kBarSdpFree + 1;
  static constexpr int kBarPdsFree = kBarPdsFull + 1;
  static constexpr int kBarDkvFull = kBarPdsFree + 1;  // [2]
  static constexpr int kBarDkvFree = kBarDkvFull + 2;  // [2]
  static constexpr int kBarRecvFull = kBarDkvFree + 2;
  static constexpr int kBarSendOk = kBarRecvFull + 1;
  static constexpr int kBarQdoFull = kBarSendOk + 1;
  static constexpr int kBarDqDone = kBarQdoFull + 1;
  static constexpr int kBarDrain = kBarDqDone + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kOffMask = kOffCtrl + 8 * kNumBars;
  static constexpr uint32_t kOffTmemHolder = kOffMask + 8 * kStages;
  static constexpr uint32_t kOffAbort = kOffTmemHolder + 4;
  static constexpr uint32_t kCtrlBytes = 512;
  static_assert(kOffAbort + 4 - kOffCtrl <= kCtrlBytes, "control block overflow");
  static constexpr uint32_t kSmemBytes = kOffCtrl + kCtrlBytes + 1024;
  static constexpr uint32_t kTmemDq = 0;
  static constexpr uint32_t kTmemS = DC;
  static constexpr uint32_t kTmemDp = DC + kBI;
  static constexpr uint32_t kTmemDkv = DC + 2 * kBI;  // + buf * kNE * kBI + e * kBI
  static constexpr uint32_t kTmemUsed = kTmemDkv + 2 * kNE * kBI;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  // warps 0-3: P / dS (thread = head row); 4-7: dKV drain (thread = head-dim
  // row); 8-9: gather; 10: TMEM owner + MMA issuer
  static constexpr int kProducerWarp0 = 8;
  static constexpr int kMmaWarp = 10;
  static constexpr int kThreads = 352;
};

template <int DC, int NC>
__global__ void __launch_bounds__(352, 1)
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
  const int t = blockIdx.x / NC;
  const uint32_t rank = NC == 2 ? cluster_ctarank() : 0u;
  const int b = t / p.S;
  const int nblk = (p.topk + L::kBI - 1) / L::kBI;
  auto bar = [&](int i) -> uint32_t { return base + L::kOffCtrl + 8u * static_cast<uint32_t>(i); };
  volatile uint64_t* masks = reinterpret_cast<volatile uint64_t*>(smem + L::kOffMask);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + L::kOffTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  const WaitCtl ctl{abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarKvFull + s), 64);  // every gather thread arrives
      mbar_init(bar(L::kBarKvEmpty + s), 1);
    }
    mbar_init(bar(L::kBarSdpFull), 1);
    mbar_init(bar(L::kBarSdpFree), 128);
    mbar_init(bar(L::kBarPdsFull), 128);
    mbar_init(bar(L::kBarPdsFree), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::kBarDkvFull + i), 1);
      mbar_init(bar(L::kBarDkvFree + i), 128);
    }
    mbar_init(bar(L::kBarRecvFull), 128);
    mbar_init(bar(L::kBarSendOk), 128);
    mbar_init(bar(L::kBarQdoFull), 1);
    mbar_init(bar(L::kBarDqDone), 1);
    mbar_init(bar(L::kBarDrain), 1);
    *abort_flag = *reinterpret_cast<volatile int*>(p.status) != 0 ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == L::kMmaWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
    }
    tmem_alloc(base + L::kOffTmemHolder, L::kTmemCols);
  }
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

  if (warp >= L::kProducerWarp0 && warp < L::kMmaWarp) {
    // ------------------------------------------------------------ gather
    // Warp pw copies slots [16 pw, 16 pw + 16) of each 32-slot block; one warp
    // instruction moves kRpi whole rows of this CTA's D slice (32 lanes x 16
    // bytes, coalesced) into the 128-byte-swizzled tile with cp.async.
    const int pw = warp - L::kProducerWarp0;
    constexpr int kCpr = DC / 8;
    constexpr int kRpi = 32 / kCpr;
    const int rsub = lane / kCpr;
    const int cc = lane % kCpr;
    const uint32_t lane_off = static_cast<uint32_t>(cc / 8) * L::kKvChunkBytes;
    const uint32_t c16 = static_cast<uint32_t>(cc % 8);
    const __nv_bfloat16* kv_col = p.kv + static_cast<size_t>(rank) * DC + cc * 8;
    const int32_t* idx_row = p.idx + static_cast<size_t>(t) * p.topk;
    auto load_idx = [&](int blk) -> int {
      const int j = blk * L::kBI + lane;
      return j < p.topk ? __ldg(idx_row + j) : -1;
    };
    int r_next = load_idx(0);
    if (warp == L::kProducerWarp0 && lane == 0) {
      mbar_arrive_expect_tx(bar(L::kBarQdoFull),
                            2u * static_cast<uint32_t>(p.H) * 128u * L::kChunks);
      for (int c = 0; c < L::kChunks; ++c) {
        const int x = static_cast<int>(rank) * DC + c * 64;
        tma_load_2d(base + L::kOffQ + c * L::kQChunkBytes, &tm_q, x, t * p.H, bar(L::kBarQdoFull));
        tma_load_2d(base + L::kOffDo + c * L::kQChunkBytes, &tm_do, x, t * p.H,
                    bar(L::kBarQdoFull));
      }
    }
    int i = 0;
    for (; i < nblk; ++i) {
      const int s = i % L::kStages;
      const int r = r_next;
      if (i + 1 < nblk) r_next = load_idx(i + 1);
      const bool v = static_cast<unsigned>(r) < static_cast<unsigned>(p.S_kv);
      const int row = b * p.S_kv + (v ? r : 0);
      const uint32_t m = __ballot_sync(0xffffffffu, v);
      if (i >= L::kStages) {
        const bool ok = mbar_wait(bar(L::kBarKvEmpty + s), ((i / L::kStages) - 1) & 1, ctl);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (pw == 0 && lane == 0) masks[s] = m;
      const uint32_t stage = base + L::kOffKv + s * L::kKvStageBytes + lane_off;
#pragma unroll
      for (int k = 0; k < 16 / kRpi; ++k) {
        const int rloc = 16 * pw + k * kRpi + rsub;
        const int rr = __shfl_sync(0xffffffffu, row, rloc);
        const uint32_t srow = static_cast<uint32_t>(rloc);
        cp_async_16(stage + srow * 128u + ((c16 ^ (srow & 7u)) << 4),
                    kv_col + static_cast<size_t>(rr) * p.D);
      }
      cp_async_commit();
      if (i >= 1) {
        cp_async_wait_group<1>();
        fence_proxy_async_smem();
        mbar_arrive(bar(L::kBarKvFull + (i - 1) % L::kStages));
      }
    }
    cp_async_wait_group<0>();
    fence_proxy_async_smem();
    if (i == nblk) mbar_arrive(bar(L::kBarKvFull + (nblk - 1) % L::kStages));
    if (warp == L::kProducerWarp0 && lane == 0) mbar_wait_drain(bar(L::kBarQdoFull), 0);
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
      const uint64_t d_ds = smem_desc(base + L::kOffDs, 16u, 512u, kSwizzle64B);
      const uint64_t d_qt = smem_desc(base + L::kOffQ, L::kQChunkBytes, 1024u, kSwizzle128B);
      const uint64_t d_dot = smem_desc(base + L::kOffDo, L::kQChunkBytes, 1024u, kSwizzle128B);
      const uint64_t d_dsmn = smem_desc(base + L::kOffDs, 8192u, 512u, kSwizzle64B);
      const uint64_t d_pmn = smem_desc(base + L::kOffP, 8192u, 512u, kSwizzle64B);
      auto issue_grad = [&](int j) -> bool {
        const int bk = j & 1;
        const int sj = j % L::kStages;
        if (!mbar_wait(bar(L::kBarPdsFull), j & 1, ctl)) return false;
        if (j >= 2 && !mbar_wait(bar(L::kBarDkvFree + bk), ((j >> 1) - 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint64_t dkv = d_kvmn + ((static_cast<uint32_t>(sj) * L::kKvStageBytes) >> 4);
        // dQ += dS' . K   (M = 128 heads, N = DC, K = 32 slots)
#pragma unroll
        for (int k = 0; k < L::kBI / 16; ++k)
          mma_ss(tmem + L::kTmemDq, d_ds + (k * 32u >> 4), dkv + (k * 2048u >> 4), idesc_dq,
                 (j > 0 || k > 0) ? 1u : 0u);
        // dKV^T[e] = Q^T[e] . dS' + dO^T[e] . P   (M = 128 dims, N = 32 slots, K = 128 heads)
#pragma unroll
        for (int e = 0; e < L::kNE; ++e) {
          const uint32_t d_tm = tmem + L::kTmemDkv + (bk * L::kNE + e) * L::kBI;
#pragma unroll
          for (int k = 0; k < L::kHPad / 16; ++k)
            mma_ss(d_tm, d_qt + ((2 * e * L::kQChunkBytes + k * 2048u) >> 4),
                   d_dsmn + (k * 1024u >> 4), idesc_dkv, k > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < L::kHPad / 16; ++k)
            mma_ss(d_tm, d_dot + ((2 * e * L::kQChunkBytes + k * 2048u) >> 4),
                   d_pmn + (k * 1024u >> 4), idesc_dkv, 1u);
        }
        mma_commit(bar(L::kBarPdsFree));
        mma_commit(bar(L::kBarKvEmpty + sj));
        mma_commit(bar(L::kBarDkvFull + bk));
        return true;
      };
      bool ok = mbar_wait(bar(L::kBarQdoFull), 0, ctl);
      for (int i = 0; ok && i < nblk; ++i) {
        const int s = i % L::kStages;
        if (!mbar_wait(bar(L::kBarKvFull + s), (i / L::kStages) & 1, ctl)) { ok = false; break; }
        if (i >= 1 && !mbar_wait(bar(L::kBarSdpFree), (i - 1) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dk = d_kv + ((static_cast<uint32_t>(s) * L::kKvStageBytes) >> 4);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t bd = dk + ((c * L::kKvChunkBytes + k * 32u) >> 4);
            const uint32_t acc = (c | k) != 0 ? 1u : 0u;
            mma_ss(tmem + L::kTmemS, d_q + ((c * L::kQChunkBytes + k * 32u) >> 4), bd, idesc_sdp,
                   acc);
            mma_ss(tmem + L::kTmemDp, d_do + ((c * L::kQChunkBytes + k * 32u) >> 4), bd,
                   idesc_sdp, acc);
          }
        }
        mma_commit(bar(L::kBarSdpFull));
        if (i >= 1 && !issue_grad(i - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_grad(nblk - 1);
      mma_commit(bar(L::kBarDqDone));
      mma_commit(bar(L::kBarDrain));
      mbar_wait_drain(bar(L::kBarDrain), 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dKV drain
    const int wq = warp - 4;  // TMEM lane quarter
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int32_t* idx_row = p.idx + static_cast<size_t>(t) * p.topk;
    const bool active = (wq * 32) < DC;  // DC = 64: rows 64..127 are padding
    for (int j = 0; j < nblk; ++j) {
      const int bk = j & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDkvFull + bk), (j >> 1) & 1, ctl));
      if (!ok) break;
      tc_fence_after();
      const int slot = j * L::kBI + lane;
      const int r = slot < p.topk ? __ldg(idx_row + slot) : -1;
      const bool v = static_cast<unsigned>(r) < static_cast<unsigned>(p.S_kv);
      const uint32_t vm = __ballot_sync(0xffffffffu, v);
      const int row = b * p.S_kv + (v ? r : 0);
      if (active) {
#pragma unroll 1
        for (int e = 0; e < L::kNE; ++e) {
          float x[32];
          tmem_ld32(tmem + lane_base + L::kTmemDkv + (bk * L::kNE + e) * L::kBI, x);
          float* col = p.dkv_acc + static_cast<size_t>(rank) * DC + e * 128 + wq * 32 + lane;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const int rk = __shfl_sync(0xffffffffu, row, k);
            if ((vm >> k) & 1u) red_add_f32(col + static_cast<size_t>(rk) * p.D, x[k]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::kBarDkvFree + bk));
    }
  } else {
    // ------------------------------------------------------------ P / dS
    const int h = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float cl2 = p.scale_log2;
    const float lse2 = h < p.H ? __ldg(p.lse + static_cast<size_t>(t) * p.H + h) : INFINITY;
    const float dlt_s =
        h < p.H ? __ldg(p.delta + static_cast<size_t>(t) * p.H + h) * p.scale : 0.f;
    uint32_t peer_recv = 0, peer_recv_bar = 0, peer_sendok = 0;
    if (NC == 2) {
      peer_recv = mapa_shared(base + L::kOffRecv, rank ^ 1u);
      peer_recv_bar = mapa_shared(bar(L::kBarRecvFull), rank ^ 1u);
      peer_sendok = mapa_shared(bar(L::kBarSendOk), rank ^ 1u);
    }
    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
      const int s = i % L::kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSdpFull), i & 1, ctl));
      if (!ok) break;
      tc_fence_after();
      float xs[32], xp[32];
      tmem_ld32(tmem + lane_base + L::kTmemS, xs);
      tmem_ld32(tmem + lane_base + L::kTmemDp, xp);
      tc_fence_before();
      mbar_arrive(bar(L::kBarSdpFree));
      // zs: score in the exp2 domain; zp: sm_scale * dP (so that
      // dS' = P (zp - sm_scale Delta) already carries the scale).
      if (NC == 2) {
        // Exchange partial S and dP with the peer CTA (the other half of D),
        // both rounded to fp16 first and summed in the same order on both
        // sides; fp16 halves the bytes on the CTA-to-CTA network.
        uint32_t hs[16], hp[16];
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          hs[w] = pack_f16x2_sat(xs[2 * w] * cl2, xs[2 * w + 1] * cl2);
          hp[w] = pack_f16x2_sat(xp[2 * w] * p.scale, xp[2 * w + 1] * p.scale);
        }
        if (i >= 1) {
          ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarSendOk), (i - 1) & 1, ctl));
          if (!ok) break;
        }
        const uint32_t row_off = static_cast<uint32_t>(h) * 128u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          st_cluster_v4u(peer_recv + row_off + ((c ^ (h & 7)) << 4), hs[4 * c], hs[4 * c + 1],
                         hs[4 * c + 2], hs[4 * c + 3]);
          st_cluster_v4u(peer_recv + row_off + (((c + 4) ^ (h & 7)) << 4), hp[4 * c],
                         hp[4 * c + 1], hp[4 * c + 2], hp[4 * c + 3]);
        }
        mbar_arrive_remote(peer_recv_bar);
        ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarRecvFull), i & 1, ctl));
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ys[4], yp[4];
          ld_shared_v4u(base + L::kOffRecv + row_off + ((c ^ (h & 7)) << 4), ys[0], ys[1], ys[2],
                        ys[3]);
          ld_shared_v4u(base + L::kOffRecv + row_off + (((c + 4) ^ (h & 7)) << 4), yp[0], yp[1],
                        yp[2], yp[3]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 ms = unpack_f16x2(hs[4 * c + k]);
            const float2 ps = unpack_f16x2(ys[k]);
            const float2 mp = unpack_f16x2(hp[4 * c + k]);
            const float2 pp2 = unpack_f16x2(yp[k]);
            xs[8 * c + 2 * k] = ms.x + ps.x;
            xs[8 * c + 2 * k + 1] = ms.y + ps.y;
            xp[8 * c + 2 * k] = mp.x + pp2.x;
            xp[8 * c + 2 * k + 1] = mp.y + pp2.y;
          }
        }
        if (i + 1 < nblk) mbar_arrive_remote(peer_sendok);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          xs[j] *= cl2;
          xp[j] *= p.scale;
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarKvFull + s), (i / L::kStages) & 1, ctl));
      if (!ok) break;
      const uint32_t msk = static_cast<uint32_t>(masks[s]);
      uint32_t pp[16], pd[16];
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        float pv[2], dv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int jj = 2 * w + u;
          const float pr = ((msk >> jj) & 1u) ? fast_exp2(xs[jj] - lse2) : 0.f;
          pv[u] = pr;
          dv[u] = pr * (xp[jj] - dlt_s);
        }
        pp[w] = pack_bf16x2(pv[0], pv[1]);
        pd[w] = pack_bf16x2(dv[0], dv[1]);
      }
      // P / dS buffers were last read by the gradient MMAs of block i-1.
      if (i >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarPdsFree), (i - 1) & 1, ctl));
        if (!ok) break;
      }
      const uint32_t row64 = static_cast<uint32_t>(h) * 64u;
      const uint32_t sw = static_cast<uint32_t>((h >> 1) & 3);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        st_shared_v4(base + L::kOffP + row64 + ((c ^ sw) << 4), pp[4 * c], pp[4 * c + 1],
                     pp[4 * c + 2], pp[4 * c + 3]);
        st_shared_v4(base + L::kOffDs + row64 + ((c ^ sw) << 4), pd[4 * c], pd[4 * c + 1],
                     pd[4 * c + 2], pd[4 * c + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::kBarPdsFull));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDqDone), 0, ctl));
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* qrow = p.dq + (static_cast<size_t>(t) * p.H + h) * p.D +
                            static_cast<size_t>(rank) * DC;
#pragma unroll 1
      for (int c = 0; c < DC / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_base + L::kTmemDq + c * 32, v);
        if (h < p.H) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
          uint4* dst = reinterpret_cast<uint4*>(qrow + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (NC == 2) cluster_sync();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int DC, int NC>
static cudaError_t launch_bwd_impl(const CUtensorMap& tm_q, const CUtensorMap& tm_do,
                                   const BwdParams& p, int tokens, cudaStream_t stream) {
  using L = BwdLayout<DC, NC>;
  auto kern = smqa_bwd_kernel<DC, NC>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tokens) * NC, 1, 1);
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
  return cudaLaunchKernelEx(&cfg, kern, tm_q, tm_do, p);
}

cudaError_t launch_bwd_main(const CUtensorMap& tm_q, const CUtensorMap& tm_do,
                            const BwdParams& p, int tokens, cudaStream_t stream) {
  if (p.D == 512) return launch_bwd_impl<256, 2>(tm_q, tm_do, p, tokens, stream);
  if (p.D == 64) return launch_bwd_impl<64, 1>(tm_q, tm_do, p, tokens, stream);
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

cudaError_t launch_bwd_postprocess(const float* acc, __nv_bfloat16* out, int64_t elems,
                                   cudaStream_t stream) {
  const int64_t vec8 = elems / 8;
  smqa_bwd_post_kernel<<<grid_for(vec8, 256), 256, 0, stream>>>(acc, out, vec8);
  return cudaGetLastError();
}

}  // namespace smqa
