// smqa_fwd.cu -- forward of top-k sparse MQA with an attention sink on sm_103a.
//
// What it computes (DeepSeek-V4 kernel pages of NeMo AutoModel,
// tilelang_sparse_mla_fwd: `sparse_mqa_fwd_interface` / `sparse_mqa_fwd`):
// for every token t = (b, s) and head h,
//   O[t,h,:] = sum_j p_j kv[b, idx[t,j], :],
//   p_j = exp(c q.k_j) / (sum_valid exp(c q.k) + exp(sink_h)),
//   lse[t,h] = log2 of that denominator,
// over the slots j whose index lies in [0, S_kv).
//
// Design (one token per CTA, or per CTA pair when D = 512):
//   * The token's H heads form the M = 128 rows of every MMA (heads beyond H
//     are zero rows), so the H heads sharing one gathered kv block make a
//     real GEMM for the tcgen05 tensor core.
//   * D = 512: a 2-CTA cluster splits the head dim; CTA r holds columns
//     [256r, 256r+256) of q, of every gathered kv row and of O.  Its O
//     accumulator (128 x 256 fp32) takes half of TMEM, the score tiles the
//     rest.  Each CTA computes partial scores over its half of D, sends them
//     to its peer with st.async into the peer's shared memory, and adds the
//     peer's half; both CTAs then run the same softmax on identical scores.
//   * Warp roles: warp 4 gathers kv rows with TMA gather4 (4 rows x 128 B
//     per instruction, 128-byte swizzle, multi-stage ring); warp 5 owns TMEM
//     and issues the MMAs from one thread; warps 0-3 (thread = head row =
//     TMEM lane) run the masked online softmax in the exp2 domain, rescale O
//     lazily (only when the running max grows by more than 2^8), write P as
//     bf16 for the P.V MMA and finish with the sink and the log2 LSE.
//   * Masked slots load a real (finite) row and get a -inf score, so their
//     probability is exactly 0.
#include <cuda_runtime.h>

#include "smqa_internal.h"
#include "smqa_ptx.cuh"

namespace smqa {

template <int DC, int NC>
struct FwdLayout {
  static constexpr int kHPad = 128;         // MMA M: heads padded to 128
  static constexpr int kBI = 64;            // slots per block
  static constexpr int kChunks = DC / 64;   // 64-column (128-byte) swizzle chunks
  static constexpr int kStages = NC == 2 ? 3 : 4;
  static constexpr uint32_t kQBytes = kHPad * DC * 2;
  static constexpr uint32_t kQChunkBytes = kHPad * 128;
  static constexpr uint32_t kKvChunkBytes = kBI * 128;
  static constexpr uint32_t kKvStageBytes = kChunks * kKvChunkBytes;
  static constexpr uint32_t kPBytes = kHPad * kBI * 2;
  static constexpr uint32_t kRecvBytes = NC == 2 ? kHPad * kBI * 4 : 0;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKv = kOffQ + kQBytes;
  static constexpr uint32_t kOffP = kOffKv + kStages * kKvStageBytes;
  static constexpr uint32_t kOffRecv = kOffP + 2 * kPBytes;
  static constexpr uint32_t kOffCtrl = kOffRecv + kRecvBytes;
  // barrier indices
  static constexpr int kBarKvFull = 0;
  static constexpr int kBarKvEmpty = kBarKvFull + kStages;
  static constexpr int kBarSFull = kBarKvEmpty + kStages;
  static constexpr int kBarSFree = kBarSFull + 2;
  static constexpr int kBarPFull = kBarSFree + 2;
  static constexpr int kBarODone = kBarPFull + 2;
  static constexpr int kBarRecvFull = kBarODone + 2;
  static constexpr int kBarSendOk = kBarRecvFull + 1;
  static constexpr int kBarQFull = kBarSendOk + 1;
  static constexpr int kBarDrain = kBarQFull + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kOffMask = kOffCtrl + 8 * kNumBars;
  static constexpr uint32_t kOffTmemHolder = kOffMask + 8 * kStages;
  static constexpr uint32_t kOffAbort = kOffTmemHolder + 4;
  static constexpr uint32_t kCtrlBytes = 512;
  static_assert(kOffAbort + 4 - kOffCtrl <= kCtrlBytes, "control block overflow");
  // +1024 so the dynamic buffer can be realigned to 1024 bytes (swizzle atoms)
  static constexpr uint32_t kSmemBytes = kOffCtrl + kCtrlBytes + 1024;
  static constexpr uint32_t kTmemO = 0;
  static constexpr uint32_t kTmemS = DC;
  static constexpr uint32_t kTmemCols = (DC + 2 * kBI) <= 256 ? 256 : 512;
  static constexpr int kThreads = 192;
};

template <int DC, int NC>
__global__ void __launch_bounds__(192, 1)
    smqa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_kv, const FwdParams p) {
  using L = FwdLayout<DC, NC>;
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
      mbar_init(bar(L::kBarKvFull + s), 1);
      mbar_init(bar(L::kBarKvEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::kBarSFull + i), 1);
      mbar_init(bar(L::kBarSFree + i), 128);
      mbar_init(bar(L::kBarPFull + i), 128);
      mbar_init(bar(L::kBarODone + i), 1);
    }
    mbar_init(bar(L::kBarRecvFull), 1);
    mbar_init(bar(L::kBarSendOk), 128);
    mbar_init(bar(L::kBarQFull), 1);
    mbar_init(bar(L::kBarDrain), 1);
    *abort_flag = *reinterpret_cast<volatile int*>(p.status) != 0 ? 1 : 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_kv);
  }
  if (warp == 5) tmem_alloc(base + L::kOffTmemHolder, L::kTmemCols);
  // Heads beyond H are zero rows of the A operand (the TMA box covers H rows).
  if (threadIdx.x < L::kHPad && static_cast<int>(threadIdx.x) >= p.H) {
    const uint32_t h = threadIdx.x;
#pragma unroll
    for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_shared_v4(base + L::kOffQ + c * L::kQChunkBytes + h * 128u + k * 16u, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if (NC == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    int issued = 0;  // blocks whose gather was issued
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(L::kBarQFull), static_cast<uint32_t>(p.H) * 128u * L::kChunks);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_2d(base + L::kOffQ + c * L::kQChunkBytes, &tm_q,
                    static_cast<int>(rank) * DC + c * 64, t * p.H, bar(L::kBarQFull));
    }
    const int32_t* idx_row = p.idx + static_cast<size_t>(t) * p.topk;
    for (int i = 0; i < nblk; ++i) {
      const int s = i % L::kStages;
      if (i >= L::kStages) {
        bool ok = mbar_wait(bar(L::kBarKvEmpty + s), ((i / L::kStages) - 1) & 1, ctl);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      const int j0 = i * L::kBI + lane;
      const int j1 = j0 + 32;
      const int r0 = j0 < p.topk ? __ldg(idx_row + j0) : -1;
      const int r1 = j1 < p.topk ? __ldg(idx_row + j1) : -1;
      const bool v0 = static_cast<unsigned>(r0) < static_cast<unsigned>(p.S_kv);
      const bool v1 = static_cast<unsigned>(r1) < static_cast<unsigned>(p.S_kv);
      const int row0 = b * p.S_kv + (v0 ? r0 : 0);
      const int row1 = b * p.S_kv + (v1 ? r1 : 0);
      const uint32_t m_lo = __ballot_sync(0xffffffffu, v0);
      const uint32_t m_hi = __ballot_sync(0xffffffffu, v1);
      int gy[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int src = 4 * (lane & 15) + k;
        const int a = __shfl_sync(0xffffffffu, row0, src & 31);
        const int c = __shfl_sync(0xffffffffu, row1, src & 31);
        gy[k] = src < 32 ? a : c;
      }
      if (lane == 0) {
        masks[s] = static_cast<uint64_t>(m_lo) | (static_cast<uint64_t>(m_hi) << 32);
        mbar_arrive_expect_tx(bar(L::kBarKvFull + s), L::kKvStageBytes);
      }
      __syncwarp();
      if (lane < 16) {
        const uint32_t dst0 = base + L::kOffKv + s * L::kKvStageBytes + lane * 4u * 128u;
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_gather4(dst0 + c * L::kKvChunkBytes, &tm_kv, static_cast<int>(rank) * DC + c * 64,
                      gy[0], gy[1], gy[2], gy[3], bar(L::kBarKvFull + s));
      }
      issued = i + 1;
    }
    // Let every copy this warp started land before the CTA can exit.
    if (lane == 0) {
      mbar_wait_drain(bar(L::kBarQFull), 0);
      for (int i = issued - L::kStages; i < issued; ++i)
        if (i >= 0) mbar_wait_drain(bar(L::kBarKvFull + i % L::kStages), (i / L::kStages) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, L::kBI, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, DC, false, true);
      auto issue_pv = [&](int j) -> bool {
        const int bj = j & 1;
        const int sj = j % L::kStages;
        if (!mbar_wait(bar(L::kBarPFull + bj), (j >> 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint32_t p_base = base + L::kOffP + bj * L::kPBytes;
        const uint32_t v_base = base + L::kOffKv + sj * L::kKvStageBytes;
#pragma unroll
        for (int k = 0; k < L::kBI / 16; ++k) {
          const uint64_t a = smem_desc(p_base + k * 32u, 16u, 1024u, kSwizzle128B);
          const uint64_t bd = smem_desc(v_base + k * 2048u, L::kKvChunkBytes, 1024u, kSwizzle128B);
          mma_ss(tmem + L::kTmemO, a, bd, idesc_o, (j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar(L::kBarKvEmpty + sj));
        mma_commit(bar(L::kBarODone + bj));
        return true;
      };
      bool ok = mbar_wait(bar(L::kBarQFull), 0, ctl);
      for (int i = 0; ok && i < nblk; ++i) {
        const int s = i % L::kStages;
        const int bb = i & 1;
        if (!mbar_wait(bar(L::kBarKvFull + s), (i / L::kStages) & 1, ctl)) { ok = false; break; }
        if (i >= 2 && !mbar_wait(bar(L::kBarSFree + bb), ((i >> 1) - 1) & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kv_base = base + L::kOffKv + s * L::kKvStageBytes;
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = smem_desc(base + L::kOffQ + c * L::kQChunkBytes + k * 32u, 16u,
                                         1024u, kSwizzle128B);
            const uint64_t bd = smem_desc(kv_base + c * L::kKvChunkBytes + k * 32u, 16u, 1024u,
                                          kSwizzle128B);
            mma_ss(tmem + L::kTmemS + bb * L::kBI, a, bd, idesc_s, (c | k) != 0 ? 1u : 0u);
          }
        }
        mma_commit(bar(L::kBarSFull + bb));
        if (i >= 1 && !issue_pv(i - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(nblk - 1);
      // No MMA may still be running when TMEM is released.
      mma_commit(bar(L::kBarDrain));
      mbar_wait_drain(bar(L::kBarDrain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int h = threadIdx.x;  // head row == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // exp2 argument: score * (c log2 e), or (score * c) * log2 e with the
    // reference-rounding flag (x * s1 * 1 is exact when the flag is off).
    const float s1 = p.ref_round ? p.scale : p.scale_log2;
    const float s2 = p.ref_round ? 1.4426950408889634f : 1.f;
    float m_run = -INFINITY;
    float l_run = 0.f;
    uint32_t peer_recv = 0, peer_recv_bar = 0, peer_sendok = 0;
    if (NC == 2) {
      peer_recv = mapa_shared(base + L::kOffRecv, rank ^ 1u);
      peer_recv_bar = mapa_shared(bar(L::kBarRecvFull), rank ^ 1u);
      peer_sendok = mapa_shared(bar(L::kBarSendOk), rank ^ 1u);
    }
    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
      const int bb = i & 1;
      const int s = i % L::kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull + bb), (i >> 1) & 1, ctl));
      if (!ok) break;
      tc_fence_after();
      float x[64];
      {
        float* x0 = x;
        tmem_ld32(tmem + lane_base + L::kTmemS + bb * L::kBI,
                  *reinterpret_cast<float(*)[32]>(x0));
        tmem_ld32(tmem + lane_base + L::kTmemS + bb * L::kBI + 32,
                  *reinterpret_cast<float(*)[32]>(x0 + 32));
      }
      tc_fence_before();
      mbar_arrive(bar(L::kBarSFree + bb));
      if (NC == 2) {
        // Exchange partial scores with the peer CTA (the other half of D).
        if (i >= 1) {
          ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarSendOk), (i - 1) & 1, ctl));
          if (!ok) break;
        }
        const uint32_t row_off = static_cast<uint32_t>(h) * 256u;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_async_v4(peer_recv + row_off + ((c ^ (h & 7)) << 4), x[4 * c], x[4 * c + 1],
                      x[4 * c + 2], x[4 * c + 3], peer_recv_bar);
        if (h == 0) mbar_arrive_expect_tx(bar(L::kBarRecvFull), L::kRecvBytes);
        ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarRecvFull), i & 1, ctl));
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float y0, y1, y2, y3;
          ld_shared_v4f(base + L::kOffRecv + row_off + ((c ^ (h & 7)) << 4), y0, y1, y2, y3);
          x[4 * c] += y0;
          x[4 * c + 1] += y1;
          x[4 * c + 2] += y2;
          x[4 * c + 3] += y3;
        }
        if (i + 1 < nblk) mbar_arrive_remote(peer_sendok);
      }
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarKvFull + s), (i / L::kStages) & 1, ctl));
      if (!ok) break;
      const uint64_t msk = masks[s];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        x[j] = ((msk >> j) & 1ull) ? (x[j] * s1) * s2 : -INFINITY;
        mx = fmaxf(mx, x[j]);
      }
      const float m_new = fmaxf(m_run, mx);
      const bool bump = (m_run == -INFINITY) ? (m_new != -INFINITY) : (m_new > m_run + 8.f);
      float alpha = 1.f;
      if (bump) {
        alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
      }
      // O was accumulated against the old max: rescale it (whole warp, since
      // the TMEM accesses are warp-collective; rows without a bump use 1).
      const bool need_rescale = bump && alpha != 0.f && i > 0;
      if (__any_sync(0xffffffffu, need_rescale)) {
        const int jp = i - 1;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(L::kBarODone + (jp & 1)), (jp >> 1) & 1, ctl));
        if (!ok) break;
        tc_fence_after();
        const float a = need_rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < DC / 32; ++c) {
          float v[32];
          tmem_ld32(tmem + lane_base + L::kTmemO + c * 32, v);
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] *= a;
          tmem_st32(tmem + lane_base + L::kTmemO + c * 32, v);
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      // P buffer `bb` was last read by the P.V MMA of block i-2.
      if (i >= 2) {
        const int jp = i - 2;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(L::kBarODone + (jp & 1)), (jp >> 1) & 1, ctl));
        if (!ok) break;
      }
      uint32_t pk[32];
      float rs = 0.f;
#pragma unroll
      for (int w = 0; w < 32; ++w) {
        const float p0 = fast_exp2(x[2 * w] - m_use);
        const float p1 = fast_exp2(x[2 * w + 1] - m_use);
        pk[w] = pack_bf16x2(p0, p1);
        rs += p0 + p1;  // fp32 probabilities: the LSE must not carry bf16 rounding
      }
      l_run += rs;
      const uint32_t p_row = base + L::kOffP + bb * L::kPBytes + static_cast<uint32_t>(h) * 128u;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(p_row + ((c ^ (h & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(L::kBarPFull + bb));
    }
    if (ok) {
      const int jl = nblk - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarODone + (jl & 1)), (jl >> 1) & 1, ctl));
    }
    if (ok) {
      tc_fence_after();
      const float sink2 = h < p.H ? __ldg(p.sink + h) * 1.4426950408889634f : 0.f;
      const float m_fin = fmaxf(m_run, sink2);
      const float so = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_fin);
      const float Z = l_run * so + fast_exp2(sink2 - m_fin);
      const float inv = so / Z;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(t) * p.H + h) * p.D +
                            static_cast<size_t>(rank) * DC;
#pragma unroll 1
      for (int c = 0; c < DC / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_base + L::kTmemO + c * 32, v);
        if (h < p.H) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(v[2 * k] * inv, v[2 * k + 1] * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
        }
      }
      if (rank == 0 && h < p.H) p.lse[static_cast<size_t>(t) * p.H + h] = m_fin + log2f(Z);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (NC == 2) cluster_sync();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int DC, int NC>
static cudaError_t launch_fwd_impl(const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                   const FwdParams& p, int tokens, cudaStream_t stream) {
  using L = FwdLayout<DC, NC>;
  auto kern = smqa_fwd_kernel<DC, NC>;
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
  return cudaLaunchKernelEx(&cfg, kern, tm_q, tm_kv, p);
}

cudaError_t launch_fwd(const CUtensorMap& tm_q, const CUtensorMap& tm_kv, const FwdParams& p,
                       int tokens, cudaStream_t stream) {
  if (p.D == 512) return launch_fwd_impl<256, 2>(tm_q, tm_kv, p, tokens, stream);
  if (p.D == 64) return launch_fwd_impl<64, 1>(tm_q, tm_kv, p, tokens, stream);
  return cudaErrorInvalidValue;
}

}  // namespace smqa
