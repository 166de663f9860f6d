// smqa_indexer.cu -- backward of the lightning indexer on sm_103a.
//
// What it computes (DeepSeek-V4 kernel pages of NeMo AutoModel,
// tilelang_indexer_bwd: `indexer_bwd_interface` for one batch element and
// `batched_indexer_bwd`): the gradient with respect to index_q of the
// indexer scores
//   score[t,j] = sum_h w[t,h] ReLU(q[t,h] . k[idx[t,j]])
// given grad_scores g[t,j]:
//   dq[t,h] = w[t,h] sum_j g[t,j] [q[t,h] . k_j > 0] k_j
// over the valid slots j (index in [0, S_kv)); the pages give the tensors but
// not the formula, so this is the plainest reading of them.
//
// One CTA per (token, batch element), two CTAs per SM.  Per 64-slot block:
//   gather (warps 4-5)  the block's key rows, 16-byte cp.async into a
//                       128-byte-swizzled K-major tile (three-stage ring), and
//                       its grad_scores with masked slots set to 0;
//   MMA (warp 6)        L = Q.K^T (M = 128 head rows, N = 64 slots, K = D)
//                       into one of two TMEM tiles, and once the block's gate
//                       operand is written, dq += G.K (K = 64 slots, N = D,
//                       the same key tile read MN-major) into a TMEM
//                       accumulator that lives for the whole token;
//   gate (warps 0-3)    thread = head row: G[h,j] = g_j if L[h,j] > 0 else 0,
//                       written bf16 as the K-major A operand of dq += G.K
//                       (one buffer, rewritten once the previous block's dq
//                       MMAs have read it).
// At the end warps 0-3 scale the accumulator by w[t,h], round it to bf16 and
// stage it in shared memory for TMA tensor stores.  Head rows H..127 of Q
// are zero, so their rows of dq are never stored.
#include <cuda_runtime.h>

#include "smqa_internal.h"
#include "smqa_ptx.cuh"

namespace smqa {

template <int D, int STAGES = 2, int GBUFS = 2, int CTAS = 2>
struct IdxLayout {
  static constexpr int kHPad = 128;
  static constexpr int kBI = 64;                    // slots per block
  static constexpr int kChunks = D / 64;            // 64-column (128-byte) chunks
  static constexpr int kStages = STAGES;            // key-tile ring
  static constexpr int kGateBufs = GBUFS;           // gate operand buffers
  static constexpr int kCtasPerSm = CTAS;
  static constexpr uint32_t kQChunkBytes = kHPad * 128;   // 16 KB
  static constexpr uint32_t kQBytes = kChunks * kQChunkBytes;
  static constexpr uint32_t kKvChunkBytes = kBI * 128;    // 8 KB
  static constexpr uint32_t kKvStageBytes = kChunks * kKvChunkBytes;
  static constexpr uint32_t kGateBytes = kHPad * kBI * 2; // 16 KB (bf16, 128-byte rows)
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKv = kOffQ + kQBytes;
  static constexpr uint32_t kOffGate = kOffKv + kStages * kKvStageBytes;  // [kGateBufs]
  static constexpr uint32_t kOffG = kOffGate + kGateBufs * kGateBytes;   // fp32 [kStages][64]
  static constexpr uint32_t kOffCtrl = kOffG + kStages * kBI * 4;
  static constexpr int kBarKvFull = 0;
  static constexpr int kBarKvEmpty = kBarKvFull + kStages;
  static constexpr int kBarLFull = kBarKvEmpty + kStages;  // [2]
  static constexpr int kBarLFree = kBarLFull + 2;          // [2]
  static constexpr int kBarGFull = kBarLFree + 2;          // [kGateBufs] gate operand written
  static constexpr int kBarGFree = kBarGFull + kGateBufs;  // [kGateBufs] gate operand read
  static constexpr int kBarQFull = kBarGFree + kGateBufs;
  static constexpr int kBarDqDone = kBarQFull + 1;
  static constexpr int kBarDrain = kBarDqDone + 1;
  static constexpr int kBarStaged = kBarDrain + 1;
  static constexpr int kNumBars = kBarStaged + 1;
  static constexpr uint32_t kOffTmemHolder = kOffCtrl + 8 * kNumBars;
  static constexpr uint32_t kOffAbort = kOffTmemHolder + 4;
  static constexpr uint32_t kOffWarpLast = kOffAbort + 4;  // int [8]
  static constexpr uint32_t kCtrlBytes = 256;
  static_assert(kOffWarpLast + 32 - kOffCtrl <= kCtrlBytes, "control block overflow");
  static constexpr uint32_t kSmemBytes = kOffCtrl + kCtrlBytes + 1024;
  static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 233472, "shared memory budget");
  static_assert(kChunks * kQChunkBytes <= kStages * kKvStageBytes, "dq staging fits the ring");
  // TMEM: two L tiles, then the dq accumulator.
  static constexpr uint32_t kTmemL = 0;
  static constexpr uint32_t kTmemDq = 2 * kBI;
  static constexpr uint32_t kTmemCols = 256;
  static_assert(kCtasPerSm * kTmemCols <= 512, "TMEM budget of the resident CTAs");
  static_assert(kTmemDq + D <= kTmemCols, "TMEM budget");
  static constexpr int kGatherWarp0 = 4;
  static constexpr int kMmaWarp = 6;
  static constexpr int kThreads = 224;
};

template <int D, int ST, int GB, int CT>
__global__ void __launch_bounds__(224, CT)
    smqa_indexer_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_dq, const IdxParams p) {
  using L = IdxLayout<D, ST, GB, CT>;
  extern __shared__ uint8_t smem_raw[];
  uint32_t base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  base += pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = static_cast<int>(blockIdx.x) / p.S;
  const int s = static_cast<int>(blockIdx.x) % p.S;
  // Row of (s, b, head 0) in q / weights / dq, and the token's index row.
  const int64_t row0 = static_cast<int64_t>(s) * p.q_tok_rows + static_cast<int64_t>(b) * p.q_b_rows;
  const int32_t* idx_row = p.idx + (static_cast<size_t>(b) * p.S + s) * p.topk;
  const float* g_row = p.g + (static_cast<size_t>(b) * p.S + s) * p.topk;
  auto bar = [&](int i) -> uint32_t { return base + L::kOffCtrl + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + L::kOffTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  const WaitCtl ctl{abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kStages; ++i) {
      // 64 cp.async completions + 64 plain arrivals (grad_scores stored).
      mbar_init(bar(L::kBarKvFull + i), 128);
      mbar_init(bar(L::kBarKvEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::kBarLFull + i), 1);
      mbar_init(bar(L::kBarLFree + i), 128);
    }
    for (int i = 0; i < L::kGateBufs; ++i) {
      mbar_init(bar(L::kBarGFull + i), 128);
      mbar_init(bar(L::kBarGFree + i), 1);
    }
    mbar_init(bar(L::kBarQFull), 1);
    mbar_init(bar(L::kBarDqDone), 1);
    mbar_init(bar(L::kBarDrain), 1);
    mbar_init(bar(L::kBarStaged), 128);
    *abort_flag = *reinterpret_cast<volatile int*>(p.status) != 0 ? 1 : 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(bar(L::kBarQFull), static_cast<uint32_t>(p.H) * 128u * L::kChunks);
    for (int c = 0; c < L::kChunks; ++c)
      tma_load_2d(base + L::kOffQ + c * L::kQChunkBytes, &tm_q, c * 64, static_cast<int>(row0),
                  bar(L::kBarQFull));
  }
  if (warp == L::kMmaWarp) {
    if (lane == 0) tma_prefetch_desc(&tm_q);
    tmem_alloc(base + L::kOffTmemHolder, L::kTmemCols);
  }
  if (threadIdx.x < L::kHPad && static_cast<int>(threadIdx.x) >= p.H) {
    const uint32_t h = threadIdx.x;
#pragma unroll
    for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_shared_v4(base + L::kOffQ + c * L::kQChunkBytes + h * 128u + k * 16u, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  volatile int* warp_last = reinterpret_cast<volatile int*>(smem + L::kOffWarpLast);
  scan_last_valid(idx_row, p.topk, p.S_kv, warp_last);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int nblk = live_blocks(warp_last, L::kBI);

  if (warp >= L::kGatherWarp0 && warp < L::kMmaWarp) {
    // ------------------------------------------------------------ gather
    // Thread = slot of the block (its index and grad_score); warp pw copies
    // the key rows of slots [32 pw, 32 pw + 32), kRpi whole rows per warp
    // instruction (32 lanes x 16 bytes, coalesced).
    const int pw = warp - L::kGatherWarp0;
    const int tid = threadIdx.x - L::kGatherWarp0 * 32;  // slot within a block
    constexpr int kCpr = D / 8;
    constexpr int kRpi = 32 / kCpr;
    const int rsub = lane / kCpr;
    const int cc = lane % kCpr;
    const uint32_t lane_off = static_cast<uint32_t>(cc / 8) * L::kKvChunkBytes;
    const uint32_t c16 = static_cast<uint32_t>(cc % 8);
    const __nv_bfloat16* k_col = p.k + static_cast<size_t>(b) * p.k_b_stride + cc * 8;
    for (int i = 0; i < nblk; ++i) {
      const int st = i % L::kStages;
      if (i >= L::kStages) {
        const bool ok = mbar_wait(bar(L::kBarKvEmpty + st), ((i / L::kStages) - 1) & 1, ctl);
        if (!__all_sync(0xffffffffu, ok)) break;
      } else if (*abort_flag) {
        break;
      }
      const int j = i * L::kBI + tid;
      const int r = j < p.topk ? __ldg(idx_row + j) : -1;
      const bool v = static_cast<unsigned>(r) < static_cast<unsigned>(p.S_kv);
      const float gj = (v && j < p.topk) ? __ldg(g_row + j) : 0.f;
      reinterpret_cast<volatile float*>(smem + L::kOffG)[st * L::kBI + tid] = gj;
      const int row = v ? r : 0;
      const uint32_t stage = base + L::kOffKv + st * L::kKvStageBytes + lane_off;
#pragma unroll
      for (int k = 0; k < 32 / kRpi; ++k) {
        const int rw = k * kRpi + rsub;  // row within this warp's 32
        const int rr = __shfl_sync(0xffffffffu, row, rw);
        const uint32_t srow = static_cast<uint32_t>(32 * pw + rw);
        cp_async_16(stage + srow * 128u + ((c16 ^ (srow & 7u)) << 4),
                    k_col + static_cast<size_t>(rr) * p.k_row_stride);
      }
      // One arrival when this thread's copies land, one now (it releases the
      // grad_score stored above).
      cp_async_arrive_noinc(bar(L::kBarKvFull + st));
      mbar_arrive(bar(L::kBarKvFull + st));
    }
    cp_async_wait_all();
    if (warp == L::kGatherWarp0 && lane == 0) mbar_wait_drain(bar(L::kBarQFull), 0);
  } else if (warp == L::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_l = idesc_bf16_f32(128, L::kBI, false, false);
      constexpr uint32_t idesc_dq = idesc_bf16_f32(128, D, false, true);
      const uint64_t d_q = smem_desc(base + L::kOffQ, 16u, 1024u, kSwizzle128B);
      const uint64_t d_kv = smem_desc(base + L::kOffKv, 16u, 1024u, kSwizzle128B);
      const uint64_t d_kvmn = smem_desc(base + L::kOffKv, L::kKvChunkBytes, 1024u, kSwizzle128B);
      const uint64_t d_gate = smem_desc(base + L::kOffGate, 16u, 1024u, kSwizzle128B);
      // L of block i (M = 128 head rows, N = 64 slots, K = D).
      auto issue_l = [&](int i) {
        const int st = i % L::kStages;
        const uint64_t dk = d_kv + ((static_cast<uint32_t>(st) * L::kKvStageBytes) >> 4);
        const uint32_t d_tm = tmem + L::kTmemL + static_cast<uint32_t>(i & 1) * L::kBI;
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(d_tm, d_q + ((c * L::kQChunkBytes + k * 32u) >> 4),
                   dk + ((c * L::kKvChunkBytes + k * 32u) >> 4), idesc_l, (c | k) != 0 ? 1u : 0u);
        mma_commit(bar(L::kBarLFull + (i & 1)));
      };
      // dq += G.K for block j (M = 128 head rows, N = D, K = 64 slots).
      auto issue_dq = [&](int j) {
        const int st = j % L::kStages;
        const uint64_t dk = d_kvmn + ((static_cast<uint32_t>(st) * L::kKvStageBytes) >> 4);
        const uint64_t dg =
            d_gate + ((static_cast<uint32_t>(j % L::kGateBufs) * L::kGateBytes) >> 4);
#pragma unroll
        for (int k = 0; k < L::kBI / 16; ++k)
          mma_ss(tmem + L::kTmemDq, dg + (k * 32u >> 4), dk + (k * 2048u >> 4), idesc_dq,
                 (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(L::kBarKvEmpty + st));
        mma_commit(bar(L::kBarGFree + j % L::kGateBufs));
      };
      // Event loop (non-blocking tests), oldest work first: dq of block n2
      // once its gate operand is written; L of block n1 once its key rows
      // have landed and its TMEM tile has been read (block n1 - 2).
      bool ok = mbar_wait(bar(L::kBarQFull), 0, ctl);
      int n1 = 0, n2 = 0;
      PollState ps = poll_start();
      uint32_t spins = 0;
      while (ok && n2 < nblk) {
        if (n2 < n1 &&
            mbar_probe(bar(L::kBarGFull + n2 % L::kGateBufs), (n2 / L::kGateBufs) & 1)) {
          tc_fence_after();
          issue_dq(n2);
          ++n2;
        } else if (n1 < nblk &&
                   mbar_probe(bar(L::kBarKvFull + n1 % L::kStages), (n1 / L::kStages) & 1) &&
                   (n1 < 2 || mbar_probe(bar(L::kBarLFree + (n1 & 1)), ((n1 - 2) >> 1) & 1))) {
          // The key tile was written by cp.async (generic proxy): order it
          // before the tensor core's (async proxy) reads.
          fence_proxy_async_smem();
          tc_fence_after();
          issue_l(n1);
          ++n1;
          if (static_cast<int>(blockIdx.x) == p.stall_cta) {  // test hook only
            ok = stall_until_limit(ctl);
            break;
          }
        } else {
          if ((++spins & 63u) == 0u && !poll_check(ctl, ps)) {
            ok = false;
            break;
          }
          continue;
        }
        ps.t0 = globaltimer_ns();  // progress: the limit counts from the last issue
      }
      mma_commit(bar(L::kBarDqDone));
      mma_commit(bar(L::kBarDrain));
      mbar_wait_drain(bar(L::kBarDrain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ gate
    // Thread = head row h: per block the row's 64 logits from TMEM, then
    // G[h,j] = g_j if L[h,j] > 0 else 0 (g_j is 0 for masked slots), bf16,
    // into the block's gate operand (128-byte rows, 128-byte swizzle).
    const int h = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t row128 = static_cast<uint32_t>(h) * 128u;
    bool ok = *abort_flag == 0;
    for (int i = 0; ok && i < nblk; ++i) {
      const int lb = i & 1;                // logit tile
      const int gb = i % L::kGateBufs;     // gate operand buffer
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarLFull + lb), (i >> 1) & 1, ctl));
      if (!ok) break;
      tc_fence_after();
      float x[64];
      const uint32_t t_l = tmem + lane_base + L::kTmemL + static_cast<uint32_t>(lb) * L::kBI;
      tmem_ld32x2(t_l, t_l + 32, *reinterpret_cast<float(*)[32]>(x),
                  *reinterpret_cast<float(*)[32]>(x + 32));
      tc_fence_before();
      mbar_arrive(bar(L::kBarLFree + lb));
      // The block's grad_scores (its key tile, and so the L tile, came after
      // them; this wait has completed and only orders the reads).
      const int st = i % L::kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarKvFull + st), (i / L::kStages) & 1, ctl));
      if (!ok) break;
      if (i >= L::kGateBufs) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(L::kBarGFree + gb), ((i / L::kGateBufs) - 1) & 1, ctl));
        if (!ok) break;
      }
      const float4* gq = reinterpret_cast<const float4*>(smem + L::kOffG + st * L::kBI * 4);
      const uint32_t gate = base + L::kOffGate + static_cast<uint32_t>(gb) * L::kGateBytes;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w4[4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float4 gv = gq[2 * c + k];
          const float* xs = x + 8 * c + 4 * k;
          w4[2 * k] = pack_bf16x2(xs[0] > 0.f ? gv.x : 0.f, xs[1] > 0.f ? gv.y : 0.f);
          w4[2 * k + 1] = pack_bf16x2(xs[2] > 0.f ? gv.z : 0.f, xs[3] > 0.f ? gv.w : 0.f);
        }
        st_shared_v4(gate + row128 + ((static_cast<uint32_t>(c) ^ static_cast<uint32_t>(h & 7)) << 4),
                     w4[0], w4[1], w4[2], w4[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::kBarGFull + gb));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarDqDone), 0, ctl));
    if (ok) {
      tc_fence_after();
      // dq = w[t,h] * accumulator, bf16, as 64-column tiles in the
      // 128-byte-swizzled layout of dq's tensor map (the key ring is free:
      // every MMA has completed); the TMA then writes whole rows.
      const float wh = h < p.H ? __ldg(p.w + row0 + h) : 0.f;
#pragma unroll 1
      for (int cc = 0; cc < L::kChunks; ++cc) {
        float v[2][32];
        if (nblk > 0) {
          tmem_ld32x2(tmem + lane_base + L::kTmemDq + cc * 64,
                      tmem + lane_base + L::kTmemDq + cc * 64 + 32, v[0], v[1]);
        } else {  // no valid slot: the gradient is 0
#pragma unroll
          for (int k = 0; k < 32; ++k) v[0][k] = v[1][k] = 0.f;
        }
        const uint32_t row = base + L::kOffKv + static_cast<uint32_t>(cc) * L::kQChunkBytes +
                             static_cast<uint32_t>(h) * 128u;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(v[u][2 * k] * wh, v[u][2 * k + 1] * wh);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t piece = static_cast<uint32_t>(4 * u + k);
            st_shared_v4(row + ((piece ^ (static_cast<uint32_t>(h) & 7u)) << 4), w[4 * k],
                         w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
          }
        }
      }
    }
    // Every gate thread arrives (also after a failed wait, so that the
    // storing thread never waits in vain); one thread ships the tiles.
    fence_proxy_async_smem();
    mbar_arrive(bar(L::kBarStaged));
    if (threadIdx.x == 0) {
      if (mbar_wait(bar(L::kBarStaged), 0, ctl) && *abort_flag == 0) {
        for (int cc = 0; cc < L::kChunks; ++cc)
          tma_store_2d(&tm_dq, base + L::kOffKv + static_cast<uint32_t>(cc) * L::kQChunkBytes,
                       cc * 64, static_cast<int>(row0));
        bulk_commit_group();
        bulk_wait_group0();  // complete before the CTA (and its shared memory) goes away
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Key-tile stages, gate buffers and CTAs per SM of the kernel (measured on
// the H=64 D=128 topk=2048 S=8192 workload: 2/2/2 1.292 ms, 3/1/2 1.049 ms,
// 4/2/1 1.685 ms, 6/2/1 1.668 ms; two resident CTAs hide each other's
// per-token prologue and epilogue, and the third stage outweighs the second
// gate buffer).
constexpr int kIdxStages = 3, kIdxGateBufs = 1, kIdxCtas = 2;

template <int D>
static cudaError_t launch_indexer_impl(const CUtensorMap& tm_q, const CUtensorMap& tm_dq,
                                       const IdxParams& p, int ctas, cudaStream_t stream) {
  using L = IdxLayout<D, kIdxStages, kIdxGateBufs, kIdxCtas>;
  auto kern = smqa_indexer_bwd_kernel<D, kIdxStages, kIdxGateBufs, kIdxCtas>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<ctas, L::kThreads, L::kSmemBytes, stream>>>(tm_q, tm_dq, p);
  return cudaGetLastError();
}

cudaError_t launch_indexer_bwd(const CUtensorMap& tm_q, const CUtensorMap& tm_dq,
                               const IdxParams& p, cudaStream_t stream) {
  const int ctas = p.B * p.S;
  if (p.D == 128) return launch_indexer_impl<128>(tm_q, tm_dq, p, ctas, stream);
  if (p.D == 64) return launch_indexer_impl<64>(tm_q, tm_dq, p, ctas, stream);
  return cudaErrorInvalidValue;
}

}  // namespace smqa
