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
// Design.  The token's H heads are the M = 128 rows of every MMA (heads
// beyond H are zero rows), so the heads sharing one gathered kv block form a
// real GEMM for the tcgen05 tensor core.
//   * D = 512: two independent CTAs per token.  CTA r owns O columns
//     [256r, 256r+256): its O accumulator (128 x 256 fp32) is half of TMEM.
//     Both CTAs compute the FULL score tile S = Q.K^T over all 512 columns,
//     so no partial sums cross between SMs (the CTA-to-CTA network moves
//     only ~8 B/clk per SM, far too little for a per-block exchange).  Q's
//     own half is an smem operand; the other half sits in TMEM as the A
//     operand of `tcgen05.mma ... [a_tmem]` (TMEM: O 256 + two 64-column
//     score tiles + Q 128 = 512 columns).  Both CTAs issue the K steps in the
//     same order, so their scores, softmax and LSE are bit-identical.
//   * D = 64: one CTA per token; Q is an smem operand.
//   * Warp roles: warps 8-11 gather full kv rows with 16-byte cp.async
//     (coalesced 512-byte row pieces, written into the 128-byte-swizzled
//     K-major tile; completion signalled per block by cp.async mbarrier
//     arrivals); warp 12 owns TMEM and issues the MMAs from one thread;
//     warps 0-7 (two warpgroups; thread = head row = TMEM lane, 32 score
//     columns each) run the masked online softmax in the exp2 domain, rescale
//     O lazily (only when the running max grows by more than 2^8), write P as
//     bf16 for the P.V MMA and finish with the sink and the log2 LSE.
//   * Masked slots load a real (finite) row and get a -inf score, so their
//     probability is exactly 0.
#include <cuda_runtime.h>

#include "smqa_internal.h"
#include "smqa_ptx.cuh"

namespace smqa {

template <int D, int NSPLIT>
struct FwdLayout {
  static constexpr int kDC = D / NSPLIT;      // O columns (and own Q columns) per CTA
  static constexpr int kHPad = 128;           // MMA M: heads padded to 128
  static constexpr int kBI = 64;              // slots per block (MMA N of the scores)
  static constexpr int kChunks = D / 64;      // 64-column (128-byte) swizzle chunks per row
  static constexpr int kOwnChunks = kDC / 64;
  static constexpr int kOthChunks = kChunks - kOwnChunks;
  static constexpr int kStages = D >= 512 ? 2 : 4;   // slots of each ring
  static constexpr uint32_t kQChunkBytes = kHPad * 128;
  static constexpr uint32_t kQBytes = kOwnChunks * kQChunkBytes;
  static constexpr uint32_t kKvChunkBytes = kBI * 128;   // kBI rows x 128 B
  static constexpr uint32_t kOwnStageBytes = kOwnChunks * kKvChunkBytes;
  static constexpr uint32_t kOthStageBytes = kOthChunks * kKvChunkBytes;
  static constexpr uint32_t kPBytes = kHPad * kBI * 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffOwn = kOffQ + kQBytes;
  static constexpr uint32_t kOffOth = kOffOwn + kStages * kOwnStageBytes;
  static constexpr uint32_t kOffP = kOffOth + kStages * kOthStageBytes;
  static constexpr uint32_t kOffCtrl = kOffP + kPBytes;
  static constexpr int kBarOwnFull = 0;
  static constexpr int kBarOwnEmpty = kBarOwnFull + kStages;
  static constexpr int kBarOthFull = kBarOwnEmpty + kStages;
  static constexpr int kBarOthEmpty = kBarOthFull + kStages;
  static constexpr int kBarSFull = kBarOthEmpty + kStages;  // phase i: S of block i ready
  static constexpr int kBarSFree = kBarSFull + 1;           // phase i: S of block i read
  static constexpr int kBarPFull = kBarSFree + 1;           // phase i: P of block i written
  static constexpr int kBarODone = kBarPFull + 1;           // phase i: P.V of block i done
  static constexpr int kBarQFull = kBarODone + 1;
  static constexpr int kBarQtFull = kBarQFull + 1;   // other half of Q stored in TMEM
  static constexpr int kBarDrain = kBarQtFull + 1;
  static constexpr int kBarXmax = kBarDrain + 1;     // [2], by block parity
  static constexpr int kBarLsum = kBarXmax + 2;
  static constexpr int kNumBars = kBarLsum + 1;
  static constexpr uint32_t kOffXmax = kOffCtrl + 8 * kNumBars;    // float [2][2][128]
  static constexpr uint32_t kOffLsum = kOffXmax + 2 * 2 * 128 * 4; // float [2][128]
  static constexpr uint32_t kOffTmemHolder = kOffLsum + 2 * 128 * 4;
  static constexpr uint32_t kOffAbort = kOffTmemHolder + 4;
  static constexpr uint32_t kOffWarpLast = kOffAbort + 4;  // int [16]
  static constexpr uint32_t kCtrlBytes = 4096;
  static_assert(kOffWarpLast + 64 - kOffCtrl <= kCtrlBytes, "control block overflow");
  static constexpr uint32_t kSmemBytes = kOffCtrl + kCtrlBytes + 1024;  // +1024: realignment
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM: O, the other half of Q (bf16 pairs), then the score tile as two
  // partial sums: chain A over the own column half, chain B over the other.
  static constexpr uint32_t kTmemO = 0;
  static constexpr uint32_t kTmemQt = kDC;
  static constexpr uint32_t kTmemSA = kDC + (D - kDC) / 2;
  static constexpr uint32_t kTmemSB = kTmemSA + kBI;
  static constexpr uint32_t kTmemUsed = kTmemSA + (kOthChunks > 0 ? 2 : 1) * kBI;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  // warps 0-7: softmax; 8-9: gather own column half; 10-11: gather the other
  // half; 12: TMEM owner + MMA issuer
  static constexpr int kSoftmaxThreads = 256;
  static constexpr int kOwnWarp0 = 8;
  static constexpr int kOthWarp0 = 10;
  static constexpr int kMmaWarp = 12;
  static constexpr int kThreads = 416;
};

// Gathers one column half of a block's kv rows into a 128-byte-swizzled
// K-major tile of `nchunks` 64-column chunks.  Warp w (0 or 1) of the pair
// issues instructions w, w+2, ...; instruction k moves 16-byte pieces
// q = 32k + lane, piece q being column piece q % (8 nchunks) of slot row
// q / (8 nchunks).
template <int NCHUNKS, int D>
__device__ __forceinline__ void gather_half(uint32_t stage, const __nv_bfloat16* kv, int col0,
                                            int row0, int row1, int w, int lane) {
  constexpr int kRcpr = NCHUNKS * 8;
  constexpr int kInstr = 64 * kRcpr / 32;
#pragma unroll 4
  for (int k = w; k < kInstr; k += 2) {
    const int q = 32 * k + lane;
    const int r = q / kRcpr;
    const int cc = q % kRcpr;
    const int a = __shfl_sync(0xffffffffu, row0, r & 31);
    const int c2 = __shfl_sync(0xffffffffu, row1, r & 31);
    const int rr = r < 32 ? a : c2;
    cp_async_16(stage + static_cast<uint32_t>(cc / 8) * (64u * 128u) +
                    static_cast<uint32_t>(r) * 128u +
                    ((static_cast<uint32_t>(cc % 8) ^ (static_cast<uint32_t>(r) & 7u)) << 4),
                kv + static_cast<size_t>(rr) * D + col0 + cc * 8);
  }
}

template <int D, int NSPLIT>
__global__ void __launch_bounds__(416, 1)
    smqa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const FwdParams p) {
  using L = FwdLayout<D, NSPLIT>;
  constexpr int DC = L::kDC;
  extern __shared__ uint8_t smem_raw[];
  uint32_t base = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (base & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  base += pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x / NSPLIT;
  const int rank = NSPLIT == 2 ? static_cast<int>(blockIdx.x % NSPLIT) : 0;
  const int b = t / p.S;
  const int32_t* idx_row = p.idx + static_cast<size_t>(t) * p.topk;
  auto bar = [&](int i) -> uint32_t { return base + L::kOffCtrl + 8u * static_cast<uint32_t>(i); };
  volatile float* xmax = reinterpret_cast<volatile float*>(smem + L::kOffXmax);
  volatile float* lsum = reinterpret_cast<volatile float*>(smem + L::kOffLsum);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + L::kOffTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  const WaitCtl ctl{abort_flag, p.status, p.limit_ns};

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarOwnFull + s), 64);  // one cp.async arrival per gather thread
      mbar_init(bar(L::kBarOwnEmpty + s), 1);
      mbar_init(bar(L::kBarOthFull + s), 64);
      mbar_init(bar(L::kBarOthEmpty + s), 1);
    }
    mbar_init(bar(L::kBarSFull), 1);
    mbar_init(bar(L::kBarSFree), L::kSoftmaxThreads);
    mbar_init(bar(L::kBarPFull), L::kSoftmaxThreads);
    mbar_init(bar(L::kBarODone), 1);
    mbar_init(bar(L::kBarQFull), 1);
    mbar_init(bar(L::kBarQtFull), L::kSoftmaxThreads);
    mbar_init(bar(L::kBarDrain), 1);
    mbar_init(bar(L::kBarXmax), L::kSoftmaxThreads);
    mbar_init(bar(L::kBarXmax + 1), L::kSoftmaxThreads);
    mbar_init(bar(L::kBarLsum), L::kSoftmaxThreads);
    *abort_flag = *reinterpret_cast<volatile int*>(p.status) != 0 ? 1 : 0;
    fence_mbar_init();
    // This CTA's column half of Q, issued before anything else waits on
    // memory (the index scan below and the other half's loads overlap it).
    mbar_arrive_expect_tx(bar(L::kBarQFull), static_cast<uint32_t>(p.H) * 128u * L::kOwnChunks);
    for (int c = 0; c < L::kOwnChunks; ++c)
      tma_load_2d(base + L::kOffQ + c * L::kQChunkBytes, &tm_q, rank * DC + c * 64, t * p.H,
                  bar(L::kBarQFull));
  }
  if (warp == L::kMmaWarp) tmem_alloc(base + L::kOffTmemHolder, L::kTmemCols);
  // Softmax threads (h, g) start loading their part of the other column half
  // of Q (stored into TMEM once it is allocated).
  uint4 qt_pre[16];
  if (NSPLIT == 2 && warp < L::kOwnWarp0) {
    const int hq = threadIdx.x & 127;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + (static_cast<size_t>(t) * p.H + (hq < p.H ? hq : 0)) * D + (1 - rank) * DC +
        (warp >> 2) * 128);
#pragma unroll
    for (int k = 0; k < 16; ++k) qt_pre[k] = hq < p.H ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
  }
  // Heads beyond H are zero rows of the smem A operand (the TMA box covers H rows).
  if (threadIdx.x < L::kHPad && static_cast<int>(threadIdx.x) >= p.H) {
    const uint32_t h = threadIdx.x;
#pragma unroll
    for (int c = 0; c < L::kOwnChunks; ++c)
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
  // Blocks up to the last one holding a valid slot (0: no valid slot).
  const int nblk = live_blocks(warp_last, L::kBI);

  if (warp >= L::kOwnWarp0 && warp < L::kMmaWarp) {
    // ------------------------------------------------------------ gather
    // Warps 8-9 fill the own-column-half ring (needed until P.V), warps
    // 10-11 the other-half ring (needed only by the scores), so the other
    // half of block i+2 can land as soon as the scores of block i are done.
    const bool own = warp < L::kOthWarp0;
    const int w = (warp - L::kOwnWarp0) & 1;
    if (own || L::kOthChunks > 0) {
      auto load_idx = [&](int blk, int half) -> int {
        const int j = blk * L::kBI + 32 * half + lane;
        return j < p.topk ? __ldg(idx_row + j) : -1;
      };
      const int full0 = own ? L::kBarOwnFull : L::kBarOthFull;
      const int empty0 = own ? L::kBarOwnEmpty : L::kBarOthEmpty;
      const uint32_t ring = base + (own ? L::kOffOwn : L::kOffOth);
      const uint32_t stage_bytes = own ? L::kOwnStageBytes : L::kOthStageBytes;
      const int col0 = (own ? rank : 1 - rank) * DC;
      int n0 = load_idx(0, 0), n1 = load_idx(0, 1);
      for (int i = 0; i < nblk; ++i) {
        const int s = i % L::kStages;
        const int r0 = n0, r1 = n1;
        if (i + 1 < nblk) {
          n0 = load_idx(i + 1, 0);
          n1 = load_idx(i + 1, 1);
        }
        const int row0 = b * p.S_kv + (static_cast<unsigned>(r0) < static_cast<unsigned>(p.S_kv) ? r0 : 0);
        const int row1 = b * p.S_kv + (static_cast<unsigned>(r1) < static_cast<unsigned>(p.S_kv) ? r1 : 0);
        if (i >= L::kStages) {
          const bool ok = mbar_wait(bar(empty0 + s), ((i / L::kStages) - 1) & 1, ctl);
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        const uint32_t stage = ring + static_cast<uint32_t>(s) * stage_bytes;
        if (own)
          gather_half<L::kOwnChunks, D>(stage, p.kv, col0, row0, row1, w, lane);
        else
          gather_half<(L::kOthChunks > 0 ? L::kOthChunks : 1), D>(stage, p.kv, col0, row0, row1,
                                                                  w, lane);
        cp_async_arrive_noinc(bar(full0 + s));
      }
      // Let every copy this warp started land before the CTA can exit.
      cp_async_wait_all();
      if (own && w == 0 && lane == 0) mbar_wait_drain(bar(L::kBarQFull), 0);
    }
  } else if (warp == L::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, L::kBI, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, DC, false, true);
      // Descriptors are built once; per MMA only the start-address field
      // (bits 0-13, in 16-byte units) moves, by compile-time offsets.
      const uint64_t d_q = smem_desc(base + L::kOffQ, 16u, 1024u, kSwizzle128B);
      const uint64_t d_p = smem_desc(base + L::kOffP, 16u, 1024u, kSwizzle128B);
      const uint64_t d_own = smem_desc(base + L::kOffOwn, 16u, 1024u, kSwizzle128B);
      const uint64_t d_oth = smem_desc(base + L::kOffOth, 16u, 1024u, kSwizzle128B);
      const uint64_t d_v = smem_desc(base + L::kOffOwn, L::kKvChunkBytes, 1024u, kSwizzle128B);
      // Chain A: own column half, Q from smem.  Chain B: the other half, Q
      // from TMEM.  Chunk j of a half is chunk j of that half on both CTAs,
      // so each chain sums the same products in the same order everywhere.
      auto issue_a = [&](int i) {
        const uint64_t dk = d_own + ((static_cast<uint32_t>(i % L::kStages) * L::kOwnStageBytes) >> 4);
#pragma unroll
        for (int c = 0; c < L::kOwnChunks; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + L::kTmemSA, d_q + ((c * L::kQChunkBytes + k * 32u) >> 4),
                   dk + ((c * L::kKvChunkBytes + k * 32u) >> 4), idesc_s, (c | k) ? 1u : 0u);
      };
      auto issue_b = [&](int i) {
        const uint64_t dk = d_oth + ((static_cast<uint32_t>(i % L::kStages) * L::kOthStageBytes) >> 4);
#pragma unroll
        for (int c = 0; c < L::kOthChunks; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tmem + L::kTmemSB, tmem + L::kTmemQt + (c * 4 + k) * 8,
                   dk + ((c * L::kKvChunkBytes + k * 32u) >> 4), idesc_s, (c | k) ? 1u : 0u);
      };
      // O += P.V for block j; V = the own column half, read MN-major.
      auto issue_pv = [&](int j) {
        const int sj = j % L::kStages;
        const uint64_t dv = d_v + ((static_cast<uint32_t>(sj) * L::kOwnStageBytes) >> 4);
#pragma unroll
        for (int k = 0; k < L::kBI / 16; ++k)
          mma_ss(tmem + L::kTmemO, d_p + (k * 32u >> 4), dv + (k * 2048u >> 4), idesc_o,
                 (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(L::kBarOwnEmpty + sj));
        mma_commit(bar(L::kBarODone));
      };
      bool ok = mbar_wait(bar(L::kBarQFull), 0, ctl);
      if (ok && NSPLIT == 2) ok = mbar_wait(bar(L::kBarQtFull), 0, ctl);
      // Event loop over three kinds of work, oldest first (polled with
      // non-blocking tests, so that waiting on one never delays another): P.V of block npv
      // once its P is written; chain A (+ completion of S) of block na once
      // the own half has landed; chain B of block nb once the other half has
      // landed.  Both score chains of a block need the previous block's
      // scores to have been read (one score tile in TMEM), and a block's
      // scores may complete at most one block ahead of P.V.
      constexpr bool kHasB = L::kOthChunks > 0;
      int nb = 0, na = 0, npv = 0;
      PollState ps = poll_start();
      uint32_t spins = 0;
      while (ok && npv < nblk) {
        if (npv < na && mbar_probe(bar(L::kBarPFull), npv & 1)) {
          tc_fence_after();
          issue_pv(npv);
          ++npv;
        } else if (na < nblk && (!kHasB || nb > na) && na <= npv + 1 &&
                   (na == 0 || mbar_probe(bar(L::kBarSFree), (na - 1) & 1)) &&
                   mbar_probe(bar(L::kBarOwnFull + na % L::kStages), (na / L::kStages) & 1)) {
          // The kv tile was written by cp.async (generic proxy): order it
          // before the tensor core's (async proxy) reads.
          fence_proxy_async_smem();
          tc_fence_after();
          issue_a(na);
          mma_commit(bar(L::kBarSFull));
          ++na;
        } else if (kHasB && nb < nblk && nb <= na &&
                   (nb == 0 || mbar_probe(bar(L::kBarSFree), (nb - 1) & 1)) &&
                   mbar_probe(bar(L::kBarOthFull + nb % L::kStages), (nb / L::kStages) & 1)) {
          fence_proxy_async_smem();
          tc_fence_after();
          issue_b(nb);
          // Only chain B reads the other column half: free its stage.
          mma_commit(bar(L::kBarOthEmpty + nb % L::kStages));
          ++nb;
        } else {
          if ((++spins & 63u) == 0u && !poll_check(ctl, ps)) {
            ok = false;
            break;
          }
          continue;
        }
        // Progress: the limit counts from the last issued work.
        ps.t0 = globaltimer_ns();
      }
      // No MMA may still be running when TMEM is released.
      mma_commit(bar(L::kBarDrain));
      mbar_wait_drain(bar(L::kBarDrain), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Thread (h, g): head row h (TMEM lane), score columns [32g, 32g+32) of
    // every block, O columns [DC/2 g, DC/2 (g+1)) for rescaling and output.
    const int g = warp >> 2;
    const int h = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    // exp2 argument: score * (c log2 e), or (score * c) * log2 e with the
    // reference-rounding flag (x * s1 * 1 is exact when the flag is off).
    const float s1 = p.ref_round ? p.scale : p.scale_log2;
    const float s2 = p.ref_round ? 1.4426950408889634f : 1.f;
    constexpr int kOHalf = DC / 2;
    if (NSPLIT == 2) {
      // The other column half of this head's q row -> TMEM (A operand of
      // score chain B), as bf16 pairs: this thread stores words [64g, 64g+64)
      // (loaded into qt_pre during the prologue).
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 w = qt_pre[half * 8 + k];
          v[4 * k] = __uint_as_float(w.x);
          v[4 * k + 1] = __uint_as_float(w.y);
          v[4 * k + 2] = __uint_as_float(w.z);
          v[4 * k + 3] = __uint_as_float(w.w);
        }
        tmem_st32(tmem + lane_base + L::kTmemQt + 64 * g + 32 * half, v);
      }
      tc_fence_before();
      mbar_arrive(bar(L::kBarQtFull));
    }
    // Slot validity: lane j of each warp holds slot 32g + j of the block;
    // the warp's ballot is this thread's 32-bit column mask (read one block
    // ahead from L2).
    auto slot_ok = [&](int blk) -> bool {
      const int j = blk * L::kBI + 32 * g + lane;
      if (j >= p.topk) return false;
      const int r = __ldg(idx_row + j);
      return static_cast<unsigned>(r) < static_cast<unsigned>(p.S_kv);
    };
    bool v_next = slot_ok(0);
    float m_run = -INFINITY;
    float l_part = 0.f;
    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
      const int bb = i & 1;
      const uint32_t msk = __ballot_sync(0xffffffffu, v_next);
      if (i + 1 < nblk) v_next = slot_ok(i + 1);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull), i & 1, ctl));
      if (!ok) break;
      tc_fence_after();
      float x[32];
      if constexpr (L::kOthChunks > 0) {
        // Both partial tiles in one TMEM round trip.
        float x2[32];
        tmem_ld32x2(tmem + lane_base + L::kTmemSA + 32 * g, tmem + lane_base + L::kTmemSB + 32 * g,
                    x, x2);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] += x2[j];
      } else {
        tmem_ld32(tmem + lane_base + L::kTmemSA + 32 * g, x);
      }
      tc_fence_before();
      mbar_arrive(bar(L::kBarSFree));
      float mq[8];
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = ((msk >> j) & 1u) ? (x[j] * s1) * s2 : -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        mq[j] = fmaxf(fmaxf(x[4 * j], x[4 * j + 1]), fmaxf(x[4 * j + 2], x[4 * j + 3]));
      const float mloc = fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])),
                               fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7])));
      // Combine with the other half of the row (the thread of the other
      // warpgroup with the same h); buffers alternate by block parity.
      xmax[(bb * 2 + g) * 128 + h] = mloc;
      mbar_arrive(bar(L::kBarXmax + bb));
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarXmax + bb), (i >> 1) & 1, ctl));
      if (!ok) break;
      const float mx = fmaxf(mloc, xmax[(bb * 2 + (g ^ 1)) * 128 + h]);
      const float m_new = fmaxf(m_run, mx);
      const bool bump = (m_run == -INFINITY) ? (m_new != -INFINITY) : (m_new > m_run + 8.f);
      float alpha = 1.f;
      if (bump) {
        alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
        l_part *= alpha;
        m_run = m_new;
      }
      // The P buffer and the O accumulator are free once P.V of block i-1
      // has completed.
      if (i >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarODone), (i - 1) & 1, ctl));
        if (!ok) break;
        tc_fence_after();
      }
      // O was accumulated against the old max: rescale this thread's half of
      // the row (whole warp, since TMEM accesses are warp-collective; rows
      // without a bump use 1).
      const bool need_rescale = bump && alpha != 0.f && i > 0;
      if (__any_sync(0xffffffffu, need_rescale)) {
        const float a = need_rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < kOHalf / 32; ++c) {
          float v[32];
          tmem_ld32(tmem + lane_base + L::kTmemO + g * kOHalf + c * 32, v);
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] *= a;
          tmem_st32(tmem + lane_base + L::kTmemO + g * kOHalf + c * 32, v);
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t pk[16];
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        const float p0 = fast_exp2(x[2 * w] - m_use);
        const float p1 = fast_exp2(x[2 * w + 1] - m_use);
        pk[w] = pack_bf16x2(p0, p1);
        rs[w & 3] += p0 + p1;  // fp32 probabilities: the LSE must not carry bf16 rounding
      }
      l_part += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      const uint32_t p_row = base + L::kOffP + static_cast<uint32_t>(h) * 128u;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared_v4(p_row + (((4 * g + c) ^ (h & 7)) << 4), pk[4 * c], pk[4 * c + 1],
                     pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(L::kBarPFull));
    }
    if (ok && nblk > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarODone), (nblk - 1) & 1, ctl));
    // Row sums: the two halves of each row meet here.
    lsum[g * 128 + h] = l_part;
    mbar_arrive(bar(L::kBarLsum));
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarLsum), 0, ctl));
    if (ok) {
      const float l_run = lsum[h] + lsum[128 + h];
      tc_fence_after();
      const float sink2 = h < p.H ? __ldg(p.sink + h) * 1.4426950408889634f : 0.f;
      const float m_fin = fmaxf(m_run, sink2);
      const float so = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_fin);
      const float Z = l_run * so + fast_exp2(sink2 - m_fin);
      const float inv = so / Z;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(t) * p.H + h) * D +
                            static_cast<size_t>(rank) * DC + g * kOHalf;
#pragma unroll 1
      for (int c = 0; c < kOHalf / 32; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_base + L::kTmemO + g * kOHalf + c * 32, v);
        if (nblk == 0) {  // no valid slot: O was never written, the output is 0
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.f;
        }
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
      if (rank == 0 && g == 0 && h < p.H)
        p.lse[static_cast<size_t>(t) * p.H + h] = m_fin + log2f(Z);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, int NSPLIT>
static cudaError_t launch_fwd_impl(const CUtensorMap& tm_q, const FwdParams& p, int tokens,
                                   cudaStream_t stream) {
  using L = FwdLayout<D, NSPLIT>;
  auto kern = smqa_fwd_kernel<D, NSPLIT>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<static_cast<unsigned>(tokens) * NSPLIT, L::kThreads, L::kSmemBytes, stream>>>(tm_q, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const CUtensorMap& tm_q, const FwdParams& p, int tokens,
                       cudaStream_t stream) {
  if (p.D == 512) return launch_fwd_impl<512, 2>(tm_q, p, tokens, stream);
  if (p.D == 64) return launch_fwd_impl<64, 1>(tm_q, p, tokens, stream);
  return cudaErrorInvalidValue;
}

}  // namespace smqa
