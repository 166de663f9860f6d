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
// real GEMM for the tcgen05 tensor core.  Slots go in blocks of 64.
//   * D = 512: a cluster of two CTAs works on each token.  CTA r owns the
//     column half [256r, 256r+256) of Q, of every gathered kv row and of O
//     (its O accumulator, 128 x 256 fp32, is half of TMEM).  Per block it computes
//     the partial scores over its half, S_r = Q_r.K_r^T, and the pair trades
//     them through an L2-resident exchange slot: each CTA scales its partial
//     into the exp2 domain and sends it in block floating point (per head
//     and block one power-of-two scale and 64 int16 mantissas, so the
//     rounding error is about 2^-15 of the head's largest partial in the
//     block: 16.5 KB per block instead of 32 KB of fp32, where fp16 would put
//     up to ~2^-8 of a score's magnitude into a single-slot LSE).  Both CTAs
//     form S = own + peer's from the same two rounded values, so the pair's
//     probabilities and LSE are bit-identical.  Each CTA then runs the same
//     online softmax and accumulates O_r += P.V_r.  The exchange slot (two
//     receivers x six block buffers) is claimed from a pool by the pair's
//     rank 0 and released at exit.
//   * Exchange flow control without a consumed-signal: a CTA frees score
//     tile i % 3 only after its softmax has read the full scores of block i
//     (formed after the peer's partial of block i was read), and it computes
//     (and sends) block i + 3 only into a freed tile, so the arrival of the
//     peer's block j + 3 proves that the peer has read block j; block j + 6
//     goes into the buffer of block j only after its own CTA has received
//     block j + 3 (six buffers rather than the four this needs at least, so
//     that a sender waits for the peer's block i - 3 rather than i - 1).
//   * Persistent CTAs (pairs): each takes tokens one after another from a
//     counter (rank 0 hands each to its peer), so the next token's gathers,
//     scores, exchange and softmax run while the current one's last P.V and
//     O read-out finish; O goes from TMEM straight to global memory with
//     32-byte stores.
//   * D = 64: single persistent CTAs, no exchange; CTA c takes tokens c,
//     c + grid, ... (static order, no counter).
//   * Warp roles (D = 512; for D = 64 the combiner and sender warps are
//     absent): warps 8-10 gather this CTA's half of the kv rows with
//     16-byte cp.async (coalesced 512-byte row pieces written into the
//     128-byte-swizzled K-major tile; completion signalled per block by
//     cp.async mbarrier arrivals) into a five-stage ring, and publish each
//     block's valid-slot mask; warp 11 owns TMEM and issues the MMAs from
//     one thread (partial scores into a ring of three 64-column TMEM tiles;
//     P.V with P, bf16, from a two-buffer ring in TMEM as the A operand);
//     warps 12-15 round each partial tile, store it to the peer's buffer
//     and then write the rounded values back into the tile (the stores'
//     way to L2 overlaps the write-back); warps 4-7 write the full scores
//     (own + peer's) back into the tile; warps 0-3 (thread = head row =
//     TMEM lane) run the masked online softmax in the exp2 domain (the mask
//     only on blocks holding an invalid slot), rescale O lazily (only when
//     the running max grows by more than 2^8), write P as bf16 into TMEM
//     for the P.V MMA and finish with the sink and the log2 LSE.
//   * Per-element arithmetic of these roles uses the packed two-lane fp32
//     instructions (add/mul/fma.rn.f32x2) and three-input maxima, which
//     halve their instruction counts; the roles' chain of latencies, not
//     the tensor core, bounds a block's time.
//   * Masked slots load a real (finite) row and get a -inf score, so their
//     probability is exactly 0; blocks past a token's last valid slot are
//     skipped.
#include <cuda_runtime.h>

#include "smqa_internal.h"
#include "smqa_ptx.cuh"

namespace smqa {

template <int D, int NSPLIT>
struct FwdLayout {
  static constexpr int kDC = D / NSPLIT;      // columns of Q, kv and O per CTA
  static constexpr int kHPad = 128;           // MMA M: heads padded to 128
  static constexpr int kBI = 64;              // slots per block (MMA N of the scores)
  static constexpr int kChunks = kDC / 64;    // 64-column (128-byte) swizzle chunks per row
  static constexpr int kStages = 5;           // kv ring (five 32 KB stages fill shared memory)
  static constexpr int kSBufs = 3;            // score tiles in TMEM
  static constexpr int kXBufs = kSBufs + 3;   // exchange buffers per receiver
  static constexpr uint32_t kQChunkBytes = kHPad * 128;
  static constexpr uint32_t kQBytes = kChunks * kQChunkBytes;
  static constexpr uint32_t kKvChunkBytes = kBI * 128;   // kBI rows x 128 B
  static constexpr uint32_t kStageBytes = kChunks * kKvChunkBytes;
  static constexpr int kTokRing = 4;          // tokens published ahead
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffKv = kOffQ + kQBytes;
  // Exchange buffer of one receiver and block: each head's 64 partial scores
  // as int16 with one power-of-two scale (block floating point), in 8 pieces
  // of 16 bytes per head, piece-major (a warp's 32 heads are 512 contiguous
  // bytes), then the 128 heads' dequantization factors (fp32).
  static constexpr int kPieces = 8;
  static constexpr uint32_t kXchgScaleOff = kPieces * 16u * kHPad;
  static constexpr uint32_t kXchgBytes = kXchgScaleOff + 4u * kHPad;
  static constexpr uint32_t kOffCtrl = kOffKv + kStages * kStageBytes;
  static constexpr int kBarKvFull = 0;                       // [kStages]
  static constexpr int kBarKvEmpty = kBarKvFull + kStages;   // [kStages]
  static constexpr int kBarSFull = kBarKvEmpty + kStages;    // [kSBufs] partial scores ready
  static constexpr int kBarSRead = kBarSFull + kSBufs;       // [kSBufs] ... read by the sender
  static constexpr int kBarSSum = kBarSRead + kSBufs;        // [kSBufs] full scores in the tile
  static constexpr int kBarSFree = kBarSSum + kSBufs;        // [kSBufs] tile read by the softmax
  static constexpr int kBarRecvFull = kBarSFree + kSBufs;    // [kXBufs] peer's partial arrived
  static constexpr int kBarPFull = kBarRecvFull + kXBufs;    // [2] P of block i in buffer i % 2
  static constexpr int kBarODone = kBarPFull + 2;            // [2] P.V of block i done
  static constexpr int kBarQFull = kBarODone + 2;            // one phase per token with blocks
  static constexpr int kBarQFree = kBarQFull + 1;            // its scores MMAs are done with Q
  static constexpr int kBarOFree = kBarQFree + 1;            // its O has been read out
  static constexpr int kBarTokFull = kBarOFree + 1;          // [kTokRing] token published
  static constexpr int kBarTokEmpty = kBarTokFull + kTokRing;  // [kTokRing] ... and read
  // The pair's token sequence: rank 0 takes each token from the counter and
  // hands it to both CTAs (IdFull); rank 1 frees an entry again (IdEmpty, on
  // rank 0) once its readers are done with it.
  static constexpr int kBarIdFull = kBarTokEmpty + kTokRing;   // [kTokRing]
  static constexpr int kBarIdEmpty = kBarIdFull + kTokRing;    // [kTokRing]
  static constexpr int kBarDrain = kBarIdEmpty + kTokRing;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr uint32_t kOffTmemHolder = kOffCtrl + 8 * kNumBars;
  static constexpr uint32_t kOffAbort = kOffTmemHolder + 4;
  static constexpr uint32_t kOffSlot = kOffAbort + 4;
  static constexpr uint32_t kOffMask = kOffSlot + 4;  // uint32 [kStages][2]
  static constexpr uint32_t kOffTokLast = kOffMask + 8 * kStages;  // int [kTokRing][kGatherWarps]
  static constexpr uint32_t kOffTokId = kOffTokLast + 4 * 3 * kTokRing;  // int [kTokRing], handed over
  static constexpr uint32_t kOffTokT = kOffTokId + 4 * kTokRing;         // int [kTokRing], published
  static constexpr uint32_t kCtrlBytes = 640;
  static_assert(kOffTokT + 4 * kTokRing - kOffCtrl <= kCtrlBytes, "control block overflow");
  static constexpr uint32_t kSmemBytes = kOffCtrl + kCtrlBytes + 1024;  // +1024: realignment
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // TMEM: O, the ring of score tiles, then two P buffers (bf16 pairs, 32
  // columns each).
  static constexpr uint32_t kTmemO = 0;
  static constexpr uint32_t kTmemS = kDC;  // + (block % kSBufs) * kBI
  static constexpr uint32_t kTmemP = kTmemS + kSBufs * kBI;  // + (block % 2) * kBI / 2
  static constexpr uint32_t kTmemUsed = kTmemP + kBI;
  static constexpr uint32_t kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  // warps 0-3: softmax; 4-7 (D split across the pair only): add the peer's
  // partial scores; then three gather warps, the TMEM owner + MMA issuer and
  // (D split only) four warps that send this CTA's partial scores.  (Three
  // gather warps, since the copies a warp keeps in flight bound its gather
  // rate.)
  static constexpr int kSoftmaxThreads = 128;
  static constexpr int kCombWarp0 = 4;
  static constexpr int kGatherWarp0 = kCombWarp0 + (NSPLIT == 2 ? 4 : 0);
  static constexpr int kGatherWarps = 3;
  static constexpr int kMmaWarp = kGatherWarp0 + kGatherWarps;
  static constexpr int kSendWarp0 = kMmaWarp + 1;
  static constexpr int kThreads = (kSendWarp0 + (NSPLIT == 2 ? 4 : 0)) * 32;
  // Readers of a published token: the MMA thread, the softmax warps and (D
  // split only) the combiner and sender warps (one arrival each).
  static constexpr int kTokReaders = 1 + 4 + (NSPLIT == 2 ? 8 : 0);
  static_assert(kGatherWarps == 3, "token ring entries hold three gather warps' scans");
  static_assert(2 * kXBufs * kXchgBytes == kFwdSlotBytes, "exchange slot size");
};

// Gathers this CTA's column half of a block's kv rows into a
// 128-byte-swizzled K-major tile of NCHUNKS 64-column chunks.  Warp w of the
// NW gather warps issues instructions w, w+NW, ...; instruction k moves
// 16-byte pieces q = 32k + lane, piece q being column piece q % (8 NCHUNKS)
// of slot row q / (8 NCHUNKS).
template <int NCHUNKS, int D, int NW>
__device__ __forceinline__ void gather_block(uint32_t stage, const __nv_bfloat16* kv, int col0,
                                             int row0, int row1, int w, int lane) {
  constexpr int kRcpr = NCHUNKS * 8;
  constexpr int kInstr = 64 * kRcpr / 32;
#pragma unroll 4
  for (int k = w; k < kInstr; k += NW) {
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

// Persistent: each CTA (pair) of the grid's p.clusters handles a sequence of
// tokens -- taken one at a time from p.tok_counter by the pair's rank 0 (so
// faster pairs take more), or c, c + p.clusters, ... without a counter -- as
// one sequence of 64-slot blocks (G counts them over the CTA's whole life),
// so that the next token's gathers, scores, exchange and softmax overlap the
// current one's last P.V and O read-out; Q (one buffer) waits only for the
// current token's last scores MMA, the next token's first P.V for the O
// read-out.  Every barrier phase follows G, or the token count k.  Ring entry
// k % kTokRing publishes token k's index (-1: no more tokens) and its last
// valid slot as scanned by the three gather warps.
template <int D, int NSPLIT>
__global__ void __launch_bounds__(NSPLIT == 2 ? 512 : 256, 1)
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
  const int cl = static_cast<int>(blockIdx.x) / NSPLIT;  // this CTA's (pair's) index
  const uint32_t rank = NSPLIT == 2 ? cluster_ctarank() : 0u;
  auto token_of = [&](int k) -> int { return cl + k * p.clusters; };  // k-th token, no counter
  auto bar = [&](int i) -> uint32_t { return base + L::kOffCtrl + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(smem + L::kOffTmemHolder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  volatile int* slot_smem = reinterpret_cast<volatile int*>(smem + L::kOffSlot);
  volatile uint32_t* vmask = reinterpret_cast<volatile uint32_t*>(smem + L::kOffMask);
  volatile int* tok_last = reinterpret_cast<volatile int*>(smem + L::kOffTokLast);
  volatile int* tok_id = reinterpret_cast<volatile int*>(smem + L::kOffTokId);
  volatile int* tok_t = reinterpret_cast<volatile int*>(smem + L::kOffTokT);
  const WaitCtl ctl{abort_flag, p.status, p.limit_ns};
  // Live blocks of the token in ring entry e (after its full barrier).
  auto tok_blocks = [&](int e) -> int {
    const int last = max(max(tok_last[3 * e], tok_last[3 * e + 1]), tok_last[3 * e + 2]);
    return last < 0 ? 0 : last / L::kBI + 1;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      // One cp.async arrival per gather thread, plus the arrival that
      // publishes the block's valid-slot mask.
      mbar_init(bar(L::kBarKvFull + s), 32 * L::kGatherWarps + 1);
      mbar_init(bar(L::kBarKvEmpty + s), 1);
    }
    for (int s = 0; s < L::kSBufs; ++s) {
      mbar_init(bar(L::kBarSFull + s), 1);
      mbar_init(bar(L::kBarSRead + s), 128);
      mbar_init(bar(L::kBarSSum + s), 128);
      mbar_init(bar(L::kBarSFree + s), L::kSoftmaxThreads);
    }
    // Exchange: the peer's four sender warps each signal a filled buffer.
    for (int s = 0; s < L::kXBufs; ++s) mbar_init(bar(L::kBarRecvFull + s), 4);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::kBarPFull + s), L::kSoftmaxThreads);
      mbar_init(bar(L::kBarODone + s), 1);
    }
    mbar_init(bar(L::kBarQFull), 1);
    mbar_init(bar(L::kBarQFree), 1);
    mbar_init(bar(L::kBarOFree), L::kSoftmaxThreads);
    for (int e = 0; e < L::kTokRing; ++e) {
      mbar_init(bar(L::kBarTokFull + e), L::kGatherWarps);
      mbar_init(bar(L::kBarTokEmpty + e), L::kTokReaders);
      mbar_init(bar(L::kBarIdFull + e), 1);
      mbar_init(bar(L::kBarIdEmpty + e), 1);
    }
    mbar_init(bar(L::kBarDrain), 1);
    *abort_flag = *reinterpret_cast<volatile int*>(p.status) != 0 ? 1 : 0;
    *slot_smem = -1;
    if (NSPLIT == 2 && rank == 0 && *abort_flag == 0) {
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
    if (lane == 0) tma_prefetch_desc(&tm_q);
    tmem_alloc(base + L::kOffTmemHolder, L::kTmemCols);
  }
  // Heads beyond H are zero rows of the smem A operand (the TMA box covers H
  // rows, so later loads leave them zero).
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
  if (NSPLIT == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // The pair's exchange slot (claimed by rank 0); without one, nothing runs.
  int slot = -1;
  if (NSPLIT == 2) {
    slot = rank == 0 ? *slot_smem : ld_shared_cluster_s32(mapa_shared(base + L::kOffSlot, 0u));
    if (slot < 0) *abort_flag = 1;
  }
  __syncwarp();
  const bool run = *abort_flag == 0;

  if (warp >= L::kGatherWarp0 && warp < L::kMmaWarp) {
    // ------------------------------------------------------------ gather
    // Per token: its index (handed over within the pair), the index row's
    // last valid slot (each warp scans a third) into ring entry k %
    // kTokRing, then its live blocks.  (An L2 prefetch of the token's Q
    // here cost 1 %.)
    const int w = warp - L::kGatherWarp0;
    const int col0 = static_cast<int>(rank) * DC;
    // Token k's setup: wait until ring entry k % kTokRing is free, learn the
    // token (for D = 512 rank 0 takes it from the counter and writes it into
    // both CTAs' entry, the peer's only once the peer has freed it), scan its
    // index row (16-byte loads issued before any compare) and publish it.
    auto setup = [&](int k) -> bool {
      const int e = k % L::kTokRing;
      if (k >= L::kTokRing &&
          !__all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokEmpty + e), ((k / L::kTokRing) - 1) & 1, ctl)))
        return false;
      int t;
      if (NSPLIT == 2 && p.tok_counter != nullptr) {
        if (w == 0) {
          if (lane == 0) {
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
          // The whole warp again before anyone waits: lanes suspended in a
          // wait while lane 0 hands the token over slowed the handover by
          // thousands of cycles.
          __syncwarp();
        }
        if (!__all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarIdFull + e), (k / L::kTokRing) & 1, ctl)))
          return false;
        t = tok_id[e];
      } else {
        t = token_of(k) < p.tokens ? token_of(k) : -1;
      }
      int last = -1;
      if (t >= 0) {
        const int32_t* row = p.idx + static_cast<size_t>(t) * p.topk;
        const int tid = 32 * w + lane;
        if ((p.topk & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
          const int4* row4 = reinterpret_cast<const int4*>(row);
          const unsigned skv = static_cast<unsigned>(p.S_kv);
#pragma unroll 8
          for (int q = tid; q < p.topk / 4; q += 32 * L::kGatherWarps) {
            const int4 v = __ldg(row4 + q);
            if (static_cast<unsigned>(v.x) < skv) last = 4 * q;
            if (static_cast<unsigned>(v.y) < skv) last = 4 * q + 1;
            if (static_cast<unsigned>(v.z) < skv) last = 4 * q + 2;
            if (static_cast<unsigned>(v.w) < skv) last = 4 * q + 3;
          }
        } else {
#pragma unroll 8
          for (int j = tid; j < p.topk; j += 32 * L::kGatherWarps)
            if (static_cast<unsigned>(__ldg(row + j)) < static_cast<unsigned>(p.S_kv)) last = j;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
      }
      if (lane == 0) {
        if (w == 0) tok_t[e] = t;
        tok_last[3 * e + w] = last;
        mbar_arrive(bar(L::kBarTokFull + e));
      }
      return true;
    };
    // The next token is set up once a couple of the current token's blocks
    // are issued (the gather waits for free kv stages then anyway), so that
    // its index, count and Q are known before the current token ends: set
    // up at the token boundary instead, the next token's first scores came
    // ~15,000 cycles after the current token's last.
    bool ok = run && setup(0);
    int G = 0;
    for (int k = 0; ok; ++k) {
      const int e = k % L::kTokRing;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokFull + e), (k / L::kTokRing) & 1, ctl));
      if (!ok) break;
      const int t = tok_t[e];
      if (t < 0) break;  // no more tokens
      const int nblk = tok_blocks(e);
      const int pre = nblk < 2 ? nblk : 2;  // blocks issued before the next token's setup
      if (pre == 0) {
        ok = setup(k + 1);
        if (!ok) break;
      }
      const int32_t* idx_row = p.idx + static_cast<size_t>(t) * p.topk;
      const int b = t / p.S;
      auto load_idx = [&](int blk, int half) -> int {
        const int j = blk * L::kBI + 32 * half + lane;
        return j < p.topk ? __ldg(idx_row + j) : -1;
      };
      int n0 = nblk > 0 ? load_idx(0, 0) : -1, n1 = nblk > 0 ? load_idx(0, 1) : -1;
      for (int i = 0; i < nblk; ++i, ++G) {
        const int s = G % L::kStages;
        const int r0 = n0, r1 = n1;
        if (i + 1 < nblk) {
          n0 = load_idx(i + 1, 0);
          n1 = load_idx(i + 1, 1);
        }
        const int row0 = b * p.S_kv + (static_cast<unsigned>(r0) < static_cast<unsigned>(p.S_kv) ? r0 : 0);
        const int row1 = b * p.S_kv + (static_cast<unsigned>(r1) < static_cast<unsigned>(p.S_kv) ? r1 : 0);
        if (G >= L::kStages) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarKvEmpty + s), ((G / L::kStages) - 1) & 1, ctl));
          if (!ok) break;
        }
        // The block's valid-slot mask (bit j of word h: slot 32h + j), read by
        // the softmax once this stage's full barrier has completed.
        const uint32_t m0 = __ballot_sync(0xffffffffu, static_cast<unsigned>(r0) < static_cast<unsigned>(p.S_kv));
        const uint32_t m1 = __ballot_sync(0xffffffffu, static_cast<unsigned>(r1) < static_cast<unsigned>(p.S_kv));
        gather_block<L::kChunks, D, L::kGatherWarps>(base + L::kOffKv + static_cast<uint32_t>(s) * L::kStageBytes,
                                    p.kv, col0, row0, row1, w, lane);
        cp_async_arrive_noinc(bar(L::kBarKvFull + s));
        if (w == 0 && lane == 0) {
          vmask[2 * s] = m0;
          vmask[2 * s + 1] = m1;
          mbar_arrive(bar(L::kBarKvFull + s));
        }
        if (i + 1 == pre) {
          ok = setup(k + 1);
          if (!ok) break;
        }
      }
    }
    // Let every copy this warp started land before the CTA can exit.
    cp_async_wait_all();
  } else if (warp == L::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, L::kBI, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, DC, false, true);
      // Descriptors are built once; per MMA only the start-address field
      // (bits 0-13, in 16-byte units) moves, by compile-time offsets.
      const uint64_t d_q = smem_desc(base + L::kOffQ, 16u, 1024u, kSwizzle128B);
      const uint64_t d_k = smem_desc(base + L::kOffKv, 16u, 1024u, kSwizzle128B);
      const uint64_t d_v = smem_desc(base + L::kOffKv, L::kKvChunkBytes, 1024u, kSwizzle128B);
      // Scores of block i over this CTA's columns (M = 128 heads, N = 64
      // slots, K = DC) into score tile i % kSBufs.
      auto issue_s = [&](int i) {
        const uint64_t dk = d_k + ((static_cast<uint32_t>(i % L::kStages) * L::kStageBytes) >> 4);
        const uint32_t d_tm = tmem + L::kTmemS + static_cast<uint32_t>(i % L::kSBufs) * L::kBI;
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(d_tm, d_q + ((c * L::kQChunkBytes + k * 32u) >> 4),
                   dk + ((c * L::kKvChunkBytes + k * 32u) >> 4), idesc_s, (c | k) ? 1u : 0u);
        mma_commit(bar(L::kBarSFull + i % L::kSBufs));
      };
      // O += P.V for block j (block jt of its token: the first overwrites);
      // P (A operand) from TMEM buffer j % 2, V = this CTA's columns of the
      // block, MN-major.
      auto issue_pv = [&](int j, int jt) {
        const int sj = j % L::kStages;
        const uint64_t dv = d_v + ((static_cast<uint32_t>(sj) * L::kStageBytes) >> 4);
        const uint32_t a_tm = tmem + L::kTmemP + static_cast<uint32_t>(j & 1) * (L::kBI / 2);
#pragma unroll
        for (int k = 0; k < L::kBI / 16; ++k)
          mma_ts(tmem + L::kTmemO, a_tm + k * 8, dv + (k * 2048u >> 4), idesc_o,
                 (jt > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(L::kBarKvEmpty + sj));
        mma_commit(bar(L::kBarODone + (j & 1)));
      };
      // Three cursors over the CTA's tokens: Q loads (token lk, one per
      // token with blocks, into the single buffer once the previous such
      // token's last scores MMA has completed), scores (token sk, its block
      // si, sequence index sG) and P.V (vk, vi, vG).  Each caches its
      // token's live-block count (-1: not read yet) and touches the
      // published counts only at token boundaries.  Event loop
      // (non-blocking tests, so that waiting on one kind of work never
      // delays the other), oldest work first: P.V of block vG once its P is
      // written (and, for a token's first block, the previous token's O has
      // been read out); scores of block sG once its kv rows have landed, its
      // score tile has been read by the softmax (block sG - kSBufs) and its
      // token's Q is in; otherwise the next Q load.
      auto tok_known = [&](int k) -> bool {
        return mbar_probe(bar(L::kBarTokFull + k % L::kTokRing), (k / L::kTokRing) & 1);
      };
      auto nblk_of = [&](int k) -> int { return tok_blocks(k % L::kTokRing); };
      int lk = 0, lnb = -1, la = 0, lt = -1;         // load cursor (token lt), loads issued
      bool l_end = false;                             // the load cursor met the end
      int sk = 0, si = 0, snb = -1, sG = 0, sa = 0;   // sa: load index of token sk
      int vk = 0, vi = 0, vnb = -1, vG = 0, va = 0;   // va: load index of token vk
      int qfree = 0;                                  // Q releases committed
      bool ok = run;
      PollState ps = poll_start();
      uint32_t spins = 0;
      while (ok) {
        // ---- cursor bookkeeping (does work only at token boundaries)
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
        if (vnb < 0 && vk < lk) vnb = nblk_of(vk);
        if (vnb >= 0 && vi == vnb && vk < sk) {       // token vk done: release its entry
          mbar_arrive(bar(L::kBarTokEmpty + vk % L::kTokRing));
          if (vnb > 0) ++va;
          ++vk;
          vi = 0;
          vnb = -1;
          continue;
        }
        if (l_end && vk == lk) break;  // every token done
        // ---- events, within the current tokens: back to the bookkeeping
        // only at a token boundary or after a Q load, so that a mid-token
        // iteration tests nothing but the events.
        const bool want_load = lnb > 0;
        const bool need_book = !want_load && lnb < 0 && !l_end && qfree >= la;
        for (;;) {
          if (vG < sG && vi < vnb && mbar_probe(bar(L::kBarPFull + (vG & 1)), (vG >> 1) & 1) &&
              (vi > 0 || va == 0 || mbar_probe(bar(L::kBarOFree), (va - 1) & 1))) {
            tc_fence_after();
            issue_pv(vG, vi);
            ++vi;
            ++vG;
            ps.t0 = globaltimer_ns();  // progress: the limit counts from the last issue
            if (vi == vnb) break;
          } else if (si < snb &&
                     mbar_probe(bar(L::kBarKvFull + sG % L::kStages), (sG / L::kStages) & 1) &&
                     (sG < L::kSBufs ||
                      mbar_probe(bar(L::kBarSFree + sG % L::kSBufs), ((sG / L::kSBufs) - 1) & 1)) &&
                     (si > 0 || mbar_probe(bar(L::kBarQFull), sa & 1))) {
            // The kv tile was written by cp.async (generic proxy): order it
            // before the tensor core's (async proxy) reads.
            fence_proxy_async_smem();
            tc_fence_after();
            issue_s(sG);
            ++si;
            ++sG;
            ps.t0 = globaltimer_ns();
            if (static_cast<int>(blockIdx.x) == p.stall_cta && sG == 1) {  // test hook only
              ok = stall_until_limit(ctl);
              break;
            }
            if (si == snb) {  // the token's last scores: Q may take the next token
              mma_commit(bar(L::kBarQFree));
              ++qfree;
              break;
            }
          } else if (want_load && (la == 0 || mbar_probe(bar(L::kBarQFree), (la - 1) & 1))) {
            // This CTA's column half of token lt's Q into the (free) buffer.
            mbar_arrive_expect_tx(bar(L::kBarQFull), static_cast<uint32_t>(p.H) * 128u * L::kChunks);
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_2d(base + L::kOffQ + c * L::kQChunkBytes, &tm_q,
                          static_cast<int>(rank) * DC + c * 64, lt * p.H, bar(L::kBarQFull));
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
      // No MMA may still be running when TMEM is released, and no Q load
      // still landing when the CTA exits.
      mma_commit(bar(L::kBarDrain));
      mbar_wait_drain(bar(L::kBarDrain), 0);
      if (la > 0) mbar_wait_drain(bar(L::kBarQFull), (la - 1) & 1);
    }
    __syncwarp();
  } else if (NSPLIT == 2 && warp >= L::kSendWarp0) {
    // ------------------------------------------------------------ sender
    // Thread = head row h: this CTA's partial scores of each block, in block
    // floating point, into the peer's receive buffer of the block (L2), then
    // one release-arrive per warp on the peer's barrier; the tile gets the
    // values the peer will see, for the combiner.
    const int sq = warp & 3;  // TMEM lane quarter
    const int h = sq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(sq * 32) << 16;
    const float s1 = p.ref_round ? p.scale : p.scale_log2;
    const uint32_t peer_full = mapa_shared(bar(L::kBarRecvFull), rank ^ 1u);
    uint8_t* peer0 = p.exch + (static_cast<size_t>(slot) * 2 + (rank ^ 1u)) *
                                  (L::kXBufs * L::kXchgBytes);
    bool ok = run;
    int G = 0;
    for (int k = 0; ok; ++k) {
      const int te = k % L::kTokRing;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokFull + te), (k / L::kTokRing) & 1, ctl));
      if (!ok || tok_t[te] < 0) break;
      const int nblk = tok_blocks(te);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kBarTokEmpty + te));
      for (int ib = 0; ib < nblk; ++ib, ++G) {
        const int i = G;  // position in the CTA's block sequence
        const int sb = i % L::kSBufs;
        const int xb = i % L::kXBufs;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull + sb), (i / L::kSBufs) & 1, ctl));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tile = tmem + lane_base + L::kTmemS + sb * L::kBI;
        float x[64];
        tmem_ld32x2(tile, tile + 32, *reinterpret_cast<float(*)[32]>(x),
                    *reinterpret_cast<float(*)[32]>(x + 32));
        const int ex = bfp16_exponent(__fmul_rn(__fmul_rn(absmax_fold_n<64>(x), s1), kExpMargin));
        const float f = __fmul_rn(s1, pow2f(14 - ex)), inv = pow2f(ex - 14);
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 r = bfp16_round2(make_float2(x[2 * k], x[2 * k + 1]), f);
          w[k] = bfp16_pack(r.x, r.y);
          const float2 v = bfp16_value2(r, inv);
          x[2 * k] = v.x;
          x[2 * k + 1] = v.y;
        }
        // The peer has read block i - kXBufs from this buffer once its block
        // i - kXBufs + kSBufs has arrived here (it computed that block into
        // the score tile it freed after reading block i - kXBufs).
        if (i >= L::kXBufs) {
          const int j = i - L::kXBufs + L::kSBufs;
          ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarRecvFull + j % L::kXBufs),
                                                       (j / L::kXBufs) & 1, ctl));
          if (!ok) break;
        }
        // The stores first, so that their way to L2 overlaps the write-back.
        uint8_t* buf = peer0 + static_cast<size_t>(xb) * L::kXchgBytes;
        uint4* dst = reinterpret_cast<uint4*>(buf) + h;
#pragma unroll
        for (int c = 0; c < L::kPieces; ++c)
          dst[c * L::kHPad] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        reinterpret_cast<int*>(buf + L::kXchgScaleOff)[h] = ex;
        // The tile now gets this CTA's partial as the peer will see it.
        tmem_st32(tile, *reinterpret_cast<float(*)[32]>(x));
        tmem_st32(tile + 32, *reinterpret_cast<float(*)[32]>(x + 32));
        tc_fence_before();
        mbar_arrive(bar(L::kBarSRead + sb));
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(peer_full + 8u * static_cast<uint32_t>(xb));
      }
    }
  } else if (NSPLIT == 2 && warp >= L::kCombWarp0 && warp < L::kGatherWarp0) {
    // ------------------------------------------------------------ combiner
    // Thread = head row h: once the peer's partial of block i has arrived
    // and the sender has rounded this CTA's partial in the tile, the tile
    // gets the full scores S = own + peer's, both as the block-floating-point
    // values that were exchanged, so both CTAs add the same two fp32 terms.
    // The peer's row is loaded first so that its L2 latency overlaps the
    // wait for the sender.
    const int sq = warp & 3;  // TMEM lane quarter
    const int h = sq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(sq * 32) << 16;
    const uint8_t* recv0 = p.exch + (static_cast<size_t>(slot) * 2 + rank) *
                                        (L::kXBufs * L::kXchgBytes);
    bool ok = run;
    int G = 0;
    for (int k = 0; ok; ++k) {
      const int te = k % L::kTokRing;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokFull + te), (k / L::kTokRing) & 1, ctl));
      if (!ok || tok_t[te] < 0) break;
      const int nblk = tok_blocks(te);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kBarTokEmpty + te));
      for (int ib = 0; ib < nblk; ++ib, ++G) {
        const int i = G;  // position in the CTA's block sequence
        const int sb = i % L::kSBufs;
        const int xb = i % L::kXBufs;
        ok = __all_sync(0xffffffffu, mbar_wait<true>(bar(L::kBarRecvFull + xb),
                                                     (i / L::kXBufs) & 1, ctl));
        if (!ok) break;
        const uint8_t* buf = recv0 + static_cast<size_t>(xb) * L::kXchgBytes;
        const uint4* src = reinterpret_cast<const uint4*>(buf) + h;
        uint4 y[L::kPieces];
#pragma unroll
        for (int c = 0; c < L::kPieces; ++c) y[c] = __ldcg(src + c * L::kHPad);
        const float pinv = pow2f(__ldcg(reinterpret_cast<const int*>(buf + L::kXchgScaleOff) + h) - 14);
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarSRead + sb), (i / L::kSBufs) & 1, ctl));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tile = tmem + lane_base + L::kTmemS + sb * L::kBI;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float x[32];
          tmem_ld32(tile + 32 * half, x);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 yc = y[4 * half + c];
            const uint32_t ya[4] = {yc.x, yc.y, yc.z, yc.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 pv = bfp16_unpack(ya[k], pinv);
              const int j = 8 * c + 2 * k;
              const float2 sum = add2(make_float2(x[j], x[j + 1]), pv);
              x[j] = sum.x;
              x[j + 1] = sum.y;
            }
          }
          tmem_st32(tile + 32 * half, x);
        }
        // The peer's values are consumed (see the flow-control note above).
        tc_fence_before();
        mbar_arrive(bar(L::kBarSSum + sb));
      }
    }
  } else if (warp < L::kSoftmaxThreads / 32) {
    // ------------------------------------------------------------ softmax
    // Thread = head row h (TMEM lane): all 64 score columns of every block,
    // the whole O row for rescaling and output.
    const int h = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // exp2 argument: score * (c log2 e), or (score * c) * log2 e with the
    // reference-rounding flag (x * s1 * 1 is exact when the flag is off).
    // With the D split the tile already holds s1 * score.
    const float s1 = NSPLIT == 2 ? 1.f : (p.ref_round ? p.scale : p.scale_log2);
    const float s2 = p.ref_round ? 1.4426950408889634f : 1.f;
    // O rows start 32-byte aligned when the tensor does (row and half
    // offsets are multiples of 64 bytes).
    const bool o32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
    bool ok = run;
    int G = 0;  // blocks so far
    for (int tk = 0; ok; ++tk) {
      const int te = tk % L::kTokRing;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarTokFull + te), (tk / L::kTokRing) & 1, ctl));
      if (!ok) break;
      const int t = tok_t[te];
      if (t < 0) break;
      const int nblk = tok_blocks(te);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::kBarTokEmpty + te));
      float m_run = -INFINITY;
      float l_run = 0.f;
      for (int ib = 0; ib < nblk; ++ib, ++G) {
        const int i = G;  // position in the CTA's block sequence
        const int sb = i % L::kSBufs;
        ok = __all_sync(0xffffffffu, mbar_wait(bar((NSPLIT == 2 ? L::kBarSSum : L::kBarSFull) + sb),
                                               (i / L::kSBufs) & 1, ctl));
        if (!ok) break;
        tc_fence_after();
        // The scores imply that the block's kv stage (and its valid-slot mask)
        // has landed; its full barrier is tested only to order the mask read.
        const int st = i % L::kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarKvFull + st), (i / L::kStages) & 1, ctl));
        if (!ok) break;
        const uint32_t msk0 = vmask[2 * st];
        const uint32_t msk1 = vmask[2 * st + 1];
        float x[64];
        tmem_ld32x2(tmem + lane_base + L::kTmemS + sb * L::kBI,
                    tmem + lane_base + L::kTmemS + sb * L::kBI + 32,
                    *reinterpret_cast<float(*)[32]>(x), *reinterpret_cast<float(*)[32]>(x + 32));
        tc_fence_before();
        mbar_arrive(bar(L::kBarSFree + sb));
        // Scale (unless the tile already holds the exp2 argument), then mask
        // (a block whose 64 slots are all valid has nothing to mask).
        if (NSPLIT == 1 || p.ref_round) {
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = (x[j] * s1) * s2;
        }
        if ((msk0 & msk1) != 0xffffffffu) {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const uint32_t bit = ((j < 32 ? msk0 : msk1) >> (j & 31)) & 1u;
            x[j] = bit ? x[j] : -INFINITY;
          }
        }
        const float mloc = max_n<64>(x);
        const float m_new = fmaxf(m_run, mloc);
        const bool bump = (m_run == -INFINITY) ? (m_new != -INFINITY) : (m_new > m_run + 8.f);
        float alpha = 1.f;
        if (bump) {
          alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        const float2 nm2 = make_float2(-m_use, -m_use);
        // P buffer i % 2 was last read by P.V of block i-2.
        if (i >= 2) {
          ok = __all_sync(0xffffffffu,
                          mbar_wait(bar(L::kBarODone + (i & 1)), ((i - 2) >> 1) & 1, ctl));
          if (!ok) break;
          tc_fence_after();
        }
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[16];
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            const float2 d = add2(make_float2(x[32 * half + 2 * w], x[32 * half + 2 * w + 1]), nm2);
            const float p0 = fast_exp2(d.x);
            const float p1 = fast_exp2(d.y);
            pk[w] = pack_bf16x2(p0, p1);
            rs[w & 3] += p0 + p1;  // fp32 probabilities: the LSE must not carry bf16 rounding
          }
          tmem_st16u(tmem + lane_base + L::kTmemP + static_cast<uint32_t>(i & 1) * (L::kBI / 2) +
                         16 * half, pk);
        }
        l_run += (rs[0] + rs[1]) + (rs[2] + rs[3]);
        // O was accumulated against the old max: once P.V of block i-1 has
        // completed, rescale this row before P.V of block i may start (whole
        // warp, since TMEM accesses are warp-collective; rows without a bump
        // use 1).
        const bool need_rescale = bump && alpha != 0.f && ib > 0;
        if (__any_sync(0xffffffffu, need_rescale)) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarODone + ((i - 1) & 1)),
                                                 ((i - 1) >> 1) & 1, ctl));
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
        tc_fence_before();
        mbar_arrive(bar(L::kBarPFull + (i & 1)));
      }
      if (!ok) break;
      // The token's last P.V, then O (normalised, bf16) straight from TMEM
      // to its rows with 32-byte stores (the kv ring, which used to stage it
      // for a TMA store, already holds the next token's rows), and the LSE.
      // 64 columns per TMEM trip (one wait for two loads; 32 at a time:
      // 4.65 against 4.60 ms on the headline workload).
      if (nblk > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(L::kBarODone + ((G - 1) & 1)),
                                               ((G - 1) >> 1) & 1, ctl));
        if (!ok) break;
        tc_fence_after();
      }
      const float sink2 = h < p.H ? __ldg(p.sink + h) * 1.4426950408889634f : 0.f;
      const float m_fin = fmaxf(m_run, sink2);
      const float so = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_fin);
      const float Z = l_run * so + fast_exp2(sink2 - m_fin);
      const float inv = so / Z;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(t) * p.H + h) * D + static_cast<size_t>(rank) * DC;
#pragma unroll 1
      for (int c2 = 0; c2 < DC / 64; ++c2) {
        float v2[2][32];
        if (nblk > 0) {
          tmem_ld32x2(tmem + lane_base + L::kTmemO + c2 * 64,
                      tmem + lane_base + L::kTmemO + c2 * 64 + 32, v2[0], v2[1]);
        } else {  // no valid slot: O was never written, the output is 0
#pragma unroll
          for (int kk = 0; kk < 32; ++kk) v2[0][kk] = v2[1][kk] = 0.f;
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * c2 + cc;
          const float* v = v2[cc];
          if (h < p.H) {
            uint32_t w[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const float2 y = mul2(make_float2(v[2 * u], v[2 * u + 1]), make_float2(inv, inv));
              w[u] = pack_bf16x2(y.x, y.y);
            }
            if (o32) {  // 32-byte stores: half the transactions of 16-byte ones
              st_global_v8(orow + 32 * c, *reinterpret_cast<const uint32_t(*)[8]>(w));
              st_global_v8(orow + 32 * c + 16, *reinterpret_cast<const uint32_t(*)[8]>(w + 8));
            } else {
              uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                dst[kk] = make_uint4(w[4 * kk], w[4 * kk + 1], w[4 * kk + 2], w[4 * kk + 3]);
            }
          }
        }
      }
      if (nblk > 0) {
        // O is in registers: the next token's first P.V may overwrite it.
        tc_fence_before();
        mbar_arrive(bar(L::kBarOFree));
      }
      if (rank == 0 && h < p.H) p.lse[static_cast<size_t>(t) * p.H + h] = m_fin + log2f(Z);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (NSPLIT == 2) cluster_sync();
  if (warp == L::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  // Release the pair's exchange slot once both CTAs are done with it.
  if (NSPLIT == 2 && rank == 0 && threadIdx.x == 0 && slot >= 0) {
    __threadfence();
    atomicExch(p.slot_flags + slot, 0);
  }
}

// Clusters (pairs, or single CTAs for D = 64) of one instantiation that fit
// on the device at once, per device (the persistent grid's size).
template <int D, int NSPLIT>
static int fwd_resident_clusters(cudaLaunchConfig_t cfg) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  int n = 0;
  auto kern = smqa_fwd_kernel<D, NSPLIT>;
  if (NSPLIT > 1) {
    cfg.gridDim = dim3(NSPLIT, 1, 1);
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

template <int D, int NSPLIT>
static cudaError_t launch_fwd_impl(const CUtensorMap& tm_q, const FwdParams& p0, int tokens,
                                   cudaStream_t stream) {
  using L = FwdLayout<D, NSPLIT>;
  auto kern = smqa_fwd_kernel<D, NSPLIT>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(L::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NSPLIT;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int resident = fwd_resident_clusters<D, NSPLIT>(cfg);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  FwdParams p = p0;
  p.tokens = tokens;
  p.clusters = tokens < resident ? tokens : resident;
  cfg.gridDim = dim3(static_cast<unsigned>(p.clusters) * NSPLIT, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, tm_q, p);
}

cudaError_t launch_fwd(const CUtensorMap& tm_q, const FwdParams& p, int tokens,
                       cudaStream_t stream) {
  if (p.D == 512) return launch_fwd_impl<512, 2>(tm_q, p, tokens, stream);
  if (p.D == 64) return launch_fwd_impl<64, 1>(tm_q, p, tokens, stream);
  return cudaErrorInvalidValue;
}

}  // namespace smqa
