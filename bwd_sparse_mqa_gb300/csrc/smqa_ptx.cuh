// smqa_ptx.cuh -- sm_103a building blocks written as inline PTX: mbarriers with
// bounded waits, cp.async, TMA tile loads and stores, tcgen05 (TMEM alloc,
// MMA, commit, ld/st), shared-memory matrix descriptors and cluster (DSMEM)
// addressing.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace smqa {

// ---------------------------------------------------------------------------
// Device status word and bounded waits
// ---------------------------------------------------------------------------
// Every wait below gives up after a wall-time limit (measured with
// %globaltimer).  The first wait that gives up sets its CTA's abort flag and
// ORs kStatusTimeout into the global status word.  From then on every wait of
// every CTA that sees the flag or the status word returns at once, every role
// loop stops, TMEM is freed and the CTA exits; CTAs that start while the
// status word is set begin aborted (the word is sticky until the host clears
// it with smqa_device_status(1)).  Results of an aborted launch are undefined.
constexpr int kStatusTimeout = 4;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy and to the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Arrive on a barrier that lives in another CTA of the cluster
// (`remote` is a shared::cluster address from mapa).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test (never suspends the thread): for loops that poll
// several barriers, where a suspending try_wait on one would delay noticing
// another.
__device__ __forceinline__ bool mbar_probe(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared per-CTA control block used by the bounded waits.
struct WaitCtl {
  volatile int* abort_flag;  // shared memory
  int* status;               // global status word
  uint64_t limit_ns;
};

__device__ __forceinline__ void ctl_abort(const WaitCtl& c) {
  if (*c.abort_flag == 0) {
    *c.abort_flag = 1;
    atomicOr(c.status, kStatusTimeout);
  }
}

// Polling state of one bounded wait.  Every 64 polls the shared abort flag
// and the wall clock are checked and the global status word is loaded; that
// load is examined only at the next check, so its L2 latency never delays
// noticing a completed phase.
struct PollState {
  uint64_t t0;
  int status_seen;
};

__device__ __forceinline__ PollState poll_start() { return PollState{globaltimer_ns(), 0}; }

// False once the CTA must give up (limit reached, or an abort seen here or
// in the status word).
__device__ __forceinline__ bool poll_check(const WaitCtl& c, PollState& ps) {
  if (*c.abort_flag || ps.status_seen != 0) {
    *c.abort_flag = 1;
    return false;
  }
  ps.status_seen = *reinterpret_cast<volatile int*>(c.status);
  if (globaltimer_ns() - ps.t0 > c.limit_ns) {
    ctl_abort(c);
    return false;
  }
  return true;
}

// Test hook (the library's smqa_debug_stall): waits for a condition that
// never comes true, bounded like every wait, until the limit runs out and
// the CTA aborts.  Returns false.
__device__ __forceinline__ bool stall_until_limit(const WaitCtl& c) {
  PollState ps = poll_start();
  while (poll_check(c, ps)) {
  }
  return false;
}

// Waits until the phase with parity `parity` of `bar` has completed.
// Returns false (and aborts the CTA) if the limit runs out or the CTA has
// already aborted.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  if (kCluster ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
  PollState ps = poll_start();
  for (uint32_t it = 1;; ++it) {
    if (kCluster ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
    if ((it & 63u) == 0u && !poll_check(c, ps)) return false;
  }
}

// Bounded wait used only on the way out of a kernel (for copies or MMAs that
// may still be in flight after an abort): ignores the abort flag.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity,
                                                uint64_t limit_ns = 200000000ull) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// ---------------------------------------------------------------------------
// Live slot range of a token
// ---------------------------------------------------------------------------
// Every thread of the CTA calls this before the CTA's first barrier: the
// warp's largest slot j < topk whose index names a row in [0, S_kv) (or -1)
// goes to warp_last[warp].  After the barrier, live_blocks() turns the
// per-warp values into the number of slot blocks that hold any valid slot;
// blocks past the last valid slot contribute nothing and are skipped.
__device__ __forceinline__ void scan_last_valid(const int32_t* idx_row, int topk, int S_kv,
                                                volatile int* warp_last) {
  int last = -1;
#pragma unroll 4
  for (int j = static_cast<int>(threadIdx.x); j < topk; j += static_cast<int>(blockDim.x))
    if (static_cast<unsigned>(__ldg(idx_row + j)) < static_cast<unsigned>(S_kv)) last = j;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
  if ((threadIdx.x & 31) == 0) warp_last[threadIdx.x >> 5] = last;
}

__device__ __forceinline__ int live_blocks(const volatile int* warp_last, int block_slots) {
  int last = -1;
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  for (int w = 0; w < nwarps; ++w) last = max(last, warp_last[w]);
  return last < 0 ? 0 : last / block_slots + 1;
}

// ---------------------------------------------------------------------------
// Proxy fences and named barriers
// ---------------------------------------------------------------------------
// Generic-proxy shared-memory writes -> later async-proxy reads (MMA / TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// 32-bit load from another CTA's shared memory (`remote` from mapa).
__device__ __forceinline__ int ld_shared_cluster_s32(uint32_t remote) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_cluster_s32(uint32_t remote, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// cp.async (16-byte global -> shared copies, L1 bypassed)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once every cp.async this thread has issued so far has
// landed (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
// Waits for every cp.async this thread started (committed or not).
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}

// 32-byte global store (eight 32-bit words; the address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* addr, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(addr), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Prefetch of one box at (x, y) into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* m, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(m), "r"(x), "r"(y) : "memory");
}
// 2-D tiled load of one box at (x, y) into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(m), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 2-D tensor store of one shared-memory box (tracked by this thread's bulk
// async-groups), and the group commit / wait for it.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(m),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor core
// ---------------------------------------------------------------------------
// Allocation is done by one full warp; the base address lands in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format).
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 descriptor version (1)
//   bits 49-51 base offset (0: atoms are aligned)      bits 61-63 swizzle
// Swizzle codes: 0 none, 2 = 128-byte, 4 = 64-byte, 6 = 32-byte.
constexpr uint32_t kSwizzle128B = 2;
constexpr uint32_t kSwizzle64B = 4;

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(swizzle & 7u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and an fp32 accumulator.
//   bits 4-5 D format (1 = f32)   bits 7-9 A format (1 = bf16)
//   bits 10-12 B format (1 = bf16) bit 15 A is MN-major   bit 16 B is MN-major
//   bits 17-22 N >> 3             bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn_major) << 15) |
         (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.  No "memory"
// clobber: the MMA touches no memory the compiler tracks, and leaving it out
// lets descriptor arithmetic for the next MMA be scheduled early (a clobber
// serialises it behind every MMA and starves the tensor core).  Ordering
// against other threads' writes comes from the barrier/fence asms around it.
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// D[tmem] (+)= A[tmem] * B[smem]; A is M rows (lanes) x K, two 16-bit
// elements per 32-bit column, element 2c in the low half of column c.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane
// (warp's lane quarter base + i), columns [col, col+32).  Includes the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 32-column loads issued together, one wait: v0 from taddr0, v1 from
// taddr1 (same lane mapping as tmem_ld32).
__device__ __forceinline__ void tmem_ld32x2(uint32_t taddr0, uint32_t taddr1, float (&v0)[32],
                                            float (&v1)[32]) {
  uint32_t r0[32], r1[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]), "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]), "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]), "=r"(r0[16]), "=r"(r0[17]), "=r"(r0[18]), "=r"(r0[19]), "=r"(r0[20]), "=r"(r0[21]), "=r"(r0[22]), "=r"(r0[23]), "=r"(r0[24]), "=r"(r0[25]), "=r"(r0[26]), "=r"(r0[27]), "=r"(r0[28]), "=r"(r0[29]), "=r"(r0[30]), "=r"(r0[31]),
        "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]), "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]), "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]), "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]), "=r"(r1[14]), "=r"(r1[15]), "=r"(r1[16]), "=r"(r1[17]), "=r"(r1[18]), "=r"(r1[19]), "=r"(r1[20]), "=r"(r1[21]), "=r"(r1[22]), "=r"(r1[23]), "=r"(r1[24]), "=r"(r1[25]), "=r"(r1[26]), "=r"(r1[27]), "=r"(r1[28]), "=r"(r1[29]), "=r"(r1[30]), "=r"(r1[31])
      : "r"(taddr0), "r"(taddr1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v0[i] = __uint_as_float(r0[i]);
    v1[i] = __uint_as_float(r1[i]);
  }
}

// 16 consecutive 32-bit columns from this thread's lane (warp-collective),
// waiting until the stores have completed.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// ---------------------------------------------------------------------------
// Small numeric helpers
// ---------------------------------------------------------------------------
// Two fp32 operations in one instruction (packed f32x2, sm_100 and later);
// each lane is the IEEE round-to-nearest result of the scalar operation.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats -> packed bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// max(a, b, c) / min(a, b, c) in one instruction (the three-input forms of
// sm_100 and later).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// The largest and the smallest of N values (N = 32 or 64), as trees of
// three-input maxima and minima.
template <int N>
__device__ __forceinline__ float2 maxmin_n(const float* x) {
  static_assert(N == 32 || N == 64, "maxmin_n: 32 or 64 values");
  constexpr int G = N / 3;  // full groups of three; N % 3 values are left over
  float a[G + 1], b[G + 1];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    a[j] = fmax3f(x[3 * j], x[3 * j + 1], x[3 * j + 2]);
    b[j] = fmin3f(x[3 * j], x[3 * j + 1], x[3 * j + 2]);
  }
  if constexpr (N % 3 == 2) {
    a[G] = fmaxf(x[N - 2], x[N - 1]);
    b[G] = fminf(x[N - 2], x[N - 1]);
  } else {
    a[G] = x[N - 1];
    b[G] = x[N - 1];
  }
  // Reduce the G + 1 partial results three at a time.
  int n = G + 1;
#pragma unroll
  for (int round = 0; round < 4; ++round) {
    if (n <= 1) break;
    int m = 0;
#pragma unroll
    for (int j = 0; j + 2 < n; j += 3, ++m) {
      a[m] = fmax3f(a[j], a[j + 1], a[j + 2]);
      b[m] = fmin3f(b[j], b[j + 1], b[j + 2]);
    }
    const int rest = n % 3;
    if (rest == 1) {
      a[m] = a[n - 1];
      b[m] = b[n - 1];
      ++m;
    } else if (rest == 2) {
      a[m] = fmaxf(a[n - 2], a[n - 1]);
      b[m] = fminf(b[n - 2], b[n - 1]);
      ++m;
    }
    n = m;
  }
  return make_float2(a[0], b[0]);
}

// The largest of N values; and the largest of their magnitudes, taken as
// max(max x, -min x) (no absolute-value instruction per element).
template <int N>
__device__ __forceinline__ float max_n(const float* x) {
  static_assert(N >= 2, "max_n: at least two values");
  float a[N / 3 + 1];
  constexpr int G = N / 3;
#pragma unroll
  for (int j = 0; j < G; ++j) a[j] = fmax3f(x[3 * j], x[3 * j + 1], x[3 * j + 2]);
  a[G] = N % 3 == 2 ? fmaxf(x[N - 2], x[N - 1]) : x[N - 1];
  int n = G + 1;
#pragma unroll
  for (int round = 0; round < 4; ++round) {
    if (n <= 1) break;
    int m = 0;
#pragma unroll
    for (int j = 0; j + 2 < n; j += 3, ++m) a[m] = fmax3f(a[j], a[j + 1], a[j + 2]);
    const int rest = n % 3;
    if (rest == 1) a[m++] = a[n - 1];
    else if (rest == 2) { a[m] = fmaxf(a[n - 2], a[n - 1]); ++m; }
    n = m;
  }
  return a[0];
}
template <int N>
__device__ __forceinline__ float absmax_n(const float* x) {
  const float2 mm = maxmin_n<N>(x);
  return fmaxf(mm.x, -mm.y);
}
// The same magnitude maximum with the absolute values taken in the first
// level of the tree (the form the forward's sender runs faster with; the
// backward's runs faster with absmax_n).
template <int N>
__device__ __forceinline__ float absmax_fold_n(const float* x) {
  float y[N / 3 + 1];
  constexpr int G = N / 3;
#pragma unroll
  for (int j = 0; j < G; ++j) y[j] = fmax3f(fabsf(x[3 * j]), fabsf(x[3 * j + 1]), fabsf(x[3 * j + 2]));
  y[G] = N % 3 == 2 ? fmaxf(fabsf(x[N - 2]), fabsf(x[N - 1])) : fabsf(x[N - 1]);
  return max_n<G + 1>(y);
}

// Block floating point of one head's partial sums of a block (the forward's
// partial scores and the backward's partial S and dP), v = s1 x with x the
// raw partial and s1 its scale (the softmax scale in the exp2 domain, or
// sm_scale for dP): exponent
// e = floor(log2(v_max (1 + 2^-15))) with v_max = s1 max|x| (clamped to
// [-100, 100]); each value becomes the integer n = rint(x * (s1 2^(14-e)))
// and stands for n 2^(e-14).  The factor 1 + 2^-15 keeps |x s1 2^(14-e)|
// below 32767.5 (with every fp32 rounding of v_max counted), so |n| <= 32767
// without a clamp; for 2^-100 <= v_max < 2^101 the absolute error of a value
// is at most 2^-15 (1 + 2^-14) v_max.  n is stored offset by 32768 as an
// unsigned 16-bit field.  One fused multiply-add rounds: x * f + kRoundBias,
// with kRoundBias = 1.5 * 2^23 + 32768, is exactly rounded to an integer
// whose low 16 bits are n + 32768; the field is unpacked by placing it under
// the exponent of 2^23.  Every step is exact or one IEEE rounding (explicit
// round-to-nearest operations), so the sender and the peer get the same value.
constexpr float kRoundBias = 12615680.f;        // 1.5 * 2^23 + 32768
constexpr float kUnpackBias = 8421376.f;         // 2^23 + 32768
constexpr float kExpMargin = 1.000030517578125f;  // 1 + 2^-15

__device__ __forceinline__ int bfp16_exponent(float vmax_abs) {
  const int e = static_cast<int>((__float_as_uint(vmax_abs) >> 23) & 0xffu) - 127;
  return min(max(e, -100), 100);
}
// 2^k as a float (k within the normal range).
__device__ __forceinline__ float pow2f(int k) {
  return __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
}
// kRoundBias + n for two raw partials x (f = s1 2^(14-e)).
__device__ __forceinline__ float2 bfp16_round2(float2 x, float f) {
  return fma2(x, make_float2(f, f), make_float2(kRoundBias, kRoundBias));
}
// The values n 2^(e-14) of two rounded kRoundBias + n (inv = 2^(e-14)).
__device__ __forceinline__ float2 bfp16_value2(float2 r, float inv) {
  return fma2(r, make_float2(inv, inv), make_float2(-kRoundBias * inv, -kRoundBias * inv));
}
// Two rounded values -> two 16-bit fields (the first in the low half).
__device__ __forceinline__ uint32_t bfp16_pack(float r_lo, float r_hi) {
  return __byte_perm(__float_as_uint(r_lo), __float_as_uint(r_hi), 0x5410);
}
// A packed pair -> the two values it stands for.
__device__ __forceinline__ float2 bfp16_unpack(uint32_t w, float inv) {
  const float lo = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7610));
  const float hi = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7632));
  return fma2(make_float2(lo, hi), make_float2(inv, inv),
              make_float2(-kUnpackBias * inv, -kUnpackBias * inv));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

}  // namespace smqa
