// Shared device helpers for the sm_103a kernels: error word, bounded
// mbarrier waits, TMA tile loads, tcgen05 (TMEM alloc / MMA / commit / load).
//
// Every inline-PTX form here is written from the PTX ISA description of the
// instruction; none is taken from a library.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda.h>

namespace dinfer {

// ---------------------------------------------------------------------------
// device status word (read by the host after a call); bits are OR-ed in
// ---------------------------------------------------------------------------
enum : uint32_t {
  ST_WAIT_TIMEOUT = 1u << 0,   // a bounded mbarrier wait gave up
  ST_BAD_TOKEN = 1u << 1,      // an id outside [0, vocab) reached the embedding
  ST_NAN_CONF = 1u << 2,       // a confidence was NaN
  ST_ITER_OVERFLOW = 1u << 3,  // a block needed more than block_len iterations
  ST_NO_COMMIT = 1u << 4,      // an iteration with masks left committed nothing
};

// Per-context device-resident loop state.  Kernels read the current block
// start from here so that one captured graph serves every block.
constexpr int kMaxBatch = 64;
constexpr int kMaxBlocks = 4096;
struct DevState {
  int32_t block_start;   // absolute position of the current block
  int32_t block_index;
  int32_t n_blocks;
  int32_t iteration;     // iterations done in the current block
  int32_t total_iterations;
  int32_t refreshes;
  uint32_t status;
  int32_t any_masked;    // 1 while some sequence of the batch has masks in the block
  uint32_t diag[4];      // first timed-out wait: (kernel << 8 | site) + 1, block x | y << 16, block z | step << 16, thread
  uint32_t moe_touched;  // (MoE layer forward, expert) pairs that received rows (measurement count)
  int32_t eos_id;        // end-of-sequence id (-1: none)
  int32_t any_left;      // 1 while some sequence has masked positions after the current block
  int32_t committed[kMaxBatch];    // commits of the last iteration, per sequence
  int32_t iters_per_block[kMaxBlocks];
};

__device__ __forceinline__ void set_status(DevState* st, uint32_t bit) {
  if (st) atomicOr(&st->status, bit);
}

// Record the first wait that timed out (kernel and site codes are the
// kernel's own) together with the CTA, the pipeline step and the thread.
constexpr uint32_t kDiagGemm = 1, kDiagLmHead = 2, kDiagAttn = 3;
__device__ __forceinline__ void record_timeout(DevState* st, uint32_t kernel, uint32_t site, uint32_t step) {
  if (!st) return;
  atomicOr(&st->status, ST_WAIT_TIMEOUT);
  if (atomicCAS(&st->diag[0], 0u, ((kernel << 8) | site) + 1u) == 0u) {
    st->diag[1] = blockIdx.x | (blockIdx.y << 16);
    st->diag[2] = blockIdx.z | (step << 16);
    st->diag[3] = threadIdx.x;
  }
}

// ---------------------------------------------------------------------------
// small math
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Feature layout of the row kernels (residual norms, MoE combine): thread t
// of a row holds 16 features of the 128-feature tile t / 8, as four groups of
// 4 consecutive features kRowGroupStride apart, starting at row_f0(t).  The 8
// threads of a tile then read or write 128 contiguous bytes of fp32 (64 of
// bf16) per instruction, so every cache line is fetched whole and once.
constexpr int kRowGroupStride = 32;
__device__ __forceinline__ int row_f0(int t) { return (t >> 3) * 128 + (t & 7) * 4; }

// Online-softmax state over a set of logits, in the log2 domain:
// m = max t, s = sum 2^(t - m), a = index of the max (lowest on ties).
struct SoftmaxState {
  float m;
  float s;
  int a;
};
__device__ __forceinline__ SoftmaxState sm_empty() { return {-INFINITY, 0.f, 0x7fffffff}; }
__device__ __forceinline__ SoftmaxState sm_merge(SoftmaxState x, SoftmaxState y) {
  if (y.m == -INFINITY) return x;
  if (x.m == -INFINITY) return y;
  SoftmaxState r;
  if (x.m > y.m || (x.m == y.m && x.a < y.a)) {
    r.m = x.m; r.a = x.a;
  } else {
    r.m = y.m; r.a = y.a;
  }
  r.s = x.s * exp2f(x.m - r.m) + y.s * exp2f(y.m - r.m);
  return r;
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}


// Wait for the phase with the given parity to complete.  Gives up after
// about kWaitCycles SM cycles (~1 s), sets *abort and returns false.
constexpr long long kWaitCycles = 2000000000LL;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort = 1;
      return false;
    }
  }
}

// mbar_wait that records where it gave up when its own bound ran out.
__device__ __forceinline__ bool mbar_wait_diag(uint64_t* bar, uint32_t parity, volatile int* abort, DevState* st,
                                               uint32_t kernel, uint32_t site, uint32_t step) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort = 1;
      record_timeout(st, kernel, site, step);
      return false;
    }
  }
}

// Wait for a phase whatever the abort flag says (operations already issued
// by this CTA: copies in flight, committed MMAs), bounded by kWaitCycles / 4.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles / 4) return false;
  return true;
}

// ---------------------------------------------------------------------------
// TMA (2-D tiled tensor loads into shared memory, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// x = innermost (element) coordinate, must be a multiple of 8 for bf16
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads
// ---------------------------------------------------------------------------
// Allocate ncols TMEM columns (power of two >= 32); the whole warp executes.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (rows of 64 bf16 = 128 B, 8-row groups 1024 B apart).
// Fields: start address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29
// (unused for swizzled K-major; 1), stride byte offset >> 4 in 32-45 (1024 B),
// descriptor version 1 in bits 46-47, base offset 0, swizzle mode 2 (128 B)
// in bits 61-63.
__device__ __forceinline__ uint64_t make_sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A/B, fp32 accumulator,
// both operands K-major: D format (F32 = 1) bits 4-5, A format (BF16 = 1)
// bits 7-9, B format (BF16 = 1) bits 10-12, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once all tcgen05 ops issued so far by this thread completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets lane
// (base lane + i), columns col..col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .b32 rx;\n .reg .pred px;\n"
      " elect.sync rx|px, %1;\n"
      " selp.u32 %0, 1, 0, px;\n}"
      : "=r"(pred)
      : "r"(0xffffffffu));
  return pred;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: wait until the preceding kernel of the
// stream has completed and its writes are visible (no-op without the launch
// attribute); allow the next kernel of the stream to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace dinfer
