// Pair-CTA tensor-core GEMM for sm_103a (tcgen05 cta_group::2): Y = X W^T for
// many token rows (the block-boundary refresh, batched blocks), where the
// GEMM is bound by the tensor cores rather than by the weight stream.
//
// A cluster of two CTAs on two SMs computes one 256 x BN tile: weight rows
// are the MMA's M dimension (256 = 128 per CTA), tokens its N dimension.
// Each CTA stages its own 128 weight rows and HALF of the BN token rows; the
// leader CTA (cluster rank 0) issues tcgen05.mma.cta_group::2, which reads
// both CTAs' shared memory and leaves each CTA's 128 x BN accumulator in its
// own TMEM.  Per SM this halves the token bytes staged and read by the tensor
// cores per MMA against a one-CTA 128 x BN tile, for the same work.
//
// Synchronisation across the pair:
//   full[s]    (leader) both CTAs' copies of stage s complete on it: the
//              leader expects the bytes of both, the peer's copies use the
//              cta_group::2 form that signals the leader's barrier;
//   empty[s]   (each CTA) the leader's commit, multicast to both CTAs, frees
//              stage s in both;
//   tfull[a]   (each CTA) the leader's commit after a tile's last k-step,
//              multicast: accumulator a is ready in both TMEMs;
//   tempty[a]  (leader) the 128 epilogue threads of BOTH CTAs arrive (the
//              peer's remotely) once they have read accumulator a.
// Work is dealt in whole tiles, or stream-K: the (pair tile, k-step) units
// split evenly over the pairs, both CTAs of a pair taking the same units for
// their own rows.  The epilogue is the one-CTA kernel's (run_epilogue), each
// CTA finishing its own 128 rows x BN tokens; a split tile leaves
// token-major fp32 partials in the CTA's two workspace slots, which the
// following residual norm adds (residual GEMMs) or splitk_fixup_pair_kernel
// sums and finishes with the same epilogue.
#pragma once
#include "gemm_tc.cuh"

namespace dinfer {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// one warp of each CTA of the pair allocates, together
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma_pair_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at this offset in both CTAs of the pair once the
// tcgen05 operations issued so far by this thread completed.
__device__ __forceinline__ void tc_commit_pair_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// mbar_wait for a barrier that the other CTA of the pair also arrives on
// (acquire at cluster scope), bounded like mbar_wait
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort = 1;
      return false;
    }
  }
}

template <int BN>  // tokens per pair tile (the MMA's N); each CTA stages BN / 2
struct Gemm2Cfg {
  static constexpr int kStageA = 128 * 64 * 2;
  static constexpr int kStageB = (BN / 2) * 64 * 2;
  static constexpr int kStage = kStageA + kStageB;
  static constexpr int kXchgBufs = 2;
  static constexpr int kXchgFloats = kXchgBufs * 128 * 17;
  static constexpr int kStageOutBytes = 2 * 16 * 128 * 2;  // QKV output staging (see epilogue_chunk)
  static constexpr int kStages = (232448 - 1024 - kXchgFloats * 4 - kStageOutBytes - 512) / kStage;
  static constexpr int kSmem = 1024 + kStages * kStage + kXchgFloats * 4 + kStageOutBytes + 512;
  // two accumulators of BN columns, allocated as a power of two
  static constexpr int kTmemCols = 2 * BN <= 256 ? 256 : 512;
  static_assert(kSmem <= 232448, "pair GEMM shared memory above 227 KB");
  static_assert(2 * BN <= 512 && BN % 16 == 0, "two accumulators of BN columns must fit in TMEM");
  static_assert((BN / 2) * 128 % 1024 == 0, "each CTA's token half must keep the 1024-byte swizzle alignment");
};

// Pair tile t -> this CTA's 128-row tile of weight pair tile np (rows
// 256 np .. 256 np + 255; this CTA's half is 128-row tile 2 np + rank) and
// token tile mt (pair_tile_coords: the pairs running at once share a few of
// each through L2).
template <int BN>
__device__ __forceinline__ TileRef pair_tile(const GemmArgs& a, int t, int rank) {
  TileRef r;
  int np;
  pair_tile_coords(t, a.m_tiles, a.n_tiles / 2, np, r.mt);
  r.nt = 2 * np + rank;
  r.a_base = 0;
  r.b_row = r.mt * BN;
  r.m_lim = a.M;
  r.out_base = 0;
  return r;
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc2_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  using C = Gemm2Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Pipe p;
  p.stages = smem;
  float* xchg = reinterpret_cast<float*>(smem + C::kStages * C::kStage);
  __nv_bfloat16* stage_out = reinterpret_cast<__nv_bfloat16*>(xchg + C::kXchgFloats);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(stage_out) + C::kStageOutBytes);
  p.full = bars;
  p.empty = bars + C::kStages;
  p.tfull = bars + 2 * C::kStages;
  p.tempty = p.tfull + 2;
  p.drain = p.tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p.drain + 1);
  volatile int* misc = reinterpret_cast<volatile int*>(tmem_slot + 1);
  p.abort_flag = misc;
  p.rec = nullptr;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const GemmArgs& a = args;
  const int rank = (int)cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int tiles = (a.n_tiles / 2) * a.m_tiles;
  SegList sl;
  if (a.stream_k) {
    Sched sc;
    sc.G = npairs;
    sc.KT = a.k_tiles;
    sc.U = (unsigned)tiles * a.k_tiles;
    sl.init(1, a.k_tiles, sc.start(pair), sc.start(pair + 1));
  } else {
    sl.init(0, a.k_tiles, pair, tiles, npairs);  // tiles pair, pair + npairs, ...
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&p.full[s], 1);
      mbar_init(&p.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p.tfull[i], 1);
      mbar_init(&p.tempty[i], 2 * 128);
    }
    mbar_init(p.drain, 1);
    misc[0] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.b);
    prefetch_tmap(&maps.a[0]);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, C::kTmemCols);
  tc_fence_before();
  // both CTAs' barriers are initialised and their TMEM allocated before any
  // copy or arrive of one CTA can reach the other
  cluster_barrier();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == 0) {
    // ------------------------------ TMA producer (both CTAs) ------------------------------
    if (elect_one_sync()) {
      const uint64_t pol_w = l2_policy_evict_normal();  // every weight tile is read by m_tiles pairs
      const uint64_t pol_x = l2_policy_evict_last();
      const uint32_t full0 = mapa_shared(smem_u32(p.full), 0);  // the leader's full barriers
      const int b_half = rank * (BN / 2);
      uint32_t it = 0;
      bool waited = false;  // griddepcontrol.wait: before the first token tile
      for (int j = 0; j < sl.nseg && !*p.abort_flag; ++j) {
        int t, kb, ke;
        sl.seg(j, t, kb, ke);
        const TileRef tr = pair_tile<BN>(a, t, rank);
        bool ok = true;
        for (int k = kb; k < ke; ++k, ++it) {
          const int s = it % C::kStages;
          const uint32_t round = it / C::kStages;
          if (!mbar_wait(&p.empty[s], (round & 1) ^ 1, p.abort_flag)) { ok = false; break; }
          if (rank == 0) mbar_arrive_expect_tx(&p.full[s], 2 * C::kStage);
          uint8_t* st = p.stages + s * C::kStage;
          const uint32_t fb = full0 + s * 8;
          // the weights do not depend on the preceding kernel
          load_stage_a<true>(maps, a, st, fb, tr, k, pol_w);
          if (!waited) {
            pdl_wait();
            waited = true;
          }
          tma_load_2d_to<true>(st + C::kStageA, &maps.b, fb, k * 64, tr.b_row + b_half, pol_x);
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer (leader only) ------------------------------
    if (rank == 0 && elect_one_sync()) {
      constexpr uint32_t idesc = make_idesc_bf16(256, BN);
      uint32_t it = 0;
      for (int j = 0; j < sl.nseg && !*p.abort_flag; ++j) {
        int t, kb, ke;
        sl.seg(j, t, kb, ke);
        const int acc = j & 1;
        const uint32_t use = j >> 1;
        if (!mbar_wait_cluster(&p.tempty[acc], (use & 1) ^ 1, p.abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * acc_stride<BN>();
        bool ok = true;
        for (int k = kb; k < ke; ++k, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait_cluster(&p.full[s], (it / C::kStages) & 1, p.abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(p.stages + s * C::kStage);
          const uint64_t ad = make_sw128_desc(sa);
          const uint64_t bd = make_sw128_desc(sa + C::kStageA);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_pair_bf16(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc,
                             (k > kb || kk > 0) ? 1u : 0u);
          tc_commit_pair_both(&p.empty[s]);
        }
        if (!ok) break;
        tc_commit_pair_both(&p.tfull[acc]);
      }
      tc_commit_pair(p.drain);
      mbar_wait(p.drain, 0, p.abort_flag);
    }
  } else {
    // ------------------------------ epilogue (both CTAs) ------------------------------
    const uint32_t tempty0 = mapa_shared(smem_u32(p.tempty), 0);  // the leader's
    run_epilogue<BN, C::kXchgBufs>(
        a, p, tmem_base, xchg, stage_out, warp, lane, sl.nseg,
        [&](int j, int& t, int& kb, int& ke, TileRef& tr) {
          sl.seg(j, t, kb, ke);
          tr = pair_tile<BN>(a, t, rank);
        },
        // this CTA's slots: 0 its part of the pair's first tile, 1 of its last
        [&](int t) { return a.ws + ((size_t)blockIdx.x * 2 + (t == sl.tf ? 0 : 1)) * (BN * 128); },
        [&](int acc) {
          if (rank == 0)
            mbar_arrive(&p.tempty[acc]);
          else
            mbar_arrive_cluster(tempty0 + acc * 8);
        });
  }

  __syncthreads();
  if (*p.abort_flag && threadIdx.x == 0) record_timeout(a.status, kDiagGemm, 4, (uint32_t)rank);
  // neither CTA leaves (or frees its TMEM) while the leader's products may
  // still read the peer's shared memory or write its TMEM, or the peer's
  // copies and arrives may still reach the leader's barriers
  tc_fence_before();
  cluster_barrier();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

// Split-K fixup of the pair GEMM: block = (pair tile, CTA rank, 16-token
// chunk), 128 threads = the rows of that CTA's half.  Sums, in pair order,
// the partial slots of the pairs whose unit ranges overlap the tile (slots of
// CTA 2 c + rank of pair c), then applies the GEMM's epilogue.  Tiles owned
// whole by one pair were finished by it.
template <int BN>
__global__ void __launch_bounds__(128) splitk_fixup_pair_kernel(const GemmArgs a) {
  __shared__ float xchg[128 * 17];
  pdl_wait();
  constexpr int chunks = BN / 16;
  const int c = blockIdx.x % chunks;
  const int half = blockIdx.x / chunks;
  const int rank = half & 1, tp = half >> 1;
  const int tiles = (a.n_tiles / 2) * a.m_tiles;
  Sched sc;
  sc.G = a.grid / 2;
  sc.KT = a.k_tiles;
  sc.U = (unsigned)tiles * a.k_tiles;
  const unsigned tu0 = (unsigned)tp * a.k_tiles;
  const int c_first = sc.owner(tu0), c_last = sc.owner(tu0 + a.k_tiles - 1);
  if (c_first == c_last) {  // whole tile: done by the GEMM
    pdl_trigger();
    return;
  }
  const int row = threadIdx.x;
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = 0.f;
#pragma unroll 1
  for (int cc = c_first; cc <= c_last; cc += 2) {
    float buf[2][16];
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (cc + x <= c_last) {
        const int w = ((unsigned)tp == sc.start(cc + x) / sc.KT) ? 0 : 1;
        const size_t slot = (size_t)(2 * (cc + x) + rank) * 2 + w;
        const float* src = a.ws + slot * (BN * 128) + (size_t)(c * 16) * 128 + row;
#pragma unroll
        for (int i = 0; i < 16; ++i) buf[x][i] = __ldcg(src + (size_t)i * 128);
      }
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (cc + x <= c_last)
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += buf[x][i];
  }
  int np, mt;
  pair_tile_coords(tp, a.m_tiles, a.n_tiles / 2, np, mt);
  epilogue_chunk<BN>(a, v, row, 2 * np + rank, mt * BN + c * 16, xchg, a.M, 0, false);
  pdl_trigger();
}

}  // namespace dinfer
