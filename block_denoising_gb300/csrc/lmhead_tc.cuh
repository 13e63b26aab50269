// Fused LM head + per-position online softmax + threshold commit (bf16, sm_103a).
//
// The method needs, per block position, only the top-1 token and its softmax
// probability, so the [rows x vocab] logits are never written: each CTA
// streams a contiguous vocabulary slice of the LM-head weight through the
// tcgen05 pipeline (weight rows = MMA M, block tokens = MMA N), keeps a
// running (max, argmax, sum of 2^(t - max)) per token in shared memory, and
// writes one partial per token.  The CTA that finishes last merges the
// partials in CTA order and applies the threshold commit to the ids / mask in
// place (see decode.cuh).  A debug pointer optionally also stores the fp32
// logits for parity tests.
#pragma once
#include "decode.cuh"
#include "gemm_tc.cuh"

namespace dinfer {

struct LmArgs {
  int V, mask_id;
  float scale;        // logit scale
  float* logits;      // optional [M, V] fp32
  DecodeArgs dec;
};

template <int BN>
struct LmCfg {
  static constexpr int kMaxM = 1024;
  // one stage fewer than a plain GEMM at 64 tokens: the running softmax
  // states take the room
  static constexpr int kStages = BN == 64 ? 8 : gemm_default_stages<BN>();
  static constexpr int kSmem = GemmCfg<BN, kStages>::kSmem + kMaxM * 12 + 4 * 16 * 12 + 128;
  static_assert(kSmem <= 232448, "LM-head shared memory above 227 KB");
};

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    lmhead_tc_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs ga, const LmArgs la) {
  constexpr int ST = LmCfg<BN>::kStages;
  using C = GemmCfg<BN, ST>;
  extern __shared__ uint8_t smem_raw[];
  float* xchg;
  uint32_t* tmem_slot;
  volatile int* misc;
  const Pipe p = setup_pipe<BN, ST>(smem_raw, xchg, tmem_slot, misc);
  volatile int* last_flag = misc + 1;
  // running softmax state per token, after the GEMM's shared memory
  uint8_t* extra = reinterpret_cast<uint8_t*>(const_cast<int*>(misc + 24));
  float* st_m = reinterpret_cast<float*>(extra);
  float* st_s = st_m + LmCfg<BN>::kMaxM;
  int* st_a = reinterpret_cast<int*>(st_s + LmCfg<BN>::kMaxM);
  float* w_m = reinterpret_cast<float*>(st_a + LmCfg<BN>::kMaxM);  // [4][16]
  float* w_s = w_m + 64;
  int* w_a = reinterpret_cast<int*>(w_s + 64);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int M = ga.M;

  Sched sc;
  sc.G = gridDim.x;
  sc.KT = 1;
  sc.U = (unsigned)(ga.m_tiles * ga.n_tiles);
  SegList sl;
  sl.init(0, ga.k_tiles, blockIdx.x, ga.m_tiles * ga.n_tiles, gridDim.x);

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.b);
    prefetch_tmap(&maps.a[0]);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  for (int m = threadIdx.x; m < M; m += blockDim.x) {
    st_m[m] = -INFINITY;
    st_s[m] = 0.f;
    st_a[m] = 0x7fffffff;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == 0) {
    if (elect_one_sync()) run_producer<BN, ST>(maps, ga, sl, p, ga.m_tiles);
  } else if (warp == 1) {
    if (elect_one_sync()) run_mma<BN, ST>(sl, p, tmem_base);
  } else {
    pdl_wait();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int ep_tid = threadIdx.x - 64;
    const float kLog2e = 1.4426950408889634f;
    const float sl2 = la.scale * kLog2e;
    for (int j = 0; j < sl.nseg; ++j) {
      const int t = sl.tf + j * sl.stride;
      const int nt = t / ga.m_tiles, mt = t % ga.m_tiles;
      const int acc = j & 1;
      if (!mbar_wait(&p.tfull[acc], (j >> 1) & 1, p.abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * acc_stride<BN>();
      const int n = nt * 128 + row;
      const bool valid = (n < la.V) && (n != la.mask_id);
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tbase + c * 16, v);
        const int m0 = mt * BN + c * 16;
        if (la.logits != nullptr && n < la.V) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (m0 + i < M) la.logits[(size_t)(m0 + i) * la.V + n] = valid ? v[i] * la.scale : -INFINITY;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float tv = valid ? v[i] * sl2 : -INFINITY;
          const float wm = warp_max(tv);
          const float e = (valid && wm != -INFINITY) ? exp2f(tv - wm) : 0.f;
          const float ws = warp_sum(e);
          const unsigned hit = __ballot_sync(0xffffffffu, valid && tv == wm);
          if (lane == i) {
            w_m[q * 16 + i] = wm;
            w_s[q * 16 + i] = ws;
            w_a[q * 16 + i] = hit ? (nt * 128 + q * 32 + __ffs(hit) - 1) : 0x7fffffff;
          }
        }
        named_bar_sync(1, 128);
        if (ep_tid < 16 && m0 + ep_tid < M) {
          const int m = m0 + ep_tid;
          SoftmaxState s{st_m[m], st_s[m], st_a[m]};
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            SoftmaxState x{w_m[qq * 16 + ep_tid], w_s[qq * 16 + ep_tid], w_a[qq * 16 + ep_tid]};
            s = sm_merge(s, x);
          }
          st_m[m] = s.m;
          st_s[m] = s.s;
          st_a[m] = s.a;
        }
        named_bar_sync(1, 128);
      }
      tc_fence_before();
      mbar_arrive(&p.tempty[acc]);
    }
    // publish this CTA's partial for every token, then take a ticket
    SoftmaxState* part = la.dec.partials + (size_t)blockIdx.x * M;
    for (int m = ep_tid; m < M; m += 128) {
      part[m].m = st_m[m];
      part[m].s = st_s[m];
      part[m].a = st_a[m];
    }
    __threadfence();
    named_bar_sync(1, 128);
    if (ep_tid == 0) {
      const int prev = atomicAdd(la.dec.ticket, 1);
      const int is_last = (prev == (int)gridDim.x - 1);
      if (is_last) *la.dec.ticket = 0;
      *last_flag = is_last;
    }
    named_bar_sync(1, 128);
    if (*last_flag) {
      __threadfence();
      // reuse the running-state arrays as scratch for tokens / confidences
      finalize_and_commit(la.dec, ep_tid, st_a, st_s, 1);
    }
  }

  __syncthreads();
  if (*p.abort_flag && threadIdx.x == 0) record_timeout(ga.status, kDiagLmHead, 0, 0);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace dinfer
