// Persistent layer chain for a cached denoising iteration (block rows <= 64,
// dense SwiGLU FFN): one launch per layer runs
//
//   O projection + residual -> FFN RMSNorm -> gate/up + SwiGLU ->
//   down projection + residual -> next RMSNorm -> next layer's QKV (+ RoPE,
//   dual-cache write of the block's K/V)
//
// between two attention launches, so the weight stream of a layer does not
// stop at the five kernel boundaries of the per-operation path.
//
// One CTA per SM, the warp roles of the weight-streaming GEMM (warp 0 TMA,
// warp 1 MMA, warps 2-5 epilogue) and its shared-memory ring and TMEM
// accumulators.  Each CTA owns a fixed list of segments (tile, k-range) of
// the four GEMMs, in phase order; every GEMM is split stream-K over the grid
// (the same number of weight bytes per SM in every phase).  A tile shared by
// several CTAs leaves fp32 partials: gate/up and QKV tiles are finished by
// their last contributor (a ticket per tile), which sums the partials in CTA
// order and applies the epilogue (SwiGLU; RoPE and the cache write); the
// residual partials of O and down are summed by the row norms.
//
// The weight tile of a ring stage never depends on another CTA, so the
// producer requests it as soon as the stage is free -- also across phase
// boundaries -- and issues the stage's token tile once its producer is done:
//   O       the attention output (programmatic dependency on the attention launch);
//   gate/up the FFN norm of every block row (counter);
//   down    k-step c needs gate/up tile c (one ready flag per tile);
//   QKV     the next norm of every block row (counter).
// The norms run on the epilogue warps of CTA r for row r, once every CTA has
// written its residual partials (counter); they sum the partials in CTA order
// (as the split-K fixup does), so results do not depend on timing.
//
// All CTAs must be resident together: the grid is at most one CTA per SM and
// a CTA needs most of an SM's shared memory; the kernels around it never wait
// for it.  Every wait is bounded; a wait that runs out sets the CTA's abort
// flag and the device status, and the CTA winds down.  The last CTA to leave
// resets the counters for the next launch.
#pragma once
#include "gemm_tc.cuh"

namespace dinfer {

enum ChainPhase : int { CH_O = 0, CH_GU = 1, CH_DN = 2, CH_QKV = 3, CH_PHASES = 4 };
// synchronisation words (uint32, zero between launches)
enum ChainSync : int { SY_O = 0, SY_N1 = 1, SY_DN = 2, SY_N2 = 3, SY_EXIT = 4, SY_GU = 32 };
constexpr int kChainMaxSegs = 64;
constexpr int kChainMaxGuTiles = 1024;
constexpr int kChainMaxQkvTiles = 1024;
constexpr int SY_TICKET_GU = SY_GU + kChainMaxGuTiles;             // tile tickets of gate/up
constexpr int SY_TICKET_QKV = SY_TICKET_GU + kChainMaxGuTiles;     // and of QKV
constexpr int kChainSyncWords = SY_TICKET_QKV + kChainMaxQkvTiles;
constexpr uint32_t kDiagChain = 4;
// weight stages requested into L2 beyond the ring while a phase waits for its
// token tiles (0: none).  Measured on the LLaDA-8B iteration, prefetching
// delays the row norms on the critical path more than it saves.
constexpr uint32_t kChainL2Ahead = 0;

struct ChainArgs {
  GemmArgs g[CH_PHASES];       // operands and epilogues of the four GEMMs (BN 64, one token tile);
                               // grid = CTAs sharing the phase's stream-K units (<= units);
                               // ws = the phase's partial slots [grid][2][64 * 128]
  int cta0[CH_PHASES];         // first CTA of each phase's grid (the phase uses g[ph].grid CTAs)
  int has_qkv;                 // 0 after the last layer
  int M, d;
  float eps;
  const __nv_bfloat16* g_ffn;  // FFN norm gain of this layer
  const __nv_bfloat16* g_next; // attention norm gain of the next layer, or the final norm gain
  float* h;                    // residual stream [M, d] fp32
  __nv_bfloat16* xn;           // normed activations [M, d]
  uint32_t* sync;              // kChainSyncWords words
  DevState* status;
};

struct ChainMaps {
  GemmMaps m[CH_PHASES];
};

struct ChainSeg {
  int ph, t, kb, ke, slot;  // slot: partial slot of a residual segment (0 first tile, 1 last)
};

using ChainCfg = GemmCfg<64>;
constexpr int kChainSmem = ChainCfg::kSmem + kChainMaxSegs * (int)sizeof(ChainSeg) + 256 + kChainMaxGuTiles / 8 +
                           2 * ChainCfg::kStages * 4 + CH_PHASES * 48 + 64;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ uint4 ld_relaxed_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
// Pause between polls of a word other CTAs write: a tight loop of loads on
// one L2 line from many SMs slows every stream that line's slice serves.
constexpr unsigned kChainPollNs = 400;
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// order this thread's generic-proxy view of global memory with its later
// tensor-memory-access (async proxy) copies, and the reverse
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ Sched chain_sched(const GemmArgs& g) {
  Sched sc;
  sc.G = g.grid;
  sc.KT = g.k_tiles;
  sc.U = (unsigned)g.n_tiles * g.k_tiles;
  return sc;
}

// The segments of this CTA, phase by phase; begin[ph] .. begin[ph + 1].
__device__ __forceinline__ int chain_segments(const ChainArgs& a, ChainSeg* seg, int* begin) {
  int n = 0;
  for (int ph = 0; ph < CH_PHASES; ++ph) {
    begin[ph] = n;
    if (ph == CH_QKV && !a.has_qkv) continue;
    const GemmArgs& g = a.g[ph];
    // CTAs cta0 .. cta0 + grid - 1 take part; stream-K phases use at most one
    // CTA per unit, so every CTA in a tile's contributor range leaves a partial
    const int b = (int)blockIdx.x - a.cta0[ph];
    if (b < 0 || b >= g.grid) continue;
    SegList sl;
    if (g.stream_k) {
      const Sched sc = chain_sched(g);
      sl.init(1, g.k_tiles, sc.start(b), sc.start(b + 1));
    } else {
      sl.init(0, g.k_tiles, b, g.n_tiles, g.grid);  // whole tiles, round-robin
    }
    for (int j = 0; j < sl.nseg && n < kChainMaxSegs; ++j) {
      ChainSeg s;
      s.ph = ph;
      sl.seg(j, s.t, s.kb, s.ke);
      s.slot = (s.t == sl.tf) ? 0 : 1;
      seg[n++] = s;
    }
  }
  begin[CH_PHASES] = n;
  return n;
}

// Kernel-parameter structs are read at compile-time offsets (constant bank);
// a run-time phase index would turn every field access into a generic load of
// parameter memory, so per-phase code is dispatched by switch.
#define CHAIN_PHASE_SWITCH(ph, STMT)                         \
  switch (ph) {                                              \
    case CH_O: { constexpr int PH = CH_O; STMT; } break;     \
    case CH_GU: { constexpr int PH = CH_GU; STMT; } break;   \
    case CH_DN: { constexpr int PH = CH_DN; STMT; } break;   \
    default: { constexpr int PH = CH_QKV; STMT; } break;     \
  }

// What the producer loads for a stage of each phase: the tensor maps and the
// tile layout, gathered once so that the per-stage path is one small block.
struct ChainLoad {
  const CUtensorMap* a[3];  // weight maps (pair: gate, up; three: q, k, v)
  const CUtensorMap* b;     // token map
  int mode;                 // AMode
  int per;                  // A_THREE: 128-row tiles per map
};

__device__ __forceinline__ void chain_load_a(const ChainLoad& L, uint8_t* stage, uint64_t* bar, int t, int k,
                                             uint64_t pol) {
  const int kx = k * 64;
  if (L.mode == A_PAIR) {
    tma_load_2d(stage, L.a[0], bar, kx, t * 64, pol);
    tma_load_2d(stage + 64 * 128, L.a[1], bar, kx, t * 64, pol);
  } else if (L.mode == A_THREE) {
    const int m = t / L.per;
    tma_load_2d(stage, L.a[m], bar, kx, (t - m * L.per) * 128, pol);
  } else {
    tma_load_2d(stage, L.a[0], bar, kx, t * 128, pol);
  }
}

__device__ __forceinline__ void chain_prefetch_a(const ChainLoad& L, int t, int k) {
  const int kx = k * 64;
  if (L.mode == A_PAIR) {
    tma_prefetch_2d(L.a[0], kx, t * 64);
    tma_prefetch_2d(L.a[1], kx, t * 64);
  } else if (L.mode == A_THREE) {
    const int m = t / L.per;
    tma_prefetch_2d(L.a[m], kx, (t - m * L.per) * 128);
  } else {
    tma_prefetch_2d(L.a[0], kx, t * 128);
  }
}


// TMA producer (one thread): weight tiles run ahead into free stages, token
// tiles follow once their data is ready.
// Gate/up tiles known ready, one bit each; flags are polled 32 at a time
// (one 128-byte line, then one acquire fence), so a down segment costs about
// one round trip per 32 k-steps rather than one per k-step.
__device__ __forceinline__ bool chain_gu_ready(const ChainArgs& a, uint32_t* bits, int k) {
  uint32_t& w = bits[k >> 5];
  if ((w >> (k & 31)) & 1u) return true;
  const int k0 = k & ~31;
  uint32_t got = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 v = ld_relaxed_v4(a.sync + SY_GU + k0 + 4 * i);
    got |= ((v.x != 0u) ? 1u : 0u) << (4 * i);
    got |= ((v.y != 0u) ? 1u : 0u) << (4 * i + 1);
    got |= ((v.z != 0u) ? 1u : 0u) << (4 * i + 2);
    got |= ((v.w != 0u) ? 1u : 0u) << (4 * i + 3);
  }
  if (!got) return false;
  fence_acquire_gpu();
  fence_proxy_async_global();
  w |= got;
  return (w >> (k & 31)) & 1u;
}

// The k-steps of one phase's segments, in order.
struct ChainStages {
  const ChainSeg* seg;
  int j, j1, t, k, ke;
  __device__ __forceinline__ ChainStages(const ChainSeg* s, int j0, int j_end) : seg(s), j(j0), j1(j_end) { open(); }
  __device__ __forceinline__ void open() {
    if (j < j1) {
      const ChainSeg g = seg[j];
      t = g.t; k = g.kb; ke = g.ke;
    }
  }
  __device__ __forceinline__ bool more() const { return j < j1; }
  __device__ __forceinline__ void next() {
    if (++k == ke) {
      ++j;
      open();
    }
  }
};

// TMA producer (one thread), the loop of a plain GEMM producer per phase: a
// free stage is awaited in its barrier (the thread sleeps), then the weight
// and token tiles are issued together.  At the start of a phase whose token
// tiles depend on other CTAs, the phase's first weight tiles are issued into
// the free stages and the ones after them requested into L2, so HBM keeps
// streaming while the dependency completes; down k-steps wait for their
// gate/up tile individually.
__device__ __forceinline__ void chain_producer(const ChainLoad* plan, const ChainArgs& a, const ChainSeg* seg,
                                               const int* begin, const Pipe& p, uint32_t* gu_bits) {
  using C = ChainCfg;
  const uint64_t pol_w = l2_policy_evict_first();
  const uint64_t pol_x = l2_policy_evict_last();
  uint32_t it = 0;  // ring position
  bool ok = true;
  // Everything another kernel writes -- the attention output and this
  // grid's counters, which the previous layer's chain resets at its end --
  // is read after the dependency wait (the kernel may start before the
  // attention, and with it the previous chain, has completed).
  pdl_wait();
  // bounded poll of a dependency; false when the wait gave up
  auto wait_until = [&](auto cond, uint32_t site) -> bool {
    const long long t0 = clock64();
    while (!cond()) {
      if (*p.abort_flag) return false;
      if (clock64() - t0 > kWaitCycles) {
        *p.abort_flag = 1;
        record_timeout(a.status, kDiagChain, site, it);
        return false;
      }
      __nanosleep(kChainPollNs);
    }
    return true;
  };
  for (int ph = 0; ph < CH_PHASES && ok; ++ph) {
    if (begin[ph] == begin[ph + 1]) continue;
    const ChainLoad& L = plan[ph];
    // is the token tile of k-step k of this phase loadable?
    auto ready = [&](int k) -> bool {
      if (ph == CH_GU) return ld_acquire_u32(a.sync + SY_N1) >= (uint32_t)a.M;
      if (ph == CH_QKV) return ld_acquire_u32(a.sync + SY_N2) >= (uint32_t)a.M;
      if (ph == CH_DN) return chain_gu_ready(a, gu_bits, k);
      return true;
    };
    auto load_b = [&](int s, int k) {
      tma_load_2d(p.stages + s * C::kStage + C::kStageA, L.b, &p.full[s], k * 64, 0, pol_x);
    };
    ChainStages st(seg, begin[ph], begin[ph + 1]);
    bool gate = ph == CH_O || ready(st.k);
    if (!gate) {
      // the phase waits for other CTAs: its first weight tiles go into the
      // free stages and the next ones into L2 while the dependency completes
      ChainStages pre = st;
      uint32_t n = 0;
      for (; n < (uint32_t)C::kStages && pre.more(); ++n, pre.next()) {
        const int s = (it + n) % C::kStages;
        if (!mbar_wait(&p.empty[s], (((it + n) / C::kStages) & 1) ^ 1, p.abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(&p.full[s], C::kStage);
        chain_load_a(L, p.stages + s * C::kStage, &p.full[s], pre.t, pre.k, pol_w);
      }
      ChainStages l2 = pre;
      for (uint32_t m = 0; m < kChainL2Ahead && l2.more() && ok; ++m, l2.next()) chain_prefetch_a(L, l2.t, l2.k);
      // their token tiles, in order, as each becomes loadable
      for (uint32_t i = 0; i < n; ++i, ++it, st.next()) {
        const int s = it % C::kStages, kk = st.k;
        if (ok && !wait_until([&]() { return ready(kk); }, 4u + ph)) ok = false;
        if (ok) fence_proxy_async_global();
        load_b(s, kk);  // also when winding down: the stage's weight tile is in flight
      }
      if (!ok) break;
    } else if (ph != CH_O) {
      fence_proxy_async_global();
    }
    for (; st.more() && ok; st.next(), ++it) {
      const int s = it % C::kStages, kk = st.k;
      if (!mbar_wait(&p.empty[s], ((it / C::kStages) & 1) ^ 1, p.abort_flag)) { ok = false; break; }
      mbar_arrive_expect_tx(&p.full[s], C::kStage);
      chain_load_a(L, p.stages + s * C::kStage, &p.full[s], st.t, kk, pol_w);
      if (ph == CH_DN && !chain_gu_ready(a, gu_bits, kk)) {
        if (!wait_until([&]() { return chain_gu_ready(a, gu_bits, kk); }, 8u)) ok = false;
      }
      load_b(s, kk);  // also when winding down: the stage's weight tile is in flight
      if (!ok) {
        ++it;
        break;
      }
    }
  }
  if (!ok) {
    // winding down: let the copies of the last stages land before the CTA's
    // shared memory is released (every issued stage got its token tile)
    const uint32_t lo = it > (uint32_t)C::kStages ? it - C::kStages : 0u;
    for (uint32_t i = lo; i < it; ++i) mbar_wait_drain(&p.full[i % C::kStages], (i / C::kStages) & 1);
  }
}

// MMA issue (one thread): the segments in order, accumulators alternating.
__device__ __forceinline__ void chain_mma(const ChainSeg* seg, int nseg, const Pipe& p, uint32_t tmem_base) {
  using C = ChainCfg;
  constexpr uint32_t idesc = make_idesc_bf16(128, 64);
  uint32_t it = 0;
  for (int j = 0; j < nseg && !*p.abort_flag; ++j) {
    const int acc = j & 1;
    const uint32_t use = j >> 1;
    if (!mbar_wait(&p.tempty[acc], (use & 1) ^ 1, p.abort_flag)) break;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * 64;
    bool ok = true;
    const int kb = seg[j].kb, ke = seg[j].ke;  // registers: re-read after each barrier otherwise
    for (int k = kb; k < ke; ++k, ++it) {
      const int s = it % C::kStages;
      if (!mbar_wait(&p.full[s], (it / C::kStages) & 1, p.abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sa = smem_u32(p.stages + s * C::kStage);
      const uint64_t ad = make_sw128_desc(sa);
      const uint64_t bd = make_sw128_desc(sa + C::kStageA);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc_mma_bf16(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, (k > kb || kk > 0) ? 1u : 0u);
      tc_commit(&p.empty[s]);
    }
    if (!ok) break;
    tc_commit(&p.tfull[acc]);
  }
  tc_commit(p.drain);
  mbar_wait_drain(p.drain, 0);
}

// Epilogue-thread 0 waits until *word >= target (bounded); the decision is
// shared through `flag` after the epilogue barrier.
__device__ __forceinline__ bool chain_wait_count(const uint32_t* word, uint32_t target, volatile int* flag,
                                                 const Pipe& p, int etid, DevState* status, uint32_t site) {
  if (etid == 0) {
    bool ok = !*p.abort_flag;
    const long long t0 = clock64();
    while (ok && ld_acquire_u32(word) < target) {
      __nanosleep(kChainPollNs);
      if (*p.abort_flag) ok = false;
      else if (clock64() - t0 > kWaitCycles) {
        *p.abort_flag = 1;
        record_timeout(status, kDiagChain, site, target);
        ok = false;
      }
    }
    *flag = ok ? 1 : 0;
  }
  named_bar_sync(1, 128);
  return *flag != 0;
}

// Contributors [c_first, c_last] of tile t of a stream-K phase (CTA order),
// and the partial slot of contributor cc (0: its first tile, 1: its last).
struct ChainContrib {
  Sched sc;
  int c_first, c_last;
  __device__ __forceinline__ ChainContrib(const GemmArgs& g, int t) : sc(chain_sched(g)) {
    const unsigned tu0 = (unsigned)t * g.k_tiles;
    c_first = sc.owner(tu0);
    c_last = sc.owner(tu0 + g.k_tiles - 1);
  }
  __device__ __forceinline__ const float* slot(const GemmArgs& g, int cc, int t) const {
    const int w = ((unsigned)t == sc.start(cc) / sc.KT) ? 0 : 1;
    return g.ws + ((size_t)cc * 2 + w) * (64 * 128);
  }
};

// x = h[row, f0 .. f0+15] plus the residual partials of the tile over those
// features (token-major slots [64 tokens][128 rows]), summed in CTA order; the
// loads of up to 4 contributors are in flight together.
__device__ __forceinline__ void chain_gather16(const ChainArgs& a, const GemmArgs& g, int row, int f0,
                                               float (&x)[16]) {
  const float4* h4 = reinterpret_cast<const float4*>(a.h + (size_t)row * a.d + f0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 t4 = h4[i];
    x[4 * i] = t4.x; x[4 * i + 1] = t4.y; x[4 * i + 2] = t4.z; x[4 * i + 3] = t4.w;
  }
  const int t = f0 / 128, fl = f0 - t * 128;
  const ChainContrib cb(g, t);
  if (cb.c_first == cb.c_last) return;  // a whole tile: its owner added it to h
  for (int c0 = cb.c_first; c0 <= cb.c_last; c0 += 4) {
    float4 buf[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (c0 + q <= cb.c_last) {
        const float4* sp = reinterpret_cast<const float4*>(cb.slot(g, c0 + q, t) + (size_t)row * 128 + fl);
#pragma unroll
        for (int i = 0; i < 4; ++i) buf[q][i] = __ldcg(sp + i);
      }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (c0 + q <= cb.c_last)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[4 * i] += buf[q][i].x;
          x[4 * i + 1] += buf[q][i].y;
          x[4 * i + 2] += buf[q][i].z;
          x[4 * i + 3] += buf[q][i].w;
        }
  }
}

// Row `row` of the block: h += residual partials (CTA order), then
// xn = bf16(RMSNorm(h) * g).  128 epilogue threads, 16 features per group;
// a thread's first two groups are gathered together (their loads in flight
// at once) and stay in registers for the second pass.
__device__ __forceinline__ void chain_norm_row(const ChainArgs& a, const GemmArgs& gp, int row,
                                               const __nv_bfloat16* g, int etid, float* red) {
  const int groups = a.d / 16;
  const int g0 = etid, g1 = etid + 128;
  float x0[16], x1[16];
  float ss = 0.f;
  {
    if (g0 < groups) chain_gather16(a, gp, row, g0 * 16, x0);
    if (g1 < groups) chain_gather16(a, gp, row, g1 * 16, x1);
    float4* h0 = reinterpret_cast<float4*>(a.h + (size_t)row * a.d + g0 * 16);
    float4* h1 = reinterpret_cast<float4*>(a.h + (size_t)row * a.d + g1 * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (g0 < groups) h0[i] = make_float4(x0[4 * i], x0[4 * i + 1], x0[4 * i + 2], x0[4 * i + 3]);
      if (g1 < groups) h1[i] = make_float4(x1[4 * i], x1[4 * i + 1], x1[4 * i + 2], x1[4 * i + 3]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (g0 < groups) ss = fmaf(x0[i], x0[i], ss);
      if (g1 < groups) ss = fmaf(x1[i], x1[i], ss);
    }
  }
  for (int gi = etid + 256; gi < groups; gi += 128) {  // d_model above 4096
    float x[16];
    chain_gather16(a, gp, row, gi * 16, x);
    float4* ho = reinterpret_cast<float4*>(a.h + (size_t)row * a.d + gi * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) ho[i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
#pragma unroll
    for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
  }
  ss = warp_sum(ss);
  if ((etid & 31) == 0) red[etid >> 5] = ss;
  named_bar_sync(1, 128);
  const float tot = (red[0] + red[1]) + (red[2] + red[3]);
  const float inv = rsqrtf(tot / (float)a.d + a.eps);
  __nv_bfloat16* out = a.xn + (size_t)row * a.d;
  if (g0 < groups) norm_store16(x0, inv, g, g0 * 16, out);
  if (g1 < groups) norm_store16(x1, inv, g, g1 * 16, out);
  for (int gi = etid + 256; gi < groups; gi += 128) {
    float x[16];
    const float4* h4 = reinterpret_cast<const float4*>(a.h + (size_t)row * a.d + gi * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 t4 = h4[i];
      x[4 * i] = t4.x; x[4 * i + 1] = t4.y; x[4 * i + 2] = t4.z; x[4 * i + 3] = t4.w;
    }
    norm_store16(x, inv, g, gi * 16, out);
  }
  named_bar_sync(1, 128);  // red is reused by the next norm
}

// v = chunk c (tokens 16 c .. 16 c + 15) of output row `row` of tile t, summed
// over the tile's row-major partial slots ([128 rows][64 tokens]) in CTA order.
__device__ __forceinline__ void chain_sum_slots(const GemmArgs& g, int t, int row, int c, float (&v)[16]) {
  const ChainContrib cb(g, t);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = 0.f;
  for (int c0 = cb.c_first; c0 <= cb.c_last; c0 += 4) {
    float4 buf[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (c0 + q <= cb.c_last) {
        const float4* sp = reinterpret_cast<const float4*>(cb.slot(g, c0 + q, t) + (size_t)row * 64 + c * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) buf[q][i] = __ldcg(sp + i);
      }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (c0 + q <= cb.c_last)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[4 * i] += buf[q][i].x;
          v[4 * i + 1] += buf[q][i].y;
          v[4 * i + 2] += buf[q][i].z;
          v[4 * i + 3] += buf[q][i].w;
        }
  }
}

// Epilogue context of the four phases.
struct ChainEpi {
  const ChainArgs& a;
  const Pipe& p;
  const ChainSeg* seg;
  const int* begin;
  uint32_t tmem_base;
  float* xchg;
  volatile int* ep_flag;
  float* red;
  int etid, q, row, base_pos;
};

// The epilogue of one phase: its segments, then (residual phases) the row
// norm.  Decisions are taken by epilogue thread 0 and shared through ep_flag
// after the epilogue barrier, so the 128 threads branch together.  Returns
// false when a wait gave up.
template <int PH>
__device__ __forceinline__ bool chain_epilogue_phase(const ChainEpi& e, int& j) {
  const ChainArgs& a = e.a;
  const Pipe& p = e.p;
  const GemmArgs& g = a.g[PH];
  constexpr bool resid = PH == CH_O || PH == CH_DN;
  const int etid = e.etid, row = e.row;
  volatile int* ep_flag = e.ep_flag;
  for (; j < e.begin[PH + 1]; ++j) {
    const ChainSeg s = e.seg[j];
    const int acc = j & 1;
    const uint32_t use = j >> 1;
    if (etid == 0) ep_flag[j & 1] = (mbar_wait(&p.tfull[acc], use & 1, p.abort_flag) && !*p.abort_flag) ? 1 : 0;
    named_bar_sync(1, 128);
    if (!ep_flag[j & 1]) return false;
    tc_fence_after();
    const uint32_t tbase = e.tmem_base + ((uint32_t)(e.q * 32) << 16) + acc * 64;
    const bool whole = s.kb == 0 && s.ke == g.k_tiles;
    bool finish = whole;
    if (!whole) {
      float* base = g.ws + ((size_t)(blockIdx.x - a.cta0[PH]) * 2 + s.slot) * (64 * 128);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[16];
        tmem_ld16(tbase + c * 16, v);
        if (resid) {  // token-major [64 tokens][128 rows]: the row norms read 16 features at a time
#pragma unroll
          for (int i = 0; i < 16; ++i) base[(size_t)(c * 16 + i) * 128 + row] = v[i];
        } else {      // row-major [128 rows][64 tokens]: the finisher reads 16 tokens at a time
          float4* sl = reinterpret_cast<float4*>(base + (size_t)row * 64 + c * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) sl[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&p.tempty[acc]);
      if (!resid) {
        // the last contributor of the tile finishes it
        named_bar_sync(1, 128);
        if (etid == 0) {
          __threadfence();
          const ChainContrib cb(g, s.t);
          uint32_t* ticket = a.sync + (PH == CH_GU ? SY_TICKET_GU : SY_TICKET_QKV) + s.t;
          const bool last = atomicAdd(ticket, 1u) + 1u == (uint32_t)(cb.c_last - cb.c_first + 1);
          if (last) __threadfence();
          ep_flag[2 + (j & 1)] = last ? 1 : 0;
        }
        named_bar_sync(1, 128);
        finish = ep_flag[2 + (j & 1)] != 0;
      }
    }
    if (finish) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[16];
        if (whole) tmem_ld16(tbase + c * 16, v);
        else chain_sum_slots(g, s.t, row, c, v);
        // whole residual tile (h += acc), gate/up (act = SiLU(gate) * up),
        // or QKV (RoPE factors loaded with the chunk)
        epilogue_chunk<64>(g, v, row, s.t, c * 16, e.xchg, g.M, 0, nullptr, e.base_pos);
      }
      if (whole) {
        tc_fence_before();
        mbar_arrive(&p.tempty[acc]);
      }
      if (PH == CH_GU) {
        // act columns [64 t, 64 t + 64) are complete: down k-step t may load them
        named_bar_sync(1, 128);
        if (etid == 0) {
          __threadfence();
          fence_proxy_async_global();
          st_release_u32(a.sync + SY_GU + s.t, 1u);
        }
      }
    }
  }
  if (resid) {
    // this CTA's residual partials are written; row blockIdx.x is normed
    // once every CTA's are
    named_bar_sync(1, 128);
    if (etid == 0) {
      __threadfence();  // the partials of all 128 threads (ordered by the barrier)
      red_release_add_u32(a.sync + (PH == CH_O ? SY_O : SY_DN), 1u);
    }
    if ((int)blockIdx.x < a.M) {
      if (!chain_wait_count(a.sync + (PH == CH_O ? SY_O : SY_DN), gridDim.x, ep_flag, p, etid, a.status,
                            PH == CH_O ? 2u : 3u))
        return false;
      chain_norm_row(a, g, blockIdx.x, PH == CH_O ? a.g_ffn : a.g_next, etid, e.red);
      if (etid == 0) {
        fence_proxy_async_global();
        __threadfence();
        red_release_add_u32(a.sync + (PH == CH_O ? SY_N1 : SY_N2), 1u);
      }
    }
  }
  return true;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    layer_chain_kernel(const __grid_constant__ ChainMaps maps, const __grid_constant__ ChainArgs a) {
  using C = ChainCfg;
  extern __shared__ uint8_t smem_raw[];
  float* xchg;
  uint32_t* tmem_slot;
  volatile int* misc;
  const Pipe p = setup_pipe<64>(smem_raw, xchg, tmem_slot, misc);
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ChainSeg* seg = reinterpret_cast<ChainSeg*>(sm + C::kStages * C::kStage + C::kXchgFloats * 4 + 512);
  int* begin = reinterpret_cast<int*>(seg + kChainMaxSegs);       // [CH_PHASES + 1]
  volatile int* ep_flag = reinterpret_cast<volatile int*>(begin + CH_PHASES + 1);  // [4]
  float* red = reinterpret_cast<float*>(const_cast<int*>(ep_flag + 4));  // [4]
  uint32_t* gu_bits = reinterpret_cast<uint32_t*>(red + 4);                // [kChainMaxGuTiles / 32]
  ChainLoad* plan = reinterpret_cast<ChainLoad*>(                          // [CH_PHASES], 16-byte aligned
      (reinterpret_cast<uintptr_t>(gu_bits + kChainMaxGuTiles / 32) + 15) & ~uintptr_t(15));
  if (threadIdx.x == 0) {
    for (int ph = 0; ph < CH_PHASES; ++ph) {
      CHAIN_PHASE_SWITCH(ph, {
        ChainLoad& L = plan[PH];
        L.a[0] = &maps.m[PH].a[0];
        L.a[1] = &maps.m[PH].a[1];
        L.a[2] = &maps.m[PH].a[2];
        L.b = &maps.m[PH].b;
        L.mode = a.g[PH].a_mode;
        L.per = a.g[PH].a_rows / 128 > 0 ? a.g[PH].a_rows / 128 : 1;
      })
    }
    chain_segments(a, seg, begin);
    for (int i = 0; i < kChainMaxGuTiles / 32; ++i) gu_bits[i] = 0u;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane == 0) {
    for (int ph = 0; ph < CH_PHASES; ++ph) {
      CHAIN_PHASE_SWITCH(ph, {
        prefetch_tmap(&maps.m[PH].a[0]);
        prefetch_tmap(&maps.m[PH].a[1]);
        prefetch_tmap(&maps.m[PH].a[2]);
        prefetch_tmap(&maps.m[PH].b);
      })
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nseg = begin[CH_PHASES];
  if (threadIdx.x == 0) pdl_trigger();  // the next attention may start on SMs this grid leaves

  if (warp == 0) {
    if (elect_one_sync()) chain_producer(plan, a, seg, begin, p, gu_bits);
  } else if (warp == 1) {
    if (elect_one_sync()) chain_mma(seg, nseg, p, tmem_base);
  } else {
    // ------------------------------ epilogue ------------------------------
    const int etid = threadIdx.x - 64;
    const int q = warp & 3;
    const int row = q * 32 + lane;  // output feature row inside the tile
    pdl_wait();
    const GemmArgs& gq = a.g[CH_QKV];
    const int base_pos = (a.has_qkv && gq.pos_from_state) ? gq.state->block_start : 0;
    int j = 0;  // segment counter = accumulator sequence
    ChainEpi e{a, p, seg, begin, tmem_base, xchg, ep_flag, red, etid, q, row, base_pos};
    bool ok = chain_epilogue_phase<CH_O>(e, j);
    ok = ok && chain_epilogue_phase<CH_GU>(e, j);
    ok = ok && chain_epilogue_phase<CH_DN>(e, j);
    ok = ok && chain_epilogue_phase<CH_QKV>(e, j);
    (void)ok;
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    // the last CTA out resets the counters for the next launch
    __threadfence();
    if (atomicAdd(a.sync + SY_EXIT, 1u) == gridDim.x - 1) {
      a.sync[SY_O] = 0;
      a.sync[SY_N1] = 0;
      a.sync[SY_DN] = 0;
      a.sync[SY_N2] = 0;
      for (int t = 0; t < a.g[CH_GU].n_tiles; ++t) {
        a.sync[SY_GU + t] = 0;
        a.sync[SY_TICKET_GU + t] = 0;
      }
      if (a.has_qkv)
        for (int t = 0; t < a.g[CH_QKV].n_tiles; ++t) a.sync[SY_TICKET_QKV + t] = 0;
      __threadfence();
      a.sync[SY_EXIT] = 0;
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace dinfer
