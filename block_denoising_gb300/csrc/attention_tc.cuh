// Bidirectional attention of query rows against the dual KV cache on the
// tcgen05 tensor cores (head_dim 128).
//
// Every query row attends over ALL L cached positions of its sequence (the
// prefix, the block slot just written with the block's fresh K/V, and the
// suffix) with no mask: o = softmax(q k^T / sqrt(128)) v.
//
// One CTA = 128 query rows x one head x one range of 128-key chunks,
// 320 threads:
//   warp 0     TMA: Q once, then K and V chunks (2-stage K and V rings with
//              their own barriers: a K stage is refilled as soon as S of its
//              chunk has been computed, a V stage once P V of its chunk has;
//              3-D tensor maps so that keys past L and rows past the sequence
//              read as zeros);
//   warp 1     TMEM allocation and the single-thread MMA issue:
//              S_j = Q K_j^T into one of two TMEM buffers, and for each key
//              half h, O_h += P_{j,h} V_{j,h} (64 keys; P from shared memory,
//              V the MN-major operand), in the order S_0, S_1, then per chunk
//              j: P V of both halves, S_{j+2};
//   warps 2-9  softmax, two threads per query row: warp w reads TMEM lane
//              quadrant w % 4 and takes key half h = (w - 2) / 4, keys
//              64 h .. 64 h + 63 of every chunk.  Each half is an online
//              softmax of its own (running max m_h, normaliser l_h and
//              accumulator O_h in TMEM), so the two warps that share an SM
//              sub-partition exchange nothing per chunk: tcgen05.ld of the
//              half row of S, log2-domain
//              softmax, P = bf16(2^(s - m_h)) written to the half's 64-key
//              slab of one of two shared-memory buffers in the
//              128-byte-swizzled K-major layout (so the softmax of chunk j
//              overlaps P_{j-1} V_{j-1}).  At the end the halves combine:
//              m = max(m_0, m_1), O = sum_h 2^(m_h - m) O_h, l likewise, and
//              each thread writes O / l for 64 output columns.  Warps whose 32
//              rows all lie past the sequence's rows (a 64-row block) only
//              keep the barrier counts.
// A running max is raised only when a chunk's max exceeds it by more than 8
// (P stays <= 2^8); then that half's O (in TMEM) and l are rescaled once.
// O / l is exact whatever max was used.
// Small grids (a batch-1 block) split the keys over up to 8 CTAs of a cluster;
// partials (m, l, O) are merged through distributed shared memory.
#pragma once
#include <cooperative_groups.h>

#include "common.cuh"

namespace dinfer {

struct AttnTcMaps {
  CUtensorMap q;  // [batch][rows_per_seq][d], box {64, 128, 1}
  CUtensorMap k;  // [batch][L][d], box {64, 128, 1}
  CUtensorMap v;
};

struct AttnTcArgs {
  __nv_bfloat16* o;  // [batch * rows_per_seq, d]
  int d, heads, L, rows_per_seq, q_tiles;
  int splits, chunks_per_split;
  float scale_log2;  // log2(e) / sqrt(128)
  DevState* status;
};

constexpr int kHd = 128;                // head dimension of the bf16 path
constexpr int kAtcThreads = 320;
constexpr int kAtcSoftmax = 256;        // softmax threads: 128 rows x 2 key halves
constexpr int kAtcKeys = 128;           // keys per chunk
constexpr int kAtcTile = 128 * 128 * 2; // one 128 x 128 bf16 operand (two 64-column swizzle slabs)
constexpr int kAtcSlab = 128 * 128;     // bytes of one 64-column slab of 128 rows
constexpr int kAtcStages = 2;           // K ring and V ring
constexpr int kAtcMaxSplits = 8;
// Q | K[2] | V[2] | P[2] | barriers | row exchange [2 halves][128]
constexpr int kAtcOffK = kAtcTile;
constexpr int kAtcOffV = kAtcOffK + kAtcStages * kAtcTile;
constexpr int kAtcOffP = kAtcOffV + kAtcStages * kAtcTile;
constexpr int kAtcOffBar = kAtcOffP + 2 * kAtcTile;
constexpr int kAtcOffX = kAtcOffBar + 256;
constexpr int kAtcSmem = 1024 + kAtcOffX + 2 * 128 * 4;
static_assert(kAtcSmem <= 232448, "attention shared memory above 227 KB");
constexpr int kAtcTmemCols = 512;       // S0 | S1 | O_0 | O_1
constexpr int kAtcColO = 256;
constexpr float kAtcLazy = 8.0f;        // log2 growth of the max tolerated before rescaling O

__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle:
// 64 MN elements (128 B) per row, one row per K index, 8-row groups 1024 B
// apart (stride byte offset), MN slabs of 64 elements `lbo` bytes apart
// (leading byte offset).
__device__ __forceinline__ uint64_t make_sw128_desc_mn(uint32_t smem_addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#define ATC_O4(x, b) "=r"(x[(b)]), "=r"(x[(b) + 1]), "=r"(x[(b) + 2]), "=r"(x[(b) + 3])
#define ATC_O32(x, b)                                                                                      \
  ATC_O4(x, b), ATC_O4(x, (b) + 4), ATC_O4(x, (b) + 8), ATC_O4(x, (b) + 12), ATC_O4(x, (b) + 16),          \
      ATC_O4(x, (b) + 20), ATC_O4(x, (b) + 24), ATC_O4(x, (b) + 28)
#define ATC_I4(x, b) "+r"(x[(b)]), "+r"(x[(b) + 1]), "+r"(x[(b) + 2]), "+r"(x[(b) + 3])
#define ATC_I32(x, b)                                                                                      \
  ATC_I4(x, b), ATC_I4(x, (b) + 4), ATC_I4(x, (b) + 8), ATC_I4(x, (b) + 12), ATC_I4(x, (b) + 16),          \
      ATC_I4(x, (b) + 20), ATC_I4(x, (b) + 24), ATC_I4(x, (b) + 28)

// 64 consecutive TMEM columns of this warp's 32 lanes, one wait for both
// loads.  The empty statement after the wait carries the second load's
// registers, so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&x)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];" : ATC_O32(x, 0) : "r"(taddr));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];" : ATC_O32(x, 32) : "r"(taddr + 32));
  asm volatile("tcgen05.wait::ld.sync.aligned;" : ATC_I32(x, 0)::"memory");
  asm volatile("" : ATC_I32(x, 32));
}

// 32 TMEM columns at each of two addresses of this warp's 32 lanes, one wait
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t (&x)[32], uint32_t tb, uint32_t (&y)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];" : ATC_O32(x, 0) : "r"(ta));
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];" : ATC_O32(y, 0) : "r"(tb));
  asm volatile("tcgen05.wait::ld.sync.aligned;" : ATC_I32(x, 0)::"memory");
  asm volatile("" : ATC_I32(y, 0));
}

// 2^x with the PTX approximate base-2 exponential (2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b2);
}

__global__ void __launch_bounds__(kAtcThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnTcMaps maps, const AttnTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kAtcOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;                  // [2]
  uint64_t* k_empty = k_full + kAtcStages;      // [2]
  uint64_t* v_full = k_empty + kAtcStages;      // [2]
  uint64_t* v_empty = v_full + kAtcStages;      // [2]
  uint64_t* s_full = v_empty + kAtcStages;      // [2]
  uint64_t* s_empty = s_full + 2;               // [2]
  uint64_t* p_full = s_empty + 2;               // [half][2]
  uint64_t* pv_done = p_full + 4;               // [half][2]
  uint64_t* drain = pv_done + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x % a.q_tiles;
  const int bi = blockIdx.x / a.q_tiles;
  const int head = blockIdx.y;
  const int split = blockIdx.z;
  const int row0 = qt * 128;
  const int q_valid = min(128, a.rows_per_seq - row0);
  const int n_chunks = (a.L + kAtcKeys - 1) / kAtcKeys;
  const int c_begin = split * a.chunks_per_split;
  const int nck = max(0, min(n_chunks, c_begin + a.chunks_per_split) - c_begin);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kAtcStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], kAtcSoftmax);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&p_full[s], kAtcSoftmax / 2);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.v);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kAtcTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the next kernel (the O projection) may become resident on the SMs this
  // grid leaves and request its first weight tiles; it reads this grid's
  // output only after griddepcontrol.wait (the whole grid complete)
  if (threadIdx.x == 0) pdl_trigger();
  // TMEM buffers at computed column offsets (not indexed arrays: local
  // memory would live in L2 on an SM whose memory is carved out as shared
  // memory): S buffer b at 128 b, O_h at 256 + 128 h
  const int hc = head * 128;  // first column of this head

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (elect_one_sync()) {
      // The cached keys / values outside the block slot do not depend on the
      // preceding kernel: request them into L2 before the dependency wait (the
      // block slot's lines are written by the preceding kernel; a prefetch only
      // warms L2, which stays coherent).
      for (int j = 0; j < nck; ++j) {
        const int key0 = (c_begin + j) * kAtcKeys;
        tma_prefetch_3d(&maps.k, hc, key0, bi);
        tma_prefetch_3d(&maps.k, hc + 64, key0, bi);
        tma_prefetch_3d(&maps.v, hc, key0, bi);
        tma_prefetch_3d(&maps.v, hc + 64, key0, bi);
      }
      pdl_wait();
      mbar_arrive_expect_tx(q_full, kAtcTile);
      tma_load_3d(sm, &maps.q, q_full, hc, row0, bi);
      tma_load_3d(sm + kAtcSlab, &maps.q, q_full, hc + 64, row0, bi);
      int k_issued = 0, v_issued = 0;
      // K of chunk j into stage j % 2 once S of chunk j - 2 completed
      auto load_k = [&](int j) -> bool {
        const int st = j % kAtcStages;
        if (!mbar_wait_diag(&k_empty[st], ((j / kAtcStages) & 1) ^ 1, abort_flag, a.status, kDiagAttn, 1, j))
          return false;
        k_issued = j + 1;
        mbar_arrive_expect_tx(&k_full[st], kAtcTile);
        uint8_t* kb = sm + kAtcOffK + st * kAtcTile;
        const int key0 = (c_begin + j) * kAtcKeys;
        tma_load_3d(kb, &maps.k, &k_full[st], hc, key0, bi);
        tma_load_3d(kb + kAtcSlab, &maps.k, &k_full[st], hc + 64, key0, bi);
        return true;
      };
      // V of chunk j into stage j % 2 once P V of chunk j - 2 completed
      auto load_v = [&](int j) -> bool {
        const int st = j % kAtcStages;
        if (!mbar_wait_diag(&v_empty[st], ((j / kAtcStages) & 1) ^ 1, abort_flag, a.status, kDiagAttn, 10, j))
          return false;
        v_issued = j + 1;
        mbar_arrive_expect_tx(&v_full[st], kAtcTile);
        uint8_t* vb = sm + kAtcOffV + st * kAtcTile;
        const int key0 = (c_begin + j) * kAtcKeys;
        tma_load_3d(vb, &maps.v, &v_full[st], hc, key0, bi);
        tma_load_3d(vb + kAtcSlab, &maps.v, &v_full[st], hc + 64, key0, bi);
        return true;
      };
      // K runs two chunks ahead of V: K_{j+2} waits for S_j, which is issued
      // before P_{j-1} V_{j-1} completes (what V_{j+1} waits for)
      bool go = true;
      for (int j = 0; j < min(nck, kAtcStages) && go; ++j) go = load_k(j);
      for (int j = 0; j < nck && go && !*abort_flag; ++j) {
        go = load_v(j);
        if (go && j + kAtcStages < nck) go = load_k(j + kAtcStages);
      }
      if (*abort_flag) {  // let the copies in flight land before the CTA exits
        mbar_wait_drain(q_full, 0);
        for (int j = max(0, k_issued - kAtcStages); j < k_issued; ++j)
          mbar_wait_drain(&k_full[j % kAtcStages], (j / kAtcStages) & 1);
        for (int j = max(0, v_issued - kAtcStages); j < v_issued; ++j)
          mbar_wait_drain(&v_full[j % kAtcStages], (j / kAtcStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (elect_one_sync()) {
      constexpr uint32_t idesc_s = make_idesc_bf16(128, 128);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, 128) | (1u << 16);  // B (V) MN-major
      const uint32_t q_addr = smem_u32(sm), p_addr = smem_u32(sm + kAtcOffP);
      // S_j = Q K_j^T into S buffer j & 1
      auto issue_s = [&](int j) -> bool {
        const int st = j % kAtcStages, sb = j & 1;
        if (!mbar_wait_diag(&k_full[st], (j / kAtcStages) & 1, abort_flag, a.status, kDiagAttn, 4, j)) return false;
        if (!mbar_wait_diag(&s_empty[sb], ((j >> 1) & 1) ^ 1, abort_flag, a.status, kDiagAttn, 5, j)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sm + kAtcOffK + st * kAtcTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // 16 head dims per step
          const uint64_t ad = make_sw128_desc(q_addr + (kk >> 2) * kAtcSlab + (kk & 3) * 32);
          const uint64_t bd = make_sw128_desc(k_addr + (kk >> 2) * kAtcSlab + (kk & 3) * 32);
          tc_mma_bf16(tmem + sb * 128, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[sb]);
        tc_commit(&k_empty[st]);
        return true;
      };
      // O_h += P_{j,h} V_{j,h}: keys 64 h .. 64 h + 63 of chunk j, P in slab h
      // of P buffer j & 1, V rows 64 h .. of V stage j % 2
      auto issue_pv = [&](int j, int h) -> bool {
        const int st = j % kAtcStages, pb = j & 1;
        if (!mbar_wait_diag(&p_full[h * 2 + pb], (j >> 1) & 1, abort_flag, a.status, kDiagAttn, 2, j)) return false;
        if (h == 0 && !mbar_wait_diag(&v_full[st], (j / kAtcStages) & 1, abort_flag, a.status, kDiagAttn, 11, j))
          return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sm + kAtcOffV + st * kAtcTile);
        const uint32_t pa = p_addr + pb * kAtcTile + h * kAtcSlab;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 16 keys per step
          const uint64_t ad = make_sw128_desc(pa + kk * 32);
          const uint64_t bd = make_sw128_desc_mn(v_addr + (h * 4 + kk) * 2048, kAtcSlab);
          tc_mma_bf16(tmem + kAtcColO + h * 128, ad, bd, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[h * 2 + pb]);
        if (h == 1) tc_commit(&v_empty[st]);  // both halves have read V_j
        return true;
      };
      bool ok = mbar_wait_diag(q_full, 0, abort_flag, a.status, kDiagAttn, 3, 0);
      for (int j = 0; j < min(nck, 2) && ok; ++j) ok = issue_s(j);
      for (int j = 0; j < nck && ok; ++j) {
        ok = issue_pv(j, 0) && issue_pv(j, 1);
        if (ok && j + 2 < nck) ok = issue_s(j + 2);
      }
      tc_commit(drain);
      mbar_wait_drain(drain, 0);
    }
  } else {
    // ------------------------------ softmax / output ------------------------------
    // Every wait's outcome is made warp-uniform: the TMEM accesses are
    // warp-collective.  The two warps of a quadrant meet only at the end, at
    // the same pair barriers whatever their waits returned (a failed wait
    // only skips work), so that a timed-out wait never leaves a warp blocked.
    const int q = warp & 3;
    const int hk = (warp - 2) >> 2;         // key half: keys 64 hk .. 64 hk + 63 of a chunk
    const int r = q * 32 + lane;            // query row inside the tile (TMEM lane)
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const bool live = q * 32 < q_valid;     // warp-uniform, the same for both halves
    const uint32_t t_oh = tmem + kAtcColO + hk * 128 + lane_off;  // this half's O
    const float sc = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nck; ++j) {
      const int sb = j & 1;
      if (ok && !__all_sync(0xffffffffu, mbar_wait_diag(&s_full[sb], (j >> 1) & 1, abort_flag, a.status,
                                                        kDiagAttn, 6, j)))
        ok = false;
      if (!live) {  // rows past the sequence: keep the counts only
        mbar_arrive(&s_empty[sb]);
        mbar_arrive(&p_full[hk * 2 + sb]);
        continue;
      }
      if (!ok) continue;
      uint32_t sv[64];
      tc_fence_after();
      tmem_ld64((tmem + sb * 128 + hk * 64) + lane_off, sv);
      tc_fence_before();
      mbar_arrive(&s_empty[sb]);
      const int nvalid = a.L - (c_begin + j) * kAtcKeys - hk * 64;  // <= 0: the upper half holds no key
      if (nvalid < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i >= nvalid) sv[i] = 0xff800000u;  // -inf: no key
      }
      float mx0 = __uint_as_float(sv[0]), mx1 = __uint_as_float(sv[1]);
      float mx2 = __uint_as_float(sv[2]), mx3 = __uint_as_float(sv[3]);
#pragma unroll
      for (int i = 4; i < 64; i += 4) {
        mx0 = fmaxf(mx0, __uint_as_float(sv[i]));
        mx1 = fmaxf(mx1, __uint_as_float(sv[i + 1]));
        mx2 = fmaxf(mx2, __uint_as_float(sv[i + 2]));
        mx3 = fmaxf(mx3, __uint_as_float(sv[i + 3]));
      }
      const float mj = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sc;  // -inf when the half holds no key
      if (m_used == -INFINITY) {
        // nothing accumulated yet (O_h and l hold zeros or nothing): start
        // from this chunk's max, -inf again if it holds no key either
        m_used = mj;
      } else {
        const bool grow = mj > m_used + kAtcLazy;
        if (__any_sync(0xffffffffu, grow)) {
          // rescale O_h: it must hold every product issued so far (P_{j-1} V_{j-1})
          if (!__all_sync(0xffffffffu, mbar_wait_diag(&pv_done[hk * 2 + ((j - 1) & 1)], ((j - 1) >> 1) & 1,
                                                      abort_flag, a.status, kDiagAttn, 7, j))) {
            ok = false;
            continue;
          }
          tc_fence_after();
          const float alpha = grow ? ex2_approx(m_used - mj) : 1.f;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float o16[16];
            tmem_ld16(t_oh + c * 16, o16);
#pragma unroll
            for (int i = 0; i < 16; ++i) o16[i] *= alpha;
            tmem_st16(t_oh + c * 16, o16);
          }
          tc_fence_before();
          l *= alpha;
          if (grow) m_used = mj;
        }
      }
      // this half's slab of buffer sb is free once P_{j-2} V_{j-2} of the half completed
      if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait_diag(&pv_done[hk * 2 + sb], ((j >> 1) & 1) ^ 1, abort_flag,
                                                             a.status, kDiagAttn, 8, j))) {
        ok = false;
        continue;
      }
      // with no key seen yet (m_used = -inf) every p is 2^-inf = 0
      const float nm = m_used == -INFINITY ? 0.f : -m_used;
      uint8_t* prow = sm + kAtcOffP + sb * kAtcTile + hk * kAtcSlab + r * 128;
      float rs0 = 0.f, rs1 = 0.f, rs2 = 0.f, rs3 = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = u * 8;
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = ex2_approx(fmaf(__uint_as_float(sv[i + e]), sc, nm));
        const uint4 w = make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                                   pack_bf16x2(p[6], p[7]));
        // l sums the bf16 values the tensor cores multiply, so that O / l
        // weights the keys exactly in proportion (one dominant key keeps
        // weight 1 whatever its rounding)
        rs0 += __uint_as_float(w.x << 16) + __uint_as_float(w.x & 0xffff0000u);
        rs1 += __uint_as_float(w.y << 16) + __uint_as_float(w.y & 0xffff0000u);
        rs2 += __uint_as_float(w.z << 16) + __uint_as_float(w.z & 0xffff0000u);
        rs3 += __uint_as_float(w.w << 16) + __uint_as_float(w.w & 0xffff0000u);
        *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) << 4)) = w;
      }
      l += (rs0 + rs1) + (rs2 + rs3);
      fence_async_shared();  // the P rows become visible to the tensor cores
      tc_fence_before();
      mbar_arrive(&p_full[hk * 2 + sb]);
    }
    if (live) {
      if (ok && nck > 0 &&
          !__all_sync(0xffffffffu, mbar_wait_diag(&pv_done[hk * 2 + ((nck - 1) & 1)], ((nck - 1) >> 1) & 1,
                                                  abort_flag, a.status, kDiagAttn, 9, nck)))
        ok = false;
      // combine the halves: both quadrant warps are past their last product,
      // so every MMA of the CTA has completed and Q is free
      const int pair_bar = 2 + q;             // named barrier of the quadrant's two warps
      float* xm = reinterpret_cast<float*>(sm + kAtcOffBar + 256);  // [half][128] running max
      float* xl = reinterpret_cast<float*>(sm);                     // [half][128] normaliser, over Q
      named_bar_sync(pair_bar, 64);
      xm[hk * 128 + r] = ok ? m_used : -INFINITY;
      xl[hk * 128 + r] = ok ? l : 0.f;
      named_bar_sync(pair_bar, 64);
      const float m_o = xm[(hk ^ 1) * 128 + r], l_o = xl[(hk ^ 1) * 128 + r];
      const float mown = ok ? m_used : -INFINITY;
      const float m = fmaxf(mown, m_o);
      // -inf - -inf is NaN: a half with no key (or a failed one) weighs 0
      const float s_own = mown == -INFINITY ? 0.f : ex2_approx(mown - m);
      const float s_oth = m_o == -INFINITY ? 0.f : ex2_approx(m_o - m);
      const float lt = (ok ? l : 0.f) * s_own + l_o * s_oth;
      const bool good = ok && lt > 0.f;
      pdl_wait();
      // this thread's 64 output columns, 32 at a time: O_own and O_other
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        const int c0 = hk * 64 + part * 32;
        uint32_t oa[32], ob[32];
        if (good) {
          tc_fence_after();
          tmem_ld32x2(tmem + kAtcColO + hk * 128 + lane_off + c0, oa,
                      tmem + kAtcColO + (hk ^ 1) * 128 + lane_off + c0, ob);
          tc_fence_before();
        }
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          o[i] = good ? __uint_as_float(oa[i]) * s_own + __uint_as_float(ob[i]) * s_oth : 0.f;
        if (a.splits == 1) {
          if (r < q_valid) {
            const float inv = good ? 1.f / lt : 0.f;
            uint4* og = reinterpret_cast<uint4*>(a.o + ((size_t)bi * a.rows_per_seq + row0 + r) * a.d + hc + c0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int i = u * 8;
              og[u] = make_uint4(pack_bf16x2(o[i] * inv, o[i + 1] * inv), pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv),
                                 pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv), pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv));
            }
          }
        } else {
          // partial (O relative to m, m, l) in this CTA's shared memory, over
          // the K ring and the P buffers, merged below; float4 column i of row
          // r at (i ^ r) mod 32: the 32 rows a warp stores at once fall in
          // different banks
          float4* po = reinterpret_cast<float4*>(sm + kAtcOffK) + r * 32;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int i = c0 / 4 + u;
            po[i ^ (r & 31)] = make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
          }
        }
      }
      if (a.splits > 1 && hk == 0) {
        float* pml = reinterpret_cast<float*>(sm + kAtcOffP) + r * 2;
        pml[0] = good ? m : -INFINITY;
        pml[1] = good ? lt : 0.f;
      }
    }
  }

  __syncthreads();
  if (a.splits > 1) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (warp >= 2) {
      // This CTA merges rows [ra, rb) of the tile over all splits.  Every
      // remote load of a step is issued before any of its values is used.
      const int t = threadIdx.x - 64;  // 0..255
      const int rank = (int)cluster.block_rank();
      const int per = (q_valid + a.splits - 1) / a.splits;
      const int ra = rank * per, nr = max(0, min(q_valid, ra + per) - ra);
      const float* pml = reinterpret_cast<const float*>(sm + kAtcOffP);
      const float* po = reinterpret_cast<const float*>(sm + kAtcOffK);
      float* coef = reinterpret_cast<float*>(sm);  // [per][8], over this CTA's Q tile
      if (t < nr) {
        const int rr = ra + t;
        float mv[kAtcMaxSplits], lv[kAtcMaxSplits];
#pragma unroll
        for (int sp = 0; sp < kAtcMaxSplits; ++sp) {
          mv[sp] = -INFINITY;
          lv[sp] = 0.f;
          if (sp < a.splits) {
            const float* rp = cluster.map_shared_rank(pml, sp);
            mv[sp] = rp[rr * 2];
            lv[sp] = rp[rr * 2 + 1];
          }
        }
        float mmax = mv[0];
#pragma unroll
        for (int sp = 1; sp < kAtcMaxSplits; ++sp) mmax = fmaxf(mmax, mv[sp]);
        float lsum = 0.f;
#pragma unroll
        for (int sp = 0; sp < kAtcMaxSplits; ++sp) {
          mv[sp] = mv[sp] == -INFINITY ? 0.f : ex2_approx(mv[sp] - mmax);
          lsum = fmaf(mv[sp], lv[sp], lsum);
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
        for (int sp = 0; sp < kAtcMaxSplits; ++sp) coef[t * kAtcMaxSplits + sp] = mv[sp] * inv;
      }
      named_bar_sync(1, kAtcSoftmax);
      // two items per thread per round: every remote load of the round is
      // issued before any of its values is used (a store in between would
      // order the next item's loads behind it)
      const int n_items = nr * 32;
      for (int base = t; base < n_items; base += 2 * kAtcSoftmax) {
        float4 o[2][kAtcMaxSplits];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int idx = base + u * kAtcSoftmax;
          if (idx < n_items) {
            const int rr = ra + (idx >> 5), c4 = (idx & 31) * 4;
#pragma unroll
            for (int sp = 0; sp < kAtcMaxSplits; ++sp)
              if (sp < a.splits)
                o[u][sp] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(po, sp) + rr * 128 +
                                                             (c4 ^ ((rr & 31) * 4)));
          }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int idx = base + u * kAtcSoftmax;
          if (idx < n_items) {
            const int row = idx >> 5, c4 = (idx & 31) * 4;
            float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
            for (int sp = 0; sp < kAtcMaxSplits; ++sp) {
              if (sp < a.splits) {
                const float w = coef[row * kAtcMaxSplits + sp];
                acc0 = fmaf(w, o[u][sp].x, acc0);
                acc1 = fmaf(w, o[u][sp].y, acc1);
                acc2 = fmaf(w, o[u][sp].z, acc2);
                acc3 = fmaf(w, o[u][sp].w, acc3);
              }
            }
            __nv_bfloat16* og = a.o + ((size_t)bi * a.rows_per_seq + row0 + ra + row) * a.d + hc + c4;
            *reinterpret_cast<uint2*>(og) = make_uint2(pack_bf16x2(acc0, acc1), pack_bf16x2(acc2, acc3));
          }
        }
      }
    }
    cluster.sync();  // keep this CTA's shared memory alive until every peer has read it
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kAtcTmemCols);
  }
}

#undef ATC_O4
#undef ATC_O32
#undef ATC_I4
#undef ATC_I32

}  // namespace dinfer
