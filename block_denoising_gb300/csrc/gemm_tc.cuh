// Weight-streaming tensor-core GEMM for sm_103a:  Y[m, n] = sum_k X[m, k] W[n, k]
//
// Operand roles are swapped relative to the usual token-major GEMM: the
// weight rows are the MMA's M dimension (128 per tile) and the tokens are its
// N dimension (BN per tile), so a batch-1 block of 64 tokens is one full MMA
// tile and the weights stream through shared memory exactly once.
//
// Structure (one CTA per SM, 192 threads):
//   warp 0  TMA producer: weight tile [128 x 64] + token tile [BN x 64] per
//           stage, 128-byte swizzle, completion on the stage's mbarrier;
//   warp 1  TMEM allocation + single-thread tcgen05.mma issue (4 x K16 per
//           stage), fp32 accumulators double-buffered in TMEM;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (one TMEM lane per
//           thread = one output feature), fused output op.
// Work is split "stream-K": the (tile, k-step) units are divided evenly over
// the CTAs, so every SM streams the same number of weight bytes whatever the
// tile count.  A CTA that owns a whole tile applies the fused epilogue
// itself; a tile shared by several CTAs is left as fp32 partials, which the
// fixup kernel below sums in CTA order (so results do not depend on timing)
// and finishes with the same epilogue -- one CTA per 16-column chunk, so the
// reduction is one parallel round trip instead of a serial tail.
#pragma once
#include "common.cuh"

namespace dinfer {

// (xr + i xi)(yr + i yi)
__device__ __forceinline__ void cmulf(float xr, float xi, float yr, float yi, float& zr, float& zi) {
  zr = fmaf(xr, yr, -xi * yi);
  zi = fmaf(xr, yi, xi * yr);
}

enum AMode : int {
  A_SINGLE = 0,  // one weight map, 128-row boxes
  A_THREE = 1,   // three maps (wq, wk, wv) of a_rows rows each, 128-row boxes
  A_PAIR = 2,    // two maps (gate, up), 64-row boxes stacked into one tile
};

struct GemmMaps {
  CUtensorMap a[3];
  CUtensorMap b;
};

struct GemmArgs {
  int M, N, K;            // tokens, output features, reduction length
  int m_tiles, n_tiles, k_tiles;
  int stream_k;           // 1: split (tile, k) units evenly; 0: whole tiles per CTA
  int a_mode, a_rows;     // see AMode; a_rows = rows per map in A_THREE
  // epilogue operands
  float* out_f32;
  __nv_bfloat16* out_bf16;
  int ldo;
  float* resid;
  __nv_bfloat16* q_out;    // [M, d]
  __nv_bfloat16* k_cache;  // this layer: [batch, L, d]
  __nv_bfloat16* v_cache;
  const float* rope_cos;   // [max_seq, head_dim / 2]
  const float* rope_sin;
  int d_model, head_dim;
  int rows_per_seq;        // rows of one sequence in X (block length or L)
  int seq_len;             // L (cache stride in positions)
  int pos_from_state;      // 1: position = block_start + local row; 0: local row
  int row_off;             // added to the position (first recomputed position of a window)
  const DevState* state;
  // stream-K partial tiles
  float* ws;               // [grid][2][BN tokens][128 rows] fp32 (token-major)
  int grid;                // CTAs of the GEMM launch (fixes the unit ranges)
  DevState* status;
  // grouped mode (mixture-of-experts): the tiles of `groups` independent
  // GEMMs that share the maps.  Group e owns rows [g_row_off[e], g_row_off[e+1])
  // of the token operand and weight rows [e * g_wrows, (e+1) * g_wrows) of the
  // weight map; its tiles are [g_tile_cum[e], g_tile_cum[e+1]) (device tables
  // written by the routing kernels), n-tile major.
  int grouped;
  int groups;
  const int* g_tile_cum;   // [groups + 1]
  const int* g_row_off;    // [groups + 1]
  int g_wrows;             // weight rows per group
  int g_a_half;            // A_PAIR: offset of the up rows inside a group
};

// Where a tile's operands and outputs are.  Token columns are local to the
// tile's group: local row m = mt * BN + c is valid when m < m_lim and lands on
// output row out_base + m.
struct TileRef {
  int nt, mt;
  int a_base;    // first weight row of the group in the weight map (0 when dense)
  int b_row;     // first token row of the token tile
  int m_lim;
  int out_base;
};

template <int BN>
__device__ __forceinline__ TileRef decode_tile(const GemmArgs& a, int t) {
  TileRef r;
  if (!a.grouped) {
    r.nt = t / a.m_tiles;
    r.mt = t - r.nt * a.m_tiles;
    r.a_base = 0;
    r.b_row = r.mt * BN;
    r.m_lim = a.M;
    r.out_base = 0;
    return r;
  }
  int lo = 0, hi = a.groups;  // e with g_tile_cum[e] <= t < g_tile_cum[e + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a.g_tile_cum + mid) <= t) lo = mid; else hi = mid;
  }
  const int row0 = __ldg(a.g_row_off + lo), rows = __ldg(a.g_row_off + lo + 1) - row0;
  const int mtiles = (rows + BN - 1) / BN;
  const int li = t - __ldg(a.g_tile_cum + lo);
  r.nt = li / mtiles;
  r.mt = li - r.nt * mtiles;
  r.a_base = lo * a.g_wrows;
  r.b_row = row0 + r.mt * BN;
  r.m_lim = rows;
  r.out_base = row0;
  return r;
}

constexpr int kGemmThreads = 192;

// Pipeline depth: as many stages as fit in shared memory beside the epilogue
// exchange buffer (the weight bytes in flight per SM set the streaming rate
// of a CTA: nine 16 KB weight tiles at 64 tokens).
template <int BN>
constexpr int gemm_default_stages() { return BN == 64 ? 9 : (BN == 128 ? 6 : 4); }
// TMEM column distance of the two accumulators: BN, or 256 for tiles wider
// than 128 tokens (each accumulator starts on a 256-column boundary)
template <int BN>
__host__ __device__ constexpr int acc_stride() { return BN <= 128 ? BN : 256; }
// the GEMM kernel stages QKV outputs where the buffers fit beside its stages
// and two exchange buffers
template <int BN>
constexpr int gemm_default_staged() {
  return 1024 + gemm_default_stages<BN>() * (128 + BN) * 128 + 2 * 128 * 17 * 4 + 2 * 16 * 128 * 2 + 512 <= 232448;
}

// STG: the QKV epilogue stages its bf16 outputs in shared memory (two
// 16-token x 128-row buffers) and stores whole 16-byte vectors.
template <int BN, int ST = gemm_default_stages<BN>(), int STG = 0>
struct GemmCfg {
  static constexpr int kStageA = 128 * 64 * 2;
  static constexpr int kStageB = BN * 64 * 2;
  static constexpr int kStage = kStageA + kStageB;
  static constexpr int kStages = ST;
  // epilogue row-pair exchange: two buffers used in turn where they fit
  // beside the stages (227 KB per CTA), else one
  static constexpr int kXchgBufs = (1024 + kStages * kStage + 2 * 128 * 17 * 4 + 512 <= 232448) ? 2 : 1;
  static constexpr int kXchgFloats = kXchgBufs * 128 * 17;
  static constexpr int kStageOutBytes = STG ? 2 * 16 * 128 * 2 : 0;
  static constexpr int kSmem = 1024 /*align slack*/ + kStages * kStage + kXchgFloats * 4 + kStageOutBytes + 512;
  static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
  static_assert(kSmem <= 232448, "GEMM shared memory above 227 KB");
};
// the configuration gemm_tc_kernel<BN> runs with
template <int BN>
using GemmKCfg = GemmCfg<BN, gemm_default_stages<BN>(), gemm_default_staged<BN>()>;

// ---------------------------------------------------------------------------
// schedule: contiguous unit ranges per CTA
// ---------------------------------------------------------------------------
struct Sched {
  // 32-bit: the launcher guarantees U * G < 2^32
  unsigned U;  // total units
  unsigned KT; // units per tile (k-steps) in stream-K mode, 1 otherwise
  unsigned G;
  __host__ __device__ __forceinline__ unsigned start(unsigned c) const { return (U * c) / G; }
  __host__ __device__ __forceinline__ int owner(unsigned u) const { return (int)(((u + 1) * G - 1) / U); }
};

// 2-D tiled TMA load into this CTA's shared memory, completing on the
// mbarrier at shared::cluster address `bar`: this CTA's own, or (kPair, the
// cta_group::2 form) the pair leader's.
template <bool kPair>
__device__ __forceinline__ void tma_load_2d_to(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                               uint64_t policy) {
  if (kPair)
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// The 128 weight rows of tile tr.nt, k-step k, into `stage`.
template <bool kPair = false>
__device__ __forceinline__ void load_stage_a(const GemmMaps& maps, const GemmArgs& a, uint8_t* stage, uint32_t bar,
                                             const TileRef& tr, int k, uint64_t pol_w) {
  uint8_t* sa = stage;
  const int kx = k * 64;
  const int nt = tr.nt;
  if (a.grouped) {
    if (a.a_mode == A_PAIR) {
      tma_load_2d_to<kPair>(sa, &maps.a[0], bar, kx, tr.a_base + nt * 64, pol_w);
      tma_load_2d_to<kPair>(sa + 64 * 128, &maps.a[0], bar, kx, tr.a_base + a.g_a_half + nt * 64, pol_w);
    } else {
      tma_load_2d_to<kPair>(sa, &maps.a[0], bar, kx, tr.a_base + nt * 128, pol_w);
    }
  } else if (a.a_mode == A_PAIR) {
    tma_load_2d_to<kPair>(sa, &maps.a[0], bar, kx, nt * 64, pol_w);
    tma_load_2d_to<kPair>(sa + 64 * 128, &maps.a[1], bar, kx, nt * 64, pol_w);
  } else if (a.a_mode == A_THREE) {
    const int per = a.a_rows / 128;
    tma_load_2d_to<kPair>(sa, &maps.a[nt / per], bar, kx, (nt % per) * 128, pol_w);
  } else {
    tma_load_2d_to<kPair>(sa, &maps.a[0], bar, kx, nt * 128, pol_w);
  }
}
template <int BN>
__device__ __forceinline__ void load_stage_b(const GemmMaps& maps, uint8_t* stage, uint64_t* bar, int b_row, int k,
                                             uint64_t pol_x) {
  tma_load_2d(stage + GemmCfg<BN>::kStageA, &maps.b, bar, k * 64, b_row, pol_x);
}

// RoPE factors of output row `row` of tile nt for the 16 tokens m0..m0+15
// (q and k rows; v rows need none).  base_pos: absolute position of token 0
// of a sequence's rows (the block start for block rows, 0 for a refresh).
// bf16 models have head_dim 128, so a 128-row tile is one head of q, k or v
// and row is the feature inside the head; its rotation frequency is row % 64.
// Token -> (sequence, row) steps along the chunk: one division per chunk.
__device__ __forceinline__ void qkv_rope_fetch(const GemmArgs& a, int base_pos, int row, int nt, int m0,
                                               float (&cs)[16], float (&sn)[16]) {
  if (nt * 128 >= 2 * a.d_model) return;
  const int j = row & 63;
  int r = m0 - (m0 / a.rows_per_seq) * a.rows_per_seq;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int pos = base_pos + r;
    cs[c] = __ldg(a.rope_cos + pos * 64 + j);
    sn[c] = __ldg(a.rope_sin + pos * 64 + j);
    if (++r == a.rows_per_seq) r = 0;
  }
}

// Epilogue of 16 tokens (m0..m0+15) of output row `row` of tile nt.  QKV
// tiles take their RoPE factors from `rope` (cos then sin, made by the
// caller) or, when it is NULL, load them here.  `xchg` (128 x 17 floats)
// pairs rows through shared memory.  A caller that finishes several chunks
// either alternates two buffers, so that a chunk's writes never meet the
// previous chunk's reads, or reuses one and asks for a barrier after the
// reads (`sync_after`).
template <int BN>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& a, float (&v)[16], int row, int nt, int m0,
                                               float* xchg, int m_lim, int out_base, bool sync_after,
                                               const float (*rope)[16] = nullptr, int base_pos_in = -1,
                                               __nv_bfloat16* stage = nullptr, bool stage_f32 = false) {
  if (a.q_out != nullptr) {
    // ---- QKV: RoPE pairs (i, i + 64) sit in rows row and row ^ 64 ----
    const int d = a.d_model;
    const int which = (nt * 128) / d;           // 0 q, 1 k, 2 v
    const int nn = nt * 128 - which * d + row;  // feature inside q/k/v
    const int base_pos =
        base_pos_in >= 0 ? base_pos_in : (a.pos_from_state ? a.state->block_start : 0) + a.row_off;
    float cs[16], sn[16];
    if (rope) {
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        cs[c] = rope[0][c];
        sn[c] = rope[1][c];
      }
    } else {
      qkv_rope_fetch(a, base_pos, row, nt, m0, cs, sn);
    }
    float* mine = xchg + row * 17;
#pragma unroll
    for (int c = 0; c < 16; ++c) mine[c] = v[c];
    named_bar_sync(1, 128);
    const float* part = xchg + (row ^ 64) * 17;
    float o[16];
    const float sgn = row < 64 ? -1.f : 1.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) o[c] = (which == 2) ? v[c] : fmaf(sgn * part[c], sn[c], v[c] * cs[c]);
    if (stage != nullptr) {
      // stage the chunk as [16 tokens][128 features] bf16, then each thread
      // stores two 16-byte pieces (8 features of one token): whole 256-byte
      // rows per token instead of 2-byte stores 2 * d bytes apart
#pragma unroll
      for (int c = 0; c < 16; ++c) stage[c * 128 + row] = __float2bfloat16_rn(o[c]);
      named_bar_sync(1, 128);
      __nv_bfloat16* __restrict__ dst0 = (which == 0 ? a.q_out : (which == 1 ? a.k_cache : a.v_cache)) +
                                         (nt * 128 - which * d);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int piece = row + h * 128;  // 16 tokens x 16 pieces
        const int c = piece >> 4, f8 = (piece & 15) * 8;
        const int m = m0 + c;
        if (m < a.M) {
          const int bi = m / a.rows_per_seq, r = m - bi * a.rows_per_seq;
          const size_t orow = which == 0 ? (size_t)m : (size_t)bi * a.seq_len + base_pos + r;
          *reinterpret_cast<uint4*>(dst0 + orow * d + f8) = *reinterpret_cast<const uint4*>(stage + c * 128 + f8);
        }
      }
      if (sync_after) named_bar_sync(1, 128);
      return;
    }
    if (sync_after) named_bar_sync(1, 128);
    __nv_bfloat16* __restrict__ dst = (which == 0 ? a.q_out : (which == 1 ? a.k_cache : a.v_cache)) + nn;
    int bi = m0 / a.rows_per_seq;
    int r = m0 - bi * a.rows_per_seq;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int m = m0 + c;
      if (m < a.M) {
        const size_t orow = which == 0 ? (size_t)m : (size_t)bi * a.seq_len + base_pos + r;
        dst[orow * d] = __float2bfloat16_rn(o[c]);
      }
      if (++r == a.rows_per_seq) {
        r = 0;
        ++bi;
      }
    }
  } else if (a.a_mode == A_PAIR) {
    // ---- SwiGLU: gate row r (< 64) pairs with up row r + 64 ----
    // the pair splits the 16 tokens: the gate row finishes tokens 0..7 and
    // hands its values of tokens 8..15 to the up row, which finishes those
    const bool gate_row = row < 64;
    float* mine = xchg + row * 17;
#pragma unroll
    for (int i = 0; i < 8; ++i) mine[i] = gate_row ? v[8 + i] : v[i];
    named_bar_sync(1, 128);
    const float* part = xchg + (row ^ 64) * 17;
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float g = gate_row ? v[i] : part[i];
      const float u = gate_row ? part[i] : v[8 + i];
      o[i] = __fdividef(g, 1.0f + __expf(-g)) * u;  // rounded to bf16 next
    }
    if (sync_after) named_bar_sync(1, 128);
    const int jf = nt * 64 + (row & 63);
    const int mh = m0 + (gate_row ? 0 : 8);
    if (jf < a.N) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (mh + i < m_lim) a.out_bf16[(size_t)(out_base + mh + i) * a.ldo + jf] = __float2bfloat16_rn(o[i]);
    }
  } else if (stage_f32 && a.resid == nullptr && a.out_bf16 == nullptr) {
    // plain fp32 output: stage the chunk as [16 tokens][128 rows] in xchg
    // (all 128 threads take part in the barrier), then each thread stores
    // four 16-byte pieces -- whole 512-byte token rows
    float* st = xchg;
#pragma unroll
    for (int c = 0; c < 16; ++c) st[c * 128 + row] = v[c];
    named_bar_sync(1, 128);
    const int n0 = nt * 128;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int piece = row + h * 128;  // 16 tokens x 32 pieces
      const int c = piece >> 5, f4 = (piece & 31) * 4;
      if (m0 + c < m_lim && n0 + f4 < a.N)
        *reinterpret_cast<float4*>(a.out_f32 + (size_t)(out_base + m0 + c) * a.ldo + n0 + f4) =
            *reinterpret_cast<const float4*>(st + c * 128 + f4);
    }
    if (sync_after) named_bar_sync(1, 128);
  } else {
    const int n = nt * 128 + row;
    if (n < a.N) {
      if (a.resid) {
        // residual add: all 16 loads in flight before the stores
        float hv[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) hv[c] = (m0 + c < a.M) ? a.resid[(size_t)(m0 + c) * a.N + n] : 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (m0 + c < a.M) a.resid[(size_t)(m0 + c) * a.N + n] = hv[c] + v[c];
      } else if (a.out_bf16) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (m0 + c < m_lim) a.out_bf16[(size_t)(out_base + m0 + c) * a.ldo + n] = __float2bfloat16_rn(v[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (m0 + c < m_lim) a.out_f32[(size_t)(out_base + m0 + c) * a.ldo + n] = v[c];
      }
    }
  }
}

// h[m0 .. m0+15, n] of a residual GEMM (zeros past M), all 16 loads in flight.
__device__ __forceinline__ void resid_load16(const GemmArgs& a, int n, int m0, float (&hv)[16]) {
#pragma unroll
  for (int c = 0; c < 16; ++c) hv[c] = (m0 + c < a.M) ? a.resid[(size_t)(m0 + c) * a.N + n] : 0.f;
}

// The segments (tile t, k-steps [kb, ke)) of one CTA's unit range.  In
// stream-K mode the range [u0, u1) covers the tail of tile tf, whole tiles,
// and the head of tile tl; the partial segments are processed FIRST so that
// the cross-CTA reduction of a shared tile happens while the other CTAs are
// still streaming, and the kernel ends on whole tiles.
struct SegList {
  int stream_k, k_tiles;
  long long u0, u1;
  int tf, nseg, first_partial, last_partial, np;
  int stride;  // whole-tile mode: tiles tf, tf + stride, ...
  // stream-K: the unit range [b, e).  Whole tiles (sk == 0): tiles are dealt
  // round-robin (b = CTA index, e = tile count, stride = grid), so that the
  // CTAs running at the same time cover consecutive tiles -- the token tiles
  // of one weight tile -- and share its weight stream through L2.
  __device__ __forceinline__ void init(int sk, int kt, long long b, long long e, int grid = 1) {
    stream_k = sk;
    k_tiles = kt;
    u0 = b;
    u1 = e;
    stride = 1;
    if (!sk) {
      tf = (int)b;
      stride = grid;
      nseg = b < e ? (int)((e - b + grid - 1) / grid) : 0;
      first_partial = last_partial = np = 0;
      return;
    }
    if (u1 <= u0) {
      nseg = 0;
      return;
    }
    tf = (int)(u0 / kt);
    const int tl = (int)((u1 - 1) / kt);
    nseg = tl - tf + 1;
    first_partial = (u0 % kt) != 0 || (nseg == 1 && (u1 % kt) != 0);
    last_partial = nseg > 1 && (u1 % kt) != 0;
    np = first_partial + last_partial;
  }
  // natural index of the j-th processed segment
  __device__ __forceinline__ int natural(int j) const {
    if (j < np) return (j == 0 && last_partial) ? nseg - 1 : 0;
    return (first_partial ? 1 : 0) + (j - np);
  }
  __device__ __forceinline__ void seg(int j, int& t, int& kb, int& ke) const {
    if (!stream_k) {
      t = tf + j * stride;
      kb = 0;
      ke = k_tiles;
      return;
    }
    const int k = natural(j);
    t = tf + k;
    const long long ts = (long long)t * k_tiles;
    const long long a = ts > u0 ? ts : u0;
    const long long b = (ts + k_tiles) < u1 ? (ts + k_tiles) : u1;
    kb = (int)(a - ts);
    ke = (int)(b - ts);
  }
};

struct Pipe {
  uint8_t* stages;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* drain;
  volatile int* abort_flag;
  int* rec;  // producer stage records [2 * kStages] (shared memory, not thread-local)
};

// Sum, in CTA order, the token-major partials of split tile t that the
// contributors of the stream-K schedule published, for this thread's output
// row and the 16 tokens of chunk c.
template <int BN>
__device__ __forceinline__ void sum_split_partials(const GemmArgs& a, int t, int row, int c, float (&v)[16]) {
  Sched sc;
  sc.G = a.grid;
  sc.KT = a.k_tiles;
  sc.U = (unsigned)(a.m_tiles * a.n_tiles) * a.k_tiles;
  const unsigned tu0 = (unsigned)t * a.k_tiles;
  const int c_first = sc.owner(tu0), c_last = sc.owner(tu0 + a.k_tiles - 1);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = 0.f;
#pragma unroll 1
  for (int cc = c_first; cc <= c_last; cc += 2) {
    float buf[2][16];
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (cc + x <= c_last) {
        const int slot = (cc + x) * 2 + (((unsigned)t == sc.start(cc + x) / sc.KT) ? 0 : 1);
        const float* src = a.ws + (size_t)slot * (BN * 128) + (size_t)(c * 16) * 128 + row;
#pragma unroll
        for (int i = 0; i < 16; ++i) buf[x][i] = __ldcg(src + (size_t)i * 128);
      }
#pragma unroll
    for (int x = 0; x < 2; ++x)
      if (cc + x <= c_last)
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += buf[x][i];
  }
}

// TMA producer loop (one elected thread of warp 0).  The weight tiles of the
// first pipeline stages do not depend on the preceding kernel, so they are
// requested before griddepcontrol.wait; the activation tiles after it.
template <int BN, int ST = gemm_default_stages<BN>()>
__device__ __forceinline__ void run_producer(const GemmMaps& maps, const GemmArgs& a, const SegList& sl,
                                             const Pipe& p, int m_tiles) {
  using C = GemmCfg<BN, ST>;
  // weight tiles used by a single token tile stream through L2 once; with
  // several token tiles the following tiles re-read them from L2
  const uint64_t pol_w = (m_tiles == 1 && !a.grouped) ? l2_policy_evict_first() : l2_policy_evict_normal();
  const uint64_t pol_x = l2_policy_evict_last();
  // phase 1: weights of the first kStages stages (dense: before the wait);
  // the stage records stay in shared memory (thread-local arrays would live
  // in L2 on an SM whose memory is carved out as shared memory)
  int* pre_b = p.rec;
  int* pre_k = p.rec + C::kStages;
  int pre = 0;
  if (!a.grouped) {
    for (int j = 0; j < sl.nseg && pre < C::kStages; ++j) {
      int t, kb, ke;
      sl.seg(j, t, kb, ke);
      const TileRef tr = decode_tile<BN>(a, t);
      for (int k = kb; k < ke && pre < C::kStages; ++k, ++pre) {
        mbar_arrive_expect_tx(&p.full[pre], C::kStage);
        load_stage_a(maps, a, p.stages + pre * C::kStage, smem_u32(&p.full[pre]), tr, k, pol_w);
        pre_b[pre] = tr.b_row;
        pre_k[pre] = k;
      }
    }
  }
  pdl_wait();
  for (int i = 0; i < pre; ++i) load_stage_b<BN>(maps, p.stages + i * C::kStage, &p.full[i], pre_b[i], pre_k[i], pol_x);
  // phase 2: the rest of the pipeline
  uint32_t it = 0;
  for (int j = 0; j < sl.nseg && !*p.abort_flag; ++j) {
    int t, kb, ke;
    sl.seg(j, t, kb, ke);
    const TileRef tr = decode_tile<BN>(a, t);
    bool ok = true;
    for (int k = kb; k < ke; ++k, ++it) {
      if (it < (uint32_t)pre) continue;
      const int s = it % C::kStages;
      const uint32_t round = it / C::kStages;
      if (!mbar_wait(&p.empty[s], (round & 1) ^ 1, p.abort_flag)) { ok = false; break; }
      mbar_arrive_expect_tx(&p.full[s], C::kStage);
      load_stage_a(maps, a, p.stages + s * C::kStage, smem_u32(&p.full[s]), tr, k, pol_w);
      load_stage_b<BN>(maps, p.stages + s * C::kStage, &p.full[s], tr.b_row, k, pol_x);
    }
    if (!ok) break;
  }
}

// MMA issue loop (one elected thread of warp 1).
template <int BN, int ST = gemm_default_stages<BN>()>
__device__ __forceinline__ void run_mma(const SegList& sl, const Pipe& p, uint32_t tmem_base) {
  using C = GemmCfg<BN, ST>;
  constexpr uint32_t idesc = make_idesc_bf16(128, BN);
  uint32_t it = 0;
  for (int j = 0; j < sl.nseg && !*p.abort_flag; ++j) {
    int t, kb, ke;
    sl.seg(j, t, kb, ke);
    const int acc = j & 1;
    const uint32_t use = j >> 1;
    if (!mbar_wait(&p.tempty[acc], (use & 1) ^ 1, p.abort_flag)) break;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + acc * acc_stride<BN>();
    bool ok = true;
    for (int k = kb; k < ke; ++k, ++it) {
      const int s = it % C::kStages;
      if (!mbar_wait(&p.full[s], (it / C::kStages) & 1, p.abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sa = smem_u32(p.stages + s * C::kStage);
      const uint32_t sb = sa + C::kStageA;
      const uint64_t ad = make_sw128_desc(sa);
      const uint64_t bd = make_sw128_desc(sb);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        tc_mma_bf16(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, (k > kb || kk > 0) ? 1u : 0u);
      }
      tc_commit(&p.empty[s]);
    }
    if (!ok) break;
    tc_commit(&p.tfull[acc]);
  }
  tc_commit(p.drain);
  mbar_wait(p.drain, 0, p.abort_flag);
}

// Carve the shared memory of a GEMM CTA and initialise its barriers.
template <int BN, int ST = gemm_default_stages<BN>(), int STG = 0>
__device__ __forceinline__ Pipe setup_pipe(uint8_t* smem_raw, float*& xchg, uint32_t*& tmem_slot,
                                           volatile int*& misc) {
  using C = GemmCfg<BN, ST, STG>;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Pipe p;
  p.stages = smem;
  xchg = reinterpret_cast<float*>(smem + C::kStages * C::kStage);
  // [kStageOutBytes of QKV output staging after the exchange buffers]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xchg + C::kXchgFloats) + C::kStageOutBytes);
  p.full = bars;
  p.empty = bars + C::kStages;
  p.tfull = bars + 2 * C::kStages;
  p.tempty = p.tfull + 2;
  p.drain = p.tempty + 2;
  tmem_slot = reinterpret_cast<uint32_t*>(p.drain + 1);
  misc = reinterpret_cast<volatile int*>(tmem_slot + 1);
  p.abort_flag = misc;
  p.rec = const_cast<int*>(misc + 2);  // misc[2 .. 2 + 2 * kStages)
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&p.full[s], 1);
      mbar_init(&p.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p.tfull[i], 1);
      mbar_init(&p.tempty[i], 128);
    }
    mbar_init(p.drain, 1);
    misc[0] = 0;
    fence_mbar_init();
  }
  return p;
}

// Epilogue warps (2-5) of a GEMM CTA: finish the accumulator of each of the
// CTA's nseg segments in turn.  seg_tile(j, t, kb, ke, tr) names segment j
// (tile t, k-steps [kb, ke), operands and outputs tr); a segment that is not
// a whole tile leaves token-major fp32 partials at partial_slot(t);
// release(acc) hands accumulator acc back to the MMA issuer.  NXB: exchange
// buffers (see epilogue_chunk); stage_out: two QKV output staging buffers
// (NULL: QKV outputs are stored directly), used in turn with NXB == 2.
template <int BN, int NXB, class SegFn, class SlotFn, class ReleaseFn>
__device__ __forceinline__ void run_epilogue(const GemmArgs& a, const Pipe& p, uint32_t tmem_base, float* xchg,
                                             __nv_bfloat16* stage_out, int warp, int lane, int nseg,
                                             SegFn seg_tile, SlotFn partial_slot, ReleaseFn release) {
  pdl_wait();  // global writes only after the preceding kernel completed
  const int base_pos =
      a.q_out != nullptr ? (a.pos_from_state ? a.state->block_start : 0) + a.row_off : 0;
  const int q = warp & 3;                 // TMEM lane quadrant of this warp
  const int row = q * 32 + lane;          // output feature row inside the tile
  // QKV: RoPE factors of this row's frequency.  A whole tile loads those of
  // its first token (and of the sequence start, where a tile wraps into
  // the next sequence) ahead of its main loop; the following tokens step
  // by one rotation of the frequency's angle (<= BN steps: an error of a
  // few fp32 ulps, far below the bf16 rounding of q and k).
  float rc = 1.f, rs = 0.f, rc0 = 1.f, rs0 = 0.f, step_c = 1.f, step_s = 0.f;
  if (a.q_out != nullptr) {
    step_c = __ldg(a.rope_cos + 64 + (row & 63));
    step_s = __ldg(a.rope_sin + 64 + (row & 63));
  }
  // rotations by 2, 4, 8 and 16 positions: a chunk's 16 factors come from
  // its first one at most four products deep, the next chunk's first one
  // from a single product
  float p2c, p2s, p4c, p4s, p8c, p8s, p16c, p16s;
  cmulf(step_c, step_s, step_c, step_s, p2c, p2s);
  cmulf(p2c, p2s, p2c, p2s, p4c, p4s);
  cmulf(p4c, p4s, p4c, p4s, p8c, p8s);
  cmulf(p8c, p8s, p8c, p8s, p16c, p16s);
  int xb = 0;  // exchange buffer of the next pairing chunk
  for (int j = 0; j < nseg; ++j) {
    int t, kb, ke;
    TileRef tr;
    seg_tile(j, t, kb, ke, tr);
    const int acc = j & 1;
    const uint32_t use = j >> 1;
    const bool whole = (kb == 0 && ke == a.k_tiles);
    const int n = tr.nt * 128 + row;
    float hcur[16];  // residual: h of the chunk being finished
    // loads of the tile's first RoPE factors or residual values overlap its
    // main loop (a whole tile's h is written by this thread only)
    int rr = 0;  // QKV: offset of the chunk's first token in its sequence
    if (a.q_out != nullptr && whole) {
      rr = (tr.mt * BN) % a.rows_per_seq;
      rc = __ldg(a.rope_cos + (base_pos + rr) * 64 + (row & 63));
      rs = __ldg(a.rope_sin + (base_pos + rr) * 64 + (row & 63));
      rc0 = __ldg(a.rope_cos + base_pos * 64 + (row & 63));
      rs0 = __ldg(a.rope_sin + base_pos * 64 + (row & 63));
    }
    if (a.resid != nullptr && whole) resid_load16(a, n, tr.mt * BN, hcur);
    if (!mbar_wait(&p.tfull[acc], use & 1, p.abort_flag)) break;
    tc_fence_after();
    const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * acc_stride<BN>();
    if (!whole) {
      // partial tile: token-major [BN][128], so a warp stores whole lines
      float* base = partial_slot(t);
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tbase + c * 16, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) base[(size_t)(c * 16 + i) * 128 + row] = v[i];
      }
      tc_fence_before();
      release(acc);
      continue;
    }
    if (a.q_out != nullptr) {
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tbase + c * 16, v);
        float rope[2][16];
        if (rr + 16 <= a.rows_per_seq) {
          // the chunk stays inside one sequence
          rope[0][0] = rc;
          rope[1][0] = rs;
          cmulf(rc, rs, step_c, step_s, rope[0][1], rope[1][1]);
#pragma unroll
          for (int i = 0; i < 2; ++i) cmulf(rope[0][i], rope[1][i], p2c, p2s, rope[0][2 + i], rope[1][2 + i]);
#pragma unroll
          for (int i = 0; i < 4; ++i) cmulf(rope[0][i], rope[1][i], p4c, p4s, rope[0][4 + i], rope[1][4 + i]);
#pragma unroll
          for (int i = 0; i < 8; ++i) cmulf(rope[0][i], rope[1][i], p8c, p8s, rope[0][8 + i], rope[1][8 + i]);
          rr += 16;
          if (rr == a.rows_per_seq) {
            rr = 0;
            rc = rc0;
            rs = rs0;
          } else {
            cmulf(rope[0][0], rope[1][0], p16c, p16s, rc, rs);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            rope[0][i] = rc;
            rope[1][i] = rs;
            if (++rr == a.rows_per_seq) {
              rr = 0;
              rc = rc0;
              rs = rs0;
            } else {
              cmulf(rope[0][i], rope[1][i], step_c, step_s, rc, rs);
            }
          }
        }
        epilogue_chunk<BN>(a, v, row, tr.nt, tr.mt * BN + c * 16, xchg + xb * (128 * 17), tr.m_lim, tr.out_base,
                           NXB == 1, rope, base_pos, stage_out ? stage_out + xb * (16 * 128) : nullptr);
        xb ^= NXB - 1;
      }
    } else if (a.resid != nullptr) {
      // residual: h of chunk c + 1 loads while chunk c is finished
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        const int m0 = tr.mt * BN + c * 16;
        float v[16], hnext[16];
        tmem_ld16(tbase + c * 16, v);
        if (c + 1 < BN / 16) resid_load16(a, n, m0 + 16, hnext);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (m0 + i < a.M) a.resid[(size_t)(m0 + i) * a.N + n] = hcur[i] + v[i];
#pragma unroll
        for (int i = 0; i < 16; ++i) hcur[i] = hnext[i];
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tbase + c * 16, v);
        epilogue_chunk<BN>(a, v, row, tr.nt, tr.mt * BN + c * 16, xchg + xb * (128 * 17), tr.m_lim, tr.out_base,
                           NXB == 1, nullptr, -1, nullptr, stage_out != nullptr && NXB == 2);
        xb ^= NXB - 1;
      }
    }
    tc_fence_before();
    release(acc);
  }
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs args) {
  using C = GemmKCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  float* xchg;
  uint32_t* tmem_slot;
  volatile int* misc;
  const Pipe p = setup_pipe<BN, C::kStages, C::kStageOutBytes ? 1 : 0>(smem_raw, xchg, tmem_slot, misc);
  __nv_bfloat16* stage_out =
      C::kStageOutBytes ? reinterpret_cast<__nv_bfloat16*>(xchg + C::kXchgFloats) : nullptr;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const GemmArgs& a = args;

  Sched sc;
  sc.G = gridDim.x;
  // grouped: the tile count is written by the routing kernels that precede
  // this launch, so it is read after the dependency wait
  if (a.grouped) pdl_wait();
  const int tiles = a.grouped ? __ldg(a.g_tile_cum + a.groups) : a.m_tiles * a.n_tiles;
  sc.KT = a.stream_k ? a.k_tiles : 1;
  sc.U = (unsigned)tiles * sc.KT;
  SegList sl;
  if (a.stream_k)
    sl.init(1, a.k_tiles, sc.start(blockIdx.x), sc.start(blockIdx.x + 1));
  else
    sl.init(0, a.k_tiles, blockIdx.x, tiles, gridDim.x);

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.b);
    prefetch_tmap(&maps.a[0]);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // one wave (<= one CTA per SM): the next kernel may start launching now
  if (threadIdx.x == 0) pdl_trigger();

  if (warp == 0) {
    if (elect_one_sync()) run_producer<BN>(maps, a, sl, p, a.m_tiles);
  } else if (warp == 1) {
    if (elect_one_sync()) run_mma<BN>(sl, p, tmem_base);
  } else {
    run_epilogue<BN, C::kXchgBufs>(
        a, p, tmem_base, xchg, stage_out, warp, lane, sl.nseg,
        [&](int j, int& t, int& kb, int& ke, TileRef& tr) {
          sl.seg(j, t, kb, ke);
          tr = decode_tile<BN>(a, t);
        },
        // slot 0 holds this CTA's part of its first tile, slot 1 of its last
        [&](int t) { return a.ws + ((size_t)blockIdx.x * 2 + (t == sl.tf ? 0 : 1)) * (BN * 128); },
        [&](int acc) { mbar_arrive(&p.tempty[acc]); });
  }

  __syncthreads();
  if (*p.abort_flag && threadIdx.x == 0) record_timeout(a.status, kDiagGemm, 0, 0);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Split-K fixup: block = (tile, 16-column chunk), 128 threads = the tile's
// output rows; the partial slots are token-major.  Sums the partial slots of the tile's contributors (the CTAs
// of the GEMM grid whose unit ranges overlap it) in CTA order, then applies
// the GEMM's epilogue.  Tiles owned whole by one CTA were finished by it.
template <int BN>
__global__ void __launch_bounds__(128) splitk_fixup_kernel(const GemmArgs a) {
  __shared__ float xchg[128 * 17];
  pdl_wait();
  const int chunks = BN / 16;
  const int t = blockIdx.x / chunks, c = blockIdx.x % chunks;
  Sched sc;
  sc.G = a.grid;
  sc.KT = a.k_tiles;
  sc.U = (unsigned)(a.m_tiles * a.n_tiles) * a.k_tiles;
  const unsigned tu0 = (unsigned)t * a.k_tiles;
  const int c_first = sc.owner(tu0);
  const int c_last = sc.owner(tu0 + a.k_tiles - 1);
  if (c_first == c_last) {  // whole tile: done by the GEMM
    pdl_trigger();
    return;
  }
  // token-major slots [BN tokens][128 rows]: for each token the 32 threads
  // of a warp read 32 consecutive rows, one whole 128-byte line
  const int row = threadIdx.x;
  float v[16];
  sum_split_partials<BN>(a, t, row, c, v);
  const int nt = t / a.m_tiles, mt = t % a.m_tiles;
  epilogue_chunk<BN>(a, v, row, nt, mt * BN + c * 16, xchg, a.M, 0, false);
  pdl_trigger();
}

// Residual GEMM finish fused with the next RMSNorm.  The O and down
// projections leave tiles shared by several CTAs as token-major fp32 partials
// (whole tiles were already added to h by the GEMM).  One CTA per output row r
// (token src(r)), d / 16 threads, 16 features per thread in the row-kernel
// layout (one weight tile of 128 features per 8 threads):
//   h[src] += sum of the partials of every shared tile, in CTA order;
//   out[r] = bf16(h[src] / sqrt(mean(h[src]^2) + eps) * g).
// Pair-GEMM tile order: pair tile t -> (weight pair tile np, token tile mt).
// Token tiles go in groups of kPairGroupM, each group swept weight-tile
// major, so that the ~76 pairs running at once read a few weight tiles and at
// most kPairGroupM token tiles (a few tens of MB, inside L2) whatever the
// token count; with <= kPairGroupM token tiles this is t = np * m_tiles + mt.
constexpr int kPairGroupM = 8;
__host__ __device__ __forceinline__ void pair_tile_coords(int t, int m_tiles, int np_tiles, int& np, int& mt) {
  const int per_group = kPairGroupM * np_tiles;
  const int g = t / per_group;
  const int w = t - g * per_group;
  const int m0 = g * kPairGroupM;
  const int gm = min(kPairGroupM, m_tiles - m0);
  np = w / gm;
  mt = m0 + (w - np * gm);
}
__host__ __device__ __forceinline__ int pair_tile_index(int np, int mt, int m_tiles, int np_tiles) {
  const int g = mt / kPairGroupM, m0 = g * kPairGroupM;
  const int gm = min(kPairGroupM, m_tiles - m0);
  return g * kPairGroupM * np_tiles + np * gm + (mt - m0);
}

struct ResidPlan {
  const float* ws;
  int m_tiles, n_tiles, k_tiles, grid, BN;
  int stream_k;  // 0: the GEMM owned whole tiles, nothing left to add
  // 1: the pair-CTA GEMM: grid counts pairs, a unit is (pair tile, k-step)
  // with pair tile pair_tile_index(nt / 2, mt), and the slots of CTA
  // 2 c + nt % 2 of pair c hold rows of 128-row tile nt
  int pair;
};

// x = h[src] at the thread's 16 features (row-kernel layout from f0) plus the
// stream-K partials of the residual GEMM
// that cover those features (the tile's contributors, summed in CTA order so
// the result does not depend on timing); h is written back when partials
// were added (a tile owned whole by one CTA was already added by it).
// kBatch contributors' loads in flight at a time.
template <int kBatch>
__device__ __forceinline__ void resid_gather16(float* __restrict__ h, size_t src, int f0, int d, const ResidPlan& rp,
                                               float (&x)[16]) {
  float* hp = h + src * d + f0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 t = *reinterpret_cast<const float4*>(hp + kRowGroupStride * i);
    x[4 * i] = t.x; x[4 * i + 1] = t.y; x[4 * i + 2] = t.z; x[4 * i + 3] = t.w;
  }
  const int m = (int)src;
  const int mt = m / rp.BN, ml = m - mt * rp.BN;
  const int nt = f0 / 128, fl = f0 - nt * 128;
  const int t = rp.pair ? pair_tile_index(nt >> 1, mt, rp.m_tiles, rp.n_tiles / 2) : nt * rp.m_tiles + mt;
  const int rank = rp.pair ? (nt & 1) : 0;
  Sched sc;
  sc.G = rp.grid;
  sc.KT = rp.k_tiles;
  sc.U = (unsigned)(rp.m_tiles * (rp.pair ? rp.n_tiles / 2 : rp.n_tiles)) * rp.k_tiles;
  const unsigned tu0 = (unsigned)t * rp.k_tiles;
  const int c_first = rp.stream_k ? sc.owner(tu0) : 0;
  const int c_last = rp.stream_k ? sc.owner(tu0 + rp.k_tiles - 1) : 0;
  if (c_first == c_last) return;
  for (int c0 = c_first; c0 <= c_last; c0 += kBatch) {
    float4 buf[kBatch][4];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int cc = c0 + q;
      if (cc <= c_last) {
        const int w = ((unsigned)t == sc.start(cc) / sc.KT) ? 0 : 1;
        const size_t slot = rp.pair ? (size_t)(2 * cc + rank) * 2 + w : (size_t)cc * 2 + w;
        const float* sp = rp.ws + slot * (rp.BN * 128) + (size_t)ml * 128 + fl;
#pragma unroll
        for (int i = 0; i < 4; ++i) buf[q][i] = __ldcg(reinterpret_cast<const float4*>(sp + kRowGroupStride * i));
      }
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q)
      if (c0 + q <= c_last)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[4 * i] += buf[q][i].x;
          x[4 * i + 1] += buf[q][i].y;
          x[4 * i + 2] += buf[q][i].z;
          x[4 * i + 3] += buf[q][i].w;
        }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(hp + kRowGroupStride * i) = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
}

// the bf16 gains of the thread's 16 features, packed in 8 registers
__device__ __forceinline__ void load_gain16(const __nv_bfloat16* __restrict__ g, int f0, uint4 (&gain)[2]) {
  uint2* gw = reinterpret_cast<uint2*>(gain);
#pragma unroll
  for (int i = 0; i < 4; ++i) gw[i] = __ldg(reinterpret_cast<const uint2*>(g + f0 + kRowGroupStride * i));
}

// the thread's 16 outputs: bf16(x * inv_rms * gain)
__device__ __forceinline__ void norm_store16g(const float (&x)[16], float inv, const uint4 (&gain)[2], int f0,
                                              __nv_bfloat16* __restrict__ out) {
  const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(gain);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 g0 = __bfloat1622float2(gb[2 * i]), g1 = __bfloat1622float2(gb[2 * i + 1]);
    __nv_bfloat162 a0 = __floats2bfloat162_rn(x[4 * i] * inv * g0.x, x[4 * i + 1] * inv * g0.y);
    __nv_bfloat162 a1 = __floats2bfloat162_rn(x[4 * i + 2] * inv * g1.x, x[4 * i + 3] * inv * g1.y);
    *reinterpret_cast<uint2*>(out + f0 + kRowGroupStride * i) =
        make_uint2(*reinterpret_cast<uint32_t*>(&a0), *reinterpret_cast<uint32_t*>(&a1));
  }
}

// kMany: a grid of many rows (a refresh), held to 64 registers a thread so
// that four 256-thread CTAs share an SM; otherwise (a block's rows, one CTA
// per SM) four contributors' partials and the gains are in flight together.
template <typename Tg, bool kMany>
__global__ void __launch_bounds__(512, kMany ? 2 : 1) resid_norm_kernel(float* __restrict__ h, const Tg* __restrict__ g,
                                                         __nv_bfloat16* __restrict__ out, int d, float eps,
                                                         int rows_per_seq, int L, int pos_from_state,
                                                         int gather_off, const DevState* st, ResidPlan rp,
                                                         int trigger_early) {
  __shared__ float red[32];
  // the next GEMM may launch once every CTA of this grid has started (they
  // are all resident by then): it becomes resident beside the last ones and
  // requests its first weight tiles meanwhile
  if (trigger_early) pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  size_t src = r;
  if (pos_from_state) {  // gather the block rows from the L rows per sequence of the residual
    const int bi = r / rows_per_seq;
    src = (size_t)bi * L + st->block_start + gather_off + (r - bi * rows_per_seq);
  }
  // blockDim is a whole number of warps; threads past d / 16 hold zeros
  const bool active = threadIdx.x * 16 < d;
  const int f0 = active ? row_f0(threadIdx.x) : 0;
  float x[16];
  uint4 gain[2] = {};
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = 0.f;
  if (active) {
    if (!kMany) load_gain16(g, f0, gain);
    resid_gather16<kMany ? 2 : 4>(h, src, f0, d, rp, x);
    if (kMany) load_gain16(g, f0, gain);  // in flight during the block reduction
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)d + eps);
  if (active) norm_store16g(x, inv, gain, f0, out + (size_t)r * d);
  if (!trigger_early) pdl_trigger();
}

}  // namespace dinfer
