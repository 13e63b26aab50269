// Bidirectional attention of query rows against the dual KV cache.
//
// Every query of the block (or, at a block boundary, every position) attends
// over ALL L cached positions of its sequence -- the prefix, the freshly
// written block slot and the suffix -- with no mask: softmax(q k^T / sqrt(hd)) v.
// Because the QKV epilogue writes the block's fresh K/V into the cache slot of
// the block before this kernel runs, attending over the whole cache equals
// attending over the concatenation [cached prefix | fresh block | cached suffix].
//
// bf16 kernel: one CTA = 64 query rows x one head x one key range; 4 warps of
// 16 rows; K/V chunks of 64 keys double-buffered with cp.async; S = Q K^T and
// O = P V on mma.sync m16n8k16 (bf16 in, fp32 accumulate), online softmax in
// the log2 domain, P rounded to bf16 for the second product.  When the keys
// are split over several CTAs (small grids: a batch-1 block), the splits of
// one (sequence, head, query tile) form a thread-block cluster; each CTA
// leaves its unnormalised partial in its own shared memory and, after a
// cluster barrier, merges a slice of the rows by reading all partials over
// distributed shared memory, in split order.
#pragma once
#include <cooperative_groups.h>

#include "common.cuh"

namespace dinfer {

struct AttnArgs {
  const __nv_bfloat16* q;   // [Mq, d]
  const __nv_bfloat16* k;   // [batch, L, d]   (this layer)
  const __nv_bfloat16* v;
  __nv_bfloat16* o;         // [Mq, d]
  int d, heads, L;
  int rows_per_seq;         // query rows per sequence
  int q_tiles;              // query tiles of 64 per sequence
  int splits, chunks_per_split;  // splits > 1: launched with cluster dims (1, 1, splits)
  float scale_log2;         // log2(e) / sqrt(hd)
};

constexpr int kMaxAttnSplits = 8;  // portable cluster size
constexpr int kAttnThreads = 128;
constexpr int kHd = 128;
constexpr int kKeyChunk = 64;
// 64 rows x 256 B per tile, 16-byte chunks XOR-swizzled by (row & 7)
constexpr int kAttnTileBytes = 64 * kHd * 2;
constexpr int kAttnStages = 3;                                     // K/V chunks in flight
constexpr int kAttnSmem = kAttnTileBytes * (1 + 2 * kAttnStages);  // Q + stages x (K, V): 112 KB, 2 CTAs/SM

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a 64x128 bf16 tile
  return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Load a 64-row x 128-col bf16 tile (rows >= valid_rows zero-filled).
__device__ __forceinline__ void load_tile_async(uint32_t sbase, const __nv_bfloat16* g, size_t row_stride,
                                                int valid_rows) {
  // 64 rows x 16 chunks = 1024 chunks / 128 threads = 8 each
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int idx = threadIdx.x + i * kAttnThreads;
    const int r = idx >> 4, c = idx & 15;
    const bool ok = r < valid_rows;
    const __nv_bfloat16* src = g + (ok ? (size_t)r * row_stride : 0) + c * 8;
    cp_async16(sbase + swz(r, c), src, ok);
  }
}

__global__ void __launch_bounds__(kAttnThreads)
    attn_bf16_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t s_q = smem_u32(sm);
  // stage i: K at s_q + (1 + 2i) tiles, V at s_q + (2 + 2i) tiles
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int qt = blockIdx.x % a.q_tiles;
  const int bi = blockIdx.x / a.q_tiles;
  const int head = blockIdx.y;
  const int split = blockIdx.z;
  const int row0 = qt * 64;                       // first query row inside the sequence
  const int q_valid = min(64, a.rows_per_seq - row0);
  const size_t qrow_base = (size_t)bi * a.rows_per_seq + row0;
  const __nv_bfloat16* qg = a.q + qrow_base * a.d + head * kHd;
  const __nv_bfloat16* kg = a.k + (size_t)bi * a.L * a.d + head * kHd;
  const __nv_bfloat16* vg = a.v + (size_t)bi * a.L * a.d + head * kHd;
  const int n_chunks = (a.L + kKeyChunk - 1) / kKeyChunk;
  const int c_begin = split * a.chunks_per_split;
  const int c_end = min(n_chunks, c_begin + a.chunks_per_split);

  pdl_wait();
  auto s_k = [&](int st) { return s_q + (uint32_t)(1 + 2 * st) * kAttnTileBytes; };
  auto s_v = [&](int st) { return s_q + (uint32_t)(2 + 2 * st) * kAttnTileBytes; };
  auto load_chunk = [&](int c, int st) {
    const int k0 = c * kKeyChunk;
    load_tile_async(s_k(st), kg + (size_t)k0 * a.d, a.d, min(kKeyChunk, a.L - k0));
    load_tile_async(s_v(st), vg + (size_t)k0 * a.d, a.d, min(kKeyChunk, a.L - k0));
  };
  // prologue: group 0 = Q + chunk 0, groups 1 .. kAttnStages-2 = the next chunks
  load_tile_async(s_q, qg, a.d, q_valid);
#pragma unroll
  for (int i = 0; i < kAttnStages - 1; ++i) {
    if (c_begin + i < c_end) load_chunk(c_begin + i, i);
    cp_async_commit();
  }
  cp_async_wait<kAttnStages - 2>();
  __syncthreads();

  // Q fragments for this warp's 16 rows, all 8 k-steps of hd
  uint32_t qf[8][4];
  {
    const int r = warp * 16 + (lane & 15);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int chunk = ks * 2 + (lane >> 4);
      ldsm_x4(s_q + swz(r, chunk), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
    }
  }
  float oacc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

  for (int c = c_begin; c < c_end; ++c) {
    const int buf = (c - c_begin) % kAttnStages;
    // refill the stage consumed in the previous iteration with chunk c + kAttnStages - 1
    const int cn = c + kAttnStages - 1;
    if (cn < c_end) load_chunk(cn, (cn - c_begin) % kAttnStages);
    cp_async_commit();
    cp_async_wait<kAttnStages - 1>();
    __syncthreads();

    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {        // pairs of key n-tiles (16 keys)
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {      // hd k-steps of 16
        const int key = kp * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int chunk = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(s_k(buf) + swz(key, chunk), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * kp], qf[ks], b0, b1);
        mma_bf16_16816(s[2 * kp + 1], qf[ks], b2, b3);
      }
    }
    // online softmax (rows g and g+8 of this warp)
    const int kbase = c * kKeyChunk;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kbase + i * 8 + 2 * t4 + (e & 1);
        const float val = (key < a.L) ? s[i][e] * a.scale_log2 : -INFINITY;
        s[i][e] = val;
        mx[e >> 1] = fmaxf(mx[e >> 1], val);
      }
    }
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mnew = fmaxf(m_r[h], mx[h]);
      alpha[h] = (m_r[h] == -INFINITY) ? 0.f : exp2f(m_r[h] - mnew);
      m_r[h] = mnew;
    }
    uint32_t pf[4][4];  // P as A fragments: 4 key k-steps of 16
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mm = m_r[e >> 1];
        p[e] = (s[i][e] == -INFINITY) ? 0.f : bf16r(exp2f(s[i][e] - mm));
        rs[e >> 1] += p[e];
      }
      const int kstep = i >> 1, hi = i & 1;
      pf[kstep][hi * 2 + 0] = pack_bf16(p[0], p[1]);
      pf[kstep][hi * 2 + 1] = pack_bf16(p[2], p[3]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) l_r[h] = l_r[h] * alpha[h] + rs[h];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      oacc[i][0] *= alpha[0];
      oacc[i][1] *= alpha[0];
      oacc[i][2] *= alpha[1];
      oacc[i][3] *= alpha[1];
    }
    // O += P V: k = keys (4 steps of 16), n = hd (16 tiles of 8)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int np = 0; np < 8; ++np) {  // pairs of hd n-tiles (16 cols)
        const int key = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int chunk = np * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(s_v(buf) + swz(key, chunk), b0, b1, b2, b3);
        mma_bf16_16816(oacc[2 * np], pf[ks], b0, b1);
        mma_bf16_16816(oacc[2 * np + 1], pf[ks], b2, b3);
      }
    }
    __syncthreads();
  }
  // row sums across the quad
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 1);
    l_r[h] += __shfl_xor_sync(0xffffffffu, l_r[h], 2);
  }
  const int r_lo = warp * 16 + g, r_hi = r_lo + 8;  // rows inside the tile
  if (threadIdx.x == 0) pdl_trigger();
  if (a.splits == 1) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = h ? r_hi : r_lo;
      if (r < q_valid) {
        const float inv = 1.f / l_r[h];
        __nv_bfloat16* og = a.o + (qrow_base + r) * a.d + head * kHd;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = i * 8 + 2 * t4;
          *reinterpret_cast<__nv_bfloat162*>(og + col) =
              __floats2bfloat162_rn(oacc[i][2 * h] * inv, oacc[i][2 * h + 1] * inv);
        }
      }
    }
    return;
  }
  // ---- split keys: partials stay in shared memory, merged across the cluster ----
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  float* po = reinterpret_cast<float*>(sm + kAttnTileBytes);          // [64][128] fp32, over the K/V buffers
  float* pml = po + 64 * kHd;                                         // [64][2]
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = h ? r_hi : r_lo;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = i * 8 + 2 * t4;
      *reinterpret_cast<float2*>(po + r * kHd + col) = make_float2(oacc[i][2 * h], oacc[i][2 * h + 1]);
    }
    if (t4 == 0) {
      pml[r * 2] = m_r[h];
      pml[r * 2 + 1] = l_r[h];
    }
  }
  cluster.sync();
  const int rank = (int)cluster.block_rank();
  const int per = (64 + a.splits - 1) / a.splits;
  const int r0 = rank * per, r1 = min(min(64, r0 + per), q_valid);
  for (int idx = threadIdx.x; idx < (r1 - r0) * (kHd / 4); idx += kAttnThreads) {
    const int r = r0 + idx / (kHd / 4), c4 = (idx % (kHd / 4)) * 4;
    float ms[kMaxAttnSplits], ls[kMaxAttnSplits];
    float4 os[kMaxAttnSplits];
    float mmax = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < kMaxAttnSplits; ++sp) {
      if (sp < a.splits) {
        const float* rpml = cluster.map_shared_rank(pml, sp);
        const float* rpo = cluster.map_shared_rank(po, sp);
        ms[sp] = rpml[r * 2];
        ls[sp] = rpml[r * 2 + 1];
        os[sp] = *reinterpret_cast<const float4*>(rpo + r * kHd + c4);
        mmax = fmaxf(mmax, ms[sp]);
      }
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, lsum = 0.f;
#pragma unroll
    for (int sp = 0; sp < kMaxAttnSplits; ++sp) {
      if (sp < a.splits && ms[sp] != -INFINITY) {
        const float w = exp2f(ms[sp] - mmax);
        lsum += ls[sp] * w;
        acc[0] += os[sp].x * w;
        acc[1] += os[sp].y * w;
        acc[2] += os[sp].z * w;
        acc[3] += os[sp].w * w;
      }
    }
    const float inv = 1.f / lsum;
    __nv_bfloat16* og = a.o + (qrow_base + r) * a.d + head * kHd + c4;
    *reinterpret_cast<__nv_bfloat162*>(og) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    *reinterpret_cast<__nv_bfloat162*>(og + 2) = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  }
  cluster.sync();  // keep this CTA's shared memory alive until every peer has read it
}

// ---------------------------------------------------------------------------
// fp32 SIMT attention (fp32 models): one CTA per (query row, head)
// ---------------------------------------------------------------------------
struct AttnF32Args {
  const float* q;   // [Mq, d]
  const float* k;   // [batch, L, d]
  const float* v;
  float* o;         // [Mq, d]
  int d, heads, hd, L, rows_per_seq;
  float scale;
};

__global__ void attn_f32_kernel(const AttnF32Args a) {
  extern __shared__ float sc[];  // [L] scores, then [hd] query
  __shared__ float red[32];
  const int m = blockIdx.x, head = blockIdx.y;
  const int bi = m / a.rows_per_seq;
  float* qs = sc + a.L;
  for (int i = threadIdx.x; i < a.hd; i += blockDim.x) qs[i] = a.q[(size_t)m * a.d + head * a.hd + i];
  __syncthreads();
  const float* kb = a.k + (size_t)bi * a.L * a.d + head * a.hd;
  const float* vb = a.v + (size_t)bi * a.L * a.d + head * a.hd;
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < a.L; j += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < a.hd; ++i) acc = fmaf(qs[i], kb[(size_t)j * a.d + i], acc);
    acc *= a.scale;
    sc[j] = acc;
    mx = fmaxf(mx, acc);
  }
  mx = warp_max(mx);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  mx = red[0];
  __syncthreads();
  float sum = 0.f;
  for (int j = threadIdx.x; j < a.L; j += blockDim.x) {
    const float e = expf(sc[j] - mx);
    sc[j] = e;
    sum += e;
  }
  sum = warp_sum(sum);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = 1.f / red[0];
  for (int i = threadIdx.x; i < a.hd; i += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < a.L; ++j) acc = fmaf(sc[j], vb[(size_t)j * a.d + i], acc);
    a.o[(size_t)m * a.d + head * a.hd + i] = acc * inv;
  }
}

}  // namespace dinfer
