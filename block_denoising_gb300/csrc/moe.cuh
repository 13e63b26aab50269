// Mixture-of-experts FFN (OLMoE-style routing, LLaDA-MoE shapes).
//
//   p = softmax(x_hat W_r^T) over the E experts; the top-k experts of each row
//   by p (ties to the lower expert index), weights not renormalised;
//   h += sum over the row's experts of p_e * (silu(x_hat W_g,e^T) * x_hat W_u,e^T) W_d,e^T
//
// Device pipeline: router logits (tcgen05 GEMM, fp32 out) -> moe_topk_kernel
// (one warp per row) -> moe_count_kernel + moe_scan_kernel (or, for at most
// 256 rows and 64 experts, moe_route_tables_kernel) + moe_scatter_kernel (a
// counting sort of the (row, expert) pairs by expert, rows in ascending
// order inside an expert, so the permutation does not depend on timing) ->
// grouped gate/up and down GEMMs over the permuted rows (gemm_tc_kernel in
// grouped mode, tile tables written here) -> moe_combine_norm_kernel
// (weighted sum of the row's k expert outputs in slot order, residual add,
// next RMSNorm).
#pragma once
#include "common.cuh"

namespace dinfer {

constexpr int kMoeMaxK = 8;
constexpr int kMoeMaxE = 256;
constexpr int kMoeChunk = 256;  // rows per counting chunk

// top-k of softmax(logits) per row; one warp per row, E <= 64 (2 per lane)
__global__ void moe_topk_kernel(const float* __restrict__ logits, int M, int E, int K, int* __restrict__ topk_id,
                                float* __restrict__ topk_w) {
  pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp < M) {
    const float* l = logits + (size_t)warp * E;
    float v0 = lane < E ? l[lane] : -INFINITY;
    float v1 = lane + 32 < E ? l[lane + 32] : -INFINITY;
    const float mx = warp_max(fmaxf(v0, v1));
    const float e0 = lane < E ? expf(v0 - mx) : 0.f, e1 = lane + 32 < E ? expf(v1 - mx) : 0.f;
    const float inv = 1.f / warp_sum(e0 + e1);
    // selection by logit (monotone in p), ties to the lower expert
    float c0 = v0, c1 = v1;
    for (int k = 0; k < K; ++k) {
      float bv = c0;
      int bi = lane;
      if (c1 > bv) { bv = c1; bi = lane + 32; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) {
        topk_id[(size_t)warp * K + k] = bi;
        topk_w[(size_t)warp * K + k] = expf(bv - mx) * inv;
      }
      if (bi == lane) c0 = -INFINITY;
      if (bi == lane + 32) c1 = -INFINITY;
    }
  }
  pdl_trigger();
}

// Per chunk of 256 rows: for every expert, the rank of each selecting row
// among the chunk's selecting rows (row order) and the chunk's count.
__global__ void __launch_bounds__(kMoeChunk) moe_count_kernel(const int* __restrict__ topk_id, int M, int E, int K,
                                                             int* __restrict__ local_rank, int* __restrict__ chunk_cnt) {
  __shared__ int warp_tot[kMoeChunk / 32];
  pdl_wait();
  const int r = blockIdx.x * kMoeChunk + threadIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ids[kMoeMaxK];
#pragma unroll
  for (int k = 0; k < kMoeMaxK; ++k) ids[k] = (r < M && k < K) ? topk_id[(size_t)r * K + k] : -1;
  for (int e = 0; e < E; ++e) {
    int slot = -1;
#pragma unroll
    for (int k = 0; k < kMoeMaxK; ++k)
      if (ids[k] == e) slot = k;
    const unsigned bal = __ballot_sync(0xffffffffu, slot >= 0);
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kMoeChunk / 32; ++w) {
      const int c = warp_tot[w];
      before += w < warp ? c : 0;
      total += c;
    }
    if (slot >= 0) local_rank[(size_t)r * K + slot] = before + __popc(bal & ((1u << lane) - 1u));
    if (threadIdx.x == 0) chunk_cnt[(size_t)blockIdx.x * E + e] = total;
    __syncthreads();
  }
  pdl_trigger();
}

// One CTA: chunk bases per expert, expert row offsets, and the tile tables of
// the two grouped GEMMs (n-tiles per expert x token tiles of that expert).
__global__ void moe_scan_kernel(const int* __restrict__ chunk_cnt, int n_chunks, int E, int* __restrict__ chunk_base,
                                int* __restrict__ row_off, int* __restrict__ tile_cum_gu, int* __restrict__ tile_cum_dn,
                                int bn_gu, int nt_gu, int bn_dn, int nt_dn, DevState* st) {
  __shared__ int tot[kMoeMaxE];
  pdl_wait();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int acc = 0;
    for (int c = 0; c < n_chunks; ++c) {
      chunk_base[(size_t)c * E + e] = acc;
      acc += chunk_cnt[(size_t)c * E + e];
    }
    tot[e] = acc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int ro = 0, tg = 0, td = 0, touched = 0;
    for (int e = 0; e < E; ++e) {
      touched += tot[e] > 0;
      row_off[e] = ro;
      tile_cum_gu[e] = tg;
      tile_cum_dn[e] = td;
      ro += tot[e];
      tg += ((tot[e] + bn_gu - 1) / bn_gu) * nt_gu;
      td += ((tot[e] + bn_dn - 1) / bn_dn) * nt_dn;
    }
    row_off[E] = ro;
    tile_cum_gu[E] = tg;
    tile_cum_dn[E] = td;
    atomicAdd(&st->moe_touched, (uint32_t)touched);
  }
  pdl_trigger();
}

// The counting sort of a block's rows (M <= kMoeChunk, E <= 64) in one CTA,
// with the results of moe_count_kernel + moe_scan_kernel for a single chunk:
// per expert a bitmask of the rows that select it (set with atomicOr, whose
// result does not depend on the order), a row's rank among the expert's rows
// = the population count of the mask below the row (ascending row order),
// then exclusive scans of the counts and tile counts over the experts (one
// warp, two experts a lane).
__global__ void __launch_bounds__(kMoeChunk) moe_route_tables_kernel(
    const int* __restrict__ topk_id, int M, int E, int K, int* __restrict__ local_rank, int* __restrict__ chunk_base,
    int* __restrict__ row_off, int* __restrict__ tile_cum_gu, int* __restrict__ tile_cum_dn, int bn_gu, int nt_gu,
    int bn_dn, int nt_dn, DevState* st) {
  constexpr int W = kMoeChunk / 32;  // mask words per expert
  __shared__ uint32_t bits[64 * W];
  __shared__ int cnt[64];
  pdl_wait();
  const int r = threadIdx.x;
  for (int i = r; i < E * W; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  int ids[kMoeMaxK];
#pragma unroll
  for (int k = 0; k < kMoeMaxK; ++k) ids[k] = (r < M && k < K) ? topk_id[(size_t)r * K + k] : -1;
#pragma unroll
  for (int k = 0; k < kMoeMaxK; ++k)
    if (ids[k] >= 0) atomicOr(&bits[ids[k] * W + (r >> 5)], 1u << (r & 31));
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kMoeMaxK; ++k) {
    if (ids[k] < 0) continue;
    const uint32_t* b = bits + ids[k] * W;
    int rank = __popc(b[r >> 5] & ((1u << (r & 31)) - 1u));
    for (int w = 0; w < (r >> 5); ++w) rank += __popc(b[w]);
    local_rank[(size_t)r * K + k] = rank;
  }
  if (r < E) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) c += __popc(bits[r * W + w]);
    cnt[r] = c;
    chunk_base[r] = 0;
  }
  __syncthreads();
  if (r < 32) {
    const int e0 = 2 * r, e1 = 2 * r + 1;
    const int c0 = e0 < E ? cnt[e0] : 0, c1 = e1 < E ? cnt[e1] : 0;
    const int g0 = ((c0 + bn_gu - 1) / bn_gu) * nt_gu, g1 = ((c1 + bn_gu - 1) / bn_gu) * nt_gu;
    const int d0 = ((c0 + bn_dn - 1) / bn_dn) * nt_dn, d1 = ((c1 + bn_dn - 1) / bn_dn) * nt_dn;
    int sc = c0 + c1, sg = g0 + g1, sd = d0 + d1;  // inclusive scans over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tc = __shfl_up_sync(0xffffffffu, sc, o), tg = __shfl_up_sync(0xffffffffu, sg, o);
      const int td = __shfl_up_sync(0xffffffffu, sd, o);
      if (r >= o) {
        sc += tc;
        sg += tg;
        sd += td;
      }
    }
    if (e0 < E) {
      row_off[e0] = sc - c0 - c1;
      tile_cum_gu[e0] = sg - g0 - g1;
      tile_cum_dn[e0] = sd - d0 - d1;
    }
    if (e1 < E) {
      row_off[e1] = sc - c1;
      tile_cum_gu[e1] = sg - g1;
      tile_cum_dn[e1] = sd - d1;
    }
    if (r == 31) {
      row_off[E] = sc;
      tile_cum_gu[E] = sg;
      tile_cum_dn[E] = sd;
    }
    // experts that received rows, for the measured byte count
    const int touched = __popc(__ballot_sync(0xffffffffu, c0 > 0)) + __popc(__ballot_sync(0xffffffffu, c1 > 0));
    if (r == 0) atomicAdd(&st->moe_touched, (uint32_t)touched);
  }
  pdl_trigger();
}

// One CTA per (row, slot): its permuted position, and a copy of the row's
// normed input into the permuted operand of the gate/up GEMM.
__global__ void moe_scatter_kernel(const __nv_bfloat16* __restrict__ xn, int d, int M, int E, int K,
                                   const int* __restrict__ topk_id, const int* __restrict__ local_rank,
                                   const int* __restrict__ chunk_base, const int* __restrict__ row_off,
                                   int* __restrict__ inv, __nv_bfloat16* __restrict__ x_perm) {
  pdl_wait();
  const int pair = blockIdx.x;
  const int r = pair / K;
  const int e = topk_id[pair];
  const int dst = row_off[e] + chunk_base[(size_t)(r / kMoeChunk) * E + e] + local_rank[pair];
  if (threadIdx.x == 0) inv[pair] = dst;
  const uint4* src = reinterpret_cast<const uint4*>(xn + (size_t)r * d);
  uint4* out = reinterpret_cast<uint4*>(x_perm + (size_t)dst * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) out[i] = src[i];
  pdl_trigger();
}

// h[src] += sum_k w[r, k] * y[inv[r, k]] (slot order); then, if out != NULL,
// out[r] = bf16(RMSNorm(h[src]) * g).  One CTA per output row, whole warps
// covering d / 16 threads (16 features each).
template <typename Tg>
__global__ void __launch_bounds__(512) moe_combine_norm_kernel(float* __restrict__ h, const float* __restrict__ y,
                                                               const float* __restrict__ topk_w,
                                                               const int* __restrict__ inv, int K,
                                                               const Tg* __restrict__ g,
                                                               __nv_bfloat16* __restrict__ out, int d, float eps,
                                                               int rows_per_seq, int L, int gather,
                                                               int gather_off, const DevState* st) {
  __shared__ float red[32];
  pdl_wait();
  const int r = blockIdx.x;
  size_t src = r;
  if (gather) {
    const int bi = r / rows_per_seq;
    src = (size_t)bi * L + st->block_start + gather_off + (r - bi * rows_per_seq);
  }
  // blockDim is a whole number of warps; threads past d / 16 hold zeros.
  // Features in the row-kernel layout (row_f0, kRowGroupStride).
  const bool active = threadIdx.x * 16 < d;
  const int f0 = active ? row_f0(threadIdx.x) : 0;
  float* hp = h + src * d + f0;
  float x[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = 0.f;
  if (active) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 t = *reinterpret_cast<const float4*>(hp + kRowGroupStride * i);
      x[4 * i] = t.x; x[4 * i + 1] = t.y; x[4 * i + 2] = t.z; x[4 * i + 3] = t.w;
    }
  }
  for (int k = 0; k < K && active; ++k) {
    const float w = topk_w[src * K + k];
    const float* yp = y + (size_t)inv[src * K + k] * d + f0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(yp + kRowGroupStride * i));
      x[4 * i] = fmaf(w, t.x, x[4 * i]);
      x[4 * i + 1] = fmaf(w, t.y, x[4 * i + 1]);
      x[4 * i + 2] = fmaf(w, t.z, x[4 * i + 2]);
      x[4 * i + 3] = fmaf(w, t.w, x[4 * i + 3]);
    }
  }
  if (active) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(hp + kRowGroupStride * i) = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
  }
  if (out == nullptr) {
    pdl_trigger();
    return;
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
  const float inv_rms = rsqrtf(red[0] / (float)d + eps);
  if (active) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int f = f0 + kRowGroupStride * i;
      __nv_bfloat162 a0 = __floats2bfloat162_rn(x[4 * i] * inv_rms * (float)g[f], x[4 * i + 1] * inv_rms * (float)g[f + 1]);
      __nv_bfloat162 a1 =
          __floats2bfloat162_rn(x[4 * i + 2] * inv_rms * (float)g[f + 2], x[4 * i + 3] * inv_rms * (float)g[f + 3]);
      *reinterpret_cast<uint2*>(out + (size_t)r * d + f) =
          make_uint2(*reinterpret_cast<uint32_t*>(&a0), *reinterpret_cast<uint32_t*>(&a1));
    }
  }
  pdl_trigger();
}

}  // namespace dinfer
