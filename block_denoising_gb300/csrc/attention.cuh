// Bidirectional attention of query rows against the dual KV cache, fp32
// models (SIMT).  Every query row attends over ALL L cached positions of its
// sequence -- the prefix, the freshly written block slot and the suffix --
// with no mask: softmax(q k^T / sqrt(hd)) v.  Because the QKV step writes the
// block's fresh K/V into the cache slot of the block before this kernel runs,
// attending over the whole cache equals attending over the concatenation
// [cached prefix | fresh block | cached suffix].  The bf16 path runs on the
// tensor cores (attention_tc.cuh).
#pragma once
#include "common.cuh"

namespace dinfer {

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
