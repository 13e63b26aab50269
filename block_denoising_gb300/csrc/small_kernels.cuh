// Row-wise kernels of the denoising iteration (embedding gather, RMSNorm),
// the fp32 (SIMT FFMA, no TF32) GEMM / epilogue / LM-head variants used by
// fp32 models, and the device-side loop-state kernels.
#pragma once
#include "common.cuh"
#include "decode.cuh"

namespace dinfer {

// Row r of a rows x d activation belongs to sequence r / rows_per_seq at
// absolute position base + row_off + r % rows_per_seq, where base is the
// current block start (pos_from_state) or 0, and row_off a fixed offset (the
// first recomputed position of a window; 0 for the block or all positions).
struct RowMap {
  int rows_per_seq, L, pos_from_state;
  int row_off;
  __device__ __forceinline__ size_t seq_index(int r, const DevState* st) const {
    const int bi = r / rows_per_seq;
    const int base = (pos_from_state ? st->block_start : 0) + row_off;
    return (size_t)bi * L + base + (r - bi * rows_per_seq);
  }
};

// h[r, :] = E[ids[seq_index(r)], :]  (fp32 residual stream)
template <typename T>
__global__ void embed_kernel(const T* __restrict__ E, const int32_t* __restrict__ ids, float* __restrict__ h,
                             int rows, int d, int vocab, RowMap rm, DevState* st) {
  pdl_wait();
  const int r = blockIdx.x;
  if (r >= rows) return;
  int id = ids[rm.seq_index(r, st)];
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) set_status(st, ST_BAD_TOKEN);
    id = 0;
  }
  const T* src = E + (size_t)id * d;
  float* dst = h + (size_t)r * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) dst[i] = (float)src[i];
  pdl_trigger();
}

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// out[r, :] = h[src(r), :] / sqrt(mean(h^2) + eps) * g, rounded to the GEMM
// input type.  src(r) = seq_index(r) when gather != 0 (block rows of a
// full-sequence residual), else r.  One CTA of 256 threads per row; rows of
// up to 8192 values are held in registers (float4) so every load is issued
// before the reduction.
__device__ __forceinline__ void load4(const float* g, int k, float (&w)[4]) {
  const float4 t = reinterpret_cast<const float4*>(g)[k];
  w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* g, int k, float (&w)[4]) {
  const uint2 t = reinterpret_cast<const uint2*>(g)[k];
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&t.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&t.y);
  w[0] = __low2float(a); w[1] = __high2float(a); w[2] = __low2float(b); w[3] = __high2float(b);
}
__device__ __forceinline__ void store4(float* o, int k, float a, float b, float c, float d) {
  reinterpret_cast<float4*>(o)[k] = make_float4(a, b, c, d);
}
__device__ __forceinline__ void store4(__nv_bfloat16* o, int k, float a, float b, float c, float d) {
  __nv_bfloat162 x = __floats2bfloat162_rn(a, b), y = __floats2bfloat162_rn(c, d);
  uint2 t;
  t.x = *reinterpret_cast<uint32_t*>(&x);
  t.y = *reinterpret_cast<uint32_t*>(&y);
  reinterpret_cast<uint2*>(o)[k] = t;
}

template <typename Tg, typename To>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ h, const Tg* __restrict__ g,
                                                      To* __restrict__ out, int rows, int d, float eps, int gather,
                                                      RowMap rm, const DevState* st) {
  pdl_wait();
  const int r = blockIdx.x;
  if (r >= rows) return;
  const size_t src = gather ? rm.seq_index(r, st) : (size_t)r;
  const float* x = h + src * d;
  To* o = out + (size_t)r * d;
  __shared__ float red[32];
  const int n4 = d >> 2;
  const bool vec = (d & 3) == 0 && n4 <= 8 * 256;
  float v[8][4];
  float ss = 0.f;
  if (vec) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = threadIdx.x + i * 256;
      if (k < n4) {
        const float4 t = reinterpret_cast<const float4*>(x)[k];
        v[i][0] = t.x; v[i][1] = t.y; v[i][2] = t.z; v[i][3] = t.w;
        ss = fmaf(t.x, t.x, fmaf(t.y, t.y, fmaf(t.z, t.z, fmaf(t.w, t.w, ss))));
      }
    }
  } else {
    for (int i = threadIdx.x; i < d; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = rsqrtf(red[0] / (float)d + eps);
  if (vec) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = threadIdx.x + i * 256;
      if (k < n4) {
        float w[4];
        load4(g, k, w);
        store4(o, k, v[i][0] * inv * w[0], v[i][1] * inv * w[1], v[i][2] * inv * w[2], v[i][3] * inv * w[3]);
      }
    }
  } else {
    for (int i = threadIdx.x; i < d; i += blockDim.x) o[i] = from_float<To>(x[i] * inv * (float)g[i]);
  }
  pdl_trigger();
}

// ---------------------------------------------------------------------------
// fp32 SIMT GEMM: Y[m, n] (+)= sum_k X[m, k] W[n, k]; 64x64 tiles, 256 threads
// ---------------------------------------------------------------------------
__global__ void gemm_f32_kernel(const float* __restrict__ X, const float* __restrict__ W, float* __restrict__ Y,
                                int M, int N, int K, int ldy, int accumulate) {
  __shared__ float xs[16][64 + 1];
  __shared__ float ws[16][64 + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 16 * 64; i += 256) {
      const int kk = i & 15, rr = i >> 4;
      xs[kk][rr] = (m0 + rr < M && k0 + kk < K) ? X[(size_t)(m0 + rr) * K + k0 + kk] : 0.f;
      ws[kk][rr] = (n0 + rr < N && k0 + kk < K) ? W[(size_t)(n0 + rr) * K + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float xv[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv[i] = xs[kk][ty * 4 + i];
        wv[i] = ws[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) {
        float* y = Y + (size_t)m * ldy + n;
        *y = accumulate ? *y + acc[i][j] : acc[i][j];
      }
    }
}

// qkv [rows, 3d] fp32 -> q [rows, d] (RoPE), cache K (RoPE), V at the rows' positions
__global__ void rope_cache_f32_kernel(const float* __restrict__ qkv, float* __restrict__ q, float* __restrict__ kc,
                                      float* __restrict__ vc, const float* __restrict__ cosv,
                                      const float* __restrict__ sinv, int rows, int d, int hd, RowMap rm,
                                      const DevState* st) {
  const int r = blockIdx.x;
  if (r >= rows) return;
  const size_t si = rm.seq_index(r, st);
  const int bi = r / rm.rows_per_seq;
  const int pos = (int)(si - (size_t)bi * rm.L);
  const int half = hd / 2;
  const float* src = qkv + (size_t)r * 3 * d;
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    const int i = n % hd, j = i % half;
    const int partner = (i < half) ? n + half : n - half;
    const float cs = cosv[pos * half + j], sn = sinv[pos * half + j];
    const float q1 = src[n], q2 = src[partner];
    const float k1 = src[d + n], k2 = src[d + partner];
    q[(size_t)r * d + n] = (i < half) ? q1 * cs - q2 * sn : q1 * cs + q2 * sn;
    kc[si * d + n] = (i < half) ? k1 * cs - k2 * sn : k1 * cs + k2 * sn;
    vc[si * d + n] = src[2 * d + n];
  }
}

// act[r, j] = silu(gu[r, j]) * gu[r, f + j]
__global__ void swiglu_f32_kernel(const float* __restrict__ gu, float* __restrict__ act, int rows, int f) {
  const size_t n = (size_t)rows * f;
  for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < n; idx += (size_t)gridDim.x * blockDim.x) {
    const size_t r = idx / f, j = idx - r * f;
    const float g = gu[r * 2 * f + j], u = gu[r * 2 * f + f + j];
    act[idx] = g / (1.f + expf(-g)) * u;
  }
}

// fp32 LM head with online softmax: each CTA a vocabulary slice, 128 threads
// (one vocabulary row each per tile), rows x d normed input in shared memory.
struct LmF32Args {
  const float* x;   // [M, d]
  const float* W;   // [V, d]
  int M, d, V, mask_id;
  float scale;
  float* logits;    // optional [M, V]
  DecodeArgs dec;
};

__global__ void __launch_bounds__(128) lmhead_f32_kernel(const LmF32Args a) {
  extern __shared__ float xs[];            // [M * d]
  __shared__ float st_m[1024], st_s[1024];
  __shared__ int st_a[1024];
  __shared__ int last_sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < a.M * a.d; i += 128) xs[i] = a.x[i];
  for (int m = tid; m < a.M; m += 128) {
    st_m[m] = -INFINITY;
    st_s[m] = 0.f;
    st_a[m] = 0x7fffffff;
  }
  __syncthreads();
  const float sl2 = a.scale * 1.4426950408889634f;
  const int tiles = (a.V + 127) / 128;
  const int t0 = (int)((long long)tiles * blockIdx.x / gridDim.x);
  const int t1 = (int)((long long)tiles * (blockIdx.x + 1) / gridDim.x);
  __shared__ float w_m[4], w_s[4];
  __shared__ int w_a[4];
  for (int t = t0; t < t1; ++t) {
    const int n = t * 128 + tid;
    const bool valid = n < a.V && n != a.mask_id;
    const float* wr = a.W + (size_t)min(n, a.V - 1) * a.d;
    for (int m = 0; m < a.M; ++m) {
      float acc = 0.f;
      const float* xr = xs + (size_t)m * a.d;
      for (int k = 0; k < a.d; ++k) acc = fmaf(xr[k], wr[k], acc);
      if (a.logits && n < a.V) a.logits[(size_t)m * a.V + n] = valid ? acc * a.scale : -INFINITY;
      const float tv = valid ? acc * sl2 : -INFINITY;
      const float wm = warp_max(tv);
      const float e = (valid && wm != -INFINITY) ? exp2f(tv - wm) : 0.f;
      const float wsum = warp_sum(e);
      const unsigned hit = __ballot_sync(0xffffffffu, valid && tv == wm);
      if (lane == 0) {
        w_m[warp] = wm;
        w_s[warp] = wsum;
        w_a[warp] = hit ? (t * 128 + warp * 32 + __ffs(hit) - 1) : 0x7fffffff;
      }
      __syncthreads();
      if (tid == 0) {
        SoftmaxState s{st_m[m], st_s[m], st_a[m]};
        for (int q = 0; q < 4; ++q) s = sm_merge(s, SoftmaxState{w_m[q], w_s[q], w_a[q]});
        st_m[m] = s.m;
        st_s[m] = s.s;
        st_a[m] = s.a;
      }
      __syncthreads();
    }
  }
  SoftmaxState* part = a.dec.partials + (size_t)blockIdx.x * a.M;
  for (int m = tid; m < a.M; m += 128) {
    part[m].m = st_m[m];
    part[m].s = st_s[m];
    part[m].a = st_a[m];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(a.dec.ticket, 1);
    last_sh = (prev == (int)gridDim.x - 1);
    if (last_sh) *a.dec.ticket = 0;
  }
  __syncthreads();
  if (!last_sh) return;
  __threadfence();
  finalize_and_commit(a.dec, tid, st_a, st_s, 1);
}

// ---------------------------------------------------------------------------
// loop state
// ---------------------------------------------------------------------------
// x = prompt | mask_id ..., mask = 0 | 1 ...; block 0 starts at P
__global__ void init_sequence_kernel(const int32_t* __restrict__ prompt, int32_t* __restrict__ ids,
                                     uint8_t* __restrict__ mask, int batch, int P, int L, int mask_id,
                                     DevState* st, int n_blocks) {
  const size_t n = (size_t)batch * L;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int b = (int)(i / L), p = (int)(i - (size_t)b * L);
    ids[i] = p < P ? prompt[(size_t)b * P + p] : mask_id;
    mask[i] = p < P ? 0 : 1;
  }
  // blocks skipped after end-of-sequence report no iterations
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < n_blocks && k < kMaxBlocks; k += gridDim.x * blockDim.x)
    st->iters_per_block[k] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    st->block_start = P;
    st->block_index = 0;
    st->n_blocks = n_blocks;
    st->iteration = 0;
    st->total_iterations = 0;
    st->refreshes = 0;
    st->status = 0;
    st->diag[0] = 0;
    st->any_masked = 1;
    st->any_left = 1;
  }
}

// start of a block: the refresh is iteration 1
__global__ void begin_block_kernel(DevState* st) {
  st->iteration = 0;
  st->refreshes += 1;
}

// inner loop condition after the refresh: iterate while masks remain
__global__ void set_inner_cond_kernel(DevState* st, cudaGraphConditionalHandle h) {
  cudaGraphSetConditional(h, (st->any_masked && st->status == 0u) ? 1u : 0u);
}

// End of a block (one CTA of 256 threads).  With an end-of-sequence id set,
// a sequence whose finished block holds it ends there: its later positions
// become the id, unmasked.  Then move to the next block; the outer loop
// continues while blocks remain and some sequence has masked positions left.
__global__ void __launch_bounds__(256) advance_block_kernel(DevState* st, int B, cudaGraphConditionalHandle h,
                                                            int use_cond, int32_t* __restrict__ ids,
                                                            uint8_t* __restrict__ mask, int batch, int L) {
  const int s0 = st->block_start, eos = st->eos_id;
  const int tail = s0 + B;
  int left = 0;
  for (int b = 0; b < batch; ++b) {
    int32_t* x = ids + (size_t)b * L;
    uint8_t* m = mask + (size_t)b * L;
    int found = 0;
    if (eos >= 0)
      for (int r = threadIdx.x; r < B; r += blockDim.x) found |= (x[s0 + r] == eos);
    if (__syncthreads_or(found)) {
      for (int p = tail + threadIdx.x; p < L; p += blockDim.x) {
        x[p] = eos;
        m[p] = 0;
      }
    }
    for (int p = tail + threadIdx.x; p < L; p += blockDim.x) left |= m[p] != 0;
  }
  left = __syncthreads_or(left);
  if (threadIdx.x == 0) {
    st->block_index += 1;
    st->block_start += B;
    st->any_left = left;
    if (use_cond)
      cudaGraphSetConditional(h, (st->block_index < st->n_blocks && st->status == 0u && left) ? 1u : 0u);
  }
}

// The end-of-sequence id of the next generation (-1: none).
__global__ void set_eos_kernel(DevState* st, int eos_id) { st->eos_id = eos_id; }

// Condition of a block's conditional node: run it while masks are left.
__global__ void set_block_cond_kernel(DevState* st, cudaGraphConditionalHandle h) {
  cudaGraphSetConditional(h, (st->any_left && st->status == 0u) ? 1u : 0u);
}

// geometry of a stand-alone prefill / block step
__global__ void set_block_kernel(DevState* st, int block_start, int reset) {
  st->block_start = block_start;
  if (reset) {
    st->iteration = 0;
    st->status = 0;
    st->diag[0] = 0;
    st->block_index = 0;
  }
}

}  // namespace dinfer
