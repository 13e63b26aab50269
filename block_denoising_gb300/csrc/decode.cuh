// Decoding strategy on the device: merge the per-CTA online-softmax partials
// of the LM head into (token, confidence) per block position, then apply the
// threshold parallel commit in place.
//
// dInfer README, "Step 3: Use the model in dInfer": the decoder is
// ThresholdParallelDecoder(0, threshold, mask_id, eos_id) -- greedy top-1
// (temperature 0), confidence = softmax probability of the top-1 token; every
// masked position of the current block whose confidence exceeds the
// threshold is unmasked, else only the single most confident one.
// Ties: lowest vocabulary index (argmax), lowest block position (fallback).
#pragma once
#include "common.cuh"

namespace dinfer {

struct DecodeArgs {
  int M;                   // block rows = batch * B
  int batch, L, B;         // sequences, sequence length, block length
  float threshold;
  int commit;              // 0: produce tok/conf only
  int32_t* ids;            // [batch, L] updated in place
  uint8_t* mask;           // [batch, L] 1 = masked, cleared in place
  int32_t* tok_out;        // optional [M]
  float* conf_out;         // optional [M]
  int32_t* committed_out;  // optional [batch]
  DevState* state;
  int count_iteration;     // 1: advance the iteration counters
  cudaGraphConditionalHandle cond;
  int use_cond;
  SoftmaxState* partials;  // [n_parts][M]
  int n_parts;
  int* ticket;             // zero between launches
};

// Executed by 128 threads (ids 0..127) of the CTA that finished last.
// scratch: >= 2 * M words of shared memory.
__device__ __forceinline__ void finalize_and_commit(const DecodeArgs& d, int tid, int* scratch_i,
                                                    float* scratch_f, int bar_id) {
  // 1. merge partials in a fixed order -> token and confidence per row
  for (int m = tid; m < d.M; m += 128) {
    SoftmaxState s = sm_empty();
    for (int c = 0; c < d.n_parts; ++c) {
      const SoftmaxState* p = d.partials + (size_t)c * d.M + m;
      SoftmaxState x;
      x.m = __ldcg(&p->m);
      x.s = __ldcg(&p->s);
      x.a = __ldcg(&p->a);
      s = sm_merge(s, x);
    }
    const float conf = 1.0f / s.s;  // the max term contributes 2^0 = 1
    scratch_i[m] = s.a;
    scratch_f[m] = conf;
    if (d.tok_out) d.tok_out[m] = s.a;
    if (d.conf_out) d.conf_out[m] = conf;
    if (!(conf == conf)) set_status(d.state, ST_NAN_CONF);
  }
  named_bar_sync(bar_id, 128);
  if (!d.commit) return;
  // 2. threshold commit, one warp per sequence
  const int warp = tid >> 5, lane = tid & 31;
  const int s0 = d.state->block_start;
  __shared__ int any_left_sh;
  if (tid == 0) any_left_sh = 0;
  named_bar_sync(bar_id, 128);
  for (int b = warp; b < d.batch; b += 4) {
    int32_t* ids = d.ids + (size_t)b * d.L + s0;
    uint8_t* msk = d.mask + (size_t)b * d.L + s0;
    const int* tok = scratch_i + b * d.B;
    const float* conf = scratch_f + b * d.B;
    int n_masked = 0, n_sel = 0;
    float best = -1.f;
    int best_r = 0x7fffffff;
    for (int r0 = 0; r0 < d.B; r0 += 32) {
      const int r = r0 + lane;
      const bool in = r < d.B;
      const bool masked = in && msk[r] != 0;
      const bool sel = masked && conf[r] > d.threshold;
      n_masked += __popc(__ballot_sync(0xffffffffu, masked));
      n_sel += __popc(__ballot_sync(0xffffffffu, sel));
      if (masked && (conf[r] > best || (conf[r] == best && r < best_r))) {
        best = conf[r];
        best_r = r;
      }
    }
    // warp argmax of (best, -best_r)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int orr = __shfl_xor_sync(0xffffffffu, best_r, o);
      if (ob > best || (ob == best && orr < best_r)) {
        best = ob;
        best_r = orr;
      }
    }
    int committed = 0;
    if (n_masked > 0) {
      if (n_sel > 0) {
        for (int r0 = 0; r0 < d.B; r0 += 32) {
          const int r = r0 + lane;
          if (r < d.B && msk[r] != 0 && conf[r] > d.threshold) {
            ids[r] = tok[r];
            msk[r] = 0;
          }
        }
        committed = n_sel;
      } else {
        if (best_r >= d.B) {  // no comparable confidence (NaN): lowest masked position
          int r_first = 0x7fffffff;
          for (int r0 = 0; r0 < d.B; r0 += 32) {
            const unsigned bm = __ballot_sync(0xffffffffu, (r0 + lane) < d.B && msk[r0 + lane] != 0);
            if (bm && r_first == 0x7fffffff) r_first = r0 + __ffs(bm) - 1;
          }
          best_r = r_first;
        }
        if (lane == 0) {
          ids[best_r] = tok[best_r];
          msk[best_r] = 0;
        }
        committed = 1;
      }
    }
    if (lane == 0) {
      if (d.committed_out) d.committed_out[b] = committed;
      d.state->committed[b] = committed;
      if (n_masked - committed > 0) atomicOr(&any_left_sh, 1);
    }
  }
  named_bar_sync(bar_id, 128);
  if (tid == 0) {
    DevState* st = d.state;
    if (d.count_iteration) {
      st->iteration += 1;
      st->total_iterations += 1;
      if (st->block_index < kMaxBlocks) st->iters_per_block[st->block_index] = st->iteration;
      if (st->iteration > d.B) set_status(st, ST_ITER_OVERFLOW);
    }
    st->any_masked = any_left_sh;
    // a device-side error ends the block loop (and, through advance_block, the sequence)
    if (d.use_cond) cudaGraphSetConditional(d.cond, (any_left_sh && st->status == 0u) ? 1u : 0u);
  }
}

}  // namespace dinfer
