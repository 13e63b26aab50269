// Host runtime behind include/dinfer.h: context, workspaces, tensor maps,
// kernel enqueue for the refresh and the cached iteration, and the CUDA
// graphs that run the whole block loop on the device.
//
// The iteration loop follows the dInfer README's system notes (CUDA Graphs and
// loop unrolling to remove stream bubbles between diffusion iterations): here
// the block loop and the per-block iteration loop are CUDA graph conditional
// WHILE nodes whose conditions are set on the device by the commit, so a
// whole generation is one graph launch with no host round trip.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstddef>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/dinfer.h"
#include "../../include/dinfer_ops.h"
#include "attention.cuh"
#include "attention_tc.cuh"
#include "gemm_tc.cuh"
#include "gemm_tc2.cuh"
#include "lmhead_tc.cuh"
#include "moe.cuh"
#include "noalloc.cuh"
#include "small_kernels.cuh"

using namespace dinfer;

namespace {

thread_local std::string g_create_error;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 matrix [rows, cols] row-major, boxes of box_rows x 64 with the 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (cols * 2) % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor [batch][rows][cols] (row-major, packed), boxes of 128 rows x 64
// columns of one batch entry with the 128-byte swizzle; rows past `rows` read
// as zeros.
bool make_map3(CUtensorMap* m, const void* base, uint64_t batch, uint64_t rows, uint64_t cols) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (cols * 2) % 16 != 0) return false;
  cuuint64_t dims[3] = {cols, rows, batch};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int bn_for_rows(int M) { return M <= 64 ? 64 : (M <= 128 ? 128 : 256); }

// Per-device set-up state (SM count, kernel attributes): a process may drive
// several GPUs, each with its own.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
int g_num_sms[kMaxDevices] = {};
bool g_attrs_done[kMaxDevices] = {};
int g_pair_clusters[kMaxDevices] = {};  // co-resident 2-CTA clusters of the pair GEMM

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 0;
  }
  return dev;
}

int num_sms() {
  const int dev = current_device();
  if (!g_num_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    std::lock_guard<std::mutex> lk(g_setup_mutex);
    g_num_sms[dev] = n > 0 ? n : 1;
  }
  return g_num_sms[dev];
}

// Launch with programmatic dependent launch (the kernel may start while the
// previous kernel of the stream finishes; it waits with griddepcontrol.wait)
// and an optional cluster along z.
bool g_pdl = true;
template <typename... ExpTypes, typename... ActTypes>
cudaError_t launchk(void (*kernel)(ExpTypes...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster_z,
                    ActTypes&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int n = 0;
  if (g_pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_z > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = 1;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = cluster_z;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<ActTypes>(args)...);
}

bool set_smem_attrs() {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_setup_mutex);
  if (g_attrs_done[dev]) return true;
  bool ok = true;
  ok &= cudaFuncSetAttribute(gemm_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GemmKCfg<64>::kSmem) == cudaSuccess;
  ok &= cudaFuncSetAttribute(gemm_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GemmKCfg<128>::kSmem) == cudaSuccess;
  ok &= cudaFuncSetAttribute(gemm_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GemmKCfg<256>::kSmem) == cudaSuccess;
  ok &= cudaFuncSetAttribute(lmhead_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             LmCfg<64>::kSmem) == cudaSuccess;
  ok &= cudaFuncSetAttribute(lmhead_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             LmCfg<128>::kSmem) == cudaSuccess;
  ok &= cudaFuncSetAttribute(lmhead_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             LmCfg<256>::kSmem) == cudaSuccess;
  ok &= cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAtcSmem) ==
        cudaSuccess;
  ok &= cudaFuncSetAttribute(gemm_tc2_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Gemm2Cfg<256>::kSmem) == cudaSuccess;
  ok &= cudaFuncSetAttribute(gemm_tc2_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Gemm2Cfg<128>::kSmem) == cudaSuccess;
  ok &= cudaFuncSetAttribute(gemm_tc2_kernel<176>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Gemm2Cfg<176>::kSmem) == cudaSuccess;
  {
    // how many pairs run at once: clusters live inside one GPC, so SMs of a
    // GPC with an odd count of free SMs may stay out
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2 * 256);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = Gemm2Cfg<256>::kSmem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = 2;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    // a failed query leaves the pair path off (one-CTA tiles everywhere)
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc2_kernel<256>, &cfg) != cudaSuccess) {
      n = 0;
      cudaGetLastError();
    }
    g_pair_clusters[dev] = n;
  }
  ok &= cudaFuncSetAttribute(lmhead_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) ==
        cudaSuccess;
  ok &= cudaFuncSetAttribute(attn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) ==
        cudaSuccess;
  g_attrs_done[dev] = ok;
  return ok;
}

// Stream-K fixup workspace: floats per CTA slot pair and the ticket count.
size_t gemm_ws_floats(int grid) { return (size_t)grid * 2 * 256 * 128; }

// GEMM schedule.  With enough output tiles to keep most SMs streaming
// (a single SM pulls ~80-90 GB/s, so ~80 busy SMs saturate HBM), every CTA
// owns whole tiles and applies the epilogue itself.  With few tiles (the
// d_model-wide O and down projections of a block), the (tile, k-step) units
// are split evenly over the SMs (stream-K) and shared tiles are finished by
// the split-K fixup kernel, or -- residual GEMMs with defer_resid -- by the
// following resid_norm_kernel.
struct GemmSched {
  int stream_k, grid;
};
GemmSched gemm_schedule(int M, int n_tiles, int K, int BN, bool whole_only = false) {
  const int m_tiles = (M + BN - 1) / BN;
  const long long tiles = (long long)m_tiles * n_tiles;
  const int k_tiles = K / 64;
  const int sms = num_sms();
  GemmSched g;
  const long long per = (tiles + sms - 1) / sms;
  const long long wgrid = (tiles + per - 1) / per;
  // weight streaming (few token rows): ~80 busy SMs already saturate HBM;
  // tensor-bound (many rows): whole tiles only if they keep >= 90% of the SMs busy
  const bool whole = whole_only || (M <= 128 ? tiles * 10 >= (long long)sms * 6 : tiles * 10 >= (long long)sms * per * 9);
  if (whole) {
    g.stream_k = 0;
    g.grid = (int)wgrid;
  } else {
    // at least k_tiles / 14 units per CTA, so that at most 16 CTAs share a tile
    const long long units = tiles * k_tiles;
    const long long min_units = (k_tiles + 13) / 14;
    g.stream_k = 1;
    g.grid = (int)std::max<long long>(1, std::min<long long>(sms, units / min_units));
  }
  return g;
}

// The schedule a GEMM launch takes: gemm_schedule, except that a GEMM whose
// split tiles would need a fixup launch (~5 us) takes whole tiles when one SM
// streaming its weight tiles (~85 GB/s) is not slower than all SMs streaming
// the whole matrix (~6.8 TB/s) plus that launch -- provided the whole tiles
// occupy at least half of the SMs (a short-K tile streams at ~35 GB/s per SM,
// so fewer whole tiles, as the MoE model's QKV and router GEMMs of a block,
// are faster split).
GemmSched launch_schedule(const GemmArgs& a, int BN, bool defer_resid, bool whole_only) {
  GemmSched gs = gemm_schedule(a.M, a.n_tiles, a.K, BN, whole_only);
  const long long all_tiles = (long long)((a.M + BN - 1) / BN) * a.n_tiles;
  if (gs.stream_k && !defer_resid && a.M <= 128 && all_tiles * 2 >= num_sms()) {
    const long long tiles = (long long)((a.M + BN - 1) / BN) * a.n_tiles;
    const long long per = (tiles + num_sms() - 1) / num_sms();
    const long long tile_bytes = (long long)std::min(a.N, 128) * a.K * 2;
    if (per * tile_bytes / 85 <= tiles * tile_bytes / 6800 + 5000) {
      gs.stream_k = 0;
      gs.grid = (int)((tiles + per - 1) / per);
    }
  }
  return gs;
}

cudaError_t launch_gemm_tc(const GemmMaps& maps, GemmArgs a, int BN, cudaStream_t s, bool defer_resid = false,
                           bool whole_only = false) {
  a.m_tiles = (a.M + BN - 1) / BN;
  a.k_tiles = a.K / 64;
  const GemmSched gs = launch_schedule(a, BN, defer_resid, whole_only);
  a.stream_k = gs.stream_k;
  a.grid = gs.grid;
  const long long units = (long long)a.m_tiles * a.n_tiles * (a.stream_k ? a.k_tiles : 1);
  if ((unsigned long long)units * (unsigned long long)a.grid >= (1ull << 32)) return cudaErrorInvalidValue;
  const int tiles = a.m_tiles * a.n_tiles;
  // split tiles are finished by the fixup kernel; residual GEMMs leave them
  // to the next residual norm
  const bool fixup = a.stream_k && !defer_resid;
  cudaError_t e = cudaSuccess;
  switch (BN) {
    case 64:
      e = launchk(gemm_tc_kernel<64>, dim3(a.grid), dim3(kGemmThreads), GemmKCfg<64>::kSmem, s, 1, maps, a);
      if (e == cudaSuccess && fixup) e = launchk(splitk_fixup_kernel<64>, dim3(tiles * 4), dim3(128), 0, s, 1, a);
      break;
    case 128:
      e = launchk(gemm_tc_kernel<128>, dim3(a.grid), dim3(kGemmThreads), GemmKCfg<128>::kSmem, s, 1, maps, a);
      if (e == cudaSuccess && fixup) e = launchk(splitk_fixup_kernel<128>, dim3(tiles * 8), dim3(128), 0, s, 1, a);
      break;
    default:
      e = launchk(gemm_tc_kernel<256>, dim3(a.grid), dim3(kGemmThreads), GemmKCfg<256>::kSmem, s, 1, maps, a);
      if (e == cudaSuccess && fixup) e = launchk(splitk_fixup_kernel<256>, dim3(tiles * 16), dim3(128), 0, s, 1, a);
      break;
  }
  return e;
}

// Pair-CTA GEMM (gemm_tc2_kernel): 256 weight rows x 256 (or 128) tokens per
// tile on a 2-CTA cluster.  It pays where the GEMM is bound by the tensor
// cores (>= 384 token rows: the time of its MMAs at ~1.8 PFLOP/s exceeds that
// of reading its weights once); below that the one-CTA kernel streams the
// weights.  Per GEMM: whole 256-token tiles dealt round-robin over the
// co-resident pairs when they keep >= 85% of the pairs busy, else whole
// 176-token tiles when those do (1536 rows: 9 x 176 tokens, 144 tiles of a
// 4096-wide projection in two waves of 76 pairs); else 256-token
// tiles in stream-K order for a residual GEMM (the following residual norm
// adds its split tiles at little cost); else, for the others, whole 128-token
// tiles when those keep >= 80% of the pairs busy (no fixup launch), and
// stream-K with splitk_fixup_pair_kernel otherwise.  (Measured at 1536 rows:
// stream-K beats whole 128-token tiles for the O and down projections; at
// 512 rows whole 128-token tiles beat stream-K + fixup for QKV and gate/up.)
constexpr int kPairBN = 256;
enum PairMode { PAIR_NONE = 0, PAIR_W256, PAIR_W176, PAIR_W128, PAIR_SK };
int pair_clusters() {
  set_smem_attrs();
  return g_pair_clusters[current_device()];
}
bool pair_balanced(int M, int n_tiles, int bn, int pct) {
  const long long P = pair_clusters();
  const long long tiles = (long long)(n_tiles / 2) * ((M + bn - 1) / bn);
  const long long per = (tiles + P - 1) / P;
  return tiles * 100 >= per * P * pct;
}
PairMode pair_mode(int M, int n_tiles, bool resid) {
  if (pair_clusters() < 1 || M < 384 || n_tiles % 2) return PAIR_NONE;
  if (pair_balanced(M, n_tiles, 256, 85)) return PAIR_W256;
  if (pair_balanced(M, n_tiles, 176, 85)) return PAIR_W176;
  if (!resid && pair_balanced(M, n_tiles, 128, 80)) return PAIR_W128;
  return PAIR_SK;
}
int pair_bn(PairMode pm) { return pm == PAIR_W128 ? 128 : (pm == PAIR_W176 ? 176 : 256); }
// Pairs of a pair-GEMM launch: all co-resident pairs in stream-K mode (at
// least k_tiles / 14 units each, so that at most 16 pairs share a tile),
// else one per tile up to that count.
int pair_grid(const GemmArgs& a, int stream_k, int bn = kPairBN) {
  const int m_tiles = (a.M + bn - 1) / bn;
  const long long tiles = (long long)(a.n_tiles / 2) * m_tiles;
  const long long P = pair_clusters();
  if (!stream_k) return (int)std::min(P, tiles);
  const int k_tiles = a.K / 64;
  const long long min_units = (k_tiles + 13) / 14;
  return (int)std::max<long long>(1, std::min(P, tiles * k_tiles / min_units));
}
// the residual norm's view of a pair GEMM: whole tiles were added to h by
// the GEMM; stream-K leaves split tiles in the pairs' slots
ResidPlan resid_plan_pair(const GemmArgs& a, const float* ws, PairMode pm) {
  if (pm != PAIR_SK) {
    ResidPlan w{};
    w.ws = ws;
    w.BN = pair_bn(pm);
    w.m_tiles = (a.M + w.BN - 1) / w.BN;
    w.n_tiles = a.n_tiles;
    w.k_tiles = a.K / 64;
    w.stream_k = 0;
    w.grid = 1;
    w.pair = 1;
    return w;
  }
  ResidPlan p;
  p.ws = ws;
  p.BN = kPairBN;
  p.m_tiles = (a.M + kPairBN - 1) / kPairBN;
  p.n_tiles = a.n_tiles;
  p.k_tiles = a.K / 64;
  p.stream_k = 1;
  p.grid = pair_grid(a, 1);
  p.pair = 1;
  return p;
}
// maps.b: the token operand with pair_bn(pm) / 2-row boxes (each CTA stages
// half a tile).
cudaError_t launch_gemm_tc2(const GemmMaps& maps, GemmArgs a, cudaStream_t s, PairMode pm) {
  const int bn = pair_bn(pm);
  const int stream_k = pm == PAIR_SK;
  a.m_tiles = (a.M + bn - 1) / bn;
  a.k_tiles = a.K / 64;
  a.stream_k = stream_k;
  const int pairs = pair_grid(a, stream_k, bn);
  if (pairs < 1 || a.n_tiles % 2) return cudaErrorInvalidValue;
  const long long units = (long long)(a.n_tiles / 2) * a.m_tiles * (stream_k ? a.k_tiles : 1);
  if ((unsigned long long)units * (unsigned long long)pairs >= (1ull << 32)) return cudaErrorInvalidValue;
  a.grid = 2 * pairs;
  const long long tiles = (long long)(a.n_tiles / 2) * a.m_tiles;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes =
      bn == 128 ? Gemm2Cfg<128>::kSmem : (bn == 176 ? Gemm2Cfg<176>::kSmem : Gemm2Cfg<256>::kSmem);
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int n = 0;
  if (g_pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  at[n].id = cudaLaunchAttributeClusterDimension;
  at[n].val.clusterDim.x = 2;
  at[n].val.clusterDim.y = 1;
  at[n].val.clusterDim.z = 1;
  ++n;
  cfg.attrs = at;
  cfg.numAttrs = n;
  cudaError_t e = bn == 128   ? cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<128>, maps, a)
                  : bn == 176 ? cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<176>, maps, a)
                              : cudaLaunchKernelEx(&cfg, gemm_tc2_kernel<256>, maps, a);
  if (e == cudaSuccess && stream_k && a.resid == nullptr)
    e = launchk(splitk_fixup_pair_kernel<kPairBN>, dim3((unsigned)(tiles * 2 * (kPairBN / 16))), dim3(128), 0, s, 1,
                a);
  return e;
}

// Grouped (MoE expert) GEMM: persistent grid, tiles from the device tables.
cudaError_t launch_gemm_grouped(const GemmMaps& maps, GemmArgs a, int BN, cudaStream_t s) {
  a.grouped = 1;
  a.stream_k = 0;
  a.m_tiles = 1;
  a.k_tiles = a.K / 64;
  a.grid = num_sms();
  switch (BN) {
    case 64:
      return launchk(gemm_tc_kernel<64>, dim3(a.grid), dim3(kGemmThreads), GemmKCfg<64>::kSmem, s, 1, maps, a);
    case 128:
      return launchk(gemm_tc_kernel<128>, dim3(a.grid), dim3(kGemmThreads), GemmKCfg<128>::kSmem, s, 1, maps, a);
    default:
      return launchk(gemm_tc_kernel<256>, dim3(a.grid), dim3(kGemmThreads), GemmKCfg<256>::kSmem, s, 1, maps, a);
  }
}

// The routed FFN of one layer for `rows` rows of xn (bf16 [rows, d]):
// router GEMM -> top-k -> counting-sort permutation -> grouped gate/up
// (SwiGLU) and down GEMMs.  Leaves y [pairs, d] (fp32, permuted order),
// topk weights and inverse positions for the combine kernel.
struct MoeBufs {
  float* logits;
  int* topk_id;
  float* topk_w;
  int* rank;
  int* chunk_cnt;
  int* chunk_base;
  int* tables;
  int* inv;
  void* x;
  void* act;
  float* y;
  float* ws;
  DevState* st;
};
cudaError_t enqueue_moe_ffn(const MoeBufs& b, const void* xn, int rows, int D, int E, int K, int FE,
                            const CUtensorMap& m_router, const CUtensorMap& m_w13, const CUtensorMap& m_w2,
                            cudaStream_t s) {
  const int BN = bn_for_rows(rows);
  GemmMaps mr{};
  mr.a[0] = m_router;
  if (!make_map(&mr.b, xn, rows, D, BN)) return cudaErrorInvalidValue;
  GemmArgs ra{};
  ra.M = rows; ra.N = E; ra.K = D; ra.n_tiles = (E + 127) / 128; ra.a_mode = A_SINGLE;
  ra.out_f32 = b.logits; ra.ldo = E; ra.ws = b.ws; ra.status = b.st; ra.state = b.st;
  cudaError_t e = launch_gemm_tc(mr, ra, BN, s);
  if (e != cudaSuccess) return e;
  e = launchk(moe_topk_kernel, dim3((rows * 32 + 255) / 256), dim3(256), 0, s, 1, (const float*)b.logits, rows, E, K,
              b.topk_id, b.topk_w);
  if (e != cudaSuccess) return e;
  const int chunks = (rows + kMoeChunk - 1) / kMoeChunk;
  const int pairs = rows * K;
  const int bng = bn_for_rows(std::max(1, (pairs + E - 1) / E));  // token tile of the expert GEMMs
  int* row_off = b.tables;
  int* cum_gu = b.tables + (E + 1);
  int* cum_dn = b.tables + 2 * (E + 1);
  if (chunks == 1 && E <= 64) {
    e = launchk(moe_route_tables_kernel, dim3(1), dim3(kMoeChunk), 0, s, 1, (const int*)b.topk_id, rows, E, K, b.rank,
                b.chunk_base, row_off, cum_gu, cum_dn, bng, FE / 64, bng, D / 128, b.st);
    if (e != cudaSuccess) return e;
  } else {
    e = launchk(moe_count_kernel, dim3(chunks), dim3(kMoeChunk), 0, s, 1, (const int*)b.topk_id, rows, E, K, b.rank,
                b.chunk_cnt);
    if (e != cudaSuccess) return e;
    e = launchk(moe_scan_kernel, dim3(1), dim3(64), 0, s, 1, (const int*)b.chunk_cnt, chunks, E, b.chunk_base,
                row_off, cum_gu, cum_dn, bng, FE / 64, bng, D / 128, b.st);
    if (e != cudaSuccess) return e;
  }
  e = launchk(moe_scatter_kernel, dim3(pairs), dim3(256), 0, s, 1, (const __nv_bfloat16*)xn, D, rows, E, K,
              (const int*)b.topk_id, (const int*)b.rank, (const int*)b.chunk_base, (const int*)row_off, b.inv,
              (__nv_bfloat16*)b.x);
  if (e != cudaSuccess) return e;
  // gate/up: SwiGLU into act [pairs, FE]
  GemmMaps mg{};
  mg.a[0] = m_w13;
  if (!make_map(&mg.b, b.x, pairs, D, bng)) return cudaErrorInvalidValue;
  GemmArgs ga{};
  ga.M = pairs; ga.N = FE; ga.K = D; ga.a_mode = A_PAIR;
  ga.groups = E; ga.g_tile_cum = cum_gu; ga.g_row_off = row_off; ga.g_wrows = 2 * FE; ga.g_a_half = FE;
  ga.out_bf16 = (__nv_bfloat16*)b.act; ga.ldo = FE; ga.status = b.st; ga.state = b.st;
  e = launch_gemm_grouped(mg, ga, bng, s);
  if (e != cudaSuccess) return e;
  // down: y [pairs, D]
  GemmMaps md{};
  md.a[0] = m_w2;
  if (!make_map(&md.b, b.act, pairs, FE, bng)) return cudaErrorInvalidValue;
  GemmArgs da{};
  da.M = pairs; da.N = D; da.K = FE; da.a_mode = A_SINGLE;
  da.groups = E; da.g_tile_cum = cum_dn; da.g_row_off = row_off; da.g_wrows = D;
  da.out_f32 = b.y; da.ldo = D; da.status = b.st; da.state = b.st;
  return launch_gemm_grouped(md, da, bng, s);
}

ResidPlan resid_plan(const GemmArgs& a, int BN, const float* ws, bool whole_only = false) {
  ResidPlan p;
  p.ws = ws;
  p.BN = BN;
  p.m_tiles = (a.M + BN - 1) / BN;
  p.n_tiles = a.n_tiles;
  p.k_tiles = a.K / 64;
  const GemmSched gs = gemm_schedule(a.M, a.n_tiles, a.K, BN, whole_only);
  p.stream_k = gs.stream_k;
  p.grid = gs.grid;
  p.pair = 0;
  return p;
}

// Residual norm over `rows` rows (one CTA each): the many-rows variant when
// the grid is larger than one CTA per SM.
cudaError_t launch_resid_norm(int rows, int nthr, cudaStream_t s, float* h, const __nv_bfloat16* g,
                              __nv_bfloat16* out, int d, float eps, int rows_per_seq, int L, int gather,
                              int gather_off, const DevState* st, const ResidPlan& rp) {
  if (rows > num_sms())
    return launchk(resid_norm_kernel<__nv_bfloat16, true>, dim3(rows), dim3(nthr), 0, s, 1, h, g, out, d, eps,
                   rows_per_seq, L, gather, gather_off, st, rp, 1);
  return launchk(resid_norm_kernel<__nv_bfloat16, false>, dim3(rows), dim3(nthr), 0, s, 1, h, g, out, d, eps,
                 rows_per_seq, L, gather, gather_off, st, rp, 1);
}

int lmhead_grid(int M, int V) {
  const int BN = bn_for_rows(M);
  const long long tiles = (long long)((M + BN - 1) / BN) * ((V + 127) / 128);
  return (int)std::min<long long>(num_sms(), tiles);
}

cudaError_t launch_lmhead_tc(const GemmMaps& maps, GemmArgs ga, LmArgs la, int BN, cudaStream_t s) {
  ga.m_tiles = (ga.M + BN - 1) / BN;
  ga.k_tiles = ga.K / 64;
  ga.stream_k = 0;
  const int grid = lmhead_grid(ga.M, ga.N);
  la.dec.n_parts = grid;
  switch (BN) {
    case 64:
      return launchk(lmhead_tc_kernel<64>, dim3(grid), dim3(kGemmThreads), LmCfg<64>::kSmem, s, 1, maps, ga, la);
    case 128:
      return launchk(lmhead_tc_kernel<128>, dim3(grid), dim3(kGemmThreads), LmCfg<128>::kSmem, s, 1, maps, ga, la);
    default:
      return launchk(lmhead_tc_kernel<256>, dim3(grid), dim3(kGemmThreads), LmCfg<256>::kSmem, s, 1, maps, ga, la);
  }
}

struct AttnPlan {
  int q_tiles, splits, cps;
};
// One CTA per SM (about 198 KB of shared memory each).  Grids smaller than
// the SM count (a batch-1 block: heads x 1 query tile) split the keys over up
// to 8 CTAs of a cluster so that the grid fills the SMs once.
AttnPlan plan_attention(int batch, int rows_per_seq, int heads, int L) {
  AttnPlan p;
  p.q_tiles = (rows_per_seq + 127) / 128;
  const int n_chunks = (L + kAtcKeys - 1) / kAtcKeys;
  const int base = batch * p.q_tiles * heads;
  int want = num_sms() / base;
  want = std::max(1, std::min(std::min(want, n_chunks), 8));
  p.cps = (n_chunks + want - 1) / want;
  p.splits = (n_chunks + p.cps - 1) / p.cps;
  return p;
}

// q [batch * rows_per_seq, heads * 128], k/v [batch, L, heads * 128] -> o
cudaError_t launch_attention(const void* q, const void* k, const void* v, void* o, int batch, int rows_per_seq,
                             int heads, int L, const AttnPlan& ap, DevState* status, cudaStream_t s) {
  const int d = heads * kHd;
  AttnTcMaps maps;
  if (!make_map3(&maps.q, q, batch, rows_per_seq, d) || !make_map3(&maps.k, k, batch, L, d) ||
      !make_map3(&maps.v, v, batch, L, d))
    return cudaErrorInvalidValue;
  AttnTcArgs aa{};
  aa.o = (__nv_bfloat16*)o;
  aa.d = d; aa.heads = heads; aa.L = L; aa.rows_per_seq = rows_per_seq;
  aa.q_tiles = ap.q_tiles; aa.splits = ap.splits; aa.chunks_per_split = ap.cps;
  aa.scale_log2 = 1.4426950408889634f / sqrtf((float)kHd);
  aa.status = status;
  dim3 g(batch * ap.q_tiles, heads, ap.splits);
  return launchk(attn_tc_kernel, g, dim3(kAtcThreads), kAtcSmem, s, ap.splits, maps, aa);
}

struct GraphSet {
  cudaGraphExec_t exec = nullptr;
  cudaGraph_t graph = nullptr;
};

}  // namespace

// ===========================================================================
// context
// ===========================================================================
struct dinfer_ctx {
  dinfer_model_desc desc{};
  std::vector<const void*> w;
  bool bf16 = true;
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  cudaStream_t cap_stream = nullptr, cap_stream2 = nullptr;
  std::string err;
  std::vector<void*> allocs;

  size_t max_rows = 0;  // max_batch * max_seq
  float* h = nullptr;
  void* xn = nullptr;
  void* q = nullptr;
  void* attn_o = nullptr;
  void* act = nullptr;
  float* qkv32 = nullptr;
  float* gu32 = nullptr;
  void* kc = nullptr;
  void* vc = nullptr;
  float* rope_cos = nullptr;
  float* rope_sin = nullptr;
  int32_t* ids = nullptr;
  uint8_t* mask = nullptr;
  int32_t* prompt_dev = nullptr;
  int32_t* committed_dev = nullptr;
  DevState* st = nullptr;
  DevState* st_host = nullptr;  // pinned
  float* gemm_ws = nullptr;
  SoftmaxState* lm_part = nullptr;
  int* lm_ticket = nullptr;

  // weight maps (bf16)
  std::vector<CUtensorMap> m_wq, m_wk, m_wv, m_wo, m_wg, m_wu, m_wd;
  std::vector<CUtensorMap> m_router, m_w13, m_w2;
  // MoE routing / permutation buffers (rows = max_rows * top_k pairs)
  float* moe_logits = nullptr;
  int* moe_topk_id = nullptr;
  float* moe_topk_w = nullptr;
  int* moe_rank = nullptr;
  int* moe_chunk_cnt = nullptr;
  int* moe_chunk_base = nullptr;
  int* moe_tables = nullptr;  // row_off | tile_cum_gu | tile_cum_dn, each [E + 1]
  int* moe_inv = nullptr;
  void* moe_x = nullptr;      // bf16 [pairs, d]
  void* moe_act = nullptr;    // bf16 [pairs, fe]
  float* moe_y = nullptr;     // fp32 [pairs, d]
  CUtensorMap m_lm{};

  float* dbg_logits = nullptr;
  int32_t* dbg_tok = nullptr;
  float* dbg_conf = nullptr;
  float* dbg_hidden = nullptr;  // [n_layers][batch * B][d] residual stream of the block rows
  void* dbg_final = nullptr;    // [batch * B][d] LM-head input (model dtype)
  int dbg_block_start = -1;     // block start of the forward being enqueued (host-known), -1 inside generate

  // geometry of the last prefill (for dinfer_block_step)
  int cur_batch = 0, cur_L = 0, cur_B = 0, cur_s = 0;
  bool have_prefill = false;
  // KV-cache policy of the cached iterations (dinfer_set_cache_mode)
  int cache_mode = DINFER_CACHE_DUAL;
  int cache_window = 0;
  int eos_id = -1;  // end-of-sequence id of dinfer_generate (-1: none)

  std::map<std::tuple<int, int, int, int, int, int>, GraphSet> graphs;  // (kind, b, L, B, extra, window)
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;

  size_t cache_layer_elems() const { return (size_t)desc.max_batch * desc.max_seq * desc.d_model; }
  size_t esize() const { return bf16 ? 2 : 4; }
  void* kc_layer(int l) const { return (char*)kc + (size_t)l * cache_layer_elems() * esize(); }
  void* vc_layer(int l) const { return (char*)vc + (size_t)l * cache_layer_elems() * esize(); }
  const void* W(int i) const { return w[i]; }
  const void* LW(int l, int j) const { return w[1 + 9 * l + j]; }
};

namespace {

dinfer_status fail(dinfer_ctx* c, dinfer_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) c->err = buf; else g_create_error = buf;
  return s;
}

#define CK(call)                                                                              \
  do {                                                                                        \
    cudaError_t e_ = (call);                                                                  \
    if (e_ != cudaSuccess) return fail(c, DINFER_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

template <typename T>
dinfer_status dalloc(dinfer_ctx* c, T** p, size_t bytes) {
  void* q = nullptr;
  if (bytes == 0) bytes = 16;
  if (cudaMalloc(&q, bytes) != cudaSuccess) {
    cudaGetLastError();
    return fail(c, DINFER_ENOMEM, "cudaMalloc of %zu bytes failed", bytes);
  }
  c->allocs.push_back(q);
  *p = reinterpret_cast<T*>(q);
  return DINFER_OK;
}

const char* validate_desc(const dinfer_model_desc* d) {
  if (!d) return "null model description";
  if (d->n_layers < 1 || d->d_model < 1 || d->n_heads < 1 || d->head_dim < 2 || d->vocab < 2)
    return "non-positive model dimension";
  if (d->n_heads * d->head_dim != d->d_model) return "n_heads * head_dim != d_model";
  if (d->head_dim % 2) return "head_dim must be even";
  if (d->mask_id < 0 || d->mask_id >= d->vocab) return "mask_id outside [0, vocab)";
  if (d->dtype != DINFER_FP32 && d->dtype != DINFER_BF16) return "dtype must be DINFER_FP32 or DINFER_BF16";
  const bool moe = d->n_experts != 0 || d->top_k != 0 || d->expert_ffn != 0;
  if (moe) {
    if (d->n_experts < 1 || d->top_k < 1 || d->top_k > d->n_experts || d->expert_ffn < 1)
      return "inconsistent MoE fields";
    if (d->dtype != DINFER_BF16) return "MoE models must be bf16";
    if (d->n_experts > 64) return "MoE models take at most 64 experts";
    if (d->top_k > kMoeMaxK) return "MoE top_k must be <= 8";
    if (d->expert_ffn % 64) return "MoE expert_ffn must be a multiple of 64";
  } else if (d->ffn < 1) {
    return "ffn must be positive";
  }
  if (d->max_batch < 1 || d->max_batch > kMaxBatch) return "max_batch must be in [1, 64]";
  if (d->max_seq < 1) return "max_seq must be positive";
  if (!(d->rms_eps >= 0.f) || !(d->rope_theta > 0.f) || !std::isfinite(d->logit_scale)) return "bad float field";
  if (d->dtype == DINFER_BF16) {
    if (d->head_dim != 128) return "bf16 models need head_dim 128";
    if (d->d_model % 128) return "bf16 models need d_model % 128 == 0";
    if (!moe && d->ffn % 64) return "bf16 models need ffn % 64 == 0";
    if (d->vocab % 8) return "bf16 models need vocab % 8 == 0";
  } else {
    if ((size_t)d->d_model * 4 * 64 > 192 * 1024) return "fp32 models need d_model <= 768";
  }
  return nullptr;
}

// ---------------------------------------------------------------------------
// geometry of one forward
// ---------------------------------------------------------------------------
struct Fwd {
  int batch, L, B;
  int rows;          // rows computed: batch * rows_per_seq
  int rows_per_seq;  // B (dual-cache iteration), L (refresh), or a window's length
  int pos_from_state;  // 1: computed rows start at the block start (read on the device)
  bool refresh;
  // decode
  int commit;
  int count_iteration;
  cudaGraphConditionalHandle cond;
  int use_cond;
  float threshold;
  int row_off = 0;   // first computed position (added to the block start when pos_from_state)
  // the block rows sit at offset (block start - first computed position) in each sequence's rows
  bool gathers_block() const { return rows_per_seq != B; }
};

// Test hook: copy the residual stream of the block rows after layer l (the
// rows of a refresh sit at the block start of each sequence).
cudaError_t debug_copy_hidden(dinfer_ctx* c, const Fwd& f, int l, cudaStream_t s) {
  if (!c->dbg_hidden || c->dbg_block_start < 0) return cudaSuccess;
  const size_t d = c->desc.d_model, brows = (size_t)f.batch * f.B;
  float* dst = c->dbg_hidden + (size_t)l * brows * d;
  if (!f.gathers_block()) return cudaMemcpyAsync(dst, c->h, brows * d * 4, cudaMemcpyDeviceToDevice, s);
  const size_t off = (size_t)(c->dbg_block_start - f.row_off);  // window rows start at row_off
  return cudaMemcpy2DAsync(dst, (size_t)f.B * d * 4, c->h + off * d, (size_t)f.rows_per_seq * d * 4,
                           (size_t)f.B * d * 4, f.batch, cudaMemcpyDeviceToDevice, s);
}

// Enqueue one forward over f.rows rows, final norm of the block rows, LM head,
// decode and (optionally) the commit.  Works eagerly or under stream capture.
// bf16 layer sequence (per layer, all on the tensor-core path):
//   [norm] -> QKV GEMM (+fixup: RoPE, q, dual-cache K/V) -> attention ->
//   O GEMM (deferred residual) -> resid_norm (h += O; ffn norm) ->
//   gate/up GEMM (+fixup: SwiGLU) -> down GEMM (deferred residual) ->
//   resid_norm (h += down; next layer's attention norm, or the final norm of
//   the block rows)
dinfer_status enqueue_layers_bf16(dinfer_ctx* c, const Fwd& f, cudaStream_t s) {
  const dinfer_model_desc& d = c->desc;
  const int D = d.d_model, F = d.ffn, H = d.n_heads, hd = d.head_dim;
  const int rows = f.rows;
  RowMap rm{f.rows_per_seq, f.L, f.pos_from_state, f.row_off};
  CK(launchk(embed_kernel<__nv_bfloat16>, dim3(rows), dim3(256), 0, s, 1, (const __nv_bfloat16*)c->W(0),
             (const int32_t*)c->ids, c->h, rows, D, d.vocab, rm, c->st));
  CK(launchk(rmsnorm_kernel<__nv_bfloat16, __nv_bfloat16>, dim3(rows), dim3(256), 0, s, 1,
             (const float*)c->h, (const __nv_bfloat16*)c->LW(0, 0), (__nv_bfloat16*)c->xn, rows, D, d.rms_eps, 0,
             rm, (const DevState*)c->st));
  const int BN = bn_for_rows(rows);
  // O projection of many rows: 128-token tiles dealt whole (three per CTA on
  // 128 SMs at 1536 x 4096) add to h in the GEMM, so the FFN norm gathers no
  // stream-K partials -- when they keep at least 80% of the SMs busy
  const long long o_tiles = (long long)((rows + 127) / 128) * (D / 128);
  const long long o_per = (o_tiles + num_sms() - 1) / num_sms();
  const bool o_whole = rows > 128 && o_tiles * 10 >= o_per * num_sms() * 8;
  const int BNo = o_whole ? 128 : BN;
  GemmMaps mx{}, mo{}, mact{};
  if (!make_map(&mx.b, c->xn, rows, D, BN) || !make_map(&mo.b, c->attn_o, rows, D, BNo) ||
      (!d.n_experts && !make_map(&mact.b, c->act, rows, F, BN)))
    return fail(c, DINFER_ECUDA, "tensor map encoding failed for activations");
  // many rows: every projection on pair-CTA tiles (pair_mode)
  const PairMode pm_qkv = pair_mode(rows, 3 * D / 128, false);
  const PairMode pm_gu = d.n_experts ? PAIR_NONE : pair_mode(rows, F / 64, false);
  const PairMode pm_o = pair_mode(rows, D / 128, true);
  const PairMode pm_down = d.n_experts ? PAIR_NONE : pair_mode(rows, D / 128, true);
  const bool pair_qkv = pm_qkv != PAIR_NONE, pair_gu = pm_gu != PAIR_NONE;
  const bool pair_o = pm_o != PAIR_NONE, pair_down = pm_down != PAIR_NONE;
  GemmMaps mxq{}, mxg{}, mo2{}, mact2{};
  if ((pair_qkv && !make_map(&mxq.b, c->xn, rows, D, pair_bn(pm_qkv) / 2)) ||
      (pair_gu && !make_map(&mxg.b, c->xn, rows, D, pair_bn(pm_gu) / 2)) ||
      (pair_o && !make_map(&mo2.b, c->attn_o, rows, D, pair_bn(pm_o) / 2)) ||
      (pair_down && !make_map(&mact2.b, c->act, rows, F, pair_bn(pm_down) / 2)))
    return fail(c, DINFER_ECUDA, "tensor map encoding failed for activations");
  const AttnPlan ap = plan_attention(f.batch, f.rows_per_seq, H, f.L);
  const int nthr = ((D / 16 + 31) / 32) * 32;  // fused-norm threads per row: whole warps
  if (nthr > 512 || D % 128) return fail(c, DINFER_EINVAL, "d_model unsupported by the fused residual norm");
  for (int l = 0; l < d.n_layers; ++l) {
    // QKV GEMM, RoPE and the dual-cache write in its epilogue
    {
      GemmMaps m = pair_qkv ? mxq : mx;
      m.a[0] = c->m_wq[l];
      m.a[1] = c->m_wk[l];
      m.a[2] = c->m_wv[l];
      GemmArgs a{};
      a.M = rows; a.N = 3 * D; a.K = D;
      a.n_tiles = 3 * D / 128;
      a.a_mode = A_THREE; a.a_rows = D;
      a.q_out = (__nv_bfloat16*)c->q;
      a.k_cache = (__nv_bfloat16*)c->kc_layer(l);
      a.v_cache = (__nv_bfloat16*)c->vc_layer(l);
      a.rope_cos = c->rope_cos; a.rope_sin = c->rope_sin;
      a.d_model = D; a.head_dim = hd;
      a.rows_per_seq = f.rows_per_seq; a.seq_len = f.L; a.pos_from_state = f.pos_from_state;
      a.row_off = f.row_off;
      a.state = c->st; a.ws = c->gemm_ws; a.status = c->st;
      CK(pair_qkv ? launch_gemm_tc2(m, a, s, pm_qkv) : launch_gemm_tc(m, a, BN, s));
    }
    // attention over the dual cache
    CK(launch_attention(c->q, c->kc_layer(l), c->vc_layer(l), c->attn_o, f.batch, f.rows_per_seq, H, f.L, ap,
                        c->st, s));
    // O projection + residual, fused with the FFN norm
    {
      GemmMaps m = pair_o ? mo2 : mo;
      m.a[0] = c->m_wo[l];
      GemmArgs a{};
      a.M = rows; a.N = D; a.K = D; a.n_tiles = D / 128; a.a_mode = A_SINGLE;
      a.resid = c->h; a.ws = c->gemm_ws; a.status = c->st; a.state = c->st;
      CK(pair_o ? launch_gemm_tc2(m, a, s, pm_o) : launch_gemm_tc(m, a, BNo, s, true, o_whole));
      CK(launch_resid_norm(rows, nthr, s, c->h, (const __nv_bfloat16*)c->LW(l, 5), (__nv_bfloat16*)c->xn, D,
                           d.rms_eps, f.rows_per_seq, f.L, 0, 0, (const DevState*)c->st,
                           pair_o ? resid_plan_pair(a, c->gemm_ws, pm_o)
                                  : resid_plan(a, BNo, c->gemm_ws, o_whole)));
    }
    const bool last = l + 1 == d.n_layers;
    const void* gn = last ? c->W(1 + 9 * d.n_layers) : c->LW(l + 1, 0);
    // after the last layer only the block rows go on (to the LM head),
    // gathered from the rows of each sequence when more rows were computed
    const int nrows = last ? f.batch * f.B : rows;
    const int gather = last && f.gathers_block() ? 1 : 0;
    if (d.n_experts) {
      // MoE FFN: routed experts, then the weighted combine + residual + next norm
      MoeBufs mb{c->moe_logits, c->moe_topk_id, c->moe_topk_w, c->moe_rank, c->moe_chunk_cnt, c->moe_chunk_base,
                 c->moe_tables, c->moe_inv, c->moe_x, c->moe_act, c->moe_y, c->gemm_ws, c->st};
      CK(enqueue_moe_ffn(mb, c->xn, rows, D, d.n_experts, d.top_k, d.expert_ffn, c->m_router[l], c->m_w13[l],
                         c->m_w2[l], s));
      CK(launchk(moe_combine_norm_kernel<__nv_bfloat16>, dim3(nrows), dim3(nthr), 0, s, 1, c->h,
                 (const float*)c->moe_y, (const float*)c->moe_topk_w, (const int*)c->moe_inv, d.top_k,
                 (const __nv_bfloat16*)gn, (__nv_bfloat16*)c->xn, D, d.rms_eps, f.B, f.rows_per_seq, gather,
                 -f.row_off, (const DevState*)c->st));
      CK(debug_copy_hidden(c, f, l, s));
      continue;
    }
    // SwiGLU FFN (gate/up with the SiLU*up epilogue, down + residual)
    {
      GemmMaps m = pair_gu ? mxg : mx;
      m.a[0] = c->m_wg[l];
      m.a[1] = c->m_wu[l];
      GemmArgs a{};
      a.M = rows; a.N = F; a.K = D; a.n_tiles = F / 64; a.a_mode = A_PAIR;
      a.out_bf16 = (__nv_bfloat16*)c->act; a.ldo = F;
      a.ws = c->gemm_ws; a.status = c->st; a.state = c->st;
      CK(pair_gu ? launch_gemm_tc2(m, a, s, pm_gu) : launch_gemm_tc(m, a, BN, s));
      GemmMaps m2 = pair_down ? mact2 : mact;
      m2.a[0] = c->m_wd[l];
      GemmArgs b{};
      b.M = rows; b.N = D; b.K = F; b.n_tiles = D / 128; b.a_mode = A_SINGLE;
      b.resid = c->h; b.ws = c->gemm_ws; b.status = c->st; b.state = c->st;
      CK(pair_down ? launch_gemm_tc2(m2, b, s, pm_down) : launch_gemm_tc(m2, b, BN, s, true));
      CK(launch_resid_norm(nrows, nthr, s, c->h, (const __nv_bfloat16*)gn, (__nv_bfloat16*)c->xn, D, d.rms_eps,
                           f.B, f.rows_per_seq, gather, -f.row_off, (const DevState*)c->st,
                           pair_down ? resid_plan_pair(b, c->gemm_ws, pm_down) : resid_plan(b, BN, c->gemm_ws)));
      CK(debug_copy_hidden(c, f, l, s));
    }
  }
  return DINFER_OK;
}

// Enqueue one forward over f.rows rows, final norm of the block rows, LM head,
// decode and (optionally) the commit.  Works eagerly or under stream capture.
dinfer_status enqueue_forward(dinfer_ctx* c, const Fwd& f, cudaStream_t s) {
  const dinfer_model_desc& d = c->desc;
  const int D = d.d_model, F = d.ffn, H = d.n_heads, hd = d.head_dim;
  const int rows = f.rows;
  RowMap rm{f.rows_per_seq, f.L, f.pos_from_state, f.row_off};
  if (c->bf16) {
    dinfer_status st = enqueue_layers_bf16(c, f, s);
    if (st != DINFER_OK) return st;
  } else {
    // fp32 models: SIMT FFMA GEMMs and separate elementwise kernels
    embed_kernel<float><<<rows, 256, 0, s>>>((const float*)c->W(0), c->ids, c->h, rows, D, d.vocab, rm, c->st);
    CK(cudaGetLastError());
    for (int l = 0; l < d.n_layers; ++l) {
      rmsnorm_kernel<float, float><<<rows, 256, 0, s>>>(c->h, (const float*)c->LW(l, 0), (float*)c->xn, rows, D,
                                                        d.rms_eps, 0, rm, c->st);
      for (int j = 0; j < 3; ++j) {
        dim3 g((D + 63) / 64, (rows + 63) / 64);
        gemm_f32_kernel<<<g, 256, 0, s>>>((const float*)c->xn, (const float*)c->LW(l, 1 + j), c->qkv32 + j * D,
                                          rows, D, D, 3 * D, 0);
      }
      rope_cache_f32_kernel<<<rows, 256, 0, s>>>(c->qkv32, (float*)c->q, (float*)c->kc_layer(l),
                                                  (float*)c->vc_layer(l), c->rope_cos, c->rope_sin, rows, D, hd, rm,
                                                  c->st);
      AttnF32Args aa{(const float*)c->q, (const float*)c->kc_layer(l), (const float*)c->vc_layer(l),
                     (float*)c->attn_o, D, H, hd, f.L, f.rows_per_seq, 1.f / sqrtf((float)hd)};
      attn_f32_kernel<<<dim3(rows, H), 128, (size_t)(f.L + hd) * sizeof(float), s>>>(aa);
      {
        dim3 g((D + 63) / 64, (rows + 63) / 64);
        gemm_f32_kernel<<<g, 256, 0, s>>>((const float*)c->attn_o, (const float*)c->LW(l, 4), c->h, rows, D, D, D,
                                          1);
      }
      rmsnorm_kernel<float, float><<<rows, 256, 0, s>>>(c->h, (const float*)c->LW(l, 5), (float*)c->xn, rows, D,
                                                        d.rms_eps, 0, rm, c->st);
      {
        dim3 g((F + 63) / 64, (rows + 63) / 64);
        gemm_f32_kernel<<<g, 256, 0, s>>>((const float*)c->xn, (const float*)c->LW(l, 6), c->gu32, rows, F, D,
                                          2 * F, 0);
        gemm_f32_kernel<<<g, 256, 0, s>>>((const float*)c->xn, (const float*)c->LW(l, 7), c->gu32 + F, rows, F, D,
                                          2 * F, 0);
        swiglu_f32_kernel<<<256, 256, 0, s>>>(c->gu32, (float*)c->act, rows, F);
        dim3 g2((D + 63) / 64, (rows + 63) / 64);
        gemm_f32_kernel<<<g2, 256, 0, s>>>((const float*)c->act, (const float*)c->LW(l, 8), c->h, rows, D, F, D, 1);
      }
      CK(cudaGetLastError());
      CK(debug_copy_hidden(c, f, l, s));
    }
    // final norm of the block rows (gathered from the full sequence at a refresh)
    const int brows = f.batch * f.B;
    RowMap rb{f.B, f.rows_per_seq, 1, -f.row_off};
    rmsnorm_kernel<float, float><<<brows, 256, 0, s>>>(c->h, (const float*)c->W(1 + 9 * d.n_layers),
                                                       (float*)c->xn, brows, D, d.rms_eps,
                                                       f.gathers_block() ? 1 : 0, rb, c->st);
    CK(cudaGetLastError());
  }

  // LM head, online softmax, threshold commit
  const int brows = f.batch * f.B;
  if (c->dbg_final)
    CK(cudaMemcpyAsync(c->dbg_final, c->xn, (size_t)brows * D * c->esize(), cudaMemcpyDeviceToDevice, s));
  DecodeArgs dec{};
  dec.M = brows; dec.batch = f.batch; dec.L = f.L; dec.B = f.B;
  dec.threshold = f.threshold; dec.commit = f.commit;
  dec.ids = c->ids; dec.mask = c->mask;
  dec.tok_out = c->dbg_tok; dec.conf_out = c->dbg_conf;
  dec.committed_out = c->committed_dev;
  dec.state = c->st; dec.count_iteration = f.count_iteration;
  dec.cond = f.cond; dec.use_cond = f.use_cond;
  dec.partials = c->lm_part; dec.ticket = c->lm_ticket;
  if (c->bf16) {
    const int BNl = bn_for_rows(brows);
    GemmMaps m{};
    m.a[0] = c->m_lm;
    if (!make_map(&m.b, c->xn, brows, D, BNl)) return fail(c, DINFER_ECUDA, "tensor map encoding failed (lm)");
    GemmArgs ga{};
    ga.M = brows; ga.N = d.vocab; ga.K = D; ga.n_tiles = (d.vocab + 127) / 128; ga.a_mode = A_SINGLE;
    ga.status = c->st; ga.state = c->st;
    LmArgs la{d.vocab, d.mask_id, d.logit_scale, c->dbg_logits, dec};
    CK(launch_lmhead_tc(m, ga, la, BNl, s));
  } else {
    const int grid = std::min(num_sms(), (d.vocab + 127) / 128);
    dec.n_parts = grid;
    LmF32Args la{(const float*)c->xn, (const float*)c->W(2 + 9 * d.n_layers), brows, D, d.vocab, d.mask_id,
                 d.logit_scale, c->dbg_logits, dec};
    lmhead_f32_kernel<<<grid, 128, (size_t)brows * D * sizeof(float), s>>>(la);
    CK(cudaGetLastError());
  }
  return DINFER_OK;
}

bool debug_on(const dinfer_ctx* c) {
  return c->dbg_logits || c->dbg_tok || c->dbg_conf || c->dbg_hidden || c->dbg_final;
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

dinfer_status read_status(dinfer_ctx* c) {
  CK(cudaMemcpyAsync(c->st_host, c->st, sizeof(DevState), cudaMemcpyDeviceToHost, c->stream));
  CK(cudaStreamSynchronize(c->stream));
  if (c->st_host->status)
    return fail(c, DINFER_EDEVICE,
                "device status word 0x%x (1 wait timeout, 2 bad token, 4 NaN confidence, 8 iteration overflow); "
                "first timeout: site 0x%x block 0x%x z/step 0x%x thread %u",
                c->st_host->status, c->st_host->diag[0], c->st_host->diag[1], c->st_host->diag[2],
                c->st_host->diag[3]);
  return DINFER_OK;
}

// Capture a graph that runs one forward (refresh or cached iteration).
dinfer_status build_step_graph(dinfer_ctx* c, const Fwd& f, GraphSet& gs) {
  cudaStream_t s = c->cap_stream;
  CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  dinfer_status st = enqueue_forward(c, f, s);
  cudaGraph_t g = nullptr;
  cudaError_t e = cudaStreamEndCapture(s, &g);
  if (st != DINFER_OK) {
    if (g) cudaGraphDestroy(g);
    return st;
  }
  if (e != cudaSuccess) return fail(c, DINFER_ECUDA, "stream capture failed: %s", cudaGetErrorString(e));
  e = cudaGraphInstantiate(&gs.exec, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return fail(c, DINFER_ECUDA, "graph instantiation failed: %s", cudaGetErrorString(e));
  }
  gs.graph = g;
  return DINFER_OK;
}

// Add a WHILE conditional node at the current capture point of stream s and
// return its body graph; subsequent captured work depends on the node.
dinfer_status add_while_node(dinfer_ctx* c, cudaStream_t s, cudaGraphConditionalHandle h, cudaGraph_t* body) {
  cudaStreamCaptureStatus cs;
  cudaGraph_t cg = nullptr;
  const cudaGraphNode_t* deps = nullptr;
  size_t ndeps = 0;
  CK(cudaStreamGetCaptureInfo(s, &cs, nullptr, &cg, &deps, nullptr, &ndeps));
  if (cs != cudaStreamCaptureStatusActive) return fail(c, DINFER_ECUDA, "stream is not capturing");
  cudaGraphNodeParams p{};
  p.type = cudaGraphNodeTypeConditional;
  p.conditional.handle = h;
  p.conditional.type = cudaGraphCondTypeWhile;
  p.conditional.size = 1;
  cudaGraphNode_t node;
  CK(cudaGraphAddNode(&node, cg, deps, nullptr, ndeps, &p));
  *body = p.conditional.phGraph_out[0];
  CK(cudaStreamUpdateCaptureDependencies(s, &node, nullptr, 1, cudaStreamSetCaptureDependencies));
  return DINFER_OK;
}

// Whole-generation graph: init; while (blocks left) { refresh + commit;
// while (masks left) { cached iteration + commit } ; next block }.
dinfer_status build_generate_graph(dinfer_ctx* c, int batch, int P, int G, int B, float thr, GraphSet& gs) {
  const int L = P + G;
  cudaStream_t s = c->cap_stream, s2 = c->cap_stream2;
  cudaGraph_t g = nullptr;
  CK(cudaGraphCreate(&g, 0));
  dinfer_status st = DINFER_OK;
  cudaGraph_t body_o = nullptr, body_i = nullptr;
  cudaGraphConditionalHandle h_o, h_i;
  // top level
  CK(cudaGraphConditionalHandleCreate(&h_o, g, 1, cudaGraphCondAssignDefault));
  CK(cudaStreamBeginCaptureToGraph(s, g, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal));
  init_sequence_kernel<<<256, 256, 0, s>>>(c->prompt_dev, c->ids, c->mask, batch, P, L, c->desc.mask_id, c->st,
                                           G / B);
  st = add_while_node(c, s, h_o, &body_o);
  {
    cudaGraph_t g2 = nullptr;
    cudaError_t e = cudaStreamEndCapture(s, &g2);
    if (st != DINFER_OK) return st;
    if (e != cudaSuccess) return fail(c, DINFER_ECUDA, "capture (top): %s", cudaGetErrorString(e));
  }
  // outer body: one block
  CK(cudaGraphConditionalHandleCreate(&h_i, body_o, 0, cudaGraphCondAssignDefault));
  CK(cudaStreamBeginCaptureToGraph(s2, body_o, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal));
  begin_block_kernel<<<1, 1, 0, s2>>>(c->st);
  Fwd fr{batch, L, B, batch * L, L, 0, true, 1, 1, 0, 0, thr};
  st = enqueue_forward(c, fr, s2);
  if (st == DINFER_OK) {
    set_inner_cond_kernel<<<1, 1, 0, s2>>>(c->st, h_i);
    st = add_while_node(c, s2, h_i, &body_i);
  }
  if (st == DINFER_OK) advance_block_kernel<<<1, 256, 0, s2>>>(c->st, B, h_o, 1, c->ids, c->mask, batch, L);
  {
    cudaGraph_t g2 = nullptr;
    cudaError_t e = cudaStreamEndCapture(s2, &g2);
    if (st != DINFER_OK) return st;
    if (e != cudaSuccess) return fail(c, DINFER_ECUDA, "capture (block): %s", cudaGetErrorString(e));
  }
  // inner body: one cached iteration
  CK(cudaStreamBeginCaptureToGraph(s2, body_i, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal));
  Fwd fi{batch, L, B, batch * B, B, 1, false, 1, 1, h_i, 1, thr};
  st = enqueue_forward(c, fi, s2);
  {
    cudaGraph_t g2 = nullptr;
    cudaError_t e = cudaStreamEndCapture(s2, &g2);
    if (st != DINFER_OK) return st;
    if (e != cudaSuccess) return fail(c, DINFER_ECUDA, "capture (iteration): %s", cudaGetErrorString(e));
  }
  cudaError_t e = cudaGraphInstantiate(&gs.exec, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return fail(c, DINFER_ECUDA, "graph instantiation failed: %s", cudaGetErrorString(e));
  }
  gs.graph = g;
  return DINFER_OK;
}

// Positions [r0, r1) a cached iteration recomputes under the context's cache
// policy (block start s0, block length B, sequence length L).
void cache_window(const dinfer_ctx* c, int s0, int B, int L, int& r0, int& r1) {
  switch (c->cache_mode) {
    case DINFER_CACHE_NONE: r0 = 0; r1 = L; break;
    case DINFER_CACHE_PREFIX: r0 = s0; r1 = L; break;
    case DINFER_CACHE_VICINITY:
      r0 = std::max(0, s0 - c->cache_window);
      r1 = std::min(L, s0 + B + c->cache_window);
      break;
    default: r0 = s0; r1 = s0 + B; break;
  }
}

// The forward of a cached iteration: the dual cache's block rows (positions
// read on the device, one graph for every block), or a window of host-known
// positions.
Fwd iteration_fwd(const dinfer_ctx* c, int batch, int L, int B, int s0, float thr, int commit,
                  cudaGraphConditionalHandle cond, int use_cond) {
  int r0, r1;
  cache_window(c, s0, B, L, r0, r1);
  if (c->cache_mode == DINFER_CACHE_DUAL) return Fwd{batch, L, B, batch * B, B, 1, false, commit, 1, cond, use_cond, thr};
  Fwd f{batch, L, B, batch * (r1 - r0), r1 - r0, 0, false, commit, 1, cond, use_cond, thr};
  f.row_off = r0;
  return f;
}

// Graph of one block for the host-driven block loop (window cache policies):
// IF (some sequence has masked positions left) { refresh + commit; WHILE
// (masks left in the block) { one cached iteration over the window of block
// start s0 }; end of block (end-of-sequence, next block) }.
dinfer_status build_block_graph(dinfer_ctx* c, int batch, int L, int B, int s0, float thr, GraphSet& gs) {
  cudaStream_t s = c->cap_stream, s2 = c->cap_stream2;
  cudaGraph_t g = nullptr;
  CK(cudaGraphCreate(&g, 0));
  cudaGraphConditionalHandle h_if, h_w;
  CK(cudaGraphConditionalHandleCreate(&h_if, g, 0, cudaGraphCondAssignDefault));
  cudaGraph_t body_if = nullptr, body_w = nullptr;
  dinfer_status st = DINFER_OK;
  auto end_capture = [&](cudaStream_t cs, const char* what) -> dinfer_status {
    cudaGraph_t g2 = nullptr;
    cudaError_t e = cudaStreamEndCapture(cs, &g2);
    if (st != DINFER_OK) return st;
    if (e != cudaSuccess) return fail(c, DINFER_ECUDA, "capture (%s): %s", what, cudaGetErrorString(e));
    return DINFER_OK;
  };
  // top level: the block's condition, then its IF node
  CK(cudaStreamBeginCaptureToGraph(s, g, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal));
  set_block_cond_kernel<<<1, 1, 0, s>>>(c->st, h_if);
  {
    cudaStreamCaptureStatus cs;
    cudaGraph_t cg = nullptr;
    const cudaGraphNode_t* deps = nullptr;
    size_t ndeps = 0;
    cudaError_t e = cudaStreamGetCaptureInfo(s, &cs, nullptr, &cg, &deps, nullptr, &ndeps);
    cudaGraphNodeParams p{};
    p.type = cudaGraphNodeTypeConditional;
    p.conditional.handle = h_if;
    p.conditional.type = cudaGraphCondTypeIf;
    p.conditional.size = 1;
    cudaGraphNode_t node;
    if (e == cudaSuccess) e = cudaGraphAddNode(&node, cg, deps, nullptr, ndeps, &p);
    if (e == cudaSuccess) e = cudaStreamUpdateCaptureDependencies(s, &node, nullptr, 1, cudaStreamSetCaptureDependencies);
    if (e != cudaSuccess) st = fail(c, DINFER_ECUDA, "conditional IF node: %s", cudaGetErrorString(e));
    else body_if = p.conditional.phGraph_out[0];
  }
  if ((st = end_capture(s, "block")) != DINFER_OK) return st;
  // IF body: refresh, the iteration loop, end of block
  CK(cudaGraphConditionalHandleCreate(&h_w, body_if, 0, cudaGraphCondAssignDefault));
  CK(cudaStreamBeginCaptureToGraph(s2, body_if, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal));
  begin_block_kernel<<<1, 1, 0, s2>>>(c->st);
  const Fwd fr{batch, L, B, batch * L, L, 0, true, 1, 1, 0, 0, thr};
  st = enqueue_forward(c, fr, s2);
  if (st == DINFER_OK) {
    set_inner_cond_kernel<<<1, 1, 0, s2>>>(c->st, h_w);
    st = add_while_node(c, s2, h_w, &body_w);
  }
  if (st == DINFER_OK) advance_block_kernel<<<1, 256, 0, s2>>>(c->st, B, 0, 0, c->ids, c->mask, batch, L);
  if ((st = end_capture(s2, "block body")) != DINFER_OK) return st;
  // WHILE body: one cached iteration over the block's window
  CK(cudaStreamBeginCaptureToGraph(s2, body_w, nullptr, nullptr, 0, cudaStreamCaptureModeThreadLocal));
  const Fwd fi = iteration_fwd(c, batch, L, B, s0, thr, 1, h_w, 1);
  st = enqueue_forward(c, fi, s2);
  if ((st = end_capture(s2, "window iteration")) != DINFER_OK) return st;
  cudaError_t e = cudaGraphInstantiate(&gs.exec, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return fail(c, DINFER_ECUDA, "graph instantiation failed: %s", cudaGetErrorString(e));
  }
  gs.graph = g;
  return DINFER_OK;
}

// A graph from the context's cache (built on first use).
template <typename Build>
dinfer_status cached_graph(dinfer_ctx* c, const std::tuple<int, int, int, int, int, int>& key, Build build,
                           cudaGraphExec_t* out) {
  GraphSet& gs = c->graphs[key];
  if (!gs.exec) {
    dinfer_status st = build(gs);
    if (st != DINFER_OK) {
      c->graphs.erase(key);
      return st;
    }
  }
  *out = gs.exec;
  return DINFER_OK;
}

dinfer_status check_geometry(dinfer_ctx* c, int batch, int L, int B) {
  if (batch < 1 || batch > c->desc.max_batch) return fail(c, DINFER_EINVAL, "batch %d outside [1, %d]", batch,
                                                          c->desc.max_batch);
  if (L < 1 || L > c->desc.max_seq) return fail(c, DINFER_EINVAL, "sequence length %d outside [1, %d]", L,
                                                c->desc.max_seq);
  if (B < 1 || B > L) return fail(c, DINFER_EINVAL, "block length %d outside [1, %d]", B, L);
  if (batch * B > 1024) return fail(c, DINFER_EINVAL, "batch * block_length must be <= 1024");
  if (!c->bf16 && (size_t)batch * B * c->desc.d_model * 4 > 200 * 1024)
    return fail(c, DINFER_EINVAL, "fp32 models: batch * block_length * d_model too large");
  return DINFER_OK;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

int32_t dinfer_num_weights(const dinfer_model_desc* desc) {
  if (!desc || desc->n_layers < 1) return -1;
  return 1 + 9 * desc->n_layers + 2;
}

const char* dinfer_last_error(const dinfer_ctx* ctx) { return ctx ? ctx->err.c_str() : g_create_error.c_str(); }

void dinfer_destroy(dinfer_ctx* c) {
  if (!c) return;
  if (c->stream) cudaStreamSynchronize(c->stream);
  for (auto& kv : c->graphs) {
    if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    if (kv.second.graph) cudaGraphDestroy(kv.second.graph);
  }
  for (void* p : c->allocs) cudaFree(p);
  if (c->st_host) cudaFreeHost(c->st_host);
  if (c->ev0) cudaEventDestroy(c->ev0);
  if (c->ev1) cudaEventDestroy(c->ev1);
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  if (c->cap_stream2) cudaStreamDestroy(c->cap_stream2);
  if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
  delete c;
}

dinfer_status dinfer_create(const dinfer_model_desc* desc, const void* const* weights, void* stream,
                            dinfer_ctx** out) {
  if (!out) return fail(nullptr, DINFER_EINVAL, "out is NULL");
  *out = nullptr;
  if (const char* why = validate_desc(desc)) return fail(nullptr, DINFER_EINVAL, "%s", why);
  if (!weights) return fail(nullptr, DINFER_EINVAL, "weights is NULL");
  const int nw = dinfer_num_weights(desc);
  for (int i = 0; i < nw; ++i)
    if (!weights[i]) return fail(nullptr, DINFER_EINVAL, "weight %d is NULL", i);
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev < 1) {
    cudaGetLastError();
    return fail(nullptr, DINFER_ECUDA, "no CUDA device");
  }
  if (!set_smem_attrs()) return fail(nullptr, DINFER_ECUDA, "cudaFuncSetAttribute failed");
  if (!get_encode_fn()) return fail(nullptr, DINFER_ECUDA, "cuTensorMapEncodeTiled unavailable");

  dinfer_ctx* c = new dinfer_ctx();
  c->desc = *desc;
  c->bf16 = desc->dtype == DINFER_BF16;
  c->w.assign(weights, weights + nw);
  auto bail = [&](dinfer_status s) {
    g_create_error = c->err;
    dinfer_destroy(c);
    return s;
  };
#define CKC(call)                                                                                     \
  do {                                                                                                \
    cudaError_t e_ = (call);                                                                          \
    if (e_ != cudaSuccess) {                                                                          \
      fail(c, DINFER_ECUDA, "%s: %s", #call, cudaGetErrorString(e_));                                 \
      return bail(DINFER_ECUDA);                                                                      \
    }                                                                                                 \
  } while (0)
#define AL(ptr, bytes)                                   \
  do {                                                   \
    dinfer_status s_ = dalloc(c, &(ptr), (bytes));       \
    if (s_ != DINFER_OK) return bail(s_);                \
  } while (0)

  c->stream = reinterpret_cast<cudaStream_t>(stream);  // NULL: the legacy default stream
  CKC(cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking));
  CKC(cudaStreamCreateWithFlags(&c->cap_stream2, cudaStreamNonBlocking));
  CKC(cudaEventCreate(&c->ev0));
  CKC(cudaEventCreate(&c->ev1));

  const size_t D = desc->d_model, F = desc->ffn, es = c->esize();
  c->max_rows = (size_t)desc->max_batch * desc->max_seq;
  AL(c->h, c->max_rows * D * 4);
  AL(c->xn, c->max_rows * D * es);
  AL(c->q, c->max_rows * D * es);
  AL(c->attn_o, c->max_rows * D * es);
  AL(c->act, c->max_rows * F * es);
  if (desc->n_experts) {
    const size_t E = desc->n_experts, K = desc->top_k, FE = desc->expert_ffn;
    const size_t pairs = c->max_rows * K, chunks = (c->max_rows + kMoeChunk - 1) / kMoeChunk;
    AL(c->moe_logits, c->max_rows * E * 4);
    AL(c->moe_topk_id, pairs * 4);
    AL(c->moe_topk_w, pairs * 4);
    AL(c->moe_rank, pairs * 4);
    AL(c->moe_chunk_cnt, chunks * E * 4);
    AL(c->moe_chunk_base, chunks * E * 4);
    AL(c->moe_tables, 3 * (E + 1) * 4);
    AL(c->moe_inv, pairs * 4);
    AL(c->moe_x, pairs * D * 2);
    AL(c->moe_act, pairs * FE * 2);
    AL(c->moe_y, pairs * D * 4);
  }
  if (!c->bf16) {
    AL(c->qkv32, c->max_rows * 3 * D * 4);
    AL(c->gu32, c->max_rows * 2 * F * 4);
  }
  AL(c->kc, c->cache_layer_elems() * desc->n_layers * es);
  AL(c->vc, c->cache_layer_elems() * desc->n_layers * es);
  const int half = desc->head_dim / 2;
  // at least two positions: the GEMM epilogue steps RoPE by position 1's angle
  const int rope_pos = desc->max_seq < 2 ? 2 : desc->max_seq;
  AL(c->rope_cos, (size_t)rope_pos * half * 4);
  AL(c->rope_sin, (size_t)rope_pos * half * 4);
  {
    // rotary table in double precision: angle = pos * theta^(-2i/hd)
    std::vector<float> cs((size_t)rope_pos * half), sn((size_t)rope_pos * half);
    for (int p = 0; p < rope_pos; ++p)
      for (int i = 0; i < half; ++i) {
        const double inv = std::pow((double)desc->rope_theta, -2.0 * i / desc->head_dim);
        const double ang = (double)p * inv;
        cs[(size_t)p * half + i] = (float)std::cos(ang);
        sn[(size_t)p * half + i] = (float)std::sin(ang);
      }
    CKC(cudaMemcpy(c->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
    CKC(cudaMemcpy(c->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice));
  }
  AL(c->ids, c->max_rows * 4);
  AL(c->mask, c->max_rows);
  AL(c->prompt_dev, c->max_rows * 4);
  AL(c->committed_dev, kMaxBatch * 4);
  AL(c->st, sizeof(DevState));
  CKC(cudaMemset(c->st, 0, sizeof(DevState)));
  CKC(cudaMallocHost((void**)&c->st_host, sizeof(DevState)));
  const int G = num_sms();
  AL(c->gemm_ws, gemm_ws_floats(G) * 4);
  AL(c->lm_part, (size_t)G * 1024 * sizeof(SoftmaxState));
  AL(c->lm_ticket, 16);
  CKC(cudaMemset(c->lm_ticket, 0, 16));

  if (c->bf16) {
    const int nl = desc->n_layers;
    c->m_wq.resize(nl); c->m_wk.resize(nl); c->m_wv.resize(nl); c->m_wo.resize(nl);
    c->m_wg.resize(nl); c->m_wu.resize(nl); c->m_wd.resize(nl);
    c->m_router.resize(nl); c->m_w13.resize(nl); c->m_w2.resize(nl);
    bool ok = true;
    const size_t E = desc->n_experts, FE = desc->expert_ffn;
    for (int l = 0; l < nl; ++l) {
      ok &= make_map(&c->m_wq[l], c->LW(l, 1), D, D, 128);
      ok &= make_map(&c->m_wk[l], c->LW(l, 2), D, D, 128);
      ok &= make_map(&c->m_wv[l], c->LW(l, 3), D, D, 128);
      ok &= make_map(&c->m_wo[l], c->LW(l, 4), D, D, 128);
      if (E) {
        ok &= make_map(&c->m_router[l], c->LW(l, 6), E, D, 128);
        ok &= make_map(&c->m_w13[l], c->LW(l, 7), E * 2 * FE, D, 64);
        ok &= make_map(&c->m_w2[l], c->LW(l, 8), E * D, FE, 128);
      } else {
        ok &= make_map(&c->m_wg[l], c->LW(l, 6), F, D, 64);
        ok &= make_map(&c->m_wu[l], c->LW(l, 7), F, D, 64);
        ok &= make_map(&c->m_wd[l], c->LW(l, 8), D, F, 128);
      }
    }
    ok &= make_map(&c->m_lm, c->W(2 + 9 * nl), desc->vocab, D, 128);
    if (!ok) {
      fail(c, DINFER_EINVAL, "weight tensor maps could not be built (weights must be 16-byte aligned bf16)");
      return bail(DINFER_EINVAL);
    }
  }
  CKC(cudaDeviceSynchronize());
  *out = c;
  return DINFER_OK;
#undef CKC
#undef AL
}

dinfer_status dinfer_set_debug_outputs(dinfer_ctx* c, float* logits, int32_t* tok, float* conf) {
  if (!c) return DINFER_EINVAL;
  c->dbg_logits = logits;
  c->dbg_tok = tok;
  c->dbg_conf = conf;
  return DINFER_OK;
}

dinfer_status dinfer_set_cache_mode(dinfer_ctx* c, int32_t mode, int32_t window) {
  if (!c) return DINFER_EINVAL;
  if (mode < DINFER_CACHE_DUAL || mode > DINFER_CACHE_VICINITY)
    return fail(c, DINFER_EINVAL, "cache mode %d is not one of DINFER_CACHE_DUAL / NONE / PREFIX / VICINITY", mode);
  if (window < 0) return fail(c, DINFER_EINVAL, "vicinity window must be >= 0 (got %d)", window);
  c->cache_mode = mode;
  c->cache_window = mode == DINFER_CACHE_VICINITY ? window : 0;
  return DINFER_OK;
}

dinfer_status dinfer_set_eos(dinfer_ctx* c, int32_t eos_id) {
  if (!c) return DINFER_EINVAL;
  if (eos_id != -1 && (eos_id < 0 || eos_id >= c->desc.vocab || eos_id == c->desc.mask_id))
    return fail(c, DINFER_EINVAL, "eos_id %d is neither -1 nor a token id in [0, vocab) other than mask_id", eos_id);
  c->eos_id = eos_id;
  return DINFER_OK;
}

dinfer_status dinfer_set_debug_hidden(dinfer_ctx* c, float* hidden, void* final_in) {
  if (!c) return DINFER_EINVAL;
  c->dbg_hidden = hidden;
  c->dbg_final = final_in;
  return DINFER_OK;
}

dinfer_status dinfer_sync(dinfer_ctx* c) {
  if (!c) return DINFER_EINVAL;
  return read_status(c);
}

dinfer_status dinfer_moe_experts_touched(dinfer_ctx* c, int64_t* touched) {
  if (!c || !touched) return fail(c, DINFER_EINVAL, "NULL argument");
  uint32_t v = 0;
  uint32_t* dev = &c->st->moe_touched;
  CK(cudaStreamSynchronize(c->stream));
  CK(cudaMemcpy(&v, dev, sizeof(v), cudaMemcpyDeviceToHost));
  CK(cudaMemset(dev, 0, sizeof(v)));
  *touched = v;
  return DINFER_OK;
}

dinfer_status dinfer_prefill_cache(dinfer_ctx* c, int32_t* ids, uint8_t* mask, int32_t batch, int32_t seq_len,
                                   int32_t block_start, int32_t block_len, float threshold, int32_t commit,
                                   int32_t* committed) {
  if (!c) return DINFER_EINVAL;
  if (!ids || !mask) return fail(c, DINFER_EINVAL, "ids / mask is NULL");
  dinfer_status st = check_geometry(c, batch, seq_len, block_len);
  if (st != DINFER_OK) return st;
  if (block_start < 0 || block_start + block_len > seq_len)
    return fail(c, DINFER_EINVAL, "block [%d, %d) outside the sequence", block_start, block_start + block_len);
  if (!(threshold == threshold)) return fail(c, DINFER_EINVAL, "threshold is NaN");
  if (!is_device_ptr(ids) || !is_device_ptr(mask)) return fail(c, DINFER_EINVAL, "ids / mask must be device memory");
  const size_t n = (size_t)batch * seq_len;
  cudaStream_t s = c->stream;
  CK(cudaMemcpyAsync(c->ids, ids, n * 4, cudaMemcpyDeviceToDevice, s));
  CK(cudaMemcpyAsync(c->mask, mask, n, cudaMemcpyDeviceToDevice, s));
  set_block_kernel<<<1, 1, 0, s>>>(c->st, block_start, 1);
  CK(cudaGetLastError());
  Fwd f{batch, seq_len, block_len, batch * seq_len, seq_len, 0, true, commit ? 1 : 0, 1, 0, 0, threshold};
  c->dbg_block_start = block_start;
  if (debug_on(c)) {
    st = enqueue_forward(c, f, s);
    if (st != DINFER_OK) return st;
  } else {
    auto key = std::make_tuple(1, batch, seq_len, block_len, (int)(commit ? 1 : 0) ^ (int)(threshold * 1e6f) * 2, 0);
    GraphSet& gs = c->graphs[key];
    if (!gs.exec) {
      st = build_step_graph(c, f, gs);
      if (st != DINFER_OK) {
        c->graphs.erase(key);
        return st;
      }
    }
    CK(cudaGraphLaunch(gs.exec, s));
  }
  CK(cudaMemcpyAsync(ids, c->ids, n * 4, cudaMemcpyDeviceToDevice, s));
  CK(cudaMemcpyAsync(mask, c->mask, n, cudaMemcpyDeviceToDevice, s));
  if (committed) CK(cudaMemcpyAsync(committed, c->committed_dev, batch * 4, cudaMemcpyDeviceToDevice, s));
  c->cur_batch = batch;
  c->cur_L = seq_len;
  c->cur_B = block_len;
  c->cur_s = block_start;
  c->have_prefill = true;
  return DINFER_OK;
}

dinfer_status dinfer_block_step(dinfer_ctx* c, int32_t* ids, uint8_t* mask, float threshold, int32_t* committed) {
  if (!c) return DINFER_EINVAL;
  if (!c->have_prefill) return fail(c, DINFER_ESTATE, "dinfer_block_step before dinfer_prefill_cache");
  if (!ids || !mask) return fail(c, DINFER_EINVAL, "ids / mask is NULL");
  if (!(threshold == threshold)) return fail(c, DINFER_EINVAL, "threshold is NaN");
  if (!is_device_ptr(ids) || !is_device_ptr(mask)) return fail(c, DINFER_EINVAL, "ids / mask must be device memory");
  const int batch = c->cur_batch, L = c->cur_L, B = c->cur_B;
  const size_t n = (size_t)batch * L;
  cudaStream_t s = c->stream;
  CK(cudaMemcpyAsync(c->ids, ids, n * 4, cudaMemcpyDeviceToDevice, s));
  CK(cudaMemcpyAsync(c->mask, mask, n, cudaMemcpyDeviceToDevice, s));
  set_block_kernel<<<1, 1, 0, s>>>(c->st, c->cur_s, 0);
  CK(cudaGetLastError());
  int r0, r1;
  cache_window(c, c->cur_s, B, L, r0, r1);
  const Fwd f = iteration_fwd(c, batch, L, B, c->cur_s, threshold, 1, 0, 0);
  c->dbg_block_start = c->cur_s;
  dinfer_status st;
  if (debug_on(c)) {
    st = enqueue_forward(c, f, s);
    if (st != DINFER_OK) return st;
  } else {
    auto key = std::make_tuple(2, batch, L, B, (int)(threshold * 1e6f), r0 * 65536 + (r1 - r0));
    GraphSet& gs = c->graphs[key];
    if (!gs.exec) {
      st = build_step_graph(c, f, gs);
      if (st != DINFER_OK) {
        c->graphs.erase(key);
        return st;
      }
    }
    CK(cudaGraphLaunch(gs.exec, s));
  }
  CK(cudaMemcpyAsync(ids, c->ids, n * 4, cudaMemcpyDeviceToDevice, s));
  CK(cudaMemcpyAsync(mask, c->mask, n, cudaMemcpyDeviceToDevice, s));
  if (committed) CK(cudaMemcpyAsync(committed, c->committed_dev, batch * 4, cudaMemcpyDeviceToDevice, s));
  return DINFER_OK;
}

dinfer_status dinfer_generate(dinfer_ctx* c, const int32_t* prompt, int32_t batch, int32_t prompt_len,
                              int32_t gen_length, int32_t block_length, float threshold, int32_t* out,
                              dinfer_stats* stats) {
  if (!c) return DINFER_EINVAL;
  if (!prompt || !out) return fail(c, DINFER_EINVAL, "prompt / out is NULL");
  if (prompt_len < 0 || gen_length < 1 || block_length < 1 || gen_length % block_length)
    return fail(c, DINFER_EINVAL, "gen_length must be a positive multiple of block_length");
  const int L = prompt_len + gen_length;
  dinfer_status st = check_geometry(c, batch, L, block_length);
  if (st != DINFER_OK) return st;
  if (gen_length / block_length > kMaxBlocks) return fail(c, DINFER_EINVAL, "too many blocks");
  if (!(threshold == threshold)) return fail(c, DINFER_EINVAL, "threshold is NaN");
  cudaStream_t s = c->stream;
  const bool p_dev = is_device_ptr(prompt), o_dev = is_device_ptr(out);
  CK(cudaEventRecord(c->ev0, s));
  if (prompt_len > 0)
    CK(cudaMemcpyAsync(c->prompt_dev, prompt, (size_t)batch * prompt_len * 4,
                       p_dev ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, s));
  const int B = block_length, nblk = gen_length / block_length;
  const bool eager = debug_on(c) || getenv("DINFER_NO_GRAPH") != nullptr;
  c->dbg_block_start = -1;  // the block start advances on the device: no hidden-state copies
  set_eos_kernel<<<1, 1, 0, s>>>(c->st, c->eos_id);
  CK(cudaGetLastError());
  if (eager) {
    init_sequence_kernel<<<256, 256, 0, s>>>(c->prompt_dev, c->ids, c->mask, batch, prompt_len, L, c->desc.mask_id,
                                             c->st, nblk);
    CK(cudaGetLastError());
    for (int b = 0; b < nblk; ++b) {
      CK(cudaMemcpyAsync(c->st_host, c->st, sizeof(DevState), cudaMemcpyDeviceToHost, s));
      CK(cudaStreamSynchronize(s));
      if (!c->st_host->any_left || c->st_host->status) break;  // every sequence ended
      begin_block_kernel<<<1, 1, 0, s>>>(c->st);
      Fwd fr{batch, L, B, batch * L, L, 0, true, 1, 1, 0, 0, threshold};
      st = enqueue_forward(c, fr, s);
      if (st != DINFER_OK) return st;
      for (int it = 1; it < B + 1; ++it) {
        CK(cudaMemcpyAsync(c->st_host, c->st, sizeof(DevState), cudaMemcpyDeviceToHost, s));
        CK(cudaStreamSynchronize(s));
        if (!c->st_host->any_masked || c->st_host->status) break;
        const Fwd fi = iteration_fwd(c, batch, L, B, prompt_len + b * B, threshold, 1, 0, 0);
        st = enqueue_forward(c, fi, s);
        if (st != DINFER_OK) return st;
      }
      advance_block_kernel<<<1, 256, 0, s>>>(c->st, B, 0, 0, c->ids, c->mask, batch, L);
      CK(cudaGetLastError());
    }
  } else if (c->cache_mode == DINFER_CACHE_DUAL) {
    // one graph: block loop and iteration loop on the device
    auto key = std::make_tuple(3, batch, prompt_len, gen_length * 4096 + block_length, (int)(threshold * 1e6f), 0);
    cudaGraphExec_t ex;
    st = cached_graph(c, key, [&](GraphSet& gs) {
      return build_generate_graph(c, batch, prompt_len, gen_length, block_length, threshold, gs);
    }, &ex);
    if (st != DINFER_OK) return st;
    CK(cudaGraphLaunch(ex, s));
  } else {
    // windows of host-known positions: the blocks are enqueued from the host
    // (no synchronisation), each as a graph that runs it only while some
    // sequence has masked positions left (refresh, then its cached iterations
    // in a device-side loop)
    init_sequence_kernel<<<256, 256, 0, s>>>(c->prompt_dev, c->ids, c->mask, batch, prompt_len, L, c->desc.mask_id,
                                             c->st, nblk);
    CK(cudaGetLastError());
    const int thr = (int)(threshold * 1e6f);
    for (int b = 0; b < nblk; ++b) {
      const int s0 = prompt_len + b * B;
      int r0, r1;
      cache_window(c, s0, B, L, r0, r1);
      cudaGraphExec_t ex;
      st = cached_graph(c, std::make_tuple(4, batch, L, B, thr, r0 * 65536 + (r1 - r0)),
                        [&](GraphSet& gs) { return build_block_graph(c, batch, L, B, s0, threshold, gs); }, &ex);
      if (st != DINFER_OK) return st;
      CK(cudaGraphLaunch(ex, s));
    }
  }
  // output: ids [batch, L]
  CK(cudaMemcpyAsync(out, c->ids, (size_t)batch * L * 4, o_dev ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost,
                     s));
  CK(cudaEventRecord(c->ev1, s));
  st = read_status(c);
  if (stats) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, c->ev0, c->ev1);
    stats->n_blocks = nblk;
    stats->iterations = c->st_host->total_iterations;
    stats->refreshes = c->st_host->refreshes;
    stats->ms_device = ms;
    if (stats->iters_per_block)
      for (int b = 0; b < nblk && b < kMaxBlocks; ++b) stats->iters_per_block[b] = c->st_host->iters_per_block[b];
  }
  return st;
}

}  // extern "C"

// ===========================================================================
// kernel-level entry points (include/dinfer_ops.h)
// ===========================================================================
namespace {
constexpr size_t kOpStateBytes = 64 * 1024;          // DevState
constexpr size_t kOpTicketBytes = 4u << 20;          // zeroed counters
constexpr size_t kOpDataBytes = 160u << 20;
struct OpWs {
  DevState* st;
  int* tickets;
  uint8_t* data;
  size_t data_bytes;
};
bool op_ws(void* ws, size_t bytes, OpWs& o) {
  if (!ws || bytes < kOpStateBytes + kOpTicketBytes + 4096) return false;
  uint8_t* p = reinterpret_cast<uint8_t*>(ws);
  o.st = reinterpret_cast<DevState*>(p);
  o.tickets = reinterpret_cast<int*>(p + kOpStateBytes);
  o.data = p + kOpStateBytes + kOpTicketBytes;
  o.data_bytes = bytes - kOpStateBytes - kOpTicketBytes;
  return true;
}
}  // namespace

extern "C" {

size_t dinfer_op_workspace_bytes(void) { return kOpStateBytes + kOpTicketBytes + kOpDataBytes; }

dinfer_status dinfer_op_gemm_bf16(const void* X, const void* W, float* Y, int32_t M, int32_t N, int32_t K,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  dinfer_ctx* c = nullptr;
  if (!X || !W || !Y) return fail(c, DINFER_EINVAL, "NULL operand");
  if (M < 1 || M > (1 << 20) || N < 128 || N % 128 || K < 64 || K % 64)
    return fail(c, DINFER_EINVAL, "unsupported GEMM shape");
  OpWs o;
  if (!op_ws(workspace, workspace_bytes, o)) return fail(c, DINFER_EINVAL, "workspace too small");
  const int G = num_sms();
  if (gemm_ws_floats(G) * 4 > o.data_bytes) return fail(c, DINFER_EINVAL, "workspace too small");
  const int BN = bn_for_rows(M);
  if ((size_t)((M + BN - 1) / BN) * (N / 128) * 4 > kOpTicketBytes) return fail(c, DINFER_EINVAL, "too many tiles");
  if (!set_smem_attrs()) return fail(c, DINFER_ECUDA, "cudaFuncSetAttribute failed");
  const PairMode pm = pair_mode(M, N / 128, false);
  const bool pair = pm != PAIR_NONE;
  GemmMaps m{};
  if (!make_map(&m.a[0], W, N, K, 128) || !make_map(&m.b, X, M, K, pair ? pair_bn(pm) / 2 : BN))
    return fail(c, DINFER_EINVAL, "tensor map encoding failed (alignment?)");
  GemmArgs a{};
  a.M = M; a.N = N; a.K = K; a.n_tiles = N / 128; a.a_mode = A_SINGLE;
  a.out_f32 = Y; a.ldo = N;
  a.ws = reinterpret_cast<float*>(o.data); a.status = o.st; a.state = o.st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CK(pair ? launch_gemm_tc2(m, a, s, pm) : launch_gemm_tc(m, a, BN, s));
  return DINFER_OK;
}

dinfer_status dinfer_op_lmhead_bf16(const void* X, const void* W, int32_t M, int32_t V, int32_t K, int32_t mask_id,
                                    float scale, int32_t* tok, float* conf, float* logits, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  dinfer_ctx* c = nullptr;
  if (!X || !W || !tok || !conf) return fail(c, DINFER_EINVAL, "NULL operand");
  if (M < 1 || M > 1024 || V < 8 || V % 8 || K < 64 || K % 64) return fail(c, DINFER_EINVAL, "unsupported shape");
  OpWs o;
  if (!op_ws(workspace, workspace_bytes, o)) return fail(c, DINFER_EINVAL, "workspace too small");
  const int G = num_sms();
  if ((size_t)G * 1024 * sizeof(SoftmaxState) > o.data_bytes) return fail(c, DINFER_EINVAL, "workspace too small");
  if (!set_smem_attrs()) return fail(c, DINFER_ECUDA, "cudaFuncSetAttribute failed");
  const int BN = bn_for_rows(M);
  GemmMaps m{};
  if (!make_map(&m.a[0], W, V, K, 128) || !make_map(&m.b, X, M, K, BN))
    return fail(c, DINFER_EINVAL, "tensor map encoding failed (alignment?)");
  GemmArgs ga{};
  ga.M = M; ga.N = V; ga.K = K; ga.n_tiles = (V + 127) / 128; ga.a_mode = A_SINGLE;
  ga.status = o.st; ga.state = o.st;
  DecodeArgs dec{};
  dec.M = M; dec.batch = 1; dec.L = M; dec.B = M; dec.commit = 0;
  dec.tok_out = tok; dec.conf_out = conf; dec.state = o.st;
  dec.partials = reinterpret_cast<SoftmaxState*>(o.data); dec.ticket = o.tickets;
  LmArgs la{V, mask_id, scale, logits, dec};
  CK(launch_lmhead_tc(m, ga, la, BN, reinterpret_cast<cudaStream_t>(stream)));
  return DINFER_OK;
}

dinfer_status dinfer_op_attention_bf16(const void* q, const void* k, const void* v, void* out, int32_t batch,
                                       int32_t rows_per_seq, int32_t L, int32_t heads, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  dinfer_ctx* c = nullptr;
  if (!q || !k || !v || !out) return fail(c, DINFER_EINVAL, "NULL operand");
  if (batch < 1 || rows_per_seq < 1 || L < 1 || heads < 1) return fail(c, DINFER_EINVAL, "unsupported shape");
  OpWs o{};
  if (workspace && !op_ws(workspace, workspace_bytes, o)) return fail(c, DINFER_EINVAL, "workspace too small");
  if (!set_smem_attrs()) return fail(c, DINFER_ECUDA, "cudaFuncSetAttribute failed");
  const AttnPlan ap = plan_attention(batch, rows_per_seq, heads, L);
  if (launch_attention(q, k, v, out, batch, rows_per_seq, heads, L, ap, o.st,
                       reinterpret_cast<cudaStream_t>(stream)) == cudaErrorInvalidValue)
    return fail(c, DINFER_EINVAL, "tensor map encoding failed (alignment?)");
  CK(cudaGetLastError());
  return DINFER_OK;
}

}  // extern "C"

extern "C" dinfer_status dinfer_op_moe_ffn_bf16(const void* X, const void* router, const void* w13, const void* w2,
                                                int32_t M, int32_t d, int32_t E, int32_t K, int32_t fe, float* out,
                                                int32_t* topk_id, float* topk_w, void* workspace,
                                                size_t workspace_bytes, void* stream) {
  dinfer_ctx* c = nullptr;
  if (!X || !router || !w13 || !w2 || !out) return fail(c, DINFER_EINVAL, "NULL operand");
  if (M < 1 || d < 128 || d % 128 || d / 16 > 512 || E < 1 || E > 64 || K < 1 || K > kMoeMaxK || K > E || fe < 64 ||
      fe % 64)
    return fail(c, DINFER_EINVAL, "unsupported MoE shape");
  OpWs o;
  if (!op_ws(workspace, workspace_bytes, o)) return fail(c, DINFER_EINVAL, "workspace too small");
  if (!set_smem_attrs()) return fail(c, DINFER_ECUDA, "cudaFuncSetAttribute failed");
  // carve the data region
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void* p = o.data + off;
    off += (bytes + 255) & ~size_t(255);
    return p;
  };
  const size_t pairs = (size_t)M * K, chunks = (M + kMoeChunk - 1) / kMoeChunk;
  MoeBufs b;
  b.ws = (float*)take(gemm_ws_floats(num_sms()) * 4);
  b.logits = (float*)take((size_t)M * E * 4);
  b.topk_id = (int*)take(pairs * 4);
  b.topk_w = (float*)take(pairs * 4);
  b.rank = (int*)take(pairs * 4);
  b.chunk_cnt = (int*)take(chunks * E * 4);
  b.chunk_base = (int*)take(chunks * E * 4);
  b.tables = (int*)take(3 * ((size_t)E + 1) * 4);
  b.inv = (int*)take(pairs * 4);
  b.x = take(pairs * d * 2);
  b.act = take(pairs * fe * 2);
  b.y = (float*)take(pairs * d * 4);
  b.st = o.st;
  if (off > o.data_bytes) return fail(c, DINFER_EINVAL, "workspace too small for this MoE shape");
  CUtensorMap mr, m13, m2;
  if (!make_map(&mr, router, E, d, 128) || !make_map(&m13, w13, (size_t)E * 2 * fe, d, 64) ||
      !make_map(&m2, w2, (size_t)E * d, fe, 128))
    return fail(c, DINFER_EINVAL, "tensor map encoding failed (alignment?)");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CK(enqueue_moe_ffn(b, X, M, d, E, K, fe, mr, m13, m2, s));
  CK(cudaMemsetAsync(out, 0, (size_t)M * d * 4, s));
  CK(launchk(moe_combine_norm_kernel<__nv_bfloat16>, dim3(M), dim3(((d / 16 + 31) / 32) * 32), 0, s, 1, out,
             (const float*)b.y,
             (const float*)b.topk_w, (const int*)b.inv, K, (const __nv_bfloat16*)nullptr, (__nv_bfloat16*)nullptr,
             d, 0.f, M, M, 0, 0, (const DevState*)o.st));
  if (topk_id) CK(cudaMemcpyAsync(topk_id, b.topk_id, pairs * 4, cudaMemcpyDeviceToDevice, s));
  if (topk_w) CK(cudaMemcpyAsync(topk_w, b.topk_w, pairs * 4, cudaMemcpyDeviceToDevice, s));
  return DINFER_OK;
}

// ===========================================================================
// allocation-free GEMM entry point (include/dinfer_ops.h)
// ===========================================================================
namespace {
// Device addresses of the fixed scratch and its status word, looked up once
// per device under the set-up mutex.
float* g_noalloc_ptr[kMaxDevices] = {};
DevState* g_noalloc_state_ptr[kMaxDevices] = {};

dinfer_status noalloc_setup(int* dev_out) {
  dinfer_ctx* c = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(c, DINFER_ECUDA, "no current CUDA device");
  }
  *dev_out = dev;
  std::lock_guard<std::mutex> lk(g_setup_mutex);
  if (g_noalloc_ptr[dev]) return DINFER_OK;
  // the host-side names of the __device__ arrays are not device addresses
  void* p = nullptr;
  void* q = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e == cudaSuccess) e = cudaGetSymbolAddress(&q, g_noalloc_state);
  if (e != cudaSuccess || !p || !q) {
    cudaGetLastError();
    return fail(c, DINFER_ECUDA, "cudaGetSymbolAddress of the fixed scratch failed: %s", cudaGetErrorString(e));
  }
  g_noalloc_state_ptr[dev] = reinterpret_cast<DevState*>(q);
  g_noalloc_ptr[dev] = reinterpret_cast<float*>(p);
  return DINFER_OK;
}
}  // namespace

extern "C" dinfer_status dinfer_op_gemm_bf16_noalloc(const void* X, const void* W, float* Y, int32_t M, int32_t N,
                                                     int32_t K, void* stream) {
  dinfer_ctx* c = nullptr;
  if (!X || !W || !Y) return fail(c, DINFER_EINVAL, "NULL operand");
  if (M < 1 || M > kNoAllocMaxRows)
    return fail(c, DINFER_EINVAL, "the allocation-free GEMM takes 1 <= M <= %d token rows (got %d)", kNoAllocMaxRows,
                M);
  if (N < 128 || N % 128 || K < 64 || K % 64) return fail(c, DINFER_EINVAL, "unsupported GEMM shape");
  int dev = 0;
  dinfer_status st = noalloc_setup(&dev);
  if (st != DINFER_OK) return st;
  if (!set_smem_attrs()) return fail(c, DINFER_ECUDA, "cudaFuncSetAttribute failed");
  constexpr int BN = 64;  // M <= 64: one token tile
  GemmMaps m{};
  if (!make_map(&m.a[0], W, N, K, 128) || !make_map(&m.b, X, M, K, BN))
    return fail(c, DINFER_EINVAL, "tensor map encoding failed (alignment?)");
  GemmArgs a{};
  a.M = M; a.N = N; a.K = K; a.n_tiles = N / 128; a.a_mode = A_SINGLE;
  a.out_f32 = Y; a.ldo = N;
  a.m_tiles = 1;
  a.k_tiles = K / 64;
  // the schedule dinfer_op_gemm_bf16 takes; the scratch holds two partial
  // tiles for each of at most kNoAllocMaxCtas CTAs
  const GemmSched gs = launch_schedule(a, BN, false, false);
  a.stream_k = gs.stream_k;
  a.grid = std::min(gs.grid, kNoAllocMaxCtas);
  if ((unsigned long long)a.n_tiles * (a.stream_k ? a.k_tiles : 1) * a.grid >= (1ull << 32))
    return fail(c, DINFER_EINVAL, "GEMM too large for the allocation-free entry point");
  a.ws = g_noalloc_ptr[dev];
  a.status = g_noalloc_state_ptr[dev];
  a.state = g_noalloc_state_ptr[dev];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // No partial tile must start at zero: every slot the fixup reads is written
  // by the GEMM launch of the same call.
  CK(launchk(gemm_tc_kernel<BN>, dim3(a.grid), dim3(kGemmThreads), GemmKCfg<BN>::kSmem, s, 1, m, a));
  if (a.stream_k) CK(launchk(splitk_fixup_kernel<BN>, dim3(a.n_tiles * 4), dim3(128), 0, s, 1, a));
  return DINFER_OK;
}

extern "C" dinfer_status dinfer_op_gemm_bf16_noalloc_status(void* stream) {
  dinfer_ctx* c = nullptr;
  int dev = 0;
  dinfer_status st = noalloc_setup(&dev);
  if (st != DINFER_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word[5] = {};  // status, diag[4]
  const size_t off = offsetof(DevState, status);
  CK(cudaStreamSynchronize(s));
  CK(cudaMemcpyFromSymbolAsync(&word[0], g_noalloc_state, 4, off, cudaMemcpyDeviceToHost, s));
  CK(cudaMemcpyFromSymbolAsync(&word[1], g_noalloc_state, 16, offsetof(DevState, diag), cudaMemcpyDeviceToHost, s));
  CK(cudaStreamSynchronize(s));
  if (word[0] == 0) return DINFER_OK;
  const uint32_t zero[5] = {};
  CK(cudaMemcpyToSymbolAsync(g_noalloc_state, &zero[0], 4, off, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyToSymbolAsync(g_noalloc_state, &zero[1], 16, offsetof(DevState, diag), cudaMemcpyHostToDevice, s));
  CK(cudaStreamSynchronize(s));
  return fail(c, DINFER_EDEVICE,
              "allocation-free GEMM: device status word 0x%x (1 = a pipeline wait timed out; the output of the "
              "calls since the last check is not valid); first timeout: site 0x%x block 0x%x z/step 0x%x thread %u",
              word[0], word[1], word[2], word[3], word[4]);
}
