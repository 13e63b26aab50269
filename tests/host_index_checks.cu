// Host-side checks of the GEMMs' index arithmetic: the library's own
// __host__ __device__ helpers, compiled by nvcc and run on the CPU (no GPU is
// touched).  Run by tests/test_host_index_checks.py.
//   * the pair-CTA GEMM's grouped tile order (pair_tile_coords) is a
//     bijection onto (weight pair tile, token tile) and pair_tile_index is
//     its inverse; every window of one group's tiles stays inside that
//     group's token tiles;
//   * the stream-K schedule (Sched) splits the units into non-empty
//     contiguous ranges, one per CTA, whose owners agree with start();
//   * the TMEM accumulator stride of each tile width leaves two
//     accumulators inside the columns the one-CTA and pair kernels allocate.
#include <cstdio>
#include <vector>

#include "../block_denoising_gb300/csrc/gemm_tc2.cuh"

using namespace dinfer;

static long long g_fail = 0;
#define CHECK(cond, ...)                   \
  do {                                     \
    if (!(cond)) {                         \
      if (g_fail < 20) {                   \
        std::printf("FAIL %s: ", #cond);   \
        std::printf(__VA_ARGS__);          \
        std::printf("\n");                 \
      }                                    \
      ++g_fail;                            \
    }                                      \
  } while (0)

static void pair_tile_order() {
  long long cases = 0;
  for (int m_tiles = 1; m_tiles <= 100; ++m_tiles) {
    for (int np_tiles = 1; np_tiles <= 96; ++np_tiles) {
      const int T = m_tiles * np_tiles;
      std::vector<int> seen(T, 0);
      for (int t = 0; t < T; ++t) {
        int np = -1, mt = -1;
        pair_tile_coords(t, m_tiles, np_tiles, np, mt);
        const bool in = np >= 0 && np < np_tiles && mt >= 0 && mt < m_tiles;
        CHECK(in, "t %d of %d x %d -> (%d, %d)", t, np_tiles, m_tiles, np, mt);
        if (!in) continue;
        CHECK(!seen[np * m_tiles + mt], "t %d repeats (%d, %d)", t, np, mt);
        seen[np * m_tiles + mt] = 1;
        CHECK(pair_tile_index(np, mt, m_tiles, np_tiles) == t, "index(%d, %d) != %d", np, mt, t);
        // the tiles of one group of kPairGroupM token tiles are consecutive
        CHECK(mt / kPairGroupM == t / (kPairGroupM * np_tiles), "t %d (token tile %d) outside its group", t, mt);
        ++cases;
      }
    }
  }
  std::printf("pair tile order: %lld tiles checked\n", cases);
}

static void stream_k_ranges() {
  const unsigned Us[] = {1, 2, 3, 7, 64, 96, 152, 153, 999, 2048, 6144, 64 * 96, 32 * 64 * 3, 576 * 64, 1000003};
  const unsigned Gs[] = {1, 2, 3, 76, 151, 152};
  long long cases = 0;
  for (unsigned U : Us) {
    for (unsigned G0 : Gs) {
      const unsigned G = G0 < U ? G0 : U;  // the launchers never start more CTAs than units
      Sched s{U, 1, G};
      CHECK(s.start(0) == 0 && s.start(G) == U, "U %u G %u: ends %u %u", U, G, s.start(0), s.start(G));
      for (unsigned c = 0; c < G; ++c) {
        const unsigned a = s.start(c), b = s.start(c + 1);
        CHECK(b > a, "U %u G %u: CTA %u empty", U, G, c);
        CHECK(s.owner(a) == (int)c && s.owner(b - 1) == (int)c, "U %u G %u: CTA %u owners %d %d", U, G, c,
              s.owner(a), s.owner(b - 1));
        ++cases;
      }
    }
  }
  std::printf("stream-K ranges: %lld CTAs checked\n", cases);
}

template <int BN>
static void tmem_fit(int alloc_cols) {
  CHECK(acc_stride<BN>() >= BN, "BN %d: stride %d", BN, acc_stride<BN>());
  CHECK(2 * acc_stride<BN>() <= alloc_cols, "BN %d: two accumulators need %d of %d columns", BN,
        2 * acc_stride<BN>(), alloc_cols);
}

int main() {
  pair_tile_order();
  stream_k_ranges();
  tmem_fit<64>(GemmKCfg<64>::kTmemCols);
  tmem_fit<128>(GemmKCfg<128>::kTmemCols);
  tmem_fit<256>(GemmKCfg<256>::kTmemCols);
  tmem_fit<128>(Gemm2Cfg<128>::kTmemCols);  // pair-CTA tiles: each CTA's accumulators
  tmem_fit<176>(Gemm2Cfg<176>::kTmemCols);
  tmem_fit<256>(Gemm2Cfg<256>::kTmemCols);
  std::printf("host index checks: %lld failures\n", g_fail);
  return g_fail ? 1 : 0;
}
