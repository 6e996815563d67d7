// Host-only driver for tests/test_plans.py: runs the launch planners of the
// row-slab, FP8 row-slab, FP8 split-activation and tile kernels over a grid of shapes and launch
// configurations and prints one JSON object per accepted plan.  No CUDA call
// is made; the kernels' headers are included for their host planners only.
#include <cstdio>

#include "sgr_rows.cuh"
#include "sgr_w8.cuh"
#include "sgr_w8s.cuh"
#include "sgr_gemm.cuh"
#include "sgr_pair.cuh"

int main() {
  const int sms = 152;
  const int Ms[] = {1, 3, 16, 17, 32, 40, 48, 64, 100, 128, 200, 256, 1024};
  // The latent-MoE shapes, ragged and tiny ones, and the large ends: N = 2^17
  // (past the row slab's 128 rows per CTA), K = 65536 and K = 2^20 (the
  // library's largest K).
  const int NKs[][2] = {{7168, 3584}, {3584, 7168}, {520, 264}, {8, 3584}, {1024, 1024}, {152, 1792},
                        {131072, 64}, {152, 65536}, {16, 1048576}};
  for (auto& nk : NKs) {
    const int N = nk[0], K = nk[1];
    for (int M : Ms) {
      const int nt = (M + 15) / 16 * 16;
      // row-slab kernel
      for (int ksp : {0, 2})
      for (int rb : {0, 8, 24, 32, 48, 64, 128})
        for (int kb : {1, 2, 4, 8})
          for (int st : {2, 3, 4, 6, 8}) {
            sgr_config c = {};
            c.path = SGR_PATH_TC_ROWS;
            c.ctas_per_sm = 1;
            c.rows_per_stage = rb;
            c.k_blocks_per_stage = kb;
            c.stages = st;
            c.token_tile = nt;
            c.k_split = ksp;
            sgr::RowsParams p;
            int grid = 0;
            size_t smem = 0;
            if (sgr::rows_plan(c, sms, M, N, K, &p, &grid, &smem) != SGR_OK) continue;
            const size_t w_ring = (size_t)st * kb * p.RB * 128, a_ring = (size_t)st * kb * p.NT * 128;
            std::printf("{\"kind\": \"rows\", \"M\": %d, \"N\": %d, \"K\": %d, \"RB\": %d, \"NT\": %d, \"G\": %d, "
                        "\"kbps\": %d, \"stages\": %d, \"prefetch\": %d, \"k_stages\": %d, \"tmem_cols\": %d, "
                        "\"issuers\": %d, \"mode\": %d, \"threads\": %d, \"grid\": %d, \"smem\": %zu, \"w_ring\": %zu, "
                        "\"a_ring\": %zu, \"slack\": %u, \"ksplit\": %d}\n",
                        M, N, K, p.RB, p.NT, p.groups, p.kbps, p.stages, p.prefetch, p.k_stages, p.tmem_cols,
                        p.issuers, sgr::rows_epi_mode(p.NT, p.groups), sgr::rows_threads(sgr::rows_epi_mode(p.NT, p.groups)),
                        grid, smem, w_ring, a_ring, (unsigned)sgr::rows_tail_slack(p.stages, p.kbps, p.RB, p.NT), p.ksplit);
          }
      // FP8 row-slab kernel
      for (int rb : {0, 8, 24, 32, 64, 128})
        for (int kb : {2, 4, 6, 8})
          for (int st : {2, 3, 4, 6, 12})
            for (int sa : {2, 3, 8}) {
              sgr_config c = {};
              c.path = SGR_PATH_W8;
              c.ctas_per_sm = 1;
              c.rows_per_stage = rb;
              c.k_blocks_per_stage = kb;
              c.stages = st;
              c.prefetch_stages = sa;
              c.token_tile = nt;
              for (int fp4 = 0; fp4 <= 1; ++fp4) {
                sgr::W8Params p;
                int grid = 0;
                size_t smem = 0;
                if (sgr::w8_plan(c, sms, M, N, K, &p, &grid, &smem, fp4 != 0) != SGR_OK) continue;
                std::printf("{\"kind\": \"w8\", \"fp4\": %d, \"M\": %d, \"N\": %d, \"K\": %d, \"RB\": %d, \"NT\": %d, "
                            "\"G\": %d, \"kbps\": %d, \"stages\": %d, \"a_stages\": %d, \"k_stages\": %d, "
                            "\"slots\": %d, \"acc_cols\": %d, \"tmem_cols\": %d, \"conv_warps\": %d, \"grid\": %d, "
                            "\"smem\": %zu, \"rtile\": %u, \"w_stage\": %u, \"w_ring\": %zu, \"a_ring\": %zu}\n",
                            fp4, M, N, K, p.RB, p.NT, p.groups, p.kbps, p.stages, p.a_stages, p.k_stages, p.slots,
                            p.acc_cols, p.tmem_cols, p.conv_warps, grid, smem, sgr::w8_rtile_bytes(p.RB, p.NT),
                            sgr::wring_stage_bytes(fp4 != 0, p.kbps, p.RB),
                            (size_t)p.stages * sgr::wring_stage_bytes(fp4 != 0, p.kbps, p.RB),
                            (size_t)p.a_stages * sgr::w8_astage_bytes(p.kbps, p.NT));
              }
            }
      // FP8 split-activation kernel (up to 16 tokens)
      if (M <= sgr::kW8sMaxTokens)
        for (int rb : {0, 24, 32, 48, 64})
          for (int kb : {1, 2, 4, 8})
            for (int st : {2, 3, 4, 7, 8}) {
              sgr_config c = {};
              c.path = SGR_PATH_W8S;
              c.ctas_per_sm = 1;
              c.rows_per_stage = rb;
              c.k_blocks_per_stage = kb;
              c.stages = st;
              c.token_tile = M <= 8 ? 8 : 16;
              sgr::W8sParams p;
              int grid = 0;
              size_t smem = 0;
              if (sgr::w8s_plan(c, sms, M, N, K, K, &p, &grid, &smem) != SGR_OK) continue;
              std::printf("{\"kind\": \"w8s\", \"M\": %d, \"N\": %d, \"K\": %d, \"RB\": %d, \"NT\": %d, \"G\": %d, "
                          "\"kbps\": %d, \"stages\": %d, \"k_stages\": %d, \"kb\": %d, \"kbp\": %d, "
                          "\"issuers\": %d, \"tmem_cols\": %d, \"grid\": %d, \"smem\": %zu, \"ring\": %zu, "
                          "\"span\": %u}\n",
                          M, N, K, p.RB, p.NT, p.groups, p.kbps, p.stages, p.k_stages, p.kb, p.kbp, p.issuers,
                          p.tmem_cols, grid, smem, (size_t)p.stages * sgr::w8s_wstage_bytes(p.kbps, p.RB),
                          sgr::w8s_operand_span(p.kbp, p.NT, p.RB));
            }
      // tile kernel
      for (int tn : {64, 128, 192, 256})
        for (int kb : {1, 2, 4})
          for (int st : {2, 4, 7})
            for (int split : {1, 2, 3, 4}) {
              sgr_config c = {};
              c.path = SGR_PATH_TILE;
              c.ctas_per_sm = 1;
              c.tile_n = tn;
              c.k_blocks_per_stage = kb;
              c.stages = st;
              c.k_split = split;
              sgr::TileParams p;
              int grid = 0;
              size_t smem = 0;
              if (sgr::tile_plan(c, sms, M, N, K, &p, &grid, &smem) != SGR_OK) continue;
              std::printf("{\"kind\": \"tile\", \"M\": %d, \"N\": %d, \"K\": %d, \"NT\": %d, \"kbps\": %d, "
                          "\"stages\": %d, \"split\": %d, \"m_tiles\": %d, \"n_tiles\": %d, \"k_blocks\": %d, "
                          "\"kb_split\": %d, \"tmem_cols\": %d, \"grid\": %d, \"smem\": %zu}\n",
                          M, N, K, p.NT, p.kbps, p.stages, split, p.m_tiles, p.n_tiles, p.k_blocks, p.kb_split,
                          p.tmem_cols, grid, smem);
            }
      // 2-CTA tile kernel (76 pairs: a 152-SM device whose SMs all pair up)
      for (int tn : {64, 96, 128, 192, 256})
        for (int kb : {1, 2, 4})
          for (int st : {2, 4, 7, 10, 16}) {
            sgr_config c = {};
            c.path = SGR_PATH_PAIR;
            c.ctas_per_sm = 1;
            c.tile_n = tn;
            c.k_blocks_per_stage = kb;
            c.stages = st;
            sgr::PairParams p;
            int grid = 0;
            size_t smem = 0;
            if (sgr::pair_plan(c, sms / 2, M, N, K, &p, &grid, &smem) != SGR_OK) continue;
            std::printf("{\"kind\": \"pair\", \"M\": %d, \"N\": %d, \"K\": %d, \"NT\": %d, \"kbps\": %d, "
                        "\"stages\": %d, \"m_tiles\": %d, \"n_tiles\": %d, \"k_blocks\": %d, \"tmem_cols\": %d, "
                        "\"grid\": %d, \"smem\": %zu, \"stage_bytes\": %u}\n",
                        M, N, K, p.NT, p.kbps, p.stages, p.m_tiles, p.n_tiles, p.k_blocks, p.tmem_cols, grid, smem,
                        sgr::pair_stage_bytes(p.NT, p.kbps));
          }
    }
  }
  // Default row-slab configurations (the K-split rule among them).
  const int dNKs[][2] = {{7168, 3584}, {3584, 7168}, {2048, 8192}, {1024, 4096}, {7168, 2048}, {2048, 2048},
                         {4096, 14336}, {4864, 4096}, {4872, 4096}, {8, 65536}, {2560, 10240}};
  for (auto& nk : dNKs)
    for (int M : {1, 16, 17, 40, 64, 65, 128}) {
      const int N = nk[0], K = nk[1];
      if (!sgr::rows_supported(sms, M, N, K)) continue;
      sgr_config c = {};
      sgr::rows_default_config(sms, M, N, K, &c);
      sgr::RowsParams p;
      int grid = 0;
      size_t smem = 0;
      const int rc = sgr::rows_plan(c, sms, M, N, K, &p, &grid, &smem);
      std::printf("{\"kind\": \"rows_default\", \"M\": %d, \"N\": %d, \"K\": %d, \"k_split\": %d, \"kbps\": %d, "
                  "\"stages\": %d, \"token_tile\": %d, \"plan_ok\": %d, \"RB\": %d}\n",
                  M, N, K, c.k_split, c.k_blocks_per_stage, c.stages, c.token_tile, rc == SGR_OK ? 1 : 0,
                  rc == SGR_OK ? p.RB : 0);
    }
  return 0;
}
