// gemm_launch.cu — instantiations of the tcgen05 GEMMs: CTA-pair kernels for many tokens,
// split-K kernels (with their fused reductions) for few tokens.
#include "gemm_tc.cuh"
#include "launch.h"

namespace gqa {

using PairSmem = GemmPairSmem<6>;
constexpr int kSkinnyStages = 8;  // one CTA per SM, 8 x 24 KB in flight (64 token columns)
using SkinnySmem = GemmSmem<64, kSkinnyStages>;
// at most 32 tokens: a 4 KB activation stage, so 11 stages (176 KB of weights) are in flight
constexpr int kNarrowStages = 11;
using NarrowSmem = GemmSmem<32, kNarrowStages>;


cudaError_t configure_gemm_kernels() {
  cudaError_t e;
  e = cudaFuncSetAttribute(gemm_tc_pair_kernel<6, kQkvRope>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairSmem::kBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_tc_pair_kernel<6, kStoreF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairSmem::kBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_splitk_cluster_kernel<kSplitKQkv, kSkinnyStages, 64>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, SkinnySmem::kBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_splitk_cluster_kernel<kSplitKOut, kSkinnyStages, 64>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, SkinnySmem::kBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_splitk_cluster_kernel<kSplitKQkv, kNarrowStages, 32>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, NarrowSmem::kBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_splitk_cluster_kernel<kSplitKOut, kNarrowStages, 32>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, NarrowSmem::kBytes);
}

int gemm_pair_max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = PairSmem::kBytes;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_pair_kernel<6, kQkvRope>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_gemm_qkv_rope(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bt,
                                 const GemmParams& p, int grid, cudaStream_t s) {
  return launch_pdl(gemm_tc_pair_kernel<6, kQkvRope>, dim3(grid), dim3(192), PairSmem::kBytes, s, 0, a, b, bt, p);
}

cudaError_t launch_gemm_store_f32(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bt,
                                  const GemmParams& p, int grid, cudaStream_t s) {
  return launch_pdl(gemm_tc_pair_kernel<6, kStoreF32>, dim3(grid), dim3(192), PairSmem::kBytes, s, 0, a, b, bt, p);
}

// One cluster of p.splits CTAs per 128-feature tile (cluster rank = k split).
// The activation map's box must be splitk_token_tile(p.N) rows.
template <int EPI>
static cudaError_t launch_splitk(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t s) {
  // the reduction serves 2..8 splits (cluster sizes) of at most 64 tokens
  if (p.splits < 2 || p.splits > 8 || p.N < 1 || p.N > 64) return cudaErrorInvalidValue;
  if (p.N <= 32)
    return launch_pdl(gemm_splitk_cluster_kernel<EPI, kNarrowStages, 32>, dim3(p.m_tiles * p.splits), dim3(192),
                      NarrowSmem::kBytes, s, p.splits, a, b, p);
  return launch_pdl(gemm_splitk_cluster_kernel<EPI, kSkinnyStages, 64>, dim3(p.m_tiles * p.splits), dim3(192),
                    SkinnySmem::kBytes, s, p.splits, a, b, p);
}

int splitk_token_tile(int n_tok) { return n_tok <= 32 ? 32 : 64; }

cudaError_t launch_gemm_splitk_qkv(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                   cudaStream_t s) {
  return launch_splitk<kSplitKQkv>(a, b, p, s);
}

cudaError_t launch_gemm_splitk_out(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                   cudaStream_t s) {
  return launch_splitk<kSplitKOut>(a, b, p, s);
}

}  // namespace gqa
