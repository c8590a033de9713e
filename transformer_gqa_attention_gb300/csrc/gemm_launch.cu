// gemm_launch.cu — instantiations of the tcgen05 GEMMs: CTA-pair kernels for many tokens,
// split-K kernels (with their fused reductions) for few tokens.
#include "gemm_tc.cuh"
#include "launch.h"

namespace gqa {

using PairSmem = GemmPairSmem<6>;
// Stage rings: two CTAs per SM (~100 KB of shared memory each) with 4 stages of 16 KB weights
// + 8 KB activations (64 token columns) or 5 stages of 16 + 4 KB (at most 32 tokens); one CTA
// per SM with 8 stages of 16 + 8 KB (the W_O kernel at 33-64 tokens, 4 splits).
constexpr int kSkinnyStages = 4;
using SkinnySmem = GemmSmem<64, kSkinnyStages>;
constexpr int kNarrowStages = 5;
using NarrowSmem = GemmSmem<32, kNarrowStages>;
constexpr int kDeepStages = 8;
using DeepSmem = GemmSmem<64, kDeepStages>;


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
  e = cudaFuncSetAttribute(gemm_splitk_cluster_kernel<kSplitKOut, kDeepStages, 64>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, DeepSmem::kBytes);
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
// Ring per case: at most 32 tokens, the 5-stage 32-column ring; 33-64 tokens, the 4-stage
// 64-column ring for Q/K/V and the 8-stage one (one CTA per SM) for W_O.
template <int EPI>
static cudaError_t launch_splitk(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p, cudaStream_t s) {
  // the reduction serves 2..8 splits (cluster sizes) of at most 64 tokens
  if (p.splits < 2 || p.splits > 8 || p.N < 1 || p.N > 64) return cudaErrorInvalidValue;
  const dim3 grid(p.m_tiles * p.splits);
  if (p.N <= 32) {
    if (!splitk_fits<32, kNarrowStages>(p.splits)) return cudaErrorInvalidValue;
    return launch_pdl(gemm_splitk_cluster_kernel<EPI, kNarrowStages, 32>, grid, dim3(192), NarrowSmem::kBytes, s,
                      p.splits, a, b, p);
  }
  if constexpr (EPI == kSplitKQkv) {
    if (!splitk_fits<64, kSkinnyStages>(p.splits)) return cudaErrorInvalidValue;
    return launch_pdl(gemm_splitk_cluster_kernel<EPI, kSkinnyStages, 64>, grid, dim3(192), SkinnySmem::kBytes, s,
                      p.splits, a, b, p);
  } else {
    if (!splitk_fits<64, kDeepStages>(p.splits)) return cudaErrorInvalidValue;
    return launch_pdl(gemm_splitk_cluster_kernel<EPI, kDeepStages, 64>, grid, dim3(192), DeepSmem::kBytes, s,
                      p.splits, a, b, p);
  }
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
