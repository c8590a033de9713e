// launch.h — internal host-side launchers of the block's kernels (C++, not part of the
// public C ABI).  Each returns the cudaError_t of its launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "params.h"

namespace gqa {

// Launch `kernel` with programmatic dependent launch (the kernel calls griddep_wait before
// touching anything an earlier kernel may write) and, if cluster_x > 0, a runtime cluster
// shape of cluster_x x 1 x 1.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster_x,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Records a failing CUDA call's error code for attn_last_cuda_error (thread-local; every
// translation unit of the library reports through it).
void set_last_cuda_error(cudaError_t e);

// One-time per-process opt-in to large dynamic shared memory on the current device.
cudaError_t configure_kernels();

// Number of 2-CTA clusters of the pair GEMM that can be resident at once (0 on error).
int gemm_pair_max_clusters();

// b: weight map with 128-row boxes (whole tiles); bt: the same weight, p.tail_w / 2-row boxes
// (pieces of a partial last round)
cudaError_t launch_gemm_qkv_rope(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bt,
                                 const GemmParams& p, int grid, cudaStream_t s);
cudaError_t launch_gemm_store_f32(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bt,
                                  const GemmParams& p, int grid, cudaStream_t s);
// Few-token split-K projections with the reduction fused (last split of each tile).  The
// activation tensor map's box holds splitk_token_tile(n_tok) rows.
int splitk_token_tile(int n_tok);
// One cluster of p.splits CTAs (2..8) per 128-feature tile, at most 64 tokens.
cudaError_t launch_gemm_splitk_qkv(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                   cudaStream_t s);
cudaError_t launch_gemm_splitk_out(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                   cudaStream_t s);

cudaError_t launch_flash_prefill(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& h, const FlashParams& p, dim3 grid, cudaStream_t s);
cudaError_t launch_decode_attn(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                               dim3 grid, cudaStream_t s);
// Short prefills (T <= 16): the decode attention kernel with 4 positions per CTA.
cudaError_t launch_short_attn(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p, dim3 grid,
                              cudaStream_t s);
cudaError_t launch_decode_combine(const DecodeParams& p, int B, cudaStream_t s);
cudaError_t launch_exp2_compare(const float* a, float* out_fma, float* out_mufu, int n, cudaStream_t s);
cudaError_t launch_rms_rstd(const void* x, int rows, float eps, float* r, cudaStream_t s);
cudaError_t launch_fold_norm_weight(const void* src, const void* w, int rows, void* dst, cudaStream_t s);

}  // namespace gqa
