// launch.h — internal host-side launchers of the block's kernels (C++, not part of the
// public C ABI).  Each returns the cudaError_t of its launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "params.h"

namespace gqa {

// Dynamic shared memory each kernel needs (bytes).
size_t gemm_wide_smem();    // 128x256 tiles (prefill)
size_t gemm_skinny_smem();  // 128x64 tiles (few tokens, split-K)
size_t flash_smem();
size_t decode_smem();

// One-time per-process opt-in to large dynamic shared memory on the current device.
cudaError_t configure_kernels();

// Number of 2-CTA clusters of the pair GEMM that can be resident at once (0 on error).
int gemm_pair_max_clusters();

cudaError_t launch_gemm_qkv_rope(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                 int grid, cudaStream_t s);
cudaError_t launch_gemm_store_f32(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                  int grid, cudaStream_t s);
cudaError_t launch_gemm_partial(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                int grid, cudaStream_t s);

// Reduction of the skinny projection partials.
struct QkvFinalizeParams {
  const float* part;  // [splits][tokens_pad][6144]
  long long slab;
  int splits, n_tok, T, S_max, start_pos;
  const float* R;     // [T,64,2]
  void* q;            // [n_tok, 4096] bf16
  void* cache_k;      // [B,S_max,8,128] bf16
  void* cache_v;
};
struct OutFinalizeParams {
  const float* part;  // [splits][tokens_pad][4096]
  long long slab;
  int splits, n_tok;
  float* delta;       // [n_tok, 4096]
};
cudaError_t launch_qkv_finalize(const QkvFinalizeParams& p, cudaStream_t s);
cudaError_t launch_out_finalize(const OutFinalizeParams& p, cudaStream_t s);

cudaError_t launch_flash_prefill(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const FlashParams& p, dim3 grid, cudaStream_t s);
cudaError_t launch_decode_attn(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                               dim3 grid, cudaStream_t s);
cudaError_t launch_decode_combine(const DecodeParams& p, int B, cudaStream_t s);

}  // namespace gqa
