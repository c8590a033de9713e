// gemm_launch.cu — instantiations of the tcgen05 GEMM and the split-K reductions of the
// skinny (few-token) projections.
#include "gemm_tc.cuh"
#include "launch.h"

namespace gqa {

using PairSmem = GemmPairSmem<6>;
using SkinnySmem = GemmSmem<64, 4>;

size_t gemm_wide_smem() { return PairSmem::kBytes; }
size_t gemm_skinny_smem() { return SkinnySmem::kBytes; }

cudaError_t configure_gemm_kernels() {
  cudaError_t e;
  e = cudaFuncSetAttribute(gemm_tc_pair_kernel<6, kQkvRope>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairSmem::kBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_tc_pair_kernel<6, kStoreF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairSmem::kBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_tc_kernel<64, 4, kPartialT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, SkinnySmem::kBytes);
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

cudaError_t launch_gemm_qkv_rope(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                 int grid, cudaStream_t s) {
  gemm_tc_pair_kernel<6, kQkvRope><<<grid, 192, PairSmem::kBytes, s>>>(a, b, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_store_f32(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                  int grid, cudaStream_t s) {
  gemm_tc_pair_kernel<6, kStoreF32><<<grid, 192, PairSmem::kBytes, s>>>(a, b, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_partial(const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                                int grid, cudaStream_t s) {
  gemm_tc_kernel<64, 4, kPartialT><<<grid, 192, SkinnySmem::kBytes, s>>>(a, b, p);
  return cudaGetLastError();
}

// Sum the split-K partials of the skinny Q/K/V projection, rotate Q and K pairs by R
// (steps 4-5) and store Q_r / the cache entries, exactly as the wide GEMM epilogue does.
// One thread per (token, 4 consecutive features).
__global__ void __launch_bounds__(256) qkv_finalize_kernel(const QkvFinalizeParams p) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.n_tok * 1536) return;
  const int n = idx / 1536;
  const int f = (idx - n * 1536) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* src = p.part + static_cast<size_t>(n) * 6144 + f;
  for (int s = 0; s < p.splits; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(src + static_cast<size_t>(s) * p.slab);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const int b = n / p.T;
  const int t = n - b * p.T;
  float o0 = acc.x, o1 = acc.y, o2 = acc.z, o3 = acc.w;
  if (f < 5120) {
    const int j = (f & 127) >> 1;
    const float4 cs = __ldg(reinterpret_cast<const float4*>(p.R + (static_cast<size_t>(t) * 64 + j) * 2));
    o0 = cs.x * acc.x - cs.y * acc.y;
    o1 = cs.y * acc.x + cs.x * acc.y;
    o2 = cs.z * acc.z - cs.w * acc.w;
    o3 = cs.w * acc.z + cs.z * acc.w;
  }
  __nv_bfloat16* dst;
  if (f < 4096) {
    dst = static_cast<__nv_bfloat16*>(p.q) + static_cast<size_t>(n) * 4096 + f;
  } else {
    const bool is_v = f >= 5120;
    const size_t row = static_cast<size_t>(b) * p.S_max + p.start_pos + t;
    dst = static_cast<__nv_bfloat16*>(is_v ? p.cache_v : p.cache_k) + row * 1024 + (f - (is_v ? 5120 : 4096));
  }
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
}

// Delta[n, f] = sum over splits of the skinny W_O partials.
__global__ void __launch_bounds__(256) out_finalize_kernel(const OutFinalizeParams p) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= p.n_tok * 1024) return;
  const int n = idx / 1024;
  const int f = (idx - n * 1024) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* src = p.part + static_cast<size_t>(n) * 4096 + f;
  for (int s = 0; s < p.splits; ++s) {
    const float4 v = *reinterpret_cast<const float4*>(src + static_cast<size_t>(s) * p.slab);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  *reinterpret_cast<float4*>(p.delta + static_cast<size_t>(n) * 4096 + f) = acc;
}

cudaError_t launch_qkv_finalize(const QkvFinalizeParams& p, cudaStream_t s) {
  const int total = p.n_tok * 1536;
  qkv_finalize_kernel<<<(total + 255) / 256, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_out_finalize(const OutFinalizeParams& p, cudaStream_t s) {
  const int total = p.n_tok * 1024;
  out_finalize_kernel<<<(total + 255) / 256, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gqa
