// attn_launch.cu — instantiations of the prefill and decode attention kernels.
#include "decode_attn.cuh"
#include "flash_prefill.cuh"
#include "launch.h"

namespace gqa {

cudaError_t configure_gemm_kernels();


cudaError_t configure_kernels() {
  cudaError_t e = configure_gemm_kernels();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flash_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FlashSmem::kBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_attn_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DecodeSmemT<4>::kBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_attn_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DecodeSmemT<16>::kBytes);
}

cudaError_t launch_flash_prefill(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& h, const FlashParams& p, dim3 grid, cudaStream_t s) {
  return launch_pdl(flash_prefill_kernel, grid, dim3(384), FlashSmem::kBytes, s, 0, q, k, v, h, p);
}

cudaError_t launch_decode_attn(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                               dim3 grid, cudaStream_t s) {
  return launch_pdl(decode_attn_kernel<1>, grid, dim3(160), DecodeSmemT<4>::kBytes, s, 0, k, v, p);
}

cudaError_t launch_short_attn(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p, dim3 grid,
                              cudaStream_t s) {
  return launch_pdl(decode_attn_kernel<4>, grid, dim3(160), DecodeSmemT<16>::kBytes, s, 0, k, v, p);
}

// Both exponentials of the softmax on n inputs (the FMA-pipe cubic and the multi-function
// unit's ex2.approx.ftz), for the test that compares them.
__global__ void exp2_compare_kernel(const float* __restrict__ a, float* __restrict__ out_fma,
                                    float* __restrict__ out_mufu, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float2 v = make_float2(a[i], i + 1 < n ? a[i + 1] : 0.f);
  const float2 r = exp2_fma2(v);
  out_fma[i] = r.x;
  out_mufu[i] = fast_exp2(v.x);
  if (i + 1 < n) {
    out_fma[i + 1] = r.y;
    out_mufu[i + 1] = fast_exp2(v.y);
  }
}

cudaError_t launch_exp2_compare(const float* a, float* out_fma, float* out_mufu, int n, cudaStream_t s) {
  exp2_compare_kernel<<<(n / 2 + 256) / 256, 256, 0, s>>>(a, out_fma, out_mufu, n);
  return cudaGetLastError();
}

cudaError_t launch_decode_combine(const DecodeParams& p, int B, cudaStream_t s) {
  decode_combine_kernel<<<dim3(8, B), 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gqa
