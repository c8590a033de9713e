// attn_launch.cu — instantiations of the prefill and decode attention kernels.
#include "decode_attn.cuh"
#include "flash_prefill.cuh"
#include "launch.h"

namespace gqa {

cudaError_t configure_gemm_kernels();

size_t flash_smem() { return FlashSmem::kBytes; }
size_t decode_smem() { return DecodeSmem::kBytes; }

cudaError_t configure_kernels() {
  cudaError_t e = configure_gemm_kernels();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flash_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FlashSmem::kBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DecodeSmem::kBytes);
}

cudaError_t launch_flash_prefill(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& h, const FlashParams& p, dim3 grid, cudaStream_t s) {
  return launch_pdl(flash_prefill_kernel, grid, dim3(384), FlashSmem::kBytes, s, 0, q, k, v, h, p);
}

cudaError_t launch_decode_attn(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                               dim3 grid, cudaStream_t s) {
  return launch_pdl(decode_attn_kernel, grid, dim3(160), DecodeSmem::kBytes, s, 0, k, v, p);
}

cudaError_t launch_decode_combine(const DecodeParams& p, int B, cudaStream_t s) {
  decode_combine_kernel<<<dim3(8, B), 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gqa
