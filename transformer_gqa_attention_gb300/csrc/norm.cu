// norm.cu — the attention_norm (RMSNorm) prologue of the block's residual form.
//
// The transformer block feeds the attention block attention_norm(x) and adds the update
// back (page "Llama 3.1 8B · Merge and project", code excerpt model.py 236-248); RMSNorm is
// read as y = x / sqrt(mean_j x_j^2 + eps) * w with eps = norm_eps = 1e-5.  Since
//     Q = y W_Q^T = diag(r) (x diag(w)) W_Q^T = diag(r) x (W_Q diag(w))^T,  r = 1 / rms(x),
// the library folds w into a second copy of the projection weights once (attn_set_norm) and
// the Q/K/V kernels multiply each token row's accumulators by r in their epilogue; only r
// needs a pass over x.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace gqa {

// r[row] = 1 / sqrt(mean_j x[row, j]^2 + eps), x [rows, 4096] bf16, fp32 accumulation.
// One 128-thread CTA per row: every thread issues its four 16-byte loads at once (one memory
// round trip per row), then a fixed-order reduction (lanes, then the four warps).
__global__ void __launch_bounds__(128) rms_rstd_kernel(const __nv_bfloat16* __restrict__ x, int rows, float eps,
                                                       float* __restrict__ r) {
  __shared__ float part[4];
  griddep_wait();  // x may come from the previous kernel on the stream
  griddep_launch_dependents();
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * 4096);
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __ldg(src + threadIdx.x + 128 * i);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = bf16lo_to_f32(w[k]), b = bf16hi_to_f32(w[k]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) part[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    const float t = (part[0] + part[1]) + (part[2] + part[3]);
    r[row] = 1.f / sqrtf(t * (1.f / 4096.f) + eps);
  }
}

// Folded weight copy: dst = src * w along the input (k) axis, both k-block-major
// [kb][row][64] bf16 with `rows` rows; w [4096] bf16.
__global__ void fold_norm_weight_kernel(const __nv_bfloat16* __restrict__ src, const __nv_bfloat16* __restrict__ w,
                                        int rows, __nv_bfloat16* __restrict__ dst) {
  const size_t n = static_cast<size_t>(rows) * 4096;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t kb = i / (static_cast<size_t>(rows) * 64);
    const int k = static_cast<int>(kb * 64 + (i & 63));
    dst[i] = __float2bfloat16_rn(__bfloat162float(src[i]) * __bfloat162float(w[k]));
  }
}

cudaError_t launch_rms_rstd(const void* x, int rows, float eps, float* r, cudaStream_t s) {
  return launch_pdl(rms_rstd_kernel, dim3(rows), dim3(128), 0, s, 0,
                    static_cast<const __nv_bfloat16*>(x), rows, eps, r);
}

cudaError_t launch_fold_norm_weight(const void* src, const void* w, int rows, void* dst, cudaStream_t s) {
  fold_norm_weight_kernel<<<1024, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src),
                                               static_cast<const __nv_bfloat16*>(w), rows,
                                               static_cast<__nv_bfloat16*>(dst));
  return cudaGetLastError();
}

}  // namespace gqa
