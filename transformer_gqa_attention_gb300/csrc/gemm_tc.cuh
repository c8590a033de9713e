// gemm_tc.cuh — warp-specialised tcgen05 GEMM, D[M,N] = A[M,K] * B[N,K]^T, both operands
// K-major bf16 (the [out, in] weight storage of the quoted F.linear layers), fp32
// accumulation in TMEM.
//
//   warp 0      TMA producer: 128x64 A box + BNx64 B box per stage, 128-byte swizzle
//   warp 1      TMEM owner + single-thread UMMA issuer (128 x BN x 16 per instruction)
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows, fused output transform
//
// Epilogues (one output tile per CTA):
//   kQkvRope  — the fused Q/K/V projection (steps 1-5 of "Llama 3.1 8B · Grouped-query
//               attention"): columns 0..4095 are Q, 4096..5119 K, 5120..6143 V of the
//               packed [6144,4096] weight.  Q and K pairs (2j, 2j+1) are rotated by
//               R[t, j] in fp32, then Q is stored to the Q_r buffer [B*T,4096] and K_r, V
//               straight into the caches [B,S_max,8,128] at position start_pos + t.
//   kStoreF32 — Delta = H W_O^T (step 14) stored fp32 row-major.
//   kPartialT — skinny (swap-AB) split-K: A holds weight rows, B the few token rows;
//               each split stores its fp32 partial slab [token][feature] for a
//               separate reduction kernel.
#pragma once

#include "params.h"
#include "ptx.cuh"

namespace gqa {

template <int BN, int STAGES>
struct GemmSmem {
  static constexpr int kABytes = 128 * 64 * 2;
  static constexpr int kBBytes = BN * 64 * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kBytes = kBarOffset + 256 + 1024;  // + barriers + alignment slack
};

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  using L = GemmSmem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::kABytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* acc_bar = empty_bar + STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int split = blockIdx.x % p.splits;
  const int tile = blockIdx.x / p.splits;
  const int n_tile = tile % p.n_tiles;
  const int m_tile = tile / p.n_tiles;
  const int m0 = m_tile * 128;
  const int n0 = n_tile * BN;
  const int kb0 = split * p.kb_per_split;
  const int nkb = (split == p.splits - 1) ? (p.num_kb - kb0) : p.kb_per_split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(acc_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&empty_bar[s], ph ^ 1u, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&full_bar[s], L::kStageBytes);
        const int kc = (kb0 + i) * 64;
        tma_load_2d(sA + s * L::kABytes, &tmA, &full_bar[s], kc, m0);
        tma_load_2d(sB + s * L::kBBytes, &tmB, &full_bar[s], kc, n0);
        ++issued;
      }
      if (*abort_flag) {  // let copies still in flight land before the CTA leaves
        for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
          mbar_wait_drain(&full_bar[i % STAGES], (i / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ UMMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, BN, 0, 0);
      const uint32_t a_base = smem_u32(sA);
      const uint32_t b_base = smem_u32(sB);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&full_bar[s], ph, abort_flag, p.status)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t da = sdesc_sw128(a_base + s * L::kABytes + k * 32, 0, 1024);
          const uint64_t db = sdesc_sw128(b_base + s * L::kBBytes + k * 32, 0, 1024);
          umma_ss(tmem_base, da, db, idesc, (i | k) != 0);
        }
        umma_commit(&empty_bar[s]);
      }
      umma_commit(acc_bar);
      if (*abort_flag) mbar_wait_drain(acc_bar, 0);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_bar, 0, abort_flag, p.status));
    tc_fence_after();
    if (ok) {
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
      const int m = m0 + row;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(t_row + c * 32, v);
        tmem_ld_wait();
        const int col0 = n0 + c * 32;
        if constexpr (EPI == kQkvRope) {
          if (m < p.M) {
            const int b = m / p.T;
            const int t = m - b * p.T;
            const bool is_v = col0 >= 5120;
            uint32_t w[16];
            if (is_v) {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                w[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            } else {
              // pairs j0 .. j0+15 of this head slice
              const int j0 = (col0 & 127) >> 1;
              const float4* rp = reinterpret_cast<const float4*>(p.R + (static_cast<size_t>(t) * 64 + j0) * 2);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 cs = __ldg(rp + i);  // (cos, sin) of pairs 2i and 2i+1
                const float e0 = __uint_as_float(v[4 * i + 0]), o0 = __uint_as_float(v[4 * i + 1]);
                const float e1 = __uint_as_float(v[4 * i + 2]), o1 = __uint_as_float(v[4 * i + 3]);
                w[2 * i + 0] = pack_bf16x2(cs.x * e0 - cs.y * o0, cs.y * e0 + cs.x * o0);
                w[2 * i + 1] = pack_bf16x2(cs.z * e1 - cs.w * o1, cs.w * e1 + cs.z * o1);
              }
            }
            __nv_bfloat16* dst;
            if (col0 < 4096) {
              dst = static_cast<__nv_bfloat16*>(p.out0) + static_cast<size_t>(m) * 4096 + col0;
            } else {
              const size_t cache_row = static_cast<size_t>(b) * p.S_max + p.start_pos + t;
              dst = static_cast<__nv_bfloat16*>(is_v ? p.out2 : p.out1) + cache_row * 1024 +
                    (col0 - (is_v ? 5120 : 4096));
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        } else if constexpr (EPI == kStoreF32) {
          if (m < p.M) {
            float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(p.out0) + static_cast<size_t>(m) * p.ldo + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                  __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          }
        } else {  // kPartialT: slab [split][token][feature]; a warp stores 32 consecutive features
          if (m < p.M) {
            float* base = static_cast<float*>(p.out0) + static_cast<size_t>(split) * p.slab +
                          static_cast<size_t>(col0) * p.ldo + m;
#pragma unroll
            for (int i = 0; i < 32; ++i) base[static_cast<size_t>(i) * p.ldo] = __uint_as_float(v[i]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, BN);
  }
}

}  // namespace gqa
