// decode_attn.cuh — attention of a few query positions per sequence against the KV cache:
// steps 6-13 of "Llama 3.1 8B · Grouped-query attention", memory-bound.  Decode (one new
// position per sequence, T = 1) and short prefills (T <= 16 new positions, each masked
// causally: the first tokens of a prompt, or a short chunk continuing a cache).
//
// The 4 query heads of kv group g = h/4 share every key and value of that group
// (K_G[h] = K_r[h/4], V_G[h] = V[h/4]), so one CTA serves (sequence b, group g, group of
// kPos positions, key split) and streams each K/V byte of its split once for all 4 heads and
// kPos positions.  The number of kv groups (8 for the whole block, fewer for a head shard)
// comes from the parameters.
//
//   warps 0..3  consumers: each takes 16 keys of every 64-key tile; S = q K^T and
//               O += P V with mma.sync m16n8k16, the (position, head) pairs being rows
//               4 x position + head of the 16-row A operand (rows 0..3 for decode); online
//               softmax in fp32 with quad-shuffle row max/sum
//   warp 4      producer: 64-key K and V tiles by TMA (128-byte swizzle), 3 stages
//
// Each CTA writes an unnormalised partial (O, running max m, running sum l) per row; the
// last split of each (b, g, position group) to finish merges the splits (log-sum-exp) and
// writes H bf16 [B, T, 512 n_kv] (or, without arrival counters, decode_combine_kernel does
// the merge).  With a single split the CTA writes H directly.
#pragma once

#include "params.h"
#include "ptx.cuh"

namespace gqa {

template <int kRows>
struct DecodeSmemT {
  static constexpr int kHalf = kDecTileKeys * 64 * 2;  // 64 keys x 64 d bf16 = 8 KB
  static constexpr int kTile = 2 * kHalf;              // 64 keys x 128 d
  static constexpr int kStage = 2 * kTile;             // K + V
  static constexpr int kRed = kDecStages * kStage;     // cross-warp reduction scratch
  static constexpr int kRedBytes = 4 * kRows * 128 * 4 + 4 * kRows * 2 * 4;
  static constexpr int kBar = kRed + kRedBytes;
  static constexpr int kBytes = kBar + 128 + 1024;
};
using DecodeSmem = DecodeSmemT<4>;  // one position per CTA: the rows are the group's 4 heads

// Byte offset of the 16-byte chunk `cd` (0..15, 8 d each) of key row `key` in a
// 64-key x 128-d tile stored as two 128-byte-swizzled 64-d halves.
__device__ __forceinline__ uint32_t dec_chunk_off(int key, int cd) {
  return (cd >> 3) * DecodeSmem::kHalf + key * 128 + (((cd & 7) ^ (key & 7)) << 4);
}

// Merge the key splits of (b, g, position group pg): for row = 4 x position + head,
// H[b, t, h] = sum_s e^{m_s - M} O_s / sum_s e^{m_s - M} l_s.  128 threads: thread ->
// (rows tid / 32, + 4, ...; 4 consecutive d).  Partials are read from L2; rows of positions
// past T are not written.
template <int kPos>
__device__ __forceinline__ void decode_merge_splits(const DecodeParams& p, int b, int g, int pg, int tid) {
  constexpr int kRows = 4 * kPos;
  const int d0 = (tid & 31) * 4;
  const size_t unit0 = ((static_cast<size_t>(b) * p.n_kv + g) * p.n_pg + pg) * p.n_splits;
#pragma unroll
  for (int row = tid >> 5; row < kRows; row += 4) {
    const int t = pg * kPos + (row >> 2);
    if (t >= p.T) continue;
    float M = -INFINITY;
    for (int s = 0; s < p.n_splits; ++s) M = fmaxf(M, __ldcg(p.part_ml + ((unit0 + s) * kRows + row) * 2));
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < p.n_splits; ++s) {
      const size_t u = (unit0 + s) * kRows + row;
      const float f = fast_exp2(__ldcg(p.part_ml + u * 2) - Mu);
      Ls += f * __ldcg(p.part_ml + u * 2 + 1);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + u * 128 + d0));
      acc[0] += f * v.x;
      acc[1] += f * v.y;
      acc[2] += f * v.z;
      acc[3] += f * v.w;
    }
    const float inv = 1.f / Ls;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.H) + (static_cast<size_t>(b) * p.T + t) * (p.n_kv * 512) +
                         (g * 4 + (row & 3)) * 128 + d0;
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  }
}

// grid (n_splits, n_kv, B n_pg), 160 threads; kPos = 1 (decode) or 4 (short prefills).
template <int kPos>
__global__ void __launch_bounds__(160)
    decode_attn_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const DecodeParams p) {
  static_assert(kPos == 1 || kPos == 4, "one position (4 rows) or four (16 rows) per CTA");
  constexpr int kRows = 4 * kPos;
  constexpr bool kTwoRows = kPos > 1;  // each thread holds two live rows (r0 and r0 + 8)
  using L = DecodeSmemT<kRows>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* empty_bar = full_bar + kDecStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty_bar + kDecStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = static_cast<int>(blockIdx.z) / p.n_pg;
  const int pg = static_cast<int>(blockIdx.z) - b * p.n_pg;
  const int t0 = pg * kPos;  // first position of this CTA's group
  // keys this group may see: through q_start + (its last position) when causal
  const int kv_hi = p.causal ? min(p.kv_len, p.q_start + min(p.T, t0 + kPos)) : p.kv_len;
  const int n_tiles_total = (kv_hi + kDecTileKeys - 1) / kDecTileKeys;
  const int t_begin = split * p.tiles_per_split;
  const int my_tiles = max(0, min(n_tiles_total, t_begin + p.tiles_per_split) - t_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();
  // q and the new cache entries come from the projection kernel; partials and counters
  // may still be in use by an earlier kernel until it has finished
  griddep_wait();

  if (warp == 4) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int issued = 0;
      // test hook: CTA (0, 0, 0) issues no loads, so its consumers wait out and abort
      const bool no_loads = p.fault && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
      for (int i = 0; i < (no_loads ? 0 : my_tiles); ++i) {
        const int s = i % kDecStages;
        const uint32_t ph = (i / kDecStages) & 1;
        if (!mbar_wait(&empty_bar[s], ph ^ 1u, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&full_bar[s], L::kStage);
        uint8_t* st = smem + s * L::kStage;
        const int key0 = (t_begin + i) * kDecTileKeys;
        tma_load_4d(st, &tmK, &full_bar[s], 0, g, key0, b);
        tma_load_4d(st + L::kHalf, &tmK, &full_bar[s], 64, g, key0, b);
        tma_load_4d(st + L::kTile, &tmV, &full_bar[s], 0, g, key0, b);
        tma_load_4d(st + L::kTile + L::kHalf, &tmV, &full_bar[s], 64, g, key0, b);
        ++issued;
      }
      if (*abort_flag) {
        for (int i = (issued > kDecStages ? issued - kDecStages : 0); i < issued; ++i)
          mbar_wait_drain(&full_bar[i % kDecStages], (i / kDecStages) & 1);
      }
    }
  } else {
    // ------------------------------------------------------------------ consumers
    // A operand (queries): this thread's rows are r0 = lane / 4 (fragment registers 0, 2)
    // and r0 + 8 (registers 1, 3); rows past 4 kPos and rows of positions past T are zero
    // and see no key.
    const int r0 = lane >> 2;  // 0..7
    const int qc = (lane & 3) * 2;
    int row_lim[2];  // last key each of the thread's two rows may see (-1: none)
    uint32_t qa[8][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = r0 + 8 * h;
      const int t = t0 + (row >> 2);
      const bool live = row < kRows && t < p.T;
      row_lim[h] = !live ? -1 : (p.causal ? min(p.kv_len - 1, p.q_start + t) : p.kv_len - 1);
      const uint32_t* qp = reinterpret_cast<const uint32_t*>(
          static_cast<const __nv_bfloat16*>(p.q) + (static_cast<size_t>(b) * p.T + (live ? t : 0)) * (p.n_kv * 512) +
          (g * 4 + (row & 3)) * 128);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][h] = live ? __ldg(qp + (kk * 16 + qc) / 2) : 0u;          // k = qc, qc + 1
        qa[kk][2 + h] = live ? __ldg(qp + (kk * 16 + qc + 8) / 2) : 0u;  // k = qc + 8, qc + 9
      }
    }
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    const int kb = warp * 16;  // this warp's 16 keys inside each tile
    bool ok = true;
    for (int i = 0; i < my_tiles; ++i) {
      const int s = i % kDecStages;
      ok = __all_sync(0xffffffffu, mbar_wait(&full_bar[s], (i / kDecStages) & 1, abort_flag, p.status));
      if (!ok) break;
      const uint32_t k_addr = smem_u32(smem + s * L::kStage);
      const uint32_t v_addr = k_addr + L::kTile;

      // S[16 rows x 16 keys]: two n8 tiles (keys kb..kb+7, kb+8..kb+15); registers 0, 1 of
      // each hold row r0, registers 2, 3 row r0 + 8
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int mi = lane >> 3;  // matrix index supplied by this lane's address
        const int key = kb + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(k_addr + dec_chunk_off(key, 2 * kk + (mi & 1)), b0, b1, b2, b3);
          const uint32_t a1 = kTwoRows ? qa[kk][1] : 0u;
          const uint32_t a3 = kTwoRows ? qa[kk][3] : 0u;
          mma_bf16_16816(sc[0], qa[kk][0], a1, qa[kk][2], a3, b0, b1);
          mma_bf16_16816(sc[1], qa[kk][0], a1, qa[kk][2], a3, b2, b3);
        }
      }
      // mask keys past each row's last visible key (cache length; causal position)
      const int kg0 = (t_begin + i) * kDecTileKeys + kb + qc;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (kg0 + nt * 8 + e > row_lim[0]) sc[nt][e] = -INFINITY;
          if (kTwoRows && kg0 + nt * 8 + e > row_lim[1]) sc[nt][2 + e] = -INFINITY;
        }
      float alpha[2] = {1.f, 1.f};
      float pr[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int h = 0; h < (kTwoRows ? 2 : 1); ++h) {
        float mx = fmaxf(fmaxf(sc[0][2 * h], sc[0][2 * h + 1]), fmaxf(sc[1][2 * h], sc[1][2 * h + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[h], mx * p.scale_log2);
        const float mu = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[h] = fast_exp2(m_run[h] - mu);
        float ls = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            pr[nt][2 * h + e] = fast_exp2(fmaf(sc[nt][2 * h + e], p.scale_log2, -mu));
            ls += pr[nt][2 * h + e];
          }
        ls += __shfl_xor_sync(0xffffffffu, ls, 1);
        ls += __shfl_xor_sync(0xffffffffu, ls, 2);
        l_run[h] = l_run[h] * alpha[h] + ls;
        m_run[h] = m_new;
      }
#pragma unroll
      for (int i2 = 0; i2 < 16; ++i2) {
        o[i2][0] *= alpha[0];
        o[i2][1] *= alpha[0];
        if (kTwoRows) {
          o[i2][2] *= alpha[1];
          o[i2][3] *= alpha[1];
        }
      }
      // O[16 x 128] += P[16 x 16 keys] V[16 keys x 128]
      const uint32_t pa0 = pack_bf16x2(pr[0][0], pr[0][1]);
      const uint32_t pa2 = pack_bf16x2(pr[1][0], pr[1][1]);
      const uint32_t pa1 = kTwoRows ? pack_bf16x2(pr[0][2], pr[0][3]) : 0u;
      const uint32_t pa3 = kTwoRows ? pack_bf16x2(pr[1][2], pr[1][3]) : 0u;
      {
        const int mi = lane >> 3;
        const int key = kb + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {  // d blocks of 16
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(v_addr + dec_chunk_off(key, 2 * dp + (mi >> 1)), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
          mma_bf16_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
    }

    // ---------------------------------------------------------- cross-warp merge
    float* red_o = reinterpret_cast<float*>(smem + L::kRed);  // [4 warps][kRows][128]
    float* red_ml = red_o + 4 * kRows * 128;                   // [4 warps][kRows][2]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = r0 + 8 * h;
      if (row < kRows) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          red_o[(warp * kRows + row) * 128 + nt * 8 + qc] = o[nt][2 * h];
          red_o[(warp * kRows + row) * 128 + nt * 8 + qc + 1] = o[nt][2 * h + 1];
        }
        if ((lane & 3) == 0) {
          red_ml[(warp * kRows + row) * 2 + 0] = m_run[h];
          red_ml[(warp * kRows + row) * 2 + 1] = l_run[h];
        }
      }
    }
    // one decision for all 128 consumer threads (the merge below uses named barriers)
    if (bar1_and_128(ok && !*abort_flag)) {
      const int tid = threadIdx.x;
      const int d0 = (tid & 31) * 4;
      const size_t unit = ((static_cast<size_t>(b) * p.n_kv + g) * p.n_pg + pg) * p.n_splits + split;
      // a single split (short caches) normalises and writes H itself: no partials, no counter
      const bool direct = p.n_splits == 1 && p.counters;
#pragma unroll
      for (int row = tid >> 5; row < kRows; row += 4) {
        float mw[4], M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          mw[w] = red_ml[(w * kRows + row) * 2];
          M = fmaxf(M, mw[w]);
        }
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float Ls = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float f = fast_exp2(mw[w] - Mu);
          Ls += f * red_ml[(w * kRows + row) * 2 + 1];
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] += f * red_o[(w * kRows + row) * 128 + d0 + e];
        }
        if (direct) {
          const int t = t0 + (row >> 2);
          if (t < p.T) {
            const float inv = 1.f / Ls;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.H) +
                                 (static_cast<size_t>(b) * p.T + t) * (p.n_kv * 512) + (g * 4 + (row & 3)) * 128 + d0;
            uint2 w;
            w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2*>(dst) = w;
          }
          continue;
        }
        *reinterpret_cast<float4*>(p.part_o + (unit * kRows + row) * 128 + d0) =
            make_float4(acc[0], acc[1], acc[2], acc[3]);
        if ((tid & 31) == 0) {
          p.part_ml[(unit * kRows + row) * 2 + 0] = M;
          p.part_ml[(unit * kRows + row) * 2 + 1] = Ls;
        }
      }
      if (p.counters && !direct) {
        // the last split of (b, g, pg) to publish its partial merges all of them
        const int ci = (b * p.n_kv + g) * p.n_pg + pg;
        volatile int* last_flag = abort_flag + 1;
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (tid == 0) *last_flag = (atomicAdd(&p.counters[ci], 1) == p.n_splits - 1);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (*last_flag) {
          __threadfence();
          decode_merge_splits<kPos>(p, b, g, pg, tid);
          if (tid == 0) p.counters[ci] = 0;  // ready for the next call
        }
      }
    }
  }
}

// Separate merge kernel (used when the decode kernel runs without arrival counters; one
// position per sequence).  grid (n_kv, B), 128 threads, launched after decode_attn_kernel
// has completed.  If a split of this call gave up a wait (*p.status non-zero), some partials
// were never written, so every H entry of the call is written as NaN instead of a merge of
// stale partials, and the status bits are OR-ed into *p.status_sticky, where they stay until
// the caller reads them.
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
  const int st = *reinterpret_cast<volatile const int*>(p.status);
  if (st != 0) {
    const int hh = threadIdx.x >> 5;
    const int d0 = (threadIdx.x & 31) * 4;
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.H) + static_cast<size_t>(blockIdx.y) * (p.n_kv * 512) +
                         (blockIdx.x * 4 + hh) * 128 + d0;
    const uint32_t nan2 = 0x7FC07FC0u;  // two bf16 quiet NaNs
    *reinterpret_cast<uint2*>(dst) = make_uint2(nan2, nan2);
    if (p.status_sticky && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.status_sticky, st);
    return;
  }
  decode_merge_splits<1>(p, blockIdx.y, blockIdx.x, 0, threadIdx.x);
}

}  // namespace gqa
