// flash_prefill.cuh — causal grouped-query attention for a prefill (steps 6-13 of
// "Llama 3.1 8B · Grouped-query attention"): S = Q_r K_G^T, S / sqrt(128), + M, row
// softmax, H = A V_G, written merged as [B*T, 4096] bf16 (head h at columns 128h..).
//
// One CTA = one (sequence b, query head h, 128-query tile).  K_G[h] = K_r[h/4] and
// V_G[h] = V[h/4] are an index map: the CTA reads kv head g = h/4 of the cache directly.
//
//   warp 0      TMA producer: Q tile once, then 128-key K and V tiles (2 stages each)
//   warp 1      TMEM owner + UMMA issuer: S_j = Q K_j^T into one of two TMEM S buffers,
//               then O += P_{j-1} V_{j-1} (P from shared memory, V MN-major)
//   warps 2..5  softmax: one thread per query row; online softmax in fp32 in the log2
//               domain with the 1/sqrt(128) scale folded into the exponent; lazy O
//               rescaling (only when a row max grows by more than 2^8); P written bf16
//               into the swizzled shared-memory tile the next UMMA reads; final O / l.
//
// TMEM columns: S buffers at 0 and 128, O at 256 (512 allocated).
#pragma once

#include "params.h"
#include "ptx.cuh"

namespace gqa {

struct FlashSmem {
  static constexpr int kTile = 128 * 128 * 2;  // one 128x128 bf16 tile (two 64-col halves)
  static constexpr int kHalf = 128 * 64 * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;          // 2 stages
  static constexpr int kV = kK + 2 * kTile;      // 2 stages
  static constexpr int kP = kV + 2 * kTile;
  static constexpr int kBar = kP + kTile;
  static constexpr int kBytes = kBar + 256 + 1024;
};

__global__ void __launch_bounds__(192, 1)
    flash_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FlashParams p) {
  using L = FlashSmem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;   // [2]
  uint64_t* v_empty = bars + 7;  // [2]
  uint64_t* s_full = bars + 9;   // [2]
  uint64_t* p_full = bars + 11;
  uint64_t* o_done = bars + 12;
  uint64_t* drain = bars + 13;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int bh = blockIdx.x;
  const int b = bh / 32;
  const int h = bh % 32;
  const int g = h >> 2;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);  // heaviest tiles first
  const int q0 = qt * 128;
  const int kv_len = p.start_pos + p.T;
  const int kv_hi = p.causal ? min(kv_len, p.start_pos + q0 + 128) : kv_len;
  const int n_kv = (kv_hi + 127) / 128;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 14; ++i) mbar_init(&bars[i], i == 11 ? 128u : 1u);  // p_full: 128 rows
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const uint32_t tmem_O = tmem_base + 256;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, L::kTile);
      tma_load_3d(smem + L::kQ, &tmQ, q_full, h * 128, q0, b);
      tma_load_3d(smem + L::kQ + L::kHalf, &tmQ, q_full, h * 128 + 64, q0, b);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1u, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&k_full[st], L::kTile);
        uint8_t* kd = smem + L::kK + st * L::kTile;
        tma_load_4d(kd, &tmK, &k_full[st], 0, g, j * 128, b);
        tma_load_4d(kd + L::kHalf, &tmK, &k_full[st], 64, g, j * 128, b);
        if (!mbar_wait(&v_empty[st], ph ^ 1u, abort_flag, p.status)) { ++issued; break; }
        mbar_arrive_expect_tx(&v_full[st], L::kTile);
        uint8_t* vd = smem + L::kV + st * L::kTile;
        tma_load_4d(vd, &tmV, &v_full[st], 0, g, j * 128, b);
        tma_load_4d(vd + L::kHalf, &tmV, &v_full[st], 64, g, j * 128, b);
        ++issued;
      }
      if (*abort_flag) {
        mbar_wait_drain(q_full, 0);
        for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) {
          mbar_wait_drain(&k_full[j & 1], (j >> 1) & 1);
          mbar_wait_drain(&v_full[j & 1], (j >> 1) & 1);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- UMMA issuer
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);   // Q, K both K-major
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, 0, 1);  // P K-major, V MN-major
      const uint32_t q_addr = smem_u32(smem + L::kQ);
      const uint32_t k_addr = smem_u32(smem + L::kK);
      const uint32_t v_addr = smem_u32(smem + L::kV);
      const uint32_t p_addr = smem_u32(smem + L::kP);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status);
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {
          const int st = j & 1;
          if (!mbar_wait(&k_full[st], (j >> 1) & 1, abort_flag, p.status)) break;
          tc_fence_after();
          const uint32_t d_s = tmem_base + st * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * L::kHalf + (kk & 3) * 32;
            umma_ss(d_s, sdesc_sw128(q_addr + off, 0, 1024),
                    sdesc_sw128(k_addr + st * L::kTile + off, 0, 1024), idesc_s, kk != 0);
          }
          umma_commit(&k_empty[st]);
          umma_commit(&s_full[st]);
        }
        if (j >= 1) {
          const int jp = j - 1;
          const int st = jp & 1;
          if (!mbar_wait(p_full, jp & 1, abort_flag, p.status)) break;
          if (!mbar_wait(&v_full[st], (jp >> 1) & 1, abort_flag, p.status)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // P: K-major, keys 16kk..16kk+15 -> half kk/4, +32 B per step inside the atom.
            const uint32_t poff = (kk >> 2) * L::kHalf + (kk & 3) * 32;
            // V: MN-major (d contiguous); 16 keys = two 8-row groups = 2048 B per step;
            // d 64..127 lives in the second half (LBO), 8-key groups 1024 B apart (SBO).
            const uint32_t voff = kk * 2048;
            umma_ss(tmem_O, sdesc_sw128(p_addr + poff, 0, 1024),
                    sdesc_sw128(v_addr + st * L::kTile + voff, L::kHalf, 1024), idesc_pv,
                    (jp | kk) != 0);
          }
          umma_commit(&v_empty[st]);
          umma_commit(o_done);
        }
      }
      if (*abort_flag) {  // let issued UMMAs finish before TMEM is released
        umma_commit(drain);
        mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int qpos = p.start_pos + q0 + r;
    uint8_t* Ps = smem + L::kP;
    float m_used = -INFINITY;
    float l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      ok = mbar_wait(&s_full[st], (j >> 1) & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem_base + lane_off + st * 128 + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[i]);
      }
      const int key0 = j * 128;
      const bool needs_mask = (key0 + 127 >= kv_len) || (p.causal && key0 + 127 > p.start_pos + q0);
      if (needs_mask) {
        const int lim = p.causal ? min(kv_len - 1, qpos) : kv_len - 1;
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (key0 + i > lim) s[i] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) mx = fmaxf(mx, s[i]);
      const float m_tile = mx * p.scale_log2;
      // PV_{j-1} must be complete before O is rescaled and before P is overwritten.
      if (j >= 1) {
        ok = mbar_wait(o_done, (j - 1) & 1, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
      }
      if (j == 0) {
        m_used = m_tile;
      } else {
        // Per-row decision (rows never influence each other's bits); the TMEM round trip is
        // warp-collective, rows that keep their max scale by exactly 1.
        const bool grow = m_tile > m_used + 8.0f;
        if (__any_sync(0xffffffffu, grow)) {
          float alpha = 1.f;
          if (grow) {
            alpha = fast_exp2(m_used - m_tile);
            l_sum *= alpha;
            m_used = m_tile;
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(tmem_O + lane_off + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(tmem_O + lane_off + c * 32, v);
          }
          tmem_st_wait();
        }
      }
      const float mu = (m_used == -INFINITY) ? 0.f : m_used;
      // P = exp2(s * scale_log2 - m_used), written bf16 into the swizzled P tile.
      float lsum = 0.f;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint8_t* prow = Ps + hf * L::kHalf + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = hf * 64 + c * 8 + 2 * e;
            const float p0 = fast_exp2(fmaf(s[i], p.scale_log2, -mu));
            const float p1 = fast_exp2(fmaf(s[i + 1], p.scale_log2, -mu));
            lsum += p0 + p1;
            w[e] = pack_bf16x2(p0, p1);
          }
          *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      l_sum += lsum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok) {
      ok = mbar_wait(o_done, (n_kv - 1) & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_sum;
      const bool valid = (q0 + r) < p.T;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.H) + (static_cast<size_t>(b) * p.T + q0 + r) * 4096 + h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem_O + lane_off + c * 32, v);
        tmem_ld_wait();
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l);
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace gqa
