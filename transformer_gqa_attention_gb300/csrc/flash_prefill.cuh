// flash_prefill.cuh — causal grouped-query attention for a prefill (steps 6-13 of
// "Llama 3.1 8B · Grouped-query attention"): S = Q_r K_G^T, S / sqrt(128), + M, row
// softmax, H = A V_G, written merged as [B*T, 4096] bf16 (head h at columns 128h..).
// A context over G of the 8 kv groups has 4 G query heads: Q_r and H rows are 512 G wide
// and the cache holds G kv heads per position; the kernel takes G from its parameters.
//
// One CTA = one sequence b, one 128-query tile and TWO query heads h0 = 2p, h1 = 2p+1 of
// the same kv group g = h0/4 (K_G[h] = K_r[h/4], V_G[h] = V[h/4] is an index map: both
// heads read the same K/V tiles of kv head g from the cache, staged once in shared memory).
// Both heads have the same causal extent, so they advance through the key tiles together.
//
//   warp 0      TMA producer: the two Q tiles once, then 128-key K and V tiles (2 stages)
//   warp 1      TMEM owner + UMMA issuer.  Per key tile j, for head slot i = 0, 1:
//                 S_i = Q_i K_j^T (both operands K-major from shared memory) into TMEM,
//                 O_i += P_i V_j with P_i read from TMEM (it overwrites S_i) and V an
//                 MN-major shared-memory operand, issued in two halves (keys 0..63 as soon
//                 as the softmax has released them, then 64..127).  Issue order S_0(j+1)
//                 before PV_1(j) keeps the tensor core busy while the other head's softmax
//                 runs.
//   warps 4..7  softmax of head slot 0, warps 8..11 of head slot 1: one thread per query
//               row (no shuffles); online softmax in fp32 in the log2 domain with the
//               1/sqrt(128) scale folded into the exponent; P = exp2(...) rounded to bf16
//               and stored back into TMEM; lazy per-row rescale of O only when the row max
//               grows by more than 2^8; final O / l stored to H.
//
// UMMAs issued by one thread complete in order, so the completion of S_i(j) (signalled to
// the softmax) also means PV_i(j-1) has finished reading P_i(j-1) and writing O_i.
//
// TMEM columns: S_0/P_0 at 0, S_1/P_1 at 128, O_0 at 256, O_1 at 384 (512 allocated).
#pragma once

#include <type_traits>

#include "params.h"
#include "ptx.cuh"

namespace gqa {

// Pairs of every 16 in a softmax chunk whose exponentials run on the FMA pipe (exp2_fma2)
// instead of the multi-function unit.  Measured on GB300 with 0, 2, 4, 6 and 8 of 16: every
// share made the kernel slower (B=1 x T=32768: 5.06-5.13 ms at 0, 5.16 at 2, 5.26-5.33 at 4,
// 5.74 at 8), so the softmax phase is not bounded by the multi-function unit here and the
// default is 0; the cubic stays available for parts where it is.
#ifndef GQA_FLASH_FMA_EXP2_PAIRS
#define GQA_FLASH_FMA_EXP2_PAIRS 0
#endif
constexpr int kFmaExp2Pairs = GQA_FLASH_FMA_EXP2_PAIRS;

struct FlashSmem {
  static constexpr int kTile = 128 * 128 * 2;  // one 128x128 bf16 tile (two 64-column halves)
  static constexpr int kHalf = 128 * 64 * 2;
  static constexpr int kQ = 0;                 // 2 tiles (head slots 0, 1)
  static constexpr int kK = kQ + 2 * kTile;    // 2 stages
  static constexpr int kV = kK + 2 * kTile;    // 2 stages
  static constexpr int kBar = kV + 2 * kTile;
  static constexpr int kBytes = kBar + 256 + 1024;
};

__global__ void __launch_bounds__(384, 1)
    flash_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmH,
                         const FlashParams p) {
  using L = FlashSmem;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2] stages
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;   // [2]
  uint64_t* v_empty = bars + 7;  // [2]
  uint64_t* s_full = bars + 9;   // [2] head slots
  uint64_t* p_lo = bars + 11;    // [2] head slots, 128 arrivals: P of keys 0..63 in TMEM
  uint64_t* p_hi = bars + 13;    // [2] head slots, 128 arrivals: P of keys 64..127
  uint64_t* o_full = bars + 15;  // [2] head slots
  uint64_t* drain = bars + 17;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work order (1-D grid, dispatched in index order): bands of groups_per_band (sequence,
  // kv group) pairs; within a band the heaviest query tiles first, across its groups and the
  // group's two head pairs.  A band's K/V are sized to stay in L2 while its CTAs run.
  const int band_ctas = p.groups_per_band * 2 * p.n_qtiles;
  const int band = static_cast<int>(blockIdx.x) / band_ctas;
  const int w_in = static_cast<int>(blockIdx.x) - band * band_ctas;
  const int qi = w_in / (2 * p.groups_per_band);
  const int gp = w_in - qi * 2 * p.groups_per_band;
  const int grp = band * p.groups_per_band + (gp >> 1);  // b * n_kv + kv group
  const int b = grp / p.n_kv;
  const int hp = ((grp - b * p.n_kv) << 1) | (gp & 1);
  const int h0 = 2 * hp;
  const int g = h0 >> 2;
  const int qt = p.n_qtiles - 1 - qi;  // heaviest tiles first
  const int q0 = qt * 128;
  const int kv_len = p.start_pos + p.T;
  const int kv_hi = p.causal ? min(kv_len, p.start_pos + q0 + 128) : kv_len;
  const int n_ktiles = (kv_hi + 127) / 128;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 18; ++i) mbar_init(&bars[i], (i >= 11 && i <= 14) ? 128u : 1u);
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
  griddep_launch_dependents();

  // registers: 168 x 384 at launch >= 72 x 128 (producer / issuer warpgroup) + 208 x 256
  // (the two softmax warpgroups)
  if (warp < 4) {
   setmaxnreg_dec<72>();
   if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      griddep_wait();  // Q_r, K_r, V come from the projection kernel
      // test hook: CTA 0 issues no loads, so its consumers wait out and abort
      const bool no_loads = p.fault && blockIdx.x == 0;
      if (!no_loads) mbar_arrive_expect_tx(q_full, 2 * L::kTile);
      for (int i = 0; i < (no_loads ? 0 : 2); ++i) {
        tma_load_3d(smem + L::kQ + i * L::kTile, &tmQ, q_full, (h0 + i) * 128, q0, b);
        tma_load_3d(smem + L::kQ + i * L::kTile + L::kHalf, &tmQ, q_full, (h0 + i) * 128 + 64, q0, b);
      }
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < (no_loads ? 0 : n_ktiles); ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&k_empty[st], ph ^ 1u, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&k_full[st], L::kTile);
        uint8_t* kd = smem + L::kK + st * L::kTile;
        tma_load_4d(kd, &tmK, &k_full[st], 0, g, j * 128, b);
        tma_load_4d(kd + L::kHalf, &tmK, &k_full[st], 64, g, j * 128, b);
        ++issued_k;
        if (!mbar_wait(&v_empty[st], ph ^ 1u, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&v_full[st], L::kTile);
        uint8_t* vd = smem + L::kV + st * L::kTile;
        tma_load_4d(vd, &tmV, &v_full[st], 0, g, j * 128, b);
        tma_load_4d(vd + L::kHalf, &tmV, &v_full[st], 64, g, j * 128, b);
        ++issued_v;
      }
      if (*abort_flag && !no_loads) {  // let copies still in flight land before the CTA leaves
        mbar_wait_drain(q_full, 0);
        for (int j = (issued_k > 2 ? issued_k - 2 : 0); j < issued_k; ++j)
          mbar_wait_drain(&k_full[j & 1], (j >> 1) & 1);
        for (int j = (issued_v > 2 ? issued_v - 2 : 0); j < issued_v; ++j)
          mbar_wait_drain(&v_full[j & 1], (j >> 1) & 1);
      }
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------------ UMMA issuer
    // The whole warp runs the loop (its waits are warp-uniform); one elected lane issues
    // the MMAs and commits.
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);   // Q, K both K-major
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 128, 0, 1);  // P (TMEM), V MN-major
    const uint32_t q_addr = smem_u32(smem + L::kQ);
    const uint32_t k_addr = smem_u32(smem + L::kK);
    const uint32_t v_addr = smem_u32(smem + L::kV);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.status));
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one_sync()) umma_commit(bar);
      __syncwarp();
    };
    // S_i(j) = Q_i K_j^T
    auto issue_s = [&](int i, int j) {
      const uint32_t d_s = tmem_base + i * 128;
      const uint64_t qd = sdesc_sw128(q_addr + i * L::kTile, 0, 1024);
      const uint64_t kd = sdesc_sw128(k_addr + (j & 1) * L::kTile, 0, 1024);
      if (elect_one_sync()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kHalf + (kk & 3) * 32) >> 4;  // descriptor address units
          umma_ss(d_s, qd + off, kd + off, idesc_s, kk != 0);
        }
        umma_commit(&s_full[i]);
      }
      __syncwarp();
    };
    // O_i += P_i(j) V_j for keys 16*kk0 .. 16*kk0+63 (kk0 = 0 or 4); P_i holds keys
    // (2c, 2c+1) in column c of S_i's TMEM columns.  V: MN-major (d contiguous); 16 keys =
    // two 8-row groups = 2048 B per step; d 64..127 lives in the second half (LBO), 8-key
    // groups 1024 B apart (SBO).
    auto issue_pv_half = [&](int i, int j, int kk0) {
      const uint32_t d_o = tmem_base + 256 + i * 128;
      const uint32_t a_p = tmem_base + i * 128;
      const uint64_t vd = sdesc_sw128(v_addr + (j & 1) * L::kTile, L::kHalf, 1024);
      if (elect_one_sync()) {
#pragma unroll
        for (int kk = kk0; kk < kk0 + 4; ++kk)
          umma_ts(d_o, a_p + kk * 8, vd + ((kk * 2048) >> 4), idesc_pv, (j | kk) != 0);
      }
      __syncwarp();
    };
    bool ok = wait(q_full, 0);
    if (ok) ok = wait(&k_full[0], 0);
    if (ok) {
      tc_fence_after();
      issue_s(0, 0);
      issue_s(1, 0);
      commit(&k_empty[0]);
    }
    for (int j = 0; ok && j < n_ktiles; ++j) {
      const bool more = j + 1 < n_ktiles;
      // head slot 0: PV_0(j) in two halves as P arrives, then S_0(j+1)
      if (!(ok = wait(&v_full[j & 1], (j >> 1) & 1))) break;
      if (!(ok = wait(&p_lo[0], j & 1))) break;
      tc_fence_after();
      issue_pv_half(0, j, 0);
      if (!(ok = wait(&p_hi[0], j & 1))) break;
      tc_fence_after();
      issue_pv_half(0, j, 4);
      if (!more) commit(&o_full[0]);
      if (more) {
        if (!(ok = wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1))) break;
        tc_fence_after();
        issue_s(0, j + 1);
      }
      // head slot 1: PV_1(j), then S_1(j+1)
      if (!(ok = wait(&p_lo[1], j & 1))) break;
      tc_fence_after();
      issue_pv_half(1, j, 0);
      if (!(ok = wait(&p_hi[1], j & 1))) break;
      tc_fence_after();
      issue_pv_half(1, j, 4);
      commit(&v_empty[j & 1]);
      if (!more) commit(&o_full[1]);
      if (more) {
        issue_s(1, j + 1);
        commit(&k_empty[(j + 1) & 1]);
      }
    }
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {  // let issued UMMAs finish before TMEM is released
      commit(drain);
      mbar_wait_drain(drain, 0);
    }
   }
  } else {
    setmaxnreg_inc<208>();
    // ------------------------------------------------------------------ softmax
    const int slot = (warp - 4) >> 2;  // head slot 0 or 1
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem_base + lane_off + slot * 128;
    const uint32_t t_o = tmem_base + lane_off + 256 + slot * 128;
    const int qpos = p.start_pos + q0 + r;
    float m_used = -INFINITY;
    float l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n_ktiles; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[slot], j & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      // All four TMEM loads in flight before the single wait.
      uint32_t sv[128];
      tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[64]));
      tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&sv[96]));
      tmem_ld_wait();
      const int key0 = j * 128;
      const bool needs_mask = (key0 + 127 >= kv_len) || (p.causal && key0 + 127 > p.start_pos + q0);
      if (needs_mask) {
        const int lim = p.causal ? min(kv_len - 1, qpos) : kv_len - 1;
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (key0 + i > lim) sv[i] = __float_as_uint(-INFINITY);
      }
      // Row max: 8 independent chains of 3-input max (max is exact in any order).
      float m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = __uint_as_float(sv[i]);
#pragma unroll
      for (int t = 0; t < 60; ++t)
        m8[t & 7] = max3f(m8[t & 7], __uint_as_float(sv[8 + 2 * t]), __uint_as_float(sv[9 + 2 * t]));
      const float mx = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      const float m_tile = mx * p.scale_log2;
      // Per-row lazy rescale decision (rows never influence each other's bits).
      float alpha = 1.f;
      bool grow = false;
      if (j == 0) {
        m_used = m_tile;
      } else if (m_tile > m_used + 8.0f) {
        grow = true;
        alpha = fast_exp2(m_used - m_tile);
        l_sum *= alpha;
        m_used = m_tile;
      }
      const float mu = (m_used == -INFINITY) ? 0.f : m_used;
      // P = exp2(s * scale_log2 - m_used), bf16, written over S_i in TMEM in two halves
      // (keys 0..63, then 64..127), each released as soon as it is stored; scale and shift
      // run as packed fp32 pairs and the row sum accumulates in 4 packed partial sums.
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
      const float2 nmu2 = make_float2(-mu, -mu);
      float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // Chunk c (keys 32c .. 32c+31) as 16 pairs.  On key tiles without masked entries the
      // last kFmaExp2Pairs pairs of each chunk take their exponentials on the FMA pipe
      // (exp2_fma2), the others on the multi-function unit, which alone would bound this
      // phase; tiles with masked (-inf) entries use the multi-function unit throughout, so
      // masked probabilities stay exactly 0.
      auto exp_chunk = [&](auto use_fma, int c, uint32_t(&w)[16]) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 a = ffma2(make_float2(__uint_as_float(sv[c * 32 + 2 * e]), __uint_as_float(sv[c * 32 + 2 * e + 1])),
                                 sc2, nmu2);
          float2 pe;
          if (decltype(use_fma)::value && e >= 16 - kFmaExp2Pairs)
            pe = exp2_fma2(a);
          else
            pe = make_float2(fast_exp2(a.x), fast_exp2(a.y));
          l4[e & 3] = fadd2(l4[e & 3], pe);
          w[e] = pack_bf16x2(pe.x, pe.y);
        }
      };
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
          uint32_t w[16];
          if constexpr (kFmaExp2Pairs > 0) {
            if (needs_mask)
              exp_chunk(std::false_type{}, c, w);
            else
              exp_chunk(std::true_type{}, c, w);
          } else {
            exp_chunk(std::false_type{}, c, w);
          }
          tmem_st16(t_s + c * 16, w);
        }
        if (hf == 0 && __any_sync(0xffffffffu, grow)) {
          // O_i holds the sum through key tile j-1 (PV_i(j-1) completed before S_i(j)); it
          // is rescaled before any part of P_i(j) is released to the tensor core.
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tmem_ld32(t_o + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(t_o + c * 32, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(hf == 0 ? &p_lo[slot] : &p_hi[slot]);
      }
      const float2 l2 = fadd2(fadd2(l4[0], l4[1]), fadd2(l4[2], l4[3]));
      l_sum += l2.x + l2.y;
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&o_full[slot], 0, abort_flag, p.status));
    if (ok) {
      // O / l as bf16 into this slot's Q tile (free once the last UMMA has completed), in the
      // 128-byte-swizzled layout the tile was loaded in: row r, 16-byte chunk c of a 64-column
      // half at chunk position c ^ (r & 7) (conflict-free); then two TMA stores, which leave
      // out the rows of a ragged last tile past T.
      tc_fence_after();
      const float inv_l = 1.f / l_sum;
      uint8_t* tile = smem + L::kQ + slot * L::kTile;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(t_o + c * 32, v);
        tmem_ld_wait();
        uint8_t* row_base = tile + (c >> 1) * L::kHalf + r * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = (c & 1) * 4 + k;
          const uint4 w4 = make_uint4(pack_bf16x2(__uint_as_float(v[8 * k + 0]) * inv_l, __uint_as_float(v[8 * k + 1]) * inv_l),
                                      pack_bf16x2(__uint_as_float(v[8 * k + 2]) * inv_l, __uint_as_float(v[8 * k + 3]) * inv_l),
                                      pack_bf16x2(__uint_as_float(v[8 * k + 4]) * inv_l, __uint_as_float(v[8 * k + 5]) * inv_l),
                                      pack_bf16x2(__uint_as_float(v[8 * k + 6]) * inv_l, __uint_as_float(v[8 * k + 7]) * inv_l));
          *reinterpret_cast<uint4*>(row_base + ((chunk ^ (r & 7)) << 4)) = w4;
        }
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(2 + slot, 128);
    if (ok && quarter == 0 && lane == 0) {
      const uint8_t* tile = smem + L::kQ + slot * L::kTile;
      tma_store_3d(&tmH, tile, (h0 + slot) * 128, q0, b);
      tma_store_3d(&tmH, tile + L::kHalf, (h0 + slot) * 128 + 64, q0, b);
      tma_store_commit();
      tma_store_wait_read();
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
