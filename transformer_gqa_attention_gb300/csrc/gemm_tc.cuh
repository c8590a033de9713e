// gemm_tc.cuh — tcgen05 GEMMs of the block's projections, D = A * B^T with both operands
// K-major bf16 (the [out, in] weight storage of the quoted F.linear layers) and fp32
// accumulation in TMEM.  Two kernels:
//
//   gemm_tc_pair_kernel (many tokens) — persistent CTA pairs (cta_group::2), 256x256
//     output tiles, double-buffered TMEM accumulators so the epilogue of one tile runs
//     under the main loop of the next.  Warp roles per CTA: warp 0 TMA producer, warp 1
//     TMEM owner (+ the single UMMA-issuing thread in CTA 0 of the pair), warps 2..5
//     epilogue.  Tiles are numbered with the n tile fastest so the pairs resident at one
//     time share A row bands through L2; the tiles of a last, partial round are cut along
//     N into narrower items spread over all pairs (pair_item).
//   gemm_splitk_cluster_kernel (few tokens) — swap-AB split-K over a thread-block cluster
//     with the reduction done through distributed shared memory.
//
// Operands are read through 3-D tensor maps (64 columns, rows, 64-column k block), box
// 64 x {32,64,128} x 1 (and 64 x tail_w/2 x 1 for the weight rows of a last-round piece), so
// the same kernels read row-major activations (k-block stride 128 B) and the k-block-major
// weight copies the context keeps (each 128-row box one contiguous 16 KB).
//
// Epilogues:
//   kQkvRope  — the fused Q/K/V projection (steps 1-5 of "Llama 3.1 8B · Grouped-query
//               attention"): columns 0..4095 are Q, 4096..5119 K, 5120..6143 V of the
//               packed [6144,4096] weight (for a context over G of the 8 kv groups:
//               512 G query, then 128 G key and 128 G value columns).  Q and K pairs
//               (2j, 2j+1) are rotated by R[t, j] in fp32, then Q is stored to the Q_r
//               buffer [B*T,512 G] and K_r, V straight into the caches [B,S_max,G,128] at
//               position start_pos + t.
//   kStoreF32 — Delta = H W_O^T (step 14) stored fp32 row-major.
//   kSplitKQkv / kSplitKOut — the same two epilogues for the few-token kernel.
#pragma once

#include "pair_sched.h"
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

// Few-token split-K kernel: whether the partial tile [BN][128] fp32 and the receive slots
// (splits x ceil(BN / splits) token rows of 512 bytes) fit in the STAGES stage buffers.
template <int BN, int STAGES>
constexpr bool splitk_fits(int splits) {
  return BN * 128 * 4 + splits * ((BN + splits - 1) / splits) * 512 <= STAGES * GemmSmem<BN, STAGES>::kStageBytes;
}

// Epilogue of 32 x 32 chunks held by a warp (lane i = output row m_base + i).  A chunk goes
// through a per-warp shared-memory tile (32 rows, stride 36 floats: conflict-free 16-byte
// writes and reads) so that global stores and the RoPE table reads cover contiguous row
// segments instead of one 16-byte piece of 32 rows each.
constexpr int kEpiStride = 36;
constexpr int kEpiWarpFloats = 32 * kEpiStride;

__device__ __forceinline__ void stage_chunk(float* stage, int lane, const uint32_t (&v)[32]) {
  float4* srow = reinterpret_cast<float4*>(stage + lane * kEpiStride);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    srow[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]), __uint_as_float(v[4 * i + 2]),
                          __uint_as_float(v[4 * i + 3]));
}

// Rows of the Q/K/V epilogue after the transpose: pass k (0..3) of a lane handles row
// 8k + lane/4 of the warp's 32 rows, columns 8 (lane & 3) .. +7 of the chunk.
struct QkvRows {
  int m[4], b[4], t[4];
  float rs[4];  // row scale (1 / rms of the token row under attention_norm; 1 for the block alone)
};

__device__ __forceinline__ QkvRows qkv_rows(const GemmParams& p, int lane, int m_base) {
  QkvRows q;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    q.m[k] = m_base + 8 * k + (lane >> 2);
    const int mc = min(q.m[k], p.M - 1);
    q.b[k] = mc / p.T;
    q.t[k] = mc - q.b[k] * p.T;
    q.rs[k] = 1.f;
  }
  return q;
}

// The rows' 1 / rms (residual form).  It comes from the previous kernel, so it is read only
// after the accumulator wait, which follows the producer's wait for that kernel.
__device__ __forceinline__ void qkv_row_scales(const GemmParams& p, QkvRows& q) {
  if (!p.row_scale) return;
#pragma unroll
  for (int k = 0; k < 4; ++k) q.rs[k] = __ldg(p.row_scale + min(q.m[k], p.M - 1));
}

// (cos, sin) of the 4 RoPE pairs a lane rotates in chunk-column block cc (0..3) of a head
// slice: pairs 16 cc + 4 (lane & 3) .. +3 of each of its 4 rows.
__device__ __forceinline__ void load_rope(const GemmParams& p, const QkvRows& q, int lane, int cc,
                                          float4 (&cs)[4][2]) {
  const int j0 = 16 * cc + 4 * (lane & 3);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4* rp = reinterpret_cast<const float4*>(p.R + (static_cast<size_t>(q.t[k]) * 64 + j0) * 2);
    cs[k][0] = __ldg(rp);
    cs[k][1] = __ldg(rp + 1);
  }
}

// Q/K/V epilogue of one staged chunk (columns col0 .. col0+31, all of one of Q, K, V: the
// boundaries are multiples of 128).
__device__ __forceinline__ void store_qkv_chunk(const GemmParams& p, const float* stage, int lane, const QkvRows& q,
                                                int col0, const float4 (&cs)[4][2]) {
  const int cq = lane & 3;
  const int col = col0 + 8 * cq;
  const int k_col0 = p.q_cols;              // first key column
  const int v_col0 = p.q_cols + p.kv_cols;  // first value column
  const bool is_v = col0 >= v_col0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = 8 * k + (lane >> 2);
    if (q.m[k] >= p.M) continue;
    float4 x0 = *reinterpret_cast<const float4*>(stage + r * kEpiStride + 8 * cq);
    float4 x1 = *reinterpret_cast<const float4*>(stage + r * kEpiStride + 8 * cq + 4);
    const float rs = q.rs[k];
    x0 = make_float4(x0.x * rs, x0.y * rs, x0.z * rs, x0.w * rs);
    x1 = make_float4(x1.x * rs, x1.y * rs, x1.z * rs, x1.w * rs);
    uint4 w;
    if (is_v) {
      w = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w), pack_bf16x2(x1.x, x1.y),
                     pack_bf16x2(x1.z, x1.w));
    } else {
      const float4 c0 = cs[k][0], c1 = cs[k][1];  // (cos, sin) of two pairs per float4
      w = make_uint4(pack_bf16x2(c0.x * x0.x - c0.y * x0.y, c0.y * x0.x + c0.x * x0.y),
                     pack_bf16x2(c0.z * x0.z - c0.w * x0.w, c0.w * x0.z + c0.z * x0.w),
                     pack_bf16x2(c1.x * x1.x - c1.y * x1.y, c1.y * x1.x + c1.x * x1.y),
                     pack_bf16x2(c1.z * x1.z - c1.w * x1.w, c1.w * x1.z + c1.z * x1.w));
    }
    __nv_bfloat16* dst;
    if (col0 < k_col0) {
      dst = static_cast<__nv_bfloat16*>(p.out0) + static_cast<size_t>(q.m[k]) * p.q_cols + col;
    } else {
      const size_t cache_row = static_cast<size_t>(q.b[k]) * p.S_max + p.start_pos + q.t[k];
      dst = static_cast<__nv_bfloat16*>(is_v ? p.out2 : p.out1) + cache_row * p.kv_cols + (col - (is_v ? v_col0 : k_col0));
    }
    *reinterpret_cast<uint4*>(dst) = w;
  }
}

// four bf16 (8 bytes) widened to fp32
__device__ __forceinline__ float4 bf16x4_to_float4(uint2 v) {
  return make_float4(bf16lo_to_f32(v.x), bf16hi_to_f32(v.x), bf16lo_to_f32(v.y), bf16hi_to_f32(v.y));
}

// Residual values (bf16, 4 per lane and pass) a lane adds in store_f32_chunk for the chunk at
// columns col0 .. col0+31.
__device__ __forceinline__ void load_residual_chunk(const GemmParams& p, int lane, int m_base, int col0,
                                                    uint2 (&rv)[8]) {
  const int c4 = col0 + 4 * (lane & 7);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int m = min(m_base + 4 * k + (lane >> 3), p.M - 1);
    rv[k] = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.residual) +
                                                 static_cast<size_t>(m) * 4096 + c4));
  }
}

// fp32 epilogue of one staged chunk: 8 passes of 4 rows, lane -> row 4k + lane/8, columns
// col0 + 4 (lane & 7) .. +3; with a residual, the values read by load_residual_chunk are added.
__device__ __forceinline__ void store_f32_chunk(const GemmParams& p, const float* stage, int lane, int m_base,
                                                int col0, const uint2 (&rv)[8]) {
  const int c4 = col0 + 4 * (lane & 7);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int r = 4 * k + (lane >> 3);
    const int m = m_base + r;
    if (m >= p.M) continue;
    float4 x = *reinterpret_cast<const float4*>(stage + r * kEpiStride + 4 * (lane & 7));
    if (p.residual) {
      const float4 h = bf16x4_to_float4(rv[k]);
      x = make_float4(h.x + x.x, h.y + x.y, h.z + x.z, h.w + x.w);
    }
    *reinterpret_cast<float4*>(static_cast<float*>(p.out0) + static_cast<size_t>(m) * p.ldo + c4) = x;
  }
}

// ---------------------------------------------------------------------------------------
// CTA-pair variant (cta_group::2) for the many-token projections: a cluster of two CTAs
// computes one 256x256 output tile.  CTA r stages its own 128 rows of A (rows m0+128r..)
// and its own 128 rows of B (rows n0+128r.., i.e. half of the tile's N) per 64-wide k
// block; the single issuing thread in CTA 0 runs 256x256x16 UMMAs that read both CTAs'
// shared memory and leave each CTA's 128 output rows (all 256 columns) in its own TMEM.
// Per CTA a stage is 32 KB instead of 48 KB for a 128x256 single-CTA tile, so six stages
// fit and each SM streams half as many B bytes per FLOP.
//   - both CTAs' TMA loads complete on CTA 0's full barrier (CTA 0 expects both halves);
//   - CTA 0's commits arrive on the empty / accumulator-full barriers of both CTAs;
//   - each CTA's epilogue warps release an accumulator on CTA 0's acc_empty barrier.
template <int STAGES>
struct GemmPairSmem {
  static constexpr int kABytes = 128 * 64 * 2;
  static constexpr int kBBytes = 128 * 64 * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOffset = STAGES * kStageBytes;
  static constexpr int kEpiOffset = kBarOffset + 256;  // 4 epilogue warps' staging tiles
  static constexpr int kBytes = kEpiOffset + 4 * kEpiWarpFloats * 4 + 1024;
  static constexpr int kTmemCols = 512;  // two 256-column accumulators
};

template <int STAGES, int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmBt, const GemmParams p) {
  using L = GemmPairSmem<STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::kABytes;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* acc_full = empty_bar + STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;       // [2], used in CTA 0 only
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 8);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, L::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer barriers initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      tma_prefetch_desc(&tmBt);
      int it = 0;
      bool ok = true;
      // B is the context's weight copy (never written after creation): its first stages are
      // fetched before waiting for the previous kernel; A (activations) only after.
      // test hook: pair 0 issues no loads, so CTA 0's issuer waits out and aborts
      // B rows of an item: CTA r holds rows n0 + w/2 * r .. + w/2 - 1 of the weight, fetched as
      // one box per stage: 128 rows for a whole tile (tmB), tail_w / 2 rows for a piece of the
      // partial round (tmBt; rows past the piece are not read by the UMMA, rows past the
      // weight are zero-filled).  CTA 0's barrier counts both CTAs' A and B boxes.
      const bool no_loads = p.fault && pair == 0;
      auto load_b = [&](int st, uint32_t bar, int n0, int w, int kb) {
        if (w == 256)
          tma_load_3d_pair(sB + st * L::kBBytes, &tmB, bar, 0, n0 + 128 * static_cast<int>(rank), kb);
        else
          tma_load_3d_pair(sB + st * L::kBBytes, &tmBt, bar, 0, n0 + (w >> 1) * static_cast<int>(rank), kb);
      };
      auto stage_tx = [&](int w) { return 2 * (L::kABytes + 64 * (w == 256 ? 256 : p.tail_w)); };
      int mt, n0, w;
      const int n_pre = (pair_item(p, pair, n_pairs, 0, mt, n0, w) && !no_loads) ? min(STAGES, p.num_kb) : 0;
      for (int i = 0; i < n_pre; ++i) {
        if (rank == 0) mbar_arrive_expect_tx(&full_bar[i], stage_tx(w));
        load_b(i, mapa_shared(smem_u32(&full_bar[i]), 0), n0, w, i);
      }
      griddep_wait();
      for (int idx = 0; ok && !no_loads && pair_item(p, pair, n_pairs, idx, mt, n0, w); ++idx) {
        const int m0 = mt * 256 + 128 * rank;
        for (int i = 0; i < p.num_kb; ++i, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          const uint32_t bar0 = mapa_shared(smem_u32(&full_bar[s]), 0);
          if (it < n_pre) {  // B already requested above
            tma_load_3d_pair(sA + s * L::kABytes, &tmA, bar0, 0, m0, i);
            continue;
          }
          if (!mbar_wait(&empty_bar[s], ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], stage_tx(w));
          tma_load_3d_pair(sA + s * L::kABytes, &tmA, bar0, 0, m0, i);
          load_b(s, bar0, n0, w, i);
        }
      }
      if (*abort_flag && rank == 0) {  // CTA 0's barriers count both CTAs' bytes
        for (int i = (it > STAGES ? it - STAGES : 0); i < it; ++i)
          mbar_wait_drain(&full_bar[i % STAGES], (i / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ------------------------------------------------------------ UMMA issuer (CTA 0)
      // The whole warp runs the loop (waits are warp-uniform); one elected lane issues.
      const uint32_t a_base = smem_u32(sA);
      const uint32_t b_base = smem_u32(sB);
      int it = 0, lt = 0;
      bool ok = true;
      int mt, n0, w;
      for (; ok && pair_item(p, pair, n_pairs, lt, mt, n0, w); ++lt) {
        const int ab = lt & 1;
        const uint32_t idesc = idesc_bf16_f32(256, w, 0, 0);
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_cluster(&acc_empty[ab], ((lt >> 1) & 1) ^ 1u, abort_flag,
                                                             p.status))))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * 256;
        for (int i = 0; i < p.num_kb; ++i, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&full_bar[s], ph, abort_flag, p.status)))) break;
          tc_fence_after();
          const uint64_t da = sdesc_sw128(a_base + s * L::kABytes, 0, 1024);
          const uint64_t db = sdesc_sw128(b_base + s * L::kBBytes, 0, 1024);
          if (elect_one_sync()) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_ss_pair(d_tmem, da + 2 * k, db + 2 * k, idesc, (i | k) != 0);
            umma_commit_pair(&empty_bar[s], 0x3);
          }
          __syncwarp();
        }
        if (ok) {
          if (elect_one_sync()) umma_commit_pair(&acc_full[ab], 0x3);
          __syncwarp();
        }
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {  // let issued UMMAs finish before TMEM is released
        if (elect_one_sync()) umma_commit_pair(drain, 0x1);
        __syncwarp();
        mbar_wait_drain(drain, 0);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    float* stage = reinterpret_cast<float*>(smem + L::kEpiOffset) + (warp - 2) * kEpiWarpFloats;
    int lt = 0;
    int mt, n0, w;
    for (; pair_item(p, pair, n_pairs, lt, mt, n0, w); ++lt) {
      const int ab = lt & 1;
      const int m_base = mt * 256 + 128 * rank + quarter * 32;
      // The item's 32-column chunks i = 0 .. w/32 - 1 sit at accumulator columns 32 i and
      // output columns n0 + 32 i; pass cp stores chunks cp and cp + 4, which lie 128 columns
      // (one head slice) apart and so rotate by the same RoPE pairs, those of position
      // ((n0 / 32) + cp) mod 4 of a head slice.  Q/K items read all their rotation
      // coefficients before waiting for the accumulator, so the latency hides under the main
      // loop (an item may mix key and value chunks: each chunk picks its own store).
      const bool rope = EPI == kQkvRope && n0 < p.q_cols + p.kv_cols;
      QkvRows qr{};
      float4 cs[4][4][2];
      // Delta items with a residual: the residual of chunk pair cp + 1 is read while pair cp
      // is stored (pair 0 before the accumulator wait)
      uint2 rva[8], rvb[8], rva_n[8], rvb_n[8];
      if constexpr (EPI == kQkvRope) {
        qr = qkv_rows(p, lane, m_base);
        if (rope) {
#pragma unroll
          for (int cp = 0; cp < 4; ++cp) load_rope(p, qr, lane, ((n0 >> 5) + cp) & 3, cs[cp]);
        }
      } else {
        if (p.residual) {
          load_residual_chunk(p, lane, m_base, n0, rva);
          if (w > 128) load_residual_chunk(p, lane, m_base, n0 + 128, rvb);
        }
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[ab], (lt >> 1) & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      if constexpr (EPI == kQkvRope) qkv_row_scales(p, qr);
      const uint32_t t_row = tmem_base + lane_off + ab * 256;
#pragma unroll
      for (int cp = 0; cp < 4; ++cp) {
        const bool has_a = 32 * cp < w, has_b = 32 * (cp + 4) < w;
        if constexpr (EPI == kStoreF32) {
          if (p.residual && cp < 3) {
            if (32 * (cp + 1) < w) load_residual_chunk(p, lane, m_base, n0 + (cp + 1) * 32, rva_n);
            if (32 * (cp + 5) < w) load_residual_chunk(p, lane, m_base, n0 + (cp + 5) * 32, rvb_n);
          }
        }
        if (!has_a) break;  // chunks are filled in order: none left
        uint32_t va[32], vb[32];
        tmem_ld32(t_row + cp * 32, va);
        if (has_b) tmem_ld32(t_row + (cp + 4) * 32, vb);
        tmem_ld_wait();
        stage_chunk(stage, lane, va);
        __syncwarp();
        if constexpr (EPI == kQkvRope) {
          store_qkv_chunk(p, stage, lane, qr, n0 + cp * 32, cs[cp]);
        } else {
          store_f32_chunk(p, stage, lane, m_base, n0 + cp * 32, rva);
        }
        __syncwarp();
        if (has_b) {
          stage_chunk(stage, lane, vb);
          __syncwarp();
          if constexpr (EPI == kQkvRope) {
            store_qkv_chunk(p, stage, lane, qr, n0 + (cp + 4) * 32, cs[cp]);
          } else {
            store_f32_chunk(p, stage, lane, m_base, n0 + (cp + 4) * 32, rvb);
          }
          __syncwarp();
        }
        if constexpr (EPI == kStoreF32) {
          if (p.residual && cp < 3) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              rva[k] = rva_n[k];
              rvb[k] = rvb_n[k];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[ab]), 0));
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's UMMAs or remote arrivals are live
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, L::kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// Few-token projections (swap-AB: A = 128 weight rows = output features, B = the <= 64
// token rows), split along K over the CTAs of one thread-block cluster (cluster rank =
// split).  Each CTA accumulates its K range in TMEM, parks the fp32 partial tile
// [BN tokens][128 features] in its own shared memory, and after one cluster barrier pushes
// to each peer, with one bulk shared-to-shared copy, the rows of the tokens that peer
// reduces; each CTA then sums its own tokens from its shared memory and applies the final
// epilogue:
//   kSplitKQkv — RoPE of Q and K pairs (adjacent lanes hold a pair), Q_r and the cache
//                entries stored bf16 (steps 1-5);
//   kSplitKOut — Delta stored fp32 (step 14).
// BN: token columns of the UMMA (64, or 32 for at most 32 tokens: a smaller activation
// stage).  STAGES <= 5 runs two CTAs per SM: a CTA's loop is bound by the tensor core's cost
// per 128 x BN x 16 instruction rather than by bytes in flight, so two CTAs over shorter k
// ranges finish sooner than one with a deeper ring.
template <int EPI, int STAGES, int BN>
__global__ void __launch_bounds__(192, (STAGES <= 5 ? 2 : 1))
    gemm_splitk_cluster_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                               const GemmParams p) {
  static_assert(BN == 32 || BN == 64, "token tile of 32 or 64");
  using L = GemmSmem<BN, STAGES>;
  // after the main loop the stage buffers hold this CTA's partial tile, token-major
  // [BN tokens][128 features] fp32, then the receive slots: per source rank the rows of the
  // tokens this CTA reduces, slot_tok = ceil(BN / splits) of them (splitk_fits checks on the
  // host that partial tile and slots fit in the stage buffers)
  constexpr int kPartBytes = BN * 128 * 4;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::kABytes;
  float* red = reinterpret_cast<float*>(smem);                // [64 tokens][128] partial tile
  float* recv = reinterpret_cast<float*>(smem + kPartBytes);  // [source rank][slot_tok][128]
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* acc_full = empty_bar + STAGES;
  uint64_t* drain = acc_full + 1;
  uint64_t* recv_bar = drain + 1;  // completes when every peer's rows for this CTA have landed
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(recv_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = static_cast<int>(cluster_ctarank());
  const int m0 = (blockIdx.x / p.splits) * 128;
  const int kb0 = split * p.num_kb / p.splits;
  const int nkb = (split + 1) * p.num_kb / p.splits - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    mbar_init(recv_bar, 1);
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
  griddep_launch_dependents();

  // CTA r reduces tokens [r N / splits, (r+1) N / splits); its recv_bar expects those rows
  // from every other split
  const int t_lo = split * p.N / p.splits;
  const int t_hi = (split + 1) * p.N / p.splits;
  const int slot_tok = (BN + p.splits - 1) / p.splits;
  if (threadIdx.x == 64)
    mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((p.splits - 1) * (t_hi - t_lo)) * 512u);
  // Epilogue warp w reduces tokens t_lo + w + 4 j, j < kTokPerWarp (at most BN / 2 tokens per
  // CTA for splits >= 2); for Q/K/V its lanes' RoPE coefficients of those tokens are read
  // while the main loop runs (an input of the call), not one L2 round trip per token pair
  // after the reduction
  constexpr int kTokPerWarp = BN / 8;
  float4 cs[kTokPerWarp];

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      // A is the context's weight copy (never written after creation): its first stages are
      // fetched before waiting for the previous kernel; B (activations) only after.
      // test hook: cluster 0 issues no loads, so its issuers wait out and abort
      const bool no_loads = p.fault && static_cast<int>(blockIdx.x) < p.splits;
      const int n_pre = no_loads ? 0 : min(STAGES, nkb);
      for (int i = 0; i < n_pre; ++i) {
        mbar_arrive_expect_tx(&full_bar[i], L::kStageBytes);
        tma_load_3d(sA + i * L::kABytes, &tmA, &full_bar[i], 0, m0, kb0 + i);
      }
      griddep_wait();
      int issued = 0;
      for (int i = 0; i < (no_loads ? 0 : nkb); ++i) {
        const int s = i % STAGES;
        if (i >= n_pre) {
          if (!mbar_wait(&empty_bar[s], ((i / STAGES) & 1) ^ 1u, abort_flag, p.status)) break;
          mbar_arrive_expect_tx(&full_bar[s], L::kStageBytes);
          tma_load_3d(sA + s * L::kABytes, &tmA, &full_bar[s], 0, m0, kb0 + i);
        }
        tma_load_3d(sB + s * L::kBBytes, &tmB, &full_bar[s], 0, 0, kb0 + i);
        ++issued;
      }
      if (*abort_flag) {
        for (int i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
          mbar_wait_drain(&full_bar[i % STAGES], (i / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // the whole warp runs the loop (waits are warp-uniform); one elected lane issues
    constexpr uint32_t idesc = idesc_bf16_f32(128, BN, 0, 0);
    const uint32_t a_base = smem_u32(sA);
    const uint32_t b_base = smem_u32(sB);
    bool ok = true;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&full_bar[s], (i / STAGES) & 1, abort_flag, p.status)))) break;
      tc_fence_after();
      const uint64_t da = sdesc_sw128(a_base + s * L::kABytes, 0, 1024);
      const uint64_t db = sdesc_sw128(b_base + s * L::kBBytes, 0, 1024);
      if (elect_one_sync()) {
#pragma unroll
        for (int k = 0; k < 4; ++k) umma_ss(tmem_base, da + 2 * k, db + 2 * k, idesc, (i | k) != 0);
        umma_commit(&empty_bar[s]);
      }
      __syncwarp();
    }
    if (elect_one_sync()) umma_commit(ok ? acc_full : drain);
    __syncwarp();
    if (!ok) mbar_wait_drain(drain, 0);
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    if constexpr (EPI == kSplitKQkv) {
      const int m = m0 + 4 * lane;  // pairs (m & 127) / 2 and the next one
      const bool rope = m < p.q_cols + p.kv_cols;
#pragma unroll
      for (int j = 0; j < kTokPerWarp; ++j) {
        const int tok = t_lo + (warp - 2) + 4 * j;
        cs[j] = make_float4(1.f, 0.f, 1.f, 0.f);  // value features: not rotated
        if (rope && tok < t_hi) {
          const int t = tok - (tok / p.T) * p.T;
          cs[j] = __ldg(reinterpret_cast<const float4*>(p.R + (static_cast<size_t>(t) * 64 + ((m & 127) >> 1)) * 2));
        }
      }
    }
    // accumulator rows (features) -> this CTA's partial tile in shared memory
    if (bar1_and_128(mbar_wait(acc_full, 0, abort_flag, p.status))) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) red[(c * 32 + i) * 128 + row] = __uint_as_float(v[i]);
      }
      fence_proxy_async_smem();  // the bulk copies below read these rows
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every split's partial tile is in its CTA's shared memory

  // Every CTA pushes the rows of its partial tile that CTA d reduces into CTA d's receive
  // slot with one bulk shared-to-shared copy, completing on CTA d's recv_bar; CTA d then sums
  // from its own shared memory.  The copies are issued even after an abort (no TMA write is
  // in flight past the barrier above), so every recv_bar completes and no CTA leaves while a
  // copy into it is landing.
  if (threadIdx.x == 64) {
    for (int d = 0; d < p.splits; ++d) {
      const int d_lo = d * p.N / p.splits;
      const int d_hi = (d + 1) * p.N / p.splits;
      if (d == split || d_hi == d_lo) continue;
      bulk_copy_smem_to_cluster(mapa_shared(smem_u32(recv) + static_cast<uint32_t>(split * slot_tok) * 512u, d),
                                smem_u32(red + d_lo * 128), static_cast<uint32_t>(d_hi - d_lo) * 512u,
                                mapa_shared(smem_u32(recv_bar), d));
    }
  }
  bool go = false;
  if (warp >= 2) {
    go = !*abort_flag;
    if (go) {
      go = mbar_wait(recv_bar, 0, abort_flag, p.status);
    } else {
      mbar_wait_drain(recv_bar, 0);
    }
    go = bar1_and_128(go);
  }
  if (go) {
    // Warp w of the four epilogue warps takes tokens t_lo + w, t_lo + w + 4, ...; lane l takes
    // features 4l .. 4l+3 of the CTA's 128 (two RoPE pairs), so every shared load is a
    // conflict-free 16-byte read and one warp store writes a token's whole 128-feature row.
    const int ew = warp - 2;
    const int f0 = 4 * lane;
    const int m = m0 + f0;
#pragma unroll
    for (int j = 0; j < kTokPerWarp; ++j) {
      const int tok = t_lo + ew + 4 * j;
      if (tok >= t_hi) break;
      float4 acc = *reinterpret_cast<const float4*>(red + tok * 128 + f0);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        if (r < p.splits && r != split) {
          const float4 v = *reinterpret_cast<const float4*>(recv + (r * slot_tok + tok - t_lo) * 128 + f0);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
      }
      if constexpr (EPI == kSplitKOut) {
        if (p.residual) {  // x + Delta
          const float4 h = bf16x4_to_float4(__ldg(reinterpret_cast<const uint2*>(
              static_cast<const __nv_bfloat16*>(p.residual) + static_cast<size_t>(tok) * 4096 + m)));
          acc = make_float4(h.x + acc.x, h.y + acc.y, h.z + acc.z, h.w + acc.w);
        }
        *reinterpret_cast<float4*>(static_cast<float*>(p.fin0) + static_cast<size_t>(tok) * 4096 + m) = acc;
      } else {
        if (p.row_scale) {  // attention_norm: the token row's 1 / rms
          const float rs = __ldg(p.row_scale + tok);
          acc = make_float4(acc.x * rs, acc.y * rs, acc.z * rs, acc.w * rs);
        }
        const int b = tok / p.T;
        const int t = tok - b * p.T;
        if (m < p.q_cols + p.kv_cols) {  // RoPE of the Q and K pairs
          const float4 c4 = cs[j];
          const float e0 = acc.x, o0 = acc.y, e1 = acc.z, o1 = acc.w;
          acc = make_float4(c4.x * e0 - c4.y * o0, c4.y * e0 + c4.x * o0, c4.z * e1 - c4.w * o1, c4.w * e1 + c4.z * o1);
        }
        const uint2 o = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        if (m < p.q_cols) {
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.fin0) + static_cast<size_t>(tok) * p.q_cols + m) = o;
        } else {
          const int v_col0 = p.q_cols + p.kv_cols;
          const bool is_v = m >= v_col0;
          const size_t crow = static_cast<size_t>(b) * p.S_max + p.start_pos + t;
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(is_v ? p.fin2 : p.fin1) + crow * p.kv_cols +
                                    (m - (is_v ? v_col0 : p.q_cols))) = o;
        }
      }
    }
  }

  // no CTA leaves while a peer's copy out of its partial tile may be in flight (every copy
  // has completed once its destination's recv_bar has, which each CTA waited for above)
  cluster_sync_relaxed();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, BN);
  }
}

}  // namespace gqa
