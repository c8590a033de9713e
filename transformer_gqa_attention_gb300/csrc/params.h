// params.h — launch parameter blocks and constants shared by the kernels and the host
// code (no device code here).
#pragma once

#include <cstdint>

namespace gqa {

// Status bits OR-ed into the context's device status word.
constexpr int kDevErrTimeout = 1;

// Upper bound for any single device-side wait (wall-clock, via %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s while draining after an abort

// kQkvRope / kStoreF32: many-token epilogues.  kSplitKQkv / kSplitKOut: the same two
// epilogues after the cluster-wide split-K reduction of the few-token kernel.
enum EpiMode : int { kQkvRope = 0, kStoreF32 = 1, kSplitKQkv = 3, kSplitKOut = 4 };

struct GemmParams {
  int M, N;          // rows of A, rows of B
  int num_kb;        // K / 64
  int splits;        // few-token kernel: k splits = cluster size
  int n_tiles;       // CTA-pair kernels: 256-wide output tiles along N (split-K kernels: 1)
  int m_tiles;       // ceil(M / 128)
  // CTA-pair kernel schedule: full_rounds rounds of whole 256x256 tiles, then the tiles of
  // the last, partial round cut into pieces of tail_w columns (0: whole tiles throughout)
  int full_rounds, tail_w;
  // Q/K/V epilogues: the packed weight's rows are q_cols query features (4 heads x 128 per
  // kv group), then kv_cols key and kv_cols value features (128 per kv group); Q_r rows are
  // q_cols wide and a cache position holds kv_cols features.  The whole block: 4096 / 1024.
  int q_cols, kv_cols;
  // epilogue operands
  void* out0;        // kQkvRope: Q_r [M,q_cols] bf16 | kStoreF32: D fp32
  void* out1;        // kQkvRope: cache_k
  void* out2;        // kQkvRope: cache_v
  const float* R;    // Q/K/V epilogues: [T,64,2]
  int T, S_max, start_pos;
  int ldo;           // kStoreF32: row stride (floats)
  void* fin0;        // split-K final outputs: Q_r [N,q_cols] bf16 | Delta [N,4096] fp32
  void* fin1;        // kSplitKQkv: cache_k
  void* fin2;        // kSplitKQkv: cache_v
  int* status;
  int fault;         // test hook: the first work unit's producer issues no loads (its waits run out)
  // residual form of the block (both null for the block alone)
  const float* row_scale;  // Q/K/V epilogues: 1 / rms of each token row (attention_norm)
  const void* residual;    // Delta epilogues: x [tokens, 4096] bf16, added to Delta
};

struct FlashParams {
  int B, T, S_max, start_pos, causal;
  int n_kv;             // kv groups (heads of K/V) of the context; 4 query heads each
  int n_qtiles;
  int groups_per_band;  // (sequence, kv group) pairs scheduled together (divides n_kv B)
  int* status;
  int fault;  // test hook: CTA 0's producer issues no loads (its waits run out)
  float scale_log2;  // log2(e) / sqrt(128)
};

constexpr int kDecStages = 3;
constexpr int kDecTileKeys = 64;

struct DecodeParams {
  int B, kv_len, n_splits, tiles_per_split;
  int n_kv;       // kv groups of the context (4 query heads each; q and H rows are 512 n_kv wide)
  // query positions: T per sequence, the first at absolute position q_start (decode: T = 1,
  // q_start = kv_len - 1); with causal, query t sees keys 0 .. q_start + t, else all kv_len
  int T, q_start, causal;
  int n_pg;       // position groups per sequence (ceil(T / positions per CTA))
  const void* q;  // [B, T, 512 n_kv] bf16 rotated queries
  float* part_o;           // [B, n_kv, n_pg, n_splits, rows, 128]
  float* part_ml;          // [B, n_kv, n_pg, n_splits, rows, 2]
  int* counters;           // [B*n_kv*n_pg] arrival counters: the last split merges (null: separate merge kernel)
  void* H;        // [B, T, 512 n_kv] bf16 (combine output)
  int* status;
  // decode_combine_kernel only: when *status is non-zero (a split of this call gave up a
  // wait), H is written as NaN and the status bits are OR-ed into *status_sticky (null: not)
  int* status_sticky;
  int fault;      // test hook: CTA (0, 0, 0)'s producer issues no loads (its waits run out)
  float scale_log2;
};

}  // namespace gqa
