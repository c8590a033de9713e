// gqa_abi.cu — the C ABI declared in include/gqa_attn.h: argument validation, the
// context (packed weights, status word, workspace), TMA descriptors and the launch
// sequence of one block forward.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "gqa_attn.h"
#include "launch.h"
#include "pair_sched.h"
#include "params.h"

using namespace gqa;

struct gqa_ctx {
  int device = -1;
  int num_sms = 0;
  int pair_clusters = 0;  // co-resident 2-CTA clusters of the pair GEMM
  // kv groups of this context: 8 for the whole block, G < 8 for a head shard (4 G query
  // heads); q_cols = 512 G query features, kv_cols = 128 G key (and value) features
  int n_kv = 8;
  int q_cols() const { return 512 * n_kv; }
  int kv_cols() const { return 128 * n_kv; }
  int qkv_rows() const { return 768 * n_kv; }
  // weights, k-block-major: W_t[kb][row][64]
  __nv_bfloat16* w_qkv = nullptr;  // qkv_rows x 4096: W_Q rows 0..q_cols-1, then W_K, then W_V
  __nv_bfloat16* w_o = nullptr;    // 4096 rows x q_cols (the columns of W_O that belong to its heads)
  // residual form: W_QKV * diag(attention_norm weight), same layout (attn_set_norm)
  __nv_bfloat16* w_qkv_norm = nullptr;
  float norm_eps = 0.f;
  int* status = nullptr;           // device status word (kDevErr* bits)
  int* counters = nullptr;         // arrival counters of the decode split merge (kCounterInts)
  uint8_t* ws = nullptr;           // workspace
  size_t ws_bytes = 0;
  const void* last_q = nullptr;
  const void* last_h = nullptr;
  // per-kernel device timing
  bool profiling = false;
  std::vector<cudaEvent_t> ev;        // 2 per recorded launch
  std::vector<int> ev_kind;           // kind of each recorded launch
  size_t ev_used = 0;                 // launches recorded so far
  int fault_kind = -1;                // test hook armed by attn_debug_inject_timeout
};

namespace {
thread_local int g_last_cuda_error = 0;
}  // namespace

void gqa::set_last_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

namespace {

gqa_status cuda_fail(cudaError_t e) {
  set_last_cuda_error(e);
  return GQA_ERR_CUDA;
}

#define GQA_CUDA(call)                          \
  do {                                          \
    cudaError_t e_ = (call);                    \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr long long kMaxTokens = 262144;
constexpr long long kMaxSMax = 1048576;
constexpr int kSkinnyMaxTokens = 64;     // at or below: swap-AB split-K projections
constexpr int kDecodeMaxBatch = 1024;
// Arrival counters of the decode split merge, one per (sequence, kv group, position group).
constexpr int kCounterInts = kDecodeMaxBatch * 8;
// Prefills of at most this many tokens per sequence run the decode attention kernel with
// kShortPos positions per CTA instead of the flash kernel (whose 128-row query tiles they
// would fill to an eighth at most) — unless the cache is long and the flash grid fills the
// GPU: each position group of the short kernel reads the keys again, and its mma.sync rows
// cost more per key than the flash kernel's tcgen05 tiles.  Measured block steps at T = 16:
// B = 1 is faster on the short kernel up to 4096 cached keys (61 vs 76 us); B = 2 ties at
// 1024 keys and loses at 4096 (81 vs 77 us); B = 4 wins up to 256 keys and loses from 512
// (54 vs 44 us; at 4096 97 vs 79 us).
constexpr int kShortMaxT = 16;
constexpr int kShortPos = 4;
constexpr int kShortAlwaysKeys = 256;     // at most this many keys: the short kernel
constexpr int kFlashMinCtas = 32;         // longer caches: flash once its grid has this many CTAs

// ------------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor map with 128-byte swizzle; dims[0] innermost; strides in bytes for dims 1..
bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
              const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, s, b, e,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// GEMM operands are addressed as (column c < 64, row r, k block kb) with box 64 x box_rows x 1.
// Row-major [rows, k_cols] activation: element (c, r, kb) at r*2*k_cols + kb*128 + 2c bytes.
bool map_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t k_cols, uint32_t box_rows) {
  const uint64_t dims[3] = {64, rows, k_cols / 64};
  const uint64_t strides[2] = {k_cols * 2, 64 * 2};
  const uint32_t box[3] = {64, box_rows, 1};
  return make_map(m, base, 3, dims, strides, box);
}

// k-block-major weight copy W_t[kb][row][64] (kbs k blocks): element (c, r, kb) at
// (kb*rows + r)*128 + 2c bytes, so one box of consecutive rows is one contiguous read.
bool map_weight_tiled(CUtensorMap* m, const void* base, uint64_t rows, uint64_t kbs, uint32_t box_rows) {
  const uint64_t dims[3] = {64, rows, kbs};
  const uint64_t strides[2] = {64 * 2, rows * 64 * 2};
  const uint32_t box[3] = {64, box_rows, 1};
  return make_map(m, base, 3, dims, strides, box);
}

// Copy a row-major [rows, 64 kbs] bf16 weight into rows row0.. of a k-block-major copy with
// total_rows rows (kbs strided 2-D copies, at context creation only).
cudaError_t copy_weight_tiled(void* dst, const void* src, size_t rows, size_t row0, size_t total_rows,
                              size_t kbs, cudaStream_t s) {
  for (size_t kb = 0; kb < kbs; ++kb) {
    uint8_t* d = static_cast<uint8_t*>(dst) + (kb * total_rows + row0) * 128;
    const uint8_t* from = static_cast<const uint8_t*>(src) + kb * 128;
    cudaError_t e = cudaMemcpy2DAsync(d, 128, from, kbs * 128, 128, rows, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// KV cache [B, S_max, n_kv, 128] bf16 seen as (d, g, s < kv_len, b); box 64 d x key_rows.
bool map_cache(CUtensorMap* m, const void* base, int B, int S_max, int n_kv, int kv_len, uint32_t key_rows) {
  const uint64_t dims[4] = {128, static_cast<uint64_t>(n_kv), static_cast<uint64_t>(kv_len), static_cast<uint64_t>(B)};
  const uint64_t strides[3] = {128 * 2, static_cast<uint64_t>(n_kv) * 128 * 2,
                               static_cast<uint64_t>(S_max) * n_kv * 128 * 2};
  const uint32_t box[4] = {64, 1, key_rows, 1};
  return make_map(m, base, 4, dims, strides, box);
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------------ workspace
struct WsLayout {
  size_t q_off, h_off, dec_o_off, dec_ml_off, rstd_off, total;
};

// Few-token projections (at most kSkinnyMaxTokens tokens): k splits per 128-feature tile.
struct SkinnyPlan {
  int splits_qkv, splits_o;
};

SkinnyPlan skinny_plan(int n_tok) {
  // k splits = cluster size.  A CTA's main loop is bound by the tensor core's cost per
  // 128 x N x 16 instruction (~110 cycles for N <= 64), so more, shorter k ranges per weight
  // tile finish sooner where two CTAs fit on an SM: Q/K/V in 4 splits (48 x 4 = 192 CTAs, two
  // per SM); W_O in 8 splits at most 32 tokens (256 CTAs, two per SM), else 4 with one CTA per
  // SM and a deeper ring.  Measured against 2 / 4 splits with one CTA per SM: 16 tokens
  // 33.7 -> 31.3 us per block step; 64 tokens (decode B=64) Q/K/V 22.4 -> 21.2 us, while W_O
  // in 8 splits went 14.5 -> 15.8 us, so it keeps 4 there.
  SkinnyPlan s;
  s.splits_qkv = 4;
  s.splits_o = n_tok <= 32 ? 8 : 4;
  return s;
}

struct DecodePlan {
  int n_splits, tiles_per_split;
};

// Key splits of the decode attention kernel for `units` (sequence, position group) pairs of
// n_kv groups each, at ctas_per_sm resident CTAs per SM (2 with one position per CTA, 1 with
// four: the larger reduction scratch).
DecodePlan decode_plan(int units_b, int n_kv, int kv_len, int num_sms, int ctas_per_sm = 2) {
  const int n_tiles = (kv_len + kDecTileKeys - 1) / kDecTileKeys;
  // aim for ~6-7 waves, at least 4 tiles (256 keys) per split (B=64 at 4096 keys: 4 splits of
  // 16 tiles measured faster than 5, 8 or 10)
  const long long units = static_cast<long long>(units_b) * n_kv;
  const long long target = 13LL * num_sms * ctas_per_sm / 2;
  int splits = static_cast<int>(std::max(1LL, (target + units - 1) / units));
  splits = std::min(splits, std::max(1, n_tiles / 4));
  DecodePlan d;
  d.tiles_per_split = (n_tiles + splits - 1) / splits;
  d.n_splits = (n_tiles + d.tiles_per_split - 1) / d.tiles_per_split;
  return d;
}

// dec_rows: rows of decode partials per (kv group, split): B x position groups x rows per CTA.
WsLayout ws_layout(long long n_tok, int n_kv, const SkinnyPlan* sk, const DecodePlan* dp, long long dec_rows) {
  WsLayout w{};
  size_t off = 0;
  const size_t q_cols = static_cast<size_t>(n_kv) * 512;
  w.q_off = off;
  off = round_up(off + static_cast<size_t>(n_tok) * q_cols * 2, 256);
  w.h_off = off;
  off = round_up(off + static_cast<size_t>(n_tok) * q_cols * 2, 256);
  w.dec_o_off = off;
  w.dec_ml_off = off;
  if (dp) {
    const size_t rows = static_cast<size_t>(dec_rows) * n_kv * dp->n_splits;
    off = round_up(off + rows * 128 * 4, 256);
    w.dec_ml_off = off;
    off = round_up(off + rows * 2 * 4, 256);
  }
  w.rstd_off = off;  // residual form: 1 / rms per token row
  off = round_up(off + static_cast<size_t>(n_tok) * 4, 256);
  w.total = off;
  return w;
}

gqa_status ensure_ws(gqa_ctx* c, size_t bytes, cudaStream_t s) {
  if (bytes <= c->ws_bytes) return GQA_OK;
  GQA_CUDA(cudaStreamSynchronize(s));
  if (c->ws) GQA_CUDA(cudaFree(c->ws));
  c->ws = nullptr;
  c->ws_bytes = 0;
  const size_t want = round_up(bytes, 1 << 20);
  if (cudaMalloc(&c->ws, want) != cudaSuccess) {
    cudaGetLastError();
    c->ws = nullptr;
    return GQA_ERR_OOM;
  }
  c->ws_bytes = want;
  return GQA_OK;
}

gqa_status check_device(gqa_ctx* c) {
  int dev = -1;
  GQA_CUDA(cudaGetDevice(&dev));
  if (dev != c->device) return GQA_ERR_DEVICE;
  return GQA_OK;
}

// One-shot test hook: 1 if the next launch of `kind` should skip its first unit's loads.
int take_fault(gqa_ctx* c, int kind) {
  if (c->fault_kind != kind) return 0;
  c->fault_kind = -1;
  return 1;
}

constexpr size_t kMaxProfiledLaunches = 65536;

// RAII bracket of one kernel launch with two events when profiling is on.
// NVTX range names of the kernel kinds (host-side ranges around each launch; without a tool
// attached an NVTX call returns at once).
const char* const kKindNames[GQA_KERNEL_KINDS] = {"gqa.qkv_gemm", "gqa.qkv_splitk", "gqa.flash_prefill",
                                                  "gqa.decode_attn", "gqa.out_gemm", "gqa.out_splitk",
                                                  "gqa.rms_norm"};

// RAII NVTX range around one entry point's host work (its launches nest inside it).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
};

struct ProfScope {
  gqa_ctx* c;
  cudaStream_t s;
  bool on;
  ProfScope(gqa_ctx* c_, int kind, cudaStream_t s_) : c(c_), s(s_), on(false) {
    nvtxRangePushA(kind >= 0 && kind < GQA_KERNEL_KINDS ? kKindNames[kind] : "gqa.kernel");
    if (c->profiling && c->ev_used < kMaxProfiledLaunches) {
      if (c->ev.size() < 2 * (c->ev_used + 1)) {
        cudaEvent_t a, b;
        if (cudaEventCreate(&a) != cudaSuccess) return;
        if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return; }
        c->ev.push_back(a);
        c->ev.push_back(b);
        c->ev_kind.push_back(kind);
      }
      c->ev_kind[c->ev_used] = kind;
      on = cudaEventRecord(c->ev[2 * c->ev_used], s) == cudaSuccess;
    }
  }
  ~ProfScope() {
    if (on) {
      cudaEventRecord(c->ev[2 * c->ev_used + 1], s);
      ++c->ev_used;
    }
    nvtxRangePop();
  }
};

const float kScaleLog2 = static_cast<float>(1.4426950408889634 / std::sqrt(128.0));

// Q/K/V projection + RoPE + cache write for n_tok tokens laid out [B, T] (steps 1-5).
gqa_status run_qkv(gqa_ctx* c, const void* x, int n_tok, int T, const float* R, void* ck, void* cv,
                   int S_max, int start_pos, void* q_out, const WsLayout& w, const SkinnyPlan* sk,
                   const float* row_scale, cudaStream_t s) {
  GemmParams p{};
  // residual form: the folded weights, each token row scaled by its 1 / rms
  const __nv_bfloat16* wqkv = row_scale ? c->w_qkv_norm : c->w_qkv;
  p.row_scale = row_scale;
  p.T = T;
  p.S_max = S_max;
  p.start_pos = start_pos;
  p.status = c->status;
  p.num_kb = 64;
  p.q_cols = c->q_cols();
  p.kv_cols = c->kv_cols();
  const int rows = c->qkv_rows();
  CUtensorMap ta, tb;
  if (sk) {
    if (!map_weight_tiled(&ta, wqkv, rows, 64, 128) || !map_rows(&tb, x, n_tok, 4096, splitk_token_tile(n_tok)))
      return cuda_fail(cudaErrorInvalidValue);
    p.M = rows;
    p.N = n_tok;
    p.splits = sk->splits_qkv;
    p.n_tiles = 1;
    p.m_tiles = rows / 128;
    p.fin0 = q_out;
    p.fin1 = ck;
    p.fin2 = cv;
    p.R = R;
    p.fault = take_fault(c, GQA_KERNEL_QKV_SPLITK);
    { ProfScope ps(c, GQA_KERNEL_QKV_SPLITK, s); GQA_CUDA(launch_gemm_splitk_qkv(ta, tb, p, s)); }
  } else {
    // CTA pairs, 256x256 tiles: each CTA loads 128-row boxes of x and of W_QKV
    if (!map_rows(&ta, x, n_tok, 4096, 128) || !map_weight_tiled(&tb, wqkv, rows, 64, 128))
      return cuda_fail(cudaErrorInvalidValue);
    p.M = n_tok;
    p.N = rows;
    p.splits = 1;
    p.n_tiles = rows / 256;
    p.m_tiles = (n_tok + 255) / 256;
    p.out0 = q_out;
    p.out1 = ck;
    p.out2 = cv;
    p.R = R;
    const int grid = plan_pair_grid(p, c->pair_clusters);
    CUtensorMap tbt = tb;  // boxes of tail_w / 2 rows for the pieces of a partial last round
    if (p.tail_w && !map_weight_tiled(&tbt, wqkv, rows, 64, p.tail_w / 2)) return cuda_fail(cudaErrorInvalidValue);
    p.fault = take_fault(c, GQA_KERNEL_QKV_GEMM);
    { ProfScope ps(c, GQA_KERNEL_QKV_GEMM, s); GQA_CUDA(launch_gemm_qkv_rope(ta, tb, tbt, p, grid, s)); }
  }
  return GQA_OK;
}

// Delta = H W_O^T (step 14).
gqa_status run_out(gqa_ctx* c, const void* h, int n_tok, float* delta, const WsLayout& w,
                   const SkinnyPlan* sk, const void* residual, cudaStream_t s) {
  GemmParams p{};
  p.residual = residual;  // residual form: x + Delta
  p.status = c->status;
  const int kc = c->q_cols();  // the contraction runs over this context's heads only
  p.num_kb = kc / 64;
  CUtensorMap ta, tb;
  if (sk) {
    if (!map_weight_tiled(&ta, c->w_o, 4096, p.num_kb, 128) || !map_rows(&tb, h, n_tok, kc, splitk_token_tile(n_tok)))
      return cuda_fail(cudaErrorInvalidValue);
    p.M = 4096;
    p.N = n_tok;
    p.splits = sk->splits_o;
    p.n_tiles = 1;
    p.m_tiles = 32;
    p.fin0 = delta;
    p.fault = take_fault(c, GQA_KERNEL_OUT_SPLITK);
    { ProfScope ps(c, GQA_KERNEL_OUT_SPLITK, s); GQA_CUDA(launch_gemm_splitk_out(ta, tb, p, s)); }
  } else {
    if (!map_rows(&ta, h, n_tok, kc, 128) || !map_weight_tiled(&tb, c->w_o, 4096, p.num_kb, 128))
      return cuda_fail(cudaErrorInvalidValue);
    p.M = n_tok;
    p.N = 4096;
    p.splits = 1;
    p.n_tiles = 16;
    p.m_tiles = (n_tok + 255) / 256;
    p.out0 = delta;
    p.ldo = 4096;
    const int grid = plan_pair_grid(p, c->pair_clusters);
    CUtensorMap tbt = tb;
    if (p.tail_w && !map_weight_tiled(&tbt, c->w_o, 4096, p.num_kb, p.tail_w / 2))
      return cuda_fail(cudaErrorInvalidValue);
    p.fault = take_fault(c, GQA_KERNEL_OUT_GEMM);
    { ProfScope ps(c, GQA_KERNEL_OUT_GEMM, s); GQA_CUDA(launch_gemm_store_f32(ta, tb, tbt, p, grid, s)); }
  }
  return GQA_OK;
}

}  // namespace

extern "C" {

const char* attn_strerror(gqa_status st) {
  switch (st) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument (null pointer, null context or bad flag)";
    case GQA_ERR_SHAPE: return "shape out of range (B, T, S_max or start_pos)";
    case GQA_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case GQA_ERR_CUDA: return "CUDA runtime error (see attn_last_cuda_error)";
    case GQA_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case GQA_ERR_OOM: return "workspace allocation failed";
    case GQA_ERR_DEVICE: return "current device is not the context's sm_103 GPU";
  }
  return "unknown status";
}

int attn_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"

namespace {

// A context over n_kv kv groups (4 n_kv query heads) from row-major weights: wq [512 n_kv,
// 4096], wk / wv [128 n_kv, 4096], wo [4096, 512 n_kv].
gqa_status create_impl(const void* wq, const void* wk, const void* wv, const void* wo, int n_kv,
                       cudaStream_t s, gqa_ctx** out) {
  if (!out) return GQA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!wq || !wk || !wv || !wo) return GQA_ERR_INVALID_ARG;
  if (n_kv < 1 || n_kv > 8) return GQA_ERR_SHAPE;
  if (!aligned16(wq) || !aligned16(wk) || !aligned16(wv) || !aligned16(wo)) return GQA_ERR_ALIGN;
  int dev = -1;
  GQA_CUDA(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  GQA_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3) return GQA_ERR_DEVICE;
  if (!encode_fn()) return cuda_fail(cudaErrorNotSupported);
  GQA_CUDA(configure_kernels());

  gqa_ctx* c = new gqa_ctx();
  c->device = dev;
  c->n_kv = n_kv;
  c->num_sms = prop.multiProcessorCount;
  c->pair_clusters = gemm_pair_max_clusters();
  if (c->pair_clusters <= 0) c->pair_clusters = prop.multiProcessorCount / 2;
  auto fail = [&](gqa_status st) {
    attn_destroy(c);
    return st;
  };
  const size_t rows = c->qkv_rows(), qc = c->q_cols(), kvc = c->kv_cols();
  if (cudaMalloc(&c->w_qkv, rows * 4096 * 2) != cudaSuccess || cudaMalloc(&c->w_o, 4096 * qc * 2) != cudaSuccess ||
      cudaMalloc(&c->status, sizeof(int)) != cudaSuccess ||
      cudaMalloc(&c->counters, kCounterInts * sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return fail(GQA_ERR_OOM);
  }
  cudaError_t e = cudaMemsetAsync(c->status, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->counters, 0, kCounterInts * sizeof(int), s);
  // k-block-major copies: W_Q rows 0..qc-1, W_K qc..qc+kvc-1, W_V qc+kvc.. of W_QKV; W_O
  if (e == cudaSuccess) e = copy_weight_tiled(c->w_qkv, wq, qc, 0, rows, 64, s);
  if (e == cudaSuccess) e = copy_weight_tiled(c->w_qkv, wk, kvc, qc, rows, 64, s);
  if (e == cudaSuccess) e = copy_weight_tiled(c->w_qkv, wv, kvc, qc + kvc, rows, 64, s);
  if (e == cudaSuccess) e = copy_weight_tiled(c->w_o, wo, 4096, 0, 4096, qc / 64, s);
  if (e != cudaSuccess) return fail(cuda_fail(e));
  *out = c;
  return GQA_OK;
}

}  // namespace

extern "C" {

gqa_status attn_create(const void* wq, const void* wk, const void* wv, const void* wo, gqa_stream_t stream,
                       gqa_ctx** out) {
  return create_impl(wq, wk, wv, wo, 8, reinterpret_cast<cudaStream_t>(stream), out);
}

gqa_status attn_create_shard(const void* wq_shard, const void* wk_shard, const void* wv_shard, const void* wo_shard,
                             int n_kv_local, gqa_stream_t stream, gqa_ctx** out) {
  return create_impl(wq_shard, wk_shard, wv_shard, wo_shard, n_kv_local, reinterpret_cast<cudaStream_t>(stream),
                     out);
}

}  // extern "C"

namespace {

// 1 / rms of each of the n_tok token rows of x (residual form), into the workspace.
gqa_status run_rms(gqa_ctx* c, const void* x, int n_tok, const WsLayout& w, cudaStream_t s) {
  float* r = reinterpret_cast<float*>(c->ws + w.rstd_off);
  { ProfScope ps(c, GQA_KERNEL_RMS_NORM, s); GQA_CUDA(launch_rms_rstd(x, n_tok, c->norm_eps, r, s)); }
  return GQA_OK;
}

// The block (residual == false: out = Delta of x) or its residual form (out = x +
// Delta(attention_norm(x))).
gqa_status prefill_impl(gqa_ctx* c, const void* x, int B, int T, const float* R, int causal, void* cache_k,
                        void* cache_v, int S_max, int start_pos, float* delta, bool residual, cudaStream_t s) {
  if (!c || !x || !R || !cache_k || !cache_v || !delta) return GQA_ERR_INVALID_ARG;
  if (B < 1 || T < 1 || start_pos < 0 || S_max < 1 || S_max > kMaxSMax) return GQA_ERR_SHAPE;
  if (static_cast<long long>(start_pos) + T > S_max) return GQA_ERR_SHAPE;
  if (static_cast<long long>(B) * T > kMaxTokens) return GQA_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(R) || !aligned16(cache_k) || !aligned16(cache_v) || !aligned16(delta))
    return GQA_ERR_ALIGN;
  if (residual && !c->w_qkv_norm) return GQA_ERR_INVALID_ARG;  // attn_set_norm not called (never on a shard)
  gqa_status st = check_device(c);
  if (st != GQA_OK) return st;

  const int n_tok = B * T;
  const int G = c->n_kv;
  const int kv_len = start_pos + T;
  SkinnyPlan sk_v = skinny_plan(n_tok);
  const SkinnyPlan* sk = n_tok <= kSkinnyMaxTokens ? &sk_v : nullptr;
  // few positions per sequence: the decode attention kernel, 4 positions per CTA
  const int n_pg = (T + kShortPos - 1) / kShortPos;
  const bool short_path = T <= kShortMaxT && static_cast<long long>(B) * G * n_pg <= kCounterInts &&
                          (kv_len <= kShortAlwaysKeys || 2LL * G * B < kFlashMinCtas);
  const DecodePlan dp = decode_plan(B * n_pg, G, kv_len, c->num_sms, 1);
  const WsLayout w = short_path ? ws_layout(n_tok, G, sk, &dp, static_cast<long long>(B) * n_pg * 4 * kShortPos)
                                : ws_layout(n_tok, G, sk, nullptr, 0);
  st = ensure_ws(c, w.total, s);
  if (st != GQA_OK) return st;
  void* q_r = c->ws + w.q_off;
  void* h = c->ws + w.h_off;
  c->last_q = q_r;
  c->last_h = h;

  const float* row_scale = nullptr;
  if (residual) {
    if ((st = run_rms(c, x, n_tok, w, s)) != GQA_OK) return st;
    row_scale = reinterpret_cast<const float*>(c->ws + w.rstd_off);
  }
  st = run_qkv(c, x, n_tok, T, R, cache_k, cache_v, S_max, start_pos, q_r, w, sk, row_scale, s);
  if (st != GQA_OK) return st;

  if (short_path) {
    // steps 6-13 for T <= 16 positions: query t sees keys 0 .. start_pos + t (causal) or all
    CUtensorMap tk, tv;
    if (!map_cache(&tk, cache_k, B, S_max, G, kv_len, kDecTileKeys) ||
        !map_cache(&tv, cache_v, B, S_max, G, kv_len, kDecTileKeys))
      return cuda_fail(cudaErrorInvalidValue);
    DecodeParams p{};
    p.B = B;
    p.n_kv = G;
    p.kv_len = kv_len;
    p.n_splits = dp.n_splits;
    p.tiles_per_split = dp.tiles_per_split;
    p.T = T;
    p.q_start = start_pos;
    p.causal = causal ? 1 : 0;
    p.n_pg = n_pg;
    p.q = q_r;
    p.part_o = reinterpret_cast<float*>(c->ws + w.dec_o_off);
    p.part_ml = reinterpret_cast<float*>(c->ws + w.dec_ml_off);
    p.H = h;
    p.status = c->status;
    p.scale_log2 = kScaleLog2;
    p.counters = c->counters;
    p.fault = take_fault(c, GQA_KERNEL_DECODE_ATTN);
    {
      ProfScope ps(c, GQA_KERNEL_DECODE_ATTN, s);
      GQA_CUDA(launch_short_attn(tk, tv, p, dim3(dp.n_splits, G, B * n_pg), s));
    }
    return run_out(c, h, n_tok, delta, w, sk, residual ? x : nullptr, s);
  }

  // steps 6-13: causal GQA flash attention over keys 0 .. start_pos+T-1
  CUtensorMap tq, tk, tv, th;
  {
    // Q_r (read) and H (written) are both [B, T, 512 G] bf16, addressed in 64 x 128 boxes
    const uint64_t qc = c->q_cols();
    const uint64_t dims[3] = {qc, static_cast<uint64_t>(T), static_cast<uint64_t>(B)};
    const uint64_t strides[2] = {qc * 2, static_cast<uint64_t>(T) * qc * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_map(&tq, q_r, 3, dims, strides, box) || !make_map(&th, h, 3, dims, strides, box) ||
        !map_cache(&tk, cache_k, B, S_max, G, kv_len, 128) ||
        !map_cache(&tv, cache_v, B, S_max, G, kv_len, 128))
      return cuda_fail(cudaErrorInvalidValue);
  }
  FlashParams fp{};
  fp.B = B;
  fp.T = T;
  fp.S_max = S_max;
  fp.start_pos = start_pos;
  fp.causal = causal ? 1 : 0;
  fp.n_kv = G;
  fp.n_qtiles = (T + 127) / 128;
  fp.status = c->status;
  fp.scale_log2 = kScaleLog2;
  fp.fault = take_fault(c, GQA_KERNEL_FLASH_PREFILL);
  // Scheduling bands: all (sequence, kv group) pairs at once while their K/V (kv_len x 512 B
  // each) total at most 64 MB; otherwise the largest count of one sequence's G groups, halved
  // while it divides G, whose K/V fit in 32 MB, so the CTAs resident together reuse K/V tiles
  // through L2.
  {
    const long long kv_bytes = static_cast<long long>(kv_len) * 512;
    int gpb = G * B;
    if (kv_bytes * gpb > (64LL << 20)) {
      gpb = G;
      while (gpb > 1 && (gpb & 1) == 0 && kv_bytes * gpb > (32LL << 20)) gpb >>= 1;
    }
    fp.groups_per_band = gpb;
  }
  { ProfScope ps(c, GQA_KERNEL_FLASH_PREFILL, s); GQA_CUDA(launch_flash_prefill(tq, tk, tv, th, fp, dim3(B * 2 * G * fp.n_qtiles), s)); }

  return run_out(c, h, n_tok, delta, w, sk, residual ? x : nullptr, s);
}

gqa_status decode_impl(gqa_ctx* c, const void* x, int B, int start_pos, const float* R_row, void* cache_k,
                       void* cache_v, int S_max, float* delta, bool residual, cudaStream_t s) {
  if (!c || !x || !R_row || !cache_k || !cache_v || !delta) return GQA_ERR_INVALID_ARG;
  if (B < 1 || B > kDecodeMaxBatch || start_pos < 0 || S_max < 1 || S_max > kMaxSMax || start_pos >= S_max)
    return GQA_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(R_row) || !aligned16(cache_k) || !aligned16(cache_v) || !aligned16(delta))
    return GQA_ERR_ALIGN;
  if (residual && !c->w_qkv_norm) return GQA_ERR_INVALID_ARG;  // attn_set_norm not called (never on a shard)
  gqa_status st = check_device(c);
  if (st != GQA_OK) return st;

  const int kv_len = start_pos + 1;
  const int G = c->n_kv;
  SkinnyPlan sk_v = skinny_plan(B);
  const SkinnyPlan* sk = B <= kSkinnyMaxTokens ? &sk_v : nullptr;
  const DecodePlan dp = decode_plan(B, G, kv_len, c->num_sms);
  const WsLayout w = ws_layout(B, G, sk, &dp, static_cast<long long>(B) * 4);
  st = ensure_ws(c, w.total, s);
  if (st != GQA_OK) return st;
  void* q_r = c->ws + w.q_off;
  void* h = c->ws + w.h_off;
  c->last_q = q_r;
  c->last_h = h;

  // steps 1-5 for the new token of each sequence (T = 1, position start_pos)
  const float* row_scale = nullptr;
  if (residual) {
    if ((st = run_rms(c, x, B, w, s)) != GQA_OK) return st;
    row_scale = reinterpret_cast<const float*>(c->ws + w.rstd_off);
  }
  st = run_qkv(c, x, B, 1, R_row, cache_k, cache_v, S_max, start_pos, q_r, w, sk, row_scale, s);
  if (st != GQA_OK) return st;

  // steps 6-13 against the cache (no mask: every key 0..start_pos is visible)
  CUtensorMap tk, tv;
  if (!map_cache(&tk, cache_k, B, S_max, G, kv_len, kDecTileKeys) ||
      !map_cache(&tv, cache_v, B, S_max, G, kv_len, kDecTileKeys))
    return cuda_fail(cudaErrorInvalidValue);
  DecodeParams p{};
  p.B = B;
  p.n_kv = G;
  p.kv_len = kv_len;
  p.n_splits = dp.n_splits;
  p.tiles_per_split = dp.tiles_per_split;
  p.T = 1;
  p.q_start = start_pos;
  p.causal = 0;  // the new position sees the whole cache
  p.n_pg = 1;
  p.q = q_r;
  p.part_o = reinterpret_cast<float*>(c->ws + w.dec_o_off);
  p.part_ml = reinterpret_cast<float*>(c->ws + w.dec_ml_off);
  p.H = h;
  p.status = c->status;
  p.scale_log2 = kScaleLog2;
  p.counters = c->counters;  // the last split of each (b, g) merges
  p.fault = take_fault(c, GQA_KERNEL_DECODE_ATTN);
  { ProfScope ps(c, GQA_KERNEL_DECODE_ATTN, s); GQA_CUDA(launch_decode_attn(tk, tv, p, dim3(dp.n_splits, G, B), s)); }

  // step 14
  return run_out(c, h, B, delta, w, sk, residual ? x : nullptr, s);
}

}  // namespace

extern "C" {

gqa_status attn_prefill(gqa_ctx* c, const void* x, int B, int T, const float* R, int causal, void* cache_k,
                        void* cache_v, int S_max, int start_pos, float* delta, gqa_stream_t stream) {
  CallRange range("gqa.attn_prefill");
  return prefill_impl(c, x, B, T, R, causal, cache_k, cache_v, S_max, start_pos, delta, false,
                      reinterpret_cast<cudaStream_t>(stream));
}

gqa_status attn_prefill_residual(gqa_ctx* c, const void* x, int B, int T, const float* R, int causal,
                                 void* cache_k, void* cache_v, int S_max, int start_pos, float* h_out,
                                 gqa_stream_t stream) {
  CallRange range("gqa.attn_prefill_residual");
  return prefill_impl(c, x, B, T, R, causal, cache_k, cache_v, S_max, start_pos, h_out, true,
                      reinterpret_cast<cudaStream_t>(stream));
}

gqa_status attn_decode(gqa_ctx* c, const void* x, int B, int start_pos, const float* R_row, void* cache_k,
                       void* cache_v, int S_max, float* delta, gqa_stream_t stream) {
  CallRange range("gqa.attn_decode");
  return decode_impl(c, x, B, start_pos, R_row, cache_k, cache_v, S_max, delta, false,
                     reinterpret_cast<cudaStream_t>(stream));
}

gqa_status attn_decode_residual(gqa_ctx* c, const void* x, int B, int start_pos, const float* R_row,
                                void* cache_k, void* cache_v, int S_max, float* h_out, gqa_stream_t stream) {
  CallRange range("gqa.attn_decode_residual");
  return decode_impl(c, x, B, start_pos, R_row, cache_k, cache_v, S_max, h_out, true,
                     reinterpret_cast<cudaStream_t>(stream));
}

gqa_status attn_set_norm(gqa_ctx* c, const void* norm_w, float eps, gqa_stream_t stream) {
  if (!c || !norm_w || !(eps > 0.f) || !std::isfinite(eps)) return GQA_ERR_INVALID_ARG;
  if (!aligned16(norm_w)) return GQA_ERR_ALIGN;
  // the residual form adds x once, after the whole sum over heads: not on a head shard
  if (c->n_kv != 8) return GQA_ERR_INVALID_ARG;
  gqa_status st = check_device(c);
  if (st != GQA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!c->w_qkv_norm && cudaMalloc(&c->w_qkv_norm, size_t(6144) * 4096 * 2) != cudaSuccess) {
    cudaGetLastError();
    c->w_qkv_norm = nullptr;
    return GQA_ERR_OOM;
  }
  GQA_CUDA(launch_fold_norm_weight(c->w_qkv, norm_w, 6144, c->w_qkv_norm, s));
  c->norm_eps = eps;
  return GQA_OK;
}

gqa_status attn_sync_status(gqa_ctx* c, gqa_stream_t stream) {
  if (!c) return GQA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GQA_CUDA(cudaStreamSynchronize(s));
  int v = 0;
  GQA_CUDA(cudaMemcpy(&v, c->status, sizeof(int), cudaMemcpyDeviceToHost));
  if (v != 0) {
    // an aborted kernel may have left arrival counters mid-count
    GQA_CUDA(cudaMemset(c->counters, 0, kCounterInts * sizeof(int)));
    GQA_CUDA(cudaMemset(c->status, 0, sizeof(int)));
    if (v & kDevErrTimeout) return GQA_ERR_TIMEOUT;
  }
  return GQA_OK;
}

gqa_status attn_debug_buffers(gqa_ctx* c, const void** q_r, const void** h) {
  if (!c) return GQA_ERR_INVALID_ARG;
  if (q_r) *q_r = c->last_q;
  if (h) *h = c->last_h;
  return GQA_OK;
}

gqa_status attn_debug_inject_timeout(gqa_ctx* c, int kind) {
  if (!c) return GQA_ERR_INVALID_ARG;
  switch (kind) {
    case GQA_KERNEL_QKV_GEMM:
    case GQA_KERNEL_QKV_SPLITK:
    case GQA_KERNEL_FLASH_PREFILL:
    case GQA_KERNEL_DECODE_ATTN:
    case GQA_KERNEL_OUT_GEMM:
    case GQA_KERNEL_OUT_SPLITK:
      c->fault_kind = kind;
      return GQA_OK;
    default:
      return GQA_ERR_INVALID_ARG;
  }
}

gqa_status attn_debug_pair_schedule(int m_tiles, int n_tiles, int n_pairs, int* full_rounds, int* tail_w,
                                    int* grid_ctas, int* items, int max_items, int* n_items) {
  if (!full_rounds || !tail_w || !grid_ctas || !n_items || (!items && max_items > 0) || m_tiles < 1 ||
      n_tiles < 1 || n_pairs < 1 || max_items < 0)
    return GQA_ERR_INVALID_ARG;
  GemmParams p{};
  p.m_tiles = m_tiles;
  p.n_tiles = n_tiles;
  const int grid = plan_pair_grid(p, n_pairs);
  *full_rounds = p.full_rounds;
  *tail_w = p.tail_w;
  *grid_ctas = grid;
  int n = 0;
  for (int pair = 0; pair < grid / 2; ++pair) {
    int mt, n0, w;
    for (int idx = 0; pair_item(p, pair, grid / 2, idx, mt, n0, w); ++idx, ++n) {
      if (n < max_items) {
        items[4 * n + 0] = pair;
        items[4 * n + 1] = mt;
        items[4 * n + 2] = n0;
        items[4 * n + 3] = w;
      }
    }
  }
  *n_items = n;
  return n > max_items ? GQA_ERR_SHAPE : GQA_OK;
}

gqa_status attn_debug_exp2(const float* a, float* out_fma, float* out_mufu, int n, gqa_stream_t stream) {
  if (!a || !out_fma || !out_mufu || n < 1) return GQA_ERR_INVALID_ARG;
  GQA_CUDA(launch_exp2_compare(a, out_fma, out_mufu, n, reinterpret_cast<cudaStream_t>(stream)));
  return GQA_OK;
}

gqa_status attn_profile_begin(gqa_ctx* c) {
  if (!c) return GQA_ERR_INVALID_ARG;
  c->profiling = true;
  c->ev_used = 0;
  return GQA_OK;
}

gqa_status attn_profile_end(gqa_ctx* c, double* ms_per_kind, int* launches_per_kind, gqa_stream_t stream) {
  if (!c) return GQA_ERR_INVALID_ARG;
  c->profiling = false;
  GQA_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
  double ms[GQA_KERNEL_KINDS] = {0};
  int n[GQA_KERNEL_KINDS] = {0};
  for (size_t i = 0; i < c->ev_used; ++i) {
    float t = 0.f;
    GQA_CUDA(cudaEventElapsedTime(&t, c->ev[2 * i], c->ev[2 * i + 1]));
    const int k = c->ev_kind[i];
    if (k >= 0 && k < GQA_KERNEL_KINDS) {
      ms[k] += t;
      n[k] += 1;
    }
  }
  c->ev_used = 0;
  for (int k = 0; k < GQA_KERNEL_KINDS; ++k) {
    if (ms_per_kind) ms_per_kind[k] = ms[k];
    if (launches_per_kind) launches_per_kind[k] = n[k];
  }
  return GQA_OK;
}

void attn_destroy(gqa_ctx* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
  if (c->w_qkv) cudaFree(c->w_qkv);
  if (c->w_o) cudaFree(c->w_o);
  if (c->w_qkv_norm) cudaFree(c->w_qkv_norm);
  if (c->status) cudaFree(c->status);
  if (c->counters) cudaFree(c->counters);
  if (c->ws) cudaFree(c->ws);
  delete c;
}

}  // extern "C"
