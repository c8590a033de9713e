// decode_noalloc.cu — attn_decode_attention_noalloc: the split-KV decode attention with its
// scratch in a fixed, file-scope device array instead of memory obtained from cudaMalloc.
//
// Who needs it: a caller that hands this library only its inputs and outputs and cannot
// let it allocate device memory — for example a serving engine that has reserved nearly
// all of HBM for its own paged KV cache and routes every allocation through its own pool,
// or a latency-critical decode loop that cannot afford cudaMalloc's implicit device-wide
// synchronisation.  The same split-KV kernels as attn_decode run here; only the location
// of their per-split partial results (and of the time-out status words) changes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "gqa_attn.h"
#include "launch.h"
#include "params.h"

using namespace gqa;

namespace {

// Capacity: at most 2048 (sequence, kv group, key split) units, i.e. B <= 256.
constexpr int kMaxUnits = 2048;
constexpr int kMaxBatch = kMaxUnits / 8;
constexpr size_t kPartOFloats = static_cast<size_t>(kMaxUnits) * 4 * 128;
constexpr size_t kPartMlFloats = static_cast<size_t>(kMaxUnits) * 4 * 2;
// Two int status words, padded to 256 bytes: [0] this call's (cleared by every call),
// [1] sticky (OR of the calls' time-outs since attn_decode_attention_noalloc_status read it).
constexpr size_t kStatusFloats = 64;
constexpr size_t kScratchFloats = kPartOFloats + kPartMlFloats + kStatusFloats;  // ~4.26 MB

// Held by every device that loads this library until the process exits.  All calls share
// it: calls that overlap on the GPU (different streams, or different host threads) race.
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
struct DeviceSetup {
  std::mutex mu;
  std::atomic<bool> ready{false};
  float* scratch = nullptr;  // device address of g_decode_scratch on this device
  int num_sms = 0;
  bool sm103 = false;
};
DeviceSetup g_setup[kMaxDevices];

// One-shot test hook (attn_decode_attention_noalloc_debug_inject_timeout).
std::atomic<int> g_inject_timeout{0};

gqa_status fail_cuda(cudaError_t e) {
  set_last_cuda_error(e);
  return GQA_ERR_CUDA;
}

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

// KV cache [B, S_max, 8, 128] bf16 as (d, kv head, position < kv_len, sequence), 64x64 boxes.
bool map_cache(CUtensorMap* m, const void* base, int B, int S_max, int kv_len) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {128, 8, static_cast<cuuint64_t>(kv_len), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {128 * 2, 1024 * 2, static_cast<cuuint64_t>(S_max) * 1024 * 2};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kDecTileKeys), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Set-up of the current device, done once per device by the first call that succeeds in it
// (a failed attempt is retried by the next call, and its CUDA error is reported each time):
// the scratch array's device address, the SM count and architecture, and the kernels'
// shared-memory opt-in.
gqa_status device_setup(DeviceSetup** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return GQA_ERR_DEVICE;
  DeviceSetup& su = g_setup[dev];
  if (!su.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(su.mu);
    if (!su.ready.load(std::memory_order_relaxed)) {
      int major = 0, minor = 0, sms = 0;
      if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return fail_cuda(e);
      su.sm103 = major == 10 && minor == 3;
      su.num_sms = sms;
      if (su.sm103) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_decode_scratch)) != cudaSuccess) return fail_cuda(e);
        if ((e = configure_kernels()) != cudaSuccess) return fail_cuda(e);
        su.scratch = static_cast<float*>(p);
      }
      su.ready.store(true, std::memory_order_release);
    }
  }
  if (!su.sm103) return GQA_ERR_DEVICE;
  *out = &su;
  return GQA_OK;
}

int* status_words(const DeviceSetup& su) { return reinterpret_cast<int*>(su.scratch + kPartOFloats + kPartMlFloats); }

}  // namespace

extern "C" gqa_status attn_decode_attention_noalloc(const void* q_r, const void* cache_k, const void* cache_v,
                                                    int B, int kv_len, int S_max, void* h,
                                                    gqa_stream_t stream) {
  if (!q_r || !cache_k || !cache_v || !h) return GQA_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxBatch || kv_len < 1 || S_max < 1 || S_max > 1048576 || kv_len > S_max)
    return GQA_ERR_SHAPE;
  if (!aligned16(q_r) || !aligned16(cache_k) || !aligned16(cache_v) || !aligned16(h)) return GQA_ERR_ALIGN;

  DeviceSetup* su = nullptr;
  gqa_status st = device_setup(&su);
  if (st != GQA_OK) return st;
  if (!encode_fn()) return fail_cuda(cudaErrorNotSupported);

  // Key splits: about 16 CTAs per SM in total, at least 4 tiles (256 keys) per split,
  // and never more units than the scratch holds.
  const int n_tiles = (kv_len + kDecTileKeys - 1) / kDecTileKeys;
  const long long units = static_cast<long long>(B) * 8;
  int splits = static_cast<int>(std::max(1LL, (16LL * su->num_sms + units - 1) / units));
  splits = std::min(splits, std::max(1, n_tiles / 4));
  splits = std::min(splits, static_cast<int>(kMaxUnits / units));
  const int tiles_per_split = (n_tiles + splits - 1) / splits;
  splits = (n_tiles + tiles_per_split - 1) / tiles_per_split;

  CUtensorMap tk, tv;
  if (!map_cache(&tk, cache_k, B, S_max, kv_len) || !map_cache(&tv, cache_v, B, S_max, kv_len))
    return fail_cuda(cudaErrorInvalidValue);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* status = status_words(*su);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);  // this call's word starts at zero
  if (e != cudaSuccess) return fail_cuda(e);

  DecodeParams p{};
  p.B = B;
  p.n_kv = 8;
  p.kv_len = kv_len;
  p.n_splits = splits;
  p.tiles_per_split = tiles_per_split;
  p.T = 1;
  p.q_start = kv_len - 1;
  p.causal = 0;  // one position per sequence, seeing the whole cache
  p.n_pg = 1;
  p.q = q_r;
  p.part_o = su->scratch;
  p.part_ml = su->scratch + kPartOFloats;
  p.H = h;
  p.status = status;
  p.status_sticky = status + 1;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / 11.313708498984761);  // log2(e) / sqrt(128)
  p.fault = g_inject_timeout.exchange(0);
  e = launch_decode_attn(tk, tv, p, dim3(splits, 8, B), s);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_decode_combine(p, B, s);
  if (e != cudaSuccess) return fail_cuda(e);
  return GQA_OK;
}

extern "C" gqa_status attn_decode_attention_noalloc_status(gqa_stream_t stream) {
  DeviceSetup* su = nullptr;
  gqa_status st = device_setup(&su);
  if (st != GQA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda(e);
  int* sticky = status_words(*su) + 1;
  int v = 0;
  if ((e = cudaMemcpy(&v, sticky, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return fail_cuda(e);
  if (v != 0) {
    if ((e = cudaMemset(sticky, 0, sizeof(int))) != cudaSuccess) return fail_cuda(e);
    if (v & kDevErrTimeout) return GQA_ERR_TIMEOUT;
  }
  return GQA_OK;
}

extern "C" gqa_status attn_decode_attention_noalloc_debug_inject_timeout(void) {
  g_inject_timeout.store(1);
  return GQA_OK;
}
