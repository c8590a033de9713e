// decode_noalloc.cu — attn_decode_attention_noalloc: the split-KV decode attention with its
// scratch in a fixed, file-scope device array instead of memory obtained from cudaMalloc.
//
// Who needs it: a caller that hands this library only its inputs and outputs and cannot
// let it allocate device memory — for example a serving engine that has reserved nearly
// all of HBM for its own paged KV cache and routes every allocation through its own pool,
// or a latency-critical decode loop that cannot afford cudaMalloc's implicit device-wide
// synchronisation.  The same split-KV kernels as attn_decode run here; only the location
// of their per-split partial results (and of the time-out status word) changes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
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
constexpr size_t kStatusFloats = 64;  // one int status word, padded to 256 bytes
constexpr size_t kScratchFloats = kPartOFloats + kPartMlFloats + kStatusFloats;  // ~4.26 MB

// Held by every device that loads this library until the process exits.  All calls share
// it: calls that overlap on the GPU (different streams, or different host threads) race.
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
struct DeviceSetup {
  std::once_flag once;
  float* scratch = nullptr;  // device address of g_decode_scratch on this device
  cudaError_t err = cudaSuccess;
};
DeviceSetup g_setup[kMaxDevices];

gqa_status fail_cuda(cudaError_t) { return GQA_ERR_CUDA; }

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

}  // namespace

extern "C" gqa_status attn_decode_attention_noalloc(const void* q_r, const void* cache_k, const void* cache_v,
                                                    int B, int kv_len, int S_max, void* h,
                                                    gqa_stream_t stream) {
  if (!q_r || !cache_k || !cache_v || !h) return GQA_ERR_INVALID_ARG;
  if (B < 1 || B > kMaxBatch || kv_len < 1 || S_max < 1 || S_max > 1048576 || kv_len > S_max)
    return GQA_ERR_SHAPE;
  if (!aligned16(q_r) || !aligned16(cache_k) || !aligned16(cache_v) || !aligned16(h)) return GQA_ERR_ALIGN;

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (dev < 0 || dev >= kMaxDevices) return GQA_ERR_DEVICE;
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return fail_cuda(e);
  if (prop.major != 10 || prop.minor != 3) return GQA_ERR_DEVICE;

  // Once per device, with that device current: look up the scratch array's device address
  // and opt the kernels in to their dynamic shared memory.
  DeviceSetup& su = g_setup[dev];
  std::call_once(su.once, [&su] {
    void* p = nullptr;
    su.err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (su.err == cudaSuccess) {
      su.scratch = static_cast<float*>(p);
      su.err = configure_kernels();
    }
  });
  if (su.err != cudaSuccess || !su.scratch) return fail_cuda(su.err != cudaSuccess ? su.err : cudaErrorUnknown);
  if (!encode_fn()) return fail_cuda(cudaErrorNotSupported);

  // Key splits: about 16 CTAs per SM in total, at least 4 tiles (256 keys) per split,
  // and never more units than the scratch holds.
  const int n_tiles = (kv_len + kDecTileKeys - 1) / kDecTileKeys;
  const long long units = static_cast<long long>(B) * 8;
  int splits = static_cast<int>(std::max(1LL, (16LL * prop.multiProcessorCount + units - 1) / units));
  splits = std::min(splits, std::max(1, n_tiles / 4));
  splits = std::min(splits, static_cast<int>(kMaxUnits / units));
  const int tiles_per_split = (n_tiles + splits - 1) / splits;
  splits = (n_tiles + tiles_per_split - 1) / tiles_per_split;

  CUtensorMap tk, tv;
  if (!map_cache(&tk, cache_k, B, S_max, kv_len) || !map_cache(&tv, cache_v, B, S_max, kv_len))
    return fail_cuda(cudaErrorInvalidValue);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* status = reinterpret_cast<int*>(su.scratch + kPartOFloats + kPartMlFloats);
  e = cudaMemsetAsync(status, 0, sizeof(int), s);  // the status word must start at zero
  if (e != cudaSuccess) return fail_cuda(e);

  DecodeParams p{};
  p.B = B;
  p.kv_len = kv_len;
  p.n_splits = splits;
  p.tiles_per_split = tiles_per_split;
  p.q = q_r;
  p.part_o = su.scratch;
  p.part_ml = su.scratch + kPartOFloats;
  p.H = h;
  p.status = status;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / 11.313708498984761);  // log2(e) / sqrt(128)
  e = launch_decode_attn(tk, tv, p, dim3(splits, 8, B), s);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_decode_combine(p, B, s);
  if (e != cudaSuccess) return fail_cuda(e);
  return GQA_OK;
}
