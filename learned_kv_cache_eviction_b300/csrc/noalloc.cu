// noalloc.cu -- dms_decode_attention_noalloc: the decode-attention kernels run
// over caller-owned buffers, with their split-K scratch in a fixed array in
// the library's own device memory instead of memory obtained from cudaMalloc.
//
// Who needs this: callers that must not allocate device memory at the point
// where they decode -- an engine whose memory is fully reserved up front by its
// own pool, code running while the CUDA caching allocator is forbidden to grow,
// or a process that only receives pointers to buffers another component owns.
// Such callers hold the K/V pools and the lengths themselves and pass them in.
//
// The scratch array lives for as long as the library is loaded, on every GPU
// that loads it.  All calls share it: two calls whose kernels overlap on the
// GPU (different streams, or different host threads on one device) race on it
// and must be serialised by the caller.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <utility>

#include "decode.cuh"
#include "dms.h"

namespace {

// Split-K scratch of one call: the device error word, one arrival counter per
// head, and the partial (acc, max, sum) of every (warp, head) segment.  8 MiB.
constexpr size_t kScratchBytes = DMS_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_scratch, per device
std::atomic<bool> g_attr_done[kMaxDevices][2][DMS_MAX_GROUP + 1] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool device_pointer_on(const void* p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

// Once per device, with that device current: look up the device address of the
// scratch array (the host-side name g_scratch is only a stand-in) and zero the
// error word kept at its start.
int scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return DMS_ERR_CUDA;
    }
    if (cudaMemset(p, 0, 256) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      return DMS_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DMS_OK;
}

template <typename... KArgs, typename... Args>
int launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) != cudaSuccess) {
    cudaGetLastError();
    return DMS_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? DMS_OK : DMS_ERR_CUDA;
}

template <int D, int G>
int run(int dev, int num_sms, unsigned char* scratch, const void* k_pool, const void* v_pool, const int32_t* len,
        int NH, int kv_heads, int capacity, const void* q, float* out, float scale, cudaStream_t st) {
  using Sh = dms::DecodeShape<D, G>;
  if ((2 * static_cast<int64_t>(NH) + 1) * 4 > Sh::SMEM) return DMS_ERR_SCRATCH_LIMIT;  // prologue prefix sums, lengths
  // Upper bound of the retained slots: every slot of every head.
  const int64_t smax = static_cast<int64_t>(NH) * capacity;
  const int64_t per_cta = int64_t(dms::kMinSlotsPerWarp) * Sh::NW;
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms, (smax + per_cta - 1) / per_cta)));
  // Scratch layout: [0, 256) error word; head counters; partial acc; partial (max, sum).
  const size_t entries = static_cast<size_t>(grid) * Sh::NW + NH;
  const size_t cnt_off = 256;
  const size_t acc_off = cnt_off + ((static_cast<size_t>(NH) * 4 + 255) / 256) * 256;
  const size_t acc_bytes = entries * G * D * sizeof(float);
  const size_t ml_bytes = entries * Sh::MLS * sizeof(float);
  if (acc_off + acc_bytes + ml_bytes > kScratchBytes) return DMS_ERR_SCRATCH_LIMIT;
  if (dev < kMaxDevices && !g_attr_done[dev][D == 128][G]) {
    if (cudaFuncSetAttribute(dms::decode_kernel<D, G, false, dms::kKvBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM) !=
        cudaSuccess) {
      cudaGetLastError();
      return DMS_ERR_CUDA;
    }
    g_attr_done[dev][D == 128][G] = true;
  }
  dms::DecodeArgs a{};
  a.K = static_cast<const uint4*>(k_pool);
  a.V = static_cast<const uint4*>(v_pool);
  a.len = len;
  a.q = static_cast<const uint16_t*>(q);
  a.out = out;
  a.err = reinterpret_cast<int32_t*>(scratch);
  a.head_cnt = reinterpret_cast<int32_t*>(scratch + cnt_off);
  a.part_acc = reinterpret_cast<float*>(scratch + acc_off);
  a.part_ml = reinterpret_cast<float*>(scratch + acc_off + acc_bytes);
  a.NH = NH;
  a.Hkv = kv_heads;
  a.cap = capacity;
  a.qscale = scale * 1.4426950408889634f;  // log2(e)
  a.Gq = G;
  a.nsplit = 1;
  a.min_tiles = dms::kMinTilesPerWarp;
  a.clamp_len = 1;  // the lengths are the caller's: never trust them to stay within the pools
  // The merge in the decode kernel needs every head counter at zero.  Calls that
  // complete leave them at zero; clearing them here (stream-ordered, no
  // allocation) also recovers from a call that stopped early.
  if (cudaMemsetAsync(a.head_cnt, 0, static_cast<size_t>(NH) * 4, st) != cudaSuccess) {
    cudaGetLastError();
    return DMS_ERR_CUDA;
  }
  return launch_dependent(dms::decode_kernel<D, G, false, dms::kKvBf16>, dim3(grid), dim3(Sh::NW * 32), Sh::SMEM, st, a);
}

template <int D>
int run_d(int G, int dev, int nsm, unsigned char* s, const void* k, const void* v, const int32_t* len, int NH,
          int H, int cap, const void* q, float* out, float scale, cudaStream_t st) {
  switch (G) {
    case 1: return run<D, 1>(dev, nsm, s, k, v, len, NH, H, cap, q, out, scale, st);
    case 2: return run<D, 2>(dev, nsm, s, k, v, len, NH, H, cap, q, out, scale, st);
    case 3: return run<D, 3>(dev, nsm, s, k, v, len, NH, H, cap, q, out, scale, st);
    case 4: return run<D, 4>(dev, nsm, s, k, v, len, NH, H, cap, q, out, scale, st);
    case 5: return run<D, 5>(dev, nsm, s, k, v, len, NH, H, cap, q, out, scale, st);
    case 6: return run<D, 6>(dev, nsm, s, k, v, len, NH, H, cap, q, out, scale, st);
    case 7: return run<D, 7>(dev, nsm, s, k, v, len, NH, H, cap, q, out, scale, st);
    case 8: return run<D, 8>(dev, nsm, s, k, v, len, NH, H, cap, q, out, scale, st);
    default: return DMS_ERR_INVALID_ARG;
  }
}

}  // namespace

extern "C" int dms_decode_attention_noalloc(const void* k_pool, const void* v_pool, const int32_t* len, int batch,
                                            int kv_heads, int capacity, int head_dim, const void* q, float* out,
                                            float scale, int q_heads, void* stream) {
  if (batch < 1 || kv_heads < 1 || capacity < 1 || (head_dim != 64 && head_dim != 128) || q_heads < 1 ||
      q_heads % kv_heads != 0 || q_heads / kv_heads > DMS_MAX_GROUP || !std::isfinite(scale))
    return DMS_ERR_INVALID_ARG;
  const int64_t NH = static_cast<int64_t>(batch) * kv_heads;
  if (NH > DMS_NOALLOC_MAX_HEADS || NH * capacity >= (int64_t(1) << 31)) return DMS_ERR_SCRATCH_LIMIT;
  if (!k_pool || !v_pool || !len || !q || !out || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(q) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(len) & 3u))
    return DMS_ERR_INVALID_ARG;
  int dev = -1, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return DMS_ERR_CUDA;
  }
  if (!device_pointer_on(k_pool, dev) || !device_pointer_on(v_pool, dev) || !device_pointer_on(len, dev) ||
      !device_pointer_on(q, dev) || !device_pointer_on(out, dev))
    return DMS_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int rc = scratch_address(dev, &scratch);
  if (rc != DMS_OK) return rc;
  unsigned char* s = static_cast<unsigned char*>(scratch);
  const int G = q_heads / kv_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return head_dim == 128
             ? run_d<128>(G, dev, nsm, s, k_pool, v_pool, len, static_cast<int>(NH), kv_heads, capacity, q, out,
                          scale, st)
             : run_d<64>(G, dev, nsm, s, k_pool, v_pool, len, static_cast<int>(NH), kv_heads, capacity, q, out,
                         scale, st);
}
