// dms_api.cu -- the C ABI of libdms.so (declared in include/dms.h): cache
// lifetime, argument checks, kernel dispatch.  All compute runs in the
// kernels of append.cuh and decode.cuh; this file only validates, allocates
// at creation time and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>
#include <utility>

#include "append.cuh"
#include "decode.cuh"
#include "dms.h"
#include "prefill.cuh"

struct dms_cache {
  int B, H, cap, D, w, NH;
  int kvf;  // DMS_KV_BF16 or DMS_KV_FP8_E4M3
  int64_t t;
  // The last call that advanced t added exactly one token, so the lengths after
  // t - 1 appends are still in their generation: the next fused step may then
  // start before the previous launch has finished (DecodeArgs::early).
  bool single_prev;
  int device;
  int num_sms;
  dms::CacheView view;
  float* part_acc;
  float* part_ml;
  int32_t* head_cnt;  // [2 NH] arrival counters of (virtual) heads split across warps (zero between calls)
  size_t part_entries;
  // The position in device memory, read by steps replayed from a CUDA graph
  // (dms_step_graph_*).  Valid while t_dev_synced; any call that advances t
  // outside a graph clears the flag, and the next graph launch re-sends t.
  int64_t* t_dev;
  bool t_dev_synced;
  // FP8 caches: one token's rows for the prefill's rounds of append + decode
  // (q bf16 [B][8 H][D] | out fp32 [B][8 H][D] | k, v bf16 [NH][D] | logit fp32 [NH]).
  uint8_t* round_buf;
  // Steps from host buffers (dms_step_host), made on first use.
  struct dms_host_pipe* host_pipe;
};

// Two sets of device rows for steps whose inputs and output live in host
// memory, with a copy-in and a copy-out stream.  Call i uses set i % 2: its
// host->device copies wait only for the kernel of call i - 2 (which read that
// set), so they run under the kernel of call i - 1; its device->host copy runs
// under the kernel of call i + 1.  The copy streams wait for kernels through
// the kern_done events; the kernels wait for the copy streams through sequence
// numbers that the copy streams write into flags (stream memory writes) and
// the kernel polls (DecodeArgs::host_flag), so that the compute stream holds
// nothing but the step kernels and each keeps its early start.
typedef CUresult (*StreamWriteValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
struct dms_host_pipe {
  cudaStream_t in_st = nullptr, out_st = nullptr;
  cudaEvent_t kern_done[2] = {}, out_done[2] = {};
  bool used[2] = {false, false};
  uint8_t* buf[2] = {nullptr, nullptr};  // each laid out as RoundLayout
  unsigned* flags = nullptr;             // [2 sets][rows landed, output read back]
  unsigned seq[2] = {0, 0};              // calls made on each set
  StreamWriteValue32Fn write_value = nullptr;
  int next = 0;
};

namespace {

constexpr size_t kAlign = 256;

std::mutex g_mu;
std::unordered_set<const dms_cache*> g_live;
thread_local int g_last_error = DMS_OK;

bool is_live(const dms_cache* c) {
  std::lock_guard<std::mutex> lk(g_mu);
  return c != nullptr && g_live.count(c) != 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Make the cache's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Is `p` device memory of device `dev` (or managed memory)?
bool device_pointer_ok(const void* p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type == cudaMemoryTypeManaged) return true;
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? DMS_OK : DMS_ERR_CUDA; }

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream is still running; every kernel of
// this library calls griddepcontrol.wait before touching global memory, so
// stream order is preserved for data while launch latency is overlapped.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
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
  return launch_status();
}

// The new token of a fused step (dms_step): its K, V rows and eviction logit;
// t_dev set when the launch is captured into a CUDA graph (the position is
// then read from device memory at replay); early: the launch may start before
// the previous one has finished (DecodeArgs::early).
struct StepInput {
  const uint4* k;
  const uint4* v;
  const float* logit;
  const int64_t* t_dev;
  bool early;
  // steps from host rows: the set's sequence flags and the values to wait for
  const unsigned* host_flag = nullptr;
  unsigned in_need = 0, out_need = 0;
};

// May the fused step of cache c at its current position start early?  Needs
// the lengths after t - 1 appends (the last advance added one token) and ring
// entries of t - 1 - w and t - w that the previous step does not write (w >= 2).
bool step_can_start_early(const dms_cache* c) { return c->w >= 2 && c->t >= 1 && c->single_prev; }

// Decode launch.  Plain (FUSED false): attention of q over the cache as it
// stands at position c->t.  Fused (FUSED true, `in` set): the token of
// position c->t is appended in the same launch and the attention runs over
// the cache after it; the caller then advances c->t.
// Opt the decode kernel into its dynamic shared memory on c's device (once;
// not a stream operation, so it is done before any stream capture).
template <int D, int G, bool FUSED, int KVF>
int decode_attr(const dms_cache* c) {
  using Sh = dms::DecodeShape<D, G, KVF>;
  static std::atomic<bool> attr_done[64] = {};  // set once per device; threads may race to set it
  if (c->device < 64 && attr_done[c->device]) return DMS_OK;
  if (cudaFuncSetAttribute(dms::decode_kernel<D, G, FUSED, KVF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Sh::SMEM) != cudaSuccess) {
    cudaGetLastError();
    return DMS_ERR_CUDA;
  }
  if (c->device < 64) attr_done[c->device] = true;
  return DMS_OK;
}

// G: query heads per warp task; nsplit: groups per KV head (query heads per KV
// head = G * nsplit), see dms::DecodeArgs.
template <int D, int G, bool FUSED, int KVF>
int launch_decode_t(dms_cache* c, const void* q, float* out, float scale, cudaStream_t st, const StepInput* in,
                    int nsplit = 1) {
  using Sh = dms::DecodeShape<D, G, KVF>;
  if (decode_attr<D, G, FUSED, KVF>(c) != DMS_OK) return DMS_ERR_CUDA;
  const int64_t NV = static_cast<int64_t>(c->NH) * nsplit;
  // The prologue's prefix sums and lengths (and, fused, each head's new and previous slot) fit in shared memory.
  if ((NV + 1 + c->NH + (FUSED ? 2 * c->NH : 0)) * 4 > Sh::SMEM) return DMS_ERR_INVALID_ARG;
  // Upper bound of the retained slots (the exact sum lives on the device); a
  // graph-replayed step runs at positions unknown now, so it takes the capacity.
  const bool graph = FUSED && in != nullptr && in->t_dev != nullptr;
  const int64_t smax = NV * (graph ? c->cap : std::min<int64_t>(c->t + (FUSED ? 1 : 0), c->cap));
  const int64_t want = (smax + int64_t(dms::kMinSlotsPerWarp) * Sh::NW - 1) / (int64_t(dms::kMinSlotsPerWarp) * Sh::NW);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(c->num_sms, want)));
  if (static_cast<size_t>(grid) * Sh::NW + NV > c->part_entries) return DMS_ERR_INVALID_ARG;
  dms::DecodeArgs a{};
  a.K = c->view.K;
  a.V = c->view.V;
  a.len = dms::len_after(c->view, c->t);
  a.q = static_cast<const uint16_t*>(q);
  a.out = out;
  a.part_acc = c->part_acc;
  a.part_ml = c->part_ml;
  a.head_cnt = c->head_cnt;
  a.err = c->view.err;
  a.NH = c->NH;
  a.Hkv = c->H;
  a.cap = c->cap;
  a.qscale = scale * 1.4426950408889634f;  // log2(e): softmax evaluated as 2^(x log2 e)
  a.Gq = G * nsplit;
  a.nsplit = nsplit;
  a.k_new = nullptr;
  a.v_new = nullptr;
  a.logit_new = nullptr;
  a.K_w = nullptr;
  a.V_w = nullptr;
  a.slot_pos = nullptr;
  a.ring_slot = c->view.ring_slot;
  a.ring_flag = c->view.ring_flag;
  a.len_w = nullptr;
  a.t_dev = nullptr;
  a.t = c->t;
  a.w = c->w;
  a.early = 0;
  a.min_tiles = dms::kMinTilesPerWarp;
  a.clamp_len = 0;
  if constexpr (FUSED) {
    a.k_new = in->k;
    a.v_new = in->v;
    a.logit_new = in->logit;
    a.K_w = c->view.K;
    a.V_w = c->view.V;
    a.slot_pos = c->view.slot_pos;
    a.len = c->view.len;  // both halves: the kernel picks them by the position's parity
    a.len_w = c->view.len;
    a.t_dev = in->t_dev;
    a.early = in->early ? 1 : 0;
    a.host_flag = in->host_flag;
    a.in_need = in->in_need;
    a.out_need = in->out_need;
  }
  return launch_pdl(dms::decode_kernel<D, G, FUSED, KVF>, dim3(grid), dim3(Sh::NW * 32), Sh::SMEM, st, a);
}

template <int D, bool FUSED, int KVF = dms::kKvBf16>
int launch_decode_d(dms_cache* c, const void* q, float* out, float scale, int G, cudaStream_t st,
                    const StepInput* in = nullptr) {
  switch (G) {
    case 1: return launch_decode_t<D, 1, FUSED, KVF>(c, q, out, scale, st, in);
    case 2: return launch_decode_t<D, 2, FUSED, KVF>(c, q, out, scale, st, in);
    case 3: return launch_decode_t<D, 3, FUSED, KVF>(c, q, out, scale, st, in);
    case 4: return launch_decode_t<D, 4, FUSED, KVF>(c, q, out, scale, st, in);
    case 5: return launch_decode_t<D, 5, FUSED, KVF>(c, q, out, scale, st, in);
    // Six and eight query heads per KV head run as two groups of three / four:
    // the 12-warp kernel of the smaller group beats the 8-warp kernel that the
    // registers of a six- or eight-head warp allow.
    case 6: return launch_decode_t<D, 3, FUSED, KVF>(c, q, out, scale, st, in, 2);
    case 7: return launch_decode_t<D, 7, FUSED, KVF>(c, q, out, scale, st, in);
    case 8: return launch_decode_t<D, 4, FUSED, KVF>(c, q, out, scale, st, in, 2);
    default: return DMS_ERR_INVALID_ARG;
  }
}

template <int D, int G>
int launch_prefill_t(dms_cache* c, const dms::PrefillArgs& a, cudaStream_t st) {
  using Sh = dms::PrefillShape<D, G>;
  static std::atomic<bool> attr_done[64] = {};  // set once per device; threads may race to set it
  if (c->device < 64 && !attr_done[c->device]) {
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device) != cudaSuccess ||
        optin < Sh::SMEM + 1024) {  // dynamic + the kernel's 1 KB of static shared memory
      cudaGetLastError();
      return DMS_ERR_CUDA;
    }
    if (cudaFuncSetAttribute(dms::prefill_attention_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Sh::SMEM) != cudaSuccess) {
      cudaGetLastError();
      return DMS_ERR_CUDA;
    }
    attr_done[c->device] = true;
  }
  const dim3 grid((a.C + Sh::PT - 1) / Sh::PT, c->NH);
  return launch_pdl(dms::prefill_attention_kernel<D, G>, grid, dim3(256), Sh::SMEM, st, a);
}

template <int D>
int launch_prefill_d(dms_cache* c, const dms::PrefillArgs& a, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_prefill_t<D, 1>(c, a, st);
    case 2: return launch_prefill_t<D, 2>(c, a, st);
    case 3: return launch_prefill_t<D, 3>(c, a, st);
    case 4: return launch_prefill_t<D, 4>(c, a, st);
    case 5: return launch_prefill_t<D, 5>(c, a, st);
    case 6: return launch_prefill_t<D, 6>(c, a, st);
    case 7: return launch_prefill_t<D, 7>(c, a, st);
    case 8: return launch_prefill_t<D, 8>(c, a, st);
    default: return DMS_ERR_INVALID_ARG;
  }
}

// decode_attr for the cache's head dim, group size and format (fused kernel).
template <int D, int KVF>
int fused_attr_k(const dms_cache* c, int G) {
  switch (G) {
    case 1: return decode_attr<D, 1, true, KVF>(c);
    case 2: return decode_attr<D, 2, true, KVF>(c);
    case 3: return decode_attr<D, 3, true, KVF>(c);
    case 4: return decode_attr<D, 4, true, KVF>(c);
    case 5: return decode_attr<D, 5, true, KVF>(c);
    case 6: return decode_attr<D, 3, true, KVF>(c);
    case 7: return decode_attr<D, 7, true, KVF>(c);
    case 8: return decode_attr<D, 4, true, KVF>(c);
    default: return DMS_ERR_INVALID_ARG;
  }
}
template <int D>
int fused_attr_d(const dms_cache* c, int G) {
  return c->kvf == DMS_KV_FP8_E4M3 ? fused_attr_k<D, dms::kKvFp8>(c, G) : fused_attr_k<D, dms::kKvBf16>(c, G);
}

// Decode launch for the cache's storage format (plain, or fused with `in`).
template <int D, bool FUSED>
int launch_decode_f(dms_cache* c, const void* q, float* out, float scale, int G, cudaStream_t st,
                    const StepInput* in = nullptr) {
  return c->kvf == DMS_KV_FP8_E4M3 ? launch_decode_d<D, FUSED, dms::kKvFp8>(c, q, out, scale, G, st, in)
                                   : launch_decode_d<D, FUSED, dms::kKvBf16>(c, q, out, scale, G, st, in);
}

// Single-token append (one warp per head) for the cache's head dim and format.
int launch_append(dms_cache* c, const void* k, const void* v, const float* logit, cudaStream_t st) {
  const int blocks = (c->NH * 32 + 255) / 256;
  const uint4* k4 = static_cast<const uint4*>(k);
  const uint4* v4 = static_cast<const uint4*>(v);
  const bool fp8 = c->kvf == DMS_KV_FP8_E4M3;
  if (c->D == 128)
    return fp8 ? launch_pdl(dms::append_kernel<128, dms::kKvFp8>, dim3(blocks), dim3(256), 0, st, c->view, k4, v4,
                            logit, c->t)
               : launch_pdl(dms::append_kernel<128, dms::kKvBf16>, dim3(blocks), dim3(256), 0, st, c->view, k4, v4,
                            logit, c->t);
  return fp8 ? launch_pdl(dms::append_kernel<64, dms::kKvFp8>, dim3(blocks), dim3(256), 0, st, c->view, k4, v4, logit,
                          c->t)
             : launch_pdl(dms::append_kernel<64, dms::kKvBf16>, dim3(blocks), dim3(256), 0, st, c->view, k4, v4,
                          logit, c->t);
}

// Chunk append: the bookkeeping (one warp per head), then the row copy.
int launch_append_chunk(dms_cache* c, const void* k, const void* v, const float* logits, int chunk, cudaStream_t st) {
  const int rc = launch_pdl(dms::append_chunk_slots_kernel, dim3((c->NH + 3) / 4), dim3(128), 0, st, c->view, logits,
                            c->t, chunk);
  if (rc != DMS_OK) return rc;
  const dim3 grid((c->cap + 255) / 256, c->NH);
  const uint4* k4 = static_cast<const uint4*>(k);
  const uint4* v4 = static_cast<const uint4*>(v);
  const bool fp8 = c->kvf == DMS_KV_FP8_E4M3;
  if (c->D == 128)
    return fp8 ? launch_pdl(dms::append_chunk_copy_kernel<128, dms::kKvFp8>, grid, dim3(256), 0, st, c->view, k4, v4,
                            c->t, chunk)
               : launch_pdl(dms::append_chunk_copy_kernel<128, dms::kKvBf16>, grid, dim3(256), 0, st, c->view, k4, v4,
                            c->t, chunk);
  return fp8 ? launch_pdl(dms::append_chunk_copy_kernel<64, dms::kKvFp8>, grid, dim3(256), 0, st, c->view, k4, v4,
                          c->t, chunk)
             : launch_pdl(dms::append_chunk_copy_kernel<64, dms::kKvBf16>, grid, dim3(256), 0, st, c->view, k4, v4,
                          c->t, chunk);
}

}  // namespace

// A decode step over several caches captured into a CUDA graph.
struct dms_step_graph {
  std::vector<dms_cache*> caches;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int64_t** pos = nullptr;  // device array: each cache's position word
  int device = 0;
  // The buffers bound at capture, for a token step run as per-layer launches
  // when the graph's early-started layers may not start early (see launch).
  std::vector<const void*> k, v, q;
  std::vector<const float*> logit;
  std::vector<float*> out;
  float scale = 1.f;
  int q_heads = 0;
};

namespace {

void free_host_pipe(dms_host_pipe* p) {
  if (p == nullptr) return;
  for (int s = 0; s < 2; ++s) {
    if (p->kern_done[s]) cudaEventDestroy(p->kern_done[s]);
    if (p->out_done[s]) cudaEventDestroy(p->out_done[s]);
    cudaFree(p->buf[s]);
  }
  cudaFree(p->flags);
  if (p->in_st) cudaStreamDestroy(p->in_st);
  if (p->out_st) cudaStreamDestroy(p->out_st);
  delete p;
}

void free_cache_memory(dms_cache* c) {
  free_host_pipe(c->host_pipe);
  c->host_pipe = nullptr;
  cudaFree(c->view.K);
  cudaFree(c->view.V);
  cudaFree(c->view.slot_pos);
  cudaFree(c->view.ring_slot);
  cudaFree(c->view.ring_flag);
  cudaFree(c->view.len);
  cudaFree(c->view.err);
  cudaFree(c->part_acc);
  cudaFree(c->part_ml);
  cudaFree(c->head_cnt);
  cudaFree(c->round_buf);
}

// Byte offsets into dms_cache::round_buf.
struct RoundLayout {
  size_t q, out, k, v, logit, total;
  explicit RoundLayout(const dms_cache* c) {
    const size_t rows_q = static_cast<size_t>(c->NH) * DMS_MAX_GROUP, d = static_cast<size_t>(c->D);
    q = 0;
    out = q + rows_q * d * 2;
    k = out + rows_q * d * 4;
    v = k + static_cast<size_t>(c->NH) * d * 2;
    logit = v + static_cast<size_t>(c->NH) * d * 2;
    total = logit + ((static_cast<size_t>(c->NH) * 4 + 255) / 256) * 256;
  }
};

// FP8 caches: the chunked prefill as its definition states it, C rounds of
// (append token c, decode token c's query), each one launch of the fused FP8
// step kernel.  Token c's rows are gathered from the chunk layouts into the
// cache's round buffer with pitched copies, and its output row is scattered
// back.  Exact by construction; one decode launch per token.
int prefill_by_rounds(dms_cache* c, const void* q, const void* k, const void* v, const float* logits, int chunk,
                      float* out, float scale, int q_heads, cudaStream_t st) {
  const RoundLayout lay(c);
  uint8_t* rb = c->round_buf;
  const size_t D = static_cast<size_t>(c->D), C = static_cast<size_t>(chunk);
  const size_t rows_q = static_cast<size_t>(c->B) * q_heads, rows_kv = static_cast<size_t>(c->NH);
  const int G = q_heads / c->H;
  for (size_t t = 0; t < C; ++t) {
    const bool ok =
        cudaMemcpy2DAsync(rb + lay.q, D * 2, static_cast<const uint8_t*>(q) + t * D * 2, C * D * 2, D * 2, rows_q,
                          cudaMemcpyDeviceToDevice, st) == cudaSuccess &&
        cudaMemcpy2DAsync(rb + lay.k, D * 2, static_cast<const uint8_t*>(k) + t * D * 2, C * D * 2, D * 2, rows_kv,
                          cudaMemcpyDeviceToDevice, st) == cudaSuccess &&
        cudaMemcpy2DAsync(rb + lay.v, D * 2, static_cast<const uint8_t*>(v) + t * D * 2, C * D * 2, D * 2, rows_kv,
                          cudaMemcpyDeviceToDevice, st) == cudaSuccess &&
        cudaMemcpy2DAsync(rb + lay.logit, 4, logits + t, C * 4, 4, rows_kv, cudaMemcpyDeviceToDevice, st) ==
            cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return DMS_ERR_CUDA;
    }
    // one fused step (append + decode) per token
    float* o = reinterpret_cast<float*>(rb + lay.out);
    const StepInput in{reinterpret_cast<const uint4*>(rb + lay.k), reinterpret_cast<const uint4*>(rb + lay.v),
                       reinterpret_cast<const float*>(rb + lay.logit), nullptr, false};
    const int rc = c->D == 128 ? launch_decode_f<128, true>(c, rb + lay.q, o, scale, G, st, &in)
                               : launch_decode_f<64, true>(c, rb + lay.q, o, scale, G, st, &in);
    if (rc != DMS_OK) return rc;
    c->t += 1;
    if (cudaMemcpy2DAsync(out + t * D, C * D * 4, o, D * 4, D * 4, rows_q, cudaMemcpyDeviceToDevice, st) !=
        cudaSuccess) {
      cudaGetLastError();
      return DMS_ERR_CUDA;
    }
  }
  return DMS_OK;
}

// The fused step (append token t, decode its query) on device rows whose
// pointers the caller has checked; advances the host position.
int step_launch(dms_cache* c, const void* k, const void* v, const float* evict_logit, const void* q, float* out,
                float scale, int G, cudaStream_t st, const unsigned* host_flag = nullptr, unsigned in_need = 0,
                unsigned out_need = 0) {
  // One launch (bf16 or FP8 storage).  The decode kernel appends the token
  // (into generations of the state that the step does not read; FP8 caches
  // quantize it) and attends over the cache after the append; after a
  // one-token advance it starts before the previous launch has finished.
  StepInput in{static_cast<const uint4*>(k), static_cast<const uint4*>(v), evict_logit, nullptr,
               step_can_start_early(c)};
  in.host_flag = host_flag;
  in.in_need = in_need;
  in.out_need = out_need;
  const int rc = c->D == 128 ? launch_decode_f<128, true>(c, q, out, scale, G, st, &in)
                             : launch_decode_f<64, true>(c, q, out, scale, G, st, &in);
  if (rc != DMS_OK) return rc;
  c->t += 1;
  c->single_prev = true;
  c->t_dev_synced = false;
  return DMS_OK;
}

// The host-buffer pipeline of a cache, made on its first use.
dms_host_pipe* host_pipe(dms_cache* c) {
  if (c->host_pipe != nullptr) return c->host_pipe;
  dms_host_pipe* p = new (std::nothrow) dms_host_pipe();
  if (p == nullptr) return nullptr;
  const size_t bytes = RoundLayout(c).total;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult qr = cudaDriverEntryPointSymbolNotFound;
  bool ok = cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fn, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess && fn != nullptr;
  p->write_value = reinterpret_cast<StreamWriteValue32Fn>(fn);
  ok = ok && cudaStreamCreateWithFlags(&p->in_st, cudaStreamNonBlocking) == cudaSuccess &&
       cudaStreamCreateWithFlags(&p->out_st, cudaStreamNonBlocking) == cudaSuccess &&
       cudaMalloc(&p->flags, 4 * sizeof(unsigned)) == cudaSuccess &&
       cudaMemset(p->flags, 0, 4 * sizeof(unsigned)) == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess;
  for (int s = 0; s < 2 && ok; ++s)
    ok = cudaEventCreateWithFlags(&p->kern_done[s], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->out_done[s], cudaEventDisableTiming) == cudaSuccess &&
         cudaMalloc(&p->buf[s], bytes) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    free_host_pipe(p);
    return nullptr;
  }
  c->host_pipe = p;
  return p;
}

// Host memory that a copy may read or write (pinned, or plain pageable memory).
bool host_pointer_ok(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return true;  // unknown to CUDA: pageable host memory
  }
  return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

}  // namespace

extern "C" {

int dms_last_error(void) { return g_last_error; }

const char* dms_error_string(int code) {
  switch (code) {
    case DMS_OK: return "ok";
    case DMS_ERR_INVALID_ARG: return "invalid argument";
    case DMS_ERR_CUDA: return "CUDA error";
    case DMS_ERR_CAPACITY: return "cache capacity exceeded (sticky)";
    case DMS_ERR_BAD_HANDLE: return "bad cache handle";
    case DMS_ERR_TIMEOUT: return "device wait timed out (sticky)";
    case DMS_ERR_EMPTY: return "cache is empty";
    case DMS_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown error";
  }
}

dms_cache_t* dms_cache_create(int batch, int kv_heads, int capacity, int head_dim, int window) {
  return dms_cache_create_ex(batch, kv_heads, capacity, head_dim, window, DMS_KV_BF16);
}

dms_cache_t* dms_cache_create_ex(int batch, int kv_heads, int capacity, int head_dim, int window, int kv_format) {
  g_last_error = DMS_OK;
  if (batch < 1 || kv_heads < 1 || capacity < 1 || window < 1 || (head_dim != 64 && head_dim != 128) ||
      (kv_format != DMS_KV_BF16 && kv_format != DMS_KV_FP8_E4M3)) {
    g_last_error = DMS_ERR_INVALID_ARG;
    return nullptr;
  }
  const int64_t NH = static_cast<int64_t>(batch) * kv_heads;
  if (NH > (1 << 20) || NH * static_cast<int64_t>(capacity) >= (int64_t(1) << 31) ||
      2 * NH * static_cast<int64_t>(window) >= (int64_t(1) << 31)) {
    g_last_error = DMS_ERR_INVALID_ARG;
    return nullptr;
  }
  dms_cache* c = new (std::nothrow) dms_cache();
  if (!c) {
    g_last_error = DMS_ERR_CUDA;
    return nullptr;
  }
  std::memset(c, 0, sizeof(*c));
  c->B = batch;
  c->H = kv_heads;
  c->cap = capacity;
  c->D = head_dim;
  c->w = window;
  c->NH = static_cast<int>(NH);
  c->kvf = kv_format;
  c->t = 0;
  c->single_prev = false;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    g_last_error = DMS_ERR_CUDA;
    return nullptr;
  }
  // bytes per slot: bf16 2 D per row; fp8 D codes per row, plus the K row's 16-byte scale chunk
  const bool fp8 = kv_format == DMS_KV_FP8_E4M3;
  const size_t kpool = static_cast<size_t>(NH) * capacity * (fp8 ? head_dim + 16 : 2 * head_dim);
  const size_t vpool = static_cast<size_t>(NH) * capacity * (fp8 ? head_dim : 2 * head_dim);
  const size_t nslot = static_cast<size_t>(NH) * capacity;
  const size_t nring = 2 * static_cast<size_t>(NH) * window;  // two generations
  // partials: one per warp and virtual head (two per KV head when its query heads are split)
  c->part_entries = static_cast<size_t>(c->num_sms) * dms::kMaxWarpsPerCta + 2 * NH;
  const size_t part_acc = c->part_entries * DMS_MAX_GROUP * head_dim * sizeof(float);
  const size_t part_ml = c->part_entries * DMS_MAX_GROUP * 2 * sizeof(float);
  bool ok = cudaMalloc(&c->view.K, kpool) == cudaSuccess && cudaMalloc(&c->view.V, vpool) == cudaSuccess &&
            cudaMalloc(&c->view.slot_pos, nslot * 4) == cudaSuccess &&
            cudaMalloc(&c->view.ring_slot, nring * 4) == cudaSuccess &&
            cudaMalloc(&c->view.ring_flag, nring) == cudaSuccess &&
            cudaMalloc(&c->view.len, dms::kLenGens * NH * 4) == cudaSuccess && cudaMalloc(&c->view.err, kAlign) == cudaSuccess &&
            cudaMalloc(&c->part_acc, part_acc) == cudaSuccess && cudaMalloc(&c->part_ml, part_ml) == cudaSuccess &&
            cudaMalloc(&c->head_cnt, 2 * NH * 4) == cudaSuccess &&
            (!fp8 || cudaMalloc(&c->round_buf, RoundLayout(c).total) == cudaSuccess);
  ok = ok && cudaMemset(c->view.K, 0, kpool) == cudaSuccess && cudaMemset(c->view.V, 0, vpool) == cudaSuccess &&
       cudaMemset(c->view.slot_pos, 0xff, nslot * 4) == cudaSuccess &&
       cudaMemset(c->view.ring_slot, 0xff, nring * 4) == cudaSuccess &&
       cudaMemset(c->view.ring_flag, 0, nring) == cudaSuccess && cudaMemset(c->view.len, 0, dms::kLenGens * NH * 4) == cudaSuccess &&
       cudaMemset(c->view.err, 0, kAlign) == cudaSuccess && cudaMemset(c->head_cnt, 0, 2 * NH * 4) == cudaSuccess &&
       cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    free_cache_memory(c);
    delete c;
    g_last_error = DMS_ERR_CUDA;
    return nullptr;
  }
  c->view.NH = c->NH;
  c->view.cap = capacity;
  c->view.D = head_dim;
  c->view.w = window;
  c->view.kvf = fp8 ? dms::kKvFp8 : dms::kKvBf16;
  c->t_dev = reinterpret_cast<int64_t*>(reinterpret_cast<char*>(c->view.err) + 64);  // zeroed with the error word
  c->t_dev_synced = true;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_live.insert(c);
  }
  return c;
}

void dms_cache_destroy(dms_cache_t* cache) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (cache == nullptr || g_live.erase(cache) == 0) return;
  }
  DeviceGuard g(cache->device);
  cudaDeviceSynchronize();
  free_cache_memory(cache);
  delete cache;
}

int64_t dms_cache_position(dms_cache_t* cache) { return is_live(cache) ? cache->t : -1; }

int dms_append(dms_cache_t* c, const void* k, const void* v, const float* evict_logit, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (!k || !v || !evict_logit || !aligned16(k) || !aligned16(v) || !aligned16(evict_logit))
    return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return DMS_ERR_CUDA;
  if (!device_pointer_ok(k, c->device) || !device_pointer_ok(v, c->device) ||
      !device_pointer_ok(evict_logit, c->device))
    return DMS_ERR_INVALID_ARG;
  const int rc = launch_append(c, k, v, evict_logit, static_cast<cudaStream_t>(stream));
  if (rc == DMS_OK) {
    c->t += 1;
    c->single_prev = true;
  }
  c->t_dev_synced = false;
  return rc;
}

int dms_append_chunk(dms_cache_t* c, const void* k, const void* v, const float* logits, int chunk, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (chunk < 1 || !k || !v || !logits || !aligned16(k) || !aligned16(v) || !aligned16(logits))
    return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return DMS_ERR_CUDA;
  if (!device_pointer_ok(k, c->device) || !device_pointer_ok(v, c->device) || !device_pointer_ok(logits, c->device))
    return DMS_ERR_INVALID_ARG;
  const int rc = launch_append_chunk(c, k, v, logits, chunk, static_cast<cudaStream_t>(stream));
  if (rc == DMS_OK) {
    c->t += chunk;
    c->single_prev = chunk == 1;
  }
  c->t_dev_synced = false;
  return rc;
}

int dms_prefill(dms_cache_t* c, const void* q, const void* k, const void* v, const float* logits, int chunk,
                float* out, float scale, int q_heads, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (chunk < 1 || !q || !k || !v || !logits || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(logits) || !aligned16(out) || q_heads < 1 || q_heads % c->H != 0 ||
      q_heads / c->H > DMS_MAX_GROUP || !std::isfinite(scale) || c->t + chunk > INT32_MAX)
    return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return DMS_ERR_CUDA;
  if (!device_pointer_ok(q, c->device) || !device_pointer_ok(k, c->device) || !device_pointer_ok(v, c->device) ||
      !device_pointer_ok(logits, c->device) || !device_pointer_ok(out, c->device))
    return DMS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->kvf == DMS_KV_FP8_E4M3) {
    // the tensor-core kernel reads bf16 rows; FP8 caches run the definition
    const int rc = prefill_by_rounds(c, q, k, v, logits, chunk, out, scale, q_heads, st);
    c->single_prev = rc == DMS_OK;  // rounds of single appends
    c->t_dev_synced = false;
    return rc;
  }
  dms::PrefillArgs a;
  a.K = c->view.K;
  a.V = c->view.V;
  a.len = dms::len_after(c->view, c->t);
  a.slot_pos = c->view.slot_pos;
  a.ring_flag = c->view.ring_flag;
  a.q = static_cast<const uint4*>(q);
  a.kc = static_cast<const uint4*>(k);
  a.vc = static_cast<const uint4*>(v);
  a.logits = logits;
  a.out = out;
  a.err = c->view.err;
  a.NH = c->NH;
  a.Hkv = c->H;
  a.cap = c->cap;
  a.w = c->w;
  a.C = chunk;
  a.t0 = static_cast<int>(c->t);
  a.qscale = scale * 1.4426950408889634f;  // log2(e)
  const int G = q_heads / c->H;
  int rc = c->D == 128 ? launch_prefill_d<128>(c, a, G, st) : launch_prefill_d<64>(c, a, G, st);
  if (rc != DMS_OK) return rc;
  rc = launch_append_chunk(c, k, v, logits, chunk, st);
  if (rc == DMS_OK) {
    c->t += chunk;
    c->single_prev = chunk == 1;
  }
  c->t_dev_synced = false;
  return rc;
}

int dms_decode_attention(dms_cache_t* c, const void* q, float* out, float scale, int q_heads, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (!q || !out || !aligned16(q) || !aligned16(out) || q_heads < 1 || q_heads % c->H != 0 ||
      q_heads / c->H > DMS_MAX_GROUP || !std::isfinite(scale))
    return DMS_ERR_INVALID_ARG;
  if (c->t == 0) return DMS_ERR_EMPTY;
  DeviceGuard g(c->device);
  if (!g.ok) return DMS_ERR_CUDA;
  if (!device_pointer_ok(q, c->device) || !device_pointer_ok(out, c->device)) return DMS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int G = q_heads / c->H;
  return c->D == 128 ? launch_decode_f<128, false>(c, q, out, scale, G, st)
                     : launch_decode_f<64, false>(c, q, out, scale, G, st);
}

int dms_step(dms_cache_t* c, const void* k, const void* v, const float* evict_logit, const void* q, float* out,
             float scale, int q_heads, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (!k || !v || !evict_logit || !q || !out || !aligned16(k) || !aligned16(v) || !aligned16(evict_logit) ||
      !aligned16(q) || !aligned16(out) || q_heads < 1 || q_heads % c->H != 0 || q_heads / c->H > DMS_MAX_GROUP ||
      !std::isfinite(scale))
    return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return DMS_ERR_CUDA;
  if (!device_pointer_ok(k, c->device) || !device_pointer_ok(v, c->device) ||
      !device_pointer_ok(evict_logit, c->device) || !device_pointer_ok(q, c->device) ||
      !device_pointer_ok(out, c->device))
    return DMS_ERR_INVALID_ARG;
  return step_launch(c, k, v, evict_logit, q, out, scale, q_heads / c->H, static_cast<cudaStream_t>(stream));
}

int dms_step_host(dms_cache_t* c, const void* k, const void* v, const float* evict_logit, const void* q, float* out,
                  float scale, int q_heads, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (!k || !v || !evict_logit || !q || !out || q_heads < 1 || q_heads % c->H != 0 ||
      q_heads / c->H > DMS_MAX_GROUP || !std::isfinite(scale))
    return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!g.ok) return DMS_ERR_CUDA;
  if (!host_pointer_ok(k) || !host_pointer_ok(v) || !host_pointer_ok(evict_logit) || !host_pointer_ok(q) ||
      !host_pointer_ok(out))
    return DMS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    return DMS_ERR_INVALID_ARG;
  }
  if (cs != cudaStreamCaptureStatusNone) return DMS_ERR_INVALID_ARG;
  dms_host_pipe* p = host_pipe(c);
  if (p == nullptr) return DMS_ERR_CUDA;
  const RoundLayout lay(c);
  const int s = p->next;
  uint8_t* b = p->buf[s];
  const size_t D = static_cast<size_t>(c->D), NH = static_cast<size_t>(c->NH);
  const size_t q_bytes = static_cast<size_t>(c->B) * q_heads * D * 2;
  const unsigned seq = p->seq[s] + 1;  // this call's number on set s; the set's last copy-out wrote seq - 1
  unsigned* flag = p->flags + 2 * s;
  const auto write_flag = [&](unsigned* addr, cudaStream_t cs) {
    return p->write_value(reinterpret_cast<CUstream>(cs), reinterpret_cast<CUdeviceptr>(addr), seq, 0) ==
           CUDA_SUCCESS;
  };
  // copy in, after the kernel that last read this set; then flag the rows as landed
  bool ok = !p->used[s] || cudaStreamWaitEvent(p->in_st, p->kern_done[s], 0) == cudaSuccess;
  ok = ok && cudaMemcpyAsync(b + lay.k, k, NH * D * 2, cudaMemcpyHostToDevice, p->in_st) == cudaSuccess &&
       cudaMemcpyAsync(b + lay.v, v, NH * D * 2, cudaMemcpyHostToDevice, p->in_st) == cudaSuccess &&
       cudaMemcpyAsync(b + lay.logit, evict_logit, NH * 4, cudaMemcpyHostToDevice, p->in_st) == cudaSuccess &&
       cudaMemcpyAsync(b + lay.q, q, q_bytes, cudaMemcpyHostToDevice, p->in_st) == cudaSuccess &&
       write_flag(flag, p->in_st);
  if (!ok) {
    cudaGetLastError();
    return DMS_ERR_CUDA;  // nothing of this call reached the compute stream; the set's numbering is unchanged
  }
  p->seq[s] = seq;
  p->used[s] = true;
  p->next = s ^ 1;
  // the step: its kernel waits (on the device) for flag[0] >= seq and flag[1] >= seq - 1
  float* o = reinterpret_cast<float*>(b + lay.out);
  const int rc = step_launch(c, b + lay.k, b + lay.v, reinterpret_cast<const float*>(b + lay.logit), b + lay.q, o,
                             scale, q_heads / c->H, st, flag, seq, seq - 1);
  // copy out after the step, then flag the output rows as read back (also when
  // the launch failed, so that the next call on this set does not wait in vain)
  ok = cudaEventRecord(p->kern_done[s], st) == cudaSuccess &&
       cudaStreamWaitEvent(p->out_st, p->kern_done[s], 0) == cudaSuccess &&
       (rc != DMS_OK || cudaMemcpyAsync(out, o, static_cast<size_t>(c->B) * q_heads * D * 4,
                                        cudaMemcpyDeviceToHost, p->out_st) == cudaSuccess) &&
       write_flag(flag + 1, p->out_st) && cudaEventRecord(p->out_done[s], p->out_st) == cudaSuccess;
  if (rc != DMS_OK) return rc;
  if (!ok) {
    cudaGetLastError();
    return DMS_ERR_CUDA;
  }
  return DMS_OK;
}

int dms_step_host_join(dms_cache_t* c, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  dms_host_pipe* p = c->host_pipe;
  if (p == nullptr) return DMS_OK;
  DeviceGuard g(c->device);
  if (!g.ok) return DMS_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int s = 0; s < 2; ++s)
    if (p->used[s] && cudaStreamWaitEvent(st, p->out_done[s], 0) != cudaSuccess) {
      cudaGetLastError();
      return DMS_ERR_CUDA;
    }
  return DMS_OK;
}

int dms_cache_lengths(dms_cache_t* c, int32_t* out_dev, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (!out_dev) return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!device_pointer_ok(out_dev, c->device)) return DMS_ERR_INVALID_ARG;
  return cudaMemcpyAsync(out_dev, dms::len_after(c->view, c->t), static_cast<size_t>(c->NH) * 4, cudaMemcpyDeviceToDevice,
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DMS_OK
             : DMS_ERR_CUDA;
}

int dms_cache_slot_positions(dms_cache_t* c, int32_t* out_dev, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (!out_dev) return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!device_pointer_ok(out_dev, c->device)) return DMS_ERR_INVALID_ARG;
  return cudaMemcpyAsync(out_dev, c->view.slot_pos, static_cast<size_t>(c->NH) * c->cap * 4,
                         cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DMS_OK
             : DMS_ERR_CUDA;
}

int dms_cache_export_kv(dms_cache_t* c, void* k_out, void* v_out, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (!k_out || !v_out || !aligned16(k_out) || !aligned16(v_out)) return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!device_pointer_ok(k_out, c->device) || !device_pointer_ok(v_out, c->device)) return DMS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int blocks = c->num_sms * 8;
  uint4* ko = static_cast<uint4*>(k_out);
  uint4* vo = static_cast<uint4*>(v_out);
  const bool fp8 = c->kvf == DMS_KV_FP8_E4M3;
  if (c->D == 128) {
    if (fp8) dms::export_kv_kernel<128, dms::kKvFp8><<<blocks, 256, 0, st>>>(c->view, ko, vo);
    else dms::export_kv_kernel<128, dms::kKvBf16><<<blocks, 256, 0, st>>>(c->view, ko, vo);
  } else {
    if (fp8) dms::export_kv_kernel<64, dms::kKvFp8><<<blocks, 256, 0, st>>>(c->view, ko, vo);
    else dms::export_kv_kernel<64, dms::kKvBf16><<<blocks, 256, 0, st>>>(c->view, ko, vo);
  }
  return launch_status();
}

int dms_cache_export_scales(dms_cache_t* c, float* k_scale, float* v_scale, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  if (!k_scale || !v_scale || c->kvf != DMS_KV_FP8_E4M3) return DMS_ERR_INVALID_ARG;
  DeviceGuard g(c->device);
  if (!device_pointer_ok(k_scale, c->device) || !device_pointer_ok(v_scale, c->device)) return DMS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int blocks = c->num_sms * 8;
  if (c->D == 128)
    dms::export_scales_kernel<128><<<blocks, 256, 0, st>>>(c->view, k_scale, v_scale);
  else
    dms::export_scales_kernel<64><<<blocks, 256, 0, st>>>(c->view, k_scale, v_scale);
  return launch_status();
}

int dms_cache_kv_format(dms_cache_t* c) { return is_live(c) ? c->kvf : DMS_ERR_BAD_HANDLE; }

int dms_cache_selftest_wait(dms_cache_t* c, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  DeviceGuard g(c->device);
  if (!g.ok) return DMS_ERR_CUDA;
  dms::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(c->view.err);
  return launch_status();
}

int dms_cache_status(dms_cache_t* c, void* stream) {
  if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  DeviceGuard g(c->device);
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DMS_ERR_CUDA;
  int32_t bits = 0;
  if (cudaMemcpy(&bits, c->view.err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return DMS_ERR_CUDA;
  if (bits & dms::kErrBitTimeout) return DMS_ERR_TIMEOUT;
  if (bits & dms::kErrBitCapacity) return DMS_ERR_CAPACITY;
  return DMS_OK;
}

dms_step_graph_t* dms_step_graph_create(dms_cache_t* const* caches, int n, const void* const* k,
                                        const void* const* v, const float* const* evict_logit,
                                        const void* const* q, float* const* out, float scale, int q_heads) {
  g_last_error = DMS_ERR_INVALID_ARG;
  if (n < 1 || !caches || !k || !v || !evict_logit || !q || !out || !std::isfinite(scale) || q_heads < 1)
    return nullptr;
  std::unordered_set<const dms_cache*> seen;
  for (int i = 0; i < n; ++i) {
    dms_cache* c = caches[i];
    if (!is_live(c)) {
      g_last_error = DMS_ERR_BAD_HANDLE;
      return nullptr;
    }
    if (!seen.insert(c).second || c->device != caches[0]->device ||
        q_heads % c->H != 0 || q_heads / c->H > DMS_MAX_GROUP || !k[i] || !v[i] || !evict_logit[i] || !q[i] ||
        !out[i] || !aligned16(k[i]) || !aligned16(v[i]) || !aligned16(evict_logit[i]) || !aligned16(q[i]) ||
        !aligned16(out[i]))
      return nullptr;
  }
  DeviceGuard g(caches[0]->device);
  g_last_error = DMS_ERR_CUDA;
  if (!g.ok) return nullptr;
  for (int i = 0; i < n; ++i) {
    dms_cache* c = caches[i];
    if (!device_pointer_ok(k[i], c->device) || !device_pointer_ok(v[i], c->device) ||
        !device_pointer_ok(evict_logit[i], c->device) || !device_pointer_ok(q[i], c->device) ||
        !device_pointer_ok(out[i], c->device)) {
      g_last_error = DMS_ERR_INVALID_ARG;
      return nullptr;
    }
    const int G = q_heads / c->H;
    if ((c->D == 128 ? fused_attr_d<128>(c, G) : fused_attr_d<64>(c, G)) != DMS_OK) return nullptr;
  }
  dms_step_graph* sg = new (std::nothrow) dms_step_graph();
  if (!sg) return nullptr;
  sg->device = caches[0]->device;
  sg->caches.assign(caches, caches + n);
  std::vector<int64_t*> pos(n);
  for (int i = 0; i < n; ++i) pos[i] = caches[i]->t_dev;
  cudaStream_t st = nullptr;
  bool ok = cudaMalloc(&sg->pos, n * sizeof(int64_t*)) == cudaSuccess &&
            cudaMemcpy(sg->pos, pos.data(), n * sizeof(int64_t*), cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
  int rc = DMS_OK;
  if (ok) {
    // One fused step per cache, each reading its position from device memory,
    // then one node that advances every position.  Layers after the first
    // start early (their launch's predecessor is another cache's step, which
    // writes none of their state); the first waits, since the node before it
    // writes the position words.
    for (int i = 0; i < n && rc == DMS_OK; ++i) {
      dms_cache* c = caches[i];
      const StepInput in{static_cast<const uint4*>(k[i]), static_cast<const uint4*>(v[i]), evict_logit[i], c->t_dev,
                         i > 0 && c->w >= 2};
      const int G = q_heads / c->H;
      rc = c->D == 128 ? launch_decode_f<128, true>(c, q[i], out[i], scale, G, st, &in)
                       : launch_decode_f<64, true>(c, q[i], out[i], scale, G, st, &in);
    }
    if (rc == DMS_OK) rc = launch_pdl(dms::advance_positions_kernel, dim3(1), dim3(32), 0, st, sg->pos, n);
    cudaGraph_t graph = nullptr;
    const bool ended = cudaStreamEndCapture(st, &graph) == cudaSuccess;
    sg->graph = graph;
    ok = rc == DMS_OK && ended && graph != nullptr &&
         cudaGraphInstantiate(&sg->exec, graph, 0) == cudaSuccess;
  }
  if (st) cudaStreamDestroy(st);
  if (!ok) {
    cudaGetLastError();
    if (sg->exec) cudaGraphExecDestroy(sg->exec);
    if (sg->graph) cudaGraphDestroy(sg->graph);
    cudaFree(sg->pos);
    delete sg;
    g_last_error = rc == DMS_ERR_INVALID_ARG ? DMS_ERR_INVALID_ARG : DMS_ERR_CUDA;
    return nullptr;
  }
  sg->k.assign(k, k + n);
  sg->v.assign(v, v + n);
  sg->logit.assign(evict_logit, evict_logit + n);
  sg->q.assign(q, q + n);
  sg->out.assign(out, out + n);
  sg->scale = scale;
  sg->q_heads = q_heads;
  g_last_error = DMS_OK;
  return sg;
}

int dms_step_graph_launch(dms_step_graph_t* sg, void* stream) {
  if (!sg) return DMS_ERR_BAD_HANDLE;
  for (dms_cache* c : sg->caches)
    if (!is_live(c)) return DMS_ERR_BAD_HANDLE;
  DeviceGuard g(sg->device);
  if (!g.ok) return DMS_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The layers captured to start early need each cache's last advance to have
  // been one token (true after any replay or dms_step).  Otherwise -- after a
  // chunk append, or on an empty cache -- this token step runs as one fused
  // launch per layer, none started early, on the same bound buffers.
  bool early_ok = true;
  for (size_t i = 1; i < sg->caches.size(); ++i) {
    const dms_cache* c = sg->caches[i];
    if (c->w >= 2 && !step_can_start_early(c)) early_ok = false;
  }
  if (!early_ok) {
    for (size_t i = 0; i < sg->caches.size(); ++i) {
      dms_cache* c = sg->caches[i];
      const StepInput in{static_cast<const uint4*>(sg->k[i]), static_cast<const uint4*>(sg->v[i]), sg->logit[i],
                         nullptr, false};
      const int G = sg->q_heads / c->H;
      const int rc = c->D == 128 ? launch_decode_f<128, true>(c, sg->q[i], sg->out[i], sg->scale, G, st, &in)
                                 : launch_decode_f<64, true>(c, sg->q[i], sg->out[i], sg->scale, G, st, &in);
      if (rc != DMS_OK) return rc;
      c->t += 1;
      c->single_prev = true;
      c->t_dev_synced = false;
    }
    return DMS_OK;
  }
  for (dms_cache* c : sg->caches) {
    if (c->t_dev_synced) continue;
    const int rc = launch_pdl(dms::set_position_kernel, dim3(1), dim3(1), 0, st, c->t_dev, c->t);
    if (rc != DMS_OK) return rc;
    c->t_dev_synced = true;
  }
  if (cudaGraphLaunch(sg->exec, st) != cudaSuccess) {
    cudaGetLastError();
    return DMS_ERR_CUDA;
  }
  for (dms_cache* c : sg->caches) {
    c->t += 1;
    c->single_prev = true;
  }
  return DMS_OK;
}

void dms_step_graph_destroy(dms_step_graph_t* sg) {
  if (!sg) return;
  DeviceGuard g(sg->device);
  cudaDeviceSynchronize();
  if (sg->exec) cudaGraphExecDestroy(sg->exec);
  if (sg->graph) cudaGraphDestroy(sg->graph);
  cudaFree(sg->pos);
  delete sg;
}

}  // extern "C"
