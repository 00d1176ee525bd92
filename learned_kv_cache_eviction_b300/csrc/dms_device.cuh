// dms_device.cuh -- device-side helpers shared by the DMS kernels:
// mbarrier / bulk-copy wrappers (inline PTX for sm_103a), warp reductions,
// bf16 unpacking, and the view of the cache's device state.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dms {

// Sticky device error bits (the host maps them to DMS_ERR_* codes).
constexpr int kErrBitCapacity = 1;
constexpr int kErrBitTimeout = 2;
constexpr int kErrBitLength = 4;  // a caller-supplied length outside [0, capacity] was clamped

// Time limit of every device-side wait on an mbarrier (ns of %globaltimer).
constexpr uint64_t kWaitLimitNs = 1500ull * 1000ull * 1000ull;

// Device state of one cache.  K is stored with a per-slot permutation of the
// 16-byte chunks of each row (chunk c of slot s lives at chunk c ^ (s & 7)),
// so that a contiguous bulk copy of consecutive slots into shared memory can
// be read one row per lane without bank conflicts.  V is stored unpermuted.
//
// The lengths are kept in three generations and the ring in two, so that one
// kernel can read a step's old state from every CTA while it writes the new
// state (the fused append + decode step): the lengths after t appends are
// len[t % 3], and the ring entry (slot, mark) of position p is
// ring[(p / w) & 1][i][p % w].  The third generation of lengths lets a fused
// step start before the previous step has finished: it derives its lengths
// from generation t - 1, which neither the previous step (writing t) nor
// itself (writing t + 1) touches.
//
// FP8 storage (kvf == kKvFp8): a K row is D E4M3 codes followed by one 16-byte
// chunk {K scale, V scale, 0, 0} (float32); a V row is D codes.  The K row
// stride, D + 16 bytes, is an odd number of 16-byte chunks, so 8 consecutive
// rows read at the same column fall into 8 different bank groups with no
// permutation.
constexpr int kKvBf16 = 0;
constexpr int kKvFp8 = 1;

struct CacheView {
  uint4* K;            // bf16: [NH][cap][D/8] 16-byte chunks (bf16 x 8); fp8: [NH][cap][D/16 + 1]
  uint4* V;            // bf16: [NH][cap][D/8]; fp8: [NH][cap][D/16]
  int32_t* slot_pos;   // [NH][cap]
  int32_t* ring_slot;  // [2][NH][w]
  uint8_t* ring_flag;  // [2][NH][w]
  int32_t* len;        // [3][NH]
  int32_t* err;        // sticky error bits
  int NH, cap, D, w;
  int kvf;  // kKvBf16 or kKvFp8
};

// Generations of the lengths kept in CacheView::len.
constexpr int kLenGens = 3;

// Generation holding the lengths after t appends (t >= 0).
__host__ __device__ __forceinline__ int64_t len_gen(int64_t t) { return t % kLenGens; }

// Lengths after t appends.
__host__ __device__ __forceinline__ int32_t* len_after(const CacheView& c, int64_t t) {
  return c.len + len_gen(t) * static_cast<int64_t>(c.NH);
}

// Index of the ring entry of position p of head i.
__host__ __device__ __forceinline__ size_t ring_index(int NH, int w, int i, int64_t p) {
  return (static_cast<size_t>((p / w) & 1) * NH + i) * w + static_cast<size_t>(p % w);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false after the time
// limit (the caller latches kErrBitTimeout and stops).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// One bulk (non-tensor) asynchronous copy global -> shared, completing on `bar`
// with `bytes` transaction bytes.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Load with acquire semantics at GPU scope (a flag written by another agent).
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Programmatic dependent launch: wait until the grids this one depends on have
// completed and their writes are visible; allow the next grid in the stream to
// be scheduled (it still waits for this grid's completion before its own wait
// returns).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2^x (PTX ex2.approx, flush-to-zero; ex2(-inf) = +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two bf16 packed in a 32-bit word (element 2j in the low half) -> float2.
// Widening bf16 to fp32 is exact: the bf16 bits become the top half.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace dms
