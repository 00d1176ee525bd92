// append.cuh -- the fused append/evict kernels of the DMS compacted cache.
//
// Method ("Inference-Time Hyper-Scaling with KV Cache Compression", AI
// research-map summary, "Approach"): every (token, KV head) carries a binary
// eviction decision whose eviction is executed after a delay window of w
// tokens.  At inference the decision is sigmoid(logit) > 0.5, evaluated here
// as the float32 compare logit > 0.
//
// Slot policy (the pages give none; this is the reading used throughout):
// at the append of token t, if t >= w and token t - w was marked, t - w
// leaves and token t takes its slot; otherwise token t takes slot len and len
// grows.  So slots [0, len) always hold exactly the retained tokens and the
// decode kernel reads a dense prefix of each head's pool.
#pragma once

#include "dms_device.cuh"
#include "fp8.cuh"

namespace dms {

// Bookkeeping of one append for head i at position t (one thread).  Returns
// the slot written, or -1 if the cache is full (the token is dropped, its ring
// entry records "no slot, keep", and the capacity error is latched).
__device__ __forceinline__ int append_bookkeeping(const CacheView& c, int i, int64_t t, float logit,
                                                  int& len_reg) {
  int s;
  const size_t old = t >= c.w ? ring_index(c.NH, c.w, i, t - c.w) : 0;
  if (t >= c.w && c.ring_flag[old]) {
    s = c.ring_slot[old];  // token t - w leaves; token t takes its slot
  } else if (len_reg < c.cap) {
    s = len_reg++;
  } else {
    s = -1;
    atomicOr(c.err, kErrBitCapacity);
  }
  const size_t now = ring_index(c.NH, c.w, i, t);
  c.ring_slot[now] = s;
  c.ring_flag[now] = (s >= 0 && logit > 0.0f) ? 1 : 0;
  if (s >= 0) c.slot_pos[static_cast<size_t>(i) * c.cap + s] = static_cast<int32_t>(t);
  return s;
}

// One warp per (sequence, KV head).  Lane 0 does the bookkeeping; the warp
// then stores the row: bf16, the K row (chunk-permuted by slot) and the V row
// with 16-byte stores; fp8, both rows quantized.  k, v: [NH][D/8] chunks;
// logit: [NH].
template <int D, int KVF = kKvBf16>
__global__ void __launch_bounds__(256) append_kernel(CacheView c, const uint4* __restrict__ k,
                                                     const uint4* __restrict__ v,
                                                     const float* __restrict__ logit, int64_t t) {
  constexpr int CH = D / 8;
  griddep_wait();
  griddep_launch_dependents();
  const int i = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= c.NH) return;
  int s = -1;
  if (lane == 0) {
    int len_reg = len_after(c, t)[i];
    s = append_bookkeeping(c, i, t, logit[i], len_reg);
    len_after(c, t + 1)[i] = len_reg;
  }
  s = __shfl_sync(0xffffffffu, s, 0);
  if (s < 0) return;
  if constexpr (KVF == kKvFp8) {
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (lane < CH) x = __ldg(k + static_cast<size_t>(i) * CH + lane);
    else if (lane < 2 * CH) x = __ldg(v + static_cast<size_t>(i) * CH + lane - CH);
    const size_t slot = static_cast<size_t>(i) * c.cap + s;
    quantize_kv_rows<D>(x, reinterpret_cast<uint8_t*>(c.K) + slot * (D + 16),
                        reinterpret_cast<uint8_t*>(c.V) + slot * D, lane);
    return;
  }
  const size_t row = (static_cast<size_t>(i) * c.cap + s) * CH;
  if (lane < CH) {
    c.K[row + (lane ^ (s & 7))] = __ldg(k + static_cast<size_t>(i) * CH + lane);
  } else if (lane < 2 * CH) {
    const int ch = lane - CH;
    c.V[row + ch] = __ldg(v + static_cast<size_t>(i) * CH + ch);
  }
}

// Bookkeeping of `chunk` appends (positions t0 .. t0 + chunk - 1) per
// (sequence, KV head), bit-identical to that many single appends; one warp per
// head, 32 tokens at a time, lane j taking token base + j.
//   * Token t retires token t - w if that one was stored and marked; it then
//     takes its slot.  Lanes j and j + w of a batch depend on each other, lanes
//     closer than w do not: the batch is resolved in runs of w lanes, each run
//     with one ballot (which lanes need a fresh slot), a prefix count (their
//     order) and two shuffles (the slot and mark of token t - w).
//   * For w <= 32 the state of the tokens before a batch comes from the
//     previous batch's lanes by shuffles; for larger w, and for the first
//     batch, from the ring in memory.
//   * Lengths and ring are the double-buffered state of CacheView: read at
//     t0, written at t0 + chunk.
//   * Fresh slots are handed out in position order from len; beyond the
//     capacity a token is dropped (ring entry "no slot, keep") and the
//     capacity error is latched, as for a single append.
// The slot -> position map, the ring and len are written here; the K/V rows
// are copied by append_chunk_copy_kernel from the final slot -> position map.
__global__ void __launch_bounds__(128) append_chunk_slots_kernel(CacheView c, const float* __restrict__ logits,
                                                                 int64_t t0, int chunk) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= c.NH) return;
  const int w = c.w;
  int32_t* sp = c.slot_pos + static_cast<size_t>(i) * c.cap;
  int len = len_after(c, t0)[i];
  bool overflow = false;
  int slot = -1, flag = 0;  // this lane's token in the current (then previous) batch
  for (int base = 0; base < chunk; base += 32) {
    const int n = min(32, chunk - base);
    const bool active = lane < n;
    const int64_t t = t0 + base + lane;
    const bool marked = active && logits[static_cast<size_t>(i) * chunk + base + lane] > 0.0f;
    // Token t - w for lanes where it precedes this batch (lane < w).
    int rslot = -1, rflag = 0;
    if (w <= 32 && base > 0) {  // the previous batch was full: t - w was its lane 32 - w + lane
      rslot = __shfl_sync(0xffffffffu, slot, (lane + 32 - w) & 31);
      rflag = __shfl_sync(0xffffffffu, flag, (lane + 32 - w) & 31);
    } else if (active && lane < w && t >= w) {
      const size_t e = ring_index(c.NH, w, i, t - w);
      rslot = c.ring_slot[e];
      rflag = c.ring_flag[e];
    }
    slot = -1;
    flag = 0;
    for (int sb = 0; sb < n; sb += w) {  // run of lanes [sb, sb + w)
      const bool in_run = active && lane >= sb && lane < sb + w;
      const int src = lane >= w ? lane - w : 0;
      const int pslot = __shfl_sync(0xffffffffu, slot, src);
      const int pflag = __shfl_sync(0xffffffffu, flag, src);
      bool retire = false;
      int rslot_eff = -1;
      if (t >= w) {
        retire = (lane >= w ? pflag : rflag) != 0;
        rslot_eff = lane >= w ? pslot : rslot;
      }
      const bool fresh = in_run && !retire;
      const unsigned m = __ballot_sync(0xffffffffu, fresh);
      const int rank = __popc(m & ((1u << lane) - 1u));
      const int room = c.cap - len;
      if (in_run) {
        slot = retire ? rslot_eff : (rank < room ? len + rank : -1);
        flag = (slot >= 0 && marked) ? 1 : 0;
      }
      const int nf = __popc(m);
      if (nf > room) overflow = true;
      len += min(nf, room);
    }
    // A lane whose slot lane + w of this batch took (it retired this token) does
    // not record its position; the later token's entry is the one that stays.
    const int nxt = __shfl_sync(0xffffffffu, slot, (lane + w) & 31);
    const bool superseded = w < 32 && lane + w < n && slot >= 0 && nxt == slot;
    if (active && slot >= 0 && !superseded) sp[slot] = static_cast<int32_t>(t);
    // The ring keeps the last 2w positions (two generations of w): each batch
    // writes the entries of its lanes that no later lane of the batch (2w
    // positions on, same entry) overwrites.
    if (active && lane + 2 * w >= n) {
      const size_t e = ring_index(c.NH, w, i, t);
      c.ring_slot[e] = slot;
      c.ring_flag[e] = static_cast<uint8_t>(flag);
    }
    __syncwarp();
  }
  if (lane == 0) {
    len_after(c, t0 + chunk)[i] = len;
    if (overflow) atomicOr(c.err, kErrBitCapacity);
  }
}

// K/V rows of a chunk appended by append_chunk_slots_kernel: every slot whose
// final position lies in [t0, t0 + chunk) receives that token's row (a token
// retired within the same chunk is no longer in the map, so each slot is
// written once).  Grid: (slot groups of 256, heads); one warp per 32 slots,
// one coalesced row (K chunks permuted by slot, then V) per step; fp8 caches
// quantize the row instead.
template <int D, int KVF = kKvBf16>
__global__ void __launch_bounds__(256) append_chunk_copy_kernel(CacheView c, const uint4* __restrict__ k,
                                                                const uint4* __restrict__ v, int64_t t0,
                                                                int chunk) {
  constexpr int CH = D / 8;
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int s0 = (static_cast<int>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * 32;
  const int L = len_after(c, t0 + chunk)[i];
  if (s0 >= L) return;
  const int s = s0 + lane;
  const int p = s < L ? c.slot_pos[static_cast<size_t>(i) * c.cap + s] : -1;
  unsigned m = __ballot_sync(0xffffffffu, p >= t0 && p < t0 + chunk);
  while (m) {
    const int src = __ffs(m) - 1;
    m &= m - 1;
    const int ss = s0 + src;
    const int tok = __shfl_sync(0xffffffffu, p, src) - static_cast<int>(t0);
    const size_t in = (static_cast<size_t>(i) * chunk + tok) * CH;
    if constexpr (KVF == kKvFp8) {
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (lane < CH) x = __ldg(k + in + lane);
      else if (lane < 2 * CH) x = __ldg(v + in + lane - CH);
      const size_t slot = static_cast<size_t>(i) * c.cap + ss;
      quantize_kv_rows<D>(x, reinterpret_cast<uint8_t*>(c.K) + slot * (D + 16),
                          reinterpret_cast<uint8_t*>(c.V) + slot * D, lane);
      continue;
    }
    const size_t row = (static_cast<size_t>(i) * c.cap + ss) * CH;
    if (lane < CH) {
      c.K[row + (lane ^ (ss & 7))] = __ldg(k + in + lane);
    } else if (lane < 2 * CH) {
      c.V[row + lane - CH] = __ldg(v + in + lane - CH);
    }
  }
}

// Self-test of the device-side time limit: one warp waits, with the same
// bounded wait the kernels use, on an mbarrier that nothing ever completes; the
// wait gives up after its limit and the timeout is latched in the cache's error
// word, as a real wait that ran out would.  Launched only by
// dms_cache_selftest_wait.
__global__ void wait_selftest_kernel(int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0);
  if (!ok && threadIdx.x == 0) atomicOr(err, kErrBitTimeout);
}

// Logical-order copy of the K and V pools (undoes the chunk permutation of K).
// One thread per 16-byte chunk.  fp8: the codes only, [NH][cap][D] bytes each
// (export_scales_kernel copies the scales).
template <int D, int KVF = kKvBf16>
__global__ void export_kv_kernel(CacheView c, uint4* __restrict__ k_out, uint4* __restrict__ v_out) {
  if constexpr (KVF == kKvFp8) {
    constexpr int U = D / 16;  // 16-byte chunks of codes per row
    const size_t n = static_cast<size_t>(c.NH) * c.cap * U;
    for (size_t x = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; x < n;
         x += static_cast<size_t>(gridDim.x) * blockDim.x) {
      const size_t row = x / U;
      k_out[x] = c.K[row * (U + 1) + x % U];
      v_out[x] = c.V[x];
    }
    return;
  }
  constexpr int CH = D / 8;
  const size_t n = static_cast<size_t>(c.NH) * c.cap * CH;
  for (size_t x = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; x < n;
       x += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t row = x / CH;
    const int ch = static_cast<int>(x % CH);
    const int s = static_cast<int>(row % c.cap);
    k_out[x] = c.K[row * CH + (ch ^ (s & 7))];
    v_out[x] = c.V[x];
  }
}

// fp8 caches: the K and V scales of every slot, [NH][cap] float32 each.
template <int D>
__global__ void export_scales_kernel(CacheView c, float* __restrict__ k_scale, float* __restrict__ v_scale) {
  const size_t n = static_cast<size_t>(c.NH) * c.cap;
  for (size_t x = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; x < n;
       x += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float2 sc = *reinterpret_cast<const float2*>(reinterpret_cast<const uint8_t*>(c.K) + x * (D + 16) + D);
    k_scale[x] = sc.x;
    v_scale[x] = sc.y;
  }
}

// Positions of caches whose steps are replayed from a CUDA graph: the last
// node of the graph advances each cache's position word by one, and a launch
// after calls made outside the graph first re-sends the host's position.
__global__ void advance_positions_kernel(int64_t* const* __restrict__ pos, int n) {
  griddep_wait();
  for (int i = threadIdx.x; i < n; i += blockDim.x) *pos[i] += 1;
}

__global__ void set_position_kernel(int64_t* pos, int64_t value) {
  griddep_wait();
  *pos = value;
}

}  // namespace dms
