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

namespace dms {

// Bookkeeping of one append for head i at position t (one thread).  Returns
// the slot written, or -1 if the cache is full (the token is dropped, its ring
// entry records "no slot, keep", and the capacity error is latched).
__device__ __forceinline__ int append_bookkeeping(const CacheView& c, int i, int64_t t, float logit,
                                                  int& len_reg) {
  const int r = static_cast<int>(t % c.w);
  int32_t* rs = c.ring_slot + static_cast<size_t>(i) * c.w;
  uint8_t* rf = c.ring_flag + static_cast<size_t>(i) * c.w;
  int s;
  if (t >= c.w && rf[r]) {
    s = rs[r];  // token t - w leaves; token t takes its slot
  } else if (len_reg < c.cap) {
    s = len_reg++;
  } else {
    s = -1;
    atomicOr(c.err, kErrBitCapacity);
  }
  rs[r] = s;
  rf[r] = (s >= 0 && logit > 0.0f) ? 1 : 0;
  if (s >= 0) c.slot_pos[static_cast<size_t>(i) * c.cap + s] = static_cast<int32_t>(t);
  return s;
}

// One warp per (sequence, KV head).  Lane 0 does the bookkeeping; the warp
// then copies the K row (chunk-permuted by slot) and the V row with 16-byte
// stores.  k, v: [NH][D/8] chunks; logit: [NH].
template <int D>
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
    int len_reg = c.len[i];
    s = append_bookkeeping(c, i, t, logit[i], len_reg);
    c.len[i] = len_reg;
  }
  s = __shfl_sync(0xffffffffu, s, 0);
  if (s < 0) return;
  const size_t row = (static_cast<size_t>(i) * c.cap + s) * CH;
  if (lane < CH) {
    c.K[row + (lane ^ (s & 7))] = __ldg(k + static_cast<size_t>(i) * CH + lane);
  } else if (lane < 2 * CH) {
    const int ch = lane - CH;
    c.V[row + ch] = __ldg(v + static_cast<size_t>(i) * CH + ch);
  }
}

// `chunk` appends per (sequence, KV head) in position order, one warp per
// head.  Lane 0 assigns the slots of up to 32 tokens at a time sequentially
// (bit-identical to single appends, including chains where a token retires
// another token of the same chunk); then the warp copies those rows, skipping
// a row whose slot a later token of the same batch takes over (that token
// retired it), so that no slot is written twice by one batch.
// k, v: [NH][chunk][D/8] chunks; logits: [NH][chunk].
template <int D>
__global__ void __launch_bounds__(128) append_chunk_kernel(CacheView c, const uint4* __restrict__ k,
                                                           const uint4* __restrict__ v,
                                                           const float* __restrict__ logits, int64_t t0,
                                                           int chunk) {
  constexpr int CH = D / 8;
  __shared__ int slots_smem[4][32];
  griddep_wait();
  griddep_launch_dependents();
  const int wl = threadIdx.x >> 5;
  const int i = static_cast<int>(blockIdx.x * 4 + wl);
  const int lane = threadIdx.x & 31;
  if (i >= c.NH) return;
  int* slots = slots_smem[wl];
  int len_reg = c.len[i];
  for (int base = 0; base < chunk; base += 32) {
    const int n = min(32, chunk - base);
    if (lane == 0) {
      for (int j = 0; j < n; ++j) {
        const float lg = logits[static_cast<size_t>(i) * chunk + base + j];
        const int s = append_bookkeeping(c, i, t0 + base + j, lg, len_reg);
        slots[j] = s;
        // Token j took the slot of token j - w (which it retired): if that token
        // is in this batch, it is not copied, so the slot is written once.
        if (s >= 0 && j >= c.w && slots[j - c.w] == s) slots[j - c.w] = -1;
      }
    }
    __syncwarp();
    // n rows x (CH K chunks + CH V chunks)
    for (int idx = lane; idx < n * 2 * CH; idx += 32) {
      const int j = idx / (2 * CH);
      const int q = idx % (2 * CH);
      const int s = slots[j];
      if (s < 0) continue;
      const size_t src = (static_cast<size_t>(i) * chunk + base + j) * CH;
      const size_t row = (static_cast<size_t>(i) * c.cap + s) * CH;
      if (q < CH) {
        c.K[row + (q ^ (s & 7))] = __ldg(k + src + q);
      } else {
        c.V[row + (q - CH)] = __ldg(v + src + (q - CH));
      }
    }
    __syncwarp();
  }
  if (lane == 0) c.len[i] = len_reg;
}

// Logical-order copy of the K and V pools (undoes the chunk permutation of K).
// One thread per 16-byte chunk.
template <int D>
__global__ void export_kv_kernel(CacheView c, uint4* __restrict__ k_out, uint4* __restrict__ v_out) {
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

}  // namespace dms
