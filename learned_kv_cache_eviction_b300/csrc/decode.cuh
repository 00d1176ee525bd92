// decode.cuh -- split-K GQA decode attention over the DMS compacted caches.
//
// What it computes: for every sequence b and query head g, softmax attention
// of q[b][g] over the retained keys of KV head h = g / G (G = Hq / Hkv).  The
// retained keys of (b, h) are exactly slots [0, len) of its pool (the slot
// policy in append.cuh keeps them dense), so the kernel reads only the
// retained K/V bytes -- the cost the method is built to cut (notes page of
// "Inference-Time Hyper-Scaling with KV Cache Compression", section
// "研究背景与动机": each decode step reads the whole KV cache; the AI
// research-map summary, "Experimental setup", counts "KV-cache token reads").
//
// Work split ("balanced by retained length"): the concatenation of all heads'
// retained slots, S = sum(len) slots, is cut into Pe equal contiguous ranges,
// one per warp of a persistent grid (one CTA of up to 12 warps per SM, so that
// each of the SM's four schedulers gets the same number of warps).  Each warp is
// an independent flash-decoding worker:
//   * lane 0 streams its range in tiles of TK = 16 slots (K tile and V tile,
//     each one contiguous bulk copy global -> shared completing on an
//     mbarrier), NST = 2 tiles per warp in flight; when a tile opens a new
//     head, the lanes also load that head's G query rows into registers, to be
//     widened into shared memory when the head's first tile is consumed;
//   * QK: lanes r and r + 16 score slot r of the tile over one half of the
//     head dim each (K rows are chunk-permuted in the pool, so these reads are
//     free of bank conflicts while q is read as a broadcast), then add;
//   * online softmax in fp32, base 2 (q is pre-scaled by scale * log2 e);
//   * PV: lane owns D/32 output elements of all G heads; packed fp32 FMAs.
// A head covered by one warp is normalised and written directly.  A head split
// across warps leaves one partial (max, sum, unnormalised acc) per warp; each
// such warp then increments the head's arrival counter, and the warp that
// arrives last merges the partials and writes the output (and resets the
// counter for the next call).  No warp ever waits for another.
#pragma once

#include "dms_device.cuh"
#include "fp8.cuh"

namespace dms {

template <int D_, int G_, int KVF_ = kKvBf16>
struct DecodeShape {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr int KVF = KVF_;
  static constexpr bool FP8 = KVF == kKvFp8;
  // Slots per tile: 16 (bf16; lanes r and r + 16 score slot r over the two
  // halves of D), or 32 (fp8; the same two lanes score slots r and r + 16, so
  // each q load serves two slots).
  static constexpr int TK = FP8 ? 32 : 16;
  static constexpr int NST = 2;                 // tiles in flight per warp
  static constexpr int CH = D / 8;              // 16-byte chunks per bf16 row
  static constexpr int HCH = CH / 2;            // chunks per half row (two lanes score one slot)
  static constexpr int EL = D / 32;             // output elements per lane in PV
  // Row bytes in HBM and in the tiles: bf16 2 D each; fp8 D codes, the K row
  // followed by its 16-byte scale chunk.
  static constexpr int ROWB_K = FP8 ? D + 16 : 2 * D;
  static constexpr int ROWB_V = FP8 ? D : 2 * D;
  static constexpr int KU4 = ROWB_K / 16;       // 16-byte units per row
  static constexpr int VU4 = ROWB_V / 16;
  static constexpr int TILEB_K = TK * ROWB_K;
  static constexpr int TILEB_V = TK * ROWB_V;
  // qs: fp32 q, per head g two half rows of D/2 floats, padded by 4 floats so
  // that the two lane halves read different banks.
  static constexpr int QHALF = D / 2 + 4;
  static constexpr int QROW = 2 * QHALF;
  // p buffer: per slot, the G probabilities as (p, p) pairs (operands of the
  // packed fp32 FMA), padded to a multiple of 4 floats.
  static constexpr int PROW = (2 * G + 3) / 4 * 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = NST * TILEB_K;
  static constexpr int OFF_QS = NST * (TILEB_K + TILEB_V);
  static constexpr int QV = (G * D / 8 + 31) / 32;  // 16-byte q chunks per lane
  static constexpr int OFF_P = OFF_QS + ((G * QROW * 4 + 15) / 16) * 16;
  static constexpr int OFF_BAR = OFF_P + TK * PROW * 4;
  // Fused step: per-warp state kept in shared memory rather than in registers
  // (the decode loop has none to spare): the new token's slots of the first
  // FX_HEADS heads of the warp's range, the first head, the current segment's,
  // and the step's position.
  static constexpr int FX_HEADS = 12;
  static constexpr int FX_I0 = FX_HEADS, FX_SEG = FX_HEADS + 1;
  static constexpr int FX_T = FX_HEADS + 2;  // the step's position t (int64, two slots)
  static constexpr int OFF_FX = OFF_BAR + NST * 8;
  static constexpr int FX_BYTES = FP8 ? 0 : (FX_HEADS + 2) * 4;  // the fused step is bf16 only
  static constexpr int WARP_BYTES = ((OFF_FX + FX_BYTES + 127) / 128) * 128;
  static constexpr int kSmemBudget = 227 * 1024 - 1024;  // leaves room for static shared memory
  // Warps per CTA: 12 (three per scheduler) where the shared memory allows.  With
  // three warps on a scheduler its register file leaves 168 registers per thread;
  // G >= 5 needs more, so those shapes run two warps per scheduler.
  static constexpr int NW_CAP = G >= 5 ? 8 : 12;
  static constexpr int NW = (kSmemBudget / WARP_BYTES) < NW_CAP ? (kSmemBudget / WARP_BYTES) : NW_CAP;
  static constexpr int SMEM = NW * WARP_BYTES;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(G >= 1 && G <= 8, "1 <= G <= 8");
  static_assert(NW >= 4, "at least four warps per CTA");
};

// Largest number of warps per CTA of any instantiation (sizes the partials).
constexpr int kMaxWarpsPerCta = 12;

// Fewest retained slots a warp is given (two tiles; bounds the number of
// partials when the cache is small).  Small caches are latency-bound per warp,
// so they are spread over as many warps as this allows.
constexpr int kMinSlotsPerWarp = 32;

struct DecodeArgs {
  const uint4* K;
  const uint4* V;
  const int32_t* len;
  const uint16_t* q;  // bf16 [B][Hq][D]
  float* out;         // fp32 [B][Hq][D]
  float* part_acc;    // [entries][G][D]
  float* part_ml;     // [entries][G][2]
  int32_t* head_cnt;  // [NH * nsplit] arrival counters of split (virtual) heads; zero between calls
  int32_t* err;
  int NH, Hkv, cap;
  float qscale;  // scale * log2(e)
  // Query heads per KV head (the q / out row stride), and how many groups of
  // G of them each KV head is split into (1, or 2 when Gq = 2 G).  With two
  // groups the kernel works on 2 NH virtual heads: virtual head v is KV head
  // v mod NH with query heads [(v / NH) G, (v / NH + 1) G) of its group.  Both
  // groups stream the same K/V rows, at about the same time, so the second
  // read is mostly served by L2.
  int Gq, nsplit;
  // Fused step only (decode_kernel<D, G, true>, dms_step): the new token of
  // position t is appended in the same launch.  `len` is then the base of the
  // double-buffered lengths [2][NH] (see CacheView): the kernel decodes over
  // the lengths after the token and writes those, the token's ring entry, slot
  // map entry and K/V row into the other halves of the double-buffered state,
  // which no CTA reads.  The position t comes from `t`, or, when t_dev is set
  // (a step replayed from a CUDA graph), from device memory.
  const uint4* k_new;     // [NH][D/8] the new token's K and V
  const uint4* v_new;
  const float* logit_new;  // [NH]
  uint4* K_w;             // the K and V pools, writable
  uint4* V_w;
  int32_t* slot_pos;      // [NH][cap]
  int32_t* ring_slot;     // [2][NH][w]
  uint8_t* ring_flag;     // [2][NH][w]
  int32_t* len_w;         // [2][NH] the lengths, writable
  const int64_t* t_dev;   // graph-replayed steps: the cache's position in device memory
  int64_t t;
  int w;
};

// The new token's slot in head x for the fused step at position t: the slot of
// token t - w if that token was stored and marked (it leaves now), else the
// next free slot, else -1 (capacity exceeded).  Reads only the state before
// the step.
__device__ __forceinline__ int fused_new_slot(const DecodeArgs& a, int64_t t, int x, int L_old) {
  if (t >= a.w) {
    const size_t e = ring_index(a.NH, a.w, x, t - a.w);
    if (a.ring_flag[e]) return a.ring_slot[e];
  }
  return L_old < a.cap ? L_old : -1;
}

// Not inlined: the slot lookup of a head beyond the first FX_HEADS of a warp's
// range (rare), kept out of the decode loop's code.
static __device__ __noinline__ int fused_new_slot_far(const DecodeArgs& a, int64_t t, int x) {
  return fused_new_slot(a, t, x, a.len[(t & 1) * a.NH + x]);
}

// Fused step, not inlined (once per head, in the warp whose tile holds the new
// token's slot): overwrite row j of the staged tile with the new token's K row
// (at the pool's chunk order for slot s_new) and V row from the step's input.
// The tile's copy of that pool row is discarded: the row is being written in
// the same launch.  The proxy fence orders these stores before the bulk copy
// that next refills the buffer.
static __device__ __noinline__ void patch_new_row(const DecodeArgs& a, uint4* Kt, uint4* Vt, int i, int j, int s_new,
                                                  int CH, int lane) {
  if (lane < CH) {
    Kt[j * CH + (lane ^ (s_new & 7))] = __ldg(a.k_new + static_cast<size_t>(i) * CH + lane);
  } else if (lane < 2 * CH) {
    Vt[j * CH + lane - CH] = __ldg(a.v_new + static_cast<size_t>(i) * CH + lane - CH);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// Retained length of head x as this launch decodes it (fused: after the
// append of position t).
template <bool FUSED>
__device__ __forceinline__ int decode_len(const DecodeArgs& a, int64_t t, int x) {
  if constexpr (FUSED) {
    const int L = a.len[(t & 1) * a.NH + x];
    const bool retire = t >= a.w && a.ring_flag[ring_index(a.NH, a.w, x, t - a.w)] != 0;
    return (!retire && L < a.cap) ? L + 1 : L;
  }
  return a.len[x];
}

// Retained-slot iterator over one warp's global range [A, E).
struct TileIter {
  int i;      // head
  int L;      // retained length of head i
  int s;      // next slot in head i
  int send;   // end of this warp's slots in head i
  int64_t P;  // global index of slot 0 of head i
  int64_t E;
  bool valid;
  bool first;  // next tile opens a new segment (head)

  template <typename LenF>
  __device__ __forceinline__ void start(const LenF& len, int i0, int64_t P0, int64_t A, int64_t E_) {
    i = i0;
    P = P0;
    E = E_;
    L = len(i0);
    s = static_cast<int>(A - P0);
    send = static_cast<int>(min(E, P0 + L) - P0);
    valid = s < send;
    first = true;
  }
  template <typename LenF>
  __device__ __forceinline__ void advance(const LenF& len, int NH, int cnt) {
    s += cnt;
    first = false;
    if (s < send) return;
    P += L;
    ++i;
    while (P < E && i < NH) {
      L = len(i);
      if (L > 0) break;
      ++i;
    }
    if (P >= E || i >= NH) {
      valid = false;
      return;
    }
    s = 0;
    send = static_cast<int>(min(E, P + L) - P);
    first = true;
  }
};

// Exclusive prefix sums of len[0..NH) into pre[0..NH] (shared memory) by the
// whole CTA, reading each length from global memory once.
template <typename LenF>
__device__ __forceinline__ void scan_lengths(const LenF& len, int NH, int* pre) {
  __shared__ int wsum[32];
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int x = tid; x < NH; x += nt) pre[x] = len(x);
  __syncthreads();
  const int per = (NH + nt - 1) / nt;
  const int b0 = min(NH, tid * per), b1 = min(NH, b0 + per);
  int sum = 0;
  for (int x = b0; x < b1; ++x) sum += pre[x];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int v = lane < (nt >> 5) ? wsum[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    wsum[lane] = inc - v;
  }
  __syncthreads();
  // Each thread rewrites only its own range [b0, b1), which no other thread reads.
  int run = wsum[wid] + incl - sum;
  for (int x = b0; x < b1; ++x) {
    const int l = pre[x];
    pre[x] = run;
    run += l;
  }
  if (tid == nt - 1) pre[NH] = run;
  __syncthreads();
}

// Merge the nseg partials (max m, sum l, unnormalised acc) of one head, stored
// at consecutive partial indices base, base + 1, ..., and write the normalised
// output (outp already offset by lane * EL).  Partials written by other SMs are
// read from L2 (ld.global.cg).  Pass 1 reduces (max, sum) with the segments
// spread over the lanes, each lane keeping its first segment's values; pass 2
// takes 32 segments at a time, each lane computing one segment's weight,
// broadcast by shuffles while the accumulators' loads of several segments are
// in flight together.
template <int D, int G>
__device__ __forceinline__ void merge_partials(const DecodeArgs& a, size_t base, int nseg, float* outp, int lane) {
  constexpr int EL = D / 32;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
  float M[G], L[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = -INFINITY;
    L[g] = 0.f;
  }
  float2 v0[G];  // this lane's segment among the first 32, kept for pass 2
  for (int k = lane; k < nseg; k += 32) {
    float2 v[G];
#pragma unroll
    for (int g = 0; g < G; ++g) v[g] = __ldcg(ml + (base + k) * G + g);
    if (k == lane) {
#pragma unroll
      for (int g = 0; g < G; ++g) v0[g] = v[g];
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mn = fmaxf(M[g], v[g].x);
      L[g] = L[g] * fast_exp2(M[g] - mn) + v[g].y * fast_exp2(v[g].x - mn);
      M[g] = mn;
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float Mo = __shfl_xor_sync(0xffffffffu, M[g], off);
      const float Lo = __shfl_xor_sync(0xffffffffu, L[g], off);
      const float mn = fmaxf(M[g], Mo);
      if (mn != -INFINITY) {
        L[g] = L[g] * fast_exp2(M[g] - mn) + Lo * fast_exp2(Mo - mn);
        M[g] = mn;
      }
    }
  }
  float2 acc[G][EL / 2];
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int e = 0; e < EL / 2; ++e) acc[g][e] = make_float2(0.f, 0.f);
  }
  for (int kb = 0; kb < nseg; kb += 32) {
    float wv[G];
    const int k = kb + lane;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mk = kb == 0 ? v0[g].x : (k < nseg ? __ldcg(ml + (base + k) * G + g).x : 0.f);
      wv[g] = k < nseg ? fast_exp2(mk - M[g]) : 0.f;
    }
    const int n = min(32, nseg - kb);
#pragma unroll 4
    for (int j = 0; j < n; ++j) {
      const size_t kk = base + kb + j;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float wk = __shfl_sync(0xffffffffu, wv[g], j);
        const float2* src = reinterpret_cast<const float2*>(a.part_acc + (kk * G + g) * D + lane * EL);
#pragma unroll
        for (int e = 0; e < EL / 2; ++e) acc[g][e] = __ffma2_rn(make_float2(wk, wk), __ldcg(src + e), acc[g][e]);
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float inv = 1.f / L[g];
#pragma unroll
    for (int e = 0; e < EL / 2; ++e)
      reinterpret_cast<float2*>(outp + g * D)[e] = make_float2(acc[g][e].x * inv, acc[g][e].y * inv);
  }
}

template <int D, int G, bool FUSED, int KVF = kKvBf16>
__global__ void __launch_bounds__(DecodeShape<D, G, KVF>::NW * 32, 1) decode_kernel(const DecodeArgs a) {
  using Sh = DecodeShape<D, G, KVF>;
  static_assert(!(FUSED && Sh::FP8), "the fused step stores bf16 rows");
  constexpr int NW = Sh::NW, TK = Sh::TK, NST = Sh::NST, CH = Sh::CH, HCH = Sh::HCH, EL = Sh::EL;
  constexpr int ROWB_K = Sh::ROWB_K, ROWB_V = Sh::ROWB_V, TILEB_K = Sh::TILEB_K, TILEB_V = Sh::TILEB_V;
  constexpr int QHALF = Sh::QHALF, QROW = Sh::QROW, PROW = Sh::PROW;
  extern __shared__ __align__(1024) uint8_t smem[];

  // Launched as a programmatic dependent of the previous kernel: everything the
  // previous kernels wrote is visible after this wait.
  griddep_wait();
  griddep_launch_dependents();

  // ---- prologue: prefix sums of the retained lengths, warp ranges ----
  const int wl = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wg = static_cast<int64_t>(blockIdx.x) * NW + wl;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * NW;
  // The step's position (fused step only): a kernel argument, or read from
  // device memory when the launch is replayed from a CUDA graph.
  int64_t t_step = a.t;
  if constexpr (FUSED) {
    if (a.t_dev != nullptr) t_step = __ldcg(a.t_dev);
  }
  // Virtual heads (see DecodeArgs::nsplit) and the KV head / query-head group of each.
  const int NV = a.NH * a.nsplit;
  auto real_head = [&](int v) { return v >= a.NH ? v - a.NH : v; };
  auto head_group = [&](int v) { return v >= a.NH ? 1 : 0; };
  int* pre = reinterpret_cast<int*>(smem);  // [NV + 1]; aliases the warp regions until the barrier below
  int* sn = pre + NV + 1;                   // fused step: [NH] the new token's slot in each KV head
  // Fused step: warp x of the grid appends the token to head x (and x + nwarps,
  // ...).  Its row chunk (K for lanes < CH, V for lanes CH .. 2 CH - 1) and
  // logit are loaded now, in flight during the scan.
  uint4 own_row = make_uint4(0u, 0u, 0u, 0u);
  float own_logit = 0.f;
  if constexpr (FUSED) {
    if (wg < a.NH) {
      if (lane < 2 * CH)
        own_row = __ldg((lane < CH ? a.k_new : a.v_new) + static_cast<size_t>(wg) * CH + (lane % CH));
      own_logit = __ldg(a.logit_new + wg);
    }
  }
  // The scan reads each head's length (and, fused, the ring entry of t - w) once;
  // the fused scan also records the new token's slot in sn.
  auto scanf = [&](int v) {
    const int x = real_head(v);
    if constexpr (FUSED) {
      const int L = a.len[(t_step & 1) * a.NH + x];
      int fl = 0, sl = 0;
      if (t_step >= a.w) {
        const size_t e = ring_index(a.NH, a.w, x, t_step - a.w);
        fl = a.ring_flag[e];
        sl = a.ring_slot[e];
      }
      if (v < a.NH) sn[x] = fl ? sl : (L < a.cap ? L : -1);
      return (fl || L >= a.cap) ? L : L + 1;
    } else {
      return a.len[x];
    }
  };
  scan_lengths(scanf, NV, pre);
  if constexpr (FUSED) {
    // Bookkeeping and row of the new token; none of it is read by this launch
    // (other halves of the double-buffered state, the slot map, and a pool row
    // that every tile copy skips: the new row is copied from the input).
    for (int64_t x = wg; x < a.NH; x += nwarps) {
      const int i = static_cast<int>(x);
      const int s_new = sn[i];
      uint4 rowc = own_row;
      float lg = own_logit;
      if (x != wg) {
        if (lane < 2 * CH) rowc = __ldg((lane < CH ? a.k_new : a.v_new) + static_cast<size_t>(i) * CH + (lane % CH));
        lg = __ldg(a.logit_new + i);
      }
      if (lane == 0) {
        a.len_w[((t_step + 1) & 1) * a.NH + i] = pre[i + 1] - pre[i];
        const size_t e = ring_index(a.NH, a.w, i, t_step);
        a.ring_slot[e] = s_new;
        a.ring_flag[e] = (s_new >= 0 && lg > 0.0f) ? 1 : 0;
        if (s_new >= 0) a.slot_pos[static_cast<size_t>(i) * a.cap + s_new] = static_cast<int32_t>(t_step);
        else atomicOr(a.err, kErrBitCapacity);
      }
      if (s_new >= 0) {
        const size_t row = (static_cast<size_t>(i) * a.cap + s_new) * CH;
        if (lane < CH) a.K_w[row + (lane ^ (s_new & 7))] = rowc;
        else if (lane < 2 * CH) a.V_w[row + lane - CH] = rowc;
      }
    }
  }
  const int64_t S = pre[NV];
  int64_t Pe = nwarps;
  if (S / kMinSlotsPerWarp < Pe) Pe = S / kMinSlotsPerWarp;
  if (Pe < 1) Pe = 1;
  const bool active = S > 0 && wg < Pe;
  int64_t A = 0, E = 0, P0 = 0;
  int i0 = 0;
  if (active) {
    A = (wg * S) / Pe;
    E = ((wg + 1) * S) / Pe;
    int lo = 0, hi = NV;  // pre[lo] <= A < pre[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] <= A) lo = mid; else hi = mid;
    }
    i0 = lo;
    P0 = pre[lo];
  }
  // Fused step: the new token's slots of heads i0, i0 + 1, ... (read before the
  // barrier, which ends the prefix sums' lease on the warp regions).
  int snl = -1;
  if constexpr (FUSED) {
    if (active && lane < Sh::FX_HEADS && i0 + lane < NV) snl = sn[real_head(i0 + lane)];
  }
  __syncthreads();

  if (!active) return;

  // ---- per-warp shared memory ----
  uint8_t* wbase = smem + wl * Sh::WARP_BYTES;
  uint8_t* Ks = wbase + Sh::OFF_K;
  uint8_t* Vs = wbase + Sh::OFF_V;
  float* qs = reinterpret_cast<float*>(wbase + Sh::OFF_QS);
  float* pb = reinterpret_cast<float*>(wbase + Sh::OFF_P);
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + Sh::OFF_BAR);  // [NST] tiles
  int* fx = reinterpret_cast<int*>(wbase + Sh::OFF_FX);               // fused-step state
  if (lane == 0) {
    for (int x = 0; x < NST; ++x) mbar_init(&bars[x], 1);
    fence_barrier_init();
  }
  if constexpr (FUSED) {
    if (lane < Sh::FX_HEADS) fx[lane] = snl;
    if (lane == 0) {
      fx[Sh::FX_I0] = i0;
      fx[Sh::FX_SEG] = -1;
      *reinterpret_cast<int64_t*>(fx + Sh::FX_T) = t_step;
    }
  }
  __syncwarp();
  // Retained length of head x after this launch's append (read per head
  // change; the position comes from shared memory, not a register).
  auto lenf = [&](int v) {
    if constexpr (FUSED) return decode_len<true>(a, *reinterpret_cast<const int64_t*>(fx + Sh::FX_T), real_head(v));
    else return decode_len<false>(a, 0, real_head(v));
  };

  const int Hq = a.Hkv * a.Gq;
  TileIter is{}, cs{};
  is.start(lenf, i0, P0, A, E);
  cs = is;
  int n_issued = 0, n_cons = 0, nq_issued = 0, nq_conv = 0;
  constexpr int QV = Sh::QV;
  uint4 qpre[QV];  // bf16 q rows of the next segment, 8 elements per chunk

  // Issue tiles ahead while buffers are free.  A segment's first tile also
  // starts the load of that segment's q into qpre, which must have been
  // consumed by the previous segment.
  auto try_issue = [&]() {
    while (is.valid && n_issued < n_cons + NST) {
      if (is.first && nq_issued != nq_conv) break;
      const int cnt = min(TK, is.send - is.s);
      const int buf = n_issued % NST;
      if (lane == 0) {
        const uint32_t kbytes = static_cast<uint32_t>(cnt * ROWB_K), vbytes = static_cast<uint32_t>(cnt * ROWB_V);
        const size_t row = static_cast<size_t>(real_head(is.i)) * a.cap + is.s;
        mbar_arrive_expect_tx(&bars[buf], kbytes + vbytes);
        bulk_copy_g2s(Ks + buf * TILEB_K, a.K + row * Sh::KU4, kbytes, &bars[buf]);
        bulk_copy_g2s(Vs + buf * TILEB_V, a.V + row * Sh::VU4, vbytes, &bars[buf]);
      }
      if (is.first) {
        const int x = real_head(is.i);
        const int b = x / a.Hkv, h = x - (x / a.Hkv) * a.Hkv;
        const uint4* qsrc =
            reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * Hq + h * a.Gq + head_group(is.i) * G) * D);
#pragma unroll
        for (int v = 0; v < QV; ++v) {
          const int x = lane + 32 * v;
          if (x < G * D / 8) qpre[v] = __ldg(qsrc + x);
        }
        ++nq_issued;
      }
      ++n_issued;
      is.advance(lenf, NV, cnt);
    }
  };

  // Latch a timeout, then wait (bounded) for this warp's copies in flight.
  auto fail_and_drain = [&]() {
    if (lane == 0) atomicOr(a.err, kErrBitTimeout);
    for (int k = n_cons; k < n_issued; ++k) (void)mbar_wait(&bars[k % NST], (k / NST) & 1);
  };

  // QK lane roles: two lanes per slot, each over half of the head dim.
  const int r = lane & 15, hf = lane >> 4;
  float m[G], l[G];
  float2 o[G][EL / 2];
  int seg_i = 0, seg_L = 0;
  int64_t seg_P = 0;

  try_issue();
  while (cs.valid) {
    if (cs.first) {
      // ---- segment start: this head's q (bf16) -> qs (fp32, pre-scaled) ----
      // (the first tile of this segment was issued, so its q is in qpre)
#pragma unroll
      for (int v = 0; v < QV; ++v) {
        const int x = lane + 32 * v;
        if (x < G * D / 8) {
          const int e0 = 8 * x, g = e0 / D, d = e0 % D;
          float* dst = qs + g * QROW + (d >= D / 2 ? QHALF + d - D / 2 : d);
          const uint4 u = qpre[v];
          const float2 f0 = bf16x2_to_float2(u.x), f1 = bf16x2_to_float2(u.y);
          const float2 f2 = bf16x2_to_float2(u.z), f3 = bf16x2_to_float2(u.w);
          const float sc = a.qscale;
          reinterpret_cast<float4*>(dst)[0] = make_float4(f0.x * sc, f0.y * sc, f1.x * sc, f1.y * sc);
          reinterpret_cast<float4*>(dst)[1] = make_float4(f2.x * sc, f2.y * sc, f3.x * sc, f3.y * sc);
        }
      }
      __syncwarp();
      ++nq_conv;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < EL / 2; ++e) o[g][e] = make_float2(0.f, 0.f);
      }
      seg_i = cs.i;
      seg_L = cs.L;
      seg_P = cs.P;
      if constexpr (FUSED) {
        const int d = cs.i - fx[Sh::FX_I0];
        const int sw =
            d < Sh::FX_HEADS ? fx[d]
                             : fused_new_slot_far(a, *reinterpret_cast<const int64_t*>(fx + Sh::FX_T), real_head(cs.i));
        __syncwarp();
        if (lane == 0) fx[Sh::FX_SEG] = sw;
        __syncwarp();
      }
      try_issue();
    }

    const int cnt = min(TK, cs.send - cs.s);
    const int s0 = cs.s;
    const int buf = n_cons % NST;
    if (n_issued <= n_cons || !mbar_wait(&bars[buf], (n_cons / NST) & 1)) {
      fail_and_drain();
      return;
    }

    if constexpr (FUSED) {
      const int sw = fx[Sh::FX_SEG];  // reloaded after the wait (the wait clobbers memory)
      if (static_cast<unsigned>(sw - s0) < static_cast<unsigned>(cnt))
        patch_new_row(a, reinterpret_cast<uint4*>(Ks + buf * TILEB_K), reinterpret_cast<uint4*>(Vs + buf * TILEB_V),
                      real_head(seg_i), sw - s0, sw, CH, lane);
    }

    // ---- QK and online softmax (base 2) ----
    if constexpr (!Sh::FP8) {
      // QK: lanes r and r + 16 score slot s0 + r over the two halves of D
      float sc[G];
      {
        const uint4* krow = reinterpret_cast<const uint4*>(Ks + buf * TILEB_K) + r * CH;
        const int sw = (s0 + r) & 7;
        const float* qh = qs + hf * QHALF;
        float2 acc0[G], acc1[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          acc0[g] = make_float2(0.f, 0.f);
          acc1[g] = make_float2(0.f, 0.f);
        }
        if (r < cnt) {
#pragma unroll
          for (int c = 0; c < HCH; ++c) {
            const uint4 kk = krow[(hf * HCH + c) ^ sw];
            const float2 k0 = bf16x2_to_float2(kk.x), k1 = bf16x2_to_float2(kk.y);
            const float2 k2 = bf16x2_to_float2(kk.z), k3 = bf16x2_to_float2(kk.w);
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float4* qp = reinterpret_cast<const float4*>(qh + g * QROW + c * 8);
              const float4 qa = qp[0], qb = qp[1];
              acc0[g] = __ffma2_rn(make_float2(qa.x, qa.y), k0, acc0[g]);
              acc1[g] = __ffma2_rn(make_float2(qa.z, qa.w), k1, acc1[g]);
              acc0[g] = __ffma2_rn(make_float2(qb.x, qb.y), k2, acc0[g]);
              acc1[g] = __ffma2_rn(make_float2(qb.z, qb.w), k3, acc1[g]);
            }
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float sg = (acc0[g].x + acc0[g].y) + (acc1[g].x + acc1[g].y);
          sg += __shfl_xor_sync(0xffffffffu, sg, 16);
          sc[g] = r < cnt ? sg : -INFINITY;
        }
      }

      // ---- online softmax (base 2); lanes r and r + 16 hold the same scores ----
      {
        bool rescale = false;
        float alpha[G], p[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float mt = sc[g];
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
          const float mn = fmaxf(m[g], mt);
          alpha[g] = fast_exp2(m[g] - mn);
          p[g] = fast_exp2(sc[g] - mn);
          l[g] = l[g] * alpha[g] + (hf == 0 ? p[g] : 0.f);
          m[g] = mn;
          rescale |= alpha[g] != 1.f;
        }
        if (hf == 0) {
          float2* prow = reinterpret_cast<float2*>(pb + r * PROW);
#pragma unroll
          for (int g = 0; g < G; ++g) prow[g] = make_float2(p[g], p[g]);
        }
        if (rescale) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float2 aa = make_float2(alpha[g], alpha[g]);
#pragma unroll
            for (int e = 0; e < EL / 2; ++e) o[g][e] = __fmul2_rn(o[g][e], aa);
          }
        }
        __syncwarp();
      }
    } else {
      // fp8, 32-slot tiles: lanes r and r + 16 score slots s0 + r and s0 + r + 16
      // over the two halves of D, each q load serving both slots.  A score is
      // the dot product with the codes times the row's K scale; the V scale is
      // folded into the slot's probability for PV.  Rows at or past cnt hold
      // stale bytes: their scores are replaced by -inf and their V scales by 0.
      const uint8_t* krA = Ks + buf * TILEB_K + r * ROWB_K;
      const uint8_t* krB = krA + 16 * ROWB_K;
      const bool okA = r < cnt, okB = r + 16 < cnt;
      const float* qh = qs + hf * QHALF;
      float2 aA0[G], aA1[G], aB0[G], aB1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        aA0[g] = make_float2(0.f, 0.f);
        aA1[g] = make_float2(0.f, 0.f);
        aB0[g] = make_float2(0.f, 0.f);
        aB1[g] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        const uint4 kA = *reinterpret_cast<const uint4*>(krA + hf * (D / 2) + c * 16);
        const uint4 kB = *reinterpret_cast<const uint4*>(krB + hf * (D / 2) + c * 16);
#pragma unroll
        for (int hw = 0; hw < 2; ++hw) {  // 8 codes of each slot at a time
          const uint32_t wa0 = hw ? kA.z : kA.x, wa1 = hw ? kA.w : kA.y;
          const uint32_t wb0 = hw ? kB.z : kB.x, wb1 = hw ? kB.w : kB.y;
          const float2 a0 = e4m3x2_to_float2(wa0 & 0xffffu), a1 = e4m3x2_to_float2(wa0 >> 16);
          const float2 a2 = e4m3x2_to_float2(wa1 & 0xffffu), a3 = e4m3x2_to_float2(wa1 >> 16);
          const float2 b0 = e4m3x2_to_float2(wb0 & 0xffffu), b1 = e4m3x2_to_float2(wb0 >> 16);
          const float2 b2 = e4m3x2_to_float2(wb1 & 0xffffu), b3 = e4m3x2_to_float2(wb1 >> 16);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float4* qp = reinterpret_cast<const float4*>(qh + g * QROW + c * 16 + hw * 8);
            const float4 qa = qp[0], qb = qp[1];
            const float2 q01 = make_float2(qa.x, qa.y), q23 = make_float2(qa.z, qa.w);
            const float2 q45 = make_float2(qb.x, qb.y), q67 = make_float2(qb.z, qb.w);
            aA0[g] = __ffma2_rn(q01, a0, aA0[g]);
            aA1[g] = __ffma2_rn(q23, a1, aA1[g]);
            aA0[g] = __ffma2_rn(q45, a2, aA0[g]);
            aA1[g] = __ffma2_rn(q67, a3, aA1[g]);
            aB0[g] = __ffma2_rn(q01, b0, aB0[g]);
            aB1[g] = __ffma2_rn(q23, b1, aB1[g]);
            aB0[g] = __ffma2_rn(q45, b2, aB0[g]);
            aB1[g] = __ffma2_rn(q67, b3, aB1[g]);
          }
        }
      }
      const float2 scA = *reinterpret_cast<const float2*>(krA + D);  // {K scale, V scale}
      const float2 scB = *reinterpret_cast<const float2*>(krB + D);
      const float vsA = okA ? scA.y : 0.f, vsB = okB ? scB.y : 0.f;
      float sA[G], sB[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float x = (aA0[g].x + aA0[g].y) + (aA1[g].x + aA1[g].y);
        float y = (aB0[g].x + aB0[g].y) + (aB1[g].x + aB1[g].y);
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        y += __shfl_xor_sync(0xffffffffu, y, 16);
        sA[g] = okA ? x * scA.x : -INFINITY;
        sB[g] = okB ? y * scB.x : -INFINITY;
      }
      // online softmax over the 32 slots; lanes r and r + 16 hold the same scores
      bool rescale = false;
      float alpha[G], pA[G], pB[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float mt = fmaxf(sA[g], sB[g]);
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        const float mn = fmaxf(m[g], mt);
        alpha[g] = fast_exp2(m[g] - mn);
        pA[g] = fast_exp2(sA[g] - mn);
        pB[g] = fast_exp2(sB[g] - mn);
        l[g] = l[g] * alpha[g] + (hf == 0 ? pA[g] + pB[g] : 0.f);
        m[g] = mn;
        rescale |= alpha[g] != 1.f;
      }
      {
        // lane r writes slot r's weights, lane r + 16 slot r + 16's
        float2* prow = reinterpret_cast<float2*>(pb + (r + hf * 16) * PROW);
        const float vs = hf ? vsB : vsA;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pw = (hf ? pB[g] : pA[g]) * vs;
          prow[g] = make_float2(pw, pw);
        }
      }
      if (rescale) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 aa = make_float2(alpha[g], alpha[g]);
#pragma unroll
          for (int e = 0; e < EL / 2; ++e) o[g][e] = __fmul2_rn(o[g][e], aa);
        }
      }
      __syncwarp();
    }

    // ---- PV: lane owns elements [lane*EL, lane*EL + EL) of every head ----
    {
      const uint8_t* Vt = Vs + buf * TILEB_V + lane * (EL * (Sh::FP8 ? 1 : 2));
      auto pv_row = [&](int j) {
        float2 v2[EL / 2];
        if constexpr (Sh::FP8) {
          if constexpr (EL == 4) {
            const uint32_t vv = *reinterpret_cast<const uint32_t*>(Vt + j * ROWB_V);
            v2[0] = e4m3x2_to_float2(vv & 0xffffu);
            v2[1] = e4m3x2_to_float2(vv >> 16);
          } else {
            v2[0] = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(Vt + j * ROWB_V));
          }
        } else if constexpr (EL == 4) {
          const uint2 vv = *reinterpret_cast<const uint2*>(Vt + j * ROWB_V);
          v2[0] = bf16x2_to_float2(vv.x);
          v2[1] = bf16x2_to_float2(vv.y);
        } else {
          v2[0] = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(Vt + j * ROWB_V));
        }
        const float4* prow = reinterpret_cast<const float4*>(pb + j * PROW);
#pragma unroll
        for (int x = 0; x < (G + 1) / 2; ++x) {
          const float4 p4 = prow[x];
#pragma unroll
          for (int e = 0; e < EL / 2; ++e) o[2 * x][e] = __ffma2_rn(make_float2(p4.x, p4.y), v2[e], o[2 * x][e]);
          if (2 * x + 1 < G) {
#pragma unroll
            for (int e = 0; e < EL / 2; ++e)
              o[2 * x + 1][e] = __ffma2_rn(make_float2(p4.z, p4.w), v2[e], o[2 * x + 1][e]);
          }
        }
      };
      if (cnt == TK) {
#pragma unroll
        for (int j = 0; j < TK; ++j) pv_row(j);
      } else {
        for (int j = 0; j < cnt; ++j) pv_row(j);
      }
    }
    __syncwarp();
    ++n_cons;
    const int cur_i = cs.i;
    cs.advance(lenf, NV, cnt);
    const bool seg_end = !cs.valid || cs.i != cur_i;

    if (seg_end) {
      // ---- segment end: direct output, or a partial merged by the last arriver ----
#pragma unroll
      for (int g = 0; g < G; ++g) l[g] = warp_sum(l[g]);
      const int x = real_head(seg_i);
      const int b = x / a.Hkv, h = x - b * a.Hkv;
      float* outp = a.out + (static_cast<size_t>(b) * Hq + h * a.Gq + head_group(seg_i) * G) * D + lane * EL;
      // Warps holding the first and the last slot of this head.
      const int64_t w0 = ((seg_P + 1) * Pe - 1) / S;
      const int64_t w1 = ((seg_P + seg_L) * Pe - 1) / S;
      if (w0 == w1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float inv = 1.f / l[g];
#pragma unroll
          for (int e = 0; e < EL / 2; ++e)
            reinterpret_cast<float2*>(outp + g * D)[e] = make_float2(o[g][e].x * inv, o[g][e].y * inv);
        }
      } else {
        // Partial of (warp wg, head seg_i) at index wg + seg_i: unique, because the
        // heads a warp covers never decrease with the warp index.
        const size_t idx = static_cast<size_t>(wg + seg_i);
        float* pa = a.part_acc + idx * G * D + lane * EL;
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int e = 0; e < EL / 2; ++e) reinterpret_cast<float2*>(pa + g * D)[e] = o[g][e];
        }
        if (lane < G) {
          float mm = m[0], ll = l[0];
#pragma unroll
          for (int g = 1; g < G; ++g) {
            if (lane == g) {
              mm = m[g];
              ll = l[g];
            }
          }
          reinterpret_cast<float2*>(a.part_ml)[idx * G + lane] = make_float2(mm, ll);
        }
        // Release the partial, then count this arrival; the last of the head's
        // nseg warps merges (acquire) and resets the counter.
        const int nseg = static_cast<int>(w1 - w0) + 1;
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(a.head_cnt + seg_i, 1) == nseg - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          merge_partials<D, G>(a, static_cast<size_t>(w0 + seg_i), nseg, outp, lane);
          if (lane == 0) a.head_cnt[seg_i] = 0;
        }
      }
    }
    try_issue();
  }
}

}  // namespace dms
