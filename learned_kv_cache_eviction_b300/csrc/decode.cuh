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
// such warp then increments the head's arrival counter (a warp's first
// segment when it ends, its last one when its range is done), and the warp
// that arrives last merges the partials and writes the output (and resets the
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
  // Per-warp state kept in shared memory rather than in registers (the decode
  // loop has none to spare): the retained lengths of the first FX_HEADS heads
  // of the warp's range (read at every head change, so no head change waits on
  // global memory), and for the fused step the new token's slots of the same
  // heads, the current segment's, and the step's position; then the first head.
  static constexpr int FX_HEADS = 6;
  static constexpr int FX_HL = 0, FX_SN = FX_HEADS;
  static constexpr int FX_I0 = 2 * FX_HEADS, FX_SEG = 2 * FX_HEADS + 1;
  static constexpr int FX_T = 2 * FX_HEADS + 2;  // the step's position t (int64, two slots)
  static constexpr int OFF_FX = OFF_BAR + NST * 8;
  static constexpr int FX_BYTES = (FX_T + 2) * 4;  // through the int64 position
  // Then two mbarriers for the bulk copies of a merge, and the warp's split
  // segments (see decode_kernel): {virtual head, index of its first partial,
  // partial count} for the first and for the last segment (head -1: none),
  // whose merges, if this warp's arrival completes them, run after its range;
  // and the merge mbarriers' phase bits.
  static constexpr int OFF_MB = OFF_FX + FX_BYTES;
  static constexpr int OFF_DEF = OFF_MB + 16;
  static constexpr int WARP_BYTES = ((OFF_DEF + 28 + 127) / 128) * 128;
  // Partials: acc [G][D] floats, and (max, sum) of the G heads padded to a
  // 16-byte record of MLS floats, so that consecutive partials form one
  // contiguous bulk copy.  A merge stages them PM at a time in two halves of
  // the warp's tile, q and probability buffers (free once its range is done),
  // the copy of one chunk in flight while the other is folded in.
  static constexpr int MLS = (2 * G + 3) / 4 * 4;
  static constexpr int STAGE_HALF = (OFF_BAR / 2) / 16 * 16;
  static constexpr int PM = STAGE_HALF / (G * D * 4 + MLS * 4);
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
  static_assert(PM >= 1 && OFF_MB % 8 == 0 && STAGE_HALF % 16 == 0, "merge staging");
  static_assert(OFF_FX % 8 == 0 && OFF_FX + FX_T * 4 + 8 <= OFF_MB, "the position word lies inside FX");
};

// Largest number of warps per CTA of any instantiation (sizes the partials).
constexpr int kMaxWarpsPerCta = 12;

// Fewest tiles a warp is given (bounds the number of partials when the cache
// is small).  Small caches are latency-bound per warp, so they are spread over
// as many warps as this allows (three tiles measured best on small caches;
// capping the warps per head instead, for fewer partials, was slower).
// kMinSlotsPerWarp sizes the grid on the host.
constexpr int kMinTilesPerWarp = 3;
constexpr int kMinSlotsPerWarp = 48;

struct DecodeArgs {
  const uint4* K;
  const uint4* V;
  const int32_t* len;
  const uint16_t* q;  // bf16 [B][Hq][D]
  float* out;         // fp32 [B][Hq][D]
  float* part_acc;    // [entries][G][D]
  float* part_ml;     // [entries][MLS]: (max, sum) of each of the G heads, padded to 16 bytes
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
  // lengths [3][NH] (see CacheView): the kernel decodes over the lengths after
  // the token and writes those, the token's ring entry, slot map entry and K/V
  // row into generations of the state that no CTA of the launch reads.  The
  // position t comes from `t`, or, when t_dev is set (a step replayed from a
  // CUDA graph), from device memory.
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
  // Fused step only: 1 when the launch may run its prologue (length scan, work
  // split) and start its first tile copies before the previous launch in the
  // stream has finished (programmatic dependent launch).  Everything it reads
  // before its grid-dependency wait was then written by earlier launches: the
  // lengths after t - 1 appends, the ring entries of positions t - 1 - w and
  // t - w (w >= 2), the position word (never written by the launch just before
  // this one), and pool rows other than the one the previous token went to.
  // The host sets it only when the previous call that advanced the cache added
  // exactly one token (so generation t - 1 of the lengths is intact).
  int early;
  // Work split: every warp gets at least min_tiles tiles.
  int min_tiles;
  // Plain decode over caller-owned lengths (the no-allocation entry point):
  // each length is clamped to [0, cap] before use, and a clamped value latches
  // kErrBitLength, so that a bad length can never send a copy past a head's pool.
  int clamp_len;
  // Fused step from host rows (dms_step_host): the step's k, v, logit and q
  // rows are copied in, and its output copied out, on copy streams of their
  // own, which write sequence numbers into host_flag[0] (rows landed) and
  // host_flag[1] (the output rows read back) when they finish.  Before it
  // reads an input or writes an output, every warp waits (bounded) until
  // host_flag[0] >= in_need and host_flag[1] >= out_need (wrap-safe), so the
  // launch needs no cross-stream dependency and keeps its early start.  Null
  // for every other call.
  const unsigned* host_flag;
  unsigned in_need, out_need;
};

// Steps from host rows: wait until the copy streams have landed this step's
// rows and read back the output rows this step will overwrite (DecodeArgs::
// host_flag).  On the time limit it latches kErrBitTimeout and returns; the
// step then reads stale rows but stays within its buffers.
__device__ __forceinline__ void wait_host_rows(const DecodeArgs& a) {
  if (a.host_flag == nullptr) return;
  uint64_t t0 = 0;
  while (true) {
    const unsigned fi = ld_acquire_u32(a.host_flag), fo = ld_acquire_u32(a.host_flag + 1);
    if (static_cast<int>(fi - a.in_need) >= 0 && static_cast<int>(fo - a.out_need) >= 0) return;
    const uint64_t now = global_timer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > kWaitLimitNs) {
      atomicOr(a.err, kErrBitTimeout);
      return;
    }
  }
}

// Length of head x in a plain decode, clamped when the lengths come from the caller.
__device__ __forceinline__ int plain_len(const DecodeArgs& a, int x) {
  int L = a.len[x];
  if (a.clamp_len && static_cast<unsigned>(L) > static_cast<unsigned>(a.cap)) {
    L = L < 0 ? 0 : a.cap;
    atomicOr(a.err, kErrBitLength);
  }
  return L;
}

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
  return fused_new_slot(a, t, x, a.len[len_gen(t) * a.NH + x]);
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
    Kt[j * CH + (lane ^ (s_new & 7))] = __ldcg(a.k_new + static_cast<size_t>(i) * CH + lane);
  } else if (lane < 2 * CH) {
    Vt[j * CH + lane - CH] = __ldcg(a.v_new + static_cast<size_t>(i) * CH + lane - CH);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// The same for FP8 storage: the new token's rows are quantized exactly as the
// append stores them (quantize_kv_rows) into row j of the staged K tile (D
// codes + the scale chunk) and V tile (D codes).  Called by the whole warp.
template <int D>
static __device__ __noinline__ void patch_new_row_fp8(const DecodeArgs& a, uint8_t* Kt, uint8_t* Vt, int i, int j,
                                                      int lane) {
  constexpr int CH = D / 8;
  uint4 x = make_uint4(0u, 0u, 0u, 0u);
  if (lane < CH) x = __ldcg(a.k_new + static_cast<size_t>(i) * CH + lane);
  else if (lane < 2 * CH) x = __ldcg(a.v_new + static_cast<size_t>(i) * CH + lane - CH);
  quantize_kv_rows<D>(x, Kt + j * (D + 16), Vt + j * D, lane);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// Fused step started early (DecodeArgs::early): head x's state as the step
// sees it, derived without reading anything the previous step wrote.  From
// the lengths after t - 1 appends and the ring entries of t - 1 - w and t - w:
// the slot the previous step's token (position t - 1) went to, the slot of
// this step's token (position t), and the length after this step's append.
// The same rule as append_bookkeeping, applied twice.
struct EarlyHead {
  int L;       // retained length after t + 1 appends
  int s_new;   // slot of token t, -1 if the cache is full
  int s_prev;  // slot of token t - 1, -1 if it was not stored
};

__device__ __forceinline__ EarlyHead early_head(const DecodeArgs& a, int64_t t, int x) {
  const int L1 = __ldcg(a.len + len_gen(t - 1) * a.NH + x);
  int f1 = 0, s1 = 0, f0 = 0, s0 = 0;
  if (t - 1 >= a.w) {
    const size_t e = ring_index(a.NH, a.w, x, t - 1 - a.w);
    f1 = __ldcg(a.ring_flag + e);
    s1 = __ldcg(a.ring_slot + e);
  }
  if (t >= a.w) {
    const size_t e = ring_index(a.NH, a.w, x, t - a.w);
    f0 = __ldcg(a.ring_flag + e);
    s0 = __ldcg(a.ring_slot + e);
  }
  EarlyHead h;
  h.s_prev = f1 ? s1 : (L1 < a.cap ? L1 : -1);
  const int L2 = (f1 || L1 >= a.cap) ? L1 : L1 + 1;
  h.s_new = f0 ? s0 : (L2 < a.cap ? L2 : -1);
  h.L = (f0 || L2 >= a.cap) ? L2 : L2 + 1;
  return h;
}

// Retained length of head x as this launch decodes it (fused: after the
// append of position t).
template <bool FUSED>
__device__ __forceinline__ int decode_len(const DecodeArgs& a, int64_t t, int x) {
  if constexpr (FUSED) {
    if (a.early) return early_head(a, t, x).L;
    const int L = a.len[len_gen(t) * a.NH + x];
    const bool retire = t >= a.w && a.ring_flag[ring_index(a.NH, a.w, x, t - a.w)] != 0;
    return (!retire && L < a.cap) ? L + 1 : L;
  }
  return plain_len(a, x);
}

// Tiles of TK slots in a head of L retained slots (the last one partial).
template <int TK>
__host__ __device__ __forceinline__ int tiles_of(int L) { return (L + TK - 1) / TK; }

// Retained-slot iterator over one warp's global range [A, E) of tiles: the
// heads' tiles concatenated, so every warp range starts and ends on a tile
// boundary of its heads and holds the same number of tiles (to within one).
template <int TK>
struct TileIter {
  int i;      // head
  int L;      // retained length of head i
  int s;      // next slot in head i
  int send;   // end of this warp's slots in head i
  int64_t P;  // global index of tile 0 of head i
  int64_t E;
  bool valid;
  bool first;  // next tile opens a new segment (head)

  __device__ __forceinline__ void set_end() {
    send = static_cast<int>(min(static_cast<int64_t>(L), (E - P) * TK));
  }
  template <typename LenF>
  __device__ __forceinline__ void start(const LenF& len, int i0, int64_t P0, int64_t A, int64_t E_) {
    i = i0;
    P = P0;
    E = E_;
    L = len(i0);
    s = static_cast<int>(A - P0) * TK;
    set_end();
    valid = s < send;
    first = true;
  }
  template <typename LenF>
  __device__ __forceinline__ void advance(const LenF& len, int NH, int cnt) {
    s += cnt;
    first = false;
    if (s < send) return;
    P += tiles_of<TK>(L);
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
    set_end();
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

// Arrival counts of split heads.  A warp writes its partials, synchronises
// (__syncwarp), and lane 0 issues a release fence at GPU scope, which publishes
// the whole warp's partials, then adds its arrivals (relaxed, issued back to
// back); an arrival that completes a count is followed by an acquire fence
// before the others' partials are read.
__device__ __forceinline__ void fence_release_gpu() { asm volatile("fence.release.gpu;" ::: "memory"); }
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acquire.gpu;" ::: "memory"); }


// Merge the nseg partials (max m, sum l, unnormalised acc) of one head, stored
// at consecutive partial indices base, base + 1, ..., and write the normalised
// output (outp already offset by lane * EL).  The partials are staged into
// shared memory (`stage`: two halves of STAGE_HALF bytes, the warp's free
// buffers) by bulk copies of PM partials at a time, chunk c + 1 in flight while
// chunk c is folded in with a running max per query head.  The caller has
// acquired the partials; the proxy fence orders those generic-proxy writes
// before the async-proxy reads of the bulk copies.  `phases` holds the two
// mbarriers' phase bits.  Returns false if a copy did not complete within the
// time limit.
template <typename Sh>
__device__ __forceinline__ bool merge_partials(const DecodeArgs& a, size_t base, int nseg, float* outp, int lane,
                                               uint8_t* stage, uint64_t* mbar, uint32_t& phases) {
  constexpr int G = Sh::G, D = Sh::D, EL = D / 32, MLS = Sh::MLS, PM = Sh::PM, HALF = Sh::STAGE_HALF;
  constexpr int ACCB = G * D * 4;
  float M[G], L[G];
  float2 acc[G][EL / 2];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    M[g] = -INFINITY;
    L[g] = 0.f;
#pragma unroll
    for (int e = 0; e < EL / 2; ++e) acc[g][e] = make_float2(0.f, 0.f);
  }
  const int nch = (nseg + PM - 1) / PM;
  auto issue = [&](int c) {
    if (lane == 0) {
      const int b = c & 1, n = min(PM, nseg - c * PM);
      uint8_t* dst = stage + b * HALF;
      const uint32_t ab = static_cast<uint32_t>(n * ACCB), mb = static_cast<uint32_t>(n * MLS * 4);
      mbar_arrive_expect_tx(&mbar[b], ab + mb);
      bulk_copy_g2s(dst, a.part_acc + (base + static_cast<size_t>(c) * PM) * G * D, ab, &mbar[b]);
      bulk_copy_g2s(dst + PM * ACCB, a.part_ml + (base + static_cast<size_t>(c) * PM) * MLS, mb, &mbar[b]);
    }
  };
  if (lane == 0) asm volatile("fence.proxy.async;" ::: "memory");
  issue(0);
  if (nch > 1) issue(1);
  for (int c = 0; c < nch; ++c) {
    const int b = c & 1, n = min(PM, nseg - c * PM);
    const uint32_t ph = (phases >> b) & 1u;
    if (!mbar_wait(&mbar[b], ph)) {
      // give the copies in flight a second bounded wait before leaving
      for (int k = c; k < min(nch, c + 2); ++k) (void)mbar_wait(&mbar[k & 1], (phases >> (k & 1)) & 1u);
      return false;
    }
    phases ^= 1u << b;
    const float* sacc = reinterpret_cast<const float*>(stage + b * HALF);
    const float* sml = reinterpret_cast<const float*>(stage + b * HALF + PM * ACCB);
    float mt[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mt[g] = M[g];
#pragma unroll
    for (int j = 0; j < PM; ++j) {
      if (j < n) {
#pragma unroll
        for (int g = 0; g < G; ++g) mt[g] = fmaxf(mt[g], sml[j * MLS + 2 * g]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float sc = fast_exp2(M[g] - mt[g]);
      L[g] *= sc;
#pragma unroll
      for (int e = 0; e < EL / 2; ++e) acc[g][e] = __fmul2_rn(acc[g][e], make_float2(sc, sc));
      M[g] = mt[g];
    }
#pragma unroll
    for (int j = 0; j < PM; ++j) {
      if (j < n) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 mlj = *reinterpret_cast<const float2*>(sml + j * MLS + 2 * g);
          const float wj = fast_exp2(mlj.x - mt[g]);
          L[g] = fmaf(wj, mlj.y, L[g]);
          const float2* src = reinterpret_cast<const float2*>(sacc + (j * G + g) * D + lane * EL);
#pragma unroll
          for (int e = 0; e < EL / 2; ++e) acc[g][e] = __ffma2_rn(make_float2(wj, wj), src[e], acc[g][e]);
        }
      }
    }
    __syncwarp();
    if (c + 2 < nch) issue(c + 2);  // this half has been read
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float inv = 1.f / L[g];
#pragma unroll
    for (int e = 0; e < EL / 2; ++e)
      reinterpret_cast<float2*>(outp + g * D)[e] = make_float2(acc[g][e].x * inv, acc[g][e].y * inv);
  }
  return true;
}

template <int D, int G, bool FUSED, int KVF = kKvBf16>
__global__ void __launch_bounds__(DecodeShape<D, G, KVF>::NW * 32, 1) decode_kernel(const DecodeArgs a) {
  using Sh = DecodeShape<D, G, KVF>;
  constexpr int NW = Sh::NW, TK = Sh::TK, NST = Sh::NST, CH = Sh::CH, HCH = Sh::HCH, EL = Sh::EL;
  constexpr int ROWB_K = Sh::ROWB_K, ROWB_V = Sh::ROWB_V, TILEB_K = Sh::TILEB_K, TILEB_V = Sh::TILEB_V;
  constexpr int QHALF = Sh::QHALF, QROW = Sh::QROW, PROW = Sh::PROW;
  extern __shared__ __align__(1024) uint8_t smem[];

  // Launched as a programmatic dependent of the previous kernel: everything the
  // previous kernels wrote is visible after griddep_wait.  A fused step started
  // early (a.early) first runs its prologue and issues its first tile copies
  // from state that earlier launches wrote (see DecodeArgs::early), and waits
  // before it reads any input or writes anything.
  const bool early = FUSED && a.early != 0;
  if (!early) {
    griddep_wait();
    griddep_launch_dependents();
    if constexpr (FUSED) wait_host_rows(a);
  }

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
  int* ln = pre + NV + 1;                   // [NH] each KV head's retained length (fused: after the append)
  int* sn = ln + a.NH;                      // fused step: [NH] the new token's slot in each KV head
  int* sp = sn + a.NH;                      // fused step started early: [NH] the previous token's slot
  // Fused step: warp x of the grid appends the token to head x (and x + nwarps,
  // ...).  Its row chunk (K for lanes < CH, V for lanes CH .. 2 CH - 1) and
  // logit are loaded now, in flight during the scan (not when started early:
  // the inputs may come from the launch just before).
  uint4 own_row = make_uint4(0u, 0u, 0u, 0u);
  float own_logit = 0.f;
  if constexpr (FUSED) {
    if (!early && wg < a.NH) {
      if (lane < 2 * CH)
        own_row = __ldcg((lane < CH ? a.k_new : a.v_new) + static_cast<size_t>(wg) * CH + (lane % CH));
      own_logit = __ldcg(a.logit_new + wg);
    }
  }
  // The scan reads each head's length (and, fused, the ring entry of t - w) once
  // and sums its tiles; the fused scan also records the new token's slot in sn
  // and the length after the append in ln.
  auto scanf = [&](int v) {
    const int x = real_head(v);
    if constexpr (FUSED) {
      if (early) {
        const EarlyHead eh = early_head(a, t_step, x);
        if (v < a.NH) {
          sn[x] = eh.s_new;
          sp[x] = eh.s_prev;
          ln[x] = eh.L;
        }
        return tiles_of<TK>(eh.L);
      }
      const int L = a.len[len_gen(t_step) * a.NH + x];
      int fl = 0, sl = 0;
      if (t_step >= a.w) {
        const size_t e = ring_index(a.NH, a.w, x, t_step - a.w);
        fl = a.ring_flag[e];
        sl = a.ring_slot[e];
      }
      const int L3 = (fl || L >= a.cap) ? L : L + 1;
      if (v < a.NH) {
        sn[x] = fl ? sl : (L < a.cap ? L : -1);
        ln[x] = L3;
      }
      return tiles_of<TK>(L3);
    } else {
      const int L = plain_len(a, x);
      if (v < a.NH) ln[x] = L;
      return tiles_of<TK>(L);
    }
  };
  scan_lengths(scanf, NV, pre);
  // Fused step: the bookkeeping and row of the new token in head i (length
  // after the append L_i, slot s_new, -1 if the cache is full).  None of it is
  // read by this launch: the next generations of the lengths and the ring, the
  // slot map, and a pool row that every tile copy skips (the new row is taken
  // from the input).
  auto append_head = [&](int i, int s_new, int L_i, uint4 rowc, float lg) {
    if (lane == 0) {
      a.len_w[len_gen(t_step + 1) * a.NH + i] = L_i;
      const size_t e = ring_index(a.NH, a.w, i, t_step);
      a.ring_slot[e] = s_new;
      a.ring_flag[e] = (s_new >= 0 && lg > 0.0f) ? 1 : 0;
      if (s_new >= 0) a.slot_pos[static_cast<size_t>(i) * a.cap + s_new] = static_cast<int32_t>(t_step);
      else atomicOr(a.err, kErrBitCapacity);
    }
    if (s_new >= 0) {
      if constexpr (Sh::FP8) {
        const size_t slot = static_cast<size_t>(i) * a.cap + s_new;
        quantize_kv_rows<D>(rowc, reinterpret_cast<uint8_t*>(a.K_w) + slot * (D + 16),
                            reinterpret_cast<uint8_t*>(a.V_w) + slot * D, lane);
      } else {
        const size_t row = (static_cast<size_t>(i) * a.cap + s_new) * CH;
        if (lane < CH) a.K_w[row + (lane ^ (s_new & 7))] = rowc;
        else if (lane < 2 * CH) a.V_w[row + lane - CH] = rowc;
      }
    }
  };
  auto load_new_row = [&](int i) {
    uint4 rowc = make_uint4(0u, 0u, 0u, 0u);
    if (lane < 2 * CH) rowc = __ldcg((lane < CH ? a.k_new : a.v_new) + static_cast<size_t>(i) * CH + (lane % CH));
    return rowc;
  };
  if constexpr (FUSED) {
    if (!early) {
      for (int64_t x = wg; x < a.NH; x += nwarps) {
        const int i = static_cast<int>(x);
        const bool own = x == wg;
        append_head(i, sn[i], ln[i], own ? own_row : load_new_row(i),
                    own ? own_logit : __ldcg(a.logit_new + i));
      }
    }
  }
  const int64_t S = pre[NV];  // tiles of all heads
  int64_t Pe = nwarps;
  if (S / a.min_tiles < Pe) Pe = S / a.min_tiles;
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
  // barrier, which ends the prefix sums' lease on the warp regions).  Started
  // early: also the slot of the previous step's token in head i0 (its tile is
  // not copied before the wait), and this warp's own head to append.
  int snl = -1, hll = 0, sprev0 = -1, own_sn = -1, own_L = 0;
  if (active && lane < Sh::FX_HEADS && i0 + lane < NV) hll = ln[real_head(i0 + lane)];
  if constexpr (FUSED) {
    if (active && lane < Sh::FX_HEADS && i0 + lane < NV) snl = sn[real_head(i0 + lane)];
    if (early) {
      if (active) sprev0 = sp[real_head(i0)];
      if (wg < a.NH) {
        own_sn = sn[wg];
        own_L = ln[wg];
      }
    }
  }
  __syncthreads();

  if (!active && !early) return;

  // ---- per-warp shared memory ----
  uint8_t* wbase = smem + wl * Sh::WARP_BYTES;
  uint8_t* Ks = wbase + Sh::OFF_K;
  uint8_t* Vs = wbase + Sh::OFF_V;
  float* qs = reinterpret_cast<float*>(wbase + Sh::OFF_QS);
  float* pb = reinterpret_cast<float*>(wbase + Sh::OFF_P);
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + Sh::OFF_BAR);  // [NST] tiles
  int* fx = reinterpret_cast<int*>(wbase + Sh::OFF_FX);               // fused-step state
  uint64_t* mbar = reinterpret_cast<uint64_t*>(wbase + Sh::OFF_MB);   // [2] merge copies
  int* def = reinterpret_cast<int*>(wbase + Sh::OFF_DEF);              // split segments, merge phases
  if (active) {
    if (lane == 0) {
      for (int x = 0; x < NST; ++x) mbar_init(&bars[x], 1);
      mbar_init(&mbar[0], 1);
      mbar_init(&mbar[1], 1);
      fence_barrier_init();
      def[0] = -1;
      def[3] = -1;
      def[6] = 0;
    }
    if (lane < Sh::FX_HEADS) fx[Sh::FX_HL + lane] = hll;
    if (lane == 0) fx[Sh::FX_I0] = i0;
    if constexpr (FUSED) {
      if (lane < Sh::FX_HEADS) fx[Sh::FX_SN + lane] = snl;
      if (lane == 0) {
        fx[Sh::FX_SEG] = -1;
        *reinterpret_cast<int64_t*>(fx + Sh::FX_T) = t_step;
      }
    }
  }
  __syncwarp();
  // Retained length of virtual head v as this launch decodes it (fused: after
  // its append), read per head change: from the warp's cached lengths, else
  // from global memory (the position comes from shared memory, not a register).
  auto lenf = [&](int v) {
    const int d = v - fx[Sh::FX_I0];
    if (static_cast<unsigned>(d) < static_cast<unsigned>(Sh::FX_HEADS)) return fx[Sh::FX_HL + d];
    if constexpr (FUSED) return decode_len<true>(a, *reinterpret_cast<const int64_t*>(fx + Sh::FX_T), real_head(v));
    else return decode_len<false>(a, 0, real_head(v));
  };

  const int Hq = a.Hkv * a.Gq;
  TileIter<TK> is{}, cs{};
  if (active) is.start(lenf, i0, P0, A, E);
  cs = is;
  int n_issued = 0, n_cons = 0, nq_issued = 0, nq_conv = 0;
  int c0_arrival = -1;  // lane 0: the count before this warp's first-segment arrival
  constexpr int QV = Sh::QV;
  uint4 qpre[QV];  // bf16 q rows of the next segment, 8 elements per chunk

  // The K and V tile copies of the iterator's next tile (lane 0).
  auto issue_tile = [&](int cnt) {
    if (lane == 0) {
      const int buf = n_issued % NST;
      const uint32_t kbytes = static_cast<uint32_t>(cnt * ROWB_K), vbytes = static_cast<uint32_t>(cnt * ROWB_V);
      const size_t row = static_cast<size_t>(real_head(is.i)) * a.cap + is.s;
      mbar_arrive_expect_tx(&bars[buf], kbytes + vbytes);
      bulk_copy_g2s(Ks + buf * TILEB_K, a.K + row * Sh::KU4, kbytes, &bars[buf]);
      bulk_copy_g2s(Vs + buf * TILEB_V, a.V + row * Sh::VU4, vbytes, &bars[buf]);
    }
  };
  // The G query rows of virtual head v into qpre.
  auto load_q = [&](int v) {
    const int x = real_head(v);
    const int b = x / a.Hkv, h = x - (x / a.Hkv) * a.Hkv;
    const uint4* qsrc =
        reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * Hq + h * a.Gq + head_group(v) * G) * D);
#pragma unroll
    for (int u = 0; u < QV; ++u) {
      const int y = lane + 32 * u;
      if (y < G * D / 8) qpre[u] = __ldcg(qsrc + y);
    }
    ++nq_issued;
  };

  // Issue tiles ahead while buffers are free.  A segment's first tile also
  // starts the load of that segment's q into qpre, which must have been
  // consumed by the previous segment.
  auto try_issue = [&]() {
    while (is.valid && n_issued < n_cons + NST) {
      if (is.first && nq_issued != nq_conv) break;
      const int cnt = min(TK, is.send - is.s);
      issue_tile(cnt);
      if (is.first) load_q(is.i);
      ++n_issued;
      is.advance(lenf, NV, cnt);
    }
  };

  if constexpr (FUSED) {
    if (early) {
      // Before the wait: up to NST tiles of the first head, stopping at the tile
      // that holds the previous step's token (its row may still be in flight).
      if (active) {
        while (is.valid && n_issued < NST && is.i == i0) {
          const int cnt = min(TK, is.send - is.s);
          if (static_cast<unsigned>(sprev0 - is.s) < static_cast<unsigned>(cnt)) break;
          issue_tile(cnt);
          ++n_issued;
          is.advance(lenf, NV, cnt);
        }
      }
      griddep_wait();
      griddep_launch_dependents();
      wait_host_rows(a);
      for (int64_t x = wg; x < a.NH; x += nwarps) {
        const int i = static_cast<int>(x);
        if (x == wg) {
          append_head(i, own_sn, own_L, load_new_row(i), __ldcg(a.logit_new + i));
        } else {
          const EarlyHead eh = early_head(a, t_step, i);
          append_head(i, eh.s_new, eh.L, load_new_row(i), __ldcg(a.logit_new + i));
        }
      }
      if (!active) return;
      if (n_issued > 0) load_q(i0);  // the first segment's q, now that the inputs are visible
    }
  }

  // Latch a timeout, then wait (bounded) for this warp's copies in flight.
  auto fail_and_drain = [&]() {
    if (lane == 0) atomicOr(a.err, kErrBitTimeout);
    for (int k = n_cons; k < n_issued; ++k) (void)mbar_wait(&bars[k % NST], (k / NST) & 1);
  };

  // Merge of split head v's nseg partials from index base into its output (the
  // last arriver); a copy that timed out latches the error.
  auto merge_head = [&](int v, size_t base, int nseg) {
    const int x = real_head(v);
    const int b = x / a.Hkv, h = x - b * a.Hkv;
    float* outp = a.out + (static_cast<size_t>(b) * Hq + h * a.Gq + head_group(v) * G) * D + lane * EL;
    uint32_t ph = static_cast<uint32_t>(def[6]);
    const bool ok = merge_partials<Sh>(a, base, nseg, outp, lane, wbase, mbar, ph);
    __syncwarp();
    if (lane == 0) {
      def[6] = static_cast<int>(ph);
      a.head_cnt[v] = 0;  // for the next call
      if (!ok) atomicOr(a.err, kErrBitTimeout);
    }
    __syncwarp();
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
            d < Sh::FX_HEADS ? fx[Sh::FX_SN + d]
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
      if (static_cast<unsigned>(sw - s0) < static_cast<unsigned>(cnt)) {
        if constexpr (Sh::FP8)
          patch_new_row_fp8<D>(a, Ks + buf * TILEB_K, Vs + buf * TILEB_V, real_head(seg_i), sw - s0, lane);
        else
          patch_new_row(a, reinterpret_cast<uint4*>(Ks + buf * TILEB_K), reinterpret_cast<uint4*>(Vs + buf * TILEB_V),
                        real_head(seg_i), sw - s0, sw, CH, lane);
      }
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
      // Warps holding the first and the last tile of this head.
      const int64_t w0 = ((seg_P + 1) * Pe - 1) / S;
      const int64_t w1 = ((seg_P + tiles_of<TK>(seg_L)) * Pe - 1) / S;
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
          reinterpret_cast<float2*>(a.part_ml + idx * Sh::MLS)[lane] = make_float2(mm, ll);
        }
        // Only a warp's first and last segments can be split.  The last one's
        // arrival is counted once the warp's range is done (below).  The first
        // one (ending mid-range) arrives now, its count read only at the end of
        // the range, so the stream does not wait on it: the head's other
        // pieces end their warps' ranges, and one of those warps merges it
        // instead of this warp merging two heads after its range.
        if (lane == 0) {
          const int k = cs.valid ? 0 : 3;
          def[k] = seg_i;
          def[k + 1] = static_cast<int>(w0 + seg_i);
          def[k + 2] = static_cast<int>(w1 - w0) + 1;
        }
        if (cs.valid) {
          __syncwarp();
          if (lane == 0) {
            fence_release_gpu();
            c0_arrival = atomicAdd(a.head_cnt + seg_i, 1);
          }
        }
      }
    }
    try_issue();
  }
  // Count the arrival of the warp's last segment if it is split (release the
  // partial first); the last of a head's nseg warps to arrive merges
  // (acquire) and resets its counter.
  __syncwarp();
  const int v0 = def[0], v1 = def[3];
  if (v0 >= 0 || v1 >= 0) {
    int last = 0;
    if (lane == 0) {
      int c1 = -1;
      if (v1 >= 0) {
        fence_release_gpu();
        c1 = atomicAdd(a.head_cnt + v1, 1);
      }
      last = (v0 >= 0 && c0_arrival == def[2] - 1 ? 1 : 0) | (v1 >= 0 && c1 == def[5] - 1 ? 2 : 0);
      if (last) fence_acquire_gpu();
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last & 2) merge_head(v1, static_cast<size_t>(def[4]), def[5]);
    if (last & 1) merge_head(v0, static_cast<size_t>(def[1]), def[2]);
  }
}

}  // namespace dms
