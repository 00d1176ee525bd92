// prefill.cuh -- chunked-prefill attention over the DMS compacted cache, on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes: C new tokens at positions t0 .. t0 + C - 1 of every
// sequence, each query attending to exactly the keys that single-token decode
// at its position would see -- the retained cache (tokens before t0) and the
// chunk's own tokens up to itself -- under the method's delayed eviction ("AI
// research-map summary" of "Inference-Time Hyper-Scaling with KV Cache
// Compression", section "Approach": a per-head eviction decision executed after
// a delay window).  Key j is visible to the query at position t iff
// pos_j <= t <= last_j, where last_j = pos_j + w - 1 for a token marked for
// eviction and +inf otherwise:
//   * a cached token marked for eviction is still in the cache only if it is
//     among the last w positions before t0 (its ring entry carries the mark);
//   * a chunk token's mark is its logit > 0.
// The chunk is appended to the cache afterwards (append_chunk_slots_kernel,
// append_chunk_copy_kernel), so the whole call equals C rounds of single-token
// append + decode attention.
//
// One CTA of 128 threads per (tile of PT = 128 / G query positions x G query
// heads, KV head).  Row r of the tile is query head g = r / PT at chunk
// position c0 + r % PT; thread r owns row r (tensor-memory lane r).  For each
// tile of 128 keys (the cache's retained slots first, then the chunk's keys up
// to the tile's last position):
//   1. the threads stage the K and V tile in shared memory in the 128-byte
//      swizzled layouts (K rows of the cache pool are stored chunk-permuted by
//      slot, which is that layout already), plus each key's (position, last);
//      K, V and the metadata are double-buffered: the next tile's asynchronous
//      copies (cp.async) are in flight while this one is computed;
//   2. one thread issues S = Q K^T (bf16 x bf16 -> fp32 in tensor memory);
//   3. every thread loads its row of S, masks it, and updates the running
//      max (only when it grows by more than 2^8, rescaling the accumulator in
//      tensor memory then) and sum; p = 2^(s - m) is written as two bf16
//      terms, hi = bf16(p) and lo = bf16(p - hi), so that P V keeps ~16 bits
//      of p;
//   4. one thread issues O += P_hi V + P_lo V (fp32 in tensor memory).
// The MMAs are ordered on two mbarriers; every wait has a time limit.
#pragma once

#include <cuda_bf16.h>

#include "dms_device.cuh"
#include "umma.cuh"

namespace dms {

template <int D_, int G_>
struct PrefillShape {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr int M = 128;                          // rows per tile
  static constexpr int PT = M / G;                       // query positions per tile
  static constexpr int ROWS = PT * G;                    // rows in use (<= 128)
  static constexpr int NK = 128;                         // keys per tile
  static constexpr int NP = D / 64;                      // 128-byte panels per row of Q, K, V
  static constexpr int PANEL = 128 * 128;                // bytes of one panel of 128 rows
  static constexpr int OFF_Q = 0;                        // Q: NP panels, K-major
  static constexpr int OFF_K = OFF_Q + NP * PANEL;       // K: 2 buffers x NP panels, K-major (B of S = Q K^T)
  static constexpr int OFF_V = OFF_K + 2 * NP * PANEL;   // V: 2 buffers x NP panels, MN-major (B of O = P V)
  static constexpr int OFF_PH = OFF_V + 2 * NP * PANEL;  // P hi: 2 panels (128 keys), K-major
  static constexpr int OFF_PL = OFF_PH + 2 * PANEL;      // P lo
  static constexpr int OFF_META = OFF_PL + 2 * PANEL;    // 2 buffers x int2 [NK]: (position, last visible)
  static constexpr int SMEM = OFF_META + 2 * NK * 8;     // 227 KB at head_dim 128
  static constexpr int TMEM_S = 0;                       // S: columns [0, NK)
  static constexpr int TMEM_O = NK;                      // O: columns [NK, NK + D)
  static constexpr uint32_t TMEM_COLS = 256;
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(G >= 1 && G <= 8, "1 <= G <= 8");
};

struct PrefillArgs {
  const uint4* K;            // cache K pool [NH][cap][D/8] (chunk-permuted rows)
  const uint4* V;            // cache V pool [NH][cap][D/8]
  const int32_t* len;        // [NH] retained lengths before the chunk
  const int32_t* slot_pos;   // [NH][cap]
  const uint8_t* ring_flag;  // [NH][w]
  const uint4* q;            // bf16 [B][Hq][C][D]
  const uint4* kc;           // bf16 [B][Hkv][C][D], the chunk's keys
  const uint4* vc;           // bf16 [B][Hkv][C][D]
  const float* logits;       // fp32 [B][Hkv][C]
  float* out;                // fp32 [B][Hq][C][D]
  int32_t* err;
  int NH, Hkv, cap, w, C;
  int t0;                    // position of the chunk's first token
  float qscale;              // scale * log2(e)
};

template <int D, int G>
__global__ void __launch_bounds__(128, 1) prefill_attention_kernel(const PrefillArgs a) {
  using Sh = PrefillShape<D, G>;
  constexpr int NK = Sh::NK, PT = Sh::PT, ROWS = Sh::ROWS, CH = D / 8, PANEL = Sh::PANEL;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_s;
  __shared__ __align__(8) uint64_t bar_o;
  __shared__ uint32_t tmem_base;
  uint8_t* sQ = smem + Sh::OFF_Q;
  uint8_t* sK0 = smem + Sh::OFF_K;
  uint8_t* sV0 = smem + Sh::OFF_V;
  uint8_t* sPH = smem + Sh::OFF_PH;
  uint8_t* sPL = smem + Sh::OFF_PL;
  int2* meta0 = reinterpret_cast<int2*>(smem + Sh::OFF_META);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int i = blockIdx.y;  // (sequence, KV head)
  const int b = i / a.Hkv, h = i - b * a.Hkv;
  const int c0 = blockIdx.x * PT;
  const int Hq = a.Hkv * G;

  // Launched as a programmatic dependent: the cache state written by earlier
  // kernels is visible after this wait.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) umma::tmem_alloc(&tmem_base, Sh::TMEM_COLS);
  if (tid == 0) {
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    fence_barrier_init();
  }
  // Q tile: row r = (head g = r / PT, chunk position c0 + r % PT); unused rows are zero.
  for (int x = tid; x < 128 * CH; x += 128) {
    const int r = x / CH, cc = x % CH;
    const int g = r / PT, c = c0 + r % PT;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < ROWS && c < a.C) val = __ldg(a.q + ((static_cast<size_t>(b) * Hq + h * G + g) * a.C + c) * CH + cc);
    *reinterpret_cast<uint4*>(sQ + (cc >> 3) * PANEL + r * 128 + (((cc & 7) ^ (r & 7)) << 4)) = val;
  }
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's lanes

  // This thread's row.
  const int r = tid;
  const int rg = r / PT, rc = c0 + r % PT;
  const bool row_ok = r < ROWS && rc < a.C;
  const int tq = a.t0 + rc;  // the row's query position
  float m_run = -INFINITY, l_run = 0.f;

  const int L = a.len[i];
  const int nkc = (L + NK - 1) / NK;          // tiles of retained cache slots
  const int kend = min(a.C, c0 + PT);         // chunk keys any row of this tile can see
  const int nkk = (kend + NK - 1) / NK;       // tiles of chunk keys
  const int ntiles = nkc + nkk;
  const int pend_lo = a.t0 - a.w;             // cached positions >= this may still carry a mark
  int n_s = 0, n_o = 0;                       // commits issued on bar_s / bar_o (uniform)
  int w_s = 0, w_o = 0;                       // of which waited for
  bool failed = false;

  // Tile it: keys [k0, k0 + kn) of the cache's retained slots (it < nkc) or of
  // the chunk.  K and V tiles go to buffer it & 1 with asynchronous 16-byte
  // copies (rows past kn are zero-filled); cache K rows already hold chunk c at
  // c ^ (slot & 7), and slot & 7 == j & 7 because tiles start at multiples of
  // 128, so their swizzled position is c itself.
  auto stage = [&](int t) {
    const bool from_cache = t < nkc;
    const int k0 = from_cache ? t * NK : (t - nkc) * NK;
    const int kn = from_cache ? min(NK, L - k0) : min(NK, kend - k0);
    uint8_t* dK = sK0 + (t & 1) * (Sh::NP * PANEL);
    uint8_t* dV = sV0 + (t & 1) * (Sh::NP * PANEL);
    const uint4* gK = from_cache ? a.K + static_cast<size_t>(i) * a.cap * CH : a.kc + static_cast<size_t>(i) * a.C * CH;
    const uint4* gV = from_cache ? a.V + static_cast<size_t>(i) * a.cap * CH : a.vc + static_cast<size_t>(i) * a.C * CH;
#pragma unroll 4
    for (int x = tid; x < NK * CH; x += 128) {
      const int j = x / CH, cc = x % CH;
      const bool ok = j < kn;
      const size_t src = ok ? static_cast<size_t>(k0 + j) * CH + cc : 0;
      const int kpos = from_cache ? (cc & 7) : ((cc & 7) ^ (j & 7));
      umma::cp_async16(dK + (cc >> 3) * PANEL + j * 128 + (kpos << 4), gK + src, ok);
      umma::cp_async16(dV + (cc >> 3) * PANEL + j * 128 + (((cc & 7) ^ (j & 7)) << 4), gV + src, ok);
    }
  };
  // Key metadata of tile t into buffer t & 1: (position, last visible position).
  auto stage_meta = [&](int t) {
    const bool from_cache = t < nkc;
    const int k0 = from_cache ? t * NK : (t - nkc) * NK;
    const int kn = from_cache ? min(NK, L - k0) : min(NK, kend - k0);
    const int j = tid;  // NK == blockDim.x
    int pos = INT_MAX, last = -1;  // invisible
    if (j < kn) {
      if (from_cache) {
        pos = a.slot_pos[static_cast<size_t>(i) * a.cap + k0 + j];
        const bool marked = pos >= pend_lo && a.ring_flag[static_cast<size_t>(i) * a.w + pos % a.w] != 0;
        last = marked ? pos + a.w - 1 : INT_MAX;
      } else {
        pos = a.t0 + k0 + j;
        const bool marked = a.logits[static_cast<size_t>(i) * a.C + k0 + j] > 0.0f;
        last = marked ? pos + a.w - 1 : INT_MAX;
      }
    }
    meta0[(t & 1) * NK + j] = make_int2(pos, last);
  };
  if (ntiles > 0) {
    stage(0);
    umma::cp_async_commit();
    stage_meta(0);
  }

  for (int it = 0; it < ntiles; ++it) {
    // The previous P V must be done: it reads the V and P tiles (and the K/V
    // buffer refilled below held tile it - 1) and writes O.
    if (w_o < n_o) {
      const bool ok = mbar_wait(&bar_o, w_o & 1);
      ++w_o;
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      umma::fence_after_sync();
    }
    // ---- 1. prefetch tile it + 1, then wait for tile it's copies ----
    if (it + 1 < ntiles) stage(it + 1);
    umma::cp_async_commit();
    umma::cp_async_wait_prior();
    const uint8_t* sK = sK0 + (it & 1) * (Sh::NP * PANEL);
    const uint8_t* sV = sV0 + (it & 1) * (Sh::NP * PANEL);
    const int2* meta = meta0 + (it & 1) * NK;
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();

    // ---- 2. S = Q K^T ----
    if (tid == 0) {
      umma::fence_after_sync();
      constexpr uint32_t idq = umma::idesc_bf16(128, NK, 0);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * PANEL + (kk & 3) * 32;
        umma::mma_bf16(tmem + Sh::TMEM_S, umma::sw128_desc(umma::smem_u32(sQ) + off, 16, 1024),
                       umma::sw128_desc(umma::smem_u32(sK) + off, 16, 1024), idq, kk > 0);
      }
      umma::commit(&bar_s);
    }
    ++n_s;
    if (it + 1 < ntiles) stage_meta(it + 1);  // overlaps the S MMA
    {
      const bool ok = mbar_wait(&bar_s, w_s & 1);
      ++w_s;
      if (__syncthreads_or(!ok)) {
        failed = true;
        break;
      }
      umma::fence_after_sync();
    }

    // ---- 3. softmax of this thread's row ----
    float s[NK];
#pragma unroll
    for (int cb = 0; cb < NK / 32; ++cb) {
      float v[32];
      umma::ld32(trow + Sh::TMEM_S + cb * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) s[cb * 32 + j] = v[j];
    }
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      const int2 mk = meta[j];
      const bool vis = row_ok && mk.x <= tq && tq <= mk.y;
      s[j] = vis ? s[j] * a.qscale : -INFINITY;
      mt = fmaxf(mt, s[j]);
    }
    bool rescale = false;
    float factor = 1.f;
    if (mt > m_run + 8.f) {  // also when m_run is still -inf and this tile has a visible key
      if (m_run != -INFINITY) {
        factor = fast_exp2(m_run - mt);
        rescale = true;
        l_run *= factor;
      }
      m_run = mt;
    }
    const float mref = m_run == -INFINITY ? 0.f : m_run;  // rows with nothing visible yet: p = 0
    float psum = 0.f;
#pragma unroll
    for (int q8 = 0; q8 < NK / 8; ++q8) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p0 = fast_exp2(s[q8 * 8 + 2 * e] - mref);
        const float p1 = fast_exp2(s[q8 * 8 + 2 * e + 1] - mref);
        psum += p0 + p1;
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
        const float2 hf = __bfloat1622float2(h2);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
        hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
        lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
      }
      const int off = (q8 >> 3) * PANEL + r * 128 + (((q8 & 7) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(sPH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sPL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    l_run += psum;
    // Rescale this warp's accumulator rows in tensor memory (warp-collective).
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        float o[32];
        umma::ld32(trow + Sh::TMEM_O + cb * 32, o);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] *= factor;
        umma::st32(trow + Sh::TMEM_O + cb * 32, o);
      }
    }
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    __syncthreads();

    // ---- 4. O += P_hi V + P_lo V ----
    if (tid == 0) {
      umma::fence_after_sync();
      constexpr uint32_t idp = umma::idesc_bf16(128, D, 1);
#pragma unroll
      for (int kk = 0; kk < NK / 16; ++kk) {
        const uint32_t aoff = (kk >> 2) * PANEL + (kk & 3) * 32;
        const uint64_t bd = umma::sw128_desc(umma::smem_u32(sV) + kk * 2048, PANEL, 1024);
        umma::mma_bf16(tmem + Sh::TMEM_O, umma::sw128_desc(umma::smem_u32(sPH) + aoff, 16, 1024), bd, idp,
                       it > 0 || kk > 0);
        umma::mma_bf16(tmem + Sh::TMEM_O, umma::sw128_desc(umma::smem_u32(sPL) + aoff, 16, 1024), bd, idp, true);
      }
      umma::commit(&bar_o);
    }
    ++n_o;
  }

  if (!failed && w_o < n_o) {
    const bool ok = mbar_wait(&bar_o, w_o & 1);
    ++w_o;
    failed = __syncthreads_or(!ok);
    umma::fence_after_sync();
  }
  if (!failed && ntiles > 0) {
    // ---- epilogue: O / l -> out ----
    const float inv = row_ok && l_run > 0.f ? 1.f / l_run : 0.f;
    float* orow = a.out + ((static_cast<size_t>(b) * Hq + h * G + rg) * a.C + rc) * D;
#pragma unroll
    for (int cb = 0; cb < D / 32; ++cb) {
      float o[32];
      umma::ld32(trow + Sh::TMEM_O + cb * 32, o);
      if (row_ok) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(orow + cb * 32 + j) =
              make_float4(o[j] * inv, o[j + 1] * inv, o[j + 2] * inv, o[j + 3] * inv);
      }
    }
  }
  if (failed) {
    if (tid == 0) atomicOr(a.err, kErrBitTimeout);
    umma::cp_async_wait_all();
    // Wait (bounded) for the tensor-core work still in flight before freeing its memory.
    for (; w_s < n_s; ++w_s) (void)mbar_wait(&bar_s, w_s & 1);
    for (; w_o < n_o; ++w_o) (void)mbar_wait(&bar_o, w_o & 1);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) umma::tmem_dealloc(tmem, Sh::TMEM_COLS);
}

}  // namespace dms
