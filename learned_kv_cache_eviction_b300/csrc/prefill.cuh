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
// One CTA of 256 threads per (tile of PT = 128 / G query positions x G query
// heads, KV head).  Row r of the tile is query head g = r / PT at chunk
// position c0 + r % PT, tensor-memory lane r; threads r and r + 128 share row
// r (the two warps of a lane quarter), each owning half of its keys in the
// softmax and half of its output columns.  For each
// tile of 128 keys (the cache's retained slots first, then the chunk's keys up
// to the tile's last position):
//   1. the threads stage the K and V tile in shared memory in the 128-byte
//      swizzled layouts (K rows of the cache pool are stored chunk-permuted by
//      slot, which is that layout already), plus each key's (position, last);
//      K, V and the metadata are double-buffered: the next tile's asynchronous
//      copies (cp.async) are in flight while this one is computed;
//   2. one thread issues S = Q K^T (bf16 x bf16 -> fp32 in tensor memory);
//   3. each thread of a row loads its half of the row of S, masks it and
//      finds its max, and the two threads swap their maxima through tensor
//      memory (so they take the same decisions); the running max
//      moves only when it grows by more than 2^8 (the accumulator in tensor
//      memory is rescaled then); each thread turns its 64 keys into
//      p = 2^(s - m) and keeps its half of the row sum; p is written as two bf16
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
  static constexpr int TMEM_S = 0;                       // S: 2 buffers, columns [0, 2 NK)
  static constexpr int TMEM_O = 2 * NK;                  // O: columns [2 NK, 2 NK + D)
  static constexpr int TMEM_X = 2 * NK + D;              // the two half-row maxima of each row
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(TMEM_X + 2 <= static_cast<int>(TMEM_COLS), "tensor memory columns");
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static_assert(G >= 1 && G <= 8, "1 <= G <= 8");
};

struct PrefillArgs {
  const uint4* K;            // cache K pool [NH][cap][D/8] (chunk-permuted rows)
  const uint4* V;            // cache V pool [NH][cap][D/8]
  const int32_t* len;        // [NH] retained lengths before the chunk (the current buffer)
  const int32_t* slot_pos;   // [NH][cap]
  const uint8_t* ring_flag;  // [2][NH][w], entry of position p at ring_index(NH, w, i, p)
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
__global__ void __launch_bounds__(256, 1) prefill_attention_kernel(const PrefillArgs a) {
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
  for (int x = tid; x < 128 * CH; x += 256) {
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
  const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);  // this warp's lanes

  // This thread's row, and which half of its columns (keys, then outputs) it owns.
  const int r = tid & 127, hh = tid >> 7;
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
  const int tq_first = a.t0 + c0;                          // query positions of the CTA's rows
  const int tq_last = a.t0 + min(a.C, c0 + PT) - 1;
  bool nomask_next = false;                   // tile-wide "no mask" flag of the next tile (uniform)
  int n_s = 0, n_o = 0;                       // commits issued on bar_s / bar_o (uniform)
  int w_s = 0, w_o = 0;                       // of which waited for
  bool failed = false;

  // Tile t: keys [k0, k0 + kn) of the cache's retained slots (t < nkc) or of
  // the chunk.  Its K and V go to buffers t & 1 with asynchronous 16-byte
  // copies (rows past kn are zero-filled); cache K rows already hold chunk c at
  // c ^ (slot & 7), and slot & 7 == j & 7 because tiles start at multiples of
  // 128, so their swizzled position is c itself.  K and V are staged
  // separately: a K buffer is free once its S = Q K^T is done, a V buffer only
  // once its P V is.
  auto tile_keys = [&](int t, int& k0, int& kn) -> bool {
    const bool from_cache = t < nkc;
    k0 = from_cache ? t * NK : (t - nkc) * NK;
    kn = from_cache ? min(NK, L - k0) : min(NK, kend - k0);
    return from_cache;
  };
  auto stage_rows = [&](int t, bool is_v) {
    int k0, kn;
    const bool from_cache = tile_keys(t, k0, kn);
    uint8_t* dst = (is_v ? sV0 : sK0) + (t & 1) * (Sh::NP * PANEL);
    const uint4* g = is_v ? (from_cache ? a.V : a.vc) : (from_cache ? a.K : a.kc);
    g += static_cast<size_t>(i) * (from_cache ? a.cap : a.C) * CH;
    const bool pre_swizzled = from_cache && !is_v;
    // Thread tid copies chunk cc = tid % CH of rows j0, j0 + JS, j0 + 2 JS, ...;
    // JS is a multiple of 8, so every one of its rows has the same swizzle.
    constexpr int JS = 256 / CH;
    static_assert(JS % 8 == 0 && NK % JS == 0, "rows per pass");
    const int cc = tid % CH, j0 = tid / CH;
    const int pos = pre_swizzled ? (cc & 7) : ((cc & 7) ^ (j0 & 7));
    uint8_t* d0 = dst + (cc >> 3) * PANEL + j0 * 128 + (pos << 4);
    const uint4* s0 = g + static_cast<size_t>(k0 + j0) * CH + cc;
#pragma unroll
    for (int k = 0; k < NK / JS; ++k) {
      const bool ok = j0 + k * JS < kn;
      umma::cp_async16(d0 + k * JS * 128, ok ? s0 + k * JS * CH : g, ok);
    }
  };
  // Key metadata of tile t into buffer t & 1: (position, last visible position).
  // Split in two so that the loads of meta_begin are in flight while the
  // softmax of the current tile runs: a key's position (and, for a chunk key,
  // its logit) first; then, in meta_end, the ring lookup that only cached keys
  // among the last w positions need, and the store.
  auto meta_begin = [&](int t, int& pos, float& lg) {
    int k0, kn;
    const bool from_cache = tile_keys(t, k0, kn);
    const int j = tid;  // threads [0, NK) handle one key each
    pos = INT_MAX;
    lg = 0.f;
    if (j < NK && j < kn) {
      if (from_cache) {
        pos = a.slot_pos[static_cast<size_t>(i) * a.cap + k0 + j];
      } else {
        pos = a.t0 + k0 + j;
        lg = a.logits[static_cast<size_t>(i) * a.C + k0 + j];
      }
    }
  };
  // Returns whether this key is a key of the tile that every row of the CTA
  // sees (or lies past the tile's end), for the tile-wide "no mask" test.
  auto meta_end = [&](int t, int pos, float lg) -> bool {
    if (tid >= NK) return true;
    int k0, kn;
    const bool from_cache = tile_keys(t, k0, kn);
    int last = -1;  // invisible unless set below
    if (pos != INT_MAX) {
      const bool marked = from_cache
                              ? (pos >= pend_lo && a.ring_flag[ring_index(a.NH, a.w, i, pos)] != 0)
                              : lg > 0.0f;
      last = marked ? pos + a.w - 1 : INT_MAX;
    }
    meta0[(t & 1) * NK + tid] = make_int2(pos, last);
    return tid >= kn || (pos <= tq_first && last >= tq_last);
  };
  auto issue_s = [&](int t) {  // S(t) = Q K(t)^T into S buffer t & 1; one thread
    constexpr uint32_t idq = umma::idesc_bf16(128, NK, 0);
    const uint32_t kbase = umma::smem_u32(sK0 + (t & 1) * (Sh::NP * PANEL));
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * PANEL + (kk & 3) * 32;
      umma::mma_bf16(tmem + Sh::TMEM_S + (t & 1) * NK, umma::sw128_desc(umma::smem_u32(sQ) + off, 16, 1024),
                     umma::sw128_desc(kbase + off, 16, 1024), idq, kk > 0);
    }
    umma::commit(&bar_s);
  };
  auto issue_pv = [&](int t) {  // O += P_hi V(t) + P_lo V(t); one thread
    constexpr uint32_t idp = umma::idesc_bf16(128, D, 1);
    const uint32_t vbase = umma::smem_u32(sV0 + (t & 1) * (Sh::NP * PANEL));
#pragma unroll
    for (int kk = 0; kk < NK / 16; ++kk) {
      const uint32_t aoff = (kk >> 2) * PANEL + (kk & 3) * 32;
      const uint64_t bd = umma::sw128_desc(vbase + kk * 2048, PANEL, 1024);
      umma::mma_bf16(tmem + Sh::TMEM_O, umma::sw128_desc(umma::smem_u32(sPH) + aoff, 16, 1024), bd, idp,
                     t > 0 || kk > 0);
      umma::mma_bf16(tmem + Sh::TMEM_O, umma::sw128_desc(umma::smem_u32(sPL) + aoff, 16, 1024), bd, idp, true);
    }
    umma::commit(&bar_o);
  };

  // ---- prologue: K and V of tile 0, K of tile 1, metadata of tile 0; S(0) ----
  if (ntiles > 0) {
    stage_rows(0, false);
    stage_rows(0, true);
    umma::cp_async_commit();
    if (ntiles > 1) stage_rows(1, false);
    umma::cp_async_commit();
    bool all_vis;
    {
      int pos;
      float lg;
      meta_begin(0, pos, lg);
      all_vis = meta_end(0, pos, lg);
    }
    umma::cp_async_wait_prior();
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    nomask_next = __syncthreads_and(all_vis);
    if (tid == 0) {
      umma::fence_after_sync();
      issue_s(0);
    }
    ++n_s;
  }

  // Tile it: the tensor core runs S(it + 1) and P V(it - 1) .. P V(it) while the
  // threads work on the softmax of tile it.
  for (int it = 0; it < ntiles; ++it) {
    const int bf = it & 1;
    const bool nomask = nomask_next;  // every valid key of tile it is visible to every row
    // (a) S(it) is done: S buffer bf can be read, K buffer bf is free again.
    // Every thread observes the commit itself; a wait that timed out is only
    // recorded here, and the CTA decides at the barrier of (g) to stop (the
    // thread meanwhile reads stale tensor memory of its own allocation).
    bool bad = !mbar_wait(&bar_s, w_s & 1);
    ++w_s;
    umma::fence_after_sync();
    // (b) prefetch K(it + 2) into K buffer bf; start loading the metadata of
    // tile it + 1 (stored in (f)).
    if (it + 2 < ntiles) stage_rows(it + 2, false);
    umma::cp_async_commit();
    int npos = INT_MAX;
    float nlg = 0.f;
    if (it + 1 < ntiles) meta_begin(it + 1, npos, nlg);

    // (c) softmax of this thread's row: each thread loads its own half of the
    // row (keys hh NK/2 .. hh NK/2 + NK/2 - 1, P panel hh), masks it and finds
    // its max; the two threads of a row (the same lane in warps w and w ^ 4)
    // swap their maxima through tensor memory, so they take the same decisions.
    const int2* meta = meta0 + bf * NK + hh * (NK / 2);
    static_assert(NK / 2 == 64, "one 64-column load per half row");
    float s[NK / 2];
    umma::ld64(trow + Sh::TMEM_S + bf * NK + hh * (NK / 2), s);
    float mt = -INFINITY;
    if (nomask && row_ok) {
      int k0, kn;
      tile_keys(it, k0, kn);
      kn -= hh * (NK / 2);  // this half's valid keys (warp-uniform)
      if (kn >= NK / 2) {   // a full half: no key to drop
#pragma unroll
        for (int j = 0; j < NK / 2; j += 2) {
          const float2 v = __fmul2_rn(make_float2(s[j], s[j + 1]), make_float2(a.qscale, a.qscale));
          s[j] = v.x;
          s[j + 1] = v.y;
        }
      } else {
#pragma unroll
        for (int j = 0; j < NK / 2; j += 2) {
          const float2 v = __fmul2_rn(make_float2(s[j], s[j + 1]), make_float2(a.qscale, a.qscale));
          s[j] = j < kn ? v.x : -INFINITY;
          s[j + 1] = j + 1 < kn ? v.y : -INFINITY;
        }
      }
#pragma unroll
      for (int j = 0; j < NK / 2; j += 4) mt = fmaxf(mt, fmaxf(fmaxf(s[j], s[j + 1]), fmaxf(s[j + 2], s[j + 3])));
    } else {
#pragma unroll
      for (int j = 0; j < NK / 2; ++j) {
        const int2 mk = meta[j];
        const bool vis = row_ok && mk.x <= tq && tq <= mk.y;
        s[j] = vis ? s[j] * a.qscale : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
    }
    // Swap the half-row maxima: write own column, pair barrier (the two warps
    // of this lane quarter; every thread of both reaches it once per tile),
    // read the other's column.
    umma::st1(trow + Sh::TMEM_X + hh, mt);
    umma::fence_before_sync();
    asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
    umma::fence_after_sync();
    mt = fmaxf(mt, umma::ld1(trow + Sh::TMEM_X + (hh ^ 1)));
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
    // Pairs of keys in packed fp32 arithmetic (each lane of a pair rounds as
    // the scalar operation would).
    const float2 nref = make_float2(-mref, -mref);
    float2 psum2 = make_float2(0.f, 0.f);
    uint32_t hi[NK / 16][4], lo[NK / 16][4];
#pragma unroll
    for (int qq = 0; qq < NK / 16; ++qq) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __fadd2_rn(make_float2(s[qq * 8 + 2 * e], s[qq * 8 + 2 * e + 1]), nref);
        const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
        psum2 = __fadd2_rn(psum2, p);
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(p.x, p.y);
        const float2 hf = __bfloat1622float2(h2);
        const float2 d = __fadd2_rn(p, make_float2(-hf.x, -hf.y));
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(d.x, d.y);
        hi[qq][e] = *reinterpret_cast<const uint32_t*>(&h2);
        lo[qq][e] = *reinterpret_cast<const uint32_t*>(&l2);
      }
    }
    const float psum = psum2.x + psum2.y;

    // (d) P V(it - 1) is done: the P buffers, O and V buffer bf ^ 1 are free
    // (observed by every thread itself, as in (a)).
    if (w_o < n_o) {
      bad = !mbar_wait(&bar_o, w_o & 1) || bad;
      ++w_o;
      umma::fence_after_sync();
    }
    // (e) prefetch V(it + 1) into V buffer bf ^ 1.
    if (it + 1 < ntiles) stage_rows(it + 1, true);
    umma::cp_async_commit();
    // (f) rescale this warp's accumulator rows (warp-collective; each half of the
    // threads owns half of the output columns), then write P.
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int cb = hh * (D / 64) + cc;
        float o[32];
        umma::ld32(trow + Sh::TMEM_O + cb * 32, o);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] *= factor;
        umma::st32(trow + Sh::TMEM_O + cb * 32, o);
      }
    }
#pragma unroll
    for (int qq = 0; qq < NK / 16; ++qq) {
      const int q8 = hh * (NK / 16) + qq;
      const int off = (q8 >> 3) * PANEL + r * 128 + (((q8 & 7) ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(sPH + off) = make_uint4(hi[qq][0], hi[qq][1], hi[qq][2], hi[qq][3]);
      *reinterpret_cast<uint4*>(sPL + off) = make_uint4(lo[qq][0], lo[qq][1], lo[qq][2], lo[qq][3]);
    }
    l_run += psum;
    const bool nvis = it + 1 < ntiles ? meta_end(it + 1, npos, nlg) : true;
    // (g) K(it + 1) and V(it) have landed (all groups but the two just committed).
    umma::cp_async_wait_two();
    umma::fence_proxy_async_smem();
    umma::fence_before_sync();
    // One barrier per tile in the common case: it also carries the "no mask"
    // vote for tile it + 1 and the waits' outcome; a second one tells them
    // apart when the vote fails (a masked next tile, or a timed-out wait).
    if (__syncthreads_and(nvis && !bad)) {
      nomask_next = true;
    } else {
      nomask_next = false;
      if (__syncthreads_or(bad)) {
        failed = true;
        break;
      }
    }
    // (h) S(it + 1) first, so that the next softmax can start, then P V(it).
    if (tid == 0) {
      umma::fence_after_sync();
      if (it + 1 < ntiles) issue_s(it + 1);
      issue_pv(it);
    }
    if (it + 1 < ntiles) ++n_s;
    ++n_o;
  }

  if (!failed && w_o < n_o) {
    const bool ok = mbar_wait(&bar_o, w_o & 1);
    ++w_o;
    failed = __syncthreads_or(!ok);
    umma::fence_after_sync();
  }
  if (!failed && ntiles > 0) {
    // ---- epilogue: O / l -> out; the row sum is the two halves' sums, swapped
    // through shared memory that no MMA reads any more ----
    float* lsw = reinterpret_cast<float*>(sPH);
    lsw[hh * 128 + r] = l_run;
    __syncthreads();
    const float l_row = l_run + lsw[(1 - hh) * 128 + r];
    const float inv = row_ok && l_row > 0.f ? 1.f / l_row : 0.f;
    float* orow = a.out + ((static_cast<size_t>(b) * Hq + h * G + rg) * a.C + rc) * D;
#pragma unroll
    for (int cc = 0; cc < D / 64; ++cc) {
      const int cb = hh * (D / 64) + cc;
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
