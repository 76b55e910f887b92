// Incremental decoding over a key/value cache (sm_103a).
//
// The NanoEuler engine generates text one token at a time with a KV cache
// (mynewscn README, generation with the KV cache; socker-news README, GPU
// generation mode `i`).  A decode step is the same attention as the training
// forward restricted to the newest positions: the Tq new queries sit at
// positions Tkv - Tq .. Tkv - 1 and attend causally to the cached positions
// 0 .. Tkv - 1, so o and lse equal those rows of the forward over T = Tkv.
//
//   k_kv_append       new keys rotated (fp16) and new values copied into the caches
//   k_decode_q        the Tq x G query rows of each key/value head rotated and
//                     packed into one 128-row tile (row t * G + g; zero rows after);
//                     with at most 32 (64) rows the tile holds 4 (2) copies of them
//                     and copy f takes key columns f * 128 / F .. of every key tile,
//                     so the exponentials of a tile are spread over four warps
//   k_decode          split sweep over the cache: one CTA per SM loops over work
//                     items (batch, key/value head, split of the key tiles);
//                     S = Q K^T and O += P V on the tensor cores, an online softmax
//                     in between; each item leaves its unnormalised O and its
//                     running max and sum for the rows of the tile, and the CTA
//                     that finishes a group's last split merges the group's
//                     partials: O = sum 2^(m_s - m) O_s / l
//
// Decode streams the cache once and does little arithmetic per byte, so the
// sweep is bound by HBM; the G query heads of a key/value head (and the Tq
// tokens) share every K/V tile through the M dimension of the MMAs.  The
// caches are head-major ([B, Hkv, Tcap, D]): a work item reads one contiguous
// stretch of each.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace ne {
namespace {

constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, 0, kStatusTimeout);
}

// ====================================================================== cache append
template <int D>
__global__ void __launch_bounds__(256) k_kv_append(const KvAppendArgs a) {
  constexpr int kCPR = D / 8;
  const uint32_t n = (uint32_t)a.B * a.Tn * a.Hkv * kCPR;
  for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < n; it += gridDim.x * blockDim.x) {
    const uint32_t row = it / kCPR;  // (b, t, g)
    const int c = (int)(it % kCPR);
    const uint32_t bt = fdiv(row, a.div_hkv);
    const uint32_t g = row - bt * a.Hkv;
    const uint32_t b = fdiv(bt, a.div_tn);
    const uint32_t t = bt - b * a.Tn;
    const int pos = a.pos0 + (int)t;
    const uint4 kv = load_rope_chunk<D>(a.k + (size_t)row * D, c, a.rope_half != 0);
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(a.v) + it);
    float4 c0, c1;
    rope_coeffs<D>(a.rope, pos, c, c0, c1);
    const size_t dst = (((size_t)b * a.Hkv + g) * a.Tcap + pos) * kCPR + c;  // head-major cache
    reinterpret_cast<uint4*>(a.kc)[dst] = rope_chunk_f16(kv, c0, c1, nullptr);
    reinterpret_cast<uint4*>(a.vc)[dst] = vv;
  }
}

// ====================================================================== merging the partials
// Row r (token r / G, head g * G + r % G) of group bk = b * Hkv + g, one warp:
// O = sum_s 2^(m_s - m) O_s / l with l = sum_s 2^(m_s - m) l_s over the
// nsplit x F partials (splits of the cache, copies of the query rows).
template <int D>
__device__ __forceinline__ void merge_row(const DecodeArgs& a, int bk, int r, int lane) {
  constexpr int kPer = D / 32;
  const int b = bk / a.Hkv, g = bk - b * a.Hkv;
  const int t = r / a.G, h = g * a.G + (r - t * a.G);
  const int npart = a.nsplit * a.F;
  const size_t base = (size_t)bk * npart;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
  float m = -INFINITY;
  for (int p = 0; p < npart; p++) m = fmaxf(m, __ldcg(&ml[(base + p) * a.R + r].x));
  float acc[kPer], L = 0.f;
#pragma unroll
  for (int e = 0; e < kPer; e++) acc[e] = 0.f;
  for (int p = 0; p < npart; p++) {
    const size_t pr = (base + p) * a.R + r;
    const float2 v = __ldcg(&ml[pr]);
    if (v.y == 0.f) continue;  // no visible key in this part
    const float w = ex2(v.x - m);
    L += w * v.y;
#pragma unroll
    for (int e = 0; e < kPer; e++) acc[e] += w * __ldcg(a.part_o + pr * D + lane + 32 * e);
  }
  const float inv = 1.f / L;
  const size_t orow = (((size_t)b * a.Tq + t) * a.Hq + h) * D;
#pragma unroll
  for (int e = 0; e < kPer; e++) {
    if (a.o_fp32)
      static_cast<float*>(a.o)[orow + lane + 32 * e] = acc[e] * inv;
    else
      static_cast<__nv_bfloat16*>(a.o)[orow + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
  }
  if (lane == 0) a.lse[((size_t)b * a.Hq + h) * a.Tq + t] = (m + __log2f(L)) * kLn2;
}

// ====================================================================== packed queries
template <int D>
__global__ void __launch_bounds__(256) k_decode_q(const DecodeArgs a) {
  constexpr int kCPR = D / 8;
  const uint32_t n = (uint32_t)a.B * a.Hkv * kTile * kCPR;
  for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < n; it += gridDim.x * blockDim.x) {
    const uint32_t row = it / kCPR;  // (b * Hkv + g) * 128 + r
    const int c = (int)(it % kCPR);
    const uint32_t bk = row / kTile;
    const int r = (int)(row % kTile) % (kTile / a.F);  // copy (row % 128) / (128 / F) of query row r
    uint4 out = make_uint4(0, 0, 0, 0);
    if (r < a.R) {
      const int t = r / a.G, gg = r - t * a.G;
      const uint32_t b = bk / a.Hkv, g = bk - b * a.Hkv;
      const int h = (int)g * a.G + gg;
      const uint4 qv = load_rope_chunk<D>(a.q + (((size_t)b * a.Tq + t) * a.Hq + h) * D, c, a.rope_half != 0);
      float4 c0, c1;
      rope_coeffs<D>(a.rope, a.Tkv - a.Tq + t, c, c0, c1);
      out = rope_chunk_f16(qv, c0, c1, nullptr);
    }
    reinterpret_cast<uint4*>(a.qpk)[it] = out;
  }
  // the sweep counts finished splits per (batch, kv head) group from zero
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)(a.B * a.Hkv); i += gridDim.x * blockDim.x)
    a.done[i] = 0u;
}

// ====================================================================== split sweep
template <int D>
struct DecCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr uint32_t kSpan = D * 2;
  static constexpr uint32_t kSwz = D == 64 ? kSw128 : kSw64;
  static constexpr uint32_t kSBO = 8 * kSpan;
  static constexpr int kStages = D == 64 ? 6 : 8;  // K/V ring: decode is bound by the bytes in flight
  static constexpr uint32_t kColO = 0, kColS = 64, kColP = 192, kTmemCols = 256;
  static constexpr int kThreads = 224;  // 0 producer, 1 S issuer, 2-5 softmax, 6 PV issuer
  static constexpr int kOffQ = 0;       // [2]
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 32 * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct DecItem {
  int bk, s, n0, n1;  // (batch, kv head) index, split, key tiles [n0, n1)
};

__device__ __forceinline__ bool dec_item(const DecodeArgs& a, int tl, DecItem& it) {
  const int w = tl * (int)gridDim.x + (int)blockIdx.x;
  const int per_s = a.B * a.Hkv;
  if (w >= per_s * a.nsplit) return false;
  it.s = w / per_s;
  it.bk = w - it.s * per_s;
  it.n0 = (int)((long long)it.s * a.ntk / a.nsplit);
  it.n1 = (int)((long long)(it.s + 1) * a.ntk / a.nsplit);
  return true;
}

// Softmax role of the decode sweep for one warp: rows of its TMEM lane quarter
// (copy f of the query rows), key columns f * W .. f * W + W - 1 of every tile.
// Returns false if a wait gave up.
template <int D, int W>
__device__ __forceinline__ bool decode_softmax(const DecodeArgs& a, uint32_t tmem, int warp, int lane, uint64_t* s_full,
                                               uint64_t* s_read, uint64_t* p_ready, uint64_t* pv_done,
                                               uint64_t* o_free, uint64_t* part_done, uint64_t* merge_go,
                                               volatile int* merge_flag, int nact, volatile int* abort) {
  using C = DecCfg<D>;
  const int q4 = warp & 3;        // TMEM lane quarter
  const int rr = q4 * 32 + lane;  // row of the packed tile
  const int span = kTile / a.F;
  const int f = rr / span, r = rr % span;  // copy, query row (token r / G, head r % G of the group)
  const int c0 = f * W;                    // this copy's first key column of a tile
  const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
  const float sl2 = a.scale_log2;
  // this row's last visible key position (-1: a padding row sees none)
  const int qpos = r < a.R ? a.Tkv - a.Tq + r / a.G : -1;
  if (W < 128) {
    // the P columns of the other copies stay zero in this warp's lanes
    uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < 8; c++) tmem_st8(trow + C::kColP + c * 8, z);
    tmem_wait_st();
  }
  bool ok = true;
  int g = 0;
  DecItem it;
  for (int tl = 0; ok && dec_item(a, tl, it); tl++) {
    float r_max = -INFINITY, l = 0.f;  // raw-logit running maximum (as used) and sum
    for (int n = it.n0; n < it.n1; n++, g++) {
      ok = __all_sync(0xffffffffu, mbar_wait(s_full, g & 1, abort));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[W];
#pragma unroll
      for (int c = 0; c < W / 32; c++)
        tmem_ld32(trow + C::kColS + c0 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32 * c));
      tmem_wait_ld();
      tc_fence_before();
      warp_arrive(s_read);  // S of the next step may overwrite the score columns
      // keys after this row's position (and past the cache) are masked
      const int lim = qpos - n * kTile - c0;  // columns 0..lim of the slice are visible
      if (lim < W - 1) {
#pragma unroll
        for (int c = 0; c < W; c++)
          if (c > lim) s[c] = 0xff800000u;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < W; c += 2) mx = fmax3(mx, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
      const float r_new = fmaxf(r_max, mx);
      // lazy rescale of O and l when the maximum grows by more than 2^8
      float r_use = r_max;
      if (r_max == -INFINITY) {
        r_use = r_new;  // first visible keys of this item (O holds zeros so far)
      } else if (__fmul_rn(r_new, sl2) > __fmul_rn(r_max, sl2) + 8.0f) {
        r_use = r_new;
      }
      const bool resc = r_max != -INFINITY && r_use != r_max;
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold every earlier P V
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (g - 1) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        const float alpha = resc ? ex2(__fmul_rn(r_max, sl2) - __fmul_rn(r_use, sl2)) : 1.f;
        l *= alpha;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < D / 32; c++) {
          tmem_ld32(trow + C::kColO + c * 32, w);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e++) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
          tmem_st32(trow + C::kColO + c * 32, w);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      r_max = r_use;
      // P = exp2(s * scale_log2 - m) (0 while the row has seen no visible key)
      const float m_use = r_use == -INFINITY ? 0.f : __fmul_rn(r_use, sl2);
      const uint64_t sl2x2 = f2(sl2, sl2), negm = f2(-m_use, -m_use);
      uint64_t sum4[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pk[W / 2];
#pragma unroll
      for (int e = 0; e < W / 2; e++) {
        float x0, x1;
        f2_split(f2_fma(f2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), sl2x2, negm), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        pk[e] = pack_bf16(p0, p1);
        sum4[e & 3] = f2_add(sum4[e & 3], f2(p0, p1));
      }
      {
        float s0, s1, s2, s3, s4, s5, s6, s7;
        f2_split(sum4[0], s0, s1);
        f2_split(sum4[1], s2, s3);
        f2_split(sum4[2], s4, s5);
        f2_split(sum4[3], s6, s7);
        l += ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
      }
      // one P buffer: the previous step's P V has read it
      if (g >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (g - 1) & 1, abort));
        if (!ok) break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < W / 16; c++)
        tmem_st8(trow + C::kColP + c0 / 2 + c * 8, *reinterpret_cast<const uint32_t(*)[8]>(pk + 8 * c));
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(p_ready);
    }
    if (!ok) break;
    // the copy's partial result: unnormalised O, the max (log2 units) and the sum
    ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (g - 1) & 1, abort));
    if (!ok) break;
    tc_fence_after();
    const size_t prow = (((size_t)it.bk * a.nsplit + it.s) * a.F + f) * a.R + r;
#pragma unroll
    for (int c = 0; c < D / 32; c++) {
      uint32_t w[32];
      tmem_ld32(trow + C::kColO + c * 32, w);
      tmem_wait_ld();
      if (r < a.R) {
        float4* dst = reinterpret_cast<float4*>(a.part_o + prow * D + c * 32);
#pragma unroll
        for (int e = 0; e < 8; e++)
          dst[e] = make_float4(__uint_as_float(w[4 * e]), __uint_as_float(w[4 * e + 1]), __uint_as_float(w[4 * e + 2]),
                               __uint_as_float(w[4 * e + 3]));
      }
    }
    if (r < a.R)
      reinterpret_cast<float2*>(a.part_ml)[prow] = make_float2(r_max == -INFINITY ? -INFINITY : __fmul_rn(r_max, sl2), l);
    tc_fence_before();
    warp_arrive(o_free);  // the next item's first P V may overwrite O
    // The CTA that completes a group's last split merges the group's partials
    // (a count of finished splits per group; fences order the partials before it).
    __threadfence();
    warp_arrive(part_done);
    if (q4 == 0) {  // quarter 0 always holds query rows
      bool good = true;
      if (lane == 0) {
        good = mbar_wait(part_done, tl & 1, abort);
        if (good) {
          __threadfence();
          *merge_flag = atomicAdd(a.done + it.bk, 1u) == (unsigned)(a.nsplit - 1) ? 1 : 0;
          __threadfence();
          mbar_arrive(merge_go);
        }
      }
      ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
      if (!ok) break;
    }
    ok = __all_sync(0xffffffffu, mbar_wait(merge_go, tl & 1, abort));
    if (!ok) break;
    if (*merge_flag) {
      __threadfence();
      for (int row = (rr >> 5) % nact; row < a.R; row += nact)  // one warp per row
        merge_row<D>(a, it.bk, row, lane);
    }
  }
  return ok;
}

template <int D>
__global__ void __launch_bounds__(224, 1) k_decode(const __grid_constant__ DecodeArgs a) {
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int S = C::kStages;
  constexpr int TB = C::kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;            // [2]
  uint64_t* q_empty = bars + 2;       // [2]
  uint64_t* kv_full = bars + 4;       // [S]
  uint64_t* kv_empty = bars + 4 + S;  // [S]
  uint64_t* s_full = bars + 4 + 2 * S;
  uint64_t* s_read = s_full + 1;      // the softmax warps hold the scores in registers
  uint64_t* p_ready = s_full + 2;
  uint64_t* pv_done = s_full + 3;
  uint64_t* o_free = s_full + 4;      // an item's O has been read out
  uint64_t* drain = s_full + 5;       // [2]
  uint64_t* part_done = s_full + 7;   // the item's partials are written (one arrival per active softmax warp)
  uint64_t* merge_go = s_full + 8;    // merge_flag says whether this CTA merges the group
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 9);
  volatile int* abort = reinterpret_cast<volatile int*>(s_full + 9) + 1;
  volatile int* merge_flag = reinterpret_cast<volatile int*>(s_full + 9) + 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // softmax warps whose TMEM lane quarter holds query rows (the others sit out)
  int nact = 0;
  for (int q = 0; q < 4; q++) nact += ((q * 32) % (kTile / a.F)) < a.R ? 1 : 0;

  if (tid == 0) {
    *abort = 0;
    for (int k = 0; k < 2; k++) {
      mbar_init(q_full + k, 1);
      mbar_init(q_empty + k, 1);
      mbar_init(drain + k, 1);
    }
    for (int k = 0; k < S; k++) {
      mbar_init(kv_full + k, 1);
      mbar_init(kv_empty + k, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_read, nact);  // one arrival per active softmax warp
    mbar_init(p_ready, nact);
    mbar_init(pv_done, 1);
    mbar_init(o_free, nact);
    mbar_init(part_done, nact);
    mbar_init(merge_go, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const volatile int never = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.map_q);
      prefetch_tmap(&a.map_k);
      prefetch_tmap(&a.map_v);
      bool ok = true;
      int g = 0, loaded = 0;
      DecItem it;
      for (int tl = 0; ok && dec_item(a, tl, it); tl++) {
        const int qb = tl & 1, b = it.bk / a.Hkv, kvh = it.bk - b * a.Hkv;
        if (tl >= 2 && !(ok = mbar_wait(q_empty + qb, ((tl >> 1) - 1) & 1, abort))) break;
        mbar_arrive_expect_tx(q_full + qb, TB);
        tma_load_4d(smem + C::kOffQ + qb * TB, &a.map_q, q_full + qb, 0, 0, it.bk * kTile, 0);
        loaded = tl + 1;
        for (int n = it.n0; n < it.n1; n++, g++) {
          const int st = g % S, use = g / S;
          if (use > 0 && !(ok = mbar_wait(kv_empty + st, (use - 1) & 1, abort))) break;
          mbar_arrive_expect_tx(kv_full + st, 2 * TB);
          tma_load_4d(smem + C::kOffK + st * TB, &a.map_k, kv_full + st, 0, n * kTile, kvh, b);
          tma_load_4d(smem + C::kOffV + st * TB, &a.map_v, kv_full + st, 0, n * kTile, kvh, b);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      // let every copy issued above land before the CTA can exit
      for (int tl = loaded - 2 < 0 ? 0 : loaded - 2; tl < loaded; tl++)
        mbar_wait(q_full + (tl & 1), (tl >> 1) & 1, &never);
      for (int x = g - S < 0 ? 0 : g - S; x < g; x++) mbar_wait(kv_full + x % S, (x / S) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S = Q K^T issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_fp16(128, 128, false, false);
      constexpr uint32_t kStepK = 32 >> 4;
      constexpr uint32_t tstep = (uint32_t)TB >> 4;
      const uint64_t dQ0 = smem_desc(smem_u32(smem + C::kOffQ), 16, C::kSBO, C::kSwz);
      const uint64_t dK0 = smem_desc(smem_u32(smem + C::kOffK), 16, C::kSBO, C::kSwz);
      bool ok = true;
      int g = 0;
      DecItem it;
      for (int tl = 0; ok && dec_item(a, tl, it); tl++) {
        const int qb = tl & 1;
        if (!(ok = mbar_wait(q_full + qb, (tl >> 1) & 1, abort))) break;
        for (int n = it.n0; n < it.n1; n++, g++) {
          const int st = g % S;
          if (!(ok = mbar_wait(kv_full + st, (g / S) & 1, abort))) break;
          // one score buffer: the previous step's scores have been read
          if (g >= 1 && !(ok = mbar_wait(s_read, (g - 1) & 1, abort))) break;
          tc_fence_after();
          mma_ss_chain<D / 16>(tmem + C::kColS, dQ0 + (uint64_t)(qb * tstep), kStepK, dK0 + (uint64_t)(st * tstep),
                               kStepK, idS, 0u);
          mma_commit(s_full);
          if (n + 1 == it.n1) mma_commit(q_empty + qb);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      mma_commit(drain);
      mbar_wait(drain, 0, &never);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ O += P V issuer
    if (lane == 0) {
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      constexpr uint32_t kStepMN = (16 * C::kSpan) >> 4;
      constexpr uint32_t tstep = (uint32_t)TB >> 4;
      const uint64_t dV0 = smem_desc(smem_u32(smem + C::kOffV), 16, C::kSBO, C::kSwz);
      bool ok = true;
      int g = 0;
      DecItem it;
      for (int tl = 0; ok && dec_item(a, tl, it); tl++) {
        for (int n = it.n0; n < it.n1; n++, g++) {
          const int st = g % S;
          if (!(ok = mbar_wait(p_ready, g & 1, abort))) break;
          if (n == it.n0 && tl > 0 && !(ok = mbar_wait(o_free, (tl - 1) & 1, abort))) break;
          tc_fence_after();
          mma_ts_chain<8, false>(tmem + C::kColO, tmem + C::kColP, dV0 + (uint64_t)(st * tstep), kStepMN, idPV,
                                 n > it.n0 ? 1u : 0u);
          mma_commit(pv_done);
          mma_commit(kv_empty + st);  // K was read by S(g), which completed before the softmax began
        }
      }
      if (!ok) record_timeout(a.status, abort);
      mma_commit(drain + 1);
      mbar_wait(drain + 1, 0, &never);
    }
  } else if ((((warp & 3) * 32) % (kTile / a.F)) < a.R) {
    // ------------------------------------------------------------ softmax, one row per thread
    bool ok;
    if (a.F == 4)
      ok = decode_softmax<D, 32>(a, tmem, warp, lane, s_full, s_read, p_ready, pv_done, o_free, part_done, merge_go,
                                 merge_flag, nact, abort);
    else if (a.F == 2)
      ok = decode_softmax<D, 64>(a, tmem, warp, lane, s_full, s_read, p_ready, pv_done, o_free, part_done, merge_go,
                                 merge_flag, nact, abort);
    else
      ok = decode_softmax<D, 128>(a, tmem, warp, lane, s_full, s_read, p_ready, pv_done, o_free, part_done, merge_go,
                                  merge_flag, nact, abort);
    if (!ok) record_timeout(a.status, abort);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    tmem_relinquish();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

int grid_for(long long items, int per_block) {
  long long blocks = (items + per_block - 1) / per_block;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

template <int D>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s, int nsm) {
  using C = DecCfg<D>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_decode<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int items = a.B * a.Hkv * a.nsplit;
  k_decode<D><<<items < nsm ? items : nsm, C::kThreads, C::kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_append(const KvAppendArgs& a, int D, cudaStream_t s) {
  const long long n = (long long)a.B * a.Tn * a.Hkv * (D / 8);
  if (D == 64)
    k_kv_append<64><<<grid_for(n, 256), 256, 0, s>>>(a);
  else
    k_kv_append<32><<<grid_for(n, 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_q(const DecodeArgs& a, cudaStream_t s) {
  const long long n = (long long)a.B * a.Hkv * kTile * (a.D / 8);
  if (a.D == 64)
    k_decode_q<64><<<grid_for(n, 256), 256, 0, s>>>(a);
  else
    k_decode_q<32><<<grid_for(n, 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, int nsm, cudaStream_t s) {
  return a.D == 64 ? launch_decode_t<64>(a, s, nsm) : launch_decode_t<32>(a, s, nsm);
}

}  // namespace ne
