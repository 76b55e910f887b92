// Forward pass of causal GQA attention with RoPE on Q/K (sm_103a).
//
// The NanoEuler GPU engine's FlashAttention is tiled, uses an online softmax
// and never forms the T x T score matrix (socker-news README, "GPU engine" /
// "Kernels and acceleration"; ojeo summary); its causal mask skips the upper
// triangle instead of masking it (openai-hub article, softmax-kernel section).
// The kernels here compute the same result with the GB300 tensor cores:
//
//   k_rope_qk     streaming pre-pass: q, k -> rotated fp16 copies in the
//                 workspace (the backward reads them too).
//   k_attn_fwd4   default precision, persistent: work items of two (query head,
//                 128-row query tile) units of one key/value head that share
//                 the K/V stream; S = Q K^T and O += P V on tcgen05 with the
//                 accumulators in TMEM; one softmax warpgroup per unit keeps the
//                 unit's row maximum and sum in registers (lazy rescale, only
//                 when the maximum grows by more than 2^8); epilogue O / l and
//                 LSE = ln(sum exp).  With F8 the rotated q, k are e4m3.
//   k_attn_fwd    split precision (NE_ATTN_PRECISE_QK), one CTA per (query
//                 tile, batch, key/value head, chunk of query heads): rotates
//                 the bf16 Q and K tiles in shared memory into fp16 hi + lo
//                 parts, S = Qhi Khi^T + Qlo Khi^T + Qhi Klo^T so the logits
//                 carry ~2^-22 relative error when |s| reaches 10^3, P = hi + lo
//                 in two bf16 parts, and a two-part LSE.
// Only the diagonal tile (j == i) is masked; tiles above it are never visited.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace ne {
namespace {

template <int D, bool PRECISE>
struct FwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr uint32_t kSpan = D * 2;  // bytes per row == swizzle span
  static constexpr uint32_t kSwz = D == 64 ? kSw128 : kSw64;
  static constexpr uint32_t kSBO = 8 * kSpan;  // one 8-row swizzle atom
  static constexpr int kMaxHC = D == 64 ? (PRECISE ? 3 : 4) : 8;  // HC*D + 2*128 TMEM columns <= 512
  static constexpr int kStages = D == 64 ? (PRECISE ? 2 : 3) : (PRECISE ? 3 : 4);
  static constexpr int kLoTiles = PRECISE ? 1 : 0;
  // shared memory map (bytes from a 1024-aligned base)
  static constexpr int kOffQ = 0;
  static constexpr int kOffQlo = kOffQ + kMaxHC * kTileBytes;
  static constexpr int kOffK = kOffQlo + kLoTiles * kMaxHC * kTileBytes;
  static constexpr int kOffKlo = kOffK + kStages * kTileBytes;
  static constexpr int kOffV = kOffKlo + kLoTiles * kStages * kTileBytes;
  static constexpr int kOffM = kOffV + kStages * kTileBytes;
  static constexpr int kOffL = kOffM + kMaxHC * kTile * 4;
  static constexpr int kOffBar = kOffL + kMaxHC * kTile * 4;
  static constexpr int kNumBars = 2 + 3 * kStages + 4 + kMaxHC + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemS = 256;  // two 128-column score buffers at 256, 384
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kMaxHC * D <= 256, "tensor memory budget");
};

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, 0, kStatusTimeout);
}

// Rotates `ntiles` consecutive 128-row tiles in place (positions pos0 + row),
// writing fp16 results; with `lo` the fp16 remainders go to the same offsets there.
// Each thread walks 16-byte chunks `nthreads` apart (consecutive threads touch
// consecutive chunks: conflict-free); the shared-memory chunks and the table
// entries of a batch of 8 chunks are all loaded before any is rotated, so the
// table's L2 latency is paid once per batch.
template <int D, int kBatch = 8>
__device__ __forceinline__ void rope_tiles(uint8_t* base, uint8_t* lo, int ntiles, int pos0, const float2* tab,
                                           int tid, int nthreads) {
  constexpr uint32_t kSpan = D * 2;
  constexpr int kCPR = D / 8;  // 16-byte chunks per row
  const int total = ntiles * kTile * kCPR;
  for (int first = tid; first < total; first += kBatch * nthreads) {
    uint4 x[kBatch];
    float4 ca[kBatch], cb[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; u++) {
      const int idx = first + u * nthreads;
      if (idx < total) {
        const int row = (idx / kCPR) % kTile;
        const int pc = idx % kCPR;
        const int lc = (int)((swz(row, pc, kSpan) - row * kSpan) / 16u);  // logical chunk
        x[u] = *reinterpret_cast<const uint4*>(base + (uint32_t)idx * 16u);
        rope_coeffs<D>(tab, pos0 + row, lc, ca[u], cb[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; u++) {
      const int idx = first + u * nthreads;
      if (idx < total) {
        const uint32_t phys = (uint32_t)idx * 16u;
        if (lo) {
          uint4 l;
          *reinterpret_cast<uint4*>(base + phys) = rope_chunk_f16(x[u], ca[u], cb[u], &l);
          *reinterpret_cast<uint4*>(lo + phys) = l;
        } else {
          *reinterpret_cast<uint4*>(base + phys) = rope_chunk_f16(x[u], ca[u], cb[u], nullptr);
        }
      }
    }
  }
}

template <int D, bool PRECISE>
__global__ void __launch_bounds__(256, 1) k_attn_fwd(const __grid_constant__ FwdArgs a) {
  using C = FwdCfg<D, PRECISE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_ready = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* k_ready = kv_full + C::kStages;
  uint64_t* kv_empty = k_ready + C::kStages;
  uint64_t* s_full = kv_empty + C::kStages;  // [2]
  uint64_t* p_ready = s_full + 2;            // [2]
  uint64_t* o_done = p_ready + 2;            // [kMaxHC]
  uint64_t* drain = o_done + C::kMaxHC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  float* sm_m = reinterpret_cast<float*>(smem + C::kOffM);
  float* sm_l = reinterpret_cast<float*>(smem + C::kOffL);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int HC = a.HC;
  const int nchunk = a.G / HC;
  const int per_i = a.B * a.Hkv * nchunk;
  const int i = a.nt - 1 - (int)blockIdx.x / per_i;
  int rem = (int)blockIdx.x % per_i;
  const int hc = rem % nchunk;
  rem /= nchunk;
  const int kvh = rem % a.Hkv;
  const int b = rem / a.Hkv;
  const int h0 = kvh * a.G + hc * HC;
  const int nkv = i + 1;

  if (tid == 0) {
    *abort = 0;
    mbar_init(q_full, 1);
    mbar_init(q_ready, 192);
    for (int s = 0; s < C::kStages; s++) {
      mbar_init(kv_full + s, 1);
      mbar_init(k_ready + s, 64);
      mbar_init(kv_empty + s, 1);
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(s_full + s, 1);
      mbar_init(p_ready + s, 128);
    }
    for (int h = 0; h < C::kMaxHC; h++) mbar_init(o_done + h, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const volatile int never = 0;

  const uint32_t sQ = smem_u32(smem + C::kOffQ);
  const uint32_t sQlo = smem_u32(smem + C::kOffQlo);
  const uint32_t sK = smem_u32(smem + C::kOffK);
  const uint32_t sKlo = smem_u32(smem + C::kOffKlo);
  const uint32_t sV = smem_u32(smem + C::kOffV);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.map_q);
      prefetch_tmap(&a.map_k);
      prefetch_tmap(&a.map_v);
      mbar_arrive_expect_tx(q_full, HC * C::kTileBytes);
      for (int hh = 0; hh < HC; hh++)
        tma_load_4d(smem + C::kOffQ + hh * C::kTileBytes, &a.map_q, q_full, 0, h0 + hh, i * kTile, b);
      int loaded = 0;
      for (int j = 0; j < nkv; j++) {
        const int st = j % C::kStages, use = j / C::kStages;
        if (use > 0 && !mbar_wait(kv_empty + st, (use - 1) & 1, abort)) {
          record_timeout(a.status, abort);
          break;
        }
        mbar_arrive_expect_tx(kv_full + st, 2 * C::kTileBytes);
        tma_load_4d(smem + C::kOffK + st * C::kTileBytes, &a.map_k, kv_full + st, 0, kvh, j * kTile, b);
        tma_load_4d(smem + C::kOffV + st * C::kTileBytes, &a.map_v, kv_full + st, 0, kvh, j * kTile, b);
        loaded = j + 1;
      }
      // Let every copy issued above land before the CTA can exit.
      mbar_wait(q_full, 0, &never);
      for (int j = loaded - C::kStages < 0 ? 0 : loaded - C::kStages; j < loaded; j++)
        mbar_wait(kv_full + j % C::kStages, (j / C::kStages) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_fp16(128, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      constexpr uint32_t kStepK = 32 >> 4, kStepMN = (16 * C::kSpan) >> 4, kTileStep = C::kTileBytes >> 4;
      // shared-memory descriptors, computed once (tile k adds k * bytes / 16 to the start address)
      const uint64_t dQ0 = smem_desc(sQ, 16, C::kSBO, C::kSwz), dQlo0 = smem_desc(sQlo, 16, C::kSBO, C::kSwz);
      const uint64_t dK0 = smem_desc(sK, 16, C::kSBO, C::kSwz), dKlo0 = smem_desc(sKlo, 16, C::kSBO, C::kSwz);
      const uint64_t dV0 = smem_desc(sV, 16, C::kSBO, C::kSwz);
      bool ok = mbar_wait(q_ready, 0, abort);
      tc_fence_after();
      auto issue_pv = [&](int m) -> bool {
        const int hh = m % HC, jm = m / HC, st = jm % C::kStages, sb = m & 1;
        if (!mbar_wait(p_ready + sb, (m >> 1) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t sP = tmem + C::kTmemS + sb * 128;
        const uint64_t dV = dV0 + (uint64_t)(st * kTileStep);
        mma_ts_chain<8>(tmem + hh * D, sP, dV, kStepMN, idPV, jm > 0 ? 1u : 0u);
        if (PRECISE)  // + P_lo V: the bf16 remainder of P sits in the buffer's upper 64 columns
          mma_ts_chain<8>(tmem + hh * D, sP + 64, dV, kStepMN, idPV, 1u);
        mma_commit(o_done + hh);
        if (hh == HC - 1) mma_commit(kv_empty + st);
        return true;
      };
      int n = 0;
      for (int j = 0; ok && j < nkv; j++) {
        const int st = j % C::kStages;
        if (!mbar_wait(k_ready + st, (j / C::kStages) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int hh = 0; hh < HC; hh++, n++) {
          const int sb = n & 1;
          // S = Qhi Khi^T (+ Qlo Khi^T + Qhi Klo^T)
          const uint64_t qd = dQ0 + (uint64_t)(hh * kTileStep), kd = dK0 + (uint64_t)(st * kTileStep);
          mma_ss_chain<D / 16>(tmem + C::kTmemS + sb * 128, qd, kStepK, kd, kStepK, idS, 0u);
          if (PRECISE) {
            mma_ss_chain<D / 16>(tmem + C::kTmemS + sb * 128, dQlo0 + (uint64_t)(hh * kTileStep), kStepK, kd,
                                 kStepK, idS, 1u);
            mma_ss_chain<D / 16>(tmem + C::kTmemS + sb * 128, qd, kStepK, dKlo0 + (uint64_t)(st * kTileStep),
                                 kStepK, idS, 1u);
          }
          mma_commit(s_full + sb);
          if (n >= 1 && !issue_pv(n - 1)) {
            ok = false;
            break;
          }
        }
      }
      if (ok && n >= 1) ok = issue_pv(n - 1);
      if (!ok) record_timeout(a.status, abort);
      // All issued MMAs must finish before the tensor memory is released.
      mma_commit(drain);
      mbar_wait(drain, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ RoPE on Q (warps 2-7 together)
    const bool ok_q = mbar_wait(q_full, 0, abort);
    if (ok_q) {
      rope_tiles<D>(smem + C::kOffQ, PRECISE ? smem + C::kOffQlo : nullptr, HC, i * kTile, a.rope, tid - 64, 192);
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    } else {
      record_timeout(a.status, abort);
    }
  }
  if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ RoPE on K
    const int rt = tid - 64;
    bool ok = !*abort;
    for (int j = 0; ok && j < nkv; j++) {
      const int st = j % C::kStages;
      if (!mbar_wait(kv_full + st, (j / C::kStages) & 1, abort)) {
        ok = false;
        break;
      }
      rope_tiles<D>(smem + C::kOffK + st * C::kTileBytes, PRECISE ? smem + C::kOffKlo + st * C::kTileBytes : nullptr,
                    1, j * kTile, a.rope, rt, 64);
      fence_proxy_async_smem();
      mbar_arrive(k_ready + st);
    }
    if (!ok) record_timeout(a.status, abort);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int r = tid - 128;               // query row within the tile
    const uint32_t lane_base = (uint32_t)(warp - 4) * 32u;
    const uint32_t trow = tmem + (lane_base << 16);
    const float sl2 = a.scale_log2;
    bool ok = true;
    int n = 0;
    for (int j = 0; ok && j < nkv; j++) {
      const bool diag = (j == i);
      for (int hh = 0; hh < HC; hh++, n++) {
        const int sb = n & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(s_full + sb, (n >> 1) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        float s[kTile];
        {
          // all four loads in flight before the single wait
          uint32_t u0[32], u1[32], u2[32], u3[32];
          const uint32_t sc = trow + C::kTmemS + sb * 128;
          tmem_ld32(sc, u0);
          tmem_ld32(sc + 32, u1);
          tmem_ld32(sc + 64, u2);
          tmem_ld32(sc + 96, u3);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e++) {
            s[e] = __uint_as_float(u0[e]);
            s[32 + e] = __uint_as_float(u1[e]);
            s[64 + e] = __uint_as_float(u2[e]);
            s[96 + e] = __uint_as_float(u3[e]);
          }
        }
        if (diag) {
#pragma unroll
          for (int c = 0; c < kTile; c++)
            if (c > r) s[c] = -INFINITY;
        }
        // The row state keeps the raw score r_use that defines the reference
        // m_use = fp32(r_use * scale_log2); the epilogue needs it for the
        // double-float LSE.  Eight partial maxima keep the dependency chain short.
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; e++) mx8[e] = s[e];
#pragma unroll
        for (int c = 8; c < kTile; c++) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
        const float mxr = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        // Every reference value is the correctly rounded product r * scale_log2
        // (no FMA contraction), so alpha, P and the LSE all use the same m.
        const float r_old = j == 0 ? -INFINITY : sm_m[hh * kTile + r];
        const float m_old = __fmul_rn(r_old, sl2);
        float l_old = j == 0 ? 0.f : sm_l[hh * kTile + r];
        float r_use = r_old, alpha = 1.f;
        if (j == 0) {
          r_use = mxr;
        } else {
          // The previous O_h += P V must be complete before O_h is read or rescaled.
          ok = __all_sync(0xffffffffu, mbar_wait(o_done + hh, (j - 1) & 1, abort));
          if (!ok) break;
          tc_fence_after();
          const float r_new = fmaxf(r_old, mxr);
          const float m_new = __fmul_rn(r_new, sl2);
          if (__any_sync(0xffffffffu, m_new > m_old + 8.0f)) {
            r_use = r_new;
            alpha = ex2(m_old - m_new);
#pragma unroll
            for (int c = 0; c < D / 16; c++) {
              uint32_t u[16];
              tmem_ld16(trow + hh * D + c * 16, u);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; e++) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
              tmem_st16(trow + hh * D + c * 16, u);
            }
          }
        }
        // Default: P is rounded to bf16 and the row sum adds the rounded values,
        // so O is the exact average of V rows under the weights the MMA uses.
        // PRECISE: P = hi + lo (two bf16 parts, ~2^-17 relative) and the row sum
        // adds the fp32 values, so O and LSE follow the exact softmax.
        const float m_use = __fmul_rn(r_use, sl2);
        float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kTile / 32; c++) {
          uint32_t pk[16], pl[16];
#pragma unroll
          for (int e = 0; e < 16; e++) {
            const float p0 = ex2(fmaf(s[c * 32 + 2 * e], sl2, -m_use));
            const float p1 = ex2(fmaf(s[c * 32 + 2 * e + 1], sl2, -m_use));
            pk[e] = pack_bf16(p0, p1);
            if (PRECISE) {
              pl[e] = pack_bf16(p0 - bf_lo(pk[e]), p1 - bf_hi(pk[e]));
              sum8[e & 7] += p0 + p1;
            } else {
              sum8[e & 7] += bf_lo(pk[e]) + bf_hi(pk[e]);
            }
          }
          tmem_st16(trow + C::kTmemS + sb * 128 + c * 16, pk);
          if (PRECISE) tmem_st16(trow + C::kTmemS + sb * 128 + 64 + c * 16, pl);
        }
        const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_ready + sb);
        sm_m[hh * kTile + r] = r_use;
        sm_l[hh * kTile + r] = l_old * alpha + sum;
      }
    }
    if (ok) {
      const int t = i * kTile + r;
      for (int hh = 0; hh < HC; hh++) {
        ok = __all_sync(0xffffffffu, mbar_wait(o_done + hh, (nkv - 1) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        const float l = sm_l[hh * kTile + r];
        const float inv = 1.f / l;
        const int h = h0 + hh;
        const size_t orow = (((size_t)b * a.T + t) * a.Hq + h) * D;
#pragma unroll
        for (int c = 0; c < D / 16; c++) {
          uint32_t u[16];
          tmem_ld16(trow + hh * D + c * 16, u);
          tmem_wait_ld();
          if (t < a.T) {
            if (a.o_fp32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.o) + orow + c * 16);
#pragma unroll
              for (int e = 0; e < 4; e++)
                dst[e] = make_float4(__uint_as_float(u[4 * e]) * inv, __uint_as_float(u[4 * e + 1]) * inv,
                                     __uint_as_float(u[4 * e + 2]) * inv, __uint_as_float(u[4 * e + 3]) * inv);
            } else {
              uint32_t w[8];
#pragma unroll
              for (int e = 0; e < 8; e++)
                w[e] = pack_bf16(__uint_as_float(u[2 * e]) * inv, __uint_as_float(u[2 * e + 1]) * inv);
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.o) + orow + c * 16);
              dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
              dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
        if (t < a.T) {
          const size_t li = ((size_t)b * a.Hq + h) * a.T + t;
          const float r_use = sm_m[hh * kTile + r];
          const float m_use = __fmul_rn(r_use, sl2);
          if (PRECISE) {
            // LSE in log2 units = r_use * scale_log2 + log2(l), carried as hi + lo
            // (exact product remainder by fma), then converted to natural log with
            // a two-part ln 2.  The backward rebuilds P from hi + lo.
            const float m_lo = fmaf(r_use, sl2, -m_use) + r_use * a.scale_log2_lo;
            float h2, l2;
            two_sum(m_use, __log2f(l), h2, l2);
            l2 += m_lo;
            const float hi = __fmul_rn(h2, kLn2Hi);
            const float lo = fmaf(h2, kLn2Hi, -hi) + h2 * kLn2Lo + l2 * kLn2Hi;
            const float H = __fadd_rn(hi, lo);
            a.lse[li] = H;
            a.lse_lo[li] = __fsub_rn(lo, __fsub_rn(H, hi));
          } else {
            a.lse[li] = (m_use + __log2f(l)) * 0.69314718055994531f;
          }
        }
      }
    }
    if (!ok) record_timeout(a.status, abort);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    tmem_relinquish();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ====================================================================== RoPE pre-pass
// q [B,T,Hq,D] and k [B,T,Hkv,D] (bf16) -> rotated fp16 copies of the same
// layout.  Every head at position t turns by the same angles, so a thread takes
// one 16-byte chunk c (four pairs) of one position (b, t) for a group of four
// heads (of the Hq query heads followed by the Hkv key heads): the chunk's
// (cos, sin) entries are read once for the four, and the four loads are in
// flight together.  Streaming work: every byte is read and written once.
template <int D>
__global__ void __launch_bounds__(256) k_rope_qk(const RopeArgs a) {
  constexpr int kCPR = D / 8;  // 16-byte chunks per row
  constexpr int kU = 4;        // heads per thread
  const int H = a.Hq + a.Hkv;
  const uint32_t ngr = (uint32_t)(H + kU - 1) / kU;
  const uint32_t n = (uint32_t)a.B * a.T * ngr * kCPR;
  const bool half = a.rope_half != 0;
  for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < n; it += gridDim.x * blockDim.x) {
    const int c = (int)(it % kCPR);
    const uint32_t rest = it / kCPR;  // (b * T + t) * ngr + head group
    const uint32_t bt = fdiv(rest, a.div_hg);
    const int h0 = (int)(rest - bt * ngr) * kU;
    const uint32_t t = bt - fdiv(bt, a.div_t) * a.T;
    float4 c0, c1;
    rope_coeffs<D>(a.rope, (int)t, c, c0, c1);
    {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; u++) {
        const int h = h0 + u;
        if (h < H) {
          const bool isq = h < a.Hq;
          const __nv_bfloat16* row = isq ? a.q + ((size_t)bt * a.Hq + h) * D : a.k + ((size_t)bt * a.Hkv + h - a.Hq) * D;
          v[u] = load_rope_chunk<D>(row, c, half);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; u++) {
        const int h = h0 + u;
        if (h < H) {
          const bool isq = h < a.Hq;
          __half* dst = isq ? a.qr + ((size_t)bt * a.Hq + h) * D : a.kr + ((size_t)bt * a.Hkv + h - a.Hq) * D;
          reinterpret_cast<uint4*>(dst)[c] = rope_chunk_f16(v[u], c0, c1, nullptr);
        }
      }
    }
  }
}

// ====================================================================== FP8 pre-passes (D = 64)
// The FP8 forward takes the rotated q and k as e4m3 with one scale per head:
// value = e4m3 code * max_h / 448, max_h the largest |rotated value| of head h
// over all batches and positions.  Pass 1 finds max_h, pass 2 rotates again and
// rounds (round to nearest even, saturating at 448).
constexpr int kMaxHeadsF8 = 256;  // Hq + Hkv at most (shared-memory maxima of pass 1)

__global__ void __launch_bounds__(256) k_rope_amax(const RopeArgs a) {
  constexpr int D = 64, kCPR = D / 8;
  __shared__ unsigned smax[kMaxHeadsF8];
  const int nh = a.Hq + a.Hkv;
  for (int i = threadIdx.x; i < nh; i += blockDim.x) smax[i] = 0u;
  __syncthreads();
  const uint32_t nq = (uint32_t)a.B * a.T * a.Hq * kCPR;
  const uint32_t n = nq + (uint32_t)a.B * a.T * a.Hkv * kCPR;
  for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < n; it += gridDim.x * blockDim.x) {
    const bool isq = it < nq;
    const uint32_t x = isq ? it : it - nq;
    const uint32_t row = x / kCPR;  // (b, t, h)
    const uint32_t bt = fdiv(row, isq ? a.div_hq : a.div_hkv);
    const uint32_t h = row - bt * (isq ? a.Hq : a.Hkv);
    const uint32_t t = bt - fdiv(bt, a.div_t) * a.T;
    const uint4 v = load_rope_chunk<D>((isq ? a.q : a.k) + (size_t)row * D, (int)(x % kCPR), a.rope_half != 0);
    float4 c0, c1;
    rope_coeffs<D>(a.rope, (int)t, (int)(x % kCPR), c0, c1);
    float y[8];
    rope_chunk_f32(v, c0, c1, y);
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < 8; e++) m = fmaxf(m, fabsf(y[e]));
    atomicMax(&smax[isq ? h : a.Hq + h], __float_as_uint(m));  // non-negative floats order as integers
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nh; i += blockDim.x)
    if (smax[i]) atomicMax(reinterpret_cast<unsigned*>(a.amax) + i, smax[i]);
}

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(256) k_rope_q8(const RopeArgs a) {
  constexpr int D = 64, kCPR = D / 8;
  const uint32_t nq = (uint32_t)a.B * a.T * a.Hq * kCPR;
  const uint32_t n = nq + (uint32_t)a.B * a.T * a.Hkv * kCPR;
  for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < n; it += gridDim.x * blockDim.x) {
    const bool isq = it < nq;
    const uint32_t x = isq ? it : it - nq;
    const uint32_t row = x / kCPR;
    const uint32_t bt = fdiv(row, isq ? a.div_hq : a.div_hkv);
    const uint32_t h = row - bt * (isq ? a.Hq : a.Hkv);
    const uint32_t t = bt - fdiv(bt, a.div_t) * a.T;
    const float mx = __ldg(a.amax + (isq ? h : a.Hq + h));
    const float inv = mx > 0.f ? 448.f / mx : 1.f;
    const uint4 v = load_rope_chunk<D>((isq ? a.q : a.k) + (size_t)row * D, (int)(x % kCPR), a.rope_half != 0);
    float4 c0, c1;
    rope_coeffs<D>(a.rope, (int)t, (int)(x % kCPR), c0, c1);
    float y[8];
    rope_chunk_f32(v, c0, c1, y);
    const uint32_t w0 = (uint32_t)e4m3x2(y[0] * inv, y[1] * inv) | ((uint32_t)e4m3x2(y[2] * inv, y[3] * inv) << 16);
    const uint32_t w1 = (uint32_t)e4m3x2(y[4] * inv, y[5] * inv) | ((uint32_t)e4m3x2(y[6] * inv, y[7] * inv) << 16);
    reinterpret_cast<uint2*>(isq ? a.q8 : a.k8)[x] = make_uint2(w0, w1);
  }
}

// ====================================================================== persistent forward, two query tiles per item
// Default-precision forward over the rotated fp16 (or, with F8, e4m3) q, k that
// the RoPE pre-pass (or the projection's epilogue) left in the workspace.  A work
// item is a pair of units of one (batch, key/value head); a unit is one query
// head's 128-row query tile.  The two units share the item's K/V stream (key
// tiles 0 .. max(i0, i1)), and each softmax warpgroup owns one unit's rows for
// the whole item: its row maximum and row sum stay in registers, so the two
// warpgroups never wait for each other.  Unit u has its own TMEM score buffer
// S_u, P buffer P_u and accumulator O_u (2 x (128 + 64 + 64) = 512 columns), so
// S_u of the next key tile goes out as soon as the scores of this one are in
// the warpgroup's registers (all 128 per row, one TMEM round trip, before the
// row maximum).  O_u += P_u V goes out in two halves of 64 keys, the first while the
// warpgroup still exponentiates the second, so that P_u of the next key tile
// rarely waits for it.
// Items come from a host-built table (fwd_pair_schedule in api.cu): pairs of
// heads of one group at the same query tile; with an odd group size the
// group's last head pairs adjacent query tiles (i, i - 1) of itself.
// Warps: 0 TMA producer (a ring of four Q slots, a K/V ring), 1 S = Q K^T
// issuer for both units, 2 and 3 O += P V issuers for units 0 and 1, 4-7 and
// 8-11 the softmax warpgroups of units 0 and 1 (one thread per query row).
// Each softmax warp stores its 32 rows of O itself (TMA boxes of 32 rows).

// Writes row r (0..31) of a 32-row slice of O (D values, fp32 when ES == 4, else
// bf16) into a staging area of column boxes of 32 rows: `span` = min(D * ES, 128)
// bytes per row, box after box, each with the TMA / UMMA swizzle of that span.
template <int D, int ES>
__device__ __forceinline__ void stage_rows32(const float (&x)[D], uint8_t* stg, int r) {
  constexpr int kSpan = D * ES < 128 ? D * ES : 128;
  constexpr int kCols = kSpan / ES;
#pragma unroll
  for (int c0 = 0, bx = 0; c0 < D; c0 += kCols, bx++) {
#pragma unroll
    for (int ch = 0; ch < kSpan / 16; ch++) {
      uint4 w;
      if constexpr (ES == 4) {
        const int i = c0 + ch * 4;
        w = make_uint4(__float_as_uint(x[i]), __float_as_uint(x[i + 1]), __float_as_uint(x[i + 2]),
                       __float_as_uint(x[i + 3]));
      } else {
        const int i = c0 + ch * 8;
        w = make_uint4(pack_bf16(x[i], x[i + 1]), pack_bf16(x[i + 2], x[i + 3]), pack_bf16(x[i + 4], x[i + 5]),
                       pack_bf16(x[i + 6], x[i + 7]));
      }
      *reinterpret_cast<uint4*>(stg + bx * 32 * kSpan + swz(r, ch, kSpan)) = w;
    }
  }
}

template <int D, bool F8 = false>
struct Fwd4Cfg {
  static constexpr int kTileBytes = kTile * D * 2;  // V tile (bf16)
  static constexpr uint32_t kSpan = D * 2;
  static constexpr uint32_t kSwz = D == 64 ? kSw128 : kSw64;
  static constexpr uint32_t kSBO = 8 * kSpan;
  static constexpr int kQKTileBytes = kTile * D * (F8 ? 1 : 2);
  static constexpr uint32_t kQKSpan = D * (F8 ? 1 : 2);
  static constexpr uint32_t kQKSwz = kQKSpan == 128 ? kSw128 : (kQKSpan == 64 ? kSw64 : kSw32);
  static constexpr uint32_t kQKSBO = 8 * kQKSpan;
  static constexpr int kQSlots = 4;                      // two items' worth of query tiles
  static constexpr int kStages = (D == 64 && !F8) ? 3 : 4;  // K/V ring
  static constexpr uint32_t kColO = 0, kColS = 128, kColP = 384;  // unit u: O at 64u, S at 128 + 128u, P at 384 + 64u
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 384;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQSlots * kQKTileBytes;
  static constexpr int kOffV = kOffK + kStages * kQKTileBytes;
  static constexpr int kOstBytes = kTile * D * 4;  // O staging per unit (fp32 rows at most)
  static constexpr int kOffOst = kOffV + kStages * kTileBytes;
  static constexpr int kOffBar = kOffOst + 2 * kOstBytes;
  static constexpr int kNumBars = 2 * kQSlots + 2 * kStages + 14 + 3;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16;  // the dynamic area is 1024-aligned
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Fwd4Item {
  int b, nu;       // batch; number of units (1 or 2)
  int h0, h1, i0, i1;  // query head and query tile of each unit; i0 >= i1
  __device__ __forceinline__ int h(int u) const { return u ? h1 : h0; }
  __device__ __forceinline__ int i(int u) const { return u ? i1 : i0; }
};

// Item tl of this CTA: entries (b, h0 | (h1 + 1) << 16, i0, i1), b = -1 past the end.
__device__ __forceinline__ bool fwd4_item(const FwdArgs& a, int tl, Fwd4Item& it) {
  if (tl >= a.sched_k) return false;
  const int4 w = __ldg(reinterpret_cast<const int4*>(a.sched) + (size_t)blockIdx.x * a.sched_k + tl);
  if (w.x < 0) return false;
  it.b = w.x;
  it.h0 = w.y & 0xffff;
  it.h1 = (int)((uint32_t)w.y >> 16) - 1;
  it.nu = it.h1 >= 0 ? 2 : 1;
  it.i0 = w.z;
  it.i1 = it.nu == 2 ? w.w : -1;
  return true;
}

template <int D, bool F8>
__global__ void __launch_bounds__(384, 1) k_attn_fwd4(const __grid_constant__ FwdArgs a) {
  using C = Fwd4Cfg<D, F8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  // the swizzled tiles need a 1024-byte aligned base; the declaration asks for it
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kStatusTimeout);
    return;
  }
  constexpr int S = C::kStages;
  constexpr int TB = C::kTileBytes;
  constexpr int TQK = C::kQKTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;                  // [4] Q slots
  uint64_t* q_empty = q_full + 4;           // [4] the slot's last S has completed
  uint64_t* kv_full = q_empty + 4;          // [S]
  uint64_t* kv_empty = kv_full + S;         // [S] both O += P V issuers are done with the stage
  uint64_t* s_full = kv_empty + S;          // [2] per unit
  uint64_t* s_read = s_full + 2;            // [2] the unit's warpgroup holds its scores in registers
  uint64_t* p_ready = s_read + 2;           // [2][2] per unit and key half: the half of P is in TMEM
  uint64_t* pv_done = p_ready + 4;          // [2][2] per unit and key half: that half of O += P V has completed
  uint64_t* o_free = pv_done + 4;           // [2] the unit's O has been read out
  uint64_t* drain = o_free + 2;             // [3] one per issuing thread
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + C::kNumBars) + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    *abort = 0;
    for (int k = 0; k < C::kQSlots; k++) {
      mbar_init(q_full + k, 1);
      mbar_init(q_empty + k, 1);
    }
    for (int k = 0; k < S; k++) {
      mbar_init(kv_full + k, 1);
      mbar_init(kv_empty + k, 2);
    }
    for (int u = 0; u < 2; u++) {
      mbar_init(s_full + u, 1);
      mbar_init(s_read + u, 4);  // one arrival per warp of the warpgroup
      mbar_init(p_ready + 2 * u, 4);
      mbar_init(p_ready + 2 * u + 1, 4);
      mbar_init(pv_done + 2 * u, 1);
      mbar_init(pv_done + 2 * u + 1, 1);
      mbar_init(o_free + u, 4);
    }
    for (int k = 0; k < 3; k++) mbar_init(drain + k, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const volatile int never = 0;
  // registers per thread: 64 for the producer and issuer warps (warps 0-3) and
  // 216 for the softmax warpgroups: 128 x 64 + 256 x 216 = 63,488 of the
  // 384 x 168 = 64,512 the block is launched with
  if (warp < 4) regs_dec<64>();  // warpgroup 0: TMA producer and MMA issuers
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.map_q);
      prefetch_tmap(&a.map_k);
      prefetch_tmap(&a.map_v);
      bool ok = true;
      int g = 0, c = 0;  // K/V stages and Q slots handed out so far
      Fwd4Item it, nx;
      bool have = fwd4_item(a, 0, it);
      for (int tl = 0; ok && have; tl++, it = nx) {
        have = fwd4_item(a, tl + 1, nx);  // the next entry loads while this item runs
        const int kvh = it.h0 / a.G;
        for (int u = 0; u < it.nu; u++, c++) {
          const int sl = c & 3, use = c >> 2;
          if (use > 0 && !(ok = mbar_wait(q_empty + sl, (use - 1) & 1, abort))) break;
          mbar_arrive_expect_tx(q_full + sl, TQK);
          tma_load_4d(smem + C::kOffQ + sl * TQK, &a.map_q, q_full + sl, 0, it.h(u), it.i(u) * kTile, it.b);
        }
        for (int j = 0; ok && j <= it.i0; j++, g++) {
          const int st = g % S, use = g / S;
          if (use > 0 && !(ok = mbar_wait(kv_empty + st, (use - 1) & 1, abort))) break;
          mbar_arrive_expect_tx(kv_full + st, TQK + TB);
          tma_load_4d(smem + C::kOffK + st * TQK, &a.map_k, kv_full + st, 0, kvh, j * kTile, it.b);
          tma_load_4d(smem + C::kOffV + st * TB, &a.map_v, kv_full + st, 0, kvh, j * kTile, it.b);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      // let every copy issued above land before the CTA can exit
      for (int x = c - 4 < 0 ? 0 : c - 4; x < c; x++) mbar_wait(q_full + (x & 3), (x >> 2) & 1, &never);
      for (int x = g - S < 0 ? 0 : g - S; x < g; x++) mbar_wait(kv_full + x % S, (x / S) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S = Q K^T issuer (both units)
    if (lane == 0) {
      constexpr uint32_t idS = F8 ? idesc_e4m3(128, 128, false, false) : idesc_fp16(128, 128, false, false);
      constexpr uint32_t kStepK = 32 >> 4;  // 16 fp16 or 32 e4m3 values of K
      constexpr uint32_t tstep = (uint32_t)TQK >> 4;
      const uint64_t dQ0 = smem_desc(smem_u32(smem + C::kOffQ), 16, C::kQKSBO, C::kQKSwz);
      const uint64_t dK0 = smem_desc(smem_u32(smem + C::kOffK), 16, C::kQKSBO, C::kQKSwz);
      bool ok = true;
      int g = 0, c = 0, n[2] = {0, 0};  // K/V stages, Q slots, S issued per unit
      Fwd4Item it, nx;
      bool have = fwd4_item(a, 0, it);
      for (int tl = 0; ok && have; tl++, it = nx) {
        have = fwd4_item(a, tl + 1, nx);
        for (int j = 0; ok && j <= it.i0; j++, g++) {
          const int st = g % S;
          if (!(ok = mbar_wait(kv_full + st, (g / S) & 1, abort))) break;
          for (int u = 0; u < it.nu; u++) {
            if (j > it.i(u)) continue;
            const int q = c + u, sl = q & 3;
            if (j == 0 && !(ok = mbar_wait(q_full + sl, (q >> 2) & 1, abort))) break;
            // the unit's previous scores are in its warpgroup's registers
            if (n[u] > 0 && !(ok = mbar_wait(s_read + u, (n[u] - 1) & 1, abort))) break;
            tc_fence_after();
            if constexpr (F8)
              mma_ss_chain2_f8(tmem + C::kColS + 128u * u, dQ0 + (uint64_t)(sl * tstep), kStepK,
                               dK0 + (uint64_t)(st * tstep), kStepK, idS, 0u);
            else
              mma_ss_chain<D / 16>(tmem + C::kColS + 128u * u, dQ0 + (uint64_t)(sl * tstep), kStepK,
                                   dK0 + (uint64_t)(st * tstep), kStepK, idS, 0u);
            mma_commit(s_full + u);
            if (j == it.i(u)) mma_commit(q_empty + sl);
            n[u]++;
          }
        }
        c += it.nu;
      }
      if (!ok) record_timeout(a.status, abort);
      mma_commit(drain);
      mbar_wait(drain, 0, &never);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ O_u += P_u V issuers
    if (lane == 0) {
      const int u = warp - 2;
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      constexpr uint32_t kStepMN = (16 * C::kSpan) >> 4;
      constexpr uint32_t tstep = (uint32_t)TB >> 4;
      const uint64_t dV0 = smem_desc(smem_u32(smem + C::kOffV), 16, C::kSBO, C::kSwz);
      bool ok = true;
      int g = 0, n = 0, e = 0;  // K/V stages, this unit's steps, this unit's items
      Fwd4Item it, nx;
      bool have = fwd4_item(a, 0, it);
      for (int tl = 0; ok && have; tl++, it = nx) {
        have = fwd4_item(a, tl + 1, nx);
        const bool act = u < it.nu;
        for (int j = 0; ok && j <= it.i0; j++, g++) {
          const int st = g % S;
          if (act && j <= it.i(u)) {
            // keys 0..63 of P go out while the warpgroup still computes keys 64..127
            if (!(ok = mbar_wait(p_ready + 2 * u, n & 1, abort))) break;
            if (j == 0 && e > 0 && !(ok = mbar_wait(o_free + u, (e - 1) & 1, abort))) break;
            tc_fence_after();
            const uint64_t dv = dV0 + (uint64_t)(st * tstep);
            mma_ts_chain<4, false>(tmem + C::kColO + 64u * u, tmem + C::kColP + 64u * u, dv, kStepMN, idPV,
                                   j > 0 ? 1u : 0u);
            mma_commit(pv_done + 2 * u);
            if (!(ok = mbar_wait(p_ready + 2 * u + 1, n & 1, abort))) break;
            tc_fence_after();
            mma_ts_chain<4, false>(tmem + C::kColO + 64u * u, tmem + C::kColP + 64u * u + 32u,
                                   dv + (uint64_t)(4 * kStepMN), kStepMN, idPV, 1u);
            mma_commit(pv_done + 2 * u + 1);
            mma_commit(kv_empty + st);  // V by this PV; K by this unit's S, complete before its P existed
            n++;
          } else {
            mbar_arrive(kv_empty + st);  // this unit does not use the stage
          }
        }
        if (act) e++;
      }
      if (!ok) record_timeout(a.status, abort);
      mma_commit(drain + 1 + u);
      mbar_wait(drain + 1 + u, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup of unit u
    regs_inc<216>();
    const int u = (warp - 4) >> 2;  // 0: warps 4-7, 1: warps 8-11
    const int q4 = warp & 3;        // TMEM lane quarter
    const int r = q4 * 32 + lane;   // query row within the tile
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t sbuf = trow + C::kColS + 128u * u;
    const uint32_t pbuf = trow + C::kColP + 64u * u;
    const uint32_t obuf = trow + C::kColO + 64u * u;
    // this warp's staging area for its 32 rows of O (boxes of 32 rows x 128 bytes)
    uint8_t* ost = smem + C::kOffOst + u * C::kOstBytes + q4 * (C::kOstBytes / 4);
    bool ok = true;
    int n = 0, ne = 0;  // this unit's steps and epilogues so far
    Fwd4Item it, nx;
    bool have = fwd4_item(a, 0, it);
    for (int tl = 0; ok && have; tl++, it = nx) {
      have = fwd4_item(a, tl + 1, nx);
      if (u >= it.nu) continue;
      const int iu = it.i(u), hu = it.h(u);
      const int t = iu * kTile + r;
      float sl2 = a.scale_log2;
      if constexpr (F8) {  // scores are in e4m3 code units: fold in the two heads' scales
        const float sq = __ldg(a.qk_amax + hu), sk = __ldg(a.qk_amax + a.Hq + hu / a.G);
        sl2 = a.scale_log2 * ((sq > 0.f ? sq : 448.f) * (1.f / 448.f)) * ((sk > 0.f ? sk : 448.f) * (1.f / 448.f));
      }
      float r_run = 0.f, l_run = 0.f;  // running maximum (raw logit units) and sum of the row
      for (int j = 0; j <= iu; j++, n++) {
        const bool diag = (j == iu);
        ok = __all_sync(0xffffffffu, mbar_wait(s_full + u, n & 1, abort));
        if (!ok) break;
        tc_fence_after();
        // pass 1: all 128 scores of the row into registers (one TMEM round trip; the
        // unit's next S may then overwrite the score buffer), the row maximum over
        // them (masked past the diagonal)
        uint32_t sc[128];
#pragma unroll
        for (int c = 0; c < 4; c++) tmem_ld32(sbuf + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sc + 32 * c));
        tmem_wait_ld();
        tc_fence_before();
        warp_arrive(s_read + u);
        if (diag) {
#pragma unroll
          for (int e = 0; e < 128; e++)
            if (e > r) sc[e] = 0xff800000u;  // -inf: key after the query (exp2(-inf) = 0)
        }
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; e++) mx8[e] = -INFINITY;
#pragma unroll
        for (int e = 0; e < 128; e += 2)
          mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], __uint_as_float(sc[e]), __uint_as_float(sc[e + 1]));
        const float mxr = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        float r_use = mxr, alpha = 1.f;
        if (j > 0) {
          r_use = r_run;
          const float m_old = __fmul_rn(r_run, sl2);
          const float r_new = fmaxf(r_run, mxr);
          const float m_new = __fmul_rn(r_new, sl2);
          // lazy rescale: only when some row's maximum grew by more than 2^8; O must
          // then hold every earlier P V (the latest is this unit's previous step)
          if (__any_sync(0xffffffffu, m_new > m_old + 8.0f)) {
            ok = __all_sync(0xffffffffu, mbar_wait(pv_done + 2 * u + 1, (n - 1) & 1, abort));
            if (!ok) break;
            tc_fence_after();
            r_use = r_new;
            alpha = ex2(m_old - m_new);
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < D / 32; c++) {
              tmem_ld32(obuf + c * 32, w);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; e++) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
              tmem_st32(obuf + c * 32, w);
            }
            tmem_wait_st();
            tc_fence_before();
          }
        }
        r_run = r_use;
        const float m_use = __fmul_rn(r_use, sl2);
        // keys 0..63 of the P buffer are free once the first half of the unit's previous
        // O += P V has completed (keys 64..127: its second half, waited for below)
        if (n > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(pv_done + 2 * u, (n - 1) & 1, abort));
          if (!ok) break;
        }
        tc_fence_after();
        // pass 2: P = exp2(s * scale_log2 - m) as bf16 into the unit's P buffer, 16 keys
        // at a time from pass 1's registers.
        // (the row sum adds the fp32 values of P; the MMA multiplies their bf16 roundings)
        uint64_t sum4[4] = {0ull, 0ull, 0ull, 0ull};
        const uint64_t sl2x2 = f2(sl2, sl2), negm = f2(-m_use, -m_use);
#pragma unroll
        for (int c = 0; c < 8; c++) {
          if (c == 4) {
            // keys 0..63 of P are stored: the first half of O += P V may start; keys
            // 64..127 wait for the second half of the previous one
            tmem_wait_st();
            tc_fence_before();
            warp_arrive(p_ready + 2 * u);
            if (n > 0 && !__all_sync(0xffffffffu, mbar_wait(pv_done + 2 * u + 1, (n - 1) & 1, abort))) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; e++) {
            const int k = 16 * c + 2 * e;
            float x0, x1;
            f2_split(f2_fma(f2(__uint_as_float(sc[k]), __uint_as_float(sc[k + 1])), sl2x2, negm), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            pk[e] = pack_bf16(p0, p1);
            sum4[e & 3] = f2_add(sum4[e & 3], f2(p0, p1));
          }
          tmem_st8(pbuf + c * 8, pk);
        }
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(p_ready + 2 * u + 1);
        {
          float s0, s1, s2, s3, s4, s5, s6, s7;
          f2_split(sum4[0], s0, s1);
          f2_split(sum4[1], s2, s3);
          f2_split(sum4[2], s4, s5);
          f2_split(sum4[3], s6, s7);
          const float l = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
          l_run = j > 0 ? fmaf(l_run, alpha, l) : l;
        }
        if (!diag) continue;
        // last key tile of the unit: O / l and the LSE
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done + 2 * u + 1, n & 1, abort));
        if (!ok) break;
        tc_fence_after();
        const float inv = 1.f / l_run;
        float x[D];
#pragma unroll
        for (int c = 0; c < D / 32; c++) {
          uint32_t w[32];
          tmem_ld32(obuf + c * 32, w);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e++) x[c * 32 + e] = __uint_as_float(w[e]) * inv;
        }
        tc_fence_before();
        warp_arrive(o_free + u);  // O is in registers: the unit's next first O += P V may overwrite it
        // each warp's 32 rows of O leave through its staging area and TMA stores (rows
        // past T are not written); the area is reused once the previous store has read it
        if (ne > 0) {
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
        if (a.o_fp32) {
          stage_rows32<D, 4>(x, ost, lane);
        } else {
          stage_rows32<D, 2>(x, ost, lane);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int span = D * (a.o_fp32 ? 4 : 2) < 128 ? D * (a.o_fp32 ? 4 : 2) : 128;
          const int cols = span / (a.o_fp32 ? 4 : 2);
          for (int c0 = 0, bx = 0; c0 < D; c0 += cols, bx++)
            tma_store_4d(&a.map_o, ost + bx * 32 * span, c0, hu, iu * kTile + q4 * 32, it.b);
          bulk_commit();
        }
        ne++;
        if (t < a.T)
          a.lse[((size_t)it.b * a.Hq + hu) * a.T + t] = (m_use + __log2f(l_run)) * 0.69314718055994531f;
      }
    }
    if (lane == 0) bulk_wait<0>();  // the O stores are done with the staging areas
    if (!ok) record_timeout(a.status, abort);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    tmem_relinquish();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool F8 = false>
cudaError_t launch_fwd4_t(const FwdArgs& a, int grid, cudaStream_t s) {
  using C = Fwd4Cfg<D, F8>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(k_attn_fwd4<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  k_attn_fwd4<D, F8><<<grid, C::kThreads, C::kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

template <int D, bool P>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s) {
  using C = FwdCfg<D, P>;
  const int grid = a.nt * a.B * a.Hkv * (a.G / a.HC);
  // the shared-memory opt-in is a per-device function attribute: set it once per device
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_fwd<D, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  k_attn_fwd<D, P><<<grid, 256, C::kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, bool precise, cudaStream_t s) {
  if (precise) return a.D == 64 ? launch_fwd_t<64, true>(a, s) : launch_fwd_t<32, true>(a, s);
  return a.D == 64 ? launch_fwd4_t<64>(a, a.grid, s) : launch_fwd4_t<32>(a, a.grid, s);
}

cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t s) { return launch_fwd4_t<64, true>(a, a.grid, s); }

cudaError_t launch_rope_amax(const RopeArgs& a, cudaStream_t s) {
  const long long n = (long long)a.B * a.T * (a.Hq + a.Hkv) * 8;
  const long long want = (n + 4 * 256 - 1) / (4 * 256);
  const int blocks = (int)(want < 4096 ? want : 4096);  // few blocks: each merges its maxima once
  k_rope_amax<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_q8(const RopeArgs& a, cudaStream_t s) {
  const long long n = (long long)a.B * a.T * (a.Hq + a.Hkv) * 8;
  const long long want = (n + 255) / 256;
  const int blocks = (int)(want < 65536 ? want : 65536);
  k_rope_q8<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_qk(const RopeArgs& a, int D, cudaStream_t s) {
  // one thread per (position, group of four heads, chunk)
  const long long n = (long long)a.B * a.T * ((a.Hq + a.Hkv + 3) / 4) * (D / 8);
  const long long want = (n + 255) / 256;
  const int blocks = (int)(want < 65536 ? want : 65536);
  if (D == 64)
    k_rope_qk<64><<<blocks, 256, 0, s>>>(a);
  else
    k_rope_qk<32><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ne
