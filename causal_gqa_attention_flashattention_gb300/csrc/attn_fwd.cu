// Forward pass of causal GQA attention with RoPE on Q/K (sm_103a).
//
// The NanoEuler GPU engine's FlashAttention is tiled, uses an online softmax
// and never forms the T x T score matrix (socker-news README, "GPU engine" /
// "Kernels and acceleration"; ojeo summary); its causal mask skips the upper
// triangle instead of masking it (openai-hub article, softmax-kernel section).
// This kernel computes the same result with the GB300 tensor cores:
//
//   CTA = (query tile i of 128 rows, batch b, key/value head g, chunk of HC
//         query heads of g's group).  Tiles are issued largest-i first.
//   warp 0      TMA producer: the HC query tiles once, then K_j / V_j for
//               j = 0..i through a ring of kStages stages.  Each K/V tile is
//               read once and used by all HC heads (GQA sharing).
//   warp 1      tcgen05 MMA issuer: S = Q_h K_j^T into one of two TMEM score
//               buffers, then O_h += P V_j with P read from TMEM.
//   warps 2-3   RoPE: rotate the Q tiles and each K tile in shared memory
//               (in place, through the swizzled layout) before the MMA reads
//               them; rotated values never go to HBM.  Rotated operands are
//               fp16 (three more mantissa bits than bf16).  With PRECISE the
//               fp16 remainder (rotated - hi) goes to a second buffer and
//               S = Qhi Khi^T + Qlo Khi^T + Qhi Klo^T, so the logits carry
//               ~2^-22 relative error even when |s| reaches 10^3.
//   warps 4-7   softmax, one thread per query row: row max, lazy rescale of
//               the TMEM accumulator (only when the max grows by > 2^8),
//               exp2, P (bf16) back into TMEM, row sum of the rounded P (so
//               O is an exact convex combination of V rows with the weights
//               the MMA used; with PRECISE, P = hi + lo in two bf16 parts and
//               O += Phi V + Plo V); epilogue O / l (bf16 or fp32) and
//               LSE = ln(sum exp).
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
// layout, one 16-byte chunk (four pairs) per thread.  Streaming work: every
// byte is read and written once, the cos/sin table stays in L2.
template <int D>
__global__ void __launch_bounds__(256) k_rope_qk(const RopeArgs a) {
  constexpr int kCPR = D / 8;  // 16-byte chunks per row
  constexpr int kShift = D == 64 ? 3 : 2;
  constexpr int kPer = 4;      // chunks per thread, loaded together
  const uint32_t nq = (uint32_t)a.B * a.T * a.Hq * kCPR;
  const uint32_t n = nq + (uint32_t)a.B * a.T * a.Hkv * kCPR;
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < n; base += kPer * stride) {
    uint4 v[kPer];
    float4 c0[kPer], c1[kPer];
#pragma unroll
    for (int u = 0; u < kPer; u++) {
      const uint32_t it = base + u * stride;
      if (it < n) {
        const bool isq = it < nq;
        const uint32_t x = isq ? it : it - nq;
        const uint32_t row = x >> kShift;  // (b, t, h)
        const uint32_t bt = fdiv(row, isq ? a.div_hq : a.div_hkv);
        const uint32_t t = bt - fdiv(bt, a.div_t) * a.T;
        v[u] = load_rope_chunk<D>((isq ? a.q : a.k) + (size_t)row * D, (int)(x & (kCPR - 1)), a.rope_half != 0);
        rope_coeffs<D>(a.rope, (int)t, (int)(x & (kCPR - 1)), c0[u], c1[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kPer; u++) {
      const uint32_t it = base + u * stride;
      if (it < n) {
        const bool isq = it < nq;
        reinterpret_cast<uint4*>(isq ? a.qr : a.kr)[isq ? it : it - nq] = rope_chunk_f16(v[u], c0[u], c1[u], nullptr);
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

// ====================================================================== persistent forward, one head per item
// Default-precision forward over the pre-rotated fp16 q, k.  One CTA per SM
// loops over work items (query tile i, batch, query head), largest first in a
// snake order.  Key tile j of an item is step n of the CTA (n counts across
// items); step n computes S into TMEM score buffer n & 1, is handled by softmax
// warpgroup n & 1 (warps 2-5 or 6-9, one thread per query row) and writes its
// P into TMEM P buffer n & 1, from which O += P V reads it.  With separate S
// and P buffers, S of step n + 2 goes out as soon as step n's scores have been
// read, and P of step n + 2 waits only for the PV of step n (issued a full
// step earlier): the warpgroups never wait for the tensor core in the steady
// state.  The row statistics pass from one step to the next through shared
// memory: the running maximum after the first pass over the scores (m_ready),
// the running sum after the second (l_ready).  The warpgroup of an item's last
// key tile writes O and the LSE.
// Warps: 0 TMA producer, 1 S = Q K^T issuer, 10 O += P V issuer.
// Writes row r of a 128-row tile (D values, fp32 when ES == 4, else bf16) into a
// staging area of column boxes: `span` = min(D * ES, 128) bytes per row, box after
// box, each with the TMA / UMMA swizzle of that span.
template <int D, int ES>
__device__ __forceinline__ void stage_rows(const float (&x)[D], uint8_t* stg, int r) {
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
      *reinterpret_cast<uint4*>(stg + bx * kTile * kSpan + swz(r, ch, kSpan)) = w;
    }
  }
}

// F8: q and k tiles hold e4m3 (one byte per value; 64-byte rows, 64-byte
// swizzle for D = 64); v, P and O keep their formats.
template <int D, bool F8 = false>
struct Fwd3Cfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr uint32_t kSpan = D * 2;
  static constexpr uint32_t kSwz = D == 64 ? kSw128 : kSw64;
  static constexpr uint32_t kSBO = 8 * kSpan;
  static constexpr int kQKTileBytes = kTile * D * (F8 ? 1 : 2);
  static constexpr uint32_t kQKSpan = D * (F8 ? 1 : 2);
  static constexpr uint32_t kQKSwz = kQKSpan == 128 ? kSw128 : (kQKSpan == 64 ? kSw64 : kSw32);
  static constexpr uint32_t kQKSBO = 8 * kQKSpan;
  static constexpr int kStages = 4;  // K/V ring
  static constexpr uint32_t kColO = 0, kColS = 128, kColP = 384;  // S buffers at 128, 256; P buffers at 384, 448
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 352;
  static constexpr int kOffQ = 0;  // [2]
  static constexpr int kOffK = 2 * kQKTileBytes;
  static constexpr int kOffV = kOffK + kStages * kQKTileBytes;
  static constexpr int kOstBytes = kTile * D * 4;                // O staging per warpgroup (fp32 rows at most)
  static constexpr int kOffOst = kOffV + kStages * kTileBytes;    // [2]
  static constexpr int kOffStat = kOffOst + 2 * kOstBytes;         // m[128], l[128]
  static constexpr int kOffBar = kOffStat + 2 * kTile * 4;
  static constexpr int kSmemBytes = kOffBar + 40 * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Fwd3Item {
  int i, b, h;
};

// Item tl of this CTA from the host-built schedule: w indexes the largest-first
// order of (query tile, batch, head), items given out longest first to the CTA
// with the least work so far.
__device__ __forceinline__ bool fwd3_item(const FwdArgs& a, int tl, Fwd3Item& it) {
  if (tl >= a.sched_k) return false;
  const int w = __ldg(a.sched + (size_t)blockIdx.x * a.sched_k + tl);
  if (w < 0) return false;
  const int per_i = a.B * a.Hq;
  it.i = a.nt - 1 - w / per_i;
  const int rem = w % per_i;
  it.h = rem % a.Hq;  // the heads of one kv group sit next to each other: their K/V tiles meet in L2
  it.b = rem / a.Hq;
  return true;
}

template <int D, bool F8>
__global__ void __launch_bounds__(352, 1) k_attn_fwd3(const __grid_constant__ FwdArgs a) {
  using C = Fwd3Cfg<D, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int S = C::kStages;
  constexpr int TB = C::kTileBytes;
  constexpr int TQK = C::kQKTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* q_full = bars;         // [2]
  uint64_t* q_empty = bars + 2;    // [2]
  uint64_t* kv_full = bars + 4;    // [S]
  uint64_t* kv_empty = bars + 8;   // [S]
  uint64_t* s_full = bars + 12;    // [2]
  uint64_t* s_read = bars + 14;    // [2] the step's warpgroup has read its scores
  uint64_t* p_ready = bars + 16;   // [2]
  uint64_t* pv_done = bars + 18;   // [2] PV of the P buffer's last step completed
  uint64_t* m_ready = bars + 20;   // running maximum of the latest step stored
  uint64_t* l_ready = bars + 21;   // running sum of the latest step stored
  uint64_t* o_free = bars + 22;    // the item's O has been read out
  uint64_t* drain = bars + 23;     // [2] one per issuing thread
  uint64_t* ost_full = bars + 26;  // [2] a warpgroup's rows of O are staged
  uint64_t* ost_free = bars + 28;  // [2] the previous store from a warpgroup's staging tile has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 30);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 30) + 1;
  float* sm_m = reinterpret_cast<float*>(smem + C::kOffStat);
  float* sm_l = sm_m + kTile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    *abort = 0;
    for (int k = 0; k < 2; k++) {
      mbar_init(q_full + k, 1);
      mbar_init(q_empty + k, 1);
      mbar_init(s_full + k, 1);
      mbar_init(s_read + k, 4);  // one arrival per warp of the warpgroup
      mbar_init(p_ready + k, 4);
      mbar_init(pv_done + k, 1);
      mbar_init(drain + k, 1);
      mbar_init(ost_full + k, 4);
      mbar_init(ost_free + k, 1);
    }
    for (int k = 0; k < S; k++) {
      mbar_init(kv_full + k, 1);
      mbar_init(kv_empty + k, 1);
    }
    mbar_init(m_ready, 4);
    mbar_init(l_ready, 4);
    mbar_init(o_free, 4);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
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
      int g = 0, loaded_items = 0;
      Fwd3Item it;
      for (int tl = 0; ok && fwd3_item(a, tl, it); tl++) {
        const int qb = tl & 1, kvh = it.h / a.G;
        if (tl >= 2 && !(ok = mbar_wait(q_empty + qb, ((tl >> 1) - 1) & 1, abort))) break;
        mbar_arrive_expect_tx(q_full + qb, TQK);
        tma_load_4d(smem + C::kOffQ + qb * TQK, &a.map_q, q_full + qb, 0, it.h, it.i * kTile, it.b);
        loaded_items = tl + 1;
        for (int j = 0; j <= it.i; j++, g++) {
          const int st = g % S, use = g / S;
          if (use > 0 && !(ok = mbar_wait(kv_empty + st, (use - 1) & 1, abort))) break;
          mbar_arrive_expect_tx(kv_full + st, TQK + TB);
          tma_load_4d(smem + C::kOffK + st * TQK, &a.map_k, kv_full + st, 0, kvh, j * kTile, it.b);
          tma_load_4d(smem + C::kOffV + st * TB, &a.map_v, kv_full + st, 0, kvh, j * kTile, it.b);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      // let every copy issued above land before the CTA can exit
      for (int tl = loaded_items - 2 < 0 ? 0 : loaded_items - 2; tl < loaded_items; tl++)
        mbar_wait(q_full + (tl & 1), (tl >> 1) & 1, &never);
      for (int x = g - S < 0 ? 0 : g - S; x < g; x++) mbar_wait(kv_full + x % S, (x / S) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S = Q K^T issuer
    if (lane == 0) {
      constexpr uint32_t idS = F8 ? idesc_e4m3(128, 128, false, false) : idesc_fp16(128, 128, false, false);
      constexpr uint32_t kStepK = 32 >> 4;  // 16 fp16 or 32 e4m3 values of K
      constexpr uint32_t tstep = (uint32_t)TQK >> 4;
      const uint64_t dQ0 = smem_desc(smem_u32(smem + C::kOffQ), 16, C::kQKSBO, C::kQKSwz);
      const uint64_t dK0 = smem_desc(smem_u32(smem + C::kOffK), 16, C::kQKSBO, C::kQKSwz);
      bool ok = true;
      int g = 0;
      Fwd3Item it;
      for (int tl = 0; ok && fwd3_item(a, tl, it); tl++) {
        const int qb = tl & 1;
        if (!(ok = mbar_wait(q_full + qb, (tl >> 1) & 1, abort))) break;
        for (int j = 0; j <= it.i; j++, g++) {
          const int st = g % S;
          if (!(ok = mbar_wait(kv_full + st, (g / S) & 1, abort))) break;
          // the score buffer's previous step (g - 2) has read its scores
          if (g >= 2 && !(ok = mbar_wait(s_read + (g & 1), ((g >> 1) - 1) & 1, abort))) break;
          tc_fence_after();
          if constexpr (F8)
            mma_ss_chain2_f8(tmem + C::kColS + (g & 1) * 128, dQ0 + (uint64_t)(qb * tstep), kStepK,
                             dK0 + (uint64_t)(st * tstep), kStepK, idS, 0u);
          else
            mma_ss_chain<D / 16>(tmem + C::kColS + (g & 1) * 128, dQ0 + (uint64_t)(qb * tstep), kStepK,
                                 dK0 + (uint64_t)(st * tstep), kStepK, idS, 0u);
          mma_commit(s_full + (g & 1));
          if (j == it.i) mma_commit(q_empty + qb);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      mma_commit(drain);
      mbar_wait(drain, 0, &never);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ O += P V issuer
    if (lane == 0) {
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      constexpr uint32_t kStepMN = (16 * C::kSpan) >> 4;
      constexpr uint32_t tstep = (uint32_t)TB >> 4;
      const uint64_t dV0 = smem_desc(smem_u32(smem + C::kOffV), 16, C::kSBO, C::kSwz);
      bool ok = true;
      int g = 0;
      Fwd3Item it;
      for (int tl = 0; ok && fwd3_item(a, tl, it); tl++) {
        for (int j = 0; j <= it.i; j++, g++) {
          const int st = g % S;
          if (!(ok = mbar_wait(p_ready + (g & 1), (g >> 1) & 1, abort))) break;
          if (j == 0 && tl > 0 && !(ok = mbar_wait(o_free, (tl - 1) & 1, abort))) break;
          tc_fence_after();
          mma_ts_chain<8, false>(tmem + C::kColO, tmem + C::kColP + (g & 1) * 64, dV0 + (uint64_t)(st * tstep),
                                 kStepMN, idPV, j > 0 ? 1u : 0u);
          mma_commit(pv_done + (g & 1));
          // K was read by S(g), which completed before this step's softmax began
          mma_commit(kv_empty + st);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      mma_commit(drain + 1);
      mbar_wait(drain + 1, 0, &never);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = (warp - 2) >> 2;  // 0: warps 2-5, 1: warps 6-9
    const int q4 = warp & 3;         // TMEM lane quarter
    const int r = q4 * 32 + lane;    // query row within the tile
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t sbuf = trow + C::kColS + wg * 128;
    const uint32_t pbuf = trow + C::kColP + wg * 64;
    uint8_t* ost = smem + C::kOffOst + wg * C::kOstBytes;
    float sl2 = a.scale_log2;
    bool ok = true;
    int g = 0, ne = 0;  // ne: this warpgroup's epilogues so far
    Fwd3Item it;
    for (int tl = 0; ok && fwd3_item(a, tl, it); tl++) {
      const int t = it.i * kTile + r;
      if constexpr (F8) {  // scores are in e4m3 code units: fold in the two heads' scales
        const float sq = __ldg(a.qk_amax + it.h), sk = __ldg(a.qk_amax + a.Hq + it.h / a.G);
        sl2 = a.scale_log2 * ((sq > 0.f ? sq : 448.f) * (1.f / 448.f)) * ((sk > 0.f ? sk : 448.f) * (1.f / 448.f));
      }
      for (int j = 0; j <= it.i; j++, g++) {
        if ((g & 1) != wg) continue;
        const bool diag = (j == it.i);
        ok = __all_sync(0xffffffffu, mbar_wait(s_full + wg, (g >> 1) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        // pass 1: row maximum over the 128 keys (masked past the diagonal); the
        // scores of keys 64..127 stay in registers for pass 2
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; e++) mx8[e] = -INFINITY;
        uint32_t hi[64];
#pragma unroll
        for (int h2 = 0; h2 < 2; h2++) {
          uint32_t lo[64];
          uint32_t(&u)[64] = h2 ? hi : lo;
          tmem_ld32(sbuf + h2 * 64, *reinterpret_cast<uint32_t(*)[32]>(u));
          tmem_ld32(sbuf + h2 * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(u + 32));
          tmem_wait_ld();
          if (diag) {
#pragma unroll
            for (int e = 0; e < 64; e++)
              if (h2 * 64 + e > r) u[e] = 0xff800000u;  // -inf: key after the query
          }
#pragma unroll
          for (int e = 0; e < 64; e += 2)
            mx8[(e >> 1) & 7] = fmax3(mx8[(e >> 1) & 7], __uint_as_float(u[e]), __uint_as_float(u[e + 1]));
        }
        const float mxr = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        // running maximum (raw logit units) after the previous key tile, from the other
        // warpgroup; at an item's first tile the wait only orders the two writes of sm_m
        float r_use = mxr, alpha = 1.f;
        if (g > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(m_ready, (g - 1) & 1, abort));
          if (!ok) break;
        }
        if (j > 0) {
          const float r_old = sm_m[r];
          r_use = r_old;
          const float m_old = __fmul_rn(r_old, sl2);
          const float r_new = fmaxf(r_old, mxr);
          const float m_new = __fmul_rn(r_new, sl2);
          // lazy rescale: only when some row's maximum grew by more than 2^8; O must
          // then hold every earlier P V (the latest is step g - 1's)
          if (__any_sync(0xffffffffu, m_new > m_old + 8.0f)) {
            ok = __all_sync(0xffffffffu, mbar_wait(pv_done + ((g - 1) & 1), ((g - 1) >> 1) & 1, abort));
            if (!ok) break;
            tc_fence_after();
            r_use = r_new;
            alpha = ex2(m_old - m_new);
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
        }
        sm_m[r] = r_use;
        warp_arrive(m_ready);
        const float m_use = __fmul_rn(r_use, sl2);
        // P's buffer is free once the PV of step g - 2 has completed
        if (g >= 2) {
          ok = __all_sync(0xffffffffu, mbar_wait(pv_done + wg, ((g >> 1) - 1) & 1, abort));
          if (!ok) break;
        }
        tc_fence_after();
        // pass 2: P = exp2(s * scale_log2 - m) as bf16 into this warpgroup's P buffer.
        // Keys 0..63 are read again, 16 at a time (the next chunk loads while this
        // one is exponentiated); keys 64..127 come from pass 1's registers.
        // (the row sum adds the fp32 values of P; the MMA multiplies their bf16 roundings)
        uint64_t sum4[4] = {0ull, 0ull, 0ull, 0ull};
        const uint64_t sl2x2 = f2(sl2, sl2), negm = f2(-m_use, -m_use);
        uint32_t ua[16], ub[16];
        tmem_ld16(sbuf, ua);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 8; c++) {
          uint32_t(&cur)[16] = c >= 4 ? *reinterpret_cast<uint32_t(*)[16]>(hi + 16 * (c - 4)) : ((c & 1) ? ub : ua);
          uint32_t(&nxt)[16] = (c & 1) ? ua : ub;
          if (c < 3) tmem_ld16(sbuf + (c + 1) * 16, nxt);
          if (diag && c < 4) {
#pragma unroll
            for (int e = 0; e < 16; e++)
              if (16 * c + e > r) cur[e] = 0xff800000u;  // exp2(-inf) = 0
          }
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; e++) {
            float x0, x1;
            f2_split(f2_fma(f2(__uint_as_float(cur[2 * e]), __uint_as_float(cur[2 * e + 1])), sl2x2, negm), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            pk[e] = pack_bf16(p0, p1);
            sum4[e & 3] = f2_add(sum4[e & 3], f2(p0, p1));
          }
          tmem_st8(pbuf + c * 8, pk);
          if (c < 3) tmem_wait_ld();
          if (c == 2) {
            // every score is in registers: S of step g + 2 may overwrite them
            tc_fence_before();
            warp_arrive(s_read + wg);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(p_ready + wg);
        float l;
        {
          float s0, s1, s2, s3, s4, s5, s6, s7;
          f2_split(sum4[0], s0, s1);
          f2_split(sum4[1], s2, s3);
          f2_split(sum4[2], s4, s5);
          f2_split(sum4[3], s6, s7);
          l = ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
        }
        // running sum after the previous key tile; at an item's first tile the wait only
        // orders this step's write of sm_l after the previous step's read
        if (g > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(l_ready, (g - 1) & 1, abort));
          if (!ok) break;
        }
        if (j > 0) l += sm_l[r] * alpha;
        if (!diag) sm_l[r] = l;
        warp_arrive(l_ready);
        if (!diag) continue;
        // last key tile of the item: O / l and the LSE
        ok = __all_sync(0xffffffffu, mbar_wait(pv_done + wg, (g >> 1) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        const float inv = 1.f / l;
        float x[D];
#pragma unroll
        for (int c = 0; c < D / 32; c++) {
          uint32_t w[32];
          tmem_ld32(trow + C::kColO + c * 32, w);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e++) x[c * 32 + e] = __uint_as_float(w[e]) * inv;
        }
        tc_fence_before();
        warp_arrive(o_free);  // O is in registers: the next item's first PV may overwrite it
        // O leaves through the warpgroup's staging tile and a TMA store (rows past T
        // are not written); the tile is reused once the previous store has read it
        if (ne > 0) {
          if (r == 0) {
            bulk_wait_read<0>();
            mbar_arrive(ost_free + wg);
          }
          ok = __all_sync(0xffffffffu, mbar_wait(ost_free + wg, (ne - 1) & 1, abort));
          if (!ok) break;
        }
        if (a.o_fp32) {
          stage_rows<D, 4>(x, ost, r);
        } else {
          stage_rows<D, 2>(x, ost, r);
        }
        fence_proxy_async_smem();
        warp_arrive(ost_full + wg);
        if (r == 0) {
          if (!(ok = mbar_wait(ost_full + wg, ne & 1, abort))) {
            record_timeout(a.status, abort);
          } else {
            const int span = D * (a.o_fp32 ? 4 : 2) < 128 ? D * (a.o_fp32 ? 4 : 2) : 128;
            const int cols = span / (a.o_fp32 ? 4 : 2);
            for (int c0 = 0, bx = 0; c0 < D; c0 += cols, bx++)
              tma_store_4d(&a.map_o, ost + bx * kTile * span, c0, it.h, it.i * kTile, it.b);
            bulk_commit();
          }
        }
        ne++;
        if (!__all_sync(0xffffffffu, ok)) break;
        if (t < a.T)
          a.lse[((size_t)it.b * a.Hq + it.h) * a.T + t] = (__fmul_rn(r_use, sl2) + __log2f(l)) * 0.69314718055994531f;
      }
    }
    if (r == 0) bulk_wait<0>();  // the O stores are done with the staging tiles
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
cudaError_t launch_fwd3_t(const FwdArgs& a, cudaStream_t s) {
  using C = Fwd3Cfg<D, F8>;
  static bool attr_set[64] = {};
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(k_attn_fwd3<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaError_t e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int items = a.nt * a.B * a.Hq;
  k_attn_fwd3<D, F8><<<items < nsm ? items : nsm, C::kThreads, C::kSmemBytes, s>>>(a);
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
  if (a.D == 64) return precise ? launch_fwd_t<64, true>(a, s) : launch_fwd3_t<64>(a, s);
  return precise ? launch_fwd_t<32, true>(a, s) : launch_fwd3_t<32>(a, s);
}

cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t s) { return launch_fwd3_t<64, true>(a, s); }

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
  const long long n = (long long)a.B * a.T * (a.Hq + a.Hkv) * (D / 8);
  const long long want = (n + 4 * 256 - 1) / (4 * 256);  // four chunks per thread
  const int blocks = (int)(want < 65536 ? want : 65536);
  if (D == 64)
    k_rope_qk<64><<<blocks, 256, 0, s>>>(a);
  else
    k_rope_qk<32><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ne
