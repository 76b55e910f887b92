// Backward pass of causal GQA attention with RoPE on Q/K (sm_103a).
//
// The NanoEuler pages hand-write the backward of every kernel and check it
// against central finite differences in double precision, RoPE and GQA
// included (socker-news README, "Verified backward"; openai-hub article on
// the hand-written forward/backward).  With P = softmax(S), S = scale Q^ K^T:
//   dV = P^T dO,  dP = dO V^T,  Delta_t = sum_j P_tj dP_tj = dO_t . O_t,
//   dS = P o (dP - Delta),  dQ^ = scale dS K^,  dK^ = scale dS^T Q^,
//   dq = R^T dQ^, dk = R^T dK^ (summed over the query heads of the group).
//
// Three kernels:
//   k_bwd_prep  (HBM-bound, one pass): Delta = rowsum(dO o O), lse*log2(e),
//               rotated copies q^, k^ (fp16; with precise logits also their
//               fp16 remainders), zeroed fp32 dQ accumulator.
//   k_bwd_dkdv  CTA = (key tile j, batch b, kv head g); sweeps query tiles
//               i >= j and the G query heads of the group:
//     warp 0    TMA producer (K^_j, V_j once; then Q^_i, dO_i, lse, Delta)
//     warp 1    tcgen05 issuer: S^T = K^ Q^T, dP^T = V dO^T, dV += P^T dO,
//               dK += dS^T Q^, dQ_tile = dS K^ (TMEM accumulators)
//     warps 4-7 one thread per key row: P^T = exp2(S^T scale log2e - lse2),
//               causal mask on the diagonal tile, dS^T = P^T o (dP^T - Delta)
//               (fp16, to shared memory in the layout both MMAs read)
//     warps 8-11 drain dQ_tile from TMEM into swizzled shared memory and add
//               it to the fp32 accumulator with a TMA tensor reduce-add.
//     dK and dV accumulate in TMEM across all (i, head) steps, so the GQA
//     group reduction happens inside the kernel; the epilogue applies scale
//     and the inverse rotation to dK.
//   k_bwd_dq    dq = scale R^T dQacc (bf16 or fp32).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace ne {
namespace {

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, 0, kStatusTimeout);
}

// ====================================================================== pre-pass
template <int D>
__global__ void __launch_bounds__(256) k_bwd_prep(const PrepArgs a) {
  constexpr int kCPR = D / 8;  // 16-byte chunks (8 bf16) per row
  constexpr int kShift = D == 64 ? 3 : 2;
  const uint32_t gtid = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t nthr = gridDim.x * blockDim.x;  // a multiple of 32

  // (A) query rows: rotate q, Delta = dO . O, lse2 = lse * log2(e)
  const uint32_t nA = (uint32_t)a.B * a.T * a.Hq * kCPR;
  const uint32_t nA32 = (nA + 31u) / 32u * 32u;
  for (uint32_t it = gtid; it < nA32; it += nthr) {
    const bool valid = it < nA;
    float part = 0.f;
    uint32_t h = 0, t = 0, b = 0;
    int c = 0;
    if (valid) {
      const uint32_t row = it >> kShift;  // (b, t, h)
      c = (int)(it & (kCPR - 1));
      const uint32_t bt = fdiv(row, a.div_hq);
      h = row - bt * a.Hq;
      b = fdiv(bt, a.div_t);
      t = bt - b * a.T;
      const uint4 dv = __ldg(reinterpret_cast<const uint4*>(a.dout) + it);
      float4 o0, o1;
      uint4 ov;
      if (a.o_fp32) {
        const float4* op = reinterpret_cast<const float4*>(a.o) + 2 * (size_t)it;
        o0 = __ldg(op);
        o1 = __ldg(op + 1);
      } else {
        ov = __ldg(reinterpret_cast<const uint4*>(a.o) + it);
      }
      if (a.rotate_qk) {
        const uint4 qv = load_rope_chunk<D>(a.q + (size_t)row * D, c, a.rope_half != 0);
        float4 c0, c1;
        rope_coeffs<D>(a.rope, (int)t, c, c0, c1);
        if (a.qlo) {
          uint4 l;
          reinterpret_cast<uint4*>(a.qr)[it] = rope_chunk_f16(qv, c0, c1, &l);
          reinterpret_cast<uint4*>(a.qlo)[it] = l;
        } else {
          reinterpret_cast<uint4*>(a.qr)[it] = rope_chunk_f16(qv, c0, c1, nullptr);
        }
      }
      const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
      if (a.o_fp32) {
        part = o0.x * bf_lo(dw[0]) + o0.y * bf_hi(dw[0]) + o0.z * bf_lo(dw[1]) + o0.w * bf_hi(dw[1]) +
               o1.x * bf_lo(dw[2]) + o1.y * bf_hi(dw[2]) + o1.z * bf_lo(dw[3]) + o1.w * bf_hi(dw[3]);
      } else {
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
        for (int p = 0; p < 4; p++) part += bf_lo(ow[p]) * bf_lo(dw[p]) + bf_hi(ow[p]) * bf_hi(dw[p]);
      }
    }
#pragma unroll
    for (int off = kCPR / 2; off >= 1; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (valid && c == 0) {
      const size_t o = ((size_t)b * a.Hq + h) * a.Tp + t;
      a.delta[o] = a.negate ? -part : part;
      const size_t li = ((size_t)b * a.Hq + h) * a.T + t;
      if (a.lse_lo) {
        // (hi + lo) * log2(e) as a two-part value, with a two-part log2(e).
        const float hi = a.lse[li], lo = a.lse_lo[li];
        const float h2 = __fmul_rn(hi, kLog2eHi);
        a.lse2[o] = h2;
        a.lse2_lo[o] = fmaf(hi, kLog2eHi, -h2) + hi * kLog2eLo + lo * kLog2eHi;
      } else {
        const float l2 = a.lse[li] * 1.4426950408889634f;
        a.lse2[o] = a.negate ? -l2 : l2;
      }
    }
  }
  // (B) key rows: rotate k (unless the forward's rotated copy is already there)
  const uint32_t nB = a.rotate_qk ? (uint32_t)a.B * a.T * a.Hkv * kCPR : 0u;
  for (uint32_t it = gtid; it < nB; it += nthr) {
    const uint32_t row = it >> kShift;
    const int c = (int)(it & (kCPR - 1));
    const uint32_t bt = fdiv(row, a.div_hkv);
    const uint32_t t = bt - fdiv(bt, a.div_t) * a.T;
    const uint4 kv = load_rope_chunk<D>(a.k + (size_t)row * D, c, a.rope_half != 0);
    float4 c0, c1;
    rope_coeffs<D>(a.rope, (int)t, c, c0, c1);
    if (a.klo) {
      uint4 l;
      reinterpret_cast<uint4*>(a.kr)[it] = rope_chunk_f16(kv, c0, c1, &l);
      reinterpret_cast<uint4*>(a.klo)[it] = l;
    } else {
      reinterpret_cast<uint4*>(a.kr)[it] = rope_chunk_f16(kv, c0, c1, nullptr);
    }
  }
  // (C) zero the dQ accumulator [B, Hq, Tp, D]
  const uint32_t nC = (uint32_t)a.B * a.Hq * a.Tp * (D / 4);
  for (uint32_t it = gtid; it < nC; it += nthr) reinterpret_cast<float4*>(a.dqacc)[it] = make_float4(0.f, 0.f, 0.f, 0.f);
  // (D) padded rows t in [T, Tp): no probability mass (lse2 = +inf), Delta = 0
  const uint32_t npad = (uint32_t)(a.Tp - a.T);
  const uint32_t nD = (uint32_t)a.B * a.Hq * npad;
  for (uint32_t it = gtid; it < nD; it += nthr) {
    const uint32_t bh = fdiv(it, a.div_pad);
    const uint32_t t = (uint32_t)a.T + (it - bh * npad);
    a.delta[(size_t)bh * a.Tp + t] = 0.f;
    a.lse2[(size_t)bh * a.Tp + t] = __int_as_float(a.negate ? 0xff800000 : 0x7f800000);
    if (a.lse2_lo) a.lse2_lo[(size_t)bh * a.Tp + t] = 0.f;
  }
}

// ====================================================================== dq epilogue
// dq = scale R_t^T dQacc.  A thread takes one 32-byte chunk c (four pairs) of
// one position (b, t) for a group of four query heads, so the chunk's
// (cos, sin) entries are read once for the four, whose loads are in flight
// together.
template <int D>
__global__ void __launch_bounds__(256) k_bwd_dq(const DqArgs a) {
  constexpr int kCPR = D / 8;
  constexpr int kU = 4;  // heads per thread
  const uint32_t ngr = (uint32_t)(a.Hq + kU - 1) / kU;
  const uint32_t n = (uint32_t)a.B * a.T * ngr * kCPR;
  for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < n; it += gridDim.x * blockDim.x) {
    const int c = (int)(it % kCPR);
    const uint32_t rest = it / kCPR;  // (b * T + t) * ngr + head group
    const uint32_t bt = fdiv(rest, a.div_hg);
    const int h0 = (int)(rest - bt * ngr) * kU;
    const uint32_t b = fdiv(bt, a.div_t);
    const uint32_t t = bt - b * a.T;
    float4 c0, c1;
    rope_coeffs<D>(a.rope, (int)t, c, c0, c1);
    const float cs[4] = {c0.x, c0.z, c1.x, c1.z}, sn[4] = {c0.y, c0.w, c1.y, c1.w};
    {
      float4 x0[kU], x1[kU];
#pragma unroll
      for (int u = 0; u < kU; u++) {
        if (h0 + u < a.Hq) {
          const float4* src = reinterpret_cast<const float4*>(
              a.dqacc + (((size_t)b * a.Hq + h0 + u) * a.Tp + t) * D + c * 8);
          x0[u] = src[0];
          x1[u] = src[1];
        }
      }
#pragma unroll
      for (int u = 0; u < kU; u++) {
        const int h = h0 + u;
        if (h >= a.Hq) continue;
        const float xs[8] = {x0[u].x, x0[u].y, x0[u].z, x0[u].w, x1[u].x, x1[u].y, x1[u].z, x1[u].w};
        float y[8];
#pragma unroll
        for (int p = 0; p < 4; p++) {
          y[2 * p] = a.scale * (xs[2 * p] * cs[p] + xs[2 * p + 1] * sn[p]);
          y[2 * p + 1] = a.scale * (xs[2 * p + 1] * cs[p] - xs[2 * p] * sn[p]);
        }
        const size_t row = (size_t)bt * a.Hq + h;  // (b, t, h)
        if (a.rope_half) {
          // pair p of the chunk is (x[4c + p], x[D/2 + 4c + p]) of the row
          const size_t r0 = row * D + 4 * c, r1 = r0 + D / 2;
          if (a.grad_fp32) {
            *reinterpret_cast<float4*>(static_cast<float*>(a.dq) + r0) = make_float4(y[0], y[2], y[4], y[6]);
            *reinterpret_cast<float4*>(static_cast<float*>(a.dq) + r1) = make_float4(y[1], y[3], y[5], y[7]);
          } else {
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.dq) + r0) =
                make_uint2(pack_bf16(y[0], y[2]), pack_bf16(y[4], y[6]));
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.dq) + r1) =
                make_uint2(pack_bf16(y[1], y[3]), pack_bf16(y[5], y[7]));
          }
        } else if (a.grad_fp32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.dq) + row * D + c * 8);
          dst[0] = make_float4(y[0], y[1], y[2], y[3]);
          dst[1] = make_float4(y[4], y[5], y[6], y[7]);
        } else {
          reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dq) + row * D)[c] =
              make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
        }
      }
    }
  }
}

// ====================================================================== dK/dV sweep
template <int D, bool PRECISE>
struct BwdCfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr uint32_t kSpan = D * 2;
  static constexpr uint32_t kSwz = D == 64 ? kSw128 : kSw64;
  static constexpr uint32_t kSBO = 8 * kSpan;
  // PRECISE runs the steps one after another (one stage, one dS and one dQ
  // buffer): its extra operands (remainder tiles, dS lo, P lo) fill the
  // shared and tensor memory the overlap would need.
  static constexpr int kStages = PRECISE ? 1 : 2;
  static constexpr int kLo = PRECISE ? 1 : 0;
  static constexpr int kDsBufs = PRECISE ? 1 : 2;
  static constexpr int kDqBufs = PRECISE ? 1 : 2;
  static constexpr int kVecBytes = kTile * 4;  // lse2 / Delta slice of one tile
  static constexpr int kDsBytes = kTile * kTile * 2;
  static constexpr int kDsParts = PRECISE ? 2 : 1;  // hi (+ lo) fp16 parts of dS
  static constexpr int kStgBytes = kTile * D * 4;
  static constexpr int kOffK = 0;
  static constexpr int kOffKlo = kOffK + kTileBytes;
  static constexpr int kOffV = kOffKlo + kLo * kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;
  static constexpr int kOffQlo = kOffQ + kStages * kTileBytes;
  static constexpr int kOffDO = kOffQlo + kLo * kStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;
  static constexpr int kOffStg = kOffDS + kDsBufs * kDsParts * kDsBytes;
  static constexpr int kOffLse = kOffStg + kStgBytes;
  static constexpr int kOffLlo = kOffLse + kStages * kVecBytes;  // lse2 remainder (PRECISE)
  static constexpr int kOffDel = kOffLlo + kLo * kStages * kVecBytes;
  static constexpr int kOffBar = kOffDel + kStages * kVecBytes;
  static constexpr int kNumBars = 1 + 2 * kStages + 4 + 2 * 2 + 2 * 2 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // tensor memory columns: S^T/P^T, dP^T, dV, dK, dQ buffers, P^T lo (PRECISE)
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D, kColDQ = 256 + 2 * D;
  static constexpr uint32_t kColPlo = kColDQ + kDqBufs * D;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kColPlo + (PRECISE ? 64 : 0) <= kTmemCols, "tensor memory budget");
};

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also returns the AND of `v` over the participating threads.
__device__ __forceinline__ bool named_sync_and(int id, int nthreads, bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* m, const void* src, int c0, int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(c0), "r"(c1), "r"(smem_u32(src))
      : "memory");
}

// Writes 32 fp16 values (packed pairs w[0..15]) for queries c*32..c*32+31 of
// key row r into a dS^T tile: two 16 KB atoms of 64 queries, 128-byte swizzle.
__device__ __forceinline__ void store_ds_chunk(uint8_t* ds, int r, int c, const uint32_t (&w)[16]) {
  uint8_t* atom = ds + (c >> 1) * 16384;
#pragma unroll
  for (int q4 = 0; q4 < 4; q4++)
    *reinterpret_cast<uint4*>(atom + swz(r, (c & 1) * 4 + q4, 128)) =
        make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
}

template <int D, bool PRECISE>
__global__ void __launch_bounds__(384, 1) k_bwd_dkdv(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D, PRECISE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* qd_full = kv_full + 1;             // [kStages]
  uint64_t* qd_empty = qd_full + C::kStages;   // [kStages]
  uint64_t* s_full = qd_empty + C::kStages;
  uint64_t* p_ready = s_full + 1;
  uint64_t* dp_full = p_ready + 1;
  uint64_t* acc_done = dp_full + 1;
  uint64_t* ds_ready = acc_done + 1;  // [kDsBufs]
  uint64_t* ds_free = ds_ready + 2;   // [kDsBufs]
  uint64_t* dq_full = ds_free + 2;    // [kDqBufs]
  uint64_t* dq_free = dq_full + 2;    // [kDqBufs]
  uint64_t* drain = dq_free + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_j = a.B * a.Hkv;
  const int j = (int)blockIdx.x / per_j;  // smallest j (longest sweep) first
  const int rem = (int)blockIdx.x % per_j;
  const int kvh = rem % a.Hkv, b = rem / a.Hkv;
  const int G = a.G;
  const int N = (a.nt - j) * G;  // (query tile, head) steps

  if (tid == 0) {
    *abort = 0;
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::kStages; s++) {
      mbar_init(qd_full + s, 1);
      mbar_init(qd_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_ready, 128);
    mbar_init(dp_full, 1);
    mbar_init(acc_done, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(ds_ready + s, 128);
      mbar_init(ds_free + s, 1);
      mbar_init(dq_full + s, 1);
      mbar_init(dq_free + s, 128);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const volatile int never = 0;
  const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
  const uint32_t sKlo = smem_u32(smem + C::kOffKlo), sQlo = smem_u32(smem + C::kOffQlo);
  const uint32_t sQ = smem_u32(smem + C::kOffQ), sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sDS = smem_u32(smem + C::kOffDS);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.map_qr);
      prefetch_tmap(&a.map_do);
      mbar_arrive_expect_tx(kv_full, (2 + C::kLo) * C::kTileBytes);
      tma_load_4d(smem + C::kOffK, &a.map_kr, kv_full, 0, kvh, j * kTile, b);
      if (PRECISE) tma_load_4d(smem + C::kOffKlo, &a.map_klo, kv_full, 0, kvh, j * kTile, b);
      tma_load_4d(smem + C::kOffV, &a.map_v, kv_full, 0, kvh, j * kTile, b);
      int loaded = 0;
      for (int n = 0; n < N; n++) {
        const int st = n % C::kStages, use = n / C::kStages;
        if (use > 0 && !mbar_wait(qd_empty + st, (use - 1) & 1, abort)) {
          record_timeout(a.status, abort);
          break;
        }
        const int i = j + n / G, h = kvh * G + n % G;
        const size_t vec = ((size_t)b * a.Hq + h) * a.Tp + (size_t)i * kTile;
        mbar_arrive_expect_tx(qd_full + st, (2 + C::kLo) * C::kTileBytes + (2 + C::kLo) * C::kVecBytes);
        tma_load_4d(smem + C::kOffQ + st * C::kTileBytes, &a.map_qr, qd_full + st, 0, h, i * kTile, b);
        if (PRECISE)
          tma_load_4d(smem + C::kOffQlo + st * C::kTileBytes, &a.map_qlo, qd_full + st, 0, h, i * kTile, b);
        tma_load_4d(smem + C::kOffDO + st * C::kTileBytes, &a.map_do, qd_full + st, 0, h, i * kTile, b);
        bulk_load(smem + C::kOffLse + st * C::kVecBytes, a.lse2 + vec, C::kVecBytes, qd_full + st);
        if (PRECISE) bulk_load(smem + C::kOffLlo + st * C::kVecBytes, a.lse2_lo + vec, C::kVecBytes, qd_full + st);
        bulk_load(smem + C::kOffDel + st * C::kVecBytes, a.delta + vec, C::kVecBytes, qd_full + st);
        loaded = n + 1;
      }
      mbar_wait(kv_full, 0, &never);
      for (int n = loaded - C::kStages < 0 ? 0 : loaded - C::kStages; n < loaded; n++)
        mbar_wait(qd_full + n % C::kStages, (n / C::kStages) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_fp16(128, 128, false, false);   // K^ Q^T (fp16)
      constexpr uint32_t idDP = idesc_bf16(128, 128, false, false);  // V dO^T (bf16)
      constexpr uint32_t idDV = idesc_bf16(128, D, false, true);     // P^T (TMEM) x dO MN-major
      constexpr uint32_t idDK = idesc_fp16(128, D, false, true);     // dS^T x Q^ MN-major
      constexpr uint32_t idDQ = idesc_fp16(128, D, true, true);      // dS (MN-major) x K^ MN-major
      auto issue_kmajor = [&](uint32_t col, uint32_t sa, uint32_t sb, uint32_t id, uint32_t acc) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ks++)
          mma_ss(tmem + col, smem_desc(sa + ks * 32, 16, C::kSBO, C::kSwz),
                 smem_desc(sb + ks * 32, 16, C::kSBO, C::kSwz), id, (acc || ks > 0) ? 1u : 0u);
      };
      // S^T = Khi Qhi^T (+ Khi Qlo^T + Klo Qhi^T): the forward's products in the
      // forward's order, so the recomputed logits round as the forward's did
      auto issue_s = [&](int stq) {
        issue_kmajor(C::kColS, sK, sQ + stq * C::kTileBytes, idS, 0);
        if (PRECISE) {
          issue_kmajor(C::kColS, sK, sQlo + stq * C::kTileBytes, idS, 1);
          issue_kmajor(C::kColS, sKlo, sQ + stq * C::kTileBytes, idS, 1);
        }
      };
      // dK += dS^T Q (A = dS^T tile read K-major), dQ = dS K (A = dS^T tile read MN-major)
      auto issue_dk = [&](uint32_t ds, uint32_t qsm, uint32_t acc) {
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ks++)
          mma_ss(tmem + C::kColDK, smem_desc(ds + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024, kSw128),
                 smem_desc(qsm + ks * 16 * C::kSpan, 16, C::kSBO, C::kSwz), idDK, (acc || ks > 0) ? 1u : 0u);
      };
      auto issue_dq = [&](uint32_t col, uint32_t ds, uint32_t ksm, uint32_t acc) {
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ks++)
          mma_ss(tmem + col, smem_desc(ds + ks * 2048, 16384, 1024, kSw128),
                 smem_desc(ksm + ks * 16 * C::kSpan, 16, C::kSBO, C::kSwz), idDQ, (acc || ks > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(kv_full, 0, abort) && mbar_wait(qd_full, 0, abort);
      tc_fence_after();
      if (ok) {
        issue_s(0);
        mma_commit(s_full);
        issue_kmajor(C::kColDP, sV, sDO, idDP, 0);
        mma_commit(dp_full);
      }
      for (int n = 0; ok && n < N; n++) {
        const int st = n % C::kStages;
        const uint32_t q_s = sQ + st * C::kTileBytes, do_s = sDO + st * C::kTileBytes;
        // dV += P^T dO   (A = P^T in TMEM: hi, and lo when PRECISE; B = dO MN-major)
        if (!(ok = mbar_wait(p_ready, n & 1, abort))) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ks++)
          mma_ts(tmem + C::kColDV, tmem + C::kColS + ks * 8,
                 smem_desc(do_s + ks * 16 * C::kSpan, 16, C::kSBO, C::kSwz), idDV, (n > 0 || ks > 0) ? 1u : 0u);
        if (PRECISE) {
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ks++)
            mma_ts(tmem + C::kColDV, tmem + C::kColPlo + ks * 8,
                   smem_desc(do_s + ks * 16 * C::kSpan, 16, C::kSBO, C::kSwz), idDV, 1u);
        }
        // Overlapped order: the next S^T goes in right after the dV MMAs that
        // read this step's P^T from the same columns.
        const int st1 = (n + 1) % C::kStages;
        if (!PRECISE && n + 1 < N) {
          if (!(ok = mbar_wait(qd_full + st1, ((n + 1) / C::kStages) & 1, abort))) break;
          tc_fence_after();
          issue_s(st1);
          mma_commit(s_full);
        }
        const int dsb = n % C::kDsBufs, qb = n % C::kDqBufs;
        const uint32_t ds = sDS + dsb * C::kDsParts * C::kDsBytes;
        if (!(ok = mbar_wait(ds_ready + dsb, (n / C::kDsBufs) & 1, abort))) break;
        tc_fence_after();
        issue_dk(ds, q_s, n > 0);
        if (PRECISE) {
          issue_dk(ds + C::kDsBytes, q_s, 1);                          // dS lo x Q hi
          issue_dk(ds, sQlo + st * C::kTileBytes, 1);                  // dS hi x Q lo
        }
        if (n >= C::kDqBufs) {
          if (!(ok = mbar_wait(dq_free + qb, ((n - C::kDqBufs) / C::kDqBufs) & 1, abort))) break;
          tc_fence_after();
        }
        const uint32_t dqcol = C::kColDQ + qb * D;
        issue_dq(dqcol, ds, sK, 0);
        if (PRECISE) {
          issue_dq(dqcol, ds + C::kDsBytes, sK, 1);                    // dS lo x K hi
          issue_dq(dqcol, ds, sKlo, 1);                                // dS hi x K lo
        }
        mma_commit(dq_full + qb);
        mma_commit(ds_free + dsb);
        mma_commit(qd_empty + st);
        if (n + 1 < N) {
          if (PRECISE) {
            // Serial order: this step's P^T (read back by the compute warps
            // for dS) stays in TMEM until ds_ready, so S^T waits until here.
            if (!(ok = mbar_wait(qd_full + st1, ((n + 1) / C::kStages) & 1, abort))) break;
            tc_fence_after();
            issue_s(st1);
            mma_commit(s_full);
          }
          // next dP^T (the compute warps finished reading dP^T before signalling ds_ready)
          issue_kmajor(C::kColDP, sV, sDO + st1 * C::kTileBytes, idDP, 0);
          mma_commit(dp_full);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      mma_commit(acc_done);
      mma_commit(drain);
      mbar_wait(drain, 0, &never);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ P and dS (one key row per thread)
    const int r = tid - 128;
    const uint32_t trow = tmem + ((uint32_t)(warp - 4) * 32u << 16);
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int n = 0; n < N; n++) {
      const int st = n % C::kStages;
      const int i = j + n / G;
      const bool diag = (i == j);
      const float* lse2 = reinterpret_cast<const float*>(smem + C::kOffLse + st * C::kVecBytes);
      const float* lse2lo = reinterpret_cast<const float*>(smem + C::kOffLlo + st * C::kVecBytes);
      const float* del = reinterpret_cast<const float*>(smem + C::kOffDel + st * C::kVecBytes);
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full, n & 1, abort)))) break;
      tc_fence_after();
      uint32_t pk[PRECISE ? 1 : kTile / 2];  // P^T row as packed bf16 pairs (default mode)
#pragma unroll
      for (int c = 0; c < kTile / 32; c++) {
        uint32_t u[32];
        tmem_ld32(trow + C::kColS + c * 32, u);
        // the 32 lse2 values of this chunk: broadcast vector loads while the TMEM load is in flight
        float l2[32], l2lo[PRECISE ? 32 : 1];
#pragma unroll
        for (int v4 = 0; v4 < 8; v4++) {
          const float4 t4 = reinterpret_cast<const float4*>(lse2 + c * 32)[v4];
          l2[4 * v4] = t4.x, l2[4 * v4 + 1] = t4.y, l2[4 * v4 + 2] = t4.z, l2[4 * v4 + 3] = t4.w;
          if (PRECISE) {
            const float4 t5 = reinterpret_cast<const float4*>(lse2lo + c * 32)[v4];
            l2lo[4 * v4] = t5.x, l2lo[4 * v4 + 1] = t5.y, l2lo[4 * v4 + 2] = t5.z, l2lo[4 * v4 + 3] = t5.w;
          }
        }
        tmem_wait_ld();
        uint32_t w[16], wl[16];
#pragma unroll
        for (int e = 0; e < 16; e++) {
          const int q0 = c * 32 + 2 * e;
          const float s0 = __uint_as_float(u[2 * e]), s1 = __uint_as_float(u[2 * e + 1]);
          float x0 = fmaf(s0, sl2, -l2[2 * e]), x1 = fmaf(s1, sl2, -l2[2 * e + 1]);
          if (PRECISE) {  // logits of 10^3..10^4: add the remainders of scale and LSE
            x0 += s0 * a.scale_log2_lo - l2lo[2 * e];
            x1 += s1 * a.scale_log2_lo - l2lo[2 * e + 1];
          }
          float p0 = ex2(x0);
          float p1 = ex2(x1);
          if (diag) {
            if (q0 < r) p0 = 0.f;
            if (q0 + 1 < r) p1 = 0.f;
          }
          w[e] = pack_bf16(p0, p1);
          if (PRECISE)
            wl[e] = pack_bf16(p0 - bf_lo(w[e]), p1 - bf_hi(w[e]));
          else
            pk[c * 16 + e] = w[e];
        }
        tmem_st16(trow + C::kColS + c * 16, w);
        if (PRECISE) tmem_st16(trow + C::kColPlo + c * 16, wl);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_ready);

      const int dsb = n % C::kDsBufs;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(dp_full, n & 1, abort)))) break;
      if (n >= C::kDsBufs &&
          !(ok = __all_sync(0xffffffffu, mbar_wait(ds_free + dsb, ((n - C::kDsBufs) / C::kDsBufs) & 1, abort))))
        break;
      tc_fence_after();
      uint8_t* ds = smem + C::kOffDS + dsb * C::kDsParts * C::kDsBytes;
#pragma unroll
      for (int c = 0; c < kTile / 32; c++) {
        uint32_t u[32];
        tmem_ld32(trow + C::kColDP + c * 32, u);
        uint32_t ph[16], pl[16];
        if (PRECISE) {
          // P^T = hi + lo (bf16 pairs) is still in TMEM: the next S^T is not issued before ds_ready.
          tmem_ld16(trow + C::kColS + c * 16, ph);
          tmem_ld16(trow + C::kColPlo + c * 16, pl);
        }
        float dl[32];
#pragma unroll
        for (int v4 = 0; v4 < 8; v4++) {
          const float4 t4 = reinterpret_cast<const float4*>(del + c * 32)[v4];
          dl[4 * v4] = t4.x, dl[4 * v4 + 1] = t4.y, dl[4 * v4 + 2] = t4.z, dl[4 * v4 + 3] = t4.w;
        }
        tmem_wait_ld();
        uint32_t w[16], wl[16];
#pragma unroll
        for (int e = 0; e < 16; e++) {
          float p0, p1;
          if (PRECISE) {
            p0 = bf_lo(ph[e]) + bf_lo(pl[e]);
            p1 = bf_hi(ph[e]) + bf_hi(pl[e]);
          } else {
            p0 = bf_lo(pk[c * 16 + e]);
            p1 = bf_hi(pk[c * 16 + e]);
          }
          const float d0 = (__uint_as_float(u[2 * e]) - dl[2 * e]) * p0;
          const float d1 = (__uint_as_float(u[2 * e + 1]) - dl[2 * e + 1]) * p1;
          w[e] = pack_f16(d0, d1);
          if (PRECISE) wl[e] = pack_f16(d0 - f16_lo(w[e]), d1 - f16_hi(w[e]));
        }
        store_ds_chunk(ds, r, c, w);
        if (PRECISE) store_ds_chunk(ds + C::kDsBytes, r, c, wl);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ds_ready + dsb);
    }
    // dK epilogue: scale, inverse rotation, store
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort));
    if (ok) {
      tc_fence_after();
      const int t = j * kTile + r;
      float x[D];
#pragma unroll
      for (int c = 0; c < D / 32; c++) {
        uint32_t u[32];
        tmem_ld32(trow + C::kColDK + c * 32, u);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e++) x[c * 32 + e] = __uint_as_float(u[e]);
      }
      if (t < a.T) {
        const size_t base = (((size_t)b * a.T + t) * a.Hkv + kvh) * D;
#pragma unroll
        for (int c = 0; c < D / 8; c++) {
          float4 c0, c1;
          rope_coeffs<D>(a.rope, t, c, c0, c1);
          const float cs[4] = {c0.x, c0.z, c1.x, c1.z}, sn[4] = {c0.y, c0.w, c1.y, c1.w};
          float y[8];
#pragma unroll
          for (int p = 0; p < 4; p++) {
            const float x0 = x[c * 8 + 2 * p], x1 = x[c * 8 + 2 * p + 1];
            y[2 * p] = a.scale * (x0 * cs[p] + x1 * sn[p]);
            y[2 * p + 1] = a.scale * (x1 * cs[p] - x0 * sn[p]);
          }
          if (a.grad_fp32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.dk) + base + c * 8);
            dst[0] = make_float4(y[0], y[1], y[2], y[3]);
            dst[1] = make_float4(y[4], y[5], y[6], y[7]);
          } else {
            reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dk) + base)[c] =
                make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
          }
        }
      }
    }
    if (!ok) record_timeout(a.status, abort);
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ drain (one query row per thread)
    const int r = tid - 256;
    const uint32_t trow = tmem + ((uint32_t)(warp - 8) * 32u << 16);
    uint8_t* stg = smem + C::kOffStg;
    bool ok = true;
    for (int n = 0; n < N; n++) {
      const int qb = n % C::kDqBufs;
      // Every drain thread reaches both named barriers of an iteration; the
      // first one agrees on `ok`, so a timeout in one warp stops all four.
      const bool got = __all_sync(0xffffffffu, mbar_wait(dq_full + qb, (n / C::kDqBufs) & 1, abort));
      uint32_t u[D];
      if (got) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; c++) {
          uint32_t v[32];
          tmem_ld32(trow + C::kColDQ + qb * D + c * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e++) u[c * 32 + e] = v[e];
        }
        tc_fence_before();
        mbar_arrive(dq_free + qb);
      }
      if (r == 0) bulk_wait_read<0>();  // previous reduction has finished reading the staging tile
      if (!(ok = named_sync_and(1, 128, got))) break;
#pragma unroll
      for (int bx = 0; bx < D / 32; bx++)
#pragma unroll
        for (int c = 0; c < 8; c++)
          *reinterpret_cast<uint4*>(stg + bx * 16384 + swz(r, c, 128)) =
              make_uint4(u[bx * 32 + 4 * c], u[bx * 32 + 4 * c + 1], u[bx * 32 + 4 * c + 2], u[bx * 32 + 4 * c + 3]);
      fence_proxy_async_smem();
      named_sync(1, 128);
      if (r == 0) {
        const int i = j + n / G, h = kvh * G + n % G;
        const int row0 = (int)(((size_t)b * a.Hq + h) * a.Tp + (size_t)i * kTile);
#pragma unroll
        for (int bx = 0; bx < D / 32; bx++) tma_reduce_add_2d(&a.map_dqacc, stg + bx * 16384, bx * 32, row0);
        bulk_commit();
      }
    }
    if (r == 0) bulk_wait<0>();
    // dV epilogue
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort));
    if (ok) {
      tc_fence_after();
      const int t = j * kTile + r;
      uint32_t u[D];
#pragma unroll
      for (int c = 0; c < D / 32; c++) {
        uint32_t v[32];
        tmem_ld32(trow + C::kColDV + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e++) u[c * 32 + e] = v[e];
      }
      if (t < a.T) {
        const size_t base = (((size_t)b * a.T + t) * a.Hkv + kvh) * D;
        if (a.grad_fp32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.dv) + base);
#pragma unroll
          for (int c = 0; c < D / 4; c++)
            dst[c] = make_float4(__uint_as_float(u[4 * c]), __uint_as_float(u[4 * c + 1]), __uint_as_float(u[4 * c + 2]),
                                 __uint_as_float(u[4 * c + 3]));
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dv) + base);
#pragma unroll
          for (int c = 0; c < D / 8; c++)
            dst[c] = make_uint4(pack_bf16(__uint_as_float(u[8 * c]), __uint_as_float(u[8 * c + 1])),
                                pack_bf16(__uint_as_float(u[8 * c + 2]), __uint_as_float(u[8 * c + 3])),
                                pack_bf16(__uint_as_float(u[8 * c + 4]), __uint_as_float(u[8 * c + 5])),
                                pack_bf16(__uint_as_float(u[8 * c + 6]), __uint_as_float(u[8 * c + 7])));
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

// ====================================================================== persistent dK/dV sweep
// One CTA per SM loops over work items (key tile j, batch, kv head), longest
// sweep first in a snake order.  An item accumulates dK and dV of its key
// tile over the query tiles i >= j of every query head of the group (one
// step per (i, head)).  S^T = K Q^T and dP^T = V dO^T read K and V from shared
// memory (double-buffered across items, so the next item's K and V load
// while this one runs); P^T gets TMEM columns of its own, so S^T of the next
// step may overwrite the score columns as soon as the compute warps have read
// them, and dP^T of the next step may overwrite its columns as soon as they
// are read.  dS goes to shared memory once, where dK reads it K-major and dQ
// MN-major.  The accumulators pass from one item to the next through acc_done
// (MMAs complete) and acc_free (the compute warps have read them).
// Warps: 0 TMA producer; 1-3 MMA issuers; 4-11 P and dS (two warpgroups, half
// the query columns each), then each item's dK / dV store; 12-15 dQ drain.
template <int D>
struct Bwd3Cfg {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr uint32_t kSpan = D * 2;
  static constexpr uint32_t kSwz = D == 64 ? kSw128 : kSw64;
  static constexpr uint32_t kSBO = 8 * kSpan;
  static constexpr int kStages = 3;
  static constexpr int kVecBytes = kTile * 4;
  static constexpr int kDsBytes = kTile * kTile * 2;
  static constexpr int kStgBytes = kTile * 32 * 4;  // one 32-column box of the fp32 dQ tile
  static constexpr int kOffKV = 0;  // [2] x (K, V)
  static constexpr int kOffQ = kOffKV + 4 * kTileBytes;
  static constexpr int kOffDO = kOffQ + kStages * kTileBytes;
  static constexpr int kOffDS = kOffDO + kStages * kTileBytes;
  static constexpr int kOffStg = kOffDS + kDsBytes;
  static constexpr int kOffLse = kOffStg + kStgBytes;
  static constexpr int kOffDel = kOffLse + kStages * kVecBytes;
  // (cos, sin) rows of the rotation table for the dK epilogue, position
  // t = t0 + 16a + b split three ways: the row of each item's t0 = 128 j (one per
  // K/V buffer), rows 16a (a < 8) and rows b (b < 16, padded so that the 16 rows
  // one warp reads start in different banks)
  static constexpr int kRotRow = D * 4;
  static constexpr int kRotStrideB = kRotRow + 16;
  static constexpr int kOffRot = kOffDel + kStages * kVecBytes;
  static constexpr int kOffRotA = kOffRot + 2 * kRotRow;
  static constexpr int kOffRotB = kOffRotA + 8 * kRotRow;
  static constexpr int kOffBar = kOffRotB + 16 * kRotStrideB;
  static constexpr int kNumBars = 32;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // TMEM: S^T | dP^T | P^T | dV | dK | dQ
  static constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDV = 320, kColDK = 320 + D,
                            kColDQ = 320 + 2 * D;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kColDQ + D <= kTmemCols, "tensor memory budget");
};

struct BwdItem {
  int j, b, kvh, N;  // N = (nt - j) * G steps
};

__device__ __forceinline__ bool bwd_item(const BwdArgs& a, int tl, BwdItem& it) {
  const int G = (int)gridDim.x, c = (int)blockIdx.x;
  const int w = (tl & 1) ? (tl + 1) * G - 1 - c : tl * G + c;  // snake over the longest-first order
  const int per_j = a.B * a.Hkv;
  if (w >= a.nt * per_j) return false;
  it.j = w / per_j;
  const int rem = w % per_j;
  it.kvh = rem % a.Hkv;
  it.b = rem / a.Hkv;
  it.N = (a.nt - it.j) * a.G;
  return true;
}

// Writes row r of a 128-row tile of a gradient (values x, fp32 when ES == 4,
// else bf16) into staging boxes of 128 rows by min(D * ES, 128) bytes with the
// TMA / UMMA swizzle of that span: box 0 at stg0, box 1 (fp32 rows of D = 64
// only) at stg1.  Returns the number of boxes.  HALF: x holds the rotated
// (interleaved) order of a half-split row, whose column j is x[2j] (j < D/2)
// or x[2(j - D/2) + 1].
template <int D, int ES, bool HALF = false>
__device__ __forceinline__ int stage_grad(const float (&x)[D], uint8_t* stg0, uint8_t* stg1, int r) {
  constexpr int kSpan = D * ES < 128 ? D * ES : 128;
  constexpr int kCols = kSpan / ES;
  auto col = [&](int j) { return HALF ? x[j < D / 2 ? 2 * j : 2 * (j - D / 2) + 1] : x[j]; };
#pragma unroll
  for (int c0 = 0, bx = 0; c0 < D; c0 += kCols, bx++) {
    uint8_t* stg = bx == 0 ? stg0 : stg1;
#pragma unroll
    for (int ch = 0; ch < kSpan / 16; ch++) {
      uint4 w;
      if constexpr (ES == 4) {
        const int i = c0 + ch * 4;
        w = make_uint4(__float_as_uint(col(i)), __float_as_uint(col(i + 1)), __float_as_uint(col(i + 2)),
                       __float_as_uint(col(i + 3)));
      } else {
        const int i = c0 + ch * 8;
        w = make_uint4(pack_bf16(col(i), col(i + 1)), pack_bf16(col(i + 2), col(i + 3)),
                       pack_bf16(col(i + 4), col(i + 5)), pack_bf16(col(i + 6), col(i + 7)));
      }
      *reinterpret_cast<uint4*>(stg + swz(r, ch, kSpan)) = w;
    }
  }
  return D / kCols;
}

// kSplit: fp32 gradients of D = 64 in the interleaved layout, whose item
// epilogue splits the columns between the two compute warpgroups.
template <int D, bool kSplit>
__global__ void __launch_bounds__(512, 1) k_bwd_dkdv3(const __grid_constant__ BwdArgs a) {
  using C = Bwd3Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;        // [2]
  uint64_t* kv_empty = bars + 2;   // [2] released by the three issuers and the item's gradient stores
  uint64_t* qd_full = bars + 4;    // [kStages]
  uint64_t* qd_empty = bars + 7;   // [kStages] released by issuers 1 and 2
  uint64_t* s_full = bars + 10;
  uint64_t* s_read = bars + 11;    // the compute warps hold S^T in registers
  uint64_t* p_ready = bars + 12;
  uint64_t* pbuf_free = bars + 13; // dV read P^T
  uint64_t* dp_full = bars + 14;
  uint64_t* ds_ready = bars + 15;
  uint64_t* ds_free = bars + 16;   // dK and dQ read the dS tile
  uint64_t* dq_full = bars + 17;
  uint64_t* dq_free = bars + 18;
  uint64_t* acc_done = bars + 19;  // an item's last dV and dK complete
  uint64_t* acc_free = bars + 20;  // the compute warps read dK and dV
  uint64_t* drain = bars + 21;     // [3]
  uint64_t* stg_full = bars + 24;  // [2] per compute warpgroup: its rows of the item's gradient are staged
  uint64_t* stg_free = bars + 26;  // [2] the gradient's TMA stores have read the staging
  uint64_t* dp_read = bars + 28;   // the compute warps hold dP^T(g): dP^T(g+1) may overwrite it
  uint64_t* rot_full = bars + 30;  // rows 16a and b of the rotation table are in shared memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G;

  if (tid == 0) {
    *abort = 0;
    for (int s = 0; s < 2; s++) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_empty + s, 5);  // the three issuers, and both compute warpgroups' gradient stores
    }
    for (int s = 0; s < C::kStages; s++) {
      mbar_init(qd_full + s, 1);
      mbar_init(qd_empty + s, 2);
    }
    mbar_init(s_full, 1);
    mbar_init(s_read, 8);  // one arrival per warp of the compute warps
    mbar_init(p_ready, 8);
    mbar_init(pbuf_free, 1);
    mbar_init(dp_full, 1);
    mbar_init(ds_ready, 8);
    mbar_init(ds_free, 2);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);
    mbar_init(acc_done, 2);
    mbar_init(acc_free, 8);
    for (int s = 0; s < 3; s++) mbar_init(drain + s, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(stg_full + s, 4);
      mbar_init(stg_free + s, 1);
    }
    mbar_init(dp_read, 8);
    mbar_init(rot_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const volatile int never = 0;
  const uint32_t sKV = smem_u32(smem + C::kOffKV);
  const uint32_t sQ = smem_u32(smem + C::kOffQ), sDO = smem_u32(smem + C::kOffDO);
  const uint32_t sDS = smem_u32(smem + C::kOffDS);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.map_qr);
      prefetch_tmap(&a.map_do);
      prefetch_tmap(&a.map_kr);
      prefetch_tmap(&a.map_v);
      bool ok = true;
      int g = 0, kv_loaded = 0;
      const uint8_t* rot = reinterpret_cast<const uint8_t*>(a.rope);
      mbar_arrive_expect_tx(rot_full, 24 * C::kRotRow);
      for (int x = 0; x < 8; x++)
        bulk_load(smem + C::kOffRotA + x * C::kRotRow, rot + (size_t)16 * x * C::kRotRow, C::kRotRow, rot_full);
      for (int x = 0; x < 16; x++)
        bulk_load(smem + C::kOffRotB + x * C::kRotStrideB, rot + (size_t)x * C::kRotRow, C::kRotRow, rot_full);
      auto load_kv = [&](int k, const BwdItem& x) -> bool {
        const int kb = k & 1;
        if (k >= 2 && !mbar_wait(kv_empty + kb, ((k >> 1) - 1) & 1, abort)) return false;
        mbar_arrive_expect_tx(kv_full + kb, 2 * C::kTileBytes + C::kRotRow);
        tma_load_4d(smem + C::kOffKV + kb * 2 * C::kTileBytes, &a.map_kr, kv_full + kb, 0, x.kvh, x.j * kTile, x.b);
        tma_load_4d(smem + C::kOffKV + (kb * 2 + 1) * C::kTileBytes, &a.map_v, kv_full + kb, 0, x.kvh, x.j * kTile,
                    x.b);
        bulk_load(smem + C::kOffRot + kb * C::kRotRow, rot + (size_t)x.j * kTile * C::kRotRow, C::kRotRow,
                  kv_full + kb);
        kv_loaded = k + 1;
        return true;
      };
      BwdItem it, nx;
      if (bwd_item(a, 0, it)) ok = load_kv(0, it);
      for (int tl = 0; ok && bwd_item(a, tl, it); tl++) {
        for (int n = 0; n < it.N; n++, g++) {
          const int st = g % C::kStages, use = g / C::kStages;
          if (use > 0 && !(ok = mbar_wait(qd_empty + st, (use - 1) & 1, abort))) break;
          const int i = it.j + n / G, h = it.kvh * G + n % G;
          const size_t vec = ((size_t)it.b * a.Hq + h) * a.Tp + (size_t)i * kTile;
          mbar_arrive_expect_tx(qd_full + st, 2 * C::kTileBytes + 2 * C::kVecBytes);
          tma_load_4d(smem + C::kOffQ + st * C::kTileBytes, &a.map_qr, qd_full + st, 0, h, i * kTile, it.b);
          tma_load_4d(smem + C::kOffDO + st * C::kTileBytes, &a.map_do, qd_full + st, 0, h, i * kTile, it.b);
          bulk_load(smem + C::kOffLse + st * C::kVecBytes, a.lse2 + vec, C::kVecBytes, qd_full + st);
          bulk_load(smem + C::kOffDel + st * C::kVecBytes, a.delta + vec, C::kVecBytes, qd_full + st);
          // the next item's K and V, once the previous user of that buffer is done
          // (after this item's second step is queued, so that wait delays no early step)
          if (n == (it.N > 1 ? 1 : 0) && bwd_item(a, tl + 1, nx) && !(ok = load_kv(tl + 1, nx))) break;
        }
      }
      if (!ok) record_timeout(a.status, abort);
      // let every copy issued above land before the CTA can exit
      for (int k = kv_loaded - 2 < 0 ? 0 : kv_loaded - 2; k < kv_loaded; k++)
        mbar_wait(kv_full + (k & 1), (k >> 1) & 1, &never);
      for (int x = g - C::kStages < 0 ? 0 : g - C::kStages; x < g; x++)
        mbar_wait(qd_full + x % C::kStages, (x / C::kStages) & 1, &never);
      mbar_wait(rot_full, 0, &never);
    }
  } else if (warp >= 1 && warp <= 3) {
    // ------------------------------------------------------------ MMA issuers
    // One thread issues about one MMA per 70-120 cycles, so each step's 32
    // MMAs are spread over three threads.  Every overwrite of a TMEM operand
    // follows its last read behind a barrier:
    //   warp 1: S^T(g+1) once the compute warps read S^T(g), and dV += P^T dO;
    //   warp 2: dP^T(g+1) once the compute warps read dP^T(g), then dK += dS^T Q;
    //   warp 3: the dQ tile = dS K (dS from shared memory).
    if (lane == 0) {
      constexpr uint32_t idS = idesc_fp16(128, 128, false, false);   // K^ x Q^ (both K-major)
      constexpr uint32_t idDP = idesc_bf16(128, 128, false, false);  // V x dO (both K-major)
      constexpr uint32_t idDV = idesc_bf16(128, D, false, true);     // P^T (TMEM) x dO MN-major
      constexpr uint32_t idDK = idesc_fp16(128, D, false, true);     // dS^T (K-major) x Q^ MN-major
      constexpr uint32_t idDQ = idesc_fp16(128, D, true, true);      // dS (MN-major) x K^ MN-major
      constexpr int KD = D / 16;                                     // k-steps over the head dimension
      constexpr uint32_t kStepK = 32 >> 4;                           // K-major: next 16 columns
      constexpr uint32_t kStepMN = (16 * C::kSpan) >> 4;             // MN-major: next 16 rows
      constexpr uint32_t kTileStep = C::kTileBytes >> 4;
      const uint64_t dQ0 = smem_desc(sQ, 16, C::kSBO, C::kSwz);
      const uint64_t dDO0 = smem_desc(sDO, 16, C::kSBO, C::kSwz);
      const uint64_t dKV0 = smem_desc(sKV, 16, C::kSBO, C::kSwz);
      const uint64_t dDS = smem_desc(sDS, 16384, 1024, kSw128);   // dS, MN-major (for dQ)
      const uint64_t dDSk = smem_desc(sDS, 16, 1024, kSw128);     // dS^T, K-major (for dK)
      auto dK = [&](int kb) { return dKV0 + (uint64_t)(2 * kb * kTileStep); };
      auto dV = [&](int kb) { return dKV0 + (uint64_t)((2 * kb + 1) * kTileStep); };
      auto dQs = [&](int st) { return dQ0 + (uint64_t)(st * kTileStep); };
      auto dDOs = [&](int st) { return dDO0 + (uint64_t)(st * kTileStep); };
      bool ok = true;
      int g = 0;
      BwdItem it;
      if (warp == 1) {
        // S^T of the first step
        BwdItem nx;
        const bool any = bwd_item(a, 0, it);
        if (any && (ok = mbar_wait(kv_full, 0, abort) && mbar_wait(qd_full, 0, abort))) {
          tc_fence_after();
          mma_ss_chain<KD>(tmem + C::kColS, dK(0), kStepK, dQs(0), kStepK, idS, 0);
          mma_commit(s_full);
        }
        for (int tl = 0; ok && bwd_item(a, tl, it); tl++) {
          const int kb = tl & 1;
          for (int n = 0; n < it.N; n++, g++) {
            const int st = g % C::kStages;
            // S^T of the next step (this item's or the next item's first) and dV of
            // this step touch different TMEM columns: issue each as soon as its
            // inputs are there, so a late Q / dO load does not hold up dV.
            const bool last = (n + 1 == it.N);
            bool need_s = !last || bwd_item(a, tl + 1, nx);
            bool need_dv = true;
            const int g1 = g + 1, st1 = g1 % C::kStages, kb1 = last ? (kb ^ 1) : kb;
            const unsigned long long t_start = globaltimer();
            while (need_s || need_dv) {
              bool progressed = false;
              if (need_s && mbar_test(s_read, g & 1) && (!last || mbar_test(kv_full + kb1, ((tl + 1) >> 1) & 1)) &&
                  mbar_test(qd_full + st1, (g1 / C::kStages) & 1)) {
                tc_fence_after();
                mma_ss_chain<KD>(tmem + C::kColS, dK(kb1), kStepK, dQs(st1), kStepK, idS, 0);
                mma_commit(s_full);
                need_s = false;
                progressed = true;
              }
              // dV += P^T dO (the first step of an item starts from zero once the
              // previous item's dV has been read out)
              if (need_dv && mbar_test(p_ready, g & 1) && (n > 0 || tl == 0 || mbar_test(acc_free, (tl - 1) & 1))) {
                tc_fence_after();
                mma_ts_chain<8, false>(tmem + C::kColDV, tmem + C::kColP, dDOs(st), kStepMN, idDV, n > 0 ? 1u : 0u);
                mma_commit(pbuf_free);
                mma_commit(qd_empty + st);  // this thread's reads of stage st: Q^ by S^T, dO by dV
                if (last) {
                  mma_commit(acc_done);
                  mma_commit(kv_empty + kb);  // K by S^T
                }
                need_dv = false;
                progressed = true;
              }
              if (!progressed) {
                if (*abort || globaltimer() - t_start > kWaitLimitNs) {
                  ok = false;
                  break;
                }
                __nanosleep(64);  // leave the issue slots to the compute warps
              }
            }
            if (!ok) break;
          }
        }
      } else if (warp == 2) {
        const bool any = bwd_item(a, 0, it);
        if (any && (ok = mbar_wait(kv_full, 0, abort) && mbar_wait(qd_full, 0, abort))) {
          tc_fence_after();
          mma_ss_chain<KD>(tmem + C::kColDP, dV(0), kStepK, dDOs(0), kStepK, idDP, 0);
          mma_commit(dp_full);
        }
        BwdItem nx;
        for (int tl = 0; ok && bwd_item(a, tl, it); tl++) {
          const int kb = tl & 1;
          for (int n = 0; n < it.N; n++, g++) {
            const int st = g % C::kStages;
            const bool last = (n + 1 == it.N);
            // dP^T(g+1) as soon as the compute warps hold dP^T(g), ahead of dK(g)
            if (!last || bwd_item(a, tl + 1, nx)) {
              const int g1 = g + 1, st1 = g1 % C::kStages, kb1 = last ? (kb ^ 1) : kb;
              if (!(ok = mbar_wait(dp_read, g & 1, abort))) break;
              if (last && !(ok = mbar_wait(kv_full + kb1, ((tl + 1) >> 1) & 1, abort))) break;
              if (!(ok = mbar_wait(qd_full + st1, (g1 / C::kStages) & 1, abort))) break;
              tc_fence_after();
              mma_ss_chain<KD>(tmem + C::kColDP, dV(kb1), kStepK, dDOs(st1), kStepK, idDP, 0);
              mma_commit(dp_full);
            }
            if (!(ok = mbar_wait(ds_ready, g & 1, abort))) break;
            if (n == 0 && tl > 0 && !(ok = mbar_wait(acc_free, (tl - 1) & 1, abort))) break;
            tc_fence_after();
            // dK += dS^T Q^: the dS tile in shared memory read K-major (queries
            // along K), one chain of four k-steps per 128-byte swizzle atom of 64 queries
            mma_ss_chain<4>(tmem + C::kColDK, dDSk, kStepK, dQs(st), kStepMN, idDK, n > 0 ? 1u : 0u);
            mma_ss_chain<4>(tmem + C::kColDK, dDSk + (16384 >> 4), kStepK, dQs(st) + 4 * kStepMN, kStepMN, idDK, 1u);
            mma_commit(ds_free);
            mma_commit(qd_empty + st);  // this thread's reads of stage st: dO by dP^T, Q^ by dK
            if (last) {
              mma_commit(acc_done);
              mma_commit(kv_empty + kb);  // V by dP^T
            }
          }
        }
      } else {
        for (int tl = 0; ok && bwd_item(a, tl, it); tl++) {
          const int kb = tl & 1;
          if (!(ok = mbar_wait(kv_full + kb, (tl >> 1) & 1, abort))) break;  // K^ in shared memory
          for (int n = 0; n < it.N; n++, g++) {
            if (!(ok = mbar_wait(ds_ready, g & 1, abort))) break;
            if (g >= 1 && !(ok = mbar_wait(dq_free, (g - 1) & 1, abort))) break;
            tc_fence_after();
            mma_ss_chain<8>(tmem + C::kColDQ, dDS, 2048 >> 4, dK(kb), kStepMN, idDQ, 0);
            mma_commit(dq_full);
            mma_commit(ds_free);
            if (n + 1 == it.N) mma_commit(kv_empty + kb);  // K by dQ
          }
        }
      }
      if (!ok) record_timeout(a.status, abort);
      uint64_t* my_drain = drain + (warp - 1);
      mma_commit(my_drain);
      mbar_wait(my_drain, 0, &never);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ P and dS, half the query columns each
    const int wg = (warp - 4) >> 2;          // 0: queries 0..63, 1: queries 64..127
    const int r = tid - 128 - wg * 128;      // key row
    const int cbase = wg * 64;
    const uint32_t trow = tmem + ((uint32_t)(warp & 3) * 32u << 16);
    const float sl2 = a.scale_log2;
    const uint32_t x7 = (uint32_t)(r & 7);  // swizzle of this key row in the dS tile
    uint8_t* atom = smem + C::kOffDS + wg * 16384;
    bool ok = true;
    int g = 0, epi = 0;  // steps and item epilogues of this warpgroup so far
    BwdItem it;
    for (int tl = 0; ok && bwd_item(a, tl, it); tl++) {
      for (int n = 0; n < it.N; n++, g++) {
        const int st = g % C::kStages;
        const int i = it.j + n / G;
        const bool diag = (i == it.j);
        const float* lse2 = reinterpret_cast<const float*>(smem + C::kOffLse + st * C::kVecBytes) + cbase;
        const float* del = reinterpret_cast<const float*>(smem + C::kOffDel + st * C::kVecBytes) + cbase;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(s_full, g & 1, abort)))) break;
        tc_fence_after();
        // P^T = exp2(s * scale_log2 - lse2) for this thread's 64 query columns (the
        // vectors hold -lse2 and -Delta): the scores arrive with one TMEM round trip
        // and turn into fp32 P in the same registers, then into bf16 pairs (for dV and dS)
        float pf[64];
        uint32_t(&pu)[64] = *reinterpret_cast<uint32_t(*)[64]>(pf);
#pragma unroll
        for (int c = 0; c < 4; c++)
          tmem_ld16(trow + C::kColS + cbase + c * 16, *reinterpret_cast<uint32_t(*)[16]>(pu + 16 * c));
        tmem_wait_ld();
        tc_fence_before();
        warp_arrive(s_read);  // S^T of the next step may overwrite the score columns
        const uint64_t sl2x2 = f2(sl2, sl2);
        auto exp_pass = [&](auto masked) {
#pragma unroll
          for (int v4 = 0; v4 < 16; v4++) {
            const float4 t4 = reinterpret_cast<const float4*>(lse2)[v4];
#pragma unroll
            for (int e = 0; e < 2; e++) {
              const int q = 4 * v4 + 2 * e;
              float x0, x1;
              f2_split(f2_fma(f2(pf[q], pf[q + 1]), sl2x2, e == 0 ? f2(t4.x, t4.y) : f2(t4.z, t4.w)), x0, x1);
              float p0 = ex2(x0), p1 = ex2(x1);
              if constexpr (decltype(masked)::value) {
                if (cbase + q < r) p0 = 0.f;
                if (cbase + q + 1 < r) p1 = 0.f;
              }
              pf[q] = p0;
              pf[q + 1] = p1;
            }
          }
        };
        // the causal mask only on the diagonal tile, in a copy of the pass of its own
        if (diag)
          exp_pass(std::true_type());
        else
          exp_pass(std::false_type());
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 32; q++) pk[q] = pack_bf16(pf[2 * q], pf[2 * q + 1]);
        // the P^T columns are free once dV(g-1) has read P^T(g-1)
        if (g > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(pbuf_free, (g - 1) & 1, abort)))) break;
        tc_fence_after();
#pragma unroll
        for (int hlf = 0; hlf < 4; hlf++)
          tmem_st8(trow + C::kColP + wg * 32 + hlf * 8, *reinterpret_cast<const uint32_t(*)[8]>(pk + 8 * hlf));
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(p_ready);

        if (!(ok = __all_sync(0xffffffffu, mbar_wait(dp_full, g & 1, abort)))) break;
        if (g > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (g - 1) & 1, abort)))) break;
        if (n == 0 && epi > 0) {
          // the previous item's gradient stores read this warpgroup's half of the dS
          // tile (and its K or V buffer): dS may go there once they have
          if (r == 0) {
            bulk_wait_read<0>();
            mbar_arrive(stg_free + wg);
            mbar_arrive(kv_empty + ((tl - 1) & 1));
          }
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(stg_free + wg, (epi - 1) & 1, abort)))) break;
        }
        tc_fence_after();
        // dS = P * (dP - Delta), 16 columns at a time; the next chunk of dP^T loads
        // while this one is computed (its columns are never the ones being stored)
        uint32_t va[16], vb[16];
        tmem_ld16(trow + C::kColDP + cbase, va);
        tmem_wait_ld();
#pragma unroll
        for (int c4 = 0; c4 < 4; c4++) {
          uint32_t(&v)[16] = (c4 & 1) ? vb : va;
          uint32_t(&nxt)[16] = (c4 & 1) ? va : vb;
          if (c4 < 3) tmem_ld16(trow + C::kColDP + cbase + (c4 + 1) * 16, nxt);
          uint32_t w[8];
#pragma unroll
          for (int v4 = 0; v4 < 4; v4++) {
            const float4 t4 = reinterpret_cast<const float4*>(del + c4 * 16)[v4];
#pragma unroll
            for (int e = 0; e < 2; e++) {
              const int q = 4 * v4 + 2 * e;  // column within this quarter
              const uint64_t d = f2_mul(f2_add(f2(__uint_as_float(v[q]), __uint_as_float(v[q + 1])),
                                               e == 0 ? f2(t4.x, t4.y) : f2(t4.z, t4.w)),
                                        f2(bf_lo(pk[c4 * 8 + (q >> 1)]), bf_hi(pk[c4 * 8 + (q >> 1)])));
              float d0, d1;
              f2_split(d, d0, d1);
              w[q >> 1] = pack_f16(d0, d1);
            }
          }
          // dS into shared memory, where both dK (K-major) and dQ (MN-major) read it
#pragma unroll
          for (int q = 0; q < 2; q++)
            *reinterpret_cast<uint4*>(atom + r * 128 + (((uint32_t)(2 * c4 + q) ^ x7) << 4)) =
                make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          if (c4 < 3) tmem_wait_ld();
          if (c4 == 2) {
            tc_fence_before();
            warp_arrive(dp_read);  // dP^T(g+1) may overwrite the dP^T columns
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(ds_ready);
      }
      if (!ok) break;
      // Item epilogue: dK = scale * (inverse rotation of the accumulated dK^) and
      // dV, stored with TMA from swizzled staging boxes of 128 rows by 128 bytes.
      // fp32 gradients of D = 64 in the interleaved layout ("split"): each
      // warpgroup takes half the columns of both accumulators (dK and dV columns
      // 32 wg .. 32 wg + 31), so the two share the rotation.  Otherwise warps
      // 4-7 store dK and warps 8-11 dV, whole rows.
      constexpr bool split = kSplit;
      // The angle of pair i at t = t0 + 16a + b is the sum of three table angles,
      // so its (cos, sin) is the product of three unit complex numbers from
      // shared memory (each table entry is rounded once; the products add a few
      // fp32 roundings).  The t0 row came with this item's K and V.
      auto rotate = [&](float* xr, int p0, auto np_c) {
        constexpr int np = decltype(np_c)::value;
        const float2* r0 = reinterpret_cast<const float2*>(smem + C::kOffRot + (tl & 1) * C::kRotRow) + p0;
        const float2* ra = reinterpret_cast<const float2*>(smem + C::kOffRotA + (r >> 4) * C::kRotRow) + p0;
        const float2* rb = reinterpret_cast<const float2*>(smem + C::kOffRotB + (r & 15) * C::kRotStrideB) + p0;
#pragma unroll
        for (int i = 0; i < np; i++) {
          const float2 e0 = r0[i], ea = ra[i], eb = rb[i];
          const float cab = fmaf(ea.x, eb.x, -ea.y * eb.y), sab = fmaf(ea.y, eb.x, ea.x * eb.y);
          const float cs = fmaf(e0.x, cab, -e0.y * sab), sn = fmaf(e0.y, cab, e0.x * sab);
          const float x0 = xr[2 * i], x1 = xr[2 * i + 1];
          xr[2 * i] = a.scale * (x0 * cs + x1 * sn);
          xr[2 * i + 1] = a.scale * (x1 * cs - x0 * sn);
        }
      };
      if (wg == 0 || split) {  // the rotation table rows used below are in shared memory
        if (epi == 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(rot_full, 0, abort)))) break;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(kv_full + (tl & 1), (tl >> 1) & 1, abort)))) break;
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(acc_done, tl & 1, abort)))) break;
      tc_fence_after();
      // Staging: the first box goes to this warpgroup's half of the dS tile, the
      // second to this item's K (warps 4-7) or V (warps 8-11) buffer; one thread
      // then stores them (rows past T are not written).  Both are free once the
      // item's last dQ has read the dS tile and K (the last S^T and dP^T, which
      // read K and V, completed before acc_done).  The wait for the stores to read
      // them comes at the next item's first dS, which also releases the K/V
      // buffer to the producer.
      uint8_t* stg1 = smem + C::kOffKV + (2 * (tl & 1) + wg) * C::kTileBytes;
      if constexpr (split) {
        // dK columns 32 wg .. 32 wg + 31 in x[0 .. 31], the same dV columns in x[32 .. 63]
        float x[64];
#pragma unroll
        for (int c = 0; c < 4; c++) {
          uint32_t u[16];
          tmem_ld16(trow + (c < 2 ? C::kColDK : C::kColDV) + wg * 32 + (c & 1) * 16, u);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e++) x[c * 16 + e] = __uint_as_float(u[e]);
        }
        tc_fence_before();
        warp_arrive(acc_free);  // the next item's first dV / dK may overwrite the accumulators
        rotate(x, wg * 16, std::integral_constant<int, 16>());
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (g - 1) & 1, abort)))) break;
        uint8_t* bk = wg == 0 ? atom : stg1;
        uint8_t* bv = wg == 0 ? stg1 : atom;
#pragma unroll
        for (int ch = 0; ch < 8; ch++) {
          *reinterpret_cast<float4*>(bk + swz(r, ch, 128)) =
              make_float4(x[4 * ch], x[4 * ch + 1], x[4 * ch + 2], x[4 * ch + 3]);
          *reinterpret_cast<float4*>(bv + swz(r, ch, 128)) =
              make_float4(x[32 + 4 * ch], x[33 + 4 * ch], x[34 + 4 * ch], x[35 + 4 * ch]);
        }
        fence_proxy_async_smem();
        warp_arrive(stg_full + wg);
        if (r == 0) {
          if ((ok = mbar_wait(stg_full + wg, epi & 1, abort))) {
            tma_store_4d(&a.map_dk, bk, wg * 32, it.kvh, it.j * kTile, it.b);
            tma_store_4d(&a.map_dv, bv, wg * 32, it.kvh, it.j * kTile, it.b);
            bulk_commit();
          }
        }
      } else {
        float x[D];
#pragma unroll
        for (int c = 0; c < D / 16; c++) {
          uint32_t u[16];
          tmem_ld16(trow + (wg == 0 ? C::kColDK : C::kColDV) + c * 16, u);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; e++) x[c * 16 + e] = __uint_as_float(u[e]);
        }
        tc_fence_before();
        warp_arrive(acc_free);
        if (wg == 0) rotate(x, 0, std::integral_constant<int, D / 2>());
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (g - 1) & 1, abort)))) break;
        const CUtensorMap* map = wg == 0 ? &a.map_dk : &a.map_dv;
        int nbox;
        if (wg == 0 && a.rope_half)
          nbox = a.grad_fp32 ? stage_grad<D, 4, true>(x, atom, stg1, r) : stage_grad<D, 2, true>(x, atom, stg1, r);
        else
          nbox = a.grad_fp32 ? stage_grad<D, 4>(x, atom, stg1, r) : stage_grad<D, 2>(x, atom, stg1, r);
        fence_proxy_async_smem();
        warp_arrive(stg_full + wg);
        if (r == 0) {
          if ((ok = mbar_wait(stg_full + wg, epi & 1, abort))) {
            const int span = nbox == 2 ? 128 : D * (a.grad_fp32 ? 4 : 2);
            const int cols = span / (a.grad_fp32 ? 4 : 2);
            tma_store_4d(map, atom, 0, it.kvh, it.j * kTile, it.b);
            if (nbox == 2) tma_store_4d(map, stg1, cols, it.kvh, it.j * kTile, it.b);
            bulk_commit();
          }
        }
      }
      epi++;
      if (!(ok = __all_sync(0xffffffffu, ok))) break;
    }
    if (ok && r == 0) bulk_wait<0>();
    if (!ok) record_timeout(a.status, abort);
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ drain (one query row per thread)
    const int r = tid - 384;
    const uint32_t trow = tmem + ((uint32_t)(warp & 3) * 32u << 16);
    uint8_t* stg = smem + C::kOffStg;
    bool ok = true;
    int g = 0;
    BwdItem it;
    for (int tl = 0; ok && bwd_item(a, tl, it); tl++) {
      for (int n = 0; n < it.N; n++, g++) {
        // Every drain thread reaches both named barriers of a step; the first
        // one agrees on `ok`, so a timeout in one warp stops all four.
        const bool got = __all_sync(0xffffffffu, mbar_wait(dq_full, g & 1, abort));
        uint32_t u[D];
        if (got) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; c++) {
            uint32_t v[32];
            tmem_ld32(trow + C::kColDQ + c * 32, v);
#pragma unroll
            for (int e = 0; e < 32; e++) u[c * 32 + e] = v[e];
          }
          tmem_wait_ld();
          tc_fence_before();
          warp_arrive(dq_free);
        }
        const int i = it.j + n / G, h = it.kvh * G + n % G;
        const int row0 = (int)(((size_t)it.b * a.Hq + h) * a.Tp + (size_t)i * kTile);
#pragma unroll
        for (int bx = 0; bx < D / 32; bx++) {
          if (r == 0) bulk_wait_read<0>();  // previous reduction has finished reading the staging box
          if (!(ok = named_sync_and(1, 128, got))) break;
#pragma unroll
          for (int c = 0; c < 8; c++)
            *reinterpret_cast<uint4*>(stg + swz(r, c, 128)) =
                make_uint4(u[bx * 32 + 4 * c], u[bx * 32 + 4 * c + 1], u[bx * 32 + 4 * c + 2], u[bx * 32 + 4 * c + 3]);
          fence_proxy_async_smem();
          named_sync(1, 128);
          if (r == 0) {
            tma_reduce_add_2d(&a.map_dqacc, stg, bx * 32, row0);
            bulk_commit();
          }
        }
        if (!ok) break;
      }
    }
    if (r == 0) bulk_wait<0>();
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

int elementwise_blocks(long long items) {
  long long blocks = (items + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace

cudaError_t launch_bwd_prep(const PrepArgs& a, cudaStream_t s) {
  const long long items = (long long)a.B * a.Tp * a.Hq * a.D / 4;
  const int blocks = elementwise_blocks(items);
  if (a.D == 64)
    k_bwd_prep<64><<<blocks, 256, 0, s>>>(a);
  else
    k_bwd_prep<32><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const DqArgs& a, cudaStream_t s) {
  // one thread per (position, group of four heads, chunk)
  const long long items = (long long)a.B * a.T * ((a.Hq + 3) / 4) * (a.D / 8);
  const int blocks = elementwise_blocks(items);
  if (a.D == 64)
    k_bwd_dq<64><<<blocks, 256, 0, s>>>(a);
  else
    k_bwd_dq<32><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, bool P>
cudaError_t launch_dkdv_t(const BwdArgs& a, cudaStream_t s) {
  using C = BwdCfg<D, P>;
  const int grid = a.nt * a.B * a.Hkv;
  // the shared-memory opt-in is a per-device function attribute: set it once per device
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_bwd_dkdv<D, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  k_bwd_dkdv<D, P><<<grid, 384, C::kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

template <int D, bool kSplit>
cudaError_t launch_dkdv3_t(const BwdArgs& a, cudaStream_t s) {
  using C = Bwd3Cfg<D>;
  static bool attr_set[64] = {};
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(k_bwd_dkdv3<D, kSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaError_t e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int items = a.nt * a.B * a.Hkv;
  k_bwd_dkdv3<D, kSplit><<<items < nsm ? items : nsm, 512, C::kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdArgs& a, bool precise, cudaStream_t s) {
  if (a.D == 64) {
    if (precise) return launch_dkdv_t<64, true>(a, s);
    return a.grad_fp32 && !a.rope_half ? launch_dkdv3_t<64, true>(a, s) : launch_dkdv3_t<64, false>(a, s);
  }
  return precise ? launch_dkdv_t<32, true>(a, s) : launch_dkdv3_t<32, false>(a, s);
}

}  // namespace ne
