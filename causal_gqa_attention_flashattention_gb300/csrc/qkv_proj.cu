// RMSNorm + fused Q/K/V projection, the step in front of attention (sm_103a).
//
// Every NanoEuler block computes x + attn(rmsnorm(x)) with a pre-norm RMSNorm
// and no bias anywhere (socker-news README, "Architecture" and the block
// order; mynewscn README, architecture list).  With
//   rstd_r = 1 / sqrt(mean_c x[r, c]^2 + eps)
// the projection is qkv[r, n] = rstd_r * sum_c x[r, c] * w[c] * W[n, c]: the
// norm weight w scales the reduction index, so it folds into the projection
// matrix, and rstd_r scales a whole output row, so it moves to the epilogue.
//
//   k_qkv_prep   rstd for every row (one warp per row) and the folded matrix
//                Wf[n', c] = W[n, c] * w[c] (bf16); for the half-split rotary
//                layout the query and key rows are reordered so that feature
//                pair (i, i + D/2) of a head comes out as adjacent columns
//                (2i, 2i + 1), the order the attention kernels take
//   k_qkv_gemm   persistent tcgen05 GEMM, one CTA per SM over 128 x BN output
//                tiles: x and Wf tiles stream in by TMA through a ring of
//                stages, 64-wide K blocks go to the tensor cores as four
//                128 x BN x 16 MMAs into one of two TMEM accumulators, and four
//                epilogue warps read the other accumulator (one output row per
//                thread), scale it by rstd and rotate query and key features
//                (the rotary embedding, socker-news README "Architecture");
//                v (bf16) and the rotated q, k (fp16, the operand format of the
//                attention forward and backward) leave through shared-memory
//                boxes that a seventh warp stores with TMA, plain q, k (bf16,
//                optional) straight from registers
//
// The rotated fp16 q and k land in the layout of the attention forward's
// workspace, so the forward can skip its own rotation pass.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ne {
namespace {

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  *abort = 1;
  atomicCAS(status, 0, kStatusTimeout);
}

// ====================================================================== row statistics and weight fold
// Blocks [0, row_blocks) take eight rows each (one warp per row); the rest fold
// the weight, one 16-byte chunk (8 values) per thread.
__global__ void __launch_bounds__(256) k_qkv_prep(const QkvArgs a, int row_blocks) {
  const int cpr = a.C / 8;  // 16-byte chunks per row
  if ((int)blockIdx.x < row_blocks) {
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= a.M) return;
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)row * a.C);
    float ss = 0.f;
    // four chunks per lane in flight at once (a 768-wide row is three)
    for (int c0 = lane; c0 < cpr; c0 += 128) {
      uint4 u[4];
#pragma unroll
      for (int k = 0; k < 4; k++) u[k] = c0 + 32 * k < cpr ? __ldg(xr + c0 + 32 * k) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint32_t w[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
#pragma unroll
        for (int p = 0; p < 4; p++) {
          const float lo = __uint_as_float(w[p] << 16), hi = __uint_as_float(w[p] & 0xFFFF0000u);
          ss = fmaf(lo, lo, ss);
          ss = fmaf(hi, hi, ss);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) a.rstd[row] = rsqrtf(ss / (float)a.C + a.eps);
    return;
  }
  const long long n = (long long)a.N * cpr;
  const int qk_rows = (a.Hq + a.Hkv) * a.D;
  for (long long it = (long long)(blockIdx.x - row_blocks) * blockDim.x + threadIdx.x; it < n;
       it += (long long)(gridDim.x - row_blocks) * blockDim.x) {
    const int nd = (int)(it / cpr), c = (int)(it - (long long)nd * cpr);
    int src = nd;
    if (a.rope_half && nd < qk_rows) {
      // destination column j of a head holds feature j / 2 (even j) or D/2 + j / 2 (odd j)
      const int j = nd % a.D;
      src = nd - j + ((j & 1) ? a.D / 2 + (j >> 1) : (j >> 1));
    }
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(a.w + (size_t)src * a.C) + c);
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(a.norm_w) + c);
    const uint32_t wu[4] = {u.x, u.y, u.z, u.w}, gu[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; p++) {
      const float lo = __uint_as_float(wu[p] << 16) * __uint_as_float(gu[p] << 16);
      const float hi = __uint_as_float(wu[p] & 0xFFFF0000u) * __uint_as_float(gu[p] & 0xFFFF0000u);
      o[p] = pack_bf16(lo, hi);
    }
    reinterpret_cast<uint4*>(a.wf + (size_t)nd * a.C)[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ====================================================================== GEMM with the rotary epilogue
template <int BN>
struct QkvCfg {
  static constexpr int kABytes = 128 * 128;  // 128 rows x 64 bf16
  static constexpr int kBBytes = BN * 128;   // BN rows x 64 bf16
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStgBytes = 128 * 64;  // one output box: 128 rows x 32 two-byte values
  static constexpr int kNStg = 8;             // staging boxes in flight
  static constexpr int kStgLag = 4;           // stores the store warp keeps unread before freeing a box
  static constexpr int kBudget = 226 * 1024;
  static constexpr int kFit = (kBudget - kNStg * kStgBytes) / kStageBytes;
  static constexpr int kStages = kFit < 6 ? kFit : 6;
  // full / empty per stage, two accumulators' full / empty, staging full / free,
  // drain, then the TMEM slot and the abort flag: all within 512 bytes
  static_assert((2 * kStages + 4 + 2 * kNStg + 1) * 8 + 8 <= 512, "barrier area");
  static constexpr int kOffStg = kStages * kStageBytes;
  static constexpr int kOffBar = kOffStg + kNStg * kStgBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;  // barriers, slot, flag; alignment slack
  static constexpr uint32_t kTmemCols = 2 * BN <= 256 ? 256 : 512;
  static constexpr int kThreads = 224;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue, warp 6 stores
};

// Eight fp32 values -> one 16-byte chunk of four bf16 pairs.
__device__ __forceinline__ uint4 pack8_bf16(const float* y) {
  return make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
}

// Plain (not rotated) q or k values of one 32-column chunk at column d0 of a
// head, straight from registers: interleaved rows as they are; half-split rows
// take columns 2i, 2i + 1 back to features d0/2 + i and D/2 + d0/2 + i.
template <int D>
__device__ __forceinline__ void store_plain_qk(__nv_bfloat16* head, const float (&y)[32], int d0, bool half) {
  if (!half) {
    uint4* dst = reinterpret_cast<uint4*>(head + d0);
#pragma unroll
    for (int c = 0; c < 4; c++) dst[c] = pack8_bf16(y + 8 * c);
    return;
  }
  uint4* lo = reinterpret_cast<uint4*>(head + d0 / 2);
  uint4* hi = reinterpret_cast<uint4*>(head + D / 2 + d0 / 2);
#pragma unroll
  for (int c = 0; c < 2; c++) {
    lo[c] = make_uint4(pack_bf16(y[16 * c], y[16 * c + 2]), pack_bf16(y[16 * c + 4], y[16 * c + 6]),
                       pack_bf16(y[16 * c + 8], y[16 * c + 10]), pack_bf16(y[16 * c + 12], y[16 * c + 14]));
    hi[c] = make_uint4(pack_bf16(y[16 * c + 1], y[16 * c + 3]), pack_bf16(y[16 * c + 5], y[16 * c + 7]),
                       pack_bf16(y[16 * c + 9], y[16 * c + 11]), pack_bf16(y[16 * c + 13], y[16 * c + 15]));
  }
}

// Rotation of the 16 pairs of one chunk by (cos, sin) entries cs[0..7] (two
// pairs per float4), rounded to fp16.
__device__ __forceinline__ void rotate_chunk_f16(const float (&y)[32], const float4* cs, uint32_t (&h)[16]) {
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const float4 e = cs[k];
    const int j = 4 * k;
    h[2 * k] = pack_f16(fmaf(y[j], e.x, -y[j + 1] * e.y), fmaf(y[j], e.y, y[j + 1] * e.x));
    h[2 * k + 1] = pack_f16(fmaf(y[j + 2], e.z, -y[j + 3] * e.w), fmaf(y[j + 2], e.w, y[j + 3] * e.z));
  }
}

// Which staging box a 32-column chunk of the tile goes through, if any: value
// chunks always, query and key chunks when the rotated copies are written.
struct ChunkDst {
  bool staged, isv, isq;
  int h, d0;
};
template <int D>
__device__ __forceinline__ ChunkDst chunk_dst(const QkvArgs& a, int n0) {
  const int qcols = a.Hq * D, qkcols = (a.Hq + a.Hkv) * D;
  ChunkDst c;
  c.isv = n0 >= qkcols;
  c.isq = n0 < qcols;
  const int nn = c.isv ? n0 - qkcols : (c.isq ? n0 : n0 - qcols);  // head * D + d0 within the tensor
  c.h = nn / D;
  c.d0 = nn - c.h * D;
  c.staged = c.isv || a.qr != nullptr;
  return c;
}

template <int BN, int D>
__global__ void __launch_bounds__(224, 1) k_qkv_gemm(const __grid_constant__ QkvArgs a) {
  using C = QkvCfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;                      // [S] x and Wf tiles landed
  uint64_t* empty = bars + S;                 // [S] the MMAs that read them completed
  uint64_t* acc_full = bars + 2 * S;          // [2] accumulator complete
  uint64_t* acc_empty = acc_full + 2;         // [2] accumulator read out
  uint64_t* stg_full = acc_full + 4;          // [kNStg] a staging box written by the four epilogue warps
  uint64_t* stg_free = stg_full + C::kNStg;   // [kNStg] its store has read it
  uint64_t* drain = stg_free + C::kNStg;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(drain + 1) + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    *abort = 0;
    for (int k = 0; k < S; k++) {
      mbar_init(full + k, 1);
      mbar_init(empty + k, 1);
    }
    for (int k = 0; k < 2; k++) {
      mbar_init(acc_full + k, 1);
      mbar_init(acc_empty + k, 4);  // one arrival per epilogue warp
    }
    for (int k = 0; k < C::kNStg; k++) {
      mbar_init(stg_full + k, 4);
      mbar_init(stg_free + k, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.map_x);
      prefetch_tmap(&a.map_w);
      bool ok = true;
      int g = 0;
      for (int tile = blockIdx.x; ok && tile < a.tiles; tile += gridDim.x) {
        const int m = tile / a.ntn, n = tile - m * a.ntn;
        for (int kb = 0; kb < a.nkb; kb++, g++) {
          const int st = g % S, use = g / S;
          if (use > 0 && !(ok = mbar_wait(empty + st, (use - 1) & 1, abort))) break;
          uint8_t* sa = smem + st * C::kStageBytes;
          mbar_arrive_expect_tx(full + st, C::kStageBytes);
          tma_load_2d(sa, &a.map_x, full + st, kb * 64, m * 128);
          tma_load_2d(sa + C::kABytes, &a.map_w, full + st, kb * 64, n * BN);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      // let the copies issued above land before the CTA can exit
      for (int x = g - S < 0 ? 0 : g - S; x < g; x++) mbar_wait(full + x % S, (x / S) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, BN, false, false);
      bool ok = true;
      int g = 0, tl = 0;
      for (int tile = blockIdx.x; ok && tile < a.tiles; tile += gridDim.x, tl++) {
        const int buf = tl & 1;
        if (tl >= 2 && !(ok = mbar_wait(acc_empty + buf, ((tl >> 1) - 1) & 1, abort))) break;
        tc_fence_after();
        for (int kb = 0; kb < a.nkb; kb++, g++) {
          const int st = g % S;
          if (!(ok = mbar_wait(full + st, (g / S) & 1, abort))) break;
          tc_fence_after();
          uint8_t* sa = smem + st * C::kStageBytes;
          const uint64_t dA = smem_desc(smem_u32(sa), 16, 1024, kSw128);
          const uint64_t dB = smem_desc(smem_u32(sa + C::kABytes), 16, 1024, kSw128);
          mma_ss_chain<4>(tmem + (uint32_t)(buf * BN), dA, 2, dB, 2, idesc, kb > 0 ? 1u : 0u);
          mma_commit(empty + st);
        }
        if (!ok) break;
        mma_commit(acc_full + buf);
      }
      if (!ok) record_timeout(a.status, abort);
      mma_commit(drain);
      mbar_wait(drain, 0, &never);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue, one output row per thread
    // Rotated q, k (fp16) and v (bf16) leave through 128-row x 32-column boxes
    // in shared memory (64-byte swizzle) that warp 6 stores with TMA; plain
    // q, k (optional) are stored from registers.
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int r = quarter * 32 + lane;
    const bool rotating = a.qr != nullptr;
    const int qkcols = (a.Hq + a.Hkv) * D;
    uint8_t* stg = smem + C::kOffStg;
    bool ok = true;
    int tl = 0, ns = 0;  // tiles done, staging boxes used
    for (int tile = blockIdx.x; ok && tile < a.tiles; tile += gridDim.x, tl++) {
      const int m = tile / a.ntn, n = tile - m * a.ntn;
      const int buf = tl & 1;
      // row data that does not depend on the accumulator, loaded before waiting for it
      const int row = m * 128 + r;
      const bool valid = row < a.M;
      const float rs = valid ? __ldg(a.rstd + row) : 0.f;
      const int t = valid ? row % a.T : 0;
      float4 cs[D / 4];  // (cos, sin) of the D/2 pairs at position t
      if (rotating && n * BN < qkcols) {
        const float4* tab = reinterpret_cast<const float4*>(a.rope + (size_t)t * (D / 2));
#pragma unroll
        for (int k = 0; k < D / 4; k++) cs[k] = __ldg(tab + k);
      }
      // every lane leaves together (the tcgen05 loads below are warp-wide)
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(acc_full + buf, (tl >> 1) & 1, abort)))) break;
      tc_fence_after();
      const uint32_t base = tmem + (uint32_t)(buf * BN) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; cc++) {
        const int n0 = n * BN + cc * 32;
        if (n0 >= a.N) break;  // the same for every thread of the tile
        uint32_t u[32];
        tmem_ld32(base + (uint32_t)(cc * 32), u);
        tmem_wait_ld();
        if (cc + 1 == BN / 32 || n0 + 32 >= a.N) {  // the accumulator is read out
          tc_fence_before();
          warp_arrive(acc_empty + buf);
        }
        float y[32];
#pragma unroll
        for (int j = 0; j < 32; j++) y[j] = __uint_as_float(u[j]) * rs;
        const ChunkDst dst = chunk_dst<D>(a, n0);
        if (!dst.isv) {
          __nv_bfloat16* plain = dst.isq ? a.q : a.k;
          if (plain && valid)
            store_plain_qk<D>(plain + ((size_t)row * (dst.isq ? a.Hq : a.Hkv) + dst.h) * D, y, dst.d0,
                              a.rope_half != 0);
        }
        if (!dst.staged) continue;
        // this row's 64 bytes of the box
        const int sb = ns % C::kNStg, use = ns / C::kNStg;
        ns++;
        if (use > 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(stg_free + sb, (use - 1) & 1, abort)))) break;
        uint32_t w[16];
        if (dst.isv) {
#pragma unroll
          for (int k = 0; k < 16; k++) w[k] = pack_bf16(y[2 * k], y[2 * k + 1]);
        } else {
#pragma unroll
          for (int hh = 0; hh < D / 32; hh++)
            if (dst.d0 == hh * 32) rotate_chunk_f16(y, cs + hh * 8, w);
        }
        uint8_t* box = stg + sb * C::kStgBytes;
#pragma unroll
        for (int c = 0; c < 4; c++)
          *reinterpret_cast<uint4*>(box + swz((uint32_t)r, (uint32_t)c, 64)) =
              make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        fence_proxy_async_smem();
        warp_arrive(stg_full + sb);
      }
    }
    if (!ok) record_timeout(a.status, abort);
  } else if (warp == 6) {
    // ------------------------------------------------------------ TMA stores of the staged boxes
    // Walks the chunks in the epilogue's order; a box is handed back once its
    // store has read it, kStgLag stores later.
    if (lane == 0) {
      bool ok = true;
      int ns = 0;
      for (int tile = blockIdx.x; ok && tile < a.tiles; tile += gridDim.x) {
        const int m = tile / a.ntn, n = tile - m * a.ntn;
        for (int cc = 0; cc < BN / 32; cc++) {
          const int n0 = n * BN + cc * 32;
          if (n0 >= a.N) break;
          const ChunkDst dst = chunk_dst<D>(a, n0);
          if (!dst.staged) continue;
          const int sb = ns % C::kNStg, use = ns / C::kNStg;
          if (!(ok = mbar_wait(stg_full + sb, use & 1, abort))) break;
          const CUtensorMap* map = dst.isv ? &a.map_vst : (dst.isq ? &a.map_qr : &a.map_kr);
          tma_store_4d(map, smem + C::kOffStg + sb * C::kStgBytes, dst.d0, dst.h, m * 128, 0);
          bulk_commit();
          ns++;
          bulk_wait_read<C::kStgLag>();
          if (ns > C::kStgLag) mbar_arrive(stg_free + (ns - 1 - C::kStgLag) % C::kNStg);
        }
      }
      if (!ok) record_timeout(a.status, abort);
      bulk_wait<0>();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    tmem_relinquish();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, int D>
cudaError_t launch_gemm_t(const QkvArgs& a, int grid, cudaStream_t s) {
  using C = QkvCfg<BN>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(k_qkv_gemm<BN, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  k_qkv_gemm<BN, D><<<grid, C::kThreads, C::kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qkv_prep(const QkvArgs& a, cudaStream_t s) {
  const int row_blocks = (a.M + 7) / 8;
  const long long chunks = (long long)a.N * (a.C / 8);
  long long fold = (chunks + 255) / 256;  // one chunk per thread: every load in flight at once
  if (fold < 1) fold = 1;
  if (fold > 16384) fold = 16384;
  k_qkv_prep<<<row_blocks + (int)fold, 256, 0, s>>>(a, row_blocks);
  return cudaGetLastError();
}

// Column-tile width: the BN in {128, 192, 256} whose rounds of tiles over the
// SMs finish first, a round costing BN + 32 columns' worth of time (the 32 a
// per-tile overhead: pipeline fill and the epilogue's tail); ties take the
// narrower tile.
int qkv_pick_bn(int M, int N, int nsm, int* grid) {
  const long long mt = (M + 127) / 128;
  int best = 128;
  long long best_cost = -1;
  for (int bn : {128, 192, 256}) {
    const long long tiles = mt * ((N + bn - 1) / bn);
    const long long rounds = (tiles + nsm - 1) / nsm;
    const long long cost = rounds * (bn + 32);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  const long long tiles = mt * ((N + best - 1) / best);
  *grid = (int)(tiles < nsm ? tiles : nsm);
  return best;
}

cudaError_t launch_qkv_gemm(const QkvArgs& a, int BN, int grid, cudaStream_t s) {
  if (a.D == 64) {
    if (BN == 128) return launch_gemm_t<128, 64>(a, grid, s);
    if (BN == 192) return launch_gemm_t<192, 64>(a, grid, s);
    return launch_gemm_t<256, 64>(a, grid, s);
  }
  if (BN == 128) return launch_gemm_t<128, 32>(a, grid, s);
  if (BN == 192) return launch_gemm_t<192, 32>(a, grid, s);
  return launch_gemm_t<256, 32>(a, grid, s);
}

}  // namespace ne
