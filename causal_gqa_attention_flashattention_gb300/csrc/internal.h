// Internal interfaces between the C-ABI layer (api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace ne {

constexpr int kTile = 128;  // query rows / key rows per tile

// Device-side status codes (mirror ne_status in include/ne_attn.h).
constexpr int kStatusTimeout = -6;

// Flag bits shared with include/ne_attn.h.
constexpr int kFlagOFp32 = 1;      // o is float32
constexpr int kFlagGradFp32 = 2;   // dq, dk, dv are float32
constexpr int kFlagPreciseQK = 4;  // logits from hi + lo fp16 parts of rotated q and k
constexpr int kFlagQKRotated = 8;  // backward: the workspace already holds the forward's rotated q and k
constexpr int kFlagRopeHalf = 16;  // RoPE pairs (x[i], x[i + D/2]) instead of (x[2i], x[2i+1])
constexpr int kFlagFp8 = 32;       // forward: rotated q, k as e4m3 with per-head scales

// Largest number of query heads one forward CTA handles (TMEM/smem budget).
inline int fwd_max_heads(int D, bool precise) { return D == 64 ? (precise ? 3 : 4) : 8; }

struct FwdArgs {
  // 4-D tiled maps over [B, T, H, D], box D x 1 x 128 x 1.  Default precision:
  // map_q / map_k cover the rotated fp16 copies in the workspace (e4m3 with
  // FP8); precise logits: the bf16 inputs (the kernel rotates them itself).
  CUtensorMap map_q, map_k, map_v;
  CUtensorMap map_o;                // store map over o (default precision): 128-byte (or 64-byte) column boxes x 32 rows
  void* o;                          // [B, T, Hq, D] bf16 or fp32
  float* lse;                       // [B, Hq, T]
  float* lse_lo;                    // [B, Hq, T] fp32 remainder of lse (precise logits only)
  const float2* rope;               // [Tcap][D/2] (cos, sin)
  int* status;                      // device status word
  int B, T, Hq, Hkv, D, G, HC;      // HC: query heads per CTA (divides G; precise-logits kernel)
  int nt;                           // number of 128-row tiles
  int o_fp32;
  float scale_log2;                 // log2(e) / sqrt(D), rounded to fp32
  float scale_log2_lo;              // remainder log2(e)/sqrt(D) - scale_log2
  const float* qk_amax;             // FP8 forward: per-head max |rotated value|, [Hq] for q then [Hkv] for k
  const int* sched;                 // [grid, sched_k] int4 work items of each CTA (b = -1: none), see fwd_pair_schedule
  int sched_k;
  int grid;                         // CTAs of the persistent forward
};

// Division of a non-negative 32-bit n < 2^31 by a runtime divisor d >= 1 with
// a multiply-high and a shift (round-up magic number):
//   l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(n, m) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) l++;
  const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
  return FastDiv{d, (uint32_t)m, l};
}

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) { return (__umulhi(n, f.m) + n) >> f.l; }
#endif

// RoPE pre-pass of the forward: q, k (bf16) -> rotated fp16 copies qr, kr.
struct RopeArgs {
  const __nv_bfloat16 *q, *k;
  __half *qr, *kr;
  const float2* rope;
  int B, T, Hq, Hkv;
  int rope_half;  // half-split pair layout of q and k
  FastDiv div_hq, div_hkv, div_t;
  FastDiv div_hg;    // by the groups of four heads (Hq + Hkv, four per thread) of k_rope_qk
  uint8_t *q8, *k8;  // FP8 forward: rotated q, k as e4m3 scaled by 448 / max |value| of their head
  float* amax;       // FP8 forward: [Hq + Hkv] per-head max |rotated value| (zeroed before the max pass)
};

struct BwdArgs {
  CUtensorMap map_qr, map_kr, map_v, map_do;  // 4-D maps as above (qr/kr: rotated fp16 copies)
  CUtensorMap map_qlo, map_klo;               // fp16 remainders (precise logits only)
  CUtensorMap map_dqacc;                      // 2-D map over [B*Hq*Tp, D] fp32, box 32 x 128
  CUtensorMap map_dk, map_dv;                 // 4-D store maps over [B, T, Hkv, D] (fp32 or bf16), box
                                              // 128 bytes of columns x 1 x 128 rows x 1, same swizzle span
  const float* lse2;                          // [B, Hq, Tp]  lse * log2(e); +inf on pad rows
  const float* lse2_lo;                       // [B, Hq, Tp]  its fp32 remainder (precise logits only)
  const float* delta;                         // [B, Hq, Tp]
  void* dk;                                   // [B, T, Hkv, D] bf16 or fp32
  void* dv;
  const float2* rope;
  int* status;
  int B, T, Hq, Hkv, D, G, nt, Tp;
  int grad_fp32;
  int rope_half;  // dk leaves in the half-split pair layout
  float scale_log2, scale_log2_lo, scale;
};

struct PrepArgs {
  const __nv_bfloat16 *q, *k, *dout;
  const void* o;  // bf16 or fp32
  const float* lse;
  const float* lse_lo;          // null unless precise logits
  __half *qr, *kr, *qlo, *klo;  // qlo/klo null unless precise logits
  float *lse2, *lse2_lo, *delta, *dqacc;
  const float2* rope;
  int B, T, Hq, Hkv, D, Tp, o_fp32;
  int rotate_qk;                            // 0: qr / kr already hold the rotated q and k
  int rope_half;                            // half-split pair layout of q and k
  int negate;                               // 1: store -lse * log2(e) and -Delta (default-precision sweep)
  FastDiv div_hq, div_hkv, div_t, div_pad;  // by Hq, Hkv, T and Tp - T (pad rows; d = 1 if none)
};

struct DqArgs {
  const float* dqacc;  // [B, Hq, Tp, D]
  void* dq;            // [B, T, Hq, D]
  const float2* rope;
  int B, T, Hq, D, Tp, grad_fp32;
  int rope_half;  // dq leaves in the half-split pair layout
  float scale;
  FastDiv div_hq, div_t;
  FastDiv div_hg;  // by the groups of four query heads (four per thread)
};

// Key/value cache append: rotated keys (fp16) and values (bf16) of Tn new positions.
struct KvAppendArgs {
  const __nv_bfloat16 *k, *v;  // [B, Tn, Hkv, D]
  __half* kc;                  // [B, Hkv, Tcap, D] rotated keys
  __nv_bfloat16* vc;           // [B, Hkv, Tcap, D]
  const float2* rope;
  int B, Tn, Hkv, Tcap, pos0;
  int rope_half;  // half-split pair layout of the new keys
  FastDiv div_hkv, div_tn;
};

// Decode over a key/value cache (see attn_decode.cu).
struct DecodeArgs {
  CUtensorMap map_q;         // packed rotated queries [B*Hkv*128, D] fp16 (4-D map, box D x 1 x 128 x 1)
  CUtensorMap map_k, map_v;  // caches [B, Hkv, Tkv valid of Tcap, D] (fp16 keys, bf16 values)
  const __nv_bfloat16* q;    // [B, Tq, Hq, D]
  __half* qpk;               // [B, Hkv, 128, D] packed rotated queries (workspace)
  float* part_o;             // [B, Hkv, nsplit, F, R, D] unnormalised O per split and copy (workspace)
  float* part_ml;            // [B, Hkv, nsplit, F, R] (max in log2 units, sum) pairs (workspace)
  unsigned* done;            // [B * Hkv] finished splits per group (workspace; zeroed by the query pass)
  void* o;                   // [B, Tq, Hq, D] bf16 or fp32
  float* lse;                // [B, Hq, Tq]
  const float2* rope;
  int* status;
  int B, Tq, Tkv, Hq, Hkv, D, G, R, ntk, nsplit, o_fp32;
  int F;                     // copies of the R query rows in the 128-row tile: 4 if R <= 32, 2 if R <= 64, else 1
  int rope_half;             // half-split pair layout of q (and of the cached keys)
  float scale_log2;
};

// RMSNorm + fused Q/K/V projection (see qkv_proj.cu).  Rows r = b * T + t of
// x [M, C]; projection features n of w_qkv [N, C], N = (Hq + 2 Hkv) D.
struct QkvArgs {
  CUtensorMap map_x;              // x [M, C] bf16, box 64 x 128, 128-byte swizzle
  CUtensorMap map_w;              // folded weight [N, C] bf16, box 64 x BN, 128-byte swizzle
  CUtensorMap map_qr, map_kr;     // store maps over the rotated fp16 q [M, Hq, D], k [M, Hkv, D]
  CUtensorMap map_vst;            // store map over v [M, Hkv, D] bf16 (boxes 32 x 1 x 128, 64-byte swizzle)
  const __nv_bfloat16* x;         // [M, C]
  const __nv_bfloat16* norm_w;    // [C]
  const __nv_bfloat16* w;         // [N, C]
  __nv_bfloat16* wf;              // [N, C] w_qkv[n', c] * norm_w[c], rows permuted for half-split q, k
  float* rstd;                    // [M]
  __nv_bfloat16 *q, *k, *v;       // [M, Hq, D], [M, Hkv, D], [M, Hkv, D] (q and k may be null)
  __half *qr, *kr;                // rotated fp16 q and k (null: not written)
  const float2* rope;
  int* status;
  int M, C, N, T, Hq, Hkv, D;
  int nkb, ntn, tiles;            // 64-wide K blocks, BN-wide column tiles, 128 x BN tiles
  int rope_half;
  float eps;
};

cudaError_t launch_qkv_prep(const QkvArgs& a, cudaStream_t s);
cudaError_t launch_qkv_gemm(const QkvArgs& a, int BN, int grid, cudaStream_t s);
int qkv_pick_bn(int M, int N, int nsm, int* grid);

cudaError_t launch_fwd(const FwdArgs& a, bool precise, cudaStream_t s);
cudaError_t launch_kv_append(const KvAppendArgs& a, int D, cudaStream_t s);
cudaError_t launch_decode_q(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, int nsm, cudaStream_t s);
cudaError_t launch_rope_qk(const RopeArgs& a, int D, cudaStream_t s);
cudaError_t launch_rope_amax(const RopeArgs& a, cudaStream_t s);  // D = 64
cudaError_t launch_rope_q8(const RopeArgs& a, cudaStream_t s);    // D = 64
cudaError_t launch_fwd_fp8(const FwdArgs& a, cudaStream_t s);      // D = 64
cudaError_t launch_bwd_prep(const PrepArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dkdv(const BwdArgs& a, bool precise, cudaStream_t s);
cudaError_t launch_bwd_dq(const DqArgs& a, cudaStream_t s);
cudaError_t launch_rope_table(float2* tab, int Tcap, int D, double base, cudaStream_t s);
cudaError_t launch_timeout_probe(int* status, long long limit_ns, cudaStream_t s);

}  // namespace ne
