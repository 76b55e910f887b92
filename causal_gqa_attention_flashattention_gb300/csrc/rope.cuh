// Rotary position embedding on packed bf16 data, driven by a cos/sin table.
//
// Rotation of pair i of the D-vector at position t (interleaved pairs, the
// original rotary-embedding layout; the NanoEuler pages apply it to queries
// and keys, socker-news README "Architecture"):
//   x'[2i]   = x[2i] cos(t theta_i) - x[2i+1] sin(t theta_i)
//   x'[2i+1] = x[2i] sin(t theta_i) + x[2i+1] cos(t theta_i),  theta_i = base^(-2i/D)
// The inverse (used on gradients) is the transpose: sin -> -sin.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace ne {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Rotates the four pairs held in one 16-byte chunk (8 bf16) by the table
// entries (cos, sin) of four consecutive pairs, in fp32, and returns the
// result rounded to fp16 (`hi`).  If `lo` is given it receives the fp16
// rounding of the remainder (rotated - hi), so hi + lo carries the rotated
// value to about 2^-22 relative.  fp16 keeps 3 more mantissa bits than bf16;
// the rotated operands feed the tensor cores as fp16.
__device__ __forceinline__ uint4 rope_chunk_f16(uint4 x, const float4 cs01, const float4 cs23, uint4* lo) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  const float c[4] = {cs01.x, cs01.z, cs23.x, cs23.z};
  const float s[4] = {cs01.y, cs01.w, cs23.y, cs23.w};
  uint32_t hi[4], lw[4];
#pragma unroll
  for (int p = 0; p < 4; p++) {
    const float x0 = bf_lo(w[p]), x1 = bf_hi(w[p]);
    const float y0 = fmaf(x0, c[p], -x1 * s[p]);
    const float y1 = fmaf(x0, s[p], x1 * c[p]);
    uint32_t h;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(y1), "f"(y0));
    hi[p] = h;
    if (lo) {
      float h0, h1;
      asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
          : "=f"(h0), "=f"(h1)
          : "r"(h));
      uint32_t l;
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(l) : "f"(y1 - h1), "f"(y0 - h0));
      lw[p] = l;
    }
  }
  if (lo) *lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  return make_uint4(hi[0], hi[1], hi[2], hi[3]);
}

// The same rotation left in fp32: y[0..7] for the four pairs of the chunk.
__device__ __forceinline__ void rope_chunk_f32(uint4 x, const float4 cs01, const float4 cs23, float (&y)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  const float c[4] = {cs01.x, cs01.z, cs23.x, cs23.z};
  const float s[4] = {cs01.y, cs01.w, cs23.y, cs23.w};
#pragma unroll
  for (int p = 0; p < 4; p++) {
    const float x0 = bf_lo(w[p]), x1 = bf_hi(w[p]);
    y[2 * p] = fmaf(x0, c[p], -x1 * s[p]);
    y[2 * p + 1] = fmaf(x0, s[p], x1 * c[p]);
  }
}

// Chunk c (pairs 4c..4c+3) of a bf16 row of D values, in the interleaved order
// the rotation works on.  Interleaved rows store it as is.  In the half-split
// layout pair i is (x[i], x[i + D/2]): the chunk gathers x[4c..4c+3] and
// x[D/2 + 4c .. D/2 + 4c + 3] next to each other, so the rotated values come out
// in the interleaved order of a feature permutation, which leaves every q . k
// dot product unchanged.
template <int D>
__device__ __forceinline__ uint4 load_rope_chunk(const __nv_bfloat16* row, int c, bool half) {
  if (!half) return __ldg(reinterpret_cast<const uint4*>(row) + c);
  const uint2 x = __ldg(reinterpret_cast<const uint2*>(row + 4 * c));
  const uint2 y = __ldg(reinterpret_cast<const uint2*>(row + D / 2 + 4 * c));
  return make_uint4(__byte_perm(x.x, y.x, 0x5410), __byte_perm(x.x, y.x, 0x7632), __byte_perm(x.y, y.y, 0x5410),
                    __byte_perm(x.y, y.y, 0x7632));
}

// Loads the (cos, sin) entries for pairs 4c..4c+3 of position `pos`.
template <int D>
__device__ __forceinline__ void rope_coeffs(const float2* tab, int pos, int chunk, float4& a, float4& b) {
  const float4* p = reinterpret_cast<const float4*>(tab + (size_t)pos * (D / 2) + chunk * 4);
  a = __ldg(p);
  b = __ldg(p + 1);
}

}  // namespace ne
