// Integer dot products of 4-bit codes with int16 activations, shared by the
// decode kernel and the attention projections.  A repacked code word (see
// internal.h) holds columns 8w..8w+3 in its low nibbles and 8w+4..8w+7 in
// its high nibbles; activations are int16 X = rint(v * 32767 / max|v|).
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace moe {

// Integer dot product of one 32-column chunk: the chunk's 16 code bytes
// (byte i of word j = column 8j+i in the low nibble, column 8j+4+i in the
// high nibble) against the int16 activation chunk x (x[j] = columns 8j..8j+7
// as four int16 pairs).  Exact in int32; two chains per nibble half.
__device__ __forceinline__ int idot_chunk(const uint4& w, const uint4 (&x)[4]) {
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
  int lo_acc[2] = {0, 0}, hi_acc[2] = {0, 0};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = words[j] & 0x0F0F0F0Fu;  // codes of columns 8j+0..3
    const uint32_t hi = words[j] & 0xF0F0F0F0u;  // 16 x codes of columns 8j+4..7
    lo_acc[j & 1] = dp2a_lo(x[j].x, lo, lo_acc[j & 1]);
    lo_acc[j & 1] = dp2a_hi(x[j].y, lo, lo_acc[j & 1]);
    hi_acc[j & 1] = dp2a_lo(x[j].z, hi, hi_acc[j & 1]);
    hi_acc[j & 1] = dp2a_hi(x[j].w, hi, hi_acc[j & 1]);
  }
  return (lo_acc[0] + lo_acc[1]) + ((hi_acc[0] + hi_acc[1]) >> 4);
}

// Sum of the int16 pairs of a uint4 (8 values, exact).
__device__ __forceinline__ int sum8_s16(const uint4& q) {
  int s = dp2a_lo(q.x, 0x01010101u, 0);
  s = dp2a_lo(q.y, 0x01010101u, s);
  s = dp2a_lo(q.z, 0x01010101u, s);
  return dp2a_lo(q.w, 0x01010101u, s);
}

// int16 quantisation factor for a vector with max |v| = m: X = rint(v * q).
__device__ __forceinline__ float quant_factor(float m) { return m > 0.f ? 32767.f / m : 0.f; }

__device__ __forceinline__ uint32_t pack_s16x2(float a, float b) {
  const int ia = __float2int_rn(a), ib = __float2int_rn(b);
  return (static_cast<uint32_t>(ia) & 0xffffu) | (static_cast<uint32_t>(ib) << 16);
}

}  // namespace moe
