// Row-wise softmax pieces shared by the forward and decode kernels: one
// thread owns one 128-column row of scores held in registers.
#pragma once
#include "common.cuh"

namespace attn {

// Maximum of a 128-column row: eight independent chains of three-input max.
__device__ __forceinline__ float row_max128(const uint32_t (&s)[128]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1]));
#pragma unroll
  for (int c = 16; c < 128; c += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k)
      m[k] = max3(m[k], __uint_as_float(s[c + 2 * k]), __uint_as_float(s[c + 2 * k + 1]));
  return max3(max3(m[0], m[1], m[2]), max3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// Row sum of four packed partial sums.
__device__ __forceinline__ float sum_acc(const uint64_t (&acc)[4]) {
  float a0, a1, b0, b1, c0, c1, d0, d1;
  f2_unpack(acc[0], a0, a1);
  f2_unpack(acc[1], b0, b1);
  f2_unpack(acc[2], c0, c1);
  f2_unpack(acc[3], d0, d1);
  return ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
}

// P = 2^(mul * s - mu) for the 128 columns of this thread's row (mul folds
// the softmax scale in; 1 when s already holds log2-unit logits), as packed
// bf16 written in place into s[0..63] (s[k] = columns 2k, 2k+1; step k reads
// only s[2k], s[2k+1], so no unread score is overwritten) and, with LO, the
// rounding residual p - bf16(p) in lo[0..63].  Returns the row sum of P.
template <bool LO>
__device__ __forceinline__ float exp_bf16(uint32_t (&s)[128], uint32_t (&lo)[64], float mul, float mu) {
  const uint64_t mul2 = f2_pack(mul, mul), nmu2 = f2_pack(-mu, -mu);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int k = 0; k < 64; ++k) {
    float y0, y1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * k]), __uint_as_float(s[2 * k + 1])), mul2, nmu2), y0, y1);
    const float p0 = ex2(y0), p1 = ex2(y1);
    acc[k & 3] = f2_add(acc[k & 3], f2_pack(p0, p1));
    const uint32_t hi = pack_bf16(p0, p1);
    s[k] = hi;
    if (LO) lo[k] = pack_bf16(p0 - bf16lo_f32(hi), p1 - bf16hi_f32(hi));
  }
  return sum_acc(acc);
}

}  // namespace attn
