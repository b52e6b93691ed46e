// FP8 prologue: signed Hadamard rotation of Q and K rows, per-(batch, head)
// amax, e4m3 quantisation of Q, K and V.
//
// FlashAttention-3 digest, "Basse précision FP8 et incoherent processing":
// queries and keys are multiplied by a random orthogonal matrix -- a Hadamard
// transform with random signs, applied per head in O(d log d) -- to spread
// outliers before FP8 quantisation; the transform is memory-bandwidth bound.
// Here each row x (d = 128) becomes (x * s) H / sqrt(128), H the natural-order
// Sylvester Hadamard matrix and s the +-1 vector of the row's KV head, so
// (q M)(k M)^T = q k^T exactly in real arithmetic; V is not rotated.
//
// Two bandwidth-bound passes over Q, K, V (one warp per 128-element row, each
// lane holding four consecutive elements; butterflies of distance 1 and 2 in
// registers, 4..64 through warp shuffles): pass 1 finds the amax of every
// (batch, head) of the rotated tensors (integer atomic max of the non-negative
// float bits, so the result does not depend on the order), pass 2 recomputes
// the rotation and writes e4m3 codes scaled by 448 / amax.
//
// Optionally RoPE is fused in front of the rotation (the digest's "fused with
// RoPE at no extra cost"): the row at position n of its head has its element
// pairs (c, c + 64) turned by n * base^(-2c/128) before the signs and the
// Hadamard butterflies, in the same registers -- lane l pairs with lane
// l ^ 16 -- so RoPE costs no extra pass over memory.
#include "common.cuh"
#include "launch.h"

namespace attn {

struct QuantTensors {
  const __nv_bfloat16* x[3];  // Q, K, V
  uint8_t* out[3];            // e4m3 codes
  long long rows[3];          // B * H * N
  int heads[3];               // H of each tensor
  unsigned* amax[3];          // [B * H] float bits (workspace)
  float* scale[3];            // [B * H] dequantisation scales (output)
  const int8_t* signs;        // [Hkv, 128] or nullptr
  float rope_k;               // RoPE: inv_freq(c) = exp2(-c * rope_k), rope_k = 2 log2(base) / 128; 0 = off
  int N, Hkv, G;              // G = Hq / Hkv
};

constexpr int ROWS_PER_WARP = 16;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Rotated (or plain) row values of this lane: elements 4 * lane .. 4 * lane + 3.
__device__ __forceinline__ void load_row(const QuantTensors& t, int ti, long long row, float (&v)[4]) {
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(t.x[ti] + row * 128) + lane_id());
  v[0] = bf16lo_f32(raw.x);
  v[1] = bf16hi_f32(raw.x);
  v[2] = bf16lo_f32(raw.y);
  v[3] = bf16hi_f32(raw.y);
  if (ti == 2) return;
  if (t.rope_k != 0.f) {  // RoPE on Q and K rows, rotate-half pairs (c, c + 64)
    const int lane = lane_id();
    const float pos = (float)(row % t.N);
    const bool first = lane < 16;  // elements 4 lane .. 4 lane + 3 < 64
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float partner = __shfl_xor_sync(0xffffffffu, v[r], 16);
      const int c = (4 * lane + r) & 63;
      float sn, cs;
      sincosf(pos * exp2f(-(float)c * t.rope_k), &sn, &cs);
      v[r] = first ? fmaf(v[r], cs, -partner * sn) : fmaf(v[r], cs, partner * sn);
    }
  }
  if (t.signs == nullptr) return;
  const int head = (int)((row / t.N) % t.heads[ti]);
  const int hk = ti == 0 ? head / t.G : head;
  const char4 sg = __ldg(reinterpret_cast<const char4*>(t.signs + hk * 128) + lane_id());
  v[0] *= (float)sg.x;
  v[1] *= (float)sg.y;
  v[2] *= (float)sg.z;
  v[3] *= (float)sg.w;
  // Walsh-Hadamard butterflies: (a, b) -> (a + b, a - b) for index pairs j, j ^ h.
  float a = v[0], b = v[1];
  v[0] = a + b;
  v[1] = a - b;
  a = v[2];
  b = v[3];
  v[2] = a + b;
  v[3] = a - b;
  a = v[0];
  b = v[2];
  v[0] = a + b;
  v[2] = a - b;
  a = v[1];
  b = v[3];
  v[1] = a + b;
  v[3] = a - b;
  const int lane = lane_id();
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float other = __shfl_xor_sync(0xffffffffu, v[r], m);
      v[r] = (lane & m) ? (other - v[r]) : (v[r] + other);
    }
  }
  const float norm = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int r = 0; r < 4; ++r) v[r] *= norm;
}

__global__ void __launch_bounds__(256) quant_amax_kernel(const QuantTensors t) {
  const int ti = blockIdx.y;
  const long long warp_g = (long long)blockIdx.x * 8 + warp_id();
  const long long r0 = warp_g * ROWS_PER_WARP;
  if (r0 >= t.rows[ti]) return;
  const long long r1 = min(r0 + ROWS_PER_WARP, t.rows[ti]);
  long long cur_bh = r0 / t.N;
  float mx = 0.f;
  for (long long row = r0; row < r1; ++row) {
    const long long bh = row / t.N;
    if (bh != cur_bh) {  // the warp's rows crossed into the next head: flush
      const float red = warp_max(mx);
      if (lane_id() == 0) atomicMax(t.amax[ti] + cur_bh, __float_as_uint(red));
      cur_bh = bh;
      mx = 0.f;
    }
    float v[4];
    load_row(t, ti, row, v);
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
  }
  mx = warp_max(mx);
  if (lane_id() == 0) atomicMax(t.amax[ti] + cur_bh, __float_as_uint(mx));
}

__global__ void quant_scale_kernel(const QuantTensors t, int B) {
  const int ti = blockIdx.y;
  const int n = B * t.heads[ti];
  for (int i = threadIdx.x + blockIdx.x * blockDim.x; i < n; i += blockDim.x * gridDim.x) {
    const float a = __uint_as_float(t.amax[ti][i]);
    t.scale[ti][i] = a > 0.f ? a / 448.0f : 1.0f;
  }
}

__global__ void __launch_bounds__(256) quant_write_kernel(const QuantTensors t) {
  const int ti = blockIdx.y;
  const long long warp_g = (long long)blockIdx.x * 8 + warp_id();
  const long long r0 = warp_g * ROWS_PER_WARP;
  if (r0 >= t.rows[ti]) return;
  const long long r1 = min(r0 + ROWS_PER_WARP, t.rows[ti]);
  for (long long row = r0; row < r1; ++row) {
    const float a = __uint_as_float(t.amax[ti][row / t.N]);
    const float inv = a > 0.f ? 448.0f / a : 1.0f;
    float v[4];
    load_row(t, ti, row, v);
    reinterpret_cast<uint32_t*>(t.out[ti] + row * 128)[lane_id()] =
        pack_e4m3x4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
  }
}

cudaError_t launch_hadamard_quant(const void* q, const void* k, const void* v, void* q8, void* k8,
                                  void* v8, float* scales, const int8_t* signs, int B, int Hq,
                                  int Hkv, int N, float rope_base, unsigned* amax_ws, cudaStream_t st) {
  QuantTensors t{};
  t.rope_k = rope_base > 0.f ? 2.0f * log2f(rope_base) / 128.0f : 0.f;
  t.x[0] = (const __nv_bfloat16*)q;
  t.x[1] = (const __nv_bfloat16*)k;
  t.x[2] = (const __nv_bfloat16*)v;
  t.out[0] = (uint8_t*)q8;
  t.out[1] = (uint8_t*)k8;
  t.out[2] = (uint8_t*)v8;
  t.heads[0] = Hq;
  t.heads[1] = t.heads[2] = Hkv;
  for (int i = 0; i < 3; ++i) t.rows[i] = (long long)B * t.heads[i] * N;
  t.amax[0] = amax_ws;
  t.amax[1] = amax_ws + B * Hq;
  t.amax[2] = amax_ws + B * Hq + B * Hkv;
  t.scale[0] = scales;
  t.scale[1] = scales + B * Hq;
  t.scale[2] = scales + B * Hq + B * Hkv;
  t.signs = signs;
  t.N = N;
  t.Hkv = Hkv;
  t.G = Hq / Hkv;
  cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(unsigned) * (size_t)(B * Hq + 2 * B * Hkv), st);
  if (e != cudaSuccess) return e;
  const long long warps = (t.rows[0] + ROWS_PER_WARP - 1) / ROWS_PER_WARP;
  const dim3 grid((unsigned)((warps + 7) / 8), 3);
  quant_amax_kernel<<<grid, 256, 0, st>>>(t);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  quant_scale_kernel<<<dim3(1, 3), 256, 0, st>>>(t, B);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  quant_write_kernel<<<grid, 256, 0, st>>>(t);
  return cudaGetLastError();
}

}  // namespace attn
