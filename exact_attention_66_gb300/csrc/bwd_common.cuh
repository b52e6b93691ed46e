// Pieces shared by the backward kernels (bwd.cu, bwd_fused.cu): MMA issue
// sequences over 128-byte swizzled shared-memory tiles, TMEM <-> register
// and shared-memory moves, and the register split of their warpgroups.
#pragma once
#include <cuda_runtime.h>
#include "common.cuh"

namespace attn {

// ------------------------------------------------------------------ bwd_pre
// Extra duties of the pre kernel for the one-kernel backward (bwd_fused.cu);
// all null for the two-kernel backward.
struct PreExtra {
  int* flags;              // dQ ordering flags to zero, n_flags of them
  long long n_flags;
  int* ticket;             // work-item counter to zero
  const int2* row_range;   // with a block map: rows of Q tiles whose range is
  int Hq, nT;              // empty get dQ = 0 here (no KV tile ever adds to them)
  __nv_bfloat16* dq;
};

// Row statistics of the backward, one pair per query row, rows padded to whole
// 128-row tiles: {LSE * log2(e), D = rowsum(dO * O)}.  Padding rows and rows
// with no allowed key get +inf (so that P = exp2(x - inf) = 0) and D = 0.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const float* __restrict__ lse,
                                                      float2* __restrict__ rowstat, int N,
                                                      long long rows_padded, const PreExtra x) {
  constexpr int TPR = D / 8;  // threads per row, 8 bf16 each
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gt / TPR;
  const int part = (int)(gt % TPR);
  const long long np = (long long)((N + TILE - 1) / TILE) * TILE;
  const long long bh = row / np;
  const int i = (int)(row - bh * np);
  const bool real = row < rows_padded && i < N;
  float acc = 0.f;
  if (real) {
    const long long src = bh * N + i;
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + src * D) + part);
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(dout + src * D) + part);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      acc = fmaf(bf16lo_f32(aw[w]), bf16lo_f32(gw[w]), acc);
      acc = fmaf(bf16hi_f32(aw[w]), bf16hi_f32(gw[w]), acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows_padded && part == 0) {
    float l2 = INFINITY;
    if (real) {
      const float v = lse[bh * N + i];
      l2 = v == -INFINITY ? INFINITY : v * LOG2E;
    }
    rowstat[row] = make_float2(l2, acc);
  }
  if (x.flags != nullptr && gt < x.n_flags) x.flags[gt] = 0;
  if (x.ticket != nullptr && gt == 0) *x.ticket = 0;
  if (x.row_range != nullptr && real) {
    const int2 r = x.row_range[(bh / x.Hq) * x.nT + i / TILE];
    if (r.x >= r.y) reinterpret_cast<uint4*>(x.dq + (bh * N + i) * D)[part] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// D(tmem, 128 x 128) = A B^T, A and B K-major 128-byte swizzled tiles of
// ROW_BYTES per row (16 KB column chunks), one MMA per 32 bytes of a row.
// Issue loops are unrolled: the tensor pipe queues few MMAs, and a rolled
// loop's per-iteration overhead in the issuing thread leaves it idle.
template <int ROW_BYTES>
__device__ __forceinline__ void issue_nt(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, false);
  const uint64_t ad = opaque(sdesc_sw128(a_smem, 16, 1024)), bd = opaque(sdesc_sw128(b_smem, 16, 1024));
#pragma unroll
  for (int kk = 0; kk < ROW_BYTES / 32; ++kk) {
    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
    mma_f16_ss(d_tmem, sdesc_add(ad, off), sdesc_add(bd, off), id, kk > 0 ? 1u : 0u);
  }
}

// D(tmem, 128 x 128) = A B^T with A packed bf16 in TMEM (128 lanes x D
// elements, D / 2 columns) and B a K-major shared-memory tile.
template <int D>
__device__ __forceinline__ void issue_nt_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, false);
  const uint64_t bd = opaque(sdesc_sw128(b_smem, 16, 1024));
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    mma_f16_ts(d_tmem, a_tmem + kk * 8, sdesc_add(bd, (kk / 4) * 16384 + (kk % 4) * 32), id,
               kk > 0 ? 1u : 0u);
}

// Copy row r of a K-major 128-byte swizzled bf16 tile (D elements per row)
// into this warp's TMEM lanes as packed bf16 (A-operand layout).
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t* tile, int r, uint32_t t_addr) {
#pragma unroll
  for (int q4 = 0; q4 < D / 64; ++q4) {  // 32 words = 64 elements = one 128-byte chunk row
    uint32_t v[32];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint4 x = *reinterpret_cast<const uint4*>(tile + q4 * 16384 + r * 128 + ((g ^ (r & 7)) << 4));
      v[4 * g] = x.x;
      v[4 * g + 1] = x.y;
      v[4 * g + 2] = x.z;
      v[4 * g + 3] = x.w;
    }
    tmem_st32(t_addr + q4 * 32, v);
  }
}

// D(tmem, 128 x D) += A(128 x 128 keys) B(128 keys x D, MN-major in shared
// memory).  A is a K-major shared-memory tile (A_TMEM false; a_tmem ignored)
// or packed bf16 in TMEM (A_TMEM true; a_smem ignored).
template <int D, bool A_TMEM>
__device__ __forceinline__ void issue_acc(uint32_t d_tmem, uint32_t a_smem, uint32_t a_tmem,
                                          uint32_t b_smem, bool first) {
  constexpr uint32_t id = idesc_bf16(128, D, false, true);
  const uint64_t ad = opaque(sdesc_sw128(a_smem, 16, 1024)), bd = opaque(sdesc_sw128(b_smem, 16384, 1024));
#pragma unroll
  for (int kk = 0; kk < TILE / 16; ++kk) {
    const uint32_t acc = (first && kk == 0) ? 0u : 1u;
    const uint64_t b = sdesc_add(bd, kk * 16 * 128);
    if (A_TMEM)
      mma_f16_ts(d_tmem, a_tmem + kk * 8, b, id, acc);
    else
      mma_f16_ss(d_tmem, sdesc_add(ad, (kk / 4) * 16384 + (kk % 4) * 32), b, id, acc);
  }
}

// Store 32 packed bf16 words (64 consecutive columns starting at 64 * w) of
// row r into a 128 x 128 bf16 K-major swizzled tile.
__device__ __forceinline__ void store_half_row(uint8_t* tile, int r, int w, const uint32_t (&v)[32]) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint32_t addr = (uint32_t)(w * 16384 + r * 128 + ((g ^ (r & 7)) << 4));
    *reinterpret_cast<uint4*>(tile + addr) = make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
  }
}

// Columns [col0, col0 + NC) of an fp32 TMEM row (NC a multiple of 32) as
// bf16 * mul into dst (global), if in range; zeros when the accumulator was
// never written.
template <int NC>
__device__ __forceinline__ void store_cols(uint32_t t_col, bool have, float mul, __nv_bfloat16* dst,
                                           bool in_range) {
#pragma unroll
  for (int q4 = 0; q4 < NC / 32; ++q4) {
    uint32_t v[32];
    if (have) {
      tmem_ld32(t_col + q4 * 32, v);
      tmem_wait_ld(v);
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) v[c] = 0u;
    }
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 16; ++k)
      pk[k] = pack_bf16(__uint_as_float(v[2 * k]) * mul, __uint_as_float(v[2 * k + 1]) * mul);
    if (in_range) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + q4 * 32);
#pragma unroll
      for (int k = 0; k < 4; ++k) d4[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
    }
  }
}

// Load 64 consecutive fp32 TMEM columns of this warp's lanes.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
}
__device__ __forceinline__ void tmem_wait64(uint32_t (&v)[64]) {
  tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&v[0]));
  tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&v[32]));
}

constexpr int BWD_LAUNCH_REGS = 168, BWD_REGS_LOW = 80, BWD_REGS_HIGH = 208;
static_assert(128 * BWD_REGS_LOW + 256 * BWD_REGS_HIGH <= 384 * BWD_LAUNCH_REGS, "register split");

// The register split inside the backward kernels assumes exactly this many
// registers per thread at launch; refuse to launch any other build.
template <typename K>
static inline cudaError_t check_regs(K kern, int& cached) {
  if (cached < 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return cudaErrorInvalidDeviceFunction;
    cached = fa.numRegs;
  }
  // The register split inside the kernel assumes this allocation at launch.
  return cached == BWD_LAUNCH_REGS ? cudaSuccess : cudaErrorInvalidConfiguration;
}

}  // namespace attn
