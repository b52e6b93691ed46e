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
//  * the work-item counter to zero;
//  * the int32 dQ accumulator [rows_padded, D] to zero;
//  * per query row, the fixed-point quantum of its dQ partials: qscale =
//    2^k with bound * qscale <= 2^30, where bound = 2 scale max|K|
//    (||dO_i|| max_j ||V_j|| + |D_i|) bounds |dQ_i| and every partial sum of
//    it (|dQ_i| <= scale max|K| sum_j |dS_ij|, sum_j |dS_ij| <= max_j |dP_ij - D_i|,
//    |dP_ij| <= ||dO_i|| ||V_j||; the factor 2 covers rounding), so the int32
//    sums can never overflow.
struct PreExtra {
  int* ticket;
  int* dqacc;
  float* qscale;         // [rows_padded]
  const float2* kvb;     // [B * Hkv]: {max |K|, max_j ||V_j||} of each KV head
  int Hq, Hkv;
  float scale;
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
  constexpr int TPR = D / 16;          // threads per row, 16 bf16 each (two 16-byte loads per tensor)
  constexpr int RPB = 256 / TPR;       // rows per block (blocks of 256 threads)
  // A block holds RPB rows of one (batch, head): one 32-bit division per
  // block index instead of a 64-bit one per thread (which cost about half the
  // kernel's issue slots).
  const int np = (N + TILE - 1) / TILE * TILE;
  const unsigned bph = (unsigned)(np / RPB);  // blocks per (batch, head)
  const unsigned bh = blockIdx.x / bph;
  const int i = (int)(blockIdx.x - bh * bph) * RPB + (int)(threadIdx.x / TPR);
  const int part = (int)(threadIdx.x % TPR);
  const long long row = (long long)bh * np + i;
  const bool real = row < rows_padded && i < N;
  float acc = 0.f, ss = 0.f;  // rowsum(dO * O), ||dO||^2
  if (real) {
    const long long src = (long long)bh * N + i;
    const uint4* ap = reinterpret_cast<const uint4*>(o + src * D) + 2 * part;
    const uint4* gp = reinterpret_cast<const uint4*>(dout + src * D) + 2 * part;
    const uint4 a0 = __ldg(ap), a1 = __ldg(ap + 1), g0 = __ldg(gp), g1 = __ldg(gp + 1);
    const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      acc = fmaf(bf16lo_f32(aw[w]), bf16lo_f32(gw[w]), acc);
      acc = fmaf(bf16hi_f32(aw[w]), bf16hi_f32(gw[w]), acc);
      ss = fmaf(bf16lo_f32(gw[w]), bf16lo_f32(gw[w]), ss);
      ss = fmaf(bf16hi_f32(gw[w]), bf16hi_f32(gw[w]), ss);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) {
    acc += __shfl_xor_sync(0xffffffffu, acc, off);
    ss += __shfl_xor_sync(0xffffffffu, ss, off);
  }
  if (row < rows_padded && part == 0) {
    float l2 = INFINITY;
    if (real) {
      const float v = lse[(long long)bh * N + i];
      l2 = v == -INFINITY ? INFINITY : v * LOG2E;
    }
    rowstat[row] = make_float2(l2, acc);
    if (x.qscale != nullptr) {
      const float2 kv = x.kvb[(bh / x.Hq) * x.Hkv + (bh % x.Hq) / (x.Hq / x.Hkv)];
      const float bound = 2.0f * x.scale * kv.x * (sqrtf(ss) * kv.y + fabsf(acc));
      float q = 1.0f;
      if (bound > 0.f && bound <= 3.0e38f) {
        int ex;
        frexpf(bound, &ex);  // bound < 2^ex
        q = ldexpf(1.0f, 30 - max(ex, -90));
      }
      x.qscale[row] = q;
    }
  }
  if (x.ticket != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *x.ticket = 0;
  if (x.dqacc != nullptr && row < rows_padded) {
    uint4* z = reinterpret_cast<uint4*>(x.dqacc + row * D + part * 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) z[k] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Bounds of the one-kernel backward's fixed-point dQ: per (batch, KV head)
// the largest |K| element and the largest row norm ||V_j||.  A block takes
// KV_BOUND_ROWS consecutive rows of one head (a grid of heads x row chunks),
// reduces them in shared memory and makes one atomic maximum per value on the
// non-negative floats' bits (order independent); kvb must be zero.
constexpr int KV_BOUND_ROWS = 256;
template <int D>
__global__ void __launch_bounds__(256) kv_bound_kernel(const __nv_bfloat16* __restrict__ k,
                                                       const __nv_bfloat16* __restrict__ v,
                                                       float2* __restrict__ kvb, int N, int chunks) {
  constexpr int TPR = D / 8;           // threads per row, 8 bf16 each
  constexpr int RPI = 256 / TPR;       // rows per iteration of the block
  const int head = blockIdx.x / chunks;
  const int r0 = (blockIdx.x % chunks) * KV_BOUND_ROWS;
  const int part = threadIdx.x % TPR;
  float km = 0.f, vn = 0.f;
  for (int rr = threadIdx.x / TPR; rr < KV_BOUND_ROWS; rr += RPI) {
    const int i = r0 + rr;
    float vs = 0.f;
    if (i < N) {
      const long long row = (long long)head * N + i;
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(k + row * D) + part);
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(v + row * D) + part);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        km = fmaxf(km, fmaxf(fabsf(bf16lo_f32(aw[w])), fabsf(bf16hi_f32(aw[w]))));
        vs = fmaf(bf16lo_f32(bw[w]), bf16lo_f32(bw[w]), vs);
        vs = fmaf(bf16hi_f32(bw[w]), bf16hi_f32(bw[w]), vs);
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) vs += __shfl_xor_sync(0xffffffffu, vs, off);
    vn = fmaxf(vn, sqrtf(vs));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, off));
    vn = fmaxf(vn, __shfl_xor_sync(0xffffffffu, vn, off));
  }
  __shared__ float red[2][8];
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = km;
    red[1][threadIdx.x >> 5] = vn;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) {
      km = fmaxf(km, red[0][w]);
      vn = fmaxf(vn, red[1][w]);
    }
    unsigned* dst = reinterpret_cast<unsigned*>(kvb + head);
    atomicMax(dst, __float_as_uint(km));
    atomicMax(dst + 1, __float_as_uint(vn));
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

// D(tmem, 128 x D) (+)= A(128 x 128 keys) B(128 keys x D, MN-major in shared
// memory), A a K-major shared-memory tile.
template <int D>
__device__ __forceinline__ void issue_acc(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, bool first) {
  constexpr uint32_t id = idesc_bf16(128, D, false, true);
  const uint64_t ad = opaque(sdesc_sw128(a_smem, 16, 1024)), bd = opaque(sdesc_sw128(b_smem, 16384, 1024));
#pragma unroll
  for (int kk = 0; kk < TILE / 16; ++kk)
    mma_f16_ss(d_tmem, sdesc_add(ad, (kk / 4) * 16384 + (kk % 4) * 32), sdesc_add(bd, kk * 16 * 128), id,
               (first && kk == 0) ? 0u : 1u);
}

// The same with A packed bf16 in TMEM, written in place over a 128-column
// fp32 tile by the two softmax warpgroups: keys [64 h, 64 h + 64) at TMEM
// columns [64 h, 64 h + 32) of a_tmem, each warpgroup inside the columns it
// read, so neither overwrites values the other has still to load.
template <int D>
__device__ __forceinline__ void issue_acc_inplace(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                                  bool first) {
  constexpr uint32_t id = idesc_bf16(128, D, false, true);
  const uint64_t bd = opaque(sdesc_sw128(b_smem, 16384, 1024));
#pragma unroll
  for (int kk = 0; kk < TILE / 16; ++kk)
    mma_f16_ts(d_tmem, a_tmem + (kk / 4) * 64 + (kk % 4) * 8, sdesc_add(bd, kk * 16 * 128), id,
               (first && kk == 0) ? 0u : 1u);
}

// e4m3 forms for the mixed backward (kind::f8f6f4, 32 keys per MMA, twice the
// bf16 rate).  D(tmem, 128 x 128) = A B^T, A and B e4m3 K-major 128-byte
// swizzled tiles of 128-byte rows (K = 128).
__device__ __forceinline__ void issue_nt_e4m3(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
  constexpr uint32_t id = idesc_e4m3(128, 128, false, false);
  const uint64_t ad = opaque(sdesc_sw128(a_smem, 16, 1024)), bd = opaque(sdesc_sw128(b_smem, 16, 1024));
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_f8_ss(d_tmem, sdesc_add(ad, kk * 32), sdesc_add(bd, kk * 32), id, kk > 0 ? 1u : 0u);
}
// D(tmem, 128 x D) (+)= A(128 x 128 keys, e4m3 K-major) B(128 keys x D, e4m3
// MN-major, 128-byte rows: 32 keys = 4 KB per MMA).
template <int D>
__device__ __forceinline__ void issue_acc_e4m3(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, bool first) {
  constexpr uint32_t id = idesc_e4m3(128, D, false, true);
  const uint64_t ad = opaque(sdesc_sw128(a_smem, 16, 1024)), bd = opaque(sdesc_sw128(b_smem, 16384, 1024));
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_f8_ss(d_tmem, sdesc_add(ad, kk * 32), sdesc_add(bd, kk * 32 * 128), id, (first && kk == 0) ? 0u : 1u);
}

// Store 16 words of e4m3 codes (64 consecutive columns starting at 64 * w)
// of row r into a 128 x 128 e4m3 K-major swizzled tile (128-byte rows).
__device__ __forceinline__ void store_half_row_e4m3(uint8_t* tile, int r, int w, const uint32_t (&v)[16]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t addr = (uint32_t)(r * 128 + (((4 * w + c) ^ (r & 7)) << 4));
    *reinterpret_cast<uint4*>(tile + addr) = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
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

// ------------------------------------------- P^T and dS^T of one KV row
// Constants of one step of a KV-row thread (thread = KV row j, 64 query
// columns c = query rows i0 + c): the score mods in log2 units and the mask
// of a partial tile as a column interval plus, for document ids that are not
// runs, an element-wise id test.
struct KvStep {
  float scale_log2;       // scale * log2(e)
  float sc_in, sc_out;    // soft-cap: scale / c and c * log2(e)
  float al2, al_base;     // ALiBi: slope * log2(e), and slope * log2(e) * (j - i0)
  int lo, hi;             // partial tiles: column c valid iff lo <= c < hi
  const int* doc_cols;    // element-wise document test: ids of query rows i0.., else nullptr
  int doc_j, n_cols;      // this row's id; columns c >= n_cols are past the sequence end
  bool sc, al, partial;
};

// P^T(j, i0 + c) = exp2(x - LSE) for the NC columns c = c0 .. c0 + NC - 1
// (0 where masked), from the scores in s[0 .. NC).  pk: P as packed bf16 (the
// A operand of dV += P^T dO); s: fp32 P times the soft-cap derivative
// 1 - tanh^2 (just P without the cap), kept for dS.  nl2[e] = -LSE * log2(e)
// of query rows i0 + e * 32 + lane, broadcast by shuffles.  fp32 arithmetic
// two lanes per instruction.
template <bool MODS, int NC>
__device__ __forceinline__ void kv_row_p_cols(uint32_t* s, uint32_t* pk, int c0, const float (&nl2)[2],
                                              const KvStep& a) {
  const uint64_t sc_in2 = f2_pack(a.sc_in, a.sc_in), sc_out2 = f2_pack(a.sc_out, a.sc_out);
  const uint64_t one2 = f2_pack(1.f, 1.f);
  const uint64_t al_base2 = f2_pack(a.al_base, a.al_base), nal2 = f2_pack(-a.al2, -a.al2);
  const uint64_t sl2 = f2_pack(a.scale_log2, a.scale_log2);
  const bool sc = MODS && a.sc, al = MODS && a.al;
#pragma unroll
  for (int k = 0; k < NC; k += 2) {
    const int c = c0 + k;  // column (query row i0 + c)
    const uint64_t nl = f2_pack(__shfl_sync(0xffffffffu, nl2[c >> 5], c & 31),
                                __shfl_sync(0xffffffffu, nl2[(c + 1) >> 5], (c + 1) & 31));
    const float s0 = __uint_as_float(s[k]), s1 = __uint_as_float(s[k + 1]);
    uint64_t x2, dmul2 = 0;
    if (sc || al) {
      uint64_t y2 = f2_pack(s0, s1);
      if (sc) {
        const uint64_t t2 = tanh2_exp(f2_mul(y2, sc_in2));
        y2 = f2_mul(t2, sc_out2);
        dmul2 = f2_fma(t2, f2_neg(t2), one2);  // 1 - t^2
      } else {
        y2 = f2_mul(y2, sl2);
      }
      if (al) y2 = f2_fma(f2_pack((float)c, (float)(c + 1)), nal2, f2_add(y2, al_base2));
      x2 = f2_add(y2, nl);
    } else {
      x2 = f2_fma(f2_pack(s0, s1), sl2, nl);
    }
    float x0, x1;
    f2_unpack(x2, x0, x1);
    float pe[2] = {ex2(x0), ex2(x1)};
    if (a.partial) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int cc = c + e;
        bool valid = (cc >= a.lo) && (cc < a.hi);
        if (a.doc_cols != nullptr && valid) valid = (cc < a.n_cols) && (__ldg(a.doc_cols + cc) == a.doc_j);
        if (!valid) pe[e] = 0.f;
      }
    }
    pk[k / 2] = pack_bf16(pe[0], pe[1]);
    if (sc) {
      float q0, q1;
      f2_unpack(f2_mul(f2_pack(pe[0], pe[1]), dmul2), q0, q1);
      s[k] = __float_as_uint(q0);
      s[k + 1] = __float_as_uint(q1);
    } else {
      s[k] = __float_as_uint(pe[0]);
      s[k + 1] = __float_as_uint(pe[1]);
    }
  }
}
template <bool MODS>
__device__ __forceinline__ void kv_row_p(uint32_t (&s)[64], uint32_t (&pk)[32], const float (&nl2)[2],
                                         const KvStep& a) {
  kv_row_p_cols<MODS, 64>(s, pk, 0, nl2, a);
}

// dS^T(j, i0 + c) = P (dP - D) (times the soft-cap derivative) for NC
// columns starting at column c0, packed bf16 into pk; P (times the
// derivative) given as packed bf16, pd[k] holding columns c0 + 2k, c0 + 2k + 1
// (half the registers of fp32); ndd[e] = -D of query rows i0 + e * 32 + lane,
// broadcast by shuffles.
// SCALED: dP is dp * dps (the dequantisation factor of an e4m3 dP).
template <int NC, bool SCALED = false>
__device__ __forceinline__ void kv_row_ds_bf16(const uint32_t* pd, const uint32_t* dp, int c0,
                                               const float (&ndd)[2], uint32_t* pk, float dps = 1.f) {
  const uint64_t dps2 = f2_pack(dps, dps);
#pragma unroll
  for (int k = 0; k < NC; k += 2) {
    const int c = c0 + k;
    const uint64_t nd = f2_pack(__shfl_sync(0xffffffffu, ndd[c >> 5], c & 31),
                                __shfl_sync(0xffffffffu, ndd[(c + 1) >> 5], (c + 1) & 31));
    const uint64_t dp2 = f2_pack(__uint_as_float(dp[k]), __uint_as_float(dp[k + 1]));
    const uint64_t g2 = SCALED ? f2_fma(dp2, dps2, nd) : f2_add(dp2, nd);
    float ds0, ds1;
    f2_unpack(f2_mul(f2_pack(bf16lo_f32(pd[k / 2]), bf16hi_f32(pd[k / 2])), g2), ds0, ds1);
    pk[k / 2] = pack_bf16(ds0, ds1);
  }
}

// Store 16 packed bf16 words (32 consecutive columns, 64 w + 32 h ..) of row
// r into a 128 x 128 bf16 K-major swizzled tile.
__device__ __forceinline__ void store_quarter_row(uint8_t* tile, int r, int w, int h, const uint32_t* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int g = 4 * h + q;
    const uint32_t addr = (uint32_t)(w * 16384 + r * 128 + ((g ^ (r & 7)) << 4));
    *reinterpret_cast<uint4*>(tile + addr) = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
}

constexpr int BWD_LAUNCH_REGS = 168, BWD_REGS_LOW = 80, BWD_REGS_HIGH = 208;
static_assert(128 * BWD_REGS_LOW + 256 * BWD_REGS_HIGH <= 384 * BWD_LAUNCH_REGS, "register split");

// The register split inside the backward kernels assumes exactly this many
// registers per thread at launch; refuse to launch any other build.
template <typename K>
static inline cudaError_t check_regs(K kern, int& cached, int expected = BWD_LAUNCH_REGS) {
  if (cached < 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return cudaErrorInvalidDeviceFunction;
    cached = fa.numRegs;
  }
  // The register split inside the kernel assumes this allocation at launch.
  return cached == expected ? cudaSuccess : cudaErrorInvalidConfiguration;
}

}  // namespace attn
