// Backward pass of exact tiled attention for sm_103a: dQ, dK, dV from Q, K, V,
// O, dO and the forward's LSE, recomputing P tile by tile instead of storing it
// (FlashAttention-3 digest, "Rappel du fonctionnement de FlashAttention":
// tiling and recomputation).  Formulas (the pages state none; textbook
// calculus of the forward):
//   P = exp(x - LSE),  dP = dO V^T,  D = rowsum(dO * O) = rowsum(P * dP),
//   dX = P (dP - D),   dZ = dX * (1 - tanh^2(z/c)) with the soft-cap, else dX,
//   dQ = scale dZ K,   dK = scale dZ^T Q,   dV = P^T dO.
//
// Three kernels:
//  * bwd_pre:  D = rowsum(dO * O) per query row (bandwidth bound).
//  * bwd_dkdv: one CTA per (batch, KV head, 128-row KV tile).  K_J and V_J stay
//    in shared memory; Q/dO tiles of every query head of the GQA group and
//    every needed Q tile stream through a 2-stage TMA ring.  S^T = K Q^T and
//    dP^T = V dO^T land in TMEM; two softmax warpgroups (a thread per KV row,
//    64 query columns each) turn them into P^T (bf16, to shared memory) and
//    dS^T (bf16, written back over dP^T in TMEM); dV += P^T dO reads P^T from
//    shared memory, dK += dS^T Q reads dS^T from TMEM.
//  * bwd_dq:   one CTA per (batch, query head, 128-row Q tile), streaming K/V
//    tiles: S = Q K^T and dP = dO V^T in TMEM, dS to shared memory,
//    dQ += dS K.
// As in the forward, the softmax copies S / dP to registers and hands the TMEM
// columns back at once, so the next tile's GEMMs run while it computes, and two
// threads issue the MMAs of independent chains (the tensor pipe queues few
// MMAs, so a single issuer that waits on a barrier would leave it idle).
// Each dQ, dK, dV tile is accumulated by exactly one CTA, in TMEM, over its
// partner tiles in a fixed order: no atomics, so the result is bitwise
// reproducible (contrast the nondeterministic block-sparse backward on the
// FlexAttention/FA4 page, "Limitations actuelles").
#include "common.cuh"
#include "launch.h"

namespace attn {

// ------------------------------------------------------------------ bwd_pre
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      float* __restrict__ delta, long long rows) {
  constexpr int TPR = D / 8;  // threads per row, 8 bf16 each
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gt / TPR;
  const int part = (int)(gt % TPR);
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + part);
    const uint4 g = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + part);
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
  if (row < rows && part == 0) delta[row] = acc;
}

// log2-unit LSE of a row; +inf (so that P = 0) past N or for rows with no key.
__device__ __forceinline__ float lse_log2(const float* lse, size_t idx, bool in_range) {
  if (!in_range) return INFINITY;
  const float v = lse[idx];
  return v == -INFINITY ? INFINITY : v * LOG2E;
}

// D(tmem, 128 x 128) = A B^T, A and B K-major 128-byte swizzled tiles of
// `row_bytes` per row (16 KB column chunks), one MMA per 32 bytes of a row.
__device__ __forceinline__ void issue_nt(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, int row_bytes) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, false);
  const uint64_t ad = sdesc_sw128(a_smem, 16, 1024), bd = sdesc_sw128(b_smem, 16, 1024);
#pragma unroll 1
  for (int kk = 0; kk < row_bytes / 32; ++kk) {
    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
    mma_f16_ss(d_tmem, sdesc_add(ad, off), sdesc_add(bd, off), id, kk > 0 ? 1u : 0u);
  }
}

// D(tmem, 128 x 128) = A B^T with A packed bf16 in TMEM (128 lanes x D
// elements, D / 2 columns) and B a K-major shared-memory tile.
template <int D>
__device__ __forceinline__ void issue_nt_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, false);
  const uint64_t bd = sdesc_sw128(b_smem, 16, 1024);
#pragma unroll 1
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
// memory).  A is a K-major shared-memory tile (a_tmem == 0) or packed bf16 in
// TMEM (a_smem ignored).
template <int D>
__device__ __forceinline__ void issue_acc(uint32_t d_tmem, uint32_t a_smem, uint32_t a_tmem,
                                          uint32_t b_smem, bool first) {
  constexpr uint32_t id = idesc_bf16(128, D, false, true);
  const uint64_t ad = sdesc_sw128(a_smem, 16, 1024), bd = sdesc_sw128(b_smem, 16384, 1024);
#pragma unroll 1
  for (int kk = 0; kk < TILE / 16; ++kk) {
    const uint32_t acc = (first && kk == 0) ? 0u : 1u;
    const uint64_t b = sdesc_add(bd, kk * 16 * 128);
    if (a_tmem)
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

struct BwdBars {
  uint64_t in_full;              // resident tiles
  uint64_t full[2], empty[2];    // streamed stages (dkdv: Q+dO; dq: K)
  uint64_t vfull[2], vempty[2];  // dq: V stages
  uint64_t s_full, s_free, p_full, acc_done;
  uint64_t a_ready;              // dq: Q and dO copied into TMEM
  uint64_t fin[2];               // per issuer: all its MMAs done
  uint32_t tmem_base;
  int abort;
};

constexpr int BWD_LAUNCH_REGS = 168, BWD_REGS_LOW = 56, BWD_REGS_HIGH = 224;
static_assert(128 * BWD_REGS_LOW + 256 * BWD_REGS_HIGH <= 384 * BWD_LAUNCH_REGS, "register split");

// ================================================================== dK, dV
template <int D>
struct KvCfg {
  static constexpr int CH = D / 64;
  static constexpr int TB = TILE * D * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TB;
  static constexpr int ST_OFF = 2 * TB;  // stage s: Q tile at +0, dO tile at +TB
  static constexpr int PT_OFF = ST_OFF + 2 * 2 * TB;  // P^T tile, 128 x 128 bf16
  static constexpr int BAR_OFF = PT_OFF + TILE * TILE * 2;
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 256 + 1024);
};
static_assert(KvCfg<128>::SMEM_BYTES <= 232448, "dK/dV shared memory exceeds 227 KB");

// Steps of a dK/dV CTA: query head g of the group (outer), non-skipped Q tile
// I (inner, ascending).
struct KvSteps {
  int J, I_first, G;
  __device__ __forceinline__ int next_I(const AttnParams& p, int b, int I) const {
    while (I < p.nT && tile_class(p, b, I, J) == CLS_SKIP) ++I;
    return I;
  }
  // Advance (g, I) to the next step; false when past the last one.
  __device__ __forceinline__ bool advance(const AttnParams& p, int b, int& g, int& I) const {
    I = next_I(p, b, I + 1);
    if (I < p.nT) return true;
    ++g;
    I = I_first;
    return g < G;
  }
};

template <int D, bool MODS>
__global__ void __launch_bounds__(384, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, const AttnParams p) {
  using C = KvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  BwdBars& S = *reinterpret_cast<BwdBars*>(smem + C::BAR_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();

  const int BHk = p.B * p.Hkv;
  const int J = (int)(blockIdx.x / BHk);  // smallest KV tile (most work under causal) first
  const int bh = (int)(blockIdx.x % BHk);
  const int b = bh / p.Hkv, hk = bh - b * p.Hkv;
  const int G = p.Hq / p.Hkv;
  const bool causal = (p.flags & MOD_CAUSAL) != 0;
  KvSteps steps{J, 0, G};
  steps.I_first = steps.next_I(p, b, causal ? J : 0);
  const bool any = steps.I_first < p.nT;

  if (threadIdx.x == 0) {
    S.abort = 0;
    mbar_init(&S.in_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 2);  // dV issuer and dK issuer
    }
    mbar_init(&S.s_full, 2);      // S^T (issuer A) and dP^T (issuer B)
    mbar_init(&S.s_free, 256);
    mbar_init(&S.p_full, 256);
    mbar_init(&S.acc_done, 1);    // dV(n) done: P^T buffer free
    mbar_init(&S.fin[0], 1);
    mbar_init(&S.fin[1], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const uint32_t sK = smem_u32(smem + C::K_OFF);
  const uint32_t sV = smem_u32(smem + C::V_OFF);
  const uint32_t sST = smem_u32(smem + C::ST_OFF);
  const uint32_t sPT = smem_u32(smem + C::PT_OFF);
  // TMEM: S^T [0,128), dP^T / dS^T [128,256), dV [256, 256+D), dK [256+D, 256+2D).
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp < 4) regs_dec<BWD_REGS_LOW>();
  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      mbar_arrive_tx(&S.in_full, 2 * C::TB);
      for (int ch = 0; ch < C::CH; ++ch) {
        tma_load_3d(smem + C::K_OFF + ch * 16384, &tk, &S.in_full, ch * 64, J * TILE, b * p.Hkv + hk);
        tma_load_3d(smem + C::V_OFF + ch * 16384, &tv, &S.in_full, ch * 64, J * TILE, b * p.Hkv + hk);
      }
      int n = 0;
      if (any) {
        int g = 0, I = steps.I_first;
        do {
          const int st = n & 1;
          if (!mbar_wait(&S.empty[st], ((n >> 1) & 1) ^ 1, ab)) break;
          const int hq = hk * G + g;
          mbar_arrive_tx(&S.full[st], 2 * C::TB);
          uint8_t* dst = smem + C::ST_OFF + st * 2 * C::TB;
          for (int ch = 0; ch < C::CH; ++ch) {
            tma_load_3d(dst + ch * 16384, &tq, &S.full[st], ch * 64, I * TILE, b * p.Hq + hq);
            tma_load_3d(dst + C::TB + ch * 16384, &tdo, &S.full[st], ch * 64, I * TILE, b * p.Hq + hq);
          }
          ++n;
        } while (steps.advance(p, b, g, I));
      }
      mbar_wait_drain(&S.in_full, 0);
      for (int s = 0; s < 2; ++s)
        if (n > s) mbar_wait_drain(&S.full[s], ((n - 1 - s) >> 1) & 1);
    }
  } else if (warp == 1 || warp == 2) {
    // ---------------------------------------------------------- MMA issuers
    // Issuer A (warp 1): S^T = K Q^T and dV += P^T dO.
    // Issuer B (warp 2): dP^T = V dO^T and dK += dS^T Q.
    if (lane == 0) {
      const bool A = warp == 1;
      bool ok = mbar_wait(&S.in_full, 0, ab);
      tc_fence_after();
      if (ok && any) {
        int g = 0, I = steps.I_first, n = 0;
        ok = mbar_wait(&S.full[0], 0, ab);
        tc_fence_after();
        if (ok) {
          if (A)
            issue_nt(tS, sK, sST, D * 2);
          else
            issue_nt(tdP, sV, sST + C::TB, D * 2);
          mma_commit(&S.s_full);
        }
        while (ok) {
          const uint32_t q_sm = sST + (n & 1) * 2 * C::TB;
          const uint32_t do_sm = q_sm + C::TB;
          int g2 = g, I2 = I;
          const bool has_next = steps.advance(p, b, g2, I2);
          const uint32_t qn_sm = sST + ((n + 1) & 1) * 2 * C::TB;
          if (A && has_next) {
            // S^T(n+1) as soon as the softmax copied S^T(n) out.
            if (!(ok = mbar_wait(&S.full[(n + 1) & 1], ((n + 1) >> 1) & 1, ab))) break;
            if (!(ok = mbar_wait(&S.s_free, n & 1, ab))) break;
            tc_fence_after();
            issue_nt(tS, sK, qn_sm, D * 2);
            mma_commit(&S.s_full);
          }
          if (!(ok = mbar_wait(&S.p_full, n & 1, ab))) break;
          tc_fence_after();
          if (A) {
            issue_acc<D>(tdV, sPT, 0, do_sm, n == 0);
            mma_commit(&S.acc_done);
          } else {
            issue_acc<D>(tdK, 0, tdP, q_sm, n == 0);
          }
          mma_commit(&S.empty[n & 1]);
          if (!A && has_next) {
            // dP^T(n+1) after dK(n) has read dS^T(n) (same columns, in order).
            if (!(ok = mbar_wait(&S.full[(n + 1) & 1], ((n + 1) >> 1) & 1, ab))) break;
            tc_fence_after();
            issue_nt(tdP, sV, qn_sm + C::TB, D * 2);
            mma_commit(&S.s_full);
          }
          if (!has_next) break;
          g = g2;
          I = I2;
          ++n;
        }
      }
      mma_commit(&S.fin[A ? 0 : 1]);
      mbar_wait_drain(&S.fin[A ? 0 : 1], 0);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------- softmax / dS warpgroups
    regs_inc<BWD_REGS_HIGH>();
    const int w = (warp - 4) >> 2;  // query columns [64 w, 64 w + 64)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int j = J * TILE + r;  // this thread's KV row
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool sc = MODS && (p.flags & MOD_SOFTCAP);
    const bool al = MODS && (p.flags & MOD_ALIBI);
    const bool win = MODS && (p.flags & MOD_WINDOW);
    const bool doc = MODS && (p.flags & MOD_DOC);
    const float sc_in = p.scale / p.softcap, sc_out = p.softcap * LOG2E;
    const int doc_j = (doc && j < p.N) ? p.doc_ids[(size_t)b * p.N + j] : 0;
    uint8_t* pt_tile = smem + C::PT_OFF;
    bool ok = true;
    if (any) {
      int g = 0, I = steps.I_first, n = 0;
      do {
        const int hq = hk * G + g;
        const int cls = tile_class(p, b, I, J);
        const float al2 = al ? alibi_slope(p, hq) * LOG2E : 0.f;
        // LSE (log2 units) and D of this warpgroup's 64 query rows: lane k
        // holds rows k and 32 + k; loaded before the wait, broadcast below.
        const int i0 = I * TILE + 64 * w;  // query row of column 0
        const size_t rbase = ((size_t)b * p.Hq + hq) * p.N;
        float my_l2[2], my_dd[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ii = i0 + 32 * h + lane;
          my_l2[h] = lse_log2(lse, rbase + ii, ii < p.N);
          my_dd[h] = ii < p.N ? delta[rbase + ii] : 0.f;
        }
        if (!(ok = wait_warp(&S.s_full, n & 1, ab))) break;
        tc_fence_after();
        uint32_t s[64], dp[64];
        tmem_ld64(tS + lane_off + 64 * w, s);
        tmem_ld64(tdP + lane_off + 64 * w, dp);
        tmem_wait64(s);
        tmem_wait64(dp);
        tc_fence_before();
        mbar_arrive(&S.s_free);

        const int lo = causal ? j - i0 : -0x7fffffff;   // valid iff c >= lo
        const int hi = win ? p.window + j - i0 : 0x7fffffff;  // valid iff c < hi
        const float al_base = al2 * (float)(j - i0);
        uint32_t pw[32], dw[32];
#pragma unroll
        for (int c4 = 0; c4 < 64; c4 += 16) {
          float l2[16], dd[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            l2[k] = __shfl_sync(0xffffffffu, my_l2[(c4 + k) >> 5], (c4 + k) & 31);
            dd[k] = __shfl_sync(0xffffffffu, my_dd[(c4 + k) >> 5], (c4 + k) & 31);
          }
#pragma unroll
          for (int k = 0; k < 16; k += 2) {
            float pe[2], ds[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = c4 + k + e;
              const float sv = __uint_as_float(s[c]);
              float x, dmul = 1.f;
              if (sc) {
                const float t = tanh_exp(sv * sc_in);
                x = t * sc_out;
                dmul = fmaf(-t, t, 1.f);
              } else {
                x = sv * p.scale_log2;
              }
              if (al) x = fmaf(-al2, (float)c, x + al_base);
              float pv = ex2(x - l2[k + e]);
              if (cls == CLS_PARTIAL) {
                bool valid = (c >= lo) && (c < hi);
                if (doc && valid)
                  valid = (i0 + c < p.N) && (__ldg(p.doc_ids + (size_t)b * p.N + i0 + c) == doc_j);
                if (!valid) pv = 0.f;
              }
              pe[e] = pv;
              ds[e] = pv * (__uint_as_float(dp[c]) - dd[k + e]) * dmul;
            }
            pw[(c4 + k) / 2] = pack_bf16(pe[0], pe[1]);
            dw[(c4 + k) / 2] = pack_bf16(ds[0], ds[1]);
          }
        }
        // dS^T over dP^T in TMEM (A operand of dK += dS^T Q), packed into the
        // first 64 columns of dP^T -- which the other warpgroup reads: wait
        // until all 256 softmax threads have copied dP^T(n) out.
        if (!(ok = wait_warp(&S.s_free, n & 1, ab))) break;
        tc_fence_after();
        tmem_st32(tdP + lane_off + 32 * w, dw);
        // P^T to shared memory once dV(n-1) has read the previous one.
        if (n > 0) {
          if (!(ok = wait_warp(&S.acc_done, (n - 1) & 1, ab))) break;
          tc_fence_after();
        }
        store_half_row(pt_tile, r, w, pw);
        tmem_wait_st();
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&S.p_full);
        ++n;
      } while (steps.advance(p, b, g, I));
    }
    if (ok) ok = wait_warp(&S.fin[0], 0, ab) && wait_warp(&S.fin[1], 0, ab);
    tc_fence_after();
    if (ok) {
      const size_t row = ((size_t)b * p.Hkv + hk) * p.N + j;
      store_cols<D / 2>(tdV + lane_off + w * (D / 2), any, 1.0f, dv + row * D + w * (D / 2), j < p.N);
      store_cols<D / 2>(tdK + lane_off + w * (D / 2), any, p.scale, dk + row * D + w * (D / 2), j < p.N);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ======================================================================= dQ
template <int D>
struct DqCfg {
  static constexpr int CH = D / 64;
  static constexpr int TB = TILE * D * 2;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = TB;
  static constexpr int K_OFF = 2 * TB;  // 2 K stages
  static constexpr int V_OFF = 4 * TB;  // 2 V stages
  static constexpr int DS_OFF = 6 * TB; // dS tile, 128 x 128 bf16
  static constexpr int BAR_OFF = DS_OFF + TILE * TILE * 2;
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 256 + 1024);
};
static_assert(DqCfg<128>::SMEM_BYTES <= 232448, "dQ shared memory exceeds 227 KB");

template <int D, bool MODS>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const float* __restrict__ lse, const float* __restrict__ delta,
                  __nv_bfloat16* __restrict__ dq, const AttnParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  BwdBars& S = *reinterpret_cast<BwdBars*>(smem + C::BAR_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();

  const int BH = p.B * p.Hq;
  const int I = p.nT - 1 - (int)(blockIdx.x / BH);  // longest rows (causal) first
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int hk = hq / (p.Hq / p.Hkv);
  const bool causal = (p.flags & MOD_CAUSAL) != 0;
  const int J_end = causal ? min(p.nT, I + 1) : p.nT;
  auto next_J = [&](int J) {
    while (J < J_end && tile_class(p, b, I, J) == CLS_SKIP) ++J;
    return J;
  };
  const int J_first = next_J(0);

  if (threadIdx.x == 0) {
    S.abort = 0;
    mbar_init(&S.in_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 2);   // K: read by S (A) and dQ (B)
      mbar_init(&S.vfull[s], 1);
      mbar_init(&S.vempty[s], 1);  // V: read by dP (A)
    }
    mbar_init(&S.s_full, 1);
    mbar_init(&S.s_free, 256);
    mbar_init(&S.p_full, 256);
    mbar_init(&S.acc_done, 1);     // dQ(n) done: dS buffer free
    mbar_init(&S.a_ready, 256);    // Q / dO in TMEM
    mbar_init(&S.fin[0], 1);
    mbar_init(&S.fin[1], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const uint32_t sQ = smem_u32(smem + C::Q_OFF);
  const uint32_t sDO = smem_u32(smem + C::DO_OFF);
  const uint32_t sK = smem_u32(smem + C::K_OFF);
  const uint32_t sV = smem_u32(smem + C::V_OFF);
  const uint32_t sDS = smem_u32(smem + C::DS_OFF);
  // TMEM: S [0,128), dP [128,256), dQ [256, 256+D), then Q and dO as packed
  // bf16 A operands (D / 2 columns each): the recompute GEMMs S = Q K^T and
  // dP = dO V^T read only K / V from shared memory.
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256;
  const uint32_t tQa = tmem + 256 + D, tDOa = tmem + 256 + D + D / 2;

  if (warp < 4) regs_dec<BWD_REGS_LOW>();
  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_tx(&S.in_full, 2 * C::TB);
      for (int ch = 0; ch < C::CH; ++ch) {
        tma_load_3d(smem + C::Q_OFF + ch * 16384, &tq, &S.in_full, ch * 64, I * TILE, b * p.Hq + hq);
        tma_load_3d(smem + C::DO_OFF + ch * 16384, &tdo, &S.in_full, ch * 64, I * TILE, b * p.Hq + hq);
      }
      int nk = 0, nv = 0;
      for (int J = J_first; J < J_end; J = next_J(J + 1)) {
        const int st = nk & 1;
        if (!mbar_wait(&S.empty[st], ((nk >> 1) & 1) ^ 1, ab)) break;
        mbar_arrive_tx(&S.full[st], C::TB);
        for (int ch = 0; ch < C::CH; ++ch)
          tma_load_3d(smem + C::K_OFF + st * C::TB + ch * 16384, &tk, &S.full[st], ch * 64, J * TILE,
                      b * p.Hkv + hk);
        ++nk;
        if (!mbar_wait(&S.vempty[st], ((nv >> 1) & 1) ^ 1, ab)) break;
        mbar_arrive_tx(&S.vfull[st], C::TB);
        for (int ch = 0; ch < C::CH; ++ch)
          tma_load_3d(smem + C::V_OFF + st * C::TB + ch * 16384, &tv, &S.vfull[st], ch * 64, J * TILE,
                      b * p.Hkv + hk);
        ++nv;
      }
      mbar_wait_drain(&S.in_full, 0);
      for (int s = 0; s < 2; ++s) {
        if (nk > s) mbar_wait_drain(&S.full[s], ((nk - 1 - s) >> 1) & 1);
        if (nv > s) mbar_wait_drain(&S.vfull[s], ((nv - 1 - s) >> 1) & 1);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // Issuer A (warp 1): S = Q K^T and dP = dO V^T.  Issuer B (warp 2): dQ += dS K.
    if (lane == 0) {
      const bool A = warp == 1;
      bool ok = mbar_wait(&S.in_full, 0, ab);
      tc_fence_after();
      int n = 0;
      for (int J = J_first; ok && J < J_end; J = next_J(J + 1), ++n) {
        const int st = n & 1;
        if (!(ok = mbar_wait(&S.full[st], (n >> 1) & 1, ab))) break;
        if (A) {
          if (!(ok = mbar_wait(&S.vfull[st], (n >> 1) & 1, ab))) break;
          if (n == 0 && !(ok = mbar_wait(&S.a_ready, 0, ab))) break;
          if (n > 0 && !(ok = mbar_wait(&S.s_free, (n - 1) & 1, ab))) break;
          tc_fence_after();
          issue_nt_tmem_a<D>(tS, tQa, sK + st * C::TB);
          issue_nt_tmem_a<D>(tdP, tDOa, sV + st * C::TB);
          mma_commit(&S.s_full);
          mma_commit(&S.vempty[st]);
          mma_commit(&S.empty[st]);
        } else {
          if (!(ok = mbar_wait(&S.p_full, n & 1, ab))) break;
          tc_fence_after();
          issue_acc<D>(tdQ, sDS, 0, sK + st * C::TB, n == 0);
          mma_commit(&S.acc_done);
          mma_commit(&S.empty[st]);
        }
      }
      mma_commit(&S.fin[A ? 0 : 1]);
      mbar_wait_drain(&S.fin[A ? 0 : 1], 0);
    }
  } else if (warp >= 4) {
    regs_inc<BWD_REGS_HIGH>();
    const int w = (warp - 4) >> 2;  // key columns [64 w, 64 w + 64)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int i = I * TILE + r;  // this thread's query row
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool sc = MODS && (p.flags & MOD_SOFTCAP);
    const bool al = MODS && (p.flags & MOD_ALIBI);
    const bool win = MODS && (p.flags & MOD_WINDOW);
    const bool doc = MODS && (p.flags & MOD_DOC);
    const float sc_in = p.scale / p.softcap, sc_out = p.softcap * LOG2E;
    const float al2 = al ? alibi_slope(p, hq) * LOG2E : 0.f;
    const size_t row = ((size_t)b * p.Hq + hq) * p.N + i;
    const float lse2 = lse_log2(lse, row, i < p.N);
    const float dd = i < p.N ? delta[row] : 0.f;
    const int doc_i = (doc && i < p.N) ? p.doc_ids[(size_t)b * p.N + i] : 0;
    uint8_t* ds_tile = smem + C::DS_OFF;
    bool ok = wait_warp(&S.in_full, 0, ab);
    if (ok) {  // warpgroup 0 copies Q, warpgroup 1 copies dO into TMEM
      tile_row_to_tmem<D>(smem + (w == 0 ? C::Q_OFF : C::DO_OFF), r, (w == 0 ? tQa : tDOa) + lane_off);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&S.a_ready);
    }
    int n = 0;
    for (int J = J_first; ok && J < J_end; J = next_J(J + 1), ++n) {
      const int cls = tile_class(p, b, I, J);
      if (!(ok = wait_warp(&S.s_full, n & 1, ab))) break;
      tc_fence_after();
      uint32_t s[64], dp[64];
      tmem_ld64(tS + lane_off + 64 * w, s);
      tmem_ld64(tdP + lane_off + 64 * w, dp);
      tmem_wait64(s);
      tmem_wait64(dp);
      tc_fence_before();
      mbar_arrive(&S.s_free);

      const int j0 = J * TILE + 64 * w;  // key row of column 0
      const int hi_lim = min(causal ? i : 0x7fffffff, p.N - 1) - j0;  // valid iff c <= hi_lim
      const int lo_lim = win ? i - p.window - j0 : -0x7fffffff;        // valid iff c > lo_lim
      const float al_base = al2 * (float)(j0 - i);
      uint32_t dw[32];
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        float ds[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = k + e;
          const float sv = __uint_as_float(s[c]);
          float x, dmul = 1.f;
          if (sc) {
            const float t = tanh_exp(sv * sc_in);
            x = t * sc_out;
            dmul = fmaf(-t, t, 1.f);
          } else {
            x = sv * p.scale_log2;
          }
          if (al) x = fmaf(al2, (float)c, x + al_base);
          float pe = ex2(x - lse2);
          if (cls == CLS_PARTIAL) {
            bool valid = (c <= hi_lim) && (c > lo_lim);
            if (doc && valid) valid = (__ldg(p.doc_ids + (size_t)b * p.N + j0 + c) == doc_i);
            if (!valid) pe = 0.f;
          }
          ds[e] = pe * (__uint_as_float(dp[c]) - dd) * dmul;
        }
        dw[k / 2] = pack_bf16(ds[0], ds[1]);
      }
      if (n > 0) {
        if (!(ok = wait_warp(&S.acc_done, (n - 1) & 1, ab))) break;
        tc_fence_after();
      }
      store_half_row(ds_tile, r, w, dw);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&S.p_full);
    }
    if (ok) ok = wait_warp(&S.fin[1], 0, ab);
    tc_fence_after();
    if (ok) store_cols<D / 2>(tdQ + lane_off + w * (D / 2), n > 0, p.scale, dq + row * D + w * (D / 2), i < p.N);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ launch
template <typename K>
static cudaError_t check_regs(K kern, int& cached) {
  if (cached < 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return cudaErrorInvalidDeviceFunction;
    cached = fa.numRegs;
  }
  // The register split inside the kernel assumes this allocation at launch.
  return cached == BWD_LAUNCH_REGS ? cudaSuccess : cudaErrorInvalidConfiguration;
}

template <int D, bool MODS>
static cudaError_t launch_bwd_t(const BwdLaunch& L, cudaStream_t st) {
  const AttnParams& p = L.p;
  const long long rows = (long long)p.B * p.Hq * p.N;
  const long long threads = rows * (D / 8);
  if (L.events[0]) cudaEventRecord(L.events[0], st);
  bwd_pre_kernel<D><<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
      (const __nv_bfloat16*)L.o, (const __nv_bfloat16*)L.dout, L.delta, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  static int kv_regs = -1, dq_regs = -1;
  auto kv = bwd_dkdv_kernel<D, MODS>;
  if ((e = check_regs(kv, kv_regs)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  if (L.events[1]) cudaEventRecord(L.events[1], st);
  kv<<<(unsigned)(p.nT * p.B * p.Hkv), 384, KvCfg<D>::SMEM_BYTES, st>>>(
      L.tq, L.tk, L.tv, L.tdo, L.lse, L.delta, (__nv_bfloat16*)L.dk, (__nv_bfloat16*)L.dv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  auto dqk = bwd_dq_kernel<D, MODS>;
  if ((e = check_regs(dqk, dq_regs)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(dqk, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  if (L.events[2]) cudaEventRecord(L.events[2], st);
  dqk<<<(unsigned)(p.nT * p.B * p.Hq), 384, DqCfg<D>::SMEM_BYTES, st>>>(
      L.tq, L.tk, L.tv, L.tdo, L.lse, L.delta, (__nv_bfloat16*)L.dq, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (L.events[3]) cudaEventRecord(L.events[3], st);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdLaunch& L, int d, bool mods, cudaStream_t st) {
  if (d == 128) return mods ? launch_bwd_t<128, true>(L, st) : launch_bwd_t<128, false>(L, st);
  return mods ? launch_bwd_t<64, true>(L, st) : launch_bwd_t<64, false>(L, st);
}

}  // namespace attn
