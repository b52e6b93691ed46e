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
//    every needed Q tile stream through a TMA ring.  S^T = K Q^T and
//    dP^T = V dO^T land in TMEM; one softmax warpgroup (a thread per KV row)
//    turns them into P^T and dS^T (bf16, written back over S^T / dP^T), and
//    dV += P^T dO, dK += dS^T Q run with their A operand read from TMEM.
//  * bwd_dq:   one CTA per (batch, query head, 128-row Q tile), streaming K/V
//    tiles: S = Q K^T and dP = dO V^T in TMEM, dS back over S, dQ += dS K.
// Each dQ, dK, dV tile is accumulated by exactly one CTA, in TMEM, over its
// partner tiles in ascending order: no atomics, so the result is bitwise
// reproducible (contrast the nondeterministic block-sparse backward on the
// FlexAttention/FA4 page, "Limitations actuelles").  Every step is split in
// two 64-column halves so the softmax of one half overlaps the MMAs of the
// other.
#include "common.cuh"
#include "launch.h"

namespace attn {

constexpr int MAX_LIST = BWD_MAX_N / TILE;  // tiles per sequence the step lists can hold

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

// Row constants shared by the two main kernels.
__device__ __forceinline__ float lse_log2(const float* lse, size_t idx, bool in_range) {
  if (!in_range) return INFINITY;  // rows past N: P = 0
  const float v = lse[idx];
  return v == -INFINITY ? INFINITY : v * LOG2E;  // rows with no key: P = 0
}

// Pack 64 fp32 (as bits) to 32 bf16x2 words.
__device__ __forceinline__ void pack64(const float (&v)[64], uint32_t (&w)[32]) {
#pragma unroll
  for (int k = 0; k < 32; ++k) w[k] = pack_bf16(v[2 * k], v[2 * k + 1]);
}

// S/dP half-tiles: D(tmem, M=128 x N=64) = A(128 rows, K-major) * B(64 rows at b_smem, K-major)^T.
template <int D>
__device__ __forceinline__ void issue_half_nt(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
  constexpr uint32_t id = idesc_bf16(128, 64, false, false);
  const uint64_t ad = sdesc_sw128(a_smem, 16, 1024), bd = sdesc_sw128(b_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
    mma_f16_ss(d_tmem, sdesc_add(ad, off), sdesc_add(bd, off), id, kk > 0 ? 1u : 0u);
  }
}

// Accumulation: D(tmem, 128 x D) += A(tmem, 128 x 64 packed bf16) * B(64 rows at b_smem, MN-major).
template <int D>
__device__ __forceinline__ void issue_half_acc(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                               bool first) {
  constexpr uint32_t id = idesc_bf16(128, D, false, true);
  const uint64_t bd = sdesc_sw128(b_smem, 16384, 1024);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_f16_ts(d_tmem, a_tmem + kk * 8, sdesc_add(bd, kk * 16 * 128), id, (first && kk == 0) ? 0u : 1u);
}

// Write a 128-column-or-less fp32 TMEM row (D columns at t_col) to a bf16 row, times mul.
template <int D>
__device__ __forceinline__ void store_row(uint32_t t_col, bool have, float mul, __nv_bfloat16* dst,
                                          bool in_range) {
#pragma unroll
  for (int q4 = 0; q4 < D / 32; ++q4) {
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
    for (int w = 0; w < 16; ++w)
      pk[w] = pack_bf16(__uint_as_float(v[2 * w]) * mul, __uint_as_float(v[2 * w + 1]) * mul);
    if (in_range) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + q4 * 32);
#pragma unroll
      for (int w = 0; w < 4; ++w) d4[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
    }
  }
}

// ================================================================== dK, dV
template <int D>
struct KvCfg {
  static constexpr int CH = D / 64;
  static constexpr int TB = TILE * D * 2;
  static constexpr int QST = 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TB;
  static constexpr int ST_OFF = 2 * TB;  // stage s: Q tile at +0, dO tile at +TB
  static constexpr int VEC_OFF = ST_OFF + QST * 2 * TB;  // stage s: lse2[128], D[128]
  static constexpr int LIST_OFF = VEC_OFF + QST * 1024;
  static constexpr int BAR_OFF = LIST_OFF + MAX_LIST * 2;
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 256 + 1024);
};

struct BwdBars {
  uint64_t in_full;         // resident tiles (K/V or Q/dO)
  uint64_t full[2], empty[2];  // streamed stages
  uint64_t s_full[2], p_full[2];
  uint64_t done, drain;
  uint32_t tmem_base;
  int n_list;
  int abort;
};

template <int D, bool MODS>
__global__ void __launch_bounds__(256, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, const AttnParams p) {
  using C = KvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  BwdBars& S = *reinterpret_cast<BwdBars*>(smem + C::BAR_OFF);
  int16_t* list = reinterpret_cast<int16_t*>(smem + C::LIST_OFF);
  float* vec = reinterpret_cast<float*>(smem + C::VEC_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();

  const int BHk = p.B * p.Hkv;
  const int J = (int)(blockIdx.x / BHk);  // smallest KV tile (most work under causal) first
  const int bh = (int)(blockIdx.x % BHk);
  const int b = bh / p.Hkv, hk = bh - b * p.Hkv;
  const int G = p.Hq / p.Hkv;
  const bool causal = (p.flags & MOD_CAUSAL) != 0;

  if (threadIdx.x == 0) {
    S.abort = 0;
    mbar_init(&S.in_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.full[s], 1 + 32);
      mbar_init(&S.empty[s], 1);
      mbar_init(&S.s_full[s], 1);
      mbar_init(&S.p_full[s], 128);
    }
    mbar_init(&S.done, 1);
    mbar_init(&S.drain, 1);
    fence_mbar_init();
    int n = 0;
    for (int I = causal ? J : 0; I < p.nT && n < MAX_LIST; ++I)
      if (tile_class(p, b, I, J) != CLS_SKIP) list[n++] = (int16_t)I;
    S.n_list = n;
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const int nI = S.n_list;
  const int T = G * nI;
  const uint32_t sK = smem_u32(smem + C::K_OFF);
  const uint32_t sV = smem_u32(smem + C::V_OFF);
  const uint32_t sST = smem_u32(smem + C::ST_OFF);

  if (warp == 0) {
    // ---------------------------------------------------------- producer warp
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tdo);
      mbar_arrive_tx(&S.in_full, 2 * C::TB);
      for (int ch = 0; ch < C::CH; ++ch) {
        tma_load_3d(smem + C::K_OFF + ch * 16384, &tk, &S.in_full, ch * 64, J * TILE, b * p.Hkv + hk);
        tma_load_3d(smem + C::V_OFF + ch * 16384, &tv, &S.in_full, ch * 64, J * TILE, b * p.Hkv + hk);
      }
    }
    int n = 0;
    for (; n < T; ++n) {
      const int st = n % C::QST;
      if (!wait_warp(&S.empty[st], ((n / C::QST) & 1) ^ 1, ab)) break;
      const int g = n / nI;
      const int I = list[n % nI];
      const int hq = hk * G + g;
      if (lane == 0) {
        mbar_arrive_tx(&S.full[st], 2 * C::TB);
        uint8_t* dst = smem + C::ST_OFF + st * 2 * C::TB;
        for (int ch = 0; ch < C::CH; ++ch) {
          tma_load_3d(dst + ch * 16384, &tq, &S.full[st], ch * 64, I * TILE, b * p.Hq + hq);
          tma_load_3d(dst + C::TB + ch * 16384, &tdo, &S.full[st], ch * 64, I * TILE, b * p.Hq + hq);
        }
      }
      float* v = vec + st * 256;
      const size_t base = ((size_t)b * p.Hq + hq) * p.N;
      for (int r = lane; r < TILE; r += 32) {
        const int i = I * TILE + r;
        v[r] = lse_log2(lse, base + i, i < p.N);
        v[TILE + r] = i < p.N ? delta[base + i] : 0.f;
      }
      mbar_arrive(&S.full[st]);
    }
    if (lane == 0) {
      mbar_wait_drain(&S.in_full, 0);
      for (int s = 0; s < C::QST; ++s)
        if (n > s) mbar_wait_drain(&S.full[s], ((n - 1 - s) / C::QST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(&S.in_full, 0, ab);
      tc_fence_after();
      if (ok && T > 0) {
        ok = mbar_wait(&S.full[0], 0, ab);
        tc_fence_after();
        if (ok) {
          for (int h = 0; h < 2; ++h) {
            issue_half_nt<D>(tmem + h * 64, sK, sST + h * 8192);
            issue_half_nt<D>(tmem + 128 + h * 64, sV, sST + C::TB + h * 8192);
            mma_commit(&S.s_full[h]);
          }
        }
      }
      for (int n = 0; ok && n < T; ++n) {
        const int st = n % C::QST;
        const uint32_t q_sm = sST + st * 2 * C::TB;
        const uint32_t do_sm = q_sm + C::TB;
        const bool has_next = n + 1 < T;
        const int stn = (n + 1) % C::QST;
        const uint32_t qn_sm = sST + stn * 2 * C::TB;
        for (int h = 0; h < 2; ++h) {
          if (!(ok = mbar_wait(&S.p_full[h], n & 1, ab))) break;
          tc_fence_after();
          issue_half_acc<D>(tmem + 256, tmem + h * 64, do_sm + h * 8192, n == 0 && h == 0);
          issue_half_acc<D>(tmem + 256 + D, tmem + 128 + h * 64, q_sm + h * 8192, n == 0 && h == 0);
          if (h == 1) mma_commit(&S.empty[st]);
          if (has_next) {
            if (h == 0) {
              if (!(ok = mbar_wait(&S.full[stn], ((n + 1) / C::QST) & 1, ab))) break;
              tc_fence_after();
            }
            issue_half_nt<D>(tmem + h * 64, sK, qn_sm + h * 8192);
            issue_half_nt<D>(tmem + 128 + h * 64, sV, qn_sm + C::TB + h * 8192);
            mma_commit(&S.s_full[h]);
          }
        }
      }
      mma_commit(&S.done);
      mma_commit(&S.drain);
      mbar_wait_drain(&S.drain, 0);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------- softmax / dS warpgroup
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
    bool ok = true;
    for (int n = 0; ok && n < T; ++n) {
      const int g = n / nI;
      const int I = list[n % nI];
      const int hq = hk * G + g;
      const int cls = tile_class(p, b, I, J);
      const float* v = vec + (n % C::QST) * 256;
      const float al2 = al ? alibi_slope(p, hq) * LOG2E : 0.f;
      for (int h = 0; h < 2; ++h) {
        if (!(ok = wait_warp(&S.s_full[h], n & 1, ab))) break;
        tc_fence_after();
        uint32_t s[64], dp[64];
        tmem_ld32(tmem + lane_off + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tmem + lane_off + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld32(tmem + lane_off + 128 + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_ld32(tmem + lane_off + 128 + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        const int i0 = I * TILE + h * 64;         // q row of column 0
        const int lo = causal ? j - i0 : -0x7fffffff;   // valid iff c >= lo
        const int hi = win ? p.window + j - i0 : 0x7fffffff;  // valid iff c < hi
        const float al_base = al2 * (float)(j - i0);
        const float* lv = v + h * 64;
        const float* dv_ = v + TILE + h * 64;
        float pv[64], dsv[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
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
          float pe = ex2(x - lv[c]);
          if (cls == CLS_PARTIAL) {
            bool valid = (c >= lo) && (c < hi);
            if (doc && valid) valid = (i0 + c < p.N) && (__ldg(p.doc_ids + (size_t)b * p.N + i0 + c) == doc_j);
            if (!valid) pe = 0.f;
          }
          pv[c] = pe;
          dsv[c] = pe * (__uint_as_float(dp[c]) - dv_[c]) * dmul;
        }
        uint32_t w[32];
        pack64(pv, w);
        tmem_st32(tmem + lane_off + h * 64, w);
        pack64(dsv, w);
        tmem_st32(tmem + lane_off + 128 + h * 64, w);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&S.p_full[h]);
      }
    }
    if (ok) ok = wait_warp(&S.done, 0, ab);
    tc_fence_after();
    if (ok) {
      const size_t row = ((size_t)b * p.Hkv + hk) * p.N + j;
      store_row<D>(tmem + lane_off + 256, T > 0, 1.0f, dv + row * D, j < p.N);
      store_row<D>(tmem + lane_off + 256 + D, T > 0, p.scale, dk + row * D, j < p.N);
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
  static constexpr int KST = 2;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = TB;
  static constexpr int ST_OFF = 2 * TB;  // stage s: K tile at +0, V tile at +TB
  static constexpr int LIST_OFF = ST_OFF + KST * 2 * TB;
  static constexpr int BAR_OFF = LIST_OFF + MAX_LIST * 2;
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 256 + 1024);
};

template <int D, bool MODS>
__global__ void __launch_bounds__(256, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const float* __restrict__ lse, const float* __restrict__ delta,
                  __nv_bfloat16* __restrict__ dq, const AttnParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  BwdBars& S = *reinterpret_cast<BwdBars*>(smem + C::BAR_OFF);
  int16_t* list = reinterpret_cast<int16_t*>(smem + C::LIST_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();

  const int BH = p.B * p.Hq;
  const int I = p.nT - 1 - (int)(blockIdx.x / BH);  // longest rows (causal) first
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int hk = hq / (p.Hq / p.Hkv);
  const bool causal = (p.flags & MOD_CAUSAL) != 0;

  if (threadIdx.x == 0) {
    S.abort = 0;
    mbar_init(&S.in_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
      mbar_init(&S.s_full[s], 1);
      mbar_init(&S.p_full[s], 128);
    }
    mbar_init(&S.done, 1);
    mbar_init(&S.drain, 1);
    fence_mbar_init();
    const int J_end = causal ? min(p.nT, I + 1) : p.nT;
    int n = 0;
    for (int J = 0; J < J_end && n < MAX_LIST; ++J)
      if (tile_class(p, b, I, J) != CLS_SKIP) list[n++] = (int16_t)J;
    S.n_list = n;
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const int T = S.n_list;
  const uint32_t sQ = smem_u32(smem + C::Q_OFF);
  const uint32_t sDO = smem_u32(smem + C::DO_OFF);
  const uint32_t sST = smem_u32(smem + C::ST_OFF);

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_tx(&S.in_full, 2 * C::TB);
      for (int ch = 0; ch < C::CH; ++ch) {
        tma_load_3d(smem + C::Q_OFF + ch * 16384, &tq, &S.in_full, ch * 64, I * TILE, b * p.Hq + hq);
        tma_load_3d(smem + C::DO_OFF + ch * 16384, &tdo, &S.in_full, ch * 64, I * TILE, b * p.Hq + hq);
      }
      int n = 0;
      for (; n < T; ++n) {
        const int st = n % C::KST;
        if (!mbar_wait(&S.empty[st], ((n / C::KST) & 1) ^ 1, ab)) break;
        const int J = list[n];
        mbar_arrive_tx(&S.full[st], 2 * C::TB);
        uint8_t* dst = smem + C::ST_OFF + st * 2 * C::TB;
        for (int ch = 0; ch < C::CH; ++ch) {
          tma_load_3d(dst + ch * 16384, &tk, &S.full[st], ch * 64, J * TILE, b * p.Hkv + hk);
          tma_load_3d(dst + C::TB + ch * 16384, &tv, &S.full[st], ch * 64, J * TILE, b * p.Hkv + hk);
        }
      }
      mbar_wait_drain(&S.in_full, 0);
      for (int s = 0; s < C::KST; ++s)
        if (n > s) mbar_wait_drain(&S.full[s], ((n - 1 - s) / C::KST) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(&S.in_full, 0, ab);
      tc_fence_after();
      if (ok && T > 0) {
        ok = mbar_wait(&S.full[0], 0, ab);
        tc_fence_after();
        if (ok) {
          for (int h = 0; h < 2; ++h) {
            issue_half_nt<D>(tmem + h * 64, sQ, sST + h * 8192);
            issue_half_nt<D>(tmem + 128 + h * 64, sDO, sST + C::TB + h * 8192);
            mma_commit(&S.s_full[h]);
          }
        }
      }
      for (int n = 0; ok && n < T; ++n) {
        const int st = n % C::KST;
        const uint32_t k_sm = sST + st * 2 * C::TB;
        const bool has_next = n + 1 < T;
        const int stn = (n + 1) % C::KST;
        const uint32_t kn_sm = sST + stn * 2 * C::TB;
        for (int h = 0; h < 2; ++h) {
          if (!(ok = mbar_wait(&S.p_full[h], n & 1, ab))) break;
          tc_fence_after();
          issue_half_acc<D>(tmem + 256, tmem + h * 64, k_sm + h * 8192, n == 0 && h == 0);
          if (h == 1) mma_commit(&S.empty[st]);
          if (has_next) {
            if (h == 0) {
              if (!(ok = mbar_wait(&S.full[stn], ((n + 1) / C::KST) & 1, ab))) break;
              tc_fence_after();
            }
            issue_half_nt<D>(tmem + h * 64, sQ, kn_sm + h * 8192);
            issue_half_nt<D>(tmem + 128 + h * 64, sDO, kn_sm + C::TB + h * 8192);
            mma_commit(&S.s_full[h]);
          }
        }
      }
      mma_commit(&S.done);
      mma_commit(&S.drain);
      mbar_wait_drain(&S.drain, 0);
    }
  } else if (warp >= 4) {
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
    bool ok = true;
    for (int n = 0; ok && n < T; ++n) {
      const int J = list[n];
      const int cls = tile_class(p, b, I, J);
      for (int h = 0; h < 2; ++h) {
        if (!(ok = wait_warp(&S.s_full[h], n & 1, ab))) break;
        tc_fence_after();
        uint32_t s[64], dp[64];
        tmem_ld32(tmem + lane_off + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(tmem + lane_off + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld32(tmem + lane_off + 128 + h * 64, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_ld32(tmem + lane_off + 128 + h * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        const int j0 = J * TILE + h * 64;  // kv row of column 0
        const int hi_lim = min(causal ? i : 0x7fffffff, p.N - 1) - j0;  // valid iff c <= hi_lim
        const int lo_lim = win ? i - p.window - j0 : -0x7fffffff;        // valid iff c > lo_lim
        const float al_base = al2 * (float)(j0 - i);
        float dsv[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
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
          dsv[c] = pe * (__uint_as_float(dp[c]) - dd) * dmul;
        }
        uint32_t w[32];
        pack64(dsv, w);
        tmem_st32(tmem + lane_off + h * 64, w);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&S.p_full[h]);
      }
    }
    if (ok) ok = wait_warp(&S.done, 0, ab);
    tc_fence_after();
    if (ok) store_row<D>(tmem + lane_off + 256, T > 0, p.scale, dq + row * D, i < p.N);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ launch
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

  auto kv = bwd_dkdv_kernel<D, MODS>;
  if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, KvCfg<D>::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  if (L.events[1]) cudaEventRecord(L.events[1], st);
  kv<<<(unsigned)(p.nT * p.B * p.Hkv), 256, KvCfg<D>::SMEM_BYTES, st>>>(
      L.tq, L.tk, L.tv, L.tdo, L.lse, L.delta, (__nv_bfloat16*)L.dk, (__nv_bfloat16*)L.dv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  auto dqk = bwd_dq_kernel<D, MODS>;
  if ((e = cudaFuncSetAttribute(dqk, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  if (L.events[2]) cudaEventRecord(L.events[2], st);
  dqk<<<(unsigned)(p.nT * p.B * p.Hq), 256, DqCfg<D>::SMEM_BYTES, st>>>(
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
