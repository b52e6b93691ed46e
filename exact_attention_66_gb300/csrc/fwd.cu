// Forward pass of exact tiled attention for sm_103a: bf16 or e4m3 operands,
// fp32 accumulation and softmax.
//
// Method (FlashAttention-3 digest, "Rappel du fonctionnement de FlashAttention"
// and "Chevauchement de GEMM et softmax grâce à l'asynchronisme"; FlashAttention-2
// (FR), "Architecture technique et principes de fonctionnement"): Q is split in
// tiles of 128 rows, K/V are streamed in tiles of 128 rows, and for every tile
// pair the two GEMMs S = Q K^T and O += P V run on the tensor cores while a
// running row max m and row sum l rescale the partial output, so the N x N
// score matrix is never stored and the result is exact.
//
// GB300 design (not a translation of the pages' Hopper/Ampere kernels):
//  * one CTA = two Q tiles (256 rows) of one (batch, query head); both tiles
//    share every K/V tile that TMA brings into shared memory;
//  * warp 0 issues TMA loads (Q once, K/V through two-stage rings guarded by
//    mbarriers); warp 1 issues tcgen05 MMAs from a single thread; warps 4-7
//    and 8-11 are the softmax warpgroups of Q tile 0 and Q tile 1;
//  * S lives in TMEM (fp32, 128 columns per tile), the softmax warpgroup
//    writes P back over S as packed bf16, and P V reads P straight from TMEM
//    (A operand in tensor memory), so P never touches shared memory;
//  * the MMA order S0(j) S1(j) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ... hides each
//    warpgroup's exponentials behind the other tile's GEMMs (the pages'
//    ping-pong idea, expressed with tcgen05 commits instead of named barriers);
//  * O is rescaled in TMEM only when a row max grows by more than 2^8
//    (lazy rescale, exact after the final division by l);
//  * on partial (masked) tiles P is split into bf16 hi + lo parts and both
//    are multiplied by V, which removes the bf16 rounding of P where few keys
//    carry the whole row (the first rows of a causal context);
//  * fully masked tiles are skipped (block-sparsity map, FlexAttention/FA4
//    page, "Limitations actuelles");
//  * the FP8 variant (FlashAttention-3 digest, "Basse précision FP8 et
//    incoherent processing") runs the same pipeline on e4m3 Q/K/V with
//    tcgen05.mma kind::f8f6f4 (twice the bf16 rate), rounds P to e4m3 for
//    P V, and folds the per-(batch, head) dequantisation scales into the
//    softmax scale (Q, K) and the epilogue (V).
#include "common.cuh"
#include "launch.h"

namespace attn {

template <int D, bool FP8>
struct FwdCfg {
  static constexpr int ESZ = FP8 ? 1 : 2;              // bytes per element
  static constexpr int ROW_BYTES = D * ESZ;
  static constexpr int CH = ROW_BYTES / 128;            // 128-byte column chunks per row
  static constexpr int BOX = 128 / ESZ;                 // elements per TMA box row
  static constexpr int TILE_BYTES = TILE * ROW_BYTES;   // one tile of 128 rows
  static constexpr int KST = TILE_BYTES >= 32768 ? 2 : (FP8 ? 4 : 3);  // K ring stages
  static constexpr int VST = KST;                       // V ring stages
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + KST * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + VST * TILE_BYTES;
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 512 + 1024);  // + alignment slack
  static constexpr uint32_t O_COL = 256;            // TMEM: S0 @0, S1 @128, O0 @256, O1 @256+D
  static constexpr int THREADS = 384;
  // Register split: launched at 168 per thread (65536 / 384, rounded down to
  // a multiple of 8); warpgroup 0 (TMA, MMA, two idle warps) gives up
  // registers to the two softmax warpgroups: 128 * 56 + 256 * 224 = 384 * 168.
  static constexpr int LAUNCH_REGS = 168, REGS_LOW = 56, REGS_HIGH = 224;
};
static_assert(128 * 56 + 256 * 224 <= 384 * 168, "register split exceeds the launch allocation");

struct FwdBars {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort;
};

// Next kv tile >= J that at least one of the CTA's two Q tiles needs.
__device__ __forceinline__ int union_next(const AttnParams& p, int b, int I0, int J, int J_end) {
  while (J < J_end && tile_class(p, b, I0, J) == CLS_SKIP && tile_class(p, b, I0 + 1, J) == CLS_SKIP)
    ++J;
  return J;
}

// S = Q K^T over d: every MMA consumes 32 bytes of each row (16 bf16 or 32
// e4m3 elements), stepping through the 128-byte swizzled chunks.
template <int D, bool FP8>
__device__ __forceinline__ void issue_S(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t id = FP8 ? idesc_e4m3(128, 128, false, false) : idesc_bf16(128, 128, false, false);
  constexpr int KSTEPS = FwdCfg<D, FP8>::ROW_BYTES / 32;
  const uint64_t qd = sdesc_sw128(q_smem, 16, 1024), kd = sdesc_sw128(k_smem, 16, 1024);
#pragma unroll 1
  for (int kk = 0; kk < KSTEPS; ++kk) {
    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
    const uint64_t a = sdesc_add(qd, off), b = sdesc_add(kd, off);
    if (FP8)
      mma_f8_ss(d_tmem, a, b, id, kk > 0 ? 1u : 0u);
    else
      mma_f16_ss(d_tmem, a, b, id, kk > 0 ? 1u : 0u);
  }
}

// O += P V with P from TMEM (8 columns = 16 bf16 or 32 e4m3 keys per MMA).
template <int D, bool FP8>
__device__ __forceinline__ void issue_PV(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool first, bool with_lo) {
  constexpr uint32_t id = FP8 ? idesc_e4m3(128, D, false, true) : idesc_bf16(128, D, false, true);
  constexpr int KV = FP8 ? 32 : 16;
  const uint64_t vd = sdesc_sw128(v_smem, 16384, 1024);
#pragma unroll 1
  for (int kk = 0; kk < TILE / KV; ++kk) {
    const uint64_t bd = sdesc_add(vd, kk * KV * 128);
    if (FP8)
      mma_f8_ts(o_tmem, p_tmem + kk * 8, bd, id, (first && kk == 0) ? 0u : 1u);
    else
      mma_f16_ts(o_tmem, p_tmem + kk * 8, bd, id, (first && kk == 0) ? 0u : 1u);
  }
  if (!FP8 && with_lo) {
#pragma unroll 1
    for (int kk = 0; kk < TILE / 16; ++kk) {
      const uint64_t bd = sdesc_add(vd, kk * 16 * 128);
      mma_f16_ts(o_tmem, p_tmem + 64 + kk * 8, bd, id, 1u);
    }
  }
}

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
// the softmax scale in; 1 when s already holds log2-unit logits), packed to
// bf16 and written over S in TMEM (columns 0..63); with LO the rounding
// residual p - bf16(p) goes to columns 64..127.  Returns the row sum of P.
template <bool LO>
__device__ __forceinline__ float store_p(const uint32_t (&s)[128], float mul, float mu, uint32_t tS) {
  const uint64_t mul2 = f2_pack(mul, mul), nmu2 = f2_pack(-mu, -mu);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t ph[32];
    uint32_t pl[32];
#pragma unroll
    for (int w = 0; w < 32; ++w) {
      const int c = h * 64 + 2 * w;
      float y0, y1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), mul2, nmu2), y0, y1);
      const float p0 = ex2(y0), p1 = ex2(y1);
      acc[w & 3] = f2_add(acc[w & 3], f2_pack(p0, p1));
      ph[w] = pack_bf16(p0, p1);
      if (LO) pl[w] = pack_bf16(p0 - bf16lo_f32(ph[w]), p1 - bf16hi_f32(ph[w]));
    }
    tmem_st32(tS + h * 32, ph);
    if (LO) tmem_st32(tS + 64 + h * 32, pl);
  }
  return sum_acc(acc);
}

// P = 2^(mul * s - mu) rounded to e4m3 (nearest even, saturating), four per
// TMEM column, over S (columns 0..31).  Returns the row sum of the fp32 P.
__device__ __forceinline__ float store_p_e4m3(const uint32_t (&s)[128], float mul, float mu, uint32_t tS) {
  const uint64_t mul2 = f2_pack(mul, mul), nmu2 = f2_pack(-mu, -mu);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
  uint32_t pw[32];
#pragma unroll
  for (int w = 0; w < 32; ++w) {
    float y0, y1, y2, y3;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * w]), __uint_as_float(s[4 * w + 1])), mul2, nmu2), y0, y1);
    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * w + 2]), __uint_as_float(s[4 * w + 3])), mul2, nmu2), y2, y3);
    const float p0 = ex2(y0), p1 = ex2(y1), p2 = ex2(y2), p3 = ex2(y3);
    acc[(2 * w) & 3] = f2_add(acc[(2 * w) & 3], f2_pack(p0, p1));
    acc[(2 * w + 1) & 3] = f2_add(acc[(2 * w + 1) & 3], f2_pack(p2, p3));
    pw[w] = pack_e4m3x4(p0, p1, p2, p3);
  }
  tmem_st32(tS, pw);
  return sum_acc(acc);
}

template <int D, bool MODS, bool FP8>
__global__ void __launch_bounds__(384, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ o,
               float* __restrict__ lse, const float* __restrict__ scales, const AttnParams p) {
  using C = FwdCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  FwdBars& S = *reinterpret_cast<FwdBars*>(smem + C::BAR_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();

  // Work item, heaviest Q blocks first (longest-processing-time order).
  const int BH = p.B * p.Hq;
  const int qblk = p.n_qblk - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int hk = hq / (p.Hq / p.Hkv);
  const int I0 = 2 * qblk;
  const int J_end = (p.flags & MOD_CAUSAL) ? min(p.nT, I0 + 2) : p.nT;

  if (threadIdx.x == 0) {
    S.abort = 0;
    mbar_init(&S.q_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&S.k_full[s], 1);
      mbar_init(&S.k_empty[s], 1);
      mbar_init(&S.v_full[s], 1);
      mbar_init(&S.v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&S.s_full[t], 1);
      mbar_init(&S.p_full[t], 128);
      mbar_init(&S.o_full[t], 1);
    }
    mbar_init(&S.mma_drain, 1);
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
  const uint32_t sK = smem_u32(smem + C::K_OFF);
  const uint32_t sV = smem_u32(smem + C::V_OFF);

  if (warp < 4) regs_dec<C::REGS_LOW>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_tx(&S.q_full, 2 * C::TILE_BYTES);
      for (int t = 0; t < 2; ++t)
        for (int ch = 0; ch < C::CH; ++ch)
          tma_load_3d(smem + C::Q_OFF + t * C::TILE_BYTES + ch * 16384, &tq, &S.q_full, ch * C::BOX,
                      (I0 + t) * TILE, b * p.Hq + hq);
      int kit = 0, vit = 0;
      for (int J = union_next(p, b, I0, 0, J_end); J < J_end; J = union_next(p, b, I0, J + 1, J_end)) {
        const int ks = kit % C::KST;
        if (!mbar_wait(&S.k_empty[ks], ((kit / C::KST) & 1) ^ 1, ab)) break;
        mbar_arrive_tx(&S.k_full[ks], C::TILE_BYTES);
        for (int ch = 0; ch < C::CH; ++ch)
          tma_load_3d(smem + C::K_OFF + ks * C::TILE_BYTES + ch * 16384, &tk, &S.k_full[ks],
                      ch * C::BOX, J * TILE, b * p.Hkv + hk);
        ++kit;
        const int vs = vit % C::VST;
        if (!mbar_wait(&S.v_empty[vs], ((vit / C::VST) & 1) ^ 1, ab)) break;
        mbar_arrive_tx(&S.v_full[vs], C::TILE_BYTES);
        for (int ch = 0; ch < C::CH; ++ch)
          tma_load_3d(smem + C::V_OFF + vs * C::TILE_BYTES + ch * 16384, &tv, &S.v_full[vs],
                      ch * C::BOX, J * TILE, b * p.Hkv + hk);
        ++vit;
      }
      // Let every copy this thread issued land before the CTA can exit: the
      // last load into each stage completes phase ((n_loads - 1) & 1).
      mbar_wait_drain(&S.q_full, 0);
      for (int s = 0; s < C::KST; ++s)
        if (kit > s) mbar_wait_drain(&S.k_full[s], ((kit - 1 - s) / C::KST) & 1);
      for (int s = 0; s < C::VST; ++s)
        if (vit > s) mbar_wait_drain(&S.v_full[s], ((vit - 1 - s) / C::VST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int npv[2] = {0, 0};
      bool ok = mbar_wait(&S.q_full, 0, ab);
      tc_fence_after();
      int J = union_next(p, b, I0, 0, J_end);
      int c0 = 0, c1 = 0;
      if (ok && J < J_end) {
        c0 = tile_class(p, b, I0, J);
        c1 = tile_class(p, b, I0 + 1, J);
        ok = mbar_wait(&S.k_full[0], 0, ab);
        tc_fence_after();
        if (ok) {
          if (c0 != CLS_SKIP) { issue_S<D, FP8>(tmem + 0, sQ, sK); mma_commit(&S.s_full[0]); }
          if (c1 != CLS_SKIP) { issue_S<D, FP8>(tmem + 128, sQ + C::TILE_BYTES, sK); mma_commit(&S.s_full[1]); }
          mma_commit(&S.k_empty[0]);
        }
      }
      int it = 0;
      while (ok && J < J_end) {
        const int Jn = union_next(p, b, I0, J + 1, J_end);
        const bool has_next = Jn < J_end;
        const int n0 = has_next ? tile_class(p, b, I0, Jn) : CLS_SKIP;
        const int n1 = has_next ? tile_class(p, b, I0 + 1, Jn) : CLS_SKIP;
        const int vs = it % C::VST;
        const int ksn = (it + 1) % C::KST;
        const uint32_t vsm = sV + vs * C::TILE_BYTES;
        const uint32_t ksm = sK + ksn * C::TILE_BYTES;
        if (!(ok = mbar_wait(&S.v_full[vs], (it / C::VST) & 1, ab))) break;
        bool k_ready = false;
        if (c0 != CLS_SKIP) {
          if (!(ok = mbar_wait(&S.p_full[0], npv[0] & 1, ab))) break;
          tc_fence_after();
          issue_PV<D, FP8>(tmem + C::O_COL, tmem + 0, vsm, npv[0] == 0, c0 == CLS_PARTIAL);
          mma_commit(&S.o_full[0]);
          ++npv[0];
        }
        if (n0 != CLS_SKIP) {
          if (!(ok = mbar_wait(&S.k_full[ksn], ((it + 1) / C::KST) & 1, ab))) break;
          k_ready = true;
          tc_fence_after();
          issue_S<D, FP8>(tmem + 0, sQ, ksm);
          mma_commit(&S.s_full[0]);
        }
        if (c1 != CLS_SKIP) {
          if (!(ok = mbar_wait(&S.p_full[1], npv[1] & 1, ab))) break;
          tc_fence_after();
          issue_PV<D, FP8>(tmem + C::O_COL + D, tmem + 128, vsm, npv[1] == 0, c1 == CLS_PARTIAL);
          mma_commit(&S.o_full[1]);
          ++npv[1];
        }
        if (n1 != CLS_SKIP) {
          if (!k_ready) {
            if (!(ok = mbar_wait(&S.k_full[ksn], ((it + 1) / C::KST) & 1, ab))) break;
            tc_fence_after();
          }
          issue_S<D, FP8>(tmem + 128, sQ + C::TILE_BYTES, ksm);
          mma_commit(&S.s_full[1]);
        }
        if (has_next) mma_commit(&S.k_empty[ksn]);
        mma_commit(&S.v_empty[vs]);
        J = Jn;
        c0 = n0;
        c1 = n1;
        ++it;
      }
      // Every MMA this thread issued completes before TMEM can be released.
      mma_commit(&S.mma_drain);
      mbar_wait_drain(&S.mma_drain, 0);
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax
    regs_inc<C::REGS_HIGH>();
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int I = I0 + t;
    const int i = I * TILE + r;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + (uint32_t)t * 128;
    const uint32_t tO = tmem + lane_off + C::O_COL + (uint32_t)t * D;
    const bool causal = (p.flags & MOD_CAUSAL) != 0;
    // FP8: the scores are q8.k8 and need the Q and K dequantisation scales.
    const float qk_scale = FP8 ? p.scale * scales[b * p.Hq + hq] * scales[p.B * p.Hq + b * p.Hkv + hk]
                               : p.scale;
    const float scale_log2 = qk_scale * LOG2E;
    RowMods rm{};
    if (MODS) {
      rm.sc_in = qk_scale / p.softcap;
      rm.sc_out = p.softcap * LOG2E;
      rm.alibi_l2 = (p.flags & MOD_ALIBI) ? alibi_slope(p, hq) * LOG2E : 0.f;
      rm.doc_i = ((p.flags & MOD_DOC) && i < p.N) ? p.doc_ids[(size_t)b * p.N + i] : 0;
    }
    float m = -INFINITY, l = 0.f;
    int ns = 0;
    bool ok = true;
    for (int J = 0; J < J_end; ++J) {
      const int cls = tile_class(p, b, I, J);
      if (cls == CLS_SKIP) continue;
      if (!(ok = wait_warp(&S.s_full[t], ns & 1, ab))) break;
      tc_fence_after();
      uint32_t s[128];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        tmem_ld32(tS + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[q4 * 32]));
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&s[q4 * 32]));

      // Scores in log2 units, masked on partial tiles.
      const int j0 = J * TILE;
      const int hi_lim = min(causal ? i : 0x7fffffff, p.N - 1) - j0;  // valid iff c <= hi_lim
      float mt;   // tile row max in log2 units
      float mul;  // factor still to apply to s inside the exponential
      if (!MODS) {
        // Raw scores: the scale is positive, so it commutes with the max and
        // is folded into the exponential's FMA.
        if (cls == CLS_PARTIAL) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > hi_lim) s[c] = __float_as_uint(-INFINITY);
        }
        mt = row_max128(s) * scale_log2;
        mul = scale_log2;
      } else {
        mul = 1.0f;
        const bool sc = (p.flags & MOD_SOFTCAP) != 0;
        const bool al = (p.flags & MOD_ALIBI) != 0;
        const bool win = (p.flags & MOD_WINDOW) != 0;
        const bool doc = (p.flags & MOD_DOC) != 0;
        const float al_row = rm.alibi_l2 * (float)(j0 - i);
        const int lo_lim = win ? (i - p.window - j0) : -0x7fffffff;  // valid iff c > lo_lim
        const int* drow = doc ? p.doc_ids + (size_t)b * p.N + j0 : nullptr;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          float x = __uint_as_float(s[c]);
          x = sc ? tanh_exp(x * rm.sc_in) * rm.sc_out : x * scale_log2;
          if (al) x = fmaf(rm.alibi_l2, (float)c, x + al_row);
          if (cls == CLS_PARTIAL) {
            bool valid = (c <= hi_lim) && (c > lo_lim);
            if (doc && valid) valid = (__ldg(drow + c) == rm.doc_i);
            if (!valid) x = -INFINITY;
          }
          s[c] = __float_as_uint(x);
        }
        mt = row_max128(s);
      }

      // Running max; O is rescaled only when some row's max grew by > 2^8.
      const float mn = fmaxf(m, mt);
      if (ns == 0) {
        m = mn;
      } else {
        const bool need = mn > m + RESCALE_THRESHOLD;
        if (__any_sync(0xffffffffu, need)) {
          if (!(ok = wait_warp(&S.o_full[t], (ns - 1) & 1, ab))) break;
          tc_fence_after();
          const float alpha = need ? ex2(m - mn) : 1.0f;
          if (need) {
            l *= alpha;
            m = mn;
          }
#pragma unroll
          for (int q4 = 0; q4 < D / 32; ++q4) {
            uint32_t ov[32];
            tmem_ld32(tO + q4 * 32, ov);
            tmem_wait_ld(ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(tO + q4 * 32, ov);
          }
          tmem_wait_st();
        }
      }
      const float mu = (m == -INFINITY) ? 0.f : m;

      // P = 2^(x - m) as bf16 (hi, plus lo on partial tiles) over S in TMEM.
      if (FP8)
        l += store_p_e4m3(s, mul, mu, tS);
      else if (cls == CLS_PARTIAL)
        l += store_p<true>(s, mul, mu, tS);
      else
        l += store_p<false>(s, mul, mu, tS);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&S.p_full[t]);
      ++ns;
    }

    // ------------------------------------------------------------ epilogue
    if (ok && ns > 0) {
      ok = wait_warp(&S.o_full[t], (ns - 1) & 1, ab);
      tc_fence_after();
    }
    if (ok) {
      const float vscale = FP8 ? scales[p.B * p.Hq + p.B * p.Hkv + b * p.Hkv + hk] : 1.0f;
      const float inv = l > 0.f ? vscale / l : 0.f;
      __nv_bfloat16* orow = o + (((size_t)b * p.Hq + hq) * p.N + i) * D;
#pragma unroll
      for (int q4 = 0; q4 < D / 32; ++q4) {
        uint32_t ov[32];
        if (ns > 0) {
          tmem_ld32(tO + q4 * 32, ov);
          tmem_wait_ld(ov);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int w = 0; w < 16; ++w)
          pk[w] = pack_bf16(__uint_as_float(ov[2 * w]) * inv, __uint_as_float(ov[2 * w + 1]) * inv);
        if (i < p.N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + q4 * 32);
#pragma unroll
          for (int w = 0; w < 4; ++w)
            dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
        }
      }
      if (i < p.N)
        lse[((size_t)b * p.Hq + hq) * p.N + i] = l > 0.f ? (m + log2f(l)) * LN2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool MODS, bool FP8>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                void* o, float* lse, const float* scales, const AttnParams& p,
                                cudaStream_t st) {
  using C = FwdCfg<D, FP8>;
  auto kern = fwd_kernel<D, MODS, FP8>;
  // The register split inside the kernel assumes exactly LAUNCH_REGS per
  // thread at launch; refuse to launch any other build of it.
  static int regs = -1;
  if (regs < 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return cudaErrorInvalidDeviceFunction;
    regs = fa.numRegs;
  }
  if (regs != C::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(p.n_qblk * p.B * p.Hq));
  kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(tq, tk, tv, (__nv_bfloat16*)o, lse, scales, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_bf16(const FwdLaunch& L, int d, bool mods, cudaStream_t st) {
  if (d == 128)
    return mods ? launch_fwd_t<128, true, false>(L.tq, L.tk, L.tv, L.o, L.lse, nullptr, L.p, st)
                : launch_fwd_t<128, false, false>(L.tq, L.tk, L.tv, L.o, L.lse, nullptr, L.p, st);
  return mods ? launch_fwd_t<64, true, false>(L.tq, L.tk, L.tv, L.o, L.lse, nullptr, L.p, st)
              : launch_fwd_t<64, false, false>(L.tq, L.tk, L.tv, L.o, L.lse, nullptr, L.p, st);
}

cudaError_t launch_fwd_fp8(const Fp8Launch& L, bool mods, cudaStream_t st) {
  return mods ? launch_fwd_t<128, true, true>(L.tq, L.tk, L.tv, L.o, L.lse, L.scales, L.p, st)
              : launch_fwd_t<128, false, true>(L.tq, L.tk, L.tv, L.o, L.lse, L.scales, L.p, st);
}

}  // namespace attn
