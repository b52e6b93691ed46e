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
//  * warp 0 issues TMA loads (Q once; K and V through one 3-stage ring in the
//    order the MMAs consume them); warps 1 and 2 each issue the tcgen05 MMAs
//    of one Q tile from a single thread (the tensor pipe queues few MMAs, so
//    one issuer waiting on a barrier would leave it idle); warps 4-7 and 8-11
//    are the softmax warpgroups of Q tile 0 / 1;
//  * S and O live in TMEM (S0, S1, O0, O1: all 512 columns).  A softmax thread
//    (one row) copies its S row to registers and immediately hands the TMEM
//    columns back, so the MMA computes S(j+1) while the softmax of tile j is
//    still running; P is written to shared memory (128-byte swizzled K-major
//    tile) and P V is a shared-memory MMA.  The tensor pipe therefore never
//    waits for an exponential unless the softmax is slower than the GEMMs
//    (the FA3 digest's overlap of softmax and GEMM, done here with tcgen05's
//    asynchronous MMAs instead of warpgroup ping-pong);
//  * O is rescaled in TMEM only when a row max grows by more than 2^8 (lazy
//    rescale, exact after the final division by l), after the previous P V
//    has completed;
//  * on partial (masked) bf16 tiles P is split into bf16 hi + lo parts and both
//    are multiplied by V (lo read from TMEM), which removes the bf16 rounding
//    of P where few keys carry the whole row (the first rows of a causal
//    context); for those tiles S(j+1) is issued after P V;
//  * fully masked tiles are skipped (block-sparsity map, FlexAttention/FA4
//    page, "Limitations actuelles");
//  * the FP8 variant (FlashAttention-3 digest, "Basse précision FP8 et
//    incoherent processing") runs the same pipeline on e4m3 Q/K/V with
//    tcgen05.mma kind::f8f6f4 (twice the bf16 rate), rounds P to e4m3 for
//    P V, and folds the per-(batch, head) dequantisation scales into the
//    softmax scale (Q, K) and the epilogue (V).
#include "common.cuh"
#include "launch.h"
#include "softmax.cuh"

namespace attn {

template <int D, bool FP8>
struct FwdCfg {
  static constexpr int ESZ = FP8 ? 1 : 2;              // bytes per element
  static constexpr int ROW_BYTES = D * ESZ;             // one Q/K/V row
  static constexpr int CH = ROW_BYTES / 128;            // 128-byte column chunks per row
  static constexpr int BOX = 128 / ESZ;                 // elements per TMA box row
  static constexpr int TILE_BYTES = TILE * ROW_BYTES;   // one Q/K/V tile of 128 rows
  static constexpr int P_BYTES = TILE * TILE * ESZ;     // one P tile (128 x 128)
  static constexpr int RST = TILE_BYTES >= 32768 ? 3 : 4;  // K/V ring stages
  static constexpr int Q_OFF = 0;
  static constexpr int R_OFF = Q_OFF + 2 * TILE_BYTES;
  static constexpr int P_OFF = R_OFF + RST * TILE_BYTES;
  static constexpr int BAR_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 256 + 1024);  // + alignment slack
  static constexpr uint32_t O_COL = 256;  // TMEM: S0 @0, S1 @128, O0 @256, O1 @256+D
  static constexpr int THREADS = 384;
  // Register split: launched at 168 per thread (65536 / 384, rounded down to
  // a multiple of 8); warpgroup 0 (TMA, MMA, two idle warps) gives up
  // registers to the two softmax warpgroups.  bf16: 64 / 216 (the softmax
  // fits in 216 once the P residual is stored as soon as it is formed; the
  // issuing warps spilled at 56: 64 / 216 was 0.6-5.3 % faster than 56 / 224
  // on the GQA 8K, MHA 2K, flex and paged workloads).  e4m3: 56 / 216, with
  // no spills, 5.2 % faster than 40 / 232 (36 / 48 bytes of spills) on the
  // 16K FP8 workload.
  static constexpr int LAUNCH_REGS = 168, REGS_LOW = FP8 ? 56 : 64, REGS_HIGH = 216;
  static_assert(128 * REGS_LOW + 256 * REGS_HIGH <= 384 * LAUNCH_REGS, "register split exceeds the launch allocation");
};
static_assert(FwdCfg<128, false>::SMEM_BYTES <= 232448, "forward shared memory exceeds 227 KB");

struct FwdBars {
  uint64_t q_full;
  uint64_t full[4], empty[4];  // K/V ring
  uint64_t s_full[2];          // S_t computed (MMA commit)
  uint64_t s_free[2];          // S_t copied out of TMEM by the softmax (128 arrivals)
  uint64_t p_full[2];          // P_t written (128 arrivals)
  uint64_t o_full[2];          // P_t V done (MMA commit)
  uint64_t mma_drain[2];
  uint64_t never;              // test hook: a phase that nothing completes
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(FwdBars) <= 256, "barrier block");

// Next kv tile >= J that at least one of the CTA's two Q tiles needs.
__device__ __forceinline__ int union_next(const AttnParams& p, int b, int I0, int J, int J_end) {
  while (J < J_end && tile_class(p, b, I0, J) == CLS_SKIP && tile_class(p, b, I0 + 1, J) == CLS_SKIP)
    ++J;
  return J;
}

// D(tmem) = A B^T with A and B K-major 128-byte swizzled tiles in shared
// memory of `row_bytes` per row; every MMA consumes 32 bytes of each row (16
// bf16 or 32 e4m3 elements), stepping through the 16 KB column chunks.
template <bool FP8, int N, int ROW_BYTES>
__device__ __forceinline__ void issue_nt(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem,
                                         bool accumulate_first) {
  constexpr uint32_t id = FP8 ? idesc_e4m3(128, N, false, false) : idesc_bf16(128, N, false, false);
  const uint64_t ad = opaque(sdesc_sw128(a_smem, 16, 1024)), bd = opaque(sdesc_sw128(b_smem, 16, 1024));
#pragma unroll
  for (int kk = 0; kk < ROW_BYTES / 32; ++kk) {
    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
    const uint32_t acc = (kk > 0 || accumulate_first) ? 1u : 0u;
    if (FP8)
      mma_f8_ss(d_tmem, sdesc_add(ad, off), sdesc_add(bd, off), id, acc);
    else
      mma_f16_ss(d_tmem, sdesc_add(ad, off), sdesc_add(bd, off), id, acc);
  }
}

// O(tmem) += P V: P (shared memory, K-major, 128 keys) times V (shared
// memory, 128 keys x D, MN-major).  With LO (bf16 partial tiles) the rounding
// residual of P, packed in TMEM at lo_tmem, is added with A read from TMEM.
template <int D, bool FP8>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_smem, uint32_t v_smem,
                                         bool first, bool with_lo, uint32_t lo_tmem) {
  constexpr uint32_t id = FP8 ? idesc_e4m3(128, D, false, true) : idesc_bf16(128, D, false, true);
  constexpr int KV = FP8 ? 32 : 16;  // keys per MMA
  const uint64_t pd = opaque(sdesc_sw128(p_smem, 16, 1024)), vd = opaque(sdesc_sw128(v_smem, 16384, 1024));
#pragma unroll
  for (int kk = 0; kk < TILE / KV; ++kk) {
    const uint32_t poff = (kk / 4) * 16384 + (kk % 4) * 32;
    const uint64_t bd = sdesc_add(vd, kk * KV * 128);
    const uint32_t acc = (first && kk == 0) ? 0u : 1u;
    if (FP8)
      mma_f8_ss(o_tmem, sdesc_add(pd, poff), bd, id, acc);
    else
      mma_f16_ss(o_tmem, sdesc_add(pd, poff), bd, id, acc);
  }
  if (!FP8 && with_lo) {
#pragma unroll
    for (int kk = 0; kk < TILE / 16; ++kk)
      mma_f16_ts(o_tmem, lo_tmem + kk * 8, sdesc_add(vd, kk * 16 * 128), id, 1u);
  }
}

// Same for e4m3 P, in place: s[k] holds the codes of columns 4k..4k+3.
__device__ __forceinline__ float exp_e4m3(uint32_t (&s)[128], float mul, float mu) {
  const uint64_t mul2 = f2_pack(mul, mul), nmu2 = f2_pack(-mu, -mu);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    float y0, y1, y2, y3;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * k]), __uint_as_float(s[4 * k + 1])), mul2, nmu2), y0, y1);
    f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * k + 2]), __uint_as_float(s[4 * k + 3])), mul2, nmu2), y2, y3);
    const float p0 = ex2(y0), p1 = ex2(y1), p2 = ex2(y2), p3 = ex2(y3);
    acc[(2 * k) & 3] = f2_add(acc[(2 * k) & 3], f2_pack(p0, p1));
    acc[(2 * k + 1) & 3] = f2_add(acc[(2 * k + 1) & 3], f2_pack(p2, p3));
    s[k] = pack_e4m3x4(p0, p1, p2, p3);
  }
  return sum_acc(acc);
}

// Store this thread's P row (row r, `row_bytes` = 256 for bf16, 128 for e4m3)
// into the 128-byte swizzled K-major tile: 16-byte granule g of the row goes
// to chunk g / 8, row r, slot (g % 8) ^ (r % 8).
template <int NWORDS>
__device__ __forceinline__ void store_p_smem(uint8_t* tile, int r, const uint32_t (&w)[128]) {
#pragma unroll
  for (int g = 0; g < NWORDS / 4; ++g) {
    const uint32_t addr = (uint32_t)((g >> 3) * 16384 + r * 128 + (((g & 7) ^ (r & 7)) << 4));
    *reinterpret_cast<uint4*>(tile + addr) = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
  }
}

// Score mods of one row of a tile, in place, in log2 units: x = scale s, or
// the soft-cap c tanh(scale s / c); minus the ALiBi bias; -inf where the mask
// (column interval [lo_lim + 1, hi_lim], and the element-wise document test
// when drow is set) forbids the pair on partial tiles.  fp32 arithmetic two
// lanes per instruction.
struct ModsArgs {
  float scale_log2, sc_in, sc_out, alibi_l2, al_row;
  int hi_lim, lo_lim;
  const int* drow;  // document ids of the tile's columns, element-wise test
  int doc_i;
  bool partial;
};
template <bool SC, bool AL>
__device__ __forceinline__ void score_mods(uint32_t (&s)[128], const ModsArgs& a) {
  const uint64_t sl2 = f2_pack(a.scale_log2, a.scale_log2);
  const uint64_t sc_in2 = f2_pack(a.sc_in, a.sc_in), sc_out2 = f2_pack(a.sc_out, a.sc_out);
  const uint64_t al2 = f2_pack(a.alibi_l2, a.alibi_l2), al_row2 = f2_pack(a.al_row, a.al_row);
#pragma unroll
  for (int c = 0; c < 128; c += 2) {
    uint64_t x2 = f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    if (SC)
      x2 = f2_mul(tanh2_exp(f2_mul(x2, sc_in2)), sc_out2);
    else
      x2 = f2_mul(x2, sl2);
    if (AL) x2 = f2_fma(f2_pack((float)c, (float)(c + 1)), al2, f2_add(x2, al_row2));
    float x0, x1;
    f2_unpack(x2, x0, x1);
    s[c] = __float_as_uint(x0);
    s[c + 1] = __float_as_uint(x1);
  }
  if (a.partial) {
#pragma unroll
    for (int c = 0; c < 128; ++c) {
      bool valid = (c <= a.hi_lim) && (c > a.lo_lim);
      if (a.drow != nullptr && valid) valid = (__ldg(a.drow + c) == a.doc_i);
      if (!valid) s[c] = __float_as_uint(-INFINITY);
    }
  }
}

// MODS: soft-cap / ALiBi score mods compiled in; MASKS: window / document
// masks compiled in (causal and the sequence end always are); PAGED: K and V
// read through a block table.
template <int D, bool MODS, bool FP8, bool MASKS, bool PAGED>
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

  // Work item.  Causal or masked launches: heaviest Q blocks first
  // (longest-processing-time order), heads interleaved.  Otherwise every Q
  // block costs the same, and the Q blocks of a head -- and the query heads of
  // a KV head -- run one after another, so the CTAs in flight share few heads'
  // K and V and L2 keeps them (32 heads of 16K keys are 128 MB of e4m3 K/V).
  const int BH = p.B * p.Hq;
  int qblk, bh;
  if (MASKS || (p.flags & MOD_CAUSAL)) {
    qblk = p.n_qblk - 1 - (int)(blockIdx.x / BH);
    bh = (int)(blockIdx.x % BH);
  } else {
    bh = (int)(blockIdx.x / p.n_qblk);
    qblk = (int)(blockIdx.x % p.n_qblk);
  }
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int hk = hq / (p.Hq / p.Hkv);
  const int I0 = 2 * qblk;
  // KV tiles [J_begin, J_end) cover every non-skipped tile of both Q tiles.
  const int2 rg0 = MASKS ? q_tile_range(p, b, I0) : make_int2(0, p.nT);
  const int2 rg1 = MASKS ? q_tile_range(p, b, I0 + 1) : make_int2(0, p.nT);
  const int J_begin = min(rg0.y > rg0.x ? rg0.x : p.nT, rg1.y > rg1.x ? rg1.x : p.nT);
  const int J_end = min((p.flags & MOD_CAUSAL) ? min(p.nT, I0 + 2) : p.nT, max(rg0.y, rg1.y));

  if (threadIdx.x == 0) {
    S.abort = 0;
    mbar_init(&S.q_full, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 2);  // one commit from each MMA issuer
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&S.s_full[t], 1);
      mbar_init(&S.s_free[t], 128);
      mbar_init(&S.p_full[t], 128);
      mbar_init(&S.o_full[t], 1);
    }
    mbar_init(&S.mma_drain[0], 1);
    mbar_init(&S.mma_drain[1], 1);
    mbar_init(&S.never, 1);
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
  const uint32_t sR = smem_u32(smem + C::R_OFF);
  const uint32_t sP = smem_u32(smem + C::P_OFF);

  if (warp < 4) regs_dec<C::REGS_LOW>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Ring order = consumption order: K(J0), then per union tile J:
    // K(next J) before V(J).
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_tx(&S.q_full, 2 * C::TILE_BYTES);
      for (int t = 0; t < 2; ++t)
        for (int ch = 0; ch < C::CH; ++ch)
          tma_load_3d(smem + C::Q_OFF + t * C::TILE_BYTES + ch * 16384, &tq, &S.q_full, ch * C::BOX,
                      (I0 + t) * TILE, b * p.Hq + hq);
    }
    // Both walks issue K(J0), then per union tile J: K(next J), V(J).  The
    // last load into each stage completes phase ((loads into it - 1) & 1):
    // lane 0 waits for all of them before the CTA can exit.
    int r = 0;
    auto drain = [&]() {
      mbar_wait_drain(&S.q_full, 0);
      for (int s = 0; s < C::RST; ++s)
        if (r > s) mbar_wait_drain(&S.full[s], ((r - 1 - s) / C::RST) & 1);
    };
    if (!PAGED) {
      // Contiguous K/V: lane 0 issues one box per 64-column chunk of a tile.
      if (lane == 0) {
        auto load = [&](const CUtensorMap* map, int J) -> bool {
          const int st = r % C::RST;
          if (!mbar_wait(&S.empty[st], ((r / C::RST) & 1) ^ 1, ab)) return false;
          mbar_arrive_tx(&S.full[st], C::TILE_BYTES);
          uint8_t* dst = smem + C::R_OFF + st * C::TILE_BYTES;
          for (int ch = 0; ch < C::CH; ++ch)
            tma_load_3d(dst + ch * 16384, map, &S.full[st], ch * C::BOX, J * TILE, b * p.Hkv + hk);
          ++r;
          return true;
        };
        int J = union_next(p, b, I0, J_begin, J_end);
        bool ok = J >= J_end || load(&tk, J);
        while (ok && J < J_end) {
          const int Jn = union_next(p, b, I0, J + 1, J_end);
          if (Jn < J_end && !(ok = load(&tk, Jn))) break;
          if (!(ok = load(&tv, J))) break;
          J = Jn;
        }
        drain();
      }
    } else {
      // Paged K/V: the tile's 8 blocks of 16 rows, each a 16-row box at its 2 KB
      // offset (the 128-byte swizzle repeats every 8 rows, so the layout
      // matches a whole-tile load), one box per lane of the warp -- small
      // boxes cost per box, so one thread issuing all of them would limit the
      // stream.  Each lane fetches its table entry while lane 0 waits for the
      // slot.  Blocks past the sequence end use an out-of-range block index:
      // TMA fills them with zeros.
      auto load = [&](const CUtensorMap* map, int J) -> bool {
        const int st = r % C::RST;
        int z = p.kv_blocks * p.Hkv;
        if (lane < 8 * C::CH) {
          const int lb = J * (TILE / 16) + lane / C::CH;
          if (lb < p.bt_stride) z = __ldg(p.block_table + (size_t)b * p.bt_stride + lb) * p.Hkv + hk;
        }
        bool good = true;
        if (lane == 0) {
          good = mbar_wait(&S.empty[st], ((r / C::RST) & 1) ^ 1, ab);
          if (good) mbar_arrive_tx(&S.full[st], C::TILE_BYTES);
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) return false;
        if (lane < 8 * C::CH)
          tma_load_3d(smem + C::R_OFF + st * C::TILE_BYTES + (lane % C::CH) * 16384 + (lane / C::CH) * 2048, map,
                      &S.full[st], (lane % C::CH) * C::BOX, 0, z);
        ++r;
        return true;
      };
      int J = union_next(p, b, I0, J_begin, J_end);
      bool ok = J >= J_end || load(&tk, J);
      while (ok && J < J_end) {
        const int Jn = union_next(p, b, I0, J + 1, J_end);
        if (Jn < J_end && !(ok = load(&tk, Jn))) break;
        if (!(ok = load(&tv, J))) break;
        J = Jn;
      }
      if (lane == 0) drain();
    }
  } else if (warp == 1 || warp == 2) {
    // ---------------------------------------------------------- MMA issuers
    // One issuing thread per Q tile (warp 1: tile 0, warp 2: tile 1).  The
    // tensor pipe queues few MMAs, so a thread that waits on a barrier leaves
    // it idle; two independent issuers keep it fed while either one waits.
    if (lane == 0) {
      const int t = warp - 1;
      const int I = I0 + t;
      const uint32_t s_tm = tmem + (uint32_t)t * 128;
      const uint32_t o_tm = tmem + C::O_COL + (uint32_t)t * D;
      const uint32_t q_sm = sQ + t * C::TILE_BYTES;
      const uint32_t p_sm = sP + t * C::P_BYTES;
      bool ok = mbar_wait(&S.q_full, 0, ab);
      tc_fence_after();
      int r = 0;    // ring slots consumed
      int nk = 0;   // S tiles issued
      int npv = 0;  // P V issued
      auto slot = [&](int& st) -> bool {  // wait for the next ring slot
        st = r % C::RST;
        const bool good = mbar_wait(&S.full[st], (r / C::RST) & 1, ab);
        ++r;
        tc_fence_after();
        return good;
      };
      auto issue_S = [&](uint32_t k_sm) {
        issue_nt<FP8, 128, C::ROW_BYTES>(s_tm, q_sm, k_sm, false);
        mma_commit(&S.s_full[t]);
        ++nk;
      };
      int J = union_next(p, b, I0, J_begin, J_end);
      int c = CLS_SKIP;
      // Half-period offset of Q tile 1 in long CTAs: its first S waits until
      // Q tile 0's softmax has produced its first P, so that tile 1's GEMMs run
      // while tile 0's exponentials do.  Left alone, the two tiles share every
      // K/V slot and run in lockstep: both softmax warpgroups compute at once
      // while the tensor pipe idles (clock stamps on the GQA 8K workload:
      // both S issued within 2 cycles of each other, 3950 cycles per KV tile
      // for 2048 of MMA).  The offset decays over some 25 KV tiles as the
      // shared ring pulls the tiles together again, and costs half a period at
      // the start, so short CTAs keep the plain start (measured: GQA 8K
      // forward -4.0 %, MHA 2K and flex workloads unchanged).
      if (ok && J < J_end) {
        int ks;
        ok = slot(ks);
        c = tile_class(p, b, I, J);
        if (ok && t == 1 && J_end - J_begin >= 24 && c != CLS_SKIP && tile_class(p, b, I0, J) != CLS_SKIP)
          ok = mbar_wait(&S.p_full[0], 0, ab);
        if (ok) {
          if (c != CLS_SKIP) issue_S(sR + ks * C::TILE_BYTES);
          mma_commit(&S.empty[ks]);
        }
      }
      while (ok && J < J_end) {
        const int Jn = union_next(p, b, I0, J + 1, J_end);
        const bool has_next = Jn < J_end;
        const int n = has_next ? tile_class(p, b, I, Jn) : CLS_SKIP;
        // Partial bf16 tiles keep their P residual in the S columns: their
        // S(Jn) goes after P V.
        const bool late = !FP8 && c == CLS_PARTIAL;
        int ks = 0, vs = 0;
        if (has_next) {
          if (!(ok = slot(ks))) break;
          // Early S(Jn): the S columns are free once the softmax copied S(J)
          // out (at once if this tile skipped J).
          if (n != CLS_SKIP && !late) {
            if (c != CLS_SKIP) {
              if (!(ok = mbar_wait(&S.s_free[t], (nk - 1) & 1, ab))) break;
              tc_fence_after();
            }
            issue_S(sR + ks * C::TILE_BYTES);
          }
          if (!late) mma_commit(&S.empty[ks]);
        }
        if (!(ok = slot(vs))) break;
        if (c != CLS_SKIP) {
          if (!(ok = mbar_wait(&S.p_full[t], npv & 1, ab))) break;
          tc_fence_after();
          issue_pv<D, FP8>(o_tm, p_sm, sR + vs * C::TILE_BYTES, npv == 0, c == CLS_PARTIAL, s_tm);
          mma_commit(&S.o_full[t]);
          ++npv;
          if (late && n != CLS_SKIP) {
            if (!(ok = mbar_wait(&S.s_free[t], (nk - 1) & 1, ab))) break;
            tc_fence_after();
            issue_S(sR + ks * C::TILE_BYTES);
          }
        }
        if (has_next && late) mma_commit(&S.empty[ks]);
        mma_commit(&S.empty[vs]);
        J = Jn;
        c = n;
      }
      // Every MMA this thread issued completes before TMEM can be released.
      mma_commit(&S.mma_drain[t]);
      mbar_wait_drain(&S.mma_drain[t], 0);
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
    uint8_t* p_tile = smem + C::P_OFF + t * C::P_BYTES;
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
    }
    const bool win = MASKS && (p.flags & MOD_WINDOW) != 0;
    const bool doc = MASKS && (p.flags & MOD_DOC) != 0;
    rm.doc_i = (doc && i < p.N) ? p.doc_ids[(size_t)b * p.N + i] : 0;
    rm.doc_runs = false;
    rm.doc_run = make_int2(0, p.N);
    if (doc) rm.doc_run = doc_run(p, b, i, rm.doc_runs);
    const bool doc_each = doc && !rm.doc_runs;  // ids tested element by element
    float m = -INFINITY, l = 0.f;
    int ns = 0;
    bool ok = true;
    // Test hook: the first tile's warpgroup waits on a phase nothing completes,
    // runs into the launch's limit and raises the abort word; every later wait
    // of the grid then gives up, and the kernel drains (attn_test_hooks).
    if ((p.stall & STALL_FWD) && t == 0) ok = wait_warp(&S.never, 0, ab, p.wait_ns);
    for (int J = J_begin; J < J_end; ++J) {
      const int cls = tile_class(p, b, I, J);
      if (cls == CLS_SKIP) continue;
      const bool partial = cls == CLS_PARTIAL;
      if (!(ok = wait_warp(&S.s_full[t], ns & 1, ab))) break;
      tc_fence_after();
      uint32_t s[128];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        tmem_ld32(tS + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[q4 * 32]));
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&s[q4 * 32]));
      if (!partial || FP8) {  // S is in registers: hand the columns back to the MMA
        tc_fence_before();
        mbar_arrive(&S.s_free[t]);
      }

      // Scores in log2 units, masked on partial tiles.
      const int j0 = J * TILE;
      const int hi_lim = min(causal ? i : 0x7fffffff, p.N - 1) - j0;  // valid iff c <= hi_lim
      float mt;   // tile row max in log2 units
      float mul;  // factor still to apply to s inside the exponential
      // Allowed columns of this row on a partial tile: (lo_lim, hi_m] (causal,
      // the sequence end, the window, the row's document run), plus the
      // element-wise document test when the ids are not runs.
      int lo_lim = win ? (i - p.window - j0) : -0x7fffffff;  // valid iff c > lo_lim
      int hi_m = hi_lim;                                      // valid iff c <= hi_m
      if (doc && rm.doc_runs) {
        lo_lim = max(lo_lim, rm.doc_run.x - 1 - j0);
        hi_m = min(hi_m, rm.doc_run.y - 1 - j0);
      }
      const int* drow = doc ? p.doc_ids + (size_t)b * p.N + j0 : nullptr;
      if (!MODS) {
        // Raw scores: the scale is positive, so it commutes with the max and
        // is folded into the exponential's FMA.
        if (partial) {
          if (!doc_each) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > hi_m || c <= lo_lim) s[c] = __float_as_uint(-INFINITY);
          } else {
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              const bool valid = c <= hi_m && c > lo_lim && __ldg(drow + c) == rm.doc_i;
              if (!valid) s[c] = __float_as_uint(-INFINITY);
            }
          }
        }
        mt = row_max128(s) * scale_log2;
        mul = scale_log2;
      } else {
        mul = 1.0f;
        const bool sc = (p.flags & MOD_SOFTCAP) != 0;
        const bool al = (p.flags & MOD_ALIBI) != 0;
        // The score mods in log2 units, specialised on soft-cap / ALiBi so the
        // unrolled loop carries no dead work.
        const float al_row = rm.alibi_l2 * (float)(j0 - i);
        const ModsArgs ma{scale_log2, rm.sc_in, rm.sc_out, rm.alibi_l2, al_row, hi_m, lo_lim,
                          doc_each ? drow : nullptr, rm.doc_i, partial};
        if (sc && al) score_mods<true, true>(s, ma);
        else if (sc) score_mods<true, false>(s, ma);
        else if (al) score_mods<false, true>(s, ma);
        else score_mods<false, false>(s, ma);
        mt = row_max128(s);
      }

      // Running max: it moves only when some row's max grew by > 2^8.
      const float mn = fmaxf(m, mt);
      bool need = false;
      float alpha = 1.0f;
      if (ns == 0) {
        m = mn;
      } else {
        need = mn > m + RESCALE_THRESHOLD;
        if (need) {
          alpha = ex2(m - mn);
          l *= alpha;
          m = mn;
        }
      }
      const float mu = (m == -INFINITY) ? 0.f : m;

      // P into registers (the previous P V may still be reading P's buffer).
      uint32_t lo[64];
      if (FP8)
        l += exp_e4m3(s, mul, mu);
      else if (partial) {
        l += exp_bf16<true>(s, lo, mul, mu);
        // The residual of P into the S columns (this warpgroup's until it
        // releases them below), for the TS MMA: stored now, so that it is not
        // live in registers across the wait and the rescale.
        tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&lo[0]));
        tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&lo[32]));
      } else
        l += exp_bf16<false>(s, lo, mul, mu);

      // The previous P V must be done before O is rescaled or P overwritten.
      if (ns > 0) {
        if (!(ok = wait_warp(&S.o_full[t], (ns - 1) & 1, ab))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int q4 = 0; q4 < D / 32; ++q4) {
            uint32_t ov[32];
            tmem_ld32(tO + q4 * 32, ov);
            tmem_wait_ld(ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(tO + q4 * 32, ov);
          }
        }
      }
      if (FP8) {
        store_p_smem<32>(p_tile, r, s);
      } else {
        store_p_smem<64>(p_tile, r, s);
      }
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
      if (partial && !FP8) mbar_arrive(&S.s_free[t]);
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

template <int D, bool MODS, bool FP8, bool MASKS, bool PAGED = false>
static cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                void* o, float* lse, const float* scales, const AttnParams& p,
                                cudaStream_t st) {
  using C = FwdCfg<D, FP8>;
  auto kern = fwd_kernel<D, MODS, FP8, MASKS, PAGED>;
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

cudaError_t launch_fwd_bf16(const FwdLaunch& L, int d, bool mods, bool masks, cudaStream_t st) {
#define ATTN_FWD(DD, MO, MA) launch_fwd_t<DD, MO, false, MA>(L.tq, L.tk, L.tv, L.o, L.lse, nullptr, L.p, st)
#define ATTN_FWDP(DD, MO, MA) launch_fwd_t<DD, MO, false, MA, true>(L.tq, L.tk, L.tv, L.o, L.lse, nullptr, L.p, st)
  if (L.p.block_table != nullptr) {  // paged K/V
    if (d == 128)
      return mods ? ATTN_FWDP(128, true, true) : masks ? ATTN_FWDP(128, false, true) : ATTN_FWDP(128, false, false);
    return mods ? ATTN_FWDP(64, true, true) : masks ? ATTN_FWDP(64, false, true) : ATTN_FWDP(64, false, false);
  }
  if (d == 128) return mods ? ATTN_FWD(128, true, true) : masks ? ATTN_FWD(128, false, true) : ATTN_FWD(128, false, false);
  return mods ? ATTN_FWD(64, true, true) : masks ? ATTN_FWD(64, false, true) : ATTN_FWD(64, false, false);
#undef ATTN_FWDP
#undef ATTN_FWD
}

cudaError_t launch_fwd_fp8(const Fp8Launch& L, bool mods, bool masks, cudaStream_t st) {
#define ATTN_FWD8(MO, MA) launch_fwd_t<128, MO, true, MA>(L.tq, L.tk, L.tv, L.o, L.lse, L.scales, L.p, st)
  return mods ? ATTN_FWD8(true, true) : masks ? ATTN_FWD8(false, true) : ATTN_FWD8(false, false);
#undef ATTN_FWD8
}

}  // namespace attn
