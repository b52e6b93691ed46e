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
//    in shared memory; Q tiles (3-slot TMA ring) and dO tiles (2-slot ring) of
//    every query head of the GQA group and every needed Q tile stream past
//    them.  S^T = K Q^T and dP^T = V dO^T land in TMEM regions of their own;
//    two softmax warpgroups (a thread per KV row, 64 query columns each) turn
//    them into P^T and dS^T, packed bf16 into the dP^T region; dV += P^T dO
//    and dK += dS^T Q read their A operand from TMEM.
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
#include "bwd_common.cuh"
#include "launch.h"

namespace attn {

// ================================================================== dK, dV
// e4m3 P^T of the mixed backward is P * P8_MUL: P <= 1 stays below the e4m3
// maximum (448), and P down to 2^-17 stays above its smallest subnormal.
constexpr float P8_MUL = 256.f;

// Shared memory: K_J, V_J, a 3-slot Q ring and a 2-slot dO ring.  TMEM (512 columns):
//   XS  [0, 128)        S^T(n), copied to registers and handed back at once
//   XD  [128, 256)      dP^T(n); then, per softmax warpgroup w (query columns
//                       [64 w, 64 w + 64)), packed bf16 dS^T(n) at columns
//                       [64 w, 64 w + 32) (A of dK += dS^T Q) and P^T(n) at
//                       [64 w + 32, 64 w + 64) (A of dV += P^T dO)
//   dV  [256, 256 + D), dK [256 + D, 256 + 2D)  fp32 accumulators
// A warpgroup writes only columns it has already loaded, so it overwrites
// nothing the other has yet to read.  The tensor pipe runs one CTA's MMAs in
// issue order, so dP^T(n+1) may be issued right behind dK(n), the last reader
// of the region.  Because P^T does not stay in XS, S^T(n+1) is computed while
// the softmax works on P(n); per step the softmax waits for one GEMM only,
// dP^T.  (P^T in place over S^T kept S^T(n+1) waiting for the exponentials of
// P(n): 3660 cycles a step against 2048 of MMA.)
// FP8 (the mixed e4m3 backward): V and dO tiles are e4m3 (128-byte rows, one
// TMA box each), and P^T goes to an e4m3 shared-memory tile, the A operand of
// the e4m3 dV GEMM.
template <int D, bool FP8 = false>
struct KvCfg {
  static constexpr int CH = D / 64;
  static constexpr int TB = TILE * D * 2;
  static constexpr int VB = FP8 ? TILE * D : TB;  // one V or dO tile
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TB;
  // Q tiles in a 3-slot ring (last read by dK, the step's final GEMM) and dO
  // tiles in a 2-slot ring (last read by dV): the load of Q(n+1) never waits
  // for dK(n-1), which runs late in step n.
  static constexpr int QS = 3, DOS = 2;
  static constexpr int Q_OFF = TB + VB;
  static constexpr int DO_OFF = Q_OFF + QS * TB;
  static constexpr int P8_OFF = DO_OFF + DOS * VB;             // e4m3 P^T tile (FP8 only)
  static constexpr int BAR_OFF = P8_OFF + (FP8 ? TILE * TILE : 0);
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 256 + 1024);
};
static_assert(KvCfg<128>::SMEM_BYTES <= 232448, "dK/dV shared memory exceeds 227 KB");
static_assert(KvCfg<128, true>::SMEM_BYTES <= 232448, "dK/dV shared memory exceeds 227 KB");

struct KvBars {
  uint64_t in_full;              // K_J, V_J
  uint64_t qfull[3], qempty[3];  // Q ring
  uint64_t dfull[2];             // dO ring (a slot is free once qempty shows its step's dK done)
  uint64_t s_full;             // S^T(n) in XS               (MMA commit)
  uint64_t xs_free;            // S^T(n) copied out of XS    (256 softmax threads)
  uint64_t dp_full;            // dP^T(n) in XD              (MMA commit)
  uint64_t p_full;             // P^T(n) stored in XD        (256)
  uint64_t ds_full;            // dS^T(n) stored in XD       (256)
  uint64_t fin;                // every MMA of the dV / dK / dP^T issuer done
  uint64_t fin_s;              // every MMA of the S^T issuer done
  uint64_t never;              // test hook: a phase that nothing completes
  uint32_t tmem_base;
  int abort;
};

// Steps of a dK/dV CTA: non-skipped Q tile I (outer, ascending), query head
// g of the group (inner).
struct KvSteps {
  int J, I_first, I_end, G;  // Q tiles of the KV tile: [I_first, I_end), skipped ones passed over
  __device__ __forceinline__ int next_I(const AttnParams& p, int b, int I) const {
    while (I < I_end && tile_class(p, b, I, J) == CLS_SKIP) ++I;
    return I < I_end ? I : p.nT;
  }
  // Advance (g, I) to the next step; false when past the last one.  The query
  // heads of the group are the inner loop.  Measured on the causal GQA 8K
  // workload against Q tiles inner: 1.8 % less time, although the Q / dO
  // tiles in use at once then span every head and DRAM reads rise from 0.85
  // to 1.43 GB per launch (0.79 TB/s, about an eighth of the HBM rate).
  __device__ __forceinline__ bool advance(const AttnParams& p, int b, int& g, int& I) const {
    if (++g < G) return true;
    g = 0;
    I = next_I(p, b, I + 1);
    return I < p.nT;
  }
};

// MODS: soft-cap / ALiBi compiled in; MASKS: window / document masks.  FP8:
// the mixed e4m3 backward (d = 128, no score mods, no window / document
// masks): tv and tdo map the e4m3 V and dO, fp8s holds their dequantisation
// scales ([B * Hkv] of dO, then [B * Hkv] of V); dP^T and dV run as e4m3 GEMMs,
// P^T rounded to e4m3 after scaling by P8_MUL, dS and dK stay bf16.
template <int D, bool MODS, bool MASKS, bool FP8 = false>
__global__ void __launch_bounds__(384, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const float2* __restrict__ rowstat, __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, const AttnParams p, const float* __restrict__ fp8s) {
  static_assert(!FP8 || (D == 128 && !MODS && !MASKS), "the e4m3 backward has d = 128 and no mods");
  using C = KvCfg<D, FP8>;
  // The dQ kernel that follows reads nothing this kernel writes: once every
  // CTA of this grid has started, its CTAs may take the SMs this grid's last
  // CTAs leave idle.
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  KvBars& S = *reinterpret_cast<KvBars*>(smem + C::BAR_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();

  const int BHk = p.B * p.Hkv;
  const int J = (int)(blockIdx.x / BHk);  // smallest KV tile (most work under causal) first
  const int bh = (int)(blockIdx.x % BHk);
  const int b = bh / p.Hkv, hk = bh - b * p.Hkv;
  const int G = p.Hq / p.Hkv;
  const bool causal = (p.flags & MOD_CAUSAL) != 0;
  const int2 rg = MASKS ? kv_tile_range(p, b, J) : make_int2(0, p.nT);
  KvSteps steps{J, 0, MASKS ? min(p.nT, rg.y) : p.nT, G};
  steps.I_first = steps.next_I(p, b, max(causal ? J : 0, rg.x));
  const bool any = steps.I_first < p.nT;

  if (threadIdx.x == 0) {
    S.abort = 0;
    mbar_init(&S.in_full, 1);
    for (int s = 0; s < C::QS; ++s) {
      mbar_init(&S.qfull[s], 1);
      mbar_init(&S.qempty[s], 1);
    }
    for (int s = 0; s < C::DOS; ++s) mbar_init(&S.dfull[s], 1);
    mbar_init(&S.s_full, 1);
    mbar_init(&S.xs_free, 256);
    mbar_init(&S.dp_full, 1);
    mbar_init(&S.p_full, 256);
    mbar_init(&S.ds_full, 256);
    mbar_init(&S.fin, 1);
    mbar_init(&S.fin_s, 1);
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
  const uint32_t sK = smem_u32(smem + C::K_OFF);
  const uint32_t sV = smem_u32(smem + C::V_OFF);
  const uint32_t sQ = smem_u32(smem + C::Q_OFF);
  const uint32_t sDO = smem_u32(smem + C::DO_OFF);
  const uint32_t tXS = tmem, tXD = tmem + 128;
  const uint32_t sP8 = smem_u32(smem + C::P8_OFF);
  const uint32_t tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp < 4) regs_dec<BWD_REGS_LOW>();
  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      mbar_arrive_tx(&S.in_full, C::TB + C::VB);
      for (int ch = 0; ch < C::CH; ++ch) {
        tma_load_3d(smem + C::K_OFF + ch * 16384, &tk, &S.in_full, ch * 64, J * TILE, b * p.Hkv + hk);
        if (!FP8)
          tma_load_3d(smem + C::V_OFF + ch * 16384, &tv, &S.in_full, ch * 64, J * TILE, b * p.Hkv + hk);
      }
      if (FP8) tma_load_3d(smem + C::V_OFF, &tv, &S.in_full, 0, J * TILE, b * p.Hkv + hk);
      int nq = 0, nd = 0;  // Q / dO loads issued
      if (any) {
        int g = 0, I = steps.I_first;
        do {
          const int hq = hk * G + g;
          const int qs = nq % C::QS, ds = nd % C::DOS;
          if (!mbar_wait(&S.qempty[qs], ((nq / C::QS) & 1) ^ 1, ab)) break;
          mbar_arrive_tx(&S.qfull[qs], C::TB);
          for (int ch = 0; ch < C::CH; ++ch)
            tma_load_3d(smem + C::Q_OFF + qs * C::TB + ch * 16384, &tq, &S.qfull[qs], ch * 64, I * TILE,
                        b * p.Hq + hq);
          ++nq;
          // dO(nd) goes over dO(nd - 2): read by dP^T and dV of step nd - 2,
          // both done once that step's dK is (issue order; one commit fewer a step).
          if (nd >= C::DOS && !mbar_wait(&S.qempty[(nd - C::DOS) % C::QS], ((nd - C::DOS) / C::QS) & 1, ab)) break;
          mbar_arrive_tx(&S.dfull[ds], C::VB);
          if (FP8)
            tma_load_3d(smem + C::DO_OFF + ds * C::VB, &tdo, &S.dfull[ds], 0, I * TILE, b * p.Hq + hq);
          else
            for (int ch = 0; ch < C::CH; ++ch)
              tma_load_3d(smem + C::DO_OFF + ds * C::TB + ch * 16384, &tdo, &S.dfull[ds], ch * 64, I * TILE,
                          b * p.Hq + hq);
          ++nd;
        } while (steps.advance(p, b, g, I));
      }
      // Loads still in flight must land before the CTA exits.
      mbar_wait_drain(&S.in_full, 0);
      for (int s = 0; s < C::QS; ++s)
        if (nq > s) mbar_wait_drain(&S.qfull[s], ((nq - 1 - s) / C::QS) & 1);
      for (int s = 0; s < C::DOS; ++s)
        if (nd > s) mbar_wait_drain(&S.dfull[s], ((nd - 1 - s) / C::DOS) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer: dV, dK, dP^T
    // Per step n: dV(n) once P^T(n) is stored, then dK(n) and dP(n+1) once
    // dS^T(n) is.  dP^T(n+1) overwrites XD behind the two GEMMs that read it
    // (issue order), and one thread issuing every accumulation fixes their
    // order.  The S^T chain has a thread of its own (warp 2): the tensor pipe
    // queues few MMAs, and one thread issuing both chains answered each
    // softmax hand-off only after issuing the other chain's GEMMs (4000 cycles
    // a step, 3050 of them spent issuing).
    if (lane == 0) {
      bool ok = mbar_wait(&S.in_full, 0, ab);
      tc_fence_after();
      if (ok && any) {
        int g = 0, I = steps.I_first, n = 0;
        auto q_at = [&](int m) { return sQ + (uint32_t)((m % C::QS) * C::TB); };
        auto do_at = [&](int m) { return sDO + (uint32_t)((m % C::DOS) * C::VB); };
        // dP^T(m) = V dO(m)^T into XD.
        auto issue_dp = [&](int m) -> bool {
          if (!mbar_wait(&S.dfull[m % C::DOS], (m / C::DOS) & 1, ab)) return false;
          tc_fence_after();
          if (FP8)
            issue_nt_e4m3(tXD, sV, do_at(m));
          else
            issue_nt<D * 2>(tXD, sV, do_at(m));
          mma_commit(&S.dp_full);
          return true;
        };
        ok = issue_dp(0);
        while (ok) {
          const bool has_next = steps.advance(p, b, g, I);
          // dV += P^T(n) dO(n).
          if (!(ok = mbar_wait(&S.p_full, n & 1, ab))) break;
          tc_fence_after();
          if (FP8)
            issue_acc_e4m3<D>(tdV, sP8, do_at(n), n == 0);
          else
            issue_acc_inplace<D>(tdV, tXD + 32, do_at(n), n == 0);
          // dK += dS^T(n) Q(n); Q(n) and dO(n) are free after it (S^T(n)
          // completed before the softmax stored dS^T(n); dV(n) ran before dK(n)).
          if (!(ok = mbar_wait(&S.ds_full, n & 1, ab))) break;
          tc_fence_after();
          issue_acc_inplace<D>(tdK, tXD, q_at(n), n == 0);
          mma_commit(&S.qempty[n % C::QS]);
          if (!has_next) break;
          if (!(ok = issue_dp(n + 1))) break;
          ++n;
        }
      }
      mma_commit(&S.fin);
      mbar_wait_drain(&S.fin, 0);
    }
  } else if (warp == 2) {
    // --------------------------------------------------- MMA issuer: S^T
    // S^T(n) = K Q(n)^T into XS once the softmax has copied S^T(n-1) out.
    // Each S^T(n) completes before the softmax goes on with step n, so none is
    // in flight when the other issuer's last commit (fin) completes.
    if (lane == 0) {
      bool ok = mbar_wait(&S.in_full, 0, ab);
      tc_fence_after();
      if (ok && any) {
        int g = 0, I = steps.I_first, n = 0;
        do {
          if (n > 0 && !(ok = mbar_wait(&S.xs_free, (n - 1) & 1, ab))) break;
          if (!(ok = mbar_wait(&S.qfull[n % C::QS], (n / C::QS) & 1, ab))) break;
          tc_fence_after();
          issue_nt<D * 2>(tXS, sK, sQ + (uint32_t)((n % C::QS) * C::TB));
          mma_commit(&S.s_full);
          ++n;
        } while (steps.advance(p, b, g, I));
      }
      // On an early exit S^T(n) may still be running: let it finish before
      // the CTA frees its TMEM.
      mma_commit(&S.fin_s);
      mbar_wait_drain(&S.fin_s, 0);
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
    const bool win = MASKS && (p.flags & MOD_WINDOW) != 0;
    const bool doc = MASKS && (p.flags & MOD_DOC) != 0;
    const float sc_in = p.scale / p.softcap, sc_out = p.softcap * LOG2E;
    const int doc_j = (doc && j < p.N) ? p.doc_ids[(size_t)b * p.N + j] : 0;
    // e4m3: dP = dP8 * sdo * sv; dV = dV8 * sdo / P8_MUL.
    const float sdo = FP8 ? fp8s[b * p.Hkv + hk] : 1.f;
    const float dps = FP8 ? sdo * fp8s[p.B * p.Hkv + b * p.Hkv + hk] : 1.f;
    bool doc_runs = false;
    const int2 run_j = doc ? doc_run(p, b, j, doc_runs) : make_int2(0, p.N);
    const bool doc_each = doc && !doc_runs;  // ids tested element by element
    bool ok = true;
    // Test hook: warpgroup 0 waits on a phase nothing completes (attn_test_hooks).
    if ((p.stall & STALL_BWD) && w == 0) ok = wait_warp(&S.never, 0, ab, p.wait_ns);
    if (ok && any) {
      int g = 0, I = steps.I_first, n = 0;
      do {
        const int hq = hk * G + g;
        const int cls = tile_class(p, b, I, J);
        const float al2 = al ? alibi_slope(p, hq) * LOG2E : 0.f;
        // {LSE log2, D} of this warpgroup's 64 query rows (columns): lane k
        // holds rows k and 32 + k (negated), broadcast by shuffles where used.
        const int i0 = I * TILE + 64 * w;  // query row of column 0
        const float2* rs = rowstat + ((size_t)b * p.Hq + hq) * ((size_t)p.nT * TILE) + i0;
        const float2 rs0 = rs[lane], rs1 = rs[32 + lane];
        const float my_nl2[2] = {-rs0.x, -rs1.x}, my_ndd[2] = {-rs0.y, -rs1.y};

        // S^T(n) -> registers, XS back to the MMA pipe (S^T(n+1)).
        if (!(ok = wait_warp(&S.s_full, n & 1, ab))) break;
        tc_fence_after();
        uint32_t s[64];
        tmem_ld64(tXS + lane_off + 64 * w, s);
        tmem_wait64(s);
        tc_fence_before();
        mbar_arrive(&S.xs_free);

        // P = exp2(x - LSE) (0 where masked); s[] keeps P (times the
        // soft-cap derivative) for dS.
        KvStep a;
        a.scale_log2 = p.scale_log2;
        a.sc_in = sc_in;
        a.sc_out = sc_out;
        a.al2 = al2;
        a.al_base = al2 * (float)(j - i0);
        a.lo = causal ? j - i0 : -0x7fffffff;
        a.hi = win ? p.window + j - i0 : 0x7fffffff;
        if (doc_runs) {  // the query rows of this KV row's document: one interval
          a.lo = max(a.lo, run_j.x - i0);
          a.hi = min(a.hi, run_j.y - i0);
        }
        a.doc_cols = doc_each ? p.doc_ids + (size_t)b * p.N + i0 : nullptr;
        a.doc_j = doc_j;
        a.n_cols = p.N - i0;
        a.sc = sc;
        a.al = al;
        a.partial = cls == CLS_PARTIAL;
        // P as packed bf16 (pk, the A operand of dV) and the factor of dS
        // (pd: P times the soft-cap derivative, else P), also bf16, which
        // keeps the registers live across the dP^T loads to pk, pd, dp and o.
        uint32_t pk[32], pd[32], p8[16];
        kv_row_p<MODS>(s, pk, my_nl2, a);
#pragma unroll
        for (int q = 0; q < 32; ++q)
          pd[q] = sc ? pack_bf16(__uint_as_float(s[2 * q]), __uint_as_float(s[2 * q + 1])) : pk[q];
        if (FP8)
#pragma unroll
          for (int q = 0; q < 16; ++q)
            p8[q] = pack_e4m3x4(__uint_as_float(s[4 * q]) * P8_MUL, __uint_as_float(s[4 * q + 1]) * P8_MUL,
                                __uint_as_float(s[4 * q + 2]) * P8_MUL, __uint_as_float(s[4 * q + 3]) * P8_MUL);

        // dS = P (dP - D) (times the soft-cap derivative), in pairs, from the
        // two 32-column halves of this warpgroup's dP^T columns: the second
        // half first, so that P^T(n) can go there at once (dV(n-1) and
        // dK(n-1) read XD before dP^T(n) overwrote it), then the first half,
        // which dS^T(n) replaces.
        if (!(ok = wait_warp(&S.dp_full, n & 1, ab))) break;
        tc_fence_after();
        if (FP8) {
          // e4m3 P^T into its shared-memory tile: dV(n-1), its last reader,
          // completed before the commit of dP^T(n) that was just seen.
          store_half_row_e4m3(smem + C::P8_OFF, r, w, p8);
          fence_async_smem();
          tc_fence_before();
          mbar_arrive(&S.p_full);
        }
        uint32_t dp[32], o[32];
        tmem_ld32(tXD + lane_off + 64 * w + 32, dp);
        tmem_wait_ld(dp);
        kv_row_ds_bf16<32, FP8>(pd + 16, dp, 32, my_ndd, o + 16, dps);
        if (!FP8) {
          tmem_st32(tXD + lane_off + 64 * w + 32, pk);
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&S.p_full);
        }
        tmem_ld32(tXD + lane_off + 64 * w, dp);
        tmem_wait_ld(dp);
        kv_row_ds_bf16<32, FP8>(pd, dp, 0, my_ndd, o, dps);
        tmem_st32(tXD + lane_off + 64 * w, o);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&S.ds_full);
        ++n;
      } while (steps.advance(p, b, g, I));
    }
    if (ok) ok = wait_warp(&S.fin, 0, ab);
    tc_fence_after();
    if (ok) {
      const size_t row = ((size_t)b * p.Hkv + hk) * p.N + j;
      store_cols<D / 2>(tdV + lane_off + w * (D / 2), any, FP8 ? sdo / P8_MUL : 1.0f, dv + row * D + w * (D / 2),
                        j < p.N);
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
// Shared memory: K tiles in a 4-slot ring (read by S and, at the end of the
// step, by dQ), V tiles in a 2-slot ring (read only by dP, early), and the dS
// tile.  Q and dO are first loaded into K slot 3 and V slot 1, copied into
// TMEM by the softmax warpgroups, and those slots then join their rings.
template <int D>
struct DqCfg {
  static constexpr int CH = D / 64;
  static constexpr int TB = TILE * D * 2;
  static constexpr int KS = 4, VS = 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = KS * TB;
  static constexpr int Q_OFF = K_OFF + 3 * TB;   // K slot 3
  static constexpr int DO_OFF = V_OFF + 1 * TB;  // V slot 1
  static constexpr int DS_OFF = V_OFF + VS * TB;  // dS tile, 128 x 128 bf16
  static constexpr int BAR_OFF = DS_OFF + TILE * TILE * 2;
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 256 + 1024);
};
static_assert(DqCfg<128>::SMEM_BYTES <= 232448, "dQ shared memory exceeds 227 KB");

struct DqBars {
  uint64_t in_full;              // Q, dO
  uint64_t kfull[4], kempty[4];  // K ring
  uint64_t vfull[2], vempty[2];  // V ring
  uint64_t s_full, s_free, p_full, acc_done;
  uint64_t a_ready;              // Q and dO copied into TMEM: their slots are free
  uint64_t fin[3];               // per issuer: all its MMAs done
  uint32_t tmem_base;
  int abort;
};

template <int D, bool MODS, bool MASKS>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const float2* __restrict__ rowstat, __nv_bfloat16* __restrict__ dq,
                  const AttnParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  DqBars& S = *reinterpret_cast<DqBars*>(smem + C::BAR_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();

  const int BH = p.B * p.Hq;
  const int I = p.nT - 1 - (int)(blockIdx.x / BH);  // longest rows (causal) first
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int hk = hq / (p.Hq / p.Hkv);
  const bool causal = (p.flags & MOD_CAUSAL) != 0;
  const int2 rg = MASKS ? q_tile_range(p, b, I) : make_int2(0, p.nT);
  const int J_end = min(causal ? min(p.nT, I + 1) : p.nT, rg.y);
  auto next_J = [&](int J) {
    while (J < J_end && tile_class(p, b, I, J) == CLS_SKIP) ++J;
    return J;
  };
  const int J_first = next_J(rg.x);

  if (threadIdx.x == 0) {
    S.abort = 0;
    mbar_init(&S.in_full, 1);
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(&S.kfull[s], 1);
      mbar_init(&S.kempty[s], 2);  // read by S (issuer A) and dQ (issuer B)
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(&S.vfull[s], 1);
      mbar_init(&S.vempty[s], 1);  // read by dP (issuer A)
    }
    mbar_init(&S.s_full, 2);       // S(n) and dP(n), one commit each
    mbar_init(&S.s_free, 256);
    mbar_init(&S.p_full, 256);
    mbar_init(&S.acc_done, 1);     // dQ(n) done: dS buffer free
    mbar_init(&S.a_ready, 256);    // Q / dO in TMEM: slots 4 and 5 free
    for (int i = 0; i < 3; ++i) mbar_init(&S.fin[i], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const uint32_t sKr = smem_u32(smem + C::K_OFF), sVr = smem_u32(smem + C::V_OFF);
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
      int nk = 0, nv = 0;  // K / V loads issued
      for (int J = J_first; J < J_end; J = next_J(J + 1)) {
        const int ks = nk % C::KS, vs = nv % C::VS;
        // K slot 3 and V slot 1 hold Q and dO until the softmax copied them.
        if (nk == 3 && !mbar_wait(&S.a_ready, 0, ab)) break;
        if (!mbar_wait(&S.kempty[ks], ((nk / C::KS) & 1) ^ 1, ab)) break;
        mbar_arrive_tx(&S.kfull[ks], C::TB);
        for (int ch = 0; ch < C::CH; ++ch)
          tma_load_3d(smem + C::K_OFF + ks * C::TB + ch * 16384, &tk, &S.kfull[ks], ch * 64, J * TILE,
                      b * p.Hkv + hk);
        ++nk;
        if (nv == 1 && !mbar_wait(&S.a_ready, 0, ab)) break;
        if (!mbar_wait(&S.vempty[vs], ((nv / C::VS) & 1) ^ 1, ab)) break;
        mbar_arrive_tx(&S.vfull[vs], C::TB);
        for (int ch = 0; ch < C::CH; ++ch)
          tma_load_3d(smem + C::V_OFF + vs * C::TB + ch * 16384, &tv, &S.vfull[vs], ch * 64, J * TILE,
                      b * p.Hkv + hk);
        ++nv;
      }
      // Loads still in flight must land before the CTA exits.
      mbar_wait_drain(&S.in_full, 0);
      for (int s = 0; s < C::KS; ++s)
        if (nk > s) mbar_wait_drain(&S.kfull[s], ((nk - 1 - s) / C::KS) & 1);
      for (int s = 0; s < C::VS; ++s)
        if (nv > s) mbar_wait_drain(&S.vfull[s], ((nv - 1 - s) / C::VS) & 1);
    }
  } else if (warp < 4) {
    // Three issuing threads, one per warp of warps 1-3, so that each SM
    // sub-partition carries at most one of them: S = Q K^T (warp 1), dP = dO V^T
    // (warp 3), dQ += dS K (warp 2).  A thread whose MMAs wait for room in the
    // tensor pipe slows the softmax warps of its sub-partition, and every
    // hand-off waits for the slowest warp: with S and dP on one thread, the
    // softmax warps beside it trailed the others by 250-400 cycles a step.
    if (lane == 0) {
      const int role = warp == 1 ? 0 : warp == 3 ? 1 : 2;  // 0: S, 1: dP, 2: dQ
      bool ok = mbar_wait(&S.in_full, 0, ab);
      tc_fence_after();
      int n = 0;
      for (int J = J_first; ok && J < J_end; J = next_J(J + 1), ++n) {
        const int ks = n % C::KS, vs = n % C::VS;
        const uint32_t k_sm = sKr + ks * C::TB, v_sm = sVr + vs * C::TB;
        if (role < 2) {
          // S(n) / dP(n) once the softmax has copied S(n-1) and dP(n-1) out.
          if (role == 0 && !(ok = mbar_wait(&S.kfull[ks], (n / C::KS) & 1, ab))) break;
          if (role == 1 && !(ok = mbar_wait(&S.vfull[vs], (n / C::VS) & 1, ab))) break;
          if (n == 0 && !(ok = mbar_wait(&S.a_ready, 0, ab))) break;
          if (n > 0 && !(ok = mbar_wait(&S.s_free, (n - 1) & 1, ab))) break;
          tc_fence_after();
          if (role == 0) {
            issue_nt_tmem_a<D>(tS, tQa, k_sm);
            mma_commit(&S.s_full);
            mma_commit(&S.kempty[ks]);
          } else {
            issue_nt_tmem_a<D>(tdP, tDOa, v_sm);
            mma_commit(&S.s_full);
            mma_commit(&S.vempty[vs]);
          }
        } else {
          if (!(ok = mbar_wait(&S.kfull[ks], (n / C::KS) & 1, ab))) break;
          if (!(ok = mbar_wait(&S.p_full, n & 1, ab))) break;
          tc_fence_after();
          issue_acc<D>(tdQ, sDS, k_sm, n == 0);
          mma_commit(&S.acc_done);
          mma_commit(&S.kempty[ks]);
        }
      }
      mma_commit(&S.fin[role]);
      mbar_wait_drain(&S.fin[role], 0);
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
    const bool win = MASKS && (p.flags & MOD_WINDOW) != 0;
    const bool doc = MASKS && (p.flags & MOD_DOC) != 0;
    const float sc_in = p.scale / p.softcap, sc_out = p.softcap * LOG2E;
    const float al2 = al ? alibi_slope(p, hq) * LOG2E : 0.f;
    const size_t row = ((size_t)b * p.Hq + hq) * p.N + i;
    const float2 rs = rowstat[((size_t)b * p.Hq + hq) * ((size_t)p.nT * TILE) + i];
    const uint64_t nl2 = f2_pack(-rs.x, -rs.x), ndd = f2_pack(-rs.y, -rs.y);
    const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
    const int doc_i = (doc && i < p.N) ? p.doc_ids[(size_t)b * p.N + i] : 0;
    bool doc_runs = false;
    const int2 run_i = doc ? doc_run(p, b, i, doc_runs) : make_int2(0, p.N);
    const bool doc_each = doc && !doc_runs;  // ids tested element by element
    const uint64_t sc_in2 = f2_pack(sc_in, sc_in), sc_out2 = f2_pack(sc_out, sc_out);
    const uint64_t one2 = f2_pack(1.f, 1.f), al2x = f2_pack(al2, al2);
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
      int hi_lim = min(causal ? i : 0x7fffffff, p.N - 1) - j0;  // valid iff c <= hi_lim
      int lo_lim = win ? i - p.window - j0 : -0x7fffffff;        // valid iff c > lo_lim
      if (doc_runs) {  // the keys of this query row's document: one interval
        hi_lim = min(hi_lim, run_i.y - 1 - j0);
        lo_lim = max(lo_lim, run_i.x - 1 - j0);
      }
      const float al_base = al2 * (float)(j0 - i);
      uint32_t dw[32];
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
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
          if (al) y2 = f2_fma(f2_pack((float)k, (float)(k + 1)), al2x, f2_add(y2, f2_pack(al_base, al_base)));
          x2 = f2_add(y2, nl2);
        } else {
          x2 = f2_fma(f2_pack(s0, s1), sl2, nl2);
        }
        float x0, x1;
        f2_unpack(x2, x0, x1);
        float pe[2] = {ex2(x0), ex2(x1)};
        if (cls == CLS_PARTIAL) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = k + e;
            bool valid = (c <= hi_lim) && (c > lo_lim);
            if (doc_each && valid) valid = (__ldg(p.doc_ids + (size_t)b * p.N + j0 + c) == doc_i);
            if (!valid) pe[e] = 0.f;
          }
        }
        uint64_t pp = f2_pack(pe[0], pe[1]);
        if (sc) pp = f2_mul(pp, dmul2);
        const uint64_t g2 = f2_add(f2_pack(__uint_as_float(dp[k]), __uint_as_float(dp[k + 1])), ndd);
        float ds0, ds1;
        f2_unpack(f2_mul(pp, g2), ds0, ds1);
        dw[k / 2] = pack_bf16(ds0, ds1);
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
    if (ok) ok = wait_warp(&S.fin[2], 0, ab);
    tc_fence_after();
    if (ok) store_cols<D / 2>(tdQ + lane_off + w * (D / 2), n > 0, p.scale, dq + row * D + w * (D / 2), i < p.N);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // Launched as a programmatic dependent of the dK/dV kernel (it may start
  // before that grid ends): no CTA of this grid completes before the dK/dV
  // grid has, so work after this kernel in the stream sees dK and dV too.
  pdl_wait();
}

// ------------------------------------------------------------------ launch
template <int D, bool MODS, bool MASKS, bool FP8 = false>
static cudaError_t launch_bwd_t(const BwdLaunch& L, cudaStream_t st) {
  const AttnParams& p = L.p;
  const long long rows = (long long)p.B * p.Hq * p.nT * TILE;
  const long long threads = rows * (D / 16);  // bwd_pre: 16 elements of a row per thread
  if (L.events[0]) cudaEventRecord(L.events[0], st);
  cudaError_t e;
  if (FP8 && (e = launch_quant_bwd_fp8(L.dout, L.v, L.do8, L.v8, L.fp8s, p.B, p.Hq, p.Hkv, p.N, L.fp8amax, p.status, st)) !=
                 cudaSuccess)
    return e;
  bwd_pre_kernel<D><<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
      (const __nv_bfloat16*)L.o, (const __nv_bfloat16*)L.dout, L.lse, L.rowstat, p.N, rows, PreExtra{});
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  static int kv_regs = -1, dq_regs = -1;
  using KC = KvCfg<D, FP8>;
  auto kv = bwd_dkdv_kernel<D, MODS, MASKS, FP8>;
  if ((e = check_regs(kv, kv_regs)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, KC::SMEM_BYTES)) != cudaSuccess)
    return e;
  if (L.events[1]) cudaEventRecord(L.events[1], st);
  kv<<<(unsigned)(p.nT * p.B * p.Hkv), 384, KC::SMEM_BYTES, st>>>(
      L.tq, L.tk, FP8 ? L.tv8 : L.tv, FP8 ? L.tdo8 : L.tdo, L.rowstat, (__nv_bfloat16*)L.dk, (__nv_bfloat16*)L.dv, p,
      L.fp8s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  auto dqk = bwd_dq_kernel<D, MODS, MASKS>;
  if ((e = check_regs(dqk, dq_regs)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(dqk, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  if (L.events[2]) cudaEventRecord(L.events[2], st);
  {
    // Programmatic dependent launch: dQ's CTAs may start on the SMs the
    // dK/dV grid's tail leaves idle (each waits for that grid before exiting).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.nT * p.B * p.Hq));
    cfg.blockDim = dim3(384);
    cfg.dynamicSmemBytes = DqCfg<D>::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, dqk, L.tq, L.tk, L.tv, L.tdo, L.rowstat, (__nv_bfloat16*)L.dq, p)) !=
        cudaSuccess)
      return e;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (L.events[3]) cudaEventRecord(L.events[3], st);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdLaunch& L, int d, bool mods, bool masks, cudaStream_t st) {
  if (L.fp8) return (d == 128 && !mods && !masks) ? launch_bwd_t<128, false, false, true>(L, st) : cudaErrorInvalidValue;
  if (d == 128)
    return mods ? launch_bwd_t<128, true, true>(L, st)
                : masks ? launch_bwd_t<128, false, true>(L, st) : launch_bwd_t<128, false, false>(L, st);
  return mods ? launch_bwd_t<64, true, true>(L, st)
              : masks ? launch_bwd_t<64, false, true>(L, st) : launch_bwd_t<64, false, false>(L, st);
}

}  // namespace attn
