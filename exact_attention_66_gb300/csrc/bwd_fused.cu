// One-kernel backward of exact tiled attention under a causal mask, sm_103a:
// dK, dV and dQ from a single pass over the tile pairs, five GEMMs per pair
// (FlashAttention-3 digest, "Rappel du fonctionnement de FlashAttention":
// tiles, recomputation of P from the LSE).  Formulas as in bwd.cu:
//   P = exp(x - LSE), dP = dO V^T, dS = P (dP - D) (times the soft-cap
//   derivative), dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K.
//
// Work items are (batch, KV head, 128-row KV tile J).  A CTA keeps K_J, V_J in
// shared memory and walks the non-skipped Q tiles I of its KV tile from the
// top down, every query head of the GQA group inner; per step:
//   S^T = K Q^T (TMEM X)  ->  P^T, packed bf16, written back into X
//   dP^T = V dO^T (TMEM Y) ->  dS^T, bf16, into shared memory
//   dV += P^T dO (A from TMEM), dK += dS^T Q, dQ_part = dS K (TMEM Y).
// dV and dK stay in TMEM for the whole item.  The 128 x d fp32 dQ partial of
// each step is added into an fp32 dQ accumulator in global memory.
//
// Determinism.  The dQ partials of one query tile (b, hq, I) come from every
// non-skipped KV tile J of its row, from different CTAs, in no fixed order.
// Each partial is rounded to an integer multiple of its row's quantum (a power
// of two chosen from a bound on |dQ_i| that holds for every partial sum,
// bwd_pre) and added as int32 (red.global.add.s32): integer addition is
// associative, so the sum -- and dQ = sum / quantum * scale, written by a
// last pass -- is bitwise the same whatever order the partials arrive in,
// with no ordering between CTAs at all (contrast the atomics-based,
// nondeterministic backward on the FlexAttention/FA4 page, "Limitations
// actuelles").  The bound leaves at least 2^30 quanta for |dQ_i|: about 19
// significant bits in the worst case the bound allows, far below the bf16
// rounding of the result.
//
// Scheduling.  The grid is persistent (one CTA per SM) and CTAs take work
// items from a global counter in ascending J: the longest items first (J = 0
// has the most Q tiles under the causal mask); no CTA ever waits on another.
//
// Roles (640 threads): warp 0 lane 0 claims items and drives TMA; warp 1
// lane 0 issues every MMA; warps 4-11 are two warpgroups of 128 threads
// (thread = TMEM lane) that compute P and dS for 64 query columns each and
// write dK / dV at the end of each item; warps 12-19 are two warpgroups that
// take the dQ partial of 64 query rows each out of TMEM and reduce it into
// global memory, off the GEMM chain.  d = 128 only (d = 64 runs the two-kernel
// backward of bwd.cu).
#include "bwd_common.cuh"
#include "launch.h"

namespace attn {

// 640 threads: warpgroup 0 (TMA producer, MMA issuer, two idle warps), two
// P / dS warpgroups and two dQ reduction warpgroups (one per half of a dQ
// tile: eight warps keep enough reductions in flight).  Launched at 96
// registers per thread (65536 / 640, rounded down to a multiple of 8);
// warpgroup 0 (down to 56) and the reduction warpgroups (down to 88) give
// registers to the P / dS warpgroups (up to 120): 56 + 2 x 120 + 2 x 88 <= 5 x 96.
constexpr int FU_THREADS = 640, FU_LAUNCH_REGS = 96, FU_REGS_LOW = 56, FU_REGS_SOFTMAX = 120,
              FU_REGS_REDUCE = 88;
static_assert(FU_REGS_LOW + 2 * FU_REGS_SOFTMAX + 2 * FU_REGS_REDUCE <= 5 * FU_LAUNCH_REGS, "register split");
static_assert(FU_REGS_LOW <= FU_LAUNCH_REGS && FU_REGS_REDUCE <= FU_LAUNCH_REGS && FU_REGS_SOFTMAX >= FU_LAUNCH_REGS,
              "setmaxnreg.dec lowers, setmaxnreg.inc raises the launch count");

template <int D>
struct FuCfg {
  static constexpr int CH = D / 64;         // 64-column chunks of a row
  static constexpr int TB = TILE * D * 2;   // one 128-row bf16 tile
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TB;
  static constexpr int Q_OFF = 2 * TB;      // 2-slot Q ring (read by S, then dK)
  static constexpr int DO_OFF = 4 * TB;     // 2-slot dO ring (read by dV, then dP)
  static constexpr int DS_OFF = 6 * TB;     // dS^T, 128 KV rows x 128 query columns bf16
  static constexpr int BAR_OFF = DS_OFF + TILE * TILE * 2;
  static constexpr int SMEM_BYTES = smem_one_cta(BAR_OFF + 512 + 1024);
};
static_assert(FuCfg<128>::SMEM_BYTES <= 232448, "fused backward shared memory exceeds 227 KB");

struct FuBars {
  uint64_t item_full[2], item_empty[2];  // work-item slots (producer -> issuer, softmax)
  uint64_t kv_full;                      // K_J, V_J of the current item landed
  uint64_t kv_free;                      // every MMA of an item done: K/V reusable, dK/dV readable (commit)
  uint64_t qfull[2], qempty[2], dfull[2], dempty[2];
  uint64_t s_full;    // S^T(m) in X                   (commit)
  uint64_t p_full;    // P^T(m) packed into X          (256 softmax threads)
  uint64_t dp_full;   // dP^T(m) in Y                  (commit)
  uint64_t ds_full;   // dS^T(m) in shared memory      (256)
  uint64_t dq_full;   // dQ(m) partial in Y            (commit; also: dK(m) done)
  uint64_t y_free;    // dQ(m) partial read out of Y   (256 reduction threads)
  uint64_t acc_free;  // dV, dK of the previous item read out of TMEM (256)
  uint64_t fin;
  uint64_t never;     // test hook: a phase that nothing completes
  int item[2];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(FuBars) <= 512, "barrier block");

// A work item: KV tile J of (batch b, KV head hk).  Its steps are the
// non-skipped Q tiles I in [I_lo, I_top] from the top down, heads inner.
struct FuItem {
  int b, hk, J;
  int I_lo, I_top;  // I_top < I_lo: no step (the tile's dK, dV are zero)
};

// Highest non-skipped Q tile <= I of the item's KV tile (I_lo - 1 if none).
__device__ __forceinline__ int fu_down(const AttnParams& p, const FuItem& it, int I) {
  while (I >= it.I_lo && tile_class(p, it.b, I, it.J) == CLS_SKIP) --I;
  return I;
}

template <bool MASKS>
__device__ __forceinline__ FuItem fu_item(const AttnParams& p, int t) {
  FuItem it;
  const int BHk = p.B * p.Hkv;
  it.J = t / BHk;
  const int bh = t - it.J * BHk;
  it.b = bh / p.Hkv;
  it.hk = bh - it.b * p.Hkv;
  int lo = it.J, hi = p.nT;  // causal: only Q tiles I >= J
  if (MASKS) {
    const int2 rg = kv_tile_range(p, it.b, it.J);
    lo = max(lo, rg.x);
    hi = min(hi, rg.y);
  }
  it.I_lo = lo;
  it.I_top = fu_down(p, it, hi - 1);
  return it;
}

// Next step: the next query head of the group, else the next Q tile down.
__device__ __forceinline__ bool fu_next(const AttnParams& p, const FuItem& it, int G, int& I, int& g) {
  if (++g < G) return true;
  g = 0;
  I = fu_down(p, it, I - 1);
  return I >= it.I_lo;
}

// Global reduction of one int32 dQ accumulator element.
__device__ __forceinline__ void red_add_s32(int* a, int v) {
  asm volatile("red.global.add.s32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

// The dQ partial of a step, dQ^T(tmem, 128 head-dimension lanes x 128 query
// columns) = K^T dS^T, with K and the dS^T tile both read MN-major (the
// head-dimension, resp. query, columns contiguous in 64-column chunks of the
// K-major tiles).  A TMEM lane then holds one head-dimension index of every
// query row, so the 32 lanes of a warp cover 32 consecutive dQ columns of one
// row: each warp-wide global reduction is one whole 128-byte line.
__device__ __forceinline__ void issue_dq(uint32_t d_tmem, uint32_t ds_smem, uint32_t k_smem) {
  constexpr uint32_t id = idesc_bf16(128, 128, true, true);
  const uint64_t dsd = opaque(sdesc_sw128(ds_smem, 16384, 1024));
  const uint64_t kd = opaque(sdesc_sw128(k_smem, 16384, 1024));
#pragma unroll
  for (int kk = 0; kk < TILE / 16; ++kk) {
    const uint32_t off = kk * 16 * 128;
    mma_f16_ss(d_tmem, sdesc_add(kd, off), sdesc_add(dsd, off), id, kk > 0 ? 1u : 0u);
  }
}

template <int D, bool MODS, bool MASKS>
__global__ void __launch_bounds__(FU_THREADS, 1)
    bwd_fused_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                     const float2* __restrict__ rowstat, const float* __restrict__ qscale,
                     int* __restrict__ dqacc, int* __restrict__ ticket, __nv_bfloat16* __restrict__ dk,
                     __nv_bfloat16* __restrict__ dv, const AttnParams p) {
  static_assert(D == 128, "the one-kernel backward is built for d = 128");
  using C = FuCfg<D>;
  constexpr int HD = D / 2;  // dQ / dK / dV columns per softmax warpgroup
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  FuBars& S = *reinterpret_cast<FuBars*>(smem + C::BAR_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();
  const int G = p.Hq / p.Hkv;
  const int n_items = p.nT * p.B * p.Hkv;

  if (threadIdx.x == 0) {
    S.abort = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.item_full[s], 1);
      mbar_init(&S.item_empty[s], 1 + 256 + 256);  // the issuer, softmax and reduction threads
      mbar_init(&S.qfull[s], 1);
      mbar_init(&S.qempty[s], 1);
      mbar_init(&S.dfull[s], 1);
      mbar_init(&S.dempty[s], 1);
    }
    mbar_init(&S.kv_full, 1);
    mbar_init(&S.kv_free, 1);
    mbar_init(&S.s_full, 1);
    mbar_init(&S.p_full, 256);
    mbar_init(&S.dp_full, 1);
    mbar_init(&S.ds_full, 256);
    mbar_init(&S.dq_full, 1);
    mbar_init(&S.y_free, 256);
    mbar_init(&S.acc_free, 256);
    mbar_init(&S.fin, 1);
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
  const uint32_t sK = smem_u32(smem + C::K_OFF), sV = smem_u32(smem + C::V_OFF);
  const uint32_t sQ = smem_u32(smem + C::Q_OFF), sDO = smem_u32(smem + C::DO_OFF);
  const uint32_t sDS = smem_u32(smem + C::DS_OFF);
  // TMEM: X [0,128) S^T then P^T; Y [128,256) dP^T then the dQ partial;
  // dV [256, 256 + D), dK [256 + D, 256 + 2D).
  const uint32_t tX = tmem, tY = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
  auto q_at = [&](int m) { return sQ + (uint32_t)((m & 1) * C::TB); };
  auto do_at = [&](int m) { return sDO + (uint32_t)((m & 1) * C::TB); };

  if (warp < 4) regs_dec<FU_REGS_LOW>();
  if (warp == 0) {
    // ------------------------------------------- work items and TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      int k = 0, c = 0;  // items published, items with steps
      int mq = 0, md = 0;  // Q / dO tiles loaded (one of each per step)
      bool ok = true;
      while (ok) {
        // The next item is claimed only once this CTA has issued every load of
        // the current one: an item claimed early would hold up the CTAs that
        // wait on its dQ partials.
        const int t = atomicAdd(ticket, 1);
        const int s = k & 1;
        if (k >= 2 && !(ok = mbar_wait(&S.item_empty[s], ((k - 2) >> 1) & 1, ab))) break;
        *(volatile int*)&S.item[s] = t < n_items ? t : -1;
        mbar_arrive(&S.item_full[s]);
        ++k;
        if (t >= n_items) break;
        const FuItem it = fu_item<MASKS>(p, t);
        if (it.I_top < it.I_lo) continue;
        if (c > 0 && !(ok = mbar_wait(&S.kv_free, (c - 1) & 1, ab))) break;
        mbar_arrive_tx(&S.kv_full, 2 * C::TB);
        for (int ch = 0; ch < C::CH; ++ch) {
          tma_load_3d(smem + C::K_OFF + ch * 16384, &tk, &S.kv_full, ch * 64, it.J * TILE, it.b * p.Hkv + it.hk);
          tma_load_3d(smem + C::V_OFF + ch * 16384, &tv, &S.kv_full, ch * 64, it.J * TILE, it.b * p.Hkv + it.hk);
        }
        ++c;
        int I = it.I_top, g = 0;
        do {
          const int plane = it.b * p.Hq + it.hk * G + g;
          const int qs = mq & 1;
          if (!(ok = mbar_wait(&S.qempty[qs], ((mq >> 1) & 1) ^ 1, ab))) break;
          mbar_arrive_tx(&S.qfull[qs], C::TB);
          for (int ch = 0; ch < C::CH; ++ch)
            tma_load_3d(smem + C::Q_OFF + qs * C::TB + ch * 16384, &tq, &S.qfull[qs], ch * 64, I * TILE, plane);
          ++mq;
          const int ds = md & 1;
          if (!(ok = mbar_wait(&S.dempty[ds], ((md >> 1) & 1) ^ 1, ab))) break;
          mbar_arrive_tx(&S.dfull[ds], C::TB);
          for (int ch = 0; ch < C::CH; ++ch)
            tma_load_3d(smem + C::DO_OFF + ds * C::TB + ch * 16384, &tdo, &S.dfull[ds], ch * 64, I * TILE, plane);
          ++md;
        } while (fu_next(p, it, G, I, g));
      }
      // Loads still in flight must land before the CTA exits.
      if (c > 0) mbar_wait_drain(&S.kv_full, (c - 1) & 1);
      for (int s = 0; s < 2; ++s) {
        if (mq > s) mbar_wait_drain(&S.qfull[s], ((mq - 1 - s) >> 1) & 1);
        if (md > s) mbar_wait_drain(&S.dfull[s], ((md - 1 - s) >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per step m: dP(m); [first step of an item: dV(m)]; S(m+1); dK(m), dQ(m);
    // dV(m+1).  The S^T -> P^T chain (X) and the dP^T -> dS -> dQ chain (Y)
    // interleave, so each GEMM finds the tensor pipe free of the other
    // chain's latency.
    if (lane == 0) {
      int k = 0, c = 0, m = 0;
      bool ok = true;
      while (ok) {
        const int s = k & 1;
        if (!(ok = mbar_wait(&S.item_full[s], (k >> 1) & 1, ab))) break;
        const int t = *(volatile int*)&S.item[s];
        mbar_arrive(&S.item_empty[s]);
        ++k;
        if (t < 0) break;
        const FuItem it = fu_item<MASKS>(p, t);
        if (it.I_top < it.I_lo) continue;
        if (!(ok = mbar_wait(&S.kv_full, c & 1, ab))) break;
        if (!(ok = mbar_wait(&S.qfull[m & 1], (m >> 1) & 1, ab))) break;
        tc_fence_after();
        issue_nt<D * 2>(tX, sK, q_at(m));
        mma_commit(&S.s_full);
        int I = it.I_top, g = 0;
        bool first = true;
        while (true) {
          int I2 = I, g2 = g;
          const bool has_next = fu_next(p, it, G, I2, g2);
          // dP(m) into Y once the previous step's dQ partial has left it.
          if (m > 0 && !(ok = mbar_wait(&S.y_free, (m - 1) & 1, ab))) break;
          if (!(ok = mbar_wait(&S.dfull[m & 1], (m >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_nt<D * 2>(tY, sV, do_at(m));
          mma_commit(&S.dp_full);
          if (first) {  // dV(m) overwrites the accumulator: the last item's dV, dK must be out
            if (!(ok = mbar_wait(&S.p_full, m & 1, ab))) break;
            if (c > 0 && !(ok = mbar_wait(&S.acc_free, (c - 1) & 1, ab))) break;
            tc_fence_after();
            issue_acc_inplace<D>(tdV, tX, do_at(m), true);
          }
          mma_commit(&S.dempty[m & 1]);  // dO(m): read by dV(m) and dP(m)
          if (has_next) {
            if (!(ok = mbar_wait(&S.qfull[(m + 1) & 1], ((m + 1) >> 1) & 1, ab))) break;
            tc_fence_after();
            issue_nt<D * 2>(tX, sK, q_at(m + 1));  // after dV(m) read P^T(m) from X
            mma_commit(&S.s_full);
          }
          if (!(ok = mbar_wait(&S.ds_full, m & 1, ab))) break;
          tc_fence_after();
          issue_acc<D>(tdK, sDS, q_at(m), first);
          mma_commit(&S.qempty[m & 1]);  // Q(m): read by S(m) and dK(m)
          issue_dq(tY, sDS, sK);
          mma_commit(&S.dq_full);
          if (!has_next) {
            mma_commit(&S.kv_free);
            ++m;
            break;
          }
          // dV(m+1) reads dO(m+1): its load must have landed too (the wait
          // before dP(m+1) comes later; a completed phase stays complete until
          // the slot is refilled, which needs dP(m+1) first).
          if (!(ok = mbar_wait(&S.p_full, (m + 1) & 1, ab))) break;
          if (!(ok = mbar_wait(&S.dfull[(m + 1) & 1], ((m + 1) >> 1) & 1, ab))) break;
          tc_fence_after();
          issue_acc_inplace<D>(tdV, tX, do_at(m + 1), false);
          I = I2;
          g = g2;
          first = false;
          ++m;
        }
        ++c;
      }
      mma_commit(&S.fin);
      mbar_wait_drain(&S.fin, 0);
    }
  } else if (warp >= 4 && warp < 12) {  // warps 4-7: query columns 0-63, 8-11: 64-127
    // ------------------------------------------ P, dS and the dK/dV epilogue
    regs_inc<FU_REGS_SOFTMAX>();
    const int w = (warp - 4) >> 2;  // query columns [64 w, 64 w + 64); dK/dV columns [HD w, HD w + HD)
    const int wq = warp & 3;
    const int r = wq * 32 + lane;   // TMEM lane = KV row of the tile
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const bool sc = MODS && (p.flags & MOD_SOFTCAP);
    const bool al = MODS && (p.flags & MOD_ALIBI);
    const bool win = MASKS && (p.flags & MOD_WINDOW) != 0;
    const bool doc = MASKS && (p.flags & MOD_DOC) != 0;
    const float sc_in = p.scale / p.softcap, sc_out = p.softcap * LOG2E;
    uint8_t* ds_tile = smem + C::DS_OFF;
    bool ok = true;
    // Test hook: warpgroup 0 waits on a phase nothing completes (attn_test_hooks).
    if ((p.stall & STALL_BWD) && w == 0) ok = wait_warp(&S.never, 0, ab, p.wait_ns);
    int k = 0, c = 0, m = 0;  // items read, items with steps, steps
    while (ok) {
      const int s = k & 1;
      if (!(ok = wait_warp(&S.item_full[s], (k >> 1) & 1, ab))) break;
      const int t = *(volatile int*)&S.item[s];
      mbar_arrive(&S.item_empty[s]);
      ++k;
      if (t < 0) break;
      const FuItem it = fu_item<MASKS>(p, t);
      const int j = it.J * TILE + r;  // this thread's KV row
      const size_t row = ((size_t)it.b * p.Hkv + it.hk) * p.N + j;
      if (it.I_top < it.I_lo) {  // no allowed pair: dK = dV = 0
        store_cols<HD>(0, false, 0.f, dv + row * D + HD * w, j < p.N);
        store_cols<HD>(0, false, 0.f, dk + row * D + HD * w, j < p.N);
        continue;
      }
      const int doc_j = (doc && j < p.N) ? p.doc_ids[(size_t)it.b * p.N + j] : 0;
      bool doc_runs = false;
      const int2 run_j = doc ? doc_run(p, it.b, j, doc_runs) : make_int2(0, p.N);
      const bool doc_each = doc && !doc_runs;
      int I = it.I_top, g = 0;
      do {
        const int hq = it.hk * G + g;
        const int cls = tile_class(p, it.b, I, it.J);
        const float al2 = al ? alibi_slope(p, hq) * LOG2E : 0.f;
        const int i0 = I * TILE + 64 * w;  // query row of column 0
        const float2* rs = rowstat + ((size_t)it.b * p.Hq + hq) * ((size_t)p.nT * TILE) + i0;
        const float2 rs0 = rs[lane], rs1 = rs[32 + lane];
        const float nl2[2] = {-rs0.x, -rs1.x}, ndd[2] = {-rs0.y, -rs1.y};

        // S^T(m) -> P^T, 32 columns at a time; P^T packed into this
        // warpgroup's X columns.  P (times the soft-cap derivative) is kept as
        // packed bf16 for dS, which halves the registers it holds.
        if (!(ok = wait_warp(&S.s_full, m & 1, ab))) break;
        tc_fence_after();
        KvStep a;
        a.scale_log2 = p.scale_log2;
        a.sc_in = sc_in;
        a.sc_out = sc_out;
        a.al2 = al2;
        a.al_base = al2 * (float)(j - i0);
        a.lo = j - i0;  // causal
        a.hi = win ? p.window + j - i0 : 0x7fffffff;
        if (doc_runs) {
          a.lo = max(a.lo, run_j.x - i0);
          a.hi = min(a.hi, run_j.y - i0);
        }
        a.doc_cols = doc_each ? p.doc_ids + (size_t)it.b * p.N + i0 : nullptr;
        a.doc_j = doc_j;
        a.n_cols = p.N - i0;
        a.sc = sc;
        a.al = al;
        a.partial = cls == CLS_PARTIAL;
        uint32_t pk[32], pd[32];  // P, and P times the soft-cap derivative (soft-cap only)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t s32[32];
          tmem_ld32(tX + lane_off + 64 * w + 32 * h, s32);
          tmem_wait_ld(s32);
          kv_row_p_cols<MODS, 32>(s32, &pk[16 * h], 32 * h, nl2, a);
          if (sc)
#pragma unroll
            for (int q = 0; q < 16; ++q)
              pd[16 * h + q] = pack_bf16(__uint_as_float(s32[2 * q]), __uint_as_float(s32[2 * q + 1]));
        }
        tmem_st32(tX + lane_off + 64 * w, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&S.p_full);

        // dP^T(m) -> dS^T(m), bf16, into the shared-memory tile (the MMAs of
        // step m - 1 that read it are done: dP(m) was issued after them).
        if (!(ok = wait_warp(&S.dp_full, m & 1, ab))) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t dp[32], o[16];
          tmem_ld32(tY + lane_off + 64 * w + 32 * h, dp);
          tmem_wait_ld(dp);
          kv_row_ds_bf16<32>(sc ? &pd[16 * h] : &pk[16 * h], dp, 32 * h, ndd, o);
          store_quarter_row(ds_tile, r, w, h, o);
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&S.ds_full);
        ++m;
      } while (fu_next(p, it, G, I, g));
      if (!ok) break;
      // dK, dV out of TMEM once every MMA of the item has completed.
      if (!(ok = wait_warp(&S.kv_free, c & 1, ab))) break;
      tc_fence_after();
      store_cols<HD>(tdV + lane_off + HD * w, true, 1.0f, dv + row * D + HD * w, j < p.N);
      store_cols<HD>(tdK + lane_off + HD * w, true, p.scale, dk + row * D + HD * w, j < p.N);
      tc_fence_before();
      mbar_arrive(&S.acc_free);
      ++c;
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------ dQ reduction
    // Warpgroup h takes query rows 64 h .. 64 h + 63 of each step's dQ^T
    // partial (lane = head-dimension column): out of Y into registers (Y goes
    // back to the MMA pipe once both halves are out), rounded to the rows'
    // quanta, added into the int32 accumulator one whole line per warp-wide
    // reduction.
    regs_dec<FU_REGS_REDUCE>();
    const int h = (warp - 12) >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    int k = 0, m = 0;
    bool ok = true;
    while (ok) {
      const int s = k & 1;
      if (!(ok = wait_warp(&S.item_full[s], (k >> 1) & 1, ab))) break;
      const int t = *(volatile int*)&S.item[s];
      mbar_arrive(&S.item_empty[s]);
      ++k;
      if (t < 0) break;
      const FuItem it = fu_item<MASKS>(p, t);
      if (it.I_top < it.I_lo) continue;
      int I = it.I_top, g = 0;
      do {
        const size_t row0 = ((size_t)(it.b * p.Hq + it.hk * G + g) * p.nT + I) * TILE + 64 * h;  // padded row
        const float q_lo = qscale[row0 + lane], q_hi = qscale[row0 + 32 + lane];  // quanta of rows lane, 32 + lane
        if (!(ok = wait_warp(&S.dq_full, m & 1, ab))) break;
        tc_fence_after();
        uint32_t y[64];
        tmem_ld32(tY + lane_off + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&y[0]));
        tmem_ld32(tY + lane_off + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&y[32]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&y[0]));
        tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&y[32]));
        tc_fence_before();
        mbar_arrive(&S.y_free);
        int* acol = dqacc + row0 * D + r;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float q = __shfl_sync(0xffffffffu, c < 32 ? q_lo : q_hi, c & 31);
          red_add_s32(acol + (size_t)c * D, __float2int_rn(__uint_as_float(y[c]) * q));
        }
        ++m;
      } while (fu_next(p, it, G, I, g));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dQ = accumulator / row quantum * scale, bf16; rows past N are not written.
template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const int* __restrict__ dqacc,
                                                         const float* __restrict__ qscale,
                                                         __nv_bfloat16* __restrict__ dq, int N, int nT,
                                                         float scale, long long rows) {
  constexpr int TPR = D / 16;  // threads per row, 16 elements each
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gt / TPR;  // row of dq, [B * Hq * N]
  const int part = (int)(gt % TPR);
  if (row >= rows) return;
  // rows < 2^31 (a dQ of 2^31 rows would not fit in device memory): 32-bit division
  const unsigned bh = (unsigned)row / (unsigned)N;
  const long long prow = (long long)bh * nT * TILE + (row - (long long)bh * N);  // padded row
  const float mul = scale / qscale[prow];
  const int4* src = reinterpret_cast<const int4*>(dqacc + prow * D + part * 16);
  uint4* dst = reinterpret_cast<uint4*>(dq + row * D) + 2 * part;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int4 a = src[2 * h], b = src[2 * h + 1];
    uint4 o;
    o.x = pack_bf16((float)a.x * mul, (float)a.y * mul);
    o.y = pack_bf16((float)a.z * mul, (float)a.w * mul);
    o.z = pack_bf16((float)b.x * mul, (float)b.y * mul);
    o.w = pack_bf16((float)b.z * mul, (float)b.w * mul);
    dst[h] = o;
  }
}

// ------------------------------------------------------------------ launch
// K/V bounds, row statistics and quanta (zeroing the accumulator), the main
// kernel, the bf16 conversion of dQ.  events[0..3]: before the bounds, before
// the main kernel, before the conversion, after it.
template <bool MODS, bool MASKS>
static cudaError_t launch_fused_t(const BwdLaunch& L, cudaStream_t st) {
  constexpr int D = 128;
  const AttnParams& p = L.p;
  const long long rows = (long long)p.B * p.Hq * p.nT * TILE;
  const long long threads = rows * (D / 16);  // bwd_pre: 16 elements of a row per thread
  if (L.events[0]) cudaEventRecord(L.events[0], st);
  cudaError_t e = cudaMemsetAsync(L.kvb, 0, (size_t)p.B * p.Hkv * sizeof(float2), st);
  if (e != cudaSuccess) return e;
  const int chunks = (p.N + KV_BOUND_ROWS - 1) / KV_BOUND_ROWS;
  kv_bound_kernel<D><<<(unsigned)(p.B * p.Hkv * chunks), 256, 0, st>>>(
      (const __nv_bfloat16*)L.k, (const __nv_bfloat16*)L.v, L.kvb, p.N, chunks);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  PreExtra x{};
  x.ticket = L.ticket;
  x.dqacc = L.dqacc;
  x.qscale = L.qscale;
  x.kvb = L.kvb;
  x.Hq = p.Hq;
  x.Hkv = p.Hkv;
  x.scale = p.scale;
  bwd_pre_kernel<D><<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
      (const __nv_bfloat16*)L.o, (const __nv_bfloat16*)L.dout, L.lse, L.rowstat, p.N, rows, x);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  static int regs = -1;
  auto kern = bwd_fused_kernel<D, MODS, MASKS>;
  if ((e = check_regs(kern, regs, FU_LAUNCH_REGS)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FuCfg<D>::SMEM_BYTES)) !=
      cudaSuccess)
    return e;
  const long long items = (long long)p.nT * p.B * p.Hkv;
  const unsigned grid = (unsigned)(items < L.sms ? items : L.sms);
  if (L.events[1]) cudaEventRecord(L.events[1], st);
  kern<<<grid, FU_THREADS, FuCfg<D>::SMEM_BYTES, st>>>(L.tq, L.tk, L.tv, L.tdo, L.rowstat, L.qscale, L.dqacc,
                                                      L.ticket, (__nv_bfloat16*)L.dk, (__nv_bfloat16*)L.dv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (L.events[2]) cudaEventRecord(L.events[2], st);
  const long long dq_rows = (long long)p.B * p.Hq * p.N;
  dq_convert_kernel<D><<<(unsigned)((dq_rows * (D / 16) + 255) / 256), 256, 0, st>>>(
      L.dqacc, L.qscale, (__nv_bfloat16*)L.dq, p.N, p.nT, p.scale, dq_rows);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (L.events[3]) cudaEventRecord(L.events[3], st);
  return cudaGetLastError();
}

cudaError_t launch_bwd_fused(const BwdLaunch& L, int d, bool mods, bool masks, cudaStream_t st) {
  if (d != 128) return cudaErrorInvalidValue;
  return mods ? launch_fused_t<true, true>(L, st)
              : masks ? launch_fused_t<false, true>(L, st) : launch_fused_t<false, false>(L, st);
}

}  // namespace attn
