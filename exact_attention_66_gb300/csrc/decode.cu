// Decode step over a paged K/V cache for sm_103a: the newest token of every
// sequence attends to all of that sequence's cached keys, which are read
// through a block table of 16-row blocks.
//
// Method ("Les kernels d'attention rapide et la fusion d'opérateurs
// accélèrent les modèles d'IA", section "Attention de type FlashAttention et
// attention paginée"): the K/V cache grows by one token per step and is
// stored in fixed-size blocks that a block table maps from logical to
// physical positions; the attention kernel translates each position through
// that table.  The softmax is the forward's exact online softmax (running
// max and sum, output divided by the sum at the end).
//
// GB300 design:
//  * a decode step reads the whole cache once and does 4 G FLOP per cached
//    key and head dimension for a GQA group of G query heads (about 8 FLOP
//    per byte at G = 8): it is bound by HBM, not by the tensor cores;
//  * the work is cut into items (sequence, KV head, chunk of `ct` key tiles of
//    128) and a persistent grid of one CTA per SM walks its items
//    round-robin.  The TMA producer runs ahead across item boundaries, so an
//    SM keeps its loads in flight from its first tile to its last;
//  * the G query heads of a KV head are the rows of one 128-row tcgen05 tile
//    (rows >= G stay zero): S = Q K^T and O += P V are each one MMA chain
//    per key tile, and every K and V row is read once for all G heads;
//  * a key tile arrives as eight 16-row TMA boxes (one per cache block) in a
//    4-slot ring, in the order K(t0), K(t1), V(t0), K(t2), V(t1), ... so that
//    S of the next tile is computed while the softmax of this one runs;
//  * each item leaves O / l (fp32) and its log2-sum-exp in a workspace, and
//    a second kernel merges the chunks of every (sequence, head) by their
//    LSE.
#include "common.cuh"
#include "launch.h"
#include "softmax.cuh"

namespace attn {

namespace {

constexpr int DEC_D = 128;
constexpr int DEC_THREADS = 256;
constexpr int DEC_TB = TILE * DEC_D * 2;  // one bf16 tile of 128 rows (32 KB)
constexpr int DEC_RST = 4;                // K/V ring slots
constexpr int DEC_Q_OFF = 0;              // two Q tiles (item parity)
constexpr int DEC_P_OFF = 2 * DEC_TB;
constexpr int DEC_R_OFF = 3 * DEC_TB;
constexpr int DEC_BAR_OFF = DEC_R_OFF + DEC_RST * DEC_TB;
constexpr int DEC_SMEM = smem_one_cta(DEC_BAR_OFF + 256 + 1024);
static_assert(DEC_SMEM <= 232448, "decode shared memory exceeds 227 KB");

struct DecBars {
  uint64_t q_full[2], q_empty[2];        // Q tile of an item (TMA) / its last S done (commit)
  uint64_t full[DEC_RST], empty[DEC_RST];  // K/V ring
  uint64_t s_full[2], s_free[2];         // S buffers
  uint64_t p_full, o_full, o_free;       // P written, P V done, O read by the epilogue
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DecBars) <= 256, "decode barrier block");

// Sequence b's length, first key tile and number of chunks.  A length outside
// [0, 16 * bt_stride] is reported and the sequence treated as empty.
__device__ __forceinline__ void seq_chunks(const DecodeParams& p, int b, int& L, int& J0, int& n) {
  L = p.seqlens[b];
  if (L < 0 || L > 16 * p.bt_stride) {
    atomicCAS(p.status, 0, DEV_ERR_BOUNDS);
    L = 0;
  }
  const int J_hi = (L + TILE - 1) / TILE;
  J0 = (p.flags & MOD_WINDOW) ? max(0, L - p.window) / TILE : 0;
  n = L > 0 ? (J_hi - J0 + p.ct - 1) / p.ct : 0;
}

// One CTA: per-sequence chunk counts and the exclusive prefix of the items
// (chunks x KV heads) over the sequences.
__global__ void __launch_bounds__(1024) decode_setup_kernel(const DecodeParams p) {
  __shared__ int part[1024];
  const int t = threadIdx.x;
  const int per = (p.B + 1023) / 1024;
  const int b0 = min(p.B, t * per), b1 = min(p.B, b0 + per);
  int sum = 0;
  for (int b = b0; b < b1; ++b) {
    int L, J0, n;
    seq_chunks(p, b, L, J0, n);
    sum += n * p.Hkv;
  }
  part[t] = sum;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan
    const int v = t >= off ? part[t - off] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  int run = t > 0 ? part[t - 1] : 0;
  for (int b = b0; b < b1; ++b) {
    int L, J0, n;
    seq_chunks(p, b, L, J0, n);
    p.seq_info[b] = make_int4(L, J0, n, run);
    run += n * p.Hkv;
  }
  if (t == 1023) *p.n_items = part[1023];
}

// A key tile of this CTA's work, in the order every role walks it.
struct DecTile {
  int b, hk, c, L, J;
  int item;          // ordinal of its item among this CTA's items
  bool first, last;  // first / last tile of the item
};

struct DecWalker {
  int x, total, item, b, hk, c, L, J, J_first, J_end;
  __device__ void init(const DecodeParams& p) {
    x = blockIdx.x;
    total = *p.n_items;
    item = -1;
    J = J_end = 0;
  }
  // Next tile; false when this CTA has none left.
  __device__ bool next(const DecodeParams& p, DecTile& t) {
    if (J >= J_end) {
      if (item >= 0) x += gridDim.x;
      if (x >= total) return false;
      ++item;
      int lo = 0, hi = p.B - 1;  // last sequence whose first item is <= x
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.seq_info[mid].w <= x) lo = mid;
        else hi = mid - 1;
      }
      const int4 si = p.seq_info[lo];
      b = lo;
      L = si.x;
      const int r = x - si.w;
      hk = r / si.z;
      c = r - hk * si.z;
      J_first = si.y + c * p.ct;
      J_end = min(J_first + p.ct, (L + TILE - 1) / TILE);
      J = J_first;
    }
    t.b = b;
    t.hk = hk;
    t.c = c;
    t.L = L;
    t.J = J;
    t.item = item;
    t.first = J == J_first;
    t.last = J + 1 == J_end;
    ++J;
    return true;
  }
};

// S(tmem, 128 x 128 fp32) = Q K^T, both K-major 128-byte swizzled bf16 tiles
// of 256-byte rows (two 16 KB column chunks).
__device__ __forceinline__ void dec_issue_s(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, false);
  const uint64_t ad = opaque(sdesc_sw128(q_smem, 16, 1024)), bd = opaque(sdesc_sw128(k_smem, 16, 1024));
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
    mma_f16_ss(d_tmem, sdesc_add(ad, off), sdesc_add(bd, off), id, kk > 0 ? 1u : 0u);
  }
}

// O(tmem) (+)= P V: P K-major (128 keys), V MN-major (128 keys x 128).
__device__ __forceinline__ void dec_issue_pv(uint32_t o_tmem, uint32_t p_smem, uint32_t v_smem, bool first) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, true);
  const uint64_t pd = opaque(sdesc_sw128(p_smem, 16, 1024)), vd = opaque(sdesc_sw128(v_smem, 16384, 1024));
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t poff = (kk / 4) * 16384 + (kk % 4) * 32;
    mma_f16_ss(o_tmem, sdesc_add(pd, poff), sdesc_add(vd, kk * 16 * 128), id, (first && kk == 0) ? 0u : 1u);
  }
}

// MODS: soft-cap / ALiBi compiled in (the window is a column interval and
// runs in both variants).
template <bool MODS>
__global__ void __launch_bounds__(DEC_THREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  DecBars& S = *reinterpret_cast<DecBars*>(smem + DEC_BAR_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();
  const int G = p.G;
  const int nsw = (G + 31) / 32;  // softmax warps (4 .. 3 + nsw): one thread per query head

  // Rows >= G of the Q tiles never receive data: zero them (and P) once.
  for (int g = threadIdx.x; g < 3 * DEC_TB / 16; g += DEC_THREADS) {
    const int row = ((g * 16) % 16384) / 128;
    if (g * 16 >= 2 * DEC_TB || row >= G)
      *reinterpret_cast<uint4*>(smem + g * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_async_smem();
  if (threadIdx.x == 0) {
    S.abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.q_full[i], 1);
      mbar_init(&S.q_empty[i], 1);
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.s_free[i], 32 * nsw);
    }
    for (int s = 0; s < DEC_RST; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.p_full, 32 * nsw);
    mbar_init(&S.o_full, 1);
    mbar_init(&S.o_free, 32 * nsw);
    mbar_init(&S.drain, 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;  // S0 @0, S1 @128, O @256
  const uint32_t sQ = smem_u32(smem + DEC_Q_OFF), sP = smem_u32(smem + DEC_P_OFF);
  const uint32_t sR = smem_u32(smem + DEC_R_OFF);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      DecWalker w;
      w.init(p);
      int r = 0, nq = 0;  // ring loads, Q loads
      auto load_q = [&](const DecTile& t) -> bool {
        const int qb = t.item & 1;
        if (t.item >= 2 && !mbar_wait(&S.q_empty[qb], ((t.item >> 1) - 1) & 1, ab)) return false;
        mbar_arrive_tx(&S.q_full[qb], 2 * G * 128);
        for (int ch = 0; ch < 2; ++ch)
          tma_load_3d(smem + DEC_Q_OFF + qb * DEC_TB + ch * 16384, &tq, &S.q_full[qb], ch * 64, 0,
                      t.b * p.Hkv + t.hk);
        ++nq;
        return true;
      };
      auto load_kv = [&](const CUtensorMap* map, const DecTile& t) -> bool {
        // The tile's 8 cache blocks; blocks wholly past the sequence end take an
        // out-of-range index (TMA fills zeros), table entries outside
        // [0, kv_blocks) are an error.
        int z[TILE / 16];
#pragma unroll
        for (int sb = 0; sb < TILE / 16; ++sb) {
          const int lb = t.J * (TILE / 16) + sb;
          z[sb] = p.kv_blocks * p.Hkv;
          if (lb * 16 < t.L) {
            const int e = __ldg(p.block_table + (size_t)t.b * p.bt_stride + lb);
            if (e < 0 || e >= p.kv_blocks) {
              raise_error(ab, DEV_ERR_BOUNDS);
              return false;
            }
            z[sb] = e * p.Hkv + t.hk;
          }
        }
        const int st = r % DEC_RST;
        if (!mbar_wait(&S.empty[st], ((r / DEC_RST) & 1) ^ 1, ab)) return false;
        mbar_arrive_tx(&S.full[st], DEC_TB);
        uint8_t* dst = smem + DEC_R_OFF + st * DEC_TB;
#pragma unroll
        for (int sb = 0; sb < TILE / 16; ++sb)
#pragma unroll
          for (int ch = 0; ch < 2; ++ch)
            tma_load_3d(dst + ch * 16384 + sb * 2048, map, &S.full[st], ch * 64, 0, z[sb]);
        ++r;
        return true;
      };
      DecTile cur, nxt;
      bool have = w.next(p, cur);
      bool ok = !have || (load_q(cur) && load_kv(&tk, cur));
      while (ok && have) {
        const bool hn = w.next(p, nxt);
        if (hn && nxt.first && !(ok = load_q(nxt))) break;
        if (hn && !(ok = load_kv(&tk, nxt))) break;
        if (!(ok = load_kv(&tv, cur))) break;
        cur = nxt;
        have = hn;
      }
      // Every copy issued lands before the CTA can exit.
      for (int qb = 0; qb < 2; ++qb)
        if (nq > qb) mbar_wait_drain(&S.q_full[qb], ((nq - 1 - qb) >> 1) & 1);
      for (int s = 0; s < DEC_RST; ++s)
        if (r > s) mbar_wait_drain(&S.full[s], ((r - 1 - s) / DEC_RST) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      DecWalker w;
      w.init(p);
      int r = 0, ns = 0;  // ring slots consumed, S tiles issued
      bool ok = true;
      auto slot = [&](int& st) -> bool {
        st = r % DEC_RST;
        const bool good = mbar_wait(&S.full[st], (r / DEC_RST) & 1, ab);
        ++r;
        tc_fence_after();
        return good;
      };
      auto issue_s = [&](const DecTile& t, int ks) -> bool {
        const int qb = t.item & 1;
        if (t.first && !mbar_wait(&S.q_full[qb], (t.item >> 1) & 1, ab)) return false;
        if (ns >= 2 && !mbar_wait(&S.s_free[ns & 1], ((ns >> 1) - 1) & 1, ab)) return false;
        tc_fence_after();
        dec_issue_s(tmem + (uint32_t)(ns & 1) * 128, sQ + qb * DEC_TB, sR + ks * DEC_TB);
        mma_commit(&S.s_full[ns & 1]);
        mma_commit(&S.empty[ks]);
        if (t.last) mma_commit(&S.q_empty[qb]);
        ++ns;
        return true;
      };
      DecTile cur, nxt;
      bool have = w.next(p, cur);
      int ks = 0, vs = 0, npv = 0;
      if (have) ok = slot(ks) && issue_s(cur, ks);
      while (ok && have) {
        const bool hn = w.next(p, nxt);
        if (hn && !(ok = slot(ks) && issue_s(nxt, ks))) break;
        if (!(ok = slot(vs))) break;
        if (!(ok = mbar_wait(&S.p_full, npv & 1, ab))) break;
        // The first P V of an item overwrites O: the epilogue of the previous
        // item must have read it.
        if (cur.first && cur.item >= 1 && !(ok = mbar_wait(&S.o_free, (cur.item - 1) & 1, ab))) break;
        tc_fence_after();
        dec_issue_pv(tmem + 256, sP, sR + vs * DEC_TB, cur.first);
        mma_commit(&S.o_full);
        mma_commit(&S.empty[vs]);
        ++npv;
        cur = nxt;
        have = hn;
      }
      // Every MMA issued completes before TMEM can be released.
      mma_commit(&S.drain);
      mbar_wait_drain(&S.drain, 0);
    }
  } else if (warp >= 4 && warp < 4 + nsw) {
    // -------------------------------------------------------------- softmax
    const int wq = warp & 3;
    const int r = wq * 32 + lane;  // query head r of the group (TMEM lane r)
    const bool active = r < G;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tO = tmem + lane_off + 256;
    uint8_t* p_tile = smem + DEC_P_OFF;
    const bool win = (p.flags & MOD_WINDOW) != 0;
    const bool sc = MODS && (p.flags & MOD_SOFTCAP);
    const bool al = MODS && (p.flags & MOD_ALIBI);
    const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t sc_in2 = f2_pack(p.sc_in, p.sc_in), sc_out2 = f2_pack(p.sc_out, p.sc_out);
    DecWalker w;
    w.init(p);
    DecTile t;
    float m = -INFINITY, l = 0.f, al2 = 0.f;
    int n = 0;  // tiles processed
    bool ok = true;
    while (ok && w.next(p, t)) {
      const int hq = t.hk * G + min(r, G - 1);
      if (t.first) {
        m = -INFINITY;
        l = 0.f;
        if (al) {
          const float slope = p.slopes != nullptr ? p.slopes[hq] : exp2f(-8.0f * (float)(hq + 1) / (float)p.Hq);
          al2 = slope * LOG2E;
        }
      }
      if (!(ok = wait_warp(&S.s_full[n & 1], (n >> 1) & 1, ab))) break;
      tc_fence_after();
      uint32_t s[128];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        tmem_ld32(tmem + lane_off + (uint32_t)(n & 1) * 128 + q4 * 32, *reinterpret_cast<uint32_t(*)[32]>(&s[q4 * 32]));
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(&s[q4 * 32]));
      tc_fence_before();
      mbar_arrive(&S.s_free[n & 1]);

      // Keys j0 + c are allowed iff lo_lim < c <= hi_lim: j <= i = L - 1, and
      // with the window i - j < W.
      const int j0 = t.J * TILE;
      const int hi_lim = t.L - 1 - j0;
      const int lo_lim = win ? t.L - p.window - 1 - j0 : -1;
      const bool partial = hi_lim < TILE - 1 || lo_lim >= 0;
      float mt, mul;
      if (!(sc || al)) {
        if (partial) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > hi_lim || c <= lo_lim) s[c] = __float_as_uint(-INFINITY);
        }
        mt = row_max128(s) * p.scale_log2;
        mul = p.scale_log2;
      } else {
        // log2-unit logits: soft-cap c tanh(scale s / c), then ALiBi
        // slope (j - i).
        const float al_base = al2 * (float)(j0 - (t.L - 1));
        const uint64_t al2x = f2_pack(al2, al2), alb = f2_pack(al_base, al_base);
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          uint64_t x2 = f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1]));
          x2 = sc ? f2_mul(tanh2_exp(f2_mul(x2, sc_in2)), sc_out2) : f2_mul(x2, sl2);
          if (al) x2 = f2_fma(f2_pack((float)c, (float)(c + 1)), al2x, f2_add(x2, alb));
          float x0, x1;
          f2_unpack(x2, x0, x1);
          s[c] = __float_as_uint(x0);
          s[c + 1] = __float_as_uint(x1);
        }
        if (partial) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > hi_lim || c <= lo_lim) s[c] = __float_as_uint(-INFINITY);
        }
        mt = row_max128(s);
        mul = 1.0f;
      }

      // Running max, moved only when the row max grows by more than 2^8.
      const float mn = fmaxf(m, mt);
      bool need = false;
      float alpha = 1.0f;
      if (t.first) {
        m = mn;
      } else if (mn > m + RESCALE_THRESHOLD) {
        need = true;
        alpha = ex2(m - mn);
        l *= alpha;
        m = mn;
      }
      const float mu = (m == -INFINITY) ? 0.f : m;
      uint32_t unused_lo[64];
      l += exp_bf16<false>(s, unused_lo, mul, mu);

      // The previous P V must be done before P is overwritten or O rescaled.
      if (n > 0) {
        if (!(ok = wait_warp(&S.o_full, (n - 1) & 1, ab))) break;
        tc_fence_after();
        if (!t.first && __any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int q4 = 0; q4 < DEC_D / 32; ++q4) {
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
      if (active) {  // P row r into the 128-byte swizzled K-major tile
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const uint32_t addr = (uint32_t)((g >> 3) * 16384 + r * 128 + (((g & 7) ^ (r & 7)) << 4));
          *reinterpret_cast<uint4*>(p_tile + addr) = make_uint4(s[4 * g], s[4 * g + 1], s[4 * g + 2], s[4 * g + 3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&S.p_full);

      if (t.last) {
        // ------------------------------------------------------ item epilogue
        if (!(ok = wait_warp(&S.o_full, n & 1, ab))) break;
        tc_fence_after();
        const float inv = l > 0.f ? 1.0f / l : 0.f;
        const size_t prow = ((size_t)t.b * p.Hq + hq) * p.max_chunks + t.c;
        float4* dst = reinterpret_cast<float4*>(p.o_part + prow * DEC_D);
#pragma unroll
        for (int q4 = 0; q4 < DEC_D / 32; ++q4) {
          uint32_t ov[32];
          tmem_ld32(tO + q4 * 32, ov);
          tmem_wait_ld(ov);
          if (active) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[q4 * 8 + c] = make_float4(__uint_as_float(ov[4 * c]) * inv, __uint_as_float(ov[4 * c + 1]) * inv,
                                            __uint_as_float(ov[4 * c + 2]) * inv, __uint_as_float(ov[4 * c + 3]) * inv);
          }
        }
        if (active) p.lse_part[prow] = l > 0.f ? m + log2f(l) : -INFINITY;
        tc_fence_before();
        mbar_arrive(&S.o_free);
      }
      ++n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// One warp per (sequence, query head): merge the chunks' O / l by their LSE.
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p, __nv_bfloat16* __restrict__ o,
                                                             float* __restrict__ lse) {
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.B * p.Hq) return;
  const int b = gw / p.Hq;
  const int n = p.seq_info[b].z;
  const float* lp = p.lse_part + (size_t)gw * p.max_chunks;
  const float4* op = reinterpret_cast<const float4*>(p.o_part + (size_t)gw * p.max_chunks * DEC_D);
  float M = -INFINITY;
  for (int c = lane; c < n; c += 32) M = fmaxf(M, lp[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -INFINITY) {
    for (int c = 0; c < n; ++c) {
      const float wc = exp2f(lp[c] - M);
      const float4 v = op[(size_t)c * (DEC_D / 4) + lane];
      W += wc;
      acc.x += wc * v.x;
      acc.y += wc * v.y;
      acc.z += wc * v.z;
      acc.w += wc * v.w;
    }
  }
  const float inv = W > 0.f ? 1.0f / W : 0.f;
  uint2 pk;
  pk.x = pack_bf16(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(o + (size_t)gw * DEC_D)[lane] = pk;
  if (lane == 0) lse[gw] = W > 0.f ? (M + log2f(W)) * LN2 : -INFINITY;
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& L, bool mods, cudaStream_t st) {
  decode_setup_kernel<<<1, 1024, 0, st>>>(L.p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = mods ? decode_kernel<true> : decode_kernel<false>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DEC_SMEM)) != cudaSuccess)
    return e;
  kern<<<(unsigned)L.grid, DEC_THREADS, DEC_SMEM, st>>>(L.tq, L.tk, L.tv, L.p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long warps = (long long)L.p.B * L.p.Hq;
  decode_combine_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(L.p, (__nv_bfloat16*)L.o, L.lse);
  return cudaGetLastError();
}

}  // namespace attn
