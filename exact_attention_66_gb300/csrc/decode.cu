// Decode step over a paged K/V cache for sm_103a: the newest token (or the T
// newest tokens, causal among themselves) of every sequence attends to that
// sequence's cached keys, which are read through a block table of 16-row
// blocks.
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
//  * the G query heads x T tokens of a KV head are the rows of one 128-row
//    tcgen05 tile (rows >= G T stay zero): S = Q K^T and O += P V are each one
//    MMA chain per key tile, and every K and V row is read once for all of
//    them;
//  * a key tile arrives as sixteen 2 KB TMA boxes (one per cache block and
//    64-column half), issued by 16 lanes of a producer warp at once: one warp
//    streams K tiles and another V tiles, each through its own 2-slot ring,
//    so that the one-box-per-instruction issue rate of a single thread does
//    not limit the stream; S of the next tile is computed while the softmax
//    of this one runs;
//  * each item leaves O / l (fp32) and its log2-sum-exp in a workspace, and
//    a second kernel merges the chunks of every (sequence, head) by their
//    LSE.
#include "common.cuh"
#include "launch.h"
#include "softmax.cuh"

namespace attn {

namespace {

constexpr int DEC_THREADS = 256;

// Shared-memory layout.  The MMAs read Q and P as 128-row tiles, of which only
// the R = G T rows of the query heads and tokens matter.  A Q or P tile keeps
// QG 8-row swizzle groups (QG KB) per 64-column chunk:
//  * QG = 1 (R <= 8): the MMA descriptor's stride between 8-row groups is 0,
//    so its other fifteen groups re-read the same eight rows;
//  * QG = 4 (R <= 32): the stride is 1 KB and groups 4..15 read the 12 KB
//    after the chunk -- the next chunk, P or the K ring, always inside the
//    CTA's shared memory, since the rings follow Q and P;
//  * QG = 16: whole 128-row tiles.
// The S and O rows that rows >= 8 QG produce are never read, and neither are
// the S / O rows >= R: one softmax thread per row < R.  The room saved goes to
// deeper K and V rings, i.e. more bytes in flight.
template <int D, int QG>
struct DecCfg {
  static constexpr int CH = D / 64;                     // 64-column chunks of a Q / K / V row
  static constexpr int TB = TILE * D * 2;               // one bf16 K or V tile of 128 rows
  static constexpr int QCH = QG * 1024;                 // one 64-column chunk of a Q / P tile
  static constexpr int QTB = CH * QCH;                  // one Q tile
  static constexpr int PTB = 2 * QCH;                   // the P tile (128 keys)
  static constexpr uint32_t QSBO = QG == 1 ? 0u : 1024u;  // MMA stride between 8-row groups
  // K ring and V ring slots (shared memory left after Q and P; twice as many
  // of the half-size tiles of d = 64)
  static constexpr int KS = (QG < 16 ? 3 : 2) * (D == 64 ? 2 : 1), VS = KS;
  static constexpr int Q_OFF = 0;                       // two Q tiles (item parity)
  static constexpr int P_OFF = 2 * QTB;
  static constexpr int K_OFF = P_OFF + PTB;
  static constexpr int V_OFF = K_OFF + KS * TB;
  static constexpr int BAR_OFF = V_OFF + VS * TB;
  static constexpr int SMEM = smem_one_cta(BAR_OFF + 512 + 1024);
  static_assert(SMEM <= 232448, "decode shared memory exceeds 227 KB");
  static_assert(K_OFF % 1024 == 0, "swizzled tiles need 1 KB alignment");
  // Reads of groups QG..15 past the last Q / P chunk stay inside the K ring.
  static_assert(QG == 1 || QG == 16 || P_OFF + PTB - QCH + 16 * 1024 <= V_OFF + VS * TB,
                "partial Q / P tiles must be followed by 16 KB of shared memory");
};
constexpr int DEC_MAX_SLOTS = 6;

struct DecBars {
  uint64_t q_full[2], q_empty[2];        // Q tile of an item (TMA) / its last S done (commit)
  uint64_t kfull[DEC_MAX_SLOTS], kempty[DEC_MAX_SLOTS];  // K ring
  uint64_t vfull[DEC_MAX_SLOTS], vempty[DEC_MAX_SLOTS];  // V ring
  uint64_t s_full[2], s_free[2];         // S buffers
  uint64_t p_full, o_full;               // P written, P V done
  uint64_t o_free[2];                    // O buffer read by its item's epilogue
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DecBars) <= 512, "decode barrier block");

// Sequence b's length, first key tile and number of chunks.  A length outside
// [0, 16 * bt_stride] is reported and the sequence treated as empty.
__device__ __forceinline__ void seq_chunks(const DecodeParams& p, int b, int& L, int& J0, int& n) {
  L = p.seqlens[b];
  if (L < 0 || L > 16 * p.bt_stride) {
    atomicCAS(p.status, 0, DEV_ERR_BOUNDS);
    L = 0;
  }
  const int J_hi = (L + TILE - 1) / TILE;
  // keys of the earliest new token, at L - T, reach back to L - T - W + 1
  J0 = (p.flags & MOD_WINDOW) ? max(0, L - p.q_len - p.window + 1) / TILE : 0;
  n = L > 0 ? (J_hi - J0 + p.ct - 1) / p.ct : 0;
}

// One CTA: per-sequence chunk counts and the exclusive prefix of the items
// (chunks x KV heads) over the sequences.  Thread t owns sequences
// [t * per, (t + 1) * per); the scan runs on warp shuffles.
constexpr int DEC_SETUP_PER = 8;  // sequences a thread keeps in registers
__global__ void __launch_bounds__(1024) decode_setup_kernel(const DecodeParams p) {
  __shared__ int warp_sum[32];
  pdl_launch_dependents();  // the main kernel's prologue needs nothing from here
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int per = (p.B + 1023) / 1024;
  const int b0 = min(p.B, t * per), b1 = min(p.B, b0 + per);
  int L[DEC_SETUP_PER], J0[DEC_SETUP_PER], n[DEC_SETUP_PER];
  int sum = 0;
  for (int base = b0; base < b1; base += DEC_SETUP_PER) {  // one pass when per <= DEC_SETUP_PER
    const int m = min(DEC_SETUP_PER, b1 - base);
#pragma unroll
    for (int k = 0; k < DEC_SETUP_PER; ++k)
      if (k < m) seq_chunks(p, base + k, L[k], J0[k], n[k]);
#pragma unroll
    for (int k = 0; k < DEC_SETUP_PER; ++k)
      if (k < m) sum += n[k] * p.Hkv;
  }
  int incl = sum;  // inclusive scan over the block
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_sum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int w = warp_sum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += v;
    }
    warp_sum[lane] = w;
  }
  __syncthreads();
  int run = incl - sum + (wid > 0 ? warp_sum[wid - 1] : 0);
  for (int base = b0; base < b1; base += DEC_SETUP_PER) {
    const int m = min(DEC_SETUP_PER, b1 - base);
    if (per > DEC_SETUP_PER) {  // more than fit in registers: recompute this group
#pragma unroll
      for (int k = 0; k < DEC_SETUP_PER; ++k)
        if (k < m) seq_chunks(p, base + k, L[k], J0[k], n[k]);
    }
#pragma unroll
    for (int k = 0; k < DEC_SETUP_PER; ++k) {
      if (k < m) {
        p.seq_info[base + k] = make_int4(L[k], J0[k], n[k], run);
        run += n[k] * p.Hkv;
      }
    }
  }
  if (t == 1023) *p.n_items = warp_sum[31];
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

// S(tmem, 128 x 128 fp32) = Q K^T: Q and K K-major 128-byte swizzled bf16
// tiles of D columns, K as 16 KB 64-column chunks, Q in the layout of C.
template <typename C>
__device__ __forceinline__ void dec_issue_s(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t id = idesc_bf16(128, 128, false, false);
  const uint64_t ad = opaque(sdesc_sw128(q_smem, 16, C::QSBO)), bd = opaque(sdesc_sw128(k_smem, 16, 1024));
#pragma unroll
  for (int kk = 0; kk < C::CH * 4; ++kk) {
    const uint32_t step = (kk % 4) * 32;
    mma_f16_ss(d_tmem, sdesc_add(ad, (kk / 4) * C::QCH + step), sdesc_add(bd, (kk / 4) * 16384 + step), id,
               kk > 0 ? 1u : 0u);
  }
}

// O(tmem) (+)= P V: P K-major (128 keys, layout of C), V MN-major (128 keys x D).
template <typename C>
__device__ __forceinline__ void dec_issue_pv(uint32_t o_tmem, uint32_t p_smem, uint32_t v_smem, bool first) {
  constexpr uint32_t id = idesc_bf16(128, C::CH * 64, false, true);
  const uint64_t pd = opaque(sdesc_sw128(p_smem, 16, C::QSBO)), vd = opaque(sdesc_sw128(v_smem, 16384, 1024));
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t poff = (kk / 4) * C::QCH + (kk % 4) * 32;
    mma_f16_ss(o_tmem, sdesc_add(pd, poff), sdesc_add(vd, kk * 16 * 128), id, (first && kk == 0) ? 0u : 1u);
  }
}

// MODS: soft-cap / ALiBi compiled in (the window is a column interval and
// runs in both variants); QG: 8-row groups of the Q / P tiles (8 QG >= R).
template <int D, bool MODS, int QG>
__global__ void __launch_bounds__(DEC_THREADS, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const DecodeParams p) {
  using C = DecCfg<D, QG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  DecBars& S = *reinterpret_cast<DecBars*>(smem + C::BAR_OFF);
  const Abort ab{&S.abort, p.status};
  const int warp = warp_id(), lane = lane_id();
  const int G = p.G;
  const int R = G * p.q_len;      // tile rows in use: (query head, token) pairs
  const int nsw = (R + 31) / 32;  // softmax warps (4 .. 3 + nsw): one thread per row

  // Rows >= R of the Q tiles never receive data: zero them (and P) once.
  for (int g = threadIdx.x; g < (2 * C::QTB + C::PTB) / 16; g += DEC_THREADS) {
    const int row = ((g * 16) % C::QCH) / 128;
    if (g * 16 >= 2 * C::QTB || row >= R)
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
    for (int s = 0; s < C::KS; ++s) {
      mbar_init(&S.kfull[s], 1);
      mbar_init(&S.kempty[s], 1);
    }
    for (int s = 0; s < C::VS; ++s) {
      mbar_init(&S.vfull[s], 1);
      mbar_init(&S.vempty[s], 1);
    }
    mbar_init(&S.p_full, 32 * nsw);
    mbar_init(&S.o_full, 1);
    mbar_init(&S.o_free[0], 32 * nsw);
    mbar_init(&S.o_free[1], 32 * nsw);
    mbar_init(&S.drain, 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  // The item table comes from the set-up kernel, which may still be running.
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;  // S0 @0, S1 @128, O0 @256, O1 @384 (by item parity)
  const uint32_t sQ = smem_u32(smem + C::Q_OFF), sP = smem_u32(smem + C::P_OFF);
  const uint32_t sK = smem_u32(smem + C::K_OFF), sV = smem_u32(smem + C::V_OFF);

  if (warp == 0 || warp == 3) {
    // ----------------------------------------------------------- TMA producers
    // Warp 0 streams Q (once per item) and the K tiles, warp 3 the V tiles.
    const bool is_k = warp == 0;
    if (lane == 0) {
      tma_prefetch_desc(is_k ? &tk : &tv);
      if (is_k) tma_prefetch_desc(&tq);
    }
    uint64_t* full = is_k ? S.kfull : S.vfull;
    uint64_t* empty = is_k ? S.kempty : S.vempty;
    const int slots = is_k ? C::KS : C::VS;
    uint8_t* ring = smem + (is_k ? C::K_OFF : C::V_OFF);
    const CUtensorMap* map = is_k ? &tk : &tv;
    DecWalker w;
    w.init(p);
    int r = 0, nq = 0;  // tiles loaded, Q loads
    bool ok = true;
    // Lane l < 16 copies box (cache block l / 2, column half l % 2) of a tile.
    // Blocks wholly past the sequence end take an out-of-range index (TMA
    // fills zeros); table entries outside [0, kv_blocks) are an error.  The
    // entries of the next tile are fetched while this one waits for its slot.
    auto lookup = [&](const DecTile& t, int& z, bool& bad) {
      z = p.kv_blocks * p.Hkv;
      bad = false;
      if (lane < 8 * C::CH) {
        const int lb = t.J * (TILE / 16) + lane / C::CH;
        if (lb * 16 < t.L) {
          const int e = __ldg(p.block_table + (size_t)t.b * p.bt_stride + lb);
          bad = e < 0 || e >= p.kv_blocks;
          z = e * p.Hkv + t.hk;
        }
      }
    };
    DecTile t, tn;
    int z = 0;
    bool bad = false;
    bool have = w.next(p, t);
    if (have) lookup(t, z, bad);
    while (ok && have) {
      if (is_k && t.first) {
        const int qb = t.item & 1;
        if (lane == 0) {
          ok = t.item < 2 || mbar_wait(&S.q_empty[qb], ((t.item >> 1) - 1) & 1, ab);
          if (ok) {
            mbar_arrive_tx(&S.q_full[qb], C::CH * R * 128);
            for (int ch = 0; ch < C::CH; ++ch)
              tma_load_3d(smem + C::Q_OFF + qb * C::QTB + ch * C::QCH, &tq, &S.q_full[qb], ch * 64, 0,
                          t.b * p.Hkv + t.hk);
          }
        }
        if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
        ++nq;
      }
      const int st = r % slots;
      if (lane == 0) ok = mbar_wait(&empty[st], ((r / slots) & 1) ^ 1, ab);
      if (!(ok = __shfl_sync(0xffffffffu, ok, 0))) break;
      if (__any_sync(0xffffffffu, bad)) {  // the table entries are needed only now
        if (lane == 0) raise_error(ab, DEV_ERR_BOUNDS);
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive_tx(&full[st], C::TB);
      __syncwarp();
      if (lane < 8 * C::CH)
        tma_load_3d(ring + st * C::TB + (lane % C::CH) * 16384 + (lane / C::CH) * 2048, map, &full[st],
                    (lane % C::CH) * 64, 0, z);
      ++r;
      have = w.next(p, tn);
      if (have) {
        t = tn;
        lookup(t, z, bad);
      }
    }
    // Every copy issued lands before the CTA can exit.
    if (lane == 0) {
      for (int qb = 0; qb < 2; ++qb)
        if (nq > qb) mbar_wait_drain(&S.q_full[qb], ((nq - 1 - qb) >> 1) & 1);
      for (int s = 0; s < slots; ++s)
        if (r > s) mbar_wait_drain(&full[s], ((r - 1 - s) / slots) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      DecWalker w;
      w.init(p);
      int nk = 0, nv = 0, ns = 0;  // K and V tiles consumed, S tiles issued
      bool ok = true;
      auto kslot = [&](int& st) -> bool {
        st = nk % C::KS;
        const bool good = mbar_wait(&S.kfull[st], (nk / C::KS) & 1, ab);
        ++nk;
        tc_fence_after();
        return good;
      };
      auto vslot = [&](int& st) -> bool {
        st = nv % C::VS;
        const bool good = mbar_wait(&S.vfull[st], (nv / C::VS) & 1, ab);
        ++nv;
        tc_fence_after();
        return good;
      };
      auto issue_s = [&](const DecTile& t, int ks) -> bool {
        const int qb = t.item & 1;
        if (t.first && !mbar_wait(&S.q_full[qb], (t.item >> 1) & 1, ab)) return false;
        if (ns >= 2 && !mbar_wait(&S.s_free[ns & 1], ((ns >> 1) - 1) & 1, ab)) return false;
        tc_fence_after();
        dec_issue_s<C>(tmem + (uint32_t)(ns & 1) * 128, sQ + qb * C::QTB, sK + ks * C::TB);
        mma_commit(&S.s_full[ns & 1]);
        mma_commit(&S.kempty[ks]);
        if (t.last) mma_commit(&S.q_empty[qb]);
        ++ns;
        return true;
      };
      DecTile cur, nxt;
      bool have = w.next(p, cur);
      int ks = 0, vs = 0, npv = 0;
      if (have) ok = kslot(ks) && issue_s(cur, ks);
      while (ok && have) {
        const bool hn = w.next(p, nxt);
        if (hn && !(ok = kslot(ks) && issue_s(nxt, ks))) break;
        if (!(ok = vslot(vs))) break;
        if (!(ok = mbar_wait(&S.p_full, npv & 1, ab))) break;
        // The first P V of an item overwrites its O buffer: the epilogue of
        // the item two before, which used the same buffer, must have read it
        // (one barrier per buffer, so a later epilogue cannot alias its phase).
        if (cur.first && cur.item >= 2 &&
            !(ok = mbar_wait(&S.o_free[cur.item & 1], ((cur.item >> 1) - 1) & 1, ab)))
          break;
        tc_fence_after();
        dec_issue_pv<C>(tmem + 256 + (uint32_t)(cur.item & 1) * 128, sP, sV + vs * C::TB, cur.first);
        mma_commit(&S.o_full);
        mma_commit(&S.vempty[vs]);
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
    const int r = wq * 32 + lane;  // tile row (TMEM lane) r: query head r / T, token r % T
    const bool active = r < R;
    const int rr = min(r, R - 1);
    const int g = rr / p.q_len, tok = rr - g * p.q_len;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tO0 = tmem + lane_off + 256;  // + 128 for odd items
    uint8_t* p_tile = smem + C::P_OFF;
    const bool win = (p.flags & MOD_WINDOW) != 0;
    const bool sc = MODS && (p.flags & MOD_SOFTCAP);
    const bool al = MODS && (p.flags & MOD_ALIBI);
    const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t sc_in2 = f2_pack(p.sc_in, p.sc_in), sc_out2 = f2_pack(p.sc_out, p.sc_out);
    // An item's output is written once the next tile's P is out (or at the
    // end), so the softmax never waits for the item's last P V by itself.
    struct Pending {
      bool on;
      int buf;      // O buffer (item parity)
      size_t prow;  // row of the partial buffers: ((b * Hq + hq) * T + token) * max_chunks + chunk
      float m, l;   // running max (log2 units) and sum
    };
    Pending pend{false, 0, 0u, 0.f, 0.f};
    auto epilogue = [&](const Pending& e) {
      const float inv = e.l > 0.f ? 1.0f / e.l : 0.f;
      float4* dst = reinterpret_cast<float4*>(p.o_part + e.prow * D);
      const uint32_t tO = tO0 + (uint32_t)e.buf * 128;
#pragma unroll
      for (int q4 = 0; q4 < D / 32; ++q4) {
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
      if (active) p.lse_part[e.prow] = e.l > 0.f ? e.m + log2f(e.l) : -INFINITY;
      tc_fence_before();
      mbar_arrive(&S.o_free[e.buf]);
    };
    DecWalker w;
    w.init(p);
    DecTile t;
    float m = -INFINITY, l = 0.f, al2 = 0.f;
    int n = 0;  // tiles processed
    bool ok = true;
    while (ok && w.next(p, t)) {
      const int hq = t.hk * G + g;
      const int i = t.L - p.q_len + tok;  // this row's token position
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

      // Keys j0 + c are allowed iff lo_lim < c <= hi_lim: j <= i, and with
      // the window i - j < W (rows differ only by their token's position).
      const int j0 = t.J * TILE;
      const int hi_lim = i - j0;
      const int lo_lim = win ? i - p.window - j0 : -1;
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
        const float al_base = al2 * (float)(j0 - i);
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
          const uint32_t tO = tO0 + (uint32_t)(t.item & 1) * 128;
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
      if (active) {  // P row r into the 128-byte swizzled K-major tile
#pragma unroll
        for (int q16 = 0; q16 < 16; ++q16) {
          const uint32_t addr = (uint32_t)((q16 >> 3) * C::QCH + r * 128 + (((q16 & 7) ^ (r & 7)) << 4));
          *reinterpret_cast<uint4*>(p_tile + addr) =
              make_uint4(s[4 * q16], s[4 * q16 + 1], s[4 * q16 + 2], s[4 * q16 + 3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&S.p_full);

      // The finished item before this one: its last P V completed before P
      // was overwritten above, and its O buffer is not the one in use.
      if (pend.on) {
        epilogue(pend);
        pend.on = false;
      }
      if (t.last)
        pend = Pending{true, t.item & 1, (((size_t)t.b * p.Hq + hq) * p.q_len + tok) * p.max_chunks + t.c, m, l};
      ++n;
    }
    if (ok && pend.on && (ok = wait_warp(&S.o_full, (n - 1) & 1, ab))) {
      tc_fence_after();
      epilogue(pend);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// One warp per (sequence, query head, token): merge the chunks' O / l by their LSE.
// Lane c holds the log2-sum-exp and weight of chunk c; every lane
// accumulates four output columns over the chunks, DEC_MERGE chunks' loads in
// flight at a time (one round for the usual chunk counts).
constexpr int DEC_MERGE = 16;
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p, __nv_bfloat16* __restrict__ o,
                                                             float* __restrict__ lse) {
  constexpr int NV = D / 64;  // float2 pairs of output columns per lane (D / 32 columns)
  pdl_wait();  // the partial results come from the main kernel
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.B * p.Hq * p.q_len) return;
  const int b = gw / (p.Hq * p.q_len);
  const int n = p.seq_info[b].z;
  const float* lp = p.lse_part + (size_t)gw * p.max_chunks;
  const float2* op = reinterpret_cast<const float2*>(p.o_part + (size_t)gw * p.max_chunks * D) + lane * NV;
  // The first DEC_MERGE chunks' partial outputs load together with the first
  // 32 log2-sum-exps, before their maximum is known: one memory round trip
  // less on the usual chunk counts.
  float2 v[DEC_MERGE][NV];
#pragma unroll
  for (int u = 0; u < DEC_MERGE; ++u)
#pragma unroll
    for (int j = 0; j < NV; ++j) v[u][j] = u < n ? op[(size_t)u * (D / 2) + j] : make_float2(0.f, 0.f);
  const float l0 = lane < n ? lp[lane] : -INFINITY;
  float M = l0;
  for (int c = 32 + lane; c < n; c += 32) M = fmaxf(M, lp[c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float W = 0.f;
  float2 acc[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) acc[j] = make_float2(0.f, 0.f);
  if (M != -INFINITY) {
    for (int c0 = 0; c0 < n; c0 += DEC_MERGE) {
      const bool mine = lane < DEC_MERGE && c0 + lane < n;
      const float wl = mine ? exp2f((c0 == 0 ? l0 : lp[c0 + lane]) - M) : 0.f;
      W += wl;
      if (c0 > 0)
#pragma unroll
        for (int u = 0; u < DEC_MERGE; ++u)
#pragma unroll
          for (int j = 0; j < NV; ++j)
            v[u][j] = c0 + u < n ? op[(size_t)(c0 + u) * (D / 2) + j] : make_float2(0.f, 0.f);
#pragma unroll
      for (int u = 0; u < DEC_MERGE; ++u) {
        const float wc = __shfl_sync(0xffffffffu, wl, u);
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          acc[j].x += wc * v[u][j].x;
          acc[j].y += wc * v[u][j].y;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  }
  const float inv = W > 0.f ? 1.0f / W : 0.f;
  uint32_t* orow = reinterpret_cast<uint32_t*>(o + (size_t)gw * D) + lane * NV;
#pragma unroll
  for (int j = 0; j < NV; ++j) orow[j] = pack_bf16(acc[j].x * inv, acc[j].y * inv);
  if (lane == 0) lse[gw] = W > 0.f ? (M + log2f(W)) * LN2 : -INFINITY;
}

}  // namespace

// Launch with programmatic stream serialisation: the kernel may start while
// the previous one in the stream finishes (it calls pdl_wait() before reading
// that kernel's results).
template <typename... Args>
static cudaError_t launch_pdl(void (*kern)(Args...), unsigned grid, unsigned threads, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D>
static cudaError_t launch_decode_d(const DecodeLaunch& L, bool mods, cudaStream_t st) {
  const int R = L.p.G * L.p.q_len;
  const int qg = R <= 8 ? 1 : R <= 32 ? 4 : 16;
  auto kern = mods ? (qg == 1 ? decode_kernel<D, true, 1> : qg == 4 ? decode_kernel<D, true, 4> : decode_kernel<D, true, 16>)
                   : (qg == 1 ? decode_kernel<D, false, 1> : qg == 4 ? decode_kernel<D, false, 4> : decode_kernel<D, false, 16>);
  const int smem = qg == 1 ? DecCfg<D, 1>::SMEM : qg == 4 ? DecCfg<D, 4>::SMEM : DecCfg<D, 16>::SMEM;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess) return e;
  if ((e = launch_pdl(kern, (unsigned)L.grid, DEC_THREADS, (size_t)smem, st, L.tq, L.tk, L.tv, L.p)) != cudaSuccess)
    return e;
  const long long warps = (long long)L.p.B * L.p.Hq * L.p.q_len;
  return launch_pdl(decode_combine_kernel<D>, (unsigned)((warps + 7) / 8), 256u, 0, st, L.p, (__nv_bfloat16*)L.o,
                    L.lse);
}

cudaError_t launch_decode(const DecodeLaunch& L, bool mods, cudaStream_t st) {
  decode_setup_kernel<<<1, 1024, 0, st>>>(L.p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return L.p.d == 64 ? launch_decode_d<64>(L, mods, st) : launch_decode_d<128>(L, mods, st);
}

}  // namespace attn
