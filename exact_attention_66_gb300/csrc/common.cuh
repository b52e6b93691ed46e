// Shared kernel-side definitions: launch parameters, tile classification and
// the per-element mask/score-mod arithmetic used by every attention kernel.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include "ptx.cuh"

namespace attn {

constexpr int TILE = 128;  // rows of a Q tile and of a K/V tile
// Every TMEM-using kernel asks for at least this much shared memory so that a
// second CTA can never share its SM (each CTA allocates all 512 TMEM columns).
constexpr int MIN_SMEM_ONE_CTA = 120 * 1024;
constexpr int smem_one_cta(int bytes) { return bytes > MIN_SMEM_ONE_CTA ? bytes : MIN_SMEM_ONE_CTA; }
// Longest sequence the backward's per-CTA tile lists hold (1024 tiles of 128).
constexpr int BWD_MAX_N = 1024 * 128;

enum : uint32_t { MOD_CAUSAL = 1u, MOD_WINDOW = 2u, MOD_DOC = 4u, MOD_SOFTCAP = 8u, MOD_ALIBI = 16u };
enum : int { CLS_SKIP = 0, CLS_PARTIAL = 1, CLS_FULL = 2 };
// Test hooks (attn_test_hooks in include/attn.h): kernels of the selected kind
// make one consumer warpgroup wait first on an mbarrier that nothing
// completes, so that the wait runs into its time limit.
enum : int { STALL_FWD = 1, STALL_BWD = 2 };

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
// Lazy rescale: the running max used for the exponentials is only moved when
// a new row maximum exceeds it by more than this (log2 units, a factor 256).
// The result is exact either way once O is divided by l.
constexpr float RESCALE_THRESHOLD = 8.0f;

// Parameters common to the attention kernels (passed by value).
struct AttnParams {
  int B, Hq, Hkv, N;
  int nT;            // ceil(N / 128)
  int n_qblk;        // forward: ceil(N / 256) blocks of two Q tiles
  float scale;       // multiplier of q.k
  float scale_log2;  // scale * log2(e)
  uint32_t flags;    // MOD_*
  int window;
  float softcap;
  const int* doc_ids;   // [B, N] or nullptr
  // Document runs: [start, end) of the run of equal ids around each position
  // ([B, N], workspace), valid when *doc_unsorted == 0 (ids non-decreasing
  // along N: every document is then one run, and the document mask of a row
  // is an interval of columns).  Both nullptr without the document mod.
  const int2* doc_bounds;
  const int* doc_unsorted;
  const float* slopes;  // [Hq] or nullptr (default slopes)
  // Paged K/V (forward only): K and V live in blocks of 16 rows,
  // cache [kv_blocks, Hkv, 16, d]; row n of batch b is row n % 16 of block
  // block_table[b * bt_stride + n / 16].  nullptr: contiguous [B, Hkv, N, d].
  const int* block_table;
  int kv_blocks, bt_stride;
  const uint8_t* map;   // [B, nT, nT] tile classes, or nullptr (analytic)
  // With a map: [first, last + 1) of the non-skipped tiles of each Q tile
  // (row_range, over J) and of each KV tile (col_range, over I), [B, nT].
  const int2* row_range;
  const int2* col_range;
  int* status;          // device status word
  unsigned long long wait_ns;  // time limit of the test hooks' stalled wait (ns)
  int stall;                   // STALL_* test hook bits, 0 normally
};

// Non-skipped KV tiles of Q tile I (a superset without a map).
__device__ __forceinline__ int2 q_tile_range(const AttnParams& p, int b, int I) {
  if (p.row_range == nullptr || I >= p.nT) return make_int2(0, p.nT);
  return p.row_range[(size_t)b * p.nT + I];
}
// Non-skipped Q tiles of KV tile J (a superset without a map).
__device__ __forceinline__ int2 kv_tile_range(const AttnParams& p, int b, int J) {
  if (p.col_range == nullptr || J >= p.nT) return make_int2(0, p.nT);
  return p.col_range[(size_t)b * p.nT + J];
}

// Class of tile (I, J) for batch row b.  With no map the mask is causal or
// none, and the class follows in closed form; the ragged last column tile
// is always partial.
__device__ __forceinline__ int tile_class(const AttnParams& p, int b, int I, int J) {
  if (I >= p.nT || J >= p.nT) return CLS_SKIP;
  if (p.map != nullptr) return p.map[((size_t)b * p.nT + I) * p.nT + J];
  int c = CLS_FULL;
  if (p.flags & MOD_CAUSAL) c = (J < I) ? CLS_FULL : (J == I ? CLS_PARTIAL : CLS_SKIP);
  if (c == CLS_FULL && (J + 1) * TILE > p.N) c = CLS_PARTIAL;
  return c;
}

__device__ __forceinline__ float alibi_slope(const AttnParams& p, int hq) {
  return p.slopes != nullptr ? p.slopes[hq] : exp2f(-8.0f * (float)(hq + 1) / (float)p.Hq);
}

// tanh from the exponential: tanh(y) = sign(y) (1 - 2 / (e^{2|y|} + 1)).
// The absolute error is a few units of 1e-7 over the whole range (no
// cancellation problem for the absolute error, which is what enters the
// logits once multiplied by the cap).
__device__ __forceinline__ float tanh_exp(float y) {
  const float e = ex2(fabsf(y) * (2.0f * LOG2E));
  const float t = fmaf(-2.0f, rcp_approx(e + 1.0f), 1.0f);
  return copysignf(t, y);
}

// The same for a pair of lanes, its fp32 arithmetic two lanes per instruction
// (scalar fp32 on the softmax warps slows the tensor pipe; the two-wide form
// does not).
__device__ __forceinline__ uint64_t tanh2_exp(uint64_t y2) {
  float y0, y1;
  f2_unpack(y2, y0, y1);
  const uint32_t b0 = __float_as_uint(y0), b1 = __float_as_uint(y1);
  float z0, z1;
  f2_unpack(f2_mul(f2_pack(__uint_as_float(b0 & 0x7fffffffu), __uint_as_float(b1 & 0x7fffffffu)),
                   f2_pack(2.0f * LOG2E, 2.0f * LOG2E)), z0, z1);
  float u0, u1;
  f2_unpack(f2_add(f2_pack(ex2(z0), ex2(z1)), f2_pack(1.0f, 1.0f)), u0, u1);
  float t0, t1;
  f2_unpack(f2_fma(f2_pack(rcp_approx(u0), rcp_approx(u1)), f2_pack(-2.0f, -2.0f), f2_pack(1.0f, 1.0f)), t0, t1);
  return f2_pack(__uint_as_float(__float_as_uint(t0) | (b0 & 0x80000000u)),
                 __uint_as_float(__float_as_uint(t1) | (b1 & 0x80000000u)));
}

// Document run [start, end) of position `pos` when the ids are runs, else
// the whole sequence (the caller then tests ids element by element).
__device__ __forceinline__ int2 doc_run(const AttnParams& p, int b, int pos, bool& runs) {
  runs = p.doc_bounds != nullptr && *p.doc_unsorted == 0;
  if (!runs || pos >= p.N) return make_int2(0, p.N);
  return p.doc_bounds[(size_t)b * p.N + pos];
}

// Every lane of the warp waits; the warp proceeds only if all of them saw the
// phase complete (keeps the warp converged for the .sync.aligned tcgen05 ops).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const Abort& ab,
                                          unsigned long long limit = ATTN_WAIT_TIMEOUT_NS) {
  const bool ok = mbar_wait(bar, parity, ab, limit);
  return __all_sync(0xffffffffu, ok);
}

// Per-row constants of the score mods, in log2 units.
struct RowMods {
  float sc_in;     // softcap: s * sc_in = scale * s / c
  float sc_out;    // softcap: c * log2(e)
  float alibi_l2;  // slope * log2(e)
  int doc_i;       // doc id of the row
  int2 doc_run;    // its document's columns [start, end) when doc_runs
  bool doc_runs;
};

}  // namespace attn
