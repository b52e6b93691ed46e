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
  const float* slopes;  // [Hq] or nullptr (default slopes)
  const uint8_t* map;   // [B, nT, nT] tile classes, or nullptr (analytic)
  int* status;          // device status word
};

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

// Every lane of the warp waits; the warp proceeds only if all of them saw the
// phase complete (keeps the warp converged for the .sync.aligned tcgen05 ops).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const Abort& ab) {
  const bool ok = mbar_wait(bar, parity, ab);
  return __all_sync(0xffffffffu, ok);
}

// Per-row constants of the score mods, in log2 units.
struct RowMods {
  float sc_in;     // softcap: s * sc_in = scale * s / c
  float sc_out;    // softcap: c * log2(e)
  float alibi_l2;  // slope * log2(e)
  int doc_i;       // doc id of the row
};

}  // namespace attn
