// FP8 prologue: signed Hadamard rotation of Q and K rows, per-(batch, head)
// amax, e4m3 quantisation of Q, K and V.
//
// FlashAttention-3 digest, "Basse précision FP8 et incoherent processing":
// queries and keys are multiplied by a random orthogonal matrix -- a Hadamard
// transform with random signs, applied per head in O(d log d) -- to spread
// outliers before FP8 quantisation; the transform is memory-bandwidth bound.
// Here each row x (d = 128) becomes (x * s) H / sqrt(128), H the natural-order
// Sylvester Hadamard matrix and s the +-1 vector of the row's KV head, so
// (q M)(k M)^T = q k^T exactly in real arithmetic; V is not rotated.
//
// Two bandwidth-bound passes over Q, K, V: pass 1 finds the amax of every
// (batch, head) of the rotated tensors (integer atomic max of the non-negative
// float bits, so the result does not depend on the order), pass 2 recomputes
// the rotation and writes e4m3 codes scaled by 448 / amax.  Rows reach
// shared memory in 64-row stages by bulk copy (one producer thread per CTA,
// a 6-slot ring); eight lanes per 128-element row, lane l8 holding elements
// 16 l8 .. 16 l8 + 15, so a compute warp takes four rows of a stage.  The
// butterflies of distance 1..8 stay in registers (two lanes of fp32 per
// instruction from distance 2 on), 16..64 go through three warp shuffles; the
// signs are applied to the bf16 bits while converting, and 1 / sqrt(128)
// is folded into the amax and the quantisation multiplier.
//
// Optionally RoPE is fused in front of the rotation (the digest's "fused with
// RoPE at no extra cost"): the row at position n of its head has its element
// pairs (c, c + 64) turned by n * base^(-2c/128) before the signs and the
// Hadamard butterflies, in the same registers -- lane l8 pairs with lane
// l8 ^ 4 -- so RoPE costs no extra pass over memory.
#include "common.cuh"
#include "launch.h"

namespace attn {

struct QuantTensors {
  const __nv_bfloat16* x[3];  // Q, K, V
  uint8_t* out[3];            // e4m3 codes
  long long rows[3];          // B * H * N
  int heads[3];               // scales of each tensor per batch entry (its H, or Hkv for dO)
  long long rps[3];           // rows per scale: N, or G * N for dO (one scale per query-head group)
  unsigned* amax[3];          // [B * H] float bits (workspace)
  float* scale[3];            // [B * H] dequantisation scales (output)
  const int8_t* signs;        // [Hkv, 128] or nullptr (no rotation)
  float rope_k;               // RoPE: inv_freq(c) = exp2(-c * rope_k), rope_k = 2 log2(base) / 128; 0 = off
  int N, Hkv, G;              // G = Hq / Hkv
  int* status;                // device status word (bounded waits report a timeout there)
};

constexpr int STAGE_ROWS = 256;                 // rows per shared-memory stage
constexpr int STAGE_BYTES = STAGE_ROWS * 256;    // 64 KB of bf16 rows (d = 128)
constexpr int QSTAGES = 3;                       // ring slots per CTA
constexpr int QWARPS = 16;                       // compute warps
constexpr int WROWS = STAGE_ROWS / QWARPS;       // rows of a stage per compute warp (16)
constexpr int SLABS = WROWS / 4;                 // four rows per warp instruction
constexpr int QTHREADS = (QWARPS + 1) * 32;      // plus one producer warp
constexpr float HAD_NORM = 0.08838834764831845f;  // 1 / sqrt(128)

// Untiled bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global to shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// This lane's 16 bf16 elements of a row.
struct Raw16 {
  uint4 a, b;
};
__device__ __forceinline__ Raw16 load16(const QuantTensors& t, int ti, long long row, int l8) {
  const uint4* p = reinterpret_cast<const uint4*>(t.x[ti] + row * 128 + 16 * l8);
  return Raw16{__ldg(p), __ldg(p + 1)};
}

// KV head whose signs rotate rows of head plane n (= b * H + h) of tensor ti.
__device__ __forceinline__ int sign_head(const QuantTensors& t, int ti, long long n) {
  const int head = (int)(n % t.heads[ti]);
  return ti == 0 ? head / t.G : head;
}

// This lane's 16 values of the row: RoPE (when on), then the signed
// Walsh-Hadamard transform without its 1 / sqrt(128) (Q and K with signs), or
// the plain values.  Every lane of the warp must call it (warp shuffles).
// hk: the row's sign head (sign_head), pos: its position in its sequence.
template <bool ROPE>
__device__ __forceinline__ void transform16(const QuantTensors& t, int ti, int hk, int pos, int l8, const Raw16& raw,
                                            const float (&inv_freq)[16], float (&v)[16]) {
  const uint32_t w[8] = {raw.a.x, raw.a.y, raw.a.z, raw.a.w, raw.b.x, raw.b.y, raw.b.z, raw.b.w};
  if (ti == 2 || (!ROPE && t.signs == nullptr)) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = bf16lo_f32(w[k]);
      v[2 * k + 1] = bf16hi_f32(w[k]);
    }
    return;
  }
  uint32_t sgn[4] = {0u, 0u, 0u, 0u};  // sign bytes of elements 4 j .. 4 j + 3
  if (t.signs != nullptr) {
    const uint4 sg = __ldg(reinterpret_cast<const uint4*>(t.signs + hk * 128 + 16 * l8));
    sgn[0] = sg.x;
    sgn[1] = sg.y;
    sgn[2] = sg.z;
    sgn[3] = sg.w;
  }
  if (ROPE) {  // RoPE first (before the signs), rotate-half pairs (c, c + 64)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[2 * k] = bf16lo_f32(w[k]);
      v[2 * k + 1] = bf16hi_f32(w[k]);
    }
    const float fpos = (float)pos;
    const bool first = l8 < 4;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float partner = __shfl_xor_sync(0xffffffffu, v[e], 4);
      // Angle reduced to [-pi, pi] by Cody and Waite's two-constant method:
      // 2 pi = C1 - C2 with C1 = fl(2 pi) and C2 = 1.7484556e-7 its excess;
      // both steps are fused multiply-adds, so k C1 enters exactly.  Then the
      // fast sine / cosine, accurate to a few 1e-7 on that interval.
      const float ang = fpos * inv_freq[e];
      const float kf = rintf(ang * 0.15915494309189535f);  // 1 / (2 pi)
      const float red = fmaf(kf, 1.7484556e-07f, fmaf(-kf, 6.28318548f, ang));
      float sn, cs;
      __sincosf(red, &sn, &cs);
      v[e] = first ? fmaf(v[e], cs, -partner * sn) : fmaf(v[e], cs, partner * sn);
    }
    if (t.signs == nullptr) return;
#pragma unroll
    for (int e = 0; e < 16; ++e)
      v[e] = __uint_as_float(__float_as_uint(v[e]) ^ (((sgn[e >> 2] >> (8 * (e & 3) + 7)) & 1u) << 31));
  } else {  // signs applied to the bf16 bits while converting
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t sb = sgn[k >> 1] >> (16 * (k & 1));  // sign bytes of elements 2 k, 2 k + 1
      v[2 * k] = __uint_as_float((w[k] << 16) ^ ((sb & 0x80u) << 24));
      v[2 * k + 1] = __uint_as_float((w[k] & 0xFFFF0000u) ^ ((sb & 0x8000u) << 16));
    }
  }
  // Butterflies (a, b) -> (a + b, a - b) on index pairs (j, j ^ h).  h = 1: scalar.
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float a0 = v[2 * k], b0 = v[2 * k + 1];
    v[2 * k] = a0 + b0;
    v[2 * k + 1] = a0 - b0;
  }
  uint64_t P[8];  // pairs (v[2 k], v[2 k + 1])
#pragma unroll
  for (int k = 0; k < 8; ++k) P[k] = f2_pack(v[2 * k], v[2 * k + 1]);
  const uint64_t m1 = f2_pack(-1.f, -1.f);
#pragma unroll
  for (int hb = 1; hb < 8; hb <<= 1) {  // h = 2, 4, 8: pair index bit hb
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k & hb) continue;
      const uint64_t a2 = P[k], b2 = P[k | hb];
      P[k] = f2_add(a2, b2);
      P[k | hb] = f2_fma(b2, m1, a2);
    }
  }
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {  // h = 16, 32, 64: lane bit m of l8
    const float sgn_self = (l8 & m) ? -1.f : 1.f;
    const uint64_t s2 = f2_pack(sgn_self, sgn_self);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float x0, x1;
      f2_unpack(P[k], x0, x1);
      const float o0 = __shfl_xor_sync(0xffffffffu, x0, m), o1 = __shfl_xor_sync(0xffffffffu, x1, m);
      P[k] = f2_fma(P[k], s2, f2_pack(o0, o1));  // lower index: a + b; upper: a' - b'
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) f2_unpack(P[k], v[2 * k], v[2 * k + 1]);
}

// RoPE inverse frequencies of this lane's 16 elements (c mod 64 = 16 (l8 & 3) + e).
__device__ __forceinline__ void rope_freqs(const QuantTensors& t, int l8, float (&f)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) f[e] = t.rope_k != 0.f ? exp2f(-(float)(16 * (l8 & 3) + e) * t.rope_k) : 0.f;
}

// Scale of the values transform16 returns for tensor ti (1 / sqrt(128) when rotated).
__device__ __forceinline__ float out_norm(const QuantTensors& t, int ti) {
  return (ti != 2 && t.signs != nullptr) ? HAD_NORM : 1.0f;
}

// Work: stages of 256 consecutive rows (64 KB) of Q, then K, then V.  One
// producer thread per CTA streams a CTA's stages (stage g = blockIdx.x +
// k * gridDim.x) into a ring of shared-memory slots with bulk copies, with the
// stage's indices (tensor, first row, scale and head of its rows) in a record
// beside each slot; sixteen compute warps take 16 rows each per stage, copy
// them to registers and hand the slot back before transforming them.  With
// the rows staged through registers instead (one 16-row group in flight per
// warp), too few bytes were in flight to keep HBM busy: a third of its
// bandwidth at 59 % issue.
struct Group {
  int ti;
  long long r0, r1;
};
__device__ __forceinline__ bool stage_of(const QuantTensors& t, long long g, Group& gr) {
#pragma unroll
  for (int ti = 0; ti < 3; ++ti) {
    const long long n = (t.rows[ti] + STAGE_ROWS - 1) / STAGE_ROWS;
    if (g < n) {
      gr.ti = ti;
      gr.r0 = g * STAGE_ROWS;
      gr.r1 = min(gr.r0 + STAGE_ROWS, t.rows[ti]);
      return true;
    }
    g -= n;
  }
  return false;
}

// A stage's indices, computed once by the producer (64-bit divisions per row
// cost more instructions than the transform).
struct StageInfo {
  long long r0, r1;  // rows [r0, r1) of tensor ti
  long long h0, n0;  // scale index and head plane of row r0
  int ti;
  int one_head;      // every row has scale h0
  int one_n;         // every row is in head plane n0
  int hk0;           // sign head of plane n0
};

struct QuantBars {
  uint64_t full[QSTAGES], empty[QSTAGES];
  StageInfo info[QSTAGES];
  int abort;
  int done[QSTAGES];  // the producer found no further stage
};
constexpr int QSMEM = QSTAGES * STAGE_BYTES + (int)sizeof(QuantBars) + 128;

// Pass 1 (WRITE false): amax of every (batch, head).  Pass 2 (WRITE true):
// e4m3 codes scaled by 448 / amax.  ROPE: rotary embedding in front (its 16
// inverse frequencies per lane are only kept in registers when it is on).
template <bool WRITE, bool ROPE>
__global__ void __launch_bounds__(QTHREADS, 1) quant_pass_kernel(const QuantTensors t) {
  extern __shared__ uint8_t qsm_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)qsm_raw + 127) & ~(uintptr_t)127);
  QuantBars& S = *reinterpret_cast<QuantBars*>(sm + QSTAGES * STAGE_BYTES);
  const Abort ab{&S.abort, t.status};
  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    S.abort = 0;
    for (int s = 0; s < QSTAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], QWARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == QWARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      long long k = 0;
      bool ok = true;
      for (long long g = blockIdx.x;; g += gridDim.x, ++k) {
        const int s = (int)(k % QSTAGES);
        if (!(ok = mbar_wait(&S.empty[s], (uint32_t)((k / QSTAGES) & 1) ^ 1u, ab))) break;
        Group gr;
        StageInfo& in = S.info[s];
        if (!stage_of(t, g, gr)) {  // tell the compute warps, with no copy
          S.done[s] = 1;
          mbar_arrive(&S.full[s]);
          break;
        }
        const long long rps = t.rps[gr.ti];
        in.r0 = gr.r0;
        in.r1 = gr.r1;
        in.ti = gr.ti;
        in.h0 = gr.r0 / rps;
        in.one_head = gr.r1 - 1 < (in.h0 + 1) * rps;
        in.n0 = gr.r0 / t.N;
        in.one_n = gr.r1 - 1 < (in.n0 + 1) * t.N;
        in.hk0 = t.signs != nullptr ? sign_head(t, gr.ti, in.n0) : 0;
        S.done[s] = 0;
        const uint32_t bytes = (uint32_t)(gr.r1 - gr.r0) * 256u;
        mbar_arrive_tx(&S.full[s], bytes);
        bulk_load(sm + s * STAGE_BYTES, t.x[gr.ti] + gr.r0 * 128, bytes, &S.full[s]);
      }
      // Copies still in flight (the compute warps stopped early) must land
      // before the CTA exits: the last phase armed in each slot completes
      // ((phases armed in it - 1) & 1).
      const long long armed = ok ? k + 1 : k;
      for (int s = 0; s < QSTAGES; ++s)
        if (armed > s) mbar_wait_drain(&S.full[s], (uint32_t)(((armed - 1 - s) / QSTAGES) & 1));
    }
    return;
  }
  // -------------------------------------------------------- compute warps
  const int l8 = lane & 7, qr = lane >> 3;
  float inv_freq[16];
  if (ROPE) rope_freqs(t, l8, inv_freq);
  for (long long k = 0;; ++k) {
    const int s = (int)(k % QSTAGES);
    if (!wait_warp(&S.full[s], (uint32_t)((k / QSTAGES) & 1), ab)) break;
    if (S.done[s]) break;
    const StageInfo in = S.info[s];
    Raw16 raw[SLABS];
#pragma unroll
    for (int sl = 0; sl < SLABS; ++sl) {
      const int lr = WROWS * warp + 4 * sl + qr;
      if (in.r0 + lr < in.r1) {
        const uint4* src = reinterpret_cast<const uint4*>(sm + s * STAGE_BYTES + lr * 256 + l8 * 32);
        raw[sl] = Raw16{src[0], src[1]};
      } else {
        raw[sl] = Raw16{make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);

    const int ti = in.ti;
    const float norm = out_norm(t, ti);
    const long long rps = t.rps[ti];
    float mx = 0.f;
#pragma unroll
    for (int sl = 0; sl < SLABS; ++sl) {
      const long long row_raw = in.r0 + WROWS * warp + 4 * sl + qr;
      const long long row = min(row_raw, in.r1 - 1);
      const long long n = in.one_n ? in.n0 : row / t.N;
      const int hk = t.signs == nullptr ? 0 : in.one_n ? in.hk0 : sign_head(t, ti, n);
      float v[16];
      transform16<ROPE>(t, ti, hk, (int)(row - n * t.N), l8, raw[sl], inv_freq, v);
      if (WRITE) {
        if (row_raw >= in.r1) continue;
        const float a = __uint_as_float(t.amax[ti][in.one_head ? in.h0 : row / rps]);
        const float mul = a > 0.f ? (448.0f / a) * norm : 1.0f;
        uint4 codes;
        codes.x = pack_e4m3x4(v[0] * mul, v[1] * mul, v[2] * mul, v[3] * mul);
        codes.y = pack_e4m3x4(v[4] * mul, v[5] * mul, v[6] * mul, v[7] * mul);
        codes.z = pack_e4m3x4(v[8] * mul, v[9] * mul, v[10] * mul, v[11] * mul);
        codes.w = pack_e4m3x4(v[12] * mul, v[13] * mul, v[14] * mul, v[15] * mul);
        reinterpret_cast<uint4*>(t.out[ti] + row * 128)[l8] = codes;
      } else {
        float rm = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) rm = fmaxf(rm, fabsf(v[e]));
        if (row_raw >= in.r1) rm = 0.f;
        if (in.one_head) {
          mx = fmaxf(mx, rm);
        } else {  // rows of two heads in this stage (short sequences): one atomic per row
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) rm = fmaxf(rm, __shfl_xor_sync(0xffffffffu, rm, o));
          if (l8 == 0 && row_raw < in.r1) atomicMax(t.amax[ti] + row / rps, __float_as_uint(rm * norm));
        }
      }
    }
    if (!WRITE && in.one_head) {
      mx = warp_max(mx);
      if (lane == 0) atomicMax(t.amax[ti] + in.h0, __float_as_uint(mx * norm));
    }
  }
}

// Whole rows per thread (every prologue without RoPE).  A stage of 256 rows
// reaches shared memory as two tensor copies (columns 0-63 and 64-127) with
// the 128-byte swizzle: 16-byte chunk c of row r sits in slot c ^ (r % 8) of
// the row's 128 bytes, so a thread reading its own row chunk by chunk meets
// eight different bank groups across any eight consecutive rows.  Each of
// eight compute warps takes 32 rows of a stage, one per thread, and runs all
// seven butterfly stages in registers with no shuffle: distance 1 in scalar
// fp32 on the two halves of a bf16 pair word, distances 2..64 two lanes per
// instruction.  The butterflies, their order and the sign and scale steps are
// those of the lane-split form above, so both give the same bits.  Codes
// leave through a per-warp transposition in shared memory (row r, chunk c in
// slot c ^ (r % 8) again), so each store instruction writes four whole rows.
constexpr int RWARPS = 8;                          // compute warps (two warpgroups)
constexpr int RTHREADS = (RWARPS + 4) * 32;        // plus a producer warpgroup (one thread works)
// Register split: launched at 168 a thread (ptxas' bound for 384 threads), the
// producer warpgroup gives registers back so a compute thread can hold its
// 128 rotated values, the sign words and the code words without spilling.
constexpr int R_LAUNCH = 168, R_LOW = 56, R_HIGH = 224;
static_assert(128 * R_LOW + 256 * R_HIGH <= RTHREADS * R_LAUNCH, "register split over the launch's allocation");
constexpr int XPOSE_BYTES = RWARPS * 32 * 128;     // one 32-row block of codes per compute warp
constexpr int RSMEM = QSTAGES * STAGE_BYTES + XPOSE_BYTES + (int)sizeof(QuantBars) + 1024;
static_assert(RWARPS * 32 == STAGE_ROWS, "one row of a stage per compute thread");

struct QuantMaps {
  CUtensorMap m[3];  // [rows, 128] bf16 of each tensor, 64 x 256 boxes, 128-byte swizzle
};

// XOR masks that negate halves of bf16 pair words: bit 15 (low half) and bit
// 31 (high half) from the sign bits of int8 signs.  sw holds the signs of four
// consecutive elements 4 j .. 4 j + 3; lo: the word of elements 4 j, 4 j + 1,
// hi: the word of 4 j + 2, 4 j + 3.
__device__ __forceinline__ uint32_t sign_mask_lo(uint32_t sw) { return __byte_perm(sw, 0u, 0x1404) & 0x80008000u; }
__device__ __forceinline__ uint32_t sign_mask_hi(uint32_t sw) { return __byte_perm(sw, 0u, 0x3424) & 0x80008000u; }

template <bool WRITE>
__global__ void __launch_bounds__(RTHREADS, 1) quant_rows_kernel(const QuantTensors t,
                                                                 const __grid_constant__ QuantMaps maps) {
  extern __shared__ uint8_t qsm_raw[];
  // The 128-byte swizzle repeats every 1024 bytes: slots start on that boundary.
  uint8_t* sm = (uint8_t*)(((uintptr_t)qsm_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* xpose = sm + QSTAGES * STAGE_BYTES;
  QuantBars& S = *reinterpret_cast<QuantBars*>(xpose + XPOSE_BYTES);
  const Abort ab{&S.abort, t.status};
  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    S.abort = 0;
    for (int s = 0; s < QSTAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], RWARPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp >= RWARPS) {
    // ------------------------------------------------------------ producer
    regs_dec<R_LOW>();
    if (warp == RWARPS && lane == 0) {
      for (int i = 0; i < 3; ++i)
        if (t.rows[i] > 0) tma_prefetch_desc(&maps.m[i]);
      long long k = 0;
      bool ok = true;
      for (long long g = blockIdx.x;; g += gridDim.x, ++k) {
        const int s = (int)(k % QSTAGES);
        if (!(ok = mbar_wait(&S.empty[s], (uint32_t)((k / QSTAGES) & 1) ^ 1u, ab))) break;
        Group gr;
        StageInfo& in = S.info[s];
        if (!stage_of(t, g, gr)) {
          S.done[s] = 1;
          mbar_arrive(&S.full[s]);
          break;
        }
        const long long rps = t.rps[gr.ti];
        in.r0 = gr.r0;
        in.r1 = gr.r1;
        in.ti = gr.ti;
        in.h0 = gr.r0 / rps;
        in.one_head = gr.r1 - 1 < (in.h0 + 1) * rps;
        in.n0 = gr.r0 / t.N;
        in.one_n = gr.r1 - 1 < (in.n0 + 1) * t.N;
        in.hk0 = t.signs != nullptr ? sign_head(t, gr.ti, in.n0) : 0;
        S.done[s] = 0;
        // Both boxes count in full: rows past the tensor's end arrive as zeros.
        mbar_arrive_tx(&S.full[s], STAGE_BYTES);
        tma_load_2d(sm + s * STAGE_BYTES, &maps.m[gr.ti], &S.full[s], 0, (int)gr.r0);
        tma_load_2d(sm + s * STAGE_BYTES + STAGE_BYTES / 2, &maps.m[gr.ti], &S.full[s], 64, (int)gr.r0);
      }
      const long long armed = ok ? k + 1 : k;
      for (int s = 0; s < QSTAGES; ++s)
        if (armed > s) mbar_wait_drain(&S.full[s], (uint32_t)(((armed - 1 - s) / QSTAGES) & 1));
    }
    return;
  }
  // -------------------------------------------------------- compute warps
  regs_inc<R_HIGH>();
  const int lr = warp * 32 + lane;  // this thread's row of every stage
  uint8_t* xw = xpose + warp * (32 * 128);
  const uint64_t m1 = f2_pack(-1.f, -1.f);
  for (long long k = 0;; ++k) {
    const int s = (int)(k % QSTAGES);
    if (!wait_warp(&S.full[s], (uint32_t)((k / QSTAGES) & 1), ab)) break;
    if (S.done[s]) break;
    const StageInfo in = S.info[s];
    uint32_t w[64];  // bf16 pair words: w[j] = elements 2 j, 2 j + 1
    {
      const uint8_t* src = sm + s * STAGE_BYTES + lr * 128;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 q = *reinterpret_cast<const uint4*>(src + (c >> 3) * (STAGE_BYTES / 2) +
                                                         (((c & 7) ^ (lr & 7)) << 4));
        w[4 * c] = q.x;
        w[4 * c + 1] = q.y;
        w[4 * c + 2] = q.z;
        w[4 * c + 3] = q.w;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);

    const int ti = in.ti;
    const long long row = in.r0 + lr;
    const bool valid = row < in.r1;
    const long long rowc = valid ? row : in.r1 - 1;
    const float norm = out_norm(t, ti);
    uint64_t P[64];  // P[j] = (y[2 j], y[2 j + 1])
    if (ti != 2 && t.signs != nullptr) {
      const int hk = in.one_n ? in.hk0 : sign_head(t, ti, rowc / t.N);
      const uint4* sg = reinterpret_cast<const uint4*>(t.signs + hk * 128);
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // elements 16 i .. 16 i + 15
        const uint4 q = __ldg(sg + i);
        const uint32_t sw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int wi = 8 * i + 2 * j + e;
            const uint32_t x = w[wi] ^ (e == 0 ? sign_mask_lo(sw[j]) : sign_mask_hi(sw[j]));
            const float a = bf16lo_f32(x), b = bf16hi_f32(x);
            P[wi] = f2_pack(a + b, a - b);  // distance 1
          }
        }
      }
#pragma unroll
      for (int hb = 1; hb < 64; hb <<= 1) {  // distances 2 .. 64: pair index bit hb
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          if (j & hb) continue;
          const uint64_t a2 = P[j], b2 = P[j | hb];
          P[j] = f2_add(a2, b2);
          P[j | hb] = f2_fma(b2, m1, a2);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) P[j] = f2_pack(bf16lo_f32(w[j]), bf16hi_f32(w[j]));
    }

    if (!WRITE) {
      float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        float y0, y1;
        f2_unpack(P[j], y0, y1);
        r4[j & 3] = max3(r4[j & 3], fabsf(y0), fabsf(y1));
      }
      float rm = valid ? fmaxf(fmaxf(r4[0], r4[1]), fmaxf(r4[2], r4[3])) : 0.f;
      if (in.one_head) {
        rm = warp_max(rm);
        if (lane == 0) atomicMax(t.amax[ti] + in.h0, __float_as_uint(rm * norm));
      } else if (valid) {  // rows of two scales in this stage (short sequences): one atomic per row
        atomicMax(t.amax[ti] + row / t.rps[ti], __float_as_uint(rm * norm));
      }
    } else {
      const float a = __uint_as_float(t.amax[ti][in.one_head ? in.h0 : rowc / t.rps[ti]]);
      const float mul = a > 0.f ? (448.0f / a) * norm : 1.0f;
      const uint64_t mul2 = f2_pack(mul, mul);
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // code bytes 16 c .. 16 c + 15 of the row
        uint32_t cw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float y0, y1, y2, y3;
          f2_unpack(f2_mul(P[8 * c + 2 * j], mul2), y0, y1);
          f2_unpack(f2_mul(P[8 * c + 2 * j + 1], mul2), y2, y3);
          cw[j] = pack_e4m3x4(y0, y1, y2, y3);
        }
        *reinterpret_cast<uint4*>(xw + lane * 128 + ((c ^ (lane & 7)) << 4)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // rows 4 i .. 4 i + 3 of the warp's block, eight lanes a row
        const int rr = 4 * i + (lane >> 3), ch = lane & 7;
        const uint4 val = *reinterpret_cast<const uint4*>(xw + rr * 128 + ((ch ^ (rr & 7)) << 4));
        const long long grow = in.r0 + warp * 32 + rr;
        if (grow < in.r1) reinterpret_cast<uint4*>(t.out[ti] + grow * 128)[ch] = val;
      }
      __syncwarp();
    }
  }
}

__global__ void quant_scale_kernel(const QuantTensors t, int B) {
  const int ti = blockIdx.y;
  const int n = B * t.heads[ti];
  for (int i = threadIdx.x + blockIdx.x * blockDim.x; i < n; i += blockDim.x * gridDim.x) {
    const float a = __uint_as_float(t.amax[ti][i]);
    t.scale[ti][i] = a > 0.f ? a / 448.0f : 1.0f;
  }
}

static cudaError_t run_quant(const QuantTensors& t, int B, unsigned* amax_ws, size_t n_amax, cudaStream_t st);

cudaError_t launch_hadamard_quant(const void* q, const void* k, const void* v, void* q8, void* k8,
                                  void* v8, float* scales, const int8_t* signs, int B, int Hq,
                                  int Hkv, int N, float rope_base, unsigned* amax_ws, int* status,
                                  cudaStream_t st) {
  QuantTensors t{};
  t.status = status;
  t.rope_k = rope_base > 0.f ? 2.0f * log2f(rope_base) / 128.0f : 0.f;
  t.x[0] = (const __nv_bfloat16*)q;
  t.x[1] = (const __nv_bfloat16*)k;
  t.x[2] = (const __nv_bfloat16*)v;
  t.out[0] = (uint8_t*)q8;
  t.out[1] = (uint8_t*)k8;
  t.out[2] = (uint8_t*)v8;
  t.heads[0] = Hq;
  t.heads[1] = t.heads[2] = Hkv;
  for (int i = 0; i < 3; ++i) {
    t.rows[i] = (long long)B * t.heads[i] * N;
    t.rps[i] = N;
  }
  t.amax[0] = amax_ws;
  t.amax[1] = amax_ws + B * Hq;
  t.amax[2] = amax_ws + B * Hq + B * Hkv;
  t.scale[0] = scales;
  t.scale[1] = scales + B * Hq;
  t.scale[2] = scales + B * Hq + B * Hkv;
  t.signs = signs;
  t.N = N;
  t.Hkv = Hkv;
  t.G = Hq / Hkv;
  return run_quant(t, B, amax_ws, (size_t)(B * Hq + 2 * B * Hkv), st);
}

// The three passes of a quantisation: amax, scales, codes.
static cudaError_t run_quant(const QuantTensors& t, int B, unsigned* amax_ws, size_t n_amax, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(amax_ws, 0, sizeof(unsigned) * n_amax, st);
  if (e != cudaSuccess) return e;
  long long stages = 0;
  for (int i = 0; i < 3; ++i) stages += (t.rows[i] + STAGE_ROWS - 1) / STAGE_ROWS;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // One CTA per SM, each walking many stages.
  const long long blocks = min(stages, (long long)sms);
  if (t.rope_k != 0.f) {  // RoPE: lane-split rows
    auto p1 = quant_pass_kernel<false, true>;
    auto p2 = quant_pass_kernel<true, true>;
    if ((e = cudaFuncSetAttribute(p1, cudaFuncAttributeMaxDynamicSharedMemorySize, QSMEM)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(p2, cudaFuncAttributeMaxDynamicSharedMemorySize, QSMEM)) != cudaSuccess) return e;
    if (blocks == 0) return cudaSuccess;
    p1<<<(unsigned)blocks, QTHREADS, QSMEM, st>>>(t);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    quant_scale_kernel<<<dim3(1, 3), 256, 0, st>>>(t, B);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    p2<<<(unsigned)blocks, QTHREADS, QSMEM, st>>>(t);
    return cudaGetLastError();
  }
  QuantMaps maps{};
  for (int i = 0; i < 3; ++i)
    if (t.rows[i] > 0 && !make_rows_map(&maps.m[i], t.x[i], t.rows[i], STAGE_ROWS)) return cudaErrorInvalidValue;
  auto p1 = quant_rows_kernel<false>;
  auto p2 = quant_rows_kernel<true>;
  // The register split inside the kernels assumes R_LAUNCH registers a thread
  // at launch: with fewer, the compute warps' increase could never be granted.
  static int regs[2] = {-1, -1};
  for (int w = 0; w < 2; ++w) {
    if (regs[w] < 0) {
      cudaFuncAttributes fa;
      if ((e = cudaFuncGetAttributes(&fa, w ? p2 : p1)) != cudaSuccess) return e;
      regs[w] = fa.numRegs;
    }
    if (regs[w] != R_LAUNCH) return cudaErrorInvalidConfiguration;
  }
  if ((e = cudaFuncSetAttribute(p1, cudaFuncAttributeMaxDynamicSharedMemorySize, RSMEM)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(p2, cudaFuncAttributeMaxDynamicSharedMemorySize, RSMEM)) != cudaSuccess) return e;
  if (blocks == 0) return cudaSuccess;
  p1<<<(unsigned)blocks, RTHREADS, RSMEM, st>>>(t, maps);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  quant_scale_kernel<<<dim3(1, 3), 256, 0, st>>>(t, B);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  p2<<<(unsigned)blocks, RTHREADS, RSMEM, st>>>(t, maps);
  return cudaGetLastError();
}

// Operands of the mixed e4m3 backward: dO with one scale per (batch, KV head)
// -- the query heads of a group are consecutive in [B, Hq, N, d], so a
// group's rows are one run of G * N rows -- and V per (batch, KV head).  No
// rotation (the dV GEMM contracts over rows, not over the rotated columns).
// scales: [B * Hkv] of dO, then [B * Hkv] of V.
cudaError_t launch_quant_bwd_fp8(const void* dout, const void* v, void* do8, void* v8, float* scales, int B,
                                 int Hq, int Hkv, int N, unsigned* amax_ws, int* status, cudaStream_t st) {
  QuantTensors t{};
  t.status = status;
  t.x[0] = (const __nv_bfloat16*)dout;
  t.x[2] = (const __nv_bfloat16*)v;
  t.out[0] = (uint8_t*)do8;
  t.out[2] = (uint8_t*)v8;
  t.heads[0] = t.heads[2] = Hkv;
  t.rows[0] = (long long)B * Hq * N;
  t.rows[2] = (long long)B * Hkv * N;
  t.rps[0] = (long long)(Hq / Hkv) * N;
  t.rps[1] = t.rps[2] = N;
  t.amax[0] = amax_ws;
  t.amax[1] = amax_ws + B * Hkv;
  t.amax[2] = amax_ws + B * Hkv;
  t.scale[0] = scales;
  t.scale[1] = scales + B * Hkv;
  t.scale[2] = scales + B * Hkv;
  t.N = N;
  t.Hkv = Hkv;
  t.G = Hq / Hkv;
  return run_quant(t, B, amax_ws, (size_t)(2 * B * Hkv), st);
}

}  // namespace attn
