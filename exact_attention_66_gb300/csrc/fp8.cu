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
// the rotation and writes e4m3 codes scaled by 448 / amax.  Each compute
// thread holds one whole 128-element row and runs the seven butterfly stages
// in registers with no shuffle: distance 1 in scalar fp32 on the two halves
// of a bf16 pair word, distances 2..64 two lanes per instruction.  The signs
// are applied to the bf16 bits while converting, and 1 / sqrt(128) is folded
// into the amax and the quantisation multiplier.
//
// Optionally RoPE is fused in front of the rotation (the digest notes that the
// rotation can ride along with RoPE for free): the row at position n of its head has its element
// pairs (c, c + 64) turned by n * base^(-2c/128) before the signs and the
// Hadamard butterflies, in the same registers, so RoPE costs no extra pass
// over memory.
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

constexpr int STAGE_ROWS = 256;                   // rows per shared-memory stage
constexpr int STAGE_BYTES = STAGE_ROWS * 256;      // 64 KB of bf16 rows (d = 128)
constexpr int QSTAGES = 3;                         // ring slots per CTA
constexpr int RWARPS = 8;                          // compute warps (two warpgroups)
constexpr int RTHREADS = (RWARPS + 4) * 32;        // plus a producer warpgroup (one thread works)
constexpr int XPOSE_BYTES = RWARPS * 32 * 128;     // one 32-row block of codes per compute warp
constexpr float HAD_NORM = 0.08838834764831845f;   // 1 / sqrt(128)
static_assert(RWARPS * 32 == STAGE_ROWS, "one row of a stage per compute thread");
// Register split: launched at 168 a thread (ptxas' bound for 384 threads), the
// producer warpgroup gives registers back so a compute thread can hold its
// 128 rotated values, the sign words and the code words without spilling.
constexpr int R_LAUNCH = 168, R_LOW = 56, R_HIGH = 224;
static_assert(128 * R_LOW + 256 * R_HIGH <= RTHREADS * R_LAUNCH, "register split over the launch's allocation");

// 2-D tile load (coordinates innermost first) completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// KV head whose signs rotate rows of head plane n (= b * H + h) of tensor ti.
__device__ __forceinline__ int sign_head(const QuantTensors& t, int ti, long long n) {
  const int head = (int)(n % t.heads[ti]);
  return ti == 0 ? head / t.G : head;
}

// Scale of the transformed values of tensor ti (1 / sqrt(128) when rotated).
__device__ __forceinline__ float out_norm(const QuantTensors& t, int ti) {
  return (ti != 2 && t.signs != nullptr) ? HAD_NORM : 1.0f;
}

// Work: stages of 256 consecutive rows (64 KB) of Q, K and V, interleaved
// round by round (stage r of Q, of K, of V, then stage r + 1 ...) while the
// tensors have stages left, so that the rotated rows (bound by their
// instructions) and the plain V rows (bound by memory) are in flight at the
// same time.  One producer thread per CTA streams a CTA's stages (stage g =
// blockIdx.x + k * gridDim.x) into a ring of shared-memory slots, with the
// stage's indices (tensor, first row, scale and head of its rows) in a record
// beside each slot; the compute warps copy their rows to registers and hand
// the slot back before transforming them.
struct Group {
  int ti;
  long long r0, r1;
};
__device__ __forceinline__ bool stage_of(const QuantTensors& t, long long g, Group& gr) {
  long long n[3];
#pragma unroll
  for (int ti = 0; ti < 3; ++ti) n[ti] = (t.rows[ti] + STAGE_ROWS - 1) / STAGE_ROWS;
  // Rounds [prev, next) have cnt tensors with stages left; at most three phases.
  long long prev = 0;
#pragma unroll 1
  for (int ph = 0; ph < 3; ++ph) {
    long long next = 0x7fffffffffffffffll;
    int cnt = 0;
#pragma unroll
    for (int ti = 0; ti < 3; ++ti)
      if (n[ti] > prev) {
        ++cnt;
        next = min(next, n[ti]);
      }
    if (cnt == 0) return false;
    const long long span = (next - prev) * cnt;
    if (g < span) {
      const long long round = prev + g / cnt;
      int k = (int)(g % cnt);
#pragma unroll
      for (int ti = 0; ti < 3; ++ti)
        if (n[ti] > prev && k-- == 0) {
          gr.ti = ti;
          gr.r0 = round * STAGE_ROWS;
          gr.r1 = min(gr.r0 + STAGE_ROWS, t.rows[ti]);
          return true;
        }
      return false;
    }
    g -= span;
    prev = next;
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
  float rope_f[64];   // RoPE inverse frequencies base^(-2c/128), c = 0..63
  int abort;
  int done[QSTAGES];  // the producer found no further stage
};
constexpr int RSMEM = QSTAGES * STAGE_BYTES + XPOSE_BYTES + (int)sizeof(QuantBars) + 1024;

struct QuantMaps {
  CUtensorMap m[3];  // [rows, 128] bf16 of each tensor, 64 x 256 boxes, 128-byte swizzle
};

// XOR masks that negate halves of bf16 pair words: bit 15 (low half) and bit
// 31 (high half) from the sign bits of int8 signs.  sw holds the signs of four
// consecutive elements 4 j .. 4 j + 3; lo: the word of elements 4 j, 4 j + 1,
// hi: the word of 4 j + 2, 4 j + 3.
__device__ __forceinline__ uint32_t sign_mask_lo(uint32_t sw) { return __byte_perm(sw, 0u, 0x1404) & 0x80008000u; }
__device__ __forceinline__ uint32_t sign_mask_hi(uint32_t sw) { return __byte_perm(sw, 0u, 0x3424) & 0x80008000u; }

// Butterflies of distances 2 .. 64 on the pairs P[j] = (y[2 j], y[2 j + 1]):
// (a, b) -> (a + b, a - b) on pair indices (j, j ^ hb).
__device__ __forceinline__ void butterflies_2_64(uint64_t (&P)[64]) {
  const uint64_t m1 = f2_pack(-1.f, -1.f);
#pragma unroll
  for (int hb = 1; hb < 64; hb <<= 1) {
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      if (j & hb) continue;
      const uint64_t a2 = P[j], b2 = P[j | hb];
      P[j] = f2_add(a2, b2);
      P[j | hb] = f2_fma(b2, m1, a2);
    }
  }
}

// Pass 1 (WRITE false): amax of every (batch, head).  Pass 2 (WRITE true):
// e4m3 codes scaled by 448 / amax.  ROPE: rotary embedding in front.
//
// A stage of 256 rows reaches shared memory as two tensor copies (columns
// 0-63 and 64-127) with the 128-byte swizzle: 16-byte chunk c of row r sits in
// slot c ^ (r % 8) of the row's 128 bytes, so a thread reading its own row
// chunk by chunk meets eight different bank groups across any eight
// consecutive rows.  Codes leave through a per-warp transposition in shared
// memory (row r, chunk c in slot c ^ (r % 8) again), so each store
// instruction writes four whole rows.  With sixteen warps of eight lanes per
// row instead (three butterfly stages through warp shuffles), the passes were
// held back by their instruction count: 0.27 ms where this form takes 0.21.
template <bool WRITE, bool ROPE>
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
  if (ROPE && threadIdx.x < 64) S.rope_f[threadIdx.x] = exp2f(-(float)threadIdx.x * t.rope_k);
  __syncthreads();
  if (warp >= RWARPS) {
    // ------------------------------------------------------------ producer
    regs_dec<R_LOW>();
    if (warp == RWARPS && lane == 0) {
      for (int i = 0; i < 3; ++i)
        if (t.rows[i] > 0) tma_prefetch_desc(&maps.m[i]);
      long long total = 0;
      for (int i = 0; i < 3; ++i) total += (t.rows[i] + STAGE_ROWS - 1) / STAGE_ROWS;
      long long k = 0;
      bool ok = true;
      for (long long g = blockIdx.x;; g += gridDim.x, ++k) {
        const int s = (int)(k % QSTAGES);
        if (!(ok = mbar_wait(&S.empty[s], (uint32_t)((k / QSTAGES) & 1) ^ 1u, ab))) break;
        Group gr;
        StageInfo& in = S.info[s];
        // Pass 2 walks the stages backwards: it starts on the rows pass 1
        // read last, which are still in L2.
        if (g >= total || !stage_of(t, WRITE ? total - 1 - g : g, gr)) {  // tell the compute warps, with no copy
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
  regs_inc<R_HIGH>();
  const int lr = warp * 32 + lane;  // this thread's row of every stage
  uint8_t* xw = xpose + warp * (32 * 128);
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
    const bool signed_rows = ti != 2 && t.signs != nullptr;
    const uint4* sg = nullptr;  // the row's 128 sign bytes
    if (signed_rows) sg = reinterpret_cast<const uint4*>(t.signs + (in.one_n ? in.hk0 : sign_head(t, ti, rowc / t.N)) * 128);
    uint64_t P[64];  // P[j] = (y[2 j], y[2 j + 1])
    if (ROPE && ti != 2) {
      float v[128];
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        v[2 * j] = bf16lo_f32(w[j]);
        v[2 * j + 1] = bf16hi_f32(w[j]);
      }
      const long long n = in.one_n ? in.n0 : rowc / t.N;
      const float fpos = (float)(int)(rowc - n * t.N);
#pragma unroll
      for (int c = 0; c < 64; ++c) {  // rotate-half pairs (c, c + 64), frequency index c
        // Angle reduced to [-pi, pi] by Cody and Waite's two-constant method:
        // 2 pi = C1 - C2 with C1 = fl(2 pi) and C2 = 1.7484556e-7 its excess;
        // both steps are fused multiply-adds, so k C1 enters exactly.  Then
        // the fast sine / cosine, accurate to a few 1e-7 on that interval.
        const float ang = fpos * S.rope_f[c];
        const float kf = rintf(ang * 0.15915494309189535f);  // 1 / (2 pi)
        const float red = fmaf(kf, 1.7484556e-07f, fmaf(-kf, 6.28318548f, ang));
        float sn, cs;
        __sincosf(red, &sn, &cs);
        const float x1 = v[c], x2 = v[c + 64];
        v[c] = fmaf(x1, cs, -x2 * sn);
        v[c + 64] = fmaf(x2, cs, x1 * sn);
      }
      if (signed_rows) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // elements 16 i .. 16 i + 15
          const uint4 q = __ldg(sg + i);
          const uint32_t sw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = 16 * i + e;
            v[c] = __uint_as_float(__float_as_uint(v[c]) ^ ((sw[e >> 2] << (24 - 8 * (e & 3))) & 0x80000000u));
          }
        }
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float a = v[2 * j], b = v[2 * j + 1];
          P[j] = f2_pack(a + b, a - b);  // distance 1
        }
        butterflies_2_64(P);
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) P[j] = f2_pack(v[2 * j], v[2 * j + 1]);
      }
    } else if (signed_rows) {
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
      butterflies_2_64(P);
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
  QuantMaps maps{};
  for (int i = 0; i < 3; ++i)
    if (t.rows[i] > 0 && !make_rows_map(&maps.m[i], t.x[i], t.rows[i], STAGE_ROWS)) return cudaErrorInvalidValue;
  const bool rope = t.rope_k != 0.f;
  auto p1 = rope ? quant_rows_kernel<false, true> : quant_rows_kernel<false, false>;
  auto p2 = rope ? quant_rows_kernel<true, true> : quant_rows_kernel<true, false>;
  // The register split inside the kernels assumes R_LAUNCH registers a thread
  // at launch: with fewer, the compute warps' increase could never be granted.
  static int regs[4] = {-1, -1, -1, -1};
  for (int w = 0; w < 2; ++w) {
    int& r = regs[2 * rope + w];
    if (r < 0) {
      cudaFuncAttributes fa;
      if ((e = cudaFuncGetAttributes(&fa, w ? p2 : p1)) != cudaSuccess) return e;
      r = fa.numRegs;
    }
    if (r != R_LAUNCH) return cudaErrorInvalidConfiguration;
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
