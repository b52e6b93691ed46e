// Host-side launch interfaces between the C-ABI layer (api.cu) and the
// kernel translation units.  Internal to the library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "common.cuh"

namespace attn {

struct FwdLaunch {
  CUtensorMap tq, tk, tv;  // Q [B*Hq, N, d], K/V [B*Hkv, N, d], 128x128-row boxes, 128-B swizzle
  void* o;
  float* lse;
  AttnParams p;
};
// mods: soft-cap / ALiBi present; masks: window / document masks present.
cudaError_t launch_fwd_bf16(const FwdLaunch& L, int d, bool mods, bool masks, cudaStream_t st);

struct Fp8Launch {
  CUtensorMap tq, tk, tv;  // e4m3 tensors
  const float* scales;     // [B*Hq] q, [B*Hkv] k, [B*Hkv] v
  void* o;
  float* lse;
  AttnParams p;
};
cudaError_t launch_fwd_fp8(const Fp8Launch& L, bool mods, bool masks, cudaStream_t st);

struct BwdLaunch {
  CUtensorMap tq, tk, tv, tdo;  // bf16 maps like the forward's
  const void* o;
  const void* dout;
  const float* lse;
  float2* rowstat;  // [B, Hq, nT*128] workspace: {LSE * log2(e) (+inf: no P), D = rowsum(dO*O)}
  void* dq;
  void* dk;
  void* dv;
  AttnParams p;
  cudaEvent_t events[4];  // optional: recorded before pre / dkdv / dq and after dq
  // One-kernel backward (causal masks, d = 128) only, all workspace:
  const void* k;   // K, V (for the fixed-point bounds)
  const void* v;
  float2* kvb;     // [B, Hkv] {max |K|, max_j ||V_j||}
  float* qscale;   // [B, Hq, nT*128] quantum multiplier of each query row's dQ
  int* dqacc;      // [B, Hq, nT*128, d] int32 dQ sums in those quanta
  int* ticket;     // work-item counter
  int sms;         // persistent CTAs
  // Mixed e4m3 backward (d = 128, causal or no mask) only, all workspace:
  bool fp8;                // dP^T and dV GEMMs in e4m3
  CUtensorMap tdo8, tv8;   // e4m3 maps of do8, v8
  void* do8;               // e4m3 [B, Hq, N, d]: dO / its scale
  void* v8;                // e4m3 [B, Hkv, N, d]: V / its scale
  float* fp8s;             // [B * Hkv] dO scales, then [B * Hkv] V scales (amax / 448)
  unsigned* fp8amax;       // [2 * B * Hkv] amax scratch
};
// Two kernels after the row statistics (dK/dV kv-stationary, dQ q-stationary).
cudaError_t launch_bwd(const BwdLaunch& L, int d, bool mods, bool masks, cudaStream_t st);
// One main kernel (plus bounds, row statistics and a dQ conversion); needs
// MOD_CAUSAL and d = 128.
cudaError_t launch_bwd_fused(const BwdLaunch& L, int d, bool mods, bool masks, cudaStream_t st);

// Decode step over a paged K/V cache (d = 64 or 128): q_len new tokens per sequence.
struct DecodeParams {
  int B, Hq, Hkv, G;       // G = Hq / Hkv query heads per KV head
  int q_len;               // new tokens per sequence (G * q_len <= 128)
  int d;                   // head dimension: 64 or 128
  int bt_stride;           // block-table row length (blocks per sequence at most)
  int kv_blocks;           // cache blocks
  int ct;                  // key tiles of 128 per work item (chunk)
  int max_chunks;          // chunks per (sequence, head) in the partial buffers
  float scale_log2;        // scale * log2(e)
  float sc_in, sc_out;     // soft-cap: scale / c and c * log2(e)
  uint32_t flags;          // MOD_WINDOW | MOD_SOFTCAP | MOD_ALIBI (causal is implied)
  int window;
  const float* slopes;     // [Hq] or nullptr (default ALiBi slopes)
  const int* block_table;  // [B, bt_stride]
  const int* seqlens;      // [B] cached tokens, the new ones the last q_len
  int4* seq_info;          // [B] workspace: {L, first key tile, chunks, first item}
  int* n_items;            // workspace: number of items
  float* o_part;           // [B, Hq, q_len, max_chunks, d] workspace: O / l of each chunk
  float* lse_part;         // [B, Hq, q_len, max_chunks] workspace: log2-sum-exp of each chunk
  int* status;             // device status word
  unsigned long long wait_ns;  // time limit of a pipeline wait (ns)
};
struct DecodeLaunch {
  CUtensorMap tq;      // Q as [B*Hkv, G*q_len, d]: box of G*q_len rows x 64 columns
  CUtensorMap tk, tv;  // cache [kv_blocks*Hkv, 16, d]: 16-row boxes
  void* o;             // bf16 [B, Hq, q_len, d]
  float* lse;          // [B, Hq, q_len]
  int grid;            // persistent CTAs
  DecodeParams p;
};
// mods: soft-cap / ALiBi present.
cudaError_t launch_decode(const DecodeLaunch& L, bool mods, cudaStream_t st);

cudaError_t launch_block_map(const AttnParams& p, uint8_t* map, cudaStream_t st);
cudaError_t launch_tile_ranges(const AttnParams& p, const uint8_t* map, int2* rows, int2* cols,
                               cudaStream_t st);
cudaError_t launch_doc_bounds(const AttnParams& p, int2* bounds, int* unsorted, cudaStream_t st);
cudaError_t launch_seq_ids(const int* cu, int n_seqs, int total, int* ids, cudaStream_t st);

// TMA descriptor of a [rows, 128] bf16 tensor: 64-column x box_rows-row boxes,
// 128-byte swizzle (api.cu).
bool make_rows_map(CUtensorMap* m, const void* ptr, long long rows, int box_rows);

// rope_base > 0: RoPE (rotate-half, position = row index) applied first.
cudaError_t launch_hadamard_quant(const void* q, const void* k, const void* v, void* q8, void* k8,
                                  void* v8, float* scales, const int8_t* signs, int B, int Hq,
                                  int Hkv, int N, float rope_base, unsigned* amax_ws, int* status,
                                  cudaStream_t st);
cudaError_t launch_quant_bwd_fp8(const void* dout, const void* v, void* do8, void* v8, float* scales, int B,
                                 int Hq, int Hkv, int N, unsigned* amax_ws, int* status, cudaStream_t st);

}  // namespace attn
