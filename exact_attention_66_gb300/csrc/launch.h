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
};
cudaError_t launch_bwd(const BwdLaunch& L, int d, bool mods, bool masks, cudaStream_t st);

cudaError_t launch_block_map(const AttnParams& p, uint8_t* map, cudaStream_t st);
cudaError_t launch_tile_ranges(const AttnParams& p, const uint8_t* map, int2* rows, int2* cols,
                               cudaStream_t st);
cudaError_t launch_doc_bounds(const AttnParams& p, int2* bounds, int* unsorted, cudaStream_t st);
cudaError_t launch_seq_ids(const int* cu, int n_seqs, int total, int* ids, cudaStream_t st);

// rope_base > 0: RoPE (rotate-half, position = row index) applied first.
cudaError_t launch_hadamard_quant(const void* q, const void* k, const void* v, void* q8, void* k8,
                                  void* v8, float* scales, const int8_t* signs, int B, int Hq,
                                  int Hkv, int N, float rope_base, unsigned* amax_ws, cudaStream_t st);

}  // namespace attn
