// Block-sparsity map: every 128 x 128 tile (b, I, J) is classified as skip /
// partial / full from the allowed (i, j) pairs it holds (FlexAttention/FA4
// page, "Limitations actuelles": block sparsity; tile size 128 as named
// there).  Tiles that the causal or window bound rules out as a whole are
// classified at once.  Otherwise one thread per row finds the row's allowed
// columns in the tile: with causal, window and the sequence end they form
// the interval [max(j_lo, i - window + 1), min(j_hi, i, N - 1)], and a
// document whose ids form one run ([start, end) from the document-run
// kernel, when every batch row's ids are non-decreasing) narrows it to
// [start, end - 1].  The tile is full when every row's interval is the whole
// tile, skip when every interval is empty.  Without the runs, or with ids
// that decrease somewhere, the document test goes pair by pair.
#include "common.cuh"
#include "launch.h"

namespace attn {

__global__ void __launch_bounds__(256) block_map_kernel(const AttnParams p, uint8_t* __restrict__ map) {
  const int J = blockIdx.x, I = blockIdx.y, b = blockIdx.z;
  const bool causal = (p.flags & MOD_CAUSAL) != 0;
  const bool win = (p.flags & MOD_WINDOW) != 0;
  const bool doc = (p.flags & MOD_DOC) != 0;
  uint8_t* out = map + ((size_t)b * p.nT + I) * p.nT + J;
  const int i_lo = I * TILE, j_lo = J * TILE;
  const int i_hi = min(i_lo + TILE, p.N) - 1;  // last real row
  // Whole-tile rejections: all pairs have j > i, or all have i - j >= window.
  if ((causal && j_lo > i_hi) || (win && i_lo - (j_lo + TILE - 1) >= p.window)) {
    if (threadIdx.x == 0) *out = CLS_SKIP;
    return;
  }
  const bool doc_pairs = doc && (p.doc_bounds == nullptr || *p.doc_unsorted != 0);
  const int r = threadIdx.x & (TILE - 1);
  const int half = threadIdx.x >> 7;
  const int i = i_lo + r;
  bool any_ok = false, all_ok = true;
  if (i < p.N && !doc_pairs) {
    if (half == 0) {
      int lo = j_lo, hi = min(j_lo + TILE, p.N) - 1;
      if (causal) hi = min(hi, i);
      if (win) lo = max(lo, i - p.window + 1);
      if (doc) {
        const int2 run = p.doc_bounds[(size_t)b * p.N + i];
        lo = max(lo, run.x);
        hi = min(hi, run.y - 1);
      }
      any_ok = lo <= hi;
      all_ok = lo == j_lo && hi == j_lo + TILE - 1;
    }
  } else if (i < p.N) {
    const int di = p.doc_ids[(size_t)b * p.N + i];
#pragma unroll 4
    for (int c = 0; c < TILE / 2; ++c) {
      const int j = j_lo + half * (TILE / 2) + c;
      bool ok = j < p.N;
      if (ok && causal) ok = j <= i;
      if (ok && win) ok = (i - j) < p.window;
      if (ok) ok = p.doc_ids[(size_t)b * p.N + j] == di;
      any_ok |= ok;
      all_ok &= ok;
    }
  }
  any_ok = __syncthreads_or(any_ok);
  all_ok = __syncthreads_and(all_ok);
  if (threadIdx.x == 0) {
    int c = !any_ok ? CLS_SKIP : ((all_ok && j_lo + TILE <= p.N) ? CLS_FULL : CLS_PARTIAL);
    *out = (uint8_t)c;
  }
}

// Runs of equal document ids: for every position, the [start, end) of the run
// holding it, by binary search on the ids of its batch row (which assumes
// they do not decrease along N), and a flag set when some id does decrease
// (the kernels then test ids element by element instead).
__global__ void __launch_bounds__(256) doc_bounds_kernel(const int* __restrict__ doc, int B, int N,
                                                         int2* __restrict__ bounds, int* __restrict__ unsorted) {
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (long long)B * N) return;
  const int b = (int)(t / N), pos = (int)(t - (long long)b * N);
  const int* d = doc + (size_t)b * N;
  const int id = d[pos];
  if (pos + 1 < N && d[pos + 1] < id) atomicOr(unsorted, 1);
  int lo = 0, hi = pos;  // first index whose id is >= id
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (d[mid] < id) lo = mid + 1; else hi = mid;
  }
  const int start = lo;
  lo = pos + 1;
  hi = N;  // first index whose id is > id
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (d[mid] <= id) lo = mid + 1; else hi = mid;
  }
  bounds[t] = make_int2(start, lo);
}

// Sequence id of every packed row from the sequence offsets: the last s with
// cu[s] <= row (binary search over cu[0..n_seqs]); -1 before cu[0].  Reads
// only cu[0..n_seqs], whatever the values.
__global__ void __launch_bounds__(256) seq_ids_kernel(const int* __restrict__ cu, int n_seqs, int total,
                                                      int* __restrict__ ids) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= total) return;
  int lo = 0, hi = n_seqs + 1;  // first index with cu[index] > row
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= row) lo = mid + 1; else hi = mid;
  }
  ids[row] = min(lo - 1, n_seqs - 1);
}

cudaError_t launch_seq_ids(const int* cu, int n_seqs, int total, int* ids, cudaStream_t st) {
  seq_ids_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(cu, n_seqs, total, ids);
  return cudaGetLastError();
}

// Per Q tile (row of the map) and per KV tile (column): the range
// [first, last + 1) of non-skipped tiles, (0, 0) when there is none.  Lets
// the attention kernels start their tile loops at the first tile they need.
// One warp per (b, x): its lanes stride over map row x and map column x,
// then min / max reductions across the warp.
__global__ void __launch_bounds__(256) tile_range_kernel(const uint8_t* __restrict__ map, int nT, int B,
                                                         int2* __restrict__ rows, int2* __restrict__ cols) {
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)B * nT) return;
  const int b = (int)(gw / nT), x = (int)(gw - (long long)b * nT);
  const uint8_t* m = map + (size_t)b * nT * nT;
  int r0 = nT, r1 = -1, c0 = nT, c1 = -1;
  for (int y = lane; y < nT; y += 32) {
    if (m[(size_t)x * nT + y] != CLS_SKIP) { r0 = min(r0, y); r1 = y; }
    if (m[(size_t)y * nT + x] != CLS_SKIP) { c0 = min(c0, y); c1 = y; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    r0 = min(r0, __shfl_xor_sync(0xffffffffu, r0, o));
    r1 = max(r1, __shfl_xor_sync(0xffffffffu, r1, o));
    c0 = min(c0, __shfl_xor_sync(0xffffffffu, c0, o));
    c1 = max(c1, __shfl_xor_sync(0xffffffffu, c1, o));
  }
  if (lane == 0) {
    rows[(size_t)b * nT + x] = r1 < 0 ? make_int2(0, 0) : make_int2(r0, r1 + 1);
    cols[(size_t)b * nT + x] = c1 < 0 ? make_int2(0, 0) : make_int2(c0, c1 + 1);
  }
}

cudaError_t launch_block_map(const AttnParams& p, uint8_t* map, cudaStream_t st) {
  const dim3 grid(p.nT, p.nT, p.B);
  block_map_kernel<<<grid, 256, 0, st>>>(p, map);
  return cudaGetLastError();
}

cudaError_t launch_tile_ranges(const AttnParams& p, const uint8_t* map, int2* rows, int2* cols,
                               cudaStream_t st) {
  const long long threads = (long long)p.B * p.nT * 32;
  tile_range_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(map, p.nT, p.B, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_doc_bounds(const AttnParams& p, int2* bounds, int* unsorted, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(unsorted, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  const long long n = (long long)p.B * p.N;
  doc_bounds_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(p.doc_ids, p.B, p.N, bounds, unsorted);
  return cudaGetLastError();
}

}  // namespace attn
