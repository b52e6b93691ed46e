// C ABI of the attention library (declared in include/attn.h): argument
// validation, workspace carve-up, TMA descriptor encoding and kernel launch.
// Every argument check runs before the first CUDA call, so a bad call returns
// its status without touching the device.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include "../../include/attn.h"
#include "launch.h"

namespace attn {
__device__ int g_status;  // device status word (DEV_OK / DEV_ERR_*)
}

using namespace attn;

namespace {

constexpr int kMaxDevices = 64;

// Test hooks (attn_test_hooks): the pipeline-wait limit and the stall bits
// copied into the parameters of every later launch.
std::atomic<unsigned long long> g_wait_ns{ATTN_WAIT_TIMEOUT_NS};
std::atomic<int> g_stall{0};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int n_tiles(int N) { return (N + TILE - 1) / TILE; }

uint32_t mod_flags(const attn_mods_t* m) { return m ? m->flags : 0u; }

bool needs_map(uint32_t flags) { return (flags & (ATTN_MOD_WINDOW | ATTN_MOD_DOC)) != 0; }

size_t map_bytes(int B, int N) { return round_up((size_t)B * n_tiles(N) * n_tiles(N), 256); }

// Workspace of the window / document mods: the block map, then (documents)
// the run bounds of every position and the "ids not sorted" flag.
size_t doc_bytes(int B, int N) { return round_up((size_t)B * N * sizeof(int2), 256) + 256; }
size_t range_bytes(int B, int N) { return round_up((size_t)B * n_tiles(N) * sizeof(int2), 256); }
size_t mods_bytes(int B, int N, uint32_t flags) {
  if (!needs_map(flags)) return 0;
  return map_bytes(B, N) + 2 * range_bytes(B, N) + ((flags & ATTN_MOD_DOC) ? doc_bytes(B, N) : 0);
}

attn_status_t check_mods(const attn_mods_t* m) {
  if (!m) return ATTN_OK;
  const uint32_t known = ATTN_MOD_CAUSAL | ATTN_MOD_WINDOW | ATTN_MOD_DOC | ATTN_MOD_SOFTCAP |
                         ATTN_MOD_ALIBI | ATTN_MOD_BWD_FP8;
  if (m->flags & ~known) return ATTN_ERR_INVALID_ARG;
  if ((m->flags & ATTN_MOD_WINDOW) && m->window < 1) return ATTN_ERR_INVALID_ARG;
  if ((m->flags & ATTN_MOD_DOC) && (m->doc_ids == nullptr || !aligned(m->doc_ids, 4)))
    return ATTN_ERR_INVALID_ARG;
  if ((m->flags & ATTN_MOD_SOFTCAP) && !(std::isfinite(m->softcap) && m->softcap > 0.f))
    return ATTN_ERR_INVALID_ARG;
  if ((m->flags & ATTN_MOD_ALIBI) && m->alibi_slopes && !aligned(m->alibi_slopes, 4))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status_t check_shape(int B, int Hq, int Hkv, int N, int d, bool fp8) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_UNSUPPORTED;
  if (fp8 ? d != 128 : (d != 64 && d != 128)) return ATTN_ERR_UNSUPPORTED;
  const long long planes = (long long)B * (Hq > Hkv ? Hq : Hkv);
  if (planes * N >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn_status_t check_tensors(std::initializer_list<const void*> ps) {
  for (const void* p : ps) {
    if (p == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(p, 16)) return ATTN_ERR_UNSUPPORTED;
  }
  return ATTN_OK;
}

attn_status_t check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return ATTN_OK;
  if (ws == nullptr || ws_bytes < need || !aligned(ws, 256)) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

// ---- device state: sm_103 check, status word address (per device) --------
struct DevState {
  int checked = 0;  // 0 unknown, 1 ok, -1 unsupported
  int* status = nullptr;
};
DevState g_dev[kMaxDevices];
std::mutex g_mu;

attn_status_t device_state(int** status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& s = g_dev[dev];
  if (s.checked == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (major != 10 || minor != 3) {
      s.checked = -1;
    } else {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return ATTN_ERR_CUDA;
      s.status = static_cast<int*>(p);
      s.checked = 1;
    }
  }
  if (s.checked < 0) return ATTN_ERR_DEVICE;
  *status = s.status;
  return ATTN_OK;
}

// ---- TMA descriptors -------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [planes, N, d] contiguous tensor; box = 128 rows x 128 bytes, 128-B swizzle.
bool make_map(CUtensorMap* m, const void* ptr, bool e4m3, int d, int N, long long planes) {
  auto enc = encode_fn();
  if (!enc) return false;
  const int es = e4m3 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)d * es, (cuuint64_t)N * d * es};
  cuuint32_t box[3] = {(cuuint32_t)(128 / es), (cuuint32_t)TILE, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K/V cache of 16-row blocks, [kv_blocks, Hkv, 16, d] bf16: 3-D map over
// (d, 16 rows, block x head) with 64-column x 16-row boxes, 128-byte swizzle.
bool make_paged_map(CUtensorMap* m, const void* ptr, int d, long long planes) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, 16, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)16 * d * 2};
  cuuint32_t box[3] = {64, 16, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

AttnParams make_params(int B, int Hq, int Hkv, int N, float scale, const attn_mods_t* mods,
                       int* status) {
  AttnParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.nT = n_tiles(N);
  p.n_qblk = (N + 2 * TILE - 1) / (2 * TILE);
  p.scale = scale;
  p.scale_log2 = scale * LOG2E;
  p.flags = mod_flags(mods);
  p.window = mods ? mods->window : 0;
  p.softcap = (mods && (mods->flags & ATTN_MOD_SOFTCAP)) ? mods->softcap : 1.0f;
  p.doc_ids = (mods && (mods->flags & ATTN_MOD_DOC)) ? mods->doc_ids : nullptr;
  p.slopes = (mods && (mods->flags & ATTN_MOD_ALIBI)) ? mods->alibi_slopes : nullptr;
  p.map = nullptr;
  p.row_range = nullptr;
  p.col_range = nullptr;
  p.doc_bounds = nullptr;
  p.doc_unsorted = nullptr;
  p.block_table = nullptr;
  p.kv_blocks = 0;
  p.bt_stride = 0;
  p.status = status;
  p.wait_ns = g_wait_ns.load();
  p.stall = g_stall.load();
  return p;
}

// Soft-cap and ALiBi change the scores; the masks (causal, window,
// documents) are column intervals or element tests on partial tiles only and
// run in both kernel variants.
bool has_score_mods(uint32_t flags) { return (flags & (ATTN_MOD_SOFTCAP | ATTN_MOD_ALIBI)) != 0; }

// Backward row statistics: one {LSE * log2(e), D} pair per query row, rows
// padded to whole 128-row tiles so that every tile's pairs are 16-byte aligned.
size_t bwd_rowstat_bytes(int B, int Hq, int N) {
  return round_up((size_t)B * Hq * ((N + 127) / 128) * 128 * sizeof(float2), 256);
}

// The one-kernel backward runs causal masks with window / document parts at
// d = 128 (measured on GB300: 20 % faster than the two kernels on the flex
// workload, whose KV tiles meet few, mostly partial Q tiles; 7-10 % slower on
// plain causal masks, where its dQ reductions slow the MMA pipe by more than
// the two saved GEMMs).  Its workspace, after the row statistics and the mods
// region: the per-row dQ quanta, the K/V bounds, the work-item counter and the
// int32 dQ accumulator.
bool bwd_fused(uint32_t flags, int d) {
  return (flags & ATTN_MOD_CAUSAL) != 0 && needs_map(flags) && d == 128;
}
size_t bwd_qscale_bytes(int B, int Hq, int N) { return round_up((size_t)B * Hq * n_tiles(N) * TILE * sizeof(float), 256); }
size_t bwd_kvb_bytes(int B, int Hkv) { return round_up((size_t)B * Hkv * sizeof(float2), 256); }
size_t bwd_dqacc_bytes(int B, int Hq, int N, int d) {
  return round_up((size_t)B * Hq * n_tiles(N) * TILE * d * sizeof(int), 256);
}
size_t bwd_fused_bytes(int B, int Hq, int Hkv, int N, int d, uint32_t flags) {
  return bwd_fused(flags, d) ? bwd_qscale_bytes(B, Hq, N) + bwd_kvb_bytes(B, Hkv) + 256 + bwd_dqacc_bytes(B, Hq, N, d)
                             : 0;
}

// Mixed e4m3 backward (ATTN_MOD_BWD_FP8): d = 128 and no mod but the causal
// mask.  Its workspace, after the row statistics: e4m3 dO and V, their scales
// (2 B Hkv floats) and the amax scratch of the quantisation (2 B Hkv words).
bool bwd_fp8(uint32_t flags) { return (flags & ATTN_MOD_BWD_FP8) != 0; }
bool bwd_fp8_supported(uint32_t flags, int d) {
  return d == 128 && (flags & ~(uint32_t)(ATTN_MOD_CAUSAL | ATTN_MOD_BWD_FP8)) == 0;
}
size_t bwd_do8_bytes(int B, int Hq, int N, int d) { return round_up((size_t)B * Hq * N * d, 256); }
size_t bwd_v8_bytes(int B, int Hkv, int N, int d) { return round_up((size_t)B * Hkv * N * d, 256); }
size_t bwd_fp8s_bytes(int B, int Hkv) { return round_up((size_t)2 * B * Hkv * sizeof(float), 256); }
size_t bwd_fp8_bytes(int B, int Hq, int Hkv, int N, int d, uint32_t flags) {
  return bwd_fp8(flags) ? bwd_do8_bytes(B, Hq, N, d) + bwd_v8_bytes(B, Hkv, N, d) + 2 * bwd_fp8s_bytes(B, Hkv) : 0;
}

attn_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Varlen workspace head: the sequence id of every packed row.
size_t varlen_ids_bytes(int total) { return round_up((size_t)total * sizeof(int32_t), 256); }

// Checks shared by the varlen entry points; on success writes the document
// mods that describe the sequences (doc_ids = the ids in the workspace).
attn_status_t varlen_setup(const int32_t* cu, int n_seqs, int Hq, int Hkv, int total, int d,
                           const attn_mods_t* mods, void* ws, size_t ws_bytes, bool bwd,
                           attn_mods_t* out, void* stream) {
  attn_status_t st;
  if (cu == nullptr || n_seqs < 1 || !aligned(cu, 4)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_shape(1, Hq, Hkv, total, d, false)) != ATTN_OK) return st;
  if ((st = check_mods(mods)) != ATTN_OK) return st;
  if (mods && (mods->flags & ATTN_MOD_DOC)) return ATTN_ERR_INVALID_ARG;
  const size_t need = attn_workspace_size(bwd ? ATTN_OP_BWD_VARLEN : ATTN_OP_FWD_VARLEN, 1, Hq, Hkv,
                                          total, d, mods);
  if ((st = check_ws(ws, ws_bytes, need)) != ATTN_OK) return st;
  int* status = nullptr;
  if ((st = device_state(&status)) != ATTN_OK) return st;
  int32_t* ids = static_cast<int32_t*>(ws);
  if ((st = cuda_status(launch_seq_ids(cu, n_seqs, total, ids, static_cast<cudaStream_t>(stream)))) != ATTN_OK)
    return st;
  attn_mods_t m{};
  if (mods) m = *mods;
  m.flags |= ATTN_MOD_DOC;
  m.doc_ids = ids;
  *out = m;
  return ATTN_OK;
}

// Fill the mods workspace (document runs, block map, tile ranges) and point
// p at it.  The runs come first: the block map classifies tiles from them
// when the ids are non-decreasing.
attn_status_t prepare_mods(AttnParams& p, uint8_t* region, cudaStream_t s) {
  if (!needs_map(p.flags)) return ATTN_OK;
  attn_status_t st;
  if (p.flags & ATTN_MOD_DOC) {
    uint8_t* dregion = region + map_bytes(p.B, p.N) + 2 * range_bytes(p.B, p.N);
    int2* bounds = reinterpret_cast<int2*>(dregion);
    int* unsorted = reinterpret_cast<int*>(dregion + doc_bytes(p.B, p.N) - 256);
    if ((st = cuda_status(launch_doc_bounds(p, bounds, unsorted, s))) != ATTN_OK) return st;
    p.doc_bounds = bounds;
    p.doc_unsorted = unsorted;
  }
  if ((st = cuda_status(launch_block_map(p, region, s))) != ATTN_OK) return st;
  p.map = region;
  int2* rows = reinterpret_cast<int2*>(region + map_bytes(p.B, p.N));
  int2* cols = reinterpret_cast<int2*>(region + map_bytes(p.B, p.N) + range_bytes(p.B, p.N));
  if ((st = cuda_status(launch_tile_ranges(p, region, rows, cols, s))) != ATTN_OK) return st;
  p.row_range = rows;
  p.col_range = cols;
  return ATTN_OK;
}

// ---- paged decode ----------------------------------------------------------
// Work items of `ct` key tiles, about this many in all (16 for each SM of a
// 152-SM part), so that every persistent CTA walks many items and the last
// ones finish together.  A pure function of the shape, so that the workspace
// size is too.
constexpr long long kDecodeTargetItems = 16 * 152;

struct DecodeSplit {
  int ct, max_chunks;
};
DecodeSplit decode_split(int B, int Hkv, int N) {
  const int tiles = n_tiles(N);
  const long long units = (long long)B * Hkv * tiles;
  long long ct = (units + kDecodeTargetItems - 1) / kDecodeTargetItems;
  if (ct < 1) ct = 1;
  if (ct > tiles) ct = tiles;
  return {(int)ct, (int)((tiles + ct - 1) / ct)};
}
size_t decode_info_bytes(int B) { return round_up((size_t)B * sizeof(int4), 256) + 256; }
size_t decode_ws_bytes(int B, int Hq, int Hkv, int T, int N, int d) {
  const size_t rows = (size_t)B * Hq * T * decode_split(B, Hkv, N).max_chunks;
  return decode_info_bytes(B) + round_up(rows * d * sizeof(float), 256) + round_up(rows * sizeof(float), 256);
}
attn_status_t check_decode(int B, int Hq, int Hkv, int T, int N, int num_blocks, int d, const attn_mods_t* mods) {
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1 || N < 16 || num_blocks < 1) return ATTN_ERR_INVALID_ARG;
  if (N % 16 != 0 || Hq % Hkv != 0 || (long long)(Hq / Hkv) * T > 128 || (d != 64 && d != 128))
    return ATTN_ERR_UNSUPPORTED;
  if ((long long)num_blocks * Hkv >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  attn_status_t st;
  if ((st = check_mods(mods)) != ATTN_OK) return st;
  if (mods && (mods->flags & ATTN_MOD_DOC)) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq * T * decode_split(B, Hkv, N).max_chunks * d >= (1ll << 40)) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hq * T >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  if ((long long)B * Hkv * decode_split(B, Hkv, N).max_chunks >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

int sm_count() {
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace

namespace attn {
// [rows, 128] bf16 rows (any row count); box = 64 columns x box_rows rows,
// 128-B swizzle, rows past the end read as zeros.
bool make_rows_map(CUtensorMap* m, const void* ptr, long long rows, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace attn

extern "C" {

size_t attn_workspace_size(int op, int B, int Hq, int Hkv, int N, int d, const attn_mods_t* mods) {
  if (op == ATTN_OP_DECODE_PAGED)
    return N % 16 == 0 ? attn_decode_workspace_size(B, Hq, Hkv, 1, N / 16, d, mods) : 0;
  if (check_shape(B, Hq, Hkv, N, d, op == ATTN_OP_FWD_FP8 || op == ATTN_OP_QUANT_FP8) != ATTN_OK ||
      check_mods(mods) != ATTN_OK)
    return 0;
  const uint32_t f = mod_flags(mods);
  switch (op) {
    case ATTN_OP_FWD:
    case ATTN_OP_FWD_FP8:
      return mods_bytes(B, N, f);
    case ATTN_OP_BWD:
      return bwd_rowstat_bytes(B, Hq, N) + mods_bytes(B, N, f) + bwd_fused_bytes(B, Hq, Hkv, N, d, f) +
             bwd_fp8_bytes(B, Hq, Hkv, N, d, f);
    case ATTN_OP_QUANT_FP8:
      return round_up((size_t)(B * Hq + 2 * B * Hkv) * sizeof(unsigned), 256);
    case ATTN_OP_FWD_VARLEN:
    case ATTN_OP_BWD_VARLEN: {
      if (B != 1 || (f & ATTN_MOD_DOC)) return 0;
      const uint32_t fd = f | ATTN_MOD_DOC;  // the sequences are the documents
      return varlen_ids_bytes(N) +
             (op == ATTN_OP_FWD_VARLEN ? mods_bytes(1, N, fd)
                                       : bwd_rowstat_bytes(1, Hq, N) + mods_bytes(1, N, fd) +
                                             bwd_fused_bytes(1, Hq, Hkv, N, d, fd));
    }
    default:
      return 0;
  }
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int N, int d, float scale, const attn_mods_t* mods,
                       void* ws, size_t ws_bytes, void* stream) {
  attn_status_t st;
  if ((st = check_shape(B, Hq, Hkv, N, d, false)) != ATTN_OK) return st;
  if ((st = check_tensors({q, k, v, o})) != ATTN_OK) return st;
  if (lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned(lse, 4)) return ATTN_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_mods(mods)) != ATTN_OK) return st;
  const size_t need = attn_workspace_size(ATTN_OP_FWD, B, Hq, Hkv, N, d, mods);
  if ((st = check_ws(ws, ws_bytes, need)) != ATTN_OK) return st;
  int* status = nullptr;
  if ((st = device_state(&status)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  FwdLaunch L{};
  L.p = make_params(B, Hq, Hkv, N, scale, mods, status);
  if (!make_map(&L.tq, q, false, d, N, (long long)B * Hq) ||
      !make_map(&L.tk, k, false, d, N, (long long)B * Hkv) ||
      !make_map(&L.tv, v, false, d, N, (long long)B * Hkv))
    return ATTN_ERR_CUDA;
  L.o = o;
  L.lse = lse;
  if ((st = prepare_mods(L.p, static_cast<uint8_t*>(ws), s)) != ATTN_OK) return st;
  return cuda_status(launch_fwd_bf16(L, d, has_score_mods(L.p.flags), needs_map(L.p.flags), s));
}

static attn_status_t bwd_impl(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int N, int d, float scale,
                              const attn_mods_t* mods, void* ws, size_t ws_bytes, void* stream,
                              void* const* events) {
  attn_status_t st;
  if ((st = check_shape(B, Hq, Hkv, N, d, false)) != ATTN_OK) return st;
  if (N > BWD_MAX_N) return ATTN_ERR_UNSUPPORTED;
  if ((st = check_tensors({q, k, v, o, dout, dq, dk, dv})) != ATTN_OK) return st;
  if (lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned(lse, 4)) return ATTN_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_mods(mods)) != ATTN_OK) return st;
  if (bwd_fp8(mod_flags(mods)) && !bwd_fp8_supported(mod_flags(mods), d)) return ATTN_ERR_UNSUPPORTED;
  const size_t need = attn_workspace_size(ATTN_OP_BWD, B, Hq, Hkv, N, d, mods);
  if ((st = check_ws(ws, ws_bytes, need)) != ATTN_OK) return st;
  int* status = nullptr;
  if ((st = device_state(&status)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  BwdLaunch L{};
  L.p = make_params(B, Hq, Hkv, N, scale, mods, status);
  if (!make_map(&L.tq, q, false, d, N, (long long)B * Hq) ||
      !make_map(&L.tk, k, false, d, N, (long long)B * Hkv) ||
      !make_map(&L.tv, v, false, d, N, (long long)B * Hkv) ||
      !make_map(&L.tdo, dout, false, d, N, (long long)B * Hq))
    return ATTN_ERR_CUDA;
  L.o = o;
  L.dout = dout;
  L.lse = lse;
  L.dq = dq;
  L.dk = dk;
  L.dv = dv;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  L.rowstat = reinterpret_cast<float2*>(wsb);
  uint8_t* mregion = wsb + bwd_rowstat_bytes(B, Hq, N);
  if ((st = prepare_mods(L.p, mregion, s)) != ATTN_OK) return st;
  if (events != nullptr)
    for (int e = 0; e < 4; ++e) L.events[e] = static_cast<cudaEvent_t>(events[e]);
  if (bwd_fp8(L.p.flags)) {  // no mods region, no one-kernel region
    uint8_t* r8 = mregion;
    L.fp8 = true;
    L.v = v;
    L.do8 = r8;
    r8 += bwd_do8_bytes(B, Hq, N, d);
    L.v8 = r8;
    r8 += bwd_v8_bytes(B, Hkv, N, d);
    L.fp8s = reinterpret_cast<float*>(r8);
    L.fp8amax = reinterpret_cast<unsigned*>(r8 + bwd_fp8s_bytes(B, Hkv));
    if (!make_map(&L.tdo8, L.do8, true, d, N, (long long)B * Hq) ||
        !make_map(&L.tv8, L.v8, true, d, N, (long long)B * Hkv))
      return ATTN_ERR_CUDA;
  }
  if (!bwd_fused(L.p.flags, d))
    return cuda_status(launch_bwd(L, d, has_score_mods(L.p.flags), needs_map(L.p.flags), s));
  uint8_t* fregion = mregion + mods_bytes(B, N, L.p.flags);
  L.k = k;
  L.v = v;
  L.qscale = reinterpret_cast<float*>(fregion);
  fregion += bwd_qscale_bytes(B, Hq, N);
  L.kvb = reinterpret_cast<float2*>(fregion);
  fregion += bwd_kvb_bytes(B, Hkv);
  L.ticket = reinterpret_cast<int*>(fregion);
  L.dqacc = reinterpret_cast<int*>(fregion + 256);
  L.sms = sm_count();
  if (L.sms < 1) return ATTN_ERR_CUDA;
  return cuda_status(launch_bwd_fused(L, d, has_score_mods(L.p.flags), needs_map(L.p.flags), s));
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int N, int d, float scale, const attn_mods_t* mods,
                       void* ws, size_t ws_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, mods, ws, ws_bytes,
                  stream, nullptr);
}

attn_status_t attn_bwd_profiled(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int Hq, int Hkv, int N, int d, float scale,
                                const attn_mods_t* mods, void* ws, size_t ws_bytes, void* stream,
                                void* const* events) {
  if (events == nullptr) return ATTN_ERR_INVALID_ARG;
  for (int e = 0; e < 4; ++e)
    if (events[e] == nullptr) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, mods, ws, ws_bytes,
                  stream, events);
}

static attn_status_t quant_impl(const void* q, const void* k, const void* v, void* q8, void* k8,
                                void* v8, float* scales, const int8_t* signs, int B, int Hq, int Hkv,
                                int N, int d, float rope_base, void* ws, size_t ws_bytes, void* stream) {
  attn_status_t st;
  if ((st = check_shape(B, Hq, Hkv, N, d, true)) != ATTN_OK) return st;
  if ((st = check_tensors({q, k, v, q8, k8, v8})) != ATTN_OK) return st;
  if (scales == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned(scales, 4)) return ATTN_ERR_UNSUPPORTED;
  if (signs != nullptr && !aligned(signs, 16)) return ATTN_ERR_UNSUPPORTED;  // read in 16-byte words
  const size_t need = attn_workspace_size(ATTN_OP_QUANT_FP8, B, Hq, Hkv, N, d, nullptr);
  if ((st = check_ws(ws, ws_bytes, need)) != ATTN_OK) return st;
  int* status = nullptr;
  if ((st = device_state(&status)) != ATTN_OK) return st;
  return cuda_status(launch_hadamard_quant(q, k, v, q8, k8, v8, scales, signs, B, Hq, Hkv, N, rope_base,
                                           static_cast<unsigned*>(ws), status,
                                           static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_hadamard_quant_fp8(const void* q, const void* k, const void* v, void* q8,
                                      void* k8, void* v8, float* scales, const int8_t* signs,
                                      int B, int Hq, int Hkv, int N, int d, void* ws,
                                      size_t ws_bytes, void* stream) {
  return quant_impl(q, k, v, q8, k8, v8, scales, signs, B, Hq, Hkv, N, d, 0.f, ws, ws_bytes, stream);
}

attn_status_t attn_rope_hadamard_quant_fp8(const void* q, const void* k, const void* v, void* q8,
                                           void* k8, void* v8, float* scales, const int8_t* signs,
                                           int B, int Hq, int Hkv, int N, int d, float rope_base,
                                           void* ws, size_t ws_bytes, void* stream) {
  if (!(std::isfinite(rope_base) && rope_base > 1.f)) return ATTN_ERR_INVALID_ARG;
  return quant_impl(q, k, v, q8, k8, v8, scales, signs, B, Hq, Hkv, N, d, rope_base, ws, ws_bytes, stream);
}

attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* scales,
                           void* o, float* lse, int B, int Hq, int Hkv, int N, int d, float scale,
                           const attn_mods_t* mods, void* ws, size_t ws_bytes, void* stream) {
  attn_status_t st;
  if ((st = check_shape(B, Hq, Hkv, N, d, true)) != ATTN_OK) return st;
  if ((st = check_tensors({q8, k8, v8, o})) != ATTN_OK) return st;
  if (lse == nullptr || scales == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(scales, 4)) return ATTN_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_mods(mods)) != ATTN_OK) return st;
  const size_t need = attn_workspace_size(ATTN_OP_FWD_FP8, B, Hq, Hkv, N, d, mods);
  if ((st = check_ws(ws, ws_bytes, need)) != ATTN_OK) return st;
  int* status = nullptr;
  if ((st = device_state(&status)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  Fp8Launch L{};
  L.p = make_params(B, Hq, Hkv, N, scale, mods, status);
  if (!make_map(&L.tq, q8, true, d, N, (long long)B * Hq) ||
      !make_map(&L.tk, k8, true, d, N, (long long)B * Hkv) ||
      !make_map(&L.tv, v8, true, d, N, (long long)B * Hkv))
    return ATTN_ERR_CUDA;
  L.scales = scales;
  L.o = o;
  L.lse = lse;
  if ((st = prepare_mods(L.p, static_cast<uint8_t*>(ws), s)) != ATTN_OK) return st;
  return cuda_status(launch_fwd_fp8(L, has_score_mods(L.p.flags), needs_map(L.p.flags), s));
}

attn_status_t attn_fwd_paged(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, int num_blocks, void* o, float* lse, int B,
                             int Hq, int Hkv, int N, int d, float scale, const attn_mods_t* mods,
                             void* ws, size_t ws_bytes, void* stream) {
  attn_status_t st;
  if ((st = check_shape(B, Hq, Hkv, N, d, false)) != ATTN_OK) return st;
  if ((st = check_tensors({q, k_cache, v_cache, o})) != ATTN_OK) return st;
  if (lse == nullptr || block_table == nullptr || num_blocks < 1) return ATTN_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(block_table, 4)) return ATTN_ERR_UNSUPPORTED;
  if (N % 16 != 0) return ATTN_ERR_UNSUPPORTED;
  if ((long long)num_blocks * Hkv >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_mods(mods)) != ATTN_OK) return st;
  const size_t need = attn_workspace_size(ATTN_OP_FWD, B, Hq, Hkv, N, d, mods);
  if ((st = check_ws(ws, ws_bytes, need)) != ATTN_OK) return st;
  int* status = nullptr;
  if ((st = device_state(&status)) != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  FwdLaunch L{};
  L.p = make_params(B, Hq, Hkv, N, scale, mods, status);
  if (!make_map(&L.tq, q, false, d, N, (long long)B * Hq) ||
      !make_paged_map(&L.tk, k_cache, d, (long long)num_blocks * Hkv) ||
      !make_paged_map(&L.tv, v_cache, d, (long long)num_blocks * Hkv))
    return ATTN_ERR_CUDA;
  L.o = o;
  L.lse = lse;
  L.p.block_table = block_table;
  L.p.kv_blocks = num_blocks;
  L.p.bt_stride = N / 16;
  if ((st = prepare_mods(L.p, static_cast<uint8_t*>(ws), s)) != ATTN_OK) return st;
  return cuda_status(launch_fwd_bf16(L, d, has_score_mods(L.p.flags), needs_map(L.p.flags), s));
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int q_len, int max_blocks, int d,
                                  const attn_mods_t* mods) {
  if (max_blocks < 1 || max_blocks > (1 << 26)) return 0;
  const int N = 16 * max_blocks;
  return check_decode(B, Hq, Hkv, q_len, N, 1, d, mods) == ATTN_OK ? decode_ws_bytes(B, Hq, Hkv, q_len, N, d) : 0;
}

attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                                int num_blocks, void* o, float* lse, int B, int Hq, int Hkv, int q_len,
                                int d, float scale, const attn_mods_t* mods, void* ws, size_t ws_bytes,
                                void* stream) {
  attn_status_t st;
  if (max_blocks < 1 || max_blocks > (1 << 26)) return max_blocks < 1 ? ATTN_ERR_INVALID_ARG : ATTN_ERR_UNSUPPORTED;
  const int N = 16 * max_blocks;
  if ((st = check_decode(B, Hq, Hkv, q_len, N, num_blocks, d, mods)) != ATTN_OK) return st;
  if ((st = check_tensors({q, k_cache, v_cache, o})) != ATTN_OK) return st;
  if (lse == nullptr || block_table == nullptr || seqlens == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned(lse, 4) || !aligned(block_table, 4) || !aligned(seqlens, 4)) return ATTN_ERR_UNSUPPORTED;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, decode_ws_bytes(B, Hq, Hkv, q_len, N, d))) != ATTN_OK) return st;
  int* status = nullptr;
  if ((st = device_state(&status)) != ATTN_OK) return st;
  const int sms = sm_count();
  if (sms < 1) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const int G = Hq / Hkv;
  const DecodeSplit sp = decode_split(B, Hkv, N);
  DecodeLaunch L{};
  {  // Q as [B*Hkv, G*q_len, d]: one box holds the G query heads x q_len tokens of a KV head
    auto enc = encode_fn();
    if (!enc) return ATTN_ERR_CUDA;
    const int R = G * q_len;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)R, (cuuint64_t)B * Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)R * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)R, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&L.tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return ATTN_ERR_CUDA;
  }
  if (!make_paged_map(&L.tk, k_cache, d, (long long)num_blocks * Hkv) ||
      !make_paged_map(&L.tv, v_cache, d, (long long)num_blocks * Hkv))
    return ATTN_ERR_CUDA;
  L.o = o;
  L.lse = lse;
  DecodeParams& p = L.p;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.q_len = q_len;
  p.d = d;
  p.bt_stride = max_blocks;
  p.kv_blocks = num_blocks;
  p.ct = sp.ct;
  p.max_chunks = sp.max_chunks;
  p.scale_log2 = scale * LOG2E;
  p.flags = mod_flags(mods) & (ATTN_MOD_WINDOW | ATTN_MOD_SOFTCAP | ATTN_MOD_ALIBI);
  p.window = (p.flags & ATTN_MOD_WINDOW) ? mods->window : 0;
  const float cap = (p.flags & ATTN_MOD_SOFTCAP) ? mods->softcap : 1.0f;
  p.sc_in = scale / cap;
  p.sc_out = cap * LOG2E;
  p.slopes = (p.flags & ATTN_MOD_ALIBI) ? mods->alibi_slopes : nullptr;
  p.block_table = block_table;
  p.seqlens = seqlens;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.wait_ns = g_wait_ns.load();
  p.seq_info = reinterpret_cast<int4*>(w);
  p.n_items = reinterpret_cast<int*>(w + decode_info_bytes(B) - 256);
  const size_t rows = (size_t)B * Hq * q_len * sp.max_chunks;
  p.o_part = reinterpret_cast<float*>(w + decode_info_bytes(B));
  p.lse_part = reinterpret_cast<float*>(w + decode_info_bytes(B) + round_up(rows * d * sizeof(float), 256));
  p.status = status;
  const long long items = (long long)B * Hkv * sp.max_chunks;
  L.grid = (int)(items < sms ? items : sms);
  return cuda_status(launch_decode(L, has_score_mods(p.flags), s));
}

attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int32_t* cu_seqlens, int n_seqs, int Hq, int Hkv, int total, int d,
                              float scale, const attn_mods_t* mods, void* ws, size_t ws_bytes,
                              void* stream) {
  attn_status_t st;
  if ((st = check_tensors({q, k, v, o})) != ATTN_OK) return st;
  if (lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  attn_mods_t m;
  if ((st = varlen_setup(cu_seqlens, n_seqs, Hq, Hkv, total, d, mods, ws, ws_bytes, false, &m, stream)) !=
      ATTN_OK)
    return st;
  const size_t head = varlen_ids_bytes(total);
  return attn_fwd(q, k, v, o, lse, 1, Hq, Hkv, total, d, scale, &m, static_cast<uint8_t*>(ws) + head,
                  ws_bytes - head, stream);
}

attn_status_t attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              const int32_t* cu_seqlens, int n_seqs, int Hq, int Hkv, int total, int d,
                              float scale, const attn_mods_t* mods, void* ws, size_t ws_bytes,
                              void* stream) {
  attn_status_t st;
  if ((st = check_tensors({q, k, v, o, dout, dq, dk, dv})) != ATTN_OK) return st;
  if (lse == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  attn_mods_t m;
  if ((st = varlen_setup(cu_seqlens, n_seqs, Hq, Hkv, total, d, mods, ws, ws_bytes, true, &m, stream)) !=
      ATTN_OK)
    return st;
  const size_t head = varlen_ids_bytes(total);
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, 1, Hq, Hkv, total, d, scale, &m,
                  static_cast<uint8_t*>(ws) + head, ws_bytes - head, stream);
}

attn_status_t attn_block_map(const attn_mods_t* mods, int B, int N, uint8_t* map, void* stream) {
  attn_status_t st;
  if (B < 1 || N < 1 || map == nullptr) return ATTN_ERR_INVALID_ARG;
  if ((st = check_mods(mods)) != ATTN_OK) return st;
  if ((long long)B * n_tiles(N) * n_tiles(N) >= (1ll << 31)) return ATTN_ERR_UNSUPPORTED;
  int* status = nullptr;
  if ((st = device_state(&status)) != ATTN_OK) return st;
  AttnParams p = make_params(B, 1, 1, N, 1.0f, mods, status);
  return cuda_status(launch_block_map(p, map, static_cast<cudaStream_t>(stream)));
}

attn_status_t attn_test_hooks(unsigned long long wait_limit_ns, int stall) {
  if (stall & ~(ATTN_STALL_FWD | ATTN_STALL_BWD)) return ATTN_ERR_INVALID_ARG;
  g_wait_ns.store(wait_limit_ns == 0 ? ATTN_WAIT_TIMEOUT_NS : wait_limit_ns);
  g_stall.store(stall);
  return ATTN_OK;
}

attn_status_t attn_status(void* stream) {
  int* status = nullptr;
  attn_status_t st = device_state(&status);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  switch (h) {
    case 0: return ATTN_OK;
    case DEV_ERR_TIMEOUT: return ATTN_ERR_TIMEOUT;
    default: return ATTN_ERR_BOUNDS;
  }
}

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape, head size or alignment";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA call or kernel launch failed";
    case ATTN_ERR_DEVICE: return "current device is not an sm_103 GPU";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_BOUNDS: return "device index check failed";
    default: return "unknown status";
  }
}

}  // extern "C"
