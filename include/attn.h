/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact tiled attention library.
 *
 * What the library computes.  Exact softmax attention, in tiles, without ever
 * storing the N x N score matrix:
 *   O = softmax(mods(scale * Q K^T), masked) V,   LSE = log sum exp of each row.
 * The tiled method reaches the plain definition exactly (up to rounding
 * order): "FlashAttention-2 (FR)", opening paragraph and section "Contexte"
 * (tiles in on-chip SRAM, linear memory, identical result); the FlashAttention-3
 * digest, section "Rappel du fonctionnement de FlashAttention" (tiling plus
 * softmax rescaling gives the exact output; the backward recomputes instead of
 * storing).  The mods are the FlexAttention variants named on the
 * FlexAttention/FA4 page (ALiBi, sliding window, document masking,
 * soft-capping), here a fixed set of flags with runtime scalars in place of a
 * Python JIT, and GQA as in the Hacker News thread of the FlashAttention-3
 * digest.  The FP8 forward with Hadamard incoherent processing follows the
 * same digest, section "Basse précision FP8 et incoherent processing".
 *
 * Conventions shared by every call
 * --------------------------------
 * Layout   : contiguous [B, H, N, d] row-major; Q/O/dO/dQ have H = Hq heads,
 *            K/V/dK/dV have H = Hkv heads; query head hq reads KV head
 *            hq / (Hq / Hkv).  LSE is fp32 [B, Hq, N], natural log.
 * Types    : Q, K, V, O, dO, dQ, dK, dV are bf16; FP8 tensors are e4m3.
 * Sizes    : d in {64, 128} (FP8: d = 128); N >= 1 (backward: N <= 131072); Hq % Hkv == 0;
 *            B * max(Hq, Hkv) * N < 2^31.
 * Pointers : device pointers, 16-byte aligned.  The caller owns every
 *            buffer, including the workspace; the library allocates nothing
 *            per call (it keeps only a device status word).
 * Streams  : every call is asynchronous on `stream` (a cudaStream_t; NULL is
 *            the legacy default stream).  The device current for the calling
 *            thread must own the buffers.
 * Errors   : argument problems are reported synchronously, before anything is
 *            launched (ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
 *            ATTN_ERR_WORKSPACE); a failed launch gives ATTN_ERR_CUDA.  Errors
 *            found on the device (a pipeline wait that timed out, a bounds
 *            check) are recorded in the status word and returned by
 *            attn_status().  There is no fallback path of any kind.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad mod scalar */
  ATTN_ERR_UNSUPPORTED = 2,  /* d not supported, Hq % Hkv != 0, misaligned pointer */
  ATTN_ERR_WORKSPACE = 3,    /* workspace missing or smaller than attn_workspace_size() */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call or a launch failed */
  ATTN_ERR_DEVICE = 5,       /* the current device is not an sm_103 GPU */
  ATTN_ERR_TIMEOUT = 6,      /* (device) a pipeline wait gave up after its time limit */
  ATTN_ERR_BOUNDS = 7        /* (device) an index check failed */
} attn_status_t;

/* Mod flags.  The mask is the AND of the enabled parts. */
enum {
  ATTN_MOD_CAUSAL = 1u << 0,  /* allowed iff j <= i */
  ATTN_MOD_WINDOW = 1u << 1,  /* allowed iff i - j < window */
  ATTN_MOD_DOC = 1u << 2,     /* allowed iff doc_ids[b][i] == doc_ids[b][j] */
  ATTN_MOD_SOFTCAP = 1u << 3, /* score x -> softcap * tanh(x / softcap), applied to scale*q.k */
  ATTN_MOD_ALIBI = 1u << 4,   /* score x -> x - slope[hq] * (i - j), after the soft-cap */
  ATTN_MOD_BWD_FP8 = 1u << 5  /* attn_bwd only: mixed e4m3 backward (see attn_bwd); ignored elsewhere */
};

/* FlexAttention variants as a fixed set of flags plus runtime scalars
 * (FlexAttention/FA4 page, opening paragraphs and "Limitations actuelles":
 * no recompilation when a scalar changes). */
typedef struct {
  uint32_t flags;             /* OR of ATTN_MOD_* */
  int32_t window;             /* ATTN_MOD_WINDOW: >= 1 */
  float softcap;              /* ATTN_MOD_SOFTCAP: > 0 */
  const int32_t* doc_ids;     /* ATTN_MOD_DOC: device int32 [B, N] */
  const float* alibi_slopes;  /* ATTN_MOD_ALIBI: device fp32 [Hq], or NULL for 2^(-8(h+1)/Hq) */
} attn_mods_t;

/* Operations for attn_workspace_size().  For the two varlen operations pass
 * B = 1 and N = total (the packed row count); for the paged decode step pass
 * N = 16 * max_blocks (the longest sequence the block table can hold). */
enum {
  ATTN_OP_FWD = 0,
  ATTN_OP_BWD = 1,
  ATTN_OP_FWD_FP8 = 2,
  ATTN_OP_QUANT_FP8 = 3,
  ATTN_OP_FWD_VARLEN = 4,
  ATTN_OP_BWD_VARLEN = 5,
  ATTN_OP_DECODE_PAGED = 6
};

/* Block-map tile classes (128 x 128 tiles). */
enum { ATTN_TILE_SKIP = 0, ATTN_TILE_PARTIAL = 1, ATTN_TILE_FULL = 2 };

/*
 * Bytes of caller-provided workspace an operation needs (0 when none).
 * mods may be NULL (no mods).  Returns 0 for invalid arguments as well; the
 * operation itself then reports the argument error.
 */
size_t attn_workspace_size(int op, int B, int Hq, int Hkv, int N, int d, const attn_mods_t* mods);

/*
 * Forward pass: O (bf16 [B,Hq,N,d]) and LSE (fp32 [B,Hq,N]) from Q, K, V.
 * The method: the FlashAttention-3 digest, "Rappel du fonctionnement de
 * FlashAttention" (tiles, online softmax rescale, never materialising S) and
 * "Chevauchement de GEMM et softmax grâce à l'asynchronisme" (GEMMs on the
 * tensor cores overlapped with the exponentials).  Rows with no allowed key
 * get O = 0 and LSE = -inf.  Fully masked 128 x 128 tiles are skipped
 * (block sparsity, FlexAttention/FA4 page, "Limitations actuelles").
 * scale : multiplier of q.k (typically 1/sqrt(d)), finite and > 0.
 * ws    : workspace of attn_workspace_size(ATTN_OP_FWD, ...) bytes (may be
 *         NULL when that size is 0; window / document mods need one for the
 *         block map, its per-tile ranges and the document runs).
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int Hq, int Hkv, int N, int d, float scale,
                       const attn_mods_t* mods, void* ws, size_t ws_bytes, void* stream);

/*
 * Backward pass: dQ (bf16 [B,Hq,N,d]), dK and dV (bf16 [B,Hkv,N,d]) from Q, K,
 * V, the forward's O and LSE, and dO.  P is recomputed from LSE (the
 * FlashAttention-3 digest, "Rappel du fonctionnement": tiling and
 * recomputation).  The result is bitwise reproducible from run to run: no
 * floating-point atomics (contrast the FlexAttention/FA4 page, "Limitations
 * actuelles": nondeterministic backward with block sparsity).  dK/dV of a KV
 * head sum over its query heads (GQA).  Two implementations, chosen by the
 * mods:
 *  - causal with window / document parts, d = 128: one kernel computes dK, dV
 *    and the dQ partials of every tile pair (5 GEMMs); each dQ partial is
 *    rounded to an integer multiple of its row's quantum -- a power of two
 *    chosen from a bound on |dQ| -- and summed as int32, so the sum does not
 *    depend on the order the partials arrive in;
 *  - otherwise: every dQ, dK and dV tile is accumulated by one CTA over its
 *    partner tiles in ascending order (two kernels, 7 GEMMs per tile pair).
 * ATTN_MOD_BWD_FP8 selects a mixed-precision form of the second one (the
 * FlashAttention-3 digest, "Basse précision FP8 et incoherent processing",
 * describes FP8 for the forward; this extends it to the two backward GEMMs
 * whose operands behave like the forward's): dO and V are rounded to e4m3
 * with one scale amax/448 per (batch, KV head) each, and in the dK/dV kernel
 * dP = dO V^T and dV = P^T dO run as e4m3 GEMMs (P scaled by 256 before
 * rounding); dS, dK = dS^T Q and the whole dQ kernel stay bf16.  Less
 * accurate than the bf16 backward (tests/test_gpu_bwd_fp8.py bounds the
 * error).  Needs d = 128 and no mod other than ATTN_MOD_CAUSAL, else
 * ATTN_ERR_UNSUPPORTED.  Also bitwise reproducible.
 * ws : workspace of attn_workspace_size(ATTN_OP_BWD, ...) bytes: the row
 *      statistics {LSE log2(e), D = rowsum(dO * O)} of every query row;
 *      with window/document mods, the block map, its per-tile ranges and
 *      (documents) the document run of every position; for the one-kernel
 *      form, the dQ quanta, K/V bounds and the int32 dQ sums (4 d bytes per
 *      query row, rows padded to whole 128-row tiles); with ATTN_MOD_BWD_FP8,
 *      the e4m3 copies of dO and V (d bytes per row) and their scales.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv,
                       int B, int Hq, int Hkv, int N, int d, float scale,
                       const attn_mods_t* mods, void* ws, size_t ws_bytes, void* stream);

/*
 * attn_bwd, plus timing: events[0..3] are cudaEvent_t handles created by the
 * caller, recorded on `stream`.  Two-kernel form: events[0] before the
 * row-sum kernel, events[1] before the dK/dV kernel, events[2] before the dQ
 * kernel, events[3] after it.  One-kernel form: events[0] before the bound and
 * row-sum kernels, events[1] before the main kernel, events[2] before the dQ
 * conversion, events[3] after it.  (The block-map kernels, when the mods need
 * them, run before events[0].)  Measurement aid for "profiler l'exécution" (the kernel
 * fusion page, "Fusion et CUDA Graphs avec torch.compile"); results are
 * identical to attn_bwd.  events must not be NULL.
 */
attn_status_t attn_bwd_profiled(const void* q, const void* k, const void* v, const void* o,
                                const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int Hq, int Hkv, int N, int d, float scale,
                                const attn_mods_t* mods, void* ws, size_t ws_bytes, void* stream,
                                void* const* events);

/* Capacity, in bytes, of the fixed device scratch array of attn_bwd_noalloc. */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * attn_bwd for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point: it is a library addition.
 *
 * Who needs it: code whose device memory is owned by someone else -- a host
 * framework with its own caching allocator, or a fixed arena that other code
 * must not allocate around -- and code that must not call cudaMalloc/cudaFree
 * because those calls synchronise the device.  Such callers can still pass Q,
 * K, V, O, dO, LSE and the dQ/dK/dV outputs, but not the workspace attn_bwd
 * takes.  This variant uses instead a scratch array compiled into the library
 * (a file-scope device array of ATTN_NOALLOC_SCRATCH_BYTES, held by every GPU
 * that loads the library until the process exits).  It calls no cudaMalloc,
 * cudaFree or any other allocating routine.
 *
 * Arguments, layout and errors are those of attn_bwd, without ws/ws_bytes.
 * Limit: the workspace attn_bwd would need, attn_workspace_size(ATTN_OP_BWD,
 * ...) (8 bytes per query row with rows padded to whole 128-row tiles, plus
 * the window / document mask data, plus 4 d + 4 bytes per padded query row
 * when the one-kernel form runs), must fit in ATTN_NOALLOC_SCRATCH_BYTES;
 * otherwise the call returns ATTN_ERR_WORKSPACE before touching the device.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current).  Because CUDA loads
 * modules lazily, that lookup is also when the library's module is loaded on
 * the device and the array is reserved there, which can synchronise the
 * device.  Make that first call once per device at set-up time, before any
 * stream capture and outside any section that must not synchronise; later
 * calls only read the cached address.
 * Sharing: every call uses the same array, which keeps the last call's
 * contents.  Each call overwrites all of the scratch it reads (nothing there
 * has to start at zero), so consecutive calls are fine; calls that overlap on
 * the GPU (different streams, or host threads without ordering) race on the
 * array and give wrong results.
 */
attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                               const void* dout, const float* lse, void* dq, void* dk, void* dv,
                               int B, int Hq, int Hkv, int N, int d, float scale,
                               const attn_mods_t* mods, void* stream);

/*
 * Forward over a paged K/V cache (the inference layout of the kernel fusion
 * page's serving discussion: keys and values in fixed blocks of 16 rows
 * addressed through a block table).  Same computation and mods as attn_fwd,
 * with K and V read through the table instead of from [B, Hkv, N, d].
 * k_cache, v_cache : bf16 [num_blocks, Hkv, 16, d]; block j of head h holds
 *                    16 consecutive key (value) rows of that head.
 * block_table      : device int32 [B, N / 16]: key rows [16 t, 16 t + 16) of
 *                    batch row b are block block_table[b][t]; an index outside
 *                    [0, num_blocks) reads zeros.
 * N must be a multiple of 16 (ATTN_ERR_UNSUPPORTED otherwise); d = 64 or 128;
 * workspace as attn_fwd (ATTN_OP_FWD).
 */
attn_status_t attn_fwd_paged(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, int num_blocks, void* o, float* lse, int B,
                             int Hq, int Hkv, int N, int d, float scale, const attn_mods_t* mods,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Decode step over a paged K/V cache ("Les kernels d'attention rapide et la
 * fusion d'opérateurs accélèrent les modèles d'IA", section "Attention de
 * type FlashAttention et attention paginée": the cache grows one token per
 * step, in fixed blocks of 16 tokens mapped through a block table).  The
 * q_len newest tokens of each sequence (1 for plain decoding; several, e.g.
 * draft tokens to verify) attend to the cached keys of their sequence, causal
 * among themselves.
 * q           : bf16 [B, Hq, q_len, d]; token t of sequence b is at position
 *               L_b - q_len + t.
 * k_cache,
 * v_cache     : bf16 [num_blocks, Hkv, 16, d], as for attn_fwd_paged.
 * block_table : device int32 [B, max_blocks]: cached rows [16 t, 16 t + 16) of
 *               sequence b are block block_table[b][t]; only the first
 *               ceil(L_b / 16) entries of a row are read.
 * seqlens     : device int32 [B]: L_b, the cached tokens of sequence b (the new
 *               ones included), 0 <= L_b <= 16 * max_blocks.  A token with no
 *               key (L_b = 0, or a position below 0) gets O = 0, LSE = -inf.
 * o, lse      : bf16 [B, Hq, q_len, d] and fp32 [B, Hq, q_len] (natural log),
 *               written.
 * mods        : CAUSAL is implied (accepted, no effect); WINDOW keeps keys with
 *               i - j < window for the token at position i; SOFTCAP and ALIBI as
 *               in attn_fwd; DOC is ATTN_ERR_UNSUPPORTED.
 * ws          : attn_decode_workspace_size(B, Hq, Hkv, q_len, max_blocks, d,
 *               mods) bytes: per-chunk partial outputs.
 * Requirements: d = 64 or 128, Hq % Hkv == 0, (Hq / Hkv) * q_len <= 128 (else
 * ATTN_ERR_UNSUPPORTED).  Device-side: a length outside [0, 16 * max_blocks]
 * or a table entry outside [0, num_blocks) is reported as ATTN_ERR_BOUNDS by
 * attn_status (the call then leaves O and LSE unspecified).
 * Asynchronous on `stream`; the caller owns every buffer.
 */
attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int max_blocks, const int32_t* seqlens,
                                int num_blocks, void* o, float* lse, int B, int Hq, int Hkv, int q_len,
                                int d, float scale, const attn_mods_t* mods, void* ws, size_t ws_bytes,
                                void* stream);

/* Workspace bytes of attn_decode_paged (0 for invalid arguments).
 * attn_workspace_size(ATTN_OP_DECODE_PAGED, B, Hq, Hkv, 16 * max_blocks, d,
 * mods) is the same for q_len = 1. */
size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int q_len, int max_blocks, int d,
                                  const attn_mods_t* mods);

/*
 * Packed variable-length sequences: n_seqs sequences stored back to back along
 * the row axis, attending only within themselves -- the unpadded form of the
 * document mask (FlexAttention/FA4 page, opening paragraphs: document
 * masking among the mods it accelerates).  Sequence s occupies rows
 * [cu_seqlens[s], cu_seqlens[s+1]) of every head.
 * Layout: Q, O, dO, dQ [1, Hq, total, d]; K, V, dK, dV [1, Hkv, total, d];
 *         LSE [1, Hq, total]; all bf16 except LSE (fp32).
 * cu_seqlens : device int32 [n_seqs + 1]: 0 = cu_seqlens[0] <= cu_seqlens[1]
 *              <= ... <= cu_seqlens[n_seqs] = total (not checked on the host;
 *              a malformed array changes which rows attend to which, never
 *              which memory is touched).
 * mods       : causal / window / soft-cap / ALiBi as for attn_fwd, applied
 *              inside each sequence (i, j are packed row indices, so i - j is
 *              the in-sequence distance); ATTN_MOD_DOC must not be set
 *              (ATTN_ERR_INVALID_ARG): the sequences are the documents.
 * ws         : attn_workspace_size(ATTN_OP_FWD_VARLEN / ATTN_OP_BWD_VARLEN,
 *              1, Hq, Hkv, total, d, mods) bytes: the per-row sequence ids,
 *              then attn_fwd's / attn_bwd's workspace for the document mask.
 * Otherwise as attn_fwd / attn_bwd (same kernels, B = 1, N = total).
 */
attn_status_t attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                              const int32_t* cu_seqlens, int n_seqs, int Hq, int Hkv, int total,
                              int d, float scale, const attn_mods_t* mods, void* ws,
                              size_t ws_bytes, void* stream);
attn_status_t attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              const int32_t* cu_seqlens, int n_seqs, int Hq, int Hkv, int total,
                              int d, float scale, const attn_mods_t* mods, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * FP8 prologue (FlashAttention-3 digest, "Basse précision FP8 et incoherent
 * processing"): every row of Q and K is multiplied by diag(s) H / sqrt(d),
 * H the natural-order Sylvester Hadamard matrix of order d and s the +-1
 * sign vector of the row's KV head (query head hq uses signs[hq/(Hq/Hkv)]);
 * V is not rotated.  Each (b, head) tensor is then scaled by 448/amax and
 * rounded to e4m3 (nearest even, saturating).
 * signs  : device int8 [Hkv, d] of +-1, 16-byte aligned (ATTN_ERR_UNSUPPORTED
 *          otherwise), or NULL to skip the rotation (the plain-FP8 variant).
 * q8     : e4m3 [B,Hq,N,d];  k8, v8 : e4m3 [B,Hkv,N,d].
 * scales : device fp32, B*Hq + 2*B*Hkv entries: the dequantisation scales
 *          amax/448 of Q [B,Hq], then K [B,Hkv], then V [B,Hkv] (1 where a
 *          head is all zero).
 * ws     : workspace of attn_workspace_size(ATTN_OP_QUANT_FP8, ...) bytes.
 * d must be 128.
 */
attn_status_t attn_hadamard_quant_fp8(const void* q, const void* k, const void* v, void* q8,
                                      void* k8, void* v8, float* scales, const int8_t* signs,
                                      int B, int Hq, int Hkv, int N, int d, void* ws,
                                      size_t ws_bytes, void* stream);

/*
 * attn_hadamard_quant_fp8 with rotary position embedding fused in front of the
 * rotation (FlashAttention-3 digest, "Basse précision FP8 et incoherent
 * processing": the Hadamard transform can be fused with RoPE at no extra
 * cost): each Q and K row is first turned by RoPE -- row n of a head has its
 * element pairs (c, c + d/2), c < d/2, rotated by the angle
 * n * rope_base^(-2c/d) -- in the same pass, then signed, rotated and
 * quantised as above.  rope_base: finite and > 1 (e.g. 10000), else
 * ATTN_ERR_INVALID_ARG.  Other arguments, workspace and errors as
 * attn_hadamard_quant_fp8 (signs may be NULL: RoPE then quantisation only).
 */
attn_status_t attn_rope_hadamard_quant_fp8(const void* q, const void* k, const void* v, void* q8,
                                           void* k8, void* v8, float* scales, const int8_t* signs,
                                           int B, int Hq, int Hkv, int N, int d, float rope_base,
                                           void* ws, size_t ws_bytes, void* stream);

/*
 * FP8 forward: O (bf16) and LSE (fp32, of the dequantised scores) from the
 * e4m3 tensors and scales written by attn_hadamard_quant_fp8.  Q K^T runs in
 * e4m3 with fp32 accumulation, P is rounded to e4m3 for P V, and the
 * dequantisation factors are folded into the softmax scale (Q, K) and the
 * epilogue (V).  Same mods, workspace rule and errors as attn_fwd; d = 128.
 */
attn_status_t attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* scales,
                           void* o, float* lse, int B, int Hq, int Hkv, int N, int d,
                           float scale, const attn_mods_t* mods, void* ws, size_t ws_bytes,
                           void* stream);

/*
 * Block-sparsity map of the mask in mods (FlexAttention/FA4 page, "Limitations
 * actuelles": block sparsity; 128 x 128 tiles as named there).  map is device
 * uint8 [B, nT, nT], nT = ceil(N/128); entry (b, I, J) classifies rows
 * [128I, 128I+128) x columns [128J, 128J+128), counting only rows i < N:
 * ATTN_TILE_SKIP when no pair with j < N is allowed, ATTN_TILE_FULL when the
 * column range lies inside [0, N) and every pair is allowed, else
 * ATTN_TILE_PARTIAL.  Only the mask flags of mods matter.
 */
attn_status_t attn_block_map(const attn_mods_t* mods, int B, int N, uint8_t* map, void* stream);

/* Stall selectors of attn_test_hooks. */
enum { ATTN_STALL_FWD = 1, ATTN_STALL_BWD = 2 };

/*
 * Test hooks for the device-side failure path.  Every pipeline wait in the
 * kernels is bounded: a wait that runs out of time records ATTN_ERR_TIMEOUT
 * in the status word, every other wait of the grid gives up, copies and MMAs
 * in flight drain, tensor memory is released and the kernel returns, so the
 * context stays usable (the FlashAttention-3 digest's asynchronous
 * producer/consumer pipeline, "Fonctionnalités des GPU Hopper", is what these
 * waits belong to; the bound itself is this library's own).
 * wait_limit_ns : time limit of the stalled wait (below) in kernels launched
 *                 after this call; 0 restores the default (1 s).  Every other
 *                 wait keeps the default, and gives up as soon as the stalled
 *                 one has.
 * stall         : 0, or an OR of ATTN_STALL_FWD (forward kernels: the first
 *                 query tile's compute warpgroup of every CTA first waits on a
 *                 barrier that nothing completes) and ATTN_STALL_BWD (the
 *                 backward's main kernel: one compute warpgroup does the same).
 *                 A stalled kernel ends with ATTN_ERR_TIMEOUT and leaves its
 *                 outputs unspecified.  Other bits: ATTN_ERR_INVALID_ARG.
 * Process-wide settings, read when a call launches its kernels; not meant to
 * change while other threads launch.  No device work, no synchronisation.
 */
attn_status_t attn_test_hooks(unsigned long long wait_limit_ns, int stall);

/*
 * Synchronise `stream`, then return and clear the device status word
 * (ATTN_OK, ATTN_ERR_TIMEOUT or ATTN_ERR_BOUNDS), or ATTN_ERR_CUDA when the
 * synchronisation itself failed.
 */
attn_status_t attn_status(void* stream);

/* Static, human-readable name of a status code. */
const char* attn_status_string(attn_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
