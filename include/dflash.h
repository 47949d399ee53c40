/*
 * dflash.h — C ABI of libdflash.so: one DFlash block-diffusion draft step, the
 * greedy verify-accept that follows it, and the draft-KV commit, on one GB300
 * (sm_103a).
 *
 * The method (sources are web pages on DFlash, cited by title and section):
 *  - The drafter is a few-layer transformer that fills a block of B positions
 *    in ONE parallel non-causal pass; position 0 holds the last accepted token,
 *    the other positions hold the mask-token embedding; it reuses the target's
 *    embedding and lm-head (mlx-dspark v0.0.3 release notes, "Highlights").
 *  - It is conditioned on intermediate target activations, not logits
 *    (dflash-mlx summary, "What It Does").
 *  - Projections are int8 with per-output-channel fp16 scales (W8A16), Q/K get
 *    a per-head RMSNorm over head_dim values, RoPE is neox split-half
 *    (mirror-sd README, "The Story", Phases 2 and 3; "How It Works").
 *  - Verify: the target scores the block in one pass; the longest prefix on
 *    which the drafts equal the target's greedy choice is accepted and the
 *    target supplies one correction token (mirror-sd README, "How It Works",
 *    step 3; agentlens dflash-mlx, "How it works").
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers unless stated otherwise; the
 *    caller allocates and owns every buffer.  The library never allocates or
 *    frees device memory; scratch comes from a caller workspace.
 *  - fp16 and bf16 tensors are passed as uint16_t bit patterns.
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *    stream.  Every call is asynchronous and stream-ordered: it enqueues work
 *    and returns.  Accept lengths and next tokens stay on the device.
 *  - Return value: DFLASH_OK or a negative dflash_status.  Host-checkable
 *    faults (null pointers, bad sizes, unsupported shapes, workspace too
 *    small) return before anything is enqueued.  A failed kernel launch
 *    returns DFLASH_ECUDA.  Faults only the device can see (KV capacity
 *    exceeded, a token or length out of range) set bits in a device status
 *    word, skip the offending writes and never trap; read it with
 *    dflash_get_status().
 *  - Workspaces: scratch regions contain counters that must be zero before
 *    the first call; zero-fill a workspace once after allocating it.  Every
 *    call leaves them zero again.  Calls that share a workspace must not
 *    overlap on the GPU (stream order them).
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dflash_status {
  DFLASH_OK = 0,
  DFLASH_EINVAL = -1,       /* null pointer, negative or inconsistent size */
  DFLASH_EUNSUPPORTED = -2, /* shape outside what the kernels implement    */
  DFLASH_ECUDA = -3,        /* a CUDA runtime/launch error                  */
  DFLASH_ECAPACITY = -4,    /* KV cache capacity exceeded (device flag)    */
  DFLASH_EWORKSPACE = -5    /* workspace missing or too small              */
} dflash_status;

/* Bits of the device status word (dflash_get_status). */
#define DFLASH_DEV_KV_CAPACITY 0x1 /* a commit would pass `cap`: skipped   */
#define DFLASH_DEV_BAD_TOKEN 0x2   /* a token id outside [0, V): row zeroed */
#define DFLASH_DEV_BAD_LENGTH 0x4  /* len < 0 or n outside [-1, B]         */

/* Element types accepted by dflash_pack_w8a16. */
#define DFLASH_DTYPE_F32 0
#define DFLASH_DTYPE_F16 1
#define DFLASH_DTYPE_BF16 2

/* Row layouts of a packed W8A16 matrix. */
#define DFLASH_LAYOUT_PLAIN 0  /* rows in logical order                    */
#define DFLASH_LAYOUT_GATEUP 1 /* logical rows [gate F | up F]; packed so
                                  each 128-row tile holds 64 gate rows and
                                  the 64 matching up rows                  */

/* Drafter shape.  Supported: d in {64, 128}; H, nq*d, nkv*d, F, k*H multiples
 * of 128; nq a multiple of nkv; B in [2, 32]; V >= 1. */
typedef struct dflash_config {
  int32_t L;        /* drafter layers                                     */
  int32_t H;        /* hidden size                                        */
  int32_t nq, nkv;  /* query / key-value heads (GQA group = nq / nkv)     */
  int32_t d;        /* head_dim                                           */
  int32_t F;        /* SwiGLU width                                       */
  int32_t V;        /* vocabulary (rows of embedding and lm-head)         */
  int32_t B;        /* block size                                         */
  int32_t k;        /* hooked target layers: hidden rows are k*H wide     */
  int32_t mask_id;  /* token whose embedding fills block slots 1..B-1     */
  float rope_theta; /* RoPE base                                          */
  float eps;        /* RMSNorm epsilon                                    */
} dflash_config;

/* A packed weight matrix, int8 or int4 codes with fp16 scales.
 *  bits 8 (or 0), output of dflash_pack_w8a16: W[N][K] = q[N][K] * s[N];
 *    `q` is N*K bytes in the library's tiled layout, `s` is N fp16 scales in
 *    logical row order.
 *  bits 4, output of dflash_pack_w4a16: W[N][K] = q[N][K] * s[N][K/128]
 *    with q in [-7, 7]; `q` is dflash_w4a16_packed_bytes(N, K) bytes of
 *    tiles that carry their own scales, so `s` is not read and may be NULL.
 * Borrowed device pointers.  All matrices of one dflash_weights use the same
 * `bits`. */
typedef struct dflash_w8 {
  const void* q;
  const uint16_t* s;
  int64_t N, K;
  int32_t layout; /* DFLASH_LAYOUT_* */
  int32_t bits;   /* 8 (or 0) or 4 */
} dflash_w8;

/* Drafter weights.  qkv/o/gu/down point to HOST arrays of L descriptors
 * (read during the call); every tensor they describe is on the device.
 *   qkv[l]:  N = (nq + 2 nkv) d, K = H; rows q heads | k heads | v heads
 *   o[l]:    N = H, K = nq d
 *   gu[l]:   N = 2F, K = H, layout DFLASH_LAYOUT_GATEUP
 *   down[l]: N = H, K = F
 *   fc:      N = H, K = k H  (target hidden -> drafter width)
 * Gammas are fp32; embed and lm_head are the target's bf16 [V][H] tables. */
typedef struct dflash_weights {
  dflash_config cfg;
  dflash_w8 fc;
  const dflash_w8* qkv;
  const dflash_w8* o;
  const dflash_w8* gu;
  const dflash_w8* down;
  const float* gamma_hid;   /* [H]    norm after fc                        */
  const float* gamma_in;    /* [L][H] pre-attention norm                 */
  const float* gamma_post;  /* [L][H] pre-FFN norm                       */
  const float* gamma_q;     /* [L][d] per-head Q norm                    */
  const float* gamma_k;     /* [L][d] per-head K norm                    */
  const float* gamma_final; /* [H]    norm before the lm-head            */
  const uint16_t* embed;    /* bf16 [V][H]                               */
  const uint16_t* lm_head;  /* bf16 [V][H]                               */
} dflash_weights;

/* Draft KV cache: K after Q/K-norm and RoPE, V as projected, fp16,
 * k and v each [L][b][nkv][cap][d]; len[b] (device int32) = committed rows of
 * each sequence.  Context row j of a sequence sits at position j. */
typedef struct dflash_kv {
  uint16_t* k;
  uint16_t* v;
  int32_t* len;
  int32_t b;   /* sequences */
  int32_t cap; /* rows per sequence; at most 2^24 - 64 (positions are carried
                  exactly in fp32 by the RoPE epilogues), else the calls that
                  take a dflash_kv return DFLASH_EUNSUPPORTED */
} dflash_kv;

/* Library version string (static storage). */
DFLASH_API const char* dflash_version(void);

/* Human-readable name of a dflash_status (static storage). */
DFLASH_API const char* dflash_status_string(int32_t status);

/* Workspace bytes for dflash_draft_block, dflash_kv_commit and
 * dflash_commit_draft_block with b sequences and up to rows_per_seq hidden
 * rows per commit call (use B for the decode loop).  One workspace serves all
 * three calls.  Returns DFLASH_EINVAL / DFLASH_EUNSUPPORTED for a bad
 * config. */
DFLASH_API int32_t dflash_workspace_size(const dflash_config* cfg, int32_t b,
                              int32_t rows_per_seq, size_t* bytes);

/* W8A16 packing (mirror-sd README, "The Story", Phase 3: int8 weights with
 * per-output-channel fp16 scales).  w: device [N][K] of w_dtype.
 *   s[n] = fp16_rne(absmax_n / 127)            (division in fp32)
 *   q[n][k] = clamp(rint(w[n][k] / s[n]), -127, 127), 0 where s[n] == 0
 * and writes q in the tiled layout the GEMM streams (q_out: N*K bytes, 16-byte
 * aligned) and s in logical order (s_out: N fp16).  N, K multiples of 128;
 * layout DFLASH_LAYOUT_GATEUP needs N/2 a multiple of 64.  Offline, once per
 * weight; not on the timed path. */
DFLASH_API int32_t dflash_pack_w8a16(const void* w, int32_t w_dtype, int64_t N, int64_t K,
                          int32_t layout, void* q_out, uint16_t* s_out,
                          void* stream);

/* Bytes of the packed tiles of an int4 matrix: (N/128)(K/128) tiles of
 * 8448 bytes (8192 of codes, then the tile's 128 rows' fp16 scales).
 * N, K multiples of 128 (else DFLASH_EUNSUPPORTED). */
DFLASH_API int32_t dflash_w4a16_packed_bytes(int64_t N, int64_t K, size_t* bytes);

/* Symmetric int4 quantisation with one scale per row and 128-column group
 * (W4A16; a 4-bit drafter is the default of mlx-dspark v0.0.3, release
 * notes "Notes"; the symmetric [-7, 7] format and the group size of 128 are
 * this library's choice) of w[N][K] (device, w_dtype DFLASH_DTYPE_*):
 *   s[n][g] = fp16_rn(max_{k in group g} |w[n][k]| / 7)  (fp32 division)
 *   q[n][k] = clamp(rint(w[n][k] / s[n][k/128]), -7, 7)  (fp32 division;
 *             0 where the scale is 0)
 * q_out (16-byte aligned, dflash_w4a16_packed_bytes(N, K) bytes) receives
 * the tiles, s_out (device, N*K/128 fp16) the scales in logical order; both
 * caller-owned.  s_out is only a by-product once packing has finished (the
 * tiles hold a copy).  Layouts, shape limits and errors as dflash_pack_w8a16.
 * Asynchronous on `stream`. */
DFLASH_API int32_t dflash_pack_w4a16(const void* w, int32_t w_dtype, int64_t N, int64_t K,
                          int32_t layout, void* q_out, uint16_t* s_out,
                          void* stream);

/* Workspace bytes for dflash_w8a16_linear (0: split-K partial sums are
 * reduced on chip, so the call needs no scratch; ws may be NULL). */
DFLASH_API int32_t dflash_w8a16_linear_workspace_size(int64_t M, int64_t N, int64_t K,
                                           size_t* bytes);

/* The W8A16 projection alone (the kernel every drafter matmul runs on):
 * y[m][n] = s[n] * sum_k x[m][k] q[n][k] (int4: sum over groups g of
 * s[n][g] * sum_{k in g} x[m][k] q[n][k]) with fp16 activations x [M][K]
 * (16-byte aligned), fp32 accumulation, fp32 output y [M][N] in logical row
 * order (mirror-sd README, "The Story", Phase 3).  M in [1, 4096]. */
DFLASH_API int32_t dflash_w8a16_linear(const dflash_w8* w, const uint16_t* x, int64_t M,
                            float* y, void* ws, size_t ws_bytes, void* stream);

/* One draft step for b = kv->b sequences (mlx-dspark v0.0.3, "Highlights";
 * mirror-sd README, "How It Works"):
 *   x[slot 0] = embed[last_tok], x[slots 1..B-1] = embed[mask_id];
 *   slot i of sequence j sits at position len[j] + i;
 *   per layer: u = RMSNorm(x; gamma_in); [q|k|v] = W8(qkv) u;
 *              q, k = RoPE(per-head RMSNorm(q|k)); attention of the block's
 *              queries over [context K/V (len[j] rows) || block K/V], no mask;
 *              x += W8(o) attn; u = RMSNorm(x; gamma_post);
 *              x += W8(down)(silu(gate) * up), [gate|up] = W8(gu) u;
 *   h = RMSNorm(x[slots 1..B-1]; gamma_final) (rounded to bf16);
 *   draft[j][i] = argmax_v h[i] . lm_head[v] (lowest index on ties).
 * last_tok: [b] int32.  draft_out: [b][B-1] int32.
 * hidden_out (nullable): [b][B-1][H] fp32, h before bf16 rounding.
 * logits_out (nullable): [b][B-1][V] fp32.
 * When both are null the lm-head's input is bf16(x * gamma_final) without
 * the final RMSNorm's positive per-row factor, which leaves each row's
 * argmax unchanged (up to bf16 rounding of near ties).
 * The cache is read, never written: the block's own K/V live in the
 * workspace, so rejecting drafts needs no cache rollback. */
DFLASH_API int32_t dflash_draft_block(const dflash_weights* w, const dflash_kv* kv,
                           const int32_t* last_tok, int32_t* draft_out,
                           float* hidden_out, float* logits_out, void* ws,
                           size_t ws_bytes, void* stream);

/* Workspace bytes for dflash_lmhead_argmax with M rows. */
DFLASH_API int32_t dflash_lmhead_workspace_size(int64_t M, size_t* bytes);

/* idx_out[m] = argmax_v sum_k h[m][k] * w[v][k] (bf16 inputs, fp32
 * accumulation, lowest index on ties), the drafter's shared lm-head
 * (mlx-dspark v0.0.3, "Highlights").  h: [M][H] bf16, w: [V][H] bf16,
 * M in [1, 128], H a multiple of 64, rows 16-byte aligned.
 * maxlogit_out (nullable): [M] fp32.  logits_out (nullable): [M][V] fp32. */
DFLASH_API int32_t dflash_lmhead_argmax(const uint16_t* h, const uint16_t* w, int64_t M,
                             int64_t V, int64_t H, int32_t* idx_out,
                             float* maxlogit_out, float* logits_out, void* ws,
                             size_t ws_bytes, void* stream);

/* Workspace bytes for dflash_verify_accept. */
DFLASH_API int32_t dflash_verify_workspace_size(int32_t b, int32_t R, int64_t V,
                                     size_t* bytes);

/* Greedy verify-accept (mirror-sd README, "How It Works", step 3; agentlens
 * dflash-mlx, "How it works").  For each sequence j:
 *   a_r = argmax_v logits[j][r][v]  (fp32, lowest index on ties)
 *   n   = number of leading i < D with draft[j][i] == a_i
 *   corr = a_n if n < R else -1
 *   emitted[j] = draft[j][0..n) ++ [corr], padded with -1 to R entries
 *   next_tok[j] = last emitted token (slot 0 of the next block)
 * logits: [b][R][V] fp32; draft: [b][D] int32, 1 <= D <= R.
 * n_out, corr_out, next_tok_out: [b] int32 (next_tok_out nullable);
 * emitted_out: [b][R] int32 (nullable).  n_out feeds dflash_kv_commit. */
DFLASH_API int32_t dflash_verify_accept(const float* logits, const int32_t* draft,
                             int32_t b, int32_t R, int32_t D, int64_t V,
                             int32_t* n_out, int32_t* corr_out,
                             int32_t* emitted_out, int32_t* next_tok_out,
                             void* ws, size_t ws_bytes, void* stream);

/* Allocation-free verify-accept.  The pages describe no counterpart to this call;
 * it exists for callers that cannot allocate device memory themselves (for
 * example code running inside a stream capture that forbids allocation,
 * embedders whose memory is fully pre-reserved by another allocator, or
 * plain C hosts without a CUDA allocator wrapper).  It computes exactly what
 * dflash_verify_accept computes, with the same arguments minus the
 * workspace: its scratch is a fixed 64 KiB array inside the library's device
 * image, resident on every GPU that loads the library until the process
 * exits.  Shapes whose scratch would exceed that (more than 1024 sequences,
 * or b*R*slices keys beyond the array) return DFLASH_EWORKSPACE.  The first
 * call on a device resolves the array's device address (cudaGetSymbolAddress
 * with that device current) and keeps it for the life of the process; make
 * that first call before any stream capture, and do not call it again on a
 * device after cudaDeviceReset there (the kept address would be stale).  Each call clears the per-sequence counters it needs with
 * cudaMemsetAsync on the stream.  All calls share the one array, which keeps
 * the last call's contents, so calls that can overlap on the GPU (different
 * streams without ordering) race: serialise them.  No cudaMalloc, cudaFree
 * or other allocating routine is ever called. */
DFLASH_API int32_t dflash_verify_accept_noalloc(const float* logits,
                                                const int32_t* draft,
                                                int32_t b, int32_t R,
                                                int32_t D, int64_t V,
                                                int32_t* n_out,
                                                int32_t* corr_out,
                                                int32_t* emitted_out,
                                                int32_t* next_tok_out,
                                                void* stream);

/* Workspace bytes for dflash_verify_accept_sample. */
DFLASH_API int32_t dflash_verify_sample_workspace_size(int32_t b, int32_t R, int64_t V,
                                                       size_t* bytes);

/* Temperature speculative-sampling accept (mlx-dspark v0.0.3 release notes,
 * "Highlights": with temperature T > 0 the loop stays lossless, each emitted
 * token an exact sample from the target at T, "via the same acceptance rule
 * as DSpark").  The pages do not write the rule out; this is the standard
 * speculative-sampling rule for this drafter's greedy (one-hot) proposals.
 * For each sequence j, with p_r = softmax(logits[j][r] / T):
 *   draft i, in order, is accepted iff u_accept[j][i] < p_i(draft[j][i])
 *   n    = number of leading accepted drafts
 *   corr = a draw from p_n with draft[j][n] removed (renormalised) if n < D,
 *          a draw from p_D if n = D < R, else -1
 *   emitted / next_tok as in dflash_verify_accept.
 * The draw is argmax_v logits[j][row][v] / T - log(-log u_sample[j][v])
 * (Gumbel-max, decided in fp32, lowest index on ties).  The random numbers
 * are inputs: u_accept [b][D] and u_sample [b][V] fp32 on the device, every
 * value in the open interval (0, 1); values outside it give unspecified
 * tokens.  temperature: finite, > 0.  Accept probabilities are formed in
 * fp32 (max and exp-sum per vocabulary slice, merged in a fixed order).
 * Other arguments, layouts and errors as in dflash_verify_accept; ws holds
 * dflash_verify_sample_workspace_size bytes, zero-filled once (every call
 * leaves its counters zero).  A draft token outside [0, V) has probability 0
 * (rejected). */
DFLASH_API int32_t dflash_verify_accept_sample(const float* logits, const int32_t* draft,
                                               int32_t b, int32_t R, int32_t D, int64_t V,
                                               float temperature, const float* u_accept,
                                               const float* u_sample, int32_t* n_out,
                                               int32_t* corr_out, int32_t* emitted_out,
                                               int32_t* next_tok_out, void* ws,
                                               size_t ws_bytes, void* stream);

/* Commit and draft in one pass: the same results as dflash_kv_commit(w, kv,
 * hid, rows_per_seq, n, ...) followed by dflash_draft_block(w, kv, last_tok,
 * ...) on the same stream (up to fp32 summation order).  The committed rows'
 * K/V projections ride along in each layer's QKV GEMM of the draft, so the
 * K/V weights are read once and the separate K/V launch disappears; the
 * block is drafted against the grown context and len[] is advanced at the
 * end.  Arguments and errors are the union of the two calls'; ws is sized by
 * dflash_workspace_size(cfg, b, rows_per_seq). */
DFLASH_API int32_t dflash_commit_draft_block(const dflash_weights* w, const dflash_kv* kv,
                                             const uint16_t* hid, int32_t rows_per_seq,
                                             const int32_t* n, const int32_t* last_tok,
                                             int32_t* draft_out, float* hidden_out,
                                             float* logits_out, void* ws, size_t ws_bytes,
                                             void* stream);

/* Draft-KV commit with rollback of the rejected suffix (mlx-dspark v0.0.3,
 * "Notes": KV rollback; dflash-mlx "What It Does": conditioning on target
 * hidden states).  hid: [b][rows_per_seq][k*H] fp16 target hidden rows of the
 * verified block; n: [b] int32 (device) accept lengths, n[j] in [-1, B].
 * For each sequence j, rows r < c_j = min(n[j] + 1, rows_per_seq):
 *   c = RMSNorm(W8(fc) hid[j][r]; gamma_hid)
 *   per layer l: K = RoPE(per-head RMSNorm(W8(Wk_l) c; gamma_k[l]),
 *                         pos = len[j] + r),  V = W8(Wv_l) c
 *   written at cache row len[j] + r;  then len[j] += c_j.
 * Rows r >= c_j are never written.  A sequence whose len[j] + c_j would pass
 * `cap` is skipped whole and flags DFLASH_DEV_KV_CAPACITY.  rows_per_seq in
 * [1, 256] with b * rows_per_seq <= 4096. */
DFLASH_API int32_t dflash_kv_commit(const dflash_weights* w, const dflash_kv* kv,
                         const uint16_t* hid, int32_t rows_per_seq,
                         const int32_t* n, void* ws, size_t ws_bytes,
                         void* stream);

/* Launch modes (dflash_set_launch_mode).
 *  DFLASH_LAUNCH_STREAM_ORDER (the default): every kernel starts after the
 *    previous work of its stream has finished.  Correct whatever else runs
 *    on the GPU at the same time.
 *  DFLASH_LAUNCH_EARLY: every kernel is launched as a programmatic dependent
 *    of the previous kernel of its stream and lets its own dependents launch
 *    early, so each kernel's weight copies start while the previous kernel
 *    finishes (about 10 % shorter draft steps on a dedicated GPU).  Only for
 *    callers that own the GPU and issue the library's calls from one stream:
 *    on GB300 (driver 580), early-launched kernels gave wrong results, now
 *    and then, while other kernels (the library's on another stream, or any
 *    other work) ran on the same GPU. */
#define DFLASH_LAUNCH_STREAM_ORDER 0
#define DFLASH_LAUNCH_EARLY 1

/* Sets the launch mode of every later call in this process (all devices,
 * all threads).  A CUDA graph keeps the mode its kernels were captured with.
 * DFLASH_EINVAL for an unknown mode.  No page describes this; it is a
 * property of this library's kernels. */
DFLASH_API int32_t dflash_set_launch_mode(int32_t mode);

/* The current launch mode. */
DFLASH_API int32_t dflash_get_launch_mode(void);

/* Reads (and, when clear != 0, resets) the device status word of the current
 * device into *host_status.  Synchronises the device. */
DFLASH_API int32_t dflash_get_status(int32_t* host_status, int32_t clear);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
