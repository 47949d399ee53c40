// kernels.h — host-side launchers shared between the C-ABI translation unit
// and the kernel translation units.  Plain C++ declarations, no device code.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dfl {

constexpr int kTile = 128;            // packed weight tile edge (rows x k-columns)
constexpr int kLayersPerLaunch = 8;   // layers batched into one commit GEMM launch
constexpr int kTileBytes = 16384;     // one packed int8 tile

// Streaming multiprocessors of the current device (queried once per device).
int num_sms();

// Whether launches may start early as programmatic dependents of the
// previous kernel in their stream (the library's launch mode).
bool launch_early();
void set_launch_mode(int mode);
int get_launch_mode();

enum Epi : int {
  EPI_STORE_F32 = 0,  // out[m][n] = y
  EPI_RESID_F32 = 1,  // out[m][n] += y
  EPI_SWIGLU = 2,     // g[m][j] = silu(gate_j) * up_j  (fp16)
  EPI_QKV = 3,        // per-head Q/K RMSNorm + RoPE; q, block k, block v (fp16)
  EPI_KVCOMMIT = 4,   // per-head K RMSNorm + RoPE; K, V appended to the cache
};

struct W8Args {
  const uint8_t* q;  // packed tiles
  const __half* s;   // logical-order scales (int8 weights only)
  int N, K, layout;
  int bits;  // 8: int8 tiles + per-row scales; 4: int4 tiles carrying their group scales
  int row0;   // first packed row used (multiple of 128)
  int nrows;  // packed rows used (multiple of 128)
  int M;      // activation rows
  int splits;  // k-splits = cluster size along y
  int epi;
  float* out_f32;
  int ldo;
  __half* out_h;  // EPI_SWIGLU: g [M][F]; EPI_QKV: q [M][nq d]
  __half* kout;   // EPI_QKV: block k [M][nkv d]; EPI_KVCOMMIT: layer's K cache
  __half* vout;
  const float* gq;
  const float* gk;
  int nq, nkv, d, F;
  float theta, eps;
  const int* len;    // [b] committed lengths
  const int* nacc;   // EPI_KVCOMMIT: accept lengths
  int rows_per_seq;  // activation rows per sequence
  int b, cap;
  int* status;
  // Deferred RMSNorm.  Reader side: when ss_in is set, the activations are
  // x * gamma (not yet normalised) and the epilogue scales each row's result
  // by rsqrt(sum_i ss_in[m][i] / K + eps), i < nss_in.  Writer side (STORE /
  // RESID): when xg_out is set, also write fp16(y * g_next) and each row's
  // sum of squares over this 128-column tile into ss_out[m][tile].
  const float* ss_in;
  int nss_in;
  float* ss_out;
  int nss_out;
  __half* xg_out;
  const float* g_next;
  // Lm-head input (RESID): when set, rows with slot m % hb_rps > 0 also go to
  // hb_out, compacted to row (m / hb_rps) (hb_rps - 1) + slot - 1, as
  // bf16(y * g_next): the final RMSNorm's per-row factor is left out, which
  // the argmax over each row's logits does not see.
  __nv_bfloat16* hb_out;
  int hb_rps;
  // A commit folded into the draft's QKV projection (EPI_QKV only; c_nacc
  // null: none): rows m >= mc0 are target-context rows, c_rps per sequence,
  // whose K/V go into this layer's cache ck / cv at len + slot for the
  // committed slots; the block's rows sit after the new length.
  int mc0;
  const int* c_nacc;
  int c_rps;
  __half* ck;
  __half* cv;
  // Several layers' projections in one launch (the K/V rows of every
  // layer's qkv for a commit): tile columns [i ntl, (i + 1) ntl) of the grid
  // belong to layer i < nl and use lq/ls/lk/lv/lgk[i] in place of
  // q/s/kout/vout/gk.  nl = 0: a single projection.
  int nl, ntl;
  const uint8_t* lq[kLayersPerLaunch];
  const __half* ls[kLayersPerLaunch];
  __half* lk[kLayersPerLaunch];
  __half* lv[kLayersPerLaunch];
  const float* lgk[kLayersPerLaunch];
  // RoPE frequencies theta^(-2p/d), p < d/2, as float pairs hi + lo of the
  // double value (per-head epilogues)
  float inv_hi[64];
  float inv_lo[64];
};

// Tensor-map encoder of the CUDA driver API (resolved once through the runtime).
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);
// Same for a 3-D tensor: dims innermost first, strides (bytes) of dims 1 and 2.
bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const uint64_t dims[3],
                    const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle swz);

// Launch helpers: the programmatic-dependent-launch attribute is set when
// `pdl` is requested and the library's launch mode allows early launches
// (launch_early()); launch_kc also groups blocks into thread-block clusters
// of shape `cluster` (no cluster when 1x1x1).
cudaError_t launch_k(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, void** args);
cudaError_t launch_kc(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, dim3 cluster,
                      void** args);

// --- W8A16 GEMM (k_gemm_w8.cu) ---
int w8_pick_splits(int units, int KT);
cudaError_t w8_gemm(const W8Args& a, const __half* x, cudaStream_t st, bool pdl);
cudaError_t w8_pack(const void* w, int w_dtype, int64_t N, int64_t K, int layout, uint8_t* q_out, __half* s_out,
                    cudaStream_t st);
// int4 packing: s_out [N][K/128] group scales in logical order, q_out the
// packed tiles of kW4TileBytes each (nibbles + the tile's rows' scales)
cudaError_t w4_pack(const void* w, int w_dtype, int64_t N, int64_t K, int layout, uint8_t* q_out, __half* s_out,
                    cudaStream_t st);
constexpr int64_t kW4TileBytes = 8192 + 256;

// --- lm-head GEMM + argmax (k_lmhead.cu) ---
size_t lmhead_ws_bytes(int64_t M);
// Vocabulary tiles the lm-head kernel reads first (lmhead_tile_rows rows
// each): tiles [0, n) start every CTA's stream.
int lmhead_first_tiles(int M, int V, int H);
// Vocabulary rows per lm-head tile for M rows (the stride of the tiles that
// lmhead_first_tiles counts).
int lmhead_tile_rows(int M, int H);
cudaError_t lmhead_argmax(const __nv_bfloat16* h, const __nv_bfloat16* w, int M, int V, int H, int* idx_out,
                          float* maxlogit, float* logits, void* ws, cudaStream_t st, bool pdl, int* status);

// --- block attention (k_attn.cu) ---
struct AttnArgs {
  const __half* q;     // [M][nq][d]
  const __half* kblk;  // [M][nkv][d]
  const __half* vblk;
  const __half* kc;  // layer's K cache [b][nkv][cap][d]
  const __half* vc;
  const int* len;
  __half* out;  // [M][nq][d]
  int b, B, nq, nkv, d, cap;
  int* status;
  int nwc;  // compute warps (16 query rows each); the rest help with loads and the merge
  // a commit folded into this pass (null: none): the context grows by
  // commit_count(len, nacc, rps, cap) rows, written by this layer's QKV kernel
  const int* nacc;
  int rps;
  // L2 prefetch issued while the kernel would otherwise leave HBM idle:
  // pieces [pf_i0, pf_i1) of base + i * pf_stride, pf_bytes each (or none)
  const uint8_t* pf_base;
  size_t pf_stride;
  uint32_t pf_bytes;
  int pf_i0, pf_i1;
};
cudaError_t attention(const AttnArgs& a, cudaStream_t st, bool pdl);

// --- small kernels (k_small.cu) ---
// ss_out null: u = RMSNorm(x; gamma).  Else the deferred form: u = x * gamma
// and ss_out[m][H/128] = sums of squares per 128-column tile.
cudaError_t embed_rmsnorm(const __nv_bfloat16* E, const int* last_tok, int mask_id, int V, int b, int B, int H,
                          const float* gamma, float eps, float* x, __half* u, float* ss_out, cudaStream_t st,
                          bool pdl, int* status);

// Rows of a sequence a commit appends: min(n + 1, rps), or 0 when n is out
// of [-1, rps], the length is negative or the rows would pass cap (the
// length-update kernel flags those cases).
__device__ __forceinline__ int commit_count(int len, int n, int rps, int cap) {
  int c = n + 1 < rps ? n + 1 : rps;
  if (c < 0) c = 0;
  return (n >= -1 && n <= rps && len >= 0 && len + c <= cap) ? c : 0;
}
cudaError_t final_norm(const float* x, int b, int B, int H, const float* gamma, float eps, __nv_bfloat16* h,
                       float* hidden_out, cudaStream_t st, bool pdl);
cudaError_t commit_len_update(int* len, const int* nacc, int b, int rows_per_seq, int cap, cudaStream_t st,
                              bool pdl, int* status);
// --- temperature speculative-sampling accept (k_sample.cu) ---
struct SampleArgs {
  const float* logits;    // [b][R][V]
  const int* draft;       // [b][D]
  const float* u_acc;     // [b][D] uniforms in (0, 1)
  const float* u_sample;  // [b][V] uniforms in (0, 1)
  int b, R, D;
  int64_t V;
  float T;
  int P, P2;              // vocabulary slices per row (stats) / per sequence (pick)
  int64_t chunk, chunk2;  // slice lengths
  int* tickets;           // [2b] zero between calls
  float2* part;           // [b R][P] (max, exp-sum) of z / T per slice
  float* zx;              // [b R] z / T of each row's draft token
  int* sel;               // [b][2] row to sample (-1: none), token it excludes
  unsigned long long* keys;  // [b][P2]
  int* n_out;
  int* corr_out;
  int* emitted;
  int* next_tok;
};
int sample_parts(int b, int R, int64_t V);
int sample_parts2(int b, int64_t V);
size_t sample_ws_bytes(int b, int R, int64_t V);
cudaError_t verify_sample(const float* logits, const int* draft, int b, int R, int D, int64_t V, float T,
                          const float* u_acc, const float* u_sample, int* n_out, int* corr_out, int* emitted,
                          int* next_tok, void* ws, cudaStream_t st, bool pdl);
size_t verify_ws_bytes(int b, int R, int64_t V);
cudaError_t verify_accept(const float* logits, const int* draft, int b, int R, int D, int64_t V, int* n_out,
                          int* corr_out, int* emitted, int* next_tok, void* ws, cudaStream_t st, bool pdl);

// Allocation-free variant of verify_accept: scratch lives in a fixed device
// array of kNoAllocScratchBytes inside the library (k_small.cu).
constexpr size_t kNoAllocScratchBytes = 64 * 1024;
size_t verify_noalloc_need(int b, int R, int64_t V);
cudaError_t verify_accept_noalloc(const float* logits, const int* draft, int b, int R, int D, int64_t V, int* n_out,
                                  int* corr_out, int* emitted, int* next_tok, cudaStream_t st);

}  // namespace dfl
