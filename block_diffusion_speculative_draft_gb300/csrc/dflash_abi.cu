// dflash_abi.cu — the extern "C" entry points declared in include/dflash.h:
// argument validation, workspace carving and the kernel sequence of one
// draft step, one verify-accept and one draft-KV commit.  No allocation ever
// happens here: every byte of scratch comes from the caller's workspace.
#include <math.h>
#include <string.h>

#include "../../include/dflash.h"
#include "kernels.h"

using namespace dfl;

namespace {

__device__ int g_status;  // device status word (DFLASH_DEV_* bits)

int* status_ptr() {
  static int* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_cfg(const dflash_config* c) {
  if (!c) return DFLASH_EINVAL;
  if (c->L < 1 || c->H < 1 || c->nq < 1 || c->nkv < 1 || c->d < 1 || c->F < 1 || c->V < 1 || c->B < 2 ||
      c->k < 1)
    return DFLASH_EINVAL;
  if (c->mask_id < 0 || c->mask_id >= c->V) return DFLASH_EINVAL;
  if (!(c->eps >= 0.f) || !(c->rope_theta > 0.f)) return DFLASH_EINVAL;
  if (c->d != 64 && c->d != 128) return DFLASH_EUNSUPPORTED;
  if (c->H % 128 || (c->nq * c->d) % 128 || (c->nkv * c->d) % 128 || c->F % 128 || (c->k * c->H) % 128)
    return DFLASH_EUNSUPPORTED;
  if (c->nq % c->nkv) return DFLASH_EUNSUPPORTED;
  if (c->B > 32 || c->H > 8192) return DFLASH_EUNSUPPORTED;
  if (c->B * (c->nq / c->nkv) > 160) return DFLASH_EUNSUPPORTED;  // one attention query tile
  return DFLASH_OK;
}

int check_w8(const dflash_w8& w, int64_t N, int64_t K, int layout) {
  if (w.bits != 0 && w.bits != 8 && w.bits != 4) return DFLASH_EINVAL;
  if (!w.q || (w.bits != 4 && !w.s)) return DFLASH_EINVAL;
  if (w.N != N || w.K != K || w.layout != layout) return DFLASH_EINVAL;
  if (!aligned16(w.q)) return DFLASH_EINVAL;
  return DFLASH_OK;
}

struct WS {
  float* x;
  __half* u;
  __half* q;
  __half* kb;
  __half* vb;
  __half* ao;
  __half* g;
  __nv_bfloat16* h;
  float* ss;  // per-row, per-128-column sums of squares of x (deferred RMSNorm)
  void* lm;
  size_t total;
};

// bytes of the lm-head table prefetched into L2 during the layers' attention
constexpr size_t kLmPrefetchBytes = (size_t)96 << 20;

// Carves the workspace; the lm-head's argmax keys and ticket come first so a
// single zero-fill of the whole buffer initialises them.
WS carve(const dflash_config& c, int b, int rps, uint8_t* base) {
  WS w;
  const int M = b * c.B, Mc = b * rps;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off += al256(bytes);
    return p;
  };
  w.lm = take(lmhead_ws_bytes(b * (c.B - 1)));
  w.x = (float*)take((size_t)M * c.H * 4);
  w.u = (__half*)take((size_t)(M + Mc) * c.H * 2);  // block rows, then commit rows
  w.q = (__half*)take((size_t)M * c.nq * c.d * 2);
  w.kb = (__half*)take((size_t)M * c.nkv * c.d * 2);
  w.vb = (__half*)take((size_t)M * c.nkv * c.d * 2);
  w.ao = (__half*)take((size_t)M * c.nq * c.d * 2);
  w.g = (__half*)take((size_t)M * c.F * 2);
  w.h = (__nv_bfloat16*)take((size_t)b * (c.B - 1) * c.H * 2);
  w.ss = (float*)take((size_t)(M + Mc) * (c.H / 128) * 4);
  w.total = off;
  return w;
}

int map_err(cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_ECUDA; }

// Every launch, the first of a call included, requests programmatic dependent
// launch, which the library's launch mode grants or not: each kernel reads
// nothing but constant weights (and, for attention, the context it is given)
// before its griddepcontrol.wait, so it may start while the stream's
// previous kernel (of this call or of an earlier one) is still finishing.

W8Args base_args(const dflash_w8& w, int M, int epi) {
  W8Args a;
  memset(&a, 0, sizeof(a));
  a.q = static_cast<const uint8_t*>(w.q);
  a.s = reinterpret_cast<const __half*>(w.s);
  a.N = (int)w.N;
  a.K = (int)w.K;
  a.layout = w.layout;
  a.bits = w.bits == 4 ? 4 : 8;
  a.row0 = 0;
  a.nrows = (int)w.N;
  a.M = M;
  a.epi = epi;
  a.status = status_ptr();
  return a;
}

// RoPE frequencies theta^(-2p/d), computed in double and split into float
// pairs hi + lo for the single-precision angle reduction of the epilogues
void split_inv_freq(float* hi, float* lo, float theta, int d) {
  for (int p = 0; p < 64; ++p) {
    const double v = p < d / 2 ? pow((double)theta, -2.0 * p / d) : 0.0;
    hi[p] = (float)v;
    lo[p] = (float)(v - (double)hi[p]);
  }
}
void fill_inv_freq(W8Args& a, float theta, int d) { split_inv_freq(a.inv_hi, a.inv_lo, theta, d); }

}  // namespace

extern "C" {

const char* dflash_version(void) { return "dflash-gb300 0.1 (sm_103a)"; }

const char* dflash_status_string(int32_t s) {
  switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_EINVAL: return "invalid argument";
    case DFLASH_EUNSUPPORTED: return "unsupported shape";
    case DFLASH_ECUDA: return "CUDA error";
    case DFLASH_ECAPACITY: return "KV capacity exceeded";
    case DFLASH_EWORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int32_t dflash_workspace_size(const dflash_config* cfg, int32_t b, int32_t rows_per_seq, size_t* bytes) {
  int r = check_cfg(cfg);
  if (r) return r;
  if (!bytes || b < 1 || rows_per_seq < 1 || rows_per_seq > 256 || (int64_t)b * rows_per_seq > 4096)
    return DFLASH_EINVAL;
  WS w = carve(*cfg, b, rows_per_seq, nullptr);
  *bytes = w.total;
  return DFLASH_OK;
}

int32_t dflash_pack_w8a16(const void* w, int32_t w_dtype, int64_t N, int64_t K, int32_t layout, void* q_out,
                          uint16_t* s_out, void* stream) {
  if (!w || !q_out || !s_out) return DFLASH_EINVAL;
  if (w_dtype < 0 || w_dtype > 2 || N < 1 || K < 1) return DFLASH_EINVAL;
  if (layout != DFLASH_LAYOUT_PLAIN && layout != DFLASH_LAYOUT_GATEUP) return DFLASH_EINVAL;
  if (N % 128 || K % 128) return DFLASH_EUNSUPPORTED;
  if (layout == DFLASH_LAYOUT_GATEUP && (N / 2) % 64) return DFLASH_EUNSUPPORTED;
  if (!aligned16(q_out)) return DFLASH_EINVAL;
  return map_err(w8_pack(w, w_dtype, N, K, layout, static_cast<uint8_t*>(q_out), reinterpret_cast<__half*>(s_out),
                         static_cast<cudaStream_t>(stream)));
}

int32_t dflash_w4a16_packed_bytes(int64_t N, int64_t K, size_t* bytes) {
  if (!bytes || N < 1 || K < 1) return DFLASH_EINVAL;
  if (N % 128 || K % 128) return DFLASH_EUNSUPPORTED;
  *bytes = (size_t)(N / 128) * (size_t)(K / 128) * (size_t)kW4TileBytes;
  return DFLASH_OK;
}

int32_t dflash_pack_w4a16(const void* w, int32_t w_dtype, int64_t N, int64_t K, int32_t layout, void* q_out,
                          uint16_t* s_out, void* stream) {
  if (!w || !q_out || !s_out) return DFLASH_EINVAL;
  if (w_dtype < 0 || w_dtype > 2 || N < 1 || K < 1) return DFLASH_EINVAL;
  if (layout != DFLASH_LAYOUT_PLAIN && layout != DFLASH_LAYOUT_GATEUP) return DFLASH_EINVAL;
  if (N % 128 || K % 128) return DFLASH_EUNSUPPORTED;
  if (layout == DFLASH_LAYOUT_GATEUP && (N / 2) % 64) return DFLASH_EUNSUPPORTED;
  if (!aligned16(q_out)) return DFLASH_EINVAL;
  return map_err(w4_pack(w, w_dtype, N, K, layout, static_cast<uint8_t*>(q_out), reinterpret_cast<__half*>(s_out),
                         static_cast<cudaStream_t>(stream)));
}

int32_t dflash_w8a16_linear(const dflash_w8* w, const uint16_t* x, int64_t M, float* y, void* ws, size_t ws_bytes,
                            void* stream) {
  (void)ws;
  (void)ws_bytes;  // split-K reduces through cluster shared memory: no scratch
  if (!w || !x || !y) return DFLASH_EINVAL;
  if (M < 1 || M > 4096) return DFLASH_EINVAL;
  if (w->N % 128 || w->K % 128 || w->N < 128) return DFLASH_EUNSUPPORTED;
  if (int r = check_w8(*w, w->N, w->K, w->layout)) return r;
  if (!aligned16(x)) return DFLASH_EINVAL;
  W8Args a = base_args(*w, (int)M, EPI_STORE_F32);
  a.out_f32 = y;
  a.ldo = (int)w->N;
  return map_err(w8_gemm(a, reinterpret_cast<const __half*>(x), static_cast<cudaStream_t>(stream), true));
}

int32_t dflash_w8a16_linear_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
  if (!bytes || M < 1 || M > 4096 || N < 128 || K < 128 || N % 128 || K % 128) return DFLASH_EINVAL;
  *bytes = 0;
  return DFLASH_OK;
}

static int check_weights(const dflash_weights* w) {
  if (!w) return DFLASH_EINVAL;
  const dflash_config& c = w->cfg;
  if (int r = check_cfg(&c)) return r;
  if (!w->qkv || !w->o || !w->gu || !w->down) return DFLASH_EINVAL;
  if (!w->gamma_hid || !w->gamma_in || !w->gamma_post || !w->gamma_q || !w->gamma_k || !w->gamma_final ||
      !w->embed || !w->lm_head)
    return DFLASH_EINVAL;
  if (!aligned16(w->lm_head) || !aligned16(w->embed) || !aligned16(w->gamma_hid) || !aligned16(w->gamma_in) ||
      !aligned16(w->gamma_post) || !aligned16(w->gamma_final))
    return DFLASH_EINVAL;
  if (int r = check_w8(w->fc, c.H, (int64_t)c.k * c.H, DFLASH_LAYOUT_PLAIN)) return r;
  const int64_t nqkv = (int64_t)(c.nq + 2 * c.nkv) * c.d;
  for (int l = 0; l < c.L; ++l) {
    if (int r = check_w8(w->qkv[l], nqkv, c.H, DFLASH_LAYOUT_PLAIN)) return r;
    if (int r = check_w8(w->o[l], c.H, (int64_t)c.nq * c.d, DFLASH_LAYOUT_PLAIN)) return r;
    if (int r = check_w8(w->gu[l], 2 * (int64_t)c.F, c.H, DFLASH_LAYOUT_GATEUP)) return r;
    if (int r = check_w8(w->down[l], c.H, c.F, DFLASH_LAYOUT_PLAIN)) return r;
  }
  // one weight format per drafter (batched launches span several layers)
  const int bits = w->fc.bits == 4 ? 4 : 8;
  for (int l = 0; l < c.L; ++l) {
    for (const dflash_w8* m : {&w->qkv[l], &w->o[l], &w->gu[l], &w->down[l]})
      if ((m->bits == 4 ? 4 : 8) != bits) return DFLASH_EINVAL;
  }
  return DFLASH_OK;
}

static int check_kv(const dflash_kv* kv) {
  if (!kv || !kv->k || !kv->v || !kv->len) return DFLASH_EINVAL;
  if (kv->b < 1 || kv->cap < 1) return DFLASH_EINVAL;
  if (kv->cap > (1 << 24) - 64) return DFLASH_EUNSUPPORTED;  // positions stay exact in fp32
  if (!aligned16(kv->k) || !aligned16(kv->v)) return DFLASH_EINVAL;
  return DFLASH_OK;
}

// A draft pass, optionally with a commit folded in (hid non-null): the
// commit's context rows ride along in each layer's QKV projection, so their
// K/V reach the cache without a separate launch and the block is drafted
// against the grown context, exactly as a commit followed by a draft.
static int32_t draft_block_impl(const dflash_weights* w, const dflash_kv* kv, const int32_t* last_tok,
                                int32_t* draft_out, float* hidden_out, float* logits_out, void* ws, size_t ws_bytes,
                                void* stream, const uint16_t* hid = nullptr, int rps = 0,
                                const int32_t* ncommit = nullptr) {
  if (int r = check_weights(w)) return r;
  if (int r = check_kv(kv)) return r;
  if (!last_tok || !draft_out) return DFLASH_EINVAL;
  if (!aligned16(hidden_out)) return DFLASH_EINVAL;
  const dflash_config& c = w->cfg;
  const int b = kv->b;
  if ((int64_t)b * c.B > 4096) return DFLASH_EUNSUPPORTED;
  const bool commit = hid != nullptr;
  if (commit) {
    if (!ncommit || !aligned16(hid)) return DFLASH_EINVAL;
    if (rps < 1 || rps > 256 || (int64_t)b * rps > 4096) return DFLASH_EINVAL;
  }
  const int rps_ws = commit ? rps : c.B;
  WS need = carve(c, b, rps_ws, nullptr);
  if (!ws || ws_bytes < need.total) return DFLASH_EWORKSPACE;
  WS s = carve(c, b, rps_ws, static_cast<uint8_t*>(ws));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = status_ptr();
  if (!status) return DFLASH_ECUDA;
  const int M = b * c.B;
  const int qd = c.nq * c.d, kd = c.nkv * c.d;
  const size_t layer_kv = (size_t)b * c.nkv * kv->cap * c.d;
  cudaError_t e;
  // L2 prefetch of the lm-head: a whole number of rows of each first-round
  // tile, about kLmPrefetchBytes in total
  const bool debug_out = hidden_out || logits_out;
  const int lm_tile = lmhead_tile_rows(b * (c.B - 1), c.H);
  int lm_first = lmhead_first_tiles(b * (c.B - 1), c.V, c.H);
  if (lm_first > c.V / lm_tile) lm_first = c.V / lm_tile;  // whole tiles only: never past the table
  const size_t row_bytes = (size_t)c.H * 2;
  size_t lm_rows = lm_first > 0 ? kLmPrefetchBytes / ((size_t)lm_first * row_bytes) : 0;
  if (lm_rows > (size_t)lm_tile) lm_rows = lm_tile;
  const uint32_t lm_pf_bytes = (uint32_t)(lm_rows * row_bytes);
  const int Mc = commit ? b * rps : 0;
  const int nss = c.H / 128;
  if (commit) {
    // c = RMSNorm(W8(fc) h; gamma_hid), deferred: u rows [M, M + Mc) = y * gamma_hid
    W8Args af = base_args(w->fc, Mc, EPI_STORE_F32);
    af.ldo = c.H;
    af.xg_out = s.u + (size_t)M * c.H;
    af.g_next = w->gamma_hid;
    af.ss_out = s.ss + (size_t)M * nss;
    af.nss_out = nss;
    if (w8_gemm(af, reinterpret_cast<const __half*>(hid), st, true) != cudaSuccess) return DFLASH_ECUDA;
  }
  // with a commit every activation row of the first QKV is in the deferred form
  e = embed_rmsnorm(reinterpret_cast<const __nv_bfloat16*>(w->embed), last_tok, c.mask_id, c.V, b, c.B, c.H,
                    w->gamma_in, c.eps, s.x, s.u, commit ? s.ss : nullptr, st, true, status);
  if (e != cudaSuccess) return DFLASH_ECUDA;
  for (int l = 0; l < c.L; ++l) {
    // [q|k|v] = W8(qkv) u ; per-head QK-RMSNorm + neox RoPE in the epilogue
    W8Args a = base_args(w->qkv[l], M + Mc, EPI_QKV);
    fill_inv_freq(a, c.rope_theta, c.d);
    a.out_h = s.q;
    a.kout = s.kb;
    a.vout = s.vb;
    a.gq = w->gamma_q + (size_t)l * c.d;
    a.gk = w->gamma_k + (size_t)l * c.d;
    a.nq = c.nq;
    a.nkv = c.nkv;
    a.d = c.d;
    a.theta = c.rope_theta;
    a.eps = c.eps;
    a.len = kv->len;
    a.rows_per_seq = c.B;
    a.b = b;
    a.cap = kv->cap;
    if (l > 0 || commit) {  // else layer 0 reads the embedding, normalised by its own kernel
      a.ss_in = s.ss;
      a.nss_in = nss;
    }
    if (commit) {
      a.mc0 = M;
      a.c_nacc = ncommit;
      a.c_rps = rps;
      a.ck = reinterpret_cast<__half*>(kv->k) + l * layer_kv;
      a.cv = reinterpret_cast<__half*>(kv->v) + l * layer_kv;
    }
    if ((e = w8_gemm(a, s.u, st, true)) != cudaSuccess) return DFLASH_ECUDA;
    // block attention over [context || block]
    AttnArgs at{};
    at.q = s.q;
    at.kblk = s.kb;
    at.vblk = s.vb;
    at.kc = reinterpret_cast<const __half*>(kv->k) + l * layer_kv;
    at.vc = reinterpret_cast<const __half*>(kv->v) + l * layer_kv;
    at.len = kv->len;
    at.out = s.ao;
    at.b = b;
    at.B = c.B;
    at.nq = c.nq;
    at.nkv = c.nkv;
    at.d = c.d;
    at.cap = kv->cap;
    at.status = status;
    if (commit) {
      at.nacc = ncommit;
      at.rps = rps;
    }
    // HBM is nearly idle during attention: pull a prefix of each vocabulary
    // tile that starts an lm-head CTA's stream into L2 (a share per layer),
    // so the lm-head reads that part from L2
    at.pf_base = reinterpret_cast<const uint8_t*>(w->lm_head);
    at.pf_stride = (size_t)lm_tile * c.H * 2;
    at.pf_bytes = lm_pf_bytes;
    at.pf_i0 = (int)((long long)lm_first * l / c.L);
    at.pf_i1 = (int)((long long)lm_first * (l + 1) / c.L);
    if ((e = attention(at, st, true)) != cudaSuccess) return DFLASH_ECUDA;
    // x += W8(o) attn
    // x += W8(o) attn; the epilogue also leaves u = x * gamma_post and the
    // row sums of squares, so the post-attention RMSNorm is applied by the
    // next GEMM's epilogue (RMSNorm is a per-row scale, which commutes with
    // the contraction)
    W8Args ao = base_args(w->o[l], M, EPI_RESID_F32);
    ao.out_f32 = s.x;
    ao.ldo = c.H;
    ao.xg_out = s.u;
    ao.g_next = w->gamma_post + (size_t)l * c.H;
    ao.ss_out = s.ss;
    ao.nss_out = c.H / 128;
    if ((e = w8_gemm(ao, s.ao, st, true)) != cudaSuccess) return DFLASH_ECUDA;
    // g = silu(gate) * up, gate/up scaled by the deferred norm factor
    W8Args ag = base_args(w->gu[l], M, EPI_SWIGLU);
    ag.out_h = s.g;
    ag.ss_in = s.ss;
    ag.nss_in = c.H / 128;
    ag.eps = c.eps;
    if ((e = w8_gemm(ag, s.u, st, true)) != cudaSuccess) return DFLASH_ECUDA;
    // x += W8(down) g; for all but the last layer also u = x * gamma_in[l+1]
    W8Args ad = base_args(w->down[l], M, EPI_RESID_F32);
    ad.out_f32 = s.x;
    ad.ldo = c.H;
    if (l + 1 < c.L) {
      ad.xg_out = s.u;
      ad.g_next = w->gamma_in + (size_t)(l + 1) * c.H;
      ad.ss_out = s.ss;
      ad.nss_out = c.H / 128;
    } else if (!debug_out) {
      // the lm-head input straight from the last residual update
      ad.hb_out = s.h;
      ad.hb_rps = c.B;
      ad.g_next = w->gamma_final;
    }
    if ((e = w8_gemm(ad, s.g, st, true)) != cudaSuccess) return DFLASH_ECUDA;
  }
  (void)qd;
  (void)kd;
  // normalised hidden rows (and so true logits) only when asked for them
  if (debug_out &&
      (e = final_norm(s.x, b, c.B, c.H, w->gamma_final, c.eps, s.h, hidden_out, st, true)) != cudaSuccess)
    return DFLASH_ECUDA;
  e = lmhead_argmax(s.h, reinterpret_cast<const __nv_bfloat16*>(w->lm_head), b * (c.B - 1), c.V, c.H, draft_out,
                    nullptr, logits_out, s.lm, st, true, status);
  if (e != cudaSuccess) return DFLASH_ECUDA;
  if (commit) e = commit_len_update(kv->len, ncommit, b, rps, kv->cap, st, true, status);
  return map_err(e);
}

int32_t dflash_draft_block(const dflash_weights* w, const dflash_kv* kv, const int32_t* last_tok, int32_t* draft_out,
                           float* hidden_out, float* logits_out, void* ws, size_t ws_bytes, void* stream) {
  return draft_block_impl(w, kv, last_tok, draft_out, hidden_out, logits_out, ws, ws_bytes, stream);
}

int32_t dflash_commit_draft_block(const dflash_weights* w, const dflash_kv* kv, const uint16_t* hid,
                                  int32_t rows_per_seq, const int32_t* n, const int32_t* last_tok, int32_t* draft_out,
                                  float* hidden_out, float* logits_out, void* ws, size_t ws_bytes, void* stream) {
  if (!hid) return DFLASH_EINVAL;
  return draft_block_impl(w, kv, last_tok, draft_out, hidden_out, logits_out, ws, ws_bytes, stream, hid,
                          rows_per_seq, n);
}

int32_t dflash_lmhead_workspace_size(int64_t M, size_t* bytes) {
  if (!bytes || M < 1 || M > 128) return DFLASH_EINVAL;
  *bytes = lmhead_ws_bytes(M);
  return DFLASH_OK;
}

int32_t dflash_lmhead_argmax(const uint16_t* h, const uint16_t* w, int64_t M, int64_t V, int64_t H, int32_t* idx_out,
                             float* maxlogit_out, float* logits_out, void* ws, size_t ws_bytes, void* stream) {
  if (!h || !w || !idx_out) return DFLASH_EINVAL;
  if (M < 1 || M > 128 || V < 1 || V > (int64_t)1 << 30 || H < 64) return DFLASH_EINVAL;
  if (H % 64) return DFLASH_EUNSUPPORTED;
  if (!aligned16(h) || !aligned16(w)) return DFLASH_EINVAL;
  if (!ws || ws_bytes < lmhead_ws_bytes(M)) return DFLASH_EWORKSPACE;
  int* status = status_ptr();
  if (!status) return DFLASH_ECUDA;
  return map_err(lmhead_argmax(reinterpret_cast<const __nv_bfloat16*>(h), reinterpret_cast<const __nv_bfloat16*>(w),
                               (int)M, (int)V, (int)H, idx_out, maxlogit_out, logits_out, ws,
                               static_cast<cudaStream_t>(stream), true, status));
}

int32_t dflash_verify_workspace_size(int32_t b, int32_t R, int64_t V, size_t* bytes) {
  if (!bytes || b < 1 || R < 1 || R > 64 || V < 1) return DFLASH_EINVAL;
  *bytes = verify_ws_bytes(b, R, V);
  return DFLASH_OK;
}

int32_t dflash_verify_accept(const float* logits, const int32_t* draft, int32_t b, int32_t R, int32_t D, int64_t V,
                             int32_t* n_out, int32_t* corr_out, int32_t* emitted_out, int32_t* next_tok_out, void* ws,
                             size_t ws_bytes, void* stream) {
  if (!logits || !draft || !n_out || !corr_out) return DFLASH_EINVAL;
  if (b < 1 || R < 1 || R > 64 || D < 1 || D > R || V < 1 || V > ((int64_t)1 << 31) - 1) return DFLASH_EINVAL;
  if ((int64_t)b * R > 65535) return DFLASH_EUNSUPPORTED;
  if (!ws || ws_bytes < verify_ws_bytes(b, R, V)) return DFLASH_EWORKSPACE;
  if ((V & 3) == 0 && !aligned16(logits)) return DFLASH_EINVAL;
  return map_err(verify_accept(logits, draft, b, R, D, V, n_out, corr_out, emitted_out, next_tok_out, ws,
                               static_cast<cudaStream_t>(stream), true));
}

int32_t dflash_verify_accept_noalloc(const float* logits, const int32_t* draft, int32_t b, int32_t R, int32_t D,
                                     int64_t V, int32_t* n_out, int32_t* corr_out, int32_t* emitted_out,
                                     int32_t* next_tok_out, void* stream) {
  if (!logits || !draft || !n_out || !corr_out) return DFLASH_EINVAL;
  if (b < 1 || R < 1 || R > 64 || D < 1 || D > R || V < 1 || V > ((int64_t)1 << 31) - 1) return DFLASH_EINVAL;
  if ((int64_t)b * R > 65535) return DFLASH_EUNSUPPORTED;
  if ((V & 3) == 0 && !aligned16(logits)) return DFLASH_EINVAL;
  const size_t need = verify_noalloc_need(b, R, V);
  if (need == (size_t)-1 || need > kNoAllocScratchBytes) return DFLASH_EWORKSPACE;
  return map_err(verify_accept_noalloc(logits, draft, b, R, D, V, n_out, corr_out, emitted_out, next_tok_out,
                                       static_cast<cudaStream_t>(stream)));
}

int32_t dflash_verify_sample_workspace_size(int32_t b, int32_t R, int64_t V, size_t* bytes) {
  if (!bytes || b < 1 || R < 1 || R > 64 || V < 1) return DFLASH_EINVAL;
  *bytes = sample_ws_bytes(b, R, V);
  return DFLASH_OK;
}

int32_t dflash_verify_accept_sample(const float* logits, const int32_t* draft, int32_t b, int32_t R, int32_t D,
                                    int64_t V, float temperature, const float* u_accept, const float* u_sample,
                                    int32_t* n_out, int32_t* corr_out, int32_t* emitted_out, int32_t* next_tok_out,
                                    void* ws, size_t ws_bytes, void* stream) {
  if (!logits || !draft || !u_accept || !u_sample || !n_out || !corr_out) return DFLASH_EINVAL;
  if (b < 1 || R < 1 || R > 64 || D < 1 || D > R || V < 1 || V > ((int64_t)1 << 31) - 1) return DFLASH_EINVAL;
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return DFLASH_EINVAL;
  if ((int64_t)b * R > 65535) return DFLASH_EUNSUPPORTED;
  if (!ws || ws_bytes < sample_ws_bytes(b, R, V)) return DFLASH_EWORKSPACE;
  return map_err(verify_sample(logits, draft, b, R, D, V, temperature, u_accept, u_sample, n_out, corr_out,
                               emitted_out, next_tok_out, ws, static_cast<cudaStream_t>(stream), true));
}

int32_t dflash_kv_commit(const dflash_weights* w, const dflash_kv* kv, const uint16_t* hid, int32_t rows_per_seq,
                         const int32_t* n, void* ws, size_t ws_bytes, void* stream) {
  if (int r = check_weights(w)) return r;
  if (int r = check_kv(kv)) return r;
  if (!hid || !n) return DFLASH_EINVAL;
  if (rows_per_seq < 1 || rows_per_seq > 256 || (int64_t)kv->b * rows_per_seq > 4096) return DFLASH_EINVAL;
  if (!aligned16(hid)) return DFLASH_EINVAL;
  const dflash_config& c = w->cfg;
  const int b = kv->b;
  WS need = carve(c, b, rows_per_seq, nullptr);
  if (!ws || ws_bytes < need.total) return DFLASH_EWORKSPACE;
  WS s = carve(c, b, rows_per_seq, static_cast<uint8_t*>(ws));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = status_ptr();
  if (!status) return DFLASH_ECUDA;
  const int Mc = b * rows_per_seq;
  const size_t layer_kv = (size_t)b * c.nkv * kv->cap * c.d;
  // c = RMSNorm(W8(fc) h; gamma_hid)
  // the epilogue writes u = y * gamma_hid and the row sums of squares; the
  // K/V GEMMs apply the RMSNorm factor to their results
  W8Args af = base_args(w->fc, Mc, EPI_STORE_F32);
  af.ldo = c.H;
  af.xg_out = s.u;
  af.g_next = w->gamma_hid;
  af.ss_out = s.ss;
  af.nss_out = c.H / 128;
  if (w8_gemm(af, reinterpret_cast<const __half*>(hid), st, true) != cudaSuccess) return DFLASH_ECUDA;
  // K = rope(knorm(W_k c)), V = W_v c for every layer: the K/V rows of each
  // layer's qkv projection, up to kLayersPerLaunch layers in one launch
  for (int l0 = 0; l0 < c.L; l0 += kLayersPerLaunch) {
    const int nl = c.L - l0 < kLayersPerLaunch ? c.L - l0 : kLayersPerLaunch;
    W8Args a = base_args(w->qkv[l0], Mc, EPI_KVCOMMIT);
    fill_inv_freq(a, c.rope_theta, c.d);
    a.row0 = c.nq * c.d;
    a.nrows = 2 * c.nkv * c.d;
    a.nl = nl;
    a.ntl = a.nrows / kTile;
    for (int i = 0; i < nl; ++i) {
      const int l = l0 + i;
      a.lq[i] = static_cast<const uint8_t*>(w->qkv[l].q);
      a.ls[i] = reinterpret_cast<const __half*>(w->qkv[l].s);
      a.lk[i] = reinterpret_cast<__half*>(kv->k) + l * layer_kv;
      a.lv[i] = reinterpret_cast<__half*>(kv->v) + l * layer_kv;
      a.lgk[i] = w->gamma_k + (size_t)l * c.d;
    }
    a.nq = c.nq;
    a.nkv = c.nkv;
    a.d = c.d;
    a.theta = c.rope_theta;
    a.eps = c.eps;
    a.len = kv->len;
    a.nacc = n;
    a.rows_per_seq = rows_per_seq;
    a.b = b;
    a.cap = kv->cap;
    a.ss_in = s.ss;
    a.nss_in = c.H / 128;
    if (w8_gemm(a, s.u, st, true) != cudaSuccess) return DFLASH_ECUDA;
  }
  return map_err(commit_len_update(kv->len, n, b, rows_per_seq, kv->cap, st, true, status));
}

int32_t dflash_set_launch_mode(int32_t mode) {
  if (mode != DFLASH_LAUNCH_STREAM_ORDER && mode != DFLASH_LAUNCH_EARLY) return DFLASH_EINVAL;
  set_launch_mode(mode);
  return DFLASH_OK;
}

int32_t dflash_get_launch_mode(void) { return get_launch_mode(); }

int32_t dflash_get_status(int32_t* host_status, int32_t clear) {
  if (!host_status) return DFLASH_EINVAL;
  if (cudaDeviceSynchronize() != cudaSuccess) return DFLASH_ECUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return DFLASH_ECUDA;
  *host_status = v;
  if (clear) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return DFLASH_ECUDA;
  }
  return DFLASH_OK;
}

}  // extern "C"
