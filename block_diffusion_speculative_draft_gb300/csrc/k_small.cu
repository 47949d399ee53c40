// k_small.cu — the latency-sized kernels of the step: block embedding + first
// RMSNorm, RMSNorm, final norm, commit-length update and the greedy
// verify-accept; plus the launch and tensor-map helpers shared by all
// kernels.
#include "kernels.h"
#include "ptx.cuh"

namespace dfl {

// ------------------------------------------------------------- helpers ----
cudaError_t launch_k(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

constexpr int kDevBadToken = 0x2;
constexpr int kDevBadLength = 0x4;
constexpr int kDevCapacity = 0x1;

__device__ __forceinline__ float block_sum(float v, float* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += sh[i];
  return s;
}

// x[m] = E[tok(m)] (fp32), u[m] = RMSNorm(x[m]; gamma) (fp16).
// Slot 0 of each sequence is its last accepted token, slots 1..B-1 the mask
// token (mlx-dspark v0.0.3, "Highlights"; mirror-sd "How It Works").
__global__ void embed_rmsnorm_kernel(const __nv_bfloat16* E, const int* last_tok, int mask_id, int V, int B, int H,
                                     const float* gamma, float eps, float* x, __half* u, int* status) {
  __shared__ float sh[32];
  pdl_wait();
  const int m = blockIdx.x;
  const int j = m / B, slot = m - j * B;
  int tok = slot == 0 ? last_tok[j] : mask_id;
  bool ok = tok >= 0 && tok < V;
  if (!ok && threadIdx.x == 0) atomicOr(status, kDevBadToken);
  const __nv_bfloat16* e = E + (size_t)(ok ? tok : 0) * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    float v = ok ? __bfloat162float(e[i]) : 0.f;
    x[(size_t)m * H + i] = v;
    ss += v * v;
  }
  float tot = block_sum(ss, sh);
  float inv = rsqrtf(tot / H + eps);
  pdl_trigger();
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    u[(size_t)m * H + i] = __float2half_rn(x[(size_t)m * H + i] * inv * gamma[i]);
}

__global__ void rmsnorm_f16_kernel(const float* x, int H, const float* gamma, float eps, __half* u) {
  __shared__ float sh[32];
  pdl_wait();
  const int m = blockIdx.x;
  const float* xr = x + (size_t)m * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    float v = xr[i];
    ss += v * v;
  }
  float inv = rsqrtf(block_sum(ss, sh) / H + eps);
  pdl_trigger();
  for (int i = threadIdx.x; i < H; i += blockDim.x) u[(size_t)m * H + i] = __float2half_rn(xr[i] * inv * gamma[i]);
}

// rows 1..B-1 of every sequence: h = RMSNorm(x; gamma_final) as bf16
__global__ void final_norm_kernel(const float* x, int B, int H, const float* gamma, float eps, __nv_bfloat16* h,
                                  float* hidden_out) {
  __shared__ float sh[32];
  pdl_wait();
  const int o = blockIdx.x;  // output row j (B-1) + i
  const int j = o / (B - 1), i = o - j * (B - 1);
  const float* xr = x + ((size_t)j * B + i + 1) * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    float v = xr[c];
    ss += v * v;
  }
  float inv = rsqrtf(block_sum(ss, sh) / H + eps);
  pdl_trigger();
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    float v = xr[c] * inv * gamma[c];
    h[(size_t)o * H + c] = __float2bfloat16_rn(v);
    if (hidden_out) hidden_out[(size_t)o * H + c] = v;
  }
}

// len[j] += min(n[j] + 1, rows_per_seq) unless that would pass cap
__global__ void commit_len_kernel(int* len, const int* nacc, int b, int rows_per_seq, int cap, int* status) {
  pdl_wait();
  int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= b) return;
  int nn = nacc[j], L = len[j];
  if (nn < -1 || nn > rows_per_seq || L < 0) {
    atomicOr(status, kDevBadLength);
    return;
  }
  int c = min(nn + 1, rows_per_seq);
  if (L + c > cap) {
    atomicOr(status, kDevCapacity);
    return;
  }
  len[j] = L + c;
}

// ------------------------------------------------------- verify-accept ----
// Greedy verify-accept (mirror-sd README, "How It Works", step 3; agentlens
// dflash-mlx, "How it works"): per target row the fp32 argmax (lowest index
// on ties) over a slice of the vocabulary per CTA; the last CTA of a
// sequence (atomic ticket) merges the slices, finds the longest prefix of
// matching drafts, the correction token and the emitted tokens.
struct VerifyArgs {
  const float* logits;
  const int* draft;
  int b, R, D;
  int64_t V;
  int P;
  int64_t chunk;
  int* n_out;
  int* corr_out;
  int* emitted;
  int* next_tok;
  unsigned long long* part;  // [b R][P]
  int* tickets;              // [b]
};

__global__ void __launch_bounds__(256) verify_kernel(const VerifyArgs a) {
  __shared__ unsigned long long sk[8];
  __shared__ int flag;
  __shared__ int amax[64];
  pdl_wait();
  const int row = blockIdx.y, p = blockIdx.x;
  const int j = row / a.R;
  const float* lr = a.logits + (size_t)row * a.V;
  const int64_t c0 = (int64_t)p * a.chunk;
  const int64_t c1 = c0 + a.chunk < a.V ? c0 + a.chunk : a.V;
  unsigned long long best = 0ull;
  if ((a.V & 3) == 0) {
    const float4* l4 = reinterpret_cast<const float4*>(lr);
    for (int64_t i = c0 / 4 + threadIdx.x; i < c1 / 4; i += blockDim.x) {
      float4 v = __ldcs(l4 + i);
      uint32_t b0 = (uint32_t)(4 * i);
      best = umax64(best, argmax_key(v.x, b0));
      best = umax64(best, argmax_key(v.y, b0 + 1));
      best = umax64(best, argmax_key(v.z, b0 + 2));
      best = umax64(best, argmax_key(v.w, b0 + 3));
    }
  } else {
    for (int64_t i = c0 + threadIdx.x; i < c1; i += blockDim.x) best = umax64(best, argmax_key(lr[i], (uint32_t)i));
  }
  best = warp_max64(best);
  if ((threadIdx.x & 31) == 0) sk[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long k = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) k = umax64(k, sk[w]);
    a.part[(size_t)row * a.P + p] = k;
    __threadfence();
    int old = atomicAdd(&a.tickets[j], 1);
    flag = (old == a.R * a.P - 1);
  }
  __syncthreads();
  pdl_trigger();
  if (!flag) return;
  __threadfence();
  for (int r = threadIdx.x; r < a.R; r += blockDim.x) {
    unsigned long long k = 0ull;
    const unsigned long long* pr = a.part + ((size_t)j * a.R + r) * a.P;
    for (int q = 0; q < a.P; ++q) k = umax64(k, __ldcg(pr + q));
    amax[r] = (int)key_index(k);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int* dr = a.draft + (size_t)j * a.D;
    int n = 0;
    while (n < a.D && dr[n] == amax[n]) ++n;
    int corr = n < a.R ? amax[n] : -1;
    a.n_out[j] = n;
    a.corr_out[j] = corr;
    if (a.next_tok) a.next_tok[j] = corr >= 0 ? corr : (n > 0 ? dr[n - 1] : -1);
    a.tickets[j] = 0;
  }
  if (a.emitted) {
    __syncthreads();
    const int* dr = a.draft + (size_t)j * a.D;
    int n = a.n_out[j];
    for (int r = threadIdx.x; r < a.R; r += blockDim.x) {
      int v = -1;
      if (r < n) v = dr[r];
      else if (r == n) v = amax[n];
      a.emitted[(size_t)j * a.R + r] = v;
    }
  }
}

int verify_parts(int b, int R, int64_t V) {
  int rows = b * R;
  int P = (4 * kNumSMs + rows - 1) / rows;
  int64_t pmax = (V + 2047) / 2048;
  if (P > pmax) P = (int)pmax;
  if (P < 1) P = 1;
  return P;
}

}  // namespace

cudaError_t embed_rmsnorm(const __nv_bfloat16* E, const int* last_tok, int mask_id, int V, int b, int B, int H,
                          const float* gamma, float eps, float* x, __half* u, cudaStream_t st, bool pdl,
                          int* status) {
  void* args[] = {&E, &last_tok, &mask_id, &V, &B, &H, &gamma, &eps, &x, &u, &status};
  return launch_k((const void*)embed_rmsnorm_kernel, dim3(b * B), dim3(256), 0, st, pdl, args);
}

cudaError_t rmsnorm_f16(const float* x, int M, int H, const float* gamma, float eps, __half* u, cudaStream_t st,
                        bool pdl) {
  void* args[] = {&x, &H, &gamma, &eps, &u};
  return launch_k((const void*)rmsnorm_f16_kernel, dim3(M), dim3(256), 0, st, pdl, args);
}

cudaError_t final_norm(const float* x, int b, int B, int H, const float* gamma, float eps, __nv_bfloat16* h,
                       float* hidden_out, cudaStream_t st, bool pdl) {
  void* args[] = {&x, &B, &H, &gamma, &eps, &h, &hidden_out};
  return launch_k((const void*)final_norm_kernel, dim3(b * (B - 1)), dim3(256), 0, st, pdl, args);
}

cudaError_t commit_len_update(int* len, const int* nacc, int b, int rows_per_seq, int cap, cudaStream_t st,
                              bool pdl, int* status) {
  void* args[] = {&len, &nacc, &b, &rows_per_seq, &cap, &status};
  return launch_k((const void*)commit_len_kernel, dim3((b + 127) / 128), dim3(128), 0, st, pdl, args);
}

size_t verify_ws_bytes(int b, int R, int64_t V) {
  int P = verify_parts(b, R, V);
  return (size_t)b * R * P * sizeof(unsigned long long) + (size_t)b * sizeof(int) + 256;
}

cudaError_t verify_accept(const float* logits, const int* draft, int b, int R, int D, int64_t V, int* n_out,
                          int* corr_out, int* emitted, int* next_tok, void* ws, cudaStream_t st, bool pdl) {
  VerifyArgs a;
  a.logits = logits;
  a.draft = draft;
  a.b = b;
  a.R = R;
  a.D = D;
  a.V = V;
  a.P = verify_parts(b, R, V);
  a.chunk = (V + a.P - 1) / a.P;
  a.chunk = (a.chunk + 3) / 4 * 4;
  a.n_out = n_out;
  a.corr_out = corr_out;
  a.emitted = emitted;
  a.next_tok = next_tok;
  a.part = reinterpret_cast<unsigned long long*>(ws);
  a.tickets = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws) + (size_t)b * R * a.P * 8);
  void* args[] = {&a};
  return launch_k((const void*)verify_kernel, dim3(a.P, b * R), dim3(256), 0, st, pdl, args);
}

}  // namespace dfl
