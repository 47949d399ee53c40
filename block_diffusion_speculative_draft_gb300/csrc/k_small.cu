// k_small.cu — the latency-sized kernels of the step: block embedding + first
// RMSNorm, RMSNorm, final norm, commit-length update and the greedy
// verify-accept; plus the launch and tensor-map helpers shared by all
// kernels.
#include <atomic>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace dfl {

// ------------------------------------------------------------- helpers ----
// Launch mode (dflash_set_launch_mode): 0 = stream order, 1 = early launch.
static std::atomic<int> g_launch_mode{0};

bool launch_early() { return g_launch_mode.load(std::memory_order_relaxed) == 1; }
void set_launch_mode(int mode) { g_launch_mode.store(mode, std::memory_order_relaxed); }
int get_launch_mode() { return g_launch_mode.load(std::memory_order_relaxed); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    cache[dev] = n;
  }
  return cache[dev];
}

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
  cfg.numAttrs = pdl && launch_early() ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_kc(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl, dim3 cluster,
                      void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl && launch_early()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster.x * cluster.y * cluster.z > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster.x;
    attr[n].val.clusterDim.y = cluster.y;
    attr[n].val.clusterDim.z = cluster.z;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
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

bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const uint64_t dims[3],
                    const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle swz) {
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
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
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

constexpr int kNormThreads = 256;
constexpr int kNormVec = 8;  // float4 per thread: rows up to 8192 wide

// Loads a fp32 row into registers (all loads issued before any use) and
// returns its sum of squares over the block.
__device__ __forceinline__ float load_row(const float* xr, int H, float4 (&v)[kNormVec], float* sh) {
  const int n4 = H >> 2;
  const float4* x4 = reinterpret_cast<const float4*>(xr);
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    int c = threadIdx.x + i * kNormThreads;
    v[i] = c < n4 ? x4[c] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  return block_sum(ss, sh);
}

__device__ __forceinline__ void store_f16_row(__half* ur, int H, const float4 (&v)[kNormVec], float inv,
                                              const float* gamma) {
  const int n4 = H >> 2;
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    int c = threadIdx.x + i * kNormThreads;
    if (c < n4) {
      float4 g = g4[c];
      __half2 a = __floats2half2_rn(v[i].x * inv * g.x, v[i].y * inv * g.y);
      __half2 b = __floats2half2_rn(v[i].z * inv * g.z, v[i].w * inv * g.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&a);
      pk.y = *reinterpret_cast<uint32_t*>(&b);
      reinterpret_cast<uint2*>(ur)[c] = pk;
    }
  }
}

// x[m] = E[tok(m)] (fp32), u[m] = RMSNorm(x[m]; gamma) (fp16).
// Slot 0 of each sequence is its last accepted token, slots 1..B-1 the mask
// token (mlx-dspark v0.0.3, "Highlights"; mirror-sd "How It Works").
__global__ void __launch_bounds__(kNormThreads) embed_rmsnorm_kernel(const __nv_bfloat16* E, const int* last_tok,
                                                                    int mask_id, int V, int B, int H,
                                                                    const float* gamma, float eps, float* x,
                                                                    __half* u, float* ss_out, int* status) {
  __shared__ float sh[32];
  pdl_wait();
  const int m = blockIdx.x;
  const int j = m / B, slot = m - j * B;
  int tok = slot == 0 ? last_tok[j] : mask_id;
  bool ok = tok >= 0 && tok < V;
  if (!ok && threadIdx.x == 0) atomicOr(status, kDevBadToken);
  const uint2* e4 = reinterpret_cast<const uint2*>(E + (size_t)(ok ? tok : 0) * H);  // 4 bf16 per uint2
  const int n4 = H >> 2;
  float4 v[kNormVec];
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    int c = threadIdx.x + i * kNormThreads;
    uint2 w = (ok && c < n4) ? e4[c] : make_uint2(0u, 0u);
    v[i].x = __uint_as_float(w.x << 16);
    v[i].y = __uint_as_float(w.x & 0xFFFF0000u);
    v[i].z = __uint_as_float(w.y << 16);
    v[i].w = __uint_as_float(w.y & 0xFFFF0000u);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  float inv = 1.f;
  if (ss_out) {
    // deferred RMSNorm: per-128-column sums of squares; for a given i one
    // warp holds one column tile (n4 is a multiple of 32)
#pragma unroll
    for (int i = 0; i < kNormVec; ++i) {
      const int c0 = (threadIdx.x & ~31) + i * kNormThreads;
      if (c0 < n4) {
        float q = v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
        if ((threadIdx.x & 31) == 0) ss_out[(size_t)m * (H >> 7) + (c0 >> 5)] = q;
      }
    }
  } else {
    inv = rsqrtf(block_sum(ss, sh) / H + eps);
  }
  pdl_trigger();
  float4* xr = reinterpret_cast<float4*>(x + (size_t)m * H);
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    int c = threadIdx.x + i * kNormThreads;
    if (c < n4) xr[c] = v[i];
  }
  store_f16_row(u + (size_t)m * H, H, v, inv, gamma);
  fence_proxy_async_global();  // the next GEMM reads u with TMA
}


// rows 1..B-1 of every sequence: h = RMSNorm(x; gamma_final) as bf16
__global__ void __launch_bounds__(kNormThreads) final_norm_kernel(const float* x, int B, int H, const float* gamma,
                                                                 float eps, __nv_bfloat16* h, float* hidden_out) {
  __shared__ float sh[32];
  pdl_wait();
  const int o = blockIdx.x;  // output row j (B-1) + i
  const int j = o / (B - 1), i = o - j * (B - 1);
  float4 v[kNormVec];
  float inv = rsqrtf(load_row(x + ((size_t)j * B + i + 1) * H, H, v, sh) / H + eps);
  pdl_trigger();
  const int n4 = H >> 2;
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
#pragma unroll
  for (int q = 0; q < kNormVec; ++q) {
    int c = threadIdx.x + q * kNormThreads;
    if (c < n4) {
      float4 g = g4[c];
      float4 y = make_float4(v[q].x * inv * g.x, v[q].y * inv * g.y, v[q].z * inv * g.z, v[q].w * inv * g.w);
      __nv_bfloat162 a = __floats2bfloat162_rn(y.x, y.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(y.z, y.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&a);
      pk.y = *reinterpret_cast<uint32_t*>(&b);
      reinterpret_cast<uint2*>(h + (size_t)o * H)[c] = pk;
      if (hidden_out) reinterpret_cast<float4*>(hidden_out + (size_t)o * H)[c] = y;
    }
  }
  fence_proxy_async_global();  // the lm-head reads h with TMA
}

// len[j] += min(n[j] + 1, rows_per_seq) unless that would pass cap.
// Deliberately no early trigger (griddepcontrol.launch_dependents): the next
// draft pass's kernels then start only after this one has completed, which is
// what lets its attention read len (and the committed context K/V) before its
// own dependency wait.
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
    const int64_t e4 = c1 / 4;
    for (int64_t i0 = c0 / 4 + threadIdx.x; i0 < e4; i0 += 4 * (int64_t)blockDim.x) {
      float4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int64_t i = i0 + q * (int64_t)blockDim.x;
        v[q] = i < e4 ? __ldcs(l4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int64_t i = i0 + q * (int64_t)blockDim.x;
        if (i < e4) {
          uint32_t b0 = (uint32_t)(4 * i);
          best = umax64(best, argmax_key(v[q].x, b0));
          best = umax64(best, argmax_key(v[q].y, b0 + 1));
          best = umax64(best, argmax_key(v[q].z, b0 + 2));
          best = umax64(best, argmax_key(v[q].w, b0 + 3));
        }
      }
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
  // merge the P slices of every row: one warp per row, lanes over slices
  for (int r = threadIdx.x >> 5; r < a.R; r += blockDim.x >> 5) {
    const unsigned long long* pr = a.part + ((size_t)j * a.R + r) * a.P;
    unsigned long long k = 0ull;
    for (int q = (threadIdx.x & 31); q < a.P; q += 32) k = umax64(k, __ldcg(pr + q));
    k = warp_max64(k);
    if ((threadIdx.x & 31) == 0) amax[r] = (int)key_index(k);
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
  int P = (4 * num_sms() + rows - 1) / rows;
  int64_t pmax = (V + 2047) / 2048;
  if (P > pmax) P = (int)pmax;
  if (P < 1) P = 1;
  return P;
}

}  // namespace

cudaError_t embed_rmsnorm(const __nv_bfloat16* E, const int* last_tok, int mask_id, int V, int b, int B, int H,
                          const float* gamma, float eps, float* x, __half* u, float* ss_out, cudaStream_t st,
                          bool pdl, int* status) {
  void* args[] = {&E, &last_tok, &mask_id, &V, &B, &H, &gamma, &eps, &x, &u, &ss_out, &status};
  return launch_k((const void*)embed_rmsnorm_kernel, dim3(b * B), dim3(kNormThreads), 0, st, pdl, args);
}


cudaError_t final_norm(const float* x, int b, int B, int H, const float* gamma, float eps, __nv_bfloat16* h,
                       float* hidden_out, cudaStream_t st, bool pdl) {
  void* args[] = {&x, &B, &H, &gamma, &eps, &h, &hidden_out};
  return launch_k((const void*)final_norm_kernel, dim3(b * (B - 1)), dim3(kNormThreads), 0, st, pdl, args);
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

// ------------------------------------------- allocation-free verify ----
// Scratch for callers that cannot allocate device memory: a fixed array in
// this library's device image, present on every GPU that loads the library
// until the process exits.  Layout: per-sequence tickets at offset 0, the
// per-slice argmax keys from offset kNoAllocTicketBytes.
constexpr size_t kNoAllocTicketBytes = 4096;
static __device__ __align__(256) unsigned char g_verify_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};
}  // namespace

size_t verify_noalloc_need(int b, int R, int64_t V) {
  int P = verify_parts(b, R, V);
  if ((size_t)b * sizeof(int) > kNoAllocTicketBytes) return (size_t)-1;
  return kNoAllocTicketBytes + (size_t)b * R * P * sizeof(unsigned long long);
}

cudaError_t verify_accept_noalloc(const float* logits, const int* draft, int b, int R, int D, int64_t V, int* n_out,
                                  int* corr_out, int* emitted, int* next_tok, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      // device-side address of the scratch array on the current device
      e = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_verify_scratch);
      if (e != cudaSuccess) {
        g_scratch_ptr[dev] = nullptr;
        return e;
      }
    }
    base = g_scratch_ptr[dev];
  }
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
  a.tickets = static_cast<int*>(base);
  a.part = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(base) + kNoAllocTicketBytes);
  // tickets must start at zero whatever an earlier (possibly failed) call left
  e = cudaMemsetAsync(a.tickets, 0, (size_t)b * sizeof(int), st);
  if (e != cudaSuccess) return e;
  void* args[] = {&a};
  return launch_k((const void*)verify_kernel, dim3(a.P, b * R), dim3(256), 0, st, false, args);
}

}  // namespace dfl
