// k_lmhead.cu — vocabulary-wide bf16 GEMM with a fused argmax:
//   idx[m] = argmax_v  h[m] . W_lm[v]   (lowest index on ties)
// The drafter reuses the target's lm-head (mlx-dspark v0.0.3 release notes,
// "Highlights"), so every draft step streams the whole [V x H] bf16 table
// once; logits never reach HBM (they are optional, for parity checks only).
//
// Layout: persistent CTAs walk 128-row vocabulary tiles; a producer warp
// streams [128 x 64] bf16 weight boxes and the matching [rows x 64] slice of
// h with 2-D TMA loads (128-byte swizzle) into a 4-stage mbarrier ring;
// four consumer warps own 32 vocabulary rows each (swap-AB: vocabulary rows
// are the MMA's 16-row operand, draft rows the 8-column one).  After each
// tile every lane folds its logits into running (value, index) keys; at the
// end the keys are reduced across lanes with shuffles, across warps in shared
// memory and across CTAs with one 64-bit atomicMax per row.  The last CTA to
// finish (atomic ticket, no spinning) converts keys to indices and re-zeroes
// the workspace for the next call.
#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace dfl {

namespace {

constexpr int kStages = 4;
constexpr int kCW = 4;  // consumer warps
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kWBox = 128 * 128;  // [128 rows][64 bf16] = 16 KB

template <int MT>
struct LG {
  static constexpr int MCH = MT * 8;
  static constexpr int HBYTES = MCH * 128;
  static constexpr int STAGE = kWBox + HBYTES;
  static constexpr size_t SMEM = 1024 + kStages * (size_t)STAGE + 2 * kStages * 8 + 64 + kCW * MCH * 8;
};

struct LmArgs {
  int M, V, H;
  int* idx;
  float* maxlogit;
  float* logits;
  unsigned long long* keys;  // [128] in the workspace
  int* ticket;               // [1]
  int* status;
};

template <int MT>
__global__ void __launch_bounds__(kThreads, 1) lmhead_kernel(const __grid_constant__ CUtensorMap wmap,
                                                              const __grid_constant__ CUtensorMap hmap,
                                                              const LmArgs a) {
  using G = LG<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * G::STAGE);
  uint64_t* empty = full + kStages;
  int* flag = reinterpret_cast<int*>(empty + kStages);
  unsigned long long* red = reinterpret_cast<unsigned long long*>(flag + 16);  // [kCW][MCH]

  const int z = blockIdx.y;
  const int ntiles = (a.V + 127) / 128;
  const int KS = a.H / 64;
  const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int total = my_tiles * KS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kCW) {
    if (lane == 0) {
      prefetch_tmap(&wmap);
      prefetch_tmap(&hmap);
      const uint64_t pol = policy_evict_first();
      const int pre = total < kStages ? total : kStages;
      for (int i = 0; i < pre; ++i) {
        int tile = blockIdx.x + (i / KS) * gridDim.x, ks = i % KS;
        mbar_arrive_expect_tx(&full[i], G::STAGE);
        tma_load_2d_hint(smem + i * G::STAGE, &wmap, ks * 64, tile * 128, &full[i], pol);
      }
      pdl_wait();
      fence_proxy_async_global();  // h was written with generic stores: order the tensor reads after them
      for (int i = 0; i < pre; ++i) {
        int ks = i % KS;
        tma_load_2d(smem + i * G::STAGE + kWBox, &hmap, ks * 64, z * G::MCH, &full[i]);
      }
      for (int i = pre; i < total; ++i) {
        const int slot = i % kStages;
        int tile = blockIdx.x + (i / KS) * gridDim.x, ks = i % KS;
        if (!mbar_wait(&empty[slot], ((i / kStages) - 1) & 1, a.status)) break;
        mbar_arrive_expect_tx(&full[slot], G::STAGE);
        tma_load_2d_hint(smem + slot * G::STAGE, &wmap, ks * 64, tile * 128, &full[slot], pol);
        tma_load_2d(smem + slot * G::STAGE + kWBox, &hmap, ks * 64, z * G::MCH, &full[slot]);
      }
    }
    pdl_trigger();
  } else {
    pdl_wait();
    const int g = lane >> 2, t = lane & 3;
    unsigned long long best[MT][2];
#pragma unroll
    for (int j = 0; j < MT; ++j) best[j][0] = best[j][1] = 0ull;
    float acc[2][MT][4];
    // ldmatrix lane roles
    const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8;  // within a 16-row group
    const int a_ch = lane >> 4;
    const int b_tok = (lane & 7) + ((lane >> 4) << 3);
    const int b_ch = (lane >> 3) & 1;
    bool dead = false;
    for (int i = 0; i < total && !dead; ++i) {
      const int slot = i % kStages, ks = i % KS;
      if (ks == 0) {
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int j = 0; j < MT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[x][j][e] = 0.f;
      }
      if (!mbar_wait(&full[slot], (i / kStages) & 1, a.status)) {
        dead = true;
        break;
      }
      const uint32_t wb = smem_u32(smem + slot * G::STAGE);
      const uint32_t hb = wb + kWBox;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t af[2][4];
#pragma unroll
        for (int mg = 0; mg < 2; ++mg) {
          int row = warp * 32 + mg * 16 + a_row;
          int ch = 2 * kk + a_ch;
          ldsm_x4(wb + row * 128 + ((ch ^ (row & 7)) << 4), af[mg][0], af[mg][1], af[mg][2], af[mg][3]);
        }
#pragma unroll
        for (int p = 0; p < MT / 2; ++p) {
          int tok = p * 16 + b_tok;
          int ch = 2 * kk + b_ch;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(hb + tok * 128 + ((ch ^ (tok & 7)) << 4), b0, b1, b2, b3);
          mma_bf16(acc[0][2 * p], af[0], b0, b1);
          mma_bf16(acc[1][2 * p], af[1], b0, b1);
          mma_bf16(acc[0][2 * p + 1], af[0], b2, b3);
          mma_bf16(acc[1][2 * p + 1], af[1], b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (ks == KS - 1) {
        const int tile = blockIdx.x + (i / KS) * gridDim.x;
#pragma unroll
        for (int mg = 0; mg < 2; ++mg)
#pragma unroll
          for (int j = 0; j < MT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              int v = tile * 128 + warp * 32 + mg * 16 + g + ((e >> 1) << 3);
              int m = z * G::MCH + j * 8 + 2 * t + (e & 1);
              if (v < a.V) {
                float val = acc[mg][j][e];
                best[j][e & 1] = umax64(best[j][e & 1], argmax_key(val, (uint32_t)v));
                if (a.logits && m < a.M) a.logits[(size_t)m * a.V + v] = val;
              }
            }
      }
    }
    // reduce over the 8 row-groups (lanes with equal t)
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        unsigned long long k = best[j][c];
        k = umax64(k, __shfl_xor_sync(0xffffffffu, k, 4));
        k = umax64(k, __shfl_xor_sync(0xffffffffu, k, 8));
        k = umax64(k, __shfl_xor_sync(0xffffffffu, k, 16));
        if (g == 0) red[warp * G::MCH + j * 8 + 2 * t + c] = k;
      }
    pdl_trigger();
  }
  __syncthreads();
  if (threadIdx.x < G::MCH) {
    unsigned long long k = 0ull;
#pragma unroll
    for (int w = 0; w < kCW; ++w) k = umax64(k, red[w * G::MCH + threadIdx.x]);
    int m = z * G::MCH + threadIdx.x;
    if (m < a.M && k != 0ull) atomicMax(&a.keys[m], k);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int old = atomicAdd(a.ticket, 1);
    *flag = (old == (int)(gridDim.x * gridDim.y) - 1);
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  for (int m = threadIdx.x; m < a.M; m += blockDim.x) {
    unsigned long long k = atomicExch(&a.keys[m], 0ull);
    a.idx[m] = (int)key_index(k);
    if (a.maxlogit) a.maxlogit[m] = key_value(k);
  }
  if (threadIdx.x == 0) *a.ticket = 0;
}

// ---- tensor-memory path (33 to 128 rows) --------------------------------
// D[token][vocabulary row] = h . W^T with tcgen05.mma (M = 128 token rows,
// N = 256 vocabulary rows per tile, K = 16, bf16 operands from 128-byte
// swizzled shared memory, fp32 accumulator in tensor memory).  Persistent
// CTAs (one per SM: the kernel holds the SM's 512 tensor-memory columns)
// walk 256-row vocabulary tiles; a producer warp streams [256 x 64] weight
// boxes and the matching [128 x 64] box of h into a 4-stage ring, one thread
// issues the MMAs into two accumulators (tile t into buffer t % 2), and four
// epilogue warps read a finished accumulator back while the next tile
// accumulates: thread r owns token row r, so its argmax over the tile's 256
// logits needs no exchange.  Keys are folded across CTAs as in the
// warp-level path.
constexpr int kTcV = 256;                       // vocabulary rows per tile (MMA N)
constexpr int kTcStages = 4;
constexpr int kTcWarps = 6;                     // 4 epilogue, producer, MMA
constexpr int kTcWBytes = kTcV * 128;           // [256 rows][64 bf16]
constexpr int kTcHBytes = 128 * 128;            // [128 rows][64 bf16]
constexpr int kTcStage = kTcWBytes + kTcHBytes;  // 48 KB, a 1 KB multiple
constexpr size_t kTcSmem = 1024 + kTcStages * (size_t)kTcStage + 256;

__global__ void __launch_bounds__(kTcWarps * 32, 1) lmhead_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                     const __grid_constant__ CUtensorMap hmap,
                                                                     const LmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTcStages * kTcStage);
  uint64_t* empty = full + kTcStages;  // 1 MMA commit
  uint64_t* dfull = empty + kTcStages;  // [2] accumulator complete (commit)
  uint64_t* dfree = dfull + 2;          // [2] accumulator read back (4 epilogue warps)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(dfree + 2);
  int* flag = reinterpret_cast<int*>(s_tmem + 1);

  const int ntiles = (a.V + kTcV - 1) / kTcV;
  const int KS = a.H / 64;
  const int my_tiles = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int total = my_tiles * KS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dfree[b], 4);
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(s_tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 4) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tmap(&wmap);
      prefetch_tmap(&hmap);
      const uint64_t pol = policy_evict_first();
      const int pre = total < kTcStages ? total : kTcStages;
      for (int i = 0; i < pre; ++i) {  // weights need nothing from the preceding kernel
        const int tile = blockIdx.x + (i / KS) * gridDim.x, ks = i % KS;
        mbar_arrive_expect_tx(&full[i], kTcStage);
        tma_load_2d_hint(smem + i * kTcStage, &wmap, ks * 64, tile * kTcV, &full[i], pol);
      }
      pdl_wait();
      fence_proxy_async_global();  // h was written with generic stores: order the tensor reads after them
      for (int i = 0; i < pre; ++i)
        tma_load_2d(smem + i * kTcStage + kTcWBytes, &hmap, (i % KS) * 64, 0, &full[i]);
      for (int i = pre; i < total; ++i) {
        const int slot = i % kTcStages;
        const int tile = blockIdx.x + (i / KS) * gridDim.x, ks = i % KS;
        if (!mbar_wait(&empty[slot], ((i / kTcStages) - 1) & 1, a.status)) break;
        mbar_arrive_expect_tx(&full[slot], kTcStage);
        tma_load_2d_hint(smem + slot * kTcStage, &wmap, ks * 64, tile * kTcV, &full[slot], pol);
        tma_load_2d(smem + slot * kTcStage + kTcWBytes, &hmap, ks * 64, 0, &full[slot]);
      }
    }
    pdl_trigger();
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc_idesc_bf16(128, kTcV);
      for (int t = 0; t < my_tiles; ++t) {
        const int db = t & 1;
        if (t >= 2 && !mbar_wait(&dfree[db], ((t >> 1) - 1) & 1, a.status)) break;
        tc_fence_after();
        for (int ks = 0; ks < KS; ++ks) {
          const int i = t * KS + ks, slot = i % kTcStages;
          if (!mbar_wait(&full[slot], (i / kTcStages) & 1, a.status)) break;
          tc_fence_after();
          const uint32_t wb = smem_u32(smem + slot * kTcStage);
          const uint32_t hb = wb + kTcWBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_ss(tmem + db * kTcV, tc_sdesc_sw128(hb + kk * 32), tc_sdesc_sw128(wb + kk * 32), idesc,
                      (ks | kk) != 0);
          tc_commit(&empty[slot]);
        }
        tc_commit(&dfull[db]);
      }
    }
    pdl_trigger();
  } else {
    // ------- epilogue warps 0..3: thread r holds token row r of the accumulator -------
    pdl_wait();
    const int r = warp * 32 + lane;
    const int m = r;
    unsigned long long best = 0ull;
    for (int t = 0; t < my_tiles; ++t) {
      const int db = t & 1;
      if (!mbar_wait(&dfull[db], (t >> 1) & 1, a.status)) break;
      tc_fence_after();
      const int v0 = (blockIdx.x + t * gridDim.x) * kTcV;
      const uint32_t td = tmem + ((uint32_t)(warp * 32) << 16) + db * kTcV;
#pragma unroll 1
      for (int c0 = 0; c0 < kTcV; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(td + c0, v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int vv = v0 + c0 + j;
          const float val = __uint_as_float(v[j]);
          if (vv < a.V) {
            best = umax64(best, argmax_key(val, (uint32_t)vv));
            if (a.logits && m < a.M) a.logits[(size_t)m * a.V + vv] = val;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dfree[db]);
    }
    if (m < a.M && best != 0ull) atomicMax(&a.keys[m], best);
    pdl_trigger();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int old = atomicAdd(a.ticket, 1);
    *flag = (old == (int)(gridDim.x * gridDim.y) - 1);
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  for (int mm = threadIdx.x; mm < a.M; mm += blockDim.x) {
    unsigned long long k = atomicExch(&a.keys[mm], 0ull);
    a.idx[mm] = (int)key_index(k);
    if (a.maxlogit) a.maxlogit[mm] = key_value(k);
  }
  if (threadIdx.x == 0) *a.ticket = 0;
}

}  // namespace

size_t lmhead_ws_bytes(int64_t M) { return 128 * sizeof(unsigned long long) + 256; }

static bool lmhead_uses_tc(int M, int H) { return M > 32 && M <= 128 && H % 64 == 0; }

int lmhead_tile_rows(int M, int H) { return lmhead_uses_tc(M, H) ? kTcV : 128; }

int lmhead_first_tiles(int M, int V, int H) {
  if (lmhead_uses_tc(M, H)) {  // one CTA per SM over 256-row tiles
    const int ntiles = (V + kTcV - 1) / kTcV;
    return ntiles < num_sms() ? ntiles : num_sms();
  }
  const int chunks = (M + (M <= 16 ? 16 : 32) - 1) / (M <= 16 ? 16 : 32);
  const int ntiles = (V + 127) / 128;
  int per_chunk = (2 * num_sms()) / chunks;
  if (per_chunk < 1) per_chunk = 1;
  return ntiles < per_chunk ? ntiles : per_chunk;  // one CTA per tile of the first round
}

cudaError_t lmhead_argmax(const __nv_bfloat16* h, const __nv_bfloat16* w, int M, int V, int H, int* idx_out,
                          float* maxlogit, float* logits, void* ws, cudaStream_t st, bool pdl, int* status) {
  const int mt = M <= 16 ? 2 : 4;
  const int mch = mt * 8;
  const int chunks = (M + mch - 1) / mch;
  LmArgs a;
  a.M = M;
  a.V = V;
  a.H = H;
  a.idx = idx_out;
  a.maxlogit = maxlogit;
  a.logits = logits;
  a.keys = reinterpret_cast<unsigned long long*>(ws);
  a.ticket = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws) + 128 * sizeof(unsigned long long));
  a.status = status;
  CUtensorMap wm, hm;
  if (!encode_tmap_2d(&wm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, 64, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&hm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, (uint64_t)H, (uint64_t)M, (uint64_t)H * 2, 64,
                      (uint32_t)mch, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (lmhead_uses_tc(M, H)) {
    // tensor-memory path: one chunk of up to 128 rows, one CTA per SM
    CUtensorMap wt, ht;
    if (!encode_tmap_2d(&wt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, 64,
                        kTcV, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tmap_2d(&ht, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h, (uint64_t)H, (uint64_t)M, (uint64_t)H * 2, 64,
                        128, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    dim3 tgrid(lmhead_first_tiles(M, V, H), 1);
    void* targs[] = {&wt, &ht, &a};
    cudaFuncSetAttribute((const void*)lmhead_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    return launch_k((const void*)lmhead_tc_kernel, tgrid, dim3(kTcWarps * 32), kTcSmem, st, pdl, targs);
  }
  dim3 grid(lmhead_first_tiles(M, V, H), chunks);
  void* args[] = {&wm, &hm, &a};
  if (mt == 2) {
    cudaFuncSetAttribute((const void*)lmhead_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)LG<2>::SMEM);
    return launch_k((const void*)lmhead_kernel<2>, grid, dim3(kThreads), LG<2>::SMEM, st, pdl, args);
  }
  cudaFuncSetAttribute((const void*)lmhead_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)LG<4>::SMEM);
  return launch_k((const void*)lmhead_kernel<4>, grid, dim3(kThreads), LG<4>::SMEM, st, pdl, args);
}

}  // namespace dfl
