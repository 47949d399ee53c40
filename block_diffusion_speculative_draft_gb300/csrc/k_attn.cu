// k_attn.cu — block attention of the drafter:
//   o = softmax(q [K_ctx || K_blk]^T / sqrt(d)) [V_ctx || V_blk]
// non-causal (the whole block is drafted in one parallel pass: mlx-dspark
// v0.0.3 release notes, "Highlights"), GQA, over the sequence's committed
// context K/V followed by the block's own K/V.
//
// One CTA per (context split, kv head, sequence).  The B block rows times the
// nq/nkv query heads that share a kv head form one query tile (64 rows for
// B = 16, group 4), so every K/V byte is read once per kv head.  One compute
// warp per 16 query rows; as many helper warps again (up to 10 warps in all)
// share the copies and the split merge, which are latency-bound, and, when a
// split spans several tiles, compute the second key half of every tile.  Long contexts
// are split along the keys (flash-decoding; the pages' long-context verify
// likewise uses a two-pass attention, dflash-mlx summary, "기술적 도전":
// JIT SDPA 2-pass for N >= 1024): the splits of one (sequence, kv head) form
// a thread-block cluster; each keeps an online softmax, leaves its normalised
// partial output and log-sum-exp in shared memory, and after a cluster
// barrier every CTA merges one slice of query rows over all splits through
// distributed shared memory, in split order.  Q.K^T and P.V run on m16n8k16
// tensor-core MMAs with fp32 accumulation; K/V tiles of 64 keys are
// double-buffered with cp.async into XOR-swizzled shared memory.
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kMaxSplits = 16;  // one (non-portable) cluster of splits
constexpr int kPortable = 8;    // largest cluster every sm_90+ part accepts
constexpr int kKT = 64;         // keys per tile

// keys [k0, k1) of split sp out of ns equal, 64-aligned chunks of `total`
__device__ __forceinline__ void split_range(int total, int sp, int ns, int& k0, int& k1) {
  int chunk = (total + ns - 1) / ns;
  chunk = (chunk + kKT - 1) / kKT * kKT;
  k0 = min(total, sp * chunk);
  k1 = min(total, k0 + chunk);
}

template <int D, int KH>
__global__ void __launch_bounds__(320, 1) attn_kernel(const AttnArgs a) {
  constexpr int RB = D * 2;  // bytes per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int sp = blockIdx.x, g = blockIdx.y, j = blockIdx.z;
  const int ns = gridDim.x;
  const int grp = a.nq / a.nkv;
  const int rows = a.B * grp;
  const int nwc = a.nwc;
  const int rows_pad = nwc * 16;
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + rows_pad * RB;        // [2][64][D]
  uint8_t* sV = sK + 2 * kKT * RB;         // [2][64][D]
  float* sLse = reinterpret_cast<float*>(sV + 2 * kKT * RB);  // [rows_pad]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // The context K/V and its length are inputs of the whole draft pass (no
  // kernel of the pass writes them), so the first tile's context keys are
  // fetched before waiting for the kernel that produces q and the block K/V.
  // (a commit folded into this pass appends rows [Lold, L), written by this
  // layer's QKV kernel: those are read only after the wait)
  int L = a.len[j];
  if (L < 0) L = 0;
  if (L > a.cap) L = a.cap;
  const int Lold = L;
  if (a.nacc) L += commit_count(a.len[j], a.nacc[j], a.rps, a.cap);
  const int total = L + a.B;
  int k0, k1;
  split_range(total, sp, ns, k0, k1);

  // part 0: context keys t < Lold only; 1: the rest (appended context rows,
  // block keys, zero fill); 2: all
  auto load_kv = [&](int buf, int t0, int part) {
    for (int c = threadIdx.x; c < kKT * (D / 8); c += blockDim.x) {
      int r = c / (D / 8), ch = c % (D / 8);
      int t = t0 + r;
      bool ok = t < k1;
      const bool ctx = ok && t < L;
      const bool old_ctx = ok && t < Lold;
      if (part == 0 && !old_ctx) continue;
      if (part == 1 && old_ctx) continue;
      const __half* ks = a.kc;
      const __half* vs = a.vc;
      if (ok) {
        if (ctx) {
          size_t off = (((size_t)j * a.nkv + g) * a.cap + t) * D + ch * 8;
          ks = a.kc + off;
          vs = a.vc + off;
        } else {
          size_t off = ((size_t)(j * a.B + (t - L)) * a.nkv + g) * D + ch * 8;
          ks = a.kblk + off;
          vs = a.vblk + off;
        }
      }
      int so = buf * kKT * RB + r * RB + ((ch ^ (r & 7)) << 4);
      cp_async16(sK + so, ks, ok);
      cp_async16(sV + so, vs, ok);
    }
  };
  const int ntile = (k1 - k0 + kKT - 1) / kKT;
  load_kv(0, k0, 0);
  if (a.pf_base && threadIdx.x == 0)
    prefetch_l2_job(a.pf_base, a.pf_stride, a.pf_bytes, a.pf_i0, a.pf_i1,
                    blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z), gridDim.x * gridDim.y * gridDim.z);
  pdl_wait();

  // ---- Q tile: row rho = tok * grp + hh  ->  q[(j B + tok)][g grp + hh][:]
  for (int c = threadIdx.x; c < rows_pad * (D / 8); c += blockDim.x) {
    int rho = c / (D / 8), ch = c % (D / 8);
    bool ok = rho < rows;
    const __half* src = a.q;
    if (ok) {
      int tok = rho / grp, hh = rho - tok * grp;
      src = a.q + ((size_t)(j * a.B + tok) * a.nq + (g * grp + hh)) * D + ch * 8;
    }
    cp_async16(sQ + rho * RB + ((ch ^ (rho & 7)) << 4), src, ok);
  }
  load_kv(0, k0, 1);
  cp_async_commit();

  const float sl2 = rsqrtf((float)D) * 1.4426950408889634f;
  const int g8 = lane >> 2, t4 = lane & 3;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  uint32_t qf[D / 16][4];

  // KH = 2: warp w computes row block w % nwc over key half w / nwc of every
  // tile, each half with its own online softmax, merged once after the last
  // tile; KH = 1: one warp per row block over all 64 keys of a tile
  constexpr int KK = kKT / KH;  // keys per warp and tile
  constexpr int NN = KK / 8;    // n8 score tiles per warp
  const int rb = warp % nwc, half = warp / nwc;
  const bool cw = warp < nwc * KH;
  for (int it = 0; it < ntile; ++it) {
    if (it + 1 < ntile) load_kv((it + 1) & 1, k0 + (it + 1) * kKT, 2);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (cw) {
      if (it == 0) {
        const uint32_t qb = smem_u32(sQ);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          int row = rb * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          int ch = 2 * ks + (lane >> 4);
          ldsm_x4(qb + row * RB + ((ch ^ (row & 7)) << 4), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
        }
      }
      const int buf = it & 1;
      const uint32_t kb = smem_u32(sK + buf * kKT * RB);
      const uint32_t vb = smem_u32(sV + buf * kKT * RB);
      // S = Q K^T : 16 rows x KK keys per warp
      float s[NN][4];
#pragma unroll
      for (int n = 0; n < NN; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int n16 = 0; n16 < NN / 2; ++n16) {
          int key = half * KK + n16 * 16 + (lane & 7) + ((lane >> 4) << 3);
          int ch = 2 * ks + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + key * RB + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
          mma_f16(s[2 * n16], qf[ks], b0, b1);
          mma_f16(s[2 * n16 + 1], qf[ks], b2, b3);
        }
      }
      // scale, mask, online softmax (rows g8 and g8 + 8 of this warp); a half
      // may see no valid key yet: its max stays -inf and contributes nothing
      const int kbase = k0 + it * kKT + half * KK;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int n = 0; n < NN; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          int key = kbase + n * 8 + 2 * t4 + (e & 1);
          float v = key < k1 ? s[n][e] * sl2 : -INFINITY;
          s[n][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      }
      float corr[2], mnew[2], rs[2] = {0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mnew[r] = fmaxf(mrow[r], mx[r]);
        corr[r] = mnew[r] == -INFINITY ? 1.f : exp2f(mrow[r] - mnew[r]);
        mrow[r] = mnew[r];
      }
      uint32_t pf[NN / 2][4];  // P as the A operand of P.V, k16 steps over KK keys
#pragma unroll
      for (int n = 0; n < NN; ++n) {
        const float q0 = mnew[0] == -INFINITY ? 0.f : mnew[0];
        const float q1 = mnew[1] == -INFINITY ? 0.f : mnew[1];
        float p0 = exp2f(s[n][0] - q0);
        float p1 = exp2f(s[n][1] - q0);
        float p2 = exp2f(s[n][2] - q1);
        float p3 = exp2f(s[n][3] - q1);
        rs[0] += p0 + p1;
        rs[1] += p2 + p3;
        __half2 h01 = __floats2half2_rn(p0, p1);
        __half2 h23 = __floats2half2_rn(p2, p3);
        pf[n >> 1][(n & 1) * 2 + 0] = *reinterpret_cast<uint32_t*>(&h01);
        pf[n >> 1][(n & 1) * 2 + 1] = *reinterpret_cast<uint32_t*>(&h23);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
        rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
        lrow[r] = lrow[r] * corr[r] + rs[r];
      }
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= corr[0];
        o[i][1] *= corr[0];
        o[i][2] *= corr[1];
        o[i][3] *= corr[1];
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < NN / 2; ++kk) {
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          int key = half * KK + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          int ch = 2 * dp + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + key * RB + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
          mma_f16(o[2 * dp], pf[kk], b0, b1);
          mma_f16(o[2 * dp + 1], pf[kk], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  if (KH == 2) {
    // merge the key halves of each row block: half 1 hands (max, sum, O) over
    // through shared memory (the K/V buffers are free once the copies land)
    constexpr int XS = D + 4;  // row stride (floats)
    cp_async_wait<0>();
    __syncthreads();
    float* xo = reinterpret_cast<float*>(sK);  // [nwc][16][XS]
    float* xm = xo + (size_t)nwc * 16 * XS;    // [nwc][16]
    float* xl = xm + nwc * 16;                 // [nwc][16]
    if (cw && half == 1) {
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          xo[(rb * 16 + g8 + ((e >> 1) << 3)) * XS + i * 8 + 2 * t4 + (e & 1)] = o[i][e];
      if (t4 == 0) {
        xm[rb * 16 + g8] = mrow[0];
        xm[rb * 16 + g8 + 8] = mrow[1];
        xl[rb * 16 + g8] = lrow[0];
        xl[rb * 16 + g8 + 8] = lrow[1];
      }
    }
    __syncthreads();
    if (cw && half == 0) {
      float c0[2], c1[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float m1 = xm[rb * 16 + g8 + 8 * r], l1 = xl[rb * 16 + g8 + 8 * r];
        const float mn = fmaxf(mrow[r], m1);
        c0[r] = mrow[r] == -INFINITY ? 0.f : exp2f(mrow[r] - mn);
        c1[r] = m1 == -INFINITY ? 0.f : exp2f(m1 - mn);
        lrow[r] = lrow[r] * c0[r] + l1 * c1[r];
        mrow[r] = mn;
      }
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[i][e] = o[i][e] * c0[e >> 1] +
                    xo[(rb * 16 + g8 + ((e >> 1) << 3)) * XS + i * 8 + 2 * t4 + (e & 1)] * c1[e >> 1];
    }
  }
  pdl_trigger();

  // normalise this split's rows; log2-domain log-sum-exp (-inf when empty)
  float inv[2], lse[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    inv[r] = lrow[r] > 0.f ? 1.f / lrow[r] : 0.f;
    lse[r] = lrow[r] > 0.f ? mrow[r] + log2f(lrow[r]) : -INFINITY;
  }
  if (ns == 1) {
    if (warp < nwc)
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int rho = warp * 16 + g8 + ((e >> 1) << 3);
        if (rho >= rows) continue;
        int tok = rho / grp, hh = rho - tok * grp;
        int dim = i * 8 + 2 * t4 + (e & 1);
        a.out[((size_t)(j * a.B + tok) * a.nq + g * grp + hh) * D + dim] = __float2half_rn(o[i][e] * inv[e >> 1]);
      }
    fence_proxy_async_global();  // the o projection reads the output with TMA
    return;
  }
  // Push this split's normalised partial rows and log-sum-exps into the
  // shared memory of the CTA that owns them (CTA p merges rows
  // [p rows / ns, (p + 1) rows / ns)); remote stores do not wait for a reply,
  // and the owner then merges from its own shared memory.  The receive area
  // is separate from Q/K/V, so no barrier is needed before the pushes.
  const int maxr = (rows + ns - 1) / ns;
  constexpr int RS = D + 4;  // row stride (floats): conflict-free float2 stores
  float* rO = reinterpret_cast<float*>(sLse + rows_pad);  // [ns][maxr][RS]
  float* rL = rO + (size_t)ns * maxr * RS;                 // [ns][maxr]
  const uint32_t rObase = smem_u32(rO), rLbase = smem_u32(rL);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (warp >= nwc) break;
    const int rho = warp * 16 + g8 + 8 * h;
    if (rho >= rows) continue;
    const int own = ((rho + 1) * ns - 1) / rows;
    const int lr = rho - (own * rows) / ns;
    const uint32_t dst = dsmem_addr(rObase + (uint32_t)((sp * maxr + lr) * RS + 2 * t4) * 4u, (uint32_t)own);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) st_dsmem_f2(dst + i * 32u, o[i][2 * h] * inv[h], o[i][2 * h + 1] * inv[h]);
    if (t4 == 0) st_dsmem_f32(dsmem_addr(rLbase + (uint32_t)(sp * maxr + lr) * 4u, (uint32_t)own), lse[h]);
  }
  cp_async_wait<0>();  // an empty split may still have zero-fill copies in flight
  cluster_sync();      // every push into this CTA is visible
  // merge the owned rows over the ns splits, in split order
  const int r0 = (sp * rows) / ns, r1 = ((sp + 1) * rows) / ns;
  for (int it = threadIdx.x; it < (r1 - r0) * (D / 4); it += blockDim.x) {
    const int lr = it / (D / 4), c4 = it % (D / 4);
    float mmax = -INFINITY;
    for (int s2 = 0; s2 < ns; ++s2) mmax = fmaxf(mmax, rL[s2 * maxr + lr]);
    float den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s2 = 0; s2 < ns; ++s2) {
      const float w = exp2f(rL[s2 * maxr + lr] - mmax);
      const float4 ov = *reinterpret_cast<const float4*>(rO + (size_t)(s2 * maxr + lr) * RS + 4 * c4);
      den += w;
      num.x += w * ov.x;
      num.y += w * ov.y;
      num.z += w * ov.z;
      num.w += w * ov.w;
    }
    const float id = 1.f / den;
    const int rho = r0 + lr;
    int tok = rho / grp, hh = rho - tok * grp;
    __half2* dst = reinterpret_cast<__half2*>(a.out + ((size_t)(j * a.B + tok) * a.nq + g * grp + hh) * D + 4 * c4);
    dst[0] = __floats2half2_rn(num.x * id, num.y * id);
    dst[1] = __floats2half2_rn(num.z * id, num.w * id);
  }
  fence_proxy_async_global();  // the o projection reads the output with TMA
}

}  // namespace

// How many clusters of ns splits can be resident at once (0 when a cluster
// of that size cannot be launched).  Non-portable sizes above 8 need the
// opt-in attribute and ns free SMs in one GPC; on a 152-SM part a cluster of
// 16 one-CTA-per-SM splits fits only seven times, not eight.  The answer is
// cached per (device, kernel, ns, threads, smem).
static int attn_max_clusters(const void* fn, int ns, int threads, size_t smem) {
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, fn, ns, threads, smem);
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, int, size_t>, int> cache;
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = 0;
  if (ns <= kPortable || cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ns, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = ns;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess)
      n = 0;
  }
  cudaGetLastError();
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  return n;
}

cudaError_t attention(const AttnArgs& a0, cudaStream_t st, bool pdl) {
  AttnArgs a = a0;
  const int rows = a.B * (a.nq / a.nkv);
  const int nw = (rows + 15) / 16;
  const int rows_pad = nw * 16;
  a.nwc = nw;
  const int nthr = (2 * nw < 10 ? 2 * nw : (nw > 10 ? nw : 10)) * 32;
  auto kernel_for = [&](bool kh2) {
    return a.d == 128 ? (kh2 ? (const void*)attn_kernel<128, 2> : (const void*)attn_kernel<128, 1>)
                      : (kh2 ? (const void*)attn_kernel<64, 2> : (const void*)attn_kernel<64, 1>);
  };
  auto smem_for = [&](int n) {
    // Q, double-buffered K/V, per-row lse, then the merge's receive area
    size_t b = 128 + (size_t)rows_pad * a.d * 2 + 4 * kKT * a.d * 2 + rows_pad * 4;
    if (n > 1) {
      const size_t maxr = (rows + n - 1) / n;
      b += (size_t)n * maxr * (a.d + 4) * 4 + (size_t)n * maxr * 4;
    }
    return b;
  };
  // Split count: the longest possible context (capacity plus the block) is
  // cut into ns chunks of whole 64-key tiles, one CTA each, the ns CTAs of a
  // (sequence, kv head) forming one cluster.  Cost model: waves of resident
  // clusters times tiles per split (the pass is latency-bound, each tile a
  // serial step), the fewest splits among equal costs; splits that would be
  // left empty by the tile rounding are not launched.
  const int total = a.cap + a.B;
  const int ntiles = (total + kKT - 1) / kKT;
  const int need = a.b * a.nkv;  // clusters
  int ns = 1;
  long best = -1;
  for (int n = 1; n <= kMaxSplits && n <= ntiles; ++n) {
    const int per = (ntiles + n - 1) / n;   // tiles per split
    const int used = (ntiles + per - 1) / per;  // splits that get keys
    if (used != n) continue;
    const int fit = attn_max_clusters(kernel_for(false), n, nthr, smem_for(n));
    if (fit <= 0) continue;
    const long cost = (long)((need + fit - 1) / fit) * per;
    if (best < 0 || cost < best) {
      best = cost;
      ns = n;
    }
  }
  const int tiles = (ntiles + ns - 1) / ns;
  size_t smem = smem_for(ns);
  // helper warps take the second key half of every tile when a split has
  // several tiles (one tile: the extra merge costs more than it saves)
  const bool kh2 = nthr >= 2 * nw * 32 && tiles >= 2;
  const void* fn = kernel_for(kh2);
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (ns > kPortable) cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  dim3 grid(ns, a.nkv, a.b);
  void* args[] = {&a};
  return launch_kc(fn, grid, dim3(nthr), smem, st, pdl, dim3(ns, 1, 1), args);
}

}  // namespace dfl
