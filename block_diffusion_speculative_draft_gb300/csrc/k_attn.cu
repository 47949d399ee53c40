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
// share the copies and, when a split spans several tiles, compute the second
// key half of every tile.  Long contexts are split along the keys
// (flash-decoding; the pages' long-context verify likewise uses a two-pass
// attention, dflash-mlx summary, "기술적 도전": JIT SDPA 2-pass for
// N >= 1024), as many splits as keep every (sequence, kv head) cluster
// resident at once: the splits of one (sequence, kv head) form a thread-block
// cluster; each keeps an online softmax, stages its normalised partial rows
// and log-sum-exps grouped by the CTA that merges them, and sends each group
// with one bulk shared-to-shared::cluster copy; every CTA then merges its
// slice of query rows over all splits, in split order.  Q.K^T and P.V run on
// m16n8k16 tensor-core MMAs with fp32 accumulation.  Whole tiles of committed
// context (64 keys) arrive by tensor-map copies (128-byte swizzle) into a ring
// of two or three stages, issued ahead by one thread; the tile where the
// context meets the block (and any rows a folded commit appends) is gathered
// row by row with cp.async into the same swizzled layout.
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

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

__device__ __forceinline__ float ex2(float x) {  // 2^x, hardware approximation; 2^-inf = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte chunk ch (of D / 8) of row r in a K or V stage:
// [D / 64 column halves][64 rows][128 bytes], chunk c of a row at c ^ (r % 8)
// (the layout a 64 x 64 fp16 tensor-map box with 128-byte swizzle writes).
__device__ __forceinline__ int kv_off(int r, int ch) {
  return ((ch >> 3) << 13) + (r << 7) + (((ch & 7) ^ (r & 7)) << 4);
}

// Gathers keys [t0, t0 + 64) of (sequence j, kv head g) row by row with
// cp.async (threads tid of nthr) into K/V stage stg, in the swizzled layout of a tensor-map tile:
// part 0 = committed context rows t < Lold only, 1 = the rest (rows a folded
// commit appends, the block's keys, zero fill past k1), 2 = all.  Cache row
// t < L of the head is row row0 + t of kc / vc; block key t - L is row
// (j B + t - L) of kblk / vblk.
template <int D>
__device__ __forceinline__ void gather_tile(const AttnArgs& a, uint8_t* sK, uint8_t* sV, int stg, int t0, int part,
                                            int k1, int Lold, int L, int row0, int j, int g, int tid, int nthr) {
  constexpr int KVB = kKT * D * 2;
  for (int c = tid; c < kKT * (D / 8); c += nthr) {
    const int r = c / (D / 8), ch = c % (D / 8);
    const int t = t0 + r;
    const bool ok = t < k1;
    const bool old_ctx = ok && t < Lold;
    if (part == 0 && !old_ctx) continue;
    if (part == 1 && old_ctx) continue;
    const __half* ks = a.kc;
    const __half* vs = a.vc;
    if (ok) {
      if (t < L) {
        const size_t off = ((size_t)row0 + t) * D + ch * 8;
        ks = a.kc + off;
        vs = a.vc + off;
      } else {
        const size_t off = ((size_t)(j * a.B + (t - L)) * a.nkv + g) * D + ch * 8;
        ks = a.kblk + off;
        vs = a.vblk + off;
      }
    }
    const int so = stg * KVB + kv_off(r, ch);
    cp_async16(sK + so, ks, ok);
    cp_async16(sV + so, vs, ok);
  }
}

// Split merge, after every split has staged its rows in `sst` grouped by
// owner ([ns owners][maxr][RSH] fp16: D normalised partial outputs, then the
// row's fp32 log2-domain log-sum-exp): each owner receives its group from
// every split with one bulk shared-to-shared::cluster copy into rO
// ([ns splits][maxr][RSH]), counted on its receive barrier, then merges its
// query rows [r0, r1) over the splits in split order and writes them out.
// Every load of an item is issued before its arithmetic.
template <int D>
__device__ __forceinline__ void merge_splits(const AttnArgs& a, __half* rO, const __half* sst, uint64_t* rbar,
                                             int rows, int grp, int ns, int sp, int maxr, int r0, int r1, int j,
                                             int g) {
  constexpr int RSH = D + 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane < ns) {
    const int p = lane;
    const int nr = ((p + 1) * rows) / ns - (p * rows) / ns;
    if (nr > 0)
      bulk_s2cluster(dsmem_addr(smem_u32(rO + (size_t)sp * maxr * RSH), (uint32_t)p),
                     smem_u32(sst + (size_t)p * maxr * RSH), (uint32_t)(nr * RSH * 2),
                     dsmem_addr(smem_u32(rbar), (uint32_t)p));
    bulk_commit();
  }
  mbar_wait(rbar, 0, a.status);
  for (int it = threadIdx.x; it < (r1 - r0) * (D / 4); it += blockDim.x) {
    const int lr = it / (D / 4), c4 = it % (D / 4);
    float lv[kMaxSplits];
    uint2 pv[kMaxSplits];
#pragma unroll
    for (int s2 = 0; s2 < kMaxSplits; ++s2)
      if (s2 < ns) {
        const __half* row = rO + (size_t)(s2 * maxr + lr) * RSH;
        lv[s2] = *reinterpret_cast<const float*>(row + D);
        pv[s2] = *reinterpret_cast<const uint2*>(row + 4 * c4);
      }
    float mmax = -INFINITY;
#pragma unroll
    for (int s2 = 0; s2 < kMaxSplits; ++s2)
      if (s2 < ns) mmax = fmaxf(mmax, lv[s2]);
    float den = 0.f;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s2 = 0; s2 < kMaxSplits; ++s2)
      if (s2 < ns) {
        const float w = ex2(lv[s2] - mmax);
        const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&pv[s2].x));
        const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&pv[s2].y));
        den += w;
        num.x += w * lo.x;
        num.y += w * lo.y;
        num.z += w * hi.x;
        num.w += w * hi.y;
      }
    const float id = 1.f / den;
    const int rho = r0 + lr;
    int tok = rho / grp, hh = rho - tok * grp;
    __half2* dst = reinterpret_cast<__half2*>(a.out + ((size_t)(j * a.B + tok) * a.nq + g * grp + hh) * D + 4 * c4);
    dst[0] = __floats2half2_rn(num.x * id, num.y * id);
    dst[1] = __floats2half2_rn(num.z * id, num.w * id);
  }
  // the staging area must outlive the copies' reads of it
  if (warp == 0 && lane < ns) bulk_wait_read_all();
}

template <int D, int KH, int NST>
__global__ void __launch_bounds__(320, 1)
    attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const __grid_constant__ CUtensorMap qmap, const AttnArgs a) {
  constexpr int RB = D * 2;             // bytes per row
  constexpr int KVB = kKT * RB;         // bytes of one K (or V) tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int sp = blockIdx.x, g = blockIdx.y, j = blockIdx.z;
  const int ns = gridDim.x;
  const int grp = a.nq / a.nkv;
  const int rows = a.B * grp;
  const int nwc = a.nwc;
  const int rows_pad = nwc * 16;
  uint8_t* sK = smem;                   // [NST][KVB], 1024-aligned
  uint8_t* sV = sK + NST * KVB;         // [NST][KVB]
  uint8_t* sQ = sV + NST * KVB;         // [D / 64][rows_pad][128 bytes], swizzled like a K/V stage
  // tile barriers [0, NST), the Q barrier at [6], the merge's receive barrier at [7]
  uint64_t* full = reinterpret_cast<uint64_t*>(sQ + rows_pad * RB);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // The context K/V and its length are inputs of the whole draft pass (no
  // kernel of the pass writes them), so context tiles are fetched before
  // waiting for the kernel that produces q and the block K/V.  (A commit
  // folded into this pass appends rows [Lold, L), written by this layer's QKV
  // kernel: those are read only after the wait.)
  int L = a.len[j];
  if (L < 0) L = 0;
  if (L > a.cap) L = a.cap;
  const int Lold = L;
  if (a.nacc) L += commit_count(a.len[j], a.nacc[j], a.rps, a.cap);
  const int total = L + a.B;
  int k0, k1;
  split_range(total, sp, ns, k0, k1);
  const int ntile = (k1 - k0 + kKT - 1) / kKT;
  const int row0 = (j * a.nkv + g) * a.cap;  // this head's first cache row in the tensor maps
  // tile i is a whole tile of committed context (one tensor-map box per 64
  // columns of K and of V) or is gathered row by row (the rest)
  auto is_tma = [&](int i) { return k0 + (i + 1) * kKT <= min(k1, Lold); };

  // split merge (ns > 1): CTA p of the cluster merges query rows
  // [p rows / ns, (p + 1) rows / ns); every split sends it those rows, counted
  // in bytes on its receive barrier
  // staged row: D fp16 partial outputs, the fp32 log-sum-exp, padding (a
  // row stride of 2 D + 16 bytes keeps the staging stores conflict-free)
  constexpr int RSH = D + 8;
  const int maxr = (rows + ns - 1) / ns;
  const int r0 = (sp * rows) / ns, r1 = ((sp + 1) * rows) / ns;
  uint64_t* qbar = full + 6;
  uint64_t* rbar = full + 7;
  auto issue_tma = [&](int i, int stg) {  // thread 0 only
    fence_proxy_async_shared();  // the stage may last have been written by cp.async
    mbar_arrive_expect_tx(&full[stg], 2 * KVB);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_2d(sK + stg * KVB + h * 8192, &kmap, h * 64, row0 + k0 + i * kKT, &full[stg]);
      tma_load_2d(sV + stg * KVB + h * 8192, &vmap, h * 64, row0 + k0 + i * kKT, &full[stg]);
    }
  };
  auto load_rows = [&](int stg, int t0, int part) {
    gather_tile<D>(a, sK, sV, stg, t0, part, k1, Lold, L, row0, j, g, threadIdx.x, blockDim.x);
  };
  // prologue: tiles 0 .. NST-2; the context part before the wait
  constexpr int PRE = NST - 1;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(&full[i], 1);
    mbar_init(qbar, 1);
    if (ns > 1) {
      mbar_init(rbar, 1);
      mbar_arrive_expect_tx(rbar, (uint32_t)(ns * (r1 - r0) * RSH * 2));
    }
    fence_mbar_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    prefetch_tmap(&qmap);
    for (int i = 0; i < PRE && i < ntile; ++i)
      if (is_tma(i)) issue_tma(i, i);
  }
  __syncthreads();  // the barriers are initialised
  // peers may target this CTA's receive barrier once they have passed the
  // matching wait (after their main loop)
  if (ns > 1) cluster_arrive_relaxed();
  for (int i = 0; i < PRE && i < ntile; ++i)
    if (!is_tma(i)) load_rows(i, k0 + i * kKT, 0);
  if (a.pf_base && threadIdx.x == 0)
    prefetch_l2_job(a.pf_base, a.pf_stride, a.pf_bytes, a.pf_i0, a.pf_i1,
                    blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z), gridDim.x * gridDim.y * gridDim.z);
  pdl_wait();

  // ---- Q tile: row rho = tok * grp + hh is q[(j B + tok)][g grp + hh][:],
  // one tensor-map box (64 columns x grp heads x B tokens) per 64 columns;
  // rows past `rows` stay unwritten and are never stored
  if (threadIdx.x == 0) {
    // q was written by the preceding kernel with generic stores
    fence_proxy_async_global();
    mbar_arrive_expect_tx(qbar, (uint32_t)((D / 64) * rows * 128));
#pragma unroll
    for (int h = 0; h < D / 64; ++h) tma_load_3d(sQ + h * rows_pad * 128, &qmap, h * 64, g * grp, j * a.B, qbar);
  }
  // one cp.async group per prologue tile (group 0 also holds every context
  // part issued above: waiting for it early is only conservative)
  for (int i = 0; i < PRE; ++i) {
    if (i < ntile && !is_tma(i)) load_rows(i, k0 + i * kKT, 1);
    cp_async_commit();
  }

  const float sl2 = rsqrtf((float)D) * 1.4426950408889634f;  // 1/sqrt(d) in log2 units
  const int g8 = lane >> 2, t4 = lane & 3;
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
  // running max (raw score units) and sum of the two rows g8, g8 + 8
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  uint32_t qf[D / 16][4];

  // KH = 2: warp w computes row block w % nwc over key half w / nwc of every
  // tile, each half with its own online softmax, merged once after the last
  // tile; KH = 1: one warp per row block over all 64 keys of a tile
  constexpr int KK = kKT / KH;  // keys per warp and tile
  constexpr int NN = KK / 8;    // n8 score tiles per warp
  const int rb = warp % nwc, half = warp / nwc;
  const bool cw = warp < nwc * KH;
  uint32_t phase = 0;  // bit s: parity of the next tensor-map fill of stage s
  int stg = 0;
  for (int it = 0; it < ntile; ++it) {
    {  // refill: tile it + PRE goes to the stage tile it - 1 used
      const int nx = it + PRE;
      const int ns2 = (stg + PRE) % NST;
      if (nx < ntile) {
        if (is_tma(nx)) {
          if (threadIdx.x == 0) issue_tma(nx, ns2);
        } else {
          load_rows(ns2, k0 + nx * kKT, 2);
        }
      }
      cp_async_commit();
    }
    const bool tma = is_tma(it);
    if (tma) {
      mbar_wait(&full[stg], (phase >> stg) & 1u, a.status);
      phase ^= 1u << stg;
    }
    cp_async_wait<PRE>();
    __syncthreads();
    if (cw) {
      if (it == 0) {
        mbar_wait(qbar, 0, a.status);
        const uint32_t qb = smem_u32(sQ);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int row = rb * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int ch = 2 * ks + (lane >> 4);
          ldsm_x4(qb + (ch >> 3) * rows_pad * 128 + row * 128 + (((ch & 7) ^ (row & 7)) << 4), qf[ks][0], qf[ks][1],
                  qf[ks][2], qf[ks][3]);
        }
      }
      const uint32_t kb = smem_u32(sK + stg * KVB);
      const uint32_t vb = smem_u32(sV + stg * KVB);
      // S = Q K^T : 16 rows x KK keys per warp (raw dot products)
      float s[NN][4];
#pragma unroll
      for (int n = 0; n < NN; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int n16 = 0; n16 < NN / 2; ++n16) {
          const int key = half * KK + n16 * 16 + (lane & 7) + ((lane >> 4) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + kv_off(key, 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_f16(s[2 * n16], qf[ks], b0, b1);
          mma_f16(s[2 * n16 + 1], qf[ks], b2, b3);
        }
      }
      // keys past the split's end only occur in its last tile
      const int kbase = k0 + it * kKT + half * KK;
      if (kbase + KK > k1) {
#pragma unroll
        for (int n = 0; n < NN; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (kbase + n * 8 + 2 * t4 + (e & 1) >= k1) s[n][e] = -INFINITY;
      }
      // online softmax in log2 units: p = 2^(s sl2 - m sl2); a half may see
      // no valid key yet: its max stays -inf and contributes nothing
      float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
      for (int n = 0; n < NN; ++n) {
        mx[0] = fmaxf(mx[0], fmaxf(s[n][0], s[n][1]));
        mx[1] = fmaxf(mx[1], fmaxf(s[n][2], s[n][3]));
      }
      float corr[2], nb[2], rs[2] = {0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        corr[r] = mx[r] == -INFINITY ? 1.f : ex2((mrow[r] - mx[r]) * sl2);
        nb[r] = mx[r] == -INFINITY ? 0.f : -mx[r] * sl2;
        mrow[r] = mx[r];
      }
      uint32_t pf[NN / 2][4];  // P as the A operand of P.V, k16 steps over KK keys
#pragma unroll
      for (int n = 0; n < NN; ++n) {
        const float p0 = ex2(fmaf(s[n][0], sl2, nb[0]));
        const float p1 = ex2(fmaf(s[n][1], sl2, nb[0]));
        const float p2 = ex2(fmaf(s[n][2], sl2, nb[1]));
        const float p3 = ex2(fmaf(s[n][3], sl2, nb[1]));
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
          const int key = half * KK + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + kv_off(key, 2 * dp + (lane >> 4)), b0, b1, b2, b3);
          mma_f16(o[2 * dp], pf[kk], b0, b1);
          mma_f16(o[2 * dp + 1], pf[kk], b2, b3);
        }
      }
    }
    __syncthreads();
    stg = stg + 1 == NST ? 0 : stg + 1;
  }
  cp_async_wait<0>();  // empty trailing groups, and zero-fill copies of an empty split
  if (threadIdx.x == 0) mbar_wait(qbar, 0, a.status);  // Q landed even where no tile was computed
  if (KH == 2) {
    // merge the key halves of each row block: half 1 hands (max, sum, O) over
    // through shared memory (the K/V stages are free once the last tile is
    // consumed: every copy issued has been waited for)
    constexpr int XS = D + 4;  // row stride (floats)
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
        c0[r] = mrow[r] == -INFINITY ? 0.f : ex2((mrow[r] - mn) * sl2);
        c1[r] = m1 == -INFINITY ? 0.f : ex2((m1 - mn) * sl2);
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
    lse[r] = lrow[r] > 0.f ? mrow[r] * sl2 + log2f(lrow[r]) : -INFINITY;
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
    return;
  }
  // Stage this split's normalised partial rows and log-sum-exps in its own
  // shared memory grouped by owner, then hand each owner its group with one
  // bulk shared-to-shared::cluster copy.  The staging area reuses the K/V
  // stages and Q (no longer read) when it fits there.
  __half* rO = reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(full) + 64);  // receive [ns][maxr][RSH]
  const size_t need = (size_t)ns * maxr * RSH * 2;
  __half* sst = need <= (size_t)2 * NST * KVB + (size_t)rows_pad * RB ? reinterpret_cast<__half*>(sK)
                                                                      : rO + (size_t)ns * maxr * RSH;
  cluster_wait();   // every peer's receive barrier is initialised and armed
  __syncthreads();  // nothing reads the K/V stages, Q or the key-half scratch any more
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (warp >= nwc) break;
    const int rho = warp * 16 + g8 + 8 * h;
    if (rho >= rows) continue;
    const int own = ((rho + 1) * ns - 1) / rows;
    const int lr = rho - (own * rows) / ns;
    __half* row = sst + (size_t)(own * maxr + lr) * RSH;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<__half2*>(row + i * 8 + 2 * t4) =
          __floats2half2_rn(o[i][2 * h] * inv[h], o[i][2 * h + 1] * inv[h]);
    if (t4 == 0) *reinterpret_cast<float*>(row + D) = lse[h];
  }
  fence_proxy_async_shared();  // each writer: the staged rows are visible to the bulk copies
  __syncthreads();
  merge_splits<D>(a, rO, sst, rbar, rows, grp, ns, sp, maxr, r0, r1, j, g);
}

// ---------------------------------------------------------------------------
// Tensor-memory form: the same grid, splits, gathers and merge; the query
// tile (rows <= 256, rows past `rows` zero) is the M side of tcgen05.mma, in
// one or two blocks of 128 rows.  Three roles run their own loops over the
// split's 64-key tiles, handing off through mbarriers only:
//  * a producer warp fills a ring of NST K/V stages (tensor-map copies for
//    whole tiles of committed context; the other tiles gathered row by row
//    with cp.async by the warp), each stage released by a tcgen05.commit once
//    the MMAs that read it are done;
//  * one thread issues S = Q K^T (M 128, N 64, K 16 per instruction; A = Q
//    from tensor memory, B = K straight from its swizzled tile) and
//    O += P V (M 128, N d, K 16: A = P from tensor memory, B = V read
//    MN-major from its tile, 64-dimension halves 8 KB apart, 8-key groups
//    1 KB apart), committing each block's S to its own mbarrier; the next
//    tile's S of block 0 is issued right after this tile's P V of block 0,
//    so with two blocks one block's softmax runs while the other block's
//    MMAs do;
//  * a warp per 32 query rows (a thread per row: the row's max and sum need
//    no shuffles) copies its Q rows to tensor memory, then per tile reads
//    its scores from tensor memory, runs the online softmax and stores P
//    back as fp16 pairs over the first half of the row's scores (the next
//    S of the block is written by an MMA issued after the P V that reads
//    them, and MMAs from one thread execute in issue order).
// O stays in tensor memory for the whole split.  A row's reference maximum
// is raised only when a tile's maximum exceeds it by more than 8 in log2
// units (the rescale of O is then a read-modify-write of the row); below
// that the reference stays, every p is at most 2^8, which the fp16 P and the
// fp32 sums hold as well, and the result is the same softmax normalised by
// the same sum.
constexpr int kTcThreads = 320;  // warps 0-7 softmax, 8 tensor memory + MMA issue, 9 producer
constexpr int kTcMmaWarp = 8;
constexpr int kTcProdWarp = 9;

template <int D, int NST>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap qmap, const AttnArgs a) {
  constexpr int RB = D * 2;
  constexpr int KVB = kKT * RB;
  constexpr int RSH = D + 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int sp = blockIdx.x, g = blockIdx.y, j = blockIdx.z;
  const int ns = gridDim.x;
  const int grp = a.nq / a.nkv;
  const int rows = a.B * grp;
  const int MB = rows > 128 ? 2 : 1;  // 128-row blocks
  const int rows_pad = MB * 128;
  uint8_t* sK = smem;            // [NST][KVB], 1024-aligned
  uint8_t* sV = sK + NST * KVB;  // [NST][KVB]
  uint8_t* sQ = sV + NST * KVB;  // [D / 64][rows_pad][128 bytes], swizzled like a K/V stage
  uint64_t* full = reinterpret_cast<uint64_t*>(sQ + rows_pad * RB);  // [NST] a stage has landed
  uint64_t* empty = full + 3;  // [NST] a stage's MMAs are done
  uint64_t* sbar = full + 6;   // [2] S of a block is in tensor memory
  uint64_t* pbar = full + 8;   // [2] P of a block is (one arrival per softmax warp of the block)
  uint64_t* ofin = full + 10;  // every MMA of the split is done
  uint64_t* qbar = full + 11;
  uint64_t* rbar = full + 12;
  uint64_t* qtm = full + 13;   // Q is in tensor memory (one arrival per softmax warp)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(full + 14);
  __half* rO = reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(full) + 128);  // receive [ns][maxr][RSH]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // softmax warp w < 8 owns query rows 128 (w / 4) + 32 (w % 4) + lane, the
  // tensor-memory lanes 32 (w % 4) + lane of row block w / 4
  const bool smx = warp < 8 && (warp >> 2) * 128 + (warp & 3) * 32 < rows;
  const int nsw0 = rows >= 128 ? 4 : (rows + 31) / 32;
  const int nsw1 = rows > 128 ? (rows - 128 + 31) / 32 : 0;
  const uint32_t ncols = MB == 2 ? 512u : 256u;
  // tensor-memory columns: O of block m at m D, S at MB D + 64 m (P, fp16
  // pairs, over its first 32), Q (fp16 pairs) at MB D + 64 MB + (D / 2) m
  const uint32_t cS = MB * D, cQ = MB * D + 64 * MB;

  int L = a.len[j];
  if (L < 0) L = 0;
  if (L > a.cap) L = a.cap;
  const int Lold = L;
  if (a.nacc) L += commit_count(a.len[j], a.nacc[j], a.rps, a.cap);
  const int total = L + a.B;
  int k0, k1;
  split_range(total, sp, ns, k0, k1);
  const int ntile = (k1 - k0 + kKT - 1) / kKT;
  const int row0 = (j * a.nkv + g) * a.cap;
  auto is_tma = [&](int i) { return k0 + (i + 1) * kKT <= min(k1, Lold); };
  const int maxr = (rows + ns - 1) / ns;
  const int r0 = (sp * rows) / ns, r1 = ((sp + 1) * rows) / ns;
  const bool prod = warp == kTcProdWarp;
  auto issue_tma = [&](int i, int stg) {  // producer lane 0
    fence_proxy_async_shared();
    mbar_arrive_expect_tx(&full[stg], 2 * KVB);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      tma_load_2d(sK + stg * KVB + h * 8192, &kmap, h * 64, row0 + k0 + i * kKT, &full[stg]);
      tma_load_2d(sV + stg * KVB + h * 8192, &vmap, h * 64, row0 + k0 + i * kKT, &full[stg]);
    }
  };
  auto gather = [&](int i, int part) {  // producer warp
    gather_tile<D>(a, sK, sV, i % NST, k0 + i * kKT, part, k1, Lold, L, row0, j, g, lane, 32);
  };
  // a gathered stage is complete once the warp's copies have landed and are
  // visible to the tensor cores
  auto gathered = [&](int stg) {
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) mbar_arrive(&full[stg]);
  };
  if (prod && lane == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int m = 0; m < 2; ++m) mbar_init(&sbar[m], 1);
    mbar_init(&pbar[0], (uint32_t)nsw0);
    mbar_init(&pbar[1], (uint32_t)(nsw1 > 0 ? nsw1 : 1));
    mbar_init(ofin, 1);
    mbar_init(qbar, 1);
    mbar_init(qtm, (uint32_t)(nsw0 + nsw1));
    if (ns > 1) {
      mbar_init(rbar, 1);
      mbar_arrive_expect_tx(rbar, (uint32_t)(ns * (r1 - r0) * RSH * 2));
    }
    fence_mbar_init();
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    prefetch_tmap(&qmap);
    // the context K/V and its length are inputs of the whole draft pass, so
    // whole context tiles are fetched before the dependency wait
    for (int i = 0; i < NST && i < ntile; ++i)
      if (is_tma(i)) issue_tma(i, i);
  }
  __syncthreads();
  if (ns > 1) cluster_arrive_relaxed();
  if (prod)
    for (int i = 0; i < NST && i < ntile; ++i)
      if (!is_tma(i)) gather(i, 0);  // committed context rows of a gathered tile
  if (a.pf_base && threadIdx.x == 0)
    prefetch_l2_job(a.pf_base, a.pf_stride, a.pf_bytes, a.pf_i0, a.pf_i1,
                    blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z), gridDim.x * gridDim.y * gridDim.z);
  pdl_wait();
  // tensor memory after the dependency wait: the preceding kernel's CTAs on
  // this SM have finished, so their columns are free
  if (warp == kTcMmaWarp) tmem_alloc(s_tmem, ncols);
  if (prod) {
    if (lane == 0) {
      fence_proxy_async_global();  // q was written by the preceding kernel with generic stores
      mbar_arrive_expect_tx(qbar, (uint32_t)((D / 64) * rows * 128));
#pragma unroll
      for (int h = 0; h < D / 64; ++h) tma_load_3d(sQ + h * rows_pad * 128, &qmap, h * 64, g * grp, j * a.B, qbar);
    }
    for (int i = 0; i < NST && i < ntile; ++i)
      if (!is_tma(i)) {
        gather(i, 1);  // rows the preceding kernels wrote: appended context, the block's keys
        gathered(i);
      }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const float sl2 = rsqrtf((float)D) * 1.4426950408889634f;  // 1/sqrt(d) in log2 units
  const int mb = warp >> 2;
  const int rho = mb * 128 + (warp & 3) * 32 + lane;  // this thread's query row (softmax warps)
  const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
  float mref = -INFINITY, lsum = 0.f;  // reference maximum (raw score units) and sum of the row
  bool dead = false;                   // a wait gave up: the status is raised, the rest only drains

  if (prod) {
    // ---------------- producer: tiles NST .. ntile-1 ----------------
    for (int i = NST; i < ntile; ++i) {
      const int stg = i % NST;
      if (!dead && !mbar_wait(&empty[stg], ((i / NST) - 1) & 1, a.status)) dead = true;
      if (is_tma(i)) {
        if (lane == 0) issue_tma(i, stg);
      } else {
        gather(i, 2);
        gathered(stg);
      }
    }
  } else if (warp == kTcMmaWarp) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0 && ntile > 0) {
      auto qk = [&](int it, int m) {  // S of block m for tile it
        const uint32_t ksb = smem_u32(sK + (it % NST) * KVB);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc_mma_f16_ta(tmem + cS + 64 * m, tmem + cQ + (D / 2) * m + 8 * ks,
                        tc_sdesc_sw128(ksb + (ks >> 2) * 8192 + (ks & 3) * 32), tc_idesc_f16(kKT), ks != 0);
        tc_commit(&sbar[m]);
      };
      auto pv = [&](int it, int m) {  // O of block m += P V for tile it
        const uint32_t vsb = smem_u32(sV + (it % NST) * KVB);
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk)
          tc_mma_f16_ta(tmem + D * m, tmem + cS + 64 * m + 8 * kk, tc_sdesc_mn_sw128(vsb + kk * 2048, 8192, 1024),
                        tc_idesc_f16_bmn(D), (it | kk) != 0);
      };
      auto landed = [&](int it) {
        if (!dead && !mbar_wait(&full[it % NST], (it / NST) & 1, a.status)) dead = true;
        tc_fence_after();
      };
      if (!dead && !mbar_wait(qtm, 0, a.status)) dead = true;
      tc_fence_after();
      landed(0);
      qk(0, 0);
      if (MB == 2) qk(0, 1);
      for (int it = 0; it < ntile; ++it) {
        const bool nxt = it + 1 < ntile;
        if (!dead && !mbar_wait(&pbar[0], it & 1, a.status)) dead = true;
        tc_fence_after();
        pv(it, 0);
        if (MB == 2) {
          if (nxt) {
            landed(it + 1);
            qk(it + 1, 0);
          }
          if (!dead && !mbar_wait(&pbar[1], it & 1, a.status)) dead = true;
          tc_fence_after();
          pv(it, 1);
          tc_commit(&empty[it % NST]);
          if (nxt) qk(it + 1, 1);
        } else {
          tc_commit(&empty[it % NST]);
          if (nxt) {
            landed(it + 1);
            qk(it + 1, 0);
          }
        }
      }
      tc_commit(ofin);
    }
  } else if (smx) {
    // ---------------- online softmax, a thread per query row ----------------
    {  // this row of Q (zero past `rows`) to tensor memory as fp16 pairs
      if (!dead && !mbar_wait(qbar, 0, a.status)) dead = true;
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        uint32_t w[32];
        const uint8_t* qrow = sQ + h * rows_pad * 128 + rho * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 u = make_uint4(0u, 0u, 0u, 0u);
          if (rho < rows) u = *reinterpret_cast<const uint4*>(qrow + ((c ^ (rho & 7)) << 4));
          w[4 * c] = u.x;
          w[4 * c + 1] = u.y;
          w[4 * c + 2] = u.z;
          w[4 * c + 3] = u.w;
        }
        tmem_st32(tmem + lanes + cQ + (D / 2) * mb + 32 * h, w);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(qtm);
    }
    for (int it = 0; it < ntile; ++it) {
      if (!dead && !mbar_wait(&sbar[mb], it & 1, a.status)) dead = true;
      tc_fence_after();
      float s[kKT];
      {
        uint32_t v[32];
        tmem_ld32_wait(tmem + lanes + cS + 64 * mb, v);
#pragma unroll
        for (int n = 0; n < 32; ++n) s[n] = __uint_as_float(v[n]);
        tmem_ld32_wait(tmem + lanes + cS + 64 * mb + 32, v);
#pragma unroll
        for (int n = 0; n < 32; ++n) s[32 + n] = __uint_as_float(v[n]);
      }
      // keys past the split's end only occur in its last tile
      const int kb = k0 + it * kKT;
      if (kb + kKT > k1) {
#pragma unroll
        for (int n = 0; n < kKT; ++n)
          if (kb + n >= k1) s[n] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int n = 1; n < kKT; ++n) mx = fmaxf(mx, s[n]);
      const float mnew = fmaxf(mref, mx);
      const bool resc = mref != -INFINITY && (mnew - mref) * sl2 > 8.f;
      const float corr = resc ? ex2((mref - mnew) * sl2) : 1.f;
      if (mref == -INFINITY || resc) mref = mnew;
      if (__any_sync(0xffffffffu, resc)) {
        // O holds the earlier tiles' P V (complete: this tile's S was
        // committed after it)
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t v[32];
          tmem_ld32_wait(tmem + lanes + mb * D + c, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * corr);
          tmem_st32(tmem + lanes + mb * D + c, v);
        }
      }
      lsum *= corr;
      const float nb = mref == -INFINITY ? 0.f : -mref * sl2;
      uint32_t pw[32];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2(fmaf(s[2 * c], sl2, nb));
        const float p1 = ex2(fmaf(s[2 * c + 1], sl2, nb));
        rs += p0 + p1;
        __half2 h = __floats2half2_rn(p0, p1);
        pw[c] = *reinterpret_cast<uint32_t*>(&h);
      }
      lsum += rs;
      tmem_st32(tmem + lanes + cS + 64 * mb, pw);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pbar[mb]);
    }
    // O is final once every MMA of the split is done
    if (ntile > 0 && !dead && !mbar_wait(ofin, 0, a.status)) dead = true;
    tc_fence_after();
  }
  if (prod) {  // zero-fill copies of an empty split
    cp_async_commit();
    cp_async_wait<0>();
  }
  if (prod && lane == 0) mbar_wait(qbar, 0, a.status);  // Q landed even where no tile was computed
  pdl_trigger();

  // normalise this split's rows; log2-domain log-sum-exp (-inf when empty)
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  const float lse = lsum > 0.f ? mref * sl2 + log2f(lsum) : -INFINITY;
  const int tok = rho / grp, hh = rho - (rho / grp) * grp;
  __half* sst = nullptr;
  if (ns > 1) {
    const size_t need = (size_t)ns * maxr * RSH * 2;
    sst = need <= (size_t)2 * NST * KVB + (size_t)rows_pad * RB ? reinterpret_cast<__half*>(sK)
                                                                : rO + (size_t)ns * maxr * RSH;
    cluster_wait();   // every peer's receive barrier is initialised and armed
    __syncthreads();  // every MMA is done: nothing reads the K/V stages or Q any more
  }
  if (smx) {
    __half* dst;
    if (ns == 1) {
      dst = a.out + ((size_t)(j * a.B + tok) * a.nq + g * grp + hh) * D;
    } else {
      const int own = ((rho + 1) * ns - 1) / rows;
      dst = sst + (size_t)(own * maxr + rho - (own * rows) / ns) * RSH;
    }
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t v[32];
      if (ntile > 0) {
        tmem_ld32_wait(tmem + lanes + mb * D + c, v);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = 0u;
      }
      if (rho < rows) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u;
          uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __half2 h = __floats2half2_rn(__uint_as_float(v[8 * q + 2 * e]) * inv,
                                          __uint_as_float(v[8 * q + 2 * e + 1]) * inv);
            w[e] = *reinterpret_cast<uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(dst + c + 8 * q) = u;
        }
      }
    }
    if (ns > 1 && rho < rows) *reinterpret_cast<float*>(dst + D) = lse;
  }
  if (ns > 1) fence_proxy_async_shared();  // each writer: the staged rows are visible to the bulk copies
  // every tensor-memory read is done (or abandoned after a timeout)
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
  if (ns == 1) return;
  merge_splits<D>(a, rO, sst, rbar, rows, grp, ns, sp, maxr, r0, r1, j, g);
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

static int max_smem_optin() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
      cudaGetLastError();
      v = 48 * 1024;
    }
    cached[dev] = v;
  }
  return cached[dev];
}

// The tensor-memory kernel runs query tiles of 129-256 rows (two 128-row MMA
// blocks) whose splits get at least this many 64-key tiles; below that its
// fixed per-split work (tensor-memory allocation, the copy of Q, the
// hand-offs of the first tile) outweighs its faster tiles.  Draft pass of the
// 27B-class drafter (5 layers, 160 query rows per kv head), us, warp-level /
// tensor-memory kernel: 674 / 676 at 1024 context rows (2 tiles per split),
// 688 / 694 at 2048 (4 tiles), 727 / 714 at 4096 (6 tiles); at 64 and 128
// rows (Qwen3-4B / 8B shapes, one MMA block) it was slower at every length.
constexpr int kTcMinTiles = 5;

cudaError_t attention(const AttnArgs& a0, cudaStream_t st, bool pdl) {
  AttnArgs a = a0;
  if (a.d != 64 && a.d != 128) return cudaErrorInvalidValue;
  const int rows = a.B * (a.nq / a.nkv);
  const int nw = (rows + 15) / 16;
  a.nwc = nw;
  const int total = a.cap + a.B;
  const int ntiles = (total + kKT - 1) / kKT;
  const int need = a.b * a.nkv;  // clusters
  struct Plan {
    bool tc;
    int nthr, ns, nst, tiles;
    size_t smem;
    const void* fn;
  };
  // the launch of one kernel family: split count, stages, shared memory
  auto plan = [&](bool tc) {
    Plan p{tc, 0, 0, 0, 0, 0, nullptr};
    // tensor-memory kernel: two 128-row blocks, else one warp per 16 rows
    const int rows_pad = tc ? 256 : nw * 16;
    p.nthr = tc ? kTcThreads : (2 * nw < 10 ? 2 * nw : (nw > 10 ? nw : 10)) * 32;
    auto kernel_for = [&](bool kh2, int nst) {
      if (tc) {
        if (a.d == 128) return nst == 3 ? (const void*)attn_tc_kernel<128, 3> : (const void*)attn_tc_kernel<128, 2>;
        return nst == 3 ? (const void*)attn_tc_kernel<64, 3> : (const void*)attn_tc_kernel<64, 2>;
      }
      if (a.d == 128)
        return nst == 3 ? (kh2 ? (const void*)attn_kernel<128, 2, 3> : (const void*)attn_kernel<128, 1, 3>)
                        : (kh2 ? (const void*)attn_kernel<128, 2, 2> : (const void*)attn_kernel<128, 1, 2>);
      return nst == 3 ? (kh2 ? (const void*)attn_kernel<64, 2, 3> : (const void*)attn_kernel<64, 1, 3>)
                      : (kh2 ? (const void*)attn_kernel<64, 2, 2> : (const void*)attn_kernel<64, 1, 2>);
    };
    auto smem_for = [&](int n, int nst) {
      // 1 KB alignment slack, K/V stages, Q, barriers (64 bytes; 128 with
      // the tensor-memory kernel's), then the merge's receive area (and its
      // staging area, unless that fits in the K/V stages and Q)
      const size_t alias = (size_t)2 * nst * kKT * a.d * 2 + (size_t)rows_pad * a.d * 2;
      size_t b = 1024 + alias + (tc ? 128 : 64);
      if (n > 1) {
        const size_t maxr = (rows + n - 1) / n;
        const size_t need = (size_t)n * maxr * (a.d + 8) * 2;
        b += need;                     // receive area
        if (need > alias) b += need;   // staging area of its own
      }
      return b;
    };
    // three stages where they fit (two tiles in flight behind the one being
    // consumed), else two
    auto stages_for = [&](int n) { return smem_for(n, 3) <= (size_t)max_smem_optin() ? 3 : 2; };
    // Split count: the longest possible context (capacity plus the block) is
    // cut into ns chunks of whole 64-key tiles, one CTA each, the ns CTAs of
    // a (sequence, kv head) forming one cluster.  Cost model: waves of
    // resident clusters times tiles per split (the pass is latency-bound,
    // each tile a serial step), the fewest splits among equal costs; splits
    // that would be left empty by the tile rounding are not launched.
    // Measured on 8 ragged sequences (256 to 8192 context rows): 2 / 3 / 4 /
    // 6 / 8 splits gave a draft pass of 1178 / 1058 / 996 / 1031 / 1086 us,
    // the fractional-wave cost's order.
    long best = -1;
    for (int n = 1; n <= kMaxSplits && n <= ntiles; ++n) {
      const int per = (ntiles + n - 1) / n;       // tiles per split
      const int used = (ntiles + per - 1) / per;  // splits that get keys
      if (used != n) continue;
      const int nst = stages_for(n);
      const int fit = attn_max_clusters(kernel_for(false, nst), n, p.nthr, smem_for(n, nst));
      if (fit <= 0) continue;
      // one sequence: every cluster carries the same keys, so a partial wave
      // costs a whole one; several (lengths unknown here, typically ragged):
      // clusters of short sequences finish early and free their SMs, so
      // waves count fractionally
      const long cost = a.b > 1 ? (long)(1000.0 * (need > fit ? (double)need / fit : 1.0) * per)
                                : 1000l * ((need + fit - 1) / fit) * per;
      if (best < 0 || cost < best) {
        best = cost;
        p.ns = n;
      }
    }
    if (p.ns == 0) return p;  // no split count fits in shared memory
    p.nst = stages_for(p.ns);
    p.tiles = (ntiles + p.ns - 1) / p.ns;
    p.smem = smem_for(p.ns, p.nst);
    // warp-level kernel: helper warps take the second key half of every tile
    // when a split has several tiles (one tile: the extra merge costs more
    // than it saves)
    const bool kh2 = !tc && p.nthr >= 2 * nw * 32 && p.tiles >= 2;
    p.fn = kernel_for(kh2, p.nst);
    return p;
  };
  Plan pl{false, 0, 0, 0, 0, 0, nullptr};
  if (rows > 128 && rows <= 256) pl = plan(true);
  if (pl.ns == 0 || pl.tiles < kTcMinTiles) pl = plan(false);
  if (pl.ns == 0) return cudaErrorInvalidConfiguration;  // no split count fits in shared memory
  const int ns = pl.ns;
  const size_t smem = pl.smem;
  const void* fn = pl.fn;
  const int nthr = pl.nthr;
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (ns > kPortable) cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  // the layer's K and V caches as [b nkv cap] rows of d fp16, read in 64 x 64
  // boxes with 128-byte swizzle
  CUtensorMap km, vm;
  const uint64_t crow = (uint64_t)a.b * a.nkv * a.cap;
  if (!encode_tmap_2d(&km, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.kc, a.d, crow, (uint64_t)a.d * 2, 64, kKT,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&vm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.vc, a.d, crow, (uint64_t)a.d * 2, 64, kKT,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // q [b B tokens][nq heads][d]: one box = 64 columns of the grp heads of a kv
  // head for the B tokens of a sequence (query rows in tok * grp + hh order)
  CUtensorMap qm;
  const uint64_t qdims[3] = {(uint64_t)a.d, (uint64_t)a.nq, (uint64_t)a.b * a.B};
  const uint64_t qstr[2] = {(uint64_t)a.d * 2, (uint64_t)a.nq * a.d * 2};
  const uint32_t qbox[3] = {64, (uint32_t)(a.nq / a.nkv), (uint32_t)a.B};
  if (a.B > 256 || a.nq / a.nkv > 256 ||
      !encode_tmap_3d(&qm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.q, qdims, qstr, qbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  dim3 grid(ns, a.nkv, a.b);
  void* args[] = {&km, &vm, &qm, &a};
  return launch_kc(fn, grid, dim3(nthr), smem, st, pdl, dim3(ns, 1, 1), args);
}

}  // namespace dfl
