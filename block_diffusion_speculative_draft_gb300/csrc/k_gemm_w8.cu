// k_gemm_w8.cu — skinny W8A16 GEMM  Y[M x N] = s[N] . (X[M x K] Q[N x K]^T)
// with fused epilogues, and the packers that produce its weight layouts.
//
// Method: int8 projection weights with one fp16 scale per output channel,
// dequantised as q * s (mirror-sd README, "The Story", Phase 3; "How It Works":
// int8 constants dequantised affinely).  At M = 16..128 activation rows the
// contraction streams every weight byte once and does 2M flops per byte, so
// it has to run at HBM speed.  Two kernels read the same packed int8 tiles:
//  * up to 32 rows, a warp-level MMA kernel (m16n8k16) — these launches are
//    short and latency-bound, and two CTAs per SM in split-K clusters keep
//    them short;
//  * above 32 rows, a fifth-generation tensor-core kernel (tcgen05) with the
//    accumulator in tensor memory — at 64 to 128 rows the contraction (128 to
//    256 flop per weight byte) outruns what the warp-level MMA sustains.
// Shared structure:
//  * swap-AB: the 128-row weight tile is the MMA's M operand, the activation
//    rows of a chunk its N operand;
//  * a producer warp streams 16 KB packed weight tiles with 1-D bulk copies
//    and the matching 128-column activation slice with a 2-D TMA load
//    (128-byte swizzle, rows past M zero-filled) into an mbarrier ring;
//  * biased int8 weights become fp16 exactly in registers (magic-number
//    conversion); the scale is applied after the K reduction;
//  * split-K over the CTAs of a thread-block cluster: each split keeps its
//    fp32 partial tile in shared memory, and after a cluster barrier every
//    CTA sums one slice of activation rows over all splits through
//    distributed shared memory, in split order (deterministic), then runs the
//    epilogue for that slice; no partial ever touches global memory;
//  * programmatic dependent launch (when the library's launch mode allows
//    it): the weight copies of the first stages are issued before
//    griddepcontrol.wait, overlapping the previous kernel's tail.
// The tensor-memory kernel: four converter warps turn each int8 weight row
// into fp16 pairs (one row per thread) and store them to tensor memory
// (tcgen05.st), double-buffered; one MMA warp issues tcgen05.mma kind::f16
// with A from tensor memory and the activations (K-major, 128-byte swizzle)
// through a shared-memory descriptor; tcgen05.commit releases ring stages
// and A buffers when their MMAs have run; the accumulator is read back with
// tcgen05.ld and the tensor memory freed before the reduction.
// int4 weights (W4A16; a 4-bit drafter is the default of mlx-dspark v0.0.3,
// release notes "Notes") run on the warp-level kernel: symmetric codes in
// [-7, 7] with one fp16 scale per row and 128-column group, packed as
// 8448-byte tiles (fragment-ordered nibbles + the tile's group scales).  A
// k-tile is one group, so each stage's partial sums are scaled per row as
// they join the accumulators.
#include <map>
#include <mutex>
#include <tuple>

#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace dfl {

namespace {

constexpr int kTStride = 132;  // epilogue tile row stride (floats)

// ------------------------------------------- warp-level MMA kernel ----
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

// packed int4 tile: 8 KB of fragment-ordered nibbles, then the 128 rows'
// fp16 scales of the tile's 128-column group
constexpr int kTile4Bytes = (int)kW4TileBytes;

template <int MT, int BITS>
struct Geo {
  static constexpr int MCH = MT * 8;          // activation rows per chunk
  // ring stages: int8 3 / 4 (3 keeps two 64-row CTAs per SM); int4 tiles are
  // half the bytes, so a deeper ring keeps as many weight bytes in flight
  // (every variant stays under 110 KB: two CTAs per SM)
  static constexpr int NST = BITS == 8 ? (MT >= 8 ? 3 : 4) : (MT >= 8 ? 4 : (MT >= 4 ? 6 : 8));
  static constexpr int ABYTES = 2 * MCH * 128;  // two [MCH][64] fp16 halves
  static constexpr int WBYTES = BITS == 8 ? kTileBytes : kTile4Bytes;  // weight bytes per stage
  static constexpr int WSLOT = (WBYTES + 1023) / 1024 * 1024;  // activations 1 KB aligned
  static constexpr int STAGE = WSLOT + ABYTES;
  static constexpr int TX = WBYTES + ABYTES;  // bytes a stage's copies deliver
  static constexpr int TBYTES = (MCH * kTStride * 4 + 1023) / 1024 * 1024;
  static_assert(2 * TBYTES <= NST * STAGE, "epilogue tiles must fit in the ring");
  // side data after the barriers: row scales, gamma, next gamma, per-row
  // positions, per-row norm factors
  static constexpr int SIDE = 128 * 4 + 128 * 4 + 128 * 4 + MCH * 4 + MCH * 4;
  static constexpr size_t SMEM = 1024 + NST * (size_t)STAGE + 2 * NST * 8 + 64 + SIDE;
  static_assert(SMEM <= 112 * 1024, "two CTAs per SM");
};

// packed row -> logical row
__device__ __forceinline__ int logical_row(int prow, int layout, int N) {
  if (layout == 1) {
    int tile = prow >> 7, r = prow & 127;
    return r < 64 ? tile * 64 + r : (N >> 1) + tile * 64 + (r - 64);
  }
  return prow;
}


// Epilogue for the chunk's activation rows [tlo, thi).  T holds the reduced,
// unscaled fp32 tile as [row][TSTRIDE]; sc[r] is packed row r's scale, gam
// the per-head gamma and pos[t] the position of row t (-1: not written), all
// staged in shared memory before the main loop so that no global load sits on
// the epilogue's critical path except the residual read, issued in batches.
template <int MCH>
__device__ void epilogue(const W8Args& a, float* T, const float* sc, const float* gam, const int* pos,
                         const float* gn, const float* rr, __half* kout, __half* vout, int nt, int z, int tlo,
                         int thi, int warp, int lane) {
  constexpr int TS = kTStride;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int ntok = thi - tlo;
  const int prow0 = a.row0 + nt * kTile;  // first packed row of this tile
  if (a.ss_in) {  // deferred RMSNorm of the input rows: one factor per row
    for (int i = tid; i < ntok * kTile; i += nthr) {
      const int tok = tlo + (i >> 7);
      T[tok * TS + (i & 127)] *= rr[tok];
    }
    __syncthreads();
  }
  if (a.epi == EPI_STORE_F32 || a.epi == EPI_RESID_F32) {
    const int items = ntok * (kTile / 4);  // groups of 4 consecutive rows
    for (int base = tid; base < items; base += 4 * nthr) {
      float4 xo[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = base + u * nthr;
        xo[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (it < items && a.epi == EPI_RESID_F32) {
          const int tok = tlo + it / (kTile / 4), r = 4 * (it % (kTile / 4));
          const int m = z * MCH + tok;
          if (m < a.M) {
            const int n = logical_row(prow0 + r, a.layout, a.N);
            xo[u] = *reinterpret_cast<const float4*>(a.out_f32 + (size_t)m * a.ldo + (n - a.row0));
          }
        }
      }
      // one row's 128 columns span exactly one warp for a given u (items is a
      // multiple of 32 and nthr of 32), so the row sum of squares is a warp sum
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = base + u * nthr;
        float ss = 0.f;
        int m = a.M;
        if (it < items) {
          const int tok = tlo + it / (kTile / 4), r = 4 * (it % (kTile / 4));
          m = z * MCH + tok;
          if (m < a.M) {
            const int n = logical_row(prow0 + r, a.layout, a.N);
            const float* t = T + tok * TS + r;
            float4 v = make_float4(t[0] * sc[r] + xo[u].x, t[1] * sc[r + 1] + xo[u].y,
                                   t[2] * sc[r + 2] + xo[u].z, t[3] * sc[r + 3] + xo[u].w);
            if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + (size_t)m * a.ldo + (n - a.row0)) = v;
            if (a.xg_out) {
              __half2 h0 = __floats2half2_rn(v.x * gn[r], v.y * gn[r + 1]);
              __half2 h1 = __floats2half2_rn(v.z * gn[r + 2], v.w * gn[r + 3]);
              uint2 pk;
              pk.x = *reinterpret_cast<uint32_t*>(&h0);
              pk.y = *reinterpret_cast<uint32_t*>(&h1);
              *reinterpret_cast<uint2*>(a.xg_out + (size_t)m * a.ldo + (n - a.row0)) = pk;
              ss = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
            if (a.hb_out) {
              const int seq = m / a.hb_rps, slot = m - seq * a.hb_rps;
              if (slot > 0) {
                __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x * gn[r], v.y * gn[r + 1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(v.z * gn[r + 2], v.w * gn[r + 3]);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&h0);
                pk.y = *reinterpret_cast<uint32_t*>(&h1);
                const size_t o = (size_t)seq * (a.hb_rps - 1) + (slot - 1);
                *reinterpret_cast<uint2*>(a.hb_out + o * a.ldo + (n - a.row0)) = pk;
              }
            }
          }
        }
        if (a.xg_out && it < items) {  // warp-uniform condition
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (lane == 0 && m < a.M) a.ss_out[(size_t)m * a.nss_out + (prow0 >> 7)] = ss;
        }
      }
    }
    return;
  }
  if (a.epi == EPI_SWIGLU) {
    const int F = a.N >> 1;
    const int items = ntok * 16;  // groups of 4 output columns
    for (int it = tid; it < items; it += nthr) {
      const int tok = tlo + it / 16, r = 4 * (it % 16);
      const int m = z * MCH + tok;
      if (m >= a.M) continue;
      const float* t = T + tok * TS;
      float g[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float gate = t[r + e] * sc[r + e];
        float up = t[r + e + 64] * sc[r + e + 64];
        g[e] = gate / (1.0f + expf(-gate)) * up;
      }
      __half2 h0 = __floats2half2_rn(g[0], g[1]), h1 = __floats2half2_rn(g[2], g[3]);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&h0);
      pk.y = *reinterpret_cast<uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(a.out_h + (size_t)m * F + nt * 64 + r) = pk;
    }
    return;
  }
  // per-head epilogues: one warp per activation row, lane holds rows lane+32i
  const int qd = a.nq * a.d, kd = a.nkv * a.d;
  const int kind = prow0 < qd ? 0 : (prow0 < qd + kd ? 1 : 2);  // q, k, v
  const int nwarps = blockDim.x >> 5;
  for (int tok = tlo + warp; tok < thi; tok += nwarps) {
    const int m = z * MCH + tok;
    const int p = pos[tok];
    if (m >= a.M || p < 0) continue;
    const bool crow = a.epi == EPI_QKV && a.c_nacc && m >= a.mc0;  // folded commit row
    if (crow && kind == 0) continue;                              // its q is not needed
    const int seq = m / a.rows_per_seq;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int r = lane + 32 * i;
      v[i] = T[tok * TS + r] * sc[r];
    }
    if (kind != 2) {
      if (a.d == 128) {
        float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        float inv = rsqrtf(ss / 128.0f + a.eps);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= inv * gam[lane + 32 * i];
        rope_rot(v[0], v[2], p, a.inv_hi[lane], a.inv_lo[lane]);
        rope_rot(v[1], v[3], p, a.inv_hi[lane + 32], a.inv_lo[lane + 32]);
      } else {  // d == 64: rows 0..63 head A, 64..127 head B
        float sa = v[0] * v[0] + v[1] * v[1];
        float sb = v[2] * v[2] + v[3] * v[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          sa += __shfl_xor_sync(0xffffffffu, sa, o);
          sb += __shfl_xor_sync(0xffffffffu, sb, o);
        }
        float ia = rsqrtf(sa / 64.0f + a.eps), ib = rsqrtf(sb / 64.0f + a.eps);
        v[0] *= ia * gam[lane];
        v[1] *= ia * gam[lane + 32];
        v[2] *= ib * gam[lane];
        v[3] *= ib * gam[lane + 32];
        rope_rot(v[0], v[1], p, a.inv_hi[lane], a.inv_lo[lane]);
        rope_rot(v[2], v[3], p, a.inv_hi[lane], a.inv_lo[lane]);
      }
    }
    if (a.epi == EPI_QKV && !crow) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        int row = prow0 + lane + 32 * i;
        __half hv = __float2half_rn(v[i]);
        if (kind == 0) a.out_h[(size_t)m * qd + row] = hv;
        else if (kind == 1) kout[(size_t)m * kd + (row - qd)] = hv;
        else vout[(size_t)m * kd + (row - qd - kd)] = hv;
      }
    } else {  // a committed context row: cache [b][nkv][cap][d]
      const int cseq = crow ? (m - a.mc0) / a.c_rps : seq;
      __half* ck = crow ? a.ck : kout;
      __half* cv = crow ? a.cv : vout;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        int row = prow0 + lane + 32 * i - qd;  // within k|v rows
        int isv = row >= kd;
        int rr = isv ? row - kd : row;
        int h = rr / a.d, e = rr - h * a.d;
        size_t off = (((size_t)cseq * a.nkv + h) * a.cap + p) * a.d + e;
        (isv ? cv : ck)[off] = __float2half_rn(v[i]);
      }
    }
  }
}

// int4 nibbles (biased by 8) of one 32-bit word to the four half2 registers
// of an m16k16 A fragment: nibble k sits at bits 4k; nibbles (0, 4), (1, 5),
// (2, 6), (3, 7) form registers 0..3.  The magic-number conversion puts a
// nibble into an fp16 mantissa under exponent 2^10 (1024 + n, or 1024 + 16 n
// for the high nibble of a byte, scaled back by 1/16) and removes the bias by
// one subtraction; every step is exact.
__device__ __forceinline__ void biased_u4x8_to_half2x4(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t lo0 = (w & 0x000F000Fu) | 0x64006400u;
  const uint32_t hi0 = (w & 0x00F000F0u) | 0x64006400u;
  const uint32_t lo1 = ((w >> 8) & 0x000F000Fu) | 0x64006400u;
  const uint32_t hi1 = ((w >> 8) & 0x00F000F0u) | 0x64006400u;
  const __half2 sub = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
  const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
  const __half2 sub16 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));  // -72
  __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo0), sub);
  __half2 b = __hfma2(*reinterpret_cast<const __half2*>(&hi0), sixteenth, sub16);
  __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&lo1), sub);
  __half2 d = __hfma2(*reinterpret_cast<const __half2*>(&hi1), sixteenth, sub16);
  r[0] = *reinterpret_cast<uint32_t*>(&a);
  r[1] = *reinterpret_cast<uint32_t*>(&b);
  r[2] = *reinterpret_cast<uint32_t*>(&c);
  r[3] = *reinterpret_cast<uint32_t*>(&d);
}


// Split-K reduction across the thread-block cluster and the epilogue, shared
// by the int8 (tensor-memory) and int4 kernels.  On entry every CTA of the
// cluster has its own fp32 partial tile P[tok][kTStride] at the start of its
// (idle) stage ring; TBYTES is that tile's size rounded to 1 KB.
template <int MCH, int TBYTES>
__device__ __forceinline__ void split_reduce_epilogue(const W8Args& a, uint8_t* smem, const float* s_sc,
                                                      const float* s_gam, const int* s_pos, const float* s_gn,
                                                      const float* s_rr, __half* kout, __half* vout, int nt, int z,
                                                      int sp, int warp, int lane) {
  float* P = reinterpret_cast<float*>(smem);
  float* T = reinterpret_cast<float*>(smem + TBYTES);
  if (a.splits == 1) {
    __syncthreads();
    epilogue<MCH>(a, P, s_sc, s_gam, s_pos, s_gn, s_rr, kout, vout, nt, z, 0, MCH, warp, lane);
    // the next kernel reads these outputs with TMA (async proxy)
    fence_proxy_async_global();
    return;
  }
  // ---- split-K reduction across the cluster through distributed smem ----
  cluster_sync();
  const int S = a.splits;
  const int tlo = (sp * MCH) / S, thi = ((sp + 1) * MCH) / S;
  const int items = (thi - tlo) * (kTile / 4);  // float4 items of this slice
  const uint32_t pbase = smem_u32(P);
  for (int it = threadIdx.x; it < items; it += blockDim.x) {
    const int tok = tlo + it / (kTile / 4), c4 = it % (kTile / 4);
    const uint32_t off = pbase + (uint32_t)(tok * kTStride + 4 * c4) * 4u;
    float4 v[8];
    float4 accv = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 8) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (s0 + q < S) v[q] = ld_dsmem_f4(dsmem_addr(off, (uint32_t)(s0 + q)));
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (s0 + q < S) {
          accv.x += v[q].x;
          accv.y += v[q].y;
          accv.z += v[q].z;
          accv.w += v[q].w;
        }
    }
    *reinterpret_cast<float4*>(T + tok * kTStride + 4 * c4) = accv;
  }
  cluster_sync();  // every peer has finished reading this CTA's partial
  epilogue<MCH>(a, T, s_sc, s_gam, s_pos, s_gn, s_rr, kout, vout, nt, z, tlo, thi, warp, lane);
  fence_proxy_async_global();  // the next kernel reads these outputs with TMA
}

template <int MT, int BITS>
__global__ void __launch_bounds__(kThreads, 1) wmma_gemm_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                 const W8Args a) {
  using G = Geo<MT, BITS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::NST * G::STAGE);
  uint64_t* empty = full + G::NST;
  float* s_sc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(empty + G::NST) + 64);  // [128]
  float* s_gam = s_sc + 128;                                                                 // [128]
  float* s_gn = s_gam + 128;                                                                 // [128]
  int* s_pos = reinterpret_cast<int*>(s_gn + 128);                                           // [MCH]
  float* s_rr = reinterpret_cast<float*>(s_pos + G::MCH);                                    // [MCH]

  const int sp = blockIdx.y, z = blockIdx.z;
  // this CTA's projection (one layer of a batched launch, or the only one)
  int nt = blockIdx.x;
  const uint8_t* wq = a.q;
  const __half* wsc = a.s;
  __half* kout = a.kout;
  __half* vout = a.vout;
  const float* gk = a.gk;
  if (a.nl > 0) {
    const int li = nt / a.ntl;
    nt -= li * a.ntl;
    wq = a.lq[li];
    wsc = a.ls[li];
    kout = a.lk[li];
    vout = a.lv[li];
    gk = a.lgk[li];
  }
  const int KT = a.K / kTile;
  const int kt0 = (int)(((long long)sp * KT) / a.splits);
  const int kt1 = (int)(((long long)(sp + 1) * KT) / a.splits);
  const int nk = kt1 - kt0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < G::NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  float acc[2][MT][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      prefetch_tmap(&xmap);
      const uint8_t* wsrc = wq + ((size_t)((a.row0 >> 7) + nt) * KT + kt0) * G::WBYTES;
      const uint64_t pol = policy_evict_first();
      const int pre = nk < G::NST ? nk : G::NST;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], G::TX);
        bulk_g2s_hint(smem + i * G::STAGE, wsrc + (size_t)i * G::WBYTES, G::WBYTES, &full[i], pol);
      }
      pdl_wait();
      // the activations were written by the previous kernel with generic
      // stores; order this thread's tensor (async-proxy) reads after them
      fence_proxy_async_global();
      for (int i = 0; i < pre; ++i) {
        uint8_t* sa = smem + i * G::STAGE + G::WSLOT;
        tma_load_2d(sa, &xmap, (kt0 + i) * kTile, z * G::MCH, &full[i]);
        tma_load_2d(sa + G::MCH * 128, &xmap, (kt0 + i) * kTile + 64, z * G::MCH, &full[i]);
      }
      for (int i = pre; i < nk; ++i) {
        const int slot = i % G::NST;
        if (!mbar_wait(&empty[slot], ((i / G::NST) - 1) & 1, a.status)) break;
        mbar_arrive_expect_tx(&full[slot], G::TX);
        uint8_t* st = smem + slot * G::STAGE;
        bulk_g2s_hint(st, wsrc + (size_t)i * G::WBYTES, G::WBYTES, &full[slot], pol);
        tma_load_2d(st + G::WSLOT, &xmap, (kt0 + i) * kTile, z * G::MCH, &full[slot]);
        tma_load_2d(st + G::WSLOT + G::MCH * 128, &xmap, (kt0 + i) * kTile + 64, z * G::MCH, &full[slot]);
      }
    }
    pdl_trigger();
  } else {
    // ---------------- consumers ----------------
    {  // weights-side data first (independent of the preceding kernel)
      const int r = threadIdx.x;  // 0..127
      const int prow = a.row0 + nt * kTile + r;
      // int4 weights carry their group scales in the tile (applied per stage)
      // int4 tiles carry their group scales, applied per stage
      s_sc[r] = BITS == 8 ? __half2float(wsc[logical_row(prow, a.layout, a.N)]) : 1.f;
      if (a.epi == EPI_QKV || a.epi == EPI_KVCOMMIT) {
        const int qd = a.nq * a.d;
        const float* gsrc = (a.row0 + nt * kTile) < qd ? a.gq : gk;
        s_gam[r] = (gsrc && r < a.d) ? gsrc[r] : 1.f;
      }
      if (a.xg_out || a.hb_out) s_gn[r] = a.g_next[logical_row(prow, a.layout, a.N) - a.row0];
    }
    pdl_wait();
    if (a.ss_in && threadIdx.x < G::MCH) {
      // deferred RMSNorm factor of each activation row (fixed summation order)
      const int m = z * G::MCH + threadIdx.x;
      float rf = 0.f;
      if (m < a.M) {
        float sum = 0.f;
        const float* row = a.ss_in + (size_t)m * a.nss_in;
        if ((a.nss_in & 3) == 0 && a.nss_in <= 64) {
          // every partial in flight at once (one round trip), summed in order
          float4 v[16];
#pragma unroll
          for (int q = 0; q < 16; ++q)
            if (4 * q < a.nss_in) v[q] = reinterpret_cast<const float4*>(row)[q];
#pragma unroll
          for (int q = 0; q < 16; ++q)
            if (4 * q < a.nss_in) sum += ((v[q].x + v[q].y) + (v[q].z + v[q].w));
        } else {
          for (int i = 0; i < a.nss_in; ++i) sum += row[i];
        }
        rf = rsqrtf(sum / a.K + a.eps);
      }
      s_rr[threadIdx.x] = rf;
    }
    if ((a.epi == EPI_QKV || a.epi == EPI_KVCOMMIT) && threadIdx.x < G::MCH) {
      // position of each activation row of this chunk, -1 when not written
      const int t = threadIdx.x, m = z * G::MCH + t;
      int p = -1;
      if (m < a.M) {
        if (a.epi == EPI_KVCOMMIT) {
          const int seq = m / a.rows_per_seq, slot = m - seq * a.rows_per_seq;
          const int L0 = a.len[seq];
          p = slot < commit_count(L0, a.nacc[seq], a.rows_per_seq, a.cap) ? L0 + slot : -1;
        } else if (a.c_nacc && m >= a.mc0) {  // a context row of the folded commit
          const int mc = m - a.mc0, seq = mc / a.c_rps, slot = mc - seq * a.c_rps;
          const int L0 = a.len[seq];
          p = slot < commit_count(L0, a.c_nacc[seq], a.c_rps, a.cap) ? L0 + slot : -1;
        } else {  // a block row: after the context (grown by the folded commit)
          const int seq = m / a.rows_per_seq, slot = m - seq * a.rows_per_seq;
          const int L0 = a.len[seq];
          int base = L0 < 0 ? 0 : L0;
          if (a.c_nacc) base += commit_count(L0, a.c_nacc[seq], a.c_rps, a.cap);
          p = base + slot;
        }
      }
      s_pos[t] = p;
    }
    const int g_tok_lo = (lane & 7) + ((lane >> 4) << 3);
    const int ch_hi = (lane >> 3) & 1;
    for (int i = 0; i < nk; ++i) {
      const int slot = i % G::NST;
      if (!mbar_wait(&full[slot], (i / G::NST) & 1, a.status)) break;
      const uint32_t abase = smem_u32(smem + slot * G::STAGE + G::WSLOT);
      if constexpr (BITS == 8) {
        // the int8 tile is [row 128][128 bytes], 16-byte chunks swizzled by
        // row, each chunk holding lane t's fragment bytes (columns 2t, 2t+1,
        // 2t+8, 2t+9 of the 16-column group) at bytes 4t..4t+3.  Read as
        // 8x8 matrices of 16-bit pairs, ldmatrix hands lane (g, t) exactly
        // word t of row g's chunk: one ldmatrix.x4 per k-step loads the
        // words of rows g, g+8, g+16, g+24 of this warp's 32 rows
        // (conflict-free: the row swizzle spreads the 8 rows of a matrix).
        const uint32_t wst = smem_u32(smem + slot * G::STAGE);
        const int wr = warp * 32 + lane;  // row this lane addresses (wr % 8 == lane % 8)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t af[2][4];
          uint32_t w00, w01, w10, w11;
          ldsm_x4(wst + wr * 128 + ((ks ^ (lane & 7)) << 4), w00, w01, w10, w11);
          biased_u8x4_to_half2x2(w00, af[0][0], af[0][2]);
          biased_u8x4_to_half2x2(w01, af[0][1], af[0][3]);
          biased_u8x4_to_half2x2(w10, af[1][0], af[1][2]);
          biased_u8x4_to_half2x2(w11, af[1][1], af[1][3]);
          const uint32_t hbase = abase + (ks >> 2) * (G::MCH * 128);
          const int ch = ((ks & 3) << 1) + ch_hi;
#pragma unroll
          for (int p = 0; p < MT / 2; ++p) {
            const int tok = p * 16 + g_tok_lo;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(hbase + tok * 128 + ((ch ^ (tok & 7)) << 4), b0, b1, b2, b3);
            mma_f16(acc[0][2 * p], af[0], b0, b1);
            mma_f16(acc[1][2 * p], af[1], b0, b1);
            mma_f16(acc[0][2 * p + 1], af[0], b2, b3);
            mma_f16(acc[1][2 * p + 1], af[1], b2, b3);
          }
        }
      } else {
        // int4: this k-tile is one scale group, so its partial sums are
        // scaled per row before joining the accumulators
        const uint8_t* wl = smem + slot * G::STAGE + (warp * 8 * 32 + lane) * 8;
        float tacc[2][MT][4];
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int jj = 0; jj < MT; ++jj)
#pragma unroll
            for (int e = 0; e < 4; ++e) tacc[x][jj][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint2 wq = *reinterpret_cast<const uint2*>(wl + ks * 32 * 8);
          uint32_t af[2][4];
          biased_u4x8_to_half2x4(wq.x, af[0]);
          biased_u4x8_to_half2x4(wq.y, af[1]);
          const uint32_t hbase = abase + (ks >> 2) * (G::MCH * 128);
          const int ch = ((ks & 3) << 1) + ch_hi;
#pragma unroll
          for (int p = 0; p < MT / 2; ++p) {
            const int tok = p * 16 + g_tok_lo;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(hbase + tok * 128 + ((ch ^ (tok & 7)) << 4), b0, b1, b2, b3);
            mma_f16(tacc[0][2 * p], af[0], b0, b1);
            mma_f16(tacc[1][2 * p], af[1], b0, b1);
            mma_f16(tacc[0][2 * p + 1], af[0], b2, b3);
            mma_f16(tacc[1][2 * p + 1], af[1], b2, b3);
          }
        }
        const __half* gsc = reinterpret_cast<const __half*>(smem + slot * G::STAGE + 8192);
        const int g = lane >> 2;
#pragma unroll
        for (int mg = 0; mg < 2; ++mg) {
          const float s_lo = __half2float(gsc[warp * 32 + mg * 16 + g]);
          const float s_hi = __half2float(gsc[warp * 32 + mg * 16 + g + 8]);
#pragma unroll
          for (int jj = 0; jj < MT; ++jj)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mg][jj][e] += tacc[mg][jj][e] * (e < 2 ? s_lo : s_hi);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    pdl_trigger();
  }
  __syncthreads();  // all stages consumed: the ring can be reused as scratch

  // own partial tile P[tok][kTStride] at the ring's start; the reduced slice
  // goes to a second buffer so peers can keep reading P meanwhile
  float* P = reinterpret_cast<float*>(smem);
  const int g = lane >> 2, t = lane & 3;
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int mg = 0; mg < 2; ++mg)
#pragma unroll
      for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          int r = warp * 32 + mg * 16 + g + ((e >> 1) << 3);
          int tok = j * 8 + 2 * t + (e & 1);
          P[tok * kTStride + r] = acc[mg][j][e];
        }
  }
  split_reduce_epilogue<G::MCH, G::TBYTES>(a, smem, s_sc, s_gam, s_pos, s_gn, s_rr, kout, vout, nt, z, sp, warp,
                                           lane);
}

// ---------------------------------------------------- int8, tcgen05 ----
// Converter warps in groups of four (warp w reaches tensor-memory lanes
// 32 (w % 4) ..; with G groups, group g converts the k-tiles i with
// i % G == g), then the producer warp and the MMA warp.  One group: six warps
// a CTA keep two CTAs on an SM within each sub-partition's register file
// (ten warps do not: three of them on one sub-partition, twice, is too many),
// and one group converts faster than the single MMA thread consumes.
constexpr int kTcConv = 4;
constexpr int kTcGroups = kTcConv / 4;
constexpr int kTcProducer = kTcConv;
constexpr int kTcMma = kTcConv + 1;
constexpr int kTcThreads = (kTcConv + 2) * 32;
// Projections of at least this many weight bytes run on the tensor-memory
// kernel from 17 activation rows (measured per shape: it wins for the 27B
// gate|up, down and fc and the Qwen3-4B gate|up at 32 rows, ties the 27B QKV
// and loses the smaller ones).
constexpr int64_t kTcMinWeightBytes = 40ll << 20;

// Tensor memory: 512 columns per SM.  The occupancy calculator reports one
// block per SM for any kernel that allocates tensor memory, but a 256-column
// CTA measurably shares its SM with a second one (a 512-column allocation
// made the 272-CTA gate|up launch run in two waves), so CTAs that fit two to
// an SM in shared memory take half the columns.

template <int MT>
struct TcGeo {
  static constexpr int MCH = MT * 8;  // activation rows per chunk = MMA N
  static_assert(MCH % 16 == 0 && MCH <= 128, "MMA N: a multiple of 16 up to 128");
  static constexpr int NST = MT == 16 ? 4 : 3;                // ring stages
  static constexpr uint32_t TCOLS = MT == 16 ? 512 : 256;  // tensor-memory columns of a CTA
  static constexpr int ABYTES = 2 * MCH * 128;  // two [MCH][64] fp16 halves
  static constexpr int WBYTES = kTileBytes;      // int8 tile
  static constexpr int STAGE = WBYTES + ABYTES;  // both 1 KB multiples
  static constexpr int TX = WBYTES + ABYTES;
  static constexpr int TBYTES = (MCH * kTStride * 4 + 1023) / 1024 * 1024;
  // the partial tile and, for split-K, the reduced tile, in the idle ring
  static_assert(2 * TBYTES <= NST * STAGE, "epilogue tiles must fit in the ring");
  // tensor memory: accumulator in columns [0, MCH), then one A buffer of 64
  // columns (one k-tile of fp16 pairs) per ring stage from column TA, so one
  // MMA completion releases a stage's A buffer and its activations together
  static constexpr int NAB = NST;
  static constexpr uint32_t TA = MCH <= 64 ? 64 : 128;
  static_assert(TA + 64 * NAB <= TCOLS, "tensor-memory columns");
  // wfull, xfull, wempty, afull, done per stage; dfull
  static constexpr int NBAR = 5 * NST + 1;
  static constexpr int SIDE = 128 * 4 + 128 * 4 + 128 * 4 + MCH * 4 + MCH * 4;
  static constexpr size_t SMEM = 1024 + NST * (size_t)STAGE + NBAR * 8 + 16 + SIDE;
  static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

// Named barrier over the converter warps and the MMA warp.
__device__ __forceinline__ void tc_bar() { asm volatile("bar.sync 1, %0;" ::"n"((kTcConv + 1) * 32) : "memory"); }

template <int MT>
__global__ void __launch_bounds__(kTcThreads, 1) w8_gemm_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                 const W8Args a) {
  using G = TcGeo<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // A ring stage holds a weight tile and the activation tile it meets; the
  // two halves are filled and released separately: the weights as soon as
  // the converter group has read them, the activations when the MMAs that
  // read them have completed
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + G::NST * G::STAGE);
  uint64_t* xfull = wfull + G::NST;
  uint64_t* wempty = xfull + G::NST;  // the converter group's 4 warps
  uint64_t* afull = wempty + G::NST;  // the stage's A buffer stored and activations landed (4 warps)
  uint64_t* done = afull + G::NST;    // the stage's MMAs complete (1 commit): A buffer and activations free
  uint64_t* dfull = done + G::NST;    // accumulator complete (commit)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(dfull + 1);
  float* s_sc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(s_tmem) + 16);  // [128]
  float* s_gam = s_sc + 128;                                                          // [128]
  float* s_gn = s_gam + 128;                                                          // [128]
  int* s_pos = reinterpret_cast<int*>(s_gn + 128);                                    // [MCH]
  float* s_rr = reinterpret_cast<float*>(s_pos + G::MCH);                             // [MCH]

  const int sp = blockIdx.y, z = blockIdx.z;
  int nt = blockIdx.x;
  const uint8_t* wq = a.q;
  const __half* wsc = a.s;
  __half* kout = a.kout;
  __half* vout = a.vout;
  const float* gk = a.gk;
  if (a.nl > 0) {
    const int li = nt / a.ntl;
    nt -= li * a.ntl;
    wq = a.lq[li];
    wsc = a.ls[li];
    kout = a.lk[li];
    vout = a.lv[li];
    gk = a.lgk[li];
  }
  const int KT = a.K / kTile;
  const int kt0 = (int)(((long long)sp * KT) / a.splits);
  const int kt1 = (int)(((long long)(sp + 1) * KT) / a.splits);
  const int nk = kt1 - kt0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < G::NST; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&xfull[i], 1);
      mbar_init(&wempty[i], 4);
      mbar_init(&afull[i], 4);
      mbar_init(&done[i], 1);
    }
    mbar_init(dfull, 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kTcProducer) {
    // ---------------- producer: lane 0 weights, lane 1 activations ----------------
    if (lane == 0) {
      const uint8_t* wsrc = wq + ((size_t)((a.row0 >> 7) + nt) * KT + kt0) * G::WBYTES;
      const uint64_t pol = policy_evict_first();
      for (int i = 0; i < nk; ++i) {
        const int slot = i % G::NST;
        if (i >= G::NST && !mbar_wait(&wempty[slot], ((i / G::NST) - 1) & 1, a.status)) break;
        mbar_arrive_expect_tx(&wfull[slot], G::WBYTES);
        bulk_g2s_hint(smem + slot * G::STAGE, wsrc + (size_t)i * G::WBYTES, G::WBYTES, &wfull[slot], pol);
      }
    } else if (lane == 1) {
      prefetch_tmap(&xmap);
      pdl_wait();
      // the activations were written by the previous kernel with generic
      // stores; order this thread's tensor (async-proxy) reads after them
      fence_proxy_async_global();
      for (int i = 0; i < nk; ++i) {
        const int slot = i % G::NST;
        if (i >= G::NST && !mbar_wait(&done[slot], ((i / G::NST) - 1) & 1, a.status)) break;
        mbar_arrive_expect_tx(&xfull[slot], G::ABYTES);
        uint8_t* sa = smem + slot * G::STAGE + G::WBYTES;
        tma_load_2d(sa, &xmap, (kt0 + i) * kTile, z * G::MCH, &xfull[slot]);
        tma_load_2d(sa + G::MCH * 128, &xmap, (kt0 + i) * kTile + 64, z * G::MCH, &xfull[slot]);
      }
    }
    pdl_trigger();
  } else {
    // ------------- converter warps 0..3 and the MMA warp -------------
    if (warp < 4) {  // weights-side data first (independent of the preceding kernel)
      const int r = threadIdx.x;  // 0..127
      const int prow = a.row0 + nt * kTile + r;
      s_sc[r] = __half2float(wsc[logical_row(prow, a.layout, a.N)]);
      if (a.epi == EPI_QKV || a.epi == EPI_KVCOMMIT) {
        const int qd = a.nq * a.d;
        const float* gsrc = (a.row0 + nt * kTile) < qd ? a.gq : gk;
        s_gam[r] = (gsrc && r < a.d) ? gsrc[r] : 1.f;
      }
      if (a.xg_out || a.hb_out) s_gn[r] = a.g_next[logical_row(prow, a.layout, a.N) - a.row0];
    }
    if (warp == 0) tmem_alloc(s_tmem, G::TCOLS);
    tc_fence_before();
    tc_bar();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();
    if (warp < 4) {
      const int rows = G::MCH < 128 ? G::MCH : 128;
      if (a.ss_in && threadIdx.x < rows) {
        // deferred RMSNorm factor of each activation row (fixed summation order)
        const int m = z * G::MCH + threadIdx.x;
        float rf = 0.f;
        if (m < a.M) {
          float sum = 0.f;
          const float* row = a.ss_in + (size_t)m * a.nss_in;
          if ((a.nss_in & 3) == 0 && a.nss_in <= 64) {
            float4 v[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
              if (4 * q < a.nss_in) v[q] = reinterpret_cast<const float4*>(row)[q];
#pragma unroll
            for (int q = 0; q < 16; ++q)
              if (4 * q < a.nss_in) sum += ((v[q].x + v[q].y) + (v[q].z + v[q].w));
          } else {
            for (int i = 0; i < a.nss_in; ++i) sum += row[i];
          }
          rf = rsqrtf(sum / a.K + a.eps);
        }
        s_rr[threadIdx.x] = rf;
      }
      if ((a.epi == EPI_QKV || a.epi == EPI_KVCOMMIT) && threadIdx.x < rows) {
        // position of each activation row of this chunk, -1 when not written
        const int t = threadIdx.x, m = z * G::MCH + t;
        int p = -1;
        if (m < a.M) {
          if (a.epi == EPI_KVCOMMIT) {
            const int seq = m / a.rows_per_seq, slot = m - seq * a.rows_per_seq;
            const int L0 = a.len[seq];
            p = slot < commit_count(L0, a.nacc[seq], a.rows_per_seq, a.cap) ? L0 + slot : -1;
          } else if (a.c_nacc && m >= a.mc0) {  // a context row of the folded commit
            const int mc = m - a.mc0, seq = mc / a.c_rps, slot = mc - seq * a.c_rps;
            const int L0 = a.len[seq];
            p = slot < commit_count(L0, a.c_nacc[seq], a.c_rps, a.cap) ? L0 + slot : -1;
          } else {  // a block row: after the context (grown by the folded commit)
            const int seq = m / a.rows_per_seq, slot = m - seq * a.rows_per_seq;
            const int L0 = a.len[seq];
            int base = L0 < 0 ? 0 : L0;
            if (a.c_nacc) base += commit_count(L0, a.c_nacc[seq], a.c_rps, a.cap);
            p = base + slot;
          }
        }
        s_pos[t] = p;
      }
    }
    if (warp < kTcConv) {
      // ---- converter: weight row r of each of this group's k-tiles -> fp16
      // pairs in tensor memory
      const int grp = warp >> 2;
      const int r = (warp & 3) * 32 + lane;
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      for (int i = grp; i < nk; i += kTcGroups) {
        const int slot = i % G::NST, ab = slot;
        // the stage's previous MMAs first: their completion means the tile
        // that last used this ring slot (i - NST) has landed, so the slot's
        // phase parity below cannot be one phase stale
        if (i >= G::NST && !mbar_wait(&done[slot], ((i / G::NST) - 1) & 1, a.status)) break;
        if (!mbar_wait(&wfull[slot], (i / G::NST) & 1, a.status)) break;
        const uint8_t* wrow = smem + slot * G::STAGE + r * 128;
        const uint32_t ta = tmem + lane_base + G::TA + 64 * ab;
        uint4 v[8];  // this thread's 128 weight bytes of the tile
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) v[cc] = *reinterpret_cast<const uint4*>(wrow + ((cc ^ (r & 7)) << 4));
        // the weight half of the slot can be refilled once every lane has read it
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty[slot]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t words[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            // chunk word t holds columns (2t, 2t+1, 2t+8, 2t+9): fp16 pairs t and t + 4
            const uint4 u = v[4 * h + c];
            biased_u8x4_to_half2x2(u.x, words[8 * c + 0], words[8 * c + 4]);
            biased_u8x4_to_half2x2(u.y, words[8 * c + 1], words[8 * c + 5]);
            biased_u8x4_to_half2x2(u.z, words[8 * c + 2], words[8 * c + 6]);
            biased_u8x4_to_half2x2(u.w, words[8 * c + 3], words[8 * c + 7]);
          }
          tmem_st32(ta + 32 * h, words);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        // the tile's activations must have landed too: waiting here keeps that
        // wait off the single MMA-issuing thread
        if (lane == 0) {
          mbar_wait(&xfull[slot], (i / G::NST) & 1, a.status);
          mbar_arrive(&afull[ab]);
        }
      }
      pdl_trigger();
      // ---- accumulator -> P[tok][kTStride] (this thread: weight row r); two
      // groups take halves of the columns (one group when MCH = 16)
      mbar_wait(dfull, 0, a.status);
      tc_fence_after();
      float* P = reinterpret_cast<float*>(smem);
      const uint32_t td = tmem + lane_base;
      constexpr bool kHalves = kTcGroups == 2 && G::MCH >= 32;
      constexpr int CW = kHalves ? G::MCH / 2 : G::MCH;
      if (kHalves || grp == 0) {
#pragma unroll
        for (int c0 = grp * CW; c0 < grp * CW + CW; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(td + c0, v);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int j = 0; j < 16; ++j) P[(c0 + j) * kTStride + r] = __uint_as_float(v[j]);
        }
      }
    } else if (warp == kTcMma && lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = tc_idesc_f16(G::MCH);
      for (int i = 0; i < nk; ++i) {
        const int slot = i % G::NST, ab = slot;
        // afull: the A buffer is stored and the stage's activations have landed
        if (!mbar_wait(&afull[slot], (i / G::NST) & 1, a.status)) break;
        tc_fence_after();
        const uint32_t act = smem_u32(smem + slot * G::STAGE + G::WBYTES);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t bdesc = tc_sdesc_sw128(act + (ks >> 2) * (G::MCH * 128) + (ks & 3) * 32);
          tc_mma_f16_ta(tmem, tmem + G::TA + 64 * ab + 8 * ks, bdesc, idesc, (i | ks) != 0);
        }
        tc_commit(&done[slot]);
      }
      tc_commit(dfull);
    }
  }
  // the accumulator has been read (or abandoned after a timeout): free the
  // tensor memory before the reduction and epilogue
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(*s_tmem, G::TCOLS);
  }
  split_reduce_epilogue<G::MCH, G::TBYTES>(a, smem, s_sc, s_gam, s_pos, s_gn, s_rr, kout, vout, nt, z, sp, warp,
                                           lane);
}

// ------------------------------------------------------------- packing ----
template <typename T>
__device__ __forceinline__ float ld_w(const void* w, size_t i);
template <>
__device__ __forceinline__ float ld_w<float>(const void* w, size_t i) {
  return static_cast<const float*>(w)[i];
}
template <>
__device__ __forceinline__ float ld_w<__half>(const void* w, size_t i) {
  return __half2float(static_cast<const __half*>(w)[i]);
}
template <>
__device__ __forceinline__ float ld_w<__nv_bfloat16>(const void* w, size_t i) {
  return __bfloat162float(static_cast<const __nv_bfloat16*>(w)[i]);
}

// s[n] = fp16(absmax_n / 127): one warp per logical row
template <typename T>
__global__ void pack_scale_kernel(const void* w, int64_t N, int64_t K, __half* s) {
  int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= N) return;
  int lane = threadIdx.x & 31;
  float m = 0.f;
  for (int64_t k = lane; k < K; k += 32) m = fmaxf(m, fabsf(ld_w<T>(w, row * K + k)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s[row] = __float2half_rn(m / 127.0f);
}

// int8 tiles: tile (nt, kt) is 16 KB of [packed row 128][128 bytes]; the
// 16 columns of group g (columns 16 g .. 16 g + 15 of the tile) of row r
// sit in the 16-byte chunk at r * 128 + (g xor (r mod 8)) * 16, and inside
// a chunk bytes 4t .. 4t + 3 hold columns 2t, 2t + 1, 2t + 8, 2t + 9 (t < 4),
// stored as q + 128.  The tensor-memory kernel reads whole chunks (one row
// per thread), the warp-level kernel one 4-byte fragment word per lane; the
// row swizzle keeps both conflict-free.  One thread per chunk.
template <typename T>
__global__ void pack_q_kernel(const void* w, int64_t N, int64_t K, int layout, const __half* s, uint8_t* q) {
  const int64_t chunk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nchunks = N * K / 16;
  if (chunk >= nchunks) return;
  const int64_t KT = K / kTile;
  const int64_t tile = chunk >> 10;  // 1024 chunks of 16 bytes per tile
  const int within = (int)(chunk & 1023);
  const int r = within >> 3, cs = within & 7;  // row, stored chunk slot
  const int c16 = cs ^ (r & 7);                // logical 16-column group of that slot
  const int64_t nt = tile / KT, kt = tile - nt * KT;
  const int64_t prow = nt * kTile + r;
  int64_t lrow = prow;
  if (layout == 1) {
    const int64_t tl = prow >> 7, rr = prow & 127;
    lrow = rr < 64 ? tl * 64 + rr : (N >> 1) + tl * 64 + (rr - 64);
  }
  const float sc = __half2float(s[lrow]);
  uint32_t word[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    int qv = 0;
    if (sc != 0.f) {
      const int col = 2 * (e >> 2) + (e & 1) + ((e >> 1) & 1) * 8;  // column of chunk byte e
      float r_ = rintf(ld_w<T>(w, lrow * K + kt * kTile + c16 * 16 + col) / sc);
      r_ = fminf(fmaxf(r_, -127.f), 127.f);
      qv = (int)r_;
    }
    word[e >> 2] |= (uint32_t)((qv + 128) & 0xFF) << (8 * (e & 3));  // byte e of the chunk
  }
  reinterpret_cast<uint4*>(q)[chunk] = make_uint4(word[0], word[1], word[2], word[3]);
}

// int4 group scales: s[n][g] = fp16(absmax of row n over columns
// [128 g, 128 g + 128) / 7), one warp per (row, group)
template <typename T>
__global__ void pack4_scale_kernel(const void* w, int64_t N, int64_t K, __half* s) {
  const int64_t G = K / kTile;
  const int64_t item = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (item >= N * G) return;
  const int64_t row = item / G, grp = item - row * G;
  const int lane = threadIdx.x & 31;
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(ld_w<T>(w, row * K + grp * kTile + lane + 32 * e)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s[item] = __float2half_rn(m / 7.0f);
}

// one thread per 8-byte lane chunk of a packed int4 tile:
// tile (nt, kt) -> [warp 4][kstep 8][lane 32][frag(2w) word | frag(2w+1) word],
// then 128 fp16 scales (group kt of the tile's packed rows).  In a fragment
// word nibble k holds element (row g + 8 (k & 1), column 2t + (k >> 2) +
// 8 ((k >> 1) & 1)) as q + 8, so nibbles (k, k + 4) are register k's halves.
template <typename T>
__global__ void pack4_q_kernel(const void* w, int64_t N, int64_t K, int layout, const __half* s, uint8_t* q) {
  const int64_t chunk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (chunk >= N * K / 16) return;
  const int64_t KT = K / kTile;
  const int64_t tile = chunk >> 10;
  const int within = (int)(chunk & 1023);
  const int wq = within >> 8, ks = (within >> 5) & 7, ln = within & 31;
  const int64_t nt = tile / KT, kt = tile - nt * KT;
  const int g = ln >> 2, t = ln & 3;
  auto lrow_of = [&](int64_t prow) {
    if (layout != 1) return prow;
    const int64_t tl = prow >> 7, rr = prow & 127;
    return rr < 64 ? tl * 64 + rr : (N >> 1) + tl * 64 + (rr - 64);
  };
  uint32_t word[2];
#pragma unroll
  for (int f = 0; f < 2; ++f) {
    const int mg = 2 * wq + f;
    uint32_t wd = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = g + (k & 1) * 8;
      const int c = 2 * t + (k >> 2) + ((k >> 1) & 1) * 8;
      const int64_t lrow = lrow_of(nt * kTile + mg * 16 + r);
      const float sc = __half2float(s[lrow * KT + kt]);
      int qv = 0;
      if (sc != 0.f) {
        float r_ = rintf(ld_w<T>(w, lrow * K + kt * kTile + ks * 16 + c) / sc);
        qv = (int)fminf(fmaxf(r_, -7.f), 7.f);
      }
      wd |= (uint32_t)(qv + 8) << (4 * k);
    }
    word[f] = wd;
  }
  uint8_t* tb = q + tile * kTile4Bytes;
  reinterpret_cast<uint2*>(tb)[within] = make_uint2(word[0], word[1]);
  if (within < kTile)
    reinterpret_cast<__half*>(tb + 8192)[within] = s[lrow_of(nt * kTile + within) * KT + kt];
}

}  // namespace

int w8_pick_splits(int units, int KT) {
  // enough CTAs for two per SM, at most one cluster of 8 splits, and at
  // least two 128-column k-tiles per split
  // one wave at two CTAs per SM (the warp-level kernel; for the tensor-memory
  // kernel, one CTA per SM, the resident-cluster check that follows lowers it)
  int target = 2 * num_sms();
  int s = target / units;
  int smax = KT >= 4 ? KT / 2 : 1;
  if (s > smax) s = smax;
  if (s > 8) s = 8;
  if (s < 1) s = 1;
  return s;
}

// Activation rows per CTA (16, 32, 64 or 128, in units of 8).
static int pick_mt(int M, bool w4) {
  if (w4) return M <= 16 ? 2 : (M <= 32 ? 4 : 8);
  return M <= 16 ? 2 : (M <= 32 ? 4 : (M <= 64 ? 8 : 16));
}

// How many clusters of (1, s, 1) CTAs can be resident at once: clusters are
// placed within one GPC, so sizes that do not divide a GPC's CTA slots leave
// slots unused and a grid that looked like one wave may need two.  Cached per
// (device, kernel, s).
static int max_active_clusters(const void* fn, int threads, size_t smem, int s) {
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, fn, s);
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int>, int> cache;
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, s, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = s;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 1 << 30;  // unknown: do not constrain the split count
  }
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  return n;
}

cudaError_t w8_gemm(const W8Args& a0, const __half* x, cudaStream_t st, bool pdl) {
  W8Args a = a0;
  const bool w4 = a.bits == 4;
  // a QKV with a folded commit runs block rows and context rows as separate
  // 16-row chunks (they share the weight tiles through L2)
  const int mt = a.c_nacc ? 2 : pick_mt(a.M, w4);
  const int mch = mt * 8;
  const int chunks = (a.M + mch - 1) / mch;
  const int ntiles = a.nrows / kTile * (a.nl > 0 ? a.nl : 1);
  const void* fn;
  size_t smem;
  int threads;
  int occ = 1;  // resident CTAs per SM beyond the occupancy calculator's count
  if (w4) {
    fn = mt == 2 ? (const void*)wmma_gemm_kernel<2, 4>
                 : mt == 4 ? (const void*)wmma_gemm_kernel<4, 4> : (const void*)wmma_gemm_kernel<8, 4>;
    smem = mt == 2 ? Geo<2, 4>::SMEM : mt == 4 ? Geo<4, 4>::SMEM : Geo<8, 4>::SMEM;
    threads = kThreads;
  } else if (mt == 2 || (mt == 4 && (int64_t)a.nrows * a.K < kTcMinWeightBytes)) {
    // up to 16 rows, and up to 32 rows of a small projection: the warp-level
    // kernel (two CTAs per SM in split-K clusters keep these latency-bound
    // launches short)
    fn = mt == 2 ? (const void*)wmma_gemm_kernel<2, 8> : (const void*)wmma_gemm_kernel<4, 8>;
    smem = mt == 2 ? Geo<2, 8>::SMEM : Geo<4, 8>::SMEM;
    threads = kThreads;
  } else {
    // 32 rows of a large projection and above: the tensor-memory kernel (the
    // contraction is heavy enough for the legacy MMA to limit the stream)
    fn = mt == 4 ? (const void*)w8_gemm_kernel<4>
                 : mt == 8 ? (const void*)w8_gemm_kernel<8> : (const void*)w8_gemm_kernel<16>;
    smem = mt == 4 ? TcGeo<4>::SMEM : mt == 8 ? TcGeo<8>::SMEM : TcGeo<16>::SMEM;
    threads = kTcThreads;
    // a 256-column CTA shares its SM with a second one, whatever the
    // occupancy calculator says (see kTmemCols' note)
    if (mt <= 8) occ = 2;
  }
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const int units = chunks * ntiles;
  a.splits = w8_pick_splits(units, a.K / kTile);
  // keep the whole grid resident in one wave
  while (a.splits > 1 && units > occ * max_active_clusters(fn, threads, smem, a.splits)) --a.splits;
  CUtensorMap map;
  if (!encode_tmap_2d(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, (uint64_t)a.K, (uint64_t)a.M,
                      (uint64_t)a.K * 2, 64, (uint32_t)mch, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  void* args[] = {&map, &a};
  dim3 grid(ntiles, a.splits, chunks);
  return launch_kc(fn, grid, dim3(threads), smem, st, pdl, dim3(1, a.splits, 1), args);
}

cudaError_t w8_pack(const void* w, int w_dtype, int64_t N, int64_t K, int layout, uint8_t* q_out, __half* s_out,
                    cudaStream_t st) {
  dim3 b1(256);
  dim3 g1((unsigned)((N + 7) / 8));
  int64_t nchunks = N * K / 16;
  dim3 g2((unsigned)((nchunks + 255) / 256));
  if (w_dtype == 0) {
    pack_scale_kernel<float><<<g1, b1, 0, st>>>(w, N, K, s_out);
    pack_q_kernel<float><<<g2, 256, 0, st>>>(w, N, K, layout, s_out, q_out);
  } else if (w_dtype == 1) {
    pack_scale_kernel<__half><<<g1, b1, 0, st>>>(w, N, K, s_out);
    pack_q_kernel<__half><<<g2, 256, 0, st>>>(w, N, K, layout, s_out, q_out);
  } else {
    pack_scale_kernel<__nv_bfloat16><<<g1, b1, 0, st>>>(w, N, K, s_out);
    pack_q_kernel<__nv_bfloat16><<<g2, 256, 0, st>>>(w, N, K, layout, s_out, q_out);
  }
  return cudaGetLastError();
}

cudaError_t w4_pack(const void* w, int w_dtype, int64_t N, int64_t K, int layout, uint8_t* q_out, __half* s_out,
                    cudaStream_t st) {
  const int64_t items = N * (K / kTile);
  dim3 g1((unsigned)((items + 7) / 8));
  const int64_t nchunks = N * K / 16;
  dim3 g2((unsigned)((nchunks + 255) / 256));
  if (w_dtype == 0) {
    pack4_scale_kernel<float><<<g1, 256, 0, st>>>(w, N, K, s_out);
    pack4_q_kernel<float><<<g2, 256, 0, st>>>(w, N, K, layout, s_out, q_out);
  } else if (w_dtype == 1) {
    pack4_scale_kernel<__half><<<g1, 256, 0, st>>>(w, N, K, s_out);
    pack4_q_kernel<__half><<<g2, 256, 0, st>>>(w, N, K, layout, s_out, q_out);
  } else {
    pack4_scale_kernel<__nv_bfloat16><<<g1, 256, 0, st>>>(w, N, K, s_out);
    pack4_q_kernel<__nv_bfloat16><<<g2, 256, 0, st>>>(w, N, K, layout, s_out, q_out);
  }
  return cudaGetLastError();
}

}  // namespace dfl
