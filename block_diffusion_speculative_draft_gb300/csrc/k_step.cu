// k_step.cu — one whole draft step as a single persistent kernel.
//
// The draft step is a chain of ~7 dependent stages per layer, each moving a
// few to a few tens of MB of weights (mirror-sd README, "Results": the draft
// is bound by FFN weight bandwidth, not attention).  Launched as separate
// kernels, every boundary costs a launch, a pipeline fill and a tail.  Here
// one CTA per SM runs the whole step (embedding, L x {QKV + QK-norm + RoPE,
// block attention, o + residual, RMSNorm, gate|up + SwiGLU, down +
// residual, RMSNorm}, final norm, lm-head + argmax):
//  * a loader warp walks the CTA's weight schedule for the whole step and
//    fills an mbarrier ring in shared memory: per stage one weight tile (1-D
//    bulk copy of a packed int8 tile, or a 2-D TMA box of the bf16 lm-head),
//    issued as soon as the slot frees so weights stream ahead through phase
//    boundaries, plus the matching activation slice (2-D TMA, 128-byte
//    swizzle, rows past M zero-filled), issued once the phase's inputs exist;
//  * four consumer warps (32 weight rows each) convert int8 to fp16 exactly in
//    registers and issue m16n8k16 MMAs (fp32 accumulate); two CTAs share each
//    SM, since one CTA's load/consume pipeline alone tops out near 30 GB/s;
//  * the GEMM work of a phase is split stream-K style: CTA c owns a
//    contiguous range of (row tile, k-tile) units; a row tile spanning several
//    CTAs is finished by the last to arrive (atomic ticket), which sums the
//    partials in CTA order (deterministic) and runs the fused epilogue;
//  * phases are separated by a grid barrier among consumer warps (one atomic
//    per CTA on a self-resetting word whose top bit flips once per barrier,
//    bounded spin); the launch is cooperative, so all CTAs are co-resident.
// Data written by other CTAs inside the kernel is read with L1-bypassing
// loads (cp.async.cg, ld.global.cg) after the grid barrier's acquire.
// Attention reuses the ring as scratch: the loader holds back every weight
// tile scheduled after a layer's attention until that attention has ended.
// Only the activation rows M = b * B <= 32 path uses this kernel.
#include "kernels.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kNC = 4;             // consumer warps (two CTAs share an SM)
constexpr int kCT = kNC * 32;      // consumer threads
constexpr int kThr = kCT + 32;     // + loader warp
constexpr int kStage = 16384;      // weight bytes of one ring stage
constexpr int kMiscPhase = 2;      // misc[] slot: grid barriers completed
constexpr int kTS = 132;           // epilogue tile stride (floats)
constexpr int kAR = kNC * 16;      // attention query rows per item
constexpr int kNV = 8192 / 4 / kCT; // float4 per thread covering a row of up to 8192

__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory"); }

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_smem(int* p, int v) {
  asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_smem(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Grid barrier among the consumer warps of every CTA.  CTA 0 adds
// 2^31 - (G - 1), every other CTA adds 1, so the word's top bit flips exactly
// once per barrier and the low bits return to their start value (the word is
// reusable across barriers and launches).  Bounded spin.  Afterwards thread 0
// publishes the number of completed barriers to the CTA's loader warp.
__device__ void grid_sync(unsigned* bar, int* status, int* phase_cnt) {
  fence_proxy_async_global();  // our global writes may be read by TMA next
  cbar();
  if (threadIdx.x == 0) {
    const unsigned inc = blockIdx.x == 0 ? (0x80000000u - (gridDim.x - 1)) : 1u;
    __threadfence();
    const unsigned old = atomicAdd(bar, inc);
    uint32_t i = 0;
    while (((ld_acquire_u32(bar) ^ old) & 0x80000000u) == 0u) {
      if (++i > (1u << 26)) {
        atomicOr(status, kDevWaitTimeout);
        break;
      }
    }
    __threadfence();
    st_release_smem(phase_cnt, ld_acquire_smem(phase_cnt) + 1);
  }
  cbar();
}

struct Geo {
  int mt, mch;  // n8 tiles of activation rows, rows per chunk (16 or 32)
};

// unit range [u0, u1) of CTA c among G for `units` units
__device__ __forceinline__ int unit_lo(int c, int units, int G) { return (int)(((long long)c * units) / G); }
__device__ __forceinline__ int unit_owner(int u, int units, int G) {
  int c = (int)(((long long)u * G) / units);
  while (c + 1 < G && unit_lo(c + 1, units, G) <= u) ++c;
  while (c > 0 && unit_lo(c, units, G) > u) --c;
  return c;
}
// CTAs holding a non-empty piece of row tile t (units [t KT, (t+1) KT)):
// their number and the rank of CTA c among them (-1 if c holds none)
__device__ __forceinline__ void tile_contrib(int t, int KT, int units, int G, int c, int& ns, int& rank) {
  const int tlo = t * KT, thi = tlo + KT;
  const int first = unit_owner(tlo, units, G), last = unit_owner(thi - 1, units, G);
  ns = 0;
  rank = -1;
  for (int cc = first; cc <= last; ++cc) {
    const int lo = max(unit_lo(cc, units, G), tlo), hi = min(unit_lo(cc + 1, units, G), thi);
    if (lo < hi) {
      if (cc == c) rank = ns;
      ++ns;
    }
  }
}

struct Smem {
  uint8_t* ring;
  uint8_t* act;  // kActBufs x abytes
  uint8_t* x;    // union region: epilogue tile / attention / lm-head reduce
  uint64_t* full;
  uint64_t* empty;
  int* misc;  // [0] ticket flag, [2] barriers done, [32..63] row positions
  float* sc;  // [128]
  float* gam; // [128]
};


// ------------------------------------------------------ weight schedule ----
// Every weight stage of this CTA in consumption order, with the number of
// grid barriers that must have completed before its activation slice exists.
struct StageRef {
  int kind;             // 0: packed int8 tile, 1: lm-head box
  const uint8_t* wsrc;  // kind 0
  int wx, wy;           // kind 1 box coordinates
  int amap;             // activation tensor map: 0 u, 1 ao, 2 g, 3 h
  int ax;               // activation column
  int ready;            // barriers needed before the activation slice
  int wready;           // barriers needed before the weight tile (the ring
                        // doubles as attention scratch until attention ends)
};

// Iterator over the schedule (GEMMs qkv, o, gu, down per layer, then the
// lm-head tiles of this CTA).
struct StageIter {
  const StepArgs* a;
  int gi;      // GEMM index 0 .. 4L-1, then 4L for the lm-head
  int u, u1, KT;
  int t, ks;   // lm-head tile / 64-column step
  __device__ void start_gemm() {
    const int G = gridDim.x, c = blockIdx.x;
    const StepW8& w = gemm_w();
    KT = w.K / kTile;
    const int units = (w.N / kTile) * KT;
    u = unit_lo(c, units, G);
    u1 = unit_lo(c + 1, units, G);
  }
  __device__ const StepW8& gemm_w() const {
    const int l = gi >> 2, k = gi & 3;
    return k == 0 ? a->qkv[l] : (k == 1 ? a->o[l] : (k == 2 ? a->gu[l] : a->down[l]));
  }
  __device__ void init(const StepArgs* args) {
    a = args;
    gi = 0;
    t = blockIdx.x;
    ks = 0;
    start_gemm();
  }
  __device__ bool next(StageRef& r) {
    const int m = a->nsa > 1 ? 1 : 0, nbl = 7 + m;
    while (gi < 4 * a->L) {
      if (u < u1) {
        const StepW8& w = gemm_w();
        const int l = gi >> 2, k = gi & 3;
        const int base = 1 + l * nbl;
        const int tt = u / KT, kt = u - tt * KT;
        r.kind = 0;
        r.wsrc = w.q + ((size_t)tt * KT + kt) * kTileBytes;
        r.wx = r.wy = 0;
        r.amap = k == 1 ? 1 : (k == 3 ? 2 : 0);
        r.ax = kt * kTile;
        r.ready = k == 0 ? base : (k == 1 ? base + 2 + m : (k == 2 ? base + 4 + m : base + 5 + m));
        // every stage scheduled after an attention phase waits for its end
        r.wready = k >= 1 ? base + 2 : (l > 0 ? base - nbl + 2 : 0);
        ++u;
        return true;
      }
      ++gi;
      if (gi < 4 * a->L) start_gemm();
    }
    const int ntv = (a->V + 127) / 128, KS = a->H / 64;
    if (t >= ntv) return false;
    r.kind = 1;
    r.wsrc = nullptr;
    r.wx = ks * 64;
    r.wy = t * 128;
    r.amap = 3;
    r.ax = ks * 64;
    r.ready = 1 + a->L * nbl;
    r.wready = 1 + (a->L - 1) * nbl + 2;
    if (++ks == KS) {
      ks = 0;
      t += gridDim.x;
    }
    return true;
  }
};

__device__ __forceinline__ const CUtensorMap* act_map(const StepMaps& mp, int i) {
  return i == 0 ? &mp.u : (i == 1 ? &mp.ao : (i == 2 ? &mp.g : &mp.h));
}

// Loader warp (one thread).  Each ring stage completes on two arrivals: the
// weight tile, issued as soon as the slot is free (weights never depend on
// activations, so they stream ahead through phase boundaries), and the
// activation slice, issued once the grid barriers its phase needs are done.
__device__ void loader(const StepArgs& a, const StepMaps& mp, Smem& S, int mch) {
  const uint64_t pol = policy_evict_first();
  const int sb = kStage + 2 * mch * 128;
  const int RS = a.ring_stages;
  StageIter iw, ia;
  iw.init(&a);
  ia.init(&a);
  StageRef rw, ra;
  bool hw = iw.next(rw), ha = ia.next(ra);
  uint32_t gw = 0, ga = 0, idle = 0;
  int seen_a = 0, seen_w = 0;  // barriers observed by each cursor
  while (hw || ha) {
    bool progress = false;
    if (ha && ga < gw) {
      if (seen_a < ra.ready) {
        const int now = ld_acquire_smem(S.misc + kMiscPhase);
        // activation data written before these barriers is read through the
        // async proxy next: order it after the generic-proxy writes
        if (now > seen_a) fence_proxy_async_global();
        seen_a = now;
      }
      if (seen_a >= ra.ready) {
        const int slot = (int)(ga % (uint32_t)RS);
        uint8_t* st = S.ring + (size_t)slot * sb + kStage;
        const CUtensorMap* am = act_map(mp, ra.amap);
        if (ra.kind == 0) {
          mbar_arrive_expect_tx(&S.full[slot], 2 * mch * 128);
          tma_load_2d(st, am, ra.ax, 0, &S.full[slot]);
          tma_load_2d(st + mch * 128, am, ra.ax + 64, 0, &S.full[slot]);
        } else {
          mbar_arrive_expect_tx(&S.full[slot], mch * 128);
          tma_load_2d(st, am, ra.ax, 0, &S.full[slot]);
        }
        ++ga;
        ha = ia.next(ra);
        progress = true;
      }
    }
    if (hw && seen_w < rw.wready) seen_w = ld_acquire_smem(S.misc + kMiscPhase);
    if (hw && seen_w >= rw.wready) {
      const int slot = (int)(gw % (uint32_t)RS);
      if (gw < (uint32_t)RS || mbar_try_wait(&S.empty[slot], ((gw / RS) - 1) & 1)) {
        uint8_t* st = S.ring + (size_t)slot * sb;
        mbar_arrive_expect_tx(&S.full[slot], kStage);
        if (rw.kind == 0) bulk_g2s_hint(st, rw.wsrc, kStage, &S.full[slot], pol);
        else tma_load_2d_hint(st, &mp.lm, rw.wx, rw.wy, &S.full[slot], pol);
        ++gw;
        hw = iw.next(rw);
        progress = true;
      }
    }
    if (progress) {
      idle = 0;
    } else if (++idle > (1u << 28)) {
      atomicOr(a.status, kDevWaitTimeout);
      return;
    }
  }
}

// ----------------------------------------------------------- consumers ----
struct Cons {
  const StepArgs& a;
  Smem& S;
  Geo geo;
  uint32_t gc;  // weight stages consumed so far
  int warp, lane;
};

// One ring stage of a W8 GEMM: warp w owns m-groups 2w and 2w+1 (32 weight
// rows), all eight k16 steps of the 128-column tile.
template <int MT>
__device__ __forceinline__ void mma_w8_stage(Cons& C, const uint8_t* stage, const uint8_t* abuf,
                                             float (&acc)[2][MT][4]) {
  const int w = C.warp, lane = C.lane;
  const uint8_t* wl = stage + ((w * 8) * 32 + lane) * 16;
  const int g_tok_lo = (lane & 7) + ((lane >> 4) << 3);
  const int ch_hi = (lane >> 3) & 1;
  const uint32_t abase = smem_u32(abuf);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint4 wv = *reinterpret_cast<const uint4*>(wl + ks * 32 * 16);
    uint32_t af[2][4];
    biased_u8x4_to_half2x2(wv.x, af[0][0], af[0][1]);
    biased_u8x4_to_half2x2(wv.y, af[0][2], af[0][3]);
    biased_u8x4_to_half2x2(wv.z, af[1][0], af[1][1]);
    biased_u8x4_to_half2x2(wv.w, af[1][2], af[1][3]);
    const uint32_t hbase = abase + (ks >> 2) * (MT * 8 * 128);
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
}

enum { EP_QKV = 0, EP_RESID = 1, EP_SWIGLU = 2 };

// Fused epilogue on the reduced, unscaled tile T[tok][kTS] of row tile t.
template <int MT>
__device__ void step_epilogue(Cons& C, int ep, const StepW8& w, int t, const float* T, int mlo, int mhi) {
  const StepArgs& a = C.a;
  const int tid = threadIdx.x;
  const float* sc = C.S.sc;
  if (ep == EP_RESID) {
    const int items = (mhi - mlo) * 32;
    for (int base = tid; base < items; base += 2 * kCT) {
      float4 xo[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int it = base + u * kCT;
        if (it < items) {
          const int m = mlo + (it >> 5), r = 4 * (it & 31);
          xo[u] = __ldcg(reinterpret_cast<const float4*>(a.x + (size_t)m * a.H + t * kTile + r));
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int it = base + u * kCT;
        if (it >= items) continue;
        const int m = mlo + (it >> 5), r = 4 * (it & 31);
        const float* tt = T + m * kTS + r;
        float4 v = make_float4(tt[0] * sc[r] + xo[u].x, tt[1] * sc[r + 1] + xo[u].y, tt[2] * sc[r + 2] + xo[u].z,
                               tt[3] * sc[r + 3] + xo[u].w);
        *reinterpret_cast<float4*>(a.x + (size_t)m * a.H + t * kTile + r) = v;
      }
    }
    return;
  }
  if (ep == EP_SWIGLU) {
    const int F = a.F;
    for (int it = tid; it < (mhi - mlo) * 16; it += kCT) {
      const int m = mlo + (it >> 4), r = 4 * (it & 15);
      const float* tt = T + m * kTS;
      float g[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float gate = tt[r + e] * sc[r + e];
        float up = tt[r + e + 64] * sc[r + e + 64];
        g[e] = gate / (1.0f + expf(-gate)) * up;
      }
      __half2 h0 = __floats2half2_rn(g[0], g[1]), h1 = __floats2half2_rn(g[2], g[3]);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&h0);
      pk.y = *reinterpret_cast<uint32_t*>(&h1);
      *reinterpret_cast<uint2*>(a.g + (size_t)m * F + t * 64 + r) = pk;
    }
    return;
  }
  // EP_QKV: per (row, head) Q/K RMSNorm + neox RoPE; one warp per row
  const int qd = a.nq * a.d, kd = a.nkv * a.d;
  const int prow0 = t * kTile;
  const int kind = prow0 < qd ? 0 : (prow0 < qd + kd ? 1 : 2);
  const float* gam = C.S.gam;
  const int lane = C.lane;
  for (int m = mlo + C.warp; m < mhi; m += kNC) {
    const int p = C.S.misc[32 + m];
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = T[m * kTS + lane + 32 * i] * sc[lane + 32 * i];
    if (kind != 2) {
      if (a.d == 128) {
        float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = rsqrtf(ss / 128.0f + a.eps);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= inv * gam[lane + 32 * i];
        rope_rot(v[0], v[2], p, a.inv_hi[lane], a.inv_lo[lane]);
        rope_rot(v[1], v[3], p, a.inv_hi[lane + 32], a.inv_lo[lane + 32]);
      } else {
        float sa = v[0] * v[0] + v[1] * v[1], sb = v[2] * v[2] + v[3] * v[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          sa += __shfl_xor_sync(0xffffffffu, sa, o);
          sb += __shfl_xor_sync(0xffffffffu, sb, o);
        }
        const float ia = rsqrtf(sa / 64.0f + a.eps), ib = rsqrtf(sb / 64.0f + a.eps);
        v[0] *= ia * gam[lane];
        v[1] *= ia * gam[lane + 32];
        v[2] *= ib * gam[lane];
        v[3] *= ib * gam[lane + 32];
        rope_rot(v[0], v[1], p, a.inv_hi[lane], a.inv_lo[lane]);
        rope_rot(v[2], v[3], p, a.inv_hi[lane], a.inv_lo[lane]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = prow0 + lane + 32 * i;
      const __half hv = __float2half_rn(v[i]);
      if (kind == 0) a.q[(size_t)m * qd + row] = hv;
      else if (kind == 1) a.kb[(size_t)m * kd + (row - qd)] = hv;
      else a.vb[(size_t)m * kd + (row - qd - kd)] = hv;
    }
  }
}

// A W8A16 GEMM phase: activations act[M][K] fp16, weights w, epilogue ep.
// Row-tile scales (and the Q/K gamma) for the epilogue, into shared memory.
__device__ __forceinline__ void load_tile_side(Cons& C, const StepW8& w, int t, int ep, const float* gq,
                                               const float* gk) {
  if (threadIdx.x < 128) {
    const int prow = t * kTile + threadIdx.x;
    int lrow = prow;
    if (w.layout == 1) {
      const int tl = prow >> 7, rr = prow & 127;
      lrow = rr < 64 ? tl * 64 + rr : (w.N >> 1) + tl * 64 + (rr - 64);
    }
    C.S.sc[threadIdx.x] = __half2float(w.s[lrow]);
    if (ep == EP_QKV) {
      const float* gsrc = t * kTile < C.a.nq * C.a.d ? gq : gk;
      C.S.gam[threadIdx.x] = threadIdx.x < C.a.d ? gsrc[threadIdx.x] : 1.f;
    }
  }
}

// A W8A16 GEMM phase: stream-K over (row tile, k-tile) units.  A row tile
// held whole by this CTA is finished at once; a shared tile's partial is
// written without waiting, and at the end of the phase every contributor
// waits (bounded) for the tile's other partials and sums and finishes its
// own slice of activation rows, in contributor order (deterministic).
template <int MT>
__device__ void gemm_phase(Cons& C, const StepW8& w, int ep, const float* gq, const float* gk) {
  const StepArgs& a = C.a;
  const int G = gridDim.x, c = blockIdx.x;
  const int KT = w.K / kTile, ntiles = w.N / kTile, units = ntiles * KT;
  const int u0 = unit_lo(c, units, G), u1 = unit_lo(c + 1, units, G);
  const int g8 = C.lane >> 2, t4 = C.lane & 3;
  const int mch = C.geo.mch;
  float* T = reinterpret_cast<float*>(C.S.x);
  int nsplit = 0, sp_t[4], sp_rank[4], sp_ns[4];
  int u = u0;
  while (u < u1) {
    const int t = u / KT, kt0 = u - t * KT;
    const int n = min(KT - kt0, u1 - u);
    int ns, rank;
    tile_contrib(t, KT, units, G, c, ns, rank);
    if (ns == 1) load_tile_side(C, w, t, ep, gq, gk);
    float acc[2][MT][4];
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[x][j][e] = 0.f;
    const int sb = kStage + 2 * mch * 128;
    for (int i = 0; i < n; ++i) {
      const int slot = (int)(C.gc % (uint32_t)a.ring_stages);
      mbar_wait(&C.S.full[slot], (C.gc / a.ring_stages) & 1, a.status);
      const uint8_t* st = C.S.ring + (size_t)slot * sb;
      mma_w8_stage<MT>(C, st, st + kStage, acc);
      __syncwarp();
      if (C.lane == 0) mbar_arrive(&C.S.empty[slot]);
      ++C.gc;
    }
    if (ns == 1) {
      cbar();
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int j = 0; j < MT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            T[(j * 8 + 2 * t4 + (e & 1)) * kTS + C.warp * 32 + x * 16 + g8 + ((e >> 1) << 3)] = acc[x][j][e];
      cbar();
      step_epilogue<MT>(C, ep, w, t, T, 0, a.M);
      cbar();
    } else {
      float* P = a.part + ((size_t)t * a.nslots + rank) * mch * kTile;
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int j = 0; j < MT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            P[(j * 8 + 2 * t4 + (e & 1)) * kTile + C.warp * 32 + x * 16 + g8 + ((e >> 1) << 3)] = acc[x][j][e];
      __threadfence();
      cbar();
      if (threadIdx.x == 0) atomicAdd(&a.tickets[t], 1);
      if (nsplit < 4) {
        sp_t[nsplit] = t;
        sp_rank[nsplit] = rank;
        sp_ns[nsplit] = ns;
        ++nsplit;
      }
    }
    u += n;
  }
  // finish this CTA's slices of its shared tiles, last segment first (its
  // other contributors start that tile first, so it completes earliest)
  for (int q = nsplit - 1; q >= 0; --q) {
    const int t = sp_t[q], rank = sp_rank[q], ns = sp_ns[q];
    const int mlo = (rank * a.M) / ns, mhi = ((rank + 1) * a.M) / ns;
    load_tile_side(C, w, t, ep, gq, gk);
    if (threadIdx.x == 0) {
      uint32_t i = 0;
      while ((int)ld_acquire_u32(reinterpret_cast<const unsigned*>(a.tickets + t)) < ns) {
        if (++i > (1u << 26)) {
          atomicOr(a.status, kDevWaitTimeout);
          break;
        }
      }
      __threadfence();
    }
    cbar();
    if (mlo < mhi) {
      const float* P0 = a.part + (size_t)t * a.nslots * mch * kTile;
      const int items = (mhi - mlo) * 32;
      for (int it = threadIdx.x; it < items; it += kCT) {
        const int m = mlo + (it >> 5), c4 = it & 31;
        const float4* src = reinterpret_cast<const float4*>(P0 + m * kTile) + c4;
        float4 sacc = __ldcg(src);
        int k = 1;
        for (; k + 3 < ns; k += 4) {
          const float4 v0 = __ldcg(src + (size_t)(k + 0) * mch * 32);
          const float4 v1 = __ldcg(src + (size_t)(k + 1) * mch * 32);
          const float4 v2 = __ldcg(src + (size_t)(k + 2) * mch * 32);
          const float4 v3 = __ldcg(src + (size_t)(k + 3) * mch * 32);
          sacc.x += v0.x; sacc.y += v0.y; sacc.z += v0.z; sacc.w += v0.w;
          sacc.x += v1.x; sacc.y += v1.y; sacc.z += v1.z; sacc.w += v1.w;
          sacc.x += v2.x; sacc.y += v2.y; sacc.z += v2.z; sacc.w += v2.w;
          sacc.x += v3.x; sacc.y += v3.y; sacc.z += v3.z; sacc.w += v3.w;
        }
        for (; k < ns; ++k) {
          const float4 v0 = __ldcg(src + (size_t)k * mch * 32);
          sacc.x += v0.x; sacc.y += v0.y; sacc.z += v0.z; sacc.w += v0.w;
        }
        *reinterpret_cast<float4*>(T + m * kTS + 4 * c4) = sacc;
      }
      cbar();
      step_epilogue<MT>(C, ep, w, t, T, mlo, mhi);
    }
    cbar();
    if (threadIdx.x == 0) {
      // the last contributor to finish resets the tile's counters
      const int d = atomicAdd(&a.tickets[a.ntmax + t], 1);
      if (d == ns - 1) {
        a.tickets[t] = 0;
        a.tickets[a.ntmax + t] = 0;
      }
    }
  }
}

// rows of x (fp32) -> RMSNorm(x; gamma) as fp16 into out (row stride H)
__device__ void norm_rows(Cons& C, const float* gamma, __half* out) {
  const StepArgs& a = C.a;
  float* red = reinterpret_cast<float*>(C.S.x);
  for (int m = blockIdx.x; m < a.M; m += gridDim.x) {
    const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)m * a.H);
    const int n4 = a.H >> 2;
    float4 v[kNV];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int c4 = threadIdx.x + i * kCT;
      v[i] = c4 < n4 ? __ldcg(xr + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kNV; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (C.lane == 0) red[C.warp] = ss;
    cbar();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kNC; ++i) tot += red[i];
    const float inv = rsqrtf(tot / a.H + a.eps);
    const float4* g4 = reinterpret_cast<const float4*>(gamma);
#pragma unroll
    for (int i = 0; i < kNV; ++i) {
      const int c4 = threadIdx.x + i * kCT;
      if (c4 < n4) {
        const float4 gg = g4[c4];
        __half2 h0 = __floats2half2_rn(v[i].x * inv * gg.x, v[i].y * inv * gg.y);
        __half2 h1 = __floats2half2_rn(v[i].z * inv * gg.z, v[i].w * inv * gg.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&h0);
        pk.y = *reinterpret_cast<uint32_t*>(&h1);
        reinterpret_cast<uint2*>(out + (size_t)m * a.H)[c4] = pk;
      }
    }
    cbar();
  }
}

// x[m] = E[token of row m] (fp32): slot 0 the last accepted token, other
// slots the mask token (mlx-dspark v0.0.3, "Highlights").
__device__ void embed_rows(Cons& C) {
  const StepArgs& a = C.a;
  for (int m = blockIdx.x; m < a.M; m += gridDim.x) {
    const int j = m / a.B, slot = m - j * a.B;
    int tok = slot == 0 ? a.last_tok[j] : a.mask_id;
    const bool ok = tok >= 0 && tok < a.V;
    if (!ok && threadIdx.x == 0) atomicOr(a.status, 0x2);
    const uint2* e4 = reinterpret_cast<const uint2*>(a.embed + (size_t)(ok ? tok : 0) * a.H);
    float4* xr = reinterpret_cast<float4*>(a.x + (size_t)m * a.H);
    for (int c4 = threadIdx.x; c4 < (a.H >> 2); c4 += kCT) {
      const uint2 wv = ok ? e4[c4] : make_uint2(0u, 0u);
      xr[c4] = make_float4(__uint_as_float(wv.x << 16), __uint_as_float(wv.x & 0xFFFF0000u),
                           __uint_as_float(wv.y << 16), __uint_as_float(wv.y & 0xFFFF0000u));
    }
  }
}

// final norm of rows 1..B-1 of each sequence -> h (bf16) and hidden_out
__device__ void final_rows(Cons& C) {
  const StepArgs& a = C.a;
  float* red = reinterpret_cast<float*>(C.S.x);
  const int M1 = a.b * (a.B - 1);
  for (int o = blockIdx.x; o < M1; o += gridDim.x) {
    const int j = o / (a.B - 1), i = o - j * (a.B - 1);
    const float4* xr = reinterpret_cast<const float4*>(a.x + ((size_t)j * a.B + i + 1) * a.H);
    const int n4 = a.H >> 2;
    float4 v[kNV];
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < kNV; ++q) {
      const int c4 = threadIdx.x + q * kCT;
      v[q] = c4 < n4 ? __ldcg(xr + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < kNV; ++q) ss += v[q].x * v[q].x + v[q].y * v[q].y + v[q].z * v[q].z + v[q].w * v[q].w;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
    if (C.lane == 0) red[C.warp] = ss;
    cbar();
    float tot = 0.f;
#pragma unroll
    for (int q = 0; q < kNC; ++q) tot += red[q];
    const float inv = rsqrtf(tot / a.H + a.eps);
    const float4* g4 = reinterpret_cast<const float4*>(a.gamma_final);
#pragma unroll
    for (int q = 0; q < kNV; ++q) {
      const int c4 = threadIdx.x + q * kCT;
      if (c4 < n4) {
        const float4 gg = g4[c4];
        const float4 y = make_float4(v[q].x * inv * gg.x, v[q].y * inv * gg.y, v[q].z * inv * gg.z,
                                     v[q].w * inv * gg.w);
        __nv_bfloat162 b0 = __floats2bfloat162_rn(y.x, y.y), b1 = __floats2bfloat162_rn(y.z, y.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&b0);
        pk.y = *reinterpret_cast<uint32_t*>(&b1);
        reinterpret_cast<uint2*>(a.h + (size_t)o * a.H)[c4] = pk;
        if (a.hidden_out) reinterpret_cast<float4*>(a.hidden_out + (size_t)o * a.H)[c4] = y;
      }
    }
    cbar();
  }
}

// Block attention of one layer: items (sequence, kv head, key split,
// query-row chunk of <= kAR rows); non-causal over [context || block]; key
// tiles of KT keys.
template <int D, int KT>
__device__ void attn_phase(Cons& C, int l) {
  const StepArgs& a = C.a;
  constexpr int RB = D * 2;
  const int grp = a.nq / a.nkv, rows = a.B * grp;
  const int nrc = (rows + kAR - 1) / kAR;
  const int NS = a.nsa;
  const int items = a.b * a.nkv * NS * nrc;
  uint8_t* sQ = C.S.ring;  // the ring is idle while attention runs
  uint8_t* sK = sQ + kAR * RB;
  uint8_t* sV = sK + 2 * KT * RB;
  const __half* kc = a.kc + (size_t)l * a.b * a.nkv * a.cap * D;
  const __half* vc = a.vc + (size_t)l * a.b * a.nkv * a.cap * D;
  const int warp = C.warp, lane = C.lane, g8 = lane >> 2, t4 = lane & 3;
  const float sl2 = rsqrtf((float)D) * 1.4426950408889634f;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int rc = item % nrc;
    const int sp = (item / nrc) % NS;
    const int g = (item / (nrc * NS)) % a.nkv;
    const int j = item / (nrc * NS * a.nkv);
    const int r0 = rc * kAR, r1 = min(rows, r0 + kAR);
    const int nrw = (r1 - r0 + 15) / 16;  // row groups in this chunk
    int L = a.len[j];
    L = L < 0 ? 0 : (L > a.cap ? a.cap : L);
    const int total = L + a.B;
    int chunk = (total + NS - 1) / NS;
    chunk = (chunk + KT - 1) / KT * KT;
    const int k0 = min(total, sp * chunk), k1 = min(total, k0 + chunk);
    const int ntile = (k1 - k0 + KT - 1) / KT;
    cbar();  // previous item's smem reads are finished
    for (int c = threadIdx.x; c < nrw * 16 * (D / 8); c += kCT) {
      const int rl = c / (D / 8), ch = c % (D / 8);
      const int rho = r0 + rl;
      const bool ok = rho < r1;
      const __half* src = a.q;
      if (ok) {
        const int tok = rho / grp, hh = rho - tok * grp;
        src = a.q + ((size_t)(j * a.B + tok) * a.nq + (g * grp + hh)) * D + ch * 8;
      }
      cp_async16(sQ + rl * RB + ((ch ^ (rl & 7)) << 4), src, ok);
    }
    auto load_kv = [&](int buf, int tt0) {
      for (int c = threadIdx.x; c < KT * (D / 8); c += kCT) {
        const int r = c / (D / 8), ch = c % (D / 8);
        const int tk = tt0 + r;
        const bool ok = tk < k1;
        const __half* ks = kc;
        const __half* vs = vc;
        if (ok) {
          if (tk < L) {
            const size_t off = (((size_t)j * a.nkv + g) * a.cap + tk) * D + ch * 8;
            ks = kc + off;
            vs = vc + off;
          } else {
            const size_t off = ((size_t)(j * a.B + (tk - L)) * a.nkv + g) * D + ch * 8;
            ks = a.kb + off;
            vs = a.vb + off;
          }
        }
        const int so = buf * KT * RB + r * RB + ((ch ^ (r & 7)) << 4);
        cp_async16(sK + so, ks, ok);
        cp_async16(sV + so, vs, ok);
      }
    };
    load_kv(0, k0);
    cp_async_commit();
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    uint32_t qf[D / 16][4];
    const bool active = warp < nrw;
    for (int it = 0; it < ntile; ++it) {
      if (it + 1 < ntile) load_kv((it + 1) & 1, k0 + (it + 1) * KT);
      cp_async_commit();
      cp_async_wait<1>();
      cbar();
      if (active) {
        if (it == 0) {
          const uint32_t qb = smem_u32(sQ);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int ch = 2 * ks + (lane >> 4);
            ldsm_x4(qb + row * RB + ((ch ^ (row & 7)) << 4), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
          }
        }
        const uint32_t kb = smem_u32(sK + (it & 1) * KT * RB);
        const uint32_t vb = smem_u32(sV + (it & 1) * KT * RB);
        float s[KT / 8][4];
#pragma unroll
        for (int n = 0; n < KT / 8; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
          for (int n16 = 0; n16 < KT / 16; ++n16) {
            const int key = n16 * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int ch = 2 * ks + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kb + key * RB + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
            mma_f16(s[2 * n16], qf[ks], b0, b1);
            mma_f16(s[2 * n16 + 1], qf[ks], b2, b3);
          }
        }
        const int kbase = k0 + it * KT;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < KT / 8; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = kbase + n * 8 + 2 * t4 + (e & 1);
            const float v = key < k1 ? s[n][e] * sl2 : -INFINITY;
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
          corr[r] = exp2f(mrow[r] - mnew[r]);
          mrow[r] = mnew[r];
        }
        uint32_t pf[KT / 16][4];
#pragma unroll
        for (int n = 0; n < KT / 8; ++n) {
          const float p0 = exp2f(s[n][0] - mnew[0]), p1 = exp2f(s[n][1] - mnew[0]);
          const float p2 = exp2f(s[n][2] - mnew[1]), p3 = exp2f(s[n][3] - mnew[1]);
          rs[0] += p0 + p1;
          rs[1] += p2 + p3;
          __half2 h01 = __floats2half2_rn(p0, p1), h23 = __floats2half2_rn(p2, p3);
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
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk) {
#pragma unroll
          for (int dp = 0; dp < D / 16; ++dp) {
            const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int ch = 2 * dp + (lane >> 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vb + key * RB + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
            mma_f16(o[2 * dp], pf[kk], b0, b1);
            mma_f16(o[2 * dp + 1], pf[kk], b2, b3);
          }
        }
      }
      cbar();
    }
    cp_async_wait<0>();
    if (active) {
      float inv[2], lse[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        inv[r] = lrow[r] > 0.f ? 1.f / lrow[r] : 0.f;
        lse[r] = lrow[r] > 0.f ? mrow[r] + log2f(lrow[r]) : -INFINITY;
      }
      const int rows_pad = nrc * kAR;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int rho = r0 + warp * 16 + g8 + ((e >> 1) << 3);
          if (rho >= r1) continue;
          const int dim = i * 8 + 2 * t4 + (e & 1);
          const float val = o[i][e] * inv[e >> 1];
          if (NS == 1) {
            const int tok = rho / grp, hh = rho - tok * grp;
            a.ao[((size_t)(j * a.B + tok) * a.nq + g * grp + hh) * D + dim] = __float2half_rn(val);
          } else {
            a.attn_o[((((size_t)j * a.nkv + g) * NS + sp) * rows_pad + rho) * D + dim] = val;
          }
        }
      if (NS > 1 && t4 == 0) {
        const size_t lb = (((size_t)j * a.nkv + g) * NS + sp) * rows_pad;
        const int rho0 = r0 + warp * 16 + g8;
        if (rho0 < r1) a.attn_lse[lb + rho0] = lse[0];
        if (rho0 + 8 < r1) a.attn_lse[lb + rho0 + 8] = lse[1];
      }
    }
  }
}

// merge of the attention splits: items (sequence, kv head, block of rows)
template <int D>
__device__ void merge_phase(Cons& C) {
  const StepArgs& a = C.a;
  const int grp = a.nq / a.nkv, rows = a.B * grp;
  const int rows_pad = ((rows + kAR - 1) / kAR) * kAR;
  const int NS = a.nsa;
  constexpr int CPR = D / 8;            // 8-dim chunks per row
  constexpr int RPI = kCT / CPR;        // rows per item
  const int rblocks = (rows + RPI - 1) / RPI;
  const int items = a.b * a.nkv * rblocks;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int rb = item % rblocks, g = (item / rblocks) % a.nkv, j = item / (rblocks * a.nkv);
    const int rho = rb * RPI + threadIdx.x / CPR, c8 = threadIdx.x % CPR;
    if (rho >= rows) continue;
    const size_t base = ((size_t)j * a.nkv + g) * NS;
    float ls[8];
    float mmax = -INFINITY;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      ls[s] = s < NS ? __ldcg(a.attn_lse + (base + s) * rows_pad + rho) : -INFINITY;
      mmax = fmaxf(mmax, ls[s]);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float den = 0.f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (s < NS) {
        const float wgt = exp2f(ls[s] - mmax);
        const float4* src = reinterpret_cast<const float4*>(a.attn_o + ((base + s) * rows_pad + rho) * D + c8 * 8);
        const float4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
        acc[0] += wgt * v0.x; acc[1] += wgt * v0.y; acc[2] += wgt * v0.z; acc[3] += wgt * v0.w;
        acc[4] += wgt * v1.x; acc[5] += wgt * v1.y; acc[6] += wgt * v1.z; acc[7] += wgt * v1.w;
        den += wgt;
      }
    }
    const float id = 1.f / den;
    const int tok = rho / grp, hh = rho - tok * grp;
    uint4 pk;
    __half2 h0 = __floats2half2_rn(acc[0] * id, acc[1] * id), h1 = __floats2half2_rn(acc[2] * id, acc[3] * id);
    __half2 h2 = __floats2half2_rn(acc[4] * id, acc[5] * id), h3 = __floats2half2_rn(acc[6] * id, acc[7] * id);
    pk.x = *reinterpret_cast<uint32_t*>(&h0);
    pk.y = *reinterpret_cast<uint32_t*>(&h1);
    pk.z = *reinterpret_cast<uint32_t*>(&h2);
    pk.w = *reinterpret_cast<uint32_t*>(&h3);
    *reinterpret_cast<uint4*>(a.ao + ((size_t)(j * a.B + tok) * a.nq + g * grp + hh) * D + c8 * 8) = pk;
  }
}

// lm-head + argmax over this CTA's vocabulary tiles (mlx-dspark v0.0.3,
// "Highlights": the target's lm-head is shared).
template <int MT>
__device__ void lmhead_phase(Cons& C) {
  const StepArgs& a = C.a;
  const int ntv = (a.V + 127) / 128, KS = a.H / 64;
  const int mch = MT * 8;
  const int M1 = a.b * (a.B - 1);
  const int lane = C.lane, w = C.warp, g8 = lane >> 2, t4 = lane & 3;
  unsigned long long best[MT][2];
#pragma unroll
  for (int jj = 0; jj < MT; ++jj) best[jj][0] = best[jj][1] = 0ull;
  int my_tiles = blockIdx.x < ntv ? (ntv - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int total = my_tiles * KS;
  const int sb = kStage + 2 * mch * 128;
  float acc[2][MT][4];
  const int a_row0 = w * 32 + (lane & 7) + ((lane >> 3) & 1) * 8;  // + 16 mg
  const int a_ch = lane >> 4;
  const int b_tok = (lane & 7) + ((lane >> 4) << 3);
  const int b_ch = (lane >> 3) & 1;
  for (int s = 0; s < total; ++s) {
    const int ks = s % KS;
    if (ks == 0) {
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int jj = 0; jj < MT; ++jj)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[x][jj][e] = 0.f;
    }
    const int slot = (int)(C.gc % (uint32_t)a.ring_stages);
    mbar_wait(&C.S.full[slot], (C.gc / a.ring_stages) & 1, a.status);
    const uint32_t wb = smem_u32(C.S.ring + (size_t)slot * sb);
    const uint32_t hb = wb + kStage;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t af[2][4];
      const int ch = 2 * kk + a_ch;
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int row = a_row0 + 16 * x;
        ldsm_x4(wb + row * 128 + ((ch ^ (row & 7)) << 4), af[x][0], af[x][1], af[x][2], af[x][3]);
      }
#pragma unroll
      for (int p = 0; p < MT / 2; ++p) {
        const int tok = p * 16 + b_tok;
        const int chb = 2 * kk + b_ch;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(hb + tok * 128 + ((chb ^ (tok & 7)) << 4), b0, b1, b2, b3);
        mma_bf16(acc[0][2 * p], af[0], b0, b1);
        mma_bf16(acc[1][2 * p], af[1], b0, b1);
        mma_bf16(acc[0][2 * p + 1], af[0], b2, b3);
        mma_bf16(acc[1][2 * p + 1], af[1], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&C.S.empty[slot]);
    ++C.gc;
    if (ks == KS - 1) {
      const int tile = blockIdx.x + (s / KS) * gridDim.x;
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int jj = 0; jj < MT; ++jj)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int v = tile * 128 + w * 32 + 16 * x + g8 + ((e >> 1) << 3);
            const int m = jj * 8 + 2 * t4 + (e & 1);
            if (v < a.V) {
              best[jj][e & 1] = umax64(best[jj][e & 1], argmax_key(acc[x][jj][e], (uint32_t)v));
              if (a.logits_out && m < M1) a.logits_out[(size_t)m * a.V + v] = acc[x][jj][e];
            }
          }
    }
  }
  cbar();
  unsigned long long* red = reinterpret_cast<unsigned long long*>(C.S.x);
#pragma unroll
  for (int jj = 0; jj < MT; ++jj)
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      unsigned long long k = best[jj][cc];
      k = umax64(k, __shfl_xor_sync(0xffffffffu, k, 4));
      k = umax64(k, __shfl_xor_sync(0xffffffffu, k, 8));
      k = umax64(k, __shfl_xor_sync(0xffffffffu, k, 16));
      if (g8 == 0) red[w * mch + jj * 8 + 2 * t4 + cc] = k;
    }
  cbar();
  if (threadIdx.x < mch) {
    unsigned long long k = 0ull;
#pragma unroll
    for (int ww = 0; ww < kNC; ++ww) k = umax64(k, red[ww * mch + threadIdx.x]);
    if ((int)threadIdx.x < M1 && k != 0ull) atomicMax(&a.keys[threadIdx.x], k);
  }
}

template <int MT>
__device__ void consumer(const StepArgs& a, Smem& S) {
  Cons C{a, S, Geo{MT, MT * 8}, 0u, (int)(threadIdx.x >> 5), (int)(threadIdx.x & 31)};
  // positions of the block rows (constant during the step)
  if (threadIdx.x < (unsigned)a.M) {
    const int m = threadIdx.x, j = m / a.B, slot = m - j * a.B;
    const int L0 = a.len[j];
    S.misc[32 + m] = (L0 < 0 ? 0 : L0) + slot;
  }
  embed_rows(C);
  cbar();  // the same CTA normalises the rows it embedded
  norm_rows(C, a.gamma_in, a.u);
  grid_sync(a.bar, a.status, S.misc + kMiscPhase);
  for (int l = 0; l < a.L; ++l) {
    gemm_phase<MT>(C, a.qkv[l], EP_QKV, a.gamma_q + (size_t)l * a.d, a.gamma_k + (size_t)l * a.d);
    grid_sync(a.bar, a.status, S.misc + kMiscPhase);
    if (a.d == 128) {
      if (a.attn_kt == 64) attn_phase<128, 64>(C, l); else attn_phase<128, 32>(C, l);
    } else {
      attn_phase<64, 64>(C, l);
    }
    grid_sync(a.bar, a.status, S.misc + kMiscPhase);
    if (a.nsa > 1) {
      if (a.d == 128) merge_phase<128>(C); else merge_phase<64>(C);
      grid_sync(a.bar, a.status, S.misc + kMiscPhase);
    }
    gemm_phase<MT>(C, a.o[l], EP_RESID, nullptr, nullptr);
    grid_sync(a.bar, a.status, S.misc + kMiscPhase);
    norm_rows(C, a.gamma_post + (size_t)l * a.H, a.u);
    grid_sync(a.bar, a.status, S.misc + kMiscPhase);
    gemm_phase<MT>(C, a.gu[l], EP_SWIGLU, nullptr, nullptr);
    grid_sync(a.bar, a.status, S.misc + kMiscPhase);
    gemm_phase<MT>(C, a.down[l], EP_RESID, nullptr, nullptr);
    grid_sync(a.bar, a.status, S.misc + kMiscPhase);
    if (l + 1 < a.L) norm_rows(C, a.gamma_in + (size_t)(l + 1) * a.H, a.u);
    else final_rows(C);
    grid_sync(a.bar, a.status, S.misc + kMiscPhase);
  }
  lmhead_phase<MT>(C);
  grid_sync(a.bar, a.status, S.misc + kMiscPhase);
  if (blockIdx.x == 0) {
    const int M1 = a.b * (a.B - 1);
    for (int m = threadIdx.x; m < M1; m += kCT) {
      const unsigned long long k = atomicExch(&a.keys[m], 0ull);
      a.draft_out[m] = (int)key_index(k);
    }
  }
}

template <int MT>
__global__ void __launch_bounds__(kThr, 2) draft_step_kernel(const __grid_constant__ StepMaps maps,
                                                              const __grid_constant__ StepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kSB = kStage + 2 * (MT * 8) * 128;
  Smem S;
  S.ring = base;
  S.act = nullptr;
  S.x = S.ring + (size_t)a.ring_stages * kSB;  // epilogue tile / reductions
  S.full = reinterpret_cast<uint64_t*>(S.x + a.xbytes);
  S.empty = S.full + a.ring_stages;
  S.misc = reinterpret_cast<int*>(S.empty + a.ring_stages);
  S.sc = reinterpret_cast<float*>(S.misc + 64);
  S.gam = S.sc + 128;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.ring_stages; ++i) {
      mbar_init(&S.full[i], 2);  // weight arrival + activation arrival
      mbar_init(&S.empty[i], kNC);
    }
    for (int i = 0; i < 64; ++i) S.misc[i] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == kCT) {
    prefetch_tmap(&maps.lm);
    prefetch_tmap(&maps.u);
    prefetch_tmap(&maps.ao);
    prefetch_tmap(&maps.g);
    prefetch_tmap(&maps.h);
    loader(a, maps, S, MT * 8);
  } else if (threadIdx.x < kCT) {
    consumer<MT>(a, S);
  }
  __syncthreads();
}

}  // namespace

int step_max_mch() { return 32; }

size_t step_stage_bytes(int mt) { return kStage + 2 * (size_t)(mt * 8) * 128; }

size_t step_smem_bytes(int mt, int ring_stages, size_t xbytes) {
  return 1024 + (size_t)ring_stages * step_stage_bytes(mt) + xbytes + 2 * ring_stages * 8 + 64 * 4 + 256 * 4;
}

size_t step_x_bytes(int mt, int d, int H) {
  const size_t tile = (size_t)(mt * 8) * kTS * 4;
  const size_t lm = (size_t)kNC * (mt * 8) * 8;
  size_t x = tile > lm ? tile : lm;
  (void)d;
  (void)H;
  return (x + 1023) / 1024 * 1024;
}

// attention scratch (aliases the ring): query rows + double-buffered K and V
size_t step_attn_bytes(int d, int kt) { return (size_t)kAR * d * 2 + 4 * (size_t)kt * d * 2; }

int step_threads() { return kThr; }

int step_occupancy(int mt, size_t smem) {
  const void* fn = mt == 2 ? (const void*)draft_step_kernel<2> : (const void*)draft_step_kernel<4>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThr, smem) != cudaSuccess) return 0;
  return n;
}

int step_nslots(int units_ntiles, int KT, int G) {
  // largest number of CTAs that share one row tile
  const int units = units_ntiles * KT;
  auto lo = [&](int c) { return (int)(((long long)c * units) / G); };
  auto owner = [&](int u) {
    int c = (int)(((long long)u * G) / units);
    while (c + 1 < G && lo(c + 1) <= u) ++c;
    while (c > 0 && lo(c) > u) --c;
    return c;
  };
  int best = 1;
  for (int t = 0; t < units_ntiles; ++t) {
    const int tlo = t * KT, thi = tlo + KT;
    int ns = 0;
    for (int cc = owner(tlo); cc <= owner(thi - 1); ++cc) {
      const int l0 = lo(cc) > tlo ? lo(cc) : tlo, h0 = lo(cc + 1) < thi ? lo(cc + 1) : thi;
      if (l0 < h0) ++ns;
    }
    if (ns > best) best = ns;
  }
  return best;
}

cudaError_t draft_step(const StepArgs& a0, const __nv_bfloat16* lm_head, cudaStream_t st, int G) {
  StepArgs a = a0;
  const int mt = a.M <= 16 ? 2 : 4;
  const uint32_t mch = mt * 8;
  StepMaps mp;
  const int M1 = a.b * (a.B - 1);
  bool ok = encode_tmap_2d(&mp.lm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, lm_head, (uint64_t)a.H, (uint64_t)a.V,
                           (uint64_t)a.H * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&mp.u, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.u, (uint64_t)a.H, (uint64_t)a.M,
                            (uint64_t)a.H * 2, 64, mch, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&mp.ao, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.ao, (uint64_t)a.nq * a.d, (uint64_t)a.M,
                            (uint64_t)a.nq * a.d * 2, 64, mch, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&mp.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.g, (uint64_t)a.F, (uint64_t)a.M,
                            (uint64_t)a.F * 2, 64, mch, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_tmap_2d(&mp.h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.h, (uint64_t)a.H, (uint64_t)M1,
                            (uint64_t)a.H * 2, 64, mch, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  const size_t smem = step_smem_bytes(mt, a.ring_stages, a.xbytes);
  const void* fn = mt == 2 ? (const void*)draft_step_kernel<2> : (const void*)draft_step_kernel<4>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {&mp, &a};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kThr);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace dfl
