// ptx.cuh — inline-PTX building blocks for the sm_103a kernels: mbarriers,
// bulk / tensor (TMA) copies, programmatic dependent launch, ldmatrix and the
// warp-level MMA used by the skinny GEMMs.  Every wait is bounded: after
// kSpinLimit polls it gives up, raises a status bit and returns false, so a
// lost arrival can never hang the GPU.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dfl {

// Status-word bit raised when a bounded wait gives up.
constexpr int kDevWaitTimeout = 0x100;
constexpr uint32_t kSpinLimit = 1u << 26;  // ~ seconds of polling

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on phase `parity`; false (and *status |= timeout) if it never
// completes.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  if (status) atomicOr(status, kDevWaitTimeout);
  return false;
}

// ------------------------------------------------------------ bulk copies --
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes, both
// addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Same, with an L2 eviction-priority hint (streamed-once weights).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 2-D tiled tensor copy (TMA) global -> shared.  x (innermost) coordinate in
// elements must keep x * elem_size a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// 3-D tiled tensor copy global -> shared (same x alignment rule).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Bring a global range (16-byte aligned, multiple of 16 bytes) into L2
// without touching shared memory.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Pieces [i0, i1) of a strided L2 prefetch job (piece i covers
// [base + i * stride, + bytes)), dealt round-robin to the ncta CTAs of the
// grid and issued in 32 KB bulk prefetches.  base, stride and bytes are
// multiples of 16 bytes.
__device__ __forceinline__ void prefetch_l2_job(const uint8_t* base, size_t stride, uint32_t bytes, int i0, int i1,
                                                unsigned cta, unsigned ncta) {
  constexpr uint32_t kPiece = 32u << 10;
  for (int i = i0 + (int)cta; i < i1; i += (int)ncta) {
    const uint8_t* p = base + (size_t)i * stride;
    for (uint32_t off = 0; off < bytes; off += kPiece)
      prefetch_l2_bulk(p + off, bytes - off < kPiece ? bytes - off : kPiece);
  }
}
// Same for one box of a 2-D tensor map.
__device__ __forceinline__ void prefetch_l2_tile(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}
// Orders this thread's generic-proxy global accesses with async-proxy (TMA)
// accesses to global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Orders this thread's earlier generic-proxy accesses to shared memory with
// its later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ------------------------------------------- programmatic dependent launch --
// Block until the preceding kernel in the stream has completed and its writes
// are visible (no-op when launched without the PDL attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to begin launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------- cp.async ----
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool pred) {
  int n = pred ? 16 : 0;  // zero-fill when out of range
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------ thread-block clusters ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Full cluster barrier: every thread of every CTA in the cluster arrives
// (release) and waits (acquire), so shared-memory writes made before it are
// visible to peer CTAs after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync, for overlapping the wait with other work.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// Arrive without release semantics (nothing this thread wrote before it
// needs to be visible to the cluster through the barrier).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Bulk copy from this CTA's shared memory into a peer's (shared::cluster
// addresses for the destination and its mbarrier), completion counted in
// bytes on that mbarrier.  16-byte aligned addresses, size a multiple of 16.
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until this thread's committed bulk copies have finished reading
// their sources.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Rotates (x1, x2) by the RoPE angle pos * inv, where inv = inv_hi + inv_lo
// (a double split into two floats on the host), in single precision only
// (FP64 issue is far too slow on this part for an epilogue).  The product is
// carried as a float pair (the FMA gives the exact rounding error of
// pos * inv_hi), and 2*pi is removed by Cody-Waite reduction with 2*pi split
// into two floats (W. J. Cody, W. Waite, "Software Manual for the Elementary
// Functions", 1980), so the reduced angle r (|r| <= pi + 1e-5) is within
// about 1e-6 rad of the exact one for pos < 2^24.  On that range the
// hardware sine/cosine approximation (__sincosf) has an absolute error near
// 2^-21, far below the fp16 rounding of the rotated outputs, at a fraction of
// the latency of the general sincosf.
__device__ __forceinline__ void rope_rot(float& x1, float& x2, int pos, float inv_hi, float inv_lo) {
  constexpr float kTwoPiHi = 0x1.921fb6p+2f;    // float(2 pi)
  constexpr float kTwoPiLo = -0x1.777a5cp-23f;  // float(2 pi - kTwoPiHi)
  constexpr float kInvTwoPi = 0x1.45f306p-3f;
  const float p = (float)pos;  // exact below 2^24
  const float a_hi = p * inv_hi;
  const float a_lo = fmaf(p, inv_lo, fmaf(p, inv_hi, -a_hi));
  const float k = rintf(a_hi * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, a_hi);
  r = fmaf(-k, kTwoPiLo, r);
  r += a_lo;
  float sn, cs;
  __sincosf(r, &sn, &cs);
  const float a = x1, b = x2;
  x1 = a * cs - b * sn;
  x2 = b * cs + a * sn;
}

// Stores into another CTA's shared memory (made visible to it by the next
// cluster barrier's release/acquire pair).
__device__ __forceinline__ void st_dsmem_f2(uint32_t addr, float x, float y) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float x) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(x) : "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------- ldmatrix --
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// --------------------------------------------------------------- warp MMA --
// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------- int8 -> fp16, exactly --
// Four biased bytes (q + 128, packed by dflash_pack_w8a16) to two half2
// holding q exactly.  Each byte b is placed under the fp16 exponent of 1024
// (bits 0x6400 | b, i.e. the value 1024 + b) and 1024 + 128 is subtracted;
// every intermediate is an integer below 2048, so no rounding occurs.  This is
// the magic-number conversion of Kim et al., "Who Says Elephants Can't Run:
// Bringing Large Scale MoE Models into Cloud Scale Production" (2022).
__device__ __forceinline__ void biased_u8x4_to_half2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t kMagic = 0x64646464u;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(w), "r"(kMagic));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(w), "r"(kMagic));
  const uint32_t kBias = 0x64806480u;  // half2(1152, 1152)
  asm("sub.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(kBias));
  asm("sub.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(kBias));
}

// ------------------------------------------------ ordered argmax keys ------
// 64-bit key whose unsigned maximum is the largest float and, among equal
// floats, the LOWEST index.  -0.0 is folded onto +0.0 first.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<unsigned long long>(ord) << 32) | static_cast<unsigned long long>(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
  return 0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
  uint32_t ord = static_cast<uint32_t>(k >> 32);
  uint32_t b = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
  return __uint_as_float(b);
}
__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long warp_max64(unsigned long long k) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k = umax64(k, __shfl_xor_sync(0xffffffffu, k, o));
  return k;
}

}  // namespace dfl
