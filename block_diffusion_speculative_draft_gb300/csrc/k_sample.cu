// k_sample.cu — temperature speculative-sampling accept (greedy proposals).
//
// At temperature T > 0 the loop stays lossless: every emitted token is an
// exact sample from the target at T (mlx-dspark v0.0.3 release notes,
// "Highlights": "the same acceptance rule as DSpark").  With this drafter's
// greedy proposals (one-hot q) the speculative-sampling rule is
//   accept draft i  iff  u_acc[i] < p_i(x_i),   p_i = softmax(logits[i] / T),
// n = leading accepted drafts, and one categorical draw: from p_n without
// x_n (the residual max(0, p_n - q_n), renormalised) when n < D, from p_D
// when n = D < R, none when n = D = R.  The draw is the Gumbel-max trick over
// caller-supplied uniforms u_sample[V]: argmax_v z_v / T - log(-log u_v).
//
// Two launches:
//  1. stats: one CTA per (vocabulary slice, row); each computes the online
//     maximum and exp-sum of z / T over its slice (and the draft token's
//     z / T); the last CTA of a sequence (atomic ticket) merges the slices,
//     takes the accept decisions in order, and records the row to sample and
//     the token it must exclude.
//  2. pick: one CTA per (vocabulary slice, sequence) over that single row;
//     64-bit (score, lowest index) keys reduced per CTA, the last CTA of the
//     sequence takes the maximum and writes the outputs.
// Only one row per sequence is scanned for the draw, so the transcendental
// work is V per sequence, not R x V.
#include "kernels.h"
#include "ptx.cuh"

namespace dfl {

namespace {

constexpr int kThr = 256;

// online (max, sum exp(t - max)) of one more value
__device__ __forceinline__ void online_add(float& m, float& s, float t) {
  if (t > m) {
    s = s * expf(m - t) + 1.f;  // s = 0 while m = -inf: exp(-inf) = 0
    m = t;
  } else {
    s += expf(t - m);
  }
}
__device__ __forceinline__ void online_merge(float& m, float& s, float m2, float s2) {
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else if (m2 > -INFINITY) {
    s += s2 * expf(m2 - m);
  }
}

__global__ void __launch_bounds__(kThr) sample_stats_kernel(const SampleArgs a) {
  __shared__ float sm[kThr / 32], ss[kThr / 32];
  __shared__ int flag;
  pdl_wait();
  const int row = blockIdx.y, p = blockIdx.x;
  const int j = row / a.R, r = row - j * a.R;
  const float* lr = a.logits + (size_t)row * a.V;
  const int64_t c0 = (int64_t)p * a.chunk;
  const int64_t c1 = c0 + a.chunk < a.V ? c0 + a.chunk : a.V;
  float m = -INFINITY, s = 0.f;
  for (int64_t i = c0 + threadIdx.x; i < c1; i += kThr) online_add(m, s, __ldcs(lr + i) / a.T);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    online_merge(m, s, m2, s2);
  }
  if ((threadIdx.x & 31) == 0) {
    sm[threadIdx.x >> 5] = m;
    ss[threadIdx.x >> 5] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = sm[0], S = ss[0];
    for (int w = 1; w < kThr / 32; ++w) online_merge(M, S, sm[w], ss[w]);
    a.part[(size_t)row * a.P + p] = make_float2(M, S);
    if (r < a.D) {
      const int x = a.draft[(size_t)j * a.D + r];
      if (x >= c0 && x < c1) a.zx[row] = lr[x] / a.T;
    }
    __threadfence();
    const int old = atomicAdd(&a.tickets[j], 1);
    flag = old == a.R * a.P - 1;
  }
  __syncthreads();
  pdl_trigger();
  if (!flag) return;
  __threadfence();
  // last CTA of sequence j: merge the slices of each row (one warp per row)
  __shared__ float pacc[64];
  for (int rr = threadIdx.x >> 5; rr < a.D; rr += kThr / 32) {
    const float2* pr = a.part + ((size_t)j * a.R + rr) * a.P;
    float M = -INFINITY, S = 0.f;
    for (int q = threadIdx.x & 31; q < a.P; q += 32) {
      const float2 v = __ldcg(pr + q);
      online_merge(M, S, v.x, v.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, M, o), s2 = __shfl_xor_sync(0xffffffffu, S, o);
      online_merge(M, S, m2, s2);
    }
    if ((threadIdx.x & 31) == 0) {
      // a draft token outside the vocabulary has probability 0: rejected
      const int x = a.draft[(size_t)j * a.D + rr];
      pacc[rr] = (x >= 0 && x < a.V) ? expf(__ldcg(a.zx + (size_t)j * a.R + rr) - M) / S : 0.f;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    while (n < a.D && a.u_acc[(size_t)j * a.D + n] < pacc[n]) ++n;
    a.n_out[j] = n;
    a.sel[2 * j] = n < a.D ? n : (a.D < a.R ? a.D : -1);
    a.sel[2 * j + 1] = n < a.D ? a.draft[(size_t)j * a.D + n] : -1;
    a.tickets[j] = 0;
  }
}

__global__ void __launch_bounds__(kThr) sample_pick_kernel(const SampleArgs a) {
  __shared__ unsigned long long sk[kThr / 32];
  __shared__ int flag;
  pdl_wait();
  const int j = blockIdx.y, p = blockIdx.x;
  const int row = __ldcg(a.sel + 2 * j), excl = __ldcg(a.sel + 2 * j + 1);
  unsigned long long best = 0ull;
  if (row >= 0) {
    const float* lr = a.logits + ((size_t)j * a.R + row) * a.V;
    const float* us = a.u_sample + (size_t)j * a.V;
    const int64_t c0 = (int64_t)p * a.chunk2;
    const int64_t c1 = c0 + a.chunk2 < a.V ? c0 + a.chunk2 : a.V;
    for (int64_t i = c0 + threadIdx.x; i < c1; i += kThr) {
      if (i == excl) continue;
      // Gumbel-max score, decided in fp32: z / T - log(-log u)
      const float sc = __ldcs(lr + i) / a.T - logf(-logf(__ldcs(us + i)));
      best = umax64(best, argmax_key(sc, (uint32_t)i));
    }
  }
  best = warp_max64(best);
  if ((threadIdx.x & 31) == 0) sk[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long k = sk[0];
    for (int w = 1; w < kThr / 32; ++w) k = umax64(k, sk[w]);
    a.keys[(size_t)j * a.P2 + p] = k;
    __threadfence();
    const int old = atomicAdd(&a.tickets[a.b + j], 1);
    flag = old == a.P2 - 1;
  }
  __syncthreads();
  pdl_trigger();
  if (!flag) return;
  __threadfence();
  if (threadIdx.x < 32) {
    unsigned long long k = 0ull;
    for (int q = threadIdx.x; q < a.P2; q += 32) k = umax64(k, __ldcg(a.keys + (size_t)j * a.P2 + q));
    k = warp_max64(k);
    if (threadIdx.x == 0) {
      const int n = __ldcg(a.n_out + j);
      const int corr = row >= 0 && k != 0ull ? (int)key_index(k) : -1;
      const int* dr = a.draft + (size_t)j * a.D;
      a.corr_out[j] = corr;
      if (a.next_tok) a.next_tok[j] = corr >= 0 ? corr : (n > 0 ? dr[n - 1] : -1);
      if (a.emitted)
        for (int q = 0; q < a.R; ++q) a.emitted[(size_t)j * a.R + q] = q < n ? dr[q] : (q == n ? corr : -1);
      a.tickets[a.b + j] = 0;
    }
  }
}

}  // namespace

int sample_parts(int b, int R, int64_t V) {
  int P = (4 * num_sms() + b * R - 1) / (b * R);
  const int64_t pmax = (V + 2047) / 2048;
  if (P > pmax) P = (int)pmax;
  return P < 1 ? 1 : P;
}
int sample_parts2(int b, int64_t V) {
  int P = (2 * num_sms() + b - 1) / b;
  const int64_t pmax = (V + 1023) / 1024;
  if (P > pmax) P = (int)pmax;
  return P < 1 ? 1 : P;
}

// Workspace layout (256-byte aligned pieces): tickets [2b], slice stats
// [b R][P], draft-token z / T [b R], selection [b][2], slice keys [b][P2].
// With base null only the size is computed.
static size_t carve_sample(int b, int R, int64_t V, uint8_t* base, SampleArgs* a) {
  const int P = sample_parts(b, R, V), P2 = sample_parts2(b, V);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* q = base ? base + off : nullptr;
    off = (off + bytes + 255) & ~size_t(255);
    return q;
  };
  int* tickets = reinterpret_cast<int*>(take((size_t)2 * b * sizeof(int)));
  float2* part = reinterpret_cast<float2*>(take((size_t)b * R * P * sizeof(float2)));
  float* zx = reinterpret_cast<float*>(take((size_t)b * R * sizeof(float)));
  int* sel = reinterpret_cast<int*>(take((size_t)2 * b * sizeof(int)));
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(take((size_t)b * P2 * sizeof(unsigned long long)));
  if (a) {
    a->P = P;
    a->P2 = P2;
    a->tickets = tickets;
    a->part = part;
    a->zx = zx;
    a->sel = sel;
    a->keys = keys;
  }
  return off;
}

size_t sample_ws_bytes(int b, int R, int64_t V) { return carve_sample(b, R, V, nullptr, nullptr); }

cudaError_t verify_sample(const float* logits, const int* draft, int b, int R, int D, int64_t V, float T,
                          const float* u_acc, const float* u_sample, int* n_out, int* corr_out, int* emitted,
                          int* next_tok, void* ws, cudaStream_t st, bool pdl) {
  SampleArgs a;
  a.logits = logits;
  a.draft = draft;
  a.u_acc = u_acc;
  a.u_sample = u_sample;
  a.b = b;
  a.R = R;
  a.D = D;
  a.V = V;
  a.T = T;
  carve_sample(b, R, V, static_cast<uint8_t*>(ws), &a);
  a.chunk = (V + a.P - 1) / a.P;
  a.chunk2 = (V + a.P2 - 1) / a.P2;
  a.n_out = n_out;
  a.corr_out = corr_out;
  a.emitted = emitted;
  a.next_tok = next_tok;
  void* args[] = {&a};
  cudaError_t e = launch_k((const void*)sample_stats_kernel, dim3(a.P, b * R), dim3(kThr), 0, st, pdl, args);
  if (e != cudaSuccess) return e;
  return launch_k((const void*)sample_pick_kernel, dim3(a.P2, b), dim3(kThr), 0, st, true, args);
}

}  // namespace dfl
