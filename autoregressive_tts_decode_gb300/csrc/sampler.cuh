// sampler.cuh -- block-wide token sampler.
//
// Controls from the "qwen3-tts-hip" README, section "Library Usage"
// (GenerateOptions: do_sample, top_k, top_p, temperature, repetition_penalty
// for the semantic token; subtalker_* without a penalty for acoustic tokens).
// The float rule, step by step (every step is rounded exactly as written, so
// the same logits and uniform always give the same token):
//   1. penalty rho != 1 over the stream's emitted semantic codes:
//      l = l > 0 ? l / rho : l * rho
//   2. greedy: argmax, lowest index on ties
//   3. l = l / T
//   4. order ids by (l desc, index asc), keep the first k (k <= 0 or k >= V: all)
//   5. w_i = exp_cw(l_i - l_first) in that order
//   6. top_p < 1: keep the shortest prefix whose running float sum >= top_p * Z
//   7. Z = running float sum of kept w, t = u * Z, pick the first id whose
//      running sum > t, else the last kept id.
// Selection (step 4) uses a radix select on order-preserving keys when k is
// small and a bitonic sort of all ids otherwise.
#pragma once

#include "common.cuh"

namespace q3 {

constexpr int SAMPLER_VMAX = 4096;  // largest vocabulary the block sampler takes
constexpr int SAMPLER_KSMALL = 64;  // top-k handled by radix select + warp sort
constexpr int SAMPLER_TIE_CAP = 256;

// exp(x) for x <= 0 in float, from the Cody-Waite method (Cody and Waite,
// "Software Manual for the Elementary Functions", 1980): k = rint(x log2 e),
// r = x - k ln2 with ln2 split so that k * hi is exact, a degree-7 Taylor
// polynomial of e^r in Horner form with fused multiply-adds, times 2^k.
// Inputs below -80 give 0.
__device__ __forceinline__ float exp_cw(float x) {
  if (!(x >= -80.0f)) return 0.0f;
  float kf = rintf(__fmul_rn(x, 1.44269504088896341f));
  float r = __fmaf_rn(-kf, 0.693145751953125f, x);
  r = __fmaf_rn(-kf, 1.42860682030941723212e-6f, r);
  float p = 1.98412698412698413e-4f;
  p = __fmaf_rn(p, r, 1.38888888888888889e-3f);
  p = __fmaf_rn(p, r, 8.33333333333333333e-3f);
  p = __fmaf_rn(p, r, 4.16666666666666667e-2f);
  p = __fmaf_rn(p, r, 1.66666666666666667e-1f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  int k = (int)kf;  // in [-116, 0]: 2^k is a normal float and the product is exact
  return __fmul_rn(p, __int_as_float((k + 127) << 23));
}

// Order-preserving key of a float: larger value <-> larger key; -0 and +0 equal.
__device__ __forceinline__ uint32_t fkey(float v) {
  uint32_t u = __float_as_uint(v);
  if (v == 0.0f) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SamplerSmem {
  float val[SAMPLER_VMAX];
  unsigned long long sortkey[SAMPLER_VMAX];  // (fkey << 32) | (~index): descending order
  uint32_t hist[256];
  float w[SAMPLER_VMAX];
  int cand[SAMPLER_VMAX];
  int ties[SAMPLER_TIE_CAP];
  float red[32];
  int ired[32];
  int n_gt, n_eq, remaining, pick, kept;
  uint32_t prefix;
};

__device__ __forceinline__ unsigned long long skey(float v, int i) {
  return ((unsigned long long)fkey(v) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)i);
}

// Bitonic sort, descending, of n (power of two) keys in shared memory.
__device__ inline void bitonic_desc(unsigned long long* a, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int ixj = i ^ j;
        if (ixj > i) {
          unsigned long long x = a[i], y = a[ixj];
          bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) { a[i] = y; a[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
}

// Block-wide sample over sm.val[0..V) (already holding the logits).  All threads
// of the block must call it; returns the token to every thread.
__device__ inline int block_sample(SamplerSmem& sm, int V, int do_sample, int top_k, float top_p,
                                   float temperature, float rep, const uint8_t* history, float u) {
  const int tid = threadIdx.x, nt = blockDim.x;
  if (history != nullptr && rep != 1.0f) {
    for (int i = tid; i < V; i += nt)
      if (history[i]) {
        float l = sm.val[i];
        sm.val[i] = l > 0.0f ? __fdiv_rn(l, rep) : __fmul_rn(l, rep);
      }
  }
  __syncthreads();
  if (!do_sample) {
    // argmax with lowest index on ties: max over (fkey, ~index)
    unsigned long long best = 0ull;
    for (int i = tid; i < V; i += nt) {
      unsigned long long k = skey(sm.val[i], i);
      best = k > best ? k : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
      best = t > best ? t : best;
    }
    __syncthreads();
    if ((tid & 31) == 0) sm.sortkey[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long b = 0ull;
      for (int w = 0; w < (nt + 31) / 32; ++w) b = sm.sortkey[w] > b ? sm.sortkey[w] : b;
      sm.pick = (int)(0xffffffffu - (uint32_t)(b & 0xffffffffull));
    }
    __syncthreads();
    return sm.pick;
  }
  for (int i = tid; i < V; i += nt) sm.val[i] = __fdiv_rn(sm.val[i], temperature);
  __syncthreads();
  const int K = (top_k <= 0 || top_k >= V) ? V : top_k;
  bool small = K <= SAMPLER_KSMALL;
  if (small) {
    // radix select of the K-th largest key, 8 bits at a time
    if (tid == 0) { sm.prefix = 0u; sm.remaining = K; }
    uint32_t mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = tid; b < 256; b += nt) sm.hist[b] = 0u;
      __syncthreads();
      uint32_t prefix = sm.prefix;
      for (int i = tid; i < V; i += nt) {
        uint32_t k = fkey(sm.val[i]);
        if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & 0xffu], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        int rem = sm.remaining;
        uint32_t cum = 0;
        int b = 255;
        for (; b > 0; --b) {
          if (cum + sm.hist[b] >= (uint32_t)rem) break;
          cum += sm.hist[b];
        }
        sm.remaining = rem - (int)cum;
        sm.prefix = prefix | ((uint32_t)b << shift);
      }
      mask |= 0xffu << shift;
      __syncthreads();
    }
    // gather: keys above the K-th all go in; equal keys by lowest index
    if (tid == 0) { sm.n_gt = 0; sm.n_eq = 0; }
    __syncthreads();
    const uint32_t kth = sm.prefix;
    for (int i = tid; i < V; i += nt) {
      uint32_t k = fkey(sm.val[i]);
      if (k > kth) {
        int slot = atomicAdd(&sm.n_gt, 1);
        sm.sortkey[slot] = skey(sm.val[i], i);
      } else if (k == kth) {
        int slot = atomicAdd(&sm.n_eq, 1);
        if (slot < SAMPLER_TIE_CAP) sm.ties[slot] = i;
      }
    }
    __syncthreads();
    if (sm.n_eq > SAMPLER_TIE_CAP) {
      small = false;  // pathological ties: fall back to the full sort
    } else {
      // ties: the `remaining` lowest indices, each appended after the n_gt keys
      const int n_gt = sm.n_gt, n_eq = sm.n_eq, rem = sm.remaining;
      for (int t = tid; t < n_eq; t += nt) {
        int idx = sm.ties[t], rank = 0;
        for (int s = 0; s < n_eq; ++s) rank += sm.ties[s] < idx;
        if (rank < rem) sm.sortkey[n_gt + rank] = skey(sm.val[idx], idx);
      }
      for (int t = n_gt + rem + tid; t < SAMPLER_KSMALL; t += nt) sm.sortkey[t] = 0ull;
      __syncthreads();
      bitonic_desc(sm.sortkey, SAMPLER_KSMALL);
    }
  }
  if (!small) {
    int n2 = 1;
    while (n2 < V) n2 <<= 1;
    for (int i = tid; i < n2; i += nt) sm.sortkey[i] = i < V ? skey(sm.val[i], i) : 0ull;
    __syncthreads();
    bitonic_desc(sm.sortkey, n2);
  }
  // sorted candidates: index = ~low32, value from val[]
  for (int i = tid; i < K; i += nt) sm.cand[i] = (int)(0xffffffffu - (uint32_t)(sm.sortkey[i] & 0xffffffffull));
  __syncthreads();
  const float m = sm.val[sm.cand[0]];
  for (int i = tid; i < K; i += nt) sm.w[i] = exp_cw(__fsub_rn(sm.val[sm.cand[i]], m));
  __syncthreads();
  if (tid == 0) {
    int kept = K;
    if (top_p < 1.0f) {
      float z = 0.0f;
      for (int i = 0; i < K; ++i) z = __fadd_rn(z, sm.w[i]);
      float tp = __fmul_rn(top_p, z), run = 0.0f;
      for (int i = 0; i < K; ++i) {
        run = __fadd_rn(run, sm.w[i]);
        if (run >= tp) { kept = i + 1; break; }
      }
    }
    float z = 0.0f;
    for (int i = 0; i < kept; ++i) z = __fadd_rn(z, sm.w[i]);
    float t = __fmul_rn(u, z), run = 0.0f;
    int pick = sm.cand[kept - 1];
    for (int i = 0; i < kept; ++i) {
      run = __fadd_rn(run, sm.w[i]);
      if (run > t) { pick = sm.cand[i]; break; }
    }
    sm.pick = pick;
  }
  __syncthreads();
  return sm.pick;
}

}  // namespace q3
