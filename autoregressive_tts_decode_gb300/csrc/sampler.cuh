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
// Selection (step 4), in the block sampler of the layered step (group_sample):
// a radix select on order-preserving keys when k is small (ties at the k-th
// value resolved by lowest index) and a bitonic sort of all ids otherwise.  In
// the persistent frame kernel (fast_sample, at the end): a lower bound on the
// k-th largest key from the lanes' maxima, the keys above it gathered and
// ranked by counting.  Both give the same ordered candidates, so the same draw.
#pragma once

#include "common.cuh"

namespace q3 {

constexpr int SAMPLER_VMAX = 4096;  // largest vocabulary the block sampler takes
constexpr int SAMPLER_KSMALL = 64;  // top-k handled by radix select + warp sort

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
  int wsum[32];
  int n_gt, remaining, pick;
  uint32_t prefix;
  static constexpr bool kFullSort = true;
};

__device__ __forceinline__ unsigned long long skey(float v, int i) {
  return ((unsigned long long)fkey(v) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)i);
}

// Sampler scratch for callers that only take greedy or 1 <= top_k <= 64
// (the persistent frame kernel): the logits plus 64-entry candidate arrays.
struct SamplerSmemSmall {
  float val[SAMPLER_VMAX];
  unsigned long long sortkey[SAMPLER_KSMALL];
  uint32_t hist[256];
  float w[SAMPLER_KSMALL];
  int cand[SAMPLER_KSMALL];
  int wsum[32];
  int n_gt, remaining, pick;
  uint32_t prefix;
  static constexpr bool kFullSort = false;  // callers keep top_k within SAMPLER_KSMALL
};

// Thread-group description for the block sampler: the participating threads
// (tid in [0, nt)) and their barrier.  BlockGroup is a whole thread block.
struct BlockGroup {
  __device__ static int tid() { return threadIdx.x; }
  __device__ static int nt() { return blockDim.x; }
  __device__ static void sync() { __syncthreads(); }
};

// Bitonic sort, descending, of n (power of two) keys in shared memory.
template <class G>
__device__ inline void bitonic_desc(unsigned long long* a, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = G::tid(); i < n; i += G::nt()) {
        int ixj = i ^ j;
        if (ixj > i) {
          unsigned long long x = a[i], y = a[ixj];
          bool desc = (i & k) == 0;
          if (desc ? (x < y) : (x > y)) { a[i] = y; a[ixj] = x; }
        }
      }
      G::sync();
    }
  }
}

template <class G, class SM>
__device__ inline void full_sort(SM& sm, int V);

// Group-wide sample over sm.val[0..V) (already holding the logits).  Every
// thread of the group must call it; returns the token to all of them.  With
// full_sort == false the caller guarantees 1 <= top_k <= SAMPLER_KSMALL (or
// greedy), so sortkey/w/cand need only SAMPLER_KSMALL entries.
template <class G, class SM>
__device__ inline int group_sample(SM& sm, int V, int do_sample, int top_k, float top_p,
                                   float temperature, float rep, const uint8_t* history, float u) {
  const int tid = G::tid(), nt = G::nt();
  if (history != nullptr && rep != 1.0f) {
    for (int i = tid; i < V; i += nt)
      if (history[i]) {
        float l = sm.val[i];
        sm.val[i] = l > 0.0f ? __fdiv_rn(l, rep) : __fmul_rn(l, rep);
      }
  }
  G::sync();
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
    G::sync();
    if ((tid & 31) == 0) sm.sortkey[tid >> 5] = best;
    G::sync();
    if (tid == 0) {
      unsigned long long b = 0ull;
      for (int w = 0; w < (nt + 31) / 32; ++w) b = sm.sortkey[w] > b ? sm.sortkey[w] : b;
      sm.pick = (int)(0xffffffffu - (uint32_t)(b & 0xffffffffull));
    }
    G::sync();
    return sm.pick;
  }
  for (int i = tid; i < V; i += nt) sm.val[i] = __fdiv_rn(sm.val[i], temperature);
  G::sync();
  const int K = (top_k <= 0 || top_k >= V) ? V : top_k;
  const bool small = K <= SAMPLER_KSMALL;
  if (small) {
    // radix select of the K-th largest key, 8 bits at a time
    if (tid == 0) { sm.prefix = 0u; sm.remaining = K; }
    uint32_t mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = tid; b < 256; b += nt) sm.hist[b] = 0u;
      G::sync();
      uint32_t prefix = sm.prefix;
      for (int i = tid; i < V; i += nt) {
        uint32_t k = fkey(sm.val[i]);
        if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> shift) & 0xffu], 1u);
      }
      G::sync();
      if (tid < 32) {
        // warp 0: lane l holds bins 255-8l .. 248-8l (descending); find the bin
        // where the running count from the top reaches `remaining`
        const int rem = sm.remaining;
        uint32_t c[8], tot = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) { c[q] = sm.hist[255 - 8 * tid - q]; tot += c[q]; }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += t;
        }
        const uint32_t excl = incl - tot;
        const bool mine = excl < (uint32_t)rem && incl >= (uint32_t)rem;
        if (mine) {
          uint32_t cum = excl;
          int q = 0;
          for (; q < 7; ++q) {
            if (cum + c[q] >= (uint32_t)rem) break;
            cum += c[q];
          }
          sm.remaining = rem - (int)cum;
          sm.prefix = prefix | ((uint32_t)(255 - 8 * tid - q) << shift);
        }
      }
      mask |= 0xffu << shift;
      G::sync();
    }
    // gather: keys above the K-th all go in (any order; sorted below); of the
    // keys equal to the K-th, the `remaining` lowest indices, found with an
    // ordered count over contiguous index ranges so any number of ties works.
    if (tid == 0) sm.n_gt = 0;
    G::sync();
    const uint32_t kth = sm.prefix;
    const int rem = sm.remaining;
    const int per = (V + nt - 1) / nt, lo = tid * per, hi = min(V, lo + per);
    int my_eq = 0;
    for (int i = lo; i < hi; ++i) {
      uint32_t k = fkey(sm.val[i]);
      if (k > kth) {
        int slot = atomicAdd(&sm.n_gt, 1);
        sm.sortkey[slot] = skey(sm.val[i], i);
      } else if (k == kth) {
        ++my_eq;
      }
    }
    // exclusive prefix of my_eq over threads in index order
    int incl = my_eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, incl, o);
      if ((tid & 31) >= o) incl += t;
    }
    if ((tid & 31) == 31) sm.wsum[tid >> 5] = incl;
    G::sync();
    if (tid < 32) {
      int v = tid < (nt + 31) / 32 ? sm.wsum[tid] : 0, vi = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, vi, o);
        if (tid >= o) vi += t;
      }
      sm.wsum[tid] = vi - v;  // exclusive over warps
    }
    G::sync();
    int rank = sm.wsum[tid >> 5] + incl - my_eq;
    const int n_gt = K - rem;
    for (int i = lo; i < hi && rank < rem; ++i)
      if (fkey(sm.val[i]) == kth) sm.sortkey[n_gt + rank++] = skey(sm.val[i], i);
    for (int t = K + tid; t < SAMPLER_KSMALL; t += nt) sm.sortkey[t] = 0ull;
    G::sync();
    bitonic_desc<G>(sm.sortkey, SAMPLER_KSMALL);
  }
  if (!small) {
    int n2 = 1;
    while (n2 < V) n2 <<= 1;
    full_sort<G>(sm, V);
  }
  // sorted candidates: index = ~low32, value from val[]
  for (int i = tid; i < K; i += nt) sm.cand[i] = (int)(0xffffffffu - (uint32_t)(sm.sortkey[i] & 0xffffffffull));
  G::sync();
  const float m = sm.val[sm.cand[0]];
  for (int i = tid; i < K; i += nt) sm.w[i] = exp_cw(__fsub_rn(sm.val[sm.cand[i]], m));
  G::sync();
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
  G::sync();
  return sm.pick;
}

template <class G, class SM>
__device__ inline void full_sort(SM& sm, int V) {
  int n2 = 1;
  while (n2 < V) n2 <<= 1;
  for (int i = G::tid(); i < n2; i += G::nt()) sm.sortkey[i] = i < V ? skey(sm.val[i], i) : 0ull;
  G::sync();
  bitonic_desc<G>(sm.sortkey, n2);
}

__device__ inline int block_sample(SamplerSmem& sm, int V, int do_sample, int top_k, float top_p,
                                   float temperature, float rep, const uint8_t* history, float u) {
  return group_sample<BlockGroup>(sm, V, do_sample, top_k, top_p, temperature, rep, history, u);
}

}  // namespace q3

namespace q3 {

// ---------------------------------------------------------------------------
// Register-resident sampler of the frame kernel (fast_sample, at the end).
constexpr int FAST_NT = 256;
constexpr int FAST_V4 = SAMPLER_VMAX / 4 / FAST_NT;  // float4 of logits per thread
constexpr int FAST_VPT = 4 * FAST_V4;              // 16 logits per thread at most
constexpr int FAST_NW = FAST_NT / 32;
constexpr int FAST_TOP = 8;                        // lane maxima per warp entering theta
constexpr int FAST_CAP = 256;                      // candidates ranked directly

struct FastSamplerSmem {
  unsigned long long cand[FAST_CAP];
  unsigned long long top[FAST_NW * FAST_TOP];
  unsigned long long sorted[SAMPLER_KSMALL];
  alignas(16) float w[SAMPLER_KSMALL];    // (read as float4 by the running sums)
  alignas(16) float run[SAMPLER_KSMALL];
  uint32_t keys[SAMPLER_VMAX];  // the fallback selection's copy of the value keys
  int wc[2][FAST_NW];
  int wscan[FAST_NW];
  unsigned long long theta;
  int n_cand, n_gt, pick;
};

__device__ __forceinline__ float key_value(unsigned long long k) {
  const uint32_t f = (uint32_t)(k >> 32);
  const uint32_t bits = (f & 0x80000000u) ? (f & 0x7fffffffu) : ~f;
  return __uint_as_float(bits);
}

__device__ __forceinline__ int key_index(unsigned long long k) {
  return (int)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
}

// Group-wide sum of one int per thread; `slot` alternates between calls so a
// single barrier suffices.
template <class G>
__device__ __forceinline__ int group_count(FastSamplerSmem& sm, int v, int slot) {
  const int lane = G::tid() & 31, warp = G::tid() >> 5;
  v = __reduce_add_sync(0xffffffffu, v);
  if (lane == 0) sm.wc[slot][warp] = v;
  G::sync();
  int tot = 0;
  for (int w = 0; w < FAST_NW; ++w) tot += sm.wc[slot][w];
  return tot;
}

// Fallback selection from the value keys in sm.keys[0..V): the K-th largest
// key t by bisection over its 32 bits (one group count per bit); keys above t
// and the lowest-index ties at t fill sm.cand[0..K), which are then ranked
// into sm.sorted.  Loops stay rolled: this path is rare and kept small.
template <class G>
__device__ __noinline__ void fast_select_bisect(FastSamplerSmem& sm, int V, int K) {
  const int tid = G::tid(), lane = tid & 31, warp = tid >> 5;
  const int per = (V + FAST_NT - 1) / FAST_NT, i0 = tid * per, i1 = min(V, i0 + per);
  uint32_t t = 0u;
  for (int b = 31; b >= 0; --b) {
    const uint32_t c = t | (1u << b);
    int cnt = 0;
    for (int i = i0; i < i1; ++i) cnt += sm.keys[i] >= c ? 1 : 0;
    if (group_count<G>(sm, cnt, b & 1) >= K) t = c;
  }
  int n_gt = 0, n_eq = 0;
  for (int i = i0; i < i1; ++i) {
    n_gt += sm.keys[i] > t ? 1 : 0;
    n_eq += sm.keys[i] == t ? 1 : 0;
  }
  // ties before this thread's (lower indices): warp scan + warp totals
  int incl = n_eq;
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) sm.wscan[warp] = incl;
  if (tid == 0) sm.n_gt = 0;
  const int above = group_count<G>(sm, n_gt, 1);  // keys above t (fewer than K)
  int before = incl - n_eq;
  for (int w = 0; w < warp; ++w) before += sm.wscan[w];
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = sm.keys[i];
    const unsigned long long k = ((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)i);
    if (key > t) {
      sm.cand[atomicAdd(&sm.n_gt, 1)] = k;
    } else if (key == t) {
      if (above + before < K) sm.cand[above + before] = k;
      ++before;
    }
  }
  G::sync();
  if (tid < K) {
    const unsigned long long my = sm.cand[tid];
    int rank = 0;
    for (int j = 0; j < K; ++j) rank += sm.cand[j] > my ? 1 : 0;
    sm.sorted[rank] = my;
  }
}

// The draw of the frame kernel: greedy, or sampling with 1 <= top_k <= 64,
// run by a group of 256 threads (8 warps) on V <= SAMPLER_VMAX logits (V a
// multiple of 4, logits 16-byte and history 4-byte aligned; the logits may
// be sm.keys itself -- they are read before their keys replace them, or any
// memory the group can read with plain loads): thread t reads
// float4 q of the logits at elements 4 (t + 256 q) (a warp's loads are
// contiguous) and keeps their 32-bit value keys in shared memory; candidates
// are 64-bit keys (value key, inverted index).  Greedy is the same rule with k = 1 and T = 1 (dividing by 1 is
// exact): the largest penalised logit, lowest index on ties.  The k largest
// keys are found without a serial search in the common case:
//   1. a lower bound theta on the k-th largest key: every lane's largest key,
//      sorted per warp; the k-th largest of the warps' 8 largest lane maxima
//      (a subset of the keys, so at least k keys are >= theta);
//   2. the keys >= theta are gathered (typically little more than k) and
//      ranked by counting, which places the k largest in order.
// If more than FAST_CAP keys pass the bound (many equal logits), the k-th
// largest key is found by bisection instead (fast_select_bisect).  The draw is
// the float rule of group_sample on the ordered candidates.
template <class G>
__device__ __noinline__ int fast_sample(FastSamplerSmem& sm, const float* logits, int V, int do_sample,
                                        int top_k, float top_p, float temperature, float rep,
                                        const uint8_t* history, float u) {
  const int tid = G::tid(), lane = tid & 31, warp = tid >> 5;
  const int K = !do_sample ? 1 : ((top_k <= 0 || top_k >= V) ? V : top_k);  // caller: K <= SAMPLER_KSMALL
  const float T = do_sample ? temperature : 1.0f;
  const float P = do_sample ? top_p : 1.0f;
  const bool pen = history != nullptr && rep != 1.0f;
  // value keys of the thread's logits (float4 q: elements 4 (tid + FAST_NT q)
  // .. + 3) into sm.keys, the lane's largest (key, index) kept: rolled loops,
  // so the float divisions of the rule appear once in the code (unrolling the
  // inner loop measured slower)
  unsigned long long lm = 0ull;
#pragma unroll 1
  for (int q = 0; q < FAST_V4; ++q) {
    const int e = 4 * (tid + FAST_NT * q);
    if (e >= V) break;
    float4 v = *reinterpret_cast<const float4*>(logits + e);
    uint32_t hb = pen ? *reinterpret_cast<const uint32_t*>(history + e) : 0u;
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
      float l = v.x;
      if (hb & 0xffu) l = l > 0.0f ? __fdiv_rn(l, rep) : __fmul_rn(l, rep);
      const uint32_t kv = fkey(__fdiv_rn(l, T));
      sm.keys[e + k] = kv;
      const unsigned long long kk = ((unsigned long long)kv << 32) | (0xffffffffu - (uint32_t)(e + k));
      lm = kk > lm ? kk : lm;
      v = make_float4(v.y, v.z, v.w, 0.f);
      hb >>= 8;
    }
  }
  // 1) theta: the lanes' largest keys sorted descending across the warp
  //    (bitonic network); lanes 0..7 post the warp's 8 largest
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, lm, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      lm = keep_max ? (o > lm ? o : lm) : (o < lm ? o : lm);
    }
  }
  if (lane < FAST_TOP) sm.top[warp * FAST_TOP + lane] = lm;
  if (tid == 0) {
    sm.theta = 0ull;  // fewer than K real keys posted: every real key is a candidate
    sm.n_cand = 0;
  }
  G::sync();
  if (warp == 0) {
    // the K-th largest posted key (posted real keys are distinct; zeros are padding)
    for (int h = 0; h < FAST_NW * FAST_TOP / 32; ++h) {
      const unsigned long long my = sm.top[lane + 32 * h];
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < FAST_NW * FAST_TOP; ++j) rank += sm.top[j] > my ? 1 : 0;
      if (my != 0ull && rank == K - 1) sm.theta = my;
    }
  }
  G::sync();
  // 2) gather the keys >= theta (a thread reads back its own keys)
  const unsigned long long theta = sm.theta;
#pragma unroll 1
  for (int q = 0; q < FAST_V4; ++q) {
    const int e = 4 * (tid + FAST_NT * q);
    if (e >= V) break;
    const uint4 kv = *reinterpret_cast<const uint4*>(&sm.keys[e]);
    const uint32_t ks[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const unsigned long long kk = ((unsigned long long)ks[k] << 32) | (0xffffffffu - (uint32_t)(e + k));
      if (kk >= theta) {
        const int slot = atomicAdd(&sm.n_cand, 1);
        if (slot < FAST_CAP) sm.cand[slot] = kk;
      }
    }
  }
  G::sync();
  const int C = sm.n_cand;
  if (C > FAST_CAP) {
    fast_select_bisect<G>(sm, V, K);  // sm.keys holds every key
  } else if (tid < C) {
    const unsigned long long my = sm.cand[tid];
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < C; ++j) rank += sm.cand[j] > my ? 1 : 0;
    if (rank < K) sm.sorted[rank] = my;
  }
  G::sync();
  if (tid < K) sm.w[tid] = exp_cw(__fsub_rn(key_value(sm.sorted[tid]), key_value(sm.sorted[0])));
  G::sync();
  if (warp == 0) {
    // running sums in order (one thread: the float rule's summation order);
    // the weights are read in blocks of four ahead of the dependent adds
    if (lane == 0) {
      float run = 0.0f;
      int i = 0;
#pragma unroll 1
      for (; i + 4 <= K; i += 4) {
        const float4 wv = *reinterpret_cast<const float4*>(&sm.w[i]);
        float4 rv;
        rv.x = run = __fadd_rn(run, wv.x);
        rv.y = run = __fadd_rn(run, wv.y);
        rv.z = run = __fadd_rn(run, wv.z);
        rv.w = run = __fadd_rn(run, wv.w);
        *reinterpret_cast<float4*>(&sm.run[i]) = rv;
      }
      for (; i < K; ++i) {
        run = __fadd_rn(run, sm.w[i]);
        sm.run[i] = run;
      }
    }
    __syncwarp();
    const float r0 = lane < K ? sm.run[lane] : 0.f, r1 = lane + 32 < K ? sm.run[lane + 32] : 0.f;
    int kept = K;
    if (P < 1.0f) {
      // the first i with run_i >= top_p * z (z = run_{K-1}) closes the nucleus
      const float tp = __fmul_rn(P, sm.run[K - 1]);
      const unsigned b0 = __ballot_sync(0xffffffffu, lane < K && r0 >= tp);
      const unsigned b1 = __ballot_sync(0xffffffffu, lane + 32 < K && r1 >= tp);
      kept = b0 ? __ffs(b0) : (b1 ? 32 + __ffs(b1) : K);
    }
    // the first i < kept with run_i > u * run_{kept-1}, else the last kept
    const float th = __fmul_rn(u, sm.run[kept - 1]);
    const unsigned c0 = __ballot_sync(0xffffffffu, lane < kept && r0 > th);
    const unsigned c1 = __ballot_sync(0xffffffffu, lane + 32 < kept && r1 > th);
    const int selk = c0 ? __ffs(c0) - 1 : (c1 ? 31 + __ffs(c1) : kept - 1);
    if (lane == 0) sm.pick = key_index(sm.sorted[selk]);
  }
  G::sync();
  const int pick = sm.pick;
  G::sync();
  return pick;
}

}  // namespace q3
