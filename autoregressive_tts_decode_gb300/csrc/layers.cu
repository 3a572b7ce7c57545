// layers.cu -- one-kernel-per-operation decoder building blocks (see layers.cuh).
#include <stdlib.h>

#include "layers.cuh"

namespace q3 {

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("Q3TTS_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

// ---------------------------------------------------------------- linear
// Skinny case (few tokens): one warp per output row, eight weights per lane per
// step with 16-byte streaming loads; the row is multiplied with up to MT token
// vectors at once.
template <class WT, int MT>
__global__ void __launch_bounds__(256) gemv_kernel(const float* __restrict__ X, int ldx,
                                                   const WT* __restrict__ W, int N, int K,
                                                   float* __restrict__ Y, int ldy, int M,
                                                   int accumulate, const float* __restrict__ sc) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int n = warp; n < N; n += nwarps) {
    const WT* wr = W + (size_t)n * K;
    for (int m0 = 0; m0 < M; m0 += MT) {
      float acc[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t] = 0.f;
      for (int k = lane * 8; k < K; k += 256) {
        float w[8];
        load_w8(wr + k, w);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          if (m0 + t < M) {
            float x[8];
            load_f8(X + (size_t)(m0 + t) * ldx + k, x);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[t] = fmaf(w[i], x[i], acc[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        float v = warp_sum(acc[t]);
        if (sc) v *= sc[n];  // FP8 rows: the row scale
        if (lane == 0 && m0 + t < M) {
          float* y = Y + (size_t)(m0 + t) * ldy + n;
          *y = accumulate ? *y + v : v;
        }
      }
    }
  }
}

// Many tokens: 64x64 output tiles, K in steps of 16, 4x4 outputs per thread.
template <class WT>
__global__ void __launch_bounds__(256) gemm_kernel(const float* __restrict__ X, int ldx,
                                                   const WT* __restrict__ W, int N, int K,
                                                   float* __restrict__ Y, int ldy, int M,
                                                   int accumulate, const float* __restrict__ sc) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int e = tid; e < 64 * 16; e += 256) {
      int r = e / 16, c = e % 16;
      int gm = m0 + r, gn = n0 + r, gk = k0 + c;
      As[c][r] = (gm < M && gk < K) ? X[(size_t)gm * ldx + gk] : 0.f;
      Bs[c][r] = (gn < N && gk < K) ? to_f(W[(size_t)gn * K + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[kk][tm + i]; b[i] = Bs[kk][tn + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int gm = m0 + tm + i, gn = n0 + tn + j;
      if (gm < M && gn < N) {
        float* y = Y + (size_t)gm * ldy + gn;
        const float v = sc ? acc[i][j] * sc[gn] : acc[i][j];  // FP8 rows: the row scale
        *y = accumulate ? *y + v : v;
      }
    }
}

template <class WT>
static void linear_t(const float* X, int ldx, const WT* W, int N, int K, float* Y, int ldy, int M,
                     bool acc, const float* sc, cudaStream_t s) {
  if (M <= 0 || N <= 0) return;
  if (M <= 16) {
    int blocks = (N + 7) / 8;
    if (blocks > 4096) blocks = 4096;
    if (M <= 1)
      launch_pdl(gemv_kernel<WT, 1>, dim3(blocks), dim3(256), 0, s, X, ldx, W, N, K, Y, ldy, M, acc, sc);
    else if (M <= 2)
      launch_pdl(gemv_kernel<WT, 2>, dim3(blocks), dim3(256), 0, s, X, ldx, W, N, K, Y, ldy, M, acc, sc);
    else if (M <= 4)
      launch_pdl(gemv_kernel<WT, 4>, dim3(blocks), dim3(256), 0, s, X, ldx, W, N, K, Y, ldy, M, acc, sc);
    else
      launch_pdl(gemv_kernel<WT, 8>, dim3(blocks), dim3(256), 0, s, X, ldx, W, N, K, Y, ldy, M, acc, sc);
  } else {
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    launch_pdl(gemm_kernel<WT>, dim3(grid), dim3(256), 0, s, X, ldx, W, N, K, Y, ldy, M, acc, sc);
  }
}

void launch_linear(int wdt, const float* X, int ldx, const void* W, int N, int K, float* Y, int ldy,
                   int M, bool accumulate, cudaStream_t s, const float* scale) {
  if (wdt == Q3TTS_FP8)
    linear_t(X, ldx, (const fp8e4*)W, N, K, Y, ldy, M, accumulate, scale, s);
  else if (wdt == Q3TTS_BF16)
    linear_t(X, ldx, (const bf16*)W, N, K, Y, ldy, M, accumulate, nullptr, s);
  else
    linear_t(X, ldx, (const float*)W, N, K, Y, ldy, M, accumulate, nullptr, s);
}

// --------------------------------------------------------------- rmsnorm
template <class WT>
__global__ void rmsnorm_kernel(const float* __restrict__ X, int ldx, int in_mul, int in_add,
                               const WT* __restrict__ g, float* __restrict__ Y, int ldy, int D,
                               float eps) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  __shared__ float red[32];
  const int m = blockIdx.x;
  const float* x = X + (size_t)(m * in_mul + in_add) * ldx;
  float ss = 0.f;
  for (int i = threadIdx.x; i < D; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)D + eps);
  for (int i = threadIdx.x; i < D; i += blockDim.x) Y[(size_t)m * ldy + i] = x[i] * inv * to_f(g[i]);
}

__device__ __forceinline__ void store_hilo(bf16* hi, bf16* lo, size_t i, float v) {
  const bf16 h = __float2bfloat16_rn(v);
  hi[i] = h;
  lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
}

template <class WT>
__global__ void rmsnorm_hilo_kernel(const float* __restrict__ X, int ldx, int in_mul, int in_add,
                                    const WT* __restrict__ g, bf16* __restrict__ hi, bf16* __restrict__ lo,
                                    int D, float eps) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  __shared__ float red[32];
  const int m = blockIdx.x;
  const float* x = X + (size_t)(m * in_mul + in_add) * ldx;
  float ss = 0.f;
  for (int i = threadIdx.x; i < D; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)D + eps);
  for (int i = threadIdx.x; i < D; i += blockDim.x) store_hilo(hi, lo, (size_t)m * D + i, x[i] * inv * to_f(g[i]));
}

void launch_rmsnorm_hilo(int wdt, const float* X, int ldx, int in_mul, int in_add, const void* g, const HiLo& y,
                         int M, int D, float eps, cudaStream_t s) {
  if (M <= 0) return;
  if (wdt == Q3TTS_BF16)
    launch_pdl(rmsnorm_hilo_kernel<bf16>, dim3(M), dim3(256), 0, s, X, ldx, in_mul, in_add, (const bf16*)g, y.hi, y.lo, D, eps);
  else
    launch_pdl(rmsnorm_hilo_kernel<float>, dim3(M), dim3(256), 0, s, X, ldx, in_mul, in_add, (const float*)g, y.hi, y.lo, D, eps);
}

void launch_rmsnorm(int wdt, const float* X, int ldx, int in_mul, int in_add, const void* g,
                    float* Y, int ldy, int M, int D, float eps, cudaStream_t s) {
  if (M <= 0) return;
  if (wdt == Q3TTS_BF16)
    launch_pdl(rmsnorm_kernel<bf16>, dim3(M), dim3(256), 0, s, X, ldx, in_mul, in_add, (const bf16*)g, Y, ldy, D, eps);
  else
    launch_pdl(rmsnorm_kernel<float>, dim3(M), dim3(256), 0, s, X, ldx, in_mul, in_add, (const float*)g, Y, ldy, D, eps);
}

// ------------------------------------------------ q/k norm + RoPE + append
// One block per token, one warp per head; lane l holds elements l + 32 j, so
// the rotate-half partners i and i + hd/2 sit in the same lane.
template <class WT, class KT, int HD>
__global__ void qk_rope_append_kernel(float* __restrict__ qkv, int ld, TokDesc td,
                                      const WT* __restrict__ gq, const WT* __restrict__ gk,
                                      int qk_norm, float eps, const float* __restrict__ rc,
                                      const float* __restrict__ rs, KVDesc kv, int layer, int Hq) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  constexpr int J = HD / 32, P = J / 2, HALF = HD / 2;
  const int m = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const int stream = td.tok_stream[m];
  const int pos = td.tok_pos ? td.tok_pos[m] : td.pos_const;
  const int Hkv = kv.Hkv;
  float* row = qkv + (size_t)m * ld;
  for (int hh = warp; hh < Hq + 2 * Hkv; hh += nw) {
    float v[J];
    float* src = row + (size_t)hh * HD;
#pragma unroll
    for (int j = 0; j < J; ++j) v[j] = src[lane + 32 * j];
    const bool is_q = hh < Hq, is_k = !is_q && hh < Hq + Hkv;
    if (is_q || is_k) {
      const WT* g = is_q ? gq : gk;
      if (qk_norm) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < J; ++j) ss = fmaf(v[j], v[j], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)HD + eps);
#pragma unroll
        for (int j = 0; j < J; ++j) v[j] = v[j] * inv * to_f(g[lane + 32 * j]);
      }
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const int i = lane + 32 * j;
        const float c = rc[(size_t)pos * HALF + i], sn = rs[(size_t)pos * HALF + i];
        const float x0 = v[j], x1 = v[j + P];
        v[j] = x0 * c - x1 * sn;
        v[j + P] = x1 * c + x0 * sn;
      }
    }
    if (is_q) {
#pragma unroll
      for (int j = 0; j < J; ++j) src[lane + 32 * j] = v[j];
    } else {
      const int head = is_k ? hh - Hq : hh - Hq - Hkv;
      KT* dst = (KT*)kv.pool + kv_offset(kv, layer, stream, pos, is_k ? 0 : 1, head);
#pragma unroll
      for (int j = 0; j < J; ++j) dst[lane + 32 * j] = from_f<KT>(v[j]);
    }
  }
}

template <class WT, class KT>
static void qk_rope_t(float* qkv, int ld, int M, TokDesc td, const void* gq, const void* gk,
                      int qk_norm, float eps, const float* rc, const float* rs, KVDesc kv, int layer,
                      int Hq, cudaStream_t s) {
  if (kv.hd == 128)
    launch_pdl(qk_rope_append_kernel<WT, KT, 128>, dim3(M), dim3(256), 0, s, qkv, ld, td, (const WT*)gq, (const WT*)gk,
                                                         qk_norm, eps, rc, rs, kv, layer, Hq);
  else
    launch_pdl(qk_rope_append_kernel<WT, KT, 64>, dim3(M), dim3(256), 0, s, qkv, ld, td, (const WT*)gq, (const WT*)gk,
                                                        qk_norm, eps, rc, rs, kv, layer, Hq);
}

void launch_qk_rope_append(int wdt, int kdt, float* qkv, int ld, int M, TokDesc td, const void* gq,
                           const void* gk, int qk_norm, float eps, const float* rc,
                           const float* rs, KVDesc kv, int layer, int Hq, cudaStream_t s) {
  if (M <= 0) return;
  if (wdt == Q3TTS_BF16) {
    if (kdt == Q3TTS_BF16)
      qk_rope_t<bf16, bf16>(qkv, ld, M, td, gq, gk, qk_norm, eps, rc, rs, kv, layer, Hq, s);
    else
      qk_rope_t<bf16, float>(qkv, ld, M, td, gq, gk, qk_norm, eps, rc, rs, kv, layer, Hq, s);
  } else {
    if (kdt == Q3TTS_BF16)
      qk_rope_t<float, bf16>(qkv, ld, M, td, gq, gk, qk_norm, eps, rc, rs, kv, layer, Hq, s);
    else
      qk_rope_t<float, float>(qkv, ld, M, td, gq, gk, qk_norm, eps, rc, rs, kv, layer, Hq, s);
  }
}

// -------------------------------------------------------------- attention
// One block per (token, q head): scores over positions 0..pos into shared
// memory, max-subtracted softmax, then the weighted sum of v.
template <class KT>
__global__ void __launch_bounds__(128) attention_kernel(const float* __restrict__ qkv, int ld,
                                                        TokDesc td, KVDesc kv, int layer, int Hq,
                                                        float* __restrict__ out, int ldo) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  extern __shared__ float sm[];
  __shared__ float red[32];
  const int m = blockIdx.x, h = blockIdx.y, hd = kv.hd;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int stream = td.tok_stream[m];
  const int pos = td.tok_pos ? td.tok_pos[m] : td.pos_const;
  const int S = pos + 1, g = h / (Hq / kv.Hkv);
  float* q = sm;
  float* sc = sm + hd;
  for (int i = threadIdx.x; i < hd; i += blockDim.x) q[i] = qkv[(size_t)m * ld + h * hd + i];
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)hd);
  for (int t = warp; t < S; t += nw) {
    const KT* k = (const KT*)kv.pool + kv_offset(kv, layer, stream, t, 0, g);
    float d = 0.f;
    for (int i = lane; i < hd; i += 32) d = fmaf(q[i], to_f(k[i]), d);
    d = warp_sum(d);
    if (lane == 0) sc[t] = d * scale;
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int t = threadIdx.x; t < S; t += blockDim.x) mx = fmaxf(mx, sc[t]);
  mx = block_max(mx, red);
  float z = 0.f;
  for (int t = threadIdx.x; t < S; t += blockDim.x) {
    float e = __expf(sc[t] - mx);
    sc[t] = e;
    z += e;
  }
  z = block_sum(z, red);
  __syncthreads();
  for (int i = threadIdx.x; i < hd; i += blockDim.x) {
    float acc = 0.f;
    for (int t = 0; t < S; ++t) {
      const KT* v = (const KT*)kv.pool + kv_offset(kv, layer, stream, t, 1, g);
      acc = fmaf(sc[t], to_f(v[i]), acc);
    }
    out[(size_t)m * ldo + h * hd + i] = acc / z;
  }
}

// Single-query attention, one CTA per (token, kv head), for launches with many
// CTAs (many tokens): the q heads of the group share every K/V read.  Four
// warps take interleaved positions with an online softmax each (lane l holds
// elements l + 32 j of a head vector), and combine through shared memory.  The
// stream's page-table row is staged in shared memory once.  hd <= 128, at
// most 4 q heads per kv head.  Few registers, so many CTAs share an SM.
template <class KT>
__global__ void __launch_bounds__(128) attention_gqa4_kernel(const float* __restrict__ qkv, int ld, TokDesc td,
                                                            KVDesc kv, int layer, int Hq,
                                                            float* __restrict__ out, int ldo) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  constexpr int NW = 4, RMAX = 4;
  extern __shared__ int pt[];  // the stream's page-table row
  __shared__ float qs[RMAX][128];
  __shared__ float wm[NW][RMAX], wl[NW][RMAX], wo[NW][RMAX][128];
  const int m = blockIdx.x, g = blockIdx.y, hd = kv.hd, rep = Hq / kv.Hkv, J = hd / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int stream = td.tok_stream[m];
  const int pos = td.tok_pos ? td.tok_pos[m] : td.pos_const;
  const int S = pos + 1, npg = (S + kv.page_size - 1) / kv.page_size;
  for (int i = threadIdx.x; i < npg; i += blockDim.x) pt[i] = kv.page_table[stream * kv.pages_per_stream + i];
  for (int e = threadIdx.x; e < rep * hd; e += blockDim.x) {
    const int r = e / hd, i = e % hd;
    qs[r][i] = qkv[(size_t)m * ld + (g * rep + r) * hd + i];
  }
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)hd);
  const size_t head_stride = (size_t)kv.page_size * hd;
  float mx[RMAX], l[RMAX], o[RMAX][4];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    mx[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) o[r][j] = 0.f;
  }
  for (int t = warp; t < S; t += NW) {
    const int page = pt[t / kv.page_size];
    const size_t base = ((((size_t)layer * kv.n_pages + page) * 2) * kv.Hkv + g) * head_stride +
                        (size_t)(t % kv.page_size) * hd;
    const KT* kp = (const KT*)kv.pool + base;
    const KT* vp = kp + (size_t)kv.Hkv * head_stride;  // the V plane of the same page
    float k[4], v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      k[j] = j < J ? to_f(kp[lane + 32 * j]) : 0.f;
      v[j] = j < J ? to_f(vp[lane + 32 * j]) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < rep) {
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < J) d = fmaf(qs[r][lane + 32 * j], k[j], d);
        d = warp_sum(d) * scale;
        const float mn = fmaxf(mx[r], d), corr = __expf(mx[r] - mn), e = __expf(d - mn);
        l[r] = l[r] * corr + e;
#pragma unroll
        for (int j = 0; j < 4; ++j) o[r][j] = o[r][j] * corr + e * v[j];
        mx[r] = mn;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r < rep) {
      if (lane == 0) {
        wm[warp][r] = mx[r];
        wl[warp][r] = l[r];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < J) wo[warp][r][lane + 32 * j] = o[r][j];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < rep * hd; e += blockDim.x) {
    const int r = e / hd, i = e % hd;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w][r]);
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = wm[w][r] == -INFINITY ? 0.f : __expf(wm[w][r] - M);
      Ls += wl[w][r] * f;
      Os += wo[w][r][i] * f;
    }
    out[(size_t)m * ldo + (g * rep + r) * hd + i] = Os / Ls;
  }
}

// Single-query attention, one CTA per (token, kv head), for launches with few
// CTAs (few tokens): the q heads of the group share every K/V read.  Eight
// warps take runs of GQA_B consecutive positions (warp w: w B .. w B + B - 1,
// then + 8 B), issuing the K/V loads of a run together before the
// online-softmax updates; lane l holds the E = hd / 32 contiguous elements
// l E .. l E + E - 1 of a head vector (one vector load per row).  The warps
// combine through shared memory; the stream's page-table row is staged in
// shared memory once.  hd = 64 or 128, at most 4 q heads per kv head.
constexpr int GQA_NW = 8, GQA_B = 4, GQA_RMAX = 4;

template <class KT, int E>
__device__ __forceinline__ void load_row(const KT* p, float (&f)[4]);
template <>
__device__ __forceinline__ void load_row<float, 4>(const float* p, float (&f)[4]) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
template <>
__device__ __forceinline__ void load_row<float, 2>(const float* p, float (&f)[4]) {
  const float2 v = __ldcg(reinterpret_cast<const float2*>(p));
  f[0] = v.x; f[1] = v.y; f[2] = 0.f; f[3] = 0.f;
}
template <>
__device__ __forceinline__ void load_row<bf16, 4>(const bf16* p, float (&f)[4]) {
  const uint2 v = __ldcg(reinterpret_cast<const uint2*>(p));
  f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
}
template <>
__device__ __forceinline__ void load_row<bf16, 2>(const bf16* p, float (&f)[4]) {
  const uint32_t v = __ldcg(reinterpret_cast<const unsigned int*>(p));
  f[0] = __uint_as_float(v << 16); f[1] = __uint_as_float(v & 0xffff0000u); f[2] = 0.f; f[3] = 0.f;
}

template <class KT, int E>
__global__ void __launch_bounds__(GQA_NW * 32) attention_gqa8_kernel(const float* __restrict__ qkv, int ld,
                                                                    TokDesc td, KVDesc kv, int layer, int Hq,
                                                                    float* __restrict__ out, int ldo) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  constexpr int NW = GQA_NW, B = GQA_B, RMAX = GQA_RMAX;
  extern __shared__ int pt[];  // the stream's page-table row
  __shared__ float wm[NW][RMAX], wl[NW][RMAX];
  __shared__ __align__(16) float wo[NW][RMAX][128];
  const int m = blockIdx.x, g = blockIdx.y, hd = E * 32, rep = Hq / kv.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int stream = td.tok_stream[m];
  const int pos = td.tok_pos ? td.tok_pos[m] : td.pos_const;
  const int S = pos + 1, npg = (S + kv.page_size - 1) / kv.page_size;
  for (int i = threadIdx.x; i < npg; i += blockDim.x) pt[i] = kv.page_table[stream * kv.pages_per_stream + i];
  float q[RMAX][4];
#pragma unroll
  for (int r = 0; r < RMAX; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      q[r][e] = (r < rep && e < E) ? qkv[(size_t)m * ld + (g * rep + r) * hd + lane * E + e] : 0.f;
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)hd);
  const size_t head_stride = (size_t)kv.page_size * hd;
  float mx[RMAX], l[RMAX], o[RMAX][4];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    mx[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[r][e] = 0.f;
  }
  for (int t0 = warp * B; t0 < S; t0 += NW * B) {
    float k[B][4], v[B][4];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int t = t0 + b;
      if (t < S) {
        const int page = pt[t / kv.page_size];
        const size_t base = ((((size_t)layer * kv.n_pages + page) * 2) * kv.Hkv + g) * head_stride +
                            (size_t)(t % kv.page_size) * hd + lane * E;
        const KT* kp = (const KT*)kv.pool + base;
        load_row<KT, E>(kp, k[b]);
        load_row<KT, E>(kp + (size_t)kv.Hkv * head_stride, v[b]);  // the V plane of the same page
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (t0 + b < S) {
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          if (r < rep) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) d = fmaf(q[r][e], k[b][e], d);
            d = warp_sum(d) * scale;
            const float mn = fmaxf(mx[r], d), corr = __expf(mx[r] - mn), ex = __expf(d - mn);
            l[r] = l[r] * corr + ex;
#pragma unroll
            for (int e = 0; e < E; ++e) o[r][e] = o[r][e] * corr + ex * v[b][e];
            mx[r] = mn;
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r < rep) {
      if (lane == 0) {
        wm[warp][r] = mx[r];
        wl[warp][r] = l[r];
      }
#pragma unroll
      for (int e = 0; e < E; ++e) wo[warp][r][lane * E + e] = o[r][e];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < rep * hd; e += blockDim.x) {
    const int r = e / hd, i = e % hd;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w][r]);
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = wm[w][r] == -INFINITY ? 0.f : __expf(wm[w][r] - M);
      Ls += wl[w][r] * f;
      Os += wo[w][r][i] * f;
    }
    out[(size_t)m * ldo + (g * rep + r) * hd + i] = Os / Ls;
  }
}

// ------------------------------------------ split-context paged attention
//
// Single-query attention for many tokens with long contexts (serving streams,
// prefill chunks).  All (token, kv head) pairs' cache pages, 16 positions
// each, form one list -- token by token, kv head by kv head -- and every warp
// of a fixed grid (one wave; the grid does not depend on the contexts, so a
// captured graph replays it unchanged) takes an equal run of consecutive
// pages (at least SPL_MINP), so all warps finish together.  A warp's run
// covers one or more segments (the pages of one (token, kv head)); per
// segment it keeps an online softmax in registers and then writes the output
// (when the run holds the whole segment) or (max, sum, unnormalised output) to
// part[], where the last of the segment's runs to finish (a counter per
// (token, kv head)) merges them and resets the counter.
//
// Per page the warp loads its K and V rows straight into registers -- lanes 2p
// and 2p + 1 take position p, the even and the odd 16-byte pieces of its row
// (each load instruction reads whole 32-byte sectors), and lane l takes
// elements l hd/32 .. of every V row -- so a whole page is in flight, with no
// shared-memory staging and no block barrier.  Scores use the group's q
// vectors from the warp's shared slot (the same address for the 16 lanes of a
// parity: a broadcast).
constexpr int SPL_PAGE = 16;   // positions of a cache page this kernel takes
constexpr int SPL_MINP = 2;    // fewest pages of a warp's run
constexpr int SPL_RMAX = 4;    // q heads per kv head
constexpr int SPL_WARPS = 4;   // warps of a CTA

struct SplitArgs {
  const float* qkv;
  int ld, M;
  TokDesc td;
  KVDesc kv;
  int layer, Hq;
  float* out;
  int ldo;
  float* part;      // [M][Hq][nsmax][hd + 2]
  int* cnt;         // [M][Hkv], zero between launches
  int nsmax;        // runs per (token, kv head) the part buffer holds
};

// The token whose segments hold list entry idx, from the exclusive prefix
// pfx[0..M] of the tokens' page counts x Hkv.
__device__ __forceinline__ int split_token(const int* pfx, int M, int idx) {
  int lo = 0, hi = M - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pfx[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <class KT, int HD, int REP>
__global__ void __launch_bounds__(SPL_WARPS * 32) attention_split_kernel(SplitArgs a) {
  pdl_wait();  // inputs come from the previous kernel (the next one is let in at the end)
  constexpr int NCH = HD * (int)sizeof(KT) / 32;   // 16-byte loads per lane: its half of a row
  constexpr int EPC = 16 / (int)sizeof(KT);        // elements per load
  constexpr int OPL = HD / 32;                     // output elements per lane
  constexpr int VW = OPL * (int)sizeof(KT);        // bytes of a lane's slice of a V row
  extern __shared__ __align__(16) uint8_t spl_smem[];
  float* qsm = reinterpret_cast<float*>(spl_smem);  // [warps][REP][HD]
  int* pfx = reinterpret_cast<int*>(qsm + SPL_WARPS * REP * HD);  // [M + 1] page-list prefix
  int* tpos = pfx + a.M + 1;                                     // [M] token positions
  int* tstr = tpos + a.M;                                        // [M] token streams
  const KVDesc& kv = a.kv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int Hkv = kv.Hkv;
  const float scale = 1.0f / sqrtf((float)HD);
  const size_t head_stride = (size_t)SPL_PAGE * HD;
  // page counts x Hkv per token (all threads), then their exclusive prefix
  // (warp 0: lane i sums a run of consecutive tokens, a shuffle scan adds the runs)
  for (int m = threadIdx.x; m < a.M; m += blockDim.x) {
    const int pos = a.td.tok_pos ? a.td.tok_pos[m] : a.td.pos_const;
    tpos[m] = pos;
    tstr[m] = a.td.tok_stream[m];
    pfx[m + 1] = (pos / SPL_PAGE + 1) * Hkv;
  }
  __syncthreads();
  if (warp == 0) {
    const int run = (a.M + 31) / 32, m0 = lane * run, m1 = min(a.M, m0 + run);
    int sum = 0;
    for (int m = m0; m < m1; ++m) sum += pfx[m + 1];
    int inc = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += v;
    }
    __syncwarp();
    int acc = inc - sum;  // pages of the tokens before this run
    for (int m = m0; m < m1; ++m) {
      const int n = pfx[m + 1];
      pfx[m + 1] = acc + n;
      acc += n;
    }
    if (lane == 0) pfx[0] = 0;
  }
  __syncthreads();
  const int total = pfx[a.M];
  const int nwarps = gridDim.x * SPL_WARPS, wid = blockIdx.x * SPL_WARPS + warp;
  const int ppw = max(SPL_MINP, (total + nwarps - 1) / nwarps);
  const int lo = wid * ppw, hi = min(total, lo + ppw);
  float* qw = qsm + warp * REP * HD;
  const int p = lane >> 1, half = lane & 1;  // position, parity of the row's 16-byte pieces
  for (int idx = lo; idx < hi;) {
    // the segment (m, g) holding idx, and this run's pages j0 .. j1 - 1 of it
    const int m = split_token(pfx, a.M, idx);
    const int npg = tpos[m] / SPL_PAGE + 1, S = tpos[m] + 1, stream = tstr[m];
    const int o = idx - pfx[m], g = o / npg, j0 = o % npg;
    const int seg0 = pfx[m] + g * npg, seg1 = seg0 + npg;
    const int j1 = j0 + (min(hi, seg1) - idx);
    idx += j1 - j0;
    // the group's q heads (contiguous in the token's qkv row)
    __syncwarp();
    {
      const float4* qg = reinterpret_cast<const float4*>(a.qkv + (size_t)m * a.ld + (size_t)g * REP * HD);
#pragma unroll
      for (int e = lane; e < REP * HD / 4; e += 32) reinterpret_cast<float4*>(qw)[e] = __ldg(qg + e);
    }
    __syncwarp();
    float M_[REP], L_[REP], ov[REP][OPL];
#pragma unroll
    for (int r = 0; r < REP; ++r) {
      M_[r] = -INFINITY;
      L_[r] = 0.f;
#pragma unroll
      for (int j = 0; j < OPL; ++j) ov[r][j] = 0.f;
    }
    const int* ptab = kv.page_table + (size_t)stream * kv.pages_per_stream;
    for (int jb = j0; jb < j1; jb += 32) {
      // page ids of up to 32 pages (lane k: page jb + k), loaded together
      const int pid = jb + lane < j1 ? ptab[jb + lane] : 0;
      const int jn = min(32, j1 - jb);
      for (int jj = 0; jj < jn; ++jj) {
        const int j = jb + jj;
        const int page = __shfl_sync(0xffffffffu, pid, jj);
        const KT* kb = (const KT*)kv.pool + ((((size_t)a.layer * kv.n_pages + page) * 2) * Hkv + g) * head_stride;
        const uint8_t* kp = reinterpret_cast<const uint8_t*>(kb) + (size_t)p * HD * sizeof(KT) + (size_t)half * 16;
        const uint8_t* vp = reinterpret_cast<const uint8_t*>(kb + (size_t)Hkv * head_stride) + (size_t)lane * VW;
        const int nvalid = min(SPL_PAGE, S - j * SPL_PAGE);
        // the page's loads, all in flight together
        uint4 kr[NCH];
#pragma unroll
        for (int i = 0; i < NCH; ++i) kr[i] = __ldcg(reinterpret_cast<const uint4*>(kp) + 2 * i);
        uint32_t vr[SPL_PAGE][VW / 4];
#pragma unroll
        for (int q = 0; q < SPL_PAGE; ++q) {
          if (q < nvalid) {  // rows past the context are not read (unwritten words may hold NaN)
            if constexpr (VW == 8) {
              const uint2 u = __ldcg(reinterpret_cast<const uint2*>(vp + (size_t)q * HD * sizeof(KT)));
              vr[q][0] = u.x; vr[q][1] = u.y;
            } else if constexpr (VW == 4) {
              vr[q][0] = __ldcg(reinterpret_cast<const unsigned int*>(vp + (size_t)q * HD * sizeof(KT)));
            } else {
              const uint4 u = __ldcg(reinterpret_cast<const uint4*>(vp + (size_t)q * HD * sizeof(KT)));
              vr[q][0] = u.x; vr[q][1] = u.y; vr[q][2] = u.z; vr[q][3] = u.w;
            }
          } else {
#pragma unroll
            for (int e = 0; e < VW / 4; ++e) vr[q][e] = 0u;
          }
        }
        // scores of position p over this lane's half, both halves added
        float d[REP];
#pragma unroll
        for (int r = 0; r < REP; ++r) d[r] = 0.f;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
          float kf[EPC];
          if constexpr (sizeof(KT) == 2) {
            unpack_bf16x8(kr[i], kf);
          } else {
            kf[0] = __uint_as_float(kr[i].x); kf[1] = __uint_as_float(kr[i].y);
            kf[2] = __uint_as_float(kr[i].z); kf[3] = __uint_as_float(kr[i].w);
          }
          const int i0 = (2 * i + half) * EPC;
#pragma unroll
          for (int r = 0; r < REP; ++r) {
#pragma unroll
            for (int e = 0; e < EPC; e += 4) {
              const float4 qv = *reinterpret_cast<const float4*>(qw + r * HD + i0 + e);
              d[r] = fmaf(qv.x, kf[e], d[r]);
              d[r] = fmaf(qv.y, kf[e + 1], d[r]);
              d[r] = fmaf(qv.z, kf[e + 2], d[r]);
              d[r] = fmaf(qv.w, kf[e + 3], d[r]);
            }
          }
        }
        float w[REP];
#pragma unroll
        for (int r = 0; r < REP; ++r) {
          float sc = (d[r] + __shfl_xor_sync(0xffffffffu, d[r], 1)) * scale;
          if (p >= nvalid) sc = -INFINITY;
          float pm = sc;  // over the 16 positions (lanes 2p and 2p + 1 hold the same value)
#pragma unroll
          for (int off = 16; off > 1; off >>= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, off));
          const float Mn = fmaxf(M_[r], pm);  // finite: position 0 of a page exists
          const float corr = __expf(M_[r] - Mn);
          const float ex = sc == -INFINITY ? 0.f : __expf(sc - Mn);
          float ps = ex;
#pragma unroll
          for (int off = 16; off > 1; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
          L_[r] = L_[r] * corr + ps;
          M_[r] = Mn;
#pragma unroll
          for (int q = 0; q < OPL; ++q) ov[r][q] *= corr;
          w[r] = ex;
        }
        // weighted values: lane l owns elements l OPL .. l OPL + OPL - 1
#pragma unroll
        for (int q = 0; q < SPL_PAGE; ++q) {
          float vf[OPL];
          if constexpr (sizeof(KT) == 2) {
#pragma unroll
            for (int e = 0; e < OPL / 2; ++e) {
              vf[2 * e] = __uint_as_float(vr[q][e] << 16);
              vf[2 * e + 1] = __uint_as_float(vr[q][e] & 0xffff0000u);
            }
          } else {
#pragma unroll
            for (int e = 0; e < OPL; ++e) vf[e] = __uint_as_float(vr[q][e]);
          }
#pragma unroll
          for (int r = 0; r < REP; ++r) {
            const float wq = __shfl_sync(0xffffffffu, w[r], 2 * q);
#pragma unroll
            for (int e = 0; e < OPL; ++e) ov[r][e] = fmaf(wq, vf[e], ov[r][e]);
          }
        }
      }
    }
    // runs covering this segment: warps seg0 / ppw .. (seg1 - 1) / ppw
    const int first = seg0 / ppw, nparts = (seg1 - 1) / ppw - first + 1;
    if (nparts == 1) {
#pragma unroll
      for (int r = 0; r < REP; ++r) {
        const float inv = 1.f / L_[r];
        float* dst = a.out + (size_t)m * a.ldo + (g * REP + r) * HD + lane * OPL;
#pragma unroll
        for (int e = 0; e < OPL; ++e) dst[e] = ov[r][e] * inv;
      }
      continue;
    }
    // this run's (max, sum, unnormalised output) per head, in slot wid - first
    float* pb0 = a.part + ((size_t)m * a.Hq + g * REP) * a.nsmax * (HD + 2);
#pragma unroll
    for (int r = 0; r < REP; ++r) {
      float* pr = pb0 + ((size_t)r * a.nsmax + (wid - first)) * (HD + 2);
#pragma unroll
      for (int e = 0; e < OPL; ++e) pr[lane * OPL + e] = ov[r][e];
      if (lane == 0) {
        pr[HD] = M_[r];
        pr[HD + 1] = L_[r];
      }
    }
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(a.cnt + (size_t)m * Hkv + g, 1) == nparts - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    // the last run merges all runs of (m, g): lane s reads run s's max and sum
    // (32 runs per pass), then each lane its OPL outputs
    __threadfence();
#pragma unroll
    for (int r = 0; r < REP; ++r) {
      const float* pr = pb0 + (size_t)r * a.nsmax * (HD + 2);
      float mx = -INFINITY;
      for (int s0 = lane; s0 < nparts; s0 += 32) mx = fmaxf(mx, __ldcg(pr + (size_t)s0 * (HD + 2) + HD));
#pragma unroll
      for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      float ls = 0.f;
      for (int s0 = lane; s0 < nparts; s0 += 32) {
        const float* q = pr + (size_t)s0 * (HD + 2);
        ls += __ldcg(q + HD + 1) * __expf(__ldcg(q + HD) - mx);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
      float acc[OPL];
#pragma unroll
      for (int e = 0; e < OPL; ++e) acc[e] = 0.f;
#pragma unroll 4
      for (int s0 = 0; s0 < nparts; ++s0) {
        const float* q = pr + (size_t)s0 * (HD + 2);
        const float f = __expf(__ldcg(q + HD) - mx);
#pragma unroll
        for (int e = 0; e < OPL; ++e) acc[e] = fmaf(__ldcg(q + lane * OPL + e), f, acc[e]);
      }
      const float inv = 1.f / ls;
      float* dst = a.out + (size_t)m * a.ldo + (g * REP + r) * HD + lane * OPL;
#pragma unroll
      for (int e = 0; e < OPL; ++e) dst[e] = acc[e] * inv;
    }
    if (lane == 0) a.cnt[(size_t)m * Hkv + g] = 0;
  }
  pdl_trigger();
}

template <class KT, int HD, int REP>
static size_t split_smem(int M) {
  return sizeof(float) * SPL_WARPS * REP * HD + sizeof(int) * (3 * (size_t)M + 1);
}

// Runs per (token, kv head) the split kernel's part buffer must hold for
// contexts of up to kv_cap positions: a segment of npg pages meets at most
// npg / SPL_MINP + 2 runs of at least SPL_MINP pages.
int attention_split_spans(int kv_cap) { return (kv_cap + SPL_PAGE - 1) / SPL_PAGE / SPL_MINP + 2; }

template <class KT, int HD, int REP>
static bool launch_split_t(const SplitArgs& a, int n_sm, cudaStream_t s) {
  static int per_sm = 0;  // resident CTAs per SM at the largest shared-memory size
  if (a.M > 1024) return false;
  if (!per_sm) {
    if (cudaFuncSetAttribute(attention_split_kernel<KT, HD, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)split_smem<KT, HD, REP>(1024)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attention_split_kernel<KT, HD, REP>, SPL_WARPS * 32,
                                                      split_smem<KT, HD, REP>(1024)) != cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      per_sm = 0;
      return false;
    }
  }
  // a persistent grid of one wave: every CTA stays resident and walks items
  // a plain launch: the grid is one wave of resident CTAs with fixed page
  // runs, so it must not start beside the previous kernel's CTAs (a CTA that
  // did not fit would run its whole run a wave late)
  attention_split_kernel<KT, HD, REP><<<n_sm * per_sm, SPL_WARPS * 32, split_smem<KT, HD, REP>(a.M), s>>>(a);
  return true;
}

template <class KT, int HD>
static bool launch_split_rep(const SplitArgs& a, int rep, int n_sm, cudaStream_t s) {
  switch (rep) {
    case 1: return launch_split_t<KT, HD, 1>(a, n_sm, s);
    case 2: return launch_split_t<KT, HD, 2>(a, n_sm, s);
    case 4: return launch_split_t<KT, HD, 4>(a, n_sm, s);
    default: return false;
  }
}

bool launch_attention_split(int kdt, const float* qkv, int ld, int M, TokDesc td, KVDesc kv, int layer, int Hq,
                            float* out, int ldo, float* part, int* cnt, int nsmax, cudaStream_t s) {
  if (M <= 0) return true;
  if (kv.page_size != SPL_PAGE || Hq / kv.Hkv > SPL_RMAX || (kv.hd != 64 && kv.hd != 128)) return false;
  static int n_sm = 0;
  if (!n_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n_sm = 1;
  }
  SplitArgs a{qkv, ld, M, td, kv, layer, Hq, out, ldo, part, cnt, nsmax};
  const int rep = Hq / kv.Hkv;
  if (kdt == Q3TTS_BF16)
    return kv.hd == 128 ? launch_split_rep<bf16, 128>(a, rep, n_sm, s) : launch_split_rep<bf16, 64>(a, rep, n_sm, s);
  return kv.hd == 128 ? launch_split_rep<float, 128>(a, rep, n_sm, s) : launch_split_rep<float, 64>(a, rep, n_sm, s);
}

void launch_attention(int kdt, const float* qkv, int ld, int M, TokDesc td, KVDesc kv, int layer,
                      int Hq, float* out, int ldo, int max_ctx, cudaStream_t s) {
  if (M <= 0) return;
  static int n_sm = 0;  // the current device's SM count (one device per process)
  if (!n_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n_sm = 1;
  }
  const size_t pts = sizeof(int) * (size_t)((max_ctx + kv.page_size - 1) / kv.page_size + 1);
  const bool bf = kdt == Q3TTS_BF16;
  if ((kv.hd == 128 || kv.hd == 64) && Hq / kv.Hkv <= GQA_RMAX && M * kv.Hkv < 2 * n_sm) {
    // few CTAs: eight warps per CTA, several K/V rows in flight per warp
    dim3 grid(M, kv.Hkv);
    const int nt = GQA_NW * 32;
    if (bf) {
      if (kv.hd == 128) launch_pdl(attention_gqa8_kernel<bf16, 4>, dim3(grid), dim3(nt), pts, s, qkv, ld, td, kv, layer, Hq, out, ldo);
      else launch_pdl(attention_gqa8_kernel<bf16, 2>, dim3(grid), dim3(nt), pts, s, qkv, ld, td, kv, layer, Hq, out, ldo);
    } else {
      if (kv.hd == 128) launch_pdl(attention_gqa8_kernel<float, 4>, dim3(grid), dim3(nt), pts, s, qkv, ld, td, kv, layer, Hq, out, ldo);
      else launch_pdl(attention_gqa8_kernel<float, 2>, dim3(grid), dim3(nt), pts, s, qkv, ld, td, kv, layer, Hq, out, ldo);
    }
    return;
  }
  if (kv.hd <= 128 && Hq / kv.Hkv <= 4) {
    dim3 grid(M, kv.Hkv);
    if (bf)
      launch_pdl(attention_gqa4_kernel<bf16>, dim3(grid), dim3(128), pts, s, qkv, ld, td, kv, layer, Hq, out, ldo);
    else
      launch_pdl(attention_gqa4_kernel<float>, dim3(grid), dim3(128), pts, s, qkv, ld, td, kv, layer, Hq, out, ldo);
    return;
  }
  dim3 grid(M, Hq);
  size_t smem = sizeof(float) * (size_t)(kv.hd + max_ctx);
  if (kdt == Q3TTS_BF16)
    launch_pdl(attention_kernel<bf16>, dim3(grid), dim3(128), smem, s, qkv, ld, td, kv, layer, Hq, out, ldo);
  else
    launch_pdl(attention_kernel<float>, dim3(grid), dim3(128), smem, s, qkv, ld, td, kv, layer, Hq, out, ldo);
}

// ---------------------------------------------------------------- SwiGLU
__global__ void silu_mul_kernel(const float* __restrict__ gu, float* __restrict__ a, int M, int F) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  size_t n = (size_t)M * F;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    size_t m = e / F, f = e % F;
    a[e] = silu(gu[m * 2 * F + f]) * gu[m * 2 * F + F + f];
  }
}

void launch_silu_mul(const float* gu, float* a, int M, int F, cudaStream_t s) {
  if (M <= 0) return;
  size_t n = (size_t)M * F;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 8192) blocks = 8192;
  launch_pdl(silu_mul_kernel, dim3(blocks), dim3(256), 0, s, gu, a, M, F);
}

__global__ void silu_mul_hilo_kernel(const float* __restrict__ gu, bf16* __restrict__ hi, bf16* __restrict__ lo,
                                     int M, int F) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  size_t n = (size_t)M * F;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    size_t m = e / F, f = e % F;
    store_hilo(hi, lo, e, silu(gu[m * 2 * F + f]) * gu[m * 2 * F + F + f]);
  }
}

void launch_silu_mul_hilo(const float* gu, const HiLo& a, int M, int F, cudaStream_t s) {
  if (M <= 0) return;
  size_t n = (size_t)M * F;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 8192) blocks = 8192;
  launch_pdl(silu_mul_hilo_kernel, dim3(blocks), dim3(256), 0, s, gu, a.hi, a.lo, M, F);
}

}  // namespace q3
