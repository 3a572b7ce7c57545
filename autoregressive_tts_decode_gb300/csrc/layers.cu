// layers.cu -- one-kernel-per-operation decoder building blocks (see layers.cuh).
#include "layers.cuh"

namespace q3 {

// ---------------------------------------------------------------- linear
// Skinny case (few tokens): one warp per output row, eight weights per lane per
// step with 16-byte streaming loads; the row is multiplied with up to MT token
// vectors at once.
template <class WT, int MT>
__global__ void __launch_bounds__(256) gemv_kernel(const float* __restrict__ X, int ldx,
                                                   const WT* __restrict__ W, int N, int K,
                                                   float* __restrict__ Y, int ldy, int M,
                                                   int accumulate) {
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
                                                   int accumulate) {
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
        *y = accumulate ? *y + acc[i][j] : acc[i][j];
      }
    }
}

template <class WT>
static void linear_t(const float* X, int ldx, const WT* W, int N, int K, float* Y, int ldy, int M,
                     bool acc, cudaStream_t s) {
  if (M <= 0 || N <= 0) return;
  if (M <= 16) {
    int blocks = (N + 7) / 8;
    if (blocks > 4096) blocks = 4096;
    if (M <= 1)
      gemv_kernel<WT, 1><<<blocks, 256, 0, s>>>(X, ldx, W, N, K, Y, ldy, M, acc);
    else if (M <= 2)
      gemv_kernel<WT, 2><<<blocks, 256, 0, s>>>(X, ldx, W, N, K, Y, ldy, M, acc);
    else if (M <= 4)
      gemv_kernel<WT, 4><<<blocks, 256, 0, s>>>(X, ldx, W, N, K, Y, ldy, M, acc);
    else
      gemv_kernel<WT, 8><<<blocks, 256, 0, s>>>(X, ldx, W, N, K, Y, ldy, M, acc);
  } else {
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    gemm_kernel<WT><<<grid, 256, 0, s>>>(X, ldx, W, N, K, Y, ldy, M, acc);
  }
}

void launch_linear(int wdt, const float* X, int ldx, const void* W, int N, int K, float* Y, int ldy,
                   int M, bool accumulate, cudaStream_t s) {
  if (wdt == Q3TTS_BF16)
    linear_t(X, ldx, (const bf16*)W, N, K, Y, ldy, M, accumulate, s);
  else
    linear_t(X, ldx, (const float*)W, N, K, Y, ldy, M, accumulate, s);
}

// --------------------------------------------------------------- rmsnorm
template <class WT>
__global__ void rmsnorm_kernel(const float* __restrict__ X, int ldx, int in_mul, int in_add,
                               const WT* __restrict__ g, float* __restrict__ Y, int ldy, int D,
                               float eps) {
  __shared__ float red[32];
  const int m = blockIdx.x;
  const float* x = X + (size_t)(m * in_mul + in_add) * ldx;
  float ss = 0.f;
  for (int i = threadIdx.x; i < D; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)D + eps);
  for (int i = threadIdx.x; i < D; i += blockDim.x) Y[(size_t)m * ldy + i] = x[i] * inv * to_f(g[i]);
}

void launch_rmsnorm(int wdt, const float* X, int ldx, int in_mul, int in_add, const void* g,
                    float* Y, int ldy, int M, int D, float eps, cudaStream_t s) {
  if (M <= 0) return;
  if (wdt == Q3TTS_BF16)
    rmsnorm_kernel<<<M, 256, 0, s>>>(X, ldx, in_mul, in_add, (const bf16*)g, Y, ldy, D, eps);
  else
    rmsnorm_kernel<<<M, 256, 0, s>>>(X, ldx, in_mul, in_add, (const float*)g, Y, ldy, D, eps);
}

// ------------------------------------------------ q/k norm + RoPE + append
// One block per token, one warp per head; lane l holds elements l + 32 j, so
// the rotate-half partners i and i + hd/2 sit in the same lane.
template <class WT, class KT, int HD>
__global__ void qk_rope_append_kernel(float* __restrict__ qkv, int ld, TokDesc td,
                                      const WT* __restrict__ gq, const WT* __restrict__ gk,
                                      int qk_norm, float eps, const float* __restrict__ rc,
                                      const float* __restrict__ rs, KVDesc kv, int layer, int Hq) {
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
    qk_rope_append_kernel<WT, KT, 128><<<M, 256, 0, s>>>(qkv, ld, td, (const WT*)gq, (const WT*)gk,
                                                         qk_norm, eps, rc, rs, kv, layer, Hq);
  else
    qk_rope_append_kernel<WT, KT, 64><<<M, 256, 0, s>>>(qkv, ld, td, (const WT*)gq, (const WT*)gk,
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

void launch_attention(int kdt, const float* qkv, int ld, int M, TokDesc td, KVDesc kv, int layer,
                      int Hq, float* out, int ldo, int max_ctx, cudaStream_t s) {
  if (M <= 0) return;
  dim3 grid(M, Hq);
  size_t smem = sizeof(float) * (size_t)(kv.hd + max_ctx);
  if (kdt == Q3TTS_BF16)
    attention_kernel<bf16><<<grid, 128, smem, s>>>(qkv, ld, td, kv, layer, Hq, out, ldo);
  else
    attention_kernel<float><<<grid, 128, smem, s>>>(qkv, ld, td, kv, layer, Hq, out, ldo);
}

// ---------------------------------------------------------------- SwiGLU
__global__ void silu_mul_kernel(const float* __restrict__ gu, float* __restrict__ a, int M, int F) {
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
  silu_mul_kernel<<<blocks, 256, 0, s>>>(gu, a, M, F);
}

}  // namespace q3
