// layers.cuh -- one-kernel-per-operation building blocks of the decoder stack.
//
// These kernels run the Talker prefill (many positions at once) and the
// layer-by-layer frame step for any number of streams.  Activations are fp32,
// weights fp32 or bf16 (template WT), the Talker KV cache fp32 or bf16 (KT).
// A "token" m is one row of the activation buffers; tok_stream[m] names its
// stream and tok_pos[m] its position (when tok_pos is NULL every token sits at
// pos_const).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "q3tts.h"

namespace q3 {

struct TokDesc {
  const int* tok_stream;
  const int* tok_pos;  // NULL: every token at pos_const
  int pos_const;
};

// Y[m, n] (+)= sum_k X[m, k] W[n, k] for m < M, n < N (FP8 W: times the row
// scale scale[n]).
void launch_linear(int wdt, const float* X, int ldx, const void* W, int N, int K, float* Y, int ldy,
                   int M, bool accumulate, cudaStream_t s, const float* scale = nullptr);

// Y[m] = X[in_row(m)] / rms * g, in_row(m) = m * in_mul + in_add.
void launch_rmsnorm(int wdt, const float* X, int ldx, int in_mul, int in_add, const void* g,
                    float* Y, int ldy, int M, int D, float eps, cudaStream_t s);

// Per token: q and k heads RMSNorm'ed (if qk_norm) and rotated at the token's
// position; q written back in place, k and v stored into the paged cache.
void launch_qk_rope_append(int wdt, int kdt, float* qkv, int ld, int M, TokDesc td, const void* gq,
                           const void* gk, int qk_norm, float eps, const float* rope_cos,
                           const float* rope_sin, KVDesc kv, int layer, int Hq, cudaStream_t s);

// Single-query attention of every token over positions 0..pos of its stream.
void launch_attention(int kdt, const float* qkv, int ld, int M, TokDesc td, KVDesc kv, int layer,
                      int Hq, float* out, int ldo, int max_ctx, cudaStream_t s);

// The same attention with all tokens' cache pages spread evenly over the
// GPU's warps (pages of 16 positions, hd 64 or 128, 1, 2 or 4 q heads per kv
// head; false if the shape is not one it takes).  part holds
// [M][Hq][nsmax][hd + 2] floats of partial results (nsmax =
// attention_split_spans(kv_cap)), cnt [M][Hkv] ints that must be zero before
// the first launch (every launch leaves them zero).
bool launch_attention_split(int kdt, const float* qkv, int ld, int M, TokDesc td, KVDesc kv, int layer, int Hq,
                            float* out, int ldo, float* part, int* cnt, int nsmax, cudaStream_t s);
int attention_split_spans(int kv_cap);

// Causal attention of a prefill chunk on the tensor cores (fa_prefill.cu):
// tokens t < T of one stream at positions pos0 + t, whose k and v are already
// in the cache; bf16 cache, hd 128, two q heads per kv head, pages of 16.
// err receives Q3TTS_ERR_TIMEOUT if a bounded wait runs out.  False if the
// shape is not one it takes (nothing launched).
bool fa_prefill_ok(const KVDesc& kv, int kdt, int Hq);
bool launch_fa_prefill(const float* qkv, int ld, int T, int stream, int pos0, KVDesc kv, int kdt, int layer, int Hq,
                       float* out, int ldo, int* err, cudaStream_t s);

// a[m, f] = silu(gu[m, f]) * gu[m, F + f]
void launch_silu_mul(const float* gu, float* a, int M, int F, cudaStream_t s);

// Activation operand of the tensor-core projections: x = hi + lo, two bf16
// matrices [rows][K] (row pitch K, the product's inner dimension), hi = bf16(x)
// and lo = bf16(x - hi).
struct HiLo {
  bf16* hi;
  bf16* lo;
  int rows;  // rows the buffers hold
};

// Whether the tensor-core path takes a product of this shape (K % 64 == 0 and
// the driver's tensor-map encoder is available).
bool tc_linear_ok(int N, int K, int M);

// Y[m, n] (+)= sum_k (hi[m, k] + lo[m, k]) W[n, k] for bf16 W [N, K] on the
// tcgen05 tensor cores (tc_gemm.cu); err receives Q3TTS_ERR_TIMEOUT if a
// bounded device wait runs out.  False if nothing was launched.
bool tc_linear(const HiLo& x, const void* W, int N, int K, float* Y, int ldy, int M, bool accumulate, int* err,
               cudaStream_t s);

// x (fp32 [M, K], row pitch ldx) -> its hi/lo terms.
void launch_split_hilo(const float* X, int ldx, const HiLo& x, int M, int K, cudaStream_t s);

// RMSNorm (as launch_rmsnorm) written as hi/lo terms.
void launch_rmsnorm_hilo(int wdt, const float* X, int ldx, int in_mul, int in_add, const void* g, const HiLo& y,
                         int M, int D, float eps, cudaStream_t s);

// silu(gu[m, f]) * gu[m, F + f] written as hi/lo terms.
void launch_silu_mul_hilo(const float* gu, const HiLo& a, int M, int F, cudaStream_t s);

}  // namespace q3
