// common.cuh -- small device helpers shared by the kernels of libq3tts.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q3 {

typedef __nv_bfloat16 bf16;

// One FP8 E4M3 weight: the byte is its code (Q3TTS_FP8 weights).
struct fp8e4 {
  uint8_t v;
};

// Four E4M3 codes (the bytes of w, lowest first) as floats: each pair goes
// through the hardware's exact E4M3 -> f16 conversion, then to float.
__device__ __forceinline__ void fp8x4_to_f32(uint32_t w, float* f) {
  uint32_t lo, hi;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(static_cast<unsigned short>(w & 0xffffu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(static_cast<unsigned short>(w >> 16)));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// Programmatic dependent launch.  A kernel started by launch_pdl may begin
// while its predecessor on the stream is still running: pdl_wait() blocks
// until that grid has completed and its memory is visible (a no-op for a
// kernel launched without the attribute), pdl_trigger() lets the next
// kernel's CTAs be scheduled (they then wait in their own pdl_wait()).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Whether launch_pdl sets the attribute (Q3TTS_PDL=0 in the environment: plain
// stream order, for comparison).
bool pdl_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The storage type of the norm gains and embedding tables of a model whose
// matrices are WT (bf16 beside FP8 matrices), and whether WT is FP8.
template <class WT>
struct GainOf {
  using T = WT;
};
template <>
struct GainOf<fp8e4> {
  using T = bf16;
};
template <class WT>
constexpr bool kFp8 = false;
template <>
constexpr bool kFp8<fp8e4> = true;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }

template <class T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// Streaming 16-byte load that bypasses L1 (weights are read once per use).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void unpack_bf16x8(uint4 u, float* w) {
  w[0] = __uint_as_float(u.x << 16);
  w[1] = __uint_as_float(u.x & 0xffff0000u);
  w[2] = __uint_as_float(u.y << 16);
  w[3] = __uint_as_float(u.y & 0xffff0000u);
  w[4] = __uint_as_float(u.z << 16);
  w[5] = __uint_as_float(u.z & 0xffff0000u);
  w[6] = __uint_as_float(u.w << 16);
  w[7] = __uint_as_float(u.w & 0xffff0000u);
}

// Eight consecutive weights as float (p: 16-byte aligned for bf16, 32 for f32).
__device__ __forceinline__ void load_w8(const bf16* p, float* w) { unpack_bf16x8(ld_stream16(p), w); }
__device__ __forceinline__ void load_w8(const float* p, float* w) {
  uint4 a = ld_stream16(p), b = ld_stream16(p + 4);
  w[0] = __uint_as_float(a.x); w[1] = __uint_as_float(a.y);
  w[2] = __uint_as_float(a.z); w[3] = __uint_as_float(a.w);
  w[4] = __uint_as_float(b.x); w[5] = __uint_as_float(b.y);
  w[6] = __uint_as_float(b.z); w[7] = __uint_as_float(b.w);
}

__device__ __forceinline__ void load_w8(const fp8e4* p, float* w) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  fp8x4_to_f32(u.x, w);
  fp8x4_to_f32(u.y, w + 4);
}
__device__ __forceinline__ float to_f(fp8e4 v) {
  float f[4];
  fp8x4_to_f32(v.v, f);
  return f[0];
}

__device__ __forceinline__ void load_f8(const float* p, float* x) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum; `red` is shared scratch of >= 32 floats; all threads get the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

__device__ __forceinline__ float block_max(float v, float* red) {
  int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : -INFINITY;
  return warp_max(t);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + __expf(-z)); }

// Paged KV cache: element (layer, page, kv, head, slot, dim) lives at
// ((((layer * n_pages + page) * 2 + kv) * Hkv + head) * page_size + slot) * hd + dim.
struct KVDesc {
  void* pool;
  const int* page_table;  // [stream][pages_per_stream]
  int pages_per_stream, page_size, n_pages, Hkv, hd;
};

__device__ __forceinline__ size_t kv_offset(const KVDesc& d, int layer, int stream, int pos, int kv,
                                            int head) {
  int page = d.page_table[stream * d.pages_per_stream + pos / d.page_size];
  return ((((size_t)layer * d.n_pages + page) * 2 + kv) * d.Hkv + head) * d.page_size * d.hd +
         (size_t)(pos % d.page_size) * d.hd;
}

}  // namespace q3
