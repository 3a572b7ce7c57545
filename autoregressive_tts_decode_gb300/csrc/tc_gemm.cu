// tc_gemm.cu -- projections of the layered path on the 5th-generation tensor
// cores: Y[m, n] (+)= sum_k X[m, k] W[n, k] for bf16 weights W [N, K] and a few
// to a few hundred tokens m.
//
// Every projection of the decoder ("Running Qwen3-TTS on an AMD R9700",
// section "Running Qwen3-TTS": the Talker and CodePredictor layers' QKV,
// o_proj, gate/up and down matrices and the heads) becomes, for several
// streams or a prompt, a product of a tall weight matrix with a short stack of
// activation rows.  The weights are the MMA's M side (128 rows per CTA) and the
// tokens its N side (16..256), so a handful of streams still fills the
// instruction; the weights stream from HBM once per launch.
//
// Design (one CTA per 128 weight rows and K range, 128 threads):
//  * thread 0 is the producer: TMA tiled loads (cp.async.bulk.tensor, 128-byte
//    swizzle) of a 128 x 64 weight tile and the matching 64-wide slices of the
//    activation terms into a ring of stages, signalled by mbarrier
//    transaction counts; weights carry an L2 evict-first hint;
//  * thread 32 issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32) into a TMEM
//    accumulator of 128 lanes x N columns and frees each stage with
//    tcgen05.commit on its "empty" barrier;
//  * the activations enter as two bf16 terms, x = hi + lo with hi = bf16(x)
//    and lo = bf16(x - hi), each multiplied by the same weight tile into the
//    same accumulator: the product keeps about 16 mantissa bits of x, close to
//    an fp32 dot product, at twice the MMA work (the weights, not the tensor
//    pipe, bound a skinny product);
//  * the four warps then read the accumulator (tcgen05.ld, warp w owns lanes
//    32w..32w+31, i.e. weight rows) and store, add, or atomically add (K split
//    over CTAs) into Y, 32 consecutive outputs of one token per warp access.
//  * Every mbarrier wait is bounded; on expiry the CTA records
//    Q3TTS_ERR_TIMEOUT, stops issuing, waits (bounded) for its copies in
//    flight and its issued MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <tuple>

#include "layers.cuh"

namespace q3 {

namespace {

constexpr int TC_ROWS = 128;                           // weight rows per CTA (MMA M)
constexpr int TC_BK = 64;                              // k per stage: one 128-byte swizzle row of bf16
constexpr int TC_UK = 16;                              // k per MMA instruction (kind::f16)
constexpr uint32_t TC_WBYTES = TC_ROWS * TC_BK * 2;    // weight tile of one stage
constexpr long long TC_WAIT_CYCLES = 4000000000ll;     // ~2 s at GB300 clocks

template <int NT>
struct TcCfg {
  static constexpr uint32_t XBYTES = NT * TC_BK * 2;  // one activation term of one stage
  static constexpr uint32_t STAGE = TC_WBYTES + 2 * XBYTES;
  static constexpr int S = NT <= 16 ? 5 : (NT <= 32 ? 4 : (NT <= 64 ? 3 : 2));  // two CTAs per SM up to 128 tokens
  static constexpr uint32_t TMEM_COLS = NT < 32 ? 32 : NT;
  // stages (1024-byte aligned), barriers and the TMEM address slot
  static constexpr size_t SMEM = 1024 + (size_t)S * STAGE + 256;
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(b), "r"(parity)
      : "memory");
  return ok != 0;
}

// 2-D tiled TMA load of box (x = k, y = row) into shared memory at dst.
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_hint(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile with 128-byte swizzle:
// rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart (stride byte
// offset), leading byte offset unused for this layout (encoded 1), descriptor
// version 1, swizzle mode 2 (128 B).  The start address advances by 32 bytes
// per 16-element k step inside the swizzle row.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t f16_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 16 consecutive fp32 columns of the warp's 32 TMEM lanes (one per thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

struct TcArgs {
  float* Y;
  int ldy, M, N;
  int kb_per, nkb;  // 64-wide k blocks per CTA, in all
  int mode;         // 0: store, 1: add (one CTA per output), 2: atomic add (K split)
  int* err;
};

// Bounded wait on an mbarrier phase; false (after raising the CTA's abort
// word and the error word) on expiry or when another role has aborted.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort_w, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  unsigned it = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++it & 63u) == 0) {
      if (*abort_w) return false;
      if (clock64() - t0 > TC_WAIT_CYCLES) {
        *abort_w = 1;
        atomicCAS(err, 0, Q3TTS_ERR_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

template <int NT>
__global__ void __launch_bounds__(128, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap hmap,
                   const __grid_constant__ CUtensorMap lmap, TcArgs a) {
  using C = TcCfg<NT>;
  extern __shared__ uint8_t tc_raw[];
  const uint32_t raw = su32(tc_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms want 1024-byte alignment
  uint8_t* ctl = tc_raw + (base - raw) + (size_t)C::S * C::STAGE;
  const uint32_t full0 = su32(ctl), empty0 = full0 + 8 * C::S, done = empty0 + 8 * C::S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctl + 16 * C::S + 8);
  volatile int* abort_w = reinterpret_cast<volatile int*>(ctl + 16 * C::S + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * TC_ROWS;
  const int kb0 = blockIdx.y * a.kb_per;
  const int nk = min(a.nkb, kb0 + a.kb_per) - kb0;  // >= 1: the host sizes the split so
  const int m0 = blockIdx.z * NT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(done, 1);
    *abort_w = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the set-up above overlaps the previous kernel; its outputs are read below
  pdl_wait();

  if (threadIdx.x == 0) {
    // producer
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
    const uint64_t pol = evict_first_policy();
    int issued = 0;
    for (int i = 0; i < nk; ++i) {
      const int s = i % C::S;
      const uint32_t ph = (uint32_t)(i / C::S) & 1u;
      if (!tc_wait(empty0 + 8 * s, ph ^ 1u, abort_w, a.err)) break;
      const uint32_t st = base + (uint32_t)s * C::STAGE, fb = full0 + 8 * s;
      const int kx = (kb0 + i) * TC_BK;
      mbar_expect_tx(fb, C::STAGE);
      tma_load_hint(st, &wmap, kx, n0, fb, pol);
      tma_load(st + TC_WBYTES, &hmap, kx, m0, fb);
      tma_load(st + TC_WBYTES + C::XBYTES, &lmap, kx, m0, fb);
      issued = i + 1;
    }
    // copies still in flight land before the CTA may exit (normally all have)
    for (int j = issued - C::S > 0 ? issued - C::S : 0; j < issued; ++j) {
      const uint32_t fb = full0 + 8 * (j % C::S);
      const uint32_t ph = (uint32_t)(j / C::S) & 1u;
      const long long t0 = clock64();
      while (!mbar_try_wait(fb, ph) && clock64() - t0 < TC_WAIT_CYCLES) {
      }
    }
  } else if (threadIdx.x == 32) {
    // MMA issuer
    constexpr uint32_t idesc = f16_idesc(TC_ROWS, NT);
    for (int i = 0; i < nk; ++i) {
      const int s = i % C::S;
      const uint32_t ph = (uint32_t)(i / C::S) & 1u;
      if (!tc_wait(full0 + 8 * s, ph, abort_w, a.err)) break;
      tc_fence_after();
      const uint32_t st = base + (uint32_t)s * C::STAGE;
      const uint64_t dw = sw128_desc(st), dh = sw128_desc(st + TC_WBYTES),
                     dl = sw128_desc(st + TC_WBYTES + C::XBYTES);
#pragma unroll
      for (int k = 0; k < TC_BK / TC_UK; ++k) {
        const uint64_t o = (uint64_t)((k * TC_UK * 2) >> 4);
        mma_bf16(tmem, dw + o, dh + o, idesc, (i | k) != 0 ? 1u : 0u);
        mma_bf16(tmem, dw + o, dl + o, idesc, 1u);
      }
      mma_commit(empty0 + 8 * s);  // the stage is free once these MMAs have read it
    }
    mma_commit(done);  // arrives when every MMA issued above has completed
  }
  __syncwarp();

  // epilogue: warp w holds weight rows n0 + 32 w + lane, all NT token columns;
  // the next kernel may start its set-up meanwhile
  pdl_trigger();
  bool ok = tc_wait(done, 0u, abort_w, a.err);
  ok = __all_sync(0xffffffffu, ok) && !*abort_w;
  tc_fence_after();
  if (ok) {
    const int n = n0 + warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int c0 = 0; c0 < NT; c0 += 16) {
      float v[16];
      tmem_ld16(trow + (uint32_t)c0, v);
      if (n < a.N) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = m0 + c0 + j;
          if (m < a.M) {
            float* y = a.Y + (size_t)m * a.ldy + n;
            if (a.mode == 0)
              *y = v[j];
            else if (a.mode == 1)
              *y += v[j];
            else
              atomicAdd(y, v[j]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
}

// ------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor map of a row-major bf16 matrix [rows, K] (row pitch ld elements) read
// in boxes of box_rows x 64 with 128-byte swizzle; cached per argument set (a
// map depends on nothing else).
bool tensor_map(const void* p, int rows, int K, int ld, int box_rows, CUtensorMap* out) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, int, int>, CUtensorMap> cache;
  const auto key = std::make_tuple(p, rows, K, ld, box_rows);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return true;
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  CUtensorMap m;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)TC_BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache.emplace(key, m);
  *out = m;
  return true;
}

template <int NT>
bool launch_nt(const CUtensorMap& wm, const HiLo& x, int N, int K, float* Y, int ldy, int M, bool acc, int* err,
               int n_sm, cudaStream_t s) {
  using C = TcCfg<NT>;
  CUtensorMap hm, lm;
  if (!tensor_map(x.hi, x.rows, K, K, NT, &hm) || !tensor_map(x.lo, x.rows, K, K, NT, &lm)) return false;
  const int nrb = (N + TC_ROWS - 1) / TC_ROWS, nkb = K / TC_BK, ntt = (M + NT - 1) / NT;
  // CTAs resident per SM at this stage count (TMEM holds 512 columns)
  const int per_sm = (int)std::min<size_t>(228 * 1024 / (C::SMEM + 1024), 512 / C::TMEM_COLS);
  const int slots = std::max(1, per_sm) * n_sm;
  // K split, only when the output tiles alone leave SMs idle: the fewest
  // splits that minimise (waves of CTAs) x (k blocks per CTA + c), c standing
  // for a CTA's fixed costs in k blocks (set-up, pipeline fill, and the
  // read-back and atomic adds of its 128 x NT outputs, repeated per split)
  int splits = 1;
  if ((long)nrb * ntt < slots) {
    constexpr int c = 2 + NT / 32;
    long best = -1;
    for (int sp = 1; sp <= nkb; ++sp) {
      const int per = (nkb + sp - 1) / sp;
      const long ctas = (long)nrb * ntt * ((nkb + per - 1) / per);
      const long cost = ((ctas + slots - 1) / slots) * (per + c);
      if (best < 0 || cost < best) {
        best = cost;
        splits = sp;
      }
    }
  }
  const int kb_per = (nkb + splits - 1) / splits;
  splits = (nkb + kb_per - 1) / kb_per;  // every CTA gets at least one k block
  TcArgs args;
  args.Y = Y;
  args.ldy = ldy;
  args.M = M;
  args.N = N;
  args.kb_per = kb_per;
  args.nkb = nkb;
  args.mode = splits > 1 ? 2 : (acc ? 1 : 0);
  args.err = err;
  if (splits > 1 && !acc &&
      cudaMemset2DAsync(Y, (size_t)ldy * sizeof(float), 0, (size_t)N * sizeof(float), M, s) != cudaSuccess)
    return false;
  launch_pdl(tc_gemm_kernel<NT>, dim3(nrb, splits, ntt), dim3(128), C::SMEM, s, wm, hm, lm, args);
  return cudaPeekAtLastError() == cudaSuccess;
}

// X = hi + lo, hi = bf16(x), lo = bf16(x - hi)
__global__ void split_hilo_kernel(const float* __restrict__ X, int ldx, bf16* __restrict__ hi,
                                  bf16* __restrict__ lo, int M, int K) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  const int m = blockIdx.y;
  for (int k = (blockIdx.x * blockDim.x + threadIdx.x) * 4; k < K; k += gridDim.x * blockDim.x * 4) {
    const float4 v = *reinterpret_cast<const float4*>(X + (size_t)m * ldx + k);
    const float xs[4] = {v.x, v.y, v.z, v.w};
    bf16 h[4], l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      h[q] = __float2bfloat16_rn(xs[q]);
      l[q] = __float2bfloat16_rn(xs[q] - __bfloat162float(h[q]));
    }
    *reinterpret_cast<uint2*>(hi + (size_t)m * K + k) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(lo + (size_t)m * K + k) = *reinterpret_cast<const uint2*>(l);
  }
}

template <int NT>
bool set_smem_attr() {
  if (cudaFuncSetAttribute(tc_gemm_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)TcCfg<NT>::SMEM) == cudaSuccess)
    return true;
  cudaGetLastError();
  return false;
}

// Kernel attributes, set once per process (outside any graph capture).
bool tc_setup() {
  static bool ok = false;
  static std::once_flag once;
  std::call_once(once, [] {
    ok = encode_fn() != nullptr && set_smem_attr<16>() && set_smem_attr<32>() && set_smem_attr<64>() &&
         set_smem_attr<128>() && set_smem_attr<256>();
  });
  return ok;
}

}  // namespace

bool tc_linear_ok(int N, int K, int M) { return N > 0 && M > 0 && K % TC_BK == 0 && tc_setup(); }

bool tc_linear(const HiLo& x, const void* W, int N, int K, float* Y, int ldy, int M, bool accumulate, int* err,
               cudaStream_t s) {
  if (!tc_linear_ok(N, K, M) || M > x.rows) return false;
  CUtensorMap wm;
  if (!tensor_map(W, N, K, K, TC_ROWS, &wm)) return false;
  int dev = 0, n_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  // the smallest token tile that covers M (at most 256 tokens per tile)
  if (M <= 16) return launch_nt<16>(wm, x, N, K, Y, ldy, M, accumulate, err, n_sm, s);
  if (M <= 32) return launch_nt<32>(wm, x, N, K, Y, ldy, M, accumulate, err, n_sm, s);
  if (M <= 64) return launch_nt<64>(wm, x, N, K, Y, ldy, M, accumulate, err, n_sm, s);
  if (M <= 128) return launch_nt<128>(wm, x, N, K, Y, ldy, M, accumulate, err, n_sm, s);
  return launch_nt<256>(wm, x, N, K, Y, ldy, M, accumulate, err, n_sm, s);
}

void launch_split_hilo(const float* X, int ldx, const HiLo& x, int M, int K, cudaStream_t s) {
  if (M <= 0) return;
  int bx = (K / 4 + 255) / 256;
  launch_pdl(split_hilo_kernel, dim3(dim3(bx, M)), dim3(256), 0, s, X, ldx, x.hi, x.lo, M, K);
}

}  // namespace q3
