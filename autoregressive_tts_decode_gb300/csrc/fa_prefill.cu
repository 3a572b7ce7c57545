// fa_prefill.cu -- causal attention of a prefill chunk on the 5th-generation
// tensor cores.
//
// A prefill chunk feeds T consecutive prompt positions of one stream through
// a decoder layer ("Running Qwen3-TTS on an AMD R9700", section "Running
// Qwen3-TTS": the Talker runs over the prompt before the first frame); its
// attention is a dense causal contraction: every query position p attends over
// the stream's cached positions 0..p.  Token by token it would re-read each
// prefix (T^2 / 2 cache rows per head); here one CTA takes 64 query tokens and
// one kv head -- the group's two q heads give 128 query rows, the M of one
// tcgen05.mma -- and walks the cache in tiles of 64 positions, each read once
// for all 128 rows:
//   S = Q K^T      (tcgen05.mma kind::f16, M 128, N 64, K 128, fp32 in TMEM;
//                   Q enters as bf16 hi + lo terms, the bf16 cache exactly);
//   online softmax, one thread per row (TMEM lane): the causal mask, running
//                   max and sum, P = exp(S - max) written as bf16 hi + lo;
//   O += P V       (M 128, N 128, K 64, fp32 in TMEM; V transposed into a
//                   K-major tile by the threads, O rescaled in TMEM when the
//                   running max moves).
// Every operand tile is K-major with 128-byte swizzle (8-row atoms 1024 bytes
// apart), the layout the GEMM path's descriptors use.  Cache pages arrive by
// 16-byte cp.async copies straight into that layout; positions past the
// chunk's last one are zero-filled (unwritten cache words may hold NaN).
// Every wait is bounded; on expiry the CTA records Q3TTS_ERR_TIMEOUT, waits
// (bounded) for its issued MMAs, frees its TMEM and returns.
#include "layers.cuh"

namespace q3 {

namespace {

constexpr int FA_QT = 64;     // query tokens of a CTA
constexpr int FA_KT = 64;     // cache positions of a tile
constexpr int FA_HD = 128;    // head dimension this kernel takes
constexpr int FA_ROWS = 128;  // query rows: 2 heads x FA_QT tokens
constexpr long long FA_WAIT_CYCLES = 4000000000ll;

// shared-memory layout (bytes from a 1024-aligned base)
constexpr uint32_t FA_Q_BLK = FA_ROWS * 128;      // one 64-wide k block of Q: 16 KB
constexpr uint32_t FA_K_BLK = FA_KT * 128;        // one 64-wide k block of K: 8 KB
constexpr uint32_t OFF_QH = 0;                    // [2 blocks] Q hi
constexpr uint32_t OFF_QL = OFF_QH + 2 * FA_Q_BLK;  // [2 blocks] Q lo
constexpr uint32_t OFF_K = OFF_QL + 2 * FA_Q_BLK;   // [2 blocks] K tile
constexpr uint32_t OFF_VT = OFF_K + 2 * FA_K_BLK;   // V^T tile [128 hd rows][64 positions]
constexpr uint32_t OFF_PH = OFF_VT + FA_HD * 128;   // P hi [128 rows][64 positions]
constexpr uint32_t OFF_PL = OFF_PH + FA_ROWS * 128;
constexpr uint32_t OFF_V = OFF_PL + FA_ROWS * 128;  // V tile staging [64][128] bf16, plain rows
constexpr uint32_t OFF_CTL = OFF_V + FA_KT * FA_HD * 2;
constexpr size_t FA_SMEM = 1024 + OFF_CTL + 64;
constexpr uint32_t FA_TMEM_COLS = 256;  // S in columns 0..63, O in 128..255

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(count) : "memory");
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
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// K-major tile with 128-byte swizzle: 128-byte rows, 8-row atoms 1024 bytes
// apart, descriptor version 1, swizzle mode 2.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major.
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
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// 8 floats into bf16 hi and lo terms (x = hi + lo), packed 8 to a uint4 each.
__device__ __forceinline__ void hilo8(const float* x, uint4& h, uint4& l) {
  uint32_t hh[4], ll[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const bf16 a = __float2bfloat16_rn(x[2 * q]), b = __float2bfloat16_rn(x[2 * q + 1]);
    const bf16 c = __float2bfloat16_rn(x[2 * q] - __bfloat162float(a));
    const bf16 d = __float2bfloat16_rn(x[2 * q + 1] - __bfloat162float(b));
    hh[q] = (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
    ll[q] = (uint32_t)__bfloat16_as_ushort(c) | ((uint32_t)__bfloat16_as_ushort(d) << 16);
  }
  h = make_uint4(hh[0], hh[1], hh[2], hh[3]);
  l = make_uint4(ll[0], ll[1], ll[2], ll[3]);
}

struct FaArgs {
  const float* qkv;  // [T][ld], q of head h at h * 128 (after q-norm and RoPE)
  int ld, T;
  int stream, pos0;  // token t sits at position pos0 + t of the stream
  KVDesc kv;         // bf16 cache, 16 positions per page, hd 128
  int layer, Hq;
  float* out;        // [T][ldo], head h at h * 128
  int ldo;
  int* err;
};

// Bounded wait on an mbarrier phase.
__device__ __forceinline__ bool fa_wait(uint32_t bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > FA_WAIT_CYCLES) {
      atomicCAS(err, 0, Q3TTS_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(128, 1) fa_prefill_kernel(FaArgs a) {
  extern __shared__ uint8_t fa_raw[];
  pdl_wait();  // q, k, v come from the previous kernels
  const uint32_t raw = su32(fa_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = fa_raw + (base - raw);
  const uint32_t bar_s = base + OFF_CTL, bar_o = bar_s + 8, bar_done = bar_s + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bp + OFF_CTL + 24);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int g = blockIdx.y, t0 = blockIdx.x * FA_QT;
  const int rep = a.Hq / a.kv.Hkv;  // 2
  const KVDesc& kv = a.kv;
  const size_t head_stride = (size_t)kv.page_size * FA_HD;

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(FA_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Q of row tid: token t0 + (tid % 64), q head g rep + tid / 64, as hi/lo
  // terms in two 64-wide k blocks; rows past the chunk are zero
  {
    const int i = tid % FA_QT, h = g * rep + tid / FA_QT, t = t0 + i;
    const float* q = a.qkv + (size_t)t * a.ld + (size_t)h * FA_HD;
#pragma unroll 4
    for (int c = 0; c < 16; ++c) {
      float x[8];
      if (t < a.T) {
        const float4 u = *reinterpret_cast<const float4*>(q + 8 * c);
        const float4 v = *reinterpret_cast<const float4*>(q + 8 * c + 4);
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w; x[4] = v.x; x[5] = v.y; x[6] = v.z; x[7] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.f;
      }
      uint4 hh, ll;
      hilo8(x, hh, ll);
      const uint32_t blk = (uint32_t)(c >> 3) * FA_Q_BLK, off = swz(tid, c & 7);
      *reinterpret_cast<uint4*>(bp + OFF_QH + blk + off) = hh;
      *reinterpret_cast<uint4*>(bp + OFF_QL + blk + off) = ll;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lanes

  // the row's query position; rows past the chunk see no key
  const int my_t = t0 + (tid % FA_QT);
  const int qpos = my_t < a.T ? a.pos0 + my_t : -1;
  const int last_t = min(t0 + FA_QT, a.T) - 1;
  const int kend = a.pos0 + last_t + 1;  // positions the CTA's rows can see
  const float scale = 1.0f / sqrtf((float)FA_HD);
  float m_run = -INFINITY, l_run = 0.f;
  const int* pt = kv.page_table + (size_t)a.stream * kv.pages_per_stream;
  constexpr uint32_t idS = f16_idesc(FA_ROWS, FA_KT), idO = f16_idesc(FA_ROWS, FA_HD);
  int ntile = 0;
  bool ok = true;

  for (int p0 = 0; p0 < kend && ok; p0 += FA_KT, ++ntile) {
    // K rows into the two k blocks (swizzled) and V rows into plain staging
    // rows; a row past kend is zero-filled
    for (int e = tid; e < FA_KT * 32; e += 128) {
      const int r = e >> 5, c = e & 31, kvsel = c >> 4, cc = c & 15;
      const int pos = p0 + r;
      const bool valid = pos < kend;
      const int page = valid ? pt[pos / kv.page_size] : 0;
      const bf16* src = (const bf16*)kv.pool +
                        ((((size_t)a.layer * kv.n_pages + page) * 2 + kvsel) * kv.Hkv + g) * head_stride +
                        (size_t)(pos % kv.page_size) * FA_HD + (size_t)cc * 8;
      const uint32_t dst = kvsel == 0 ? base + OFF_K + (uint32_t)(cc >> 3) * FA_K_BLK + swz(r, cc & 7)
                                      : base + OFF_V + (uint32_t)(r * 256 + cc * 16);
      cp_async16(dst, valid ? (const void*)src : (const void*)kv.pool, valid ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // V^T: row d (thread d) holds positions 0..63 of head dimension d
    {
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(bp + OFF_V);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = (uint32_t)vs[(8 * c + 2 * q) * FA_HD + tid] | ((uint32_t)vs[(8 * c + 2 * q + 1) * FA_HD + tid] << 16);
        *reinterpret_cast<uint4*>(bp + OFF_VT + swz(tid, c)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    proxy_fence();  // the tensor cores read what the threads and cp.async wrote
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // S = Q K^T: two 64-wide k blocks, 4 k steps each, hi then lo
    if (tid == 0) {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t o = (uint64_t)(k * 2);
          mma_bf16(tS, sw128_desc(base + OFF_QH + kb * FA_Q_BLK) + o, sw128_desc(base + OFF_K + kb * FA_K_BLK) + o,
                   idS, (kb | k) != 0 ? 1u : 0u);
          mma_bf16(tS, sw128_desc(base + OFF_QL + kb * FA_Q_BLK) + o, sw128_desc(base + OFF_K + kb * FA_K_BLK) + o,
                   idS, 1u);
        }
      mma_commit(bar_s);
    }
    __syncwarp();
    ok = fa_wait(bar_s, (uint32_t)ntile & 1u, a.err);
    ok = __syncthreads_and(ok);
    if (!ok) break;
    tc_fence_after();
    // online softmax of this row over the tile
    float s[FA_KT];
#pragma unroll
    for (int c = 0; c < FA_KT / 16; ++c) {
      float v[16];
      tmem_ld16(tS + lane_off + (uint32_t)(16 * c), v);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int kp = p0 + 16 * c + e;
        s[16 * c + e] = (kp <= qpos) ? v[e] * scale : -INFINITY;
      }
    }
    float mt = -INFINITY;
#pragma unroll
    for (int e = 0; e < FA_KT; ++e) mt = fmaxf(mt, s[e]);
    const float m_new = fmaxf(m_run, mt);
    const float corr = m_run == -INFINITY ? 0.f : __expf(m_run - m_new);
    float lsum = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = s[8 * c + e];
        pv[e] = x == -INFINITY ? 0.f : __expf(x - m_new);
        lsum += pv[e];
      }
      uint4 hh, ll;
      hilo8(pv, hh, ll);
      *reinterpret_cast<uint4*>(bp + OFF_PH + swz(tid, c)) = hh;
      *reinterpret_cast<uint4*>(bp + OFF_PL + swz(tid, c)) = ll;
    }
    l_run = l_run * corr + lsum;
    m_run = m_new;
    // rescale the running output (after the first tile)
    if (ntile > 0) {
#pragma unroll 1
      for (int c = 0; c < FA_HD / 16; ++c) {
        float v[16];
        tmem_ld16(tO + lane_off + (uint32_t)(16 * c), v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= corr;
        tmem_st16(tO + lane_off + (uint32_t)(16 * c), v);
      }
    }
    proxy_fence();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // O += P V: 4 k steps of 16 positions, hi then lo
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t o = (uint64_t)(k * 2);
        mma_bf16(tO, sw128_desc(base + OFF_PH) + o, sw128_desc(base + OFF_VT) + o, idO,
                 (ntile > 0 || k > 0) ? 1u : 0u);
        mma_bf16(tO, sw128_desc(base + OFF_PL) + o, sw128_desc(base + OFF_VT) + o, idO, 1u);
      }
      mma_commit(bar_o);
    }
    __syncwarp();
    ok = fa_wait(bar_o, (uint32_t)ntile & 1u, a.err);
    ok = __syncthreads_and(ok);
    tc_fence_after();
  }
  // the output of row tid: O / l (every lane takes part in the warp-wide
  // TMEM loads; rows past the chunk store nothing)
  if (ok) {
    const int h = g * rep + tid / FA_QT;
    float* dst = a.out + (size_t)(qpos >= 0 ? my_t : 0) * a.ldo + (size_t)h * FA_HD;
    const float inv = qpos >= 0 ? 1.f / l_run : 0.f;
#pragma unroll 1
    for (int c = 0; c < FA_HD / 16; ++c) {
      float v[16];
      tmem_ld16(tO + lane_off + (uint32_t)(16 * c), v);
      if (qpos >= 0) {
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *reinterpret_cast<float4*>(dst + 16 * c + e) = make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv,
                                                                     v[e + 3] * inv);
      }
    }
  }
  pdl_trigger();
  // every MMA issued above has completed before the TMEM is given back
  if (tid == 0) mma_commit(bar_done);
  __syncwarp();
  fa_wait(bar_done, 0u, a.err);
  tc_fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(FA_TMEM_COLS) : "memory");
}

}  // namespace

bool fa_prefill_ok(const KVDesc& kv, int kdt, int Hq) {
  return kdt == Q3TTS_BF16 && kv.hd == FA_HD && kv.page_size == 16 && Hq == 2 * kv.Hkv;
}

bool launch_fa_prefill(const float* qkv, int ld, int T, int stream, int pos0, KVDesc kv, int kdt, int layer, int Hq,
                       float* out, int ldo, int* err, cudaStream_t s) {
  if (T <= 0) return true;
  if (!fa_prefill_ok(kv, kdt, Hq)) return false;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(fa_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FA_SMEM) !=
        cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    attr = true;
  }
  FaArgs a{qkv, ld, T, stream, pos0, kv, layer, Hq, out, ldo, err};
  return launch_pdl(fa_prefill_kernel, dim3((T + FA_QT - 1) / FA_QT, kv.Hkv), dim3(128), FA_SMEM, s, a) ==
         cudaSuccess;
}

}  // namespace q3
