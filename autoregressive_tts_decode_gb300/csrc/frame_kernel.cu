// frame_kernel.cu -- one acoustic frame of one stream in a single persistent
// launch.
//
// The frame ("Running Qwen3-TTS on an AMD R9700", section "Running Qwen3-TTS"):
// draw the semantic token from the pending Talker logits, run 15 CodePredictor
// passes (pass 0 over [Talker hidden, semantic embedding], pass j over the
// embedding of acoustic token j; each ends in head j and a draw), sum the 16
// code embeddings ("qwen3-tts-hip" README, "Python Parity Fixtures") and run
// one Talker step whose final norm and codec head leave the next pending
// logits.  The page's cost model -- bytes(Talker) + 15 bytes(CodePredictor)
// per frame -- makes this a weight-streaming problem: at batch 1 every weight
// byte is used by one multiply-add.
//
// Design (GB300, one CTA per SM, cooperative launch, 320 threads):
//  * A producer warp walks the frame's weight schedule for its CTA -- the
//    same slices the consumers will need, in frame order -- and streams them
//    through a 20-deep ring of 8 KB chunks in shared memory with 1-D bulk
//    copies (cp.async.bulk + mbarrier transaction counts, L2 evict-first).
//    Weights do not depend on activations, so the stream runs ahead across
//    phase boundaries.  A second warp prefetches 8 chunks further ahead into
//    L2 (a deeper prefetch delays the latency-bound phases).
//  * Eight consumer warps.  A private chunk (rows of a GEMV, an o_proj tile,
//    gate and up rows) belongs to one warp, which computes whole dot
//    products over it alone; a shared chunk (rows of the transposed down
//    projection) is read by every warp for its own output columns.  No
//    block-wide barrier sits inside a streaming loop.
//  * RMSNorm is lazy: the staged input is g * x (one CTA-wide pass), and
//    each GEMV output is scaled by the one inverse RMS afterwards.
//  * The residual stream of layer k is a base vector plus an attention delta
//    and an FFN delta (FK_KC copies of the latter, so that the split-K
//    atomics of 152 CTAs spread over more addresses); the next layer's
//    RMSNorm sums them while staging and folds the sum into its own base.
//  * FFN in two stages without a grid barrier between them: a CTA computes
//    silu(gate) * up for its own intermediate channels (rows of the caller's
//    gate/up tensor), then adds their rank-k contribution to all outputs
//    through rows of W_down^T (a copy made at create) with float4 atomics.
//    o_proj works the same way over 32-column tiles of one head.
//  * Values that one phase hands to the next without a reduction -- QKV
//    rows, the CodePredictor input projection, Talker attention partials,
//    CodePredictor logits -- are 64-bit words (value, step tag) written with
//    relaxed stores; a reader polls the words it needs until their tag is
//    this step's.  Grid barriers remain only where the next phase reads a
//    complete atomic sum (after o_proj and after the FFN, plus one at the
//    frame start): 207 per 1.7B frame.
//  * Draws are made redundantly by every CTA from the full logit vector
//    (sampler.cuh, fast_sample), so a sampled code needs no barrier.
//  * The frame is a list of steps decoded from a (pass, step) position, each
//    step kind with one call site, so every phase's code exists once; the
//    consumers' loop state, the launch parameters and the CTA's share of
//    every phase (the plan, computed on the host) live in shared memory, so
//    that no phase starts with a division or a global load of its bounds.
//  * The grid barrier is a release-add / acquire-load counter polled by one
//    thread per CTA.  Every wait (ring slots, side slots, tags, grid barrier)
//    is bounded; on expiry the kernel records Q3TTS_ERR_TIMEOUT, raises an
//    abort flag, stops waiting, lets in-flight copies land and returns.
#include <algorithm>
#include <cmath>
#include <atomic>
#include <mutex>
#include <new>
#include <type_traits>
#include <vector>

#include "engine.cuh"
#include "sampler.cuh"

namespace q3 {

constexpr int FK_CONSUMER_WARPS = 8;
constexpr int FK_CONSUMERS = FK_CONSUMER_WARPS * 32;
constexpr int FK_PRODUCER_THREADS = 32;  // one warp; one thread issues the copies
constexpr int FK_PREFETCH_THREADS = 32;  // one warp; one thread issues L2 prefetches
constexpr int FK_THREADS = FK_PRODUCER_THREADS + FK_CONSUMERS + FK_PREFETCH_THREADS;
constexpr int FK_STAGE = 8192;  // one ring chunk: 2 rows of 2048 bf16, one o_proj tile of 32 x 128 bf16
constexpr int FK_NSTAGE = 20;
constexpr int FK_PF_AHEAD = 8;  // default distance (chunks) the L2 prefetch runs ahead of the ring (measured on GB300: 8 best of 0, 8, 24, 64; deeper prefetch queues up memory traffic that delays the latency-bound phases)
constexpr int FK_TMAX = 2;     // tokens per pass (CodePredictor pass 0 carries two)
constexpr int FK_DMAX = 2048;  // widest hidden state staged in shared memory
constexpr int FK_HDMAX = 128;
constexpr int FK_REPMAX = 2;   // q heads per kv head
constexpr int FK_MAXCTA = 256;
constexpr int FK_PAIRS = 4;    // (head, token) pairs of one CTA in a CodePredictor attention
constexpr long long FK_WAIT_CYCLES = 4000000000ll;  // ~2 s at GB300 clocks: the default wait bound
// Per-layer "side block" (norm gains g_attn | g_ffn | g_q | g_k, weight dtype),
// copied into a double-buffered shared-memory slot one layer ahead.
// Largest over the configurations the kernel takes (bf16 at D = 2048, fp32 at
// D <= 1024); checked at create.
constexpr int FK_SIDE_BYTES = 9216;
constexpr int FK_FIN_BYTES = 8192;  // final-norm gains of both stacks
constexpr int FK_MAXLAYERS = 64;  // Talker + CodePredictor layers held in shared memory
constexpr int FK_RMAX = 8;        // rows of one ring chunk a warp keeps in flight
constexpr int FK_KC = 4;          // copies of each residual buffer the split-K sums are spread over
constexpr int FK_UMAX = 64;       // FFN units of one CTA

static_assert(FAST_NT == FK_CONSUMERS, "the register sampler runs on the consumer warps");

struct LayerDev {
  const void* side;   // [g_attn D | g_ffn D | g_q hd | g_k hd], weight dtype, contiguous
  const void* w_qkv;
  const void* w_oT;   // o_proj tiles [Hq][ceil(D/32)][hd/8][32][8] (see oproj_step)
  const void* w_gu;   // [2F][D]: gate rows, then up rows (the caller's tensor)
  const void* w_dT;   // [F][D]: W_down transposed, row f = column f of W_down
  // FP8 matrices: per-output-row scales (W_qkv rows, W_o rows = output
  // columns of o_proj, gate rows then up rows, W_down rows = output columns)
  const float* s_qkv;
  const float* s_o;
  const float* s_gu;
  const float* s_d;
};

// A CTA's share of every phase of a frame.  It depends only on the
// configuration and the CTA's index, so the host computes it once
// (frame_kernel_create) and each CTA copies its row into shared memory at the
// start of a frame: no phase divides on its critical path.  Index s: 0 the
// CodePredictor, 1 the Talker.
struct FKRange {
  int lo, hi, nch;  // items [lo, hi), in nch ring chunks
};
struct FKPlan {
  FKRange qkv[2];   // rows of W_qkv
  FKRange proj;     // rows of the CodePredictor input projection (width D_t)
  FKRange head[2];  // rows of the CodePredictor head / of the Talker head
  FKRange ffn[2];   // FFN units [f0, f1) in nch gate/up chunks
  int ffn_nd[2];    // chunks of the units' W_down^T rows
  int op_t0[2], op_t1[2], op_h0[2], op_h1[2];  // o_proj tiles [t0, t1) and the heads h0..h1 they cover
  int sl_lo[3], sl_hi[3];  // the CTA's slice of a D_c-, D_t- and xstride-long vector
  int rpc[2];       // rows of width D_c / D_t per ring chunk
  int upc[2];       // FFN units of width D_c / D_t per ring chunk
  float invD[2];    // 1 / D_c, 1 / D_t
  float inv_nt[2];  // 1 / (o_proj tiles per head), for D_c / D_t
  int cpg, tg, tch; // Talker attention: CTAs per kv group; this CTA's group and chunk
  int hd_shift, rep_shift;   // log2 head_dim, log2 (q heads per kv head)
  float inv_hd, attn_scale;  // 1 / head_dim, 1 / sqrt(head_dim)
};

struct FKParams {
  int ncta;
  int Dt, Dc, Ft, Fc, Hq, Hkv, hd, Vt, Vc, Lt, Lc, qkv_rows, has_proj, qk_norm, dmax;
  float eps;
  const LayerDev* tl;
  const LayerDev* cl;
  const FKPlan* plan;  // [ncta]
  const void *t_head, *e_codec, *cp_heads, *cp_embeds, *cp_proj, *t_gfinal, *cp_gfinal;
  const float *s_head, *s_cp_heads, *s_cp_proj;  // FP8: the heads' and projection's row scales
  float* pending_h;
  float* pending_logits;
  uint8_t* history;
  uint8_t* finished;  // per stream: its end-of-stream code was fed
  KVDesc tkv, ckv;
  const float* rope_cos;
  const float* rope_sin;
  // residual stream (see xbase), by layer parity: base vectors, attention
  // deltas, FFN deltas (FK_KC copies); each [tokens][D] within xstride floats
  float* xb;  // [2][xstride]
  float* xa;  // [2][xstride]
  float* xf;  // [2][FK_KC][xstride]
  int xstride;
  // values handed from one phase to the next without a grid barrier, each
  // stored with the tag of the step that wrote it (see tag_of)
  uint64_t* qkv;        // [FK_TMAX][qkv_rows]
  uint64_t* z;          // [FK_TMAX][Dc]: the CodePredictor input projection
  uint64_t* part;       // [Hq][cpg][hd + 2]: Talker attention partials
  uint64_t* cp_logits;  // [Vc]
  uint32_t seq;         // this launch's sequence number
  int pf_ahead;         // chunks the L2 prefetch warp may run ahead of the ring (0: off)
  unsigned* bar;
  unsigned* done;
  int* err;
  int* abort_flag;
  long long wait_cycles;  // bound of every wait on another thread or CTA (clock64 cycles)
  int fail_bar;           // grid barrier whose arrival CTA 0 skips (-1: none; failure-path test)
  // this call
  int sid, pos, newpage;
  q3tts_sampling sp;
  const float* uniforms;
  int32_t* codes;
  const int32_t* forced;
  float* dump;
};

struct FKState {
  void* base;
  char* sideT;
  char* sideC;
  LayerDev* tl;
  LayerDev* cl;
  FKPlan* plan;  // [ncta]
  float *xb, *xa, *xf;
  uint64_t *qkv, *z, *part, *cp_logits;
  uint32_t seq;  // launches of this handle with its workspace scratch
  int pf_ahead;  // L2 prefetch distance in chunks (Q3TTS_PF_AHEAD at create; 0 turns it off)
  unsigned *bar, *done;
  int* abort_flag;
  int ncta, dmax;
  size_t smem;
  bool ok;
};

}  // namespace q3

struct q3::FrameKernelState : q3::FKState {};

namespace q3 {

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t* b, unsigned n) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(n) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

#ifdef Q3TTS_TRACE
// Whether the phase has completed, without suspending the thread.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* b, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
#endif

// As mbar_try_wait, but the thread may be suspended up to about `ns`
// nanoseconds while the phase is incomplete (woken early when it completes),
// so a waiting thread issues few instructions.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* b, unsigned parity, unsigned ns) {
  unsigned ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Weight bytes are read once per use: the copy carries an L2 evict-first
// policy so the stream does not push activations, KV rows and code out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                         uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Moves bytes at src (16-byte aligned, a multiple of 16) towards L2 ahead of
// their copy into shared memory.
__device__ __forceinline__ void prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(FK_CONSUMERS) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_volatile(const int* p) { return *(const volatile int*)p; }

// A value handed between CTAs without a grid barrier travels with a tag in
// one 64-bit word (value bits | tag << 32), written and read as relaxed
// gpu-scope accesses: an aligned 64-bit access is single-copy atomic, so a
// reader that sees the expected tag sees the value stored with it.
__device__ __forceinline__ uint64_t tag_word(float v, uint32_t tag) {
  return ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v);
}
// (No compiler memory clobber on the store: nothing is ordered against it but
// through the tag itself, and a clobber would keep the compiler from issuing
// the next rows' shared-memory loads ahead of it.)
__device__ __forceinline__ void st_tagged(uint64_t* p, float v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(tag_word(v, tag)));
}
__device__ __forceinline__ uint64_t ld_relaxed64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// Part i of n items cut into `parts` near-equal parts.  32-bit unsigned
// arithmetic: n * parts stays far below 2^32 for every split made here (rows,
// FFN units, tiles, vector elements; parts = CTAs <= 256), and a 64-bit
// division would be a long software routine on the critical path of a phase.
__device__ __forceinline__ void split(int n, int parts, int i, int& lo, int& hi) {
  lo = (int)((unsigned)n * (unsigned)i / (unsigned)parts);
  hi = (int)((unsigned)n * (unsigned)(i + 1) / (unsigned)parts);
}

__device__ __forceinline__ int rows_per_chunk(int row_bytes) {
  const int r = FK_STAGE / row_bytes;
  return r < 1 ? 1 : (r > FK_RMAX ? FK_RMAX : r);
}

// Activations staged for a GEMV use a "plane" layout so that lane reads of 8
// consecutive elements are bank-conflict free: for a vector of length K,
// float4 j of plane 0 holds elements 8j..8j+3 and float4 j of plane 1 (at
// offset K/2) holds 8j+4..8j+7.  plane_first(p, K) is the first element of
// plane float4 p (p < K/4).
__device__ __forceinline__ int plane_first(int p, int K) {
  const int half = K >> 3;
  return p < half ? 8 * p : 8 * (p - half) + 4;
}

// ------------------------------------------------------------ shared memory

// The block's dynamic shared memory.  Hot loops address it through 32-bit
// offsets from this array (shared-window loads), not through generic pointers.
extern __shared__ __align__(128) unsigned char fk_smem_raw[];

__device__ __forceinline__ uint32_t soff(const void* p) {
  return (uint32_t)((const unsigned char*)p - fk_smem_raw);
}
__device__ __forceinline__ float4 lds_f4(uint32_t off) {
  return *reinterpret_cast<const float4*>(fk_smem_raw + off);
}
__device__ __forceinline__ uint4 lds_u4(uint32_t off) {
  return *reinterpret_cast<const uint4*>(fk_smem_raw + off);
}
template <class WT>
__device__ __forceinline__ void lds_w8(uint32_t off, float* w);
template <>
__device__ __forceinline__ void lds_w8<bf16>(uint32_t off, float* w) {
  unpack_bf16x8(lds_u4(off), w);
}
template <>
__device__ __forceinline__ void lds_w8<float>(uint32_t off, float* w) {
  const float4 a = lds_f4(off), b = lds_f4(off + 16);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}
template <>
__device__ __forceinline__ void lds_w8<fp8e4>(uint32_t off, float* w) {
  const uint2 u = *reinterpret_cast<const uint2*>(fk_smem_raw + off);
  fp8x4_to_f32(u.x, w);
  fp8x4_to_f32(u.y, w + 4);
}

struct AttnScratch {
  float m[FK_CONSUMER_WARPS][FK_PAIRS];
  float l[FK_CONSUMER_WARPS][FK_PAIRS];
  float o[FK_CONSUMER_WARPS][FK_PAIRS][FK_HDMAX];
  float q[FK_PAIRS][FK_HDMAX];
  float kcur[FK_PAIRS][FK_HDMAX];  // current-position keys (token, kv group), normalised and rotated
  float vcur[FK_PAIRS][FK_HDMAX];  // current-position values (token, kv group)
};
static_assert(FK_PAIRS >= FK_REPMAX, "talker attention keeps one partial per q head of a group");

// Per consumer warp: ring chunks consumed, grid barriers passed, layers
// started (side-slot index), whether the warp gave up after a timeout, and
// the position in the frame's schedule.
struct ConsState {
  uint32_t n, phase, layer;
  int aborted;
  int j, k, s, src, fed0;  // the frame schedule's loop state: pass j, its step k, step s of the frame;
                           // where the next QKV step finds its input (SRC_*)
};

constexpr int FK_MAXPAGES = 256;  // Talker pages per stream kept in shared memory

struct FKSmem {
  alignas(128) unsigned char ring[FK_NSTAGE][FK_STAGE];
  // Launch parameters and per-layer pointer tables live in shared memory: a
  // read through a pointer to the parameter block or a global table costs a
  // memory round trip, which the short phases cannot afford.
  FKParams prm;
  LayerDev lay[FK_MAXLAYERS];  // Talker layers, then CodePredictor layers
  // Arrays read or written with 16-byte vector accesses are 16-byte aligned
  // whatever the size of the fields before them.
  union alignas(16) {
    struct {
      float xs[FK_TMAX * FK_DMAX];      // staged activations of the current GEMV (plane layout)
    } g;
    FastSamplerSmem smp;
    AttnScratch att;
  } u;
  alignas(16) float os[2][FK_TMAX][FK_HDMAX];  // attention outputs of the CTA's (<= 2) heads, plane layout
  alignas(16) float red[FK_TMAX][FK_CONSUMER_WARPS];
  alignas(16) float act[FK_TMAX][FK_UMAX];  // the CTA's FFN activations silu(gate) * up
  alignas(16) float rope_c[17][FK_HDMAX / 2];  // rows 0..15: CodePredictor positions; 16: the Talker position
  alignas(16) float rope_s[17][FK_HDMAX / 2];
  alignas(128) unsigned char side[2][FK_SIDE_BYTES];
  alignas(16) unsigned char fin[FK_FIN_BYTES];  // final-norm gains: CodePredictor then Talker
  float uni[Q3TTS_N_CODEBOOKS];
  int forced[Q3TTS_N_CODEBOOKS];
  int fedc[Q3TTS_N_CODEBOOKS];  // the frame's codes fed forward so far
  int fin_state;                 // CTA 0: 0 running, 1 ended by this frame, 2 ended before
  int tpage[FK_MAXPAGES];  // the stream's Talker page table (when it has at most FK_MAXPAGES pages)
  int cpage;               // the stream's CodePredictor page
  alignas(8) uint64_t full[FK_NSTAGE];
  alignas(8) uint64_t empty[FK_NSTAGE];
  alignas(8) uint64_t side_full[2];
  alignas(8) uint64_t side_empty[2];
  int flag;
  uint32_t pf_gate;  // chunks the ring's producer has issued (read by the prefetch warp)
  ConsState cs[FK_CONSUMER_WARPS];
  FKPlan plan;  // this CTA's row of the plan
  int ta_s0, ta_s1;  // this frame: the Talker positions [s0, s1) this CTA's attention chunk covers
#ifdef Q3TTS_TRACE
  int trace_n;
  long long trace_wait[FK_CONSUMER_WARPS];  // clock64 cycles each consumer warp spent in ring waits this step
#endif
};
static_assert(sizeof(FKSmem) <= 227 * 1024, "persistent kernel shared memory");
static_assert(offsetof(FKSmem, u) % 16 == 0 && offsetof(FKSmem, os) % 16 == 0 && offsetof(FKSmem, act) % 16 == 0 &&
                  offsetof(FKSmem, fin) % 16 == 0 && offsetof(FKSmem, side) % 16 == 0,
              "vector-accessed shared-memory arrays are 16-byte aligned");

// ---------------------------------------------------------------- context

// The consumer warps' context.  Nothing of it lives in local memory: the
// launch parameters and the shared-memory layout sit at fixed shared
// addresses, thread and block indices come from special registers, and each
// warp's mutable state (ConsState) is a shared-memory record.  A local-memory
// context would put a dependent load -- which can miss the small L1 left
// beside the ring -- in front of every phase.  Cons is an empty tag passed by
// value to the phase functions.
struct Cons {};

__device__ __forceinline__ FKSmem* fk_sm() { return reinterpret_cast<FKSmem*>(fk_smem_raw); }
__device__ __forceinline__ const FKParams* fk_prm() { return &fk_sm()->prm; }

// Offsets of the stream's K/V rows in the paged caches.  The page ids come
// from the copies of the stream's page tables staged in shared memory at the
// start of the frame: read from global memory, they would put a second
// dependent memory round trip in front of every cache access.
__device__ __forceinline__ size_t kv_row(const KVDesc& d, int page, int layer, int slot, int kv, int head) {
  return ((((size_t)layer * d.n_pages + page) * 2 + kv) * d.Hkv + head) * d.page_size * d.hd + (size_t)slot * d.hd;
}
// Page and slot of a position (the persistent kernel takes power-of-two page
// sizes only, so a shift and a mask, with no division code in the kernel).
__device__ __forceinline__ void page_slot(const KVDesc& d, int pos, int& pi, int& slot) {
  const int ps = d.page_size;
  pi = pos >> (__ffs(ps) - 1);
  slot = pos & (ps - 1);
}
__device__ __forceinline__ size_t tkv_offset(const FKParams& p, int layer, int pos, int kv, int head) {
  const KVDesc& d = p.tkv;
  int pi, slot;
  page_slot(d, pos, pi, slot);
  const int page = d.pages_per_stream <= FK_MAXPAGES ? fk_sm()->tpage[pi]
                                                     : __ldcg(d.page_table + p.sid * d.pages_per_stream + pi);
  return kv_row(d, page, layer, slot, kv, head);
}
// The CodePredictor cache holds a stream's 16 positions in one page: the k
// (kv = 0) or v row of position pos of kv group `head` is pos * hd past the
// row of position 0.
__device__ __forceinline__ size_t ckv_base(const FKParams& p, int layer, int kv, int head) {
  return kv_row(p.ckv, fk_sm()->cpage, layer, 0, kv, head);
}
__device__ __forceinline__ int ctid() { return (int)threadIdx.x - FK_PRODUCER_THREADS; }
__device__ __forceinline__ int cwarp() { return ctid() >> 5; }
__device__ __forceinline__ int clane() { return (int)threadIdx.x & 31; }
__device__ __forceinline__ int ccta() { return (int)blockIdx.x; }
__device__ __forceinline__ ConsState& cst() { return fk_sm()->cs[cwarp()]; }

// Updates a field of the warp's record from all 32 lanes: the new value is
// computed (from the old one) by every lane before any lane stores it, so the
// identical stores cannot race with a lagging lane's read.
template <class T>
__device__ __forceinline__ void warp_set(T& field, T v) {
  __syncwarp();
  field = v;
  __syncwarp();
}

struct ConsGroup {
  __device__ static int tid() { return threadIdx.x - FK_PRODUCER_THREADS; }
  __device__ static int nt() { return FK_CONSUMERS; }
  __device__ static void sync() { consumer_sync(); }
};

// Phase timestamps for profiling builds (compiled only with -DQ3TTS_TRACE):
// consumer thread 0 of each CTA appends {globaltimer, clock64, tag, aux} to
// the CTA's row of fk_trace_buf.  Without the define FK_MARK is empty.
#ifdef Q3TTS_TRACE
constexpr int FK_TRACE_EV = 8192;
__device__ uint4 fk_trace_buf[FK_MAXCTA * FK_TRACE_EV];
__device__ __forceinline__ void fk_mark(int tag, int aux) {
  if (ctid() != 0) return;
  int& n = fk_sm()->trace_n;
  if (n >= FK_TRACE_EV) return;
  unsigned long long g;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g));
  const unsigned long long c = clock64();
  fk_trace_buf[blockIdx.x * FK_TRACE_EV + n] =
      make_uint4((unsigned)g, (unsigned)(g >> 32), (unsigned)c, ((unsigned)tag << 16) | ((unsigned)aux & 0xffffu));
  n++;
}
#define FK_MARK(tag, aux) fk_mark(tag, aux)
#else
#define FK_MARK(tag, aux) ((void)0)
#endif
enum { TR_STEP = 1, TR_NORM = 2, TR_ARRIVE = 3, TR_PASS = 4, TR_WAIT0 = 5, TR_WAIT1 = 6, TR_END = 7,
       TR_CW0 = 8, TR_CW1 = 9, TR_REL = 10, TR_SUB = 11 };

__device__ __forceinline__ void raise_abort(const FKParams& p, int code) {
  atomicCAS(p.err, 0, code);
  atomicExch(p.abort_flag, 1);
}

// The tag of frame step s: unique over the launches of a workspace (the host
// numbers them), so a word left by an earlier step or frame never passes for
// the current one.
constexpr int FK_MAXSTEPS = 1024;  // steps of a frame (checked at create)
__device__ __forceinline__ uint32_t tag_of(int s) { return fk_prm()->seq * (uint32_t)FK_MAXSTEPS + (uint32_t)s; }

// Whether a thread waiting for tagged words should stop: the abort flag, or
// its bound (wait_cycles since t0) ran out, which it records.
__device__ __noinline__ bool tag_give_up(long long t0) {
  if (ld_volatile(fk_prm()->abort_flag)) return true;
  if (clock64() - t0 > fk_prm()->wait_cycles) {
    raise_abort(*fk_prm(), Q3TTS_ERR_TIMEOUT);
    return true;
  }
  return false;
}

// Resolves N words loaded (raw) from base + off[i]: each poll re-loads every
// word whose tag is not yet `tag`, all together, so the wait ends about one
// round trip after the last of them is written.  Entries a caller does not
// need hold a word already tagged `tag`.  After an abort or a timeout the
// words stay as they are.
template <int N>
__device__ __forceinline__ void tag_resolve(uint64_t (&raw)[N], const uint64_t* base, const int (&off)[N],
                                            uint32_t tag) {
  bool ok = true;
#pragma unroll
  for (int i = 0; i < N; ++i) ok = ok && (uint32_t)(raw[i] >> 32) == tag;
  if (ok) return;
  const long long t0 = clock64();
  unsigned it = 0;
  while (true) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((uint32_t)(raw[i] >> 32) != tag) raw[i] = ld_relaxed64(base + off[i]);
    ok = true;
#pragma unroll
    for (int i = 0; i < N; ++i) ok = ok && (uint32_t)(raw[i] >> 32) == tag;
    if (ok || ((++it & 15u) == 0 && tag_give_up(t0))) break;
  }
}

__device__ __forceinline__ float tag_float(uint64_t w) { return __uint_as_float((uint32_t)w); }
__device__ __forceinline__ uint64_t tag_filler(uint32_t tag) { return (uint64_t)tag << 32; }

// Bounded wait on an arbitrary mbarrier phase (all lanes of the calling warp).
__device__ __forceinline__ void wait_bar(Cons c, uint64_t* bar, unsigned par) {
  if (cst().aborted) return;
  long long t0 = clock64();
  unsigned it = 0;
  bool ab = false;
  while (!mbar_try_wait(bar, par)) {
    if ((++it & 255u) == 0 && (ld_volatile(fk_prm()->abort_flag) || clock64() - t0 > fk_prm()->wait_cycles)) {
      ab = true;
      break;
    }
  }
  ab = __any_sync(0xffffffffu, ab);  // one decision per warp
  if (ab && clane() == 0) raise_abort(*fk_prm(), Q3TTS_ERR_TIMEOUT);
  warp_set(cst().aborted, ab ? 1 : 0);
}

// The side block of the layer being started (waits for its copy).
template <class WT>
__device__ __forceinline__ const WT* side_begin(Cons c) {
  const int slot = cst().layer & 1;
  wait_bar(c, &fk_sm()->side_full[slot], (cst().layer >> 1) & 1u);
  return reinterpret_cast<const WT*>(fk_sm()->side[slot]);
}

// Done with the current layer's gains: the slot may be refilled (not after an
// abort, for the reason given at release_at).
__device__ __forceinline__ void side_end(Cons c) {
  if (ctid() == 0 && !cst().aborted) mbar_arrive(&fk_sm()->side_empty[cst().layer & 1]);
  warp_set(cst().layer, cst().layer + 1u);
}

// Grid-wide barrier of all CTAs' consumers: a monotonic arrival counter,
// release-add to arrive, acquire-load to wait (the last CTA to finish the
// launch resets it).
__device__ void grid_sync(Cons c) {
  consumer_sync();
  FK_MARK(TR_ARRIVE, 0);
  if (ctid() == 0) {
    const FKParams& p = *fk_prm();
    // the failure-path test leaves one arrival out, so every CTA's wait below
    // runs out of its bound
    if (!(ccta() == 0 && cst().phase == (unsigned)p.fail_bar)) red_release_add(p.bar, 1u);
    cst().phase++;
    const unsigned target = cst().phase * (unsigned)p.ncta;
    int fail = cst().aborted ? 1 : 0;
    if (!fail) {
      long long t0 = clock64();
      unsigned it = 0;
      while (ld_acquire(p.bar) < target) {
        if ((++it & 63u) == 0 && (ld_volatile(p.abort_flag) || clock64() - t0 > p.wait_cycles)) {
          raise_abort(p, Q3TTS_ERR_TIMEOUT);
          fail = 1;
          break;
        }
      }
    }
    fk_sm()->flag = fail;
  }
  consumer_sync();
  FK_MARK(TR_PASS, 0);
  if (fk_sm()->flag) warp_set(cst().aborted, 1);
}

// ------------------------------------------------------------ streaming
//
// A ring chunk is consumed in one of two ways.  A private chunk (rows of a
// GEMV, an o_proj tile, the gate and up rows of a few FFN units) belongs to
// warp n % 8, which computes whole dot products over it alone: no exchange
// between warps and no barrier inside a streaming loop.  A shared chunk (rows
// of the transposed down projection) is read by every warp, each for its own
// output columns.  A slot's "empty" barrier expects FK_CONSUMER_WARPS
// arrivals: the owner of a private chunk arrives with that count, every warp
// once for a shared chunk.  A streaming loop keeps what it touches per chunk
// in registers.

struct Stream {
  int lane, warp;
  bool aborted;
};

__device__ __forceinline__ Stream stream_begin(Cons c) {
  Stream s;
  s.lane = clane();
  s.warp = cwarp();
  s.aborted = cst().aborted;
  return s;
}

// The warp's first private chunk at or after n0.
__device__ __forceinline__ uint32_t first_chunk(uint32_t n0, int warp) {
  return n0 + (uint32_t)((warp - (int)(n0 % FK_CONSUMER_WARPS) + FK_CONSUMER_WARPS) % FK_CONSUMER_WARPS);
}

// The slow path of chunk_wait (out of line: it keeps the streaming loops'
// code short): waits for the mbarrier phase at shared offset bar with a bound;
// returns whether the warp gave up (timeout or abort flag), after recording
// the timeout.
__device__ __noinline__ bool chunk_wait_slow(uint32_t bar, unsigned par) {
  const long long t0 = clock64();
  unsigned it = 0;
  bool ab = false;
  uint64_t* b = reinterpret_cast<uint64_t*>(fk_smem_raw + bar);
  while (!mbar_try_wait(b, par)) {
    if ((++it & 255u) == 0 && (ld_volatile(fk_prm()->abort_flag) || clock64() - t0 > fk_prm()->wait_cycles)) {
      ab = true;
      break;
    }
  }
  ab = __any_sync(0xffffffffu, ab);  // one decision per warp
  if (ab && clane() == 0) raise_abort(*fk_prm(), Q3TTS_ERR_TIMEOUT);
  return ab;
}

// Waits (bounded) for ring chunk n; returns its shared-memory offset.
__device__ __forceinline__ uint32_t chunk_wait(Stream& s, uint32_t n) {
  FKSmem* sm = fk_sm();
  const uint32_t slot = n % FK_NSTAGE;
  if (!s.aborted) {
    const unsigned par = (n / FK_NSTAGE) & 1u;
#ifdef Q3TTS_TRACE
    // profiling builds test without suspending, so that the wait is seen
    const long long tw = clock64();
    if (!__all_sync(0xffffffffu, mbar_test_wait(&sm->full[slot], par)))
      s.aborted = chunk_wait_slow(soff(&sm->full[slot]), par);
    if (clane() == 0) sm->trace_wait[cwarp()] += clock64() - tw;
#else
    if (!__all_sync(0xffffffffu, mbar_try_wait(&sm->full[slot], par)))
      s.aborted = chunk_wait_slow(soff(&sm->full[slot]), par);
#endif
  }
  return soff(sm->ring[slot]);
}

// Hands ring chunk n back to the producer once the whole warp is done with it.
// After an abort a consumer has stopped waiting for data, so it must not free
// slots either: the producer then blocks, sees the abort flag and lets its
// in-flight copies land before the CTA can exit.
__device__ __forceinline__ void release_private(const Stream& s, uint32_t n) {
  __syncwarp();
  if (s.lane == 0 && !s.aborted) mbar_arrive_n(&fk_sm()->empty[n % FK_NSTAGE], FK_CONSUMER_WARPS);
}
__device__ __forceinline__ void release_shared(const Stream& s, uint32_t n) {
  __syncwarp();
  if (s.lane == 0 && !s.aborted) mbar_arrive_n(&fk_sm()->empty[n % FK_NSTAGE], 1u);
}

// 8 weights at shared offset w times 8 activations (plane halves xa, xb) into
// the two partial sums a, b.
template <class WT>
__device__ __forceinline__ void fma8(uint32_t w, const float4& xa, const float4& xb, float& a, float& b) {
  float wv[8];
  lds_w8<WT>(w, wv);
  a = fmaf(wv[0], xa.x, a); a = fmaf(wv[1], xa.y, a); a = fmaf(wv[2], xa.z, a); a = fmaf(wv[3], xa.w, a);
  b = fmaf(wv[4], xb.x, b); b = fmaf(wv[5], xb.y, b); b = fmaf(wv[6], xb.z, b); b = fmaf(wv[7], xb.w, b);
}

// acc + w . (a, c): two short chains of four, then one add.
__device__ __forceinline__ float dot8(const float (&w)[8], const float4& a, const float4& c, float acc) {
  const float s = fmaf(w[0], a.x, fmaf(w[1], a.y, fmaf(w[2], a.z, w[3] * a.w)));
  const float s2 = fmaf(w[4], c.x, fmaf(w[5], c.y, fmaf(w[6], c.z, w[7] * c.w)));
  return acc + (s + s2);
}

// Dot products of NR rows of a chunk at shared offset w (row i at w + ro[i];
// K elements each) with the T staged vectors at shared offset xs (plane
// layout, token t at xs + 4 K t): acc[i][t], the full sums in every lane.
// Lane l takes elements 256 b + 8 l .. + 7 of each 256-wide block b (lanes past
// a ragged last block take none); a block's activations are loaded once for
// all rows, and the NR T sums are reduced together so that their shuffle
// chains overlap.  NR and T are compile-time: a guard on a runtime row count
// inside an unrolled loop would issue the skipped rows' instructions anyway.
// Four bf16 rows of 1024 against one token (the CodePredictor's QKV, head and
// gate/up rows): every shared-memory load of the group -- the lane's 32
// activations and its 4 x 4 weight vectors -- is issued before the first
// multiply, so their latencies overlap (measured on GB300: 1,330 cycles per
// 8 KB chunk and warp, against 2,270 for the block loop below).
template <int NR>
__device__ __forceinline__ void dots4_k1024(uint32_t w, const uint32_t (&ro)[NR], uint32_t xs, int lane,
                                            float (&acc)[NR][1]) {
  constexpr int K = 1024;
  const uint32_t wl = w + (uint32_t)(lane * 16), xl = xs + (uint32_t)(lane * 16);
  float4 xa[4], xc[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    xa[b] = lds_f4(xl + (uint32_t)(b * 512));
    xc[b] = lds_f4(xl + (uint32_t)(b * 512 + K * 2));
  }
  uint4 wr[NR][4];
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int b = 0; b < 4; ++b) wr[r][b] = lds_u4(wl + ro[r] + (uint32_t)(b * 512));
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    float a = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float f[8];
      unpack_bf16x8(wr[r][b], f);
      a = dot8(f, xa[b], xc[b], a);
    }
    acc[r][0] = a;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r][0] += __shfl_xor_sync(0xffffffffu, acc[r][0], o);
}

template <class WT, int T, int NR>
__device__ __forceinline__ void dots(uint32_t w, const uint32_t (&ro)[NR], int K, uint32_t xs, int lane,
                                     float (&acc)[NR][T]) {
  if constexpr (T == 1 && NR == 4 && std::is_same<WT, bf16>::value) {
    if (K == 1024) {
      dots4_k1024<NR>(w, ro, xs, lane, acc);
      return;
    }
  }
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int t = 0; t < T; ++t) acc[r][t] = 0.f;
  const uint32_t wl = w + (uint32_t)(lane * 8 * (int)sizeof(WT));
  const uint32_t xl = xs + (uint32_t)(lane * 16);
  const int nb = (K >> 8) + (lane * 8 < (K & 255) ? 1 : 0);  // blocks with elements of this lane
#pragma unroll 1
  for (int b = 0; b < nb; ++b) {
    float4 xa[T], xc[T];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const uint32_t o = xl + (uint32_t)(b * 512 + t * K * 4);
      xa[t] = lds_f4(o);
      xc[t] = lds_f4(o + (uint32_t)K * 2u);
    }
    const uint32_t wb = wl + (uint32_t)(b * 256 * (int)sizeof(WT));
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float wv[8];
      lds_w8<WT>(wb + ro[r], wv);
#pragma unroll
      for (int t = 0; t < T; ++t) acc[r][t] = dot8(wv, xa[t], xc[t], acc[r][t]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int t = 0; t < T; ++t) acc[r][t] += __shfl_xor_sync(0xffffffffu, acc[r][t], o);
}

// Where a row GEMV puts its outputs: out[t * ts + row] as a plain float, or
// out64[t * ts + row] as a word tagged `tag` (out64 non-null).
struct RowsOut {
  float* out;
  uint64_t* out64;
  uint32_t tag;
  int ts;
  const float* sc;  // FP8: the matrix's row scales
};

// Rows base + r0 .. base + r0 + NR - 1 of a chunk (row stride rb) against T
// tokens, inv_t (row . x_t) stored by lane r T + t (the stores go out
// together) for the nv (<= NR) rows that exist.  The others are computed on
// whatever their shared-memory bytes hold (still inside the CTA's shared
// memory) and not stored: one row-group shape serves every chunk.
template <class WT, int T, int NR>
__device__ __forceinline__ void rows_group(uint32_t buf, int rb, int r0, int K, uint32_t xs, int lane,
                                           const RowsOut& o, int base, const float (&inv)[T], int nv) {
  uint32_t ro[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) ro[r] = (uint32_t)((r0 + r) * rb);
  float acc[NR][T];
  dots<WT, T, NR>(buf, ro, K, xs, lane, acc);
#pragma unroll
  for (int r = 0; r < NR; ++r)
#pragma unroll
    for (int t = 0; t < T; ++t)
      if (lane == r * T + t && r < nv) {
        const int i = t * o.ts + base + r0 + r;
        float v = acc[r][t] * inv[t];
        if constexpr (kFp8<WT>) v *= __ldg(o.sc + base + r0 + r);
        if (o.out64)
          st_tagged(o.out64 + i, v, o.tag);
        else
          o.out[i] = v;
      }
}

// Rows [r0, r1) of a row-major [*, K] matrix streamed from the ring (the
// private chunks the producer cut them into) against T staged vectors at
// shared offset xs: output row of token t = inv_t (row . x_t), placed as o
// says.  A chunk's rows go in groups of four when it holds a multiple of four
// rows (the activations are read from shared memory once per group, and they
// are half of a group's shared-memory traffic at two rows), else in pairs (a
// ragged last row computed with its neighbour's bytes and not stored).
// Advances the ring position past the rows' chunks.
template <class WT, int T>
__device__ __forceinline__ void stream_rows_t(Cons c, const FKRange& rg, int rpc, int K, uint32_t xs,
                                              const RowsOut& o, const float (&inv)[T]) {
  Stream s = stream_begin(c);
  const int rb = K * (int)sizeof(WT);
  const int r0 = rg.lo, r1 = rg.hi;
  const uint32_t n0 = cst().n;
  const uint32_t nch = (uint32_t)rg.nch;
  for (uint32_t n = first_chunk(n0, s.warp); n < n0 + nch; n += FK_CONSUMER_WARPS) {
    const uint32_t buf = chunk_wait(s, n);
    const int base = r0 + (int)(n - n0) * rpc, R = min(rpc, r1 - base);
    if ((rpc & 3) == 0) {
#pragma unroll 1
      for (int r = 0; r < R; r += 4) rows_group<WT, T, 4>(buf, rb, r, K, xs, s.lane, o, base, inv, R - r);
    } else {
#pragma unroll 1
      for (int r = 0; r < R; r += 2) rows_group<WT, T, 2>(buf, rb, r, K, xs, s.lane, o, base, inv, R - r);
    }
    release_private(s, n);
  }
  warp_set(cst().aborted, s.aborted ? 1 : 0);
  warp_set(cst().n, n0 + nch);
}

template <class WT>
__device__ __forceinline__ void stream_rows(Cons c, const FKRange& rg, int rpc, int K, int T, uint32_t xs,
                                            const RowsOut& o, float inv0, float inv1) {
  if (T == 1) {
    const float inv[1] = {inv0};
    stream_rows_t<WT, 1>(c, rg, rpc, K, xs, o, inv);
  } else {
    const float inv[2] = {inv0, inv1};
    stream_rows_t<WT, 2>(c, rg, rpc, K, xs, o, inv);
  }
}

// ------------------------------------------------------- residual helpers

// Residual stream.  Layer k of the frame (CodePredictor layers of the 15
// passes, then the Talker's) keeps, by the parity of k, [tokens][D] vectors
// (D the width of its stack): xbase(k), its input x_k, which the QKV phase
// writes (each CTA its slice; nobody adds into it); xattn(k), which the o_proj
// tiles of all CTAs add into; and xffn(k), FK_KC copies which the FFN's
// split-K sums of CTA c add into (copy c % FK_KC, so fewer CTAs add into one
// cache line).  So the FFN phase reads x_k + a_k = xbase + xattn, and layer
// k + 1 (or a head) reads x_{k+1} = xbase + xattn + the sum of the xffn copies.
// The FFN phase of layer k clears its CTA's slice of xattn(k + 1) and xffn(k +
// 1) (their last readers -- layer k's QKV phase -- are past the grid barrier
// that closed layer k's attention); the frame's first layer finds its deltas
// cleared at the start of the frame.
__device__ __forceinline__ float* xbase(const FKParams& p, int k) { return p.xb + (size_t)(k & 1) * p.xstride; }
__device__ __forceinline__ float* xattn(const FKParams& p, int k) { return p.xa + (size_t)(k & 1) * p.xstride; }
__device__ __forceinline__ float* xffn(const FKParams& p, int k, int copy) {
  return p.xf + ((size_t)(k & 1) * FK_KC + copy) * p.xstride;
}

// Where load_norm finds its input: raw tokens in xs, the tagged projection z,
// or the residual of a layer (x + a + f, or x + a within the FFN phase).
enum { SRC_XS = 0, SRC_Z = 1, SRC_RES = 2, SRC_RES_A = 3 };

// Gains g[i .. i+3] (weight dtype) as floats.
template <class WT>
__device__ __forceinline__ float4 gain4(const WT* g, int i);
template <>
__device__ __forceinline__ float4 gain4<bf16>(const bf16* g, int i) {
  const uint2 u = *reinterpret_cast<const uint2*>(g + i);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                     __uint_as_float(u.y & 0xffff0000u));
}
template <>
__device__ __forceinline__ float4 gain4<float>(const float* g, int i) {
  return *reinterpret_cast<const float4*>(g + i);
}

// The CTA's slice [lo, hi) of a vector: which = 0 (D_c long), 1 (D_t), 2
// (xstride), from the plan.
__device__ __forceinline__ void cta_slice(int which, int& lo, int& hi) {
  lo = fk_sm()->plan.sl_lo[which];
  hi = fk_sm()->plan.sl_hi[which];
}

// 1 / rms of staged token t of stack s (width D_s), from load_norm's partial
// sums (the mean square as sum * (1 / D_s); rsqrt within 2 ulp).
__device__ __forceinline__ float norm_inv(int t, int s) {
  const float* r = fk_sm()->red[t];
  float a = 0.f;
#pragma unroll
  for (int w = 0; w < FK_CONSUMER_WARPS; ++w) a += r[w];
  return rsqrtf(fmaf(a, fk_sm()->plan.invD[s], fk_prm()->eps));
}

// Stages y_t = g * x_t in xs (plane layout) for t < T, where x_t comes from
// src: SRC_XS, xs itself (raw plane layout); SRC_Z, token t of the tagged
// projection z (tag ztag); SRC_RES / SRC_RES_A, token t0 + t of layer kp's
// residual.  Leaves x_t's partial sums of squares in red[t][warp]:
// RMSNorm(x_t) * g = y_t / rms_t, and the GEMVs that follow scale their sums
// by 1 / rms_t (norm_inv) instead of normalising first, so staging takes one
// block-wide barrier.  Thread e handles plane float4 e + 256 u of the T
// tokens, all of its loads issued together.  With fold >= 0 the CTA's slice of
// each raw x_t goes to xbase(fold).  If out is given, the CTA's slice of the
// normed x_0 goes there.  g points into shared memory (4-element aligned
// groups).  sd: the stack (0 CodePredictor, 1 Talker) whose width D is.
template <class WT>
__device__ __noinline__ void load_norm(Cons c, int src, int kp, uint32_t ztag, int t0, int T, int D, int sd,
                                       const WT* g, int fold, float* out) {
  const FKParams& p = *fk_prm();
  float* xs = fk_sm()->u.g.xs;
  constexpr int PER = FK_DMAX / 4 / FK_CONSUMERS;  // float4 per thread: T D <= FK_DMAX (checked at create)
  const int nq = D >> 2, tot = T * nq, tid = ctid();
  float4 xv[PER];
  if (src == SRC_XS) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + FK_CONSUMERS * u;
      xv[u] = e < tot ? reinterpret_cast<const float4*>(xs)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  } else if (src == SRC_Z) {
    uint64_t raw[PER * 4];
    int off[PER * 4];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + FK_CONSUMERS * u;
      const int t = e >= nq ? 1 : 0;
      const int o = e < tot ? t * D + plane_first(e - t * nq, D) : 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        off[4 * u + k] = o + k;
        raw[4 * u + k] = e < tot ? ld_relaxed64(p.z + o + k) : tag_filler(ztag);
      }
    }
    tag_resolve<PER * 4>(raw, p.z, off, ztag);
#pragma unroll
    for (int u = 0; u < PER; ++u)
      xv[u] = make_float4(tag_float(raw[4 * u]), tag_float(raw[4 * u + 1]), tag_float(raw[4 * u + 2]),
                          tag_float(raw[4 * u + 3]));
  } else {
    const float* xg = xbase(p, kp) + t0 * D;
    const float* ag = xattn(p, kp) + t0 * D;
    const float* fg = xffn(p, kp, 0) + t0 * D;
    const int xst = p.xstride;
    const bool with_f = src == SRC_RES;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + FK_CONSUMERS * u;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < tot) {
        const int t = e >= nq ? 1 : 0;
        const int o = t * D + plane_first(e - t * nq, D);
        float4 cv[2 + FK_KC];
        cv[0] = ldcg4(xg + o);
        cv[1] = ldcg4(ag + o);
#pragma unroll
        for (int k = 0; k < FK_KC; ++k) cv[2 + k] = with_f ? ldcg4(fg + k * xst + o) : make_float4(0.f, 0.f, 0.f, 0.f);
        v = cv[0];
#pragma unroll
        for (int k = 1; k < 2 + FK_KC; ++k) {
          v.x += cv[k].x; v.y += cv[k].y; v.z += cv[k].z; v.w += cv[k].w;
        }
      }
      xv[u] = v;
    }
  }
  float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int e = tid + FK_CONSUMERS * u;
    const float v = xv[u].x * xv[u].x + xv[u].y * xv[u].y + xv[u].z * xv[u].z + xv[u].w * xv[u].w;
    if (e >= nq) ss1 += v; else ss0 += v;
  }
  ss0 = warp_sum(ss0);
  ss1 = warp_sum(ss1);
  FK_MARK(TR_SUB, 2);
  if (clane() == 0) {
    fk_sm()->red[0][cwarp()] = ss0;
    fk_sm()->red[1][cwarp()] = ss1;
  }
  int lo, hi;
  cta_slice(sd, lo, hi);
  if (fold >= 0) {
    float* fb = xbase(p, fold);
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + FK_CONSUMERS * u;
      if (e < tot) {
        const int t = e >= nq ? 1 : 0, i = plane_first(e - t * nq, D);
        if (i + 3 >= lo && i < hi) {
          const float vals[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (i + q >= lo && i + q < hi) fb[t * D + i + q] = vals[q];
        }
      }
    }
  }
  float4 y[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int e = tid + FK_CONSUMERS * u;
    if (e < tot) {
      const int t = e >= nq ? 1 : 0;
      const float4 gv = gain4<WT>(g, plane_first(e - t * nq, D));
      y[u] = make_float4(xv[u].x * gv.x, xv[u].y * gv.y, xv[u].z * gv.z, xv[u].w * gv.w);
      reinterpret_cast<float4*>(xs)[e] = y[u];
    }
  }
  consumer_sync();
  if (out) {
    const float iv = norm_inv(0, sd);
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = tid + FK_CONSUMERS * u;
      if (e < nq) {
        const int i = plane_first(e, D);
        if (i + 3 >= lo && i < hi) {
          const float vals[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (i + q >= lo && i + q < hi) out[i + q] = vals[q] * iv;
        }
      }
    }
  }
  FK_MARK(TR_NORM, 0);
}

// Writes a raw vector (natural order, D floats at src) into xs token t (plane layout).
__device__ __forceinline__ void put_plane(float* xs_t, int D, int i, float v) {
  const int j = i >> 3, r = i & 7;
  xs_t[r < 4 ? 4 * j + r : (D >> 1) + 4 * j + (r - 4)] = v;
}

// ----------------------------------------------- q/k head normalisation

// One warp: v (hd elements, lane holds l + 32 j) <- RoPE(RMSNorm(v) * g) with
// gains g (shared memory) and the rotation of shared-memory rope row `rr`.
template <class WT>
__device__ __forceinline__ void norm_rope_head(const FKParams& p, const FKSmem* sm, float (&v)[4],
                                               const WT* g, int rr, int lane) {
  const int hd = p.hd, J = hd / 32;
  if (p.qk_norm) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < J) ss = fmaf(v[j], v[j], ss);
    ss = warp_sum(ss);
    const float inv = rsqrtf(fmaf(ss, sm->plan.inv_hd, p.eps));
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < J) v[j] = v[j] * inv * to_f(g[lane + 32 * j]);
  }
  // rotate-half pairs (i, i + hd/2): (v0, v2), (v1, v3) for hd = 128; (v0, v1) for hd = 64
  const float c0 = sm->rope_c[rr][lane], s0 = sm->rope_s[rr][lane];
  if (J == 4) {
    const float c1 = sm->rope_c[rr][lane + 32], s1 = sm->rope_s[rr][lane + 32];
    const float a0 = v[0], a2 = v[2], a1 = v[1], a3 = v[3];
    v[0] = a0 * c0 - a2 * s0;
    v[2] = a2 * c0 + a0 * s0;
    v[1] = a1 * c1 - a3 * s1;
    v[3] = a3 * c1 + a1 * s1;
  } else {
    const float a0 = v[0], a1 = v[1];
    v[0] = a0 * c0 - a1 * s0;
    v[1] = a1 * c0 + a0 * s0;
  }
}

// Row of the shared-memory rope table for a position: CodePredictor positions
// map to themselves, the Talker position to row 16.
__device__ __forceinline__ int cp_rope_row(int pos) { return pos; }
constexpr int TALKER_ROPE_ROW = 16;

// ------------------------------------------------------------ the sampler

// Draws code j of the frame (0: semantic from the pending Talker logits; 1..15:
// acoustic from the last CodePredictor head, whose words carry tag ltag) in
// every CTA, identically.  The logits are staged in shared memory (the
// sampler turns them into keys in place).  Returns the code fed forward (the
// forced code under teacher forcing).
__device__ __noinline__ int draw_code(Cons c, int j, uint32_t ltag) {
  const FKParams& p = *fk_prm();
  const bool sem = j == 0;
  const int V = sem ? p.Vt : p.Vc;
  float* lv = reinterpret_cast<float*>(fk_sm()->u.smp.keys);
  {
    // float4 q of thread t: elements 4 (t + FK_CONSUMERS q) .. + 3 (V % 4 == 0)
    const float* pl = p.pending_logits + (size_t)p.sid * p.Vt;
    float4 v[FAST_V4];
    if (sem) {
#pragma unroll
      for (int q = 0; q < FAST_V4; ++q) {
        const int e = 4 * (ctid() + FK_CONSUMERS * q);
        if (e < V) v[q] = ldcg4(pl + e);
      }
    } else {
      uint64_t raw[4 * FAST_V4];
      int off[4 * FAST_V4];
#pragma unroll
      for (int q = 0; q < FAST_V4; ++q) {
        const int e = 4 * (ctid() + FK_CONSUMERS * q);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          off[4 * q + k] = e < V ? e + k : 0;
          raw[4 * q + k] = e < V ? ld_relaxed64(p.cp_logits + e + k) : tag_filler(ltag);
        }
      }
      tag_resolve<4 * FAST_V4>(raw, p.cp_logits, off, ltag);
#pragma unroll
      for (int q = 0; q < FAST_V4; ++q)
        v[q] = make_float4(tag_float(raw[4 * q]), tag_float(raw[4 * q + 1]), tag_float(raw[4 * q + 2]),
                           tag_float(raw[4 * q + 3]));
    }
    float* dump = p.dump && ccta() == 0 ? p.dump + (sem ? 0 : p.Vt + (j - 1) * p.Vc) : nullptr;
    // special semantic codes other than the end-of-stream code are never
    // drawn (the dump keeps the raw logits)
    const int sf = sem ? p.sp.special_from : 0;
#pragma unroll
    for (int q = 0; q < FAST_V4; ++q) {
      const int e = 4 * (ctid() + FK_CONSUMERS * q);
      if (e < V) {
        if (dump) *reinterpret_cast<float4*>(dump + e) = v[q];
        if (sf > 0) {
          float* f = reinterpret_cast<float*>(&v[q]);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (e + k >= sf && e + k != p.sp.eos_token) f[k] = -INFINITY;
        }
        *reinterpret_cast<float4*>(lv + e) = v[q];
      }
    }
  }
  consumer_sync();
  int code = fast_sample<ConsGroup>(fk_sm()->u.smp, lv, V, sem ? p.sp.do_sample : p.sp.sub_do_sample,
                                    sem ? p.sp.top_k : p.sp.sub_top_k, sem ? p.sp.top_p : p.sp.sub_top_p,
                                    sem ? p.sp.temperature : p.sp.sub_temperature,
                                    sem ? p.sp.repetition_penalty : 1.0f,
                                    sem ? p.history + (size_t)p.sid * p.Vt : nullptr, fk_sm()->uni[j]);
  FK_MARK(TR_SUB, 7);  // (draw done)
  code = min(max(code, 0), V - 1);
  int fed = code;
  if (p.forced) {
    fed = fk_sm()->forced[j];
    if (fed < 0 || fed >= V) {
      if (ccta() == 0 && ctid() == 0) atomicCAS(p.err, 0, Q3TTS_ERR_ARG);
      fed = code;
    }
  }
  // codes out (CTA 0, thread 0 alone): a finished stream writes -1; the frame
  // that feeds the end-of-stream code keeps its semantic code and ends the
  // stream.  The frame itself is computed either way.
  if (ccta() == 0 && ctid() == 0) {
    FKSmem* sm = fk_sm();
    if (sem) {
      const bool before = p.finished[p.sid] != 0;
      const bool eos = p.sp.eos_token >= 0 && fed == p.sp.eos_token;
      sm->fin_state = before ? 2 : (eos ? 1 : 0);
      if (eos && !before) p.finished[p.sid] = 1;
      p.codes[0] = before ? -1 : code;
    } else {
      p.codes[j] = sm->fin_state ? -1 : code;
    }
  }
  return fed;
}

// Gains of the current layer inside its side slot.
template <class WT>
__device__ __forceinline__ const WT* side_cur(Cons c) {
  return reinterpret_cast<const WT*>(fk_sm()->side[cst().layer & 1]);
}
template <class WT>
__device__ __forceinline__ const WT* side_gq(Cons c, int D) { return side_cur<WT>(c) + 2 * D; }
template <class WT>
__device__ __forceinline__ const WT* side_gk(Cons c, int D) { return side_cur<WT>(c) + 2 * D + fk_prm()->hd; }

// ---------------------------------------------------------------- phases

// o_proj is cut into tiles of 32 output columns of one head.  A tile is
// stored lane-interleaved, [hd/8][32][8]: lane l's 8 weights of hd block kb
// (column 32 j + l of W_o, inputs h hd + 8 kb ..) sit at (kb 32 + l) 8, so a
// warp reads a tile with conflict-free 16-byte loads and every lane owns one
// output column -- no cross-lane reduction.  The CTA's tiles are [t0, t1)
// of Hq * ceil(D / 32) (the plan's op_t0, op_t1 for stack s).
__device__ __forceinline__ int oproj_nt(int D) { return (D + 31) >> 5; }

// The CTA's o_proj tiles, one per ring chunk and private to a warp, against
// the attention outputs of the CTA's (<= 2) heads (os, plane layout) for T
// tokens; lane l owns column 32 j + l of its tile, and each column's sum is
// added into xattn(k).  Closes the attention phase of layer k with a grid
// barrier.
template <class WT>
__device__ __forceinline__ void oproj_step(Cons c, int D, int sd, int T, int k, const float* so) {
  const FKParams& p = *fk_prm();
  Stream s = stream_begin(c);
  const int hd = p.hd, nt = oproj_nt(D), nkb = hd >> 3;
  const int t0 = fk_sm()->plan.op_t0[sd], t1 = fk_sm()->plan.op_t1[sd];
  const int h_first = fk_sm()->plan.op_h0[sd];
  float* XA = xattn(p, k);
  const uint32_t os0 = soff(fk_sm()->os[0][0]);
  constexpr uint32_t OS_HEAD = FK_TMAX * FK_HDMAX * 4, OS_TOK = FK_HDMAX * 4;
  const uint32_t n0 = cst().n;
  const uint32_t nch = t1 > t0 ? (uint32_t)(t1 - t0) : 0u;
  for (uint32_t n = first_chunk(n0, s.warp); n < n0 + nch; n += FK_CONSUMER_WARPS) {
    const uint32_t buf = chunk_wait(s, n);
    // head of tile ti: floor((ti + 0.5) / nt) in float is exact here (ti < 16 nt, nt <= 64)
    const int ti = t0 + (int)(n - n0), h = (int)(((float)ti + 0.5f) * fk_sm()->plan.inv_nt[sd]);
    const int col = (ti - h * nt) * 32 + s.lane;
    const uint32_t w = buf + (uint32_t)(s.lane * 8 * (int)sizeof(WT));
    float sc = 1.f;
    if constexpr (kFp8<WT>) sc = col < D ? __ldg(so + col) : 0.f;  // W_o row (output column) scale
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
      const uint32_t xo = os0 + (uint32_t)(h - h_first) * OS_HEAD + (uint32_t)t * OS_TOK;
      float u = 0.f, v = 0.f;
#pragma unroll 4
      for (int kb = 0; kb < nkb; ++kb)
        fma8<WT>(w + (uint32_t)(kb * 256 * (int)sizeof(WT)), lds_f4(xo + (uint32_t)(kb * 16)),
                 lds_f4(xo + (uint32_t)(2 * hd + kb * 16)), u, v);
      if (col < D) atomicAdd(XA + t * D + col, (u + v) * sc);
    }
    release_private(s, n);
  }
  warp_set(cst().aborted, s.aborted ? 1 : 0);
  warp_set(cst().n, n0 + nch);
  grid_sync(c);
}

// Stores a warp's head vector (lane holds l + 32 j) into plane layout.
__device__ __forceinline__ void store_head_plane(float* dst, int hd, const float* v, int lane) {
  for (int j = 0; j < hd / 32; ++j) put_plane(dst, hd, lane + 32 * j, v[j]);
}

// CodePredictor phase B: attention of the CTA's one or two heads for each of
// the pass's tokens over positions 0..pos0+t (at most 16), then o_proj.
// Warp w takes positions w and w + 8: their cached K/V rows are loaded first,
// into registers, so that the loads are in flight while the q and current k
// rows are resolved; per-warp partial softmax sums are combined across warps.
// The CTA owning column 0 of the first q head of a kv group appends that
// group's current k, v to the cache.  The loops over pairs and positions are
// not unrolled: this phase runs once per layer and pass, and its code has to
// stay in the instruction cache with the rest of the pass.
template <class WT>
__device__ __forceinline__ void phase_cp_attn(Cons c, int layer, int T, int pos0, int k, uint32_t qtag) {
  const FKParams& p = *fk_prm();
  const FKPlan& pl = fk_sm()->plan;
  const int D = p.Dc, hd = p.hd, Hq = p.Hq, Hkv = p.Hkv, rs = pl.rep_shift, rep = 1 << rs, J = hd >> 5;
  const int nt = oproj_nt(D), ts = T - 1;  // tokens of the pass: 1 or 2 (shift ts)
  const int v0 = pl.op_t0[0], v1 = pl.op_t1[0];  // the CTA's o_proj tiles
  const int h_first = pl.op_h0[0], h_last = pl.op_h1[0];
  const int nh = v1 > v0 ? h_last - h_first + 1 : 0;
  const int npair = nh * T;
  const int g_first = h_first >> rs;
  const int ng = nh ? (h_last >> rs) - g_first + 1 : 0;  // kv groups touched (<= 2)
  const int gs = ng > 1 ? 1 : 0;
  AttnScratch& as = fk_sm()->u.att;
  const float scale = pl.attn_scale;
  const int w = cwarp(), lane = clane();
  const float* ckb = (const float*)p.ckv.pool + ckv_base(p, layer, 0, g_first);  // group g_first, k, position 0
  const int gstride = p.ckv.page_size * hd, vstride = Hkv * gstride;  // next kv group; k -> v
  // 0) cached k, v rows of positions w, w + 8 (< pos0) of the touched groups
  float kk[2][2][4], vv[2][2][4];
#pragma unroll
  for (int np = 0; np < 2; ++np) {
    const int sp = w + FK_CONSUMER_WARPS * np;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const bool cached = sp < pos0 && gi < ng;
      const float* kc = ckb + (cached ? gi * gstride + sp * hd : 0);
      const float* vc = kc + vstride;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        kk[np][gi][j] = cached && j < J ? __ldcg(kc + lane + 32 * j) : 0.f;
        vv[np][gi][j] = cached && j < J ? __ldcg(vc + lane + 32 * j) : 0.f;
      }
    }
  }
  // 1) q of each (head, token) pair, normalised and rotated (warps < npair);
  //    the k and v of the pass's positions, one (token, kv group) per warp
  //    from warp 4 on, k normalised and rotated; both kept in shared memory.
  //    The CTA owning the first o_proj tile of the group appends k and v.
  {
    const bool isq = w < npair, isk = w >= FK_CONSUMER_WARPS - FK_PAIRS && w - (FK_CONSUMER_WARPS - FK_PAIRS) < T * ng;
    if (isq || isk) {
      const int it = w - (FK_CONSUMER_WARPS - FK_PAIRS);
      const int t = isq ? (w & ts) : it >> gs, gi = isq ? 0 : (it & gs);
      const int h = h_first + (w >> ts), g = g_first + gi;
      const int so = t * p.qkv_rows + (isq ? h * hd : (Hq + g) * hd) + lane;
      const int vo = t * p.qkv_rows + (Hq + Hkv + g) * hd + lane;
      const bool app = isk && g * rep * nt >= v0 && g * rep * nt < v1;  // this CTA appends k, v
      uint64_t raw[8];  // the q or k row, then (for a k job) the v row
      int off[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        off[j] = so + 32 * j;
        off[4 + j] = vo + 32 * j;
        raw[j] = j < J ? ld_relaxed64(p.qkv + so + 32 * j) : tag_filler(qtag);
        raw[4 + j] = (j < J && isk) ? ld_relaxed64(p.qkv + vo + 32 * j) : tag_filler(qtag);
      }
      tag_resolve<8>(raw, p.qkv, off, qtag);
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = j < J ? tag_float(raw[j]) : 0.f;
      norm_rope_head(p, fk_sm(), v, isq ? side_gq<typename GainOf<WT>::T>(c, D) : side_gk<typename GainOf<WT>::T>(c, D),
                     cp_rope_row(pos0 + t), lane);
      float* dst = isq ? as.q[w] : as.kcur[it];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < J) dst[lane + 32 * j] = v[j];
      if (isk) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < J) as.vcur[it][lane + 32 * j] = tag_float(raw[4 + j]);
      }
      if (app) {
        float* kc = const_cast<float*>(ckb) + gi * gstride + (pos0 + t) * hd;
        float* vc = kc + vstride;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < J) {
            kc[lane + 32 * j] = v[j];
            vc[lane + 32 * j] = tag_float(raw[4 + j]);
          }
      }
    }
  }
  FK_MARK(TR_SUB, 3);
  consumer_sync();
  FK_MARK(TR_SUB, 4);
  // 2) per-warp partial softmax over its positions, for every pair
#pragma unroll 1
  for (int pr = 0; pr < npair; ++pr) {
    const int h = h_first + (pr >> ts), t = pr & ts, gsel = (h >> rs) - g_first;
    float m = -INFINITY, l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int np = 0; np < 2; ++np) {
      const int sp = w + FK_CONSUMER_WARPS * np;
      if (sp > pos0 + t) break;  // causal (and sp < S)
      float kr[4], vr[4];
      if (sp < pos0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          kr[j] = np ? (gsel ? kk[1][1][j] : kk[1][0][j]) : (gsel ? kk[0][1][j] : kk[0][0][j]);
          vr[j] = np ? (gsel ? vv[1][1][j] : vv[1][0][j]) : (gsel ? vv[0][1][j] : vv[0][0][j]);
        }
      } else {
        const int ci = (sp - pos0) * ng + gsel;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          kr[j] = j < J ? as.kcur[ci][lane + 32 * j] : 0.f;
          vr[j] = j < J ? as.vcur[ci][lane + 32 * j] : 0.f;
        }
      }
      float d = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < J) d = fmaf(as.q[pr][lane + 32 * j], kr[j], d);
      d = warp_sum(d) * scale;
      const float mn = fmaxf(m, d), corr = __expf(m - mn), e = __expf(d - mn);
      l = l * corr + e;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = o[j] * corr + e * vr[j];
      m = mn;
    }
    if (lane == 0) { as.m[w][pr] = m; as.l[w][pr] = l; }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < J) as.o[w][pr][lane + 32 * j] = o[j];
  }
  FK_MARK(TR_SUB, 5);
  consumer_sync();
  // 3) combine the warps: thread (pair, d)
  for (int e = ctid(); e < npair * hd; e += FK_CONSUMERS) {
    const int pr = e >> pl.hd_shift, d = e & (hd - 1);
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < FK_CONSUMER_WARPS; ++q) M = fmaxf(M, as.m[q][pr]);
    float Ls = 0.f, Os = 0.f;
#pragma unroll
    for (int q = 0; q < FK_CONSUMER_WARPS; ++q) {
      const float f = as.m[q][pr] == -INFINITY ? 0.f : __expf(as.m[q][pr] - M);
      Ls += as.l[q][pr] * f;
      Os += as.o[q][pr][d] * f;
    }
    put_plane(fk_sm()->os[pr >> ts][pr & ts], hd, d, __fdividef(Os, Ls));  // Ls >= 1 (the max term)
  }
  consumer_sync();
  FK_MARK(TR_SUB, 6);
  oproj_step<WT>(c, D, 0, T, k, p.cl[layer].s_o);
}

// Talker phase B1: attention partials.  Work item = (kv group g, position
// chunk); the q heads of the group share the K/V reads.  The item holding the
// current position appends its k, v to the cache.
// J (1, 2 or 4) consecutive elements of a cache row, widened: one vector load.
template <class KT>
__device__ __forceinline__ void ld_kv(const KT* p, int J, float (&o)[4]);
template <>
__device__ __forceinline__ void ld_kv<float>(const float* p, int J, float (&o)[4]) {
  o[1] = o[2] = o[3] = 0.f;
  if (J == 4) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  } else if (J == 2) {
    const float2 a = *reinterpret_cast<const float2*>(p);
    o[0] = a.x; o[1] = a.y;
  } else {
    o[0] = *p;
  }
}
template <>
__device__ __forceinline__ void ld_kv<bf16>(const bf16* p, int J, float (&o)[4]) {
  o[1] = o[2] = o[3] = 0.f;
  if (J == 4) {
    const uint2 a = *reinterpret_cast<const uint2*>(p);
    o[0] = __uint_as_float(a.x << 16); o[1] = __uint_as_float(a.x & 0xffff0000u);
    o[2] = __uint_as_float(a.y << 16); o[3] = __uint_as_float(a.y & 0xffff0000u);
  } else if (J == 2) {
    const uint32_t a = *reinterpret_cast<const uint32_t*>(p);
    o[0] = __uint_as_float(a << 16); o[1] = __uint_as_float(a & 0xffff0000u);
  } else {
    o[0] = to_f(*p);
  }
}

// K and v rows of Talker positions sb and sb + 8 of kv group g, lane l holding
// elements J l .. J l + J - 1 of each (cached positions from the cache; the
// current position: v from the QKV rows and a zero key, which the caller
// replaces; beyond it: zeros).
template <class KT>
__device__ __forceinline__ void talker_kv_rows(const FKParams& p, int layer, int g, int pos, int sb, int J,
                                               uint32_t qtag, float (&k)[2][4], float (&v)[2][4]) {
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const int sp = sb + b * FK_CONSUMER_WARPS;
    if (sp < pos) {
      const KT* kc = (const KT*)p.tkv.pool + tkv_offset(p, layer, sp, 0, g) + J * clane();
      const KT* vc = (const KT*)p.tkv.pool + tkv_offset(p, layer, sp, 1, g) + J * clane();
      ld_kv<KT>(kc, J, k[b]);
      ld_kv<KT>(vc, J, v[b]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) k[b][j] = v[b][j] = 0.f;
      if (sp == pos) {  // v of the current position: the tagged QKV rows
        const int vo = (p.Hq + p.Hkv + g) * p.hd + J * clane();
        uint64_t raw[4];
        int off[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          off[j] = vo + j;
          raw[j] = j < J ? ld_relaxed64(p.qkv + vo + j) : tag_filler(qtag);
        }
        tag_resolve<4>(raw, p.qkv, off, qtag);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < J) v[b][j] = tag_float(raw[j]);
      }
    }
  }
}

template <class WT, class KT>
__device__ __forceinline__ void phase_talker_attn(Cons c, int layer, uint32_t qtag, uint32_t ptag) {
  const FKParams& p = *fk_prm();
  const FKPlan& pl = fk_sm()->plan;
  const int hd = p.hd, Hq = p.Hq, Hkv = p.Hkv, rep = 1 << pl.rep_shift, J = hd >> 5;
  const int cpg = pl.cpg, g = pl.tg, ch = pl.tch;
  const int pos = p.pos;
  AttnScratch& as = fk_sm()->u.att;
  const float scale = pl.attn_scale;
  if (g < Hkv) {
    const int s0 = fk_sm()->ta_s0, s1 = fk_sm()->ta_s1;
    constexpr int BATCH = 2;
    float k[BATCH][4], v[BATCH][4];
    // the warp's first K/V rows are loaded before step 1 (they do not depend
    // on it), so the loads are in flight while it runs
    talker_kv_rows<KT>(p, layer, g, pos, s0 + cwarp(), J, qtag, k, v);
    // q of the group's heads (warps < rep); the current key (warp rep, in
    // the item holding the current position), normalised, rotated, kept in
    // shared memory and appended to the cache with its v
    const bool isk = cwarp() == rep && pos >= s0 && pos < s1;
    if (cwarp() < rep || isk) {
      const int so = (isk ? (Hq + g) * hd : (g * rep + cwarp()) * hd) + clane();
      const int vo = (Hq + Hkv + g) * hd + clane();
      uint64_t raw[8];  // the q or k row, then (for the key) the v row
      int off[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        off[j] = so + 32 * j;
        off[4 + j] = vo + 32 * j;
        raw[j] = j < J ? ld_relaxed64(p.qkv + so + 32 * j) : tag_filler(qtag);
        raw[4 + j] = (j < J && isk) ? ld_relaxed64(p.qkv + vo + 32 * j) : tag_filler(qtag);
      }
      tag_resolve<8>(raw, p.qkv, off, qtag);
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = j < J ? tag_float(raw[j]) : 0.f;
      norm_rope_head(p, fk_sm(), v, isk ? side_gk<typename GainOf<WT>::T>(c, p.Dt) : side_gq<typename GainOf<WT>::T>(c, p.Dt),
                     TALKER_ROPE_ROW, clane());
      float* dst = isk ? as.kcur[0] : as.q[cwarp()];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < J) dst[clane() + 32 * j] = v[j];
      if (isk) {
        KT* kc = (KT*)p.tkv.pool + tkv_offset(p, layer, pos, 0, g);
        KT* vc = (KT*)p.tkv.pool + tkv_offset(p, layer, pos, 1, g);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < J) {
            kc[clane() + 32 * j] = from_f<KT>(v[j]);
            vc[clane() + 32 * j] = from_f<KT>(tag_float(raw[4 + j]));
          }
      }
    }
    consumer_sync();
    float m[FK_REPMAX], l[FK_REPMAX], o[FK_REPMAX][4];
#pragma unroll
    for (int r = 0; r < FK_REPMAX; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[r][j] = 0.f;
    }
    for (int sb = s0 + cwarp(); sb < s1; sb += BATCH * FK_CONSUMER_WARPS) {
      if (sb != s0 + cwarp()) talker_kv_rows<KT>(p, layer, g, pos, sb, J, qtag, k, v);
#pragma unroll
      for (int b = 0; b < BATCH; ++b)  // the current key comes from step 1
        if (sb + b * FK_CONSUMER_WARPS == pos) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j < J) k[b][j] = as.kcur[0][J * clane() + j];
        }
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        const int sp = sb + b * FK_CONSUMER_WARPS;
        if (sp < s1) {
#pragma unroll
          for (int r = 0; r < FK_REPMAX; ++r) {
            if (r < rep) {
              float d = 0.f;  // lane l: elements J l .. J l + J - 1
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (j < J) d = fmaf(as.q[r][J * clane() + j], k[b][j], d);
              d = warp_sum(d) * scale;
              const float mn = fmaxf(m[r], d), corr = __expf(m[r] - mn), e = __expf(d - mn);
              l[r] = l[r] * corr + e;
#pragma unroll
              for (int j = 0; j < 4; ++j) o[r][j] = o[r][j] * corr + e * v[b][j];
              m[r] = mn;
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < FK_REPMAX; ++r) {
      if (r < rep) {
        if (clane() == 0) {
          as.m[cwarp()][r] = m[r];
          as.l[cwarp()][r] = l[r];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < J) as.o[cwarp()][r][J * clane() + j] = o[r][j];
      }
    }
    consumer_sync();
    for (int e = ctid(); e < rep * hd; e += FK_CONSUMERS) {
      const int r = e >> pl.hd_shift, d = e & (hd - 1);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < FK_CONSUMER_WARPS; ++w) M = fmaxf(M, as.m[w][r]);
      float Ls = 0.f, Os = 0.f;
      if (M > -INFINITY) {
#pragma unroll
        for (int w = 0; w < FK_CONSUMER_WARPS; ++w) {
          const float f = as.m[w][r] == -INFINITY ? 0.f : __expf(as.m[w][r] - M);
          Ls += as.l[w][r] * f;
          Os += as.o[w][r][d] * f;
        }
      }
      uint64_t* dst = p.part + ((size_t)(g * rep + r) * cpg + ch) * (hd + 2);
      st_tagged(dst + 2 + d, Os, ptag);
      if (d == 0) {
        st_tagged(dst, M, ptag);
        st_tagged(dst + 1, Ls, ptag);
      }
    }
  }
  // no grid barrier: the combine reads the partials by their tag
}

// Talker phase B2: combine the partials of the CTA's heads (all partial loads
// of a thread issued together), then o_proj.
template <class WT>
__device__ __forceinline__ void phase_talker_oproj(Cons c, int k, uint32_t ptag, int l) {
  const FKParams& p = *fk_prm();
  const FKPlan& pl = fk_sm()->plan;
  const int D = p.Dt, hd = p.hd, cpg = pl.cpg;
  const int v0 = pl.op_t0[1], v1 = pl.op_t1[1];  // the CTA's o_proj tiles
  const int h_first = pl.op_h0[1], h_last = pl.op_h1[1];
  const int nh = v1 > v0 ? h_last - h_first + 1 : 0;
  // warp-cooperative: thread (hh, d) = ctid() of the CTA's nh heads (whole
  // warps, as hd is a multiple of 32); lane c of a warp reads chunk c's
  // (m, l) header and the warp reduces them, then every lane reads its d of
  // the chunks' partial outputs, weighted by the header weights it gets by
  // shuffle
  const int e = ctid();
  if (e < nh * hd) {
    const int hh = e >> pl.hd_shift, d = e & (hd - 1), lane = clane();
    const uint64_t* base = p.part + (size_t)(h_first + hh) * cpg * (hd + 2);
    float M = -INFINITY;
    for (int c0 = 0; c0 < cpg; c0 += 32) {
      const bool in = c0 + lane < cpg;
      uint64_t raw[1];
      const int off[1] = {(in ? c0 + lane : 0) * (hd + 2)};
      raw[0] = in ? ld_relaxed64(base + off[0]) : tag_filler(ptag);
      tag_resolve<1>(raw, base, off, ptag);
      M = fmaxf(M, warp_max(in ? tag_float(raw[0]) : -INFINITY));
    }
    float L = 0.f, O = 0.f;
    for (int c0 = 0; c0 < cpg; c0 += 32) {
      const bool in = c0 + lane < cpg;
      uint64_t raw[2];
      const int o = (in ? c0 + lane : 0) * (hd + 2);
      const int off[2] = {o, o + 1};
      raw[0] = in ? ld_relaxed64(base + o) : tag_filler(ptag);
      raw[1] = in ? ld_relaxed64(base + o + 1) : tag_filler(ptag);
      tag_resolve<2>(raw, base, off, ptag);
      const float m = in ? tag_float(raw[0]) : -INFINITY;
      const float f = m == -INFINITY ? 0.f : __expf(m - M);
      L += warp_sum(in ? tag_float(raw[1]) * f : 0.f);
      const int nc = min(32, cpg - c0);
      for (int cb = 0; cb < nc; cb += 8) {
        uint64_t ro[8];
        int oo[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const bool iq = cb + q < nc;
          oo[q] = (iq ? c0 + cb + q : 0) * (hd + 2) + 2 + d;
          ro[q] = iq ? ld_relaxed64(base + oo[q]) : tag_filler(ptag);
        }
        tag_resolve<8>(ro, base, oo, ptag);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float fq = __shfl_sync(0xffffffffu, f, (cb + q) & 31);
          if (cb + q < nc) O = fmaf(fq, tag_float(ro[q]), O);
        }
      }
    }
    put_plane(fk_sm()->os[hh][0], hd, d, __fdividef(O, L));  // L >= 1 (the max term)
  }
  consumer_sync();
  oproj_step<WT>(c, D, 1, 1, k, p.tl[l].s_o);  // the Talker's stack, one token
}

// Units u0 .. u0 + G - 1 of a chunk that holds the gate rows of U units and
// then their up rows: a_{f,t} = silu(gate_f . y_t / rms_t) * (up_f . y_t /
// rms_t) into act[t][a0 + u] (lane u T + t writes one).
template <class WT, int T, int G>
__device__ __forceinline__ void ffn_units(uint32_t buf, int rb, int U, int u0, int D, uint32_t xs, int lane,
                                          const float (&inv)[T], float (*act)[FK_UMAX], int a0, const float* sgu,
                                          int F, int f0, int nv) {
  uint32_t ro[2 * G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    ro[2 * g] = (uint32_t)((u0 + g) * rb);
    ro[2 * g + 1] = (uint32_t)((U + u0 + g) * rb);
  }
  float acc[2 * G][T];
  dots<WT, T, 2 * G>(buf, ro, D, xs, lane, acc);
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int t = 0; t < T; ++t)
      if (lane == g * T + t && g < nv) {  // units past nv: computed on other bytes of shared memory, not kept
        float gs = 1.f, us = 1.f;
        if constexpr (kFp8<WT>) {  // gate row f and up row F + f of W_gateup
          gs = __ldg(sgu + f0 + a0 + u0 + g);
          us = __ldg(sgu + F + f0 + a0 + u0 + g);
        }
        act[t][a0 + u0 + g] = silu(acc[2 * g][t] * inv[t] * gs) * (acc[2 * g + 1][t] * inv[t] * us);
      }
}

// The down projection of the CTA's FFN units [f0, f1): shared chunks of
// W_down^T rows from ring position n0; lane l of warp w owns output columns
// 8 (32 w + l) .. + 7, accumulates a_{f,t} W_down[:, f] over the units in
// registers and adds the CTA's partial sums into copy CTA % FK_KC of
// xffn(k) with float4 atomics.
template <class WT, int T>
__device__ __forceinline__ void ffn_down(Stream& s, int D, int f0, int f1, int rpc, uint32_t nd, uint32_t n0, int k,
                                         const float* sd) {
  const FKParams& p = *fk_prm();
  const float(*act)[FK_UMAX] = fk_sm()->act;
  const int rb = D * (int)sizeof(WT);
  const int col = (s.warp * 32 + s.lane) * 8;  // the lane's first output column
  const bool active = col < D;
  float y[T][8];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int k = 0; k < 8; ++k) y[t][k] = 0.f;
  for (uint32_t n = n0; n < n0 + nd; ++n) {
    const uint32_t buf = chunk_wait(s, n);
    const int fb = f0 + (int)(n - n0) * rpc, R = min(rpc, f1 - fb);
    if (active) {
      const uint32_t w = buf + (uint32_t)(col * (int)sizeof(WT));
      if (R == 4) {  // a full chunk of four rows: every load first, then the multiplies
        float d8[4][8], a[4][T];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          lds_w8<WT>(w + (uint32_t)(r * rb), d8[r]);
#pragma unroll
          for (int t = 0; t < T; ++t) a[r][t] = act[t][fb - f0 + r];
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int t = 0; t < T; ++t)
#pragma unroll
            for (int k = 0; k < 8; ++k) y[t][k] = fmaf(a[r][t], d8[r][k], y[t][k]);
      } else {
        for (int r = 0; r < R; ++r) {
          float d8[8];
          lds_w8<WT>(w + (uint32_t)(r * rb), d8);
#pragma unroll
          for (int t = 0; t < T; ++t) {
            const float a = act[t][fb - f0 + r];
#pragma unroll
            for (int k = 0; k < 8; ++k) y[t][k] = fmaf(a, d8[k], y[t][k]);
          }
        }
      }
    }
    release_shared(s, n);
  }
  warp_set(cst().aborted, s.aborted ? 1 : 0);
  warp_set(cst().n, n0 + nd);
  if (active && nd) {
    if constexpr (kFp8<WT>) {  // W_down row (output column) scales
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float sc = __ldg(sd + col + q);
#pragma unroll
        for (int t = 0; t < T; ++t) y[t][q] *= sc;
      }
    }
    float* X = xffn(p, k, ccta() % FK_KC);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      atomicAdd(reinterpret_cast<float4*>(X + t * D + col), make_float4(y[t][0], y[t][1], y[t][2], y[t][3]));
      atomicAdd(reinterpret_cast<float4*>(X + t * D + col + 4), make_float4(y[t][4], y[t][5], y[t][6], y[t][7]));
    }
  }
}

// FFN units of the CTA whose gate and up rows share one ring chunk.
__device__ __forceinline__ int units_per_chunk(int row_bytes) {
  const int u = FK_STAGE / (2 * row_bytes);
  return u < 1 ? 1 : (u > FK_RMAX / 2 ? FK_RMAX / 2 : u);
}

// Phase C of layer k: x_k + a_k staged for RMSNorm, then the CTA's FFN
// units [f0, f1) (split-K over the FFN width) in two streams.  First the gate
// and up rows: a private chunk holds the gate rows of U units and then their
// up rows, and its warp forms a_{f,t} = silu(gate_f . y_t / rms_t) *
// (up_f . y_t / rms_t) into act.  After one block-wide barrier, the rows of the
// transposed down projection W_down^T[f] (shared chunks): lane l of warp w
// owns output columns 8 (32 w + l) .. + 7 and adds a_{f,t} W_down[:, f] over
// the CTA's units in registers.  The CTA's partial D-vector goes into copy
// CTA % FK_KC of xffn(k) with float4 atomics.  The CTA also clears its slice
// of layer k + 1's deltas (see xbase).
template <class WT>
__device__ __forceinline__ void phase_ffn(Cons c, int sd, int T, int k, const LayerDev* lw) {
  using GT = typename GainOf<WT>::T;
  const FKParams& p = *fk_prm();
  const FKPlan& pl = fk_sm()->plan;
  const int D = sd ? p.Dt : p.Dc, F = sd ? p.Ft : p.Fc;
  load_norm<GT>(c, SRC_RES_A, k, 0u, 0, T, D, sd, side_cur<GT>(c) + D, -1, nullptr);
  side_end(c);
  const float inv0 = norm_inv(0, sd), inv1 = T > 1 ? norm_inv(1, sd) : 0.f;
  const int f0 = pl.ffn[sd].lo, f1 = pl.ffn[sd].hi;
  const int rb = D * (int)sizeof(WT);
  const int upc = pl.upc[sd];
  FKSmem* sm = fk_sm();
  const uint32_t xs = soff(sm->u.g.xs);
  Stream s = stream_begin(c);
  uint32_t n0 = cst().n;
  const uint32_t nch = (uint32_t)pl.ffn[sd].nch;
  for (uint32_t n = first_chunk(n0, s.warp); n < n0 + nch; n += FK_CONSUMER_WARPS) {
    const uint32_t buf = chunk_wait(s, n);
    const int fb = f0 + (int)(n - n0) * upc, U = min(upc, f1 - fb);
    // the chunk holds the gate rows of units fb .. fb + U - 1, then their up rows
    // two units (their gate and up rows) at a time, an odd last unit alone
    int u = 0;
    if (T == 1) {
      const float inv[1] = {inv0};
#pragma unroll 1
      for (; u + 2 <= U; u += 2) ffn_units<WT, 1, 2>(buf, rb, U, u, D, xs, s.lane, inv, sm->act, fb - f0, lw->s_gu, F, f0, 2);
      if (u < U) ffn_units<WT, 1, 1>(buf, rb, U, u, D, xs, s.lane, inv, sm->act, fb - f0, lw->s_gu, F, f0, 1);
    } else {
      const float inv[2] = {inv0, inv1};
#pragma unroll 1
      for (; u + 2 <= U; u += 2) ffn_units<WT, 2, 2>(buf, rb, U, u, D, xs, s.lane, inv, sm->act, fb - f0, lw->s_gu, F, f0, 2);
      if (u < U) ffn_units<WT, 2, 1>(buf, rb, U, u, D, xs, s.lane, inv, sm->act, fb - f0, lw->s_gu, F, f0, 1);
    }
    release_private(s, n);
  }
  warp_set(cst().n, n0 + nch);
  n0 += nch;
  if (s.warp == (int)(n0 % FK_CONSUMER_WARPS)) {
    // the CTA's slice of layer k + 1's deltas is cleared here, by the warp
    // the next chunk would have gone to: the round-robin gave it the fewest
    // gate/up chunks, so it would wait below anyway
    int lo, hi;
    cta_slice(2, lo, hi);
    float* a1 = xattn(p, k + 1);
    float* f1 = xffn(p, k + 1, 0);
    for (int i = lo + s.lane; i < hi; i += 32) {
      a1[i] = 0.f;
#pragma unroll
      for (int q = 0; q < FK_KC; ++q) f1[q * p.xstride + i] = 0.f;
    }
  }
  consumer_sync();  // act complete
  if (T == 1)
    ffn_down<WT, 1>(s, D, f0, f1, pl.rpc[sd], (uint32_t)pl.ffn_nd[sd], n0, k, lw->s_d);
  else
    ffn_down<WT, 2>(s, D, f0, f1, pl.rpc[sd], (uint32_t)pl.ffn_nd[sd], n0, k, lw->s_d);
  grid_sync(c);
}

// The CodePredictor input token(s) of pass j into xs (plane layout, D_t wide):
// pass 0: [h_T, E_t[c0]]; pass j >= 1: E_cp[j-1][c_j].
// Eight consecutive weights from global memory as floats (16-byte aligned).
template <class WT>
__device__ __forceinline__ void ld8(const WT* src, float (&f)[8]);
template <>
__device__ __forceinline__ void ld8<bf16>(const bf16* src, float (&f)[8]) {
  const uint4 u = __ldcg(reinterpret_cast<const uint4*>(src));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void ld8<float>(const float* src, float (&f)[8]) {
  const float4 a = __ldcg(reinterpret_cast<const float4*>(src)), b = __ldcg(reinterpret_cast<const float4*>(src) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// Elements 8 b .. 8 b + 7 of a plane-layout vector of width D (D % 8 == 0).
__device__ __forceinline__ void put_plane8(float* xs_t, int D, int b, const float (&f)[8]) {
  *reinterpret_cast<float4*>(xs_t + 4 * b) = make_float4(f[0], f[1], f[2], f[3]);
  *reinterpret_cast<float4*>(xs_t + (D >> 1) + 4 * b) = make_float4(f[4], f[5], f[6], f[7]);
}

// Row `code` of embedding table j of the frame: j = 0 the Talker codec table,
// j >= 1 the CodePredictor table of codebook j (width D_t).
template <class WT>
__device__ __forceinline__ const WT* code_row(const FKParams& p, int j, int code) {
  return j == 0 ? (const WT*)p.e_codec + (size_t)code * p.Dt
                : (const WT*)p.cp_embeds + ((size_t)(j - 1) * p.Vc + code) * p.Dt;
}

// The CodePredictor input token(s) of pass j into xs (plane layout, D_t wide):
// pass 0: [h_T, E_t[c0]]; pass j >= 1: E_cp[j-1][c_j].
template <class WT>
__device__ __forceinline__ void cp_tokens(Cons c, int j, int fed) {
  const FKParams& p = *fk_prm();
  const int Dt = p.Dt;
  float* xs = fk_sm()->u.g.xs;
  using GT = typename GainOf<WT>::T;
  const GT* e = code_row<GT>(p, j, fed);
  for (int b = ctid(); b < (Dt >> 3); b += FK_CONSUMERS) {
    float f[8];
    ld8<GT>(e + 8 * b, f);
    put_plane8(j == 0 ? xs + Dt : xs, Dt, b, f);
    if (j == 0) {
      ld8<float>(p.pending_h + (size_t)p.sid * Dt + 8 * b, f);
      put_plane8(xs, Dt, b, f);
    }
  }
  consumer_sync();
}

// The Talker input of the next position: the fp32 sum of the frame's 16 code
// embeddings, E_t[c0] + E_cp[0][c1] + ... + E_cp[14][c15], added in that
// order, into xs (plane layout).  Every CTA forms the whole vector from the
// codes it drew (the row reads are independent of one another).  Rows are
// read 8 weights at a time: the kernel is only set up for D_t % 8 == 0 and
// 16-byte aligned embedding tables.
template <class WT>
__device__ __forceinline__ void talker_input(Cons c, int fed15) {
  using GT = typename GainOf<WT>::T;
  const FKParams& p = *fk_prm();
  const int Dt = p.Dt;
  float* xs = fk_sm()->u.g.xs;
  const int* fedc = fk_sm()->fedc;
  for (int b = ctid(); b < (Dt >> 3); b += FK_CONSUMERS) {
    float s[8];
    ld8<GT>(code_row<GT>(p, 0, fedc[0]) + 8 * b, s);
#pragma unroll 5
    for (int j = 1; j < Q3TTS_N_CODEBOOKS; ++j) {
      float f[8];
      ld8<GT>(code_row<GT>(p, j, j < Q3TTS_N_CODEBOOKS - 1 ? fedc[j] : fed15) + 8 * b, f);
#pragma unroll
      for (int k = 0; k < 8; ++k) s[k] += f[k];
    }
    put_plane8(xs, Dt, b, s);
  }
  consumer_sync();
}

// The frame's schedule as a sequence of steps.  Per CodePredictor pass j
// (0..14): DRAW (code j; embedding sum; input tokens), PROJ (when D_t != D_c),
// L_c x (QKV, CP_ATTN (+ o_proj), FFN), CP_HEAD.  Then DRAW (code 15; Talker
// input), L_t x (QKV, T_ATTN, T_OPROJ (combine + o_proj), FFN), T_HEAD.  Every step kind has one call
// site in the loop below, so each phase's code exists once.
enum StepKind { S_DRAW, S_PROJ, S_QKV, S_CP_ATTN, S_FFN, S_CP_HEAD, S_T_ATTN, S_T_OPROJ, S_T_HEAD };

struct Step {
  int kind, j, l;  // j: CodePredictor pass (15: Talker), l: layer
};

__device__ __forceinline__ int steps_per_pass(const FKParams& p) { return 2 + (p.has_proj ? 1 : 0) + 3 * p.Lc; }

// Steps of pass j (j < 15: CodePredictor pass j; 15: the Talker step).
__device__ __forceinline__ int pass_steps(const FKParams& p, int j) {
  return j < Q3TTS_N_CODEBOOKS - 1 ? steps_per_pass(p) : 2 + 4 * p.Lt;
}

// Step r of pass j.  The schedule position is kept as (pass, step) so that
// decoding it needs no division by a runtime value.
__device__ __forceinline__ Step decode_step(const FKParams& p, int j, int r) {
  Step st;
  st.j = j;
  st.l = 0;
  if (j < Q3TTS_N_CODEBOOKS - 1) {
    const int hp = p.has_proj ? 1 : 0;
    if (r == 0) {
      st.kind = S_DRAW;
    } else if (r <= hp) {
      st.kind = S_PROJ;
    } else if (r == steps_per_pass(p) - 1) {
      st.kind = S_CP_HEAD;
    } else {
      const int q = r - 1 - hp, w = q % 3;
      st.l = q / 3;
      st.kind = w == 0 ? S_QKV : (w == 1 ? S_CP_ATTN : S_FFN);
    }
  } else {
    if (r == 0) {
      st.kind = S_DRAW;
    } else if (r == 1 + 4 * p.Lt) {
      st.kind = S_T_HEAD;
    } else {
      const int q = r - 1, w = q & 3;
      st.l = q >> 2;
      st.kind = w == 0 ? S_QKV : (w == 1 ? S_T_ATTN : (w == 2 ? S_T_OPROJ : S_FFN));
    }
  }
  return st;
}

// Moves the warp's schedule position to the next step.
__device__ __forceinline__ void next_step(ConsState& L) {
  __syncwarp();
  const int j = L.j, k = L.k + 1, s = L.s + 1;
  const bool wrap = k >= pass_steps(*fk_prm(), j);
  __syncwarp();
  L.k = wrap ? 0 : k;
  L.j = wrap ? j + 1 : j;
  L.s = s;
  __syncwarp();
}

// DRAW step: draw code j; code 0..14 starts CodePredictor pass j (its input
// tokens), code 15 starts the Talker step (its input is the sum of the frame's
// 16 code embeddings).
template <class WT>
__device__ __forceinline__ void draw_step(Cons c, int j) {
  ConsState& L = cst();
  const int fed = draw_code(c, j, tag_of(L.s - 1));
  if (j == 0) warp_set(L.fed0, fed);
  if (ctid() == 0) fk_sm()->fedc[j] = fed;  // read in later steps, after barriers
  if (j < Q3TTS_N_CODEBOOKS - 1)
    cp_tokens<WT>(c, j, fed);
  else
    talker_input<WT>(c, fed);
  warp_set(L.src, (int)SRC_XS);
}

// Row-GEMV steps (QKV, PROJ, the heads): stage the input -- RMSNorm of the
// layer input (QKV, folding it into the next two residual buffers), of the
// stack output (heads), or the raw tokens already in xs (PROJ) -- then the
// CTA's rows, then (all but the last step of the frame) a grid barrier.
template <class WT>
__device__ __forceinline__ void rows_step(Cons c, const Step& st) {
  ConsState& L = cst();
  const FKParams& p = *fk_prm();
  const bool cp = st.j < Q3TTS_N_CODEBOOKS - 1;
  const int Tp = cp && st.j == 0 ? 2 : 1;  // tokens of the pass
  const uint32_t tag = tag_of(L.s);
  const int sd = cp ? 0 : 1;  // the stack
  const FKPlan& pl = fk_sm()->plan;
  int K, T, rpc;
  const FKRange* rg;
  RowsOut o;
  o.out = nullptr;
  o.out64 = nullptr;
  o.tag = tag;
  o.ts = 0;
  o.sc = nullptr;
  if (st.kind == S_QKV) {
    K = cp ? p.Dc : p.Dt;
    T = Tp;
    rg = &pl.qkv[sd];
    rpc = pl.rpc[sd];
    o.out64 = p.qkv;
    o.ts = p.qkv_rows;
    if constexpr (kFp8<WT>) o.sc = (cp ? p.cl : p.tl)[st.l].s_qkv;
  } else if (st.kind == S_PROJ) {
    K = p.Dt;
    T = Tp;
    rg = &pl.proj;
    rpc = pl.rpc[1];
    o.out64 = p.z;
    o.ts = p.Dc;
    o.sc = p.s_cp_proj;
  } else if (st.kind == S_CP_HEAD) {
    K = p.Dc;
    T = 1;
    rg = &pl.head[0];
    rpc = pl.rpc[0];
    o.out64 = p.cp_logits;
    if constexpr (kFp8<WT>) o.sc = p.s_cp_heads + (size_t)st.j * p.Vc;
  } else {
    K = p.Dt;
    T = 1;
    rg = &pl.head[1];
    rpc = pl.rpc[1];
    o.out = p.pending_logits + (size_t)p.sid * p.Vt;
    o.sc = p.s_head;
  }
  float inv0 = 1.f, inv1 = 1.f;  // the projection's input is not normed
  if (st.kind != S_PROJ) {
    using GT = typename GainOf<WT>::T;
    const GT* g;
    int src = SRC_RES, fold = -1, t0 = 0;
    const int k = (int)L.layer;  // QKV: this layer; heads: the layers done so far
    float* hout = nullptr;
    if (st.kind == S_QKV) {
      g = side_begin<GT>(c);
      FK_MARK(TR_SUB, 1);
      src = L.src;  // the raw tokens, the projection, or layer k - 1's residual
      fold = k;
    } else {
      g = reinterpret_cast<const GT*>(fk_sm()->fin) + (cp ? 0 : p.Dc);
      t0 = Tp - 1;
      if (!cp) hout = p.pending_h + (size_t)p.sid * p.Dt;
    }
    load_norm<GT>(c, src, k - 1, tag_of(L.s - 1), t0, T, K, sd, g, fold, hout);
    inv0 = norm_inv(0, sd);
    inv1 = T > 1 ? norm_inv(1, sd) : 0.f;
  }
  stream_rows<WT>(c, *rg, rpc, K, T, soff(fk_sm()->u.g.xs), o, inv0, inv1);
  FK_MARK(TR_SUB, 8);
  // no grid barrier after a row GEMV: its readers wait for the outputs' tags
  // (the Talker head is the frame's last step); the CTA's warps still meet,
  // since the next step reuses the staging area
  if (st.kind != S_T_HEAD) consumer_sync();
  FK_MARK(TR_SUB, 9);
  warp_set(L.src, st.kind == S_PROJ ? (int)SRC_Z : (int)SRC_RES);
}

// The consumer warps' schedule for one frame (steps above).  Loop state lives
// in the warp's shared-memory record (cst()).
template <class WT, class KT>
__device__ void consumer() {
  Cons c;
  {
    const FKParams& p = *fk_prm();
    FKSmem* sm = fk_sm();
    cst().n = 0;
    cst().phase = 0;
    cst().layer = 0;
    cst().aborted = false;
    if (ctid() < Q3TTS_N_CODEBOOKS) {
      sm->uni[ctid()] = p.uniforms[ctid()];
      sm->forced[ctid()] = p.forced ? p.forced[ctid()] : 0;
    }
    using GT = typename GainOf<WT>::T;
    GT* fin = reinterpret_cast<GT*>(sm->fin);
    for (int i = ctid(); i < p.Dc; i += FK_CONSUMERS) fin[i] = ((const GT*)p.cp_gfinal)[i];
    for (int i = ctid(); i < p.Dt; i += FK_CONSUMERS) fin[p.Dc + i] = ((const GT*)p.t_gfinal)[i];
    if (ccta() == 0 && ctid() == 0 && p.newpage >= 0)
      const_cast<int*>(p.tkv.page_table)[p.sid * p.tkv.pages_per_stream + (p.pos >> (__ffs(p.tkv.page_size) - 1))] = p.newpage;
    // the stream's page tables (the page entered this frame from the launch
    // parameters: CTA 0's store above need not be visible yet)
    const int tp = p.tkv.pages_per_stream;
    if (tp <= FK_MAXPAGES)
      for (int i = ctid(); i < tp; i += FK_CONSUMERS)
        sm->tpage[i] = (p.newpage >= 0 && i == (p.pos >> (__ffs(p.tkv.page_size) - 1))) ? p.newpage
                                                                         : p.tkv.page_table[p.sid * tp + i];
    if (ctid() == 0) {
      sm->cpage = p.ckv.page_table[p.sid * p.ckv.pages_per_stream];
      // this frame's Talker attention chunk of the CTA: positions [s0, s1)
      const FKPlan& gp = p.plan[ccta()];
      const int S = p.pos + 1, cs = (S + gp.cpg - 1) / gp.cpg;
      sm->ta_s0 = gp.tch * cs;
      sm->ta_s1 = min(S, sm->ta_s0 + cs);
    }
    // this CTA's plan row (read before any phase, after the barrier below)
    static_assert(sizeof(FKPlan) % 4 == 0 && sizeof(FKPlan) / 4 <= FK_CONSUMERS, "one plan word per consumer thread");
    if (ctid() < (int)(sizeof(FKPlan) / 4))
      reinterpret_cast<int*>(&sm->plan)[ctid()] = reinterpret_cast<const int*>(p.plan + ccta())[ctid()];
    // rope rows: CodePredictor positions 0..15 and the Talker position
    const int half = p.hd / 2;
    for (int e = ctid(); e < 17 * half; e += FK_CONSUMERS) {
      const int r = e / half, i = e % half, pos = r < 16 ? r : p.pos;
      sm->rope_c[r][i] = p.rope_cos[(size_t)pos * half + i];
      sm->rope_s[r][i] = p.rope_sin[(size_t)pos * half + i];
    }
  }
  consumer_sync();
#ifdef Q3TTS_TRACE
  if (ctid() == 0) fk_sm()->trace_n = 0;
  if (clane() == 0) fk_sm()->trace_wait[cwarp()] = 0;
#endif
  FK_MARK(TR_STEP, 15);
  ConsState& L = cst();
  warp_set(L.j, 0);
  warp_set(L.k, 0);
  warp_set(L.s, 0);
  warp_set(L.src, (int)SRC_XS);
  {
    // the frame's first layer finds its deltas cleared (later layers' are
    // cleared by the FFN phase before them); one grid barrier orders this
    // before any CTA adds into them
    const FKParams& p = *fk_prm();
    int lo, hi;
    cta_slice(2, lo, hi);
    float* a0 = xattn(p, 0);
    float* f0 = xffn(p, 0, 0);
    for (int i = lo + ctid(); i < hi; i += FK_CONSUMERS) {
      a0[i] = 0.f;
#pragma unroll
      for (int q = 0; q < FK_KC; ++q) f0[q * p.xstride + i] = 0.f;
    }
    grid_sync(c);
  }
  for (; L.j < Q3TTS_N_CODEBOOKS; next_step(L)) {
    const Step st = decode_step(*fk_prm(), L.j, L.k);
#ifdef Q3TTS_TRACE
    consumer_sync();  // (profiling builds) every warp's waits of the previous step are in
    if (ctid() == 0) {  // the previous step's largest ring wait of a warp, in units of 16 cycles
      long long w = 0;
      for (int q = 0; q < FK_CONSUMER_WARPS; ++q) w = max(w, fk_sm()->trace_wait[q] >> 4);
      fk_mark(TR_CW0, (int)(w > 0xffff ? 0xffff : w));
    }
    consumer_sync();
    if (clane() == 0) fk_sm()->trace_wait[cwarp()] = 0;
#endif
    FK_MARK(TR_STEP, st.kind | (st.j << 4) | (st.l << 9));
    const bool cp = st.j < Q3TTS_N_CODEBOOKS - 1;
    const int T = cp && st.j == 0 ? 2 : 1;
    switch (st.kind) {
      case S_DRAW:
        draw_step<WT>(c, st.j);
        break;
      case S_CP_ATTN:
        phase_cp_attn<WT>(c, st.l, T, st.j == 0 ? 0 : st.j + 1, (int)L.layer, tag_of(L.s - 1));
        break;
      case S_T_ATTN:
        phase_talker_attn<WT, KT>(c, st.l, tag_of(L.s - 1), tag_of(L.s));
        break;
      case S_T_OPROJ:
        phase_talker_oproj<WT>(c, (int)L.layer, tag_of(L.s - 1), st.l);
        break;
      case S_FFN:
        phase_ffn<WT>(c, cp ? 0 : 1, T, (int)L.layer, (cp ? fk_prm()->cl : fk_prm()->tl) + st.l);
        break;
      default:
        rows_step<WT>(c, st);
        break;
    }
  }
  {
    const FKParams& q = *fk_prm();
    if (ccta() == 0 && ctid() == 0) q.history[(size_t)q.sid * q.Vt + L.fed0] = 1;
    FK_MARK(TR_END, 0);
    consumer_sync();
    if (ctid() == 0) {
      __threadfence();
      if (atomicAdd(q.done, 1u) == (unsigned)q.ncta - 1) {
        *q.bar = 0u;
        *q.done = 0u;
      }
    }
  }
}

// ---------------------------------------------------------------- producer

// The frame's weight schedule for one CTA, walked twice: by the ring's
// producer (PF false: bulk copies into the ring, side blocks into their
// slots) and by the prefetch warp (PF true: the same chunks as L2 prefetches,
// at most FK_PF_AHEAD chunks ahead of the producer), so that HBM keeps
// streaming while the consumers sit in barriers, attention and draws, and the
// ring's copies hit L2.
template <class WT, bool PF>
struct Producer {
  const FKParams& p;
  FKSmem* sm;
  int cta;
  uint32_t n = 0;
  bool stop = false;
  uint64_t pol;

  __device__ Producer(const FKParams& pp, FKSmem* s, int c) : p(pp), sm(s), cta(c) {
    pol = l2_evict_first_policy();
  }

  // Waits (bounded) until slot s may be refilled with chunk n; false after an
  // abort or a timeout (the producer then stops issuing).
  __device__ bool wait_empty(int s) {
    const unsigned par = ((n / FK_NSTAGE) - 1) & 1u;
    long long t0 = clock64();
    unsigned it = 0;
    // the ring is full most of the time: wait suspended so this warp does
    // not take issue slots from the consumer warps of its scheduler
    while (!mbar_try_wait_sleep(&sm->empty[s], par, 2000)) {
      if ((++it & 15u) == 0 && (ld_volatile(p.abort_flag) || clock64() - t0 > p.wait_cycles)) {
        raise_abort(p, Q3TTS_ERR_TIMEOUT);
        stop = true;
        return false;
      }
    }
    return true;
  }

  // Prefetch mode: waits (bounded) until chunk n is at most FK_PF_AHEAD
  // chunks ahead of the producer; false to stop (an abort, or a producer that
  // no longer advances -- it reports the timeout itself).
  __device__ bool pf_gate_wait() {
    const volatile uint32_t* gate = &sm->pf_gate;
    long long t0 = clock64();
    unsigned it = 0;
    while (n >= *gate + (uint32_t)p.pf_ahead) {
      __nanosleep(256);
      if ((++it & 15u) == 0 && (ld_volatile(p.abort_flag) || clock64() - t0 > p.wait_cycles)) {
        stop = true;
        return false;
      }
    }
    return true;
  }

  __device__ void publish() {
    if (!PF) *(volatile uint32_t*)&sm->pf_gate = n;
  }

  __device__ void issue(const void* src, unsigned bytes) {
    if (stop) return;
    if (PF) {
      if (pf_gate_wait()) {
        prefetch_l2(src, bytes);
        n++;
      }
      return;
    }
    const int s = n % FK_NSTAGE;
    if (n >= (uint32_t)FK_NSTAGE && !wait_empty(s)) return;
    mbar_expect_tx(&sm->full[s], bytes);
    bulk_g2s(sm->ring[s], src, bytes, &sm->full[s], pol);
    n++;
    publish();
  }

  // One chunk from two sources (the gate rows and the up rows of a few FFN units).
  __device__ void issue2(const void* a, const void* b, unsigned bytes) {
    if (stop) return;
    if (PF) {
      if (pf_gate_wait()) {
        prefetch_l2(a, bytes);
        prefetch_l2(b, bytes);
        n++;
      }
      return;
    }
    const int s = n % FK_NSTAGE;
    if (n >= (uint32_t)FK_NSTAGE && !wait_empty(s)) return;
    mbar_expect_tx(&sm->full[s], 2 * bytes);
    bulk_g2s(sm->ring[s], a, bytes, &sm->full[s], pol);
    bulk_g2s(sm->ring[s] + bytes, b, bytes, &sm->full[s], pol);
    n++;
    publish();
  }

  int nlayers = 0;  // layers in the frame (15 CodePredictor passes, then the Talker)
  int side_last[2] = {-1, -1};  // last layer whose side block was copied into each slot

  __device__ const LayerDev& layer_at(int k) const {
    const int ncp = (Q3TTS_N_CODEBOOKS - 1) * p.Lc;
    return k < ncp ? sm->lay[p.Lt + k % p.Lc] : sm->lay[k - ncp];
  }

  // Side block of layer k into slot k & 1 (after the consumers freed it).
  __device__ void side(int k) {
    if (PF || stop || k >= nlayers) return;
    const int slot = k & 1;
    if (k >= 2) {
      const unsigned par = ((k >> 1) - 1) & 1u;
      long long t0 = clock64();
      unsigned it = 0;
      while (!mbar_try_wait_sleep(&sm->side_empty[slot], par, 2000)) {
        if ((++it & 15u) == 0 && (ld_volatile(p.abort_flag) || clock64() - t0 > p.wait_cycles)) {
          raise_abort(p, Q3TTS_ERR_TIMEOUT);
          stop = true;
          return;
        }
      }
    }
    const int ncp = (Q3TTS_N_CODEBOOKS - 1) * p.Lc;
    const int D = k < ncp ? p.Dc : p.Dt;
    const unsigned bytes = (unsigned)((2 * D + 2 * p.hd) * (int)sizeof(typename GainOf<WT>::T));
    mbar_expect_tx(&sm->side_full[slot], bytes);
    bulk_g2s(sm->side[slot], layer_at(k).side, bytes, &sm->side_full[slot], pol);
    side_last[slot] = k;
  }

  // The frame's weight schedule as a list of segments, each one matrix (or
  // matrix pair) of which the CTA streams its share: per CodePredictor pass
  // [projection], per layer [QKV rows, o_proj tiles, gate/up units, W_down^T
  // rows], head j; then the Talker's layers and its head.  One loop with two
  // copy sites walks it (the producer's code runs beside the consumers' on
  // every SM, so it is kept small).
  __device__ void run() {
    const int esz = (int)sizeof(WT);
    nlayers = (Q3TTS_N_CODEBOOKS - 1) * p.Lc + p.Lt;
    const int hp = p.has_proj ? 1 : 0;
    const int cp_seg = hp + 4 * p.Lc + 1;  // segments of a CodePredictor pass
    const int nseg = (Q3TTS_N_CODEBOOKS - 1) * cp_seg + 4 * p.Lt + 1;
    side(0);
    int layer = 0;  // layer of the frame the schedule is in
    for (int sg = 0; sg < nseg && !stop; ++sg) {
      // decode: pass j (15: the Talker), position q inside it
      int j = 0, q = sg;
      if (sg >= (Q3TTS_N_CODEBOOKS - 1) * cp_seg) {
        j = Q3TTS_N_CODEBOOKS - 1;
        q = sg - (Q3TTS_N_CODEBOOKS - 1) * cp_seg;
      } else {
        j = sg / cp_seg;
        q = sg - j * cp_seg;
      }
      const bool cp = j < Q3TTS_N_CODEBOOKS - 1;
      const int D = cp ? p.Dc : p.Dt, F = cp ? p.Fc : p.Ft;
      const int lq = cp ? q - hp : q;  // position within the layers (-1: projection)
      const char* base;
      const char* up = nullptr;  // gate/up segment: the up rows
      int N, rb;
      bool layer_end = false, one = false;  // one: one row (o_proj tile) per chunk
      if (cp && q < hp) {
        base = (const char*)p.cp_proj;
        N = p.Dc;
        rb = p.Dt * esz;
      } else if (lq >= 4 * (cp ? p.Lc : p.Lt)) {  // the head
        base = cp ? (const char*)p.cp_heads + (size_t)j * p.Vc * p.Dc * esz : (const char*)p.t_head;
        N = cp ? p.Vc : p.Vt;
        rb = D * esz;
      } else {
        const LayerDev& L = layer_at(layer);
        const int m = lq & 3;
        if (m == 0) {
          base = (const char*)L.w_qkv;
          N = p.qkv_rows;
          rb = D * esz;
        } else if (m == 1) {
          base = (const char*)L.w_oT;
          N = p.Hq * oproj_nt(D);
          rb = 32 * p.hd * esz;
          one = true;  // the consumers take one tile per chunk, however small
        } else if (m == 2) {
          base = (const char*)L.w_gu;
          up = base + (size_t)F * D * esz;
          N = F;
          rb = D * esz;
        } else {
          base = (const char*)L.w_dT;
          N = F;
          rb = D * esz;
          layer_end = true;
        }
      }
      int lo, hi;
      split(N, p.ncta, cta, lo, hi);
      const int per = one ? 1 : (up ? units_per_chunk(rb) : rows_per_chunk(rb));
      for (int r = lo; r < hi && !stop; r += per) {
        const unsigned bytes = (unsigned)(min(per, hi - r) * rb);
        if (up)
          issue2(base + (size_t)r * rb, up + (size_t)r * rb, bytes);
        else
          issue(base + (size_t)r * rb, bytes);
      }
      if (layer_end) {
        // the next layer's gains go out once this layer's weights are queued:
        // their slot was freed when the consumers began the previous layer's
        // FFN, which lies at least a ring's depth behind this point
        ++layer;
        side(layer);
      }
    }
    if (!PF) drain();  // prefetches leave nothing in flight that the CTA owns
  }

  // Copies still in flight must land before the CTA may exit: the last side
  // block copied into each slot (after an abort the producer stops early, so
  // these need not be the frame's last two layers) and the last FK_NSTAGE
  // ring chunks.
  __device__ void drain() {
    for (int slot = 0; slot < 2; ++slot) {
      const int k = side_last[slot];
      if (k < 0) continue;
      long long t0 = clock64();
      while (!mbar_try_wait(&sm->side_full[slot], (k >> 1) & 1u))
        if (clock64() - t0 > FK_WAIT_CYCLES) break;
    }
    const uint32_t first = n > (uint32_t)FK_NSTAGE ? n - FK_NSTAGE : 0;
    for (uint32_t m = first; m < n; ++m) {
      long long t0 = clock64();
      while (!mbar_try_wait(&sm->full[m % FK_NSTAGE], (m / FK_NSTAGE) & 1u))
        if (clock64() - t0 > FK_WAIT_CYCLES) break;
    }
  }
};

template <class WT, class KT>
__global__ void __launch_bounds__(FK_THREADS, 1) frame_kernel(const __grid_constant__ FKParams p) {
  FKSmem* sm = reinterpret_cast<FKSmem*>(fk_smem_raw);
  if (threadIdx.x == 0) sm->prm = p;
  for (int i = threadIdx.x; i < p.Lt + p.Lc; i += blockDim.x)
    sm->lay[i] = i < p.Lt ? p.tl[i] : p.cl[i - p.Lt];
  if (threadIdx.x == 0) {
    sm->pf_gate = 0;
    for (int s = 0; s < FK_NSTAGE; ++s) {
      mbar_init(&sm->full[s], 1);
      mbar_init(&sm->empty[s], FK_CONSUMER_WARPS);  // see release_private / release_shared
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm->side_full[s], 1);
      mbar_init(&sm->side_empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x < FK_PRODUCER_THREADS) {
    if (threadIdx.x == 0) {
      Producer<WT, false> pr(sm->prm, sm, blockIdx.x);
      pr.run();
    }
    return;
  }
  if (threadIdx.x >= FK_PRODUCER_THREADS + FK_CONSUMERS) {
    if (threadIdx.x == FK_PRODUCER_THREADS + FK_CONSUMERS && sm->prm.pf_ahead > 0) {
      Producer<WT, true> pf(sm->prm, sm, blockIdx.x);
      pf.run();
    }
    return;
  }
  consumer<WT, KT>();
}

// ------------------------------------------------------------- host side

template <class T>
__global__ void repack_oT_kernel(const T* __restrict__ w_o, T* __restrict__ w_oT, int D, int Hq, int hd) {
  // tile (h, j): w_oT[((h NT + j) (hd/8) + kb) 256 + 8 l + e] = w_o[32 j + l][h hd + 8 kb + e], 0 past D
  const int NT = (D + 31) / 32, nkb = hd / 8;
  const size_t n = (size_t)Hq * NT * 32 * hd;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(i % 8), l = (int)((i / 8) % 32);
    const size_t rest = i / 256;
    const int kb = (int)(rest % nkb);
    const size_t tile = rest / nkb;
    const int j = (int)(tile % NT), h = (int)(tile / NT);
    const int col = 32 * j + l;
    w_oT[i] = col < D ? w_o[(size_t)col * Hq * hd + (size_t)h * hd + 8 * kb + e] : T(0.f);
  }
}

template <class T>
__global__ void transpose_kernel(const T* __restrict__ in, T* __restrict__ out, int rows, int cols,
                                 size_t ostride) {
  // out[c * ostride + r] = in[r][c]
  __shared__ T tile[32][33];
  for (int r0 = blockIdx.y * 32; r0 < rows; r0 += gridDim.y * 32)
    for (int c0 = blockIdx.x * 32; c0 < cols; c0 += gridDim.x * 32) {
      for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, cc = c0 + threadIdx.x;
        if (r < rows && cc < cols) tile[i][threadIdx.x] = in[(size_t)r * cols + cc];
      }
      __syncthreads();
      for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int cc = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && cc < cols) out[(size_t)cc * ostride + r] = tile[threadIdx.x][i];
      }
      __syncthreads();
    }
}

static size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

// Floats between the copies of a residual buffer: the widest [tokens][D]
// either stack stages (the Talker's one token, or the CodePredictor's two),
// rounded to 256 bytes.
static int fk_xstride(const q3tts_config& c) {
  const int w = std::max(c.talker_hidden, FK_TMAX * c.cp_hidden);
  return (w + 63) & ~63;
}

// Bytes of one matrix element and of one gain / embedding element.
static int mat_esz(int wdt) { return wdt == Q3TTS_F32 ? 4 : (wdt == Q3TTS_FP8 ? 1 : 2); }
static int gain_esz(int wdt) { return wdt == Q3TTS_F32 ? 4 : 2; }

static size_t fk_layout(const q3tts_config& c, int ncta, FKState* st, char* base) {
  const int esz = mat_esz(c.weight_dtype), gsz = gain_esz(c.weight_dtype);
  const int Hq = c.n_q_heads, hd = c.head_dim, Hkv = c.n_kv_heads;
  const int dmax = std::max(c.talker_hidden, c.cp_hidden);
  const int qkv_rows = (Hq + 2 * Hkv) * hd;
  const int cpg = std::max(1, ncta / Hkv);
  const size_t xst = (size_t)fk_xstride(c);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = al256(off + bytes);
    return base ? base + o : nullptr;
  };
  const size_t oT_t = (size_t)Hq * hd * 32 * ((c.talker_hidden + 31) / 32);
  const size_t oT_c = (size_t)Hq * hd * 32 * ((c.cp_hidden + 31) / 32);
  // re-laid-out weights per layer: o_proj tiles, W_down^T
  char* reT = take((size_t)c.talker_layers * (oT_t + (size_t)c.talker_ffn * c.talker_hidden) * esz);
  char* reC = take((size_t)c.cp_layers * (oT_c + (size_t)c.cp_ffn * c.cp_hidden) * esz);
  char* sideT = take((size_t)c.talker_layers * (2 * c.talker_hidden + 2 * hd) * gsz);
  char* sideC = take((size_t)c.cp_layers * (2 * c.cp_hidden + 2 * hd) * gsz);
  char* tl = take(sizeof(LayerDev) * c.talker_layers);
  char* cl = take(sizeof(LayerDev) * c.cp_layers);
  char* plan = take(sizeof(FKPlan) * ncta);
  char* xb = take(sizeof(float) * 2 * xst);
  char* xa = take(sizeof(float) * 2 * xst);
  char* xf = take(sizeof(float) * 2 * FK_KC * xst);
  char* qkv = take(sizeof(uint64_t) * FK_TMAX * qkv_rows);
  char* z = take(sizeof(uint64_t) * FK_TMAX * c.cp_hidden);
  char* part = take(sizeof(uint64_t) * (size_t)Hq * cpg * (hd + 2));
  char* lg = take(sizeof(uint64_t) * c.cp_vocab);
  char* sync = take(sizeof(unsigned) * 4);
  if (st) {
    st->base = base;
    st->tl = (LayerDev*)tl;
    st->cl = (LayerDev*)cl;
    st->plan = (FKPlan*)plan;
    st->xb = (float*)xb; st->xa = (float*)xa; st->xf = (float*)xf;
    st->qkv = (uint64_t*)qkv; st->z = (uint64_t*)z; st->part = (uint64_t*)part; st->cp_logits = (uint64_t*)lg;
    st->bar = (unsigned*)sync;
    st->done = st->bar + 1;
    st->abort_flag = (int*)(st->bar + 2);
    st->dmax = dmax;
    st->sideT = sideT;
    st->sideC = sideC;
    (void)reT; (void)reC;
  }
  return off;
}

size_t frame_kernel_workspace(const q3tts_config& c, int) { return fk_layout(c, FK_MAXCTA, nullptr, nullptr) + 256; }

// The CTAs' plan rows: the producer's split of every phase (the same
// arithmetic it does on the device), with the chunk counts the consumers walk.
static void fk_plan(const q3tts_config& c, int ncta, std::vector<FKPlan>& plan) {
  const int esz = mat_esz(c.weight_dtype);
  const int D[2] = {c.cp_hidden, c.talker_hidden}, F[2] = {c.cp_ffn, c.talker_ffn},
            V[2] = {c.cp_vocab, c.codec_vocab};
  const int qkv_rows = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  const int SL[3] = {c.cp_hidden, c.talker_hidden, fk_xstride(c)};
  auto part = [&](int n, int i, int& lo, int& hi) {
    lo = (int)((unsigned)n * (unsigned)i / (unsigned)ncta);
    hi = (int)((unsigned)n * (unsigned)(i + 1) / (unsigned)ncta);
  };
  auto rows_pc = [](int rb) {
    const int r = FK_STAGE / rb;
    return r < 1 ? 1 : (r > FK_RMAX ? FK_RMAX : r);
  };
  auto units_pc = [](int rb) {
    const int u = FK_STAGE / (2 * rb);
    return u < 1 ? 1 : (u > FK_RMAX / 2 ? FK_RMAX / 2 : u);
  };
  auto range = [&](int n, int i, int per, FKRange& r) {
    part(n, i, r.lo, r.hi);
    r.nch = r.hi > r.lo ? (r.hi - r.lo + per - 1) / per : 0;
  };
  plan.assign(ncta, FKPlan{});
  for (int i = 0; i < ncta; ++i) {
    FKPlan& q = plan[i];
    for (int sd = 0; sd < 2; ++sd) {
      q.rpc[sd] = rows_pc(D[sd] * esz);
      q.upc[sd] = units_pc(D[sd] * esz);
      q.invD[sd] = 1.0f / (float)D[sd];
      range(qkv_rows, i, q.rpc[sd], q.qkv[sd]);
      range(V[sd], i, q.rpc[sd], q.head[sd]);
      range(F[sd], i, q.upc[sd], q.ffn[sd]);
      q.ffn_nd[sd] = q.ffn[sd].hi > q.ffn[sd].lo ? (q.ffn[sd].hi - q.ffn[sd].lo + q.rpc[sd] - 1) / q.rpc[sd] : 0;
      const int nt = (D[sd] + 31) / 32;
      part(c.n_q_heads * nt, i, q.op_t0[sd], q.op_t1[sd]);
      q.op_h0[sd] = q.op_t0[sd] / nt;
      q.op_h1[sd] = (q.op_t1[sd] - 1) / nt;
      q.inv_nt[sd] = 1.0f / (float)nt;
    }
    q.cpg = std::max(1, ncta / c.n_kv_heads);  // as the partials' layout (fk_layout)
    q.tg = i / q.cpg;
    q.tch = i % q.cpg;
    int hs = 0, rs = 0;
    while ((1 << hs) < c.head_dim) ++hs;
    while ((1 << rs) < c.n_q_heads / c.n_kv_heads) ++rs;
    q.hd_shift = hs;
    q.rep_shift = rs;
    q.inv_hd = 1.0f / (float)c.head_dim;
    q.attn_scale = 1.0f / std::sqrt((float)c.head_dim);
    range(c.cp_hidden, i, q.rpc[1], q.proj);  // rows of width D_t
    for (int w = 0; w < 3; ++w) {
      q.sl_lo[w] = SL[w] * i / ncta;
      q.sl_hi[w] = SL[w] * (i + 1) / ncta;
    }
  }
}

template <class WT, class KT>
static void* kernel_ptr() {
  return (void*)frame_kernel<WT, KT>;
}

static void* pick_kernel(int wdt, int kdt) {
  if (wdt == Q3TTS_FP8) return kdt == Q3TTS_BF16 ? kernel_ptr<fp8e4, bf16>() : kernel_ptr<fp8e4, float>();
  if (wdt == Q3TTS_BF16) return kdt == Q3TTS_BF16 ? kernel_ptr<bf16, bf16>() : kernel_ptr<bf16, float>();
  return kdt == Q3TTS_BF16 ? kernel_ptr<float, bf16>() : kernel_ptr<float, float>();
}

int frame_kernel_create(q3tts_handle* h) {
  FrameKernelState* st = new (std::nothrow) FrameKernelState();
  if (!st) return Q3TTS_ERR_ARG;
  st->ok = false;
  st->seq = 0;
  {
    const char* e = getenv("Q3TTS_PF_AHEAD");
    st->pf_ahead = e ? std::max(0, std::min(atoi(e), 1024)) : FK_PF_AHEAD;
  }
  h->fk = st;
  const q3tts_config& c = h->c;
  // eligibility: shapes the kernel's shared-memory layout covers
  if (c.talker_hidden > FK_DMAX || c.cp_hidden > FK_DMAX || c.head_dim > FK_HDMAX ||
      c.talker_layers + c.cp_layers > FK_MAXLAYERS ||
      c.n_q_heads / c.n_kv_heads > FK_REPMAX || c.codec_vocab > SAMPLER_VMAX ||
      c.cp_vocab > SAMPLER_VMAX || (c.codec_vocab % 4) || (c.cp_vocab % 4) || (c.talker_hidden % 8) ||
      (c.cp_hidden % 8) ||
      ((uintptr_t)h->w.talker_e_codec & 15) || ((uintptr_t)h->w.cp_embeds & 15))
    return Q3TTS_OK;
  const int ncta = std::min(h->n_sm, FK_MAXCTA);
  // every CTA's o_proj tile range must touch at most two heads (32-column
  // tiles, at most one head's worth per CTA); Talker attention needs a CTA
  // per kv head
  auto tiles_ok = [&](int D) {
    const int nt = (D + 31) / 32;
    return (c.n_q_heads * nt + ncta - 1) / ncta <= nt;
  };
  if (ncta < c.n_kv_heads || !tiles_ok(c.talker_hidden) || !tiles_ok(c.cp_hidden)) return Q3TTS_OK;
  // a ring chunk holds the gate and up rows of one FFN unit (2 D weights) and
  // one o_proj tile (32 hd weights); a CTA's FFN activations fit act
  const int esz_w = mat_esz(c.weight_dtype), esz_g = gain_esz(c.weight_dtype);
  if (2 * std::max(c.talker_hidden, c.cp_hidden) * esz_w > FK_STAGE || 32 * c.head_dim * esz_w > FK_STAGE)
    return Q3TTS_OK;
  if ((std::max(c.talker_ffn, c.cp_ffn) + ncta - 1) / ncta > FK_UMAX) return Q3TTS_OK;
  // RMSNorm staging holds at most FK_DMAX values: the CodePredictor's first
  // pass stages two tokens
  if (FK_TMAX * c.cp_hidden > FK_DMAX) return Q3TTS_OK;
  // cache pages and heads of a power-of-two size (positions and head
  // elements split by shift and mask), at least one warp wide
  if ((c.page_size & (c.page_size - 1)) || (c.head_dim & (c.head_dim - 1)) || c.head_dim < 32 ||
      c.n_q_heads % c.n_kv_heads)
    return Q3TTS_OK;
  // tags number a frame's steps below FK_MAXSTEPS
  const int steps = (Q3TTS_N_CODEBOOKS - 1) * (2 + (c.talker_hidden != c.cp_hidden ? 1 : 0) + 3 * c.cp_layers) +
                    2 + 4 * c.talker_layers;
  if (steps >= FK_MAXSTEPS) return Q3TTS_OK;
  // per-layer gains and both final norms fit their shared-memory slots
  if ((2 * std::max(c.talker_hidden, c.cp_hidden) + 2 * c.head_dim) * esz_g > FK_SIDE_BYTES ||
      (c.talker_hidden + c.cp_hidden) * esz_g > FK_FIN_BYTES)
    return Q3TTS_OK;
  st->smem = sizeof(FKSmem);
  void* k = pick_kernel(c.weight_dtype, c.kv_dtype);
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st->smem) != cudaSuccess) {
    cudaGetLastError();
    return Q3TTS_OK;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, FK_THREADS, st->smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    return Q3TTS_OK;
  }
  int coop = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->dev);
  if (!coop) return Q3TTS_OK;
  st->ncta = ncta;
  char* base = (char*)h->fk_base;  // workspace tail reserved by frame_kernel_workspace
  fk_layout(c, ncta, st, base);
  // re-laid-out weights
  const int esz = esz_w, gsz = esz_g;
  const int Hq = c.n_q_heads, hd = c.head_dim;
  std::vector<LayerDev> tl(c.talker_layers), cl(c.cp_layers);
  char* re = base;
  auto fill = [&](const q3tts_layer_weights& w, LayerDev& d, int D, int F, char* side) -> bool {
    const size_t gd = (size_t)D * gsz, gh = (size_t)hd * gsz;
    if (cudaMemcpyAsync(side, w.g_attn_norm, gd, cudaMemcpyDeviceToDevice, h->s) != cudaSuccess ||
        cudaMemcpyAsync(side + gd, w.g_ffn_norm, gd, cudaMemcpyDeviceToDevice, h->s) != cudaSuccess ||
        (w.g_q_norm && cudaMemcpyAsync(side + 2 * gd, w.g_q_norm, gh, cudaMemcpyDeviceToDevice, h->s) != cudaSuccess) ||
        (w.g_k_norm && cudaMemcpyAsync(side + 2 * gd + gh, w.g_k_norm, gh, cudaMemcpyDeviceToDevice, h->s) != cudaSuccess))
      return false;
    d.side = side;
    d.w_qkv = w.w_qkv;
    d.w_gu = w.w_gateup;
    d.s_qkv = w.s_qkv;
    d.s_o = w.s_o;
    d.s_gu = w.s_gateup;
    d.s_d = w.s_down;
    char* oT = re;
    re += (size_t)Hq * hd * 32 * ((D + 31) / 32) * esz;
    char* dT = re;
    re += (size_t)F * D * esz;
    d.w_oT = oT;
    d.w_dT = dT;
    // W_down^T [F][D]: dT[f][d] = W_down[d][f]
    dim3 tb(32, 8), tg((F + 31) / 32 < 1024 ? (F + 31) / 32 : 1024, (D + 31) / 32 < 1024 ? (D + 31) / 32 : 1024);
    if (esz == 1) {
      repack_oT_kernel<uint8_t><<<1024, 256, 0, h->s>>>((const uint8_t*)w.w_o, (uint8_t*)oT, D, Hq, hd);
      transpose_kernel<uint8_t><<<tg, tb, 0, h->s>>>((const uint8_t*)w.w_down, (uint8_t*)dT, D, F, (size_t)D);
    } else if (esz == 2) {
      repack_oT_kernel<bf16><<<1024, 256, 0, h->s>>>((const bf16*)w.w_o, (bf16*)oT, D, Hq, hd);
      transpose_kernel<bf16><<<tg, tb, 0, h->s>>>((const bf16*)w.w_down, (bf16*)dT, D, F, (size_t)D);
    } else {
      repack_oT_kernel<float><<<1024, 256, 0, h->s>>>((const float*)w.w_o, (float*)oT, D, Hq, hd);
      transpose_kernel<float><<<tg, tb, 0, h->s>>>((const float*)w.w_down, (float*)dT, D, F, (size_t)D);
    }
    return cudaGetLastError() == cudaSuccess;
  };
  for (int l = 0; l < c.talker_layers; ++l)
    if (!fill(h->tl[l], tl[l], c.talker_hidden, c.talker_ffn,
              st->sideT + (size_t)l * (2 * c.talker_hidden + 2 * hd) * gsz))
      return Q3TTS_ERR_CUDA;
  for (int l = 0; l < c.cp_layers; ++l)
    if (!fill(h->cl[l], cl[l], c.cp_hidden, c.cp_ffn, st->sideC + (size_t)l * (2 * c.cp_hidden + 2 * hd) * gsz))
      return Q3TTS_ERR_CUDA;
  std::vector<FKPlan> plan;
  fk_plan(c, ncta, plan);
  if (cudaMemcpyAsync(st->plan, plan.data(), sizeof(FKPlan) * plan.size(), cudaMemcpyHostToDevice, h->s) != cudaSuccess ||
      cudaMemcpyAsync(st->tl, tl.data(), sizeof(LayerDev) * tl.size(), cudaMemcpyHostToDevice, h->s) != cudaSuccess ||
      cudaMemcpyAsync(st->cl, cl.data(), sizeof(LayerDev) * cl.size(), cudaMemcpyHostToDevice, h->s) != cudaSuccess ||
      cudaMemsetAsync(st->bar, 0, sizeof(unsigned) * 4, h->s) != cudaSuccess ||
      cudaStreamSynchronize(h->s) != cudaSuccess)
    return Q3TTS_ERR_CUDA;
  st->ok = true;
  return Q3TTS_OK;
}

void frame_kernel_destroy(q3tts_handle* h) {
  delete h->fk;
  h->fk = nullptr;
}

static bool sampling_ok(int do_sample, int top_k) {
  return !do_sample || (top_k >= 1 && top_k <= SAMPLER_KSMALL);
}

// The persistent kernel takes one stream per launch and draws with top-k
// within the sampler's small-candidate path (or greedily).
bool frame_kernel_supports(const q3tts_handle* h, int n_active, const q3tts_sampling* sp) {
  if (!h->fk || !h->fk->ok || n_active != 1 || h->frame_kernel_off) return false;
  return sampling_ok(sp[0].do_sample, sp[0].top_k) && sampling_ok(sp[0].sub_do_sample, sp[0].sub_top_k);
}

// Launch parameters of one frame of stream sid at Talker position pos, with the
// per-frame scratch taken from the handle's workspace.
static void frame_params(FKParams& p, const q3tts_handle* h, int sid, int pos, int newpage,
                         const q3tts_sampling& sp, const float* uniforms, int32_t* codes,
                         const int32_t* forced, float* logits) {
  const FrameKernelState* st = h->fk;
  const q3tts_config& c = h->c;
  p.ncta = st->ncta;
  p.Dt = c.talker_hidden; p.Dc = c.cp_hidden; p.Ft = c.talker_ffn; p.Fc = c.cp_ffn;
  p.Hq = c.n_q_heads; p.Hkv = c.n_kv_heads; p.hd = c.head_dim; p.Vt = c.codec_vocab; p.Vc = c.cp_vocab;
  p.Lt = c.talker_layers; p.Lc = c.cp_layers; p.qkv_rows = h->qkv_rows;
  p.has_proj = h->w.cp_w_proj != nullptr; p.qk_norm = c.qk_norm; p.dmax = st->dmax; p.eps = c.rms_eps;
  p.xstride = fk_xstride(c);
  p.tl = st->tl; p.cl = st->cl; p.plan = st->plan;
  p.t_head = h->w.talker_w_head; p.e_codec = h->w.talker_e_codec; p.cp_heads = h->w.cp_heads;
  p.cp_embeds = h->w.cp_embeds; p.cp_proj = h->w.cp_w_proj; p.t_gfinal = h->w.talker_g_final;
  p.cp_gfinal = h->w.cp_g_final;
  p.s_head = h->w.s_head; p.s_cp_heads = h->w.s_cp_heads; p.s_cp_proj = h->w.s_cp_proj;
  p.pending_h = h->pending_h; p.pending_logits = h->pending_logits; p.history = h->history;
  p.finished = h->finished;
  p.tkv = talker_kv(h); p.ckv = cp_kv(h); p.rope_cos = h->rope_cos; p.rope_sin = h->rope_sin;
  p.xb = st->xb; p.xa = st->xa; p.xf = st->xf;
  p.qkv = st->qkv; p.z = st->z; p.part = st->part; p.cp_logits = st->cp_logits;
  p.bar = st->bar; p.done = st->done; p.err = h->d_err; p.abort_flag = st->abort_flag;
  p.wait_cycles = h->dbg_wait_cycles > 0 ? h->dbg_wait_cycles : FK_WAIT_CYCLES;
  p.fail_bar = h->dbg_fail_bar;
  p.pf_ahead = st->pf_ahead;
  p.sid = sid; p.pos = pos; p.newpage = newpage; p.sp = sp;
  p.uniforms = uniforms; p.codes = codes; p.forced = forced; p.dump = logits;
}

static int frame_launch(q3tts_handle* h, FKParams& p) {
  void* args[] = {&p};
  cudaError_t e = cudaLaunchCooperativeKernel(pick_kernel(h->c.weight_dtype, h->c.kv_dtype),
                                              dim3(h->fk->ncta), dim3(FK_THREADS), args, h->fk->smem, h->s);
  h->launches += 1;
  h->dbg_fail_bar = -1;  // an armed failure-path test covers one launch
  h->dbg_wait_cycles = 0;
  return e == cudaSuccess ? Q3TTS_OK : Q3TTS_ERR_CUDA;
}

// The next sequence number of a scratch area (its tagged words start at 0,
// so the numbers start at 1 and skip 0 when they wrap).
static uint32_t next_seq(uint32_t& s) {
  s = s + 1 == 0 ? 1 : s + 1;
  return s;
}

int frame_kernel_step(q3tts_handle* h, const StepDesc& d, const float* uniforms, int32_t* codes,
                      const int32_t* forced, float* logits) {
  FKParams p;
  frame_params(p, h, d.sid[0], d.pos[0], d.newpage[0], d.sp[0], uniforms, codes, forced, logits);
  p.seq = next_seq(h->fk->seq);
  return frame_launch(h, p);
}

#ifdef Q3TTS_TRACE
// Profiling builds: copies the timestamp buffer to host memory.
extern "C" int q3tts_trace_fetch(void* host, size_t bytes) {
  return cudaMemcpyFromSymbol(host, fk_trace_buf, bytes) == cudaSuccess ? 0 : -3;
}
#endif

// Arms the failure-path test for the handle's next persistent launch.
int frame_kernel_debug_fail(q3tts_handle* h, int barrier, int wait_us) {
  if (!h->fk || !h->fk->ok) return Q3TTS_ERR_UNSUPPORTED;
  h->dbg_fail_bar = barrier;
  h->dbg_wait_cycles = (long long)wait_us * 2070;  // clock64 ticks at the highest SM clock
  return Q3TTS_OK;
}

// After a device-side error: clear the barrier counters and the abort flag.
int frame_kernel_recover(q3tts_handle* h) {
  if (!h->fk || !h->fk->ok) return Q3TTS_OK;
  return cudaMemsetAsync(h->fk->bar, 0, sizeof(unsigned) * 4, h->s) == cudaSuccess ? Q3TTS_OK
                                                                                   : Q3TTS_ERR_CUDA;
}


// ------------------------------------------- frame step with static scratch
//
// q3tts_step_frame_static runs the same kernel with its per-frame scratch (the
// three residual vectors, QKV rows, attention partials, CodePredictor logits
// and the grid-barrier words) in this file-scope
// device array instead of the caller's workspace, so a frame needs no memory
// from the caller beyond what q3tts_create was given, and the call itself
// makes no device or host allocation.  Layout: the barrier words (bar, done,
// abort flag) in the first 256 bytes -- at the same place for every handle,
// since a completed frame leaves them zero for whichever call comes next --
// then the vectors, each 256-byte aligned.  Every other byte is written by a
// frame before it is read, so only the barrier words must start at zero.
static __device__ __align__(256) unsigned char fk_static_scratch[Q3TTS_STATIC_SCRATCH_BYTES];

constexpr int FK_MAX_DEVICES = 64;
static std::mutex g_static_mu;
static std::atomic<unsigned char*> g_static_addr[FK_MAX_DEVICES];
// Launches that used each device's static scratch (tags: the array is shared
// by every handle, so its sequence numbers are too).
static std::atomic<uint32_t> g_static_seq[FK_MAX_DEVICES];

// Places the scratch vectors of config c behind the barrier words at base
// (size only when base is null); returns the bytes used.
static size_t fk_static_layout(const q3tts_config& c, int ncta, char* base, FKParams* p) {
  const size_t xst = (size_t)fk_xstride(c);
  const int qkv_rows = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
  const int cpg = std::max(1, ncta / c.n_kv_heads);
  size_t off = 256;  // barrier words
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = al256(off + bytes);
    return base ? base + o : nullptr;
  };
  char* xb = take(sizeof(float) * 2 * xst);
  char* xa = take(sizeof(float) * 2 * xst);
  char* xf = take(sizeof(float) * 2 * FK_KC * xst);
  char* qkv = take(sizeof(uint64_t) * FK_TMAX * qkv_rows);
  char* z = take(sizeof(uint64_t) * FK_TMAX * c.cp_hidden);
  char* part = take(sizeof(uint64_t) * (size_t)c.n_q_heads * cpg * (c.head_dim + 2));
  char* lg = take(sizeof(uint64_t) * c.cp_vocab);
  if (p) {
    p->xb = (float*)xb; p->xa = (float*)xa; p->xf = (float*)xf;
    p->qkv = (uint64_t*)qkv; p->z = (uint64_t*)z; p->part = (uint64_t*)part; p->cp_logits = (uint64_t*)lg;
    p->bar = (unsigned*)base;
    p->done = p->bar + 1;
    p->abort_flag = (int*)(p->bar + 2);
  }
  return off;
}

// Address of the scratch array on the handle's device.  The first call on a
// device looks the symbol up (with that device current) and clears the
// barrier words on the handle's stream; later calls only read the cached
// address.
static int static_scratch(q3tts_handle* h, unsigned char** out) {
  if (h->dev < 0 || h->dev >= FK_MAX_DEVICES) return Q3TTS_ERR_UNSUPPORTED;
  unsigned char* a = g_static_addr[h->dev].load(std::memory_order_acquire);
  if (!a) {
    std::lock_guard<std::mutex> lock(g_static_mu);
    a = g_static_addr[h->dev].load(std::memory_order_relaxed);
    if (!a) {
      int cur = -1;
      if (cudaGetDevice(&cur) != cudaSuccess) return Q3TTS_ERR_CUDA;
      if (cur != h->dev && cudaSetDevice(h->dev) != cudaSuccess) return Q3TTS_ERR_CUDA;
      void* sym = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&sym, fk_static_scratch);
      if (e == cudaSuccess) e = cudaMemsetAsync(sym, 0, 256, h->s);
      if (e == cudaSuccess) e = cudaStreamSynchronize(h->s);
      if (cur != h->dev) cudaSetDevice(cur);
      if (e != cudaSuccess || !sym) {
        cudaGetLastError();
        return Q3TTS_ERR_CUDA;
      }
      a = (unsigned char*)sym;
      g_static_addr[h->dev].store(a, std::memory_order_release);
    }
  }
  *out = a;
  return Q3TTS_OK;
}

// Whether q3tts_step_frame_static can run this handle with these sampling
// settings; Q3TTS_ERR_SCRATCH if the scratch would not fit the array.
int frame_kernel_static_check(const q3tts_handle* h, const q3tts_sampling& sp) {
  if (!h->fk || !h->fk->ok) return Q3TTS_ERR_UNSUPPORTED;
  if (!sampling_ok(sp.do_sample, sp.top_k) || !sampling_ok(sp.sub_do_sample, sp.sub_top_k))
    return Q3TTS_ERR_UNSUPPORTED;
  if (fk_static_layout(h->c, h->fk->ncta, nullptr, nullptr) > (size_t)Q3TTS_STATIC_SCRATCH_BYTES)
    return Q3TTS_ERR_SCRATCH;
  return Q3TTS_OK;
}

int frame_kernel_step_static(q3tts_handle* h, int sid, int pos, int newpage, const q3tts_sampling& sp,
                             const float* uniforms, int32_t* codes, const int32_t* forced, float* logits) {
  unsigned char* base = nullptr;
  int rc = static_scratch(h, &base);
  if (rc != Q3TTS_OK) return rc;
  h->used_static = true;
  FKParams p;
  frame_params(p, h, sid, pos, newpage, sp, uniforms, codes, forced, logits);
  fk_static_layout(h->c, h->fk->ncta, (char*)base, &p);
  uint32_t sq = g_static_seq[h->dev].fetch_add(1u, std::memory_order_relaxed) + 1u;
  if (sq == 0) sq = g_static_seq[h->dev].fetch_add(1u, std::memory_order_relaxed) + 1u;
  p.seq = sq;
  return frame_launch(h, p);
}

// After a device-side error in a frame that used the static scratch.
int frame_kernel_recover_static(q3tts_handle* h) {
  if (!h->used_static || h->dev < 0 || h->dev >= FK_MAX_DEVICES) return Q3TTS_OK;
  unsigned char* a = g_static_addr[h->dev].load(std::memory_order_acquire);
  if (!a) return Q3TTS_OK;
  return cudaMemsetAsync(a, 0, 256, h->s) == cudaSuccess ? Q3TTS_OK : Q3TTS_ERR_CUDA;
}

}  // namespace q3
