// step.cu -- prefill and the layer-by-layer frame step (one kernel per operation).
//
// Frame structure ("Running Qwen3-TTS on an AMD R9700", section "Running
// Qwen3-TTS"): the semantic token comes from the Talker's pending logits, the
// CodePredictor then produces acoustic tokens 1..15 one pass at a time (pass 0
// over the Talker hidden and the semantic token's embedding, pass j over the
// embedding of token j), and the sum of the frame's 16 code embeddings
// ("qwen3-tts-hip" README, "Python Parity Fixtures": embedding-sum parity) is
// the input of one Talker step whose final norm and codec head leave the next
// pending logits.
#include "engine.cuh"
#include "layers.cuh"
#include "sampler.cuh"

namespace q3 {

KVDesc talker_kv(const q3tts_handle* h) {
  KVDesc d;
  d.pool = h->kv_pool;
  d.page_table = h->page_table;
  d.pages_per_stream = h->pps;
  d.page_size = h->c.page_size;
  d.n_pages = h->n_pages;
  d.Hkv = h->Hkv;
  d.hd = h->hd;
  return d;
}

KVDesc cp_kv(const q3tts_handle* h) {
  KVDesc d;
  d.pool = h->cp_kv;
  d.page_table = h->cp_page_table;
  d.pages_per_stream = 1;
  d.page_size = Q3TTS_N_CODEBOOKS;
  d.n_pages = h->c.max_streams;
  d.Hkv = h->Hkv;
  d.hd = h->hd;
  return d;
}

// ----------------------------------------------------------- small kernels

__global__ void setup_kernel(const StepDesc* __restrict__ dd, int* sid, int* pos, q3tts_sampling* sp,
                             int* page_table, int pps, int page_size, int* tok_stream, int* tok_pos) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  const StepDesc& d = *dd;
  for (int b = threadIdx.x; b < d.n; b += blockDim.x) {
    sid[b] = d.sid[b];
    pos[b] = d.pos[b];
    sp[b] = d.sp[b];
    if (d.newpage[b] >= 0) page_table[d.sid[b] * pps + d.pos[b] / page_size] = d.newpage[b];
    // CodePredictor pass 0: two tokens per stream at positions 0 and 1
    tok_stream[2 * b] = d.sid[b];
    tok_stream[2 * b + 1] = d.sid[b];
    tok_pos[2 * b] = 0;
    tok_pos[2 * b + 1] = 1;
  }
}

__global__ void fill_tokens_kernel(int* tok_stream, int* tok_pos, int T, int sid, int pos0) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < T; m += gridDim.x * blockDim.x) {
    tok_stream[m] = sid;
    tok_pos[m] = pos0 + m;
  }
}

// One block per active stream.  semantic != 0: the Talker's pending logits of
// the stream, its repetition history and the semantic controls; otherwise row
// b of `logits` with the sub-talker controls.
// Codes out follow the stop conditions: a stream whose end-of-stream code was
// fed writes -1; the frame that feeds it keeps its semantic code, marks the
// stream finished, and writes -1 for its acoustic codes (the frame itself is
// computed either way).  Special semantic codes other than the end-of-stream
// code are masked before the draw (the dump keeps the raw logits).
__global__ void __launch_bounds__(256) sample_kernel(
    const float* __restrict__ logits, int V, int semantic, const int* __restrict__ sid,
    const q3tts_sampling* __restrict__ sp, uint8_t* history, uint8_t* finished,
    const float* __restrict__ uniforms, int cb, const int32_t* __restrict__ forced,
    int32_t* __restrict__ codes, int* __restrict__ fed, float* __restrict__ dump, int dump_ld, int dump_off,
    int* err) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smraw[];
  SamplerSmem& sm = *reinterpret_cast<SamplerSmem*>(smraw);
  const int b = blockIdx.x, s = sid[b];
  const q3tts_sampling p = sp[b];
  const float* row = semantic ? logits + (size_t)s * V : logits + (size_t)b * V;
  const int sf = semantic ? p.special_from : 0;
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    float v = row[i];
    if (dump) dump[(size_t)b * dump_ld + dump_off + i] = v;
    if (sf > 0 && i >= sf && i != p.eos_token) v = -INFINITY;
    sm.val[i] = v;
  }
  __syncthreads();
  const uint8_t* hist = semantic ? history + (size_t)s * V : nullptr;
  int code = semantic
                 ? block_sample(sm, V, p.do_sample, p.top_k, p.top_p, p.temperature,
                                p.repetition_penalty, hist, uniforms[b * 16 + cb])
                 : block_sample(sm, V, p.sub_do_sample, p.sub_top_k, p.sub_top_p,
                                p.sub_temperature, 1.0f, nullptr, uniforms[b * 16 + cb]);
  code = min(max(code, 0), V - 1);
  if (threadIdx.x == 0) {
    int f = forced ? forced[b * 16 + cb] : code;
    if (f < 0 || f >= V) {
      atomicExch(err, Q3TTS_ERR_ARG);
      f = code;
    }
    fed[b * 16 + cb] = f;
    if (semantic) {
      const bool before = finished[s] != 0;
      if (!before && p.eos_token >= 0 && f == p.eos_token) finished[s] = 1;
      codes[b * 16 + cb] = before ? -1 : code;
      history[(size_t)s * V + f] = 1;
    } else {
      codes[b * 16 + cb] = finished[s] ? -1 : code;
    }
  }
}

template <class WT>
__global__ void cp_input_kernel(int j, int n, const int* __restrict__ sid,
                                const int* __restrict__ fed, const float* __restrict__ pending_h,
                                const WT* __restrict__ e_codec, const WT* __restrict__ cp_embeds,
                                int Dt, int Vc, float* __restrict__ uin) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  const int r = blockIdx.x;  // output row
  const float* srcf = nullptr;
  const WT* srcw = nullptr;
  if (j == 0) {
    int b = r / 2;
    if ((r & 1) == 0)
      srcf = pending_h + (size_t)sid[b] * Dt;
    else
      srcw = e_codec + (size_t)fed[b * 16] * Dt;
  } else {
    srcw = cp_embeds + ((size_t)(j - 1) * Vc + fed[r * 16 + j]) * Dt;
  }
  for (int i = threadIdx.x; i < Dt; i += blockDim.x)
    uin[(size_t)r * Dt + i] = srcf ? srcf[i] : to_f(srcw[i]);
}

template <class WT>
__global__ void embed_sum_kernel(const int* __restrict__ fed, const WT* __restrict__ e_codec,
                                 const WT* __restrict__ cp_embeds, int Dt, int Vc,
                                 float* __restrict__ x) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  const int b = blockIdx.y;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= Dt) return;
  float acc = to_f(e_codec[(size_t)fed[b * 16] * Dt + i]);
  for (int j = 1; j < Q3TTS_N_CODEBOOKS; ++j)
    acc += to_f(cp_embeds[((size_t)(j - 1) * Vc + fed[b * 16 + j]) * Dt + i]);
  x[(size_t)b * Dt + i] = acc;
}

__global__ void scatter_pending_kernel(const int* __restrict__ sid, const float* __restrict__ hn,
                                       const float* __restrict__ lg, int Dt, int Vt,
                                       float* __restrict__ pending_h,
                                       float* __restrict__ pending_logits) {
  pdl_wait();  // inputs come from the previous kernel
  pdl_trigger();
  const int b = blockIdx.x, s = sid[b];
  for (int i = threadIdx.x; i < Dt; i += blockDim.x)
    pending_h[(size_t)s * Dt + i] = hn[(size_t)b * Dt + i];
  for (int i = threadIdx.x; i < Vt; i += blockDim.x)
    pending_logits[(size_t)s * Vt + i] = lg[(size_t)b * Vt + i];
}

// ------------------------------------------------------------ stack pass

static HiLo hilo(const q3tts_handle* h) { return HiLo{h->xh, h->xl, h->m_max}; }

// Y (+)= X W^T.  On the tensor-core path X is the hi/lo pair already written
// by the producing kernel (xf unused); otherwise xf (fp32, row pitch ldx).
static void proj(q3tts_handle* h, const float* xf, int ldx, const void* W, int N, int K, float* Y, int ldy,
                 int M, bool acc, const float* scale = nullptr) {
  if (h->tc) {
    if (!tc_linear(hilo(h), W, N, K, Y, ldy, M, acc, h->d_err, h->s)) h->tc_failed = true;
  } else {
    launch_linear(h->c.weight_dtype, xf, ldx, W, N, K, Y, ldy, M, acc, h->s, scale);
  }
}

// dtype of the norm gains and embedding tables (bf16 beside FP8 matrices)
static int gain_dt(const q3tts_handle* h) {
  return h->c.weight_dtype == Q3TTS_FP8 ? Q3TTS_BF16 : h->c.weight_dtype;
}

// RMSNorm of M rows of X into the next projection's input: hi/lo terms on the
// tensor-core path, else fp32 in h->hb.
static void norm_in(q3tts_handle* h, const float* X, int ldx, int in_mul, int in_add, const void* g, int M, int D) {
  if (h->tc)
    launch_rmsnorm_hilo(gain_dt(h), X, ldx, in_mul, in_add, g, hilo(h), M, D, h->c.rms_eps, h->s);
  else
    launch_rmsnorm(gain_dt(h), X, ldx, in_mul, in_add, g, h->hb, D, M, D, h->c.rms_eps, h->s);
}

// M tokens through all layers of one decoder stack (residual stream x [M, D]).
// pf_sid >= 0: the tokens are a prefill chunk of stream pf_sid at positions
// pf_pos0 .. pf_pos0 + M - 1.
static void stack_pass(q3tts_handle* h, const q3tts_layer_weights* lw, int layers, int D, int F,
                       float* x, int M, TokDesc td, KVDesc kv, int kdt, int max_ctx, int pf_sid = -1,
                       int pf_pos0 = 0) {
  cudaStream_t s = h->s;
  const int gdt = gain_dt(h), HqD = h->Hq * h->hd;
  for (int l = 0; l < layers; ++l) {
    const q3tts_layer_weights& L = lw[l];
    norm_in(h, x, D, 1, 0, L.g_attn_norm, M, D);
    proj(h, h->hb, D, L.w_qkv, h->qkv_rows, D, h->qkv, h->qkv_rows, M, false, L.s_qkv);
    launch_qk_rope_append(gdt, kdt, h->qkv, h->qkv_rows, M, td, L.g_q_norm, L.g_k_norm,
                          h->c.qk_norm, h->c.rms_eps, h->rope_cos, h->rope_sin, kv, l, h->Hq, s);
    // a prefill chunk: query tiles on the tensor cores; contexts longer than
    // one span: spread over the GPU by span
    const bool fa = pf_sid >= 0 && launch_fa_prefill(h->qkv, h->qkv_rows, M, pf_sid, pf_pos0, kv, kdt, l, h->Hq,
                                                      h->att, HqD, h->d_err, s);
    if (!fa && (max_ctx <= 64 || !launch_attention_split(kdt, h->qkv, h->qkv_rows, M, td, kv, l, h->Hq, h->att,
                                                         HqD, h->spl_part, h->spl_cnt, h->spl_nsmax, s)))
      launch_attention(kdt, h->qkv, h->qkv_rows, M, td, kv, l, h->Hq, h->att, HqD, max_ctx, s);
    if (h->tc) launch_split_hilo(h->att, HqD, hilo(h), M, HqD, s);
    proj(h, h->att, HqD, L.w_o, D, HqD, x, D, M, true, L.s_o);
    norm_in(h, x, D, 1, 0, L.g_ffn_norm, M, D);
    proj(h, h->hb, D, L.w_gateup, 2 * F, D, h->gu, 2 * F, M, false, L.s_gateup);
    if (h->tc)
      launch_silu_mul_hilo(h->gu, hilo(h), M, F, s);
    else
      launch_silu_mul(h->gu, h->act, M, F, s);
    proj(h, h->act, F, L.w_down, D, F, x, D, M, true, L.s_down);
  }
  h->launches += (h->tc ? 10ull : 9ull) * layers;
}

static size_t wbytes(const q3tts_handle* h) { return (size_t)h->esz; }

int prefill_layered(q3tts_handle* h, int sid, const float* embeds, int len) {
  cudaStream_t s = h->s;
  const int Dt = h->Dt;
  for (int c0 = 0; c0 < len; c0 += h->chunk) {
    int T = len - c0 < h->chunk ? len - c0 : h->chunk;
    cudaMemcpyAsync(h->x, embeds + (size_t)c0 * Dt, sizeof(float) * (size_t)T * Dt,
                    cudaMemcpyDeviceToDevice, s);
    launch_pdl(fill_tokens_kernel, dim3((T + 255) / 256), dim3(256), 0, s, h->d_tok_stream, h->d_tok_pos, T, sid, c0);
    h->launches += 1;
    TokDesc td{h->d_tok_stream, h->d_tok_pos, 0};
    stack_pass(h, h->tl.data(), h->c.talker_layers, Dt, h->Ft, h->x, T, td, talker_kv(h),
               h->c.kv_dtype, c0 + T, sid, c0);
    if (c0 + T == len) {
      launch_rmsnorm(gain_dt(h), h->x, Dt, 1, T - 1, h->w.talker_g_final,
                     h->pending_h + (size_t)sid * Dt, Dt, 1, Dt, h->c.rms_eps, s);
      launch_linear(h->c.weight_dtype, h->pending_h + (size_t)sid * Dt, Dt, h->w.talker_w_head,
                    h->Vt, Dt, h->pending_logits + (size_t)sid * h->Vt, h->Vt, 1, false, s, h->w.s_head);
      h->launches += 2;
    }
  }
  if (h->tc_failed) {
    h->tc_failed = false;
    return Q3TTS_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? Q3TTS_OK : Q3TTS_ERR_CUDA;
}

// The layered step's kernels for n active streams, whose descriptor is in
// h->d_desc; the attention kernels are sized for contexts up to max_ctx.
static void step_kernels(q3tts_handle* h, int n, int max_ctx, const float* uniforms, int32_t* codes,
                         const int32_t* forced, float* logits) {
  cudaStream_t s = h->s;
  const int Dt = h->Dt, Dc = h->Dc, Vt = h->Vt, Vc = h->Vc, gdt = gain_dt(h);
  const int dump_ld = Vt + (Q3TTS_N_CODEBOOKS - 1) * Vc;
  const size_t smem = sizeof(SamplerSmem);
  launch_pdl(setup_kernel, dim3(1), dim3(256), 0, s, h->d_desc, h->d_sid, h->d_pos, h->d_sp, h->page_table, h->pps,
                                 h->c.page_size, h->d_tok_stream, h->d_tok_pos);
  launch_pdl(sample_kernel, dim3(n), dim3(256), smem, s, h->pending_logits, Vt, 1, h->d_sid, h->d_sp, h->history, h->finished,
                                     uniforms, 0, forced, codes, h->d_fed, logits, dump_ld, 0,
                                     h->d_err);
  const size_t es = wbytes(h);
  for (int j = 0; j < Q3TTS_N_CODEBOOKS - 1; ++j) {
    const int M = j == 0 ? 2 * n : n;
    if (gdt == Q3TTS_BF16)
      launch_pdl(cp_input_kernel<bf16>, dim3(M), dim3(256), 0, s, j, n, h->d_sid, h->d_fed, h->pending_h,
                                              (const bf16*)h->w.talker_e_codec,
                                              (const bf16*)h->w.cp_embeds, Dt, Vc, h->uin);
    else
      launch_pdl(cp_input_kernel<float>, dim3(M), dim3(256), 0, s, j, n, h->d_sid, h->d_fed, h->pending_h,
                                               (const float*)h->w.talker_e_codec,
                                               (const float*)h->w.cp_embeds, Dt, Vc, h->uin);
    if (h->w.cp_w_proj) {
      if (h->tc) {
        launch_split_hilo(h->uin, Dt, hilo(h), M, Dt, s);
        h->launches += 1;
      }
      proj(h, h->uin, Dt, h->w.cp_w_proj, Dc, Dt, h->cpx, Dc, M, false, h->w.s_cp_proj);
    } else
      cudaMemcpyAsync(h->cpx, h->uin, sizeof(float) * (size_t)M * Dc, cudaMemcpyDeviceToDevice, s);
    TokDesc td = j == 0 ? TokDesc{h->d_tok_stream, h->d_tok_pos, 0} : TokDesc{h->d_sid, nullptr, j + 1};
    stack_pass(h, h->cl.data(), h->c.cp_layers, Dc, h->Fc, h->cpx, M, td, cp_kv(h), Q3TTS_F32,
               Q3TTS_N_CODEBOOKS);
    norm_in(h, h->cpx, Dc, j == 0 ? 2 : 1, j == 0 ? 1 : 0, h->w.cp_g_final, n, Dc);
    const void* head = (const char*)h->w.cp_heads + (size_t)j * Vc * Dc * es;
    proj(h, h->hb, Dc, head, Vc, Dc, h->logits, Vc, n, false,
         h->w.s_cp_heads ? h->w.s_cp_heads + (size_t)j * Vc : nullptr);
    launch_pdl(sample_kernel, dim3(n), dim3(256), smem, s, h->logits, Vc, 0, h->d_sid, h->d_sp, nullptr, h->finished, uniforms,
                                       j + 1, forced, codes, h->d_fed, logits, dump_ld,
                                       Vt + j * Vc, h->d_err);
    h->launches += 4 + (h->w.cp_w_proj ? 1 : 0);
  }
  if (gdt == Q3TTS_BF16)
    launch_pdl(embed_sum_kernel<bf16>, dim3(dim3((Dt + 255) / 256, n)), dim3(256), 0, s, 
        h->d_fed, (const bf16*)h->w.talker_e_codec, (const bf16*)h->w.cp_embeds, Dt, Vc, h->x);
  else
    launch_pdl(embed_sum_kernel<float>, dim3(dim3((Dt + 255) / 256, n)), dim3(256), 0, s, 
        h->d_fed, (const float*)h->w.talker_e_codec, (const float*)h->w.cp_embeds, Dt, Vc, h->x);
  TokDesc td{h->d_sid, h->d_pos, 0};
  stack_pass(h, h->tl.data(), h->c.talker_layers, Dt, h->Ft, h->x, n, td, talker_kv(h),
             h->c.kv_dtype, max_ctx);
  // the normed hidden is also the stream's pending h_T (fp32)
  launch_rmsnorm(gdt, h->x, Dt, 1, 0, h->w.talker_g_final, h->hb, Dt, n, Dt, h->c.rms_eps, s);
  if (h->tc) {
    launch_split_hilo(h->hb, Dt, hilo(h), n, Dt, s);
    h->launches += 1;
  }
  proj(h, h->hb, Dt, h->w.talker_w_head, Vt, Dt, h->logits, Vt, n, false, h->w.s_head);
  launch_pdl(scatter_pending_kernel, dim3(n), dim3(256), 0, s, h->d_sid, h->hb, h->logits, Dt, Vt, h->pending_h,
                                           h->pending_logits);
  h->launches += 6;  // setup, semantic sample, embed-sum, final norm, head, scatter
}

void step_graph_destroy(q3tts_handle* h) {
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  h->gexec = nullptr;
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  h->cap_stream = nullptr;
}

// Captures the step's kernels for n streams into h->gexec (inputs and
// outputs in the handle's fixed buffers); false if capture is not possible.
static bool step_graph_build(q3tts_handle* h, int n, bool with_forced) {
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  h->gexec = nullptr;
  if (!h->cap_stream && cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
    h->cap_stream = nullptr;
    return false;
  }
  cudaStream_t user = h->s;
  h->s = h->cap_stream;
  const uint64_t l0 = h->launches;
  cudaGraph_t g = nullptr;
  bool ok = cudaStreamBeginCapture(h->s, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
  if (ok) {
    step_kernels(h, n, h->c.kv_cap_steps, h->g_uni, h->g_codes, with_forced ? h->g_forced : nullptr, nullptr);
    ok = cudaStreamEndCapture(h->s, &g) == cudaSuccess && g != nullptr;
  }
  h->s = user;
  h->g_launches = h->launches - l0;
  h->launches = l0;
  if (ok) ok = cudaGraphInstantiate(&h->gexec, g, 0) == cudaSuccess;
  if (g) cudaGraphDestroy(g);
  cudaGetLastError();
  if (!ok) {  // not capturable here: launch kernel by kernel from now on
    h->gexec = nullptr;
    h->graph_off = true;
    return false;
  }
  h->g_n = n;
  h->g_forced_on = with_forced;
  return true;
}

// The layered frame step.  Without a logits dump it is replayed from a CUDA
// graph captured once per (active streams, forced or not): the descriptor
// goes to the device ahead of it, the caller's uniforms and forced codes are
// copied into the handle's buffers and the codes copied out after it.
int step_layered(q3tts_handle* h, const StepDesc& d, const float* uniforms, int32_t* codes,
                 const int32_t* forced, float* logits) {
  cudaStream_t s = h->s;
  const int n = d.n;
  // pageable source: the copy is staged before the call returns, so d may change
  if (cudaMemcpyAsync(h->d_desc, &d, sizeof(StepDesc), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return Q3TTS_ERR_CUDA;
  const size_t att_smem = sizeof(float) * (size_t)(h->hd + h->c.kv_cap_steps);  // non-grouped attention
  const bool graph = !h->graph_off && !logits && (((h->hd == 128 || h->hd == 64) && h->Hq / h->Hkv <= 4) || att_smem <= 48 * 1024);
  if (graph && ((h->gexec && h->g_n == n && h->g_forced_on == (forced != nullptr)) ||
                step_graph_build(h, n, forced != nullptr))) {
    const size_t nb = sizeof(int32_t) * (size_t)n * Q3TTS_N_CODEBOOKS;
    cudaMemcpyAsync(h->g_uni, uniforms, nb, cudaMemcpyDeviceToDevice, s);
    if (forced) cudaMemcpyAsync(h->g_forced, forced, nb, cudaMemcpyDeviceToDevice, s);
    cudaGraphLaunch(h->gexec, s);
    cudaMemcpyAsync(codes, h->g_codes, nb, cudaMemcpyDeviceToDevice, s);
    h->launches += h->g_launches;
  } else {
    int max_ctx = 0;
    for (int b = 0; b < n; ++b) max_ctx = d.pos[b] + 1 > max_ctx ? d.pos[b] + 1 : max_ctx;
    step_kernels(h, n, max_ctx, uniforms, codes, forced, logits);
  }
  if (h->tc_failed) {
    h->tc_failed = false;
    return Q3TTS_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? Q3TTS_OK : Q3TTS_ERR_CUDA;
}

int sampler_setup() {
  cudaError_t e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(SamplerSmem));
  return e == cudaSuccess ? Q3TTS_OK : Q3TTS_ERR_CUDA;
}

}  // namespace q3
