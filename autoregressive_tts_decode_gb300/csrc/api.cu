// api.cu -- the C ABI of libq3tts (declared in include/q3tts.h): configuration
// checks, workspace layout, stream bookkeeping (lengths, KV pages, capacity),
// and dispatch to the frame kernels.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "engine.cuh"
#include "layers.cuh"

namespace q3 {
int sampler_setup();
int frame_kernel_create(q3tts_handle* h);
void frame_kernel_destroy(q3tts_handle* h);
bool frame_kernel_supports(const q3tts_handle* h, int n_active, const q3tts_sampling* sp);
int frame_kernel_recover(q3tts_handle* h);
int frame_kernel_step(q3tts_handle* h, const StepDesc& d, const float* uniforms, int32_t* codes,
                      const int32_t* forced, float* logits);
size_t frame_kernel_workspace(const q3tts_config& c, int n_sm);
int frame_kernel_static_check(const q3tts_handle* h, const q3tts_sampling& sp);
int frame_kernel_step_static(q3tts_handle* h, int sid, int pos, int newpage, const q3tts_sampling& sp,
                             const float* uniforms, int32_t* codes, const int32_t* forced, float* logits);
int frame_kernel_recover_static(q3tts_handle* h);
int frame_kernel_debug_fail(q3tts_handle* h, int barrier, int wait_us);
}  // namespace q3

namespace {

struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base((char*)b) {}
  template <class T>
  T* take(size_t count) {
    off = (off + 255) & ~(size_t)255;
    T* p = base ? (T*)(base + off) : nullptr;
    off += sizeof(T) * count;
    return p;
  }
};

bool pos_int(int v) { return v > 0; }

// A non-null pointer that is not 16-byte aligned (NULL passes: optional tensors).
bool misaligned16(const void* p) { return ((uintptr_t)p & 15u) != 0; }

int check_config(const q3tts_config* c) {
  if (!c) return Q3TTS_ERR_ARG;
  if (!pos_int(c->talker_layers) || !pos_int(c->talker_hidden) || !pos_int(c->talker_ffn) ||
      !pos_int(c->cp_layers) || !pos_int(c->cp_hidden) || !pos_int(c->cp_ffn) ||
      !pos_int(c->n_q_heads) || !pos_int(c->n_kv_heads) || !pos_int(c->head_dim) ||
      !pos_int(c->codec_vocab) || !pos_int(c->cp_vocab) || !pos_int(c->max_streams) ||
      !pos_int(c->kv_cap_steps) || !pos_int(c->page_size))
    return Q3TTS_ERR_ARG;
  if (c->n_codebooks != Q3TTS_N_CODEBOOKS) return Q3TTS_ERR_UNSUPPORTED;
  if (c->weight_dtype != Q3TTS_F32 && c->weight_dtype != Q3TTS_BF16 && c->weight_dtype != Q3TTS_FP8)
    return Q3TTS_ERR_ARG;
  if (c->kv_dtype != Q3TTS_F32 && c->kv_dtype != Q3TTS_BF16) return Q3TTS_ERR_ARG;
  if (c->n_q_heads % c->n_kv_heads) return Q3TTS_ERR_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return Q3TTS_ERR_UNSUPPORTED;
  // every matrix inner dimension is consumed 8 elements at a time
  if (c->talker_hidden % 8 || c->cp_hidden % 8 || c->talker_ffn % 8 || c->cp_ffn % 8)
    return Q3TTS_ERR_UNSUPPORTED;
  if (c->codec_vocab > 4096 || c->cp_vocab > 4096) return Q3TTS_ERR_UNSUPPORTED;
  if (c->max_streams > Q3TTS_MAX_STREAMS) return Q3TTS_ERR_UNSUPPORTED;
  if (c->kv_cap_steps < Q3TTS_N_CODEBOOKS) return Q3TTS_ERR_ARG;
  if (c->kv_pages < 0 || c->prefill_chunk < 0) return Q3TTS_ERR_ARG;
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f)) return Q3TTS_ERR_ARG;
  return Q3TTS_OK;
}

struct Dims {
  int Dt, Dc, Ft, Fc, Hq, Hkv, hd, Vt, Vc, qkv_rows, pps, n_pages, chunk, m_max, esz, kvesz, S;
};

Dims dims_of(const q3tts_config& c) {
  Dims d;
  d.Dt = c.talker_hidden; d.Dc = c.cp_hidden; d.Ft = c.talker_ffn; d.Fc = c.cp_ffn;
  d.Hq = c.n_q_heads; d.Hkv = c.n_kv_heads; d.hd = c.head_dim;
  d.Vt = c.codec_vocab; d.Vc = c.cp_vocab;
  d.qkv_rows = (d.Hq + 2 * d.Hkv) * d.hd;
  d.pps = (c.kv_cap_steps + c.page_size - 1) / c.page_size;
  d.S = c.max_streams;
  d.n_pages = c.kv_pages > 0 ? c.kv_pages : d.pps * d.S;
  // default prefill chunk: up to 1024 positions (long prompts read the
  // weights fewer times and give the attention more query tiles per launch)
  d.chunk = c.prefill_chunk > 0 ? c.prefill_chunk : std::min(std::max(c.kv_cap_steps, 16), 1024);
  d.m_max = std::max(d.chunk, 2 * d.S);
  d.esz = c.weight_dtype == Q3TTS_F32 ? 4 : (c.weight_dtype == Q3TTS_FP8 ? 1 : 2);  // matrix elements
  d.kvesz = c.kv_dtype == Q3TTS_F32 ? 4 : 2;
  return d;
}

// Carves the workspace (base == NULL: size only).
size_t carve(const q3tts_config& c, void* base, q3tts_handle* h) {
  Dims d = dims_of(c);
  Carver cv(base);
  const int D = std::max(d.Dt, d.Dc), F = std::max(d.Ft, d.Fc), V = std::max(d.Vt, d.Vc);
  float* rope_cos = cv.take<float>((size_t)c.kv_cap_steps * d.hd / 2);
  float* rope_sin = cv.take<float>((size_t)c.kv_cap_steps * d.hd / 2);
  char* kv_pool = cv.take<char>((size_t)c.talker_layers * d.n_pages * 2 * d.Hkv * c.page_size * d.hd * d.kvesz);
  int* page_table = cv.take<int>((size_t)d.S * d.pps);
  float* cpkv = cv.take<float>((size_t)c.cp_layers * d.S * 2 * d.Hkv * Q3TTS_N_CODEBOOKS * d.hd);
  int* cp_pt = cv.take<int>((size_t)d.S);
  float* pend_h = cv.take<float>((size_t)d.S * d.Dt);
  float* pend_l = cv.take<float>((size_t)d.S * d.Vt);
  uint8_t* hist = cv.take<uint8_t>((size_t)d.S * d.Vt);
  uint8_t* fin = cv.take<uint8_t>((size_t)d.S);
  int* sid = cv.take<int>(d.S);
  int* pos = cv.take<int>(d.S);
  q3tts_sampling* sp = cv.take<q3tts_sampling>(d.S);
  int* fed = cv.take<int>((size_t)d.S * Q3TTS_N_CODEBOOKS);
  int* tok_s = cv.take<int>(d.m_max);
  int* tok_p = cv.take<int>(d.m_max);
  float* x = cv.take<float>((size_t)d.m_max * d.Dt);
  float* hb = cv.take<float>((size_t)d.m_max * D);
  float* qkv = cv.take<float>((size_t)d.m_max * d.qkv_rows);
  float* att = cv.take<float>((size_t)d.m_max * d.Hq * d.hd);
  float* gu = cv.take<float>((size_t)d.m_max * 2 * F);
  float* act = cv.take<float>((size_t)d.m_max * F);
  const int Kx = std::max(std::max(D, F), d.Hq * d.hd);
  q3::bf16* xh = cv.take<q3::bf16>((size_t)d.m_max * Kx);
  q3::bf16* xl = cv.take<q3::bf16>((size_t)d.m_max * Kx);
  const int nsmax = q3::attention_split_spans(c.kv_cap_steps);
  float* spl_part = cv.take<float>((size_t)d.m_max * d.Hq * nsmax * (d.hd + 2));
  int* spl_cnt = cv.take<int>((size_t)d.m_max * d.Hkv);
  float* uin = cv.take<float>((size_t)2 * d.S * d.Dt);
  float* cpx = cv.take<float>((size_t)2 * d.S * d.Dc);
  float* logits = cv.take<float>((size_t)d.S * V);
  int* err = cv.take<int>(64);
  q3::StepDesc* desc = cv.take<q3::StepDesc>(1);
  float* g_uni = cv.take<float>((size_t)d.S * Q3TTS_N_CODEBOOKS);
  int32_t* g_forced = cv.take<int32_t>((size_t)d.S * Q3TTS_N_CODEBOOKS);
  int32_t* g_codes = cv.take<int32_t>((size_t)d.S * Q3TTS_N_CODEBOOKS);
  if (h) {
    h->rope_cos = rope_cos; h->rope_sin = rope_sin; h->kv_pool = kv_pool;
    h->page_table = page_table; h->cp_kv = cpkv; h->cp_page_table = cp_pt;
    h->pending_h = pend_h; h->pending_logits = pend_l; h->history = hist; h->finished = fin;
    h->d_sid = sid; h->d_pos = pos; h->d_sp = sp; h->d_fed = fed;
    h->d_tok_stream = tok_s; h->d_tok_pos = tok_p;
    h->x = x; h->hb = hb; h->qkv = qkv; h->att = att; h->gu = gu; h->act = act;
    h->xh = xh; h->xl = xl;
    h->spl_part = spl_part; h->spl_cnt = spl_cnt; h->spl_nsmax = nsmax;
    h->uin = uin; h->cpx = cpx; h->logits = logits; h->d_err = err;
    h->d_desc = desc; h->g_uni = g_uni; h->g_forced = g_forced; h->g_codes = g_codes;
  }
  cv.off = (cv.off + 255) & ~(size_t)255;
  return cv.off;
}

void free_stream_pages(q3tts_handle* h, int sid) {
  for (int p : h->pages[sid]) h->free_pages.push_back(p);
  h->pages[sid].clear();
}

bool check_sampling(const q3tts_sampling& p, int Vt) {
  if (p.do_sample && !(p.temperature > 0.f)) return false;
  if (p.sub_do_sample && !(p.sub_temperature > 0.f)) return false;
  if (!(p.top_p > 0.f) || !(p.sub_top_p > 0.f)) return false;
  if (!(p.repetition_penalty > 0.f)) return false;
  if (p.eos_token >= Vt || p.special_from > Vt) return false;
  return true;
}

// The controls as the kernels take them: with special codes masked, a
// disabled semantic top-k (<= 0 or >= the allowed count) keeps exactly the
// allowed codes, which the masked logits' order puts first.
q3tts_sampling device_sampling(const q3tts_sampling& p, int Vt) {
  q3tts_sampling d = p;
  if (p.special_from > 0 && p.special_from < Vt) {
    const int allowed = p.special_from + (p.eos_token >= p.special_from ? 1 : 0);
    if (d.top_k <= 0 || d.top_k >= allowed) d.top_k = allowed;
  } else {
    d.special_from = 0;
  }
  return d;
}

}  // namespace

extern "C" {

size_t q3tts_workspace_size(const q3tts_config* cfg) {
  if (check_config(cfg) != Q3TTS_OK) return 0;
  int dev = 0, n_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    n_sm = 0;
  return carve(*cfg, nullptr, nullptr) + q3::frame_kernel_workspace(*cfg, n_sm);
}

int q3tts_create(const q3tts_config* cfg, const q3tts_weights* w, void* workspace,
                 size_t workspace_bytes, void* cuda_stream, q3tts_handle** out) {
  if (out) *out = nullptr;
  int rc = check_config(cfg);
  if (rc != Q3TTS_OK) return rc;
  if (!w || !workspace || !out || !w->talker_layers || !w->cp_layers) return Q3TTS_ERR_ARG;
  if (((uintptr_t)workspace) & 255) return Q3TTS_ERR_ARG;
  const q3tts_config& c = *cfg;
  if (!w->talker_g_final || !w->talker_w_head || !w->talker_e_codec || !w->cp_g_final ||
      !w->cp_heads || !w->cp_embeds)
    return Q3TTS_ERR_ARG;
  if ((c.talker_hidden != c.cp_hidden) != (w->cp_w_proj != nullptr)) return Q3TTS_ERR_ARG;
  // every weight and gain is read with 16-byte vector loads or bulk copies
  if (misaligned16(w->talker_g_final) || misaligned16(w->talker_w_head) ||
      misaligned16(w->talker_e_codec) || misaligned16(w->cp_g_final) ||
      misaligned16(w->cp_heads) || misaligned16(w->cp_embeds) || misaligned16(w->cp_w_proj))
    return Q3TTS_ERR_ARG;
  for (int l = 0; l < c.talker_layers + c.cp_layers; ++l) {
    const q3tts_layer_weights& L =
        l < c.talker_layers ? w->talker_layers[l] : w->cp_layers[l - c.talker_layers];
    if (!L.w_qkv || !L.w_o || !L.w_gateup || !L.w_down || !L.g_attn_norm || !L.g_ffn_norm ||
        (c.qk_norm && (!L.g_q_norm || !L.g_k_norm)))
      return Q3TTS_ERR_ARG;
    if (misaligned16(L.w_qkv) || misaligned16(L.w_o) || misaligned16(L.w_gateup) ||
        misaligned16(L.w_down) || misaligned16(L.g_attn_norm) || misaligned16(L.g_ffn_norm) ||
        misaligned16(L.g_q_norm) || misaligned16(L.g_k_norm))
      return Q3TTS_ERR_ARG;
    // FP8 matrices come with their row scales
    if (c.weight_dtype == Q3TTS_FP8 && (!L.s_qkv || !L.s_o || !L.s_gateup || !L.s_down)) return Q3TTS_ERR_ARG;
  }
  if (c.weight_dtype == Q3TTS_FP8 && (!w->s_head || !w->s_cp_heads || (w->cp_w_proj && !w->s_cp_proj)))
    return Q3TTS_ERR_ARG;
  if (workspace_bytes < q3tts_workspace_size(cfg)) return Q3TTS_ERR_ARG;

  q3tts_handle* h = new (std::nothrow) q3tts_handle();
  if (!h) return Q3TTS_ERR_ARG;
  h->c = c;
  h->tl.assign(w->talker_layers, w->talker_layers + c.talker_layers);
  h->cl.assign(w->cp_layers, w->cp_layers + c.cp_layers);
  h->w = *w;
  h->w.talker_layers = h->tl.data();
  h->w.cp_layers = h->cl.data();
  h->s = (cudaStream_t)cuda_stream;
  h->fk = nullptr;
  if (cudaGetDevice(&h->dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->dev) != cudaSuccess) {
    delete h;
    return Q3TTS_ERR_CUDA;
  }
  Dims d = dims_of(c);
  h->Dt = d.Dt; h->Dc = d.Dc; h->Ft = d.Ft; h->Fc = d.Fc; h->Hq = d.Hq; h->Hkv = d.Hkv;
  h->hd = d.hd; h->Vt = d.Vt; h->Vc = d.Vc; h->qkv_rows = d.qkv_rows; h->pps = d.pps;
  h->n_pages = d.n_pages; h->chunk = d.chunk; h->m_max = d.m_max; h->esz = d.esz;
  h->fk_base = (char*)workspace + carve(c, nullptr, nullptr);
  carve(c, workspace, h);
  const char* env = getenv("Q3TTS_FRAME_KERNEL");
  h->frame_kernel_off = env && env[0] == '0';
  const char* genv = getenv("Q3TTS_GRAPH");
  h->graph_off = genv && genv[0] == '0';
  // the tensor-core projections: bf16 weights, every inner dimension a
  // multiple of 64 (Q3TTS_TC=0: the fp32-FMA kernels instead)
  const char* tenv = getenv("Q3TTS_TC");
  h->tc = !(tenv && tenv[0] == '0') && c.weight_dtype == Q3TTS_BF16 &&
          q3::tc_linear_ok(d.qkv_rows, d.Dt, 1) && q3::tc_linear_ok(d.qkv_rows, d.Dc, 1) &&
          q3::tc_linear_ok(d.Dt, d.Ft, 1) && q3::tc_linear_ok(d.Dc, d.Fc, 1) &&
          q3::tc_linear_ok(d.Dt, d.Hq * d.hd, 1);

  // RoPE tables: angle pos * theta^(-2i/hd), computed in double, stored as float.
  const int half = d.hd / 2;
  std::vector<float> cs((size_t)c.kv_cap_steps * half), sn((size_t)c.kv_cap_steps * half);
  for (int p = 0; p < c.kv_cap_steps; ++p)
    for (int i = 0; i < half; ++i) {
      double a = (double)p * pow((double)c.rope_theta, -2.0 * i / d.hd);
      cs[(size_t)p * half + i] = (float)cos(a);
      sn[(size_t)p * half + i] = (float)sin(a);
    }
  std::vector<int> cp_pt(d.S);
  for (int s = 0; s < d.S; ++s) cp_pt[s] = s;
  bool ok = cudaMemcpy(h->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(h->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemcpy(h->cp_page_table, cp_pt.data(), cp_pt.size() * 4, cudaMemcpyHostToDevice) == cudaSuccess &&
            cudaMemset(h->page_table, 0, sizeof(int) * (size_t)d.S * d.pps) == cudaSuccess &&
            cudaMemset(h->history, 0, (size_t)d.S * d.Vt) == cudaSuccess &&
            cudaMemset(h->finished, 0, (size_t)d.S) == cudaSuccess &&
            cudaMemset(h->d_err, 0, sizeof(int) * 64) == cudaSuccess &&
            cudaMemset(h->spl_cnt, 0, sizeof(int) * (size_t)d.m_max * d.Hkv) == cudaSuccess;
  for (cudaEvent_t& e : h->chunk_ev)
    ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
  if (!ok || q3::sampler_setup() != Q3TTS_OK) {
    for (cudaEvent_t& e : h->chunk_ev)
      if (e) cudaEventDestroy(e);
    delete h;
    return Q3TTS_ERR_CUDA;
  }
  h->len.assign(d.S, -1);
  h->pages.assign(d.S, std::vector<int>());
  h->free_pages.clear();
  for (int p = d.n_pages - 1; p >= 0; --p) h->free_pages.push_back(p);
  rc = q3::frame_kernel_create(h);
  if (rc != Q3TTS_OK) {
    for (cudaEvent_t& e : h->chunk_ev) cudaEventDestroy(e);
    delete h;
    return rc;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    q3::frame_kernel_destroy(h);
    for (cudaEvent_t& e : h->chunk_ev) cudaEventDestroy(e);
    delete h;
    return Q3TTS_ERR_CUDA;
  }
  *out = h;
  return Q3TTS_OK;
}

int q3tts_prefill(q3tts_handle* h, int sid, const float* embeds_dev, int len) {
  if (!h || !embeds_dev || sid < 0 || sid >= h->c.max_streams || len < 1) return Q3TTS_ERR_ARG;
  if (len >= h->c.kv_cap_steps) return Q3TTS_ERR_CAPACITY;
  const int ps = h->c.page_size;
  const int need = (len + ps - 1) / ps;
  free_stream_pages(h, sid);
  // the stream has no prompt until this call succeeds: an error below (pool
  // exhausted, a failed copy or launch) leaves it that way, never with its old
  // length over pages it no longer holds
  h->len[sid] = -1;
  if ((int)h->free_pages.size() < need) return Q3TTS_ERR_CAPACITY;
  std::vector<int> row(need);
  for (int i = 0; i < need; ++i) {
    row[i] = h->free_pages.back();
    h->free_pages.pop_back();
    h->pages[sid].push_back(row[i]);
  }
  cudaStream_t s = h->s;
  // pageable source: staged before the call returns, so `row` may go away
  if (cudaMemcpyAsync(h->page_table + (size_t)sid * h->pps, row.data(), sizeof(int) * need,
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemsetAsync(h->history + (size_t)sid * h->Vt, 0, h->Vt, s) != cudaSuccess ||
      cudaMemsetAsync(h->finished + sid, 0, 1, s) != cudaSuccess)
    return Q3TTS_ERR_CUDA;
  int rc = q3::prefill_layered(h, sid, embeds_dev, len);
  h->len[sid] = rc == Q3TTS_OK ? len : -1;
  return rc;
}

int q3tts_step_frame(q3tts_handle* h, const q3tts_sampling* params, const int32_t* stream_ids,
                     int n_active, const float* uniforms_dev, int32_t* codes_dev,
                     const int32_t* forced_dev, float* logits_dev) {
  if (!h || !params || !stream_ids || !uniforms_dev || !codes_dev) return Q3TTS_ERR_ARG;
  if (n_active < 1 || n_active > h->c.max_streams) return Q3TTS_ERR_ARG;
  static thread_local q3::StepDesc d;
  d.n = n_active;
  std::vector<char> seen(h->c.max_streams, 0);
  int pages_needed = 0;
  for (int b = 0; b < n_active; ++b) {
    int s = stream_ids[b];
    if (s < 0 || s >= h->c.max_streams || seen[s]) return Q3TTS_ERR_ARG;
    seen[s] = 1;
    if (!check_sampling(params[b], h->Vt)) return Q3TTS_ERR_ARG;
    if (h->len[s] < 1) return Q3TTS_ERR_STATE;
    if (h->len[s] >= h->c.kv_cap_steps) return Q3TTS_ERR_CAPACITY;
    if (h->len[s] / h->c.page_size >= (int)h->pages[s].size()) ++pages_needed;
  }
  if (pages_needed > (int)h->free_pages.size()) return Q3TTS_ERR_CAPACITY;
  // pages are picked from the top of the free list here and taken off it only
  // once the frame is launched, so a failed launch leaves every list as it was
  int taken = 0;
  for (int b = 0; b < n_active; ++b) {
    int s = stream_ids[b];
    d.sid[b] = s;
    d.pos[b] = h->len[s];
    d.sp[b] = device_sampling(params[b], h->Vt);
    d.newpage[b] = -1;
    if (h->len[s] / h->c.page_size >= (int)h->pages[s].size())
      d.newpage[b] = h->free_pages[h->free_pages.size() - 1 - taken++];
  }
  int rc;
  if (q3::frame_kernel_supports(h, n_active, d.sp))
    rc = q3::frame_kernel_step(h, d, uniforms_dev, codes_dev, forced_dev, logits_dev);
  else
    rc = q3::step_layered(h, d, uniforms_dev, codes_dev, forced_dev, logits_dev);
  if (rc != Q3TTS_OK) return rc;
  for (int b = 0; b < n_active; ++b) {
    if (d.newpage[b] >= 0) h->pages[stream_ids[b]].push_back(d.newpage[b]);
    h->len[stream_ids[b]] += 1;
  }
  h->free_pages.resize(h->free_pages.size() - taken);
  return Q3TTS_OK;
}

int q3tts_step_frames(q3tts_handle* h, const q3tts_sampling* params, const int32_t* stream_ids,
                      int n_active, int n_frames, const float* uniforms_dev, int32_t* codes_dev,
                      int32_t* codes_host, const int32_t* forced_dev) {
  if (!h || !params || !stream_ids || !uniforms_dev || !codes_dev) return Q3TTS_ERR_ARG;
  if (n_frames < 1 || n_frames > Q3TTS_MAX_CHUNK || n_active < 1 || n_active > h->c.max_streams)
    return Q3TTS_ERR_ARG;
  h->chunk_n = 0;
  const size_t per = (size_t)n_active * Q3TTS_N_CODEBOOKS;
  for (int f = 0; f < n_frames; ++f) {
    const int rc = q3tts_step_frame(h, params, stream_ids, n_active, uniforms_dev + f * per, codes_dev + f * per,
                                    forced_dev ? forced_dev + f * per : nullptr, nullptr);
    if (rc != Q3TTS_OK) return rc;
    if (codes_host && cudaMemcpyAsync(codes_host + f * per, codes_dev + f * per, per * sizeof(int32_t),
                                      cudaMemcpyDeviceToHost, h->s) != cudaSuccess)
      return Q3TTS_ERR_CUDA;
    if (cudaEventRecord(h->chunk_ev[f], h->s) != cudaSuccess) return Q3TTS_ERR_CUDA;
    h->chunk_n = f + 1;
  }
  return Q3TTS_OK;
}

int q3tts_frames_ready(q3tts_handle* h) {
  if (!h) return Q3TTS_ERR_ARG;
  int n = 0;
  while (n < h->chunk_n) {
    const cudaError_t e = cudaEventQuery(h->chunk_ev[n]);
    if (e == cudaErrorNotReady) {
      cudaGetLastError();
      break;
    }
    if (e != cudaSuccess) return Q3TTS_ERR_CUDA;
    ++n;
  }
  return n;
}

// Batch-1 frame with the persistent kernel's per-frame scratch in a static
// device array.  Validation and stream bookkeeping follow q3tts_step_frame,
// but nothing here allocates: no std::vector, no thread-local descriptor, and
// the page lists were reserved to their maximum length by the handle's first
// call, so pushing a page never grows them.
int q3tts_step_frame_static(q3tts_handle* h, const q3tts_sampling* params, int stream_id,
                            const float* uniforms_dev, int32_t* codes_dev,
                            const int32_t* forced_dev, float* logits_dev) {
  if (!h || !params || !uniforms_dev || !codes_dev) return Q3TTS_ERR_ARG;
  const int s = stream_id;
  if (s < 0 || s >= h->c.max_streams || !check_sampling(*params, h->Vt)) return Q3TTS_ERR_ARG;
  const q3tts_sampling sp = device_sampling(*params, h->Vt);
  int rc = q3::frame_kernel_static_check(h, sp);
  if (rc != Q3TTS_OK) return rc;
  if (h->len[s] < 1) return Q3TTS_ERR_STATE;
  if (h->len[s] >= h->c.kv_cap_steps) return Q3TTS_ERR_CAPACITY;
  if (!h->static_ready) {
    for (auto& v : h->pages) v.reserve(h->pps);
    h->static_ready = true;
  }
  const bool grow = h->len[s] / h->c.page_size >= (int)h->pages[s].size();
  if (grow && h->free_pages.empty()) return Q3TTS_ERR_CAPACITY;
  const int newpage = grow ? h->free_pages.back() : -1;
  rc = q3::frame_kernel_step_static(h, s, h->len[s], newpage, sp, uniforms_dev, codes_dev,
                                    forced_dev, logits_dev);
  if (rc != Q3TTS_OK) return rc;
  if (grow) {
    h->free_pages.pop_back();
    h->pages[s].push_back(newpage);
  }
  h->len[s] += 1;
  return Q3TTS_OK;
}

int q3tts_read_pending(q3tts_handle* h, int sid, float* hidden_dev, float* logits_dev) {
  if (!h || sid < 0 || sid >= h->c.max_streams) return Q3TTS_ERR_ARG;
  if (h->len[sid] < 1) return Q3TTS_ERR_STATE;
  if (hidden_dev &&
      cudaMemcpyAsync(hidden_dev, h->pending_h + (size_t)sid * h->Dt, sizeof(float) * h->Dt,
                      cudaMemcpyDeviceToDevice, h->s) != cudaSuccess)
    return Q3TTS_ERR_CUDA;
  if (logits_dev &&
      cudaMemcpyAsync(logits_dev, h->pending_logits + (size_t)sid * h->Vt, sizeof(float) * h->Vt,
                      cudaMemcpyDeviceToDevice, h->s) != cudaSuccess)
    return Q3TTS_ERR_CUDA;
  return Q3TTS_OK;
}

int q3tts_reset(q3tts_handle* h, int sid) {
  if (!h || sid < -1 || sid >= h->c.max_streams) return Q3TTS_ERR_ARG;
  int lo = sid < 0 ? 0 : sid, hi = sid < 0 ? h->c.max_streams : sid + 1;
  for (int s = lo; s < hi; ++s) {
    free_stream_pages(h, s);
    h->len[s] = -1;
  }
  size_t n = (size_t)(hi - lo) * h->Vt;
  if (cudaMemsetAsync(h->history + (size_t)lo * h->Vt, 0, n, h->s) != cudaSuccess ||
      cudaMemsetAsync(h->finished + lo, 0, (size_t)(hi - lo), h->s) != cudaSuccess)
    return Q3TTS_ERR_CUDA;
  return Q3TTS_OK;
}

int q3tts_stream_finished(q3tts_handle* h, int sid, int* finished) {
  if (!h || !finished || sid < 0 || sid >= h->c.max_streams) return Q3TTS_ERR_ARG;
  uint8_t f = 0;
  if (cudaMemcpyAsync(&f, h->finished + sid, 1, cudaMemcpyDeviceToHost, h->s) != cudaSuccess ||
      cudaStreamSynchronize(h->s) != cudaSuccess)
    return Q3TTS_ERR_CUDA;
  *finished = f ? 1 : 0;
  return Q3TTS_OK;
}

int q3tts_stream_length(q3tts_handle* h, int sid) {
  if (!h || sid < 0 || sid >= h->c.max_streams) return Q3TTS_ERR_ARG;
  return h->len[sid] < 0 ? 0 : h->len[sid];
}

int q3tts_sync_status(q3tts_handle* h) {
  if (!h) return Q3TTS_ERR_ARG;
  if (cudaStreamSynchronize(h->s) != cudaSuccess) return Q3TTS_ERR_CUDA;
  int e = 0;
  if (cudaMemcpy(&e, h->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return Q3TTS_ERR_CUDA;
  if (e != 0) {
    cudaMemset(h->d_err, 0, sizeof(int));
    q3::frame_kernel_recover(h);
    q3::frame_kernel_recover_static(h);
    cudaStreamSynchronize(h->s);
    return e;
  }
  return cudaGetLastError() == cudaSuccess ? Q3TTS_OK : Q3TTS_ERR_CUDA;
}

uint64_t q3tts_kernel_launches(const q3tts_handle* h) { return h ? h->launches : 0; }

int q3tts_debug_fail_barrier(q3tts_handle* h, int barrier, int wait_us) {
  if (!h || barrier < 0 || wait_us < 1 || wait_us > 2000000) return Q3TTS_ERR_ARG;
  return q3::frame_kernel_debug_fail(h, barrier, wait_us);
}

void q3tts_destroy(q3tts_handle* h) {
  if (!h) return;
  for (cudaEvent_t& e : h->chunk_ev)
    if (e) cudaEventDestroy(e);
  q3::frame_kernel_destroy(h);
  q3::step_graph_destroy(h);
  delete h;
}

const char* q3tts_strerror(int code) {
  switch (code) {
    case Q3TTS_OK: return "ok";
    case Q3TTS_ERR_ARG: return "invalid argument";
    case Q3TTS_ERR_CAPACITY: return "KV cache capacity exceeded";
    case Q3TTS_ERR_CUDA: return "CUDA runtime error";
    case Q3TTS_ERR_TIMEOUT: return "device-side wait timed out";
    case Q3TTS_ERR_UNSUPPORTED: return "unsupported configuration";
    case Q3TTS_ERR_STATE: return "stream has no prompt";
    case Q3TTS_ERR_SCRATCH: return "static scratch array too small for this configuration";
    default: return "unknown error";
  }
}

}  // extern "C"
