// engine.cuh -- the handle behind the C ABI and the workspace layout.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "common.cuh"
#include "q3tts.h"

namespace q3 {

// Per-call description of a frame step, passed by value to the set-up kernel.
struct StepDesc {
  int n;
  int sid[Q3TTS_MAX_STREAMS];       // stream id of active slot b
  int pos[Q3TTS_MAX_STREAMS];       // Talker position the frame writes
  int newpage[Q3TTS_MAX_STREAMS];   // page id to enter at pos / page_size, or -1
  q3tts_sampling sp[Q3TTS_MAX_STREAMS];
};

struct FrameKernelState;  // persistent frame kernel (frame_kernel.cu)

}  // namespace q3

struct q3tts_handle {
  q3tts_config c;
  std::vector<q3tts_layer_weights> tl, cl;
  q3tts_weights w;
  cudaStream_t s;
  int dev, n_sm;

  // dimensions
  int Dt, Dc, Ft, Fc, Hq, Hkv, hd, Vt, Vc, qkv_rows, pps, n_pages, chunk, m_max, esz;

  // workspace carve-up
  float* rope_cos;  // [kv_cap][hd/2]
  float* rope_sin;
  void* kv_pool;    // Talker KV, paged
  int* page_table;  // [max_streams][pps]
  float* cp_kv;     // CodePredictor KV: one 16-slot page per stream, fp32
  int* cp_page_table;
  float* pending_h;       // [max_streams][D_t]
  float* pending_logits;  // [max_streams][V_t]
  uint8_t* history;       // [max_streams][V_t]
  uint8_t* finished;      // [max_streams]: the stream fed its end-of-stream code
  int* d_sid;             // [max_streams]
  int* d_pos;
  q3tts_sampling* d_sp;
  int* d_fed;             // [max_streams][16] codes fed forward
  int* d_tok_stream;      // [m_max]
  int* d_tok_pos;         // [m_max]
  float *x, *hb, *qkv, *att, *gu, *act, *uin, *cpx, *logits;
  // hi/lo bf16 terms of the activations the tensor-core projections read
  // ([m_max][K] each); tc: bf16 weights whose every inner dimension is a
  // multiple of 64 take that path (Q3TTS_TC=0 turns it off)
  q3::bf16 *xh, *xl;
  bool tc = false;
  bool tc_failed = false;  // a projection could not be launched
  // split-context attention: span results [m_max][Hq][spl_nsmax][hd + 2] and
  // per-(token, kv head) counters [m_max][Hkv] (zero between launches)
  float* spl_part;
  int* spl_cnt;
  int spl_nsmax;
  int* d_err;
  // layered step replayed as a CUDA graph: the step's descriptor and its
  // per-call inputs/outputs pass through these fixed device buffers
  q3::StepDesc* d_desc;
  float* g_uni;      // [max_streams][16]
  int32_t* g_forced;  // [max_streams][16]
  int32_t* g_codes;   // [max_streams][16]

  // host-side stream bookkeeping
  std::vector<int> len;  // Talker positions held; -1 = no prompt yet
  std::vector<std::vector<int>> pages;
  std::vector<int> free_pages;

  q3::FrameKernelState* fk;
  char* fk_base;           // workspace region of the persistent frame kernel
  bool frame_kernel_off;   // Q3TTS_FRAME_KERNEL=0: always use the layered step
  bool used_static = false;   // q3tts_step_frame_static has run on this handle
  // failure-path test (q3tts_debug_fail_barrier), armed for one persistent launch
  int dbg_fail_bar = -1;
  long long dbg_wait_cycles = 0;
  bool static_ready = false;  // per-stream page lists reserved for it
  uint64_t launches = 0;
  // streaming chunks (q3tts_step_frames): one event per frame, recorded after
  // the frame's codes are copied out
  cudaEvent_t chunk_ev[Q3TTS_MAX_CHUNK] = {};
  int chunk_n = 0;
  // the captured layered step (valid for g_n active streams, with or without
  // forced codes); g_launches kernels per replay
  cudaGraphExec_t gexec = nullptr;
  int g_n = 0;
  bool g_forced_on = false;
  uint64_t g_launches = 0;
  cudaStream_t cap_stream = nullptr;  // stream the step is captured on
  bool graph_off = false;             // Q3TTS_GRAPH=0: launch the layered step kernel by kernel
};

namespace q3 {

// Layered frame step (one kernel per operation), any number of streams.
int step_layered(q3tts_handle* h, const StepDesc& d, const float* uniforms, int32_t* codes,
                 const int32_t* forced, float* logits);
int prefill_layered(q3tts_handle* h, int sid, const float* embeds, int len);
void step_graph_destroy(q3tts_handle* h);

KVDesc talker_kv(const q3tts_handle* h);
KVDesc cp_kv(const q3tts_handle* h);

}  // namespace q3
