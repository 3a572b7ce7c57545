/*
 * q3tts.h -- C ABI of libq3tts: GB300 (sm_103a) frame decode of a
 * Qwen3-TTS-style model.
 *
 * One acoustic frame is 80 ms of audio, 16 codebook tokens [semantic token,
 * acoustic tokens 1..15]: the Talker (main decoder) produces the semantic
 * token, the CodePredictor fills in the 15 acoustic tokens of the same frame
 * one at a time, and the sum of the frame's 16 code embeddings is the next
 * Talker input.  ("Running Qwen3-TTS on an AMD R9700", section "Running
 * Qwen3-TTS"; embedding sum: "qwen3-tts-hip" README, section "Python Parity
 * Fixtures".)  The calls below mirror the engine surface of the "qwen3-tts-hip"
 * README, section "Library Usage": a model loaded once with a fixed KV-cache
 * capacity (EngineOptions::max_cache_steps), per-request sampling controls
 * (GenerateOptions) and persistent frame-incremental streams
 * (HipTtsEngine::start_stream), with errors returned as status codes.
 *
 * Conventions for every call:
 *   - All pointers documented "device" are CUDA device pointers in the
 *     current context; "host" pointers are ordinary host memory.
 *   - The library allocates no device memory.  The caller owns the weights
 *     and one workspace buffer (size from q3tts_workspace_size); both must
 *     outlive the handle.  The workspace holds the KV caches, per-stream state,
 *     activations and the library's re-laid-out copies of some weights.
 *   - Work is enqueued on the CUDA stream given to q3tts_create and is
 *     asynchronous unless stated; q3tts_sync_status waits for it.
 *   - Every call returns Q3TTS_OK (0) or a negative Q3TTS_ERR_* code.  Argument
 *     checks happen before anything is launched; no C++ exception and no abort
 *     crosses this boundary.
 */
#ifndef Q3TTS_H
#define Q3TTS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q3TTS_OK 0
#define Q3TTS_ERR_ARG (-1)         /* invalid argument, shape or pointer */
#define Q3TTS_ERR_CAPACITY (-2)    /* KV cache or page pool full; stream limit */
#define Q3TTS_ERR_CUDA (-3)        /* a CUDA runtime call failed */
#define Q3TTS_ERR_TIMEOUT (-4)     /* a device-side wait gave up (bounded spin) */
#define Q3TTS_ERR_UNSUPPORTED (-5) /* configuration outside what the kernels handle */
#define Q3TTS_ERR_STATE (-6)       /* e.g. a frame requested before prefill */
#define Q3TTS_ERR_SCRATCH (-7)     /* static scratch array too small (q3tts_step_frame_static) */

#define Q3TTS_F32 0
#define Q3TTS_BF16 1
/* Weight streaming in 8 bits: every matrix (w_qkv, w_o, w_gateup, w_down,
 * talker_w_head, cp_heads, cp_w_proj) holds FP8 E4M3 codes (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits, subnormals, no infinities; codes
 * 0x7f and 0xff are NaN), one byte per element, with one fp32 scale per output
 * row (the element is code value x scale); norm gains and embedding tables
 * stay bf16.  Weight dtype only. */
#define Q3TTS_FP8 2

#define Q3TTS_MAX_STREAMS 256
#define Q3TTS_N_CODEBOOKS 16
#define Q3TTS_MAX_CHUNK 64  /* frames one q3tts_step_frames call enqueues at most */

/* Size of the library's static device scratch array (768 KiB), used only by
 * q3tts_step_frame_static. */
#define Q3TTS_STATIC_SCRATCH_BYTES 786432

/* Model and engine shape.  Dimensions follow the Qwen3-style decoder: RMSNorm
 * (eps rms_eps), per-head q/k RMSNorm when qk_norm != 0, rotate-half RoPE
 * (base rope_theta), grouped-query attention (n_q_heads over n_kv_heads),
 * SwiGLU FFN.  The CodePredictor has the same head layout as the Talker.
 * kv_cap_steps is the per-stream Talker KV capacity in positions
 * (max_cache_steps); the KV cache is paged in pages of page_size positions
 * drawn from a pool of kv_pages pages shared by all streams (0 = enough for
 * max_streams full streams).  prefill_chunk bounds the positions one prefill
 * launch processes (0 = min(kv_cap_steps, 1024)). */
typedef struct q3tts_config {
  int talker_layers, talker_hidden, talker_ffn;
  int cp_layers, cp_hidden, cp_ffn;
  int n_q_heads, n_kv_heads, head_dim;
  int codec_vocab; /* V_t: Talker codec vocabulary (semantic token) */
  int cp_vocab;    /* V_c: vocabulary of each acoustic codebook */
  int n_codebooks; /* must be 16 */
  int max_streams, kv_cap_steps, page_size, kv_pages, prefill_chunk;
  int weight_dtype; /* Q3TTS_F32 or Q3TTS_BF16: every weight tensor; Q3TTS_FP8: the
                       matrices (gains and embeddings bf16) */
  int kv_dtype;     /* Talker KV cache: Q3TTS_F32 or Q3TTS_BF16 */
  int qk_norm;
  float rms_eps, rope_theta;
} q3tts_config;

/* One decoder layer; device pointers, row-major [out, in], weight_dtype.
 * With Q3TTS_FP8 the s_* arrays hold each matrix's per-output-row scales
 * (fp32, one per row: s_qkv [(Hq + 2 Hkv) hd], s_o [D], s_gateup [2 F],
 * s_down [D]) and the gains are bf16; otherwise the s_* pointers are unused.
 * Every weight and gain pointer (here and in q3tts_weights) must be 16-byte
 * aligned: the kernels read them with 16-byte vector loads and bulk copies.
 * q3tts_create returns Q3TTS_ERR_ARG for a pointer that is not, before it
 * launches or copies anything.
 *   w_qkv    [(Hq + 2 Hkv) hd, D]   q rows, then k rows, then v rows
 *   w_o      [D, Hq hd]
 *   w_gateup [2 F, D]                gate rows, then up rows
 *   w_down   [D, F]
 *   g_attn_norm [D], g_ffn_norm [D], g_q_norm [hd], g_k_norm [hd] */
typedef struct q3tts_layer_weights {
  const void* w_qkv;
  const void* w_o;
  const void* w_gateup;
  const void* w_down;
  const void* g_attn_norm;
  const void* g_ffn_norm;
  const void* g_q_norm;
  const void* g_k_norm;
  const float* s_qkv;
  const float* s_o;
  const float* s_gateup;
  const float* s_down;
} q3tts_layer_weights;

/* All weights.  talker_layers / cp_layers are HOST arrays of per-layer device
 * pointer sets (copied during q3tts_create).  Device tensors:
 *   talker_g_final [D_t], talker_w_head [V_t, D_t], talker_e_codec [V_t, D_t]
 *   cp_g_final [D_c], cp_heads [15, V_c, D_c], cp_embeds [15, V_c, D_t]
 *   cp_w_proj [D_c, D_t]: the CodePredictor input projection, required when
 *   D_t != D_c and NULL otherwise.
 * With Q3TTS_FP8: s_head [V_t], s_cp_heads [15 V_c], s_cp_proj [D_c] (NULL
 * when cp_w_proj is) are the scales of the FP8 heads and projection. */
typedef struct q3tts_weights {
  const q3tts_layer_weights* talker_layers;
  const void* talker_g_final;
  const void* talker_w_head;
  const void* talker_e_codec;
  const q3tts_layer_weights* cp_layers;
  const void* cp_g_final;
  const void* cp_heads;
  const void* cp_embeds;
  const void* cp_w_proj;
  const float* s_head;
  const float* s_cp_heads;
  const float* s_cp_proj;
} q3tts_weights;

/* Sampling controls of one stream ("qwen3-tts-hip" README, "Library Usage",
 * GenerateOptions): semantic token (do_sample, top_k, top_p, temperature,
 * repetition_penalty) and acoustic tokens (sub_*; no repetition penalty).
 * top_k <= 0 or >= vocabulary disables top-k; top_p >= 1 disables top-p;
 * temperature must be > 0 when sampling.  The rule applied, in float:
 * penalty over the stream's emitted semantic codes (l>0 ? l/rho : l*rho), then
 * greedy argmax (lowest index on ties) or: l/T, order by (value desc, index
 * asc), keep top-k, w = exp(l - max) in that order, optional top-p prefix,
 * pick the first id whose running float sum exceeds u * (float sum of w). */
typedef struct q3tts_sampling {
  int do_sample, top_k;
  float top_p, temperature, repetition_penalty;
  int sub_do_sample, sub_top_k;
  float sub_top_p, sub_temperature;
  /* Stop conditions (the README lists end-of-stream handling as open parity
   * work; this is the plainest reading).  eos_token >= 0: a frame whose fed
   * semantic code equals it ends the stream -- its codes are [c0, -1 x 15] --
   * and every later frame of the stream writes sixteen -1 (it is still
   * computed; the stream's state is undefined until q3tts_prefill or
   * q3tts_reset).  special_from > 0: semantic codes >= special_from other than
   * eos_token are never drawn (the draw runs over the allowed codes; a
   * disabled top-k keeps all of them).  eos_token < 0 and special_from <= 0:
   * no stop condition, every code may be drawn. */
  int eos_token, special_from;
} q3tts_sampling;

typedef struct q3tts_handle q3tts_handle;

/* *finished receives 1 if `stream` has fed its end-of-stream code since its
 * last prefill or reset, else 0.  Waits for the handle's stream (the flag is
 * written on the device).  Q3TTS_ERR_ARG for a bad stream id. */
int q3tts_stream_finished(q3tts_handle* h, int stream, int* finished);

/* Bytes of workspace q3tts_create needs for cfg (0 if cfg is invalid). */
size_t q3tts_workspace_size(const q3tts_config* cfg);

/* Counterpart of loading the engine once with a fixed KV-cache capacity
 * ("qwen3-tts-hip" README, "Library Usage": load_with_max_frames,
 * EngineOptions::max_cache_steps).
 * Builds a handle over caller-owned weights and workspace (device memory of at
 * least q3tts_workspace_size(cfg) bytes, 256-byte aligned).  cuda_stream is a
 * cudaStream_t (NULL = legacy default stream).  Uploads RoPE tables and the
 * library's re-laid-out weight copies into the workspace and synchronises
 * once.  On success *out receives the handle. */
int q3tts_create(const q3tts_config* cfg, const q3tts_weights* w, void* workspace,
                 size_t workspace_bytes, void* cuda_stream, q3tts_handle** out);

/* Counterpart of the engine's prompt-conditioned start of a stream
 * ("qwen3-tts-hip" README, "Library Usage": a model loaded with
 * load_with_max_frames / EngineOptions::max_cache_steps, then
 * start_stream over the prompt), with random prompt vectors standing in for
 * the text conditioning.
 * Restarts stream stream_id with a prompt: embeds_dev is a device fp32
 * [len, D_t] array of Talker input vectors for positions 0..len-1.  Writes
 * their KV and leaves the final-normed hidden and codec logits of position
 * len-1 as the stream's pending state, from which the next frame's semantic
 * token is drawn.  Q3TTS_ERR_CAPACITY if len >= kv_cap_steps or the page pool
 * is exhausted.  Argument errors and len >= kv_cap_steps leave the stream as
 * it was; any later error (page pool exhausted, a CUDA failure) leaves it
 * without a prompt, so its frames get Q3TTS_ERR_STATE until a prefill
 * succeeds. */
int q3tts_prefill(q3tts_handle* h, int stream_id, const float* embeds_dev, int len);

/* One acoustic frame as defined at the top of this header ("Running Qwen3-TTS
 * on an AMD R9700", section "Running Qwen3-TTS"): the semantic draw from the
 * pending Talker logits, 15 CodePredictor passes each ending in a head and a
 * draw, the sum of the 16 code embeddings, and one Talker step.  The draws
 * follow the GenerateOptions controls ("qwen3-tts-hip" README, "Library
 * Usage").
 * Decodes one frame for each of n_active streams (distinct ids, host array
 * stream_ids[n_active]; params: host array [n_active]).
 *   uniforms_dev     device fp32 [n_active, 16]: the uniform in [0,1) for each
 *                    draw (codebook order); ignored by greedy draws.
 *   codes_dev        device int32 [n_active, 16]: the drawn codes.
 *   forced_dev       NULL, or device int32 [n_active, 16]: teacher forcing --
 *                    these codes are fed forward instead of the drawn ones.
 *   logits_dev       NULL, or device fp32 [n_active, V_t + 15 V_c]: the raw
 *                    logits behind each draw (pending Talker logits, then the
 *                    15 CodePredictor heads).
 * Each stream advances by one Talker position.  Q3TTS_ERR_STATE if a stream
 * has no prompt, Q3TTS_ERR_CAPACITY if its cache is full.
 * Execution: one stream whose configuration and sampling settings the
 * persistent frame kernel covers runs as one launch of that kernel.  It covers
 * hidden sizes up to 2048 (multiples of 8; the CodePredictor's up to 1024),
 * at most 64 layers in all, power-of-two head sizes from 32 to 128 with at
 * most 2 query heads per KV head, power-of-two page sizes,
 * vocabularies up to 4096 (multiples of 4), and draws that are greedy or keep
 * at most 64 candidates (top_k 1..64).  Otherwise the frame runs layer by
 * layer, and without a logits dump that sequence is
 * captured into a CUDA graph on the first call for a given n_active (and
 * forced_dev NULL or not) and replayed on later calls, the inputs and codes
 * passing through buffers in the workspace.  Q3TTS_FRAME_KERNEL=0 and
 * Q3TTS_GRAPH=0 in the environment at q3tts_create turn either off. */
int q3tts_step_frame(q3tts_handle* h, const q3tts_sampling* params, const int32_t* stream_ids,
                     int n_active, const float* uniforms_dev, int32_t* codes_dev,
                     const int32_t* forced_dev, float* logits_dev);

/* Frame-incremental streaming, the counterpart of the engine's streaming
 * session ("qwen3-tts-hip" README, "Library Usage": start_stream, then
 * next_audio_chunk until the stream ends): enqueues n_frames (1 ..
 * Q3TTS_MAX_CHUNK) frames for the n_active streams back to back on the
 * handle's stream, with no host synchronisation between them, and copies each
 * frame's codes to host memory as soon as that frame is done.  The call
 * returns once the frames are enqueued; q3tts_frames_ready tells how many of
 * them have landed, so a caller double-buffers: enqueue chunk k + 1, then
 * consume chunk k.  Larger chunks cost fewer host round trips; smaller ones
 * deliver the first codes sooner.
 *   uniforms_dev  device fp32 [n_frames][n_active][16]
 *   codes_dev     device int32 [n_frames][n_active][16]
 *   codes_host    NULL, or host int32 [n_frames][n_active][16] (pinned memory
 *                 keeps the copies asynchronous); caller-owned, not read or
 *                 written by the host side of the library after the call
 *   forced_dev    NULL, or device int32 [n_frames][n_active][16] (teacher
 *                 forcing, as in q3tts_step_frame)
 * Frame f runs exactly as q3tts_step_frame would with the f-th slices.  A
 * frame that cannot be enqueued (e.g. Q3TTS_ERR_CAPACITY) stops the call with
 * that code; the frames before it stay enqueued and count as this chunk. */
int q3tts_step_frames(q3tts_handle* h, const q3tts_sampling* params, const int32_t* stream_ids,
                      int n_active, int n_frames, const float* uniforms_dev, int32_t* codes_dev,
                      int32_t* codes_host, const int32_t* forced_dev);

/* Frames of the latest q3tts_step_frames chunk whose codes have reached the
 * host buffer (codes_dev when no host buffer was given), counted in order;
 * does not block.  A negative value is an error code. */
int q3tts_frames_ready(q3tts_handle* h);

/* One frame of one stream, like q3tts_step_frame with n_active = 1, but with
 * the frame's scratch (residual vectors, QKV rows, attention partials,
 * CodePredictor logits, grid-barrier words) in a static device
 * array of Q3TTS_STATIC_SCRATCH_BYTES bytes compiled into the library instead
 * of the handle's workspace.  The method's description has no counterpart to
 * this call.  It exists for callers that must not allocate while decoding: a
 * real-time audio thread that cannot afford an allocator's locks or an
 * implicit device synchronisation, or a host embedding the library under a
 * fixed memory budget.  After the set-up below the call requests no device
 * memory and builds no host container (q3tts_step_frame builds a host-side
 * list per call).
 *   params           host, one q3tts_sampling; top_k must be in 1..64 for a
 *                    sampled draw (or the draw greedy), else
 *                    Q3TTS_ERR_UNSUPPORTED.
 *   stream_id        the stream to advance by one Talker position.
 *   uniforms_dev, codes_dev, forced_dev, logits_dev
 *                    as for q3tts_step_frame with n_active = 1.
 * Set-up: the first call on a device (from any handle) looks up the array's
 * device address with that device current, clears its barrier words and
 * synchronises the handle's stream once; the first call on a handle also
 * reserves its per-stream page lists (a host allocation).  Make one call
 * before any stream capture and before any code that must not allocate.
 * The barrier words must be zero when a frame starts: module load and the
 * set-up leave them zero, every completed frame leaves them zero, and
 * q3tts_sync_status clears them after a frame that reported an error.
 * The array is one per device and process, shared by every handle: calls
 * that overlap on the device (two streams, two threads, two handles) race on
 * it and corrupt each other's frames -- serialise them.
 * Errors, all returned before anything is launched and with the stream left
 * as it was: Q3TTS_ERR_ARG for a bad pointer, stream id or sampling value;
 * then the configuration checks -- Q3TTS_ERR_UNSUPPORTED if the persistent
 * frame kernel cannot run this handle or these sampling settings,
 * Q3TTS_ERR_SCRATCH if this configuration's scratch exceeds the array; then
 * Q3TTS_ERR_STATE / Q3TTS_ERR_CAPACITY as for q3tts_step_frame.  A failed
 * launch returns Q3TTS_ERR_CUDA; device-side errors are reported by
 * q3tts_sync_status. */
int q3tts_step_frame_static(q3tts_handle* h, const q3tts_sampling* params, int stream_id,
                            const float* uniforms_dev, int32_t* codes_dev,
                            const int32_t* forced_dev, float* logits_dev);

/* Copies a stream's pending state to device buffers (either may be NULL):
 * hidden_dev fp32 [D_t], logits_dev fp32 [V_t].  Asynchronous. */
int q3tts_read_pending(q3tts_handle* h, int stream_id, float* hidden_dev, float* logits_dev);

/* Forgets a stream (-1 = all): length, semantic history, pending state; its
 * KV pages return to the pool -- the end of a persistent stream of the
 * "qwen3-tts-hip" README ("Library Usage"), whose KV capacity is fixed by
 * max_cache_steps. */
int q3tts_reset(q3tts_handle* h, int stream_id);

/* Talker positions held by a stream (0 after reset), or a negative error. */
int q3tts_stream_length(q3tts_handle* h, int stream_id);

/* Waits for the handle's stream and reports any error recorded by a kernel
 * (Q3TTS_ERR_TIMEOUT for a device-side wait that gave up), or a CUDA error --
 * the status-code counterpart of the Result every engine call of the
 * "qwen3-tts-hip" README ("Library Usage") returns.  After a kernel error it
 * clears the error word and the frame kernels' barrier words, so the next
 * frame runs normally. */
int q3tts_sync_status(q3tts_handle* h);

/* Number of kernel launches this handle has issued since q3tts_create (a
 * diagnostic for launch-overhead accounting). */
uint64_t q3tts_kernel_launches(const q3tts_handle* h);

/* Test hook for the failure path (no counterpart in the method's
 * description): arms the handle's next persistent-kernel frame
 * (q3tts_step_frame with one stream, or q3tts_step_frame_static) so that CTA 0
 * leaves out its arrival at grid barrier `barrier` (0-based, in frame order)
 * and every device-side wait of that frame gives up after about wait_us
 * microseconds.  No GPU fault, trap or endless wait is involved: the other
 * CTAs' bounded waits run out, the kernel records Q3TTS_ERR_TIMEOUT, raises
 * its abort flag, lets its in-flight copies land and returns.
 * q3tts_sync_status then returns Q3TTS_ERR_TIMEOUT and clears the error and
 * barrier words; the decoded stream's state is undefined (prefill it again),
 * every other stream and the handle stay usable.  A barrier index past the
 * frame's last barrier arms nothing that fires, and the frame runs normally.
 * The arming covers exactly one launch.  Q3TTS_ERR_ARG for barrier < 0 or
 * wait_us outside 1..2,000,000; Q3TTS_ERR_UNSUPPORTED if this handle has no
 * persistent frame kernel. */
int q3tts_debug_fail_barrier(q3tts_handle* h, int barrier, int wait_us);

/* Releases the handle: its host state, events and captured graphs.  It does
 * not wait for work queued on the handle's stream, so call q3tts_sync_status
 * first if the workspace or the weights are freed right after; neither is
 * touched by this call (both stay caller-owned).  NULL is a no-op. */
void q3tts_destroy(q3tts_handle* h);

/* A static, never-NULL description of a status code ("unknown error" for a
 * code this library does not return). */
const char* q3tts_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* Q3TTS_H */
