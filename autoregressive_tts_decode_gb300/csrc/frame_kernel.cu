// frame_kernel.cu -- persistent whole-frame kernel (placeholder until built).
#include "engine.cuh"

namespace q3 {
size_t frame_kernel_workspace(const q3tts_config&, int) { return 0; }
int frame_kernel_create(q3tts_handle*) { return Q3TTS_OK; }
void frame_kernel_destroy(q3tts_handle*) {}
bool frame_kernel_supports(const q3tts_handle*, int) { return false; }
int frame_kernel_step(q3tts_handle*, const StepDesc&, const float*, int32_t*, const int32_t*,
                      float*) {
  return Q3TTS_ERR_UNSUPPORTED;
}
}  // namespace q3
