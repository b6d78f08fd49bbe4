// wave_mel.cu -- waveform -> mel spectrogram (placeholder entry points until
// the FFT kernel lands; every call reports LM_ERR_UNSUPPORTED).
#include "internal.h"

extern "C" lm_status lm_mel_plan_create(const lm_mel_params *params, lm_mel_plan **plan) {
  if (!params || !plan) return LM_ERR_INVALID_ARG;
  *plan = nullptr;
  return LM_ERR_UNSUPPORTED;
}
extern "C" lm_status lm_mel_plan_destroy(lm_mel_plan *plan) { return plan ? LM_ERR_UNSUPPORTED : LM_OK; }
extern "C" lm_status lm_mel_n_frames(const lm_mel_plan *plan, int64_t T, int64_t *n_frames) {
  (void)T;
  if (!plan || !n_frames) return LM_ERR_INVALID_ARG;
  return LM_ERR_UNSUPPORTED;
}
extern "C" lm_status lm_mel_workspace_size(const lm_mel_plan *plan, int64_t B, size_t *bytes) {
  (void)B;
  if (!plan || !bytes) return LM_ERR_INVALID_ARG;
  return LM_ERR_UNSUPPORTED;
}
extern "C" lm_status lm_mel_spectrogram(const lm_mel_plan *plan, const void *wave, int32_t in_dtype, int64_t B,
                                        int64_t T, void *out, int32_t out_dtype, void *workspace,
                                        size_t workspace_bytes, lm_stream_t stream) {
  (void)wave; (void)in_dtype; (void)B; (void)T; (void)out; (void)out_dtype; (void)workspace;
  (void)workspace_bytes; (void)stream;
  if (!plan) return LM_ERR_INVALID_ARG;
  return LM_ERR_UNSUPPORTED;
}
