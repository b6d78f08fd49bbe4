// internal.h -- declarations shared by the library's translation units.
// Not part of the public C ABI (that is include/logmel.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "logmel.h"

namespace lm {

// Per-device facts the launchers need, queried once per device.
struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int max_smem_optin = 0;  // bytes of dynamic shared memory a block may opt into
};

// Fills `info` for the current device.  Returns LM_ERR_CUDA on failure.
lm_status current_device_info(DeviceInfo *info);

// Records a failed CUDA call for lm_last_cuda_error() and maps it to a status.
lm_status cuda_fail(cudaError_t e);

// Checks the result of a CUDA call; on failure records it and returns LM_ERR_CUDA.
#define LM_CUDA_TRY(expr)                               \
  do {                                                  \
    cudaError_t lm_e_ = (expr);                         \
    if (lm_e_ != cudaSuccess) return ::lm::cuda_fail(lm_e_); \
  } while (0)

// Sets a kernel's dynamic shared memory limit once per (kernel, device).
lm_status ensure_smem_attribute(const void *kernel, int bytes);

// Every workspace starts with a 16-byte header whose first u32 is the
// device error word (bit flags set by kernels whose bounded waits ran out).
constexpr size_t kWorkspaceHeaderBytes = 16;

// Reads an environment override once; returns `fallback` when unset.
const char *env_or(const char *name, const char *fallback);

// A token that names one launch: nonzero and never repeated in this process
// (a 64-bit counter started at a random value).  Kernels that get one clear
// the workspace words that must start at zero themselves and publish the
// token once they have; peers wait for it before their first access, so the
// call needs no memset in front of it.  Returns 0 -- clear the workspace
// with a memset -- while `stream` is being captured into a graph (a token
// baked into a graph would repeat on every replay) or when the query fails.
uint64_t call_token(cudaStream_t stream);

// --- log_mel_from_stft -----------------------------------------------------

// Workspace bytes of lm_log_mel_from_stft for this shape.
size_t stft_workspace_bytes(int64_t B, int64_t F, int32_t NF, int32_t NM);

// Fault injection for tests of the bounded waits: the maximum of tile
// `withhold_tile` is never published, and the resolver gives up waiting for
// a clip maximum after `clip_wait_ns`.
struct StftFault {
  uint64_t clip_wait_ns;
  int64_t withhold_tile;
};

// Validated launch; arguments as in lm_log_mel_from_stft.  `err_word`, when
// set, receives the kernel's error bits instead of the workspace header (a
// device u32 the caller clears).  `fault` is null outside tests.
lm_status stft_logmel_run(const void *stft, const float *filters, float *out, int64_t B, int64_t F,
                          int32_t NF, int32_t NM, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream,
                          const void *packed = nullptr, uint32_t *err_word = nullptr,
                          const StftFault *fault = nullptr);

// Per-clip floor and rescale in place: out[b] = (max(out[b], hi_b - 8) + 4) / 4,
// hi_b = the largest of the clip's tiles_per_clip order-preserving keys.
lm_status launch_clip_clamp(float *out, const uint32_t *tile_key, int64_t B, int64_t per_clip,
                            int32_t tiles_per_clip, cudaStream_t stream);

lm_status stft_describe(int64_t B, int64_t F, int32_t NF, int32_t NM, lm_stft_launch_info *info);

// --- mel_spectrogram ----------------------------------------------------------

// Argument rules of lm_mel_spectrogram that need no pointers.
lm_status mel_spectrogram_check(const lm_mel_plan *plan, int32_t in_dtype, int64_t B, int64_t T,
                                int32_t out_dtype);

// The plan's number of mel bands.
lm_status mel_plan_n_mels(const lm_mel_plan *plan, int32_t *n_mels);

// Validated launch; arguments as in lm_mel_spectrogram, plus `err_word` as
// for stft_logmel_run.
lm_status mel_spectrogram_run(const lm_mel_plan *plan, const void *wave, int32_t in_dtype, int64_t B,
                              int64_t T, void *out, int32_t out_dtype, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream, uint32_t *err_word = nullptr);

}  // namespace lm
