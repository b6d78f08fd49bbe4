/*
 * c_abi_consumer.c -- a plain C99 program that drives liblogmel.so through
 * include/logmel.h alone (no Python, no torch), as a C or C++ host
 * application would.  tests/test_c_consumer.py builds and runs it.
 *
 * Usage: c_abi_consumer DIR
 *   DIR/stft.bin      B*F*NF complex64 (interleaved f32 pairs)
 *   DIR/filters.bin   NM*NF f32
 *   DIR/wave.bin      WB*WT f32
 *   DIR/shape.txt     "B F NF NM WB WT"
 * Writes DIR/out_device.bin (lm_log_mel_from_stft), DIR/out_host.bin
 * (lm_log_mel_from_stft_host from pageable host buffers) and DIR/mel.bin
 * (lm_mel_spectrogram, Whisper parameters, log).  Exit status 0 on success;
 * any failure prints the call and its status.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "logmel.h"

#define CHECK_LM(call)                                                                   \
  do {                                                                                   \
    lm_status st_ = (call);                                                              \
    if (st_ != LM_OK) {                                                                  \
      fprintf(stderr, "%s failed: %s (cuda %d)\n", #call, lm_status_string(st_),         \
              lm_last_cuda_error());                                                     \
      return 1;                                                                          \
    }                                                                                    \
  } while (0)

#define CHECK_CUDA(call)                                                                 \
  do {                                                                                   \
    cudaError_t e_ = (call);                                                             \
    if (e_ != cudaSuccess) {                                                             \
      fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));                 \
      return 1;                                                                          \
    }                                                                                    \
  } while (0)

static void *read_file(const char *dir, const char *name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (!f) return NULL;
  void *p = malloc(bytes ? bytes : 1);
  if (p && fread(p, 1, bytes, f) != bytes) {
    free(p);
    p = NULL;
  }
  fclose(f);
  return p;
}

static int write_file(const char *dir, const char *name, const void *p, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (!f) return 1;
  const int bad = fwrite(p, 1, bytes, f) != bytes;
  return fclose(f) != 0 || bad;
}

int main(int argc, char **argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s DIR\n", argv[0]);
    return 2;
  }
  const char *dir = argv[1];
  long long B, F, NF, NM, WB, WT;
  {
    char path[4096];
    snprintf(path, sizeof path, "%s/shape.txt", dir);
    FILE *f = fopen(path, "r");
    if (!f || fscanf(f, "%lld %lld %lld %lld %lld %lld", &B, &F, &NF, &NM, &WB, &WT) != 6) {
      fprintf(stderr, "cannot read %s\n", path);
      return 2;
    }
    fclose(f);
  }
  const size_t stft_bytes = (size_t)(B * F * NF) * 8, filt_bytes = (size_t)(NM * NF) * 4;
  const size_t out_bytes = (size_t)(B * F * NM) * 4, wave_bytes = (size_t)(WB * WT) * 4;
  void *h_stft = read_file(dir, "stft.bin", stft_bytes);
  void *h_filt = read_file(dir, "filters.bin", filt_bytes);
  void *h_wave = read_file(dir, "wave.bin", wave_bytes);
  float *h_out = (float *)malloc(out_bytes);
  float *h_out2 = (float *)malloc(out_bytes);
  if (!h_stft || !h_filt || !h_wave || !h_out || !h_out2) {
    fprintf(stderr, "input files missing or short\n");
    return 2;
  }
  printf("liblogmel version %d\n", lm_version());

  cudaStream_t stream;
  CHECK_CUDA(cudaStreamCreate(&stream));
  lm_stream_t s = (lm_stream_t)stream;

  /* 1. device buffers */
  void *d_stft = NULL, *d_ws = NULL;
  float *d_filt = NULL, *d_out = NULL;
  size_t ws_bytes = 0;
  CHECK_LM(lm_log_mel_from_stft_workspace_size(B, F, (int32_t)NF, (int32_t)NM, &ws_bytes));
  CHECK_CUDA(cudaMalloc(&d_stft, stft_bytes));
  CHECK_CUDA(cudaMalloc((void **)&d_filt, filt_bytes));
  CHECK_CUDA(cudaMalloc((void **)&d_out, out_bytes));
  CHECK_CUDA(cudaMalloc(&d_ws, ws_bytes));
  CHECK_CUDA(cudaMemcpyAsync(d_stft, h_stft, stft_bytes, cudaMemcpyHostToDevice, stream));
  CHECK_CUDA(cudaMemcpyAsync(d_filt, h_filt, filt_bytes, cudaMemcpyHostToDevice, stream));
  CHECK_LM(lm_log_mel_from_stft(d_stft, d_filt, d_out, B, F, (int32_t)NF, (int32_t)NM, d_ws, ws_bytes, s));
  uint32_t device_error = 0;
  CHECK_LM(lm_workspace_error(d_ws, ws_bytes, &device_error, s));
  CHECK_CUDA(cudaMemcpy(h_out, d_out, out_bytes, cudaMemcpyDeviceToHost));
  if (write_file(dir, "out_device.bin", h_out, out_bytes)) return 3;

  /* 2. host buffers (pageable), pipelined by the library in 2-clip chunks */
  size_t hws_bytes = 0;
  void *d_hws = NULL;
  CHECK_LM(lm_log_mel_from_stft_host_workspace_size(B, F, (int32_t)NF, (int32_t)NM, 2, &hws_bytes));
  CHECK_CUDA(cudaMalloc(&d_hws, hws_bytes));
  CHECK_LM(lm_log_mel_from_stft_host(h_stft, d_filt, NULL, h_out2, B, F, (int32_t)NF, (int32_t)NM, 2, d_hws,
                                     hws_bytes, s));
  CHECK_CUDA(cudaStreamSynchronize(stream));
  CHECK_LM(lm_workspace_error(d_hws, hws_bytes, &device_error, s));
  if (memcmp(h_out, h_out2, out_bytes) != 0) {
    fprintf(stderr, "host-buffer result differs from the device result\n");
    return 4;
  }
  if (write_file(dir, "out_host.bin", h_out2, out_bytes)) return 3;

  /* 3. waveform -> Whisper log-mel */
  lm_mel_params p;
  memset(&p, 0, sizeof p);
  p.sample_rate = 16000;
  p.n_fft = 400;
  p.hop_length = 160;
  p.n_mels = 80;
  p.f_max = 8000.0f;
  p.center = 1;
  p.pad_mode = LM_PAD_REFLECT;
  p.power = 2.0f;
  p.mel_scale = LM_MEL_HTK;
  p.log_mel = 1;
  lm_mel_plan *plan = NULL;
  CHECK_LM(lm_mel_plan_create(&p, &plan));
  int64_t n_frames = 0;
  size_t mws_bytes = 0;
  CHECK_LM(lm_mel_n_frames(plan, WT, &n_frames));
  CHECK_LM(lm_mel_workspace_size(plan, WB, WT, &mws_bytes));
  const size_t mel_bytes = (size_t)(WB * p.n_mels * n_frames) * 4;
  void *d_wave = NULL, *d_mel = NULL, *d_mws = NULL;
  CHECK_CUDA(cudaMalloc(&d_wave, wave_bytes));
  CHECK_CUDA(cudaMalloc(&d_mel, mel_bytes));
  CHECK_CUDA(cudaMalloc(&d_mws, mws_bytes));
  CHECK_CUDA(cudaMemcpyAsync(d_wave, h_wave, wave_bytes, cudaMemcpyHostToDevice, stream));
  CHECK_LM(lm_mel_spectrogram(plan, d_wave, LM_F32, WB, WT, d_mel, LM_F32, d_mws, mws_bytes, s));
  CHECK_LM(lm_workspace_error(d_mws, mws_bytes, &device_error, s));
  float *h_mel = (float *)malloc(mel_bytes);
  if (!h_mel) return 2;
  CHECK_CUDA(cudaMemcpy(h_mel, d_mel, mel_bytes, cudaMemcpyDeviceToHost));
  if (write_file(dir, "mel.bin", h_mel, mel_bytes)) return 3;
  CHECK_LM(lm_mel_plan_destroy(plan));

  cudaFree(d_stft);
  cudaFree(d_filt);
  cudaFree(d_out);
  cudaFree(d_ws);
  cudaFree(d_hws);
  cudaFree(d_wave);
  cudaFree(d_mel);
  cudaFree(d_mws);
  cudaStreamDestroy(stream);
  free(h_stft);
  free(h_filt);
  free(h_wave);
  free(h_out);
  free(h_out2);
  free(h_mel);
  printf("ok %lld frames\n", (long long)n_frames);
  return 0;
}
