/*
 * logmel_oracle.c -- the CPU oracle for the log-mel front end.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; it exists so the tests, the smoke check and the benchmark's
 * CPU baseline have an obviously correct answer to compare against.  It shares
 * no code, header, table or constant generator with the CUDA library.
 *
 * Every quantity is computed in double from the f32/i16 inputs and rounded to
 * the output type once, at the end.  Loops are the plain definitions: a dense
 * mel projection over every bin, an O(N^2) DFT, an explicitly materialised
 * padded signal.  Parallelism is OpenMP over independent clips only.
 *
 * Sources (page title, then the part of the page):
 *  - "audio_mel_spectrogram_fused.py" (KBench task spec), the reference
 *    function and the five-line per-clip definition in its spec text:
 *    power, mel projection, log10 of the value floored at 1e-10, per-clip max,
 *    clamp at max - 8 and the (x + 4) / 4 rescale.
 *  - "flashmel" (PyPI page), its usage and argument list: torchaudio-style
 *    MelSpectrogram with center/pad_mode framing, periodic Hann window,
 *    one-sided real FFT, |X|^power, mel filterbank (HTK or Slaney scale,
 *    optional Slaney area norm), int16 input scaled by 1/32768, f16 output.
 *
 * Readings where the pages are silent:
 *  - mel scale formulas are the textbook HTK and Slaney definitions;
 *  - the filterbank's frequency grid is bin k <-> k * (sr/2) / (n_freqs-1),
 *    with triangles in Hz between mel-spaced points;
 *  - "reflect" does not repeat the edge sample;
 *  - the clip maximum on the waveform log path runs over (n_mels, n_frames).
 *
 * Parity pins live in tests/test_oracle_*.py; every function here has at
 * least one check that does not go through this file's own formulas.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEM 2

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* log-mel from a complex STFT (KBench spec, per-clip definition).           */
/* ------------------------------------------------------------------------ */

/* One clip: stft[F][NF] interleaved (re, im) f32 pairs; filters[NM][NF] f32;
 * writes ls[F][NM] = log10(max(mel, 1e-10)) in double and returns the clip max. */
static double clip_log_spec(const float *stft, const float *filters, int64_t F, int64_t NF,
                            int64_t NM, double *mag, double *ls) {
  double hi = -INFINITY;
  for (int64_t f = 0; f < F; ++f) {
    const float *row = stft + 2 * f * NF;
    for (int64_t k = 0; k < NF; ++k) {
      double re = (double)row[2 * k], im = (double)row[2 * k + 1];
      mag[k] = re * re + im * im; /* power, not magnitude */
    }
    for (int64_t n = 0; n < NM; ++n) {
      double mel = 0.0;
      for (int64_t k = 0; k < NF; ++k) mel += mag[k] * (double)filters[n * NF + k];
      double v = log10(mel > 1e-10 ? mel : 1e-10); /* floor before the log */
      ls[f * NM + n] = v;
      if (v > hi) hi = v;
    }
  }
  return hi;
}

/* out[B][F][NM] f32.  Returns ORACLE_OK or an error code. */
int oracle_log_mel_from_stft(const float *stft, const float *filters, int64_t B, int64_t F,
                             int64_t NF, int64_t NM, float *out) {
  if (!stft || !filters || !out || B < 0 || F < 0 || NF < 1 || NM < 1) return ORACLE_BAD_ARG;
  int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t b = 0; b < B; ++b) {
    double *mag = (double *)malloc(sizeof(double) * (size_t)NF);
    double *ls = (double *)malloc(sizeof(double) * (size_t)(F * NM + 1));
    if (!mag || !ls) {
      err = ORACLE_NO_MEM;
    } else {
      double hi = clip_log_spec(stft + 2 * b * F * NF, filters, F, NF, NM, mag, ls);
      double floor_v = hi - 8.0; /* 80 dB below the clip's loudest band */
      for (int64_t i = 0; i < F * NM; ++i) {
        double v = ls[i] > floor_v ? ls[i] : floor_v;
        out[b * F * NM + i] = (float)((v + 4.0) / 4.0);
      }
    }
    free(mag);
    free(ls);
  }
  return err;
}

/* Deliberately WRONG variants, used only by the negative tests to show the
 * comparison gate is tight enough to reject them:
 *   scope 1 = clamp per frame instead of per clip,
 *   scope 2 = clamp per batch (one max over all clips),
 *   bf16_projection = round the power and the filter to bf16 before the
 *   projection. */
static float round_to_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u = (u + 0x7fffu + lsb) & 0xffff0000u; /* round to nearest even on the upper 16 bits */
  memcpy(&f, &u, 4);
  return f;
}

int oracle_log_mel_from_stft_wrong(const float *stft, const float *filters, int64_t B, int64_t F,
                                   int64_t NF, int64_t NM, int scope, int bf16_projection,
                                   float *out) {
  if (!stft || !filters || !out || B < 1 || F < 1 || NF < 1 || NM < 1) return ORACLE_BAD_ARG;
  double *ls = (double *)malloc(sizeof(double) * (size_t)(B * F * NM));
  double *mag = (double *)malloc(sizeof(double) * (size_t)NF);
  if (!ls || !mag) {
    free(ls);
    free(mag);
    return ORACLE_NO_MEM;
  }
  for (int64_t b = 0; b < B; ++b)
    for (int64_t f = 0; f < F; ++f) {
      const float *row = stft + 2 * (b * F + f) * NF;
      for (int64_t k = 0; k < NF; ++k) {
        double re = row[2 * k], im = row[2 * k + 1];
        mag[k] = re * re + im * im;
        if (bf16_projection) mag[k] = round_to_bf16(mag[k]);
      }
      for (int64_t n = 0; n < NM; ++n) {
        double mel = 0.0;
        for (int64_t k = 0; k < NF; ++k) {
          double w = filters[n * NF + k];
          if (bf16_projection) w = round_to_bf16(w);
          mel += mag[k] * w;
        }
        ls[(b * F + f) * NM + n] = log10(mel > 1e-10 ? mel : 1e-10);
      }
    }
  double batch_hi = -INFINITY;
  for (int64_t i = 0; i < B * F * NM; ++i)
    if (ls[i] > batch_hi) batch_hi = ls[i];
  for (int64_t b = 0; b < B; ++b) {
    double clip_hi = -INFINITY;
    for (int64_t i = 0; i < F * NM; ++i)
      if (ls[b * F * NM + i] > clip_hi) clip_hi = ls[b * F * NM + i];
    for (int64_t f = 0; f < F; ++f) {
      double hi = clip_hi;
      if (scope == 1) {
        hi = -INFINITY;
        for (int64_t n = 0; n < NM; ++n)
          if (ls[(b * F + f) * NM + n] > hi) hi = ls[(b * F + f) * NM + n];
      } else if (scope == 2) {
        hi = batch_hi;
      }
      for (int64_t n = 0; n < NM; ++n) {
        double v = ls[(b * F + f) * NM + n];
        if (v < hi - 8.0) v = hi - 8.0;
        out[(b * F + f) * NM + n] = (float)((v + 4.0) / 4.0);
      }
    }
  }
  free(ls);
  free(mag);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Waveform -> mel spectrogram (flashmel / torchaudio MelSpectrogram).        */
/* ------------------------------------------------------------------------ */

#define ORACLE_PAD_REFLECT 0
#define ORACLE_PAD_CONSTANT 1
#define ORACLE_PAD_REPLICATE 2
#define ORACLE_PAD_CIRCULAR 3

#define ORACLE_SCALE_HTK 0
#define ORACLE_SCALE_SLANEY 1

/* Hz -> mel.  HTK: 2595 log10(1 + f/700).  Slaney: linear 3 mels per 200 Hz
 * below 1 kHz, then logarithmic with 27 mels per factor 6.4. */
double oracle_hz_to_mel(double f, int scale) {
  if (scale == ORACLE_SCALE_HTK) return 2595.0 * log10(1.0 + f / 700.0);
  const double f_sp = 200.0 / 3.0, min_log_hz = 1000.0;
  const double min_log_mel = min_log_hz / f_sp;
  const double logstep = log(6.4) / 27.0;
  if (f < min_log_hz) return f / f_sp;
  return min_log_mel + log(f / min_log_hz) / logstep;
}

double oracle_mel_to_hz(double m, int scale) {
  if (scale == ORACLE_SCALE_HTK) return 700.0 * (pow(10.0, m / 2595.0) - 1.0);
  const double f_sp = 200.0 / 3.0, min_log_hz = 1000.0;
  const double min_log_mel = min_log_hz / f_sp;
  const double logstep = log(6.4) / 27.0;
  if (m < min_log_mel) return f_sp * m;
  return min_log_hz * exp(logstep * (m - min_log_mel));
}

/* fb[n_mels][n_freqs] in double.  Triangles in Hz between n_mels + 2 points
 * equally spaced on the mel scale from f_min to f_max; bin k sits at
 * k * (sr/2) / (n_freqs - 1) Hz.  slaney_norm scales each triangle to unit
 * area: 2 / (f_{n+2} - f_n). */
int oracle_mel_filterbank(int64_t n_freqs, double f_min, double f_max, int64_t n_mels,
                          double sample_rate, int scale, int slaney_norm, double *fb) {
  if (!fb || n_freqs < 2 || n_mels < 1 || !(f_max > f_min)) return ORACLE_BAD_ARG;
  double *f_pts = (double *)malloc(sizeof(double) * (size_t)(n_mels + 2));
  if (!f_pts) return ORACLE_NO_MEM;
  double m_min = oracle_hz_to_mel(f_min, scale), m_max = oracle_hz_to_mel(f_max, scale);
  for (int64_t i = 0; i < n_mels + 2; ++i) {
    double m = m_min + (m_max - m_min) * (double)i / (double)(n_mels + 1);
    f_pts[i] = oracle_mel_to_hz(m, scale);
  }
  for (int64_t n = 0; n < n_mels; ++n) {
    double lo = f_pts[n], mid = f_pts[n + 1], hi = f_pts[n + 2];
    double scale_n = slaney_norm ? 2.0 / (hi - lo) : 1.0;
    for (int64_t k = 0; k < n_freqs; ++k) {
      double fk = (double)k * (sample_rate / 2.0) / (double)(n_freqs - 1);
      double up = (fk - lo) / (mid - lo);
      double down = (hi - fk) / (hi - mid);
      double w = up < down ? up : down;
      if (w < 0.0) w = 0.0;
      fb[n * n_freqs + k] = w * scale_n;
    }
  }
  free(f_pts);
  return ORACLE_OK;
}

/* Periodic Hann window of length n: 0.5 - 0.5 cos(2 pi j / n). */
int oracle_hann_window(int64_t n, double *w) {
  if (!w || n < 1) return ORACLE_BAD_ARG;
  for (int64_t j = 0; j < n; ++j) w[j] = 0.5 - 0.5 * cos(2.0 * M_PI * (double)j / (double)n);
  return ORACLE_OK;
}

int64_t oracle_n_frames(int64_t T, int64_t n_fft, int64_t hop, int center) {
  if (hop < 1 || n_fft < 1 || T < 0) return -1;
  int64_t len = center ? T + 2 * (n_fft / 2) : T;
  if (len < n_fft) return 0;
  return 1 + (len - n_fft) / hop;
}

/* Padded copy of x[T] with p samples on each side. */
static int pad_signal(const double *x, int64_t T, int64_t p, int mode, double *out) {
  for (int64_t i = 0; i < T + 2 * p; ++i) {
    int64_t s = i - p; /* position in the unpadded signal */
    double v;
    if (s >= 0 && s < T) {
      v = x[s];
    } else if (mode == ORACLE_PAD_CONSTANT) {
      v = 0.0;
    } else if (mode == ORACLE_PAD_REPLICATE) {
      v = x[s < 0 ? 0 : T - 1];
    } else if (mode == ORACLE_PAD_CIRCULAR) {
      v = x[((s % T) + T) % T];
    } else { /* reflect about the edge sample, which is not repeated */
      if (p >= T) return ORACLE_BAD_ARG;
      v = x[s < 0 ? -s : 2 * (T - 1) - s];
    }
    out[i] = v;
  }
  return ORACLE_OK;
}

/* Power spectrogram of one signal with the full torchaudio Spectrogram
 * argument set: spec[n_frames][n_fft/2 + 1] in double.
 *   1. pad > 0: `pad` zeros are added on both sides first;
 *   2. center: n_fft/2 more samples on both sides, filled per pad_mode;
 *   3. the window is a periodic Hann of length win_length (0 = n_fft),
 *      centred in n_fft samples with zeros around it;
 *   4. X_k = sum_j x_pad[t*hop + j] w[j] exp(-2 pi i j k / n_fft), summed
 *      directly (O(n_fft^2) per frame);
 *   5. normalized: X is divided by sqrt(sum_j w[j]^2);
 *   6. spec = |X_k|^power. */
int oracle_power_spectrogram_ex(const double *x, int64_t T, int64_t n_fft, int64_t win_length, int64_t hop,
                                int64_t pad, int center, int pad_mode, int normalized, double power,
                                double *spec) {
  if (!x || !spec || n_fft < 1 || hop < 1 || T < 1 || pad < 0) return ORACLE_BAD_ARG;
  int64_t wl = win_length > 0 ? win_length : n_fft;
  if (wl > n_fft) return ORACLE_BAD_ARG;
  int64_t T1 = T + 2 * pad;
  int64_t p = center ? n_fft / 2 : 0;
  int64_t n_frames = oracle_n_frames(T1, n_fft, hop, center);
  if (n_frames < 1) return ORACLE_BAD_ARG;
  int64_t n_freqs = n_fft / 2 + 1;
  double *x1 = (double *)calloc((size_t)T1, sizeof(double));
  double *xp = (double *)malloc(sizeof(double) * (size_t)(T1 + 2 * p));
  double *w = (double *)calloc((size_t)n_fft, sizeof(double));
  double *cs = (double *)malloc(sizeof(double) * (size_t)n_fft);
  double *sn = (double *)malloc(sizeof(double) * (size_t)n_fft);
  double *fr = (double *)malloc(sizeof(double) * (size_t)n_fft);
  int err = (x1 && xp && w && cs && sn && fr) ? ORACLE_OK : ORACLE_NO_MEM;
  if (err == ORACLE_OK) {
    memcpy(x1 + pad, x, sizeof(double) * (size_t)T);
    err = pad_signal(x1, T1, p, pad_mode, xp);
  }
  if (err == ORACLE_OK) {
    int64_t left = (n_fft - wl) / 2;
    oracle_hann_window(wl, w + left);
    double scale = 1.0;
    if (normalized) {
      double e = 0.0;
      for (int64_t j = 0; j < n_fft; ++j) e += w[j] * w[j];
      scale = 1.0 / sqrt(e);
    }
    for (int64_t m = 0; m < n_fft; ++m) { /* e^{-2 pi i m / n_fft} for m = (j k) mod n_fft */
      double ang = 2.0 * M_PI * (double)m / (double)n_fft;
      cs[m] = cos(ang);
      sn[m] = sin(ang);
    }
    for (int64_t t = 0; t < n_frames; ++t) {
      for (int64_t j = 0; j < n_fft; ++j) fr[j] = xp[t * hop + j] * w[j];
      for (int64_t k = 0; k < n_freqs; ++k) {
        double re = 0.0, im = 0.0;
        for (int64_t j = 0; j < n_fft; ++j) {
          int64_t m = (j * k) % n_fft;
          re += fr[j] * cs[m];
          im -= fr[j] * sn[m];
        }
        re *= scale;
        im *= scale;
        double p2 = re * re + im * im;
        spec[t * n_freqs + k] = (power == 2.0) ? p2 : pow(sqrt(p2), power);
      }
    }
  }
  free(x1);
  free(xp);
  free(w);
  free(cs);
  free(sn);
  free(fr);
  return err;
}

/* The common case: window of n_fft samples, no extra padding, no normalisation. */
int oracle_power_spectrogram(const double *x, int64_t T, int64_t n_fft, int64_t hop, int center,
                             int pad_mode, double power, double *spec) {
  return oracle_power_spectrogram_ex(x, T, n_fft, 0, hop, 0, center, pad_mode, 0, power, spec);
}

/* Round a double to IEEE binary16, nearest-even, directly (no trip through
 * float, so there is a single rounding). */
uint16_t oracle_f64_to_f16(double v) {
  uint16_t sign = signbit(v) ? 0x8000u : 0u;
  if (isnan(v)) return 0x7e00u;
  double a = fabs(v);
  if (a >= 65520.0) return sign | 0x7c00u; /* halfway above 65504 rounds to inf */
  if (a < ldexp(1.0, -14)) {               /* subnormal range: multiples of 2^-24 */
    double r = nearbyint(ldexp(a, 24));
    return sign | (uint16_t)r; /* r == 1024 encodes the smallest normal */
  }
  int e;
  frexp(a, &e);                         /* a = m 2^e, m in [0.5, 1) */
  double r = nearbyint(ldexp(a, 11 - e)); /* 11 significant bits: [1024, 2048] */
  int exp16 = e - 1 + 15;
  if (r >= 2048.0) {
    r = 1024.0;
    exp16 += 1;
  }
  if (exp16 >= 31) return sign | 0x7c00u;
  return (uint16_t)(sign | (uint16_t)(exp16 << 10) | (uint16_t)((uint32_t)r - 1024u));
}

#define ORACLE_IN_F32 0
#define ORACLE_IN_I16 1
#define ORACLE_OUT_F32 0
#define ORACLE_OUT_F16 2

/* out[B][n_mels][n_frames] as f32 or f16 (raw bits).  log_mel = 1 applies the
 * log10 floor / per-clip clamp / rescale of the KBench spec over the whole
 * (n_mels, n_frames) plane of each clip. */
int oracle_mel_spectrogram_ex(const void *wave, int in_dtype, int64_t B, int64_t T,
                              int64_t sample_rate, int64_t n_fft, int64_t win_length, int64_t hop,
                              int64_t pad, int64_t n_mels, double f_min, double f_max, int center,
                              int pad_mode, int normalized, double power, int mel_scale,
                              int slaney_norm, int log_mel, int out_dtype, void *out) {
  if (!wave || !out || B < 1 || T < 1 || n_fft < 2 || hop < 1 || n_mels < 1 || pad < 0) return ORACLE_BAD_ARG;
  int64_t n_freqs = n_fft / 2 + 1;
  int64_t n_frames = oracle_n_frames(T + 2 * pad, n_fft, hop, center);
  if (n_frames < 1) return ORACLE_BAD_ARG;
  if (center && pad_mode == ORACLE_PAD_REFLECT && n_fft / 2 >= T + 2 * pad) return ORACLE_BAD_ARG;
  double *fb = (double *)malloc(sizeof(double) * (size_t)(n_mels * n_freqs));
  if (!fb) return ORACLE_NO_MEM;
  int err = oracle_mel_filterbank(n_freqs, f_min, f_max, n_mels, (double)sample_rate, mel_scale,
                                  slaney_norm, fb);
  if (err != ORACLE_OK) {
    free(fb);
    return err;
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t b = 0; b < B; ++b) {
    double *x = (double *)malloc(sizeof(double) * (size_t)T);
    double *spec = (double *)malloc(sizeof(double) * (size_t)(n_frames * n_freqs));
    double *mel = (double *)malloc(sizeof(double) * (size_t)(n_frames * n_mels));
    int e = (x && spec && mel) ? ORACLE_OK : ORACLE_NO_MEM;
    if (e == ORACLE_OK) {
      for (int64_t i = 0; i < T; ++i) {
        if (in_dtype == ORACLE_IN_I16)
          x[i] = (double)((const int16_t *)wave)[b * T + i] / 32768.0;
        else
          x[i] = (double)((const float *)wave)[b * T + i];
      }
      e = oracle_power_spectrogram_ex(x, T, n_fft, win_length, hop, pad, center, pad_mode, normalized, power,
                                      spec);
    }
    if (e == ORACLE_OK) {
      double hi = -INFINITY;
      for (int64_t n = 0; n < n_mels; ++n)
        for (int64_t t = 0; t < n_frames; ++t) {
          double acc = 0.0;
          for (int64_t k = 0; k < n_freqs; ++k) acc += fb[n * n_freqs + k] * spec[t * n_freqs + k];
          if (log_mel) {
            acc = log10(acc > 1e-10 ? acc : 1e-10);
            if (acc > hi) hi = acc;
          }
          mel[n * n_frames + t] = acc;
        }
      for (int64_t i = 0; i < n_mels * n_frames; ++i) {
        double v = mel[i];
        if (log_mel) {
          if (v < hi - 8.0) v = hi - 8.0;
          v = (v + 4.0) / 4.0;
        }
        int64_t o = b * n_mels * n_frames + i;
        if (out_dtype == ORACLE_OUT_F16)
          ((uint16_t *)out)[o] = oracle_f64_to_f16(v);
        else
          ((float *)out)[o] = (float)v;
      }
    } else {
      err = e;
    }
    free(x);
    free(spec);
    free(mel);
  }
  free(fb);
  return err;
}

/* The common case: window of n_fft samples, no extra padding, no normalisation. */
int oracle_mel_spectrogram(const void *wave, int in_dtype, int64_t B, int64_t T,
                           int64_t sample_rate, int64_t n_fft, int64_t hop, int64_t n_mels,
                           double f_min, double f_max, int center, int pad_mode, double power,
                           int mel_scale, int slaney_norm, int log_mel, int out_dtype,
                           void *out) {
  return oracle_mel_spectrogram_ex(wave, in_dtype, B, T, sample_rate, n_fft, 0, hop, 0, n_mels, f_min, f_max,
                                   center, pad_mode, 0, power, mel_scale, slaney_norm, log_mel, out_dtype, out);
}
