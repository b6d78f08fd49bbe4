/*
 * logmel.h -- C ABI of liblogmel.so, the GB300 (sm_103a) log-mel front end.
 *
 * Two operations:
 *
 *  1. lm_log_mel_from_stft: Whisper's log-mel spectrogram from a complex
 *     STFT, as defined by the KBench task spec "audio_mel_spectrogram_fused.py"
 *     (its reference function and the per-clip definition in its spec text):
 *         mag[b,f,k]      = re^2 + im^2                      (power)
 *         mel[b,f,n]      = sum_k mag[b,f,k] * mel_filters[n,k]
 *         log_spec[b,f,n] = log10(max(mel[b,f,n], 1e-10))
 *         hi[b]           = max over (f, n) of log_spec[b,f,n]  (per clip)
 *         out[b,f,n]      = (max(log_spec[b,f,n], hi[b] - 8) + 4) / 4
 *     All arithmetic is f32 (the spec's precision section rules out bf16,
 *     fp16 and fp8 anywhere on this path).
 *
 *  2. lm_mel_spectrogram: waveform -> mel spectrogram, the torchaudio-style
 *     MelSpectrogram described on the "flashmel" PyPI page (usage section and
 *     argument list): framing with center padding, periodic Hann window,
 *     one-sided real FFT, |X|^power, triangular mel filterbank (HTK or Slaney
 *     scale), f32 or int16 input (int16 scaled by 1/32768), f32 or f16
 *     output, laid out [B, n_mels, n_frames].  Optionally followed by the same
 *     log10 / per-clip clamp / rescale as operation 1.
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must point to memory of the current
 *    CUDA device; the caller owns all buffers.  Inputs are read-only.
 *  - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *    stream); results are ready once the stream reaches that point.
 *  - Nothing is allocated on the compute path: scratch comes from the
 *    caller's `workspace`, sized by the matching *_workspace_size call.
 *  - Errors are returned as lm_status, never by aborting or trapping.
 *    Argument errors are detected on the host before anything is enqueued.
 *    LM_ERR_CUDA means a CUDA runtime call failed; lm_last_cuda_error()
 *    returns its code (per host thread).
 *  - Kernels bound every wait they perform.  A wait that runs out (which
 *    correct use never triggers) sets a device error word in the workspace
 *    instead of hanging; lm_workspace_error() reads it.
 */
#ifndef LOGMEL_H_
#define LOGMEL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *lm_stream_t;

typedef enum lm_status {
  LM_OK = 0,
  LM_ERR_INVALID_ARG = 1,   /* null pointer, negative or inconsistent size */
  LM_ERR_UNSUPPORTED = 2,   /* a valid request this library does not implement */
  LM_ERR_MISALIGNED = 3,    /* a pointer lacks the stated alignment */
  LM_ERR_CUDA = 4,          /* a CUDA runtime call failed, see lm_last_cuda_error */
  LM_ERR_OUT_OF_MEMORY = 5, /* plan creation could not allocate its tables */
  LM_ERR_DEVICE_FAULT = 6,  /* a kernel reported a bounded wait that ran out */
  LM_ERR_WORKSPACE = 7      /* workspace null or smaller than required */
} lm_status;

typedef enum lm_dtype { LM_F32 = 0, LM_I16 = 1, LM_F16 = 2 } lm_dtype;

typedef enum lm_pad_mode {
  LM_PAD_REFLECT = 0,   /* mirror about the edge sample, edge not repeated */
  LM_PAD_CONSTANT = 1,  /* zeros */
  LM_PAD_REPLICATE = 2, /* repeat the edge sample */
  LM_PAD_CIRCULAR = 3   /* wrap around */
} lm_pad_mode;

typedef enum lm_mel_scale { LM_MEL_HTK = 0, LM_MEL_SLANEY = 1 } lm_mel_scale;

/* Human-readable name of a status code.  Never NULL. */
const char *lm_status_string(int status);

/* The cudaError_t of the last failed CUDA call made by this host thread
 * inside the library (0 if none). */
int lm_last_cuda_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int lm_version(void);

/* ------------------------------------------------------------------------ */
/* 1. log-mel from a complex STFT                                           */
/* ------------------------------------------------------------------------ */

/* Bytes of device workspace lm_log_mel_from_stft needs for this shape
 * (a header, one u32 per clip and one u32 per tile of frames).  Host-only. */
lm_status lm_log_mel_from_stft_workspace_size(int64_t B, int64_t F, int32_t NF, int32_t NM,
                                              size_t *bytes);

/*
 * Whisper log-mel from a complex STFT (KBench "audio_mel_spectrogram_fused"
 * spec: reference function, per-clip definition and I/O contract).
 *
 *   stft        device, [B][F][NF] complex64 = interleaved (re, im) f32
 *               pairs, contiguous, 8-byte aligned (the alignment of a
 *               complex64 element; any contiguous view of a complex64
 *               tensor qualifies).                             (read-only)
 *   mel_filters device, [NM][NF] f32 row-major, 4-byte aligned; any dense
 *               matrix (only the span between the first and the last
 *               nonzero of each row is read).                  (read-only)
 *   out         device, [B][F][NM] f32, 4-byte aligned; must not overlap
 *               the inputs.
 *   B, F        clips and frames per clip (B, F >= 0; F may be ragged).
 *   NF, NM      bins per frame (1..8193) and mel bands (1..512).
 *   workspace   device, >= lm_log_mel_from_stft_workspace_size(B, F, NF, NM) bytes,
 *               4-byte aligned; its contents are overwritten.
 *
 * Errors: LM_ERR_INVALID_ARG (null pointer with B*F > 0, negative sizes),
 * LM_ERR_UNSUPPORTED (NF or NM out of range), LM_ERR_MISALIGNED (stft not
 * 8-byte aligned, out or workspace not 4-byte aligned), LM_ERR_WORKSPACE,
 * LM_ERR_CUDA.  B == 0 or F == 0 returns LM_OK and enqueues nothing.
 * Concurrent calls must use distinct workspaces.
 */
lm_status lm_log_mel_from_stft(const void *stft, const float *mel_filters, float *out, int64_t B,
                               int64_t F, int32_t NF, int32_t NM, void *workspace,
                               size_t workspace_bytes, lm_stream_t stream);

/* How lm_log_mel_from_stft will run a problem of this shape on the current
 * device (pure host-side planning; no work is enqueued).  Fields:
 *   resident       1 = single cooperative launch, one persistent CTA per SM,
 *                  that keeps each tile's log values on chip until its clip
 *                  maximum is known and writes the output once.
 *   cluster        > 0 = single launch of one thread-block cluster of this
 *                  many CTAs per clip (small batches, when the device runs
 *                  every clip's cluster at once): each CTA keeps its share
 *                  of the clip's log values in shared memory, the cluster
 *                  exchanges maxima through distributed shared memory, and
 *                  the output is written once.
 *                  resident = 0 and cluster = 0: two launches (log values,
 *                  then the in-place floor/rescale pass).
 *   kernels        kernel launches per call (1 or 2; plus one memset of the
 *                  workspace).
 *   grid           CTAs of the main kernel.
 *   frames_per_tile, stages, lag: tile height, shared-memory ring depth, and
 *                  how many tiles each thread holds back before writing.
 *   smem_bytes     dynamic shared memory per CTA.
 * LOGMEL_K1_VARIANT=resident|twopass|cluster forces a variant, and
 * =nocluster leaves the cluster variant out (A/B), and LOGMEL_FPB=1|2|4|6|8
 * forces the frames each consumer thread takes per tile (the workspace size
 * follows it); a forced variant or tile that cannot run returns
 * LM_ERR_UNSUPPORTED. */
typedef struct lm_stft_launch_info {
  int32_t resident;
  int32_t kernels;
  int32_t grid;
  int32_t frames_per_tile;
  int32_t stages;
  int32_t lag;
  int64_t smem_bytes;
  int32_t cluster;
  int32_t reserved;
} lm_stft_launch_info;

lm_status lm_log_mel_from_stft_describe(int64_t B, int64_t F, int32_t NF, int32_t NM,
                                        lm_stft_launch_info *info);

/* ---- Pre-packed filters (the "flashmel" page, "How it works": triangular
 * filters packed as start / width / weights) ----
 *
 * lm_log_mel_from_stft derives each band's support (first..last nonzero bin of
 * its row of the dense matrix) and first weights on every call; at kernel
 * start that costs a sweep of the whole matrix plus a second round of loads,
 * several microseconds that dominate small batches.  A caller that reuses
 * one filter matrix can pack it once and pass the pack:
 *
 *   lm_mel_filters_pack_size(NF, NM, &bytes)   bytes of device memory a pack
 *                                              needs (LM_ERR_INVALID_ARG /
 *                                              LM_ERR_UNSUPPORTED as for the
 *                                              shapes of lm_log_mel_from_stft).
 *   lm_mel_filters_pack(mel_filters, NF, NM, packed, bytes, stream)
 *       enqueues on `stream` the packing of the dense [NM][NF] f32 matrix
 *       (device, 4-byte aligned, read-only) into `packed` (device, caller
 *       owned, 16-byte aligned, >= the size above): a header with the shape,
 *       then {first bin, width} per band, then each band's first 8 weights
 *       from its first bin (zero past the width).  Errors:
 *       LM_ERR_INVALID_ARG (null), LM_ERR_MISALIGNED, LM_ERR_WORKSPACE (too
 *       small), LM_ERR_CUDA.
 *   lm_log_mel_from_stft_packed(stft, mel_filters, packed, out, ...)
 *       the same computation, arguments and results as lm_log_mel_from_stft,
 *       reading supports and first weights from `packed` (which must be made
 *       from this mel_filters, and be complete in stream order; bands wider
 *       than 8 bins still read the rest from mel_filters).  A pack whose
 *       header does not match NF, NM is not used: the call falls back to the
 *       dense matrix and sets bit 4 of the device error word
 *       (lm_workspace_error).  Errors: as lm_log_mel_from_stft, plus
 *       LM_ERR_INVALID_ARG for a null pack and LM_ERR_MISALIGNED for one not
 *       16-byte aligned.
 */
lm_status lm_mel_filters_pack_size(int32_t NF, int32_t NM, size_t *bytes);
lm_status lm_mel_filters_pack(const float *mel_filters, int32_t NF, int32_t NM, void *packed,
                              size_t packed_bytes, lm_stream_t stream);
lm_status lm_log_mel_from_stft_packed(const void *stft, const float *mel_filters, const void *packed,
                                      float *out, int64_t B, int64_t F, int32_t NF, int32_t NM,
                                      void *workspace, size_t workspace_bytes, lm_stream_t stream);

/* ---- Allocation-free variant (the source pages have no counterpart) ----
 *
 * Same computation, arguments and results as lm_log_mel_from_stft, without
 * the workspace argument.  It is meant for callers that cannot allocate
 * device memory themselves: code on a real-time audio thread, where a
 * cudaMalloc may block or synchronise the whole device, or a host
 * application that owns every byte of device memory and has no scratch to
 * hand out.
 *
 * Scratch comes from one fixed array of LM_NOALLOC_SCRATCH_BYTES compiled
 * into the library; every GPU that loads the library holds that array until
 * the process exits.  The call allocates and frees nothing.
 *  - Its first LM_NOALLOC_SCRATCH_BYTES - 256 bytes stand in for the
 *    workspace.  A problem needing more than that (about 16 bytes plus 4
 *    bytes per tile of frames; for NF = 201, NM = 128 a tile is 25 frames,
 *    so up to about 262,000 tiles, e.g. 256 clips of up to 25,500 frames)
 *    returns LM_ERR_WORKSPACE and enqueues nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept for the life of the
 *    process: after a cudaDeviceReset of that device it is stale, so do not
 *    call these entry points after one.
 *  - Every call uses the same array, which keeps the previous call's
 *    contents; each call clears the part it needs before its kernel runs.
 *    Calls whose work can overlap on the GPU (different streams, or host
 *    threads without ordering between them) race on the array: the caller
 *    must order them.
 *  - The kernels' device error bits go to a word in the array's last 256
 *    bytes, which no call clears: bits accumulate over calls until
 *    lm_log_mel_from_stft_noalloc_error reads and clears them.
 */
#define LM_NOALLOC_SCRATCH_BYTES (1u << 20)

lm_status lm_log_mel_from_stft_noalloc(const void *stft, const float *mel_filters, float *out,
                                       int64_t B, int64_t F, int32_t NF, int32_t NM,
                                       lm_stream_t stream);

/* Synchronises `stream`, then reads the accumulated device error word of
 * lm_log_mel_from_stft_noalloc calls on the current device (0 = no kernel
 * reported a problem) into *device_error, and clears it when `clear` is
 * nonzero (the clearing is ordered on `stream`).  Allocates nothing.
 * Returns LM_ERR_DEVICE_FAULT when the word was nonzero, LM_ERR_INVALID_ARG
 * for a null pointer, LM_ERR_CUDA when a CUDA call failed. */
lm_status lm_log_mel_from_stft_noalloc_error(uint32_t *device_error, int32_t clear, lm_stream_t stream);

/* Synchronises `stream`, then reads the device error word of a workspace
 * used by lm_log_mel_from_stft or lm_mel_spectrogram.  *device_error = 0
 * means no kernel reported a problem; otherwise it holds bit flags:
 *   1  an mbarrier wait inside a kernel ran out (2 s)
 *   2  waiting for another CTA's result ran out (a clip's maximum, or
 *      the launch token of the CTA that clears the workspace)
 *   4  a filter pack did not match the call (the dense matrix was used)
 *   8  (only in the bounds-checked debug build, compiled with
 *      -DLOGMEL_CHECKED) a computed global-memory index fell outside its
 *      buffer; the access was skipped
 * Returns LM_ERR_DEVICE_FAULT when it is nonzero. */
lm_status lm_workspace_error(const void *workspace, size_t workspace_bytes, uint32_t *device_error,
                             lm_stream_t stream);

/* ---- Fault injection for tests of the bounded waits (the source pages
 * have no counterpart) ----
 *
 * Runs lm_log_mel_from_stft on its one-CTA-per-SM kernel (same arguments,
 * results and errors; the cluster variant has no cross-CTA waits) with two
 * changes that make one of its cross-CTA waits run out on purpose, so that
 * a test can check that the kernel gives up cleanly instead of hanging:
 *   withheld_tile  the maximum of this tile of frames is never published
 *                  (tiles are numbered clip by clip; a clip has
 *                  ceil(F / frames_per_tile) of them, see
 *                  lm_log_mel_from_stft_describe); >= 0.
 *   clip_wait_ns   how long a CTA waits for a clip's maximum before giving
 *                  up (the regular calls wait 2 s); 1e5 .. 2e9.
 * When a wait gives up, the CTA sets bit 2 of the workspace's device error
 * word, its warps stop without further stores, and it exits once its
 * in-flight copies have landed.  The outputs of the clip whose tile was
 * withheld (and, where a CTA ran tiles of several clips, of the clips it
 * had not finished) are left incomplete.  Only single-kernel (resident)
 * launches wait across CTAs; for two-launch shapes the tile's slot stays
 * zero and the epilogue reduces the clip maximum over the other tiles.
 * Returns LM_ERR_INVALID_ARG for arguments out of range. */
lm_status lm_debug_log_mel_from_stft_withhold(const void *stft, const float *mel_filters, float *out,
                                              int64_t B, int64_t F, int32_t NF, int32_t NM, void *workspace,
                                              size_t workspace_bytes, int64_t withheld_tile,
                                              uint64_t clip_wait_ns, lm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* 2. waveform -> mel spectrogram                                            */
/* ------------------------------------------------------------------------ */

/* Parameters of a mel spectrogram, named as torchaudio's MelSpectrogram
 * arguments listed on the flashmel page (window is always periodic Hann,
 * onesided always true). */
typedef struct lm_mel_params {
  int32_t sample_rate; /* Hz, > 0 */
  int32_t n_fft;       /* 400, or a power of two in [64, 16384] */
  int32_t win_length;  /* 0 = n_fft; otherwise 1..n_fft, window centred in the frame */
  int32_t hop_length;  /* > 0 */
  int32_t n_mels;      /* 1..256 */
  float f_min;         /* Hz, >= 0 */
  float f_max;         /* Hz, > f_min; <= 0 means sample_rate / 2 */
  int32_t pad;         /* zeros added on both sides before centre padding, >= 0 */
  int32_t center;      /* 1: pad n_fft/2 on both sides with pad_mode */
  int32_t pad_mode;    /* lm_pad_mode */
  float power;         /* 1 (magnitude) or 2 (power) */
  int32_t normalized;  /* 1: scale the window by 1/sqrt(sum w^2) */
  int32_t mel_scale;   /* lm_mel_scale */
  int32_t slaney_norm; /* 1: each triangle scaled to unit area */
  int32_t log_mel;     /* 1: log10(max(x,1e-10)), per-clip clamp at max-8, (x+4)/4 */
} lm_mel_params;

typedef struct lm_mel_plan lm_mel_plan;

/* Validates `params`, builds the window, filterbank and FFT tables on the
 * host in double and uploads them (rounded to f32) to the current device.
 * Errors: LM_ERR_INVALID_ARG, LM_ERR_UNSUPPORTED, LM_ERR_OUT_OF_MEMORY,
 * LM_ERR_CUDA; on any error *plan is NULL and nothing stays allocated.
 * The plan is immutable and may be shared by streams.
 * For tests of that error path, the environment variable
 * LOGMEL_FAULT=plan_alloc (or plan_alloc:k) makes the first (k-th) of the
 * plan's device allocations fail as if the device were out of memory. */
lm_status lm_mel_plan_create(const lm_mel_params *params, lm_mel_plan **plan);

/* Frees the plan's device tables (synchronises the device first). */
lm_status lm_mel_plan_destroy(lm_mel_plan *plan);

/* Number of output frames for a signal of T samples. */
lm_status lm_mel_n_frames(const lm_mel_plan *plan, int64_t T, int64_t *n_frames);

/* Bytes of device workspace lm_mel_spectrogram needs for B clips of T
 * samples (a header and, for log plans, one u32 per tile of frames and two
 * per clip). */
lm_status lm_mel_workspace_size(const lm_mel_plan *plan, int64_t B, int64_t T, size_t *bytes);

/*
 * Mel spectrogram of B waveforms (flashmel page, usage and "how it works").
 *
 *   wave      device, [B][T] f32 (in_dtype LM_F32) or int16 (LM_I16, scaled
 *             by 1/32768), contiguous, 4-byte aligned.          (read-only)
 *   out       device, [B][n_mels][n_frames] f32 (LM_F32) or f16 (LM_F16),
 *             4-byte aligned.  log_mel plans require LM_F32.
 *   workspace device, >= lm_mel_workspace_size(plan, B, T) bytes, 4-byte
 *             aligned; its contents on entry do not matter.  An 8-byte
 *             aligned workspace needs no memset before the kernel (the
 *             kernel clears its error word, tile counter and clip words
 *             itself, keyed by a per-launch token); a 4-byte aligned one,
 *             or any call made while the stream is being captured into a
 *             graph, gets a memset first.
 *
 * Log plans run as two launches: the transform, then a clamp-only kernel
 * launched as a programmatic dependent (its launch overlaps the first
 * kernel's tail).  With LOGMEL_K3_EPILOGUE=fused, where n_fft is 64, 128,
 * 256, 400, 512 or 1024, the clip floor and rescale are applied by the same
 * cooperative grid instead (one launch, the same bits; measured slower).
 * Non-log plans are one launch.
 *
 * Errors: LM_ERR_INVALID_ARG (null pointers, T too short for reflect
 * padding, n_frames < 1), LM_ERR_UNSUPPORTED (dtype combination),
 * LM_ERR_MISALIGNED, LM_ERR_WORKSPACE, LM_ERR_CUDA.
 */
lm_status lm_mel_spectrogram(const lm_mel_plan *plan, const void *wave, int32_t in_dtype, int64_t B,
                             int64_t T, void *out, int32_t out_dtype, void *workspace,
                             size_t workspace_bytes, lm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* 3. host buffers in and out (the source pages have no counterpart)        */
/* ------------------------------------------------------------------------ */

/*
 * The same computations as lm_log_mel_from_stft(_packed) and
 * lm_mel_spectrogram, for inputs and results in host memory.  The library
 * cuts the batch into chunks of whole clips and pipelines them through
 * three staging slots in the workspace: the copy in of one chunk, the
 * kernels of the previous one and the copy out of the one before run at
 * the same time, on two internal streams of the library and `stream`.
 * Results equal those of the device entry points bit for bit (clips are
 * independent; the per-clip maximum never crosses a chunk).
 *
 *   stft_host / wave_host  host, laid out as the device entry point's input.
 *   out_host               host, laid out as the device entry point's output;
 *                          must not overlap the input.
 *                          Both should be page-locked (cudaHostAlloc or
 *                          cudaHostRegister) for the copies to overlap;
 *                          pageable memory gives the same results, with the
 *                          copies serialised and the call blocking the host.
 *   mel_filters, packed    device, as for lm_log_mel_from_stft_packed;
 *                          packed may be NULL (dense filters).
 *   chunk_clips            clips per chunk; 0 = the library's choice: whole
 *                          clips filling about 32 MB of input, and at most a
 *                          third of the batch (rounded up).
 *   workspace              device, 256-byte aligned, >= the matching
 *                          *_host_workspace_size (a 256-byte header whose
 *                          first u32 is the device error word of every
 *                          chunk, the operation's workspace for one chunk,
 *                          then three input and three output slots).
 *   stream                 the call is ordered on it: the copy streams
 *                          start after its earlier work, and it waits for
 *                          the last copy out.  out_host is complete once
 *                          `stream` reaches that point (e.g. after
 *                          cudaStreamSynchronize(stream)).
 *
 * The first call on a device, and each further call that overlaps in time
 * with the others, creates two streams and twelve events that the library
 * keeps for reuse until the process exits; no memory is allocated.
 *
 * Errors: as the device entry points, plus LM_ERR_INVALID_ARG when the host
 * buffers overlap, and LM_ERR_UNSUPPORTED when `stream` is capturing a
 * CUDA graph (the pipeline is not capturable).  Argument errors are found
 * before anything is enqueued; lm_workspace_error reads the error word.
 * Calls that overlap in time need distinct workspaces.
 */
lm_status lm_log_mel_from_stft_host_workspace_size(int64_t B, int64_t F, int32_t NF, int32_t NM,
                                                   int64_t chunk_clips, size_t *bytes);
lm_status lm_log_mel_from_stft_host(const void *stft_host, const float *mel_filters, const void *packed,
                                    float *out_host, int64_t B, int64_t F, int32_t NF, int32_t NM,
                                    int64_t chunk_clips, void *workspace, size_t workspace_bytes,
                                    lm_stream_t stream);

lm_status lm_mel_spectrogram_host_workspace_size(const lm_mel_plan *plan, int64_t B, int64_t T,
                                                 int32_t in_dtype, int32_t out_dtype, int64_t chunk_clips,
                                                 size_t *bytes);
lm_status lm_mel_spectrogram_host(const lm_mel_plan *plan, const void *wave_host, int32_t in_dtype,
                                  int64_t B, int64_t T, void *out_host, int32_t out_dtype,
                                  int64_t chunk_clips, void *workspace, size_t workspace_bytes,
                                  lm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LOGMEL_H_ */
