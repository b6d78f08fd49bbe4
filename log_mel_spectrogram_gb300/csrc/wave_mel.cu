// wave_mel.cu -- waveform -> mel spectrogram (the torchaudio-style
// MelSpectrogram on the "flashmel" PyPI page: usage, argument list and
// "How it works"), with the optional log10 / per-clip clamp / rescale of
// the KBench "audio_mel_spectrogram_fused" spec.
//
// Plan (host, once): periodic Hann window (win_length centred in n_fft,
// optional 1/sqrt(sum w^2) normalisation folded in), FFT twiddles and the
// triangular mel filterbank, all computed in double and rounded to f32; the
// filterbank is packed per band as first nonzero bin, width and weights.
//
// n_fft 64...1024 run the register kernels of wave_reg.cuh, which keep each
// frame's transform inside one warp and finish log plans in the same launch.
// The generic kernel below serves the larger sizes (and LOGMEL_K3=stockham):
//
// Kernel (one persistent CTA per SM slot, tiles of TF consecutive frames of
// one clip):
//  1. framing: frame t reads samples t*hop - n_fft/2 + j of the clip; the
//     padding (reflect / constant / replicate / circular) is index
//     arithmetic, and tiles that touch no edge load samples directly.  Pairs
//     of windowed samples form the N/2 complex points z[n] = x[2n] + i x[2n+1];
//  2. an N/2-point complex FFT in shared memory (fft.cuh): Stockham passes
//     between two buffers, or in place in one buffer at 8192 and 16384 points;
//  3. the real-input untangle X[k] = E[k] + exp(-2 pi i k/N) O[k], with
//     E = (Z[k] + conj Z[N/2-k]) / 2 and O = (Z[k] - conj Z[N/2-k]) / (2i),
//     straight into a power tile |X[k]|^power (odd row stride);
//  4. the banded mel projection, one output per thread, lanes over frames so
//     each band's row of the output [B, n_mels, n_frames] is written as a run
//     of consecutive frames (one-frame tiles above 4096 points: a warp per
//     band, lanes over its taps, the weights copied into the transform's
//     buffer once the power row is complete); f32 or f16 (round to nearest
//     even) at the store;
//  5. log plans store log10(max(mel, 1e-10)) and publish each tile's maximum
//     into a per-tile slot; a second kernel (the clamp epilogue shared with
//     the STFT path) turns slots into clip maxima and rescales in place.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

#include <cuda_fp16.h>

#include "fft.cuh"
#include "internal.h"
#include "ptx.cuh"

struct lm_mel_plan {
  lm_mel_params p;
  int device;
  int n_freqs;   // n_fft / 2 + 1
  int wmax;      // widest filter row, in bins
  float *window; // [n_fft]
  float2 *tw_m;  // [n_fft/2]      FFT twiddles, per-pass rows (fft::rows_offset)
  float2 *tw_n;  // [n_fft/2 + 1]  exp(-2 pi i k / n_fft)
  int *fstart;   // [n_mels]
  int *fwidth;   // [n_mels]
  float *fw;     // [n_mels][wmax]
  unsigned char *tables;  // n_fft <= 4096: tw_m | tw_n | window | {fstart, fwidth} | fw, the shared-memory image
  uint32_t tables_bytes;  // its size, a multiple of 16
  unsigned char *reg_tables;  // n_fft 64...1024: the register kernels' image (reg::Tables)
  uint32_t reg_tables_bytes;
  unsigned char *mel_image;   // n_fft 8192, 16384: the filterbank image (mel_image_bytes_for), or null
  uint32_t mel_image_bytes;
};

namespace lm {
namespace {

// Four floats from a 16-byte aligned shared-memory address.
__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

struct WaveArgs {
  const void *wave;
  void *out;
  uint32_t *tile_key;
  int64_t B, T, n_frames;
  int32_t in_i16, out_f16, log_mel, power_is_one;
  int32_t hop, pad_left, pad_mode;  // pad_left: centre padding plus the zero `pad`, in samples
  int32_t pad_zero;                 // zeros added on both sides before centre padding
  int32_t n_mels, wmax, tiles_per_clip, TF;
  uint32_t *err;           // device error word (workspace header)
  uint32_t *next_tile;     // tile counter (workspace header), zero at launch
  uint32_t *clip_key;      // [B] fused log epilogue: the clip's maximum key (0 = none yet)
  uint32_t *clip_done;     // [B] fused log epilogue: tiles of the clip whose maximum is folded in
  uint32_t *rescale_next;  // fused log epilogue: the next tile to floor and rescale
  int32_t fused;           // 1: the register kernel applies the clip floor and rescale itself
  int32_t clear_err;       // 1: the error word is this call's own (CTA 0 clears it when there is a token)
  uint64_t token;          // launch token (0: the host cleared the workspace with a memset)
  uint64_t *ready;         // with a token: CTA 0 stores it here once the words above that start at zero are
                           // clear; every CTA waits for it before its first tile claim
  uint64_t total_bytes;    // B * T * sample size
  uint32_t seg_offset;     // shared-memory offset of the two sample-span buffers
  uint32_t seg_bytes;      // bytes per span buffer (multiple of 128)
  int32_t use_seg;         // 1: stage interior tiles' samples with bulk copies
  const float *window;
  const float2 *tw_m;
  const float2 *tw_n;
  const int *fstart;
  const int *fwidth;
  const float *fw;
  const unsigned char *tables;  // shared-memory image of the tables (n_fft <= 4096)
  uint32_t tables_bytes;
  const unsigned char *mel_image;  // in place: the filterbank image copied into the transform's buffer, or null
  uint32_t mel_image_bytes;
};

// Launch token (CTA 0, thread 0): clears the error word (when it is this
// call's own) and the tile counter, then publishes the token with release
// order.  The fused epilogue's clip words are cleared by all of CTA 0 before
// its first block barrier, which this thread passes before publishing.
__device__ __forceinline__ void publish_cleared(const WaveArgs &a) {
  if (a.clear_err) *a.err = 0u;
  *a.next_tile = 0u;
  __threadfence();
  st_release_gpu_u64(a.ready, a.token);
}

// Thread 0: the CTA's next tile from the shared counter.  The first claim of
// a launch with a token waits (bounded) for CTA 0's token; if that runs out
// the CTA claims nothing more and the error word says why.
__device__ __forceinline__ int claim_tile(const WaveArgs &a, bool *token_seen, int *abort_flag_p, int n_tiles) {
  if (!*token_seen) {
    if (!wait_token(a.ready, a.token, kWaitTimeoutNs, abort_flag_p)) {
      *abort_flag_p = 1;
      atomicOr(a.err, kErrClipTimeout);
      return n_tiles;
    }
    *token_seen = true;
  }
  return static_cast<int>(gridDim.x + atomicAdd(a.next_tile, 1u));
}

__device__ __forceinline__ int64_t map_index(int64_t s, int64_t T, int mode, bool *zero) {
  *zero = false;
  if (s >= 0 && s < T) return s;
  switch (mode) {
    case LM_PAD_CONSTANT: *zero = true; return 0;
    case LM_PAD_REPLICATE: return s < 0 ? 0 : T - 1;
    case LM_PAD_CIRCULAR: { int64_t r = s % T; return r < 0 ? r + T : r; }
    default: return s < 0 ? -s : 2 * (T - 1) - s;  // reflect, edge not repeated
  }
}

__device__ __forceinline__ float load_sample(const WaveArgs &a, int64_t b, int64_t s) {
  if (!LM_IN_BOUNDS(b * a.T + s, a.B * a.T, a.err)) return 0.f;  // (checked builds)
  if (a.in_i16) return static_cast<float>(static_cast<const int16_t *>(a.wave)[b * a.T + s]) * (1.0f / 32768.0f);
  return static_cast<const float *>(a.wave)[b * a.T + s];
}

#include "wave_reg.cuh"

// Above 4096 points one frame's two Stockham buffers and the twiddle table
// (199 KB at 16384) leave room for a single CTA per SM.  Those sizes
// transform in place instead (one buffer laid out with fft::LayoutIP, the
// twiddle rows read through L1, a separate power row, samples loaded
// without staging), which fits two 512-thread CTAs per SM.  32 clips of
// 160000 samples, hop n_fft / 4, L2 flushed, us per call: 8192: 155.6 with
// one 1024-thread Stockham CTA, 145.4 in place with one padding level,
// 141.1 with LayoutIP's two; 16384: 137.2 Stockham, 147.5 in place with one
// level, 133.1 with two.  (With direct framing, the filterbank image, and
// the radix-16 first pass fused with the framing: 94.7 and 99.9.)
constexpr bool in_place_nfft(int n_fft) { return n_fft >= 8192; }

template <int NFFT>
struct WaveCfg {
  static constexpr int M = NFFT / 2;
  static constexpr bool kInPlace = in_place_nfft(NFFT);
  static constexpr int NF = NFFT / 2 + 1;
  static constexpr int NFP = NF | 1;  // odd power-tile row stride
  // Frames per tile, bounded by shared memory.  Up to 1024 points, 8: at
  // n_fft 400 two 16-frame CTAs per SM were 8% slower than eight-frame ones
  // (more CTAs hide each other's barriers), and at 1024 four frames were 22%
  // slower.
  static constexpr int TF = NFFT <= 1024 ? 8 : (NFFT <= 4096 ? 2 : 1);
  // Threads per CTA (a multiple of TF: the mel phase maps a thread to one
  // frame of a band group).  256 with 8-frame tiles beat every other pairing
  // tried at 400 points (160-640 threads, 8 or 16 frames: 50-79 us against
  // 48) and at 1024 (128-512 threads, 4-16 frames: 101-129 us against 95).
  // Above that shared memory allows one CTA per SM, whose barrier-separated
  // passes need more warps to hide their latency: 32 clips of 160000 samples,
  // hop n_fft / 4, 128 bands, L2 flushed, us per call with 256 / 512 / 1024
  // threads: 2048: 84.0 / 124.9 / 147.5; 4096: 105.5 / 94.2 / 106.5; 8192:
  // 303.1 / 188.4 / 155.6; 16384: 313.3 / 190.5 / 138.2.  8192 and 16384 now
  // run in place (see in_place_nfft): 16384 with two 512-thread CTAs per SM,
  // 8192 with four of 256 threads, whose 50 KB of shared memory allow it
  // (86.5 us against 94.3 with two of 512).
  static constexpr int NT = (NFFT == 4096 || NFFT == 16384) ? 512 : 256;
  static_assert(NT % 32 == 0 && NT % TF == 0, "thread count");
  // Up to 4096 every table sits in shared memory; beyond, only the FFT
  // twiddles do and the window, untangle twiddles and filterbank are read
  // through L1 from global memory.
  static constexpr bool kSmallTables = NFFT <= 4096;
  // CTAs per SM that shared memory allows at these sizes; registers are
  // capped to match so they do not lower the occupancy further.  400 points
  // gets no minimum (0): the compiler's own choice there is 64 registers,
  // while an explicit 4 made it spill and 1 let it take 104.
  static constexpr int kMinBlocks =
      NFFT == 400 ? 0 : (NFFT <= 512 || NFFT == 8192 ? 4 : (NFFT <= 1024 || kInPlace ? 2 : 1));
  static constexpr bool kFuseFirst = (M & (M - 1)) == 0;
  // The power tile (TF rows of NFP floats) lives in whichever FFT buffer does
  // not hold the transform's result; it needs at most half of it.
  static constexpr bool kResultInB = fft::num_passes<M>() % 2 == 1;
  using L = std::conditional_t<kInPlace, fft::LayoutIP<M>, fft::Layout<M>>;
  static constexpr int BUF = L::size(TF * M);  // float2 slots per FFT buffer
  static_assert(TF * NFP * sizeof(float) <= BUF * sizeof(float2), "power tile must fit an FFT buffer");
};

// Bytes of the table image up to 4096 points: tw_m [M] float2 | tw_n [M+1]
// float2 and one float2 of padding | fw [n_mels*wmax] | window [NFFT] |
// {fstart, fwidth} [n_mels] int2, rounded up to 16 (one bulk copy).  fw
// starts 16-byte aligned (M is even) and wmax is a multiple of 4, so the
// mel phase reads four weights with one 16-byte load.
inline uint32_t wave_tables_bytes(int n_fft, int n_mels, int wmax) {
  const size_t M = n_fft / 2;
  const size_t b = 8 * (2 * M + 2) + 4 * static_cast<size_t>(n_mels) * wmax + 4 * static_cast<size_t>(n_fft) +
                   8 * static_cast<size_t>(n_mels);
  return static_cast<uint32_t>((b + 15) / 16 * 16);
}

// Shared memory: bufA, bufB [BUF] float2 (TF frames of M points at Layout<M>
// positions; the power tile reuses one) | the table image (tw_m only above
// 4096 points) | keys
//
// In place (above 4096 points): buf [BUF] float2 | power row [NFP + 1] | keys.
template <int NFFT>
size_t wave_smem_bytes(int n_mels, int wmax) {
  using C = WaveCfg<NFFT>;
  size_t b = 2 * sizeof(float2) * C::BUF;
  b += sizeof(float2) * C::M;
  if (C::kSmallTables) {
    b -= sizeof(float2) * C::M;
    b += wave_tables_bytes(NFFT, n_mels, wmax);
  }
  if (C::kInPlace) b = sizeof(float2) * C::BUF + sizeof(float) * (C::NFP + 1);
  b += 16;  // tile key, abort flag, next tile
  return (b + 127) / 128 * 128;  // the sample-span buffers follow, 128-byte aligned
}

// The in-place transform's filterbank image, copied into the transform's
// buffer once the power row is complete: n_mels + 1 int2 {first bin of band
// m, offset of its weights} (the last holds only the total, so band m's
// width is the difference of two offsets), then every band's weights back
// to back.  Zero (the projection then reads the plan's global tables) when
// it does not fit the buffer: 128 bands fit at both sizes.
inline uint32_t mel_image_bytes_for(int n_fft, int n_mels, const std::vector<int> &fwidth) {
  size_t taps = 0;
  for (int m = 0; m < n_mels; ++m) taps += static_cast<size_t>(fwidth[m]);
  const size_t bytes = (8 * (static_cast<size_t>(n_mels) + 1) + 4 * taps + 15) / 16 * 16;
  size_t room = 0;
  if (n_fft == 8192) room = sizeof(float2) * WaveCfg<8192>::BUF;
  if (n_fft == 16384) room = sizeof(float2) * WaveCfg<16384>::BUF;
  return bytes <= room ? static_cast<uint32_t>(bytes) : 0u;
}

// A sample pair as a complex point: f32 pairs as they are, int16 pairs (one
// 32-bit word) scaled by 1/32768.
__device__ __forceinline__ float2 pair_point(float2 v) { return v; }
__device__ __forceinline__ float2 pair_point(int v) {
  return make_float2(static_cast<float>(static_cast<int16_t>(v & 0xffff)) * (1.0f / 32768.0f),
                     static_cast<float>(static_cast<int16_t>(v >> 16)) * (1.0f / 32768.0f));
}

// Framing of an interior frame for the in-place transform, its sample pairs
// aligned, fused with the transform's first pass (radix 16, span 1, no
// twiddle factors): thread g < M/16 loads the 16 points g + j M/16 (sample
// pairs and window pairs, 8 of each in flight at a time), windows them, runs
// the 16-point DFT in registers and stores output l at 16 dit_pos<M/16>(g) + l,
// where the pass would have written it.  src points at the frame's first
// sample pair.
template <int M, int NT, typename Pair>
__device__ __forceinline__ void frame_first_pass(const Pair *src, const float2 *win2, float2 *buf) {
  constexpr int S = M / 16;
  static_assert(fft::ip_radix<M, 1>() == 16 && S <= NT, "one first-pass butterfly per thread");
  const int g = static_cast<int>(threadIdx.x);
  if (S < NT && g >= S) return;
  float2 u[16];
#pragma unroll
  for (int c = 0; c < 16; c += 8) {
    Pair x[8];
    float2 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = g + (c + j) * S;
      x[j] = __ldg(src + n);
      w[j] = __ldg(win2 + n);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 v = pair_point(x[j]);
      u[c + j] = make_float2(v.x * w[j].x, v.y * w[j].y);
    }
  }
  fft::Dft<16>::run(u);
  const int base = 16 * fft::dit_pos<S>(g);
#pragma unroll
  for (int l = 0; l < 16; ++l) buf[fft::LayoutIP<M>::at(base + l)] = u[l];
}

template <int NFFT>
__global__ void __launch_bounds__(WaveCfg<NFFT>::NT, WaveCfg<NFFT>::kMinBlocks) wave_mel_kernel(const WaveArgs a) {
  using C = WaveCfg<NFFT>;
  constexpr int M = C::M, TF = C::TF, NFP = C::NFP, NT = C::NT;
  extern __shared__ __align__(16) unsigned char smem[];
  float2 *bufA = reinterpret_cast<float2 *>(smem);
  float2 *bufB = bufA + C::BUF;  // (not used in place)
  float *pw = C::kInPlace ? reinterpret_cast<float *>(bufA + C::BUF)
                          : reinterpret_cast<float *>(C::kResultInB ? bufA : bufB);
  float2 *twm = bufB + C::BUF;
  float2 *twn_s = twm + M;
  float *fw_s = reinterpret_cast<float *>(twn_s + M + 2);  // 16-byte aligned
  float *win_s = fw_s + a.n_mels * a.wmax;
  int2 *fsw_s = reinterpret_cast<int2 *>(win_s + NFFT);  // {first bin, width} per band
  uint32_t *blk_key = C::kSmallTables ? reinterpret_cast<uint32_t *>(reinterpret_cast<unsigned char *>(twm) + a.tables_bytes)
                      : C::kInPlace   ? reinterpret_cast<uint32_t *>(pw + NFP + 1)
                                      : reinterpret_cast<uint32_t *>(twm + M);
  const float2 *twn = C::kSmallTables ? twn_s : a.tw_n;
  const float *win = C::kSmallTables ? win_s : a.window;
  const int *fstart = a.fstart;  // global: one-frame tiles only
  const int *fwidth = a.fwidth;
  const float *fw = C::kSmallTables ? fw_s : a.fw;
  int *abort_flag_p = reinterpret_cast<int *>(blk_key + 1);
  volatile int *abort_flag = abort_flag_p;
  unsigned char *seg = smem + a.seg_offset;  // two buffers of seg_bytes
  uint64_t *seg_bar = reinterpret_cast<uint64_t *>(seg + 2 * static_cast<size_t>(a.seg_bytes));  // [2]: tables
  const int es = a.in_i16 ? 2 : 4;

  // The contiguous samples an interior tile (no padding in play) reads:
  // bulk-copy range [a0, a0 + bytes) of the waveform, 16-byte aligned.
  auto span_of = [&](int64_t tile, uint64_t *a0, uint32_t *bytes) -> bool {
    if constexpr (C::kInPlace) return false;  // no staging buffers in that layout
    if (!a.use_seg) return false;
    const int64_t b = tile / a.tiles_per_clip;
    const int64_t t0 = (tile - b * a.tiles_per_clip) * static_cast<int64_t>(TF);
    const int64_t left = a.n_frames - t0;
    const int nf = left < TF ? static_cast<int>(left) : TF;
    const int64_t s_first = t0 * a.hop - a.pad_left;
    const int64_t s_last = (t0 + nf - 1) * a.hop - a.pad_left + NFFT - 1;
    if (s_first < 0 || s_last >= a.T) return false;
    const uint64_t start = static_cast<uint64_t>(b * a.T + s_first) * es;
    const uint64_t end = static_cast<uint64_t>(b * a.T + s_last + 1) * es;
    *a0 = start & ~15ull;
    const uint64_t a1 = (end + 15ull) & ~15ull;
    if (a1 > a.total_bytes) return false;
    *bytes = static_cast<uint32_t>(a1 - *a0);
    return true;
  };
  uint32_t issued[2] = {0u, 0u};  // span copies issued per buffer (thread 0)
  auto issue_span = [&](int64_t tile, int buf) {
    uint64_t a0;
    uint32_t bytes;
    if (span_of(tile, &a0, &bytes)) {
      // (checked builds) the span lies inside the waveform and fits its
      // buffer; if not, nothing is copied and the error word says so
      const bool ok = LM_IN_BOUNDS(a0, a.total_bytes, a.err) && LM_IN_BOUNDS(a0 + bytes - 1, a.total_bytes, a.err) &&
                      LM_IN_BOUNDS(bytes - 1, a.seg_bytes, a.err);
      mbar_arrive_expect_tx(&seg_bar[buf], ok ? bytes : 0u);
      if (ok)
        bulk_g2s(seg + buf * static_cast<size_t>(a.seg_bytes), static_cast<const char *>(a.wave) + a0, bytes,
                 &seg_bar[buf], policy_evict_first());
      ++issued[buf];
    }
  };
  // Before the CTA exits, thread 0 waits until every copy it issued has
  // landed (immediate unless a wait gave up and the loop was left early).
  auto drain = [&](bool tables) {
    if (threadIdx.x != 0) return;
    if (tables) mbar_wait_drain(&seg_bar[2], 0u, a.err);
    for (int b = 0; b < 2; ++b)
      if (issued[b] > 0) mbar_wait_drain(&seg_bar[b], (issued[b] - 1u) & 1u, a.err);
  };
  if (threadIdx.x == 0) {
    if (a.token != 0 && blockIdx.x == 0) publish_cleared(a);
    mbar_init(&seg_bar[0], 1);
    mbar_init(&seg_bar[1], 1);
    mbar_init(&seg_bar[2], 1);
    *abort_flag_p = 0;
    fence_mbar_init();
    if constexpr (C::kSmallTables) {
      // every table in one bulk copy of the plan's shared-memory image
      mbar_arrive_expect_tx(&seg_bar[2], a.tables_bytes);
      bulk_g2s_plain(twm, a.tables, a.tables_bytes, &seg_bar[2]);
    }
    if (blockIdx.x < a.B * a.tiles_per_clip) issue_span(blockIdx.x, 0);
  }
  uint32_t fill0 = 0u, fill1 = 0u;  // completed span copies per buffer (the same in every thread)

  if constexpr (C::kSmallTables) {
    __syncthreads();  // the barrier is initialised
    // Without the tables every later shared-memory index is meaningless:
    // if any thread's wait gave up, the whole CTA stops here.
    const bool ok = mbar_wait(&seg_bar[2], 0, abort_flag, a.err);
    if (__syncthreads_or(!ok)) {
      drain(true);
      return;
    }
  } else {
    if constexpr (!C::kInPlace) {
      for (int i = threadIdx.x; i < M; i += blockDim.x) twm[i] = a.tw_m[i];
    }
    // Thread 0's abort flag and barriers are initialised before any thread
    // reads the flag below (that read precedes the loop's first barrier).
    __syncthreads();
  }

  // Tiles are handed out dynamically: a CTA's first tile is its index, each
  // later one comes from a counter in the workspace header (zeroed per
  // call), claimed at the start of the tile before it; once that tile's
  // framing is done, the claimed tile's samples are prefetched.  (Claiming
  // two ahead measured slower: the last tiles go to CTAs that are not yet
  // free.)
  const int64_t n_tiles = a.B * a.tiles_per_clip;
  volatile int *next_s = reinterpret_cast<volatile int *>(blk_key + 2);  // n_tiles < 2^31 (host check)
  int it = 0;
  uint32_t mel_phase = 0u;  // filterbank image copies completed (in place)
  bool token_seen = a.token == 0;  // thread 0
  for (int64_t tile = blockIdx.x, nxt; tile < n_tiles; tile = nxt, ++it) {
    const int buf = it & 1;
    const int64_t b = tile / a.tiles_per_clip;
    const int tloc = static_cast<int>(tile - b * a.tiles_per_clip);
    const int64_t t0 = static_cast<int64_t>(tloc) * TF;
    const int64_t left = a.n_frames - t0;
    const int nf = left < TF ? static_cast<int>(left) : TF;
    // Thread 0 claims the next tile now and uses the answer only after this
    // tile's framing, so the counter's round trip overlaps the framing.
    int claimed = 0;
    if (threadIdx.x == 0) {
      *blk_key = 0u;
      claimed = claim_tile(a, &token_seen, abort_flag_p, static_cast<int>(n_tiles));
    }
    // Tables loaded / previous tile finished with every buffer.  A wait that
    // gave up in the previous tile (its values are then wrong, but every
    // index stayed in bounds) ends the loop in every thread together.
    if (__syncthreads_or(*abort_flag != 0)) break;
    uint64_t span_a0;
    uint32_t span_bytes;
    const bool staged = span_of(tile, &span_a0, &span_bytes);
    if (staged) {
      mbar_wait(&seg_bar[buf], (buf ? fill1 : fill0) & 1u, abort_flag, a.err);
      if (buf) ++fill1; else ++fill0;
    }

    // 1. framing, padding, window, pairing into complex points
    const int64_t s_first = t0 * a.hop - a.pad_left;
    const int64_t s_last = (t0 + nf - 1) * a.hop - a.pad_left + NFFT - 1;
    const bool interior = s_first >= 0 && s_last < a.T;
    // staged: sample s of the clip is element (s - s_first) + head of the span buffer
    const int64_t head = staged ? (static_cast<int64_t>(b * a.T + s_first) * es - static_cast<int64_t>(span_a0)) / es : 0;
    const float *segf = reinterpret_cast<const float *>(seg + buf * static_cast<size_t>(a.seg_bytes));
    const int16_t *segh = reinterpret_cast<const int16_t *>(segf);
    // Staged tile whose sample pairs (2n, 2n+1) are aligned in the span
    // buffer (even head and hop): one 8-byte (f32) or 4-byte (i16) load per
    // complex point, the window as pairs too, compile-time trip count.
    const bool paired = staged && ((static_cast<int>(head) | a.hop) & 1) == 0;
    // Power-of-two sizes fuse the framing into the first FFT pass; at 400
    // points the fused radix-5 pass measured slower than framing on its own.
    const bool fused = paired && C::kFuseFirst;
    bool gathered = false;  // in place: the frame is in the buffer, its first pass done
    if constexpr (C::kInPlace) {
      const int64_t p0 = b * a.T + s_first;  // the frame's first sample
      if (interior && ((reinterpret_cast<uintptr_t>(a.wave) & (a.in_i16 ? 3u : 7u)) == 0) && (p0 & 1) == 0 &&
          LM_IN_BOUNDS(p0 + NFFT - 1, a.B * a.T, a.err)) {
        const float2 *win2 = reinterpret_cast<const float2 *>(win);
        if (a.in_i16)
          frame_first_pass<M, NT>(reinterpret_cast<const int *>(static_cast<const int16_t *>(a.wave) + p0), win2,
                                  bufA);
        else
          frame_first_pass<M, NT>(reinterpret_cast<const float2 *>(static_cast<const float *>(a.wave) + p0), win2,
                                  bufA);
        gathered = true;
      }
    }
    if (paired && !fused) {
      // 32-bit shared addresses; thread idx handles point n of frame f.
      constexpr int ITEMS = TF * M;
      const uint32_t seg0 = smem_u32(segf) + static_cast<uint32_t>(head) * es;
      const uint32_t win0 = C::kSmallTables ? smem_u32(win) : 0u;
      const float2 *win_g = reinterpret_cast<const float2 *>(win);
      const uint32_t dst0 = smem_u32(bufA);
      const bool i16 = a.in_i16 != 0;
#pragma unroll 4
      for (int r = 0; r < (ITEMS + NT - 1) / NT; ++r) {
        const int idx = static_cast<int>(threadIdx.x) + r * NT;
        if (ITEMS % NT != 0 && idx >= ITEMS) break;
        const int f = idx / M;
        const int n = idx - f * M;
        float2 z = make_float2(0.f, 0.f);
        if (f < nf) {
          const uint32_t e = static_cast<uint32_t>(f * a.hop + 2 * n);  // sample offset from head, even
          float2 x;
          if (i16) {
            const int v = lds_s32(seg0 + 2u * e);
            x = make_float2(static_cast<float>(static_cast<int16_t>(v & 0xffff)) * (1.0f / 32768.0f),
                            static_cast<float>(static_cast<int16_t>(v >> 16)) * (1.0f / 32768.0f));
          } else {
            x = lds_f32x2(seg0 + 4u * e);
          }
          float2 w;
          if constexpr (C::kSmallTables) {
            w = lds_f32x2(win0 + 8u * static_cast<uint32_t>(n));
          } else {
            w = win_g[n];
          }
          z = make_float2(x.x * w.x, x.y * w.y);
        }
        sts_f32x2(dst0 + 8u * static_cast<uint32_t>(C::L::at(idx)), z);
      }
    }
    if constexpr (C::kFuseFirst) if (fused) {
      // Framing fused into the first FFT pass (span P = 1, radix R0): the
      // thread of butterfly i of frame f loads its R0 complex points
      // n = i + j M/R0 straight from the span buffer (one 8-byte f32 or
      // 4-byte i16 load per point), windows them, transforms and stores to
      // bufB -- one shared-memory round trip and one barrier fewer.
      constexpr int R0 = fft::next_radix<M, 1>();
      constexpr int T = M / R0;
      constexpr int ITEMS = TF * T;
      const uint32_t seg0 = smem_u32(segf) + static_cast<uint32_t>(head) * es;
      const uint32_t win0 = C::kSmallTables ? smem_u32(win) : 0u;  // the window is in shared memory only with the small tables
      const float2 *win_g = reinterpret_cast<const float2 *>(win);
      const uint32_t dst0 = smem_u32(bufB);
      const bool i16 = a.in_i16 != 0;
#pragma unroll 2
      for (int r = 0; r < (ITEMS + NT - 1) / NT; ++r) {
        const int g = static_cast<int>(threadIdx.x) + r * NT;
        if (ITEMS % NT != 0 && g >= ITEMS) break;
        const int f = g / T;
        const int i = g - f * T;
        float2 u[R0];
#pragma unroll
        for (int j = 0; j < R0; ++j) {
          const int n = i + j * T;
          u[j] = make_float2(0.f, 0.f);
          if (f < nf) {
            const uint32_t e = static_cast<uint32_t>(f * a.hop + 2 * n);  // sample offset from head, even
            float2 x;
            if (i16) {
              const int v = lds_s32(seg0 + 2u * e);
              x = make_float2(static_cast<float>(static_cast<int16_t>(v & 0xffff)) * (1.0f / 32768.0f),
                              static_cast<float>(static_cast<int16_t>(v >> 16)) * (1.0f / 32768.0f));
            } else {
              x = lds_f32x2(seg0 + 4u * e);
            }
            float2 w;
            if constexpr (C::kSmallTables) {
              w = lds_f32x2(win0 + 8u * static_cast<uint32_t>(n));
            } else {
              w = win_g[n];
            }
            u[j] = make_float2(x.x * w.x, x.y * w.y);
          }
        }
        fft::Dft<R0>::run(u);
#pragma unroll
        for (int l = 0; l < R0; ++l)
          sts_f32x2(dst0 + 8u * static_cast<uint32_t>(C::L::at(f * M + i * R0 + l)), u[l]);
      }
    }
    for (int idx = (paired || gathered) ? TF * M : static_cast<int>(threadIdx.x); idx < TF * M; idx += blockDim.x) {
      const int f = idx / M;
      const int n = idx - f * M;
      float2 z = make_float2(0.f, 0.f);
      if (f < nf) {
        const int64_t s = (t0 + f) * a.hop - a.pad_left + 2 * n;
        float x0, x1;
        if (staged) {
          const int e = static_cast<int>(head) + f * a.hop + 2 * n;
          if (a.in_i16) {
            x0 = static_cast<float>(segh[e]) * (1.0f / 32768.0f);
            x1 = static_cast<float>(segh[e + 1]) * (1.0f / 32768.0f);
          } else {
            x0 = segf[e];
            x1 = segf[e + 1];
          }
        } else if (interior) {
          x0 = load_sample(a, b, s);
          x1 = load_sample(a, b, s + 1);
        } else {
          // Centre padding applies to the signal already extended by pad_zero
          // zeros on both sides (length T + 2 pad_zero); map there, then back.
          const int64_t Tz = a.T + 2 * a.pad_zero;
          bool z0, z1;
          const int64_t i0 = map_index(s + a.pad_zero, Tz, a.pad_mode, &z0) - a.pad_zero;
          const int64_t i1 = map_index(s + 1 + a.pad_zero, Tz, a.pad_mode, &z1) - a.pad_zero;
          x0 = (z0 || i0 < 0 || i0 >= a.T) ? 0.f : load_sample(a, b, i0);
          x1 = (z1 || i1 < 0 || i1 >= a.T) ? 0.f : load_sample(a, b, i1);
        }
        z = make_float2(x0 * win[2 * n], x1 * win[2 * n + 1]);
      }
      // in place, point n goes to its digit-reversed position (one frame a tile)
      bufA[C::L::at(C::kInPlace ? fft::dit_pos<M>(n) : idx)] = z;
    }
    __syncthreads();
    // Publish the next tile (read after the untangle's barrier) and prefetch
    // its samples into the other span buffer, whose last reader, the previous
    // tile's framing, finished two barriers ago.
    if (threadIdx.x == 0) {
      *next_s = claimed;
      if (claimed < n_tiles) issue_span(claimed, buf ^ 1);
    }

    // 2. N/2-point complex FFT of every frame (its first pass already done
    // for aligned staged tiles, whose result is then in bufB)
    bool in_b;
    if constexpr (C::kInPlace) {
      // (frames gathered point by point still need the first pass)
      constexpr int R0 = fft::ip_radix<M, 1>();
      if (!gathered) {
        fft::pass_inplace<M, R0, 1, NT>(bufA, a.tw_m);
        __syncthreads();
      }
      fft::run_inplace<M, NT, R0>(bufA, a.tw_m);
      in_b = false;
    } else if constexpr (C::kFuseFirst) {
      if (fused) {
        in_b = !fft::run<M, TF, NT, fft::next_radix<M, 1>()>(bufB, bufA, twm);
      } else {
        in_b = fft::run<M, TF, NT>(bufA, bufB, twm);
      }
    } else {
      in_b = fft::run<M, TF, NT>(bufA, bufB, twm);
    }
    const float2 *Z = in_b ? bufB : bufA;  // == kResultInB; pw is the other buffer

    // 3. untangle the real spectrum and take |X|^power.  Bins k and M - k
    // come from the same two values: with A = Z[k], B = Z[M-k],
    // E = (A + conj B) / 2, O = (A - conj B) / (2i) and tw = exp(-2 pi i k / N),
    // X[k] = E + tw O and X[M-k] = conj(E - tw O).  k = 0 gives X[0] and
    // X[M]; k = M/2 is its own partner.
    {
      constexpr int KP = M / 2 + 1;  // pairs per frame (M is even)
      constexpr int ITEMS = TF * KP;
      constexpr int ROUNDS = (ITEMS + NT - 1) / NT;
      auto untangle = [&](int idx, float2 tw) {
        const int f = idx / KP;
        const int k = idx - f * KP;
        const float2 A = Z[C::L::at(f * M + k)];
        const float2 Bz = Z[C::L::at(f * M + (k == 0 ? 0 : M - k))];
        const float2 E = make_float2(0.5f * (A.x + Bz.x), 0.5f * (A.y - Bz.y));
        // O = (A - conj B) / (2i) = -i (A - conj B) / 2
        const float2 O = make_float2(0.5f * (A.y + Bz.y), -0.5f * (A.x - Bz.x));
        const float2 TO = fft::cmul(tw, O);
        float p0 = fmaf(E.x + TO.x, E.x + TO.x, (E.y + TO.y) * (E.y + TO.y));
        float p1 = fmaf(E.x - TO.x, E.x - TO.x, (E.y - TO.y) * (E.y - TO.y));
        if (a.power_is_one) {
          p0 = sqrtf(p0);
          p1 = sqrtf(p1);
        }
        pw[f * NFP + k] = p0;
        if (k != M / 2) pw[f * NFP + M - k] = p1;
      };
      if constexpr (C::kInPlace) {
        // One frame (TF = 1, so idx = k); the twiddles come from global
        // memory, all of this thread's in flight at once.
        float2 tw[ROUNDS];
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
          const int idx = static_cast<int>(threadIdx.x) + r * NT;
          tw[r] = (ITEMS % NT == 0 || idx < ITEMS) ? __ldg(twn + idx) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
          const int idx = static_cast<int>(threadIdx.x) + r * NT;
          if (ITEMS % NT != 0 && idx >= ITEMS) break;
          untangle(idx, tw[r]);
        }
      } else {
#pragma unroll 2
        for (int r = 0; r < ROUNDS; ++r) {
          const int idx = static_cast<int>(threadIdx.x) + r * NT;
          if (ITEMS % NT != 0 && idx >= ITEMS) break;
          untangle(idx, twn[idx - (idx / KP) * KP]);
        }
      }
    }
    __syncthreads();
    nxt = *next_s;

    // 4. mel projection and store
    float lmax = -INFINITY;
    const int64_t orow0 = b * a.n_mels * a.n_frames + t0;  // output index of (band 0, frame 0) of this tile
    auto emit = [&](int m, int f, float acc) {
      const int64_t o = orow0 + static_cast<int64_t>(m) * a.n_frames + f;
      if (a.log_mel) {
        float l2;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(fmaxf(acc, 1e-10f)));
        const float v = l2 * 0.30102999566398120f;  // log10(x) = log2(x) log10(2)
        lmax = fmaxf(lmax, v);
        if (LM_IN_BOUNDS(o, a.B * a.n_mels * a.n_frames, a.err)) static_cast<float *>(a.out)[o] = v;
      } else if (a.out_f16) {
        if (LM_IN_BOUNDS(o, a.B * a.n_mels * a.n_frames, a.err)) static_cast<__half *>(a.out)[o] = __float2half_rn(acc);
      } else {
        if (LM_IN_BOUNDS(o, a.B * a.n_mels * a.n_frames, a.err)) static_cast<float *>(a.out)[o] = acc;
      }
    };
    if constexpr (TF == 1) {
      // One frame, filters hundreds of bins wide: a warp per band, lanes
      // over taps, then a shuffle reduction.
      const int lane = threadIdx.x & 31;
      bool from_smem = false, skip = false;
      if constexpr (C::kInPlace) {
        if (a.mel_image != nullptr) {
          // The transform's buffer is free once the power row is complete:
          // the plan's filterbank image goes there in one bulk copy, and the
          // projection then reads shared memory only (from global memory
          // every band paid dependent L2 round trips for its support and
          // its weights).
          if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&seg_bar[0], a.mel_image_bytes);
            bulk_g2s_plain(bufA, a.mel_image, a.mel_image_bytes, &seg_bar[0]);
            ++issued[0];
          }
          const bool ok = mbar_wait(&seg_bar[0], mel_phase & 1u, abort_flag, a.err);
          ++mel_phase;
          // a wait that gave up leaves this tile's output unwritten (the
          // abort flag ends the loop at the next barrier)
          from_smem = __all_sync(0xffffffffu, ok);
          skip = !from_smem;
        }
      }
      if (skip) {
      } else if (from_smem) {
        // G bands of the warp at a time (m, m + NW, ...): their tap loops and
        // shuffle reductions are independent chains, interleaved.  Each
        // band's sum is formed in the same order as one band at a time.
        constexpr int G = 4, NW = NT / 32;
        const uint32_t hdr = smem_u32(bufA);
        const uint32_t wts = hdr + 8u * static_cast<uint32_t>(a.n_mels + 1);
        const uint32_t pw0 = smem_u32(pw);
        for (int m0 = threadIdx.x >> 5; m0 < a.n_mels; m0 += G * NW) {
          uint32_t wa[G], pa[G];
          int wd[G], wmx = 0;
          float acc[G];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const int m = m0 + g * NW;
            const int2 h = m < a.n_mels ? lds_s32x2(hdr + 8u * m) : make_int2(0, 0);  // {first bin, offset}
            wd[g] = m < a.n_mels ? lds_s32(hdr + 8u * (m + 1) + 4u) - h.y : 0;
            wa[g] = wts + 4u * static_cast<uint32_t>(h.y);
            pa[g] = pw0 + 4u * static_cast<uint32_t>(h.x);
            acc[g] = 0.f;
            wmx = max(wmx, wd[g]);
          }
          for (int t = lane; t < wmx; t += 32) {
#pragma unroll
            for (int g = 0; g < G; ++g)
              if (t < wd[g]) acc[g] = fmaf(lds_f32(wa[g] + 4u * t), lds_f32(pa[g] + 4u * t), acc[g]);
          }
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], d);
          }
          if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g)
              if (m0 + g * NW < a.n_mels) emit(m0 + g * NW, 0, acc[g]);
          }
        }
      } else {
        for (int m = threadIdx.x >> 5; m < a.n_mels; m += NT / 32) {
          const int st = fstart[m], wd = fwidth[m];
          const float *w = fw + m * a.wmax;
          float acc = 0.f;
          for (int t = lane; t < wd; t += 32) acc = fmaf(w[t], pw[st + t], acc);
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
          if (lane == 0) emit(m, 0, acc);
        }
      }
    } else {
      // Thread = (frame f, band group): lanes run over the TF frames of one
      // band, so each band's output row is written as a run of consecutive
      // frames; the group walks bands m0, m0 + NG, ...  Shared memory is
      // addressed with 32-bit offsets.
      constexpr int NG = NT / TF;
      const int f = static_cast<int>(threadIdx.x) % TF;
      if (f < nf) {
        const uint32_t prow = smem_u32(pw) + static_cast<uint32_t>(f * NFP) * 4u;
        const int m0 = static_cast<int>(threadIdx.x) / TF;
        uint32_t fsw = smem_u32(fsw_s) + static_cast<uint32_t>(m0) * 8u;
        uint32_t wa = smem_u32(fw_s) + static_cast<uint32_t>(m0 * a.wmax) * 4u;
        const uint32_t wstep = static_cast<uint32_t>(NG * a.wmax) * 4u;
        for (int m = m0; m < a.n_mels; m += NG, fsw += NG * 8, wa += wstep) {
          const int2 sw = lds_s32x2(fsw);
          const uint32_t pa = prow + static_cast<uint32_t>(sw.x) * 4u;
          float acc = 0.f;
          int t = 0;
          // Weight rows start 16-byte aligned (wmax is a multiple of 4): four
          // weights per load; the power row has no such alignment.
          for (; t + 4 <= sw.y; t += 4) {
            const float4 w4 = lds_f32x4(wa + 4 * t);
            acc = fmaf(w4.x, lds_f32(pa + 4 * t), acc);
            acc = fmaf(w4.y, lds_f32(pa + 4 * t + 4), acc);
            acc = fmaf(w4.z, lds_f32(pa + 4 * t + 8), acc);
            acc = fmaf(w4.w, lds_f32(pa + 4 * t + 12), acc);
          }
          if (t < sw.y) {
            const float4 w4 = lds_f32x4(wa + 4 * t);
            acc = fmaf(w4.x, lds_f32(pa + 4 * t), acc);
            if (t + 1 < sw.y) acc = fmaf(w4.y, lds_f32(pa + 4 * t + 4), acc);
            if (t + 2 < sw.y) acc = fmaf(w4.z, lds_f32(pa + 4 * t + 8), acc);
          }
          emit(m, f, acc);
        }
      }
    }
    if (a.log_mel) {
      const uint32_t key = __reduce_max_sync(0xffffffffu, float_to_ordered(lmax));
      if ((threadIdx.x & 31) == 0) atomicMax(blk_key, key);
      __syncthreads();
      if (threadIdx.x == 0 && LM_IN_BOUNDS(tile, a.B * a.tiles_per_clip, a.err)) a.tile_key[tile] = *blk_key;
    }
  }
  drain(false);
  // This CTA is done: a programmatically dependent epilogue may be scheduled
  // (it still waits for the whole grid before reading).
  asm volatile("griddepcontrol.launch_dependents;");
}

using WaveKernel = void (*)(WaveArgs);

template <int NFFT>
void wave_entry(WaveKernel *k, size_t *smem, int *tf, int *nt, int n_mels, int wmax) {
  *k = wave_mel_kernel<NFFT>;
  *smem = wave_smem_bytes<NFFT>(n_mels, wmax);
  *tf = WaveCfg<NFFT>::TF;
  *nt = WaveCfg<NFFT>::NT;
}

// The register kernel of a size and its launch shape.
template <int NFFT>
void reg_entry(WaveKernel *k, size_t *smem, int *tf, int *nt, int n_mels, int wmax) {
  *k = reg::wave_reg_kernel<NFFT>;
  *smem = reg::smem_bytes<NFFT>(n_mels, wmax);
  *tf = reg::Cfg<NFFT>::TF;
  *nt = reg::Cfg<NFFT>::NT;
}

bool pick_wave_kernel(int n_fft, int n_mels, int wmax, WaveKernel *k, size_t *smem, int *tf, int *nt) {
  switch (n_fft) {
    case 64: wave_entry<64>(k, smem, tf, nt, n_mels, wmax); return true;
    case 128: wave_entry<128>(k, smem, tf, nt, n_mels, wmax); return true;
    case 256: wave_entry<256>(k, smem, tf, nt, n_mels, wmax); return true;
    case 400: wave_entry<400>(k, smem, tf, nt, n_mels, wmax); return true;
    case 512: wave_entry<512>(k, smem, tf, nt, n_mels, wmax); return true;
    case 1024: wave_entry<1024>(k, smem, tf, nt, n_mels, wmax); return true;
    case 2048: wave_entry<2048>(k, smem, tf, nt, n_mels, wmax); return true;
    case 4096: wave_entry<4096>(k, smem, tf, nt, n_mels, wmax); return true;
    case 8192: wave_entry<8192>(k, smem, tf, nt, n_mels, wmax); return true;
    case 16384: wave_entry<16384>(k, smem, tf, nt, n_mels, wmax); return true;
    default: return false;
  }
}

bool supported_nfft(int n) {
  if (n == 400) return true;
  if (n < 64 || n > 16384) return false;
  return (n & (n - 1)) == 0;
}

// ---- host-side tables, double precision ----

double hz_to_mel(double hz, int scale) {
  if (scale == LM_MEL_HTK) return 2595.0 * std::log10(1.0 + hz / 700.0);
  // Slaney: 3 mels per 200 Hz up to 1 kHz (mel 15), then 27 mels per factor 6.4
  if (hz < 1000.0) return 3.0 * hz / 200.0;
  return 15.0 + 27.0 * std::log(hz / 1000.0) / std::log(6.4);
}

double mel_to_hz(double mel, int scale) {
  if (scale == LM_MEL_HTK) return 700.0 * (std::pow(10.0, mel / 2595.0) - 1.0);
  if (mel < 15.0) return 200.0 * mel / 3.0;
  return 1000.0 * std::exp((mel - 15.0) * std::log(6.4) / 27.0);
}

struct HostTables {
  std::vector<float> window;
  std::vector<float2> tw_m, tw_n;
  std::vector<int> fstart, fwidth;
  std::vector<float> fw;
  int wmax = 0;
};

void build_tables(const lm_mel_params &p, HostTables *t) {
  const int N = p.n_fft, M = N / 2, n_freqs = N / 2 + 1;
  const int wl = p.win_length > 0 ? p.win_length : N;
  std::vector<double> w(N, 0.0);
  const int left = (N - wl) / 2;
  double energy = 0.0;
  for (int j = 0; j < wl; ++j) {
    const double v = 0.5 - 0.5 * std::cos(2.0 * M_PI * j / wl);  // periodic Hann of length wl
    w[left + j] = v;
    energy += v * v;
  }
  const double norm = p.normalized ? 1.0 / std::sqrt(energy) : 1.0;
  t->window.resize(N);
  for (int j = 0; j < N; ++j) t->window[j] = static_cast<float>(w[j] * norm);
  // FFT twiddles in the per-pass row layout of fft::rows_offset: for each
  // pass after the first (span P, radix R, the radix rule of
  // fft::next_radix), row k holds exp(-2 pi i j k / (P R)) for j = 1..R-1
  // at stride R - 1 (radix 5: 5).  The rows fill fewer than M entries.
  t->tw_m.assign(M, make_float2(0.f, 0.f));
  {
    size_t off = 0;
    for (int P = 1; P < M;) {
      const int q = M / P;
      // (the in-place sizes open with a radix-16 pass: fft::ip_radix)
      const int R = (P == 1 && in_place_nfft(N) && M % 16 == 0) ? 16
                    : q % 5 == 0                                 ? 5
                    : q % 8 == 0                                 ? 8
                    : q % 4 == 0                                 ? 4
                                                                 : 2;
      if (P > 1) {
        const int stride = R == 5 ? 5 : R - 1;
        for (int k = 0; k < P; ++k) {
          for (int j = 1; j < R; ++j) {
            const double ang = -2.0 * M_PI * static_cast<double>(j) * k / (static_cast<double>(P) * R);
            t->tw_m[off + static_cast<size_t>(k) * stride + j - 1] =
                make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang)));
          }
        }
        off += static_cast<size_t>(P) * stride;
      }
      P *= R;
    }
  }
  t->tw_n.resize(M + 1);
  for (int k = 0; k <= M; ++k) {
    const double ang = -2.0 * M_PI * k / N;
    t->tw_n[k] = make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang)));
  }
  // triangles in Hz between n_mels + 2 points equally spaced in mel
  const double f_max = p.f_max > 0.f ? p.f_max : p.sample_rate / 2.0;
  const double m0 = hz_to_mel(p.f_min, p.mel_scale), m1 = hz_to_mel(f_max, p.mel_scale);
  std::vector<double> edge(p.n_mels + 2);
  for (int i = 0; i < p.n_mels + 2; ++i) edge[i] = mel_to_hz(m0 + (m1 - m0) * i / (p.n_mels + 1), p.mel_scale);
  const double bin_hz = (p.sample_rate / 2.0) / (n_freqs - 1);
  std::vector<std::vector<double>> rows(p.n_mels);
  t->fstart.assign(p.n_mels, 0);
  t->fwidth.assign(p.n_mels, 0);
  for (int m = 0; m < p.n_mels; ++m) {
    const double lo = edge[m], c = edge[m + 1], hi = edge[m + 2];
    const double area = p.slaney_norm ? 2.0 / (hi - lo) : 1.0;
    int first = -1, last = -1;
    std::vector<double> row(n_freqs);
    for (int k = 0; k < n_freqs; ++k) {
      const double f = k * bin_hz;
      const double rise = (f - lo) / (c - lo), fall = (hi - f) / (hi - c);
      row[k] = std::max(0.0, std::min(rise, fall)) * area;
      if (row[k] > 0.0) {
        if (first < 0) first = k;
        last = k;
      }
    }
    if (first >= 0) {
      t->fstart[m] = first;
      t->fwidth[m] = last - first + 1;
      rows[m].assign(row.begin() + first, row.begin() + last + 1);
    }
    t->wmax = std::max(t->wmax, t->fwidth[m]);
  }
  // Rows at a stride of a multiple of 4 taps (zero-padded): the kernel reads
  // four weights at a time from 16-byte aligned rows.
  t->wmax = (std::max(t->wmax, 1) + 3) / 4 * 4;
  t->fw.assign(static_cast<size_t>(p.n_mels) * t->wmax, 0.f);
  for (int m = 0; m < p.n_mels; ++m)
    for (int j = 0; j < t->fwidth[m]; ++j) t->fw[static_cast<size_t>(m) * t->wmax + j] = static_cast<float>(rows[m][j]);
}

// Host-side fault injection for tests: with LOGMEL_FAULT=plan_alloc (or
// plan_alloc:k) the first (k-th, counting from 1) device allocation of a plan
// creation fails as if the device were out of memory, before any CUDA call
// is made for it.  Unset, nothing changes.
bool plan_alloc_fault(int index) {
  const char *v = env_or("LOGMEL_FAULT", "");
  const char *key = "plan_alloc";
  const size_t n = std::strlen(key);
  if (std::strncmp(v, key, n) != 0) return false;
  int k = 1;
  if (v[n] == ':') k = std::atoi(v + n + 1);
  else if (v[n] != '\0') return false;
  return index == k;
}

template <typename T>
lm_status upload(const std::vector<T> &h, T **d, int *n_alloc) {
  *d = nullptr;
  if (h.empty()) return LM_OK;
  if (plan_alloc_fault(++*n_alloc)) return LM_ERR_OUT_OF_MEMORY;
  cudaError_t e = cudaMalloc(reinterpret_cast<void **>(d), h.size() * sizeof(T));
  if (e == cudaErrorMemoryAllocation) {
    (void)cudaGetLastError();
    return LM_ERR_OUT_OF_MEMORY;
  }
  if (e != cudaSuccess) return cuda_fail(e);
  LM_CUDA_TRY(cudaMemcpy(*d, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice));
  return LM_OK;
}

void free_plan(lm_mel_plan *pl) {
  if (!pl) return;
  for (void *ptr : {static_cast<void *>(pl->window), static_cast<void *>(pl->tw_m), static_cast<void *>(pl->tw_n),
                    static_cast<void *>(pl->fstart), static_cast<void *>(pl->fwidth), static_cast<void *>(pl->fw),
                    static_cast<void *>(pl->tables), static_cast<void *>(pl->reg_tables),
                    static_cast<void *>(pl->mel_image)})
    if (ptr) cudaFree(ptr);
  delete pl;
}

lm_status validate(const lm_mel_params &p) {
  if (p.sample_rate <= 0 || p.hop_length <= 0 || p.n_mels <= 0 || p.n_fft <= 0) return LM_ERR_INVALID_ARG;
  if (!(p.f_min >= 0.f) || (p.f_max > 0.f && !(p.f_max > p.f_min))) return LM_ERR_INVALID_ARG;
  if (p.f_max <= 0.f && !(p.sample_rate / 2.0 > p.f_min)) return LM_ERR_INVALID_ARG;
  if (p.win_length < 0 || p.win_length > p.n_fft || p.pad < 0) return LM_ERR_INVALID_ARG;
  if (p.pad_mode < LM_PAD_REFLECT || p.pad_mode > LM_PAD_CIRCULAR) return LM_ERR_INVALID_ARG;
  if (p.mel_scale != LM_MEL_HTK && p.mel_scale != LM_MEL_SLANEY) return LM_ERR_INVALID_ARG;
  if (!supported_nfft(p.n_fft) || p.n_mels > 256) return LM_ERR_UNSUPPORTED;
  if (p.power != 1.f && p.power != 2.f) return LM_ERR_UNSUPPORTED;
  return LM_OK;
}

int64_t frames_for(const lm_mel_params &p, int64_t T) {
  const int64_t Tz = T + 2 * static_cast<int64_t>(p.pad);
  const int64_t len = p.center ? Tz + 2 * (p.n_fft / 2) : Tz;
  if (len < p.n_fft) return 0;
  return 1 + (len - p.n_fft) / p.hop_length;
}

// The register kernels' table image (reg::Tables<NFFT>) for n_fft 400 and
// 1024, in double and rounded to f32: window pairs, each stage-2 lane's
// twiddles exp(-2 pi i b c / M) for its inputs b, each lane's untangle
// twiddles exp(-2 pi i k / N) for its bins k, and the filter rows times
// 2^-power (the kernels form |2X|^power; scaling by a power of two is exact)
// with their supports.
template <int NFFT>
std::vector<unsigned char> reg_image(const lm_mel_params &p, const HostTables &t) {
  using C = reg::Cfg<NFFT>;
  using Tb = reg::Tables<NFFT>;
  std::vector<unsigned char> img(Tb::bytes(p.n_mels, t.wmax), 0);
  auto put2 = [&](size_t off, double re, double im) {
    const float v[2] = {static_cast<float>(re), static_cast<float>(im)};
    std::memcpy(img.data() + off, v, sizeof(v));
  };
  auto root = [&](size_t off, long num, long den) {  // exp(-2 pi i num / den)
    const double ang = -2.0 * M_PI * static_cast<double>(num % den) / static_cast<double>(den);
    put2(off, std::cos(ang), std::sin(ang));
  };
  for (int n = 0; n < C::M; ++n) put2(8 * static_cast<size_t>(n), t.window[2 * n], t.window[2 * n + 1]);
  for (int lane = 0; lane < C::LANES2; ++lane) {
    for (int j = 0; j < C::R2; ++j) {
      long b, c, k;  // stage-2 input row b of the lane's column c; bin k of its j-th output
      if (NFFT != 1024) {  // one lane per column
        c = lane;
        b = j;
        k = lane + static_cast<long>(C::N1) * j;
      } else {
        c = lane >> 1;
        const int h = lane & 1;
        b = 2 * j + h;
        k = c + 16 * j + 256 * h;
      }
      root(Tb::tw2_off() + 8 * (static_cast<size_t>(lane) * C::TWROW + j), b * c, C::M);
      root(Tb::twu_off() + 8 * (static_cast<size_t>(lane) * C::TWROW + j), k, NFFT);
    }
  }
  const float scale = p.power == 1.f ? 0.5f : 0.25f;
  std::vector<float> fw(t.fw);
  for (float &v : fw) v *= scale;
  std::memcpy(img.data() + Tb::fw_off(), fw.data(), fw.size() * sizeof(float));
  for (int m = 0; m < p.n_mels; ++m) {
    const int sw[2] = {t.fstart[m], t.fwidth[m]};
    std::memcpy(img.data() + Tb::fsw_off(p.n_mels, t.wmax) + 8 * static_cast<size_t>(m), sw, sizeof(sw));
  }
  return img;
}

// Frames per tile of the generic kernel (the register kernels' tiles are
// taller, so a workspace sized with this holds the tile keys of either).
int tile_frames(int n_fft) {
  WaveKernel k;
  size_t smem;
  int tf = 1, nt = 0;
  pick_wave_kernel(n_fft, 1, 1, &k, &smem, &tf, &nt);
  return tf;
}

}  // namespace
}  // namespace lm

extern "C" lm_status lm_mel_plan_create(const lm_mel_params *params, lm_mel_plan **plan) {
  if (!params || !plan) return LM_ERR_INVALID_ARG;
  *plan = nullptr;
  if (lm_status st = lm::validate(*params); st != LM_OK) return st;
  lm::HostTables t;
  lm::build_tables(*params, &t);
  auto *pl = new lm_mel_plan{};
  pl->p = *params;
  pl->n_freqs = params->n_fft / 2 + 1;
  pl->wmax = t.wmax;
  // The tables go to the current device, which the plan records.
  int n_alloc = 0;
  lm_status st = lm::upload(t.window, &pl->window, &n_alloc);
  if (st == LM_OK) st = lm::upload(t.tw_m, &pl->tw_m, &n_alloc);
  if (st == LM_OK) st = lm::upload(t.tw_n, &pl->tw_n, &n_alloc);
  if (st == LM_OK) st = lm::upload(t.fstart, &pl->fstart, &n_alloc);
  if (st == LM_OK) st = lm::upload(t.fwidth, &pl->fwidth, &n_alloc);
  if (st == LM_OK) st = lm::upload(t.fw, &pl->fw, &n_alloc);
  if (st == LM_OK && params->n_fft <= 4096) {
    // the shared-memory image the kernel copies in one piece
    pl->tables_bytes = lm::wave_tables_bytes(params->n_fft, params->n_mels, t.wmax);
    std::vector<unsigned char> img(pl->tables_bytes, 0);
    size_t o = 0;
    auto put = [&](const void *src, size_t n) {
      std::memcpy(img.data() + o, src, n);
      o += n;
    };
    put(t.tw_m.data(), t.tw_m.size() * sizeof(float2));
    put(t.tw_n.data(), t.tw_n.size() * sizeof(float2));
    o += sizeof(float2);  // padding: fw starts 16-byte aligned
    put(t.fw.data(), t.fw.size() * sizeof(float));
    put(t.window.data(), t.window.size() * sizeof(float));
    for (int m = 0; m < params->n_mels; ++m) {
      const int sw[2] = {t.fstart[m], t.fwidth[m]};
      put(sw, sizeof(sw));
    }
    st = lm::upload(img, &pl->tables, &n_alloc);
  }
  if (st == LM_OK) {
    std::vector<unsigned char> img;
    switch (params->n_fft) {
      case 64: img = lm::reg_image<64>(*params, t); break;
      case 128: img = lm::reg_image<128>(*params, t); break;
      case 256: img = lm::reg_image<256>(*params, t); break;
      case 400: img = lm::reg_image<400>(*params, t); break;
      case 512: img = lm::reg_image<512>(*params, t); break;
      case 1024: img = lm::reg_image<1024>(*params, t); break;
      default: break;  // the generic kernel only
    }
    if (!img.empty()) {
      pl->reg_tables_bytes = static_cast<uint32_t>(img.size());
      st = lm::upload(img, &pl->reg_tables, &n_alloc);
    }
  }
  if (st == LM_OK && lm::in_place_nfft(params->n_fft)) {
    // the filterbank image the in-place kernel copies into its buffer
    pl->mel_image_bytes = lm::mel_image_bytes_for(params->n_fft, params->n_mels, t.fwidth);
    if (pl->mel_image_bytes > 0) {
      std::vector<unsigned char> img(pl->mel_image_bytes, 0);
      const size_t w0 = 8 * (static_cast<size_t>(params->n_mels) + 1);
      int off = 0;
      for (int m = 0; m <= params->n_mels; ++m) {
        const int h[2] = {m < params->n_mels ? t.fstart[m] : 0, off};
        std::memcpy(img.data() + 8 * static_cast<size_t>(m), h, sizeof(h));
        if (m == params->n_mels) break;
        std::memcpy(img.data() + w0 + 4 * static_cast<size_t>(off), t.fw.data() + static_cast<size_t>(m) * t.wmax,
                    4 * static_cast<size_t>(t.fwidth[m]));
        off += t.fwidth[m];
      }
      st = lm::upload(img, &pl->mel_image, &n_alloc);
    }
  }
  if (st == LM_OK) {
    if (cudaError_t e = cudaGetDevice(&pl->device); e != cudaSuccess) st = lm::cuda_fail(e);
  }
  if (st != LM_OK) {
    lm::free_plan(pl);
    return st;
  }
  *plan = pl;
  return LM_OK;
}

extern "C" lm_status lm_mel_plan_destroy(lm_mel_plan *plan) {
  if (!plan) return LM_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(plan->device);
  cudaDeviceSynchronize();
  lm::free_plan(plan);
  cudaSetDevice(prev);
  return LM_OK;
}

extern "C" lm_status lm_mel_n_frames(const lm_mel_plan *plan, int64_t T, int64_t *n_frames) {
  if (!plan || !n_frames || T < 0) return LM_ERR_INVALID_ARG;
  *n_frames = lm::frames_for(plan->p, T);
  return LM_OK;
}

extern "C" lm_status lm_mel_workspace_size(const lm_mel_plan *plan, int64_t B, int64_t T, size_t *bytes) {
  if (!plan || !bytes || B < 0 || T < 0) return LM_ERR_INVALID_ARG;
  const int64_t nfr = lm::frames_for(plan->p, T);
  const int tf = lm::tile_frames(plan->p.n_fft);
  const int64_t tpc = nfr > 0 ? (nfr + tf - 1) / tf : 0;
  // header | tile keys [B * tpc] | (log plans) clip keys [B] | clip counters [B] | rescale counter
  const size_t clip_arrays = plan->p.log_mel ? (2 * static_cast<size_t>(B) + 1) * sizeof(uint32_t) : 0;
  *bytes = (lm::kWorkspaceHeaderBytes + static_cast<size_t>(B * tpc) * sizeof(uint32_t) + clip_arrays + 255) / 256 *
           256;
  return LM_OK;
}

lm_status lm::mel_plan_n_mels(const lm_mel_plan *plan, int32_t *n_mels) {
  if (!plan || !n_mels) return LM_ERR_INVALID_ARG;
  *n_mels = plan->p.n_mels;
  return LM_OK;
}

lm_status lm::mel_spectrogram_check(const lm_mel_plan *plan, int32_t in_dtype, int64_t B, int64_t T,
                                    int32_t out_dtype) {
  if (!plan || B < 0 || T < 0) return LM_ERR_INVALID_ARG;
  if (in_dtype != LM_F32 && in_dtype != LM_I16) return LM_ERR_UNSUPPORTED;
  if (out_dtype != LM_F32 && out_dtype != LM_F16) return LM_ERR_UNSUPPORTED;
  if (plan->p.log_mel && out_dtype != LM_F32) return LM_ERR_UNSUPPORTED;
  const lm_mel_params &p = plan->p;
  const int64_t nfr = lm::frames_for(p, T);
  if (B == 0) return LM_OK;
  if (T < 1 || nfr < 1) return LM_ERR_INVALID_ARG;
  if (p.center && p.pad_mode == LM_PAD_REFLECT && T + 2 * static_cast<int64_t>(p.pad) <= p.n_fft / 2)
    return LM_ERR_INVALID_ARG;
  return LM_OK;
}

lm_status lm::mel_spectrogram_run(const lm_mel_plan *plan, const void *wave, int32_t in_dtype, int64_t B,
                                  int64_t T, void *out, int32_t out_dtype, void *workspace,
                                  size_t workspace_bytes, cudaStream_t stream, uint32_t *err_word) {
  if (lm_status st = mel_spectrogram_check(plan, in_dtype, B, T, out_dtype); st != LM_OK) return st;
  if (B == 0) return LM_OK;
  const lm_mel_params &p = plan->p;
  const int64_t nfr = lm::frames_for(p, T);
  if (!wave || !out || !workspace) return workspace ? LM_ERR_INVALID_ARG : LM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(wave) & 3) || (reinterpret_cast<uintptr_t>(out) & 3) ||
      (reinterpret_cast<uintptr_t>(workspace) & 3))
    return LM_ERR_MISALIGNED;
  size_t need = 0;
  lm_mel_workspace_size(plan, B, T, &need);
  if (workspace_bytes < need) return LM_ERR_WORKSPACE;
  int dev = 0;
  LM_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != plan->device) return LM_ERR_INVALID_ARG;

  lm::WaveKernel kern;
  size_t smem = 0;
  int tf = 1;
  int nt = 0;
  const int esize = in_dtype == LM_I16 ? 2 : 4;
  lm::DeviceInfo di;
  if (lm_status st = lm::current_device_info(&di); st != LM_OK) return st;
  // n_fft 64, 128, 256, 400, 512 and 1024 run the register kernels (wave_reg.cuh) unless
  // LOGMEL_K3=stockham selects the generic shared-memory kernel (for A/B).
  // (The register kernels index samples of a clip with 32 bits at its edges.)
  bool use_reg = plan->reg_tables != nullptr && T < (int64_t{1} << 31) - 2 * (p.n_fft + p.pad) &&
                 std::strcmp(lm::env_or("LOGMEL_K3", "auto"), "stockham") != 0;
  if (use_reg) {
    switch (p.n_fft) {
      case 64: lm::reg_entry<64>(&kern, &smem, &tf, &nt, p.n_mels, plan->wmax); break;
      case 128: lm::reg_entry<128>(&kern, &smem, &tf, &nt, p.n_mels, plan->wmax); break;
      case 256: lm::reg_entry<256>(&kern, &smem, &tf, &nt, p.n_mels, plan->wmax); break;
      case 400: lm::reg_entry<400>(&kern, &smem, &tf, &nt, p.n_mels, plan->wmax); break;
      case 512: lm::reg_entry<512>(&kern, &smem, &tf, &nt, p.n_mels, plan->wmax); break;
      default: lm::reg_entry<1024>(&kern, &smem, &tf, &nt, p.n_mels, plan->wmax); break;
    }
    use_reg = smem <= static_cast<size_t>(di.max_smem_optin);
  }
  bool use_seg = false;
  size_t seg_offset = 0, seg_used = 0;
  if (!use_reg) {
    lm::pick_wave_kernel(p.n_fft, p.n_mels, plan->wmax, &kern, &smem, &tf, &nt);
    // Two buffers for the contiguous samples of one tile of frames (plus 32
    // bytes of alignment slack), then two mbarriers.
    const size_t seg_bytes =
        (static_cast<size_t>((tf - 1) * static_cast<int64_t>(p.hop_length) + p.n_fft) * esize + 32 + 127) / 128 * 128;
    seg_offset = smem;
    use_seg = !lm::in_place_nfft(p.n_fft) && (reinterpret_cast<uintptr_t>(wave) & 15) == 0 &&
              seg_offset + 2 * seg_bytes + 32 <= static_cast<size_t>(di.max_smem_optin);
    // Without staging (unaligned input, or a hop so long the spans do not fit)
    // every tile gathers its samples from global memory; the two mbarriers are
    // still reserved, right after the tables, since every CTA initialises them.
    seg_used = use_seg ? seg_bytes : 0;
    smem = seg_offset + 2 * seg_used + 32;  // three mbarriers
  }
  if (smem > static_cast<size_t>(di.max_smem_optin)) return LM_ERR_UNSUPPORTED;
  if (lm_status st = lm::ensure_smem_attribute(reinterpret_cast<const void *>(kern), static_cast<int>(smem));
      st != LM_OK)
    return st;
  int per_sm = 0;
  LM_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nt, smem));
  if (per_sm < 1) return LM_ERR_UNSUPPORTED;

  lm::WaveArgs a{};
  a.wave = wave;
  a.out = out;
  a.tile_key = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + lm::kWorkspaceHeaderBytes);
  a.B = B;
  a.T = T;
  a.n_frames = nfr;
  a.in_i16 = in_dtype == LM_I16;
  a.out_f16 = out_dtype == LM_F16;
  a.log_mel = p.log_mel != 0;
  a.power_is_one = p.power == 1.f;
  a.hop = p.hop_length;
  a.pad_left = (p.center ? p.n_fft / 2 : 0) + p.pad;
  a.pad_zero = p.pad;
  a.pad_mode = p.pad_mode;
  a.n_mels = p.n_mels;
  a.wmax = plan->wmax;
  a.TF = tf;
  a.tiles_per_clip = static_cast<int32_t>((nfr + tf - 1) / tf);
  a.window = plan->window;
  a.tw_m = plan->tw_m;
  a.tw_n = plan->tw_n;
  a.fstart = plan->fstart;
  a.fwidth = plan->fwidth;
  a.fw = plan->fw;
  a.tables = use_reg ? plan->reg_tables : plan->tables;
  a.tables_bytes = use_reg ? plan->reg_tables_bytes : plan->tables_bytes;
  a.mel_image = plan->mel_image;
  a.mel_image_bytes = plan->mel_image_bytes;
  a.err = err_word ? err_word : static_cast<uint32_t *>(workspace);
  a.next_tile = static_cast<uint32_t *>(workspace) + 1;
  a.total_bytes = static_cast<uint64_t>(B) * static_cast<uint64_t>(T) * esize;
  a.seg_offset = static_cast<uint32_t>(seg_offset);
  a.seg_bytes = static_cast<uint32_t>(seg_used);
  a.use_seg = use_seg;
  const int64_t n_tiles = B * a.tiles_per_clip;
  if (n_tiles > INT32_MAX / 2) return LM_ERR_UNSUPPORTED;  // tile indices and the counter are 32-bit
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(n_tiles, static_cast<int64_t>(di.sm_count) * per_sm));
  // Log plans finish with the clamp kernel, launched as a programmatic
  // dependent so that its launch overlaps the main kernel's tail.  With
  // LOGMEL_K3_EPILOGUE=fused the register kernels apply the clip floor and
  // rescale in the same launch instead (one cooperative grid; its CTAs wait
  // for each other's clip maxima).  Both give the same bits; the two
  // launches measured faster at every batch tried (n_fft 400, 30 s clips, L2
  // flushed: 8 clips 34.1 against 34.4 us, 32: 93.5 / 96.7, 128: 352.8 /
  // 370.8, 442: 1189 / 1261): the fused epilogue rescales only after every
  // tile has been claimed, so it re-reads as much as the clamp kernel and
  // adds its polling.
  {
    const int64_t tpc_ws = (nfr + lm::tile_frames(p.n_fft) - 1) / lm::tile_frames(p.n_fft);  // the workspace layout's
    a.clip_key = a.tile_key + B * tpc_ws;
    a.clip_done = a.clip_key + B;
    a.rescale_next = a.clip_done + B;
    a.fused = use_reg && a.log_mel && std::strcmp(lm::env_or("LOGMEL_K3_EPILOGUE", "separate"), "fused") == 0;
  }
  cudaStream_t s = stream;
  // The device error word, the tile counter and the fused epilogue's clip
  // keys and counters start at zero (tile slots are each written before they
  // are read).  With a launch token CTA 0 clears them; without one (stream
  // capture, or a workspace that is not 8-byte aligned) a memset does.
  a.clear_err = err_word == nullptr;
  a.ready = reinterpret_cast<uint64_t *>(static_cast<char *>(workspace) + 8);
  a.token = (reinterpret_cast<uintptr_t>(workspace) & 7) == 0 ? lm::call_token(s) : 0;
  if (a.token == 0)
    LM_CUDA_TRY(cudaMemsetAsync(workspace, 0, a.log_mel ? need : lm::kWorkspaceHeaderBytes, s));
  if (a.fused) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(static_cast<unsigned>(nt));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    LM_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, a));
    return LM_OK;
  }
  kern<<<grid, static_cast<unsigned>(nt), smem, s>>>(a);
  LM_CUDA_TRY(cudaGetLastError());
  if (a.log_mel) {
    if (lm_status st = lm::launch_clip_clamp(static_cast<float *>(out), a.tile_key, B, p.n_mels * nfr,
                                             a.tiles_per_clip, s);
        st != LM_OK)
      return st;
  }
  return LM_OK;
}

extern "C" lm_status lm_mel_spectrogram(const lm_mel_plan *plan, const void *wave, int32_t in_dtype, int64_t B,
                                        int64_t T, void *out, int32_t out_dtype, void *workspace,
                                        size_t workspace_bytes, lm_stream_t stream) {
  return lm::mel_spectrogram_run(plan, wave, in_dtype, B, T, out, out_dtype, workspace, workspace_bytes,
                                 reinterpret_cast<cudaStream_t>(stream), nullptr);
}
