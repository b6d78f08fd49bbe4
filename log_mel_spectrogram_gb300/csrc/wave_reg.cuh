// wave_reg.cuh -- waveform -> mel kernels for n_fft 64, 128, 256, 400, 512 and
// 1024 whose transforms run mostly in registers (included by wave_mel.cu,
// inside its namespace, after WaveArgs and map_index).
//
// The real FFT of a frame is the N/2 = M point complex FFT of its folded
// samples z[n] = x[2n] + i x[2n+1] followed by the real-input untangle
// ("flashmel" page, "How it works": the folded R2C for powers of two; here it
// is used for 400 points too).  M = N1 * N2 is split Cooley-Tukey style,
// input n = N2 a + b, output k = c + N1 d:
//
//   stage 1  thread b (N2 per frame) loads the points b, b + N2, ... straight
//            from the waveform -- framing, centre padding and the window folded
//            into the loads -- runs the N1-point DFT over a in registers and
//            writes row b of the frame's shared-memory region;
//   stage 2  the lane of column c multiplies column c by exp(-2 pi i b c / M)
//            and runs the N2-point DFT over b in registers, which gives bins
//            c + N1 d.  Bin k pairs with bin M - k in the real-input untangle,
//            and the lane that holds M - k is in the same warp.  With
//            A = Z[k], B = Z[M - k], S = A + conj B and
//            T = exp(-2 pi i k / N) (-i) (A - conj B), 2 X[k] = S + T and
//            2 conj X[M - k] = S - T: each of the two lanes forms both bins
//            of half of their common pairs, fetching half of the partner's
//            values by shuffle.  The factor 2 is folded into the filter
//            weights (scaled by 2^-power, exactly).
//
// Sizes:
//   n_fft 64, 128, 256, 400, 512: M = 32 = 8 x 4, 64 = 8 x 8, 128 = 16 x 8,
//     200 = 25 x 8, 256 = 16 x 16.  Stage 1: N2 threads per frame, each an
//     N1-point DFT; stage 2: one lane per column, each an N2-point DFT; 32
//     frames per tile, four per warp.
//   n_fft 1024: M = 512 = 16 x 32.  Stage 1: 32 threads per frame, a 16-point
//     DFT each.  Stage 2: the 32-point DFT of column c is shared by lanes 2c
//     and 2c + 1: each transforms one parity of b (16 points), the two swap
//     results with one shuffle per value, and lane 2c + h keeps the outputs
//     d = d' + 16 h, X = V0[d'] + (-1)^h exp(-2 pi i d' / 32) V1[d'].
//
// A frame stays inside one warp from its samples to its power row, so the
// stages synchronise with __syncwarp; the CTA synchronises twice per tile of
// TF frames (power rows complete; mel projection done with the region).  The
// mel projection runs lanes over the frames of a band, so each band's output
// row is stored as one run of consecutive frames.
//
// Log plans finish in the same launch (the KBench spec's per-clip floor and
// rescale, its "clip-resident" design note): each tile folds its maximum log
// value into its clip's key and then counts itself into the clip's counter
// with release order.  A CTA that finds no tile left to compute takes tiles
// to floor and rescale from a second counter, in tile (so clip) order, waits
// (bounded) for each one's clip counter to complete and rescales the tile in
// place while it is still in L2 -- so CTAs that run out of work early
// rescale the early clips while the others still compute the late ones.
// The grid is cooperative and no CTA waits before every tile has been
// claimed for computing, so every wait ends.
#pragma once

namespace reg {

using fft::cadd;
using fft::cmul;
using fft::csub;

// cos(2 pi r / N) for r in the first quadrant of N = 16 and N = 32, and cos
// and sin(2 pi m / 25): the roots of unity rounded to f32.  Called with
// arguments that are constants after unrolling, so every value folds into an
// immediate operand.
__device__ __forceinline__ float cos16(int r) {
  switch (r) {
    case 0: return 1.0f;
    case 1: return 0.923879533f;
    case 2: return 0.707106781f;
    default: return 0.382683432f;
  }
}
__device__ __forceinline__ float cos32(int r) {
  switch (r) {
    case 0: return 1.0f;
    case 1: return 0.98078528f;
    case 2: return 0.923879533f;
    case 3: return 0.831469612f;
    case 4: return 0.707106781f;
    case 5: return 0.555570233f;
    case 6: return 0.382683432f;
    default: return 0.195090322f;
  }
}
__device__ __forceinline__ float cos25(int m) {
  switch (m) {  // cos(2 pi m / 25) = cos(2 pi (25 - m) / 25)
    case 0: return 1.0f;
    case 1: case 24: return 0.968583161f;
    case 2: case 23: return 0.87630668f;
    case 3: case 22: return 0.728968627f;
    case 4: case 21: return 0.535826795f;
    case 5: case 20: return 0.309016994f;
    case 6: case 19: return 0.0627905195f;
    case 7: case 18: return -0.187381315f;
    case 8: case 17: return -0.425779292f;
    case 9: case 16: return -0.63742399f;
    case 10: case 15: return -0.809016994f;
    case 11: case 14: return -0.929776486f;
    default: return -0.992114701f;  // 12, 13
  }
}
__device__ __forceinline__ float sin25(int m) {
  const float sgn = m > 12 ? -1.0f : 1.0f;  // sin(2 pi m / 25) = -sin(2 pi (25 - m) / 25)
  switch (m > 12 ? 25 - m : m) {
    case 0: return 0.0f;
    case 1: return sgn * 0.248689887f;
    case 2: return sgn * 0.481753674f;
    case 3: return sgn * 0.684547106f;
    case 4: return sgn * 0.844327926f;
    case 5: return sgn * 0.951056516f;
    case 6: return sgn * 0.998026728f;
    case 7: return sgn * 0.982287251f;
    case 8: return sgn * 0.904827052f;
    case 9: return sgn * 0.770513243f;
    case 10: return sgn * 0.587785252f;
    case 11: return sgn * 0.368124553f;
    default: return sgn * 0.125333234f;  // 12
  }
}

// cos and sin of 2 pi m / N for N = 16 or 32 from the first quadrant.
template <int N>
__device__ __forceinline__ float2 cs_pow2(int m) {
  constexpr int Q = N / 4;
  m &= N - 1;
  const int q = m / Q, r = m % Q;
  // sin(2 pi r / N) = cos(2 pi (Q - r) / N)
  const float cr = N == 16 ? cos16(r) : cos32(r);
  const float sr = r == 0 ? 0.0f : (N == 16 ? cos16(Q - r) : cos32(Q - r));
  switch (q) {
    case 0: return make_float2(cr, sr);
    case 1: return make_float2(-sr, cr);
    case 2: return make_float2(-cr, -sr);
    default: return make_float2(sr, -cr);
  }
}

// z * exp(-2 pi i m / N), m a compile-time constant after unrolling; the
// quarter turns are exact.
template <int N>
__device__ __forceinline__ float2 rot(float2 z, int m) {
  m %= N;
  if (m == 0) return z;
  if (4 * m == N) return make_float2(z.y, -z.x);        // -i
  if (2 * m == N) return make_float2(-z.x, -z.y);       // -1
  if (4 * m == 3 * N) return make_float2(-z.y, z.x);    // +i
  float2 w;
  if constexpr (N == 25) {
    w = make_float2(cos25(m), -sin25(m));
  } else {
    const float2 cs = cs_pow2<N>(m);
    w = make_float2(cs.x, -cs.y);
  }
  return cmul(z, w);
}

template <int R>
struct Dft;
template <>
struct Dft<4> {
  __device__ __forceinline__ static void run(float2 (&u)[4]) { fft::Dft<4>::run(u); }
};
template <>
struct Dft<5> {
  __device__ __forceinline__ static void run(float2 (&u)[5]) { fft::Dft<5>::run(u); }
};
template <>
struct Dft<8> {
  __device__ __forceinline__ static void run(float2 (&u)[8]) { fft::Dft<8>::run(u); }
};

// In-place N1*N2-point DFT, natural order in and out: input n = N2 a + b,
// output k = c + N1 d; N2 DFTs of size N1, the twiddles exp(-2 pi i b c / N),
// N1 DFTs of size N2.  Every index is a compile-time constant.
template <int N1, int N2>
__device__ __forceinline__ void dft_ct(float2 (&u)[N1 * N2]) {
  constexpr int N = N1 * N2;
#pragma unroll
  for (int b = 0; b < N2; ++b) {
    float2 t[N1];
#pragma unroll
    for (int a = 0; a < N1; ++a) t[a] = u[N2 * a + b];
    Dft<N1>::run(t);
#pragma unroll
    for (int c = 0; c < N1; ++c) u[N2 * c + b] = rot<N>(t[c], b * c);
  }
  float2 out[N];
#pragma unroll
  for (int c = 0; c < N1; ++c) {
    float2 t[N2];
#pragma unroll
    for (int b = 0; b < N2; ++b) t[b] = u[N2 * c + b];
    Dft<N2>::run(t);
#pragma unroll
    for (int d = 0; d < N2; ++d) out[c + N1 * d] = t[d];
  }
#pragma unroll
  for (int k = 0; k < N; ++k) u[k] = out[k];
}

template <>
struct Dft<16> {
  __device__ __forceinline__ static void run(float2 (&u)[16]) { dft_ct<4, 4>(u); }
};
template <>
struct Dft<32> {
  __device__ __forceinline__ static void run(float2 (&u)[32]) { dft_ct<4, 8>(u); }
};
template <>
struct Dft<25> {
  __device__ __forceinline__ static void run(float2 (&u)[25]) { dft_ct<5, 5>(u); }
};

template <int NFFT>
struct Cfg;

// The sizes whose stage 2 gives each column one lane: M = N1 x N2, stage 1
// with N2 threads per frame (an N1-point DFT each), stage 2 with N1 lanes per
// frame (an N2-point DFT each), tiles of TF frames (a multiple of 32), TF / 8
// frames per warp.  Rows of stage-1 output hold N1 values at a stride of ROW
// (odd where that spreads a column over the banks).
template <int NFFT_, int N1_, int N2_, int ROW_, int MINB_, int TF_ = 32>
struct ColCfg {
  static constexpr int M = NFFT_ / 2;
  static constexpr int N1 = N1_;     // stage-1 DFT size; stage-2 lanes per frame
  static constexpr int N2 = N2_;     // stage-1 threads per frame; stage-2 DFT size
  static constexpr int ROW = ROW_;   // complex values per stage-1 row (N1 used)
  static constexpr int TF = TF_;     // frames per tile
  static constexpr int NT = 256;
  static constexpr int FPW = TF / (NT / 32);  // frames per warp
  static constexpr int REGION = 2 * N2 * ROW;  // floats per frame region
  static constexpr int LANES2 = N1;  // table rows: one per column
  static constexpr int R2 = N2;      // twiddles per column
  static constexpr int TWROW = N2 + 2;  // float2 per table row: an odd number of 16-byte units
  static constexpr int kMinBlocks = MINB_;
  // A power row (M + 1 floats at an offset of up to 15) and the mel
  // projection's reads up to 3 floats past it stay inside the frame's region.
  static_assert(M == N1 * N2 && N1 <= 32 && 15 + M + 1 + 3 <= REGION && TF % 32 == 0, "column layout");
};
// 64-frame tiles at 64 and 128 points: stage 1's N2 threads per frame then
// fill whole warps, and the per-tile work spreads over twice the frames (32
// clips x 160000 samples, hop n_fft / 4, 128 bands: 64 points 96.3 -> 84.0
// us, 128 points 57.3 -> 51.2; 128-frame tiles at 64 points 91.1, 64-frame
// tiles at 256 points 49.2 against 45.1, with two CTAs per SM).
template <>
struct Cfg<64> : ColCfg<64, 8, 4, 9, 4, 64> {};
template <>
struct Cfg<128> : ColCfg<128, 8, 8, 9, 4, 64> {};
template <>
struct Cfg<256> : ColCfg<256, 16, 8, 17, 4> {};
template <>
struct Cfg<400> : ColCfg<400, 25, 8, 25, 3> {};  // rows of 25 already spread a column over the banks
template <>
struct Cfg<512> : ColCfg<512, 16, 16, 17, 2> {};

// n_fft 1024: stage 2's 32-point column DFTs are shared by lane pairs.
template <>
struct Cfg<1024> {
  static constexpr int M = 512;
  static constexpr int N1 = 16;
  static constexpr int N2 = 32;
  static constexpr int ROW = 17;     // 16 values per row, padded: rows of one column fall in distinct banks
  static constexpr int TF = 16;
  static constexpr int NT = 256;
  static constexpr int FPW = TF / (NT / 32);  // 2
  static constexpr int REGION = 2 * N2 * ROW;  // 1088 floats
  static constexpr int TWROW = 18;   // float2 per lane row (16 used)
  static constexpr int LANES2 = 32;
  static constexpr int R2 = 16;
  static constexpr int kMinBlocks = 2;
};

// Table image (float2 units unless noted), one bulk copy per CTA:
//   win2 [M]             (w[2n], w[2n+1]) per point n
//   tw2  [LANES2][TWROW] stage-2 twiddles exp(-2 pi i b c / M) of each lane
//   twu  [LANES2][TWROW] untangle twiddles exp(-2 pi i k / N) of each lane's bins
//   fw   [n_mels][wmax]  f32 filter rows times 2^-power (wmax a multiple of 4)
//   fsw  [n_mels]        int2 {first bin, width}
template <int NFFT>
struct Tables {
  using C = Cfg<NFFT>;
  __host__ __device__ static constexpr size_t tw2_off() { return 8 * static_cast<size_t>(C::M); }
  __host__ __device__ static constexpr size_t twu_off() { return tw2_off() + 8 * C::LANES2 * C::TWROW; }
  __host__ __device__ static constexpr size_t fw_off() { return twu_off() + 8 * C::LANES2 * C::TWROW; }
  __host__ __device__ static size_t fsw_off(int n_mels, int wmax) {
    return fw_off() + 4 * static_cast<size_t>(n_mels) * wmax;
  }
  __host__ __device__ static size_t bytes(int n_mels, int wmax) {
    return (fsw_off(n_mels, wmax) + 8 * static_cast<size_t>(n_mels) + 15) / 16 * 16;
  }
};

// Shared memory: TF frame regions | table image | 16 bytes (tile key, abort
// flag, next tile, next tile to rescale) | one mbarrier, the clip floor and
// 4 spare bytes.
template <int NFFT>
size_t smem_bytes(int n_mels, int wmax) {
  using C = Cfg<NFFT>;
  return 4 * static_cast<size_t>(C::TF) * C::REGION + Tables<NFFT>::bytes(n_mels, wmax) + 16 + 16;
}

// (max(ls, floor) + 4) / 4 for floor = hi - 8; fma(x, 1/4, 1) rounds exactly
// like (x + 4) / 4.
__device__ __forceinline__ float rescale_log(float ls, float floor_v) { return fmaf(fmaxf(ls, floor_v), 0.25f, 1.0f); }

// For a frame that touches the signal's edge: the index in the clip of each
// sample s0 + 2 (stride i + lane_off) + e (i < k, e < 2) after the padding
// rule, or -1 for a padding zero, written to idx[2 i + e].  One call per
// frame, out of line (edge frames are two or three per clip); it touches no
// global memory, so the caller's loads of the frame then go out together.
// All indices fit 32 bits: the host sends clips of 2^31 samples or more to
// the generic kernel.
static __device__ __noinline__ void edge_indices(const WaveArgs &a, int s0, int lane_off, int stride, int k,
                                                 int *idx) {
  const int T = static_cast<int>(a.T), pz = a.pad_zero, mode = a.pad_mode;
  // Centre padding applies to the signal already extended by pad_zero zeros
  // on both sides (length T + 2 pad_zero); map there, then back.
  const int Tz = T + 2 * pz;
  for (int j = 0; j < 2 * k; ++j) {
    const int sz = s0 + 2 * (stride * (j >> 1) + lane_off) + (j & 1) + pz;
    int m = sz;
    bool zero = false;
    if (sz < 0 || sz >= Tz) {
      switch (mode) {
        case LM_PAD_CONSTANT: zero = true; break;
        case LM_PAD_REPLICATE: m = sz < 0 ? 0 : Tz - 1; break;
        case LM_PAD_CIRCULAR: m = sz % Tz; m = m < 0 ? m + Tz : m; break;
        default: m = sz < 0 ? -sz : 2 * (Tz - 1) - sz;  // reflect, edge not repeated
      }
    }
    const int i = m - pz;
    idx[j] = (zero || i < 0 || i >= T) ? -1 : i;
  }
}

// The K folded points n = STRIDE i + lane_off (i < K) of one frame, windowed:
// u[i] = (x[2n] w[2n], x[2n+1] w[2n+1]).  s0 is the frame's first sample
// (t hop - pad_left).  One branch per frame picks the load form: interior
// frames read sample pairs directly (8-byte f32 or 4-byte int16 pairs where
// the pair is aligned), edge frames map each sample.  `scratch` is this
// thread's row of at least K float2 in shared memory.
template <int K, int STRIDE>
__device__ __forceinline__ void load_frame(const WaveArgs &a, int64_t b, int64_t s0, int lane_off, bool wave_aligned,
                                           const float2 *win2, float2 *scratch, float2 (&u)[K]) {
  constexpr float kI16 = 1.0f / 32768.0f;
  if (!LM_IN_BOUNDS(b, a.B, a.err)) {  // (checked builds) the clip exists
#pragma unroll
    for (int i = 0; i < K; ++i) u[i] = make_float2(0.f, 0.f);
    return;
  }
  const bool interior = s0 >= 0 && s0 + 2 * (STRIDE * (K - 1) + lane_off) + 1 < a.T;
  const bool paired = wave_aligned && (((b * a.T + s0) & 1) == 0);
  if (interior && a.in_i16) {
    const int16_t *w = static_cast<const int16_t *>(a.wave) + b * a.T + s0 + 2 * lane_off;
    if (paired) {
      const int *w2 = reinterpret_cast<const int *>(w);
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int v = __ldg(w2 + STRIDE * i);
        u[i] = make_float2(static_cast<float>(static_cast<int16_t>(v & 0xffff)) * kI16,
                           static_cast<float>(static_cast<int16_t>(v >> 16)) * kI16);
      }
    } else {
#pragma unroll
      for (int i = 0; i < K; ++i)
        u[i] = make_float2(static_cast<float>(__ldg(w + 2 * STRIDE * i)) * kI16,
                           static_cast<float>(__ldg(w + 2 * STRIDE * i + 1)) * kI16);
    }
  } else if (interior) {
    const float *w = static_cast<const float *>(a.wave) + b * a.T + s0 + 2 * lane_off;
    if (paired) {
      const float2 *w2 = reinterpret_cast<const float2 *>(w);
#pragma unroll
      for (int i = 0; i < K; ++i) u[i] = __ldg(w2 + STRIDE * i);
    } else {
#pragma unroll
      for (int i = 0; i < K; ++i) u[i] = make_float2(__ldg(w + 2 * STRIDE * i), __ldg(w + 2 * STRIDE * i + 1));
    }
  } else if (a.pad_mode == LM_PAD_REFLECT && a.pad_zero == 0) {
    // Reflect padding (the common case): an index folds once, without
    // branches (T > n_fft / 2, so one reflection is enough), and every load
    // is in flight at once.
    const int T = static_cast<int>(a.T);
    const int base0 = static_cast<int>(s0) + 2 * lane_off;
    auto fold = [T](int j) {
      j = j < 0 ? -j : j;
      return j >= T ? 2 * (T - 1) - j : j;
    };
    if (a.in_i16) {
      const int16_t *w = static_cast<const int16_t *>(a.wave) + b * a.T;
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int j0 = fold(base0 + 2 * STRIDE * i), j1 = fold(base0 + 2 * STRIDE * i + 1);
        u[i] = make_float2(LM_IN_BOUNDS(j0, T, a.err) ? static_cast<float>(__ldg(w + j0)) * kI16 : 0.f,
                           LM_IN_BOUNDS(j1, T, a.err) ? static_cast<float>(__ldg(w + j1)) * kI16 : 0.f);
      }
    } else {
      const float *w = static_cast<const float *>(a.wave) + b * a.T;
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int j0 = fold(base0 + 2 * STRIDE * i), j1 = fold(base0 + 2 * STRIDE * i + 1);
        u[i] = make_float2(LM_IN_BOUNDS(j0, T, a.err) ? __ldg(w + j0) : 0.f,
                           LM_IN_BOUNDS(j1, T, a.err) ? __ldg(w + j1) : 0.f);
      }
    }
  } else {
    // Other padding: indices first, into this lane's own stage-1 row (free
    // until the DFT result overwrites it), then a gather without branches --
    // a clamped index and a select -- so that every load is in flight at once.
    int *idx = reinterpret_cast<int *>(scratch);
    edge_indices(a, static_cast<int>(s0), lane_off, STRIDE, K, idx);
    if (a.in_i16) {
      const int16_t *w = static_cast<const int16_t *>(a.wave) + b * a.T;
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int j0 = idx[2 * i], j1 = idx[2 * i + 1];
        const int k0 = j0 < 0 ? 0 : j0, k1 = j1 < 0 ? 0 : j1;
        const float x0 = LM_IN_BOUNDS(k0, a.T, a.err) ? static_cast<float>(__ldg(w + k0)) * kI16 : 0.f;
        const float x1 = LM_IN_BOUNDS(k1, a.T, a.err) ? static_cast<float>(__ldg(w + k1)) * kI16 : 0.f;
        u[i] = make_float2(j0 < 0 ? 0.f : x0, j1 < 0 ? 0.f : x1);
      }
    } else {
      const float *w = static_cast<const float *>(a.wave) + b * a.T;
#pragma unroll
      for (int i = 0; i < K; ++i) {
        const int j0 = idx[2 * i], j1 = idx[2 * i + 1];
        const int k0 = j0 < 0 ? 0 : j0, k1 = j1 < 0 ? 0 : j1;
        const float x0 = LM_IN_BOUNDS(k0, a.T, a.err) ? __ldg(w + k0) : 0.f;
        const float x1 = LM_IN_BOUNDS(k1, a.T, a.err) ? __ldg(w + k1) : 0.f;
        u[i] = make_float2(j0 < 0 ? 0.f : x0, j1 < 0 ? 0.f : x1);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const float2 wv = win2[STRIDE * i + lane_off];
    u[i] = make_float2(u[i].x * wv.x, u[i].y * wv.y);
  }
}

// Both bins of the untangle pair (k, M - k) from A = Z[k], B = Z[M - k] and
// tw = exp(-2 pi i k / N): 2 X[k] = S + T and 2 conj X[M - k] = S - T, with
// S = A + conj B and T = tw (-i) (A - conj B).  Returns |2 X[k]|^power in *pk
// and |2 X[M - k]|^power in *pm.
__device__ __forceinline__ void untangle_pair(float2 A, float2 B, float2 tw, bool power_one, float *pk, float *pm) {
  const float2 S = make_float2(A.x + B.x, A.y - B.y);
  const float2 D = make_float2(A.x - B.x, A.y + B.y);
  const float2 T = make_float2(fmaf(tw.x, D.y, tw.y * D.x), fmaf(tw.y, D.y, -tw.x * D.x));
  const float2 P = make_float2(S.x + T.x, S.y + T.y);
  const float2 Q = make_float2(S.x - T.x, S.y - T.y);
  float p = fmaf(P.x, P.x, P.y * P.y);
  float q = fmaf(Q.x, Q.x, Q.y * Q.y);
  if (power_one) {
    p = sqrtf(p);
    q = sqrtf(q);
  }
  *pk = p;
  *pm = q;
}

// Stage 2 of the one-lane-per-column sizes for the frames f0 .. of one
// iteration (32 / N1 frames, N1 lanes each): lane c transforms column c and
// holds bins c + N1 d.  The untangle pair of bin k = c + N1 d is bin
// M - k = (N1 - c) + N1 (N2 - 1 - d), the value N2 - 1 - d of the lane of
// column N1 - c; lane c forms both bins of its pairs d < N2 / 2 (the partner
// forms the others), so it fetches only the partner's values N2 - 1 ..
// N2 / 2.  Column 0 pairs with itself (d with N2 - d; d = 0 gives bins 0 and
// M, and bin M / 2 stands alone), and for even N1 so does column N1 / 2
// (d with N2 - 1 - d).  Lanes without a column (N1 = 25) run column 0 of the
// first frame and discard it.
template <int NFFT>
__device__ __forceinline__ void stage2_cols(float *regions, int f0, int nf, int lane, const float2 *tw2,
                                            const float2 *twu, bool power_one) {
  using C = Cfg<NFFT>;
  constexpr int M = C::M, N1 = C::N1, N2 = C::N2;
  constexpr int FPI = 32 / N1;  // frames per iteration
  const int q = lane / N1;
  const int c = lane - q * N1;
  const int f = f0 + q;
  const bool act = q < FPI && f < nf;
  const int cc = act ? c : 0;
  const int fr = act ? f : f0;
  const bool middle = (N1 % 2 == 0) && c == N1 / 2;
  const float2 *Y = reinterpret_cast<const float2 *>(regions + fr * C::REGION);
  const float2 *tr = tw2 + cc * C::TWROW;
  float2 v[N2];
#pragma unroll
  for (int i = 0; i < N2; ++i) v[i] = Y[i * C::ROW + cc];
#pragma unroll
  for (int i = 1; i < N2; ++i) v[i] = cmul(v[i], tr[i]);
  Dft<N2>::run(v);  // v[d] = Z[c + N1 d]
  const int src = (act && c != 0 && !middle) ? q * N1 + (N1 - c) : lane;
  float2 r[N2 / 2];  // the partner's values N2 - 1 .. N2 / 2
#pragma unroll
  for (int i = 0; i < N2 / 2; ++i) {
    r[i].x = __shfl_sync(0xffffffffu, v[N2 - 1 - i].x, src);
    r[i].y = __shfl_sync(0xffffffffu, v[N2 - 1 - i].y, src);
  }
  __syncwarp();  // every lane has read the regions before power rows overwrite them
  if (act) {
    const float2 *tu = twu + c * C::TWROW;
    // the power row's offset inside the region: as the mel projection's prow
    float *pw = regions + f * C::REGION + ((f >> 1) & 15);
#pragma unroll
    for (int d = 0; d < N2 / 2; ++d) {
      const float2 B = c == 0 ? v[(N2 - d) % N2] : (middle ? v[N2 - 1 - d] : r[d]);
      float pk, pm;
      untangle_pair(v[d], B, tu[d], power_one, &pk, &pm);
      pw[c + N1 * d] = pk;
      pw[M - c - N1 * d] = pm;
    }
    if (c == 0) {
      float pk, pm;
      untangle_pair(v[N2 / 2], v[N2 / 2], tu[N2 / 2], power_one, &pk, &pm);
      pw[M / 2] = pk;
    }
  }
}

template <int NFFT>
__global__ void __launch_bounds__(Cfg<NFFT>::NT, Cfg<NFFT>::kMinBlocks) wave_reg_kernel(const WaveArgs a) {
  using C = Cfg<NFFT>;
  using Tb = Tables<NFFT>;
  constexpr int M = C::M, TF = C::TF, NT = C::NT, REGION = C::REGION;
  extern __shared__ __align__(16) unsigned char smem[];
  float *regions = reinterpret_cast<float *>(smem);
  unsigned char *tables = smem + 4 * static_cast<size_t>(TF) * REGION;
  const float2 *win2 = reinterpret_cast<const float2 *>(tables);
  const float2 *tw2 = reinterpret_cast<const float2 *>(tables + Tb::tw2_off());
  const float2 *twu = reinterpret_cast<const float2 *>(tables + Tb::twu_off());
  const float *fw = reinterpret_cast<const float *>(tables + Tb::fw_off());
  const int2 *fsw = reinterpret_cast<const int2 *>(tables + Tb::fsw_off(a.n_mels, a.wmax));
  uint32_t *blk_key = reinterpret_cast<uint32_t *>(tables + a.tables_bytes);
  int *abort_flag_p = reinterpret_cast<int *>(blk_key + 1);
  volatile int *next_s = reinterpret_cast<volatile int *>(blk_key + 2);
  volatile int *resc_s = reinterpret_cast<volatile int *>(blk_key + 3);
  uint64_t *tbar = reinterpret_cast<uint64_t *>(blk_key + 4);
  volatile float *floor_s = reinterpret_cast<volatile float *>(blk_key + 6);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(tbar, 1);
    *abort_flag_p = 0;
    *blk_key = 0u;
    fence_mbar_init();
    mbar_arrive_expect_tx(tbar, a.tables_bytes);
    bulk_g2s_plain(tables, a.tables, a.tables_bytes, tbar);
  }
  if (a.token != 0 && blockIdx.x == 0 && a.log_mel && a.fused) {
    // clip_key, clip_done and the rescale counter are adjacent
    for (int64_t i = threadIdx.x; i < 2 * a.B + 1; i += NT) a.clip_key[i] = 0u;
  }
  __syncthreads();  // the barrier is initialised (and CTA 0's clip words are clear)
  if (a.token != 0 && blockIdx.x == 0 && threadIdx.x == 0) publish_cleared(a);
  {
    // While the tables are in flight, pull the first tile's samples into L2
    // (one prefetch per 128-byte line of the tile's span, spread over the
    // threads), so that the two latencies overlap.
    const int64_t tile = blockIdx.x;
    const int64_t b = tile / a.tiles_per_clip;
    const int64_t t0 = (tile - b * a.tiles_per_clip) * static_cast<int64_t>(a.TF);
    const int64_t left = a.n_frames - t0;
    const int nf = left < a.TF ? static_cast<int>(left) : a.TF;
    int64_t s_lo = t0 * a.hop - a.pad_left;
    int64_t s_hi = (t0 + nf - 1) * a.hop - a.pad_left + NFFT;  // one past the last sample
    s_lo = s_lo < 0 ? 0 : s_lo;
    s_hi = s_hi > a.T ? a.T : s_hi;
    if (tile < a.B * a.tiles_per_clip && s_lo < s_hi) {
      const int es = a.in_i16 ? 2 : 4;
      const char *p0 = static_cast<const char *>(a.wave) + (b * a.T + s_lo) * es;
      const int64_t lines = ((s_hi - s_lo) * es + 127) / 128 + 1;
      const uintptr_t l0 = reinterpret_cast<uintptr_t>(p0) & ~uintptr_t{127};
      for (int64_t i = threadIdx.x; i < lines; i += NT) {
        const uintptr_t line = l0 + 128 * static_cast<uintptr_t>(i);
        if (line < reinterpret_cast<uintptr_t>(a.wave) + a.total_bytes)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(line));
      }
    }
  }
  {
    // Without the tables every later shared-memory index is meaningless: if
    // any thread's wait gave up, the whole CTA stops (after the copy lands).
    const bool ok = mbar_wait(tbar, 0, abort_flag_p, a.err);
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) mbar_wait_drain(tbar, 0, a.err);
      return;
    }
  }

  const int64_t n_tiles = a.B * a.tiles_per_clip;
  const bool fused = a.log_mel && a.fused;
  bool token_seen = a.token == 0;  // thread 0
  for (int64_t tile = blockIdx.x, nxt; tile < n_tiles; tile = nxt) {
    const int64_t b = tile / a.tiles_per_clip;
    // a.TF (= TF) frames per tile
    const int64_t t0 = (tile - b * a.tiles_per_clip) * static_cast<int64_t>(a.TF);
    const int64_t left = a.n_frames - t0;
    const int nf = left < a.TF ? static_cast<int>(left) : a.TF;
    const bool wave_pair_aligned =
        (reinterpret_cast<uintptr_t>(a.wave) & (a.in_i16 ? 3u : 7u)) == 0;

    // ---------------- stage 1: framing + N1-point DFTs ----------------
    // Thread b of frame f: N2 threads per frame (32 / N2 frames per pass).
    {
      constexpr int PER = C::N2;
      constexpr int FPP = 32 / PER < C::FPW ? 32 / PER : C::FPW;  // frames per pass
      constexpr int PASSES = C::FPW / FPP;
#pragma unroll 1
      for (int ps = 0; ps < PASSES; ++ps) {
        const int q = ps * FPP + lane / PER;
        const int bb = lane % PER;
        const int f = warp * C::FPW + q;
        if (lane / PER < FPP && f < nf) {
          float2 u[C::N1];
          float2 *row = reinterpret_cast<float2 *>(regions + f * REGION) + bb * C::ROW;
          load_frame<C::N1, C::N2>(a, b, (t0 + f) * a.hop - a.pad_left, bb, wave_pair_aligned, win2, row, u);
          Dft<C::N1>::run(u);
#pragma unroll
          for (int c = 0; c < C::N1; ++c) row[c] = u[c];
          // The row's padding slots hold zeros, not stale bits: the mel
          // projection may read (and multiply by a zero weight) a few floats
          // past a power row, and those must be finite.
#pragma unroll
          for (int c = C::N1; c < C::ROW; ++c) row[c] = make_float2(0.f, 0.f);
        }
      }
    }
    __syncwarp();

    // ------- stage 2: N2-point DFTs, untangle, |2X|^power into the power rows -------
    // Frame f's power row sits inside its own region, at float offset
    // f * REGION + shift(f): lanes over the frames of one bin then hit
    // distinct banks in the mel projection.
    auto prow = [&](int f) { return regions + f * REGION + (NFFT == 1024 ? f : ((f >> 1) & 15)); };
    if constexpr (NFFT != 1024) {
#pragma unroll 1
      for (int q = 0; q < C::FPW; q += 32 / C::N1) {
        const int f0 = warp * C::FPW + q;
        if (f0 >= nf) break;  // warp-uniform
        stage2_cols<NFFT>(regions, f0, nf, lane, tw2, twu, a.power_is_one);
      }
    }
    if constexpr (NFFT == 1024) {
#pragma unroll 1
    for (int q = 0; q < C::FPW; ++q) {
      const int f = warp * C::FPW + q;
      if (f >= nf) break;  // warp-uniform
      const float2 *Y = reinterpret_cast<const float2 *>(regions + f * REGION);
      {
        const int c = lane >> 1, h = lane & 1;
        float2 v[16];
        const float2 *tr = tw2 + lane * C::TWROW;
#pragma unroll
        for (int m = 0; m < 16; ++m) v[m] = cmul(Y[(2 * m + h) * C::ROW + c], tr[m]);
        Dft<16>::run(v);  // V_h[d']
        // Lane 2c + h keeps d = d' + 16 h: X = V0 + (-1)^h W32^d' V1.
#pragma unroll
        for (int d = 0; d < 16; ++d) {
          float2 o;
          o.x = __shfl_xor_sync(0xffffffffu, v[d].x, 1);
          o.y = __shfl_xor_sync(0xffffffffu, v[d].y, 1);
          const float2 V0 = h ? o : v[d];
          const float2 V1 = h ? v[d] : o;
          const float2 T = rot<32>(V1, d);
          v[d] = h ? csub(V0, T) : cadd(V0, T);  // Z[c + 16 d + 256 h]
        }
        // The untangle pair of bin k = c + 16 d + 256 h is bin M - k, lane
        // (lane >= 2 ? 33 - lane : 1 - lane)'s value 15 - d (lanes 0 and 1,
        // column 0: value 16 - d, and d = 0 pairs with itself).  A lane forms
        // both bins of its pairs d = 0..7 (the partner forms d = 8..15; lane 0
        // also forms d = 8, bins 128 and 384), so it fetches only the
        // partner's values 15..8.
        const int src = lane >= 2 ? 33 - lane : 1 - lane;
        float2 r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          r[i].x = __shfl_sync(0xffffffffu, v[15 - i].x, src);
          r[i].y = __shfl_sync(0xffffffffu, v[15 - i].y, src);
        }
        __syncwarp();
        const float2 *tu = twu + lane * C::TWROW;
        float *pwf = regions + f * REGION + f;
        const int k0 = c + 256 * h;
#pragma unroll
        for (int d = 0; d < 8; ++d) {
          const float2 B = lane >= 2 ? r[d] : (d == 0 ? v[0] : r[d - 1]);
          float pk, pm;
          untangle_pair(v[d], B, tu[d], a.power_is_one, &pk, &pm);
          pwf[k0 + 16 * d] = pk;
          pwf[M - k0 - 16 * d] = pm;
        }
        if (lane == 0) {
          float pk, pm;
          untangle_pair(v[8], r[7], tu[8], a.power_is_one, &pk, &pm);
          pwf[128] = pk;
          pwf[384] = pm;
        }
      }
    }
    }
    if (threadIdx.x == 0) *next_s = claim_tile(a, &token_seen, abort_flag_p, static_cast<int>(n_tiles));
    __syncthreads();  // every power row of the tile is complete

    // ---------------- mel projection and store ----------------
    // Lanes run over frames (32 at a time: a warp per band; TF = 16: a
    // half-warp per band), band groups over the rest.
    float lmax = -INFINITY;
    constexpr int LF = TF < 32 ? TF : 32;  // lanes per band
#pragma unroll 1
    for (int fb = 0; fb < TF; fb += LF) {
      constexpr int NG = NT / LF;  // band groups
      const int f = fb + static_cast<int>(threadIdx.x) % LF;
      const int g = static_cast<int>(threadIdx.x) / LF;
      if (f < nf) {
        // The first four taps of every band are read unconditionally: filter
        // rows are zero-padded to a multiple of four, and the floats after a
        // power row are the frame's own finite stage-1 values, so a padded
        // tap adds exactly 0.  Bands are then straight-line code (wider bands
        // finish in a loop) and two bands' chains overlap.
        const float *pr = prow(f);
        const int64_t orow0 = b * a.n_mels * a.n_frames + t0 + f;
#pragma unroll 2
        for (int m = g; m < a.n_mels; m += NG) {
          const int2 sw = fsw[m];
          const float *pa = pr + sw.x;
          const float *wr = fw + m * a.wmax;
          const float4 w4 = *reinterpret_cast<const float4 *>(wr);
          float acc = w4.x * pa[0];
          acc = fmaf(w4.y, pa[1], acc);
          acc = fmaf(w4.z, pa[2], acc);
          acc = fmaf(w4.w, pa[3], acc);
          for (int t = 4; t < sw.y; t += 4) {
            const float4 v4 = *reinterpret_cast<const float4 *>(wr + t);
            acc = fmaf(v4.x, pa[t], acc);
            acc = fmaf(v4.y, pa[t + 1], acc);
            acc = fmaf(v4.z, pa[t + 2], acc);
            acc = fmaf(v4.w, pa[t + 3], acc);
          }
          const int64_t o = orow0 + static_cast<int64_t>(m) * a.n_frames;
          if (a.log_mel) {
            float l2;
            asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(fmaxf(acc, 1e-10f)));
            const float v = l2 * 0.30102999566398120f;  // log10(x) = log2(x) log10(2)
            lmax = fmaxf(lmax, v);
            if (LM_IN_BOUNDS(o, a.B * a.n_mels * a.n_frames, a.err)) static_cast<float *>(a.out)[o] = v;
          } else if (a.out_f16) {
            if (LM_IN_BOUNDS(o, a.B * a.n_mels * a.n_frames, a.err))
              static_cast<__half *>(a.out)[o] = __float2half_rn(acc);
          } else {
            if (LM_IN_BOUNDS(o, a.B * a.n_mels * a.n_frames, a.err)) static_cast<float *>(a.out)[o] = acc;
          }
        }
      }
    }
    if (a.log_mel) {
      const uint32_t key = __reduce_max_sync(0xffffffffu, float_to_ordered(lmax));
      if (lane == 0) atomicMax(blk_key, key);
    }
    nxt = *next_s;
    __syncthreads();  // the regions are free for the next tile; the tile key is complete
    if (a.log_mel && threadIdx.x == 0) {
      if (fused) {
        // Fold the tile maximum into its clip's, then count the tile in with
        // release order: a CTA that sees the count complete sees the maximum.
        if (LM_IN_BOUNDS(b, a.B, a.err)) {
          atomicMax(a.clip_key + b, *blk_key);
          red_add_release_gpu(a.clip_done + b, 1u);
        }
      } else {
        if (LM_IN_BOUNDS(tile, a.B * a.tiles_per_clip, a.err)) a.tile_key[tile] = *blk_key;
      }
      *blk_key = 0u;
    }
  }

  if (fused) {
    // Fused epilogue: every tile has been claimed for computing; take tiles to
    // floor and rescale from the shared counter, in tile order, each once its
    // clip's counter is complete (its log values are still in L2).  Thread 0
    // claims the next tile before waiting for the current one's clip.
    int r_next = 0;  // thread 0
    if (threadIdx.x == 0) r_next = static_cast<int>(atomicAdd(a.rescale_next, 1u));
    for (;;) {
      if (threadIdx.x == 0) {
        const int r = r_next;
        float fl = 0.f;
        if (r < n_tiles) {
          r_next = static_cast<int>(atomicAdd(a.rescale_next, 1u));
          const int64_t b = r / a.tiles_per_clip;
          bool ok = true;
          uint64_t tw0 = 0;
          for (uint32_t it = 0; ld_acquire_gpu(a.clip_done + b) < static_cast<uint32_t>(a.tiles_per_clip); ++it) {
            if ((it & 15u) == 15u) {
              const uint64_t now = global_timer_ns();
              if (tw0 == 0) {
                tw0 = now;
              } else if (now - tw0 > kWaitTimeoutNs) {
                atomicOr(a.err, kErrClipTimeout);
                ok = false;
                break;
              }
            }
            __nanosleep(128);
          }
          fl = ok ? ordered_to_float(ld_relaxed_gpu(a.clip_key + b)) - 8.0f : __int_as_float(0x7fc00000);
        }
        *resc_s = r;
        *floor_s = fl;
      }
      __syncthreads();
      const int64_t tile = *resc_s;
      const float floor_v = *floor_s;
      // every tile is taken, or a wait gave up (the error word says so; the
      // tiles left keep their log values)
      if (tile >= n_tiles || floor_v != floor_v) break;
      const int64_t b = tile / a.tiles_per_clip;
      const int64_t t0 = (tile - b * a.tiles_per_clip) * static_cast<int64_t>(a.TF);
      const int64_t left = a.n_frames - t0;
      const int nf = left < a.TF ? static_cast<int>(left) : a.TF;
      constexpr int LF = TF < 32 ? TF : 32;
      constexpr int NG = NT / LF;
#pragma unroll 1
      for (int fb = 0; fb < TF; fb += LF) {
      const int f = fb + static_cast<int>(threadIdx.x) % LF;
      if (f < nf) {
        // Up to U bands per thread and pass, every load before any store, so
        // the L2 round trips overlap (in place, one at a time they would
        // serialise).  Eight where the kernel runs four CTAs per SM: sixteen
        // would set its register peak above 64.
        constexpr int U = C::kMinBlocks >= 4 ? 8 : 16;
        float *o = static_cast<float *>(a.out) + b * a.n_mels * a.n_frames + t0 + f;
        for (int m0 = static_cast<int>(threadIdx.x) / LF; m0 < a.n_mels; m0 += NG * U) {
          float v[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int m = m0 + u * NG;
            v[u] = (m < a.n_mels && LM_IN_BOUNDS((o - static_cast<float *>(a.out)) + static_cast<int64_t>(m) * a.n_frames,
                                                 a.B * a.n_mels * a.n_frames, a.err))
                       ? o[static_cast<int64_t>(m) * a.n_frames]
                       : 0.f;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int m = m0 + u * NG;
            if (m < a.n_mels && LM_IN_BOUNDS((o - static_cast<float *>(a.out)) + static_cast<int64_t>(m) * a.n_frames,
                                             a.B * a.n_mels * a.n_frames, a.err))
              o[static_cast<int64_t>(m) * a.n_frames] = rescale_log(v[u], floor_v);
          }
        }
      }
      }
      __syncthreads();  // resc_s and floor_s are rewritten for the next tile
    }
  }
  // This CTA is done: a programmatically dependent epilogue may be scheduled
  // (it still waits for the whole grid before reading).
  asm volatile("griddepcontrol.launch_dependents;");
}

}  // namespace reg
