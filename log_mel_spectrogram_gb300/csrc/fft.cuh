// fft.cuh -- shared-memory mixed-radix complex FFT for the waveform path:
// Stockham autosort between two buffers, and an in-place decimation-in-time
// form in one buffer for the largest sizes (end of file); plus the small
// in-register DFT kernels both are made of.
//
// Forward transform, X[k] = sum_n x[n] exp(-2 pi i n k / M).  A pass of
// radix R after earlier passes whose radices multiply to P takes element
// i + j*M/R (j < R) of every frame, multiplies it by exp(-2 pi i j k / (P R))
// with k = i mod P, applies an R-point DFT and writes output l to position
// (i - k) R + k + l P.  After the last pass (P = M) the result is in natural
// order, so no bit reversal is needed.  The twiddle factors are built on the
// host in double precision and laid out pass by pass (see rows_offset).
#pragma once

#include <cuda_runtime.h>

namespace lm {
namespace fft {

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
// (-i) * z
__device__ __forceinline__ float2 mul_neg_i(float2 z) { return make_float2(z.y, -z.x); }
__device__ __forceinline__ float2 cscale(float2 z, float s) { return make_float2(z.x * s, z.y * s); }

// Frame buffers of power-of-two transforms hold element x at x + x / 32: one
// padding slot every 32 elements, so the power-of-radix strides of the
// passes do not land in the same banks (a radix-8 pass over 512 points
// otherwise stores with a 64-byte stride, 16 lanes to one bank).  Mixed-radix
// sizes (400) are laid out unpadded: their strides spread over the banks and
// the extra index arithmetic measured slower.
template <int M>
struct Layout {
  static constexpr bool kPad = (M & (M - 1)) == 0;
  __host__ __device__ static constexpr int at(int x) { return kPad ? x + (x >> 5) : x; }
  // slots a buffer of n logical elements occupies
  __host__ __device__ static constexpr int size(int n) { return kPad ? n + (n >> 5) + 1 : n; }
};

// The in-place layout adds a second padding slot every 512 elements: the
// digit-reversed stores of the framing step (consecutive inputs to positions
// 64, 512 and 4096 apart) then spread over the banks instead of landing in
// one or two.
template <int M>
struct LayoutIP {
  __host__ __device__ static constexpr int at(int x) { return x + (x >> 5) + (x >> 9); }
  __host__ __device__ static constexpr int size(int n) { return n + (n >> 5) + (n >> 9) + 1; }
};

template <int R>
struct Dft;

template <>
struct Dft<2> {
  __device__ __forceinline__ static void run(float2 (&u)[2]) {
    const float2 a = u[0], b = u[1];
    u[0] = cadd(a, b);
    u[1] = csub(a, b);
  }
};

template <>
struct Dft<4> {
  __device__ __forceinline__ static void run(float2 (&u)[4]) {
    const float2 t0 = cadd(u[0], u[2]), t1 = csub(u[0], u[2]);
    const float2 t2 = cadd(u[1], u[3]), t3 = mul_neg_i(csub(u[1], u[3]));
    u[0] = cadd(t0, t2);
    u[2] = csub(t0, t2);
    u[1] = cadd(t1, t3);
    u[3] = csub(t1, t3);
  }
};

template <>
struct Dft<8> {
  // Two 4-point DFTs over the even and odd inputs, joined with the eighth
  // roots of unity exp(-2 pi i l / 8), l < 4.
  __device__ __forceinline__ static void run(float2 (&u)[8]) {
    constexpr float h = 0.70710678118654752f;  // sqrt(1/2)
    float2 e[4] = {u[0], u[2], u[4], u[6]};
    float2 o[4] = {u[1], u[3], u[5], u[7]};
    Dft<4>::run(e);
    Dft<4>::run(o);
    const float2 o1 = make_float2(h * (o[1].x + o[1].y), h * (o[1].y - o[1].x));   // (1 - i)/sqrt2
    const float2 o2 = mul_neg_i(o[2]);                                               // -i
    const float2 o3 = make_float2(h * (o[3].y - o[3].x), -h * (o[3].x + o[3].y));  // (-1 - i)/sqrt2
    u[0] = cadd(e[0], o[0]);
    u[4] = csub(e[0], o[0]);
    u[1] = cadd(e[1], o1);
    u[5] = csub(e[1], o1);
    u[2] = cadd(e[2], o2);
    u[6] = csub(e[2], o2);
    u[3] = cadd(e[3], o3);
    u[7] = csub(e[3], o3);
  }
};

template <>
struct Dft<5> {
  // U_l = sum_j u_j w^{jl}, w = exp(-2 pi i / 5) = c1 - i s1, w^2 = c2 - i s2.
  __device__ __forceinline__ static void run(float2 (&u)[5]) {
    constexpr float c1 = 0.30901699437494742f;   // cos(2 pi / 5)
    constexpr float c2 = -0.80901699437494742f;  // cos(4 pi / 5)
    constexpr float s1 = 0.95105651629515357f;   // sin(2 pi / 5)
    constexpr float s2 = 0.58778525229247313f;   // sin(4 pi / 5)
    const float2 a1 = cadd(u[1], u[4]), a2 = cadd(u[2], u[3]);
    const float2 b1 = csub(u[1], u[4]), b2 = csub(u[2], u[3]);
    const float2 t1 = make_float2(u[0].x + c1 * a1.x + c2 * a2.x, u[0].y + c1 * a1.y + c2 * a2.y);
    const float2 t2 = make_float2(u[0].x + c2 * a1.x + c1 * a2.x, u[0].y + c2 * a1.y + c1 * a2.y);
    const float2 r1 = make_float2(s1 * b1.x + s2 * b2.x, s1 * b1.y + s2 * b2.y);  // U1 = t1 - i r1
    const float2 r2 = make_float2(s2 * b1.x - s1 * b2.x, s2 * b1.y - s1 * b2.y);  // U2 = t2 - i r2
    u[0] = make_float2(u[0].x + a1.x + a2.x, u[0].y + a1.y + a2.y);
    u[1] = cadd(t1, mul_neg_i(r1));
    u[4] = csub(t1, mul_neg_i(r1));
    u[2] = cadd(t2, mul_neg_i(r2));
    u[3] = csub(t2, mul_neg_i(r2));
  }
};

template <>
struct Dft<16> {
  // 16 = 4 x 4: inputs j = 4a + b, outputs l = c + 4d.  Four 4-point DFTs
  // over a, the factors exp(-2 pi i b c / 16), four 4-point DFTs over b.
  __device__ __forceinline__ static void run(float2 (&u)[16]) {
    constexpr float c1 = 0.92387953251128674f;  // cos(pi / 8)
    constexpr float s1 = 0.38268343236508977f;  // sin(pi / 8)
    constexpr float h = 0.70710678118654752f;   // sqrt(1/2)
    float2 v[4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float2 t[4] = {u[b], u[4 + b], u[8 + b], u[12 + b]};
      Dft<4>::run(t);
#pragma unroll
      for (int c = 0; c < 4; ++c) v[b][c] = t[c];
    }
    // exp(-2 pi i m / 16) for m = b c: 1 = (c1, -s1), 2 = (h, -h), 3 = (s1, -c1),
    // 4 = -i, 6 = (-h, -h), 9 = (-c1, s1)
    v[1][1] = cmul(v[1][1], make_float2(c1, -s1));
    v[1][2] = cmul(v[1][2], make_float2(h, -h));
    v[1][3] = cmul(v[1][3], make_float2(s1, -c1));
    v[2][1] = cmul(v[2][1], make_float2(h, -h));
    v[2][2] = mul_neg_i(v[2][2]);
    v[2][3] = cmul(v[2][3], make_float2(-h, -h));
    v[3][1] = cmul(v[3][1], make_float2(s1, -c1));
    v[3][2] = cmul(v[3][2], make_float2(-h, -h));
    v[3][3] = cmul(v[3][3], make_float2(-c1, s1));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float2 t[4] = {v[0][c], v[1][c], v[2][c], v[3][c]};
      Dft<4>::run(t);
#pragma unroll
      for (int d = 0; d < 4; ++d) u[c + 4 * d] = t[d];
    }
  }
};

// Radix of the pass that follows span P: 5 while M/P has a factor 5, then 8
// while possible, then the leftover 4 or 2.
template <int M, int P>
__host__ __device__ constexpr int next_radix() {
  return ((M / P) % 5 == 0) ? 5 : ((M / P) % 8 == 0) ? 8 : ((M / P) % 4 == 0) ? 4 : 2;
}

// Twiddle table layout.  The pass with span P > 1 and radix R multiplies
// input j of a butterfly with k = i mod P by exp(-2 pi i j k / (P R)); its
// factors for j = 1..R-1 form row k, rows of row_stride<R>() values, P rows
// per pass, passes back to back in order (the first pass, P = 1, needs
// none).  A thread reads its R - 1 factors from one row at fixed offsets,
// and the stride (7, 3 or 1 for radix 8, 4 or 2; radix 5 padded to 5) is
// odd, so the rows of 16 consecutive butterflies fall in 16 distinct 8-byte
// bank slots.  The rows take fewer than M entries for every supported M.
template <int R>
__host__ __device__ constexpr int row_stride() {
  return R == 5 ? 5 : R - 1;
}

// Offset of the rows of the pass with span Q.
template <int M, int Q, int P = 1>
__host__ __device__ constexpr int rows_offset() {
  if constexpr (P >= Q) {
    return 0;
  } else {
    constexpr int R = next_radix<M, P>();
    return (P > 1 ? P * row_stride<R>() : 0) + rows_offset<M, Q, P * R>();
  }
}

// One Stockham pass over FRAMES frames of M points stored back to back (at
// Layout<M> positions), by NT threads (the block size); every loop bound is
// a compile-time constant.
template <int M, int R, int P, int FRAMES, int NT>
__device__ __forceinline__ void pass(const float2 *__restrict__ in, float2 *__restrict__ out,
                                     const float2 *__restrict__ W) {
  constexpr int T = M / R;
  constexpr int ITEMS = FRAMES * T;
#pragma unroll
  for (int r = 0; r < (ITEMS + NT - 1) / NT; ++r) {
    const int g = static_cast<int>(threadIdx.x) + r * NT;
    if (ITEMS % NT != 0 && g >= ITEMS) break;
    const int f = g / T;
    const int i = g - f * T;
    const int k = i % P;
    const int base = f * M + i;
    float2 u[R];
#pragma unroll
    for (int j = 0; j < R; ++j) u[j] = in[Layout<M>::at(base + j * T)];
    if constexpr (P > 1) {
      const float2 *row = W + rows_offset<M, P>() + k * row_stride<R>();
#pragma unroll
      for (int j = 1; j < R; ++j) u[j] = cmul(u[j], row[j - 1]);
    }
    Dft<R>::run(u);
    const int obase = f * M + (i - k) * R + k;
#pragma unroll
    for (int l = 0; l < R; ++l) out[Layout<M>::at(obase + l * P)] = u[l];
  }
}

// Number of passes for an M-point transform (the result ends in the second
// buffer when it is odd).
template <int M, int P = 1>
__host__ __device__ constexpr int num_passes() {
  if constexpr (P == M) {
    return 0;
  } else {
    return 1 + num_passes<M, P * next_radix<M, P>()>();
  }
}

// Runs every pass over FRAMES frames with NT threads, ping-ponging between a
// and b.  Returns true when the result ends in b.
template <int M, int FRAMES, int NT, int P = 1>
__device__ __forceinline__ bool run(float2 *a, float2 *b, const float2 *W) {
  if constexpr (P == M) {
    return false;
  } else {
    constexpr int R = next_radix<M, P>();
    pass<M, R, P, FRAMES, NT>(a, b, W);
    __syncthreads();
    return !run<M, FRAMES, NT, P * R>(b, a, W);
  }
}

// Radix of the in-place pass that follows span P: 16 for the first pass of
// the in-place sizes (M >= 4096; it needs no twiddle factors, so its 16
// points fit the registers of two 512-thread CTAs per SM), then the rule of
// next_radix.  One pass fewer than radix 8 at M = 8192, and no pass with span
// 8, whose butterflies fall two lanes to a bank.
template <int M, int P>
__host__ __device__ constexpr int ip_radix() {
  return (P == 1 && M >= 4096 && M % 16 == 0) ? 16 : next_radix<M, P>();
}

// Offset of the in-place pass with span Q in the twiddle table (the rows of
// rows_offset, for the passes of ip_radix).
template <int M, int Q, int P = 1>
__host__ __device__ constexpr int ip_rows_offset() {
  if constexpr (P >= Q) {
    return 0;
  } else {
    constexpr int R = ip_radix<M, P>();
    return (P > 1 ? P * row_stride<R>() : 0) + ip_rows_offset<M, Q, P * R>();
  }
}

// In-place form (decimation in time) for transforms too large for two
// buffers: the input goes to the digit-reversed position dit_pos(n), and the
// pass of radix R after span P applies butterfly (g, k), k < P, to the
// elements g R P + k + j P (j < R), multiplying element j by
// exp(-2 pi i j k / (P R)) -- the same factors, and the same row layout, as
// the Stockham pass, for the radices of ip_radix -- and writing output l back
// to g R P + k + l P.  After the last pass the result is in natural order.
//
// Position of input n: the first pass transforms the R1 inputs n' + j M/R1
// (j < R1) of group n' < M/R1, which sit at R1 dit_pos<M/R1>(n') + j.
template <int M>
__device__ __forceinline__ int dit_pos(int n) {
  if constexpr (M == 1) {
    return 0;
  } else {
    constexpr int R = ip_radix<M, 1>();
    constexpr int S = M / R;
    return dit_pos<S>(n % S) * R + n / S;
  }
}

// One in-place pass over one frame of M points (at LayoutIP<M> positions) by
// NT threads; the twiddle rows are read through L1 from global memory.
// When a thread's factors for the whole pass take at most 16 float2, it
// loads all of them before its first butterfly, so their L2 round trips
// overlap instead of following one another butterfly by butterfly.
template <int M, int R, int P, int NT>
__device__ __forceinline__ void pass_inplace(float2 *x, const float2 *__restrict__ W) {
  constexpr int ITEMS = M / R;
  constexpr int ROUNDS = (ITEMS + NT - 1) / NT;
  constexpr bool kAhead = P > 1 && ITEMS % NT == 0 && ROUNDS * (R - 1) <= 16;
  float2 tw[kAhead ? ROUNDS : 1][R];
  if constexpr (kAhead) {
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
      const int t = static_cast<int>(threadIdx.x) + r * NT;
      const float2 *row = W + ip_rows_offset<M, P>() + (t % P) * row_stride<R>();
#pragma unroll
      for (int j = 1; j < R; ++j) tw[r][j] = __ldg(row + j - 1);
    }
  }
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int t = static_cast<int>(threadIdx.x) + r * NT;
    if (ITEMS % NT != 0 && t >= ITEMS) break;
    const int k = t % P;
    const int base = (t / P) * R * P + k;
    float2 u[R];
#pragma unroll
    for (int j = 0; j < R; ++j) u[j] = x[LayoutIP<M>::at(base + j * P)];
    if constexpr (kAhead) {
#pragma unroll
      for (int j = 1; j < R; ++j) u[j] = cmul(u[j], tw[r][j]);
    } else if constexpr (P > 1) {
      const float2 *row = W + ip_rows_offset<M, P>() + k * row_stride<R>();
#pragma unroll
      for (int j = 1; j < R; ++j) u[j] = cmul(u[j], __ldg(row + j - 1));
    }
    Dft<R>::run(u);
#pragma unroll
    for (int l = 0; l < R; ++l) x[LayoutIP<M>::at(base + l * P)] = u[l];
  }
}

// Every pass from span P on, in place; a block barrier follows each.
template <int M, int NT, int P = 1>
__device__ __forceinline__ void run_inplace(float2 *x, const float2 *W) {
  if constexpr (P < M) {
    constexpr int R = ip_radix<M, P>();
    pass_inplace<M, R, P, NT>(x, W);
    __syncthreads();
    run_inplace<M, NT, P * R>(x, W);
  }
}

}  // namespace fft
}  // namespace lm
