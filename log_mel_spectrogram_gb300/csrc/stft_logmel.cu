// stft_logmel.cu -- Whisper log-mel spectrogram from a complex STFT.
//
// Computes, per clip b (KBench "audio_mel_spectrogram_fused" spec, per-clip
// definition):
//   mag = re^2 + im^2;  mel = mag . W^T;  ls = log10(max(mel, 1e-10));
//   hi[b] = max over the clip of ls;  out = (max(ls, hi[b] - 8) + 4) / 4.
//
// Design (GB300; HBM-bound: 8 bytes read per bin, 4 written per band):
//
//  * One persistent CTA per SM walks frame tiles in clip order
//    (tile = blockIdx.x + k * gridDim.x).  A tile is TF consecutive frames
//    of one clip and is contiguous in memory.  Tiles are numbered clip-major.
//  * A producer warp streams tiles into an S-stage shared-memory ring with
//    1-D bulk copies (cp.async.bulk, L2 evict-first), each stage guarded by a
//    full/empty mbarrier pair.  Frames are 8*NF bytes, so a tile may start 8
//    bytes off a 16-byte boundary: the copy starts at the aligned address
//    below and the consumers index from the remainder.
//  * CW consumer warps compute the tile.  Thread (n, g) owns mel band n and
//    frames g, g+FG, ...; its band's support (first..last nonzero of the
//    dense filter row, found once per CTA) and up to kRegTaps weights sit in
//    registers.  Each tap is one 8-byte shared load and two packed f32x2
//    operations: acc += (w*re, w*im) * (re, im), so power and projection are
//    formed together and the two halves are summed once per output.
//  * Per-clip maximum without a second HBM pass: each warp reduces its tile
//    maximum with shuffles into a shared slot; a publisher warp stores the
//    tile's maximum (order-preserving u32 key, 0 = not yet published) into a
//    per-tile slot in global memory with one plain store -- no atomics, no
//    fences.  Tiles of a clip have contiguous slots.
//  * Resident mode (default): consumers keep each tile's log values in a
//    shared-memory ring for kLag more steps.  A resolver warp, once its own
//    CTA has published every step the clip can reach, reads the clip's slots
//    in one warp-wide pass (repeating until none is zero), and hands the
//    clip maximum to the consumers through an mbarrier; they then write the
//    final values once.  The output is written to HBM exactly once and never
//    re-read: one read of the source and one write of the result, the spec's
//    canonical traffic.  Cross-CTA waits need all CTAs resident, so this mode
//    is launched cooperatively.
//  * Two-pass mode (a clip spans more steps than kLag, or forced with
//    LOGMEL_K1_VARIANT=twopass): consumers write the log values, the
//    publisher still fills the tile slots, and a second kernel reduces each
//    clip's slots and applies the floor and rescale in place.
#include <algorithm>
#include <array>
#include <cfloat>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace lm {
namespace {

constexpr int kLag = 7;          // resident mode: steps a tile's log values wait in shared memory
constexpr int kResolveSteps = 8;  // steps the resolver polls together
constexpr int kSlots = 32;       // ring of per-step handshake slots (> kLag + kMaxStages)
constexpr int kMaxStages = 8;
constexpr int kRegTaps = 8;      // filter taps held in registers per band (packed filters assume 8)
constexpr int kMaxBands = 512;
constexpr int kMaxBins = 8193;
constexpr int kStageTargetBytes = 41 * 1024;

constexpr int threads_for(int cw) { return (cw + 3) * 32; }

struct StftArgs {
  const float2 *stft;
  const float *filters;
  float *out;
  uint32_t *err;
  uint32_t *tile_key;      // [n_tiles] key of each tile's max log value, 0 = not yet published
  int64_t B, F;
  int32_t NF, NM;
  int32_t FG;              // frame groups: active consumer threads = FG * NM
  int32_t TF;              // frames per tile (FG * FPT)
  int32_t tiles_per_clip;  // ceil(F / TF)
  int32_t span;            // steps a clip can extend past any of its steps on one CTA
  int64_t n_tiles;         // B * tiles_per_clip
  int64_t grid_q;          // gridDim.x / tiles_per_clip
  int32_t grid_r;          // gridDim.x % tiles_per_clip
  int32_t n_stages;
  uint32_t stage_stride;   // bytes per stage, multiple of 128
  uint32_t aux_offset;     // shared-memory offset of SmemAux (after the stages and the ring)
  uint64_t total_bytes;    // B * F * NF * 8
  const int32_t *packed;   // packed filter supports and first taps (see PackLayout), or null
  uint64_t clip_wait_ns;   // how long the resolver waits for a clip's maximum before giving up
  int64_t withhold_tile;   // fault injection (tests only): this tile's maximum is never published; -1 = none
  int32_t cluster;         // cluster variant: CTAs per clip (one thread-block cluster)
  int32_t frames_per_cta;  // cluster variant: frames of the clip per CTA
  uint32_t obuf_offset;    // cluster variant: shared-memory offset of the CTA's output slice
  int32_t clear_err;       // cluster variant: CTA 0 clears the error word (it is this call's own)
};

// Packed filters: header {magic, NF, NM, widest support}, then {first bin,
// width} per band, then the first kRegTaps weights of each band's support
// (zero past its width).  Built once by mel_filters_pack_kernel so that a
// call's prologue is one memory round trip instead of a sweep of the dense
// matrix followed by the tap loads.
struct PackLayout {
  static constexpr int32_t kMagic = 0x464d4c50;  // "PLMF"
  static constexpr size_t kHeader = 16;
  __host__ __device__ static size_t sw_offset() { return kHeader; }
  // the taps start 16-byte aligned (they are read as float4)
  __host__ __device__ static size_t taps_offset(int32_t NM) {
    return kHeader + (8 * static_cast<size_t>(NM) + 15) / 16 * 16;
  }
  __host__ __device__ static size_t bytes(int32_t NM) {
    return taps_offset(NM) + 4 * static_cast<size_t>(kRegTaps) * NM;  // a multiple of 16: kRegTaps = 8
  }
};

struct SmemAux {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tmax_bar[kSlots];  // consumers -> publisher: tile maximum folded in
  uint64_t pub_bar[kSlots];   // publisher -> resolver: tile maximum stored
  uint64_t hi_bar[kSlots];    // resolver -> consumers: clip maximum available
  uint32_t tmax_key[kSlots];
  float hi_val[kSlots];
  int64_t desc_frame0[kSlots];  // producer -> consumers: first frame of step k's tile
  int32_t desc_nf[kSlots];      // frames in the tile
  int32_t desc_head[kSlots];    // byte offset of the tile inside its stage (0 or 8)
  int32_t band_start[kMaxBands];
  int32_t band_width[kMaxBands];
  int32_t max_width;
  int32_t abort_flag;
};

// Walks this CTA's tiles: clip index b and tile index within the clip.
struct TileIter {
  int64_t b;
  int32_t loc;
  __device__ __forceinline__ void init(int64_t tile, int32_t tpc) {
    b = tile / tpc;
    loc = static_cast<int32_t>(tile - b * tpc);
  }
  __device__ __forceinline__ void next(const StftArgs &a) {
    b += a.grid_q;
    loc += a.grid_r;
    if (loc >= a.tiles_per_clip) {
      loc -= a.tiles_per_clip;
      ++b;
    }
  }
  __device__ __forceinline__ int64_t first_frame(const StftArgs &a) const {
    return b * a.F + static_cast<int64_t>(loc) * a.TF;
  }
  __device__ __forceinline__ int frames(const StftArgs &a) const {
    const int64_t left = a.F - static_cast<int64_t>(loc) * a.TF;
    return left < a.TF ? static_cast<int>(left) : a.TF;
  }
};

// sum_t w[t] * |fr[t]|^2 over the first `wd` taps, weights from registers
// (each w2[t] holds the weight twice).  Accumulates (w re^2, w im^2) in one
// packed pair and adds the halves at the end.
template <int W>
__device__ __forceinline__ float band_sum(const float2 *fr, int wd, const float2 (&w2)[kRegTaps]) {
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int t = 0; t < W; ++t) {
    if (t < wd) {
      const float2 c = fr[t];
      acc = __ffma2_rn(__fmul2_rn(w2[t], c), c, acc);
    }
  }
  return acc.x + acc.y;
}

// Bands wider than kRegTaps: the remaining weights come through L1 (the
// filter matrix is read-only).
__device__ __forceinline__ float band_sum_wide(const float2 *fr, int wd, const float2 (&w2)[kRegTaps],
                                               const float *wrow) {
  float acc = band_sum<kRegTaps>(fr, wd, w2);
  for (int t = kRegTaps; t < wd; ++t) {
    const float2 c = fr[t];
    acc = fmaf(__ldg(wrow + t), fmaf(c.x, c.x, c.y * c.y), acc);
  }
  return acc;
}

// log10(x) = log2(x) * log10(2) for normal x > 0 (the argument is floored
// at 1e-10 first).  The hardware base-2 logarithm has an absolute error
// below 2^-22 for these arguments, far inside the output tolerance.
__device__ __forceinline__ float fast_log10(float x) {
  float l2;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(x));
  return l2 * 0.30102999566398120f;
}

__device__ __forceinline__ float rescale(float ls, float floor_v) {
  // (max(ls, hi - 8) + 4) / 4; fma(x, 1/4, 1) rounds exactly like (x + 4) / 4.
  return fmaf(fmaxf(ls, floor_v), 0.25f, 1.0f);
}

// Per-thread constants of a consumer: its mel band, frame group and the
// band's support with the first kRegTaps weights in registers.
struct Band {
  int n, fg;
  bool active;
  int st, wd;
  float2 w2[kRegTaps];
  const float *wrow;
};

// Consumer main loop.  W = number of register taps (4 or 8), or 0 for bands
// wider than kRegTaps.
template <int FPT, int W, bool kResident, int CW>
__device__ __forceinline__ void consume(const StftArgs &a, unsigned char *smem, SmemAux &aux, float *ring,
                                        int64_t my_tiles, const Band &c, int lane) {
  volatile int *abort_flag = &aux.abort_flag;
  const int S = a.n_stages;
  const int fstep = a.FG * a.NF;    // complex values between a thread's frames
  const int ostep = a.FG * a.NM;    // outputs between a thread's frames
  const int slot_stride = a.TF * a.NM;
  const int own = c.fg * a.NM + c.n;  // this thread's first output inside a tile
  int s = 0, slot = 0, sslot = 0;
  uint32_t ph = 0;

  // Final values of step q from this thread's own ring entries.  The tile
  // descriptor of step q is still in its slot: the producer runs at most
  // n_stages (< kSlots - kLag) steps ahead of the consumers.
  // Returns false, storing nothing, when the wait for the clip maximum gave
  // up (the CTA is aborting).
  auto store_final = [&](int64_t q) -> bool {
    const int d = static_cast<int>(q & (kSlots - 1));
    const bool ok = mbar_wait(&aux.hi_bar[d], static_cast<uint32_t>((q / kSlots) & 1), abort_flag, a.err);
    if (!__all_sync(0xffffffffu, ok)) return false;
    const float floor_v = aux.hi_val[d] - 8.0f;
    const int nf = aux.desc_nf[d];
    const float *r = ring + sslot * slot_stride + own;
    float *o = a.out + aux.desc_frame0[d] * a.NM + own;
    if (c.active) {
#pragma unroll
      for (int j = 0; j < FPT; ++j)
        if (c.fg + j * a.FG < nf && LM_IN_BOUNDS((o - a.out) + j * ostep, a.B * a.F * a.NM, a.err))
          __stcs(o + j * ostep, rescale(r[j * ostep], floor_v));
    }
    if (++sslot == kLag + 1) sslot = 0;
    return true;
  };

  for (int64_t k = 0; k < my_tiles; ++k) {
    if constexpr (!kResident) {
      // Nothing else holds the consumers back in this mode: stay at most
      // kSlots / 2 steps ahead of the publisher so no handshake slot is
      // reused before the publisher has read it.
      if (k >= kSlots / 2) {
        const int64_t j = k - kSlots / 2;
        const bool ok =
            mbar_wait(&aux.pub_bar[j & (kSlots - 1)], static_cast<uint32_t>((j / kSlots) & 1), abort_flag, a.err);
        if (!__all_sync(0xffffffffu, ok)) return;
      }
    }
    // A wait that gave up means the CTA is aborting: the warp leaves without
    // touching the stage (the producer may never have filled it) or global
    // memory.  The vote keeps the lanes together.
    if (!__all_sync(0xffffffffu, mbar_wait(&aux.full[s], ph, abort_flag, a.err))) return;
    const int d = static_cast<int>(k & (kSlots - 1));
    const int64_t frame0 = aux.desc_frame0[d];
    const int nf = aux.desc_nf[d];
    const float2 *fr = reinterpret_cast<const float2 *>(smem + static_cast<size_t>(s) * a.stage_stride +
                                                        aux.desc_head[d]) +
                       (c.st + c.fg * a.NF);
    float *dst = kResident ? ring + slot * slot_stride + own : a.out + frame0 * a.NM + own;
    float lmax = -INFINITY;
    if (c.active) {
#pragma unroll
      for (int j = 0; j < FPT; ++j) {
        if (nf == a.TF || c.fg + j * a.FG < nf) {
          float acc;
          if constexpr (W > 0) {
            acc = band_sum<W>(fr + j * fstep, c.wd, c.w2);
          } else {
            acc = band_sum_wide(fr + j * fstep, c.wd, c.w2, c.wrow);
          }
          const float v = fast_log10(fmaxf(acc, 1e-10f));
          lmax = fmaxf(lmax, v);
          if constexpr (kResident) {
            dst[j * ostep] = v;  // the shared-memory ring
          } else {
            if (LM_IN_BOUNDS((dst - a.out) + j * ostep, a.B * a.F * a.NM, a.err)) dst[j * ostep] = v;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&aux.empty[s]);
    const uint32_t wkey = __reduce_max_sync(0xffffffffu, float_to_ordered(lmax));
    if (lane == 0) {
      atomicMax(&aux.tmax_key[d], wkey);
      mbar_arrive(&aux.tmax_bar[d]);
    }
    if constexpr (kResident) {
      if (k >= kLag && !store_final(k - kLag)) return;
      if (++slot == kLag + 1) slot = 0;
    }
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  if constexpr (kResident) {
    for (int64_t q = my_tiles > kLag ? my_tiles - kLag : 0; q < my_tiles; ++q)
      if (!store_final(q)) return;
  }
}

// A consumer thread's band: its index, frame group and support, with the
// first kRegTaps weights in registers (from a matching pack in one round of
// loads, else from a sweep of the dense matrix by all CW * 32 consumer
// threads, which synchronise on named barrier 1).  Returns the widest
// support of any band.
template <int CW>
__device__ __forceinline__ int setup_band(const StftArgs &a, SmemAux &aux, Band &band) {
  constexpr int kConsumers = CW * 32;
  band.n = threadIdx.x % a.NM;
  band.fg = threadIdx.x / a.NM;
  band.active = band.fg < a.FG;
  int maxw;
  // Packed filters that match this call: supports and first taps in one
  // round of loads.  Anything else (no pack, or one made for another shape)
  // derives them from the dense matrix; a mismatched pack is reported.
  bool use_pack = a.packed != nullptr;
  int4 hdr = make_int4(0, 0, 0, 0);
  if (use_pack) {
    hdr = __ldg(reinterpret_cast<const int4 *>(a.packed));
    use_pack = hdr.x == PackLayout::kMagic && hdr.y == a.NF && hdr.z == a.NM;
    if (!use_pack && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(a.err, kErrBadPack);  // once per call
  }
  if (use_pack) {
    const int2 *sw = reinterpret_cast<const int2 *>(reinterpret_cast<const char *>(a.packed) + PackLayout::sw_offset());
    const float4 *tw = reinterpret_cast<const float4 *>(reinterpret_cast<const char *>(a.packed) +
                                                        PackLayout::taps_offset(a.NM)) +
                       static_cast<int64_t>(band.n) * (kRegTaps / 4);
    const int2 v = __ldg(sw + band.n);
    float wt[kRegTaps];
#pragma unroll
    for (int q = 0; q < kRegTaps / 4; ++q) {
      const float4 t4 = __ldg(tw + q);
      wt[4 * q] = t4.x;
      wt[4 * q + 1] = t4.y;
      wt[4 * q + 2] = t4.z;
      wt[4 * q + 3] = t4.w;
    }
    maxw = hdr.w;
    band.st = band.active ? v.x : 0;
    band.wd = band.active ? v.y : 0;
#pragma unroll
    for (int t = 0; t < kRegTaps; ++t) band.w2[t] = band.active ? make_float2(wt[t], wt[t]) : make_float2(0.f, 0.f);
  } else {
    // Support of each filter row: first and last nonzero bin.  All consumer
    // threads sweep the dense matrix together with eight independent loads in
    // flight each, folding nonzeros into shared minima and maxima
    // (band_width holds the last nonzero bin until the final pass).
    for (int n = threadIdx.x; n < a.NM; n += kConsumers) {
      aux.band_start[n] = INT_MAX;
      aux.band_width[n] = -1;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
    {
      // 32-bit indices (NM * NF < 2^23): a 64-bit division here cost microseconds.
      constexpr int U = 8;
      const int total = a.NM * a.NF;
      for (int i0 = threadIdx.x; i0 < total; i0 += U * kConsumers) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + u * kConsumers;
          v[u] = i < total ? __ldg(a.filters + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (v[u] != 0.f) {
            const int i = i0 + u * kConsumers;
            const int r = i / a.NF;
            atomicMin(&aux.band_start[r], i - r * a.NF);
            atomicMax(&aux.band_width[r], i - r * a.NF);
          }
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
    for (int n = threadIdx.x; n < a.NM; n += kConsumers) {
      const int first = aux.band_start[n], last = aux.band_width[n];
      const int width = last >= 0 ? last - first + 1 : 0;
      aux.band_start[n] = last >= 0 ? first : 0;
      aux.band_width[n] = width;
      atomicMax(&aux.max_width, width);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");

    maxw = aux.max_width;
    band.st = band.active ? aux.band_start[band.n] : 0;
    band.wd = band.active ? aux.band_width[band.n] : 0;
#pragma unroll
    for (int t = 0; t < kRegTaps; ++t) {
      const float wt = (t < band.wd) ? __ldg(a.filters + static_cast<int64_t>(band.n) * a.NF + band.st + t) : 0.f;
      band.w2[t] = make_float2(wt, wt);
    }
  }
  band.wrow = a.filters + static_cast<int64_t>(band.n) * a.NF + band.st;
  return maxw;
}

template <int FPT, bool kResident, int CW>
__global__ void __launch_bounds__(threads_for(CW), 1) stft_logmel_kernel(const StftArgs a) {
  constexpr int kProducerWarp = CW;
  constexpr int kPublisherWarp = CW + 1;
  constexpr int kResolverWarp = CW + 2;
  extern __shared__ __align__(128) unsigned char smem[];
  SmemAux &aux = *reinterpret_cast<SmemAux *>(smem + a.aux_offset);
  volatile int *abort_flag = &aux.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int64_t my_tiles = (a.n_tiles - 1 - blockIdx.x) / G + 1;
  const int S = a.n_stages;

  // Warp 0 initialises the barriers, a lane per handshake slot (kSlots =
  // 32), each lane fencing its own initialisations.
  static_assert(kSlots == 32 && kMaxStages <= 32, "one lane per slot");
  if (warp == 0) {
    if (lane < S) {
      mbar_init(&aux.full[lane], 1);
      mbar_init(&aux.empty[lane], CW);
    }
    mbar_init(&aux.tmax_bar[lane], CW);
    mbar_init(&aux.pub_bar[lane], 1);
    mbar_init(&aux.hi_bar[lane], 1);
    aux.tmax_key[lane] = 0u;
    if (lane == 0) {
      aux.max_width = 0;
      aux.abort_flag = 0;
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------- producer: bulk copies of frame tiles ----------------
    // Addresses are absolute: the tensor need only be 8-byte aligned.  A
    // tile's copy covers the 16-byte aligned range around it; where that
    // range would start before the tensor (its first value sits 8 bytes past
    // a boundary) or end after it, the one complex value concerned is copied
    // by hand and the bulk copy shrinks to the aligned part.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint64_t base = reinterpret_cast<uint64_t>(a.stft);
      const uint64_t limit = base + a.total_bytes;
      TileIter it;
      it.init(blockIdx.x, a.tiles_per_clip);
      int s = 0;
      uint32_t ph = 0;
      uint32_t generic_written = 0;  // stages holding a hand-copied value
      int64_t issued = 0;
      for (int64_t k = 0; k < my_tiles; ++k) {
        if (k >= S && !mbar_wait(&aux.empty[s], ph ^ 1u, abort_flag, a.err)) break;
        const uint64_t start = base + static_cast<uint64_t>(it.first_frame(a)) * a.NF * 8ull;
        const uint64_t end = start + static_cast<uint64_t>(it.frames(a)) * a.NF * 8ull;
        const uint64_t a0 = start & ~15ull;  // the address stage byte 0 stands for
        uint64_t lo = a0;
        uint64_t hi = (end + 15ull) & ~15ull;
        unsigned char *dst = smem + static_cast<size_t>(s) * a.stage_stride;
        if ((generic_written >> s) & 1u) {
          // the bulk copy below may overwrite bytes written by hand earlier
          fence_proxy_async_smem();
          generic_written &= ~(1u << s);
        }
        if (lo < base) {
          // the first tile of a tensor that starts 8 bytes past a boundary
          if (LM_IN_BOUNDS(start - base, a.total_bytes - 7, a.err))
            *reinterpret_cast<float2 *>(dst + (start - a0)) = *reinterpret_cast<const float2 *>(start);
          lo += 16;
          generic_written |= 1u << s;
        }
        if (hi > limit) {
          // the last tile of a tensor that ends 8 bytes past a boundary
          if (LM_IN_BOUNDS(end - 8 - base, a.total_bytes - 7, a.err))
            *reinterpret_cast<float2 *>(dst + (end - 8 - a0)) = *reinterpret_cast<const float2 *>(end - 8);
          hi = end & ~15ull;
          generic_written |= 1u << s;
        }
        uint32_t bytes = hi > lo ? static_cast<uint32_t>(hi - lo) : 0u;
        // (checked builds) the copied range lies inside the tensor; if not,
        // nothing is copied and the error word says so
        if (bytes > 0 && !(LM_IN_BOUNDS(lo - base, a.total_bytes, a.err) &&
                           LM_IN_BOUNDS(hi - 1 - base, a.total_bytes, a.err)))
          bytes = 0;
        const int d = static_cast<int>(k & (kSlots - 1));
        aux.desc_frame0[d] = it.first_frame(a);
        aux.desc_nf[d] = it.frames(a);
        aux.desc_head[d] = static_cast<int32_t>(start - a0);
        mbar_arrive_expect_tx(&aux.full[s], bytes);
        if (bytes > 0) bulk_g2s(dst + (lo - a0), reinterpret_cast<const void *>(lo), bytes, &aux.full[s], pol);
        ++issued;
        it.next(a);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      // Every copy issued lands before the CTA may exit: wait for the last
      // phase of each stage in use (immediate unless the CTA is aborting).
      for (int64_t k = issued > S ? issued - S : 0; k < issued; ++k)
        mbar_wait_drain(&aux.full[k % S], static_cast<uint32_t>((k / S) & 1), a.err);
    }
    return;
  }

  if (warp == kPublisherWarp) {
    // ---- publisher: one plain store per tile of the tile's maximum key ----
    if (lane != 0) return;
    volatile uint32_t *tkey = aux.tmax_key;
    for (int64_t k = 0; k < my_tiles; ++k) {
      const int r = static_cast<int>(k & (kSlots - 1));
      if (!mbar_wait(&aux.tmax_bar[r], static_cast<uint32_t>((k / kSlots) & 1), abort_flag, a.err)) return;
      const uint32_t key = tkey[r];
      tkey[r] = 0u;
      const int64_t tile = blockIdx.x + k * G;
      if (tile != a.withhold_tile && LM_IN_BOUNDS(tile, a.n_tiles, a.err)) st_relaxed_gpu(a.tile_key + tile, key);
      mbar_arrive(&aux.pub_bar[r]);
    }
    return;
  }

  if (warp == kResolverWarp) {
    // ---- resolver: clip maxima over a sliding window of steps ----
    // Step q is served (its clip maximum handed to the consumers) once this
    // CTA has published step q -- which also keeps the resolver less than
    // kSlots steps ahead of the consumers, so no handshake slot is reused
    // before it was read -- and every tile slot of its clip is nonzero.  Each
    // pass polls the first kResolveSteps unserved steps that this CTA has
    // published, with the loads of all of them in flight together (16-byte
    // relaxed loads by the whole warp), so a step is served about one L2
    // round trip after its clip completes, in any order.
    if (!kResident) return;
    constexpr int M = kResolveSteps;
    const int tpc = a.tiles_per_clip;
    TileIter it0;  // at step q_next
    it0.init(blockIdx.x, tpc);
    int64_t q_next = 0;  // lowest step not yet served
    unsigned done = 0;   // bit w: step q_next + w already served
    uint64_t t0 = 0;
    // Polling step q starts once this CTA has published step q + span: the
    // clip of q ends by that step on every CTA, and the CTAs run nearly in
    // step, so earlier polls would mostly fail and only take issue slots
    // from the consumers.
    auto gate = [&](int64_t q) { return min(q + a.span, my_tiles - 1); };
    while (q_next < my_tiles) {
      const int64_t g0 = gate(q_next);
      // Every lane waits; the vote keeps the warp together for the
      // warp-wide operations below when some lane's wait gave up.
      if (!__all_sync(0xffffffffu, mbar_wait(&aux.pub_bar[g0 & (kSlots - 1)],
                                             static_cast<uint32_t>((g0 / kSlots) & 1), abort_flag, a.err)))
        return;
      // Lane w < M tests the gate of step q_next + w; the publisher goes in
      // step order, so the open steps are a prefix.  A gate is fewer than
      // kSlots steps past a published step, so its parity is unambiguous.
      int open = 0;
      if (lane < M) {
        const int64_t q = q_next + lane;
        if (q < my_tiles) {
          const int64_t g = gate(q);
          open = lane == 0 || mbar_test_wait(smem_u32(&aux.pub_bar[g & (kSlots - 1)]),
                                             static_cast<uint32_t>((g / kSlots) & 1));
        }
      }
      const unsigned openmask = __ballot_sync(0xffffffffu, open);
      const unsigned poll = ((1u << (__ffs(~openmask) - 1)) - 1u) & ~done;
      const uint32_t *base[M];
      int head[M];
      TileIter it = it0;
#pragma unroll
      for (int w = 0; w < M; ++w) {
        const uint32_t *slots = a.tile_key + it.b * tpc;
        head[w] = static_cast<int>((reinterpret_cast<uintptr_t>(slots) & 15) >> 2);  // slots before the clip's first
        base[w] = slots - head[w];                                                   // 16-byte aligned
        it.next(a);
      }
      uint32_t m[M];
      bool ok[M];
#pragma unroll
      for (int w = 0; w < M; ++w) {
        m[w] = 0;
        ok[w] = true;
        if ((poll >> w) & 1u) {
          const int nvec = (head[w] + tpc + 3) >> 2;
          for (int v = lane; v < nvec; v += 32) {
            // (checked builds) the 16-byte group lies inside the slots, the
            // 16-byte header before them or the 16 bytes of slack after
            const uint4 x = LM_IN_BOUNDS((base[w] + 4 * v) - a.tile_key + 4, a.n_tiles + 5, a.err)
                                ? ld_relaxed_gpu_v4(base[w] + 4 * v)
                                : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int slot = 4 * v + j - head[w];
              if (slot >= 0 && slot < tpc) {
                ok[w] = ok[w] && (e[j] != 0u);
                m[w] = max(m[w], e[j]);
              }
            }
          }
        }
      }
      unsigned served = 0;
#pragma unroll
      for (int w = 0; w < M; ++w) {
        if ((poll >> w) & 1u) {
          const bool all = __all_sync(0xffffffffu, ok[w]);
          const uint32_t mx = __reduce_max_sync(0xffffffffu, m[w]);
          if (all) {
            const int64_t q = q_next + w;
            if (lane == 0) {
              aux.hi_val[q & (kSlots - 1)] = ordered_to_float(mx);
              mbar_arrive(&aux.hi_bar[q & (kSlots - 1)]);
            }
            served |= 1u << w;
          }
        }
      }
      done |= served;
      const int adv = __ffs(~done) - 1;  // served prefix
      if (adv > 0) {
        q_next += adv;
        done >>= adv;
        for (int i = 0; i < adv; ++i) it0.next(a);
      }
      if (served) {
        t0 = 0;
        continue;
      }
      int stop = 0;
      if (lane == 0) {
        const uint64_t now = global_timer_ns();
        if (t0 == 0) t0 = now;
        if (!*abort_flag && now - t0 > a.clip_wait_ns) {
          *abort_flag = 1;
          atomicOr(a.err, kErrClipTimeout);
        }
        stop = *abort_flag;
      }
      // give up: the consumers' waits end on the abort flag
      if (__shfl_sync(0xffffffffu, stop, 0)) return;
      __nanosleep(64);
    }
    return;
  }

  // ---------------------------- consumers ----------------------------
  Band band;
  const int maxw = setup_band<CW>(a, aux, band);
  float *ring = reinterpret_cast<float *>(smem + static_cast<size_t>(a.n_stages) * a.stage_stride);
  if (maxw <= 4)
    consume<FPT, 4, kResident, CW>(a, smem, aux, ring, my_tiles, band, lane);
  else if (maxw <= kRegTaps)
    consume<FPT, kRegTaps, kResident, CW>(a, smem, aux, ring, my_tiles, band, lane);
  else
    consume<FPT, 0, kResident, CW>(a, smem, aux, ring, my_tiles, band, lane);
}

// ---- cluster variant (small batches) -----------------------------------------
// One thread-block cluster of a.cluster CTAs per clip; CTA r of clip b takes
// frames [r * frames_per_cta, (r + 1) * frames_per_cta) and keeps their log
// values in its own shared memory.  After the last tile each CTA reduces its
// maximum, the cluster exchanges maxima through distributed shared memory,
// and every CTA writes its slice once, floored and rescaled.  No global
// slots, no cross-CTA polling and no workspace beyond the error word: the
// KBench spec's "clip-resident" design note, with the clip spread over the
// shared memory of one cluster.

// Consumer loop of the cluster variant: thread (n, fg) computes band n of
// its frames of each tile into the output slice; returns the key of its
// largest value (0: none).
template <int FPT, int W>
__device__ __forceinline__ uint32_t consume_slice(const StftArgs &a, unsigned char *smem, SmemAux &aux,
                                                  float *obuf, int ntiles, const Band &c, int lane) {
  volatile int *abort_flag = &aux.abort_flag;
  const int S = a.n_stages;
  const int fstep = a.FG * a.NF;
  const int ostep = a.FG * a.NM;
  const int own = c.fg * a.NM + c.n;
  float lmax = -INFINITY;
  int s = 0;
  uint32_t ph = 0;
  for (int k = 0; k < ntiles; ++k) {
    // a wait that gave up: the CTA is aborting; stop without touching the stage
    if (!__all_sync(0xffffffffu, mbar_wait(&aux.full[s], ph, abort_flag, a.err))) break;
    const int d = k & (kSlots - 1);
    const int nf = aux.desc_nf[d];
    const float2 *fr = reinterpret_cast<const float2 *>(smem + static_cast<size_t>(s) * a.stage_stride +
                                                        aux.desc_head[d]) +
                       (c.st + c.fg * a.NF);
    float *dst = obuf + k * a.TF * a.NM + own;
    if (c.active) {
#pragma unroll
      for (int j = 0; j < FPT; ++j) {
        if (nf == a.TF || c.fg + j * a.FG < nf) {
          float acc;
          if constexpr (W > 0) {
            acc = band_sum<W>(fr + j * fstep, c.wd, c.w2);
          } else {
            acc = band_sum_wide(fr + j * fstep, c.wd, c.w2, c.wrow);
          }
          const float v = fast_log10(fmaxf(acc, 1e-10f));
          lmax = fmaxf(lmax, v);
          dst[j * ostep] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&aux.empty[s]);
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  return lmax == -INFINITY ? 0u : float_to_ordered(lmax);
}

template <int FPT, int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 1) stft_logmel_cluster_kernel(const StftArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  SmemAux &aux = *reinterpret_cast<SmemAux *>(smem + a.aux_offset);
  float *obuf = reinterpret_cast<float *>(smem + a.obuf_offset);
  volatile int *abort_flag = &aux.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = a.n_stages;
  const int64_t b = blockIdx.x / a.cluster;
  const uint32_t rank = cluster_ctarank();
  const int64_t f0 = static_cast<int64_t>(rank) * a.frames_per_cta;
  int64_t nloc = a.F - f0;
  nloc = nloc < 0 ? 0 : (nloc > a.frames_per_cta ? a.frames_per_cta : nloc);
  const int ntiles = static_cast<int>((nloc + a.TF - 1) / a.TF);

  // This launch needs no workspace but its error word, so there is no memset
  // before it: CTA 0 clears the word first thing.  Every CTA of the grid is
  // resident from the start (the host launches this variant only when all
  // clusters fit at once), errors other than a mismatched pack (which CTA 0
  // alone reports) come from waits that ran out after 2 s, so none is set
  // before the clear.  A word shared with other calls is left alone.
  if (a.clear_err && blockIdx.x == 0 && threadIdx.x == 0) *a.err = 0u;
  if (warp == 0) {
    if (lane < S) {
      mbar_init(&aux.full[lane], 1);
      mbar_init(&aux.empty[lane], CW);
    }
    if (lane == 0) {
      aux.max_width = 0;
      aux.abort_flag = 0;
      aux.tmax_key[0] = 0u;
    }
    fence_mbar_init();
  }
  __syncthreads();

  uint32_t key = 0u;
  if (warp == CW) {
    // ------------- producer: bulk copies of the slice's frame tiles -------------
    // (8-byte aligned source: as in the one-CTA-per-SM kernel, a value that
    // the 16-byte aligned copy would take from outside the tensor is copied
    // by hand.)
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint64_t base = reinterpret_cast<uint64_t>(a.stft);
      const uint64_t limit = base + a.total_bytes;
      int s = 0;
      uint32_t ph = 0;
      uint32_t generic_written = 0;
      int issued = 0;
      for (int k = 0; k < ntiles; ++k) {
        if (k >= S && !mbar_wait(&aux.empty[s], ph ^ 1u, abort_flag, a.err)) break;
        const int64_t left = nloc - static_cast<int64_t>(k) * a.TF;
        const int nf = left < a.TF ? static_cast<int>(left) : a.TF;
        const uint64_t start =
            base + static_cast<uint64_t>(b * a.F + f0 + static_cast<int64_t>(k) * a.TF) * a.NF * 8ull;
        const uint64_t end = start + static_cast<uint64_t>(nf) * a.NF * 8ull;
        const uint64_t a0 = start & ~15ull;
        uint64_t lo = a0;
        uint64_t hi = (end + 15ull) & ~15ull;
        unsigned char *dst = smem + static_cast<size_t>(s) * a.stage_stride;
        if ((generic_written >> s) & 1u) {
          fence_proxy_async_smem();
          generic_written &= ~(1u << s);
        }
        if (lo < base) {
          if (LM_IN_BOUNDS(start - base, a.total_bytes - 7, a.err))
            *reinterpret_cast<float2 *>(dst + (start - a0)) = *reinterpret_cast<const float2 *>(start);
          lo += 16;
          generic_written |= 1u << s;
        }
        if (hi > limit) {
          if (LM_IN_BOUNDS(end - 8 - base, a.total_bytes - 7, a.err))
            *reinterpret_cast<float2 *>(dst + (end - 8 - a0)) = *reinterpret_cast<const float2 *>(end - 8);
          hi = end & ~15ull;
          generic_written |= 1u << s;
        }
        uint32_t bytes = hi > lo ? static_cast<uint32_t>(hi - lo) : 0u;
        // (checked builds) the copied range lies inside the tensor; if not,
        // nothing is copied and the error word says so
        if (bytes > 0 && !(LM_IN_BOUNDS(lo - base, a.total_bytes, a.err) &&
                           LM_IN_BOUNDS(hi - 1 - base, a.total_bytes, a.err)))
          bytes = 0;
        const int d = k & (kSlots - 1);
        aux.desc_nf[d] = nf;
        aux.desc_head[d] = static_cast<int32_t>(start - a0);
        mbar_arrive_expect_tx(&aux.full[s], bytes);
        if (bytes > 0) bulk_g2s(dst + (lo - a0), reinterpret_cast<const void *>(lo), bytes, &aux.full[s], pol);
        ++issued;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      for (int k = issued > S ? issued - S : 0; k < issued; ++k)
        mbar_wait_drain(&aux.full[k % S], static_cast<uint32_t>((k / S) & 1), a.err);
    }
  } else {
    // ----------------------------- consumers -----------------------------
    Band band;
    const int maxw = setup_band<CW>(a, aux, band);
    band.wrow = a.filters + static_cast<int64_t>(band.n) * a.NF + band.st;
    if (maxw <= 4)
      key = consume_slice<FPT, 4>(a, smem, aux, obuf, ntiles, band, lane);
    else if (maxw <= kRegTaps)
      key = consume_slice<FPT, kRegTaps>(a, smem, aux, obuf, ntiles, band, lane);
    else
      key = consume_slice<FPT, 0>(a, smem, aux, obuf, ntiles, band, lane);
  }
  // Every thread of every CTA of the cluster reaches both cluster barriers
  // below, whatever happened above: no CTA leaves a peer waiting.
  key = __reduce_max_sync(0xffffffffu, key);
  if (lane == 0) atomicMax(&aux.tmax_key[0], key);
  __syncthreads();  // this CTA's maximum is in aux.tmax_key[0]; the slice is complete
  cluster_sync_all();
  if (warp == 0) {
    uint32_t k = lane < a.cluster ? ld_dsmem_u32(smem_u32(&aux.tmax_key[0]), static_cast<uint32_t>(lane)) : 0u;
    k = __reduce_max_sync(0xffffffffu, k);
    if (lane == 0) aux.hi_val[0] = ordered_to_float(k);
  }
  __syncthreads();
  if (!*abort_flag) {
    // the slice is contiguous in the output: frames f0.. of clip b, NM each
    const float floor_v = aux.hi_val[0] - 8.0f;
    const int64_t n = nloc * a.NM;
    float *o = a.out + (b * a.F + f0) * a.NM;
    const int nthreads = static_cast<int>(blockDim.x);
    if ((reinterpret_cast<uintptr_t>(o) & 15) == 0) {
      const int64_t n4 = n / 4;
      for (int64_t i = threadIdx.x; i < n4; i += nthreads) {
        float4 v = *reinterpret_cast<const float4 *>(obuf + 4 * i);
        v.x = rescale(v.x, floor_v);
        v.y = rescale(v.y, floor_v);
        v.z = rescale(v.z, floor_v);
        v.w = rescale(v.w, floor_v);
        if (LM_IN_BOUNDS((o - a.out) + 4 * i + 3, a.B * a.F * a.NM, a.err)) __stcs(reinterpret_cast<float4 *>(o) + i, v);
      }
      for (int64_t i = 4 * n4 + threadIdx.x; i < n; i += nthreads)
        if (LM_IN_BOUNDS((o - a.out) + i, a.B * a.F * a.NM, a.err)) __stcs(o + i, rescale(obuf[i], floor_v));
    } else {
      for (int64_t i = threadIdx.x; i < n; i += nthreads)
        if (LM_IN_BOUNDS((o - a.out) + i, a.B * a.F * a.NM, a.err)) __stcs(o + i, rescale(obuf[i], floor_v));
    }
  }
  cluster_sync_all();  // the peers have read this CTA's maximum
}

// Two-pass epilogue for one slice of one clip: the clip maximum is the
// maximum of its tile slots; out = (max(out, hi - 8) + 4) / 4 in place.
__global__ void __launch_bounds__(256) logmel_clamp_kernel(float *out, const uint32_t *tile_key, int64_t B,
                                                           int64_t per_clip, int32_t tiles_per_clip, int vec4) {
  __shared__ uint32_t warp_keys[8];
  // Launched as a programmatic dependent of the kernel that wrote the
  // values: wait until that grid has finished and its writes are visible
  // (a no-op for an ordinary launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int U = 8;  // 16-byte loads in flight per thread before any store
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
    float *o = out + b * per_clip;
    float4 *o4 = reinterpret_cast<float4 *>(o);
    const int64_t n4 = vec4 ? per_clip / 4 : 0;
    // The first values' loads do not depend on the clip maximum: they are
    // issued before the tile slots are reduced, so the two L2 round trips
    // overlap.
    int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * stride < n4) v[u] = o4[i0 + u * stride];
    uint32_t m = 0;
    for (int i = threadIdx.x; i < tiles_per_clip; i += blockDim.x) m = max(m, tile_key[b * tiles_per_clip + i]);
    m = __reduce_max_sync(0xffffffffu, m);
    if ((threadIdx.x & 31) == 0) warp_keys[threadIdx.x >> 5] = m;
    __syncthreads();
    m = warp_keys[0];
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = max(m, warp_keys[w]);
    __syncthreads();
    const float floor_v = ordered_to_float(m) - 8.0f;
    if (vec4) {
      // In place: every load of a pass before any of its stores, so that
      // one-at-a-time does not wait an L2 round trip per vector.
      while (i0 < n4) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (i0 + u * stride < n4) {
            float4 w = v[u];
            w.x = rescale(w.x, floor_v);
            w.y = rescale(w.y, floor_v);
            w.z = rescale(w.z, floor_v);
            w.w = rescale(w.w, floor_v);
            o4[i0 + u * stride] = w;
          }
        }
        i0 += U * stride;
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (i0 + u * stride < n4) v[u] = o4[i0 + u * stride];
      }
    } else {
      for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < per_clip; i += stride)
        o[i] = rescale(o[i], floor_v);
    }
  }
}

// Packs the dense [NM, NF] filter matrix: a warp per row finds the first
// and last nonzero bin with ballots (as the kernel's own sweep defines the
// support) and stores {first, width} and the first kRegTaps weights from
// `first` (zero past the width).  The header is zeroed before launch; block 0
// writes the shape and the magic, and every row folds its width into the
// widest.
__global__ void __launch_bounds__(256) mel_filters_pack_kernel(const float *filters, int32_t NF, int32_t NM,
                                                               int32_t *packed) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    packed[0] = PackLayout::kMagic;
    packed[1] = NF;
    packed[2] = NM;
  }
  if (n >= NM) return;
  const float *row = filters + static_cast<int64_t>(n) * NF;
  int first = INT_MAX, last = -1;
  for (int k0 = 0; k0 < NF; k0 += 32) {
    const int k = k0 + lane;
    const unsigned m = __ballot_sync(0xffffffffu, k < NF && row[k] != 0.f);
    if (m) {
      if (first == INT_MAX) first = k0 + __ffs(m) - 1;
      last = k0 + 31 - __clz(m);
    }
  }
  const int st = last >= 0 ? first : 0;
  const int wd = last >= 0 ? last - first + 1 : 0;
  int2 *sw = reinterpret_cast<int2 *>(reinterpret_cast<char *>(packed) + PackLayout::sw_offset());
  float *taps = reinterpret_cast<float *>(reinterpret_cast<char *>(packed) + PackLayout::taps_offset(NM));
  if (lane == 0) {
    sw[n] = make_int2(st, wd);
    atomicMax(&packed[3], wd);
  }
  if (lane < kRegTaps) taps[static_cast<int64_t>(n) * kRegTaps + lane] = lane < wd ? row[st + lane] : 0.f;
}

using KernelFn = void (*)(StftArgs);

template <int FPT, int CW>
KernelFn pick_variant(bool resident) {
  return resident ? stft_logmel_kernel<FPT, true, CW> : stft_logmel_kernel<FPT, false, CW>;
}

template <int CW>
KernelFn pick_fpt(int fpt, bool resident) {
  switch (fpt) {
    case 1: return pick_variant<1, CW>(resident);
    case 2: return pick_variant<2, CW>(resident);
    case 4: return pick_variant<4, CW>(resident);
    case 6: return pick_variant<6, CW>(resident);
    default: return pick_variant<8, CW>(resident);
  }
}

KernelFn pick_kernel(int cw, int fpt, bool resident) {
  if (cw == 20) return fpt == 5 ? pick_variant<5, 20>(resident) : pick_variant<4, 20>(resident);
  return pick_fpt<16>(fpt, resident);
}

template <int CW>
KernelFn pick_cluster_fpt(int fpt) {
  switch (fpt) {
    case 1: return stft_logmel_cluster_kernel<1, CW>;
    case 2: return stft_logmel_cluster_kernel<2, CW>;
    case 4: return stft_logmel_cluster_kernel<4, CW>;
    case 6: return stft_logmel_cluster_kernel<6, CW>;
    default: return stft_logmel_cluster_kernel<8, CW>;
  }
}

KernelFn pick_cluster_kernel(int cw, int fpt) {
  if (cw == 20) return fpt == 5 ? stft_logmel_cluster_kernel<5, 20> : stft_logmel_cluster_kernel<4, 20>;
  return pick_cluster_fpt<16>(fpt);
}

struct TilePlan {
  int CW, FG, FPT, TF, S;
  uint32_t stride;
  int64_t ring_bytes;
  uint32_t aux_offset;
  size_t smem;
};

// Consumer warps CW, frame groups FG of NM threads, FPT frames per thread,
// with a stage of at most about kStageTargetBytes.  Sixteen consumer warps,
// or twenty where NM divides 640 and that gives a tile at least as tall with
// 4 or 5 frames per thread (NM = 128: 5 x 5 = 25 frames against 4 x 6).  The
// loop is latency-bound: twenty warps were 3% faster at NM = 128, and halving
// the warps (with twice the frames per thread) was 37% slower.  A function
// of the shape alone: the workspace size depends on it.
void tile_height(int NF, int NM, int *CW, int *FG, int *FPT) {
  *CW = 16;
  const int fg_max = (*CW * 32) / NM;
  const int64_t frame_bytes = static_cast<int64_t>(NF) * 8;
  *FG = fg_max;
  // LOGMEL_FPB=1|2|4|6|8 forces the frames per consumer thread (sixteen
  // consumer warps; A/B only): the workspace size follows it, and a stage
  // that leaves no room for two of them in shared memory is refused later.
  const int forced = std::atoi(env_or("LOGMEL_FPB", "0"));
  if (fg_max >= 1 && (forced == 1 || forced == 2 || forced == 4 || forced == 6 || forced == 8)) {
    *FPT = forced;
    return;
  }
  *FPT = 0;
  for (int fpt : {8, 6, 4, 2, 1}) {
    if (static_cast<int64_t>(fg_max) * fpt * frame_bytes <= kStageTargetBytes) {
      *FPT = fpt;
      break;
    }
  }
  if (*FPT == 0) {
    *FPT = 1;
    *FG = std::max<int>(1, std::min<int64_t>(fg_max, kStageTargetBytes / frame_bytes));
    return;
  }
  if (NM <= 640 && 640 % NM == 0) {
    const int fg20 = 640 / NM;
    for (int fpt : {5, 4}) {
      if (static_cast<int64_t>(fg20) * fpt * frame_bytes <= kStageTargetBytes && fg20 * fpt >= *FG * *FPT) {
        *CW = 20;
        *FG = fg20;
        *FPT = fpt;
        return;
      }
    }
  }
}

// Shared memory: S stages | (resident) kLag+1 output slots of TF x NM | SmemAux.
TilePlan plan_tiles(int NF, int NM, int max_smem, bool resident) {
  TilePlan p{};
  tile_height(NF, NM, &p.CW, &p.FG, &p.FPT);
  p.TF = p.FG * p.FPT;
  const int64_t stage = static_cast<int64_t>(p.TF) * NF * 8 + 16;
  p.stride = static_cast<uint32_t>((stage + 127) / 128 * 128);
  p.ring_bytes = resident ? static_cast<int64_t>(kLag + 1) * p.TF * NM * 4 : 0;
  p.ring_bytes = (p.ring_bytes + 127) / 128 * 128;
  const int64_t budget = static_cast<int64_t>(std::min(max_smem, 227 * 1024)) -
                         static_cast<int64_t>(sizeof(SmemAux)) - p.ring_bytes - 128;
  p.S = budget > 0 ? static_cast<int>(std::min<int64_t>(kMaxStages, budget / p.stride)) : 0;
  p.aux_offset = static_cast<uint32_t>(static_cast<int64_t>(p.S) * p.stride + p.ring_bytes);
  p.smem = static_cast<size_t>(p.aux_offset) + sizeof(SmemAux);
  return p;
}

struct StftLaunch {
  TilePlan tp;
  int64_t tpc = 0;   // tiles per clip
  int64_t grid = 0;  // CTAs
  int64_t span = 0;  // steps a clip can reach past any of its steps on one CTA
  int L = 0;         // lag in steps (resident mode)
  bool resident = false;
  int cluster = 0;   // cluster variant: CTAs per clip (0: not used)
  int64_t frames_per_cta = 0;
  uint32_t obuf_offset = 0;
  KernelFn kern = nullptr;
};

// The cluster variant with C CTAs per clip: tile shape as the one-CTA-per-SM
// kernel, shared memory = S stages | the output slice (ceil(F / C) frames x
// NM f32) | SmemAux.  Fails (returns false) when two stages do not fit
// beside the slice or no cluster of C such CTAs fits the device; sets
// *max_clusters to the clusters the device runs at once.
bool plan_cluster(int64_t F, int32_t NF, int32_t NM, int C, const DeviceInfo &dev, StftLaunch *ln,
                  int *max_clusters) {
  int CW = 0, FG = 0, FPT = 0;
  tile_height(NF, NM, &CW, &FG, &FPT);
  TilePlan p{};
  p.CW = CW;
  p.FG = FG;
  p.FPT = FPT;
  p.TF = FG * FPT;
  const int64_t fc = (F + C - 1) / C;
  const int64_t obuf = (fc * NM * 4 + 127) / 128 * 128;
  const int64_t stage = static_cast<int64_t>(p.TF) * NF * 8 + 16;
  p.stride = static_cast<uint32_t>((stage + 127) / 128 * 128);
  const int64_t budget = static_cast<int64_t>(std::min(dev.max_smem_optin, 227 * 1024)) -
                         static_cast<int64_t>(sizeof(SmemAux)) - obuf - 128;
  p.S = budget > 0 ? static_cast<int>(std::min<int64_t>(kMaxStages, budget / p.stride)) : 0;
  if (p.S < 2) return false;
  p.ring_bytes = 0;
  p.aux_offset = static_cast<uint32_t>(p.S * static_cast<int64_t>(p.stride) + obuf);
  p.smem = static_cast<size_t>(p.aux_offset) + sizeof(SmemAux);
  KernelFn kern = pick_cluster_kernel(CW, FPT);
  if (ensure_smem_attribute(reinterpret_cast<const void *>(kern), static_cast<int>(p.smem)) != LM_OK) return false;
  if (C > 8 && cudaFuncSetAttribute(reinterpret_cast<const void *>(kern),
                                    cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  // Clusters the device runs at once, queried once per (device, kernel,
  // shared memory, cluster size): the query costs host time on every call of
  // exactly the small batches this variant serves.
  static std::mutex mu;
  static std::vector<std::array<int64_t, 5>> cache;  // device, kernel, smem, C -> clusters (or -1)
  int n = 0;
  bool cached = false;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const auto &e : cache)
      if (e[0] == dev.device && e[1] == reinterpret_cast<int64_t>(kern) && e[2] == static_cast<int64_t>(p.smem) &&
          e[3] == C) {
        n = static_cast<int>(e[4]);
        cached = true;
      }
  }
  if (!cached) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    cfg.blockDim = dim3(static_cast<unsigned>((CW + 1) * 32));
    cfg.dynamicSmemBytes = p.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = -1;
    }
    std::lock_guard<std::mutex> lk(mu);
    cache.push_back({dev.device, reinterpret_cast<int64_t>(kern), static_cast<int64_t>(p.smem), C, n});
  }
  if (n < 1) return false;
  *max_clusters = n;
  ln->tp = p;
  ln->cluster = C;
  ln->frames_per_cta = fc;
  ln->obuf_offset = static_cast<uint32_t>(p.S * static_cast<int64_t>(p.stride));
  ln->kern = kern;
  ln->tpc = (F + p.TF - 1) / p.TF;
  ln->resident = false;
  ln->L = 0;
  return true;
}

// Chooses tile shape, ring depth, variant and grid for a problem shape.
lm_status plan_launch(int64_t B, int64_t F, int32_t NF, int32_t NM, StftLaunch *ln, bool allow_cluster = true) {
  DeviceInfo dev;
  if (lm_status st = current_device_info(&dev); st != LM_OK) return st;
  int CW = 0, FG = 0, FPT = 0;
  tile_height(NF, NM, &CW, &FG, &FPT);
  const int TF = FG * FPT;
  ln->tpc = (F + TF - 1) / TF;
  if (ln->tpc > INT32_MAX / 2) return LM_ERR_UNSUPPORTED;
  const int64_t n_tiles = B * ln->tpc;
  ln->grid = std::min<int64_t>(n_tiles, dev.sm_count);
  // On the static round-robin schedule the tiles of the clip of step q lie
  // at steps <= q + span.  Resident mode needs span < kLag: the values of
  // step q are written at step q + kLag, after every tile of its clip.
  ln->span = (ln->grid + ln->tpc - 2) / ln->grid;
  const char *variant = env_or("LOGMEL_K1_VARIANT", "auto");
  const bool force_two = std::strcmp(variant, "twopass") == 0;
  const bool force_res = std::strcmp(variant, "resident") == 0;
  const bool force_cluster = std::strcmp(variant, "cluster") == 0;
  if (std::strcmp(variant, "nocluster") == 0) allow_cluster = false;
  // Small batches: one cluster per clip, when the device runs every clip's
  // cluster at once -- the largest cluster (16 CTAs down to 8) for which it
  // does (clusters are placed within a GPC; GB300 runs only seven of 16 CTAs
  // with one CTA per SM) -- and the clusters keep at least as many SMs
  // streaming as the one-CTA-per-SM kernel would (capped at 70% of them).
  // Measured on 8 x 3000 x 201 -> 80 style batches, L2 flushed: B = 7, 112
  // CTAs: 18.8 us against 20.6; B = 8, 96 CTAs: 20.7 against 21.0; B = 1,
  // 16 CTAs against 125: 16.6 against 13.8.
  if (allow_cluster && (force_cluster || (!force_two && !force_res))) {
    const int64_t want = std::min<int64_t>(n_tiles, (7 * static_cast<int64_t>(dev.sm_count)) / 10);
    for (int C = 16; C >= 8; --C) {
      int n = 0;
      StftLaunch c = *ln;
      if (plan_cluster(F, NF, NM, C, dev, &c, &n) && (force_cluster || (B <= n && B * C >= want))) {
        *ln = c;
        ln->grid = B * C;
        return LM_OK;
      }
    }
    if (force_cluster) return LM_ERR_UNSUPPORTED;
  }
  // Consumers wait for step q's clip maximum after computing step q + kLag,
  // so every tile of that clip (steps <= q + span on every CTA) is computed
  // by then if span < kLag; the resolver serves q as soon as they are all
  // published.  One step of slack is kept for the hand-off itself.
  ln->resident = !force_two && ln->span + 1 <= kLag;
  if (ln->resident) {
    ln->tp = plan_tiles(NF, NM, dev.max_smem_optin, true);
    if (ln->tp.S < 2) ln->resident = false;  // the output ring does not fit beside two stages
  }
  if (force_res && !ln->resident) return LM_ERR_UNSUPPORTED;
  if (!ln->resident) ln->tp = plan_tiles(NF, NM, dev.max_smem_optin, false);
  if (ln->tp.S < 2) return LM_ERR_UNSUPPORTED;
  ln->L = ln->resident ? kLag : 0;
  ln->kern = pick_kernel(ln->tp.CW, ln->tp.FPT, ln->resident);
  if (lm_status st = ensure_smem_attribute(reinterpret_cast<const void *>(ln->kern), static_cast<int>(ln->tp.smem));
      st != LM_OK)
    return st;
  int per_sm = 0;
  LM_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ln->kern, threads_for(ln->tp.CW), ln->tp.smem));
  if (per_sm < 1) return LM_ERR_UNSUPPORTED;
  return LM_OK;
}

// Workspace layout: header | tile_key[B * tiles_per_clip].
size_t tile_key_offset() { return kWorkspaceHeaderBytes; }

}  // namespace

size_t stft_workspace_bytes(int64_t B, int64_t F, int32_t NF, int32_t NM) {
  if (B < 1 || F < 1 || NF < 1 || NM < 1 || NF > kMaxBins || NM > kMaxBands) return kWorkspaceHeaderBytes;
  int CW = 0, FG = 0, FPT = 0;
  tile_height(NF, NM, &CW, &FG, &FPT);
  const int64_t TF = static_cast<int64_t>(FG) * FPT;
  const int64_t tpc = (F + TF - 1) / TF;
  // + 16: the resolver reads slots in aligned 16-byte groups and may touch
  // up to three slots past the last clip.
  return (tile_key_offset() + static_cast<size_t>(B * tpc) * sizeof(uint32_t) + 16 + 255) / 256 * 256;
}

lm_status stft_logmel_run(const void *stft, const float *filters, float *out, int64_t B, int64_t F,
                          int32_t NF, int32_t NM, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream, const void *packed, uint32_t *err_word, const StftFault *fault) {
  if (B < 0 || F < 0 || NF < 1 || NM < 1) return LM_ERR_INVALID_ARG;
  if (NF > kMaxBins || NM > kMaxBands) return LM_ERR_UNSUPPORTED;
  if (B == 0 || F == 0) return LM_OK;
  if (!stft || !filters || !out || !workspace) return workspace ? LM_ERR_INVALID_ARG : LM_ERR_WORKSPACE;
  if (F > (int64_t{1} << 40) || B > (int64_t{1} << 40) || (B * F) > (int64_t{1} << 50) / NF)
    return LM_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(stft) & 7) || (reinterpret_cast<uintptr_t>(filters) & 3) ||
      (reinterpret_cast<uintptr_t>(out) & 3) || (reinterpret_cast<uintptr_t>(workspace) & 3))
    return LM_ERR_MISALIGNED;
  if (packed && (reinterpret_cast<uintptr_t>(packed) & 15)) return LM_ERR_MISALIGNED;
  const size_t ws_needed = stft_workspace_bytes(B, F, NF, NM);
  if (workspace_bytes < ws_needed) return LM_ERR_WORKSPACE;
  {  // the output may not overlap either input
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + static_cast<uintptr_t>(B * F * NM) * 4;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(stft), s1 = s0 + static_cast<uintptr_t>(B * F * NF) * 8;
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(filters), w1 = w0 + static_cast<uintptr_t>(NM) * NF * 4;
    if ((o0 < s1 && s0 < o1) || (o0 < w1 && w0 < o1)) return LM_ERR_INVALID_ARG;
  }

  StftLaunch ln;
  // (fault injection exercises the cross-CTA waits of the one-CTA-per-SM kernel)
  if (lm_status st = plan_launch(B, F, NF, NM, &ln, fault == nullptr); st != LM_OK) return st;
  const TilePlan &tp = ln.tp;

  StftArgs a{};
  a.stft = static_cast<const float2 *>(stft);
  a.filters = filters;
  a.out = out;
  a.err = err_word ? err_word : static_cast<uint32_t *>(workspace);
  a.tile_key = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + tile_key_offset());
  a.B = B;
  a.F = F;
  a.NF = NF;
  a.NM = NM;
  a.FG = tp.FG;
  a.TF = tp.TF;
  a.tiles_per_clip = static_cast<int32_t>(ln.tpc);
  a.span = static_cast<int32_t>(ln.span);
  a.n_tiles = B * ln.tpc;
  a.n_stages = tp.S;
  a.stage_stride = tp.stride;
  a.aux_offset = tp.aux_offset;
  a.total_bytes = static_cast<uint64_t>(B) * static_cast<uint64_t>(F) * static_cast<uint64_t>(NF) * 8ull;
  a.grid_q = ln.grid / ln.tpc;
  a.grid_r = static_cast<int32_t>(ln.grid % ln.tpc);
  a.packed = static_cast<const int32_t *>(packed);
  a.clip_wait_ns = fault ? fault->clip_wait_ns : kWaitTimeoutNs;
  a.withhold_tile = fault ? fault->withhold_tile : -1;
  a.cluster = ln.cluster;
  a.frames_per_cta = static_cast<int32_t>(ln.frames_per_cta);
  a.obuf_offset = ln.obuf_offset;
  a.clear_err = err_word == nullptr;

  // The workspace (error word and tile slots) starts zeroed; the cluster
  // variant uses only the error word and clears it itself.
  if (ln.cluster == 0) LM_CUDA_TRY(cudaMemsetAsync(workspace, 0, ws_needed, stream));

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(ln.grid));
  cfg.blockDim = dim3(threads_for(tp.CW));
  cfg.dynamicSmemBytes = tp.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ln.resident ? 1 : 0;
  if (ln.cluster > 0) {
    cfg.blockDim = dim3(static_cast<unsigned>((tp.CW + 1) * 32));
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(ln.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  }
  LM_CUDA_TRY(cudaLaunchKernelEx(&cfg, ln.kern, a));
  if (ln.cluster > 0) return LM_OK;

  if (!ln.resident) return launch_clip_clamp(out, a.tile_key, B, F * NM, a.tiles_per_clip, stream);
  return LM_OK;
}

lm_status launch_clip_clamp(float *out, const uint32_t *tile_key, int64_t B, int64_t per_clip,
                            int32_t tiles_per_clip, cudaStream_t stream) {
  const int vec4 = (per_clip % 4 == 0) && ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
  const int64_t work = vec4 ? per_clip / 4 : per_clip;
  DeviceInfo dev;
  if (lm_status st = current_device_info(&dev); st != LM_OK) return st;
  // About four resident blocks per SM in all: every block first reduces its
  // clip's tile slots, so one block per 256 items would repeat that
  // reduction thousands of times for a few bytes of work each.
  const int64_t gy64 = std::min<int64_t>(B, 65535);
  const int64_t per_clip_blocks = (4 * static_cast<int64_t>(dev.sm_count) + gy64 - 1) / gy64;
  const unsigned gx = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, per_clip_blocks)));
  const unsigned gy = static_cast<unsigned>(gy64);
  // Programmatic dependent launch: the epilogue's blocks are staged while
  // the previous kernel drains and start the moment it completes.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(gx, gy);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LM_CUDA_TRY(cudaLaunchKernelEx(&cfg, logmel_clamp_kernel, out, tile_key, B, per_clip, tiles_per_clip, vec4));
  return LM_OK;
}

lm_status stft_describe(int64_t B, int64_t F, int32_t NF, int32_t NM, lm_stft_launch_info *info) {
  if (!info || B < 1 || F < 1 || NF < 1 || NM < 1) return LM_ERR_INVALID_ARG;
  if (NF > kMaxBins || NM > kMaxBands) return LM_ERR_UNSUPPORTED;
  StftLaunch ln;
  if (lm_status st = plan_launch(B, F, NF, NM, &ln); st != LM_OK) return st;
  info->resident = ln.resident ? 1 : 0;
  info->kernels = (ln.resident || ln.cluster > 0) ? 1 : 2;
  info->cluster = ln.cluster;
  info->grid = static_cast<int32_t>(ln.grid);
  info->frames_per_tile = ln.tp.TF;
  info->stages = ln.tp.S;
  info->lag = ln.L;
  info->smem_bytes = static_cast<int64_t>(ln.tp.smem);
  return LM_OK;
}

}  // namespace lm

extern "C" lm_status lm_log_mel_from_stft_workspace_size(int64_t B, int64_t F, int32_t NF, int32_t NM,
                                                         size_t *bytes) {
  if (!bytes || B < 0 || F < 0 || NF < 1 || NM < 1) return LM_ERR_INVALID_ARG;
  if (NF > 8193 || NM > 512) return LM_ERR_UNSUPPORTED;
  *bytes = lm::stft_workspace_bytes(B, F, NF, NM);
  return LM_OK;
}

extern "C" lm_status lm_log_mel_from_stft(const void *stft, const float *mel_filters, float *out, int64_t B,
                                          int64_t F, int32_t NF, int32_t NM, void *workspace,
                                          size_t workspace_bytes, lm_stream_t stream) {
  return lm::stft_logmel_run(stft, mel_filters, out, B, F, NF, NM, workspace, workspace_bytes,
                             reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" lm_status lm_debug_log_mel_from_stft_withhold(const void *stft, const float *mel_filters, float *out,
                                                         int64_t B, int64_t F, int32_t NF, int32_t NM,
                                                         void *workspace, size_t workspace_bytes,
                                                         int64_t withheld_tile, uint64_t clip_wait_ns,
                                                         lm_stream_t stream) {
  if (withheld_tile < 0 || clip_wait_ns < 100000ull || clip_wait_ns > lm::kWaitTimeoutNs) return LM_ERR_INVALID_ARG;
  const lm::StftFault fault{clip_wait_ns, withheld_tile};
  return lm::stft_logmel_run(stft, mel_filters, out, B, F, NF, NM, workspace, workspace_bytes,
                             reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, &fault);
}

extern "C" lm_status lm_log_mel_from_stft_describe(int64_t B, int64_t F, int32_t NF, int32_t NM,
                                                   lm_stft_launch_info *info) {
  return lm::stft_describe(B, F, NF, NM, info);
}

// ---- allocation-free variant -------------------------------------------------
// Scratch for lm_log_mel_from_stft_noalloc: one fixed array in device memory,
// present on every GPU that loads this library until the process exits.  Host
// code may not pass `g_noalloc_scratch` itself to a kernel (in host code the
// name is a host-side stand-in, not a device address); its device address is
// looked up once per device below.  The first LM_NOALLOC_SCRATCH_BYTES - 256
// bytes serve as the call's workspace and are cleared by every call; the
// last 256 bytes hold a sticky device error word that no call clears.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LM_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kNoallocMaxDevices = 64;
constexpr size_t kNoallocWorkspaceBytes = LM_NOALLOC_SCRATCH_BYTES - 256;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kNoallocMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).  The cache outlives a
// cudaDeviceReset, after which the address is stale: the entry points that
// use it document that.
lm_status noalloc_scratch(void **scratch) {
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) return lm::cuda_fail(e);
  if (dev < 0 || dev >= kNoallocMaxDevices) return LM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void *p = nullptr;
    if (cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch); e != cudaSuccess) return lm::cuda_fail(e);
    g_noalloc_addr[dev] = p;
  }
  *scratch = g_noalloc_addr[dev];
  return LM_OK;
}
}  // namespace

extern "C" lm_status lm_log_mel_from_stft_noalloc(const void *stft, const float *mel_filters, float *out,
                                                  int64_t B, int64_t F, int32_t NF, int32_t NM,
                                                  lm_stream_t stream) {
  if (B < 0 || F < 0 || NF < 1 || NM < 1) return LM_ERR_INVALID_ARG;
  if (NF > 8193 || NM > 512) return LM_ERR_UNSUPPORTED;
  if (B == 0 || F == 0) return LM_OK;
  if (lm::stft_workspace_bytes(B, F, NF, NM) > kNoallocWorkspaceBytes) return LM_ERR_WORKSPACE;
  void *scratch = nullptr;
  if (lm_status st = noalloc_scratch(&scratch); st != LM_OK) return st;
  uint32_t *sticky_err = reinterpret_cast<uint32_t *>(static_cast<char *>(scratch) + kNoallocWorkspaceBytes);
  // stft_logmel_run clears the workspace part it uses before launching; the
  // kernel's error bits go to the sticky word past it.
  return lm::stft_logmel_run(stft, mel_filters, out, B, F, NF, NM, scratch, kNoallocWorkspaceBytes,
                             reinterpret_cast<cudaStream_t>(stream), nullptr, sticky_err);
}

extern "C" lm_status lm_log_mel_from_stft_noalloc_error(uint32_t *device_error, int32_t clear, lm_stream_t stream) {
  if (!device_error) return LM_ERR_INVALID_ARG;
  *device_error = 0;
  void *scratch = nullptr;
  if (lm_status st = noalloc_scratch(&scratch); st != LM_OK) return st;
  uint32_t *sticky_err = reinterpret_cast<uint32_t *>(static_cast<char *>(scratch) + kNoallocWorkspaceBytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  LM_CUDA_TRY(cudaMemcpyAsync(&v, sticky_err, sizeof(v), cudaMemcpyDeviceToHost, s));
  if (clear) LM_CUDA_TRY(cudaMemsetAsync(sticky_err, 0, sizeof(uint32_t), s));
  LM_CUDA_TRY(cudaStreamSynchronize(s));
  *device_error = v;
  return v ? LM_ERR_DEVICE_FAULT : LM_OK;
}

extern "C" lm_status lm_mel_filters_pack_size(int32_t NF, int32_t NM, size_t *bytes) {
  if (!bytes) return LM_ERR_INVALID_ARG;
  *bytes = 0;
  if (NF < 1 || NM < 1) return LM_ERR_INVALID_ARG;
  if (NF > lm::kMaxBins || NM > lm::kMaxBands) return LM_ERR_UNSUPPORTED;
  *bytes = lm::PackLayout::bytes(NM);
  return LM_OK;
}

extern "C" lm_status lm_mel_filters_pack(const float *mel_filters, int32_t NF, int32_t NM, void *packed,
                                         size_t packed_bytes, lm_stream_t stream) {
  size_t need = 0;
  if (lm_status st = lm_mel_filters_pack_size(NF, NM, &need); st != LM_OK) return st;
  if (!mel_filters || !packed) return LM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(mel_filters) & 3) || (reinterpret_cast<uintptr_t>(packed) & 15))
    return LM_ERR_MISALIGNED;
  if (packed_bytes < need) return LM_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LM_CUDA_TRY(cudaMemsetAsync(packed, 0, lm::PackLayout::kHeader, s));
  lm::mel_filters_pack_kernel<<<(NM + 7) / 8, 256, 0, s>>>(mel_filters, NF, NM, static_cast<int32_t *>(packed));
  LM_CUDA_TRY(cudaGetLastError());
  return LM_OK;
}

extern "C" lm_status lm_log_mel_from_stft_packed(const void *stft, const float *mel_filters, const void *packed,
                                                 float *out, int64_t B, int64_t F, int32_t NF, int32_t NM,
                                                 void *workspace, size_t workspace_bytes, lm_stream_t stream) {
  if (!packed) return LM_ERR_INVALID_ARG;
  return lm::stft_logmel_run(stft, mel_filters, out, B, F, NF, NM, workspace, workspace_bytes,
                             reinterpret_cast<cudaStream_t>(stream), packed);
}
