// stft_logmel.cu -- Whisper log-mel spectrogram from a complex STFT.
//
// Computes, per clip b (KBench "audio_mel_spectrogram_fused" spec, per-clip
// definition):
//   mag = re^2 + im^2;  mel = mag . W^T;  ls = log10(max(mel, 1e-10));
//   hi[b] = max over the clip of ls;  out = (max(ls, hi[b] - 8) + 4) / 4.
//
// Design (GB300, HBM-bound: 8 bytes read per bin, 4 written per band):
//
//  * One persistent CTA per SM walks frame tiles in clip order
//    (tile = blockIdx.x + k * gridDim.x).  A tile is TF consecutive frames
//    of one clip and is contiguous in memory.
//  * A producer warp streams tiles into an S-stage shared-memory ring with
//    1-D bulk copies (cp.async.bulk, L2 evict-first), each stage guarded by a
//    full/empty mbarrier pair.  Frames are 8*NF bytes, so a tile may start 8
//    bytes off a 16-byte boundary: the copy starts at the aligned address
//    below and the consumers index from the remainder.
//  * 16 consumer warps compute the tile.  Thread (n, g) owns mel band n and
//    frames g, g+FG, ...; its band's support (first..last nonzero of the
//    dense filter row, found once per CTA) and up to 8 weights sit in
//    registers, so the projection is a handful of FMAs per output fed
//    straight from the staged complex values (power is formed on the fly).
//  * The per-clip maximum: each warp reduces its tile maximum with shuffles
//    and folds it into a shared slot; a monitor warp turns the slot into one
//    atomicMax on the clip's order-preserving u32 key plus a release
//    increment of the clip's tile counter.
//  * Resident mode (default): consumers keep each tile's log values in
//    registers for L more steps.  By then every tile of that clip has been
//    published; the monitor confirms it (acquire load of the counter, bounded
//    wait), hands the clip maximum over through an mbarrier, and the
//    consumers write the final values once.  The output is written to HBM
//    exactly once and never re-read: 1 read of the source + 1 write of the
//    result, the spec's canonical traffic.  Cross-CTA waits need all CTAs
//    resident, so this mode is launched cooperatively.
//  * Two-pass mode (fallback when a clip spans too many steps, or forced by
//    LOGMEL_K1_VARIANT=twopass): consumers write log values and atomicMax
//    the clip key; a second kernel applies the floor and rescale in place.
#include <algorithm>
#include <cfloat>
#include <climits>
#include <cstdlib>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace lm {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kPublisherWarp = kConsumerWarps + 1;
constexpr int kResolverWarp = kConsumerWarps + 2;
constexpr int kThreads = (kConsumerWarps + 3) * 32;
constexpr int kLag = 8;          // resident mode: steps a tile's log values stay in registers
constexpr int kSlots = 32;       // ring of per-step tile-max and clip-max slots (> 2 kLag)
constexpr int kMaxStages = 8;
constexpr int kRegTaps = 8;      // filter taps held in registers per band
constexpr int kMaxBands = 512;   // = kConsumers: one band per consumer thread
constexpr int kMaxBins = 8193;
constexpr int kStageTargetBytes = 48 * 1024;

struct StftArgs {
  const float2 *stft;
  const float *filters;
  float *out;
  uint32_t *err;
  uint32_t *clip_key;   // [B] two-pass mode: order-preserving key of the clip's max log value
  uint32_t *tile_key;   // [n_tiles] resident mode: key of each tile's max, 0 = not yet published
  int64_t B, F;
  int32_t NF, NM;
  int32_t FG;              // frame groups: active consumer threads = FG * NM
  int32_t TF;              // frames per tile (FG * FPT)
  int32_t tiles_per_clip;  // ceil(F / TF)
  int64_t n_tiles;         // B * tiles_per_clip
  int64_t grid_q;          // gridDim.x / tiles_per_clip
  int32_t grid_r;          // gridDim.x % tiles_per_clip
  int32_t n_stages;
  uint32_t stage_stride;   // bytes per stage, multiple of 128
  uint32_t aux_offset;     // shared-memory offset of SmemAux (after the stages and the ring)
  uint64_t total_bytes;    // B * F * NF * 8
};

struct SmemAux {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tmax_bar[kSlots];
  uint64_t hi_bar[kSlots];
  uint32_t tmax_key[kSlots];
  float hi_val[kSlots];
  int32_t band_start[kMaxBands];
  int32_t band_width[kMaxBands];
  int32_t max_width;
  int32_t abort_flag;
  int64_t published;  // resident mode: steps whose tile maximum is in global memory
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

// sum_t w[t] * |fr[t]|^2 over the first `wd` taps, all from registers.
template <int W>
__device__ __forceinline__ float band_sum(const float2 *fr, int wd, const float (&w)[kRegTaps]) {
  float acc = 0.f;
#pragma unroll
  for (int t = 0; t < W; ++t) {
    if (t < wd) {
      const float2 c = fr[t];
      acc = fmaf(w[t], fmaf(c.x, c.x, c.y * c.y), acc);
    }
  }
  return acc;
}

// Bands wider than kRegTaps: the remaining weights come from global memory
// (L1-cached; the filter matrix is read-only).
__device__ __forceinline__ float band_sum_wide(const float2 *fr, int wd, const float (&w)[kRegTaps],
                                               const float *wrow) {
  float acc = band_sum<kRegTaps>(fr, wd, w);
  for (int t = kRegTaps; t < wd; ++t) {
    const float2 c = fr[t];
    acc = fmaf(__ldg(wrow + t), fmaf(c.x, c.x, c.y * c.y), acc);
  }
  return acc;
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
  float w[kRegTaps];
  const float *wrow;
};

// Consumer main loop.  W = number of register taps used (4 or 8), or 0 for
// bands wider than kRegTaps (tail weights read through L1).
template <int FPT, int W, bool kResident>
__device__ __forceinline__ void consume(const StftArgs &a, unsigned char *smem, SmemAux &aux, float *ring,
                                        int64_t my_tiles, const Band &c, int lane) {
  volatile int *abort_flag = &aux.abort_flag;
  const int S = a.n_stages;
  const int64_t fstep = static_cast<int64_t>(a.FG) * a.NF;  // complex values between a thread's frames
  const int ostep = a.FG * a.NM;                           // outputs between a thread's frames
  const int slot_stride = a.TF * a.NM;
  TileIter cit, sit;
  cit.init(blockIdx.x, a.tiles_per_clip);
  sit.init(blockIdx.x, a.tiles_per_clip);
  int s = 0, slot = 0, sslot = 0;
  uint32_t ph = 0;

  // Final values of step q: (max(ls, hi - 8) + 4) / 4 from this thread's own ring entries.
  auto store_final = [&](int64_t q) {
    mbar_wait(&aux.hi_bar[q & (kSlots - 1)], static_cast<uint32_t>((q / kSlots) & 1), abort_flag, a.err);
    const float floor_v = aux.hi_val[q & (kSlots - 1)] - 8.0f;
    const int nf = sit.frames(a);
    const float *r = ring + sslot * slot_stride + c.fg * a.NM + c.n;
    float *o = a.out + sit.first_frame(a) * a.NM + c.fg * a.NM + c.n;
#pragma unroll
    for (int j = 0; j < FPT; ++j) {
      if (c.active && c.fg + j * a.FG < nf) __stcs(o, rescale(*r, floor_v));
      r += ostep;
      o += ostep;
    }
    sit.next(a);
    if (++sslot == kLag + 1) sslot = 0;
  };

  for (int64_t k = 0; k < my_tiles; ++k) {
    mbar_wait(&aux.full[s], ph, abort_flag, a.err);
    const int64_t frame0 = cit.first_frame(a);
    const int nf = cit.frames(a);
    const float2 *fr = reinterpret_cast<const float2 *>(smem + static_cast<size_t>(s) * a.stage_stride +
                                                        (((frame0 * a.NF) & 1) ? 8 : 0)) +
                       c.st + static_cast<int64_t>(c.fg) * a.NF;
    float *dst = kResident ? ring + slot * slot_stride + c.fg * a.NM + c.n
                           : a.out + frame0 * a.NM + c.fg * a.NM + c.n;
    float lmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < FPT; ++j) {
      if (c.active && c.fg + j * a.FG < nf) {
        float acc;
        if constexpr (W > 0) {
          acc = band_sum<W>(fr, c.wd, c.w);
        } else {
          acc = band_sum_wide(fr, c.wd, c.w, c.wrow);
        }
        const float v = __log10f(fmaxf(acc, 1e-10f));
        lmax = fmaxf(lmax, v);
        *dst = v;
      }
      fr += fstep;
      dst += ostep;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&aux.empty[s]);
    lmax = warp_max(lmax);

    if constexpr (kResident) {
      const int r = static_cast<int>(k & (kSlots - 1));
      if (lane == 0) {
        atomicMax(&aux.tmax_key[r], float_to_ordered(lmax));
        mbar_arrive(&aux.tmax_bar[r]);
      }
      if (k >= kLag) store_final(k - kLag);
      if (++slot == kLag + 1) slot = 0;
    } else {
      if (lane == 0) atomicMax(a.clip_key + cit.b, float_to_ordered(lmax));
    }
    cit.next(a);
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  if constexpr (kResident) {
    for (int64_t q = my_tiles > kLag ? my_tiles - kLag : 0; q < my_tiles; ++q) store_final(q);
  }
}

template <int FPT, bool kResident>
__global__ void __launch_bounds__(kThreads, 1) stft_logmel_kernel(const StftArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  SmemAux &aux = *reinterpret_cast<SmemAux *>(smem + a.aux_offset);
  volatile int *abort_flag = &aux.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int64_t my_tiles = (a.n_tiles - 1 - blockIdx.x) / G + 1;
  const int S = a.n_stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&aux.full[s], 1);
      mbar_init(&aux.empty[s], kConsumerWarps);
    }
    for (int r = 0; r < kSlots; ++r) {
      mbar_init(&aux.tmax_bar[r], kConsumerWarps);
      mbar_init(&aux.hi_bar[r], 1);
      aux.tmax_key[r] = 0u;
    }
    aux.max_width = 0;
    aux.abort_flag = 0;
    aux.published = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------- producer: bulk copies of frame tiles ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const char *src = reinterpret_cast<const char *>(a.stft);
      TileIter it;
      it.init(blockIdx.x, a.tiles_per_clip);
      int s = 0;
      uint32_t ph = 0;
      for (int64_t k = 0; k < my_tiles; ++k) {
        if (k >= S && !mbar_wait(&aux.empty[s], ph ^ 1u, abort_flag, a.err)) break;
        const uint64_t start = static_cast<uint64_t>(it.first_frame(a)) * a.NF * 8ull;
        const uint64_t end = start + static_cast<uint64_t>(it.frames(a)) * a.NF * 8ull;
        const uint64_t a0 = start & ~15ull;
        uint64_t a1 = (end + 15ull) & ~15ull;
        unsigned char *dst = smem + static_cast<size_t>(s) * a.stage_stride;
        if (a1 > a.total_bytes) {
          // The tensor ends 8 bytes past a 16-byte boundary: copy its last
          // complex value by hand; the bulk copy stops at the boundary.
          a1 = end & ~15ull;
          *reinterpret_cast<float2 *>(dst + (end - 8 - a0)) =
              *reinterpret_cast<const float2 *>(src + end - 8);
        }
        const uint32_t bytes = static_cast<uint32_t>(a1 - a0);
        mbar_arrive_expect_tx(&aux.full[s], bytes);
        if (bytes > 0) bulk_g2s(dst, src + a0, bytes, &aux.full[s], pol);
        it.next(a);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    return;
  }

  if (warp == kPublisherWarp) {
    // ---- publisher: one store per tile of the tile's maximum key ----
    if (!kResident || lane != 0) return;
    volatile uint32_t *tkey = aux.tmax_key;
    volatile int64_t *published = &aux.published;
    for (int64_t k = 0; k < my_tiles; ++k) {
      const int r = static_cast<int>(k & (kSlots - 1));
      mbar_wait(&aux.tmax_bar[r], static_cast<uint32_t>((k / kSlots) & 1), abort_flag, a.err);
      const uint32_t key = tkey[r];
      tkey[r] = 0u;
      st_relaxed_gpu(a.tile_key + blockIdx.x + k * G, key);
      *published = k + 1;
    }
    return;
  }

  if (warp == kResolverWarp) {
    // ---- resolver: clip maximum once every tile of the clip is published ----
    // The slots of a clip are contiguous (tiles are numbered clip-major), so
    // one warp-wide load pass reads them all; a zero slot means a tile of the
    // clip is still in flight on some CTA.  Before handing over the maximum
    // for step q the resolver waits until this CTA has published step q: that
    // both covers this CTA's own tile and guarantees the consumers have taken
    // the slot's previous value (step q - kSlots), so an mbarrier phase is
    // never completed twice ahead of its waiters.
    if (!kResident) return;
    volatile int64_t *published = &aux.published;
    TileIter res;
    res.init(blockIdx.x, a.tiles_per_clip);
    int64_t cached_b = -1;
    float cached_hi = 0.f;
    bool gave_up = false;
    for (int64_t q = 0; q < my_tiles; ++q) {
      uint64_t t0 = 0;
      while (!gave_up && *published <= q) {
        int stop = 0;
        if (lane == 0) {
          const uint64_t now = global_timer_ns();
          if (t0 == 0) t0 = now;
          if (!*abort_flag && now - t0 > kWaitTimeoutNs) {
            *abort_flag = 1;
            atomicOr(a.err, kErrClipTimeout);
          }
          stop = *abort_flag;
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) gave_up = true;
        else __nanosleep(32);
      }
      if (res.b != cached_b && !gave_up) {
        const uint32_t *slots = a.tile_key + res.b * a.tiles_per_clip;
        uint32_t m = 0;
        t0 = 0;
        for (;;) {
          bool ok = true;
          m = 0;
#pragma unroll 4
          for (int i = lane; i < a.tiles_per_clip; i += 32) {
            const uint32_t v = ld_relaxed_gpu(slots + i);
            ok = ok && (v != 0u);
            m = max(m, v);
          }
          if (__all_sync(0xffffffffu, ok)) break;
          int stop = 0;
          if (lane == 0) {
            const uint64_t now = global_timer_ns();
            if (t0 == 0) t0 = now;
            if (!*abort_flag && now - t0 > kWaitTimeoutNs) {
              *abort_flag = 1;
              atomicOr(a.err, kErrClipTimeout);
            }
            stop = *abort_flag;
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) {
            gave_up = true;
            break;
          }
          __nanosleep(128);
        }
        cached_b = res.b;
        cached_hi = ordered_to_float(__reduce_max_sync(0xffffffffu, m));
      }
      if (lane == 0) {
        aux.hi_val[q & (kSlots - 1)] = cached_hi;
        mbar_arrive(&aux.hi_bar[q & (kSlots - 1)]);
      }
      __syncwarp();
      res.next(a);
    }
    return;
  }

  // ---------------------------- consumers ----------------------------
  // Support of each filter row: first and last nonzero bin.
  for (int n = warp; n < a.NM; n += kConsumerWarps) {
    const float *row = a.filters + static_cast<int64_t>(n) * a.NF;
    int first = INT_MAX, last = -1;
    for (int k0 = 0; k0 < a.NF; k0 += 32) {
      const int k = k0 + lane;
      const float v = k < a.NF ? __ldg(row + k) : 0.f;
      const unsigned m = __ballot_sync(0xffffffffu, v != 0.f);
      if (m) {
        if (first == INT_MAX) first = k0 + __ffs(m) - 1;
        last = k0 + 31 - __clz(m);
      }
    }
    if (lane == 0) {
      const int width = last >= 0 ? last - first + 1 : 0;
      aux.band_start[n] = last >= 0 ? first : 0;
      aux.band_width[n] = width;
      atomicMax(&aux.max_width, width);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");

  Band band;
  band.n = threadIdx.x % a.NM;
  band.fg = threadIdx.x / a.NM;
  band.active = band.fg < a.FG;
  band.st = band.active ? aux.band_start[band.n] : 0;
  band.wd = band.active ? aux.band_width[band.n] : 0;
  band.wrow = a.filters + static_cast<int64_t>(band.n) * a.NF + band.st;
#pragma unroll
  for (int t = 0; t < kRegTaps; ++t) band.w[t] = (t < band.wd) ? __ldg(band.wrow + t) : 0.f;
  float *ring = reinterpret_cast<float *>(smem + static_cast<size_t>(a.n_stages) * a.stage_stride);
  const int maxw = aux.max_width;
  if (maxw <= 4)
    consume<FPT, 4, kResident>(a, smem, aux, ring, my_tiles, band, lane);
  else if (maxw <= kRegTaps)
    consume<FPT, kRegTaps, kResident>(a, smem, aux, ring, my_tiles, band, lane);
  else
    consume<FPT, 0, kResident>(a, smem, aux, ring, my_tiles, band, lane);
}

// Two-pass epilogue: out = (max(out, hi[b] - 8) + 4) / 4 in place.
__global__ void logmel_clamp_kernel(float *out, const uint32_t *clip_key, int64_t B, int64_t per_clip,
                                    int vec4) {
  for (int64_t b = blockIdx.y; b < B; b += gridDim.y) {
    const float floor_v = ordered_to_float(clip_key[b]) - 8.0f;
    float *o = out + b * per_clip;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (vec4) {
      float4 *o4 = reinterpret_cast<float4 *>(o);
      for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < per_clip / 4; i += stride) {
        float4 v = o4[i];
        v.x = rescale(v.x, floor_v);
        v.y = rescale(v.y, floor_v);
        v.z = rescale(v.z, floor_v);
        v.w = rescale(v.w, floor_v);
        o4[i] = v;
      }
    } else {
      for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < per_clip; i += stride)
        o[i] = rescale(o[i], floor_v);
    }
  }
}

using KernelFn = void (*)(StftArgs);

template <int FPT>
KernelFn pick_variant(bool resident) {
  return resident ? stft_logmel_kernel<FPT, true> : stft_logmel_kernel<FPT, false>;
}

KernelFn pick_kernel(int fpt, bool resident) {
  switch (fpt) {
    case 1: return pick_variant<1>(resident);
    case 2: return pick_variant<2>(resident);
    case 4: return pick_variant<4>(resident);
    default: return pick_variant<8>(resident);
  }
}

struct TilePlan {
  int FG, FPT, TF, S;
  uint32_t stride;
  int64_t ring_bytes;
  uint32_t aux_offset;
  size_t smem;
};

// Tile height: FG frame groups of NM threads, FPT frames per thread, with a
// stage of roughly kStageTargetBytes.
void tile_height(int NF, int NM, int *FG, int *FPT) {
  const int fg_max = kConsumers / NM;
  const int64_t frame_bytes = static_cast<int64_t>(NF) * 8;
  *FG = fg_max;
  *FPT = 0;
  for (int fpt : {8, 4, 2, 1}) {
    if (static_cast<int64_t>(fg_max) * fpt * frame_bytes <= kStageTargetBytes) {
      *FPT = fpt;
      break;
    }
  }
  if (*FPT == 0) {
    *FPT = 1;
    *FG = std::max<int>(1, std::min<int64_t>(fg_max, kStageTargetBytes / frame_bytes));
  }
}

// Shared memory: S stages | (resident) kLag+1 output slots of TF x NM | SmemAux.
TilePlan plan_tiles(int NF, int NM, int max_smem, bool resident) {
  TilePlan p{};
  tile_height(NF, NM, &p.FG, &p.FPT);
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
  int L = 0;         // lag in steps (resident mode)
  bool resident = false;
  KernelFn kern = nullptr;
};

// Chooses tile shape, ring depth, variant and grid for a problem shape.
lm_status plan_launch(int64_t B, int64_t F, int32_t NF, int32_t NM, StftLaunch *ln) {
  DeviceInfo dev;
  if (lm_status st = current_device_info(&dev); st != LM_OK) return st;
  int FG = 0, FPT = 0;
  tile_height(NF, NM, &FG, &FPT);
  const int TF = FG * FPT;
  ln->tpc = (F + TF - 1) / TF;
  if (ln->tpc > INT32_MAX / 2) return LM_ERR_UNSUPPORTED;
  const int64_t n_tiles = B * ln->tpc;
  ln->grid = std::min<int64_t>(n_tiles, dev.sm_count);
  // Resident mode never deadlocks when every tile of the clip of step q sits
  // at a step <= q + L - 1 of the static round-robin schedule; the clip of
  // tile q spans at most (grid + tpc - 2) / grid further steps.
  const int64_t L_need = 1 + (ln->grid + ln->tpc - 2) / ln->grid;
  const char *variant = env_or("LOGMEL_K1_VARIANT", "auto");
  const bool force_two = std::strcmp(variant, "twopass") == 0;
  const bool force_res = std::strcmp(variant, "resident") == 0;
  ln->resident = !force_two && L_need <= kLag;
  if (ln->resident) {
    ln->tp = plan_tiles(NF, NM, dev.max_smem_optin, true);
    if (ln->tp.S < 2) ln->resident = false;  // the output ring does not fit beside two stages
  }
  if (force_res && !ln->resident) return LM_ERR_UNSUPPORTED;
  if (!ln->resident) ln->tp = plan_tiles(NF, NM, dev.max_smem_optin, false);
  if (ln->tp.S < 2) return LM_ERR_UNSUPPORTED;
  ln->L = ln->resident ? kLag : 0;
  ln->kern = pick_kernel(ln->tp.FPT, ln->resident);
  if (lm_status st = ensure_smem_attribute(reinterpret_cast<const void *>(ln->kern), static_cast<int>(ln->tp.smem));
      st != LM_OK)
    return st;
  int per_sm = 0;
  LM_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ln->kern, kThreads, ln->tp.smem));
  if (per_sm < 1) return LM_ERR_UNSUPPORTED;
  return LM_OK;
}

}  // namespace

// Workspace layout: header | clip_key[B] | tile_key[B * tiles_per_clip].
static size_t tile_key_offset(int64_t B) {
  return (kWorkspaceHeaderBytes + static_cast<size_t>(B) * sizeof(uint32_t) + 15) / 16 * 16;
}

size_t stft_workspace_bytes(int64_t B, int64_t F, int32_t NF, int32_t NM) {
  if (B < 1 || F < 1 || NF < 1 || NM < 1 || NF > kMaxBins || NM > kMaxBands) return kWorkspaceHeaderBytes;
  int FG = 0, FPT = 0;
  tile_height(NF, NM, &FG, &FPT);
  const int64_t tpc = (F + static_cast<int64_t>(FG) * FPT - 1) / (static_cast<int64_t>(FG) * FPT);
  return (tile_key_offset(B) + static_cast<size_t>(B * tpc) * sizeof(uint32_t) + 255) / 256 * 256;
}

lm_status stft_logmel_run(const void *stft, const float *filters, float *out, int64_t B, int64_t F,
                          int32_t NF, int32_t NM, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
  if (B < 0 || F < 0 || NF < 1 || NM < 1) return LM_ERR_INVALID_ARG;
  if (NF > kMaxBins || NM > kMaxBands) return LM_ERR_UNSUPPORTED;
  if (B == 0 || F == 0) return LM_OK;
  if (!stft || !filters || !out || !workspace) return workspace ? LM_ERR_INVALID_ARG : LM_ERR_WORKSPACE;
  if (F > (int64_t{1} << 40) || B > (int64_t{1} << 40) || (B * F) > (int64_t{1} << 50) / NF)
    return LM_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(stft) & 15) || (reinterpret_cast<uintptr_t>(filters) & 3) ||
      (reinterpret_cast<uintptr_t>(out) & 3) || (reinterpret_cast<uintptr_t>(workspace) & 3))
    return LM_ERR_MISALIGNED;
  const size_t ws_needed = stft_workspace_bytes(B, F, NF, NM);
  if (workspace_bytes < ws_needed) return LM_ERR_WORKSPACE;
  {  // the output may not overlap either input
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + static_cast<uintptr_t>(B * F * NM) * 4;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(stft), s1 = s0 + static_cast<uintptr_t>(B * F * NF) * 8;
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(filters), w1 = w0 + static_cast<uintptr_t>(NM) * NF * 4;
    if ((o0 < s1 && s0 < o1) || (o0 < w1 && w0 < o1)) return LM_ERR_INVALID_ARG;
  }

  StftLaunch ln;
  if (lm_status st = plan_launch(B, F, NF, NM, &ln); st != LM_OK) return st;
  const TilePlan &tp = ln.tp;
  const bool resident = ln.resident;
  const KernelFn kern = ln.kern;
  const int64_t G = ln.grid;
  const int64_t tpc = ln.tpc;

  StftArgs a{};
  a.stft = static_cast<const float2 *>(stft);
  a.filters = filters;
  a.out = out;
  a.err = static_cast<uint32_t *>(workspace);
  a.clip_key = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + kWorkspaceHeaderBytes);
  a.tile_key = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + tile_key_offset(B));
  a.B = B;
  a.F = F;
  a.NF = NF;
  a.NM = NM;
  a.FG = tp.FG;
  a.TF = tp.TF;
  a.tiles_per_clip = static_cast<int32_t>(tpc);
  a.n_tiles = B * tpc;
  a.n_stages = tp.S;
  a.stage_stride = tp.stride;
  a.aux_offset = tp.aux_offset;
  a.total_bytes = static_cast<uint64_t>(B) * static_cast<uint64_t>(F) * static_cast<uint64_t>(NF) * 8ull;
  a.grid_q = G / tpc;
  a.grid_r = static_cast<int32_t>(G % tpc);

  LM_CUDA_TRY(cudaMemsetAsync(workspace, 0, ws_needed, stream));

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(G));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = tp.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = resident ? 1 : 0;
  LM_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, a));

  if (!resident) {
    const int64_t per_clip = F * NM;
    const int vec4 = (per_clip % 4 == 0) && ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
    const int64_t work = vec4 ? per_clip / 4 : per_clip;
    const unsigned gx = static_cast<unsigned>(std::min<int64_t>((work + 255) / 256, 1024));
    const unsigned gy = static_cast<unsigned>(std::min<int64_t>(B, 65535));
    logmel_clamp_kernel<<<dim3(gx, gy), 256, 0, stream>>>(out, a.clip_key, B, per_clip, vec4);
    LM_CUDA_TRY(cudaGetLastError());
  }
  return LM_OK;
}

lm_status stft_describe(int64_t B, int64_t F, int32_t NF, int32_t NM, lm_stft_launch_info *info) {
  if (!info || B < 1 || F < 1 || NF < 1 || NM < 1) return LM_ERR_INVALID_ARG;
  if (NF > kMaxBins || NM > kMaxBands) return LM_ERR_UNSUPPORTED;
  StftLaunch ln;
  if (lm_status st = plan_launch(B, F, NF, NM, &ln); st != LM_OK) return st;
  info->resident = ln.resident ? 1 : 0;
  info->kernels = ln.resident ? 1 : 2;
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
                             reinterpret_cast<cudaStream_t>(stream));
}

extern "C" lm_status lm_log_mel_from_stft_describe(int64_t B, int64_t F, int32_t NF, int32_t NM,
                                                   lm_stft_launch_info *info) {
  return lm::stft_describe(B, F, NF, NM, info);
}
