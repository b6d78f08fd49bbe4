// ptx.cuh -- small inline-PTX helpers for sm_103a: mbarriers, 1-D bulk
// (TMA) copies, L2 cache policies, the global timer and acquire/release
// global accesses.  Every wait helper is bounded and reports a timeout
// instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace lm {

// A wait that has not completed after this many nanoseconds is abandoned and
// reported through the device error word.  Correct use never comes close.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

// Device error word bits.
constexpr uint32_t kErrMbarTimeout = 1u;    // an mbarrier wait ran out
constexpr uint32_t kErrClipTimeout = 2u;    // waiting for another CTA (a clip's maximum, a launch token) ran out
constexpr uint32_t kErrBadPack = 4u;        // packed filters do not match the call (the dense matrix was used)
constexpr uint32_t kErrBounds = 8u;         // checked builds: an index fell outside its buffer (access skipped)

// Checked builds (-DLOGMEL_CHECKED, a debug variant of the library) test the
// computed indices of global-memory accesses against their buffers: an index
// outside [0, n) sets kErrBounds in the error word and the access is skipped,
// so a wrong index shows up as an error bit instead of a fault.  In regular
// builds LM_IN_BOUNDS is the constant true and costs nothing.
#ifdef LOGMEL_CHECKED
__device__ __forceinline__ bool in_bounds_checked(int64_t i, int64_t n, uint32_t *err) {
  if (i >= 0 && i < n) return true;
  atomicOr(err, kErrBounds);
  return false;
}
#define LM_IN_BOUNDS(i, n, err) (::lm::in_bounds_checked(static_cast<int64_t>(i), static_cast<int64_t>(n), (err)))
#else
#define LM_IN_BOUNDS(i, n, err) true
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t tx_bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(tx_bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Slow path of mbar_wait, kept out of line so the hot loops that wait carry
// only the first try_wait: inlining the bounded loop into them measured 4.5%
// slower.  Gives up when the CTA-wide abort flag is set or after
// kWaitTimeoutNs; in the latter case it sets the abort flag and the device
// error word.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t addr, uint32_t parity, volatile int *abort_flag,
                                                   uint32_t *err_word) {
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort_flag) return false;
      const uint64_t now = global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitTimeoutNs) {
        *abort_flag = 1;
        atomicOr(err_word, kErrMbarTimeout);
        return false;
      }
    }
  }
}

// Waits for the phase with the given parity to complete (bounded; see
// mbar_wait_slow).  Returns true on success.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          uint32_t *err_word) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  return mbar_wait_slow(addr, parity, abort_flag, err_word);
}

// Waits for a phase that a bulk copy this thread issued completes: used
// before a CTA exits, so that no copy into its shared memory outlives it.
// Ignores the abort flag (the copy lands whatever the other warps did);
// bounded all the same, reporting kErrMbarTimeout if it ever ran out.
static __device__ __noinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity, uint32_t *err_word) {
  const uint32_t addr = smem_u32(bar);
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(addr, parity)) return true;
    if ((it & 63u) == 0u) {
      const uint64_t now = global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitTimeoutNs) {
        atomicOr(err_word, kErrMbarTimeout);
        return false;
      }
    }
  }
}

// Orders this thread's earlier generic-proxy shared-memory writes before
// later async-proxy (bulk copy) accesses to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory loads and stores by 32-bit shared-window address.  Volatile,
// so the compiler keeps them in program order with the barriers and
// mbarrier waits around them.
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ int lds_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ float2 lds_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v));
}

__device__ __forceinline__ void sts_f32x2(uint32_t addr, float2 v) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y));
}

__device__ __forceinline__ int2 lds_s32x2(uint32_t addr) {
  int2 v;
  asm volatile("ld.shared.v2.s32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Same, with the default L2 policy: for data that every CTA reads.
__device__ __forceinline__ void bulk_g2s_plain(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// This CTA's rank in its thread-block cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives (release) and waits
// (acquire); executed by all threads of each warp together.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A u32 from the shared memory of CTA `rank` of this cluster, at the offset
// that `local_addr` has in this CTA's shared memory.
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint4 ld_relaxed_gpu_v4(const uint32_t *p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu_u64(uint64_t *p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Waits (bounded by `limit_ns`) until the launch token at `p` reads `token`:
// the words a peer cleared before publishing it are then visible to the
// caller.  Returns false when the wait ran out or `abort_flag` was set.
static __device__ __noinline__ bool wait_token(const uint64_t *p, uint64_t token, uint64_t limit_ns,
                                               volatile int *abort_flag) {
  uint64_t t0 = 0;
  for (;;) {
    if (ld_acquire_gpu_u64(p) == token) return true;
    if (abort_flag && *abort_flag) return false;
    const uint64_t now = global_timer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > limit_ns) {
      return false;
    }
    __nanosleep(100);
  }
}

__device__ __forceinline__ void red_add_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Order-preserving map f32 -> u32: a < b  <=>  key(a) < key(b) for all
// non-NaN floats, and key(x) > 0.  Lets atomicMax on u32 reduce floats.
__device__ __forceinline__ uint32_t float_to_ordered(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float ordered_to_float(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace lm
