// host_pipeline.cu -- the entry points that take host buffers.
//
// The batch is cut into chunks of whole clips (both operations treat clips
// independently, the per-clip maximum included).  Chunk k goes through
// staging slot k % kPipeSlots of the device workspace:
//
//   copy-in stream   wait until the kernel of chunk k - kPipeSlots has read
//                    the slot; host -> slot input;        record loaded[slot]
//   caller's stream  wait loaded[slot] and, for the slot's output buffer,
//                    drained[slot] of chunk k - kPipeSlots; the operation on
//                    the chunk;                           record computed[slot]
//   copy-out stream  wait computed[slot]; slot output -> host;
//                                                         record drained[slot]
//
// so the copy in of chunk k + 1, the kernels of chunk k and the copy out of
// chunk k - 1 run at the same time, and both directions of the host link stay
// busy.  The two copy streams start after the caller's earlier work (one
// event) and the caller's stream waits for both at the end (two events), so
// the whole call is ordered on the caller's stream like any other entry point.
#include <algorithm>
#include <mutex>
#include <vector>

#include "internal.h"

namespace lm {
namespace {

constexpr int kPipeSlots = 3;
// Default chunk: the whole clips that fit in about this many input bytes,
// and at most a third of the batch.  The first bound keeps filling and
// draining the pipeline cheap against the transfer of a large batch; the
// second gives a small batch at least three chunks to overlap.  Smaller
// chunks lose more than they gain: a chunk's kernels then fill only part of
// the GPU, and the host spends longer enqueueing than the copies take.
constexpr size_t kChunkTargetBytes = size_t{32} << 20;
constexpr int64_t kMinChunks = 3;

struct PipeStreams {
  int device = -1;
  cudaStream_t in = nullptr;
  cudaStream_t out = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t join_in = nullptr;
  cudaEvent_t join_out = nullptr;
  cudaEvent_t loaded[kPipeSlots] = {};
  cudaEvent_t computed[kPipeSlots] = {};
  cudaEvent_t drained[kPipeSlots] = {};
};

// Idle stream sets of every device.  A call takes one for its duration, so
// concurrent calls from several host threads never share events.
std::mutex g_pipe_mu;
std::vector<PipeStreams *> g_pipe_idle;

void destroy_streams(PipeStreams *p) {
  if (!p) return;
  if (p->in) cudaStreamDestroy(p->in);
  if (p->out) cudaStreamDestroy(p->out);
  cudaEvent_t *events[] = {&p->fork, &p->join_in, &p->join_out};
  for (cudaEvent_t *e : events)
    if (*e) cudaEventDestroy(*e);
  for (int i = 0; i < kPipeSlots; ++i) {
    if (p->loaded[i]) cudaEventDestroy(p->loaded[i]);
    if (p->computed[i]) cudaEventDestroy(p->computed[i]);
    if (p->drained[i]) cudaEventDestroy(p->drained[i]);
  }
  delete p;
}

lm_status create_streams(int dev, PipeStreams **out) {
  PipeStreams *p = new PipeStreams;
  p->device = dev;
  cudaError_t e = cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking);
  cudaEvent_t *events[] = {&p->fork, &p->join_in, &p->join_out};
  for (cudaEvent_t *ev : events)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  for (int i = 0; i < kPipeSlots && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&p->loaded[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->computed[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->drained[i], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    destroy_streams(p);
    return cuda_fail(e);
  }
  *out = p;
  return LM_OK;
}

lm_status acquire_streams(int dev, PipeStreams **out) {
  {
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    for (size_t i = 0; i < g_pipe_idle.size(); ++i) {
      if (g_pipe_idle[i]->device == dev) {
        *out = g_pipe_idle[i];
        g_pipe_idle.erase(g_pipe_idle.begin() + static_cast<std::ptrdiff_t>(i));
        return LM_OK;
      }
    }
  }
  return create_streams(dev, out);
}

void release_streams(PipeStreams *p) {
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  g_pipe_idle.push_back(p);
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// One chunk's work, enqueued on `s`: input slot -> output slot for clips
// [b0, b0 + n).
struct ChunkOp {
  virtual ~ChunkOp() = default;
  virtual lm_status run(const void *din, void *dout, int64_t n, cudaStream_t s) = 0;
};

// Workspace layout shared by both host entry points:
//   header (16 B; its first u32 is the device error word of every chunk)
//   | the operation's own workspace for one chunk
//   | kPipeSlots input slots | kPipeSlots output slots     (each 256-aligned)
struct PipeLayout {
  int64_t chunk = 0;
  size_t op_ws = 0, in_slot = 0, out_slot = 0;
  size_t op_offset() const { return 256; }
  size_t in_offset() const { return op_offset() + round256(op_ws); }
  size_t out_offset() const { return in_offset() + kPipeSlots * round256(in_slot); }
  size_t bytes() const { return out_offset() + kPipeSlots * round256(out_slot); }
};

int64_t pick_chunk(int64_t B, size_t in_per_clip, int64_t chunk_clips) {
  if (chunk_clips > 0) return std::min(chunk_clips, std::max<int64_t>(B, 1));
  const int64_t by_bytes = static_cast<int64_t>(kChunkTargetBytes / std::max<size_t>(in_per_clip, 1));
  const int64_t by_count = (std::max<int64_t>(B, 1) + kMinChunks - 1) / kMinChunks;
  return std::max<int64_t>(1, std::min(by_bytes, by_count));
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Runs the pipeline over B clips; argument checks are done by the caller.
lm_status run_pipeline(const char *host_in, size_t in_per_clip, char *host_out, size_t out_per_clip, int64_t B,
                       const PipeLayout &L, char *ws, cudaStream_t s, ChunkOp &op) {
  int dev = 0;
  LM_CUDA_TRY(cudaGetDevice(&dev));
  PipeStreams *ps = nullptr;
  if (lm_status st = acquire_streams(dev, &ps); st != LM_OK) return st;

  cudaError_t e = cudaMemsetAsync(ws, 0, kWorkspaceHeaderBytes, s);
  if (e == cudaSuccess) e = cudaEventRecord(ps->fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ps->in, ps->fork, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ps->out, ps->fork, 0);
  if (e != cudaSuccess) {
    release_streams(ps);
    return cuda_fail(e);
  }
  lm_status st = LM_OK;
  const int64_t n_chunks = (B + L.chunk - 1) / L.chunk;
  for (int64_t k = 0; k < n_chunks && st == LM_OK && e == cudaSuccess; ++k) {
    const int slot = static_cast<int>(k % kPipeSlots);
    const int64_t b0 = k * L.chunk;
    const int64_t n = std::min(L.chunk, B - b0);
    char *din = ws + L.in_offset() + slot * round256(L.in_slot);
    char *dout = ws + L.out_offset() + slot * round256(L.out_slot);
    const bool reuse = k >= kPipeSlots;
    if (reuse) e = cudaStreamWaitEvent(ps->in, ps->computed[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(din, host_in + static_cast<size_t>(b0) * in_per_clip, static_cast<size_t>(n) * in_per_clip,
                          cudaMemcpyDefault, ps->in);
    if (e == cudaSuccess) e = cudaEventRecord(ps->loaded[slot], ps->in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ps->loaded[slot], 0);
    if (e == cudaSuccess && reuse) e = cudaStreamWaitEvent(s, ps->drained[slot], 0);
    if (e != cudaSuccess) break;
    st = op.run(din, dout, n, s);
    if (st != LM_OK) break;
    e = cudaEventRecord(ps->computed[slot], s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ps->out, ps->computed[slot], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(host_out + static_cast<size_t>(b0) * out_per_clip, dout,
                          static_cast<size_t>(n) * out_per_clip, cudaMemcpyDefault, ps->out);
    if (e == cudaSuccess) e = cudaEventRecord(ps->drained[slot], ps->out);
  }
  // Join both copy streams back into the caller's stream, also after a
  // failure, so that nothing the call enqueued outlives its stream order.
  cudaError_t j = cudaEventRecord(ps->join_in, ps->in);
  if (j == cudaSuccess) j = cudaEventRecord(ps->join_out, ps->out);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(s, ps->join_in, 0);
  if (j == cudaSuccess) j = cudaStreamWaitEvent(s, ps->join_out, 0);
  release_streams(ps);
  if (e != cudaSuccess) return cuda_fail(e);
  if (st != LM_OK) return st;
  if (j != cudaSuccess) return cuda_fail(j);
  return LM_OK;
}

lm_status refuse_capture(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  LM_CUDA_TRY(cudaStreamIsCapturing(s, &cs));
  return cs == cudaStreamCaptureStatusNone ? LM_OK : LM_ERR_UNSUPPORTED;
}

// --- log_mel_from_stft ------------------------------------------------------

lm_status stft_host_layout(int64_t B, int64_t F, int32_t NF, int32_t NM, int64_t chunk_clips, PipeLayout *L) {
  if (B < 0 || F < 0 || NF < 1 || NM < 1 || chunk_clips < 0) return LM_ERR_INVALID_ARG;
  if (NF > 8193 || NM > 512) return LM_ERR_UNSUPPORTED;
  if (F > (int64_t{1} << 40) || B > (int64_t{1} << 40) || (F > 0 && B > (int64_t{1} << 50) / (F * NF)))
    return LM_ERR_UNSUPPORTED;
  const size_t in_clip = static_cast<size_t>(F) * NF * 8, out_clip = static_cast<size_t>(F) * NM * 4;
  L->chunk = pick_chunk(B, in_clip, chunk_clips);
  L->op_ws = stft_workspace_bytes(L->chunk, F, NF, NM);
  L->in_slot = static_cast<size_t>(L->chunk) * in_clip;
  L->out_slot = static_cast<size_t>(L->chunk) * out_clip;
  return LM_OK;
}

struct StftChunk final : ChunkOp {
  const float *filters;
  const void *packed;
  int64_t F;
  int32_t NF, NM;
  void *op_ws;
  size_t op_ws_bytes;
  uint32_t *err;
  lm_status run(const void *din, void *dout, int64_t n, cudaStream_t s) override {
    return stft_logmel_run(din, filters, static_cast<float *>(dout), n, F, NF, NM, op_ws, op_ws_bytes, s, packed,
                           err);
  }
};

// --- mel_spectrogram --------------------------------------------------------

lm_status mel_host_layout(const lm_mel_plan *plan, int64_t B, int64_t T, int32_t in_dtype, int32_t out_dtype,
                          int64_t chunk_clips, PipeLayout *L, size_t *in_clip, size_t *out_clip) {
  if (!plan || B < 0 || T < 0 || chunk_clips < 0) return LM_ERR_INVALID_ARG;
  if (in_dtype != LM_F32 && in_dtype != LM_I16) return LM_ERR_UNSUPPORTED;
  if (out_dtype != LM_F32 && out_dtype != LM_F16) return LM_ERR_UNSUPPORTED;
  int32_t n_mels = 0;
  if (lm_status st = mel_plan_n_mels(plan, &n_mels); st != LM_OK) return st;
  int64_t nfr = 0;
  if (lm_status st = lm_mel_n_frames(plan, T, &nfr); st != LM_OK) return st;
  if (nfr < 0) nfr = 0;
  if (T > (int64_t{1} << 40) || B > (int64_t{1} << 40) || (T > 0 && B > (int64_t{1} << 50) / T) ||
      (nfr > 0 && B > (int64_t{1} << 50) / (nfr * n_mels)))
    return LM_ERR_UNSUPPORTED;
  *in_clip = static_cast<size_t>(T) * (in_dtype == LM_I16 ? 2 : 4);
  *out_clip = static_cast<size_t>(nfr) * n_mels * (out_dtype == LM_F16 ? 2 : 4);
  L->chunk = pick_chunk(B, *in_clip, chunk_clips);
  size_t ws = 0;
  if (lm_status st = lm_mel_workspace_size(plan, L->chunk, T, &ws); st != LM_OK) return st;
  L->op_ws = ws;
  L->in_slot = static_cast<size_t>(L->chunk) * *in_clip;
  L->out_slot = static_cast<size_t>(L->chunk) * *out_clip;
  return LM_OK;
}

struct MelChunk final : ChunkOp {
  const lm_mel_plan *plan;
  int64_t T;
  int32_t in_dtype, out_dtype;
  void *op_ws;
  size_t op_ws_bytes;
  uint32_t *err;
  lm_status run(const void *din, void *dout, int64_t n, cudaStream_t s) override {
    return mel_spectrogram_run(plan, din, in_dtype, n, T, dout, out_dtype, op_ws, op_ws_bytes, s, err);
  }
};

}  // namespace
}  // namespace lm

extern "C" lm_status lm_log_mel_from_stft_host_workspace_size(int64_t B, int64_t F, int32_t NF, int32_t NM,
                                                              int64_t chunk_clips, size_t *bytes) {
  if (!bytes) return LM_ERR_INVALID_ARG;
  lm::PipeLayout L;
  if (lm_status st = lm::stft_host_layout(B, F, NF, NM, chunk_clips, &L); st != LM_OK) return st;
  *bytes = L.bytes();
  return LM_OK;
}

extern "C" lm_status lm_log_mel_from_stft_host(const void *stft_host, const float *mel_filters, const void *packed,
                                               float *out_host, int64_t B, int64_t F, int32_t NF, int32_t NM,
                                               int64_t chunk_clips, void *workspace, size_t workspace_bytes,
                                               lm_stream_t stream) {
  lm::PipeLayout L;
  if (lm_status st = lm::stft_host_layout(B, F, NF, NM, chunk_clips, &L); st != LM_OK) return st;
  if (B == 0 || F == 0) return LM_OK;
  if (!stft_host || !mel_filters || !out_host) return LM_ERR_INVALID_ARG;
  if (!workspace) return LM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(mel_filters) & 3) || (reinterpret_cast<uintptr_t>(workspace) & 255) ||
      (packed && (reinterpret_cast<uintptr_t>(packed) & 15)))
    return LM_ERR_MISALIGNED;
  if (workspace_bytes < L.bytes()) return LM_ERR_WORKSPACE;
  const size_t in_clip = static_cast<size_t>(F) * NF * 8, out_clip = static_cast<size_t>(F) * NM * 4;
  if (lm::overlaps(stft_host, static_cast<size_t>(B) * in_clip, out_host, static_cast<size_t>(B) * out_clip))
    return LM_ERR_INVALID_ARG;
  // The chunk shape must be one the kernel launches (plan checks only).
  lm_stft_launch_info info;
  if (lm_status st = lm::stft_describe(L.chunk, F, NF, NM, &info); st != LM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (lm_status st = lm::refuse_capture(s); st != LM_OK) return st;
  char *ws = static_cast<char *>(workspace);
  lm::StftChunk op;
  op.filters = mel_filters;
  op.packed = packed;
  op.F = F;
  op.NF = NF;
  op.NM = NM;
  op.op_ws = ws + L.op_offset();
  op.op_ws_bytes = L.op_ws;
  op.err = reinterpret_cast<uint32_t *>(ws);
  return lm::run_pipeline(static_cast<const char *>(stft_host), in_clip, reinterpret_cast<char *>(out_host), out_clip,
                          B, L, ws, s, op);
}

extern "C" lm_status lm_mel_spectrogram_host_workspace_size(const lm_mel_plan *plan, int64_t B, int64_t T,
                                                            int32_t in_dtype, int32_t out_dtype,
                                                            int64_t chunk_clips, size_t *bytes) {
  if (!bytes) return LM_ERR_INVALID_ARG;
  lm::PipeLayout L;
  size_t in_clip = 0, out_clip = 0;
  if (lm_status st = lm::mel_host_layout(plan, B, T, in_dtype, out_dtype, chunk_clips, &L, &in_clip, &out_clip);
      st != LM_OK)
    return st;
  *bytes = L.bytes();
  return LM_OK;
}

extern "C" lm_status lm_mel_spectrogram_host(const lm_mel_plan *plan, const void *wave_host, int32_t in_dtype,
                                             int64_t B, int64_t T, void *out_host, int32_t out_dtype,
                                             int64_t chunk_clips, void *workspace, size_t workspace_bytes,
                                             lm_stream_t stream) {
  lm::PipeLayout L;
  size_t in_clip = 0, out_clip = 0;
  if (lm_status st = lm::mel_host_layout(plan, B, T, in_dtype, out_dtype, chunk_clips, &L, &in_clip, &out_clip);
      st != LM_OK)
    return st;
  if (B == 0) return LM_OK;
  if (!wave_host || !out_host) return LM_ERR_INVALID_ARG;
  if (!workspace) return LM_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return LM_ERR_MISALIGNED;
  if (workspace_bytes < L.bytes()) return LM_ERR_WORKSPACE;
  if (lm::overlaps(wave_host, static_cast<size_t>(B) * in_clip, out_host, static_cast<size_t>(B) * out_clip))
    return LM_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (lm_status st = lm::refuse_capture(s); st != LM_OK) return st;
  char *ws = static_cast<char *>(workspace);
  // The chunk's shape rules, checked before anything is enqueued.
  if (lm_status st = lm::mel_spectrogram_check(plan, in_dtype, L.chunk, T, out_dtype); st != LM_OK) return st;
  lm::MelChunk op;
  op.plan = plan;
  op.T = T;
  op.in_dtype = in_dtype;
  op.out_dtype = out_dtype;
  op.op_ws = ws + L.op_offset();
  op.op_ws_bytes = L.op_ws;
  op.err = reinterpret_cast<uint32_t *>(ws);
  return lm::run_pipeline(static_cast<const char *>(wave_host), in_clip, static_cast<char *>(out_host), out_clip, B,
                          L, ws, s, op);
}
