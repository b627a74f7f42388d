// fp4idx_host.cu -- the fused pre-pass for inputs and outputs in host memory
// (fp4idx_indexer_prepass_host in include/fp4idx.h): the tokens go through
// in chunks, with the upload of chunk c+1, the fused launch of chunk c and the
// download of chunk c-1 overlapped on three streams.  Host code only; the
// arithmetic is the device entry point's (fp4idx_indexer_prepass).
//
// The library allocates no memory: the caller passes the device staging
// buffer (two slots of fp4idx_host_staging_bytes / 2 each).  The streams and
// events of the pipeline are created once per device, under a lock, and kept.
// Every copy is one cudaMemcpyAsync.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fp4idx.h"
#include "fp4idx_common.cuh"

namespace {

constexpr int kMaxDevicesH = 64;
constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// One staging slot: the chunk's inputs and query outputs, each 256-aligned.
struct Slot {
  size_t q, k, w, pos, slots, qf, qs, wt, bytes;
};

Slot slot_layout(int64_t chunk, int64_t H) {
  const size_t c = (size_t)chunk, h = (size_t)H;
  Slot s;
  size_t o = 0;
  s.q = o;     o += up(c * h * FP4IDX_HEAD_DIM * 2);
  s.k = o;     o += up(c * FP4IDX_HEAD_DIM * 2);
  s.w = o;     o += up(c * h * 2);
  s.pos = o;   o += up(c * 8);
  s.slots = o; o += up(c * 8);
  s.qf = o;    o += up(c * h * 64);
  s.qs = o;    o += up(c * h * 4);
  s.wt = o;    o += up(c * h * 4);
  s.bytes = o;
  return s;
}

// The pipeline's streams and events for one device, created once.  The
// events of the last call stay recorded, so a later call waits for the
// staging slots the earlier one still reads or writes.
struct Pipe {
  bool ready = false;
  cudaStream_t s_in = nullptr, s_run = nullptr, s_out = nullptr;
  cudaEvent_t ev_in[2], ev_run[2], ev_out[2], ev_start, ev_end_run, ev_end_out;
};

std::mutex g_pipe_mutex;  // held while a call enqueues
Pipe g_pipes[kMaxDevicesH];

bool make_pipe(Pipe& p) {
  if (p.ready) return true;
  const unsigned ev = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p.s_run, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking) != cudaSuccess)
    return false;
  for (int b = 0; b < 2; ++b)
    if (cudaEventCreateWithFlags(&p.ev_in[b], ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.ev_run[b], ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.ev_out[b], ev) != cudaSuccess)
      return false;
  if (cudaEventCreateWithFlags(&p.ev_start, ev) != cudaSuccess ||
      cudaEventCreateWithFlags(&p.ev_end_run, ev) != cudaSuccess ||
      cudaEventCreateWithFlags(&p.ev_end_out, ev) != cudaSuccess)
    return false;
  p.ready = true;
  return true;
}

// The staging of fp4idx_indexer_prepass_host_static: one buffer per device
// (a module global), never allocated by a call.  Its address is looked up
// once per device, under the pipeline lock.
__device__ __align__(256) uint8_t g_static_staging[FP4IDX_STATIC_STAGING_BYTES];
void* g_static_addr[kMaxDevicesH];

}  // namespace

extern "C" {

size_t fp4idx_host_staging_bytes(int64_t chunk_tokens, int64_t num_heads) {
  if (chunk_tokens < 1 || num_heads < 1 || chunk_tokens >= (1ll << 30) ||
      num_heads >= (1ll << 30) / chunk_tokens)
    return 0;
  return 2 * slot_layout(chunk_tokens, num_heads).bytes;
}

fp4idx_status fp4idx_indexer_prepass_host(
    const void* k, const int64_t* slot_mapping, const void* gamma, float eps, uint8_t* kv_cache,
    int64_t num_blocks, const void* q, const void* w, int64_t num_heads, float weight_scale,
    uint8_t* q_fp4, uint8_t* q_scale, float* weights_out, const int64_t* positions,
    const float* cos_cache, const float* sin_cache, int64_t max_pos, int rope_style,
    int64_t num_tokens, int64_t chunk_tokens, void* staging, uint32_t* err_flags,
    void* stream) {
  if (num_tokens < 0 || num_heads < 1 || chunk_tokens < 1) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0) return FP4IDX_OK;
  if (!k || !slot_mapping || !gamma || !kv_cache || !q || !w || !q_fp4 || !q_scale ||
      !weights_out || !positions || !cos_cache || !sin_cache || !staging)
    return FP4IDX_ERR_NULL;
  if (fp4idx_host_staging_bytes(chunk_tokens, num_heads) == 0) return FP4IDX_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(staging) % kAlign) != 0) return FP4IDX_ERR_ALIGN;
  const int64_t H = num_heads, chunk = chunk_tokens < num_tokens ? chunk_tokens : num_tokens;
  const Slot L = slot_layout(chunk_tokens, H);  // the caller sized staging for chunk_tokens
  {  // the device call's own checks, on the first chunk, before anything is enqueued
    uint8_t* const s0 = static_cast<uint8_t*>(staging);
    const fp4idx_status st = fp4idx_impl::prepass_check(
        s0 + L.k, FP4IDX_HEAD_DIM, gamma, eps, reinterpret_cast<const int64_t*>(s0 + L.slots),
        kv_cache, num_blocks, s0 + L.q, H * FP4IDX_HEAD_DIM, FP4IDX_HEAD_DIM, s0 + L.w,
        weight_scale, s0 + L.qf, s0 + L.qs, reinterpret_cast<const float*>(s0 + L.wt), H,
        reinterpret_cast<const int64_t*>(s0 + L.pos), cos_cache, sin_cache, max_pos, rope_style,
        chunk, err_flags, 0);
    if (st != FP4IDX_OK) return st;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesH) return FP4IDX_ERR_CUDA;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);

  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  Pipe& p = g_pipes[dev];
  if (!make_pipe(p)) return FP4IDX_ERR_CUDA;
  bool ok = true;
  auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
  // Work already queued on the caller's stream comes first, and so does an
  // earlier call: its kernels read the staging inputs (ev_run) and its
  // downloads read the staging outputs (ev_out) this call overwrites.  A
  // wait for an event never recorded returns at once.
  chk(cudaEventRecord(p.ev_start, caller));
  chk(cudaStreamWaitEvent(p.s_in, p.ev_start, 0));
  chk(cudaStreamWaitEvent(p.s_run, p.ev_start, 0));
  chk(cudaStreamWaitEvent(p.s_out, p.ev_start, 0));
  for (int b = 0; b < 2; ++b) {
    chk(cudaStreamWaitEvent(p.s_in, p.ev_run[b], 0));
    chk(cudaStreamWaitEvent(p.s_run, p.ev_out[b], 0));
  }
  fp4idx_status st = FP4IDX_OK;
  const size_t row_q = (size_t)H * FP4IDX_HEAD_DIM * 2;  // bytes per token of q
  const int64_t nchunks = (num_tokens + chunk - 1) / chunk;
  for (int64_t c = 0; c < nchunks && ok && st == FP4IDX_OK; ++c) {
    const int b = (int)(c & 1);
    const int64_t t0 = c * chunk, n = (num_tokens - t0) < chunk ? (num_tokens - t0) : chunk;
    uint8_t* const slot = static_cast<uint8_t*>(staging) + (size_t)b * L.bytes;
    if (c >= 2) chk(cudaStreamWaitEvent(p.s_in, p.ev_run[b], 0));  // inputs free
    const uint8_t* qh = static_cast<const uint8_t*>(q) + (size_t)t0 * row_q;
    const uint8_t* kh = static_cast<const uint8_t*>(k) + (size_t)t0 * FP4IDX_HEAD_DIM * 2;
    const uint8_t* wh = static_cast<const uint8_t*>(w) + (size_t)t0 * H * 2;
    chk(cudaMemcpyAsync(slot + L.q, qh, (size_t)n * row_q, cudaMemcpyHostToDevice, p.s_in));
    chk(cudaMemcpyAsync(slot + L.k, kh, (size_t)n * FP4IDX_HEAD_DIM * 2, cudaMemcpyHostToDevice,
                        p.s_in));
    chk(cudaMemcpyAsync(slot + L.w, wh, (size_t)n * H * 2, cudaMemcpyHostToDevice, p.s_in));
    chk(cudaMemcpyAsync(slot + L.pos, positions + t0, (size_t)n * 8, cudaMemcpyHostToDevice,
                        p.s_in));
    chk(cudaMemcpyAsync(slot + L.slots, slot_mapping + t0, (size_t)n * 8,
                        cudaMemcpyHostToDevice, p.s_in));
    chk(cudaEventRecord(p.ev_in[b], p.s_in));
    chk(cudaStreamWaitEvent(p.s_run, p.ev_in[b], 0));
    if (c >= 2) chk(cudaStreamWaitEvent(p.s_run, p.ev_out[b], 0));  // outputs free
    if (!ok) break;
    st = fp4idx_indexer_prepass(
        slot + L.k, FP4IDX_HEAD_DIM, gamma, eps, reinterpret_cast<const int64_t*>(slot + L.slots),
        kv_cache, num_blocks, slot + L.q, H * FP4IDX_HEAD_DIM, FP4IDX_HEAD_DIM, slot + L.w, H,
        weight_scale, slot + L.qf, slot + L.qs, reinterpret_cast<float*>(slot + L.wt), H,
        reinterpret_cast<const int64_t*>(slot + L.pos), cos_cache, sin_cache, max_pos,
        rope_style, n, err_flags, p.s_run);
    chk(cudaEventRecord(p.ev_run[b], p.s_run));
    chk(cudaStreamWaitEvent(p.s_out, p.ev_run[b], 0));
    chk(cudaMemcpyAsync(q_fp4 + (size_t)t0 * H * 64, slot + L.qf, (size_t)n * H * 64,
                        cudaMemcpyDeviceToHost, p.s_out));
    chk(cudaMemcpyAsync(q_scale + (size_t)t0 * H * 4, slot + L.qs, (size_t)n * H * 4,
                        cudaMemcpyDeviceToHost, p.s_out));
    chk(cudaMemcpyAsync(weights_out + (size_t)t0 * H, slot + L.wt, (size_t)n * H * 4,
                        cudaMemcpyDeviceToHost, p.s_out));
    chk(cudaEventRecord(p.ev_out[b], p.s_out));
  }
  // the caller's stream continues once every launch and download is done
  chk(cudaEventRecord(p.ev_end_run, p.s_run));
  chk(cudaEventRecord(p.ev_end_out, p.s_out));
  chk(cudaStreamWaitEvent(caller, p.ev_end_run, 0));
  chk(cudaStreamWaitEvent(caller, p.ev_end_out, 0));
  if (st != FP4IDX_OK) return st;
  return ok ? FP4IDX_OK : FP4IDX_ERR_CUDA;
}

fp4idx_status fp4idx_indexer_prepass_host_static(
    const void* k, const int64_t* slot_mapping, const void* gamma, float eps, uint8_t* kv_cache,
    int64_t num_blocks, const void* q, const void* w, int64_t num_heads, float weight_scale,
    uint8_t* q_fp4, uint8_t* q_scale, float* weights_out, const int64_t* positions,
    const float* cos_cache, const float* sin_cache, int64_t max_pos, int rope_style,
    int64_t num_tokens, int64_t chunk_tokens, uint32_t* err_flags, void* stream) {
  if (num_tokens < 0 || num_heads < 1 || chunk_tokens < 1) return FP4IDX_ERR_SHAPE;
  if (num_tokens == 0) return FP4IDX_OK;
  const size_t need = fp4idx_host_staging_bytes(chunk_tokens, num_heads);
  if (need == 0) return FP4IDX_ERR_SHAPE;
  if (need > (size_t)FP4IDX_STATIC_STAGING_BYTES) return FP4IDX_ERR_SCRATCH;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesH) return FP4IDX_ERR_CUDA;
  void* staging = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    if (g_static_addr[dev] == nullptr) {
      void* a = nullptr;
      if (cudaGetSymbolAddress(&a, g_static_staging) != cudaSuccess || a == nullptr)
        return FP4IDX_ERR_CUDA;
      g_static_addr[dev] = a;
    }
    staging = g_static_addr[dev];
  }
  return fp4idx_indexer_prepass_host(k, slot_mapping, gamma, eps, kv_cache, num_blocks, q, w,
                                     num_heads, weight_scale, q_fp4, q_scale, weights_out,
                                     positions, cos_cache, sin_cache, max_pos, rope_style,
                                     num_tokens, chunk_tokens, staging, err_flags, stream);
}

}  // extern "C"
