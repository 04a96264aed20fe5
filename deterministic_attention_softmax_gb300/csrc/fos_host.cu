// fos_host.cu -- the softmax step from host buffers: fos_softmax_step_host and its workspace
// query (declared in include/fos_softmax.h).
//
// Rows are cut into chunks that cycle through kSlots device slots of the caller's workspace.
// Three streams overlap the work of consecutive chunks: an upload stream copies chunk c + 1's
// scores and dP from host memory while the caller's stream runs the forward and backward
// kernels on chunk c (P over the scores in place, dScores over dP in place) and a download
// stream copies chunk c - 1's P and dScores back to host memory (LSE and delta, 4 bytes per
// row, follow the last chunk).  Events order the three: a slot is refilled only after its
// previous chunk has been downloaded.  The kernels
// and their arithmetic are those of fos_softmax_fwd / fos_softmax_bwd; a chunk launch covers a
// row range of the problem, so every row keeps its batch entry, head and query index, and the
// results are the bits of the device-buffer entry points.
#include <stdint.h>

#include <mutex>

#include "fos_internal.h"

namespace fos {
namespace {

constexpr int kSlots = 3;                      // chunks in flight: up, compute, down
constexpr size_t kAlign = 256;                 // workspace sub-buffer alignment
constexpr size_t kChunkTarget = 16u << 20;     // default bytes of one tensor chunk
constexpr int kMaxDevices = 64;

size_t round_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Byte layout of the workspace: full LSE and delta (the sink gradient reads every row), d_sink,
// then kSlots slots of two chunk tensors each (scores -> P, dP -> dScores), all 256-aligned.
struct Layout {
  int64_t chunk = 0;
  size_t lse = 0, delta = 0, dsink = 0, slot0 = 0, tensor = 0, total = 0;
};

Layout layout(const fos_desc *d, int esz, int64_t chunk_rows) {
  Layout o;
  int64_t c = chunk_rows;
  if (c <= 0) {
    c = (int64_t)(kChunkTarget / ((size_t)d->ld * esz));
    if (c < 1) c = 1;
  }
  if (c > d->rows) c = d->rows;
  o.chunk = c;
  size_t off = 0;
  o.lse = off;
  off = round_up(off + (size_t)d->rows * sizeof(float));
  o.delta = off;
  off = round_up(off + (size_t)d->rows * sizeof(float));
  o.dsink = off;
  off = round_up(off + (size_t)d->heads * sizeof(float));
  o.slot0 = off;
  o.tensor = round_up((size_t)c * d->ld * esz);
  o.total = off + (size_t)kSlots * 2 * o.tensor;
  return o;
}

// Per-device streams and events of the pipeline, created on first use and kept.
struct Pipe {
  bool ready = false;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in_ready[kSlots] = {}, computed[kSlots] = {}, freed[kSlots] = {};
  std::mutex enqueue;  // one pipeline is enqueued at a time per device
};

Pipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

fos_status get_pipe(Pipe **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FOS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FOS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  Pipe &p = g_pipe[dev];
  if (!p.ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.up, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.down, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.end, ef) != cudaSuccess)
      return FOS_ERR_CUDA;
    for (int i = 0; i < kSlots; ++i)
      if (cudaEventCreateWithFlags(&p.in_ready[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.computed[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.freed[i], ef) != cudaSuccess)
        return FOS_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return FOS_OK;
}

// n rows of `width` bytes at `pitch` bytes apart (the same pitch on both sides).
cudaError_t copy_rows(void *dst, const void *src, size_t pitch, size_t width, int64_t n,
                      cudaMemcpyKind kind, cudaStream_t s) {
  if (pitch == width) return cudaMemcpyAsync(dst, src, (size_t)n * pitch, kind, s);
  return cudaMemcpy2DAsync(dst, pitch, src, pitch, width, (size_t)n, kind, s);
}

}  // namespace
}  // namespace fos

using namespace fos;

extern "C" size_t fos_step_host_workspace_bytes(const fos_desc *desc, fos_dtype dtype,
                                                int64_t chunk_rows) {
  if (check_desc(desc) != FOS_OK || dtype_size(dtype) == 0 || chunk_rows < 0) return 0;
  if (desc->rows == 0) return 0;
  return layout(desc, dtype_size(dtype), chunk_rows).total;
}

extern "C" fos_status fos_softmax_step_host(const fos_desc *desc, fos_dtype dtype,
                                            const void *scores, const void *dprobs, void *probs,
                                            float *lse, void *dscores, float *delta,
                                            float *d_sink, void *workspace,
                                            size_t workspace_bytes, int64_t chunk_rows,
                                            cudaStream_t stream, const fos_launch *launch) {
  fos_status st = check_desc(desc);
  if (st != FOS_OK) return st;
  if ((st = check_launch(launch)) != FOS_OK) return st;
  const int esz = dtype_size(dtype);
  if (esz == 0 || chunk_rows < 0) return FOS_ERR_INVALID;
  if (d_sink != nullptr && desc->sink == nullptr) return FOS_ERR_INVALID;
  if (desc->rows == 0) return FOS_OK;  // nothing to do; empty buffers may be null
  if (scores == nullptr || dprobs == nullptr || probs == nullptr || lse == nullptr ||
      dscores == nullptr || delta == nullptr)
    return FOS_ERR_INVALID;
  const Layout lay = layout(desc, esz, chunk_rows);
  if (workspace == nullptr || workspace_bytes < lay.total ||
      (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
    return FOS_ERR_INVALID;
  Pipe *p = nullptr;
  if ((st = get_pipe(&p)) != FOS_OK) return st;
  std::lock_guard<std::mutex> lock(p->enqueue);

  unsigned char *ws = static_cast<unsigned char *>(workspace);
  float *d_lse = reinterpret_cast<float *>(ws + lay.lse);
  float *d_delta = reinterpret_cast<float *>(ws + lay.delta);
  float *d_dsink = reinterpret_cast<float *>(ws + lay.dsink);
  const size_t pitch = (size_t)desc->ld * esz, width = (size_t)desc->key_len * esz;
  const unsigned char *hs = static_cast<const unsigned char *>(scores);
  const unsigned char *hdp = static_cast<const unsigned char *>(dprobs);
  unsigned char *hp = static_cast<unsigned char *>(probs);
  unsigned char *hds = static_cast<unsigned char *>(dscores);

#define FOS_CU(call)                             \
  do {                                           \
    if ((call) != cudaSuccess) return FOS_ERR_CUDA; \
  } while (0)
  // everything the caller enqueued before (earlier use of the workspace included) comes first
  FOS_CU(cudaEventRecord(p->start, stream));
  FOS_CU(cudaStreamWaitEvent(p->up, p->start, 0));
  const int64_t rows = desc->rows;
  int64_t r0 = 0;
  for (int64_t c = 0; r0 < rows; ++c) {
    const int slot = (int)(c % kSlots);
    const int64_t n = (rows - r0 < lay.chunk) ? rows - r0 : lay.chunk;
    unsigned char *bx = ws + lay.slot0 + (size_t)slot * 2 * lay.tensor;  // scores, then P
    unsigned char *bd = bx + lay.tensor;                                  // dP, then dScores
    const size_t off = (size_t)r0 * pitch;
    if (c >= kSlots) FOS_CU(cudaStreamWaitEvent(p->up, p->freed[slot], 0));
    FOS_CU(copy_rows(bx, hs + off, pitch, width, n, cudaMemcpyHostToDevice, p->up));
    FOS_CU(copy_rows(bd, hdp + off, pitch, width, n, cudaMemcpyHostToDevice, p->up));
    FOS_CU(cudaEventRecord(p->in_ready[slot], p->up));

    FOS_CU(cudaStreamWaitEvent(stream, p->in_ready[slot], 0));
    if ((st = run_fwd(desc, dtype, r0, n, bx, bx, d_lse + r0, stream, launch)) != FOS_OK)
      return st;
    if ((st = run_bwd(desc, dtype, r0, n, bx, bd, bd, d_delta + r0, stream, launch)) != FOS_OK)
      return st;
    FOS_CU(cudaEventRecord(p->computed[slot], stream));

    FOS_CU(cudaStreamWaitEvent(p->down, p->computed[slot], 0));
    FOS_CU(copy_rows(hp + off, bx, pitch, width, n, cudaMemcpyDeviceToHost, p->down));
    FOS_CU(copy_rows(hds + off, bd, pitch, width, n, cudaMemcpyDeviceToHost, p->down));
    FOS_CU(cudaEventRecord(p->freed[slot], p->down));
    r0 += n;
  }
  // LSE and delta (4 bytes per row) follow the last chunk in one copy each
  FOS_CU(cudaMemcpyAsync(lse, d_lse, (size_t)rows * sizeof(float), cudaMemcpyDeviceToHost,
                         p->down));
  FOS_CU(cudaMemcpyAsync(delta, d_delta, (size_t)rows * sizeof(float), cudaMemcpyDeviceToHost,
                         p->down));
  if (d_sink != nullptr && desc->heads > 0) {
    if ((st = run_sink(desc, d_lse, d_delta, d_dsink, stream, launch)) != FOS_OK) return st;
    FOS_CU(cudaMemcpyAsync(d_sink, d_dsink, (size_t)desc->heads * sizeof(float),
                           cudaMemcpyDeviceToHost, stream));
  }
  // the caller's stream completes only after the last download
  FOS_CU(cudaEventRecord(p->end, p->down));
  FOS_CU(cudaStreamWaitEvent(stream, p->end, 0));
#undef FOS_CU
  return FOS_OK;
}

// ----------------------------------------------------------------- the allocation-free variant
//
// Some callers cannot allocate device memory for the step's workspace: a host application
// whose memory manager has already reserved the device memory it is allowed (a serving
// engine that pre-allocates its cache pool, a framework whose caching allocator must see every
// block), or a code path where cudaMalloc / cudaFree are not acceptable because cudaFree
// synchronises the device.  fos_softmax_step_host_static serves them with a fixed scratch
// array that is part of the library image: every GPU that loads the library holds it until the
// process exits.  Calls share it, so calls that overlap on the GPU (two streams with no order
// between them) race; calls on one stream are ordered.  Nothing in it needs to start at zero:
// every byte a call reads there was written earlier in the same call.

namespace fos {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)32 << 20;  // FOS_STEP_HOST_STATIC_SCRATCH_BYTES
static_assert(kStaticScratchBytes == FOS_STEP_HOST_STATIC_SCRATCH_BYTES, "header and library disagree");

static __device__ __align__(256) unsigned char g_step_scratch[kStaticScratchBytes];

// Device address of g_step_scratch per device, taken once with that device current (in host
// code the array's name is only a host-side stand-in).
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

fos_status static_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FOS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FOS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_step_scratch) != cudaSuccess || p == nullptr)
      return FOS_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FOS_OK;
}

}  // namespace
}  // namespace fos

extern "C" fos_status fos_softmax_step_host_static(const fos_desc *desc, fos_dtype dtype,
                                                   const void *scores, const void *dprobs,
                                                   void *probs, float *lse, void *dscores,
                                                   float *delta, float *d_sink,
                                                   int64_t chunk_rows, cudaStream_t stream,
                                                   const fos_launch *launch) {
  fos_status st = check_desc(desc);
  if (st != FOS_OK) return st;
  const int esz = dtype_size(dtype);
  if (esz == 0 || chunk_rows < 0) return FOS_ERR_INVALID;
  if (desc->rows == 0) {
    return fos_softmax_step_host(desc, dtype, scores, dprobs, probs, lse, dscores, delta, d_sink,
                                 nullptr, 0, chunk_rows, stream, launch);
  }
  int64_t chunk = chunk_rows;
  if (chunk == 0) {
    // the default chunk, shrunk until the whole workspace fits the static array (the
    // 256-byte rounding of the slots costs at most a few more rows)
    const size_t fixed = layout(desc, esz, 1).slot0;
    if (fixed >= kStaticScratchBytes) return FOS_ERR_UNSUPPORTED;
    const size_t row_bytes = (size_t)desc->ld * esz;
    const int64_t fit = (int64_t)((kStaticScratchBytes - fixed) / (2 * kSlots) / row_bytes);
    chunk = layout(desc, esz, 0).chunk;
    if (fit < chunk) chunk = fit;
    if (chunk < 1) chunk = 1;
    while (chunk > 1 && layout(desc, esz, chunk).total > kStaticScratchBytes) --chunk;
  }
  if (layout(desc, esz, chunk).total > kStaticScratchBytes) return FOS_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  if ((st = static_scratch(&scratch)) != FOS_OK) return st;
  return fos_softmax_step_host(desc, dtype, scores, dprobs, probs, lse, dscores, delta, d_sink,
                               scratch, kStaticScratchBytes, chunk, stream, launch);
}
