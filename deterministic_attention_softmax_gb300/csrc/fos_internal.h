// fos_internal.h -- host/device interface between the C ABI (fos_api.cu) and the kernel
// translation units.  Not installed; the public interface is include/fos_softmax.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/fos_softmax.h"

namespace fos {

constexpr int kTileK = 256;  // keys per tile: part of the arithmetic contract

// n / d for 32-bit unsigned n by a multiply-high and two shifts, d fixed and at least 1:
// Granlund and Montgomery, "Division by invariant integers using multiplication" (1994),
// Figure 4.1.  l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, s1 = min(l, 1),
// s2 = max(l - 1, 0); then t = mulhi(m, n) and n / d = (t + ((n - t) >> s1)) >> s2.
struct FastDiv {
  uint32_t m, s1, s2;
};

inline FastDiv make_fastdiv(uint32_t d) {
  if (d < 1) d = 1;
  uint32_t l = 0;
  while (l < 32 && (1ull << l) < d) ++l;
  FastDiv f;
  f.m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
  f.s1 = l > 0 ? 1u : 0u;
  f.s2 = l > 0 ? l - 1 : 0u;
  return f;
}

// n / d with the constants of make_fastdiv (exact for every 32-bit n).
__host__ __device__ inline uint32_t fast_div(uint32_t n, const FastDiv &f) {
#if defined(__CUDA_ARCH__)
  const uint32_t t = __umulhi(n, f.m);
#else
  const uint32_t t = (uint32_t)(((uint64_t)n * f.m) >> 32);
#endif
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// Geometry and masks shared by the forward and backward row kernels.
struct RowArgs {
  int64_t rows;                // rows of this launch
  int64_t row_base;            // problem row of local row 0 (a launch may cover a row range)
  int64_t ld;                  // elements between row starts
  int32_t L;                   // key length
  int32_t heads, q_len, causal;
  const int32_t *kv_valid_len; // [batch] or null
  const uint8_t *key_mask;     // [batch * L] or null
  int32_t T;                   // tiles per row, ceil(L / 256)
  int32_t stages;              // rows (or row segments) in flight per CTA; 1 on the plain path
  uint32_t stage_bytes;        // shared-memory bytes of one stage: T * 256 * esz for a whole
                               // row, seg_tiles * 256 * esz for the streaming kernels
  int32_t seg_tiles;           // streaming kernels: tiles per segment (0: whole rows)
  int32_t use_bulk;            // 1: 1-D bulk copies (TMA) into the ring; 0: plain loads
  int32_t in_vec;              // input rows start 16-byte aligned
  int32_t out_vec;             // output rows start 16-byte aligned
  uint64_t timeout_ns;         // limit of every bounded wait
  int32_t test_stall;          // test only: CTA 0 never issues its first copy
  int32_t need_geo;            // rows need b / h / limit (a mask or a sink is given)
  int32_t geo32;               // row_base + rows fits in int32: 32-bit geometry arithmetic
  FastDiv qdiv, hdiv;          // 32-bit division by q_len and by heads
  unsigned *err;               // device error word
};

struct FwdArgs : RowArgs {
  const void *scores;
  void *probs;
  float *lse;
  const float *sink;   // [heads] or null
  int32_t keep_e;      // CTA kernel: e_j are kept between the passes (every warp has at most
                       // KT tiles); otherwise they are recomputed in the second pass
  uint32_t tmem_cols;  // tensor-memory columns a CTA allocates to keep them in; 0 when none
                       // (two tiles per warp stay in registers)
  int32_t group_warps; // group kernel: compute warps per row group (blockDim / 32 / groups)
};

// Tensor-memory columns per SM, and the columns a forward CTA of `warps` compute warps with
// `kt` tiles per warp allocates (a power of two, at least 32).
constexpr uint32_t kTmemColsPerSm = 512;
uint32_t fwd_tmem_cols(int warps, int kt);

struct BwdArgs : RowArgs {
  const void *probs;
  const void *dprobs;
  void *dscores;
  float *delta;  // [rows] or null
  // The sink gradient fused into the backward: rows are taken by octets, 8 consecutive
  // positions (b, i) of one head (octet o: head o / oct_per_head, positions 8m .. 8m + 7 with
  // m = o % oct_per_head, those below pos_end), and each octet's ascending float32 sum of
  // c_r = -(exp(sink_h - lse_r) * delta_r) is written to oct_sums[o].
  const float *lse;       // [rows]
  const float *sink;      // [heads]
  float *oct_sums;        // [heads * oct_per_head]
  int64_t oct_per_head;   // ceil(batch * q_len / 8)
  int64_t pos_end;        // batch * q_len
  FastDiv octdiv;         // division by oct_per_head
  int32_t oct32;          // octet indices and positions fit 32 bits
};

struct SinkArgs {
  int32_t batch, heads, q_len;
  const float *sink;
  const float *lse;
  const float *delta;
  float *d_sink;
  FastDiv qdiv;   // division by q_len
  int32_t pos32;  // batch * q_len < 2^32: positions divide in 32 bits
};

// The fields of SinkArgs every sink launch shares.
inline void fill_sink_args(const fos_desc *d, SinkArgs *a) {
  a->batch = d->batch;
  a->heads = d->heads;
  a->q_len = d->q_len;
  a->sink = d->sink;
  a->qdiv = make_fastdiv((uint32_t)d->q_len);
  a->pos32 = ((int64_t)d->batch * d->q_len < ((int64_t)1 << 32)) ? 1 : 0;
}

// Shared memory used by a row kernel besides its ring of staged rows.
size_t fwd_extra_smem(int T, int stages);
size_t fwd_stream_extra_smem(int T, int stages);  // the streaming forward (merge warp)
size_t bwd_extra_smem(int T, int stages);

// Kernel instances per dtype: set the dynamic shared-memory limit, query residency, launch.
// The forward parks e_j of `kt` tiles per warp (kt = 2, 4, 6 or 8) in tensor memory between
// its passes when a.tmem_cols is set; `fast` selects the instance specialised for the common
// case (same arithmetic).
int fwd_tiles_per_warp(int T, int warps);
// Default compute warps per CTA (1..16).
int fwd_default_warps(int T);
int bwd_default_warps(int T);
cudaError_t fwd_prepare(fos_dtype dt, int max_smem);
// Registers, static shared memory and limits of a forward CTA instance (its residency is
// computed on the host: the runtime's query counts a kernel that allocates tensor memory as
// filling its SM).
cudaError_t fwd_attributes(fos_dtype dt, int kt, bool fast, cudaFuncAttributes *fa);
cudaError_t fwd_launch(fos_dtype dt, int kt, bool fast, const FwdArgs &a, int grid, int threads,
                       size_t smem, cudaStream_t s);
// Several row groups per CTA (each `a.group_warps` warps, one row at a time, its own ring of
// a.stages buffers, no producer warp); kt = 4, 6 or 8 tiles per warp parked in tensor memory.
size_t fwd_group_smem(int groups, int stages, size_t stage_bytes, int T);
cudaError_t fwd_group_attributes(fos_dtype dt, int kt, bool fast, cudaFuncAttributes *fa);
cudaError_t fwd_group_launch(fos_dtype dt, int kt, bool fast, const FwdArgs &a, int grid,
                             int threads, size_t smem, cudaStream_t s);
// Rows of at most 8 tiles, one warp per row: kt = 2, 4 or 8 tiles parked in a.tmem_cols
// tensor-memory columns; `warps` warps per CTA, each with a.stages row buffers of
// a.stage_bytes.
size_t fwd_rowwarp_smem(int warps, int stages, size_t stage_bytes);
cudaError_t fwd_rowwarp_attributes(fos_dtype dt, int kt, cudaFuncAttributes *fa);
cudaError_t fwd_rowwarp_launch(fos_dtype dt, int kt, const FwdArgs &a, int grid, int threads,
                               size_t smem, cudaStream_t s);
// Rows longer than shared memory: segments of a.seg_tiles tiles, each read twice.
cudaError_t fwd_stream_occupancy(fos_dtype dt, int threads, size_t smem, int *blocks_per_sm);
cudaError_t fwd_stream_launch(fos_dtype dt, const FwdArgs &a, int grid, int threads, size_t smem,
                              cudaStream_t s);

cudaError_t bwd_prepare(fos_dtype dt, int max_smem);
cudaError_t bwd_occupancy(fos_dtype dt, bool fast, int threads, size_t smem, int *blocks_per_sm);
// `sink`: the instance that takes rows by octets and writes their sink-gradient sums.
cudaError_t bwd_launch(fos_dtype dt, bool fast, const BwdArgs &a, int grid, int threads,
                       size_t smem, cudaStream_t s, bool sink = false);
// Short rows, one warp per row (P and dP of a row per buffer; T4 floats of partials per warp).
size_t bwd_rowwarp_smem(int warps, int stages, size_t stage_bytes, int T);
cudaError_t bwd_rowwarp_occupancy(fos_dtype dt, int threads, size_t smem, int *blocks_per_sm);
cudaError_t bwd_rowwarp_launch(fos_dtype dt, const BwdArgs &a, int grid, int threads, size_t smem,
                               cudaStream_t s, bool sink = false);
cudaError_t bwd_stream_occupancy(fos_dtype dt, int threads, size_t smem, int *blocks_per_sm);
cudaError_t bwd_stream_launch(fos_dtype dt, const BwdArgs &a, int grid, int threads, size_t smem,
                              cudaStream_t s);

cudaError_t sink_launch(const SinkArgs &a, int threads, cudaStream_t s);
// d_sink from the octet sums the fused backward wrote (the chunk tree and left-to-right sum of
// sink_launch on them).
cudaError_t sink_merge_launch(const SinkArgs &a, const float *oct_sums, int64_t oct_per_head,
                              int threads, cudaStream_t s);
// Chunk partials of the batch entries [b0, b1) (arrays hold their rows from b0 * heads * q_len).
cudaError_t sink_partials_launch(const SinkArgs &a, int64_t b0, int64_t b1, float *partials,
                                 int threads, cudaStream_t s);

// The QK contraction (fos_qk.cu): dynamic shared memory of a CTA, and the launch on validated
// arguments (err: the device error word).
size_t qk_smem_bytes(int head_dim, int tile_n);
fos_status run_qk(const fos_qk_desc *d, fos_dtype in_dt, fos_dtype out_dt, const void *q,
                  const void *k, void *scores, cudaStream_t stream, unsigned *err, int max_smem,
                  int sms);

// The PV contraction (fos_pv.cu), as the QK one.
size_t pv_smem_bytes(int head_dim);
fos_status run_pv(const fos_pv_desc *d, fos_dtype in_dt, fos_dtype out_dt, const void *p,
                  const void *v, void *out, cudaStream_t stream, unsigned *err, int max_smem);
// The key / value gradient contraction (fos_kvgrad.cu): out = scale * a^T m per key head, the
// group's query heads and positions accumulated in order.
size_t kvgrad_smem_bytes(int head_dim);
fos_status run_kvgrad(const fos_pv_desc *d, fos_dtype in_dt, fos_dtype out_dt, const void *a,
                      const void *m, void *out, cudaStream_t stream, unsigned *err, int max_smem);

// Host-side checks shared by the C ABI entry points (fos_api.cu).
int dtype_size(fos_dtype dt);
fos_status check_desc(const fos_desc *d);
fos_status check_launch(const fos_launch *l);

// The three operations on already validated arguments.  run_fwd / run_bwd cover rows
// [row_base, row_base + nrows) of the problem in d; their array pointers address local row 0
// of that range (lse / delta included), while masks and sink keep their problem-wide indexing.
fos_status run_fwd(const fos_desc *d, fos_dtype dt, int64_t row_base, int64_t nrows,
                   const void *scores, void *probs, float *lse, cudaStream_t s,
                   const fos_launch *l);
// With oct_sums (and lse) given, the backward may also take the sink gradient's octet sums
// (rows taken by octets; whole problem only, row_base 0); *fused tells whether it did.  When
// it did not and delta is null, delta is written to oct_sums instead (which must then hold
// nrows floats).
fos_status run_bwd(const fos_desc *d, fos_dtype dt, int64_t row_base, int64_t nrows,
                   const void *probs, const void *dprobs, void *dscores, float *delta,
                   cudaStream_t s, const fos_launch *l, const float *lse = nullptr,
                   float *oct_sums = nullptr, bool *fused = nullptr);
fos_status run_sink(const fos_desc *d, const float *lse, const float *delta, float *d_sink,
                    cudaStream_t s, const fos_launch *l);

}  // namespace fos
