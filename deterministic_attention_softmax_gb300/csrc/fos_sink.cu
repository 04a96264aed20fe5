// fos_sink.cu -- per-head sink-logit gradient, reduced in a fixed order without atomics.
//
// "[ROCm] Jax Add softmax sink (learnable off-by-one) support": one sink logit per head,
// shared by every batch entry, whose gradient is summed per head over batch and query rows
// (the CK kernels there zero d_sink and accumulate with atomicAdd).  Here one CTA owns one
// head and walks that head's rows in (b, i) order in chunks of 256:
//
//   c_r        = -(exp(sink_h - lse_r) * delta_r)        (0 when sink_h is -inf)
//   chunk q    = xor-tree sum over lanes of the ascending lane sums of c over rows
//                256q + 8l .. 256q + 8l + 7
//   d_sink[h]  = chunk partials added left to right
//
// Warps take the chunks of one round in parallel; thread 0 adds the round's partials in
// chunk order, so the result does not depend on the number of warps.  For rows sharded by
// batch entry, fos_sink_partials_kernel writes the chunk partials of one shard instead; the
// shards' partials, concatenated in chunk order and added left to right (fos_sink_grad_merge),
// give these bits.
#include "fos_device.cuh"
#include "fos_internal.h"

namespace fos {
namespace {

// Chunk c of head h (positions 256c .. 256c+255 of the head's rows in (b, i) order, those
// below `pos_end`): the xor-tree sum of the lanes' ascending sums of c_r.  Rows are read at
// r - row_base (the arrays may hold a range of rows that starts at row_base).
__device__ __forceinline__ float sink_chunk(const SinkArgs &a, int h, float sk, int64_t c,
                                            int64_t pos_end, int64_t row_base, int lane) {
  float acc = 0.0f;
#pragma unroll
  for (int q = 0; q < kLaneKeys; ++q) {
    const int64_t p = c * kTileK + lane * kLaneKeys + q;
    if (p < pos_end) {
      int64_t b;
      if (a.pos32) {
        b = fast_div((uint32_t)p, a.qdiv);
      } else {
        b = p / a.q_len;
      }
      const int64_t r = (b * a.heads + h) * a.q_len + (p - b * a.q_len) - row_base;
      const float ps = (sk == -INFINITY) ? 0.0f : scale_fos(sk, a.lse[r]);
      acc = __fadd_rn(acc, -__fmul_rn(ps, a.delta[r]));
    }
  }
  return warp_sum_xor(acc);
}

// The chunk partials of one shard: batch entries [b0, b1), whose rows the arrays hold from row
// b0 * heads * q_len on.  partials[h * (c1 - c0) + k] = chunk c0 + k of head h, where
// [c0, c1) are the chunks of positions [b0 * q_len, b1 * q_len).
__global__ void __launch_bounds__(1024) fos_sink_partials_kernel(const SinkArgs a, int64_t b0,
                                                                 int64_t b1, float *partials) {
  const int h = blockIdx.x;
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int64_t p0 = b0 * a.q_len, p1 = b1 * a.q_len;
  const int64_t c0 = p0 / kTileK, c1 = (p1 + kTileK - 1) / kTileK;
  const int64_t row_base = b0 * a.heads * a.q_len;
  const float sk = a.sink[h];
  for (int64_t c = c0 + w; c < c1; c += nw) {
    const float v = sink_chunk(a, h, sk, c, p1, row_base, lane);
    if (lane == 0) partials[(int64_t)h * (c1 - c0) + (c - c0)] = v;
  }
}

__global__ void __launch_bounds__(1024) fos_sink_kernel(const SinkArgs a) {
  __shared__ float part[32];
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  const int nw = blockDim.x >> 5;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int64_t n = (int64_t)a.batch * a.q_len;  // rows of this head
  const int64_t nchunks = (n + kTileK - 1) / kTileK;
  const float sk = a.sink[h];
  float total = 0.0f;

  for (int64_t base = 0; base < nchunks; base += nw) {
    const int64_t c = base + w;
    if (c < nchunks) {
      const float acc = sink_chunk(a, h, sk, c, n, 0, lane);
      if (lane == 0) part[w] = acc;
    }
    __syncthreads();
    if (tid == 0) {
      for (int q = 0; q < nw && base + q < nchunks; ++q) total = __fadd_rn(total, part[q]);
    }
    __syncthreads();
  }
  if (tid == 0) a.d_sink[h] = total;
}

// d_sink from the octet sums the backward wrote when it took the sink gradient along: lane l
// of chunk c holds octet 32c + l's sum (+0 past the head's last octet), which is that lane's
// ascending sum in sink_chunk, so the tree and the left-to-right chunk sum below give the bits
// of fos_sink_kernel.
__global__ void __launch_bounds__(1024) fos_sink_merge_kernel(const SinkArgs a,
                                                              const float *oct_sums,
                                                              int64_t oct_per_head) {
  __shared__ float part[32];
  const int h = blockIdx.x;
  const int tid = threadIdx.x;
  const int nw = blockDim.x >> 5;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int64_t nchunks = (oct_per_head + 31) / 32;
  const float *os = oct_sums + (int64_t)h * oct_per_head;
  float total = 0.0f;
  for (int64_t base = 0; base < nchunks; base += nw) {
    const int64_t c = base + w;
    if (c < nchunks) {
      const int64_t m = c * 32 + lane;
      const float acc = warp_sum_xor(m < oct_per_head ? os[m] : 0.0f);
      if (lane == 0) part[w] = acc;
    }
    __syncthreads();
    if (tid == 0) {
      for (int q = 0; q < nw && base + q < nchunks; ++q) total = __fadd_rn(total, part[q]);
    }
    __syncthreads();
  }
  if (tid == 0) a.d_sink[h] = total;
}

}  // namespace

cudaError_t sink_merge_launch(const SinkArgs &a, const float *oct_sums, int64_t oct_per_head,
                              int threads, cudaStream_t s) {
  fos_sink_merge_kernel<<<a.heads, threads, 0, s>>>(a, oct_sums, oct_per_head);
  return cudaGetLastError();
}

cudaError_t sink_launch(const SinkArgs &a, int threads, cudaStream_t s) {
  fos_sink_kernel<<<a.heads, threads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t sink_partials_launch(const SinkArgs &a, int64_t b0, int64_t b1, float *partials,
                                 int threads, cudaStream_t s) {
  fos_sink_partials_kernel<<<a.heads, threads, 0, s>>>(a, b0, b1, partials);
  return cudaGetLastError();
}

}  // namespace fos
