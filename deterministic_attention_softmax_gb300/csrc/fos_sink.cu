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
// chunk order, so the result does not depend on the number of warps.
#include "fos_device.cuh"
#include "fos_internal.h"

namespace fos {
namespace {

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
      float acc = 0.0f;
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) {
        const int64_t p = c * kTileK + lane * kLaneKeys + q;
        if (p < n) {
          const int64_t r = ((p / a.q_len) * a.heads + h) * a.q_len + (p % a.q_len);
          const float ps = (sk == -INFINITY) ? 0.0f : scale_fos(sk, a.lse[r]);
          acc = __fadd_rn(acc, -__fmul_rn(ps, a.delta[r]));
        }
      }
      acc = warp_sum_xor(acc);
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

cudaError_t sink_launch(const SinkArgs &a, int threads, cudaStream_t s) {
  fos_sink_kernel<<<a.heads, threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace fos
