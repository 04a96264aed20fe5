// fos_fwd.cu -- forward kernel of the fixed-order row softmax (P and LSE), sm_103a.
//
// One CTA owns one complete row at a time ("[WS1][kernels] Add fixed-order joint-attention
// softmax for Qwen-Image", Summary: fixed-order online softmax).  CTAs are persistent: CTA c
// takes rows c, c + grid, c + 2*grid, ...  On the bulk-copy path every CTA keeps a ring of
// `stages` shared-memory row buffers; thread 0 refills a buffer with a 1-D TMA bulk copy as
// soon as the CTA is done with it, so several rows per CTA are in flight from HBM while the
// current one is computed.  Per row:
//
//   pass 1   warp w takes tiles w, w + nw, ...; per tile: lane max, xor-tree max m_t,
//            e_j = exp(x_j - m_t) kept in registers, ascending lane sum, xor-tree sum s_t.
//   merge    warp 0 folds the tile states left to right, from (sink_h, 1) or (-inf, 0):
//              M_t = max(M_{t-1}, m_t)
//              S_t = S_{t-1} * exp(M_{t-1} - M_t) + s_t * exp(m_t - M_t)
//            (the factors are formed lane-parallel; the fold itself is sequential), then
//            LSE = M + log S and, per tile, c_t = exp(m_t - M) / S.
//   pass 2   P_j = e_j * c_t, rounded once to the I/O dtype, 16-byte stores.
//
// Masked keys (causal bound, valid length, key mask, -inf input) enter as -inf, tiles past
// the row's last candidate key are neither read nor reduced, and their P is written as +0.
#include "fos_device.cuh"
#include "fos_internal.h"

namespace fos {
namespace {

constexpr int kKT = 4;             // tiles per warp whose e_j stay in registers
constexpr int kBarBytes = 128;     // room for up to 16 mbarriers at the start of smem

template <typename T>
__device__ __forceinline__ void mask_keys(float (&x)[8], int j0, int lim, const uint8_t *km) {
#pragma unroll
  for (int q = 0; q < kLaneKeys; ++q) {
    const int j = j0 + q;
    const bool v = (j < lim) && (km == nullptr || km[j] != 0);
    x[q] = v ? x[q] : -INFINITY;
  }
}

// Pass 1 for tile t: returns e_j in e and leaves (m_t, s_t) in tm/ts (lane 0).
template <typename T>
__device__ __forceinline__ void tile_stats(const unsigned char *stage, int t, int lane, int lim,
                                           const uint8_t *km, float (&e)[8], float *tm,
                                           float *ts) {
  const int j0 = t * kTileK + lane * kLaneKeys;
  float x[8];
  Io<T>::widen(Io<T>::lds(stage + (size_t)j0 * Io<T>::kEsz), x);
  mask_keys<T>(x, j0, lim, km);
  float m = x[0];
#pragma unroll
  for (int q = 1; q < kLaneKeys; ++q) m = fmaxf(m, x[q]);
  m = warp_max_xor(m);
  float s = 0.0f;
  if (m != -INFINITY) {
#pragma unroll
    for (int q = 0; q < kLaneKeys; ++q) {
      e[q] = exp_fos(__fsub_rn(x[q], m));
      s = __fadd_rn(s, e[q]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < kLaneKeys; ++q) e[q] = 0.0f;
  }
  s = warp_sum_xor(s);
  if (lane == 0) {
    tm[t] = m;
    ts[t] = s;
  }
}

// e_j of tile t again, from the staged row and the stored tile maximum (same bits as pass 1).
template <typename T>
__device__ __forceinline__ void tile_exp(const unsigned char *stage, int t, int lane, int lim,
                                         const uint8_t *km, float m, float (&e)[8]) {
  const int j0 = t * kTileK + lane * kLaneKeys;
  float x[8];
  Io<T>::widen(Io<T>::lds(stage + (size_t)j0 * Io<T>::kEsz), x);
  mask_keys<T>(x, j0, lim, km);
#pragma unroll
  for (int q = 0; q < kLaneKeys; ++q) e[q] = (m != -INFINITY) ? exp_fos(__fsub_rn(x[q], m)) : 0.0f;
}

// Copy keys [0, lim) of a row into the stage with plain loads (unaligned or forced path).
template <typename T>
__device__ __forceinline__ void plain_stage(unsigned char *stage, const unsigned char *src,
                                            int lim, bool vec) {
  constexpr int esz = Io<T>::kEsz;
  int start = 0;
  if (vec) {
    const int n16 = (lim * esz) >> 4;
    for (int c = threadIdx.x; c < n16; c += blockDim.x)
      reinterpret_cast<uint4 *>(stage)[c] = reinterpret_cast<const uint4 *>(src)[c];
    start = (n16 << 4) / esz;
  }
  for (int j = start + threadIdx.x; j < lim; j += blockDim.x) {
    if (esz == 4)
      reinterpret_cast<uint32_t *>(stage)[j] = reinterpret_cast<const uint32_t *>(src)[j];
    else
      reinterpret_cast<uint16_t *>(stage)[j] = reinterpret_cast<const uint16_t *>(src)[j];
  }
}

template <typename T>
__device__ __forceinline__ void issue_row(const FwdArgs &a, int64_t rr, unsigned char *stage,
                                          uint64_t *bar) {
  constexpr int esz = Io<T>::kEsz;
  int b, h;
  const int lim = row_limit(rr, a.L, a.heads, a.q_len, a.causal, a.kv_valid_len, &b, &h);
  // Rounded up to 16 bytes; never past the row since L * esz is a multiple of 16 here.
  const uint32_t bytes = ((uint32_t)lim * esz + 15u) & ~15u;
  const uint32_t bar_a = smem_addr(bar);
  mbar_arrive_expect_tx(bar_a, bytes);
  if (bytes)
    bulk_g2s(smem_addr(stage),
             static_cast<const unsigned char *>(a.scores) + (size_t)rr * a.ld * esz, bytes,
             bar_a);
}

template <typename T>
__global__ void __launch_bounds__(512, 1) fos_fwd_kernel(const FwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
  unsigned char *ring = smem + kBarBytes;
  float *tm = reinterpret_cast<float *>(ring + (size_t)a.stages * a.stage_bytes);
  float *ts = tm + a.T;
  float *tc = ts + a.T;

  const int tid = threadIdx.x;
  const int nw = blockDim.x >> 5;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t r0 = blockIdx.x;
  if (r0 >= a.rows) return;
  const int64_t nmine = (a.rows - 1 - r0) / G + 1;
  const int NS = a.stages;
  const bool stall = a.test_stall && blockIdx.x == 0;
  int64_t issued_end = 0;  // rows [0, issued_end) of this CTA have had their copy issued

  if (a.use_bulk) {
    if (tid == 0) {
      for (int s = 0; s < NS; ++s) mbar_init(smem_addr(&bars[s]), 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      for (int64_t kk = 0; kk < nmine && kk < NS; ++kk)
        if (!(stall && kk == 0)) issue_row<T>(a, r0 + kk * G, ring + (size_t)kk * a.stage_bytes, &bars[kk]);
    }
    issued_end = nmine < NS ? nmine : NS;
  }

  for (int64_t k = 0; k < nmine; ++k) {
    const int64_t r = r0 + k * G;
    const int s = a.use_bulk ? (int)(k % NS) : 0;
    unsigned char *stage = ring + (size_t)s * a.stage_bytes;
    int b, h;
    const int lim = row_limit(r, a.L, a.heads, a.q_len, a.causal, a.kv_valid_len, &b, &h);
    const int Te = (lim + kTileK - 1) / kTileK;
    const uint8_t *km = a.key_mask ? a.key_mask + (int64_t)b * a.L : nullptr;
    const bool in_regs = Te <= nw * kKT;

    bool timed_out = false;
    if (a.use_bulk) {
      timed_out = !mbar_wait_bounded(smem_addr(&bars[s]), (uint32_t)((k / NS) & 1), a.timeout_ns);
    } else {
      plain_stage<T>(stage, static_cast<const unsigned char *>(a.scores) + (size_t)r * a.ld * esz,
                     lim, a.in_vec != 0);
      __syncthreads();
    }

    // ---- pass 1: tile statistics
    float e[kKT][8];
    if (in_regs) {
#pragma unroll
      for (int kk = 0; kk < kKT; ++kk) {
        const int t = w + kk * nw;
        if (t < Te) tile_stats<T>(stage, t, lane, lim, km, e[kk], tm, ts);
      }
    } else {
      for (int t = w; t < Te; t += nw) {
        float tmp[8];
        tile_stats<T>(stage, t, lane, lim, km, tmp, tm, ts);
      }
    }

    if (__syncthreads_or(timed_out)) {
      // A copy never landed: record it, let the copies still in flight land, stop.
      if (tid == 0) {
        raise_device_error(a.err, kDevErrTimeout);
        for (int64_t kk = k; kk < issued_end; ++kk) {
          if (stall && kk == 0) continue;
          mbar_wait_bounded(smem_addr(&bars[kk % NS]), (uint32_t)((kk / NS) & 1), a.timeout_ns);
        }
      }
      return;
    }

    // The stage is free once pass 1 has read it (when e_j stayed in registers).
    if (a.use_bulk && in_regs && tid == 0 && k + NS < nmine) {
      issue_row<T>(a, r0 + (k + NS) * G, stage, &bars[s]);
      issued_end = k + NS + 1;
    }

    // ---- merge (warp 0): ordered fold of the tile states, LSE, per-tile output scale
    if (w == 0) {
      const bool has_sink = a.sink != nullptr;
      float M = has_sink ? a.sink[h] : -INFINITY;
      float S = has_sink ? 1.0f : 0.0f;
      for (int base = 0; base < Te; base += 32) {
        const int t = base + lane;
        const float mt = t < Te ? tm[t] : -INFINITY;
        const float st = t < Te ? ts[t] : 0.0f;
        float pm = mt;  // inclusive prefix maximum inside this group of 32 tiles
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(kFull, pm, o);
          if (lane >= o) pm = fmaxf(pm, y);
        }
        pm = fmaxf(pm, M);                      // M_t
        float prev = __shfl_up_sync(kFull, pm, 1);
        if (lane == 0) prev = M;                // M_{t-1}
        const float alpha = scale_fos(prev, pm);
        const float beta = (mt == -INFINITY) ? 0.0f : __fmul_rn(st, scale_fos(mt, pm));
        const int n = min(32, Te - base);
        for (int q = 0; q < n; ++q) {
          const float aq = __shfl_sync(kFull, alpha, q);
          const float bq = __shfl_sync(kFull, beta, q);
          S = __fadd_rn(__fmul_rn(S, aq), bq);
        }
        M = __shfl_sync(kFull, pm, n - 1);
      }
      for (int t = lane; t < Te; t += 32) {
        const float mt = tm[t];
        tc[t] = (mt == -INFINITY) ? 0.0f : __fdiv_rn(scale_fos(mt, M), S);
      }
      if (lane == 0) a.lse[r] = (M == -INFINITY) ? -INFINITY : __fadd_rn(M, logf(S));
    }
    __syncthreads();

    // ---- pass 2: P = e * c_t, one rounding, 16-byte stores
    unsigned char *prow = static_cast<unsigned char *>(a.probs) + (size_t)r * a.ld * esz;
    const bool ovec = a.out_vec != 0;
    if (in_regs) {
#pragma unroll
      for (int kk = 0; kk < kKT; ++kk) {
        const int t = w + kk * nw;
        if (t < Te) {
          const float c = tc[t];
          float v[8];
#pragma unroll
          for (int q = 0; q < kLaneKeys; ++q) v[q] = __fmul_rn(e[kk][q], c);
          store_lane8<T>(prow, t * kTileK + lane * kLaneKeys, a.L, ovec, v);
        }
      }
    } else {
      for (int t = w; t < Te; t += nw) {
        float ee[8], v[8];
        tile_exp<T>(stage, t, lane, lim, km, tm[t], ee);
        const float c = tc[t];
#pragma unroll
        for (int q = 0; q < kLaneKeys; ++q) v[q] = __fmul_rn(ee[q], c);
        store_lane8<T>(prow, t * kTileK + lane * kLaneKeys, a.L, ovec, v);
      }
    }
    for (int t = Te + w; t < a.T; t += nw) {
      float z[8];
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) z[q] = 0.0f;
      store_lane8<T>(prow, t * kTileK + lane * kLaneKeys, a.L, ovec, z);
    }

    if (!in_regs) {
      __syncthreads();  // everyone is done with the stage and the tile maxima
      if (a.use_bulk && tid == 0 && k + NS < nmine) {
        issue_row<T>(a, r0 + (k + NS) * G, stage, &bars[s]);
        issued_end = k + NS + 1;
      }
    }
  }
}

template <typename T>
const void *fwd_fn() {
  return reinterpret_cast<const void *>(&fos_fwd_kernel<T>);
}

const void *fwd_fn(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return fwd_fn<float>();
    case FOS_BF16: return fwd_fn<__nv_bfloat16>();
    case FOS_F16: return fwd_fn<__half>();
  }
  return nullptr;
}

}  // namespace

size_t fwd_extra_smem(int T, int stages) {
  (void)stages;
  return (size_t)kBarBytes + (size_t)3 * T * sizeof(float);
}

cudaError_t fwd_prepare(fos_dtype dt, int max_smem) {
  return cudaFuncSetAttribute(fwd_fn(dt), cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

cudaError_t fwd_occupancy(fos_dtype dt, int threads, size_t smem, int *blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fwd_fn(dt), threads, smem);
}

cudaError_t fwd_launch(fos_dtype dt, const FwdArgs &a, int grid, int threads, size_t smem,
                       cudaStream_t s) {
  switch (dt) {
    case FOS_F32: fos_fwd_kernel<float><<<grid, threads, smem, s>>>(a); break;
    case FOS_BF16: fos_fwd_kernel<__nv_bfloat16><<<grid, threads, smem, s>>>(a); break;
    case FOS_F16: fos_fwd_kernel<__half><<<grid, threads, smem, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace fos
