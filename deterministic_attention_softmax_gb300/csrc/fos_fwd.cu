// fos_fwd.cu -- forward kernel of the fixed-order row softmax (P and LSE), sm_103a.
//
// One CTA owns one complete row at a time ("[WS1][kernels] Add fixed-order joint-attention
// softmax for Qwen-Image", Summary: fixed-order online softmax).  CTAs are persistent: CTA c
// takes rows c, c + grid, c + 2*grid, ...  On the bulk-copy path every CTA keeps a ring of
// `stages` shared-memory row buffers; thread 0 refills a buffer with a 1-D TMA bulk copy as
// soon as the CTA is done with it (and writes that row's geometry next to it), so several
// rows per CTA are in flight from HBM while the current one is computed.  Per row:
//
//   pass 1   warp w takes tiles w, w + nw, ...; per tile: lane max, xor-tree max m_t,
//            e_j = exp(x_j - m_t), ascending lane sum, xor-tree sum s_t.
//   merge    warp 0 folds the tile states left to right, from (sink_h, 1) or (-inf, 0):
//              M_t = max(M_{t-1}, m_t)
//              S_t = S_{t-1} * exp(M_{t-1} - M_t) + s_t * exp(m_t - M_t)
//            (the factors are formed lane-parallel; the fold itself is sequential), then
//            LSE = M + log S and, per tile, c_t = exp(m_t - M) / S.
//   pass 2   P_j = e_j * c_t, rounded once to the I/O dtype, 16-byte stores.
//
// e_j stays in registers when every warp has at most KT tiles (the register mode, whose
// stage is refilled right after pass 1); longer rows recompute e_j from the staged row in
// pass 2 (same bits) and release their stage at the next row's first barrier.  Masked keys
// (causal bound, valid length, key mask, -inf input) enter as -inf; tiles past the row's last
// candidate key are neither read nor reduced, and their P is written as +0.
#include "fos_device.cuh"
#include "fos_internal.h"

namespace fos {
namespace {

constexpr int kBarBytes = 128;  // up to 16 mbarriers at the start of shared memory
constexpr int kGeoBytes = 256;  // up to 16 per-stage row records (int4) after them

__device__ __forceinline__ void mask_keys(float (&x)[8], int j0, int lim, const uint8_t *km) {
#pragma unroll
  for (int q = 0; q < kLaneKeys; ++q) {
    const int j = j0 + q;
    const bool v = (j < lim) && (km == nullptr || km[j] != 0);
    x[q] = v ? x[q] : -INFINITY;
  }
}

// The 8 keys of lane `lane` in tile t, widened, with masked keys set to -inf.  Per-key
// checks are only needed in the tile holding the row limit, or when a key mask is given.
template <typename T>
__device__ __forceinline__ void tile_keys(const unsigned char *stage, int t, int lane, int lim,
                                          const uint8_t *km, float (&x)[8]) {
  const int j0 = t * kTileK + lane * kLaneKeys;
  Io<T>::widen(Io<T>::lds(stage + (size_t)j0 * Io<T>::kEsz), x);
  if (km != nullptr || (t + 1) * kTileK > lim) mask_keys(x, j0, lim, km);
}

// Pass 1 for tile t: e_j into e and (m_t, s_t) into tm/ts (lane 0).  A tile with no valid
// key has m_t = -inf: its e_j are exp(-inf) = +0 and s_t = +0.
template <typename T>
__device__ __forceinline__ void tile_stats(const unsigned char *stage, int t, int lane, int lim,
                                           const uint8_t *km, float (&e)[8], float *tm,
                                           float *ts) {
  float x[8];
  tile_keys<T>(stage, t, lane, lim, km, x);
  float m = x[0];
#pragma unroll
  for (int q = 1; q < kLaneKeys; ++q) m = fmaxf(m, x[q]);
  m = warp_max_xor(m);
  const float mm = (m == -INFINITY) ? 0.0f : m;
  float s = 0.0f;
#pragma unroll
  for (int q = 0; q < kLaneKeys; ++q) {
    e[q] = exp_fos(__fsub_rn(x[q], mm));
    s = __fadd_rn(s, e[q]);
  }
  s = warp_sum_xor(s);
  if (lane == 0) {
    tm[t] = m;
    ts[t] = s;
  }
}

// e_j of tile t again from the staged row and the stored tile maximum (same bits as pass 1).
template <typename T>
__device__ __forceinline__ void tile_exp(const unsigned char *stage, int t, int lane, int lim,
                                         const uint8_t *km, float m, float (&e)[8]) {
  float x[8];
  tile_keys<T>(stage, t, lane, lim, km, x);
  const float mm = (m == -INFINITY) ? 0.0f : m;
#pragma unroll
  for (int q = 0; q < kLaneKeys; ++q) e[q] = exp_fos(__fsub_rn(x[q], mm));
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

// Thread 0: record row rr's geometry in geo and start its bulk copy into `stage`.
template <typename T>
__device__ __forceinline__ void issue_row(const FwdArgs &a, int64_t rr, unsigned char *stage,
                                          uint64_t *bar, int4 *geo, bool skip_copy) {
  constexpr int esz = Io<T>::kEsz;
  const int4 g = row_geometry(a, rr);
  *geo = g;
  // Rounded up to 16 bytes; never past the row since L * esz is a multiple of 16 here.
  const uint32_t bytes = ((uint32_t)g.x * esz + 15u) & ~15u;
  if (skip_copy) return;  // test only: this row's copy is never issued
  const uint32_t bar_a = smem_addr(bar);
  mbar_arrive_expect_tx(bar_a, bytes);  // release: the geometry record is visible to waiters
  if (bytes)
    bulk_g2s(smem_addr(stage),
             static_cast<const unsigned char *>(a.scores) + (size_t)rr * a.ld * esz, bytes,
             bar_a);
}

template <typename T, int KT>
__global__ void __maxnreg__(KT == 4 ? 80 : 128) fos_fwd_kernel(const FwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
  int4 *geos = reinterpret_cast<int4 *>(smem + kBarBytes);
  unsigned char *ring = smem + kBarBytes + kGeoBytes;
  float *tm = reinterpret_cast<float *>(ring + (size_t)a.stages * a.stage_bytes);
  float *ts = tm + a.T;
  float *tc = ts + a.T;
  float *ab = tc + a.T;  // merge factors: alpha at ab[0..31], beta at ab[32..63]

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
  const bool reg_mode = a.T <= nw * KT;  // every row's e_j fit in registers
  const bool defer = NS >= 2;            // outside register mode: refill one row later
  int64_t issued_end = 0;                // rows [0, issued_end) of this CTA have been issued

  if (a.use_bulk) {
    if (tid == 0) {
      for (int s = 0; s < NS; ++s) mbar_init(smem_addr(&bars[s]), 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0)
      for (int64_t kk = 0; kk < nmine && kk < NS; ++kk)
        issue_row<T>(a, r0 + kk * G, ring + (size_t)kk * a.stage_bytes, &bars[kk], &geos[kk],
                     stall && kk == 0);
    issued_end = nmine < NS ? nmine : NS;
  }

  for (int64_t k = 0; k < nmine; ++k) {
    const int64_t r = r0 + k * G;
    const int s = a.use_bulk ? (int)(k % NS) : 0;
    unsigned char *stage = ring + (size_t)s * a.stage_bytes;

    bool timed_out = false;
    int4 g;
    if (a.use_bulk) {
      timed_out = !mbar_wait_bounded(smem_addr(&bars[s]), (uint32_t)((k / NS) & 1), a.timeout_ns);
      g = geos[s];
    } else {
      if (tid == 0) geos[0] = row_geometry(a, r);
      __syncthreads();  // also: every warp is done with the previous row's stage
      g = geos[0];
      plain_stage<T>(stage, static_cast<const unsigned char *>(a.scores) + (size_t)r * a.ld * esz,
                     g.x, a.in_vec != 0);
      __syncthreads();
    }
    const int lim = g.x;
    const int Te = (lim + kTileK - 1) / kTileK;
    const uint8_t *km = a.key_mask ? a.key_mask + (int64_t)g.y * a.L : nullptr;

    // ---- pass 1: tile statistics
    float e[KT][8];
    if (reg_mode) {
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
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

    // Refill a free stage: this row's in register mode (pass 1 was its last reader); with
    // two or more stages, the previous row's (its pass 2 ended before this barrier); with a
    // single stage outside register mode, this row's after an end-of-row barrier below.
    if (a.use_bulk && tid == 0 && (reg_mode || defer)) {
      const int64_t kr = reg_mode ? k : k - 1;
      if (kr >= 0 && kr + NS < nmine) {
        const int sr = (int)(kr % NS);
        issue_row<T>(a, r0 + (kr + NS) * G, ring + (size_t)sr * a.stage_bytes, &bars[sr],
                     &geos[sr], false);
        issued_end = kr + NS + 1;
      }
    }

    // ---- merge (warp 0): ordered fold of the tile states, LSE, per-tile output scale
    if (w == 0) {
      const bool has_sink = a.sink != nullptr;
      float M = has_sink ? a.sink[g.z] : -INFINITY;
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
        pm = fmaxf(pm, M);  // M_t
        float prev = __shfl_up_sync(kFull, pm, 1);
        if (lane == 0) prev = M;  // M_{t-1}
        ab[lane] = scale_fos(prev, pm);
        ab[32 + lane] = (mt == -INFINITY) ? 0.0f : __fmul_rn(st, scale_fos(mt, pm));
        __syncwarp();
        const int n = min(32, Te - base);
        for (int q = 0; q < n; ++q) S = __fadd_rn(__fmul_rn(S, ab[q]), ab[32 + q]);
        M = __shfl_sync(kFull, pm, n - 1);
        __syncwarp();
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
    if (reg_mode) {
#pragma unroll
      for (int kk = 0; kk < KT; ++kk) {
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
    // Tile t's tm entry is written (pass 1) and re-read (pass 2) by warp t % nw only, and tc
    // is rewritten after the next row's first barrier, so no barrier is needed here unless a
    // single stage must be refilled now.
    if (!reg_mode && !defer) {
      __syncthreads();
      if (a.use_bulk && tid == 0 && k + NS < nmine) {
        issue_row<T>(a, r0 + (k + NS) * G, stage, &bars[s], &geos[s], false);
        issued_end = k + NS + 1;
      }
    }
  }
}

template <int KT>
const void *fwd_fn(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_fwd_kernel<float, KT>);
    case FOS_BF16: return reinterpret_cast<const void *>(&fos_fwd_kernel<__nv_bfloat16, KT>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_fwd_kernel<__half, KT>);
  }
  return nullptr;
}

const void *fwd_fn(fos_dtype dt, int kt) { return kt <= 4 ? fwd_fn<4>(dt) : fwd_fn<8>(dt); }

template <typename T, int KT>
void launch_t(const FwdArgs &a, int grid, int threads, size_t smem, cudaStream_t s) {
  fos_fwd_kernel<T, KT><<<grid, threads, smem, s>>>(a);
}

}  // namespace

size_t fwd_extra_smem(int T, int stages) {
  (void)stages;
  return (size_t)kBarBytes + kGeoBytes + (size_t)(3 * T + 64) * sizeof(float);
}

int fwd_tiles_per_warp(int T, int warps) {
  // 4 tiles per warp when they fit, else 8; beyond 8 per warp e_j are recomputed.
  return (T <= 4 * warps) ? 4 : 8;
}

cudaError_t fwd_prepare(fos_dtype dt, int max_smem) {
  for (int kt : {4, 8}) {
    cudaError_t e =
        cudaFuncSetAttribute(fwd_fn(dt, kt), cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t fwd_occupancy(fos_dtype dt, int kt, int threads, size_t smem, int *blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fwd_fn(dt, kt), threads,
                                                       smem);
}

cudaError_t fwd_launch(fos_dtype dt, int kt, const FwdArgs &a, int grid, int threads,
                       size_t smem, cudaStream_t s) {
  const bool k4 = kt <= 4;
  switch (dt) {
    case FOS_F32: k4 ? launch_t<float, 4>(a, grid, threads, smem, s)
                     : launch_t<float, 8>(a, grid, threads, smem, s); break;
    case FOS_BF16: k4 ? launch_t<__nv_bfloat16, 4>(a, grid, threads, smem, s)
                      : launch_t<__nv_bfloat16, 8>(a, grid, threads, smem, s); break;
    case FOS_F16: k4 ? launch_t<__half, 4>(a, grid, threads, smem, s)
                     : launch_t<__half, 8>(a, grid, threads, smem, s); break;
  }
  return cudaGetLastError();
}

}  // namespace fos
