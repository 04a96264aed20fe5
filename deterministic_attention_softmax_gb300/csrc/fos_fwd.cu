// fos_fwd.cu -- forward kernel of the fixed-order row softmax (P and LSE), sm_103a.
//
// One CTA owns one complete row at a time ("[WS1][kernels] Add fixed-order joint-attention
// softmax for Qwen-Image", Summary: fixed-order online softmax).  CTAs are persistent: CTA c
// takes rows c, c + grid, c + 2*grid, ...  On the bulk-copy path every CTA keeps a ring of
// `stages` shared-memory row buffers; a producer warp refills a buffer with a 1-D TMA bulk copy
// as soon as the compute warps release it (and writes that row's geometry next to it), so
// several rows per CTA are in flight from HBM while the current one is computed.  Per row, in
// the compute warps:
//
//   pass 1   warp w takes tiles w, w + nw, ... in pairs; per tile: lane max, warp max m_t,
//            e_j = exp(x_j - m_t), ascending lane sum, xor-tree sum s_t.
//   merge    warp 0 folds the tile states left to right, from (sink_h, 1) or (-inf, 0):
//              M_t = max(M_{t-1}, m_t)
//              S_t = S_{t-1} * exp(M_{t-1} - M_t) + s_t * exp(m_t - M_t)
//            (the factors are formed lane-parallel; the fold itself is sequential), then,
//            per tile, c_t = exp(m_t - M) / S, and LSE = M + log S.
//   pass 2   P_j = e_j * c_t, rounded once to the I/O dtype, 16-byte stores.
//
// The two tiles of a pair are independent, so their shuffle trees and exponentials overlap.
// When every warp has at most KT tiles, e_j are parked in tensor memory between the passes
// (each warp in its own lane quarter and columns) and the stage is released right after pass
// 1; registers then hold one tile pair at a time, which lets twice the CTAs share an SM.  A
// single pair per warp (KT = 2) simply stays in registers.  Longer rows recompute e_j from the
// staged row in pass 2 (same bits).  Masked
// keys (causal bound, valid length, key mask, -inf input) enter as -inf; tiles past the row's
// last candidate key are neither read nor reduced, and their P is written as +0.
#include <float.h>

#include "fos_device.cuh"
#include "fos_internal.h"

namespace fos {
namespace {

constexpr int kBarBytes = 256;  // 16 "full" and 16 "empty" mbarriers at the start
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

// e_j = exp(x_j - m) and their ascending lane sum.  For a tile with no valid key (m = -inf)
// the shift is -FLT_MAX instead, so every e_j is exp(-inf) = +0; otherwise it is m itself.
// Unless some key of the tile lies more than 87 below the maximum (a warp-uniform test), no
// e_j can be below 2^-126 and the flush-to-zero exponential gives the same bits.  On that
// path neighbouring keys go two at a time through the packed float32 operations of the
// sm_100 family (__fadd2_rn, __fmul2_rn), which round each component exactly as the scalar
// operation does; x - m is computed as x + (-m), the same IEEE operation.
__device__ __forceinline__ float tile_exp_sum(const float (&x)[8], float m, float (&e)[8]) {
  const float mm = fmaxf(m, -FLT_MAX);
  const bool deep = __any_sync(kFull, __fsub_rn(min8(x), mm) < -87.0f);
  if (!deep) {
    const float2 neg = make_float2(-mm, -mm);
    const float2 l2e = make_float2(kLog2e, kLog2e);
#pragma unroll
    for (int q = 0; q < kLaneKeys; q += 2) {
      const float2 t = __fmul2_rn(__fadd2_rn(make_float2(x[q], x[q + 1]), neg), l2e);
      e[q] = ex2_ftz(t.x);
      e[q + 1] = ex2_ftz(t.y);
    }
  } else {
#pragma unroll
    for (int q = 0; q < kLaneKeys; ++q) e[q] = exp_fos(__fsub_rn(x[q], mm));
  }
  float s = e[0];
#pragma unroll
  for (int q = 1; q < kLaneKeys; ++q) s = __fadd_rn(s, e[q]);
  return s;
}

// Pass 1 for one tile: e_j into e, (m_t, s_t) into tm/ts (lane 0).
template <typename T>
__device__ __forceinline__ void tile_stats1(const unsigned char *stage, int t, int lane, int lim,
                                            const uint8_t *km, float (&e)[8], float *tm,
                                            float *ts) {
  float x[8];
  tile_keys<T>(stage, t, lane, lim, km, x);
  const float m = warp_max(max8(x));
  float s = warp_sum_xor(tile_exp_sum(x, m, e));
  if (lane == 0) {
    tm[t] = m;
    ts[t] = s;
  }
}

// Pass 1 for two tiles at once (same bits as two single calls).
template <typename T>
__device__ __forceinline__ void tile_stats2(const unsigned char *stage, int t0, int t1, int lane,
                                            int lim, const uint8_t *km, float (&e0)[8],
                                            float (&e1)[8], float *tm, float *ts) {
  float x0[8], x1[8];
  tile_keys<T>(stage, t0, lane, lim, km, x0);
  tile_keys<T>(stage, t1, lane, lim, km, x1);
  const float m0 = warp_max(max8(x0));
  const float m1 = warp_max(max8(x1));
  float s0 = tile_exp_sum(x0, m0, e0);
  float s1 = tile_exp_sum(x1, m1, e1);
  warp_sum_xor2(s0, s1);
  if (lane == 0) {
    tm[t0] = m0;
    ts[t0] = s0;
    tm[t1] = m1;
    ts[t1] = s1;
  }
}

// The same pass 1 with the lane's key pointers given (p0, p1: keys 8 * lane of tiles t0, t1 in
// the stage), so that a warp walking neighbouring tiles advances one pointer instead of
// recomputing addresses; t0 / t1 still name the tiles for the masks and the statistics.
template <typename T>
__device__ __forceinline__ void lane_keys(const unsigned char *p, int t, int lane, int lim,
                                          const uint8_t *km, float (&x)[8]) {
  Io<T>::widen(Io<T>::lds(p), x);
  if (km != nullptr || (t + 1) * kTileK > lim) mask_keys(x, t * kTileK + lane * kLaneKeys, lim, km);
}

template <typename T>
__device__ __forceinline__ void tile_stats1p(const unsigned char *p0, int t0, int lane, int lim,
                                             const uint8_t *km, float (&e)[8], float *tm,
                                             float *ts) {
  float x[8];
  lane_keys<T>(p0, t0, lane, lim, km, x);
  const float m = warp_max(max8(x));
  float s = warp_sum_xor(tile_exp_sum(x, m, e));
  if (lane == 0) {
    tm[t0] = m;
    ts[t0] = s;
  }
}

template <typename T>
__device__ __forceinline__ void tile_stats2p(const unsigned char *p0, const unsigned char *p1,
                                             int t0, int lane, int lim, const uint8_t *km,
                                             float (&e0)[8], float (&e1)[8], float *tm,
                                             float *ts) {
  float x0[8], x1[8];
  lane_keys<T>(p0, t0, lane, lim, km, x0);
  lane_keys<T>(p1, t0 + 1, lane, lim, km, x1);
  const float m0 = warp_max(max8(x0));
  const float m1 = warp_max(max8(x1));
  float s0 = tile_exp_sum(x0, m0, e0);
  float s1 = tile_exp_sum(x1, m1, e1);
  warp_sum_xor2(s0, s1);
  if (lane == 0) {
    tm[t0] = m0;
    ts[t0] = s0;
    tm[t0 + 1] = m1;
    ts[t0 + 1] = s1;
  }
}

// Pass 2's store of one tile at the lane's output pointer q (keys j0 .. j0 + 7 of the row).
template <typename T>
__device__ __forceinline__ void tile_store_p(unsigned char *q, int j0, int L, bool ovec,
                                             const float (&e)[8], float c) {
  float v[8];
  const float2 cc = make_float2(c, c);
#pragma unroll
  for (int k = 0; k < kLaneKeys; k += 2) {  // packed: one rounding per component
    const float2 pq = __fmul2_rn(make_float2(e[k], e[k + 1]), cc);
    v[k] = pq.x;
    v[k + 1] = pq.y;
  }
  if (ovec && j0 + kLaneKeys <= L) {
    Io<T>::st8(q, v);
  } else {
#pragma unroll
    for (int k = 0; k < kLaneKeys; ++k)
      if (j0 + k < L) Io<T>::st1(q + k * Io<T>::kEsz, v[k]);
  }
}

// tile_store_p for a lane whose 8 keys all lie in the row and whose output is 16-byte aligned.
template <typename T>
__device__ __forceinline__ void tile_store_full(unsigned char *q, const float (&e)[8], float c) {
  float v[8];
  const float2 cc = make_float2(c, c);
#pragma unroll
  for (int k = 0; k < kLaneKeys; k += 2) {  // packed: one rounding per component
    const float2 pq = __fmul2_rn(make_float2(e[k], e[k + 1]), cc);
    v[k] = pq.x;
    v[k + 1] = pq.y;
  }
  Io<T>::st8(q, v);
}

// e_j of tile t again from the staged row and the stored tile maximum (same bits as pass 1).
template <typename T>
__device__ __forceinline__ void tile_exp(const unsigned char *stage, int t, int lane, int lim,
                                         const uint8_t *km, float m, float (&e)[8]) {
  float x[8];
  tile_keys<T>(stage, t, lane, lim, km, x);
  (void)tile_exp_sum(x, m, e);
}

template <typename T>
__device__ __forceinline__ void tile_store(unsigned char *prow, int t, int lane, int L, bool ovec,
                                           const float (&e)[8], float c) {
  float v[8];
  const float2 cc = make_float2(c, c);
#pragma unroll
  for (int q = 0; q < kLaneKeys; q += 2) {  // packed: one rounding per component
    const float2 pq = __fmul2_rn(make_float2(e[q], e[q + 1]), cc);
    v[q] = pq.x;
    v[q + 1] = pq.y;
  }
  store_lane8<T>(prow, t * kTileK + lane * kLaneKeys, L, ovec, v);
}

// Warp 0: fold the Te tile states left to right, starting from (M, S) = (sink, 1) or (-inf, 0)
// (the prefix maxima and the rescale factors are formed lane-parallel, the fold itself is
// sequential), then write the per-tile scales c_t = exp(m_t - M) / S to tc.  Every lane ends
// with the final (M, S).  tc doubles as the fold's 64-float scratch.
__device__ __forceinline__ void merge_tiles(int Te, int lane, const float *tm, const float *ts,
                                            float *tc, float &M, float &S) {
  for (int base = 0; base < Te; base += 32) {
    const int t = base + lane;
    const float mt = t < Te ? tm[t] : -INFINITY;
    const float st = t < Te ? ts[t] : 0.0f;
    float pm = mt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(kFull, pm, o);
      if (lane >= o) pm = fmaxf(pm, y);
    }
    pm = fmaxf(pm, M);
    float prev = __shfl_up_sync(kFull, pm, 1);
    if (lane == 0) prev = M;
    // flushing these factors cannot change S (see scale_ftz)
    const float alpha = scale_ftz(prev, pm);
    const float beta = (mt == -INFINITY) ? 0.0f : __fmul_rn(st, scale_ftz(mt, pm));
    // The fold itself is sequential: every lane reads the factors back from shared
    // memory (broadcast 16-byte reads) and runs the same chain.  Slots past the last
    // tile hold (1, 0), an exact no-op on S (S * 1 = S, S + 0 = S), so the chain always
    // runs in steps of four.  tc doubles as the scratch: it is rewritten after the fold.
    const int n = min(32, Te - base);
    float *ab = tc;
    ab[lane] = (lane < n) ? alpha : 1.0f;
    ab[32 + lane] = (lane < n) ? beta : 0.0f;
    __syncwarp();
    for (int q0 = 0; q0 < n; q0 += 4) {
      const float4 av = *reinterpret_cast<const float4 *>(ab + q0);
      const float4 bv = *reinterpret_cast<const float4 *>(ab + 32 + q0);
      S = __fadd_rn(__fmul_rn(S, av.x), bv.x);
      S = __fadd_rn(__fmul_rn(S, av.y), bv.y);
      S = __fadd_rn(__fmul_rn(S, av.z), bv.z);
      S = __fadd_rn(__fmul_rn(S, av.w), bv.w);
    }
    __syncwarp();
    M = __shfl_sync(kFull, pm, n - 1);
  }
  for (int t = lane; t < Te; t += 32) {
    const float mt = tm[t];
    tc[t] = (mt == -INFINITY) ? 0.0f : __fdiv_rn(scale_fos(mt, M), S);
  }
}

// merge_tiles for rows of at most 8 tiles (one warp per row): the same bits.  Lane t < 8 holds
// tile t; its inclusive prefix maximum needs the shuffle distances 1, 2, 4 only (a lane below
// the distance gets its own value back, which the maximum leaves unchanged).  The final maximum
// is known once the prefix maxima are, so the numerators exp(m_t - M) of the scales are formed
// beside the sequential fold, which then leaves only the division.
__device__ __forceinline__ void merge_tiles8(int Te, int lane, const float *tm, const float *ts,
                                             float *tc, float &M, float &S) {
  if (Te <= 0) return;
  const float mt = lane < Te ? tm[lane] : -INFINITY;
  const float st = lane < Te ? ts[lane] : 0.0f;
  float pm = mt;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) pm = fmaxf(pm, __shfl_up_sync(kFull, pm, o));
  pm = fmaxf(pm, M);
  float prev = __shfl_up_sync(kFull, pm, 1);
  if (lane == 0) prev = M;
  const float Mf = __shfl_sync(kFull, pm, Te - 1);
  // flushing these factors cannot change S (see scale_ftz)
  const float alpha = scale_ftz(prev, pm);
  const float beta = (mt == -INFINITY) ? 0.0f : __fmul_rn(st, scale_ftz(mt, pm));
  const float num = scale_fos(mt, Mf);
  float *ab = tc;  // scratch: the factors, read back by every lane (slots past Te: (1, 0))
  if (lane < 8) {
    ab[lane] = (lane < Te) ? alpha : 1.0f;
    ab[32 + lane] = (lane < Te) ? beta : 0.0f;
  }
  __syncwarp();
#pragma unroll
  for (int q0 = 0; q0 < 8; q0 += 4) {
    if (q0 < Te) {
      const float4 av = *reinterpret_cast<const float4 *>(ab + q0);
      const float4 bv = *reinterpret_cast<const float4 *>(ab + 32 + q0);
      S = __fadd_rn(__fmul_rn(S, av.x), bv.x);
      S = __fadd_rn(__fmul_rn(S, av.y), bv.y);
      S = __fadd_rn(__fmul_rn(S, av.z), bv.z);
      S = __fadd_rn(__fmul_rn(S, av.w), bv.w);
    }
  }
  __syncwarp();
  M = Mf;
  if (lane < Te) tc[lane] = (mt == -INFINITY) ? 0.0f : __fdiv_rn(num, S);
}

// Copy keys [0, lim) of a row into the stage with plain loads (unaligned or forced path).
template <typename T>
__device__ __forceinline__ void plain_stage(unsigned char *stage, const unsigned char *src,
                                            int lim, bool vec, int nthreads) {
  constexpr int esz = Io<T>::kEsz;
  int start = 0;
  if (vec) {
    const int n16 = (lim * esz) >> 4;
    for (int c = threadIdx.x; c < n16; c += nthreads)
      reinterpret_cast<uint4 *>(stage)[c] = reinterpret_cast<const uint4 *>(src)[c];
    start = (n16 << 4) / esz;
  }
  for (int j = start + threadIdx.x; j < lim; j += nthreads) {
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

// Producer (lane 0 of the last warp): for each of the CTA's rows, wait until the compute
// warps have released the stage (the "empty" barrier, one arrival per compute warp), write the
// row's geometry next to it and start its bulk copy (the "full" barrier).  Issuing a copy can
// block the issuing thread for a long time, so no compute warp ever issues one.  Before it
// exits, the producer waits for every copy it issued, so shared memory is never released
// under a copy in flight.
template <typename T>
__device__ void fwd_produce(const FwdArgs &a, int64_t r0, int64_t G, int64_t nmine,
                            uint64_t *full, uint64_t *empty, int4 *geos, unsigned char *ring,
                            bool stall) {
  const int NS = a.stages;
  uint32_t issued = 0, last_ph = 0;  // per stage: a copy was issued / parity of the last one
  int s = 0;
  uint32_t ph = 0;
  for (int64_t kk = 0; kk < nmine; ++kk) {
    if (kk >= NS && !mbar_wait_bounded(smem_addr(&empty[s]), ph ^ 1u, a.timeout_ns)) {
      raise_device_error(a.err, kDevErrTimeout);
      break;
    }
    const bool skip = stall && kk == 0;
    issue_row<T>(a, r0 + kk * G, ring + (size_t)s * a.stage_bytes, &full[s], &geos[s], skip);
    if (!skip) {
      issued |= 1u << s;
      last_ph = (last_ph & ~(1u << s)) | (ph << s);
    }
    if (++s == NS) {
      s = 0;
      ph ^= 1u;
    }
  }
  for (int t = 0; t < NS; ++t)
    if (issued & (1u << t))
      mbar_wait_bounded(smem_addr(&full[t]), (last_ph >> t) & 1u, a.timeout_ns);
}

// kFast: the common case fixed at compile time (bulk copies, every row's e_j kept, no mask,
// no sink, 16-byte aligned output).  Both instances do the same arithmetic in the same order.
template <typename T, int KT, bool kFast>
__global__ void __maxnreg__(KT == 2 ? 72 : 64) fos_fwd_kernel(const FwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + 16;
  int4 *geos = reinterpret_cast<int4 *>(smem + kBarBytes);
  unsigned char *ring = smem + kBarBytes + kGeoBytes;
  const int T4 = (a.T + 3) & ~3;  // stats arrays padded for 16-byte reads
  float *tm = reinterpret_cast<float *>(ring + (size_t)a.stages * a.stage_bytes);
  float *ts = tm + T4;
  float *tc = ts + T4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tc + (T4 > 64 ? T4 : 64));

  const int tid = threadIdx.x;
  const int nw = (blockDim.x >> 5) - 1;  // compute warps; the last warp is the producer
  const int ncomp = nw * 32;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t r0 = blockIdx.x;
  if (r0 >= a.rows) return;
  const int64_t nmine = (a.rows - 1 - r0) / G + 1;
  const int NS = a.stages;
  // keep mode: every warp has at most KT tiles (the fast instance is only launched so); they
  // are parked in tensor memory unless one pair per warp stays in registers
  constexpr bool kRegs = KT == 2;
  const bool keep = kFast || a.keep_e != 0;
  const bool park = keep && !kRegs;
  const bool use_bulk = kFast || a.use_bulk != 0;

  if (tid == 0 && use_bulk) {
    for (int t = 0; t < NS; ++t) {
      mbar_init(smem_addr(&full[t]), 1);
      mbar_init(smem_addr(&empty[t]), nw);
    }
    fence_mbar_init();
  }
  if (park) {
    if (w == 0) tmem_alloc(smem_addr(tmem_slot), a.tmem_cols);
    tmem_fence_before();
  }
  __syncthreads();
  uint32_t tbase = 0;
  if (park) {
    tmem_fence_after();
    tbase = *tmem_slot;
  }
  if (w == nw) {
    if (use_bulk && lane == 0)
      fwd_produce<T>(a, r0, G, nmine, full, empty, geos, ring, a.test_stall && blockIdx.x == 0);
    return;
  }
  // this warp's tile slots: lane quarter w % 4, KT * 8 columns from (w / 4) * KT * 8
  // The pair loops stay rolled up to three pairs (their slots are addressed at run time): the
  // smaller code measured 9-12 % faster on 17- and 18-tile rows, the unrolled one 1-4 % faster
  // at four pairs.
  constexpr int kPairUnroll = KT <= 6 ? 1 : KT / 2;
  const uint32_t tw = tbase + ((uint32_t)((w & 3) * 32) << 16) + (uint32_t)((w >> 2) * KT * 8);

  // stage index and phase parity of row k, carried rather than computed
  int s = 0;
  uint32_t ph = 0;
  for (int64_t k = 0; k < nmine; ++k, s = (s + 1 == NS) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
    const int64_t r = r0 + k * G;
    unsigned char *stage = ring + (size_t)s * a.stage_bytes;

    bool timed_out = false;
    int4 g;
    if (use_bulk) {
      timed_out = !mbar_wait_bounded(smem_addr(&full[s]), ph, a.timeout_ns);
      g = kFast ? make_int4(a.L, 0, 0, 0) : geos[s];
    } else {
      if (tid == 0) geos[0] = row_geometry(a, r);
      compute_sync(ncomp);  // also: every warp is done with the previous row's stage
      g = geos[0];
      plain_stage<T>(stage, static_cast<const unsigned char *>(a.scores) + (size_t)r * a.ld * esz,
                     g.x, a.in_vec != 0, ncomp);
      compute_sync(ncomp);
    }
    const int lim = g.x;
    const int Te = (lim + kTileK - 1) / kTileK;
    const uint8_t *km = (!kFast && a.key_mask) ? a.key_mask + (int64_t)g.y * a.L : nullptr;

    // ---- pass 1: tile statistics, two tiles at a time
    float er0[8], er1[8];  // kRegs: the warp's pair, kept for pass 2
    if (keep) {
#pragma unroll(kPairUnroll)
      for (int kk = 0; kk < KT; kk += 2) {
        const int t0 = w + kk * nw, t1 = t0 + nw;
        float e0[8], e1[8];
        if (!dbg_ok(a.err, Te <= a.T && (uint32_t)(Te * kTileK * esz) <= a.stage_bytes &&
                               (!park || ((tw - tbase) & 0xffffu) + kk * 8 + 16 <= a.tmem_cols)))
          continue;
        if (t1 < Te) {
          tile_stats2<T>(stage, t0, t1, lane, lim, km, e0, e1, tm, ts);
          if constexpr (kRegs) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              er0[q] = e0[q];
              er1[q] = e1[q];
            }
          } else {
            __syncwarp();
            tmem_st8(tw + kk * 8, e0);
            tmem_st8(tw + kk * 8 + 8, e1);
          }
        } else if (t0 < Te) {
          tile_stats1<T>(stage, t0, lane, lim, km, e0, tm, ts);
          if constexpr (kRegs) {
#pragma unroll
            for (int q = 0; q < 8; ++q) er0[q] = e0[q];
          } else {
            __syncwarp();
            tmem_st8(tw + kk * 8, e0);
          }
        }
      }
      if (use_bulk) {  // the stage is free: e_j are parked
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
      }
    } else {
      int t = w;
      for (; t + nw < Te; t += 2 * nw) {
        float e0[8], e1[8];
        tile_stats2<T>(stage, t, t + nw, lane, lim, km, e0, e1, tm, ts);
      }
      if (t < Te) {
        float e0[8];
        tile_stats1<T>(stage, t, lane, lim, km, e0, tm, ts);
      }
    }

    if (compute_sync_or(ncomp, timed_out)) {
      // A copy never landed: record it and stop (the producer drains the copies in flight;
      // the tensor memory is freed below).
      if (tid == 0) raise_device_error(a.err, kDevErrTimeout);
      break;
    }

    // ---- merge (warp 0)
    float M = -INFINITY, S = 0.0f;
    if (w == 0) {
      if (!kFast && a.sink != nullptr) {
        M = a.sink[g.z];
        S = 1.0f;
      }
      merge_tiles(Te, lane, tm, ts, tc, M, S);
    }
    compute_sync(ncomp);
    if (w == 0 && lane == 0) a.lse[r] = (M == -INFINITY) ? -INFINITY : __fadd_rn(M, logf(S));

    // ---- pass 2: P = e * c_t, one rounding, 16-byte stores
    if (!dbg_ok(a.err, r < a.rows)) break;
    unsigned char *prow = static_cast<unsigned char *>(a.probs) + (size_t)r * a.ld * esz;
    const bool ovec = kFast || a.out_vec != 0;
    if (keep) {
      if (park) {
        __syncwarp();
        tmem_wait_st();  // this warp's pass-1 values have landed
      }
#pragma unroll(kPairUnroll)
      for (int kk = 0; kk < KT; kk += 2) {
        const int t0 = w + kk * nw, t1 = t0 + nw;
        float e0[8], e1[8];
        if (t1 < Te) {
          if constexpr (kRegs) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              e0[q] = er0[q];
              e1[q] = er1[q];
            }
          } else {
            tmem_ld16(tw + kk * 8, e0, e1);
          }
          const float c0 = tc[t0], c1 = tc[t1];
          tile_store<T>(prow, t0, lane, a.L, ovec, e0, c0);
          tile_store<T>(prow, t1, lane, a.L, ovec, e1, c1);
        } else if (t0 < Te) {
          if constexpr (kRegs) {
#pragma unroll
            for (int q = 0; q < 8; ++q) e0[q] = er0[q];
          } else {
            tmem_ld8(tw + kk * 8, e0);
          }
          tile_store<T>(prow, t0, lane, a.L, ovec, e0, tc[t0]);
        }
      }
    } else {
      for (int t = w; t < Te; t += nw) {
        float ee[8];
        tile_exp<T>(stage, t, lane, lim, km, tm[t], ee);
        tile_store<T>(prow, t, lane, a.L, ovec, ee, tc[t]);
      }
      if (use_bulk) {  // done with the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
      }
    }
    for (int t = Te + w; t < a.T; t += nw) {
      float z[8];
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) z[q] = 0.0f;
      store_lane8<T>(prow, t * kTileK + lane * kLaneKeys, a.L, ovec, z);
    }
    // Tile t's tm entry is written (pass 1) and re-read (pass 2) by warp t % nw only, and tc
    // is rewritten after the next row's first barrier: no barrier is needed here.
  }
  if (park) {  // every compute warp is done with its columns: free them
    tmem_wait_st();
    tmem_fence_before();
    compute_sync(ncomp);
    if (w == 0) {
      tmem_fence_after();
      tmem_dealloc(tbase, a.tmem_cols);
    }
  }
}

// Lane 0: the geometry of row rr into *geo and its bulk copy into `stage` on barrier `bar`.
template <typename T>
__device__ __forceinline__ void rw_issue(const FwdArgs &a, int64_t rr, unsigned char *stage,
                                         uint64_t *bar, int4 *geo) {
  constexpr int esz = Io<T>::kEsz;
  const int4 g = row_geometry(a, rr);
  *geo = g;
  const uint32_t bytes = ((uint32_t)g.x * esz + 15u) & ~15u;  // never past the row
  const uint32_t bar_a = smem_addr(bar);
  fence_proxy_async_smem();  // the warp's reads of this buffer come before the copy
  mbar_arrive_expect_tx(bar_a, bytes);
  if (bytes)
    bulk_g2s(smem_addr(stage),
             static_cast<const unsigned char *>(a.scores) + (size_t)rr * a.ld * esz, bytes,
             bar_a);
}

// ------------------------------------------------ several row groups per CTA
//
// The CTA kernel above gives every CTA a warp that only issues copies, and that warp's
// registers count against the SM like a compute warp's.  Here a CTA holds `ng` groups of
// `nw` compute warps and no producer warp.  Group gg = blockIdx.x * ng + g takes rows gg,
// gg + gridDim.x * ng, ... one at a time, through its own ring of a.stages row buffers, and its
// last warp issues its copies: the copy of row k + stages goes into row k's buffer right after
// the group barrier that ends pass 1 of row k (the e_j are parked in tensor memory by then, so
// the buffer is free), while the group's warp 0 merges.  Pass 1, the merge and pass 2 are the
// CTA kernel's functions in the same order, so a row gives the same bits on either kernel.
// Taken when every warp parks its tiles (4, 6 or 8 per warp) and rows come by bulk copy.

constexpr int kGrpMaxBars = 128;  // "full" mbarriers (groups x stages) at the start
constexpr int kGrpHead = kGrpMaxBars * 8 + kGrpMaxBars * 16;  // barriers, then row records

template <typename T, int KT, bool kFast>
__global__ void __maxnreg__(64) fos_fwd_group_kernel(const FwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  const int nw = a.group_warps;
  const int ng = (blockDim.x >> 5) / nw;
  const int NS = a.stages;
  const int W = threadIdx.x >> 5;  // warp of the CTA: its tensor-memory lane quarter is W % 4
  const int g = W / nw;
  const int w = W - g * nw;  // warp of the group
  const int lane = threadIdx.x & 31;
  const int T4 = (a.T + 3) & ~3;
  const int nstat = 2 * T4 + (T4 > 64 ? T4 : 64);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
  uint64_t *full = bars + g * NS;
  int4 *geos = reinterpret_cast<int4 *>(smem + kGrpMaxBars * 8) + g * NS;
  unsigned char *ring = smem + kGrpHead + (size_t)g * NS * a.stage_bytes;
  float *stats = reinterpret_cast<float *>(smem + kGrpHead + (size_t)ng * NS * a.stage_bytes);
  float *tm = stats + g * nstat;
  float *ts = tm + T4;
  float *tc = ts + T4;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(stats + ng * nstat);

  const int64_t GG = (int64_t)gridDim.x * ng;  // groups in the grid
  const int64_t r0 = (int64_t)blockIdx.x * ng + g;
  const int bar_id = 1 + g;  // named barrier of the group (ids 1..15)
  const int gthreads = nw * 32;
  const bool issuer = (w == nw - 1) && lane == 0;
  const bool stall = a.test_stall && blockIdx.x == 0 && g == 0;

  if (threadIdx.x == 0) {
    for (int t = 0; t < ng * NS; ++t) mbar_init(smem_addr(&bars[t]), 1);
    fence_mbar_init();
  }
  if (W == 0) tmem_alloc(smem_addr(tmem_slot), a.tmem_cols);
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tbase = *tmem_slot;
  // this warp's tile slots: lane quarter W % 4, KT * 8 columns from (W / 4) * KT * 8
  const uint32_t tw = tbase + ((uint32_t)((W & 3) * 32) << 16) + (uint32_t)((W >> 2) * KT * 8);
  constexpr int kPairUnroll = KT <= 6 ? 1 : KT / 2;

  // prologue: the group's first rows (test only: the very first copy is never issued)
  if (issuer)
    for (int t = 0; t < NS && r0 + t * GG < a.rows; ++t)
      if (!(stall && t == 0))
        rw_issue<T>(a, r0 + t * GG, ring + (size_t)t * a.stage_bytes, &full[t], &geos[t]);

  // Row j of the group always goes through stage j % NS, phase (j / NS) & 1, and the copies
  // issued before row k's barrier are those of rows 0 .. k + NS - 1: after a timeout at row k
  // the issuer knows which copies may still be in flight without keeping a record.
  int s = 0;
  uint32_t ph = 0;
  int64_t r = r0;
  bool ok = true;
  for (; r < a.rows; r += GG) {
    unsigned char *stage = ring + (size_t)s * a.stage_bytes;
    const bool timed_out = !mbar_wait_bounded(smem_addr(&full[s]), ph, a.timeout_ns);
    // a copy that never landed leaves its record unwritten: no tile is then read
    int4 gm = kFast ? make_int4(a.L, 0, 0, 0) : geos[s];
    if (timed_out) gm.x = 0;
    const int lim = gm.x;
    const int Te = (lim + kTileK - 1) / kTileK;
    const uint8_t *km = (!kFast && a.key_mask) ? a.key_mask + (int64_t)gm.y * a.L : nullptr;

    // ---- pass 1: tile statistics, two neighbouring tiles at a time, e_j parked in tensor
    // memory.  Warp w owns tiles tb .. tb + KT - 1 (any assignment gives the same bits); its
    // lane pointer steps by two tiles.
    const int tb = w * KT;
    const int nt = Te - tb;  // tiles of this warp (at most KT; <= 0 when it has none)
    {
      const unsigned char *sp = stage + (size_t)(tb * kTileK + lane * kLaneKeys) * esz;
#pragma unroll(kPairUnroll)
      for (int kk = 0; kk < KT; kk += 2, sp += 2 * kTileK * esz) {
        float e0[8], e1[8];
        if (!dbg_ok(a.err, Te <= a.T && (uint32_t)(Te * kTileK * esz) <= a.stage_bytes &&
                               ((tw - tbase) & 0xffffu) + kk * 8 + 16 <= a.tmem_cols &&
                               r < a.rows))
          continue;
        if (kk + 1 < nt) {
          tile_stats2p<T>(sp, sp + kTileK * esz, tb + kk, lane, lim, km, e0, e1, tm, ts);
          __syncwarp();
          tmem_st8(tw + kk * 8, e0);
          tmem_st8(tw + kk * 8 + 8, e1);
        } else if (kk < nt) {
          tile_stats1p<T>(sp, tb + kk, lane, lim, km, e0, tm, ts);
          __syncwarp();
          tmem_st8(tw + kk * 8, e0);
        }
      }
    }
    if (named_sync_or(bar_id, gthreads, timed_out)) {
      // A copy never landed: record it and stop (the issuer waits for its copies in flight;
      // the tensor memory is freed below).
      if (w == 0 && lane == 0) raise_device_error(a.err, kDevErrTimeout);
      ok = false;
      break;
    }
    // every warp of the group is done with the buffer: refill it with row r + stages
    if (issuer && r + NS * GG < a.rows) rw_issue<T>(a, r + NS * GG, stage, &full[s], &geos[s]);

    // ---- merge (warp 0 of the group)
    float M = -INFINITY, S = 0.0f;
    if (w == 0) {
      if (!kFast && a.sink != nullptr) {
        M = a.sink[gm.z];
        S = 1.0f;
      }
      merge_tiles(Te, lane, tm, ts, tc, M, S);
    }
    named_sync(bar_id, gthreads);
    if (w == 0 && lane == 0) a.lse[r] = (M == -INFINITY) ? -INFINITY : __fadd_rn(M, logf(S));

    // ---- pass 2: P = e * c_t from the parked e_j, one rounding, 16-byte stores
    unsigned char *prow = static_cast<unsigned char *>(a.probs) + (size_t)r * a.ld * esz;
    const bool ovec = kFast || a.out_vec != 0;
    __syncwarp();
    tmem_wait_st();  // this warp's pass-1 values have landed
    {
      const int j0 = tb * kTileK + lane * kLaneKeys;  // the lane's first key
      unsigned char *pp = prow + (size_t)j0 * esz;
#pragma unroll(kPairUnroll)
      for (int kk = 0; kk < KT; kk += 2, pp += 2 * kTileK * esz) {
        float e0[8], e1[8];
        if (!dbg_ok(a.err, ((tw - tbase) & 0xffffu) + kk * 8 + 16 <= a.tmem_cols && r < a.rows))
          continue;
        const int jk = j0 + kk * kTileK;
        if (kk + 1 < nt) {
          tmem_ld16(tw + kk * 8, e0, e1);
          const float2 c = *reinterpret_cast<const float2 *>(tc + tb + kk);
          // Both tiles' keys of this lane in the row: one check for the pair.  Measured on
          // warps of at most 6 tiles (rolled pair loops): Qwen-Image forward 50.2 -> 48.7 us;
          // with 8 tiles (unrolled) the larger code cost 0.7 %, so those keep the per-tile check.
          if (KT <= 6 && ovec && jk + kTileK + kLaneKeys <= a.L) {
            tile_store_full<T>(pp, e0, c.x);
            tile_store_full<T>(pp + kTileK * esz, e1, c.y);
          } else {
            tile_store_p<T>(pp, jk, a.L, ovec, e0, c.x);
            tile_store_p<T>(pp + kTileK * esz, jk + kTileK, a.L, ovec, e1, c.y);
          }
        } else if (kk < nt) {
          tmem_ld8(tw + kk * 8, e0);
          tile_store_p<T>(pp, jk, a.L, ovec, e0, tc[tb + kk]);
        }
      }
    }
    // tiles past the row's last candidate key: P = +0 (this warp's tiles below T)
    for (int t = (Te > tb ? Te : tb); t < tb + KT && t < a.T; ++t) {
      float z[8];
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) z[q] = 0.0f;
      store_lane8<T>(prow, t * kTileK + lane * kLaneKeys, a.L, ovec, z);
    }
    // Tile t's tm / ts entries are written by its warp in pass 1 and read by warp 0's merge
    // between the group's two barriers; tc is rewritten after the next row's first barrier.
    if (++s == NS) {
      s = 0;
      ph ^= 1u;
    }
  }
  // after a timeout at row k, every copy the issuer started (rows k .. k + NS - 1; row 0 not
  // in the test's stall) lands before the CTA can exit
  if (!ok && issuer) {
    const int64_t k = (r - r0) / GG;
    for (int64_t j = k; j < k + NS && r0 + j * GG < a.rows; ++j)
      if (!(stall && j == 0))
        mbar_wait_bounded(smem_addr(&full[j % NS]), (uint32_t)(j / NS) & 1u, a.timeout_ns);
  }
  // every warp is done with its columns: free them
  __syncwarp();
  tmem_wait_st();
  tmem_fence_before();
  __syncthreads();
  if (W == 0) {
    tmem_fence_after();
    tmem_dealloc(tbase, a.tmem_cols);
  }
}

// ------------------------------------------------ rows longer than shared memory (streaming)
//
// A row whose staged copy would not fit in shared memory is read twice, in segments of
// a.seg_tiles tiles that cycle through the same ring: pass 1 takes the tile statistics
// segment by segment while a merge warp folds them behind it (the steps of merge_tiles, chunk
// by chunk), and pass 2 reads every segment again and recomputes e_j from the stored tile
// maxima, as the staged kernel's recompute mode does.  The per-tile arithmetic and the fold are
// those of fos_fwd_kernel, so a row gives the same bits on either path; the price is a second
// read of the scores.

// Producer: each row's segments twice (pass 1, then pass 2), in order through the ring, with
// the row's record {limit, batch entry, head, segment} beside every segment.  A row with no
// valid key still gets one (empty) segment per pass, so its record reaches the compute warps.
template <typename T>
__device__ void fwd_stream_produce(const FwdArgs &a, int64_t r0, int64_t G, int64_t nmine,
                                   uint64_t *full, uint64_t *empty, int4 *geos,
                                   unsigned char *ring, bool stall) {
  constexpr int esz = Io<T>::kEsz;
  const int NS = a.stages;
  const int seg_keys = a.seg_tiles * kTileK;
  uint32_t issued = 0, last_ph = 0;
  int s = 0;
  uint32_t ph = 0;
  int64_t n = 0;  // segments issued so far
  bool stop = false;
  for (int64_t kk = 0; kk < nmine && !stop; ++kk) {
    const int64_t rr = r0 + kk * G;
    const int4 g = row_geometry(a, rr);
    const int nseg = g.x > 0 ? (g.x + seg_keys - 1) / seg_keys : 1;
    const unsigned char *src = static_cast<const unsigned char *>(a.scores) + (size_t)rr * a.ld * esz;
    for (int pass = 0; pass < 2 && !stop; ++pass) {
      for (int seg = 0; seg < nseg; ++seg, ++n) {
        if (n >= NS && !mbar_wait_bounded(smem_addr(&empty[s]), ph ^ 1u, a.timeout_ns)) {
          raise_device_error(a.err, kDevErrTimeout);
          stop = true;
          break;
        }
        const int k0 = seg * seg_keys;
        const int nk = min(seg_keys, max(0, g.x - k0));
        geos[s] = make_int4(g.x, g.y, g.z, seg);
        // rounded up to 16 bytes; never past the row since L * esz is a multiple of 16 here
        const uint32_t bytes = ((uint32_t)nk * esz + 15u) & ~15u;
        if (!(stall && n == 0)) {  // test only: the first copy is never issued
          const uint32_t bar_a = smem_addr(&full[s]);
          mbar_arrive_expect_tx(bar_a, bytes);
          if (bytes) bulk_g2s(smem_addr(ring + (size_t)s * a.stage_bytes), src + (size_t)k0 * esz,
                              bytes, bar_a);
          issued |= 1u << s;
          last_ph = (last_ph & ~(1u << s)) | (ph << s);
        }
        if (++s == NS) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  }
  for (int t = 0; t < NS; ++t)
    if (issued & (1u << t))
      mbar_wait_bounded(smem_addr(&full[t]), (last_ph >> t) & 1u, a.timeout_ns);
}

// One chunk of at most 32 tiles of the fold, in order, continuing from the running (M, S):
// lane t takes tile t of the chunk.  The steps are those of merge_tiles (prefix maxima from
// the running maximum, the factors, the sequential fold), so folding a row chunk by chunk, at
// any chunk boundaries, gives the bits of merge_tiles.  ab is a 64-float scratch.
__device__ __forceinline__ void fold_chunk(const float *tmc, const float *tsc, int n, int lane,
                                           float *ab, float &M, float &S) {
  const float mt = lane < n ? tmc[lane] : -INFINITY;
  const float st = lane < n ? tsc[lane] : 0.0f;
  float pm = mt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) pm = fmaxf(pm, __shfl_up_sync(kFull, pm, o));
  pm = fmaxf(pm, M);
  float prev = __shfl_up_sync(kFull, pm, 1);
  if (lane == 0) prev = M;
  // flushing these factors cannot change S (see scale_ftz)
  const float alpha = scale_ftz(prev, pm);
  const float beta = (mt == -INFINITY) ? 0.0f : __fmul_rn(st, scale_ftz(mt, pm));
  ab[lane] = (lane < n) ? alpha : 1.0f;
  ab[32 + lane] = (lane < n) ? beta : 0.0f;
  __syncwarp();
  for (int q0 = 0; q0 < n; q0 += 4) {
    const float4 av = *reinterpret_cast<const float4 *>(ab + q0);
    const float4 bv = *reinterpret_cast<const float4 *>(ab + 32 + q0);
    S = __fadd_rn(__fmul_rn(S, av.x), bv.x);
    S = __fadd_rn(__fmul_rn(S, av.y), bv.y);
    S = __fadd_rn(__fmul_rn(S, av.z), bv.z);
    S = __fadd_rn(__fmul_rn(S, av.w), bv.w);
  }
  __syncwarp();
  M = __shfl_sync(kFull, pm, n - 1);
}

// The merge warp: it follows the ring through the same segments as the compute warps.  For
// each pass-1 segment it waits until every compute warp has written that segment's tile
// statistics (the stage's "statistics" barrier), folds them into the running (M, S) and then
// releases the stage (its arrival on "empty" is one of the nw + 1 the producer waits for, so the
// ring never runs more than a ring ahead of the fold).  After the row's last segment it writes
// the scales c_t and the LSE, and meets the compute warps at barrier 1; pass 2 takes no part of
// it (warp 0 arrives for it on "empty"), and barrier 2 ends the row for both.  A wait that runs
// out stops the warp: it says so at the next barrier, where the compute warps learn of it.
template <typename T>
__device__ void fwd_stream_merge(const FwdArgs &a, int64_t r0, int64_t G, int64_t nmine,
                                 uint64_t *empty, uint64_t *stat, const int4 *geos,
                                 const float *tm, const float *ts, float *tc, float *ab, int nsync) {
  const int lane = threadIdx.x & 31;
  const int NS = a.stages;
  const int SEG = a.seg_tiles;
  int s = 0;
  uint32_t stat_ph = 0;  // per stage: parity of its next "statistics" phase
  for (int64_t k = 0; k < nmine; ++k) {
    const int64_t r = r0 + k * G;
    bool bad = false;
    int Te = 0, nseg = 1;
    float M = -INFINITY, S = 0.0f;
    for (int seg = 0; seg < nseg; ++seg) {
      if (!mbar_wait_bounded(smem_addr(&stat[s]), (stat_ph >> s) & 1u, a.timeout_ns)) {
        bad = true;
        break;
      }
      stat_ph ^= 1u << s;
      if (seg == 0) {
        const int4 g = geos[s];
        Te = (g.x + kTileK - 1) / kTileK;
        nseg = Te > 0 ? (Te + SEG - 1) / SEG : 1;
        if (a.sink != nullptr) {
          M = a.sink[g.z];
          S = 1.0f;
        }
      }
      const int t0 = seg * SEG, nt = min(SEG, Te - t0);
      for (int c0 = 0; c0 < nt; c0 += 32)
        fold_chunk(tm + t0 + c0, ts + t0 + c0, min(32, nt - c0), lane, ab, M, S);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
      if (++s == NS) s = 0;
    }
    if (!bad) {
#pragma unroll 4
      for (int t = lane; t < Te; t += 32) {
        const float mt = tm[t];
        tc[t] = (mt == -INFINITY) ? 0.0f : __fdiv_rn(scale_fos(mt, M), S);
      }
      if (lane == 0) a.lse[r] = (M == -INFINITY) ? -INFINITY : __fadd_rn(M, logf(S));
    }
    if (named_sync_or(1, nsync, bad)) {
      if (lane == 0 && bad) raise_device_error(a.err, kDevErrTimeout);
      return;
    }
    s = (int)((s + nseg) % NS);  // the row's pass-2 segments
    if (named_sync_or(2, nsync, false)) return;
  }
}

template <typename T>
__global__ void __maxnreg__(64) fos_fwd_stream_kernel(const FwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + 16;
  int4 *geos = reinterpret_cast<int4 *>(smem + kBarBytes);
  unsigned char *ring = smem + kBarBytes + kGeoBytes;
  const int T4 = (a.T + 3) & ~3;
  float *tm = reinterpret_cast<float *>(ring + (size_t)a.stages * a.stage_bytes);
  float *ts = tm + T4;
  float *tc = ts + T4;
  // after tc (and the 16 bytes kept for a tensor-memory address by the other kernels' layout):
  // the stages' "statistics" barriers, then the merge warp's fold scratch
  uint64_t *stat = reinterpret_cast<uint64_t *>(tc + (T4 > 64 ? T4 : 64) + 4);
  float *ab = reinterpret_cast<float *>(stat + 16);

  const int tid = threadIdx.x;
  const int nw = (blockDim.x >> 5) - 2;  // compute warps; then the merge warp and the producer
  const int nsync = (nw + 1) * 32;       // compute warps and the merge warp
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t r0 = blockIdx.x;
  if (r0 >= a.rows) return;
  const int64_t nmine = (a.rows - 1 - r0) / G + 1;
  const int NS = a.stages;
  const int SEG = a.seg_tiles;

  if (tid == 0) {
    for (int t = 0; t < NS; ++t) {
      mbar_init(smem_addr(&full[t]), 1);
      mbar_init(smem_addr(&empty[t]), nw + 1);
      mbar_init(smem_addr(&stat[t]), nw);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (w == nw + 1) {
    if (lane == 0)
      fwd_stream_produce<T>(a, r0, G, nmine, full, empty, geos, ring,
                            a.test_stall && blockIdx.x == 0);
    return;
  }
  if (w == nw) {
    fwd_stream_merge<T>(a, r0, G, nmine, empty, stat, geos, tm, ts, tc, ab, nsync);
    return;
  }

  int s = 0;
  uint32_t ph = 0;
  for (int64_t k = 0; k < nmine; ++k) {
    const int64_t r = r0 + k * G;
    bool timed_out = false;
    int4 g = make_int4(0, 0, 0, 0);
    int lim = 0, Te = 0, nseg = 1;
    const uint8_t *km = nullptr;

    // ---- pass 1: tile statistics, segment by segment; the merge warp folds them behind
    for (int seg = 0; seg < nseg; ++seg) {
      if (!mbar_wait_bounded(smem_addr(&full[s]), ph, a.timeout_ns)) {
        timed_out = true;
        break;
      }
      if (seg == 0) {
        g = geos[s];
        lim = g.x;
        Te = (lim + kTileK - 1) / kTileK;
        nseg = Te > 0 ? (Te + SEG - 1) / SEG : 1;
        km = a.key_mask ? a.key_mask + (int64_t)g.y * a.L : nullptr;
      }
      const unsigned char *stage = ring + (size_t)s * a.stage_bytes;
      const int t0 = seg * SEG, nt = min(SEG, Te - t0);
      const int lim_l = lim - t0 * kTileK;  // the segment's keys are numbered from 0
      const uint8_t *kms = km ? km + t0 * kTileK : nullptr;
      if (!dbg_ok(a.err, Te <= a.T && (nt <= 0 || (uint32_t)(nt * kTileK * esz) <= a.stage_bytes)))
        timed_out = true;  // stop the row as a failed wait would
      int tl = timed_out ? nt : w;
      for (; tl + nw < nt; tl += 2 * nw) {
        float e0[8], e1[8];
        tile_stats2<T>(stage, tl, tl + nw, lane, lim_l, kms, e0, e1, tm + t0, ts + t0);
      }
      if (tl < nt) {
        float e0[8];
        tile_stats1<T>(stage, tl, lane, lim_l, kms, e0, tm + t0, ts + t0);
      }
      if (timed_out) break;  // (index check failed) its statistics are not announced
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&stat[s]));  // release: this warp's tm / ts entries
        mbar_arrive(smem_addr(&empty[s]));
      }
      if (++s == NS) {
        s = 0;
        ph ^= 1u;
      }
    }
    // the merge warp has folded the row and written tc and the LSE
    if (named_sync_or(1, nsync, timed_out)) {
      if (tid == 0) raise_device_error(a.err, kDevErrTimeout);
      return;
    }

    // ---- pass 2: every segment again, e_j recomputed, P written
    unsigned char *prow = static_cast<unsigned char *>(a.probs) + (size_t)r * a.ld * esz;
    const bool ovec = a.out_vec != 0;
    for (int seg = 0; seg < nseg; ++seg) {
      if (!mbar_wait_bounded(smem_addr(&full[s]), ph, a.timeout_ns)) {
        timed_out = true;
        break;
      }
      const unsigned char *stage = ring + (size_t)s * a.stage_bytes;
      const int t0 = seg * SEG, nt = min(SEG, Te - t0);
      const int lim_l = lim - t0 * kTileK;
      const uint8_t *kms = km ? km + t0 * kTileK : nullptr;
      for (int tl = w; tl < nt; tl += nw) {
        float ee[8];
        tile_exp<T>(stage, tl, lane, lim_l, kms, tm[t0 + tl], ee);
        tile_store<T>(prow, t0 + tl, lane, a.L, ovec, ee, tc[t0 + tl]);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&empty[s]));
        if (w == 0) mbar_arrive(smem_addr(&empty[s]));  // the merge warp's share in pass 2
      }
      if (++s == NS) {
        s = 0;
        ph ^= 1u;
      }
    }
    for (int t = Te + w; t < a.T; t += nw) {
      float z[8];
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) z[q] = 0.0f;
      store_lane8<T>(prow, t * kTileK + lane * kLaneKeys, a.L, ovec, z);
    }
    // a wait that ran out in pass 2 stops every compute warp and the merge warp
    if (named_sync_or(2, nsync, timed_out)) {
      if (tid == 0) raise_device_error(a.err, kDevErrTimeout);
      return;
    }
    // Each warp writes (pass 1) and reads (pass 2) the tm entries of its own tiles only; the
    // merge warp reads a segment's entries once its warps have announced them, and tc is
    // rewritten after the next row's pass 1.
  }
}

const void *fwd_stream_fn(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_fwd_stream_kernel<float>);
    case FOS_BF16: return reinterpret_cast<const void *>(&fos_fwd_stream_kernel<__nv_bfloat16>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_fwd_stream_kernel<__half>);
  }
  return nullptr;
}

// ------------------------------------------------------ short rows: one warp per row
//
// A row of at most KT (<= 8) tiles is taken by one warp alone: it waits for the row's copy,
// runs pass 1 on all its tiles (pairs of neighbouring tiles), folds the tile states with
// merge_tiles8 (merge_tiles' steps for at most 8 tiles), and writes P from the e_j it parked in
// tensor memory (its lane quarter w % 4, warps sharing a quarter side by side in its columns).
// No barrier joins the warps of a CTA, so the merge of one row does not idle the others.  Each
// warp keeps its own ring of a.stages row buffers and its lane 0 issues its own copies: the copy
// of row k + stages goes into the buffer of row k as soon as pass 1 of row k has read it.  The
// per-tile arithmetic, the merge and pass 2 are those of fos_fwd_kernel, so a row gives the same
// bits on either kernel.

template <typename T, int KT>
__global__ void __maxnreg__(KT == 2 ? 72 : 64) fos_fwd_rowwarp_kernel(const FwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  constexpr int kStat = 80;  // floats per warp: tm[8], ts[8], tc[64] (tc is the merge scratch)
  const int nw = blockDim.x >> 5;
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = a.stages;  // row buffers per warp
  uint64_t *full = reinterpret_cast<uint64_t *>(smem) + w * NS;
  int4 *geos = reinterpret_cast<int4 *>(smem + kBarBytes) + w * NS;
  unsigned char *ring = smem + kBarBytes + kGeoBytes + (size_t)w * NS * a.stage_bytes;
  float *stats = reinterpret_cast<float *>(smem + kBarBytes + kGeoBytes +
                                           (size_t)nw * NS * a.stage_bytes);
  float *tm = stats + w * kStat;
  float *ts = tm + 8;
  float *tc = tm + 16;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(stats + nw * kStat);

  const int64_t GW = (int64_t)gridDim.x * nw;           // warps in the grid
  const int64_t r0 = (int64_t)blockIdx.x * nw + w;        // this warp's first row
  const int64_t nmine = r0 < a.rows ? (a.rows - 1 - r0) / GW + 1 : 0;
  const bool stall = a.test_stall && blockIdx.x == 0 && w == 0;

  if (lane == 0) {
    for (int t = 0; t < NS; ++t) mbar_init(smem_addr(&full[t]), 1);
    fence_mbar_init();
  }
  // one pair per row (KT = 2) stays in registers; longer rows are parked in tensor memory
  constexpr bool kRegs = KT == 2;
  if constexpr (!kRegs) {
    if (w == 0) tmem_alloc(smem_addr(tmem_slot), a.tmem_cols);
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
  }
  __syncwarp();  // this warp's barriers are initialised
  const uint32_t tw =
      kRegs ? 0u : *tmem_slot + ((uint32_t)((w & 3) * 32) << 16) + (uint32_t)((w >> 2) * KT * 8);
  // the four-pair loops stay rolled (measured 11 % faster on 8-tile rows), shorter ones are
  // unrolled (2 % faster on 4-tile rows)
  constexpr int kPairUnroll = KT >= 8 ? 1 : KT / 2;
  // prologue: the first rows' copies (test only: the very first one is never issued)
  uint32_t issued = 0, last_ph = 0;
  if (lane == 0)
    for (int t = 0; t < NS && t < nmine; ++t)
      if (!(stall && t == 0)) {
        rw_issue<T>(a, r0 + t * GW, ring + (size_t)t * a.stage_bytes, &full[t], &geos[t]);
        issued |= 1u << t;
      }

  int s = 0;
  uint32_t ph = 0;
  bool ok = true;
  for (int64_t k = 0; k < nmine; ++k) {
    const int64_t r = r0 + k * GW;
    unsigned char *stage = ring + (size_t)s * a.stage_bytes;
    // every lane waits; the warp stops as one if any lane's wait ran out
    const bool landed = mbar_wait_bounded(smem_addr(&full[s]), ph, a.timeout_ns);
    if (!__all_sync(kFull, landed)) {
      if (lane == 0) raise_device_error(a.err, kDevErrTimeout);
      ok = false;
      break;
    }
    const int4 g = geos[s];
    const int lim = g.x;
    const int Te = (lim + kTileK - 1) / kTileK;
    const uint8_t *km = a.key_mask ? a.key_mask + (int64_t)g.y * a.L : nullptr;
    if (!dbg_ok(a.err, Te <= KT && (uint32_t)(Te * kTileK * esz) <= a.stage_bytes &&
                           r < a.rows &&
                           (kRegs || ((tw - *tmem_slot) & 0xffffu) + KT * 8 <= a.tmem_cols))) {
      ok = false;
      break;
    }
    // the head's sink logit, loaded now so that its latency passes under pass 1
    const float sink_h = a.sink != nullptr ? a.sink[g.z] : -INFINITY;
    // the rolled loops (KT = 8) stop after the row's last tile; the unrolled ones test each pair
    const int kend = kPairUnroll == 1 ? Te : KT;

    // ---- pass 1: every tile of the row, two neighbouring tiles at a time (the lane's key
    // pointer steps by two tiles)
    float er0[8], er1[8];  // kRegs: the row's pair, kept for pass 2
    const unsigned char *sp = stage + (size_t)(lane * kLaneKeys) * esz;
#pragma unroll(kPairUnroll)
    for (int kk = 0; kk < kend; kk += 2, sp += 2 * kTileK * esz) {
      if constexpr (kRegs) {
        if (kk + 1 < Te)
          tile_stats2<T>(stage, kk, kk + 1, lane, lim, km, er0, er1, tm, ts);
        else if (kk < Te)
          tile_stats1<T>(stage, kk, lane, lim, km, er0, tm, ts);
      } else {
        float e0[8], e1[8];
        if (kk + 1 < Te) {
          tile_stats2p<T>(sp, sp + kTileK * esz, kk, lane, lim, km, e0, e1, tm, ts);
          __syncwarp();
          tmem_st8(tw + kk * 8, e0);
          tmem_st8(tw + kk * 8 + 8, e1);
        } else if (kk < Te) {
          tile_stats1p<T>(sp, kk, lane, lim, km, e0, tm, ts);
          __syncwarp();
          tmem_st8(tw + kk * 8, e0);
        }
      }
    }
    __syncwarp();  // tm / ts (lane 0) for the merge; every lane is done with the buffer
    if (lane == 0 && k + NS < nmine) {
      rw_issue<T>(a, r + NS * GW, stage, &full[s], &geos[s]);
      issued |= 1u << s;
      last_ph = (last_ph & ~(1u << s)) | ((ph ^ 1u) << s);
    }

    // ---- merge (this warp)
    float M = -INFINITY, S = 0.0f;
    if (a.sink != nullptr) {
      M = sink_h;
      S = 1.0f;
    }
    merge_tiles8(Te, lane, tm, ts, tc, M, S);
    __syncwarp();  // tc
    if (lane == 0) a.lse[r] = (M == -INFINITY) ? -INFINITY : __fadd_rn(M, logf(S));

    // ---- pass 2: P from the kept e_j
    unsigned char *prow = static_cast<unsigned char *>(a.probs) + (size_t)r * a.ld * esz;
    const bool ovec = a.out_vec != 0;
    if constexpr (kRegs) {
      if (1 < Te) {
        tile_store<T>(prow, 0, lane, a.L, ovec, er0, tc[0]);
        tile_store<T>(prow, 1, lane, a.L, ovec, er1, tc[1]);
      } else if (0 < Te) {
        tile_store<T>(prow, 0, lane, a.L, ovec, er0, tc[0]);
      }
    } else {
      __syncwarp();
      tmem_wait_st();
    }
    unsigned char *pp = prow + (size_t)(lane * kLaneKeys) * esz;
#pragma unroll(kPairUnroll)
    for (int kk = 0; kk < (kRegs ? 0 : kend); kk += 2, pp += 2 * kTileK * esz) {
      float e0[8], e1[8];
      if (kk + 1 < Te) {
        tmem_ld16(tw + kk * 8, e0, e1);
        if (ovec && (kk + 2) * kTileK <= a.L) {  // both tiles whole in the row: no key checks
          tile_store_full<T>(pp, e0, tc[kk]);
          tile_store_full<T>(pp + kTileK * esz, e1, tc[kk + 1]);
        } else {
          tile_store<T>(prow, kk, lane, a.L, ovec, e0, tc[kk]);
          tile_store<T>(prow, kk + 1, lane, a.L, ovec, e1, tc[kk + 1]);
        }
      } else if (kk < Te) {
        tmem_ld8(tw + kk * 8, e0);
        tile_store<T>(prow, kk, lane, a.L, ovec, e0, tc[kk]);
      }
    }
    for (int t = Te; t < a.T; ++t) {
      float z[8];
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) z[q] = 0.0f;
      store_lane8<T>(prow, t * kTileK + lane * kLaneKeys, a.L, ovec, z);
    }
    __syncwarp();  // tc and tm / ts are rewritten by the next row
    if (++s == NS) {
      s = 0;
      ph ^= 1u;
    }
  }
  // every copy this warp issued has landed before it exits (its buffers stay allocated until
  // the whole CTA is done, but no copy may outlive the CTA)
  if (!ok && lane == 0)
    for (int t = 0; t < NS; ++t)
      if (issued & (1u << t))
        mbar_wait_bounded(smem_addr(&full[t]), (last_ph >> t) & 1u, a.timeout_ns);
  // every warp is done with its columns: free them
  if constexpr (!kRegs) {
    __syncwarp();
    tmem_wait_st();
    tmem_fence_before();
    __syncthreads();
    if (w == 0) {
      tmem_fence_after();
      tmem_dealloc(*tmem_slot, a.tmem_cols);
    }
  }
}

template <int KT, bool kFast>
const void *fwd_group_fn_kt(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_fwd_group_kernel<float, KT, kFast>);
    case FOS_BF16:
      return reinterpret_cast<const void *>(&fos_fwd_group_kernel<__nv_bfloat16, KT, kFast>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_fwd_group_kernel<__half, KT, kFast>);
  }
  return nullptr;
}

template <bool kFast>
const void *fwd_group_fn_f(fos_dtype dt, int kt) {
  return kt <= 4 ? fwd_group_fn_kt<4, kFast>(dt)
                 : (kt <= 6 ? fwd_group_fn_kt<6, kFast>(dt) : fwd_group_fn_kt<8, kFast>(dt));
}

const void *fwd_group_fn(fos_dtype dt, int kt, bool fast) {
  return fast ? fwd_group_fn_f<true>(dt, kt) : fwd_group_fn_f<false>(dt, kt);
}

template <int KT>
const void *fwd_rowwarp_fn_kt(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_fwd_rowwarp_kernel<float, KT>);
    case FOS_BF16: return reinterpret_cast<const void *>(&fos_fwd_rowwarp_kernel<__nv_bfloat16, KT>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_fwd_rowwarp_kernel<__half, KT>);
  }
  return nullptr;
}

const void *fwd_rowwarp_fn(fos_dtype dt, int kt) {
  return kt <= 2 ? fwd_rowwarp_fn_kt<2>(dt) : (kt <= 4 ? fwd_rowwarp_fn_kt<4>(dt)
                                                        : fwd_rowwarp_fn_kt<8>(dt));
}

template <int KT, bool kFast>
const void *fwd_fn_kt(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_fwd_kernel<float, KT, kFast>);
    case FOS_BF16: return reinterpret_cast<const void *>(&fos_fwd_kernel<__nv_bfloat16, KT, kFast>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_fwd_kernel<__half, KT, kFast>);
  }
  return nullptr;
}

template <bool kFast>
const void *fwd_fn_f(fos_dtype dt, int kt) {
  switch (kt) {
    case 2: return fwd_fn_kt<2, kFast>(dt);
    case 4: return fwd_fn_kt<4, kFast>(dt);
    case 6: return fwd_fn_kt<6, kFast>(dt);
    default: return fwd_fn_kt<8, kFast>(dt);
  }
}

const void *fwd_fn(fos_dtype dt, int kt, bool fast) {
  return fast ? fwd_fn_f<true>(dt, kt) : fwd_fn_f<false>(dt, kt);
}

}  // namespace

size_t fwd_extra_smem(int T, int stages) {
  (void)stages;
  // tm and ts (T rounded up to 4), then tc, which is also the merge's 64-float scratch
  const int T4 = (T + 3) & ~3;
  // (and 16 bytes for the tensor-memory address)
  return (size_t)kBarBytes + kGeoBytes + (size_t)(2 * T4 + (T4 > 64 ? T4 : 64)) * sizeof(float) +
         16;
}

size_t fwd_stream_extra_smem(int T, int stages) {
  // fwd_extra_smem's layout, then 16 "statistics" mbarriers and the merge warp's 64-float scratch
  return fwd_extra_smem(T, stages) + 16 * sizeof(uint64_t) + 64 * sizeof(float);
}

uint32_t fwd_tmem_cols(int warps, int kt) {
  // warps sharing a lane quarter take consecutive column ranges of kt * 8
  const uint32_t need = (uint32_t)(((warps + 3) / 4) * kt * 8);
  uint32_t cols = 32;
  while (cols < need) cols <<= 1;
  return cols;
}

int fwd_tiles_per_warp(int T, int warps) {
  // the smallest even count of 2..8 that holds the row; past 8 per warp e_j are recomputed
  const int need = (T + warps - 1) / warps;
  if (need <= 2) return 2;
  if (need <= 4) return 4;
  if (need <= 6) return 6;
  return 8;
}

int fwd_default_warps(int T) {
  // Fitted to timings of the unmasked and causal bf16 forward on GB300 over 256..16384 keys
  // (any choice gives the same bits), with e_j parked in tensor memory: four tiles per warp on
  // short rows, six on 17..24 tiles, eight (the most a warp parks) on longer ones.
  if (T <= 1) return 1;
  if (T <= 16) return (T + 3) / 4;
  if (T <= 24) return (T + 5) / 6;
  if (T <= 128) return (T + 7) / 8;  // up to 16 warps
  return 8;                          // e_j recomputed in the second pass
}

cudaError_t fwd_prepare(fos_dtype dt, int max_smem) {
  for (int kt : {2, 4, 6, 8})
    for (bool fast : {false, true}) {
      cudaError_t e = cudaFuncSetAttribute(fwd_fn(dt, kt, fast),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
      if (e != cudaSuccess) return e;
      // all of the SM's on-chip memory as shared memory: the host's residency count for these
      // instances (which allocate tensor memory) assumes it
      e = cudaFuncSetAttribute(fwd_fn(dt, kt, fast), cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
    }
  for (int kt : {4, 6, 8})
    for (bool fast : {false, true}) {
      cudaError_t e = cudaFuncSetAttribute(fwd_group_fn(dt, kt, fast),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fwd_group_fn(dt, kt, fast),
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
    }
  for (int kt : {2, 4, 8}) {
    cudaError_t e = cudaFuncSetAttribute(fwd_rowwarp_fn(dt, kt),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fwd_rowwarp_fn(dt, kt), cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaFuncSetAttribute(fwd_stream_fn(dt), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_smem);
}

size_t fwd_group_smem(int groups, int stages, size_t stage_bytes, int T) {
  // barriers and row records, the groups' rings, their statistics, the tensor-memory address
  const int T4 = (T + 3) & ~3;
  const size_t nstat = (size_t)(2 * T4 + (T4 > 64 ? T4 : 64));
  return (size_t)kGrpHead + (size_t)groups * stages * stage_bytes +
         (size_t)groups * nstat * sizeof(float) + 16;
}

cudaError_t fwd_group_attributes(fos_dtype dt, int kt, bool fast, cudaFuncAttributes *fa) {
  return cudaFuncGetAttributes(fa, fwd_group_fn(dt, kt, fast));
}

cudaError_t fwd_group_launch(fos_dtype dt, int kt, bool fast, const FwdArgs &a, int grid,
                             int threads, size_t smem, cudaStream_t s) {
  void *args[] = {const_cast<FwdArgs *>(&a)};
  return cudaLaunchKernel(fwd_group_fn(dt, kt, fast), dim3(grid), dim3(threads), args, smem, s);
}

cudaError_t fwd_rowwarp_launch(fos_dtype dt, int kt, const FwdArgs &a, int grid, int threads,
                               size_t smem, cudaStream_t s) {
  void *args[] = {const_cast<FwdArgs *>(&a)};
  return cudaLaunchKernel(fwd_rowwarp_fn(dt, kt), dim3(grid), dim3(threads), args, smem, s);
}

size_t fwd_rowwarp_smem(int warps, int stages, size_t stage_bytes) {
  // per warp: its buffers and 80 floats of tile statistics; then the tensor-memory address
  return (size_t)kBarBytes + kGeoBytes + (size_t)warps * stages * stage_bytes +
         (size_t)warps * 80 * sizeof(float) + 16;
}

cudaError_t fwd_rowwarp_attributes(fos_dtype dt, int kt, cudaFuncAttributes *fa) {
  return cudaFuncGetAttributes(fa, fwd_rowwarp_fn(dt, kt));
}

cudaError_t fwd_stream_occupancy(fos_dtype dt, int threads, size_t smem, int *blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fwd_stream_fn(dt), threads,
                                                       smem);
}

cudaError_t fwd_stream_launch(fos_dtype dt, const FwdArgs &a, int grid, int threads, size_t smem,
                              cudaStream_t s) {
  void *args[] = {const_cast<FwdArgs *>(&a)};
  return cudaLaunchKernel(fwd_stream_fn(dt), dim3(grid), dim3(threads), args, smem, s);
}

cudaError_t fwd_attributes(fos_dtype dt, int kt, bool fast, cudaFuncAttributes *fa) {
  return cudaFuncGetAttributes(fa, fwd_fn(dt, kt, fast));
}

cudaError_t fwd_launch(fos_dtype dt, int kt, bool fast, const FwdArgs &a, int grid, int threads,
                       size_t smem, cudaStream_t s) {
  const void *fn = fwd_fn(dt, kt, fast);
  void *args[] = {const_cast<FwdArgs *>(&a)};
  return cudaLaunchKernel(fn, dim3(grid), dim3(threads), args, smem, s);
}

}  // namespace fos
