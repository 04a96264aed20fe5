// fos_bwd.cu -- backward kernel of the fixed-order row softmax (delta, dScores), sm_103a.
//
// The softmax VJP on the P the caller passes in ("[WS1][kernels] Add fixed-order
// joint-attention softmax for Qwen-Image", Summary, "Fixed-order backward"):
//
//   delta = fixed_sum(P * dP)          dScores_j = P_j * (dP_j - delta)
//
// with the forward's tile layout and order: inside tile t lane l multiplies and accumulates
// keys 256t + 8l .. +7 in ascending order with fused multiply-adds, the lanes are combined by
// the xor tree (16, 8, 4, 2, 1), and tile partials are added left to right.  dScores is formed
// as fma(P_j, dP_j - delta, +0) so that a zero product is +0 whatever the sign of the
// difference, and rounded once.  Masked keys are skipped in the sum and written as +0.
//
// Structure as in the forward: persistent CTAs, a producer warp that alone issues the 1-D bulk
// copies (P and dP of a row on one mbarrier) into a ring of staged rows, compute warps that
// own one complete row at a time; thread 0 adds the tile partials, everything else is
// tile-parallel over the compute warps.  Pass 2 re-reads P and dP from shared memory, and each
// compute warp releases the stage to the producer when its pass 2 is done.
#include "fos_device.cuh"
#include "fos_internal.h"

namespace fos {
namespace {

constexpr int kBarBytes = 256;  // 16 "full" and 16 "empty" mbarriers
constexpr int kGeoBytes = 256;  // up to 16 per-stage row records (int4)

__device__ __forceinline__ bool key_ok(int j, int lim, const uint8_t *km) {
  return (j < lim) && (km == nullptr || km[j] != 0);
}

template <typename T>
__device__ __forceinline__ void tile_pdp(const unsigned char *sp, const unsigned char *sd, int j0,
                                         float (&p)[8], float (&d)[8]) {
  constexpr int esz = Io<T>::kEsz;
  Io<T>::widen(Io<T>::lds(sp + (size_t)j0 * esz), p);
  Io<T>::widen(Io<T>::lds(sd + (size_t)j0 * esz), d);
}

// Lane-local ascending fused multiply-add over the lane's 8 keys (the xor tree follows).
__device__ __forceinline__ float lane_dot(const float (&p)[8], const float (&d)[8], int j0,
                                          int lim, const uint8_t *km, bool masked) {
  float acc = 0.0f;
  if (masked) {
#pragma unroll
    for (int q = 0; q < kLaneKeys; ++q)
      if (key_ok(j0 + q, lim, km)) acc = __fmaf_rn(p[q], d[q], acc);
  } else {
#pragma unroll
    for (int q = 0; q < kLaneKeys; ++q) acc = __fmaf_rn(p[q], d[q], acc);
  }
  return acc;
}

// lane_dot of two unmasked tiles at once, packed (.x: first tile, .y: second).  The packed
// float32 fused multiply-add of the sm_100 family (__ffma2_rn) rounds each component as
// __fmaf_rn does, so each component has the bits of lane_dot on its own tile.
__device__ __forceinline__ float2 lane_dot2(const float (&p0)[8], const float (&d0)[8],
                                            const float (&p1)[8], const float (&d1)[8]) {
  float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int q = 0; q < kLaneKeys; ++q)
    acc = __ffma2_rn(make_float2(p0[q], p1[q]), make_float2(d0[q], d1[q]), acc);
  return acc;
}

// dScores of the lane's 8 keys: fma(P, dP - delta, +0), +0 for masked keys.  Unmasked tiles
// take neighbouring keys two at a time in packed form (dP - delta as dP + (-delta), the same
// IEEE operation; same bits per key).
__device__ __forceinline__ void tile_grad(const float (&p)[8], const float (&d)[8], int j0,
                                          int lim, const uint8_t *km, bool masked, float delta,
                                          float (&v)[8]) {
  if (!masked) {
    const float2 nd = make_float2(-delta, -delta), zero = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < kLaneKeys; q += 2) {
      const float2 x = __fadd2_rn(make_float2(d[q], d[q + 1]), nd);
      const float2 g = __ffma2_rn(make_float2(p[q], p[q + 1]), x, zero);
      v[q] = g.x;
      v[q + 1] = g.y;
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < kLaneKeys; ++q) {
    const float g = __fmaf_rn(p[q], __fsub_rn(d[q], delta), 0.0f);
    v[q] = key_ok(j0 + q, lim, km) ? g : 0.0f;
  }
}

// Pass 1 over the staged tiles tl = w, w + nw, ... < nt (a whole row, or one segment of it,
// whose keys are numbered from 0 and valid below lim): the tile partials of delta into td[tl],
// two tiles at a time.
template <typename T>
__device__ __forceinline__ void delta_partials(const unsigned char *sp, const unsigned char *sd,
                                               int nt, int w, int nw, int lane, int lim,
                                               const uint8_t *km, float *td) {
  int t = w;
  for (; t + nw < nt; t += 2 * nw) {
    const int t1 = t + nw;
    const int j0 = t * kTileK + lane * kLaneKeys, j1 = t1 * kTileK + lane * kLaneKeys;
    float p0[8], d0[8], p1[8], d1[8];
    tile_pdp<T>(sp, sd, j0, p0, d0);
    tile_pdp<T>(sp, sd, j1, p1, d1);
    const bool m0 = km != nullptr || (t + 1) * kTileK > lim;
    const bool m1 = km != nullptr || (t1 + 1) * kTileK > lim;
    float2 acc = (m0 || m1) ? make_float2(lane_dot(p0, d0, j0, lim, km, m0),
                                          lane_dot(p1, d1, j1, lim, km, m1))
                            : lane_dot2(p0, d0, p1, d1);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)  // the xor tree of both tiles, packed
      acc = __fadd2_rn(acc, make_float2(__shfl_xor_sync(kFull, acc.x, o),
                                        __shfl_xor_sync(kFull, acc.y, o)));
    if (lane == 0) {
      td[t] = acc.x;
      td[t1] = acc.y;
    }
  }
  if (t < nt) {
    const int j0 = t * kTileK + lane * kLaneKeys;
    float p0[8], d0[8];
    tile_pdp<T>(sp, sd, j0, p0, d0);
    const float a0 =
        warp_sum_xor(lane_dot(p0, d0, j0, lim, km, km != nullptr || (t + 1) * kTileK > lim));
    if (lane == 0) td[t] = a0;
  }
}

// Pass 2 over the same staged tiles: dScores of tile tl written at tile t_base + tl of the row.
template <typename T>
__device__ __forceinline__ void grad_tiles(const unsigned char *sp, const unsigned char *sd,
                                           int nt, int w, int nw, int lane, int lim,
                                           const uint8_t *km, float delta, unsigned char *grow,
                                           int t_base, int L, bool ovec) {
  for (int t = w; t < nt; t += nw) {
    const int j0 = t * kTileK + lane * kLaneKeys;
    float p[8], d[8], v[8];
    tile_pdp<T>(sp, sd, j0, p, d);
    const bool masked = km != nullptr || (t + 1) * kTileK > lim;
    tile_grad(p, d, j0, lim, km, masked, delta, v);
    store_lane8<T>(grow, (t_base + t) * kTileK + lane * kLaneKeys, L, ovec, v);
  }
}

// ---- the rows a CTA or a warp takes, in order
//
// Plain: rows first, first + step, ... below a.rows.  Octets (the sink gradient fused into
// the backward): octets first, first + step, ... of all heads (octet o: head o / oct_per_head,
// positions 8m .. 8m + 7 below pos_end, m = o % oct_per_head), each octet's rows in position
// order, position p of head h being row (p / q_len * heads + h) * q_len + p % q_len.  The
// cursor tells where an octet ends, so that its sum can be written.
template <bool kOct>
struct RowCursor;

// Rows are taken from the last to the first.  The forward writes P from the first row to the
// last, so a backward that follows it starts on the rows whose P the forward wrote last, the
// likeliest to be still in L2.  The order of rows never changes a row's bits.
template <>
struct RowCursor<false> {
  int64_t k;     // rows counted from the last one
  int64_t last;  // the launch's last row
  __device__ RowCursor(const BwdArgs &a, int64_t first) : k(first), last(a.rows - 1) {}
  __device__ bool valid(const BwdArgs &a) const { return k < a.rows; }
  __device__ int64_t row() const { return last - k; }
  __device__ void next(const BwdArgs &, int64_t step) { k += step; }
};

// The octet cursor moves from row to row incrementally: the next position of a head is the next
// row (b, h, i + 1), or, past the last query of a batch entry, row (b + 1, h, 0), which lies
// 1 + (heads - 1) * q_len rows further on.  Only a new octet needs divisions.
template <>
struct RowCursor<true> {
  int64_t o;  // octet
  int64_t r;  // current row
  int32_t q;  // position within the octet
  int32_t n;  // positions of this octet (8, fewer at the end of a head)
  int32_t i;  // query index of the current row
  int32_t h;  // head
  __device__ RowCursor(const BwdArgs &a, int64_t first) : o(first) { seek(a); }
  __device__ void seek(const BwdArgs &a) {
    q = 0;
    if (!valid(a)) return;
    const int64_t hh = a.oct32 ? (int64_t)fast_div((uint32_t)o, a.octdiv) : o / a.oct_per_head;
    const int64_t p = 8 * (o - hh * a.oct_per_head);
    const int64_t b = a.oct32 ? (int64_t)fast_div((uint32_t)p, a.qdiv) : p / a.q_len;
    h = (int32_t)hh;
    i = (int32_t)(p - b * a.q_len);
    n = (int32_t)min((int64_t)8, a.pos_end - p);
    r = (b * a.heads + hh) * a.q_len + i;
  }
  __device__ bool valid(const BwdArgs &a) const { return o < (int64_t)a.heads * a.oct_per_head; }
  __device__ int64_t row() const { return r; }
  __device__ int64_t head() const { return h; }
  __device__ bool octet_end() const { return q + 1 == n; }  // the current row is its octet's last
  __device__ void next(const BwdArgs &a, int64_t step) {
    if (octet_end()) {
      o += step;
      seek(a);
    } else {
      ++q;
      if (++i == a.q_len) {
        i = 0;
        r += 1 + (int64_t)(a.heads - 1) * a.q_len;
      } else {
        ++r;
      }
    }
  }
};

// Row r's term of the sink gradient, as the sink-gradient kernel forms it: c_r = -(exp(sink_h -
// lse_r) * delta_r), with exp(sink_h - lse_r) taken as 0 for a -inf sink.  The sink and LSE
// values are loaded when the row starts (sink_inputs), so their latency hides behind pass 1.
__device__ __forceinline__ float2 sink_inputs(const BwdArgs &a, int64_t h, int64_t r) {
  return make_float2(a.sink[h], a.lse[r]);
}

__device__ __forceinline__ float sink_term(float2 sl, float delta) {
  const float ps = (sl.x == -INFINITY) ? 0.0f : scale_fos(sl.x, sl.y);
  return -__fmul_rn(ps, delta);
}

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

// Thread 0: record row rr's geometry and start the bulk copies of its P and dP.
template <typename T>
__device__ __forceinline__ void issue_row(const BwdArgs &a, int64_t rr, unsigned char *stage,
                                          uint64_t *bar, int4 *geo, bool skip_copy) {
  constexpr int esz = Io<T>::kEsz;
  const int4 g = row_geometry(a, rr);
  *geo = g;
  const uint32_t bytes = ((uint32_t)g.x * esz + 15u) & ~15u;
  if (skip_copy) return;  // test only: this row's copies are never issued
  const uint32_t bar_a = smem_addr(bar);
  mbar_arrive_expect_tx(bar_a, 2u * bytes);
  if (bytes) {
    const size_t off = (size_t)rr * a.ld * esz;
    bulk_g2s(smem_addr(stage), static_cast<const unsigned char *>(a.probs) + off, bytes, bar_a);
    bulk_g2s(smem_addr(stage + a.stage_bytes), static_cast<const unsigned char *>(a.dprobs) + off,
             bytes, bar_a);
  }
}

// Producer (lane 0 of the last warp): as in the forward, it alone issues the bulk copies
// (P and dP of a row on one "full" barrier) once the compute warps have released the stage,
// and waits for every copy it issued before it exits.
template <typename T, bool kOct>
__device__ void bwd_produce(const BwdArgs &a, RowCursor<kOct> cur, int64_t step, uint64_t *full,
                            uint64_t *empty, int4 *geos, unsigned char *ring, size_t slot,
                            bool stall) {
  const int NS = a.stages;
  uint32_t issued = 0, last_ph = 0;
  int s = 0;
  uint32_t ph = 0;
  for (int64_t kk = 0; cur.valid(a); ++kk, cur.next(a, step)) {
    if (kk >= NS && !mbar_wait_bounded(smem_addr(&empty[s]), ph ^ 1u, a.timeout_ns)) {
      raise_device_error(a.err, kDevErrTimeout);
      break;
    }
    const bool skip = stall && kk == 0;
    issue_row<T>(a, cur.row(), ring + (size_t)s * slot, &full[s], &geos[s], skip);
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

// kFast: the common case fixed at compile time (bulk copies, no mask, 16-byte aligned output).
// Both instances do the same arithmetic in the same order.
template <typename T, bool kFast, bool kSink>
__global__ void __maxnreg__(72) fos_bwd_kernel(const BwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + 16;
  int4 *geos = reinterpret_cast<int4 *>(smem + kBarBytes);
  unsigned char *ring = smem + kBarBytes + kGeoBytes;
  const size_t slot = 2 * (size_t)a.stage_bytes;
  float *td = reinterpret_cast<float *>(ring + (size_t)a.stages * slot);
  float *dsm = td + ((a.T + 3) & ~3);  // delta of the current row, for every warp

  const int tid = threadIdx.x;
  const int nw = (blockDim.x >> 5) - 1;  // compute warps; the last warp is the producer
  const int ncomp = nw * 32;
  const int w = tid >> 5;
  const int lane = tid & 31;
  const int64_t G = gridDim.x;
  RowCursor<kSink> cur(a, blockIdx.x);
  if (!cur.valid(a)) return;
  const int NS = a.stages;
  const bool use_bulk = kFast || a.use_bulk != 0;

  if (use_bulk) {
    if (tid == 0) {
      for (int t = 0; t < NS; ++t) {
        mbar_init(smem_addr(&full[t]), 1);
        mbar_init(smem_addr(&empty[t]), nw);
      }
      fence_mbar_init();
    }
    __syncthreads();
  }
  if (w == nw) {
    if (use_bulk && lane == 0)
      bwd_produce<T, kSink>(a, cur, G, full, empty, geos, ring, slot,
                            a.test_stall && blockIdx.x == 0);
    return;
  }

  // stage index and phase parity of the current row, carried rather than computed
  int s = 0;
  uint32_t ph = 0;
  float acc = 0.0f;  // thread 0, sink fusion: the octet's ascending sum of c_r
  for (; cur.valid(a); cur.next(a, G), s = (s + 1 == NS) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
    const int64_t r = cur.row();
    unsigned char *sp = ring + (size_t)s * slot;
    unsigned char *sd = sp + a.stage_bytes;
    float2 sl = make_float2(0.0f, 0.0f);
    if constexpr (kSink)
      if (tid == 0) sl = sink_inputs(a, cur.head(), r);

    bool timed_out = false;
    int4 g;
    if (use_bulk) {
      timed_out = !mbar_wait_bounded(smem_addr(&full[s]), ph, a.timeout_ns);
      g = kFast ? make_int4(a.L, 0, 0, 0) : geos[s];
    } else {
      if (tid == 0) geos[0] = row_geometry(a, r);
      compute_sync(ncomp);  // also: every warp is done with the previous row's stage
      g = geos[0];
      const size_t off = (size_t)r * a.ld * esz;
      plain_stage<T>(sp, static_cast<const unsigned char *>(a.probs) + off, g.x, a.in_vec != 0,
                     ncomp);
      plain_stage<T>(sd, static_cast<const unsigned char *>(a.dprobs) + off, g.x, a.in_vec != 0,
                     ncomp);
      compute_sync(ncomp);
    }
    const int lim = g.x;
    int Te = (lim + kTileK - 1) / kTileK;
    const uint8_t *km = (!kFast && a.key_mask) ? a.key_mask + (int64_t)g.y * a.L : nullptr;
    if (!dbg_ok(a.err, Te <= a.T && (uint32_t)(Te * kTileK * esz) <= a.stage_bytes &&
                           r < a.rows)) {
      Te = 0;  // no tile is read, and the row stops below as after a wait that ran out
      timed_out = true;
    }

    // ---- pass 1: tile partials of delta, two tiles at a time
    delta_partials<T>(sp, sd, Te, w, nw, lane, lim, km, td);

    if (compute_sync_or(ncomp, timed_out)) {
      if (tid == 0) raise_device_error(a.err, kDevErrTimeout);
      return;
    }

    // ---- tile partials added left to right (one thread)
    if (tid == 0) {
      // four partials per shared-memory load (td is 16-byte aligned)
      float delta = 0.0f;
      int t = 0;
      for (; t + 4 <= Te; t += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(td + t);
        delta = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(delta, v.x), v.y), v.z), v.w);
      }
      for (; t < Te; ++t) delta = __fadd_rn(delta, td[t]);
      dsm[0] = delta;
      if (a.delta) a.delta[r] = delta;
      if constexpr (kSink) {
        acc = __fadd_rn(acc, sink_term(sl, delta));
        if (cur.octet_end()) {
          a.oct_sums[cur.o] = acc;
          acc = 0.0f;
        }
      }
    }
    compute_sync(ncomp);
    const float delta = dsm[0];

    // ---- pass 2: dScores
    unsigned char *grow = static_cast<unsigned char *>(a.dscores) + (size_t)r * a.ld * esz;
    const bool ovec = kFast || a.out_vec != 0;
    grad_tiles<T>(sp, sd, Te, w, nw, lane, lim, km, delta, grow, 0, a.L, ovec);
    if (use_bulk) {  // done with the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    }
    for (int t = Te + w; t < a.T; t += nw) {
      float z[8];
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) z[q] = 0.0f;
      store_lane8<T>(grow, t * kTileK + lane * kLaneKeys, a.L, ovec, z);
    }
  }
}

// ------------------------------------------------------ short rows: one warp per row
//
// As in the forward, a row of at most 8 tiles is taken by one warp alone: pass 1 (tile
// partials of delta), the left-to-right sum of the partials (every lane adds them in the same
// order, so no thread has to broadcast delta) and pass 2 (dScores), with no barrier between
// the warps of a CTA.  Each warp keeps its own ring of a.stages buffers (P and dP of a row) and
// its lane 0 refills a buffer with the copies of row k + stages once pass 2 of row k is done.
// The per-tile arithmetic and the order of the delta sum are fos_bwd_kernel's.

// Lane 0: geometry of row rr into *geo and the bulk copies of its P and dP into `stage`.
template <typename T>
__device__ __forceinline__ void rw_issue(const BwdArgs &a, int64_t rr, unsigned char *stage,
                                         uint64_t *bar, int4 *geo) {
  constexpr int esz = Io<T>::kEsz;
  const int4 g = row_geometry(a, rr);
  *geo = g;
  const uint32_t bytes = ((uint32_t)g.x * esz + 15u) & ~15u;  // never past the row
  const uint32_t bar_a = smem_addr(bar);
  fence_proxy_async_smem();  // the warp's reads of this buffer come before the copies
  mbar_arrive_expect_tx(bar_a, 2u * bytes);
  if (bytes) {
    const size_t off = (size_t)rr * a.ld * esz;
    bulk_g2s(smem_addr(stage), static_cast<const unsigned char *>(a.probs) + off, bytes, bar_a);
    bulk_g2s(smem_addr(stage + a.stage_bytes), static_cast<const unsigned char *>(a.dprobs) + off,
             bytes, bar_a);
  }
}

template <typename T, bool kSink>
__global__ void __maxnreg__(72) fos_bwd_rowwarp_kernel(const BwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  const int nw = blockDim.x >> 5;
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = a.stages;  // row buffers per warp
  const size_t slot = 2 * (size_t)a.stage_bytes;
  const int T4 = (a.T + 3) & ~3;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem) + w * NS;
  int4 *geos = reinterpret_cast<int4 *>(smem + kBarBytes) + w * NS;
  unsigned char *ring = smem + kBarBytes + kGeoBytes + (size_t)w * NS * slot;
  float *td = reinterpret_cast<float *>(smem + kBarBytes + kGeoBytes + (size_t)nw * NS * slot) +
              w * T4;

  const int64_t GW = (int64_t)gridDim.x * nw;               // warps in the grid
  RowCursor<kSink> cur(a, (int64_t)blockIdx.x * nw + w);      // the row being computed
  const bool stall = a.test_stall && blockIdx.x == 0 && w == 0;

  if (lane == 0) {
    for (int t = 0; t < NS; ++t) mbar_init(smem_addr(&full[t]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  uint32_t issued = 0, last_ph = 0;
  {
    RowCursor<kSink> iss = cur;
    for (int t = 0; t < NS && iss.valid(a); ++t, iss.next(a, GW))
      if (lane == 0 && !(stall && t == 0)) {  // test only: the very first copies never issued
        rw_issue<T>(a, iss.row(), ring + (size_t)t * slot, &full[t], &geos[t]);
        issued |= 1u << t;
      }
  }

  int s = 0;
  uint32_t ph = 0;
  bool ok = true;
  float acc = 0.0f;  // sink fusion: the octet's ascending sum of c_r (every lane the same)
  while (cur.valid(a)) {
    RowCursor<kSink> nxt = cur;  // the warp's next row, for the copy and for the next iteration
    nxt.next(a, GW);
    const int64_t r = cur.row();
    unsigned char *sp = ring + (size_t)s * slot;
    float2 sl = make_float2(0.0f, 0.0f);
    if constexpr (kSink) sl = sink_inputs(a, cur.head(), r);
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
    if (!dbg_ok(a.err, Te <= a.T && (uint32_t)(Te * kTileK * esz) <= a.stage_bytes &&
                           r < a.rows)) {
      ok = false;  // the warp stops as after a wait that ran out
      break;
    }

    // ---- pass 1: tile partials of delta, then their sum left to right (every lane)
    delta_partials<T>(sp, sp + a.stage_bytes, Te, 0, 1, lane, lim, km, td);
    __syncwarp();
    float delta = 0.0f;
    {
      int t = 0;
      for (; t + 4 <= Te; t += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(td + t);
        delta = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(delta, v.x), v.y), v.z), v.w);
      }
      for (; t < Te; ++t) delta = __fadd_rn(delta, td[t]);
    }
    if (lane == 0 && a.delta) a.delta[r] = delta;
    if constexpr (kSink) {
      acc = __fadd_rn(acc, sink_term(sl, delta));
      if (cur.octet_end()) {
        if (lane == 0) a.oct_sums[cur.o] = acc;
        acc = 0.0f;
      }
    }

    // ---- pass 2: dScores
    unsigned char *grow = static_cast<unsigned char *>(a.dscores) + (size_t)r * a.ld * esz;
    const bool ovec = a.out_vec != 0;
    grad_tiles<T>(sp, sp + a.stage_bytes, Te, 0, 1, lane, lim, km, delta, grow, 0, a.L, ovec);
    for (int t = Te; t < a.T; ++t) {
      float z[8];
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) z[q] = 0.0f;
      store_lane8<T>(grow, t * kTileK + lane * kLaneKeys, a.L, ovec, z);
    }
    __syncwarp();  // td is rewritten by the next row; every lane is done with the buffer
    {
      // the row `stages` rows after this one goes into this buffer
      RowCursor<kSink> iss = nxt;
      for (int t = 1; t < NS && iss.valid(a); ++t) iss.next(a, GW);
      if (iss.valid(a) && lane == 0) {
        rw_issue<T>(a, iss.row(), sp, &full[s], &geos[s]);
        issued |= 1u << s;
        last_ph = (last_ph & ~(1u << s)) | ((ph ^ 1u) << s);
      }
    }
    cur = nxt;
    if (++s == NS) {
      s = 0;
      ph ^= 1u;
    }
  }
  // every copy this warp issued has landed before it exits
  if (!ok && lane == 0)
    for (int t = 0; t < NS; ++t)
      if (issued & (1u << t))
        mbar_wait_bounded(smem_addr(&full[t]), (last_ph >> t) & 1u, a.timeout_ns);
}

template <bool kSink>
const void *bwd_rowwarp_fn_s(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_bwd_rowwarp_kernel<float, kSink>);
    case FOS_BF16:
      return reinterpret_cast<const void *>(&fos_bwd_rowwarp_kernel<__nv_bfloat16, kSink>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_bwd_rowwarp_kernel<__half, kSink>);
  }
  return nullptr;
}

const void *bwd_rowwarp_fn(fos_dtype dt, bool sink = false) {
  return sink ? bwd_rowwarp_fn_s<true>(dt) : bwd_rowwarp_fn_s<false>(dt);
}

// ------------------------------------------------ rows longer than shared memory (streaming)
//
// As in the forward: a row too long to stage is read twice, in segments of a.seg_tiles tiles
// of P and dP that cycle through the ring; pass 1 takes the tile partials of delta segment by
// segment, one thread adds them left to right, and pass 2 reads every segment again for
// dScores.  The per-tile arithmetic and the order of the delta sum are those of
// fos_bwd_kernel, so a row gives the same bits on either path.  Rows are taken from the last
// to the first, as in fos_bwd_kernel (the forward's last rows of P are the likeliest in L2).

// Producer: each row's segments of P and dP twice (pass 1, then pass 2), with the row's record
// beside every segment; a row with no valid key still gets one empty segment per pass.
template <typename T>
__device__ void bwd_stream_produce(const BwdArgs &a, int64_t r0, int64_t G, int64_t nmine,
                                   uint64_t *full, uint64_t *empty, int4 *geos,
                                   unsigned char *ring, size_t slot, bool stall) {
  constexpr int esz = Io<T>::kEsz;
  const int NS = a.stages;
  const int seg_keys = a.seg_tiles * kTileK;
  uint32_t issued = 0, last_ph = 0;
  int s = 0;
  uint32_t ph = 0;
  int64_t n = 0;  // segments issued so far
  bool stop = false;
  for (int64_t kk = 0; kk < nmine && !stop; ++kk) {
    const int64_t rr = a.rows - 1 - (r0 + kk * G);
    const int4 g = row_geometry(a, rr);
    const int nseg = g.x > 0 ? (g.x + seg_keys - 1) / seg_keys : 1;
    const size_t off = (size_t)rr * a.ld * esz;
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
        const uint32_t bytes = ((uint32_t)nk * esz + 15u) & ~15u;  // never past the row
        if (!(stall && n == 0)) {  // test only: the first copies are never issued
          const uint32_t bar_a = smem_addr(&full[s]);
          mbar_arrive_expect_tx(bar_a, 2u * bytes);
          if (bytes) {
            unsigned char *st = ring + (size_t)s * slot;
            const size_t so = off + (size_t)k0 * esz;
            bulk_g2s(smem_addr(st), static_cast<const unsigned char *>(a.probs) + so, bytes, bar_a);
            bulk_g2s(smem_addr(st + a.stage_bytes),
                     static_cast<const unsigned char *>(a.dprobs) + so, bytes, bar_a);
          }
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

template <typename T>
__global__ void __maxnreg__(80) fos_bwd_stream_kernel(const BwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int esz = Io<T>::kEsz;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + 16;
  int4 *geos = reinterpret_cast<int4 *>(smem + kBarBytes);
  unsigned char *ring = smem + kBarBytes + kGeoBytes;
  const size_t slot = 2 * (size_t)a.stage_bytes;
  float *td = reinterpret_cast<float *>(ring + (size_t)a.stages * slot);
  float *dsm = td + ((a.T + 3) & ~3);

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
  const int SEG = a.seg_tiles;

  if (tid == 0) {
    for (int t = 0; t < NS; ++t) {
      mbar_init(smem_addr(&full[t]), 1);
      mbar_init(smem_addr(&empty[t]), nw);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (w == nw) {
    if (lane == 0)
      bwd_stream_produce<T>(a, r0, G, nmine, full, empty, geos, ring, slot,
                            a.test_stall && blockIdx.x == 0);
    return;
  }

  int s = 0;
  uint32_t ph = 0;
  for (int64_t k = 0; k < nmine; ++k) {
    const int64_t r = a.rows - 1 - (r0 + k * G);
    bool timed_out = false;
    int lim = 0, Te = 0, nseg = 1;
    const uint8_t *km = nullptr;

    // ---- pass 1: tile partials of delta, segment by segment
    for (int seg = 0; seg < nseg; ++seg) {
      if (!mbar_wait_bounded(smem_addr(&full[s]), ph, a.timeout_ns)) {
        timed_out = true;
        break;
      }
      if (seg == 0) {
        const int4 g = geos[s];
        lim = g.x;
        Te = (lim + kTileK - 1) / kTileK;
        nseg = Te > 0 ? (Te + SEG - 1) / SEG : 1;
        km = a.key_mask ? a.key_mask + (int64_t)g.y * a.L : nullptr;
      }
      const unsigned char *sp = ring + (size_t)s * slot;
      const int t0 = seg * SEG;
      delta_partials<T>(sp, sp + a.stage_bytes, min(SEG, Te - t0), w, nw, lane,
                        lim - t0 * kTileK, km ? km + t0 * kTileK : nullptr, td + t0);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
      if (++s == NS) {
        s = 0;
        ph ^= 1u;
      }
    }
    if (compute_sync_or(ncomp, timed_out)) {
      if (tid == 0) raise_device_error(a.err, kDevErrTimeout);
      return;
    }

    // ---- tile partials added left to right (one thread), as in fos_bwd_kernel
    if (tid == 0) {
      float delta = 0.0f;
      int t = 0;
      for (; t + 4 <= Te; t += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(td + t);
        delta = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(delta, v.x), v.y), v.z), v.w);
      }
      for (; t < Te; ++t) delta = __fadd_rn(delta, td[t]);
      dsm[0] = delta;
      if (a.delta) a.delta[r] = delta;
    }
    compute_sync(ncomp);
    const float delta = dsm[0];

    // ---- pass 2: every segment again, dScores
    unsigned char *grow = static_cast<unsigned char *>(a.dscores) + (size_t)r * a.ld * esz;
    const bool ovec = a.out_vec != 0;
    for (int seg = 0; seg < nseg; ++seg) {
      if (!mbar_wait_bounded(smem_addr(&full[s]), ph, a.timeout_ns)) {
        timed_out = true;
        break;
      }
      const unsigned char *sp = ring + (size_t)s * slot;
      const int t0 = seg * SEG;
      grad_tiles<T>(sp, sp + a.stage_bytes, min(SEG, Te - t0), w, nw, lane, lim - t0 * kTileK,
                    km ? km + t0 * kTileK : nullptr, delta, grow, t0, a.L, ovec);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
      if (++s == NS) {
        s = 0;
        ph ^= 1u;
      }
    }
    for (int t = Te + w; t < a.T; t += nw) {
      float z[8];
#pragma unroll
      for (int q = 0; q < kLaneKeys; ++q) z[q] = 0.0f;
      store_lane8<T>(grow, t * kTileK + lane * kLaneKeys, a.L, ovec, z);
    }
    // a wait that ran out in pass 2 stops every compute warp (none is left at a barrier)
    if (compute_sync_or(ncomp, timed_out)) {
      if (tid == 0) raise_device_error(a.err, kDevErrTimeout);
      return;
    }
  }
}

const void *bwd_stream_fn(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_bwd_stream_kernel<float>);
    case FOS_BF16: return reinterpret_cast<const void *>(&fos_bwd_stream_kernel<__nv_bfloat16>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_bwd_stream_kernel<__half>);
  }
  return nullptr;
}

template <bool kFast, bool kSink>
const void *bwd_fn_f(fos_dtype dt) {
  switch (dt) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_bwd_kernel<float, kFast, kSink>);
    case FOS_BF16:
      return reinterpret_cast<const void *>(&fos_bwd_kernel<__nv_bfloat16, kFast, kSink>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_bwd_kernel<__half, kFast, kSink>);
  }
  return nullptr;
}

const void *bwd_fn(fos_dtype dt, bool fast, bool sink = false) {
  if (sink) return fast ? bwd_fn_f<true, true>(dt) : bwd_fn_f<false, true>(dt);
  return fast ? bwd_fn_f<true, false>(dt) : bwd_fn_f<false, false>(dt);
}

}  // namespace

size_t bwd_extra_smem(int T, int stages) {
  (void)stages;
  return (size_t)kBarBytes + kGeoBytes + (size_t)(((T + 3) & ~3) + 4) * sizeof(float);
}

int bwd_default_warps(int T) {
  // About four tiles per warp, three from 17 to 24 tiles, never a single warp for more than
  // one tile (fitted to GB300 timings of the bf16 backward; any choice gives the same bits).
  if (T <= 1) return 1;
  if (T <= 4) return 2;
  if (T <= 6) return 3;
  if (T <= 8) return 2;
  const int w = (T >= 17 && T <= 24) ? (T + 2) / 3 : (T + 3) / 4;
  return w > 16 ? 16 : w;
}

cudaError_t bwd_prepare(fos_dtype dt, int max_smem) {
  for (bool sink : {false, true}) {
    for (bool fast : {false, true}) {
      cudaError_t e = cudaFuncSetAttribute(bwd_fn(dt, fast, sink),
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaFuncSetAttribute(bwd_rowwarp_fn(dt, sink),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
  }
  return cudaFuncSetAttribute(bwd_stream_fn(dt), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_smem);
}

size_t bwd_rowwarp_smem(int warps, int stages, size_t stage_bytes, int T) {
  return (size_t)kBarBytes + kGeoBytes + (size_t)warps * stages * 2 * stage_bytes +
         (size_t)warps * ((T + 3) & ~3) * sizeof(float);
}

cudaError_t bwd_rowwarp_occupancy(fos_dtype dt, int threads, size_t smem, int *blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, bwd_rowwarp_fn(dt), threads,
                                                       smem);
}

cudaError_t bwd_rowwarp_launch(fos_dtype dt, const BwdArgs &a, int grid, int threads, size_t smem,
                               cudaStream_t s, bool sink) {
  void *args[] = {const_cast<BwdArgs *>(&a)};
  return cudaLaunchKernel(bwd_rowwarp_fn(dt, sink), dim3(grid), dim3(threads), args, smem, s);
}

cudaError_t bwd_stream_occupancy(fos_dtype dt, int threads, size_t smem, int *blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, bwd_stream_fn(dt), threads,
                                                       smem);
}

cudaError_t bwd_stream_launch(fos_dtype dt, const BwdArgs &a, int grid, int threads, size_t smem,
                              cudaStream_t s) {
  void *args[] = {const_cast<BwdArgs *>(&a)};
  return cudaLaunchKernel(bwd_stream_fn(dt), dim3(grid), dim3(threads), args, smem, s);
}

cudaError_t bwd_occupancy(fos_dtype dt, bool fast, int threads, size_t smem, int *blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, bwd_fn(dt, fast), threads,
                                                       smem);
}

cudaError_t bwd_launch(fos_dtype dt, bool fast, const BwdArgs &a, int grid, int threads,
                       size_t smem, cudaStream_t s, bool sink) {
  void *args[] = {const_cast<BwdArgs *>(&a)};
  return cudaLaunchKernel(bwd_fn(dt, fast, sink), dim3(grid), dim3(threads), args, smem, s);
}

}  // namespace fos
