// fos_device.cuh -- device-side building blocks of the fixed-order row softmax (sm_103a).
//
// Everything that fixes a result bit lives here, so the forward, backward and sink kernels
// share one arithmetic contract:
//   * exp_fos / scale_fos  -- the exponential and the guarded rescale factor;
//   * warp_max_xor / warp_sum_xor -- the fixed xor-shuffle trees (offsets 16, 8, 4, 2, 1);
//   * Io<T> -- widening loads of 8 keys and the single rounding to the I/O dtype.
// The rest is data movement: mbarrier and 1-D bulk-copy (TMA) wrappers with bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fos_internal.h"

#ifdef __USE_FAST_MATH__
#error "libfos_softmax must be built without fast-math: it would change the arithmetic contract"
#endif

namespace fos {

constexpr int kLaneKeys = 8;   // contiguous keys per lane inside a tile
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned kDevErrTimeout = 1u;  // value stored in the device error word
constexpr unsigned kDevErrIndex = 2u;    // an index check of the debug build failed

// ------------------------------------------------------------------ arithmetic contract

// exp(d) by the base change exp(d) = 2^(d * log2 e): one round-to-nearest float32 multiply by
// log2 e (rounded to float32), then the hardware base-2 approximation (PTX ex2.approx.f32,
// which keeps subnormal results).  exp_fos(-inf) = +0.
__device__ __forceinline__ float exp_fos(float d) {
  const float t = __fmul_rn(d, 1.44269504088896340736f);
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(t));
  return y;
}

// exp(a - b) for a <= b, exactly 1 when a == b (both -inf included), 0 when only a is -inf.
// Used wherever a rescale must be an exact no-op when the maximum does not move.
__device__ __forceinline__ float scale_fos(float a, float b) {
  return (a == b) ? 1.0f : exp_fos(__fsub_rn(a, b));
}

// The same exponential with results below 2^-126 flushed to zero (PTX ex2.approx.ftz.f32): one
// instruction instead of the subnormal-keeping sequence.  For arguments whose result is at least
// 2^-126 it returns the same bits as exp_fos.  Used only where a flushed value provably cannot
// change a result: when no key of a tile lies more than 87 below the tile maximum
// (87 * log2 e < 126), and for the merge's rescale factors, whose subnormal values are always
// added to a term of at least 1 (the tile or sink holding the running maximum contributes
// exp(0) = 1), far below half an ulp of it.
constexpr float kLog2e = 1.44269504088896340736f;  // log2 e rounded to float32

// The base-2 step of exp_ftz alone, for an argument already multiplied by log2 e.
__device__ __forceinline__ float ex2_ftz(float t) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
  return y;
}

__device__ __forceinline__ float exp_ftz(float d) { return ex2_ftz(__fmul_rn(d, kLog2e)); }

__device__ __forceinline__ float scale_ftz(float a, float b) {
  return (a == b) ? 1.0f : exp_ftz(__fsub_rn(a, b));
}

// Maximum over the 32 lanes.  A maximum is exact, so any combining order gives the same
// value; the single-instruction warp reduction (PTX redux.sync .max.f32, sm_100a family) is
// used.  NaN inputs are outside the contract.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum / minimum of a lane's 8 values (exact, so the grouping does not matter; three-input
// min/max instructions of the sm_100 family).
__device__ __forceinline__ float max8(const float (&x)[8]) {
  return max3f(max3f(x[0], x[1], x[2]), max3f(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
}

__device__ __forceinline__ float min8(const float (&x)[8]) {
  return min3f(min3f(x[0], x[1], x[2]), min3f(x[3], x[4], x[5]), fminf(x[6], x[7]));
}

// Sum over the 32 lanes by the xor butterfly 16, 8, 4, 2, 1.  IEEE addition is commutative,
// so every lane ends with the same bits.
__device__ __forceinline__ float warp_sum_xor(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// The same butterfly on two independent values, interleaved (each gets the bits above).
__device__ __forceinline__ void warp_sum_xor2(float &a, float &b) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float ya = __shfl_xor_sync(kFull, a, o);
    const float yb = __shfl_xor_sync(kFull, b, o);
    a = __fadd_rn(a, ya);
    b = __fadd_rn(b, yb);
  }
}

// ------------------------------------------------------------------ dtype traits

// Io<T>: raw storage of 8 keys (Raw), exact widening to float, and the single rounding of a
// float result back to T (round to nearest even).
template <typename T>
struct Io;

template <>
struct Io<float> {
  static constexpr int kEsz = 4;
  struct Raw { float4 a, b; };
  __device__ __forceinline__ static Raw lds(const unsigned char *p) {
    Raw r;
    r.a = *reinterpret_cast<const float4 *>(p);
    r.b = *reinterpret_cast<const float4 *>(p + 16);
    return r;
  }
  __device__ __forceinline__ static void widen(const Raw &r, float (&x)[8]) {
    x[0] = r.a.x; x[1] = r.a.y; x[2] = r.a.z; x[3] = r.a.w;
    x[4] = r.b.x; x[5] = r.b.y; x[6] = r.b.z; x[7] = r.b.w;
  }
  __device__ __forceinline__ static void st8(void *g, const float (&v)[8]) {
    float4 *q = reinterpret_cast<float4 *>(g);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  __device__ __forceinline__ static void st1(void *g, float v) { *reinterpret_cast<float *>(g) = v; }
};

template <>
struct Io<__nv_bfloat16> {
  static constexpr int kEsz = 2;
  using Raw = uint4;
  __device__ __forceinline__ static Raw lds(const unsigned char *p) {
    return *reinterpret_cast<const uint4 *>(p);
  }
  // bf16 -> f32 widening is exact: the 16 bits become the high half of the float.
  __device__ __forceinline__ static void widen(const Raw &r, float (&x)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  __device__ __forceinline__ static void st8(void *g, const float (&v)[8]) {
    *reinterpret_cast<uint4 *>(g) =
        make_uint4(pack(v[0], v[1]), pack(v[2], v[3]), pack(v[4], v[5]), pack(v[6], v[7]));
  }
  __device__ __forceinline__ static void st1(void *g, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(g) = __float2bfloat16_rn(v);
  }
};

template <>
struct Io<__half> {
  static constexpr int kEsz = 2;
  using Raw = uint4;
  __device__ __forceinline__ static Raw lds(const unsigned char *p) {
    return *reinterpret_cast<const uint4 *>(p);
  }
  __device__ __forceinline__ static void widen(const Raw &r, float (&x)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
      float2 f = __half22float2(h);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  __device__ __forceinline__ static void st8(void *g, const float (&v)[8]) {
    *reinterpret_cast<uint4 *>(g) =
        make_uint4(pack(v[0], v[1]), pack(v[2], v[3]), pack(v[4], v[5]), pack(v[6], v[7]));
  }
  __device__ __forceinline__ static void st1(void *g, float v) {
    *reinterpret_cast<__half *>(g) = __float2half_rn(v);
  }
};

// Store the 8 results of one lane (keys j0..j0+7) to a row of the output.  `vec` says the row
// start is 16-byte aligned; keys at or beyond L are not written.
template <typename T>
__device__ __forceinline__ void store_lane8(unsigned char *row, int j0, int L, bool vec,
                                            const float (&v)[8]) {
  constexpr int esz = Io<T>::kEsz;
  if (vec && j0 + kLaneKeys <= L) {
    Io<T>::st8(row + (size_t)j0 * esz, v);
  } else {
#pragma unroll
    for (int q = 0; q < kLaneKeys; ++q)
      if (j0 + q < L) Io<T>::st1(row + (size_t)(j0 + q) * esz, v[q]);
  }
}

// ------------------------------------------------------------------ row geometry and masks

// Rows are ordered [batch][heads][q_len]; local row r of a launch is problem row
// a.row_base + r.  Returns {lim, b, h, 0}: lim is the number of leading keys of the row that
// can be valid (causal bound and valid length; key_mask and -inf
// are applied per key), b and h its batch entry and head.  Only computed when a mask or a
// sink needs it (one thread per row calls this, when it issues the row's copy).
__device__ __forceinline__ int4 row_geometry(const RowArgs &a, int64_t r) {
  int4 g = make_int4(a.L, 0, 0, 0);
  if (!a.need_geo) return g;
  r += a.row_base;
  int64_t b, h, i;
  if (a.geo32) {  // 32-bit arithmetic suffices; the divisions are multiply-highs
    const uint32_t rr = (uint32_t)r, q = fast_div(rr, a.qdiv);
    i = rr - q * (uint32_t)a.q_len;
    b = fast_div(q, a.hdiv);
    h = q - (uint32_t)b * (uint32_t)a.heads;
  } else {
    const int64_t q = r / a.q_len;
    i = r - q * a.q_len;
    b = q / a.heads;
    h = q - b * a.heads;
  }
  int lim = a.L;
  if (a.causal) lim = min(lim, (int)(a.L - a.q_len + i + 1));
  if (a.kv_valid_len) lim = min(lim, max(0, min(a.kv_valid_len[b], a.L)));
  g.x = lim;
  g.y = (int)b;
  g.z = (int)h;
  return g;
}

// ------------------------------------------------------------------ mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses (and those of threads it synchronised
// with) before its later asynchronous-proxy accesses, e.g. a bulk copy into a buffer the warp
// has just read.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` transactions on `bar`.  Both addresses
// must be 16-byte aligned and bytes a multiple of 16 (checked by the host launchers).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar`, giving up after timeout_ns of the global timer or, should
// the timer not advance, after a fixed number of polls.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  const uint64_t max_polls = (timeout_ns >> 4) + 1000000ull;
  for (uint64_t n = 0; n < max_polls; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > timeout_ns) return false;
  }
  return false;
}

// Plain arrive (count 1) on an mbarrier, e.g. a consumer warp releasing a stage.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named CTA barrier 1 over the first `nthreads` threads (the compute warps), and the same
// barrier combined with an OR of a per-thread flag.
__device__ __forceinline__ void compute_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

__device__ __forceinline__ bool compute_sync_or(int nthreads, bool flag) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)flag), "r"(nthreads)
      : "memory");
  return out != 0;
}

// The same two barriers with a barrier id of the caller's (1..15): one per group of warps
// when a CTA holds several independent groups.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ bool named_sync_or(int id, int nthreads, bool flag) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)flag), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void raise_device_error(unsigned *err, unsigned code) {
  *reinterpret_cast<volatile unsigned *>(err) = code;
}

// Debug build (compiled with FOS_DEBUG): an index the caller is about to use lies outside its
// array when `in_range` is false; that is recorded in the device error word and the caller skips
// the access.  In the normal build this is `true` and compiles away.
__device__ __forceinline__ bool dbg_ok(unsigned *err, bool in_range) {
#ifdef FOS_DEBUG
  if (!in_range) raise_device_error(err, kDevErrIndex);
  return in_range;
#else
  (void)err;
  (void)in_range;
  return true;
#endif
}

// ------------------------------------------------------------------ tensor memory (tcgen05)
//
// The forward parks e_j in tensor memory between its two passes instead of holding them in
// registers, which is what bounds its CTAs per SM otherwise.  An SM has 512 columns of 128
// lanes x 32 bits; a CTA allocates a power of two of at least 32 columns for its lifetime, and
// warp w may touch only lanes 32 * (w % 4) .. 32 * (w % 4) + 31.  Values go through unchanged
// (32-bit moves), so parking changes no result bit.  Address: lane in bits 31..16, column in
// bits 15..0.

// One warp: allocate `ncols` columns, their base address written to shared memory at `slot`,
// and give up the right to allocate again (this CTA allocates once).
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// One warp (the allocating one): free the columns.  Every tensor-memory access of the CTA must
// be complete and ordered before it (tmem_fence_before, a barrier, tmem_fence_after).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-wide: each lane writes its 8 values to 8 consecutive columns of its own lane.
__device__ __forceinline__ void tmem_st8(uint32_t ta, const float (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(ta),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
      : "memory");
}

// Wait until this thread's earlier tmem_st8 have completed (before reading them back).
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Warp-wide: each lane reads 8 (or 16) consecutive columns of its own lane.  The load and its
// wait are one statement, so the registers are never used before the data has arrived.
__device__ __forceinline__ void tmem_ld8(uint32_t ta, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(ta)
      : "memory");
#pragma unroll
  for (int q = 0; q < 8; ++q) v[q] = __uint_as_float(r[q]);
}

__device__ __forceinline__ void tmem_ld16(uint32_t ta, float (&v)[8], float (&u)[8]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(ta)
      : "memory");
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    v[q] = __uint_as_float(r[q]);
    u[q] = __uint_as_float(r[8 + q]);
  }
}

}  // namespace fos
