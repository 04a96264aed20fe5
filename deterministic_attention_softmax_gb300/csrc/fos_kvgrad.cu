// fos_kvgrad.cu -- the fixed-order contraction behind the key and value gradients of attention,
// on the sm_103a tensor cores (tcgen05):
//   out[b, g, j, d] = scale * sum over the query heads h of group g (ascending) and the query
//                     positions i (ascending) of a[b, h, i, j] * m[b, h, i, d]
// with (a, m, scale) = (P, dO, 1) for dV and (dScores, Q, the score scale) for dK.
//
// "Batch-invariant attention (standard softmax--cuda version)", GQA backward: each dK and dV
// element has one writer, which accumulates the group's query heads in order and, within a
// head, the query positions in order; no split over keys, no atomics.  "[WS1][kernels] Add
// fixed-order joint-attention softmax for Qwen-Image", Summary: the backward of the chain the
// softmax sits in.
//
// Order.  One CTA computes one block of 128 keys x D outputs (D = 64 or 128) of one key head,
// its accumulator in tensor memory.  It takes the group's query heads in ascending order and,
// within a head, the query positions in steps of 16 (one tcgen05.mma of shape 128 x D x 16
// each), ascending from position 0, the first step writing and every later one accumulating in
// float32; positions past the end read as zero (the last block's padding adds exact zeros).  The
// steps, their operands and their order depend only on the key, the output column and the
// group's rows, never on the batch, the block's position or the grid.  The float32 sum is
// multiplied by `scale` (one rounding) and rounded once more to the output dtype when that is
// not float32.
//
// Data movement.  Both operands have the contracted dimension (query positions) outermost, so
// both are MN-major: the a block (64 positions x 128 keys, two 64-key halves) and the m block (64
// positions x D, 64-column halves) arrive by TMA tensor copies with the 128-byte swizzle through
// a ring of stages, as the V operand of fos_pv.cu does.  Lane 0 of warp 0 issues the copies,
// lane 0 of warp 1 the MMAs; each stage's MMAs are committed to that stage's "empty" mbarrier,
// and the last commit releases the epilogue (fos_pv.cu's, with the scale).  Every wait is
// bounded.
#include "fos_device.cuh"
#include "fos_internal.h"
#include "fos_tc.cuh"

namespace fos {
namespace {

constexpr int kKgBM = 128;                  // keys per CTA (MMA M)
constexpr int kKgQB = 64;                   // query positions per block (the contracted K)
constexpr int kKgUK = 16;                   // positions per MMA
constexpr int kKgThreads = 128;
constexpr int kKgStages = 6;
constexpr int kKgHalf = kKgQB * 64 * 2;     // 8 KB: 64 positions x 64 keys (or columns)
constexpr int kKgABytes = 2 * kKgHalf;      // 16 KB: 64 positions x 128 keys
constexpr int kKgStage = 32 * 128;          // epilogue staging block: 32 rows x 128 bytes

struct KgArgs {
  int32_t dblocks;          // head dimension / 64 (1 or 2)
  int32_t q_heads, group;   // query heads; query heads per key/value head
  int32_t kv_heads;
  int32_t qblocks;          // ceil(q_len / 64)
  float scale;
  uint64_t timeout_ns;
  unsigned *err;
};

template <typename OutT>
__global__ void __launch_bounds__(kKgThreads, 1)
    fos_kvgrad_kernel(const __grid_constant__ CUtensorMap amap,
                      const __grid_constant__ CUtensorMap mmap,
                      const __grid_constant__ CUtensorMap omap, const KgArgs a, uint32_t idesc) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int stage_bytes = kKgABytes + a.dblocks * kKgHalf;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kKgStages * stage_bytes);
  uint64_t *full = bars, *empty = bars + kKgStages, *done = bars + 2 * kKgStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j0 = blockIdx.x * kKgBM, zk = blockIdx.y;  // zk = b * kv_heads + key head
  const int zq0 = (zk / a.kv_heads) * a.q_heads + (zk % a.kv_heads) * a.group;  // first query head
  const uint32_t ncols = a.dblocks == 2 ? 128u : 64u;
  const int nsteps = a.group * a.qblocks;  // (query head, block of 64 positions), in order

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKgStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), 1);
    }
    mbar_init(smem_addr(done), 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), ncols);
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tacc = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- copies: step n (head zq0 + n / qblocks, positions 64 * (n % qblocks) ..) into stage
    // n % stages once the MMAs of step n - stages have completed
    int issued = 0;
    for (int n = 0; n < nsteps; ++n) {
      const int s = n % kKgStages;
      if (n >= kKgStages &&
          !mbar_wait_bounded(smem_addr(&empty[s]), (uint32_t)((n / kKgStages) & 1) ^ 1u,
                             a.timeout_ns)) {
        raise_device_error(a.err, kDevErrTimeout);
        break;
      }
      const int zq = zq0 + n / a.qblocks, i0 = (n % a.qblocks) * kKgQB;
      unsigned char *st = smem + s * stage_bytes;
      const uint32_t fb = smem_addr(&full[s]);
      mbar_arrive_expect_tx(fb, (uint32_t)stage_bytes);
      for (int h = 0; h < 2; ++h)
        tma_load3(smem_addr(st + h * kKgHalf), &amap, j0 + h * 64, i0, zq, fb);
      for (int h = 0; h < a.dblocks; ++h)
        tma_load3(smem_addr(st + kKgABytes + h * kKgHalf), &mmap, h * 64, i0, zq, fb);
      ++issued;
    }
    // every copy issued lands before the CTA can exit (bounded, in case the MMA side stopped)
    for (int n = issued > kKgStages ? issued - kKgStages : 0; n < issued; ++n)
      mbar_wait_bounded(smem_addr(&full[n % kKgStages]), (uint32_t)((n / kKgStages) & 1),
                        a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ---- MMAs: the query heads in order, within a head the positions in steps of 16,
    // ascending; the first step overwrites
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      const int s = n % kKgStages;
      if (!mbar_wait_bounded(smem_addr(&full[s]), (uint32_t)((n / kKgStages) & 1), a.timeout_ns)) {
        raise_device_error(a.err, kDevErrTimeout);
        ok = false;
        break;
      }
      tmem_fence_after();
      unsigned char *st = smem + s * stage_bytes;
      for (int k = 0; k < kKgQB / kKgUK; ++k) {
        const uint64_t ad = sw128_mn_desc(smem_addr(st + k * kKgUK * 128), kKgHalf);
        const uint64_t bd = sw128_mn_desc(smem_addr(st + kKgABytes + k * kKgUK * 128), kKgHalf);
        mma_f16(tacc, ad, bd, idesc, (n | k) != 0 ? 1u : 0u);
      }
      mma_commit(smem_addr(&empty[s]));  // the stage may be refilled once these complete
    }
    if (ok) mma_commit(smem_addr(done));
  }
  __syncwarp();
  // every thread waits for the accumulator (bounded); a stop anywhere skips the epilogue
  const bool fin = __all_sync(kFull, mbar_wait_bounded(smem_addr(done), 0, a.timeout_ns));
  tmem_fence_after();
  if (!fin) {
    if (lane == 0) raise_device_error(a.err, kDevErrTimeout);
  } else {
    // ---- epilogue: keys j0 + 32 * warp + lane, blocks of 128 bytes of output per key; the
    // stages are free (every MMA has completed), so they hold the staging
    constexpr int kCols = 128 / (int)sizeof(OutT);  // 32 float or 64 bf16 / fp16 columns
    unsigned char *stage0 = smem + warp * 2 * kKgStage;
    const uint32_t trow = tacc + ((uint32_t)(warp * 32) << 16);
    const int nblk = (int)ncols / kCols;
    for (int c = 0; c < nblk; ++c) {
      unsigned char *st = stage0 + (c & 1) * kKgStage;
      if (lane == 0 && c >= 2) bulk_wait_read(1);  // the store from this buffer has read it
      __syncwarp();
      uint32_t packed[32];
#pragma unroll
      for (int h = 0; h < kCols / 32; ++h) {
        float v[32];
        tmem_ld32(trow + (uint32_t)(c * kCols + h * 32), v);
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = __fmul_rn(v[q], a.scale);
        if constexpr (sizeof(OutT) == 4) {
#pragma unroll
          for (int q = 0; q < 32; ++q) packed[q] = __float_as_uint(v[q]);
        } else {
#pragma unroll
          for (int q = 0; q < 32; q += 2) packed[h * 16 + q / 2] = Io<OutT>::pack(v[q], v[q + 1]);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 *dst = reinterpret_cast<uint4 *>(st + lane * 128 + ((j ^ (lane & 7)) << 4));
        *dst = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store3(&omap, c * kCols, j0 + warp * 32, zk, smem_addr(st));
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_read(0);
  }
  tmem_fence_before();
  __syncthreads();
  if (warp == 0) {
    tmem_fence_after();
    tmem_dealloc(tacc, ncols);
  }
}

const void *kvgrad_fn_for(fos_dtype out) {
  switch (out) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_kvgrad_kernel<float>);
    case FOS_BF16: return reinterpret_cast<const void *>(&fos_kvgrad_kernel<__nv_bfloat16>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_kvgrad_kernel<__half>);
  }
  return nullptr;
}

}  // namespace

size_t kvgrad_smem_bytes(int head_dim) {
  // alignment slack, the stages, 2 * stages + 1 barriers and the tensor-memory address; the
  // epilogue's staging (32 KB) reuses the stages
  return 1024 + (size_t)kKgStages * (kKgABytes + (head_dim / 64) * kKgHalf) +
         (2 * kKgStages + 1) * 8 + 16;
}

fos_status run_kvgrad(const fos_pv_desc *d, fos_dtype in_dt, fos_dtype out_dt, const void *am,
                      const void *m, void *out, cudaStream_t stream, unsigned *err, int max_smem) {
  const size_t smem = kvgrad_smem_bytes(d->head_dim);
  if (smem > (size_t)max_smem) return FOS_ERR_UNSUPPORTED;
  static std::mutex mu;
  static bool prepared[3] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!prepared[out_dt]) {
      if (cudaFuncSetAttribute(kvgrad_fn_for(out_dt),
                               cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
          cudaSuccess)
        return FOS_ERR_CUDA;
      prepared[out_dt] = true;
    }
  }
  const CUtensorMapDataType in_ty =
      in_dt == FOS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType out_ty = out_dt == FOS_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : out_dt == FOS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int osz = dtype_size(out_dt);
  const uint64_t D = (uint64_t)d->head_dim;
  alignas(64) CUtensorMap amap, mmap, omap;
  // a: [B * Hq][Sq][ld] with the keys innermost; m: [B * Hq][Sq][D]; out: [B * Hkv][Skv][D]
  if (!make_map3(&amap, in_ty, am, (uint64_t)d->kv_len, (uint64_t)d->q_len,
                 (uint64_t)d->batch * d->q_heads, (uint64_t)d->ld_probs * 2,
                 (uint64_t)d->q_len * d->ld_probs * 2, 64, kKgQB) ||
      !make_map3(&mmap, in_ty, m, D, (uint64_t)d->q_len, (uint64_t)d->batch * d->q_heads, D * 2,
                 (uint64_t)d->q_len * D * 2, 64, kKgQB) ||
      !make_map3(&omap, out_ty, out, D, (uint64_t)d->kv_len, (uint64_t)d->batch * d->kv_heads,
                 D * osz, (uint64_t)d->kv_len * D * osz, (uint32_t)(128 / osz), 32))
    return FOS_ERR_UNSUPPORTED;
  KgArgs a{};
  a.dblocks = d->head_dim / 64;
  a.q_heads = d->q_heads;
  a.group = d->q_heads / d->kv_heads;
  a.kv_heads = d->kv_heads;
  a.qblocks = (d->q_len + kKgQB - 1) / kKgQB;
  a.scale = d->scale;
  a.timeout_ns = 2000000000ull;
  a.err = err;
  const uint32_t idesc = f16_idesc(in_dt == FOS_BF16, kKgBM, d->head_dim, true, true);
  const dim3 grid((unsigned)((d->kv_len + kKgBM - 1) / kKgBM), (unsigned)(d->batch * d->kv_heads));
  void *args[] = {&amap, &mmap, &omap, &a, const_cast<uint32_t *>(&idesc)};
  if (cudaLaunchKernel(kvgrad_fn_for(out_dt), grid, dim3(kKgThreads), args, smem, stream) !=
      cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

}  // namespace fos
