// fos_pv.cu -- the fixed-order PV contraction behind the softmax, on the sm_103a tensor cores
// (tcgen05): out = P V per (batch, query head), grouped-query heads allowed.
//
// "Batch-invariant attention (standard softmax--cuda version)", Fixed Reduction Contract: each
// output element is the probability-weighted sum of one value column over the keys, with one
// writer per output and the keys accumulated in a fixed order.  "[WS1][kernels] Add
// fixed-order joint-attention softmax for Qwen-Image", Summary: the softmax's P feeds this
// contraction.
//
// Order.  One CTA computes one 128 x D block of outputs (D = 64 or 128), its accumulator in
// tensor memory.  The keys are taken in steps of 16 (one tcgen05.mma of shape 128 x D x 16 each),
// in ascending order from key 0, the first step writing and every later one accumulating in
// float32; keys past the end read as zero (the last block's padding adds exact zeros).  The
// steps, their operands and their order depend only on the query row, the value columns and the
// key count, never on the batch, the head, the block's position or the grid.  The float32 sum is
// rounded once to the output dtype when that is not float32.
//
// Data movement.  P blocks (128 rows x 64 keys, K-major) and V blocks (64 keys x 64 value
// columns, the value columns contiguous: an MN-major operand) arrive by TMA tensor copies with
// the 128-byte swizzle through a ring of stages.  Lane 0 of warp 0 issues the copies, lane 0 of
// warp 1 the MMAs; each stage's MMAs are committed to that stage's "empty" mbarrier, which lets
// the copies of a later block into it, and the last commit releases the epilogue.  Every wait is
// bounded.  The epilogue is fos_qk.cu's: lanes of the accumulator to registers, the scale (1
// for P V, the score scale for dQ = scale * dScores K), one rounding, 128-byte-swizzled
// staging, TMA tensor stores.
#include "fos_device.cuh"
#include "fos_internal.h"
#include "fos_tc.cuh"

namespace fos {
namespace {

constexpr int kPvBM = 128;     // query rows per CTA (MMA M)
constexpr int kPvKB = 64;      // keys per block (128 bytes of bf16 along K in the P tile)
constexpr int kPvUK = 16;      // keys per MMA
constexpr int kPvThreads = 128;
constexpr int kPvStages = 6;
constexpr int kPvABytes = kPvBM * kPvKB * 2;  // 16 KB
constexpr int kPvBHalf = kPvKB * 64 * 2;      // 8 KB: 64 keys x 64 value columns
constexpr int kPvStage = 32 * 128;            // epilogue staging block: 32 rows x 128 bytes

struct PvArgs {
  int32_t dblocks;         // head dimension / 64 (1 or 2)
  int32_t q_heads, group;  // query heads; query heads per key/value head
  int32_t kblocks;         // ceil(kv_len / 64)
  float scale;             // multiplies the float32 sum (1 for P V: an exact no-op)
  uint64_t timeout_ns;
  unsigned *err;
};

template <typename OutT>
__global__ void __launch_bounds__(kPvThreads, 1)
    fos_pv_kernel(const __grid_constant__ CUtensorMap pmap,
                  const __grid_constant__ CUtensorMap vmap,
                  const __grid_constant__ CUtensorMap omap, const PvArgs a, uint32_t idesc) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int stage_bytes = kPvABytes + a.dblocks * kPvBHalf;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPvStages * stage_bytes);
  uint64_t *full = bars, *empty = bars + kPvStages, *done = bars + 2 * kPvStages;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kPvBM, zq = blockIdx.y;
  const int zv = (zq / a.q_heads) * (a.q_heads / a.group) + (zq % a.q_heads) / a.group;
  const uint32_t ncols = a.dblocks == 2 ? 128u : 64u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPvStages; ++s) {
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
    // ---- copies: block kb of the keys into stage kb % stages once the MMAs of block
    // kb - stages (the stage's previous contents) have completed
    int64_t issued = 0;
    for (int kb = 0; kb < a.kblocks; ++kb) {
      const int s = kb % kPvStages;
      if (kb >= kPvStages &&
          !mbar_wait_bounded(smem_addr(&empty[s]), (uint32_t)((kb / kPvStages) & 1) ^ 1u,
                             a.timeout_ns)) {
        raise_device_error(a.err, kDevErrTimeout);
        break;
      }
      unsigned char *st = smem + s * stage_bytes;
      const uint32_t fb = smem_addr(&full[s]);
      mbar_arrive_expect_tx(fb, (uint32_t)stage_bytes);
      tma_load3(smem_addr(st), &pmap, kb * kPvKB, m0, zq, fb);
      for (int h = 0; h < a.dblocks; ++h)
        tma_load3(smem_addr(st + kPvABytes + h * kPvBHalf), &vmap, h * 64, kb * kPvKB, zv, fb);
      ++issued;
    }
    // every copy issued lands before the CTA can exit (they complete on their own; the wait is
    // bounded in case the MMA side stopped)
    for (int64_t kb = issued > kPvStages ? issued - kPvStages : 0; kb < issued; ++kb)
      mbar_wait_bounded(smem_addr(&full[kb % kPvStages]), (uint32_t)((kb / kPvStages) & 1),
                        a.timeout_ns);
  } else if (warp == 1 && lane == 0) {
    // ---- MMAs: the keys in steps of 16, ascending; the first step overwrites
    bool ok = true;
    for (int kb = 0; kb < a.kblocks; ++kb) {
      const int s = kb % kPvStages;
      if (!mbar_wait_bounded(smem_addr(&full[s]), (uint32_t)((kb / kPvStages) & 1),
                             a.timeout_ns)) {
        raise_device_error(a.err, kDevErrTimeout);
        ok = false;
        break;
      }
      tmem_fence_after();
      unsigned char *st = smem + s * stage_bytes;
      for (int k = 0; k < kPvKB / kPvUK; ++k) {
        const uint64_t ad = sw128_desc(smem_addr(st + k * kPvUK * 2));
        const uint64_t bd = sw128_mn_desc(smem_addr(st + kPvABytes + k * kPvUK * 128), kPvBHalf);
        mma_f16(tacc, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
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
    // ---- epilogue: rows m0 + 32 * warp + lane, blocks of 128 bytes of output per row; the
    // stages are free (every MMA has completed), so they hold the staging
    constexpr int kCols = 128 / (int)sizeof(OutT);  // 32 float or 64 bf16 / fp16 columns
    unsigned char *stage0 = smem + warp * 2 * kPvStage;
    const uint32_t trow = tacc + ((uint32_t)(warp * 32) << 16);
    const int nblk = (int)ncols / kCols;
    for (int c = 0; c < nblk; ++c) {
      unsigned char *st = stage0 + (c & 1) * kPvStage;
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
        tma_store3(&omap, c * kCols, m0 + warp * 32, zq, smem_addr(st));
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

const void *pv_fn_for(fos_dtype out) {
  switch (out) {
    case FOS_F32: return reinterpret_cast<const void *>(&fos_pv_kernel<float>);
    case FOS_BF16: return reinterpret_cast<const void *>(&fos_pv_kernel<__nv_bfloat16>);
    case FOS_F16: return reinterpret_cast<const void *>(&fos_pv_kernel<__half>);
  }
  return nullptr;
}

}  // namespace

size_t pv_smem_bytes(int head_dim) {
  // alignment slack, the stages, 2 * stages + 1 barriers and the tensor-memory address; the
  // epilogue's staging (32 KB) reuses the stages
  return 1024 + (size_t)kPvStages * (kPvABytes + (head_dim / 64) * kPvBHalf) +
         (2 * kPvStages + 1) * 8 + 16;
}

fos_status run_pv(const fos_pv_desc *d, fos_dtype in_dt, fos_dtype out_dt, const void *p,
                  const void *v, void *out, cudaStream_t stream, unsigned *err, int max_smem) {
  const size_t smem = pv_smem_bytes(d->head_dim);
  if (smem > (size_t)max_smem) return FOS_ERR_UNSUPPORTED;
  static std::mutex mu;
  static bool prepared[3] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!prepared[out_dt]) {
      if (cudaFuncSetAttribute(pv_fn_for(out_dt), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               max_smem) != cudaSuccess)
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
  alignas(64) CUtensorMap pm, vm, om;
  if (!make_map3(&pm, in_ty, p, (uint64_t)d->kv_len, (uint64_t)d->q_len,
                 (uint64_t)d->batch * d->q_heads, (uint64_t)d->ld_probs * 2,
                 (uint64_t)d->q_len * d->ld_probs * 2, kPvKB, kPvBM) ||
      !make_map3(&vm, in_ty, v, D, (uint64_t)d->kv_len, (uint64_t)d->batch * d->kv_heads, D * 2,
                 (uint64_t)d->kv_len * D * 2, 64, kPvKB) ||
      !make_map3(&om, out_ty, out, D, (uint64_t)d->q_len, (uint64_t)d->batch * d->q_heads,
                 D * osz, (uint64_t)d->q_len * D * osz, (uint32_t)(128 / osz), 32))
    return FOS_ERR_UNSUPPORTED;
  PvArgs a{};
  a.dblocks = d->head_dim / 64;
  a.q_heads = d->q_heads;
  a.group = d->q_heads / d->kv_heads;
  a.kblocks = (d->kv_len + kPvKB - 1) / kPvKB;
  a.scale = d->scale;
  a.timeout_ns = 2000000000ull;
  a.err = err;
  const uint32_t idesc = f16_idesc(in_dt == FOS_BF16, kPvBM, d->head_dim, true);
  const dim3 grid((unsigned)((d->q_len + kPvBM - 1) / kPvBM), (unsigned)(d->batch * d->q_heads));
  void *args[] = {&pm, &vm, &om, &a, const_cast<uint32_t *>(&idesc)};
  if (cudaLaunchKernel(pv_fn_for(out_dt), grid, dim3(kPvThreads), args, smem, stream) !=
      cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

}  // namespace fos
