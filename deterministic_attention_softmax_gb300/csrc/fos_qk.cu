// fos_qk.cu -- the fixed-order QK contraction in front of the softmax, on the sm_103a tensor
// cores (tcgen05): scores = scale * Q K^T per (batch, query head), grouped-query heads allowed.
//
// "Batch-invariant attention (standard softmax--cuda version)", Fixed Reduction Contract: each
// score is the dot product of one query row and one key row over the head dimension, with one
// writer per score and the head dimension accumulated in a fixed order.  "[WS1][kernels] Add
// fixed-order joint-attention softmax for Qwen-Image", Summary: this contraction feeds the
// softmax its materialised score matrix.
//
// Order.  One CTA computes one 128 x BN tile of scores (BN = 128 or 256 keys).  Its accumulator
// lives in tensor memory; the head dimension is taken in steps of 16 (one tcgen05.mma of shape
// 128 x BN x 16 each), in ascending order, the first step writing and every later one accumulating in
// float32.  The steps, their operands and their order depend only on the two rows a score
// joins, never on the batch, the head, the tile's position or the grid, so a score has the
// same bits wherever its rows sit.  The float32 sum is then multiplied by `scale` (one
// rounding) and rounded once more to the output dtype when that is not float32.
//
// Data movement.  Q and K tiles arrive by TMA tensor copies (3-D maps [rows of a head, head
// dimension] x heads, 128-byte swizzle, out-of-range rows read as zero) into shared memory
// laid out as the tensor core's K-major swizzled operands; one thread issues the copies and
// the eight (D = 128) or four (D = 64) MMAs and commits them to an mbarrier.  The epilogue's
// four warps read their 32 lanes of the accumulator (rows 32w .. 32w + 31) in blocks of 32
// columns, scale and round them, write each block to a 128-byte-swizzled staging buffer and
// store it with a TMA tensor store, which clips rows and columns past the end of the head.
// The staging reuses the operand buffers (free once the MMAs have completed).
#include <cuda.h>

#include <mutex>

#include "fos_device.cuh"
#include "fos_internal.h"
#include "fos_tc.cuh"

namespace fos {
namespace {

constexpr int kBM = 128;   // query rows per tile (MMA M, TMEM lanes)
constexpr int kKB = 64;    // head-dimension elements per 128-byte swizzle block
constexpr int kUK = 16;    // head-dimension elements per MMA
constexpr int kQkThreads = 128;
// A CTA per tile (tile_n 128 or 256 keys): 128 lets three CTAs share an SM (about 65 KB of
// shared memory and 128 tensor-memory columns each), 256 two.  The default is the persistent
// form below.

// Shared-memory layout (dynamic; 1024-byte aligned operand blocks), BN keys per tile (128 or
// 256, the MMA's N and the accumulator's columns):
//   [A: D / 64 blocks of 128 x 64 16-bit (16 KB)] [B: D / 64 blocks of BN x 64 16-bit]
//   [barriers and the tensor-memory address]
// After the MMAs, the operand region holds the epilogue's staging: 4 warps x 2 buffers x 4 KB.
constexpr int kABlock = kBM * kKB * 2;
constexpr int kStage = 32 * 128;  // 32 rows x 128 bytes

struct QkArgs {
  int32_t dblocks;    // head dimension / 64 (1 or 2)
  int32_t q_heads, group;  // query heads; query heads per key head
  float scale;
  uint64_t timeout_ns;
  unsigned *err;
};

// One 128 x BN tile of scores: blockIdx.x = key tile, blockIdx.y = query tile, blockIdx.z =
// batch * q_heads + query head.  OutT is the output dtype (float, bf16 or fp16).
template <typename OutT, int kBN>
__global__ void __launch_bounds__(kQkThreads, 1)
    fos_qk_kernel(const __grid_constant__ CUtensorMap qmap,
                  const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap smap, const QkArgs a, uint32_t idesc) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  constexpr int kBBlock = kBN * kKB * 2;
  // the staging buffers (4 warps x 2 x 4 KB) reuse the operand region, even at D = 64
  static_assert(kABlock + kBBlock >= 4 * 2 * kStage, "staging must fit the operand region");
  // the operand blocks must start on 1024-byte boundaries (swizzle atoms)
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *sa = smem;
  unsigned char *sb = smem + a.dblocks * kABlock;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sb + a.dblocks * kBBlock);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2);
  const uint32_t load_bar = smem_addr(&bars[0]), mma_bar = smem_addr(&bars[1]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM, zq = blockIdx.z;
  const int zk = (zq / a.q_heads) * (a.q_heads / a.group) + (zq % a.q_heads) / a.group;

  if (threadIdx.x == 0) {
    mbar_init(load_bar, 1);
    mbar_init(mma_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), (uint32_t)kBN);
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tacc = *tmem_slot;

  bool ok = true;
  if (threadIdx.x == 0) {
    // operands: the tile's Q rows and K rows, head dimension in 64-element blocks
    mbar_arrive_expect_tx(load_bar, (uint32_t)a.dblocks * (kABlock + kBBlock));
    for (int kb = 0; kb < a.dblocks; ++kb) {
      tma_load3(smem_addr(sa + kb * kABlock), &qmap, kb * kKB, m0, zq, load_bar);
      tma_load3(smem_addr(sb + kb * kBBlock), &kmap, kb * kKB, n0, zk, load_bar);
    }
    ok = mbar_wait_bounded(load_bar, 0, a.timeout_ns);
    if (ok) {
      tmem_fence_after();
      // the head dimension in steps of 16, ascending; the first step overwrites
      for (int kb = 0; kb < a.dblocks; ++kb)
        for (int k = 0; k < kKB / kUK; ++k) {
          const uint64_t ad = sw128_desc(smem_addr(sa + kb * kABlock + k * kUK * 2));
          const uint64_t bd = sw128_desc(smem_addr(sb + kb * kBBlock + k * kUK * 2));
          mma_f16(tacc, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
        }
      mma_commit(mma_bar);
    } else {
      raise_device_error(a.err, kDevErrTimeout);
    }
  }
  __syncwarp();
  // every thread waits for the accumulator (bounded); a stop anywhere skips the epilogue
  const bool done = __all_sync(kFull, mbar_wait_bounded(mma_bar, 0, a.timeout_ns));
  tmem_fence_after();
  if (!done) {
    if (lane == 0) raise_device_error(a.err, kDevErrTimeout);
  } else {
    // ---- epilogue: rows m0 + 32 * warp + lane, blocks of 128 bytes of output per row
    constexpr int kCols = 128 / (int)sizeof(OutT);  // 32 float or 64 bf16 / fp16 columns
    unsigned char *stage0 = smem + warp * 2 * kStage;
    const uint32_t trow = tacc + ((uint32_t)(warp * 32) << 16);
    for (int c = 0; c < kBN / kCols; ++c) {
      unsigned char *st = stage0 + (c & 1) * kStage;
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
          for (int q = 0; q < 32; q += 2) {
            const uint32_t lo = Io<OutT>::pack(v[q], v[q + 1]);
            packed[h * 16 + q / 2] = lo;
          }
        }
      }
      // row `lane` of the staging block: 16-byte chunk j at position j ^ (lane % 8)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 *dst = reinterpret_cast<uint4 *>(st + lane * 128 + ((j ^ (lane & 7)) << 4));
        *dst = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
      }
      fence_proxy_async_smem();  // the generic writes come before the tensor store reads them
      __syncwarp();
      if (lane == 0) {
        tma_store3(&smap, n0 + c * kCols, m0 + warp * 32, zq, smem_addr(st));
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_read(0);  // shared memory stays until the stores have read it
  }
  tmem_fence_before();
  __syncthreads();
  if (warp == 0) {
    tmem_fence_after();
    tmem_dealloc(tacc, (uint32_t)kBN);
  }
}

// ---- persistent form: one CTA per SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ... of
// 128 x 128 scores (key tile fastest), so that the CTAs of the grid write one compact band of
// the output at a time.  Warp 0 issues the copies into a ring of `stages` operand stages (a
// tile's Q and K blocks are reloaded, mostly from L2; three stages at D = 128), warp 1 the MMAs
// into kPqAcc accumulators of 128 tensor-memory columns, and warps 2..5 drain an accumulator
// (one warp per lane quarter, all 128 columns) while the MMAs of the next tiles proceed into
// the other accumulators.  Measured on the Qwen-Image shape against two stages, two
// accumulators and eight epilogue warps (two per lane quarter): float32 scores 53.3 -> 51.7 us,
// bf16 38.9 -> 37.3 us.  Each tile's scores are the same instructions on the same operands as
// in fos_qk_kernel, so the bits are the same.
constexpr int kPqBN = 128;
constexpr int kPqEpiWarps = 4;
constexpr int kPqEpiCols = kPqBN * 4 / kPqEpiWarps;  // columns per epilogue warp
constexpr int kPqAcc = 4;
constexpr int kPqThreads = (2 + kPqEpiWarps) * 32;
constexpr int kPqMaxStages = 4;
static_assert(kPqEpiWarps == 4 || kPqEpiWarps == 8, "one or two warps per lane quarter");

struct QkTiles {
  int32_t nx, ny;  // key tiles, query tiles per (batch, head)
  int64_t ntiles;  // nx * ny * batch * q_heads
  int32_t stages;  // operand stages (2 .. kPqMaxStages)
};

template <typename OutT>
__global__ void __launch_bounds__(kPqThreads, 1)
    fos_qk_persistent_kernel(const __grid_constant__ CUtensorMap qmap,
                             const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap smap, const QkArgs a,
                             const QkTiles tl, uint32_t idesc) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  constexpr int kBBlock = kPqBN * kKB * 2;  // 16 KB
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int NS = tl.stages;
  const int stage_bytes = a.dblocks * (kABlock + kBBlock);
  unsigned char *staging = smem + NS * stage_bytes;  // epilogue warps x 2 x 4 KB
  uint64_t *bars = reinterpret_cast<uint64_t *>(staging + kPqEpiWarps * 2 * kStage);
  uint64_t *full = bars, *empty = bars + kPqMaxStages, *accf = bars + 2 * kPqMaxStages,
           *acce = accf + kPqAcc;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acce + kPqAcc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), 1);
    }
    for (int i = 0; i < kPqAcc; ++i) {
      mbar_init(smem_addr(&accf[i]), 1);
      mbar_init(smem_addr(&acce[i]), kPqEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(tmem_slot), kPqAcc * kPqBN);
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tacc = *tmem_slot;
  const int64_t per_z = (int64_t)tl.nx * tl.ny;

  if (warp == 0) {
    if (lane == 0) {  // ---- copies
      int64_t i = 0;
      for (int64_t t = blockIdx.x; t < tl.ntiles; t += gridDim.x, ++i) {
        const int s = (int)(i % NS);
        if (i >= NS && !mbar_wait_bounded(smem_addr(&empty[s]), (uint32_t)((i / NS) & 1) ^ 1u,
                                          a.timeout_ns)) {
          raise_device_error(a.err, kDevErrTimeout);
          break;
        }
        const int zq = (int)(t / per_z);
        const int rem = (int)(t - (int64_t)zq * per_z);
        const int y = rem / tl.nx, x = rem - y * tl.nx;
        const int zk = (zq / a.q_heads) * (a.q_heads / a.group) + (zq % a.q_heads) / a.group;
        unsigned char *sa = smem + s * stage_bytes;
        unsigned char *sb = sa + a.dblocks * kABlock;
        const uint32_t fb = smem_addr(&full[s]);
        mbar_arrive_expect_tx(fb, (uint32_t)stage_bytes);
        for (int kb = 0; kb < a.dblocks; ++kb) {
          tma_load3(smem_addr(sa + kb * kABlock), &qmap, kb * kKB, y * kBM, zq, fb);
          tma_load3(smem_addr(sb + kb * kBBlock), &kmap, kb * kKB, x * kPqBN, zk, fb);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMAs: tile i into accumulator i % kPqAcc, head dimension ascending
      int64_t i = 0;
      for (int64_t t = blockIdx.x; t < tl.ntiles; t += gridDim.x, ++i) {
        const int s = (int)(i % NS), b = (int)(i % kPqAcc);
        if (!mbar_wait_bounded(smem_addr(&full[s]), (uint32_t)((i / NS) & 1), a.timeout_ns) ||
            (i >= kPqAcc &&
             !mbar_wait_bounded(smem_addr(&acce[b]), (uint32_t)((i / kPqAcc) & 1) ^ 1u,
                                a.timeout_ns))) {
          raise_device_error(a.err, kDevErrTimeout);
          break;
        }
        tmem_fence_after();
        unsigned char *sa = smem + s * stage_bytes;
        unsigned char *sb = sa + a.dblocks * kABlock;
        const uint32_t dacc = tacc + (uint32_t)(b * kPqBN);
        for (int kb = 0; kb < a.dblocks; ++kb)
          for (int k = 0; k < kKB / kUK; ++k) {
            const uint64_t ad = sw128_desc(smem_addr(sa + kb * kABlock + k * kUK * 2));
            const uint64_t bd = sw128_desc(smem_addr(sb + kb * kBBlock + k * kUK * 2));
            mma_f16(dacc, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
        mma_commit(smem_addr(&empty[s]));  // the stage may be refilled
        mma_commit(smem_addr(&accf[b]));   // the accumulator may be drained
      }
    }
  } else {
    // ---- epilogue: warp w drains lane quarter w % 4, kPqEpiCols columns from
    // kPqEpiCols * ((w - 2) / 4)
    constexpr int kCols = 128 / (int)sizeof(OutT);  // 32 float or 64 bf16 / fp16 columns
    const int ew = warp - 2, quarter = warp & 3, c0 = (ew >> 2) * kPqEpiCols;
    unsigned char *stage0 = staging + ew * 2 * kStage;
    int nst = 0;  // stores issued by this warp
    int64_t i = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < tl.ntiles && ok; t += gridDim.x, ++i) {
      const int b = (int)(i % kPqAcc);
      ok = __all_sync(kFull, mbar_wait_bounded(smem_addr(&accf[b]), (uint32_t)((i / kPqAcc) & 1),
                                               a.timeout_ns));
      if (!ok) {
        if (lane == 0) raise_device_error(a.err, kDevErrTimeout);
        break;
      }
      tmem_fence_after();
      const int zq = (int)(t / per_z);
      const int rem = (int)(t - (int64_t)zq * per_z);
      const int y = rem / tl.nx, x = rem - y * tl.nx;
      const uint32_t trow =
          tacc + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * kPqBN + c0);
      for (int c = 0; c < kPqEpiCols / kCols; ++c, ++nst) {
        unsigned char *st = stage0 + (nst & 1) * kStage;
        if (lane == 0 && nst >= 2) bulk_wait_read(1);
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
            for (int q = 0; q < 32; q += 2)
              packed[h * 16 + q / 2] = Io<OutT>::pack(v[q], v[q + 1]);
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4 *dst = reinterpret_cast<uint4 *>(st + lane * 128 + ((j ^ (lane & 7)) << 4));
          *dst = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2],
                            packed[4 * j + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store3(&smap, x * kPqBN + c0 + c * kCols, y * kBM + quarter * 32, zq,
                     smem_addr(st));
          bulk_commit();
        }
      }
      // this warp is done reading the accumulator: the MMAs of tile i + kPqAcc may overwrite it
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&acce[b]));
    }
    if (lane == 0) bulk_wait_read(0);  // shared memory stays until the stores have read it
  }
  tmem_fence_before();
  __syncthreads();
  if (warp == 0) {
    tmem_fence_after();
    tmem_dealloc(tacc, kPqAcc * kPqBN);
  }
}

template <typename OutT>
const void *qk_fn(int bn) {
  return bn == 128 ? reinterpret_cast<const void *>(&fos_qk_kernel<OutT, 128>)
                   : reinterpret_cast<const void *>(&fos_qk_kernel<OutT, 256>);
}

const void *qk_fn_for(fos_dtype out, int bn) {
  switch (out) {
    case FOS_F32: return qk_fn<float>(bn);
    case FOS_BF16: return qk_fn<__nv_bfloat16>(bn);
    case FOS_F16: return qk_fn<__half>(bn);
  }
  return nullptr;
}

}  // namespace

size_t qk_smem_bytes(int head_dim, int bn) {
  const int db = head_dim / kKB;
  // operands (their blocks 1024-byte aligned inside the buffer), barriers, the tensor-memory
  // address; the staging (32 KB) fits in the B region
  return 1024 + (size_t)db * (kABlock + (size_t)bn * kKB * 2) + 64;
}

template <typename OutT>
const void *qk_persistent_fn() {
  return reinterpret_cast<const void *>(&fos_qk_persistent_kernel<OutT>);
}

const void *qk_persistent_fn_for(fos_dtype out) {
  switch (out) {
    case FOS_F32: return qk_persistent_fn<float>();
    case FOS_BF16: return qk_persistent_fn<__nv_bfloat16>();
    case FOS_F16: return qk_persistent_fn<__half>();
  }
  return nullptr;
}

// Shared memory of the persistent form with `stages` operand stages: alignment slack, the
// stages, the epilogue's staging, the barriers and the tensor-memory address.
size_t qk_persistent_smem_bytes(int head_dim, int stages) {
  const int db = head_dim / kKB;
  return 1024 + (size_t)stages * db * (kABlock + kPqBN * kKB * 2) + kPqEpiWarps * 2 * kStage +
         (2 * kPqMaxStages + 2 * kPqAcc) * 8 + 16;
}

// The deepest operand ring (up to kPqMaxStages) that fits `max_smem`; 0 if not even two do.
int qk_persistent_stages(int head_dim, int max_smem) {
  for (int ns = kPqMaxStages; ns >= 2; --ns)
    if (qk_persistent_smem_bytes(head_dim, ns) <= (size_t)max_smem) return ns;
  return 0;
}

fos_status run_qk(const fos_qk_desc *d, fos_dtype in_dt, fos_dtype out_dt, const void *q,
                  const void *k, void *scores, cudaStream_t stream, unsigned *err,
                  int max_smem, int sms) {
  const bool persistent = d->tile_n == 0;
  const int bn = persistent ? kPqBN : d->tile_n;
  const int stages = persistent ? qk_persistent_stages(d->head_dim, max_smem) : 0;
  if (persistent && stages == 0) return FOS_ERR_UNSUPPORTED;
  const size_t smem = persistent ? qk_persistent_smem_bytes(d->head_dim, stages)
                                 : qk_smem_bytes(d->head_dim, bn);
  if (smem > (size_t)max_smem) return FOS_ERR_UNSUPPORTED;
  const void *fn = persistent ? qk_persistent_fn_for(out_dt) : qk_fn_for(out_dt, bn);
  static std::mutex mu;
  static bool prepared[3][3] = {};
  {
    const int kind = persistent ? 2 : (bn == 256);
    std::lock_guard<std::mutex> lock(mu);
    if (!prepared[out_dt][kind]) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
          cudaSuccess)
        return FOS_ERR_CUDA;
      prepared[out_dt][kind] = true;
    }
  }
  const CUtensorMapDataType in_ty =
      in_dt == FOS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType out_ty = out_dt == FOS_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                     : out_dt == FOS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int osz = dtype_size(out_dt);
  const uint64_t D = (uint64_t)d->head_dim;
  alignas(64) CUtensorMap qm, km, sm;
  if (!make_map3(&qm, in_ty, q, D, (uint64_t)d->q_len, (uint64_t)d->batch * d->q_heads, D * 2,
                 (uint64_t)d->q_len * D * 2, kKB, kBM) ||
      !make_map3(&km, in_ty, k, D, (uint64_t)d->kv_len, (uint64_t)d->batch * d->kv_heads, D * 2,
                 (uint64_t)d->kv_len * D * 2, kKB, (uint32_t)bn) ||
      !make_map3(&sm, out_ty, scores, (uint64_t)d->kv_len, (uint64_t)d->q_len,
                 (uint64_t)d->batch * d->q_heads, (uint64_t)d->ld_scores * osz,
                 (uint64_t)d->q_len * d->ld_scores * osz, (uint32_t)(128 / osz), 32))
    return FOS_ERR_UNSUPPORTED;
  QkArgs a{};
  a.dblocks = d->head_dim / kKB;
  a.q_heads = d->q_heads;
  a.group = d->q_heads / d->kv_heads;
  a.scale = d->scale;
  a.timeout_ns = 2000000000ull;
  a.err = err;
  const uint32_t idesc = f16_idesc(in_dt == FOS_BF16, kBM, bn, false);
  if (persistent) {
    QkTiles tl{};
    tl.nx = (d->kv_len + kPqBN - 1) / kPqBN;
    tl.ny = (d->q_len + kBM - 1) / kBM;
    tl.ntiles = (int64_t)tl.nx * tl.ny * d->batch * d->q_heads;
    tl.stages = stages;
    const int grid = (int)(tl.ntiles < sms ? tl.ntiles : sms);
    void *args[] = {&qm, &km, &sm, &a, &tl, const_cast<uint32_t *>(&idesc)};
    if (cudaLaunchKernel(fn, dim3(grid), dim3(kPqThreads), args, smem, stream) != cudaSuccess)
      return FOS_ERR_CUDA;
    return FOS_OK;
  }
  const dim3 grid((unsigned)((d->kv_len + bn - 1) / bn), (unsigned)((d->q_len + kBM - 1) / kBM),
                  (unsigned)(d->batch * d->q_heads));
  void *args[] = {&qm, &km, &sm, &a, const_cast<uint32_t *>(&idesc)};
  if (cudaLaunchKernel(fn, grid, dim3(kQkThreads), args, smem, stream) != cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

}  // namespace fos
