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

namespace fos {
namespace {

constexpr int kBM = 128;   // query rows per tile (MMA M, TMEM lanes)
constexpr int kKB = 64;    // head-dimension elements per 128-byte swizzle block
constexpr int kUK = 16;    // head-dimension elements per MMA
constexpr int kQkThreads = 128;
constexpr int kQkDefaultTileN = 128;
// Keys per tile by default: 128 lets three CTAs share an SM (about 65 KB of shared memory and
// 128 tensor-memory columns each), so more CTAs drain their scores while others load and
// multiply; 256 takes two.

// Shared-memory layout (dynamic; 1024-byte aligned operand blocks), BN keys per tile (128 or
// 256, the MMA's N and the accumulator's columns):
//   [A: D / 64 blocks of 128 x 64 16-bit (16 KB)] [B: D / 64 blocks of BN x 64 16-bit]
//   [barriers and the tensor-memory address]
// After the MMAs, the operand region holds the epilogue's staging: 4 warps x 2 buffers x 4 KB.
constexpr int kABlock = kBM * kKB * 2;
constexpr int kStage = 32 * 128;  // 32 rows x 128 bytes

// ---- tcgen05 operand descriptors (PTX ISA, "Matrix Descriptors" of the tcgen05 family)
//
// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle layout: rows of
// 128 bytes (64 bf16 of the head dimension), 8-row swizzle atoms of 1024 bytes, atoms
// 1024 bytes apart (stride byte offset); bits 0-13 start address >> 4, 16-29 leading byte
// offset >> 4 (unused by this layout, set to 1), 32-45 stride byte offset >> 4, 46-48 the
// fixed value 0b001, 49-51 base offset (0: every block starts 1024-byte aligned), 61-63 the
// layout (2 = 128-byte swizzle).  A step of 16 elements along K inside the 128-byte row
// advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: float32 accumulator (bits 4-5 = 1), A and B of the
// same 16-bit type (bits 7-9 and 10-12: 0 = f16, 1 = bf16), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t qk_idesc(bool bf16, int bn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(dtmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every MMA this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap *map, int x, int y,
                                          int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_store3(const CUtensorMap *map, int x, int y, int z,
                                           uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most `n` (0 or 1) of this thread's bulk store groups still read shared memory.
__device__ __forceinline__ void bulk_wait_read(int n) {
  if (n == 0)
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  else
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Warp-wide: each lane reads 32 consecutive columns of its own lane.
__device__ __forceinline__ void tmem_ld32(uint32_t ta, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(ta)
      : "memory");
#pragma unroll
  for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(r[q]);
}

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

// ---- host: tensor maps through the driver's entry point (no link against libcuda)

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// A 3-D map over [heads][rows][cols] elements, rows `row_bytes` apart, heads `head_bytes`
// apart, with a box of box_cols x box_rows x 1 and the 128-byte swizzle.
bool make_map3(CUtensorMap *m, CUtensorMapDataType ty, const void *base, uint64_t cols,
               uint64_t rows, uint64_t heads, uint64_t row_bytes, uint64_t head_bytes,
               uint32_t box_cols, uint32_t box_rows) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {cols, rows, heads};
  const cuuint64_t strides[2] = {row_bytes, head_bytes};
  const cuuint32_t box[3] = {box_cols, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, ty, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

fos_status run_qk(const fos_qk_desc *d, fos_dtype in_dt, fos_dtype out_dt, const void *q,
                  const void *k, void *scores, cudaStream_t stream, unsigned *err,
                  int max_smem) {
  const int bn = d->tile_n ? d->tile_n : kQkDefaultTileN;
  const size_t smem = qk_smem_bytes(d->head_dim, bn);
  if (smem > (size_t)max_smem) return FOS_ERR_UNSUPPORTED;
  static std::mutex mu;
  static bool prepared[3][2] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!prepared[out_dt][bn == 256]) {
      if (cudaFuncSetAttribute(qk_fn_for(out_dt, bn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               max_smem) != cudaSuccess)
        return FOS_ERR_CUDA;
      prepared[out_dt][bn == 256] = true;
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
  const uint32_t idesc = qk_idesc(in_dt == FOS_BF16, bn);
  const dim3 grid((unsigned)((d->kv_len + bn - 1) / bn), (unsigned)((d->q_len + kBM - 1) / kBM),
                  (unsigned)(d->batch * d->q_heads));
  void *args[] = {&qm, &km, &sm, &a, const_cast<uint32_t *>(&idesc)};
  if (cudaLaunchKernel(qk_fn_for(out_dt, bn), grid, dim3(kQkThreads), args, smem, stream) !=
      cudaSuccess)
    return FOS_ERR_CUDA;
  return FOS_OK;
}

}  // namespace fos
