// fos_tc.cuh -- tensor-core building blocks shared by the contractions around the softmax
// (fos_qk.cu: scores = scale * Q K^T; fos_pv.cu: out = P V), sm_103a: tcgen05 operand and
// instruction descriptors, the MMA and its commit, TMA tensor loads and stores, tensor-memory
// loads, and the host's tensor maps.  Data movement and instruction encoding only; the order
// in which a contraction accumulates is fixed by the kernels that use these.
#pragma once

#include <cuda.h>

#include <mutex>

#include "fos_device.cuh"

namespace fos {

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

// The same descriptor for an MN-major operand in the 128-byte swizzle layout: rows of 128 bytes
// now hold 64 consecutive MN elements of one K index, 8 such rows (8 K indices) form a 1024-byte
// atom; the stride byte offset (bits 32-45) steps to the next 8 K indices, the leading byte
// offset (bits 16-29) to the next 64 MN elements.  A step of 16 along K advances the start
// address by 2 atoms.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t mn_block_bytes) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((mn_block_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: float32 accumulator (bits 4-5 = 1), A and B of the
// same 16-bit type (bits 7-9 and 10-12: 0 = f16, 1 = bf16), A K-major (bit 15 = 0) or MN-major
// (bit 15 = 1), B K-major (bit 16 = 0) or MN-major (bit 16 = 1), N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t f16_idesc(bool bf16, int m, int n, bool b_mn_major,
                                                 bool a_mn_major = false) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
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

// ---- host: tensor maps through the driver's entry point (no link against libcuda)

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiled encode_fn() {
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
inline bool make_map3(CUtensorMap *m, CUtensorMapDataType ty, const void *base, uint64_t cols,
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

}  // namespace fos
