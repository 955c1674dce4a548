// Tensor-memory-accelerator (TMA) helpers: host-side encoding of 2-D bf16
// tensor maps with 128-byte swizzle, and the device-side tile / gather4 loads.
//
// The encode function is fetched from the driver through the runtime's entry
// point query, so the library links no libcuda.  Every map describes a
// row-major [rows][cols] bf16 tensor; the box is 64 columns (128 bytes, one
// swizzle row) by `box_rows` rows.  Out-of-range boxes are zero-filled.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace b4 {

typedef CUresult (*TmapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline TmapEncodeFn tmap_encode_fn() {
  static TmapEncodeFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TmapEncodeFn>(p);
  }
  return fn;
}

// Returns false when the driver entry point is missing or rejects the map
// (base not 16-byte aligned, row pitch not a multiple of 16 bytes, ...).
inline bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  TmapEncodeFn fn = tmap_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Box at (column c0, row r0) -> shared memory (1024-byte aligned for the swizzle).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int c0, int r0, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(c0), "r"(r0), "r"(smem_u32(bar))
      : "memory");
}

// Four arbitrary rows (a map whose box is one row high), columns [c0, c0+64).
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* tm, int c0, int r0, int r1, int r2, int r3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor, canonical K-major layout with 128-byte
// swizzle: rows of 128 bytes (64 bf16 of K), 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;             // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;             // layout type: 128-byte swizzle
  return d;
}

}  // namespace b4
