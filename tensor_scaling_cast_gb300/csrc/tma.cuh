// Tensor-memory-accelerator (TMA) tile loads with mbarrier completion, for
// sm_90+ (used here on sm_103a), written as inline PTX.
//
// A CTA-local pipeline: one thread arms an mbarrier with the expected byte
// count and issues cp.async.bulk.tensor; every consumer waits on the
// barrier's phase parity.  Every wait is bounded by a clock deadline: on
// timeout it reports failure instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace fp8q {

// Upper bound of one barrier wait, in SM clock cycles (about half a second
// at 2 GHz; a healthy tile arrives within microseconds).
constexpr long long kWaitCycles = 1ll << 30;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy ones (a TMA write into a stage the CTA has read).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// 2-D tiled load of the box at (c0 = innermost coordinate, c1) into dst.
// c0 * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// 2-D tiled store of the box at (c0, c1) from shared memory src (bulk-group
// completion).  c0 * element size must be a multiple of 16 bytes and both
// coordinates non-negative; the parts of the box outside the tensor are not
// written.  Every thread that wrote src must have executed
// fence_proxy_async() before the issuing thread saw those writes.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed bulk store groups have
// not finished reading their shared-memory sources (the buffers of the
// others may be written again).
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for the barrier phase with the given parity; false after kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long deadline = clock64() + kWaitCycles;
  while (clock64() < deadline)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// cuTensorMapEncodeTiled from the driver, fetched through the runtime so the
// library links no driver library of its own.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map of a row-major [rows, cols] bf16 / fp32 matrix with a
// 32-row x tile_cols box, zero fill outside the matrix.  The row pitch
// (cols * element size) must be a multiple of 16 bytes.  swizzle128: the box
// rows must be 128 bytes and the shared destination 1024-byte aligned; the
// 16-byte chunk c of box row r then lands at chunk c ^ (r & 7) of that row.
// l2_promotion: 0, 128 or 256 (bytes the L2 fetches per request).
inline cudaError_t encode_tile_map(CUtensorMap* map, const void* x, bool bf16, int64_t rows,
                                   int64_t cols, int tile_cols, bool swizzle128 = false, int l2_promotion = 256) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * (bf16 ? 2u : 4u)};
  const cuuint32_t box[2] = {(cuuint32_t)tile_cols, 32u};
  const cuuint32_t estride[2] = {1u, 1u};
  if (encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
             const_cast<void*>(x), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             l2_promotion == 256   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
             : l2_promotion == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                   : CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// Tensor map of a row-major [outer, inner] byte matrix (an 8-bit output)
// for tiled stores of box_inner x box_outer boxes.  inner (the row pitch in
// bytes) and box_inner must be multiples of 16.  swizzle_bytes 0, 32 or 64:
// within each box row of box_inner bytes the 16-byte chunk c sits in shared
// memory at chunk c ^ ((r >> 2) & 1) for 32 (32-byte rows) and
// c ^ ((r >> 1) & 3) for 64 (64-byte rows); the source must be 1024-byte
// aligned.
inline cudaError_t encode_byte_map(CUtensorMap* map, void* q, int64_t outer, int64_t inner, int box_inner,
                                   int box_outer, int swizzle_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)inner};
  const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  const cuuint32_t estride[2] = {1u, 1u};
  const CUtensorMapSwizzle sw = swizzle_bytes == 64   ? CU_TENSOR_MAP_SWIZZLE_64B
                                : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q, dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
             sw, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

}  // namespace fp8q
