// Tensor-core building blocks shared by the LM-head kernels (sm_100 family):
// 2-D TMA tile copies, tcgen05 shared-memory and instruction descriptors,
// the MMA issue and commit, TMEM loads, bounded waits, and tensor-map
// encoding.  The descriptor fields are written from the PTX ISA's tables for
// tcgen05 (shared-memory matrix descriptor; instruction descriptor of
// kind::f16).
#pragma once

#include <cuda.h>

#include "vpce_device.cuh"

namespace vpce {
namespace tc {

// ---------------------------------------------------------------------------
// TMA tiles
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global tile store (bulk group of the issuing thread)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_addr(src))
               : "memory");
}

// shared -> global tile reduction: global += shared, element by element in
// the tensor map's type (fp32 adds rounded to nearest), clipped to the
// tensor's extent like a store; bulk group of the issuing thread.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_addr(src))
               : "memory");
}

// ---------------------------------------------------------------------------
// shared-memory matrix descriptors (128-byte swizzle, descriptor version 1)
// ---------------------------------------------------------------------------
// K-major tile stored as 128-byte rows (64 bf16 of K per row): start address,
// stride between 8-row groups 1024 B.  The leading offset is not used by the
// swizzled K-major layout.  K advances by 32 B per 16-element MMA step inside
// the swizzle atom.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t(1u) << 16;             // leading byte offset (unused for swizzled K-major)
  d |= uint64_t(1024u >> 4) << 32;     // stride byte offset: 8-row groups
  d |= uint64_t(1u) << 46;             // version
  d |= uint64_t(2u) << 61;             // 128-byte swizzle
  return d;
}

// MN-major tile: each K row holds 64 bf16 of M (or N) in 128 bytes, 8 K rows
// form a 1024-byte swizzle atom.  The leading byte offset is the distance
// between consecutive 64-element blocks along M/N (`mn_block_bytes`), the
// stride byte offset the distance between 8-row K groups (1024 B: the K rows
// of a block are contiguous).  A 16-deep MMA step spans two atoms, so K
// advances by 2048 B per step and every start stays atom aligned.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t mn_block_bytes) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);
  d |= uint64_t((mn_block_bytes >> 4) & 0x3FFFu) << 16;  // leading byte offset: next 64 of M/N
  d |= uint64_t(1024u >> 4) << 32;                        // stride byte offset: next 8 of K
  d |= uint64_t(1u) << 46;
  d |= uint64_t(2u) << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (D format bit 4), bf16 A
// and B (bits 7 and 10), A / B major-ness (bits 15 / 16: 0 K-major, 1
// MN-major), N / 8 at bit 17, M / 16 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u) |
         (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

// D[tmem] (+)= A * B for one 16-deep K step, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// The mbarrier gets one arrival once every MMA this thread issued so far has
// completed (and stopped reading shared memory).
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.  The load and its
// wait sit in one asm statement, so no use of the registers can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// ---------------------------------------------------------------------------
// bounded waits that also give up once another role of the CTA aborted
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ld_abort(const int* f) { return *const_cast<const volatile int*>(f); }

__device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t parity, const int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (ld_abort(abort_flag) || clock64() - t0 > kWaitLimitCycles) return false;
  }
}

__device__ __forceinline__ bool waitw(uint64_t* bar, uint32_t parity, const int* abort_flag) {
  if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  for (;;) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(kFull, ld_abort(abort_flag) != 0 || clock64() - t0 > kWaitLimitCycles)) return false;
  }
}

// ---------------------------------------------------------------------------
// tensor maps (host)
// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library; resolved once).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// A [rows, cols] row-major bf16 matrix (row stride ld elements) as a 2-D
// tensor map with a box of box_cols x box_rows and the 128-byte swizzle
// (box_cols = 64: one 128-byte swizzle row per box row).  Reads past the
// extent fill zeros; stores past it are clipped.
inline bool make_map_bf16(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld,
                          int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(ld) * 2u};
  const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [rows, cols] row-major fp32 matrix (row stride ld elements) as a 2-D
// tensor map with a box of 32 x 32 and the 128-byte swizzle (tile stores and
// reductions staged per warp).
inline bool make_map_f32(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(ld) * 4u};
  const cuuint32_t box[2] = {32u, 32u};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
}  // namespace vpce
