// KV gather-copy: the defragmentation step of the verify path.
//
// What it computes ("The Plan Document: A Pivot Point in Custom CUDA Kernel
// Development", sections "Context: The Bottleneck That Demanded a Custom Kernel", where
// K/V defragmentation is the second avenue, and "Output Knowledge Created", Phase 3).
// Those sections give no algorithm, so the plainest reading is taken: the scattered
// page_size=1 prefix rows of a batch are copied, in index order, into consecutive rows
// of a destination, and each index entry is rewritten to the row's new slot.  A verify
// call that then reads the destination through the new indices reads contiguous rows.
// For every index entry i in [kv_indptr[0], kv_indptr[bs]), with j = i - kv_indptr[0]:
//   dst[j] = kv[kv_indices[i]]     (1152 bytes, bit for bit; zero if the slot is outside
//                                   the pool, which is flagged)
//   new_indices[i] = dst_slot0 + j
//
// Layout on the GPU.  The copy is bound by HBM bandwidth, so it is written for that:
// a fixed grid of 4 CTAs per SM (capturable; the batch extent is read on the device),
// each warp moving four rows per step.  Four rows are 288 granules of 16 bytes, nine per
// lane; every lane issues its nine streaming loads (no L1 allocation) before its nine
// streaming stores, so 36 KB per CTA and 144 KB per SM are in flight.  At 64 registers a
// few values spill to the stack; the fourth CTA gains more than that costs (5337 against
// 5240 GB/s with three CTAs; two CTAs moving eight rows a step reached 3944).
#include <cstdint>

#include "mtv_common.cuh"

namespace mtv {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kCtasPerSm = 4;   // resident together (64 registers a thread)
constexpr int kRowVec = kRowBytes / 16;                  // 72 granules per row
constexpr int kRowsPerStep = 4;                          // rows a warp moves per step
constexpr int kVecPerLane = kRowsPerStep * kRowVec / 32; // 9
static_assert(kVecPerLane * 32 == kRowsPerStep * kRowVec, "granules per lane");

constexpr uint32_t kGatherBadSlot = 1u;   // a slot outside [0, num_slots): its row is zero
constexpr uint32_t kGatherBadArgs = 2u;   // indptr negative, decreasing, past the index
                                          // array, or more rows than dst holds

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__global__ void __launch_bounds__(kGatherThreads, kCtasPerSm)
    kv_gather_kernel(const uint4* kv, int64_t num_slots, const int32_t* kv_indices,
                     int64_t num_kv_indices, const int32_t* kv_indptr, int32_t bs, uint4* dst, int64_t dst_rows,
                     int32_t dst_slot0, int32_t* new_indices, uint32_t* status) {
  const int64_t i0 = kv_indptr[0], i1 = kv_indptr[bs];
  if (i0 < 0 || i1 < i0 || i1 > num_kv_indices || i1 - i0 > dst_rows) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kGatherBadArgs);
    return;
  }
  const int64_t n = i1 - i0;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (kGatherThreads / 32);
  for (int64_t r0 = warp * kRowsPerStep; r0 < n; r0 += nwarps * kRowsPerStep) {
    // lanes 0-3: the four rows' slots, and their new indices
    int32_t my_slot = -1;
    if (lane < kRowsPerStep && r0 + lane < n) {
      const int64_t s = kv_indices[i0 + r0 + lane];
      if (s >= 0 && s < num_slots) my_slot = (int32_t)s;
      else atomicOr(status, kGatherBadSlot);
      new_indices[i0 + r0 + lane] = dst_slot0 + (int32_t)(r0 + lane);
    }
    uint4 v[kVecPerLane];
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) {
      const int g = lane + 32 * k;            // granule of the 4-row block
      const int row = g / kRowVec, col = g - row * kRowVec;
      const int32_t s = __shfl_sync(0xffffffffu, my_slot, row);
      v[k] = (r0 + row < n && s >= 0) ? ld_stream(kv + (int64_t)s * kRowVec + col)
                                      : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) {
      const int g = lane + 32 * k;
      const int row = g / kRowVec, col = g - row * kRowVec;
      if (r0 + row < n) st_stream(dst + (r0 + row) * kRowVec + col, v[k]);
    }
  }
}

}  // namespace

int kv_gather_ctas_per_sm() { return kCtasPerSm; }

int launch_kv_gather(const void* kv, int64_t num_slots, const int32_t* kv_indices,
                     int64_t num_kv_indices, const int32_t* kv_indptr, int32_t bs, void* dst, int64_t dst_rows,
                     int32_t dst_slot0, int32_t* new_indices, uint32_t* status, int grid,
                     cudaStream_t stream) {
  kv_gather_kernel<<<grid, kGatherThreads, 0, stream>>>(
      (const uint4*)kv, num_slots, kv_indices, num_kv_indices, kv_indptr, bs, (uint4*)dst, dst_rows, dst_slot0,
      new_indices, status);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mtv
