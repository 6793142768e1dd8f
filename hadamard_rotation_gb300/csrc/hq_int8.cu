// hq_int8.cu -- C ABI entry point of the INT8 per-token rotate-quant (include/hq.h)
// and its launch logic.  The kernel is in hq_int8.cuh.
#include <cuda_runtime.h>

#include <cstdint>

#include "hq.h"
#include "hq_int8.cuh"
#include "hq_internal.h"

namespace {

using hq::cuda_fail;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Dynamic shared memory the parking kernel may take: the 227 KB a CTA may opt in to, less
// 2 KB for its static shared memory and the 1 KB alignment of the dynamic part.
constexpr size_t kI8ParkSmemLimit = 227 * 1024 - 2 * 1024;

// INT8 per-token rotate-quant: one CTA of kI8Threads per SM, looping over row groups.
template <int G, bool BF16, int MODE, bool FULL>
hq_status launch_int8(const hq::I8Params& p, hq_stream stream) {
  // G <= 16 is bound by memory: fixed warp places (L = 1); G >= 64: round robin.
  auto kernel = hq::k_rotate_quant_int8<G, BF16, MODE, FULL, (G > 16)>;
  const size_t smem = (MODE == hq::kLoadTma) ? static_cast<size_t>(hq::kI8RingBytes) : 0;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e);
  if (smem > 48 * 1024 &&
      (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem))) != cudaSuccess)
    return cuda_fail(e);
  const int64_t row_groups = (p.M + p.rows_per_block - 1) / p.rows_per_block;
  const unsigned grid = static_cast<unsigned>(row_groups < sms ? row_groups : sms);
  kernel<<<grid, hq::kI8Threads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return HQ_OK;
}

// Rows longer than the chip can park: one CTA of kI8Threads per SM, each row read twice.
template <int G, bool BF16>
hq_status launch_int8_long(const hq::I8Params& p, hq_stream stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e);
  const unsigned grid = static_cast<unsigned>(p.M < sms ? p.M : sms);
  hq::k_rotate_quant_int8_long<G, BF16><<<grid, hq::kI8Threads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return HQ_OK;
}

// Rows of 17 to 59 warp tiles: parked whole on chip (tensor memory and shared memory), one
// CTA of kI8Threads per SM; bf16 rows load through a TMA ring of 2 or 1 tiles per warp when
// shared memory has room for it beside the parked tiles.
template <int G, bool BF16, int STAGES>
hq_status launch_int8_park_ring(const hq::I8Params& p, size_t park_bytes, hq_stream stream) {
  auto kernel = p.rows_per_block > 1 ? hq::k_rotate_quant_int8_park<G, BF16, true, STAGES>
                                     : hq::k_rotate_quant_int8_park<G, BF16, false, STAGES>;
  const size_t smem = park_bytes + static_cast<size_t>(hq::i8_park_ring_bytes(STAGES));
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return cuda_fail(e);
  if (smem > 48 * 1024 &&
      (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem))) != cudaSuccess)
    return cuda_fail(e);
  const int64_t n_blocks = (p.M + p.rows_per_block - 1) / p.rows_per_block;
  const unsigned grid = static_cast<unsigned>(n_blocks < sms ? n_blocks : sms);
  kernel<<<grid, hq::kI8Threads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return HQ_OK;
}

template <int G, bool BF16>
hq_status launch_int8_park(const hq::I8Params& p, hq_stream stream) {
  const int n_g = p.rows_per_block * p.tiles_per_row;
  const int smem_tiles = n_g > hq::kI8ParkTmemTiles ? n_g - hq::kI8ParkTmemTiles : 0;
  const size_t park = static_cast<size_t>(smem_tiles) * hq::kI8ParkTileBytes;
  if constexpr (BF16) {
    if (park + hq::i8_park_ring_bytes(2) <= kI8ParkSmemLimit)
      return launch_int8_park_ring<G, true, 2>(p, park, stream);
    if (park + hq::i8_park_ring_bytes(1) <= kI8ParkSmemLimit)
      return launch_int8_park_ring<G, true, 1>(p, park, stream);
  }
  return launch_int8_park_ring<G, BF16, 0>(p, park, stream);
}

template <int G>
hq_status dispatch_int8(const hq::I8Params& p, bool bf16, hq_stream s) {
  if (p.tiles_per_row > hq::kI8ParkMaxTiles)
    return bf16 ? launch_int8_long<G, true>(p, s) : launch_int8_long<G, false>(p, s);
  if (p.K > hq::kI8MaxK)
    return bf16 ? launch_int8_park<G, true>(p, s) : launch_int8_park<G, false>(p, s);
  const bool full = p.K % hq::kI8TileElems == 0;
  if (bf16)
    return full ? launch_int8<G, true, hq::kLoadTma, true>(p, s)
                : launch_int8<G, true, hq::kLoadTma, false>(p, s);
  return full ? launch_int8<G, false, hq::kLoadDirect, true>(p, s)
              : launch_int8<G, false, hq::kLoadDirect, false>(p, s);
}

}  // namespace

namespace hq {
// The bounded-wait self-test in this translation unit (see k_selftest_bounded_wait in hq.cu).
__global__ void k_int8_selftest_bounded_wait() {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(b, 0);  // phase 0 never completes
  if (!__all_sync(0xFFFFFFFFu, ok) && threadIdx.x == 0) atomicOr(&g_hq_fault, kFaultWaitTimeout);
}
}  // namespace hq

cudaError_t hq::int8_selftest_bounded_wait(cudaStream_t stream) {
  k_int8_selftest_bounded_wait<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

cudaError_t hq::int8_fault_word(unsigned int* fault, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(fault, g_hq_fault, sizeof(unsigned int));
  if (e == cudaSuccess && clear && *fault) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_hq_fault, &zero, sizeof(unsigned int));
  }
  return e;
}

extern "C" {

hq_status hq_rotate_quant_int8(const void* x, hq_dtype dtype, int64_t M, int64_t K, int64_t ldx,
                               int group, int8_t* q, float* scales, hq_stream stream) {
  if (dtype != HQ_F32 && dtype != HQ_BF16) return HQ_ERR_DTYPE;
  if (group != 4 && group != 16 && group != 64 && group != 256 && group != 1024) return HQ_ERR_GROUP;
  if (M < 0 || K < 0 || ldx < K || K % group != 0 || K % 16 != 0) return HQ_ERR_SHAPE;
  if (K / hq::kI8TileElems >= (int64_t{1} << 30)) return HQ_ERR_SHAPE;  // tiles per row in an int
  const int64_t es = dtype == HQ_BF16 ? 2 : 4;
  if ((K > 0 && M > INT64_MAX / K) || ldx > INT64_MAX / es) return HQ_ERR_SHAPE;
  if (M == 0 || K == 0) return HQ_OK;
  if (!x || !q || !scales) return HQ_ERR_NULL;
  if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scales, 4)) return HQ_ERR_ALIGN;
  if (M > 1 && (ldx * es) % 16 != 0) return HQ_ERR_ALIGN;
  hq::I8Params p = {};
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = (M > 1 ? ldx : K) * es;
  p.M = M;
  p.K = K;
  p.tiles_per_row = static_cast<int>((K + hq::kI8TileElems - 1) / hq::kI8TileElems);
  int a = p.tiles_per_row, b = hq::kI8Warps;  // lcm(T, 16) = T * 16 / gcd(T, 16)
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  const int lcm = p.tiles_per_row / a * hq::kI8Warps;
  if (p.tiles_per_row > hq::kI8ParkMaxTiles) {  // the long-row kernel: one row at a time
    p.rows_per_block = 1;
    p.tiles_per_warp = 0;
  } else if (p.tiles_per_row > hq::kI8Warps) {
    // rows parked on chip: B rows per CTA step (B T <= 59), the B whose B T tiles fill the
    // 16 warps' rounds best (the smaller B on a tie)
    int best_b = 1, best_used = 0, best_slots = 1;
    for (int b = 1; b <= hq::kI8ParkMaxRows && b * p.tiles_per_row <= hq::kI8ParkMaxTiles; ++b) {
      const int used = b * p.tiles_per_row;
      const int slots = (used + hq::kI8Warps - 1) / hq::kI8Warps * hq::kI8Warps;
      if (static_cast<int64_t>(used) * best_slots > static_cast<int64_t>(best_used) * slots) {
        best_b = b;
        best_used = used;
        best_slots = slots;
      }
    }
    p.rows_per_block = best_b;
    p.tiles_per_warp = 0;
  } else if (group <= 16) {  // memory-bound: whole rows, one tile per warp (see hq_int8.cuh)
    p.rows_per_block = hq::kI8Warps / p.tiles_per_row;
    p.tiles_per_warp = 1;
  } else {
    p.rows_per_block = lcm / p.tiles_per_row;
    p.tiles_per_warp = lcm / hq::kI8Warps;
  }
  p.q = q;
  p.scales = scales;
  const bool bf16 = dtype == HQ_BF16;
  switch (group) {
    case 4: return dispatch_int8<4>(p, bf16, stream);
    case 16: return dispatch_int8<16>(p, bf16, stream);
    case 64: return dispatch_int8<64>(p, bf16, stream);
    case 256: return dispatch_int8<256>(p, bf16, stream);
    default: return dispatch_int8<1024>(p, bf16, stream);
  }
}

}  // extern "C"
