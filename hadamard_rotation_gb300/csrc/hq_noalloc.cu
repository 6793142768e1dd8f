// hq_noalloc.cu -- quantize a host tensor without any device allocation.
//
// hq_quantize_nvfp4_host_noalloc does what one submission of the host pipeline
// does (copy x in, pass 1, pass 2, copy codes, scales and s_global out), but its
// device staging lives in the fixed array below instead of in memory the caller
// allocated.  It exists for callers that cannot allocate device memory
// themselves; see include/hq.h.
//
// The array is a file-scope __device__ object: the CUDA runtime reserves it on
// each device where this library's code is loaded and keeps it until the process
// exits.  Host code must not use its name as an address (on the host the name
// only stands for the symbol); the device address is obtained once per device
// with cudaGetSymbolAddress, with that device current, and then handed to the
// kernels like any other device pointer.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "hq.h"
#include "hq_internal.h"

static __device__ __align__(256) uint8_t g_hq_noalloc_scratch[HQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 256;
constexpr size_t kAlign = 256;

std::mutex g_scratch_mu;
uint8_t* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Device address of the scratch array on device `dev` (which must be current).
// The first call in a context looks the address up; later calls in the same context reuse
// it.  After cudaDeviceReset the device's context is a new one, where the array has to be
// looked up again: the cache is keyed on the context's unique ID (0 = unknown, never cached).
cudaError_t scratch_on(int dev, uint8_t** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long ctx = hq::context_id();
  if (ctx == 0 || g_scratch_ctx[dev] != ctx || g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_hq_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<uint8_t*>(p);
    g_scratch_ctx[dev] = hq::context_id();  // the lookup made a context current if none was
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" hq_status hq_quantize_nvfp4_host_noalloc(const void* x_host, hq_dtype dtype,
                                                    int64_t M, int64_t K, int group,
                                                    uint8_t* q_host, uint8_t* scales_host,
                                                    float* s_global_host, hq_stream stream) {
  if (dtype != HQ_F32 && dtype != HQ_BF16) return HQ_ERR_DTYPE;
  if (group != 0 && group != 16 && group != 256) return HQ_ERR_GROUP;
  if (M < 0 || K < 0 || K % (group > 16 ? group : 16) != 0) return HQ_ERR_SHAPE;
  if (K > 0 && M > INT64_MAX / K) return HQ_ERR_SHAPE;
  if (M == 0 || K == 0) return HQ_OK;
  if (!x_host || !q_host || !scales_host || !s_global_host) return HQ_ERR_NULL;

  // Staging layout in the array: x | codes | scales | amax | s_global.
  const uint64_t n = static_cast<uint64_t>(M) * static_cast<uint64_t>(K);
  const uint64_t es = dtype == HQ_BF16 ? 2 : 4;
  if (n > (uint64_t{1} << 40)) return HQ_ERR_TOO_LARGE;
  const size_t xb = static_cast<size_t>(n * es), qb = static_cast<size_t>(n / 2),
               sb = static_cast<size_t>(n / 16);
  const size_t need = round_up(xb) + round_up(qb) + round_up(sb) + 2 * kAlign;
  if (need > HQ_NOALLOC_SCRATCH_BYTES) return HQ_ERR_TOO_LARGE;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return hq::cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return hq::cuda_fail(cudaErrorInvalidDevice);
  uint8_t* base = nullptr;
  if ((e = scratch_on(dev, &base)) != cudaSuccess) return hq::cuda_fail(e);
  uint8_t* x_d = base;
  uint8_t* q_d = x_d + round_up(xb);
  uint8_t* s_d = q_d + round_up(qb);
  float* amax_d = reinterpret_cast<float*>(s_d + round_up(sb));
  float* sg_d = reinterpret_cast<float*>(s_d + round_up(sb) + kAlign);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((e = cudaMemcpyAsync(x_d, x_host, xb, cudaMemcpyHostToDevice, st)) != cudaSuccess)
    return hq::cuda_fail(e);
  // hq_rot_amax zeroes amax before reducing into it: nothing else in the array has
  // to start at zero, since every byte read later is written first in this call.
  hq_status s = hq_rot_amax(x_d, dtype, M, K, K, group, amax_d, nullptr, stream);
  if (s != HQ_OK) return s;
  s = hq_rotate_quant_nvfp4(x_d, dtype, M, K, K, group, amax_d, q_d, s_d, sg_d, stream);
  if (s != HQ_OK) return s;
  if ((e = cudaMemcpyAsync(q_host, q_d, qb, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(scales_host, s_d, sb, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaMemcpyAsync(s_global_host, sg_d, sizeof(float), cudaMemcpyDeviceToHost, st)) !=
          cudaSuccess)
    return hq::cuda_fail(e);
  return HQ_OK;
}
