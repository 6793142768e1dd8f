// hq_host.cu -- host pipeline of libhq: quantize tensors that live in host memory.
//
// One submission = copy x host -> device, pass 1 (hq_rot_amax), pass 2
// (hq_rotate_quant_nvfp4), codes, scales and s_global device -> host.
// Consecutive submissions overlap: two buffer sets in the caller's device
// workspace alternate, and the three phases run on three streams ordered by
// events, so the input copy of submission n+1 runs while submission n computes
// and while its outputs travel back.  The input moves by a copy engine; the
// outputs are stored into the host buffers by a kernel (k_copy_out) wherever the
// device can write them (pinned or registered memory, or pageable memory on a
// device that reaches it through the host page tables), else copied.  Separate
// device-to-host copies had shared a copy engine with the next input copy.
//
//   in stream      H2D(n) ........ H2D(n+1) ........ H2D(n+2)
//   compute stream        pass1,2(n)         pass1,2(n+1)
//   out stream                      D2H(n) ........  D2H(n+1)
//
// Slot reuse: submission n+2 overwrites the buffers of submission n, so its input
// copy waits until pass 2 of n has finished reading x, and its kernels wait until
// the output copy of n has finished reading the codes.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "hq.h"
#include "hq_internal.h"

struct hq_host_pipeline {
  int device = 0;
  int64_t M = 0, K = 0;
  hq_dtype dtype = HQ_BF16;
  int group = 16;
  size_t x_bytes = 0, q_bytes = 0, s_bytes = 0;
  struct Slot {
    uint8_t* x = nullptr;
    uint8_t* q = nullptr;
    uint8_t* s = nullptr;
    float* amax = nullptr;
    float* sglobal = nullptr;
    cudaEvent_t in_done = nullptr;       // input copy finished
    cudaEvent_t compute_done = nullptr;  // pass 2 finished
    cudaEvent_t out_done = nullptr;      // output copies finished
    bool used = false;
  } slot[2];
  cudaStream_t in = nullptr, compute = nullptr, out = nullptr;
  uint64_t submitted = 0;
  bool pageable_writable = false;  // the device writes pageable host memory through the host page tables
  int copy_out_ctas = 0;
  int broken_error = 0;  // the cudaError_t of a submission that failed after enqueueing work
  int inject_step = -1;  // hq_host_pipeline_inject_failure: the step the next submission fails at
};

namespace {

hq_status fail(cudaError_t e) { return hq::cuda_fail(e); }

// Results to host memory by SMs rather than a copy engine.  Several device-to-host
// copies per submission shared a copy engine with the next submission's host-to-device
// copy and serialised with it; SM stores to host memory run beside that copy.
__global__ void k_copy_out(const uint8_t* __restrict__ q, uint8_t* __restrict__ q_host, size_t q_bytes,
                           const uint8_t* __restrict__ s, uint8_t* __restrict__ s_host, size_t s_bytes,
                           const float* __restrict__ sg, float* __restrict__ sg_host) {
  const size_t i0 = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  auto copy = [&](const uint8_t* src, uint8_t* dst, size_t n) {
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0;
    const size_t nv = vec ? n / 16 : 0;
    for (size_t k = i0; k < nv; k += stride)
      reinterpret_cast<uint4*>(dst)[k] = __ldcs(reinterpret_cast<const uint4*>(src) + k);
    for (size_t k = nv * 16 + i0; k < n; k += stride) dst[k] = src[k];
  };
  copy(q, q_host, q_bytes);
  copy(s, s_host, s_bytes);
  if (i0 == 0) sg_host[0] = sg[0];
}

// The device address through which a kernel may write host buffer p, or nullptr if
// it may not (then a copy engine moves the data).
void* device_view(const void* p, bool pageable_writable) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return nullptr;
  }
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;  // pinned or registered
  if (a.type == cudaMemoryTypeUnregistered && pageable_writable) return const_cast<void*>(p);
  return nullptr;
}

constexpr size_t kAlign = 256;

size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool sizes(int64_t M, int64_t K, hq_dtype dt, size_t* xb, size_t* qb, size_t* sb) {
  if (M <= 0 || K <= 0 || K % 16 != 0) return false;
  if (M > INT64_MAX / K) return false;
  if (K / 16 > 0xFFFFFFFFll) return false;  // a row the kernels can index (hq_rot_amax's bound)
  const uint64_t n = static_cast<uint64_t>(M) * static_cast<uint64_t>(K);
  if (n > (uint64_t{1} << 58)) return false;  // keeps every byte count below from wrapping
  *xb = n * (dt == HQ_BF16 ? 2u : 4u);
  *qb = n / 2;
  *sb = n / 16;
  return true;
}

size_t slot_bytes(size_t xb, size_t qb, size_t sb) {
  return round_up(xb) + round_up(qb) + round_up(sb) + 2 * kAlign;
}

void destroy_objects(hq_host_pipeline* p) {
  for (auto& s : p->slot) {
    if (s.in_done) cudaEventDestroy(s.in_done);
    if (s.compute_done) cudaEventDestroy(s.compute_done);
    if (s.out_done) cudaEventDestroy(s.out_done);
  }
  if (p->in) cudaStreamDestroy(p->in);
  if (p->compute) cudaStreamDestroy(p->compute);
  if (p->out) cudaStreamDestroy(p->out);
}

}  // namespace

extern "C" {

size_t hq_host_pipeline_workspace_bytes(int64_t M, int64_t K, hq_dtype dtype) {
  size_t xb, qb, sb;
  if ((dtype != HQ_F32 && dtype != HQ_BF16) || !sizes(M, K, dtype, &xb, &qb, &sb)) return 0;
  return 2 * slot_bytes(xb, qb, sb);
}

hq_status hq_host_pipeline_create(int64_t M, int64_t K, hq_dtype dtype, int group, void* d_work,
                                  size_t work_bytes, hq_host_pipeline** out) {
  if (!out || !d_work) return HQ_ERR_NULL;
  *out = nullptr;
  if (dtype != HQ_F32 && dtype != HQ_BF16) return HQ_ERR_DTYPE;
  if (group != 0 && group != 16 && group != 256) return HQ_ERR_GROUP;
  size_t xb, qb, sb;
  if (!sizes(M, K, dtype, &xb, &qb, &sb) || K % (group > 16 ? group : 16) != 0)
    return HQ_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(d_work) % kAlign != 0) return HQ_ERR_ALIGN;
  const size_t per_slot = slot_bytes(xb, qb, sb);
  if (work_bytes < 2 * per_slot) return HQ_ERR_SHAPE;

  hq_host_pipeline* p = new (std::nothrow) hq_host_pipeline();
  if (!p) return HQ_ERR_NULL;
  cudaError_t e = cudaGetDevice(&p->device);
  if (e != cudaSuccess) {
    delete p;
    return fail(e);
  }
  p->M = M;
  p->K = K;
  p->dtype = dtype;
  p->group = group;
  p->x_bytes = xb;
  p->q_bytes = qb;
  p->s_bytes = sb;
  uint8_t* base = static_cast<uint8_t*>(d_work);
  for (int i = 0; i < 2; ++i) {
    auto& s = p->slot[i];
    uint8_t* b = base + i * per_slot;
    s.x = b;
    b += round_up(xb);
    s.q = b;
    b += round_up(qb);
    s.s = b;
    b += round_up(sb);
    s.amax = reinterpret_cast<float*>(b);
    s.sglobal = reinterpret_cast<float*>(b + kAlign);
  }
  const unsigned ev_flags = cudaEventDisableTiming;
  for (auto& s : p->slot) {
    if ((e = cudaEventCreateWithFlags(&s.in_done, ev_flags)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&s.compute_done, ev_flags)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&s.out_done, ev_flags)) != cudaSuccess) {
      destroy_objects(p);
      delete p;
      return fail(e);
    }
  }
  int pma = 0, host_tables = 0, sms = 0;
  if ((e = cudaDeviceGetAttribute(&pma, cudaDevAttrPageableMemoryAccess, p->device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&host_tables, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                                  p->device)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device)) != cudaSuccess) {
    destroy_objects(p);
    delete p;
    return fail(e);
  }
  p->pageable_writable = pma && host_tables;
  p->copy_out_ctas = sms;
  if ((e = cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&p->compute, cudaStreamNonBlocking)) != cudaSuccess ||
      (e = cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking)) != cudaSuccess) {
    destroy_objects(p);
    delete p;
    return fail(e);
  }
  *out = p;
  return HQ_OK;
}

hq_status hq_host_pipeline_submit(hq_host_pipeline* p, const void* x_host, uint8_t* q_host,
                                  uint8_t* scales_host, float* s_global_host) {
  if (!p || !x_host || !q_host || !scales_host || !s_global_host) return HQ_ERR_NULL;
  if (p->broken_error != 0) return fail(static_cast<cudaError_t>(p->broken_error));
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(e);
  if (dev != p->device && (e = cudaSetDevice(p->device)) != cudaSuccess) return fail(e);
  auto& s = p->slot[p->submitted & 1];
  // A refused step (or the injected one) ends the submission.  Steps 0..3: input copy, pass 1,
  // pass 2, output transfer.
  const int inject = p->inject_step;
  p->inject_step = -1;
  hq_status st = HQ_OK;
  bool enqueued = false;  // some work of this submission is on a stream
  auto injected = [&](int step) {
    if (st == HQ_OK && step == inject) st = fail(cudaErrorNotPermitted);
    return st != HQ_OK;
  };
  // input copy: the slot's x must no longer be read by an earlier pass 2
  if (!injected(0)) {
    if (s.used && (e = cudaStreamWaitEvent(p->in, s.compute_done, 0)) != cudaSuccess) st = fail(e);
    if (st == HQ_OK &&
        (e = cudaMemcpyAsync(s.x, x_host, p->x_bytes, cudaMemcpyHostToDevice, p->in)) != cudaSuccess)
      st = fail(e);
    if (st == HQ_OK) enqueued = true;
    if (st == HQ_OK && (e = cudaEventRecord(s.in_done, p->in)) != cudaSuccess) st = fail(e);
    // both passes: after the input arrived and after the slot's last outputs left
    if (st == HQ_OK && (e = cudaStreamWaitEvent(p->compute, s.in_done, 0)) != cudaSuccess)
      st = fail(e);
    if (st == HQ_OK && s.used && (e = cudaStreamWaitEvent(p->compute, s.out_done, 0)) != cudaSuccess)
      st = fail(e);
  }
  if (!injected(1))
    st = hq_rot_amax(s.x, p->dtype, p->M, p->K, p->K, p->group, s.amax, nullptr, p->compute);
  if (!injected(2)) {
    st = hq_rotate_quant_nvfp4(s.x, p->dtype, p->M, p->K, p->K, p->group, s.amax, s.q, s.s,
                               s.sglobal, p->compute);
    if (st == HQ_OK && (e = cudaEventRecord(s.compute_done, p->compute)) != cudaSuccess)
      st = fail(e);
  }
  // outputs to the host: stored by a kernel where the device can write the buffers,
  // otherwise copied
  if (!injected(3)) {
    if ((e = cudaStreamWaitEvent(p->out, s.compute_done, 0)) != cudaSuccess) st = fail(e);
    void* qv = device_view(q_host, p->pageable_writable);
    void* sv = device_view(scales_host, p->pageable_writable);
    void* gv = device_view(s_global_host, p->pageable_writable);
    if (st == HQ_OK && qv && sv && gv) {
      k_copy_out<<<p->copy_out_ctas, 512, 0, p->out>>>(s.q, static_cast<uint8_t*>(qv), p->q_bytes,
                                                       s.s, static_cast<uint8_t*>(sv), p->s_bytes,
                                                       s.sglobal, static_cast<float*>(gv));
      if ((e = cudaGetLastError()) != cudaSuccess) st = fail(e);
    } else if (st == HQ_OK) {
      if ((e = cudaMemcpyAsync(q_host, s.q, p->q_bytes, cudaMemcpyDeviceToHost, p->out)) !=
          cudaSuccess)
        st = fail(e);
      if (st == HQ_OK && (e = cudaMemcpyAsync(scales_host, s.s, p->s_bytes,
                                              cudaMemcpyDeviceToHost, p->out)) != cudaSuccess)
        st = fail(e);
      if (st == HQ_OK && (e = cudaMemcpyAsync(s_global_host, s.sglobal, sizeof(float),
                                              cudaMemcpyDeviceToHost, p->out)) != cudaSuccess)
        st = fail(e);
    }
    if (st == HQ_OK && (e = cudaEventRecord(s.out_done, p->out)) != cudaSuccess) st = fail(e);
  }
  if (st == HQ_OK) {
    s.used = true;
    ++p->submitted;
  } else if (enqueued) {
    // The slot's events may not cover what is in flight: no later submission may reuse it.
    p->broken_error = hq_last_cuda_error();
    if (p->broken_error == 0) p->broken_error = static_cast<int>(cudaErrorUnknown);
  }
  if (dev != p->device) cudaSetDevice(dev);
  return st;
}

hq_status hq_host_pipeline_wait(hq_host_pipeline* p) {
  if (!p) return HQ_ERR_NULL;
  cudaError_t e = cudaStreamSynchronize(p->out);
  if (e != cudaSuccess) return fail(e);
  e = cudaStreamSynchronize(p->compute);
  if (e != cudaSuccess) return fail(e);
  e = cudaStreamSynchronize(p->in);
  if (e != cudaSuccess) return fail(e);
  return HQ_OK;
}

hq_status hq_host_pipeline_inject_failure(hq_host_pipeline* p, int step) {
  if (!p) return HQ_ERR_NULL;
  if (step > 3) return HQ_ERR_SHAPE;
  p->inject_step = step < 0 ? -1 : step;
  return HQ_OK;
}

hq_status hq_host_pipeline_destroy(hq_host_pipeline* p) {
  if (!p) return HQ_OK;
  hq_status st = hq_host_pipeline_wait(p);
  destroy_objects(p);
  delete p;
  return st;
}

}  // extern "C"
