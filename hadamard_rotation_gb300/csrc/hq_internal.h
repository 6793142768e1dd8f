// hq_internal.h -- library-private helpers shared by the translation units of libhq.
#pragma once

#include <cuda_runtime.h>

#include "hq.h"

namespace hq {

// Record `e` as the calling thread's last CUDA error (read by hq_last_cuda_error())
// and return HQ_ERR_CUDA.
hq_status cuda_fail(cudaError_t e);

// The device fault word of the int8 translation unit (hq_int8.cu has its own copy
// of g_hq_fault): read it into *fault and, when `clear`, reset it.  The caller has
// synchronised the device.
cudaError_t int8_fault_word(unsigned int* fault, bool clear);

// Launch the bounded-wait self-test kernel of the int8 translation unit on `stream`.
cudaError_t int8_selftest_bounded_wait(cudaStream_t stream);

// Unique ID of the CUDA context current on the calling thread (the driver's cuCtxGetId, which
// never repeats within a process), or 0 when no context is current or the driver does not
// report one.  Per-device caches of context state (a symbol's device address, a kernel's
// shared-memory attribute) key on it: after cudaDeviceReset the device's primary context is a
// new one with a new ID, so a cache entry of the old context no longer matches.
unsigned long long context_id();

}  // namespace hq
