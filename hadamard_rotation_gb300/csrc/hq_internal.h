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

}  // namespace hq
