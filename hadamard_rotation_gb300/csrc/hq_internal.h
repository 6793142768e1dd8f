// hq_internal.h -- library-private helpers shared by the translation units of libhq.
#pragma once

#include <cuda_runtime.h>

#include "hq.h"

namespace hq {

// Record `e` as the calling thread's last CUDA error (read by hq_last_cuda_error())
// and return HQ_ERR_CUDA.
hq_status cuda_fail(cudaError_t e);

}  // namespace hq
