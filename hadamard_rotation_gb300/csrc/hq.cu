// hq.cu -- C ABI of libhq (declared in include/hq.h) and the launch logic.
//
// Every entry point validates its arguments on the host, picks the kernel
// instance for (rotation group, element type, contiguous/strided rows), sizes a
// persistent grid (resident CTAs per SM x SM count, capped by the work), and
// enqueues on the caller's stream.  Nothing here allocates, synchronises or
// waits on the device.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "hq.h"
#include "hq_internal.h"
#include "hq_kernels.cuh"

namespace hq {

// ---------------------------------------------------------------------------
// Self-test of the bounded wait: one warp waits on an mbarrier that nothing
// completes; the wait gives up after about kWaitLimitNs and the fault is recorded.
// ---------------------------------------------------------------------------
__global__ void k_selftest_bounded_wait() {
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

namespace {
thread_local int g_last_cuda_error = 0;
}  // namespace

hq_status hq::cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return HQ_ERR_CUDA;
}

namespace {

// cuCtxGetCurrent and cuCtxGetId, reached through the runtime's driver entry points (so the
// library needs no link against the driver library).  CUcontext is an opaque pointer and
// CUresult an int enum whose success value is 0.
using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);

struct DriverCtxCalls {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverCtxCalls& driver_ctx_calls() {
  static const DriverCtxCalls calls = [] {
    DriverCtxCalls c;
    auto lookup = [](const char* name) -> void* {
      void* f = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess) {
        cudaGetLastError();  // a failed lookup leaves no error behind for the caller's next call
        return nullptr;
      }
      return q == cudaDriverEntryPointSuccess ? f : nullptr;
    };
    c.get_current = reinterpret_cast<CtxGetCurrentFn>(lookup("cuCtxGetCurrent"));
    c.get_id = reinterpret_cast<CtxGetIdFn>(lookup("cuCtxGetId"));
    return c;
  }();
  return calls;
}

}  // namespace

unsigned long long hq::context_id() {
  const DriverCtxCalls& c = driver_ctx_calls();
  if (!c.get_current || !c.get_id) return 0;
  void* ctx = nullptr;
  if (c.get_current(&ctx) != 0 || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (c.get_id(ctx, &id) != 0) return 0;
  return id;
}

namespace {

using hq::cuda_fail;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_size(hq_dtype dt) { return dt == HQ_BF16 ? 2 : 4; }

// Divider constants for hq::fast_div (Granlund & Montgomery 1994, Figure 4.1).
hq::FastDiv make_fast_div(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t{1} << l) < d) ++l;
  const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1;
  hq::FastDiv f;
  f.m = static_cast<uint32_t>(m);
  f.s1 = l ? 1u : 0u;
  f.s2 = l ? l - 1 : 0u;
  return f;
}

// Resident CTAs per SM for a kernel, cached per device and context (the dynamic
// shared-memory attribute set below belongs to the context: after cudaDeviceReset it is
// set again), and the SM count, cached per device.
struct GridCache {
  std::mutex mu;
  static constexpr int kSlots = 128;
  const void* fn[kSlots] = {};
  int dev[kSlots] = {};
  unsigned long long ctx[kSlots] = {};
  int ctas[kSlots] = {};
  int n = 0;
  int sms[64] = {};
};
GridCache g_grid;

cudaError_t persistent_grid(const void* fn, uint64_t n_tiles, size_t smem, unsigned* grid) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long ctx = hq::context_id();
  int per_sm = 0, sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_grid.mu);
    for (int i = 0; i < g_grid.n; ++i)
      if (g_grid.fn[i] == fn && g_grid.dev[i] == dev && ctx != 0 && g_grid.ctx[i] == ctx)
        per_sm = g_grid.ctas[i];
    if (dev >= 0 && dev < 64) sms = g_grid.sms[dev];
  }
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_grid.mu);
    if (dev >= 0 && dev < 64) g_grid.sms[dev] = sms;
  }
  if (per_sm == 0) {
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, hq::kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    // The calls above made a context current if none was: key the entry on it.
    const unsigned long long now = ctx != 0 ? ctx : hq::context_id();
    if (now != 0) {
      std::lock_guard<std::mutex> lock(g_grid.mu);
      int slot = -1;
      for (int i = 0; i < g_grid.n; ++i)
        if (g_grid.fn[i] == fn && g_grid.dev[i] == dev) slot = i;  // an older context's entry
      if (slot < 0 && g_grid.n < GridCache::kSlots) slot = g_grid.n++;
      if (slot >= 0) {
        g_grid.fn[slot] = fn;
        g_grid.dev[slot] = dev;
        g_grid.ctx[slot] = now;
        g_grid.ctas[slot] = per_sm;
      }
    }
  }
  const uint64_t want = (n_tiles + hq::kWarpsPerCta - 1) / hq::kWarpsPerCta;
  const uint64_t cap = static_cast<uint64_t>(sms) * static_cast<uint64_t>(per_sm);
  *grid = static_cast<unsigned>(want < cap ? want : cap);
  if (*grid == 0) *grid = 1;
  return cudaSuccess;
}

// Launch with `smem` bytes of dynamic shared memory (the TMA ring of the
// contiguous-row kernels; 0 for the others).  pdl: allow programmatic dependent launch,
// so that the grid may be launched while the kernel before it on the stream is still
// running; the kernel must then execute griddepcontrol.wait before it touches global
// memory (pass 2 does so first thing), which makes it wait for that kernel's completion
// and memory, exactly as without the attribute.  Only the launch and the CTAs' start
// overlap the previous kernel's end.
template <typename Kernel>
hq_status launch(Kernel kernel, const hq::Params& p, hq_stream stream, size_t smem = 0, bool pdl = false) {
  unsigned grid = 0;
  cudaError_t e = persistent_grid(reinterpret_cast<const void*>(kernel), p.n_tiles, smem, &grid);
  if (e != cudaSuccess) return cuda_fail(e);
  if (pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(hq::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess) return cuda_fail(e);
  } else {
    kernel<<<grid, hq::kThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return HQ_OK;
}

// Shape checks shared by the two quantization passes.
// An empty tensor (M == 0 or K == 0) may come with NULL data pointers.
hq_status check_x(const void* x, hq_dtype dt, int64_t M, int64_t K, int64_t ldx, int group) {
  if (dt != HQ_F32 && dt != HQ_BF16) return HQ_ERR_DTYPE;
  if (group != 0 && group != 16 && group != 256) return HQ_ERR_GROUP;
  if (M < 0 || K < 0 || ldx < K) return HQ_ERR_SHAPE;
  const int64_t unit = group > 16 ? group : 16;
  if (K % unit != 0) return HQ_ERR_SHAPE;
  // The kernels count the 16-element blocks of one row in 32 bits.
  if (K / 16 > static_cast<int64_t>(UINT32_MAX)) return HQ_ERR_SHAPE;
  if (K > 0 && M > INT64_MAX / K) return HQ_ERR_SHAPE;
  const int64_t es = elem_size(dt);
  if (ldx > INT64_MAX / es) return HQ_ERR_SHAPE;
  if (M == 0 || K == 0) return HQ_OK;
  if (!x) return HQ_ERR_NULL;
  if (!aligned(x, 16)) return HQ_ERR_ALIGN;
  if (M > 1 && (ldx * es) % 16 != 0) return HQ_ERR_ALIGN;
  return HQ_OK;
}

// Workspace words (HQ_QUANTIZE_WORKSPACE_WORDS in all): [0] unused, [1] the amax being
// reduced (pass 1 of hq_quantize_nvfp4, or the next amax of the delayed pass), [2] CTAs of
// that kernel done, [3] warps done with the tile counters; then the tile counters of the
// run-time split from word kSchedWord on, each on its own 128-byte line.  A call that records
// no fault leaves every word 0.
constexpr int kSchedWord = hq::kSchedStrideWords;
static_assert(kSchedWord + hq::kSchedClasses * hq::kSchedStrideWords <= HQ_QUANTIZE_WORKSPACE_WORDS,
              "workspace too small for the tile counters");

// The run-time split: contiguous rows only (it reads through the TMA ring), from 16384 warp
// tiles (32 M elements) on: below that a warp has a few tiles, there is little to balance,
// and the fixed split measured faster (bf16 [4096, 4096]: 10.5 against 11.8 us per pass 2);
// up to 2^34 tiles (a tile's class index is a 32-bit counter value).
bool schedulable(const hq::Params& p, const uint32_t* workspace, bool strided) {
  return workspace != nullptr && !strided && p.n_tiles >= 16384 && p.n_tiles < (uint64_t{1} << 34);
}

hq::Params base_params(const void* x, hq_dtype dt, int64_t M, int64_t K, int64_t ldx) {
  hq::Params p = {};
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = ldx * elem_size(dt);
  p.nb = static_cast<uint64_t>(M) * static_cast<uint64_t>(K / 16);
  p.nbr = static_cast<uint32_t>(K / 16);  // check_x bounds it
  if (p.nbr > 0) p.div_nbr = make_fast_div(p.nbr);
  p.n_tiles = (p.nb + hq::kTileBlocks - 1) / hq::kTileBlocks;
  return p;
}

// Rows are read as a flat array when they are back to back.
bool is_strided(int64_t M, int64_t K, int64_t ldx) { return M > 1 && ldx != K; }

// How contiguous rows are read (hq::LoadMode): through the per-warp TMA ring
// (default) or with direct vector loads.
#ifndef HQ_PASS1_MODE
#define HQ_PASS1_MODE hq::kLoadTma
#endif
#ifndef HQ_PASS2_MODE
#define HQ_PASS2_MODE hq::kLoadTma
#endif

template <int STAGES>
size_t ring_bytes(int mode, bool bf16) {
  if (mode != hq::kLoadTma) return 0;
  return bf16 ? hq::Ring<true, STAGES>::kSmemBytes : hq::Ring<false, STAGES>::kSmemBytes;
}

template <int G, bool BF16, int MODE>
hq_status launch_rot_amax(const hq::Params& p, bool write_y, hq_stream s) {
  const size_t smem = ring_bytes<HQ_PASS1_STAGES>(MODE, BF16);
  return write_y ? launch(hq::k_rot_amax<G, BF16, MODE, true>, p, s, smem, p.sync != nullptr)
                 : launch(hq::k_rot_amax<G, BF16, MODE, false>, p, s, smem, p.sync != nullptr);
}

// Pass 1 for G <= 16 on contiguous, 32-byte aligned rows uses the streaming kernel
// (1 = on).
#ifndef HQ_PASS1_STREAM
#define HQ_PASS1_STREAM 1
#endif

template <int G>
hq_status dispatch_rot_amax(const hq::Params& p, bool bf16, bool strided, bool write_y,
                            hq_stream s) {
  if constexpr (G <= 16) {
    if (HQ_PASS1_STREAM && !strided && !write_y && aligned(p.x, 32))
      return bf16 ? launch(hq::k_rot_amax_stream<G, true>, p, s, 0, p.sync != nullptr)
                  : launch(hq::k_rot_amax_stream<G, false>, p, s, 0, p.sync != nullptr);
  }
  constexpr int kMode = HQ_PASS1_MODE;
  if (bf16)
    return strided ? launch_rot_amax<G, true, hq::kLoadStrided>(p, write_y, s)
                   : launch_rot_amax<G, true, kMode>(p, write_y, s);
  return strided ? launch_rot_amax<G, false, hq::kLoadStrided>(p, write_y, s)
                 : launch_rot_amax<G, false, kMode>(p, write_y, s);
}

template <int G, bool NEXT>
hq_status dispatch_quant(const hq::Params& p, bool bf16, bool strided, hq_stream s) {
  using hq::k_rotate_quant_nvfp4;
  constexpr int kMode = HQ_PASS2_MODE;
  if constexpr (kMode == hq::kLoadTma) {
    if (p.sched != nullptr && !strided)  // tiles handed out at run time
      return bf16 ? launch(k_rotate_quant_nvfp4<G, true, kMode, NEXT, false, true>, p, s,
                           ring_bytes<HQ_PASS2_STAGES>(kMode, true), true)
                  : launch(k_rotate_quant_nvfp4<G, false, kMode, NEXT, false, true>, p, s,
                           ring_bytes<HQ_PASS2_STAGES>(kMode, false), true);
  }
  if (bf16)
    return strided ? launch(k_rotate_quant_nvfp4<G, true, hq::kLoadStrided, NEXT>, p, s, 0, true)
                   : launch(k_rotate_quant_nvfp4<G, true, kMode, NEXT>, p, s,
                            ring_bytes<HQ_PASS2_STAGES>(kMode, true), true);
  return strided ? launch(k_rotate_quant_nvfp4<G, false, hq::kLoadStrided, NEXT>, p, s, 0, true)
                 : launch(k_rotate_quant_nvfp4<G, false, kMode, NEXT>, p, s,
                          ring_bytes<HQ_PASS2_STAGES>(kMode, false), true);
}

hq_status dispatch_quant_group(const hq::Params& p, int group, bool bf16, bool strided, hq_stream s) {
  switch (group) {
    case 0: return dispatch_quant<0, false>(p, bf16, strided, s);
    case 16: return dispatch_quant<16, false>(p, bf16, strided, s);
    default: return dispatch_quant<256, false>(p, bf16, strided, s);
  }
}

// Pass 2 with swizzled scales: row-group tiles through the TMA ring, one bulk copy
// per row, so contiguous and strided rows take the same kernel.
template <int G>
hq_status dispatch_quant_swizzled(const hq::Params& p, bool bf16, hq_stream s) {
  using hq::k_rotate_quant_nvfp4;
  if (p.sched != nullptr)  // units handed out at run time
    return bf16 ? launch(k_rotate_quant_nvfp4<G, true, hq::kLoadTma, false, true, true>, p, s,
                         ring_bytes<HQ_PASS2_STAGES>(hq::kLoadTma, true))
                : launch(k_rotate_quant_nvfp4<G, false, hq::kLoadTma, false, true, true>, p, s,
                         ring_bytes<HQ_PASS2_STAGES>(hq::kLoadTma, false));
  if (bf16)
    return launch(k_rotate_quant_nvfp4<G, true, hq::kLoadTma, false, true>, p, s,
                  ring_bytes<HQ_PASS2_STAGES>(hq::kLoadTma, true));
  return launch(k_rotate_quant_nvfp4<G, false, hq::kLoadTma, false, true>, p, s,
                ring_bytes<HQ_PASS2_STAGES>(hq::kLoadTma, false));
}

}  // namespace

extern "C" {

hq_status hq_rot_amax(const void* x, hq_dtype dtype, int64_t M, int64_t K, int64_t ldx,
                      int group, float* amax, float* y, hq_stream stream) {
  hq_status st = check_x(x, dtype, M, K, ldx, group);
  if (st != HQ_OK) return st;
  if (!amax) return HQ_ERR_NULL;
  if (!aligned(amax, 4) || (y && !aligned(y, 16))) return HQ_ERR_ALIGN;
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  if (M == 0 || K == 0) return HQ_OK;
  hq::Params p = base_params(x, dtype, M, K, ldx);
  p.amax_out = amax;
  p.y = y;
  const bool bf16 = dtype == HQ_BF16;
  const bool strided = is_strided(M, K, ldx);
  switch (group) {
    case 0: return dispatch_rot_amax<0>(p, bf16, strided, y != nullptr, stream);
    case 16: return dispatch_rot_amax<16>(p, bf16, strided, y != nullptr, stream);
    default: return dispatch_rot_amax<256>(p, bf16, strided, y != nullptr, stream);
  }
}

hq_status hq_rotate_quant_nvfp4_ws(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                   int64_t ldx, int group, const float* amax, uint8_t* q,
                                   uint8_t* scales, float* s_global, uint32_t* workspace,
                                   hq_stream stream) {
  hq_status st = check_x(x, dtype, M, K, ldx, group);
  if (st != HQ_OK) return st;
  if (workspace && !aligned(workspace, 4)) return HQ_ERR_ALIGN;
  if (M == 0 || K == 0) return HQ_OK;
  if (!amax || !q || !scales) return HQ_ERR_NULL;
  if (!aligned(amax, 4) || !aligned(q, 16) || !aligned(scales, 4) ||
      (s_global && !aligned(s_global, 4)))
    return HQ_ERR_ALIGN;
  hq::Params p = base_params(x, dtype, M, K, ldx);
  p.amax_in = amax;
  p.q = q;
  p.s = scales;
  p.sglobal_out = s_global;
  if (schedulable(p, workspace, is_strided(M, K, ldx))) {
    p.sched = workspace + kSchedWord;
    p.sched_done = workspace + 3;
  }
  const bool bf16 = dtype == HQ_BF16;
  const bool strided = is_strided(M, K, ldx);
  switch (group) {
    case 0: return dispatch_quant<0, false>(p, bf16, strided, stream);
    case 16: return dispatch_quant<16, false>(p, bf16, strided, stream);
    default: return dispatch_quant<256, false>(p, bf16, strided, stream);
  }
}

hq_status hq_rotate_quant_nvfp4(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                int64_t ldx, int group, const float* amax, uint8_t* q,
                                uint8_t* scales, float* s_global, hq_stream stream) {
  return hq_rotate_quant_nvfp4_ws(x, dtype, M, K, ldx, group, amax, q, scales, s_global, nullptr,
                                  stream);
}

hq_status hq_quantize_nvfp4(const void* x, hq_dtype dtype, int64_t M, int64_t K, int64_t ldx,
                            int group, float* amax, uint8_t* q, uint8_t* scales,
                            float* s_global, uint32_t* workspace, hq_stream stream) {
  hq_status st = check_x(x, dtype, M, K, ldx, group);
  if (st != HQ_OK) return st;
  if (!amax) return HQ_ERR_NULL;
  if (!aligned(amax, 4) || (workspace && !aligned(workspace, 4))) return HQ_ERR_ALIGN;
  // Every argument is checked before pass 1 is enqueued.
  if (M > 0 && K > 0) {
    if (!q || !scales) return HQ_ERR_NULL;
    if (!aligned(q, 16) || !aligned(scales, 4) || (s_global && !aligned(s_global, 4)))
      return HQ_ERR_ALIGN;
  }
  if (!workspace || M == 0 || K == 0) {
    st = hq_rot_amax(x, dtype, M, K, ldx, group, amax, nullptr, stream);
    if (st != HQ_OK) return st;
    return hq_rotate_quant_nvfp4(x, dtype, M, K, ldx, group, amax, q, scales, s_global, stream);
  }
  const bool bf16 = dtype == HQ_BF16;
  const bool strided = is_strided(M, K, ldx);
  // Pass 1 reduces into the workspace (0 on entry) and its last CTA writes *amax, so no
  // memset separates it from the kernel before it: it is launched as a programmatic
  // dependent and waits for that kernel's completion before it reads x.
  hq::Params p1 = base_params(x, dtype, M, K, ldx);
  p1.amax_out = reinterpret_cast<float*>(workspace + 1);
  p1.sync = workspace;
  p1.amax_copy = amax;
  switch (group) {
    case 0: st = dispatch_rot_amax<0>(p1, bf16, strided, false, stream); break;
    case 16: st = dispatch_rot_amax<16>(p1, bf16, strided, false, stream); break;
    default: st = dispatch_rot_amax<256>(p1, bf16, strided, false, stream); break;
  }
  if (st != HQ_OK) return st;
  // Pass 2 as hq_rotate_quant_nvfp4_ws; since pass 1 released it only after waiting for x's
  // producer, it fetches its first tiles of x before it waits for pass 1.
  hq::Params p = base_params(x, dtype, M, K, ldx);
  p.amax_in = amax;
  p.q = q;
  p.s = scales;
  p.sglobal_out = s_global;
  if (schedulable(p, workspace, strided)) {
    p.sched = workspace + kSchedWord;
    p.sched_done = workspace + 3;
  }
  p.x_ready = 1;
  return dispatch_quant_group(p, group, bf16, strided, stream);
}

int64_t hq_swizzled_scales_bytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0 || K % 16 != 0) return -1;
  const int64_t row_tiles = M / 128 + (M % 128 != 0);
  const int64_t cols = (K / 16 + 3) / 4 * 4;
  if (cols > 0 && row_tiles > INT64_MAX / 128 / cols) return -1;
  return row_tiles * 128 * cols;
}

hq_status hq_rotate_quant_nvfp4_swizzled_ws(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                            int64_t ldx, int group, const float* amax, uint8_t* q,
                                            uint8_t* scales, float* s_global, uint32_t* workspace,
                                            hq_stream stream) {
  hq_status st = check_x(x, dtype, M, K, ldx, group);
  if (st != HQ_OK) return st;
  if (workspace && !aligned(workspace, 4)) return HQ_ERR_ALIGN;
  if (M == 0 || K == 0) return HQ_OK;
  if (!amax || !q || !scales) return HQ_ERR_NULL;
  if (!aligned(amax, 4) || !aligned(q, 16) || !aligned(scales, 32) ||
      (s_global && !aligned(s_global, 4)))
    return HQ_ERR_ALIGN;
  hq::Params p = base_params(x, dtype, M, K, ldx);
  p.amax_in = amax;
  p.q = q;
  p.s = scales;
  p.sglobal_out = s_global;
  // Row-group units: 16 per 128-row tile and column chunk of 128 blocks, 8 tiles each.
  p.rows = static_cast<uint64_t>(M);
  const uint64_t n_cc = (static_cast<uint64_t>(K / 16) + hq::kTileBlocks - 1) / hq::kTileBlocks;
  const uint64_t n_units = static_cast<uint64_t>((M + 127) / 128) * 16u * n_cc;
  if (n_units > 0x1FFFFFFFull) return HQ_ERR_SHAPE;
  const uint64_t n_tiles = n_units * 8u;
  p.n_cc = static_cast<uint32_t>(n_cc);
  p.div_ncc = make_fast_div(p.n_cc);
  p.n_tiles = n_tiles;
  p.swz_col_tiles = static_cast<uint64_t>((K / 16 + 3) / 4);
  if (schedulable(p, workspace, false)) {  // every row is its own copy: strided rows too
    p.sched = workspace + kSchedWord;
    p.sched_done = workspace + 3;
  }
  const bool bf16 = dtype == HQ_BF16;
  switch (group) {
    case 0: return dispatch_quant_swizzled<0>(p, bf16, stream);
    case 16: return dispatch_quant_swizzled<16>(p, bf16, stream);
    default: return dispatch_quant_swizzled<256>(p, bf16, stream);
  }
}

hq_status hq_rotate_quant_nvfp4_swizzled(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                         int64_t ldx, int group, const float* amax, uint8_t* q,
                                         uint8_t* scales, float* s_global, hq_stream stream) {
  return hq_rotate_quant_nvfp4_swizzled_ws(x, dtype, M, K, ldx, group, amax, q, scales, s_global,
                                           nullptr, stream);
}

hq_status hq_rotate_quant_nvfp4_delayed_ws(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                           int64_t ldx, int group, const float* amax_prev,
                                           float* amax_next, uint8_t* q, uint8_t* scales,
                                           float* s_global, uint32_t* workspace, hq_stream stream) {
  hq_status st = check_x(x, dtype, M, K, ldx, group);
  if (st != HQ_OK) return st;
  if (!amax_next) return HQ_ERR_NULL;
  if (!aligned(amax_next, 4) || (workspace && !aligned(workspace, 4))) return HQ_ERR_ALIGN;
  if (M > 0 && K > 0) {
    if (!amax_prev || !q || !scales) return HQ_ERR_NULL;
    if (amax_prev == amax_next) return HQ_ERR_ALIAS;
    if (!aligned(amax_prev, 4) || !aligned(q, 16) || !aligned(scales, 4) ||
        (s_global && !aligned(s_global, 4)))
      return HQ_ERR_ALIGN;
  }
  if (M == 0 || K == 0 || !workspace) {
    cudaError_t e = cudaMemsetAsync(amax_next, 0, sizeof(float), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    if (M == 0 || K == 0) return HQ_OK;
  }
  hq::Params p = base_params(x, dtype, M, K, ldx);
  p.amax_in = amax_prev;
  p.amax_out = amax_next;
  p.q = q;
  p.s = scales;
  p.sglobal_out = s_global;
  const bool bf16 = dtype == HQ_BF16;
  const bool strided = is_strided(M, K, ldx);
  if (workspace) {  // the next amax reduced into word 1, the last CTA moves it to *amax_next
    p.amax_out = reinterpret_cast<float*>(workspace + 1);
    p.sync = workspace;
    p.amax_copy = amax_next;
    if (schedulable(p, workspace, strided)) {
      p.sched = workspace + kSchedWord;
      p.sched_done = workspace + 3;
    }
  }
  switch (group) {
    case 0: return dispatch_quant<0, true>(p, bf16, strided, stream);
    case 16: return dispatch_quant<16, true>(p, bf16, strided, stream);
    default: return dispatch_quant<256, true>(p, bf16, strided, stream);
  }
}

hq_status hq_rotate_quant_nvfp4_delayed(const void* x, hq_dtype dtype, int64_t M, int64_t K,
                                        int64_t ldx, int group, const float* amax_prev,
                                        float* amax_next, uint8_t* q, uint8_t* scales,
                                        float* s_global, hq_stream stream) {
  return hq_rotate_quant_nvfp4_delayed_ws(x, dtype, M, K, ldx, group, amax_prev, amax_next, q, scales,
                                          s_global, nullptr, stream);
}

hq_status hq_dequant_nvfp4(const uint8_t* q, const uint8_t* scales, const float* s_global,
                           int64_t M, int64_t K, int group, int unrotate, float* out,
                           hq_stream stream) {
  if (unrotate && group != 16 && group != 256) return HQ_ERR_GROUP;
  if (!unrotate && group != 0 && group != 16 && group != 256) return HQ_ERR_GROUP;
  if (M < 0 || K < 0) return HQ_ERR_SHAPE;
  const int64_t unit = (unrotate && group > 16) ? group : 16;
  if (K % unit != 0) return HQ_ERR_SHAPE;
  if (K > 0 && M > INT64_MAX / K) return HQ_ERR_SHAPE;
  if (M == 0 || K == 0) return HQ_OK;
  if (!q || !scales || !s_global || !out) return HQ_ERR_NULL;
  if (!aligned(q, 8) || !aligned(s_global, 4) || !aligned(out, 16)) return HQ_ERR_ALIGN;
  hq::Params p = {};
  p.nb = static_cast<uint64_t>(M) * static_cast<uint64_t>(K / 16);
  p.n_tiles = (p.nb + hq::kTileBlocks - 1) / hq::kTileBlocks;
  p.dq_q = q;
  p.dq_s = scales;
  p.dq_sglobal = s_global;
  p.dq_out = out;
  const int g = unrotate ? group : 0;
  switch (g) {
    case 0: return launch(hq::k_dequant_nvfp4<0, false>, p, stream);
    case 16: return launch(hq::k_dequant_nvfp4<16, false>, p, stream);
    default: return launch(hq::k_dequant_nvfp4<256, false>, p, stream);
  }
}

hq_status hq_rotate_quant_mxfp4_ws(const void* x, hq_dtype dtype, int64_t M, int64_t K, int64_t ldx,
                                   int group, uint8_t* q, uint8_t* scales, uint32_t* workspace,
                                   hq_stream stream) {
  hq_status st = check_x(x, dtype, M, K, ldx, group);
  if (st != HQ_OK) return st;
  if (K % 32 != 0) return HQ_ERR_SHAPE;
  if (workspace && !aligned(workspace, 4)) return HQ_ERR_ALIGN;
  if (M == 0 || K == 0) return HQ_OK;
  if (!q || !scales) return HQ_ERR_NULL;
  if (!aligned(q, 16)) return HQ_ERR_ALIGN;
  hq::Params p = base_params(x, dtype, M, K, ldx);
  p.q = q;
  p.s = scales;
  const bool bf16 = dtype == HQ_BF16;
  const bool strided = is_strided(M, K, ldx);
  if (schedulable(p, workspace, strided)) {
    p.sched = workspace + kSchedWord;
    p.sched_done = workspace + 3;
  }
  using hq::k_rotate_quant_mxfp4;
  constexpr int kMode = HQ_PASS2_MODE;
  // programmatic dependent launch; contiguous rows through the TMA ring take the run-time
  // split when the workspace allows it
  auto go = [&](auto k_strided, auto k_flat, auto k_dyn, size_t smem) {
    if (strided) return launch(k_strided, p, stream, 0, true);
    if (kMode == hq::kLoadTma && p.sched != nullptr) return launch(k_dyn, p, stream, smem, true);
    return launch(k_flat, p, stream, smem, true);
  };
  const size_t smem = bf16 ? ring_bytes<HQ_PASS2_STAGES>(kMode, true) : ring_bytes<HQ_PASS2_STAGES>(kMode, false);
  switch (group) {
    case 0:
      return bf16 ? go(k_rotate_quant_mxfp4<0, true, hq::kLoadStrided>, k_rotate_quant_mxfp4<0, true, kMode>,
                       k_rotate_quant_mxfp4<0, true, hq::kLoadTma, true>, smem)
                  : go(k_rotate_quant_mxfp4<0, false, hq::kLoadStrided>, k_rotate_quant_mxfp4<0, false, kMode>,
                       k_rotate_quant_mxfp4<0, false, hq::kLoadTma, true>, smem);
    case 16:
      return bf16 ? go(k_rotate_quant_mxfp4<16, true, hq::kLoadStrided>, k_rotate_quant_mxfp4<16, true, kMode>,
                       k_rotate_quant_mxfp4<16, true, hq::kLoadTma, true>, smem)
                  : go(k_rotate_quant_mxfp4<16, false, hq::kLoadStrided>, k_rotate_quant_mxfp4<16, false, kMode>,
                       k_rotate_quant_mxfp4<16, false, hq::kLoadTma, true>, smem);
    default:
      return bf16 ? go(k_rotate_quant_mxfp4<256, true, hq::kLoadStrided>, k_rotate_quant_mxfp4<256, true, kMode>,
                       k_rotate_quant_mxfp4<256, true, hq::kLoadTma, true>, smem)
                  : go(k_rotate_quant_mxfp4<256, false, hq::kLoadStrided>, k_rotate_quant_mxfp4<256, false, kMode>,
                       k_rotate_quant_mxfp4<256, false, hq::kLoadTma, true>, smem);
  }
}

hq_status hq_rotate_quant_mxfp4(const void* x, hq_dtype dtype, int64_t M, int64_t K, int64_t ldx,
                                int group, uint8_t* q, uint8_t* scales, hq_stream stream) {
  return hq_rotate_quant_mxfp4_ws(x, dtype, M, K, ldx, group, q, scales, nullptr, stream);
}

hq_status hq_dequant_mxfp4(const uint8_t* q, const uint8_t* scales, int64_t M, int64_t K,
                           int group, int unrotate, float* out, hq_stream stream) {
  if (unrotate && group != 16 && group != 256) return HQ_ERR_GROUP;
  if (!unrotate && group != 0 && group != 16 && group != 256) return HQ_ERR_GROUP;
  if (M < 0 || K < 0 || K % 32 != 0) return HQ_ERR_SHAPE;
  if (unrotate && K % group != 0) return HQ_ERR_SHAPE;
  if (K > 0 && M > INT64_MAX / K) return HQ_ERR_SHAPE;
  if (M == 0 || K == 0) return HQ_OK;
  if (!q || !scales || !out) return HQ_ERR_NULL;
  if (!aligned(q, 8) || !aligned(out, 16)) return HQ_ERR_ALIGN;
  hq::Params p = {};
  p.nb = static_cast<uint64_t>(M) * static_cast<uint64_t>(K / 16);
  p.n_tiles = (p.nb + hq::kTileBlocks - 1) / hq::kTileBlocks;
  p.dq_q = q;
  p.dq_s = scales;
  p.dq_out = out;
  switch (unrotate ? group : 0) {
    case 0: return launch(hq::k_dequant_nvfp4<0, true>, p, stream);
    case 16: return launch(hq::k_dequant_nvfp4<16, true>, p, stream);
    default: return launch(hq::k_dequant_nvfp4<256, true>, p, stream);
  }
}

const char* hq_status_string(hq_status status) {
  switch (status) {
    case HQ_OK: return "HQ_OK";
    case HQ_ERR_NULL: return "HQ_ERR_NULL: a required pointer is NULL";
    case HQ_ERR_SHAPE: return "HQ_ERR_SHAPE: bad M, K or ldx";
    case HQ_ERR_ALIGN: return "HQ_ERR_ALIGN: pointer or row stride misaligned";
    case HQ_ERR_DTYPE: return "HQ_ERR_DTYPE: unknown element type";
    case HQ_ERR_GROUP: return "HQ_ERR_GROUP: rotation group must be 0, 16 or 256";
    case HQ_ERR_CUDA: return "HQ_ERR_CUDA: CUDA runtime error";
    case HQ_ERR_TOO_LARGE:
      return "HQ_ERR_TOO_LARGE: tensor exceeds the fixed scratch of the allocation-free entry point";
    case HQ_ERR_ALIAS: return "HQ_ERR_ALIAS: two buffers that must be distinct are the same";
  }
  return "unknown hq_status";
}

int hq_last_cuda_error(void) { return g_last_cuda_error; }

hq_status hq_read_fault(unsigned int* fault, int clear) {
  if (!fault) return HQ_ERR_NULL;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpyFromSymbol(fault, g_hq_fault, sizeof(unsigned int));
  if (e != cudaSuccess) return cuda_fail(e);
  if (clear && *fault) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_hq_fault, &zero, sizeof(unsigned int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  unsigned int int8_word = 0;  // the int8 kernels' copy (hq_int8.cu)
  e = hq::int8_fault_word(&int8_word, clear != 0);
  if (e != cudaSuccess) return cuda_fail(e);
  *fault |= int8_word;
  return HQ_OK;
}

hq_status hq_selftest_bounded_wait(int unit, hq_stream stream) {
  if (unit < 0 || unit > 1) return HQ_ERR_SHAPE;
  if (unit == 1) {
    const cudaError_t e = hq::int8_selftest_bounded_wait(static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? HQ_OK : cuda_fail(e);
  }
  hq::k_selftest_bounded_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? HQ_OK : cuda_fail(e);
}

int hq_version(void) { return 100; }

}  // extern "C"
