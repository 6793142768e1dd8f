// hq_kernels.cuh -- device code of libhq (sm_103a).
//
// The kernels of the fused Hadamard rotation + NVFP4 quantization ("A Fused
// Hadamard + NVFP4 Quantization Kernel in Triton", §1 "The format, precisely" and
// §2 "The kernel"):
//
//   k_rot_amax_stream     pass 1 for G <= 16 on contiguous rows: stream x, rotate,
//                         reduce max |y| into one float.
//   k_rot_amax            pass 1 in tiles (G = 256, strided rows, or a rotated output).
//   k_rotate_quant_nvfp4  pass 2: stream x once, rotate in registers, block amax,
//                         E4M3 block scale, E2M1 codes, write codes + scales once.
//   k_rotate_quant_mxfp4  MXFP4 (E8M0 scale per 32 values), one pass.
//   k_dequant_nvfp4       round trip: codes * scales, optional inverse rotation.
//
// Work decomposition.  A warp owns a "tile" of 128 NVFP4 blocks (2048 elements,
// 4 KB of bf16); each lane holds 4 whole blocks (64 values) in registers.  Which
// 4 blocks a lane holds depends on the rotation group:
//   G <= 16 : block 32*j + lane of the tile (j = 0..3);
//   G == 256: the 4 lanes of a quad hold the 16 blocks of one 256-group.  In the
//             plain layout (dequant) block 16*(lane/4) + (lane%4)
//             + 4*j: index bits 4,5 of the group are the lane bits, bits 6,7 the
//             register block j.  Pass 1, pass 2 (all its forms) and MXFP4 use exchange layouts
//             (slot_block) in which each cross-lane stage moves half of the values.
// The 64 values sit in float2 pairs (block 0 with block 1, block 2 with block 3)
// so the butterfly and the division run on the packed fp32x2 pipe of sm_100-
// family parts (FADD2/FFMA2/FMUL2): one instruction per two values.
//
// Data movement.  When the rows of x are back to back (the normal case) every
// warp runs its own TMA pipeline: a ring of kStages tile slots in shared memory,
// each filled by one cp.async.bulk global->shared copy that completes on the
// slot's mbarrier.  A warp keeps kStages tiles in flight while it computes
// (pass 1: 16 warps x 3 x 4 KB = 192 KB per SM, pass 2: 16 warps x 2 x 4 KB)
// without spending registers on them.  Strided rows (ldx != K) load directly into
// registers (LoadMode below).
// Every mbarrier wait is bounded (about one second of %globaltimer); a wait that
// runs out records kFaultWaitTimeout in g_hq_fault, waits (bounded) for the
// warp's copies still in flight and leaves the loop, so nothing can hang.
//
// Launch order.  Pass 2 and MXFP4 are launched as programmatic dependents of the
// kernel before them on the stream, and so is pass 1 when hq_quantize_nvfp4 passes
// it a workspace: each executes griddepcontrol.wait before it touches global memory,
// which waits for that kernel to complete.  The pass-1 kernels execute
// griddepcontrol.launch_dependents as they start, so pass 2's grid is launched while
// pass 1 runs and its CTAs start as pass 1's leave the SMs.
//
// Bit-exactness.  The butterfly performs the stages h = 1, 2, 4, 8 (inside a
// block), then for G = 256 h = 16, 32, 64, 128 (across blocks: in registers, or
// across the quad's lanes), each stage an fp32 add/sub with one rounding, exactly
// as the definition.  The final multiply by 1/sqrt(G) is folded into the division
// (see k_rotate_quant_nvfp4); that fold is exact on the fast path's domain, and the
// slow path evaluates the definition literally.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hq {

constexpr int kThreads = 256;            // 8 warps per CTA
constexpr int kWarpsPerCta = kThreads / 32;
constexpr int kBlocksPerLane = 4;
constexpr int kTileBlocks = 32 * kBlocksPerLane;  // 128 NVFP4 blocks per warp tile

// Dynamic tile schedule: tile t belongs to class t % kSchedClasses, and warp w of every CTA
// takes the tiles of class w from that class's counter.  The counters sit a 128-byte line
// apart so that the atomic traffic of different classes does not meet at one address.
constexpr int kSchedClasses = kWarpsPerCta;
constexpr int kSchedStrideWords = 32;
static_assert(kSchedClasses == kThreads / 32, "one class per warp of a CTA");

// Fault bits recorded by the kernels (read back with hq_read_fault()).
constexpr unsigned kFaultWaitTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // one second

}  // namespace hq

// Device-side fault word.  The library is compiled without relocatable device
// code, so every translation unit that includes this header has its own copy
// (one per device that loads the library); hq_read_fault() combines them.
__device__ unsigned int g_hq_fault;

namespace hq {

// ---------------------------------------------------------------------------
// Unsigned 32-bit division by an invariant divisor with one multiply-high:
// Granlund & Montgomery, "Division by Invariant Integers using Multiplication"
// (PLDI 1994), Figure 4.1.  Used only for strided rows (ldx != K).
// ---------------------------------------------------------------------------
struct FastDiv {
  uint32_t m;
  uint32_t s1;
  uint32_t s2;
};

__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

struct Params {
  const uint8_t* x;        // input, bytes
  int64_t ldx_bytes;       // row stride of x in bytes
  uint64_t nb;             // number of 16-element blocks, M*K/16
  uint32_t nbr;            // blocks per row, K/16
  FastDiv div_nbr;         // divider for nbr (valid when nb < 2^32)
  uint64_t n_tiles;        // ceil(nb / kTileBlocks)
  // pass 1
  float* amax_out;         // atomically max-reduced (zeroed by the host call, or a workspace word)
  float* y;                // optional fp32 rotated output [M, K]
  // pass 2
  const float* amax_in;
  uint8_t* q;              // [M, K/2]
  uint8_t* s;              // [M, K/16], or the swizzled tile layout (swz_col_tiles > 0)
  float* sglobal_out;      // optional
  uint64_t swz_col_tiles;  // swizzled scales: ceil(K/64) tiles of 4 scale columns per tile row
  uint64_t rows;           // M (row-group tiles)
  uint32_t n_cc;           // row-group tiles: column chunks of 16 blocks per row, ceil(K/256)
  FastDiv div_ncc;         // divider for n_cc
  // pass 1 with a workspace (hq_quantize_nvfp4)
  unsigned* sync;          // [1] amax bits, [2] CTAs done; 0 on entry and exit
  float* amax_copy;        // the tensor's amax, written by the last CTA
  // run-time tile split (for_each_tile, DYN): kSchedClasses counters kSchedStrideWords apart
  // and the count of warps done with them, all 0 on entry and put back to 0 by the last warp
  unsigned* sched;
  unsigned* sched_done;
  int x_ready;             // pass 2: x is complete at launch (the pass 1 before it waited for
                           // x's producer before releasing it), so tiles may be fetched before
                           // griddepcontrol.wait
  // dequant
  const uint8_t* dq_q;
  const uint8_t* dq_s;
  const float* dq_sglobal;
  float* dq_out;
};

// ---------------------------------------------------------------------------
// Packed fp32x2 helpers (round to nearest even, one rounding per lane).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// a - b with one rounding per lane (the packed subtract: two register pairs read, where the
// fma form RN(b * -1 + a) read three; bf16 [32768, 28672] pass 2: 351.4 -> 348.4 us).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  const unsigned long long ra = *reinterpret_cast<unsigned long long*>(&a);
  const unsigned long long rb = *reinterpret_cast<unsigned long long*>(&b);
  unsigned long long rd;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2*>(&rd);
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// max that keeps a NaN once seen (so a non-finite input surfaces in amax).
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// Three-input max that keeps a NaN (sm_100 family).
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// max |v[i]| over 16 values (the .x or .y lane of each pair), exact; NaN if any is NaN.
template <bool Y>
__device__ __forceinline__ float block_absmax(const float2 (&v)[16]) {
  auto g = [&](int i) { return fabsf(Y ? v[i].y : v[i].x); };
  float m = max3_nan(g(0), g(1), g(2));
#pragma unroll
  for (int i = 3; i < 15; i += 2) m = max3_nan(m, g(i), g(i + 1));
  return max_nan(m, g(15));
}

// max over the CTA of each thread's `v`, then one atomicMax into *out.  Non-negative
// floats (and NaN, with the sign bit clear) order like their bit patterns as unsigned
// integers.  Every thread of the CTA must call this.
// With `count` (pass 1 of hq_quantize_nvfp4 with a workspace): *out is a workspace word
// that is 0 on entry; each CTA counts itself out in *count after its atomicMax, and the
// last one moves the tensor's amax to *final_out and puts both words back to 0.  No
// memset then precedes the launch.
__device__ __forceinline__ void cta_amax_to_global(float v, float* out, unsigned* count = nullptr,
                                                   float* final_out = nullptr) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = max_nan(v, __shfl_xor_sync(0xFFFFFFFFu, v, m));
  __shared__ float red[kWarpsPerCta];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = red[0];
#pragma unroll
    for (int w = 1; w < kWarpsPerCta; ++w) m = max_nan(m, red[w]);
    atomicMax(reinterpret_cast<unsigned int*>(out), __float_as_uint(m));
    if (count) {
      __threadfence();
      if (atomicAdd(count, 1u) == gridDim.x - 1) {
        __threadfence();
        *final_out = __uint_as_float(atomicExch(reinterpret_cast<unsigned int*>(out), 0u));
        atomicExch(count, 0u);
      }
    }
  }
}

// a / b rounded to nearest even from r = RN(1/b), by Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(a r), e = a - q0 b (exact),
// q = RN(q0 + e r).  Valid while a, b, r, q0 and e stay normal.
__device__ __forceinline__ float div_markstein(float a, float b, float r) {
  const float q0 = __fmul_rn(a, r);
  const float e = __fmaf_rn(-q0, b, a);
  return __fmaf_rn(e, r, q0);
}

// ---------------------------------------------------------------------------
// Conversions.
// ---------------------------------------------------------------------------
// Eight fp32 quotients -> eight E2M1 codes packed in a u32, element 0 in the
// lowest nibble.  cvt.rn.satfinite.e2m1x2.f32 d, a, b puts a in the high
// nibble of d and b in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8(float q0, float q1, float q2, float q3, float q4,
                                           float q5, float q6, float q7) {
  uint32_t r;
  asm("{\n\t.reg .b8 %%hq_b0, %%hq_b1, %%hq_b2, %%hq_b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 %%hq_b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 %%hq_b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 %%hq_b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 %%hq_b3, %8, %7;\n\t"
      "mov.b32 %0, {%%hq_b0, %%hq_b1, %%hq_b2, %%hq_b3};\n\t}"
      : "=r"(r)
      : "f"(q0), "f"(q1), "f"(q2), "f"(q3), "f"(q4), "f"(q5), "f"(q6), "f"(q7));
  return r;
}

// Two non-negative fp32 -> two E4M3 patterns (round to nearest even, saturate
// at 448); lo in bits 0..7, hi in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 patterns (lo in bits 0..7) -> their exact fp32 values.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t two) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(two);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Two E2M1 codes (one byte, element 0 in the low nibble) -> exact fp32 values.
__device__ __forceinline__ float2 e2m1x2_to_f32(uint32_t byte) {
  uint32_t h2;
  const uint16_t in = static_cast<uint16_t>(byte & 0xFF);
  asm("{\n\t.reg .b8 %%hq_t;\n\tcvt.u8.u16 %%hq_t, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, %%hq_t;\n\t}"
      : "=r"(h2)
      : "h"(in));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// ---------------------------------------------------------------------------
// TMA bulk copies and mbarriers (inline PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared accesses (and those it has
// synchronised with) before later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// x is streamed once: its lines are the first to leave L2.
__device__ __forceinline__ uint64_t l2_stream_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory, completing `bytes` transactions on `bar`.
__device__ __forceinline__ void tma_load(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 32 bytes to global memory in one 256-bit store (32-byte aligned address).
__device__ __forceinline__ void st_v8(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                      uint32_t e, uint32_t f, uint32_t g, uint32_t h) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a), "r"(b),
               "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
               : "memory");
}

// Arrive on `bar` announcing `bytes` of copies to come (0: a plain arrive).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with parity `parity` to complete.  Gives up after
// about kWaitLimitNs and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((i & 15u) == 0) {
      const uint64_t now = global_timer_ns();
      if (i == 0)
        t0 = now;
      else if (now - t0 > kWaitLimitNs)
        return false;
    }
  }
}

// ---------------------------------------------------------------------------
// Tile geometry.
// ---------------------------------------------------------------------------
template <int G>
__device__ __forceinline__ uint32_t lane_block(int lane, int j) {
  if constexpr (G == 256) {
    return static_cast<uint32_t>((lane >> 2) * 16 + (lane & 3) + 4 * j);
  } else {
    return static_cast<uint32_t>(32 * j + lane);
  }
}

template <bool STRIDED>
__device__ __forceinline__ const uint8_t* block_ptr(const Params& p, uint64_t b, int es) {
  if constexpr (STRIDED) {
    uint64_t row, col;
    if (p.nb <= 0xFFFFFFFFull) {
      row = fast_div(static_cast<uint32_t>(b), p.div_nbr);
    } else {
      row = b / p.nbr;
    }
    col = b - row * p.nbr;
    return p.x + row * static_cast<uint64_t>(p.ldx_bytes) + col * 16u * es;
  } else {
    return p.x + b * 16u * es;
  }
}

// Widen 16 elements (bf16 -> fp32 is exact: the bf16 bits are the top half).
template <bool BF16>
__device__ __forceinline__ void widen(const uint4* w4, float (&f)[16]) {
  if constexpr (BF16) {
    const uint32_t w[8] = {w4[0].x, w4[0].y, w4[0].z, w4[0].w, w4[1].x, w4[1].y, w4[1].z, w4[1].w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[4 * k + 0] = __uint_as_float(w4[k].x);
      f[4 * k + 1] = __uint_as_float(w4[k].y);
      f[4 * k + 2] = __uint_as_float(w4[k].z);
      f[4 * k + 3] = __uint_as_float(w4[k].w);
    }
  }
}

// Widen 16 bf16 values and apply the butterfly's first stage (h = 1) on the way:
// (x[2m], x[2m + 1]) -> (x[2m] + x[2m + 1], x[2m] - x[2m + 1]).  Each output is one
// mixed-precision add or subtract (sm_100 family): the bf16 operand is widened
// exactly and the fp32 result rounded once, so it equals the stage on the widened
// values bit for bit.  x[2m + 1] is the word's top half, which is already its fp32
// pattern with the low half cleared.
__device__ __forceinline__ void widen_stage1_bf16(const uint4* w4, float (&f)[16]) {
  const uint32_t w[8] = {w4[0].x, w4[0].y, w4[0].z, w4[0].w, w4[1].x, w4[1].y, w4[1].z, w4[1].w};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float hi = __uint_as_float(w[k] & 0xFFFF0000u);
    asm("{\n\t.reg .b16 %%hq_lo, %%hq_hi;\n\t"
        "mov.b32 {%%hq_lo, %%hq_hi}, %2;\n\t"
        "add.rn.f32.bf16 %0, %%hq_lo, %3;\n\t"
        "sub.rn.f32.bf16 %1, %%hq_lo, %3;\n\t}"
        : "=f"(f[2 * k]), "=f"(f[2 * k + 1])
        : "r"(w[k]), "f"(hi));
  }
}

// widen, or widen plus the first butterfly stage (S1, bf16 only).
template <bool BF16, bool S1>
__device__ __forceinline__ void widen_s(const uint4* w4, float (&f)[16]) {
  if constexpr (BF16 && S1)
    widen_stage1_bf16(w4, f);
  else
    widen<BF16>(w4, f);
}

// The lane's 4 blocks as two float2 arrays: P[0][i] = (blk0[i], blk1[i]),
// P[1][i] = (blk2[i], blk3[i]).
struct Lane4 {
  float2 P[2][16];
};

__device__ __forceinline__ void put_block(Lane4& t, int j, const float (&f)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    if (j & 1)
      t.P[j >> 1][i].y = f[i];
    else
      t.P[j >> 1][i].x = f[i];
  }
}

// The tile block held in register slot s of a lane (slot s is P[s >> 1], component
// s & 1), and whether its two halves (positions 0..7 and 8..15) sit swapped.
//   ORDER 0: slot j holds block lane_block<G>(lane, j), halves in place.
//   ORDER 1 (pass 1 of the 256-group, see absmax256_x): lane l of quad q = l / 4
//   (the tile's 256-group q), with A = l & 1 and B = (l >> 1) & 1, holds the four
//   blocks of the group whose block-index bits 0 and 2 are A and B: slot 2k + c holds
//   block A + 2 (k ^ B) + 4 B + 8 c of the group, its halves swapped when
//   A ^ (q & 1) = 1.  (Within a warp, each 16-byte shared-memory load then covers
//   all eight 16-byte columns of a 128-byte row: no bank conflict for bf16.)
//   ORDER 2 (pass 2 of the 256-group, see rotate_tile_x256): lane l of quad q with
//   a = l & 1 and b = (l >> 1) & 1 holds, in slot 2k + c, block
//   (k ^ a) + 2 (a ^ b) + 4 c + 8 b of group q as loaded, and block
//   a + 2 (a ^ b) + 4 c + 8 (k ^ b) once rotated (out_block).
template <int G, int ORDER>
__device__ __forceinline__ uint32_t slot_block(int lane, int s) {
  const int a = lane & 1, b = (lane >> 1) & 1, k = s >> 1, c = s & 1;
  if constexpr (ORDER == 1) {
    return static_cast<uint32_t>((lane >> 2) * 16 + a + 2 * (k ^ b) + 4 * b + 8 * c);
  } else if constexpr (ORDER == 2) {
    return static_cast<uint32_t>((lane >> 2) * 16 + (k ^ a) + 2 * (a ^ b) + 4 * c + 8 * b);
  } else {
    return lane_block<G>(lane, s);
  }
}

// The tile block whose rotated values register slot s holds after the rotation.
template <int G, int ORDER>
__device__ __forceinline__ uint32_t out_block(int lane, int s) {
  if constexpr (ORDER == 2) {
    const int a = lane & 1, b = (lane >> 1) & 1, k = s >> 1, c = s & 1;
    return static_cast<uint32_t>((lane >> 2) * 16 + a + 2 * (a ^ b) + 4 * c + 8 * (k ^ b));
  } else {
    return slot_block<G, ORDER>(lane, s);
  }
}

template <int ORDER>
__device__ __forceinline__ bool halves_swapped(int lane) {
  return ORDER == 1 && ((lane ^ (lane >> 2)) & 1);
}

// Direct global loads (strided rows).
template <int G, bool BF16, bool STRIDED, int ORDER = 0, bool S1 = false>
__device__ __forceinline__ void load_tile_global(const Params& p, uint64_t tile_base, int lane,
                                                 bool (&valid)[4], Lane4& t) {
  constexpr int es = BF16 ? 2 : 4;
  constexpr int n16 = BF16 ? 2 : 4;
  const int hx = halves_swapped<ORDER>(lane) ? n16 / 2 : 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint64_t b = tile_base + slot_block<G, ORDER>(lane, s);
    valid[s] = b < p.nb;
    uint4 w4[n16];
    if (valid[s]) {
      const uint4* src = reinterpret_cast<const uint4*>(block_ptr<STRIDED>(p, b, es));
#pragma unroll
      for (int k = 0; k < n16; ++k) w4[k] = __ldg(src + (k ^ hx));
    } else {
#pragma unroll
      for (int k = 0; k < n16; ++k) w4[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    float f[16];
    widen_s<BF16, S1>(w4, f);
    put_block(t, s, f);
  }
}

// Loads from a tile staged in shared memory (block b of the tile at b*16*es).
// FULL: the caller knows that all kTileBlocks blocks of the tile lie inside the tensor.
template <int G, bool BF16, int ORDER = 0, bool S1 = false, bool FULL = false>
__device__ __forceinline__ void load_tile_smem(const uint8_t* slot, uint64_t tile_base, uint64_t nb,
                                               int lane, bool (&valid)[4], Lane4& t) {
  constexpr int es = BF16 ? 2 : 4;
  constexpr int n16 = BF16 ? 2 : 4;
  const int hx = halves_swapped<ORDER>(lane) ? n16 / 2 : 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t bl = slot_block<G, ORDER>(lane, s);
    valid[s] = FULL || tile_base + bl < nb;
    uint4 w4[n16];
    if (valid[s]) {
      const uint4* src = reinterpret_cast<const uint4*>(slot + bl * 16u * es);
#pragma unroll
      for (int k = 0; k < n16; ++k) w4[k] = src[k ^ hx];
    } else {
#pragma unroll
      for (int k = 0; k < n16; ++k) w4[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    float f[16];
    widen_s<BF16, S1>(w4, f);
    put_block(t, s, f);
  }
}

// Ring depth (tiles in flight per warp) and CTAs per SM.  Both passes run two
// CTAs of 8 warps per SM (16 warps); pass 1 keeps 3 tiles per warp in flight,
// pass 2, which needs more registers, 2.
#ifndef HQ_PASS1_STAGES
#define HQ_PASS1_STAGES 3
#endif
#ifndef HQ_PASS1_MIN_CTAS
#define HQ_PASS1_MIN_CTAS 2
#endif
#ifndef HQ_PASS2_STAGES
#define HQ_PASS2_STAGES 2
#endif
// Shared-memory ring geometry of the TMA pipeline.
template <bool BF16, int STAGES>
struct Ring {
  static constexpr int kElemBytes = BF16 ? 2 : 4;
  static constexpr int kTileBytes = kTileBlocks * 16 * kElemBytes;  // 4 KB / 8 KB
  // fp32 tiles are twice as large: at most 3 of them per warp (192 KB per CTA).
  static constexpr int kStages = BF16 ? STAGES : (STAGES > 3 ? 3 : STAGES);
  static constexpr int kDataBytes = kWarpsPerCta * kStages * kTileBytes;
  static constexpr int kSmemBytes = kDataBytes + kWarpsPerCta * kStages * 8;
};

// How a kernel reads x.
enum LoadMode : int {
  kLoadTma = 0,      // contiguous rows, per-warp TMA ring in shared memory
  kLoadDirect = 1,   // contiguous rows, vector loads straight into registers
  kLoadStrided = 2,  // rows ldx apart, vector loads straight into registers
};

// Row-group units (pass 2 with swizzled scales).  Unit u covers the columns
// c0 = 128 cc .. c0 + 127 (blocks) of the 8 rows 128 rt + 2 k + {0, 1, 32, 33, 64,
// 65, 96, 97}, k = 0..15: the rows whose scales of 4 consecutive columns make one
// 32-byte piece of the swizzled layout.  Its 8 tiles rs = 0..7 (one row each, as
// contiguous as a plain tile) go to one warp in order.
// Units run over column chunks fastest, then k, then row tiles rt = 0 ..
// ceil(M / 128) - 1; rows past M give empty tiles.
struct RgTile {      // 32-bit fields: the host keeps units below 2^29, so rows below 2^32
  uint32_t row;     // row of the tile (may be >= M)
  uint32_t rt;      // row tile (128 rows)
  uint32_t k;       // row pair within a 32-row band
  uint32_t c0;      // first column (block) of the chunk
  uint32_t ncols;   // blocks of the chunk inside the row: 1..128
  int rs;           // tile within the unit
  bool present;     // row < M
};


// A prologue that does nothing (for_each_tile's default).
struct NoPrologue {
  __device__ __forceinline__ void operator()() const {}
};

constexpr uint64_t kNoTile = ~uint64_t{0};

// 64-bit broadcast from lane 0.
__device__ __forceinline__ uint64_t bcast0(uint64_t v) {
  const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), 0);
  const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), 0);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// A warp of the run-time split whose class has no tile left for it (its last counter fetch
// came back past the end, or it never had a tile) counts itself out; the last warp of the grid
// to do so puts the counters and the count back to 0 for the next call.  Called by lane 0,
// once per warp, as soon as that is known: usually a tile or two before the warp's end, so
// the reset overlaps the work still in flight.  Every counter atomic of a warp has returned
// its value before the warp counts itself out, and all warps have counted themselves out
// before the reset, so no fetch of this launch can follow it.
__device__ __forceinline__ void sched_retire(const Params& p) {
  if (atomicAdd(p.sched_done, 1u) == gridDim.x * static_cast<unsigned>(kWarpsPerCta) - 1u) {
    __threadfence();
#pragma unroll
    for (int c = 0; c < kSchedClasses; ++c) atomicExch(p.sched + c * kSchedStrideWords, 0u);
    atomicExch(p.sched_done, 0u);
  }
}

// body(tile_base, lane, valid, t), compiled twice: for a tile whose blocks all lie inside the
// tensor (every tile but the last) `valid` is a constant, so the body's per-block checks and
// branches drop out of the path that runs for all other tiles.
template <typename Tile, typename Body>
__device__ __forceinline__ void call_body(bool full, const Tile& tile, int lane, bool (&valid)[4], Lane4& t,
                                          Body& body) {
  if (full) {
    bool all[4] = {true, true, true, true};
    body(tile, lane, all, t);
  } else {
    body(tile, lane, valid, t);
  }
}

// Run `body(tile_base, lane, valid, t)` over this warp's tiles with the tile's values in
// registers.
//
// Which tiles.  Fixed split (DYN false): warp w of W takes the tiles w, w + W, w + 2W, ...
// Run-time split (DYN, contiguous rows only): tile t belongs to class t % C (C =
// kSchedClasses) and warp c of every CTA serves class c, tiles c + C j.  Its first R class
// indices are fixed, j = blockIdx.x + s gridDim.x (s < R, the ring depth), so the first
// copies need no atomic; every later j is R gridDim.x + the value of an atomicAdd on the
// class counter p.sched[c * kSchedStrideWords].  Only lane 0 keeps this schedule: it reads
// the counter one tile ahead (the atomic's latency hides behind the tile in between), issues
// the copies, and the other lanes learn each tile's index from it when they read that slot,
// long after it was chosen.  Warps that run ahead take more tiles, and all warps run out of
// work within about one tile of each other.  The counters are 0 on entry, and the last warp
// to run out of tiles puts them back to 0 (sched_retire).
//
// GDC: the kernel was launched as a programmatic dependent and has not yet executed
// griddepcontrol.wait; the loop does, before its first access to global memory, or, when
// p.x_ready declares x complete, right after issuing its first tile copies.
// `pre()` runs once in every warp before the first tile is read: in the TMA form after the
// warp's first copies have been issued, so that work the tiles need (reading the amax,
// building the divisor table) overlaps their flight instead of delaying it.  Every warp of
// the CTA calls it, so it may hold a __syncthreads().
// x is read with an L2 evict-first hint (it is streamed once).  REVERSE (fixed split only):
// the k-th tile of the sequence is tile
// n_tiles - 1 - k, so the pass walks x from its end (pass 1 of the two-launch path: pass 2
// walks it from the start, and each pass then begins where the previous one ended, with
// that part of x still in L2).
template <int G, bool BF16, int MODE, int STAGES, int ORDER = 0, bool S1 = false, bool REVERSE = false,
          bool GDC = false, bool DYN = false, typename Body, typename Pre = NoPrologue>
__device__ __forceinline__ void for_each_tile(const Params& p, Body&& body, Pre&& pre = Pre()) {
  static_assert(!(DYN && (REVERSE || MODE != kLoadTma)), "run-time split: TMA ring, forward walk");
  // The 256-group's quantizing tile bodies (layout ORDER 2) are compiled a second time for
  // whole tiles (call_body); elsewhere the single form measured as fast or faster.
  constexpr bool kSplitFull = G == 256 && ORDER == 2;
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const uint64_t gw = static_cast<uint64_t>(blockIdx.x) * kWarpsPerCta + wid;
  const uint64_t nw = static_cast<uint64_t>(gridDim.x) * kWarpsPerCta;
  auto tile_of = [&](uint64_t seq) { return REVERSE ? p.n_tiles - 1 - seq : seq; };
  auto gdc_wait = []() { asm volatile("griddepcontrol.wait;" ::: "memory"); };
  if constexpr (MODE != kLoadTma) {
    if constexpr (GDC) gdc_wait();
    pre();
    for (uint64_t seq = gw; seq < p.n_tiles; seq += nw) {
      const uint64_t base = tile_of(seq) * kTileBlocks;
      bool valid[4];
      Lane4 t;
      load_tile_global<G, BF16, MODE == kLoadStrided, ORDER, S1>(p, base, lane, valid, t);
      body(base, lane, valid, t);
    }
  } else {
    using R = Ring<BF16, STAGES>;
    extern __shared__ __align__(1024) uint8_t hq_smem[];
    uint8_t* ring = hq_smem + wid * R::kStages * R::kTileBytes;
    const uint32_t ring_s = smem_addr(ring);
    const uint32_t bar0 = smem_addr(hq_smem + R::kDataBytes) + wid * R::kStages * 8;
    const uint64_t policy = l2_stream_policy();

    auto issue = [&](uint64_t seq, int slot) {
      const uint64_t first = tile_of(seq) * kTileBlocks;
      const uint64_t nblk = (p.nb - first < kTileBlocks) ? (p.nb - first) : kTileBlocks;
      tma_load(ring_s + slot * R::kTileBytes, p.x + first * 16u * R::kElemBytes,
               static_cast<uint32_t>(nblk * 16u * R::kElemBytes), bar0 + slot * 8, policy);
    };
    auto timed_out = [&](uint64_t k, uint64_t issued) {
      if (lane == 0) atomicOr(&g_hq_fault, kFaultWaitTimeout);
      for (uint64_t m = k; m < issued; ++m)
        mbar_wait(bar0 + static_cast<int>(m % R::kStages) * 8, static_cast<uint32_t>((m / R::kStages) & 1));
    };

    if (lane == 0) {
      for (int s = 0; s < R::kStages; ++s) mbar_init(bar0 + s * 8, 1);
      fence_mbar_init();
    }
    __syncwarp();
    const bool early = GDC && p.x_ready;
    if (GDC && !early) gdc_wait();

    if constexpr (!DYN) {
      uint64_t issued = 0;  // tiles of this warp handed to TMA so far
      if (lane == 0) {
        for (int s = 0; s < R::kStages; ++s)
          if (gw + s * nw < p.n_tiles) issue(gw + s * nw, s);
      }
      for (int s = 0; s < R::kStages; ++s)
        if (gw + s * nw < p.n_tiles) ++issued;
      if (early) gdc_wait();
      pre();

      uint64_t k = 0;
      for (uint64_t seq = gw; seq < p.n_tiles; seq += nw, ++k) {
        const int slot = static_cast<int>(k % R::kStages);
        const uint32_t parity = static_cast<uint32_t>((k / R::kStages) & 1);
        const bool ok = mbar_wait(bar0 + slot * 8, parity);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          timed_out(k, issued);
          return;
        }
        const uint64_t base = tile_of(seq) * kTileBlocks;
        const bool full = kSplitFull && p.nb - base >= kTileBlocks;  // the same in every lane
        bool valid[4];
        Lane4 t;
        if (full)
          load_tile_smem<G, BF16, ORDER, S1, true>(ring + slot * R::kTileBytes, base, p.nb, lane, valid, t);
        else
          load_tile_smem<G, BF16, ORDER, S1>(ring + slot * R::kTileBytes, base, p.nb, lane, valid, t);
        __syncwarp();  // every lane has read the slot
        const uint64_t next = seq + R::kStages * nw;
        if (next < p.n_tiles) {
          if (lane == 0) {
            fence_proxy_async_smem();
            issue(next, slot);
          }
          ++issued;
        }
        call_body(full, base, lane, valid, t, body);
      }
    } else {
      // Lane 0's schedule: queue[s] is the tile held by the s-th slot to be read (kNoTile:
      // none, and none after it).
      const uint64_t cls = static_cast<uint64_t>(wid);
      unsigned* const counter = p.sched + wid * kSchedStrideWords;
      uint64_t queue[R::kStages];
      uint64_t issued = 0;
      unsigned pend = 0;
      bool more = true;  // lane 0: this warp's class may still have tiles for it
      if (lane == 0) {
#pragma unroll
        for (int s = 0; s < R::kStages; ++s) {
          const uint64_t tile = cls + kSchedClasses * (blockIdx.x + static_cast<uint64_t>(s) * gridDim.x);
          queue[s] = more && tile < p.n_tiles ? tile : kNoTile;
          more = queue[s] != kNoTile;
          if (more) {
            issue(queue[s], s);
            ++issued;
          }
        }
      }
      if (early) gdc_wait();
      if (lane == 0) {  // the counters are ready once the kernel before has completed
        if (more)
          pend = atomicAdd(counter, 1u);
        else
          sched_retire(p);
      }
      pre();

      for (uint64_t k = 0;; ++k) {
        const uint64_t cur = bcast0(lane == 0 ? queue[0] : 0);
        if (cur == kNoTile) break;
        const int slot = static_cast<int>(k % R::kStages);
        const uint32_t parity = static_cast<uint32_t>((k / R::kStages) & 1);
        const bool ok = mbar_wait(bar0 + slot * 8, parity);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          timed_out(k, bcast0(issued));
          return;
        }
        const uint64_t base = cur * kTileBlocks;
        const bool full = kSplitFull && p.nb - base >= kTileBlocks;  // the same in every lane
        bool valid[4];
        Lane4 t;
        if (full)
          load_tile_smem<G, BF16, ORDER, S1, true>(ring + slot * R::kTileBytes, base, p.nb, lane, valid, t);
        else
          load_tile_smem<G, BF16, ORDER, S1>(ring + slot * R::kTileBytes, base, p.nb, lane, valid, t);
        __syncwarp();  // every lane has read the slot
        if (lane == 0) {
          uint64_t nt = kNoTile;
          if (more) {
            nt = cls + kSchedClasses * (static_cast<uint64_t>(R::kStages) * gridDim.x + pend);
            if (nt < p.n_tiles) {
              pend = atomicAdd(counter, 1u);  // the one after, read ahead
              fence_proxy_async_smem();
              issue(nt, slot);
              ++issued;
            } else {
              nt = kNoTile;
              more = false;
              sched_retire(p);
            }
          }
#pragma unroll
          for (int s = 0; s + 1 < R::kStages; ++s) queue[s] = queue[s + 1];
          queue[R::kStages - 1] = nt;
        }
        call_body(full, base, lane, valid, t, body);
      }
    }
  }
}

// Row-group units through the TMA ring, each unit as its 8 tiles in order: body(tile, lane,
// valid, t) is called with the RgTile.  A unit's geometry (row tile, row pair, column chunk)
// comes from its index by one division, once per unit; a tile adds its row offset.
// Fixed split (DYN false): warp w of W takes the units w, w + W, ...  Run-time split (DYN):
// unit u belongs to class u % C (C = kSchedClasses) and warp c of every CTA serves class c,
// units c + C j: its first j is blockIdx.x, every later one gridDim.x + the value of an
// atomicAdd on the class counter p.sched[c * kSchedStrideWords], read by lane 0 a unit ahead
// (as for_each_tile's run-time split; the last warp to run out puts the counters back to 0).
// Lane 0 keeps the schedule: the unit it fetches tiles from and, once the reader reaches a
// unit, that unit's index for the other lanes (the fetcher is STAGES < 8 tiles ahead, so at
// most two units are in flight).
template <int G, bool BF16, int STAGES, bool DYN = false, int ORDER = 0, bool S1 = false, typename Body,
          typename Pre = NoPrologue>
__device__ __forceinline__ void for_each_rg_tile(const Params& p, Body&& body, Pre&& pre = Pre()) {
  using R = Ring<BF16, STAGES>;
  static_assert(R::kStages < 8, "the fetcher stays within one unit of the reader");
  constexpr uint32_t kNoUnit = ~0u;
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const uint32_t n_units = static_cast<uint32_t>(p.n_tiles >> 3);  // < 2^29
  struct Unit {
    uint32_t rt, k, row0, c0, ncols;
  };
  auto unit_of = [&](uint32_t u) {
    Unit s;
    const uint32_t rg = fast_div(u, p.div_ncc);  // row group: 16 per row tile of 128 rows
    s.rt = rg >> 4;
    s.k = rg & 15u;
    s.row0 = s.rt * 128u + 2u * s.k;
    s.c0 = (u - rg * p.n_cc) * static_cast<uint32_t>(kTileBlocks);
    const uint32_t left = p.nbr - s.c0;
    s.ncols = left < kTileBlocks ? left : kTileBlocks;
    return s;
  };
  auto tile_in = [&](const Unit& s, int rs) {  // rows 2k + {0, 1, 32, 33, 64, 65, 96, 97}
    RgTile g;
    g.rt = s.rt;
    g.k = s.k;
    g.rs = rs;
    g.row = s.row0 + static_cast<uint32_t>(rs & 1) + 32u * static_cast<uint32_t>(rs >> 1);
    g.c0 = s.c0;
    g.ncols = s.ncols;
    g.present = g.row < p.rows;
    return g;
  };

  extern __shared__ __align__(1024) uint8_t hq_smem[];
  uint8_t* ring = hq_smem + wid * R::kStages * R::kTileBytes;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar0 = smem_addr(hq_smem + R::kDataBytes) + wid * R::kStages * 8;
  const uint64_t policy = l2_stream_policy();
  auto issue = [&](const RgTile& g, int slot) {
    if (g.present)
      tma_load(ring_s + slot * R::kTileBytes,
               p.x + static_cast<uint64_t>(g.row) * p.ldx_bytes + g.c0 * 16u * R::kElemBytes,
               g.ncols * 16u * R::kElemBytes, bar0 + slot * 8, policy);
    else
      mbar_expect_tx(bar0 + slot * 8, 0);  // an empty tile: the phase completes at once
  };

  if (lane == 0) {
    for (int s = 0; s < R::kStages; ++s) mbar_init(bar0 + s * 8, 1);
    fence_mbar_init();
  }
  __syncwarp();

  // Lane 0's fetch position: unit fu (kNoUnit: none left), tile frs, and its geometry.
  const uint32_t cls = static_cast<uint32_t>(wid);
  unsigned* const counter = p.sched + (DYN ? wid * kSchedStrideWords : 0);
  uint32_t fu = DYN ? cls + kSchedClasses * blockIdx.x : blockIdx.x * kWarpsPerCta + wid;
  if (fu >= n_units) fu = kNoUnit;
  unsigned pend = 0;
  if constexpr (DYN) {
    if (lane == 0) {  // the kernel waited for the one before it: the counters are ready
      if (fu != kNoUnit)
        pend = atomicAdd(counter, 1u);
      else
        sched_retire(p);
    }
  }
  const uint32_t first = fu;
  auto next_unit = [&]() {  // lane 0: the unit after fu
    uint32_t u;
    if constexpr (DYN) {
      const uint64_t j = static_cast<uint64_t>(gridDim.x) + pend;
      u = j < (uint64_t{1} << 29) ? cls + kSchedClasses * static_cast<uint32_t>(j) : kNoUnit;
      if (u < n_units) {
        pend = atomicAdd(counter, 1u);  // the one after, read ahead
      } else {
        u = kNoUnit;
        sched_retire(p);
      }
    } else {
      const uint32_t nw = gridDim.x * kWarpsPerCta;
      u = (n_units - fu > nw) ? fu + nw : kNoUnit;
    }
    return u;
  };
  Unit fg = unit_of(fu == kNoUnit ? 0u : fu);
  int frs = 0;
  uint64_t issued = 0;  // lane 0: tiles handed to TMA
  auto fetch = [&](int slot) {  // lane 0: issue the next tile, if any, into `slot`
    if (fu == kNoUnit) return;
    issue(tile_in(fg, frs), slot);
    ++issued;
    if (++frs == 8) {
      frs = 0;
      fu = next_unit();
      if (fu != kNoUnit) fg = unit_of(fu);
    }
  };
  if (lane == 0)
    for (int s = 0; s < R::kStages; ++s) fetch(s);
  pre();

  uint32_t cu = bcast0(lane == 0 ? first : 0u) & 0xFFFFFFFFu;  // the unit being read
  Unit cg;
  int crs = 0;
  for (uint64_t k = 0;; ++k) {
    if (crs == 0) {
      if (cu == kNoUnit) break;
      cg = unit_of(cu);
    }
    const int slot = static_cast<int>(k % R::kStages);
    const uint32_t parity = static_cast<uint32_t>((k / R::kStages) & 1);
    const bool ok = mbar_wait(bar0 + slot * 8, parity);
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      if (lane == 0) atomicOr(&g_hq_fault, kFaultWaitTimeout);
      const uint64_t n_issued = bcast0(issued);
      for (uint64_t m = k; m < n_issued; ++m)
        mbar_wait(bar0 + static_cast<int>(m % R::kStages) * 8, static_cast<uint32_t>((m / R::kStages) & 1));
      return;
    }
    const RgTile g = tile_in(cg, crs);
    bool valid[4];
    Lane4 t;
    // the 256-group's body compiled a second time for whole tiles, as in for_each_tile
    const bool full = G == 256 && ORDER == 2 && g.present && g.ncols == kTileBlocks;
    if (full)
      load_tile_smem<G, BF16, ORDER, S1, true>(ring + slot * R::kTileBytes, 0, kTileBlocks, lane, valid, t);
    else
      load_tile_smem<G, BF16, ORDER, S1>(ring + slot * R::kTileBytes, 0, g.present ? g.ncols : 0, lane, valid, t);
    __syncwarp();  // every lane has read the slot
    if (lane == 0) {
      fence_proxy_async_smem();
      fetch(slot);
    }
    call_body(full, g, lane, valid, t, body);
    if (++crs == 8) {
      crs = 0;
      // the fetcher is past this unit's end and within the next one (or out of units)
      cu = static_cast<uint32_t>(bcast0(lane == 0 ? fu : 0u));
    }
  }
}

// ---------------------------------------------------------------------------
// The butterfly.  Stage h maps (a, b) = (z[i], z[i+h]) -> (a + b, a - b).
// Result: the unscaled transform z; the caller applies 1/sqrt(G).
// ---------------------------------------------------------------------------
template <int HEND = 16, int HBEG = 1>  // stages h = HBEG, 2 HBEG, ... below HEND
__device__ __forceinline__ void butterfly16(float2 (&v)[16]) {
#pragma unroll
  for (int h = HBEG; h < HEND; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float2 a = v[i];
        const float2 b = v[i + h];
        v[i] = add2(a, b);
        v[i + h] = sub2(a, b);
      }
    }
  }
}

// H256 stages h = 16, 32: the partner block sits in lane ^ 1, lane ^ 2 of the
// quad.  The lane holding the lower index computes a + b = own * 1 + partner,
// the other a - b = own * (-1) + partner; both are one rounding (fma with an
// exact product).  Every register slot is treated alike.
__device__ __forceinline__ void cross_lane_stages(Lane4& t, int lane) {
#pragma unroll
  for (int m = 1; m <= 2; m <<= 1) {
    const float sg = (lane & m) ? -1.0f : 1.0f;
    const float2 s2 = make_float2(sg, sg);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float2 o;
        o.x = __shfl_xor_sync(0xFFFFFFFFu, t.P[k][i].x, m);
        o.y = __shfl_xor_sync(0xFFFFFFFFu, t.P[k][i].y, m);
        t.P[k][i] = fma2(t.P[k][i], s2, o);
      }
    }
  }
}

// S1: the loads already applied the stage h = 1 (widen_stage1_bf16).
template <int G, bool S1 = false>
__device__ __forceinline__ void rotate_tile(Lane4& t, int lane) {
  if constexpr (G == 0) {
    return;
  } else {
    butterfly16<16, S1 ? 2 : 1>(t.P[0]);
    butterfly16<16, S1 ? 2 : 1>(t.P[1]);
    if constexpr (G == 256) {
      cross_lane_stages(t, lane);
      // h = 64: register block j <-> j ^ 1, i.e. the two halves of each pair:
      // (a, b) -> (a + b, a - b) = fma((a, b), (1, -1), (b, a)), one rounding each.
#pragma unroll
      for (int k = 0; k < 2; ++k) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 v = t.P[k][i];
          t.P[k][i] = fma2(v, make_float2(1.0f, -1.0f), make_float2(v.y, v.x));
        }
      }
      // h = 128: register block j <-> j ^ 2, i.e. pair 0 against pair 1.
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 a = t.P[0][i];
        const float2 b = t.P[1][i];
        t.P[0][i] = add2(a, b);
        t.P[1][i] = sub2(a, b);
      }
    }
  }
}

template <int G>
__device__ __forceinline__ constexpr float inv_sqrt_g() {
  return G == 16 ? 0.25f : (G == 256 ? 0.0625f : 1.0f);
}

template <int G>
__device__ __forceinline__ constexpr float sqrt_g() {
  return G == 16 ? 4.0f : (G == 256 ? 16.0f : 1.0f);
}

// ---------------------------------------------------------------------------
// Pass 1: rotate + amax.
// ---------------------------------------------------------------------------
// One butterfly stage on a register pair whose order may be swapped: with
// s = (1, 1) the pair holds (a, b) = (lower, upper index) and becomes (a + b, a - b);
// with s = (-1, -1) it holds (b, a) and becomes (a - b, a + b), i.e. the swap is
// kept.  Each output is one fma with an exact product (+-1 times a value), so it
// equals RN(a + b) or RN(a - b) bit for bit, signed zeros included.
__device__ __forceinline__ void stage_pair(float2& r0, float2& r1, float2 s, float2 ns) {
  const float2 u = fma2(r0, s, r1);
  const float2 v = fma2(r1, ns, r0);
  r0 = u;
  r1 = v;
}

// The 256-group rotation on the slot order 2 layout (slot_block), for pass 2.  The
// quad's lane bits stand for block-index bits 1 ^ 3 (lane bit 0, a) and 3 (lane bit
// 1, b); the register bit k (P[0] / P[1]) starts as block bit 0, the component as
// block bit 2.  The two stages whose partners sit in another lane each exchange
// P[1] only, and the register bit k takes the stage's output bit:
//   h = 1..8   in each block;
//   h = 16     P[0] against P[1] (block bit 0 = k ^ a);
//   h = 32     P[1] exchanged with lane ^ 1 (same bit 3, other bit 1); the lane keeps
//              the pairs of block bit 0 = a, and P[k] becomes block bit 1 = k ^ a ^ b;
//   h = 64     .x against .y;
//   h = 128    P[1] exchanged with lane ^ 2 (same bit 0, other bit 3); the lane keeps
//              the pairs of block bit 1 = a ^ b, and P[k] becomes block bit 3 = k ^ b.
// Every lane ends with four whole rotated blocks (out_block), each value the
// definition's, bit for bit (stage_pair).
template <bool S1 = false>
__device__ __forceinline__ void rotate_tile_x256(Lane4& t, int lane) {
  const float sa = (lane & 1) ? -1.0f : 1.0f;
  const float sb = (lane & 2) ? -1.0f : 1.0f;
  const float sab = sa * sb;
  butterfly16<16, S1 ? 2 : 1>(t.P[0]);
  butterfly16<16, S1 ? 2 : 1>(t.P[1]);
#pragma unroll
  for (int i = 0; i < 16; ++i)
    stage_pair(t.P[0][i], t.P[1][i], make_float2(sa, sa), make_float2(-sa, -sa));
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    t.P[1][i].x = __shfl_xor_sync(0xFFFFFFFFu, t.P[1][i].x, 1);
    t.P[1][i].y = __shfl_xor_sync(0xFFFFFFFFu, t.P[1][i].y, 1);
    stage_pair(t.P[0][i], t.P[1][i], make_float2(sab, sab), make_float2(-sab, -sab));
  }
  // h = 64: (x, y) -> (x + y, x - y) = fma((x, y), (1, -1), (y, x)), one rounding each.
#pragma unroll
  for (int k = 0; k < 2; ++k) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 v = t.P[k][i];
      t.P[k][i] = fma2(v, make_float2(1.0f, -1.0f), make_float2(v.y, v.x));
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    t.P[1][i].x = __shfl_xor_sync(0xFFFFFFFFu, t.P[1][i].x, 2);
    t.P[1][i].y = __shfl_xor_sync(0xFFFFFFFFu, t.P[1][i].y, 2);
    stage_pair(t.P[0][i], t.P[1][i], make_float2(sb, sb), make_float2(-sb, -sb));
  }
}

// max |z| over the lane's blocks of a 256-group tile loaded in slot order 1
// (slot_block), without forming the outputs of the last stage.  The two stages
// whose partner values sit in another lane of the quad (h = 16 across lane bit 0,
// h = 64 across lane bit 1) each move half of the lane's values instead of all of
// them: the lane keeps the pairs whose other index bit (position bit 3 for h = 16,
// the register bit of h = 32 for h = 64) equals its own lane bit, sends the other
// half and receives the partner's values for the pairs it keeps.  Which register of
// a pair holds the lower index depends on the lane; stage_pair's sign vector
// follows it.  Stage order and rounding are those of the definition:
//   h = 1, 2, 4    in each block (positions in place);
//   h = 8          positions i, i + 8, halves swapped when A ^ (q & 1) = 1;
//   h = 16         registers i + 8 exchanged with lane ^ 1, lower index in the lane with A = 0;
//   h = 32         P[0] against P[1], block bit 1 = k ^ B;
//   h = 64         P[1] exchanged with lane ^ 2, lower index in the lane with B = 0;
//   h = 128        .x against .y, and only feeds the max: for any a, b,
//                  max(|RN(a + b)|, |RN(a - b)|) = RN(|a| + |b|) (one of a + b, a - b
//                  has magnitude |a| + |b|, the other at most that, and RN is monotone
//                  and odd), which holds with a NaN too.  (An a, b = +-inf of opposite
//                  signs gives inf where the stage gives a NaN, so non-finite input
//                  still surfaces.)
// The lane ends up with outputs of positions other than the ones it loaded, which
// does not matter for a maximum.
template <bool S1 = false>
__device__ __forceinline__ float absmax256_x(Lane4& t, int lane) {
  const float sA = (lane & 1) ? -1.0f : 1.0f;
  const float sB = (lane & 2) ? -1.0f : 1.0f;
  const float sH = ((lane ^ (lane >> 2)) & 1) ? -1.0f : 1.0f;
  butterfly16<8, S1 ? 2 : 1>(t.P[0]);
  butterfly16<8, S1 ? 2 : 1>(t.P[1]);
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      stage_pair(t.P[k][i], t.P[k][i + 8], make_float2(sH, sH), make_float2(-sH, -sH));
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      t.P[k][i + 8].x = __shfl_xor_sync(0xFFFFFFFFu, t.P[k][i + 8].x, 1);
      t.P[k][i + 8].y = __shfl_xor_sync(0xFFFFFFFFu, t.P[k][i + 8].y, 1);
      stage_pair(t.P[k][i], t.P[k][i + 8], make_float2(sA, sA), make_float2(-sA, -sA));
    }
#pragma unroll
  for (int i = 0; i < 16; ++i)
    stage_pair(t.P[0][i], t.P[1][i], make_float2(sB, sB), make_float2(-sB, -sB));
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    t.P[1][i].x = __shfl_xor_sync(0xFFFFFFFFu, t.P[1][i].x, 2);
    t.P[1][i].y = __shfl_xor_sync(0xFFFFFFFFu, t.P[1][i].y, 2);
    stage_pair(t.P[0][i], t.P[1][i], make_float2(sB, sB), make_float2(-sB, -sB));
  }
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int i = 0; i < 16; i += 2)
      m = max3_nan(m, __fadd_rn(fabsf(t.P[k][i].x), fabsf(t.P[k][i].y)),
                   __fadd_rn(fabsf(t.P[k][i + 1].x), fabsf(t.P[k][i + 1].y)));
  return m;
}

// This thread's max |z| (unscaled butterfly output) over its tiles of x; y is
// written too when WRITE_Y.
template <int G, bool BF16, int MODE, bool WRITE_Y>
__device__ __forceinline__ float rot_amax_tiles(const Params& p) {
  // Without a rotated output, the 256-group takes slot order 1 and skips the
  // last stage's outputs (absmax256_x).
  constexpr bool kAbsTrick = G == 256 && !WRITE_Y;
  // bf16 tiles of the 256-group arrive with the first butterfly stage applied
  // (widen_stage1_bf16), with or without a rotated output.
  constexpr bool kS1 = BF16 && G == 256;
  float zmax = 0.0f;
  // Walk x from its end (for_each_tile, REVERSE): pass 2 walks it from the start.
  for_each_tile<G, BF16, MODE, HQ_PASS1_STAGES, kAbsTrick ? 1 : 0, kS1, true>(
      p, [&](uint64_t base, int lane, bool (&valid)[4], Lane4& t) {
    if constexpr (kAbsTrick) {
      zmax = max_nan(zmax, absmax256_x<kS1>(t, lane));
      return;
    }
    rotate_tile<G, kS1>(t, lane);
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        zmax = max_nan(zmax, max_nan(fabsf(t.P[k][i].x), fabsf(t.P[k][i].y)));
    if constexpr (WRITE_Y) {
      const float c = inv_sqrt_g<G>();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t b = base + lane_block<G>(lane, j);
        if (!valid[j]) continue;
        float4* dst = reinterpret_cast<float4*>(p.y + b * 16u);
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          float e[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 pr = t.P[j >> 1][4 * i4 + u];
            e[u] = __fmul_rn((j & 1) ? pr.y : pr.x, c);
          }
          dst[i4] = make_float4(e[0], e[1], e[2], e[3]);
        }
      }
    }
  });
  return zmax;
}

template <int G, bool BF16, int MODE, bool WRITE_Y>
__global__ void __launch_bounds__(kThreads, HQ_PASS1_MIN_CTAS) k_rot_amax(Params p) {
  // As k_rot_amax_stream: wait for the kernel before, then let the next one be launched.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  // |y| = RN(|z| / sqrt(G)) is monotone in |z|, so max |y| = RN(max |z| / sqrt(G))
  // exactly; the scaling commutes with the max over the CTA.
  cta_amax_to_global(__fmul_rn(rot_amax_tiles<G, BF16, MODE, WRITE_Y>(p), inv_sqrt_g<G>()), p.amax_out,
                     p.sync ? p.sync + 2 : nullptr, p.amax_copy);
}

// ---------------------------------------------------------------------------
// Pass 1, streaming form for G <= 16 on contiguous rows: every thread takes two
// whole blocks per step (block b and b + S, S = threads in the grid), each with
// one 256-bit load per 32 bytes, and keeps the next two in flight while it
// rotates the current pair.  It needs no shared memory and about 60 registers,
// so 32 warps per SM keep 64 KB of loads outstanding; x must be 32-byte aligned.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld_v8_stream(const uint8_t* src, uint32_t* w) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
        "=r"(w[7])
      : "l"(src));
}

#ifndef HQ_STREAM_DEPTH
#define HQ_STREAM_DEPTH 1
#endif

template <int G, bool BF16>
__global__ void __launch_bounds__(kThreads, HQ_STREAM_DEPTH == 1 ? 4 : 3) k_rot_amax_stream(Params p) {
  // When this grid was launched as a programmatic dependent (hq_quantize_nvfp4 with a
  // workspace), wait for the kernel before it to complete before reading x.  Then let the
  // next kernel on the stream (pass 2) be launched: it waits for this grid's completion
  // before it reads the amax, and since the launch comes after this wait, whatever wrote x
  // has completed by then (pass 2 of hq_quantize_nvfp4 reads its first tiles of x early).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int kWords = BF16 ? 8 : 16;  // 32-bit words per 16-element block
  const uint64_t S = static_cast<uint64_t>(gridDim.x) * kThreads;
  uint64_t b = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;
  // The k-th block of the walk is block nb - 1 - k: x is read from its end, where pass
  // 2 (which walks it from the start) of the previous call stopped and part of it is
  // still in L2.
  auto load = [&](uint64_t blk, uint32_t (&w)[kWords]) {
    if (blk < p.nb) {
      const uint8_t* src = p.x + (p.nb - 1 - blk) * (16u * (BF16 ? 2u : 4u));
#pragma unroll
      for (int k = 0; k < kWords; k += 8) ld_v8_stream(src + 4 * k, w + k);
    } else {
#pragma unroll
      for (int k = 0; k < kWords; ++k) w[k] = 0u;
    }
  };
  auto value = [&](const uint32_t (&w)[kWords], int i) {
    if constexpr (BF16)
      return __uint_as_float((i & 1) ? (w[i >> 1] & 0xFFFF0000u) : (w[i >> 1] << 16));
    else
      return __uint_as_float(w[i]);
  };
  float zmax = 0.0f;
  auto consume = [&](const uint32_t (&a)[kWords], const uint32_t (&c)[kWords]) {
    float2 v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = make_float2(value(a, i), value(c, i));
    if constexpr (G == 16) butterfly16(v);
#pragma unroll
    for (int i = 0; i < 16; ++i) zmax = max3_nan(zmax, fabsf(v[i].x), fabsf(v[i].y));
  };
#if HQ_STREAM_DEPTH == 1
  uint32_t wa[kWords], wb[kWords];
  load(b, wa);
  load(b + S, wb);
  for (; b < p.nb; b += 2 * S) {
    uint32_t ca[kWords], cb[kWords];
#pragma unroll
    for (int k = 0; k < kWords; ++k) { ca[k] = wa[k]; cb[k] = wb[k]; }
    load(b + 2 * S, wa);
    load(b + 3 * S, wb);
    consume(ca, cb);
  }
#else
  // two pairs in flight: (wa, wb) for step b, (wc, wd) for step b + 2S
  uint32_t wa[kWords], wb[kWords], wc[kWords], wd[kWords];
  load(b, wa);
  load(b + S, wb);
  load(b + 2 * S, wc);
  load(b + 3 * S, wd);
  for (; b < p.nb; b += 4 * S) {
    uint32_t ca[kWords], cb[kWords];
#pragma unroll
    for (int k = 0; k < kWords; ++k) { ca[k] = wa[k]; cb[k] = wb[k]; }
    load(b + 4 * S, wa);
    load(b + 5 * S, wb);
    consume(ca, cb);
    if (b + 2 * S >= p.nb) break;
#pragma unroll
    for (int k = 0; k < kWords; ++k) { ca[k] = wc[k]; cb[k] = wd[k]; }
    load(b + 6 * S, wc);
    load(b + 7 * S, wd);
    consume(ca, cb);
  }
#endif
  cta_amax_to_global(__fmul_rn(zmax, inv_sqrt_g<G>()), p.amax_out, p.sync ? p.sync + 2 : nullptr,
                     p.amax_copy);
}

// ---------------------------------------------------------------------------
// Pass 2: rotate + quantize + pack.
// ---------------------------------------------------------------------------
// SWZ: write the scales in the swizzled tile layout of block-scaled NVFP4 GEMMs
// (cuBLASLt's layout for 16-element block scales): the [M, K/16] scale matrix,
// padded to whole tiles of 128 rows x 4 columns, each tile 512 contiguous bytes,
// tiles row-major; inside a tile, row r and column c at (r % 32) * 16 + (r / 32) *
// 4 + c.  The tiles of this mode are row groups (RgTile), so that every scale
// store fills whole 32-byte pieces of that layout, padding included.
// amax: where the global amax is read, once the first tile copies are in flight.
// GDC: the kernel was launched as a programmatic dependent and has not yet executed
// griddepcontrol.wait; the tile loop does.
template <int G, bool BF16, int MODE, bool REDUCE_NEXT, bool SWZ = false, bool GDC = false,
          bool DYN = false>
__device__ __forceinline__ void rotate_quant_tiles(const Params& p, const float* amax) {
  const float r6 = __frcp_rn(6.0f);
  float s_global, rg;  // s_global and its reciprocal (Markstein fast path of the block scales)
  bool sg_ok, q_fast;

  constexpr float c = inv_sqrt_g<G>();
  constexpr float sq = sqrt_g<G>();
  // Register layout of a tile: the 256-group's exchange form (slot_block order 2), also for
  // row-group tiles (SWZ), whose scale gather follows out_block.
  constexpr int kOrder = G == 256 ? 2 : 0;
  // bf16 tiles of the 256-group arrive with the first butterfly stage applied
  // (widen_stage1_bf16).  (For G = 16 the separate widen and packed stage measured
  // faster: 364 against 381 us on bf16 [32768, 28672].)
  constexpr bool kS1 = BF16 && G == 256;

  // The fast path's divisor pair for each E4M3 block scale, indexed by its byte
  // (0..126; the NaN 0x7F never comes out of the satfinite conversion):
  // d = RN(s_f * sqrt(G)) and nr = -RN(1 / d), with s_f = RN(s_block * s_global).
  // On the fast path's domain s_f is a normal float for every non-zero s_block, so
  // s_f == 0 exactly for byte 0, whose entry is d = 1, nr = -1 (its codes are then
  // masked to 0).  The entries are what each block would compute for its own scale,
  // computed once per CTA instead of once per block.
  __shared__ float tab_d[128];
  __shared__ float tab_nr[128];
  auto prologue = [&]() {
    // s_global = amax / (448 * 6), or 1 if that is 0.
    s_global = __fdiv_rn(*amax, 2688.0f);
    if (s_global == 0.0f) s_global = 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.sglobal_out) *p.sglobal_out = s_global;
    rg = __frcp_rn(s_global);
    sg_ok = s_global >= 0x1p-60f && s_global <= 0x1p60f;
    q_fast = s_global >= 0x1p-87f && s_global <= 0x1p91f;
    if (q_fast) {  // the same for every thread of the grid
      for (int e = threadIdx.x; e < 128; e += kThreads) {
        const float sfe = __fmul_rn(e4m3x2_to_f32(static_cast<uint32_t>(e)).x, s_global);
        const float d = (sfe == 0.0f) ? 1.0f : __fmul_rn(sfe, sq);
        tab_d[e] = d;
        tab_nr[e] = -__frcp_rn(d);
      }
      __syncthreads();
    }
  };
  float next_amax = 0.0f;  // max of the block amaxes this thread saw (REDUCE_NEXT)
  uint32_t swz_acc[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // SWZ: scale words of the unit's rows

  // tile: the tile's first block (flat tiles) or its RgTile (SWZ).
  auto tile_body = [&](const auto& tile, int lane, bool (&valid)[4], Lane4& t) {
    if constexpr (kOrder == 2)
      rotate_tile_x256<kS1>(t, lane);
    else
      rotate_tile<G, kS1>(t, lane);

    // Block amax of z, then of y = z / sqrt(G): RN(max|z| * c) = max RN(|z| * c).
    float am[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      am[2 * k] = __fmul_rn(block_absmax<false>(t.P[k]), c);
      am[2 * k + 1] = __fmul_rn(block_absmax<true>(t.P[k]), c);
    }
    if constexpr (REDUCE_NEXT)
      next_amax = max3_nan(next_amax, max_nan(am[0], am[1]), max_nan(am[2], am[3]));

    // Block scales: v = (amax_b / 6) / s_global, two correctly rounded
    // divisions, then E4M3 (RNE, satfinite).  The Markstein form is exact for
    // amax_b in [2^-90, 2^90] and s_global in [2^-60, 2^60]; below 2^-90 it can be
    // off by an ulp of a value under 2^-29, which rounds to the E4M3 zero either
    // way, so only the upper bound needs a check.
    bool v_fast = sg_ok;
#pragma unroll
    for (int j = 0; j < 4; ++j) v_fast &= am[j] <= 0x1p90f;
    float v[4];
    if (v_fast) {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = div_markstein(div_markstein(am[j], 6.0f, r6), s_global, rg);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __fdiv_rn(__fdiv_rn(am[j], 6.0f), s_global);
    }
    uint32_t sb2[2];    // two E4M3 patterns per pair
#pragma unroll
    for (int k = 0; k < 2; ++k) sb2[k] = e4m3x2(v[2 * k], v[2 * k + 1]);
    uint32_t keep[4];   // all ones, or 0 where s_f == 0 (every code of the block is 0)

    // Fast path: q = RN(y / s_f) = RN(z / D), D = s_f * sqrt(G), by Markstein's
    // correction with r = RN(1/D) (as div_markstein).  The domain s_f in
    // [2^-96, 2^100] keeps D, r, z and e normal wherever the rounding decides a
    // code (|q| >= 1/8); a smaller quotient gives code 0 with the sign of z either
    // way, and y = RN(z c) equals z c there except for values that only give such
    // codes.  A non-zero s_block lies in [2^-9, 448], so q_fast (s_global in
    // [2^-87, 2^91]) puts every non-zero s_f of the tensor in that domain.
    //
    // The steps run on negated values, with nr = -r:  q0n = RN(z nr) = -q0,
    // e = RN(z + q0n D), qn = RN(q0n + e nr) = -q.  In this form qn is -q even for
    // z = +-0 (the direct form turns -0 into +0, since e = +0 and +0 + -0 = +0),
    // so code(q) = code(qn) with the sign bit flipped: one XOR per 8 codes.
    uint32_t w[4][2];  // packed codes per block: elements 0..7, 8..15
    if (q_fast) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t ex = sb2[k] & 0xFFu, ey = (sb2[k] >> 8) & 0xFFu;
        const float2 nr = make_float2(tab_nr[ex], tab_nr[ey]);
        const float2 d = make_float2(tab_d[ex], tab_d[ey]);
        keep[2 * k] = ex ? 0xFFFFFFFFu : 0u;
        keep[2 * k + 1] = ey ? 0xFFFFFFFFu : 0u;
        float2 qv[16];  // -q
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 z = t.P[k][i];
          if constexpr (G == 256) {
            // Scalar here: bf16 [8192, 16384] 73.4 -> 71.7 us (the packed form keeps the
            // FMA pipe's heavy half busy two cycles per instruction; G = 16 is faster packed)
            const float q0x = __fmul_rn(z.x, nr.x), q0y = __fmul_rn(z.y, nr.y);
            const float ex = __fmaf_rn(q0x, d.x, z.x), ey = __fmaf_rn(q0y, d.y, z.y);
            qv[i] = make_float2(__fmaf_rn(ex, nr.x, q0x), __fmaf_rn(ey, nr.y, q0y));
          } else {
            const float2 q0n = mul2(z, nr);
            const float2 e = fma2(q0n, d, z);
            qv[i] = fma2(e, nr, q0n);
          }
        }
        constexpr uint32_t kFlip = 0x88888888u;  // sign bit of every nibble
        w[2 * k][0] = kFlip ^ e2m1x8(qv[0].x, qv[1].x, qv[2].x, qv[3].x, qv[4].x, qv[5].x, qv[6].x, qv[7].x);
        w[2 * k][1] = kFlip ^ e2m1x8(qv[8].x, qv[9].x, qv[10].x, qv[11].x, qv[12].x, qv[13].x, qv[14].x, qv[15].x);
        w[2 * k + 1][0] = kFlip ^ e2m1x8(qv[0].y, qv[1].y, qv[2].y, qv[3].y, qv[4].y, qv[5].y, qv[6].y, qv[7].y);
        w[2 * k + 1][1] = kFlip ^ e2m1x8(qv[8].y, qv[9].y, qv[10].y, qv[11].y, qv[12].y, qv[13].y, qv[14].y, qv[15].y);
      }
    } else {
      // The definition, literally: y = RN(z / sqrt(G)), q = RN(y / s_f).
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float sbf = e4m3x2_to_f32(sb2[j >> 1] >> ((j & 1) * 8)).x;
        const float sfj = __fmul_rn(sbf, s_global);
        keep[j] = (sfj == 0.0f) ? 0u : 0xFFFFFFFFu;
        float qv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float z = (j & 1) ? t.P[j >> 1][i].y : t.P[j >> 1][i].x;
          const float y = __fmul_rn(z, c);
          qv[i] = (sfj == 0.0f) ? 0.0f : __fdiv_rn(y, sfj);
        }
        w[j][0] = e2m1x8(qv[0], qv[1], qv[2], qv[3], qv[4], qv[5], qv[6], qv[7]);
        w[j][1] = e2m1x8(qv[8], qv[9], qv[10], qv[11], qv[12], qv[13], qv[14], qv[15]);
      }
    }

    if constexpr (!SWZ) {
      const uint64_t base = tile;
      // Stores: 8 code bytes and 1 scale byte per block, streaming (evict-first).
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!valid[j]) continue;
        const uint64_t b = base + out_block<G, kOrder>(lane, j);
        __stcs(reinterpret_cast<uint2*>(p.q + b * 8u), make_uint2(w[j][0] & keep[j], w[j][1] & keep[j]));
        const uint32_t sbyte = (sb2[j >> 1] >> ((j & 1) * 8)) & 0xFFu;
        __stcs(reinterpret_cast<unsigned char*>(p.s + b), static_cast<unsigned char>(sbyte));
      }
    } else {
      // Row-group unit tile (base = tile index): one row segment, as a flat tile.
      const RgTile& g = tile;
      uint8_t* q_tile = p.q + (static_cast<uint64_t>(g.row) * p.nbr + g.c0) * 8u;  // codes of block c0
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!valid[j]) continue;
        __stcs(reinterpret_cast<uint2*>(q_tile + out_block<G, kOrder>(lane, j) * 8u),
               make_uint2(w[j][0] & keep[j], w[j][1] & keep[j]));
      }
      // Scales.  Row r, column c of the scale matrix sits at 512 * (row tile *
      // swz_col_tiles + c / 4) + (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4, so the
      // unit's 8 rows x 4 columns are the 32 bytes at 32 k of a column tile, row rs
      // in word 4 (rs & 1) + (rs >> 1).  Lane L collects column group L (columns
      // c0 + 4L .. + 3) of the unit's rows and writes its 32 bytes after the last
      // tile.  Blocks outside the tensor carry scale 0, which the padding must hold.
      // G <= 16: column group L sits in lanes 4 (L % 8) + m, slot L / 8 (block 32 j + lane),
      // m = 0..3 for its 4 columns.  G = 256 (the exchange layout, out_block): with u = L % 4,
      // its columns 0, 1, 2, 3 sit in lanes 4 (L / 4) + 0, 3, 2, 1, slots u, u ^ 2, u ^ 2, u
      // (lane (a, b) of the quad holds column a + 2 (a ^ b), slot 2 (u / 2 ^ b) + u % 2).  Each
      // lane packs its 4 slot bytes into one word; lane L reads the words of its 4 source
      // lanes and keeps one byte of each (byte permutes).
      const uint32_t all4 = __byte_perm(sb2[0], sb2[1], 0x5410);  // slot j in byte j
      const int src = (G == 256) ? (lane & ~3) : 4 * (lane & 7);
      const uint32_t r0 = __shfl_sync(0xFFFFFFFFu, all4, src);
      const uint32_t r1 = __shfl_sync(0xFFFFFFFFu, all4, src + 1);
      const uint32_t r2 = __shfl_sync(0xFFFFFFFFu, all4, src + 2);
      const uint32_t r3 = __shfl_sync(0xFFFFFFFFu, all4, src + 3);
      uint32_t mine;
      if constexpr (kOrder == 2) {
        const uint32_t u = lane & 3, v = u ^ 2u;
        mine = __byte_perm(__byte_perm(r0, r3, u | ((4u + v) << 4)), __byte_perm(r2, r1, v | ((4u + u) << 4)),
                           0x5410);
      } else {
        const uint32_t want = lane >> 3;
        const uint32_t sel = want | ((want + 4u) << 4);
        mine = __byte_perm(__byte_perm(r0, r1, sel), __byte_perm(r2, r3, sel), 0x5410);
      }
#pragma unroll
      for (int i = 0; i < 7; ++i) swz_acc[i] = swz_acc[i + 1];
      swz_acc[7] = mine;  // swz_acc[rs] holds row rs once rs = 7
      if (g.rs == 7) {
        const uint64_t ct = g.c0 / 4 + lane;
        if (ct < p.swz_col_tiles)
          st_v8(p.s + (static_cast<uint64_t>(g.rt) * p.swz_col_tiles + ct) * 512u + 32u * g.k, swz_acc[0],
                swz_acc[2], swz_acc[4], swz_acc[6], swz_acc[1], swz_acc[3], swz_acc[5], swz_acc[7]);
      }
    }
  };
  if constexpr (SWZ)
    for_each_rg_tile<G, BF16, HQ_PASS2_STAGES, DYN, kOrder, kS1>(p, tile_body, prologue);
  else
    for_each_tile<G, BF16, MODE, HQ_PASS2_STAGES, kOrder, kS1, false, GDC, DYN>(p, tile_body, prologue);
  // with p.sync (a workspace): reduced into the workspace, the last CTA moves it to p.amax_copy
  if constexpr (REDUCE_NEXT)
    cta_amax_to_global(next_amax, p.amax_out, p.sync ? p.sync + 2 : nullptr, p.amax_copy);
}

template <int G, bool BF16, int MODE, bool REDUCE_NEXT, bool SWZ = false, bool DYN = false>
__global__ void __launch_bounds__(kThreads, 2) k_rotate_quant_nvfp4(Params p) {
  // Launched with programmatic dependent launch: wait for the kernel before this one on
  // the stream (normally pass 1, which writes *amax_in) to complete before any access to
  // global memory other than the first tiles of an x that p.x_ready declares complete.
  // The plain tile loop waits itself, after its first tile copies when x is known to be
  // complete (p.x_ready); the row-group loop waits here.
  if constexpr (SWZ) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    rotate_quant_tiles<G, BF16, MODE, REDUCE_NEXT, SWZ, false, DYN>(p, p.amax_in);
  } else {
    rotate_quant_tiles<G, BF16, MODE, REDUCE_NEXT, SWZ, true, DYN>(p, p.amax_in);
  }
}

// ---------------------------------------------------------------------------
// MXFP4: one E8M0 scale per 32 consecutive elements, no per-tensor scale.
//   X = 2^(floor(log2 amax_32) - 2) (amax_32 / X in [4, 8)); E8M0 byte = that
//   exponent + 127, clamped at 0; codes = E2M1(y / X).  For a finite amax the
//   byte is max(biased fp32 exponent of amax - 2, 0), two integer operations.
// A 32-block is two consecutive 16-blocks, held by lanes l and l ^ 1 in both
// lane mappings; its amax is one xor-shuffle away.  Division by X is an exact
// multiply by 2^(127 - byte), with 1/sqrt(G) folded in; a lane holding a block
// whose byte is below 8 (amax below 2^-117, where folding could round subnormal
// values differently) applies the two steps literally.
// ---------------------------------------------------------------------------
//
// The 256-group takes pass 2's exchange layout (rotate_tile_x256, out_block): there the
// other half of a 32-block sits in lane ^ 3, in the other register of the P[0] / P[1]
// pair (block bit 0 is lane bit 0 and block bits 1 and 3 are unchanged), and bf16
// tiles arrive with the first butterfly stage applied.
// DYN: the run-time tile split of for_each_tile (tile counters in p.sched).
template <int G, bool BF16, int MODE, bool DYN = false>
__global__ void __launch_bounds__(kThreads, 2) k_rotate_quant_mxfp4(Params p) {
  // Launched with programmatic dependent launch, as pass 2: wait for the kernel before this
  // one on the stream to complete before any access to global memory.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr float c = inv_sqrt_g<G>();
  constexpr int kOrder = G == 256 ? 2 : 0;
  constexpr bool kS1 = BF16 && G == 256;
  for_each_tile<G, BF16, MODE, HQ_PASS2_STAGES, kOrder, kS1, false, false, DYN>(
      p, [&](uint64_t base, int lane, bool (&valid)[4], Lane4& t) {
    if constexpr (kOrder == 2)
      rotate_tile_x256<kS1>(t, lane);
    else
      rotate_tile<G>(t, lane);
    float am[4];  // block amax of y, slot 2k + h
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      am[2 * k] = __fmul_rn(block_absmax<false>(t.P[k]), c);
      am[2 * k + 1] = __fmul_rn(block_absmax<true>(t.P[k]), c);
    }
    uint32_t code[4];
    float inv[4];
    bool literal = false;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = 2 * k + h;
        const float other = kOrder == 2 ? __shfl_xor_sync(0xFFFFFFFFu, am[2 * (1 - k) + h], 3)
                                        : __shfl_xor_sync(0xFFFFFFFFu, am[j], 1);
        const float a32 = max_nan(am[j], other);
        const int eb = static_cast<int>(__float_as_uint(a32) >> 23);
        code[j] = static_cast<uint32_t>(eb > 2 ? eb - 2 : 0);
        inv[j] = __uint_as_float((254u - code[j]) << 23);  // 2^(127 - code), normal for code <= 253
        // a subnormal y (|y| < 2^-126) reaches a quotient of 2^(3 - biased exponent):
        // it can only decide a code in blocks whose byte is below 3; 8 leaves a margin
        literal |= code[j] < 8;
      }
    }
    uint32_t w[4][2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float2 f;
      if (!literal) f = make_float2(__fmul_rn(inv[2 * k], c), __fmul_rn(inv[2 * k + 1], c));
      float2 qv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (!literal) {
          qv[i] = mul2(t.P[k][i], f);
        } else {
          const float2 y = mul2(t.P[k][i], make_float2(c, c));
          qv[i] = mul2(y, make_float2(inv[2 * k], inv[2 * k + 1]));
        }
      }
      w[2 * k][0] = e2m1x8(qv[0].x, qv[1].x, qv[2].x, qv[3].x, qv[4].x, qv[5].x, qv[6].x, qv[7].x);
      w[2 * k][1] = e2m1x8(qv[8].x, qv[9].x, qv[10].x, qv[11].x, qv[12].x, qv[13].x, qv[14].x, qv[15].x);
      w[2 * k + 1][0] = e2m1x8(qv[0].y, qv[1].y, qv[2].y, qv[3].y, qv[4].y, qv[5].y, qv[6].y, qv[7].y);
      w[2 * k + 1][1] = e2m1x8(qv[8].y, qv[9].y, qv[10].y, qv[11].y, qv[12].y, qv[13].y, qv[14].y, qv[15].y);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!valid[j]) continue;
      const uint64_t b = base + out_block<G, kOrder>(lane, j);
      __stcs(reinterpret_cast<uint2*>(p.q + b * 8u), make_uint2(w[j][0], w[j][1]));
      if ((lane & 1) == 0)  // the even half (block bit 0 = lane bit 0) writes the scale byte
        __stcs(reinterpret_cast<unsigned char*>(p.s + (b >> 1)), static_cast<unsigned char>(code[j]));
    }
  });
}

// ---------------------------------------------------------------------------
// Dequant: value = (+-grid[c]) * (s_block * s_global), then optionally the
// rotation again (y = RN(z / sqrt(G)) after the same butterfly).  MX: value =
// (+-grid[c]) * 2^(byte - 127) for the 32-block's E8M0 byte.
// ---------------------------------------------------------------------------
template <int G, bool MX>
__global__ void __launch_bounds__(kThreads, 2) k_dequant_nvfp4(Params p) {
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (static_cast<uint64_t>(blockIdx.x) * kWarpsPerCta) + (threadIdx.x >> 5);
  const uint64_t n_warps = static_cast<uint64_t>(gridDim.x) * kWarpsPerCta;
  const float s_global = MX ? 1.0f : *p.dq_sglobal;
  for (uint64_t tile = warp; tile < p.n_tiles; tile += n_warps) {
    const uint64_t base = tile * kTileBlocks;
    bool valid[4];
    Lane4 t;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint64_t b = base + lane_block<G>(lane, j);
      valid[j] = b < p.nb;
      uint2 qw = make_uint2(0u, 0u);
      float s_f = 0.0f;
      if (valid[j]) {
        qw = __ldg(reinterpret_cast<const uint2*>(p.dq_q + b * 8u));
        if constexpr (MX) {
          const uint32_t e = __ldg(p.dq_s + (b >> 1));
          s_f = e >= 1u ? __uint_as_float(e << 23) : 0x1p-127f;  // 2^(e - 127)
        } else {
          const float sb = e4m3x2_to_f32(__ldg(p.dq_s + b)).x;
          s_f = __fmul_rn(sb, s_global);
        }
      }
      const float2 s2 = make_float2(s_f, s_f);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t byte = ((m < 4 ? qw.x : qw.y) >> (8 * (m & 3))) & 0xFFu;
        const float2 v = mul2(e2m1x2_to_f32(byte), s2);
        if (j & 1) {
          t.P[j >> 1][2 * m].y = v.x;
          t.P[j >> 1][2 * m + 1].y = v.y;
        } else {
          t.P[j >> 1][2 * m].x = v.x;
          t.P[j >> 1][2 * m + 1].x = v.y;
        }
      }
    }
    if constexpr (G != 0) {
      rotate_tile<G>(t, lane);
      const float2 c2 = make_float2(inv_sqrt_g<G>(), inv_sqrt_g<G>());
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int i = 0; i < 16; ++i) t.P[k][i] = mul2(t.P[k][i], c2);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!valid[j]) continue;
      const uint64_t b = base + lane_block<G>(lane, j);
      float4* dst = reinterpret_cast<float4*>(p.dq_out + b * 16u);
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        float e[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 pr = t.P[j >> 1][4 * i4 + u];
          e[u] = (j & 1) ? pr.y : pr.x;
        }
        __stcs(dst + i4, make_float4(e[0], e[1], e[2], e[3]));
      }
    }
  }
}

}  // namespace hq
