// hq_kernels.cuh -- device code of libhq (sm_103a).
//
// The three kernels of the fused Hadamard rotation + NVFP4 quantization
// ("A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §1 "The format,
// precisely" and §2 "The kernel"):
//
//   k_rot_amax            pass 1: stream x, rotate, reduce max |y| into one float.
//   k_rotate_quant_nvfp4  pass 2: stream x once, rotate in registers, block amax,
//                         E4M3 block scale, E2M1 codes, write codes + scales once.
//   k_dequant_nvfp4       round trip: codes * scales, optional inverse rotation.
//
// Work decomposition (all three kernels): a warp owns a "tile" of 128 NVFP4
// blocks (2048 elements); each lane holds 4 whole blocks (64 values) in
// registers.  Which 4 blocks a lane holds depends on the rotation group:
//   G <= 16 : block 32*j + lane of the tile (j = 0..3) -- each warp-wide memory
//             instruction covers 32 consecutive blocks;
//   G == 256: block 16*(lane/4) + (lane%4) + 4*j -- the 4 lanes of a quad hold
//             the 16 blocks of one 256-group; index bits 4,5 of the group are the
//             lane bits, bits 6,7 select the register block j.
// The 64 values sit in float2 pairs (block 0 with block 1, block 2 with block 3)
// so the butterfly and the division run on the packed fp32x2 pipe of sm_100-
// family parts (FADD2/FFMA2/FMUL2): one instruction per two values.
//
// Bit-exactness.  The butterfly performs the stages h = 1, 2, 4, 8 (inside a
// block), then for G = 256 h = 16, 32 (across the quad's lanes), 64, 128
// (across the lane's register blocks), each stage an fp32 add/sub with one
// rounding, exactly as the definition.  The final multiply by 1/sqrt(G) is
// folded into the division (see k_rotate_quant_nvfp4); that fold is exact on the
// fast path's domain, and the slow path evaluates the definition literally.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hq {

constexpr int kThreads = 256;            // 8 warps per CTA
constexpr int kWarpsPerCta = kThreads / 32;
constexpr int kBlocksPerLane = 4;
constexpr int kTileBlocks = 32 * kBlocksPerLane;  // 128 NVFP4 blocks per warp tile

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
  float* amax_out;         // atomically max-reduced (zeroed by the host call)
  float* y;                // optional fp32 rotated output [M, K]
  // pass 2
  const float* amax_in;
  uint8_t* q;              // [M, K/2]
  uint8_t* s;              // [M, K/16]
  float* sglobal_out;      // optional
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

__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 %%hq_a, %%hq_b, %%hq_d;\n\t"
      "mov.b64 %%hq_a, {%2, %3};\n\t"
      "mov.b64 %%hq_b, {%4, %5};\n\t"
      "sub.rn.f32x2 %%hq_d, %%hq_a, %%hq_b;\n\t"
      "mov.b64 {%0, %1}, %%hq_d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// max that keeps a NaN once seen (so a non-finite input surfaces in amax).
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
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

// Load one 16-element block and widen to fp32 (bf16 -> fp32 is exact).
// Element i of block `jb` goes to the .x (jb even) or .y (jb odd) lane of v[i].
template <bool BF16>
__device__ __forceinline__ void load_block(const uint8_t* ptr, float (&f)[16]) {
  if constexpr (BF16) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(ptr));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(ptr) + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      f[2 * k] = __uint_as_float(w[k] << 16);
      f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(ptr) + k);
      f[4 * k + 0] = __uint_as_float(a.x);
      f[4 * k + 1] = __uint_as_float(a.y);
      f[4 * k + 2] = __uint_as_float(a.z);
      f[4 * k + 3] = __uint_as_float(a.w);
    }
  }
}

// The lane's 4 blocks as two float2 arrays: P[0][i] = (blk0[i], blk1[i]),
// P[1][i] = (blk2[i], blk3[i]).
struct Lane4 {
  float2 P[2][16];
};

template <int G, bool BF16, bool STRIDED>
__device__ __forceinline__ void load_tile(const Params& p, uint64_t tile_base, int lane,
                                          bool (&valid)[4], Lane4& t) {
  constexpr int es = BF16 ? 2 : 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint64_t b = tile_base + lane_block<G>(lane, j);
    valid[j] = b < p.nb;
    float f[16];
    if (valid[j]) {
      load_block<BF16>(block_ptr<STRIDED>(p, b, es), f);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (j & 1)
        t.P[j >> 1][i].y = f[i];
      else
        t.P[j >> 1][i].x = f[i];
    }
  }
}

// ---------------------------------------------------------------------------
// The butterfly.  Stage h maps (a, b) = (z[i], z[i+h]) -> (a + b, a - b).
// Result: the unscaled transform z; the caller applies 1/sqrt(G).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void butterfly16(float2 (&v)[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
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

template <int G>
__device__ __forceinline__ void rotate_tile(Lane4& t, int lane) {
  if constexpr (G == 0) {
    return;
  } else {
    butterfly16(t.P[0]);
    butterfly16(t.P[1]);
    if constexpr (G == 256) {
      // h = 16, 32: partner block sits in lane ^ 1, lane ^ 2 of the quad.  The
      // lane holding the lower index computes a + b = own * 1 + partner, the
      // other a - b = own * (-1) + partner; both are one rounding (fma with an
      // exact product).
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
      // h = 64: register block j <-> j ^ 1, i.e. the two halves of each pair.
#pragma unroll
      for (int k = 0; k < 2; ++k) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = t.P[k][i].x;
          const float b = t.P[k][i].y;
          t.P[k][i].x = __fadd_rn(a, b);
          t.P[k][i].y = __fsub_rn(a, b);
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
template <int G, bool BF16, bool STRIDED, bool WRITE_Y>
__global__ void __launch_bounds__(kThreads, 2) k_rot_amax(Params p) {
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (static_cast<uint64_t>(blockIdx.x) * kWarpsPerCta) + (threadIdx.x >> 5);
  const uint64_t n_warps = static_cast<uint64_t>(gridDim.x) * kWarpsPerCta;
  float zmax = 0.0f;
  for (uint64_t tile = warp; tile < p.n_tiles; tile += n_warps) {
    const uint64_t base = tile * kTileBlocks;
    bool valid[4];
    Lane4 t;
    load_tile<G, BF16, STRIDED>(p, base, lane, valid, t);
    rotate_tile<G>(t, lane);
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
  }
  // max over the CTA, then one atomic per CTA.  |y| = RN(|z| / sqrt(G)) is
  // monotone in |z|, so max |y| = RN(max |z| / sqrt(G)) exactly.
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) zmax = max_nan(zmax, __shfl_xor_sync(0xFFFFFFFFu, zmax, m));
  __shared__ float red[kWarpsPerCta];
  if (lane == 0) red[threadIdx.x >> 5] = zmax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = red[0];
#pragma unroll
    for (int w = 1; w < kWarpsPerCta; ++w) m = max_nan(m, red[w]);
    const float a = __fmul_rn(m, inv_sqrt_g<G>());
    // non-negative floats (and NaN, with the sign cleared by fabs) order like
    // their bit patterns as unsigned integers.
    atomicMax(reinterpret_cast<unsigned int*>(p.amax_out), __float_as_uint(a));
  }
}

// ---------------------------------------------------------------------------
// Pass 2: rotate + quantize + pack.
// ---------------------------------------------------------------------------
template <int G, bool BF16, bool STRIDED>
__global__ void __launch_bounds__(kThreads, 2) k_rotate_quant_nvfp4(Params p) {
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (static_cast<uint64_t>(blockIdx.x) * kWarpsPerCta) + (threadIdx.x >> 5);
  const uint64_t n_warps = static_cast<uint64_t>(gridDim.x) * kWarpsPerCta;

  // s_global = amax / (448 * 6), or 1 if that is 0.
  const float amax = *p.amax_in;
  float s_global = __fdiv_rn(amax, 2688.0f);
  if (s_global == 0.0f) s_global = 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.sglobal_out) *p.sglobal_out = s_global;

  constexpr float c = inv_sqrt_g<G>();
  constexpr float sq = sqrt_g<G>();

  for (uint64_t tile = warp; tile < p.n_tiles; tile += n_warps) {
    const uint64_t base = tile * kTileBlocks;
    bool valid[4];
    Lane4 t;
    load_tile<G, BF16, STRIDED>(p, base, lane, valid, t);
    rotate_tile<G>(t, lane);

    // Block amax of z, then of y = z / sqrt(G): RN(max|z| * c) = max RN(|z| * c).
    float2 zm[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float mx = 0.0f, my = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        mx = fmaxf(mx, fabsf(t.P[k][i].x));
        my = fmaxf(my, fabsf(t.P[k][i].y));
      }
      zm[k] = make_float2(mx, my);
    }

    // Block scales: v = (amax_b / 6) / s_global -> E4M3 (RNE, satfinite).
    uint32_t sb2[2];    // two E4M3 patterns per pair
    float2 sf[2];       // s_f = s_block * s_global
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float ax = __fmul_rn(zm[k].x, c);
      const float ay = __fmul_rn(zm[k].y, c);
      const float vx = __fdiv_rn(__fdiv_rn(ax, 6.0f), s_global);
      const float vy = __fdiv_rn(__fdiv_rn(ay, 6.0f), s_global);
      sb2[k] = e4m3x2(vx, vy);
      const float2 sbf = e4m3x2_to_f32(sb2[k]);
      sf[k] = make_float2(__fmul_rn(sbf.x, s_global), __fmul_rn(sbf.y, s_global));
    }

    // Fast path: q = RN(y / s_f) = RN(z / D), D = s_f * sqrt(G), by Markstein's
    // correction: r = RN(1/D), q0 = RN(z r), e = z - q0 D (exact), q = RN(q0 + e r)
    // (P. Markstein, "Computation of elementary functions on the IBM RISC
    // System/6000 processor", IBM J. Res. Dev. 34(1), 1990; the theorem that q is
    // the correctly rounded quotient when r is the correctly rounded reciprocal
    // and nothing under/overflows).  The domain s_f in [2^-96, 2^100] keeps D,
    // r, z and e normal wherever the rounding decides a code (|q| >= 1/8); a
    // smaller quotient gives code 0 with the sign of z either way, and
    // y = RN(z c) equals z c there except for values that only give such codes.
    //
    // The steps run on negated values, with nr = -r:  q0n = RN(z nr) = -q0,
    // e = RN(z + q0n D), qn = RN(q0n + e nr) = -q.  In this form qn is -q even for
    // z = +-0 (the direct form turns -0 into +0, since e = +0 and +0 + -0 = +0),
    // so code(q) = code(qn) with the sign bit flipped: one XOR per 8 codes.
    bool fast = true;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float a = sf[k].x, b = sf[k].y;
      fast &= (a == 0.0f) || (a >= 0x1p-96f && a <= 0x1p100f);
      fast &= (b == 0.0f) || (b >= 0x1p-96f && b <= 0x1p100f);
    }

    uint32_t w[4][2];  // packed codes per block: elements 0..7, 8..15
    if (fast) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float dx = (sf[k].x == 0.0f) ? 1.0f : __fmul_rn(sf[k].x, sq);
        const float dy = (sf[k].y == 0.0f) ? 1.0f : __fmul_rn(sf[k].y, sq);
        const float2 nr = make_float2(-__frcp_rn(dx), -__frcp_rn(dy));
        const float2 d = make_float2(dx, dy);
        float2 qv[16];  // -q
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 z = t.P[k][i];
          const float2 q0n = mul2(z, nr);
          const float2 e = fma2(q0n, d, z);
          qv[i] = fma2(e, nr, q0n);
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
        const float sfj = (j & 1) ? sf[j >> 1].y : sf[j >> 1].x;
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

    // Stores: 8 code bytes and 1 scale byte per block, streaming (evict-first).
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!valid[j]) continue;
      const uint64_t b = base + lane_block<G>(lane, j);
      const float sfj = (j & 1) ? sf[j >> 1].y : sf[j >> 1].x;
      const uint32_t keep = (sfj == 0.0f) ? 0u : 0xFFFFFFFFu;  // s_f == 0: all codes 0
      __stcs(reinterpret_cast<uint2*>(p.q + b * 8u), make_uint2(w[j][0] & keep, w[j][1] & keep));
      const uint32_t sbyte = (sb2[j >> 1] >> ((j & 1) * 8)) & 0xFFu;
      __stcs(reinterpret_cast<unsigned char*>(p.s + b), static_cast<unsigned char>(sbyte));
    }
  }
}

// ---------------------------------------------------------------------------
// Dequant: value = (+-grid[c]) * (s_block * s_global), then optionally the
// rotation again (y = RN(z / sqrt(G)) after the same butterfly).
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(kThreads, 2) k_dequant_nvfp4(Params p) {
  const int lane = threadIdx.x & 31;
  const uint64_t warp = (static_cast<uint64_t>(blockIdx.x) * kWarpsPerCta) + (threadIdx.x >> 5);
  const uint64_t n_warps = static_cast<uint64_t>(gridDim.x) * kWarpsPerCta;
  const float s_global = *p.dq_sglobal;
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
        const float sb = e4m3x2_to_f32(__ldg(p.dq_s + b)).x;
        s_f = __fmul_rn(sb, s_global);
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
