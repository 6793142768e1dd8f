// hq_int8.cuh -- INT8 per-token rotate-quant (sm_103a).
//
// The second workload of the pages ("hyperflow_h3_flash_int8.py", HyperFlow:
// regular_hadamard, rotate_quant_kernel):
//   y     = x . R_G per run of G channels, R_G = kron(H4/2, ..., H4/2), G in {16, 64, 256},
//           H4 = [[1,1,1,-1],[1,1,-1,1],[1,-1,1,1],[-1,1,1,1]];
//   scale = max(amax_row |y|, 1e-12) / 127, one fp32 per row;
//   q     = clamp(rint(y * (1 / scale)), -127, 127), int8.
// Evaluation order (the reading the CPU oracle defines): the Kronecker factors
// act digit by digit on the base-4 channel index, the least significant digit
// first; one 4-point step maps (v0, v1, v2, v3) to out_k = RN(S/2 - v_(3-k)),
// S = (v0 + v1) + (v2 + v3) (H4 = J - 2P, P the exchange matrix).
//
// Work decomposition.  A CTA of 16 warps handles whole rows: a row of K channels
// is T = ceil(K / 2048) warp tiles (K <= 32768), the CTA takes R = 16 / T rows at
// a time, and warp w handles tile (w mod T) of row (w / T).  Within a tile the
// lane holds 4 blocks of 16 channels as in the NVFP4 kernels (G = 16: blocks
// 32j + lane; G = 64, 256: blocks 16*(lane/4) + lane%4 + 4j, so the 4 lanes of a
// quad hold 16 consecutive blocks).  Every value stays in registers from load to
// store: the row's amax is reduced through shared memory between the two
// halves, so x is read once.  bf16 rows stream through the per-warp TMA ring.
//
// The 4-point steps run on negated values: new_k = fma(S, -1/2, a_(3-k)) =
// RN(a_(3-k) - S/2) = -out_k, one FFMA2 per two values and no negation; the sign
// alternates from step to step (the sum S of negated inputs is exactly -S), so
// after an odd number of steps (G = 64) the quantizer multiplies by -1/scale.
// The step on digit 2 (G = 64, 256) runs across the quad: S comes from two
// xor-shuffles, and each lane keeps its own input a_c and produces the output of
// digit value 3 - c, which relabels the lane's block for the stores.
#pragma once

#include "hq_kernels.cuh"

namespace hq {

constexpr int kI8Warps = 16;
constexpr int kI8Threads = kI8Warps * 32;
constexpr int kI8TileElems = kTileBlocks * 16;  // 2048 channels per warp tile
constexpr int kI8MaxK = kI8Warps * kI8TileElems;  // 32768
constexpr int kI8Stages = 2;                      // TMA ring depth per warp (bf16)
constexpr int kI8RingBytes = kI8Warps * kI8Stages * kI8TileElems * 2 + kI8Warps * kI8Stages * 8;

struct I8Params {
  const uint8_t* x;
  int64_t ldx_bytes;
  int64_t M;
  int64_t K;
  int tiles_per_row;  // T
  int rows_per_iter;  // R
  int8_t* q;          // [M, K]
  float* scales;      // [M]
};

// One negated 4-point step on four float2 values (in place): a_k <- fma(S, -1/2, a_(3-k)).
__device__ __forceinline__ void h4_step(float2& a0, float2& a1, float2& a2, float2& a3) {
  const float2 s = add2(add2(a0, a1), add2(a2, a3));
  const float2 nh = make_float2(-0.5f, -0.5f);
  const float2 n0 = fma2(s, nh, a3);
  const float2 n1 = fma2(s, nh, a2);
  const float2 n2 = fma2(s, nh, a1);
  const float2 n3 = fma2(s, nh, a0);
  a0 = n0;
  a1 = n1;
  a2 = n2;
  a3 = n3;
}

// The regular-Hadamard rotation of the lane's 4 blocks, digit by digit.
// Returns +1 if the registers hold y, -1 if they hold -y.
template <int G>
__device__ __forceinline__ float rotate_regular(Lane4& t, int lane) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    // digit 0: channels 4b .. 4b+3 of a block
#pragma unroll
    for (int b = 0; b < 4; ++b) h4_step(t.P[k][4 * b], t.P[k][4 * b + 1], t.P[k][4 * b + 2], t.P[k][4 * b + 3]);
    // digit 1: channels b, b+4, b+8, b+12
#pragma unroll
    for (int b = 0; b < 4; ++b) h4_step(t.P[k][b], t.P[k][b + 4], t.P[k][b + 8], t.P[k][b + 12]);
  }
  if constexpr (G == 16) {
    return 1.0f;
  } else {
    // digit 2: the 4 blocks of the quad (lane % 4 is the digit), values now
    // carry their true sign again (two negated steps).
    const float2 nh = make_float2(-0.5f, -0.5f);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 a = t.P[k][i];
        float2 p;
        p.x = __shfl_xor_sync(0xFFFFFFFFu, a.x, 1);
        p.y = __shfl_xor_sync(0xFFFFFFFFu, a.y, 1);
        const float2 u = add2(a, p);  // v0 + v1 on lanes 0,1; v2 + v3 on lanes 2,3
        float2 w;
        w.x = __shfl_xor_sync(0xFFFFFFFFu, u.x, 2);
        w.y = __shfl_xor_sync(0xFFFFFFFFu, u.y, 2);
        const float2 s = add2(u, w);  // (v0 + v1) + (v2 + v3) on every lane
        t.P[k][i] = fma2(s, nh, a);   // -out of digit value 3 - (lane % 4)
      }
    }
    if constexpr (G == 64) {
      return -1.0f;
    } else {
      // digit 3: the lane's register blocks j = 0..3 (P[0].x, P[0].y, P[1].x, P[1].y)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a0 = t.P[0][i].x, a1 = t.P[0][i].y, a2 = t.P[1][i].x, a3 = t.P[1][i].y;
        const float s = __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3));
        t.P[0][i].x = __fmaf_rn(s, -0.5f, a3);
        t.P[0][i].y = __fmaf_rn(s, -0.5f, a2);
        t.P[1][i].x = __fmaf_rn(s, -0.5f, a1);
        t.P[1][i].y = __fmaf_rn(s, -0.5f, a0);
      }
      return 1.0f;
    }
  }
}

// Block index (within the tile) that the lane's register block j holds after the
// rotation (the digit-2 step relabels the quad's blocks c -> 3 - c).
template <int G>
__device__ __forceinline__ uint32_t i8_out_block(int lane, int j) {
  if constexpr (G == 16)
    return static_cast<uint32_t>(32 * j + lane);
  else
    return static_cast<uint32_t>((lane >> 2) * 16 + 4 * j + (3 - (lane & 3)));
}

template <int G>
__device__ __forceinline__ uint32_t i8_in_block(int lane, int j) {
  return lane_block<G == 16 ? 16 : 256>(lane, j);
}

// Low byte of rint(v) for |v| < 2^22: adding 1.5 * 2^23 rounds to an integer
// (half to even) and leaves it in the low mantissa bits, two's complement.
__device__ __forceinline__ uint32_t int8_bits(float v) {
  return __float_as_uint(__fadd_rn(v, 12582912.0f));
}

template <int G, bool BF16, int MODE>
__global__ void __launch_bounds__(kI8Threads, 1) k_rotate_quant_int8(I8Params p) {
  constexpr int es = BF16 ? 2 : 4;
  constexpr int kTileBytes = kI8TileElems * es;
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int T = p.tiles_per_row;
  const int R = p.rows_per_iter;
  const int row_local = wid / T;
  const int chunk = wid % T;
  const bool has_role = row_local < R;
  const int64_t chunk0 = static_cast<int64_t>(chunk) * kI8TileElems;
  const int64_t nvalid = has_role ? (p.K - chunk0 < kI8TileElems ? p.K - chunk0 : kI8TileElems) : 0;

  __shared__ float tile_max[kI8Warps];
  extern __shared__ __align__(1024) uint8_t hq_smem[];
  uint8_t* ring = hq_smem + wid * kI8Stages * kI8TileElems * 2;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar0 = smem_addr(hq_smem + kI8Warps * kI8Stages * kI8TileElems * 2) + wid * kI8Stages * 8;
  const uint64_t policy = l2_stream_policy();

  auto row_of = [&](int64_t it) -> int64_t {
    return (static_cast<int64_t>(blockIdx.x) + it * gridDim.x) * R + row_local;
  };
  auto issue = [&](int64_t it) {  // TMA copy of this warp's tile of iteration it
    const int64_t r = row_of(it);
    tma_load(ring_s + static_cast<int>(it % kI8Stages) * kTileBytes,
             p.x + r * p.ldx_bytes + chunk0 * es, static_cast<uint32_t>(nvalid * es),
             bar0 + static_cast<int>(it % kI8Stages) * 8, policy);
  };
  auto mine = [&](int64_t it) { return has_role && row_of(it) < p.M; };

  bool broken = false;   // a wait timed out: stop touching memory, keep the barriers
  int64_t issued = 0;    // this warp's iterations handed to TMA: 0 .. issued-1
  if constexpr (MODE == kLoadTma) {
    if (lane == 0) {
      for (int s = 0; s < kI8Stages; ++s) mbar_init(bar0 + s * 8, 1);
      fence_mbar_init();
    }
    __syncwarp();
    for (int s = 0; s < kI8Stages; ++s) {
      if (!mine(s)) break;  // mine() is monotone in the iteration
      if (lane == 0) issue(s);
      issued = s + 1;
    }
  }

  const int64_t first_rows = static_cast<int64_t>(blockIdx.x) * R;
  for (int64_t it = 0; first_rows + it * gridDim.x * R < p.M; ++it) {
    const int64_t r = row_of(it);
    const bool active = mine(it);
    Lane4 t;
    bool valid[4];
    float sign = 1.0f;
    float amax = 0.0f;
    if (active) {
      if constexpr (MODE == kLoadTma) {
        const int slot = static_cast<int>(it % kI8Stages);
        const bool ok = !broken && mbar_wait(bar0 + slot * 8, static_cast<uint32_t>((it / kI8Stages) & 1));
        if (!broken && !__all_sync(0xFFFFFFFFu, ok)) {
          if (lane == 0) atomicOr(&g_hq_fault, kFaultWaitTimeout);
          // wait (bounded) for the copies still in flight: iterations it .. issued-1
          for (int64_t m = it; m < issued; ++m)
            mbar_wait(bar0 + static_cast<int>(m % kI8Stages) * 8, static_cast<uint32_t>((m / kI8Stages) & 1));
          broken = true;
        }
        if (!broken) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t bl = i8_in_block<G>(lane, j);
            valid[j] = static_cast<int64_t>(bl) * 16 < nvalid;
            uint4 w4[2];
            if (valid[j]) {
              const uint4* src = reinterpret_cast<const uint4*>(ring + slot * kTileBytes + bl * 32u);
              w4[0] = src[0];
              w4[1] = src[1];
            } else {
              w4[0] = w4[1] = make_uint4(0u, 0u, 0u, 0u);
            }
            float f[16];
            widen<true>(w4, f);
            put_block(t, j, f);
          }
          __syncwarp();
          if (mine(it + kI8Stages)) {
            if (lane == 0) {
              fence_proxy_async_smem();
              issue(it + kI8Stages);
            }
            issued = it + kI8Stages + 1;
          }
        }
      } else {
        const uint8_t* rowp = p.x + r * p.ldx_bytes + chunk0 * es;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t bl = i8_in_block<G>(lane, j);
          valid[j] = static_cast<int64_t>(bl) * 16 < nvalid;
          uint4 w4[BF16 ? 2 : 4];
#pragma unroll
          for (int k = 0; k < (BF16 ? 2 : 4); ++k)
            w4[k] = valid[j] ? __ldg(reinterpret_cast<const uint4*>(rowp + bl * 16u * es) + k)
                             : make_uint4(0u, 0u, 0u, 0u);
          float f[16];
          widen<BF16>(w4, f);
          put_block(t, j, f);
        }
      }
      if (!broken) {
        sign = rotate_regular<G>(t, lane);
#pragma unroll
        for (int k = 0; k < 2; ++k)
          amax = max3_nan(amax, block_absmax<false>(t.P[k]), block_absmax<true>(t.P[k]));
      }
    }
    // amax of the row: warp max, then the row's T warps through shared memory.
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = max_nan(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
    if (lane == 0) tile_max[wid] = amax;
    __syncthreads();
    if (active && !broken) {
      float row_amax = tile_max[row_local * T];
      for (int c = 1; c < T; ++c) row_amax = max_nan(row_amax, tile_max[row_local * T + c]);
      const float scale = __fdiv_rn(fmaxf(row_amax, 1e-12f), 127.0f);
      const float inv = __fdiv_rn(1.0f, scale) * sign;  // -inv when the registers hold -y
      if (chunk == 0 && lane == 0) p.scales[r] = scale;
      const float2 inv2 = make_float2(inv, inv);
      int8_t* qrow = p.q + r * p.K + chunk0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t bo = i8_out_block<G>(lane, j);
        if (static_cast<int64_t>(bo) * 16 >= nvalid) continue;
        uint32_t w[4];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          uint32_t b[4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const float2 pr = t.P[j >> 1][4 * k4 + u];
            const float2 pr1 = t.P[j >> 1][4 * k4 + u + 1];
            const float2 v = mul2(make_float2((j & 1) ? pr.y : pr.x, (j & 1) ? pr1.y : pr1.x), inv2);
            b[u] = int8_bits(v.x);
            b[u + 1] = int8_bits(v.y);
          }
          w[k4] = __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
        }
        __stcs(reinterpret_cast<uint4*>(qrow + bo * 16u), make_uint4(w[0], w[1], w[2], w[3]));
      }
    }
    __syncthreads();  // tile_max is reused by the next iteration
  }
}

}  // namespace hq
