// hq_int8.cuh -- INT8 per-token rotate-quant (sm_103a).
//
// The second workload of the pages ("hyperflow_h3_flash_int8.py", HyperFlow:
// regular_hadamard, rotate_quant_kernel):
//   y     = x . R_G per run of G channels, R_G = kron(H4/2, ..., H4/2), G in {4, 16, 64, 256, 1024},
//           H4 = [[1,1,1,-1],[1,1,-1,1],[1,-1,1,1],[-1,1,1,1]];
//   scale = max(amax_row |y|, 1e-12) / 127, one fp32 per row;
//   q     = clamp(rint(y * (1 / scale)), -127, 127), int8.
// Evaluation order (the reading the CPU oracle defines): the Kronecker factors
// act digit by digit on the base-4 channel index, the least significant digit
// first; one 4-point step maps (v0, v1, v2, v3) to out_k = RN(S/2 - v_(3-k)),
// S = (v0 + v1) + (v2 + v3) (H4 = J - 2P, P the exchange matrix).
//
// Work decomposition.  A CTA of 16 warps handles whole rows: a row of K channels
// is T = ceil(K / 2048) warp tiles (K <= 32768; longer rows: k_rotate_quant_int8_park and
// k_rotate_quant_int8_long below).  The CTA takes rows in blocks of
// B rows, B T tiles numbered row by row, and warp w handles the tiles w, w + 16,
// ..., L of them.  For G = 64 and 256, which are bound by instruction issue,
// B = lcm(T, 16) / T and L = lcm(T, 16) / 16, so all 16 warps have work whatever T
// is (T = 14: 8 rows, 7 tiles per warp).  For G = 16, bound by memory, B =
// floor(16 / T) and L = 1: whole rows per CTA step, some warps idle when T does not
// divide 16 (finer row blocks balance the grid better).  Within a tile the
// lane holds 4 blocks of 16 channels (G = 16: blocks 32j + lane; G = 64, 256: the
// 4 lanes of a quad hold 16 consecutive blocks, lane % 4 being the block's digit
// 2 and the slot (i8_d3) its digit 3; every other lane holds the two 8-channel halves
// of its blocks swapped, i8_half).  The rotated values never go to
// global memory: between the rotation and the quantization, which needs the whole
// row's amax, they wait in tensor memory (the pipeline note at the kernel), so x
// is read once.  bf16 rows stream through the per-warp TMA ring.
//
// The 4-point steps run on negated values: new_k = fma(S, -1/2, a_(3-k)) =
// RN(a_(3-k) - S/2) = -out_k, one FFMA2 per two values and no negation; the sign
// alternates from step to step (the sum S of negated inputs is exactly -S), so
// after an odd number of steps (G = 64) the quantizer multiplies by -1/scale.
// The step on digit 2 (G = 64, 256) runs across the quad: the lanes c and c ^ 1 trade
// one half of their blocks, so that each holds both values of the pair on the other
// half, and the pair sums are traded with the lanes c ^ 2 (one shuffle per value); a
// lane then holds, on its half of each block, the outputs of digit values 3 - c and
// 3 - (c ^ 1), which relabels its registers for the stores.  Digit 3 (G >= 256) is
// in-lane, packed two positions per FADD2; digit 4 (G = 1024) pairs lanes as digit 2 does,
// on the two float2 arrays instead of the block halves.
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
  int tiles_per_row;   // T
  int rows_per_block;  // B = lcm(T, 16) / T
  int tiles_per_warp;  // L = lcm(T, 16) / 16 (per block)
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

// Which digit-3 value (block index bits 2..3 within a 256-group, or which
// 64-group of the quad for G = 64) register slot j of a lane holds, for G >= 64.
// Slot j is P[j >> 1], component j & 1; add2(P[0][i], P[1][i]) pairs digit-3 values
// {0, 1} and {2, 3}.  For G = 64 and 256 the map is the same in every lane.  For
// G = 1024 lane bit 2 (the low bit of digit 4) swaps the two float2 arrays, which the
// digit-4 step (i8_digit4_step) needs.
template <int G>
__device__ __forceinline__ int i8_d3(int lane, int j) {
  const int lb = (G == 1024) ? ((lane >> 2) & 1) : 0;
  return ((j & 1) << 1) | ((j >> 1) ^ lb);
}

// For G >= 64: 1 if the lane's registers 0..7 of a block hold its channels 8..15 (and
// registers 8..15 channels 0..7), else 0.  The lanes c and c ^ 1 of a quad differ, c and
// c ^ 2 agree (the digit-2 step needs that); for G = 64 and 256 the quads with odd index
// flip it as well, so that the 8 lanes of a quarter warp read the 32 banks once when
// they load their blocks' first 16 bytes from shared memory.  For G = 1024 the four lanes
// of a digit-4 step (l, l ^ 4, l ^ 8, l ^ 12) must agree, so it is lane bit 0 alone.
// G <= 16: 0.
template <int G>
__device__ __forceinline__ int i8_half(int lane) {
  if constexpr (G <= 16)
    return 0;
  else if constexpr (G == 1024)
    return lane & 1;
  else
    return (lane ^ (lane >> 2)) & 1;
}

// Block (of 16 channels, within the warp tile) that slot j of the lane loads.
//   G <= 16: block 32 j + lane.
//   G >= 64: the quad q = lane / 4 holds blocks 16 q .. 16 q + 15, lane % 4 being the
//   block's digit 2 and the slot's digit-3 value (i8_d3) its digit 3; for G = 1024, q % 4
//   is digit 4 and q / 4 the 1024-group of the tile.
template <int G>
__device__ __forceinline__ int i8_in_block(int lane, int j) {
  if constexpr (G <= 16)
    return 32 * j + lane;
  else
    return (lane >> 2) * 16 + (lane & 3) + 4 * i8_d3<G>(lane, j);
}

// Block that slot j holds after the rotation, in registers 0..7 (r = 0) or 8..15
// (r = 1) of the slot: each in-lane 4-point step leaves, in the register that held
// input digit value d, the output of digit value 3 - d; after the digit-2 step the
// lane's registers 0..7 hold digit value 3 - c and registers 8..15 digit value 3 - (c ^ 1)
// (c = lane % 4), each on the half i8_half of the block; after the digit-4 step (G = 1024)
// P[0] holds digit-4 value 3 - e and P[1] 3 - (e ^ 1) (e = (lane / 4) % 4).  G <= 16: the
// whole block, r = 0.
template <int G>
__device__ __forceinline__ int i8_out_block(int lane, int j, int r) {
  const int d2 = 3 ^ (lane & 3) ^ r;
  if constexpr (G <= 16)
    return 32 * j + lane;
  else if constexpr (G == 64)
    return (lane >> 2) * 16 + d2 + 4 * i8_d3<G>(lane, j);
  else if constexpr (G == 256)
    return (lane >> 2) * 16 + d2 + 4 * (3 - i8_d3<G>(lane, j));
  else  // the digit-4 step leaves P[0] and P[1] on the digit-3 values of P[0]
    return (lane >> 4) * 64 + (3 ^ ((lane >> 2) & 3) ^ (j >> 1)) * 16 + d2 + 4 * (3 - i8_d3<G>(lane, j & 1));
}

// The digit-2 step (G >= 64): the four values of a position sit in the same register of
// the lanes of a quad (digit value c = lane % 4), and the lanes c and c ^ 1 hold opposite
// halves of each block in registers 0..7 (i8_half).  The lanes c and c ^ 1 trade
// registers 8..15, so each holds v_c and v_(c ^ 1) on its own half; the pair sums are
// traded with the lanes c ^ 2, and every lane forms S = (v0 + v1) + (v2 + v3) (the two
// pair sums added in either order, the same value) and the negated outputs
// fma(S, -1/2, v_c) of digit value 3 - c and fma(S, -1/2, v_(c ^ 1)) of 3 - (c ^ 1).
// One shuffle per value.
__device__ __forceinline__ void i8_quad_step(Lane4& t) {
  const float2 nh = make_float2(-0.5f, -0.5f);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 o;  // the pair lane's value on this lane's half
      o.x = __shfl_xor_sync(0xFFFFFFFFu, t.P[k][8 + i].x, 1);
      o.y = __shfl_xor_sync(0xFFFFFFFFu, t.P[k][8 + i].y, 1);
      const float2 pr = add2(t.P[k][i], o);
      float2 q;  // the other pair's sum
      q.x = __shfl_xor_sync(0xFFFFFFFFu, pr.x, 2);
      q.y = __shfl_xor_sync(0xFFFFFFFFu, pr.y, 2);
      const float2 s = add2(pr, q);
      t.P[k][i] = fma2(s, nh, t.P[k][i]);
      t.P[k][8 + i] = fma2(s, nh, o);
    }
  }
}

// The digit-4 step (G = 1024): the four values of a position sit in the lanes l, l ^ 4,
// l ^ 8, l ^ 12 (digit value e = (lane / 4) % 4), which agree on what every register holds
// but for the digit-3 values of the two float2 arrays, swapped by lane bit 2 (i8_d3).  The
// lanes e and e ^ 1 trade P[1], so each holds v_e and v_(e ^ 1) on the digit-3 values of
// its own P[0]; the pair sums are traded with the lanes e ^ 2, and every lane forms S and
// the negated outputs fma(S, -1/2, v_e) of digit value 3 - e (into P[0]) and
// fma(S, -1/2, v_(e ^ 1)) of 3 - (e ^ 1) (into P[1]).  One shuffle per value.
__device__ __forceinline__ void i8_digit4_step(Lane4& t) {
  const float2 nh = make_float2(-0.5f, -0.5f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float2 o;  // the pair lane's value on this lane's P[0] positions
    o.x = __shfl_xor_sync(0xFFFFFFFFu, t.P[1][i].x, 4);
    o.y = __shfl_xor_sync(0xFFFFFFFFu, t.P[1][i].y, 4);
    const float2 pr = add2(t.P[0][i], o);
    float2 q;  // the other pair's sum
    q.x = __shfl_xor_sync(0xFFFFFFFFu, pr.x, 8);
    q.y = __shfl_xor_sync(0xFFFFFFFFu, pr.y, 8);
    const float2 s = add2(pr, q);
    t.P[0][i] = fma2(s, nh, t.P[0][i]);
    t.P[1][i] = fma2(s, nh, o);
  }
}

// The regular-Hadamard rotation of the lane's 4 blocks, digit by digit.
// Returns +1 if the registers hold y, -1 if they hold -y (an odd number of steps).
template <int G>
__device__ __forceinline__ float rotate_regular(Lane4& t) {
  static_assert(G == 4 || G == 16 || G == 64 || G == 256 || G == 1024, "group");
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    // digit 0: channels 4b .. 4b+3 of a block
#pragma unroll
    for (int b = 0; b < 4; ++b) h4_step(t.P[k][4 * b], t.P[k][4 * b + 1], t.P[k][4 * b + 2], t.P[k][4 * b + 3]);
    if constexpr (G >= 16) {
      // digit 1: channels b, b+4, b+8, b+12
#pragma unroll
      for (int b = 0; b < 4; ++b) h4_step(t.P[k][b], t.P[k][b + 4], t.P[k][b + 8], t.P[k][b + 12]);
    }
  }
  if constexpr (G == 4) {
    return -1.0f;
  } else if constexpr (G == 16) {
    return 1.0f;
  } else {
    i8_quad_step(t);  // digit 2: the four lanes of a quad (lane % 4)
    if constexpr (G == 64) {
      return -1.0f;
    } else {
      // digit 3: the lane's four slots; add2 pairs digit values {0,1} and {2,3}.
      const float2 nh = make_float2(-0.5f, -0.5f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 u = add2(t.P[0][i], t.P[1][i]);
        const float sum = __fadd_rn(u.x, u.y);
        const float2 s2 = make_float2(sum, sum);
        t.P[0][i] = fma2(s2, nh, t.P[0][i]);
        t.P[1][i] = fma2(s2, nh, t.P[1][i]);
      }
      if constexpr (G == 256) {
        return 1.0f;
      } else {
        i8_digit4_step(t);  // digit 4: the four quads of a 1024-group ((lane / 4) % 4)
        return -1.0f;
      }
    }
  }
}

// Four packed int8 bytes (channel order) from the magic-add results of four channels.
__device__ __forceinline__ uint32_t pack_i8x4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
}

// Channels of warp tile `chunk` inside a row of K channels (at most one tile, 2048).
__device__ __forceinline__ int i8_chunk_valid(int64_t K, int chunk) {
  const int64_t rest = K - static_cast<int64_t>(chunk) * kI8TileElems;
  return rest < kI8TileElems ? static_cast<int>(rest) : kI8TileElems;
}

// The codes q = rint(y * inv) of the lane's rotated tile t (inv2 = (inv, inv), inv the
// signed reciprocal of the row's scale) to the row's chunk qrow: blocks at or past
// `nvalid` (<= 2048) channels are not written (FULL: the caller knows the whole tile lies
// inside the row).  Block offsets are signed ints, so that the compiler may fold a
// store's fixed part into its address.  rint by the magic constant 1.5 * 2^23: |y * inv| <= 127 < 2^22, so the sum
// rounds (half to even) to an integer held, two's complement, in the low bits.  The sum
// is written fma(p, 1, magic) on the rounded product p: ptxas (CUDA 13.0, -O3) fuses a
// packed multiply whose only use is a packed add into one fused multiply-add even when
// both carry an explicit .rn, and rint of the unrounded product differs where RN(y * inv)
// is exactly k + 1/2.  G <= 16: one 16-byte store per block; G >= 64: one 8-byte store per
// half block (i8_out_block, i8_half).
template <int G, bool FULL = false>
__device__ __forceinline__ void i8_store_codes(int8_t* qrow, int lane, const Lane4& t, float2 inv2, int nvalid) {
  const float2 magic2 = make_float2(12582912.0f, 12582912.0f);
  const float2 one2 = make_float2(1.0f, 1.0f);
  auto ok = [&](int bl) { return FULL || bl * 16 < nvalid; };
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    uint32_t b[2][16];  // slots 2k and 2k + 1
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 w = fma2(mul2(t.P[k][i], inv2), one2, magic2);
      b[0][i] = __float_as_uint(w.x);
      b[1][i] = __float_as_uint(w.y);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if constexpr (G <= 16) {
        const int bl = i8_out_block<G>(lane, 2 * k + c, 0);
        if (ok(bl))
          __stcs(reinterpret_cast<uint4*>(qrow + bl * 16),
                 make_uint4(pack_i8x4(b[c][0], b[c][1], b[c][2], b[c][3]),
                            pack_i8x4(b[c][4], b[c][5], b[c][6], b[c][7]),
                            pack_i8x4(b[c][8], b[c][9], b[c][10], b[c][11]),
                            pack_i8x4(b[c][12], b[c][13], b[c][14], b[c][15])));
      } else {
        const int half = 8 * i8_half<G>(lane);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int bl = i8_out_block<G>(lane, 2 * k + c, r);
          if (ok(bl))
            __stcs(reinterpret_cast<uint2*>(qrow + (bl * 16 + half)),
                   make_uint2(pack_i8x4(b[c][8 * r], b[c][8 * r + 1], b[c][8 * r + 2], b[c][8 * r + 3]),
                              pack_i8x4(b[c][8 * r + 4], b[c][8 * r + 5], b[c][8 * r + 6], b[c][8 * r + 7])));
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Tensor memory (TMEM) for parking a rotated tile.  The CTA allocates all 512
// columns once; warp w may touch TMEM lanes 32 (w % 4) .. + 31 only, and parks a
// tile (64 fp32 values per lane) in 64 consecutive columns of its lanes.
// ---------------------------------------------------------------------------
constexpr uint32_t kI8TmemCols = 512;

__device__ __forceinline__ void tmem_alloc_all(uint32_t smem_dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst),
               "r"(kI8TmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_all(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kI8TmemCols)
               : "memory");
}

__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 64 32-bit registers of each lane -> 64 consecutive TMEM columns of its lane.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]),
        "r"(v[32]), "r"(v[33]), "r"(v[34]), "r"(v[35]), "r"(v[36]), "r"(v[37]), "r"(v[38]), "r"(v[39]),
        "r"(v[40]), "r"(v[41]), "r"(v[42]), "r"(v[43]), "r"(v[44]), "r"(v[45]), "r"(v[46]), "r"(v[47]),
        "r"(v[48]), "r"(v[49]), "r"(v[50]), "r"(v[51]), "r"(v[52]), "r"(v[53]), "r"(v[54]), "r"(v[55]),
        "r"(v[56]), "r"(v[57]), "r"(v[58]), "r"(v[59]), "r"(v[60]), "r"(v[61]), "r"(v[62]), "r"(v[63])
      : "memory");
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
        "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]),
        "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]),
        "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
        "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
      : "r"(taddr)
      : "memory");
}


__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void lane4_to_words(const Lane4& t, uint32_t (&v)[64]) {
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[32 * k + 2 * i] = __float_as_uint(t.P[k][i].x);
      v[32 * k + 2 * i + 1] = __float_as_uint(t.P[k][i].y);
    }
}

__device__ __forceinline__ void words_to_lane4(const uint32_t (&v)[64], Lane4& t) {
#pragma unroll
  for (int k = 0; k < 2; ++k)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      t.P[k][i] = make_float2(__uint_as_float(v[32 * k + 2 * i]), __uint_as_float(v[32 * k + 2 * i + 1]));
}

// One arrival on an mbarrier (release semantics at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Max of a non-negative float (or NaN with the sign bit clear) over the warp:
// such floats order like their bit patterns as unsigned integers.
__device__ __forceinline__ float warp_max_nonneg(float v) {
  return __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(v)));
}

// FULL: every warp tile of a row is complete (K a multiple of the tile), so no
// block needs a bounds check.
//
// Software pipeline.  Step i rotates this warp's tile i, publishes its amax and
// parks the rotated values in TMEM (slot i % 2); then it waits for the row of tile
// i - 1 to be complete, takes that tile back from TMEM and quantizes it.  A row's
// T tiles meet on an mbarrier (T arrivals), not a CTA barrier, so while one warp
// waits the others rotate.  Row barriers and tile maxima come in 4 sets, one per
// row block modulo 4.  A random-interleaving model of this protocol (parity-only
// waits, as the hardware checks them) finds no deadlock, no set reused before every
// warp has read it, and no barrier two phases ahead of a waiter, for every T from 1
// to 16; with 2 or 3 sets it fails.
// RR: tiles dealt round robin over the warps (L >= 1); otherwise L = 1 and each warp
// has a fixed place in the row block.
template <int G, bool BF16, int MODE, bool FULL, bool RR>
__global__ void __launch_bounds__(kI8Threads, 1) k_rotate_quant_int8(I8Params p) {
  constexpr int es = BF16 ? 2 : 4;
  constexpr int kTileBytes = kI8TileElems * es;
  constexpr int kSets = 4;
  const int lane = threadIdx.x & 31;
  // the block halves this lane loads swapped (i8_half): in 16-byte words of a block and of its
  // bf16 copy in shared memory
  const int hs = i8_half<G>(lane);
  const int hw = hs * ((BF16 ? 2 : 4) / 2);
  const int wid = threadIdx.x >> 5;
  const int T = p.tiles_per_row;
  const int B = p.rows_per_block;
  const int L = RR ? p.tiles_per_warp : 1;

  // Row barriers and tile maxima come in 4 sets, one per block modulo 4: a warp
  // reuses a set only after every warp has read it (see the pipeline note above).
  __shared__ float tile_max[kSets][kI8Warps][kI8Warps];      // [set][row in block][tile]
  __shared__ __align__(8) uint64_t row_bar[kSets][kI8Warps];  // [set][row in block], T arrivals
  __shared__ uint32_t tmem_base_slot;
  __shared__ volatile int cta_broken;  // a wait ran out somewhere in the CTA: everyone stops
  extern __shared__ __align__(1024) uint8_t hq_smem[];
  uint8_t* ring = hq_smem + wid * kI8Stages * kI8TileElems * 2;
  const uint32_t ring_s = smem_addr(ring);
  const uint32_t bar0 = smem_addr(hq_smem + kI8Warps * kI8Stages * kI8TileElems * 2) + wid * kI8Stages * 8;
  const uint64_t policy = l2_stream_policy();

  if (threadIdx.x == 0) {
    for (int st = 0; st < kSets; ++st)
      for (int b = 0; b < B; ++b) mbar_init(smem_addr(&row_bar[st][b]), static_cast<uint32_t>(T));
    cta_broken = 0;
    fence_mbar_init();
  }
  if (wid == 0) tmem_alloc_all(smem_addr(&tmem_base_slot));
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem_warp = tmem_base_slot + ((32u * static_cast<uint32_t>(wid & 3)) << 16) +
                             128u * static_cast<uint32_t>(wid >> 2);

  // Tile i of this warp: block q = i / L, tile g = wid + 16 (i % L) of the block, row
  // b = g / T of the block, chunk g % T of the row.  Cursors walk i with (q, k = i % L)
  // carried along; g / T is (g * ceil(2^16 / T)) >> 16, exact for g < 256 and T <= 16.
  struct TileRef {
    int64_t row;
    int set, parity, b, chunk;
    int64_t nvalid;  // channels of the chunk inside the row
  };
  struct Cursor {
    int64_t i, q;
    int k;
  };
  const uint32_t inv_T = (65536u + static_cast<uint32_t>(T) - 1u) / static_cast<uint32_t>(T);
  auto advance = [&](Cursor& c) {
    ++c.i;
    if (++c.k == L) {
      c.k = 0;
      ++c.q;
    }
  };
  // Without round robin (L = 1) the warp's tile of every block is the same.
  const int b1 = static_cast<int>((static_cast<uint32_t>(wid) * inv_T) >> 16);
  const int c1 = wid - b1 * T;
  auto tile = [&](const Cursor& c) {
    TileRef r;
    if constexpr (!RR) {
      r.b = b1;
      r.chunk = c1;
    } else {
      const uint32_t g = static_cast<uint32_t>(wid + 16 * c.k);
      r.b = static_cast<int>((g * inv_T) >> 16);
      r.chunk = static_cast<int>(g) - r.b * T;
    }
    r.row = (static_cast<int64_t>(blockIdx.x) + c.q * gridDim.x) * B + r.b;
    r.set = static_cast<int>(c.q & (kSets - 1));
    r.parity = static_cast<int>((c.q >> 2) & 1);
    const int64_t c0 = static_cast<int64_t>(r.chunk) * kI8TileElems;
    r.nvalid = FULL ? kI8TileElems : (p.K - c0 < kI8TileElems ? p.K - c0 : kI8TileElems);
    return r;
  };
  const int64_t row_blocks = (p.M + B - 1) / B;
  int64_t n_blocks = 0;  // row blocks of this CTA
  if (blockIdx.x < row_blocks) n_blocks = (row_blocks - blockIdx.x + gridDim.x - 1) / gridDim.x;
  // With L = 1 and B T < 16 (one tile per warp and row block) the warps past B T
  // have no tiles; otherwise B T = 16 L and every warp has L tiles per block.
  const int64_t n_it = (wid < B * T) ? n_blocks * L : 0;  // tiles of this warp

  bool broken = false;   // stop touching memory and waiting
  int64_t issued = 0;    // this warp's tiles 0 .. issued-1 handed to TMA (rows only increase
                         // with i, so once a tile lies past M every later one does too)
  Cursor ci = {0, 0, 0};  // the next tile to hand to TMA
  auto issue_ahead = [&](int64_t upto) {
    for (; ci.i < upto && ci.i < n_it; advance(ci)) {
      const TileRef r = tile(ci);
      if (r.row >= p.M) break;
      if (lane == 0)
        tma_load(ring_s + static_cast<int>(ci.i % kI8Stages) * kTileBytes,
                 p.x + r.row * p.ldx_bytes + static_cast<int64_t>(r.chunk) * kI8TileElems * es,
                 static_cast<uint32_t>(r.nvalid * es), bar0 + static_cast<int>(ci.i % kI8Stages) * 8,
                 policy);
      issued = ci.i + 1;
    }
  };
  if constexpr (MODE == kLoadTma) {
    if (lane == 0) {
      for (int st = 0; st < kI8Stages; ++st) mbar_init(bar0 + st * 8, 1);
      fence_mbar_init();
    }
    __syncwarp();
    issue_ahead(kI8Stages);
  }
  auto fail = [&](int64_t from) {  // record the fault, drain this warp's copies, stop
    if (lane == 0) atomicOr(&g_hq_fault, kFaultWaitTimeout);
    cta_broken = 1;
    if constexpr (MODE == kLoadTma)
      for (int64_t m = from; m < issued; ++m)
        mbar_wait(bar0 + static_cast<int>(m % kI8Stages) * 8, static_cast<uint32_t>((m / kI8Stages) & 1));
    broken = true;
  };

  int64_t drained_from = 0;  // first tile whose copy may still be in flight
  constexpr float kSign = (G == 4 || G == 64 || G == 1024) ? -1.0f : 1.0f;  // registers hold kSign * y
  Cursor ca = {0, 0, 0};  // tile it (rotate)
  Cursor cb = {0, 0, 0};  // tile it - 1 (quantize)
  for (int64_t it = 0; it <= n_it; ++it) {
    if (!broken && cta_broken) {
      fail(drained_from);
      break;
    }
    if (broken) break;
    // ---- A: rotate tile it, publish its amax, park it in TMEM ----
    if (it < n_it) {
      const TileRef r = tile(ca);
      advance(ca);
      const bool active = r.row < p.M;
      auto block_ok = [&](int bl) { return FULL || static_cast<int64_t>(bl) * 16 < r.nvalid; };
      Lane4 t;
      float amax = 0.0f;
      if (active) {
        if constexpr (MODE == kLoadTma) {
          const int slot = static_cast<int>(it % kI8Stages);
          const bool ok = mbar_wait(bar0 + slot * 8, static_cast<uint32_t>((it / kI8Stages) & 1));
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            fail(it);
            break;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int bl = i8_in_block<G>(lane, j);
            uint4 w4[2];
            if (block_ok(bl)) {
              const uint4* src = reinterpret_cast<const uint4*>(ring + slot * kTileBytes + bl * 32);
              w4[0] = src[hs];
              w4[1] = src[hs ^ 1];
            } else {
              w4[0] = w4[1] = make_uint4(0u, 0u, 0u, 0u);
            }
            float f[16];
            widen<true>(w4, f);
            put_block(t, j, f);
          }
          __syncwarp();
          drained_from = it + 1;
          if (lane == 0) fence_proxy_async_smem();
          issue_ahead(it + 1 + kI8Stages);
        } else {
          const uint8_t* rowp = p.x + r.row * p.ldx_bytes + static_cast<int64_t>(r.chunk) * kI8TileElems * es;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int bl = i8_in_block<G>(lane, j);
            const bool ok = block_ok(bl);
            uint4 w4[BF16 ? 2 : 4];
#pragma unroll
            for (int k = 0; k < (BF16 ? 2 : 4); ++k)
              w4[k] = ok ? __ldg(reinterpret_cast<const uint4*>(rowp + bl * 16 * es) + (k ^ hw))
                         : make_uint4(0u, 0u, 0u, 0u);
            float f[16];
            widen<BF16>(w4, f);
            put_block(t, j, f);
          }
        }
        rotate_regular<G>(t);
#pragma unroll
        for (int k = 0; k < 2; ++k)
          amax = max3_nan(amax, block_absmax<false>(t.P[k]), block_absmax<true>(t.P[k]));
        uint32_t v[64];
        lane4_to_words(t, v);
        tmem_st64(tmem_warp + 64u * static_cast<uint32_t>(it & 1), v);
      }
      amax = warp_max_nonneg(amax);
      if (lane == 0) {
        tile_max[r.set][r.b][r.chunk] = amax;
        mbar_arrive(smem_addr(&row_bar[r.set][r.b]));
      }
    }
    // ---- B: quantize tile it - 1 once its row is complete ----
    if (it >= 1) {
      const int64_t jt = it - 1;
      const TileRef r = tile(cb);
      advance(cb);
      const bool ok = mbar_wait(smem_addr(&row_bar[r.set][r.b]), static_cast<uint32_t>(r.parity));
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        fail(drained_from);
        break;
      }
      if (r.row < p.M) {
        // T <= 16: each half-warp reads the row's T tile maxima.
        const int c = lane & 15;
        const float row_amax = warp_max_nonneg(c < T ? tile_max[r.set][r.b][c] : 0.0f);
        const float scale = __fdiv_rn(fmaxf(row_amax, 1e-12f), 127.0f);
        const float inv = __fdiv_rn(1.0f, scale) * kSign;  // -inv when the registers hold -y
        if (r.chunk == 0 && lane == 0) p.scales[r.row] = scale;
        uint32_t v[64];
        tmem_wait_st();
        tmem_ld64(tmem_warp + 64u * static_cast<uint32_t>(jt & 1), v);
        tmem_wait_ld();
        Lane4 t;
        words_to_lane4(v, t);
        int8_t* qrow = p.q + r.row * p.K + static_cast<int64_t>(r.chunk) * kI8TileElems;
        i8_store_codes<G, FULL>(qrow, lane, t, make_float2(inv, inv), static_cast<int>(r.nvalid));
      }
    }
  }
  // Wait for this thread's TMEM traffic (a warp that stopped early may have a store
  // in flight), then free the columns.
  tmem_wait_st();
  tmem_wait_ld();
  tmem_fence_before_sync();
  __syncthreads();
  if (wid == 0) {
    tmem_fence_after_sync();
    tmem_dealloc_all(tmem_base_slot);
  }
}

// ---------------------------------------------------------------------------
// Rows of 17 to 59 warp tiles (32768 < K <= 120832 channels): the whole rotated row
// stays on chip until its amax is known, so x is read once and every value rotated once.
// A CTA of 16 warps takes blocks of B rows (B T <= 59; B = 2 or 3 for T <= 24, which
// evens out the warps' shares), blocks blockIdx.x, blockIdx.x + gridDim.x, ...; the
// block's tiles g = 0 .. B T - 1 (row g / T, chunk g % T) are dealt round robin, warp w
// taking g = w, w + 16, ... (its j-th: g = w + 16 j).  Tiles 0 .. 31 of a block park in
// tensor memory (two per warp, as above), tiles 32 .. in shared memory (8 KB each).
// Walk 1 loads, rotates, keeps the per-row tile amax and parks the tile; the CTA meets at
// a barrier (per row and warp one amax word, double-buffered by block parity, so a warp
// can be at most one block ahead of a reader); walk 2 takes each tile back, quantizes and
// stores it.
// Loads: with STAGES > 0 (bf16, when shared memory has room beside the parked tiles) a
// per-warp TMA ring of STAGES tiles: the warp's first STAGES tiles of a block are copied
// while the block before is in walk 2 (which reads no x), tile j + STAGES once tile j is
// parked.  A ring wait is bounded: a warp whose wait runs out records
// the fault, waits (bounded) for its copies in flight and marks the CTA broken, and
// every warp leaves after the next barrier.  STAGES = 0: 16-byte vector loads straight
// into registers.
// ---------------------------------------------------------------------------
constexpr int kI8ParkTmemTiles = 2 * kI8Warps;                          // 32
constexpr int kI8ParkTileBytes = kI8TileElems * 4;                      // 8 KB of fp32
constexpr int kI8ParkSmemTiles = 27;                                    // 216 KB
constexpr int kI8ParkMaxTiles = kI8ParkTmemTiles + kI8ParkSmemTiles;  // 59
constexpr int kI8ParkMaxRows = 3;                                       // B (T >= 17)
// Shared memory of the ring: STAGES bf16 tiles and as many mbarriers per warp.
__host__ __device__ constexpr int i8_park_ring_bytes(int stages) {
  return kI8Warps * stages * (kI8TileElems * 2 + 8);
}

// MULTI: blocks of B > 1 rows (B = 1 takes a leaner path).
template <int G, bool BF16, bool MULTI, int STAGES>
__global__ void __launch_bounds__(kI8Threads, 1) k_rotate_quant_int8_park(I8Params p) {
  static_assert(STAGES == 0 || BF16, "the ring holds bf16 tiles");
  constexpr int kRows = MULTI ? kI8ParkMaxRows : 1;
  constexpr int es = BF16 ? 2 : 4;
  constexpr int n16 = BF16 ? 2 : 4;  // 16-byte words per block of 16 channels
  constexpr int kRingTile = kI8TileElems * 2;
  constexpr float kSign = (G == 4 || G == 64 || G == 1024) ? -1.0f : 1.0f;
  const int lane = threadIdx.x & 31;
  // the block halves this lane loads swapped (i8_half): in 16-byte words of a block and of its
  // bf16 copy in shared memory
  const int hs = i8_half<G>(lane);
  const int hw = hs * ((BF16 ? 2 : 4) / 2);
  const int wid = threadIdx.x >> 5;
  const int T = p.tiles_per_row;
  const int B = MULTI ? p.rows_per_block : 1;
  const int n_g = B * T;  // tiles per block
  // g / T = (g * inv_T) >> 16, exact for g < 64 and 17 <= T <= 59
  const uint32_t inv_T = (65536u + static_cast<uint32_t>(T) - 1u) / static_cast<uint32_t>(T);
  __shared__ float row_max[2][kRows][kI8Warps];
  __shared__ uint32_t tmem_base_slot;
  __shared__ volatile int cta_broken;
  // [ring: 16 warps x STAGES tiles][ring mbarriers][tiles 32 .. n_g - 1 of a block]
  extern __shared__ __align__(1024) uint8_t hq_smem[];
  uint8_t* const park_base = hq_smem + i8_park_ring_bytes(STAGES);
  uint8_t* const ring = hq_smem + wid * STAGES * kRingTile;
  const uint32_t bar0 = smem_addr(hq_smem + kI8Warps * STAGES * kRingTile) + wid * STAGES * 8;

  if (threadIdx.x == 0) cta_broken = 0;
  if constexpr (STAGES > 0) {
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + s * 8, 1);
      fence_mbar_init();
    }
  }
  if (wid == 0) tmem_alloc_all(smem_addr(&tmem_base_slot));
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem_warp = tmem_base_slot + ((32u * static_cast<uint32_t>(wid & 3)) << 16) +
                             128u * static_cast<uint32_t>(wid >> 2);
  const int64_t n_blocks = (p.M + B - 1) / B;
  auto row_of = [&](int g) { return MULTI ? static_cast<int>((static_cast<uint32_t>(g) * inv_T) >> 16) : 0; };

  uint32_t k = 0;       // this warp's tiles read from the ring (its position)
  uint32_t issued = 0;  // lane 0: tiles handed to TMA
  // lane 0: copy the warp's j-th tile of the block whose first row is row0, if it exists,
  // into the slot the ring gives it
#define HQ_I8_PARK_FETCH(row0_, j_)                                                              \
  do {                                                                                          \
    const int g_ = wid + kI8Warps * (j_);                                                       \
    if (g_ < n_g) {                                                                             \
      const int b_ = row_of(g_);                                                                \
      if ((row0_) + b_ < p.M) {                                                                 \
        const int64_t c0_ = static_cast<int64_t>(g_ - b_ * T) * kI8TileElems;                   \
        const int64_t nv_ = p.K - c0_ < kI8TileElems ? p.K - c0_ : kI8TileElems;                \
        const int slot_ = static_cast<int>(issued % STAGES);                                    \
        tma_load(smem_addr(ring + slot_ * kRingTile), p.x + ((row0_) + b_) * p.ldx_bytes + c0_ * es, \
                 static_cast<uint32_t>(nv_ * es), bar0 + slot_ * 8, l2_stream_policy());        \
        ++issued;                                                                               \
      }                                                                                         \
    }                                                                                           \
  } while (0)
  if constexpr (STAGES > 0) {
    __syncwarp();
    if (lane == 0 && blockIdx.x < n_blocks)
      for (int j = 0; j < STAGES; ++j) HQ_I8_PARK_FETCH(static_cast<int64_t>(blockIdx.x) * B, j);
  }

  // The warp tile `chunk` of row `row` into registers (blocks past the row's end read 0;
  // `full`: the whole tile lies inside the row, and the call is written once with a
  // literal true and once with false, so each copy is compiled for its case); from the
  // ring: false if the wait ran out (the CTA is then broken).
  auto load = [&](int64_t row, int chunk, int nvalid, bool full, Lane4& t) {
    const int64_t c0 = static_cast<int64_t>(chunk) * kI8TileElems;
    if constexpr (STAGES > 0) {
      const int slot = static_cast<int>(k % STAGES);
      const bool ok = mbar_wait(bar0 + slot * 8, (k / STAGES) & 1u);
      if (!__all_sync(0xFFFFFFFFu, ok)) return false;  // handled after walk 1
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int bl = i8_in_block<G>(lane, q);
        uint4 w4[2];
        if (full || bl * 16 < nvalid) {
          const uint4* src = reinterpret_cast<const uint4*>(ring + slot * kRingTile + bl * 32);
          w4[0] = src[hs];
          w4[1] = src[hs ^ 1];
        } else {
          w4[0] = w4[1] = make_uint4(0u, 0u, 0u, 0u);
        }
        float f[16];
        widen<true>(w4, f);
        put_block(t, q, f);
      }
      __syncwarp();  // every lane has read the slot (refilled after the tile is parked)
      ++k;
    } else {
      const uint8_t* src = p.x + row * p.ldx_bytes + c0 * es;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int bl = i8_in_block<G>(lane, q);
        uint4 w4[n16];
        const bool ok = full || bl * 16 < nvalid;
#pragma unroll
        for (int e = 0; e < n16; ++e)
          w4[e] = ok ? __ldg(reinterpret_cast<const uint4*>(src + bl * 16 * es) + (e ^ hw)) : make_uint4(0u, 0u, 0u, 0u);
        float f[16];
        widen<BF16>(w4, f);
        put_block(t, q, f);
      }
    }
    return true;
  };
  // Tile g of the block in its place: TMEM slot g / 16 of this warp for g < 32, else
  // shared-memory slot g - 32, 16 float4 per lane, float4 i of lane l at 16 (32 i + l) (each
  // warp-wide 16-byte access covers 512 consecutive bytes).
  auto park = [&](int g, const Lane4& t) {
    uint32_t v[64];
    lane4_to_words(t, v);
    if (g < kI8ParkTmemTiles) {
      tmem_st64(tmem_warp + 64u * static_cast<uint32_t>(g >> 4), v);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(park_base + (g - kI8ParkTmemTiles) * kI8ParkTileBytes) + lane;
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[32 * i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  };
  auto unpark = [&](int g, Lane4& t) {
    uint32_t v[64];
    if (g < kI8ParkTmemTiles) {
      tmem_ld64(tmem_warp + 64u * static_cast<uint32_t>(g >> 4), v);
      tmem_wait_ld();
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(park_base + (g - kI8ParkTmemTiles) * kI8ParkTileBytes) + lane;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint4 w = src[32 * i];
        v[4 * i] = w.x;
        v[4 * i + 1] = w.y;
        v[4 * i + 2] = w.z;
        v[4 * i + 3] = w.w;
      }
    }
    words_to_lane4(v, t);
  };

  int64_t n = 0;
  for (int64_t blk = blockIdx.x; blk < n_blocks; blk += gridDim.x, ++n) {
    const int64_t row0 = blk * B;
    // walk 1: rotate, the per-row tile amax, park
    float amax[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) amax[r] = 0.0f;
    int j = 0;
    bool timed_out = false;
    for (int g = wid; g < n_g; g += kI8Warps, ++j) {
      const int b = row_of(g);
      if (MULTI && row0 + b >= p.M) break;  // rows past the end: every later g is past it too
      Lane4 t;
      const int chunk = g - b * T;
      const int nvalid = i8_chunk_valid(p.K, chunk);
      bool loaded;
      if constexpr (STAGES > 0)  // shared-memory reads: the block checks cost little
        loaded = load(row0 + b, chunk, nvalid, false, t);
      else
        loaded = nvalid == kI8TileElems ? load(row0 + b, chunk, nvalid, true, t)
                                        : load(row0 + b, chunk, nvalid, false, t);
      if (!loaded) {
        timed_out = true;
        break;
      }
      rotate_regular<G>(t);
      float m = 0.0f;
#pragma unroll
      for (int q = 0; q < 2; ++q) m = max3_nan(m, block_absmax<false>(t.P[q]), block_absmax<true>(t.P[q]));
#pragma unroll
      for (int r = 0; r < kRows; ++r)
        if (r == b) amax[r] = max_nan(amax[r], m);
      park(g, t);
      if constexpr (STAGES > 0) {  // the slot this tile came from takes tile j + STAGES
        if (lane == 0) {
          fence_proxy_async_smem();
          HQ_I8_PARK_FETCH(row0, j + STAGES);
        }
      }
    }
    if constexpr (STAGES > 0) {
      if (timed_out) {  // record it, wait (bounded) for this warp's copies still in flight
        if (lane == 0) atomicOr(&g_hq_fault, kFaultWaitTimeout);
        const uint32_t n_issued = __shfl_sync(0xFFFFFFFFu, issued, 0);
        for (uint32_t m = k; m < n_issued; ++m)
          mbar_wait(bar0 + static_cast<int>(m % STAGES) * 8, (m / STAGES) & 1u);
        cta_broken = 1;
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const float a = warp_max_nonneg(amax[r]);
      if (lane == 0) row_max[n & 1][r][wid] = a;
    }
    tmem_wait_st();  // this thread's parked columns are written before it reads them back
    __syncthreads();
    if (cta_broken) break;  // the same in every thread after the barrier
    if constexpr (STAGES > 0) {  // the next block's first tiles, while this one is in walk 2
      if (lane == 0 && blk + gridDim.x < n_blocks)
        for (int a = 0; a < STAGES; ++a) HQ_I8_PARK_FETCH((blk + gridDim.x) * B, a);
    }
    float inv[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const float row_amax = warp_max_nonneg(lane < kI8Warps ? row_max[n & 1][r][lane] : 0.0f);
      const float scale = __fdiv_rn(fmaxf(row_amax, 1e-12f), 127.0f);
      inv[r] = __fdiv_rn(1.0f, scale) * kSign;  // -inv when the registers hold -y
      if (threadIdx.x == 0 && r < B && row0 + r < p.M) p.scales[row0 + r] = scale;
    }
    // walk 2: the codes
    for (int g = wid; g < n_g; g += kI8Warps) {
      const int b = row_of(g);
      if (MULTI && row0 + b >= p.M) break;
      const int chunk = g - b * T;
      float inv_b = inv[0];
#pragma unroll
      for (int r = 1; r < kRows; ++r)
        if (r == b) inv_b = inv[r];
      const float2 inv2 = make_float2(inv_b, inv_b);
      Lane4 t;
      unpark(g, t);
      int8_t* const qrow = p.q + (row0 + b) * p.K + static_cast<int64_t>(chunk) * kI8TileElems;
      const int nvalid = i8_chunk_valid(p.K, chunk);
      if (nvalid == kI8TileElems)
        i8_store_codes<G, true>(qrow, lane, t, inv2, nvalid);
      else
        i8_store_codes<G, false>(qrow, lane, t, inv2, nvalid);
    }
  }
  // Every thread's TMEM traffic is complete before the columns are freed.
  tmem_wait_st();
  tmem_wait_ld();
  tmem_fence_before_sync();
  __syncthreads();
  if (wid == 0) {
    tmem_fence_after_sync();
    tmem_dealloc_all(tmem_base_slot);
  }
}
#undef HQ_I8_PARK_FETCH

// ---------------------------------------------------------------------------
// Rows longer than the chip can park (K > 120832 channels).  A CTA of 16 warps takes
// rows blockIdx.x, blockIdx.x + gridDim.x, ...; warp w takes the warp tiles w, w + 16,
// ... of a row (at least one each, since T > 16).  Each row is read twice: the first
// walk rotates the tiles and keeps only their amax; the CTA meets at a barrier (the
// row's amax, one word per warp, double-buffered by row parity, so a warp can be at
// most one row ahead of a reader); the second walk reads the tiles again, rotates and
// quantizes them.  The second read mostly hits L2 (a row's x is K * 2 or 4 bytes per
// CTA).  Loads are 16-byte vector loads straight into registers (contiguous or
// strided rows alike); nothing waits except the CTA barrier, so no bound is needed.
// ---------------------------------------------------------------------------
template <int G, bool BF16>
__global__ void __launch_bounds__(kI8Threads, 1) k_rotate_quant_int8_long(I8Params p) {
  constexpr int es = BF16 ? 2 : 4;
  constexpr int n16 = BF16 ? 2 : 4;  // 16-byte words per block of 16 channels
  constexpr float kSign = (G == 4 || G == 64 || G == 1024) ? -1.0f : 1.0f;
  const int lane = threadIdx.x & 31;
  // the block halves this lane loads swapped (i8_half): in 16-byte words of a block and of its
  // bf16 copy in shared memory
  const int hs = i8_half<G>(lane);
  const int hw = hs * ((BF16 ? 2 : 4) / 2);
  const int wid = threadIdx.x >> 5;
  const int T = p.tiles_per_row;
  __shared__ float row_max[2][kI8Warps];

  // The warp tile `chunk` of row `row` into registers (blocks past the row's end read 0;
  // `full` as in k_rotate_quant_int8_park).
  auto load = [&](int64_t row, int chunk, int nvalid, bool full, Lane4& t) {
    const int64_t c0 = static_cast<int64_t>(chunk) * kI8TileElems;
    const uint8_t* src = p.x + row * p.ldx_bytes + c0 * es;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int bl = i8_in_block<G>(lane, j);
      uint4 w4[n16];
      const bool ok = full || bl * 16 < nvalid;
#pragma unroll
      for (int k = 0; k < n16; ++k)
        w4[k] = ok ? __ldg(reinterpret_cast<const uint4*>(src + bl * 16 * es) + (k ^ hw)) : make_uint4(0u, 0u, 0u, 0u);
      float f[16];
      widen<BF16>(w4, f);
      put_block(t, j, f);
    }
  };

  int64_t n = 0;
  for (int64_t row = blockIdx.x; row < p.M; row += gridDim.x, ++n) {
    // walk 1: the row's amax
    float amax = 0.0f;
    for (int chunk = wid; chunk < T; chunk += kI8Warps) {
      Lane4 t;
      const int nvalid = i8_chunk_valid(p.K, chunk);
      if (nvalid == kI8TileElems)
        load(row, chunk, nvalid, true, t);
      else
        load(row, chunk, nvalid, false, t);
      rotate_regular<G>(t);
#pragma unroll
      for (int k = 0; k < 2; ++k)
        amax = max3_nan(amax, block_absmax<false>(t.P[k]), block_absmax<true>(t.P[k]));
    }
    amax = warp_max_nonneg(amax);
    if (lane == 0) row_max[n & 1][wid] = amax;
    __syncthreads();
    const float row_amax = warp_max_nonneg(lane < kI8Warps ? row_max[n & 1][lane] : 0.0f);
    const float scale = __fdiv_rn(fmaxf(row_amax, 1e-12f), 127.0f);
    const float inv = __fdiv_rn(1.0f, scale) * kSign;  // -inv when the registers hold -y
    if (threadIdx.x == 0) p.scales[row] = scale;
    // walk 2: the codes
    const float2 inv2 = make_float2(inv, inv);
    for (int chunk = wid; chunk < T; chunk += kI8Warps) {
      Lane4 t;
      int8_t* const qrow = p.q + row * p.K + static_cast<int64_t>(chunk) * kI8TileElems;
      const int nvalid = i8_chunk_valid(p.K, chunk);
      if (nvalid == kI8TileElems) {
        load(row, chunk, nvalid, true, t);
        rotate_regular<G>(t);
        i8_store_codes<G, true>(qrow, lane, t, inv2, nvalid);
      } else {
        load(row, chunk, nvalid, false, t);
        rotate_regular<G>(t);
        i8_store_codes<G, false>(qrow, lane, t, inv2, nvalid);
      }
    }
  }
}

}  // namespace hq
