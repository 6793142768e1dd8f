// hq_oracle.cpp -- CPU oracle for the fused Hadamard rotation + NVFP4 quantization.
//
// TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
// definition that the CUDA library is checked against.  Only the tests, the
// smoke check and the benchmark's CPU-baseline leg load it.  It shares no code,
// header, table or constant with the CUDA library, and the library never calls it.
//
// Build: g++ -O2 -ffp-contract=off (no fast-math), scalar fp32 arithmetic, so
// every float operation below is one IEEE-754 binary32 operation rounded to
// nearest-even, in exactly the order written.
//
// Sources (the method):
//   [P1] "A Fused Hadamard + NVFP4 Quantization Kernel in Triton"
//        §1 "The format, precisely" (format table; rotation paragraph),
//        §2 "The kernel" (hadamard16, _e2m1_code, _round_e4m3, quantize, dequantize),
//        §3 "Bit-exact against a reference" (reference(): RNE float8 cast),
//        §4 "The trap: trusting the downcast" (E4M3 rounding examples).
//   [P4] "NVFP4 Quantization" (Atlas docs), "The numeric format" (storage
//        layout [N,K/2] codes, [N,K/16] E4M3 scales along K) and the software
//        E2M1 section (sign taken from the fp32 sign bit).
//
// Readings adopted where the pages are silent or disagree (all listed in the
// design notes):
//   * rotation order: stages h = 1, 2, 4, ..., G/2 in that order, then one
//     multiply by 1/sqrt(G) (0.25 for G=16, 0.0625 for G=256);
//   * H256 is the Sylvester matrix H16 (x) H16 with +-1 entries, scaled by 1/16;
//   * s_global = amax / 2688 in one fp32 division (the [P1] §1 table form),
//     replaced by 1.0 when the quotient is 0 ([P1] §2 quantize: "or 1.0");
//   * block scale rounding is round-to-nearest-even onto E4M3, saturating at 448;
//   * a block whose reconstructed scale s_f is 0 gets all-zero codes;
//   * E2M1 ties go to the even code ([P1] §2 _e2m1_code); the sign nibble bit
//     copies the sign bit of the quotient (as [P4]), so -0.0 encodes as 0x8;
//   * a quotient beyond 6 saturates to magnitude code 7.
//
// Parity pins (what ties this file to something other than itself) are the
// "not gpu" tests: Sylvester H vs scipy.linalg.hadamard, H.H^T = I, exhaustive
// E2M1/E4M3 checks against independent rules and torch's float8_e4m3fn cast,
// the [P1] §3/§5 printed error figures, closed forms and brute force.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Element types.  bf16 -> fp32 widening is exact: the bf16 bits are the top 16
// bits of the fp32 pattern.
// ---------------------------------------------------------------------------
enum { DT_F32 = 0, DT_BF16 = 1 };

inline float bits_to_float(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

inline float load_elem(const void* x, int dtype, int64_t idx) {
  if (dtype == DT_BF16) {
    uint16_t h;
    std::memcpy(&h, static_cast<const uint8_t*>(x) + 2 * idx, 2);
    return bits_to_float(static_cast<uint32_t>(h) << 16);
  }
  float f;
  std::memcpy(&f, static_cast<const uint8_t*>(x) + 4 * idx, 4);
  return f;
}

// ---------------------------------------------------------------------------
// Rotation.  [P1] §1: y = x . H / sqrt(G) with H the Sylvester-Hadamard matrix
// (built by H <- [[H, H], [H, -H]]), orthonormal and symmetric after scaling.
// Written as the in-place fast Walsh-Hadamard butterfly, stage h = 1, 2, 4, ...
// Each stage maps (z[i], z[i+h]) -> (z[i] + z[i+h], z[i] - z[i+h]) for every i
// with bit h clear.  For G=256 the first four stages act inside each run of 16
// (the H16 factor on the inner index) and the last four across the 16 runs
// (the H16 factor on the outer index), i.e. H256 = H16 (x) H16.
// ---------------------------------------------------------------------------
void rotate_group(float* z, int G) {
  if (G == 0) return;  // rotation off: y = x
  for (int h = 1; h < G; h *= 2) {
    for (int i = 0; i < G; ++i) {
      if ((i & h) == 0) {
        const float u = z[i];
        const float v = z[i + h];
        z[i] = u + v;
        z[i + h] = u - v;
      }
    }
  }
  const float inv_sqrt_g = (G == 16) ? 0.25f : 0.0625f;  // 1/4 or 1/16, exact
  for (int i = 0; i < G; ++i) z[i] = z[i] * inv_sqrt_g;
}

// ---------------------------------------------------------------------------
// E2M1 code.  [P1] §2 _e2m1_code: the magnitude code is the number of grid
// midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0 that |q| exceeds, with '>'
// at the midpoints whose lower neighbour has the even code (0, 1, 2 -> codes
// 0, 2, 4, 6 are even) and '>=' at the others, so exact ties land on the even
// code.  Anything above 5.0 is code 7 (value 6): saturation.
// Sign: bit 3 copies the fp32 sign bit of q ([P4] software E2M1).
// ---------------------------------------------------------------------------
uint8_t e2m1_code(float q) {
  const float a = std::fabs(q);
  int c = 0;
  c += (a > 0.25f);
  c += (a >= 0.75f);
  c += (a > 1.25f);
  c += (a >= 1.75f);
  c += (a > 2.5f);
  c += (a >= 3.5f);
  c += (a > 5.0f);
  if (std::signbit(q)) c |= 8;
  return static_cast<uint8_t>(c);
}

// E2M1 magnitude grid, [P1] §1 table: {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
const float kE2M1Grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

// ---------------------------------------------------------------------------
// E4M3 (float8 e4m3fn): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
// smallest normal 2^-6, subnormal spacing 2^-9, largest finite 448
// (exponent field 15, mantissa 6); 0x7F is NaN.  [P1] §2 _round_e4m3 gives the
// quantum 2^(max(floor(log2 v), -6) - 3); [P1] §3 rounds with the
// round-to-nearest-even float8 cast, and [P1] §2 clamps to 448.
// ---------------------------------------------------------------------------
uint8_t e4m3_rne_code(float v) {
  if (std::isnan(v)) return 0x7F;
  if (!(v > 0.0f)) return 0x00;             // v == 0 (scales are never negative)
  if (v >= 448.0f) return 0x7E;             // saturate (covers +inf)
  int e2;
  std::frexp(v, &e2);                       // v = m * 2^e2, m in [0.5, 1)
  int e = e2 - 1;                           // v in [2^e, 2^(e+1))
  if (e < -6) e = -6;                       // subnormal range shares the 2^-9 quantum
  const int qexp = e - 3;                   // quantum Q = 2^qexp
  // v / Q is exact (power-of-two scaling of a value far from the fp32 limits
  // for every v that can reach this line); rint rounds half to even.
  const float n = std::rint(std::ldexp(v, -qexp));
  int ni = static_cast<int>(n);             // 0 .. 16
  int ef;
  int mant;
  if (ni == 0) return 0x00;
  if (ni == 16) {                           // rounded up into the next binade
    ni = 8;
    e += 1;
  }
  if (ni < 8) {                             // subnormal: only possible for e == -6
    ef = 0;
    mant = ni;
  } else {
    ef = e + 7;
    mant = ni - 8;
  }
  if (ef > 15 || (ef == 15 && mant > 6)) return 0x7E;  // beyond 448 -> 448
  return static_cast<uint8_t>((ef << 3) | mant);
}

float e4m3_value(uint8_t code) {
  const int ef = (code >> 3) & 0xF;
  const int mant = code & 0x7;
  float mag;
  if (ef == 0)
    mag = std::ldexp(static_cast<float>(mant), -9);
  else
    mag = std::ldexp(static_cast<float>(8 + mant), ef - 7 - 3);
  return (code & 0x80) ? -mag : mag;
}

// |a| > m, or a NaN: the running maximum keeps a NaN once it has seen one, so a
// non-finite input shows up in amax.
inline float amax_update(float m, float a) {
  if (std::isnan(m)) return m;
  if (std::isnan(a) || a > m) return a;
  return m;
}

// Rotate one row's worth of groups: yrow[k] for k in [0, K).
void rotate_row(const void* x, int dtype, int64_t row, int64_t K, int64_t ldx, int group,
                float* yrow) {
  for (int64_t k = 0; k < K; ++k) yrow[k] = load_elem(x, dtype, row * ldx + k);
  if (group > 0)
    for (int64_t g0 = 0; g0 < K; g0 += group) rotate_group(yrow + g0, group);
}

template <typename F>
void parallel_rows(int64_t M, int nthreads, F&& f) {
  if (nthreads <= 1 || M < 2) {
    f(0, M, 0);
    return;
  }
  const int64_t nt = std::min<int64_t>(nthreads, M);
  std::vector<std::thread> pool;
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t r0 = M * t / nt;
    const int64_t r1 = M * (t + 1) / nt;
    pool.emplace_back([&f, r0, r1, t] { f(r0, r1, static_cast<int>(t)); });
  }
  for (auto& th : pool) th.join();
}

bool shape_ok(int64_t M, int64_t K, int64_t ldx, int group) {
  if (M < 0 || K < 0 || ldx < K) return false;
  if (!(group == 0 || group == 16 || group == 256)) return false;
  const int64_t unit = group > 16 ? group : 16;
  return K % unit == 0;
}

// Global scale, [P1] §1 table: s_global = global_amax / (448 * 6); [P1] §2
// quantize replaces a zero quotient by 1.0.
float global_scale(float amax) {
  const float s = amax / 2688.0f;
  return (s == 0.0f) ? 1.0f : s;
}

}  // namespace

extern "C" {

// Status codes of the oracle entry points.
enum { HQO_OK = 0, HQO_ERR_ARG = 1 };

// y = rotation of each row (groups of `group` along the row); amax = max |y|
// over the whole tensor.  y_out (fp32 [M,K], row stride K) may be null.
int hqo_rot_amax(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, int group,
                 float* amax_out, float* y_out, int nthreads) {
  if (!x || !amax_out || !shape_ok(M, K, ldx, group)) return HQO_ERR_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return HQO_ERR_ARG;
  std::vector<float> part(std::max(1, nthreads), 0.0f);
  parallel_rows(M, nthreads, [&](int64_t r0, int64_t r1, int t) {
    std::vector<float> y(static_cast<size_t>(K));
    float m = 0.0f;
    for (int64_t r = r0; r < r1; ++r) {
      rotate_row(x, dtype, r, K, ldx, group, y.data());
      for (int64_t k = 0; k < K; ++k) m = amax_update(m, std::fabs(y[k]));
      if (y_out) std::memcpy(y_out + r * K, y.data(), sizeof(float) * K);
    }
    part[t] = m;
  });
  float m = 0.0f;
  for (float p : part) m = amax_update(m, p);
  *amax_out = m;
  return HQO_OK;
}

// The whole quantizer of [P1] §2/§3 for one tensor:
//   pass 1: amax of the rotated tensor (skipped when amax_in is given);
//   pass 2: per 16-element block of a row, block amax, E4M3 block scale,
//           E2M1 codes, two codes per byte with the even element in the low
//           nibble (the packing step of [P1] §2, and the storage layout of [P4]
//           "The numeric format").
// q: [M, K/2] bytes, s: [M, K/16] E4M3 bytes, both row-major and contiguous.
int hqo_quantize(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, int group,
                 const float* amax_in, uint8_t* q, uint8_t* s, float* amax_out,
                 float* sglobal_out, int nthreads) {
  if (!x || !q || !s || !shape_ok(M, K, ldx, group)) return HQO_ERR_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return HQO_ERR_ARG;
  float amax;
  if (amax_in) {
    amax = *amax_in;
  } else {
    const int rc = hqo_rot_amax(x, dtype, M, K, ldx, group, &amax, nullptr, nthreads);
    if (rc != HQO_OK) return rc;
  }
  const float s_global = global_scale(amax);
  if (amax_out) *amax_out = amax;
  if (sglobal_out) *sglobal_out = s_global;

  parallel_rows(M, nthreads, [&](int64_t r0, int64_t r1, int) {
    std::vector<float> y(static_cast<size_t>(K));
    for (int64_t r = r0; r < r1; ++r) {
      rotate_row(x, dtype, r, K, ldx, group, y.data());
      for (int64_t b = 0; b < K / 16; ++b) {
        const float* yb = y.data() + 16 * b;
        // block amax ([P1] §2: amax over the 16 rotated values)
        float amax_b = 0.0f;
        for (int i = 0; i < 16; ++i) amax_b = amax_update(amax_b, std::fabs(yb[i]));
        // block scale ([P1] §1 table: (block_amax / 6) / s_global)
        const float v = (amax_b / 6.0f) / s_global;
        const uint8_t sb = e4m3_rne_code(v);
        s[r * (K / 16) + b] = sb;
        // reconstructed scale and codes ([P1] §1: q = round(x / (s_block * s_global)))
        const float s_f = e4m3_value(sb) * s_global;
        uint8_t codes[16];
        for (int i = 0; i < 16; ++i) codes[i] = (s_f == 0.0f) ? 0 : e2m1_code(yb[i] / s_f);
        for (int j = 0; j < 8; ++j)
          q[r * (K / 2) + 8 * b + j] =
              static_cast<uint8_t>(codes[2 * j] | (codes[2 * j + 1] << 4));
      }
    }
  });
  return HQO_OK;
}

// Dequantization, [P1] §2 dequantize: value = (+-grid[c & 7]) * (s_block * s_global),
// then, when `unrotate`, the rotation again (H/sqrt(G) is symmetric and
// orthonormal, so it is its own inverse).  out: fp32 [M, K], row stride K.
int hqo_dequant(const uint8_t* q, const uint8_t* s, float s_global, int64_t M, int64_t K,
                int group, int unrotate, float* out, int nthreads) {
  if (!q || !s || !out || !shape_ok(M, K, K, unrotate ? group : 0)) return HQO_ERR_ARG;
  if (K % 16 != 0) return HQO_ERR_ARG;
  parallel_rows(M, nthreads, [&](int64_t r0, int64_t r1, int) {
    for (int64_t r = r0; r < r1; ++r) {
      float* o = out + r * K;
      for (int64_t k = 0; k < K; ++k) {
        const uint8_t byte = q[r * (K / 2) + k / 2];
        const uint8_t c = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        const float mag = kE2M1Grid[c & 7];
        const float val = (c & 8) ? -mag : mag;
        const float s_f = e4m3_value(s[r * (K / 16) + k / 16]) * s_global;
        o[k] = val * s_f;
      }
      if (unrotate && group > 0)
        for (int64_t g0 = 0; g0 < K; g0 += group) rotate_group(o + g0, group);
    }
  });
  return HQO_OK;
}

// Rotation of a flat array of n values in groups of `group` (n % group == 0).
int hqo_rotate(const float* in, int64_t n, int group, float* out) {
  if (!in || !out || n < 0) return HQO_ERR_ARG;
  if (!(group == 16 || group == 256) || n % group != 0) return HQO_ERR_ARG;
  std::memcpy(out, in, sizeof(float) * n);
  for (int64_t g0 = 0; g0 < n; g0 += group) rotate_group(out + g0, group);
  return HQO_OK;
}

// Element-wise format helpers for the exhaustive tests.
void hqo_e2m1_codes(const float* in, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e2m1_code(in[i]);
}

// Codes of the consecutive fp32 bit patterns first, first+1, ..., first+count-1.
void hqo_e2m1_codes_bits(uint32_t first, int64_t count, uint8_t* out, int nthreads) {
  parallel_rows(count, nthreads, [&](int64_t i0, int64_t i1, int) {
    for (int64_t i = i0; i < i1; ++i)
      out[i] = e2m1_code(bits_to_float(first + static_cast<uint32_t>(i)));
  });
}

void hqo_e4m3_codes(const float* in, int64_t n, uint8_t* out, int nthreads) {
  parallel_rows(n, nthreads, [&](int64_t i0, int64_t i1, int) {
    for (int64_t i = i0; i < i1; ++i) out[i] = e4m3_rne_code(in[i]);
  });
}

void hqo_e4m3_codes_bits(uint32_t first, int64_t count, uint8_t* out, int nthreads) {
  parallel_rows(count, nthreads, [&](int64_t i0, int64_t i1, int) {
    for (int64_t i = i0; i < i1; ++i)
      out[i] = e4m3_rne_code(bits_to_float(first + static_cast<uint32_t>(i)));
  });
}

void hqo_e4m3_values(const uint8_t* codes, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

float hqo_global_scale(float amax) { return global_scale(amax); }

}  // extern "C"

// ===========================================================================
// MXFP4: E2M1 codes with one power-of-two (E8M0) scale per 32 consecutive
// elements of a row, no per-tensor scale ("A Fused Hadamard + NVFP4
// Quantization Kernel in Triton", §1, where the format table sets MXFP4 beside
// NVFP4 with 32-element blocks and power-of-two E8M0 scales; "Try this", which
// repeats the error study in MXFP4 with the rotation applied as before).  The pages give no rule for the scale; the
// reading adopted is the usual MX rule: X = 2^(floor(log2 amax_b) - 2), 2 being
// the exponent of E2M1's largest value 6, so amax_b / X lies in [4, 8); the E8M0
// byte is that exponent + 127, clamped to [0, 254] (0 for an all-zero block);
// codes are E2M1 (ties to even, saturating at 6) of y / X.
// ===========================================================================
namespace {

int e8m0_code(float amax_b) {
  if (!(amax_b > 0.0f)) return 0;
  int e2;
  std::frexp(amax_b, &e2);           // amax_b = m 2^e2, m in [0.5, 1): floor(log2) = e2 - 1
  int code = (e2 - 1) - 2 + 127;
  if (code < 0) code = 0;
  if (code > 254) code = 254;
  return code;
}

float e8m0_value(int code) { return std::ldexp(1.0f, code - 127); }

}  // namespace

extern "C" {

// q: [M, K/2] packed codes (even element low), s: [M, K/32] E8M0 bytes.
int hqo_quantize_mxfp4(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, int group,
                       uint8_t* q, uint8_t* s, int nthreads) {
  if (!x || !q || !s || M < 0 || K < 0 || ldx < K) return HQO_ERR_ARG;
  if (!(group == 0 || group == 16 || group == 256)) return HQO_ERR_ARG;
  if (K % 32 != 0 || (group > 0 && K % group != 0)) return HQO_ERR_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return HQO_ERR_ARG;
  parallel_rows(M, nthreads, [&](int64_t r0, int64_t r1, int) {
    std::vector<float> y(static_cast<size_t>(K));
    for (int64_t r = r0; r < r1; ++r) {
      rotate_row(x, dtype, r, K, ldx, group, y.data());
      for (int64_t b = 0; b < K / 32; ++b) {
        const float* yb = y.data() + 32 * b;
        float amax_b = 0.0f;
        for (int i = 0; i < 32; ++i) amax_b = amax_update(amax_b, std::fabs(yb[i]));
        const int code = e8m0_code(amax_b);
        s[r * (K / 32) + b] = static_cast<uint8_t>(code);
        const float X = e8m0_value(code);
        uint8_t codes[32];
        for (int i = 0; i < 32; ++i) codes[i] = e2m1_code(yb[i] / X);
        for (int j = 0; j < 16; ++j)
          q[r * (K / 2) + 16 * b + j] =
              static_cast<uint8_t>(codes[2 * j] | (codes[2 * j + 1] << 4));
      }
    }
  });
  return HQO_OK;
}

// value = (+-grid[c & 7]) * X, then the rotation again when `unrotate`.
int hqo_dequant_mxfp4(const uint8_t* q, const uint8_t* s, int64_t M, int64_t K, int group,
                      int unrotate, float* out, int nthreads) {
  if (!q || !s || !out || M < 0 || K < 0 || K % 32 != 0) return HQO_ERR_ARG;
  if (unrotate && !(group == 16 || group == 256)) return HQO_ERR_ARG;
  if (unrotate && K % group != 0) return HQO_ERR_ARG;
  parallel_rows(M, nthreads, [&](int64_t r0, int64_t r1, int) {
    for (int64_t r = r0; r < r1; ++r) {
      float* o = out + r * K;
      for (int64_t k = 0; k < K; ++k) {
        const uint8_t byte = q[r * (K / 2) + k / 2];
        const uint8_t c = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        const float mag = kE2M1Grid[c & 7];
        const float val = (c & 8) ? -mag : mag;
        o[k] = val * e8m0_value(s[r * (K / 32) + k / 32]);
      }
      if (unrotate)
        for (int64_t g0 = 0; g0 < K; g0 += group) rotate_group(o + g0, group);
    }
  });
  return HQO_OK;
}

}  // extern "C"

// ===========================================================================
// INT8 per-token rotate-quant ("hyperflow_h3_flash_int8.py", HyperFlow: module
// docstring, regular_hadamard, rotate_quant_kernel).
//
//   R_G      = kron(H4/2, ..., H4/2) (G a power of 4), with
//              H4 = [[1,1,1,-1],[1,1,-1,1],[1,-1,1,1],[-1,1,1,1]]: orthonormal,
//              symmetric, rows summing to one.
//   y        = x . R_G on every run of G consecutive channels of a row.
//   scale    = max(amax_row |y|, 1e-12) / 127 (one per row, fp32)
//   inv      = 1 / scale
//   q        = clamp(rint(y * inv), -127, 127) as int8 (round half to even).
//
// Readings (the page's rotation is a tensor-core dot product of unspecified
// order): the Kronecker factors are applied digit by digit, least significant
// base-4 digit (contiguous channels) first, as the page's factored kernel does
// (inner factor, then outer).  H4 = J - 2 P (J all ones, P the exchange matrix),
// so one 4-point step of H4/2 on (v0, v1, v2, v3) is out_k = S/2 - v_(3-k) with
// S = (v0 + v1) + (v2 + v3); out_k is rounded once (fmaf: S/2 is exact inside).
// ===========================================================================
namespace {

void regular_hadamard_group(float* z, int G) {
  for (int stride = 1; stride < G; stride *= 4) {
    for (int base = 0; base < G; ++base) {
      if ((base / stride) % 4 != 0) continue;  // base has digit 0 at this position
      float v[4];
      for (int k = 0; k < 4; ++k) v[k] = z[base + k * stride];
      const float S = (v[0] + v[1]) + (v[2] + v[3]);
      for (int k = 0; k < 4; ++k) z[base + k * stride] = std::fmaf(0.5f, S, -v[3 - k]);
    }
  }
}

bool int8_group_ok(int G) { return G == 4 || G == 16 || G == 64 || G == 256 || G == 1024; }

}  // namespace

extern "C" {

// y = x . R_G on a flat array of n values (n % G == 0).
int hqo_int8_rotate(const float* in, int64_t n, int group, float* out) {
  if (!in || !out || n < 0 || !int8_group_ok(group) || n % group != 0) return HQO_ERR_ARG;
  std::memcpy(out, in, sizeof(float) * n);
  for (int64_t g0 = 0; g0 < n; g0 += group) regular_hadamard_group(out + g0, group);
  return HQO_OK;
}

// q: int8 [M, K] (row stride K); scales: fp32 [M].
int hqo_rotate_quant_int8(const void* x, int dtype, int64_t M, int64_t K, int64_t ldx, int group,
                          int8_t* q, float* scales, int nthreads) {
  if (!x || !q || !scales || M < 0 || K < 0 || ldx < K) return HQO_ERR_ARG;
  if (!int8_group_ok(group) || K % group != 0) return HQO_ERR_ARG;
  if (dtype != DT_F32 && dtype != DT_BF16) return HQO_ERR_ARG;
  parallel_rows(M, nthreads, [&](int64_t r0, int64_t r1, int) {
    std::vector<float> y(static_cast<size_t>(K));
    for (int64_t r = r0; r < r1; ++r) {
      for (int64_t k = 0; k < K; ++k) y[k] = load_elem(x, dtype, r * ldx + k);
      for (int64_t g0 = 0; g0 < K; g0 += group) regular_hadamard_group(y.data() + g0, group);
      float amax = 0.0f;
      for (int64_t k = 0; k < K; ++k) amax = amax_update(amax, std::fabs(y[k]));
      const float scale = ((amax > 1e-12f) ? amax : 1e-12f) / 127.0f;
      const float inv = 1.0f / scale;
      scales[r] = scale;
      for (int64_t k = 0; k < K; ++k) {
        float v = std::rint(y[k] * inv);
        if (v > 127.0f) v = 127.0f;
        if (v < -127.0f) v = -127.0f;
        q[r * K + k] = static_cast<int8_t>(v);
      }
    }
  });
  return HQO_OK;
}

}  // extern "C"
