// Quantizer decisions of the append path, shared by rq_append.cu (append
// kernel) and rq_decode.cu (the anchor-loop call that also appends the current
// token).  Every decision that fixes a stored byte is taken exactly; see the
// precision note at the top of rq_append.cu.
#pragma once

#include <cuda_fp8.h>

#include "rq_internal.cuh"

namespace rq {
namespace {

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t b) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
  return __half2float(__half(hr));
}

// E4M3 byte nearest to D / qmax (D >= 0 exact in float64), ties to the even
// code, saturating at 448.  A float32 estimate gives a candidate; the exact
// comparison |D - qmax * v(c)| over the candidate and its two neighbours
// (all products exact: 4-bit significand times a 4-bit integer) decides.
__device__ __noinline__ uint8_t e4m3_nearest_ratio(double D, int qmax) {
  float est = __fdiv_rn((float)D, (float)qmax);
  int c0 = f32_to_e4m3(est);
  int best = -1;
  double best_d = 0.0;
  for (int c = c0 - 1; c <= c0 + 1; ++c) {
    if (c < 0 || c > 0x7E) continue;
    double dist = fabs(D - (double)qmax * (double)e4m3_to_f32((uint8_t)c));
    if (best < 0 || dist < best_d || (dist == best_d && (c & 1) == 0)) {
      best = c;
      best_d = dist;
    }
  }
  return (uint8_t)best;
}

// Nearest k of v to o + k s (exact), ties to even k, clamped to [0, qmax].
__device__ __noinline__ int nearest_code(float v, float o, float s, int qmax) {
  if (!(s > 0.f)) return 0;
  double t = (double)v - (double)o;                 // exact: fp32 minus an E4M3 value
  float kf = rintf(__fdiv_rn((float)t, s));
  kf = fminf(fmaxf(kf, -1.f), (float)(qmax + 1));
  int k = (int)kf;
  double sd = (double)s;
  double r = t - (double)k * sd;                    // exact
  if (2.0 * r > sd) ++k;
  else if (2.0 * r < -sd) --k;
  r = t - (double)k * sd;
  if (2.0 * fabs(r) == sd && (k & 1)) k += (r > 0.0) ? 1 : -1;
  return min(max(k, 0), qmax);
}

// e4m3_nearest_ratio for D = hi - lo: a float32 estimate decides unless it lies
// within its error bound (relative 2^-22: one rounding in hi - lo, one in the
// division) of a midpoint between two E4M3 values; then the exact routine.
__device__ __forceinline__ uint8_t e4m3_ratio(float hi, float lo, int qmax) {
  const float est = __fdiv_rn(hi - lo, (float)qmax);
  const int c0 = f32_to_e4m3(est);                       // est >= 0: codes 0 .. 0x7E
  const float v0 = e4m3_to_f32((uint8_t)c0);
  const float vlo = c0 > 0 ? e4m3_to_f32((uint8_t)(c0 - 1)) : -INFINITY;
  const float vhi = c0 < 0x7E ? e4m3_to_f32((uint8_t)(c0 + 1)) : INFINITY;
  const float tol = est * 0x1p-20f;
  // midpoints of neighbouring E4M3 values are exact in float32 (few significant bits)
  if (est > 0.5f * (vlo + v0) + tol && est < 0.5f * (v0 + vhi) - tol) return (uint8_t)c0;
  return e4m3_nearest_ratio((double)hi - (double)lo, qmax);
}

// nearest_code with a float32 first pass: (v - o) / s is within |x| 2^-22 of
// the exact quotient, so a fractional part far enough from 1/2 decides.
__device__ __forceinline__ int nearest_code_fast(float v, float o, float s, int qmax) {
  if (!(s > 0.f)) return 0;
  const float x = __fdiv_rn(v - o, s);
  const float kf = rintf(x);
  const float tol = fmaxf(0x1p-14f, fabsf(x) * 0x1p-20f);
  if (fabsf(x - kf) < 0.5f - tol) {
    const float kc = fminf(fmaxf(kf, 0.f), (float)qmax);
    return (int)kc;
  }
  return nearest_code(v, o, s, qmax);
}

// Group quantizer for one element per lane; the g lanes of a group are
// consecutive lanes of one warp (g = 16 or 32).  Returns the code; writes
// the dequantized value and (on every lane) the scale/offset bytes.
__device__ __forceinline__ int quantize_lane(float v, bool active, int g, int qmax, uint8_t* s_byte,
                             uint8_t* o_byte, float* vhat) {
  float lo = active ? v : INFINITY, hi = active ? v : -INFINITY;
  for (int off = g / 2; off > 0; off >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off, g));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off, g));
  }
  uint8_t ob = f32_to_e4m3(lo);
  uint8_t sb = e4m3_ratio(hi, lo, qmax);
  float o = e4m3_to_f32(ob), s = e4m3_to_f32(sb);
  int code = nearest_code_fast(v, o, s, qmax);
  *s_byte = sb;
  *o_byte = ob;
  *vhat = fmaf(s, (float)code, o);                  // exact (few significant bits)
  return code;
}

// BF16 bits of the float64 value x, round to nearest even: round-to-odd to
// float32 first (exact for the later 8-bit rounding), then RNE to BF16.
__device__ uint16_t f64_to_bf16_bits(double x) {
  float f = __double2float_rz(x);
  if ((double)f != x) f = __uint_as_float(__float_as_uint(f) | 1u);
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

// BF16 bits of the scaling coefficient of x against the reference y (d
// elements in shared memory or any memory the warp can read), computed by one
// whole warp; every lane returns the same bits.  Least squares:
// <x, y> / <y, y> (0 when <y, y> = 0); norm ratio: sqrt(<x, x> / <y, y>).
// Rounded to BF16 from the value of the float64 sums (exact products; sums
// exact for data of moderate dynamic range): float32 sums with an error bound
// decide when both ends of the bound round to the same BF16 value; otherwise
// the float64 sums do.
__device__ __forceinline__ float row_value(float x) { return x; }
__device__ __forceinline__ float row_value(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>   // x rows held as float or as their exact BF16 values
__device__ uint16_t coefficient_bits(const T* x_row, const float* y_row, int d, bool norm_ratio, int lane) {
  // least squares: num = <x, y>, mag = sum |x y|; norm ratio: num = <x, x>
  float num = 0.f, den = 0.f, mag = 0.f;
  for (int k = lane; k < d; k += 32) {
    const float y = y_row[k], x = row_value(x_row[k]);
    num = fmaf(x, norm_ratio ? x : y, num);
    den = fmaf(y, y, den);
    mag = fmaf(fabsf(x), fabsf(y), mag);
  }
  for (int off = 16; off > 0; off >>= 1) {
    num += __shfl_xor_sync(0xffffffffu, num, off);
    den += __shfl_xor_sync(0xffffffffu, den, off);
    mag += __shfl_xor_sync(0xffffffffu, mag, off);
  }
  // every lane holds the same sums: the branches below are uniform over the warp
  if (!(den > 0.f)) return 0;   // c = 0
  // at most 4 + 5 roundings per term (< 2^-20 relative to the sums of magnitudes);
  // norm ratio: sums of squares carry at most 2^-20 relative error each, so the
  // square root of their quotient is within 2^-19 (with its own rounding)
  const float c = norm_ratio ? sqrtf(__fdiv_rn(num, den)) : __fdiv_rn(num, den);
  const float err = norm_ratio ? c * 0x1p-19f : (mag + fabsf(c) * den) * 0x1p-20f / den + fabsf(c) * 0x1p-22f;
  const __nv_bfloat16 lo = __float2bfloat16_rn(c - err), hi = __float2bfloat16_rn(c + err);
  const uint16_t blo = *reinterpret_cast<const uint16_t*>(&lo);
  const uint16_t bhi = *reinterpret_cast<const uint16_t*>(&hi);
  if (blo == bhi) return blo;
  double num64 = 0.0, den64 = 0.0;
  for (int k = lane; k < d; k += 32) {
    const double y = y_row[k], x = row_value(x_row[k]);
    num64 = fma(x, norm_ratio ? x : y, num64);
    den64 = fma(y, y, den64);
  }
  for (int off = 16; off > 0; off >>= 1) {
    num64 += __shfl_xor_sync(0xffffffffu, num64, off);
    den64 += __shfl_xor_sync(0xffffffffu, den64, off);
  }
  const double q64 = den64 > 0.0 ? num64 / den64 : 0.0;
  return f64_to_bf16_bits(norm_ratio ? sqrt(q64) : q64);
}

}  // namespace
}  // namespace rq
