// mx_quantize.cuh -- bandwidth-bound quantizer kernels for sm_103a.
//
//  * mx_quantize_kernel: MX (OCP) block quantization of a bf16 matrix, row-wise (1x32 blocks
//    along the row) and column-wise (32x1 blocks down each column, stored transposed) from a
//    single read of the input.  "MXFP8 on SM120: software support" (xuesongtap.github.io),
//    sec 0.1 (block format, E8M0 scale, q = Q(x/s)) and sec 1.2 (a transpose needs its own
//    blocks, scales and codes).
//  * ds_quantize_1x128_kernel / ds_quantize_128x128_kernel: DeepSeek fine-grained FP8 with
//    FP32 scales s = amax/448.  "Why FP8 training is stable" (magicnetworld.com), sec 4 and 5.
//  * nvfp4_amax_kernel / nvfp4_quantize_kernel: NVFP4 two-level quantization.
//    "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 5.4 and 5.6.
//
// Every kernel streams its input once with 128-bit loads, reduces block maxima in registers
// (warp shuffles where a block spans lanes), and writes codes with vector stores.  Scales are
// written in the 512-byte chunk layout the GEMMs read (see include/mx.h).
#pragma once

#include "mx_device.cuh"

namespace mxgb {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// offset of (row i, block j) inside a 512-byte scale chunk (128 rows x 4 blocks)
__device__ __forceinline__ int chunk_offset(int i, int j) { return (i & 31) * 16 + (i >> 5) * 4 + j; }

// ---------------------------------------------------------------------------------------------
// MX quantize.  One CTA = one 128 x 128 tile of the input (256 threads).  The tile maps to
// exactly one 512-byte row-wise scale chunk and one column-wise scale chunk.
// ---------------------------------------------------------------------------------------------
template <int ELEM>  // 0 = E4M3 (emax 8), 1 = E5M2 (emax 15)
struct MxElem;
template <>
struct MxElem<0> {
  static constexpr int emax = 8;
  __device__ static uint32_t cvt2(float lo, float hi) { return cvt_e4m3x2(lo, hi); }
};
template <>
struct MxElem<1> {
  static constexpr int emax = 15;
  __device__ static uint32_t cvt2(float lo, float hi) { return cvt_e5m2x2(lo, hi); }
};
// MXFP4: E2M1 elements (largest value 6 = 1.5 * 2^2), two codes per byte, element 2i in the low
// nibble.  "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 5.5.
template <>
struct MxElem<2> {
  static constexpr int emax = 2;
  __device__ static uint32_t cvt2(float lo, float hi) { return cvt_e2m1x2(lo, hi); }
};

// E8M0 scale byte from the largest |x| bit pattern (bf16 bits & 0x7fff) of a finite block:
// k = floor(log2 amax) - emax clamped to >= -127; byte = k + 127 = max(expfield - emax, 0).
template <int ELEM>
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax_bits) {
  const int e = static_cast<int>(amax_bits >> 7);  // biased exponent (0 for zero / subnormal)
  const int c = e - MxElem<ELEM>::emax;
  return c > 0 ? static_cast<uint32_t>(c) : 0u;
}

// 2^-k for scale byte c (k = c - 127): an FP32 with exponent field 254 - c (always normal).
__device__ __forceinline__ float mx_inv_scale(uint32_t c) { return __uint_as_float((254u - c) << 23); }

// Quantize 8 bf16 values (one uint4) with inverse scale `inv`; returns 8 packed codes.
template <int ELEM>
__device__ __forceinline__ uint2 mx_codes8(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __fmul_rn(bf16_bits_to_float(w[i] & 0xFFFFu), inv);
    const float hi = __fmul_rn(bf16_bits_to_float(w[i] >> 16), inv);
    p[i] = MxElem<ELEM>::cvt2(lo, hi);
  }
  return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// Quantize 8 bf16 values to E2M1 with inverse scale `inv`; returns 4 bytes of packed codes.
__device__ __forceinline__ uint32_t mx_codes8_e2m1(uint4 v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t p = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __fmul_rn(bf16_bits_to_float(w[i] & 0xFFFFu), inv);
    const float hi = __fmul_rn(bf16_bits_to_float(w[i] >> 16), inv);
    p |= cvt_e2m1x2(lo, hi) << (8 * i);
  }
  return p;
}

// largest |x| bit pattern (bf16 bits with the sign cleared) of 8 bf16 values; the two halves of
// each word are compared as packed 16-bit unsigned integers
__device__ __forceinline__ uint32_t absmax_bits8(uint4 v) {
  uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu), __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
  return max(m & 0xFFFFu, m >> 16);
}

// ---------------------------------------------------------------------------------------------
// Codes of fl32(x / d) without a per-element IEEE division.
//
// The recipes define the code as the rounding of the FP32 quotient fl32(x / d).  With
// r = rcp.approx(d) (relative error at most 1 ulp = 2^-23), x * r * (1 - 2^-19) and
// x * r * (1 + 2^-19) bracket fl32(x / d) with room to spare; the conversions are monotonic,
// so when both ends give the same code no rounding boundary of the format lies in between and
// that code is the code of fl32(x / d).  When they differ (a boundary within ~2^-19 of the
// quotient, rare) the IEEE quotient decides.  The result is therefore identical to converting
// __fdiv_rn(x, d).  `d` must be a normal float no larger than 2^125 (callers check).
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float rcp_approx(float v) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

constexpr float kBracketDown = 1.0f - 1.9073486328125e-06f;  // 1 - 2^-19
constexpr float kBracketUp = 1.0f + 1.9073486328125e-06f;    // 1 + 2^-19

// (a * s.x, b * s.y) with one paired multiply, each product rounded to nearest as __fmul_rn
__device__ __forceinline__ void mul2_rn(float a, float b, uint64_t s, float& ra, float& rb) {
  asm("{\n\t.reg .b64 x, y;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mul.rn.f32x2 y, x, %4;\n\t"
      "mov.b64 {%0, %1}, y;\n\t}"
      : "=f"(ra), "=f"(rb)
      : "f"(a), "f"(b), "l"(s));
}

struct QuotientBracket {
  float lo, hi;  // rcp(d) scaled by (1 - 2^-19) and (1 + 2^-19)
  float d;
  uint64_t lo2, hi2;  // lo and hi twice, as the second operand of mul2_rn
  __device__ __forceinline__ explicit QuotientBracket(float div) : d(div) {
    const float r = rcp_approx(div);
    lo = __fmul_rn(r, kBracketDown);
    hi = __fmul_rn(r, kBracketUp);
    lo2 = pack_f32x2(lo, lo);
    hi2 = pack_f32x2(hi, hi);
  }
  __device__ __forceinline__ static bool usable(float div) { return div >= 1.17549435e-38f && div <= 4.2535296e37f; }
};

// E4M3 pair (lo byte = a) of fl32(a / d), fl32(b / d)
__device__ __forceinline__ uint32_t e4m3x2_quotient(float a, float b, const QuotientBracket& q) {
  const uint32_t c0 = cvt_e4m3x2(__fmul_rn(a, q.lo), __fmul_rn(b, q.lo));
  const uint32_t c1 = cvt_e4m3x2(__fmul_rn(a, q.hi), __fmul_rn(b, q.hi));
  if (c0 == c1) return c0;
  return cvt_e4m3x2(__fdiv_rn(a, q.d), __fdiv_rn(b, q.d));
}

// E2M1 pair (low nibble = a) of fl32(a / d), fl32(b / d).  The bracket's products as paired
// multiplies: 67.6 against 68.6 us for an 8192 x 8192 NVFP4 quantization (the same pairing in
// the E4M3 bracket made the DeepSeek 1x128 kernel 8% slower: two more registers).
__device__ __forceinline__ uint32_t e2m1x2_quotient(float a, float b, const QuotientBracket& q) {
  float a0, b0, a1, b1;
  mul2_rn(a, b, q.lo2, a0, b0);
  mul2_rn(a, b, q.hi2, a1, b1);
  const uint32_t c0 = cvt_e2m1x2(a0, b0);
  const uint32_t c1 = cvt_e2m1x2(a1, b1);
  if (c0 == c1) return c0;
  return cvt_e2m1x2(__fdiv_rn(a, q.d), __fdiv_rn(b, q.d));
}

// Output pointers of one MX quantize launch: up to two element formats (F0, then F0 + 1).
struct MxOut {
  uint8_t* q_row[2];
  uint8_t* s_row[2];
  uint8_t* q_col[2];
  uint8_t* s_col[2];
};

template <int FMT>
__device__ __forceinline__ uint32_t mx_cvt2(float lo, float hi) {
  return MxElem<FMT>::cvt2(lo, hi);
}

// NF = 1: format F0 only; NF = 2: E4M3 and E5M2 from the same read of x (F0 = 0).
// Four resident CTAs per SM (64 registers a thread) keep enough loads in flight.
// B2D: 2-D 32x32 blocks (one scale per 32x32 block of x, the MX rule over the whole block;
// "MXFP8 on SM120: software support" (xuesongtap.github.io), sec 1.3).  Both copies then carry
// the block's scale on each of their 1x32 blocks, so the transposed copy's codes are the
// transpose of the row-wise codes.
template <int F0, int NF, bool ROW, bool COL, bool B2D = false>
__global__ void __launch_bounds__(256, 4) mx_quantize_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                          int64_t cols, const MxOut o) {
  pdl_prologue();
  __shared__ __align__(16) uint32_t tile[COL ? 128 * 64 : 1];  // 128 rows x 128 bf16 (as bf16x2 words)
  __shared__ __align__(16) uint8_t srow[NF][512];
  __shared__ __align__(16) uint8_t scol[NF][512];
  __shared__ uint32_t bmax[B2D ? 16 : 1];  // 2-D: largest |x| bits of the tile's 4 x 4 blocks

  // grid: x = row tile, y = column tile (no 64-bit division per thread)
  const int64_t tiles_c = cols >> 7;
  const int64_t tr = blockIdx.x;
  const int64_t tc = blockIdx.y;
  const int t = threadIdx.x;
  const int lc = t & 15;     // 16 threads per row, 8 bf16 (one uint4) each
  const int r0 = t >> 4;     // rows r0 + 16*i

  const uint16_t* xt = x + (tr * 128) * cols + tc * 128;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ld_stream_v4(xt + static_cast<int64_t>(r0 + 16 * i) * cols + lc * 8);

  if (COL) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<uint4*>(&tile[(r0 + 16 * i) * 64 + lc * 4]) = v[i];
  }

  if constexpr (B2D) {
    // block (br, bc): rows 32 br .. (this thread's rows r0 + 16 i with i >> 1 == br), columns
    // 32 bc .. (lc >> 2 == bc); the 4 lanes of a block column and the two r0 of a warp combine
    // by shuffles, the 8 warps through shared memory
    if (t < 16) bmax[t] = 0;
    __syncthreads();
#pragma unroll
    for (int br = 0; br < 4; ++br) {
      uint32_t m = max(absmax_bits8(v[2 * br]), absmax_bits8(v[2 * br + 1]));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
      if ((t & 19) == 0) atomicMax(&bmax[br * 4 + (lc >> 2)], m);  // lc % 4 == 0, even r0
    }
    __syncthreads();
  }

  if (ROW) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + 16 * i;
      uint32_t m;
      if constexpr (B2D) {
        m = bmax[(i >> 1) * 4 + (lc >> 2)];
      } else {
        m = absmax_bits8(v[i]);
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      }
      if constexpr (F0 == 2) {  // MXFP4: packed E2M1, a NaN or Inf block gets codes 0x7
        uint32_t packed, sbyte;
        if (m >= 0x7F80u) {
          sbyte = 0xFF;
          packed = 0x77777777u;
        } else {
          sbyte = mx_scale_byte<2>(m);
          packed = mx_codes8_e2m1(v[i], mx_inv_scale(sbyte));
        }
        *reinterpret_cast<uint32_t*>(o.q_row[0] + (tr * 128 + r) * (cols >> 1) + tc * 64 + lc * 4) = packed;
        if ((lc & 3) == 0) srow[0][chunk_offset(r, lc >> 2)] = static_cast<uint8_t>(sbyte);
      } else {
#pragma unroll
      for (int f = 0; f < NF; ++f) {
        uint2 codes;
        uint32_t sbyte;
        if (m >= 0x7F80u) {  // NaN or Inf in the block
          sbyte = 0xFF;
          codes = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
        } else if (F0 + f == 0) {
          sbyte = mx_scale_byte<0>(m);
          codes = mx_codes8<0>(v[i], mx_inv_scale(sbyte));
        } else {
          sbyte = mx_scale_byte<1>(m);
          codes = mx_codes8<1>(v[i], mx_inv_scale(sbyte));
        }
        *reinterpret_cast<uint2*>(o.q_row[f] + (tr * 128 + r) * cols + tc * 128 + lc * 8) = codes;
        if ((lc & 3) == 0) srow[f][chunk_offset(r, lc >> 2)] = static_cast<uint8_t>(sbyte);
      }
      }
    }
  }

  if (COL) {
    __syncthreads();
    // thread -> (column quad cq, row block rb, half hb): 16 rows x 4 columns, two bf16x2 words
    // (one conflict-free 8-byte shared load) per row; the partner thread (lane ^ 1) holds the
    // block's other 16 rows
    const int lane = t & 31;
    const int hb = lane & 1;
    const int cq = (lane >> 1) + 16 * ((t >> 5) & 1);
    const int rb = t >> 6;
    uint2 u[16];
    uint32_t m[4] = {0, 0, 0, 0};
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      u[r] = *reinterpret_cast<const uint2*>(&tile[(rb * 32 + hb * 16 + r) * 64 + 2 * cq]);
      m[0] = max(m[0], u[r].x & 0x7FFFu);
      m[1] = max(m[1], (u[r].x >> 16) & 0x7FFFu);
      m[2] = max(m[2], u[r].y & 0x7FFFu);
      m[3] = max(m[3], (u[r].y >> 16) & 0x7FFFu);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) m[j] = max(m[j], __shfl_xor_sync(0xFFFFFFFFu, m[j], 1));
    if constexpr (B2D) {  // the 32x32 block's maximum instead of the column block's
#pragma unroll
      for (int j = 0; j < 4; ++j) m[j] = bmax[rb * 4 + ((4 * cq + j) >> 5)];
    }
    if constexpr (F0 == 2) {  // MXFP4: 16 codes per column -> 8 bytes
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 4 * cq + j;
        uint32_t w2[2], sbyte;
        if (m[j] >= 0x7F80u) {
          sbyte = 0xFF;
          w2[0] = w2[1] = 0x77777777u;
        } else {
          sbyte = mx_scale_byte<2>(m[j]);
          const float inv = mx_inv_scale(sbyte);
          const int sh = (j & 1) ? 16 : 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t acc = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // rows 8h + 2k, 8h + 2k + 1 -> byte k
              const int ra = 8 * h + 2 * k;
              const uint32_t ea = ((j < 2) ? u[ra].x : u[ra].y) >> sh;
              const uint32_t eb = ((j < 2) ? u[ra + 1].x : u[ra + 1].y) >> sh;
              const float fa = __fmul_rn(bf16_bits_to_float(ea & 0xFFFFu), inv);
              const float fb = __fmul_rn(bf16_bits_to_float(eb & 0xFFFFu), inv);
              acc |= cvt_e2m1x2(fa, fb) << (8 * k);
            }
            w2[h] = acc;
          }
        }
        uint8_t* dst = o.q_col[0] + (tc * 128 + c) * (rows >> 1) + tr * 64 + rb * 16 + hb * 8;
        *reinterpret_cast<uint2*>(dst) = make_uint2(w2[0], w2[1]);
        if (hb == 0) scol[0][chunk_offset(c, rb)] = static_cast<uint8_t>(sbyte);
      }
    } else {
#pragma unroll
    for (int f = 0; f < NF; ++f) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 4 * cq + j;  // column inside the tile = row of the transposed tile
        uint32_t packed[4];
        uint32_t sbyte;
        if (m[j] >= 0x7F80u) {  // NaN or Inf in the block
          sbyte = 0xFF;
#pragma unroll
          for (int k = 0; k < 4; ++k) packed[k] = 0x7F7F7F7Fu;
        } else {
          sbyte = (F0 + f == 0) ? mx_scale_byte<0>(m[j]) : mx_scale_byte<1>(m[j]);
          const float inv = mx_inv_scale(sbyte);
          const int sh = (j & 1) ? 16 : 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t e[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) e[i] = ((j < 2) ? u[4 * k + i].x : u[4 * k + i].y) >> sh;
            const float f0 = __fmul_rn(bf16_bits_to_float(e[0] & 0xFFFFu), inv);
            const float f1 = __fmul_rn(bf16_bits_to_float(e[1] & 0xFFFFu), inv);
            const float f2 = __fmul_rn(bf16_bits_to_float(e[2] & 0xFFFFu), inv);
            const float f3 = __fmul_rn(bf16_bits_to_float(e[3] & 0xFFFFu), inv);
            packed[k] = (F0 + f == 0) ? (mx_cvt2<0>(f0, f1) | (mx_cvt2<0>(f2, f3) << 16))
                                      : (mx_cvt2<1>(f0, f1) | (mx_cvt2<1>(f2, f3) << 16));
          }
        }
        uint8_t* dst = o.q_col[f] + (tc * 128 + c) * rows + tr * 128 + rb * 32 + hb * 16;
        *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        if (hb == 0) scol[f][chunk_offset(c, rb)] = static_cast<uint8_t>(sbyte);
      }
    }
    }
  }

  __syncthreads();
  // scale chunks: 32 threads per (format, copy), one 16-byte piece each
  const int f = t >> 6;
  const int u = t & 63;
  if (f < NF) {
    if (u < 32) {
      uint8_t* srp = (NF == 1 || f == 0) ? o.s_row[0] : o.s_row[1];
      if (ROW) reinterpret_cast<uint4*>(srp + (tr * tiles_c + tc) * 512)[u] = reinterpret_cast<const uint4*>(srow[f])[u];
    } else if (COL) {
      const int64_t tiles_r = rows >> 7;
      uint8_t* scp = (NF == 1 || f == 0) ? o.s_col[0] : o.s_col[1];
      reinterpret_cast<uint4*>(scp + (tc * tiles_r + tr) * 512)[u - 32] = reinterpret_cast<const uint4*>(scol[f])[u - 32];
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Power-of-two block scales and their E8M0 form
// ---------------------------------------------------------------------------------------------
// 2^n as an FP32 for -127 <= n <= 127 (2^-127 is the subnormal 0x00400000)
__device__ __forceinline__ float pow2f(int n) {
  return __uint_as_float(n >= -126 ? static_cast<uint32_t>(n + 127) << 23 : 0x00400000u);
}

// k = the smallest integer with 448 * 2^k >= amax, clamped to [-127, 127], from the bf16 bits of
// amax (finite, sign cleared); 0 when amax == 0.  448 = 1.75 * 2^8 and 1.75 is the bf16
// mantissa 0x60: amax = 1.m * 2^e needs k = e - 8 when 1.m <= 1.75 and e - 7 otherwise.  A bf16
// subnormal amax is below 448 * 2^-127 and gets the clamp.
__device__ __forceinline__ int pow2_scale_exp(uint32_t amax_bits) {
  if (amax_bits == 0) return 0;
  const int e = static_cast<int>(amax_bits >> 7);
  if (e == 0) return -127;
  const int k = (e - 127) - 8 + ((amax_bits & 0x7Fu) > 0x60u ? 1 : 0);
  return k < -127 ? -127 : (k > 127 ? 127 : k);
}

// E8M0 code of an FP32 scale: k + 127 for exactly 2^k, -127 <= k <= 127; otherwise 0xFF (NaN)
__device__ __forceinline__ uint32_t e8m0_of_pow2(float sc) {
  const uint32_t b = __float_as_uint(sc);
  if (b == 0x00400000u) return 0;                           // 2^-127
  const uint32_t e = b >> 23;                               // sign bit set -> e > 255
  return ((b & 0x7FFFFFu) == 0 && e >= 1 && e <= 254) ? e : 0xFFu;
}

// Per-32 E8M0 scales in the MX GEMM layout of a [rows][cols] code matrix from power-of-two FP32
// block scales: block_rows 1 -> s float[cols/128][rows] (1x128 tiles), block_rows 128 -> s
// float[rows/128][cols/128].  The four 32-blocks of a 128-block keep its scale; a 2-D block's
// scale is broadcast to its 128 rows.  Grid: x = 128-row block, y = 128-column chunk; one thread
// per row writes the row's 4 bytes of the chunk.
__global__ void __launch_bounds__(128) mx_scales_from_blocks_kernel(const float* __restrict__ s, int64_t rows,
                                                                    int64_t cols, int block_rows,
                                                                    uint8_t* __restrict__ out) {
  pdl_prologue();
  const int64_t rb = blockIdx.x, kc = blockIdx.y;
  const int i = threadIdx.x;
  const int64_t nkc = cols >> 7;
  const float sc = (block_rows == 1) ? s[kc * rows + rb * 128 + i] : s[rb * nkc + kc];
  const uint32_t code = e8m0_of_pow2(sc);
  *reinterpret_cast<uint32_t*>(out + (rb * nkc + kc) * 512 + chunk_offset(i, 0)) = code * 0x01010101u;
}

// Byte permutation between the GEMM scale layout (512-byte chunks of 128 rows x 4 blocks, chunk
// (rb, kc) at (rb * nblocks/4 + kc) * 512, in-chunk byte chunk_offset(i, j)) and a plain
// [rows][nblocks] byte matrix.  The 16 bytes at in-chunk offset 16 * r hold rows r, r + 32,
// r + 64, r + 96, four blocks each, so one thread moves one 16-byte piece as four 4-byte rows.
// TO_PLAIN: src = GEMM layout, dst = plain; otherwise the inverse.
template <bool TO_PLAIN>
__global__ void __launch_bounds__(256) scale_layout_kernel(const uint8_t* __restrict__ src,
                                                           uint8_t* __restrict__ dst, int64_t rows,
                                                           int64_t nblocks) {
  pdl_prologue();
  const int64_t kchunks = nblocks >> 2;
  const int64_t pieces = (rows >> 7) * kchunks * 32;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < pieces;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t chunk = t >> 5;
    const int r = static_cast<int>(t & 31);
    const int64_t rb = chunk / kchunks, kc = chunk - rb * kchunks;
    const int64_t swz = chunk * 512 + chunk_offset(r, 0);
    const int64_t plain = ((rb << 7) + r) * nblocks + (kc << 2);
    if constexpr (TO_PLAIN) {
      const uint4 v = *reinterpret_cast<const uint4*>(src + swz);
      *reinterpret_cast<uint32_t*>(dst + plain) = v.x;
      *reinterpret_cast<uint32_t*>(dst + plain + 32 * nblocks) = v.y;
      *reinterpret_cast<uint32_t*>(dst + plain + 64 * nblocks) = v.z;
      *reinterpret_cast<uint32_t*>(dst + plain + 96 * nblocks) = v.w;
    } else {
      uint4 v;
      v.x = *reinterpret_cast<const uint32_t*>(src + plain);
      v.y = *reinterpret_cast<const uint32_t*>(src + plain + 32 * nblocks);
      v.z = *reinterpret_cast<const uint32_t*>(src + plain + 64 * nblocks);
      v.w = *reinterpret_cast<const uint32_t*>(src + plain + 96 * nblocks);
      *reinterpret_cast<uint4*>(dst + swz) = v;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// DeepSeek 1x128: s = fl32(amax / 448) (1 if amax == 0), q = E4M3(fl32(x / s)); s stored
// [K/128][rows].  CTA = 64 rows x one 128-column k-block; 4 lanes per row, 32 bf16 per lane (four
// 128-bit loads, the row's 4 lanes covering 64 contiguous bytes per load), so the per-row scale
// and reciprocal are computed by 4 lanes, not 16.
// ---------------------------------------------------------------------------------------------
// POW2: Float8BlockScaling with power-of-two scales ("MXFP8 on SM120: software support"
// (xuesongtap.github.io), sec 1.3): s = 2^k, k the smallest integer with 448 * 2^k >= amax
// (clamped to [-127, 127]; 0 when amax == 0), q = E4M3(x * 2^-k), which is exact scaling.
template <bool POW2>
__global__ void __launch_bounds__(256) ds_quantize_1x128_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                int64_t cols, uint8_t* __restrict__ q,
                                                                float* __restrict__ s) {
  pdl_prologue();
  const int64_t kb = blockIdx.y;  // grid: x = group of 64 rows, y = k-block
  const int t = threadIdx.x;
  const int l4 = t & 3;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * 64 + (t >> 2);
  const uint16_t* xr = x + r * cols + kb * 128;
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = ld_stream_v4(xr + (4 * i + l4) * 8);
  uint32_t m = max(max(absmax_bits8(v[0]), absmax_bits8(v[1])), max(absmax_bits8(v[2]), absmax_bits8(v[3])));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  float sc, inv = 1.0f;
  if (POW2) {
    const int k = pow2_scale_exp(m);
    sc = pow2f(k);
    inv = pow2f(-k);
  } else {
    sc = (m == 0) ? 1.0f : __fdiv_rn(bf16_bits_to_float(m), 448.0f);
  }
  const bool fast = QuotientBracket::usable(sc);
  const QuotientBracket qb(fast ? sc : 1.0f);
  uint8_t* qr = q + r * cols + kb * 128;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_bits_to_float(w[j] & 0xFFFFu), b = bf16_bits_to_float(w[j] >> 16);
      if (POW2) p[j] = cvt_e4m3x2(__fmul_rn(a, inv), __fmul_rn(b, inv));
      else p[j] = fast ? e4m3x2_quotient(a, b, qb) : cvt_e4m3x2(__fdiv_rn(a, sc), __fdiv_rn(b, sc));
    }
    *reinterpret_cast<uint2*>(qr + (4 * i + l4) * 8) = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
  }
  if (l4 == 0) s[kb * rows + r] = sc;
}

// DeepSeek 128x128 weight blocks: one CTA per block.  The block (32 KB) arrives in shared memory
// as two TMA boxes of 128 rows x 64 columns; the threads read it twice from there (block maximum,
// then codes), so few registers stay live and six CTAs share an SM: a 2048 x 7168 weight (896
// blocks) runs as one wave on 152 SMs, and larger weights keep six blocks in flight per SM.
// Piece i of thread t: box i & 1, row (t >> 3) + 32 (i >> 1), 16-byte chunk t & 7, so the eight
// threads of each quarter-warp read eight different chunks of one 128-byte row (no bank
// conflicts).  The copy wait is bounded; on a timeout the CTA records it and leaves.
template <bool POW2>
__global__ void __launch_bounds__(256) ds_quantize_128x128_kernel(const __grid_constant__ CUtensorMap tmx,
                                                                  int64_t rows, int64_t cols,
                                                                  uint8_t* __restrict__ q, float* __restrict__ s) {
  pdl_prologue();
  __shared__ __align__(128) uint8_t tile[2 * 128 * 128];
  __shared__ uint64_t full;
  __shared__ uint32_t wmax[8];
  __shared__ int abort_flag;
  const int64_t nbc = cols >> 7;
  const int64_t br = blockIdx.x, bc = blockIdx.y;  // grid: x = block row, y = block column
  const int t = threadIdx.x;
  if (t == 0) {
    abort_flag = 0;
    mbar_init(&full, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&full, 2 * 128 * 128);
    tma_load_2d(tile, &tmx, &full, static_cast<int32_t>(bc * 256), static_cast<int32_t>(br * 128));
    tma_load_2d(tile + 128 * 128, &tmx, &full, static_cast<int32_t>(bc * 256 + 128), static_cast<int32_t>(br * 128));
  }
  __syncthreads();
  const bool ok = mbar_wait(&full, 0, &abort_flag, kSiteQuantLoad);
  if (__syncthreads_or(!ok)) {
    if (t == 0) mbar_drain(&full, 0, 100000000ull);
    return;
  }
  const int ch = t & 7, r0 = t >> 3;
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m = max(m, absmax_bits8(*reinterpret_cast<const uint4*>(tile + (i & 1) * 16384 + (r0 + 32 * (i >> 1)) * 128 + ch * 16)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((t & 31) == 0) wmax[t >> 5] = m;
  __syncthreads();
  m = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = max(m, wmax[i]);
  float sc, inv = 1.0f;
  if (POW2) {
    const int k = pow2_scale_exp(m);
    sc = pow2f(k);
    inv = pow2f(-k);
  } else {
    sc = (m == 0) ? 1.0f : __fdiv_rn(bf16_bits_to_float(m), 448.0f);
  }
  const bool fast = QuotientBracket::usable(sc);
  const QuotientBracket qb(fast ? sc : 1.0f);
#pragma unroll 2
  for (int i = 0; i < 8; ++i) {
    const int row = r0 + 32 * (i >> 1);
    const uint4 v = *reinterpret_cast<const uint4*>(tile + (i & 1) * 16384 + row * 128 + ch * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_bits_to_float(w[j] & 0xFFFFu), b = bf16_bits_to_float(w[j] >> 16);
      if (POW2) p[j] = cvt_e4m3x2(__fmul_rn(a, inv), __fmul_rn(b, inv));
      else p[j] = fast ? e4m3x2_quotient(a, b, qb) : cvt_e4m3x2(__fdiv_rn(a, sc), __fdiv_rn(b, sc));
    }
    *reinterpret_cast<uint2*>(q + (br * 128 + row) * cols + bc * 128 + (i & 1) * 64 + ch * 8) =
        make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
  }
  if (t == 0) s[br * nbc + bc] = sc;
}

// ---------------------------------------------------------------------------------------------
// NVFP4 training options ("Why FP8 training is stable" (magicnetworld.com), sec 13; "NVFP4: high
// accuracy with 4 bits" (theluyuan.com), sec 3.2).
// ---------------------------------------------------------------------------------------------
// 16 bf16 values as FP32
__device__ __forceinline__ void load_block16(const uint16_t* p, float (&f)[16]) {
  const uint4 v0 = ld_stream_v4(p), v1 = ld_stream_v4(p + 8);
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}

// v <- 0.25 * H16 * (d .* v), d_i = -1 where bit i of `signs` is set; Sylvester butterflies in
// the order h = 1, 2, 4, 8 (each sum rounded once in FP32), then an exact scaling by 1/4.
__device__ __forceinline__ void fwht16(float (&v)[16], uint32_t signs) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((signs >> i) & 1u) v[i] = -v[i];
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

// E2M1 code of y by stochastic rounding with random byte r: for |y| < 6 between grid values
// lo <= |y| < hi, round up iff r < floor(256 (|y| - lo) / (hi - lo)); |y| >= 6 gives 6.  Every
// step is exact in FP32 (|y| - lo by Sterbenz, the step is a power of two).
__device__ __forceinline__ uint32_t e2m1_stochastic(float y, uint32_t r) {
  const uint32_t sign = (__float_as_uint(y) >> 31) << 3;
  const float a = fabsf(y);
  if (a >= 6.0f) return sign | 7u;
  const int lo = (a >= 0.5f) + (a >= 1.0f) + (a >= 1.5f) + (a >= 2.0f) + (a >= 3.0f) + (a >= 4.0f);
  const float lo_val = lo <= 4 ? 0.5f * lo : (lo == 5 ? 3.0f : 4.0f);
  const float inv_step = lo < 4 ? 2.0f : (lo < 6 ? 1.0f : 0.5f);
  const float t = floorf(__fmul_rn(__fmul_rn(__fsub_rn(a, lo_val), inv_step), 256.0f));
  return sign | static_cast<uint32_t>(lo + (static_cast<float>(r) < t ? 1 : 0));
}

// E4M3 code of t = fl32(fl32(bamax / 6) / s_g): bamax * fl32(1/6) * rcp(s_g) is within 2^-21 of
// t, so a +-2^-19 bracket that converts to one code decides it; otherwise the two IEEE quotients
__device__ __forceinline__ uint32_t nv_block_scale_code(float bamax, float sg, float rsg) {
  if (QuotientBracket::usable(sg)) {
    const float y = __fmul_rn(__fmul_rn(bamax, 0.16666667163372040f), rsg);
    const uint32_t c0 = cvt_e4m3x2(__fmul_rn(y, kBracketDown), 0.0f) & 0xFFu;
    const uint32_t c1 = cvt_e4m3x2(__fmul_rn(y, kBracketUp), 0.0f) & 0xFFu;
    if (c0 == c1) return c0;
  }
  return cvt_e4m3x2(__fdiv_rn(__fdiv_rn(bamax, 6.0f), sg), 0.0f) & 0xFFu;
}

// ---------------------------------------------------------------------------------------------
// NVFP4 pass 1: global amax (as FP32 bits, atomicMax; non-negative floats order as integers).
// ---------------------------------------------------------------------------------------------
// RHT: the maximum is taken over the transformed values (every 1x16 block along a row), one block
// (two 128-bit loads) per step.
template <bool RHT = false>
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const uint16_t* __restrict__ x, int64_t n_vec8,
                                                         unsigned int* __restrict__ amax_bits, uint32_t signs = 0) {
  pdl_prologue();
  __shared__ uint32_t wmax[8];
  uint32_t m = 0;  // bf16 bits (RHT: FP32 bits) of the largest magnitude
  if (RHT) {
    for (int64_t i = blockIdx.x * 256ll + threadIdx.x; 2 * i < n_vec8; i += static_cast<int64_t>(gridDim.x) * 256) {
      float f[16];
      load_block16(x + i * 16, f);
      fwht16(f, signs);
      float a = 0.0f;
#pragma unroll
      for (int k = 0; k < 16; ++k) a = fmaxf(a, fabsf(f[k]));
      m = max(m, __float_as_uint(a));
    }
  } else {
    for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n_vec8; i += static_cast<int64_t>(gridDim.x) * 256)
      m = max(m, absmax_bits8(ld_stream_v4(x + i * 8)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) m = max(m, wmax[i]);
    atomicMax(amax_bits, RHT ? m : m << 16);  // as FP32 bits (non-negative floats order as integers)
  }
}

__device__ __forceinline__ float e4m3_to_float(uint32_t code) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\t"
      "cvt.u16.u32 t, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(code));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Clears n words (the NVFP4 amax workspace) as a kernel of the stream's dependent-launch chain,
// after the previous kernel (which may still read them) has completed.
__global__ void __launch_bounds__(256) zero_words_kernel(unsigned int* __restrict__ p, int n) {
  pdl_prologue();
  for (int i = blockIdx.x * 256 + threadIdx.x; i < n; i += gridDim.x * 256) p[i] = 0u;
}

// Grouped NVFP4 (row groups of one matrix quantized as tensors of their own, e.g. the weights of
// MoE experts; "NVFP4: high accuracy with 4 bits" (theluyuan.com), sec 5.4 applied per group).
// The group of row r: the last g < G with off[g] <= r.  Always in [0, G), whatever off holds, so
// offsets that break their contract cannot send an access out of bounds.
__device__ __forceinline__ int nv_group_of(const int64_t* __restrict__ off, int groups, int64_t r) {
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Grouped pass 1: the maximum of each group (FP32 bits in amax[g], cleared by the host).  Work
// unit = 16 rows (inside one group: offsets are multiples of 128); grid-stride over units.  CTA 0
// also checks the offsets' contract (0 = off[0] <= ... <= off[G] = rows, multiples of 128) and
// reports a broken one through the error word.
__global__ void __launch_bounds__(256) nvfp4_amax_grouped_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                 int64_t cols, const int64_t* __restrict__ off,
                                                                 int groups, unsigned int* __restrict__ amax) {
  pdl_prologue();
  __shared__ uint32_t wmax[8];
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    bool good = __ldg(off) == 0 && __ldg(off + groups) == rows;
    for (int g = 0; g < groups; ++g) {
      const int64_t a = __ldg(off + g), b = __ldg(off + g + 1);
      good = good && b >= a && (b & 127) == 0;
    }
    if (!good) atomicOr(&g_mx_error_word, kSiteBadGroups);
  }
  const int64_t units = rows >> 4;
  const int64_t nvec = 2 * cols;  // 16 rows x cols / 8 vectors of 8
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const uint16_t* xu = x + u * 16 * cols;
    uint32_t m = 0;
    for (int64_t i = threadIdx.x; i < nvec; i += 256) m = max(m, absmax_bits8(ld_stream_v4(xu + i * 8)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < 8; ++i) m = max(m, wmax[i]);
      atomicMax(amax + nv_group_of(off, groups, u * 16), m << 16);
    }
    __syncthreads();
  }
}

// NVFP4 pass 2.  CTA = 32 rows x 128 columns; thread = one 16-element block.  RHT: the block is
// transformed first (same signs as pass 1); SR: element codes by stochastic rounding of the IEEE
// quotient with one random byte per element from rbits[rows][cols].
// GROUPED: amax_bits[G] and gscale[G] per row group (off[G + 1]); a CTA's 32 rows lie in one group.
template <bool RHT = false, bool SR = false, bool GROUPED = false>
__global__ void __launch_bounds__(256) nvfp4_quantize_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                             int64_t cols, uint8_t* __restrict__ qp,
                                                             uint8_t* __restrict__ sf, float* __restrict__ gscale,
                                                             const unsigned int* __restrict__ amax_bits,
                                                             uint32_t signs = 0, const uint8_t* __restrict__ rbits = nullptr,
                                                             const int64_t* __restrict__ off = nullptr, int groups = 1) {
  pdl_prologue();
  // grid: x = 32-row tile, y = 128-column tile; the last column tile may be half full
  // (cols % 128 == 64)
  __shared__ float s_glob[2];  // s_g and rcp(s_g), computed once per CTA
  const int64_t tr = blockIdx.x, tc = blockIdx.y;
  const int t = threadIdx.x;
  if (t == 0) {
    const int grp = GROUPED ? nv_group_of(off, groups, tr * 32) : 0;
    const float amax = __uint_as_float(amax_bits[grp]);
    const float g = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
    s_glob[0] = g;
    s_glob[1] = rcp_approx(g);
    if (!GROUPED && tr == 0 && tc == 0) *gscale = g;
  }
  if (GROUPED && tr == 0 && tc == 0) {  // every group's scale, empty groups included
    for (int k = t; k < groups; k += 256) {
      const float a = __uint_as_float(amax_bits[k]);
      gscale[k] = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 2688.0f);
    }
  }
  __syncthreads();
  const float sg = s_glob[0], rsg = s_glob[1];
  const int64_t r = tr * 32 + (t >> 3);
  const int64_t c = tc * 128 + (t & 7) * 16;
  if (c >= cols) return;

  float f[16];
  float bamax;
  if (RHT) {
    load_block16(x + r * cols + c, f);
    fwht16(f, signs);
    bamax = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) bamax = fmaxf(bamax, fabsf(f[k]));
  } else {
    const uint4 v0 = ld_stream_v4(x + r * cols + c);
    const uint4 v1 = ld_stream_v4(x + r * cols + c + 8);
    bamax = bf16_bits_to_float(max(absmax_bits8(v0), absmax_bits8(v1)));
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
      f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
  }
  const uint32_t scode = nv_block_scale_code(bamax, sg, rsg);
  const float s_hat = __fmul_rn(e4m3_to_float(scode), sg);
  uint32_t lo = 0, hi = 0;
  if (s_hat != 0.0f) {
    if (SR) {
      // the IEEE quotient per element (bracketing it and evaluating the rounding at both ends
      // measured slower: 229 against 151 us at 8192 x 8192)
      const uint4 rb = *reinterpret_cast<const uint4*>(rbits + r * cols + c);
      const uint32_t rw[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t code = e2m1_stochastic(__fdiv_rn(f[e], s_hat), (rw[e >> 2] >> (8 * (e & 3))) & 0xFFu);
        if (e < 8) lo |= code << (4 * e);
        else hi |= code << (4 * (e - 8));
      }
    } else {
      const bool fast = QuotientBracket::usable(s_hat);
      const QuotientBracket qb(fast ? s_hat : 1.0f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float a = f[2 * i], b = f[2 * i + 1];
        const uint32_t byte = fast ? e2m1x2_quotient(a, b, qb) : cvt_e2m1x2(__fdiv_rn(a, s_hat), __fdiv_rn(b, s_hat));
        if (i < 4) lo |= byte << (8 * i);
        else hi |= byte << (8 * (i - 4));
      }
    }
  }
  *reinterpret_cast<uint2*>(qp + r * (cols >> 1) + (c >> 1)) = make_uint2(lo, hi);
  // scale chunk (r / 128, c / 64), 128 rows x 4 blocks of 16
  const int64_t chunk = (r >> 7) * (cols >> 6) + (c >> 6);
  sf[chunk * 512 + chunk_offset(static_cast<int>(r & 127), static_cast<int>((c >> 4) & 3))] =
      static_cast<uint8_t>(scode);
}

// NVFP4 with 16x16 2-D blocks (weights; "Why FP8 training is stable" (magicnetworld.com),
// sec 13): one E4M3 scale per 16x16 block of x, so the row-wise copy and the transposed
// (column-wise) copy hold the same codes and scales.  CTA = one 128 x 128 tile (8 x 8 blocks).
// The codes are computed once (row-wise) and the transposed copy is a nibble transpose of them
// through shared memory.  Pass 1 is nvfp4_amax_kernel<false>.  Outputs: q_row[rows][cols/2]
// packed, s_row in the NVFP4 GEMM layout of [rows][cols/16]; q_col[cols][rows/2], s_col the
// layout of [cols][rows/16].
__global__ void __launch_bounds__(256) nvfp4_quantize_2d_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                int64_t cols, uint8_t* __restrict__ q_row,
                                                                uint8_t* __restrict__ s_row,
                                                                uint8_t* __restrict__ q_col,
                                                                uint8_t* __restrict__ s_col, float* __restrict__ gscale,
                                                                const unsigned int* __restrict__ amax_bits) {
  pdl_prologue();
  __shared__ __align__(16) uint32_t ctile[128 * 16];  // 128 rows x 128 packed codes
  __shared__ __align__(16) uint8_t srow[1024], scol[1024];
  __shared__ uint32_t bmax[64];
  __shared__ float shat[64];
  __shared__ float s_glob[2];
  const int64_t tr = blockIdx.x, tc = blockIdx.y;  // grid: x = row tile, y = column tile
  const int t = threadIdx.x;
  const int lc = t & 15, r0 = t >> 4;
  if (t < 64) bmax[t] = 0;
  if (t == 0) {
    const float amax = __uint_as_float(*amax_bits);
    const float g = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
    s_glob[0] = g;
    s_glob[1] = rcp_approx(g);
    if (tr == 0 && tc == 0) *gscale = g;
  }
  const uint16_t* xt = x + (tr * 128) * cols + tc * 128;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = ld_stream_v4(xt + static_cast<int64_t>(r0 + 16 * i) * cols + lc * 8);
  __syncthreads();
  // block (i, lc >> 1) holds this thread's row r0 + 16 i, columns lc * 8 .. + 7: combine the two
  // lanes of a block's 16 columns and the warp's two rows, then the 8 warps in shared memory
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t m = absmax_bits8(v[i]);
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
    if ((t & 17) == 0) atomicMax(&bmax[i * 8 + (lc >> 1)], m);
  }
  __syncthreads();
  const float sg = s_glob[0], rsg = s_glob[1];
  if (t < 64) {  // block (t / 8, t % 8): scale code and s_hat
    const uint32_t code = nv_block_scale_code(bf16_bits_to_float(bmax[t]), sg, rsg);
    shat[t] = __fmul_rn(e4m3_to_float(code), sg);
    bmax[t] = code;
  }
  __syncthreads();
  // row-wise codes: 8 values of row r0 + 16 i per thread, also kept in shared memory
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + 16 * i;
    const float sh = shat[i * 8 + (lc >> 1)];
    uint32_t packed = 0;
    if (sh != 0.0f) {
      const bool fast = QuotientBracket::usable(sh);
      const QuotientBracket qb(fast ? sh : 1.0f);
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = bf16_bits_to_float(w[k] & 0xFFFFu), b = bf16_bits_to_float(w[k] >> 16);
        packed |= (fast ? e2m1x2_quotient(a, b, qb) : cvt_e2m1x2(__fdiv_rn(a, sh), __fdiv_rn(b, sh))) << (8 * k);
      }
    }
    ctile[r * 16 + lc] = packed;
    *reinterpret_cast<uint32_t*>(q_row + (tr * 128 + r) * (cols >> 1) + tc * 64 + lc * 4) = packed;
    if ((lc & 1) == 0) {  // block column b = lc / 2 -> chunk b / 4, byte (r, b % 4)
      const int b = lc >> 1;
      srow[(b >> 2) * 512 + chunk_offset(r, b & 3)] = static_cast<uint8_t>(bmax[i * 8 + b]);
    }
  }
  __syncthreads();
  // column-wise copy: thread (cq, rb, hb) transposes the codes of columns 4 cq .. 4 cq + 3 over
  // rows 32 rb + 16 hb .. + 15 (one 16x16 block), 8 bytes per column
  {
    const int lane = t & 31;
    const int hb = lane & 1;
    const int cq = (lane >> 1) + 16 * ((t >> 5) & 1);
    const int rb = t >> 6;
    const uint16_t* c16 = reinterpret_cast<const uint16_t*>(ctile);
    uint32_t p[8];  // rows 2k, 2k + 1: nibbles of columns 4 cq .. + 3 in bits 0-15 and 16-31
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int ra = rb * 32 + hb * 16 + 2 * k;
      p[k] = static_cast<uint32_t>(c16[ra * 32 + cq]) | (static_cast<uint32_t>(c16[(ra + 1) * 32 + cq]) << 16);
    }
    const int blk = (2 * rb + hb) * 8 + (cq >> 2);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w2[2] = {0, 0};
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // byte k: row 2k's nibble low, row 2k + 1's high
        const uint32_t byte = ((p[k] >> (4 * j)) & 0xFu) | ((p[k] >> (12 + 4 * j)) & 0xF0u);
        w2[k >> 2] |= byte << (8 * (k & 3));
      }
      const int c = 4 * cq + j;
      *reinterpret_cast<uint2*>(q_col + (tc * 128 + c) * (rows >> 1) + tr * 64 + rb * 16 + hb * 8) =
          make_uint2(w2[0], w2[1]);
      const int bt = 2 * rb + hb;  // block index along the transposed row
      scol[(bt >> 2) * 512 + chunk_offset(c, bt & 3)] = static_cast<uint8_t>(bmax[blk]);
    }
  }
  __syncthreads();
  // two scale chunks per copy: rows of this tile x 8 blocks of 16
  if (t < 64) {
    const int k = t >> 5, u = t & 31;
    reinterpret_cast<uint4*>(s_row + (tr * (cols >> 6) + tc * 2 + k) * 512)[u] =
        reinterpret_cast<const uint4*>(srow + k * 512)[u];
  } else if (t < 128) {
    const int k = (t - 64) >> 5, u = t & 31;
    reinterpret_cast<uint4*>(s_col + (tc * (rows >> 6) + tr * 2 + k) * 512)[u] =
        reinterpret_cast<const uint4*>(scol + k * 512)[u];
  }
}

}  // namespace mxgb
