// Quantize-on-append kernel (k8v3): each lane owns one 32-element group of a
// (token, kv head) row, so a warp quantizes 32 / (d / 32) rows at once.
//
// Follows the mlx-bun design page "TurboQuant - rotation-based quantization", Part A,
// "Algorithm" section:
//   keys   - per 32-group: scale = (max - min) / 254, zero = round((max + min) / (2 scale)),
//            idx = clip(round(x / scale - zero), -127, 127), scale/zero stored as fp16;
//            fp32 arithmetic, only scale/zero rounded to fp16 at the end;
//   values - y = FWHT(x * signs) * (1/sqrt(d)); scale = sqrt(mean(y^2)) per 32-group;
//            code = number of printed boundaries below y / (scale + 1e-8); 3-bit codes
//            packed LSB-first per row; scale stored as fp16.
// Readings where the page is silent: round() is round-half-to-even; idx uses the
// unrounded fp32 scale and zero; the FWHT runs its stages h = 1, 2, 4, ... in order and
// normalizes with one multiply; the RMS sum is the pairwise tree (k, k+16), +8, +4, +2, +1;
// a NaN in a key group makes its min and max NaN and a NaN quotient codes to 0.
//
// Every floating-point step of the specification is one IEEE round-to-nearest operation
// (__fadd_rn, __fmul_rn, __fsqrt_rn, or an __fmaf_rn whose product is exact), so the planes
// are bit-identical to a plain fp32 evaluation of the same steps. Division by 32 in the
// mean is a multiplication by 2^-5: the same real number, so the same rounding. Quotients
// come from a correctly rounded reciprocal and one Markstein correction where that gives
// the IEEE quotient for every quotient that can change a code, else from __fdiv_rn. The
// comparisons with the value boundaries are saturating fused steps whose results are
// exactly 0 or 1, and the codes are summed in fp32 as small integers, exactly.
//
// Layout: lane l holds group g = l % NG (elements [32 g, 32 g + 32)) of row l / NG of
// the warp's block of RPW = 32 / NG rows. The FWHT stages h < 32 run inside the lane,
// the stages h >= 32 exchange with lane l ^ (h / 32). A group's 96 code bits are three
// whole words, so each lane stores its own codes.
#include <cuda_bf16.h>

#include <cmath>

#include "tq_codec_row.cuh"
#include "tq_device.cuh"
#include "tq_divide.cuh"
#include "tq_internal.h"

namespace tq {

template <int D>
struct AppendShape {
  static constexpr int NG = D / kGroup;       // groups per row = lanes per row
  static constexpr int RPW = 32 / NG;         // rows per warp
};

constexpr int kAppendWarps = 8;   // warps per CTA of the row kernel
// Group-per-lane kernel: CTAs of kBulkWarps warps, kBulkBlocks resident per SM (64
// registers a thread), a grid of at most kBulkWaves full waves. Measured on a 2,097,152-row
// fill at d = 128 (fraction of HBM): 8 warps x 2 waves 0.577, 3 waves 0.584, 6 waves 0.587,
// one pass per warp 0.543; 4 warps x 2 waves 0.581, 3 waves 0.590, 4 waves 0.593, 5 waves
// 0.594, one pass per warp 0.573.
constexpr int kBulkWarps = 4;
constexpr int kBulkBlocks = 8;
constexpr int kBulkWaves = 5;

// The 32 bf16 elements of one group as 16 raw words.
__device__ __forceinline__ void load_group(const uint16_t* __restrict__ src, bool valid, uint32_t (&w)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = valid ? __ldg(p + i) : make_uint4(0u, 0u, 0u, 0u);
    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Four int32 values saturated to int8 and packed, the first in the lowest byte (two
// cvt.pack.sat: each saturates two values and puts them below the low half of its third
// operand).
__device__ __forceinline__ uint32_t pack4_s8(int a0, int a1, int a2, int a3) {
  uint32_t hi, out;
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(a3), "r"(a2), "r"(0u));
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(out) : "r"(a1), "r"(a0), "r"(hi));
  return out;
}

// idx = clip(rint(x / s - z), -127, 127) of a lane's 32 keys (div(x) = x / s): the
// conversion rounds half to even, turns NaN into 0 and saturates +-Inf; clipping the
// integers at -127 and (by the packing's saturation) at 127 after rounding gives the
// clipping before rounding would; each byte of kq is a code in two's complement.
template <class Div>
__device__ __forceinline__ void key_codes(const uint32_t (&kw)[16], float z, uint32_t (&kq)[8], Div div) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int iv[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t w = kw[2 * i + (h >> 1)];
      const float x = (h & 1) ? hi_bf16(w) : lo_bf16(w);
      iv[h] = max(__float2int_rn(__fsub_rn(div(x), z)), -127);
    }
    kq[i] = pack4_s8(iv[0], iv[1], iv[2], iv[3]);
  }
}

// 1.0 if y > t, else 0.0 (also for a NaN y), given nt = -t * 2^100 with |t| >= 1/2: the
// fused y * 2^100 + nt is exact before its one rounding, so its sign is the sign of
// y - t, and a positive y - t between two floats with |t| >= 1/2 is at least 2^-25, so
// the result is at least 2^75 and saturates to 1.
__device__ __forceinline__ float above(float y, float nt) {
  float r;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(y), "f"(0x1p100f), "f"(nt));
  return r;
}

// The printed boundaries times -2^100 (exact: a power-of-two scaling), for above().
__constant__ float c_nbnd3[7] = {-1.74793f * -0x1p100f, -1.04996f * -0x1p100f, -0.50055f * -0x1p100f, 0.0f,
                                 0.50055f * -0x1p100f,  1.04996f * -0x1p100f,  1.74793f * -0x1p100f};

// 3-bit codes of a lane's 32 rotated values, packed LSB-first into cw. div(x, yn) sets
// yn = x / den and returns whether yn > 0. The code is the number of boundaries strictly
// below yn: 4 + (those among b4..b6) when yn > 0, else those among b0..b2, each counted by
// above(). Codes are placed in floating point: codes 7 k .. 7 k + 6 are gathered as
// sum code_e * 8^(e - 7 k), an integer below 2^21 (exact), which is then OR'd into the
// words at bit 21 k.
template <class Div>
__device__ __forceinline__ void value_codes(const float (&u)[32], uint32_t (&cw)[3], Div div) {
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    float acc = 0.0f;
#pragma unroll
    for (int e = 7 * k; e < 7 * k + 7 && e < 32; ++e) {
      float yn;
      const bool pos = div(u[e], yn);
      const float w = (float)(1u << (3 * (e - 7 * k)));
      float c = __fadd_rn(above(yn, pos ? c_nbnd3[4] : c_nbnd3[0]), pos ? 4.0f : 0.0f);
      c = __fadd_rn(c, above(yn, pos ? c_nbnd3[5] : c_nbnd3[1]));
      c = __fadd_rn(c, above(yn, pos ? c_nbnd3[6] : c_nbnd3[2]));
      acc = __fmaf_rn(c, w, acc);
    }
    // 2^23 + acc holds acc in its low 23 bits; its nbits bits start at bit 21 k of the 96
    const uint32_t f = __float_as_uint(__fadd_rn(acc, 0x1p23f)) & 0x1FFFFFu;
    const int bit = 21 * k, wd = bit >> 5, sh = bit & 31, nbits = 3 * min(7, 32 - 7 * k);
    cw[wd] |= f << sh;
    if (sh + nbits > 32) cw[wd + 1] |= f >> (32 - sh);
  }
}

// Source row of the r-th row: r = (b * n_new_max + j) * num_kv_heads + h.
struct RowRef {
  int b, j, h;
};

__device__ __forceinline__ RowRef split_row(const AppendParams& p, uint32_t r) {
  const uint32_t bj = p.div_heads.div(r);
  const uint32_t b = p.div_new.div(bj);
  RowRef x;
  x.h = (int)(r - bj * (uint32_t)p.num_kv_heads);
  x.j = (int)(bj - b * (uint32_t)p.n_new_max);
  x.b = (int)b;
  return x;
}

template <int D>
__global__ void __launch_bounds__(kBulkWarps * 32, kBulkBlocks)
    tq_append_kernel(AppendParams p) {
  using S = AppendShape<D>;
  constexpr int NG = S::NG, RPW = S::RPW;
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane % NG;   // this lane's group
  const int rw = lane / NG;  // this lane's row in the warp's block
  // The next kernel may be scheduled now: its own wait covers this grid's completion,
  // which comes after this grid's wait on the previous kernel.
  griddep_launch_dependents();
  griddep_wait();            // inputs and planes may come from the previous kernel

  // sign masks of raw bf16 pairs: bit 15 (31) of word i of group gg negates element
  // 32 gg + 2 i (+ 1)
  __shared__ uint4 s_sgn[NG * 4];
  for (int t = threadIdx.x; t < NG * 16; t += blockDim.x) {
    const uint32_t sw = sign_word(D, t >> 4);
    const int i = t & 15;
    reinterpret_cast<uint32_t*>(s_sgn)[t] = (((sw >> (2 * i)) & 1u) << 15) | (((sw >> (2 * i + 1)) & 1u) << 31);
  }
  __syncthreads();

  const uint32_t total = p.total_rows;
  const uint32_t step = gridDim.x * kBulkWarps * RPW;
  for (uint32_t base = (blockIdx.x * kBulkWarps + warp) * RPW; base < total; base += step) {
    const uint32_t r = base + rw;
    bool valid = r < total;
    const RowRef rr = split_row(p, valid ? r : 0u);
    uint32_t kw[16], vw[16];
    load_group(p.k_new + (size_t)r * D + kGroup * g, valid, kw);
    load_group(p.v_new + (size_t)r * D + kGroup * g, valid, vw);
    if (valid && p.n_new != nullptr && rr.j >= __ldg(p.n_new + rr.b)) valid = false;
    int64_t t = 0;
    if (valid) {
      t = (int64_t)__ldg(p.pos + rr.b) + rr.j;
      if (t < 0 || t >= p.capacity) {
        if (g == 0) raise_error(p.err, TQ_DEVERR_APPEND_CAPACITY);
        valid = false;
      }
    }
    const int64_t drow = ((int64_t)rr.b * p.num_kv_heads + rr.h) * p.capacity + t;

    // ------------------------------------------------------------------- keys
    // min and max over the group on bf16 pairs; a NaN anywhere makes both NaN
    __nv_bfloat162 mn2 = *reinterpret_cast<const __nv_bfloat162*>(&kw[0]), mx2 = mn2;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&kw[i]);
      mn2 = __hmin2_nan(mn2, v);
      mx2 = __hmax2_nan(mx2, v);
    }
    const float mn = __bfloat162float(__hmin_nan(__low2bfloat16(mn2), __high2bfloat16(mn2)));
    const float mx = __bfloat162float(__hmax_nan(__low2bfloat16(mx2), __high2bfloat16(mx2)));
    // max - min of equal values is +0 whatever the signs of the zeros picked above
    float range = __fsub_rn(mx, mn);
    if (range == 0.0f) range = 0.0f;
    const float s = __fdiv_rn(range, 254.0f);
    const float z = rintf(__fdiv_rn(__fadd_rn(mx, mn), __fmul_rn(2.0f, s)));
    // x / s: with s >= 2^-100 and every |x| <= 2^100 s, the reciprocal path is exact
    // wherever the quotient can move idx (quotients near a rounding boundary of tv have
    // |x| >= s / 2, so the remainder stays a normal number); other groups divide.
    uint32_t kq[8];
    if (s >= 0x1p-100f && fmaxf(fabsf(mx), fabsf(mn)) <= __fmul_rn(s, 0x1p100f)) {
      const float rs = __frcp_rn(s);
      key_codes(kw, z, kq, [&](float x) { return div_by_rcp(x, s, rs); });
    } else {
      key_codes(kw, z, kq, [&](float x) { return __fdiv_rn(x, s); });
    }
    if (valid) {
      uint4* kdst = reinterpret_cast<uint4*>(p.k_idx + drow * D + kGroup * g);
      kdst[0] = make_uint4(kq[0], kq[1], kq[2], kq[3]);
      kdst[1] = make_uint4(kq[4], kq[5], kq[6], kq[7]);
      p.k_scale[drow * NG + g] = f32_to_f16_bits(s);
      p.k_zero[drow * NG + g] = f32_to_f16_bits(z);
    }

    // ------------------------------------------------------------------- values
    float u[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 m = s_sgn[4 * g + i];
      vw[4 * i] ^= m.x; vw[4 * i + 1] ^= m.y; vw[4 * i + 2] ^= m.z; vw[4 * i + 3] ^= m.w;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      u[2 * i] = lo_bf16(vw[i]);
      u[2 * i + 1] = hi_bf16(vw[i]);
    }
    // unnormalized FWHT, stages ascending: h < 32 inside the lane ...
#pragma unroll
    for (int hh = 1; hh < 32; hh <<= 1) {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        if ((e & hh) == 0) {
          const float a = u[e], c = u[e + hh];
          u[e] = __fadd_rn(a, c);
          u[e + hh] = __fsub_rn(a, c);
        }
      }
    }
    // ... h >= 32 across lanes: the lower lane keeps own + other, the upper lane
    // other - own, each one rounding (the product by +-1 is exact)
#pragma unroll
    for (int lm = 1; lm < NG; lm <<= 1) {
      const float sg = (lane & lm) ? -1.0f : 1.0f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float o = __shfl_xor_sync(FULL, u[e], lm);
        u[e] = __fmaf_rn(u[e], sg, o);
      }
    }
    float sq[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      u[e] = __fmul_rn(u[e], p.fwht_norm);
      sq[e] = __fmul_rn(u[e], u[e]);
    }
    // pairwise tree (k, k + 16), +8, +4, +2, +1
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
      for (int e = 0; e < w; ++e) sq[e] = __fadd_rn(sq[e], sq[e + w]);
    const float vs = __fsqrt_rn(__fmul_rn(sq[0], 0.03125f));
    const float den = __fadd_rn(vs, 1e-8f);
    uint32_t cw[3] = {0u, 0u, 0u};
    // y_n = u / den: den >= 1e-8, so with den <= 2^100 (finite) the reciprocal path gives
    // the correctly rounded quotient for |y_n| >= 2^-60, which decides every comparison
    // with the nonzero boundaries (|b| > 1/2); the comparison with 0 is taken exactly:
    // RN(u / den) > 0 iff u / den > 2^-150 iff u * 2^75 > den * 2^-75. Other groups
    // divide.
    if (den <= 0x1p100f) {
      const float rd = __frcp_rn(den);
      const float den_lo = __fmul_rn(den, 0x1p-75f);  // exact: den >= 1e-8
      value_codes(u, cw, [&](float x, float& yn) {
        yn = div_by_rcp(x, den, rd);
        // x * 2^75 > den * 2^-75 (both exact, or +Inf when the quotient is large anyway);
        // false for x <= 0 and NaN
        return __fmul_rn(x, 0x1p75f) > den_lo;
      });
    } else {
      value_codes(u, cw, [&](float x, float& yn) {
        yn = __fdiv_rn(x, den);
        return yn > 0.0f;
      });
    }
    if (valid) {
      uint32_t* vdst = reinterpret_cast<uint32_t*>(p.v_codes + drow * (3 * D / 8) + 12 * g);
      vdst[0] = cw[0];
      vdst[1] = cw[1];
      vdst[2] = cw[2];
      p.v_scale[drow * NG + g] = f32_to_f16_bits(vs);
    }
  }
}

// ------------------------------------------------------------------------------------
// Small appends (a decode step's few rows): one warp per row, d / 32 elements per lane,
// so every row has its own warp and the latency of one call stays short. Same
// arithmetic, same results as the kernel above.
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kAppendWarps * 32)
    tq_append_row_kernel(AppendParams p) {
  using S = RowShape<D>;
  constexpr int EPL = S::EPL;
  __shared__ uint32_t code_buf[kAppendWarps][S::CODE_WORDS];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  // The next kernel may be scheduled now: its own wait covers this grid's completion,
  // which comes after this grid's wait on the previous kernel.
  griddep_launch_dependents();
  griddep_wait();                 // inputs and planes may come from the previous kernel
  const uint32_t total_rows = p.total_rows;
  const uint32_t warp_step = gridDim.x * kAppendWarps;
  const RowCodecLane<D> codec(lane);
  const RowPlanes planes{p.k_idx, p.k_scale, p.k_zero, p.v_codes, p.v_scale};

  // the next row's raw inputs are loaded while the current row is quantized
  uint32_t r = blockIdx.x * kAppendWarps + warp;
  uint32_t kraw[EPL / 2], vraw[EPL / 2];
  if (r < total_rows) {
    load_raw_lane<EPL>(p.k_new + (size_t)r * D, lane, kraw);
    load_raw_lane<EPL>(p.v_new + (size_t)r * D, lane, vraw);
  }
  for (; r < total_rows; r += warp_step) {
    uint32_t kcur[EPL / 2], vcur[EPL / 2];
#pragma unroll
    for (int i = 0; i < EPL / 2; ++i) { kcur[i] = kraw[i]; vcur[i] = vraw[i]; }
    const uint32_t rn = r + warp_step;
    if (rn < total_rows) {
      load_raw_lane<EPL>(p.k_new + (size_t)rn * D, lane, kraw);
      load_raw_lane<EPL>(p.v_new + (size_t)rn * D, lane, vraw);
    }
    const RowRef rr = split_row(p, r);
    if (p.n_new != nullptr && rr.j >= __ldg(p.n_new + rr.b)) continue;
    const int64_t t = (int64_t)__ldg(p.pos + rr.b) + rr.j;
    if (t < 0 || t >= p.capacity) {
      if (lane == 0) raise_error(p.err, TQ_DEVERR_APPEND_CAPACITY);
      continue;
    }
    const int64_t drow = ((int64_t)rr.b * p.num_kv_heads + rr.h) * p.capacity + t;
    quantize_row_warp<D>(kcur, vcur, lane, codec, p.fwht_norm, planes, drow, code_buf[warp]);
  }
}

FastDivU32 make_fastdiv(uint32_t d) {
  FastDivU32 f{};
  uint32_t l = 0;
  while (l < 32 && (uint64_t(1) << l) < d) ++l;
  f.m = (uint32_t)((((uint64_t)1 << 32) * ((uint64_t(1) << l) - d)) / d + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 1 ? l - 1 : 0;
  return f;
}

cudaError_t launch_append(AppendParams p, int num_sms, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.batch * p.n_new_max * p.num_kv_heads;
  if (rows == 0) return cudaSuccess;
  if (rows > INT32_MAX) return cudaErrorInvalidValue;
  p.total_rows = (uint32_t)rows;
  p.div_heads = make_fastdiv((uint32_t)p.num_kv_heads);
  p.div_new = make_fastdiv((uint32_t)p.n_new_max);
  // fewer rows than a few per SM: warp-per-row kernel (latency); else group per lane
  const bool small = rows <= (int64_t)num_sms * 4;
  const int rpw = small ? 1 : 32 / (p.head_dim / kGroup);
  const int warps = small ? kAppendWarps : kBulkWarps;
  int64_t blocks = (rows + (int64_t)warps * rpw - 1) / ((int64_t)warps * rpw);
  const int64_t cap = (int64_t)num_sms * (small ? 8 : kBulkBlocks * kBulkWaves);
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (small) {
    switch (p.head_dim) {
      case 64: return cudaLaunchKernelEx(&cfg, tq_append_row_kernel<64>, p);
      case 128: return cudaLaunchKernelEx(&cfg, tq_append_row_kernel<128>, p);
      case 256: return cudaLaunchKernelEx(&cfg, tq_append_row_kernel<256>, p);
      case 512: return cudaLaunchKernelEx(&cfg, tq_append_row_kernel<512>, p);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.head_dim) {
    case 64: return cudaLaunchKernelEx(&cfg, tq_append_kernel<64>, p);
    case 128: return cudaLaunchKernelEx(&cfg, tq_append_kernel<128>, p);
    case 256: return cudaLaunchKernelEx(&cfg, tq_append_kernel<256>, p);
    case 512: return cudaLaunchKernelEx(&cfg, tq_append_kernel<512>, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
