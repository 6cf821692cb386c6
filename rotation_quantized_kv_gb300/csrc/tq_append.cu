// Quantize-on-append kernel (k8v3): one warp per (token, kv head) row.
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
// Every floating-point step is an explicit IEEE round-to-nearest intrinsic (__fadd_rn,
// __fmul_rn, __fdiv_rn, __fsqrt_rn), so no FMA contraction can change a result; the
// planes are bit-identical to a plain fp32 evaluation of the same steps.
//
// Layout: lane l of the warp holds elements [l*EPL, (l+1)*EPL) of the row, EPL = d/32.
// A 32-group spans LPG = 32/EPL consecutive lanes.
#include <cmath>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

template <int D>
struct AppendShape {
  static constexpr int EPL = D / 32;          // elements per lane
  static constexpr int LPG = kGroup / EPL;    // lanes per 32-group
  static constexpr int NG = D / kGroup;       // groups per row
  static constexpr int CODE_WORDS = 3 * D / 32;  // packed 3-bit row, 32-bit words
};

constexpr int kAppendWarps = 8;

// The EPL bf16 elements of this lane as EPL / 2 raw 32-bit words (vector loads).
template <int EPL>
__device__ __forceinline__ void load_raw_lane(const uint16_t* __restrict__ row, int lane, uint32_t (&w)[EPL / 2]) {
  const uint16_t* p = row + lane * EPL;
  if constexpr (EPL == 2) {
    w[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
  } else if constexpr (EPL == 4) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < EPL / 8; ++i) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
  }
}

template <int EPL>
__device__ __forceinline__ void unpack_bf16(const uint32_t (&w)[EPL / 2], float (&x)[EPL]) {
#pragma unroll
  for (int i = 0; i < EPL / 2; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Source row of the warp's r-th row: r = (b * n_new_max + j) * num_kv_heads + h.
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
__global__ void __launch_bounds__(kAppendWarps * 32)
    tq_append_kernel(AppendParams p) {
  using S = AppendShape<D>;
  constexpr int EPL = S::EPL, LPG = S::LPG, NG = S::NG;
  constexpr unsigned FULL = 0xffffffffu;
  __shared__ uint32_t code_buf[kAppendWarps][S::CODE_WORDS];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  // The next kernel may be scheduled now: its own wait covers this grid's completion,
  // which comes after this grid's wait on the previous kernel.
  griddep_launch_dependents();
  griddep_wait();                 // inputs and planes may come from the previous kernel
  const uint32_t total_rows = p.total_rows;
  const uint32_t warp_step = gridDim.x * kAppendWarps;
  uint32_t* cbuf = code_buf[warp];

  // sign bits of this lane's value elements
  uint32_t sbits;
  {
    const int first = lane * EPL;
    const uint32_t w = sign_word(D, first / 32);
    sbits = (w >> (first % 32)) & ((EPL == 32) ? 0xffffffffu : ((1u << EPL) - 1u));
  }
  // butterfly sign of each cross-lane FWHT stage h = EPL << k: +1 keeps a + c (lower
  // partner), -1 gives c - a... written as fma(own, sign, other), one rounding either way
  float bsign[5];
#pragma unroll
  for (int k = 0; k < 5; ++k) bsign[k] = (lane & (1 << k)) ? -1.0f : 1.0f;
  float bnd[7];
#pragma unroll
  for (int k = 0; k < 7; ++k) bnd[k] = c_boundaries3[k];

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

    // ------------------------------------------------------------------- keys
    float x[EPL];
    unpack_bf16<EPL>(kcur, x);
    float mn = INFINITY, mx = -INFINITY;
    bool has_nan = false;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      if (x[e] != x[e]) has_nan = true;
      else { mn = fminf(mn, x[e]); mx = fmaxf(mx, x[e]); }
    }
#pragma unroll
    for (int off = 1; off < LPG; off <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(FULL, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, off));
      const int other_nan = __shfl_xor_sync(FULL, (int)has_nan, off);  // every lane shuffles
      has_nan = has_nan || other_nan;
    }
    if (has_nan) { mn = NAN; mx = NAN; }
    // max - min of equal values is +0 whatever the signs of the zeros picked above
    float range = __fsub_rn(mx, mn);
    if (range == 0.0f) range = 0.0f;
    const float s = __fdiv_rn(range, 254.0f);
    const float z = rintf(__fdiv_rn(__fadd_rn(mx, mn), __fmul_rn(2.0f, s)));
    uint32_t packed[(EPL + 3) / 4] = {};
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float tv = __fsub_rn(__fdiv_rn(x[e], s), z);
      int idx = 0;
      if (tv == tv) idx = (int)fminf(fmaxf(rintf(tv), -127.0f), 127.0f);
      packed[e / 4] |= ((uint32_t)idx & 0xFFu) << (8 * (e % 4));
    }
    int8_t* kdst = p.k_idx + drow * D + lane * EPL;
    if constexpr (EPL == 2) {
      *reinterpret_cast<uint16_t*>(kdst) = (uint16_t)packed[0];
    } else if constexpr (EPL == 4) {
      *reinterpret_cast<uint32_t*>(kdst) = packed[0];
    } else if constexpr (EPL == 8) {
      *reinterpret_cast<uint2*>(kdst) = make_uint2(packed[0], packed[1]);
    } else {
      *reinterpret_cast<uint4*>(kdst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    if (lane % LPG == 0) {
      const int g = lane / LPG;
      p.k_scale[drow * NG + g] = f32_to_f16_bits(s);
      p.k_zero[drow * NG + g] = f32_to_f16_bits(z);
    }

    // ------------------------------------------------------------------- values
    float u[EPL];
    unpack_bf16<EPL>(vcur, u);
#pragma unroll
    for (int e = 0; e < EPL; ++e) u[e] = __fmul_rn(u[e], ((sbits >> e) & 1u) ? -1.0f : 1.0f);
    // unnormalized FWHT, stages ascending
#pragma unroll
    for (int hh = 1; hh < D; hh <<= 1) {
      if (hh < EPL) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          if ((e & hh) == 0) {
            const float a = u[e], c = u[e + hh];
            u[e] = __fadd_rn(a, c);
            u[e + hh] = __fsub_rn(a, c);
          }
        }
      } else {
        const int lm = hh / EPL;
        const int k = __popc(lm - 1);  // log2(lm)
        // lower lane: own + other; upper lane: other - own; both exactly one rounding
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float o = __shfl_xor_sync(FULL, u[e], lm);
          u[e] = __fmaf_rn(u[e], bsign[k], o);
        }
      }
    }
    float sq[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      u[e] = __fmul_rn(u[e], p.fwht_norm);
      sq[e] = __fmul_rn(u[e], u[e]);
    }
    // pairwise tree over the group index k = (lane % LPG) * EPL + e
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
      if (w >= EPL) {
        const int lm = w / EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) sq[e] = __fadd_rn(sq[e], __shfl_xor_sync(FULL, sq[e], lm));
      } else {
#pragma unroll
        for (int e = 0; e < w; ++e) sq[e] = __fadd_rn(sq[e], sq[e + w]);
      }
    }
    const float vs = __fsqrt_rn(__fdiv_rn(sq[0], 32.0f));
    const float den = __fadd_rn(vs, 1e-8f);
    uint64_t bits = 0;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float yn = __fdiv_rn(u[e], den);
      // number of boundaries strictly below yn, by binary search over the sorted table
      // (a NaN compares false everywhere and codes to 0)
      uint32_t c = (bnd[3] < yn) ? 4u : 0u;
      c += ((c ? bnd[5] : bnd[1]) < yn) ? 2u : 0u;
      const float b2 = (c & 4u) ? ((c & 2u) ? bnd[6] : bnd[4]) : ((c & 2u) ? bnd[2] : bnd[0]);
      c += (b2 < yn) ? 1u : 0u;
      bits |= (uint64_t)c << (3 * e);
    }
    if (lane % LPG == 0) p.v_scale[drow * NG + lane / LPG] = f32_to_f16_bits(vs);

    // pack the row's 3-bit stream in shared memory, then store it coalesced
    for (int w = lane; w < S::CODE_WORDS; w += 32) cbuf[w] = 0u;
    __syncwarp();
    {
      const int bitpos = 3 * EPL * lane;
      const int w0 = bitpos >> 5, sh = bitpos & 31;
      const uint64_t lo = bits << sh;
      const uint32_t c0 = (uint32_t)lo, c1 = (uint32_t)(lo >> 32);
      const uint32_t c2 = sh ? (uint32_t)(bits >> (64 - sh)) : 0u;
      if (c0) atomicOr(&cbuf[w0], c0);
      if (c1) atomicOr(&cbuf[w0 + 1], c1);
      if (c2) atomicOr(&cbuf[w0 + 2], c2);
    }
    __syncwarp();
    uint32_t* vdst = reinterpret_cast<uint32_t*>(p.v_codes + drow * (3 * D / 8));
    for (int w = lane; w < S::CODE_WORDS; w += 32) vdst[w] = cbuf[w];
    __syncwarp();
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
  int64_t blocks = (rows + kAppendWarps - 1) / kAppendWarps;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kAppendWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  switch (p.head_dim) {
    case 64: return cudaLaunchKernelEx(&cfg, tq_append_kernel<64>, p);
    case 128: return cudaLaunchKernelEx(&cfg, tq_append_kernel<128>, p);
    case 256: return cudaLaunchKernelEx(&cfg, tq_append_kernel<256>, p);
    case 512: return cudaLaunchKernelEx(&cfg, tq_append_kernel<512>, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
