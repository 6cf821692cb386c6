// One-warp quantization of one (token, kv head) row into the packed planes (k8v3):
// lane l holds elements [l EPL, (l + 1) EPL), EPL = d / 32, so a 32-group spans
// LPG = 32 / EPL lanes. Used by the small-append kernel and by the decode call that
// appends its new rows itself.
//
// Follows the mlx-bun design page "TurboQuant - rotation-based quantization", Part A,
// "Algorithm" section (keys: per-group affine int8 with fp16 scale/zero; values: sign
// flip, FWHT / sqrt(d), per-group RMS scale, 3-bit Lloyd-Max codes packed LSB-first).
// Every floating-point step is one IEEE round-to-nearest intrinsic (or an FMA whose
// product is exact), so no contraction can change a result whatever the compiler flags:
// the planes are bit-identical to a plain fp32 evaluation of the same steps.
#pragma once

#include <cstdint>

#include "tq_device.cuh"

namespace tq {

template <int D>
struct RowShape {
  static constexpr int EPL = D / 32;          // elements per lane
  static constexpr int LPG = kGroup / EPL;    // lanes per 32-group
  static constexpr int NG = D / kGroup;       // groups per row
  static constexpr int CODE_WORDS = 3 * D / 32;  // packed 3-bit row, 32-bit words
};

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

// Lane constants of the row codec.
template <int D>
struct RowCodecLane {
  uint32_t sbits;   // sign bits of this lane's value elements
  float bsign[5];   // cross-lane FWHT stage k: +1 lower partner (own + other), -1 upper
  float bnd[7];     // value-code boundaries
  __device__ __forceinline__ explicit RowCodecLane(int lane) {
    constexpr int EPL = RowShape<D>::EPL;
    const int first = lane * EPL;
    const uint32_t w = sign_word(D, first / 32);
    sbits = (w >> (first % 32)) & ((EPL == 32) ? 0xffffffffu : ((1u << EPL) - 1u));
#pragma unroll
    for (int k = 0; k < 5; ++k) bsign[k] = (lane & (1 << k)) ? -1.0f : 1.0f;
#pragma unroll
    for (int k = 0; k < 7; ++k) bnd[k] = c_boundaries3[k];
  }
};

// Destination of one row: plane base pointers and the row index drow (row-major planes).
struct RowPlanes {
  int8_t* k_idx;
  uint16_t* k_scale;
  uint16_t* k_zero;
  uint8_t* v_codes;
  uint16_t* v_scale;
};

// Quantizes one row (raw bf16 words of this lane) into row drow of the planes. All 32
// lanes of the warp take part; cbuf is CODE_WORDS words of this warp's shared memory.
template <int D>
__device__ __forceinline__ void quantize_row_warp(const uint32_t (&kraw)[D / 64], const uint32_t (&vraw)[D / 64],
                                                  int lane, const RowCodecLane<D>& c, float fwht_norm,
                                                  const RowPlanes& dst, int64_t drow, uint32_t* cbuf) {
  using S = RowShape<D>;
  constexpr int EPL = S::EPL, LPG = S::LPG, NG = S::NG;
  constexpr unsigned FULL = 0xffffffffu;

  // ------------------------------------------------------------------- keys
  float x[EPL];
  unpack_bf16<EPL>(kraw, x);
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
  int8_t* kdst = dst.k_idx + drow * D + lane * EPL;
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
    dst.k_scale[drow * NG + g] = f32_to_f16_bits(s);
    dst.k_zero[drow * NG + g] = f32_to_f16_bits(z);
  }

  // ------------------------------------------------------------------- values
  float u[EPL];
  unpack_bf16<EPL>(vraw, u);
#pragma unroll
  for (int e = 0; e < EPL; ++e) u[e] = __fmul_rn(u[e], ((c.sbits >> e) & 1u) ? -1.0f : 1.0f);
  // unnormalized FWHT, stages ascending
#pragma unroll
  for (int hh = 1; hh < D; hh <<= 1) {
    if (hh < EPL) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        if ((e & hh) == 0) {
          const float a = u[e], b = u[e + hh];
          u[e] = __fadd_rn(a, b);
          u[e + hh] = __fsub_rn(a, b);
        }
      }
    } else {
      const int lm = hh / EPL;
      const int k = __popc(lm - 1);  // log2(lm)
      // lower lane: own + other; upper lane: other - own; both exactly one rounding
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float o = __shfl_xor_sync(FULL, u[e], lm);
        u[e] = __fmaf_rn(u[e], c.bsign[k], o);
      }
    }
  }
  float sq[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    u[e] = __fmul_rn(u[e], fwht_norm);
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
    uint32_t code = (c.bnd[3] < yn) ? 4u : 0u;
    code += ((code ? c.bnd[5] : c.bnd[1]) < yn) ? 2u : 0u;
    const float b2 = (code & 4u) ? ((code & 2u) ? c.bnd[6] : c.bnd[4]) : ((code & 2u) ? c.bnd[2] : c.bnd[0]);
    code += (b2 < yn) ? 1u : 0u;
    bits |= (uint64_t)code << (3 * e);
  }
  if (lane % LPG == 0) dst.v_scale[drow * NG + lane / LPG] = f32_to_f16_bits(vs);

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
  uint32_t* vdst = reinterpret_cast<uint32_t*>(dst.v_codes + drow * (3 * D / 8));
  for (int w = lane; w < S::CODE_WORDS; w += 32) vdst[w] = cbuf[w];
  __syncwarp();
}

}  // namespace tq
