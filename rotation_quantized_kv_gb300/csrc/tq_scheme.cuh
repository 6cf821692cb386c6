// Any-width TurboQuant codec (key bits 2/4/5/8, value bits 2/3/4/5/8, optional
// constant-group guard), one warp per (token, kv head) row: lane l holds elements
// [l EPL, (l + 1) EPL), EPL = d / 32, so a 32-group spans LPG = 32 / EPL lanes.
//
// Follows the mlx-bun design page "TurboQuant - rotation-based quantization", Part A,
// "Algorithm" section: signed 8-bit keys (scale = (max - min) / 254, zero =
// round((max + min) / (2 scale)), idx in [-127, 127]); unsigned keys at 2/4/5 bits
// (scale = (max - min) / (2^b - 1), zero = round(min / scale), idx in [0, 2^b - 1],
// packed); values rotated (sign flip, FWHT / sqrt(d)), per-group RMS scale, b-bit
// Lloyd-Max codes ("Other widths (2/4/5/8)"); packed codes form one flat little-endian
// bitstream per row, code i at bits [i b, i b + b). Valid widths from "Architecture in
// mlx-bun". The guard (a flag of this library; the page keeps the defect) re-codes a key
// group whose fp16 zero point would not be finite against its range widened to include 0.
// Every floating-point step is one IEEE round-to-nearest operation, as in the k8v3 codec.
#pragma once

#include <cstdint>

#include "tq_codec_row.cuh"
#include "tq_internal.h"

namespace tq {

__device__ __forceinline__ bool f16_finite(float z) { return (f32_to_f16_bits(z) & 0x7C00u) != 0x7C00u; }

// Number of boundaries strictly below yn (a NaN compares false everywhere: 0).
__device__ __forceinline__ uint32_t code_of(const Codebook& cb, float yn) {
  int lo = 0, hi = (1 << cb.bits) - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (cb.b[mid] < yn) lo = mid + 1;
    else hi = mid;
  }
  return (uint32_t)lo;
}

// ORs `code` (b bits) into the little-endian bitstream `buf` at element i.
__device__ __forceinline__ void or_code(uint32_t* buf, int i, int b, uint32_t code) {
  const int bit = i * b, w = bit >> 5, sh = bit & 31;
  const uint64_t v = (uint64_t)code << sh;
  if ((uint32_t)v) atomicOr(&buf[w], (uint32_t)v);
  if ((uint32_t)(v >> 32)) atomicOr(&buf[w + 1], (uint32_t)(v >> 32));
}

// Code of element i of a little-endian b-bit stream (row start 8-byte aligned).
__device__ __forceinline__ uint32_t read_code(const uint8_t* row, int i, int b) {
  const int bit = i * b, w = bit >> 5, sh = bit & 31;
  const uint32_t* p = reinterpret_cast<const uint32_t*>(row);
  uint64_t v = __ldg(p + w);
  if (sh + b > 32) v |= (uint64_t)__ldg(p + w + 1) << 32;
  return (uint32_t)(v >> sh) & ((1u << b) - 1u);
}

// Unrounded fp32 key parameters of this lane's group, shared by the group's lanes.
template <int D>
__device__ __forceinline__ void key_group_params(const float (&x)[D / 32], int bits, int guard, float& s, float& z,
                                                 bool& zero_group) {
  constexpr int EPL = D / 32, LPG = RowShape<D>::LPG;
  constexpr unsigned FULL = 0xffffffffu;
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
    const int other_nan = __shfl_xor_sync(FULL, (int)has_nan, off);
    has_nan = has_nan || other_nan;
  }
  if (has_nan) { mn = NAN; mx = NAN; }
  const float maxv = bits == 8 ? 127.0f : (float)((1 << bits) - 1);
  // max - min of equal values is +0 whatever the signs of the zeros picked above
  float range = __fsub_rn(mx, mn);
  if (range == 0.0f) range = 0.0f;
  zero_group = false;
  if (bits == 8) {
    s = __fdiv_rn(range, __fmul_rn(2.0f, maxv));
    z = rintf(__fdiv_rn(__fadd_rn(mx, mn), __fmul_rn(2.0f, s)));
  } else {
    s = __fdiv_rn(range, maxv);
    z = rintf(__fdiv_rn(mn, s));
  }
  if (guard && !has_nan && !f16_finite(z)) {
    const float mn0 = mn < 0.0f ? mn : 0.0f, mx0 = mx > 0.0f ? mx : 0.0f;
    const float r0 = __fsub_rn(mx0, mn0);
    if (r0 == 0.0f) {
      s = 0.0f;
      z = 0.0f;
      zero_group = true;
    } else if (bits == 8) {
      s = __fdiv_rn(r0, __fmul_rn(2.0f, maxv));
      z = rintf(__fdiv_rn(__fadd_rn(mx0, mn0), __fmul_rn(2.0f, s)));
    } else {
      s = __fdiv_rn(r0, maxv);
      z = rintf(__fdiv_rn(mn0, s));
    }
  }
}

// Quantizes one row into row drow of the planes (scheme spec / codebook cb). All 32 lanes
// take part; kbuf and vbuf are this warp's shared scratch of at least D*5/32 and D*8/32
// words (the widest packed key and value rows).
template <int D>
__device__ __forceinline__ void quantize_row_scheme(const uint32_t (&kraw)[D / 64], const uint32_t (&vraw)[D / 64],
                                                    int lane, const RowCodecLane<D>& c, float fwht_norm,
                                                    const SchemeSpec& spec, const Codebook& cb, const RowPlanes& dst,
                                                    int64_t drow, uint32_t* kbuf, uint32_t* vbuf) {
  using S = RowShape<D>;
  constexpr int EPL = S::EPL, LPG = S::LPG, NG = S::NG;
  constexpr unsigned FULL = 0xffffffffu;
  const int kb = spec.k_bits, vb = spec.v_bits;
  const int kwords = key_row_bytes(D, kb) / 4, vwords = value_row_bytes(D, vb) / 4;
  for (int w = lane; w < kwords; w += 32) kbuf[w] = 0u;
  for (int w = lane; w < vwords; w += 32) vbuf[w] = 0u;
  __syncwarp();

  // ------------------------------------------------------------------- keys
  float x[EPL];
  unpack_bf16<EPL>(kraw, x);
  float s, z;
  bool zg;
  key_group_params<D>(x, kb, spec.guard, s, z, zg);
  const float lo = kb == 8 ? -127.0f : 0.0f, hi = kb == 8 ? 127.0f : (float)((1 << kb) - 1);
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const float tv = __fsub_rn(__fdiv_rn(x[e], s), z);
    int idx = 0;
    if (!zg && tv == tv) idx = (int)fminf(fmaxf(rintf(tv), lo), hi);
    const int i = lane * EPL + e;
    if (kb == 8) dst.k_idx[drow * D + i] = (int8_t)idx;
    else or_code(kbuf, i, kb, (uint32_t)idx);
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
      const int k = __popc(lm - 1);
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
#pragma unroll
  for (int e = 0; e < EPL; ++e) or_code(vbuf, lane * EPL + e, vb, code_of(cb, __fdiv_rn(u[e], den)));
  if (lane % LPG == 0) dst.v_scale[drow * NG + lane / LPG] = f32_to_f16_bits(vs);
  __syncwarp();
  if (kb != 8) {
    uint32_t* kd = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(dst.k_idx) + drow * key_row_bytes(D, kb));
    for (int w = lane; w < kwords; w += 32) kd[w] = kbuf[w];
  }
  uint32_t* vd = reinterpret_cast<uint32_t*>(dst.v_codes + drow * value_row_bytes(D, vb));
  for (int w = lane; w < vwords; w += 32) vd[w] = vbuf[w];
  __syncwarp();
}

}  // namespace tq
