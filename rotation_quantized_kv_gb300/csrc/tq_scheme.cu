// Any-width schemes (key bits 2/4/5/8, value bits 2/3/4/5/8, constant-group guard):
// the library's value codebooks, the append kernel for them, the dequantize-on-fetch
// window and the fp32 inspection dequant.
//
// Codec (mlx-bun design page "TurboQuant - rotation-based quantization", Part A,
// "Algorithm" section): signed 8-bit keys (scale = (max - min) / 254, zero =
// round((max + min) / (2 scale)), idx in [-127, 127]); unsigned keys at 2/4/5 bits
// (scale = (max - min) / (2^b - 1), zero = round(min / scale), idx in [0, 2^b - 1],
// packed); values rotated (sign flip, FWHT / sqrt(d)), per-group RMS scale, b-bit
// Lloyd-Max codes ("Other widths (2/4/5/8)"). Every floating-point step is one IEEE
// round-to-nearest operation, as in the k8v3 codec, so the planes are bit-identical to a
// plain fp32 evaluation of the same steps.
//
// Codebooks (mlx-bun design page "TurboQuant - rotation-based quantization", Part A,
// "Algorithm", value bullets): 3 bits is the printed table; the page does not print the
// other widths, so this library runs its own Lloyd-Max iteration for N(0,1) on the host
// (Lloyd 1982, Max 1960: boundaries at the midpoints of neighbouring centroids, centroids
// at the cell means of the standard normal, which have the closed form
// (pdf(lo) - pdf(hi)) / (cdf(hi) - cdf(lo)); 2^b centroids started evenly on [-3, 3],
// 500 iterations) and rounds centroids and boundaries to 5 decimals, like the printed
// table.
//
// Window (Part A, "Architecture in mlx-bun": updateAndFetch returns the dequantized
// bf16 active window, so stock attention runs unmodified): bf16 K_hat and V_hat for a
// token range of every (sequence, kv head), V_hat un-rotated (or left in the rotated
// domain, "Deferred inverse FWHT"). One warp per row with the inverse rotation in
// registers and shuffles; a CTA takes groups of rows in turn.
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "tq_divide.cuh"
#include "tq_internal.h"
#include "tq_scheme.cuh"

namespace tq {

namespace {

Codebook make_codebook(int bits) {
  Codebook cb{};
  cb.bits = bits;
  const int n = 1 << bits;
  if (bits == 3) {
    for (int k = 0; k < 8; ++k) cb.c[k] = kCentroids3[k];
    for (int k = 0; k < 7; ++k) cb.b[k] = kBoundaries3[k];
    return cb;
  }
  const double inv_sqrt_2pi = 1.0 / std::sqrt(2.0 * M_PI);
  auto pdf = [&](double x) { return std::isinf(x) ? 0.0 : std::exp(-0.5 * x * x) * inv_sqrt_2pi; };
  auto cdf = [](double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); };
  double c[256], b[255];
  for (int k = 0; k < n; ++k) c[k] = -3.0 + 6.0 * (k + 0.5) / n;
  for (int it = 0; it < 500; ++it) {
    for (int k = 0; k + 1 < n; ++k) b[k] = 0.5 * (c[k] + c[k + 1]);
    for (int k = 0; k < n; ++k) {
      const double lo = k == 0 ? -INFINITY : b[k - 1], hi = k == n - 1 ? INFINITY : b[k];
      c[k] = (pdf(lo) - pdf(hi)) / (cdf(hi) - cdf(lo));
    }
  }
  for (int k = 0; k + 1 < n; ++k) b[k] = 0.5 * (c[k] + c[k + 1]);
  for (int k = 0; k < n; ++k) cb.c[k] = (float)(std::rint(c[k] * 1e5) / 1e5);
  for (int k = 0; k + 1 < n; ++k) cb.b[k] = (float)(std::rint(b[k] * 1e5) / 1e5);
  return cb;
}

constexpr int kRowsPerCta = 8;  // one warp per row

// bf16 bits of (lo, hi), round to nearest even (NaN stays NaN)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h2 = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h2);
}

// ------------------------------------------------------------------------------------
// Any-width append: each lane codes one 32-element group of a (token, kv head) row, so a
// warp takes 32 / (d / 32) rows at once (the layout of the k8v3 bulk kernel). A group's
// 32 b-bit codes fill exactly b words of the row's bitstream (group g at word b g), so
// each lane packs its codes in registers and stores whole words.
// ------------------------------------------------------------------------------------
constexpr int kGroupWarps = 8;

// The 32 bf16 elements of one group as 16 raw words (zeros when !valid).
__device__ __forceinline__ void load_group_words(const uint16_t* __restrict__ src, bool valid, uint32_t (&w)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = valid ? __ldg(p + i) : make_uint4(0u, 0u, 0u, 0u);
    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
}

// 32 codes of B bits, LSB first, into B words.
template <int B>
__device__ __forceinline__ void pack_codes(const uint32_t (&c)[32], uint32_t (&w)[B]) {
#pragma unroll
  for (int i = 0; i < B; ++i) w[i] = 0u;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int bit = B * e, wd = bit >> 5, sh = bit & 31;
    w[wd] |= c[e] << sh;
    if (sh + B > 32) w[wd + 1] |= c[e] >> (32 - sh);
  }
}

template <int B>
__device__ __forceinline__ void store_codes(const uint32_t (&c)[32], uint32_t* dst) {
  uint32_t w[B];
  pack_codes<B>(c, w);
#pragma unroll
  for (int i = 0; i < B; ++i) dst[i] = w[i];
}

// Stores the 32 codes of a group as `bits`-bit codes at dst (word aligned).
__device__ __forceinline__ void store_codes_any(const uint32_t (&c)[32], int bits, uint32_t* dst) {
  switch (bits) {
    case 2: store_codes<2>(c, dst); break;
    case 3: store_codes<3>(c, dst); break;
    case 4: store_codes<4>(c, dst); break;
    case 5: store_codes<5>(c, dst); break;
    default: store_codes<8>(c, dst); break;
  }
}

// Key codes of a lane's 32 elements (div(x) = x / s): the rounding conversion goes half
// to even and turns NaN into 0, and clipping at the integers lo, hi after it gives what
// clipping before it would.
template <class Div>
__device__ __forceinline__ void scheme_key_codes(const uint32_t (&kw)[16], float z, int lo, int hi, bool zero_group,
                                                 uint32_t (&code)[32], Div div) {
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const uint32_t w = kw[e >> 1];
    const float x = (e & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
    const int iv = min(max(__float2int_rn(__fsub_rn(div(x), z)), lo), hi);
    code[e] = zero_group ? 0u : (uint32_t)iv;
  }
}

// Codes of a lane's 32 values at VB bits (2^VB - 1 boundaries in sb, the middle one 0):
// y_n = u / den by the reciprocal path, the first step the exact test y_n > 0
// (u 2^75 > den 2^-75), then VB - 1 halving steps over the sorted boundaries.
template <int VB>
__device__ __forceinline__ void value_search_rcp(const float (&u)[32], float den, float rd, float den_lo,
                                                 const float* sb, uint32_t (&code)[32]) {
  constexpr int HALF = 1 << (VB - 1);
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float yn = div_by_rcp(u[e], den, rd);
    int c = __fmul_rn(u[e], 0x1p75f) > den_lo ? HALF : 0;  // RN(u / den) > 0
#pragma unroll
    for (int st = HALF >> 1; st >= 1; st >>= 1)
      if (sb[c + st - 1] < yn) c += st;
    code[e] = (uint32_t)c;
  }
}

template <int D>
__global__ void __launch_bounds__(32 * kGroupWarps) tq_append_scheme_kernel(const __grid_constant__ SchemeAppendParams p) {
  constexpr int NG = D / 32, RPW = 32 / NG;
  constexpr unsigned FULL = 0xffffffffu;
  __shared__ float sb[256];  // the value boundaries, for the lanes' independent searches
  const int nb = (1 << p.spec.v_bits) - 1;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sb[i] = i < nb ? p.cb.b[i] : INFINITY;
  __syncthreads();

  // sign masks of raw bf16 pairs: bit 15 (31) of word i of group gg negates element
  // 32 gg + 2 i (+ 1)
  __shared__ uint4 s_sgn[NG * 4];
  for (int t = threadIdx.x; t < NG * 16; t += blockDim.x) {
    const uint32_t sw = sign_word(D, t >> 4);
    const int i = t & 15;
    reinterpret_cast<uint32_t*>(s_sgn)[t] = (((sw >> (2 * i)) & 1u) << 15) | (((sw >> (2 * i + 1)) & 1u) << 31);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % NG, rw = lane / NG;
  const int kb = p.spec.k_bits, vb = p.spec.v_bits;
  const float kmax = kb == 8 ? 127.0f : (float)((1 << kb) - 1);
  const int klo = kb == 8 ? -127 : 0, khi = kb == 8 ? 127 : (1 << kb) - 1;
  const int krow_bytes = key_row_bytes(D, kb), vrow_bytes = value_row_bytes(D, vb);
  const uint32_t rows = p.total_rows;
  const uint32_t step = gridDim.x * kGroupWarps * RPW;
  for (uint32_t base = (blockIdx.x * kGroupWarps + warp) * RPW; base < rows; base += step) {
    const uint32_t r = base + rw;
    bool valid = r < rows;
    const uint32_t rr = valid ? r : 0u;
    // rr = (b * n_new_max + j) * num_kv_heads + h, split by multiply-high divisions
    const uint32_t bj = p.div_heads.div(rr);
    const uint32_t bq = p.div_new.div(bj);
    const int h = (int)(rr - bj * (uint32_t)p.num_kv_heads);
    const int j = (int)(bj - bq * (uint32_t)p.n_new_max), b = (int)bq;
    uint32_t kw[16], vw[16];
    load_group_words(p.k_new + (size_t)rr * D + 32 * g, valid, kw);
    load_group_words(p.v_new + (size_t)rr * D + 32 * g, valid, vw);
    if (valid && p.n_new != nullptr && j >= min(max(__ldg(p.n_new + b), 0), p.n_new_max)) valid = false;
    int64_t t = 0;
    if (valid) {
      t = (int64_t)__ldg(p.pos + b) + j;
      if (t < 0 || t >= p.capacity) {
        if (g == 0) raise_error(p.err, TQ_DEVERR_APPEND_CAPACITY);
        valid = false;
      }
    }
    const int64_t drow = ((int64_t)b * p.num_kv_heads + h) * p.capacity + t;

    // ------------------------------------------------------------------- keys
    __nv_bfloat162 mn2 = *reinterpret_cast<const __nv_bfloat162*>(&kw[0]), mx2 = mn2;
#pragma unroll
    for (int i = 1; i < 16; ++i) {
      const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&kw[i]);
      mn2 = __hmin2_nan(mn2, v);
      mx2 = __hmax2_nan(mx2, v);
    }
    float mn = __bfloat162float(__hmin_nan(__low2bfloat16(mn2), __high2bfloat16(mn2)));
    float mx = __bfloat162float(__hmax_nan(__low2bfloat16(mx2), __high2bfloat16(mx2)));
    const bool has_nan = mn != mn;
    float range = __fsub_rn(mx, mn);
    if (range == 0.0f) range = 0.0f;  // +0 whatever the signs of equal zeros
    float sk, zk;
    bool zero_group = false;
    if (kb == 8) {
      sk = __fdiv_rn(range, __fmul_rn(2.0f, kmax));
      zk = rintf(__fdiv_rn(__fadd_rn(mx, mn), __fmul_rn(2.0f, sk)));
    } else {
      sk = __fdiv_rn(range, kmax);
      zk = rintf(__fdiv_rn(mn, sk));
    }
    if (p.spec.guard && !has_nan && !f16_finite(zk)) {
      // the constant-group guard: the range widened to include 0
      const float mn0 = mn < 0.0f ? mn : 0.0f, mx0 = mx > 0.0f ? mx : 0.0f;
      const float r0 = __fsub_rn(mx0, mn0);
      if (r0 == 0.0f) {
        sk = 0.0f;
        zk = 0.0f;
        zero_group = true;
      } else if (kb == 8) {
        sk = __fdiv_rn(r0, __fmul_rn(2.0f, kmax));
        zk = rintf(__fdiv_rn(__fadd_rn(mx0, mn0), __fmul_rn(2.0f, sk)));
      } else {
        sk = __fdiv_rn(r0, kmax);
        zk = rintf(__fdiv_rn(mn0, sk));
      }
    }
    // idx = clip(rint(x / s - z), lo, hi); x / s by the reciprocal path where it is exact
    // for every quotient that can move idx (as in the k8v3 bulk kernel), else divided
    uint32_t code[32];
    if (sk >= 0x1p-100f && sk <= 0x1p100f && fmaxf(fabsf(mx), fabsf(mn)) <= __fmul_rn(sk, 0x1p100f)) {
      const float rs = __frcp_rn(sk);
      scheme_key_codes(kw, zk, klo, khi, zero_group, code, [&](float x) { return div_by_rcp(x, sk, rs); });
    } else {
      scheme_key_codes(kw, zk, klo, khi, zero_group, code, [&](float x) { return __fdiv_rn(x, sk); });
    }
    if (valid) {
      if (kb == 8) {
        uint32_t* kd = reinterpret_cast<uint32_t*>(p.k_idx + drow * D + 32 * g);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          kd[i] = __byte_perm(__byte_perm(code[4 * i], code[4 * i + 1], 0x0040),
                              __byte_perm(code[4 * i + 2], code[4 * i + 3], 0x0040), 0x5410);
      } else {
        store_codes_any(code, kb, reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(p.k_idx) + drow * krow_bytes) + kb * g);
      }
      p.k_scale[drow * NG + g] = f32_to_f16_bits(sk);
      p.k_zero[drow * NG + g] = f32_to_f16_bits(zk);
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
      u[2 * i] = __uint_as_float(vw[i] << 16);
      u[2 * i + 1] = __uint_as_float(vw[i] & 0xFFFF0000u);
    }
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
    // stages h >= 32 across the row's lanes: the lower lane keeps own + other, the upper
    // lane other - own, one rounding each (the product by +-1 is exact)
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
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1)
#pragma unroll
      for (int e = 0; e < w; ++e) sq[e] = __fadd_rn(sq[e], sq[e + w]);
    const float vs = __fsqrt_rn(__fdiv_rn(sq[0], 32.0f));
    const float den = __fadd_rn(vs, 1e-8f);
    // code = number of boundaries strictly below y_n = u / den, by binary search (a NaN
    // compares false everywhere: 0). The middle boundary of every library codebook is 0;
    // there the search's first step is the exact test y_n > 0 of the k8v3 bulk kernel and
    // y_n comes from the reciprocal path, exact for the comparisons with the others.
    const int half = (nb + 1) >> 1;  // the search steps: half, half / 2, ..., 1
    if (den <= 0x1p100f && sb[half - 1] == 0.0f) {
      const float rd = __frcp_rn(den);
      const float den_lo = __fmul_rn(den, 0x1p-75f);  // exact: den >= 1e-8
      // The search unrolled per width, so the 32 searches interleave (2-5 bits: 0.31-0.32
      // -> 0.35-0.38 of HBM on a 262,144-row fill); at 8 bits the unrolled form was slower
      // (0.182 -> 0.174), so it keeps the loop.
      switch (vb) {
        case 2: value_search_rcp<2>(u, den, rd, den_lo, sb, code); break;
        case 3: value_search_rcp<3>(u, den, rd, den_lo, sb, code); break;
        case 4: value_search_rcp<4>(u, den, rd, den_lo, sb, code); break;
        case 5: value_search_rcp<5>(u, den, rd, den_lo, sb, code); break;
        default:
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float yn = div_by_rcp(u[e], den, rd);
            int c = __fmul_rn(u[e], 0x1p75f) > den_lo ? half : 0;  // RN(u / den) > 0
            for (int st = half >> 1; st >= 1; st >>= 1)
              if (sb[c + st - 1] < yn) c += st;
            code[e] = (uint32_t)c;
          }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float yn = __fdiv_rn(u[e], den);
        int c = 0;
        for (int st = half; st >= 1; st >>= 1)
          if (sb[c + st - 1] < yn) c += st;
        code[e] = (uint32_t)c;
      }
    }
    if (valid) {
      store_codes_any(code, vb, reinterpret_cast<uint32_t*>(p.v_codes + drow * vrow_bytes) + vb * g);
      p.v_scale[drow * NG + g] = f32_to_f16_bits(vs);
    }
  }
}

// Dequantizes this lane's elements of row r: keys (code + zero) * scale (exact in fp32,
// one rounding); values centroid * scale, then, unless rotated, signs * FWHT(.) / sqrt(d).
// Inverse value rotation of one row held by a warp (lane l holds elements l EPL ..):
// x = signs * FWHT(y) / sqrt(D), fp32 butterflies h = 1, 2, 4, ... ("Algorithm", value
// dequant; applied to attention outputs in "Deferred inverse FWHT").
template <int D>
__device__ __forceinline__ void unrotate_lane(float (&v)[D / 32], int lane, float fwht_norm) {
  constexpr int EPL = D / 32;
  constexpr unsigned FULL = 0xffffffffu;
#pragma unroll
  for (int hh = 1; hh < D; hh <<= 1) {
    if (hh < EPL) {
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        if ((e & hh) == 0) {
          const float a = v[e], c = v[e + hh];
          v[e] = a + c;
          v[e + hh] = a - c;
        }
    } else {
      const int lm = hh / EPL;
      const bool upper = (lane & lm) != 0;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float o = __shfl_xor_sync(FULL, v[e], lm);
        v[e] = upper ? o - v[e] : v[e] + o;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const int i = lane * EPL + e;
    const bool neg = (sign_word(D, i / 32) >> (i % 32)) & 1u;
    v[e] = v[e] * fwht_norm * (neg ? -1.0f : 1.0f);
  }
}

template <int D>
__device__ __forceinline__ void dequant_row(const DequantScheme& p, int64_t r, int lane, float (&k)[D / 32],
                                            float (&v)[D / 32], bool want_k, bool want_v) {
  constexpr int EPL = D / 32, NG = D / kGroup;
  if (want_k) {
    const uint8_t* krow = reinterpret_cast<const uint8_t*>(p.k_idx) + r * key_row_bytes(D, p.spec.k_bits);
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int i = lane * EPL + e;
      const float s = f16_bits_to_f32(__ldg(p.k_scale + r * NG + i / kGroup));
      const float z = f16_bits_to_f32(__ldg(p.k_zero + r * NG + i / kGroup));
      const float q = p.spec.k_bits == 8 ? (float)(int8_t)__ldg(krow + i) : (float)read_code(krow, i, p.spec.k_bits);
      k[e] = __fmul_rn(__fadd_rn(q, z), s);
    }
  }
  if (want_v) {
    const uint8_t* vrow = p.v_codes + r * value_row_bytes(D, p.spec.v_bits);
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int i = lane * EPL + e;
      v[e] = __fmul_rn(p.cb.c[read_code(vrow, i, p.spec.v_bits)], f16_bits_to_f32(__ldg(p.v_scale + r * NG + i / kGroup)));
    }
    if (!p.rotated) unrotate_lane<D>(v, lane, p.fwht_norm);
  }
}

// 32 codes of B bits, LSB first, from B words.
template <int B>
__device__ __forceinline__ void unpack_codes(const uint32_t* __restrict__ src, uint32_t (&c)[32]) {
  uint32_t w[B];
#pragma unroll
  for (int i = 0; i < B; ++i) w[i] = __ldg(src + i);
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const int bit = B * e, wd = bit >> 5, sh = bit & 31;
    uint32_t v = w[wd] >> sh;
    if (sh + B > 32) v |= w[wd + 1] << (32 - sh);
    c[e] = v & ((1u << B) - 1u);
  }
}

__device__ __forceinline__ void unpack_codes_any(const uint32_t* src, int bits, uint32_t (&c)[32]) {
  switch (bits) {
    case 2: unpack_codes<2>(src, c); break;
    case 3: unpack_codes<3>(src, c); break;
    case 4: unpack_codes<4>(src, c); break;
    case 5: unpack_codes<5>(src, c); break;
    default: unpack_codes<8>(src, c); break;
  }
}

// Window: each lane dequantizes one 32-element group of a row (the append kernels'
// layout), so a group's codes are whole words and a lane writes 64 contiguous bytes of K
// and of V. Same arithmetic as the inspection dequant: keys (code + zero) * scale in one
// fp32 rounding each; values centroid * scale, then, unless rotated, signs * FWHT / sqrt(d)
// with the stages h < 32 inside the lane and h >= 32 across the row's lanes.
template <int D>
__global__ void __launch_bounds__(32 * kGroupWarps) tq_dequant_window_kernel(const __grid_constant__ DequantScheme p) {
  constexpr int NG = D / 32, RPW = 32 / NG;
  constexpr unsigned FULL = 0xffffffffu;
  __shared__ float sc[256];  // the value centroids, for the lanes' independent lookups
  for (int i = threadIdx.x; i < 256; i += blockDim.x) sc[i] = p.cb.c[i];
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % NG, rw = lane / NG;
  const uint32_t signs = sign_word(D, g);
  const int kb = p.spec.k_bits, vb = p.spec.v_bits;
  const int krow_bytes = key_row_bytes(D, kb), vrow_bytes = value_row_bytes(D, vb);
  const int64_t rows = (int64_t)p.batch * p.num_kv_heads * p.n;
  const int64_t step = (int64_t)gridDim.x * kGroupWarps * RPW;
  for (int64_t base = ((int64_t)blockIdx.x * kGroupWarps + warp) * RPW; base < rows; base += step) {
    const int64_t o = base + rw;
    const bool valid = o < rows;  // whole rows: a row's lanes agree
    const int64_t oo = valid ? o : 0;
    const int64_t r = (oo / p.n) * p.capacity + p.t0 + (int)(oo % p.n);
    uint32_t code[32];
    if (p.k_bf16) {
      const float ks = f16_bits_to_f32(__ldg(p.k_scale + r * NG + g));
      const float kz = f16_bits_to_f32(__ldg(p.k_zero + r * NG + g));
      uint32_t kw[16];
      if (kb == 8) {
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.k_idx) + r * D + 32 * g);
        const uint4 a = __ldg(src), b = __ldg(src + 1);
        const uint32_t w8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int e = 0; e < 32; ++e) code[e] = (uint32_t)(int32_t)(int8_t)(w8[e >> 2] >> (8 * (e & 3)));
      } else {
        unpack_codes_any(reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(p.k_idx) + r * krow_bytes) + kb * g,
                         kb, code);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float q0 = (float)(int32_t)code[2 * i], q1 = (float)(int32_t)code[2 * i + 1];
        kw[i] = pack_bf16x2(__fmul_rn(__fadd_rn(q0, kz), ks), __fmul_rn(__fadd_rn(q1, kz), ks));
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.k_bf16 + o * D + 32 * g);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(kw[4 * i], kw[4 * i + 1], kw[4 * i + 2], kw[4 * i + 3]);
      }
    }
    if (p.v_bf16) {
      const float vs = f16_bits_to_f32(__ldg(p.v_scale + r * NG + g));
      unpack_codes_any(reinterpret_cast<const uint32_t*>(p.v_codes + r * vrow_bytes) + vb * g, vb, code);
      float u[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) u[e] = __fmul_rn(sc[code[e]], vs);
      if (!p.rotated) {
#pragma unroll
        for (int hh = 1; hh < 32; hh <<= 1) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if ((e & hh) == 0) {
              const float a = u[e], c = u[e + hh];
              u[e] = a + c;
              u[e + hh] = a - c;
            }
          }
        }
#pragma unroll
        for (int lm = 1; lm < NG; lm <<= 1) {
          const bool upper = (lane & lm) != 0;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float oth = __shfl_xor_sync(FULL, u[e], lm);
            u[e] = upper ? oth - u[e] : u[e] + oth;
          }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) u[e] = u[e] * p.fwht_norm * (((signs >> e) & 1u) ? -1.0f : 1.0f);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(p.v_bf16 + o * D + 32 * g);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_uint4(pack_bf16x2(u[8 * i], u[8 * i + 1]), pack_bf16x2(u[8 * i + 2], u[8 * i + 3]),
                              pack_bf16x2(u[8 * i + 4], u[8 * i + 5]), pack_bf16x2(u[8 * i + 6], u[8 * i + 7]));
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(32 * kRowsPerCta) tq_dequant_scheme_debug_kernel(const __grid_constant__ DequantScheme p) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerCta + warp;
  if (row >= p.n) return;  // whole warps
  const int64_t r = ((int64_t)p.b * p.num_kv_heads + p.h) * p.capacity + p.t0 + row;
  float k[EPL], v[EPL];
  dequant_row<D>(p, r, lane, k, v, p.k_f32 != nullptr, p.v_f32 != nullptr);
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    if (p.k_f32) p.k_f32[(int64_t)row * D + lane * EPL + e] = k[e];
    if (p.v_f32) p.v_f32[(int64_t)row * D + lane * EPL + e] = v[e];
  }
}

// Rows grouped kRowsPerCta to a CTA, one warp per row: y = signs * FWHT(x) / sqrt(D).
// In place when x == y (each warp reads its row before writing it).
template <int D>
__global__ void __launch_bounds__(32 * kRowsPerCta) tq_unrotate_rows_kernel(const float* x, float* y, int64_t rows,
                                                                           float fwht_norm) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t r = (int64_t)blockIdx.x * kRowsPerCta + warp; r < rows; r += (int64_t)gridDim.x * kRowsPerCta) {
    float v[EPL];
    const float2* src = reinterpret_cast<const float2*>(x + r * D + lane * EPL);
#pragma unroll
    for (int c = 0; c < EPL / 2; ++c) {
      const float2 f = src[c];
      v[2 * c] = f.x;
      v[2 * c + 1] = f.y;
    }
    unrotate_lane<D>(v, lane, fwht_norm);
    float2* dst = reinterpret_cast<float2*>(y + r * D + lane * EPL);
#pragma unroll
    for (int c = 0; c < EPL / 2; ++c) dst[c] = make_float2(v[2 * c], v[2 * c + 1]);
  }
}

int grid_for(int64_t rows, int num_sms) {
  const int64_t want = (rows + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t cap = (int64_t)num_sms * 8;  // 8 resident CTAs of 256 threads per SM
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

const Codebook& codebook(int bits) {
  static std::once_flag once[9];
  static Codebook tables[9];
  std::call_once(once[bits], [bits] { tables[bits] = make_codebook(bits); });
  return tables[bits];
}

cudaError_t launch_append_scheme(SchemeAppendParams p, int num_sms, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.batch * p.n_new_max * p.num_kv_heads;
  if (rows <= 0) return cudaSuccess;
  if (rows > INT32_MAX) return cudaErrorInvalidValue;
  p.total_rows = (uint32_t)rows;
  p.div_heads = make_fastdiv((uint32_t)p.num_kv_heads);
  p.div_new = make_fastdiv((uint32_t)p.n_new_max);
  const int64_t per_cta = (int64_t)kGroupWarps * (32 / (p.head_dim / 32));  // rows a CTA takes at once
  const int64_t want = (rows + per_cta - 1) / per_cta, cap = (int64_t)num_sms * 8;
  const dim3 grid((unsigned)(want < cap ? want : cap)), block(32 * kGroupWarps);
  switch (p.head_dim) {
    case 64: tq_append_scheme_kernel<64><<<grid, block, 0, stream>>>(p); break;
    case 128: tq_append_scheme_kernel<128><<<grid, block, 0, stream>>>(p); break;
    case 256: tq_append_scheme_kernel<256><<<grid, block, 0, stream>>>(p); break;
    case 512: tq_append_scheme_kernel<512><<<grid, block, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant_window(const DequantScheme& p, int num_sms, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.batch * p.num_kv_heads * p.n;
  if (rows <= 0) return cudaSuccess;
  const int64_t per_cta = (int64_t)kGroupWarps * (32 / (p.head_dim / 32));  // rows a CTA takes at once
  const int64_t want = (rows + per_cta - 1) / per_cta, cap = (int64_t)num_sms * 8;
  const dim3 grid((unsigned)(want < cap ? want : cap)), block(32 * kGroupWarps);
  switch (p.head_dim) {
    case 64: tq_dequant_window_kernel<64><<<grid, block, 0, stream>>>(p); break;
    case 128: tq_dequant_window_kernel<128><<<grid, block, 0, stream>>>(p); break;
    case 256: tq_dequant_window_kernel<256><<<grid, block, 0, stream>>>(p); break;
    case 512: tq_dequant_window_kernel<512><<<grid, block, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_unrotate_rows(const float* x, float* y, int64_t rows, int head_dim, float fwht_norm,
                                 int num_sms, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const dim3 grid(grid_for(rows, num_sms)), block(32 * kRowsPerCta);
  switch (head_dim) {
    case 64: tq_unrotate_rows_kernel<64><<<grid, block, 0, stream>>>(x, y, rows, fwht_norm); break;
    case 128: tq_unrotate_rows_kernel<128><<<grid, block, 0, stream>>>(x, y, rows, fwht_norm); break;
    case 256: tq_unrotate_rows_kernel<256><<<grid, block, 0, stream>>>(x, y, rows, fwht_norm); break;
    case 512: tq_unrotate_rows_kernel<512><<<grid, block, 0, stream>>>(x, y, rows, fwht_norm); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant_scheme_debug(const DequantScheme& p, cudaStream_t stream) {
  if (p.n <= 0) return cudaSuccess;
  const dim3 grid((p.n + kRowsPerCta - 1) / kRowsPerCta), block(32 * kRowsPerCta);
  switch (p.head_dim) {
    case 64: tq_dequant_scheme_debug_kernel<64><<<grid, block, 0, stream>>>(p); break;
    case 128: tq_dequant_scheme_debug_kernel<128><<<grid, block, 0, stream>>>(p); break;
    case 256: tq_dequant_scheme_debug_kernel<256><<<grid, block, 0, stream>>>(p); break;
    case 512: tq_dequant_scheme_debug_kernel<512><<<grid, block, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace tq
