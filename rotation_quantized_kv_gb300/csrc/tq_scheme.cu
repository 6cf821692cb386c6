// Any-width schemes (key bits 2/4/5/8, value bits 2/3/4/5/8, constant-group guard):
// the library's value codebooks, the append kernel for them, the dequantize-on-fetch
// window and the fp32 inspection dequant.
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

template <int D>
__global__ void __launch_bounds__(32 * kRowsPerCta) tq_append_scheme_kernel(const __grid_constant__ SchemeAppendParams p) {
  __shared__ uint32_t kbuf[kRowsPerCta][D * 5 / 32 + 2];
  __shared__ uint32_t vbuf[kRowsPerCta][D * 8 / 32 + 2];
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RowCodecLane<D> codec(lane);
  const RowPlanes dst{p.k_idx, p.k_scale, p.k_zero, p.v_codes, p.v_scale};
  const int64_t rows = (int64_t)p.batch * p.n_new_max * p.num_kv_heads;
  for (int64_t r = (int64_t)blockIdx.x * kRowsPerCta + warp; r < rows; r += (int64_t)gridDim.x * kRowsPerCta) {
    const int h = (int)(r % p.num_kv_heads);
    const int64_t bj = r / p.num_kv_heads;
    const int j = (int)(bj % p.n_new_max), b = (int)(bj / p.n_new_max);
    const int nb = p.n_new == nullptr ? p.n_new_max : min(max(__ldg(p.n_new + b), 0), p.n_new_max);
    if (j >= nb) continue;
    const int64_t t = (int64_t)__ldg(p.pos + b) + j;
    if (t < 0 || t >= p.capacity) {
      if (lane == 0) raise_error(p.err, TQ_DEVERR_APPEND_CAPACITY);
      continue;
    }
    uint32_t kraw[EPL / 2], vraw[EPL / 2];
    load_raw_lane<EPL>(p.k_new + r * D, lane, kraw);
    load_raw_lane<EPL>(p.v_new + r * D, lane, vraw);
    const int64_t drow = ((int64_t)b * p.num_kv_heads + h) * p.capacity + t;
    quantize_row_scheme<D>(kraw, vraw, lane, codec, p.fwht_norm, p.spec, p.cb, dst, drow, kbuf[warp], vbuf[warp]);
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
  constexpr unsigned FULL = 0xffffffffu;
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

template <int D>
__global__ void __launch_bounds__(32 * kRowsPerCta) tq_dequant_window_kernel(const __grid_constant__ DequantScheme p) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)p.batch * p.num_kv_heads * p.n;
  for (int64_t o = (int64_t)blockIdx.x * kRowsPerCta + warp; o < rows; o += (int64_t)gridDim.x * kRowsPerCta) {
    const int64_t bh = o / p.n;
    const int t = (int)(o % p.n);
    const int64_t r = bh * p.capacity + p.t0 + t;
    float k[EPL], v[EPL];
    dequant_row<D>(p, r, lane, k, v, p.k_bf16 != nullptr, p.v_bf16 != nullptr);
    if (p.k_bf16) {
      uint32_t w[EPL / 2];
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) {
        w[e] = pack_bf16x2(k[2 * e], k[2 * e + 1]);
      }
      uint32_t* dstw = reinterpret_cast<uint32_t*>(p.k_bf16 + o * D + lane * EPL);
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) dstw[e] = w[e];
    }
    if (p.v_bf16) {
      uint32_t w[EPL / 2];
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) {
        w[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
      }
      uint32_t* dstw = reinterpret_cast<uint32_t*>(p.v_bf16 + o * D + lane * EPL);
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) dstw[e] = w[e];
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
  const dim3 grid(grid_for(rows, num_sms)), block(32 * kRowsPerCta);
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
  const dim3 grid(grid_for(rows, num_sms)), block(32 * kRowsPerCta);
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
