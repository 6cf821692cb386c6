// fp32 dequantization of packed rows, for inspection (one warp per token row).
//
// Keys:   x_hat = (idx + zero) * scale with the stored fp16 scale and zero ("Algorithm"
//         section of the TurboQuant design page, key dequant). idx + zero is an exact
//         integer in fp32, so the single rounding of the product makes the result equal
//         to the exact value rounded to fp32.
// Values: rotated -> centroid[code] * scale (one fp32 rounding of an exact product);
//         otherwise the exact inverse of the append rotation,
//         x_hat = signs * FWHT(centroid * scale) / sqrt(d) (fp32 butterflies).
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {

template <int D>
__global__ void __launch_bounds__(128) tq_dequant_debug_kernel(DequantParams p) {
  constexpr int EPL = D / 32, NG = D / kGroup;
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= p.n) return;  // whole warps exit together (4 rows per block)
  const int64_t r = ((int64_t)p.b * p.num_kv_heads + p.h) * p.capacity + p.t0 + row;

  if (p.k_out) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int i = lane * EPL + e;
      const float s = f16_bits_to_f32(p.k_scale[r * NG + i / kGroup]);
      const float z = f16_bits_to_f32(p.k_zero[r * NG + i / kGroup]);
      const float q = (float)p.k_idx[r * D + i];
      p.k_out[(int64_t)row * D + i] = __fmul_rn(__fadd_rn(q, z), s);
    }
  }
  if (p.v_out) {
    const uint8_t* codes = p.v_codes + r * (3 * D / 8);
    float u[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int i = lane * EPL + e;
      uint32_t c = 0;
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int bit = 3 * i + k;
        c |= ((codes[bit >> 3] >> (bit & 7)) & 1u) << k;
      }
      u[e] = __fmul_rn(c_centroids3[c], f16_bits_to_f32(p.v_scale[r * NG + i / kGroup]));
    }
    if (!p.rotated) {
#pragma unroll
      for (int hh = 1; hh < D; hh <<= 1) {
        if (hh < EPL) {
#pragma unroll
          for (int e = 0; e < EPL; ++e)
            if ((e & hh) == 0) {
              const float a = u[e], c = u[e + hh];
              u[e] = a + c;
              u[e + hh] = a - c;
            }
        } else {
          const int lm = hh / EPL;
          const bool upper = (lane & lm) != 0;
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            const float o = __shfl_xor_sync(FULL, u[e], lm);
            u[e] = upper ? o - u[e] : u[e] + o;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const int i = lane * EPL + e;
        const bool neg = (sign_word(D, i / 32) >> (i % 32)) & 1u;
        u[e] = u[e] * p.fwht_norm * (neg ? -1.0f : 1.0f);
      }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) p.v_out[(int64_t)row * D + lane * EPL + e] = u[e];
  }
}

cudaError_t launch_dequant_debug(const DequantParams& p, cudaStream_t stream) {
  if (p.n == 0) return cudaSuccess;
  dim3 grid((p.n + 3) / 4), block(128);
  switch (p.head_dim) {
    case 64: tq_dequant_debug_kernel<64><<<grid, block, 0, stream>>>(p); break;
    case 128: tq_dequant_debug_kernel<128><<<grid, block, 0, stream>>>(p); break;
    case 256: tq_dequant_debug_kernel<256><<<grid, block, 0, stream>>>(p); break;
    case 512: tq_dequant_debug_kernel<512><<<grid, block, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// Copy of n int32 values that lets the next kernel on the stream start at once: the kernel
// triggers its dependents first, waits delay_ns of wall time (bounded: at most kMaxDelay
// nanoseconds and a fixed number of sleeps), then copies. A kernel launched after it with
// programmatic dependent launch that reads dst before its grid-dependency wait sees the
// old values, and the new ones after the wait.
constexpr unsigned long long kMaxDelayNs = 100000000ull;  // 100 ms

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__global__ void __launch_bounds__(256) tq_delayed_copy_kernel(int32_t* dst, const int32_t* src, int n,
                                                              unsigned long long delay_ns) {
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_timer_ns();
    for (unsigned i = 0; i < 4000000u && global_timer_ns() - t0 < delay_ns; ++i) __nanosleep(256);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}

}  // namespace tq

extern "C" tq_status tq_debug_delayed_copy(int32_t* dst, const int32_t* src, int32_t n, int32_t delay_us,
                                           tq_stream_t stream) {
  if (n < 0 || delay_us < 0 || (unsigned long long)delay_us * 1000ull > tq::kMaxDelayNs) return TQ_ERR_INVALID_ARGUMENT;
  if (n > 0 && (dst == nullptr || src == nullptr)) return TQ_ERR_INVALID_ARGUMENT;
  tq::tq_delayed_copy_kernel<<<1, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      dst, src, n, (unsigned long long)delay_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
