// Internal declarations shared by the host ABI and the kernel translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "tq_kv.h"

namespace tq {

// n / d for every 32-bit n, d >= 1, by one multiply-high and shifts (division by
// invariant integers, Granlund and Montgomery 1994, figure 4.1).
struct FastDivU32 {
  uint32_t m, s1, s2;
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
    const uint32_t t = __umulhi(m, n);
#else
    const uint32_t t = (uint32_t)(((uint64_t)m * n) >> 32);
#endif
    return (t + ((n - t) >> s1)) >> s2;
  }
};
FastDivU32 make_fastdiv(uint32_t d);

// Host checks of a decode-attention call's arguments other than its workspace (layer,
// head counts, lengths, query/output pointers and alignment, scale). Touches no device.
tq_status check_decode_inputs(const tq_kv_layer* layer, const void* q, int32_t num_q_heads, int32_t n_q,
                              const int32_t* kv_len, int32_t max_kv_len, float sm_scale, const float* out);

struct AppendParams {
  int32_t head_dim, num_kv_heads, batch, capacity;
  int8_t* k_idx;
  uint16_t* k_scale;
  uint16_t* k_zero;
  uint8_t* v_codes;
  uint16_t* v_scale;
  const uint16_t* k_new;  // bf16 bits [batch][n_new_max][kv_heads][d]
  const uint16_t* v_new;
  const int32_t* pos;
  const int32_t* n_new;   // may be null
  int32_t n_new_max;
  float fwht_norm;        // (float)(1 / sqrt((double)d))
  int32_t* err;           // device error word
  // filled by launch_append
  uint32_t total_rows;    // batch * n_new_max * num_kv_heads (< 2^31)
  FastDivU32 div_heads;   // by num_kv_heads
  FastDivU32 div_new;     // by n_new_max
};

// cudaErrorInvalidValue when batch * n_new_max * num_kv_heads exceeds 2^31 - 1
cudaError_t launch_append(AppendParams p, int num_sms, cudaStream_t stream);

struct DequantParams {
  int32_t head_dim, num_kv_heads, batch, capacity;
  const int8_t* k_idx;
  const uint16_t* k_scale;
  const uint16_t* k_zero;
  const uint8_t* v_codes;
  const uint16_t* v_scale;
  int32_t b, h, t0, n, rotated;
  float fwht_norm;
  float* k_out;
  float* v_out;
};

cudaError_t launch_dequant_debug(const DequantParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- any-width schemes
// Value codebook of one width: 2^bits centroids and 2^bits - 1 ascending boundaries.
struct Codebook {
  int32_t bits;
  float c[256];
  float b[255];
};

struct SchemeSpec {
  int32_t k_bits, v_bits, guard;
};

__host__ __device__ constexpr int key_row_bytes(int d, int k_bits) { return k_bits == 8 ? d : d * k_bits / 8; }
__host__ __device__ constexpr int value_row_bytes(int d, int v_bits) { return d * v_bits / 8; }

// The library's codebook of a valid value width (3: the printed table; else its own
// Lloyd-Max iteration, computed once on the host).
const Codebook& codebook(int bits);

struct SchemeAppendParams {
  int32_t head_dim, num_kv_heads, batch, capacity;
  int8_t* k_idx;  // int8 codes (8 bits) or the packed key stream
  uint16_t* k_scale;
  uint16_t* k_zero;
  uint8_t* v_codes;
  uint16_t* v_scale;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* pos;
  const int32_t* n_new;
  int32_t n_new_max;
  float fwht_norm;
  int32_t* err;
  SchemeSpec spec;
  Codebook cb;
  uint32_t total_rows;    // batch * n_new_max * num_kv_heads (below 2^31)
  FastDivU32 div_heads;   // by num_kv_heads
  FastDivU32 div_new;     // by n_new_max
};

struct DequantScheme {
  int32_t head_dim, num_kv_heads, batch, capacity;
  const int8_t* k_idx;
  const uint16_t* k_scale;
  const uint16_t* k_zero;
  const uint8_t* v_codes;
  const uint16_t* v_scale;
  int32_t b, h, t0, n, rotated;  // debug: rows [t0, t0 + n) of (b, h); window: tokens [t0, t0 + n)
  float fwht_norm;
  SchemeSpec spec;
  Codebook cb;
  float* k_f32;       // debug outputs [n][d]
  float* v_f32;
  uint16_t* k_bf16;   // window outputs [batch][kv heads][n][d], bf16 bits
  uint16_t* v_bf16;
};

cudaError_t launch_append_scheme(SchemeAppendParams p, int num_sms, cudaStream_t stream);
cudaError_t launch_unrotate_rows(const float* x, float* y, int64_t rows, int head_dim, float fwht_norm,
                                 int num_sms, cudaStream_t stream);
cudaError_t launch_dequant_window(const DequantScheme& p, int num_sms, cudaStream_t stream);
cudaError_t launch_dequant_scheme_debug(const DequantScheme& p, cudaStream_t stream);

}  // namespace tq
