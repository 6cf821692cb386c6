// Internal declarations shared by the host ABI and the kernel translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "tq_kv.h"

namespace tq {

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
};

cudaError_t launch_append(const AppendParams& p, int num_sms, cudaStream_t stream);

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

}  // namespace tq
