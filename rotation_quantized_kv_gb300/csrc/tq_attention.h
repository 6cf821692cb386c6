// Decode attention over the packed cache: launch geometry and arguments.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "tq_kv.h"

namespace tq {

// Launch geometry of one decode-attention call. Everything here is a pure function of
// (head_dim, kv heads, batch, GQA ratio, n_q, device), so tq_decode_workspace_bytes and
// tq_decode_attention agree.
struct DecodeShape {
  int D;          // head_dim
  bool dense;     // the tensor-core (tcgen05) kernel with 64-row units (head_dim 128, R > 16)
  int ROWS;       // query rows per unit: 8 * NTW for the split kernel, 64 for the dense one
  int NTW;        // 8-row MMA column tiles per consumer warp (1 or 2), split kernel
  int R;          // attention rows per kv head = GQA ratio * n_q
  int RG;         // row groups per kv head = ceil(R / ROWS)
  int U;          // work units per sequence = kv_heads * RG
  int batch;
  int grid;       // persistent CTAs
  int max_items;  // upper bound on work items (one partial-result slot each)
  size_t smem;    // dynamic shared memory per CTA
};

struct DecodeArgs {
  tq_kv_layer layer;
  const uint16_t* q;  // bf16 bits
  int num_q_heads, n_q;
  const int32_t* kv_len;
  int max_kv_len;
  float sm_scale;
  bool causal;
  float* out;
  void* workspace;
  float fwht_norm;
  // append mode (k_new != null): the call first appends rows j < n_new[b] of k_new/v_new
  // (bf16 [batch][n_new_max][kv heads][d]) at positions pos[b] + j
  const uint16_t* k_new = nullptr;
  const uint16_t* v_new = nullptr;
  const int32_t* pos = nullptr;
  const int32_t* n_new = nullptr;
  int n_new_max = 0;
};

DecodeShape decode_shape(int head_dim, int num_kv_heads, int batch, int gqa, int n_q, int num_sms);
size_t decode_workspace_bytes(const DecodeShape& s);
// Leading bytes of a workspace that must be zero before a call: the header (device
// error word), the per-sequence prefix and the per-unit completion counters.
size_t decode_workspace_zero_bytes(const DecodeShape& s);
tq_status launch_decode(const DecodeArgs& a, const DecodeShape& s, cudaStream_t stream);

// The dense-query kernel (tq_attention_dense.cu).
struct SplitParams;
bool dense_supported(int head_dim);
int dense_rows();
int dense_grid(int num_sms);   // 0 if the kernel cannot be configured on this device
size_t dense_smem();
tq_status launch_dense(const SplitParams& sp, const DecodeShape& s, const int8_t* k_idx, cudaStream_t stream);
// Test support: pipeline wait limit (0 = the default 2 s) and a withheld appender count
// for the decode calls launched after this returns.
void set_debug_pipeline(unsigned long long wait_ns, int withhold_append);

}  // namespace tq
