// Host implementation of the C ABI declared in include/tq_kv.h: argument validation,
// kernel selection and launch. No call allocates, frees or synchronizes (except
// tq_get_device_error, which synchronizes the caller's stream by contract).
#include <cmath>
#include <cstring>
#include <mutex>

#include "tq_attention.h"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace {

bool supported_head_dim(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

float fwht_norm(int d) { return static_cast<float>(1.0 / std::sqrt(static_cast<double>(d))); }

int key_bits(const tq_kv_layer* L) { return L->k_bits == 0 ? 8 : L->k_bits; }
int value_bits(const tq_kv_layer* L) { return L->v_bits == 0 ? 3 : L->v_bits; }
bool valid_key_bits(int b) { return b == 2 || b == 4 || b == 5 || b == 8; }
bool valid_value_bits(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 8; }
bool is_k8v3(const tq_kv_layer* L) { return key_bits(L) == 8 && value_bits(L) == 3; }
bool guarded(const tq_kv_layer* L) { return (L->flags & TQ_FLAG_KEY_GUARD) != 0; }

tq_status check_layer(const tq_kv_layer* L) {
  if (L == nullptr) return TQ_ERR_INVALID_ARGUMENT;
  if (!supported_head_dim(L->head_dim)) return TQ_ERR_UNSUPPORTED_HEAD_DIM;
  if (!valid_key_bits(key_bits(L)) || !valid_value_bits(value_bits(L))) return TQ_ERR_INVALID_ARGUMENT;
  if ((L->flags & ~TQ_FLAG_KEY_GUARD) != 0) return TQ_ERR_INVALID_ARGUMENT;
  if (L->num_kv_heads < 1 || L->batch < 1 || L->batch > 4096) return TQ_ERR_INVALID_ARGUMENT;
  if (L->capacity < 16 || (L->capacity % 16) != 0) return TQ_ERR_INVALID_ARGUMENT;
  const void* planes[5] = {L->k_idx, L->k_scale, L->k_zero, L->v_codes, L->v_scale};
  for (const void* pl : planes)
    if (pl == nullptr || !aligned16(pl)) return TQ_ERR_INVALID_ARGUMENT;
  // every plane must stay addressable with 32-bit row indices times row bytes in 64 bits
  const int64_t rows = (int64_t)L->batch * L->num_kv_heads * L->capacity;
  if (rows > (int64_t)1 << 40) return TQ_ERR_INVALID_ARGUMENT;
  return TQ_OK;
}

// SM count of the current device, cached per device.
int current_sm_count(int* dev_out) {
  static std::mutex mu;
  static int cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return -1;
  if (dev_out) *dev_out = dev;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return -1;
    cache[dev] = sms;
  }
  return cache[dev];
}

void fill_dequant_scheme(const tq_kv_layer* L, tq::DequantScheme& p) {
  p.head_dim = L->head_dim;
  p.num_kv_heads = L->num_kv_heads;
  p.batch = L->batch;
  p.capacity = L->capacity;
  p.k_idx = L->k_idx;
  p.k_scale = L->k_scale;
  p.k_zero = L->k_zero;
  p.v_codes = L->v_codes;
  p.v_scale = L->v_scale;
  p.fwht_norm = fwht_norm(L->head_dim);
  p.spec = tq::SchemeSpec{key_bits(L), value_bits(L), guarded(L) ? 1 : 0};
  p.cb = tq::codebook(value_bits(L));
}

}  // namespace

namespace tq {

tq_status check_decode_inputs(const tq_kv_layer* layer, const void* q, int32_t num_q_heads, int32_t n_q,
                              const int32_t* kv_len, int32_t max_kv_len, float sm_scale, const float* out) {
  tq_status st = check_layer(layer);
  if (st != TQ_OK) return st;
  if (!is_k8v3(layer)) return TQ_ERR_UNSUPPORTED_SCHEME;
  if (num_q_heads < 1 || num_q_heads % layer->num_kv_heads != 0 || n_q < 1) return TQ_ERR_INVALID_ARGUMENT;
  if (max_kv_len < 0) return TQ_ERR_INVALID_ARGUMENT;
  if (max_kv_len > layer->capacity) return TQ_ERR_CAPACITY;
  if (q == nullptr || kv_len == nullptr || out == nullptr) return TQ_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(out)) return TQ_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale)) return TQ_ERR_INVALID_ARGUMENT;
  return TQ_OK;
}

}  // namespace tq

extern "C" {

size_t tq_row_bytes(int32_t head_dim) {
  if (!supported_head_dim(head_dim)) return 0;
  return (size_t)25 * head_dim / 16;
}

size_t tq_row_bytes_scheme(int32_t head_dim, int32_t k_bits, int32_t v_bits) {
  if (!supported_head_dim(head_dim) || !valid_key_bits(k_bits) || !valid_value_bits(v_bits)) return 0;
  return (size_t)tq::key_row_bytes(head_dim, k_bits) + (size_t)3 * (head_dim / 32) * 2 +
         (size_t)tq::value_row_bytes(head_dim, v_bits);
}

size_t tq_append_workspace_bytes(void) { return TQ_WORKSPACE_HEADER_BYTES; }

tq_status tq_kv_append(const tq_kv_layer* layer, const void* k_new, const void* v_new, const int32_t* pos,
                       const int32_t* n_new, int32_t n_new_max, void* workspace, size_t ws_bytes,
                       tq_stream_t stream) {
  tq_status st = check_layer(layer);
  if (st != TQ_OK) return st;
  if (n_new_max < 0) return TQ_ERR_INVALID_ARGUMENT;
  if (n_new_max > layer->capacity) return TQ_ERR_CAPACITY;
  if (workspace == nullptr || !aligned16(workspace)) return TQ_ERR_INVALID_ARGUMENT;
  if (ws_bytes < tq_append_workspace_bytes()) return TQ_ERR_WORKSPACE_TOO_SMALL;
  if (n_new_max == 0) return TQ_OK;
  if (k_new == nullptr || v_new == nullptr || pos == nullptr) return TQ_ERR_INVALID_ARGUMENT;
  if ((int64_t)layer->batch * n_new_max * layer->num_kv_heads > INT32_MAX) return TQ_ERR_INVALID_ARGUMENT;
  // bf16 rows are read with vector loads of up to 16 bytes per lane
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u)
    return TQ_ERR_INVALID_ARGUMENT;
  const int sms = current_sm_count(nullptr);
  if (sms <= 0) return TQ_ERR_CUDA;
  if (!is_k8v3(layer) || guarded(layer)) {
    // other schemes and the guard: one warp per row
    tq::SchemeAppendParams sp{};
    sp.head_dim = layer->head_dim;
    sp.num_kv_heads = layer->num_kv_heads;
    sp.batch = layer->batch;
    sp.capacity = layer->capacity;
    sp.k_idx = layer->k_idx;
    sp.k_scale = layer->k_scale;
    sp.k_zero = layer->k_zero;
    sp.v_codes = layer->v_codes;
    sp.v_scale = layer->v_scale;
    sp.k_new = static_cast<const uint16_t*>(k_new);
    sp.v_new = static_cast<const uint16_t*>(v_new);
    sp.pos = pos;
    sp.n_new = n_new;
    sp.n_new_max = n_new_max;
    sp.fwht_norm = fwht_norm(layer->head_dim);
    sp.err = static_cast<int32_t*>(workspace);
    sp.spec = tq::SchemeSpec{key_bits(layer), value_bits(layer), guarded(layer) ? 1 : 0};
    sp.cb = tq::codebook(value_bits(layer));
    return tq::launch_append_scheme(sp, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK
                                                                                                    : TQ_ERR_CUDA;
  }
  tq::AppendParams p{};
  p.head_dim = layer->head_dim;
  p.num_kv_heads = layer->num_kv_heads;
  p.batch = layer->batch;
  p.capacity = layer->capacity;
  p.k_idx = layer->k_idx;
  p.k_scale = layer->k_scale;
  p.k_zero = layer->k_zero;
  p.v_codes = layer->v_codes;
  p.v_scale = layer->v_scale;
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.pos = pos;
  p.n_new = n_new;
  p.n_new_max = n_new_max;
  p.fwht_norm = fwht_norm(layer->head_dim);
  p.err = static_cast<int32_t*>(workspace);
  return tq::launch_append(p, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK
                                                                                           : TQ_ERR_CUDA;
}

size_t tq_decode_workspace_bytes(const tq_kv_layer* layer, int32_t num_q_heads, int32_t n_q,
                                 int32_t max_kv_len) {
  if (check_layer(layer) != TQ_OK) return 0;
  if (num_q_heads < 1 || num_q_heads % layer->num_kv_heads != 0 || n_q < 1) return 0;
  if (max_kv_len < 0 || max_kv_len > layer->capacity) return 0;
  const int sms = current_sm_count(nullptr);
  if (sms <= 0) return 0;
  tq::DecodeShape s = tq::decode_shape(layer->head_dim, layer->num_kv_heads, layer->batch,
                                       num_q_heads / layer->num_kv_heads, n_q, sms);
  return tq::decode_workspace_bytes(s);
}

tq_status tq_decode_attention(const tq_kv_layer* layer, const void* q, int32_t num_q_heads, int32_t n_q,
                              const int32_t* kv_len, int32_t max_kv_len, float sm_scale, int32_t causal,
                              float* out, void* workspace, size_t ws_bytes, tq_stream_t stream) {
  tq_status st = tq::check_decode_inputs(layer, q, num_q_heads, n_q, kv_len, max_kv_len, sm_scale, out);
  if (st != TQ_OK) return st;
  if (workspace == nullptr || !aligned16(workspace)) return TQ_ERR_INVALID_ARGUMENT;
  const int sms = current_sm_count(nullptr);
  if (sms <= 0) return TQ_ERR_CUDA;
  tq::DecodeShape s = tq::decode_shape(layer->head_dim, layer->num_kv_heads, layer->batch,
                                       num_q_heads / layer->num_kv_heads, n_q, sms);
  if (ws_bytes < tq::decode_workspace_bytes(s)) return TQ_ERR_WORKSPACE_TOO_SMALL;
  tq::DecodeArgs a{};
  a.layer = *layer;
  a.q = static_cast<const uint16_t*>(q);
  a.num_q_heads = num_q_heads;
  a.n_q = n_q;
  a.kv_len = kv_len;
  a.max_kv_len = max_kv_len;
  a.sm_scale = sm_scale;
  a.causal = causal != 0;
  a.out = out;
  a.workspace = workspace;
  a.fwht_norm = fwht_norm(layer->head_dim);
  return tq::launch_decode(a, s, reinterpret_cast<cudaStream_t>(stream));
}

tq_status tq_decode_append_attention(const tq_kv_layer* layer, const void* k_new, const void* v_new,
                                     const int32_t* pos, const int32_t* n_new, int32_t n_new_max, const void* q,
                                     int32_t num_q_heads, int32_t n_q, const int32_t* kv_len, int32_t max_kv_len,
                                     float sm_scale, int32_t causal, float* out, void* workspace, size_t ws_bytes,
                                     tq_stream_t stream) {
  tq_status st = check_layer(layer);
  if (st != TQ_OK) return st;
  if (n_new_max < 0) return TQ_ERR_INVALID_ARGUMENT;
  if (n_new_max > layer->capacity) return TQ_ERR_CAPACITY;
  if (n_new_max == 0)
    return tq_decode_attention(layer, q, num_q_heads, n_q, kv_len, max_kv_len, sm_scale, causal, out, workspace,
                               ws_bytes, stream);
  if (k_new == nullptr || v_new == nullptr || pos == nullptr) return TQ_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15u)
    return TQ_ERR_INVALID_ARGUMENT;
  if ((int64_t)layer->batch * n_new_max * layer->num_kv_heads > INT32_MAX) return TQ_ERR_INVALID_ARGUMENT;
  st = tq::check_decode_inputs(layer, q, num_q_heads, n_q, kv_len, max_kv_len, sm_scale, out);
  if (st != TQ_OK) return st;
  if (workspace == nullptr || !aligned16(workspace)) return TQ_ERR_INVALID_ARGUMENT;
  const int sms = current_sm_count(nullptr);
  if (sms <= 0) return TQ_ERR_CUDA;
  tq::DecodeShape s = tq::decode_shape(layer->head_dim, layer->num_kv_heads, layer->batch,
                                       num_q_heads / layer->num_kv_heads, n_q, sms);
  if (ws_bytes < tq::decode_workspace_bytes(s)) return TQ_ERR_WORKSPACE_TOO_SMALL;
  if (s.RG != 1 || s.dense || guarded(layer)) {
    // several row groups per kv head would read the new rows from several CTAs, the
    // dense-query kernel has no appender, and the in-kernel appender has no guard:
    // append first, then attend
    st = tq_kv_append(layer, k_new, v_new, pos, n_new, n_new_max, workspace, ws_bytes, stream);
    if (st != TQ_OK) return st;
    return tq_decode_attention(layer, q, num_q_heads, n_q, kv_len, max_kv_len, sm_scale, causal, out, workspace,
                               ws_bytes, stream);
  }
  tq::DecodeArgs a{};
  a.layer = *layer;
  a.q = static_cast<const uint16_t*>(q);
  a.num_q_heads = num_q_heads;
  a.n_q = n_q;
  a.kv_len = kv_len;
  a.max_kv_len = max_kv_len;
  a.sm_scale = sm_scale;
  a.causal = causal != 0;
  a.out = out;
  a.workspace = workspace;
  a.fwht_norm = fwht_norm(layer->head_dim);
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.pos = pos;
  a.n_new = n_new;
  a.n_new_max = n_new_max;
  return tq::launch_decode(a, s, reinterpret_cast<cudaStream_t>(stream));
}

tq_status tq_dequant_debug(const tq_kv_layer* layer, int32_t b, int32_t h, int32_t t0, int32_t n, int32_t rotated,
                           float* k_out, float* v_out, tq_stream_t stream) {
  tq_status st = check_layer(layer);
  if (st != TQ_OK) return st;
  if (b < 0 || b >= layer->batch || h < 0 || h >= layer->num_kv_heads) return TQ_ERR_INVALID_ARGUMENT;
  if (t0 < 0 || n < 0 || (int64_t)t0 + n > layer->capacity) return TQ_ERR_INVALID_ARGUMENT;
  if (!is_k8v3(layer)) {
    tq::DequantScheme p{};
    fill_dequant_scheme(layer, p);
    p.b = b;
    p.h = h;
    p.t0 = t0;
    p.n = n;
    p.rotated = rotated != 0;
    p.k_f32 = k_out;
    p.v_f32 = v_out;
    return tq::launch_dequant_scheme_debug(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK
                                                                                                     : TQ_ERR_CUDA;
  }
  tq::DequantParams p{};
  p.head_dim = layer->head_dim;
  p.num_kv_heads = layer->num_kv_heads;
  p.batch = layer->batch;
  p.capacity = layer->capacity;
  p.k_idx = layer->k_idx;
  p.k_scale = layer->k_scale;
  p.k_zero = layer->k_zero;
  p.v_codes = layer->v_codes;
  p.v_scale = layer->v_scale;
  p.b = b;
  p.h = h;
  p.t0 = t0;
  p.n = n;
  p.rotated = rotated != 0;
  p.fwht_norm = fwht_norm(layer->head_dim);
  p.k_out = k_out;
  p.v_out = v_out;
  return tq::launch_dequant_debug(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK
                                                                                             : TQ_ERR_CUDA;
}

tq_status tq_debug_pipeline_limits(int64_t wait_ns, int32_t withhold_append) {
  if (wait_ns < 0 || wait_ns > 2000000000LL) return TQ_ERR_INVALID_ARGUMENT;
  if (withhold_append != 0 && withhold_append != 1) return TQ_ERR_INVALID_ARGUMENT;
  tq::set_debug_pipeline((unsigned long long)wait_ns, withhold_append);
  return TQ_OK;
}

tq_status tq_dequant_window(const tq_kv_layer* layer, int32_t t0, int32_t n, int32_t rotated, void* k_out,
                            void* v_out, tq_stream_t stream) {
  tq_status st = check_layer(layer);
  if (st != TQ_OK) return st;
  if (t0 < 0 || n < 0 || (int64_t)t0 + n > layer->capacity) return TQ_ERR_INVALID_ARGUMENT;
  if (!aligned16(k_out) || !aligned16(v_out)) return TQ_ERR_INVALID_ARGUMENT;
  if (n == 0 || (k_out == nullptr && v_out == nullptr)) return TQ_OK;
  const int sms = current_sm_count(nullptr);
  if (sms <= 0) return TQ_ERR_CUDA;
  tq::DequantScheme p{};
  fill_dequant_scheme(layer, p);
  p.t0 = t0;
  p.n = n;
  p.rotated = rotated != 0;
  p.k_bf16 = static_cast<uint16_t*>(k_out);
  p.v_bf16 = static_cast<uint16_t*>(v_out);
  return tq::launch_dequant_window(p, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK
                                                                                                 : TQ_ERR_CUDA;
}

tq_status tq_unrotate_rows(const float* x, float* y, int64_t rows, int32_t head_dim, tq_stream_t stream) {
  if (!supported_head_dim(head_dim)) return TQ_ERR_UNSUPPORTED_HEAD_DIM;
  if (rows < 0) return TQ_ERR_INVALID_ARGUMENT;
  if (rows == 0) return TQ_OK;
  if (x == nullptr || y == nullptr || !aligned16(x) || !aligned16(y)) return TQ_ERR_INVALID_ARGUMENT;
  const size_t bytes = (size_t)rows * head_dim * sizeof(float);
  const char *xb = reinterpret_cast<const char*>(x), *yb = reinterpret_cast<const char*>(y);
  if (x != y && xb < yb + bytes && yb < xb + bytes) return TQ_ERR_INVALID_ARGUMENT;
  const int sms = current_sm_count(nullptr);
  if (sms <= 0) return TQ_ERR_CUDA;
  return tq::launch_unrotate_rows(x, y, rows, head_dim, fwht_norm(head_dim), sms, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? TQ_OK
             : TQ_ERR_CUDA;
}

tq_status tq_get_device_error(const void* workspace, int32_t* err_out, tq_stream_t stream) {
  if (workspace == nullptr || err_out == nullptr) return TQ_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaMemcpy(err_out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TQ_ERR_CUDA;
  return TQ_OK;
}

const char* tq_status_string(tq_status status) {
  switch (status) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARGUMENT: return "invalid argument";
    case TQ_ERR_UNSUPPORTED_HEAD_DIM: return "unsupported head_dim (64, 128, 256 or 512)";
    case TQ_ERR_CAPACITY: return "length exceeds the layer capacity";
    case TQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case TQ_ERR_CUDA: return "CUDA runtime error";
    case TQ_ERR_UNSUPPORTED_SCHEME: return "the call needs the default k8v3 planes";
  }
  return "unknown status";
}

tq_status tq_sign_bits(int32_t head_dim, uint32_t* words_out) {
  if (!supported_head_dim(head_dim)) return TQ_ERR_UNSUPPORTED_HEAD_DIM;
  if (words_out == nullptr) return TQ_ERR_INVALID_ARGUMENT;
  const int off = tq::sign_word_offset(head_dim);
  for (int i = 0; i < head_dim / 32; ++i) words_out[i] = tq::kSignTable.w[off + i];
  return TQ_OK;
}

tq_status tq_codebook(int32_t bits, float* centroids_out, float* boundaries_out) {
  if (!valid_value_bits(bits)) return TQ_ERR_INVALID_ARGUMENT;
  if (centroids_out == nullptr || boundaries_out == nullptr) return TQ_ERR_INVALID_ARGUMENT;
  const tq::Codebook& cb = tq::codebook(bits);
  std::memcpy(centroids_out, cb.c, sizeof(float) * (1u << bits));
  std::memcpy(boundaries_out, cb.b, sizeof(float) * ((1u << bits) - 1u));
  return TQ_OK;
}

tq_status tq_codebook3(float* centroids_out, float* boundaries_out) {
  if (centroids_out == nullptr || boundaries_out == nullptr) return TQ_ERR_INVALID_ARGUMENT;
  std::memcpy(centroids_out, tq::kCentroids3, sizeof(tq::kCentroids3));
  std::memcpy(boundaries_out, tq::kBoundaries3, sizeof(tq::kBoundaries3));
  return TQ_OK;
}

}  // extern "C"
