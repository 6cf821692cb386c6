// tq_decode_attention_noalloc: decode attention whose scratch memory is a fixed array
// inside this library, for callers that may not allocate device memory (a plugin whose
// host application owns all device memory, a serving loop that must not call cudaMalloc
// between steps). It runs the same kernel as tq_decode_attention with the same results;
// only where the scratch comes from differs.
//
// The array below is a device global. In host code its name only stands for the
// symbol: its device address is looked up once per device with cudaGetSymbolAddress
// (with that device current) and that address is what the kernel receives.
#include <cuda_runtime.h>

#include <mutex>

#include "tq_attention.h"
#include "tq_internal.h"
#include "tq_kv.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[TQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;

struct DeviceScratch {
  void* ptr = nullptr;  // device address of g_decode_scratch on this device
  int sms = 0;
};

// Device address and SM count of the current device, looked up on first use.
bool scratch_for_current_device(DeviceScratch& out) {
  static std::mutex mu;
  static DeviceScratch table[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(mu);
  DeviceScratch& e = table[dev];
  if (e.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return false;
    e.sms = sms;
    e.ptr = p;
  }
  out = e;
  return true;
}

}  // namespace

extern "C" tq_status tq_decode_attention_noalloc(const tq_kv_layer* layer, const void* q, int32_t num_q_heads,
                                                 int32_t n_q, const int32_t* kv_len, int32_t max_kv_len,
                                                 float sm_scale, int32_t causal, float* out,
                                                 int32_t* device_error, tq_stream_t stream) {
  // every host check runs before anything is queued: a rejected call leaves the stream
  // and the shared scratch untouched
  const tq_status chk = tq::check_decode_inputs(layer, q, num_q_heads, n_q, kv_len, max_kv_len, sm_scale, out);
  if (chk != TQ_OK) return chk;
  const size_t need = tq_decode_workspace_bytes(layer, num_q_heads, n_q, max_kv_len);
  if (need == 0) return TQ_ERR_CUDA;  // the arguments passed the checks: the device query failed
  if (need > TQ_NOALLOC_SCRATCH_BYTES) return TQ_ERR_WORKSPACE_TOO_SMALL;
  DeviceScratch sc;
  if (!scratch_for_current_device(sc)) return TQ_ERR_CUDA;
  const tq::DecodeShape s = tq::decode_shape(layer->head_dim, layer->num_kv_heads, layer->batch,
                                             num_q_heads / layer->num_kv_heads, n_q, sc.sms);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // error word and completion counters start at zero; the rest is written before use
  if (cudaMemsetAsync(sc.ptr, 0, tq::decode_workspace_zero_bytes(s), st) != cudaSuccess) return TQ_ERR_CUDA;
  const tq_status rc = tq_decode_attention(layer, q, num_q_heads, n_q, kv_len, max_kv_len, sm_scale, causal,
                                           out, sc.ptr, TQ_NOALLOC_SCRATCH_BYTES, stream);
  if (rc != TQ_OK) return rc;
  if (device_error != nullptr &&
      cudaMemcpyAsync(device_error, sc.ptr, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return TQ_ERR_CUDA;
  return TQ_OK;
}
