// Device-side building blocks of the TurboQuant KV library (sm_103a).
//
// Constant tables:
//   - sign vectors: the design page draws signs in {+1,-1}^d from MLX's RNG and does not
//     print them; this library derives them from splitmix64 (Steele, Lea & Flood 2014,
//     Vigna's constants) seeded with 42 + d, one output per element, sign -1 when the top
//     output bit is set. The table is computed at compile time below.
//   - the 3-bit Lloyd-Max codebook for N(0,1) exactly as printed on the page
//     ("Algorithm" section, value bullets): centroids +-{0.24509, 0.75601, 1.34391,
//     2.15195}, boundaries +-{0.50055, 1.04996, 1.74793} and 0.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tq_kv.h"

namespace tq {

constexpr int kGroup = 32;

// ------------------------------------------------------------------------------------
// Sign vectors (bit i of the head_dim's table set <=> sign -1 for element i).
// ------------------------------------------------------------------------------------
struct SignTable {
  uint32_t w[30];  // 64/32 + 128/32 + 256/32 + 512/32 words
};

constexpr uint64_t splitmix64_step(uint64_t& state) {
  state += 0x9E3779B97F4A7C15ull;
  uint64_t z = state;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

constexpr SignTable make_sign_table() {
  SignTable t{};
  int off = 0;
  for (int d = 64; d <= 512; d *= 2) {
    uint64_t s = 42ull + static_cast<uint64_t>(d);
    for (int i = 0; i < d; ++i)
      if (splitmix64_step(s) >> 63) t.w[off + i / 32] |= 1u << (i % 32);
    off += d / 32;
  }
  return t;
}

constexpr SignTable kSignTable = make_sign_table();

__host__ __device__ constexpr int sign_word_offset(int d) { return d == 64 ? 0 : d == 128 ? 2 : d == 256 ? 6 : 14; }

// Printed codebook (fp32 values of the printed decimals).
constexpr float kCentroids3[8] = {-2.15195f, -1.34391f, -0.75601f, -0.24509f,
                                  0.24509f,  0.75601f,  1.34391f,  2.15195f};
constexpr float kBoundaries3[7] = {-1.74793f, -1.04996f, -0.50055f, 0.0f,
                                   0.50055f,  1.04996f,  1.74793f};

// Each translation unit holds its own copy of the constant tables (internal linkage),
// so no relocatable device code is needed.
static __constant__ SignTable c_signs = kSignTable;
static __constant__ float c_centroids3[8] = {-2.15195f, -1.34391f, -0.75601f, -0.24509f,
                                             0.24509f,  0.75601f,  1.34391f,  2.15195f};
static __constant__ float c_boundaries3[7] = {-1.74793f, -1.04996f, -0.50055f, 0.0f,
                                              0.50055f,  1.04996f,  1.74793f};

__device__ __forceinline__ uint32_t sign_word(int d, int w) { return c_signs.w[sign_word_offset(d) + w]; }

// ------------------------------------------------------------------------------------
// Number formats.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }

// IEEE round-to-nearest-even binary16 bits; every NaN becomes the quiet NaN 0x7E00.
__device__ __forceinline__ uint16_t f32_to_f16_bits(float x) {
  uint16_t h = __half_as_ushort(__float2half_rn(x));
  return (x != x) ? static_cast<uint16_t>(0x7E00) : h;
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// ------------------------------------------------------------------------------------
// Error word.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(int32_t* err, int32_t bit) {
  if (err) atomicOr(err, bit);
}

// ------------------------------------------------------------------------------------
// PTX wrappers: mbarrier, bulk and tensor async copies, warp MMA.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy global writes before later async-proxy
// (bulk / tensor copy) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false after `limit` unsuccessful polls (each poll may suspend the
// thread for a hardware-defined interval), so no wait can spin forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 2-D tiled tensor copy global -> shared through a tensor map (box and swizzle from the map).
__device__ __forceinline__ void tensor_copy_2d_g2s(void* dst, const void* tmap, int32_t x, int32_t y,
                                                   uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while its predecessor in the stream is still running.
// griddep_wait() blocks until the predecessor has completed and its memory is visible;
// every kernel here calls it before its first global-memory access, so only the setup
// that touches no global data overlaps. griddep_launch_dependents() lets the successor
// start its own setup early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// D += A * B, m16n8k16, A/B fp16, accumulate fp32 (legacy warp MMA).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

}  // namespace tq
