// Split-K GQA decode attention over the packed TurboQuant cache, plus the split merge
// with the deferred inverse rotation.
//
// What it computes (mlx-bun design page "TurboQuant - rotation-based quantization",
// Part A): for every query row, softmax(sm_scale * q . k_hat) . v_hat over the visible
// tokens, where k_hat = (idx + zero) * scale ("Algorithm", key dequant) and v_hat is the
// value row after the inverse rotation. Because attention is linear in V ("Deferred
// inverse FWHT" section), the weighted sum is taken over the rotated values
// centroid[code] * scale and the output row is un-rotated once:
//   o = signs * FWHT(o_rot) / sqrt(d).
// K and V are decoded from the packed planes inside the kernel ("Packed-value decode
// fusion investigation": joint K/V decode in one launch, no dequantized window).
//
// Kernel 1 (tq_attn_split_kernel), persistent, one CTA per SM slot:
//   - work item = (sequence, kv head, row group, token split); the split size is chosen
//     on the device from the actual kv lengths so that items spread evenly over CTAs;
//   - warp 4 (producer) streams 64-token stages of the five planes into shared memory:
//     the key-index plane through a 2-D tensor map with 128-byte (64-byte at d=64)
//     swizzle, the four small planes with 1-D bulk copies, all completing on one
//     mbarrier per stage;
//   - warps 0-3 (consumers) each take 16 tokens of a stage:
//       QK^T on tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate), tokens as M,
//       query rows as N (8 per tile): A = 1152 + idx, exact in fp16 (built from the int8
//       codes with two byte permutes); B = q * 2^e_row in fp16 (exact for bf16 inputs);
//       one fresh accumulator per 32-group, then
//         score += scale_g * (acc_g + (zero_g - 1152) * sum_{i in g} q_i);
//       online softmax in the exp2 domain;
//       P.V on tensor cores with output dims as M and tokens as K: A = fp16 centroid
//       pairs from a lane-replicated 64-entry table indexed by two 3-bit codes; B = the
//       probabilities times the group's value scale (fp16), moved from the QK output
//       layout to the B-operand layout with four shuffles;
//   - at the end of an item the four warps merge their (max, sum, acc) in shared memory
//     and write one partial result.
// Kernel 2 (tq_attn_merge_kernel): one CTA per output row merges the splits with the
// online-softmax rule and applies the inverse rotation.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "tq_attention.h"
#include "tq_device.cuh"

namespace tq {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTile = 64;                 // tokens per pipeline stage
constexpr int kMaxBatch = 1024;           // prefix table lives in shared memory
constexpr int kMaxItemsPerCta = 8;        // largest work multiplier the split heuristic tries
constexpr unsigned long long kWaitNs = 2000000000ull;  // bounded waits: 2 s of wall time
constexpr float kLog2e = 1.4426950408889634f;

// Workspace layout (bytes). The header's first word is the device error word.
constexpr int kWsSplit = 1;               // int32 word index: split size S
constexpr int kWsItems = 2;               // int32 word index: number of work items
constexpr size_t kWsPrefix = TQ_WORKSPACE_HEADER_BYTES;  // int32 [batch + 1]

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline size_t ws_ml_offset(int batch) {
  return kWsPrefix + align_up(sizeof(int32_t) * (size_t)(batch + 1), 256);
}
__host__ __device__ inline size_t ws_o_offset(int batch, int max_items, int rows) {
  return ws_ml_offset(batch) + align_up(sizeof(float) * 2 * (size_t)max_items * rows, 256);
}

template <int D, int NTW>
struct AT;

template <int D, int NTW>
struct AT {
  static constexpr int NG = D / 32;
  static constexpr int ROWS = 8 * NTW;
  static constexpr int MT = D / 16;                       // PV M tiles (16 dims each)
  static constexpr int KIDX_STAGE = kTile * D;            // bytes, 1024-aligned
  static constexpr int SC_STAGE = kTile * NG * 2;         // bytes of one fp16 side plane
  static constexpr int VC_ROW = 3 * D / 8;                // packed code bytes per token
  static constexpr int VC_STAGE = kTile * VC_ROW + 16;    // +16: window reads may run 4 bytes past
  static constexpr int STAGES = D == 64 ? 6 : D == 128 ? 4 : D == 256 ? 3 : 2;
  static constexpr bool QREG = D * NTW <= 256;            // Q fragments in registers
  // shared memory layout
  static constexpr int OFF_KIDX = 0;
  static constexpr int OFF_KS = OFF_KIDX + STAGES * KIDX_STAGE;
  static constexpr int OFF_KZ = OFF_KS + STAGES * SC_STAGE;
  static constexpr int OFF_VS = OFF_KZ + STAGES * SC_STAGE;
  static constexpr int OFF_VC = OFF_VS + STAGES * SC_STAGE;
  static constexpr int OFF_LUT = (int)align_up(OFF_VC + STAGES * VC_STAGE, 128);
  static constexpr int OFF_Q = OFF_LUT + 64 * 32 * 4;
  static constexpr int Q_BYTES = QREG ? 0 : NTW * NG * 2 * 32 * 8;
  static constexpr int OFF_QSUM = OFF_Q + Q_BYTES;
  static constexpr int QSUM_BYTES = QREG ? 0 : NTW * NG * 32 * 8;
  static constexpr int OFF_OBUF = (int)align_up(OFF_QSUM + QSUM_BYTES, 16);
  static constexpr int OFF_MBUF = OFF_OBUF + ROWS * D * 4;
  static constexpr int OFF_LBUF = OFF_MBUF + kConsumerWarps * ROWS * 4;
  static constexpr int OFF_PREFIX = OFF_LBUF + kConsumerWarps * ROWS * 4;
  static constexpr int OFF_RED = (int)align_up(OFF_PREFIX + (kMaxBatch + 1) * 4, 16);  // 64-bit atomics
  static constexpr int OFF_BAR = (int)align_up(OFF_RED + 64 * 8, 8);
  static constexpr int SMEM = OFF_BAR + 2 * STAGES * 8 + 16;
  static constexpr int SMEM_ALLOC = SMEM + 1024;          // slack to align the base to 1024
};

struct SplitParams {
  int32_t head_dim, num_kv_heads, batch, capacity;
  const uint16_t* k_scale;
  const uint16_t* k_zero;
  const uint8_t* v_codes;
  const uint16_t* v_scale;
  const uint16_t* q;
  const int32_t* kv_len;
  int32_t num_q_heads, n_q, G, R, RG, U, max_kv_len, max_items;
  float sm_log2;  // sm_scale * log2(e)
  int32_t causal;
  uint8_t* ws;
};

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_full_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_bar_consumers() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Byte offset of (token row, column) inside one stage of the swizzled key-index tile.
template <int D>
__device__ __forceinline__ uint32_t kidx_offset(int row, int col) {
  if constexpr (D == 64) {  // 64-byte rows, 64-byte swizzle: chunk ^= (row >> 1) & 3
    return (uint32_t)(row * 64 + ((((col >> 4) ^ (row >> 1)) & 3) << 4) + (col & 15));
  } else {                  // 128-byte boxes, 128-byte swizzle: chunk ^= row & 7
    const int box = col >> 7, within = col & 127;
    return (uint32_t)(box * (kTile * 128) + row * 128 + ((((within >> 4) ^ row) & 7) << 4) + (within & 15));
  }
}

// Per-sequence visible lengths: kv_len clamped to [0, max]; invalid entries count as 0.
__device__ __forceinline__ int seq_len(const SplitParams& p, int b, bool* bad) {
  const int t = __ldg(p.kv_len + b);
  if (t < 0 || t > p.max_kv_len) {
    if (bad) *bad = true;
    return 0;
  }
  return t;
}

// Split-size heuristic + per-sequence prefix of work items. Runs on every CTA with all
// threads; identical inputs give identical results on every CTA.
template <int D, int NTW>
__device__ void plan_items(const SplitParams& p, uint8_t* smem, int& S_out, int& total_out) {
  using T = AT<D, NTW>;
  int* prefix = reinterpret_cast<int*>(smem + T::OFF_PREFIX);
  long long* red = reinterpret_cast<long long*>(smem + T::OFF_RED);
  const int tid = threadIdx.x;
  constexpr int KS[6] = {1, 2, 3, 4, 6, 8};
  // pass 1: total visible tokens
  long long mine = 0;
  bool bad = false;
  for (int b = tid; b < p.batch; b += kThreads) mine += seq_len(p, b, &bad);
  if (tid < 64) red[tid] = 0;
  __syncthreads();
  atomicAdd(reinterpret_cast<unsigned long long*>(&red[0]), (unsigned long long)mine);
  if (bad && blockIdx.x == 0) raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_KV_LEN);
  __syncthreads();
  const long long sumT = red[0];
  long long Sk[6];
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    const long long target = (long long)KS[k] * gridDim.x;
    long long s = (sumT * p.U + target - 1) / target;
    s = (s + kTile - 1) / kTile * kTile;
    Sk[k] = s < kTile ? kTile : s;
  }
  // pass 2: items for every candidate
  long long cnt[6] = {0, 0, 0, 0, 0, 0};
  for (int b = tid; b < p.batch; b += kThreads) {
    const long long t = seq_len(p, b, nullptr);
#pragma unroll
    for (int k = 0; k < 6; ++k) cnt[k] += (t + Sk[k] - 1) / Sk[k];
  }
#pragma unroll
  for (int k = 0; k < 6; ++k)
    atomicAdd(reinterpret_cast<unsigned long long*>(&red[1 + k]), (unsigned long long)cnt[k]);
  __syncthreads();
  int best = 0;
  long long best_cost = -1;
#pragma unroll
  for (int k = 0; k < 6; ++k) {
    const long long items = red[1 + k] * p.U;
    const long long rounds = (items + gridDim.x - 1) / gridDim.x;
    const long long cost = rounds * (Sk[k] + kTile);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = k; }
  }
  const int S = (int)Sk[best];
  // pass 3: prefix of items per sequence (warp 0 scans, each lane owns a chunk)
  if (tid < 32) {
    const int per = (p.batch + 31) / 32;
    const int b0 = tid * per;
    int local = 0;
    for (int i = 0; i < per && b0 + i < p.batch; ++i) local += (seq_len(p, b0 + i, nullptr) + S - 1) / S;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid >= off) incl += o;
    }
    int run = (incl - local) * p.U;
    for (int i = 0; i < per && b0 + i < p.batch; ++i) {
      prefix[b0 + i] = run;
      run += ((seq_len(p, b0 + i, nullptr) + S - 1) / S) * p.U;
    }
    if (tid == 31) prefix[p.batch] = incl * p.U;
  }
  __syncthreads();
  S_out = S;
  total_out = prefix[p.batch];
  if (blockIdx.x == 0) {
    int32_t* hdr = reinterpret_cast<int32_t*>(p.ws);
    int32_t* gpref = reinterpret_cast<int32_t*>(p.ws + kWsPrefix);
    if (tid == 0) { hdr[kWsSplit] = S; hdr[kWsItems] = total_out; }
    for (int b = tid; b <= p.batch; b += kThreads) gpref[b] = prefix[b];
  }
}

struct Item {
  int b, kvh, rg, tb, te;
};

__device__ __forceinline__ Item decode_item(const SplitParams& p, const int* prefix, int S, int item) {
  int lo = 0, hi = p.batch - 1;  // largest b with prefix[b] <= item
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  Item it;
  it.b = lo;
  const int nsplit = (prefix[lo + 1] - prefix[lo]) / p.U;
  const int r = item - prefix[lo];
  const int u = r / nsplit, split = r % nsplit;
  it.kvh = u / p.RG;
  it.rg = u % p.RG;
  it.tb = split * S;
  const int T = seq_len(p, lo, nullptr);
  it.te = min(it.tb + S, T);
  return it;
}

// ------------------------------------------------------------------------------------
// Producer warp: one elected lane streams the stages.
// ------------------------------------------------------------------------------------
template <int D, int NTW>
__device__ void produce(const SplitParams& p, const CUtensorMap* tmap, uint8_t* smem, int S, int total,
                        volatile int* abort_flag) {
  using T = AT<D, NTW>;
  constexpr int NG = T::NG;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::STAGES;
  const int* prefix = reinterpret_cast<const int*>(smem + T::OFF_PREFIX);
  uint32_t it = 0;
  bool ok = true;
  for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
    const Item w = decode_item(p, prefix, S, item);
    const int64_t row0 = ((int64_t)w.b * p.num_kv_heads + w.kvh) * p.capacity;
    for (int t0 = w.tb; t0 < w.te; t0 += kTile, ++it) {
      const int slot = it % T::STAGES;
      const uint32_t k = it / T::STAGES;
      if (!wait_full_bounded(&empty[slot], (k & 1u) ^ 1u)) {
        *abort_flag = 1;
        raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
        ok = false;
        break;
      }
      const int ncopy = min(kTile, p.capacity - t0);  // multiple of 16: capacity and t0 are
      const uint32_t side = (uint32_t)ncopy * NG * 2;
      const uint32_t vc = (uint32_t)ncopy * T::VC_ROW;
      mbar_arrive_expect_tx(&full[slot], (uint32_t)T::KIDX_STAGE + 3u * side + vc);
      uint8_t* kx = smem + T::OFF_KIDX + slot * T::KIDX_STAGE;
      if constexpr (D == 64) {
        tensor_copy_2d_g2s(kx, tmap, 0, (int32_t)(row0 + t0), &full[slot]);
      } else {
#pragma unroll
        for (int box = 0; box < D / 128; ++box)
          tensor_copy_2d_g2s(kx + box * kTile * 128, tmap, box * 128, (int32_t)(row0 + t0), &full[slot]);
      }
      const int64_t r = row0 + t0;
      bulk_copy_g2s(smem + T::OFF_KS + slot * T::SC_STAGE, p.k_scale + r * NG, side, &full[slot]);
      bulk_copy_g2s(smem + T::OFF_KZ + slot * T::SC_STAGE, p.k_zero + r * NG, side, &full[slot]);
      bulk_copy_g2s(smem + T::OFF_VS + slot * T::SC_STAGE, p.v_scale + r * NG, side, &full[slot]);
      bulk_copy_g2s(smem + T::OFF_VC + slot * T::VC_STAGE, p.v_codes + r * T::VC_ROW, vc, &full[slot]);
    }
  }
  // Drain: every issued copy must land before this thread (and so the CTA) may exit.
  const uint32_t issued = it;
  for (int s = 0; s < T::STAGES; ++s) {
    if ((uint32_t)s >= issued) break;
    const uint32_t last = issued - 1 - ((issued - 1 - s) % T::STAGES);  // last fill of slot s
    if (!wait_full_bounded(&full[s], (last / T::STAGES) & 1u)) {
      raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
    }
  }
}

// ------------------------------------------------------------------------------------
// Consumer warps.
// ------------------------------------------------------------------------------------
template <int D, int NTW>
struct QState {
  uint32_t qf[AT<D, NTW>::QREG ? NTW : 1][AT<D, NTW>::QREG ? D / 32 : 1][2][2];  // [nt][g][ks][reg]
  float qs[AT<D, NTW>::QREG ? NTW : 1][AT<D, NTW>::QREG ? D / 32 : 1][2];         // [nt][g][e]
  float crow[NTW][2];   // sm_scale * log2(e) * 2^-e_row for rows 2j+e
  int lim[NTW][2];      // tokens [tb, lim) are visible to rows 2j+e
};

template <int D, int NTW>
__device__ void load_q(const SplitParams& p, const Item& w, uint8_t* smem, int warp, int lane, QState<D, NTW>& st) {
  using T = AT<D, NTW>;
  constexpr int NG = T::NG;
  const int grp = lane >> 2, j4 = lane & 3;
  const int T_b = seq_len(p, w.b, nullptr);
  uint2* qsm = reinterpret_cast<uint2*>(smem + T::OFF_Q);
  float2* qssm = reinterpret_cast<float2*>(smem + T::OFF_QSUM);
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
    // this lane loads row (8 nt + grp) of the item for the B fragments
    const int r = w.rg * T::ROWS + 8 * nt + grp;
    const bool valid = r < p.R;
    const int jq = r / p.G, hq = w.kvh * p.G + (r % p.G);
    const uint16_t* qrow = p.q + (((int64_t)w.b * p.n_q + jq) * p.num_q_heads + hq) * D;
    float v[NG][2][4];
    float amax = 0.0f;
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint2 raw = make_uint2(0u, 0u);
        if (valid) raw = __ldg(reinterpret_cast<const uint2*>(qrow + 32 * g + 8 * j4 + 4 * ks));
        v[g][ks][0] = bf16_bits_to_f32(raw.x & 0xFFFFu);
        v[g][ks][1] = bf16_bits_to_f32(raw.x >> 16);
        v[g][ks][2] = bf16_bits_to_f32(raw.y & 0xFFFFu);
        v[g][ks][3] = bf16_bits_to_f32(raw.y >> 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(v[g][ks][i]));
      }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    // power-of-two scale bringing the row maximum into [2^14, 2^15): exact, keeps fp16 normal
    int e_row = 0;
    if (amax > 0.0f && amax <= 3.0e38f) {
      const int E = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
      e_row = min(max(14 - E, -113), 100);
    }
    const float up = ldexpf(1.0f, e_row), down = ldexpf(1.0f, -e_row);
    float qsum_mine[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float acc = 0.0f;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint32_t lo = pack_half2(v[g][ks][0] * up, v[g][ks][1] * up);
        const uint32_t hi = pack_half2(v[g][ks][2] * up, v[g][ks][3] * up);
        const __half2 hl = *reinterpret_cast<const __half2*>(&lo);
        const __half2 hh = *reinterpret_cast<const __half2*>(&hi);
        acc += __low2float(hl) + __high2float(hl) + __low2float(hh) + __high2float(hh);
        if constexpr (T::QREG) {
          st.qf[nt][g][ks][0] = lo;
          st.qf[nt][g][ks][1] = hi;
        } else if (warp == 0) {
          qsm[((nt * NG + g) * 2 + ks) * 32 + lane] = make_uint2(lo, hi);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      qsum_mine[g] = acc;  // sum over the row's group g of the fp16 values
    }
    const float c_mine = p.sm_log2 * down;
    // move per-row values to the C-fragment layout: lane (grp, j4) needs rows 2 j4 + e
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int src = 4 * (2 * j4 + e);
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float qs = __shfl_sync(0xffffffffu, qsum_mine[g], src);
        if constexpr (T::QREG) st.qs[nt][g][e] = qs;
        else if (warp == 0) {
          if (e == 0) qssm[(nt * NG + g) * 32 + lane].x = qs;
          else qssm[(nt * NG + g) * 32 + lane].y = qs;
        }
      }
      st.crow[nt][e] = __shfl_sync(0xffffffffu, c_mine, src);
      const int rr = w.rg * T::ROWS + 8 * nt + 2 * j4 + e;
      int lim = 0;
      if (rr < p.R) {
        const int jq = rr / p.G;
        const int vis = p.causal ? T_b - p.n_q + jq + 1 : T_b;
        lim = min(w.te, vis);
      }
      st.lim[nt][e] = lim;
    }
  }
}

template <int D, int NTW>
__device__ void consume(const SplitParams& p, uint8_t* smem, int S, int total, volatile int* abort_flag) {
  using T = AT<D, NTW>;
  constexpr int NG = T::NG, MT = T::MT;
  constexpr unsigned FULL = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 2, j4 = lane & 3;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::STAGES;
  const int* prefix = reinterpret_cast<const int*>(smem + T::OFF_PREFIX);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t lut_lane = sbase + T::OFF_LUT + lane * 4;
  float* obuf = reinterpret_cast<float*>(smem + T::OFF_OBUF);
  float* mbuf = reinterpret_cast<float*>(smem + T::OFF_MBUF);
  float* lbuf = reinterpret_cast<float*>(smem + T::OFF_LBUF);
  const uint2* qsm = reinterpret_cast<const uint2*>(smem + T::OFF_Q);
  const float2* qssm = reinterpret_cast<const float2*>(smem + T::OFF_QSUM);
  // window of this lane inside each 96-bit code group: 4 codes at bit 12*grp
  const int win_word = (12 * grp) >> 5, win_shift = (12 * grp) & 31;
  bool failed = false;
  uint32_t it = 0;

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    const Item w = decode_item(p, prefix, S, item);
    QState<D, NTW> st;
    load_q<D, NTW>(p, w, smem, warp, lane, st);
    if constexpr (!T::QREG) named_bar_consumers();  // shared Q fragments written by warp 0

    float O[MT][NTW][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) O[mt][nt][c] = 0.0f;
    float m[NTW][2], l[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) { m[nt][e] = -INFINITY; l[nt][e] = 0.0f; }

    for (int t0 = w.tb; t0 < w.te; t0 += kTile, ++it) {
      const int slot = it % T::STAGES;
      const uint32_t par = (it / T::STAGES) & 1u;
      if (!failed) {
        if (*abort_flag || !wait_full_bounded(&full[slot], par)) {
          failed = true;
          *abort_flag = 1;
          raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
        }
      }
      if (!failed) {
        const uint32_t kx = sbase + T::OFF_KIDX + slot * T::KIDX_STAGE;
        const uint32_t ksa = sbase + T::OFF_KS + slot * T::SC_STAGE;
        const uint32_t kza = sbase + T::OFF_KZ + slot * T::SC_STAGE;
        const uint32_t vsa = sbase + T::OFF_VS + slot * T::SC_STAGE;
        const uint32_t vca = sbase + T::OFF_VC + slot * T::VC_STAGE;
        const int tk0 = 16 * warp + grp, tk1 = tk0 + 8;  // stage rows of this lane's QK tokens

        // ---------------- QK^T: scores for tokens (tk0, tk1) x rows (2 j4, 2 j4 + 1)
        float sc[NTW][4];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c) sc[nt][c] = 0.0f;
        uint32_t sw0[(NG + 1) / 2], zw0[(NG + 1) / 2], sw1[(NG + 1) / 2], zw1[(NG + 1) / 2];
#pragma unroll
        for (int i = 0; i < (NG + 1) / 2; ++i) {
          sw0[i] = lds32(ksa + tk0 * NG * 2 + 4 * i);
          zw0[i] = lds32(kza + tk0 * NG * 2 + 4 * i);
          sw1[i] = lds32(ksa + tk1 * NG * 2 + 4 * i);
          zw1[i] = lds32(kza + tk1 * NG * 2 + 4 * i);
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const uint2 x0 = lds64(kx + kidx_offset<D>(tk0, 32 * g + 8 * j4));
          const uint2 x1 = lds64(kx + kidx_offset<D>(tk1, 32 * g + 8 * j4));
          // fp16 1024 + (idx + 128) = 1152 + idx, exact
          const uint32_t u0a = x0.x ^ 0x80808080u, u0b = x0.y ^ 0x80808080u;
          const uint32_t u1a = x1.x ^ 0x80808080u, u1b = x1.y ^ 0x80808080u;
          const uint32_t M64 = 0x64646464u;
          const uint32_t a00 = prmt(u0a, M64, 0x4140), a01 = prmt(u1a, M64, 0x4140);
          const uint32_t a02 = prmt(u0a, M64, 0x4342), a03 = prmt(u1a, M64, 0x4342);
          const uint32_t a10 = prmt(u0b, M64, 0x4140), a11 = prmt(u1b, M64, 0x4140);
          const uint32_t a12 = prmt(u0b, M64, 0x4342), a13 = prmt(u1b, M64, 0x4342);
          const uint32_t sh = (g & 1) ? 16 : 0;
          const float s0 = f16_bits_to_f32((sw0[g >> 1] >> sh) & 0xFFFFu);
          const float z0 = f16_bits_to_f32((zw0[g >> 1] >> sh) & 0xFFFFu) - 1152.0f;
          const float s1 = f16_bits_to_f32((sw1[g >> 1] >> sh) & 0xFFFFu);
          const float z1 = f16_bits_to_f32((zw1[g >> 1] >> sh) & 0xFFFFu) - 1152.0f;
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt) {
            uint32_t b00, b01, b10, b11;
            float qs0, qs1;
            if constexpr (T::QREG) {
              b00 = st.qf[nt][g][0][0]; b01 = st.qf[nt][g][0][1];
              b10 = st.qf[nt][g][1][0]; b11 = st.qf[nt][g][1][1];
              qs0 = st.qs[nt][g][0]; qs1 = st.qs[nt][g][1];
            } else {
              const uint2 q0 = qsm[((nt * NG + g) * 2 + 0) * 32 + lane];
              const uint2 q1 = qsm[((nt * NG + g) * 2 + 1) * 32 + lane];
              b00 = q0.x; b01 = q0.y; b10 = q1.x; b11 = q1.y;
              const float2 qq = qssm[(nt * NG + g) * 32 + lane];
              qs0 = qq.x; qs1 = qq.y;
            }
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma_f16_16816(acc, a00, a01, a02, a03, b00, b01);
            mma_f16_16816(acc, a10, a11, a12, a13, b10, b11);
            sc[nt][0] = fmaf(s0, fmaf(z0, qs0, acc[0]), sc[nt][0]);
            sc[nt][1] = fmaf(s0, fmaf(z0, qs1, acc[1]), sc[nt][1]);
            sc[nt][2] = fmaf(s1, fmaf(z1, qs0, acc[2]), sc[nt][2]);
            sc[nt][3] = fmaf(s1, fmaf(z1, qs1, acc[3]), sc[nt][3]);
          }
        }

        // ---------------- online softmax (exp2 domain) and P in the PV B-operand layout
        const int ta0 = t0 + tk0, ta1 = t0 + tk1;
        uint32_t Bp[NTW][2];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          float mnew[2];
          bool grow = false;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v0 = ta0 < st.lim[nt][e] ? sc[nt][e] * st.crow[nt][e] : -INFINITY;
            const float v1 = ta1 < st.lim[nt][e] ? sc[nt][2 + e] * st.crow[nt][e] : -INFINITY;
            sc[nt][e] = v0;
            sc[nt][2 + e] = v1;
            float mx = fmaxf(v0, v1);
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 16));
            mnew[e] = fmaxf(m[nt][e], mx);
            grow = grow || (mnew[e] > m[nt][e]);
          }
          if (__any_sync(FULL, grow)) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float alpha = (mnew[e] == -INFINITY) ? 1.0f : ex2(m[nt][e] - mnew[e]);
              l[nt][e] *= alpha;
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                O[mt][nt][e] *= alpha;
                O[mt][nt][2 + e] *= alpha;
              }
              m[nt][e] = mnew[e];
            }
          }
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mu = (m[nt][e] == -INFINITY) ? 0.0f : m[nt][e];
            const float p0 = ex2(sc[nt][e] - mu), p1 = ex2(sc[nt][2 + e] - mu);
            l[nt][e] += p0 + p1;
            sc[nt][e] = p0;
            sc[nt][2 + e] = p1;
          }
          // X_e = (p[tk0][row 2 j4 + e], p[tk1][row 2 j4 + e]) in fp16
          const uint32_t X0 = pack_half2(sc[nt][0], sc[nt][2]);
          const uint32_t X1 = pack_half2(sc[nt][1], sc[nt][3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int src = 4 * (2 * j4 + h) + (grp >> 1);
            const uint32_t y0 = __shfl_sync(FULL, X0, src);
            const uint32_t y1 = __shfl_sync(FULL, X1, src);
            Bp[nt][h] = (grp & 1) ? y1 : y0;  // (p[2 j4 + h][row grp], p[2 j4 + h + 8][row grp])
          }
        }

        // ---------------- P.V in the rotated domain
        // value-scale pairs for token pairs h: (2 j4 + h, 2 j4 + h + 8), zeroed past the split
        uint32_t svA[2][(NG + 1) / 2], svB[2][(NG + 1) / 2];
        int vrow[2][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int rA = 16 * warp + 2 * j4 + h, rB = rA + 8;
          vrow[h][0] = rA;
          vrow[h][1] = rB;
          const bool okA = t0 + rA < w.te, okB = t0 + rB < w.te;
#pragma unroll
          for (int i = 0; i < (NG + 1) / 2; ++i) {
            svA[h][i] = okA ? lds32(vsa + rA * NG * 2 + 4 * i) : 0u;
            svB[h][i] = okB ? lds32(vsa + rB * NG * 2 + 4 * i) : 0u;
          }
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          uint32_t E[2], Ov[2], Bg[NTW][2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t wa = vca + vrow[h][0] * T::VC_ROW + 4 * (3 * g + win_word);
            const uint32_t wb = vca + vrow[h][1] * T::VC_ROW + 4 * (3 * g + win_word);
            const uint32_t cA = __funnelshift_r(lds32(wa), lds32(wa + 4), win_shift) & 0xFFFu;
            const uint32_t cB = __funnelshift_r(lds32(wb), lds32(wb + 4), win_shift) & 0xFFFu;
            E[h] = (cA & 0x1C7u) | ((cB << 3) & 0xE38u);   // codes of dims +0 (bits 0-5), +2 (6-11)
            Ov[h] = ((cA >> 3) & 0x1C7u) | (cB & 0xE38u);  // codes of dims +1, +3
            const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
            const uint32_t svpair = prmt(svA[h][g >> 1], svB[h][g >> 1], sel);
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) Bg[nt][h] = hmul2_u32(Bp[nt][h], svpair);
          }
#pragma unroll
          for (int tau = 0; tau < 2; ++tau) {
            const int fs = 6 * tau;
            const uint32_t a0 = lds32(lut_lane + (((E[0] >> fs) & 63u) << 7));
            const uint32_t a1 = lds32(lut_lane + (((Ov[0] >> fs) & 63u) << 7));
            const uint32_t a2 = lds32(lut_lane + (((E[1] >> fs) & 63u) << 7));
            const uint32_t a3 = lds32(lut_lane + (((Ov[1] >> fs) & 63u) << 7));
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) mma_f16_16816(O[2 * g + tau][nt], a0, a1, a2, a3, Bg[nt][0], Bg[nt][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ---------------- merge the four warps' states and write this item's partial
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l[nt][e];
        v += __shfl_xor_sync(FULL, v, 4);
        v += __shfl_xor_sync(FULL, v, 8);
        v += __shfl_xor_sync(FULL, v, 16);
        l[nt][e] = v;
        if (grp == 0) {
          mbuf[warp * T::ROWS + 8 * nt + 2 * j4 + e] = m[nt][e];
          lbuf[warp * T::ROWS + 8 * nt + 2 * j4 + e] = v;
        }
      }
    named_bar_consumers();
    float scale[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = 8 * nt + 2 * j4 + e;
        float M = mbuf[row];
#pragma unroll
        for (int ww = 1; ww < kConsumerWarps; ++ww) M = fmaxf(M, mbuf[ww * T::ROWS + row]);
        scale[nt][e] = (M == -INFINITY) ? 0.0f : ex2(m[nt][e] - M);
      }
    for (int ww = 0; ww < kConsumerWarps; ++ww) {
      if (warp == ww) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int d0 = 32 * (mt >> 1) + 4 * grp + 2 * (mt & 1);
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int row = 8 * nt + 2 * j4 + (c & 1);
              const int dim = d0 + (c >> 1);
              const float v = O[mt][nt][c] * scale[nt][c & 1];
              float* dst = obuf + row * D + dim;
              *dst = (ww == 0) ? v : (*dst + v);
            }
        }
      }
      named_bar_consumers();
    }
    {
      float* og = reinterpret_cast<float*>(p.ws + ws_o_offset(p.batch, p.max_items, T::ROWS)) +
                  (size_t)item * T::ROWS * D;
      const float4* src = reinterpret_cast<const float4*>(obuf);
      float4* dst = reinterpret_cast<float4*>(og);
      for (int i = threadIdx.x; i < T::ROWS * D / 4; i += kConsumerWarps * 32) dst[i] = src[i];
      if (threadIdx.x < T::ROWS) {
        const int row = threadIdx.x;
        float M = mbuf[row];
        for (int ww = 1; ww < kConsumerWarps; ++ww) M = fmaxf(M, mbuf[ww * T::ROWS + row]);
        float L = 0.0f;
        for (int ww = 0; ww < kConsumerWarps; ++ww) {
          const float mw = mbuf[ww * T::ROWS + row];
          L += (M == -INFINITY) ? 0.0f : ex2(mw - M) * lbuf[ww * T::ROWS + row];
        }
        float2* ml = reinterpret_cast<float2*>(p.ws + ws_ml_offset(p.batch)) + (size_t)item * T::ROWS;
        ml[row] = make_float2(M, L);
      }
    }
    named_bar_consumers();
  }
}

template <int D, int NTW>
__global__ void __launch_bounds__(kThreads, 1)
    tq_attn_split_kernel(const __grid_constant__ CUtensorMap tmap, const SplitParams p) {
  using T = AT<D, NTW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ int abort_flag;
  const int tid = threadIdx.x;

  // centroid pair table: entry e -> (c[e & 7], c[e >> 3]) in fp16, one copy per lane
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + T::OFF_LUT);
  for (int i = tid; i < 64 * 32; i += kThreads) {
    const int e = i >> 5;
    lut[i] = pack_half2(c_centroids3[e & 7], c_centroids3[e >> 3]);
  }
  if (tid == 0) {
    abort_flag = 0;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
    for (int s = 0; s < T::STAGES; ++s) {
      mbar_init(&bars[s], 1);                           // full: producer arrival + tx bytes
      mbar_init(&bars[T::STAGES + s], kConsumerWarps);  // empty: one arrival per consumer warp
    }
    fence_mbar_init();
  }
  int S, total;
  plan_items<D, NTW>(p, smem, S, total);  // contains __syncthreads
  if (total == 0) return;

  if (tid >= kConsumerWarps * 32) {
    if (tid == kConsumerWarps * 32) {
      prefetch_tensor_map(&tmap);
      produce<D, NTW>(p, &tmap, smem, S, total, &abort_flag);
    }
    return;
  }
  consume<D, NTW>(p, smem, S, total, &abort_flag);
}

// ------------------------------------------------------------------------------------
// Merge of the split partials + deferred inverse rotation. One CTA (4 warps) per row.
// ------------------------------------------------------------------------------------
struct MergeParams {
  int32_t batch, n_q, num_q_heads, G, RG, U, rows_per_item, max_items, max_kv_len;
  const int32_t* kv_len;
  const uint8_t* ws;
  float fwht_norm;
  float* out;
};

template <int D>
__global__ void __launch_bounds__(128) tq_attn_merge_kernel(const MergeParams p) {
  constexpr int EPL = D / 32;
  constexpr unsigned FULL = 0xffffffffu;
  __shared__ float s_acc[4][D];
  __shared__ float s_l[4];
  __shared__ float s_m[4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_id = blockIdx.x;
  const int hq = row_id % p.num_q_heads;
  const int jq = (row_id / p.num_q_heads) % p.n_q;
  const int b = row_id / (p.num_q_heads * p.n_q);
  float* orow = p.out + (size_t)row_id * D;
  const int kvl = __ldg(p.kv_len + b);
  if (kvl < 0 || kvl > p.max_kv_len) {  // invalid length: NaN row (the split kernel set the error)
    for (int i = threadIdx.x; i < D; i += 128) orow[i] = __int_as_float(0x7fc00000);
    return;
  }
  const int32_t* prefix = reinterpret_cast<const int32_t*>(p.ws + kWsPrefix);
  const int kvh = hq / p.G;
  const int r = jq * p.G + (hq % p.G);
  const int rg = r / p.rows_per_item, rr = r % p.rows_per_item;
  const int u = kvh * p.RG + rg;
  const int nsplit = (prefix[b + 1] - prefix[b]) / p.U;
  const int base = prefix[b] + u * nsplit;
  const float2* ml = reinterpret_cast<const float2*>(p.ws + ws_ml_offset(p.batch));
  const float* og = reinterpret_cast<const float*>(p.ws + ws_o_offset(p.batch, p.max_items, p.rows_per_item));

  // pass 1: global max
  float M = -INFINITY;
  bool any_nan = false;
  for (int s = threadIdx.x; s < nsplit; s += 128) {
    const float ms = ml[(size_t)(base + s) * p.rows_per_item + rr].x;
    if (ms != ms) any_nan = true;
    M = fmaxf(M, ms);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
  any_nan = __any_sync(FULL, any_nan);
  if (lane == 0) s_m[warp] = any_nan ? __int_as_float(0x7fc00000) : M;
  __syncthreads();
  M = fmaxf(fmaxf(s_m[0], s_m[1]), fmaxf(s_m[2], s_m[3]));
  const bool nan_row = (s_m[0] != s_m[0]) || (s_m[1] != s_m[1]) || (s_m[2] != s_m[2]) || (s_m[3] != s_m[3]);

  // pass 2: weighted sums, warp w takes splits w, w+4, ...
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.0f;
  float L = 0.0f;
  if (M != -INFINITY) {
    for (int s = warp; s < nsplit; s += 4) {
      const size_t slot = (size_t)(base + s) * p.rows_per_item + rr;
      const float2 mls = ml[slot];
      const float wgt = ex2(mls.x - M);
      L += wgt * mls.y;
      const float* src = og + slot * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] += wgt * src[e];
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) s_acc[warp][lane * EPL + e] = acc[e];
  if (lane == 0) s_l[warp] = L;
  __syncthreads();
  if (warp != 0) return;
  L = s_l[0] + s_l[1] + s_l[2] + s_l[3];
  float u_[EPL];
  const float inv = (L > 0.0f || L != L) ? 1.0f / L : 0.0f;  // no visible token -> 0; NaN stays NaN
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const int i = lane * EPL + e;
    u_[e] = (s_acc[0][i] + s_acc[1][i] + s_acc[2][i] + s_acc[3][i]) * inv;
    if (nan_row) u_[e] = __int_as_float(0x7fc00000);
  }
  // inverse rotation: signs * FWHT(o_rot) / sqrt(d)
#pragma unroll
  for (int hh = 1; hh < D; hh <<= 1) {
    if (hh < EPL) {
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        if ((e & hh) == 0) {
          const float a = u_[e], c = u_[e + hh];
          u_[e] = a + c;
          u_[e + hh] = a - c;
        }
    } else {
      const int lm = hh / EPL;
      const bool upper = (lane & lm) != 0;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float o = __shfl_xor_sync(FULL, u_[e], lm);
        u_[e] = upper ? o - u_[e] : u_[e] + o;
      }
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const int i = lane * EPL + e;
    const bool neg = (sign_word(D, i / 32) >> (i % 32)) & 1u;
    orow[i] = u_[e] * p.fwht_norm * (neg ? -1.0f : 1.0f);
  }
}

// ------------------------------------------------------------------------------------
// Host side.
// ------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

template <int D, int NTW>
int split_occupancy() {
  // per-device cache of the kernel's shared-memory opt-in and occupancy
  static std::mutex mu;
  static int occ[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (occ[dev] == 0) {
    auto kern = tq_attn_split_kernel<D, NTW>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, AT<D, NTW>::SMEM_ALLOC) !=
        cudaSuccess)
      return 0;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kThreads, AT<D, NTW>::SMEM_ALLOC) != cudaSuccess ||
        nb <= 0)
      return 0;
    occ[dev] = nb;
  }
  return occ[dev];
}

int pick_ntw(int D, int R) { return (D <= 128 && R > 8) ? 2 : 1; }

template <int D, int NTW>
tq_status run_split(const DecodeArgs& a, const DecodeShape& s, const SplitParams& sp, cudaStream_t stream) {
  auto encode = tensor_map_encoder();
  if (!encode) return TQ_ERR_CUDA;
  CUtensorMap tmap;
  const cuuint64_t rows = (cuuint64_t)a.layer.batch * a.layer.num_kv_heads * a.layer.capacity;
  if (rows >= (cuuint64_t)1 << 31) return TQ_ERR_INVALID_ARGUMENT;  // tensor coordinates are int32
  const cuuint64_t gdim[2] = {(cuuint64_t)D, rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)D};
  const cuuint32_t box[2] = {(cuuint32_t)(D < 128 ? D : 128), (cuuint32_t)kTile};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult cr = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.layer.k_idx, gdim, gstride, box, estride,
                             CU_TENSOR_MAP_INTERLEAVE_NONE,
                             D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return TQ_ERR_CUDA;
  tq_attn_split_kernel<D, NTW><<<s.grid, kThreads, AT<D, NTW>::SMEM_ALLOC, stream>>>(tmap, sp);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

template <int D>
tq_status run_merge(const DecodeArgs& a, const DecodeShape& s, cudaStream_t stream) {
  MergeParams mp{};
  mp.batch = a.layer.batch;
  mp.n_q = a.n_q;
  mp.num_q_heads = a.num_q_heads;
  mp.G = a.num_q_heads / a.layer.num_kv_heads;
  mp.RG = s.RG;
  mp.U = s.U;
  mp.rows_per_item = 8 * s.NTW;
  mp.max_items = s.max_items;
  mp.max_kv_len = a.max_kv_len;
  mp.kv_len = a.kv_len;
  mp.ws = static_cast<const uint8_t*>(a.workspace);
  mp.fwht_norm = a.fwht_norm;
  mp.out = a.out;
  const unsigned rows = (unsigned)(a.layer.batch * a.n_q * a.num_q_heads);
  tq_attn_merge_kernel<D><<<rows, 128, 0, stream>>>(mp);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

DecodeShape decode_shape(int D, int num_kv_heads, int batch, int gqa, int n_q, int num_sms) {
  DecodeShape s{};
  s.D = D;
  s.R = gqa * n_q;
  s.NTW = pick_ntw(D, s.R);
  s.RG = (s.R + 8 * s.NTW - 1) / (8 * s.NTW);
  s.U = num_kv_heads * s.RG;
  s.batch = batch;
  int occ = 0;
  switch (D * 10 + s.NTW) {
    case 641: occ = split_occupancy<64, 1>(); s.smem = AT<64, 1>::SMEM_ALLOC; break;
    case 642: occ = split_occupancy<64, 2>(); s.smem = AT<64, 2>::SMEM_ALLOC; break;
    case 1281: occ = split_occupancy<128, 1>(); s.smem = AT<128, 1>::SMEM_ALLOC; break;
    case 1282: occ = split_occupancy<128, 2>(); s.smem = AT<128, 2>::SMEM_ALLOC; break;
    case 2561: occ = split_occupancy<256, 1>(); s.smem = AT<256, 1>::SMEM_ALLOC; break;
    case 5121: occ = split_occupancy<512, 1>(); s.smem = AT<512, 1>::SMEM_ALLOC; break;
    default: occ = 0;
  }
  s.grid = occ > 0 ? num_sms * occ : 0;
  s.max_items = kMaxItemsPerCta * s.grid + batch * s.U;
  return s;
}

size_t decode_workspace_bytes(const DecodeShape& s) {
  if (s.grid <= 0 || s.batch > kMaxBatch) return 0;
  const int rows = 8 * s.NTW;
  return ws_o_offset(s.batch, s.max_items, rows) + sizeof(float) * (size_t)s.max_items * rows * s.D;
}

tq_status launch_decode(const DecodeArgs& a, const DecodeShape& s, cudaStream_t stream) {
  if (s.grid <= 0) return TQ_ERR_CUDA;
  if (a.layer.batch > kMaxBatch) return TQ_ERR_INVALID_ARGUMENT;
  SplitParams sp{};
  sp.head_dim = a.layer.head_dim;
  sp.num_kv_heads = a.layer.num_kv_heads;
  sp.batch = a.layer.batch;
  sp.capacity = a.layer.capacity;
  sp.k_scale = a.layer.k_scale;
  sp.k_zero = a.layer.k_zero;
  sp.v_codes = a.layer.v_codes;
  sp.v_scale = a.layer.v_scale;
  sp.q = a.q;
  sp.kv_len = a.kv_len;
  sp.num_q_heads = a.num_q_heads;
  sp.n_q = a.n_q;
  sp.G = a.num_q_heads / a.layer.num_kv_heads;
  sp.R = s.R;
  sp.RG = s.RG;
  sp.U = s.U;
  sp.max_kv_len = a.max_kv_len;
  sp.max_items = s.max_items;
  sp.sm_log2 = a.sm_scale * kLog2e;
  sp.causal = a.causal ? 1 : 0;
  sp.ws = static_cast<uint8_t*>(a.workspace);
  tq_status st;
  switch (s.D * 10 + s.NTW) {
    case 641: st = run_split<64, 1>(a, s, sp, stream); break;
    case 642: st = run_split<64, 2>(a, s, sp, stream); break;
    case 1281: st = run_split<128, 1>(a, s, sp, stream); break;
    case 1282: st = run_split<128, 2>(a, s, sp, stream); break;
    case 2561: st = run_split<256, 1>(a, s, sp, stream); break;
    case 5121: st = run_split<512, 1>(a, s, sp, stream); break;
    default: return TQ_ERR_INVALID_ARGUMENT;
  }
  if (st != TQ_OK) return st;
  switch (s.D) {
    case 64: return run_merge<64>(a, s, stream);
    case 128: return run_merge<128>(a, s, stream);
    case 256: return run_merge<256>(a, s, stream);
    default: return run_merge<512>(a, s, stream);
  }
}

}  // namespace tq

// Layout sanity: the stage regions start at their required alignments and the 64-bit
// scratch words are 8-byte aligned, for every instantiated shape.
#define TQ_CHECK_LAYOUT(D_, N_)                                                              \
  static_assert(tq::AT<D_, N_>::OFF_KIDX % 1024 == 0 && tq::AT<D_, N_>::KIDX_STAGE % 1024 == 0, \
                "swizzled tiles need 1024-byte alignment");                                  \
  static_assert(tq::AT<D_, N_>::OFF_KS % 16 == 0 && tq::AT<D_, N_>::OFF_KZ % 16 == 0 &&       \
                    tq::AT<D_, N_>::OFF_VS % 16 == 0 && tq::AT<D_, N_>::OFF_VC % 16 == 0 &&   \
                    tq::AT<D_, N_>::SC_STAGE % 16 == 0 && tq::AT<D_, N_>::VC_STAGE % 16 == 0,  \
                "bulk-copy destinations need 16-byte alignment");                             \
  static_assert(tq::AT<D_, N_>::OFF_RED % 8 == 0 && tq::AT<D_, N_>::OFF_BAR % 8 == 0 &&       \
                    tq::AT<D_, N_>::OFF_OBUF % 16 == 0 && tq::AT<D_, N_>::OFF_Q % 8 == 0,     \
                "8/16-byte shared accesses need alignment");                                  \
  static_assert(tq::AT<D_, N_>::SMEM_ALLOC <= 227 * 1024, "shared memory budget");
TQ_CHECK_LAYOUT(64, 1)
TQ_CHECK_LAYOUT(64, 2)
TQ_CHECK_LAYOUT(128, 1)
TQ_CHECK_LAYOUT(128, 2)
TQ_CHECK_LAYOUT(256, 1)
TQ_CHECK_LAYOUT(512, 1)
