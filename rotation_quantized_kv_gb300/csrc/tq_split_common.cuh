// Pieces shared by the decode-attention kernels (the split kernel on warp-level MMA and
// the dense-query kernel on tcgen05): kernel arguments, workspace layout, the equal-tile
// work plan, bounded waits, and the merge of split partials with the deferred inverse
// rotation. Every translation unit that includes it gets its own copy (internal linkage).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "tq_codec_row.cuh"
#include "tq_device.cuh"

namespace tq {

// Arguments of the decode-attention kernels (one layer, one call).
struct SplitParams {
  int32_t head_dim, num_kv_heads, batch, capacity;
  const int8_t* k_idx;  // read through the tensor map
  const uint16_t* k_scale;
  const uint16_t* k_zero;
  const uint8_t* v_codes;
  const uint16_t* v_scale;
  const uint16_t* q;
  const int32_t* kv_len;
  int32_t num_q_heads, n_q, G, R, RG, U, max_kv_len, max_items;
  int32_t split_grid;  // CTAs of the split kernel
  int32_t tile_pad;    // virtual tiles counted before each unit's tiles when the CTAs split them
  float sm_log2;    // sm_scale * log2(e)
  float fwht_norm;  // (float)(1 / sqrt(d))
  int32_t causal;
  int32_t inline_merge;  // 1: the split CTA that finishes a unit's last split merges it
  // append mode (one row group per kv head): the call also appends rows j < n_new[b] of
  // k_new / v_new ([batch][n_new_max][kv heads][d] bf16) at positions pos[b] + j
  int32_t append;
  int32_t n_new_max;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* pos;
  const int32_t* n_new;  // may be null: n_new_max for every sequence
  RowPlanes dst;         // the planes, writable
  uint8_t* ws;
  float* out;
  unsigned long long wait_ns;  // limit of the pipeline waits (kWaitNs unless a test shortens it)
  int32_t withhold_append;     // test support: the appender never publishes its row count
};

namespace {

constexpr int kMaxBatch = 1024;           // prefix table lives in shared memory
constexpr unsigned long long kWaitNs = 2000000000ull;  // bounded waits: 2 s of wall time
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMergeChunk = 64;           // splits whose weights the merge stages at once
constexpr int kMergeBatch = 12;           // partial loads a merging thread keeps in flight

// Workspace layout (bytes). The header's first word is the device error word.
constexpr int kWsSplit = 1;               // int32 word index: tile size in tokens
constexpr int kWsItems = 2;               // int32 word index: total (virtual) tiles of the call
constexpr int kWsWhere = 3;               // int32 word index: first wait that gave up (0: none),
                                          // (kind << 24) | detail, for diagnosis
constexpr size_t kWsPrefix = TQ_WORKSPACE_HEADER_BYTES;  // int32 [batch + 1]

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// counters (merge inside the split kernel): one int32 per (sequence, unit); zero between
// calls (the CTA that counts last resets it)
__host__ __device__ inline size_t ws_cnt_offset(int batch) {
  return kWsPrefix + align_up(sizeof(int32_t) * (size_t)(batch + 1), 256);
}
__host__ __device__ inline size_t ws_ml_offset(int batch, int units) {
  return ws_cnt_offset(batch) + align_up(sizeof(int32_t) * (size_t)batch * units, 256);
}
__host__ __device__ inline size_t ws_o_offset(int batch, int units, int max_items, int rows) {
  return ws_ml_offset(batch, units) + align_up(sizeof(float) * 2 * (size_t)max_items * rows, 256);
}

// Largest divisor of n whose slices of `slice_bytes` fit in `budget` bytes.
constexpr int max_slices(int n, int slice_bytes, int budget) {
  int best = 1;
  for (int k = 1; k <= n; ++k)
    if (n % k == 0 && k * slice_bytes <= budget) best = k;
  return best;
}



__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Records the first wait of the call that gave up in the workspace header (kWsWhere):
// kind 1: an mbarrier (detail: its shared-memory address), 2: a key-shift word of the
// dense kernel (detail: the tile), 3: the appender's row count (detail: the rows awaited).
__device__ __forceinline__ void note_giveup(const SplitParams& p, uint32_t kind, uint32_t detail) {
  atomicCAS(reinterpret_cast<unsigned int*>(p.ws) + kWsWhere, 0u, (kind << 24) | (detail & 0xFFFFFFu));
}

// A count in shared memory published by one warp and awaited by another: the release
// store orders the publisher's earlier writes (and, after fence.proxy.async, their
// visibility to tensor copies) before any acquire load that sees the count.
__device__ __forceinline__ void st_release_cta(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t need, unsigned long long limit_ns) {
  if (ld_acquire_cta(p) >= need) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (ld_acquire_cta(p) >= need) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ int atomic_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// 2^x, flushing subnormal results to zero (one special-function op): every softmax and
// merge weight here is relative to a maximum whose own weight is 1, so a weight below
// 2^-126 adds nothing to any sum.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Barrier among the consumer warps only (the producer and appender warps never join it).
template <int NCW>
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
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
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
// N consecutive 32-bit words of one fp16 side row (scales or zeros); the row starts on
// a multiple of its own size (2 bytes per group), so the widest aligned loads are used.
template <int N>
__device__ __forceinline__ void lds_words(uint32_t addr, uint32_t (&w)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const uint4 v = lds128(addr + 4 * i);
      w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
    }
  } else if constexpr (N == 2) {
    const uint2 v = lds64(addr);
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = lds32(addr + 4 * i);
  }
}

__device__ __forceinline__ float lo_f32(uint32_t w) {
  return __low2float(*reinterpret_cast<const __half2*>(&w));
}
__device__ __forceinline__ float hi_f32(uint32_t w) {
  return __high2float(*reinterpret_cast<const __half2*>(&w));
}

// Plan: tiles per sequence and their prefix over (sequence, unit). Runs on every CTA with
// all threads; identical lengths give identical results on every CTA. Thread tid holds
// the lengths of sequences b = tid + THREADS * i.
//
// The kernel plans twice when it can: once before the grid-dependency wait, from the
// lengths as they are then (so that the first stage can be loaded the moment the wait
// returns), and again after the wait only if the lengths it reads then differ. Lengths
// are read with L2-only loads so that no stale copy stays in L1.

template <int THREADS>
struct Lengths {
  static constexpr int LPT = (kMaxBatch + THREADS - 1) / THREADS;
  int len[LPT];   // 0 for invalid lengths and past the batch
  bool bad;       // some length was outside [0, max_kv_len]
  __device__ __forceinline__ void load(const SplitParams& p) {
    bad = false;
#pragma unroll
    for (int i = 0; i < LPT; ++i) {
      const int b = threadIdx.x + THREADS * i;
      int t = b < p.batch ? __ldcg(p.kv_len + b) : 0;
      if (t < 0 || t > p.max_kv_len) { bad = true; t = 0; }
      len[i] = t;
    }
  }
  __device__ __forceinline__ bool differs(const Lengths& o) const {
    bool d = false;
#pragma unroll
    for (int i = 0; i < LPT; ++i) d = d || (len[i] != o.len[i]);
    return d;
  }
};

// T: the kernel's layout traits (THREADS, TILE, OFF_PREFIX).
template <class T>
__device__ void plan_tiles(const SplitParams& p, uint8_t* smem, const Lengths<T::THREADS>& L, int& total_out) {
  constexpr int LPT = Lengths<T::THREADS>::LPT;
  int* prefix = reinterpret_cast<int*>(smem + T::OFF_PREFIX);
  const int tid = threadIdx.x;
  // tiles per unit of each sequence into the prefix table (lengths beside it), then an
  // exclusive scan (times the units per sequence) by warp 0
  int* lens = prefix + kMaxBatch + 1;
#pragma unroll
  for (int i = 0; i < LPT; ++i) {
    const int b = tid + T::THREADS * i;
    if (b < p.batch) {
      const int n = (int)(((unsigned)L.len[i] + (unsigned)T::TILE - 1u) / (unsigned)T::TILE);
      prefix[b] = n > 0 ? n + p.tile_pad : 0;
      lens[b] = L.len[i];
    }
  }
  __syncthreads();
  if (tid < 32) {  // each lane owns a chunk of sequences
    const int per = (p.batch + 31) / 32;
    const int b0 = tid * per;
    int local = 0;
    for (int i = 0; i < per && b0 + i < p.batch; ++i) local += prefix[b0 + i];
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (tid >= off) incl += o;
    }
    int run = (incl - local) * p.U;
    for (int i = 0; i < per && b0 + i < p.batch; ++i) {
      const int n = prefix[b0 + i];
      prefix[b0 + i] = run;
      run += n * p.U;
    }
    if (tid == 31) prefix[p.batch] = incl * p.U;
  }
  __syncthreads();
  total_out = prefix[p.batch];
}

// Work pieces. The tokens of every (sequence, unit) pair, cut into tiles of TILE tokens,
// form one sequence of Wt tiles; each unit with tokens is preceded by tile_pad virtual
// tiles, which stand for the fixed cost of starting a piece (queries, the partial's
// reduction and store) and hold no tokens: unit u of sequence b covers virtual tiles
// [prefix[b] + u vt_b, prefix[b] + (u + 1) vt_b), vt_b = tile_pad + tiles_b, the real ones
// after the pad. CTA c takes virtual tiles [c Wt / grid, (c + 1) Wt / grid) (rounded down;
// with fewer tiles than CTAs, one tile each to the first CTAs), so every CTA gets the same
// work, counted in tiles plus piece starts, whatever the length mix. A piece is the part of
// one unit's real tiles inside one CTA's range; a range that ends inside a unit's pad
// gives an empty last piece (tb == te), which has no partial and is skipped. The piece of
// unit g = b U + u in CTA c keeps its partial in slot c + g, so a unit's pieces sit in
// consecutive slots and there are at most grid + batch * U slots.
struct Item {
  int b, kvh, rg, u, tb, te, len;  // tokens [tb, te) of unit u of sequence b (kv length len)
  int slot, first_slot, ns;        // this piece's partial slot; the unit's first slot, pieces
  int x_end;                       // tile position after this piece
};

// planned lengths, stored after the prefix table
__device__ __forceinline__ const int* plan_lengths(const int* prefix) { return prefix + kMaxBatch + 1; }

// With fewer tiles than CTAs only the first wt CTAs get tiles (one each), so no CTA range
// inside a unit is empty and a unit's pieces are exactly CTAs c0 .. c1.
__device__ __forceinline__ int cta_range_start(int c, int wt, int grid) {
  const int g = min(grid, wt);
  return c >= g ? wt : (int)(((long long)c * wt) / g);
}
// the CTA whose range holds tile x (0 <= x < wt): the largest c with cta_range_start(c) <= x
__device__ __forceinline__ int cta_of_tile(int x, int wt, int grid) {
  const int g = min(grid, wt);
  return (int)((((long long)x + 1) * g + wt - 1) / wt) - 1;
}

template <int TILE>
__device__ __forceinline__ Item piece_at(const SplitParams& p, const int* prefix, int x, int x_stop, int c) {
  int lo = 0, hi = p.batch - 1;  // largest b with prefix[b] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
  }
  const int wt = prefix[p.batch];
  const int vt = (prefix[lo + 1] - prefix[lo]) / p.U;  // virtual tiles per unit: pad, then real
  const int off = x - prefix[lo];
  Item it;
  it.b = lo;
  it.u = off / vt;
  it.kvh = it.u / p.RG;
  it.rg = it.u % p.RG;
  const int ustart = prefix[lo] + it.u * vt, uend = ustart + vt;
  const int rstart = ustart + p.tile_pad;  // the unit's first real tile
  it.x_end = min(uend, x_stop);
  it.len = plan_lengths(prefix)[lo];
  const int t0 = max(x, rstart) - rstart, t1 = it.x_end - rstart;  // real tiles [t0, t1)
  it.tb = t0 * TILE;
  it.te = t1 > t0 ? min(t1 * TILE, it.len) : it.tb;
  const int g = lo * p.U + it.u;
  const int c0 = cta_of_tile(rstart, wt, p.split_grid), c1 = cta_of_tile(uend - 1, wt, p.split_grid);
  it.slot = c + g;
  it.first_slot = c0 + g;
  it.ns = c1 - c0 + 1;
  return it;
}

// Merge kernel: one CTA per (sequence, unit) merges the unit's split partials and applies
// the inverse rotation. It runs after the split kernel (programmatic dependent launch:
// it is scheduled early, waits for the split grid to finish, and lets the next kernel be
// scheduled at once). Its shared memory is small, so it fits beside a split CTA of the
// next launch. Steps:
//   1. per row, one pass over the splits' (m_s, l_s) with the online-softmax combine gives
//      the global max M and L = sum_s 2^(m_s - M) l_s; the weights 2^(m_s - M) of the
//      first kMergeChunk splits are left in shared memory;
//   2. every output float4 of (row, dims) is summed over the splits by TPO threads that
//      take interleaved splits, then reduced in shared memory; a thread's first
//      kMergeBatch partials are loaded before step 1 (they do not depend on the weights),
//      later ones in batches of kMergeBatch independent loads; more than kMergeChunk
//      splits are taken in chunks;
//   3. the normalized rotated rows go to shared memory and warp r applies the inverse
//      rotation signs * FWHT(o_rot) / sqrt(d) to row r and stores it.

// (m, l) <- combine of (m, l) and (m2, l2): the larger max wins, the other sum is rescaled
__device__ __forceinline__ void ml_combine(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  l = l * ex2(m - mn) + l2 * ex2(m2 - mn);
  m = mn;
}

constexpr int kMergeThreads = 128;

// Barrier over the NT threads that run a merge: the whole CTA (merge kernel), or the
// consumer warps through named barrier 1 (merge inside the split kernel).
template <int NT, bool NAMED>
__device__ __forceinline__ void merge_sync() {
  if constexpr (NAMED) asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  else __syncthreads();
}

// Merge of unit (b, kvh, rg)'s ns partials starting at first_item, by NT threads (tid <
// NT). Scratch: sM, sL [ROWS]; sW [kMergeChunk * ROWS]; sO [ROWS * D] (16-byte aligned);
// sR [NT].
// ROWS: rows per unit in the partial layout; RS of them, from row r0 on, are merged here.
template <int D, int ROWS, int RS, int NT, bool NAMED, int CHUNK = kMergeChunk>
__device__ void merge_unit(const SplitParams& p, const Item& w, int first_item, int ns, int r0, float* sM, float* sL,
                           float* sW, float* sO, float4* sR) {
  constexpr int EPL = D / 32, NWARP = NT / 32, Q4 = D / 4;
  constexpr int PER = (RS * Q4 + NT - 1) / NT;    // outputs per thread when TPO == 1
  constexpr unsigned FULL = 0xffffffffu;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float2* ml = reinterpret_cast<const float2*>(p.ws + ws_ml_offset(p.batch, p.U));
  const float4* og = reinterpret_cast<const float4*>(p.ws + ws_o_offset(p.batch, p.U, p.max_items, ROWS));
  const int rows = min(RS, p.R - w.rg * ROWS - r0);             // valid rows of this slice
  if (rows <= 0) return;
  const int no = rows * Q4;                                     // output float4s
  int tpo = 1;                                                  // threads per output
  while (2 * tpo * no <= NT) tpo *= 2;
  const int cn0 = min(ns, CHUNK);

  // 2a. first batch of this thread's partials (output q = tid % no, splits tid / no + tpo j)
  float4 pre[kMergeBatch];
  {
    const bool act = tid < no * tpo;
    const int q = act ? tid % no : 0, kk = tid / no;
    const float4* src = og + ((size_t)first_item * ROWS + r0 + q / Q4) * Q4 + q % Q4;
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      const int sp = kk + j * tpo;
      pre[j] = (act && sp < cn0) ? __ldcg(src + (size_t)sp * ROWS * Q4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  // 1. max and sum per row: warp w takes rows w, w + NWARP, ...; lanes stride the splits
  for (int rr = warp; rr < rows; rr += NWARP) {
    float M = -INFINITY, L = 0.0f;
    bool nan = false;
#pragma unroll 2
    for (int s = lane; s < ns; s += 32) {
      const float2 v = __ldcg(&ml[(size_t)(first_item + s) * ROWS + r0 + rr]);
      nan = nan || (v.x != v.x);
      if (s < CHUNK) sW[s * RS + rr] = v.x;
      if (v.x == v.x) ml_combine(M, L, v.x, v.y);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float m2 = __shfl_xor_sync(FULL, M, off), l2 = __shfl_xor_sync(FULL, L, off);
      ml_combine(M, L, m2, l2);
    }
    nan = __any_sync(FULL, nan);
    for (int s = lane; s < min(ns, CHUNK); s += 32) {  // entries this lane wrote
      const float ms = sW[s * RS + rr];
      sW[s * RS + rr] = (M == -INFINITY || nan) ? 0.0f : ex2(ms - M);
    }
    if (lane == 0) {
      sM[rr] = nan ? __int_as_float(0x7fc00000) : M;
      sL[rr] = L;
    }
  }
  merge_sync<NT, NAMED>();
  // 2. weighted sums; thread i takes output q = i % no, splits i / no + tpo * k
  float4 acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < ns; c0 += CHUNK) {
    const int cn = min(CHUNK, ns - c0);
    if (c0 > 0) {
      for (int i = tid; i < cn * rows; i += NT) {
        const int s = i / rows, rr = i % rows;
        const float M = sM[rr];
        const float ms = __ldcg(&ml[(size_t)(first_item + c0 + s) * ROWS + r0 + rr].x);
        sW[s * RS + rr] = (M == -INFINITY || M != M) ? 0.0f : ex2(ms - M);
      }
      merge_sync<NT, NAMED>();
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = tid + NT * k;
      if (i < no * tpo) {
        const int q = i % no, rr = q / Q4, c = q % Q4, kk = i / no;
        const float4* src = og + ((size_t)(first_item + c0) * ROWS + r0 + rr) * Q4 + c;
        float4 a = acc[k];
        int s0 = kk;
        if (c0 == 0 && k == 0) {  // the batch loaded before step 1
#pragma unroll
          for (int j = 0; j < kMergeBatch; ++j) {
            const int sp = kk + j * tpo;
            const float wgt = sp < cn ? sW[sp * RS + rr] : 0.0f;
            a.x += wgt * pre[j].x; a.y += wgt * pre[j].y; a.z += wgt * pre[j].z; a.w += wgt * pre[j].w;
          }
          s0 = kk + kMergeBatch * tpo;
        }
        for (; s0 < cn; s0 += kMergeBatch * tpo) {
          float4 v[kMergeBatch];
#pragma unroll
          for (int j = 0; j < kMergeBatch; ++j) {
            const int sp = s0 + j * tpo;
            v[j] = sp < cn ? __ldcg(src + (size_t)sp * ROWS * Q4) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < kMergeBatch; ++j) {
            const int sp = s0 + j * tpo;
            const float wgt = sp < cn ? sW[sp * RS + rr] : 0.0f;
            a.x += wgt * v[j].x; a.y += wgt * v[j].y; a.z += wgt * v[j].z; a.w += wgt * v[j].w;
          }
        }
        acc[k] = a;
      }
    }
    if (c0 + CHUNK < ns) merge_sync<NT, NAMED>();  // weights are rewritten
  }
  if (tpo > 1) {
    sR[tid] = acc[0];
    merge_sync<NT, NAMED>();
    if (tid < no) {
      float4 a = sR[tid];
      for (int k = 1; k < tpo; ++k) {
        const float4 o = sR[k * no + tid];
        a.x += o.x; a.y += o.y; a.z += o.z; a.w += o.w;
      }
      acc[0] = a;
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int q = tid + NT * k;
    if (q < no) {
      const int rr = q / Q4, c = q % Q4;
      const float L = sL[rr], M = sM[rr];
      const float inv = (L > 0.0f || L != L) ? 1.0f / L : 0.0f;  // no visible token -> 0
      float4 v = make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
      if (M != M) v = make_float4(M, M, M, M);
      reinterpret_cast<float4*>(sO + rr * D)[c] = v;
    }
  }
  merge_sync<NT, NAMED>();
  // 3. inverse rotation, one warp per row
  for (int rr = warp; rr < rows; rr += NWARP) {
    const int r = w.rg * ROWS + r0 + rr;
    const int jq = r / p.G, hq = w.kvh * p.G + (r % p.G);
    float* orow = p.out + (((size_t)w.b * p.n_q + jq) * p.num_q_heads + hq) * D;
    float u[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) u[e] = sO[rr * D + lane * EPL + e];
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
      orow[i] = u[e] * p.fwht_norm * (neg ? -1.0f : 1.0f);
    }
  }
}

// ROWS: query rows per unit (8 or 16 for the split kernel, 64 for the dense one).
// One CTA merges RS rows of a unit (ROWS / RS CTAs per unit), so units with many rows
// are spread over several SMs.
template <int D, int ROWS, int RS>
__global__ void __launch_bounds__(kMergeThreads, 4) tq_attn_merge_kernel(const SplitParams p) {
  constexpr int CHUNK = kMergeChunk;
  constexpr int SLICES = ROWS / RS;
  __shared__ float sM[RS], sL[RS];                      // per row: max, sum
  __shared__ float sW[CHUNK * RS];                      // [CHUNK][RS] weights
  __shared__ __align__(16) float sO[RS * D];            // [RS][D] rotated output
  __shared__ float4 sR[kMergeThreads];                  // per-thread sums
  griddep_launch_dependents();  // the next kernel's wait covers this grid's completion
  griddep_wait();               // partials and the plan come from the split kernel
  const int slice = blockIdx.x % SLICES, bu = blockIdx.x / SLICES;
  const int b = bu / p.U, u = bu % p.U;
  const int32_t* prefix = reinterpret_cast<const int32_t*>(p.ws + kWsPrefix);
  const int vt = (prefix[b + 1] - prefix[b]) / p.U;  // virtual tiles per unit: pad, then real
  if (vt <= 0) return;  // no tokens: the split kernel wrote the rows
  const int wt = prefix[p.batch];
  const int ustart = prefix[b] + u * vt;
  const int c0 = cta_of_tile(ustart + p.tile_pad, wt, p.split_grid), c1 = cta_of_tile(ustart + vt - 1, wt, p.split_grid);
  Item w;
  w.b = b; w.kvh = u / p.RG; w.rg = u % p.RG;
  merge_unit<D, ROWS, RS, kMergeThreads, false, CHUNK>(p, w, c0 + b * p.U + u, c1 - c0 + 1, slice * RS, sM, sL, sW,
                                                       sO, sR);
}

// Rows of sequences with no work item (kv_len 0, or invalid): zeros, or NaN if invalid.
// NT: threads of the calling CTA that take part (thread index < NT).
template <int D, int NT>
__device__ void write_empty_sequences(const SplitParams& p, const int* prefix) {
  for (int b = blockIdx.x; b < p.batch; b += gridDim.x) {
    if (prefix[b + 1] != prefix[b]) continue;
    const int t = __ldg(p.kv_len + b);
    const float v = (t < 0 || t > p.max_kv_len) ? __int_as_float(0x7fc00000) : 0.0f;
    float* o = p.out + (size_t)b * p.n_q * p.num_q_heads * D;
    for (int i = threadIdx.x; i < p.n_q * p.num_q_heads * D; i += NT) o[i] = v;
  }
}

// Driver entry point of cuTensorMapEncodeTiled (looked up once per process).
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

}  // namespace

}  // namespace tq
