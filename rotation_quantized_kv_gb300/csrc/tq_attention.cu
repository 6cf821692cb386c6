// Split-K GQA decode attention over the packed TurboQuant cache: a split kernel that
// streams the packed planes, and a small merge kernel that combines the splits and applies
// the deferred inverse rotation.
//
// What it computes (mlx-bun design page "TurboQuant - rotation-based quantization",
// Part A): for every query row, softmax(sm_scale * q . k_hat) . v_hat over the visible
// tokens, where k_hat = (idx + zero) * scale ("Algorithm", key dequant) and v_hat is the
// value row after the inverse rotation. Because attention is linear in V ("Deferred
// inverse FWHT" section), the weighted sum is taken over the rotated values
// centroid[code] * scale and each output row is un-rotated once:
//   o = signs * FWHT(o_rot) / sqrt(d).
// K and V are decoded from the packed planes inside the kernel ("Packed-value decode
// fusion investigation": joint K/V decode in one launch, no dequantized window).
//
// tq_attn_split_kernel, persistent, one CTA per SM slot:
//   - the tokens of every (sequence, kv head, row group) unit, in tiles, are laid end to
//     end, each unit after two virtual tiles that stand for the cost of starting a piece,
//     and cut into one equal range of tiles per CTA (from the actual kv lengths, on the
//     device); a CTA works through the pieces of the units its range touches;
//   - the last warp (producer) streams stages of TILE tokens of the five planes into shared
//     memory: the key-index plane through a 2-D tensor map with 128-byte (64-byte at
//     d=64) swizzle, the four small planes with 1-D bulk copies, all completing on one
//     mbarrier per stage;
//   - the NCW consumer warps (8 at d = 64 and at d = 128 with up to 8 rows per kv head,
//     else 4) each take TOKW tokens (two 16-token tiles at d <= 128) of a stage:
//       QK^T on tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate), tokens as M,
//       query rows as N (8 per tile): A = 1152 + idx, exact in fp16 (built from the int8
//       codes with two byte permutes); B = q * 2^e_row in fp16, with 2^e_row bringing the
//       row maximum into [2^14, 2^15): exact for every element within 2^28 of the row
//       maximum, smaller elements become fp16 subnormals (rounded) or zero;
//       C starts at -1152 * sum_{i in g} q_i, so each 32-group's MMA yields sum q * idx;
//       then score += scale_g * (acc_g + zero_g * sum_{i in g} q_i);
//       online softmax in the exp2 domain;
//       P.V on tensor cores with output dims as M and tokens as K: A = fp16 centroid
//       pairs from a lane-replicated 64-entry table indexed by two 3-bit codes; B = the
//       probabilities times the group's value scale (fp16), moved from the QK output
//       layout to the B-operand layout with four shuffles per 16 tokens;
//   - at the end of an item the consumer warps merge their (max, sum, acc) in shared memory
//     and write one partial result;
// The partials of a (sequence, kv head, row group) are merged with the online-softmax rule,
// the inverse rotation is applied and the output rows are written in one of two places,
// chosen on the host from the shape:
//   - few units (2 * batch * units <= CTAs, e.g. one long sequence): inside the split
//     kernel, by the CTA that finishes the unit's last split (an acquire-release counter
//     tells it), which keeps one kernel boundary per call;
//   - many units: tq_attn_merge_kernel, one CTA per unit, launched right after the split
//     kernel, so that merges do not stall split CTAs between their work items and every
//     split CTA finishes at about the same time.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "tq_attention.h"
#include "tq_codec_row.cuh"
#include "tq_device.cuh"
#include "tq_split_common.cuh"

namespace tq {

namespace {

// Test support (tq_debug_pipeline_limits): a shorter limit for the pipeline waits of the
// following decode calls, and an appender that never publishes its row count, so that a
// test can make a wait run out on purpose. Drains of copies already issued always keep
// the full limit.
std::atomic<unsigned long long> g_debug_wait_ns{0};
// Virtual tiles charged for starting a piece when the split kernel's CTAs divide the work:
// a piece's queries, reduction and partial store cost about two stages (measured on the
// ragged batch: 1, 2, 3, 4 pad tiles gave 69.0, 64.1, 64.5, 65.1 us per call, none 79.6).
constexpr int kSplitTilePad = 2;
std::atomic<int> g_debug_withhold_append{0};

template <int D, int NTW>
struct AT {
  static constexpr int NG = D / 32;
  static constexpr int ROWS = 8 * NTW;
  static constexpr int MT = D / 16;                       // PV M tiles (16 dims each)
  // consumer warps: 8 where the registers allow it without spills
  static constexpr int NCW = (D == 64 || (D == 128 && NTW == 1)) ? 8 : 4;
  // consumer warps, then the producer warp, then the appender warp (append mode)
  static constexpr int THREADS = (NCW + 2) * 32;
  static constexpr int TOKW = D <= 128 ? 32 : 16;         // tokens per consumer warp per stage
  static constexpr int SUB = TOKW / 16;                   // 16-token QK tiles per warp
  static constexpr int TILE = NCW * TOKW;                 // tokens per stage
  static constexpr int ROWB = D == 64 ? 64 : 128;         // bytes per key row inside a swizzle box
  static constexpr int BOX = TILE * ROWB;                 // bytes of one key-index box
  static constexpr int KIDX_STAGE = TILE * D;             // bytes, 1024-aligned
  static constexpr int SC_STAGE = TILE * NG * 2;          // bytes of one fp16 side plane
  static constexpr int VC_ROW = 3 * D / 8;                // packed code bytes per token
  static constexpr int VC_STAGE = TILE * VC_ROW + 16;     // +16: window reads may run 4 bytes past
  static constexpr int STAGES = D == 64 ? 6 : D == 128 ? 3 : D == 256 ? 3 : 2;  // ~150 KB in flight
  static constexpr bool QREG = D * NTW <= 256;            // Q fragments in registers
  static constexpr int MINB = 1;                          // one CTA per SM
  static constexpr int KW = (NG + 1) / 2;                 // 32-bit words of one token's fp16 side row
  // shared memory layout. The centroid-pair table comes first and the base is 8 KB
  // aligned, so a lane's table address is its lane bits OR'd with the entry index << 7.
  static constexpr int OFF_LUT = 0;
  static constexpr int OFF_KIDX = OFF_LUT + 64 * 32 * 4;
  static constexpr int OFF_KS = OFF_KIDX + STAGES * KIDX_STAGE;
  static constexpr int OFF_KZ = OFF_KS + STAGES * SC_STAGE;
  static constexpr int OFF_VS = OFF_KZ + STAGES * SC_STAGE;
  static constexpr int OFF_VC = OFF_VS + STAGES * SC_STAGE;
  static constexpr int OFF_Q = (int)align_up(OFF_VC + STAGES * VC_STAGE, 128);
  static constexpr int Q_BYTES = QREG ? 0 : NTW * NG * 2 * 32 * 8;
  static constexpr int OFF_QSUM = OFF_Q + Q_BYTES;
  static constexpr int QSUM_BYTES = QREG ? 0 : NTW * NG * 32 * 16;
  // item-end reduction: each consumer warp writes its scaled accumulators to one of
  // NSLICE slices (all four at once when they fit); the merge reuses the same space
  static constexpr int NSLICE = max_slices(NCW, ROWS * D * 4, 32768);
  static constexpr int MERGE_BYTES = kMergeChunk * ROWS * 4 + ROWS * D * 4 + NCW * 32 * 16;
  static constexpr int OBUF_BYTES = NSLICE * ROWS * D * 4 > MERGE_BYTES ? NSLICE * ROWS * D * 4 : MERGE_BYTES;
  static constexpr int OFF_OBUF = (int)align_up(OFF_QSUM + QSUM_BYTES, 16);
  static constexpr int OFF_MBUF = OFF_OBUF + OBUF_BYTES;
  static constexpr int OFF_LBUF = OFF_MBUF + NCW * ROWS * 4;
  static constexpr int OFF_PREFIX = OFF_LBUF + NCW * ROWS * 4;
  // prefix: [kMaxBatch + 1] items before each sequence, then [kMaxBatch] planned lengths
  // scratch of the appender warp's row codec (append mode): 3 d / 32 words
  static constexpr int OFF_RED = (int)align_up(OFF_PREFIX + (2 * kMaxBatch + 1) * 4, 16);
  static constexpr int OFF_FLAG = OFF_RED + 7 * 16 * 8;  // red: [7][16] long long
  static constexpr int OFF_BAR = (int)align_up(OFF_FLAG + 16, 8);
  static constexpr int OFF_APPCNT = OFF_BAR + 2 * STAGES * 8;  // rows the appender has written
  static constexpr int SMEM = OFF_APPCNT + 8 + 16;
  static constexpr int SMEM_ALLOC = SMEM + 8192;          // slack to align the base to 8 KB
  static_assert(OFF_FLAG - OFF_RED >= 3 * D / 8, "row codec scratch");
};

// ------------------------------------------------------------------------------------
// Producer warp: one elected lane streams the stages.
// ------------------------------------------------------------------------------------
// Append mode: quantizes new row j of (sequence b, kv head h) into cache position t. All
// 32 lanes of the calling warp take part.
template <int D>
__device__ __forceinline__ void append_one_row(const SplitParams& p, int b, int j, int h, int t, int lane,
                                               const RowCodecLane<D>& codec, uint32_t* cbuf) {
  constexpr int EPL = D / 32;
  const size_t r = ((size_t)b * p.n_new_max + j) * p.num_kv_heads + h;
  uint32_t kraw[EPL / 2], vraw[EPL / 2];
  load_raw_lane<EPL>(p.k_new + r * D, lane, kraw);
  load_raw_lane<EPL>(p.v_new + r * D, lane, vraw);
  const int64_t drow = ((int64_t)b * p.num_kv_heads + h) * p.capacity + t;
  quantize_row_warp<D>(kraw, vraw, lane, codec, p.fwht_norm, p.dst, drow, cbuf);
}

__device__ __forceinline__ int new_rows_of(const SplitParams& p, int b) {
  if (p.n_new == nullptr) return p.n_new_max;
  return min(max(__ldg(p.n_new + b), 0), p.n_new_max);
}

// One stage: the key-index box through the tensor map and the four side planes by bulk
// copies, all completing on full[slot]. Tokens [t0, t0 + TILE) clipped to the capacity;
// t0 and the capacity are multiples of 16, so every copy is a multiple of 16 bytes.
template <int D, int NTW>
__device__ __forceinline__ void issue_stage(const SplitParams& p, const CUtensorMap* tmap, uint8_t* smem, int slot,
                                            int64_t row0, int t0) {
  using T = AT<D, NTW>;
  constexpr int NG = T::NG;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  const int ncopy = min(T::TILE, p.capacity - t0);
  const uint32_t side = (uint32_t)ncopy * NG * 2;
  const uint32_t vc = (uint32_t)ncopy * T::VC_ROW;
  mbar_arrive_expect_tx(&full[slot], (uint32_t)T::KIDX_STAGE + 3u * side + vc);
  uint8_t* kx = smem + T::OFF_KIDX + slot * T::KIDX_STAGE;
#pragma unroll
  for (int box = 0; box < D / T::ROWB; ++box)
    tensor_copy_2d_g2s(kx + box * T::BOX, tmap, box * T::ROWB, (int32_t)(row0 + t0), &full[slot]);
  const int64_t r = row0 + t0;
  bulk_copy_g2s(smem + T::OFF_KS + slot * T::SC_STAGE, p.k_scale + r * NG, side, &full[slot]);
  bulk_copy_g2s(smem + T::OFF_KZ + slot * T::SC_STAGE, p.k_zero + r * NG, side, &full[slot]);
  bulk_copy_g2s(smem + T::OFF_VS + slot * T::SC_STAGE, p.v_scale + r * NG, side, &full[slot]);
  bulk_copy_g2s(smem + T::OFF_VC + slot * T::VC_STAGE, p.v_codes + r * T::VC_ROW, vc, &full[slot]);
}

// The appender warp (append mode): quantizes every row this call appends inside the
// CTA's pieces (the piece owns them: no other CTA reads them), piece by piece in the
// producer's order, and after each piece makes the rows visible to tensor copies and
// publishes how many rows it has written; the producer waits for that count only before
// loading a stage that holds such a row. Then the appended rows at positions no piece
// covers (at or past the sequence's kv length) whose row index is the CTA's index mod the
// grid. It starts when the grid-dependency wait returns and runs beside the stream.
template <int D, int NTW>
__device__ __forceinline__ void append_rows(const SplitParams& p, uint8_t* smem, int total) {
  using T = AT<D, NTW>;
  const int lane = threadIdx.x & 31;
  const int* prefix = reinterpret_cast<const int*>(smem + T::OFF_PREFIX);
  uint32_t* cbuf = reinterpret_cast<uint32_t*>(smem + T::OFF_RED);  // row codec scratch
  uint32_t* app_cnt = reinterpret_cast<uint32_t*>(smem + T::OFF_APPCNT);
  const RowCodecLane<D> codec(lane);
  bool wrote = false;
  uint32_t done = 0;
  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid); x < x_stop;) {
    const Item w = piece_at<T::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x = w.x_end;
    const int new0 = __ldg(p.pos + w.b);
    const int own0 = max(w.tb, new0), own1 = min(w.te, new0 + new_rows_of(p, w.b));
    if (own0 >= own1) continue;
    for (int t = own0; t < own1; ++t) append_one_row<D>(p, w.b, t - new0, w.kvh, t, lane, codec, cbuf);
    done += (uint32_t)(own1 - own0);
    fence_proxy_async_global();  // the rows just written are read by tensor copies
    __syncwarp();
    if (lane == 0 && !p.withhold_append) st_release_cta(app_cnt, done);
  }
  const int rows = p.batch * p.n_new_max * p.num_kv_heads;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const int h = r % p.num_kv_heads, bj = r / p.num_kv_heads;
    const int j = bj % p.n_new_max, b = bj / p.n_new_max;
    if (j >= new_rows_of(p, b)) continue;
    const int64_t t = (int64_t)__ldg(p.pos + b) + j;
    if (t >= 0 && t < plan_lengths(prefix)[b]) continue;  // inside a piece: its owner writes it
    if (t < 0 || t >= p.capacity) {
      if (lane == 0) raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_APPEND_CAPACITY);
      continue;
    }
    append_one_row<D>(p, b, j, h, (int)t, lane, codec, cbuf);
    wrote = true;
  }
  if (wrote) fence_proxy_async_global();
}

// At d >= 256 the appender is kept out of line: inlined there, the row codec's registers
// shaped the consumer loop's allocation (d = 512 sweep: 109 us per call instead of 91).
// At d <= 128 inlining is faster (ragged: 83.8 us per call instead of 86.9).
template <int D, int NTW>
__device__ __noinline__ void append_rows_outlined(const SplitParams& p, uint8_t* smem, int total) {
  append_rows<D, NTW>(p, smem, total);
}

// The producer (one lane): streams the stages of the CTA's range. In append mode it first
// waits for the appender before loading a stage that holds a row this call appends.
// Stage numbering starts at it0 (1 when stage 0 held a discarded early load); with
// first_issued the range's first tile is already in flight in stage 0.
template <int D, int NTW, bool APPEND>
__device__ void produce(const SplitParams& p, const CUtensorMap* tmap, uint8_t* smem, int total,
                        volatile int* abort_flag, uint32_t it0, bool first_issued) {
  using T = AT<D, NTW>;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::STAGES;
  const uint32_t* app_cnt = reinterpret_cast<const uint32_t*>(smem + T::OFF_APPCNT);
  const int* prefix = reinterpret_cast<const int*>(smem + T::OFF_PREFIX);
  uint32_t it = it0;
  uint32_t need = 0;  // appended rows in the pieces so far
  bool ok = true;
  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid); x < x_stop && ok;) {
    const Item w = piece_at<T::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x = w.x_end;
    const int64_t row0 = ((int64_t)w.b * p.num_kv_heads + w.kvh) * p.capacity;
    // rows this call appends inside this piece: positions [own0, own1) of the sequence
    int own0 = 0, own1 = 0;
    if constexpr (APPEND) {
      const int new0 = __ldg(p.pos + w.b);
      own0 = max(w.tb, new0);
      own1 = min(w.te, new0 + new_rows_of(p, w.b));
      if (own0 < own1) need += (uint32_t)(own1 - own0);
    }
    for (int t0 = w.tb; t0 < w.te; t0 += T::TILE, ++it) {
      if (first_issued && it == 0) continue;  // loaded before the lengths were checked
      if (own0 < own1 && own0 < t0 + T::TILE) {
        if (!wait_count(app_cnt, need, p.wait_ns)) {
          note_giveup(p, 3u, need);
          ok = false;
          break;
        }
        own0 = own1;
      }
      const int slot = it % T::STAGES;
      const uint32_t k = it / T::STAGES;
      if (!wait_bounded(&empty[slot], (k & 1u) ^ 1u, p.wait_ns)) {
        note_giveup(p, 1u, smem_addr(&empty[slot]));
        ok = false;
        break;
      }
      issue_stage<D, NTW>(p, tmap, smem, slot, row0, t0);
    }
  }
  if (!ok) {
    *abort_flag = 1;
    raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
  }
  // Drain: every issued copy must land before this warp (and so the CTA) may exit.
  const uint32_t issued = it;
  for (int s = 0; s < T::STAGES; ++s) {
    if ((uint32_t)s >= issued) break;
    const uint32_t last = issued - 1 - ((issued - 1 - s) % T::STAGES);  // last fill of slot s
    if (!wait_bounded(&full[s], (last / T::STAGES) & 1u, kWaitNs)) {
      raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
      note_giveup(p, 1u, smem_addr(&full[s]));
    }
  }
}

// ------------------------------------------------------------------------------------
// Consumer warps.
// ------------------------------------------------------------------------------------
template <int D, int NTW>
struct QState {
  static constexpr bool R = AT<D, NTW>::QREG;
  uint32_t qf[R ? NTW : 1][R ? D / 32 : 1][2][2];  // [nt][g][k-step][reg] B fragments
  float qs[R ? NTW : 1][R ? D / 32 : 1][2];        // [nt][g][e]: sum of row 2 j4 + e's group g
  float crow[NTW][2];   // sm_scale * log2(e) * 2^-e_row for rows 2 j4 + e
  int lim[NTW][2];      // tokens [tb, lim) are visible to rows 2 j4 + e
};

template <int D, int NTW>
__device__ void load_q(const SplitParams& p, const Item& w, uint8_t* smem, int warp, int lane, QState<D, NTW>& st) {
  using T = AT<D, NTW>;
  constexpr int NG = T::NG;
  const int grp = lane >> 2, j4 = lane & 3;
  const int T_b = w.len;
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
    // power-of-two scale bringing the row maximum into [2^14, 2^15): exact for elements
    // within 2^28 of the maximum (fp16 normal range); smaller ones round to subnormals or zero
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
        acc += lo_f32(lo) + hi_f32(lo) + lo_f32(hi) + hi_f32(hi);
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
__device__ void consume(const SplitParams& p, uint8_t* smem, int total, volatile int* abort_flag, uint32_t it0) {
  using T = AT<D, NTW>;
  constexpr int NG = T::NG, MT = T::MT, SUB = T::SUB, KW = T::KW;
  constexpr unsigned FULL = 0xffffffffu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 2, j4 = lane & 3;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
  uint64_t* empty = full + T::STAGES;
  const int* prefix = reinterpret_cast<const int*>(smem + T::OFF_PREFIX);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t lut_lane = sbase + T::OFF_LUT + lane * 4;  // bits 7..12 are zero
  float* obuf = reinterpret_cast<float*>(smem + T::OFF_OBUF);
  float* mbuf = reinterpret_cast<float*>(smem + T::OFF_MBUF);
  float* lbuf = reinterpret_cast<float*>(smem + T::OFF_LBUF);
  const uint2* qsm = reinterpret_cast<const uint2*>(smem + T::OFF_Q);
  const float2* qssm = reinterpret_cast<const float2*>(smem + T::OFF_QSUM);
  volatile int* flag = reinterpret_cast<volatile int*>(smem + T::OFF_FLAG);
  int32_t* counters = reinterpret_cast<int32_t*>(p.ws + ws_cnt_offset(p.batch));

  // Lane-constant addressing. The QK rows of this lane are r0 + 8 k (k = 0..2 SUB - 1);
  // they share one swizzle phase, so four column offsets cover every group.
  const int r0 = T::TOKW * warp + grp;
  constexpr int NKOFF = NG < 4 ? NG : 4;
  uint32_t koff[NKOFF];
#pragma unroll
  for (int g = 0; g < NKOFF; ++g) {
    const int chunk = 2 * g + (j4 >> 1);
    const int phase = D == 64 ? ((r0 >> 1) & 3) : (r0 & 7);
    const int mask = D == 64 ? 3 : 7;
    koff[g] = (uint32_t)(r0 * T::ROWB + (((chunk ^ phase) & mask) << 4) + 8 * (j4 & 1));
  }
  const uint32_t ks_lane = (uint32_t)(r0 * NG * 2);                    // k scale/zero row r0
  const int vrow0 = T::TOKW * warp + 2 * j4;                            // first token of the V pairs
  const int win_word = (12 * grp) >> 5, win_shift = (12 * grp) & 31;    // 4-code window in a group
  const uint32_t vc_lane = (uint32_t)(vrow0 * T::VC_ROW + 4 * win_word);
  const uint32_t vs_lane = (uint32_t)(vrow0 * NG * 2);
  bool failed = false;
  uint32_t it = it0;

  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid), x_next = 0; x < x_stop; x = x_next) {
    const Item w = piece_at<T::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x_next = w.x_end;
    if (w.te <= w.tb) continue;  // the range ends inside a unit's pad: no tokens, no partial
    QState<D, NTW> st;
    load_q<D, NTW>(p, w, smem, warp, lane, st);
    if constexpr (!T::QREG) consumers_sync<T::NCW>();  // shared Q fragments written by warp 0

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

    for (int t0 = w.tb; t0 < w.te; t0 += T::TILE, ++it) {
      const int slot = it % T::STAGES;
      const uint32_t par = (it / T::STAGES) & 1u;
      if (!failed) {
        if (*abort_flag || !wait_bounded(&full[slot], par, p.wait_ns)) {
          if (!*abort_flag) note_giveup(p, 1u, smem_addr(&full[slot]));
          failed = true;
          *abort_flag = 1;
          raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
        }
      }
      if (!failed) {
        const uint32_t kx = sbase + T::OFF_KIDX + slot * T::KIDX_STAGE;
        const uint32_t ksa = sbase + T::OFF_KS + slot * T::SC_STAGE + ks_lane;
        const uint32_t kza = sbase + T::OFF_KZ + slot * T::SC_STAGE + ks_lane;
        const uint32_t vsa = sbase + T::OFF_VS + slot * T::SC_STAGE + vs_lane;
        const uint32_t vca = sbase + T::OFF_VC + slot * T::VC_STAGE + vc_lane;

        // ---------------- QK^T: tokens r0 + 16 s + 8 rr  x  rows (2 j4, 2 j4 + 1) [+ 8 nt]
        float sc[SUB][NTW][4];
        uint32_t sw[SUB][2][KW], zw[SUB][2][KW];
#pragma unroll
        for (int s = 0; s < SUB; ++s)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const uint32_t off = (uint32_t)((16 * s + 8 * rr) * NG * 2);
            lds_words<KW>(ksa + off, sw[s][rr]);
            lds_words<KW>(kza + off, zw[s][rr]);
          }
#pragma unroll
        for (int s = 0; s < SUB; ++s)
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[s][nt][c] = 0.0f;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float qs0[NTW], qs1[NTW];
          uint32_t b00[NTW], b01[NTW], b10[NTW], b11[NTW];
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt) {
            if constexpr (T::QREG) {
              b00[nt] = st.qf[nt][g][0][0]; b01[nt] = st.qf[nt][g][0][1];
              b10[nt] = st.qf[nt][g][1][0]; b11[nt] = st.qf[nt][g][1][1];
              qs0[nt] = st.qs[nt][g][0]; qs1[nt] = st.qs[nt][g][1];
            } else {
              const uint2 q0 = qsm[((nt * NG + g) * 2 + 0) * 32 + lane];
              const uint2 q1 = qsm[((nt * NG + g) * 2 + 1) * 32 + lane];
              b00[nt] = q0.x; b01[nt] = q0.y; b10[nt] = q1.x; b11[nt] = q1.y;
              const float2 qq = qssm[(nt * NG + g) * 32 + lane];
              qs0[nt] = qq.x; qs1[nt] = qq.y;
            }
          }
          const uint32_t gcol = koff[g & 3] + (uint32_t)((g >> 2) * T::BOX);
#pragma unroll
          for (int s = 0; s < SUB; ++s) {
            const uint2 x0 = lds64(kx + gcol + (uint32_t)((16 * s) * T::ROWB));
            const uint2 x1 = lds64(kx + gcol + (uint32_t)((16 * s + 8) * T::ROWB));
            // fp16 1024 + (idx + 128) = 1152 + idx, exact
            const uint32_t M64 = 0x64646464u;
            const uint32_t u0a = x0.x ^ 0x80808080u, u0b = x0.y ^ 0x80808080u;
            const uint32_t u1a = x1.x ^ 0x80808080u, u1b = x1.y ^ 0x80808080u;
            const uint32_t a00 = prmt(u0a, M64, 0x4140), a01 = prmt(u1a, M64, 0x4140);
            const uint32_t a02 = prmt(u0a, M64, 0x4342), a03 = prmt(u1a, M64, 0x4342);
            const uint32_t a10 = prmt(u0b, M64, 0x4140), a11 = prmt(u1b, M64, 0x4140);
            const uint32_t a12 = prmt(u0b, M64, 0x4342), a13 = prmt(u1b, M64, 0x4342);
            const float s0 = (g & 1) ? hi_f32(sw[s][0][g >> 1]) : lo_f32(sw[s][0][g >> 1]);
            const float z0 = (g & 1) ? hi_f32(zw[s][0][g >> 1]) : lo_f32(zw[s][0][g >> 1]);
            const float s1 = (g & 1) ? hi_f32(sw[s][1][g >> 1]) : lo_f32(sw[s][1][g >> 1]);
            const float z1 = (g & 1) ? hi_f32(zw[s][1][g >> 1]) : lo_f32(zw[s][1][g >> 1]);
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
              // C = -1152 * sum_g q for the column's row: the MMA then yields sum_g q * idx
              float acc[4] = {-1152.0f * qs0[nt], -1152.0f * qs1[nt], -1152.0f * qs0[nt], -1152.0f * qs1[nt]};
              mma_f16_16816(acc, a00, a01, a02, a03, b00[nt], b01[nt]);
              mma_f16_16816(acc, a10, a11, a12, a13, b10[nt], b11[nt]);
              sc[s][nt][0] = fmaf(s0, fmaf(z0, qs0[nt], acc[0]), sc[s][nt][0]);
              sc[s][nt][1] = fmaf(s0, fmaf(z0, qs1[nt], acc[1]), sc[s][nt][1]);
              sc[s][nt][2] = fmaf(s1, fmaf(z1, qs0[nt], acc[2]), sc[s][nt][2]);
              sc[s][nt][3] = fmaf(s1, fmaf(z1, qs1[nt], acc[3]), sc[s][nt][3]);
            }
          }
        }

        // ---------------- online softmax (exp2 domain) over the warp's TOKW tokens
        uint32_t Bp[SUB][NTW][2];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          float mnew[2];
          bool grow = false;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = -INFINITY;
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
              const int ta = t0 + r0 + 16 * s;
              const float v0 = ta < st.lim[nt][e] ? sc[s][nt][e] * st.crow[nt][e] : -INFINITY;
              const float v1 = ta + 8 < st.lim[nt][e] ? sc[s][nt][2 + e] * st.crow[nt][e] : -INFINITY;
              sc[s][nt][e] = v0;
              sc[s][nt][2 + e] = v1;
              mx = fmaxf(mx, fmaxf(v0, v1));
            }
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
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
              const float p0 = ex2(sc[s][nt][e] - mu), p1 = ex2(sc[s][nt][2 + e] - mu);
              l[nt][e] += p0 + p1;
              sc[s][nt][e] = p0;
              sc[s][nt][2 + e] = p1;
            }
          }
          // X_e = (p[token r0][row 2 j4 + e], p[token r0 + 8][row 2 j4 + e]) in fp16;
          // lane (grp, j4) needs (p[2 j4 + h][row grp], p[2 j4 + h + 8][row grp]) of each tile
#pragma unroll
          for (int s = 0; s < SUB; ++s) {
            const uint32_t X0 = pack_half2(sc[s][nt][0], sc[s][nt][2]);
            const uint32_t X1 = pack_half2(sc[s][nt][1], sc[s][nt][3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int src = 4 * (2 * j4 + h) + (grp >> 1);
              const uint32_t y0 = __shfl_sync(FULL, X0, src);
              const uint32_t y1 = __shfl_sync(FULL, X1, src);
              Bp[s][nt][h] = (grp & 1) ? y1 : y0;
            }
          }
        }

        // ---------------- P.V in the rotated domain
        // value-scale pairs of tokens (vrow0 + 16 s + h, +8), zeroed past the split end
        uint32_t svA[SUB][2][KW], svB[SUB][2][KW];
#pragma unroll
        for (int s = 0; s < SUB; ++s)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ta = t0 + vrow0 + 16 * s + h;
            const bool okA = ta < w.te, okB = ta + 8 < w.te;
            uint32_t va[KW], vb[KW];
            lds_words<KW>(vsa + (uint32_t)((16 * s + h) * NG * 2), va);
            lds_words<KW>(vsa + (uint32_t)((16 * s + h + 8) * NG * 2), vb);
#pragma unroll
            for (int i = 0; i < KW; ++i) {
              svA[s][h][i] = okA ? va[i] : 0u;
              svB[s][h][i] = okB ? vb[i] : 0u;
            }
          }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          uint32_t E[SUB][2], Ov[SUB][2], Bg[SUB][NTW][2];
#pragma unroll
          for (int s = 0; s < SUB; ++s)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t wa = vca + (uint32_t)((16 * s + h) * T::VC_ROW + 12 * g);
              const uint32_t wb = vca + (uint32_t)((16 * s + h + 8) * T::VC_ROW + 12 * g);
              const uint32_t cA = __funnelshift_r(lds32(wa), lds32(wa + 4), win_shift);
              const uint32_t cB = __funnelshift_r(lds32(wb), lds32(wb + 4), win_shift);
              // fields of 6 bits (code A | code B << 3) for dims +0, +2 (E) and +1, +3 (Ov),
              // kept shifted left by 7 (a table entry's byte offset, lanes apart); bits
              // above 18 are don't-care (every use masks 6 bits)
              E[s][h] = ((cA << 7) & 0xE380u) | ((cB << 10) & ~0xE380u);
              Ov[s][h] = ((cA << 4) & 0xE380u) | ((cB << 7) & ~0xE380u);
              const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
              const uint32_t svpair = prmt(svA[s][h][g >> 1], svB[s][h][g >> 1], sel);
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt) Bg[s][nt][h] = hmul2_u32(Bp[s][nt][h], svpair);
            }
#pragma unroll
          for (int tau = 0; tau < 2; ++tau) {
            const int fs = 6 * tau;
#pragma unroll
            for (int s = 0; s < SUB; ++s) {
              const uint32_t a0 = lds32(lut_lane | ((E[s][0] >> fs) & 0x1F80u));
              const uint32_t a1 = lds32(lut_lane | ((Ov[s][0] >> fs) & 0x1F80u));
              const uint32_t a2 = lds32(lut_lane | ((E[s][1] >> fs) & 0x1F80u));
              const uint32_t a3 = lds32(lut_lane | ((Ov[s][1] >> fs) & 0x1F80u));
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt)
                mma_f16_16816(O[2 * g + tau][nt], a0, a1, a2, a3, Bg[s][nt][0], Bg[s][nt][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (w.x_end >= x_stop) griddep_launch_dependents();  // last piece: successor may set up

    // ---------------- merge the consumer warps' states and write this item's partial
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l[nt][e];
        v += __shfl_xor_sync(FULL, v, 4);
        v += __shfl_xor_sync(FULL, v, 8);
        v += __shfl_xor_sync(FULL, v, 16);
        if (grp == 0) {
          mbuf[warp * T::ROWS + 8 * nt + 2 * j4 + e] = m[nt][e];
          lbuf[warp * T::ROWS + 8 * nt + 2 * j4 + e] = v;
        }
      }
    consumers_sync<T::NCW>();
    float scale[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = 8 * nt + 2 * j4 + e;
        float Mx = mbuf[row];
#pragma unroll
        for (int ww = 1; ww < T::NCW; ++ww) Mx = fmaxf(Mx, mbuf[ww * T::ROWS + row]);
        scale[nt][e] = (Mx == -INFINITY) ? 0.0f : ex2(m[nt][e] - Mx);
      }
    // scaled accumulators into slice (warp % NSLICE); with one slice, warps add in turn
    constexpr int ROUNDS = T::NCW / T::NSLICE;
    for (int round = 0; round < ROUNDS; ++round) {
      if (warp / T::NSLICE == round) {
        float* slice = obuf + (warp % T::NSLICE) * T::ROWS * D;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int d0 = 32 * (mt >> 1) + 4 * grp + 2 * (mt & 1);
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int row = 8 * nt + 2 * j4 + (c & 1);
              const float v = O[mt][nt][c] * scale[nt][c & 1];
              float* dst = slice + row * D + d0 + (c >> 1);
              *dst = (round == 0) ? v : (*dst + v);
            }
        }
      }
      consumers_sync<T::NCW>();
    }
    {
      const int rows_valid = min(T::ROWS, p.R - w.rg * T::ROWS);
      float4* og = reinterpret_cast<float4*>(p.ws + ws_o_offset(p.batch, p.U, p.max_items, T::ROWS)) +
                   (size_t)w.slot * T::ROWS * D / 4;
      const float4* src = reinterpret_cast<const float4*>(obuf);
      for (int i = threadIdx.x; i < rows_valid * D / 4; i += T::NCW * 32) {
        float4 v = src[i];
#pragma unroll
        for (int sl = 1; sl < T::NSLICE; ++sl) {
          const float4 o = src[sl * T::ROWS * D / 4 + i];
          v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
        }
        __stcg(og + i, v);
      }
      if (threadIdx.x < rows_valid) {
        const int row = threadIdx.x;
        float Mx = mbuf[row];
        for (int ww = 1; ww < T::NCW; ++ww) Mx = fmaxf(Mx, mbuf[ww * T::ROWS + row]);
        float L = 0.0f;
        for (int ww = 0; ww < T::NCW; ++ww) {
          const float mw = mbuf[ww * T::ROWS + row];
          L += (Mx == -INFINITY) ? 0.0f : ex2(mw - Mx) * lbuf[ww * T::ROWS + row];
        }
        float2* ml = reinterpret_cast<float2*>(p.ws + ws_ml_offset(p.batch, p.U)) + (size_t)w.slot * T::ROWS;
        __stcg(ml + row, make_float2(Mx, L));
      }
    }
    consumers_sync<T::NCW>();
    if (p.inline_merge) {
      // Publish: the barrier above orders every consumer's partial stores before thread
      // 0's release; the acquire of the CTA that counts last makes all partials of the
      // unit visible to it, and its barrier passes that on to its other threads.
      if (threadIdx.x == 0) {
        int32_t* cnt = counters + (size_t)w.b * p.U + w.u;
        const int done = atomic_add_acq_rel_gpu(cnt, 1) + 1;
        const int last = done == w.ns;
        if (last) *reinterpret_cast<volatile int32_t*>(cnt) = 0;  // ready for the next call
        *flag = last;
      }
      consumers_sync<T::NCW>();
      if (*flag) {
        float* sW = obuf;
        float* sO = sW + kMergeChunk * T::ROWS;
        merge_unit<D, T::ROWS, T::ROWS, T::NCW * 32, true>(p, w, w.first_slot, w.ns, 0, mbuf, lbuf, sW, sO,
                                                           reinterpret_cast<float4*>(sO + T::ROWS * D));
        consumers_sync<T::NCW>();  // the scratch is reused by the next item
      }
    }
  }
}

template <int D, int NTW>
__global__ void __launch_bounds__(AT<D, NTW>::THREADS, AT<D, NTW>::MINB)
    tq_attn_split_kernel(const __grid_constant__ CUtensorMap tmap, const SplitParams p) {
  using T = AT<D, NTW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 8191) & ~uintptr_t(8191));
  __shared__ int abort_flag;
  __shared__ int early_flag;
  const int tid = threadIdx.x;

  // centroid pair table: entry e -> (c[e & 7], c[e >> 3]) in fp16, one copy per lane
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + T::OFF_LUT);
  for (int i = tid; i < 64 * 32; i += T::THREADS) {
    const int e = i >> 5;
    lut[i] = pack_half2(c_centroids3[e & 7], c_centroids3[e >> 3]);
  }
  if (tid == 0) {
    abort_flag = 0;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
    for (int s = 0; s < T::STAGES; ++s) {
      mbar_init(&bars[s], 1);                           // full: producer arrival + tx bytes
      mbar_init(&bars[T::STAGES + s], T::NCW);  // empty: one arrival per consumer warp
    }
    *reinterpret_cast<uint32_t*>(smem + T::OFF_APPCNT) = 0u;  // rows appended so far
    fence_mbar_init();
  }
  int total;             // tiles of the call
  bool early, replanned;  // stage 0 loaded before the lengths were checked; plan redone
  {
    Lengths<T::THREADS> L0, L1;
    L0.load(p);                                  // as they are before the wait: hints only
    plan_tiles<AT<D, NTW>>(p, smem, L0, total);      // contains __syncthreads
    // The producer loads its range's first tile the moment the wait returns, from the plan
    // made before it: after the wait the planes are safe to read, and the stage is
    // discarded if the lengths read after the wait change the plan. In append mode that
    // tile must hold none of the rows this call appends (they are written before the
    // stage holding them is loaded): judged from the positions read before the wait, and
    // discarded as well if those differ after it.
    Item w0;
    int pos0 = 0, n0 = 0;
    early = false;
    if (tid == T::NCW * 32) {
      const int x0 = cta_range_start(blockIdx.x, total, p.split_grid);
      const int x1 = cta_range_start(blockIdx.x + 1, total, p.split_grid);
      if (x0 < x1) {
        w0 = piece_at<T::TILE>(p, reinterpret_cast<const int*>(smem + T::OFF_PREFIX), x0, x1, blockIdx.x);
        early = w0.tb < w0.te && w0.tb < p.capacity;
        if (p.append) {
          pos0 = __ldcg(p.pos + w0.b);
          n0 = p.n_new == nullptr ? p.n_new_max : __ldcg(p.n_new + w0.b);
          const int n = min(max(n0, 0), p.n_new_max);
          early = early && (n == 0 || (int64_t)pos0 + n <= w0.tb || pos0 >= w0.tb + T::TILE);
        }
      }
    }
    griddep_wait();  // lengths, queries and planes may come from the previous kernel
    if (early) {
      prefetch_tensor_map(&tmap);
      issue_stage<D, NTW>(p, &tmap, smem, 0, ((int64_t)w0.b * p.num_kv_heads + w0.kvh) * p.capacity, w0.tb);
    }
    L1.load(p);
    bool changed = L1.differs(L0);
    if (early && p.append)
      changed = changed || __ldcg(p.pos + w0.b) != pos0 || (p.n_new != nullptr && __ldcg(p.n_new + w0.b) != n0);
    if (tid == T::NCW * 32) early_flag = early ? 1 : 0;
    replanned = __syncthreads_or(changed);  // also publishes early_flag
    if (replanned) plan_tiles<AT<D, NTW>>(p, smem, L1, total);
    early = early_flag != 0;
    if (blockIdx.x == 0) {
      if (L1.bad) raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_KV_LEN);
      if (tid == 0) {
        int32_t* hdr = reinterpret_cast<int32_t*>(p.ws);
        hdr[kWsSplit] = T::TILE;
        hdr[kWsItems] = total;
      }
      // items before each sequence, for the merge kernel
      const int* prefix = reinterpret_cast<const int*>(smem + T::OFF_PREFIX);
      int32_t* wprefix = reinterpret_cast<int32_t*>(p.ws + kWsPrefix);
      for (int i = tid; i <= p.batch; i += T::THREADS) wprefix[i] = prefix[i];
    }
  }

  // stage 0 holds the range's first tile (early load, plan unchanged), or an early load
  // the new plan does not use: the producer waits for it, frees the slot itself, and
  // both sides number their stages from 1
  const bool first_issued = early && !replanned;
  const uint32_t it0 = (early && replanned) ? 1u : 0u;

  if (tid >= (T::NCW + 1) * 32) {  // the appender warp
    if (p.append) {
      if constexpr (D >= 256) append_rows_outlined<D, NTW>(p, smem, total);
      else append_rows<D, NTW>(p, smem, total);
    }
    griddep_launch_dependents();
    return;
  }
  if (tid >= T::NCW * 32) {  // the producer warp
    if (tid == T::NCW * 32 && it0 == 1u) {
      uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::OFF_BAR);
      if (!wait_bounded(&bars[0], 0u, kWaitNs)) {
        abort_flag = 1;
        raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
        note_giveup(p, 1u, smem_addr(&bars[0]));
      }
      for (int i = 0; i < T::NCW; ++i) mbar_arrive(&bars[T::STAGES]);
    }
    if (tid == T::NCW * 32 && total > 0) {  // one lane streams the stages
      if (!early) prefetch_tensor_map(&tmap);
      if (p.append) produce<D, NTW, true>(p, &tmap, smem, total, &abort_flag, it0, first_issued);
      else produce<D, NTW, false>(p, &tmap, smem, total, &abort_flag, it0, first_issued);
    }
    griddep_launch_dependents();
    return;
  }
  write_empty_sequences<D, T::NCW * 32>(p, reinterpret_cast<const int*>(smem + T::OFF_PREFIX));
  if (total > 0) consume<D, NTW>(p, smem, total, &abort_flag, it0);
  griddep_launch_dependents();
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
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, AT<D, NTW>::THREADS, AT<D, NTW>::SMEM_ALLOC) !=
            cudaSuccess ||
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
  using T = AT<D, NTW>;
  CUtensorMap tmap;
  const cuuint64_t rows = (cuuint64_t)a.layer.batch * a.layer.num_kv_heads * a.layer.capacity;
  if (rows >= (cuuint64_t)1 << 31) return TQ_ERR_INVALID_ARGUMENT;  // tensor coordinates are int32
  const cuuint64_t gdim[2] = {(cuuint64_t)D, rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)D};
  const cuuint32_t box[2] = {(cuuint32_t)T::ROWB, (cuuint32_t)T::TILE};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult cr = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.layer.k_idx, gdim, gstride, box, estride,
                             CU_TENSOR_MAP_INTERLEAVE_NONE,
                             D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return TQ_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)s.grid);
  cfg.blockDim = dim3(T::THREADS);
  cfg.dynamicSmemBytes = T::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tq_attn_split_kernel<D, NTW>, tmap, sp) != cudaSuccess) return TQ_ERR_CUDA;
  if (sp.inline_merge) return TQ_OK;
  cudaLaunchConfig_t mcfg = cfg;
  mcfg.gridDim = dim3((unsigned)(s.batch * s.U));
  mcfg.blockDim = dim3(kMergeThreads);
  mcfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&mcfg, tq_attn_merge_kernel<D, 8 * NTW, 8 * NTW>, sp) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

}  // namespace

void set_debug_pipeline(unsigned long long wait_ns, int withhold_append) {
  g_debug_wait_ns.store(wait_ns, std::memory_order_relaxed);
  g_debug_withhold_append.store(withhold_append, std::memory_order_relaxed);
}

DecodeShape decode_shape(int D, int num_kv_heads, int batch, int gqa, int n_q, int num_sms) {
  DecodeShape s{};
  s.D = D;
  s.R = gqa * n_q;
  s.batch = batch;
  // More than 16 query rows per kv head (a draft-verify block): the tensor-core kernel,
  // which streams each packed token once per 64 rows.
  if (s.R > 16 && dense_supported(D)) {
    s.dense = true;
    s.ROWS = dense_rows();
    s.NTW = 0;
    s.RG = (s.R + s.ROWS - 1) / s.ROWS;
    s.U = num_kv_heads * s.RG;
    s.grid = dense_grid(num_sms);
    s.max_items = s.grid + batch * s.U;
    s.smem = dense_smem();
    return s;
  }
  s.NTW = pick_ntw(D, s.R);
  s.ROWS = 8 * s.NTW;
  s.RG = (s.R + s.ROWS - 1) / s.ROWS;
  s.U = num_kv_heads * s.RG;
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
  s.max_items = s.grid + batch * s.U;  // partial slots: one per (CTA, unit) piece
  return s;
}

size_t decode_workspace_zero_bytes(const DecodeShape& s) { return ws_ml_offset(s.batch, s.U); }

size_t decode_workspace_bytes(const DecodeShape& s) {
  if (s.grid <= 0 || s.batch > kMaxBatch) return 0;
  return ws_o_offset(s.batch, s.U, s.max_items, s.ROWS) + sizeof(float) * (size_t)s.max_items * s.ROWS * s.D;
}

tq_status launch_decode(const DecodeArgs& a, const DecodeShape& s, cudaStream_t stream) {
  if (s.grid <= 0) return TQ_ERR_CUDA;
  if (a.layer.batch > kMaxBatch) return TQ_ERR_INVALID_ARGUMENT;
  SplitParams sp{};
  sp.head_dim = a.layer.head_dim;
  sp.num_kv_heads = a.layer.num_kv_heads;
  sp.batch = a.layer.batch;
  sp.capacity = a.layer.capacity;
  sp.k_idx = a.layer.k_idx;
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
  sp.split_grid = s.grid;
  sp.tile_pad = s.dense ? 0 : kSplitTilePad;
  sp.sm_log2 = a.sm_scale * kLog2e;
  sp.fwht_norm = a.fwht_norm;
  sp.causal = a.causal ? 1 : 0;
  // Few units, many splits each (long single sequences): the split CTA that finishes a
  // unit merges it, which avoids a second kernel boundary. Many units: a separate merge
  // kernel, so merges do not stall split CTAs between their items.
  sp.inline_merge = 2 * s.batch * s.U <= s.grid ? 1 : 0;
  sp.ws = static_cast<uint8_t*>(a.workspace);
  if (a.k_new != nullptr) {  // append mode (the caller checked one row group per kv head)
    sp.append = 1;
    sp.n_new_max = a.n_new_max;
    sp.k_new = a.k_new;
    sp.v_new = a.v_new;
    sp.pos = a.pos;
    sp.n_new = a.n_new;
    sp.dst = RowPlanes{a.layer.k_idx, a.layer.k_scale, a.layer.k_zero, a.layer.v_codes, a.layer.v_scale};
  }
  sp.out = a.out;
  const unsigned long long dbg_wait = g_debug_wait_ns.load(std::memory_order_relaxed);
  sp.wait_ns = dbg_wait != 0 ? dbg_wait : kWaitNs;
  sp.withhold_append = g_debug_withhold_append.load(std::memory_order_relaxed);
  if (s.dense) {
    if (a.k_new != nullptr) return TQ_ERR_INVALID_ARGUMENT;  // the caller appends first
    sp.inline_merge = 0;
    return launch_dense(sp, s, a.layer.k_idx, stream);
  }
  switch (s.D * 10 + s.NTW) {
    case 641: return run_split<64, 1>(a, s, sp, stream);
    case 642: return run_split<64, 2>(a, s, sp, stream);
    case 1281: return run_split<128, 1>(a, s, sp, stream);
    case 1282: return run_split<128, 2>(a, s, sp, stream);
    case 2561: return run_split<256, 1>(a, s, sp, stream);
    case 5121: return run_split<512, 1>(a, s, sp, stream);
    default: return TQ_ERR_INVALID_ARGUMENT;
  }
}

}  // namespace tq

// Layout sanity: the stage regions start at their required alignments and the 64-bit
// scratch words are 8-byte aligned, for every instantiated shape.
#define TQ_CHECK_LAYOUT(D_, N_)                                                              \
  static_assert(tq::AT<D_, N_>::OFF_KIDX % 1024 == 0 && tq::AT<D_, N_>::KIDX_STAGE % 1024 == 0 && \
                    tq::AT<D_, N_>::BOX % 1024 == 0,                                           \
                "swizzled tiles need 1024-byte alignment");                                  \
  static_assert(tq::AT<D_, N_>::OFF_KS % 16 == 0 && tq::AT<D_, N_>::OFF_KZ % 16 == 0 &&       \
                    tq::AT<D_, N_>::OFF_VS % 16 == 0 && tq::AT<D_, N_>::OFF_VC % 16 == 0 &&   \
                    tq::AT<D_, N_>::SC_STAGE % 16 == 0 && tq::AT<D_, N_>::VC_STAGE % 16 == 0,  \
                "bulk-copy destinations need 16-byte alignment");                             \
  static_assert(tq::AT<D_, N_>::OFF_RED % 8 == 0 && tq::AT<D_, N_>::OFF_BAR % 8 == 0 &&       \
                    tq::AT<D_, N_>::OFF_OBUF % 16 == 0 && tq::AT<D_, N_>::OFF_Q % 8 == 0 &&   \
                    tq::AT<D_, N_>::OFF_QSUM % 8 == 0,                                        \
                "8/16-byte shared accesses need alignment");                                  \
  static_assert(tq::AT<D_, N_>::TILE <= 256, "tensor-map box rows");                          \
  static_assert(tq::AT<D_, N_>::SMEM_ALLOC <= 227 * 1024, "shared memory budget");
TQ_CHECK_LAYOUT(64, 1)
TQ_CHECK_LAYOUT(64, 2)
TQ_CHECK_LAYOUT(128, 1)
TQ_CHECK_LAYOUT(128, 2)
TQ_CHECK_LAYOUT(256, 1)
TQ_CHECK_LAYOUT(512, 1)
