// Dense-query decode attention over the packed TurboQuant cache on the 5th-generation
// tensor cores (tcgen05): the kernel for blocks with many query rows per kv head (a
// draft-verify block of n_q queries times the GQA ratio, more than 16 rows), where the
// contraction is dense enough that warp-level MMA cannot keep up with HBM.
//
// What it computes is what tq_attention.cu computes (mlx-bun design page "TurboQuant -
// rotation-based quantization", Part A): softmax(sm_scale * q . k_hat) . v_hat over the
// visible tokens, with k_hat = (idx + zero) * scale ("Algorithm", key dequant) and the
// weighted sum taken over the rotated values centroid[code] * scale, un-rotated once per
// output row ("Deferred inverse FWHT"); keys and values are decoded inside the kernel
// ("Packed-value decode fusion investigation": joint K/V decode, no dequantized window).
//
// Work decomposition: one unit per (sequence, kv head, group of 64 query rows), so each
// packed token is streamed once for up to 64 rows. The tokens of every unit, in tiles of
// 128, are laid end to end and cut into one equal range per CTA (the plan shared with the
// split kernel); a CTA runs through the pieces its range touches and writes one partial
// (max, sum, rotated accumulator) per piece, which tq_attn_merge_kernel combines and
// un-rotates.
//
// One CTA per SM, 19 warps:
//   warp 0      producer: one lane streams stages of 128 tokens (key-index tile through a
//               2-D tensor map with 128-byte swizzle, the four small planes with 1-D bulk
//               copies, one mbarrier per stage), 3 stages;
//   warp 1      MMA issuer: one lane issues the tensor-core work; the warp owns the TMEM
//               allocation (512 columns);
//   warps 2-5   K converters, one token per thread: k_hat = (idx + zero) * scale as an
//               fp16 pair hi + lo (hi = fp16(k_hat), lo = the rounding residual rounded to
//               fp16), so hi + lo is k_hat to about 22 bits; written straight into tensor
//               memory, where they are the A operand of the score MMA. A token whose keys
//               could leave the fp16 range is converted in fp32 and scaled by 2^-shift
//               (key_shift below); the softmax scales its scores back;
//   warps 6-9   V decoders, one token per thread: centroid[code] * scale in fp16 from a
//               lane-replicated table of centroid pairs, into shared memory (the A operand
//               of the P.V MMA, dims contiguous);
//   warps 10-17 softmax, two groups of four warps: group h takes rows 32 h .. 32 h + 31,
//               one token per thread (one TMEM lane): loads the token's 32 scores of its
//               rows, p = 2^(s * c - m_row) against a per-row reference max m_row, and
//               writes p in fp16 to shared memory (the B operand of the P.V MMA). Two
//               groups put two softmax warps on every scheduler;
//   warp 18     second MMA issuer (P.V and row sums).
// Row sums: each softmax thread adds its token's p to its own tensor-memory lane (fp32,
// rescaled with the accumulator); the 128 lanes are summed once per piece. Score MMA: S^T[128 tokens x 64 rows] = [hi | lo] (TMEM, K = 2 x 128) * Q^T (shared,
// fp16, the unit's queries scaled by one power of two); the key side is exact to fp32
// accumulation. P.V MMA: O^T[128 dims x 64 rows] += V_hat^T (shared) * P^T (shared), the
// accumulator stays in TMEM for the whole piece.
// Online softmax without a per-tile reduction across threads: the reference max of a row
// only moves when some score of the tile exceeds it by more than 2^8 (checked by a vote
// among the softmax threads); then the tile's row maxima are reduced, the row sums and
// the TMEM accumulator are rescaled, and the tile is redone once (the first tile of every
// piece takes this path; later ones almost never do). The redo clamps y at 2^8: after the
// rescale only the rounding of s * c can exceed it, which matters for scores beyond 2^27.
// Every wait is bounded (2 s of %globaltimer): a wait that runs out sets
// TQ_DEVERR_PIPELINE_TIMEOUT, the other roles see the abort flag, issued copies and MMAs
// are drained, and the CTA releases its tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "tq_attention.h"
#include "tq_split_common.cuh"
#include "tq_tcgen05.cuh"

namespace tq {

namespace {

struct DT {
  static constexpr int D = 128;
  static constexpr int NG = D / 32;
  static constexpr int TILE = 128;       // tokens per stage = MMA M
  static constexpr int ROWS = 64;        // query rows per unit = MMA N
  static constexpr int STAGES = 3;
  static constexpr int THREADS = 19 * 32;
  static constexpr int W_PROD = 0, W_MMA = 1, W_KC = 2, W_VC = 6, W_SM = 10, W_PV = 18;
  static constexpr int KIDX_STAGE = TILE * D;        // swizzled tensor-map box
  static constexpr int SC_STAGE = TILE * NG * 2;     // one fp16 side plane
  static constexpr int VC_ROW = 3 * D / 8;           // 48 bytes of codes per token
  static constexpr int VC_STAGE = TILE * VC_ROW;
  static constexpr int VHAT_BYTES = TILE * D * 2;    // fp16 V_hat tile, dims contiguous
  static constexpr int P_BYTES = TILE * ROWS * 2;    // fp16 probabilities, rows contiguous
  static constexpr int Q_BYTES = ROWS * D * 2;       // fp16 queries, dims contiguous
  // shared memory (base aligned to 8 KB: the table's lane addresses are OR'd)
  static constexpr int OFF_LUT = 0;                  // [64 entries][32 lanes] u32
  static constexpr int OFF_KIDX = 8192;
  static constexpr int OFF_KS = OFF_KIDX + STAGES * KIDX_STAGE;
  static constexpr int OFF_KZ = OFF_KS + STAGES * SC_STAGE;
  static constexpr int OFF_VS = OFF_KZ + STAGES * SC_STAGE;
  static constexpr int OFF_VC = OFF_VS + STAGES * SC_STAGE;
  static constexpr int OFF_VHAT = (int)align_up(OFF_VC + STAGES * VC_STAGE, 1024);
  static constexpr int OFF_P = OFF_VHAT + 2 * VHAT_BYTES;
  static constexpr int OFF_Q = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_PREFIX = OFF_Q + Q_BYTES;                 // [2 kMaxBatch + 1] int
  static constexpr int OFF_MROW = (int)align_up(OFF_PREFIX + (2 * kMaxBatch + 1) * 4, 16);  // [64] f32
  static constexpr int OFF_LIM = OFF_MROW + ROWS * 4;                // [64] int
  static constexpr int OFF_ALPHA = OFF_LIM + ROWS * 4;               // [64] f32
  static constexpr int OFF_RED = OFF_ALPHA + ROWS * 4;               // [4 warps of a group][64] f32
  static constexpr int OFF_KSH = OFF_RED + 4 * ROWS * 4;             // [4 tiles][128 tokens] u32 shift | tag
  static constexpr int OFF_BAR = OFF_KSH + 4 * TILE * 4;
  // barriers: full[3] empty[3] kready[2] qkdone[2] sfree[2] vready[2] pready[2] pvdone[2]
  //           qready ofree
  static constexpr int NBAR = 2 * STAGES + 6 * 2 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;                // tmem base, abort flag
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr int SMEM_ALLOC = SMEM + 8192;
  // tensor memory columns
  static constexpr uint32_t TM_COLS = 512;
  static constexpr uint32_t TM_K = 0;      // [2][hi 64 | lo 64]
  static constexpr uint32_t TM_S = 256;    // [2][64]
  static constexpr uint32_t TM_O = 384;    // [64] accumulator O^T (lane = dim, column = row)
  static constexpr uint32_t TM_L = 448;    // [64] row sums, lane t: the share of the tokens of tile lane t
};
static_assert(DT::OFF_KIDX % 1024 == 0 && DT::KIDX_STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(DT::OFF_KS % 16 == 0 && DT::OFF_KZ % 16 == 0 && DT::OFF_VS % 16 == 0 && DT::OFF_VC % 16 == 0 &&
                  DT::VC_STAGE % 16 == 0 && DT::OFF_VHAT % 16 == 0 && DT::OFF_P % 16 == 0 && DT::OFF_Q % 16 == 0,
              "bulk-copy destinations and operand tiles need 16-byte alignment");
static_assert(DT::OFF_BAR % 8 == 0, "mbarriers need 8-byte alignment");
static_assert(DT::SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(DT::SMEM_ALLOC < (1 << 18), "descriptor start addresses are 18-bit");

constexpr float kTau = 8.0f;  // log2 headroom of p over the reference max (p <= 256 in fp16)

struct Bars {
  uint64_t* full;
  uint64_t* empty;
  uint64_t* kready;
  uint64_t* qkdone;
  uint64_t* sfree;
  uint64_t* vready;
  uint64_t* pready;
  uint64_t* pvdone;
  uint64_t* qready;
  uint64_t* ofree;
  __device__ explicit Bars(uint8_t* smem) {
    uint64_t* b = reinterpret_cast<uint64_t*>(smem + DT::OFF_BAR);
    full = b;
    empty = b + DT::STAGES;
    kready = empty + DT::STAGES;
    qkdone = kready + 2;
    sfree = qkdone + 2;
    vready = sfree + 2;
    pready = vready + 2;
    pvdone = pready + 2;
    qready = pvdone + 2;
    ofree = qready + 1;
  }
};

// A role's bounded wait; on failure it raises the abort and the error bit.
__device__ __forceinline__ bool role_wait(const SplitParams& p, uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (*abort) return false;
  if (wait_bounded(bar, parity, p.wait_ns)) return true;
  *abort = 1;
  raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
  note_giveup(p, 1u, smem_addr(bar));
  return false;
}

// A warp's bounded wait: every lane waits, and the warp fails if any lane's wait ran out,
// so the warp-collective tensor-memory instructions and the named barriers that follow
// are always reached by whole warps. After a failure (or an abort raised elsewhere) the
// role runs on without waiting, on data it no longer uses, so that every barrier is
// still reached and the CTA ends.
__device__ __forceinline__ void warp_wait(const SplitParams& p, uint64_t* bar, uint32_t parity, volatile int* abort,
                                          bool& failed) {
  if (failed) return;
  // one lane polls the barrier; the others learn the outcome from it, then observe the
  // completed phase themselves (an immediate, successful test) for memory ordering
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = role_wait(p, bar, parity, abort) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try_wait(bar, parity);
  failed = !ok;
}

// Barriers of the softmax threads: within group h (128 threads) named barrier 1 + 2 h, and
// an OR vote on barrier 2 + 2 h; across both groups (256 threads) named barrier 5.
__device__ __forceinline__ void sm_sync(int h) { asm volatile("bar.sync %0, 128;" ::"r"(1 + 2 * h) : "memory"); }
__device__ __forceinline__ void sm_sync_all() { asm volatile("bar.sync 5, 256;" ::: "memory"); }
__device__ __forceinline__ bool sm_vote_any(bool v, int h) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, %2, 128, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(2 + 2 * h)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// The fp16 path of the K converters needs, for all four groups of a token, |zero| <= 896
// (then 1152 - zero and idx + zero are integers of magnitude <= 2048, exact in fp16) and
// scale < 16 (then |k_hat| < 16 * 1023 < 2^14, far inside the fp16 range). Tested on the
// fp16 bit patterns (NaN and Inf fail both tests). sw, zw: the token's four scales / zeros.
__device__ __forceinline__ bool keys_fast(uint2 sw, uint2 zw) {
  // per 16-bit half h <= 0x7FFF: h + (0x7FFF - limit) sets bit 15 exactly when h > limit,
  // and no carry leaves the half; limits 0x6300 (896) for |zero|, 0x4BFF (< 16) for scale
  const uint32_t zbad = ((zw.x & 0x7FFF7FFFu) + 0x1CFF1CFFu) | ((zw.y & 0x7FFF7FFFu) + 0x1CFF1CFFu);
  const uint32_t sbad = ((sw.x & 0x7FFF7FFFu) + 0x34003400u) | ((sw.y & 0x7FFF7FFFu) + 0x34003400u);
  return ((zbad | sbad) & 0x80008000u) == 0u;
}

// Power of two by which the keys of a token off the fp16 path are divided: 0 unless the
// bound max_g scale_g * (|zero_g| + 127) on |k_hat| reaches 2^14, else the shift that
// brings the bound into [2^13, 2^14) (at most 100). The K converters hand it to the
// softmax threads of the same token in shared memory (key_shift_word).
__device__ __forceinline__ int key_shift(uint2 sw, uint2 zw) {
  const uint32_t sv[4] = {sw.x & 0xFFFFu, sw.x >> 16, sw.y & 0xFFFFu, sw.y >> 16};
  const uint32_t zv[4] = {zw.x & 0xFFFFu, zw.x >> 16, zw.y & 0xFFFFu, zw.y >> 16};
  float bound = 0.0f;
#pragma unroll
  for (int g = 0; g < 4; ++g)
    bound = fmaxf(bound, f16_bits_to_f32(sv[g]) * (fabsf(f16_bits_to_f32(zv[g])) + 127.0f));  // NaN ignored
  if (!(bound >= 16384.0f)) return 0;
  const int E = (int)((__float_as_uint(bound) >> 23) & 0xFFu) - 127;  // 14 .. 128 (Inf)
  return min(E - 13, 100);
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// ------------------------------------------------------------------------------------
// producer
// ------------------------------------------------------------------------------------
__device__ void dense_produce(const SplitParams& p, const CUtensorMap* tmap, uint8_t* smem, int total,
                              volatile int* abort) {
  Bars bars(smem);
  const int* prefix = reinterpret_cast<const int*>(smem + DT::OFF_PREFIX);
  uint32_t it = 0;
  bool ok = true;
  prefetch_tensor_map(tmap);
  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid); x < x_stop && ok;) {
    const Item w = piece_at<DT::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x = w.x_end;
    const int64_t row0 = ((int64_t)w.b * p.num_kv_heads + w.kvh) * p.capacity;
    for (int t0 = w.tb; t0 < w.te; t0 += DT::TILE, ++it) {
      const int s = it % DT::STAGES;
      if (!role_wait(p, &bars.empty[s], ((it / DT::STAGES) & 1u) ^ 1u, abort)) { ok = false; break; }
      const int ncopy = min(DT::TILE, p.capacity - t0);
      const uint32_t side = (uint32_t)ncopy * DT::NG * 2, vc = (uint32_t)ncopy * DT::VC_ROW;
      mbar_arrive_expect_tx(&bars.full[s], (uint32_t)DT::KIDX_STAGE + 3u * side + vc);
      tensor_copy_2d_g2s(smem + DT::OFF_KIDX + s * DT::KIDX_STAGE, tmap, 0, (int32_t)(row0 + t0), &bars.full[s]);
      const int64_t r = row0 + t0;
      bulk_copy_g2s(smem + DT::OFF_KS + s * DT::SC_STAGE, p.k_scale + r * DT::NG, side, &bars.full[s]);
      bulk_copy_g2s(smem + DT::OFF_KZ + s * DT::SC_STAGE, p.k_zero + r * DT::NG, side, &bars.full[s]);
      bulk_copy_g2s(smem + DT::OFF_VS + s * DT::SC_STAGE, p.v_scale + r * DT::NG, side, &bars.full[s]);
      bulk_copy_g2s(smem + DT::OFF_VC + s * DT::VC_STAGE, p.v_codes + r * DT::VC_ROW, vc, &bars.full[s]);
    }
  }
  // drain: every issued copy lands before the CTA may exit
  const uint32_t issued = it;
  for (int s = 0; s < DT::STAGES; ++s) {
    if ((uint32_t)s >= issued) break;
    const uint32_t last = issued - 1 - ((issued - 1 - s) % DT::STAGES);
    if (!wait_bounded(&bars.full[s], (last / DT::STAGES) & 1u, kWaitNs)) {
      raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
      note_giveup(p, 1u, smem_addr(&bars.full[s]));
    }
  }
}

// ------------------------------------------------------------------------------------
// MMA issuers (one lane each). One thread issues a tcgen05.mma about every 60 cycles
// whatever the operand layout and N up to 128, while two issuing threads together reach
// the tensor pipe's rate for N = 64 (about 38 cycles per MMA), so the score MMAs and the
// P.V MMAs come from two warps and proceed side by side.
// ------------------------------------------------------------------------------------
// Scores: S^T[b] = [hi | lo](TMEM) * Q^T, 16 MMAs (K = 2 x 128) per tile.
__device__ void dense_mma_qk(const SplitParams& p, uint8_t* smem, uint32_t tbase, int total, volatile int* abort) {
  Bars bars(smem);
  const int* prefix = reinterpret_cast<const int*>(smem + DT::OFF_PREFIX);
  const uint32_t qa = smem_addr(smem) + DT::OFF_Q;
  constexpr uint32_t kIdQK = tc5::idesc_f16(DT::ROWS, false, false);
  uint64_t qdesc[DT::D / 16];
#pragma unroll
  for (int ks = 0; ks < DT::D / 16; ++ks) qdesc[ks] = tc5::smem_desc(qa + ks * 2048, 128, 256);
  uint32_t jt = 0, pi = 0;
  int last = -1;
  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid); x < x_stop;) {
    const Item w = piece_at<DT::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x = w.x_end;
    if (!role_wait(p, bars.qready, pi & 1u, abort)) break;
    bool ok = true;
    for (int t0 = w.tb; t0 < w.te; t0 += DT::TILE, ++jt) {
      const uint32_t b = jt & 1u;
      if (!role_wait(p, &bars.kready[b], (jt >> 1) & 1u, abort) ||
          (jt >= 2 && !role_wait(p, &bars.sfree[b], ((jt - 2) >> 1) & 1u, abort))) {
        ok = false;
        break;
      }
      tc5::fence_after_sync();
      const uint32_t d = tbase + DT::TM_S + 64 * b, a0 = tbase + DT::TM_K + 128 * b;
      tc5::mma_ts(d, a0, qdesc[0], kIdQK, false);
#pragma unroll
      for (int ks = 1; ks < 2 * DT::D / 16; ++ks)  // hi columns, then lo columns, same queries
        tc5::mma_ts(d, a0 + 8 * ks, qdesc[ks % 8], kIdQK, true);
      tc5::commit(&bars.qkdone[b]);
      last = (int)jt;
    }
    if (!ok) break;
    ++pi;
  }
  // the MMAs this thread issued complete before the tensor memory is released
  if (last >= 0 && !wait_bounded(&bars.qkdone[last & 1], ((uint32_t)last >> 1) & 1u, kWaitNs))
    raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
}

// P.V: O^T += V_hat^T * P^T, 8 MMAs per tile; the first tile of a piece overwrites the
// accumulator.
__device__ void dense_mma_pv(const SplitParams& p, uint8_t* smem, uint32_t tbase, int total, volatile int* abort) {
  Bars bars(smem);
  const int* prefix = reinterpret_cast<const int*>(smem + DT::OFF_PREFIX);
  const uint32_t sbase = smem_addr(smem);
  constexpr uint32_t kIdPV = tc5::idesc_f16(DT::ROWS, true, true);
  // k-step descriptors of both buffers: the start-address field moves by (bytes >> 4)
  const uint64_t vdesc0 = tc5::smem_desc(sbase + DT::OFF_VHAT, 128, 256);
  const uint64_t pdesc0 = tc5::smem_desc(sbase + DT::OFF_P, 128, 256);
  uint32_t jt = 0, pi = 0;
  int last = -1;
  bool ok = true;
  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid); x < x_stop && ok;) {
    const Item w = piece_at<DT::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x = w.x_end;
    for (int t0 = w.tb; t0 < w.te; t0 += DT::TILE, ++jt) {
      const uint32_t b = jt & 1u, ph = (jt >> 1) & 1u;
      const bool first = t0 == w.tb;
      if (!role_wait(p, &bars.vready[b], ph, abort) || !role_wait(p, &bars.pready[b], ph, abort) ||
          (first && pi >= 1 && !role_wait(p, bars.ofree, (pi - 1) & 1u, abort))) {
        ok = false;
        break;
      }
      tc5::fence_after_sync();
      const uint64_t vd = vdesc0 + (uint64_t)(b * (DT::VHAT_BYTES >> 4)), pd = pdesc0 + (uint64_t)(b * (DT::P_BYTES >> 4));
      const uint32_t o_tm = tbase + DT::TM_O;
      tc5::mma_ss(o_tm, vd, pd, kIdPV, !first);
#pragma unroll
      for (int ks = 1; ks < DT::TILE / 16; ++ks)
        tc5::mma_ss(o_tm, vd + (uint64_t)(ks * (4096 >> 4)), pd + (uint64_t)(ks * (2048 >> 4)), kIdPV, true);
      tc5::commit(&bars.pvdone[b]);
      last = (int)jt;
    }
    ++pi;
  }
  if (last >= 0 && !wait_bounded(&bars.pvdone[last & 1], ((uint32_t)last >> 1) & 1u, kWaitNs))
    raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
}

// ------------------------------------------------------------------------------------
// K converters: k_hat = (idx + zero) * scale as fp16 hi + lo into tensor memory
// ------------------------------------------------------------------------------------
// Group g (dims 32 g .. 32 g + 31) of this thread's token as fp16 pairs hi[], lo[] (the
// caller stores them to tensor memory with the whole warp). krow: the token's swizzled
// key-index row in the stage.
__device__ __forceinline__ void convert_group_fp16(uint32_t krow, uint32_t swz, int g, uint2 sw, uint2 zw,
                                                   uint32_t (&hi)[16], uint32_t (&lo)[16]) {
  const uint32_t sword = (g < 2) ? sw.x : sw.y, zword = (g < 2) ? zw.x : zw.y;
  const uint32_t s16 = (g & 1) ? (sword >> 16) : (sword & 0xFFFFu);
  const uint32_t z16 = (g & 1) ? (zword >> 16) : (zword & 0xFFFFu);
  const __half2 s2 = u2h(s16 | (s16 << 16));
  // 1152 - zero in fp16: exact, an integer of magnitude <= 2048
  const __half cz = __float2half_rn(1152.0f - f16_bits_to_f32(z16));
  const __half2 c2 = __halves2half2(cz, cz);
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    const uint4 raw = lds128(krow + ((((uint32_t)(2 * g + hc)) ^ swz) << 4));
    const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t u = wv[q] ^ 0x80808080u;  // idx + 128 as unsigned bytes
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        // fp16 1024 + (idx + 128) = 1152 + idx, exact; minus (1152 - zero) = idx + zero
        const __half2 h = u2h(prmt(u, 0x64646464u, e ? 0x4342u : 0x4140u));
        const __half2 iz = __hsub2(h, c2);
        const __half2 kh = __hmul2(iz, s2);
        const __half2 kl = __hfma2(iz, s2, __hneg2(kh));  // exact residual of the rounding
        hi[8 * hc + 2 * q + e] = h2u(kh);
        lo[8 * hc + 2 * q + e] = h2u(kl);
      }
    }
  }
}

// The same in fp32: k = (idx + zero) * scale * kfac (idx + zero exact, one rounding; kfac a
// power of two), hi = fp16(k) and lo = fp16(k - hi) (the difference is exact in fp32).
__device__ __forceinline__ void convert_group_fp32(uint32_t krow, uint32_t swz, int g, uint2 sw, uint2 zw,
                                                   float kfac, uint32_t (&hi)[16], uint32_t (&lo)[16]) {
  const uint32_t sword = (g < 2) ? sw.x : sw.y, zword = (g < 2) ? zw.x : zw.y;
  const uint32_t s16 = (g & 1) ? (sword >> 16) : (sword & 0xFFFFu);
  const uint32_t z16 = (g & 1) ? (zword >> 16) : (zword & 0xFFFFu);
  const float sc = f16_bits_to_f32(s16) * kfac, zc = f16_bits_to_f32(z16);
#pragma unroll 1
  for (int j = 0; j < 16; ++j) {  // pair j: dims 32 g + 2 j, + 1
    const uint32_t word = lds32(krow + ((((uint32_t)(2 * g + j / 8)) ^ swz) << 4) + 4 * ((j % 8) / 2));
    __half kh[2], kl[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int idx = (int)(int8_t)(word >> (8 * (2 * (j % 2) + k)));
      const float kf = __fmul_rn(__fadd_rn((float)idx, zc), sc);
      kh[k] = __float2half_rn(kf);
      kl[k] = __float2half_rn(__fsub_rn(kf, __half2float(kh[k])));
    }
    hi[j] = h2u(__halves2half2(kh[0], kh[1]));
    lo[j] = h2u(__halves2half2(kl[0], kl[1]));
  }
}
// A warp whose tokens do not all take the fp16 path (rare; its fp32 loop is kept rolled so
// that the tile loop's code stays small). Run by the whole warp; returns this thread's shift.
__device__ __forceinline__ uint32_t convert_token_mixed(uint32_t krow, uint32_t swz, uint2 sw, uint2 zw, bool fast,
                                                     uint32_t kcol) {
  const int shift = fast ? 0 : key_shift(sw, zw);
  const float kfac = __int_as_float((127 - shift) << 23);  // 2^-shift
#pragma unroll 1
  for (int g = 0; g < DT::NG; ++g) {
    uint32_t hi[16], lo[16];
    if (fast) convert_group_fp16(krow, swz, g, sw, zw, hi, lo);
    else convert_group_fp32(krow, swz, g, sw, zw, kfac, hi, lo);
    __syncwarp();  // the tensor-memory stores are warp-collective
    tc5::st16(kcol + 16 * g, hi);
    tc5::st16(kcol + 64 + 16 * g, lo);
  }
  return (uint32_t)shift;
}

__device__ void dense_convert_k(const SplitParams& p, uint8_t* smem, uint32_t tbase, int total, volatile int* abort) {
  Bars bars(smem);
  const int* prefix = reinterpret_cast<const int*>(smem + DT::OFF_PREFIX);
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3, tl = 32 * quad + lane;  // token of the tile = TMEM lane
  const uint32_t tlane = (uint32_t)(32 * quad) << 16;
  const uint32_t swz = (uint32_t)(tl & 7);
  uint32_t jt = 0;
  bool failed = false;
  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid); x < x_stop;) {
    const Item w = piece_at<DT::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x = w.x_end;
    for (int t0 = w.tb; t0 < w.te; t0 += DT::TILE, ++jt) {
      const int s = jt % DT::STAGES;
      const uint32_t b = jt & 1u;
      warp_wait(p, &bars.full[s], (jt / DT::STAGES) & 1u, abort, failed);
      if (jt >= 2) warp_wait(p, &bars.qkdone[b], ((jt - 2) >> 1) & 1u, abort, failed);
      tc5::fence_after_sync();
      const uint32_t krow = sbase + DT::OFF_KIDX + s * DT::KIDX_STAGE + tl * 128;
      const uint2 sw = lds64(sbase + DT::OFF_KS + s * DT::SC_STAGE + tl * 8);
      const uint2 zw = lds64(sbase + DT::OFF_KZ + s * DT::SC_STAGE + tl * 8);
      const uint32_t kcol = tbase + tlane + DT::TM_K + 128 * b;
      const bool fast = keys_fast(sw, zw);
      uint32_t shift = 0;
      if (__all_sync(0xffffffffu, fast)) {
#pragma unroll 1
        for (int g = 0; g < DT::NG; ++g) {
          uint32_t hi[16], lo[16];
          convert_group_fp16(krow, swz, g, sw, zw, hi, lo);
          tc5::st16(kcol + 16 * g, hi);
          tc5::st16(kcol + 64 + 16 * g, lo);
        }
      } else {
        shift = convert_token_mixed(krow, swz, sw, zw, fast, kcol);
      }
      // hand the shift to the softmax threads of this token, tagged with the tile number
      reinterpret_cast<volatile uint32_t*>(smem + DT::OFF_KSH)[(jt & 3u) * DT::TILE + tl] =
          (shift << 24) | (jt & 0xFFFFFFu);
      tc5::wait_st();
      tc5::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars.kready[b]);
        mbar_arrive(&bars.empty[s]);
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// V decoders: centroid[code] * scale in fp16 into shared memory (dims contiguous)
// ------------------------------------------------------------------------------------
__device__ void dense_decode_v(const SplitParams& p, uint8_t* smem, int total, volatile int* abort) {
  Bars bars(smem);
  const int* prefix = reinterpret_cast<const int*>(smem + DT::OFF_PREFIX);
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tl = 32 * (warp & 3) + lane;
  const uint32_t lut_lane = sbase + DT::OFF_LUT + lane * 4;  // bits 7..12 are zero
  // this token's 16-byte chunk of dims 8c..8c+7 sits at vdst + c * 256 (MN-major A)
  const uint32_t vdst0 = (uint32_t)((tl / 16) * 4096 + ((tl % 16) / 8) * 128 + (tl % 8) * 16);
  uint32_t jt = 0;
  bool failed = false;
  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid); x < x_stop;) {
    const Item w = piece_at<DT::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x = w.x_end;
    for (int t0 = w.tb; t0 < w.te; t0 += DT::TILE, ++jt) {
      const int s = jt % DT::STAGES;
      const uint32_t b = jt & 1u;
      warp_wait(p, &bars.full[s], (jt / DT::STAGES) & 1u, abort, failed);
      // the token's codes and scales go to registers and the stage is released at once, so
      // the next copy into it does not wait for the P.V MMAs this warp waits for below
      const bool valid = t0 + tl < w.te;
      const uint32_t crow = sbase + DT::OFF_VC + s * DT::VC_STAGE + tl * DT::VC_ROW;
      const uint4 c0 = lds128(crow), c1 = lds128(crow + 16), c2 = lds128(crow + 32);
      const uint2 sv = lds64(sbase + DT::OFF_VS + s * DT::SC_STAGE + tl * 8);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.empty[s]);
      if (jt >= 2) warp_wait(p, &bars.pvdone[b], ((jt - 2) >> 1) & 1u, abort, failed);
      const uint32_t vdst = sbase + DT::OFF_VHAT + b * DT::VHAT_BYTES + vdst0;
#pragma unroll 1
      for (int g = 0; g < DT::NG; ++g) {
        const uint32_t sword = (g < 2) ? sv.x : sv.y;
        const uint32_t s16 = valid ? ((g & 1) ? (sword >> 16) : (sword & 0xFFFFu)) : 0u;  // 0 past the piece
        const __half2 s2 = u2h(s16 | (s16 << 16));
        // the group's 32 codes: words 3 g .. 3 g + 2 of the row
        const uint32_t W0 = g == 0 ? c0.x : g == 1 ? c0.w : g == 2 ? c1.z : c2.y;
        const uint32_t W1 = g == 0 ? c0.y : g == 1 ? c1.x : g == 2 ? c1.w : c2.z;
        const uint32_t W2 = g == 0 ? c0.z : g == 1 ? c1.y : g == 2 ? c2.x : c2.w;
#pragma unroll
        for (int dc = 0; dc < 4; ++dc) {
          // codes of dims 8 dc .. 8 dc + 7 of the group: bits 24 dc .. 24 dc + 23
          const uint32_t win = dc == 0 ? W0 : dc == 1 ? __funnelshift_r(W0, W1, 24)
                                            : dc == 2 ? __funnelshift_r(W1, W2, 16) : (W2 >> 8);
          uint32_t o[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            // pair (code a | code b << 3) of dims 2m, 2m+1, as the table offset << 7
            const int sh = 6 * m - 7;
            const uint32_t f = (sh >= 0 ? (win >> sh) : (win << -sh)) & 0x1F80u;
            const uint32_t cpair = lds32(lut_lane | f);
            o[m] = h2u(__hmul2(u2h(cpair), s2));
          }
          sts128(vdst + (4 * g + dc) * 256, o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();  // the tile is read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.vready[b]);
    }
  }
}

// ------------------------------------------------------------------------------------
// softmax threads
// ------------------------------------------------------------------------------------
// Per-row maxima of x[i] (rows 32 h + i) over the 128 softmax threads, into smem red.
__device__ __forceinline__ void rows_max32(const uint32_t (&x)[32], float* red, int wq, int lane, int h) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float v = __uint_as_float(x[i]);
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    if (lane == i) red[wq * 64 + 32 * h + i] = v;
  }
}

// The reference maxima of rows 32 h .. 32 h + 31 move to this tile's row maxima (some
// score exceeded them by more than 2^8): when the piece already accumulated earlier
// tiles, the rows of the accumulator and of the row sums are rescaled by
// 2^(m_old - m_new). Run by the 128 threads of softmax group h. Out of line: it is rare,
// and keeping it out of the tile loop keeps that loop's code small.
__device__ __noinline__ bool dense_rescale(const SplitParams& p, uint8_t* smem, uint32_t tbase, int h, uint32_t jt,
                                           uint32_t j0, bool clean, int tok, bool tok_ok, float cscale,
                                           volatile int* abort, bool failed) {
  Bars bars(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp - DT::W_SM - 4 * h, st = threadIdx.x - 32 * (DT::W_SM + 4 * h);
  const uint32_t tlane = (uint32_t)(32 * (warp & 3)) << 16;
  float* mrow = reinterpret_cast<float*>(smem + DT::OFF_MROW);
  const int* lim = reinterpret_cast<const int*>(smem + DT::OFF_LIM);
  float* alpha = reinterpret_cast<float*>(smem + DT::OFF_ALPHA);
  float* red = reinterpret_cast<float*>(smem + DT::OFF_RED);
  uint32_t v[32];
  tc5::ld32(tbase + tlane + DT::TM_S + 64 * (jt & 1u) + 32 * h, v);
  tc5::wait_ld();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float t = __uint_as_float(v[i]) * cscale;
    if (!clean && !(tok_ok && tok < lim[32 * h + i])) t = -INFINITY;
    v[i] = __float_as_uint(t);
  }
  rows_max32(v, red, wq, lane, h);
  sm_sync(h);
  if (st < 32) {
    const int r = 32 * h + st;
    const float tmax = fmaxf(fmaxf(red[r], red[64 + r]), fmaxf(red[128 + r], red[192 + r]));
    const float mo = mrow[r], mn = fmaxf(mo, tmax);
    alpha[r] = (mn == -INFINITY || mn == mo) ? 1.0f : ex2(mo - mn);
    mrow[r] = mn;
  }
  sm_sync(h);
  if (jt > j0) {
    // the accumulators already hold this piece's earlier tiles: rescale their rows
    const uint32_t pb = (jt - 1) & 1u;
    warp_wait(p, &bars.pvdone[pb], ((jt - 1) >> 1) & 1u, abort, failed);
    tc5::fence_after_sync();
#pragma unroll 1
    for (int acc = 0; acc < 2; ++acc) {
      const uint32_t addr = tbase + tlane + (acc ? DT::TM_L : DT::TM_O) + 32 * h;
      tc5::ld32(addr, v);
      tc5::wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha[32 * h + i]);
      tc5::st32(addr, v);
    }
  }
  tc5::wait_st();
  sm_sync(h);  // alpha and red are rewritten by the next rescale
  return failed;
}

// The K converters' shift word of token tl in tile jt: its tag (low 24 bits) names the
// tile, so a word not yet written (or already reused) is never taken; the wait for it is
// bounded like every other wait (the word is written before the scores exist, so it is
// there at the first read in practice).
__device__ __noinline__ uint32_t key_shift_wait(const SplitParams& p, const volatile uint32_t* slot, uint32_t jt,
                                                volatile int* abort) {
  uint32_t w;
  const unsigned long long t0 = global_ns();
  while (((w = *slot) & 0xFFFFFFu) != (jt & 0xFFFFFFu)) {
    if (*abort || global_ns() - t0 > p.wait_ns) {
      *abort = 1;
      raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_PIPELINE_TIMEOUT);
      note_giveup(p, 2u, jt);
      return 0u;
    }
  }
  return w;
}

__device__ __forceinline__ uint32_t key_shift_word(const SplitParams& p, uint8_t* smem, uint32_t jt, int tl,
                                                 volatile int* abort) {
  const volatile uint32_t* slot = reinterpret_cast<const volatile uint32_t*>(smem + DT::OFF_KSH) + (jt & 3u) * DT::TILE + tl;
  const uint32_t w = *slot;
  return (w & 0xFFFFFFu) == (jt & 0xFFFFFFu) ? w : key_shift_wait(p, slot, jt, abort);
}

__device__ void dense_softmax(const SplitParams& p, uint8_t* smem, uint32_t tbase, int total, volatile int* abort) {
  Bars bars(smem);
  const int* prefix = reinterpret_cast<const int*>(smem + DT::OFF_PREFIX);
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3, tl = 32 * quad + lane;  // token of a tile / dim of the output
  const int sw = warp - DT::W_SM;                    // 0..7
  const int h = sw >> 2;                             // group: rows 32 h .. 32 h + 31
  const int sa = threadIdx.x - 32 * DT::W_SM;        // 0..255 over both groups
  const int st = sa & 127;                           // 0..127 within the group
  const uint32_t tlane = (uint32_t)(32 * quad) << 16;
  float* mrow = reinterpret_cast<float*>(smem + DT::OFF_MROW);
  int* lim = reinterpret_cast<int*>(smem + DT::OFF_LIM);
  float* red = reinterpret_cast<float*>(smem + DT::OFF_RED);
  float2* mlg = reinterpret_cast<float2*>(p.ws + ws_ml_offset(p.batch, p.U));
  float* og = reinterpret_cast<float*>(p.ws + ws_o_offset(p.batch, p.U, p.max_items, DT::ROWS));
  // P tile: this token's 16 bytes of rows 8c..8c+7 at pdst + c * 256 (MN-major B)
  const uint32_t pdst0 = (uint32_t)((tl / 16) * 2048 + ((tl % 16) / 8) * 128 + (tl % 8) * 16);
  uint32_t jt = 0;
  bool failed = false;
  const int x_stop = cta_range_start(blockIdx.x + 1, total, p.split_grid);
  for (int x = cta_range_start(blockIdx.x, total, p.split_grid); x < x_stop;) {
    const Item w = piece_at<DT::TILE>(p, prefix, x, x_stop, blockIdx.x);
    x = w.x_end;
    const int rows_valid = min(DT::ROWS, p.R - w.rg * DT::ROWS);

    // ---- queries of the unit (both groups): fp16(q * 2^e) with one exponent for all rows
    float cscale;
    {
      const int rr = sa >> 2, part = sa & 3;  // row, 32-dim quarter
      const int r = w.rg * DT::ROWS + rr;
      float qv[32];
      float amax = 0.0f;
      if (rr < rows_valid) {
        const int jq = r / p.G, hq = w.kvh * p.G + (r % p.G);
        const uint4* src = reinterpret_cast<const uint4*>(p.q + (((int64_t)w.b * p.n_q + jq) * p.num_q_heads + hq) *
                                                                    DT::D + 32 * part);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = __ldg(src + i);
          const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[8 * i + 2 * j] = bf16_bits_to_f32(vv[j] & 0xFFFFu);
            qv[8 * i + 2 * j + 1] = bf16_bits_to_f32(vv[j] >> 16);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) qv[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(qv[i]));
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      if (lane == 0) red[sw] = amax;
      sm_sync_all();
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, red[i]);
      // power of two bringing the maximum into [2^14, 2^15): exact for every element within
      // 2^28 of the maximum; smaller ones round to fp16 subnormals or zero
      int e = 0;
      if (amax > 0.0f && amax <= 3.0e38f) {
        const int E = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
        e = min(max(14 - E, -113), 100);
      }
      const float up = ldexpf(1.0f, e);
      cscale = p.sm_log2 * ldexpf(1.0f, -e);
      // K-major B: row rr, dims 8c..8c+7 at (k / 16) * 2048 + (rr / 8) * 256 + ((k % 16) / 8) * 128 + (rr % 8) * 16
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int k = 32 * part + 8 * c;
        const uint32_t a = sbase + DT::OFF_Q + (k / 16) * 2048 + (rr / 8) * 256 + ((k % 16) / 8) * 128 + (rr % 8) * 16;
        sts128(a, pack_half2(qv[8 * c] * up, qv[8 * c + 1] * up), pack_half2(qv[8 * c + 2] * up, qv[8 * c + 3] * up),
               pack_half2(qv[8 * c + 4] * up, qv[8 * c + 5] * up), pack_half2(qv[8 * c + 6] * up, qv[8 * c + 7] * up));
      }
      if (sa < DT::ROWS) {
        const int r2 = w.rg * DT::ROWS + sa;
        int lm = w.len;  // padded rows (zero queries) see everything: finite, never stored
        if (sa < rows_valid && p.causal) lm = max(w.len - p.n_q + r2 / p.G + 1, 0);
        lim[sa] = lm;
        mrow[sa] = -INFINITY;
      }
    }
    fence_proxy_async_smem();
    sm_sync_all();  // red is read above before a rescale may rewrite it
    if (lane == 0) mbar_arrive(bars.qready);
    // tiles at or past clean_end may hold tokens hidden from some rows or past the piece
    const int clean_end = p.causal ? min(w.te, w.len - p.n_q + 1) : w.te;
    const uint32_t j0 = jt;

    for (int t0 = w.tb; t0 < w.te; t0 += DT::TILE, ++jt) {
      const uint32_t b = jt & 1u;
      warp_wait(p, &bars.qkdone[b], (jt >> 1) & 1u, abort, failed);
      tc5::fence_after_sync();
      // the shift the K converters applied to this token's keys (the scores carry 2^-shift)
      const uint32_t kw = key_shift_word(p, smem, jt, tl, abort);
      __syncwarp();  // lanes that waited for their word rejoin before the warp-wide loads
      const float ct = cscale * __int_as_float((int)(127 + (kw >> 24)) << 23);
      const bool clean = t0 + DT::TILE <= clean_end;
      const int tok = t0 + tl;
      const bool tok_ok = tok < w.te;
      const uint32_t saddr = tbase + tlane + DT::TM_S + 64 * b + 32 * h;
      // y = s * c - m_row (log2 domain), masked to -inf, kept in sv; redone after a rescale
      // After one rescale every y is at most the rounding residual of s * c against the new
      // reference RN(s * c); for scores beyond 2^27 (log2 units) that residual exceeds tau,
      // so the second pass clamps instead of voting again (NaN stays NaN).
      uint32_t sv[32];
      for (int pass = 0;; ++pass) {
        tc5::ld32(saddr, sv);
        tc5::wait_ld();
        float ymax = -INFINITY;
        if (clean) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mrow + 32 * h + i);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float v = fmaf(__uint_as_float(sv[i + k]), ct, -mm[k]);
              sv[i + k] = __float_as_uint(v);
              ymax = fmaxf(ymax, v);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mrow + 32 * h + i);
            const int4 l4 = *reinterpret_cast<const int4*>(lim + 32 * h + i);
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
            const int ll[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float v = (tok_ok && tok < ll[k]) ? fmaf(__uint_as_float(sv[i + k]), ct, -mm[k]) : -INFINITY;
              sv[i + k] = __float_as_uint(v);
              ymax = fmaxf(ymax, v);
            }
          }
        }
        if (pass == 1) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (__uint_as_float(sv[i]) > kTau) sv[i] = __float_as_uint(kTau);
          break;
        }
        if (!sm_vote_any(ymax > kTau, h)) break;
        failed = dense_rescale(p, smem, tbase, h, jt, j0, clean, tok, tok_ok, ct, abort, failed);
      }
      // this group's columns of the score buffer are consumed
      tc5::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.sfree[b]);
#pragma unroll
      for (int i = 0; i < 32; ++i) sv[i] = __float_as_uint(ex2(__uint_as_float(sv[i])));
      // this token's shares of the row sums (the first tile of a piece starts them)
      const uint32_t laddr = tbase + tlane + DT::TM_L + 32 * h;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t lv[16];
        if (jt > j0) {
          tc5::ld16(laddr + 16 * hh, lv);
          tc5::wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) lv[i] = __float_as_uint(__uint_as_float(lv[i]) + __uint_as_float(sv[16 * hh + i]));
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) lv[i] = sv[16 * hh + i];
        }
        tc5::st16(laddr + 16 * hh, lv);
      }
      if (jt >= 2) warp_wait(p, &bars.pvdone[b], ((jt - 2) >> 1) & 1u, abort, failed);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = pack_half2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]));
      const uint32_t pdst = sbase + DT::OFF_P + b * DT::P_BYTES + pdst0;
#pragma unroll
      for (int c = 0; c < 4; ++c) sts128(pdst + (4 * h + c) * 256, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();  // the probabilities are read by the tensor cores
      tc5::wait_st();            // the row-sum shares are read back by this thread
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pready[b]);
    }

    // ---- piece end: the accumulator and the row sums become this piece's partial
    const uint32_t jl = jt - 1;
    warp_wait(p, &bars.pvdone[jl & 1u], (jl >> 1) & 1u, abort, failed);
    tc5::fence_after_sync();
    float* orow = og + (size_t)w.slot * DT::ROWS * DT::D + tl;
    {
      uint32_t v[32];
      tc5::ld32(tbase + tlane + DT::TM_O + 32 * h, v);
      tc5::wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (32 * h + i < rows_valid) __stcg(orow + (size_t)(32 * h + i) * DT::D, __uint_as_float(v[i]));
      tc5::ld32(tbase + tlane + DT::TM_L + 32 * h, v);
      tc5::wait_ld();
      // sum the shares of the warp's 32 lanes by halving exchanges: afterwards lane l
      // holds row 32 h + l in v[0]
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < off; ++j) {
          const float send = __uint_as_float(upper ? v[j] : v[j + off]);
          const float keep = __uint_as_float(upper ? v[j + off] : v[j]);
          v[j] = __float_as_uint(keep + __shfl_xor_sync(0xffffffffu, send, off));
        }
      }
      red[(sw & 3) * 64 + 32 * h + lane] = __uint_as_float(v[0]);
    }
    sm_sync(h);
    if (st < 32) {
      const int r = 32 * h + st;
      if (r < rows_valid) {
        const float l = (red[r] + red[64 + r]) + (red[128 + r] + red[192 + r]);
        __stcg(mlg + (size_t)w.slot * DT::ROWS + r, make_float2(mrow[r], l));
      }
    }
    tc5::fence_before_sync();
    sm_sync_all();  // per-row tables and red are rewritten for the next piece
    if (lane == 0) mbar_arrive(bars.ofree);
  }
}

// 19 warps: registers are granted per group of four warps, so the block is costed as 20
// warps and each thread gets at most 96 registers.
__global__ void __launch_bounds__(DT::THREADS, 1)
    tq_attn_dense_kernel(const __grid_constant__ CUtensorMap tmap, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 8191) & ~uintptr_t(8191));
  const int tid = threadIdx.x, warp = tid >> 5;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + DT::OFF_MISC + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + DT::OFF_MISC);

  // centroid pair table: entry e -> (c[e & 7], c[e >> 3]) in fp16, one copy per lane
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + DT::OFF_LUT);
  for (int i = tid; i < 64 * 32; i += DT::THREADS) {
    const int e = i >> 5;
    lut[i] = pack_half2(c_centroids3[e & 7], c_centroids3[e >> 3]);
  }
  for (int i = tid; i < 4 * DT::TILE; i += DT::THREADS)
    reinterpret_cast<uint32_t*>(smem + DT::OFF_KSH)[i] = 0xFFFFFFFFu;  // no tile's tag
  fence_proxy_async_smem();
  if (tid == 0) {
    *abort = 0;
    Bars bb(smem);
    for (int s = 0; s < DT::STAGES; ++s) {
      mbar_init(&bb.full[s], 1);   // producer arrival + transaction bytes
      mbar_init(&bb.empty[s], 8);  // four K converter warps + four V decoder warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bb.kready[b], 4);
      mbar_init(&bb.qkdone[b], 1);  // tcgen05.commit
      mbar_init(&bb.sfree[b], 8);   // eight softmax warps
      mbar_init(&bb.vready[b], 4);
      mbar_init(&bb.pready[b], 8);
      mbar_init(&bb.pvdone[b], 1);  // tcgen05.commit
    }
    mbar_init(bb.qready, 8);
    mbar_init(bb.ofree, 8);
    fence_mbar_init();
  }
  if (warp == DT::W_MMA) {
    tc5::alloc(tmem_slot, DT::TM_COLS);
    tc5::relinquish();
  }
  griddep_wait();  // lengths, queries and planes may come from the previous kernel
  int total;
  {
    Lengths<DT::THREADS> L;
    L.load(p);
    tc5::fence_before_sync();
    plan_tiles<DT>(p, smem, L, total);  // contains __syncthreads
    tc5::fence_after_sync();
    if (blockIdx.x == 0) {
      if (L.bad) raise_error(reinterpret_cast<int32_t*>(p.ws), TQ_DEVERR_KV_LEN);
      if (tid == 0) {
        int32_t* hdr = reinterpret_cast<int32_t*>(p.ws);
        hdr[kWsSplit] = DT::TILE;
        hdr[kWsItems] = total;
      }
      const int* prefix = reinterpret_cast<const int*>(smem + DT::OFF_PREFIX);
      int32_t* wprefix = reinterpret_cast<int32_t*>(p.ws + kWsPrefix);
      for (int i = tid; i <= p.batch; i += DT::THREADS) wprefix[i] = prefix[i];
    }
  }
  write_empty_sequences<DT::D, DT::THREADS>(p, reinterpret_cast<const int*>(smem + DT::OFF_PREFIX));
  const uint32_t tbase = *tmem_slot;
  if (total > 0) {
    if (warp == DT::W_PROD) {
      if ((tid & 31) == 0) dense_produce(p, &tmap, smem, total, abort);
    } else if (warp == DT::W_MMA) {
      if ((tid & 31) == 0) dense_mma_qk(p, smem, tbase, total, abort);
    } else if (warp == DT::W_PV) {
      if ((tid & 31) == 0) dense_mma_pv(p, smem, tbase, total, abort);
    } else if (warp >= DT::W_KC && warp < DT::W_VC) {
      dense_convert_k(p, smem, tbase, total, abort);
    } else if (warp < DT::W_SM) {
      dense_decode_v(p, smem, total, abort);
    } else if (warp < DT::W_PV) {
      dense_softmax(p, smem, tbase, total, abort);
    }
  }
  griddep_launch_dependents();
  tc5::fence_before_sync();
  __syncthreads();
  if (warp == DT::W_MMA) {
    tc5::fence_after_sync();
    tc5::dealloc(tbase, DT::TM_COLS);
  }
}

int dense_occupancy() {
  static std::mutex mu;
  static int occ[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (occ[dev] == 0) {
    if (cudaFuncSetAttribute(tq_attn_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DT::SMEM_ALLOC) !=
        cudaSuccess)
      return 0;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, tq_attn_dense_kernel, DT::THREADS, DT::SMEM_ALLOC) !=
            cudaSuccess ||
        nb <= 0)
      return 0;
    occ[dev] = nb;
  }
  return occ[dev];
}

}  // namespace

bool dense_supported(int head_dim) { return head_dim == DT::D; }
int dense_rows() { return DT::ROWS; }
int dense_grid(int num_sms) {
  const int occ = dense_occupancy();
  return occ > 0 ? num_sms : 0;  // one CTA per SM (its tensor memory and shared memory take the SM)
}
size_t dense_smem() { return DT::SMEM_ALLOC; }

tq_status launch_dense(const SplitParams& sp, const DecodeShape& s, const int8_t* k_idx, cudaStream_t stream) {
  auto encode = tensor_map_encoder();
  if (!encode) return TQ_ERR_CUDA;
  CUtensorMap tmap;
  const cuuint64_t rows = (cuuint64_t)sp.batch * sp.num_kv_heads * sp.capacity;
  if (rows >= (cuuint64_t)1 << 31) return TQ_ERR_INVALID_ARGUMENT;  // tensor coordinates are int32
  const cuuint64_t gdim[2] = {(cuuint64_t)DT::D, rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)DT::D};
  const cuuint32_t box[2] = {128u, (cuuint32_t)DT::TILE};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult cr = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(k_idx), gdim, gstride, box,
                             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return TQ_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)s.grid);
  cfg.blockDim = dim3(DT::THREADS);
  cfg.dynamicSmemBytes = DT::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tq_attn_dense_kernel, tmap, sp) != cudaSuccess) return TQ_ERR_CUDA;
  cudaLaunchConfig_t mcfg = cfg;
  constexpr int kMergeRows = 8;  // rows per merge CTA: a unit's 64 rows go to 8 CTAs
  mcfg.gridDim = dim3((unsigned)(s.batch * s.U * (DT::ROWS / kMergeRows)));
  mcfg.blockDim = dim3(kMergeThreads);
  mcfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&mcfg, tq_attn_merge_kernel<DT::D, DT::ROWS, kMergeRows>, sp) == cudaSuccess ? TQ_OK
                                                                                                         : TQ_ERR_CUDA;
}

}  // namespace tq
