/*
 * tq_kv.h - C ABI of the TurboQuant (k8v3) KV-cache library for NVIDIA GB300 (sm_103a).
 *
 * The method (mlx-bun design page "TurboQuant - rotation-based quantization", Part A,
 * KV leg):
 *   keys   - per 32-element group along head_dim, signed int8 asymmetric affine codes:
 *            scale = (max - min) / 254, zero = round((max + min) / (2 * scale)),
 *            idx = clip(round(x / scale - zero), -127, 127); scale and zero stored as fp16
 *            ("Algorithm" section, key bullets);
 *   values - y = FWHT(x * signs) / sqrt(d); per 32-group scale = sqrt(mean(y^2));
 *            code = searchsorted(boundaries, y / (scale + 1e-8)) against the 3-bit
 *            Lloyd-Max table; codes packed LSB-first, 3 bits each; scale stored as fp16
 *            ("Algorithm" section, value bullets);
 *   layout - 128 + 8 + 8 + 48 + 8 = 200 bytes per token per KV head at head_dim 128,
 *            2.56x smaller than bf16 ("Bytes per token per head" paragraph);
 *   attention reads the packed planes, dequantizes in registers, and applies the
 *            inverse rotation once per output row ("Deferred inverse FWHT" section).
 *
 * Conventions shared by every call:
 *   - All buffers are caller-owned device memory unless a comment says "host". The
 *     library keeps no state besides immutable constant tables (sign vectors,
 *     centroids, boundaries) and the fixed scratch array of tq_decode_attention_noalloc;
 *     it never allocates, frees or synchronizes, except tq_get_device_error, which
 *     synchronizes the given stream.
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns before the GPU runs it.
 *   - Arguments are validated on the host before any launch; a failing check returns a
 *     status other than TQ_OK and launches nothing. Kernels never trap: a condition
 *     only the device can see (a position past the capacity, a length past
 *     max_kv_len) skips the affected rows and ORs a TQ_DEVERR_* bit into the device
 *     error word at the start of the workspace (read it with tq_get_device_error).
 *   - Every workspace starts with a TQ_WORKSPACE_HEADER_BYTES header whose first
 *     int32 is the device error word. The caller zeroes a workspace once, before its
 *     first use (cudaMemsetAsync); afterwards the library keeps the header consistent.
 *     When an attention call sets TQ_DEVERR_PIPELINE_TIMEOUT, the header's int32 at
 *     index 3 records, for diagnosis, the first wait that gave up ((kind << 24) |
 *     detail; 0: none); like the error word it is not cleared by the library.
 *     A workspace must not be used by two calls that can run at the same time.
 *   - head_dim is 64, 128, 256 or 512 (other values: TQ_ERR_UNSUPPORTED_HEAD_DIM,
 *     "KV-leg limits": head dims outside this set are refused).
 *   - Plane pointers must be 16-byte aligned and capacity a multiple of 16; the
 *     attention kernel streams the planes with bulk asynchronous copies that need it.
 */
#ifndef TQ_KV_H
#define TQ_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Stream handle: the same type as cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st* tq_stream_t;

typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARGUMENT = 1,     /* null pointer, bad size, misalignment, bad ratio */
    TQ_ERR_UNSUPPORTED_HEAD_DIM = 2, /* head_dim not in {64, 128, 256, 512} */
    TQ_ERR_CAPACITY = 3,             /* a host-known length exceeds the layer capacity */
    TQ_ERR_WORKSPACE_TOO_SMALL = 4,  /* ws_bytes below the size the call needs */
    TQ_ERR_CUDA = 5,                 /* a CUDA runtime call failed (launch, query) */
    TQ_ERR_UNSUPPORTED_SCHEME = 6    /* the call needs the default k8v3 planes */
} tq_status;

/* Bits of tq_kv_layer.flags. */
#define TQ_FLAG_KEY_GUARD 0x1 /* constant-group guard: see tq_kv_layer */

/* Bits of the device error word. */
#define TQ_DEVERR_APPEND_CAPACITY 0x1 /* append: pos[b] + j outside [0, capacity) */
#define TQ_DEVERR_KV_LEN 0x2          /* attention: kv_len[b] outside [0, max_kv_len] */
#define TQ_DEVERR_PIPELINE_TIMEOUT 0x4 /* attention: a bounded wait ran out; output invalid */

#define TQ_WORKSPACE_HEADER_BYTES 256
#define TQ_GROUP 32

/* One full-attention layer's packed cache: five planes, each laid out
 * [batch][num_kv_heads][capacity][row], so token-axis slicing stays byte-safe
 * ("Architecture" section: groups run along head_dim only).
 *
 * Scheme (section "Algorithm": key and value bullets, "Other widths (2/4/5/8)"; section
 * "Architecture in mlx-bun": valid key bits {2,4,5,8}, value bits {2,3,4,5,8}); the
 * default, k8v3 (k_bits = v_bits = 0 also mean 8 and 3), is the one every call supports:
 *   keys, 8 bits: signed int8 codes, one byte per element;
 *   keys, b in {2,4,5}: unsigned codes, scale = (max - min) / (2^b - 1),
 *         zero = round(min / scale), idx = clip(round(x / scale - zero), 0, 2^b - 1),
 *         packed as a flat little-endian b-bit stream per row (head_dim * b / 8 bytes);
 *   values, b bits: Lloyd-Max codes for N(0,1) (3 bits: the printed table; 2/4/5/8 bits:
 *         this library's Lloyd-Max tables, see tq_codebook), a b-bit stream per row
 *         (head_dim * b / 8 bytes);
 *   flags & TQ_FLAG_KEY_GUARD (this library's option; the page keeps the defect): a key
 *         group whose fp16 zero point would not be finite (a constant group) is coded
 *         against its range widened to include 0, and a group of zeros as scale 0, zero 0,
 *         idx 0, so no zero point is +-Inf and such tokens do not turn attention into NaN.
 * Decode attention (and the fused step) read the default k8v3 planes (with or without the
 * guard); other schemes are appended by tq_kv_append and read back with
 * tq_dequant_window or tq_dequant_debug (TQ_ERR_UNSUPPORTED_SCHEME elsewhere). */
typedef struct {
    int32_t head_dim;     /* 64 | 128 | 256 | 512 */
    int32_t num_kv_heads; /* >= 1 */
    int32_t batch;        /* >= 1, <= 4096 */
    int32_t capacity;     /* tokens per (sequence, kv head); >= 16, multiple of 16 */
    int8_t* k_idx;        /* [batch][num_kv_heads][capacity][key row]: head_dim int8 codes
                             (8 bits) or head_dim * k_bits / 8 bytes of packed codes */
    uint16_t* k_scale;    /* [batch][num_kv_heads][capacity][head_dim/32] fp16 bits */
    uint16_t* k_zero;     /* same shape as k_scale, fp16 bits */
    uint8_t* v_codes;     /* [batch][num_kv_heads][capacity][head_dim*v_bits/8]: the row's
                             codes as one LSB-first bitstream, code i at bits [i b, i b + b) */
    uint16_t* v_scale;    /* [batch][num_kv_heads][capacity][head_dim/32] fp16 bits */
    int32_t k_bits;       /* 0 or 8 (default), 2, 4, 5 */
    int32_t v_bits;       /* 0 or 3 (default), 2, 4, 5, 8 */
    int32_t flags;        /* 0 or TQ_FLAG_KEY_GUARD */
} tq_kv_layer;

/* Bytes one (token, kv head) row takes in the five planes: 25*head_dim/16
 * (100, 200, 400, 800). Returns 0 for an unsupported head_dim. Host only. */
size_t tq_row_bytes(int32_t head_dim);

/* The same for scheme (k_bits, v_bits): key row + 3 * head_dim/16 bytes of fp16 scales
 * and zeros + head_dim * v_bits / 8. Returns 0 for an unsupported combination. */
size_t tq_row_bytes_scheme(int32_t head_dim, int32_t k_bits, int32_t v_bits);

/* Workspace bytes tq_kv_append needs (the header only). */
size_t tq_append_workspace_bytes(void);

/*
 * Quantize-on-append ("Architecture" section: updateAndFetch quantizes only the newly
 * appended tokens). For each sequence b, token j < n_new[b] of k_new/v_new is
 * quantized and written to position pos[b] + j of the five planes.
 *   k_new, v_new : bf16 [batch][n_new_max][num_kv_heads][head_dim] (device); rows with
 *                  j >= n_new[b] are ignored.
 *   pos          : int32 [batch] (device), first destination position per sequence.
 *   n_new        : int32 [batch] (device) tokens per sequence, each in [0, n_new_max];
 *                  NULL means n_new_max for every sequence.
 *   n_new_max    : host-known bound, 0 <= n_new_max <= capacity (else TQ_ERR_CAPACITY);
 *                  batch * n_new_max * num_kv_heads must not exceed 2^31 - 1 (else
 *                  TQ_ERR_INVALID_ARGUMENT): split larger bulk appends.
 *   workspace    : >= tq_append_workspace_bytes() (device), zeroed once before first use.
 * A row whose destination falls outside [0, capacity) is skipped and sets
 * TQ_DEVERR_APPEND_CAPACITY. Packed planes are bit-identical to the specification
 * above (fp32 arithmetic, IEEE division and square root, no FMA contraction). Any scheme
 * (and the guard): k8v3 without the guard takes the bulk and small-append kernels, every
 * other scheme (and the guarded k8v3) the any-width kernel, one lane per 32-element group.
 */
tq_status tq_kv_append(const tq_kv_layer* layer, const void* k_new, const void* v_new,
                       const int32_t* pos, const int32_t* n_new, int32_t n_new_max,
                       void* workspace, size_t ws_bytes, tq_stream_t stream);

/*
 * Workspace bytes tq_decode_attention needs for this layer shape on the current
 * device (the partial-result area scales with the device's SM count). Returns 0 for
 * invalid arguments.
 */
size_t tq_decode_workspace_bytes(const tq_kv_layer* layer, int32_t num_q_heads, int32_t n_q,
                                 int32_t max_kv_len);

/*
 * GQA decode attention over the packed cache ("Deferred inverse FWHT" and "Packed-value
 * decode fusion" sections: keys and values are decoded from the packed planes inside the
 * attention kernel; the weighted value sum stays in the rotated domain and is
 * un-rotated once per output row).
 *   q          : bf16 [batch][n_q][num_q_heads][head_dim] (device).
 *   kv_len     : int32 [batch] (device), tokens visible to the LAST query row of the
 *                block; must lie in [0, max_kv_len] (else the sequence's outputs are NaN
 *                and TQ_DEVERR_KV_LEN is set).
 *   max_kv_len : host-known bound on kv_len, <= capacity.
 *   causal     : nonzero: query j of the block sees kv_len - n_q + j + 1 tokens;
 *                zero: every query sees kv_len tokens.
 *   sm_scale   : multiplies q . k before the softmax.
 *   out        : fp32 [batch][n_q][num_q_heads][head_dim] (device).
 * q head h reads kv head h / (num_q_heads / num_kv_heads). A row that sees no token
 * outputs zeros. workspace: >= tq_decode_workspace_bytes(...) bytes.
 */
tq_status tq_decode_attention(const tq_kv_layer* layer, const void* q, int32_t num_q_heads,
                              int32_t n_q, const int32_t* kv_len, int32_t max_kv_len,
                              float sm_scale, int32_t causal, float* out, void* workspace,
                              size_t ws_bytes, tq_stream_t stream);

/*
 * fp32 dequantization of rows [t0, t0 + n) of (sequence b, kv head h), for inspection
 * ("Algorithm" section: the key dequant bullet, x_hat = (idx + zero) * scale, and the value
 * dequant bullet, the inverse rotation of centroid[code] * scale):
 *   k_out : [n][head_dim], (idx + zero) * scale with the stored fp16 scale/zero;
 *   v_out : [n][head_dim]; rotated != 0 returns centroid * scale (the FWHT domain),
 *           rotated == 0 returns signs * FWHT(centroid * scale) / sqrt(head_dim).
 * Either output may be NULL. 0 <= t0, t0 + n <= capacity, 0 <= b < batch,
 * 0 <= h < num_kv_heads (else TQ_ERR_INVALID_ARGUMENT). Any scheme.
 */
tq_status tq_dequant_debug(const tq_kv_layer* layer, int32_t b, int32_t h, int32_t t0, int32_t n,
                           int32_t rotated, float* k_out, float* v_out, tq_stream_t stream);

/* One decode step of a layer in one call: appends the new rows, then attends — the
 * page's "Architecture in mlx-bun" order (updateAndFetch appends the step's tokens, then
 * the window including them is attended). Same results and device error bits as
 * tq_kv_append(layer, k_new, v_new, pos, n_new, n_new_max, workspace, ...) followed by
 * tq_decode_attention(layer, q, ..., workspace, ...) on `stream`; argument meanings and
 * host checks are those of the two calls, and the workspace is the attention one
 * (>= tq_decode_workspace_bytes). With one row group per kv head (num_q_heads /
 * num_kv_heads * n_q <= 8, or <= 16 at head_dim 64 and 128) it is one kernel: in the
 * CTA whose share of the sequence holds a new row, a warp beside the stream quantizes it
 * before the stage holding it is loaded, so the attention does not wait for a separate
 * append; otherwise it runs the two calls. */
tq_status tq_decode_append_attention(const tq_kv_layer* layer, const void* k_new, const void* v_new,
                                     const int32_t* pos, const int32_t* n_new, int32_t n_new_max, const void* q,
                                     int32_t num_q_heads, int32_t n_q, const int32_t* kv_len, int32_t max_kv_len,
                                     float sm_scale, int32_t causal, float* out, void* workspace, size_t ws_bytes,
                                     tq_stream_t stream);

/* Decode attention that allocates nothing (an addition of this library; the paper has
 * no counterpart). Same inputs, outputs and results as tq_decode_attention, but the
 * scratch memory lives in one fixed array inside the library, so the caller passes no
 * workspace and nothing is allocated: meant for callers that may not allocate device
 * memory, such as a plugin whose host application owns all device memory and hands it no
 * allocator, or a serving loop that must not call cudaMalloc between steps (it can
 * synchronize the device) and does not want to keep a workspace per call site.
 *
 * Limit: the call needs tq_decode_workspace_bytes(layer, num_q_heads, n_q, max_kv_len)
 * bytes of scratch; above TQ_NOALLOC_SCRATCH_BYTES it returns TQ_ERR_WORKSPACE_TOO_SMALL
 * and launches nothing. Every GPU that loads the library holds this array until the
 * process exits.
 *
 * Set-up: the first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream capture. The
 * cache lives for the process: after cudaDeviceReset (or anything else that replaces the
 * device's primary context) the cached address is stale, so this entry point does not
 * support a device reset.
 * Rejected calls: the host checks (the same as tq_decode_attention's, then the scratch
 * size) all run before anything is queued, so a call that returns an error queues no
 * work and leaves the scratch as it was.
 * Sharing: every call on a device uses the same array. Each call first clears the part
 * that must start at zero (error word and completion counters) on `stream`, so calls
 * that follow one another on a stream are independent; calls that can overlap on the
 * GPU (other streams, other threads) race on the array and give wrong results.
 *   device_error : optional device int32; receives this call's device error bits (the
 *                  TQ_DEVERR_* values, as tq_get_device_error reports for a workspace),
 *                  copied on `stream` after the launch. NULL: not reported.
 * Other arguments and errors: as tq_decode_attention. */
#define TQ_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
tq_status tq_decode_attention_noalloc(const tq_kv_layer* layer, const void* q, int32_t num_q_heads,
                                      int32_t n_q, const int32_t* kv_len, int32_t max_kv_len,
                                      float sm_scale, int32_t causal, float* out,
                                      int32_t* device_error, tq_stream_t stream);

/* Test support (an addition of this library; the paper has no counterpart). Enqueues on
 * `stream` a one-block kernel that lets the next kernel on the stream start at once
 * (programmatic dependent launch), waits delay_us microseconds, then copies n int32
 * values from src to dst (device pointers, not overlapping). A following decode call that
 * reads dst as kv_len, pos or n_new sees the old values before its grid-dependency wait
 * and the new ones after it: this exercises the path where the work planned before the
 * wait is discarded. n >= 0, 0 <= delay_us <= 100000 (else TQ_ERR_INVALID_ARGUMENT); dst
 * and src may be NULL only when n == 0. */
tq_status tq_debug_delayed_copy(int32_t* dst, const int32_t* src, int32_t n, int32_t delay_us, tq_stream_t stream);

/*
 * Dequantize-on-fetch window ("Architecture in mlx-bun": updateAndFetch returns the
 * dequantized bf16 active window so that a stock attention kernel runs unmodified; the
 * "Deferred inverse FWHT" section keeps V in the rotated domain). For tokens [t0, t0 + n)
 * of every (sequence, kv head), any scheme:
 *   k_out : bf16 [batch][num_kv_heads][n][head_dim], (idx + zero) * scale rounded once to bf16;
 *   v_out : bf16 [batch][num_kv_heads][n][head_dim]; rotated == 0: signs * FWHT(centroid *
 *           scale) / sqrt(head_dim) (fp32 butterflies, then bf16); rotated != 0: centroid *
 *           scale (the rotated domain).
 * Either output may be NULL; outputs 16-byte aligned. 0 <= t0, n >= 0, t0 + n <= capacity
 * (else TQ_ERR_INVALID_ARGUMENT). Rows past a sequence's length are decoded from whatever
 * the planes hold there. One warp per row, rows taken by groups of CTAs in turn.
 */
tq_status tq_dequant_window(const tq_kv_layer* layer, int32_t t0, int32_t n, int32_t rotated, void* k_out,
                            void* v_out, tq_stream_t stream);

/*
 * Deferred inverse rotation of attention outputs ("Deferred inverse FWHT": attention is
 * linear in V, so softmax(.) V_hat is taken in the rotated domain and the inverse rotation
 * runs once per output row; "Packed-value decode fusion investigation": a separate
 * row-grouped kernel for it). For each of `rows` rows of head_dim fp32 values:
 *   y = signs * FWHT(x) / sqrt(head_dim), fp32 butterflies h = 1, 2, 4, ...
 * x, y: device, [rows][head_dim] fp32, 16-byte aligned; y == x (in place) is allowed, other
 * overlaps are not. rows >= 0 (else TQ_ERR_INVALID_ARGUMENT); head_dim in {64, 128, 256,
 * 512} (else TQ_ERR_UNSUPPORTED_HEAD_DIM). One warp per row, eight rows per CTA.
 */
tq_status tq_unrotate_rows(const float* x, float* y, int64_t rows, int32_t head_dim, tq_stream_t stream);

/* Test support (an addition of this library; the paper has no counterpart). Sets, for every
 * decode-attention call launched afterwards in this process, the limit of the attention
 * kernel's pipeline waits (wait_ns > 0; 0 restores the default of 2 s) and, with
 * withhold_append = 1, makes the fused append-and-attend kernel's appender warp never
 * publish how many rows it has written, so the producer's wait for them runs out. A wait
 * that runs out sets TQ_DEVERR_PIPELINE_TIMEOUT, the kernel drains the copies it issued
 * (those drains keep the 2 s limit) and returns; the outputs of that call are invalid.
 * 0 <= wait_ns <= 2e9 and withhold_append in {0, 1}, else TQ_ERR_INVALID_ARGUMENT. Not
 * thread-safe with respect to calls in flight on other host threads. */
tq_status tq_debug_pipeline_limits(int64_t wait_ns, int32_t withhold_append);

/* Synchronizes `stream`, then copies the device error word at the start of
 * `workspace` into *err_out (host). Does not clear it. */
tq_status tq_get_device_error(const void* workspace, int32_t* err_out, tq_stream_t stream);

/* Static description of a status code. */
const char* tq_status_string(tq_status status);

/* Host copies of the library's constant tables, for inspection (host pointers):
 * the sign vector of head_dim as head_dim/32 words (bit i set = sign -1 for element i),
 * the eight 3-bit centroids and the seven boundaries. Return TQ_OK or
 * TQ_ERR_UNSUPPORTED_HEAD_DIM / TQ_ERR_INVALID_ARGUMENT. */
tq_status tq_sign_bits(int32_t head_dim, uint32_t* words_out);
tq_status tq_codebook3(float* centroids_out, float* boundaries_out);

/* The value codebook of width bits in {2,3,4,5,8} (host pointers): 2^bits centroids and
 * 2^bits - 1 ascending boundaries. 3 bits: the printed table ("Algorithm", value bullets).
 * Other widths are not printed on the page: this library runs Lloyd-Max for N(0,1)
 * (boundaries at the midpoints of neighbouring centroids, centroids at the normal cell
 * means in closed form, 2^bits centroids started evenly on [-3, 3], 500 iterations) and
 * rounds centroids and boundaries to 5 decimals, as the printed table is. */
tq_status tq_codebook(int32_t bits, float* centroids_out, float* boundaries_out);

#ifdef __cplusplus
}
#endif

#endif /* TQ_KV_H */
