/*
 * fa3.h -- C ABI of the GB300 (sm_103a) per-head INT8 attention-quantization
 * library (libfa3.so).
 *
 * The library implements the data-parallel hot path of "FA3" activation
 * quantization as described by msModelSlim's algorithm page
 * ("FA3量化：Flash Attention 3激活量化算法说明", section 原理 / 算法流程) and used by
 * MindIE ("FA3 quantization" and "Attention Quantization", Overview):
 *   - per-head Recall-Window calibration with a running min/max,
 *   - symmetric per-head INT8 parameters and quantize-on-append,
 *   - decode-phase attention that reads the INT8 KV cache directly
 *     (absorbed MLA with a bf16 RoPE key, and GQA with INT8 q/k/v).
 *
 * Conventions shared by every call:
 *   - Array arguments are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or synchronizes; every call only enqueues work on
 *     `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *     stream) and returns.
 *   - bf16 data is passed as uint16_t bit patterns.
 *   - The return value is an fa3_status.  Host-side validation (null
 *     pointers, sizes, alignment, options) happens before anything is
 *     enqueued: on any error other than FA3_ECUDA nothing was enqueued.
 *   - Errors that depend on device data (an append position, a context
 *     length) cannot be seen on the host.  Kernels OR the FA3_DEVERR_* bits
 *     into the optional caller-owned device word `dev_err` (int32, may be
 *     NULL) and skip the offending row; the caller reads the word when it
 *     likes.  Kernels never trap and every wait inside them is bounded.
 *   - Calls on the same stream are ordered; calls that share a workspace
 *     must not run concurrently on different streams.  The library's kernels
 *     are launched as programmatic dependents of the work before them on the
 *     stream (their launch overlaps its tail), and each waits for that work to
 *     complete before it reads or writes memory, so stream order holds for
 *     every buffer a caller passes.
 */
#ifndef FA3_H_
#define FA3_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum fa3_status {
  FA3_OK = 0,
  FA3_EINVAL = 1,       /* null pointer, non-positive size, bad option            */
  FA3_ERANGE = 2,       /* a size or alignment outside what the kernels support    */
  FA3_ECUDA = 3,        /* the CUDA runtime reported an error while enqueuing      */
  FA3_EWORKSPACE = 4,   /* workspace pointer NULL or smaller than required         */
  FA3_EDEVICE = 5       /* current device is not an sm_103 (GB300-class) GPU       */
};

/* Bits written into the optional device error word. */
#define FA3_DEVERR_POS 1      /* append: pos[b] < 0 or pos[b] + T_new > T_max (row skipped)    */
#define FA3_DEVERR_LENS 2     /* decode: lens[b] < 0 or lens[b] > T_max (output row set to 0) */
#define FA3_DEVERR_TIMEOUT 4  /* a bounded wait inside a kernel gave up (output not valid)    */
#define FA3_DEVERR_PAGE 8     /* paged calls: a block-table entry outside [0, num_pages)       */
#define FA3_DEVERR_CALIB 16   /* float32 calibration: a head's tail counts disagreed (non-finite
                                 input); that head's range is left unchanged                  */

/* Human-readable name of a status code (static string). */
const char* fa3_status_string(int status);

/* Library ABI version (major*100 + minor). */
int fa3_version(void);

/* Measurement aid (no counterpart in the pages).  When both events are
 * non-NULL, every later call of fa3_decode_attn_mla, fa3_decode_attn_gqa,
 * fa3_prefill_attn_gqa and fa3_calibrate_perhead records start_event on its
 * stream just before its main kernel (the MLA decode, the GQA decode, the
 * prefill attention, the calibration's pass over its input) and
 * stop_event just after it, so that the caller can time that kernel alone
 * (cudaEventElapsedTime).  The events are cudaEvent_t passed as void*, owned
 * by the caller and must outlive their use; NULL, NULL turns this off.  One
 * setting for the whole process, not synchronized between host threads.
 * Returns FA3_EINVAL when exactly one of the two is NULL. */
int fa3_set_kernel_timing(void* start_event, void* stop_event);

/* ------------------------------------------------------------------------
 * Calibration -- msModelSlim FA3量化, 原理 / 算法流程 steps 1-3.
 *
 * Step 1: every head h collects the N = B*L values x[b, h, 0..L) of all b
 *   (L = S*D for an activation of shape (B, H, S, D)).
 * Step 2 (Recall Window): sort the N values, target_num = int(ratio * N)
 *   (float64 product, truncated, at least 1), and among the windows
 *   [sorted[i], sorted[i + target_num - 1]], i = 0 .. N - target_num, take
 *   the narrowest (exact width: the true difference of the two values, not
 *   a rounded one; ties -> smallest i).
 * Step 3: min_io[h] = min(min_io[h], lo[h]), max_io[h] = max(max_io[h], hi[h]).
 *   -0.0 orders before +0.0 in both the sort and the min/max.
 *
 * x        bf16 values; element (b, h, l) at x[b*stride_b + h*stride_h + l]
 *          (strides in elements; l is contiguous).  Values must be finite and
 *          of magnitude below 2^127, so that every window width is below the
 *          largest float (not checked).
 * B, H, L  B >= 1, 1 <= H, L >= 1, B*L < 2^32.
 * ratio    in (0, 1]; the pages' default is 0.9999.
 * min_io, max_io  float[H], in/out.  Initialise to +inf / -inf before the
 *          first batch; pass them back unchanged to accumulate more batches.
 * workspace  device buffer of fa3_calibrate_workspace_size(H) bytes, 256-byte
 *          aligned, ZERO-FILLED before its first use.  Every successful call
 *          leaves it zero-filled again, so it can be reused without clearing,
 *          also by a call with another H.  (After an FA3_ECUDA error, zero it
 *          again.)
 * Results are exact: the same bits as the sorted definition above.
 * ------------------------------------------------------------------------ */
size_t fa3_calibrate_workspace_size(int H);

int fa3_calibrate_perhead(const uint16_t* x, int64_t B, int H, int64_t L,
                          int64_t stride_b, int64_t stride_h, double ratio,
                          float* min_io, float* max_io,
                          void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Calibration of float32 activations -- the same steps and readings as
 * fa3_calibrate_perhead (msModelSlim FA3量化, 原理 / 算法流程 steps 1-3) for
 * float32 input: x float32, element (b, h, l) at x[b*stride_b + h*stride_h + l].
 * Supported: N - target_num + 1 <= 4096 window starts (the pages' ratio 0.9999
 * keeps that up to N = 40.96 million values per head), N < 2^31, H <= 65535;
 * values finite with magnitude below 2^127 (not checked: a head whose internal
 * counts then disagree sets FA3_DEVERR_CALIB and keeps its range).
 * workspace  fa3_calibrate_f32_workspace_size(H) bytes, 16-byte aligned,
 *            ZERO-FILLED before its first use; every call leaves it zeroed.
 * ------------------------------------------------------------------------ */
size_t fa3_calibrate_f32_workspace_size(int H);

int fa3_calibrate_perhead_f32(const float* x, int64_t B, int H, int64_t L,
                              int64_t stride_b, int64_t stride_h, double ratio,
                              float* min_io, float* max_io, void* workspace, size_t workspace_bytes,
                              int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Running-range merge -- msModelSlim FA3量化, 原理 / 算法流程 step 3 applied to
 * R ranges at once (e.g. the ranges that R ranks computed on their shares of
 * the calibration batches, gathered by the caller's collective):
 *   min_io[h] = min(min_io[h], mins[r][h]),  max_io[h] = max(max_io[h], maxs[r][h])
 * over r = 0 .. R-1, in IEEE totalOrder (-0.0 below +0.0).  min and max are
 * associative and commutative, so sharding the batches over ranks and merging
 * gives the same bits as accumulating every batch in one process.
 * mins, maxs  float [R][H], device;  min_io, max_io  float[H], in/out.
 * ------------------------------------------------------------------------ */
int fa3_range_merge(const float* mins, const float* maxs, int R, int H, float* min_io, float* max_io,
                    void* stream);

/* ------------------------------------------------------------------------
 * Quantization parameters -- msModelSlim FA3量化, 原理 / 算法流程 step 4:
 *   abs_max[h] = max(|min[h]|, |max[h]|);  scale[h] = abs_max[h] / 127
 * (one IEEE float32 division).  min, max, scale: float[H].
 * ------------------------------------------------------------------------ */
int fa3_qparams(const float* min_v, const float* max_v, float* scale, int H, void* stream);

/* ------------------------------------------------------------------------
 * Quantize-on-append -- the input_scale step of MindIE "FA3 quantization" /
 * "Attention Quantization" (Overview): activations become INT8 codes
 *   q = clamp(round_half_even(x / scale[h]), -127, 127)     (scale 0 -> 0)
 * with x / scale one IEEE float32 division.
 *
 * kv       bf16 [B][T_new][H][D] new rows.
 * scale    float[H].
 * cache    int8 [B][T_max][H][D]; row t of sequence b goes to position
 *          pos[b] + t.  Other rows are untouched.
 * pos      int32[B] device array.  A sequence with pos[b] < 0 or
 *          pos[b] + T_new > T_max is skipped and FA3_DEVERR_POS is set.
 * rope_src, rope_cache, Dr  optional pass-through of the unquantized RoPE key
 *          of MLA ("FA3 quantization", Overview: the RoPE part of K is not
 *          quantized): bf16 [B][T_new][Dr] copied to bf16 [B][T_max][Dr] at
 *          the same positions.  Pass NULL, NULL, 0 to skip.
 * Also used to quantize a GQA query: T_new = T_max = 1 and pos = 0.
 * ------------------------------------------------------------------------ */
int fa3_quantize_append(const uint16_t* kv, const float* scale, int8_t* cache, const int32_t* pos,
                        int B, int T_new, int H, int D, int T_max,
                        const uint16_t* rope_src, uint16_t* rope_cache, int Dr,
                        int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Per-channel parameters -- MindIE Turbo "Attention量化", 表1 / 表2: scale and
 * offset tensors of shape [head_num, head_dim], one pair per (head, channel).
 * The pages give the tensors' shapes, not the arithmetic; this library takes
 * the plain readings below (float32 IEEE operations throughout):
 *   symmetric   scale = max(|min|, |max|) / 127,  offset = 0
 *               q = clamp(round_half_even(x / scale), -127, 127)
 *   asymmetric  [lo, hi] = [min(min, 0), max(max, 0)]  (0 stays exact)
 *               scale = (hi - lo) / 255,  offset = round_half_even(-lo / scale) - 128
 *               q = clamp(round_half_even(x / scale) + offset, -128, 127)
 *               dequantized value (q - offset) * scale
 * scale = 0 (an all-zero channel) gives offset 0 and code 0 (symmetric) or
 * offset (asymmetric).  min / max must be finite.
 * ------------------------------------------------------------------------ */

/* Per-channel Recall-Window calibration: msModelSlim FA3量化 算法流程 steps 2-3
 * on each (head, channel) -- the N = B*S values x[b, h, s, d] of channel d of
 * head h -- with the per-head call's readings (target_num = int(ratio * N),
 * exact widths, ties to the smallest start, totalOrder running min/max).
 * x        bf16; element (b, h, s, d) at x[b*stride_b + h*stride_h + s*stride_s + d].
 * min_io, max_io  float [H][D], in/out (start at +inf / -inf).
 * Supported: N - target_num + 1 <= 32 window starts (FA3_ERANGE otherwise),
 *            H <= 65535.  No workspace. */
int fa3_calibrate_perchannel(const uint16_t* x, int64_t B, int H, int64_t S, int D,
                             int64_t stride_b, int64_t stride_h, int64_t stride_s, double ratio,
                             float* min_io, float* max_io, void* stream);

/* min_v, max_v, scale, offset: float[n] (n = heads * head_dim), device. */
int fa3_qparams_channel(const float* min_v, const float* max_v, int n, int asymmetric,
                        float* scale, float* offset, void* stream);

/* Quantize-on-append with per-channel parameters (fa3_quantize_append's layout).
 * kv bf16 [B][T_new][H][D]; scale, offset float [H][D] (offset may be NULL when
 * asymmetric is 0); cache int8 [B][T_max][H][D] written at pos[b] + t.
 * Supported: D % 8 == 0; kv, scale, offset 16-byte aligned, cache 8-byte aligned.
 * A sequence with pos[b] < 0 or pos[b] + T_new > T_max is skipped and sets
 * FA3_DEVERR_POS. */
int fa3_quantize_append_channel(const uint16_t* kv, const float* scale, const float* offset,
                                int asymmetric, int8_t* cache, const int32_t* pos,
                                int B, int T_new, int H, int D, int T_max, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Absorbed-MLA decode attention over an INT8 latent cache -- MindIE
 * "FA3 quantization", Overview (non-RoPE K quantized to 8 bits per head,
 * RoPE K left unquantized; decode-phase attention reads the INT8 cache),
 * with the per-head scales of msModelSlim FA3量化 step 4.
 *
 * For every sequence b and head h (one decoded query token):
 *   q8[h]   = quantize(q[b, h, 0:Dl], q_scale[h])          (the latent query)
 *   acc[j]  = sum_c q8[h, c] * ckv[b, j, c]                 (exact integer)
 *   s[j]    = (acc[j] * q_scale[h] * kv_scale[0] + q[b, h, Dl:] . krope[b, j, :])
 *             * softmax_scale,                  j < lens[b]
 *   out[b, h, :] = kv_scale[0] * sum_j softmax(s)_j * ckv[b, j, :]
 *
 * q        bf16 [B][H][Dl + Dr] (latent part first).
 * ckv      int8 [B][T_max][Dl] latent cache (shared K-nope / V), one KV head.
 * krope    bf16 [B][T_max][Dr] RoPE key.
 * q_scale  float[H];  kv_scale float[1].
 * lens     int32[B]; 0 gives a zero row; < 0 or > T_max sets FA3_DEVERR_LENS.
 * out      float32 [B][H][Dl].
 * Supported: H <= 128, Dl in {64, 128, ..., 512} (multiple of 64),
 *            Dr a multiple of 16 up to 64, T_max >= 1; ckv/krope rows 16-byte
 *            aligned (Dl % 16 == 0, Dr % 8 == 0).
 * workspace  fa3_mla_workspace_size(B, H, Dl, T_max) bytes (split-K partials).
 * ------------------------------------------------------------------------ */
size_t fa3_mla_workspace_size(int B, int H, int Dl, int T_max);

int fa3_decode_attn_mla(const uint16_t* q, const int8_t* ckv, const uint16_t* krope,
                        const float* q_scale, const float* kv_scale, const int32_t* lens,
                        float* out, int B, int H, int Dl, int Dr, int T_max, float softmax_scale,
                        void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * GQA decode attention with INT8 q, k and v -- MindIE "Attention
 * Quantization", Overview, and MindIE Turbo "Attention量化" (q, k, v all
 * 8-bit; deq_scale brings the result back to floating point).
 *
 * Query head h reads KV head g = h / (Hq / Hkv):
 *   s[j] = (q[b, h] . k[b, j, g]) * q_scale[h] * k_scale[g] * softmax_scale
 *   out[b, h, :] = bf16( v_scale[g] * sum_j softmax(s)_j * v[b, j, g, :] ),  j < lens[b]
 *
 * q        int8 [B][Hq][D];  k, v  int8 [B][T_max][Hkv][D].
 * q_scale  float[Hq];  k_scale, v_scale  float[Hkv].
 * lens     int32[B] (as for MLA).   out  bf16 [B][Hq][D].
 * Supported: D = 128, 1 <= Hq / Hkv <= 8; 16-byte aligned rows.
 * workspace  fa3_gqa_workspace_size(B, Hq, Hkv, D, T_max) bytes.
 * ------------------------------------------------------------------------ */
size_t fa3_gqa_workspace_size(int B, int Hq, int Hkv, int D, int T_max);

int fa3_decode_attn_gqa(const int8_t* q, const int8_t* k, const int8_t* v,
                        const float* q_scale, const float* k_scale, const float* v_scale,
                        const int32_t* lens, uint16_t* out, int B, int Hq, int Hkv, int D, int T_max,
                        float softmax_scale, void* workspace, size_t workspace_bytes,
                        int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * GQA decode with per-channel (asymmetric) INT8 q, k and v -- MindIE Turbo
 * "Attention量化", 表1 / 表2 (q/k/v_scale and q/k/v_offset, [heads][head_dim]),
 * with the dequantization of fa3_qparams_channel: x = (code - offset) * scale.
 *   s[j] = sum_d xq[d] * xk_j[d] * softmax_scale,  out = bf16( sum_j softmax(s)_j * xv_j )
 * q_scale, q_offset float [Hq][D]; k_scale, k_offset, v_scale, v_offset float [Hkv][D].
 * k_offset moves every score of a row by the same amount, which the softmax
 * removes: it must be passed and is not read.  Other arguments, layouts,
 * limits and the workspace (fa3_gqa_workspace_size) as fa3_decode_attn_gqa.
 * ------------------------------------------------------------------------ */
int fa3_decode_attn_gqa_channel(const int8_t* q, const int8_t* k, const int8_t* v,
                                const float* q_scale, const float* q_offset,
                                const float* k_scale, const float* k_offset,
                                const float* v_scale, const float* v_offset,
                                const int32_t* lens, uint16_t* out, int B, int Hq, int Hkv, int D, int T_max,
                                float softmax_scale, void* workspace, size_t workspace_bytes,
                                int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Prefill-phase GQA attention with INT8 q, k and v -- MindIE "Attention
 * Quantization", Overview, and MindIE Turbo "Attention量化" (q, k, v all 8-bit
 * with per-head scales; deq_scale restores floating point); at long sequence
 * lengths these activations dominate memory (msModelSlim "FA3量化", 简介).
 *
 * The q_lens[b] new rows of sequence b are the last tokens of its kv_lens[b]-
 * token context (kv_lens[b] - q_lens[b] cached tokens, then the new rows); new
 * row i sits at position pos = kv_lens[b] - q_lens[b] + i and attends causally
 * to keys 0 .. pos.  Query head h reads KV head g = h / (Hq / Hkv):
 *   s[t] = (q[b, i, h] . k[b, t, g]) * q_scale[h] * k_scale[g] * softmax_scale
 *   out[b, i, h, :] = bf16( v_scale[g] * sum_{t <= pos} softmax(s)_t * v[b, t, g, :] )
 *
 * q        int8 [B][S][Hq][D] (rows i >= q_lens[b] are not read).
 * k, v     int8 [B][T][Hkv][D] (rows t >= kv_lens[b] are not read).
 * q_scale  float[Hq];  k_scale, v_scale  float[Hkv].
 * q_lens, kv_lens  int32[B]; 0 <= q_lens[b] <= S and q_lens[b] <= kv_lens[b] <= T,
 *          otherwise FA3_DEVERR_LENS is set and sequence b is skipped.
 * out      bf16 [B][S][Hq][D]; rows i >= q_lens[b] are left untouched.
 * Supported: D = 128, Hq / Hkv dividing 128; 16-byte aligned q, k, v, out.
 * No workspace.
 * ------------------------------------------------------------------------ */
int fa3_prefill_attn_gqa(const int8_t* q, const int8_t* k, const int8_t* v,
                         const float* q_scale, const float* k_scale, const float* v_scale,
                         const int32_t* q_lens, const int32_t* kv_lens, uint16_t* out,
                         int B, int S, int T, int Hq, int Hkv, int D, float softmax_scale,
                         int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Allocation-free GQA decode.  No counterpart in the pages: a convenience for
 * callers that cannot allocate device memory when they run attention (code
 * inside an allocator or memory-pool callback, runtimes that plan every
 * allocation ahead of time, deployments that forbid allocation after start-up).
 *
 * Same arguments and results as fa3_decode_attn_gqa, without the workspace:
 * the split-K partials go to a fixed 8 MiB array in the library's own device
 * memory, which every GPU that loads libfa3.so holds until the process exits.
 * Sizes whose partials would need more than 8 MiB (fa3_gqa_workspace_size() >
 * 8 MiB) return FA3_EWORKSPACE; the split plan (at most one wave of resident
 * CTAs, 4 KB of partials each) keeps every size below 2 MiB on GB300.
 * The first call on each device looks up the array's device address (this
 * may initialise the module on that device): make that first call before any
 * stream capture.  All calls share the one array and it keeps the last call's
 * contents (nothing in it needs to start at zero); calls that overlap on the
 * GPU -- on different streams, or from different host threads -- race on it.
 * ------------------------------------------------------------------------ */
int fa3_decode_attn_gqa_noalloc(const int8_t* q, const int8_t* k, const int8_t* v,
                                const float* q_scale, const float* k_scale, const float* v_scale,
                                const int32_t* lens, uint16_t* out, int B, int Hq, int Hkv, int D, int T_max,
                                float softmax_scale, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Paged INT8 KV cache.  The pages leave the KV cache's storage to the serving
 * runtime (MindIE "FA3 quantization", usage steps: the runtime is told which
 * format to keep the cache in); these calls take the block-table layout of
 * paged serving runtimes.  The cache of every sequence is a list of pages of
 * page_size token rows in one pool shared by all sequences:
 *   block_table  int32 [B][max_pages], device; entry i of sequence b is the
 *                pool page that holds that sequence's tokens
 *                [i * page_size, (i + 1) * page_size).
 *   num_pages    pages in the pool; the per-sequence capacity is
 *                T_max = max_pages * page_size.
 * Token t of sequence b lives in pool row
 *   block_table[b][t / page_size] * page_size + t % page_size,
 * so a pool is the contiguous [B][T_max] cache of the calls above with its
 * rows regrouped; results are exactly those of the contiguous call on the
 * gathered cache.  Only the entries a call needs are read (pages of tokens
 * below lens[b], or of the appended positions); such an entry outside
 * [0, num_pages) sets FA3_DEVERR_PAGE: the append skips that token row, the
 * decode reads that page as zeros (that sequence's output is not valid).
 * Pages may be shared between sequences (read-only prefixes).
 * ------------------------------------------------------------------------ */

/* Quantize-on-append into a paged cache (fa3_quantize_append's arithmetic).
 * cache      int8 [num_pages][page_size][H][D] pool.
 * rope_cache optional bf16 [num_pages][page_size][Dr] pool (NULL, NULL, 0 to skip).
 * Positions as for fa3_quantize_append with T_max = max_pages * page_size.
 * Supported: any page_size >= 1. */
int fa3_quantize_append_paged(const uint16_t* kv, const float* scale, int8_t* cache,
                              const int32_t* block_table, const int32_t* pos,
                              int B, int T_new, int H, int D, int num_pages, int page_size, int max_pages,
                              const uint16_t* rope_src, uint16_t* rope_cache, int Dr,
                              int32_t* dev_err, void* stream);

/* Absorbed-MLA decode over a paged cache (fa3_decode_attn_mla's arithmetic).
 * ckv    int8 [num_pages][page_size][Dl] pool;  krope  bf16 [num_pages][page_size][Dr] pool.
 * Supported: as fa3_decode_attn_mla, page_size a multiple of 64 (one 64-token
 * tile never spans two pages), num_pages * page_size < 2^31.
 * workspace  fa3_mla_workspace_size(B, H, Dl, max_pages * page_size) bytes. */
int fa3_decode_attn_mla_paged(const uint16_t* q, const int8_t* ckv, const uint16_t* krope,
                              const float* q_scale, const float* kv_scale, const int32_t* lens,
                              const int32_t* block_table, float* out, int B, int H, int Dl, int Dr,
                              int num_pages, int page_size, int max_pages, float softmax_scale,
                              void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream);

/* GQA decode over a paged cache (fa3_decode_attn_gqa's arithmetic).
 * k, v   int8 [num_pages][page_size][Hkv][D] pools.
 * Supported: as fa3_decode_attn_gqa, page_size a multiple of 16.
 * workspace  fa3_gqa_workspace_size(B, Hq, Hkv, D, max_pages * page_size) bytes. */
int fa3_decode_attn_gqa_paged(const int8_t* q, const int8_t* k, const int8_t* v,
                              const float* q_scale, const float* k_scale, const float* v_scale,
                              const int32_t* lens, const int32_t* block_table, uint16_t* out,
                              int B, int Hq, int Hkv, int D, int num_pages, int page_size, int max_pages,
                              float softmax_scale, void* workspace, size_t workspace_bytes,
                              int32_t* dev_err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA3_H_ */
