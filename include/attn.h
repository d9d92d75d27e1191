/*
 * Exact softmax attention for one GB300 GPU (sm_103a): C ABI.
 *
 * Two operations:
 *   attn_fwd           O = softmax(scale * Q K^T + mask) V and the per-row log-sum-exp,
 *                      tiled with the online-softmax recurrence so that the score matrix
 *                      never reaches device memory ("FlashAttention: not computing less,
 *                      moving less", sections 01-03; "FlashAttention-4: Blackwell
 *                      algorithm-pipeline co-design", all sections on the forward pass).
 *   attn_decode_paged  one query token per sequence against a paged KV cache, split over
 *                      the keys and merged by log-sum-exp ("Faster, more flexible FA4 for
 *                      LLM inference", PR 1999/2104, PR 1940, PR 2186 sections).
 *
 * Conventions shared by every entry point
 *  - All pointers named as device pointers must point to device memory of the current
 *    CUDA device; the caller owns every buffer and keeps it alive until the work on
 *    `stream` completes.
 *  - `stream` is a cudaStream_t passed as void* (NULL selects the legacy default stream).
 *    Every compute call is asynchronous on `stream` and never synchronises the host.
 *  - bf16 tensors are IEEE bfloat16 bit patterns; the innermost dimension (d) is
 *    contiguous. Results are identical to the exact definition up to floating-point
 *    rounding: fp32 accumulation of bf16 products, bf16 probabilities and bf16 output.
 *  - A call that returns an error code other than ATTN_ERR_CUDA has launched nothing and
 *    written nothing. Errors found by the device while a kernel runs (a timed-out wait,
 *    an out-of-range page index or sequence length) are recorded in a per-device status
 *    word read by attn_get_device_status(); kernels never trap.
 */
#ifndef EXACT_SOFTMAX_ATTENTION_GB300_ATTN_H
#define EXACT_SOFTMAX_ATTENTION_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int attn_status_t;

#define ATTN_OK 0
#define ATTN_ERR_NULL_PTR (-1)          /* a required pointer is NULL */
#define ATTN_ERR_BAD_SHAPE (-2)         /* unsupported or inconsistent sizes */
#define ATTN_ERR_ALIGN (-3)             /* a pointer is not aligned as documented */
#define ATTN_ERR_UNSUPPORTED_ARCH (-4)  /* the current device is not sm_103 */
#define ATTN_ERR_CUDA (-5)              /* a CUDA runtime or driver call failed */
#define ATTN_ERR_DEVICE_TIMEOUT (-6)    /* a kernel gave up on a pipeline wait (device status) */
#define ATTN_ERR_DEVICE_BAD_INDEX (-7)  /* a page index or sequence length was out of range (device status) */
#define ATTN_ERR_BAD_ARG (-8)           /* an unknown option name or an invalid value */
#define ATTN_ERR_SCRATCH_TOO_SMALL (-9) /* attn_decode_paged_noalloc: sizes exceed its fixed scratch */

/* 8-bit floating-point formats (OCP FP8) of attn_fwd_fp8 and attn_decode_paged_fp8 */
#define ATTN_FP8_E4M3 0 /* 4 exponent bits (bias 7), 3 mantissa bits, largest 448, no infinities */
#define ATTN_FP8_E5M2 1 /* 5 exponent bits (bias 15), 2 mantissa bits, largest 57344 */

/*
 * Forward attention ("FlashAttention: not computing less, moving less", section 01
 * formula O = softmax(QK^T / sqrt(d)) V with a general scale; section 02 online-softmax
 * recurrence; section 03 log-sum-exp statistics; causal masking as in "FlashAttention4
 * 精读" section 3.3; grouped-query heads as in section 3.3, GQA paragraph; packed
 * variable-length sequences as in "FlashAttention: not computing less, moving less",
 * section 05, training paragraph).
 *
 * q   device, bf16 [T, Hq, d]    queries, T = B*Nq (dense) or Nq (packed)
 * k   device, bf16 [Tk, Hkv, d]  keys,    Tk = B*Nk (dense) or Nk (packed)
 * v   device, bf16 [Tk, Hkv, d]  values
 * o   device, bf16 [T, Hq, d]    output (written)
 * lse device, fp32 [T, Hq]       natural-log log-sum-exp of the scaled scores of each row,
 *                                so softmax_ij = exp(scale * q_i.k_j - lse_i) (written)
 * B         number of sequences (>= 0)
 * Hq, Hkv   query and key/value heads; Hq % Hkv == 0, query head h reads kv head h/(Hq/Hkv)
 * Nq, Nk    dense: query and key length of every sequence. Packed: the rows of q/o and of
 *           k/v (the sequence lengths come from cu_seqlens and queries and keys share them;
 *           a sequence reaching past Nq or Nk is treated as empty and recorded as
 *           ATTN_ERR_DEVICE_BAD_INDEX)
 * d         head dimension, 64, 128 or 256 (256: one 128-row query tile per CTA at a time,
 *           key/value tiles streamed in 128-column halves; the CTAs take query tiles from a
 *           counter as they become free, and the call takes that 8-byte counter from the
 *           library's stream-ordered pool on `stream`, zeroes it there and returns it there,
 *           so calls on different streams never share one)
 * scale     multiplier of q.k (typically 1/sqrt(d)); must be finite
 * causal    0: every key is visible. 1: bottom-right aligned mask, key j visible to query
 *           row i of its sequence iff j <= i + (Nk - Nq). Rows that see no key get o = 0
 *           and lse = -inf.
 * cu_seqlens NULL for dense batches, else device int32 [B+1] prefix offsets of packed
 *           sequences (non-decreasing). One kernel launch takes up to 1024 sequences (64 at
 *           d = 256); a larger B runs as consecutive launches of that many sequences each.
 * Alignment: q, k, v, o 16 bytes; lse 4 bytes.
 * Returns ATTN_OK or an error code; see the conventions above.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int Nq, int Nk, int d, float scale, int causal, const int* cu_seqlens, void* stream);

/*
 * attn_fwd with values (and outputs) narrower than queries and keys: head dims (d, dv) =
 * (192, 128), the DeepSeek-V3 configuration ("FlashAttention-4: Blackwell algorithm-pipeline
 * co-design", performance section). Scores use all d = 192 columns of q and k; the output
 * is the probability-weighted sum of the dv = 128 wide values.
 *
 * q           device, bf16 [T, Hq, d]      k  device, bf16 [Tk, Hkv, d]
 * v           device, bf16 [Tk, Hkv, dv]   o  device, bf16 [T, Hq, dv] (written)
 * lse         device, fp32 [T, Hq] (written)
 * d, dv       (192, 128); (64, 64), (128, 128) and (256, 256) are also accepted and behave as
 *             attn_fwd.
 *             Anything else is ATTN_ERR_BAD_SHAPE.
 * Everything else is as for attn_fwd. With (192, 128) the kernel uses 96-key tiles (the
 * 192-wide query and key tiles leave no room in shared memory for 128-key tiles), and one
 * launch takes up to 256 packed sequences (a larger batch runs as several launches).
 */
attn_status_t attn_fwd_hd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nq, int Nk, int d, int dv, float scale, int causal, const int* cu_seqlens, void* stream);

/*
 * attn_fwd on Q/K/V given in 8-bit floating point ("Faster, more flexible FA4 for LLM
 * inference", PR 2109: e4m3 or e5m2 inputs).
 *
 * q, k, v     device, 8-bit codes in the layouts of attn_fwd, OCP FP8 format fp8_format
 *             (ATTN_FP8_E4M3 or ATTN_FP8_E5M2, defined below); each tensor stands for its
 *             descale times the decoded values (one factor per tensor, finite)
 * o, lse      bf16 [T, Hq, d] and fp32 [T, Hq] as for attn_fwd
 * d           128 only (other values: ATTN_ERR_BAD_SHAPE)
 * Everything else (masks, packed sequences, GQA, alignment, errors) is as for attn_fwd.
 * An unknown format, a non-finite descale or a score scale that overflows a float is
 * ATTN_ERR_BAD_ARG.
 * Arithmetic: S = Q K^T on the tensor cores in 8-bit floating point with fp32 accumulation
 * (products of 8-bit values are exact); the softmax as for attn_fwd; P rounded to f16; V
 * widened exactly to f16 in shared memory; O += P V in f16 with fp32 accumulation.
 */
attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int Nq, int Nk, int d, float scale, int causal, const int* cu_seqlens, void* stream,
                           int fp8_format, float q_descale, float k_descale, float v_descale);

/*
 * Paged-KV decode ("Faster, more flexible FA4 for LLM inference": PR 1999/2104 arbitrary
 * page sizes gathered with cp.async, PR 1940 split-KV with a separate combine kernel,
 * PR 2186 query heads of one kv head packed into one tile; "FlashAttention: not computing
 * less, moving less", section 05, inference paragraph: decode over a paged KV cache).
 * One query token per sequence; every cached key of the sequence is visible.
 *
 * q          device, bf16 [B, Hq, d]
 * k_cache    device, bf16 [num_pages, page_size, Hkv, d]  physical pages of keys
 * v_cache    device, bf16 [num_pages, page_size, Hkv, d]  physical pages of values
 * page_table device, int32 [B, max_pages_per_seq]; token t of sequence b lives in physical
 *            page page_table[b][t / page_size], slot t % page_size. Entries may repeat
 *            (shared prefixes); entries past a sequence's last page are never read.
 * seqlens    device, int32 [B], cached tokens per sequence, 0 <= seqlens[b] <=
 *            max_pages_per_seq * page_size. A sequence of length 0 gets o = 0, lse = -inf.
 * page_size  tokens per page, >= 1 (any value)
 * o          device, bf16 [B, Hq, d] (written);  lse device, fp32 [B, Hq] (written)
 * B, Hq, Hkv, d  as for attn_fwd (d = 64 or 128); the query heads of a kv head are the rows
 *            of one tile, so more than 16 per kv head run as groups of 16 (one CTA each, in the
 *            same launch, neighbours in the grid so that they share the cache rows in the L2)
 * max_pages_per_seq  columns of page_table (>= 1)
 * num_pages  physical pages in each cache (>= 1, num_pages * page_size <= 2^31 - 1 cache rows);
 *            a page index outside [0, num_pages) is not read: its rows count as zeros and
 *            ATTN_ERR_DEVICE_BAD_INDEX is recorded
 * scale      as for attn_fwd
 * num_splits 0: choose the number of key splits from the SM count and the sizes;
 *            n > 0: split every sequence's keys into at most n chunks.
 * Workspace: partial outputs of the splits live in memory taken from a library-owned
 * stream-ordered pool on `stream` and returned to it on `stream` after the combine.
 * Launches: a split kernel and, when a sequence has more than one split, a combine kernel
 * launched as its programmatic dependent (it may start while the split kernel finishes and
 * waits on the device for its results). Work after the call on `stream` sees both done, as
 * for any pair of launches; a kernel the caller launches with programmatic stream
 * serialization must wait (griddepcontrol.wait) before it reads o or lse.
 * Alignment: q, o, k_cache, v_cache 16 bytes; lse, page_table, seqlens 4 bytes.
 */
attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* page_table,
                                const int* seqlens, int page_size, void* o, float* lse, void* stream, int B, int Hq,
                                int Hkv, int d, int max_pages_per_seq, int num_pages, float scale, int num_splits);

/*
 * attn_decode_paged over key/value caches in 8-bit floating point ("Faster, more flexible
 * FA4 for LLM inference", PR 2109: e4m3 or e5m2 inputs; half the cache bytes of bf16).
 *
 * k_cache, v_cache  device, 8-bit codes [num_pages, page_size, Hkv, d] in the OCP FP8
 *                   format kv_format: ATTN_FP8_E4M3 (4 exponent bits, bias 7, largest 448,
 *                   no infinities) or ATTN_FP8_E5M2 (5 exponent bits, bias 15).
 * k_descale, v_descale  one factor per tensor: key code c stands for k_descale * fp8(c),
 *                   value code c for v_descale * fp8(c). Finite; otherwise
 *                   ATTN_ERR_BAD_ARG. An unknown kv_format is ATTN_ERR_BAD_ARG.
 * Everything else (q in bf16, page table, seqlens, o, lse, sizes, num_splits, workspace,
 * alignment, errors) is as for attn_decode_paged.
 * Arithmetic: the products run on the tensor cores in f16 with fp32 accumulation. Every
 * FP8 value is exact in f16; q is converted from bf16 to f16, which is exact for
 * |q| in [2^-14, 65504] (smaller magnitudes lose low bits, larger ones overflow), and the
 * probabilities are rounded to f16 before the P V product.
 */
attn_status_t attn_decode_paged_fp8(const void* q, const void* k_cache, const void* v_cache, const int* page_table,
                                    const int* seqlens, int page_size, void* o, float* lse, void* stream, int B,
                                    int Hq, int Hkv, int d, int max_pages_per_seq, int num_pages, float scale,
                                    int num_splits, int kv_format, float k_descale, float v_descale);

/*
 * attn_decode_paged without any memory allocation. The pages have no counterpart to this
 * call; it exists for callers that cannot allocate device memory when they run decode:
 * a serving engine that has already given nearly all of the GPU's memory to its own
 * KV-cache pool, or code that must not enter the driver's allocator, which can block the
 * device or fail late under memory pressure.
 *
 * Same arguments, layouts, results and error behaviour as attn_decode_paged. The split
 * partials go to one fixed 32 MiB device array built into the library (every GPU that
 * loads the library holds it until the process exits) instead of memory taken per call.
 * - Sizes whose partials need more than 32 MiB, that is B * Hq * splits * (d + 1) * 4
 *   bytes with splits from attn_decode_plan, are rejected with
 *   ATTN_ERR_SCRATCH_TOO_SMALL before anything is launched (lower num_splits to fit).
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before any
 *   stream capture begins.
 * - All calls on a device share the one array, and it keeps the last call's contents.
 *   Nothing in it needs clearing, because the combine step reads only partials the same
 *   call wrote. Calls whose work overlaps on the GPU (on different streams, say) race on
 *   the array and may produce wrong results: order them.
 * - No cudaMalloc, cudaFree or other allocating routine is called.
 */
attn_status_t attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache, const int* page_table,
                                        const int* seqlens, int page_size, void* o, float* lse, void* stream, int B,
                                        int Hq, int Hkv, int d, int max_pages_per_seq, int num_pages, float scale,
                                        int num_splits);

/*
 * Host-side split choice of attn_decode_paged (the num_splits = 0 heuristic of "Faster,
 * more flexible FA4 for LLM inference", PR 1940 section; the pages give no formula).
 * Writes the tokens per split (*chunk, a multiple of 64) and the splits the workspace
 * holds per sequence (*max_splits) for the given sizes. The heuristic aims at about 32
 * (sequence, kv head, split) items per SM, with at least 256 and at least 128 * Hq / Hkv
 * tokens per split (so that the fp32 partials of the query heads stay small next to the
 * cache bytes of a split) and at most 8192. num_sms <= 0 uses the current device's SM
 * count. Pure host arithmetic; needs no GPU when num_sms > 0.
 */
attn_status_t attn_decode_plan(int B, int Hq, int Hkv, int max_pages_per_seq, int page_size, int num_splits,
                               int num_sms, int* chunk, int* max_splits);

/*
 * Bytes of split-KV workspace attn_decode_paged takes for these sizes: B * Hq * max_splits
 * partial outputs of d floats plus as many partial log-sum-exps (fp32), with max_splits
 * from attn_decode_plan (a call with max_splits = 1 writes its results directly and needs
 * none). Returns 0 for max_splits <= 1 or non-positive sizes. Pure host arithmetic.
 * attn_decode_paged takes this memory from a library-owned stream-ordered pool;
 * attn_decode_paged_noalloc compares it with its fixed 32 MiB array.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int d, int max_splits);

/* Static description of a status code. Never NULL. */
const char* attn_status_string(attn_status_t status);

/*
 * Synchronises `stream`, then reads and clears the current device's status word.
 * Returns ATTN_OK, the first device-side error recorded since the last call
 * (ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_DEVICE_BAD_INDEX), or ATTN_ERR_CUDA.
 */
attn_status_t attn_get_device_status(void* stream);

/*
 * Process-wide tuning options (not needed for correct use):
 *   "exp_poly"           0: every exponential on MUFU.EX2 (default); 1: one column in
 *                        eight on the Cody-Waite cubic polynomial ("FlashAttention4 精读"
 *                        section 3.1.3, partial emulation)
 *   "rescale_threshold"  rescale O only when the row maximum grows by more than this many
 *                        powers of two (default 8, i.e. a factor 256, "FlashAttention4 精读"
 *                        section 3.1.4); 0 rescales on every increase
 *   "decode_chunk"       tokens per decode split when num_splits = 0 (0 = heuristic)
 *   "sec_heads"          forward scheduling section (0 = heuristic): dense batches, the
 *                        (batch, query head) pairs ordered together (rounded up to whole
 *                        GQA groups; by default all of them unless the work spans 16 or more
 *                        waves of the grid); packed sequences, query heads per section
 *   "count"              1: count softmax rescale decisions and exponentials (attn_read_counters)
 *   "watchdog_ms"        device wait limit before a kernel gives up (default 4000)
 *   "dynamic_order"      head width 256: 1 (default) CTAs take query tiles from a counter in
 *                        the order of head sections (16 heads unless "sec_heads" says
 *                        otherwise), heaviest blocks first within each, so that the running
 *                        CTAs share key/value tiles in the L2 ("FlashAttention4 精读" section
 *                        3.3, L2-sized sections with LPT); 0 the static order of the other widths
 *   "correction"         1: the rescale of O is done by a separate correction warp per TMEM lane
 *                        quarter ("FlashAttention4 精读" section 3.1), bf16 at d = 128 only;
 *                        0 (default): by the softmax warp itself, in the rare steps that need it
 *   "unroll_kv"          1: the last O += P V of a work tile and the first S = Q K^T of the next
 *                        are issued as one burst ("Low-precision FA4" section 2.1.2), bf16 and
 *                        e4m3 at d = 128; 0 (default): separate bursts
 *   "packed_order"       packed sequences: 1 (default) orders work heaviest first across all
 *                        sequences ("FlashAttention4 精读" section 3.3, LPT for varlen);
 *                        0 keeps the sequences in the caller's order (each sequence's
 *                        blocks still heaviest first), for measuring what the sort gains
 *   "decode_order"       paged decode: 1 (default) the CTAs of every sequence's last split
 *                        (shorter than the others in general) start after all other splits,
 *                        longest first for up to 256 sequences, so they fill the SMs that the
 *                        last full-length splits leave idle (LPT, as for the forward); 0 the
 *                        splits sequence by sequence
 *   "decode_maps"        8-bit paged decode at d = 128 with a page size that is a multiple of
 *                        16 and at most 8 or more than 16 query heads per kv head: 1 (default)
 *                        each group of 16 tokens (within one page) is loaded per kv head with
 *                        one tensor-map copy for K and one for V; 0 every lane copies 16-byte
 *                        pieces of its token's rows (the path of the other shapes). Both give
 *                        the same bytes
 * Returns ATTN_ERR_BAD_ARG for an unknown name or an invalid value.
 */
attn_status_t attn_set_option(const char* name, double value);
attn_status_t attn_get_option(const char* name, double* value);

/*
 * Reads and clears the current device's counters (enabled by option "count"):
 * out[0] softmax warp-tile steps (one warp's 32 rows against one key tile), out[1] of which
 * raised the running maximum, out[2] exponentials on the polynomial, out[3] exponentials on
 * MUFU, out[4] steps after the first key tile of a Q tile (O already holds a partial sum),
 * out[5] of which rescaled O ("FlashAttention-4: Blackwell algorithm-pipeline co-design",
 * conditional softmax rescaling: the fraction out[5] / out[4] is the rescale rate).
 * n <= 6 values are written. Synchronises the device.
 */
attn_status_t attn_read_counters(unsigned long long* out, int n);

/*
 * Diagnostics. attn_debug_exp2 evaluates the device exponentials on n fp32 inputs:
 * mode 0 the software 2^x of the hybrid exponential ("FlashAttention-4: Blackwell
 * algorithm-pipeline co-design", section "hybrid exponential"), mode 1 MUFU ex2.approx.ftz.
 * x, y device fp32 [n]. attn_debug_watchdog launches a kernel that waits on a barrier no
 * thread ever arrives on, with the bounded wait of the attention kernels and the given
 * limit, so that the next attn_get_device_status() reports ATTN_ERR_DEVICE_TIMEOUT.
 */
attn_status_t attn_debug_exp2(const float* x, float* y, long long n, int mode, void* stream);
attn_status_t attn_debug_watchdog(unsigned long long limit_ns, void* stream);

/* Library version string. */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_SOFTMAX_ATTENTION_GB300_ATTN_H */
