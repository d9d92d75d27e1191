// Internal interface between the C-ABI layer (attn_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace attn {

// Raise a kernel's dynamic shared-memory limit once per device (the current one). The flags
// are atomics because launches can come from several host threads at once; setting the
// attribute twice is harmless, so a race only repeats that call.
constexpr int kMaxAttrDevices = 64;
template <typename Kernel>
// min_regs: registers per thread the kernel must have been built with (a kernel that moves
// registers between warp groups with setmaxnreg hands out exactly the launch's total); a build
// with fewer is refused (cudaErrorInvalidConfiguration) instead of launched.
inline cudaError_t ensure_smem_attr(Kernel kernel, int bytes, std::atomic<bool> (&done)[kMaxAttrDevices],
                                    int min_regs = 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxAttrDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    if (min_regs > 0) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        if (fa.numRegs < min_regs) return cudaErrorInvalidConfiguration;
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < kMaxAttrDevices) done[dev].store(true, std::memory_order_release);
    return e;
}

// Device status word layout (int[4]): [0] first error code (0 = ok), [1] detail, [2..3] reserved.
enum DeviceErr : int {
    kDevOk = 0,
    kDevTimeout = -6,   // matches ATTN_ERR_DEVICE_TIMEOUT
    kDevBadIndex = -7,  // matches ATTN_ERR_DEVICE_BAD_INDEX
};

// Counters (unsigned long long[6]) when enabled: [0] softmax warp-tile decisions, [1] of which raised the
// running maximum, [2] polynomial exponentials evaluated, [3] MUFU exponentials evaluated, [4] decisions
// after the first key tile of a Q tile (O already holds a partial sum), [5] of which rescaled O.
constexpr int kNumCounters = 6;

struct FwdParams {
    __nv_bfloat16* o;
    float* lse;
    const int* cu_seqlens;  // device int32 [B+1] or nullptr for dense batches
    int B, Hq, Hkv, G, Nq, Nk;
    int causal;
    float scale;        // softmax scale applied to q.k
    float scale_log2;   // scale * log2(e)
    float rescale_thr;  // rescale O only when the row max grows by more than this (base-2 exponent units)
    float out_scale;    // multiplies O at the end (8-bit inputs: the value descale; else 1)
    int sec_q;          // scheduling section, a multiple of G: dense, (batch, head) pairs; packed, query heads (divides Hq)
    int total_tiles;    // dense: number of work tiles; varlen: ignored (computed on device)
    int packed_plain;   // packed sequences: 1 = sequences in the caller's order (no heaviest-first sort)
    int corr_warp;      // 1: O is rescaled by the correction role (epilogue warps; a separate instantiation,
                        // bf16 at d = 128); 0: by the softmax warps
    int unroll_kv;      // 1: the last P V product of a work tile and the first S = Q K^T of the next share a
                        // burst (a separate instantiation, for bf16 and e4m3 inputs at d = 128)
    unsigned int* sched;  // head width 256: zeroed unit counter of this launch (dynamic order), or nullptr
    int* status;
    unsigned long long* counters;  // nullptr unless counting is enabled
    unsigned long long watchdog_ns;
};

struct FwdTmaps {
    CUtensorMap q, k, v;
};

// Launch the forward kernel for head dim d in {64, 128}; exp_poly selects the MUFU/polynomial split.
cudaError_t launch_attn_fwd(const FwdTmaps& tm, const FwdParams& p, int d, int exp_poly, int grid,
                            cudaStream_t stream);
// 8-bit Q/K/V codes (fmt 0 = e4m3, 1 = e5m2), d = 128; p.scale already includes the q and k
// descales and p.out_scale is the v descale.
cudaError_t launch_attn_fwd_fp8(const FwdTmaps& tm, const FwdParams& p, int d, int fmt, int grid,
                                cudaStream_t stream);
// Head dims (d, dv) = (192, 128): q, k 192 wide, v, o 128 wide; key tiles of 96 rows.
cudaError_t launch_attn_fwd_hd(const FwdTmaps& tm, const FwdParams& p, int d, int dv, int grid, cudaStream_t stream);
// Head width 256 (q, k, v, o): one 128-row Q tile at a time, two S buffers in TMEM.
cudaError_t launch_attn_fwd_wide(const FwdTmaps& tm, const FwdParams& p, int grid, cudaStream_t stream);
// Largest number of packed sequences of one call for query/key width d.
int fwd_max_varlen_batch(int d);

struct DecodeParams {
    const __nv_bfloat16* q;        // [B, Hq, d]
    const __nv_bfloat16* k_cache;  // [num_pages, page_size, Hkv, d]
    const __nv_bfloat16* v_cache;
    const int* page_table;         // [B, max_pages]
    const int* seqlens;            // [B]
    __nv_bfloat16* o;              // [B, Hq, d]
    float* lse;                    // [B, Hq]
    float* ws_o;                   // [B, Hq, max_splits, d] partial outputs
    float* ws_lse;                 // [B, Hq, max_splits] partial LSE
    int B, Hq, Hkv, page_size, max_pages, num_pages;
    // Query heads: g_stride = Hq / Hkv per kv head (query head h reads kv head h / g_stride). The
    // split kernels take them in n_groups groups of at most 16 (one CTA each); the combine
    // merges heads g_base .. g_base + G - 1 of every kv head (all of them: g_base 0, G = g_stride).
    int G, g_base, g_stride, n_groups;
    int chunk;       // tokens per split (multiple of 64)
    int max_splits;  // splits per sequence the workspace holds
    // Work order of the split kernels. order (set by the caller): 1 = the last split of every
    // sequence after all the others, 0 = one grid row per sequence with all its splits. The
    // launcher derives full_rows and lpt: grid rows y < full_rows list the splits of sequence y
    // before its last one, the rows after them the last split of every sequence (in decreasing
    // length when lpt != 0); full_rows < 0: row y holds all splits of sequence y.
    int order, full_rows, lpt;
    // tok / page_size for 0 <= tok < 2^31 is __umulhi(tok, ps_magic) >> ps_shift (set by the
    // launcher; page_size 1: ps_magic = 0 and the quotient is tok).
    unsigned int ps_magic;
    int ps_shift;
    float scale, scale_log2, rescale_thr;
    float v_descale;  // FP8 caches: value descale applied to the output (bf16 caches: unused)
    int* status;
};

cudaError_t launch_attn_decode(const DecodeParams& p, int d, cudaStream_t stream);
// FP8 caches (k_cache / v_cache hold 8-bit codes); fmt 0 = e4m3, 1 = e5m2. p.scale and
// p.scale_log2 already include the key descale.
cudaError_t launch_attn_decode_fp8(const DecodeParams& p, int d, int fmt, cudaStream_t stream);

// Status word and SM count of the current device (checks that it is an sm_103 GPU);
// returns an attn_status_t code.
int current_device_info(int** status, int* num_sms);

// Diagnostics
cudaError_t launch_exp2_probe(const float* x, float* y, long long n, int mode, cudaStream_t stream);
cudaError_t launch_watchdog_probe(int* status, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace attn
