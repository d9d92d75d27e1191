// C ABI of the attention library: argument checks, TMA descriptors, launch planning,
// the device status word and process-wide options. Every compute step runs in the
// kernels of attn_fwd.cu and attn_decode.cu.
#include "attn.h"
#include "decode_maps.cuh"
#include "kernels.cuh"

#include <cudaTypedefs.h>

#include <float.h>
#include <math.h>
#include <mutex>
#include <string.h>

namespace {

using attn::DecodeParams;
using attn::FwdParams;
using attn::FwdTmaps;

constexpr int kMaxDevices = 64;

__device__ int g_status[4];
__device__ unsigned long long g_counters[attn::kNumCounters];

struct Options {
    int exp_poly = 0;
    double rescale_threshold = 8.0;
    int decode_chunk = 0;
    int sec_heads = 0;
    int count = 0;
    double watchdog_ms = 4000.0;
    int packed_order = 1;
    int correction = 0;
    int unroll_kv = 0;
    int dynamic_order = 1;
    int decode_order = 1;
    int decode_maps = 1;
};

std::mutex g_mu;
Options g_opt;

struct DeviceState {
    bool init = false;
    bool arch_ok = false;
    int num_sms = 0;
    int* status = nullptr;
    unsigned long long* counters = nullptr;
    cudaMemPool_t pool = nullptr;
};
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

attn_status_t device_state(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return ATTN_ERR_CUDA;
        st.arch_ok = (major == 10 && minor == 3);
        st.num_sms = sms;
        if (st.arch_ok) {
            if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status), g_status) != cudaSuccess) return ATTN_ERR_CUDA;
            if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.counters), g_counters) != cudaSuccess)
                return ATTN_ERR_CUDA;
        }
        st.init = true;
    }
    if (!st.arch_ok) return ATTN_ERR_UNSUPPORTED_ARCH;
    *out = &st;
    return ATTN_OK;
}

attn_status_t encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return ATTN_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return ATTN_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return ATTN_OK;
}

// 3-D map over a [rows, heads, d] tensor of bf16 (elem 2) or 8-bit codes (elem 1); box =
// 128 bytes of d x 1 head x 128 rows, 128-byte swizzle (the K-major / MN-major canonical
// layout the MMAs read), zero fill outside [0, rows).
attn_status_t make_map(CUtensorMap* m, const void* base, long long rows, int heads, int d, int elem = 2,
                       int box_rows = 128) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)d * elem, (cuuint64_t)heads * d * elem};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem), 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                          const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// 2-D map over a paged cache of 8-bit codes viewed as [rows, row_bytes] (row_bytes = Hkv * d):
// box d bytes x 16 rows, 128-byte swizzle (the layout the decode kernel's rings use).
attn_status_t make_cache_map(CUtensorMap* m, const void* base, long long rows, int row_bytes, int d) {
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)d, (cuuint32_t)attn::kDecodeMapRows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

Options options() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_opt;
}

int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

// The library's stream-ordered memory pool on the current device (created on first use; it
// keeps what it has reserved, so later calls take their memory without the driver).
attn_status_t device_pool(DeviceState* ds, cudaMemPool_t* out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!ds->pool) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
        cudaMemPoolProps props;
        memset(&props, 0, sizeof props);
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if (cudaMemPoolCreate(&ds->pool, &props) != cudaSuccess) return ATTN_ERR_CUDA;
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(ds->pool, cudaMemPoolAttrReleaseThreshold, &keep);
    }
    *out = ds->pool;
    return ATTN_OK;
}

}  // namespace

extern "C" {

const char* attn_version(void) { return "exact_softmax_attention_gb300 0.1 (sm_103a)"; }

const char* attn_status_string(attn_status_t s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULL_PTR: return "a required pointer is NULL";
        case ATTN_ERR_BAD_SHAPE: return "unsupported or inconsistent sizes";
        case ATTN_ERR_ALIGN: return "a pointer is not aligned as required";
        case ATTN_ERR_UNSUPPORTED_ARCH: return "the current device is not an sm_103 GPU";
        case ATTN_ERR_CUDA: return "a CUDA call failed";
        case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on its pipeline (device watchdog)";
        case ATTN_ERR_DEVICE_BAD_INDEX: return "a page index or sequence length was out of range";
        case ATTN_ERR_BAD_ARG: return "unknown option or invalid value";
        case ATTN_ERR_SCRATCH_TOO_SMALL: return "the sizes need more split workspace than the fixed scratch array holds";
        default: return "unknown status";
    }
}

attn_status_t attn_set_option(const char* name, double value) {
    if (!name) return ATTN_ERR_NULL_PTR;
    if (!isfinite(value)) return ATTN_ERR_BAD_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!strcmp(name, "exp_poly")) {
        if (value != 0 && value != 1) return ATTN_ERR_BAD_ARG;
        g_opt.exp_poly = (int)value;
    } else if (!strcmp(name, "rescale_threshold")) {
        if (value < 0 || value > 60) return ATTN_ERR_BAD_ARG;
        g_opt.rescale_threshold = value;
    } else if (!strcmp(name, "decode_chunk")) {
        if (value < 0 || value > (1 << 24)) return ATTN_ERR_BAD_ARG;
        g_opt.decode_chunk = (int)value;
    } else if (!strcmp(name, "sec_heads")) {
        if (value < 0 || value > 65536) return ATTN_ERR_BAD_ARG;
        g_opt.sec_heads = (int)value;
    } else if (!strcmp(name, "count")) {
        if (value != 0 && value != 1) return ATTN_ERR_BAD_ARG;
        g_opt.count = (int)value;
    } else if (!strcmp(name, "watchdog_ms")) {
        if (value < 1 || value > 600000) return ATTN_ERR_BAD_ARG;
        g_opt.watchdog_ms = value;
    } else if (!strcmp(name, "packed_order")) {
        if (value != 0 && value != 1) return ATTN_ERR_BAD_ARG;
        g_opt.packed_order = (int)value;
    } else if (!strcmp(name, "correction")) {
        if (value != 0 && value != 1) return ATTN_ERR_BAD_ARG;
        g_opt.correction = (int)value;
    } else if (!strcmp(name, "unroll_kv")) {
        if (value != 0 && value != 1) return ATTN_ERR_BAD_ARG;
        g_opt.unroll_kv = (int)value;
    } else if (!strcmp(name, "dynamic_order")) {
        if (value != 0 && value != 1) return ATTN_ERR_BAD_ARG;
        g_opt.dynamic_order = (int)value;
    } else if (!strcmp(name, "decode_order")) {
        if (value != 0 && value != 1) return ATTN_ERR_BAD_ARG;
        g_opt.decode_order = (int)value;
    } else if (!strcmp(name, "decode_maps")) {
        if (value != 0 && value != 1) return ATTN_ERR_BAD_ARG;
        g_opt.decode_maps = (int)value;
    } else {
        return ATTN_ERR_BAD_ARG;
    }
    return ATTN_OK;
}

attn_status_t attn_get_option(const char* name, double* value) {
    if (!name || !value) return ATTN_ERR_NULL_PTR;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!strcmp(name, "exp_poly")) *value = g_opt.exp_poly;
    else if (!strcmp(name, "rescale_threshold")) *value = g_opt.rescale_threshold;
    else if (!strcmp(name, "decode_chunk")) *value = g_opt.decode_chunk;
    else if (!strcmp(name, "sec_heads")) *value = g_opt.sec_heads;
    else if (!strcmp(name, "count")) *value = g_opt.count;
    else if (!strcmp(name, "watchdog_ms")) *value = g_opt.watchdog_ms;
    else if (!strcmp(name, "packed_order")) *value = g_opt.packed_order;
    else if (!strcmp(name, "correction")) *value = g_opt.correction;
    else if (!strcmp(name, "unroll_kv")) *value = g_opt.unroll_kv;
    else if (!strcmp(name, "dynamic_order")) *value = g_opt.dynamic_order;
    else if (!strcmp(name, "decode_order")) *value = g_opt.decode_order;
    else if (!strcmp(name, "decode_maps")) *value = g_opt.decode_maps;
    else return ATTN_ERR_BAD_ARG;
    return ATTN_OK;
}

// Shared body of the forward entry points. fp8 < 0: bf16 Q/K/V; 0 / 1: e4m3 / e5m2 codes
// with per-tensor descales (d = 128 only). dv: value / output width (= d, or 128 with d = 192).
static attn_status_t fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                         int Nq, int Nk, int d, float scale, int causal, const int* cu_seqlens, void* stream, int fp8,
                         float q_descale, float k_descale, float v_descale, int dv = -1) {
    if (dv < 0) dv = d;
    if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL_PTR;
    const bool shape_ok = (d == dv && (d == 64 || d == 128 || d == 256)) || (d == 192 && dv == 128);
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq < 0 || Nk < 0 || !shape_ok) return ATTN_ERR_BAD_SHAPE;
    if (fp8 >= 0 && d != 128) return ATTN_ERR_BAD_SHAPE;
    if (causal != 0 && causal != 1) return ATTN_ERR_BAD_SHAPE;
    if (!isfinite(scale)) return ATTN_ERR_BAD_SHAPE;
    if (Hq > 65535 || Hkv > 65535) return ATTN_ERR_BAD_SHAPE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        (cu_seqlens && !aligned(cu_seqlens, 4)))
        return ATTN_ERR_ALIGN;
    // rows of q/o and of k/v: dense B*N; packed: Nq and Nk are the total packed rows
    const long long Tq = cu_seqlens ? (long long)Nq : (long long)B * Nq;
    const long long Tk = cu_seqlens ? (long long)Nk : (long long)B * Nk;
    if (Tq > INT32_MAX - 1024 || Tk > INT32_MAX - 1024) return ATTN_ERR_BAD_SHAPE;
    if (B == 0 || Tq == 0) return ATTN_OK;
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    if ((st = encode_fn()) != ATTN_OK) return st;
    FwdTmaps tm;
    const int elem = fp8 >= 0 ? 1 : 2;
    const int kv_rows = d == 192 ? 96 : 128;  // keys per K/V tile of the kernel instantiation
    if (make_map(&tm.q, q, Tq, Hq, d, elem) != ATTN_OK || make_map(&tm.k, k, Tk, Hkv, d, elem, kv_rows) != ATTN_OK ||
        make_map(&tm.v, v, Tk, Hkv, dv, elem, kv_rows) != ATTN_OK)
        return ATTN_ERR_CUDA;
    const Options opt = options();
    FwdParams p;
    memset(&p, 0, sizeof p);
    p.o = reinterpret_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.cu_seqlens = cu_seqlens;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.Nq = Nq;
    p.Nk = Nk;
    p.causal = causal;
    const double score_scale = fp8 < 0 ? (double)scale : (double)scale * (double)q_descale * (double)k_descale;
    p.scale = (float)score_scale;
    p.scale_log2 = (float)(score_scale * 1.4426950408889634);
    p.out_scale = fp8 < 0 ? 1.0f : v_descale;
    p.rescale_thr = (float)opt.rescale_threshold;
    p.status = ds->status;
    p.counters = opt.count ? ds->counters : nullptr;
    p.watchdog_ns = (unsigned long long)(opt.watchdog_ms * 1e6);
    p.packed_plain = opt.packed_order == 0;
    p.corr_warp = opt.correction;
    p.unroll_kv = opt.unroll_kv;
    int grid = ds->num_sms;
    if (!cu_seqlens) {
        const long long nblk = cdiv(Nq, 256);
        const long long pairs = (long long)B * Hq;
        const long long tiles = pairs * nblk;
        if (tiles > INT32_MAX / 2) return ATTN_ERR_BAD_SHAPE;
        p.total_tiles = (int)tiles;
        const long long units = d == 256 ? 2 * tiles : tiles;  // the d = 256 kernel takes one Q tile at a time
        if (units < grid) grid = (int)units;
        // Section of (batch, head) pairs: all of them unless the tiles make 16 or more waves
        // of the grid; then sections of at least 8 waves each, which keeps the heaviest-first
        // order balanced within a section while fewer key/value heads share the L2.
        // Head width 256 with the dynamic order: the CTAs take units in order as they become
        // free, so balance needs no long sections. Measured on the long causal geometry
        // (B1 H32 N8192): 4-head sections bring DRAM reads to the algorithmic bytes but no
        // time (the kernel is bounded by shared-memory traffic, not DRAM); 16 heads were the
        // fastest and still halve the DRAM traffic of the static order.
        const bool dyn = d == 256 && opt.dynamic_order;
        long long sec = pairs;
        if (opt.sec_heads > 0) sec = opt.sec_heads;
        else if (dyn) sec = 16;
        else if (nblk > 0 && tiles >= 16LL * grid) sec = cdiv(8LL * grid, nblk);
        sec = ((sec + p.G - 1) / p.G) * p.G;
        if (sec > pairs) sec = pairs;
        p.sec_q = (int)sec;
    } else {
        // packed: largest multiple of G dividing Hq that is <= the target heads per section
        int target = opt.sec_heads > 0 ? opt.sec_heads : 8;
        if (target < p.G) target = p.G;
        int sec = p.G;
        for (int c = p.G; c <= Hq && c <= target; c += p.G)
            if (Hq % c == 0) sec = c;
        p.sec_q = sec;
        p.total_tiles = 0;
    }
    if (grid <= 0) return ATTN_OK;
    const cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    // Head width 256, dynamic order: a unit counter per call, from the library's stream-ordered
    // pool, zeroed on the call's stream before every launch (so concurrent calls on other
    // streams never share one) and returned after the last.
    unsigned int* sched = nullptr;
    if (d == 256 && opt.dynamic_order) {
        cudaMemPool_t pool = nullptr;
        if ((st = device_pool(ds, &pool)) != ATTN_OK) return st;
        if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&sched), 2 * sizeof(unsigned int), pool, st_) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    auto launch = [&](const FwdParams& lp) {
        if (sched && cudaMemsetAsync(sched, 0, 2 * sizeof(unsigned int), st_) != cudaSuccess) return cudaErrorUnknown;
        FwdParams q = lp;
        q.sched = sched;
        return fp8 >= 0   ? attn::launch_attn_fwd_fp8(tm, q, d, fp8, grid, st_)
               : d != dv  ? attn::launch_attn_fwd_hd(tm, q, d, dv, grid, st_)
               : d == 256 ? attn::launch_attn_fwd_wide(tm, q, grid, st_)
                          : attn::launch_attn_fwd(tm, q, d, opt.exp_poly, grid, st_);
    };
    auto done = [&](attn_status_t r) {
        if (sched && cudaFreeAsync(sched, st_) != cudaSuccess && r == ATTN_OK) r = ATTN_ERR_CUDA;
        return r;
    };
    if (!cu_seqlens) return done(launch(p) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA);
    // Packed sequences: one launch builds its work order in shared memory for at most maxB
    // sequences, so a larger batch runs as consecutive launches of maxB sequences each (the
    // offsets in cu_seqlens are absolute rows of q/k, so a launch only needs its slice of them).
    const int maxB = attn::fwd_max_varlen_batch(d);
    for (int b0 = 0; b0 < B; b0 += maxB) {
        FwdParams lp = p;
        lp.cu_seqlens = cu_seqlens + b0;
        lp.B = B - b0 < maxB ? B - b0 : maxB;
        if (launch(lp) != cudaSuccess) return done(ATTN_ERR_CUDA);
    }
    return done(ATTN_OK);
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int Nq, int Nk, int d, float scale, int causal, const int* cu_seqlens, void* stream) {
    return fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens, stream, -1, 1.0f, 1.0f, 1.0f);
}

attn_status_t attn_fwd_hd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nq, int Nk, int d, int dv, float scale, int causal, const int* cu_seqlens, void* stream) {
    return fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens, stream, -1, 1.0f, 1.0f, 1.0f, dv);
}

attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                           int Nq, int Nk, int d, float scale, int causal, const int* cu_seqlens, void* stream,
                           int fp8_format, float q_descale, float k_descale, float v_descale) {
    if (fp8_format != ATTN_FP8_E4M3 && fp8_format != ATTN_FP8_E5M2) return ATTN_ERR_BAD_ARG;
    if (!isfinite(q_descale) || !isfinite(k_descale) || !isfinite(v_descale)) return ATTN_ERR_BAD_ARG;
    const double score_scale_log2 = (double)scale * (double)q_descale * (double)k_descale * 1.4426950408889634;
    if (!(fabs(score_scale_log2) <= (double)FLT_MAX)) return ATTN_ERR_BAD_ARG;  // the kernel uses it as a float
    return fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, cu_seqlens, stream, fp8_format, q_descale,
               k_descale, v_descale);
}

size_t attn_decode_workspace_bytes(int B, int Hq, int d, int max_splits) {
    if (B <= 0 || Hq <= 0 || d <= 0 || max_splits <= 1) return 0;
    return (size_t)B * (size_t)Hq * (size_t)max_splits * ((size_t)d + 1) * sizeof(float);
}

attn_status_t attn_decode_plan(int B, int Hq, int Hkv, int max_pages_per_seq, int page_size, int num_splits,
                               int num_sms, int* chunk, int* max_splits) {
    if (!chunk || !max_splits) return ATTN_ERR_NULL_PTR;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_pages_per_seq <= 0 || page_size <= 0 || num_splits < 0)
        return ATTN_ERR_BAD_SHAPE;
    const long long lmax = (long long)max_pages_per_seq * page_size;
    if (lmax > INT32_MAX / 2) return ATTN_ERR_BAD_SHAPE;
    if (num_sms <= 0) {
        DeviceState* ds = nullptr;
        const attn_status_t st = device_state(&ds);
        if (st != ATTN_OK) return st;
        num_sms = ds->num_sms;
    }
    const Options opt = options();
    long long c;
    if (num_splits > 0) {
        c = (lmax + num_splits - 1) / num_splits;
    } else if (opt.decode_chunk > 0) {
        c = opt.decode_chunk;
    } else {
        // About 18 (sequence, kv head, split) items per SM, assuming the average sequence fills
        // half of its page-table row; at least 256 tokens per split. Each split costs a few
        // microseconds beyond its bytes (pipeline fill and drain, the warp merge), and the split
        // kernels start every sequence's last split after all the others, so fewer, longer
        // splits win until the last wave gets coarse. Measured on 64 sequences of U[1K, 32K]
        // tokens, 8 kv heads: 1728 / 2048 / 2560 / 3072 / 3456 tokens per split (32 to 16 items
        // per SM) gave 6093 / 6186 / 6274 / 6287 / 6221 GB/s with e4m3 caches and 6883 / 6897 /
        // 6952 / 6990 / 6963 GB/s with bf16 caches.
        const long long work = (long long)(B > 0 ? B : 1) * Hkv * ((lmax + 1) / 2);
        const long long items = 18LL * num_sms;
        c = (work + items - 1) / items;
        if (c < 256) c = 256;
        // Each split writes d + 1 floats per query head; with few kv heads (MQA) small splits
        // would write partials of a size close to their cache bytes (measured on 32 query heads
        // per kv head: 256-token splits 1616 GB/s, 4096-token splits 3870 GB/s).
        if (c < 128LL * (Hq / Hkv)) c = 128LL * (Hq / Hkv);
        if (c > 8192) c = 8192;
    }
    c = ((c + 63) / 64) * 64;
    if (c > lmax) c = ((lmax + 63) / 64) * 64;
    if (c < 64) c = 64;
    if (cdiv(lmax, c) * (long long)Hkv > INT32_MAX) return ATTN_ERR_BAD_SHAPE;  // one grid row per (split, kv head)
    *chunk = (int)c;
    *max_splits = cdiv(lmax, c);
    return ATTN_OK;
}

// Shared body of the paged decode entry points. kv_format < 0: bf16 caches; 0 / 1: FP8
// e4m3 / e5m2 caches with the given descales.
static attn_status_t decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* page_table,
                                  const int* seqlens, int page_size, void* o, float* lse, void* stream, int B, int Hq,
                                  int Hkv, int d, int max_pages_per_seq, int num_pages, float scale, int num_splits,
                                  int kv_format, float k_descale, float v_descale) {
    if (!q || !k_cache || !v_cache || !page_table || !seqlens || !o || !lse) return ATTN_ERR_NULL_PTR;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || (d != 64 && d != 128) || page_size <= 0 ||
        max_pages_per_seq <= 0 || num_pages <= 0 || num_splits < 0 || B > 65535 || Hkv > 65535)
        return ATTN_ERR_BAD_SHAPE;
    if ((long long)num_pages * page_size > INT32_MAX) return ATTN_ERR_BAD_SHAPE;  // cache rows are 32-bit indices
    if (!isfinite(scale)) return ATTN_ERR_BAD_SHAPE;
    if (!aligned(q, 16) || !aligned(o, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(lse, 4) ||
        !aligned(page_table, 4) || !aligned(seqlens, 4))
        return ATTN_ERR_ALIGN;
    if (B == 0) return ATTN_OK;
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    int chunk = 0, max_splits = 0;
    st = attn_decode_plan(B, Hq, Hkv, max_pages_per_seq, page_size, num_splits, ds->num_sms, &chunk, &max_splits);
    if (st != ATTN_OK) return st;
    // one grid column per (split, kv head, group of 16 query heads)
    if ((long long)max_splits * Hkv * ((Hq / Hkv + 15) / 16) > INT32_MAX) return ATTN_ERR_BAD_SHAPE;
    const Options opt = options();
    DecodeParams p;
    memset(&p, 0, sizeof p);
    p.q = reinterpret_cast<const __nv_bfloat16*>(q);
    p.k_cache = reinterpret_cast<const __nv_bfloat16*>(k_cache);
    p.v_cache = reinterpret_cast<const __nv_bfloat16*>(v_cache);
    p.page_table = page_table;
    p.seqlens = seqlens;
    p.o = reinterpret_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.g_stride = Hq / Hkv;  // more than 16 per kv head run as groups of 16 within one launch
    p.page_size = page_size;
    p.max_pages = max_pages_per_seq;
    p.num_pages = num_pages;
    p.chunk = chunk;
    p.max_splits = max_splits;
    const double score_scale = kv_format < 0 ? (double)scale : (double)scale * (double)k_descale;
    p.scale = (float)score_scale;
    p.scale_log2 = (float)(score_scale * 1.4426950408889634);
    p.rescale_thr = (float)opt.rescale_threshold;
    p.order = opt.decode_order;
    p.v_descale = kv_format < 0 ? 1.0f : v_descale;
    p.status = ds->status;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void* ws = nullptr;
    if (max_splits > 1) {
        cudaMemPool_t pool = nullptr;
        if ((st = device_pool(ds, &pool)) != ATTN_OK) return st;
        const size_t n_o = (size_t)B * Hq * max_splits * d;
        if (cudaMallocFromPoolAsync(&ws, attn_decode_workspace_bytes(B, Hq, d, max_splits), pool, s) != cudaSuccess)
            return ATTN_ERR_CUDA;
        p.ws_o = reinterpret_cast<float*>(ws);
        p.ws_lse = p.ws_o + n_o;
    }
    cudaError_t e;
    if (kv_format < 0) {
        e = attn::launch_attn_decode(p, d, s);
    } else if (d == 128 && page_size % attn::kDecodeMapRows == 0 && opt.decode_maps) {
        // the 16 tokens of a token group lie in one page: one map load per group and tensor (the
        // launcher keeps the per-row copies for the head counts where those measured faster)
        attn::DecodeTmaps tm;
        if ((st = encode_fn()) != ATTN_OK ||
            (st = make_cache_map(&tm.k, k_cache, (long long)num_pages * page_size, Hkv * d, d)) != ATTN_OK ||
            (st = make_cache_map(&tm.v, v_cache, (long long)num_pages * page_size, Hkv * d, d)) != ATTN_OK) {
            if (ws) cudaFreeAsync(ws, s);
            return st;
        }
        e = attn::launch_attn_decode_fp8_maps(p, tm, d, kv_format, s);
    } else {
        e = attn::launch_attn_decode_fp8(p, d, kv_format, s);
    }
    if (ws) cudaFreeAsync(ws, s);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* page_table,
                                const int* seqlens, int page_size, void* o, float* lse, void* stream, int B, int Hq,
                                int Hkv, int d, int max_pages_per_seq, int num_pages, float scale, int num_splits) {
    return decode_paged(q, k_cache, v_cache, page_table, seqlens, page_size, o, lse, stream, B, Hq, Hkv, d,
                        max_pages_per_seq, num_pages, scale, num_splits, -1, 1.0f, 1.0f);
}

attn_status_t attn_decode_paged_fp8(const void* q, const void* k_cache, const void* v_cache, const int* page_table,
                                    const int* seqlens, int page_size, void* o, float* lse, void* stream, int B,
                                    int Hq, int Hkv, int d, int max_pages_per_seq, int num_pages, float scale,
                                    int num_splits, int kv_format, float k_descale, float v_descale) {
    if (kv_format != ATTN_FP8_E4M3 && kv_format != ATTN_FP8_E5M2) return ATTN_ERR_BAD_ARG;
    if (!isfinite(k_descale) || !isfinite(v_descale)) return ATTN_ERR_BAD_ARG;
    const double score_scale_log2 = (double)scale * (double)k_descale * 1.4426950408889634;
    if (!(fabs(score_scale_log2) <= (double)FLT_MAX)) return ATTN_ERR_BAD_ARG;  // the kernels use it as a float
    return decode_paged(q, k_cache, v_cache, page_table, seqlens, page_size, o, lse, stream, B, Hq, Hkv, d,
                        max_pages_per_seq, num_pages, scale, num_splits, kv_format, k_descale, v_descale);
}

attn_status_t attn_get_device_status(void* stream) {
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int h[4] = {0, 0, 0, 0};
    if (cudaMemcpy(h, ds->status, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    const int zero[4] = {0, 0, 0, 0};
    if (cudaMemcpy(ds->status, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
    return h[0];
}

attn_status_t attn_read_counters(unsigned long long* out, int n) {
    if (!out) return ATTN_ERR_NULL_PTR;
    if (n < 0) return ATTN_ERR_BAD_ARG;
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned long long h[attn::kNumCounters] = {};
    if (cudaMemcpy(h, ds->counters, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    unsigned long long z[attn::kNumCounters] = {};
    if (cudaMemcpy(ds->counters, z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
    for (int i = 0; i < n && i < attn::kNumCounters; ++i) out[i] = h[i];
    return ATTN_OK;
}

attn_status_t attn_debug_exp2(const float* x, float* y, long long n, int mode, void* stream) {
    if (!x || !y) return ATTN_ERR_NULL_PTR;
    if (n < 0 || (mode != 0 && mode != 1)) return ATTN_ERR_BAD_ARG;
    if (!aligned(x, 4) || !aligned(y, 4)) return ATTN_ERR_ALIGN;
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    return attn::launch_exp2_probe(x, y, n, mode, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

attn_status_t attn_debug_watchdog(unsigned long long limit_ns, void* stream) {
    if (limit_ns == 0 || limit_ns > 10000000000ull) return ATTN_ERR_BAD_ARG;
    DeviceState* ds = nullptr;
    attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    return attn::launch_watchdog_probe(ds->status, limit_ns, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
}

}  // extern "C"

namespace attn {
int current_device_info(int** status, int* num_sms) {
    DeviceState* ds = nullptr;
    const attn_status_t st = device_state(&ds);
    if (st != ATTN_OK) return st;
    *status = ds->status;
    *num_sms = ds->num_sms;
    return ATTN_OK;
}
}  // namespace attn
