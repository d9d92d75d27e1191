// Paged decode that allocates nothing: the split-KV partial outputs live in a fixed
// device array that is part of the library image instead of memory taken per call.
//
// Meant for callers that cannot call cudaMalloc (or any allocator) at the point where they
// run attention: for example a serving engine that has already handed nearly all device
// memory to its own KV-cache pool, or code that must not enter the driver's allocator
// because that can block the device or fail late under memory pressure.
#include "attn.h"
#include "kernels.cuh"

#include <math.h>
#include <mutex>
#include <string.h>

namespace {

// Fixed scratch for the split partials: [B, Hq, splits, d] fp32 outputs followed by
// [B, Hq, splits] fp32 log-sum-exps. Every GPU that loads the library keeps it until exit.
constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device. In host code the array's
// name is only a host-side stand-in, so the address comes from cudaGetSymbolAddress, once
// per device, with that device current.
attn_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return ATTN_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" attn_status_t attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                   const int* page_table, const int* seqlens, int page_size, void* o,
                                                   float* lse, void* stream, int B, int Hq, int Hkv, int d,
                                                   int max_pages_per_seq, int num_pages, float scale, int num_splits) {
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
    int* status = nullptr;
    int num_sms = 0;
    attn_status_t st = attn::current_device_info(&status, &num_sms);
    if (st != ATTN_OK) return st;
    int chunk = 0, max_splits = 0;
    st = attn_decode_plan(B, Hq, Hkv, max_pages_per_seq, page_size, num_splits, num_sms, &chunk, &max_splits);
    if (st != ATTN_OK) return st;
    // one grid column per (split, kv head, group of 16 query heads)
    if ((long long)max_splits * Hkv * ((Hq / Hkv + 15) / 16) > INT32_MAX) return ATTN_ERR_BAD_SHAPE;
    const size_t n_o = (size_t)B * Hq * max_splits * d;
    const size_t n_l = (size_t)B * Hq * max_splits;
    if (max_splits > 1 && (n_o + n_l) * sizeof(float) > kScratchBytes) return ATTN_ERR_SCRATCH_TOO_SMALL;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != ATTN_OK) return st;
    double rescale = 8.0;
    attn_get_option("rescale_threshold", &rescale);
    double order = 1.0;
    attn_get_option("decode_order", &order);

    attn::DecodeParams p;
    memset(&p, 0, sizeof p);
    p.q = reinterpret_cast<const __nv_bfloat16*>(q);
    p.k_cache = reinterpret_cast<const __nv_bfloat16*>(k_cache);
    p.v_cache = reinterpret_cast<const __nv_bfloat16*>(v_cache);
    p.page_table = page_table;
    p.seqlens = seqlens;
    p.o = reinterpret_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    // The combine reads only partials of the same call, all written by the split kernel
    // first, so nothing in the scratch has to start at zero.
    p.ws_o = reinterpret_cast<float*>(scratch);
    p.ws_lse = p.ws_o + n_o;
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
    p.scale = scale;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.rescale_thr = (float)rescale;
    p.order = (int)order;
    p.status = status;
    const cudaError_t e = attn::launch_attn_decode(p, d, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
