// Paged-KV split-KV decode for sm_103a (GB300): one query token per sequence.
//
// "Faster, more flexible FA4 for LLM inference":
//  - PR 1999/2104: pages of any size are gathered with per-thread cp.async rather than
//    TMA, and each row's location (page-table lookup, then a 32-bit cache row index) is
//    resolved once per row and handed out by warp shuffles ("transposed" address
//    generation) instead of being recomputed by every thread that copies a piece of it;
//  - PR 1940: split-KV (Flash-Decoding): several CTAs share one sequence's keys, each
//    writes a partial output and its log-sum-exp, and a separate combine kernel merges
//    them; num_splits = 0 picks the split size from the SM count and the lengths;
//  - PR 2186: GQA packing: all query heads of one key/value head are computed from one
//    copy of each K/V row.
// The online-softmax recurrence ("FlashAttention: not computing less, moving less",
// section 02) runs per warp over its tokens; the warps of a CTA and then the splits
// are merged with the same max-shifted LSE weighting.
//
// Split kernel: one CTA of 4 warps per (sequence, split, kv head), the kv heads of one split
// adjacent in the grid, so CTAs running side by side read neighbouring pieces of the same
// cache rows. The grid lists every split but the last of each sequence first and the last
// splits (shorter in general) after them, longest first, so that they fill the SMs freed
// while the last full-length splits finish (LPT); the combine kernel is launched as a
// programmatic dependent and waits on the device, not behind a launch.
// Each warp owns a private cp.async ring of NST stages of 16 tokens (K and V rows,
// 128-byte XOR swizzle) and processes token groups w, w+4, w+8, ... of the split, so the
// main loop needs no CTA-wide barrier. Scores S = Q K^T use m16n8k16 bf16 MMAs with the (up to 16) query
// heads of the group as rows; O^T += V^T P^T reuses the score accumulators as the B
// operand directly.
#include "decode_maps.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

#include <math.h>

namespace attn {
namespace {

constexpr int kWarps = 4;
constexpr int kGroup = 16;  // tokens per warp-stage

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Page-table index and slot of token tok (0 <= tok < 2^31) without an integer division: the
// launcher's multiplier m = ceil(2^(31+k) / page_size), k = ceil(log2 page_size), makes
// floor(tok * m / 2^(31+k)) the exact quotient for every 31-bit tok (Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994).
__device__ __forceinline__ int page_index(const DecodeParams& p, int tok, int& slot) {
    const int q = p.ps_magic ? (int)(__umulhi((unsigned)tok, p.ps_magic) >> p.ps_shift) : tok;
    slot = tok - q * p.page_size;
    return q;
}

template <int D>
struct DecLayout {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTileBytes = kGroup * kRowBytes;  // one K or V warp-stage
    static constexpr int kChunksPerRow = D / 8;             // 16-byte chunks
};

// Byte offset of 16-byte chunk c of row r inside a [16 x D] bf16 warp-stage tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// Sequence whose last split has rank `rank` in decreasing length (ties: lower sequence index
// first), and its length as stored (*raw_len). Every thread of the CTA calls it; scratch holds
// 2 B + 2 ints of shared memory.
__device__ __forceinline__ int seq_of_rank(const DecodeParams& p, int rank, uint8_t* scratch, int* raw_len) {
    int* key = reinterpret_cast<int*>(scratch);
    int* raw = key + p.B;
    int* sel = raw + p.B;
    const long long max_len = (long long)p.max_pages * p.page_size;
    for (int t = threadIdx.x; t < p.B; t += blockDim.x) {
        const int r = __ldg(p.seqlens + t);
        const int len = r < 0 ? 0 : (r > max_len ? (int)max_len : r);
        const int ns = cdiv(len, p.chunk);
        key[t] = len - (ns > 0 ? ns - 1 : 0) * p.chunk;  // tokens of the last split
        raw[t] = r;
    }
    if (threadIdx.x == 0) sel[0] = 0;
    __syncthreads();
    for (int t = threadIdx.x; t < p.B; t += blockDim.x) {
        const int kt = key[t];
        int r = 0;
        for (int u = 0; u < p.B; ++u) {
            const int ku = key[u];
            r += (ku > kt) || (ku == kt && u < t);
        }
        if (r == rank) sel[0] = t;
    }
    __syncthreads();
    const int b = sel[0];
    *raw_len = raw[b];
    __syncthreads();  // the scratch is the ring's memory
    return b;
}

// Work item of a split-kernel CTA: sequence, split (or -1: the sequence's last split) and
// head-group index hg = kv head * n_groups + group. The grid lists every split but the last
// of each sequence (row = sequence, column = split * HG + hg) before the last splits, which
// are shorter in general: CTAs start in grid order, so the short items fill the SMs that
// free up while the last full-length ones finish, the longest first when p.lpt is set.
// Returns false (for the whole CTA) when the CTA has no item. has_len: len holds the
// sequence length as stored (read while ranking).
struct DecItem {
    int b, split, hg, len;
    bool has_len;
};
__device__ __forceinline__ bool decode_item(const DecodeParams& p, uint8_t* scratch, DecItem& it) {
    const int HG = p.Hkv * p.n_groups;
    it.has_len = false;
    it.len = 0;
    if (p.full_rows < 0 || (int)blockIdx.y < p.full_rows) {
        it.b = blockIdx.y;
        it.split = (int)(blockIdx.x / (unsigned)HG);
        it.hg = (int)(blockIdx.x % (unsigned)HG);
        return true;
    }
    const long long j = (long long)(blockIdx.y - p.full_rows) * gridDim.x + blockIdx.x;
    if (j >= (long long)p.B * HG) return false;
    it.hg = (int)(j % HG);
    if (p.lpt) {
        it.b = seq_of_rank(p, (int)(j / HG), scratch, &it.len);
        it.has_len = true;
    } else {
        it.b = (int)(j / HG);
    }
    it.split = -1;
    return true;
}

// Merge the 4 warps' partial results of a split kernel (max-shifted LSE weighting) and
// store: directly as bf16 o / lse when the sequence has one split, else as an fp32 partial
// for the combine kernel. PERM_D: the accumulator rows follow the FP8 kernel's permuted d
// order (row 16 mt + i of O^T holds d = (D/8) i + 2 mt, row 16 mt + i + 8 holds the next d);
// otherwise row r holds d = r. out_scale multiplies the output (the value descale).
template <int D, int GN, bool PERM_D>
__device__ __forceinline__ void merge_and_store(const DecodeParams& p, uint8_t* smem, float (&oacc)[GN / 8][D / 16][4],
                                                float m0, float m1, float l0, float l1, int split, int nsplit, int kvh,
                                                int b, float out_scale, int G, int g_base) {
    constexpr int NH = GN / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g0 = lane >> 2;
    const float sl2 = p.scale_log2;
    // row sums over the quad
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    __syncthreads();  // every warp is done with its ring: reuse shared memory for the merge

    // ---- merge the 4 warps: sm_o[w][head][d], sm_m[w][head], sm_l[w][head]
    float* sm_o = reinterpret_cast<float*>(smem);
    float* sm_m = sm_o + kWarps * GN * D;
    float* sm_l = sm_m + kWarps * GN;
    if ((lane & 3) == 0) {
        sm_m[warp * GN + g0] = m0;
        sm_l[warp * GN + g0] = l0;
        if (GN == 16) {
            sm_m[warp * GN + g0 + 8] = m1;
            sm_l[warp * GN + g0 + 8] = l1;
        }
    }
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            const int hd = nh * 8 + 2 * (lane & 3);
            const int dr0 = PERM_D ? (D / 8) * g0 + 2 * mt : mt * 16 + g0;
            const int dr1 = PERM_D ? dr0 + 1 : dr0 + 8;
            float* base = sm_o + (long long)warp * GN * D;
            base[hd * D + dr0] = oacc[nh][mt][0];
            base[(hd + 1) * D + dr0] = oacc[nh][mt][1];
            base[hd * D + dr1] = oacc[nh][mt][2];
            base[(hd + 1) * D + dr1] = oacc[nh][mt][3];
        }
    __syncthreads();

    const bool direct = nsplit == 1;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int hh = idx / D, d = idx - hh * D;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, sm_m[w * GN + hh]);
        float ll = 0.0f, acc = 0.0f;
        if (mm != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float sw = ex2_mufu((sm_m[w * GN + hh] - mm) * sl2);
                ll += sw * sm_l[w * GN + hh];
                acc += sw * sm_o[(w * GN + hh) * D + d];
            }
        }
        const float o = ll > 0.0f ? acc / ll * out_scale : 0.0f;
        const float lse = ll > 0.0f ? mm * p.scale + logf(ll) : -INFINITY;
        const long long bh = (long long)b * p.Hq + kvh * p.g_stride + g_base + hh;
        if (direct) {
            p.o[bh * D + d] = __float2bfloat16(o);
            if (d == 0) p.lse[bh] = lse;
        } else {
            p.ws_o[(bh * p.max_splits + split) * D + d] = o;
            if (d == 0) p.ws_lse[bh * p.max_splits + split] = lse;
        }
    }
}

template <int D, int GN, int NST>
__global__ void __launch_bounds__(kWarps * 32) decode_split_kernel(const DecodeParams p) {
    grid_dependents_launch();  // the combine kernel may be scheduled once every split CTA runs
    using L = DecLayout<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    // hg = kv head * n_groups + group of 16 query heads: the groups of one kv head are neighbours
    // in launch order, so they read the same cache rows at about the same time and all but the
    // first find them in the L2.
    DecItem item;
    if (!decode_item(p, smem, item)) return;
    const int grp = item.hg % p.n_groups, kvh = item.hg / p.n_groups, b = item.b;
    const int g_base = 16 * grp;
    const int G = p.n_groups > 1 ? min(16, p.g_stride - g_base) : p.g_stride;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long max_len = (long long)p.max_pages * p.page_size;

    int len = item.has_len ? item.len : __ldg(p.seqlens + b);
    if (len < 0 || len > max_len) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevBadIndex);
        len = len < 0 ? 0 : (int)max_len;
    }
    const int nsplit = cdiv(len, p.chunk);
    int split = item.split;
    if (split < 0)
        split = nsplit > 0 ? nsplit - 1 : 0;
    else if (p.full_rows >= 0 && split >= nsplit - 1)
        return;  // the last split has its own CTA after the full rows
    const int t_begin = split * p.chunk;
    if (len == 0) {
        // No cached keys: the output is 0 and the log-sum-exp is -inf (written by split 0).
        if (split == 0) {
            for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
                const int h = kvh * p.g_stride + g_base + i / D;
                p.o[((long long)b * p.Hq + h) * D + (i % D)] = __float2bfloat16(0.0f);
            }
            if (threadIdx.x < G) p.lse[(long long)b * p.Hq + kvh * p.g_stride + g_base + threadIdx.x] = -INFINITY;
        }
        return;
    }
    if (t_begin >= len) return;
    const int t_end = min(len, t_begin + p.chunk);

    // ---- query fragments: rows = query heads of this kv head (padded to 16), k = d
    const int g0 = lane >> 2;
    const int h0 = kvh * p.g_stride + g_base + g0, h1 = kvh * p.g_stride + g_base + g0 + 8;
    const bool v0 = g0 < G, v1 = (GN == 16) && (g0 + 8 < G);
    const uint32_t* q0p = reinterpret_cast<const uint32_t*>(p.q + ((long long)b * p.Hq + h0) * D);
    const uint32_t* q1p = reinterpret_cast<const uint32_t*>(p.q + ((long long)b * p.Hq + h1) * D);
    uint32_t aq[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int c = kk * 8 + (lane & 3);  // u32 index of columns kk*16 + 2*(lane%4)
        aq[kk][0] = v0 ? __ldg(q0p + c) : 0u;
        aq[kk][1] = v1 ? __ldg(q1p + c) : 0u;
        aq[kk][2] = v0 ? __ldg(q0p + c + 4) : 0u;
        aq[kk][3] = v1 ? __ldg(q1p + c + 4) : 0u;
    }

    // ---- per-warp ring
    uint8_t* ring = smem + warp * NST * 2 * L::kTileBytes;
    const uint32_t ring_s = smem_u32(ring);
    const int row_stride = p.Hkv * D;  // elements between consecutive cache rows
    const int* pt = p.page_table + (long long)b * p.max_pages;
    constexpr int kRowsPerIter = 32 / L::kChunksPerRow;
    constexpr int kIters = kGroup / kRowsPerIter;
    const int my_chunk = lane % L::kChunksPerRow;
    const int my_row0 = lane / L::kChunksPerRow;
    const int col = kvh * D + my_chunk * 8;  // this lane's chunk of its kv head's row (Hkv * D < 2^23)

    // groups handled by this warp: t_begin + 16 * (warp + 4 * i)
    const int n_groups_total = cdiv(t_end - t_begin, kGroup);
    const int my_groups = n_groups_total > warp ? cdiv(n_groups_total - warp, kWarps) : 0;

    auto issue = [&](int i) {
        const int slot = i % NST;
        const int g = t_begin + kGroup * (warp + kWarps * i);
        // lane r (r < 16) resolves row r of the group once; others mirror lanes 0-15
        const int tok = g + (lane & 15);
        int row = -1;  // cache row (page * page_size + slot) of this lane's token, -1: none
        if (tok < t_end) {
            int pslot;
            const int pg = __ldg(pt + page_index(p, tok, pslot));
            if (pg >= 0 && pg < p.num_pages)
                row = pg * p.page_size + pslot;  // < num_pages * page_size <= INT32_MAX
            else
                atomicCAS(p.status, 0, kDevBadIndex);
        }
        const uint32_t kdst = ring_s + slot * 2 * L::kTileBytes;
        const uint32_t vdst = kdst + L::kTileBytes;
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
            const int r = it * kRowsPerIter + my_row0;
            const int rr = __shfl_sync(0xffffffffu, row, r);
            const long long ro = (long long)rr * row_stride + col;
            const __nv_bfloat16* ks = rr >= 0 ? p.k_cache + ro : p.k_cache;
            const __nv_bfloat16* vs = rr >= 0 ? p.v_cache + ro : p.v_cache;
            cp_async16(kdst + swz<D>(r, my_chunk), ks, rr >= 0 ? 16u : 0u);
            cp_async16(vdst + swz<D>(r, my_chunk), vs, rr >= 0 ? 16u : 0u);
        }
    };

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    constexpr int NH = GN / 8;
    float oacc[NH][D / 16][4];
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[nh][mt][e] = 0.0f;

    const float sl2 = p.scale_log2;
    // ldmatrix row/chunk for this lane: token (lane % 8) + 8 * (lane / 16), chunk parity (lane / 8) & 1
    const int lm_row = (lane & 7) + ((lane >> 4) << 3);
    const int lm_par = (lane >> 3) & 1;

#pragma unroll
    for (int i = 0; i < NST - 1; ++i) {
        if (i < my_groups) issue(i);
        cp_async_commit();
    }
    for (int i = 0; i < my_groups; ++i) {
        cp_async_wait<NST - 2>();
        __syncwarp();
        if (i + NST - 1 < my_groups) issue(i + NST - 1);
        cp_async_commit();

        const int slot = i % NST;
        const uint32_t kt = ring_s + slot * 2 * L::kTileBytes;
        const uint32_t vt = kt + L::kTileBytes;
        const int g = t_begin + kGroup * (warp + kWarps * i);

        // S = Q K^T : rows = heads, columns = 16 tokens (two n8 tiles)
        float sc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(kt + swz<D>(lm_row, 2 * kk + lm_par), b0, b1, b2, b3);
            mma_bf16_16816(sc[0], aq[kk], b0, b1);
            mma_bf16_16816(sc[1], aq[kk], b2, b3);
        }
        // mask tokens past the split end
        const int tk = g + 2 * (lane & 3);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (tk + nt * 8 + (e & 1) >= t_end) sc[nt][e] = -INFINITY;

        // online softmax per head row (row0 = head g0, row1 = head g0 + 8)
        float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mc0 = fmaxf(m0, mx0), mc1 = fmaxf(m1, mx1);
        const bool need = ((mc0 - m0) * sl2 > p.rescale_thr) || (GN == 16 && (mc1 - m1) * sl2 > p.rescale_thr);
        if (__any_sync(0xffffffffu, need)) {
            const float a0 = (m0 == -INFINITY) ? 0.0f : ex2_mufu((m0 - mc0) * sl2);
            const float a1 = (m1 == -INFINITY) ? 0.0f : ex2_mufu((m1 - mc1) * sl2);
            l0 *= a0;
            l1 *= a1;
            m0 = mc0;
            m1 = mc1;
            // O^T columns are heads 2*(lane%4) and +1 (and +8 for the second n8 tile)
            const int src = (lane & 3) * 8;  // lane holding row 2*(lane%4): lane = 4 * head
            const float c00 = __shfl_sync(0xffffffffu, a0, src);
            const float c01 = __shfl_sync(0xffffffffu, a0, src + 4);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                oacc[0][mt][0] *= c00;
                oacc[0][mt][1] *= c01;
                oacc[0][mt][2] *= c00;
                oacc[0][mt][3] *= c01;
            }
            if (GN == 16) {
                const float c10 = __shfl_sync(0xffffffffu, a1, src);
                const float c11 = __shfl_sync(0xffffffffu, a1, src + 4);
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    oacc[NH - 1][mt][0] *= c10;
                    oacc[NH - 1][mt][1] *= c11;
                    oacc[NH - 1][mt][2] *= c10;
                    oacc[NH - 1][mt][3] *= c11;
                }
            }
        }
        const float n0 = (m0 == -INFINITY) ? 0.0f : -m0 * sl2;
        const float n1 = (m1 == -INFINITY) ? 0.0f : -m1 * sl2;
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            pr[nt][0] = ex2_mufu(fmaf(sc[nt][0], sl2, n0));
            pr[nt][1] = ex2_mufu(fmaf(sc[nt][1], sl2, n0));
            pr[nt][2] = ex2_mufu(fmaf(sc[nt][2], sl2, n1));
            pr[nt][3] = ex2_mufu(fmaf(sc[nt][3], sl2, n1));
        }
        l0 += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        l1 += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
        // P^T as the B operand: k = tokens 2*(lane%4) (+8), n = head lane/4 (+8)
        const uint32_t pb0 = pack_bf16x2(pr[0][0], pr[0][1]);
        const uint32_t pb1 = pack_bf16x2(pr[1][0], pr[1][1]);
        const uint32_t pb2 = pack_bf16x2(pr[0][2], pr[0][3]);
        const uint32_t pb3 = pack_bf16x2(pr[1][2], pr[1][3]);
        // O^T += V^T P^T : rows = d (16 per m-tile), k = 16 tokens
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a[4];
            ldmatrix_x4_trans(vt + swz<D>(lm_row, 2 * mt + lm_par), a[0], a[1], a[2], a[3]);
            mma_bf16_16816(oacc[0][mt], a, pb0, pb1);
            if (GN == 16) mma_bf16_16816(oacc[NH - 1][mt], a, pb2, pb3);
        }
    }
    cp_async_wait<0>();
    merge_and_store<D, GN, false>(p, smem, oacc, m0, m1, l0, l1, split, nsplit, kvh, b, 1.0f, G, g_base);
}

// ---------------------------------------------------------------------------- FP8 caches
// "Faster, more flexible FA4 for LLM inference", PR 2109: key/value caches in 8-bit floating
// point, e4m3 or e5m2. Key code c stands for k_descale * fp8(c) and value code c for
// v_descale * fp8(c) (one factor per tensor). The split kernel keeps the structure of the
// bf16 one (per-warp cp.async rings of 16 tokens, GQA heads as MMA rows, online softmax,
// warp merge) with three changes:
//  - the products are f16 m16n8k16 MMAs. One cvt turns two cached codes into the f16 pair
//    an operand register holds, exactly (every e4m3 and e5m2 value is an f16 value); the
//    query is converted from bf16 to f16 once (exact for |q| in [2^-14, 65504]), and the
//    probabilities are rounded to f16 instead of bf16;
//  - the order of d inside Q K^T is permuted, identically in Q and K, and so is the order of
//    d among the value rows (undone when the output is stored), so that the bytes of each
//    lane's operands are contiguous in shared memory: one 16-byte load feeds several MMAs,
//    without ldmatrix;
//  - k_descale is folded into the softmax scale by the host; v_descale scales the output.

// Byte offset of 16-byte chunk c of row r inside a [16 x D] byte warp-stage tile.
template <int D>
__device__ __forceinline__ uint32_t swz8(int r, int c) {
    constexpr int kChunks = D / 16;
    return (uint32_t)(r * D + ((c ^ (r & (kChunks - 1))) << 4));
}

// Two FP8 codes (low byte first) to an f16 pair (low half first).
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint32_t two_codes) {
    const uint16_t v = (uint16_t)two_codes;
    uint32_t d;
    if (FMT == 0)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
    else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(d) : "h"(v));
    return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t* w) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void lds64(uint32_t addr, uint32_t* w) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(addr) : "memory");
}

// 2-D tiled tensor load into shared memory (dst: shared-window address, 1024-byte aligned for
// the 128-byte swizzle), completing on an mbarrier.
__device__ __forceinline__ void map_load_2d(uint32_t dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Orders this thread's earlier shared-memory accesses before its later bulk copies into shared
// memory (the copies write through the async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Bounded wait for a token group's map loads: false after kStageWaitNs of global time.
constexpr uint64_t kStageWaitNs = 2000000000ull;
__device__ __forceinline__ bool stage_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 15u && global_timer_ns() - t0 > kStageWaitNs) return false;
    }
}

// TG tokens per warp-stage (16 or 32). Launch bound: as many CTAs per SM as their rings fit in
// shared memory, at most four.
template <int D, int TG, int NST>
constexpr int fp8_min_blocks() {
    return (232448 / (kWarps * NST * 2 * TG * D)) < 4 ? (232448 / (kWarps * NST * 2 * TG * D)) : 4;
}

// TM: the K/V rows of a token group come from one tensor-map load each (the group lies within
// one page); else every lane copies 16-byte pieces of its token's rows with cp.async.
template <int D, int GN, int NST, int FMT, int TG, bool TM>
__global__ void __launch_bounds__(kWarps * 32, (fp8_min_blocks<D, TG, NST>()))
    decode_split_fp8_kernel(const DecodeParams p, const __grid_constant__ DecodeTmaps tm) {
    grid_dependents_launch();  // the combine kernel may be scheduled once every split CTA runs
    static_assert(TG == 16 || TG == 32, "tokens per warp-stage");
    static_assert(!TM || (D == 128 && TG == kDecodeMapRows), "map loads: 128-byte rows, one group per load");
    constexpr int kTile = TG * D;       // bytes of one K or V warp-stage tile
    constexpr int NT = TG / 8;          // n-tiles of 8 tokens in S = Q K^T
    constexpr int KS = TG / 16;         // k-steps of 16 tokens in O^T += V^T P^T
    constexpr int kChunks = D / 16;     // 16-byte chunks per cache row
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // map loads write the 128-byte swizzle relative to 1024-byte boundaries: the rings start on one
    uint8_t* smem = TM ? smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u) : smem_raw;
    // hg = kv head * n_groups + group of 16 query heads: the groups of one kv head are neighbours
    // in launch order, so they read the same cache rows at about the same time and all but the
    // first find them in the L2.
    DecItem item;
    if (!decode_item(p, smem, item)) return;
    const int grp = item.hg % p.n_groups, kvh = item.hg / p.n_groups, b = item.b;
    const int g_base = 16 * grp;
    const int G = p.n_groups > 1 ? min(16, p.g_stride - g_base) : p.g_stride;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long max_len = (long long)p.max_pages * p.page_size;

    int len = item.has_len ? item.len : __ldg(p.seqlens + b);
    if (len < 0 || len > max_len) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, kDevBadIndex);
        len = len < 0 ? 0 : (int)max_len;
    }
    const int nsplit = cdiv(len, p.chunk);
    int split = item.split;
    if (split < 0)
        split = nsplit > 0 ? nsplit - 1 : 0;
    else if (p.full_rows >= 0 && split >= nsplit - 1)
        return;  // the last split has its own CTA after the full rows
    const int t_begin = split * p.chunk;
    if (len == 0) {
        if (split == 0) {
            for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
                const int h = kvh * p.g_stride + g_base + i / D;
                p.o[((long long)b * p.Hq + h) * D + (i % D)] = __float2bfloat16(0.0f);
            }
            if (threadIdx.x < G) p.lse[(long long)b * p.Hq + kvh * p.g_stride + g_base + threadIdx.x] = -INFINITY;
        }
        return;
    }
    if (t_begin >= len) return;
    const int t_end = min(len, t_begin + p.chunk);

    // ---- query fragments (f16), rows = query heads of this kv head. Permuted d: column
    // 2 qd + e of k-step kk is d = (D/4) qd + 4 kk + e, column 2 qd + 8 + e is that + 2.
    const int g0 = lane >> 2, qd = lane & 3;
    const int h0 = kvh * p.g_stride + g_base + g0, h1 = kvh * p.g_stride + g_base + g0 + 8;
    const bool v0 = g0 < G, v1 = (GN == 16) && (g0 + 8 < G);
    const uint32_t* q0p = reinterpret_cast<const uint32_t*>(p.q + ((long long)b * p.Hq + h0) * D);
    const uint32_t* q1p = reinterpret_cast<const uint32_t*>(p.q + ((long long)b * p.Hq + h1) * D);
    uint32_t aq[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int c = (D / 8) * qd + 2 * kk;  // u32 index of d = (D/4) qd + 4 kk
        aq[kk][0] = v0 ? bf16x2_to_f16x2(__ldg(q0p + c)) : 0u;
        aq[kk][1] = v1 ? bf16x2_to_f16x2(__ldg(q1p + c)) : 0u;
        aq[kk][2] = v0 ? bf16x2_to_f16x2(__ldg(q0p + c + 1)) : 0u;
        aq[kk][3] = v1 ? bf16x2_to_f16x2(__ldg(q1p + c + 1)) : 0u;
    }

    // ---- per-warp ring of NST stages x (K tile, V tile), 16 rows of D bytes each
    uint8_t* ring = smem + warp * NST * 2 * kTile;
    const uint32_t ring_s = smem_u32(ring);
    const uint8_t* kc = reinterpret_cast<const uint8_t*>(p.k_cache);
    const uint8_t* vc = reinterpret_cast<const uint8_t*>(p.v_cache);
    const int* pt = p.page_table + (long long)b * p.max_pages;
    constexpr int kRowsPerIter = 32 / kChunks;
    constexpr int kIters = TG / kRowsPerIter;
    const int my_chunk = lane % kChunks;
    const int my_row0 = lane / kChunks;
    const int col = kvh * D + my_chunk * 16;  // this lane's chunk of its kv head's row (Hkv * D < 2^23)
    const int n_groups_total = cdiv(t_end - t_begin, TG);
    const int my_groups = n_groups_total > warp ? cdiv(n_groups_total - warp, kWarps) : 0;

    const int row_stride = p.Hkv * D;  // bytes between consecutive cache rows
    auto issue = [&](int i) {
        const int slot = i % NST;
        const int g = t_begin + TG * (warp + kWarps * i);
        const int tok = g + (lane & (TG - 1));
        int row = -1;  // cache row (page * page_size + slot) of this lane's token, -1: none
        if (tok < t_end) {
            int pslot;
            const int pg = __ldg(pt + page_index(p, tok, pslot));
            if (pg >= 0 && pg < p.num_pages)
                row = pg * p.page_size + pslot;  // < num_pages * page_size <= INT32_MAX
            else
                atomicCAS(p.status, 0, kDevBadIndex);
        }
        const uint32_t kdst = ring_s + slot * 2 * kTile;
        const uint32_t vdst = kdst + kTile;
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
            const int r = it * kRowsPerIter + my_row0;
            const int rr = __shfl_sync(0xffffffffu, row, r);
            const long long ro = (long long)rr * row_stride + col;
            cp_async16(kdst + swz8<D>(r, my_chunk), rr >= 0 ? kc + ro : kc, rr >= 0 ? 16u : 0u);
            cp_async16(vdst + swz8<D>(r, my_chunk), rr >= 0 ? vc + ro : vc, rr >= 0 ? 16u : 0u);
        }
    };

    // map loads: one barrier per warp-stage after the rings (one arrival: lane 0, with the bytes)
    uint64_t* sbar = reinterpret_cast<uint64_t*>(smem + kWarps * NST * 2 * kTile) + warp * NST;
    if constexpr (TM) {
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < NST; ++i) mbar_init(&sbar[i], 1);
            fence_mbar_init();
        }
        __syncwarp();
    }
    auto issue_map = [&](int i) {
        if (lane == 0) {
            const int slot = i % NST;
            const int g = t_begin + TG * (warp + kWarps * i);  // a multiple of 16: the group lies in one page
            int pslot;
            const int pg = __ldg(pt + page_index(p, g, pslot));
            // a page index out of range is not read: the copy starts at the first row past the
            // cache (num_pages * page_size <= INT32_MAX), so the map fills the rows with zeros,
            // as the per-row copies do
            int row0 = p.num_pages * p.page_size;
            if (pg >= 0 && pg < p.num_pages)
                row0 = pg * p.page_size + pslot;
            else
                atomicCAS(p.status, 0, kDevBadIndex);
            uint64_t* bar = &sbar[slot];
            fence_async_smem();  // the warp's reads of this slot (ordered by __syncwarp) before the copies
            mbar_arrive_expect_tx(bar, 2 * kTile);
            const uint32_t kdst = ring_s + slot * 2 * kTile;
            map_load_2d(kdst, &tm.k, bar, kvh * D, row0);
            map_load_2d(kdst + kTile, &tm.v, bar, kvh * D, row0);
        }
    };

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    constexpr int NH = GN / 8;
    float oacc[NH][D / 16][4];
#pragma unroll
    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[nh][mt][e] = 0.0f;
    const float sl2 = p.scale_log2;

    if constexpr (TM) {
        for (int i = 0; i < NST - 1 && i < my_groups; ++i) issue_map(i);
    } else {
#pragma unroll
        for (int i = 0; i < NST - 1; ++i) {
            if (i < my_groups) issue(i);
            cp_async_commit();
        }
    }
    for (int i = 0; i < my_groups; ++i) {
        const int slot = i % NST;
        const uint32_t kt = ring_s + slot * 2 * kTile;
        const uint32_t vt = kt + kTile;
        const int g = t_begin + TG * (warp + kWarps * i);
        if constexpr (TM) {
            if (!__all_sync(0xffffffffu, stage_wait(&sbar[slot], (uint32_t)(i / NST) & 1u))) {
                // loads that never landed: report, let the groups in flight land (bounded), and
                // leave the loop (the warp still takes part in the merge's barriers)
                if (lane == 0) atomicCAS(p.status, 0, kDevTimeout);
                for (int j = i + 1; j < i + NST - 1 && j < my_groups; ++j) stage_wait(&sbar[j % NST], (uint32_t)(j / NST) & 1u);
                break;
            }
            __syncwarp();
            if (i + NST - 1 < my_groups) issue_map(i + NST - 1);
            if (g + TG > t_end) {
                // rows past the sequence's end come from the same page but need not hold finite
                // codes: zero their V rows (their scores are masked below)
                const int nv = t_end - g;
                for (int c = lane; c < (TG - nv) * kChunks; c += 32)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vt + (nv + c / kChunks) * D +
                                                                                 (c % kChunks) * 16),
                                 "r"(0u)
                                 : "memory");
                __syncwarp();
            }
        } else {
            cp_async_wait<NST - 2>();
            __syncwarp();
            if (i + NST - 1 < my_groups) issue(i + NST - 1);
            cp_async_commit();
        }

        // K operand bytes: tokens g0 + 8 nt, bytes [(D/4) qd, (D/4) qd + D/4) of the row
        uint32_t kw[NT][D / 16];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < D / 64; ++j) lds128(kt + swz8<D>(g0 + 8 * nt, (D / 64) * qd + j), &kw[nt][4 * j]);
        // S = Q K^T : rows = heads, columns = TG tokens (NT n8 tiles)
        float sc[NT][4] = {};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma_f16_16816(sc[nt], aq[kk], fp8x2_to_f16x2<FMT>(kw[nt][kk]), fp8x2_to_f16x2<FMT>(kw[nt][kk] >> 16));
        const int tk = g + 2 * qd;
        if (TG == 16 || g + TG > t_end) {  // (the 16-token form is the one measured fastest at d = 128)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (tk + nt * 8 + (e & 1) >= t_end) sc[nt][e] = -INFINITY;
        }

        // online softmax per head row (row0 = head g0, row1 = head g0 + 8)
        float mx0, mx1;
        if constexpr (TG == 16) {
            mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
            mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        } else {
            mx0 = fmaxf(sc[0][0], sc[0][1]);
            mx1 = fmaxf(sc[0][2], sc[0][3]);
#pragma unroll
            for (int nt = 1; nt < NT; ++nt) {
                mx0 = max3f(mx0, sc[nt][0], sc[nt][1]);
                mx1 = max3f(mx1, sc[nt][2], sc[nt][3]);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mc0 = fmaxf(m0, mx0), mc1 = fmaxf(m1, mx1);
        const bool need = ((mc0 - m0) * sl2 > p.rescale_thr) || (GN == 16 && (mc1 - m1) * sl2 > p.rescale_thr);
        if (__any_sync(0xffffffffu, need)) {
            const float a0 = (m0 == -INFINITY) ? 0.0f : ex2_mufu((m0 - mc0) * sl2);
            const float a1 = (m1 == -INFINITY) ? 0.0f : ex2_mufu((m1 - mc1) * sl2);
            l0 *= a0;
            l1 *= a1;
            m0 = mc0;
            m1 = mc1;
            const int src = qd * 8;  // lane holding head 2 qd: lane = 4 * head
            const float c00 = __shfl_sync(0xffffffffu, a0, src);
            const float c01 = __shfl_sync(0xffffffffu, a0, src + 4);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                oacc[0][mt][0] *= c00;
                oacc[0][mt][1] *= c01;
                oacc[0][mt][2] *= c00;
                oacc[0][mt][3] *= c01;
            }
            if (GN == 16) {
                const float c10 = __shfl_sync(0xffffffffu, a1, src);
                const float c11 = __shfl_sync(0xffffffffu, a1, src + 4);
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    oacc[NH - 1][mt][0] *= c10;
                    oacc[NH - 1][mt][1] *= c11;
                    oacc[NH - 1][mt][2] *= c10;
                    oacc[NH - 1][mt][3] *= c11;
                }
            }
        }
        const float n0 = (m0 == -INFINITY) ? 0.0f : -m0 * sl2;
        const float n1 = (m1 == -INFINITY) ? 0.0f : -m1 * sl2;
        float pr[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            pr[nt][0] = ex2_mufu(fmaf(sc[nt][0], sl2, n0));
            pr[nt][1] = ex2_mufu(fmaf(sc[nt][1], sl2, n0));
            pr[nt][2] = ex2_mufu(fmaf(sc[nt][2], sl2, n1));
            pr[nt][3] = ex2_mufu(fmaf(sc[nt][3], sl2, n1));
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            l0 += (pr[2 * ks][0] + pr[2 * ks][1]) + (pr[2 * ks + 1][0] + pr[2 * ks + 1][1]);
            l1 += (pr[2 * ks][2] + pr[2 * ks][3]) + (pr[2 * ks + 1][2] + pr[2 * ks + 1][3]);
        }
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            // the P^T operand of tokens 16 ks .. 16 ks + 15 (n-tiles 2 ks and 2 ks + 1)
            const uint32_t pb0 = pack_f16x2(pr[2 * ks][0], pr[2 * ks][1]);
            const uint32_t pb1 = pack_f16x2(pr[2 * ks + 1][0], pr[2 * ks + 1][1]);
            const uint32_t pb2 = pack_f16x2(pr[2 * ks][2], pr[2 * ks][3]);
            const uint32_t pb3 = pack_f16x2(pr[2 * ks + 1][2], pr[2 * ks + 1][3]);
            // V operand bytes: tokens 16 ks + {2qd, 2qd+1, 2qd+8, 2qd+9}; bytes [(D/8) g0, (D/8) g0 + D/8).
            // Row 16 mt + g0 of V^T is d = (D/8) g0 + 2 mt, row 16 mt + g0 + 8 is d + 1.
            uint32_t vw[4][D / 32];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int tok = 16 * ks + 2 * qd + (t & 1) + 8 * (t >> 1);
                if (D == 128)
                    lds128(vt + swz8<D>(tok, g0), vw[t]);
                else
                    lds64(vt + swz8<D>(tok, g0 >> 1) + (g0 & 1) * 8, vw[t]);
            }
            // O^T += V^T P^T : rows = permuted d (16 per m-tile), k = 16 tokens
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;  // bytes 2j and 2j+1 of both tokens
                const uint32_t lo = __byte_perm(vw[0][mt >> 1], vw[1][mt >> 1], sel);
                const uint32_t hi = __byte_perm(vw[2][mt >> 1], vw[3][mt >> 1], sel);
                const uint32_t a[4] = {fp8x2_to_f16x2<FMT>(lo), fp8x2_to_f16x2<FMT>(lo >> 16), fp8x2_to_f16x2<FMT>(hi),
                                       fp8x2_to_f16x2<FMT>(hi >> 16)};
                mma_f16_16816(oacc[0][mt], a, pb0, pb1);
                if (GN == 16) mma_f16_16816(oacc[NH - 1][mt], a, pb2, pb3);
            }
        }
    }
    if constexpr (!TM) cp_async_wait<0>();
    merge_and_store<D, GN, true>(p, smem, oacc, m0, m1, l0, l1, split, nsplit, kvh, b, p.v_descale, G, g_base);
}

// One warp per (sequence, query head of this launch): LSE = log sum_s exp(lse_s) (max-shifted,
// warp shuffles over the splits), O = sum_s exp(lse_s - LSE) O_s, summed in split order.
// Launched as a programmatic dependent of the split kernel: its CTAs may start while the last
// split CTAs run. What the split kernel does not write (the lengths) is read before waiting for
// that grid to finish; after it, the split LSEs and the first 8 partial rows are loaded together.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // row (b, kv head, g) of this launch's heads -> query row b * Hq + kvh * g_stride + g_base + g
    const long long row = (long long)blockIdx.x * 4 + warp;
    const long long per_b = (long long)p.Hkv * p.G;
    const bool active = row < (long long)p.B * per_b;
    const int b = active ? (int)(row / per_b) : 0;
    const int rem = active ? (int)(row - b * per_b) : 0;
    const long long bh = (long long)b * p.Hq + (long long)(rem / p.G) * p.g_stride + p.g_base + rem % p.G;
    const long long max_len = (long long)p.max_pages * p.page_size;
    int len = active ? __ldg(p.seqlens + b) : 0;
    len = len < 0 ? 0 : (len > max_len ? (int)max_len : len);
    const int ns = cdiv(len, p.chunk);
    grid_dependency_wait();
    if (ns <= 1) return;  // written directly by the split kernel
    constexpr int PER = D / 32;
    constexpr int UNR = 8;  // partial rows loaded before any is accumulated
    const float* wl = p.ws_lse + bh * p.max_splits;
    const float* wo = p.ws_o + bh * p.max_splits * D + lane * PER;
    auto load_rows = [&](int s0, int cnt, float (&v)[UNR][PER]) {
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const float* src = wo + (long long)(s0 + min(u, cnt - 1)) * D;  // clamped: always a valid row
            if (PER == 4) {
                const float4 t = *reinterpret_cast<const float4*>(src);
                v[u][0] = t.x;
                v[u][1 % PER] = t.y;
                v[u][2 % PER] = t.z;
                v[u][3 % PER] = t.w;
            } else {
                const float2 t = *reinterpret_cast<const float2*>(src);
                v[u][0] = t.x;
                v[u][1 % PER] = t.y;
            }
        }
    };
    float v[UNR][PER];
    const float l_first = lane < ns ? wl[lane] : -INFINITY;
    load_rows(0, min(UNR, ns), v);
    float mx = l_first;
    for (int s = lane + 32; s < ns; s += 32) mx = fmaxf(mx, wl[s]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.0f;
    if (mx != -INFINITY) {
        sum = lane < ns ? __expf(l_first - mx) : 0.0f;
        for (int s = lane + 32; s < ns; s += 32) sum += __expf(wl[s] - mx);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float lse = sum > 0.0f ? mx + logf(sum) : -INFINITY;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
    if (sum > 0.0f) {
        for (int s0 = 0; s0 < ns; s0 += 32) {
            const int cnt32 = min(32, ns - s0);  // warp-uniform
            // the weight of split s0 + i sits in lane i
            const float w_lane = lane < cnt32 ? __expf((s0 == 0 ? l_first : wl[s0 + lane]) - lse) : 0.0f;
            for (int j = 0; j < cnt32; j += UNR) {
                if (s0 + j > 0) load_rows(s0 + j, min(UNR, cnt32 - j), v);
#pragma unroll
                for (int u = 0; u < UNR; ++u) {
                    const float w = __shfl_sync(0xffffffffu, w_lane, (j + u) & 31);
                    if (j + u < cnt32) {
#pragma unroll
                        for (int e = 0; e < PER; ++e) acc[e] += w * v[u][e];
                    }
                }
            }
        }
    }
    __nv_bfloat16* out = p.o + bh * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(out + e) = pack_bf16x2(acc[e], acc[e + 1]);
    if (lane == 0) p.lse[bh] = lse;
}

// Grid of a split kernel, and the work order it encodes (p.full_rows, p.lpt): rows 0..B-1
// hold the splits before the last of each sequence (column = split * HG + head group), the
// rows after them the last split of every sequence, HG columns each, in decreasing length for
// up to 256 sequences (each CTA of that part ranks the B lengths). Within a row the head
// groups of one kv head, then the kv heads of one split, are neighbours. With too many rows
// for the grid (more than 32767 sequences), or with p.order = 0, row b holds all splits of
// sequence b.
dim3 split_grid(DecodeParams& p) {
    const long long HG = (long long)p.Hkv * p.n_groups;
    const long long X = (p.max_splits > 1 ? p.max_splits - 1 : 1) * HG;
    const long long full_rows = p.max_splits > 1 ? p.B : 0;
    const long long part_rows = ((long long)p.B * HG + X - 1) / X;
    if (p.order != 0 && full_rows + part_rows <= 65535) {
        p.full_rows = (int)full_rows;
        p.lpt = p.B <= 256;
        return dim3((unsigned)X, (unsigned)(full_rows + part_rows));
    }
    p.full_rows = -1;
    p.lpt = 0;
    return dim3((unsigned)(p.max_splits * HG), (unsigned)p.B);
}

// The combine kernel after a split kernel on the same stream, as its programmatic dependent.
template <int D>
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream) {
    const long long rows = (long long)p.B * p.Hkv * p.G;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, p);
}

template <int D, int GN, int NST>
cudaError_t launch_t(DecodeParams p, cudaStream_t stream) {
    constexpr int ring = kWarps * NST * 2 * DecLayout<D>::kTileBytes;
    constexpr int merge = (kWarps * GN * D + 2 * kWarps * GN) * 4;
    constexpr int bytes = ring > merge ? ring : merge;
    static std::atomic<bool> attr_set[kMaxAttrDevices];
    cudaError_t e = ensure_smem_attr(decode_split_kernel<D, GN, NST>, bytes, attr_set);
    if (e != cudaSuccess) return e;
    const dim3 grid = split_grid(p);
    decode_split_kernel<D, GN, NST><<<grid, kWarps * 32, bytes, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.max_splits > 1) e = launch_combine<D>(p, stream);
    return e;
}

template <int D, int GN, int NST, int FMT, int TG, bool TM>
cudaError_t launch_fp8_t(DecodeParams p, const DecodeTmaps& tm, cudaStream_t stream) {
    constexpr int ring = kWarps * NST * 2 * TG * D;
    constexpr int merge = (kWarps * GN * D + 2 * kWarps * GN) * 4;
    // map loads: the stage barriers after the rings, and up to 1 KB to align the rings
    constexpr int bytes = (ring > merge ? ring : merge) + (TM ? kWarps * NST * 8 + 1024 : 0);
    static std::atomic<bool> attr_set[kMaxAttrDevices];
    cudaError_t e = ensure_smem_attr(decode_split_fp8_kernel<D, GN, NST, FMT, TG, TM>, bytes, attr_set);
    if (e != cudaSuccess) return e;
    const dim3 grid = split_grid(p);
    decode_split_fp8_kernel<D, GN, NST, FMT, TG, TM><<<grid, kWarps * 32, bytes, stream>>>(p, tm);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.max_splits > 1) e = launch_combine<D>(p, stream);
    return e;
}

// Tokens per warp-stage of the 8-bit kernels, three stages each: 16 at d = 128 (48 KB of rings per
// CTA, four CTAs per SM), 32 at d = 64 (the same 48 KB). Measured on the paged decode workload
// with e4m3 caches: d = 128, 16 tokens 6100 GB/s against 5755 for 32 (two CTAs per SM) and 6070
// for 32 tokens in two stages; d = 64 (Hkv 16), 32 tokens 6178 against 5250 for 16.
// Map loads (tm != nullptr) against per-row copies, e4m3 paged decode workload (64 sequences of
// U[1024, 32768] tokens, page 16): 4 query heads per kv head 6450 against 6415 GB/s, 32 (two
// groups of 16) 2526 against 2437; 16 query heads per kv head 5420 against 5470, so that shape
// keeps the per-row copies.
template <int FMT>
cudaError_t launch_fp8_fmt(const DecodeParams& p, const DecodeTmaps* tm, int d, cudaStream_t stream) {
    constexpr int NST = 3;
    static const DecodeTmaps no_maps = {};
    if (d == 128 && tm && (p.G <= 8 || p.n_groups > 1))
        return p.G <= 8 ? launch_fp8_t<128, 8, NST, FMT, 16, true>(p, *tm, stream)
                        : launch_fp8_t<128, 16, NST, FMT, 16, true>(p, *tm, stream);
    if (d == 128)
        return p.G <= 8 ? launch_fp8_t<128, 8, NST, FMT, 16, false>(p, no_maps, stream)
                        : launch_fp8_t<128, 16, NST, FMT, 16, false>(p, no_maps, stream);
    return p.G <= 8 ? launch_fp8_t<64, 8, NST, FMT, 32, false>(p, no_maps, stream)
                    : launch_fp8_t<64, 16, NST, FMT, 32, false>(p, no_maps, stream);
}

}  // namespace

// The query heads of a kv head are the rows of the kernels' tensor-core products (at most 16):
// more than 16 run as one launch (split kernel, then combine) per group of 16.
// The split kernels take at most 16 query heads of a kv head (the rows of their tensor-core
// products); more run as groups of 16 in the same launch, one CTA per group, neighbours in the
// grid (so the groups share the cache rows in the L2). The combine then merges all heads.
static DecodeParams grouped(const DecodeParams& p_in) {
    DecodeParams p = p_in;
    // page divisor: m = ceil(2^(31+k) / page_size) < 2^32 with k = ceil(log2 page_size)
    p.ps_magic = 0;
    p.ps_shift = 0;
    if (p.page_size > 1) {
        int k = 0;
        while ((1LL << k) < p.page_size) ++k;
        const unsigned long long num = 1ULL << (31 + k);
        p.ps_magic = (unsigned)((num + (unsigned long long)p.page_size - 1) / (unsigned long long)p.page_size);
        p.ps_shift = k - 1;
    }
    p.n_groups = (p_in.g_stride + 15) / 16;
    p.g_base = 0;
    p.G = p_in.g_stride;
    return p;
}

cudaError_t launch_attn_decode_fp8(const DecodeParams& p_in, int d, int fmt, cudaStream_t stream) {
    const DecodeParams p = grouped(p_in);
    return fmt == 0 ? launch_fp8_fmt<0>(p, nullptr, d, stream) : launch_fp8_fmt<1>(p, nullptr, d, stream);
}

cudaError_t launch_attn_decode_fp8_maps(const DecodeParams& p_in, const DecodeTmaps& tm, int d, int fmt,
                                        cudaStream_t stream) {
    if (d != 128 || p_in.page_size % kDecodeMapRows != 0) return cudaErrorInvalidValue;
    const DecodeParams p = grouped(p_in);
    return fmt == 0 ? launch_fp8_fmt<0>(p, &tm, d, stream) : launch_fp8_fmt<1>(p, &tm, d, stream);
}

cudaError_t launch_attn_decode(const DecodeParams& p_in, int d, cudaStream_t stream) {
    constexpr int NST = 3;
    const DecodeParams p = grouped(p_in);
    return d == 128 ? (p.G <= 8 ? launch_t<128, 8, NST>(p, stream) : launch_t<128, 16, NST>(p, stream))
                    : (p.G <= 8 ? launch_t<64, 8, NST>(p, stream) : launch_t<64, 16, NST>(p, stream));
}

}  // namespace attn
