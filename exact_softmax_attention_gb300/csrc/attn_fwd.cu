// Exact softmax attention forward for sm_103a (GB300).
//
// Computes O = softmax(scale * Q K^T + mask) V and the per-row log-sum-exp with the
// online-softmax recurrence ("FlashAttention: not computing less, moving less",
// section 02: running max m, sum l, unnormalised accumulator a, rescale by
// exp(m - m'), o = a / l at the end), so no score tile ever leaves the SM.
//
// One persistent CTA per SM walks a list of work tiles (sequence, query head,
// 256-row query block = two 128-row Q tiles). Warp roles (16 warps):
//   warp 0       TMA producer: Q tiles once per work tile, then a ring of K/V tiles
//   warps 1-2    MMA issuers, one per Q tile: S = Q K^T and O += P V with tcgen05.mma,
//                accumulators in tensor memory; warp 1 owns the TMEM allocation
//   warps 4-7    softmax for Q tile 0, warps 8-11 softmax for Q tile 1: one thread per
//                row reads S from TMEM, masks, takes the row max, decides whether to
//                rescale O (warp-uniform, only when the max grew by more than the
//                threshold), computes exponentials (MUFU ex2 and, optionally, a cubic
//                polynomial on the FMA pipes for a fraction of columns), row sums, and
//                writes P as bf16 into TMEM over S in two stages (keys 0-95, then 96-127),
//                each signalled at once, so that O += P V starts on the first three
//                quarters while the last quarter is computed ("FlashAttention-4:
//                Blackwell algorithm-pipeline co-design", section on warp roles and
//                barriers; "FlashAttention4 精读", P staging)
//   warps 12-15  epilogue: O / l, LSE, bf16 store of finished rows
// The GEMM issue order per KV step follows the two-tile ping-pong of
// "Low-precision FA4" section 2.1.1 (S0 = Q0 K0, S1 = Q1 K0; then O0 += P0 V_n,
// S0 = Q0 K_{n+1}, O1 += P1 V_n, S1 = Q1 K_{n+1}; then the last two PV products).
// The conditional rescale follows "FlashAttention-4: Blackwell algorithm-pipeline
// co-design", section "conditional softmax rescaling", and "FlashAttention4 精读"
// section 3.1.4 (warp-uniform decision).
//
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512); P_s (bf16,
// 64 columns) overlays the first half of S_s. Because S_s(n) is issued after
// PV_s(n-1) by the same thread, the S_s(n) completion barrier also covers
// PV_s(n-1), so the softmax warps may rescale O_s right after reading S_s(n).
#include "kernels.cuh"
#include "ptx.cuh"

#include <math.h>

namespace attn {
namespace {

constexpr int BM = 128;  // rows per Q tile
constexpr int BN = 128;  // keys per K/V tile
constexpr int kBNWide = 96;  // keys per K/V tile when Q/K rows are 192 wide (shared-memory bound)
constexpr int kThreads = 512;
constexpr int kMaxVarlenB = 1024;
constexpr int kMaxLevels = 2048;  // 256-row blocks per packed sequence for the level order
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
constexpr int kReqRescale = 1, kReqEpilogue = 3;  // request codes of the correction role (+ Q tile)
constexpr uint32_t kTmemCols = 512;

// D: width of queries and keys; DV: width of values and outputs; BNT: keys per K/V tile.
template <int D, int F8 = 0, int DV = D, int BNT = BN>
struct Layout {
    // F8 != 0: Q, K and V arrive as 8-bit floating-point codes (1 = e4m3, 2 = e5m2); V is
    // widened to f16 in shared memory before the P V product.
    static constexpr int kElem = F8 ? 1 : 2;             // bytes per loaded Q/K/V element
    static constexpr int kQBytes = BM * D * kElem;
    static constexpr int kKBytes = BNT * D * kElem;      // K tile as loaded
    static constexpr int kV8Bytes = F8 ? BNT * DV : 0;   // 8-bit V tile as loaded
    static constexpr int kVBytes = BNT * DV * 2;         // 16-bit V tile read by the MMA
    // Ring entry n holds what burst n reads: K tile n (for S = Q K_n^T) and V tile n-1
    // (for O += P_{n-1} V_{n-1}); with 8-bit inputs also the 8-bit V tile it is widened from.
    static constexpr int kV8Off = kKBytes;
    static constexpr int kVOff = kKBytes + kV8Bytes;
    static constexpr int kEntryBytes = kKBytes + kV8Bytes + kVBytes;
    static constexpr int kEntries = (D == 64) ? 4 : 2;
    static constexpr int kChunks = D * kElem / 128;      // 128-byte swizzle chunks per Q/K row
    static constexpr int kVChunks = DV / 64;             // 128-byte chunks per 16-bit V row
    static constexpr int kChunkBytesQ = BM * 128;        // one [BM rows x 128 bytes] chunk
    static constexpr int kChunkBytesKV = BNT * 128;      // one [BNT rows x 128 bytes] chunk
    // packed-sequence order tables: smaller where Q/K tiles leave less shared memory
    static constexpr int kMaxB = D > 128 ? 256 : kMaxVarlenB;
    static constexpr int kMaxLv = D > 128 ? 512 : kMaxLevels;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = 2 * kQBytes;
    static constexpr int kBarOff = kKVOff + kEntries * kEntryBytes;
    // barrier indices
    static constexpr int bQFull = 0, bQEmpty = 2, bEFull = 4, bEEmpty = 4 + kEntries;
    static constexpr int bSFull = 4 + 2 * kEntries, bPFull = bSFull + 2, bOFull = bSFull + 4, bOEmpty = bSFull + 6;
    static constexpr int bStats = bSFull + 8, bDrain = bSFull + 10, bIssued = bSFull + 12;
    static constexpr int bPRest = bSFull + 14;  // P stage 2 (keys 96-127); bPFull is stage 1
    // 8-bit inputs: [kEntries] the entry's 8-bit V tile has landed / has been widened. Only
    // entries that carry V advance them.
    static constexpr int bV8Full = bSFull + 16, bVConv = bV8Full + (F8 ? kEntries : 0);
    // correction role: [quarter] a request is posted in the quarter's slot (bReq); [4 s +
    // quarter] in a step whose O rescale was handed over, the softmax warp's first P stage is
    // written (bPStage), after which the correction warp arrives on bPFull in its place
    static constexpr int bReq = bVConv + (F8 ? kEntries : 0), bPStage = bReq + 4;
    static constexpr int kNumBars = bPStage + 8;
    static constexpr int kStatsOff = kBarOff + ((kNumBars * 8 + 15) / 16) * 16;
    // m[2][128], l[2][128], alpha[2][128], request slots [4]
    static constexpr int kMiscOff = kStatsOff + (3 * 2 * BM + 4) * 4;
    // misc: tmem base, abort flag, packed-order levels, packed work tiles
    // packed-sequence work order (built once per CTA): pre, lvl, perm, nbs
    static constexpr int kPreOff = kMiscOff + 16;
    static constexpr int kLvlOff = kPreOff + ((kMaxB + 1) * 4 + 15) / 16 * 16;
    static constexpr int kPermOff = kLvlOff + ((kMaxLv + 2) * 4 + 15) / 16 * 16;
    static constexpr int kNbOff = kPermOff + kMaxB * 4;
    static constexpr int kBytes = kNbOff + kMaxB * 4;
    static constexpr int kAlloc = kBytes + 1024;                   // slack for 1024-byte alignment
};

struct Tile {
    int h, kvh;
    int q0, k0;   // first token of the sequence in q/o and in k/v
    int Lq, Lk;   // sequence lengths
    int r0;       // first row (within the sequence) of Q tile 0
    int n[2];     // K/V tiles for Q tile 0 and Q tile 1 (0 = tile not computed)
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Wait of a converged warp: every lane polls the same phase (measured faster than one lane
// polling and broadcasting), and the result is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint64_t limit_ns) {
    const bool ok = mbar_wait(bar, parity, abort, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Optional event timeline of CTA 0 for pipeline tuning (compile with -DATTN_TIMELINE).
#ifdef ATTN_TIMELINE
__device__ long long g_timeline[5][4096][4];
__device__ int g_timeline_n[5];
#define ATTN_TL_DECL(x) x
#define ATTN_TL(role, a, b, c, d)                                                         \
    do {                                                                                  \
        if (blockIdx.x == 0 && (threadIdx.x & 31) == 0 && tl_idx < 4096) {                \
            g_timeline[role][tl_idx][0] = (a); g_timeline[role][tl_idx][1] = (b);        \
            g_timeline[role][tl_idx][2] = (c); g_timeline[role][tl_idx][3] = (d);        \
            g_timeline_n[role] = ++tl_idx;                                                \
        }                                                                                 \
    } while (0)
#else
#define ATTN_TL_DECL(x)
#define ATTN_TL(role, a, b, c, d) ((void)0)
#endif

// Packed sequence b: first token and length. Offsets outside [0, Nq] (total packed
// query rows) or [0, Nk] (total key rows), or decreasing, make the sequence empty; the
// work-order build records that as a device error.
__device__ __forceinline__ bool packed_seq(const FwdParams& p, int b, int& first, int& len) {
    const int a = __ldg(p.cu_seqlens + b), e = __ldg(p.cu_seqlens + b + 1);
    const bool ok = a >= 0 && e >= a && e <= p.Nq && e <= p.Nk;
    first = ok ? a : 0;
    len = ok ? e - a : 0;
    return ok;
}

// ------------------------------------------------------------------ 8-bit inputs
// Instruction descriptor of kind::f8f6f4 with fp32 accumulation; fmt 0 = e4m3, 1 = e5m2
// for both A and B ([7,10) A format, [10,13) B format), both K-major.
__host__ __device__ constexpr uint32_t idesc_f8_f32(uint32_t M, uint32_t N, uint32_t fmt) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Instruction descriptor of kind::f16 with f16 A and B (format 0) and fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N, uint32_t b_mn_major) {
    return (1u << 4) | (b_mn_major << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_ss_f8_by(uint32_t issue, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 e, %5, 0;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two 8-bit codes (low byte first) to an f16 pair (low half first); exact for every code.
template <int F8>
__device__ __forceinline__ uint32_t f8x2_to_f16x2(uint32_t two_codes) {
    const uint16_t v = (uint16_t)two_codes;
    uint32_t d;
    if (F8 == 1)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
    else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(d) : "h"(v));
    return d;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Store packed P columns [C0, C1) (two 16-bit probabilities per column) to TMEM at tS.
template <int C0, int C1>
__device__ __forceinline__ void store_p_cols(uint32_t tS, const uint32_t* pk) {
    static_assert((C1 - C0) % 16 == 0, "whole 16-column stores");
    if constexpr (C1 - C0 >= 32) {
        tmem_st32(tS + C0, pk + C0);
        store_p_cols<C0 + 32, C1>(tS, pk);
    } else if constexpr (C1 - C0 >= 16) {
        tmem_st16(tS + C0, pk + C0);
        store_p_cols<C0 + 16, C1>(tS, pk);
    }
}

// Widen row r of the 8-bit V tile at v8 ([BN keys x D bytes], rows of 128 bytes in the TMA's
// 128-byte swizzle: 16-byte unit u of row r at r*128 + ((u ^ (r & 7)) << 4)) into the 16-bit
// V tile at v16, in the layout a TMA load of 16-bit V would have produced: D/64 chunks of
// [BN rows x 128 bytes], unit u of row r of chunk c at c*BN*128 + r*128 + ((u ^ (r & 7)) << 4).
template <int D, int F8>
__device__ __forceinline__ void widen_v_rows(uint32_t v8, uint32_t v16, int r) {
    static_assert(D == 128, "8-bit inputs: one 128-byte row per key");
    {
        const uint32_t sw = (uint32_t)(r & 7);
#pragma unroll 2
        for (int u = 0; u < 8; ++u) {  // 16 codes: d = 16u .. 16u + 15
            uint32_t w[4];
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(v8 + r * 128 + ((u ^ sw) << 4))
                         : "memory");
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                h[2 * i] = f8x2_to_f16x2<F8>(w[i]);
                h[2 * i + 1] = f8x2_to_f16x2<F8>(w[i] >> 16);
            }
            const int c = u >> 2;                 // 64-column chunk
            const uint32_t u0 = (uint32_t)((u & 3) * 2);  // first 16-byte unit of these 16 values
            const uint32_t base = v16 + c * (BN * 128) + r * 128;
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + ((u0 ^ sw) << 4)), "r"(h[0]), "r"(h[1]),
                         "r"(h[2]), "r"(h[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + (((u0 + 1) ^ sw) << 4)), "r"(h[4]),
                         "r"(h[5]), "r"(h[6]), "r"(h[7])
                         : "memory");
        }
    }
}

// Work order of packed sequences, built once per CTA in shared memory by build_packed_order.
struct PackedOrder {
    const int* pre;   // [B + 1] work tiles before the i-th sequence of perm (sequence-major order)
    const int* lvl;   // lvl[j + 2] = work tiles at block levels above j (level order)
    const int* perm;  // [B] sequences by 256-row block count, most first (stable)
    int levels;       // > 0: level order over this many levels; 0: sequence-major order
};

// Map a work-tile index to its tile (a work tile is two consecutive 128-row Q tiles of one
// (sequence, query head)). The order puts the heaviest tiles first so that the snake walk
// below balances the persistent CTAs (longest-processing-time first; under a causal mask a
// tile's cost grows with its query block index j, whatever the sequence).
//   dense batches: sections of sec_q (batch, head) pairs, then query blocks, then the pairs
//     of the section; sec_q is all pairs unless the problem spans many waves, where smaller
//     sections keep the key/value heads being read together within the L2;
//   packed sequences, causal: block levels j from the highest down, then the sequences that
//     reach level j (longest first), then heads;
//   packed sequences, no mask: sequences longest first, then sections of sec_q query heads,
//     then query blocks, then the heads of the section.
// The query heads of one key/value head are adjacent in all three.
template <int BNT>
__device__ __forceinline__ void get_tile(const FwdParams& p, const PackedOrder& po, int w, Tile& t) {
    int b, Lq, Lk, q0, k0, j, h;
    if (p.cu_seqlens) {
        int i;
        if (po.levels > 0) {
            int lo = 0, hi = po.levels - 1;  // smallest level j with lvl[j + 2] <= w
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (po.lvl[mid + 2] <= w) hi = mid; else lo = mid + 1;
            }
            j = lo;
            const int k = w - po.lvl[j + 2];
            i = k / p.Hq;
            h = k - i * p.Hq;
        } else {
            int lo = 0, hi = p.B;  // pre[i] <= w < pre[i + 1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (po.pre[mid] <= w) lo = mid; else hi = mid;
            }
            i = lo;
            j = -1;
        }
        b = po.perm[i];
        int first, len;
        packed_seq(p, b, first, len);
        q0 = k0 = first;
        Lq = Lk = len;
        if (j < 0) {
            const int u = w - po.pre[i];
            const int nblk = cdiv(Lq, 2 * BM);
            const int sec = p.sec_q;
            const int per_sec = nblk * sec;
            const int si = u / per_sec;
            const int rem = u - si * per_sec;
            const int jj = rem / sec;
            h = si * sec + (rem - jj * sec);
            j = p.causal ? (nblk - 1 - jj) : jj;
        }
    } else {
        Lq = p.Nq;
        Lk = p.Nk;
        const int nblk = cdiv(Lq, 2 * BM);
        const int pairs = p.B * p.Hq;
        const int sec = p.sec_q;
        const int si = w / (sec * nblk);
        const int rem = w - si * (sec * nblk);
        const int len = min(sec, pairs - si * sec);  // the last section may be shorter
        const int jj = rem / len;
        const int pair = si * sec + (rem - jj * len);
        b = pair / p.Hq;
        h = pair - b * p.Hq;
        q0 = b * p.Nq;
        k0 = b * p.Nk;
        j = p.causal ? (nblk - 1 - jj) : jj;
    }
    t.h = h;
    t.kvh = t.h / p.G;
    t.q0 = q0;
    t.k0 = k0;
    t.Lq = Lq;
    t.Lk = Lk;
    t.r0 = j * 2 * BM;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int r = t.r0 + s * BM;
        int n = 0;
        if (r < Lq && Lk > 0) {
            if (p.causal) {
                const int rl = min(r + BM - 1, Lq - 1);
                const int kmax = min(Lk, rl + (Lk - Lq) + 1);
                n = kmax > 0 ? cdiv(kmax, BNT) : 0;
            } else {
                n = cdiv(Lk, BNT);
            }
        }
        t.n[s] = n;
    }
}

// Build the packed-sequence work order (one warp). Blocks per sequence nb = ceil(len / 256);
// a counting sort by nb, stable so that every CTA derives the same order, gives perm.
// Level order (causal, nb <= max_levels): with c_j = #{sequences with nb > j}, level j holds
// Hq * c_j tiles, and lvl[j + 2] = Hq * sum over levels above j of c. Returns the number of
// levels (0 selects the sequence-major order) and the number of work tiles.
__device__ void build_packed_order(const FwdParams& p, int* pre, int* lvl, int* perm, int* nbs, int lane,
                                   int max_levels, int& levels, int& total) {
    const int B = p.B;
    int maxnb = 0;
    for (int base = 0; base < B; base += 32) {
        const int b = base + lane;
        if (b < B) {
            int first, len;
            if (!packed_seq(p, b, first, len) && p.status && blockIdx.x == 0) atomicCAS(p.status, 0, kDevBadIndex);
            nbs[b] = len > 0 ? cdiv(len, 2 * BM) : 0;
            maxnb = max(maxnb, nbs[b]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) maxnb = max(maxnb, __shfl_xor_sync(0xffffffffu, maxnb, o));
    const bool sorted = maxnb <= max_levels && !p.packed_plain;
    if (sorted) {
        for (int v = lane; v <= maxnb + 1; v += 32) lvl[v] = 0;
        __syncwarp();
        for (int b = lane; b < B; b += 32) atomicAdd(&lvl[nbs[b]], 1);
        __syncwarp();
        // lvl[v] = #{nb > v}: exclusive suffix sums of the histogram, 32 values per pass from the top
        int carry = 0;
        for (int top = maxnb + 1; top >= 0; top -= 32) {
            const int v = top - lane;
            const int x = v >= 0 ? lvl[v] : 0;
            int incl = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (v >= 0) lvl[v] = carry + incl - x;
            carry += __shfl_sync(0xffffffffu, incl, 31);
            __syncwarp();
        }
        // stable scatter; afterwards lvl[v] = #{nb >= v}
        for (int base = 0; base < B; base += 32) {
            const int b = base + lane;
            const int v = b < B ? nbs[b] : -1;
            const unsigned same = __match_any_sync(0xffffffffu, v);
            const int rank = __popc(same & ((1u << lane) - 1u));
            if (b < B) perm[lvl[v] + rank] = b;
            __syncwarp();
            if (b < B && rank == 0) lvl[v] += __popc(same);
            __syncwarp();
        }
        // inclusive suffix sums times Hq: lvl[v] = Hq * sum_{u >= v} #{nb >= u}
        carry = 0;
        for (int top = maxnb + 1; top >= 0; top -= 32) {
            const int v = top - lane;
            const int x = v >= 0 ? lvl[v] : 0;
            int incl = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (v >= 0) lvl[v] = p.Hq * (carry + incl);
            carry += __shfl_sync(0xffffffffu, incl, 31);
            __syncwarp();
        }
    } else {
        for (int b = lane; b < B; b += 32) perm[b] = b;
        __syncwarp();
    }
    // sequence-major prefix over perm
    int carry = 0;
    for (int base = 0; base < B; base += 32) {
        const int i = base + lane;
        const int cnt = i < B ? p.Hq * nbs[perm[i]] : 0;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (i < B) pre[i] = carry + incl - cnt;
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pre[B] = carry;
    __syncwarp();
    levels = (sorted && p.causal) ? maxnb : 0;
    total = carry;
}

// The r-th work tile of this CTA: rounds of gridDim.x consecutive tiles, walked in
// alternating direction (a snake), so that a CTA given one of the heaviest tiles of a round
// is given one of the lightest of the next.
__device__ __forceinline__ int snake_index(int r) {
    const int c = (r & 1) ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    return r * (int)gridDim.x + c;
}

// Software 2^x on the FMA/ALU pipes ("FlashAttention-4: Blackwell algorithm-pipeline
// co-design", section "hybrid exponential"; "FlashAttention4 精读" section 3.1.3):
// clamp at -127; n = floor(x) from the round-down add of the magic bias 1.5 * 2^23,
// whose low mantissa bits then hold n; 2^f by the Horner cubic with the printed
// coefficients; 2^n applied by adding n to the exponent field (the bias bits of the
// magic constant vanish when shifted left by 23).
__device__ __forceinline__ float ex2_poly(float x) {
    x = fmaxf(x, -127.0f);
    const float t = __fadd_rd(x, 12582912.0f);
    const float f = __fsub_rn(x, __fsub_rn(t, 12582912.0f));
    float q = __fmaf_rn(0.0771f, f, 0.2276f);
    q = __fmaf_rn(q, f, 0.6951f);
    q = __fmaf_rn(q, f, 1.0f);
    return __uint_as_float(__float_as_uint(q) + (__float_as_uint(t) << 23));
}

template <int D, int POLY_EVERY, int F8, int DV, int BNT, int UKV, int CORR>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using L = Layout<D, F8, DV, BNT>;
    constexpr int BN = BNT;  // keys per K/V tile (shadows the default)
    static_assert(BN % 32 == 0 && BN <= 128 && DV <= 128 && DV % 64 == 0 && D % 64 == 0, "tile shape");
    static_assert(L::kAlloc <= 232448, "shared memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    float* st_m = reinterpret_cast<float*>(smem + L::kStatsOff);  // [2][128]
    float* st_l = st_m + 2 * BM;                                    // [2][128]
    float* st_a = st_l + 2 * BM;                                    // [2][128] rescale factors handed over
    int* st_req = reinterpret_cast<int*>(st_a + 2 * BM);            // [4] request slot per lane quarter
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    ATTN_TL_DECL(int tl_idx = 0);

    if (threadIdx.x == 0) {
        mbar_init(&bars[L::bQFull + 0], 1);
        mbar_init(&bars[L::bQFull + 1], 1);
        mbar_init(&bars[L::bQEmpty + 0], 1);
        mbar_init(&bars[L::bQEmpty + 1], 1);
        for (int i = 0; i < L::kEntries; ++i) {
            mbar_init(&bars[L::bEFull + i], 1);
            mbar_init(&bars[L::bEEmpty + i], 2);  // released by both MMA warps
            if (F8) {
                mbar_init(&bars[L::bV8Full + i], 1);
                mbar_init(&bars[L::bVConv + i], 4);  // the four widening (epilogue) warps
            }
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[L::bSFull + s], 1);
            mbar_init(&bars[L::bPFull + s], 4);
            mbar_init(&bars[L::bPRest + s], 4);
            mbar_init(&bars[L::bOFull + s], 1);
            mbar_init(&bars[L::bOEmpty + s], 4);
            mbar_init(&bars[L::bStats + s], 4);
            for (int q = 0; q < 4; ++q) mbar_init(&bars[L::bPStage + 4 * s + q], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[L::bDrain + s], 1);
            mbar_init(&bars[L::bIssued + s], 1);
        }
        for (int q = 0; q < 4; ++q) {
            mbar_init(&bars[L::bReq + q], 1);
            st_req[q] = 0;
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    // Work order over packed sequences (warp 2).
    int* misc = reinterpret_cast<int*>(smem + L::kMiscOff);
    int* pre = reinterpret_cast<int*>(smem + L::kPreOff);
    int* lvl = reinterpret_cast<int*>(smem + L::kLvlOff);
    int* perm = reinterpret_cast<int*>(smem + L::kPermOff);
    if (p.cu_seqlens && warp == 2) {
        int levels, tiles;
        build_packed_order(p, pre, lvl, perm, reinterpret_cast<int*>(smem + L::kNbOff), lane, L::kMaxLv, levels, tiles);
        if (lane == 0) {
            misc[2] = levels;
            misc[3] = tiles;
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int total = p.total_tiles;
    const PackedOrder po{pre, lvl, perm, p.cu_seqlens ? misc[2] : 0};
    if (p.cu_seqlens) total = misc[3];
    const uint32_t tmem = *tmem_slot;
    const uint64_t wd = p.watchdog_ns;

    // Register split per warpgroup (producer/MMA, softmax, softmax, correction/epilogue): 72,
    // 184, 184, 72; 80, 176, 176, 72 for 192-wide rows (the MMA warps need more, the softmax of
    // 96-key tiles less); 80, 184, 184, 64 for the unroll-KV schedule. Each sums to at most
    // 512 = 4 x 128, the registers the CTA is launched with.
    constexpr int kRegLow = (D > 128 || UKV) ? 80 : 72;
    constexpr int kRegSoftmax = D > 128 ? 176 : 184;
    constexpr int kRegEpi = (UKV && D <= 128) ? 64 : 72;
    static_assert(kRegLow + 2 * kRegSoftmax + kRegEpi <= 512, "register split");
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegLow));
    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        // The whole warp walks the schedule so that addresses and coordinates stay
        // warp-uniform; lane 0 issues the copies.
        const uint32_t leader = lane == 0;
        uint32_t stage = 0, phase = 0, qphase[2] = {0, 0};
        int issued = 0;
        bool ok = true;
        for (int r = 0; r * (int)gridDim.x < total && ok; ++r) {
            const int w = snake_index(r);
            if (w >= total) continue;
            Tile t;
            get_tile<BN>(p, po, w, t);
            const int nmax = max(t.n[0], t.n[1]);
            if (nmax == 0) continue;  // no visible key in the block: the other roles skip it too
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                if (!ok || t.n[s] == 0) continue;
                ATTN_TL_DECL(long long tq = clock64());
                if (!(ok = warp_wait(&bars[L::bQEmpty + s], qphase[s] ^ 1u, abort_flag, wd))) continue;
                qphase[s] ^= 1u;
                uint8_t* dst = smem + L::kQOff + s * L::kQBytes;
                mbar_arrive_expect_tx_by(leader, &bars[L::bQFull + s], L::kQBytes);
#pragma unroll
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_3d_by(leader, dst + c * L::kChunkBytesQ, &tmQ, &bars[L::bQFull + s],
                                   c * (128 / L::kElem), t.h, t.q0 + t.r0 + s * BM);
                ATTN_TL(0, 10 + s, w, tq, clock64());
            }
            for (int e = 0; e <= nmax && ok; ++e) {
                ATTN_TL_DECL(long long tw = clock64());
                if (!(ok = warp_wait(&bars[L::bEEmpty + stage], phase ^ 1u, abort_flag, wd))) break;
                uint8_t* ent = smem + L::kKVOff + stage * L::kEntryBytes;
                const uint32_t bytes = (e < nmax ? (uint32_t)L::kKBytes : 0u) + (!F8 && e >= 1 ? (uint32_t)L::kVBytes : 0u);
                mbar_arrive_expect_tx_by(leader, &bars[L::bEFull + stage], bytes);
                if (e < nmax) {
#pragma unroll
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_3d_by(leader, ent + c * L::kChunkBytesKV, &tmK, &bars[L::bEFull + stage],
                                       c * (128 / L::kElem), t.kvh, t.k0 + e * BN);
                }
                if (e >= 1) {  // 16-bit V tile, or the 8-bit tile it is widened from (own barrier)
                    constexpr int kBoxes = F8 ? L::kChunks : L::kVChunks;
                    uint64_t* vbar = &bars[(F8 ? L::bV8Full : L::bEFull) + stage];
                    if (F8) mbar_arrive_expect_tx_by(leader, vbar, L::kV8Bytes);
#pragma unroll
                    for (int c = 0; c < kBoxes; ++c)
                        tma_load_3d_by(leader, ent + (F8 ? L::kV8Off : L::kVOff) + c * L::kChunkBytesKV, &tmV, vbar,
                                       c * (128 / L::kElem), t.kvh, t.k0 + (e - 1) * BN);
                }
                ATTN_TL(0, 0, e, tw, clock64());
                ++issued;
                if (++stage == (uint32_t)L::kEntries) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok) {
            // Let copies already in flight land before the CTA can exit.
            uint32_t st = stage, ph = phase;
            for (int i = 0; i < L::kEntries && i < issued; ++i) {
                if (st == 0) { st = L::kEntries; ph ^= 1u; }
                --st;
                int dummy = 0;
                mbar_wait(&bars[L::bEFull + st], ph, &dummy, 20000000ull);
            }
            for (int s = 0; s < 2; ++s) {
                int dummy = 0;
                mbar_wait(&bars[L::bQFull + s], qphase[s] ^ 1u, &dummy, 20000000ull);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------------ MMA issuers
        // Warp 1 issues Q tile 0's products, warp 2 Q tile 1's. Per KV step n the tensor pipe
        // receives
        //   burst 0 (warp 1): PV0(n-1), S0(n)     burst 1 (warp 2): PV1(n-1), S1(n)
        // so it computes one tile's products while the other tile's softmax works; S_s(n) is
        // issued after PV_s(n-1) by the same thread, so its completion covers PV_s(n-1).
        // A token pair keeps the bursts in that alternating order: each warp passes the token
        // as soon as its MMAs are issued, before its completion signals, so the other warp's
        // waits and descriptor set-up overlap the commits. Both warps walk the same schedule;
        // ring entry n is released once both have committed their reads of it (count 2).
        // Within a warp, lane 0 issues every tcgen05 instruction while the whole warp keeps the
        // descriptors and slots warp-uniform.
        // unroll-KV at work-tile boundaries ("Low-precision FA4", section 2.1.2; UKV = 1): the
        // last burst of a work tile holds only PV(last), and the first of the next only S(0),
        // so the tensor pipe would idle while the other tile's softmax finishes. With UKV the
        // two are one burst: PV_s(last) of this tile, then S_s(0) = Q'_s K'_0^T of the next
        // (from the next ring entry; it overwrites P_s(last) only after the PV has read it).
        const int s = warp - 1;
        const uint32_t leader = lane == 0;
        constexpr uint32_t idS = F8 ? idesc_f8_f32(BM, BN, F8 - 1) : idesc_bf16_f32(BM, BN, 0);
        constexpr uint32_t idO = F8 ? idesc_f16_f32(BM, DV, 1) : idesc_bf16_f32(BM, DV, 1);
        constexpr int kPA = (3 * BN / 4) / 16;  // P stage 1: k-steps (16 keys each) 0 .. kPA-1
        const uint32_t colS = s ? kColS1 : kColS0;
        const uint32_t colO = s ? kColO1 : kColO0;
        uint32_t stage = 0, phase = 0;
        uint32_t qf = 0, pf = 0, oe = 0, burst = 0;
        uint32_t vcv = 0;  // 8-bit inputs: phase bit per ring slot of the V-widened barrier
        const uint32_t q_base = smem_u32(smem + L::kQOff) + s * L::kQBytes;
        const uint32_t kv_base = smem_u32(smem + L::kKVOff);
        const uint64_t dq = smem_desc_sw128(q_base, 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(kv_base, 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(kv_base, L::kChunkBytesKV, 1024);
        bool ok = true, any = false;
        if constexpr (UKV) {
            // The next work tile (from round r on) with at least one key tile; advances r past it.
            auto next_tile = [&](int& r, Tile& t) -> bool {
                for (; r * (int)gridDim.x < total; ++r) {
                    const int w = snake_index(r);
                    if (w >= total) continue;
                    get_tile<BN>(p, po, w, t);
                    if (max(t.n[0], t.n[1]) > 0) {
                        ++r;
                        return true;
                    }
                }
                return false;
            };
            // S = Q K^T of this warp's Q tile with the K tile in ring slot `slot`
            auto issue_s = [&](uint32_t slot) {
                // K steps of 32 bytes (16 bf16 or 32 8-bit elements), 4 per 128-byte chunk
                const uint64_t kd = dk0 + (uint64_t)((slot * L::kEntryBytes) >> 4);
    #pragma unroll
                for (int k = 0; k < D * L::kElem / 32; ++k) {
                    const uint64_t oq = (uint64_t)(((k >> 2) * L::kChunkBytesQ + (k & 3) * 32) >> 4);
                    const uint64_t ok_ = (uint64_t)(((k >> 2) * L::kChunkBytesKV + (k & 3) * 32) >> 4);
                    if (F8)
                        tc_mma_ss_f8_by(leader, tmem + colS, dq + oq, kd + ok_, idS, k > 0 ? 1u : 0u);
                    else
                        tc_mma_ss_by(leader, tmem + colS, dq + oq, kd + ok_, idS, k > 0 ? 1u : 0u);
                }
            };
            int r = 0;
            Tile t;
            bool have = next_tile(r, t);
            int n_first = 0;  // 1 when the previous burst already issued this tile's S(0)
            while (have && ok) {
                const int nmax = max(t.n[0], t.n[1]);
                const int ns = s ? t.n[1] : t.n[0];
                if (n_first == 0 && ns > 0) {
                    if (!(ok = warp_wait(&bars[L::bQFull + s], qf, abort_flag, wd))) break;
                    qf ^= 1u;
                    any = true;
                }
                Tile nt;
                int r_next = r;
                bool merged = false;
                for (int n = n_first; n <= nmax && ok; ++n) {
                    const bool do_pv = n >= 1 && n - 1 < ns, do_s = n < ns;
                    const uint32_t e_slot = stage, e_par = phase;
                    if (++stage == (uint32_t)L::kEntries) { stage = 0; phase ^= 1u; }
                    ATTN_TL_DECL(long long tp = clock64());
                    if (!(ok = warp_wait(&bars[L::bEFull + e_slot], e_par, abort_flag, wd))) break;
                    if (do_pv) {
                        if (!(ok = warp_wait(&bars[L::bPFull + s], pf, abort_flag, wd))) break;
                        if (n - 1 == 0) {
                            if (!(ok = warp_wait(&bars[L::bOEmpty + s], oe ^ 1u, abort_flag, wd))) break;
                            oe ^= 1u;
                        }
                    }
                    if (F8 && n >= 1) {  // every entry that carries V: wait until it has been widened
                        if (!(ok = warp_wait(&bars[L::bVConv + e_slot], (vcv >> e_slot) & 1u, abort_flag, wd))) break;
                        vcv ^= 1u << e_slot;
                    }
                    // unroll-KV: the next work tile's first entry and Q tile join the last burst
                    bool mg = false;
                    int nns = 0;
                    uint32_t m_slot = 0;
                    if (n == nmax && next_tile(r_next, nt)) {
                        mg = true;
                        nns = s ? nt.n[1] : nt.n[0];
                        m_slot = stage;
                        const uint32_t m_par = phase;
                        if (++stage == (uint32_t)L::kEntries) { stage = 0; phase ^= 1u; }
                        if (!(ok = warp_wait(&bars[L::bEFull + m_slot], m_par, abort_flag, wd))) break;
                        if (nns > 0) {
                            if (!(ok = warp_wait(&bars[L::bQFull + s], qf, abort_flag, wd))) break;
                            qf ^= 1u;
                            any = true;
                        }
                    }
                    // token: burst 0 of step n follows burst 1 of step n-1; burst 1 follows burst 0
                    if (s == 0) {
                        if (burst > 0 && !(ok = warp_wait(&bars[L::bIssued + 1], (burst - 1) & 1u, abort_flag, wd))) break;
                    } else {
                        if (!(ok = warp_wait(&bars[L::bIssued + 0], burst & 1u, abort_flag, wd))) break;
                    }
                    ATTN_TL(s ? 4 : 1, 100 + s, n, tp, clock64());
                    tc_fence_after();
                    const uint32_t ent_off = e_slot * L::kEntryBytes;
                    if (do_pv) {
                        const uint64_t vd = dv0 + (uint64_t)((ent_off + L::kVOff) >> 4);
                        const uint32_t acc0 = n - 1 > 0 ? 1u : 0u;
    #pragma unroll
                        for (int k = 0; k < kPA; ++k)  // P stage 1
                            tc_mma_ts_by(leader, tmem + colO, tmem + colS + k * 8, vd + (uint64_t)(k * (2048 >> 4)), idO,
                                         k == 0 ? acc0 : 1u);
                        if (!(ok = warp_wait(&bars[L::bPRest + s], pf, abort_flag, wd))) break;
                        pf ^= 1u;
                        tc_fence_after();
    #pragma unroll
                        for (int k = kPA; k < BN / 16; ++k)  // P stage 2
                            tc_mma_ts_by(leader, tmem + colO, tmem + colS + k * 8, vd + (uint64_t)(k * (2048 >> 4)), idO, 1u);
                    }
                    if (do_s) issue_s(e_slot);
                    __syncwarp();
                    if (mg) {
                        // this tile's completions first, so that its epilogue starts without waiting
                        // for the next tile's S(0)
                        if (do_pv && n - 1 == ns - 1) tc_commit_by(leader, &bars[L::bOFull + s]);
                        tc_commit_by(leader, &bars[L::bEEmpty + e_slot]);
                        if (nns > 0) issue_s(m_slot);
                        __syncwarp();
                        if (leader) mbar_arrive(&bars[L::bIssued + s]);
                        if (nns > 0) tc_commit_by(leader, &bars[L::bSFull + s]);
                        if (nns == 1) tc_commit_by(leader, &bars[L::bQEmpty + s]);
                        tc_commit_by(leader, &bars[L::bEEmpty + m_slot]);
                    } else {
                        if (leader) mbar_arrive(&bars[L::bIssued + s]);
                        if (do_s) tc_commit_by(leader, &bars[L::bSFull + s]);
                        if (do_pv && n - 1 == ns - 1) tc_commit_by(leader, &bars[L::bOFull + s]);
                        if (do_s && n == ns - 1) tc_commit_by(leader, &bars[L::bQEmpty + s]);
                        tc_commit_by(leader, &bars[L::bEEmpty + e_slot]);
                    }
                    ATTN_TL(s ? 4 : 1, 200 + s, n, clock64(), 0);
                    ++burst;
                    merged = mg;
                }
                if (!ok) break;
                if (merged) {
                    t = nt;
                    r = r_next;
                    n_first = 1;
                } else {
                    have = next_tile(r, t);
                    n_first = 0;
                }
            }
        } else {
            for (int r = 0; r * (int)gridDim.x < total && ok; ++r) {
                const int w = snake_index(r);
                if (w >= total) continue;
                Tile t;
                get_tile<BN>(p, po, w, t);
                const int nmax = max(t.n[0], t.n[1]);
                const int ns = s ? t.n[1] : t.n[0];
                if (nmax == 0) continue;
                if (ns > 0) {
                    if (!(ok = warp_wait(&bars[L::bQFull + s], qf, abort_flag, wd))) break;
                    qf ^= 1u;
                    any = true;
                }
                for (int n = 0; n <= nmax && ok; ++n) {
                    const bool do_pv = n >= 1 && n - 1 < ns, do_s = n < ns;
                    const uint32_t e_slot = stage, e_par = phase;
                    if (++stage == (uint32_t)L::kEntries) { stage = 0; phase ^= 1u; }
                    ATTN_TL_DECL(long long tp = clock64());
                    if (!(ok = warp_wait(&bars[L::bEFull + e_slot], e_par, abort_flag, wd))) break;
                    if (do_pv) {
                        if (!(ok = warp_wait(&bars[L::bPFull + s], pf, abort_flag, wd))) break;
                        if (n - 1 == 0) {
                            if (!(ok = warp_wait(&bars[L::bOEmpty + s], oe ^ 1u, abort_flag, wd))) break;
                            oe ^= 1u;
                        }
                    }
                    if (F8 && n >= 1) {  // every entry that carries V: wait until it has been widened
                        if (!(ok = warp_wait(&bars[L::bVConv + e_slot], (vcv >> e_slot) & 1u, abort_flag, wd))) break;
                        vcv ^= 1u << e_slot;
                    }
                    // token: burst 0 of step n follows burst 1 of step n-1; burst 1 follows burst 0
                    if (s == 0) {
                        if (burst > 0 && !(ok = warp_wait(&bars[L::bIssued + 1], (burst - 1) & 1u, abort_flag, wd))) break;
                    } else {
                        if (!(ok = warp_wait(&bars[L::bIssued + 0], burst & 1u, abort_flag, wd))) break;
                    }
                    ATTN_TL(s ? 4 : 1, 100 + s, n, tp, clock64());
                    tc_fence_after();
                    const uint32_t ent_off = e_slot * L::kEntryBytes;
                    if (do_pv) {
                        const uint64_t vd = dv0 + (uint64_t)((ent_off + L::kVOff) >> 4);
                        const uint32_t acc0 = n - 1 > 0 ? 1u : 0u;
    #pragma unroll
                        for (int k = 0; k < kPA; ++k)  // P stage 1
                            tc_mma_ts_by(leader, tmem + colO, tmem + colS + k * 8, vd + (uint64_t)(k * (2048 >> 4)), idO,
                                         k == 0 ? acc0 : 1u);
                        if (!(ok = warp_wait(&bars[L::bPRest + s], pf, abort_flag, wd))) break;
                        pf ^= 1u;
                        tc_fence_after();
    #pragma unroll
                        for (int k = kPA; k < BN / 16; ++k)  // P stage 2
                            tc_mma_ts_by(leader, tmem + colO, tmem + colS + k * 8, vd + (uint64_t)(k * (2048 >> 4)), idO, 1u);
                    }
                    if (do_s) {
                        // K steps of 32 bytes (16 bf16 or 32 8-bit elements), 4 per 128-byte chunk
                        const uint64_t kd = dk0 + (uint64_t)(ent_off >> 4);
    #pragma unroll
                        for (int k = 0; k < D * L::kElem / 32; ++k) {
                            const uint64_t oq = (uint64_t)(((k >> 2) * L::kChunkBytesQ + (k & 3) * 32) >> 4);
                            const uint64_t ok_ = (uint64_t)(((k >> 2) * L::kChunkBytesKV + (k & 3) * 32) >> 4);
                            if (F8)
                                tc_mma_ss_f8_by(leader, tmem + colS, dq + oq, kd + ok_, idS, k > 0 ? 1u : 0u);
                            else
                                tc_mma_ss_by(leader, tmem + colS, dq + oq, kd + ok_, idS, k > 0 ? 1u : 0u);
                        }
                    }
                    __syncwarp();
                    if (leader) mbar_arrive(&bars[L::bIssued + s]);
                    if (do_s) tc_commit_by(leader, &bars[L::bSFull + s]);
                    if (do_pv && n - 1 == ns - 1) tc_commit_by(leader, &bars[L::bOFull + s]);
                    if (do_s && n == ns - 1) tc_commit_by(leader, &bars[L::bQEmpty + s]);
                    tc_commit_by(leader, &bars[L::bEEmpty + e_slot]);
                    ATTN_TL(s ? 4 : 1, 200 + s, n, clock64(), 0);
                    ++burst;
                }
            }
        }
        if (any) {
            // Wait until every MMA this warp issued has completed before TMEM can be released.
            tc_commit_by(leader, &bars[L::bDrain + s]);
            int dummy = 0;
            if (leader) mbar_wait(&bars[L::bDrain + s], 0, &dummy, 50000000ull);
            __syncwarp();
        }
    }
    } else if (warp < 12) {
        // ------------------------------------------------------------------ softmax
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegSoftmax));
        const int s = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + (s ? kColS1 : kColS0);
        const uint32_t tO = tmem + lane_off + (s ? kColO1 : kColO0);
        const float sl2 = p.scale_log2;
        uint32_t sf = 0, oe = 0;
        uint32_t c_dec = 0, c_res = 0, c_first = 0, c_ores = 0;  // per warp: far below 2^32
        bool ok = true;
        for (int r = 0; r * (int)gridDim.x < total && ok; ++r) {
            const int w = snake_index(r);
            if (w >= total) continue;
            Tile t;
            get_tile<BN>(p, po, w, t);
            const int ns = s ? t.n[1] : t.n[0];
            if (ns == 0) continue;
            const int tile_row0 = t.r0 + s * BM;
            const int qrow = tile_row0 + row;
            const int off = t.Lk - t.Lq;
            float m = -INFINITY, l = 0.0f;
            ++c_first;
            for (int n = 0; n < ns; ++n) {
                ATTN_TL_DECL(long long ts0 = clock64());
                if (!warp_wait(&bars[L::bSFull + s], sf, abort_flag, wd)) { ok = false; break; }
                sf ^= 1u;
                tc_fence_after();
                ATTN_TL_DECL(long long ts1 = clock64());
                uint32_t r[BN / 32][32];
#pragma unroll
                for (int i = 0; i < BN / 32; ++i) tmem_ld32(tS + 32 * i, r[i]);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < BN / 32; ++i) reg_fence(r[i]);
                float sv[BN];
#pragma unroll
                for (int c = 0; c < BN; ++c) sv[c] = __uint_as_float(r[c >> 5][c & 31]);
                const int kb = n * BN;
                const bool need_mask = (kb + BN > t.Lk) || (p.causal && kb + BN - 1 > tile_row0 + off);
                if (need_mask) {
                    const int lim = (p.causal ? min(t.Lk, qrow + off + 1) : t.Lk) - kb;
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c >= lim) sv[c] = -INFINITY;
                }
                // row maximum: eight chains of three-input maxima
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = fmaxf(sv[i], sv[i + 8]);
#pragma unroll
                for (int c = 16; c < BN; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = max3f(mx[i], sv[c + i], sv[c + 8 + i]);
                const float mt = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                const float m_cand = fmaxf(m, mt);
                const bool need = (m_cand - m) * sl2 > p.rescale_thr;  // NaN (both -inf) is false
                const bool warp_need = __any_sync(0xffffffffu, need);
                bool handed = false;  // O's rescale for this step handed to the correction warp
                if (warp_need) {
                    const float alpha = (m == -INFINITY) ? 0.0f : ex2_mufu((m - m_cand) * sl2);
                    if (n > 0) {
                        ++c_ores;
                        if constexpr (CORR != 0) {
                            // hand the rescale to the correction warp of this quarter, which
                            // works while the exponentials below are computed (rows that keep
                            // their maximum have alpha = 1); if the quarter's request slot is
                            // taken, rescale here
                            st_a[s * BM + row] = alpha;
                            __syncwarp();
                            int posted = 0;
                            if (lane == 0 && atomicCAS(&st_req[quarter], 0, kReqRescale + s) == 0) {
                                mbar_arrive(&bars[L::bReq + quarter]);
                                posted = 1;
                            }
                            handed = __shfl_sync(0xffffffffu, posted, 0) != 0;
                        }
                        if (!handed) {
#pragma unroll 1
                            for (int c = 0; c < DV; c += 16) {
                                uint32_t o[16];
                                tmem_ld16(tO + c, o);
                                tc_wait_ld();
                                reg_fence(o);
#pragma unroll
                                for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                                tmem_st16(tO + c, o);
                            }
                        }
                    }
                    l *= alpha;
                    m = m_cand;
                    ++c_res;
                }
                ++c_dec;
                const float neg = (m == -INFINITY) ? 0.0f : -m * sl2;
                // exponent arguments two at a time (packed FMA), exponentials, packed row sums;
                // P goes out in two stages (keys 0-95, then 96-127)
                float sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                uint32_t pk[BN / 2];
                constexpr int kSA = (3 * BN / 4) / 16 * 16;  // keys in P stage 1 (whole MMA k-steps)
                auto exp_pair = [&](int c) {
                    float x0, x1;
                    ffma2(x0, x1, sv[c], sv[c + 1], sl2, sl2, neg, neg);
                    float p0, p1;
                    if (POLY_EVERY > 0 && (c % (POLY_EVERY > 0 ? POLY_EVERY : 1)) == POLY_EVERY - 2) {
                        p0 = ex2_mufu(x0);
                        p1 = ex2_poly(x1);
                    } else {
                        p0 = ex2_mufu(x0);
                        p1 = ex2_mufu(x1);
                    }
                    const int a = ((c >> 1) & 3) * 2;
                    fadd2(sum[a], sum[a + 1], sum[a], sum[a + 1], p0, p1);
                    pk[c >> 1] = F8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
                };
#pragma unroll
                for (int c = 0; c < kSA; c += 2) exp_pair(c);
                store_p_cols<0, kSA / 2>(tS, pk);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                // P stage 1 is written; in a handed-over step the correction warp passes this on
                // to the MMA warp once O_s is rescaled
                if (lane == 0) mbar_arrive(handed ? &bars[L::bPStage + 4 * s + quarter] : &bars[L::bPFull + s]);
#pragma unroll
                for (int c = kSA; c < BN; c += 2) exp_pair(c);
                store_p_cols<kSA / 2, BN / 2>(tS, pk);
                l += ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[L::bPRest + s]);
                if (quarter == 0) ATTN_TL(2 + s, n, ts0, ts1, clock64());
            }
            if (!ok) break;
            // Publish (m, l) once the epilogue has drained the previous tile of this stage.
            if (!warp_wait(&bars[L::bOEmpty + s], oe ^ 1u, abort_flag, wd)) { ok = false; break; }
            oe ^= 1u;
            st_m[s * BM + row] = m;
            st_l[s * BM + row] = l;
            __syncwarp();
            if constexpr (CORR != 0) {
                // the finished tile is a request too: wait (bounded) until the quarter's slot is
                // free; the correction warp frees it as soon as it has read the one there
                int posted = 1;
                if (lane == 0) {
                    const uint64_t t0 = global_timer_ns();
                    while (atomicCAS(&st_req[quarter], 0, kReqEpilogue + s) != 0) {
                        if (*abort_flag || global_timer_ns() - t0 > wd) {
                            *abort_flag = 1;
                            posted = 0;
                            break;
                        }
                    }
                    if (posted) mbar_arrive(&bars[L::bReq + quarter]);
                }
                if (!__shfl_sync(0xffffffffu, posted, 0)) { ok = false; break; }
            } else {
                if (lane == 0) mbar_arrive(&bars[L::bStats + s]);
            }
        }
        if (p.counters && lane == 0) {
            atomicAdd(p.counters + 0, (unsigned long long)c_dec);
            atomicAdd(p.counters + 1, (unsigned long long)c_res);
            const unsigned long long ex = c_dec * 32ull * BN;
            const unsigned long long poly = POLY_EVERY > 0 ? ex / POLY_EVERY : 0ull;
            atomicAdd(p.counters + 2, poly);
            atomicAdd(p.counters + 3, ex - poly);
            atomicAdd(p.counters + 4, (unsigned long long)(c_dec - c_first));
            atomicAdd(p.counters + 5, (unsigned long long)c_ores);
        }
    } else {
        // ------------------------------------------------------------------ correction + epilogue
        // Warp 12 + q serves TMEM lane quarter q of both Q tiles: it writes O / l and the LSE
        // of finished rows and, with 8-bit inputs, widens V tiles. With CORR it is also the
        // correction warp ("FlashAttention4 精读" section 3.1, correction warpgroup;
        // "FlashAttention-4: Blackwell algorithm-pipeline co-design", conditional softmax
        // rescaling) and is driven by requests: the softmax warps of its quarter post, in the
        // quarter's slot, either "tile s is finished" (once per Q tile) or, in the rare step
        // where they raise their rows' maxima by more than the threshold, "rescale O_s". For
        // the latter the softmax warp publishes its factors and goes on with its exponentials,
        // and this warp rescales the quarter's rows of O_s in TMEM meanwhile, then passes the
        // softmax warp's "P stage 1 written" (bPStage) on to the MMA warp (bPFull), so the next
        // O += P V starts on the rescaled accumulator. The warp sleeps on one barrier (bReq)
        // and is woken only by requests; the MMA warp never waits for it otherwise.
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegEpi));
        if constexpr (CORR != 0) {
            static_assert(F8 == 0, "the correction role is built for 16-bit inputs");
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            volatile int* slot = st_req + quarter;
            uint32_t rq = 0, pst = 0;  // pst bit s: next phase parity of bPStage of tile s
            uint32_t of0 = 0, of1 = 0;  // per Q tile: next phase parity of bOFull
            int cur0 = 0, cur1 = 0;     // per Q tile: next round of the schedule to write out
            bool ok = true;
            // Write O / l and the LSE of Q tile s of the next work tile that has keys for it;
            // rows of work tiles without keys for it on the way get O = 0, LSE = -inf. With
            // `finish`, only those rows are written, up to the end of the schedule.
            auto write_out = [&](const int s, int& cur, uint32_t& of, bool finish) -> bool {
                for (; cur * (int)gridDim.x < total; ++cur) {
                    const int w = snake_index(cur);
                    if (w >= total) continue;
                    Tile t;
                    get_tile<BN>(p, po, w, t);
                    const int qrow = t.r0 + s * BM + row;
                    if (t.r0 + s * BM >= t.Lq) continue;
                    const bool valid = qrow < t.Lq;
                    const long long tok = (long long)t.q0 + qrow;
                    __nv_bfloat16* orow = p.o + (tok * p.Hq + t.h) * DV;
                    if (t.n[s] == 0) {
                        if (valid) {
                            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                            for (int c = 0; c < DV / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
                            p.lse[tok * p.Hq + t.h] = -INFINITY;
                        }
                        continue;
                    }
                    if (finish) return false;  // a finished tile nobody reported: a timeout elsewhere
                    ++cur;
                    if (!warp_wait(&bars[L::bOFull + s], of, abort_flag, wd)) return false;
                    of ^= 1u;
                    tc_fence_after();
                    const float m = st_m[s * BM + row];
                    const float l = st_l[s * BM + row];
                    const float inv = l > 0.0f ? p.out_scale / l : 0.0f;
                    const uint32_t tO = tmem + lane_off + (s ? kColO1 : kColO0);
#pragma unroll 1
                    for (int c = 0; c < DV; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tO + c, o);
                        tc_wait_ld();
                        reg_fence(o);
                        if (valid) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[L::bOEmpty + s]);
                    if (valid) p.lse[tok * p.Hq + t.h] = l > 0.0f ? m * p.scale + logf(l) : -INFINITY;
                    return true;
                }
                return finish;
            };
            // tiles this warp will be told about: one per Q tile with keys
            int pending = 0;
            for (int r = 0; r * (int)gridDim.x < total; ++r) {
                const int w = snake_index(r);
                if (w >= total) continue;
                Tile t;
                get_tile<BN>(p, po, w, t);
                pending += (t.n[0] > 0) + (t.n[1] > 0);
            }
            while (pending > 0 && ok) {
                if (!(ok = warp_wait(&bars[L::bReq + quarter], rq, abort_flag, wd))) break;
                rq ^= 1u;
                const int req = *slot;
                __syncwarp();
                if (lane == 0) *slot = 0;  // read: the slot may take the next request
                if (req >= kReqEpilogue) {
                    ok = req == kReqEpilogue ? write_out(0, cur0, of0, false) : write_out(1, cur1, of1, false);
                    --pending;
                } else {
                    // O_s of this quarter's rows times the published factors, then the softmax
                    // warp's first P stage on to the MMA warp
                    const int s = req - kReqRescale;
                    tc_fence_after();
                    const float a = st_a[s * BM + row];
                    const uint32_t tO = tmem + lane_off + (s ? kColO1 : kColO0);
#pragma unroll 1
                    for (int c = 0; c < DV; c += 16) {
                        uint32_t o[16];
                        tmem_ld16(tO + c, o);
                        tc_wait_ld();
                        reg_fence(o);
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                        tmem_st16(tO + c, o);
                    }
                    tc_wait_st();
                    if (!(ok = warp_wait(&bars[L::bPStage + 4 * s + quarter], (pst >> s) & 1u, abort_flag, wd))) break;
                    pst ^= 1u << s;
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[L::bPFull + s]);
                }
            }
            if (ok) {
                write_out(0, cur0, of0, true);
                write_out(1, cur1, of1, true);
            }
        } else {
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            uint32_t of[2] = {0, 0}, sp[2] = {0, 0};
            uint32_t stage = 0, v8ph = 0;  // 8-bit inputs: ring slot and per-slot phase bits of bV8Full
            bool ok = true;
            for (int r = 0; r * (int)gridDim.x < total && ok; ++r) {
                const int w = snake_index(r);
                if (w >= total) continue;
                Tile t;
                get_tile<BN>(p, po, w, t);
                if constexpr (F8 != 0) {
                    // Widen this tile's 8-bit V tiles first (rows 32*quarter .. +31 of each), in ring
                    // order. The MMA warps wait for them (bVConv) before each P V product and only
                    // then release the entry, so the 8-bit tile is never overwritten while read here.
                    const int nmax = max(t.n[0], t.n[1]);
                    for (int e = 0; e <= nmax && nmax > 0 && ok; ++e) {
                        const uint32_t e_slot = stage;
                        if (++stage == (uint32_t)L::kEntries) stage = 0;
                        if (e == 0) continue;
                        if (!(ok = warp_wait(&bars[L::bV8Full + e_slot], (v8ph >> e_slot) & 1u, abort_flag, wd))) break;
                        v8ph ^= 1u << e_slot;
                        const uint32_t ent = smem_u32(smem + L::kKVOff) + e_slot * L::kEntryBytes;
                        widen_v_rows<D, F8>(ent + L::kV8Off, ent + L::kVOff, quarter * 32 + lane);
                        fence_proxy_async_smem();  // make the generic-proxy stores visible to the MMA
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars[L::bVConv + e_slot]);
                    }
                    if (!ok) break;
                }
                for (int s = 0; s < 2; ++s) {
                    const int qrow = t.r0 + s * BM + row;
                    if (t.r0 + s * BM >= t.Lq) continue;
                    const bool valid = qrow < t.Lq;
                    const long long tok = (long long)t.q0 + qrow;
                    __nv_bfloat16* orow = p.o + (tok * p.Hq + t.h) * DV;
                    if (t.n[s] == 0) {
                        if (valid) {
                            uint4 z = make_uint4(0, 0, 0, 0);
    #pragma unroll
                            for (int c = 0; c < DV / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
                            p.lse[tok * p.Hq + t.h] = -INFINITY;
                        }
                        continue;
                    }
                    if (!warp_wait(&bars[L::bOFull + s], of[s], abort_flag, wd)) { ok = false; break; }
                    of[s] ^= 1u;
                    if (!warp_wait(&bars[L::bStats + s], sp[s], abort_flag, wd)) { ok = false; break; }
                    sp[s] ^= 1u;
                    tc_fence_after();
                    const float m = st_m[s * BM + row];
                    const float l = st_l[s * BM + row];
                    const float inv = l > 0.0f ? p.out_scale / l : 0.0f;
                    const uint32_t tO = tmem + lane_off + (s ? kColO1 : kColO0);
    #pragma unroll 1
                    for (int c = 0; c < DV; c += 32) {
                        uint32_t o[32];
                        tmem_ld32(tO + c, o);
                        tc_wait_ld();
                        reg_fence(o);
                        if (valid) {
                            uint32_t pk[16];
    #pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                            uint4* dst = reinterpret_cast<uint4*>(orow + c);
    #pragma unroll
                            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[L::bOEmpty + s]);
                    if (valid) p.lse[tok * p.Hq + t.h] = l > 0.0f ? m * p.scale + logf(l) : -INFINITY;
                }
            }
        }
    }

    // ---------------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, kThreads);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    if (threadIdx.x == 0 && *abort_flag && p.status) {
        atomicCAS(p.status, 0, kDevTimeout);
        atomicAdd(p.status + 1, 1);
    }
}

template <int D, int POLY, int F8, int DV = D, int BNT = BN, int UKV = 0, int CORR = 0>
cudaError_t launch_t(const FwdTmaps& tm, const FwdParams& p, int grid, cudaStream_t stream) {
    using L = Layout<D, F8, DV, BNT>;
    static std::atomic<bool> attr_set[kMaxAttrDevices];
    // the warp groups' setmaxnreg shares add up to the launch's 512 x 128 registers
    const cudaError_t e = ensure_smem_attr(attn_fwd_kernel<D, POLY, F8, DV, BNT, UKV, CORR>, L::kAlloc, attr_set, 128);
    if (e != cudaSuccess) return e;
    attn_fwd_kernel<D, POLY, F8, DV, BNT, UKV, CORR><<<grid, kThreads, L::kAlloc, stream>>>(tm.q, tm.k, tm.v, p);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ d = 256
// Head width 256: the accumulator O of one 128-row Q tile takes 256 of the 512 TMEM columns,
// so a CTA works on one Q tile at a time and uses the other 256 columns for two S buffers. The
// unit of work is one Q tile; the two Q tiles of a 256-row work tile are consecutive units, so
// neighbouring CTAs of a round take them and stream the same K/V tiles at about the same time
// (the second read of each tile can hit the L2). S(n+1) = Q K_{n+1}^T is computed while the
// softmax works on S(n), and each KV step issues O += P(n) V_n then S(n+2) = Q K_{n+2}^T into
// the buffer P(n) came from. K and V tiles (128 keys x 256) travel as 32 KB halves
// (d 0-127 and 128-255) through a ring of five slots. The softmax warps also write the
// finished rows, so no separate epilogue warps or statistics exchange are needed.
// TMEM columns: O [0,256), S0 [256,384), S1 [384,512).
constexpr int kWideD = 256;
constexpr int kWideThreads = 256;  // warp 0 TMA, warp 1 MMA, warp 2 packed order, warps 4-7 softmax
constexpr uint32_t kWideColO = 0, kWideColS = 256;

struct LayoutWide {
    static constexpr int kQBytes = BM * kWideD * 2;          // 4 chunks of [128 rows x 128 bytes]
    static constexpr int kChunkBytes = 128 * 128;            // one [128 rows x 128 bytes] chunk
    static constexpr int kSlots = 5;
    static constexpr int kSlotBytes = 2 * kChunkBytes;       // half a K or V tile: d 0-127 or 128-255
    static constexpr int kQOff = 0;
    static constexpr int kSlotOff = kQBytes;
    static constexpr int kBarOff = kSlotOff + kSlots * kSlotBytes;
    // S-buffer barriers come in pairs: the softmax may finish P(n) and P(n+1) before the MMA
    // warp reads either, so P's barriers are per buffer like S's (one phase per use of a buffer).
    static constexpr int bQFull = 0, bQEmpty = 1, bSlot = 2, bSFull = bSlot + kSlots, bPFull = bSFull + 2,
                         bPRest = bPFull + 2, bVDone = bPRest + 2, bOFull = bVDone + 1, bDrain = bOFull + 1;
    // dynamic unit order: [2] a unit index is in the slot / every consumer has read it
    static constexpr int bUFull = bDrain + 1, bUEmpty = bUFull + 2;
    static constexpr int kNumBars = bUEmpty + 2;
    static constexpr int kMiscOff = kBarOff + ((kNumBars * 8 + 15) / 16) * 16;
    // misc: tmem base, abort flag, packed-order levels, work tiles, two unit slots
    // packed-sequence order tables (small: the tiles leave about 2 KB)
    static constexpr int kMaxB = 64;
    static constexpr int kMaxLv = 192;
    static constexpr int kPreOff = kMiscOff + 32;
    static constexpr int kLvlOff = kPreOff + ((kMaxB + 1) * 4 + 15) / 16 * 16;
    static constexpr int kPermOff = kLvlOff + ((kMaxLv + 2) * 4 + 15) / 16 * 16;
    static constexpr int kNbOff = kPermOff + kMaxB * 4;
    static constexpr int kBytes = kNbOff + kMaxB * 4;
    static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

// K/V half tiles in the order the MMA warp consumes them, per Q tile with ns key tiles:
// K0a K0b K1a K1b | V0a V0b K2a K2b | V1a V1b K3a K3b | ... (K_{n+2} only while n + 2 < ns).
// Item i lives in slot i % 5. The producer refills a slot once the products that read its
// item are complete: S(m) = Q K_m^T for a K half (the S-buffer barrier of m % 2), O += P(n)
// V_n for a V half (bVDone, one phase per step). Those barriers are shared by several items,
// and a parity wait is only meaningful while the barrier is at most one phase past the phase
// waited for, so the producer observes every phase of them in order and, before loading the
// item that lets the next product of a barrier start (the second half of V_n or of K_m), it
// first observes that barrier's previous product. A barrier then never completes a phase
// the producer has not yet observed and the one after it.
constexpr uint32_t kNoEvent = 0xffffffffu;
constexpr uint32_t kEvPV = 0u, kEvS0 = 1u, kEvS1 = 2u;  // event kinds: bVDone, bSFull + 0, bSFull + 1

// Events observed so far per barrier, and the release events of the items in the ring
// (kind << 30 | index of the event on its barrier), oldest first.
struct WideEvents {
    uint32_t seen[3];
    uint32_t r0, r1, r2, r3, r4;
};

// Wait until the event barrier of `kind` has completed phases 0 .. upto-1, one phase at a time.
__device__ __forceinline__ bool wide_observe(uint64_t* bars, WideEvents& ev, uint32_t kind, uint32_t upto,
                                             volatile int* abort_flag, uint64_t wd) {
    using L = LayoutWide;
    uint64_t* bar = &bars[kind == kEvPV ? L::bVDone : L::bSFull + (kind - kEvS0)];
    uint32_t seen = kind == kEvPV ? ev.seen[0] : (kind == kEvS0 ? ev.seen[1] : ev.seen[2]);
    while (seen < upto) {
        if (!warp_wait(bar, seen & 1u, abort_flag, wd)) return false;
        ++seen;
    }
    if (kind == kEvPV) ev.seen[0] = seen;
    else if (kind == kEvS0) ev.seen[1] = seen;
    else ev.seen[2] = seen;
    return true;
}

// Load K or V half h (d 128h .. 128h+127) of the key tile at key row `row` into the next ring
// slot, once the item it replaces has been released; `rel` is the event that will release
// this item (kind << 30 | index). False on a timeout.
__device__ __forceinline__ bool wide_load_half(uint64_t* bars, uint8_t* smem, WideEvents& ev, long long& item,
                                               const CUtensorMap* map, int kvh, int row, int h, uint32_t rel,
                                               uint32_t leader, volatile int* abort_flag, uint64_t wd) {
    using L = LayoutWide;
    static_assert(L::kSlots == 5, "ring of five slots");
    if (ev.r0 != kNoEvent && !wide_observe(bars, ev, ev.r0 >> 30, (ev.r0 & 0x3fffffffu) + 1u, abort_flag, wd))
        return false;
    ev.r0 = ev.r1, ev.r1 = ev.r2, ev.r2 = ev.r3, ev.r3 = ev.r4, ev.r4 = rel;
    const int slot = (int)(item % L::kSlots);
    uint8_t* dst = smem + L::kSlotOff + slot * L::kSlotBytes;
    mbar_arrive_expect_tx_by(leader, &bars[L::bSlot + slot], L::kSlotBytes);
#pragma unroll
    for (int c = 0; c < 2; ++c)
        tma_load_3d_by(leader, dst + c * L::kChunkBytes, map, &bars[L::bSlot + slot], (2 * h + c) * 64, kvh, row);
    ++item;
    return true;
}

__global__ void __launch_bounds__(kWideThreads, 1)
    attn_fwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using L = LayoutWide;
    static_assert(L::kAlloc <= 232448, "shared memory");
    constexpr int D = kWideD;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
    int* misc = reinterpret_cast<int*>(smem + L::kMiscOff);
    int* pre = reinterpret_cast<int*>(smem + L::kPreOff);
    int* lvl = reinterpret_cast<int*>(smem + L::kLvlOff);
    int* perm = reinterpret_cast<int*>(smem + L::kPermOff);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    ATTN_TL_DECL(int tl_idx = 0);

    if (threadIdx.x == 0) {
        mbar_init(&bars[L::bQFull], 1);
        mbar_init(&bars[L::bQEmpty], 1);
        for (int i = 0; i < L::kSlots; ++i) mbar_init(&bars[L::bSlot + i], 1);
        mbar_init(&bars[L::bSFull + 0], 1);
        mbar_init(&bars[L::bSFull + 1], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[L::bPFull + b], 4);
            mbar_init(&bars[L::bPRest + b], 4);
        }
        mbar_init(&bars[L::bVDone], 1);
        mbar_init(&bars[L::bOFull], 1);
        mbar_init(&bars[L::bDrain], 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(&bars[L::bUFull + k], 1);
            mbar_init(&bars[L::bUEmpty + k], 5);  // the MMA warp and the four softmax warps
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (p.cu_seqlens && warp == 2) {
        int levels, tiles;
        build_packed_order(p, pre, lvl, perm, reinterpret_cast<int*>(smem + L::kNbOff), lane, L::kMaxLv, levels, tiles);
        if (lane == 0) {
            misc[2] = levels;
            misc[3] = tiles;
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int total = p.total_tiles;
    const PackedOrder po{pre, lvl, perm, p.cu_seqlens ? misc[2] : 0};
    if (p.cu_seqlens) total = misc[3];
    const uint32_t tmem = *tmem_slot;
    const uint64_t wd = p.watchdog_ns;
    // Units (128-row Q tiles) this CTA works on, the k-th one per call. Static order: the snake
    // over rounds of the grid. Dynamic order (p.sched, a zeroed counter per call): the warp 0
    // takes the next unit of the order from the counter when it is ready for one and passes it
    // to the MMA and softmax warps through two shared-memory slots, so CTAs that finish early
    // take more units and all CTAs work on neighbouring units (the same few heads) at any time.
    // Returns false when no unit is left, or on a timeout (then ok = false); u = -1 for a round
    // without a unit.
    const int units = 2 * total;
    volatile int* uslot = misc + 4;
    auto next_unit = [&](int k, int& u, bool producer, bool& ok) -> bool {
        if (!p.sched) {
            if (k * (int)gridDim.x >= units) return false;
            u = snake_index(k);
            if (u >= units) u = -1;
            return true;
        }
        const int sl = k & 1;
        if (producer) {
            if (k >= 2 && !(ok = warp_wait(&bars[L::bUEmpty + sl], ((k >> 1) & 1) ^ 1, abort_flag, wd))) return false;
            int v = 0;
            if (lane == 0) {
                v = (int)atomicAdd(p.sched, 1u);
                uslot[sl] = v;
                mbar_arrive(&bars[L::bUFull + sl]);
            }
            u = __shfl_sync(0xffffffffu, v, 0);
        } else {
            if (!(ok = warp_wait(&bars[L::bUFull + sl], (k >> 1) & 1, abort_flag, wd))) return false;
            u = uslot[sl];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[L::bUEmpty + sl]);
        }
        return u < units;
    };

    if (warp == 0) {
        // ------------------------------------------------------------------ TMA producer
        const uint32_t leader = lane == 0;
        uint32_t qph = 0;
        WideEvents ev{{0, 0, 0}, kNoEvent, kNoEvent, kNoEvent, kNoEvent, kNoEvent};
        uint32_t n_pv = 0, n_s0 = 0, n_s1 = 0;  // products assigned so far: O += P V steps, S per buffer
        long long item = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int u;
            if (!next_unit(k, u, true, ok)) break;
            if (u < 0) continue;
            Tile t;
            get_tile<BN>(p, po, u >> 1, t);
            {
                const int s = u & 1;
                const int ns = s ? t.n[1] : t.n[0];
                if (ns == 0) continue;
                if (!(ok = warp_wait(&bars[L::bQEmpty], qph ^ 1u, abort_flag, wd))) break;
                qph ^= 1u;
                mbar_arrive_expect_tx_by(leader, &bars[L::bQFull], L::kQBytes);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tma_load_3d_by(leader, smem + L::kQOff + c * L::kChunkBytes, &tmQ, &bars[L::bQFull], c * 64, t.h,
                                   t.q0 + t.r0 + s * BM);
                // S(m) on buffer m % 2: its two K halves; the second lets the product start
                auto load_k = [&](int m) {
                    const uint32_t b = (uint32_t)(m & 1), kind = b ? kEvS1 : kEvS0, idx = b ? n_s1++ : n_s0++;
                    ok = wide_load_half(bars, smem, ev, item, &tmK, t.kvh, t.k0 + m * BN, 0, (kind << 30) | idx, leader,
                                        abort_flag, wd) &&
                         wide_observe(bars, ev, kind, idx, abort_flag, wd) &&
                         wide_load_half(bars, smem, ev, item, &tmK, t.kvh, t.k0 + m * BN, 1, (kind << 30) | idx, leader,
                                        abort_flag, wd);
                };
                for (int m = 0; m < ns && m < 2 && ok; ++m) load_k(m);
                for (int n = 0; n < ns && ok; ++n) {
                    ATTN_TL_DECL(long long tv = clock64());
                    // O += P(n) V_n: its two V halves; the second lets the product start
                    const uint32_t idx = n_pv++;
                    ok = wide_load_half(bars, smem, ev, item, &tmV, t.kvh, t.k0 + n * BN, 0, (kEvPV << 30) | idx, leader,
                                        abort_flag, wd) &&
                         wide_observe(bars, ev, kEvPV, idx, abort_flag, wd) &&
                         wide_load_half(bars, smem, ev, item, &tmV, t.kvh, t.k0 + n * BN, 1, (kEvPV << 30) | idx, leader,
                                        abort_flag, wd);
                    ATTN_TL(0, 0, n, tv, clock64());
                    if (n + 2 < ns && ok) {
                        ATTN_TL_DECL(long long tk = clock64());
                        load_k(n + 2);
                        ATTN_TL(0, 1, n, tk, clock64());
                    }
                }
            }
        }
        if (!ok) {
            // Let copies already in flight land before the CTA can exit.
            for (int i = 0; i < L::kSlots && i < item; ++i) {
                const long long it = item - 1 - i;
                int dummy = 0;
                mbar_wait(&bars[L::bSlot + (int)(it % L::kSlots)], (uint32_t)((it / L::kSlots) & 1), &dummy, 20000000ull);
            }
            int dummy = 0;
            mbar_wait(&bars[L::bQFull], qph ^ 1u, &dummy, 20000000ull);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        // Per Q tile: S(0), S(1); then per step n: O += P(n) V_n (both 128-column halves of O,
        // the first three quarters of the keys as soon as P stage 1 is written), one commit
        // (bVDone), then S(n+2) into the buffer of P(n) and its commit. The S(n+2) products
        // follow O += P(n) V_n in issue order, so they overwrite P(n) only after it is read.
        const uint32_t leader = lane == 0;
        constexpr uint32_t idS = idesc_bf16_f32(BM, BN, 0);
        constexpr uint32_t idO = idesc_bf16_f32(BM, 128, 1);
        constexpr int kPA = (3 * BN / 4) / 16;  // P stage 1: k-steps 0 .. kPA-1
        const uint32_t q_base = smem_u32(smem + L::kQOff);
        const uint32_t slot_base = smem_u32(smem + L::kSlotOff);
        const uint64_t dq = smem_desc_sw128(q_base, 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(slot_base, 16, 1024);
        const uint64_t dv0 = smem_desc_sw128(slot_base, L::kChunkBytes, 1024);
        uint32_t qf = 0, pf = 0;  // pf bit b: parity of the next P phase of S buffer b
        long long item = 0;
        bool ok = true, any = false;
        // Wait for the next ring item; returns its slot.
        auto next_slot = [&](int& slot) -> bool {
            slot = (int)(item % L::kSlots);
            const uint32_t par = (uint32_t)((item / L::kSlots) & 1);
            ++item;
            return warp_wait(&bars[L::bSlot + slot], par, abort_flag, wd);
        };
        // S(m) = Q K_m^T into S buffer sb: the k-steps of the first K half (d 0-127) as soon as it
        // has landed, then those of the second; false on a timeout
        auto issue_s = [&](uint32_t sb) -> bool {
            const uint32_t colS = kWideColS + 128u * sb;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int slot;
                if (!next_slot(slot)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int k = 8 * h + kk;
                    const uint64_t oq = (uint64_t)(((k >> 2) * L::kChunkBytes + (k & 3) * 32) >> 4);
                    const uint64_t ok_ =
                        (uint64_t)((slot * L::kSlotBytes + ((kk >> 2) & 1) * L::kChunkBytes + (k & 3) * 32) >> 4);
                    tc_mma_ss_by(leader, tmem + colS, dq + oq, dk0 + ok_, idS, k > 0 ? 1u : 0u);
                }
            }
            return true;
        };
        for (int k = 0; ok; ++k) {
            int u;
            if (!next_unit(k, u, false, ok)) break;
            if (u < 0) continue;
            Tile t;
            get_tile<BN>(p, po, u >> 1, t);
            {
                const int s = u & 1;
                const int ns = s ? t.n[1] : t.n[0];
                if (ns == 0) continue;
                if (!(ok = warp_wait(&bars[L::bQFull], qf, abort_flag, wd))) break;
                qf ^= 1u;
                any = true;
                tc_fence_after();
                for (int m = 0; m < ns && m < 2; ++m) {
                    if (!(ok = issue_s((uint32_t)(m & 1)))) break;
                    __syncwarp();
                    tc_commit_by(leader, &bars[L::bSFull + (m & 1)]);
                    if (m == ns - 1) tc_commit_by(leader, &bars[L::bQEmpty]);
                }
                for (int n = 0; n < ns && ok; ++n) {
                    const uint32_t sb = (uint32_t)(n & 1);
                    const uint32_t colS = kWideColS + 128u * sb;
                    ATTN_TL_DECL(long long t0 = clock64());
                    if (!(ok = warp_wait(&bars[L::bPFull + sb], (pf >> sb) & 1u, abort_flag, wd))) break;
                    ATTN_TL_DECL(long long t1 = clock64());
                    // P stage 1 (keys 0-95) with each V half as soon as it has landed: O columns
                    // 0-127 from V_n's d 0-127, then columns 128-255 from d 128-255
                    const uint32_t acc0 = n > 0 ? 1u : 0u;
                    int va, vb;
                    if (!(ok = next_slot(va))) break;
                    ATTN_TL(1, 100, n, t0, t1);
                    ATTN_TL(1, 101, n, clock64(), 0);
                    tc_fence_after();
                    const uint64_t vda = dv0 + (uint64_t)((va * L::kSlotBytes) >> 4);
#pragma unroll
                    for (int k = 0; k < kPA; ++k)
                        tc_mma_ts_by(leader, tmem + kWideColO, tmem + colS + k * 8, vda + (uint64_t)(k * (2048 >> 4)),
                                     idO, k == 0 ? acc0 : 1u);
                    if (!(ok = next_slot(vb))) break;
                    tc_fence_after();
                    const uint64_t vdb = dv0 + (uint64_t)((vb * L::kSlotBytes) >> 4);
#pragma unroll
                    for (int k = 0; k < kPA; ++k)
                        tc_mma_ts_by(leader, tmem + kWideColO + 128, tmem + colS + k * 8,
                                     vdb + (uint64_t)(k * (2048 >> 4)), idO, k == 0 ? acc0 : 1u);
                    if (!(ok = warp_wait(&bars[L::bPRest + sb], (pf >> sb) & 1u, abort_flag, wd))) break;
                    pf ^= 1u << sb;
                    tc_fence_after();
#pragma unroll
                    for (int k = kPA; k < BN / 16; ++k) {  // P stage 2
                        tc_mma_ts_by(leader, tmem + kWideColO, tmem + colS + k * 8, vda + (uint64_t)(k * (2048 >> 4)),
                                     idO, 1u);
                        tc_mma_ts_by(leader, tmem + kWideColO + 128, tmem + colS + k * 8,
                                     vdb + (uint64_t)(k * (2048 >> 4)), idO, 1u);
                    }
                    __syncwarp();
                    tc_commit_by(leader, &bars[L::bVDone]);
                    if (n == ns - 1) tc_commit_by(leader, &bars[L::bOFull]);
                    ATTN_TL(1, 102, n, clock64(), 0);
                    if (n + 2 < ns) {
                        ATTN_TL(1, 103, n, clock64(), 0);
                        if (!(ok = issue_s(sb))) break;
                        __syncwarp();
                        tc_commit_by(leader, &bars[L::bSFull + sb]);
                        if (n + 2 == ns - 1) tc_commit_by(leader, &bars[L::bQEmpty]);
                        ATTN_TL(1, 104, n, clock64(), 0);
                    }
                }
            }
        }
        if (any) {
            // Wait until every MMA this warp issued has completed before TMEM can be released.
            tc_commit_by(leader, &bars[L::bDrain]);
            int dummy = 0;
            if (leader) mbar_wait(&bars[L::bDrain], 0, &dummy, 50000000ull);
            __syncwarp();
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------------ softmax + output
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + kWideColO;
        const float sl2 = p.scale_log2;
        uint32_t sf = 0, of = 0, pv_done = 0;  // sf bit b: S buffer b parity; pv_done: O += P V steps before this tile
        unsigned long long c_dec = 0, c_res = 0, c_dec1 = 0, c_ores = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int u;
            if (!next_unit(k, u, false, ok)) break;
            if (u < 0) continue;
            Tile t;
            get_tile<BN>(p, po, u >> 1, t);
            {
                const int s = u & 1;
                const int tile_row0 = t.r0 + s * BM;
                if (tile_row0 >= t.Lq) continue;
                const int ns = s ? t.n[1] : t.n[0];
                const int qrow = tile_row0 + row;
                const bool valid = qrow < t.Lq;
                const long long tok = (long long)t.q0 + qrow;
                __nv_bfloat16* orow = p.o + (tok * p.Hq + t.h) * D;
                if (ns == 0) {  // no visible key: zero output, LSE -inf
                    if (valid) {
                        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
                        p.lse[tok * p.Hq + t.h] = -INFINITY;
                    }
                    continue;
                }
                const int off = t.Lk - t.Lq;
                float m = -INFINITY, l = 0.0f;
                for (int n = 0; n < ns; ++n) {
                    const uint32_t sb = (uint32_t)(n & 1);
                    const uint32_t tS = tmem + lane_off + kWideColS + 128u * sb;
                    ATTN_TL_DECL(long long ts0 = clock64());
                    if (!warp_wait(&bars[L::bSFull + sb], (sf >> sb) & 1u, abort_flag, wd)) { ok = false; break; }
                    ATTN_TL_DECL(long long ts1 = clock64());
                    sf ^= 1u << sb;
                    tc_fence_after();
                    uint32_t rr[BN / 32][32];
#pragma unroll
                    for (int i = 0; i < BN / 32; ++i) tmem_ld32(tS + 32 * i, rr[i]);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < BN / 32; ++i) reg_fence(rr[i]);
                    float sv[BN];
#pragma unroll
                    for (int c = 0; c < BN; ++c) sv[c] = __uint_as_float(rr[c >> 5][c & 31]);
                    const int kb = n * BN;
                    const bool need_mask = (kb + BN > t.Lk) || (p.causal && kb + BN - 1 > tile_row0 + off);
                    if (need_mask) {
                        const int lim = (p.causal ? min(t.Lk, qrow + off + 1) : t.Lk) - kb;
#pragma unroll
                        for (int c = 0; c < BN; ++c)
                            if (c >= lim) sv[c] = -INFINITY;
                    }
                    float mx[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = fmaxf(sv[i], sv[i + 8]);
#pragma unroll
                    for (int c = 16; c < BN; c += 16)
#pragma unroll
                        for (int i = 0; i < 8; ++i) mx[i] = max3f(mx[i], sv[c + i], sv[c + 8 + i]);
                    const float mt = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                    const float m_cand = fmaxf(m, mt);
                    const bool need = (m_cand - m) * sl2 > p.rescale_thr;  // NaN (both -inf) is false
                    if (__any_sync(0xffffffffu, need)) {
                        const float alpha = (m == -INFINITY) ? 0.0f : ex2_mufu((m - m_cand) * sl2);
                        if (n > 0) {
                            ++c_ores;
                            // O += P(n-1) V_{n-1} must be complete before O is rescaled (S(n) was
                            // issued before it, so the S barrier does not cover it).
                            if (!warp_wait(&bars[L::bVDone], (pv_done + (uint32_t)n - 1u) & 1u, abort_flag, wd)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
#pragma unroll 1
                            for (int c = 0; c < D; c += 16) {
                                uint32_t o[16];
                                tmem_ld16(tO + c, o);
                                tc_wait_ld();
                                reg_fence(o);
#pragma unroll
                                for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                                tmem_st16(tO + c, o);
                            }
                        }
                        l *= alpha;
                        m = m_cand;
                        ++c_res;
                    }
                    ++c_dec;
                    if (n > 0) ++c_dec1;
                    const float neg = (m == -INFINITY) ? 0.0f : -m * sl2;
                    float sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    uint32_t pk[BN / 2];
                    constexpr int kSA = (3 * BN / 4) / 16 * 16;
                    auto exp_pair = [&](int c) {
                        float x0, x1;
                        ffma2(x0, x1, sv[c], sv[c + 1], sl2, sl2, neg, neg);
                        const float p0 = ex2_mufu(x0), p1 = ex2_mufu(x1);
                        const int a = ((c >> 1) & 3) * 2;
                        fadd2(sum[a], sum[a + 1], sum[a], sum[a + 1], p0, p1);
                        pk[c >> 1] = pack_bf16x2(p0, p1);
                    };
#pragma unroll
                    for (int c = 0; c < kSA; c += 2) exp_pair(c);
                    store_p_cols<0, kSA / 2>(tS, pk);
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[L::bPFull + sb]);
#pragma unroll
                    for (int c = kSA; c < BN; c += 2) exp_pair(c);
                    store_p_cols<kSA / 2, BN / 2>(tS, pk);
                    l += ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[L::bPRest + sb]);
                    if (quarter == 0) ATTN_TL(2, n, ts0, ts1, clock64());
                }
                if (!ok) break;
                pv_done += (uint32_t)ns;
                // output: O / l in bf16 and the LSE, once the last O += P V is complete
                if (!warp_wait(&bars[L::bOFull], of, abort_flag, wd)) { ok = false; break; }
                of ^= 1u;
                tc_fence_after();
                const float inv = l > 0.0f ? p.out_scale / l : 0.0f;
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + c, o);
                    tc_wait_ld();
                    reg_fence(o);
                    if (valid) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                        uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
                // the next tile's first P V product overwrites O: the loads above are ordered
                // before it by the fence and arrive that publish that tile's P
                if (valid) p.lse[tok * p.Hq + t.h] = l > 0.0f ? m * p.scale + logf(l) : -INFINITY;
            }
        }
        if (p.counters && lane == 0) {
            atomicAdd(p.counters + 0, c_dec);
            atomicAdd(p.counters + 1, c_res);
            atomicAdd(p.counters + 3, c_dec * 32ull * BN);
            atomicAdd(p.counters + 4, c_dec1);
            atomicAdd(p.counters + 5, c_ores);
        }
    }

    // ---------------------------------------------------------------------- teardown
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, kWideThreads);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    if (threadIdx.x == 0 && *abort_flag && p.status) {
        atomicCAS(p.status, 0, kDevTimeout);
        atomicAdd(p.status + 1, 1);
    }
}

cudaError_t launch_wide(const FwdTmaps& tm, const FwdParams& p, int grid, cudaStream_t stream) {
    static std::atomic<bool> attr_set[kMaxAttrDevices];
    const cudaError_t e = ensure_smem_attr(attn_fwd_wide_kernel, LayoutWide::kAlloc, attr_set);
    if (e != cudaSuccess) return e;
    attn_fwd_wide_kernel<<<grid, kWideThreads, LayoutWide::kAlloc, stream>>>(tm.q, tm.k, tm.v, p);
    return cudaGetLastError();
}

}  // namespace

int fwd_max_varlen_batch(int d) {
    if (d == kWideD) return LayoutWide::kMaxB;
    return d > 128 ? Layout<192, 0, 128, kBNWide>::kMaxB : kMaxVarlenB;
}

cudaError_t launch_attn_fwd_wide(const FwdTmaps& tm, const FwdParams& p, int grid, cudaStream_t stream) {
    return launch_wide(tm, p, grid, stream);
}

cudaError_t launch_attn_fwd_hd(const FwdTmaps& tm, const FwdParams& p, int d, int dv, int grid, cudaStream_t stream) {
    if (d == 192 && dv == 128) return launch_t<192, 0, 0, 128, kBNWide>(tm, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_fwd(const FwdTmaps& tm, const FwdParams& p, int d, int exp_poly, int grid,
                            cudaStream_t stream) {
    if (d == 128) {
        if (exp_poly) return launch_t<128, 8, 0>(tm, p, grid, stream);
        if (p.unroll_kv) return launch_t<128, 0, 0, 128, BN, 1>(tm, p, grid, stream);
        return p.corr_warp ? launch_t<128, 0, 0, 128, BN, 0, 1>(tm, p, grid, stream) : launch_t<128, 0, 0>(tm, p, grid, stream);
    }
    return exp_poly ? launch_t<64, 8, 0>(tm, p, grid, stream) : launch_t<64, 0, 0>(tm, p, grid, stream);
}

cudaError_t launch_attn_fwd_fp8(const FwdTmaps& tm, const FwdParams& p, int d, int fmt, int grid,
                                cudaStream_t stream) {
    if (d != 128) return cudaErrorInvalidValue;
    if (fmt == 0)
        return p.unroll_kv ? launch_t<128, 0, 1, 128, BN, 1>(tm, p, grid, stream) : launch_t<128, 0, 1>(tm, p, grid, stream);
    return launch_t<128, 0, 2>(tm, p, grid, stream);
}

// ------------------------------------------------------------------------------ diagnostics

namespace {
__global__ void exp2_probe_kernel(const float* x, float* y, long long n, int mode) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        y[i] = mode == 0 ? ex2_poly(x[i]) : ex2_mufu(x[i]);
}

// Waits on an mbarrier that nothing ever arrives on, with the same bounded wait the
// attention kernels use, and reports the timeout through the status word.
__global__ void watchdog_probe_kernel(int* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, &abort_flag, limit_ns);
    __syncthreads();
    if (threadIdx.x == 0 && !ok) {
        atomicCAS(status, 0, kDevTimeout);
        atomicAdd(status + 1, 1);
    }
}
}  // namespace

cudaError_t launch_exp2_probe(const float* x, float* y, long long n, int mode, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    exp2_probe_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, y, n, mode);
    return cudaGetLastError();
}

cudaError_t launch_watchdog_probe(int* status, unsigned long long limit_ns, cudaStream_t stream) {
    watchdog_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace attn

#ifdef ATTN_TIMELINE
extern "C" int attn_timeline_read(long long* out, int* counts) {
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(out, attn::g_timeline, sizeof(long long) * 5 * 4096 * 4);
    cudaMemcpyFromSymbol(counts, attn::g_timeline_n, sizeof(int) * 5);
    int z[5] = {0, 0, 0, 0, 0};
    cudaMemcpyToSymbol(attn::g_timeline_n, z, sizeof(z));
    return 0;
}
#endif
