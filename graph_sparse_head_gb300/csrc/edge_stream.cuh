// The streaming edge-attention kernel (kpnn2 PackedMultiheadAttention,
// Notes steps 2-4), templated on its lane shape. Included by the
// translation units that instantiate it for fp16 and float32 intermediates.
//
// Work decomposition. The CSR positions of one sample are cut into units of
// kUnitEdges consecutive positions (edges of consecutive targets, each
// target's edges ordered by source). A unit is walked by one "slot": the LPE
// lanes that own one row of channels, a lane owning CPL consecutive channels
// (one whole head when the head has at most 16 channels). A warp runs the
// same unit for 32 / LPE samples side by side, so its slots never diverge.
// Every slot does the same gather work whatever the in-degrees: a target
// inside one unit is finished there; a target crossing a unit boundary leaves
// partial softmax states, and the slot that writes its last piece (counted
// with one atomic per sample and target) combines them in unit order.
//
// Per edge, a lane gathers its chunks of the source's k and v rows through
// cp.async into a per-lane ring of shared-memory stages, kDepth edges ahead
// of use, so the loads in flight hold no registers. Edges go two per step:
// when both belong to the current target their scores are independent and
// share one rescale; at a target boundary they go one at a time. Source
// indices (three windows of LPE positions), target bounds (row_ptr) and the
// next target's q row are prefetched in registers. When a head spans several lanes, its dot
// product is a butterfly sum over them, so those lanes hold the same score.
//
// The softmax is online, in log2 units: s = (q . k) * log2(e)/sqrt(d). With
// fp16 rows the dot product takes mixed-precision FMAs on the packed halves
// (fp16 products are exact in fp32, so no widening is needed) and is scaled
// once; fp32 rows use q pre-scaled in fp32 pairs. m is a lazy reference: it
// moves to a new score only when that score exceeds it by more than kLazy, so
// most edges skip the rescale of l and acc; l = running sum of 2^(s - m), acc
// = running sum of 2^(s - m) v, updated with paired fp32 FMAs. The (m, l)
// arithmetic uses explicit round-to-nearest operations so that it is identical in the variants with and without values; that makes
// pmha_edge_weights bit-identical to the weights of pmha_forward.
#pragma once

#include <math.h>

#include <type_traits>

#include "pmha_internal.h"

namespace pmha {
namespace stream {

#ifndef PMHA_STREAM_DEPTH
#define PMHA_STREAM_DEPTH 4
#endif
#ifndef PMHA_STREAM_WARPS
#define PMHA_STREAM_WARPS 2
#endif
#ifndef PMHA_STREAM_LINE_COPY
#define PMHA_STREAM_LINE_COPY 1
#endif
#ifndef PMHA_STREAM_MIXED_FMA
#define PMHA_STREAM_MIXED_FMA 1
#endif
#ifndef PMHA_STREAM_LAZY
#define PMHA_STREAM_LAZY 8
#endif
constexpr int kWarps = PMHA_STREAM_WARPS;  // warps per block
constexpr int kDepth = PMHA_STREAM_DEPTH;  // edges in flight per slot (even: two per step)
constexpr int kRing = kDepth + 2;          // stages: a stage is refilled one step after it was read
// The running reference m moves only when a score exceeds it by more than
// kLazy (log2 units), so 2^(s - m) <= 2^kLazy; 0 moves it at every new maximum.
constexpr float kLazy = (float)PMHA_STREAM_LAZY;

struct Args {
    const void *q;
    long long q_ld;
    const void *kv;
    long long kv_ld, v_off;
    void *mixed;
    float *part;
    float *ml;
    float *scores;  // (B, nnz, H) raw scores by CSR position, or null
    const int32_t *row_ptr;
    const int32_t *col;
    const int32_t *unit_first_t;
    const int32_t *unit_order;  // units by decreasing estimated work (the ring kernel's queue order)
    unsigned *task_counter;     // next task of the ring kernel's queue (zero at launch)
    const uint8_t *kpm;  // (B, S) key_padding_mask, nonzero = key dropped; or null
    const uint32_t *kpm_bits;  // (B, n_kw) the mask per CSR position, 32 positions a word
    long long n_kw;
    int *counters;             // (B, n_merge) pieces written per crossing target (zero at launch)
    const int32_t *merge_pos;  // L, index of a target in the merge list
    long long n_merge;
    long long n_units, nnz;
    int B, L, S, E, H, d;
    float score_scale;
    // out_proj inside the ring kernel (edge_out.cuh); out = null: none
    void *out;                 // (B, L, E) bf16 rows
    const uint32_t *wo_frag;   // Wo as fp16 in wo_frag_pos order
    const void *bo;            // (E) bf16, or null (no bias)
    int *blk_count;            // (B, n_blk) finished targets per block of kOutRows (zero at launch)
    int n_blk;
    int *err;                  // device error word (a poll that gave up sets kErrTimeoutBit)
};

template <typename T, int CPL, bool WV>
constexpr int smem_bytes()
{
    return kWarps * kRing * (WV ? 2 : 1) * 32 * CPL * (int)sizeof(T);
}

// x += a.lo * b.lo, y += a.hi * b.hi for two fp16 pairs, one rounding each
// (the fp16 product is exact in fp32, so this equals widening then fma.rn.f32)
__device__ __forceinline__ void fma_h2(float &x, float &y, uint32_t a, uint32_t b)
{
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %2;\n\tmov.b32 {b0, b1}, %3;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %1, a1, b1, %1;\n\t}"
        : "+f"(x), "+f"(y)
        : "r"(a), "r"(b));
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// f(std::integral_constant<int, I>) for I = FIRST .. LAST-1, unrolled at compile time
template <int I, int N, typename F>
__device__ __forceinline__ void static_for(F &&f)
{
    if constexpr (I < N) {
        f(std::integral_constant<int, I>{});
        static_for<I + 1, N>(f);
    }
}

// One 16-byte cp.async from src + SOFF to dst + DOFF, the offsets as
// immediates of the address operands (no address arithmetic per chunk).
template <int DOFF, int SOFF>
__device__ __forceinline__ void cp_async16_at(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%3], 16;" ::"r"(dst), "l"(src), "n"(DOFF), "n"(SOFF)
                 : "memory");
}

template <int CB>
__device__ __forceinline__ void cp_async(uint32_t dst, const void *src)
{
    if constexpr (CB >= 16) {
        static_for<0, CB / 16>([&](auto ic) {
            constexpr int i = decltype(ic)::value;
            cp_async16_at<16 * i, 16 * i>(dst, src);
        });
    } else {
        asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(dst), "l"(src), "n"(CB) : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int CB>
struct Raw {
    uint32_t w[CB / 4];
};

template <int CB>
__device__ __forceinline__ Raw<CB> lds_raw(uint32_t addr)
{
    Raw<CB> r;
    if constexpr (CB % 16 == 0) {
        static_for<0, CB / 16>([&](auto ic) {
            constexpr int i = decltype(ic)::value;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
                         : "=r"(r.w[4 * i]), "=r"(r.w[4 * i + 1]), "=r"(r.w[4 * i + 2]), "=r"(r.w[4 * i + 3])
                         : "r"(addr), "n"(16 * i));
        });
    } else if constexpr (CB == 8) {
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "r"(addr));
    } else {
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r.w[0]) : "r"(addr));
    }
    return r;
}

template <int CB>
__device__ __forceinline__ Raw<CB> ldg_raw(const void *p)
{
    Raw<CB> r;
    if constexpr (CB % 16 == 0) {
#pragma unroll
        for (int i = 0; i < CB / 16; ++i) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p) + i);
            r.w[4 * i] = u.x;
            r.w[4 * i + 1] = u.y;
            r.w[4 * i + 2] = u.z;
            r.w[4 * i + 3] = u.w;
        }
    } else if constexpr (CB == 8) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        r.w[0] = u.x;
        r.w[1] = u.y;
    } else {
        r.w[0] = __ldg(reinterpret_cast<const unsigned int *>(p));
    }
    return r;
}

// ---- paired fp32 arithmetic (each half rounds exactly like its scalar op)
typedef unsigned long long f2;
__device__ __forceinline__ f2 pk(float x, float y)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 upk(f2 r)
{
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
    return f;
}
__device__ __forceinline__ f2 ffma2(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 fmul2(f2 a, f2 b)
{
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// CPL channels of type T in `r`, widened to CPL / 2 fp32 pairs.
template <typename T, int CPL>
__device__ __forceinline__ void widen2(const Raw<CPL * (int)sizeof(T)> &r, f2 (&f)[CPL / 2])
{
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int j = 0; j < CPL / 2; ++j) {
            const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&r.w[j]));
            f[j] = pk(x.x, x.y);
        }
    } else {
#pragma unroll
        for (int j = 0; j < CPL / 2; ++j) f[j] = pk(__uint_as_float(r.w[2 * j]), __uint_as_float(r.w[2 * j + 1]));
    }
}

template <typename T, int CPL>
__device__ __forceinline__ void store_row(T *p, const f2 (&v)[CPL / 2])
{
    if constexpr (sizeof(T) == 2) {
        uint32_t w[CPL / 2];
#pragma unroll
        for (int j = 0; j < CPL / 2; ++j) {
            const float2 x = upk(v[j]);
            __half2 h = __floats2half2_rn(x.x, x.y);
            w[j] = *reinterpret_cast<uint32_t *>(&h);
        }
        if constexpr (CPL * 2 >= 16) {
#pragma unroll
            for (int i = 0; i < CPL * 2 / 16; ++i)
                reinterpret_cast<uint4 *>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        } else if constexpr (CPL * 2 == 8) {
            *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
        } else {
            *reinterpret_cast<uint32_t *>(p) = w[0];
        }
    } else {
#pragma unroll
        for (int j = 0; j < CPL / 2; ++j) reinterpret_cast<float2 *>(p)[j] = upk(v[j]);
    }
}

// WV: mix values (else scores and (m, l) only); WS: write raw scores;
// KPM: read a key_padding_mask (a dropped key scores -inf).
template <typename T, int CPL, int LPE, bool WV, bool WS, bool KPM>
__global__ void __launch_bounds__(kWarps * 32) k_edge_stream(Args a)
{
    constexpr int P = 32 / LPE;               // slots per warp
    constexpr int CB = CPL * (int)sizeof(T);  // bytes per lane per row
    constexpr int NR = WV ? 2 : 1;            // rows staged per edge: k (and v)
    constexpr int NP = CPL / 2;               // fp32 pairs per lane
    constexpr int STAGE = NR * 32 * CB;       // bytes of one stage of one warp
    extern __shared__ __align__(16) unsigned char smem_dyn[];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slot = lane / LPE, grp = lane % LPE;
    const unsigned smask = LPE == 32 ? 0xffffffffu : (((1u << LPE) - 1u) << (slot * LPE));
    // the P slots of a warp walk the same unit for P consecutive samples: the
    // graph is shared by all samples, so their control flow is identical
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const long long groups = (a.B + P - 1) / P;
    if (gw >= groups * a.n_units) return;
    const int u = (int)(gw % a.n_units);
    const int b = (int)(gw / a.n_units) * P + slot;
    const unsigned live = __ballot_sync(0xffffffffu, b < a.B);  // lanes of the slots that run
    if (b >= a.B) return;  // the whole slot leaves together
    const int e0 = u * kUnitEdges;
    const int n = (int)min((long long)kUnitEdges, a.nnz - e0);
    const int e1 = e0 + n;

    const int c0 = grp * CPL;
    const int head = c0 / a.d;
    const int lph = a.d / CPL;  // lanes per head (1 when a lane owns a whole head)
    const bool head_leader = (grp & (lph - 1)) == 0;

    const uint32_t sbase = smem_u32(smem_dyn) + (uint32_t)(warp * kRing * STAGE + lane * CB);
    // Row copies by the whole slot: the k|v bytes of a row (v right after k)
    // are cut into 16-byte chunks and lane grp copies chunks q * LPE + grp, so
    // every cp.async instruction reads whole 32-byte sectors (a lane copying
    // only its own 32 bytes reads half sectors, twice). A chunk lands where
    // its consumer lane reads it, so each wait is followed by a warp barrier.
    constexpr bool kLineCopy = PMHA_STREAM_LINE_COPY && CB >= 16;
    constexpr int RK = LPE * CB;  // bytes of a row's k part (= E elements)
    const uint32_t sslot = smem_u32(smem_dyn) + (uint32_t)(warp * kRing * STAGE + slot * LPE * CB);
    const char *KVs = (const char *)a.kv + (long long)b * a.S * a.kv_ld * (long long)sizeof(T);
    auto copy_row = [&](uint32_t dst, const char *row) {
        // chunk q * LPE + grp: one base address per row, the chunk offsets as immediates
        const uint32_t d0 = dst + 16 * grp;
        const char *s0 = row + 16 * grp;
        static_for<0, NR * CB / 16>([&](auto qc) {
            constexpr int q = decltype(qc)::value;
            cp_async16_at<16 * q * LPE + (q >= CB / 16 ? 32 * CB - RK : 0), 16 * q * LPE>(d0, s0);
        });
    };
    const char *KVb = (const char *)a.kv + ((long long)b * a.S * a.kv_ld + c0) * (long long)sizeof(T);
    const long long row_bytes = a.kv_ld * (long long)sizeof(T);
    const long long v_bytes = a.v_off * (long long)sizeof(T);
    const T *Qb = (const T *)a.q + (long long)b * a.L * a.q_ld + c0;
    float *scores_b = WS ? a.scores + (long long)b * a.nnz * a.H : nullptr;
    const int32_t *colu = a.col + e0;

    // ---- gathers: windows w, w + 1, w + 2 of source indices (lane grp holds position w * LPE + grp)
    auto ldcol = [&](int w) -> int {
        const int p = w * LPE + grp;
        return p < n ? colu[p] : 0;
    };
    int iw = 0;
    int cw0 = ldcol(0), cw1 = ldcol(1), cw2 = ldcol(2);
    // edges j and j + 1 (j even) in one commit group, into ring stages sj and
    // sj + 1 (sj = j mod kRing, even since kRing is); both lie in one window
    auto issue2 = [&](int j, int sj) {
        if (j >= (iw + 1) * LPE) {
            ++iw;
            cw0 = cw1;
            cw1 = cw2;
            cw2 = ldcol(iw + 2);
        }
        const int s0 = __shfl_sync(smask, cw0, j & (LPE - 1), LPE);
        const int s1 = __shfl_sync(smask, cw0, (j + 1) & (LPE - 1), LPE);
        if constexpr (kLineCopy) {
            if (j < n) copy_row(sslot + (uint32_t)(sj * STAGE), KVs + (long long)s0 * row_bytes);
            if (j + 1 < n) copy_row(sslot + (uint32_t)((sj + 1) * STAGE), KVs + (long long)s1 * row_bytes);
        } else {
            if (j < n) {
                const char *row = KVb + (long long)s0 * row_bytes;
                const uint32_t dst = sbase + (uint32_t)(sj * STAGE);
                cp_async<CB>(dst, row);
                if constexpr (WV) cp_async<CB>(dst + 32 * CB, row + v_bytes);
            }
            if (j + 1 < n) {
                const char *row = KVb + (long long)s1 * row_bytes;
                const uint32_t dst = sbase + (uint32_t)((sj + 1) * STAGE);
                cp_async<CB>(dst, row);
                if constexpr (WV) cp_async<CB>(dst + 32 * CB, row + v_bytes);
            }
        }
        cp_async_commit();
    };
    static_assert(kDepth % 2 == 0, "edges go two per step");
#pragma unroll
    for (int j = 0; j < kDepth; j += 2) issue2(j, j);

    // ---- key_padding_mask per CSR position (one bit each, 32 positions a
    // word, the next word prefetched): every lane holds the same word
    const uint32_t *kb = KPM ? a.kpm_bits + (long long)b * a.n_kw : nullptr;
    auto ldword = [&](int w) -> uint32_t { return (KPM && w < a.n_kw) ? kb[w] : 0u; };
    int kwi = e0 >> 5;
    uint32_t kw_cur = ldword(kwi), kw_nxt = ldword(kwi + 1);
    auto masked = [&](int j) -> bool {  // j never decreases, by at most 32 per call
        const int pos = e0 + j;
        if ((pos >> 5) != kwi) {
            ++kwi;
            kw_cur = kw_nxt;
            kw_nxt = ldword(kwi + 1);
        }
        return (kw_cur >> (pos & 31)) & 1u;
    };

    // ---- target bounds: lane grp holds row_ptr[tw + grp + 1], the end of target tw + grp
    int t = a.unit_first_t[u];
    int tw = t;
    int rp_cur = tw + grp < a.L ? a.row_ptr[tw + grp + 1] : (int)a.nnz;
    int rp_nxt = tw + LPE + grp < a.L ? a.row_ptr[tw + LPE + grp + 1] : (int)a.nnz;
    auto end_of = [&](int tt) -> int {  // row_ptr[tt + 1]; tt never decreases
        while (tt - tw >= LPE) {
            tw += LPE;
            rp_cur = rp_nxt;
            rp_nxt = tw + LPE + grp < a.L ? a.row_ptr[tw + LPE + grp + 1] : (int)a.nnz;
        }
        return __shfl_sync(smask, rp_cur, tt - tw, LPE);
    };
    int bound = end_of(t);
    const bool first_started_here = a.row_ptr[t] == e0;
    bool is_first = true;

    // fp16 rows: q stays packed and the scores take mixed-precision FMAs (no
    // widening), scaled once per score; fp32 rows: q pre-scaled in fp32 pairs
    constexpr bool kMixed = PMHA_STREAM_MIXED_FMA && sizeof(T) == 2;
    f2 q2[kMixed ? 1 : NP];
    Raw<CB> qr;
    const f2 sc2 = pk(a.score_scale, a.score_scale);
    auto set_q = [&](const Raw<CB> &r) {
        if constexpr (kMixed) {
            qr = r;
        } else {
            widen2<T, CPL>(r, q2);
#pragma unroll
            for (int j = 0; j < NP; ++j) q2[j] = fmul2(q2[j], sc2);
        }
    };
    set_q(ldg_raw<CB>(Qb + (long long)t * a.q_ld));
    Raw<CB> qnext = ldg_raw<CB>(Qb + (long long)min(t + 1, a.L - 1) * a.q_ld);

    float m = -INFINITY, l = 0.f;
    f2 acc2[NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) acc2[j] = 0ull;

    // Combine the partial states (m, l, acc) of target t's pieces, unit order:
    // M = max m_i, L = sum l_i 2^(m_i - M), acc = sum acc_i 2^(m_i - M); an
    // empty piece (every key dropped) has m = -inf, l = 0 and adds nothing.
    auto merge_pieces = [&](int beg, int u0, int n_pieces) {
        const long long stride = 2 * a.H + a.E;
        const float *base = a.part + (long long)b * 2 * a.n_units * stride;
        auto piece = [&](int i) -> const float * {
            const int sid = 2 * (u0 + i) + ((i == 0 && beg != u0 * kUnitEdges) ? 1 : 0);
            return base + (long long)sid * stride;
        };
        // two passes over the pieces, loads unrolled so that several are in
        // flight: the maximum, then L and acc together (each summed in piece order)
        float Mh = -INFINITY;
#pragma unroll 4
        for (int i = 0; i < n_pieces; ++i) Mh = fmaxf(Mh, piece(i)[head]);
        const float mo = Mh == -INFINITY ? 0.f : Mh;
        float Lh = 0.f;
        f2 macc[NP];
#pragma unroll
        for (int j = 0; j < NP; ++j) macc[j] = 0ull;
#pragma unroll 2
        for (int i = 0; i < n_pieces; ++i) {
            const float *pp = piece(i);
            const float w = ex2(__fsub_rn(pp[head], mo));
            Lh = __fadd_rn(Lh, __fmul_rn(pp[a.H + head], w));
            if constexpr (WV) {
                const f2 w2 = pk(w, w);
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    const float2 v = reinterpret_cast<const float2 *>(pp + 2 * a.H + c0)[j];
                    macc[j] = ffma2(pk(v.x, v.y), w2, macc[j]);
                }
            }
        }
        if (a.ml && head_leader) {
            float *q = a.ml + (((long long)b * a.L + t) * a.H + head) * 2;
            q[0] = Mh;
            q[1] = Lh;
        }
        if constexpr (WV) {
            const float inv = Lh > 0.f ? __frcp_rn(Lh) : 0.f;
            const f2 inv2 = pk(inv, inv);
            f2 o[NP];
#pragma unroll
            for (int j = 0; j < NP; ++j) o[j] = fmul2(macc[j], inv2);
            store_row<T, CPL>((T *)a.mixed + ((long long)b * a.L + t) * a.E + c0, o);
        }
    };

    // finish target t in this unit: a complete target writes its result, a
    // target crossing a unit boundary its partial state
    auto finish = [&]() {
        const bool complete = (is_first ? first_started_here : true) && bound <= e1;
        if (complete) {
            if constexpr (WV) {
                const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
                const f2 inv2 = pk(inv, inv);
                f2 o[NP];
#pragma unroll
                for (int j = 0; j < NP; ++j) o[j] = fmul2(acc2[j], inv2);
                store_row<T, CPL>((T *)a.mixed + ((long long)b * a.L + t) * a.E + c0, o);
            }
            if (a.ml && head_leader) {
                float *p = a.ml + (((long long)b * a.L + t) * a.H + head) * 2;
                p[0] = m;
                p[1] = l;
            }
        } else {
            const int slot_id = 2 * u + (is_first ? 0 : 1);
            float *p = a.part + ((long long)b * 2 * a.n_units + slot_id) * (2 * a.H + a.E);
            if (head_leader) {
                p[head] = m;
                p[a.H + head] = l;
            }
            if constexpr (WV) {
#pragma unroll
                for (int j = 0; j < NP; ++j) reinterpret_cast<float2 *>(p + 2 * a.H + c0)[j] = upk(acc2[j]);
            }
            // The slot that writes a target's last piece merges all its
            // pieces: each writer publishes its piece (fence) and counts it;
            // the one that completes the count reads every piece in piece order.
            {
            __threadfence();
            __syncwarp(smask);
            const int beg = a.row_ptr[t], end = a.row_ptr[t + 1];
            const int u0 = beg / kUnitEdges, n_pieces = (end - 1) / kUnitEdges - u0 + 1;
            int prev = 0;
            if (grp == 0) prev = atomicAdd(a.counters + (long long)b * a.n_merge + a.merge_pos[t], 1);
            prev = __shfl_sync(smask, prev, 0, LPE);
            if (prev == n_pieces - 1) {
                __threadfence();
                merge_pieces(beg, u0, n_pieces);
            }
            }
        }
    };
    // move from t to the target of position pos (> the end of t)
    auto advance = [&](int pos) {
        finish();
        is_first = false;
        const int t_prev = t;
        do {
            ++t;
            bound = end_of(t);
        } while (bound <= pos);
        set_q(t == t_prev + 1 ? qnext : ldg_raw<CB>(Qb + (long long)t * a.q_ld));
        qnext = ldg_raw<CB>(Qb + (long long)min(t + 1, a.L - 1) * a.q_ld);
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int i = 0; i < NP; ++i) acc2[i] = 0ull;
    };
    // the head's score of one staged k row (two independent partial sums)
    auto score = [&](const Raw<CB> &kr) -> float {
        float dot;
        if constexpr (kMixed) {
            float ax = 0.f, ay = 0.f, bx = 0.f, by = 0.f;
#pragma unroll
            for (int i = 0; i < NP; i += 2) {
                fma_h2(ax, ay, qr.w[i], kr.w[i]);
                if (i + 1 < NP) fma_h2(bx, by, qr.w[i + 1], kr.w[i + 1]);
            }
            dot = __fadd_rn(__fadd_rn(ax, bx), __fadd_rn(ay, by));
        } else {
            f2 k2[NP];
            widen2<T, CPL>(kr, k2);
            f2 da = 0ull, db = 0ull;
#pragma unroll
            for (int i = 0; i < NP; i += 2) {
                da = ffma2(q2[i], k2[i], da);
                if (i + 1 < NP) db = ffma2(q2[i + 1], k2[i + 1], db);
            }
            const float2 fa = upk(da), fb = upk(db);
            dot = __fadd_rn(__fadd_rn(fa.x, fb.x), __fadd_rn(fa.y, fb.y));
        }
        for (int o = 1; o < lph; o <<= 1) dot = __fadd_rn(dot, __shfl_xor_sync(smask, dot, o, LPE));
        if constexpr (kMixed) dot = __fmul_rn(dot, a.score_scale);
        return dot;
    };
    auto mix = [&](const Raw<CB> &vr, float p) {
        f2 v2[NP];
        widen2<T, CPL>(vr, v2);
        const f2 p2 = pk(p, p);
#pragma unroll
        for (int i = 0; i < NP; ++i) acc2[i] = ffma2(p2, v2[i], acc2[i]);
    };
    auto rescale = [&](float scale) {
        const f2 s2 = pk(scale, scale);
#pragma unroll
        for (int i = 0; i < NP; ++i) acc2[i] = fmul2(acc2[i], s2);
    };
    // Move the reference m to mx where mx > m + kLazy (m = -inf: any finite
    // mx), rescaling l and acc; the vote keeps the branch uniform over the warp.
    auto lift = [&](float mx) {
        const bool move = mx > __fadd_rn(m, kLazy);
        if (__any_sync(live, move)) {
            const float scale = !move ? 1.f : (m == -INFINITY ? 0.f : ex2(__fsub_rn(m, mx)));
            l = __fmul_rn(l, scale);
            if constexpr (WV) rescale(scale);
            if (move) m = mx;
        }
    };
    // one edge through the online softmax (used at target boundaries); its
    // v row is read from stage address vst once the score is known
    auto one = [&](int j, const Raw<CB> &kr, uint32_t vst) {
        const int pos = e0 + j;
        if (pos >= bound) advance(pos);
        float dot = score(kr);
        Raw<CB> vr;
        if constexpr (WV) vr = lds_raw<CB>(vst);
        if constexpr (KPM)
            if (masked(j)) dot = -INFINITY;
        if constexpr (WS) {
            if (head_leader) scores_b[(long long)(e0 + j) * a.H + head] = dot;
        }
        lift(dot);
        // ex2.approx(-inf) is +0, so a dropped edge gives p = 0 once some key
        // is live; before that m is -inf and the offset 0 avoids -inf - -inf
        const float p = ex2(__fsub_rn(dot, (KPM && m == -INFINITY) ? 0.f : m));
        l = __fadd_rn(l, p);
        if constexpr (WV) mix(vr, p);
    };

    // rs = j mod kRing, stepped by 2 with a wrap (no division in the loop);
    // edge j + kDepth goes to stage (rs + kDepth) mod kRing = the stage read
    // one step earlier
    int rs = 0;
    for (int j = 0; j < n; j += 2) {
        cp_async_wait<kDepth / 2 - 1>();
        if constexpr (kLineCopy) __syncwarp(live);  // the other lanes' chunks of these rows
        const uint32_t st0 = sbase + (uint32_t)(rs * STAGE);
        const uint32_t st1 = st0 + (uint32_t)STAGE;
        const Raw<CB> kr0 = lds_raw<CB>(st0);
        const Raw<CB> kr1 = lds_raw<CB>(st1);
        // the v rows are read after the scores (fewer live registers; the
        // softmax covers the load latency). Stages st0 and st1 are refilled
        // only by the next step's issue2.
        issue2(j + kDepth, rs == 0 ? kRing - 2 : rs - 2);
        rs = rs + 2 == kRing ? 0 : rs + 2;

        const int pos = e0 + j;
        if (j + 1 < n && pos + 1 < bound) {
            // both edges belong to t: two independent scores, one rescale
            float d0 = score(kr0), d1 = score(kr1);
            Raw<CB> vr0, vr1;
            if constexpr (WV) {
                vr0 = lds_raw<CB>(st0 + 32 * CB);
                vr1 = lds_raw<CB>(st1 + 32 * CB);
            }
            if constexpr (KPM) {
                if (masked(j)) d0 = -INFINITY;
                if (masked(j + 1)) d1 = -INFINITY;
            }
            if constexpr (WS) {
                if (head_leader) {
                    scores_b[(long long)(e0 + j) * a.H + head] = d0;
                    scores_b[(long long)(e0 + j + 1) * a.H + head] = d1;
                }
            }
            lift(fmaxf(d0, d1));
            const float m_off = (KPM && m == -INFINITY) ? 0.f : m;
            const float p0 = ex2(__fsub_rn(d0, m_off));
            const float p1 = ex2(__fsub_rn(d1, m_off));
            l = __fadd_rn(__fadd_rn(l, p0), p1);
            if constexpr (WV) {
                mix(vr0, p0);
                mix(vr1, p1);
            }
        } else {
            one(j, kr0, st0 + 32 * CB);
            if (j + 1 < n) one(j + 1, kr1, st1 + 32 * CB);
        }
    }
    cp_async_wait<0>();
    finish();
}

// Instantiated in edge_attn_f16.cu / edge_attn_f32.cu.
template <typename T, int CPL, int LPE, bool WV>
pmha_status launch(const Args &k, long long slots, cudaStream_t s)
{
    constexpr int smem = smem_bytes<T, CPL, WV>();
    constexpr int P = 32 / LPE;
    const long long warps = (k.B + P - 1) / P * k.n_units;
    const long long blocks = (warps + kWarps - 1) / kWarps;
    (void)slots;
    auto kern = k.kpm ? (k.scores ? k_edge_stream<T, CPL, LPE, WV, true, true>
                                  : k_edge_stream<T, CPL, LPE, WV, false, true>)
                      : (k.scores ? k_edge_stream<T, CPL, LPE, WV, true, false>
                                  : k_edge_stream<T, CPL, LPE, WV, false, false>);
    if constexpr (smem > 48 * 1024) {
        PMHA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    }
    kern<<<(unsigned)blocks, kWarps * 32, smem, s>>>(k);
    return PMHA_OK;
}

template <typename T, int CPL, bool WV>
pmha_status launch_lpe(int lpe, const Args &k, long long slots, cudaStream_t s)
{
    switch (lpe) {
    case 2: return launch<T, CPL, 2, WV>(k, slots, s);
    case 4: return launch<T, CPL, 4, WV>(k, slots, s);
    case 8: return launch<T, CPL, 8, WV>(k, slots, s);
    case 16: return launch<T, CPL, 16, WV>(k, slots, s);
    case 32: return launch<T, CPL, 32, WV>(k, slots, s);
    default: return PMHA_ERR_UNSUPPORTED;
    }
}

// Entry points of the two instantiating translation units.
pmha_status launch_f16(int cpl, int lpe, bool wv, const Args &k, long long slots, cudaStream_t s);
pmha_status launch_f32(int cpl, int lpe, bool wv, const Args &k, long long slots, cudaStream_t s);

}  // namespace stream
}  // namespace pmha
