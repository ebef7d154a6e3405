// Streaming variants of the per-edge backward kernels (chain rule of kpnn2
// PackedMultiheadAttention, Notes steps 2-4) for fp16 intermediates with 8
// or 16 channels per lane. Same walk, arguments and outputs as k_bwd_dq /
// k_bwd_dkv in backward.cu; the rows gathered per edge go through a per-lane
// ring of shared-memory stages filled by cp.async kDepth edges ahead (so the
// loads in flight hold no registers), and the arithmetic runs on paired fp32
// FMAs (fma.rn.f32x2) over half2-widened channels.
//
//   dq  (per-target view): per edge the source's k and v rows
//   dkv (per-source view): per edge the target's q and dmixed rows and its
//       (m, l) and D for the lane's head
// Included by backward.cu after WalkArgs and head_sum_rt.
#pragma once

#include "edge_stream.cuh"

namespace pmha {
namespace bwds {
using stream::cp_async;
using stream::cp_async_commit;
using stream::cp_async_wait;
using stream::f2;
using stream::ffma2;
using stream::lds_raw;
using stream::pk;
using stream::Raw;
using stream::upk;
using stream::widen2;

#ifndef PMHA_BWDS_DEPTH
#define PMHA_BWDS_DEPTH 4
#endif
#ifndef PMHA_BWDS_WARPS
#define PMHA_BWDS_WARPS 2
#endif
#ifndef PMHA_BWDS_MINB
#define PMHA_BWDS_MINB 1
#endif
constexpr int kDepth = PMHA_BWDS_DEPTH;  // edges in flight per lane
constexpr int kRing = kDepth + 1;        // stages: the one read and the kDepth being filled
constexpr int kWarps = PMHA_BWDS_WARPS;  // warps per block
constexpr int kMinBlocks = PMHA_BWDS_MINB;  // resident blocks per SM the register budget aims at

template <int CPL>
__device__ __forceinline__ float dot2(const f2 (&x)[CPL / 2], const f2 (&y)[CPL / 2])
{
    f2 da = 0ull, db = 0ull;
#pragma unroll
    for (int i = 0; i < CPL / 2; i += 2) {
        da = ffma2(x[i], y[i], da);
        if (i + 1 < CPL / 2) db = ffma2(x[i + 1], y[i + 1], db);
    }
    const float2 fa = upk(da), fb = upk(db);
    return __fadd_rn(__fadd_rn(fa.x, fb.x), __fadd_rn(fa.y, fb.y));
}

template <int CPL>
__device__ __forceinline__ void load_widen(const __half *p, f2 (&out)[CPL / 2])
{
    constexpr int CB = CPL * 2;
    Raw<CB> r;
#pragma unroll
    for (int i = 0; i < CB / 16; ++i) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p) + i);
        r.w[4 * i] = u.x;
        r.w[4 * i + 1] = u.y;
        r.w[4 * i + 2] = u.z;
        r.w[4 * i + 3] = u.w;
    }
    widen2<__half, CPL>(r, out);
}

// dq over the per-target view: per edge the k and v rows of the source.
template <int CPL, int LPE>
__global__ void __launch_bounds__(kWarps * 32, kMinBlocks) k_bwd_dq_s(WalkArgs a)
{
    constexpr int P = 32 / LPE, CB = CPL * 2, NP = CPL / 2;
    constexpr int STG = 2 * 32 * CB;  // one stage of one warp: 32 lanes' k pieces, then their v pieces
    __shared__ __align__(16) unsigned char ring[kWarps][kRing][STG];
    __shared__ int sidx[kWarps][kUnitEdges];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int slot = lane / LPE, grp = lane % LPE;
    const long long gw = (long long)blockIdx.x * kWarps + wib;
    const long long groups = (a.B + P - 1) / P;
    if (gw >= groups * a.n_units) return;
    const int u = (int)(gw % a.n_units);
    const int b0 = (int)(gw / a.n_units) * P;
    const int b = min(b0 + slot, a.B - 1);
    const bool live_slot = b0 + slot < a.B;
    const int e0 = u * kUnitEdges;
    const int e1 = (int)min((long long)e0 + kUnitEdges, a.nnz);
    const int c0 = grp * CPL;
    const int d = a.E / a.H, head = c0 / d, lph = d / CPL > 1 ? d / CPL : 1;
    const __half *Q = (const __half *)a.q + (long long)b * a.L * a.q_ld + c0;
    const __half *G = (const __half *)a.g + (long long)b * a.L * a.E + c0;
    const __half *K = (const __half *)a.k + (long long)b * a.S * a.kv_ld + c0;
    const __half *V = (const __half *)a.v + (long long)b * a.S * a.kv_ld + c0;
    const uint8_t *kpm = a.kpm ? a.kpm + (long long)b * a.S : nullptr;
    for (int p = e0 + lane; p < e1; p += 32) sidx[wib][p - e0] = a.idx[p];
    __syncwarp();

    const uint32_t sbase = stream::smem_u32(&ring[wib][0][lane * CB]);
    // edge p (absolute position) into stage st; one commit group per edge, empty past the unit
    auto issue = [&](int p, int st) {
        if (p < e1) {
            const long long s = sidx[wib][p - e0];
            const uint32_t dst = sbase + (uint32_t)(st * STG);
            cp_async<CB>(dst, K + s * a.kv_ld);
            cp_async<CB>(dst + 32 * CB, V + s * a.kv_ld);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kDepth; ++j) issue(e0 + j, j);

    int t = a.unit_first[u];
    const bool first_started_here = a.row_ptr[t] == e0;
    bool is_first = true;
    int bound = a.row_ptr[t + 1];
    f2 q2[NP], g2[NP], acc[NP];
    float m = 0.f, inv_l = 0.f, Dt = 0.f;
    auto load_row = [&]() {
        load_widen<CPL>(Q + (long long)t * a.q_ld, q2);
        load_widen<CPL>(G + (long long)t * a.E, g2);
#pragma unroll
        for (int i = 0; i < NP; ++i) acc[i] = 0ull;
        const long long st = ((long long)b * a.L + t) * a.H + head;
        m = a.ml[2 * st];
        const float l = a.ml[2 * st + 1];
        inv_l = l > 0.f ? __frcp_rn(l) : 0.f;
        Dt = a.D[st];
    };
    auto finish = [&]() {
        const bool complete = (is_first ? first_started_here : true) && bound <= e1;
        if (!live_slot) return;
        float *o = complete ? a.out0 + ((long long)b * a.L + t) * a.E + c0
                            : a.part + ((long long)b * 2 * a.n_units + 2 * u + (is_first ? 0 : 1)) * a.E + c0;
        const f2 sc = pk(a.inv_sqrt_d, a.inv_sqrt_d);
#pragma unroll
        for (int i = 0; i < NP; ++i) reinterpret_cast<float2 *>(o)[i] = upk(stream::fmul2(acc[i], sc));
    };
    load_row();
    int rd = 0, wr = kDepth;  // ring stage read this edge / filled next
    for (int p = e0; p < e1; ++p) {
        if (p >= bound) {
            finish();
            is_first = false;
            do {
                ++t;
                bound = a.row_ptr[t + 1];
            } while (bound <= p);
            load_row();
        }
        cp_async_wait<kDepth - 1>();  // edge p's rows have landed (this lane's own copies)
        const uint32_t src = sbase + (uint32_t)(rd * STG);
        const Raw<CB> kr = lds_raw<CB>(src);
        const Raw<CB> vr = lds_raw<CB>(src + 32 * CB);
        const bool drop = kpm && kpm[sidx[wib][p - e0]];
        issue(p + kDepth, wr);
        rd = rd + 1 == kRing ? 0 : rd + 1;
        wr = wr + 1 == kRing ? 0 : wr + 1;
        f2 k2[NP], v2[NP];
        widen2<__half, CPL>(kr, k2);
        widen2<__half, CPL>(vr, v2);
        float d1 = dot2<CPL>(q2, k2), d2 = dot2<CPL>(g2, v2);
        d1 = head_sum_rt(d1, lph);
        d2 = head_sum_rt(d2, lph);
        // a dropped key (key_padding_mask) has weight 0
        const float w =
            (inv_l > 0.f && !drop) ? __fmul_rn(stream::ex2(__fsub_rn(__fmul_rn(d1, a.score_scale), m)), inv_l) : 0.f;
        const float ds = __fmul_rn(w, __fsub_rn(d2, Dt));
        const f2 ds2 = pk(ds, ds);
#pragma unroll
        for (int i = 0; i < NP; ++i) acc[i] = ffma2(ds2, k2[i], acc[i]);
    }
    cp_async_wait<0>();
    finish();
}

// dk and dv over the per-source view: per edge the target's q and dmixed
// rows and its (m, l) and D for the lane's head.
template <int CPL, int LPE>
__global__ void __launch_bounds__(kWarps * 32, kMinBlocks) k_bwd_dkv_s(WalkArgs a)
{
    constexpr int P = 32 / LPE, CB = CPL * 2, NP = CPL / 2;
    constexpr int STG = 32 * (2 * CB + 16);  // one stage of one warp: q pieces, dmixed pieces, {m, l, D, -}
    __shared__ __align__(16) unsigned char ring[kWarps][kRing][STG];
    __shared__ int sidx[kWarps][kUnitEdges];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int slot = lane / LPE, grp = lane % LPE;
    const long long gw = (long long)blockIdx.x * kWarps + wib;
    const long long groups = (a.B + P - 1) / P;
    if (gw >= groups * a.n_units) return;
    const int u = (int)(gw % a.n_units);
    const int b0 = (int)(gw / a.n_units) * P;
    const int b = min(b0 + slot, a.B - 1);
    const bool live_slot = b0 + slot < a.B;
    const int e0 = u * kUnitEdges;
    const int e1 = (int)min((long long)e0 + kUnitEdges, a.nnz);
    const int c0 = grp * CPL;
    const int d = a.E / a.H, head = c0 / d, lph = d / CPL > 1 ? d / CPL : 1;
    const __half *Q = (const __half *)a.q + (long long)b * a.L * a.q_ld + c0;
    const __half *G = (const __half *)a.g + (long long)b * a.L * a.E + c0;
    const __half *K = (const __half *)a.k + (long long)b * a.S * a.kv_ld + c0;
    const __half *V = (const __half *)a.v + (long long)b * a.S * a.kv_ld + c0;
    const float *ML = a.ml + (long long)b * a.L * a.H * 2 + 2 * head;
    const float *DD = a.D + (long long)b * a.L * a.H + head;
    const uint8_t *kpm = a.kpm ? a.kpm + (long long)b * a.S : nullptr;
    for (int p = e0 + lane; p < e1; p += 32) sidx[wib][p - e0] = a.idx[p];
    __syncwarp();

    const uint32_t sbase = stream::smem_u32(&ring[wib][0][0]);
    const uint32_t q_off = (uint32_t)(lane * CB), g_off = (uint32_t)(32 * CB + lane * CB),
                   s_off = (uint32_t)(64 * CB + lane * 16);
    // edge p (absolute position) into stage st; one commit group per edge, empty past the unit
    auto issue = [&](int p, int st) {
        if (p < e1) {
            const long long t = sidx[wib][p - e0];
            const uint32_t dst = sbase + (uint32_t)(st * STG);
            cp_async<CB>(dst + q_off, Q + t * a.q_ld);
            cp_async<CB>(dst + g_off, G + t * a.E);
            cp_async<8>(dst + s_off, ML + t * a.H * 2);
            cp_async<4>(dst + s_off + 8, DD + t * a.H);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kDepth; ++j) issue(e0 + j, j);

    int s = a.unit_first[u];
    const bool first_started_here = a.row_ptr[s] == e0;
    bool is_first = true;
    int bound = a.row_ptr[s + 1];
    bool dropped = false;
    f2 k2[NP], v2[NP], ak[NP], av[NP];
    auto load_row = [&]() {
        dropped = kpm && kpm[s];
        load_widen<CPL>(K + (long long)s * a.kv_ld, k2);
        load_widen<CPL>(V + (long long)s * a.kv_ld, v2);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            ak[i] = 0ull;
            av[i] = 0ull;
        }
    };
    auto finish = [&]() {
        const bool complete = (is_first ? first_started_here : true) && bound <= e1;
        if (!live_slot) return;
        float *ok, *ov;
        if (complete) {
            ok = a.out0 + ((long long)b * a.S + s) * a.E + c0;
            ov = a.out1 + ((long long)b * a.S + s) * a.E + c0;
        } else {
            ok = a.part + ((long long)b * 2 * a.n_units + 2 * u + (is_first ? 0 : 1)) * 2 * a.E + c0;
            ov = ok + a.E;
        }
        const f2 sc = pk(a.inv_sqrt_d, a.inv_sqrt_d);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            reinterpret_cast<float2 *>(ok)[i] = upk(stream::fmul2(ak[i], sc));
            reinterpret_cast<float2 *>(ov)[i] = upk(av[i]);
        }
    };
    load_row();
    int rd = 0, wr = kDepth;  // ring stage read this edge / filled next
    for (int p = e0; p < e1; ++p) {
        if (p >= bound) {
            finish();
            is_first = false;
            do {
                ++s;
                bound = a.row_ptr[s + 1];
            } while (bound <= p);
            load_row();
        }
        cp_async_wait<kDepth - 1>();  // edge p's rows have landed (this lane's own copies)
        const uint32_t src = sbase + (uint32_t)(rd * STG);
        const Raw<CB> qr = lds_raw<CB>(src + q_off);
        const Raw<CB> gr = lds_raw<CB>(src + g_off);
        float m, l, Dt;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(m), "=f"(l) : "r"(src + s_off));
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(Dt) : "r"(src + s_off + 8));
        issue(p + kDepth, wr);
        rd = rd + 1 == kRing ? 0 : rd + 1;
        wr = wr + 1 == kRing ? 0 : wr + 1;
        f2 q2[NP], g2[NP];
        widen2<__half, CPL>(qr, q2);
        widen2<__half, CPL>(gr, g2);
        float d1 = dot2<CPL>(q2, k2), d2 = dot2<CPL>(g2, v2);
        d1 = head_sum_rt(d1, lph);
        d2 = head_sum_rt(d2, lph);
        // every edge of a dropped key (key_padding_mask) has weight 0
        const float w = (l > 0.f && !dropped)
                            ? __fmul_rn(stream::ex2(__fsub_rn(__fmul_rn(d1, a.score_scale), m)), __frcp_rn(l))
                            : 0.f;
        const float ds = __fmul_rn(w, __fsub_rn(d2, Dt));
        const f2 ds2 = pk(ds, ds), w2 = pk(w, w);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            ak[i] = ffma2(ds2, q2[i], ak[i]);
            av[i] = ffma2(w2, g2[i], av[i]);
        }
    }
    cp_async_wait<0>();
    finish();
}

}  // namespace bwds
}  // namespace pmha
