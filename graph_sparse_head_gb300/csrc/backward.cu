// Backward pass of the layer: the chain rule of kpnn2 PackedMultiheadAttention,
// Notes steps 1-5, given dL/d(output). Like the page's training path it
// recomputes the forward instead of keeping per-edge tensors: the caller's
// inputs are projected again, the edge kernel gives each target's softmax
// statistics (m, l) and its mix, and every per-edge weight is recomputed
// from those when needed.
//
//   step 5   dmixed = dout Wo;  dWo = dout^T mixed;  dbo = sum dout
//   steps 2-4, for each live edge e = (s -> t) and head h, with
//            w_e = 2^(s_e - m_t) / l_t and D_t = dot(dmixed_t, mixed_t)
//            (= sum_e w_e dw_e, since mixed_t = sum_e w_e v_s):
//              dw_e = dot(dmixed_t, v_s),  ds_e = w_e (dw_e - D_t)
//              dq_t += ds_e k_s / sqrt(d)  (a sum over the edges INTO t)
//              dk_s += ds_e q_t / sqrt(d)  (a sum over the edges OUT of s)
//              dv_s += w_e dmixed_t        (likewise)
//            Both sums are segmented reductions without atomics: dq walks
//            the per-target view, dk and dv the per-source view, each in
//            units of kUnitEdges positions; a row that crosses a unit
//            boundary leaves partial sums that an ordered merge adds up.
//   step 1   dX = dq Wq (+ dk Wk + dv Wv for one shared input tensor),
//            dWq = dq^T Xq, dbq = sum dq, likewise for k and v.
// All sums run in a fixed order: results are deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "pmha_internal.h"

namespace pmha {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------- D = dot(dmixed, mixed) per (row, head)
// One thread per (row, head): the head's d channels of both rows come in as
// 16-byte vectors (consecutive threads read consecutive heads, so a warp
// reads whole rows); products are rounded and summed in channel order.
template <typename T>
__device__ __forceinline__ void widen16(const uint4 &u, float (&f)[16 / sizeof(T)]);
template <>
__device__ __forceinline__ void widen16<__half>(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}
template <>
__device__ __forceinline__ void widen16<float>(const uint4 &u, float (&f)[4])
{
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}

template <typename T>
__global__ void __launch_bounds__(256) k_rowdot(const T *__restrict__ dmixed, const T *__restrict__ mixed,
                                                long long rows, int E, int H, float *__restrict__ D,
                                                const float *__restrict__ ml, float2 *__restrict__ rec)
{
    constexpr int PER = 16 / (int)sizeof(T);  // channels per vector
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // row * H + head
    if (i >= rows * H) return;
    const int d = E / H;
    const long long r = i / H;
    const int h = (int)(i - r * H);
    const T *gs = dmixed + r * E + (long long)h * d, *os = mixed + r * E + (long long)h * d;
    float acc = 0.f;
    if (d % PER) {  // heads narrower than a vector (float32 heads of 1 or 2 channels)
        for (int c = 0; c < d; ++c) acc = __fadd_rn(acc, __fmul_rn(to_f(gs[c]), to_f(os[c])));
    } else {
        const uint4 *g = reinterpret_cast<const uint4 *>(gs);
        const uint4 *o = reinterpret_cast<const uint4 *>(os);
        for (int v = 0; v < d / PER; ++v) {
            float fg[PER], fo[PER];
            widen16<T>(__ldg(g + v), fg);
            widen16<T>(__ldg(o + v), fo);
#pragma unroll
            for (int c = 0; c < PER; ++c) acc = __fadd_rn(acc, __fmul_rn(fg[c], fo[c]));
        }
    }
    D[i] = acc;
    if (rec) {  // the ring kernels' record of (row, head): w = 2^(s - c) with c = m + log2(l)
        const float2 s = reinterpret_cast<const float2 *>(ml)[i];
        rec[i] = make_float2(s.y > 0.f ? __fadd_rn(s.x, log2f(s.y)) : INFINITY, acc);
    }
}

struct WalkArgs {
    const void *q;    // (B, L) rows of pitch q_ld (intermediate type)
    long long q_ld;
    const void *k;    // (B, S) rows of pitch kv_ld
    const void *v;
    long long kv_ld;
    const void *g;    // dmixed (B, L, E), intermediate type
    const float *ml;  // (B, L, H, 2): m (log2 units), l
    const float *D;   // (B, L, H)
    const uint8_t *kpm;
    const int32_t *row_ptr, *idx, *unit_first;  // the walked view: row pointers, the other end, unit plan
    long long n_units, nnz;
    int B, L, S, E, H, n_rows;  // n_rows: rows of the walked view (L for dq, S for dk/dv)
    float score_scale;          // log2(e) / sqrt(d)
    float inv_sqrt_d;
    float *out0, *out1;   // dq (B, L, E) | dk, dv (B, S, E)
    float *part;          // (B, 2 n_units, W) partial sums of rows crossing a unit boundary
};

// Sum over the lanes of one head (LPH lanes, aligned groups).
template <int LPH>
__device__ __forceinline__ float head_sum(float x)
{
#pragma unroll
    for (int o = 1; o < LPH; o <<= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

#ifndef PMHA_BWD_PF
#define PMHA_BWD_PF 1
#endif
#ifndef PMHA_BWD_WARPS
#define PMHA_BWD_WARPS 4
#endif
constexpr int kBwdWarps = PMHA_BWD_WARPS;  // warps per block of the per-edge kernels
constexpr int kPF = PMHA_BWD_PF;           // edges ahead in flight per slot (raw rows in registers)

// A lane's CPL channels of one row, loaded as raw words (one vector load)
// and converted to float only when used, so a prefetch does not wait.
template <typename T, int CPL>
struct RawRow {
    static constexpr int kBytes = CPL * (int)sizeof(T);
    static constexpr int kWords = kBytes >= 4 ? kBytes / 4 : 1;
    uint32_t w[kWords];
    __device__ __forceinline__ void load(const T *p, bool act)
    {
        if (!act) {
#pragma unroll
            for (int i = 0; i < kWords; ++i) w[i] = 0u;
            return;
        }
        if constexpr (kBytes % 16 == 0) {
#pragma unroll
            for (int i = 0; i < kBytes / 16; ++i) {
                const uint4 v = *reinterpret_cast<const uint4 *>(reinterpret_cast<const char *>(p) + 16 * i);
                w[4 * i] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
            }
        } else if constexpr (kBytes == 8) {
            const uint2 v = *reinterpret_cast<const uint2 *>(p);
            w[0] = v.x;
            w[1] = v.y;
        } else if constexpr (kBytes == 4) {
            w[0] = *reinterpret_cast<const uint32_t *>(p);
        } else {
            w[0] = *reinterpret_cast<const unsigned short *>(p);
        }
    }
    __device__ __forceinline__ float at(int c) const
    {
        if constexpr (sizeof(T) == 4) {
            return __uint_as_float(w[c]);
        } else {
            const unsigned short h = (unsigned short)(w[c >> 1] >> ((c & 1) * 16));
            return to_f(*reinterpret_cast<const T *>(&h));
        }
    }
};

// Sum over the lph lanes of one head (aligned groups inside a slot).
__device__ __forceinline__ float head_sum_rt(float x, int lph)
{
    for (int o = 1; o < lph; o <<= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

}  // namespace
}  // namespace pmha

#include "bwd_stream.cuh"  // the streaming variants (fp16, 8 or 16 channels per lane)

namespace pmha {
namespace {

// The per-edge backward kernels. Like the forward's streaming kernel, a
// "slot" of LPE = E / CPL lanes owns one sample (a lane owns CPL channels),
// and the P = 32 / LPE slots of a warp walk the same unit of the view for P
// consecutive samples: the graph is shared, so their walks are identical.
// The unit's other-end indices are staged in shared memory; the rows of the
// next kPF edges are in flight in a register ring of raw words.
//
// dq: the per-target view; per edge it gathers k_s and v_s.
template <typename T, int CPL, int LPE>
__global__ void __launch_bounds__(kBwdWarps * 32) k_bwd_dq(WalkArgs a)
{
    constexpr int P = 32 / LPE;
    __shared__ int sidx[kBwdWarps][kUnitEdges];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int slot = lane / LPE, grp = lane % LPE;
    const long long gw = (long long)blockIdx.x * kBwdWarps + wib;
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
    const T *Q = (const T *)a.q + (long long)b * a.L * a.q_ld;
    const T *G = (const T *)a.g + (long long)b * a.L * a.E;
    const T *K = (const T *)a.k + (long long)b * a.S * a.kv_ld;
    const T *V = (const T *)a.v + (long long)b * a.S * a.kv_ld;
    const uint8_t *kpm = a.kpm ? a.kpm + (long long)b * a.S : nullptr;
    for (int p = e0 + lane; p < e1; p += 32) sidx[wib][p - e0] = a.idx[p];
    __syncwarp();

    RawRow<T, CPL> kr[kPF], vr[kPF];
    auto fetch = [&](RawRow<T, CPL> &kd, RawRow<T, CPL> &vd, int p) {
        if (p < e1) {
            const int s = sidx[wib][p - e0];
            kd.load(K + (long long)s * a.kv_ld + c0, true);
            vd.load(V + (long long)s * a.kv_ld + c0, true);
        }
    };
#pragma unroll
    for (int j = 0; j < kPF; ++j) fetch(kr[j], vr[j], e0 + j);

    int t = a.unit_first[u];
    const bool first_started_here = a.row_ptr[t] == e0;
    bool is_first = true;
    int bound = a.row_ptr[t + 1];
    float q[CPL], gv[CPL], acc[CPL], m = 0.f, inv_l = 0.f, Dt = 0.f;
    auto load_row = [&]() {
        RawRow<T, CPL> rq, rg;
        rq.load(Q + (long long)t * a.q_ld + c0, true);
        rg.load(G + (long long)t * a.E + c0, true);
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            q[c] = rq.at(c);
            gv[c] = rg.at(c);
            acc[c] = 0.f;
        }
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
#pragma unroll
        for (int c = 0; c < CPL; ++c) o[c] = __fmul_rn(acc[c], a.inv_sqrt_d);
    };
    load_row();
    for (int base = e0; base < e1; base += kPF) {
#pragma unroll
        for (int j = 0; j < kPF; ++j) {
            const int p = base + j;
            if (p >= e1) break;
            if (p >= bound) {
                finish();
                is_first = false;
                do {
                    ++t;
                    bound = a.row_ptr[t + 1];
                } while (bound <= p);
                load_row();
            }
            const int s = sidx[wib][p - e0];
            float kk[CPL], vv[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                kk[c] = kr[j].at(c);
                vv[c] = vr[j].at(c);
            }
            fetch(kr[j], vr[j], p + kPF);
            float d1 = 0.f, d2 = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                d1 = __fmaf_rn(q[c], kk[c], d1);
                d2 = __fmaf_rn(gv[c], vv[c], d2);
            }
            d1 = head_sum_rt(d1, lph);
            d2 = head_sum_rt(d2, lph);
            // a dropped key (key_padding_mask) has weight 0
            const bool drop = kpm && kpm[s];
            const float w =
                (inv_l > 0.f && !drop) ? __fmul_rn(ex2f(__fsub_rn(__fmul_rn(d1, a.score_scale), m)), inv_l) : 0.f;
            const float ds = __fmul_rn(w, __fsub_rn(d2, Dt));
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = __fmaf_rn(ds, kk[c], acc[c]);
        }
    }
    finish();
}

// dk and dv: the per-source view; per edge it gathers q_t, dmixed_t and the
// target's (m, l, D) of the lane's head.
template <typename T, int CPL, int LPE>
__global__ void __launch_bounds__(kBwdWarps * 32) k_bwd_dkv(WalkArgs a)
{
    constexpr int P = 32 / LPE;
    __shared__ int sidx[kBwdWarps][kUnitEdges];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int slot = lane / LPE, grp = lane % LPE;
    const long long gw = (long long)blockIdx.x * kBwdWarps + wib;
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
    const T *Q = (const T *)a.q + (long long)b * a.L * a.q_ld;
    const T *G = (const T *)a.g + (long long)b * a.L * a.E;
    const T *K = (const T *)a.k + (long long)b * a.S * a.kv_ld;
    const T *V = (const T *)a.v + (long long)b * a.S * a.kv_ld;
    const float *ML = a.ml + (long long)b * a.L * a.H * 2;
    const float *DD = a.D + (long long)b * a.L * a.H;
    const uint8_t *kpm = a.kpm ? a.kpm + (long long)b * a.S : nullptr;
    for (int p = e0 + lane; p < e1; p += 32) sidx[wib][p - e0] = a.idx[p];
    __syncwarp();

    RawRow<T, CPL> qr[kPF], gr[kPF];
    float mr[kPF], lr[kPF], dr[kPF];
    auto fetch = [&](RawRow<T, CPL> &qd, RawRow<T, CPL> &gd, float &md, float &ld, float &dd, int p) {
        if (p < e1) {
            const int t = sidx[wib][p - e0];
            qd.load(Q + (long long)t * a.q_ld + c0, true);
            gd.load(G + (long long)t * a.E + c0, true);
            const long long st = (long long)t * a.H + head;
            md = ML[2 * st];
            ld = ML[2 * st + 1];
            dd = DD[st];
        }
    };
#pragma unroll
    for (int j = 0; j < kPF; ++j) fetch(qr[j], gr[j], mr[j], lr[j], dr[j], e0 + j);

    int s = a.unit_first[u];
    const bool first_started_here = a.row_ptr[s] == e0;
    bool is_first = true;
    int bound = a.row_ptr[s + 1];
    bool dropped = false;
    float kk[CPL], vv[CPL], ak[CPL], av[CPL];
    auto load_row = [&]() {
        dropped = kpm && kpm[s];
        RawRow<T, CPL> rk, rv;
        rk.load(K + (long long)s * a.kv_ld + c0, true);
        rv.load(V + (long long)s * a.kv_ld + c0, true);
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            kk[c] = rk.at(c);
            vv[c] = rv.at(c);
            ak[c] = 0.f;
            av[c] = 0.f;
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
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            ok[c] = __fmul_rn(ak[c], a.inv_sqrt_d);
            ov[c] = av[c];
        }
    };
    load_row();
    for (int base = e0; base < e1; base += kPF) {
#pragma unroll
        for (int j = 0; j < kPF; ++j) {
            const int p = base + j;
            if (p >= e1) break;
            if (p >= bound) {
                finish();
                is_first = false;
                do {
                    ++s;
                    bound = a.row_ptr[s + 1];
                } while (bound <= p);
                load_row();
            }
            float qq[CPL], gg[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                qq[c] = qr[j].at(c);
                gg[c] = gr[j].at(c);
            }
            const float m = mr[j], l = lr[j], Dt = dr[j];
            fetch(qr[j], gr[j], mr[j], lr[j], dr[j], p + kPF);
            float d1 = 0.f, d2 = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                d1 = __fmaf_rn(qq[c], kk[c], d1);
                d2 = __fmaf_rn(gg[c], vv[c], d2);
            }
            d1 = head_sum_rt(d1, lph);
            d2 = head_sum_rt(d2, lph);
            // every edge of a dropped key (key_padding_mask) has weight 0
            const float w = (l > 0.f && !dropped)
                                ? __fmul_rn(ex2f(__fsub_rn(__fmul_rn(d1, a.score_scale), m)), __frcp_rn(l))
                                : 0.f;
            const float ds = __fmul_rn(w, __fsub_rn(d2, Dt));
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                ak[c] = __fmaf_rn(ds, qq[c], ak[c]);
                av[c] = __fmaf_rn(w, gg[c], av[c]);
            }
        }
    }
    finish();
}

// Rows of a view that cross a unit boundary, or have no edges: add the
// pieces in unit order (no edges: zeros). One warp per (sample, row);
// width W floats per piece, written to out (+ out1 for the second half
// when W = 2E).
__global__ void __launch_bounds__(256) k_bwd_merge(const int32_t *__restrict__ merge_rows, long long n_merge,
                                                   const int32_t *__restrict__ row_ptr, const float *__restrict__ part,
                                                   long long n_units, int B, int n_rows, int E, int W,
                                                   float *__restrict__ out0, float *__restrict__ out1)
{
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gw >= (long long)B * n_merge) return;
    const int b = (int)(gw / n_merge);
    const int r = merge_rows[gw - (long long)b * n_merge];
    const int beg = row_ptr[r], end = row_ptr[r + 1];
    const float *base = part + (long long)b * 2 * n_units * W;
    const int u0 = beg / kUnitEdges, n_pc = end > beg ? (end - 1) / kUnitEdges - u0 + 1 : 0;
    const int first_slot = 2 * u0 + (beg != u0 * kUnitEdges ? 1 : 0);  // piece 0; piece i > 0 is slot 2 (u0 + i)
    float *o0 = out0 + ((long long)b * n_rows + r) * E;
    float *o1 = out1 ? out1 + ((long long)b * n_rows + r) * E : nullptr;  // column c >= E goes to o1[c - E]
    if ((E & 3) == 0) {
        // four columns a lane (16-byte loads and stores; a group of four never straddles E)
        for (int c = 4 * lane; c < W; c += 128) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int i = 0; i < n_pc; ++i) {
                const int slot = i == 0 ? first_slot : 2 * (u0 + i);
                const float4 v = *reinterpret_cast<const float4 *>(base + (long long)slot * W + c);
                acc.x = __fadd_rn(acc.x, v.x);
                acc.y = __fadd_rn(acc.y, v.y);
                acc.z = __fadd_rn(acc.z, v.z);
                acc.w = __fadd_rn(acc.w, v.w);
            }
            *reinterpret_cast<float4 *>(c < E ? o0 + c : o1 + (c - E)) = acc;
        }
        return;
    }
    for (int c = lane; c < W; c += 32) {
        float acc = 0.f;
        for (int i = 0; i < n_pc; ++i) {
            const int slot = i == 0 ? first_slot : 2 * (u0 + i);
            acc = __fadd_rn(acc, base[(long long)slot * W + c]);
        }
        *(c < E ? o0 + c : o1 + (c - E)) = acc;
    }
}

// ---------------------------------------------------------------- CUDA-core GEMMs (fp32 accumulation)
// C (M x N, pitch ldc) (+)= A (M x K, pitch lda) . B (K x N, pitch ldb)
template <typename TA, typename TB, typename TC, bool ACC>
__global__ void __launch_bounds__(256) k_gemm_nn(const TA *__restrict__ A, long long lda, const TB *__restrict__ B,
                                                 long long ldb, TC *__restrict__ C, long long ldc, long long M, int N,
                                                 int K)
{
    __shared__ float As[16][68], Bs[16][68];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const long long m0 = (long long)blockIdx.x * 64;
    const int n0 = blockIdx.y * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int r = i / 16, c = i % 16;  // A tile: 64 rows x 16 k
            const long long gm = m0 + r;
            As[c][r] = (gm < M && k0 + c < K) ? to_f(A[gm * lda + k0 + c]) : 0.f;
            const int kr = i / 64, nc = i % 64;  // B tile: 16 k x 64 cols
            Bs[kr][nc] = (k0 + kr < K && n0 + nc < N) ? to_f(B[(long long)(k0 + kr) * ldb + n0 + nc]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = As[kk][ty + 16 * i];
                bv[i] = Bs[kk][tx + 16 * i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const long long gm = m0 + ty + 16 * i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gn = n0 + tx + 16 * j;
            if (gn >= N) continue;
            float v = acc[i][j];
            if (ACC) v = __fadd_rn(to_f(C[gm * ldc + gn]), v);
            C[gm * ldc + gn] = from_f<TC>(v);
        }
    }
}

// P[chunk] (K x N) = A[rows of chunk]^T . B[rows of chunk]; A (M x K), B (M x N).
// With B null, P[chunk] (K) = column sums of A over the chunk.
template <typename TA, typename TB>
__global__ void __launch_bounds__(256) k_gemm_tn_part(const TA *__restrict__ A, long long lda,
                                                      const TB *__restrict__ B, long long ldb, long long M, int K,
                                                      int N, long long rows_per_chunk, float *__restrict__ P)
{
    __shared__ float As[16][68], Bs[16][68];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int k0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
    const long long chunk = blockIdx.z;
    const long long r_beg = chunk * rows_per_chunk, r_end = min(M, r_beg + rows_per_chunk);
    float acc[4][4] = {};
    for (long long r0 = r_beg; r0 < r_end; r0 += 16) {
        for (int i = threadIdx.x; i < 16 * 64; i += 256) {
            const int rr = i / 64, cc = i % 64;
            const long long gr = r0 + rr;
            As[rr][cc] = (gr < r_end && k0 + cc < K) ? to_f(A[gr * lda + k0 + cc]) : 0.f;
            Bs[rr][cc] = (gr < r_end && n0 + cc < N) ? to_f(B[gr * ldb + n0 + cc]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = As[rr][ty + 16 * i];
                bv[i] = Bs[rr][tx + 16 * i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *out = P + chunk * (long long)K * N;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gk = k0 + ty + 16 * i;
        if (gk >= K) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gn = n0 + tx + 16 * j;
            if (gn < N) out[(long long)gk * N + gn] = acc[i][j];
        }
    }
}

template <typename TA>
__global__ void __launch_bounds__(256) k_colsum_part(const TA *__restrict__ A, long long lda, long long M, int K,
                                                     long long rows_per_chunk, float *__restrict__ P)
{
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const long long chunk = blockIdx.y;
    if (c >= K) return;
    const long long r_beg = chunk * rows_per_chunk, r_end = min(M, r_beg + rows_per_chunk);
    float acc = 0.f;
    for (long long r = r_beg; r < r_end; ++r) acc = __fadd_rn(acc, to_f(A[r * lda + c]));
    P[chunk * K + c] = acc;
}

// out[c] = sum over tiles of P[tile][c] (P has n columns); one block per c
__global__ void __launch_bounds__(256) k_sum_tiles(const float *__restrict__ P, long long n, int tiles,
                                                   float *__restrict__ out)
{
    __shared__ float red[256];
    const long long c = blockIdx.x;
    float acc = 0.f;
    for (int t = threadIdx.x; t < tiles; t += 256) acc = __fadd_rn(acc, P[(long long)t * n + c]);
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] = __fadd_rn(red[threadIdx.x], red[threadIdx.x + w]);
        __syncthreads();
    }
    if (threadIdx.x == 0) out[c] = red[0];
}

// out[i] = sum over chunks of P[chunk][i], in a fixed order
__global__ void __launch_bounds__(256) k_sum_chunks(const float *__restrict__ P, long long n, int chunks,
                                                    float *__restrict__ out)
{
    // out[i] = sum over c of P[c * n + i]. Eight warps share 32 consecutive
    // outputs: warp g adds the g-th eighth of the chunks in chunk order
    // (sixteen loads in flight at a time), then warp 0 adds the eight sums in
    // order. A fixed order, so the result is deterministic; a single thread
    // per output made this pass a chain of dependent L2 round trips.
    __shared__ float part[8][32];
    const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
    const long long i = (long long)blockIdx.x * 32 + lane;
    const int per = (chunks + 7) / 8, c_lo = min(chunks, g * per), c_hi = min(chunks, c_lo + per);
    float acc = 0.f;
    if (i < n) {
        int c = c_lo;
        for (; c + 16 <= c_hi; c += 16) {
            float v[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = P[(long long)(c + q) * n + i];
#pragma unroll
            for (int q = 0; q < 16; ++q) acc = __fadd_rn(acc, v[q]);
        }
        for (; c < c_hi; ++c) acc = __fadd_rn(acc, P[(long long)c * n + i]);
    }
    part[g][lane] = acc;
    __syncthreads();
    if (g == 0 && i < n) {
        float t = part[0][lane];
#pragma unroll
        for (int q = 1; q < 8; ++q) t = __fadd_rn(t, part[q][lane]);
        out[i] = t;
    }
}

template <typename TO>
__global__ void k_convert(const float *__restrict__ in, long long n, TO *__restrict__ out)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = from_f<TO>(in[i]);
}

// out[c * ld_out + r] = in[r * ld_in + c] for r < M, c < E (converted to a
// 16-bit type); the columns r in [M, Mpad) of out are zero. 64 x 64 tiles
// through shared memory, 16-byte global loads and stores: a thread loads
// 16-byte pieces of input rows and stores 8 consecutive r of one output row.
// With colsum non-null, also writes the tile's 64-row column sums of the
// input (in row order) to colsum[blockIdx.x * E + c]. With rows16 non-null,
// also writes the input rows in fp16, untransposed (pitch ld16).
// Shapes (checked by transpose_cvt): E and Mpad multiples of 64; ld_in,
// ld_out and ld16 multiples of 8 elements; every pointer 16-byte aligned.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256) k_transpose_cvt(const TIn *__restrict__ in, long long ld_in, long long M, int E,
                                                       long long Mpad, TOut *__restrict__ out, long long ld_out,
                                                       float *__restrict__ colsum, __half *__restrict__ rows16,
                                                       long long ld16)
{
    static_assert(sizeof(TOut) == 2, "16-bit outputs");
    constexpr int V = 16 / (int)sizeof(TIn);  // elements per 16-byte load: 4 (fp32) or 8
    constexpr int TPR = 64 / V;              // threads per tile row
    constexpr int RPP = 256 / TPR;           // tile rows per pass
    constexpr int NP = 64 / RPP;             // passes
    __shared__ float tile[64][65];
    const long long r0 = (long long)blockIdx.x * 64;
    const int c0 = blockIdx.y * 64;
    const int cl = (threadIdx.x % TPR) * V, rl = threadIdx.x / TPR;
    uint4 raw[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k) {  // every load in flight before the first use
        const long long r = r0 + rl + k * RPP;
        raw[k] = r < M ? *reinterpret_cast<const uint4 *>(in + r * ld_in + c0 + cl) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        const int rr = rl + k * RPP;
        const TIn *x = reinterpret_cast<const TIn *>(&raw[k]);
        float v[V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            v[j] = to_f(x[j]);
            tile[rr][cl + j] = v[j];
        }
        if (rows16 && r0 + rr < M) {
            __half *dst = rows16 + (r0 + rr) * ld16 + c0 + cl;
            if constexpr (V == 8) {
                uint4 w;
                uint32_t *wp = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
                    wp[j] = *reinterpret_cast<const uint32_t *>(&h);
                }
                *reinterpret_cast<uint4 *>(dst) = w;
            } else {
                uint2 w;
                const __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
                w.x = *reinterpret_cast<const uint32_t *>(&a);
                w.y = *reinterpret_cast<const uint32_t *>(&b);
                *reinterpret_cast<uint2 *>(dst) = w;
            }
        }
    }
    __syncthreads();
    if (colsum && threadIdx.x < 64) {
        float acc = 0.f;
        for (int rr = 0; rr < 64; ++rr) acc = __fadd_rn(acc, tile[rr][threadIdx.x]);
        colsum[(long long)blockIdx.x * E + c0 + threadIdx.x] = acc;
    }
    // output row c0 + cc, tile rows 8 seg .. 8 seg + 7: a warp takes 8 columns
    // x 4 segments (shared-memory banks (8 seg + cc + i) mod 32 all differ)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cc = warp * 8 + (lane >> 2);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int seg = 4 * k + (lane & 3);
        uint4 w;
        uint32_t *wp = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const TOut lo = from_f<TOut>(tile[8 * seg + 2 * j][cc]), hi = from_f<TOut>(tile[8 * seg + 2 * j + 1][cc]);
            wp[j] = (uint32_t)*reinterpret_cast<const unsigned short *>(&lo) |
                    ((uint32_t)*reinterpret_cast<const unsigned short *>(&hi) << 16);
        }
        *reinterpret_cast<uint4 *>(out + (long long)(c0 + cc) * ld_out + r0 + 8 * seg) = w;
    }
}

// fp32 rows -> fp16 rows of another pitch (a slot of a concatenated row);
// four channels per thread (E % 4 == 0, pitches multiples of 4)
__global__ void k_rows_f16(const float *__restrict__ in, long long rows, int E, __half *__restrict__ out,
                           long long ld_out)
{
    const long long i = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= rows * E) return;
    const long long r = i / E;
    const int c = (int)(i - r * E);
    const float4 v = *reinterpret_cast<const float4 *>(in + i);
    const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t *>(&a);
    w.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(out + r * ld_out + c) = w;
}

inline unsigned blocks(long long n, int t) { return (unsigned)((n + t - 1) / t); }

template <typename T, int CPL>
bool launch_walks_lpe(int lpe, const WalkArgs &dq, const WalkArgs &dkv, cudaStream_t s)
{
    const long long groups = (dq.B + 32 / lpe - 1) / (32 / lpe);
    if constexpr (std::is_same<T, __half>::value && (CPL == 8 || CPL == 16)) {
        // rows gathered through a cp.async ring, paired fp32 arithmetic
        const unsigned grid_s = blocks(groups * dq.n_units, bwds::kWarps);
        switch (lpe) {
#define PMHA_WALK_S(L)                                                                   \
    case L:                                                                              \
        bwds::k_bwd_dq_s<CPL, L><<<grid_s, bwds::kWarps * 32, 0, s>>>(dq);               \
        bwds::k_bwd_dkv_s<CPL, L><<<grid_s, bwds::kWarps * 32, 0, s>>>(dkv);             \
        return true;
            PMHA_WALK_S(1) PMHA_WALK_S(2) PMHA_WALK_S(4) PMHA_WALK_S(8) PMHA_WALK_S(16) PMHA_WALK_S(32)
#undef PMHA_WALK_S
        default: return false;
        }
    }
    const unsigned grid = blocks(groups * dq.n_units, kBwdWarps);
    switch (lpe) {
#define PMHA_WALK(L)                                                    \
    case L:                                                             \
        k_bwd_dq<T, CPL, L><<<grid, kBwdWarps * 32, 0, s>>>(dq);        \
        k_bwd_dkv<T, CPL, L><<<grid, kBwdWarps * 32, 0, s>>>(dkv);      \
        return true;
        PMHA_WALK(1) PMHA_WALK(2) PMHA_WALK(4) PMHA_WALK(8) PMHA_WALK(16) PMHA_WALK(32)
#undef PMHA_WALK
    default: return false;
    }
}

template <typename T>
bool launch_walks(int cpl, int lpe, const WalkArgs &dq, const WalkArgs &dkv, cudaStream_t s)
{
    switch (cpl) {
    case 1: return launch_walks_lpe<T, 1>(lpe, dq, dkv, s);
    case 2: return launch_walks_lpe<T, 2>(lpe, dq, dkv, s);
    case 4: return launch_walks_lpe<T, 4>(lpe, dq, dkv, s);
    case 8: return launch_walks_lpe<T, 8>(lpe, dq, dkv, s);
    case 16: return launch_walks_lpe<T, 16>(lpe, dq, dkv, s);
    default: return false;
    }
}

}  // namespace

// Channels per lane (CPL) and lanes per sample (LPE = E / CPL) of the
// per-edge backward kernels: CPL the largest power of two up to 16 (fp16) or
// 8 (fp32) that divides the head size, LPE a power of two up to 32.
bool bwd_shape(int64_t E, int64_t H, int *cpl, int *lpe, TcType t)
{
    if (H < 1 || E % H) return false;
#ifndef PMHA_BWD_CMAX
#define PMHA_BWD_CMAX 16
#endif
    const int64_t d = E / H, cmax = t == TcType::F16 ? PMHA_BWD_CMAX : 8;
    int64_t c = 1;
    while (c * 2 <= cmax && d % (c * 2) == 0) c *= 2;
    if (E % c) return false;
    const int64_t l = E / c;
    if (l < 1 || l > 32 || (l & (l - 1))) return false;
    *cpl = (int)c;
    *lpe = (int)l;
    return true;
}

pmha_status bwd_rowdot(TcType t, const void *dmixed, const void *mixed, int64_t rows, int64_t E, int64_t H, float *D,
                       const float *ml, float2 *rec, cudaStream_t s)
{
    StageTimer timer("bwd_rowdot", s);
    if (t == TcType::F16)
        k_rowdot<__half><<<blocks(rows * H, 256), 256, 0, s>>>((const __half *)dmixed, (const __half *)mixed, rows,
                                                              (int)E, (int)H, D, ml, rec);
    else
        k_rowdot<float><<<blocks(rows * H, 256), 256, 0, s>>>((const float *)dmixed, (const float *)mixed, rows,
                                                             (int)E, (int)H, D, ml, rec);
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

pmha_status bwd_attention(TcType t, const pmha_graph *g, const BwdAttnArgs &x, cudaStream_t s)
{
    int cpl, lpe;
    if (!bwd_shape(x.E, x.H, &cpl, &lpe, t)) {
        set_error("backward: no kernel for embed_dim %lld, num_heads %lld", (long long)x.E, (long long)x.H);
        return PMHA_ERR_UNSUPPORTED;
    }
    WalkArgs dq;
    dq.q = x.q;
    dq.q_ld = x.q_ld;
    dq.k = x.k;
    dq.v = x.v;
    dq.kv_ld = x.kv_ld;
    dq.g = x.dmixed;
    dq.ml = x.ml;
    dq.D = x.D;
    dq.kpm = x.kpm;
    dq.n_units = g->n_units;
    dq.nnz = g->nnz;
    dq.B = (int)x.B;
    dq.L = (int)g->L;
    dq.S = (int)g->S;
    dq.E = (int)x.E;
    dq.H = (int)x.H;
    dq.score_scale = (float)(1.4426950408889634 / sqrt((double)(x.E / x.H)));
    dq.inv_sqrt_d = (float)(1.0 / sqrt((double)(x.E / x.H)));
    WalkArgs dkv = dq;
    dq.row_ptr = g->row_ptr;
    dq.idx = g->col;
    dq.unit_first = g->unit_first_t;
    dq.n_rows = (int)g->L;
    dq.out0 = x.dq;
    dq.out1 = nullptr;
    dq.part = x.part_dq;
    dkv.row_ptr = g->src_row_ptr;
    dkv.idx = g->tgt_by_src;
    dkv.unit_first = g->unit_first_s;
    dkv.n_rows = (int)g->S;
    dkv.out0 = x.dk;
    dkv.out1 = x.dv;
    dkv.part = x.part_dkv;
    if (x.B * g->n_units > 0 && x.rec && t == TcType::F16 && bwd_ring_supported(x.E, x.H)) {
        // the ring kernels: persistent warps on a queue per view
        StageTimer timer("bwd_edges", s);
        PMHA_CUDA_TRY(cudaMemsetAsync(x.ctr, 0, 2 * sizeof(unsigned), s));
        BwdRingArgs r;
        r.q = x.q;
        r.q_ld = x.q_ld;
        r.k = x.k;
        r.v = x.v;
        r.kv_ld = x.kv_ld;
        r.g = x.dmixed;
        r.rec = x.rec;
        r.kpm = x.kpm;
        r.n_units = g->n_units;
        r.nnz = g->nnz;
        r.B = (int)x.B;
        r.L = (int)g->L;
        r.S = (int)g->S;
        r.E = (int)x.E;
        r.H = (int)x.H;
        r.score_scale = dq.score_scale;
        r.inv_sqrt_d = dq.inv_sqrt_d;
        BwdRingArgs rk = r;
        r.row_ptr = g->row_ptr;
        r.idx = g->col;
        r.unit_first = g->unit_first_t;
        r.unit_order = g->unit_order;
        r.n_rows = (int)g->L;
        r.out0 = x.dq;
        r.out1 = nullptr;
        r.part = x.part_dq;
        r.task_counter = x.ctr;
        rk.row_ptr = g->src_row_ptr;
        rk.idx = g->tgt_by_src;
        rk.unit_first = g->unit_first_s;
        rk.unit_order = nullptr;
        rk.n_rows = (int)g->S;
        rk.out0 = x.dk;
        rk.out1 = x.dv;
        rk.part = x.part_dkv;
        rk.task_counter = x.ctr + 1;
        pmha_status st = launch_bwd_ring(false, r, s);
        if (st == PMHA_OK) st = launch_bwd_ring(true, rk, s);
        if (st != PMHA_OK) return st;
        count_launch(2);
        PMHA_CUDA_TRY(cudaGetLastError());
    } else if (x.B * g->n_units > 0) {
        StageTimer timer("bwd_edges", s);
        const bool ok = t == TcType::F16 ? launch_walks<__half>(cpl, lpe, dq, dkv, s)
                                         : launch_walks<float>(cpl, lpe, dq, dkv, s);
        if (!ok) {
            set_error("backward: no kernel for %d channels per lane", cpl);
            return PMHA_ERR_UNSUPPORTED;
        }
        count_launch(2);
        PMHA_CUDA_TRY(cudaGetLastError());
    }
    StageTimer timer("bwd_merge", s);
    if (g->n_merge > 0) {
        k_bwd_merge<<<blocks(x.B * g->n_merge, 8), 256, 0, s>>>(g->merge_t, g->n_merge, g->row_ptr, x.part_dq,
                                                                g->n_units, (int)x.B, (int)g->L, (int)x.E, (int)x.E,
                                                                x.dq, nullptr);
        count_launch();
    }
    if (g->n_merge_s > 0) {
        k_bwd_merge<<<blocks(x.B * g->n_merge_s, 8), 256, 0, s>>>(g->merge_s, g->n_merge_s, g->src_row_ptr,
                                                                  x.part_dkv, g->n_units, (int)x.B, (int)g->S,
                                                                  (int)x.E, (int)(2 * x.E), x.dk, x.dv);
        count_launch();
    }
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

// ---------------------------------------------------------------- GEMM entry points
namespace {
template <typename TA, typename TB, typename TC>
void nn_launch(const void *A, long long lda, const void *B, long long ldb, void *C, long long ldc, long long M, int N,
               int K, bool acc, cudaStream_t s)
{
    dim3 grid(blocks(M, 64), blocks(N, 64));
    if (acc)
        k_gemm_nn<TA, TB, TC, true><<<grid, 256, 0, s>>>((const TA *)A, lda, (const TB *)B, ldb, (TC *)C, ldc, M, N,
                                                          K);
    else
        k_gemm_nn<TA, TB, TC, false><<<grid, 256, 0, s>>>((const TA *)A, lda, (const TB *)B, ldb, (TC *)C, ldc, M,
                                                           N, K);
}
}  // namespace

// C (M x N) (+)= A (M x K) . B (K x N); types: A in {F32, BF16, F16}, B in
// {F32, BF16}, C in {F32, F16}.
pmha_status bwd_gemm_nn(TcType ta, TcType tb, TcType tc, const void *A, int64_t lda, const void *B, int64_t ldb,
                        void *C, int64_t ldc, int64_t M, int64_t N, int64_t K, bool accumulate, cudaStream_t s)
{
    if (M <= 0) return PMHA_OK;
#define PMHA_NN(TA_, TB_, TC_) nn_launch<TA_, TB_, TC_>(A, lda, B, ldb, C, ldc, M, (int)N, (int)K, accumulate, s)
    if (tc == TcType::F32) {
        if (ta == TcType::F32 && tb == TcType::F32) PMHA_NN(float, float, float);
        else if (ta == TcType::F32 && tb == TcType::BF16) PMHA_NN(float, __nv_bfloat16, float);
        else if (ta == TcType::BF16 && tb == TcType::BF16) PMHA_NN(__nv_bfloat16, __nv_bfloat16, float);
        else {
            set_error("bwd_gemm_nn: unsupported operand types");
            return PMHA_ERR_UNSUPPORTED;
        }
    } else if (tc == TcType::F16) {
        if (ta == TcType::BF16 && tb == TcType::BF16) PMHA_NN(__nv_bfloat16, __nv_bfloat16, __half);
        else {
            set_error("bwd_gemm_nn: unsupported operand types");
            return PMHA_ERR_UNSUPPORTED;
        }
    } else {
        set_error("bwd_gemm_nn: unsupported output type");
        return PMHA_ERR_UNSUPPORTED;
    }
#undef PMHA_NN
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

// dW (K x N, fp32) = A^T B over M rows (A: M x K, B: M x N), and, when db is
// given, db (K) = column sums of A; `scratch` holds the per-chunk partials.
pmha_status bwd_gemm_tn(TcType ta, TcType tb, const void *A, int64_t lda, const void *B, int64_t ldb, int64_t M,
                        int64_t K, int64_t N, float *dW, float *db, float *scratch, int64_t chunks, cudaStream_t s)
{
    if (chunks < 1) chunks = 1;
    const long long rpc = (M + chunks - 1) / chunks;
    if (dW) {
        dim3 grid(blocks(K, 64), blocks(N, 64), (unsigned)chunks);
#define PMHA_TN(TA_, TB_)                                                                                       \
    k_gemm_tn_part<TA_, TB_><<<grid, 256, 0, s>>>((const TA_ *)A, lda, (const TB_ *)B, ldb, M, (int)K, (int)N, \
                                                  rpc, scratch)
        if (ta == TcType::F32 && tb == TcType::F32) PMHA_TN(float, float);
        else if (ta == TcType::F32 && tb == TcType::BF16) PMHA_TN(float, __nv_bfloat16);
        else if (ta == TcType::F32 && tb == TcType::F16) PMHA_TN(float, __half);
        else if (ta == TcType::BF16 && tb == TcType::F16) PMHA_TN(__nv_bfloat16, __half);
        else if (ta == TcType::BF16 && tb == TcType::BF16) PMHA_TN(__nv_bfloat16, __nv_bfloat16);
        else {
            set_error("bwd_gemm_tn: unsupported operand types");
            return PMHA_ERR_UNSUPPORTED;
        }
#undef PMHA_TN
        k_sum_chunks<<<blocks(K * N, 32), 256, 0, s>>>(scratch, K * N, (int)chunks, dW);
        count_launch(2);
    }
    if (db) {
        dim3 grid(blocks(K, 256), (unsigned)chunks);
        if (ta == TcType::F32) k_colsum_part<float><<<grid, 256, 0, s>>>((const float *)A, lda, M, (int)K, rpc, scratch);
        else k_colsum_part<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16 *)A, lda, M, (int)K, rpc, scratch);
        k_sum_chunks<<<blocks(K, 32), 256, 0, s>>>(scratch, K, (int)chunks, db);
        count_launch(2);
    }
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

// ---------------------------------------------------------------- steps 5 and 1
namespace {
bool use_tc(const BwdGemmArgs &g) { return g.pt == TcType::BF16 && g.E % 128 == 0 && gemm_tc_supported(g.E); }
int64_t pad64(int64_t m) { return (m + 63) / 64 * 64; }
constexpr int64_t kMaxSplit = 256;

// bump allocator over the caller's scratch (256-byte steps)
struct Bump {
    char *p;
    size_t used = 0;
    template <typename T>
    T *take(size_t n)
    {
        T *r = (T *)(p + used);
        used += (n * sizeof(T) + 255) & ~(size_t)255;
        return r;
    }
};

template <typename TIn, typename TOut>
pmha_status transpose_cvt(const void *in, int64_t ld_in, int64_t M, int64_t E, int64_t Mpad, void *out, int64_t ld_out,
                          cudaStream_t s, float *colsum = nullptr, __half *rows16 = nullptr, int64_t ld16 = 0)
{
    auto a16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    if (E % 64 || Mpad % 64 || Mpad < M || ld_in % 8 || ld_out % 8 || (rows16 && ld16 % 8) || !a16(in) || !a16(out) ||
        !a16(rows16)) {
        set_error("backward transpose: shape or alignment outside what its kernel takes (E %lld, Mpad %lld)",
                  (long long)E, (long long)Mpad);
        return PMHA_ERR_UNSUPPORTED;
    }
    StageTimer timer("bwd_transpose", s);
    dim3 grid(blocks(Mpad, 64), blocks(E, 64));
    k_transpose_cvt<TIn, TOut><<<grid, 256, 0, s>>>((const TIn *)in, ld_in, M, (int)E, Mpad, (TOut *)out, ld_out,
                                                    colsum, rows16, ld16);
    count_launch();
    return PMHA_OK;
}

// db (E) = column sums of an (M x E) matrix from the per-64-row-tile sums a
// transpose_cvt left in colsum: one block per column, thread i adds tiles
// i, i + 256, ... in order, then a fixed-order tree over the 256 threads
void bias_from_tiles(const float *colsum, int64_t M, int64_t E, float *db, cudaStream_t s)
{
    StageTimer timer("bwd_bias", s);
    k_sum_tiles<<<(unsigned)E, 256, 0, s>>>(colsum, E, (int)((M + 63) / 64), db);
    count_launch();
}

// dW (E x E) = sum_r dYT[o][r] XT[i][r] on the tensor cores (split K, fp32 partials, ordered sum)
pmha_status dw_tc(const __half *dyT, const __half *xT, int64_t E, int64_t Mpad, float *dW, float *part,
                  cudaStream_t s)
{
    const int64_t ksplit = std::min<int64_t>(kMaxSplit, std::max<int64_t>(1, Mpad / 64));
    pmha_status st = gemm_tc_general(TcType::F16, TcType::F32, dyT, Mpad, E, Mpad, xT, Mpad, E, part, E, ksplit,
                                     "bwd_dw", s);
    if (st != PMHA_OK) return st;
    const int64_t kb = Mpad / 64, per = (kb + ksplit - 1) / ksplit, used = (kb + per - 1) / per;
    k_sum_chunks<<<blocks(E * E, 32), 256, 0, s>>>(part, E * E, (int)used, dW);
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}
}  // namespace

size_t bwd_gemm_scratch_bytes(int64_t B, int64_t L, int64_t S, int64_t E, TcType pt)
{
    const int64_t Mq = B * L, Mk = B * S, M = std::max(Mq, Mk);
    const int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(64, M / 4096));
    size_t simt = ((size_t)(chunks * E * E) * 4 + 255) & ~(size_t)255;
    if (!(pt == TcType::BF16 && E % 128 == 0)) return simt;
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const int64_t Mqp = pad64(Mq), Mkp = pad64(Mk), Mp = std::max(Mqp, Mkp);
    size_t tc = al((size_t)(E * E) * 2)                  // Wo^T
                + al((size_t)(E * 3 * E) * 2)            // the weights of one input's roles, transposed
                + 2 * al((size_t)(E * Mqp) * 2)          // dout^T, mixed^T
                + 3 * al((size_t)(E * Mp) * 2)           // dq^T, dk^T, dv^T
                + 3 * al((size_t)(E * Mp) * 2)           // the inputs transposed
                + al((size_t)(M * 3 * E) * 2)            // one input's dY rows in fp16
                + al((size_t)(kMaxSplit * E * E) * 4)    // split-K partials
                + al((size_t)(Mp / 64 * E) * 4);         // per-tile column sums
    return std::max(simt, tc) + 256;
}

pmha_status bwd_step5(const BwdGemmArgs &g, cudaStream_t s)
{
    const int64_t E = g.E, M = g.B * g.L;
    pmha_status st;
    if (use_tc(g)) {
        Bump bump{(char *)g.scratch};
        __nv_bfloat16 *woT = bump.take<__nv_bfloat16>((size_t)(E * E));
        if ((st = transpose_cvt<__nv_bfloat16, __nv_bfloat16>(g.w[3], E, E, E, E, woT, E, s)) != PMHA_OK) return st;
        // dmixed = dout Wo = dout (Wo^T)^T
        if ((st = gemm_tc_general(TcType::BF16, g.it, g.dout, E, M, E, woT, E, E, g.dmixed, E, 1, "bwd_dmixed", s)) !=
            PMHA_OK)
            return st;
        if (g.gw[3]) {
            const int64_t Mp = pad64(M);
            __half *doutT = bump.take<__half>((size_t)(E * Mp));
            __half *mixT = bump.take<__half>((size_t)(E * Mp));
            float *part = bump.take<float>((size_t)(kMaxSplit * E * E));
            float *cs = g.gb[3] ? bump.take<float>((size_t)(Mp / 64 * E)) : nullptr;
            if ((st = transpose_cvt<__nv_bfloat16, __half>(g.dout, E, M, E, Mp, doutT, Mp, s, cs)) != PMHA_OK) return st;
            if ((st = transpose_cvt<__half, __half>(g.mixed, E, M, E, Mp, mixT, Mp, s)) != PMHA_OK) return st;
            if ((st = dw_tc(doutT, mixT, E, Mp, g.gw[3], part, s)) != PMHA_OK) return st;
            if (cs) bias_from_tiles(cs, M, E, g.gb[3], s);
        }
        if (g.gb[3] && !g.gw[3])
            if ((st = bwd_gemm_tn(g.pt, g.it, g.dout, E, g.mixed, E, M, E, E, nullptr, g.gb[3], (float *)g.scratch,
                                  g.chunks, s)) != PMHA_OK)
                return st;
        PMHA_CUDA_TRY(cudaGetLastError());
        return PMHA_OK;
    }
    if ((st = bwd_gemm_nn(g.pt, g.pt, g.it, g.dout, E, g.w[3], E, g.dmixed, E, M, E, E, false, s)) != PMHA_OK) return st;
    if (g.gw[3] || g.gb[3])
        if ((st = bwd_gemm_tn(g.pt, g.it, g.dout, E, g.mixed, E, M, E, E, g.gw[3], g.gb[3], (float *)g.scratch,
                              g.chunks, s)) != PMHA_OK)
            return st;
    return PMHA_OK;
}

pmha_status bwd_step1(const BwdGemmArgs &g, cudaStream_t s)
{
    const int64_t E = g.E;
    const int64_t rows[3] = {g.B * g.L, g.B * g.S, g.B * g.S};
    pmha_status st;
    if (!use_tc(g)) {
        // bias gradients: column sums of dq, dk, dv (ordered chunks)
        for (int r = 0; r < 3; ++r)
            if (g.gb[r])
                if ((st = bwd_gemm_tn(TcType::F32, g.pt, g.dy[r], E, g.in[r], E, rows[r], E, E, nullptr, g.gb[r],
                                      (float *)g.scratch, g.chunks, s)) != PMHA_OK)
                    return st;
        for (int r = 0; r < 3; ++r)
            if (g.gw[r])
                if ((st = bwd_gemm_tn(TcType::F32, g.pt, g.dy[r], E, g.in[r], E, rows[r], E, E, g.gw[r], nullptr,
                                      (float *)g.scratch, g.chunks, s)) != PMHA_OK)
                    return st;
        for (int r = 0; r < 3; ++r) {
            bool seen = false;
            for (int q = 0; q < r; ++q) seen |= g.in[q] == g.in[r];
            if (seen || !g.gx[r]) continue;
            bool first = true;
            for (int q = r; q < 3; ++q) {
                if (g.in[q] != g.in[r]) continue;
                if ((st = bwd_gemm_nn(TcType::F32, g.pt, TcType::F32, g.dy[q], E, g.w[q], E, g.dx32, E, rows[r], E, E,
                                      !first, s)) != PMHA_OK)
                    return st;
                first = false;
            }
            if ((st = bwd_convert(g.dx32, rows[r] * E, g.pt, g.gx[r], s)) != PMHA_OK) return st;
        }
        return PMHA_OK;
    }
    Bump bump{(char *)g.scratch};
    (void)bump.take<__nv_bfloat16>((size_t)(E * E));  // Wo^T of step 5 (not needed here; keeps offsets stable)
    __half *wsub = bump.take<__half>((size_t)(E * 3 * E));
    const int64_t Mp = pad64(std::max(rows[0], rows[1]));
    (void)bump.take<__half>((size_t)(E * pad64(rows[0])));
    (void)bump.take<__half>((size_t)(E * pad64(rows[0])));
    __half *dyT[3], *xT[3];
    for (int r = 0; r < 3; ++r) dyT[r] = bump.take<__half>((size_t)(E * Mp));
    for (int r = 0; r < 3; ++r) xT[r] = bump.take<__half>((size_t)(E * Mp));
    __half *dy16 = bump.take<__half>((size_t)(std::max(rows[0], rows[1]) * 3 * E));
    float *part = bump.take<float>((size_t)(kMaxSplit * E * E));
    float *cs = bump.take<float>((size_t)(Mp / 64 * E));
    // The input gradient of each input (below) is one product over the roles it
    // feeds, with their dY rows side by side in fp16: the roles of input group
    // lead (its first role) fill a region of dy16 of rows x (n_roles E), slot
    // i of role i of the group. Regions of different inputs do not overlap.
    __half *pack16[3] = {nullptr, nullptr, nullptr};  // where role r's fp16 dY rows go (null: no input gradient)
    int64_t pack_ld[3] = {0, 0, 0};
    {
        int64_t off = 0;
        for (int r = 0; r < 3; ++r) {
            bool seen = false;
            for (int q = 0; q < r; ++q) seen |= g.in[q] == g.in[r];
            if (seen || !g.gx[r]) continue;
            int nr = 0;
            for (int q = r; q < 3; ++q) nr += g.in[q] == g.in[r];
            for (int q = r, i = 0; q < 3; ++q)
                if (g.in[q] == g.in[r]) {
                    pack16[q] = dy16 + off + i++ * E;
                    pack_ld[q] = nr * E;
                }
            off += rows[r] * nr * E;
        }
    }
    bool packed[3] = {false, false, false};
    // weight gradients dW_r = dY_r^T X_r: both transposed to fp16 (tokens along K);
    // the bias gradient (column sums of dY_r) comes out of the same transpose, and
    // so do dY_r's fp16 rows for the input gradient
    for (int r = 0; r < 3; ++r) {
        if (!g.gw[r] && !g.gb[r]) continue;
        const int64_t mp = pad64(rows[r]);
        if ((st = transpose_cvt<float, __half>(g.dy[r], E, rows[r], E, mp, dyT[r], mp, s, g.gb[r] ? cs : nullptr,
                                               pack16[r], pack_ld[r])) != PMHA_OK)
            return st;
        packed[r] = pack16[r] != nullptr;
        if (g.gb[r]) bias_from_tiles(cs, rows[r], E, g.gb[r], s);
        if (!g.gw[r]) continue;
        int src = r;
        for (int q = 0; q < r; ++q)
            if (g.in[q] == g.in[r] && g.gw[q]) {
                src = q;
                break;
            }
        if (src == r)
            if ((st = transpose_cvt<__nv_bfloat16, __half>(g.in[r], E, rows[r], E, mp, xT[r], mp, s)) != PMHA_OK)
                return st;
        if ((st = dw_tc(dyT[r], xT[src], E, mp, g.gw[r], part, s)) != PMHA_OK) return st;
    }
    // input gradients: dX = sum over the roles of X of dY_r W_r, one K = n_roles * E product
    for (int r = 0; r < 3; ++r) {
        bool seen = false;
        for (int q = 0; q < r; ++q) seen |= g.in[q] == g.in[r];
        if (seen || !g.gx[r]) continue;
        int roles[3], nr = 0;
        for (int q = r; q < 3; ++q)
            if (g.in[q] == g.in[r]) roles[nr++] = q;
        const int64_t K = nr * E;
        for (int i = 0; i < nr; ++i) {
            const int q = roles[i];
            if (!packed[q]) {
                StageTimer pack_timer("bwd_pack", s);
                k_rows_f16<<<blocks(rows[r] * E / 4, 256), 256, 0, s>>>(g.dy[q], rows[r], (int)E, pack16[q], K);
                count_launch();
            }
            if ((st = transpose_cvt<__nv_bfloat16, __half>(g.w[q], E, E, E, E, wsub + i * E, K, s)) != PMHA_OK)
                return st;
        }
        if ((st = gemm_tc_general(TcType::F16, g.pt, pack16[r], K, rows[r], K, wsub, K, E, g.gx[r], E, 1, "bwd_dx",
                                  s)) != PMHA_OK)
            return st;
    }
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

pmha_status bwd_convert(const float *in, int64_t n, TcType out_t, void *out, cudaStream_t s)
{
    if (n <= 0) return PMHA_OK;
    if (out_t == TcType::BF16) k_convert<__nv_bfloat16><<<blocks(n, 256), 256, 0, s>>>(in, n, (__nv_bfloat16 *)out);
    else if (out_t == TcType::F32) k_convert<float><<<blocks(n, 256), 256, 0, s>>>(in, n, (float *)out);
    else k_convert<__half><<<blocks(n, 256), 256, 0, s>>>(in, n, (__half *)out);
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

}  // namespace pmha
