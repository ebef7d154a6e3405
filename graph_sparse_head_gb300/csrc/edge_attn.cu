// Edge attention: scores, segmented softmax and value mix over the live edges
// into each target (kpnn2 PackedMultiheadAttention, Notes steps 2-4, and the
// paragraph after them: a target without live keys mixes to zeros).
//
// One warp per work item = (sample b, target t, a range of t's edges in CSR
// order). The warp covers all H heads of the target. Lane layout for a row of
// E channels: a lane owns CPL consecutive channels (16 bytes of fp16 when
// CPL = 8), E / CPL lanes cover one row, so 32 / (E / CPL) "slots" of lanes
// walk different edges of the same target side by side. A head's channels
// sit in d / CPL adjacent lanes; the per-head dot product is a butterfly sum
// over them, so every lane of a head holds the same score.
//
// Per slot the softmax is online, in log2 units: s = (q . k) * log2(e)/sqrt(d)
// with q pre-scaled in fp32 registers; m = running max, l = running sum of
// 2^(s - m), acc = running sum of 2^(s - m) * v. U edges are loaded before
// they are used, then folded in with one rescale. Slots merge at the end with
// the same rule; split targets write (m, l, acc) partials that a second
// kernel merges in chunk order. The (m, l) arithmetic uses explicit
// round-to-nearest intrinsics so that it is identical in the kernel variants
// with and without values, which makes pmha_edge_weights bit-identical to the
// weights of pmha_forward.
#include <math.h>

#include "pmha_internal.h"

namespace pmha {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct KArgs {
    const void *q;
    long long q_ld;
    const void *kv;
    long long kv_ld, v_off;
    void *mixed;
    float *part;
    float *ml;
    float *scores;
    const int32_t *col;
    const int32_t *perm;
    const Item *items;
    long long n_items, n_parts, nnz;
    int B, L, S, E, H, d;
    float score_scale;
};

// CPL consecutive channels of a row, widened to fp32, with the widest aligned
// vector loads (16 bytes per access when CPL * sizeof(T) >= 16).
template <int CPL>
__device__ __forceinline__ void load_channels_h(const __half *p, float (&f)[CPL])
{
    constexpr int bytes = CPL * 2;
    if constexpr (bytes >= 16) {
#pragma unroll
        for (int v = 0; v < bytes / 16; ++v) {
            uint4 u = __ldg(reinterpret_cast<const uint4 *>(p) + v);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&w[j]));
                f[v * 8 + 2 * j] = x.x;
                f[v * 8 + 2 * j + 1] = x.y;
            }
        }
    } else if constexpr (bytes == 8) {
        uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
        f[0] = a.x;
        f[1] = a.y;
        f[2] = b.x;
        f[3] = b.y;
    } else {
        unsigned int u = __ldg(reinterpret_cast<const unsigned int *>(p));
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&u));
        f[0] = a.x;
        f[1] = a.y;
    }
}

template <int CPL>
__device__ __forceinline__ void load_channels_f32(const float *p, float (&f)[CPL])
{
    if constexpr (CPL >= 4) {
#pragma unroll
        for (int v = 0; v < CPL / 4; ++v) {
            float4 u = __ldg(reinterpret_cast<const float4 *>(p) + v);
            f[4 * v] = u.x;
            f[4 * v + 1] = u.y;
            f[4 * v + 2] = u.z;
            f[4 * v + 3] = u.w;
        }
    } else {
        float2 u = __ldg(reinterpret_cast<const float2 *>(p));
        f[0] = u.x;
        f[1] = u.y;
    }
}

template <typename T, int CPL>
__device__ __forceinline__ void load_row(const T *p, float (&f)[CPL])
{
    if constexpr (sizeof(T) == 2) load_channels_h<CPL>(reinterpret_cast<const __half *>(p), f);
    else load_channels_f32<CPL>(reinterpret_cast<const float *>(p), f);
}

template <typename T, int CPL>
__device__ __forceinline__ void store_row(T *p, const float (&f)[CPL])
{
    if constexpr (sizeof(T) == 2) {
        uint32_t w[CPL / 2];
#pragma unroll
        for (int j = 0; j < CPL / 2; ++j) {
            __half2 h = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t *>(&h);
        }
        if constexpr (CPL * 2 >= 16) {
#pragma unroll
            for (int v = 0; v < CPL * 2 / 16; ++v)
                reinterpret_cast<uint4 *>(p)[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        } else if constexpr (CPL * 2 == 8) {
            *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
        } else {
            *reinterpret_cast<uint32_t *>(p) = w[0];
        }
    } else {
        if constexpr (CPL >= 4) {
#pragma unroll
            for (int v = 0; v < CPL / 4; ++v)
                reinterpret_cast<float4 *>(p)[v] = make_float4(f[4 * v], f[4 * v + 1], f[4 * v + 2], f[4 * v + 3]);
        } else {
            *reinterpret_cast<float2 *>(p) = make_float2(f[0], f[1]);
        }
    }
}

// Merge softmax state (m2, l2, acc2) into (m, l, acc). Symmetric in its two
// operands, so lanes that merge with each other end with identical state.
template <int CPL, bool WV>
__device__ __forceinline__ void merge_state(float &m, float &l, float (&acc)[CPL], float m2, float l2,
                                            const float (&acc2)[CPL])
{
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    const float s1 = (m == -INFINITY) ? 0.f : ex2(__fsub_rn(m, M));
    const float s2 = (m2 == -INFINITY) ? 0.f : ex2(__fsub_rn(m2, M));
    l = __fadd_rn(__fmul_rn(l, s1), __fmul_rn(l2, s2));
    if constexpr (WV) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] = __fadd_rn(__fmul_rn(acc[c], s1), __fmul_rn(acc2[c], s2));
    }
    m = M;
}

template <typename T, int CPL, int U, bool WV>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) k_edge_attn(KArgs a)
{
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= (long long)a.B * a.n_items) return;
    const int b = (int)(gw / a.n_items);
    const Item it = a.items[gw - (long long)b * a.n_items];

    const int lpe = a.E / CPL;  // lanes per row
    const int P = 32 / lpe;     // slots
    const int slot = lane / lpe, grp = lane - slot * lpe;
    const int c0 = grp * CPL;
    const int head = c0 / a.d;
    const int lph = a.d / CPL;  // lanes per head
    const bool head_leader = (grp % lph) == 0;

    const T *Q = (const T *)a.q;
    const T *KV = (const T *)a.kv;
    float qf[CPL];
    load_row<T, CPL>(Q + ((long long)b * a.L + it.t) * a.q_ld + c0, qf);
#pragma unroll
    for (int c = 0; c < CPL; ++c) qf[c] = __fmul_rn(qf[c], a.score_scale);

    float m = -INFINITY, l = 0.f;
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;

    const long long kv_sample = (long long)b * a.S;
    float *scores_b = a.scores ? a.scores + (long long)b * a.nnz * a.H : nullptr;

    for (int base = it.begin; base < it.end; base += 32) {
        const int n = min(32, it.end - base);
        const int my_col = lane < n ? a.col[base + lane] : 0;
        const int my_perm = (scores_b && lane < n) ? a.perm[base + lane] : 0;
        for (int j = 0; j < n; j += P * U) {
            float kf[U][CPL];
            float vf[WV ? U : 1][CPL];
            bool valid[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int idx = j + slot + P * u;
                valid[u] = idx < n;
                const int s = __shfl_sync(0xffffffffu, my_col, idx & 31);
                if (valid[u]) {
                    const T *row = KV + (kv_sample + s) * a.kv_ld + c0;
                    load_row<T, CPL>(row, kf[u]);
                    if constexpr (WV) load_row<T, CPL>(row + a.v_off, vf[u]);
                } else {
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        kf[u][c] = 0.f;
                        if constexpr (WV) vf[u][c] = 0.f;
                    }
                }
            }
            float sc[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float dot = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) dot = __fmaf_rn(qf[c], kf[u][c], dot);
                for (int o = 1; o < lph; o <<= 1) dot = __fadd_rn(dot, __shfl_xor_sync(0xffffffffu, dot, o));
                sc[u] = valid[u] ? dot : -INFINITY;
                const int e = __shfl_sync(0xffffffffu, my_perm, (j + slot + P * u) & 31);
                if (scores_b && valid[u] && head_leader) scores_b[(long long)e * a.H + head] = sc[u];
            }
            float mx = m;
#pragma unroll
            for (int u = 0; u < U; ++u) mx = fmaxf(mx, sc[u]);
            if (mx != -INFINITY) {
                const float scale = (m == -INFINITY) ? 0.f : ex2(__fsub_rn(m, mx));
                l = __fmul_rn(l, scale);
                if constexpr (WV) {
#pragma unroll
                    for (int c = 0; c < CPL; ++c) acc[c] = __fmul_rn(acc[c], scale);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float p = valid[u] ? ex2(__fsub_rn(sc[u], mx)) : 0.f;
                    l = __fadd_rn(l, p);
                    if constexpr (WV) {
#pragma unroll
                        for (int c = 0; c < CPL; ++c) acc[c] = __fmaf_rn(p, vf[u][c], acc[c]);
                    }
                }
                m = mx;
            }
        }
    }

    // merge the slots: butterfly over lanes that own the same channels
    for (int o = lpe; o < 32; o <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        float acc2[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc2[c] = WV ? __shfl_xor_sync(0xffffffffu, acc[c], o) : 0.f;
        merge_state<CPL, WV>(m, l, acc, m2, l2, acc2);
    }
    if (slot != 0) return;

    if (it.slot < 0) {
        if constexpr (WV) {
            const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = __fmul_rn(acc[c], inv);
            store_row<T, CPL>((T *)a.mixed + ((long long)b * a.L + it.t) * a.E + c0, acc);
        }
        if (a.ml && head_leader) {
            float *p = a.ml + (((long long)b * a.L + it.t) * a.H + head) * 2;
            p[0] = m;
            p[1] = l;
        }
    } else {
        float *p = a.part + ((long long)b * a.n_parts + it.slot) * (2 * a.H + a.E);
        if (head_leader) {
            p[head] = m;
            p[a.H + head] = l;
        }
        if constexpr (WV) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) p[2 * a.H + c0 + c] = acc[c];
        }
    }
}

// One warp per (sample, split target): merges the target's chunk partials in
// chunk order with the rule of merge_state, lane-per-channel.
template <typename T, bool WV>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
k_split_merge(const Heavy *__restrict__ heavy, long long n_heavy, const float *__restrict__ part,
              long long n_parts, int B, int L, int E, int H, int d, void *mixed, float *ml)
{
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= (long long)B * n_heavy) return;
    const int b = (int)(gw / n_heavy);
    const Heavy hv = heavy[gw - (long long)b * n_heavy];
    const int stride = 2 * H + E;
    const float *pb = part + ((long long)b * n_parts + hv.first_slot) * stride;
    for (int c0 = 0; c0 < E; c0 += 32) {
        const int ch = c0 + lane;
        const bool live = ch < E;
        const int h = live ? ch / d : 0;
        float m = -INFINITY, l = 0.f;
        float acc[1] = {0.f};
        for (int i = 0; i < hv.n_chunks; ++i) {
            const float *p = pb + (long long)i * stride;
            const float acc2[1] = {WV && live ? p[2 * H + ch] : 0.f};
            merge_state<1, WV>(m, l, acc, p[h], p[H + h], acc2);
        }
        if (WV && live) {
            const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
            const float v = __fmul_rn(acc[0], inv);
            T *dst = (T *)mixed + ((long long)b * L + hv.t) * E + ch;
            if constexpr (sizeof(T) == 2) *reinterpret_cast<__half *>(dst) = __float2half_rn(v);
            else *reinterpret_cast<float *>(dst) = v;
        }
        if (ml && live && ch % d == 0) {
            float *q = ml + (((long long)b * L + hv.t) * H + h) * 2;
            q[0] = m;
            q[1] = l;
        }
    }
}

// weights[b, e, h] = 2^(s - m) / l for the target of edge e; averaged over
// heads when out has one entry per edge. Runs in place when out == scores
// (per-head layout: each thread reads its H scores before writing them).
__global__ void k_weights(const float *scores, const float *__restrict__ ml,
                          const int32_t *__restrict__ tgt_of_edge, long long B, long long nnz, int L,
                          int H, bool average, float *out)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * nnz) return;
    const long long b = i / nnz, e = i - b * nnz;
    const int t = tgt_of_edge[e];
    const float *s = scores + i * H;
    const float *st = ml + ((b * L + t) * H) * 2;
    float sum = 0.f;
    for (int h = 0; h < H; ++h) {
        const float w = __fmul_rn(ex2(__fsub_rn(s[h], st[2 * h])), __frcp_rn(st[2 * h + 1]));
        if (average) sum = __fadd_rn(sum, w);
        else out[i * H + h] = w;
    }
    if (average) out[i] = __fdiv_rn(sum, (float)H);
}

int pick_cpl(int64_t E, int64_t d, TcType t)
{
    static const int h_order[] = {8, 16, 32, 4, 2};
    static const int f32_order[] = {4, 8, 16, 2};
    const bool half = t != TcType::F32;
    const int *order = half ? h_order : f32_order;
    const int n = half ? 5 : 4;
    const int elem = half ? 2 : 4;
    if ((E * elem) % 16) return 0;
    auto pow2 = [](int64_t x) { return x > 0 && (x & (x - 1)) == 0; };
    for (int i = 0; i < n; ++i) {
        const int c = order[i];
        if (E % c || d % c) continue;
        if (E / c > 32 || !pow2(E / c) || !pow2(d / c)) continue;
        return c;
    }
    return 0;
}

template <typename T, int CPL, bool WV>
void launch_edge(const KArgs &k, long long warps, cudaStream_t s)
{
    constexpr int U = (CPL * sizeof(T) <= 16) ? 4 : 2;
    const long long blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    k_edge_attn<T, CPL, U, WV><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, s>>>(k);
}

template <typename T, bool WV>
bool dispatch_cpl(int cpl, const KArgs &k, long long warps, cudaStream_t s)
{
    switch (cpl) {
    case 2: launch_edge<T, 2, WV>(k, warps, s); return true;
    case 4: launch_edge<T, 4, WV>(k, warps, s); return true;
    case 8: launch_edge<T, 8, WV>(k, warps, s); return true;
    case 16: launch_edge<T, 16, WV>(k, warps, s); return true;
    case 32:
        if constexpr (sizeof(T) == 2) {
            launch_edge<T, 32, WV>(k, warps, s);
            return true;
        }
        return false;
    default: return false;
    }
}

}  // namespace

bool edge_supported(int64_t E, int64_t H, TcType t)
{
    if (H < 1 || E % H) return false;
    return pick_cpl(E, E / H, t) != 0;
}

pmha_status edge_attention(TcType dt, const pmha_graph *g, const EdgeArgs &a, cudaStream_t s)
{
    const int cpl = pick_cpl(a.E, a.E / a.H, dt);
    if (!cpl) {
        set_error("edge_attention: no kernel for embed_dim %lld, num_heads %lld", (long long)a.E, (long long)a.H);
        return PMHA_ERR_UNSUPPORTED;
    }
    KArgs k;
    k.q = a.q;
    k.q_ld = a.q_ld;
    k.kv = a.kv;
    k.kv_ld = a.kv_ld;
    k.v_off = a.v_off;
    k.mixed = a.mixed;
    k.part = a.part;
    k.ml = a.ml;
    k.scores = a.scores;
    k.col = g->col;
    k.perm = g->perm;
    k.items = g->items;
    k.n_items = g->n_items;
    k.n_parts = g->n_parts;
    k.nnz = g->nnz;
    k.B = (int)a.B;
    k.L = (int)g->L;
    k.S = (int)g->S;
    k.E = (int)a.E;
    k.H = (int)a.H;
    k.d = (int)(a.E / a.H);
    k.score_scale = a.score_scale;
    const long long warps = a.B * g->n_items;
    if (warps == 0) return PMHA_OK;
    StageTimer timer(a.with_values ? "edge_attn" : "edge_scores", s);
    bool ok;
    if (dt == TcType::F16)
        ok = a.with_values ? dispatch_cpl<__half, true>(cpl, k, warps, s)
                           : dispatch_cpl<__half, false>(cpl, k, warps, s);
    else
        ok = a.with_values ? dispatch_cpl<float, true>(cpl, k, warps, s) : dispatch_cpl<float, false>(cpl, k, warps, s);
    if (!ok) return PMHA_ERR_UNSUPPORTED;
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

pmha_status split_merge(TcType dt, const pmha_graph *g, const EdgeArgs &a, cudaStream_t s)
{
    if (g->n_heavy == 0) return PMHA_OK;
    const long long warps = a.B * g->n_heavy;
    const unsigned blocks = (unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
    const int d = (int)(a.E / a.H);
    StageTimer timer("split_merge", s);
    if (dt == TcType::F16) {
        if (a.with_values)
            k_split_merge<__half, true><<<blocks, kWarpsPerBlock * 32, 0, s>>>(
                g->heavy, g->n_heavy, a.part, g->n_parts, (int)a.B, (int)g->L, (int)a.E, (int)a.H, d, a.mixed, a.ml);
        else
            k_split_merge<__half, false><<<blocks, kWarpsPerBlock * 32, 0, s>>>(
                g->heavy, g->n_heavy, a.part, g->n_parts, (int)a.B, (int)g->L, (int)a.E, (int)a.H, d, a.mixed, a.ml);
    } else {
        if (a.with_values)
            k_split_merge<float, true><<<blocks, kWarpsPerBlock * 32, 0, s>>>(
                g->heavy, g->n_heavy, a.part, g->n_parts, (int)a.B, (int)g->L, (int)a.E, (int)a.H, d, a.mixed, a.ml);
        else
            k_split_merge<float, false><<<blocks, kWarpsPerBlock * 32, 0, s>>>(
                g->heavy, g->n_heavy, a.part, g->n_parts, (int)a.B, (int)g->L, (int)a.E, (int)a.H, d, a.mixed, a.ml);
    }
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

pmha_status weights_finalize(const pmha_graph *g, const EdgeArgs &a, pmha_wmode mode, float *out, cudaStream_t s)
{
    const long long n = a.B * g->nnz;
    if (n == 0) return PMHA_OK;
    const int TB = 256;
    StageTimer timer("weights", s);
    k_weights<<<(unsigned)((n + TB - 1) / TB), TB, 0, s>>>(a.scores, a.ml, g->tgt_of_edge, a.B, g->nnz, (int)g->L,
                                                           (int)a.H, mode == PMHA_WEIGHTS_AVG, out);
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

}  // namespace pmha
