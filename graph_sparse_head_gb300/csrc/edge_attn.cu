// Edge attention (kpnn2 PackedMultiheadAttention, Notes steps 2-4, and the
// paragraph after them: a target without live keys mixes to zeros): the
// choice of lane shape and the launch of the streaming kernel
// (edge_stream.cuh), the merge of targets that cross a unit boundary, and
// the per-edge weights in the given edge order.
#include <math.h>

#include "edge_ring.cuh"

#ifndef PMHA_EDGE_RING
#define PMHA_EDGE_RING 1
#endif

namespace pmha {
namespace {

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Targets without edges (paragraph after the Notes steps: they mix to
// zeros): one warp per (sample, merge-list target) writes the zero mix and
// (m, l) = (-inf, 0) for the targets without edges and skips the others
// (targets that cross a unit boundary, merged by the edge kernel itself).
template <typename T, bool WV>
__global__ void __launch_bounds__(256) k_empty_targets(const int32_t *__restrict__ merge_t, long long n_merge,
                                                       const int32_t *__restrict__ row_ptr, int B, int L, int E,
                                                       int H, void *mixed, float *ml)
{
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long long gw = (long long)blockIdx.x * 8 + wib;
    if (gw >= (long long)B * n_merge) return;
    const int b = (int)(gw / n_merge);
    const int t = merge_t[gw - (long long)b * n_merge];
    if (row_ptr[t] != row_ptr[t + 1]) return;
    if constexpr (WV) {
        T *mrow = (T *)mixed + ((long long)b * L + t) * E;
        for (int c = lane; c < E; c += 32) mrow[c] = T(0.f);
    }
    if (ml) {
        float *mlrow = ml + ((long long)b * L + t) * H * 2;
        for (int h = lane; h < H; h += 32) {
            mlrow[2 * h] = -INFINITY;
            mlrow[2 * h + 1] = 0.f;
        }
    }
}

// key_padding_mask per CSR position: warp w reads the sources of positions
// 32 w .. 32 w + 31 once and, for every sample b, sets bit p of word (b, w)
// when the source at position 32 w + p is dropped in b.
__global__ void __launch_bounds__(256) k_kpm_bits(const int32_t *__restrict__ col, long long nnz,
                                                  const uint8_t *__restrict__ kpm, int S, int B, long long n_kw,
                                                  uint32_t *__restrict__ bits)
{
    const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= n_kw) return;  // whole warps
    const long long pos = w * 32 + lane;
    const int src = pos < nnz ? col[pos] : -1;
#pragma unroll 4
    for (int b = 0; b < B; ++b) {
        const bool drop = src >= 0 && kpm[(long long)b * S + src] != 0;
        const unsigned word = __ballot_sync(0xffffffffu, drop);
        if (lane == 0) bits[(long long)b * n_kw + w] = word;
    }
}

// weights[b, e, h] = 2^(s - m) / l for the target of edge e; averaged over
// heads when out has one entry per edge. Runs in place when out == scores
// (per-head layout: each thread reads its H scores before writing them).
// HC = H known at compile time (every score and (m, l) pair of the edge is
// loaded with 16-byte loads before any arithmetic), or 0 for any H.
__device__ __forceinline__ float edge_weight(float s, float m, float l)
{
    // a dropped key (score -inf) or a target with no live key (l = 0) weighs 0
    return (l == 0.f || s == -INFINITY) ? 0.f : __fmul_rn(ex2(__fsub_rn(s, m)), __frcp_rn(l));
}

// The edges are walked in CSR order, so the scores (written at CSR positions
// by the edge kernel) and the targets' (m, l) are read in sequence; each
// weight goes to its given-order place (the averaged weights, 4 bytes an
// edge, are a small array that stays in L2 while it fills).
template <int HC>
__global__ void __launch_bounds__(256) k_weights(const float *__restrict__ scores, const float *__restrict__ ml,
                                                 const int32_t *__restrict__ tgt_of_pos,
                                                 const int32_t *__restrict__ perm, long long B, long long nnz,
                                                 int L, int H_rt, bool average, float *out)
{
    const long long si = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (sample, CSR position)
    if (si >= B * nnz) return;
    const long long b = si / nnz, p = si - b * nnz;
    const int t = __ldg(tgt_of_pos + p);
    const long long i = b * nnz + __ldg(perm + p);  // (sample, given-order edge id)
    if constexpr (HC > 0) {
        static_assert(HC % 4 == 0, "16-byte loads of the scores");
        float s[HC], st[2 * HC];
#pragma unroll
        for (int j = 0; j < HC / 4; ++j) {
            const float4 v = reinterpret_cast<const float4 *>(scores + si * HC)[j];
            s[4 * j] = v.x;
            s[4 * j + 1] = v.y;
            s[4 * j + 2] = v.z;
            s[4 * j + 3] = v.w;
        }
        const float4 *mlp = reinterpret_cast<const float4 *>(ml + ((b * L + t) * HC) * 2);
#pragma unroll
        for (int j = 0; j < HC / 2; ++j) {
            const float4 v = __ldg(mlp + j);
            st[4 * j] = v.x;
            st[4 * j + 1] = v.y;
            st[4 * j + 2] = v.z;
            st[4 * j + 3] = v.w;
        }
        float w[HC], sum = 0.f;
#pragma unroll
        for (int h = 0; h < HC; ++h) {
            w[h] = edge_weight(s[h], st[2 * h], st[2 * h + 1]);
            sum = __fadd_rn(sum, w[h]);
        }
        if (average) {
            out[i] = __fdiv_rn(sum, (float)HC);
        } else {
#pragma unroll
            for (int j = 0; j < HC / 4; ++j)
                reinterpret_cast<float4 *>(out + i * HC)[j] = make_float4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
    } else {
        const int H = H_rt;
        const float *s = scores + si * H;
        const float *st = ml + ((b * L + t) * H) * 2;
        float sum = 0.f;
        for (int h = 0; h < H; ++h) {
            const float w = edge_weight(s[h], st[2 * h], st[2 * h + 1]);
            if (average) sum = __fadd_rn(sum, w);
            else out[i * H + h] = w;
        }
        if (average) out[i] = __fdiv_rn(sum, (float)H);
    }
}

// Lane shape: a lane owns CPL channels (a whole head when the head has at
// most 16 fp16 / 8 fp32 channels), LPE = E / CPL lanes own a row; both
// powers of two, LPE <= 32.
bool pick_shape(int64_t E, int64_t d, TcType t, int *cpl, int *lpe)
{
    auto pow2 = [](int64_t x) { return x > 0 && (x & (x - 1)) == 0; };
#ifndef PMHA_STREAM_HALF_CPL_MAX
#define PMHA_STREAM_HALF_CPL_MAX 16
#endif
    const int64_t cmax = t == TcType::F32 ? 8 : PMHA_STREAM_HALF_CPL_MAX;
    const int64_t cmin = t == TcType::F32 ? 4 : 8;
    if (!pow2(d) || d < cmin) return false;
    const int64_t c = d < cmax ? d : cmax;
    if (E % c || !pow2(E / c) || E / c < 2 || E / c > 32) return false;
    *cpl = (int)c;
    *lpe = (int)(E / c);
    return true;
}

}  // namespace

bool fused_out_supported(TcType t, int64_t E, int64_t H)
{
    int cpl, lpe;
    if (!PMHA_EDGE_RING || t != TcType::F16 || H < 1 || E % H || !pick_shape(E, E / H, t, &cpl, &lpe)) return false;
    return cpl == 16 && lpe == 8;
}

bool edge_supported(int64_t E, int64_t H, TcType t)
{
    int cpl, lpe;
    if (H < 1 || E % H) return false;
    return pick_shape(E, E / H, t, &cpl, &lpe);
}

pmha_status edge_attention(TcType dt, const pmha_graph *g, const EdgeArgs &a, cudaStream_t s)
{
    int cpl, lpe;
    if (!pick_shape(a.E, a.E / a.H, dt, &cpl, &lpe)) {
        set_error("edge_attention: no kernel for embed_dim %lld, num_heads %lld", (long long)a.E, (long long)a.H);
        return PMHA_ERR_UNSUPPORTED;
    }
    stream::Args k;
    k.q = a.q;
    k.q_ld = a.q_ld;
    k.kv = a.kv;
    k.kv_ld = a.kv_ld;
    k.v_off = a.v_off;
    k.mixed = a.mixed;
    k.part = a.part;
    k.ml = a.ml;
    k.scores = a.scores;
    k.row_ptr = g->row_ptr;
    k.col = g->col;
    k.unit_first_t = g->unit_first_t;
    k.unit_order = g->unit_order;
    k.task_counter = (unsigned *)a.counters;  // the first word of the counter region
    k.kpm = a.kpm;
    k.kpm_bits = a.kpm_bits;
    k.n_kw = (g->nnz + 31) / 32;
    k.counters = a.counters + kCounterHead;
    k.merge_pos = g->merge_pos;
    k.n_merge = g->n_merge;
    k.n_units = g->n_units;
    k.nnz = g->nnz;
    k.B = (int)a.B;
    k.L = (int)g->L;
    k.S = (int)g->S;
    k.E = (int)a.E;
    k.H = (int)a.H;
    k.d = (int)(a.E / a.H);
    k.score_scale = a.score_scale;
    const bool fused = a.out != nullptr;
    if (fused && (!a.with_values || !a.wo_frag || !fused_out_supported(dt, a.E, a.H))) {
        set_error("edge attention: no fused out_proj for embed_dim %lld, num_heads %lld", (long long)a.E,
                  (long long)a.H);
        return PMHA_ERR_UNSUPPORTED;
    }
    k.out = a.out;
    k.wo_frag = (const uint32_t *)a.wo_frag;
    k.bo = a.bo;
    k.n_blk = (int)out_blocks(g->L);
    k.blk_count = k.counters + a.B * g->n_merge;
    k.err = device_error_word();
    if (!k.err) return PMHA_ERR_CUDA;
    const long long slots = a.B * g->n_units;
    if (slots == 0) return PMHA_OK;
    if (a.v_off != a.E) {  // the kernel copies a row's k and v bytes as one run
        set_error("edge attention: v must follow k in the projected rows");
        return PMHA_ERR_UNSUPPORTED;
    }
    if (a.kpm) {
        // the mask per CSR position, as bits
        StageTimer bits_timer("kpm_bits", s);
        k_kpm_bits<<<(unsigned)((k.n_kw + 7) / 8), 256, 0, s>>>(g->col, g->nnz, a.kpm, (int)g->S, (int)a.B, k.n_kw,
                                                               a.kpm_bits);
        count_launch();
    }
    // the ring kernel's task counter and the arrival counts of the pieces of
    // crossing targets (the edge kernel merges them)
    // (and, with out_proj tasks, the finished targets per block)
    PMHA_CUDA_TRY(cudaMemsetAsync(
        a.counters, 0, (size_t)(kCounterHead + a.B * g->n_merge + (fused ? a.B * k.n_blk : 0)) * 4, s));
    StageTimer timer(fused ? "edge_attn_out" : (a.with_values ? "edge_attn" : "edge_scores"), s);
    // fp16 rows of 16 channels a lane and 8 to 32 lanes: the ring kernel
    // (edge_ring.cuh); other shapes and float32 layers: the streaming kernel
    const bool ring = PMHA_EDGE_RING && dt == TcType::F16 && cpl == 16 && lpe >= 8;
    const pmha_status st = fused ? stream::launch_ring_out_f16(lpe, k, s)
                           : ring ? stream::launch_ring_f16(lpe, a.with_values, k, s)
                           : dt == TcType::F16 ? stream::launch_f16(cpl, lpe, a.with_values, k, slots, s)
                                               : stream::launch_f32(cpl, lpe, a.with_values, k, slots, s);
    if (st != PMHA_OK) return st;
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

// Targets that cross a unit boundary are merged inside the edge kernel (by
// the slot that writes their last piece); this launch only gives the targets
// without edges their zero mix and (m, l) = (-inf, 0).
pmha_status empty_targets(TcType dt, const pmha_graph *g, const EdgeArgs &a, cudaStream_t s)
{
    if (g->n_merge == 0 || g->n_empty == 0) return PMHA_OK;
    const long long warps = a.B * g->n_merge;
    const unsigned blocks = (unsigned)((warps + 7) / 8);
    StageTimer timer("empty_targets", s);
    auto go = [&](auto kern) {
        kern<<<blocks, 256, 0, s>>>(g->merge_t, g->n_merge, g->row_ptr, (int)a.B, (int)g->L, (int)a.E, (int)a.H,
                                    a.mixed, a.ml);
    };
    if (dt == TcType::F16) {
        if (a.with_values) go(k_empty_targets<__half, true>);
        else go(k_empty_targets<__half, false>);
    } else {
        if (a.with_values) go(k_empty_targets<float, true>);
        else go(k_empty_targets<float, false>);
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
    const unsigned blocks = (unsigned)((n + TB - 1) / TB);
    const bool avg = mode == PMHA_WEIGHTS_AVG;
    // the 16-byte loads need 16-byte aligned scores, (m, l) and per-head output rows
    const bool vec = ((uintptr_t)a.scores % 16 == 0) && ((uintptr_t)a.ml % 16 == 0) &&
                     (avg || (uintptr_t)out % 16 == 0);
    if (vec && a.H == 8)
        k_weights<8><<<blocks, TB, 0, s>>>(a.scores, a.ml, g->tgt_of_pos, g->perm, a.B, g->nnz, (int)g->L, 8, avg, out);
    else if (vec && a.H == 4)
        k_weights<4><<<blocks, TB, 0, s>>>(a.scores, a.ml, g->tgt_of_pos, g->perm, a.B, g->nnz, (int)g->L, 4, avg, out);
    else if (vec && a.H == 16)
        k_weights<16><<<blocks, TB, 0, s>>>(a.scores, a.ml, g->tgt_of_pos, g->perm, a.B, g->nnz, (int)g->L, 16, avg, out);
    else
        k_weights<0><<<blocks, TB, 0, s>>>(a.scores, a.ml, g->tgt_of_pos, g->perm, a.B, g->nnz, (int)g->L, (int)a.H, avg,
                                           out);
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

}  // namespace pmha
