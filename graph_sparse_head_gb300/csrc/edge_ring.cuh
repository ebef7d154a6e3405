// The edge-attention kernel for fp16 intermediates with 16 channels a lane
// (kpnn2 PackedMultiheadAttention, Notes steps 2-4; a target without live
// keys mixes to zeros), for rows of 8 to 32 lanes (embed_dim 128 to 512,
// heads of at least 16 channels).
//
// Work decomposition (as in edge_stream.cuh): the CSR positions of one
// sample are cut into units of kUnitEdges consecutive positions; a warp
// walks one unit for P = 32 / LPE consecutive samples at once (a "slot" of
// LPE lanes per sample, a lane owning 16 channels), so the slots never
// diverge. A target inside one unit is finished there; a target crossing a
// unit boundary leaves partial softmax states and the slot that writes its
// last piece merges them in unit order.
//
// What this kernel adds:
//  * Everything a step reads comes through one per-warp ring of shared-
//    memory stages that cp.async fills kRDepth edges ahead: the source's k
//    and v rows and, when the edge is the first of a target, that target's
//    q rows (an issuing cursor walks the target bounds ahead of the
//    consumer). A target switch therefore never waits on a q row from DRAM;
//    with in-degrees of 1 to 3 (most targets of a power-law graph) that
//    wait was the cost of a switch.
//  * Each cp.async instruction copies whole 128-byte lines of one slot's
//    row (lane grp copies 16-byte chunks q * LPE + grp to their own place),
//    so a quarter-warp fills 8 consecutive chunks. A lane reads its two
//    chunks 2 grp and 2 grp + 1 in the order 2 grp + sw, 2 grp + 1 - sw
//    with sw = (grp >> 2) & 1, so the 8 lanes of a quarter-warp touch 8
//    distinct 16-byte bank groups on each read: no shared-memory bank
//    conflicts on either side. A lane with sw = 1 therefore holds its two
//    chunks swapped; its q and k are swapped alike (the dot product does not
//    care), and its mix is swapped back when stored.
//  * Source indices and target bounds come from 32-wide windows shared by
//    the whole warp (one coalesced load per 32 positions or targets).
//    Slots past the batch compute on the last sample and store nothing, so
//    the warp stays converged for the shuffles and votes.
//  * The mix takes mixed-precision FMAs (fp16 value x fp16 weight, fp32
//    accumulate): the weight 2^(s - m) <= 2^8 is rounded to fp16 for the mix
//    only (relative error 2^-11); the running sum l, the (m, l) pair and the
//    returned weights keep fp32.
#pragma once

#include <algorithm>

#include "edge_out.cuh"
#include "edge_stream.cuh"

namespace pmha {
namespace stream {

#ifndef PMHA_RING_DEPTH
#define PMHA_RING_DEPTH 4
#endif
#ifndef PMHA_RING_WARPS
#define PMHA_RING_WARPS 2
#endif
#ifndef PMHA_RING_MIX_F16
#define PMHA_RING_MIX_F16 1
#endif
#ifndef PMHA_RING_EARLY
#define PMHA_RING_EARLY 1
#endif
#ifndef PMHA_RING_ACQREL
#define PMHA_RING_ACQREL 1
#endif

constexpr int kRWarps = PMHA_RING_WARPS;  // warps per block
constexpr int kRDepth = PMHA_RING_DEPTH;  // edges in flight ahead of the pair being read (even)
// Early release: a step reads its k and v rows into registers first and
// refills the same two stages at once, so kRDepth stages keep kRDepth edges
// in flight; otherwise a stage is refilled one step after it was read.
constexpr bool kREarly = PMHA_RING_EARLY;
constexpr int kRRing = kREarly ? kRDepth : kRDepth + 2;
constexpr int kRCB = 32;                  // bytes of one row per lane: 16 fp16 channels
static_assert(kRDepth % 2 == 0 && kRDepth >= 2, "edges go two per step");

template <bool WV>
__host__ __device__ constexpr int ring_stage_bytes()
{
    return ((WV ? 2 : 1) + 1) * 32 * kRCB;  // k (and v) rows, then q rows, of the warp's slots
}
template <bool WV>
__host__ __device__ constexpr int ring_smem_bytes()
{
    return kRWarps * kRRing * ring_stage_bytes<WV>();
}
// With out_proj tasks (edge_out.cuh, embed_dim 128): one block of kFOWarps
// warps per SM, their rings, then Wo (fp16, wo_frag_pos order) and bo (fp32)
// for the whole block, loaded once: 16 x 12 KB + 32 KB + 512 B.
constexpr int kFOWarps = 16;
constexpr int kFOE = 128;
__host__ __device__ constexpr int ring_fo_wo_offset() { return kFOWarps * kRRing * ring_stage_bytes<true>(); }
__host__ __device__ constexpr int ring_fo_smem_bytes() { return ring_fo_wo_offset() + kFOE * kFOE * 2 + kFOE * 4; }

// 32 bytes of shared memory as two 16-byte loads, from a0 and from a1
__device__ __forceinline__ Raw<32> lds_pair(uint32_t a0, uint32_t a1)
{
    Raw<32> r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
                 : "r"(a0));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.w[4]), "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
                 : "r"(a1));
    return r;
}

// Orders this thread's prior global writes before its later ones and its
// later reads after earlier acquires (release and acquire at GPU scope; the
// pieces of a crossing target are published and read across CTAs with it).
__device__ __forceinline__ void fence_gpu()
{
#if PMHA_RING_ACQREL
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
#else
    __threadfence();
#endif
}

// x += p * v.lo, y += p * v.hi: fp16 operands, fp32 accumulate, one rounding
__device__ __forceinline__ void fma_h2p(float &x, float &y, uint32_t v, uint16_t p)
{
    asm("{\n\t.reg .b16 a0, a1;\n\tmov.b32 {a0, a1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, %3, %0;\n\tfma.rn.f32.f16 %1, a1, %3, %1;\n\t}"
        : "+f"(x), "+f"(y)
        : "r"(v), "h"(p));
}

// WV: mix values (else scores and (m, l) only); WS: write raw scores;
// KPM: read a key_padding_mask (a dropped key scores -inf); FO: out_proj
// tasks in the queue (edge_out.cuh).
template <int LPE, bool WV, bool WS, bool KPM, bool FO>
__global__ void __launch_bounds__((FO ? kFOWarps : kRWarps) * 32, FO ? 1 : 16 / kRWarps) k_edge_ring(Args a)
{
    static_assert(LPE >= 8 && LPE <= 32, "8 to 32 lanes per row");
    static_assert(!FO || (WV && 16 * LPE == kFOE), "out_proj needs the mixed rows, embed_dim 128");
    constexpr int P = 32 / LPE;             // slots (samples) per warp
    constexpr int NR = WV ? 2 : 1;          // row parts staged per edge: k (and v)
    constexpr int PART = LPE * kRCB;        // bytes of one row part of one slot
    constexpr int SLOT_ROW = NR * PART;     // a slot's k|v bytes in a stage
    constexpr int QOFF = NR * 32 * kRCB;    // q rows of the stage
    constexpr int STAGE = ring_stage_bytes<WV>();
    constexpr unsigned kAll = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char smem_dyn[];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slot = lane / LPE, grp = lane % LPE;
    const int c0 = grp * 16;
    const int head = c0 / a.d;
    const int lph = a.d / 16;  // lanes per head
    const int sw = (grp >> 2) & 1;  // the lane's two chunks sit swapped in shared memory

    // ---- shared-memory addresses (stage offsets are added per step)
    const uint32_t wbase = smem_u32(smem_dyn) + (uint32_t)(warp * kRRing * STAGE);
    if constexpr (FO) {
        // the block's copy of Wo (fragment order) and bo (fp32), read by every out_proj task
        const uint4 *wsrc = reinterpret_cast<const uint4 *>(a.wo_frag);
        uint4 *wdst = reinterpret_cast<uint4 *>(smem_dyn + ring_fo_wo_offset());
        for (int i = threadIdx.x; i < kFOE * kFOE * 2 / 16; i += blockDim.x) wdst[i] = wsrc[i];
        float *bs = reinterpret_cast<float *>(smem_dyn + ring_fo_wo_offset() + kFOE * kFOE * 2);
        const unsigned short *bo = (const unsigned short *)a.bo;
        for (int i = threadIdx.x; i < kFOE; i += blockDim.x)
            bs[i] = bo ? __bfloat162float(__ushort_as_bfloat16(bo[i])) : 0.f;
        __syncthreads();
    }
    // reads: the lane's first and second 16-byte chunk (swapped when sw = 1)
    const uint32_t rd_kv0 = wbase + (uint32_t)(slot * SLOT_ROW + 32 * grp + 16 * sw);
    const uint32_t rd_kv1 = wbase + (uint32_t)(slot * SLOT_ROW + 32 * grp + 16 * (1 - sw));
    const uint32_t rd_q0 = wbase + (uint32_t)(QOFF + slot * PART + 32 * grp + 16 * sw);
    const uint32_t rd_q1 = wbase + (uint32_t)(QOFF + slot * PART + 32 * grp + 16 * (1 - sw));
    // fills: chunk q * LPE + grp of a row part lands at its own place
    const uint32_t fill_kv = wbase + (uint32_t)(slot * SLOT_ROW + 16 * grp);
    const uint32_t fill_q = wbase + (uint32_t)(QOFF + slot * PART + 16 * grp);

    // Persistent warps: each takes tasks (sample group, unit) from one queue,
    // sample groups in order (their k|v rows stay in L2 meanwhile), within a
    // group the units with the most estimated work first, so the last tasks
    // to start are short ones. With FO the out_proj tasks (a block of
    // kOutRows targets of one sample each) follow all edge tasks, group by
    // group: the warps that run out of edge tasks take the blocks of the
    // groups already done while the last units finish.
    const unsigned n_groups = (unsigned)((a.B + P - 1) / P);
    const unsigned n_u = (unsigned)a.n_units;
    const unsigned n_o = FO ? (unsigned)(P * a.n_blk) : 0u;
    const unsigned n_tasks = n_groups * (n_u + n_o);
    for (;;) {
    unsigned task = 0;
    if (lane == 0) task = atomicAdd(a.task_counter, 1u);
    task = __shfl_sync(kAll, task, 0);
    if (task >= n_tasks) break;
    unsigned grp_i = task / n_u, idx = task % n_u;
    if constexpr (FO) {
        if (task >= n_groups * n_u) {
            const unsigned y = task - n_groups * n_u;
            grp_i = y / n_o;
            idx = y % n_o;
            const int bb = (int)grp_i * P + (int)(idx % P);
            if (bb < a.B)
                out_proj_block<kFOE, kRRing * STAGE>(a, bb, (int)(idx / P), wbase,
                                                     smem_u32(smem_dyn) + (uint32_t)ring_fo_wo_offset(), lane);
            continue;
        }
    }
    const int u = a.unit_order[idx];
    const int b_slot = (int)grp_i * P + slot;
    const bool own = b_slot < a.B;  // slots past the batch store nothing
    const int b = own ? b_slot : a.B - 1;
    const int e0 = u * kUnitEdges;
    const int n = (int)min((long long)kUnitEdges, a.nnz - e0);
    const int e1 = e0 + n;
    const bool head_leader = own && (grp & (lph - 1)) == 0;

    // ---- global rows (byte pointers at this lane's first chunk)
    const char *KV0 = (const char *)a.kv + (long long)b * a.S * a.kv_ld * 2 + 16 * grp;
    const unsigned kv_row = (unsigned)(a.kv_ld * 2);  // row pitches in bytes (< 2^32)
    const char *Q0 = (const char *)a.q + (long long)b * a.L * a.q_ld * 2 + 16 * grp;
    const unsigned q_row = (unsigned)(a.q_ld * 2);
    float *scores_b = WS ? a.scores + (long long)b * a.nnz * a.H : nullptr;
    const int32_t *colu = a.col + e0;

    auto copy_kv = [&](uint32_t st, int s) {
        const char *src = KV0 + (unsigned long long)(unsigned)s * kv_row;  // one 32 x 32 -> 64-bit multiply-add
        static_for<0, 2 * NR>([&](auto qc) {
            constexpr int q = decltype(qc)::value;
            constexpr int doff = (q / 2) * PART + (q % 2) * (PART / 2);
            cp_async16_at<doff, 16 * q * LPE>(fill_kv + st, src);
        });
    };
    auto copy_q = [&](uint32_t st, int t) {
        const char *src = Q0 + (unsigned long long)(unsigned)t * q_row;
        cp_async16_at<0, 0>(fill_q + st, src);
        cp_async16_at<PART / 2, 16 * LPE>(fill_q + st, src);
    };

    // ---- 32-wide windows of source indices: lane i holds col[e0 + 32 w + i]
    auto ldcol = [&](int w) -> int {
        const int p = 32 * w + lane;
        return p < n ? colu[p] : 0;
    };
    int cwi = 0;
    int cw_cur = ldcol(0), cw_nxt = ldcol(1);

    // ---- target bounds: a window of 32 targets, lane i holds row_ptr[tw + i + 1]
    struct Bounds {
        int tw, cur, nxt;
    };
    auto ldrp = [&](int tt) -> int { return tt < a.L ? a.row_ptr[tt + 1] : (int)a.nnz; };
    auto end_in = [&](Bounds &w, int tt) -> int {  // row_ptr[tt + 1]; tt never decreases
        while (tt - w.tw >= 32) {
            w.tw += 32;
            w.cur = w.nxt;
            w.nxt = ldrp(w.tw + 32 + lane);
        }
        return __shfl_sync(kAll, w.cur, tt - w.tw);
    };
    const int t_first = a.unit_first_t[u];
    // issuing cursor: the target of the position being issued
    Bounds wi{t_first, ldrp(t_first + lane), ldrp(t_first + 32 + lane)};
    int ti = t_first;
    int bi = end_in(wi, ti);

    // positions j, j + 1 (j even; both in one 32-window) into stages sj, sj + 1;
    // the first position of a target also brings its q rows
    auto issue2 = [&](int j, int sj) {
        if (j >= 32 * (cwi + 1)) {
            ++cwi;
            cw_cur = cw_nxt;
            cw_nxt = ldcol(cwi + 1);
        }
        const int s0 = __shfl_sync(kAll, cw_cur, j & 31);
        const int s1 = __shfl_sync(kAll, cw_cur, (j + 1) & 31);
        const uint32_t st0 = (uint32_t)(sj * STAGE);
        if (j < n) {
            copy_kv(st0, s0);
            if (e0 + j >= bi) {
                do {
                    ++ti;
                    bi = end_in(wi, ti);
                } while (bi <= e0 + j);
                copy_q(st0, ti);
            }
        }
        if (j + 1 < n) {
            copy_kv(st0 + STAGE, s1);
            if (e0 + j + 1 >= bi) {
                do {
                    ++ti;
                    bi = end_in(wi, ti);
                } while (bi <= e0 + j + 1);
                copy_q(st0 + STAGE, ti);
            }
        }
        cp_async_commit();
    };
    // prologue: the unit's first target's q rows with its first edge
    copy_q(0, t_first);
#pragma unroll
    for (int j = 0; j < kRDepth; j += 2) issue2(j, j);
    static_assert(!kREarly || kRRing == kRDepth, "early release keeps every stage in flight");

    // ---- key_padding_mask per CSR position (one bit each, 32 positions a word)
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

    // ---- consumer state
    Bounds wc{t_first, ldrp(t_first + lane), ldrp(t_first + 32 + lane)};
    int t = t_first;
    int bound = end_in(wc, t);
    const bool first_started_here = a.row_ptr[t] == e0;
    bool is_first = true;
    // FO: targets whose final row this slot wrote, in block cur_blk, not yet counted
    int cur_blk = t_first / kOutRows, fin_cnt = 0;
    auto count_block = [&]() {
        if constexpr (FO) {
            fence_gpu();
            __syncwarp(kAll);
            if (grp == 0 && fin_cnt) atomicAdd(a.blk_count + (long long)b * a.n_blk + cur_blk, fin_cnt);
            fin_cnt = 0;
        }
    };
    Raw<kRCB> qr;
    float m = -INFINITY, l = 0.f;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;

    // the lane's 16 mixed channels (v * inv), stored in row order
    auto write_mixed = [&](const float (&v)[16], float inv) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            __half2 h = __floats2half2_rn(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv));
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        char *row = (char *)a.mixed + (((long long)b * a.L + t) * a.E + c0) * 2;
        *reinterpret_cast<uint4 *>(row + 16 * sw) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4 *>(row + 16 * (1 - sw)) = make_uint4(w[4], w[5], w[6], w[7]);
    };

    // Combine the partial states (m, l, acc) of target t's pieces in unit
    // order, in one pass with a running maximum M: a piece with m_i > M first
    // rescales L and acc by 2^(M - m_i); then L += l_i 2^(m_i - M) and acc +=
    // acc_i 2^(m_i - M). An empty piece (every key dropped: m = -inf, l = 0)
    // adds nothing. Pieces are pulled into L1 eight ahead of their use, so the
    // pass is not a chain of L2 round trips (a target with thousands of edges
    // has dozens of pieces).
    auto merge_pieces = [&](int beg, int u0, int n_pieces) {
        const long long stride = 2 * a.H + a.E;
        const float *base = a.part + (long long)b * 2 * a.n_units * stride;
        auto piece = [&](int i) -> const float * {
            const int sid = 2 * (u0 + i) + ((i == 0 && beg != u0 * kUnitEdges) ? 1 : 0);
            return base + (long long)sid * stride;
        };
        auto pull = [&](int i) {
            if (i < n_pieces) {
                const float *pp = piece(i);
                asm volatile("prefetch.global.L1 [%0];" ::"l"(pp + head));
                if constexpr (WV) asm volatile("prefetch.global.L1 [%0];" ::"l"(pp + 2 * a.H + c0));
            }
        };
#pragma unroll
        for (int i = 0; i < 8; ++i) pull(i);
        float Mh = -INFINITY, Lh = 0.f;
        float macc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) macc[j] = 0.f;
        for (int i = 0; i < n_pieces; ++i) {
            pull(i + 8);
            const float *pp = piece(i);
            const float mi = pp[head], li = pp[a.H + head];
            if (mi > Mh) {
                const float sc = ex2(__fsub_rn(Mh, mi));  // 0 while M is -inf
                Lh = __fmul_rn(Lh, sc);
                if constexpr (WV) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) macc[j] = __fmul_rn(macc[j], sc);
                }
                Mh = mi;
            }
            const float w = mi == -INFINITY ? 0.f : ex2(__fsub_rn(mi, Mh));
            Lh = __fmaf_rn(li, w, Lh);
            if constexpr (WV) {
                // a piece row is 2H + E floats: 8-byte aligned for any H
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 v = reinterpret_cast<const float2 *>(pp + 2 * a.H + c0)[j];
                    macc[2 * j] = __fmaf_rn(v.x, w, macc[2 * j]);
                    macc[2 * j + 1] = __fmaf_rn(v.y, w, macc[2 * j + 1]);
                }
            }
        }
        if (a.ml && head_leader) {
            float *q = a.ml + (((long long)b * a.L + t) * a.H + head) * 2;
            q[0] = Mh;
            q[1] = Lh;
        }
        if constexpr (WV) write_mixed(macc, Lh > 0.f ? __frcp_rn(Lh) : 0.f);
    };

    // finish target t in this unit: a complete target writes its result, a
    // target crossing a unit boundary its partial state
    auto finish = [&]() {
        const bool complete = (is_first ? first_started_here : true) && bound <= e1;
        if (complete) {
            if (own) {
                if constexpr (FO) ++fin_cnt;
                if constexpr (WV) write_mixed(acc, l > 0.f ? __frcp_rn(l) : 0.f);
                if (a.ml && head_leader) {
                    float *p = a.ml + (((long long)b * a.L + t) * a.H + head) * 2;
                    p[0] = m;
                    p[1] = l;
                }
            }
        } else {
            const int slot_id = 2 * u + (is_first ? 0 : 1);
            float *p = a.part + ((long long)b * 2 * a.n_units + slot_id) * (2 * a.H + a.E);
            if (own) {
                if (head_leader) {
                    p[head] = m;
                    p[a.H + head] = l;
                }
                if constexpr (WV) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        reinterpret_cast<float2 *>(p + 2 * a.H + c0)[j] = make_float2(acc[2 * j], acc[2 * j + 1]);
                }
            }
            // The slot that writes a target's last piece merges all its
            // pieces: each writer publishes its piece (fence) and counts it;
            // the one that completes the count reads every piece in piece order.
            fence_gpu();
            __syncwarp(kAll);
            const int beg = a.row_ptr[t], end = a.row_ptr[t + 1];
            const int u0 = beg / kUnitEdges, n_pieces = (end - 1) / kUnitEdges - u0 + 1;
            int prev = 0;
            if (grp == 0 && own) prev = atomicAdd(a.counters + (long long)b * a.n_merge + a.merge_pos[t], 1);
            prev = __shfl_sync(kAll, prev, slot * LPE);
            if (own && prev == n_pieces - 1) {
                fence_gpu();
                merge_pieces(beg, u0, n_pieces);
                if constexpr (FO) ++fin_cnt;
            }
        }
    };
    auto set_q = [&](uint32_t st) { qr = lds_pair(rd_q0 + st, rd_q1 + st); };
    // move from t to the target of position pos (> the end of t); its q rows
    // sit in stage st
    auto advance = [&](int pos, uint32_t st) {
        finish();
        is_first = false;
        do {
            ++t;
            bound = end_in(wc, t);
        } while (bound <= pos);
        if constexpr (FO) {
            if (t / kOutRows != cur_blk) {
                count_block();
                cur_blk = t / kOutRows;
            }
        }
        set_q(st);
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    };
    // the head's score of one staged k row (two independent partial sums)
    auto score = [&](const Raw<kRCB> &kr) -> float {
        float ax = 0.f, ay = 0.f, bx = 0.f, by = 0.f;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            fma_h2(ax, ay, qr.w[i], kr.w[i]);
            fma_h2(bx, by, qr.w[i + 1], kr.w[i + 1]);
        }
        float dot = __fadd_rn(__fadd_rn(ax, bx), __fadd_rn(ay, by));
        for (int o = 1; o < lph; o <<= 1) dot = __fadd_rn(dot, __shfl_xor_sync(kAll, dot, o));
        return __fmul_rn(dot, a.score_scale);
    };
    auto mix = [&](const Raw<kRCB> &vr, float p) {
#if PMHA_RING_MIX_F16
        const __half ph = __float2half_rn(p);
        const uint16_t pb = __half_as_ushort(ph);
#pragma unroll
        for (int i = 0; i < 8; ++i) fma_h2p(acc[2 * i], acc[2 * i + 1], vr.w[i], pb);
#else
        const f2 p2 = pk(p, p);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&vr.w[i]));
            const float2 r = upk(ffma2(p2, pk(x.x, x.y), pk(acc[2 * i], acc[2 * i + 1])));
            acc[2 * i] = r.x;
            acc[2 * i + 1] = r.y;
        }
#endif
    };
    auto rescale = [&](float scale) {
        const f2 s2 = pk(scale, scale);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float2 r = upk(fmul2(pk(acc[2 * i], acc[2 * i + 1]), s2));
            acc[2 * i] = r.x;
            acc[2 * i + 1] = r.y;
        }
    };
    // Move the reference m to mx where mx > m + kLazy (m = -inf: any finite
    // mx), rescaling l and acc; the vote keeps the branch uniform over the warp.
    auto lift = [&](float mx) {
        const bool move = mx > __fadd_rn(m, kLazy);
        if (__any_sync(kAll, move)) {
            const float scale = !move ? 1.f : (m == -INFINITY ? 0.f : ex2(__fsub_rn(m, mx)));
            l = __fmul_rn(l, scale);
            if constexpr (WV) rescale(scale);
            if (move) m = mx;
        }
    };
    // one edge through the online softmax (used at target boundaries)
    auto one = [&](int j, const Raw<kRCB> &kr, uint32_t st) {
        const int pos = e0 + j;
        if (pos >= bound) advance(pos, st);
        float dot = score(kr);
        Raw<kRCB> vr;
        if constexpr (WV) vr = lds_pair(rd_kv0 + st + PART, rd_kv1 + st + PART);
        if constexpr (KPM)
            if (masked(j)) dot = -INFINITY;
        if constexpr (WS)
            if (head_leader) scores_b[(long long)(e0 + j) * a.H + head] = dot;
        lift(dot);
        // ex2.approx(-inf) is +0, so a dropped edge gives p = 0 once some key
        // is live; before that m is -inf and the offset 0 avoids -inf - -inf
        const float p = ex2(__fsub_rn(dot, (KPM && m == -INFINITY) ? 0.f : m));
        l = __fadd_rn(l, p);
        if constexpr (WV) mix(vr, p);
    };

    // the first stages (and the unit's first q rows) have landed
    cp_async_wait<kRDepth / 2 - 1>();
    __syncwarp(kAll);
    set_q(0);

    // rs = j mod kRRing, stepped by 2 with a wrap. Without early release,
    // edge j + kRDepth goes to stage (rs + kRDepth) mod kRRing = the stage
    // read one step earlier; with it, edge j + kRRing goes to the stage of
    // edge j as soon as this step has its rows in registers (a step with a
    // target switch reads q and v from the stages as it goes, and refills
    // them at its end).
    int rs = 0;
    for (int j = 0; j < n; j += 2) {
        cp_async_wait<kRDepth / 2 - 1>();
        __syncwarp(kAll);  // the other lanes' chunks of these rows
        const uint32_t st0 = (uint32_t)(rs * STAGE);
        const uint32_t st1 = st0 + (uint32_t)STAGE;
        const int rs_now = rs;
        const Raw<kRCB> kr0 = lds_pair(rd_kv0 + st0, rd_kv1 + st0);
        const Raw<kRCB> kr1 = lds_pair(rd_kv0 + st1, rd_kv1 + st1);
        if constexpr (!kREarly) issue2(j + kRDepth, rs == 0 ? kRRing - 2 : rs - 2);
        rs = rs + 2 == kRRing ? 0 : rs + 2;

        const int pos = e0 + j;
        if (j + 1 < n && pos + 1 < bound) {
            // both edges belong to t: two independent scores, one rescale
            Raw<kRCB> vr0, vr1;
            if constexpr (WV && kREarly) {
                vr0 = lds_pair(rd_kv0 + st0 + PART, rd_kv1 + st0 + PART);
                vr1 = lds_pair(rd_kv0 + st1 + PART, rd_kv1 + st1 + PART);
            }
            float d0 = score(kr0), d1 = score(kr1);
            if constexpr (kREarly) {
                // every lane's loads of both stages have returned (each of
                // the four 16-byte loads of v is read once) before the
                // warp refills them
                if constexpr (WV) {
                    const uint32_t touch = vr0.w[0] ^ vr0.w[4] ^ vr1.w[0] ^ vr1.w[4];
                    asm volatile("" ::"r"(touch));
                }
                __syncwarp(kAll);
                issue2(j + kRRing, rs_now);
            }
            if constexpr (WV && !kREarly) {
                vr0 = lds_pair(rd_kv0 + st0 + PART, rd_kv1 + st0 + PART);
                vr1 = lds_pair(rd_kv0 + st1 + PART, rd_kv1 + st1 + PART);
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
            one(j, kr0, st0);
            if (j + 1 < n) one(j + 1, kr1, st1);
            if constexpr (kREarly) {
                __syncwarp(kAll);
                issue2(j + kRRing, rs_now);
            }
        }
    }
    cp_async_wait<0>();
    finish();
    count_block();
    }  // task loop
}

// Resident blocks per SM of a kernel at its launch shape (occupancy query,
// once per device and kernel).
int ring_blocks_per_sm(const void *kern, int threads, int smem);

template <int LPE, bool WV, bool FO>
pmha_status launch_ring(const Args &k, cudaStream_t s)
{
    constexpr int smem = FO ? ring_fo_smem_bytes() : ring_smem_bytes<WV>();
    constexpr int NW = FO ? kFOWarps : kRWarps;
    constexpr int P = 32 / LPE;
    const long long warps = (k.B + P - 1) / P * k.n_units;
    if ((k.B + P - 1) / P * (k.n_units + (FO ? (long long)P * k.n_blk : 0)) > 0xffffffffLL) {
        set_error("edge attention: more than 2^32 tasks");
        return PMHA_ERR_UNSUPPORTED;
    }
    auto kern = k.kpm ? (k.scores ? k_edge_ring<LPE, WV, true, true, FO> : k_edge_ring<LPE, WV, false, true, FO>)
                      : (k.scores ? k_edge_ring<LPE, WV, true, false, FO> : k_edge_ring<LPE, WV, false, false, FO>);
    if constexpr (smem > 48 * 1024) {
        PMHA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    }
    const int per_sm = ring_blocks_per_sm((const void *)kern, NW * 32, smem);
    if (per_sm < 1) {
        set_error("edge attention: the ring kernel does not fit on an SM");
        return PMHA_ERR_UNSUPPORTED;
    }
    // (with out_proj tasks: one block per SM, which the out_proj tasks keep busy)
    const long long blocks =
        FO ? (long long)per_sm * num_sms() : std::min<long long>((warps + NW - 1) / NW, (long long)per_sm * num_sms());
    kern<<<(unsigned)blocks, NW * 32, smem, s>>>(k);
    return PMHA_OK;
}

// Entry points of the instantiating translation units: lpe 8, 16 or 32; and
// with out_proj tasks (k.out set), lpe 8.
pmha_status launch_ring_f16(int lpe, bool wv, const Args &k, cudaStream_t s);
pmha_status launch_ring_out_f16(int lpe, const Args &k, cudaStream_t s);

}  // namespace stream
}  // namespace pmha
