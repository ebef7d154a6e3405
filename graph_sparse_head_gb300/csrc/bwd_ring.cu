// The per-edge backward kernels for fp16 intermediates with 16 channels a
// lane (chain rule of kpnn2 PackedMultiheadAttention, Notes steps 2-4), on
// the structure of the forward's ring kernel (edge_ring.cuh):
//
//   dq  (per-target view): per edge the source's k and v rows; per row the
//       target's q and dmixed rows and its record {c, D}, c = m + log2(l)
//       w = 2^(q.k log2(e)/sqrt(d) - c) (= 2^(s - m) / l), ds = w (dmixed.v - D),
//       dq_t = sum ds k / sqrt(d)
//   dkv (per-source view): per edge the target's q and dmixed rows and its
//       record; per row the source's k and v rows
//       dk_s = sum ds q / sqrt(d), dv_s = sum w dmixed
//
// Work decomposition as in the forward: the positions of a view are cut into
// units of kUnitEdges; a warp walks one unit for P = 32 / LPE consecutive
// samples (a slot of LPE lanes per sample, 16 channels a lane). Persistent
// warps take (sample group, unit) tasks from one queue, sample groups in
// order, the units of a group in the order given (longest first for dq).
// A row inside one unit is finished there; a row crossing a unit boundary
// leaves partial sums in the unit's slots 2u / 2u + 1, which k_bwd_merge
// adds in unit order.
//
// Everything a step reads comes through a per-warp ring of kBRDepth shared-
// memory stages that cp.async fills kBRDepth edges ahead: the edge's rows
// and, when the edge is the first of a row, that row's rows (an issuing
// cursor walks the row bounds ahead of the consumer), so a row switch never
// waits on a global load. Steps take two edges; when both belong to the
// current row, the step reads both stages into registers and refills them
// at once (early release). Chunk placement and the swapped read order of
// lanes with sw = 1 are the forward's (no shared-memory bank conflicts);
// a lane's accumulators are swapped alike and stored back in row order.
// Dot products take mixed-precision FMAs (fp16 x fp16, fp32 accumulate) or,
// where a row is widened to fp32 anyway (dq's k, summed into dq, and the
// target's q), paired fp32 FMAs: fp16 products are exact in fp32, so both
// forms give the same dot product for the same summation order. The sums
// over edges widen the fp16 rows (paired fp32 FMAs).
#include <cuda_fp16.h>

#include <algorithm>

#include "edge_ring.cuh"
#include "pmha_internal.h"

namespace pmha {
namespace bwdr {
using stream::cp_async16_at;
using stream::cp_async_commit;
using stream::cp_async_wait;
using stream::ex2;
using stream::f2;
using stream::ffma2;
using stream::fma_h2;
using stream::fmul2;
using stream::lds_pair;
using stream::pk;
using stream::Raw;
using stream::smem_u32;
using stream::upk;

#ifndef PMHA_BRING_DEPTH
#define PMHA_BRING_DEPTH 4
#endif
constexpr int kBRWarps = 2;                 // warps per block
constexpr int kBRDepth = PMHA_BRING_DEPTH;  // stages = edges in flight (early release)
static_assert(kBRDepth % 2 == 0 && kBRDepth >= 2, "edges go two per step");
constexpr int kPartBytes = 32 * 32;         // one row part of the warp: 32 lanes x 16 fp16
// a stage: parts A, B (the edge's rows), C, D (the row's rows), then one
// 8-byte record per lane
constexpr int kOffA = 0, kOffB = kPartBytes, kOffC = 2 * kPartBytes, kOffD = 3 * kPartBytes,
              kOffRec = 4 * kPartBytes;
constexpr int kStage = 4 * kPartBytes + 32 * 8;
constexpr int kBRSmem = kBRWarps * kBRDepth * kStage;

// dot product of a lane's 16 channels (two independent partial sums each
// way), summed over the lph lanes of its head
__device__ __forceinline__ float dot16(const Raw<32> &x, const Raw<32> &y, int lph)
{
    float ax = 0.f, ay = 0.f, bx = 0.f, by = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        fma_h2(ax, ay, x.w[i], y.w[i]);
        fma_h2(bx, by, x.w[i + 1], y.w[i + 1]);
    }
    float d = __fadd_rn(__fadd_rn(ax, bx), __fadd_rn(ay, by));
    for (int o = 1; o < lph; o <<= 1) d = __fadd_rn(d, __shfl_xor_sync(0xffffffffu, d, o));
    return d;
}

// the lane's 16 fp16 channels as fp32 pairs
__device__ __forceinline__ void widen16(const Raw<32> &x, f2 (&f)[8])
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&x.w[i]));
        f[i] = pk(v.x, v.y);
    }
}

// dot16 on widened channels: the same products (exact in fp32), sums and
// order, so the same result
__device__ __forceinline__ float dot16w(const f2 (&x)[8], const f2 (&y)[8], int lph)
{
    f2 a2 = 0ull, b2 = 0ull;
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        a2 = ffma2(x[i], y[i], a2);
        b2 = ffma2(x[i + 1], y[i + 1], b2);
    }
    const float2 fa = upk(a2), fb = upk(b2);
    float d = __fadd_rn(__fadd_rn(fa.x, fb.x), __fadd_rn(fa.y, fb.y));
    for (int o = 1; o < lph; o <<= 1) d = __fadd_rn(d, __shfl_xor_sync(0xffffffffu, d, o));
    return d;
}

// acc += c * x for the lane's 16 widened channels
__device__ __forceinline__ void axpy16(f2 (&acc)[8], float c, const f2 (&x)[8])
{
    const f2 c2 = pk(c, c);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = ffma2(c2, x[i], acc[i]);
}

// 16 fp32 values of a lane (its two chunks in read order) times `scale` to
// row + c0: the first read chunk is chunk 2 grp + sw of the lane's pair
__device__ __forceinline__ void store16(float *row, const f2 (&acc)[8], float scale, int sw)
{
    const f2 s2 = pk(scale, scale);
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 lo = upk(fmul2(acc[2 * i], s2)), hi = upk(fmul2(acc[2 * i + 1], s2));
        v[i] = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    float4 *first = reinterpret_cast<float4 *>(row + 8 * sw), *second = reinterpret_cast<float4 *>(row + 8 * (1 - sw));
    first[0] = v[0];
    first[1] = v[1];
    second[0] = v[2];
    second[1] = v[3];
}

// DKV: the per-source view (dk, dv), else the per-target view (dq).
// KPM: a key_padding_mask drops keys (their edges have weight 0).
// Shared memory allows 6 blocks (12 warps) per SM, so the register budget
// is set for that many (168 a thread).
template <int LPE, bool DKV, bool KPM>
__global__ void __launch_bounds__(kBRWarps * 32, 6) k_bwd_ring(BwdRingArgs a)
{
    static_assert(LPE >= 8 && LPE <= 32, "8 to 32 lanes per row");
    constexpr int P = 32 / LPE;      // slots (samples) per warp
    constexpr int PART = LPE * 32;   // bytes of one slot's row in a part
    constexpr unsigned kAll = 0xffffffffu;
    extern __shared__ __align__(16) unsigned char smem_dyn[];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slot = lane / LPE, grp = lane % LPE;
    const int c0 = grp * 16;
    const int head = c0 / (a.E / a.H);
    const int lph = a.E / a.H / 16;  // lanes per head
    const int sw = (grp >> 2) & 1;   // the lane's two chunks sit swapped in shared memory

    const uint32_t wbase = smem_u32(smem_dyn) + (uint32_t)(warp * kBRDepth * kStage);
    const uint32_t rd0 = wbase + (uint32_t)(slot * PART + 32 * grp + 16 * sw);
    const uint32_t rd1 = wbase + (uint32_t)(slot * PART + 32 * grp + 16 * (1 - sw));
    const uint32_t fill = wbase + (uint32_t)(slot * PART + 16 * grp);
    const uint32_t rec_at = wbase + (uint32_t)(kOffRec + 8 * lane);

    const unsigned n_groups = (unsigned)((a.B + P - 1) / P);
    const unsigned n_u = (unsigned)a.n_units;
    const unsigned n_tasks = n_groups * n_u;
    for (;;) {
    unsigned task = 0;
    if (lane == 0) task = atomicAdd(a.task_counter, 1u);
    task = __shfl_sync(kAll, task, 0);
    if (task >= n_tasks) break;
    const unsigned grp_i = task / n_u, idx_u = task % n_u;
    const int u = a.unit_order ? a.unit_order[idx_u] : (int)idx_u;
    const int b_slot = (int)grp_i * P + slot;
    const bool own = b_slot < a.B;  // slots past the batch store nothing
    const int b = own ? b_slot : a.B - 1;
    const int e0 = u * kUnitEdges;
    const int n = (int)min((long long)kUnitEdges, a.nnz - e0);
    const int e1 = e0 + n;

    // byte pointers at this lane's first chunk of row 0 of sample b
    const char *Q0 = (const char *)a.q + ((long long)b * a.L * a.q_ld) * 2 + 16 * grp;
    const char *G0 = (const char *)a.g + ((long long)b * a.L * a.E) * 2 + 16 * grp;
    const char *K0 = (const char *)a.k + ((long long)b * a.S * a.kv_ld) * 2 + 16 * grp;
    const char *V0 = (const char *)a.v + ((long long)b * a.S * a.kv_ld) * 2 + 16 * grp;
    const unsigned q_row = (unsigned)(a.q_ld * 2), g_row = (unsigned)(a.E * 2), kv_row = (unsigned)(a.kv_ld * 2);
    const float2 *REC = a.rec + (long long)b * a.L * a.H + head;
    const uint8_t *kpm_b = KPM ? a.kpm + (long long)b * a.S : nullptr;

    // two 16-byte chunks (grp and LPE + grp) of a row into part `off` of stage st
    auto copy_row = [&](uint32_t st, uint32_t off, const char *src) {
        cp_async16_at<0, 0>(fill + st + off, src);
        cp_async16_at<PART / 2, 16 * LPE>(fill + st + off, src);
    };
    auto copy_rec = [&](uint32_t st, int t) {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(rec_at + st),
                     "l"(REC + (long long)(unsigned)t * a.H)
                     : "memory");
    };
    // the rows an edge brings from its other end o (and, for DKV, o's record)
    auto copy_edge = [&](uint32_t st, int o) {
        if constexpr (DKV) {  // o is a target
            copy_row(st, kOffA, Q0 + (unsigned long long)(unsigned)o * q_row);
            copy_row(st, kOffB, G0 + (unsigned long long)(unsigned)o * g_row);
            copy_rec(st, o);
        } else {              // o is a source
            copy_row(st, kOffA, K0 + (unsigned long long)(unsigned)o * kv_row);
            copy_row(st, kOffB, V0 + (unsigned long long)(unsigned)o * kv_row);
        }
    };
    // the rows of view row r (a source for DKV, a target for dq)
    auto copy_view_row = [&](uint32_t st, int r) {
        if constexpr (DKV) {
            copy_row(st, kOffC, K0 + (unsigned long long)(unsigned)r * kv_row);
            copy_row(st, kOffD, V0 + (unsigned long long)(unsigned)r * kv_row);
        } else {
            copy_row(st, kOffC, Q0 + (unsigned long long)(unsigned)r * q_row);
            copy_row(st, kOffD, G0 + (unsigned long long)(unsigned)r * g_row);
            copy_rec(st, r);
        }
    };

    // ---- 32-wide windows of the other ends: lane i holds idx[e0 + 32 w + i]
    const int32_t *idxu = a.idx + e0;
    auto ldidx = [&](int w) -> int {
        const int p = 32 * w + lane;
        return p < n ? idxu[p] : 0;
    };
    int cwi = 0;
    int cw_cur = ldidx(0), cw_nxt = ldidx(1);

    // ---- row bounds: a window of 32 rows, lane i holds row_ptr[tw + i + 1]
    struct Bounds {
        int tw, cur, nxt;
    };
    auto ldrp = [&](int rr) -> int { return rr < a.n_rows ? a.row_ptr[rr + 1] : (int)a.nnz; };
    auto end_in = [&](Bounds &w, int rr) -> int {  // row_ptr[rr + 1]; rr never decreases
        while (rr - w.tw >= 32) {
            w.tw += 32;
            w.cur = w.nxt;
            w.nxt = ldrp(w.tw + 32 + lane);
        }
        return __shfl_sync(kAll, w.cur, rr - w.tw);
    };
    const int r_first = a.unit_first[u];
    Bounds wi{r_first, ldrp(r_first + lane), ldrp(r_first + 32 + lane)};
    int ri = r_first;
    int bi = end_in(wi, ri);

    // positions j, j + 1 (j even; one 32-window) into stages sj, sj + 1; the
    // first position of a row also brings that row's rows
    auto issue2 = [&](int j, int sj) {
        if (j >= 32 * (cwi + 1)) {
            ++cwi;
            cw_cur = cw_nxt;
            cw_nxt = ldidx(cwi + 1);
        }
        const int o0 = __shfl_sync(kAll, cw_cur, j & 31);
        const int o1 = __shfl_sync(kAll, cw_cur, (j + 1) & 31);
        const uint32_t st0 = (uint32_t)(sj * kStage);
        if (j < n) {
            copy_edge(st0, o0);
            if (e0 + j >= bi) {
                do {
                    ++ri;
                    bi = end_in(wi, ri);
                } while (bi <= e0 + j);
                copy_view_row(st0, ri);
            }
        }
        if (j + 1 < n) {
            copy_edge(st0 + kStage, o1);
            if (e0 + j + 1 >= bi) {
                do {
                    ++ri;
                    bi = end_in(wi, ri);
                } while (bi <= e0 + j + 1);
                copy_view_row(st0 + kStage, ri);
            }
        }
        cp_async_commit();
    };
    copy_view_row(0, r_first);
#pragma unroll
    for (int j = 0; j < kBRDepth; j += 2) issue2(j, j);

    // ---- consumer state: row r and its rows / record, the sums
    Bounds wc{r_first, ldrp(r_first + lane), ldrp(r_first + 32 + lane)};
    int r = r_first;
    int bound = end_in(wc, r);
    const bool first_started_here = a.row_ptr[r] == e0;
    bool is_first = true;
    // dq: the target's q (widened) and dmixed; dkv: the source's k and v
    f2 rowCw[8];
    Raw<32> rowC, rowD;
    float rc = 0.f, rD = 0.f;  // dq: the target's record
    bool r_dropped = false;       // dkv: the source is a padded key
    f2 acc0[8], acc1[8];          // dq: acc0; dkv: dk (acc0), dv (acc1)
    auto zero = [&]() {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            acc0[i] = 0ull;
            if constexpr (DKV) acc1[i] = 0ull;
        }
    };
    auto set_row = [&](uint32_t st) {
        rowC = lds_pair(rd0 + st + kOffC, rd1 + st + kOffC);
        rowD = lds_pair(rd0 + st + kOffD, rd1 + st + kOffD);
        if constexpr (!DKV) widen16(rowC, rowCw);
        if constexpr (!DKV) {
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(rc), "=f"(rD) : "r"(rec_at + st));
        } else if constexpr (KPM) {
            r_dropped = kpm_b[r] != 0;
        }
    };
    auto finish = [&]() {
        if (!own) return;
        const bool complete = (is_first ? first_started_here : true) && bound <= e1;
        if (complete) {
            float *o = a.out0 + ((long long)b * a.n_rows + r) * a.E + c0;
            store16(o, acc0, a.inv_sqrt_d, sw);
            if constexpr (DKV) store16(a.out1 + ((long long)b * a.n_rows + r) * a.E + c0, acc1, 1.f, sw);
        } else {
            const int W = DKV ? 2 * a.E : a.E;
            float *p = a.part + ((long long)b * 2 * a.n_units + 2 * u + (is_first ? 0 : 1)) * W + c0;
            store16(p, acc0, a.inv_sqrt_d, sw);
            if constexpr (DKV) store16(p + a.E, acc1, 1.f, sw);
        }
    };
    // move from r to the row of position pos (> the end of r); its rows sit in stage st
    auto advance = [&](int pos, uint32_t st) {
        finish();
        is_first = false;
        do {
            ++r;
            bound = end_in(wc, r);
        } while (bound <= pos);
        set_row(st);
        zero();
    };
    // one edge: A, B are the edge's rows (dq: k, v; dkv: q, dmixed), rec its
    // target's record (dkv), o its other end (dq: the source, for the mask)
    auto edge = [&](const Raw<32> &A, const Raw<32> &B, float2 rec, int o) {
        if constexpr (DKV) {
            const float d1 = dot16(A, rowC, lph), d2 = dot16(B, rowD, lph);
            // c = +inf for a target without a live key: ex2(-inf) = +0
            const float w = r_dropped ? 0.f : ex2(__fsub_rn(__fmul_rn(d1, a.score_scale), rec.x));
            const float ds = __fmul_rn(w, __fsub_rn(d2, rec.y));
            f2 xw[8];
            widen16(A, xw);
            axpy16(acc0, ds, xw);
            widen16(B, xw);
            axpy16(acc1, w, xw);
        } else {
            f2 kw[8];
            widen16(A, kw);
            const float d1 = dot16w(rowCw, kw, lph), d2 = dot16(rowD, B, lph);
            const bool drop = KPM && kpm_b[o] != 0;
            const float w = drop ? 0.f : ex2(__fsub_rn(__fmul_rn(d1, a.score_scale), rc));
            const float ds = __fmul_rn(w, __fsub_rn(d2, rD));
            axpy16(acc0, ds, kw);
        }
    };
    auto ld_rec = [&](uint32_t st) -> float2 {
        float2 v = make_float2(0.f, 0.f);
        if constexpr (DKV) asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(rec_at + st));
        return v;
    };
    auto other_end = [&](int j) -> int {  // dq with a mask: the source of position e0 + j
        if constexpr (KPM && !DKV) return idxu[j];
        return 0;
    };
    auto one = [&](int j, uint32_t st) {
        const int pos = e0 + j;
        if (pos >= bound) advance(pos, st);
        const Raw<32> A = lds_pair(rd0 + st + kOffA, rd1 + st + kOffA);
        const Raw<32> B = lds_pair(rd0 + st + kOffB, rd1 + st + kOffB);
        edge(A, B, ld_rec(st), other_end(j));
    };

    cp_async_wait<kBRDepth / 2 - 1>();
    __syncwarp(kAll);
    set_row(0);
    zero();
    int rs = 0;
    for (int j = 0; j < n; j += 2) {
        cp_async_wait<kBRDepth / 2 - 1>();
        __syncwarp(kAll);  // the other lanes' chunks of these rows
        const uint32_t st0 = (uint32_t)(rs * kStage), st1 = st0 + (uint32_t)kStage;
        const int rs_now = rs;
        rs = rs + 2 == kBRDepth ? 0 : rs + 2;
        const int pos = e0 + j;
        if (j + 1 < n && pos + 1 < bound) {
            // both edges belong to r: read both stages, refill them, then compute
            const Raw<32> A0 = lds_pair(rd0 + st0 + kOffA, rd1 + st0 + kOffA);
            const Raw<32> B0 = lds_pair(rd0 + st0 + kOffB, rd1 + st0 + kOffB);
            const Raw<32> A1 = lds_pair(rd0 + st1 + kOffA, rd1 + st1 + kOffA);
            const Raw<32> B1 = lds_pair(rd0 + st1 + kOffB, rd1 + st1 + kOffB);
            const float2 q0 = ld_rec(st0), q1 = ld_rec(st1);
            const int o0 = other_end(j), o1 = other_end(j + 1);
            // every lane's loads of both stages have returned before the warp
            // refills them (one word of each 16-byte load is an input here)
            asm volatile("" ::"r"(A0.w[0]), "r"(A0.w[4]), "r"(B0.w[0]), "r"(B0.w[4]), "r"(A1.w[0]), "r"(A1.w[4]),
                         "r"(B1.w[0]), "r"(B1.w[4]), "f"(q0.x), "f"(q1.x));
            __syncwarp(kAll);
            issue2(j + kBRDepth, rs_now);
            edge(A0, B0, q0, o0);
            edge(A1, B1, q1, o1);
        } else {
            one(j, st0);
            if (j + 1 < n) one(j + 1, st1);
            __syncwarp(kAll);
            issue2(j + kBRDepth, rs_now);
        }
    }
    cp_async_wait<0>();
    finish();
    __syncwarp(kAll);  // every lane is done with the ring before the next task fills it
    }  // task loop
}

template <int LPE, bool DKV>
pmha_status launch_one(const BwdRingArgs &a, cudaStream_t s)
{
    auto kern = a.kpm ? k_bwd_ring<LPE, DKV, true> : k_bwd_ring<LPE, DKV, false>;
    static_assert(kBRSmem <= 48 * 1024, "static launch without the large-shared-memory attribute");
    const int per_sm = stream::ring_blocks_per_sm((const void *)kern, kBRWarps * 32, kBRSmem);
    if (per_sm < 1) {
        set_error("backward: the ring kernel does not fit on an SM");
        return PMHA_ERR_UNSUPPORTED;
    }
    constexpr int P = 32 / LPE;
    const long long tasks = (a.B + P - 1) / P * a.n_units;
    if (tasks > 0xffffffffLL) {
        set_error("backward: more than 2^32 tasks");
        return PMHA_ERR_UNSUPPORTED;
    }
    const long long blocks = std::min<long long>((tasks + kBRWarps - 1) / kBRWarps, (long long)per_sm * num_sms());
    if (blocks > 0) kern<<<(unsigned)blocks, kBRWarps * 32, kBRSmem, s>>>(a);
    return PMHA_OK;
}

}  // namespace bwdr

bool bwd_ring_supported(int64_t E, int64_t H)
{
    if (H < 1 || E % H) return false;
    const int64_t d = E / H;
    return (E == 128 || E == 256 || E == 512) && d % 16 == 0;
}

pmha_status launch_bwd_ring(bool dkv, const BwdRingArgs &a, cudaStream_t s)
{
    const int lpe = a.E / 16;
    switch (lpe) {
    case 8: return dkv ? bwdr::launch_one<8, true>(a, s) : bwdr::launch_one<8, false>(a, s);
    case 16: return dkv ? bwdr::launch_one<16, true>(a, s) : bwdr::launch_one<16, false>(a, s);
    case 32: return dkv ? bwdr::launch_one<32, true>(a, s) : bwdr::launch_one<32, false>(a, s);
    default: set_error("backward: no ring kernel for embed_dim %d", a.E); return PMHA_ERR_UNSUPPORTED;
    }
}

}  // namespace pmha
