// out_proj (kpnn2 PackedMultiheadAttention, Notes step 5: the joined heads
// times Wo^T plus bo) as a task of the ring edge kernel.
//
// The ring kernel's queue interleaves two kinds of task: a unit of edges for
// a group of samples, and the out_proj of kOutRows consecutive targets of one
// sample. A slot that writes a target's final mixed row counts it, per
// (sample, block of kOutRows targets), after a release fence; the out_proj
// task of a block polls that count (with an acquire load, at most about a
// second) until every target of the block that has edges is counted, and
// then reads the block's mixed rows from L2. The queue places every
// out_proj task after every edge task, so the warps that find no edge task
// left take the blocks of finished sample groups while the last units run.
// Every edge task is taken from the queue before any out_proj task, and an
// edge task waits for nothing, so every poll ends.
//
// A task computes 16 rows at a time with mma.sync m16n8k16 (fp16 operands,
// fp32 accumulate): A = 16 mixed rows staged in the warp's ring (16-byte
// chunks placed at chunk c ^ (row & 7), so ldmatrix reads no bank twice),
// B = Wo from the block's shared-memory copy in the fragment order of
// wo_frag_pos (one 16-byte load per lane, n-tile and pair of k-steps, 512
// consecutive bytes per warp: no bank conflicts). Targets without edges mix
// to zeros, so their rows are bo.
#pragma once

#include "edge_stream.cuh"

namespace pmha {
namespace stream {

constexpr unsigned kOutWaitPolls = 1u << 22;  // polls 256 ns apart: about a second

__device__ __forceinline__ int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void lds_v4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d += a . b: one m16n8k16 product, fp16 operands, fp32 accumulators
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void st_zero16(uint32_t addr)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// out[b, t0 .. t0 + kOutRows) = mixed . Wo^T + bo for one sample b, by one
// warp; `ring` is the warp's ring (RING_BYTES of shared memory, idle), `wo`
// the block's copy of Wo followed by bo as E floats. Not inlined: its
// registers are then allocated apart from the edge loop's, which otherwise
// spills at the 128-register cap.
template <int E, int RING_BYTES>
__device__ __noinline__ void out_proj_block(const Args &a, int b, int blk, uint32_t ring, uint32_t wo, int lane)
{
    static_assert(E % 64 == 0, "64-column output chunks");
    constexpr unsigned kAll = 0xffffffffu;
    constexpr int CPR = E / 8;                   // 16-byte chunks per row
    constexpr int ROW = 2 * E;                   // bytes per row
    constexpr int TILE = 16 * ROW;               // a 16-row tile
    constexpr int NBUF = 2 * TILE <= RING_BYTES ? 2 : 1;
    constexpr int NSUB = kOutRows / 16;
    constexpr int KP = E / 32;                   // pairs of 16-deep k-steps
    constexpr int PER_LANE = 16 * CPR / 32;      // chunks a lane copies per tile
    static_assert(TILE <= RING_BYTES, "a 16-row tile fits the ring");
    static_assert(kOutRows == 64, "two 32-bit masks of targets");
    const int t0 = blk * kOutRows;

    // which targets of the block have edges (the others mix to zeros)
    auto has_edges = [&](int i) -> bool {
        const int t = t0 + i;
        return t < a.L && a.row_ptr[t + 1] > a.row_ptr[t];
    };
    const unsigned live_lo = __ballot_sync(kAll, has_edges(lane));
    const unsigned live_hi = __ballot_sync(kAll, has_edges(32 + lane));
    const int expect = __popc(live_lo) + __popc(live_hi);
    int ok = 1;
    if (lane == 0) {
        const int *cnt = a.blk_count + (long long)b * a.n_blk + blk;
        unsigned polls = 0;
        while (ld_acquire_gpu(cnt) < expect) {
            if (++polls > kOutWaitPolls) {
                ok = 0;
                atomicOr(a.err, kErrTimeoutBit);
                break;
            }
            __nanosleep(256);
        }
    }
    ok = __shfl_sync(kAll, ok, 0);
    if (!ok) return;
    asm volatile("fence.acq_rel.gpu;" ::: "memory");  // this lane's reads of the rows come after the count

    const char *mixed_b = (const char *)a.mixed + (long long)b * a.L * ROW;
    auto fill = [&](int sub, uint32_t buf) {
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int q = i * 32 + lane, r = q / CPR, c = q % CPR;
            const int rr = 16 * sub + r;
            const bool live = ((rr < 32 ? live_lo >> rr : live_hi >> (rr - 32)) & 1u) != 0;
            const uint32_t dst = buf + (uint32_t)(r * ROW + 16 * (c ^ (r & 7)));
            if (live) cp_async16_at<0, 0>(dst, mixed_b + (long long)(t0 + rr) * ROW + 16 * c);
            else st_zero16(dst);
        }
        cp_async_commit();
    };

    const uint32_t bias = wo + (uint32_t)(E * E * 2);
    __nv_bfloat16 *out_b = (__nv_bfloat16 *)a.out + (long long)b * a.L * E;
    // the lane's ldmatrix row: rows 0-7 / 8-15 of the low k half, then of the high half
    const int ar = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int kh = lane >> 4;

    fill(0, ring);
    if (NBUF == 2) fill(1, ring + TILE);
#pragma unroll 1
    for (int sub = 0; sub < NSUB; ++sub) {
        const uint32_t buf = ring + (uint32_t)((NBUF == 2 ? (sub & 1) : 0) * TILE);
        if (NBUF == 2 && sub + 1 < NSUB) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncwarp(kAll);  // every lane's chunks (and zero rows) of the tile are in place
        const uint32_t arow = buf + (uint32_t)(ar * ROW);
#pragma unroll 1
        for (int ch = 0; ch < E / 64; ++ch) {
            float acc[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
#pragma unroll 1
            for (int kp = 0; kp < KP; ++kp) {
                uint32_t a0[4], a1[4];
                ldsm_x4(arow + (uint32_t)(16 * ((4 * kp + kh) ^ (ar & 7))), a0);
                ldsm_x4(arow + (uint32_t)(16 * ((4 * kp + 2 + kh) ^ (ar & 7))), a1);
                const uint32_t wk = wo + (uint32_t)((((ch * 8) * KP + kp) * 32 + lane) * 16);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // four n-tiles at a time
                    uint32_t bf[4][4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) lds_v4(wk + (uint32_t)((4 * h + j) * KP * 512), bf[j]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        mma_16816(acc[4 * h + j], a0, bf[j][0], bf[j][1]);
                        mma_16816(acc[4 * h + j], a1, bf[j][2], bf[j][3]);
                    }
                }
            }
            // rows lane / 4 and lane / 4 + 8 of the tile, columns 2 (lane % 4) + {0, 1} of each n-tile
            const int ta = t0 + 16 * sub + (lane >> 2), tb = ta + 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = 64 * ch + 8 * j + 2 * (lane & 3);
                float b0, b1;
                asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(b0), "=f"(b1) : "r"(bias + 4 * col));
                if (ta < a.L) {
                    const __nv_bfloat162 v = __floats2bfloat162_rn(__fadd_rn(acc[j][0], b0), __fadd_rn(acc[j][1], b1));
                    *reinterpret_cast<__nv_bfloat162 *>(out_b + (long long)ta * E + col) = v;
                }
                if (tb < a.L) {
                    const __nv_bfloat162 v = __floats2bfloat162_rn(__fadd_rn(acc[j][2], b0), __fadd_rn(acc[j][3], b1));
                    *reinterpret_cast<__nv_bfloat162 *>(out_b + (long long)tb * E + col) = v;
                }
            }
        }
        if (sub + NBUF < NSUB) {
            __syncwarp(kAll);  // every lane's ldmatrix of this buffer has returned
            fill(sub + NBUF, buf);
        }
    }
}

}  // namespace stream
}  // namespace pmha
