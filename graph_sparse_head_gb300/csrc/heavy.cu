// Edge attention for targets with many incoming edges, on the tensor cores
// (kpnn2 PackedMultiheadAttention, Notes steps 2-4 for one target).
//
// The edge-packed scores and mix of one target t, head h, are rewritten
// through the projections of step 1 (k_s = Wk x_s + bk, v_s = Wv x_s + bv,
// x_s the key token, which is also the value token here):
//
//   q_t,h . k_s,h = (Wk_h^T q_t,h) . x_s + q_t,h . bk_h
//   sum_e w_e v_s,h = Wv_h (sum_e w_e x_s) + bv_h          (sum_e w_e = 1)
//
// The second score term does not depend on the edge, so the softmax over the
// edges of t drops it; with qt_h = Wk_h^T q_t,h the scores of 128 edges and
// every head are one product X_tile (128 x E) . [qt_0 .. qt_H-1] (E x H),
// and the mix of the tile is X_tile^T (E x 128) . P (128 x H): two dense
// 128 x 16 x E contractions per tile of edges, and the gathered rows are the
// tokens x_s (E bf16 values) instead of k_s and v_s.
//
// Three launches:
//   k_heavy_qt    qt of every (sample, heavy target), scaled by log2(e)/sqrt(d),
//                 stored as the 128-byte-swizzled K-major image the MMA reads
//   k_heavy_attn  persistent, two CTAs per SM, 6 warps each:
//                 warp 0    gathers the source tokens of 128 edges with TMA
//                           (tile::gather4, 4 rows per copy) into a 3-stage
//                           ring, and copies the item's qt image
//                 warp 1    issues the two MMAs per tile from one thread:
//                           S = X qt (fp32 in tensor memory) and, once the
//                           softmax warps wrote P, Y = X^T P
//                 warps 2-5 one thread per tile row: scores from tensor
//                           memory, P = 2^(s - m_ref) in bf16 against a
//                           reference per (item, head) that moves only when a
//                           score passes it by more than kLazy (then the mix
//                           in tensor memory and the sums are rescaled), the
//                           running sums l; Y accumulates in tensor memory
//                           over the item's tiles and is read once, during
//                           the next item's first tile
//                 An item is one (sample, heavy target); items run in order
//                 of decreasing in-degree, dealt to the CTAs back and forth.
//   k_heavy_out   mixed[t] = Wv_h (Y_h / l_h) + bv_h per head, fp16 rows
//
// Every mbarrier wait is bounded (1 s of wall clock); a wait that gives up
// sets PMHA_ERR_TIMEOUT, the CTA stops, lets its own copies land and frees
// its tensor memory.
#include <cuda.h>

#include <algorithm>
#include <mutex>
#include <set>
#include <vector>

#include "pmha_internal.h"
#include "tc_util.cuh"

namespace pmha {
namespace {
using namespace tcu;

constexpr int kE = 128;                        // embed_dim of this path
constexpr int kRows = 128;                     // edges per tile (MMA M of the score product)
constexpr int kHMax = 8;                       // heads kept in one 16-column accumulator
constexpr int kStages = 3;                     // X tiles in flight per CTA
constexpr int kHalfBytes = kRows * 128;        // 128 rows x 64 bf16 channels, 128-byte swizzle
constexpr int kTileBytes = 2 * kHalfBytes;     // one X tile (both channel halves)
constexpr int kSmallBytes = 4096;              // a 16 x 128 K-major operand (two 2 KB k-blocks)
constexpr int kQtBytes = 2048;                 // the qt image of one item (the two data atoms)
constexpr int kThreads = 192;
constexpr int kTmemCols = 64;                  // S[2] at 0 and 16, Y[2] at 32 and 48
constexpr int kOffQ = kStages * kTileBytes;    // qt operands [2]
constexpr int kOffP = kOffQ + 2 * kSmallBytes; // P operands [2]
constexpr int kOffBar = kOffP + 2 * kSmallBytes;
constexpr int kSmemBytes = kOffBar + 704;  // barriers, words, tile maxima [2][4][8], sums [4][8], reference [8]
static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");

struct HeavyArgs {
    const int32_t *row_ptr;   // L + 1
    const int32_t *col;       // nnz, source per CSR position
    const int4 *info;         // n_heavy heavy targets {t, first CSR position, in-degree, tiles}, in-degree non-increasing
    int n_heavy, B, S;
    const uint8_t *qt;        // (n_heavy * B) images of kQtBytes
    __half *yh;               // (n_heavy * B, E, 8): Y / l per channel and head, fp16
    int *err;
};

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Four rows of a 2-D bf16 tensor (box: 64 columns, one row) into shared
// memory, 512 bytes, swizzled by the destination address like a tiled load.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, int x, int y0, int y1, int y2,
                                            int y3, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(bar)
        : "memory");
}

// Contiguous global -> shared copy (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Descriptor of an MN-major operand with 128-byte swizzle: atoms of 64
// elements along M (128 bytes) by 8 rows along K; atoms along M `lbo` bytes
// apart, 8-row groups along K `sbo` bytes apart.
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: D fp32, A and B bf16, A K-major (mn_a =
// 0) or MN-major (mn_a = 1), B K-major, N = 16, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t mn_a)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (mn_a << 15) | ((uint32_t)(16 >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// named barrier 1 over the 128 softmax threads; true when any thread passes `pred`
__device__ __forceinline__ bool sm_sync_or(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Byte offset of element (row n, column k) of a 16-row K-major operand of
// 128 bf16 columns: two k-blocks of 64 columns, 2 KB apart, each two 8-row
// atoms of 8 x 128 bytes with the 128-byte swizzle (16-byte unit u of row n
// stored at u ^ (n % 8)).
__host__ __device__ __forceinline__ uint32_t small_off(int n, int k)
{
    return (uint32_t)((k >> 6) * 2048 + (n >> 3) * 1024 + (n & 7) * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) +
                      (k & 7) * 2);
}

// The item sequence of one CTA: round r takes item r*G + c (r even) or
// r*G + G-1-c (r odd) of the items sorted by decreasing in-degree.
__device__ __forceinline__ long long item_of(int r, int c, int G)
{
    return (long long)r * G + ((r & 1) ? (G - 1 - c) : c);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// P of a tile is 2^(s - m_ref) with a reference m_ref per (item, head) that
// changes only when a score passes it by more than kLazy (log2 units): then
// the item's running mix in tensor memory and the running sums are rescaled.
// P <= 2^kLazy keeps every sum far inside the fp32 range.
constexpr float kLazy = 16.f;

__global__ void __launch_bounds__(kThreads, 2) k_heavy_attn(const __grid_constant__ CUtensorMap tm_x, HeavyArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *xr = smem;             // X ring [kStages]
    uint8_t *qs = smem + kOffQ;     // qt operand [2], by item parity
    uint8_t *ps = smem + kOffP;     // P operand [2], by tile parity
    uint64_t *bars = (uint64_t *)(smem + kOffBar);
    uint64_t *xfull = bars, *xempty = bars + 3, *qfull = bars + 6, *qempty = bars + 8, *sfull = bars + 10,
             *sempty = bars + 12, *pfull = bars + 14, *ydone = bars + 16, *yfull = bars + 18, *yempty = bars + 20,
             *done = bars + 22;
    uint32_t *tmem_holder = (uint32_t *)(bars + 23);
    volatile int *abort_flag = (volatile int *)(tmem_holder + 1);
    int *issued = (int *)(tmem_holder + 2);   // [3] X copies armed per stage
    int *qissued = (int *)(tmem_holder + 5);  // [2] qt copies armed per buffer
    float *red = (float *)(smem + kOffBar + 256);   // [2][4][8] per-warp tile maxima
    float *lred = (float *)(smem + kOffBar + 512);  // [4][8] per-warp sums of an item
    float *mref_s = (float *)(smem + kOffBar + 640);  // [8] reference of an item's first tile
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long n_items = (long long)a.n_heavy * a.B;
    const int G = (int)gridDim.x, c = (int)blockIdx.x;

    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(a.err, kErrInternalBit);
        return;
    }
    // rows of a partial tile that no copy fills must hold finite values: zero
    // the operand buffers once (generic writes, then made visible to the MMA)
    for (int i = threadIdx.x; i < kOffBar / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_shared();
    if (threadIdx.x == 0) {
        for (int s = 0; s < 3; ++s) {
            mbar_init(smem_u32(&xfull[s]), 1);
            mbar_init(smem_u32(&xempty[s]), 1);
            issued[s] = 0;
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&qfull[s]), 1);
            mbar_init(smem_u32(&qempty[s]), 1);
            mbar_init(smem_u32(&sfull[s]), 1);
            mbar_init(smem_u32(&sempty[s]), 4);
            mbar_init(smem_u32(&pfull[s]), 4);
            mbar_init(smem_u32(&ydone[s]), 1);
            mbar_init(smem_u32(&yfull[s]), 1);
            mbar_init(smem_u32(&yempty[s]), 4);
            qissued[s] = 0;
        }
        mbar_init(smem_u32(done), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ---------------- producer: the item's qt image, then the source tokens of
        // each tile. Item metadata is loaded an item ahead and a tile's source
        // indices a tile ahead, so no dependent global load waits in line
        // before a copy is issued.
        int T = 0, it = 0;
        bool ok = true;
        long long k = item_of(0, c, G);
        if (k < n_items) {
            int4 inf = a.info[(int)(k / a.B)];
            long long kn = item_of(1, c, G);
            int4 infn = kn < n_items ? a.info[(int)(kn / a.B)] : make_int4(0, 0, 0, 0);
            // rows 4 lane .. 4 lane + 3 of tile i of item kk (past the last edge, the last edge again)
            auto load_idx = [&](long long kk, const int4 &f, int i, int (&y)[4]) {
                const int rows = min(kRows, f.z - kRows * i);
                if (lane < ((rows + 3) >> 2)) {
                    const int rowbase = (int)(kk % a.B) * a.S;
                    const int32_t *colp = a.col + f.y;
                    const int e0 = kRows * i + 4 * lane, last = kRows * i + rows - 1;
#pragma unroll
                    for (int u = 0; u < 4; ++u) y[u] = rowbase + colp[min(e0 + u, last)];
                }
            };
            int y[4] = {0, 0, 0, 0};
            load_idx(k, inf, 0, y);
            for (int r = 0; ok; ++r) {
                const int qb = it & 1;
                if (lane == 0) {
                    ok = mbar_wait(smem_u32(&qempty[qb]), (uint32_t)((it >> 1) & 1) ^ 1u, abort_flag, a.err);
                    if (ok) {
                        const uint32_t fb = smem_u32(&qfull[qb]);
                        mbar_arrive_expect_tx(fb, kQtBytes);
                        qissued[qb] += 1;
                        const uint8_t *src = a.qt + k * kQtBytes;
                        const uint32_t dst = smem_u32(qs + qb * kSmallBytes);
                        bulk_copy(dst, src, 1024, fb);                // k-block 0, rows 0-7
                        bulk_copy(dst + 2048, src + 1024, 1024, fb);  // k-block 1, rows 0-7
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                for (int i = 0; i < inf.w; ++i, ++T) {
                    const int st = T % 3;
                    const int groups = (min(kRows, inf.z - kRows * i) + 3) >> 2;
                    if (lane == 0) {
                        ok = mbar_wait(smem_u32(&xempty[st]), (uint32_t)((T / 3) & 1) ^ 1u, abort_flag, a.err);
                        if (ok) {
                            mbar_arrive_expect_tx(smem_u32(&xfull[st]), (uint32_t)groups * 1024u);
                            issued[st] += 1;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane < groups) {
                        const uint32_t dst = smem_u32(xr + st * kTileBytes + lane * 512);
                        const uint32_t fb = smem_u32(&xfull[st]);
                        tma_gather4(dst, &tm_x, 0, y[0], y[1], y[2], y[3], fb);
                        tma_gather4(dst + kHalfBytes, &tm_x, 64, y[0], y[1], y[2], y[3], fb);
                    }
                    if (i + 1 < inf.w) load_idx(k, inf, i + 1, y);
                    else if (kn < n_items) load_idx(kn, infn, 0, y);
                }
                if (!ok) break;
                ++it;
                if (kn >= n_items) break;
                k = kn;
                inf = infn;
                kn = item_of(r + 2, c, G);
                if (kn < n_items) infn = a.info[(int)(kn / a.B)];
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: S(T), then Y(T - 1) once its P is written.
            // Y of an item accumulates in tensor memory region it % 2.
            int T = 0, it = 0;
            bool ok = true;
            bool have = false, pf = false, pl = false;  // a pending Y: its tile, first / last of its item
            int pU = 0, pit = 0;
            auto issue_y = [&]() -> bool {
                const int sb = pU & 1, yb = pit & 1;
                if (!mbar_wait(smem_u32(&pfull[sb]), (uint32_t)((pU >> 1) & 1), abort_flag, a.err)) return false;
                if (pf && !mbar_wait(smem_u32(&yempty[yb]), (uint32_t)((pit >> 1) & 1) ^ 1u, abort_flag, a.err))
                    return false;
                tc_fence_after();
                const uint32_t xa = smem_u32(xr + (pU % 3) * kTileBytes);
                const uint32_t pb = smem_u32(ps + sb * kSmallBytes);
                const uint32_t d = tmem_base + 32u + (uint32_t)(yb * 16);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    // K step j = tile rows 16 j .. 16 j + 15: two 8-row groups of both channel halves
                    const uint64_t da = smem_desc_mn(xa + (uint32_t)(j * 2048), (uint32_t)kHalfBytes, 1024u);
                    const uint64_t db = smem_desc(pb + (uint32_t)((j >> 2) * 2048 + (j & 3) * 32));
                    mma_f16kind(d, da, db, idesc_bf16(1), (j > 0 || !pf) ? 1u : 0u);
                }
                mma_commit(smem_u32(&ydone[sb]));
                mma_commit(smem_u32(&xempty[pU % 3]));
                if (pl) mma_commit(smem_u32(&yfull[yb]));
                return true;
            };
            // tiles per item, one item ahead
            long long kn = item_of(0, c, G);
            int ntn = kn < n_items ? a.info[(int)(kn / a.B)].w : 0;
            for (int r = 0; ok; ++r) {
                if (kn >= n_items) break;
                const int nt = ntn;
                kn = item_of(r + 1, c, G);
                if (kn < n_items) ntn = a.info[(int)(kn / a.B)].w;
                const int qb = it & 1;
                if (!(ok = mbar_wait(smem_u32(&qfull[qb]), (uint32_t)((it >> 1) & 1), abort_flag, a.err))) break;
                const uint32_t qa = smem_u32(qs + qb * kSmallBytes);
                for (int i = 0; i < nt; ++i, ++T) {
                    const int st = T % 3, sb = T & 1;
                    if (!(ok = mbar_wait(smem_u32(&xfull[st]), (uint32_t)((T / 3) & 1), abort_flag, a.err))) break;
                    if (!(ok = mbar_wait(smem_u32(&sempty[sb]), (uint32_t)((T >> 1) & 1) ^ 1u, abort_flag, a.err)))
                        break;
                    tc_fence_after();
                    const uint32_t xa = smem_u32(xr + st * kTileBytes);
                    const uint32_t d = tmem_base + (uint32_t)(sb * 16);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        // K step j = channels 16 j .. 16 j + 15 (+32 bytes inside a swizzle atom)
                        const uint64_t da = smem_desc(xa + (uint32_t)((j >> 2) * kHalfBytes + (j & 3) * 32));
                        const uint64_t db = smem_desc(qa + (uint32_t)((j >> 2) * 2048 + (j & 3) * 32));
                        mma_f16kind(d, da, db, idesc_bf16(0), j > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&sfull[sb]));
                    if (i == nt - 1) mma_commit(smem_u32(&qempty[qb]));
                    if (have && !(ok = issue_y())) break;
                    have = true;
                    pU = T;
                    pit = it;
                    pf = i == 0;
                    pl = i == nt - 1;
                }
                if (!ok) break;
                ++it;
            }
            if (ok && have) issue_y();
            // every MMA issued by this thread has finished once this arrives
            mma_commit(smem_u32(done));
            int dummy = 0;
            mbar_wait(smem_u32(done), 0, (volatile int *)&dummy, a.err);
        }
    } else {
        // ---------------- softmax warps: thread r owns tile row r (scores) and channel r (mix).
        // `bad` (a wait gave up) may differ between warps; the loops stop only
        // on `stop`, decided by all 128 threads at a named barrier.
        const int q = warp & 3, r = q * 32 + lane;
        const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
        int T = 0, it = 0;
        bool bad = false, stop = false;
        bool has_prev = false;  // the previous item is finished during the next item's first tile
        long long k_prev = 0;
        float lp_prev[kHMax], m_ref[kHMax], lp[kHMax];
        // the previous item's per-warp sums into lred (read after the next barrier)
        auto put_sums = [&]() {
#pragma unroll
            for (int h = 0; h < kHMax; ++h) {
                const float lw = warp_sum(lp_prev[h]);
                if (lane == 0) lred[q * kHMax + h] = lw;
            }
        };
        // item ip's mix Y / l, channel r, into yh; hands its tensor memory back
        auto finish = [&](int ip, long long kp) {
            const int yb = ip & 1;
            bool ok = !bad && mbar_wait(smem_u32(&yfull[yb]), (uint32_t)((ip >> 1) & 1), abort_flag, a.err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                bad = true;
                return;
            }
            tc_fence_after();
            float y[kHMax];
            tmem_ld8(trow + 32u + (uint32_t)(yb * 16), y);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&yempty[yb]));
            uint32_t packed[kHMax / 2];
#pragma unroll
            for (int h = 0; h < kHMax; h += 2) {
                const float l0 = (lred[h] + lred[kHMax + h]) + (lred[2 * kHMax + h] + lred[3 * kHMax + h]);
                const float l1 =
                    (lred[h + 1] + lred[kHMax + h + 1]) + (lred[2 * kHMax + h + 1] + lred[3 * kHMax + h + 1]);
                __half2 hv = __floats2half2_rn(l0 > 0.f ? y[h] / l0 : 0.f, l1 > 0.f ? y[h + 1] / l1 : 0.f);
                packed[h / 2] = *reinterpret_cast<uint32_t *>(&hv);
            }
            *reinterpret_cast<uint4 *>(a.yh + (kp * kE + r) * kHMax) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
        };
        long long kn = item_of(0, c, G);  // in-degree of the next item, loaded an item ahead
        int degn = kn < n_items ? a.info[(int)(kn / a.B)].z : 0;
        for (int rr = 0; !stop; ++rr) {
            if (kn >= n_items) break;
            const long long k = kn;
            const int deg = degn;
            const int nt = (deg + kRows - 1) / kRows;
            kn = item_of(rr + 1, c, G);
            if (kn < n_items) degn = a.info[(int)(kn / a.B)].z;
#pragma unroll
            for (int h = 0; h < kHMax; ++h) lp[h] = 0.f;
            for (int i = 0; i < nt; ++i, ++T) {
                const int sb = T & 1;
                bool ok = !bad && mbar_wait(smem_u32(&sfull[sb]), (uint32_t)((T >> 1) & 1), abort_flag, a.err);
                ok = __all_sync(0xffffffffu, ok);
                float s[kHMax];
                if (ok) {
                    tc_fence_after();
                    tmem_ld8(trow + (uint32_t)(sb * 16), s);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sempty[sb]));
                    // P[sb] was last read by Y(T - 2)
                    if (T >= 2) ok = mbar_wait(smem_u32(&ydone[sb]), (uint32_t)(((T - 2) >> 1) & 1), abort_flag, a.err);
                    ok = __all_sync(0xffffffffu, ok);
                }
                const bool valid = ok && kRows * i + r < deg;
#pragma unroll
                for (int h = 0; h < kHMax; ++h) s[h] = valid ? s[h] : -INFINITY;
                if (i == 0) {
                    if (has_prev) put_sums();
                    if (r == 0)  // row 0 of an item is an edge: its scores are the first reference
#pragma unroll
                        for (int h = 0; h < kHMax; ++h) mref_s[h] = s[h];
                    if (sm_sync_or(!ok || bad)) {
                        bad = stop = true;
                        break;
                    }
#pragma unroll
                    for (int h = 0; h < kHMax; ++h) m_ref[h] = mref_s[h];
                }
                bool need = false;
#pragma unroll
                for (int h = 0; h < kHMax; ++h) need |= s[h] > m_ref[h] + kLazy;
                if (sm_sync_or(need || !ok || bad)) {
                    if (sm_sync_or(!ok || bad)) {
                        bad = stop = true;
                        break;
                    }
                    // a score passed the reference by more than kLazy: raise the
                    // reference to the tile maximum, rescale the sums and the mix
                    float f[kHMax];
#pragma unroll
                    for (int h = 0; h < kHMax; ++h) {
                        const float mw = warp_max(s[h]);
                        if (lane == 0) red[(sb * 4 + q) * kHMax + h] = mw;
                    }
                    sm_sync_or(false);
#pragma unroll
                    for (int h = 0; h < kHMax; ++h) {
                        const float *rm = red + sb * 4 * kHMax + h;
                        const float M = fmaxf(fmaxf(rm[0], rm[kHMax]), fmaxf(rm[2 * kHMax], rm[3 * kHMax]));
                        const float mn = fmaxf(m_ref[h], M);
                        f[h] = ex2f(m_ref[h] - mn);
                        m_ref[h] = mn;
                        lp[h] *= f[h];
                    }
                    if (i > 0) {
                        // the item's earlier Y products are all complete once Y(T - 1) is
                        bool ok2 = !bad && mbar_wait(smem_u32(&ydone[(T - 1) & 1]), (uint32_t)(((T - 1) >> 1) & 1),
                                                     abort_flag, a.err);
                        ok2 = __all_sync(0xffffffffu, ok2);
                        if (ok2) {
                            tc_fence_after();
                            const uint32_t ya = trow + 32u + (uint32_t)((it & 1) * 16);
                            float y[kHMax];
                            tmem_ld8(ya, y);
#pragma unroll
                            for (int h = 0; h < kHMax; ++h) y[h] *= f[h];
                            tmem_st8(ya, y);
                            tc_fence_before();
                        } else {
                            bad = true;
                        }
                    }
                }
                uint8_t *pbuf = ps + sb * kSmallBytes;
#pragma unroll
                for (int h = 0; h < kHMax; ++h) {
                    const __nv_bfloat16 pb = __float2bfloat16_rn(valid ? ex2f(s[h] - m_ref[h]) : 0.f);
                    lp[h] += __bfloat162float(pb);
                    *reinterpret_cast<__nv_bfloat16 *>(pbuf + small_off(h, r)) = pb;
                }
                // P is read by the tensor cores (async proxy)
                fence_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&pfull[sb]));
                if (i == 0 && has_prev) finish(it - 1, k_prev);
            }
            if (stop) break;
#pragma unroll
            for (int h = 0; h < kHMax; ++h) lp_prev[h] = lp[h];
            has_prev = true;
            k_prev = k;
            ++it;
        }
        if (!stop && has_prev) {
            put_sums();
            if (!sm_sync_or(bad)) finish(it - 1, k_prev);
        }
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let the copies this CTA started land before its shared memory goes away
        int dummy = 0;
        for (int s = 0; s < 3; ++s)
            if (issued[s] > 0)
                mbar_wait(smem_u32(&xfull[s]), (uint32_t)((issued[s] - 1) & 1), (volatile int *)&dummy, a.err);
        for (int s = 0; s < 2; ++s)
            if (qissued[s] > 0)
                mbar_wait(smem_u32(&qfull[s]), (uint32_t)((qissued[s] - 1) & 1), (volatile int *)&dummy, a.err);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
    }
}

// qt[item] = log2(e)/sqrt(d) * Wk_h^T q_t,h for every head h (zero for h >=
// H), as rows 0-7 of the 16-row K-major operand: one 1 KB atom per k-block
// (channels 0-63, then 64-127). Thread c computes channel c of every head
// for 8 items at a time (one weight read feeds 8 FMAs).
constexpr int kBatch = 8;
__global__ void __launch_bounds__(128) k_heavy_qt(const __half *__restrict__ q, long long q_ld,
                                                 const __nv_bfloat16 *__restrict__ wk,
                                                 const int4 *__restrict__ info, long long n_items, int B, int L,
                                                 int H, int d, float scale, int per_block, uint8_t *__restrict__ qt)
{
    __shared__ __align__(16) __nv_bfloat16 w_s[kE * kE];
    __shared__ __align__(16) float q_s[kE * kBatch];  // [input channel][item]
    const int c = threadIdx.x;
    {
        uint4 w[kE * kE / 8 / 128];  // all 16 loads in flight at once
#pragma unroll
        for (int m = 0; m < kE * kE / 8 / 128; ++m) w[m] = reinterpret_cast<const uint4 *>(wk)[c + 128 * m];
#pragma unroll
        for (int m = 0; m < kE * kE / 8 / 128; ++m) reinterpret_cast<uint4 *>(w_s)[c + 128 * m] = w[m];
    }
    const long long first = (long long)blockIdx.x * per_block;
    const long long last = min(n_items, first + per_block);
    // channel c of the q rows of 8 items, loaded a batch ahead
    auto load_q = [&](long long base, float (&v)[kBatch]) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const long long k = base + i;
            v[i] = k < last ? __half2float(q[((long long)(k % B) * L + info[(int)(k / B)].x) * q_ld + c]) : 0.f;
        }
    };
    float qv[kBatch];
    load_q(first, qv);
    for (long long base = first; base < last; base += kBatch) {
        __syncthreads();  // weights staged / the previous batch's q rows read
#pragma unroll
        for (int i = 0; i < kBatch; ++i) q_s[c * kBatch + i] = qv[i];
        __syncthreads();
        if (base + kBatch < last) load_q(base + kBatch, qv);
#pragma unroll 1
        for (int h = 0; h < kHMax; ++h) {
            float acc[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) acc[i] = 0.f;
            if (h < H) {
                for (int j = h * d; j < (h + 1) * d; ++j) {
                    const float w = __bfloat162float(w_s[j * kE + c]);
                    const float4 qa = reinterpret_cast<const float4 *>(q_s + j * kBatch)[0];
                    const float4 qb = reinterpret_cast<const float4 *>(q_s + j * kBatch)[1];
                    acc[0] = fmaf(qa.x, w, acc[0]);
                    acc[1] = fmaf(qa.y, w, acc[1]);
                    acc[2] = fmaf(qa.z, w, acc[2]);
                    acc[3] = fmaf(qa.w, w, acc[3]);
                    acc[4] = fmaf(qb.x, w, acc[4]);
                    acc[5] = fmaf(qb.y, w, acc[5]);
                    acc[6] = fmaf(qb.z, w, acc[6]);
                    acc[7] = fmaf(qb.w, w, acc[7]);
                }
            }
            const int off = (c >> 6) * 1024 + h * 128 + ((((c & 63) >> 3) ^ h) << 4) + (c & 7) * 2;
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                if (base + i < last)
                    *reinterpret_cast<__nv_bfloat16 *>(qt + (base + i) * kQtBytes + off) =
                        __float2bfloat16_rn(acc[i] * scale);
        }
    }
}

// mixed[b, t, j] = sum_c Wv[j, c] yh[item, c, h(j)] + bv[j]: thread j, Wv in
// shared memory as fp32 rows of pitch kE + 1 (conflict-free column reads),
// 8 items at a time ([head][channel][item] in shared memory).
constexpr int kOutSmem = (kE * (kE + 1) + kHMax * kE * kBatch) * 4;
__global__ void __launch_bounds__(128) k_heavy_out(const __half *__restrict__ yh, const __nv_bfloat16 *__restrict__ wv,
                                                  const __nv_bfloat16 *__restrict__ bv,
                                                  const int4 *__restrict__ info, long long n_items, int B, int L,
                                                  int d, int per_block, __half *__restrict__ mixed, int *err)
{
    extern __shared__ __align__(16) float o_s[];
    float *w_s = o_s;                  // [kE][kE + 1]
    float *y_s = o_s + kE * (kE + 1);  // [8 heads][kE channels][kBatch items]
    const int j = threadIdx.x;
    {
        uint4 w[kE * kE / 8 / 128];  // all 16 loads in flight at once
#pragma unroll
        for (int m = 0; m < kE * kE / 8 / 128; ++m) w[m] = reinterpret_cast<const uint4 *>(wv)[j + 128 * m];
#pragma unroll
        for (int m = 0; m < kE * kE / 8 / 128; ++m) {
            const int u = j + 128 * m, row = u / (kE / 8), col = (u % (kE / 8)) * 8;
            const __nv_bfloat162 *bp = reinterpret_cast<const __nv_bfloat162 *>(&w[m]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(bp[e]);
                w_s[row * (kE + 1) + col + 2 * e] = f.x;
                w_s[row * (kE + 1) + col + 2 * e + 1] = f.y;
            }
        }
    }
    const float bias = bv ? __bfloat162float(bv[j]) : 0.f;
    const int h = j / d;
    bool range_bad = false;
    const long long first = (long long)blockIdx.x * per_block;
    const long long last = min(n_items, first + per_block);
    // channel j of 8 items' rows (8 heads each), loaded a batch ahead
    auto load_y = [&](long long base, uint4 (&raw)[kBatch]) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            raw[i] = base + i < last ? reinterpret_cast<const uint4 *>(yh + ((base + i) * kE + j) * kHMax)[0]
                                     : make_uint4(0u, 0u, 0u, 0u);
    };
    uint4 raw[kBatch];
    load_y(first, raw);
    for (long long base = first; base < last; base += kBatch) {
        float v[kBatch][kHMax];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const __half2 *hp = reinterpret_cast<const __half2 *>(&raw[i]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __half22float2(hp[u]);
                v[i][2 * u] = f.x;
                v[i][2 * u + 1] = f.y;
            }
        }
        __syncthreads();  // weights staged / the previous batch read
#pragma unroll
        for (int hh = 0; hh < kHMax; ++hh) {
            float4 *dst = reinterpret_cast<float4 *>(y_s + (hh * kE + j) * kBatch);
            dst[0] = make_float4(v[0][hh], v[1][hh], v[2][hh], v[3][hh]);
            dst[1] = make_float4(v[4][hh], v[5][hh], v[6][hh], v[7][hh]);
        }
        __syncthreads();
        if (base + kBatch < last) load_y(base + kBatch, raw);
        const float *wr = w_s + j * (kE + 1);
        const float *yr = y_s + h * kE * kBatch;
        float acc[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) acc[i] = 0.f;
#pragma unroll 4
        for (int cc = 0; cc < kE; ++cc) {
            const float w = wr[cc];
            const float4 ya = reinterpret_cast<const float4 *>(yr + cc * kBatch)[0];
            const float4 yb = reinterpret_cast<const float4 *>(yr + cc * kBatch)[1];
            acc[0] = fmaf(w, ya.x, acc[0]);
            acc[1] = fmaf(w, ya.y, acc[1]);
            acc[2] = fmaf(w, ya.z, acc[2]);
            acc[3] = fmaf(w, ya.w, acc[3]);
            acc[4] = fmaf(w, yb.x, acc[4]);
            acc[5] = fmaf(w, yb.y, acc[5]);
            acc[6] = fmaf(w, yb.z, acc[6]);
            acc[7] = fmaf(w, yb.w, acc[7]);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const long long k = base + i;
            if (k >= last) break;
            const float out = acc[i] + bias;
            if (!(fabsf(out) <= 65504.f)) range_bad = true;
            mixed[((k % B) * L + info[(int)(k / B)].x) * kE + j] = __float2half_rn(out);
        }
    }
    if (range_bad) atomicOr(err, kErrRangeBit);
}

constexpr int kItemsPerBlock = 32;  // items per block of the qt and output kernels

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device)
template <typename K>
cudaError_t set_smem_once(K kern, int bytes)
{
    static std::mutex mu;
    static std::set<int> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(dev)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert(dev);
    return e;
}

}  // namespace

bool heavy_supported(const pmha_graph *g, int64_t E, int64_t H, TcType t)
{
    return g && g->light && g->n_heavy > 0 && t == TcType::F16 && E == kE && H >= 1 && H <= kHMax &&
           (kE % H) == 0;
}

size_t heavy_workspace_bytes(const pmha_graph *g, int64_t B)
{
    if (!g || !g->light || g->n_heavy <= 0) return 0;
    const size_t items = (size_t)g->n_heavy * (size_t)B;
    return items * (size_t)kQtBytes + items * (size_t)kE * kHMax * 2;
}

pmha_status heavy_attention(const pmha_graph *g, const HeavyInputs &in, cudaStream_t s)
{
    const long long n_items = (long long)g->n_heavy * in.B;
    if (n_items == 0) return PMHA_OK;
    if (in.B * g->S >= (1ll << 31)) {
        set_error("heavy-target path: batch x key_features exceeds the TMA row range");
        return PMHA_ERR_UNSUPPORTED;
    }
    const int H = (int)in.H, d = (int)(kE / in.H);
    uint8_t *qt = (uint8_t *)in.workspace;
    __half *yh = (__half *)((uint8_t *)in.workspace + (size_t)n_items * kQtBytes);
    CUtensorMap tm_x;
    if (!make_map_box(&tm_x, in.x, in.B * g->S, kE, kE, true, 64, 1)) {
        set_error("heavy-target path: cuTensorMapEncodeTiled failed for the key tokens");
        return PMHA_ERR_CUDA;
    }
    const unsigned pre_blocks = (unsigned)((n_items + kItemsPerBlock - 1) / kItemsPerBlock);
    {
        StageTimer timer("heavy_qt", s);
        k_heavy_qt<<<pre_blocks, 128, 0, s>>>((const __half *)in.q, (long long)in.q_ld,
                                              (const __nv_bfloat16 *)in.wk, g->heavy_info, n_items, (int)in.B,
                                              (int)g->L, H, d, (float)(1.4426950408889634 / sqrt((double)d)),
                                              kItemsPerBlock, qt);
        count_launch();
        PMHA_CUDA_TRY(cudaGetLastError());
    }
    PMHA_CUDA_TRY(set_smem_once(k_heavy_attn, kSmemBytes));
    {
        HeavyArgs a;
        a.row_ptr = g->row_ptr;
        a.col = g->col;
        a.info = g->heavy_info;
        a.n_heavy = (int)g->n_heavy;
        a.B = (int)in.B;
        a.S = (int)g->S;
        a.qt = qt;
        a.yh = yh;
        a.err = device_error_word();
        const long long grid = std::min<long long>(n_items, 2ll * num_sms());
        StageTimer timer("heavy_attn", s);
        k_heavy_attn<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(tm_x, a);
        count_launch();
        PMHA_CUDA_TRY(cudaGetLastError());
    }
    PMHA_CUDA_TRY(set_smem_once(k_heavy_out, kOutSmem));
    {
        StageTimer timer("heavy_out", s);
        k_heavy_out<<<pre_blocks, 128, kOutSmem, s>>>(yh, (const __nv_bfloat16 *)in.wv, (const __nv_bfloat16 *)in.bv,
                                                      g->heavy_info, n_items, (int)in.B, (int)g->L, d, kItemsPerBlock,
                                                      (__half *)in.mixed, device_error_word());
        count_launch();
        PMHA_CUDA_TRY(cudaGetLastError());
    }
    return PMHA_OK;
}

}  // namespace pmha
