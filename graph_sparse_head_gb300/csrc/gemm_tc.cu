// Projection GEMM on the 5th-generation tensor cores (sm_103a): tcgen05.mma
// with fp32 accumulators in tensor memory, operands streamed into shared
// memory by TMA, bias add and bf16 rounding fused into the epilogue.
//
// kpnn2 PackedMultiheadAttention, Notes step 1 (q_proj, k_proj, v_proj) and
// step 5 (out_proj): Y = X W^T + b, W stored (out, in) like nn.Linear. The
// head split of step 1 is a layout fact: row r of Y, columns [h*d, (h+1)*d),
// is head h, so no data movement is needed. Up to three projections that
// read the same X (Q|K|V of attention within one graph, K|V of a bipartite
// map) run as one GEMM whose N axis walks the weight matrices in turn; the
// output row then holds [Q | K | V] side by side.
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0    TMA producer: X tile 128 x 64 and W tile 128 x 64 per stage,
//             128-byte swizzle, into a 4-stage shared-memory ring
//   warp 1    allocates 256 TMEM columns (two 128 x 128 fp32 accumulators)
//             and issues tcgen05.mma (M=128, N=128, K=16) from one thread
//   warps 2-  epilogue, kEpi groups of 4 warps; group g drains the tiles
//             whose accumulator is g (a CTA's tiles alternate between the
//             two): tcgen05.ld 32 columns at a time (warp w reads TMEM lanes
//             32*(w%4) .. +31), + bias (staged in shared memory once per
//             tile), rounded to the output type, written to a
//             128-byte-swizzled shared tile that one thread stores with TMA
// Layers with E a multiple of 256 use 128 x 256 tiles instead (W tile
// 256 x 64, a 3-stage ring, 512 TMEM columns): both epilogue groups drain
// every tile, group g columns 128 g .. 128 g + 127.
// Tiles are visited m-major with the N tiles of one row block adjacent, so
// CTAs that share an X tile run together and the re-reads hit L2.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the CTA
// records PMHA_ERR_TIMEOUT in a device word, drains its own TMA copies and
// MMAs (again bounded), frees its tensor memory and returns.
#include <cuda.h>

#include <mutex>
#include <set>
#include <type_traits>
#include <utility>

#include "pmha_internal.h"
#include "tc_util.cuh"

namespace pmha {
namespace {
using namespace tcu;

constexpr int BM = 128, BN = 128, BK = 64;
#ifndef PMHA_GEMM_STAGES
#define PMHA_GEMM_STAGES 4
#endif
constexpr int kStages = PMHA_GEMM_STAGES;
constexpr int kTileABytes = BM * BK * 2;
// Row blocks are taken last-first, so the first rows of the output are the
// last ones written and are still in L2 when the next kernel starts on them
// (the edge kernel walks samples from the first; measured -1.7 % on the n=20k
// layer with L2 flushed before each call).
#ifndef PMHA_GEMM_REVERSE_M
#define PMHA_GEMM_REVERSE_M 1
#endif
#ifndef PMHA_GEMM_EPI_GROUPS
#define PMHA_GEMM_EPI_GROUPS 2
#endif
constexpr int kEpi = PMHA_GEMM_EPI_GROUPS;  // epilogue warpgroups (1 to 3)
static_assert(kEpi >= 1 && kEpi <= 3, "one to three epilogue groups");
constexpr int kAcc = kEpi == 1 ? 2 : kEpi;   // TMEM accumulators (one per group, or two for one group)
constexpr int kThreads = 64 + 128 * kEpi;
constexpr int kOutBoxBytes = BM * 128;             // 128 rows x 64 16-bit columns, 128-byte swizzle
constexpr int kOutTileBytes = 2 * kOutBoxBytes;     // one 128 x 128 output tile

// Tile width WN: 128 columns (BN), or 256 for the wide layers. A tile whose
// operands dominate its traffic waits for them: they reach shared memory at
// about 95 GB/s per SM (a 128 x 128 x 16 MMA itself takes 65 cycles when its
// operands are in place), and a 256-column tile reads 25 % fewer operand
// bytes per output. Wide tiles hold three 48 KB stages; both epilogue
// groups drain every wide tile, group g its columns 128 g .. 128 g + 127,
// through its own staging tile and TMA store.
template <int WN>
struct Tile {
    static_assert(WN == 128 || WN == 256, "128- or 256-column tiles");
    static constexpr bool kSplit = WN > BN;  // every epilogue group takes 128 columns of every tile
    static_assert(!kSplit || kEpi == WN / BN, "one epilogue group per 128 columns of a wide tile");
    static constexpr int kStages = kSplit ? 3 : ::pmha::kStages;
    static constexpr int kTileB = WN * BK * 2;
    static constexpr int kStage = kTileABytes + kTileB;
    static constexpr int kBufs = kEpi == 1 ? 2 : kEpi;                 // staging tiles
    static constexpr int kTmemCols = kAcc * WN <= 256 ? 256 : 512;      // a power of two
    static constexpr int kBias = kEpi * BN * 4;                         // fp32 bias of 128 columns, per group
    static constexpr int kSmem = kStages * kStage + kBufs * kOutTileBytes + kBias + 1024 /*align*/ + 256 /*barriers*/;
    static_assert(kAcc * WN <= 512, "the accumulators fit in tensor memory");
    static_assert(kSmem <= 232448, "shared memory of one CTA");
};

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B of one 16-bit type (bits 7-9 and 10-12: 0 = f16, 1 = bf16), both
// K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
template <typename TIn, int WN>
__host__ __device__ constexpr uint32_t idesc()
{
    constexpr uint32_t f = std::is_same<TIn, __nv_bfloat16>::value ? 1u : 0u;
    return (1u << 4) | (f << 7) | (f << 10) | ((uint32_t)(WN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

struct TcArgs {
    int M, N, K, E;
    const __nv_bfloat16 *bias[3];  // parameters are bf16
    void *out;
    long long ldy;
    int *err;
    // split-K (float output only): tile t covers K blocks [ks * kb_per, ..) of
    // split ks = t % ksplit and writes its partial at out + ks * part_stride
    int ksplit, kb_per;
    long long part_stride;
    // side job: bf16 -> fp16 copy of cvt_n values (out of range sets kErrRangeBit)
    const __nv_bfloat16 *cvt_src;
    __half *cvt_dst;
    int cvt_n;
    int cvt_frag_E;  // nonzero: write the copy in wo_frag_pos order of this E x E matrix
};

// Two fp32 values to one 32-bit word of the output type. fp16 outputs also
// report values outside the fp16 range (or not finite) in *range_bad.
template <typename TOut>
__device__ __forceinline__ uint32_t pack2(float v0, float v1, bool &range_bad);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float v0, float v1, bool &)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float v0, float v1, bool &range_bad)
{
    if (!(fabsf(v0) <= 65504.f) || !(fabsf(v1) <= 65504.f)) range_bad = true;
    __half2 h = __floats2half2_rn(v0, v1);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// named barrier 1 + g over the 128 threads of epilogue group g
__device__ __forceinline__ void epi_sync(int g) { asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory"); }
// same barrier, returning whether any of the 128 threads passed `pred`
__device__ __forceinline__ bool epi_sync_or(int g, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(1 + g)
        : "memory");
    return r != 0;
}

template <typename TIn, typename TOut, int WN>
__global__ void __launch_bounds__(kThreads, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w0,
          const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_w2,
          const __grid_constant__ CUtensorMap tm_y, TcArgs a)
{
    using TL = Tile<WN>;
    constexpr int kStages = TL::kStages, kStageBytes = TL::kStage, kBufs = TL::kBufs, kTmemCols = TL::kTmemCols;
    constexpr int kBiasBytes = TL::kBias;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *tiles = smem;
    uint8_t *staging = smem + kStages * kStageBytes;  // output staging tiles (none for wide tiles)
    float *bias_s = (float *)(staging + kBufs * kOutTileBytes);  // [kEpi][BN]
    uint64_t *bars = (uint64_t *)(staging + kBufs * kOutTileBytes + kBiasBytes);
    uint64_t *full = bars;                    // [kStages]
    uint64_t *empty = bars + kStages;         // [kStages]
    uint64_t *acc_full = bars + 2 * kStages;  // [kAcc]
    uint64_t *acc_empty = acc_full + kAcc;    // [kAcc]
    uint64_t *mma_done = acc_empty + kAcc;    // [1]
    uint32_t *tmem_holder = (uint32_t *)(mma_done + 1);
    volatile int *abort_flag = (volatile int *)(tmem_holder + 1);
    int *issued = (int *)(tmem_holder + 2);  // [kStages]: TMA phases armed per stage

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles_n = a.N / WN;
    const int n_tiles = ((a.M + BM - 1) / BM) * n_tiles_n * a.ksplit;
    const int k_blocks = a.K / BK;
    // tile -> (row block, column block, K split)
    auto decode = [&](int tile, int &m_blk, int &n_blk, int &kb0, int &kb1) {
        const int ks = tile % a.ksplit, mn = tile / a.ksplit;
        m_blk = mn / n_tiles_n;
        n_blk = mn % n_tiles_n;
        if (PMHA_GEMM_REVERSE_M) m_blk = (a.M + BM - 1) / BM - 1 - m_blk;
        kb0 = ks * a.kb_per;
        kb1 = min(k_blocks, kb0 + a.kb_per);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
            issued[s] = 0;
        }
        for (int i = 0; i < kAcc; ++i) {
            mbar_init(smem_u32(&acc_full[i]), 1);
            mbar_init(smem_u32(&acc_empty[i]), 128 * (WN / BN));  // every group that drains the accumulator
        }
        mbar_init(smem_u32(mma_done), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                int m_blk, n_blk, kb0, kb1;
                decode(tile, m_blk, n_blk, kb0, kb1);
                const int n_glob = n_blk * WN;
                const int seg = n_glob / a.E;
                const int n_loc = n_glob - seg * a.E;
                const CUtensorMap *tw = seg == 0 ? &tm_w0 : (seg == 1 ? &tm_w1 : &tm_w2);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, a.err)) break;
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, kStageBytes);
                    issued[stage] += 1;
                    const uint32_t sa = smem_u32(tiles + stage * kStageBytes);
                    tma_load_2d(sa, &tm_x, kb * BK, m_blk * BM, fb);
                    tma_load_2d(sa + kTileABytes, tw, kb * BK, n_loc, fb);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                if (!mbar_wait(smem_u32(&acc_empty[acc]), acc_phase ^ 1u, abort_flag, a.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * WN);
                int m_blk, n_blk, kb0, kb1;
                decode(tile, m_blk, n_blk, kb0, kb1);
                bool ok = true;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(tiles + stage * kStageBytes);
                    const uint64_t da = smem_desc(sa), db = smem_desc(sa + kTileABytes);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // +32 bytes along K inside the swizzle atom = +2 in the address field
                        mma_f16kind(d_tmem, da + (uint64_t)(2 * k), db + (uint64_t)(2 * k), idesc<TIn, WN>(),
                                    (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&acc_full[acc]));
                if (++acc == kAcc) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // all MMAs issued by this thread have finished once this arrives
            mma_commit(smem_u32(mma_done));
            int dummy = 0;
            mbar_wait(smem_u32(mma_done), 0, (volatile int *)&dummy, a.err);
        }
    } else {
        // ---------------- epilogue, kEpi groups of 128 threads: TMEM -> registers
        // (+ bias, rounding) -> swizzled shared tile -> TMA tensor store. The
        // CTA's i-th tile uses accumulator i % 2 and goes to group i % kEpi;
        // the two staging tiles alternate within one group or are one per group.
        const int quarter = warp & 3;
        const int g = (warp - 2) >> 2;          // epilogue group
        const int et = threadIdx.x - 64 - 128 * g;  // 0..127 within the group
        const int r = quarter * 32 + lane;  // tile row of this thread
        float *bias_g = bias_s + g * BN;  // the group's 128 columns of bias
        {
            // Side job before the first accumulator is ready: this CTA's share
            // of the bf16 -> fp16 copy, 8 values (one 16-byte load) a thread
            // and step. (On the producer's idle lanes it held the first TMA
            // loads back by up to 14 us at E = 512: divergent lanes of one warp.)
            const int n8 = a.cvt_n / 8;  // cvt_n is a multiple of 8 (E x E, E a multiple of 64)
            const int per = (n8 + (int)gridDim.x - 1) / (int)gridDim.x;
            const int end = min(n8, ((int)blockIdx.x + 1) * per);
            bool bad = false;
            for (int c = (int)blockIdx.x * per + (threadIdx.x - 64); c < end; c += 128 * kEpi) {
                const uint4 raw = reinterpret_cast<const uint4 *>(a.cvt_src)[c];
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                __half h[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float v = __bfloat162float(__ushort_as_bfloat16((unsigned short)(w[q / 2] >> (16 * (q % 2)))));
                    bad |= !(fabsf(v) <= 65504.f);
                    h[q] = __float2half_rn(v);
                }
                const int i0 = 8 * c;
                if (a.cvt_frag_E) {
                    // k .. k + 7 of one row n: pairs land in four lanes' words
#pragma unroll
                    for (int q = 0; q < 8; q += 2) {
                        const int64_t at = wo_frag_pos((i0 + q) / a.cvt_frag_E, (i0 + q) % a.cvt_frag_E, a.cvt_frag_E);
                        *reinterpret_cast<__half2 *>(a.cvt_dst + at) = __halves2half2(h[q], h[q + 1]);
                    }
                } else {
                    uint4 o;
                    o.x = (uint32_t)__half_as_ushort(h[0]) | ((uint32_t)__half_as_ushort(h[1]) << 16);
                    o.y = (uint32_t)__half_as_ushort(h[2]) | ((uint32_t)__half_as_ushort(h[3]) << 16);
                    o.z = (uint32_t)__half_as_ushort(h[4]) | ((uint32_t)__half_as_ushort(h[5]) << 16);
                    o.w = (uint32_t)__half_as_ushort(h[6]) | ((uint32_t)__half_as_ushort(h[7]) << 16);
                    reinterpret_cast<uint4 *>(a.cvt_dst)[c] = o;
                }
            }
            if (bad) atomicOr(a.err, kErrRangeBit);
        }
        // narrow tiles alternate between the groups; a wide tile goes to both
        const int cg = TL::kSplit ? g * BN : 0;  // the group's first column in the tile
        for (int i = TL::kSplit ? 0 : g;; i += TL::kSplit ? 1 : kEpi) {
            const int tile = blockIdx.x + i * gridDim.x;
            if (tile >= n_tiles) break;
            const int acc = i % kAcc;
            const uint32_t acc_phase = (uint32_t)(i / kAcc) & 1u;
            const int buf = kEpi == 1 ? acc : g;
            int m_blk, n_blk, kb0, kb1;
            decode(tile, m_blk, n_blk, kb0, kb1);
            const int n_glob = n_blk * WN;
            const int seg = n_glob / a.E;
            const int n_loc = n_glob - seg * a.E;
            const __nv_bfloat16 *bias = a.bias[seg];
            // this thread's bias value (column cg + et of the tile), loaded
            // before the accumulator wait so that the wait covers the load
            float bias_v = 0.f;
            if constexpr (!std::is_same<TOut, float>::value)
                if (bias) bias_v = __bfloat162float(bias[n_loc + cg + et]);
            const bool ok = mbar_wait(smem_u32(&acc_full[acc]), acc_phase, abort_flag, a.err);
            // the store that last read this group's staging tile is done
            if (et == 0) {
                if constexpr (kEpi >= 2) bulk_wait_read0();
                else bulk_wait_read1();
            }
            // the readers of the previous tile's bias passed the barrier before its store
            if constexpr (!std::is_same<TOut, float>::value) bias_g[et] = bias_v;
            if (epi_sync_or(g, !ok)) break;  // one decision for all 128 threads
            tc_fence_after();
            const bool live = m_blk * BM + r < a.M;
            if constexpr (std::is_same<TOut, float>::value) {
                // fp32 partial of this K split, stored straight from registers
                float *dst = (float *)a.out + (long long)(tile % a.ksplit) * a.part_stride +
                             (long long)(m_blk * BM + r) * a.ldy + n_glob;
#pragma unroll 1
                for (int c = 0; c < WN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * WN + c * 32), v);
                    if (live) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<uint4 *>(dst + c * 32 + 4 * q) =
                                make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&acc_empty[acc]));
                continue;
            } else {
            uint8_t *sb = staging + buf * kOutTileBytes;
            bool range_bad = false;
            // columns [32c, 32c + 32) of the accumulator: + bias, rounded, into the staging tile
            auto emit = [&](int c, const uint32_t (&v)[32]) {
                uint32_t packed[16];
                bool bad = false;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float v0 = __uint_as_float(v[2 * j]), v1 = __uint_as_float(v[2 * j + 1]);
                    if (bias) {
                        const float2 bb = *reinterpret_cast<const float2 *>(bias_g + c * 32 + 2 * j);
                        v0 = __fadd_rn(v0, bb.x);
                        v1 = __fadd_rn(v1, bb.y);
                    }
                    packed[j] = pack2<TOut>(v0, v1, bad);
                }
                range_bad |= bad && live;
                // 16-byte unit u of the 128-byte row of box c / 2 sits at u ^ (r % 8)
                uint8_t *rowp = sb + (c >> 1) * kOutBoxBytes + r * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int u = (c & 1) * 4 + q;
                    *reinterpret_cast<uint4 *>(rowp + ((u ^ (r & 7)) << 4)) =
                        make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                }
            };
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * WN + cg);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(t_row + (uint32_t)(c * 32), v);
                emit(c, v);
            }
            if (range_bad) atomicOr(a.err, kErrRangeBit);
            // the accumulator has been read: hand it back to the MMA warp
            tc_fence_before();
            mbar_arrive(smem_u32(&acc_empty[acc]));
            // staged tile -> global (rows past M are clipped by the tensor map)
            fence_async_shared();
            epi_sync(g);
            if (et == 0) {
                tma_store_2d(&tm_y, smem_u32(sb), n_glob + cg, m_blk * BM);
                tma_store_2d(&tm_y, smem_u32(sb + kOutBoxBytes), n_glob + cg + 64, m_blk * BM);
                bulk_commit();
            }
            }  // 16-bit output
        }
        if (et == 0) bulk_wait_all();  // the CTA's shared memory must outlive its stores
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let the copies this CTA started land before its shared memory goes away
        int dummy = 0;
        for (int s = 0; s < kStages; ++s)
            if (issued[s] > 0)
                mbar_wait(smem_u32(&full[s]), (uint32_t)((issued[s] - 1) & 1), (volatile int *)&dummy, a.err);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

// 2-D 16-bit row-major tensor (rows x cols, row pitch `pitch` elements),
// box 128 rows x 64 columns, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, bool bf16, int64_t pitch = 0)
{
    return make_map_box(m, base, rows, cols, pitch ? pitch : cols, bf16, BK, BM);
}

}  // namespace

bool gemm_tc_supported(int64_t E)
{
    return E >= BN && E % BN == 0 && E <= 65536;
}

pmha_status gemm_tc(TcType in, TcType out, const void *X, int64_t M, int64_t E, const GemmSegments &seg, void *Y,
                    int64_t ldy, const char *stage, cudaStream_t stream)
{
    if (M <= 0) return PMHA_OK;
    if (M > (int64_t)0x7fffffff - BM) {
        set_error("gemm_tc: %lld rows exceed the 32-bit tile index", (long long)M);
        return PMHA_ERR_UNSUPPORTED;
    }
    if (((uintptr_t)Y & 15) || (ldy * 2) % 16) {
        set_error("gemm_tc: output must be 16-byte aligned with a 16-byte row pitch");
        return PMHA_ERR_INVALID_ARG;
    }
    const bool in_bf16 = in == TcType::BF16;
    // 256-column tiles where every tile lies inside one weight matrix
    const bool wide = E % 256 == 0;
    CUtensorMap mx, mw[3];
    if (!make_map(&mx, X, M, E, in_bf16)) {
        set_error("gemm_tc: cuTensorMapEncodeTiled failed for X (pointer %p)", X);
        return PMHA_ERR_CUDA;
    }
    for (int i = 0; i < 3; ++i) {
        const void *w = seg.w[i < seg.n_seg ? i : 0];
        if (!make_map_box(&mw[i], w, E, E, E, in_bf16, BK, wide ? 256 : BN)) {
            set_error("gemm_tc: cuTensorMapEncodeTiled failed for W (pointer %p)", w);
            return PMHA_ERR_CUDA;
        }
    }
    CUtensorMap my;
    if (!make_map(&my, Y, M, E * seg.n_seg, out == TcType::BF16, ldy)) {
        set_error("gemm_tc: cuTensorMapEncodeTiled failed for Y (pointer %p, pitch %lld)", Y, (long long)ldy);
        return PMHA_ERR_CUDA;
    }
    TcArgs a;
    a.M = (int)M;
    a.N = (int)(E * seg.n_seg);
    a.K = (int)E;
    a.E = (int)E;
    for (int i = 0; i < 3; ++i) a.bias[i] = (const __nv_bfloat16 *)(i < seg.n_seg ? seg.b[i] : nullptr);
    a.out = Y;
    a.ldy = ldy;
    a.err = device_error_word();
    if (!a.err) return PMHA_ERR_CUDA;
    a.ksplit = 1;
    a.kb_per = a.K / BK;
    a.part_stride = 0;
    a.cvt_src = (const __nv_bfloat16 *)seg.cvt_src;
    a.cvt_dst = (__half *)seg.cvt_dst;
    a.cvt_n = seg.cvt_src && seg.cvt_dst ? (int)seg.cvt_n : 0;
    a.cvt_frag_E = (int)seg.cvt_frag_E;
    if (seg.cvt_frag_E && (seg.cvt_frag_E % 64 || seg.cvt_n != seg.cvt_frag_E * seg.cvt_frag_E)) {
        set_error("gemm_tc: fragment-order conversion needs an E x E matrix with E a multiple of 64");
        return PMHA_ERR_UNSUPPORTED;
    }
    if (seg.cvt_n > 0x7fffffff) {
        set_error("gemm_tc: side conversion of %lld values exceeds the 32-bit index", (long long)seg.cvt_n);
        return PMHA_ERR_UNSUPPORTED;
    }

    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcArgs);
    if (wide) {
        if (in_bf16 && out == TcType::F16) kern = k_gemm_tc<__nv_bfloat16, __half, 256>;
        else if (in_bf16) kern = k_gemm_tc<__nv_bfloat16, __nv_bfloat16, 256>;
        else if (out == TcType::BF16) kern = k_gemm_tc<__half, __nv_bfloat16, 256>;
        else kern = k_gemm_tc<__half, __half, 256>;
    } else {
        if (in_bf16 && out == TcType::F16) kern = k_gemm_tc<__nv_bfloat16, __half, BN>;
        else if (in_bf16) kern = k_gemm_tc<__nv_bfloat16, __nv_bfloat16, BN>;
        else if (out == TcType::BF16) kern = k_gemm_tc<__half, __nv_bfloat16, BN>;
        else kern = k_gemm_tc<__half, __half, BN>;
    }
    const int smem_bytes = wide ? Tile<256>::kSmem : Tile<BN>::kSmem;
    static std::mutex mu;
    static std::set<std::pair<int, void *>> configured;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!configured.count({dev, (void *)kern})) {
            PMHA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes));
            configured.insert({dev, (void *)kern});
        }
    }
    const int n_tiles = (int)(((M + BM - 1) / BM) * (a.N / (wide ? 256 : BN)));
    const int grid = std::min(n_tiles, num_sms());
    StageTimer timer(stage, stream);
    kern<<<grid, kThreads, smem_bytes, stream>>>(mx, mw[0], mw[1], mw[2], my, a);
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

pmha_status gemm_tc_general(TcType in, TcType out, const void *X, int64_t ldx, int64_t M, int64_t K, const void *W,
                            int64_t ldw, int64_t N, void *Y, int64_t ldy, int64_t ksplit, const char *stage,
                            cudaStream_t stream)
{
    if (M <= 0) return PMHA_OK;
    if (K % BK || N % BN || K <= 0 || N <= 0 || M > (int64_t)0x7fffffff - BM) {
        set_error("gemm_tc_general: K must be a multiple of %d and N of %d", BK, BN);
        return PMHA_ERR_UNSUPPORTED;
    }
    if (((uintptr_t)X & 15) || ((uintptr_t)W & 15) || ((uintptr_t)Y & 15) || (ldx * 2) % 16 || (ldw * 2) % 16 ||
        (ldy * (out == TcType::F32 ? 4 : 2)) % 16) {
        set_error("gemm_tc_general: operands must be 16-byte aligned with 16-byte row pitches");
        return PMHA_ERR_INVALID_ARG;
    }
    if (in == TcType::F32) {
        set_error("gemm_tc_general: 16-bit operands only");
        return PMHA_ERR_UNSUPPORTED;
    }
    const bool in_bf16 = in == TcType::BF16;
    CUtensorMap mx, mw, my;
    if (!make_map(&mx, X, M, K, in_bf16, ldx) || !make_map(&mw, W, N, K, in_bf16, ldw)) {
        set_error("gemm_tc_general: cuTensorMapEncodeTiled failed for X or W");
        return PMHA_ERR_CUDA;
    }
    if (out != TcType::F32) {
        if (!make_map(&my, Y, M, N, out == TcType::BF16, ldy)) {
            set_error("gemm_tc_general: cuTensorMapEncodeTiled failed for Y");
            return PMHA_ERR_CUDA;
        }
    } else {
        my = mx;  // unused: float partials are stored without TMA
    }
    const int k_blocks = (int)(K / BK);
    if (out != TcType::F32) ksplit = 1;
    ksplit = std::max<int64_t>(1, std::min<int64_t>(ksplit, k_blocks));
    const int kb_per = (int)((k_blocks + ksplit - 1) / ksplit);
    ksplit = (k_blocks + kb_per - 1) / kb_per;  // every split gets at least one K block
    TcArgs a;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.E = (int)N;  // one weight matrix
    for (int i = 0; i < 3; ++i) a.bias[i] = nullptr;
    a.out = Y;
    a.ldy = ldy;
    a.err = device_error_word();
    if (!a.err) return PMHA_ERR_CUDA;
    a.ksplit = (int)ksplit;
    a.kb_per = kb_per;
    a.part_stride = M * ldy;
    a.cvt_src = nullptr;
    a.cvt_dst = nullptr;
    a.cvt_n = 0;
    a.cvt_frag_E = 0;
    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcArgs);
    if (out == TcType::F32) kern = in_bf16 ? k_gemm_tc<__nv_bfloat16, float, BN> : k_gemm_tc<__half, float, BN>;
    else if (in_bf16)
        kern = out == TcType::F16 ? k_gemm_tc<__nv_bfloat16, __half, BN> : k_gemm_tc<__nv_bfloat16, __nv_bfloat16, BN>;
    else kern = out == TcType::BF16 ? k_gemm_tc<__half, __nv_bfloat16, BN> : k_gemm_tc<__half, __half, BN>;
    static std::mutex mu;
    static std::set<std::pair<int, void *>> configured;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!configured.count({dev, (void *)kern})) {
            PMHA_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Tile<BN>::kSmem));
            configured.insert({dev, (void *)kern});
        }
    }
    const int n_tiles = (int)(((M + BM - 1) / BM) * (N / BN) * ksplit);
    const int grid = std::min(n_tiles, num_sms());
    StageTimer timer(stage, stream);
    kern<<<grid, kThreads, Tile<BN>::kSmem, stream>>>(mx, mw, mw, mw, my, a);
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

}  // namespace pmha
