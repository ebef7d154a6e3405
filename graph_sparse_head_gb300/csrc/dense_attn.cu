// Edge attention of a dense graph on the 5th-generation tensor cores
// (kpnn2 PackedMultiheadAttention, Notes steps 2-4). The page observes that
// restricting attention to the graph's edges gives the same mix as dense
// attention whose score matrix is masked to the edges; when most (target,
// source) pairs are edges, the masked dense form is the cheaper one: the
// scores of a 128-target x 128-source tile are one tensor-core product, and
// every k|v row is read once per tile instead of once per edge.
//
// One CTA per (sample b, head h, tile of 128 targets), 6 warps:
//   warp 4   TMA producer: the q tile once, then per 128-source step the k tile
//            (128 sources x d) and the v^T tile (d x 128 sources), 128-byte
//            swizzle, two stages
//   warp 5   allocates 256 TMEM columns and issues, from one thread,
//            S = Q K^T (M=128, N=128, fp32 in TMEM columns 0-127) and
//            O_step = P V (M=128, N=d, TMEM columns 128-..) with tcgen05.mma
//   warps 0-3 one thread per target row: read S from TMEM, mask it (the
//            graph's adjacency bits, key_padding_mask, sources past S),
//            online softmax in log2 units, P in fp16 into a swizzled shared
//            tile (the A operand of P V), then O = O * alpha + O_step in
//            registers; finally mixed = O / l in fp16.
// V enters transposed (channels x tokens, written by a transpose kernel from
// the projection) so that both products take K-major operands.
//
// Every mbarrier wait is bounded; on expiry the CTA records PMHA_ERR_TIMEOUT,
// drains its own copies and MMAs (bounded), frees its tensor memory and returns.
#include <cuda_fp16.h>

#include <set>

#include "tc_util.cuh"

namespace pmha {
namespace {
using namespace tcu;

constexpr int kTM = 128;       // targets per CTA
constexpr int kTN = 128;       // sources per step
constexpr int kThreads = 192;  // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr int kTmemCols = 256;

template <int D>
struct DenseLayout {
    static constexpr int DC = D / 64;               // 64-channel chunks of a head
    static constexpr int kQBytes = DC * kTM * 128;   // q tile
    static constexpr int kKBytes = DC * kTN * 128;   // k tile (two stages)
    static constexpr int kVBytes = 2 * D * 128;      // v^T tile: 2 chunks of 64 sources (two stages)
    static constexpr int kPBytes = 2 * kTM * 128;    // P: 2 chunks of 64 sources
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + 2 * kKBytes;
    static constexpr int kOffP = kOffV + 2 * kVBytes;
    static constexpr int kOffWords = kOffP + kPBytes;  // uint32 [2][4] source-validity words
    static constexpr int kOffBars = kOffWords + 32;
    static constexpr int kSmem = kOffBars + 160;     // the base is 1024-byte aligned (checked)
};
static_assert(2 * (DenseLayout<64>::kSmem + 1024) <= 233472, "two CTAs per SM at head_dim 64");

struct DenseArgs {
    int B, L, S, H, n_tiles_t;
    int S_pad;                    // columns per sample in V^T (S rounded up to 8)
    float score_scale;            // log2(e) / sqrt(d)
    const uint32_t *adj;          // L x words_per_row adjacency bits, or null (complete graph)
    long long words_per_row;
    const uint8_t *kpm;           // (B, S) or null
    __half *mixed;                // (B, L, E)
    int E;
    int *err;
};

// Instruction descriptor, kind::f16 with f16 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// barrier 1 over the 128 softmax threads, returning whether any of them passed `pred`
__device__ __forceinline__ bool softmax_vote(bool pred)
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
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// 32 columns of this warp's 32 TMEM lanes, without waiting for them
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// a row's reference maximum moves only when a score passes it by more than this (log2 units)
constexpr float kLazy = 8.f;

// 2^x on the FMA pipe, for a share of the softmax's exponentials (the
// multi-function unit gives 16 exponentials a clock per SM, a quarter of
// what the tensor pipe feeds at head_dim 64). Range reduction x = j + f with
// j = round(x) (the 1.5 * 2^23 shift puts j in the low mantissa bits of t)
// and f in [-1/2, 1/2]; 2^f from a cubic fitted for this kernel as the
// minimax of the relative error on [-1/2, 1/2] (7.5e-5, under half an fp16
// step: P enters P V in fp16); j is added to the exponent field (the bits of
// t shifted by 23 are j << 23, since those of 1.5 * 2^23 end in 23 zeros).
// x is at most kLazy + the step's rounding; inputs below -125 give about
// 2^-125 instead of 0, which rounds to 0 in fp16 and is nothing against a
// row sum of at least 2^-kLazy.
constexpr float kExpC0 = 9.999280572e-01f, kExpC1 = 6.932609677e-01f, kExpC2 = 2.426113188e-01f,
                kExpC3 = 5.517175049e-02f;
__device__ __forceinline__ float ex2_fma(float x)
{
    x = fmaxf(x, -125.f);
    const float t = __fadd_rn(x, 12582912.f);
    const float f = __fsub_rn(x, __fsub_rn(t, 12582912.f));
    float p = __fmaf_rn(kExpC3, f, kExpC2);
    p = __fmaf_rn(p, f, kExpC1);
    p = __fmaf_rn(p, f, kExpC0);
    return __int_as_float(__float_as_int(p) + (int)((uint32_t)__float_as_int(t) << 23));
}
// Pairs of columns (of 16 in 32) whose exponentials take ex2_fma: every
// (16 / kEmuPairs)-th pair. 0 keeps every exponential on ex2.approx.
#ifndef PMHA_DENSE_EMU_PAIRS
#define PMHA_DENSE_EMU_PAIRS 0
#endif
constexpr int kEmuPairs = PMHA_DENSE_EMU_PAIRS;
static_assert(kEmuPairs == 0 || (16 % (kEmuPairs > 0 ? kEmuPairs : 1) == 0), "an even spread of emulated pairs");
__device__ __forceinline__ constexpr bool emulated_pair(int i)
{
    return kEmuPairs > 0 && (i % (16 / (kEmuPairs > 0 ? kEmuPairs : 1))) == (16 / (kEmuPairs > 0 ? kEmuPairs : 1)) - 1;
}

// Paired fp32 arithmetic for the softmax pass (each half rounds like the
// scalar instruction) and a three-input maximum: fewer instructions per
// score in a pass that is bound by instruction issue.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float x, float y)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 unpack2(f32x2 r)
{
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
    return f;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// head_dim 64: two CTAs per SM (registers capped at 170 a thread); 128: one
template <int D>
__global__ void __launch_bounds__(kThreads, D == 64 ? 2 : 1)
k_dense_attn(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_vt, DenseArgs a)
{
    using LY = DenseLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint32_t *words = (uint32_t *)(smem + LY::kOffWords);
    uint64_t *bars = (uint64_t *)(smem + LY::kOffBars);
    uint64_t *q_full = bars;         // [1]
    uint64_t *k_full = bars + 1;     // [2]
    uint64_t *k_empty = bars + 3;    // [2]
    uint64_t *v_full = bars + 5;     // [2]
    uint64_t *v_empty = bars + 7;    // [2]
    uint64_t *s_full = bars + 9;     // [1]
    uint64_t *s_free = bars + 10;    // [1]
    uint64_t *p_full = bars + 11;    // [1]
    uint64_t *o_full = bars + 12;    // [1] one phase per P V product
    uint64_t *mma_done = bars + 13;  // [1]
    uint32_t *tmem_holder = (uint32_t *)(bars + 14);
    volatile int *abort_flag = (volatile int *)(tmem_holder + 1);
    int *issued = (int *)(tmem_holder + 2);  // [5]: TMA phases armed (q, k stages 0 and 1, v stages 0 and 1)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int it = blockIdx.x % a.n_tiles_t;
    const int bh = blockIdx.x / a.n_tiles_t;
    const int h = bh % a.H, b = bh / a.H;
    const int t0 = it * kTM;
    const int n_steps = (a.S + kTN - 1) / kTN;

    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(a.err, kErrInternalBit);
        return;
    }
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(q_full), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&k_full[s]), 1);
            mbar_init(smem_u32(&k_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&v_full[s]), 1);
            mbar_init(smem_u32(&v_empty[s]), 1);
        }
        mbar_init(smem_u32(s_full), 1);
        mbar_init(smem_u32(s_free), 128);
        mbar_init(smem_u32(p_full), 128);
        mbar_init(smem_u32(o_full), 1);
        mbar_init(smem_u32(mma_done), 1);
        issued[0] = issued[1] = issued[2] = issued[3] = issued[4] = 0;
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5) {
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
    const uint32_t tmem_s = tmem_base, tmem_o = tmem_base + kTN;

    if (warp == 4) {
        if (lane == 0) {
            // ---------------- TMA producer: q, k_0, then per step v_j and k_{j+1}
            const uint32_t qb = smem_u32(q_full);
            mbar_arrive_expect_tx(qb, LY::kQBytes);
            issued[0] = 1;
#pragma unroll
            for (int c = 0; c < LY::DC; ++c)
                tma_load_2d(smem_u32(smem + LY::kOffQ + c * kTM * 128), &tm_q, h * D + c * 64, b * a.L + t0, qb);
            auto load_k = [&](int j) -> bool {
                const int s = j & 1;
                if (!mbar_wait(smem_u32(&k_empty[s]), ((j >> 1) & 1) ^ 1u, abort_flag, a.err)) return false;
                const uint32_t fb = smem_u32(&k_full[s]);
                mbar_arrive_expect_tx(fb, LY::kKBytes);
                issued[1 + s] += 1;
                const uint32_t kdst = smem_u32(smem + LY::kOffK + s * LY::kKBytes);
#pragma unroll
                for (int c = 0; c < LY::DC; ++c)
                    tma_load_2d(kdst + c * kTN * 128, &tm_k, h * D + c * 64, b * a.S + j * kTN, fb);
                return true;
            };
            bool ok = load_k(0);
            for (int j = 0; ok && j < n_steps; ++j) {
                const int vs = j & 1;
                if (!mbar_wait(smem_u32(&v_empty[vs]), ((j >> 1) & 1) ^ 1u, abort_flag, a.err)) break;
                const uint32_t fb = smem_u32(&v_full[vs]);
                mbar_arrive_expect_tx(fb, LY::kVBytes);
                issued[3 + vs] += 1;
                const uint32_t vdst = smem_u32(smem + LY::kOffV + vs * LY::kVBytes);
#pragma unroll
                for (int kc = 0; kc < 2; ++kc)
                    tma_load_2d(vdst + kc * D * 128, &tm_vt, b * a.S_pad + j * kTN + kc * 64, h * D, fb);
                if (j + 1 < n_steps) ok = load_k(j + 1);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ---------------- MMA issuer: S(j + 1) as soon as the softmax has read
            // S(j), then O += P(j) V(j) (O accumulates in tensor memory)
            bool ok = mbar_wait(smem_u32(q_full), 0, abort_flag, a.err);
            tc_fence_after();
            const uint32_t qa = smem_u32(smem + LY::kOffQ);
            const uint32_t pa = smem_u32(smem + LY::kOffP);
            auto issue_s = [&](int j) -> bool {
                const int s = j & 1;
                if (!mbar_wait(smem_u32(&k_full[s]), (j >> 1) & 1, abort_flag, a.err)) return false;
                if (j > 0 && !mbar_wait(smem_u32(s_free), (j - 1) & 1, abort_flag, a.err)) return false;
                tc_fence_after();
                const uint32_t ka = smem_u32(smem + LY::kOffK + s * LY::kKBytes);
#pragma unroll
                for (int c = 0; c < LY::DC; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16kind(tmem_s, smem_desc(qa + c * kTM * 128) + (uint64_t)(2 * k),
                                    smem_desc(ka + c * kTN * 128) + (uint64_t)(2 * k), idesc_f16(kTM, kTN),
                                    (c > 0 || k > 0) ? 1u : 0u);
                mma_commit(smem_u32(s_full));
                mma_commit(smem_u32(&k_empty[s]));
                return true;
            };
            ok = ok && issue_s(0);
            for (int j = 0; ok && j < n_steps; ++j) {
                if (j + 1 < n_steps && !(ok = issue_s(j + 1))) break;
                const int vs = j & 1;
                if (!(ok = mbar_wait(smem_u32(p_full), j & 1, abort_flag, a.err))) break;
                if (!(ok = mbar_wait(smem_u32(&v_full[vs]), (j >> 1) & 1, abort_flag, a.err))) break;
                tc_fence_after();
                const uint32_t va = smem_u32(smem + LY::kOffV + vs * LY::kVBytes);
#pragma unroll
                for (int kc = 0; kc < 2; ++kc)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_f16kind(tmem_o, smem_desc(pa + kc * kTM * 128) + (uint64_t)(2 * k),
                                    smem_desc(va + kc * D * 128) + (uint64_t)(2 * k), idesc_f16(kTM, D),
                                    (j > 0 || kc > 0 || k > 0) ? 1u : 0u);
                mma_commit(smem_u32(o_full));
                mma_commit(smem_u32(&v_empty[vs]));
            }
            // all MMAs issued by this thread have finished once this arrives
            mma_commit(smem_u32(mma_done));
            int dummy = 0;
            mbar_wait(smem_u32(mma_done), 0, (volatile int *)&dummy, a.err);
        }
    } else {
        // ---------------- softmax and accumulation: thread r owns target row t0 + r
        const int r = threadIdx.x;  // 0..127
        const int t = t0 + r;
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        // m: the row's reference (log2 units), raised only when a step's maximum
        // passes it by more than kLazy; P <= 2^kLazy stays well inside fp16
        float m = -INFINITY, l = 0.f;
        const uint32_t *adj_row = (a.adj && t < a.L) ? a.adj + (long long)t * a.words_per_row : nullptr;
        uint8_t *P = smem + LY::kOffP;
        bool ok = true;
        for (int j = 0; j < n_steps; ++j) {
            // A step whose 128 sources all exist and are all live for every row
            // (complete graph, no padding mask, not past S) needs no mask.
            const bool full = !a.adj && !a.kpm && (j + 1) * kTN <= a.S;
            uint32_t rb[4] = {~0u, ~0u, ~0u, ~0u};
            if (!full) {
                // sources that exist and are not padding: one bit per column, one word per warp
                const int sc = j * kTN + r;
                bool col_ok = sc < a.S;
                if (col_ok && a.kpm) col_ok = a.kpm[(long long)b * a.S + sc] == 0;
                const unsigned wbits = __ballot_sync(0xffffffffu, col_ok);
                if (lane == 0) words[(j & 1) * 4 + warp] = wbits;
                if (a.adj) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const long long wi = (long long)j * 4 + w;
                        rb[w] = (adj_row && wi < a.words_per_row) ? adj_row[wi] : 0u;
                    }
                }
                softmax_sync();
#pragma unroll
                for (int w = 0; w < 4; ++w) rb[w] &= words[(j & 1) * 4 + w];
            }

            ok = !softmax_vote(!mbar_wait(smem_u32(s_full), j & 1, abort_flag, a.err));
            if (!ok) break;
            tc_fence_after();
            uint32_t v0[32], v1[32];
            // pass 1: the step's row max of the raw products (the scale is positive)
            float mx = -INFINITY;
            tmem_ld32_async(tmem_s + lane_off, v0);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < kTN / 32; ++c) {
                uint32_t(&cur)[32] = (c & 1) ? v1 : v0;
                uint32_t(&nxt)[32] = (c & 1) ? v0 : v1;
                if (c + 1 < kTN / 32) tmem_ld32_async(tmem_s + lane_off + (uint32_t)((c + 1) * 32), nxt);
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float x0 = __uint_as_float(cur[2 * i]), x1 = __uint_as_float(cur[2 * i + 1]);
                    m4[i & 3] = max3(m4[i & 3], full ? x0 : (((rb[c] >> (2 * i)) & 1u) ? x0 : -INFINITY),
                                     full ? x1 : (((rb[c] >> (2 * i + 1)) & 1u) ? x1 : -INFINITY));
                }
                mx = fmaxf(mx, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
                if (c + 1 < kTN / 32) tmem_wait_ld();
            }
            const float mxs = __fmul_rn(mx, a.score_scale);
            const bool move = mxs > m + kLazy;  // also when m is still -inf and the step has a live source
            const float m_new = move ? mxs : m;
            // ex2.approx(-inf) is +0: masked columns add nothing; the offset 0
            // stands in for a reference that is still -inf (no live source yet)
            const float m_off = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = move ? ex2_approx(__fsub_rn(m, m_off)) : 1.f;
            // pass 2: P = 2^(s * scale - m) in fp16 (kept in registers) and the row sum
            f32x2 sum2[2] = {pack2(0.f, 0.f), pack2(0.f, 0.f)};
            const f32x2 scale2 = pack2(a.score_scale, a.score_scale), neg_m2 = pack2(-m_off, -m_off);
            uint32_t pk[kTN / 32][16];
            tmem_ld32_async(tmem_s + lane_off, v0);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < kTN / 32; ++c) {
                uint32_t(&cur)[32] = (c & 1) ? v1 : v0;
                uint32_t(&nxt)[32] = (c & 1) ? v0 : v1;
                if (c + 1 < kTN / 32) tmem_ld32_async(tmem_s + lane_off + (uint32_t)((c + 1) * 32), nxt);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float2 x = unpack2(
                        fma2(pack2(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), scale2, neg_m2));
                    float p0 = emulated_pair(i) ? ex2_fma(x.x) : ex2_approx(x.x);
                    float p1 = emulated_pair(i) ? ex2_fma(x.y) : ex2_approx(x.y);
                    if (!full) {
                        p0 = ((rb[c] >> (2 * i)) & 1u) ? p0 : 0.f;
                        p1 = ((rb[c] >> (2 * i + 1)) & 1u) ? p1 : 0.f;
                    }
                    sum2[i & 1] = add2(sum2[i & 1], pack2(p0, p1));
                    const __half2 hp = __floats2half2_rn(p0, p1);
                    pk[c][i] = *reinterpret_cast<const uint32_t *>(&hp);
                }
                if (c + 1 < kTN / 32) tmem_wait_ld();
            }
            // S has been read: the MMA warp may compute S(j + 1)
            tc_fence_before();
            mbar_arrive(smem_u32(s_free));
            if (j > 0) {
                // P(j - 1) has been consumed and O holds steps 0 .. j-1 once P V(j - 1) is done;
                // a row whose reference moved rescales its O in tensor memory now, before P V(j)
                ok = !softmax_vote(!mbar_wait(smem_u32(o_full), (j - 1) & 1, abort_flag, a.err));
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, move)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        const uint32_t oa = tmem_o + lane_off + (uint32_t)(c * 32);
                        tmem_ld32_async(oa, v0);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) v0[i] = __float_as_uint(__fmul_rn(__uint_as_float(v0[i]), alpha));
                        tmem_st32(oa, v0);
                    }
                    tmem_wait_st();
                }
            }
            // P into the swizzled A tile: columns c*32 .. c*32+31 = chunk c/2, 16-byte units 4*(c%2) .. +3
#pragma unroll
            for (int c = 0; c < kTN / 32; ++c) {
                uint8_t *rowp = P + (c >> 1) * (kTM * 128) + r * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int u = (c & 1) * 4 + q;
                    *reinterpret_cast<uint4 *>(rowp + ((u ^ (r & 7)) << 4)) =
                        make_uint4(pk[c][4 * q], pk[c][4 * q + 1], pk[c][4 * q + 2], pk[c][4 * q + 3]);
                }
            }
            // P is ready for the tensor cores (and O rescaled)
            tc_fence_before();
            fence_async_shared();
            mbar_arrive(smem_u32(p_full));
            const float2 sa = unpack2(sum2[0]), sb = unpack2(sum2[1]);
            const float sum = __fadd_rn(__fadd_rn(sa.x, sb.x), __fadd_rn(sa.y, sb.y));
            l = __fadd_rn(__fmul_rn(l, alpha), sum);
            m = m_new;
        }
        if (ok) {
            // the last P V product completes O
            ok = !softmax_vote(!mbar_wait(smem_u32(o_full), (n_steps - 1) & 1, abort_flag, a.err));
            if (ok) tc_fence_after();
        }
        if (ok) {
            // mixed = O / l (a target without a live source mixes to zeros). The
            // tensor-memory loads are warp-collective: every lane runs them,
            // only rows of real targets (t < L) store.
            const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
            __half *dst = a.mixed + ((long long)b * a.L + t) * a.E + h * D;
            bool bad = false;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                tmem_ld32_async(tmem_o + lane_off + (uint32_t)(cc * 32), ov);
                tmem_wait_ld();
                if (t >= a.L) continue;
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float x0 = __fmul_rn(__uint_as_float(ov[c + 2 * i]), inv);
                        const float x1 = __fmul_rn(__uint_as_float(ov[c + 2 * i + 1]), inv);
                        if (!(fabsf(x0) <= 65504.f) || !(fabsf(x1) <= 65504.f)) bad = true;
                        const __half2 hv = __floats2half2_rn(x0, x1);
                        w[i] = *reinterpret_cast<const uint32_t *>(&hv);
                    }
                    *reinterpret_cast<uint4 *>(dst + cc * 32 + c) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            if (bad) atomicOr(a.err, kErrRangeBit);
        }
        if (warp < 4) tc_fence_before();
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let the copies this CTA started land before its shared memory goes away
        int dummy = 0;
        if (issued[0]) mbar_wait(smem_u32(q_full), 0, (volatile int *)&dummy, a.err);
        for (int s = 0; s < 2; ++s)
            if (issued[1 + s] > 0)
                mbar_wait(smem_u32(&k_full[s]), (uint32_t)((issued[1 + s] - 1) & 1), (volatile int *)&dummy,
                          a.err);
        for (int s = 0; s < 2; ++s)
            if (issued[3 + s] > 0)
                mbar_wait(smem_u32(&v_full[s]), (uint32_t)((issued[3 + s] - 1) & 1), (volatile int *)&dummy,
                          a.err);
    }
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// V (B*S rows of pitch v_ld, E channels) -> V^T (E rows, B*S_pad columns;
// sample b at columns b*S_pad.., its padding columns zero). 64 x 64 tiles:
// 16-byte loads of 8 channels, a shared tile with a 66-element pitch (the
// transposed reads hit 8 different banks), 16-byte stores of 8 tokens.
// E, v_ld and S_pad are multiples of 8.
__global__ void __launch_bounds__(256) k_transpose_v(const __half *__restrict__ v, long long v_ld, int S, int S_pad,
                                                     long long cols, int E, __half *__restrict__ vt)
{
    __shared__ __half tile[64][66];
    const long long r0 = (long long)blockIdx.x * 64;  // padded token index
    const int c0 = blockIdx.y * 64;                    // channel
    const int t = threadIdx.x;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int idx = t + 256 * k;
        const int row = idx >> 3, cu = idx & 7;
        const long long r = r0 + row;
        const long long b = r / S_pad, s = r - b * S_pad;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < cols && s < S && c0 + cu * 8 < E)
            val = *reinterpret_cast<const uint4 *>(v + (b * S + s) * v_ld + c0 + cu * 8);
        const __half *hv = reinterpret_cast<const __half *>(&val);
#pragma unroll
        for (int i = 0; i < 8; ++i) tile[row][cu * 8 + i] = hv[i];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int idx = t + 256 * k;
        const int ch = idx >> 3, tu = idx & 7;
        __align__(16) __half hv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) hv[i] = tile[tu * 8 + i][ch];
        const long long r = r0 + tu * 8;
        if (c0 + ch < E && r < cols)
            *reinterpret_cast<uint4 *>(vt + (long long)(c0 + ch) * cols + r) = *reinterpret_cast<const uint4 *>(hv);
    }
}

template <int D>
pmha_status launch_dense(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mvt, const DenseArgs &a,
                         cudaStream_t s)
{
    using LY = DenseLayout<D>;
    static std::mutex mu;
    static std::set<int> configured;
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!configured.count(dev)) {
            PMHA_CUDA_TRY(
                cudaFuncSetAttribute(k_dense_attn<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kSmem));
            configured.insert(dev);
        }
    }
    const long long grid = (long long)a.B * a.H * a.n_tiles_t;
    k_dense_attn<D><<<(unsigned)grid, kThreads, LY::kSmem, s>>>(mq, mk, mvt, a);
    return PMHA_OK;
}

}  // namespace

bool dense_supported(const pmha_graph *g, int64_t E, int64_t H, TcType t)
{
    if (!g->dense || t != TcType::F16 || H < 1 || E % H) return false;
    const int64_t d = E / H;
    return d == 64 || d == 128;
}

static int64_t s_pad(const pmha_graph *g) { return (g->S + 7) / 8 * 8; }

size_t dense_vt_bytes(const pmha_graph *g, int64_t B, int64_t E) { return (size_t)(B * s_pad(g) * E) * 2; }

pmha_status dense_attention(const pmha_graph *g, const DenseInputs &in, cudaStream_t s)
{
    const int64_t E = in.E, H = in.H, d = E / H, B = in.B, L = g->L, S = g->S, SP = s_pad(g);
    if (B * SP > 0x7fffffffLL || B * L > 0x7fffffffLL) {
        set_error("dense attention: more than 2^31 token rows");
        return PMHA_ERR_UNSUPPORTED;
    }
    {
        StageTimer timer("transpose_v", s);
        dim3 grid((unsigned)((B * SP + 63) / 64), (unsigned)((E + 63) / 64));
        k_transpose_v<<<grid, 256, 0, s>>>((const __half *)in.v, in.v_ld, (int)S, (int)SP, B * SP, (int)E,
                                           (__half *)in.vt);
        count_launch();
        PMHA_CUDA_TRY(cudaGetLastError());
    }
    CUtensorMap mq, mk, mvt;
    if (!make_map_box(&mq, in.q, B * L, E, in.q_ld, false, 64, kTM) ||
        !make_map_box(&mk, in.k, B * S, E, in.k_ld, false, 64, kTN) ||
        !make_map_box(&mvt, in.vt, E, B * SP, B * SP, false, 64, (uint32_t)d)) {
        set_error("dense attention: cuTensorMapEncodeTiled failed");
        return PMHA_ERR_CUDA;
    }
    DenseArgs a;
    a.B = (int)B;
    a.L = (int)L;
    a.S = (int)S;
    a.S_pad = (int)SP;
    a.H = (int)H;
    a.n_tiles_t = (int)((L + kTM - 1) / kTM);
    a.score_scale = (float)(1.4426950408889634 / sqrt((double)d));
    a.adj = g->dense_complete ? nullptr : g->adj;
    a.words_per_row = g->adj_words_per_row;
    a.kpm = in.kpm;
    a.mixed = (__half *)in.mixed;
    a.E = (int)E;
    a.err = device_error_word();
    if (!a.err) return PMHA_ERR_CUDA;
    StageTimer timer("dense_attn", s);
    const pmha_status st = d == 64 ? launch_dense<64>(mq, mk, mvt, a, s) : launch_dense<128>(mq, mk, mvt, a, s);
    if (st != PMHA_OK) return st;
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

}  // namespace pmha
