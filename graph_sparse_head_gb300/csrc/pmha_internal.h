// Internal declarations shared by the translation units of libpmha.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pmha.h"

namespace pmha {

// --------------------------------------------------------------------------
// Graph: the live edges grouped by target, plus the work plan of the edge
// kernel. Everything lives in one device allocation owned by the graph.
//
// Work plan: the CSR positions [0, nnz) of one sample are cut into units of
// kUnitEdges consecutive positions. A unit walks the targets its positions
// belong to, in order. A target whose edges all lie in one unit is finished
// there; a target that crosses a unit boundary is finished by the slot that
// writes its last piece, from partial softmax states that the units write to
// two slots per unit: slot 2u for the unit's first target, slot 2u + 1 for
// its last. Targets with no edge get their zero mix from a small kernel.
// --------------------------------------------------------------------------

#ifndef PMHA_UNIT_EDGES
#define PMHA_UNIT_EDGES 176
#endif
constexpr int kUnitEdges = PMHA_UNIT_EDGES;

}  // namespace pmha

struct pmha_graph {
    int64_t L = 0, S = 0;
    int64_t nnz_given = 0, nnz = 0;   // nnz counts appended self-loops
    int64_t max_deg = 0;
    int64_t n_units = 0;              // units per sample, ceil(nnz / kUnitEdges)
    int64_t n_merge = 0;              // targets crossing a unit boundary or without edges
    int device = 0;
    int32_t *row_ptr = nullptr;       // L + 1
    int32_t *col = nullptr;           // nnz, source per CSR position
    int32_t *perm = nullptr;          // nnz, given-order edge id per CSR position
    int32_t *tgt_of_edge = nullptr;   // nnz, target per given-order edge id
    int32_t *tgt_of_pos = nullptr;    // nnz, target per CSR position
    int32_t *unit_first_t = nullptr;  // n_units, target of each unit's first position
    int32_t *unit_order = nullptr;    // n_units, the units by decreasing estimated work (ties by index)
    int32_t *merge_t = nullptr;       // n_merge, targets to merge (crossing a unit boundary, or without edges)
    int32_t *merge_pos = nullptr;     // L, index of each target in merge_t, or -1
    int64_t n_empty = 0;              // targets without edges
    // The same edges by source (for the backward pass): positions sorted by
    // (source, target); units of kUnitEdges positions; sources to merge.
    int32_t *src_row_ptr = nullptr;   // S + 1
    int32_t *tgt_by_src = nullptr;    // nnz, target per by-source position
    int32_t *unit_first_s = nullptr;  // n_units, source of each unit's first position
    int32_t *merge_s = nullptr;       // n_merge_s, sources crossing a unit boundary, or without edges
    int64_t n_merge_s = 0;
    int64_t max_out_deg = 0;
    // Dense graphs (most (target, source) pairs are edges): the adjacency as
    // bits, row t = words [t * adj_words_per_row, ...), bit s % 32 of word s / 32.
    bool dense = false;               // the masked-dense kernel may run this graph
    bool dense_complete = false;      // every pair is an edge: no mask needed
    uint32_t *adj = nullptr;          // L * adj_words_per_row words (own allocation), or null
    int64_t adj_words_per_row = 0;
    void *mem = nullptr;              // the single allocation behind the arrays above
    // Targets with at least heavy_min_deg edges run on the tensor cores
    // (heavy.cu); the others keep the per-edge kernel, which then walks
    // `light`: the same L targets and S sources with only the light targets'
    // edges (heavy targets have none there). No split: light == nullptr.
    int64_t heavy_min_deg = 0;
    int64_t n_heavy = 0;
    int4 *heavy_info = nullptr;       // n_heavy {target, first CSR position, in-degree, 128-edge tiles},
                                      // in-degree non-increasing (own allocation)
    pmha_graph *light = nullptr;
};

namespace pmha {

// ---------------------------------------------------------------- errors
void set_error(const char *fmt, ...);
pmha_status cuda_fail(cudaError_t e, const char *what);
#define PMHA_CUDA_TRY(expr)                                     \
    do {                                                        \
        cudaError_t _e = (expr);                                \
        if (_e != cudaSuccess) return ::pmha::cuda_fail(_e, #expr); \
    } while (0)

// Device word of sticky error bits set by kernels: a bounded wait gave up,
// or an fp16 intermediate left the fp16 range. Read by pmha_device_status.
int *device_error_word();
constexpr int kErrTimeoutBit = 1;
constexpr int kErrRangeBit = 2;
constexpr int kErrInternalBit = 4;  // a kernel found its launch unusable (e.g. shared memory misaligned) and did nothing

// ---------------------------------------------------------------- profiling
// Records an event pair around a launch when profiling is on.
struct StageTimer {
    StageTimer(const char *stage, cudaStream_t s);
    ~StageTimer();
    const char *stage;
    cudaStream_t stream;
    int slot;
};
void count_launch(int n = 1);
int num_sms();

// ---------------------------------------------------------------- CSR build
pmha_status build_csr(const int64_t *src, const int64_t *tgt, int64_t nnz, int64_t L, int64_t S,
                      bool self_loops, cudaStream_t stream, pmha_graph **out);

// ---------------------------------------------------------------- GEMMs
// Y[m, n] = sum_k X[m, k] * W_seg[n - seg*E, k] + bias_seg[n - seg*E]
// for n in [0, n_seg * E), where seg = n / E; X is (M, E) with row stride E,
// Y has row stride ldy. Up to three weight segments (Q|K|V fused).
struct GemmSegments {
    const void *w[3];
    const void *b[3];
    int n_seg;
    // optional side job of the tensor-core kernel: convert cvt_n bf16 values
    // at cvt_src to fp16 at cvt_dst (out_proj's weight, while step 1 runs)
    const void *cvt_src = nullptr;
    void *cvt_dst = nullptr;
    int64_t cvt_n = 0;
    // nonzero: cvt_src is an E x E matrix (E = cvt_frag_E) and the copy is
    // written in the mma.sync fragment order of wo_frag_pos
    int64_t cvt_frag_E = 0;
};

// Place (in fp16 elements) of W[n][k] of an E x E matrix (E a multiple of
// 64) in the B-fragment order of mma.sync m16n8k16 with B[k][n] = W[n][k]:
// for output tile j (columns 8 j .. 8 j + 7) and k-steps 2 kp, 2 kp + 1, lane
// l's four 32-bit registers (b0, b1 of step 2 kp, then of step 2 kp + 1) are
// 16 consecutive bytes, and the 32 lanes' 512 bytes follow one another. b0
// of a step holds k = 2 (l % 4) + {0, 1}, b1 the same k + 8, both for
// n = 8 j + l / 4.
__host__ __device__ inline int64_t wo_frag_pos(int n, int k, int E)
{
    const int j = n >> 3, nn = n & 7, ks = k >> 4, kk = k & 15;
    const int kp = ks >> 1, kh = ks & 1;
    const int lane = nn * 4 + ((kk & 7) >> 1);
    const int r = kh * 2 + (kk >> 3);
    const int64_t word = (((int64_t)j * (E / 32) + kp) * 32 + lane) * 4 + r;
    return word * 2 + (kk & 1);
}
// Element types on the projection path. Layers stored in bf16 keep their
// intermediates (q, k, v, mixed) in fp16; float32 layers stay float32.
enum class TcType { BF16, F16, F32 };
inline size_t type_size(TcType t) { return t == TcType::F32 ? 4 : 2; }

// Tensor-core GEMM: X and W both `in` (bf16 or fp16), biases bf16, Y `out`.
// `stage` names the launch for the stage timer (a string literal).
bool gemm_tc_supported(int64_t E);
pmha_status gemm_tc(TcType in, TcType out, const void *X, int64_t M, int64_t E, const GemmSegments &seg, void *Y,
                    int64_t ldy, const char *stage, cudaStream_t stream);
// CUDA-core GEMM with independent types for X, W (and bias) and Y.
pmha_status gemm_simt(TcType tx, TcType tw, TcType ty, const void *X, int64_t M, int64_t E,
                      const GemmSegments &seg, void *Y, int64_t ldy, const char *stage, cudaStream_t stream);
// dst[i] = fp16(src[i]) for n bf16 values (the out_proj weight of a bf16 layer).
pmha_status convert_bf16_to_f16(const void *src, void *dst, int64_t n, cudaStream_t stream);

// ---------------------------------------------------------------- edge attention
struct EdgeArgs {
    const void *q;        // (B, L) rows, row stride q_ld elements, head h at columns h*d..
    int64_t q_ld;
    const void *kv;       // (B, S) rows: K at columns [0, E), V at [v_off, v_off + E)
    int64_t kv_ld;
    int64_t v_off;
    void *mixed;          // (B, L, E) output of the mix (light targets written directly)
    float *part;          // (B, 2 n_units, 2H + E): per slot m[H], l[H], acc[E] of a crossing target
    float *ml;            // (B, L, H, 2): softmax reference m (log2 units, at most 8 below the largest
                          // score) and l = sum of 2^(s - m), per target/head
    float *scores;        // (B, nnz, H): raw scores (log2 units) by CSR position, or null
    int *counters;        // kCounterHead words (a task counter), then (B, n_merge) pieces written per
                          // crossing target; zeroed by edge_attention before the edge kernel
    const uint8_t *kpm;   // (B, S) key_padding_mask, nonzero = key dropped, or null
    uint32_t *kpm_bits;   // (B, ceil(nnz / 32)) scratch: bit p of word w = key of CSR position 32 w + p dropped
    int64_t B, L, S, E, H, nnz;
    float score_scale;    // log2(e) / sqrt(d)
    bool with_values;     // false: scores and (m, l) only
    // out_proj inside the edge kernel (fused_out_supported): out (B, L, E)
    // layer-type rows = mixed . Wo^T + bo, with Wo as fp16 in wo_frag_pos
    // order; the mixed rows still pass through `mixed`. Null: mixed only.
    void *out = nullptr;
    const void *wo_frag = nullptr;
    const void *bo = nullptr;
};
constexpr int kCounterHead = 64;  // words before the merge counters (256 bytes)
// Targets per out_proj task of the fused edge kernel; the counter region
// ends with (B, ceil(L / kOutRows)) counts of finished targets per block.
constexpr int kOutRows = 64;
inline int64_t out_blocks(int64_t L) { return (L + kOutRows - 1) / kOutRows; }
// The fused out_proj runs in the ring edge kernel for fp16 intermediates,
// embed_dim 128 (with heads of at least 16 channels): each block holds Wo.
bool fused_out_supported(TcType t, int64_t E, int64_t H);
// `t` is the intermediate type (F16 or F32) of q, k, v and mixed.
bool edge_supported(int64_t E, int64_t H, TcType t);
pmha_status edge_attention(TcType t, const pmha_graph *g, const EdgeArgs &a, cudaStream_t s);
pmha_status empty_targets(TcType t, const pmha_graph *g, const EdgeArgs &a, cudaStream_t s);

// Y (M x N) = X (M x K, pitch ldx) . W^T (W: N x K, pitch ldw) on the tensor
// cores, one weight matrix, no bias, 16-bit operands of one type; out F16 or
// BF16 (Y pitch ldy), or F32: K split in up to ksplit parts, part i stored at
// Y + i * M * ldy (the caller sums them). K % 64 == 0, N % 128 == 0.
pmha_status gemm_tc_general(TcType in, TcType out, const void *X, int64_t ldx, int64_t M, int64_t K, const void *W,
                            int64_t ldw, int64_t N, void *Y, int64_t ldy, int64_t ksplit, const char *stage,
                            cudaStream_t stream);

// ---------------------------------------------------------------- backward
struct BwdAttnArgs {
    const void *q;         // projected q rows (B, L) of pitch q_ld, intermediate type
    int64_t q_ld;
    const void *k, *v;     // projected k, v rows (B, S) of pitch kv_ld
    int64_t kv_ld;
    const void *dmixed;    // (B, L, E) intermediate type
    const float *ml;       // (B, L, H, 2) forward softmax statistics (log2 units)
    const float *D;        // (B, L, H) dot(dmixed, mixed) per head
    const float2 *rec;     // (B, L, H) {m + log2(l), D}, or null (then no ring kernels)
    unsigned *ctr;         // two task counters for the ring kernels
    const uint8_t *kpm;    // (B, S) or null
    float *dq, *dk, *dv;   // (B, L, E), (B, S, E), (B, S, E), scaled
    float *part_dq;        // (B, 2 n_units, E) partial sums of rows crossing a unit
    float *part_dkv;       // (B, 2 n_units, 2E)
    int64_t B, E, H;
};
// The per-edge backward kernels on the ring design (bwd_ring.cu): fp16
// intermediates, embed_dim 128, 256 or 512, heads of a multiple of 16
// channels. One launch walks one view: dq over the per-target view (rows =
// targets, idx = sources) or dk, dv over the per-source view.
struct BwdRingArgs {
    const void *q;          // projected q rows (B, L) of pitch q_ld, fp16
    long long q_ld;
    const void *k, *v;      // projected k, v rows (B, S) of pitch kv_ld, fp16
    long long kv_ld;
    const void *g;          // dmixed (B, L, E), fp16
    const float2 *rec;      // (B, L, H): c = m + log2(l) (log2 units; +inf when l = 0), D
    const uint8_t *kpm;     // (B, S) or null
    const int32_t *row_ptr, *idx, *unit_first;  // the walked view
    const int32_t *unit_order;                  // the order of its units in the queue, or null (index order)
    long long n_units, nnz;
    int B, L, S, E, H, n_rows;                  // n_rows: L (dq) or S (dk, dv)
    float score_scale;      // log2(e) / sqrt(d)
    float inv_sqrt_d;
    float *out0, *out1;     // dq | dk, dv rows (B, n_rows, E), fp32
    float *part;            // (B, 2 n_units, W) partial sums of rows crossing a unit (W = E, or 2E for dk|dv)
    unsigned *task_counter; // zero before the launch
};
bool bwd_ring_supported(int64_t E, int64_t H);
pmha_status launch_bwd_ring(bool dkv, const BwdRingArgs &a, cudaStream_t s);
// Lane shape of the per-edge backward kernels for intermediate type t
// (channels per lane, lanes per sample; false: no kernel).
bool bwd_shape(int64_t E, int64_t H, int *cpl, int *lpe, TcType t);
// D (rows, H) = dmixed . mixed per head; with rec non-null also the records
// {m + log2(l) (+inf when l = 0), D} from ml (rows, H, 2).
pmha_status bwd_rowdot(TcType t, const void *dmixed, const void *mixed, int64_t rows, int64_t E, int64_t H, float *D,
                       const float *ml, float2 *rec, cudaStream_t s);
// Steps 2-4 backward: dq over the per-target view, dk and dv over the per-source view.
pmha_status bwd_attention(TcType t, const pmha_graph *g, const BwdAttnArgs &x, cudaStream_t s);
// C (M x N) (+)= A (M x K) . B (K x N) on CUDA cores, fp32 accumulation.
pmha_status bwd_gemm_nn(TcType ta, TcType tb, TcType tc, const void *A, int64_t lda, const void *B, int64_t ldb,
                        void *C, int64_t ldc, int64_t M, int64_t N, int64_t K, bool accumulate, cudaStream_t s);
// dW (K x N) = A^T B over M rows and/or db (K) = column sums of A; deterministic chunked sums.
pmha_status bwd_gemm_tn(TcType ta, TcType tb, const void *A, int64_t lda, const void *B, int64_t ldb, int64_t M,
                        int64_t K, int64_t N, float *dW, float *db, float *scratch, int64_t chunks, cudaStream_t s);
pmha_status bwd_convert(const float *in, int64_t n, TcType out_t, void *out, cudaStream_t s);
// Steps 5 and 1 of the backward pass: dmixed, out_proj's and the
// projections' weight and bias gradients, the input gradients. Tensor cores
// for bf16 layers with embed_dim % 128 == 0, else CUDA cores.
struct BwdGemmArgs {
    TcType pt, it;              // layer (parameter) type, intermediate type
    int64_t B, L, S, E;
    const void *dout, *mixed;   // (B, L, E) layer type, intermediate type
    const void *w[4];           // wq, wk, wv, wo (E, E) layer type
    const void *in[3];          // query, key, value (layer type)
    const float *dy[3];         // dq, dk, dv (fp32)
    void *gx[3];                // input gradients (layer type) or null; shared for shared inputs
    float *gw[4], *gb[4];       // parameter gradients (q, k, v, o) or null
    void *dmixed;               // out: (B, L, E) intermediate type
    float *dx32;                // (max(B L, B S), E) fp32 accumulator (CUDA-core path)
    void *scratch;              // bwd_gemm_scratch_bytes()
    int64_t chunks;             // row chunks of the CUDA-core column sums
};
size_t bwd_gemm_scratch_bytes(int64_t B, int64_t L, int64_t S, int64_t E, TcType pt);
pmha_status bwd_step5(const BwdGemmArgs &g, cudaStream_t s);
pmha_status bwd_step1(const BwdGemmArgs &g, cudaStream_t s);

// ---------------------------------------------------------------- dense graphs
struct DenseInputs {
    const void *q;   // (B, L) fp16 rows of pitch q_ld, head h at columns h*d..
    int64_t q_ld;
    const void *k;   // (B, S) fp16 rows of pitch k_ld
    int64_t k_ld;
    const void *v;   // (B, S) fp16 rows of pitch v_ld
    int64_t v_ld;
    void *vt;        // workspace: E x (B * S) fp16, V transposed
    void *mixed;     // (B, L, E) fp16 output of the mix
    const uint8_t *kpm;  // (B, S) key_padding_mask or null
    int64_t B, E, H;
};
// The tensor-core path for dense graphs applies: the graph was built dense,
// fp16 intermediates, head_dim 64 or 128.
bool dense_supported(const pmha_graph *g, int64_t E, int64_t H, TcType t);
size_t dense_vt_bytes(const pmha_graph *g, int64_t B, int64_t E);
// Steps 2-4 for every target of a dense graph: V transposed, then the
// masked-dense tile kernel writes `mixed`.
pmha_status dense_attention(const pmha_graph *g, const DenseInputs &in, cudaStream_t s);
// ---------------------------------------------------------------- heavy targets
struct HeavyInputs {
    const void *q;        // projected q rows (B, L) fp16 of pitch q_ld
    int64_t q_ld;
    const void *x;        // key tokens (B, S, E) bf16: the key and value input (one tensor)
    const void *wk, *wv;  // (E, E) bf16
    const void *bv;       // (E) bf16 or null
    void *mixed;          // (B, L, E) fp16: the heavy targets' rows are written
    void *workspace;      // heavy_workspace_bytes(g, B), 256-byte aligned
    int64_t B, H;
};
// The tensor-core path for heavy targets applies: the graph was split, fp16
// intermediates, embed_dim 128, at most 8 heads.
bool heavy_supported(const pmha_graph *g, int64_t E, int64_t H, TcType t);
size_t heavy_workspace_bytes(const pmha_graph *g, int64_t B);
// Steps 2-4 for the heavy targets of g (writes their mixed rows).
pmha_status heavy_attention(const pmha_graph *g, const HeavyInputs &in, cudaStream_t s);
// Splits a built graph: targets with at least min_deg edges become heavy,
// the rest form g->light. No split when min_deg <= 0, the graph is dense,
// or either side would be empty. Synchronizes the stream.
pmha_status split_heavy(pmha_graph *g, int64_t min_deg, cudaStream_t stream);
void destroy_graph(pmha_graph *g);

// weights[b, e(, h)] from raw scores and (m, l); in place when out == scores.
pmha_status weights_finalize(const pmha_graph *g, const EdgeArgs &a, pmha_wmode mode, float *out,
                             cudaStream_t s);

}  // namespace pmha
