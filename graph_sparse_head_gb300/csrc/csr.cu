// One-time build of the per-target edge view (CSR by target) and of the
// edge kernel's work plan.
//
// The kpnn2 PackedMultiheadAttention page (constructor parameters and Raises
// table) fixes what is accepted: indices in range, length >= 1, no repeated
// (source, target) pair, and add_self_loops appending every missing (i, i)
// after the given pairs. The pages never group edges by target (they gather
// per edge); this view exists so the attention kernel can run a segmented
// softmax per target without atomics. Positions of one target are ordered by
// source, which makes the view unique for a given edge set.
//
// Steps, all on the device of the calling thread:
//   keys      key = target * S + source, value = edge id; range check
//   loops     flags of present (i, i); exclusive scan; append missing loops
//   sort      LSD radix sort, 8-bit digits, stable scatter per tile
//   checks    adjacent equal keys -> duplicate
//   view      row_ptr by binary search; col, perm, target of each edge id
//   plan      first target of every unit of kUnitEdges positions; list of
//             targets crossing a unit boundary (their pieces are merged by
//             the edge kernel) or without edges, with their positions in it
// followed by a single device-to-host copy of a summary and one synchronize.
#include <algorithm>
#include <vector>

#include "pmha_internal.h"

namespace pmha {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortItems = 16;                       // per lane
constexpr int kSortTile = kSortThreads * kSortItems;  // 4096 keys per block
constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;

enum : int { kFlagRange = 1, kFlagDuplicate = 2 };

struct Summary {
    int flags;
    int nnz_total;
    int n_merge;
    int max_deg;
    int n_empty;  // rows without edges
};

__device__ __forceinline__ int warp_inclusive_sum(int v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

// Exclusive scan of one value per thread across a block of kScanThreads
// threads; returns the exclusive prefix and writes the block total.
__device__ __forceinline__ int block_exclusive_sum(int v, int *smem_warp, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = warp_inclusive_sum(v);
    if (lane == 31) smem_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kScanThreads / 32 ? smem_warp[lane] : 0;
        int wi = warp_inclusive_sum(w);
        if (lane < kScanThreads / 32) smem_warp[lane] = wi - w;
        if (lane == kScanThreads / 32 - 1) smem_warp[kScanThreads / 32] = wi;
    }
    __syncthreads();
    int r = smem_warp[warp] + inc - v;
    *total = smem_warp[kScanThreads / 32];
    __syncthreads();
    return r;
}

__global__ void k_scan_reduce(const int *__restrict__ in, int n, int *__restrict__ block_sums)
{
    __shared__ int sw[kScanThreads / 32 + 1];
    const int base = blockIdx.x * kScanTile + threadIdx.x * kScanItems;
    int s = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i)
        if (base + i < n) s += in[base + i];
    int total;
    block_exclusive_sum(s, sw, &total);
    if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

// Single block: exclusive scan of the block sums in place; total to *total.
__global__ void k_scan_blocks(int *__restrict__ sums, int n, int *__restrict__ total)
{
    __shared__ int sw[kScanThreads / 32 + 1];
    int carry = 0;
    for (int base = 0; base < n; base += kScanTile) {
        const int b = base + threadIdx.x * kScanItems;
        int v[kScanItems];
        int s = 0;
#pragma unroll
        for (int i = 0; i < kScanItems; ++i) {
            v[i] = (b + i < n) ? sums[b + i] : 0;
            s += v[i];
        }
        int chunk_total;
        int pre = block_exclusive_sum(s, sw, &chunk_total) + carry;
#pragma unroll
        for (int i = 0; i < kScanItems; ++i) {
            if (b + i < n) sums[b + i] = pre;
            pre += v[i];
        }
        carry += chunk_total;
    }
    if (threadIdx.x == 0 && total) *total = carry;
}

__global__ void k_scan_apply(const int *__restrict__ in, int n, const int *__restrict__ block_off,
                             int *__restrict__ out)
{
    __shared__ int sw[kScanThreads / 32 + 1];
    const int base = blockIdx.x * kScanTile + threadIdx.x * kScanItems;
    int v[kScanItems];
    int s = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
        v[i] = (base + i < n) ? in[base + i] : 0;
        s += v[i];
    }
    int total;
    int pre = block_exclusive_sum(s, sw, &total) + block_off[blockIdx.x];
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
        if (base + i < n) out[base + i] = pre;
        pre += v[i];
    }
}

// Exclusive scan; `in` may equal `out`. `tmp` holds ceil(n / kScanTile) ints.
// `total` (device, nullable) receives the sum.
void exclusive_scan(const int *in, int *out, int n, int *total, int *tmp, cudaStream_t s)
{
    const int nb = std::max(1, (n + kScanTile - 1) / kScanTile);
    k_scan_reduce<<<nb, kScanThreads, 0, s>>>(in, n, tmp);
    k_scan_blocks<<<1, kScanThreads, 0, s>>>(tmp, nb, total);
    k_scan_apply<<<nb, kScanThreads, 0, s>>>(in, n, tmp, out);
    count_launch(3);
}

// ------------------------------------------------------------ radix sort

template <typename K>
__global__ void k_radix_hist(const K *__restrict__ keys, int n, int shift, int n_tiles,
                             int *__restrict__ hist)
{
    __shared__ int h[kRadix];
    for (int i = threadIdx.x; i < kRadix; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const int base = blockIdx.x * kSortTile;
    for (int i = threadIdx.x; i < kSortTile; i += blockDim.x) {
        const int idx = base + i;
        if (idx < n) atomicAdd(&h[(int)((keys[idx] >> shift) & (kRadix - 1))], 1);
    }
    __syncthreads();
    for (int d = threadIdx.x; d < kRadix; d += blockDim.x) hist[d * n_tiles + blockIdx.x] = h[d];
}

// Stable scatter of one tile. Warp w owns the tile's keys
// [w * 32 * kSortItems, (w + 1) * 32 * kSortItems) and walks them in rounds of
// 32 consecutive keys, so (warp, round, lane) is the input order. Within a
// round, lanes with the same digit find each other with match.any and rank by
// lane; a per-warp count per digit carries the rank across rounds. Warps are
// then offset by an exclusive scan of the per-warp counts, and the tile by the
// global digit-major scan of the histograms.
template <typename K>
__global__ void __launch_bounds__(kSortThreads)
k_radix_scatter(const K *__restrict__ keys_in, const int *__restrict__ vals_in, int n, int shift,
                int n_tiles, const int *__restrict__ offsets, K *__restrict__ keys_out,
                int *__restrict__ vals_out)
{
    __shared__ int cnt[kSortWarps][kRadix];
    __shared__ int tile_base[kRadix];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = lane; i < kRadix; i += 32) cnt[warp][i] = 0;
    __syncwarp();
    const unsigned lt_mask = (1u << lane) - 1u;
    const int base = blockIdx.x * kSortTile + warp * 32 * kSortItems;
    K key[kSortItems];
    int val[kSortItems];
    int rank[kSortItems];
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
        const int idx = base + r * 32 + lane;
        const bool valid = idx < n;
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        rank[r] = 0;
        if (valid) {
            key[r] = keys_in[idx];
            val[r] = vals_in[idx];
            const int d = (int)((key[r] >> shift) & (kRadix - 1));
            const unsigned peers = __match_any_sync(vmask, d);
            const int leader = __ffs(peers) - 1;
            const int before = cnt[warp][d];
            rank[r] = before + __popc(peers & lt_mask);
            __syncwarp(vmask);
            if (lane == leader) cnt[warp][d] = before + __popc(peers);
        }
        __syncwarp();
    }
    __syncthreads();
    for (int d = threadIdx.x; d < kRadix; d += blockDim.x) {
        int acc = 0;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) {
            const int c = cnt[w][d];
            cnt[w][d] = acc;
            acc += c;
        }
        tile_base[d] = offsets[d * n_tiles + blockIdx.x];
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kSortItems; ++r) {
        const int idx = base + r * 32 + lane;
        if (idx < n) {
            const int d = (int)((key[r] >> shift) & (kRadix - 1));
            const int pos = tile_base[d] + cnt[warp][d] + rank[r];
            keys_out[pos] = key[r];
            vals_out[pos] = val[r];
        }
    }
}

// Sorts (keys, vals) by the low `bits` bits of the keys. Returns pointers to
// the sorted arrays (one of the two buffers).
template <typename K>
void radix_sort(K *keys_a, int *vals_a, K *keys_b, int *vals_b, int n, int bits, int *hist,
                int *scan_tmp, cudaStream_t s, K **keys_sorted, int **vals_sorted)
{
    const int n_tiles = std::max(1, (n + kSortTile - 1) / kSortTile);
    K *ki = keys_a, *ko = keys_b;
    int *vi = vals_a, *vo = vals_b;
    for (int shift = 0; shift < bits; shift += kRadixBits) {
        k_radix_hist<K><<<n_tiles, kSortThreads, 0, s>>>(ki, n, shift, n_tiles, hist);
        count_launch();
        exclusive_scan(hist, hist, kRadix * n_tiles, nullptr, scan_tmp, s);
        k_radix_scatter<K><<<n_tiles, kSortThreads, 0, s>>>(ki, vi, n, shift, n_tiles, hist, ko, vo);
        count_launch();
        std::swap(ki, ko);
        std::swap(vi, vo);
    }
    *keys_sorted = ki;
    *vals_sorted = vi;
}

// ------------------------------------------------------------ build kernels

template <typename K>
__global__ void k_make_keys(const int64_t *__restrict__ src, const int64_t *__restrict__ tgt,
                            int nnz, int64_t L, int64_t S, bool self_loops, K *__restrict__ keys,
                            int *__restrict__ vals, int *__restrict__ has_loop,
                            Summary *__restrict__ sum)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= nnz) return;
    const int64_t s = src[e], t = tgt[e];
    const bool ok = s >= 0 && s < S && t >= 0 && t < L;
    if (!ok) atomicOr(&sum->flags, kFlagRange);
    keys[e] = ok ? (K)(t * S + s) : (K)0;
    vals[e] = e;
    if (self_loops && ok && s == t) has_loop[t] = 1;
}

__global__ void k_missing_loops(const int *__restrict__ has_loop, int n, int *__restrict__ miss)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) miss[i] = has_loop[i] ? 0 : 1;
}

template <typename K>
__global__ void k_fill(K *__restrict__ keys, int *__restrict__ vals, int from, int to, K value)
{
    const int i = from + blockIdx.x * blockDim.x + threadIdx.x;
    if (i < to) {
        keys[i] = value;
        vals[i] = -1;
    }
}

template <typename K>
__global__ void k_append_loops(const int *__restrict__ has_loop, const int *__restrict__ pos, int n,
                               int nnz, int64_t S, K *__restrict__ keys, int *__restrict__ vals)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n && !has_loop[i]) {
        keys[nnz + pos[i]] = (K)((int64_t)i * S + i);
        vals[nnz + pos[i]] = nnz + pos[i];
    }
}

__global__ void k_set_total(Summary *sum, int nnz, const int *missing_total)
{
    sum->nnz_total = nnz + (missing_total ? *missing_total : 0);
}

template <typename K>
__global__ void k_check_and_view(const K *__restrict__ keys, const int *__restrict__ vals,
                                 int64_t S, Summary *__restrict__ sum, int32_t *__restrict__ col,
                                 int32_t *__restrict__ perm, int32_t *__restrict__ tgt_of_edge,
                                 int32_t *__restrict__ tgt_of_pos)
{
    const int n = sum->nnz_total;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const K k = keys[i];
    if (i > 0 && keys[i - 1] == k) atomicOr(&sum->flags, kFlagDuplicate);
    const int64_t t = (int64_t)(k / (K)S);
    col[i] = (int32_t)((int64_t)k - t * S);
    perm[i] = vals[i];
    tgt_of_edge[vals[i]] = (int32_t)t;
    tgt_of_pos[i] = (int32_t)t;
}

// Adjacency bits of a dense graph: block t sets bit s of row t for every
// source s of target t.
__global__ void k_adj_bits(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col, int64_t words,
                           uint32_t *__restrict__ adj)
{
    const int t = blockIdx.x;
    const int beg = row_ptr[t], end = row_ptr[t + 1];
    uint32_t *row = adj + (int64_t)t * words;
    for (int p = beg + (int)threadIdx.x; p < end; p += blockDim.x) {
        const int s = col[p];
        atomicOr(&row[s >> 5], 1u << (s & 31));
    }
}

template <typename K>
__global__ void k_row_ptr(const K *__restrict__ keys, const Summary *__restrict__ sum, int64_t L,
                          int64_t S, int32_t *__restrict__ row_ptr)
{
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t > L) return;
    const K target_key = (K)(t * S);
    int lo = 0, hi = sum->nnz_total;  // first position with key >= target_key
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (keys[mid] < target_key) lo = mid + 1;
        else hi = mid;
    }
    row_ptr[t] = lo;
}

// Target of the first position of every unit: the largest t with
// row_ptr[t] <= u * kUnitEdges (it has an edge there, since positions are < nnz).
__global__ void k_unit_first(const int32_t *__restrict__ row_ptr, int L, const Summary *__restrict__ sum,
                             int32_t *__restrict__ unit_first_t)
{
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    const int n_units = (sum->nnz_total + kUnitEdges - 1) / kUnitEdges;
    if (u >= n_units) return;
    const int pos = u * kUnitEdges;
    int lo = 0, hi = L;  // invariant: row_ptr[lo] <= pos < row_ptr[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (row_ptr[mid] <= pos) lo = mid;
        else hi = mid;
    }
    unit_first_t[u] = lo;
}

// Work estimate of every unit (its positions plus kSwitchCost per target it
// touches: a target switch costs the edge kernel about that many edges), as
// a 16-bit key that sorts the slowest unit first; padding units past the
// real count get the largest key. vals receive the unit indices.
#ifndef PMHA_SWITCH_COST
#define PMHA_SWITCH_COST 4
#endif
constexpr int kSwitchCost = PMHA_SWITCH_COST;
__global__ void k_unit_cost(const int32_t *__restrict__ row_ptr, int L, const Summary *__restrict__ sum,
                            const int32_t *__restrict__ unit_first_t, int max_units, uint32_t *__restrict__ key,
                            int *__restrict__ val)
{
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= max_units) return;
    const int nnz = sum->nnz_total;
    const int n_units = (nnz + kUnitEdges - 1) / kUnitEdges;
    val[u] = u;
    if (u >= n_units) {
        key[u] = 0xffffu;
        return;
    }
    const int e0 = u * kUnitEdges, e1 = min(e0 + kUnitEdges, nnz);
    int lo = 0, hi = L;  // target of position e1 - 1: row_ptr[lo] <= e1 - 1 < row_ptr[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (row_ptr[mid] <= e1 - 1) lo = mid;
        else hi = mid;
    }
    const int cost = (e1 - e0) + kSwitchCost * (lo - unit_first_t[u] + 1);
    key[u] = 0xfffeu - (uint32_t)min(cost, 0xfffe);
}

__global__ void k_merge_flags(const int32_t *__restrict__ row_ptr, int L, int *__restrict__ flag,
                              Summary *__restrict__ sum)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= L) return;
    const int b = row_ptr[t], e = row_ptr[t + 1], deg = e - b;
    flag[t] = (deg == 0 || b / kUnitEdges != (e - 1) / kUnitEdges) ? 1 : 0;
    atomicMax(&sum->max_deg, deg);
    if (deg == 0) atomicAdd(&sum->n_empty, 1);
}

__global__ void k_merge_write(const int *__restrict__ flag, const int *__restrict__ off, int L,
                              int32_t *__restrict__ merge_t)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < L && flag[t]) merge_t[off[t]] = t;
}

// Index of each target in the merge list (-1 when it is not there).
__global__ void k_merge_pos(const int *__restrict__ flag, const int *__restrict__ off, int L,
                            int32_t *__restrict__ merge_pos)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < L) merge_pos[t] = flag[t] ? off[t] : -1;
}

// Keys of the by-source view: for CSR position p (target t, source s),
// key = s * L + t; positions past nnz_total get the sentinel (sorted last).
template <typename K>
__global__ void k_csc_keys(const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col, int64_t L,
                           const Summary *__restrict__ sum, int cap, K sentinel, K *__restrict__ keys,
                           int *__restrict__ vals)
{
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= cap) return;
    vals[p] = p;
    if (p >= sum->nnz_total) {
        keys[p] = sentinel;
        return;
    }
    int lo = 0, hi = (int)L;  // row_ptr[lo] <= p < row_ptr[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (row_ptr[mid] <= p) lo = mid;
        else hi = mid;
    }
    keys[p] = (K)col[p] * (K)L + (K)lo;
}

// Target of each by-source position.
template <typename K>
__global__ void k_csc_view(const K *__restrict__ keys, const Summary *__restrict__ sum, int64_t L,
                           int32_t *__restrict__ tgt_by_src)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= sum->nnz_total) return;
    tgt_by_src[i] = (int32_t)((int64_t)(keys[i] % (K)L));
}

__global__ void k_copy_total(const Summary *__restrict__ from, Summary *__restrict__ to)
{
    to->nnz_total = from->nnz_total;
}

inline int blocks_for(int64_t n, int threads) { return (int)std::max<int64_t>(1, (n + threads - 1) / threads); }

template <typename K>
pmha_status build_typed(const int64_t *src, const int64_t *tgt, int64_t nnz64, int64_t L, int64_t S,
                        bool self_loops, cudaStream_t stream, pmha_graph **out)
{
    const int nnz = (int)nnz64;
    const int cap = (int)(nnz64 + (self_loops ? L : 0));
    const int max_units = cap / kUnitEdges + 1;
    int bits = 0;
    {
        const unsigned long long ls = (unsigned long long)L * (unsigned long long)S;
        while (bits < 64 && (ls >> bits) != 0ull) ++bits;
        bits = std::max(bits, 1);
    }
    const K sentinel = (bits >= (int)(8 * sizeof(K))) ? (K)~(K)0 : (K)(((K)1 << bits) - 1);

    pmha_graph *g = new pmha_graph();
    g->L = L;
    g->S = S;
    g->nnz_given = nnz64;
    cudaGetDevice(&g->device);

    // graph allocation
    auto align = [](size_t x) { return (x + 255) & ~(size_t)255; };
    size_t off_row = 0;
    size_t off_col = off_row + align((size_t)(L + 1) * 4);
    size_t off_perm = off_col + align((size_t)cap * 4);
    size_t off_tge = off_perm + align((size_t)cap * 4);
    size_t off_inv = off_tge + align((size_t)cap * 4);
    size_t off_units = off_inv + align((size_t)cap * 4);
    size_t off_order = off_units + align((size_t)max_units * 4);
    size_t off_merge = off_order + align((size_t)max_units * 4);
    size_t off_mpos = off_merge + align((size_t)L * 4);
    size_t off_srp = off_mpos + align((size_t)L * 4);
    size_t off_tbs = off_srp + align((size_t)(S + 1) * 4);
    size_t off_ufs = off_tbs + align((size_t)cap * 4);
    size_t off_ms = off_ufs + align((size_t)max_units * 4);
    size_t graph_bytes = off_ms + align((size_t)S * 4);

    // temporaries
    const int n_tiles = std::max(1, (cap + kSortTile - 1) / kSortTile);
    const int64_t LS1 = std::max(L, S) + 1;  // room for the per-target and the per-source passes
    const int64_t scan_max = std::max<int64_t>({(int64_t)kRadix * n_tiles, LS1, 1});
    size_t t_keys_a = 0;
    size_t t_keys_b = t_keys_a + align((size_t)cap * sizeof(K));
    size_t t_vals_a = t_keys_b + align((size_t)cap * sizeof(K));
    size_t t_vals_b = t_vals_a + align((size_t)cap * 4);
    size_t t_hist = t_vals_b + align((size_t)cap * 4);
    size_t t_scan = t_hist + align((size_t)kRadix * n_tiles * 4);
    size_t t_loop = t_scan + align((size_t)(scan_max / kScanTile + 2) * 4);
    size_t t_miss = t_loop + align((size_t)(L + 1) * 4);
    size_t t_c1 = t_miss + align((size_t)LS1 * 4);
    size_t t_c2 = t_c1 + align((size_t)LS1 * 4);
    size_t t_c3 = t_c2 + align((size_t)LS1 * 4);
    size_t t_tot = t_c3 + align((size_t)LS1 * 4);
    size_t t_sum = t_tot + align(4 * sizeof(int));
    size_t tmp_bytes = t_sum + align(2 * sizeof(Summary));

    char *gm = nullptr, *tm = nullptr;
    Summary *host_sum = nullptr;
    pmha_status st = PMHA_OK;
    cudaError_t ce;
    if ((ce = cudaMalloc(&gm, graph_bytes)) != cudaSuccess) { delete g; return cuda_fail(ce, "cudaMalloc(graph)"); }
    if ((ce = cudaMalloc(&tm, tmp_bytes)) != cudaSuccess) {
        cudaFree(gm);
        delete g;
        return cuda_fail(ce, "cudaMalloc(build temporaries)");
    }
    if ((ce = cudaMallocHost(&host_sum, 2 * sizeof(Summary))) != cudaSuccess) {
        cudaFree(gm);
        cudaFree(tm);
        delete g;
        return cuda_fail(ce, "cudaMallocHost(summary)");
    }
    g->mem = gm;
    g->row_ptr = (int32_t *)(gm + off_row);
    g->col = (int32_t *)(gm + off_col);
    g->perm = (int32_t *)(gm + off_perm);
    g->tgt_of_edge = (int32_t *)(gm + off_tge);
    g->tgt_of_pos = (int32_t *)(gm + off_inv);
    g->unit_first_t = (int32_t *)(gm + off_units);
    g->unit_order = (int32_t *)(gm + off_order);
    g->merge_t = (int32_t *)(gm + off_merge);
    g->merge_pos = (int32_t *)(gm + off_mpos);
    g->src_row_ptr = (int32_t *)(gm + off_srp);
    g->tgt_by_src = (int32_t *)(gm + off_tbs);
    g->unit_first_s = (int32_t *)(gm + off_ufs);
    g->merge_s = (int32_t *)(gm + off_ms);

    K *keys_a = (K *)(tm + t_keys_a), *keys_b = (K *)(tm + t_keys_b);
    int *vals_a = (int *)(tm + t_vals_a), *vals_b = (int *)(tm + t_vals_b);
    int *hist = (int *)(tm + t_hist), *scan_tmp = (int *)(tm + t_scan);
    int *has_loop = (int *)(tm + t_loop), *miss = (int *)(tm + t_miss);
    int *c1 = (int *)(tm + t_c1), *c2 = (int *)(tm + t_c2);
    int *tot = (int *)(tm + t_tot);
    Summary *dsum = (Summary *)(tm + t_sum);
    Summary *dsum_src = dsum + 1;  // the by-source pass

    const int TB = 256;
    do {
        if ((ce = cudaMemsetAsync(dsum, 0, sizeof(Summary), stream)) != cudaSuccess) break;
        if ((ce = cudaMemsetAsync(has_loop, 0, (size_t)(L + 1) * 4, stream)) != cudaSuccess) break;
        k_make_keys<K><<<blocks_for(nnz, TB), TB, 0, stream>>>(src, tgt, nnz, L, S, self_loops, keys_a,
                                                               vals_a, has_loop, dsum);
        count_launch();
        if (self_loops) {
            k_fill<K><<<blocks_for(cap - nnz, TB), TB, 0, stream>>>(keys_a, vals_a, nnz, cap, sentinel);
            k_missing_loops<<<blocks_for(L, TB), TB, 0, stream>>>(has_loop, (int)L, miss);
            count_launch(2);
            exclusive_scan(miss, miss, (int)L, &tot[0], scan_tmp, stream);
            k_append_loops<K><<<blocks_for(L, TB), TB, 0, stream>>>(has_loop, miss, (int)L, nnz, S, keys_a,
                                                                    vals_a);
            k_set_total<<<1, 1, 0, stream>>>(dsum, nnz, &tot[0]);
            count_launch(2);
        } else {
            k_set_total<<<1, 1, 0, stream>>>(dsum, nnz, nullptr);
            count_launch();
        }
        K *keys_s;
        int *vals_s;
        radix_sort<K>(keys_a, vals_a, keys_b, vals_b, cap, bits, hist, scan_tmp, stream, &keys_s, &vals_s);
        k_check_and_view<K><<<blocks_for(cap, TB), TB, 0, stream>>>(keys_s, vals_s, S, dsum, g->col, g->perm,
                                                                    g->tgt_of_edge, g->tgt_of_pos);
        k_row_ptr<K><<<blocks_for(L + 1, TB), TB, 0, stream>>>(keys_s, dsum, L, S, g->row_ptr);
        k_unit_first<<<blocks_for(max_units, TB), TB, 0, stream>>>(g->row_ptr, (int)L, dsum, g->unit_first_t);
        k_merge_flags<<<blocks_for(L, TB), TB, 0, stream>>>(g->row_ptr, (int)L, c1, dsum);
        count_launch(4);
        {
            // the units by decreasing estimated work, for the edge kernel's queue
            uint32_t *ck_a = (uint32_t *)keys_a, *ck_b = (uint32_t *)keys_b;
            k_unit_cost<<<blocks_for(max_units, TB), TB, 0, stream>>>(g->row_ptr, (int)L, dsum, g->unit_first_t,
                                                                      max_units, ck_a, vals_a);
            count_launch();
            uint32_t *ck_s;
            int *cv_s;
            radix_sort<uint32_t>(ck_a, vals_a, ck_b, vals_b, max_units, 16, hist, scan_tmp, stream, &ck_s, &cv_s);
            if ((ce = cudaMemcpyAsync(g->unit_order, cv_s, (size_t)max_units * 4, cudaMemcpyDeviceToDevice,
                                      stream)) != cudaSuccess)
                break;
        }
        exclusive_scan(c1, c2, (int)L, &dsum->n_merge, scan_tmp, stream);
        k_merge_write<<<blocks_for(L, TB), TB, 0, stream>>>(c1, c2, (int)L, g->merge_t);
        k_merge_pos<<<blocks_for(L, TB), TB, 0, stream>>>(c1, c2, (int)L, g->merge_pos);
        count_launch(2);
        if ((ce = cudaGetLastError()) != cudaSuccess) break;
        // the by-source view (for the backward pass): sort (source, target) keys
        if ((ce = cudaMemsetAsync(dsum_src, 0, sizeof(Summary), stream)) != cudaSuccess) break;
        k_copy_total<<<1, 1, 0, stream>>>(dsum, dsum_src);
        k_csc_keys<K><<<blocks_for(cap, TB), TB, 0, stream>>>(g->row_ptr, g->col, L, dsum, cap, sentinel, keys_a,
                                                              vals_a);
        count_launch(2);
        {
            K *keys_s2;
            int *vals_s2;
            radix_sort<K>(keys_a, vals_a, keys_b, vals_b, cap, bits, hist, scan_tmp, stream, &keys_s2, &vals_s2);
            k_csc_view<K><<<blocks_for(cap, TB), TB, 0, stream>>>(keys_s2, dsum, L, g->tgt_by_src);
            k_row_ptr<K><<<blocks_for(S + 1, TB), TB, 0, stream>>>(keys_s2, dsum, S, L, g->src_row_ptr);
            k_unit_first<<<blocks_for(max_units, TB), TB, 0, stream>>>(g->src_row_ptr, (int)S, dsum,
                                                                       g->unit_first_s);
            k_merge_flags<<<blocks_for(S, TB), TB, 0, stream>>>(g->src_row_ptr, (int)S, c1, dsum_src);
            count_launch(4);
            exclusive_scan(c1, c2, (int)S, &dsum_src->n_merge, scan_tmp, stream);
            k_merge_write<<<blocks_for(S, TB), TB, 0, stream>>>(c1, c2, (int)S, g->merge_s);
            count_launch();
        }
        if ((ce = cudaGetLastError()) != cudaSuccess) break;
        if ((ce = cudaMemcpyAsync(host_sum, dsum, 2 * sizeof(Summary), cudaMemcpyDeviceToHost, stream)) !=
            cudaSuccess)
            break;
        ce = cudaStreamSynchronize(stream);
    } while (0);

    if (ce != cudaSuccess) {
        st = cuda_fail(ce, "CSR build");
    } else if (host_sum->flags & kFlagRange) {
        set_error("pmha_build_csr: an index lies outside [0, key_features) or [0, query_features)");
        st = PMHA_ERR_INDEX_RANGE;
    } else if (host_sum->flags & kFlagDuplicate) {
        set_error("pmha_build_csr: a (source, target) pair is given more than once");
        st = PMHA_ERR_DUPLICATE_EDGE;
    }
    if (st == PMHA_OK) {
        g->nnz = host_sum->nnz_total;
        g->max_deg = host_sum->max_deg;
        g->n_units = (g->nnz + kUnitEdges - 1) / kUnitEdges;
        g->n_merge = host_sum->n_merge;
        g->n_empty = host_sum->n_empty;
        g->n_merge_s = host_sum[1].n_merge;
        g->max_out_deg = host_sum[1].max_deg;
        // A graph with at least a quarter of all (target, source) pairs may run
        // the masked-dense tensor-core kernel; it keeps the pairs as bits
        // (none for a complete graph). Without room for the bits the graph
        // simply stays on the per-edge path.
        const double pairs = (double)L * (double)S;
        if ((double)g->nnz * 4.0 >= pairs && pairs <= (double)(1ull << 29)) {
            g->dense_complete = g->nnz == L * S;
            g->dense = true;
            if (!g->dense_complete) {
                g->adj_words_per_row = (S + 31) / 32;
                const size_t bytes = (size_t)L * (size_t)g->adj_words_per_row * 4;
                if (cudaMalloc(&g->adj, bytes) != cudaSuccess) {
                    cudaGetLastError();
                    g->adj = nullptr;
                    g->dense = false;
                } else {
                    do {
                        if ((ce = cudaMemsetAsync(g->adj, 0, bytes, stream)) != cudaSuccess) break;
                        k_adj_bits<<<(unsigned)L, 256, 0, stream>>>(g->row_ptr, g->col, g->adj_words_per_row, g->adj);
                        count_launch();
                        if ((ce = cudaGetLastError()) != cudaSuccess) break;
                        ce = cudaStreamSynchronize(stream);
                    } while (0);
                    if (ce != cudaSuccess) {
                        st = cuda_fail(ce, "CSR build (adjacency bits)");
                        cudaFree(g->adj);
                    }
                }
            }
        }
    }
    cudaFree(tm);
    cudaFreeHost(host_sum);
    if (st != PMHA_OK) {
        cudaFree(gm);
        delete g;
        return st;
    }
    *out = g;
    return PMHA_OK;
}

}  // namespace

pmha_status build_csr(const int64_t *src, const int64_t *tgt, int64_t nnz, int64_t L, int64_t S,
                      bool self_loops, cudaStream_t stream, pmha_graph **out)
{
    const unsigned long long ls = (unsigned long long)L * (unsigned long long)S;
    if (ls < (1ull << 32)) return build_typed<uint32_t>(src, tgt, nnz, L, S, self_loops, stream, out);
    return build_typed<unsigned long long>(src, tgt, nnz, L, S, self_loops, stream, out);
}

void destroy_graph(pmha_graph *g)
{
    if (!g) return;
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != g->device) cudaSetDevice(g->device);
    if (g->light) destroy_graph(g->light);
    if (g->heavy_info) cudaFree(g->heavy_info);
    if (g->mem) cudaFree(g->mem);
    if (g->adj) cudaFree(g->adj);
    if (cur != g->device) cudaSetDevice(cur);
    delete g;
}

// Host-side split (one-time, like the build): the per-target degrees and
// sources come back to the host, the heavy targets are listed by
// non-increasing in-degree, and the light targets' edges are built into a
// graph of their own by the same device pipeline.
pmha_status split_heavy(pmha_graph *g, int64_t min_deg, cudaStream_t stream)
{
    if (min_deg <= 0 || g->dense || g->max_deg < min_deg) return PMHA_OK;
    const int64_t L = g->L, nnz = g->nnz;
    std::vector<int32_t> rp((size_t)L + 1), col((size_t)nnz);
    PMHA_CUDA_TRY(cudaMemcpyAsync(rp.data(), g->row_ptr, (size_t)(L + 1) * 4, cudaMemcpyDeviceToHost, stream));
    PMHA_CUDA_TRY(cudaMemcpyAsync(col.data(), g->col, (size_t)nnz * 4, cudaMemcpyDeviceToHost, stream));
    PMHA_CUDA_TRY(cudaStreamSynchronize(stream));
    std::vector<int32_t> heavy;
    int64_t n_light = 0;
    for (int64_t t = 0; t < L; ++t) {
        const int64_t deg = rp[(size_t)t + 1] - rp[(size_t)t];
        if (deg >= min_deg) heavy.push_back((int32_t)t);
        else n_light += deg;
    }
    if (heavy.empty() || n_light == 0) return PMHA_OK;
    std::stable_sort(heavy.begin(), heavy.end(), [&](int32_t x, int32_t y) {
        return rp[(size_t)x + 1] - rp[(size_t)x] > rp[(size_t)y + 1] - rp[(size_t)y];
    });
    std::vector<int64_t> lsrc, ltgt;
    lsrc.reserve((size_t)n_light);
    ltgt.reserve((size_t)n_light);
    for (int64_t t = 0; t < L; ++t) {
        const int32_t b = rp[(size_t)t], e = rp[(size_t)t + 1];
        if (e - b >= min_deg) continue;
        for (int32_t p = b; p < e; ++p) {
            lsrc.push_back(col[(size_t)p]);
            ltgt.push_back(t);
        }
    }
    std::vector<int4> info(heavy.size());
    for (size_t i = 0; i < heavy.size(); ++i) {
        const int32_t t = heavy[i], b = rp[(size_t)t], deg = rp[(size_t)t + 1] - b;
        info[i] = make_int4(t, b, deg, (deg + 127) / 128);
    }
    int64_t *dl = nullptr;
    int4 *dh = nullptr;
    PMHA_CUDA_TRY(cudaMalloc(&dl, (size_t)n_light * 16));
    cudaError_t ce = cudaMalloc(&dh, heavy.size() * sizeof(int4));
    if (ce != cudaSuccess) {
        cudaFree(dl);
        return cuda_fail(ce, "cudaMalloc(heavy targets)");
    }
    pmha_graph *light = nullptr;
    pmha_status st = PMHA_OK;
    do {
        if ((ce = cudaMemcpyAsync(dl, lsrc.data(), (size_t)n_light * 8, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
            break;
        if ((ce = cudaMemcpyAsync(dl + n_light, ltgt.data(), (size_t)n_light * 8, cudaMemcpyHostToDevice, stream)) !=
            cudaSuccess)
            break;
        if ((ce = cudaMemcpyAsync(dh, info.data(), info.size() * sizeof(int4), cudaMemcpyHostToDevice, stream)) !=
            cudaSuccess)
            break;
        st = build_csr(dl, dl + n_light, n_light, L, g->S, false, stream, &light);  // synchronizes
    } while (0);
    if (ce != cudaSuccess) st = cuda_fail(ce, "heavy-target split");
    cudaFree(dl);
    if (st != PMHA_OK) {
        cudaFree(dh);
        return st;
    }
    g->light = light;
    g->heavy_info = dh;
    g->n_heavy = (int64_t)heavy.size();
    g->heavy_min_deg = min_deg;
    return PMHA_OK;
}

}  // namespace pmha
