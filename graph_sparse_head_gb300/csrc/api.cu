// Host side of the C ABI declared in include/pmha.h: argument checks, the
// workspace layout, and the order of launches for one forward pass
// (kpnn2 PackedMultiheadAttention, Notes steps 1-5):
//   projections (tensor-core GEMM, Q|K|V fused when the tokens are shared)
//   -> edge attention (scores, segmented softmax, value mix)
//   -> merge of split targets -> per-edge weights (if requested)
//   -> out_proj GEMM.
// Everything is queued on the caller's stream; nothing here synchronizes
// except pmha_build_csr (once) and the explicit status / profiling reads.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "pmha_internal.h"

namespace pmha {

// ---------------------------------------------------------------- errors

static thread_local char t_err[512] = "";

void set_error(const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
}

pmha_status cuda_fail(cudaError_t e, const char *what)
{
    set_error("%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
    return PMHA_ERR_CUDA;
}

static __device__ int g_device_error;

int *device_error_word()
{
    static std::mutex mu;
    static int *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
            set_error("cudaGetSymbolAddress(device error word) failed");
            return nullptr;
        }
        addr[dev] = (int *)p;
    }
    return addr[dev];
}

int num_sms()
{
    static std::atomic<int> cached[64];  // zero-initialised (static storage)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (!n) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// ---------------------------------------------------------------- profiling

static std::atomic<long long> g_launches{0};
void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {
struct Record {
    const char *stage;
    cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

StageTimer::StageTimer(const char *stage_, cudaStream_t s) : stage(stage_), stream(s), slot(-1)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return;
    Record r;
    r.stage = stage;
    r.start = take_event();
    r.stop = take_event();
    if (!r.start || !r.stop) {  // keep whichever one was created
        if (r.start) g_event_pool.push_back(r.start);
        if (r.stop) g_event_pool.push_back(r.stop);
        return;
    }
    cudaEventRecord(r.start, stream);
    slot = (int)g_records.size();
    g_records.push_back(r);
}

StageTimer::~StageTimer()
{
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (slot < (int)g_records.size()) cudaEventRecord(g_records[slot].stop, stream);
}

// ---------------------------------------------------------------- helpers

namespace {

size_t elem_size(pmha_dtype dt) { return dt == PMHA_BF16 ? 2 : 4; }
TcType param_type(pmha_dtype dt) { return dt == PMHA_BF16 ? TcType::BF16 : TcType::F32; }
// q, k, v and mixed of a bf16 layer are kept in fp16 (same width, 3 more
// mantissa bits); a float32 layer keeps them in float32.
TcType inter_type(pmha_dtype dt) { return dt == PMHA_BF16 ? TcType::F16 : TcType::F32; }
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

pmha_status check_params(const pmha_graph *g, const pmha_params *p, int64_t batch)
{
    if (!g) {
        set_error("graph is NULL");
        return PMHA_ERR_INVALID_ARG;
    }
    if (!p) {
        set_error("params is NULL");
        return PMHA_ERR_INVALID_ARG;
    }
    if (p->dtype != PMHA_F32 && p->dtype != PMHA_BF16) {
        set_error("dtype %d is neither PMHA_F32 nor PMHA_BF16", (int)p->dtype);
        return PMHA_ERR_INVALID_ARG;
    }
    if (p->embed_dim < 1 || p->num_heads < 1 || p->embed_dim % p->num_heads) {
        set_error("embed_dim %lld must be positive and divisible by num_heads %lld", (long long)p->embed_dim,
                  (long long)p->num_heads);
        return PMHA_ERR_INVALID_ARG;
    }
    if (batch < 1) {
        set_error("batch %lld must be >= 1", (long long)batch);
        return PMHA_ERR_INVALID_ARG;
    }
    const void *w[4] = {p->wq, p->wk, p->wv, p->wo};
    for (int i = 0; i < 4; ++i)
        if (!w[i] || !aligned16(w[i])) {
            set_error("projection weight %d is NULL or not 16-byte aligned", i);
            return PMHA_ERR_INVALID_ARG;
        }
    const void *b[4] = {p->bq, p->bk, p->bv, p->bo};
    for (int i = 0; i < 4; ++i)
        if (b[i] && ((uintptr_t)b[i] % elem_size(p->dtype))) {
            set_error("bias %d is not aligned to its element size", i);
            return PMHA_ERR_INVALID_ARG;
        }
    if (!edge_supported(p->embed_dim, p->num_heads, inter_type(p->dtype))) {
        set_error("no edge kernel for embed_dim %lld, num_heads %lld in this dtype (needs a power-of-two split "
                  "of the row and of each head over at most 32 lanes)",
                  (long long)p->embed_dim, (long long)p->num_heads);
        return PMHA_ERR_UNSUPPORTED;
    }
    if (batch * g->L * p->embed_dim > (int64_t)1 << 46 || batch * g->S * p->embed_dim > (int64_t)1 << 46) {
        set_error("tensor too large");
        return PMHA_ERR_INVALID_ARG;
    }
    return PMHA_OK;
}

struct Layout {
    size_t qkv = 0, mixed = 0, part = 0, ml = 0, scores = 0, wo16 = 0, vt = 0, counters = 0, kpm_bits = 0, heavy = 0,
           total = 0;
};

// In-degree from which a target runs on the tensor-core path (graphs are
// split when they are built): PMHA_HEAVY_MIN_DEGREE, default 0 (no split,
// every target on the per-edge kernel, which is the faster of the two on
// the measured workloads).
int64_t heavy_min_degree()
{
    const char *e = getenv("PMHA_HEAVY_MIN_DEGREE");
    if (e && *e) {
        char *end = nullptr;
        const long long v = strtoll(e, &end, 10);
        if (end && *end == '\0' && v >= 0) return (int64_t)v;
    }
    return 0;
}

// Step 5 inside the edge kernel (where it can run there) when
// PMHA_FUSED_OUT_PROJ=1 (read on every call); by default it runs as its own
// tensor-core GEMM, which is the faster of the two on the measured workloads
// (the edge kernel's warp-level products re-read Wo from shared memory for
// every 16 rows and are bound by that bandwidth).
bool fuse_out_proj()
{
    const char *e = getenv("PMHA_FUSED_OUT_PROJ");
    return e && e[0] == '1' && e[1] == '\0';
}

bool out_proj_on_tensor_cores(const pmha_params *p)
{
    return p->dtype == PMHA_BF16 && gemm_tc_supported(p->embed_dim);
}

// Offsets inside the workspace. qkv holds B*L*E + B*S*(kv_width) intermediate
// elements: Q, then K|V rows (or the fused [Q|K|V] / [Q|K] rows, which take
// the same room); wo16 holds an fp16 copy of out_proj's weight when out_proj
// runs on the tensor cores with fp16 operands.
Layout layout(const pmha_graph *g, const pmha_params *p, int64_t B, pmha_wmode wmode, bool with_values)
{
    const int64_t E = p->embed_dim, H = p->num_heads;
    const size_t es = type_size(inter_type(p->dtype));
    Layout l;
    size_t o = 0;
    l.qkv = o;
    o += align256((size_t)(B * g->L * E + B * g->S * E * (with_values ? 2 : 1)) * es);
    l.mixed = o;
    if (with_values) o += align256((size_t)(B * g->L * E) * es);
    l.part = o;
    o += align256((size_t)(B * 2 * g->n_units * (2 * H + E)) * 4);
    l.ml = o;
    if (wmode != PMHA_WEIGHTS_NONE) o += align256((size_t)(B * g->L * H * 2) * 4);
    l.scores = o;  // raw scores by CSR position; the weights pass puts them in the given order
    if (wmode != PMHA_WEIGHTS_NONE) o += align256((size_t)(B * g->nnz * H) * 4);
    l.wo16 = o;
    if (with_values && out_proj_on_tensor_cores(p)) o += align256((size_t)(E * E) * 2);
    l.vt = o;
    if (with_values && dense_supported(g, E, H, inter_type(p->dtype))) o += align256(dense_vt_bytes(g, B, E));
    l.counters = o;  // the light part of a split graph has its own merge list; then the out_proj block counts
    o += align256((size_t)(kCounterHead + B * std::max(g->n_merge, g->light ? g->light->n_merge : (int64_t)0) +
                           B * out_blocks(g->L)) * 4);
    l.kpm_bits = o;  // a key_padding_mask per CSR position, when one is given
    o += align256((size_t)(B * ((g->nnz + 31) / 32)) * 4);
    l.heavy = o;  // the heavy-target path's qt images and per-head mixes
    if (with_values && wmode == PMHA_WEIGHTS_NONE && p->dtype == PMHA_BF16 &&
        heavy_supported(g, E, H, inter_type(p->dtype)))
        o += align256(heavy_workspace_bytes(g, B));
    l.total = o;
    return l;
}

// Step 1: tokens (layer dtype) -> q / k / v (intermediate type).
pmha_status project(pmha_dtype dt, const void *X, int64_t M, int64_t E, const GemmSegments &seg, void *Y,
                    int64_t ldy, const char *stage, cudaStream_t s)
{
    if (dt == PMHA_BF16 && gemm_tc_supported(E))
        return gemm_tc(TcType::BF16, TcType::F16, X, M, E, seg, Y, ldy, stage, s);
    if (seg.cvt_frag_E) {
        set_error("%s: the fragment-order copy of Wo needs the tensor-core GEMM", stage);
        return PMHA_ERR_UNSUPPORTED;
    }
    if (seg.cvt_n > 0) {
        const pmha_status st = convert_bf16_to_f16(seg.cvt_src, seg.cvt_dst, seg.cvt_n, s);
        if (st != PMHA_OK) return st;
    }
    return gemm_simt(param_type(dt), param_type(dt), inter_type(dt), X, M, E, seg, Y, ldy, stage, s);
}

GemmSegments segs(const void *w0, const void *b0, const void *w1 = nullptr, const void *b1 = nullptr,
                  const void *w2 = nullptr, const void *b2 = nullptr)
{
    GemmSegments s;
    s.w[0] = w0;
    s.b[0] = b0;
    s.w[1] = w1;
    s.b[1] = b1;
    s.w[2] = w2;
    s.b[2] = b2;
    s.n_seg = w2 ? 3 : (w1 ? 2 : 1);
    return s;
}

// Steps 1-4 (and the weights); with_values = false stops after the scores.
// A non-null wo16 receives the fp16 copy of Wo that out_proj on the tensor
// cores needs; the first projection GEMM writes it as a side job. A non-null
// fused_out asks for step 5 inside the edge kernel, into fused_out, where
// that kernel runs and supports it (fused_out_supported); *fused_done tells
// whether it did (then wo16 holds Wo in the fragment order it reads).
pmha_status attend(const pmha_graph *g, const pmha_params *p, const void *query, const void *key,
                   const void *value, const uint8_t *kpm, int64_t B, pmha_wmode wmode, float *weights, char *ws, const Layout &lay,
                   bool with_values, cudaStream_t s, const void **mixed_out, float *ml_keep = nullptr,
                   bool allow_dense = true, EdgeArgs *args_out = nullptr, void *wo16 = nullptr,
                   void *fused_out = nullptr, bool *fused_done = nullptr)
{
    const int64_t E = p->embed_dim, H = p->num_heads, L = g->L, S = g->S;
    const TcType it = inter_type(p->dtype);
    // which kernels run steps 2-4: masked-dense tiles, the heavy/light split, or the edge kernel
    const bool dense_path = allow_dense && with_values && dense_supported(g, E, H, it);
    const bool heavy_path = !dense_path && with_values && wmode == PMHA_WEIGHTS_NONE && !kpm && !ml_keep &&
                            !args_out && key == value && p->dtype == PMHA_BF16 && heavy_supported(g, E, H, it);
    const bool fuse = fused_out && wo16 && with_values && !dense_path && !heavy_path && p->dtype == PMHA_BF16 &&
                      gemm_tc_supported(E) && fused_out_supported(it, E, H);
    if (fused_done) *fused_done = fuse;
    auto with_wo = [&](GemmSegments sg) {
        if (wo16) {
            sg.cvt_src = p->wo;
            sg.cvt_dst = wo16;
            sg.cvt_n = p->embed_dim * p->embed_dim;
            sg.cvt_frag_E = fuse ? E : 0;
        }
        return sg;
    };
    const size_t es = type_size(inter_type(p->dtype));
    char *qkv = ws + lay.qkv;
    EdgeArgs a;
    pmha_status st;
    const bool same_qkv = query == key && (!with_values || key == value) && L == S;
    const int width = with_values ? 3 : 2;
    if (same_qkv) {
        // one GEMM: rows [Q | K | V] (or [Q | K])
        st = with_values ? project(p->dtype, query, B * L, E,
                                   with_wo(segs(p->wq, p->bq, p->wk, p->bk, p->wv, p->bv)), qkv, 3 * E, "proj_qkv", s)
                         : project(p->dtype, query, B * L, E, with_wo(segs(p->wq, p->bq, p->wk, p->bk)), qkv, 2 * E,
                                   "proj_qk", s);
        if (st != PMHA_OK) return st;
        a.q = qkv;
        a.q_ld = width * E;
        a.kv = qkv + E * es;
        a.kv_ld = width * E;
    } else {
        char *kvbuf = qkv + (size_t)(B * L * E) * es;
        const int64_t kv_w = with_values ? 2 * E : E;
        st = project(p->dtype, query, B * L, E, with_wo(segs(p->wq, p->bq)), qkv, E, "proj_q", s);
        if (st != PMHA_OK) return st;
        if (with_values && key == value) {
            st = project(p->dtype, key, B * S, E, segs(p->wk, p->bk, p->wv, p->bv), kvbuf, kv_w, "proj_kv", s);
            if (st != PMHA_OK) return st;
        } else {
            st = project(p->dtype, key, B * S, E, segs(p->wk, p->bk), kvbuf, kv_w, "proj_k", s);
            if (st != PMHA_OK) return st;
            if (with_values) {
                st = project(p->dtype, value, B * S, E, segs(p->wv, p->bv), kvbuf + E * es, kv_w, "proj_v", s);
                if (st != PMHA_OK) return st;
            }
        }
        a.q = qkv;
        a.q_ld = E;
        a.kv = kvbuf;
        a.kv_ld = kv_w;
    }
    a.v_off = E;
    a.mixed = with_values ? ws + lay.mixed : nullptr;
    a.part = (float *)(ws + lay.part);
    a.ml = ml_keep ? ml_keep : (wmode != PMHA_WEIGHTS_NONE ? (float *)(ws + lay.ml) : nullptr);
    a.scores = wmode == PMHA_WEIGHTS_NONE ? nullptr : (float *)(ws + lay.scores);
    a.B = B;
    a.L = L;
    a.S = S;
    a.E = E;
    a.H = H;
    a.nnz = g->nnz;
    a.score_scale = (float)(1.4426950408889634 / sqrt((double)(E / H)));
    a.with_values = with_values;
    a.kpm = kpm;
    a.counters = (int *)(ws + lay.counters);
    a.kpm_bits = (uint32_t *)(ws + lay.kpm_bits);
    if (args_out) *args_out = a;
    if (dense_path) {
        // most (target, source) pairs are edges: steps 2-4 as masked-dense tiles
        DenseInputs din;
        din.q = a.q;
        din.q_ld = a.q_ld;
        din.k = a.kv;
        din.k_ld = a.kv_ld;
        din.v = (const char *)a.kv + (size_t)a.v_off * es;
        din.v_ld = a.kv_ld;
        din.vt = ws + lay.vt;
        din.mixed = a.mixed;
        din.kpm = kpm;
        din.B = B;
        din.E = E;
        din.H = H;
        if ((st = dense_attention(g, din, s)) != PMHA_OK) return st;
        if (wmode != PMHA_WEIGHTS_NONE) {
            // weights from the per-edge scores: the kernels pmha_edge_weights runs
            EdgeArgs w = a;
            w.with_values = false;
            if ((st = edge_attention(it, g, w, s)) != PMHA_OK) return st;
            if ((st = empty_targets(it, g, w, s)) != PMHA_OK) return st;
            if ((st = weights_finalize(g, w, wmode, weights, s)) != PMHA_OK) return st;
        }
        if (mixed_out) *mixed_out = a.mixed;
        return PMHA_OK;
    }
    if (heavy_path) {
        // heavy targets on the tensor cores, the others on the per-edge kernel
        // over the light part of the graph (whose empty targets include the
        // heavy ones: their zero rows are overwritten by the heavy path)
        if ((st = edge_attention(it, g->light, a, s)) != PMHA_OK) return st;
        if ((st = empty_targets(it, g->light, a, s)) != PMHA_OK) return st;
        HeavyInputs hin;
        hin.q = a.q;
        hin.q_ld = a.q_ld;
        hin.x = key;
        hin.wk = p->wk;
        hin.wv = p->wv;
        hin.bv = p->bv;
        hin.mixed = a.mixed;
        hin.workspace = ws + lay.heavy;
        hin.B = B;
        hin.H = H;
        if ((st = heavy_attention(g, hin, s)) != PMHA_OK) return st;
        if (mixed_out) *mixed_out = a.mixed;
        return PMHA_OK;
    }
    if (fuse) {
        a.out = fused_out;
        a.wo_frag = wo16;
        a.bo = p->bo;
    }
    if ((st = edge_attention(inter_type(p->dtype), g, a, s)) != PMHA_OK) return st;
    if ((st = empty_targets(inter_type(p->dtype), g, a, s)) != PMHA_OK) return st;
    if (wmode != PMHA_WEIGHTS_NONE)
        if ((st = weights_finalize(g, a, wmode, weights, s)) != PMHA_OK) return st;
    if (mixed_out) *mixed_out = a.mixed;
    return PMHA_OK;
}

pmha_status check_wmode(pmha_wmode wmode, const float *weights, bool allow_none)
{
    if (wmode != PMHA_WEIGHTS_NONE && wmode != PMHA_WEIGHTS_AVG && wmode != PMHA_WEIGHTS_PER_HEAD) {
        set_error("weight mode %d is not a pmha_wmode", (int)wmode);
        return PMHA_ERR_INVALID_ARG;
    }
    if (wmode == PMHA_WEIGHTS_NONE && !allow_none) {
        set_error("pmha_edge_weights needs PMHA_WEIGHTS_AVG or PMHA_WEIGHTS_PER_HEAD");
        return PMHA_ERR_INVALID_ARG;
    }
    if ((wmode == PMHA_WEIGHTS_NONE) != (weights == nullptr)) {
        set_error("weights must be given exactly when a weight mode is requested");
        return PMHA_ERR_INVALID_ARG;
    }
    if (weights && ((uintptr_t)weights & 3u)) {
        set_error("weights must be 4-byte aligned");
        return PMHA_ERR_INVALID_ARG;
    }
    return PMHA_OK;
}

pmha_status forward_device(const pmha_graph *g, const pmha_params *p, const void *query, const void *key,
                           const void *value, const uint8_t *kpm, int64_t B, void *output, pmha_wmode wmode, float *weights,
                           void *workspace, size_t ws_bytes, cudaStream_t s)
{
    pmha_status st = check_params(g, p, B);
    if (st != PMHA_OK) return st;
    if ((st = check_wmode(wmode, weights, true)) != PMHA_OK) return st;
    if (!query || !key || !value || !output || !aligned16(query) || !aligned16(key) || !aligned16(value) ||
        !aligned16(output)) {
        set_error("query, key, value and output must be non-NULL, 16-byte aligned device pointers");
        return PMHA_ERR_INVALID_ARG;
    }
    if ((p->embed_dim * (int64_t)elem_size(p->dtype)) % 16) {
        set_error("embed_dim %lld gives rows that are not a multiple of 16 bytes", (long long)p->embed_dim);
        return PMHA_ERR_UNSUPPORTED;
    }
    const Layout lay = layout(g, p, B, wmode, true);
    if (!workspace || ws_bytes < lay.total || ((uintptr_t)workspace & 255u)) {
        set_error("workspace needs %zu bytes, 256-byte aligned (got %zu at %p)", lay.total, ws_bytes, workspace);
        return PMHA_ERR_WORKSPACE;
    }
    char *ws = (char *)workspace;
    const void *mixed = nullptr;
    // both MMA operands of out_proj on the tensor cores must share one type:
    // step 1's GEMM (same condition) leaves an fp16 copy of Wo in wo16
    const bool tc_out = out_proj_on_tensor_cores(p);
    void *wo16 = tc_out ? ws + lay.wo16 : nullptr;
    bool fused = false;
    st = attend(g, p, query, key, value, kpm, B, wmode, weights, ws, lay, true, s, &mixed, nullptr, true, nullptr, wo16,
                fuse_out_proj() ? output : nullptr, &fused);
    if (st != PMHA_OK) return st;
    if (fused) return PMHA_OK;  // step 5 ran inside the edge kernel
    // step 5: out_proj over the joined heads, mixed (intermediate type) -> output (layer dtype)
    const int64_t E = p->embed_dim;
    if (tc_out)
        return gemm_tc(TcType::F16, TcType::BF16, mixed, B * g->L, E, segs(wo16, p->bo), output, E, "out_proj", s);
    return gemm_simt(inter_type(p->dtype), param_type(p->dtype), param_type(p->dtype), mixed, B * g->L, E,
                     segs(p->wo, p->bo), output, E, "out_proj", s);
}

// Workspace of the backward pass: the forward's regions, then (m, l), D,
// the per-row records {m + log2(l), D} and task counters of the ring kernels,
// dmixed, dq, dk, dv, partial sums, an fp32 input-gradient accumulator and
// the chunk partials of the weight-gradient sums.
struct BwdLayout {
    Layout f;
    size_t ml = 0, D = 0, rec = 0, ctr = 0, dmixed = 0, dq = 0, dk = 0, dv = 0, pdq = 0, pdkv = 0, dx = 0, scratch = 0,
           total = 0;
    int64_t chunks = 1;
};

BwdLayout bwd_layout(const pmha_graph *g, const pmha_params *p, int64_t B)
{
    const int64_t E = p->embed_dim, H = p->num_heads, L = g->L, S = g->S;
    const size_t es = type_size(inter_type(p->dtype));
    BwdLayout b;
    b.f = layout(g, p, B, PMHA_WEIGHTS_NONE, true);
    size_t o = b.f.total;
    b.ml = o;
    o += align256((size_t)(B * L * H * 2) * 4);
    b.D = o;
    o += align256((size_t)(B * L * H) * 4);
    b.rec = o;
    o += align256((size_t)(B * L * H) * 8);
    b.ctr = o;
    o += 256;
    b.dmixed = o;
    o += align256((size_t)(B * L * E) * es);
    b.dq = o;
    o += align256((size_t)(B * L * E) * 4);
    b.dk = o;
    o += align256((size_t)(B * S * E) * 4);
    b.dv = o;
    o += align256((size_t)(B * S * E) * 4);
    b.pdq = o;
    o += align256((size_t)(B * 2 * g->n_units * E) * 4);
    b.pdkv = o;
    o += align256((size_t)(B * 2 * g->n_units * 2 * E) * 4);
    b.dx = o;
    o += align256((size_t)(std::max(B * L, B * S) * E) * 4);
    b.chunks = std::max<int64_t>(1, std::min<int64_t>(64, std::max(B * L, B * S) / 4096));
    b.scratch = o;
    o += align256(bwd_gemm_scratch_bytes(B, L, S, E, param_type(p->dtype)));
    b.total = o;
    return b;
}

}  // namespace
}  // namespace pmha

using namespace pmha;

extern "C" {

pmha_status pmha_build_csr(const int64_t *source_index, const int64_t *target_index, int64_t nnz,
                           int64_t query_features, int64_t key_features, int add_self_loops, pmha_stream stream,
                           pmha_graph **out)
{
    if (!out) {
        set_error("pmha_build_csr: out is NULL");
        return PMHA_ERR_INVALID_ARG;
    }
    *out = nullptr;
    if (nnz < 1) {
        set_error("pmha_build_csr: the index arrays are empty (nnz must be >= 1)");
        return PMHA_ERR_EMPTY;
    }
    if (!source_index || !target_index) {
        set_error("pmha_build_csr: NULL index array");
        return PMHA_ERR_INVALID_ARG;
    }
    if (((uintptr_t)source_index & 7u) || ((uintptr_t)target_index & 7u)) {
        set_error("pmha_build_csr: index arrays must be 8-byte aligned");
        return PMHA_ERR_INVALID_ARG;
    }
    if (query_features < 1 || key_features < 1 || query_features > 0x7ffffffe || key_features > 0x7ffffffe) {
        set_error("pmha_build_csr: query_features and key_features must be in [1, 2^31 - 2]");
        return PMHA_ERR_INVALID_ARG;
    }
    if (add_self_loops && query_features != key_features) {
        set_error("pmha_build_csr: add_self_loops needs query_features == key_features");
        return PMHA_ERR_INVALID_ARG;
    }
    const int64_t cap = nnz + (add_self_loops ? query_features : 0);
    if (cap > 0x7fffffffLL - 8192) {
        set_error("pmha_build_csr: more than 2^31 - 8193 edges");
        return PMHA_ERR_INVALID_ARG;
    }
    cudaPointerAttributes at;
    for (const int64_t *ptr : {source_index, target_index}) {
        if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess || (at.type != cudaMemoryTypeDevice &&
                                                                  at.type != cudaMemoryTypeManaged)) {
            cudaGetLastError();
            set_error("pmha_build_csr: index arrays must be device memory");
            return PMHA_ERR_INVALID_ARG;
        }
    }
    pmha_status st = build_csr(source_index, target_index, nnz, query_features, key_features, add_self_loops != 0,
                               (cudaStream_t)stream, out);
    if (st != PMHA_OK) return st;
    if ((st = split_heavy(*out, heavy_min_degree(), (cudaStream_t)stream)) != PMHA_OK) {
        destroy_graph(*out);
        *out = nullptr;
    }
    return st;
}

pmha_status pmha_graph_info(const pmha_graph *g, int64_t *nnz_total, int64_t *L, int64_t *S, int64_t *max_deg)
{
    if (!g) {
        set_error("graph is NULL");
        return PMHA_ERR_INVALID_ARG;
    }
    if (nnz_total) *nnz_total = g->nnz;
    if (L) *L = g->L;
    if (S) *S = g->S;
    if (max_deg) *max_deg = g->max_deg;
    return PMHA_OK;
}

pmha_status pmha_graph_split_info(const pmha_graph *g, int64_t *n_heavy, int64_t *heavy_min_degree, int64_t *light_nnz)
{
    if (!g) {
        set_error("graph is NULL");
        return PMHA_ERR_INVALID_ARG;
    }
    if (n_heavy) *n_heavy = g->light ? g->n_heavy : 0;
    if (heavy_min_degree) *heavy_min_degree = g->heavy_min_deg;
    if (light_nnz) *light_nnz = g->light ? g->light->nnz : g->nnz;
    return PMHA_OK;
}

pmha_status pmha_graph_export(const pmha_graph *g, int32_t *row_ptr, int32_t *col, int32_t *perm,
                              pmha_stream stream)
{
    if (!g) {
        set_error("graph is NULL");
        return PMHA_ERR_INVALID_ARG;
    }
    cudaStream_t s = (cudaStream_t)stream;
    if (row_ptr)
        PMHA_CUDA_TRY(cudaMemcpyAsync(row_ptr, g->row_ptr, (size_t)(g->L + 1) * 4, cudaMemcpyDeviceToDevice, s));
    if (col) PMHA_CUDA_TRY(cudaMemcpyAsync(col, g->col, (size_t)g->nnz * 4, cudaMemcpyDeviceToDevice, s));
    if (perm) PMHA_CUDA_TRY(cudaMemcpyAsync(perm, g->perm, (size_t)g->nnz * 4, cudaMemcpyDeviceToDevice, s));
    return PMHA_OK;
}

pmha_status pmha_graph_export_by_source(const pmha_graph *g, int32_t *src_row_ptr, int32_t *target,
                                        pmha_stream stream)
{
    if (!g) {
        set_error("graph is NULL");
        return PMHA_ERR_INVALID_ARG;
    }
    cudaStream_t s = (cudaStream_t)stream;
    if (src_row_ptr)
        PMHA_CUDA_TRY(cudaMemcpyAsync(src_row_ptr, g->src_row_ptr, (size_t)(g->S + 1) * 4, cudaMemcpyDeviceToDevice,
                                      s));
    if (target) PMHA_CUDA_TRY(cudaMemcpyAsync(target, g->tgt_by_src, (size_t)g->nnz * 4, cudaMemcpyDeviceToDevice, s));
    return PMHA_OK;
}

void pmha_graph_destroy(pmha_graph *g)
{
    destroy_graph(g);
}

size_t pmha_forward_workspace_size(const pmha_graph *g, const pmha_params *p, int64_t batch, pmha_wmode wmode)
{
    if (check_params(g, p, batch) != PMHA_OK) return 0;
    if (wmode != PMHA_WEIGHTS_NONE && wmode != PMHA_WEIGHTS_AVG && wmode != PMHA_WEIGHTS_PER_HEAD) return 0;
    return layout(g, p, batch, wmode, true).total;
}

size_t pmha_edge_weights_workspace_size(const pmha_graph *g, const pmha_params *p, int64_t batch, pmha_wmode wmode)
{
    if (check_params(g, p, batch) != PMHA_OK) return 0;
    if (wmode != PMHA_WEIGHTS_AVG && wmode != PMHA_WEIGHTS_PER_HEAD) return 0;
    return layout(g, p, batch, wmode, false).total;
}

pmha_status pmha_forward(const pmha_graph *g, const pmha_params *p, const void *query, const void *key,
                         const void *value, const uint8_t *key_padding_mask, int64_t batch, void *output,
                         pmha_wmode wmode, float *weights, void *workspace, size_t ws_bytes, pmha_stream stream)
{
    return forward_device(g, p, query, key, value, key_padding_mask, batch, output, wmode, weights, workspace, ws_bytes,
                          (cudaStream_t)stream);
}

// Host-buffer variant: [inputs | key_padding_mask | output | weights | forward workspace].
static size_t host_staging(const pmha_graph *g, const pmha_params *p, int64_t B, pmha_wmode wmode, size_t *off_in,
                           size_t *off_mask, size_t *off_out, size_t *off_w, size_t *off_ws)
{
    const size_t es = elem_size(p->dtype);
    const size_t q = align256((size_t)(B * g->L * p->embed_dim) * es);
    const size_t kv = align256((size_t)(B * g->S * p->embed_dim) * es);
    size_t o = 0;
    *off_in = o;
    o += q + 2 * kv;
    *off_mask = o;
    o += align256((size_t)(B * g->S));
    *off_out = o;
    o += q;
    *off_w = o;
    if (wmode == PMHA_WEIGHTS_AVG) o += align256((size_t)(B * g->nnz) * 4);
    if (wmode == PMHA_WEIGHTS_PER_HEAD) o += align256((size_t)(B * g->nnz * p->num_heads) * 4);
    *off_ws = o;
    return o + layout(g, p, B, wmode, true).total;
}

size_t pmha_forward_host_workspace_size(const pmha_graph *g, const pmha_params *p, int64_t batch, pmha_wmode wmode)
{
    if (check_params(g, p, batch) != PMHA_OK) return 0;
    if (wmode != PMHA_WEIGHTS_NONE && wmode != PMHA_WEIGHTS_AVG && wmode != PMHA_WEIGHTS_PER_HEAD) return 0;
    size_t a, b, c, d, e;
    return host_staging(g, p, batch, wmode, &a, &b, &c, &d, &e);
}

pmha_status pmha_forward_host(const pmha_graph *g, const pmha_params *p, const void *qh, const void *kh,
                              const void *vh, const uint8_t *mh, int64_t B, void *oh, pmha_wmode wmode, float *wh, void *workspace,
                              size_t ws_bytes, pmha_stream stream)
{
    pmha_status st = check_params(g, p, B);
    if (st != PMHA_OK) return st;
    if ((st = check_wmode(wmode, wh, true)) != PMHA_OK) return st;
    if (!qh || !kh || !vh || !oh) {
        set_error("pmha_forward_host: NULL host buffer");
        return PMHA_ERR_INVALID_ARG;
    }
    size_t off_in, off_mask, off_out, off_w, off_ws;
    const size_t need = host_staging(g, p, B, wmode, &off_in, &off_mask, &off_out, &off_w, &off_ws);
    if (!workspace || ws_bytes < need || ((uintptr_t)workspace & 255u)) {
        set_error("pmha_forward_host: workspace needs %zu bytes, 256-byte aligned", need);
        return PMHA_ERR_WORKSPACE;
    }
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = (char *)workspace;
    const size_t es = elem_size(p->dtype);
    const size_t qb = (size_t)(B * g->L * p->embed_dim) * es, kb = (size_t)(B * g->S * p->embed_dim) * es;
    char *dq = ws + off_in;
    char *dk = dq + align256(qb);
    char *dv = dk + align256(kb);
    const void *q_dev = dq, *k_dev = dk, *v_dev = dv;
    {
        StageTimer timer("h2d", s);
        PMHA_CUDA_TRY(cudaMemcpyAsync(dq, qh, qb, cudaMemcpyHostToDevice, s));
        if (kh == qh && g->L == g->S) k_dev = dq;
        else PMHA_CUDA_TRY(cudaMemcpyAsync(dk, kh, kb, cudaMemcpyHostToDevice, s));
        if (vh == kh) v_dev = k_dev;
        else if (vh == qh && g->L == g->S) v_dev = dq;
        else PMHA_CUDA_TRY(cudaMemcpyAsync(dv, vh, kb, cudaMemcpyHostToDevice, s));
        if (mh) PMHA_CUDA_TRY(cudaMemcpyAsync(ws + off_mask, mh, (size_t)(B * g->S), cudaMemcpyHostToDevice, s));
    }
    const uint8_t *m_dev = mh ? (const uint8_t *)(ws + off_mask) : nullptr;
    float *dw = wmode != PMHA_WEIGHTS_NONE ? (float *)(ws + off_w) : nullptr;
    st = forward_device(g, p, q_dev, k_dev, v_dev, m_dev, B, ws + off_out, wmode, dw, ws + off_ws, ws_bytes - off_ws, s);
    if (st != PMHA_OK) return st;
    {
        StageTimer timer("d2h", s);
        PMHA_CUDA_TRY(cudaMemcpyAsync(oh, ws + off_out, qb, cudaMemcpyDeviceToHost, s));
        if (dw) {
            const size_t wb = (size_t)(B * g->nnz) * 4 * (wmode == PMHA_WEIGHTS_PER_HEAD ? p->num_heads : 1);
            PMHA_CUDA_TRY(cudaMemcpyAsync(wh, dw, wb, cudaMemcpyDeviceToHost, s));
        }
    }
    return PMHA_OK;
}

pmha_status pmha_edge_weights(const pmha_graph *g, const pmha_params *p, const void *query, const void *key,
                              const uint8_t *key_padding_mask, int64_t B, pmha_wmode wmode, float *weights, void *workspace, size_t ws_bytes,
                              pmha_stream stream)
{
    pmha_status st = check_params(g, p, B);
    if (st != PMHA_OK) return st;
    if ((st = check_wmode(wmode, weights, false)) != PMHA_OK) return st;
    if (!query || !key || !aligned16(query) || !aligned16(key)) {
        set_error("query and key must be non-NULL, 16-byte aligned device pointers");
        return PMHA_ERR_INVALID_ARG;
    }
    if ((p->embed_dim * (int64_t)elem_size(p->dtype)) % 16) {
        set_error("embed_dim %lld gives rows that are not a multiple of 16 bytes", (long long)p->embed_dim);
        return PMHA_ERR_UNSUPPORTED;
    }
    const Layout lay = layout(g, p, B, wmode, false);
    if (!workspace || ws_bytes < lay.total || ((uintptr_t)workspace & 255u)) {
        set_error("workspace needs %zu bytes, 256-byte aligned (got %zu)", lay.total, ws_bytes);
        return PMHA_ERR_WORKSPACE;
    }
    return attend(g, p, query, key, key, key_padding_mask, B, wmode, weights, (char *)workspace, lay, false, (cudaStream_t)stream,
                  nullptr);
}

size_t pmha_backward_workspace_size(const pmha_graph *g, const pmha_params *p, int64_t batch)
{
    if (check_params(g, p, batch) != PMHA_OK) return 0;
    int cpl, lpe;
    if (!bwd_shape(p->embed_dim, p->num_heads, &cpl, &lpe, inter_type(p->dtype))) return 0;
    return bwd_layout(g, p, batch).total;
}

pmha_status pmha_backward(const pmha_graph *g, const pmha_params *p, const void *query, const void *key,
                          const void *value, const uint8_t *key_padding_mask, int64_t B, const void *dout,
                          void *dquery, void *dkey, void *dvalue, const pmha_grads *grads, void *workspace,
                          size_t ws_bytes, pmha_stream stream)
{
    pmha_status st = check_params(g, p, B);
    if (st != PMHA_OK) return st;
    const int64_t E = p->embed_dim, H = p->num_heads, L = g->L, S = g->S;
    if (!query || !key || !value || !dout || !aligned16(query) || !aligned16(key) || !aligned16(value) ||
        !aligned16(dout)) {
        set_error("pmha_backward: query, key, value and dout must be non-NULL, 16-byte aligned device pointers");
        return PMHA_ERR_INVALID_ARG;
    }
    if ((E * (int64_t)elem_size(p->dtype)) % 16) {
        set_error("embed_dim %lld gives rows that are not a multiple of 16 bytes", (long long)E);
        return PMHA_ERR_UNSUPPORTED;
    }
    int cpl, lpe;
    if (!bwd_shape(E, H, &cpl, &lpe, inter_type(p->dtype))) {
        set_error("pmha_backward: no kernel for embed_dim %lld, num_heads %lld", (long long)E, (long long)H);
        return PMHA_ERR_UNSUPPORTED;
    }
    if ((query == key || query == value) && L != S) {
        set_error("pmha_backward: one tensor cannot be the query (%lld tokens) and a key/value (%lld tokens)",
                  (long long)L, (long long)S);
        return PMHA_ERR_INVALID_ARG;
    }
    // roles sharing one input tensor must share (or leave NULL) their gradient buffer
    const void *in[3] = {query, key, value};
    void *gx[3] = {dquery, dkey, dvalue};
    for (int i = 0; i < 3; ++i)
        for (int j = i + 1; j < 3; ++j)
            if (in[i] == in[j] && gx[i] && gx[j] && gx[i] != gx[j]) {
                set_error("pmha_backward: inputs %d and %d are one tensor, so their gradients must be one buffer", i,
                          j);
                return PMHA_ERR_INVALID_ARG;
            }
    const BwdLayout bl = bwd_layout(g, p, B);
    if (!workspace || ws_bytes < bl.total || ((uintptr_t)workspace & 255u)) {
        set_error("pmha_backward: workspace needs %zu bytes, 256-byte aligned (got %zu)", bl.total, ws_bytes);
        return PMHA_ERR_WORKSPACE;
    }
    cudaStream_t s = (cudaStream_t)stream;
    char *ws = (char *)workspace;
    const TcType it = inter_type(p->dtype), pt = param_type(p->dtype);
    const size_t es = type_size(it);
    float *ml = (float *)(ws + bl.ml), *D = (float *)(ws + bl.D);
    void *dmixed = ws + bl.dmixed;
    float *dq = (float *)(ws + bl.dq), *dk = (float *)(ws + bl.dk), *dv = (float *)(ws + bl.dv);
    float *dx = (float *)(ws + bl.dx), *scratch = (float *)(ws + bl.scratch);

    // forward recompute: projections, (m, l) of every target, the mix
    EdgeArgs a;
    const void *mixed = nullptr;
    st = attend(g, p, query, key, value, key_padding_mask, B, PMHA_WEIGHTS_NONE, nullptr, ws, bl.f, true, s, &mixed,
                ml, false, &a);
    if (st != PMHA_OK) return st;
    // step 5
    BwdGemmArgs gm;
    gm.pt = pt;
    gm.it = it;
    gm.B = B;
    gm.L = L;
    gm.S = S;
    gm.E = E;
    gm.dout = dout;
    gm.mixed = mixed;
    gm.w[0] = p->wq;
    gm.w[1] = p->wk;
    gm.w[2] = p->wv;
    gm.w[3] = p->wo;
    for (int r = 0; r < 3; ++r) {
        gm.in[r] = in[r];
        gm.gx[r] = gx[r];
    }
    gm.dy[0] = dq;
    gm.dy[1] = dk;
    gm.dy[2] = dv;
    gm.gw[0] = grads ? grads->wq : nullptr;
    gm.gw[1] = grads ? grads->wk : nullptr;
    gm.gw[2] = grads ? grads->wv : nullptr;
    gm.gw[3] = grads ? grads->wo : nullptr;
    gm.gb[0] = grads ? grads->bq : nullptr;
    gm.gb[1] = grads ? grads->bk : nullptr;
    gm.gb[2] = grads ? grads->bv : nullptr;
    gm.gb[3] = grads ? grads->bo : nullptr;
    gm.dmixed = dmixed;
    gm.dx32 = dx;
    gm.scratch = scratch;
    gm.chunks = bl.chunks;
    if ((st = bwd_step5(gm, s)) != PMHA_OK) return st;
    // steps 2-4
    float2 *rec = (float2 *)(ws + bl.rec);
    if ((st = bwd_rowdot(it, dmixed, mixed, B * L, E, H, D, ml, rec, s)) != PMHA_OK) return st;
    BwdAttnArgs x;
    x.q = a.q;
    x.q_ld = a.q_ld;
    x.k = a.kv;
    x.v = (const char *)a.kv + (size_t)a.v_off * es;
    x.kv_ld = a.kv_ld;
    x.dmixed = dmixed;
    x.ml = ml;
    x.D = D;
    x.rec = rec;
    x.ctr = (unsigned *)(ws + bl.ctr);
    x.kpm = key_padding_mask;
    x.dq = dq;
    x.dk = dk;
    x.dv = dv;
    x.part_dq = (float *)(ws + bl.pdq);
    x.part_dkv = (float *)(ws + bl.pdkv);
    x.B = B;
    x.E = E;
    x.H = H;
    if ((st = bwd_attention(it, g, x, s)) != PMHA_OK) return st;
    // step 1: weight, bias and input gradients of the projections
    if ((st = bwd_step1(gm, s)) != PMHA_OK) return st;
    return PMHA_OK;
}

pmha_status pmha_device_status(pmha_stream stream)
{
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "pmha_device_status");
    int *w = device_error_word();
    if (!w) return PMHA_ERR_CUDA;
    int v = 0;
    e = cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "pmha_device_status");
    if (v != 0) {
        const int zero = 0;
        cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (v & kErrInternalBit) {
            set_error("a kernel found its launch configuration unusable and did nothing");
            return PMHA_ERR_CUDA;
        }
        if (v & kErrTimeoutBit) {
            set_error("a bounded device-side wait gave up");
            return PMHA_ERR_TIMEOUT;
        }
        set_error("an intermediate (q, k, v or mixed) left the fp16 range; the results since the last check "
                  "are not valid");
        return PMHA_ERR_OVERFLOW;
    }
    return PMHA_OK;
}

const char *pmha_last_error(void) { return t_err; }

pmha_status pmha_profile_enable(int on)
{
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = on != 0;
    return PMHA_OK;
}

pmha_status pmha_profile_read(int max_stages, char *names, int64_t *launches, double *total_ms, int *n_stages)
{
    std::vector<Record> recs;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        recs.swap(g_records);
    }
    std::vector<std::string> stage_names;
    std::vector<int64_t> counts;
    std::vector<double> totals;
    pmha_status st = PMHA_OK;
    for (const Record &r : recs) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(r.stop);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
        if (e != cudaSuccess) {
            st = cuda_fail(e, "pmha_profile_read");
            continue;
        }
        size_t i = 0;
        while (i < stage_names.size() && stage_names[i] != r.stage) ++i;
        if (i == stage_names.size()) {
            stage_names.push_back(r.stage);
            counts.push_back(0);
            totals.push_back(0.0);
        }
        counts[i] += 1;
        totals[i] += ms;
    }
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        for (const Record &r : recs) {
            g_event_pool.push_back(r.start);
            g_event_pool.push_back(r.stop);
        }
    }
    const int n = (int)stage_names.size();
    if (n_stages) *n_stages = n;
    for (int i = 0; i < n && i < max_stages; ++i) {
        if (names) {
            strncpy(names + 32 * i, stage_names[i].c_str(), 31);
            names[32 * i + 31] = '\0';
        }
        if (launches) launches[i] = counts[i];
        if (total_ms) total_ms[i] = totals[i];
    }
    return st;
}

int64_t pmha_launch_count(void) { return g_launches.load(); }

}  // extern "C"
