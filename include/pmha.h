/*
 * pmha.h - C ABI of the edge-packed multi-head attention library for GB300.
 *
 * The layer (kpnn2 0.3.0 API reference, page "PackedMultiheadAttention"):
 * each query token (a target node) attends only to the key tokens (its
 * sources) along live edges (source_index[e], target_index[e]). For every
 * sample, target t and head h (d = embed_dim / num_heads channels):
 *   Notes step 1   q = Wq x_q + bq, k = Wk x_k + bk, v = Wv x_v + bv
 *   Notes step 2   score[e] = dot(q[t], k[s]) / sqrt(d)
 *   Notes step 3   softmax of the scores over the edges into t only
 *   Notes step 4   mixed[t] = sum over edges e into t of weight[e] * v[s]
 *   Notes step 5   join the heads' slices and apply out_proj (Wo, bo)
 * and, from the paragraph after the steps, a target with no live key mixes
 * to zeros (its output is bo).
 *
 * Conventions for every call:
 *  - Pointers marked "device" point to memory of the current CUDA device;
 *    pointers marked "host" to host memory (pinned memory makes the copies
 *    asynchronous). All device pointers must be 16-byte aligned.
 *  - Tensors are dense row-major: query (B, L, E), key and value (B, S, E),
 *    output (B, L, E), weights (B, nnz) or (B, nnz, H) in float32. Projection
 *    weights are (E, E) stored (out_features, in_features) like nn.Linear.
 *  - The caller owns every buffer it passes, including the workspace. The
 *    library owns only the arrays inside a pmha_graph, released by
 *    pmha_graph_destroy. It keeps no pointer to caller memory after a call.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *    unless stated. Every call returns a pmha_status; on failure
 *    pmha_last_error() gives a message for the calling thread. A failing call
 *    writes nothing to its outputs unless it says otherwise.
 *  - Nothing in this library waits on another CTA or launch inside a kernel;
 *    the only bounded device-side waits are the tensor-core GEMM's pipeline
 *    barriers, which give up with PMHA_ERR_TIMEOUT (see pmha_device_status).
 */
#ifndef PMHA_H
#define PMHA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header needs no CUDA header. */
typedef struct CUstream_st *pmha_stream;

typedef enum {
    PMHA_OK = 0,
    PMHA_ERR_INVALID_ARG = 1,    /* a size, pointer, alignment or option is not accepted */
    PMHA_ERR_INDEX_RANGE = 2,    /* an index lies outside [0, key_features) / [0, query_features) */
    PMHA_ERR_DUPLICATE_EDGE = 3, /* a (source, target) pair is given twice */
    PMHA_ERR_EMPTY = 4,          /* nnz < 1 */
    PMHA_ERR_UNSUPPORTED = 5,    /* a valid combination this build has no kernel for */
    PMHA_ERR_WORKSPACE = 6,      /* workspace NULL or smaller than the matching *_workspace_size */
    PMHA_ERR_CUDA = 7,           /* a CUDA runtime or launch error; see pmha_last_error() */
    PMHA_ERR_TIMEOUT = 8,        /* a bounded device-side wait gave up (reported by pmha_device_status) */
    PMHA_ERR_OVERFLOW = 9        /* an fp16 intermediate overflowed (reported by pmha_device_status) */
} pmha_status;

/* Precision. A PMHA_BF16 layer takes bf16 tokens, projections and biases and
 * returns bf16 output; all arithmetic accumulates in fp32, and the
 * intermediates q, k, v and the per-target mix are stored in fp16 (same width
 * as bf16, 3 more mantissa bits). A projected value outside the fp16 range
 * (|x| > 65504) is flagged and reported as PMHA_ERR_OVERFLOW by
 * pmha_device_status. A PMHA_F32 layer keeps everything in float32. */

typedef enum { PMHA_F32 = 0, PMHA_BF16 = 1 } pmha_dtype;

/* need_weights / average_attn_weights of kpnn2's forward(): NONE = no weights,
 * AVG = mean over heads, shape (B, nnz); PER_HEAD = shape (B, nnz, H). */
typedef enum { PMHA_WEIGHTS_NONE = 0, PMHA_WEIGHTS_AVG = 1, PMHA_WEIGHTS_PER_HEAD = 2 } pmha_wmode;

/* The four learned projections (kpnn2 PackedMultiheadAttention, attribute
 * table: q_proj, k_proj, v_proj, out_proj, separate embed_dim x embed_dim
 * nn.Linear layers). All pointers are device pointers in `dtype`. A NULL bias
 * pointer means that projection has no bias (bias=False). */
typedef struct {
    int64_t embed_dim;   /* E, positive, divisible by num_heads */
    int64_t num_heads;   /* H */
    pmha_dtype dtype;    /* storage type of tokens, projections and output */
    const void *wq, *wk, *wv, *wo;  /* (E, E) (out, in) */
    const void *bq, *bk, *bv, *bo;  /* (E,) or NULL */
} pmha_params;

/* Opaque graph: the live edges grouped by target (CSR by target), kept on the device. */
typedef struct pmha_graph pmha_graph;

/*
 * pmha_build_csr - validate the packed edge index and build the per-target
 * view used by every later call. (kpnn2 PackedMultiheadAttention,
 * constructor parameters source_index, target_index, query_features,
 * key_features, add_self_loops, and the constructor's Raises table.)
 *
 *  source_index, target_index  device int64 arrays of length nnz, paired by
 *        position; source_index[e] in [0, key_features), target_index[e] in
 *        [0, query_features); no pair may repeat. Their order is the order of
 *        the per-edge weights. Read during the call only (copy semantics).
 *  nnz   number of given pairs, >= 1.
 *  query_features (L), key_features (S)  positive sequence lengths.
 *  add_self_loops  nonzero: every missing (i, i) is appended after the given
 *        pairs, i ascending; requires L == S. Existing self-loops are kept.
 *  out   receives the new graph on PMHA_OK (NULL on failure).
 *
 * Edges into one target are ordered by source index, so the graph (and every
 * result computed on it) does not depend on the order of the given pairs
 * except for the order of the returned weights.
 * Errors: PMHA_ERR_EMPTY, PMHA_ERR_INVALID_ARG (sizes, L != S with self-loops,
 * more than 2^31 - 1 edges), PMHA_ERR_INDEX_RANGE, PMHA_ERR_DUPLICATE_EDGE,
 * PMHA_ERR_CUDA. The call allocates device memory and synchronizes `stream`
 * once, to read the validation result; it is the only synchronizing call.
 */
pmha_status pmha_build_csr(const int64_t *source_index, const int64_t *target_index, int64_t nnz,
                           int64_t query_features, int64_t key_features, int add_self_loops,
                           pmha_stream stream, pmha_graph **out);

/* Sizes of a built graph (host outputs, any may be NULL). nnz_total counts
 * appended self-loops (kpnn2 attribute nnz); max_in_degree is the largest
 * number of edges into one target. */
pmha_status pmha_graph_info(const pmha_graph *graph, int64_t *nnz_total, int64_t *query_features,
                            int64_t *key_features, int64_t *max_in_degree);

/* How pmha_build_csr split the targets for pmha_forward (host outputs, any
 * may be NULL). Targets with at least heavy_min_degree incoming edges
 * ("heavy") run on the tensor-core path when pmha_forward computes values
 * without weights and without a key_padding_mask, for a bf16 layer with
 * embed_dim 128, at most 8 heads and key == value (the same pointer): their
 * scores and mix are two dense products per 128 edges over the gathered key
 * tokens (Notes steps 2-4 rewritten through the step 1 projections:
 * q.k_s = (Wk^T q).x_s + a per-target constant, sum w v_s = Wv (sum w x_s)
 * + bv). The other targets keep the per-edge kernel. The threshold is the
 * value of the environment variable PMHA_HEAVY_MIN_DEGREE when the graph is
 * built; unset or 0 means no split (the default: on the measured workloads
 * the per-edge kernel is faster). n_heavy = 0 means no split (no threshold,
 * no target reaches it, every target does, or the graph is dense);
 * light_nnz counts the edges of the other targets.
 * Errors: PMHA_ERR_INVALID_ARG (graph NULL). */
pmha_status pmha_graph_split_info(const pmha_graph *graph, int64_t *n_heavy, int64_t *heavy_min_degree,
                                  int64_t *light_nnz);

/* Copy the per-target view into caller device buffers (int32):
 *  row_ptr (L + 1)  edges into target t are positions row_ptr[t] .. row_ptr[t+1]-1,
 *  col (nnz_total)  source index of each position, ascending within a target,
 *  perm (nnz_total) position of that edge in the given order (appended
 *                   self-loops numbered after the given pairs).
 * Any pointer may be NULL to skip it. Asynchronous on `stream`. */
pmha_status pmha_graph_export(const pmha_graph *graph, int32_t *row_ptr, int32_t *col,
                              int32_t *perm, pmha_stream stream);

/* Release a graph (NULL is ignored). Waits for nothing: the caller must make
 * sure no call that uses the graph is still running on the device. */
void pmha_graph_destroy(pmha_graph *graph);

/*
 * Workspace (device bytes) that pmha_forward / pmha_edge_weights need for this
 * graph, parameters, batch and weight mode. Returns 0 when the arguments are
 * invalid. A workspace may be reused by later calls on the same stream.
 */
size_t pmha_forward_workspace_size(const pmha_graph *graph, const pmha_params *params,
                                   int64_t batch, pmha_wmode wmode);
size_t pmha_edge_weights_workspace_size(const pmha_graph *graph, const pmha_params *params,
                                        int64_t batch, pmha_wmode wmode);

/*
 * pmha_forward - one forward pass of the layer (kpnn2 PackedMultiheadAttention,
 * forward(): Notes steps 1-5; Returns table).
 *
 *  query  device (B, L, E); key, value device (B, S, E), all in params->dtype.
 *         Passing the same pointer for all three (with L == S) is attention
 *         within one graph and lets the library project them in one GEMM;
 *         key == value shares one GEMM for both.
 *  key_padding_mask  device (B, S) bytes or NULL (forward()'s key_padding_mask):
 *         a nonzero byte drops key s of sample b from the softmax of every
 *         target it feeds; such an edge weighs 0, and a target whose keys
 *         are all dropped mixes to zeros, so its output row is out_proj's
 *         bias. Read-only; NULL drops nothing.
 *  batch  B >= 1.
 *  output device (B, L, E) in params->dtype; must not overlap the inputs.
 *  wmode  PMHA_WEIGHTS_NONE, _AVG or _PER_HEAD (need_weights /
 *         average_attn_weights).
 *  weights device float32, (B, nnz_total) for AVG or (B, nnz_total, H) for
 *         PER_HEAD, one entry per live edge in the given order followed by
 *         appended self-loops; NULL when wmode is NONE. The weights into one
 *         target sum to 1 (to 0 when it has no edge).
 *  workspace, workspace_bytes  device scratch of at least
 *         pmha_forward_workspace_size() bytes, 256-byte aligned.
 * With the environment variable PMHA_FUSED_OUT_PROJ=1 (read at each call),
 * a bf16 layer with embed_dim 128 whose attention runs on the per-edge
 * kernel computes out_proj inside that kernel instead of as its own GEMM
 * (same results within rounding; slower on the measured workloads). A
 * bounded wait there that gives up is reported by pmha_device_status as
 * PMHA_ERR_TIMEOUT.
 * Errors: PMHA_ERR_INVALID_ARG, PMHA_ERR_UNSUPPORTED (a head size or width
 * without a kernel), PMHA_ERR_WORKSPACE, PMHA_ERR_CUDA (launch errors only;
 * the call does not synchronize).
 */
pmha_status pmha_forward(const pmha_graph *graph, const pmha_params *params, const void *query,
                         const void *key, const void *value, const uint8_t *key_padding_mask,
                         int64_t batch, void *output, pmha_wmode wmode, float *weights,
                         void *workspace, size_t workspace_bytes, pmha_stream stream);

/*
 * pmha_forward_host - pmha_forward on HOST buffers: copies query / key / value
 * from host memory to the device, runs the forward pass, and copies output
 * (and weights, if requested) back to host memory, all on `stream`; the call
 * returns after queuing the work, so synchronize `stream` before reading the
 * results. Host buffers should be pinned for the copies to overlap.
 * Same shapes as pmha_forward; equal host pointers for query / key / value
 * are copied once. key_padding_mask_host is a host (B, S) byte array or NULL. The workspace must hold pmha_forward_host_workspace_size()
 * bytes (the device copies of inputs and results live there).
 */
size_t pmha_forward_host_workspace_size(const pmha_graph *graph, const pmha_params *params,
                                        int64_t batch, pmha_wmode wmode);
pmha_status pmha_forward_host(const pmha_graph *graph, const pmha_params *params,
                              const void *query_host, const void *key_host,
                              const void *value_host, const uint8_t *key_padding_mask_host,
                              int64_t batch, void *output_host,
                              pmha_wmode wmode, float *weights_host, void *workspace,
                              size_t workspace_bytes, pmha_stream stream);

/*
 * pmha_edge_weights - the per-edge softmax weights only (kpnn2 forward(),
 * need_weights=True, "for example to draw edge thickness on the prior graph"):
 * projects query and key, scores the live edges and normalizes them, without
 * the value projection, the mix or out_proj. The weights are bit-identical to
 * the ones pmha_forward writes for the same inputs.
 *  wmode  PMHA_WEIGHTS_AVG or PMHA_WEIGHTS_PER_HEAD.
 * Other arguments as in pmha_forward.
 */
pmha_status pmha_edge_weights(const pmha_graph *graph, const pmha_params *params,
                              const void *query, const void *key,
                              const uint8_t *key_padding_mask, int64_t batch, pmha_wmode wmode,
                              float *weights, void *workspace, size_t workspace_bytes,
                              pmha_stream stream);

/*
 * pmha_device_status - synchronize `stream` and report what kernels flagged
 * since the last check: a bounded device-side wait gave up (PMHA_ERR_TIMEOUT),
 * or an fp16 intermediate overflowed (PMHA_ERR_OVERFLOW); PMHA_ERR_CUDA if the
 * stream holds a CUDA error. Clears the flags. PMHA_OK otherwise.
 * The compute calls return as soon as their work is queued, so these
 * conditions never show in their own status: a bfloat16 layer keeps q, k, v
 * and the mix in fp16, and inputs large enough to leave the fp16 range give
 * invalid outputs that only this call reports. Callers that cannot bound
 * their inputs poll it after the calls they want checked.
 */
pmha_status pmha_device_status(pmha_stream stream);

/*
 * pmha_forward_noalloc - pmha_forward for callers that cannot allocate device
 * memory when they call the layer (a host whose allocator owns all device
 * memory, or a call site where cudaMalloc / cudaFree may not run). The pages
 * have no counterpart: it is a property of this library, not of the method.
 *
 * The caller passes inputs and outputs exactly as for pmha_forward; the
 * workspace comes from a scratch array of PMHA_NOALLOC_SCRATCH_BYTES built
 * into the library, which every GPU that loads this code keeps until the
 * process exits. Problems whose pmha_forward_workspace_size exceeds it are
 * rejected with PMHA_ERR_WORKSPACE and a message. Apart from its first call on
 * a device, the call allocates nothing. That first call (with the device
 * current) looks up the array's device address; under CUDA's lazy module
 * loading it is also the moment the array is loaded onto the device, so it
 * reserves the PMHA_NOALLOC_SCRATCH_BYTES and can fail (PMHA_ERR_CUDA, "could
 * not reserve") when other allocations already hold the device's memory: make
 * it early, before an allocator claims the memory, and before any stream
 * capture. The address is cached per device and driver context; it does not
 * survive cudaDeviceReset, so do not use this entry point on a device reset in
 * the same process. All calls share the array: calls whose GPU work overlaps
 * (other streams, unordered threads) race on it; calls queued on one stream
 * are safe.
 */
#define PMHA_NOALLOC_SCRATCH_BYTES (64u << 20)
pmha_status pmha_forward_noalloc(const pmha_graph *graph, const pmha_params *params, const void *query,
                                 const void *key, const void *value,
                                 const uint8_t *key_padding_mask, int64_t batch, void *output,
                                 pmha_wmode wmode, float *weights, pmha_stream stream);

/*
 * pmha_backward - gradients of the layer (the chain rule of kpnn2
 * PackedMultiheadAttention, Notes steps 1-5) for dout = dLoss/d(output).
 * Like the page's training path it recomputes the forward from the inputs
 * instead of keeping per-edge tensors, so it takes the forward's inputs:
 *  query, key, value, key_padding_mask, batch  as for pmha_forward;
 *  dout    device (B, L, E), params->dtype;
 *  dquery  device (B, L, E), dkey and dvalue device (B, S, E), params->dtype,
 *          or NULL (not computed). When two inputs are one tensor (the same
 *          pointer), their gradient is the sum of both roles' gradients and
 *          goes to the one buffer they share (their non-NULL gradient
 *          pointers must then be equal). Written, not accumulated.
 *  grads   device float32 parameter gradients, any member NULL to skip it:
 *          wq, wk, wv, wo (E, E) like the weights, bq, bk, bv, bo (E);
 *          summed over the batch; written, not accumulated. NULL skips all.
 *  workspace  device scratch of pmha_backward_workspace_size() bytes,
 *          256-byte aligned.
 * Sums run in a fixed order: results are deterministic. Supported shapes:
 * embed_dim <= 512 whose lanes split evenly over heads (returns
 * PMHA_ERR_UNSUPPORTED otherwise, and the size function returns 0).
 * Errors as pmha_forward; the call does not synchronize.
 */
typedef struct {
    float *wq, *wk, *wv, *wo;
    float *bq, *bk, *bv, *bo;
} pmha_grads;
size_t pmha_backward_workspace_size(const pmha_graph *graph, const pmha_params *params, int64_t batch);
pmha_status pmha_backward(const pmha_graph *graph, const pmha_params *params, const void *query,
                          const void *key, const void *value, const uint8_t *key_padding_mask,
                          int64_t batch, const void *dout, void *dquery, void *dkey, void *dvalue,
                          const pmha_grads *grads, void *workspace, size_t workspace_bytes,
                          pmha_stream stream);

/*
 * pmha_graph_export_by_source - the per-source view the backward pass walks:
 * src_row_ptr (S + 1) and, per position, its target (nnz_total), positions
 * ordered by (source, target). Device int32 buffers; NULL skips one.
 */
pmha_status pmha_graph_export_by_source(const pmha_graph *graph, int32_t *src_row_ptr, int32_t *target,
                                        pmha_stream stream);

/* Message describing the last failure of a call made by this thread ("" if none). */
const char *pmha_last_error(void);

/*
 * Stage timing. With pmha_profile_enable(1), pmha_forward / pmha_edge_weights
 * record a CUDA event pair around each kernel launch on the caller's stream.
 * pmha_profile_read() synchronizes those events and returns, per stage, the
 * number of launches and their total device time in milliseconds, then clears
 * the records. names receives up to max_stages NUL-terminated names of at
 * most 31 characters, 32 bytes apart.
 */
pmha_status pmha_profile_enable(int on);
pmha_status pmha_profile_read(int max_stages, char *names, int64_t *launches, double *total_ms,
                              int *n_stages);

/* Number of kernel launches this library queued since load (all calls, all threads). */
int64_t pmha_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PMHA_H */
