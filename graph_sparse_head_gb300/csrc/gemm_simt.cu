// Projection GEMM on the CUDA cores: the float32 path, and widths the
// tensor-core kernel does not tile (E not a multiple of 128).
//
// kpnn2 PackedMultiheadAttention, Notes step 1 / step 5: each projection is an
// nn.Linear, Y = X W^T + b with W stored (out, in). Every operand is widened
// to fp32; each output element accumulates in ascending k order with fused
// multiply-adds, then adds its bias and rounds once to the output type.
#include "pmha_internal.h"

namespace pmha {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;
constexpr int TM = 4, TN = 4;  // outputs per thread; 16 x 16 threads

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v, int *err);
template <> __device__ __forceinline__ float from_f<float>(float v, int *) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v, int *) { return __float2bfloat16_rn(v); }
template <> __device__ __forceinline__ __half from_f<__half>(float v, int *err)
{
    if (!(fabsf(v) <= 65504.f)) atomicOr(err, kErrRangeBit);
    return __float2half_rn(v);
}

struct SimtArgs {
    const void *X;
    const void *w[3];
    const void *b[3];
    void *Y;
    int64_t M, E, N, ldy;
    int *err;
};

template <typename TX, typename TW, typename TY>
__global__ void __launch_bounds__(256) k_gemm_simt(SimtArgs a)
{
    __shared__ float xs[BK][BM + 1];
    __shared__ float ws[BK][BN + 1];
    const TX *X = (const TX *)a.X;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int64_t m0 = (int64_t)blockIdx.x * BM, n0 = (int64_t)blockIdx.y * BN;
    const int64_t K = a.E;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    for (int64_t k0 = 0; k0 < K; k0 += BK) {
        for (int idx = threadIdx.x; idx < BM * BK; idx += 256) {
            const int r = idx / BK, c = idx % BK;
            const int64_t m = m0 + r, k = k0 + c;
            xs[c][r] = (m < a.M && k < K) ? to_f<TX>(X[m * K + k]) : 0.f;
        }
        for (int idx = threadIdx.x; idx < BN * BK; idx += 256) {
            const int r = idx / BK, c = idx % BK;
            const int64_t n = n0 + r, k = k0 + c;
            float v = 0.f;
            if (n < a.N && k < K) {
                const int seg = (int)(n / a.E);
                const TW *W = (const TW *)a.w[seg];
                v = to_f<TW>(W[(n - seg * a.E) * K + k]);
            }
            ws[c][r] = v;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float xv[TM], wv[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) xv[i] = xs[kk][ty * TM + i];
#pragma unroll
            for (int j = 0; j < TN; ++j) wv[j] = ws[kk][tx * TN + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(xv[i], wv[j], acc[i][j]);
        }
        __syncthreads();
    }
    TY *Y = (TY *)a.Y;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t m = m0 + ty * TM + i;
        if (m >= a.M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int64_t n = n0 + tx * TN + j;
            if (n >= a.N) continue;
            const int seg = (int)(n / a.E);
            float v = acc[i][j];
            if (a.b[seg]) v = __fadd_rn(v, to_f<TW>(((const TW *)a.b[seg])[n - seg * a.E]));
            Y[m * a.ldy + n] = from_f<TY>(v, a.err);
        }
    }
}

__global__ void k_bf16_to_f16(const __nv_bfloat16 *__restrict__ src, __half *__restrict__ dst, int64_t n, int *err)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const float v = __bfloat162float(src[i]);
        if (!(fabsf(v) <= 65504.f)) atomicOr(err, kErrRangeBit);
        dst[i] = __float2half_rn(v);
    }
}

}  // namespace

pmha_status gemm_simt(TcType tx, TcType tw, TcType ty, const void *X, int64_t M, int64_t E, const GemmSegments &seg,
                      void *Y, int64_t ldy, const char *stage, cudaStream_t stream)
{
    SimtArgs a;
    a.X = X;
    for (int i = 0; i < 3; ++i) {
        a.w[i] = i < seg.n_seg ? seg.w[i] : nullptr;
        a.b[i] = i < seg.n_seg ? seg.b[i] : nullptr;
    }
    a.Y = Y;
    a.M = M;
    a.E = E;
    a.N = E * seg.n_seg;
    a.ldy = ldy;
    a.err = device_error_word();
    if (!a.err) return PMHA_ERR_CUDA;
    dim3 grid((unsigned)((M + BM - 1) / BM), (unsigned)((a.N + BN - 1) / BN));
    if (grid.y > 65535u) {
        set_error("gemm_simt: %lld output columns exceed the grid limit", (long long)a.N);
        return PMHA_ERR_UNSUPPORTED;
    }
    StageTimer timer(stage, stream);
    if (tx == TcType::F32 && tw == TcType::F32 && ty == TcType::F32)
        k_gemm_simt<float, float, float><<<grid, 256, 0, stream>>>(a);
    else if (tx == TcType::BF16 && tw == TcType::BF16 && ty == TcType::F16)
        k_gemm_simt<__nv_bfloat16, __nv_bfloat16, __half><<<grid, 256, 0, stream>>>(a);
    else if (tx == TcType::F16 && tw == TcType::BF16 && ty == TcType::BF16)
        k_gemm_simt<__half, __nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, stream>>>(a);
    else {
        set_error("gemm_simt: no kernel for this type combination");
        return PMHA_ERR_UNSUPPORTED;
    }
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

pmha_status convert_bf16_to_f16(const void *src, void *dst, int64_t n, cudaStream_t stream)
{
    int *err = device_error_word();
    if (!err) return PMHA_ERR_CUDA;
    const int TB = 256;
    StageTimer timer("convert_wo", stream);
    k_bf16_to_f16<<<(unsigned)((n + TB - 1) / TB), TB, 0, stream>>>((const __nv_bfloat16 *)src, (__half *)dst, n, err);
    count_launch();
    PMHA_CUDA_TRY(cudaGetLastError());
    return PMHA_OK;
}

}  // namespace pmha
