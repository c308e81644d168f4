// combine.cu -- row a5: out[t] = bf16( sum_j w[t,j] * y[t,j] + sum_s y_shared[t,s] ).
//
// Source: "vLLM Day-0 support for Recursive's Flint", "Optimisation strategy"
// (the low-latency path folds routing and the expert combine into adjacent
// kernels).  The sum runs in FP32 in a fixed order -- the routed experts in
// selection order, then the shared experts -- so the output is deterministic,
// and is rounded once to BF16 (round to nearest even).
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) combine_kernel(DevLayer d, int T,
                                                           __nv_bfloat16 *__restrict__ out,
                                                           int *__restrict__ ids_out,
                                                           float *__restrict__ w_out) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.y;
    const int K = d.k, P = d.k + d.S;
    const int m4 = blockIdx.x * kThreads + threadIdx.x;      // float4 index along H
    if (blockIdx.x == 0 && threadIdx.x < K) {
        if (ids_out) ids_out[t * K + threadIdx.x] = __ldcg(d.ids + t * K + threadIdx.x);
        if (w_out) w_out[t * K + threadIdx.x] = __ldcg(d.wsel + t * K + threadIdx.x);
    }
    if (4 * m4 >= d.H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < P; ++j) {
        const int p = __ldcg(d.pair_of + t * P + j);
        const float w = j < K ? __ldcg(d.pair_w + p) : 1.0f;
        const float4 y = __ldcg(reinterpret_cast<const float4 *>(d.y_ws + (size_t)p * d.H) + m4);
        acc.x = fmaf(w, y.x, acc.x);
        acc.y = fmaf(w, y.y, acc.y);
        acc.z = fmaf(w, y.z, acc.z);
        acc.w = fmaf(w, y.w, acc.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t *>(&lo);
    v.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(out + (size_t)t * d.H + 4 * m4) = v;
}

}  // namespace

cudaError_t launch_combine(const DevLayer &d, int T, __nv_bfloat16 *out, int *ids, float *w,
                           cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((d.H / 4 + kThreads - 1) / kThreads, T);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, d, T, out, ids, w);
}

}  // namespace moe
