// route_static.cu -- moe_route_topk_static: the routing step (FP32 router GEMV,
// sigmoid top-k, normalised weights) for callers that cannot allocate device
// memory.
//
// Why it exists: the regular entry points need a handle from moe_init, which
// calls cudaMalloc for the repacked weights and a per-handle workspace.  Some
// callers cannot do that at the point where they route tokens -- an engine
// that has already handed all free device memory to its KV cache, code that
// runs under an allocator which forbids raw cudaMalloc/cudaFree after start-up,
// or code that must not risk the implicit device synchronisation those calls
// may cause.  This entry point allocates nothing: its scratch (the [T, E] FP32
// logits and the arrival counter of the last-block-finishes pattern) lives in
// the file-scope array below, which every GPU that loads the library holds
// until the process exits.  Limits: T <= 64 tokens, E <= 512 experts
// (128 KiB of logits).
//
// The array is shared by every call on a device and keeps the last call's
// contents.  The arrival counter is cleared (cudaMemsetAsync on the array's
// device address, no allocation) before every launch.  Two calls whose kernels
// may overlap on the GPU -- different streams, or different host threads on
// one device -- race on the array: order them on one stream.
//
// Host code must not pass `g_route_scratch` itself to a kernel: in host code
// that name is only a stand-in for the symbol.  The device address is looked
// up once per device with cudaGetSymbolAddress, with that device current, on
// the first call made on that device; make that first call before any stream
// capture begins.
#include <mutex>
#include <string>

#include "moe_internal.cuh"

namespace moe {
void record_error(const std::string &msg);
}

namespace {

constexpr int kStaticMaxTokens = 64;
constexpr int kStaticMaxExperts = 512;
constexpr size_t kLogitBytes = (size_t)kStaticMaxTokens * kStaticMaxExperts * sizeof(float);
constexpr size_t kScratchBytes = kLogitBytes + 256;          // logits, then the counter

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kTokGroup = 8;
constexpr int kMaxDevices = 64;

// Ranking on logit_key(logit): larger first, the lower id on equal keys.
__device__ __forceinline__ bool ranks_before(unsigned s, int e, unsigned bs, int be) {
    return s > bs || (s == bs && e < be);
}

// One warp per expert computes its logits for all tokens; the block that
// arrives last selects the top-k of every token.
__global__ void __launch_bounds__(kThreads)
route_static_kernel(const float *__restrict__ Wr, const float *__restrict__ bias, int E, int H, int K,
                    int normalize, float routed_scale, const __nv_bfloat16 *__restrict__ x, int T,
                    int *__restrict__ ids_out, float *__restrict__ w_out, unsigned char *scratch) {
    float *logits = reinterpret_cast<float *>(scratch);
    unsigned *counter = reinterpret_cast<unsigned *>(scratch + kLogitBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kWarps + warp;
    const int nvec = H / 4;

    if (e < E) {
        const float *wr = Wr + (size_t)e * H;
        const float b = bias ? bias[e] : 0.f;
        for (int t0 = 0; t0 < T; t0 += kTokGroup) {
            const int nt = min(kTokGroup, T - t0);
            float acc[kTokGroup];
#pragma unroll
            for (int t = 0; t < kTokGroup; ++t) acc[t] = 0.f;
            for (int v = lane; v < nvec; v += 32) {
                const float4 w = __ldg(reinterpret_cast<const float4 *>(wr) + v);
#pragma unroll
                for (int t = 0; t < kTokGroup; ++t) {
                    if (t < nt) {
                        const uint2 xb = __ldcg(reinterpret_cast<const uint2 *>(x + (size_t)(t0 + t) * H) + v);
                        acc[t] = fmaf(__uint_as_float(xb.x << 16), w.x, acc[t]);
                        acc[t] = fmaf(__uint_as_float(xb.x & 0xFFFF0000u), w.y, acc[t]);
                        acc[t] = fmaf(__uint_as_float(xb.y << 16), w.z, acc[t]);
                        acc[t] = fmaf(__uint_as_float(xb.y & 0xFFFF0000u), w.w, acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kTokGroup; ++t) {
                float a = acc[t];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
                if (lane == 0 && t < nt) logits[(size_t)(t0 + t) * E + e] = a + b;
            }
        }
    }

    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(counter, 1u) == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    for (int t = warp; t < T; t += kWarps) {
        unsigned sc[kStaticMaxExperts / 32];
#pragma unroll
        for (int m = 0; m < kStaticMaxExperts / 32; ++m) {
            const int ee = lane + 32 * m;
            sc[m] = ee < E ? moe::logit_key(__ldcg(logits + (size_t)t * E + ee)) : 0u;
        }
        unsigned taken = 0u;
        unsigned sel_k = 0u;
        int sel_e = 0;
        for (int j = 0; j < K; ++j) {
            unsigned bs = 0u;
            int be = 0x7fffffff;
#pragma unroll
            for (int m = 0; m < kStaticMaxExperts / 32; ++m) {
                const int ee = lane + 32 * m;
                if (ee < E && !(taken & (1u << m)) && ranks_before(sc[m], ee, bs, be)) {
                    bs = sc[m];
                    be = ee;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const unsigned os = __shfl_xor_sync(0xffffffffu, bs, off);
                const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (ranks_before(os, oe, bs, be)) {
                    bs = os;
                    be = oe;
                }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            if (lane == j) {
                sel_k = bs;
                sel_e = be;
            }
        }
        const float sel_s = moe::key_score(sel_k);
        float sum = 0.f;
        for (int j = 0; j < K; ++j) sum += __shfl_sync(0xffffffffu, sel_s, j);
        if (lane < K) {
            const float w = (normalize ? sel_s / sum : sel_s) * routed_scale;
            ids_out[t * K + lane] = sel_e;
            w_out[t * K + lane] = w;
        }
    }
    if (threadIdx.x == 0) *counter = 0u;
}

std::mutex g_mu;
unsigned char *g_dev_scratch[kMaxDevices] = {};

// Device address of g_route_scratch on the current device (looked up once).
cudaError_t scratch_address(unsigned char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev_scratch[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_dev_scratch[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_dev_scratch[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_route_topk_static(const float *router_w, const float *router_b,
                                            int num_experts, int hidden, int top_k,
                                            int normalize_topk, float routed_scale, const void *x,
                                            int T, int *topk_ids, float *topk_w, void *stream) {
    std::string why;
    auto add = [&](const std::string &m) { why += (why.empty() ? "" : "; ") + m; };
    if (T < 1 || T > kStaticMaxTokens)
        add("T=" + std::to_string(T) + " outside [1, 64] (the static scratch holds 64 tokens x 512 experts)");
    if (num_experts < 1 || num_experts > kStaticMaxExperts)
        add("num_experts=" + std::to_string(num_experts) +
            " outside [1, 512] (the static scratch holds 64 tokens x 512 experts)");
    if (top_k < 1 || top_k > 8 || top_k > num_experts) add("top_k must be in [1, min(8, num_experts)]");
    if (hidden < 64 || hidden > 16384 || hidden % 64) add("hidden must be a multiple of 64 in [64, 16384]");
    if (normalize_topk != 0 && normalize_topk != 1) add("normalize_topk must be 0 or 1");
    if (!why.empty()) {
        moe::record_error(why);
        return MOE_ERR_UNSUPPORTED;
    }
    if (!router_w || !x || !topk_ids || !topk_w || ((uintptr_t)router_w & 15) || ((uintptr_t)x & 15)) {
        moe::record_error("router_w, x, topk_ids and topk_w must be non-NULL; router_w and x 16-byte aligned");
        return MOE_ERR_INVALID_ARG;
    }
    unsigned char *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(scratch + kLogitBytes, 0, sizeof(unsigned), st);
    if (e == cudaSuccess) {
        const int blocks = (num_experts + kWarps - 1) / kWarps;
        route_static_kernel<<<blocks, kThreads, 0, st>>>(router_w, router_b, num_experts, hidden, top_k,
                                                        normalize_topk, routed_scale,
                                                        static_cast<const __nv_bfloat16 *>(x), T,
                                                        topk_ids, topk_w, scratch);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        moe::record_error(std::string("moe_route_topk_static: ") + cudaGetErrorString(e));
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
