// route.cu -- rows a1 + a2: FP32 router GEMV, sigmoid, top-k with
// lowest-index tie-break, weight normalisation, and the work list of the
// distinct selected experts.
//
// Sources: "Inkling 2 Small on vLLM: Day-0 Support", "Accuracy evaluation"
// (the router runs in FP32); "Day 0 support for Mistral Large 4 on vLLM",
// "Breakable CUDA graphs and fusions" (FP32 routing GEMM);
// "vLLM Day-0 support for Recursive's Flint", "Flint model architecture"
// (sigmoid top-6 over 256 experts plus one shared expert) and "Optimisation
// strategy" (the expert GEMVs read only the selected experts, which is what the
// work list built here enables).
//
// One launch.  Each warp computes one expert's logits for every token (the
// router row is streamed once with 16-byte loads; the first part is fetched
// before the programmatic-launch wait because router weights do not depend on
// the previous kernel).  The CTA that finishes last (atomic ticket, no
// spinning) then runs sigmoid/top-k per token (one warp per token), counts the
// tokens per expert with 64-bit token masks, scans them into slots (shared
// experts first, then routed experts in ascending id) and numbers the
// (expert, token) pairs so that each expert's pairs are contiguous.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kThreads = 32 * kRouteWarps;
constexpr int kTokGroup = 8;
constexpr int kPre = 16;    // float4 per lane fetched before the wait (2048 K)

__device__ __forceinline__ void bf16x4_to_f(uint2 v, float &a, float &b, float &c, float &e) {
    a = __uint_as_float(v.x << 16);
    b = __uint_as_float(v.x & 0xFFFF0000u);
    c = __uint_as_float(v.y << 16);
    e = __uint_as_float(v.y & 0xFFFF0000u);
}

__device__ __forceinline__ void dot4_tokens(const float4 &w, const __nv_bfloat16 *__restrict__ x,
                                            int H, int t0, int nt, int v, float (&acc)[kTokGroup]) {
#pragma unroll
    for (int t = 0; t < kTokGroup; ++t) {
        if (t < nt) {
            uint2 xb = __ldcg(reinterpret_cast<const uint2 *>(x + (size_t)(t0 + t) * H + 4 * v));
            float x0, x1, x2, x3;
            bf16x4_to_f(xb, x0, x1, x2, x3);
            acc[t] = fmaf(x0, w.x, acc[t]);
            acc[t] = fmaf(x1, w.y, acc[t]);
            acc[t] = fmaf(x2, w.z, acc[t]);
            acc[t] = fmaf(x3, w.w, acc[t]);
        }
    }
}

__device__ __forceinline__ bool better(float s, int e, float bs, int be) {
    return s > bs || (s == bs && e < be);
}

__global__ void __launch_bounds__(kThreads) route_kernel(DevLayer d,
                                                         const __nv_bfloat16 *__restrict__ x, int T) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = d.H, E = d.E, K = d.k, S = d.S;
    const int e = blockIdx.x * kRouteWarps + warp;
    const int nvec = H / 4;
    const float *wr = d.router_w + (size_t)(e < E ? e : 0) * H;

    float4 pre[kPre];
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
        int v = lane + 32 * j;
        pre[j] = (e < E && v < nvec) ? ld_f4(wr + 4 * v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();
    pdl_trigger();

    if (e < E) {
        const float bias = d.router_b ? d.router_b[e] : 0.f;
        for (int t0 = 0; t0 < T; t0 += kTokGroup) {
            const int nt = min(kTokGroup, T - t0);
            float acc[kTokGroup];
#pragma unroll
            for (int t = 0; t < kTokGroup; ++t) acc[t] = 0.f;
#pragma unroll
            for (int j = 0; j < kPre; ++j) {
                int v = lane + 32 * j;
                if (v < nvec) dot4_tokens(pre[j], x, H, t0, nt, v, acc);
            }
            for (int v = lane + 32 * kPre; v < nvec; v += 32)
                dot4_tokens(ld_f4(wr + 4 * v), x, H, t0, nt, v, acc);
#pragma unroll
            for (int t = 0; t < kTokGroup; ++t) {
                float a = acc[t];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
                if (lane == 0 && t < nt) d.logits[(size_t)(t0 + t) * E + e] = a + bias;
            }
        }
    }

    // ---- last CTA to finish builds the routing result and the work list ----
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned tk = atomicAdd(d.ticket, 1u);
        s_last = (tk == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    __shared__ int s_ids[kMaxTokens][kMaxTopK];
    __shared__ float s_w[kMaxTokens][kMaxTopK];
    __shared__ unsigned long long s_mask[kMaxExperts];
    __shared__ int s_pbase[kMaxExperts];
    __shared__ int s_wsum_f[kRouteWarps], s_wsum_c[kRouteWarps];

    for (int i = threadIdx.x; i < E; i += kThreads) s_mask[i] = 0ull;
    __syncthreads();

    // a2: sigmoid + top-k + weights, one warp per token.
    for (int t = warp; t < T; t += kRouteWarps) {
        float sc[kMaxExperts / 32];
#pragma unroll
        for (int m = 0; m < kMaxExperts / 32; ++m) {
            int ee = lane + 32 * m;
            float s = -INFINITY;
            if (ee < E) {
                float z = __ldcg(d.logits + (size_t)t * E + ee);
                s = isnan(z) ? -INFINITY : 1.0f / (1.0f + expf(-z));
            }
            sc[m] = s;
        }
        unsigned taken = 0u;
        float sel_s = 0.f;
        int sel_e = 0;
        for (int j = 0; j < K; ++j) {
            float bs = -INFINITY;
            int be = 0x7fffffff;
#pragma unroll
            for (int m = 0; m < kMaxExperts / 32; ++m) {
                int ee = lane + 32 * m;
                if (ee < E && !(taken & (1u << m)) && better(sc[m], ee, bs, be)) {
                    bs = sc[m];
                    be = ee;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                float os = __shfl_xor_sync(0xffffffffu, bs, off);
                int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (better(os, oe, bs, be)) {
                    bs = os;
                    be = oe;
                }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            if (lane == j) {
                sel_s = bs;
                sel_e = be;
            }
        }
        // weights: normalised over the k selected scores (summed in selection order)
        float sum = 0.f;
        for (int j = 0; j < K; ++j) sum += __shfl_sync(0xffffffffu, sel_s, j);
        if (lane < K) {
            float w = d.normalize ? sel_s / sum : sel_s;
            w *= d.routed_scale;
            s_ids[t][lane] = sel_e;
            s_w[t][lane] = w;
            d.ids[(size_t)t * K + lane] = sel_e;
            d.wsel[(size_t)t * K + lane] = w;
            atomicOr(&s_mask[sel_e], 1ull << t);
        }
    }
    __syncthreads();

    // Slots: shared experts first, then routed experts with >= 1 token in
    // ascending id.  Exclusive scans of (used?, token count) over experts.
    const int per = (E + kThreads - 1) / kThreads;
    const int e0 = threadIdx.x * per;
    int fsum = 0, csum = 0;
    for (int i = 0; i < per; ++i) {
        int ee = e0 + i;
        if (ee < E) {
            int c = __popcll(s_mask[ee]);
            fsum += c > 0;
            csum += c;
        }
    }
    int finc = fsum, cinc = csum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int a = __shfl_up_sync(0xffffffffu, finc, off);
        int b = __shfl_up_sync(0xffffffffu, cinc, off);
        if (lane >= off) {
            finc += a;
            cinc += b;
        }
    }
    if (lane == 31) {
        s_wsum_f[warp] = finc;
        s_wsum_c[warp] = cinc;
    }
    __syncthreads();
    int fbase = finc - fsum, cbase = cinc - csum;
    for (int w = 0; w < warp; ++w) {
        fbase += s_wsum_f[w];
        cbase += s_wsum_c[w];
    }
    for (int i = 0; i < per; ++i) {
        int ee = e0 + i;
        if (ee < E) {
            int c = __popcll(s_mask[ee]);
            if (c > 0) {
                int slot = S + fbase;
                int p0 = S * T + cbase;
                d.slot_expert[slot] = ee;
                d.slot_m[slot] = c;
                d.slot_p0[slot] = p0;
                s_pbase[ee] = p0;
                fbase += 1;
                cbase += c;
            }
        }
    }
    if (threadIdx.x == kThreads - 1) *d.nslots = S + fbase;   // last thread: total U
    if (threadIdx.x < S) {
        d.slot_expert[threadIdx.x] = -(threadIdx.x + 1);
        d.slot_m[threadIdx.x] = T;
        d.slot_p0[threadIdx.x] = threadIdx.x * T;
    }
    __syncthreads();

    // Pairs: an expert's tokens are numbered in ascending token order.
    const int P = K + S;
    for (int it = threadIdx.x; it < T * K; it += kThreads) {
        int t = it / K, j = it % K;
        int ee = s_ids[t][j];
        unsigned long long below = (t == 0) ? 0ull : (s_mask[ee] & ((1ull << t) - 1ull));
        int p = s_pbase[ee] + __popcll(below);
        d.pair_tok[p] = t;
        d.pair_w[p] = s_w[t][j];
        d.pair_of[t * P + j] = p;
    }
    for (int it = threadIdx.x; it < T * S; it += kThreads) {
        int sidx = it / T, t = it % T;
        int p = sidx * T + t;
        d.pair_tok[p] = t;
        d.pair_w[p] = 1.0f;
        d.pair_of[t * P + K + sidx] = p;
    }
    for (int p = threadIdx.x; p < T * P; p += kThreads) d.hmax[p] = 0u;

    // Power-of-two prescale of each activation row so that it fits the f16
    // operands of the expert GEMVs exactly: max|x| * 2^-xexp < 2^15.
    for (int t = warp; t < T; t += kRouteWarps) {
        float mx = 0.f;
        for (int v = lane; v < nvec; v += 32) {
            uint2 xb = __ldcg(reinterpret_cast<const uint2 *>(x + (size_t)t * H + 4 * v));
            float a, b, c, f;
            bf16x4_to_f(xb, a, b, c, f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(a), fabsf(b)), fmaxf(fabsf(c), fabsf(f))));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) {
            int ex = 0;
            if (mx > 0.f && isfinite(mx)) ex = max(0, ilogbf(mx) - 14);
            d.xexp[t] = ex;
        }
    }
    if (threadIdx.x == 0) *d.ticket = 0u;
}

}  // namespace

cudaError_t launch_route(const DevLayer &d, const __nv_bfloat16 *x, int T, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((d.E + kRouteWarps - 1) / kRouteWarps);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_kernel, d, x, T);
}

}  // namespace moe
