// route.cu -- rows a1 + a2: FP32 router GEMV, sigmoid (or softmax) scores,
// top-k with lowest-index tie-break, weight normalisation, and the work list of
// the distinct selected experts (the three-kernel chain; the single launch has
// its own copy of these steps, sigmoid only).
//
// Sources: "Inkling 2 Small on vLLM: Day-0 Support", "Accuracy evaluation"
// (the router runs in FP32); "Day 0 support for Mistral Large 4 on vLLM",
// "Breakable CUDA graphs and fusions" (FP32 routing GEMM);
// "Day 0 support for Mistral Large 4 on vLLM", "Specialized decode" (its
// fused layer runs a softmax top-4 router);
// "vLLM Day-0 support for Recursive's Flint", "Flint model architecture"
// (sigmoid top-6 over 256 experts plus one shared expert) and "Optimisation
// strategy" (the expert GEMVs read only the selected experts, which is what the
// work list built here enables).
//
// Grid: (E/8 expert groups) x (token groups of up to 8 tokens) x (K ranges:
// the router rows are split along H until the grid covers the SMs).  A
// block's threads form two halves of four experts; a thread takes 4-column
// groups of the K range for its half's four experts, whose router columns it
// fetches into registers BEFORE the programmatic-launch wait (router weights
// do not depend on the previous kernel).  The block stages its token group's
// activation columns in shared memory (BF16, by asynchronous copies) and each
// x group a thread reads there serves four experts' FP32 partial logits (one
// accumulator per expert and token, so the FMA chains run side by side); a
// transposing butterfly and a fixed-order sum over a half's warps give the
// logits.  With several K ranges the partial sums go to the
// workspace and the ticket's last block adds them in a fixed order, into
// shared memory.  Two tickets follow, with no spinning:
//   * the last expert group of a token group to finish runs the scores and
//     top-k for those tokens (one warp per token) and ORs each token into a
//     64-bit mask per selected expert;
//   * the last token group to finish turns the masks into slots (shared
//     experts first, then routed experts in ascending id), numbers the
//     (expert, token) pairs so that each expert's pairs are contiguous, lists
//     the slots with many tokens for the grouped kernels, and clears the masks.
// With a single token group the first ticket's last block is also the last
// overall: it keeps the choices and masks in shared memory and skips the
// second ticket.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kThreads = 32 * kRouteWarps;
constexpr int kTokGroup = 8;
constexpr int kEPT = 4;                                  // experts per thread (a block half's)
constexpr int kRouteHalfWarps = kRouteWarps / 2;
constexpr int kHalfThreads = 32 * kRouteHalfWarps;
constexpr int kPre = 4;     // 4-column groups per thread fetched before the wait (2048 K)
static_assert(kRouteWarps == 2 * kEPT, "two halves of four experts");

// 16-byte asynchronous copy global -> shared (L2 only)
__device__ __forceinline__ void cp_async16_cg(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(__cvta_generic_to_global(src))
                 : "memory");
}

__device__ __forceinline__ void bf16x4_to_f(uint2 v, float &a, float &b, float &c, float &e) {
    a = __uint_as_float(v.x << 16);
    b = __uint_as_float(v.x & 0xFFFF0000u);
    c = __uint_as_float(v.y << 16);
    e = __uint_as_float(v.y & 0xFFFF0000u);
}

// Top-k of one token's FP32 logits (lane L holds experts i * 32 + L, i < M)
// by sort keys; lane j < k returns the j-th choice.
template <int M>
__device__ __forceinline__ unsigned long long token_topk(const float *z, bool in_smem, int E, int K, int lane) {
    unsigned long long c[M];
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const int e = i * 32 + lane;
        c[i] = e < E ? ((unsigned long long)logit_key(in_smem ? z[e] : __ldcg(z + e)) << 32) | (unsigned)~e : 0ull;
    }
    if constexpr (M <= 8) return warp_topk_sorted<M>(c, K, lane);
    else return warp_topk_tree<M>(c, K, lane);
}

// Softmax denominator of one token relative to its largest logit z0: the sum
// over all experts of exp(z_e - z0), lane-strided, then across the warp; every
// lane gets lane 0's total.
__device__ __forceinline__ float softmax_den(const float *z, bool in_smem, int E, float z0, int lane) {
    float acc = 0.f;
    for (int e = lane; e < E; e += 32) acc += expf((in_smem ? z[e] : __ldcg(z + e)) - z0);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    return __shfl_sync(0xffffffffu, acc, 0);
}

__global__ void __launch_bounds__(kThreads) route_kernel(DevLayer d, const __nv_bfloat16 *__restrict__ x,
                                                         int T, int tg, int *__restrict__ ids_out,
                                                         float *__restrict__ w_out) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = d.H, E = d.E, K = d.k, S = d.S;
    // this block's experts: e0 .. e0 + kRouteWarps - 1
    const int e0 = blockIdx.x * kRouteWarps;
    // K split: block z takes columns [k0, k0 + Hk) of the router rows
    const int KH = gridDim.z, Hk = H / KH, k0 = blockIdx.z * Hk;
    const int nvec = Hk / 4;
    const int t0 = blockIdx.y * tg, nt = min(tg, T - t0);

    MOE_TRACE_POINT(0, 0);
    // The block's threads form two halves (warps 0-3 and 4-7), half h taking
    // experts e0 + 4h .. e0 + 4h + 3; thread i of a half takes the 4-column
    // groups v = i + 128 j of the K range for its four experts, so that each
    // x group it reads from shared memory serves four experts.  The first
    // kPre groups' router columns are loaded before the dependency wait.
    const int half = warp / kRouteHalfWarps, hi_ = threadIdx.x % (32 * kRouteHalfWarps);
    const int eh = e0 + kEPT * half;
    float4 pre[kPre][kEPT];
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
        const int v = hi_ + kHalfThreads * j;
#pragma unroll
        for (int i = 0; i < kEPT; ++i) {
            if (eh + i < E && v < nvec) {
                // volatile loads: issued here, before the wait, not sunk past it
                const float *wr = d.router_w + (size_t)(eh + i) * H + k0 + 4 * v;
                const float2 lo = ld_nc_f2(wr), hi = ld_nc_f2(wr + 2);
                pre[j][i] = make_float4(lo.x, lo.y, hi.x, hi.y);
            } else {
                pre[j][i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    pdl_wait();
    pdl_trigger();
    MOE_TRACE_POINT(0, 1);

    // ---- stage the token group's activation columns [k0, k0 + Hk) (16-byte
    // loads, all in flight) ----
    __shared__ float s_rmax[kTokGroup];
    if (threadIdx.x < kTokGroup) s_rmax[threadIdx.x] = 0.f;
    // x columns as BF16, copied by 16-byte asynchronous copies (all in
    // flight, no register round trip); the dot products below unpack them
    const uint2 *xs = reinterpret_cast<const uint2 *>(smem);   // [nt][Hk/4] groups of four
    {
        const int r16 = Hk / 8, n16 = nt * r16;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t0 * H + k0);
#pragma unroll 4
        for (int i = threadIdx.x; i < n16; i += kThreads)
            cp_async16_cg(smem + (size_t)16 * i, src + (size_t)(i / r16) * (H / 8) + i % r16);
        asm volatile("cp.async.wait_all;\n" ::: "memory");
        __syncthreads();
        if (blockIdx.x == 0) {
            // per-token max |x| for the GEMVs' power-of-two prescale
            // (non-negative, so its bits order as unsigned integers)
#pragma unroll 1
            for (int i0 = 0; i0 < n16; i0 += kThreads) {
                const int i = i0 + threadIdx.x;
                float m = 0.f;
                if (i < n16) {
                    const uint4 v = reinterpret_cast<const uint4 *>(smem)[i];
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[q] << 16)),
                                           fabsf(__uint_as_float(w4[q] & 0xFFFF0000u))));
                }
                if ((r16 & 31) == 0) {
                    // a warp's 32 pieces are one token's (and all in range or
                    // all out): one shared atomic per warp
                    const unsigned mw = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
                    if (lane == 0 && i < n16) atomicMax(reinterpret_cast<unsigned *>(&s_rmax[i / r16]), mw);
                } else if (i < n16) {
                    atomicMax(reinterpret_cast<unsigned *>(&s_rmax[i / r16]), __float_as_uint(m));
                }
            }
            __syncthreads();
        }
    }
    MOE_TRACE_POINT(0, 2);
    if (blockIdx.x == 0 && threadIdx.x < nt) {
        // this K range's max; the exponent is taken from the whole row below
        atomicMax(d.xmaxb + t0 + threadIdx.x, __float_as_uint(s_rmax[threadIdx.x]));
    }
    // ---- logits of the group's tokens for the block's experts ----
    {
        // acc[i][t]: expert eh + i, token t0 + t, over this thread's columns
        float acc[kEPT][kTokGroup];
#pragma unroll
        for (int i = 0; i < kEPT; ++i)
#pragma unroll
            for (int t = 0; t < kTokGroup; ++t) acc[i][t] = 0.f;
        auto group = [&](int v, const float4 (&w)[kEPT]) {
#pragma unroll
            for (int t = 0; t < kTokGroup; ++t) {
                if (t < nt) {
                    float4 xv;
                    bf16x4_to_f(xs[t * nvec + v], xv.x, xv.y, xv.z, xv.w);
#pragma unroll
                    for (int i = 0; i < kEPT; ++i)
                        acc[i][t] = fmaf(xv.w, w[i].w, fmaf(xv.z, w[i].z, fmaf(xv.y, w[i].y, fmaf(xv.x, w[i].x, acc[i][t]))));
                }
            }
        };
#pragma unroll
        for (int j = 0; j < kPre; ++j) {
            const int v = hi_ + kHalfThreads * j;
            if (v < nvec) group(v, pre[j]);
        }
        // the rest of a longer K range, one column group at a time
#pragma unroll 1
        for (int v = hi_ + kHalfThreads * kPre; v < nvec; v += kHalfThreads) {
            float4 w[kEPT];
#pragma unroll
            for (int i = 0; i < kEPT; ++i)
                w[i] = eh + i < E ? ld_f4(d.router_w + (size_t)(eh + i) * H + k0 + 4 * v) : make_float4(0.f, 0.f, 0.f, 0.f);
            group(v, w);
        }
        MOE_TRACE_POINT(0, 8);
        // warp sums of the 32 values by a transposing butterfly: at the step
        // of distance w every lane keeps the half of its values selected by
        // bit w of its lane index and adds the partner's copy of that half;
        // lane L ends with value L (expert eh + L / 8, token L % 8)
        float *s_part = reinterpret_cast<float *>(smem + (size_t)nt * nvec * 8);   // [kRouteWarps][32]
        static_assert(kEPT * kTokGroup == 32, "one value per lane");
        {
            float a[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) a[u] = acc[u / kTokGroup][u % kTokGroup];
#pragma unroll
            for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
                for (int u = 0; u < w; ++u) {
                    const bool up = (lane & w) != 0;
                    const float send = up ? a[u] : a[u + w];
                    const float keep = up ? a[u + w] : a[u];
                    a[u] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                }
            }
            s_part[warp * 32 + lane] = a[0];
        }
        __syncthreads();
        if (threadIdx.x < kRouteWarps * kTokGroup) {
            // the sums of a half's warps in a fixed order
            const int i = threadIdx.x / kTokGroup, t = threadIdx.x % kTokGroup, e = e0 + i;
            const int h = i / kEPT, u = (i % kEPT) * kTokGroup + t;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kRouteHalfWarps; ++w) v += s_part[(h * kRouteHalfWarps + w) * 32 + u];
            if (e < E && t < nt) {
                if (KH == 1) d.logits[(size_t)(t0 + t) * E + e] = v + (d.router_b ? d.router_b[e] : 0.f);
                else d.lpart[((size_t)blockIdx.z * d.max_tokens + t0 + t) * E + e] = v;
            }
        }
    }

    // ---- the last expert group of this token group: top-k of its tokens ----
    __shared__ int s_last;
    __shared__ int s_ids[kMaxTokens][kMaxTopK];
    __shared__ float s_w[kMaxTokens][kMaxTopK];
    __shared__ unsigned long long s_mask[kMaxExperts];
    __syncthreads();
    MOE_TRACE_POINT(0, 3);
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(d.tg_ticket + blockIdx.y, 1u) == gridDim.x * gridDim.z - 1;
    }
    MOE_TRACE_POINT(0, 9);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // With one token group this block is also the last one overall: the
    // choices and the expert masks stay in shared memory (no second ticket).
    const bool one = gridDim.y == 1;
    if (one)
        for (int i = threadIdx.x; i < E; i += kThreads) s_mask[i] = 0ull;
    float *s_lg = reinterpret_cast<float *>(smem);   // [nt][E]: x is no longer read
    if (KH > 1) {
        // the token group's logits: the K ranges' sums in a fixed order; kept
        // in shared memory for the top-k below.  One block reads all the
        // partials, so the number of requests sets the time: four experts
        // per 16-byte load when E allows, a thread's items kLgBatch at a time
        // with all their partial loads in flight together.
        if ((E & 3) == 0) {
            constexpr int kLgBatch = 2;
            const int nq = nt * E / 4;
            const float4 *lp = reinterpret_cast<const float4 *>(d.lpart);
#pragma unroll 1
            for (int i0 = 0; i0 < nq; i0 += kLgBatch * kThreads) {
                float4 part[kLgBatch][kMaxKSplit];
#pragma unroll
                for (int r = 0; r < kLgBatch; ++r) {
                    const int i = i0 + r * kThreads + threadIdx.x;
                    const int t = (4 * i) / E, e4 = 4 * i - t * E;
#pragma unroll
                    for (int z = 0; z < kMaxKSplit; ++z)
                        part[r][z] = (z < KH && i < nq)
                                         ? __ldcg(lp + (((size_t)z * d.max_tokens + t0 + t) * E + e4) / 4)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int r = 0; r < kLgBatch; ++r) {
                    const int i = i0 + r * kThreads + threadIdx.x;
                    if (i < nq) {
                        const int t = (4 * i) / E, e4 = 4 * i - t * E;
                        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int z = 0; z < kMaxKSplit; ++z)
                            if (z < KH) {
                                v[0] += part[r][z].x;
                                v[1] += part[r][z].y;
                                v[2] += part[r][z].z;
                                v[3] += part[r][z].w;
                            }
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            v[u] += d.router_b ? d.router_b[e4 + u] : 0.f;
                            s_lg[4 * i + u] = v[u];
                        }
                        *reinterpret_cast<float4 *>(d.logits + (size_t)(t0 + t) * E + e4) =
                            make_float4(v[0], v[1], v[2], v[3]);
                    }
                }
            }
        } else {
            for (int i = threadIdx.x; i < nt * E; i += kThreads) {
                const int t = i / E, ee = i - t * E;
                float part[kMaxKSplit];
#pragma unroll
                for (int z = 0; z < kMaxKSplit; ++z)
                    part[z] = z < KH ? __ldcg(d.lpart + ((size_t)z * d.max_tokens + t0 + t) * E + ee) : 0.f;
                float v = 0.f;
#pragma unroll
                for (int z = 0; z < kMaxKSplit; ++z)
                    if (z < KH) v += part[z];
                v += d.router_b ? d.router_b[ee] : 0.f;
                s_lg[i] = v;
                d.logits[(size_t)(t0 + t) * E + ee] = v;
            }
        }
    }
    __syncthreads();
    MOE_TRACE_POINT(0, 4);
    if (warp < nt) {
        // sort keys logit_key(logit) << 32 | ~id: larger is better, equal
        // logits go to the lower id; lane j < k ends with the j-th choice
        const int t = t0 + warp;
        const bool lsm = KH > 1;
        const float *zt = lsm ? s_lg + (size_t)warp * E : d.logits + (size_t)t * E;
        unsigned long long sel;
        switch (d.E <= 32 ? 1 : d.E <= 64 ? 2 : d.E <= 128 ? 4 : d.E <= 256 ? 8 : 16) {
            case 1: sel = token_topk<1>(zt, lsm, E, K, lane); break;
            case 2: sel = token_topk<2>(zt, lsm, E, K, lane); break;
            case 4: sel = token_topk<4>(zt, lsm, E, K, lane); break;
            case 8: sel = token_topk<8>(zt, lsm, E, K, lane); break;
            default: sel = token_topk<16>(zt, lsm, E, K, lane); break;
        }
        MOE_TRACE_POINT(0, 10);
        const unsigned sel_key = (unsigned)(sel >> 32);
        const int sel_e = (int)~(unsigned)sel;
        // the choices' scores: the sigmoid of the logit, or (softmax routing)
        // its exponential relative to the largest logit, lane 0's choice
        const bool smax = d.score_func == 1;
        const float zsel = key_logit(sel_key);
        const float z0 = __shfl_sync(0xffffffffu, zsel, 0);
        const float sel_s = smax ? expf(zsel - z0) : key_score(sel_key);
        // weights: normalised over the k selected scores (summed in selection
        // order); softmax scores without normalisation are divided by the sum
        // over all experts
        float sum = 0.f;
        for (int j = 0; j < K; ++j) sum += __shfl_sync(0xffffffffu, sel_s, j);
        const float den = smax && !d.normalize ? softmax_den(zt, lsm, E, z0, lane) : 1.f;
        if (lane < K) {
            const float w = (d.normalize ? sel_s / sum : sel_s / den) * d.routed_scale;
            d.ids[(size_t)t * K + lane] = sel_e;
            d.wsel[(size_t)t * K + lane] = w;
            if (ids_out) ids_out[(size_t)t * K + lane] = sel_e;
            if (w_out) w_out[(size_t)t * K + lane] = w;
            if (one) {
                s_ids[t][lane] = sel_e;
                s_w[t][lane] = w;
                atomicOr(s_mask + sel_e, 1ull << t);
            } else {
                atomicOr(d.emask + sel_e, 1ull << t);
            }
        }
    }
    // this token group's power-of-two prescales from their whole-row maxima
    // (every block of the group has added its part before the ticket above);
    // with W4A4 the quantiser, running beside this kernel, writes them from
    // the quantised rows
    if (threadIdx.x < nt) {
        const int t = t0 + threadIdx.x;
        if (!d.w4a4) d.xexp[t] = max(-100, exp_for_f16(__uint_as_float(__ldcg(d.xmaxb + t))));
        d.xmaxb[t] = 0u;
    }
    MOE_TRACE_POINT(0, 11);
    // ---- the last token group: slots, pairs, hot list ----
    __syncthreads();
    if (!one) {
        if (threadIdx.x == 0) {
            d.tg_ticket[blockIdx.y] = 0u;
            __threadfence();
            s_last = atomicAdd(d.ticket, 1u) == gridDim.y - 1;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
    } else if (threadIdx.x == 0) {
        d.tg_ticket[0] = 0u;
    }
    MOE_TRACE_POINT(0, 5);

    __shared__ int s_pbase[kMaxExperts];
    __shared__ int s_wsum_f[kRouteWarps], s_wsum_c[kRouteWarps];
    __shared__ short s_slotm[kMaxTokens * kMaxTopK + kMaxShared];   // tokens per slot
    if (!one) {
        for (int i = threadIdx.x; i < E; i += kThreads) {
            s_mask[i] = __ldcg(d.emask + i);
            d.emask[i] = 0ull;
        }
        for (int i = threadIdx.x; i < T * K; i += kThreads) {
            s_ids[i / K][i % K] = __ldcg(d.ids + i);
            s_w[i / K][i % K] = __ldcg(d.wsel + i);
        }
    }
    __syncthreads();
    MOE_TRACE_POINT(0, 6);
    // Slots: shared experts first, then routed experts with >= 1 token in
    // ascending id.  Exclusive scans of (used?, token count) over experts.
    const int per = (E + kThreads - 1) / kThreads;
    const int eb = threadIdx.x * per;
    int fsum = 0, csum = 0;
    for (int i = 0; i < per; ++i) {
        const int ee = eb + i;
        if (ee < E) {
            const int c = __popcll(s_mask[ee]);
            fsum += c > 0;
            csum += c;
        }
    }
    int finc = fsum, cinc = csum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, finc, off);
        const int b = __shfl_up_sync(0xffffffffu, cinc, off);
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
    MOE_TRACE_POINT(0, 12);
    int fbase = finc - fsum, cbase = cinc - csum;
    for (int w = 0; w < warp; ++w) {
        fbase += s_wsum_f[w];
        cbase += s_wsum_c[w];
    }
    for (int i = 0; i < per; ++i) {
        const int ee = eb + i;
        if (ee < E) {
            const int c = __popcll(s_mask[ee]);
            if (c > 0) {
                const int slot = S + fbase;
                const int p0 = S * T + cbase;
                d.slot_expert[slot] = ee;
                d.slot_m[slot] = c;
                d.slot_p0[slot] = p0;
                s_slotm[slot] = (short)c;
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
        s_slotm[threadIdx.x] = (short)T;
    }
    __syncthreads();
    MOE_TRACE_POINT(0, 13);
    if (warp == 0) {
        // slots with at least grouped_min tokens (in slot order) go to the
        // grouped tensor-core kernels; the GEMV kernels skip them
        int ns = S;
        for (int w = 0; w < kRouteWarps; ++w) ns += s_wsum_f[w];
        // (and the routed ones below it, which the GEMV kernels take).  Where
        // the GEMV kernels take slots of up to 15 tokens, a routed slot's
        // threshold is raised from grouped_min (up to 16) until the grouped
        // kernels' items fit one per block: their time is that of the block
        // with the most items, the GEMV kernels' units are handed out on demand.
        int tau = d.grouped_min;
        if (T > 8 && d.tau_max > d.grouped_min) {
            // routed slots by token count (counts of 16 and more together):
            // lane b < 17 ends with the number of count b.  Per 32 slots the
            // lanes of one count meet in a match and the lowest of them adds
            // them up (one writer per entry).
            __shared__ int s_hist[17];
            if (lane < 17) s_hist[lane] = 0;
            __syncwarp();
            for (int b0 = S; b0 < ns; b0 += 32) {
                const int sl = b0 + lane;
                const int m = sl < ns ? s_slotm[sl] : 0;
                const int bin = sl < ns && m >= d.grouped_min ? min(m, 16) : -1;
                const unsigned mm = __match_any_sync(0xffffffffu, bin);
                if (bin >= 0 && lane == __ffs(mm) - 1) s_hist[bin] += __popc(mm);
                __syncwarp();
            }
            const int h = lane < 17 ? s_hist[lane] : 0;
            int shot = 0;   // shared slots stay hot at grouped_min
            for (int j = 0; j < S; ++j) shot += s_slotm[j] >= d.grouped_min;
            // routed slots with at least cand tokens
            int cnt = __reduce_add_sync(0xffffffffu, lane >= d.tau_max ? h : 0);
            // from the top: the smallest threshold whose items still fit
            tau = d.tau_max;
            for (int cand = d.tau_max; cand >= d.grouped_min; --cand) {
                const long up = (long)cnt * (d.I / 64) + (long)shot * (d.Is / 64);
                const long dn = (long)(cnt + shot) * (d.H / 128);
                if (up > d.nsm || dn > d.nsm) break;
                tau = cand;
                if (cand > d.grouped_min) cnt += __shfl_sync(0xffffffffu, h, cand - 1);
            }
        }
        int nh = 0, nc = 0;
        for (int b = 0; b < ns; b += 32) {
            const int sl = b + lane;
            const bool hot = d.grouped_min > 0 && sl < ns && s_slotm[sl] >= (sl < S ? d.grouped_min : tau);
            const bool cold = sl >= S && sl < ns && !hot;
            const unsigned bal = __ballot_sync(0xffffffffu, hot);
            const unsigned bcl = __ballot_sync(0xffffffffu, cold);
            if (hot) d.hot_slots[nh + __popc(bal & ((1u << lane) - 1u))] = sl;
            if (cold) d.cold_slots[nc + __popc(bcl & ((1u << lane) - 1u))] = sl;
            nh += __popc(bal);
            nc += __popc(bcl);
        }
        if (lane == 0) {
            *d.nhot = nh;
            *d.ncold = nc;
        }
    }

    MOE_TRACE_POINT(0, 14);
    // Pairs: an expert's tokens are numbered in ascending token order.
    const int P = K + S;
    for (int it = threadIdx.x; it < T * K; it += kThreads) {
        const int t = it / K, j = it % K;
        const int ee = s_ids[t][j];
        const unsigned long long below = (t == 0) ? 0ull : (s_mask[ee] & ((1ull << t) - 1ull));
        const int p = s_pbase[ee] + __popcll(below);
        d.pair_tok[p] = t;
        d.pair_w[p] = s_w[t][j];
        d.pair_of[t * P + j] = p;
    }
    for (int it = threadIdx.x; it < T * S; it += kThreads) {
        const int sidx = it / T, t = it % T;
        const int p = sidx * T + t;
        d.pair_tok[p] = t;
        d.pair_w[p] = 1.0f;
        d.pair_of[t * P + K + sidx] = p;
    }
    MOE_TRACE_POINT(0, 15);
    for (int p = threadIdx.x; p < T * P; p += kThreads) d.hmax[p] = 0u;
    if (threadIdx.x == 0) {
        *d.ticket = 0u;
        d.wave_ctr[0] = 0u;
        d.wave_ctr[1] = 0u;
    }
    MOE_TRACE_POINT(0, 7);
}

}  // namespace

// K splits of the router rows: enough blocks for the SMs, K ranges of a
// multiple of 64 columns, at most kMaxKSplit.
int route_ksplit(const DevLayer &d, int T, int sm_count) {
    const int gx = (d.E + kRouteWarps - 1) / kRouteWarps, gy = (T + kTokGroup - 1) / kTokGroup;
    int kh = 1;
    while (2 * kh <= kMaxKSplit && gx * gy * kh < sm_count && d.H % (64 * 2 * kh) == 0) kh *= 2;
    return kh;
}

size_t route_smem_bytes(const DevLayer &d, int T, int kh, int *tg_out) {
    // activation columns of one token group as FP32 (at most 8 tokens, at
    // most 96 KB), later the group's logits,
    const int Hk = d.H / kh;
    int tg = kTokGroup;
    while (tg > 1 && (size_t)tg * Hk * 4 > 96 * 1024) --tg;
    if (tg > T) tg = T;
    if (tg_out) *tg_out = tg;
    // plus the warps' partial logits [kRouteWarps][32] behind the columns
    return (size_t)tg * (size_t)std::max(Hk, d.E) * 4 + (size_t)kRouteWarps * 32 * 4;
}

cudaError_t launch_route(const DevLayer &d, const __nv_bfloat16 *x, int T, int *ids_out, float *w_out,
                         int sm_count, cudaStream_t s) {
    int tg = 1;
    const int kh = route_ksplit(d, T, sm_count);
    const size_t smem = route_smem_bytes(d, T, kh, &tg);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((d.E + kRouteWarps - 1) / kRouteWarps, (T + tg - 1) / tg, kh);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, route_kernel, d, x, T, tg, ids_out, w_out);
}

cudaError_t prepare_route_kernel(int optin_bytes) {
    return allow_max_dynamic_smem(route_kernel, optin_bytes);
}

}  // namespace moe
