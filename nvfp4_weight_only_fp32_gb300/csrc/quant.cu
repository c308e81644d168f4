// quant.cu -- "Four Over Six" NVFP4 quantisation of activation rows, for the
// W4A4 option (moe_config.w4a4): "Inkling 2 Small on vLLM: Day-0 Support",
// "Mixed-precision MoE and Four-Over-Six NVFP4" (a per-token global scale
// plus, per 16-element block, the block maximum scaled to 6 and to 4, the
// lower reconstruction error kept) and "MoE with fused activation
// quantisation" (tokens quantised before gate/up, the SwiGLU output before
// down).
//
// Every decision is taken in FP32 with each step rounded on its own (the
// __f*_rn intrinsics are never contracted into fused multiply-adds), in this
// order, per row v of n BF16 values:
//   a = max |v|;  gs = a / 1792 (a = 0: gs = 1)
//   per 16-element block, m = its max |v|, for c = 6 then 4:
//     s_c = e4m3(m / (c * gs))              round to nearest even, saturating
//     q_k = e2m1(v_k / (s_c * gs))          nearest grid value, ties to the
//                                           code with mantissa bit 0, +-6 max
//     err_c = sum_k |v_k - e2m1(q_k) * s_c * gs|, k = 0..15 in order
//   the block keeps 4 if err_4 < err_6, else 6.
// The row is written back as the exact products e2m1 * e4m3 (at most six
// significant bits: exact in BF16) and the global scale gs goes to its own
// array; the GEMM epilogues multiply by it.  Optionally the codes themselves
// are written too (E2M1 codes two per byte, element 2j in the low nibble, and
// one E4M3 scale code per block), for the block-scaled tensor-core MMAs.  The power-of-two prescale the
// kernels use for the f16 operand (exponent of the row's new maximum) and,
// for h rows, the row maximum's bits are written as well.
#include "moe_internal.cuh"

namespace moe {

namespace {

// E2M1 code of the nearest grid value to |v| (0, .5, 1, 1.5, 2, 3, 4, 6), a
// midpoint going to the code with mantissa bit 0; saturating at 6: 7 less the
// number of the seven midpoints that |v| does not pass.
__device__ __forceinline__ uint32_t e2m1_code_rne(float v) {
    const float a = fabsf(v);
    const uint32_t c = 7u - ((a <= 0.25f) + (a < 0.75f) + (a <= 1.25f) + (a < 1.75f) + (a <= 2.5f) + (a < 3.5f) +
                             (a <= 5.0f));
    return (v < 0.f && c) ? (c | 8u) : c;
}

// FP32 -> E4M3 (fn) code, round to nearest even, saturating (v >= 0)
__device__ __forceinline__ uint32_t e4m3_code_rn(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(v), "f"(v));   // both bytes
    return r & 0xFFu;
}
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    const uint32_t h2 = e4m3x2_to_f16x2(code);
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

constexpr int kFosMaxThreads = 1024;
constexpr int kFosMaxCluster = 8;

// E2M1 value of a code: the magnitudes times 2 are 0,1,2,3,4,6,8,12, one per
// nibble of 0xC8643210.
__device__ __forceinline__ float e2m1_value(uint32_t code) {
    const float m = (float)((0xC8643210u >> (4 * (code & 7u))) & 15u) * 0.5f;
    return (code & 8u) ? -m : m;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// every thread of every CTA of the cluster; orders the shared-memory writes
// before it with the reads after it, across the cluster
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t ld_cluster_u32(const void *p, uint32_t rank) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p), ra, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(ra) : "memory");
    return v;
}
__device__ __forceinline__ void st_cluster_u32(void *p, uint32_t rank, uint32_t v) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p), ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(ra), "r"(v) : "memory");
}

// one candidate scale c (6 or 4) of a 16-element block whose maximum is m:
// this lane's four elements v[0..3] get their codes q and error terms t
__device__ __forceinline__ void fos_candidate(const float (&v)[4], float m, float cg, float gs, uint32_t &scode,
                                              float &sc, uint32_t &q, float (&t)[4]) {
    scode = e4m3_code_rn(__fdiv_rn(m, cg));
    sc = e4m3_value(scode);
    const float dv = __fmul_rn(sc, gs);
    q = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t c = 0;
        if (sc > 0.f) {
            const float z = __fdiv_rn(v[j], dv);
            c = e2m1_code_rne(z);
        }
        const float rv = __fmul_rn(__fmul_rn(e2m1_value(c), sc), gs);
        t[j] = fabsf(__fsub_rn(v[j], rv));
        q |= c << (4 * j);
    }
}

// Rows are split over a cluster of S CTAs (S = gridDim.x / nrows, the
// cluster's extent); CTA s takes the s-th run of the row's 16-element blocks,
// four lanes to a block, four consecutive elements to a lane, so that a warp
// covers 128 elements.  The row maximum and the maximum of the written row
// are reduced over the cluster through distributed shared memory.  A block's
// two error sums run through its four lanes in element order (each lane adds
// its four terms to its left neighbour's sum), one FP32 accumulator per
// candidate as in the definition.
// src may equal dst: each element is read, then written, by one thread, and
// the row maximum is taken over the values read before any write.
__global__ void __launch_bounds__(kFosMaxThreads)
fos_kernel(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int S, int stride, int len_long, int n_short,
           int len_short, float *__restrict__ gs_out, int *__restrict__ exp_out, unsigned *__restrict__ max_out,
           uint8_t *__restrict__ codes, uint8_t *__restrict__ sfc, int code_stride, int sf_stride, int wait_late) {
    // The next kernel may start at once: its own wait covers this kernel's
    // completion.  The rows come from the kernels before (the SwiGLU output),
    // complete once the wait returns; it also orders the writes below after
    // those of the SwiGLU epilogue (h maxima).  With wait_late (the tokens,
    // launched right after the router, which releases its dependents only
    // once its own wait has returned: the tokens are complete by then) the
    // work runs beside the router and the wait comes last, so that this grid
    // still completes after the router's.
    pdl_trigger();
    if (!wait_late) pdl_wait();
    __shared__ unsigned s_red[kFosMaxThreads / 32];
    __shared__ unsigned s_part[kFosMaxCluster];   // rank 0: each CTA's maximum of the written values
    __shared__ unsigned s_amax;                    // this CTA's maximum of the values read
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    const int r = blockIdx.x / S;
    const uint32_t rank = S > 1 ? cluster_rank() : 0u;
    const int n = r < n_short ? len_short : len_long;
    const int nblk = n >> 4, per = (nblk + S - 1) / S;
    const int b0 = min(nblk, (int)rank * per), b1 = min(nblk, b0 + per);
    const int step = blockDim.x >> 2;   // blocks per round
    const __nv_bfloat16 *row = src + (size_t)r * stride;
    __nv_bfloat16 *out = dst + (size_t)r * stride;

    // a = max |v| over the row (a >= 0, not NaN: its bits order as unsigned)
    uint2 first = make_uint2(0u, 0u);   // the first round's values, kept for the second pass
    float a = 0.f;
    for (int b = b0 + (tid >> 2), i = 0; b < b1; b += step, ++i) {
        const uint2 u = *reinterpret_cast<const uint2 *>(row + 16 * b + 4 * (tid & 3));
        if (i == 0) first = u;
        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
        const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
        a = fmaxf(a, fmaxf(fmaxf(fabsf(__low2float(p0)), fabsf(__high2float(p0))),
                           fmaxf(fabsf(__low2float(p1)), fabsf(__high2float(p1)))));
    }
    unsigned am = __reduce_max_sync(0xffffffffu, __float_as_uint(a));
    if (lane == 0) s_red[wid] = am;
    __syncthreads();
    if (wid == 0) {
        am = __reduce_max_sync(0xffffffffu, lane < nw ? s_red[lane] : 0u);
        if (lane == 0) s_amax = am;
    }
    if (S > 1) {
        cluster_barrier();
        am = __reduce_max_sync(0xffffffffu, lane < S ? ld_cluster_u32(&s_amax, (uint32_t)lane) : 0u);
    } else {
        __syncthreads();
        am = s_amax;
    }
    a = __uint_as_float(am);
    const float gs = a > 0.f ? __fdiv_rn(a, 1792.0f) : 1.0f;
    const float cg6 = __fmul_rn(6.0f, gs), cg4 = __fmul_rn(4.0f, gs);

    float newmax = 0.f;
    const int ql = lane & 3;   // this lane's place in its block
    for (int bb = b0, i = 0; bb < b1; bb += step, ++i) {
        const int b = bb + (tid >> 2);
        const bool on = b < b1;   // the same for the block's four lanes
        uint2 u = first;
        if (i > 0 && on) u = *reinterpret_cast<const uint2 *>(row + 16 * b + 4 * ql);
        if (!on) u = make_uint2(0u, 0u);
        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
        const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
        const float v[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
        float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));   // the block maximum
        uint32_t sc6, sc4, q6, q4;
        float s6, s4, t6[4], t4[4];
        fos_candidate(v, m, cg6, gs, sc6, s6, q6, t6);
        fos_candidate(v, m, cg4, gs, sc4, s4, q4, t4);
        // err_c = (((0 + t_0) + t_1) + ...) + t_15: lane ql adds its terms to
        // the sum of lanes 0..ql-1, which arrives from its left neighbour
        float e6 = 0.f, e4 = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float l6 = __shfl_up_sync(0xffffffffu, e6, 1, 4);
            const float l4 = __shfl_up_sync(0xffffffffu, e4, 1, 4);
            if (ql == j) {
                e6 = j ? l6 : 0.f;
                e4 = j ? l4 : 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    e6 = __fadd_rn(e6, t6[k]);
                    e4 = __fadd_rn(e4, t4[k]);
                }
            }
        }
        e6 = __shfl_sync(0xffffffffu, e6, 3, 4);
        e4 = __shfl_sync(0xffffffffu, e4, 3, 4);
        const bool pick4 = e4 < e6;   // ties: 6
        const uint32_t q = pick4 ? q4 : q6;
        const float sv = pick4 ? s4 : s6;
        if (on) {
            float w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                w[j] = __fmul_rn(e2m1_value(q >> (4 * j)), sv);   // exact
                newmax = fmaxf(newmax, fabsf(w[j]));
            }
            const __nv_bfloat162 o0 = __floats2bfloat162_rn(w[0], w[1]);
            const __nv_bfloat162 o1 = __floats2bfloat162_rn(w[2], w[3]);
            uint2 o;
            o.x = *reinterpret_cast<const uint32_t *>(&o0);
            o.y = *reinterpret_cast<const uint32_t *>(&o1);
            *reinterpret_cast<uint2 *>(out + 16 * b + 4 * ql) = o;
            if (codes) {
                // elements 2j and 2j+1 share a byte, the first in the low nibble
                *reinterpret_cast<uint16_t *>(codes + (size_t)r * code_stride + 8 * b + 2 * ql) = (uint16_t)q;
                if (ql == 0) sfc[(size_t)r * sf_stride + b] = (uint8_t)(pick4 ? sc4 : sc6);
            }
        }
    }
    unsigned nm = __reduce_max_sync(0xffffffffu, __float_as_uint(newmax));
    if (lane == 0) s_red[wid] = nm;   // every read of s_red above came before the barrier after it
    __syncthreads();
    if (wid == 0) {
        nm = __reduce_max_sync(0xffffffffu, lane < nw ? s_red[lane] : 0u);
        if (lane == 0) {
            if (S > 1) st_cluster_u32(&s_part[rank], 0u, nm);
            else s_part[0] = nm;
        }
    }
    if (S > 1) cluster_barrier();   // also keeps rank 0's shared memory alive for the stores above
    if (rank == 0 && tid == 0) {
        nm = 0u;
        for (int i = 0; i < S; ++i) nm = max(nm, s_part[i]);
        gs_out[r] = gs;
        if (exp_out) exp_out[r] = max(-100, exp_for_f16(__uint_as_float(nm)));
        if (max_out) max_out[r] = nm;
    }
    if (wait_late) pdl_wait();
}

}  // namespace

// GB300's SM count, for the split heuristic below only: any value gives the
// same results (no device query in the launch path, which may be captured).
constexpr int kFosSmsHint = 152;

// The cluster size: the fewest CTAs per row (1, 2, 4 or 8) that give at
// least two CTAs per SM in all, or blocks of at most 32 16-element runs (128
// threads) per CTA.
static int fos_split(int nrows, int len) {
    const int nblk = len / 16;
    int S = 1;
    while (S < kFosMaxCluster && (long long)nrows * S < 2LL * kFosSmsHint && (nblk + S - 1) / S > 32) S *= 2;
    while (S < kFosMaxCluster && (nblk + S - 1) / S > kFosMaxThreads / 4) S *= 2;
    return S;
}

cudaError_t launch_fos(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int nrows, int stride, int len_long,
                       int n_short, int len_short, float *gs, int *exp_out, unsigned *max_out, uint8_t *codes,
                       uint8_t *sfc, int code_stride, int sf_stride, cudaStream_t s, bool wait_late) {
    if (nrows <= 0) return cudaSuccess;
    const int len = n_short > 0 ? max(len_long, len_short) : len_long;
    const int S = fos_split(nrows, len);
    const int per = (len / 16 + S - 1) / S;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nrows * S));
    cfg.blockDim = dim3(min(kFosMaxThreads, (4 * per + 31) / 32 * 32));
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = S > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, fos_kernel, src, dst, S, stride, len_long, n_short, len_short, gs, exp_out,
                              max_out, codes, sfc, code_stride, sf_stride, wait_late ? 1 : 0);
}

}  // namespace moe
