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
// midpoint going to the code with mantissa bit 0; saturating at 6.
__device__ __forceinline__ int e2m1_code_rne(float v) {
    const float a = fabsf(v);
    int c;
    if (a <= 0.25f) c = 0;
    else if (a < 0.75f) c = 1;
    else if (a <= 1.25f) c = 2;
    else if (a < 1.75f) c = 3;
    else if (a <= 2.5f) c = 4;
    else if (a < 3.5f) c = 5;
    else if (a <= 5.0f) c = 6;
    else c = 7;
    return (v < 0.f && c) ? (c | 8) : c;
}

__device__ __forceinline__ float e2m1_value(int code) {
    const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
    const float m = mag[code & 7];
    return (code & 8) ? -m : m;
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

// One CTA per row (rows r < nrows of length len(r): n for x rows; for h rows
// I or Is by pair, the first n_short rows of len_short).  Each half-warp takes
// one 16-element block at a time, a lane per element, so that both
// candidates cost one element's work per lane and the error sums are 16
// shuffles; a row of 4096 takes four such rounds at 1024 threads.
// src may equal dst: every element is read and written by one thread, after
// the row maximum is complete.
__global__ void __launch_bounds__(kFosMaxThreads)
fos_kernel(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int stride, int len_long, int n_short, int len_short,
           float *__restrict__ gs_out, int *__restrict__ exp_out, unsigned *__restrict__ max_out,
           uint8_t *__restrict__ codes, uint8_t *__restrict__ sfc, int code_stride, int sf_stride) {
    // The next kernel may start at once: its own wait covers this kernel's
    // completion.  The rows come from the kernels before (the router's input,
    // the SwiGLU output), complete once this wait returns; it also orders
    // the writes below after those of the router (x's exponents) and of the
    // SwiGLU epilogue (h maxima).
    pdl_trigger();
    pdl_wait();
    __shared__ unsigned s_red[kFosMaxThreads / 32];
    const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    const int n = r < n_short ? len_short : len_long;
    const __nv_bfloat16 *row = src + (size_t)r * stride;
    __nv_bfloat16 *out = dst + (size_t)r * stride;

    // a = max |v| over the row (a >= 0, not NaN: its bits order as unsigned)
    float a = 0.f;
    for (int k = tid; k < n; k += blockDim.x) a = fmaxf(a, fabsf(__bfloat162float(row[k])));
    unsigned am = __reduce_max_sync(0xffffffffu, __float_as_uint(a));
    if (lane == 0) s_red[wid] = am;
    __syncthreads();
    am = __reduce_max_sync(0xffffffffu, lane < nw ? s_red[lane] : 0u);
    a = __uint_as_float(am);
    const float gs = a > 0.f ? __fdiv_rn(a, 1792.0f) : 1.0f;

    float newmax = 0.f;
    const int hb = lane & 16;   // this half-warp's first lane
    for (int base = 0; base < n; base += blockDim.x) {
        const int k = base + tid;
        const bool on = k < n;   // the same for a whole half-warp: n and blockDim are multiples of 16
        const float v = on ? __bfloat162float(row[k]) : 0.f;
        float m = fabsf(v);      // the block maximum
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float t[2], sv[2];
        int q[2];
        uint32_t scode[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float cg = __fmul_rn(i == 0 ? 6.0f : 4.0f, gs);
            scode[i] = e4m3_code_rn(__fdiv_rn(m, cg));
            const float sc = e4m3_value(scode[i]);
            const float dv = __fmul_rn(sc, gs);
            q[i] = sc > 0.f ? e2m1_code_rne(__fdiv_rn(v, dv)) : 0;
            const float rv = __fmul_rn(__fmul_rn(e2m1_value(q[i]), sc), gs);
            t[i] = fabsf(__fsub_rn(v, rv));
            sv[i] = sc;
        }
        // each candidate's error: the 16 terms added in element order, one
        // FP32 accumulator (every lane of the half-warp forms the same sums)
        float e6 = 0.f, e4 = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            e6 = __fadd_rn(e6, __shfl_sync(0xffffffffu, t[0], hb + j));
            e4 = __fadd_rn(e4, __shfl_sync(0xffffffffu, t[1], hb + j));
        }
        const int pick = e4 < e6 ? 1 : 0;   // ties: 6
        const float w = __fmul_rn(e2m1_value(q[pick]), sv[pick]);   // exact
        if (on) {
            out[k] = __float2bfloat16_rn(w);
            newmax = fmaxf(newmax, fabsf(w));
        }
        if (codes) {
            const uint32_t c = (uint32_t)q[pick] & 15u;
            const uint32_t hi = __shfl_down_sync(0xffffffffu, c, 1);
            if (on && (lane & 1) == 0) codes[(size_t)r * code_stride + k / 2] = (uint8_t)(c | (hi << 4));
            if (on && (lane & 15) == 0) sfc[(size_t)r * sf_stride + k / 16] = (uint8_t)scode[pick];
        }
    }
    unsigned nm = __reduce_max_sync(0xffffffffu, __float_as_uint(newmax));
    __syncthreads();   // every warp has read s_red above
    if (lane == 0) s_red[wid] = nm;
    __syncthreads();
    if (wid == 0) {
        nm = __reduce_max_sync(0xffffffffu, lane < nw ? s_red[lane] : 0u);
        if (lane == 0) {
            gs_out[r] = gs;
            if (exp_out) exp_out[r] = max(-100, exp_for_f16(__uint_as_float(nm)));
            if (max_out) max_out[r] = nm;
        }
    }
}

}  // namespace

cudaError_t launch_fos(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int nrows, int stride, int len_long,
                       int n_short, int len_short, float *gs, int *exp_out, unsigned *max_out, uint8_t *codes,
                       uint8_t *sfc, int code_stride, int sf_stride, cudaStream_t s) {
    if (nrows <= 0) return cudaSuccess;
    const int len = n_short > 0 ? max(len_long, len_short) : len_long;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nrows);
    cfg.blockDim = dim3(min(kFosMaxThreads, (len + 31) / 32 * 32));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fos_kernel, src, dst, stride, len_long, n_short, len_short, gs, exp_out,
                              max_out, codes, sfc, code_stride, sf_stride);
}

}  // namespace moe
