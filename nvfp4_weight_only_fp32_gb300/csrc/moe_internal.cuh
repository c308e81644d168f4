// moe_internal.cuh -- private declarations shared by the library's CUDA files.
//
// Streaming layout of the repacked NVFP4 weights (built once by moe_init):
//
//   A weight matrix is cut into tiles of 16 rows (the M of one
//   mma.m16n8k16) and each tile's K range into chunks of 64 elements (four
//   16-element NVFP4 blocks).  One chunk is 576 contiguous bytes:
//
//     bytes [0, 512)   codes.  Lane L = 4g + q of a warp owns bytes
//                      [16L, 16L+16): word i (i = 0..3) holds the A-fragment
//                      codes of block 4c+i for that lane, byte b of the word
//                      being fragment register b:
//                        b=0  row g,    k = 16(4c+i) + 2q + {0,1}
//                        b=1  row g+8,  same k
//                        b=2  row g,    k + 8
//                        b=3  row g+8,  k + 8
//                      (low nibble = the lower k, as in the canonical layout,
//                      so each byte is a copy of one canonical byte).
//     bytes [512, 576) E4M3 block scales: byte 8g + 2i + h is the scale of
//                      row g + 8h for block 4c+i.
//
//   One warp therefore streams a chunk with one 16-byte load of codes and one
//   8-byte load of scales per lane, and every loaded byte is used.
//
//   Gate/up (w13): tile r holds gate rows 8r..8r+7 as MMA rows 0..7 and the
//   matching up rows as MMA rows 8..15, so SwiGLU pairs are lane-local in the
//   accumulator.  Down (w2): tile r holds output rows 16r..16r+15.
//   Offset of chunk c of tile r of expert e: ((e*NT + r)*NC + c) * 576.
//
// FP8 experts (E4M3 codes with a scale per row and 32 elements: MXFP8, or the
// FP32 scale of a 128 x 128 block) use "F8 chunks" of the same 576 bytes:
// 16 rows x 32 K elements (two MMA K blocks kb = 0, 1).
//     bytes [0, 512)   codes.  Lane L = 4g + q owns bytes [16L, 16L+16):
//                      byte 8kb + 2j + e is element k = 16kb + 2q + e (+8
//                      for j = 2, 3) of row g (j = 0, 2) or g+8 (j = 1, 3),
//                      i.e. fragment register j of block kb, low byte first.
//     bytes [512, 576) the FP32 scales of the 16 rows for these 32 elements:
//                      bytes 8g + 4h hold the scale of row g + 8h.
//   A tile has K/32 F8 chunks.  The same two loads per lane (16 code bytes at
//   16L, 8 scale bytes at 512 + 8g) fetch a chunk in either format.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_nvfp4.h"

namespace moe {

constexpr int kBlockK = 16;        // NVFP4 block length along K
constexpr int kChunkK8 = 32;       // K elements per F8 chunk
constexpr int kChunkK = 64;        // K elements per streamed chunk
constexpr int kChunkBytes = 576;   // 512 code bytes + 64 scale bytes
constexpr int kCodeBytes = 512;
constexpr int kGemvWarps = 8;      // warps per GEMV CTA
constexpr int kMaxTokens = 64;
constexpr int kMaxTopK = 8;
constexpr int kMaxExperts = 512;
constexpr int kMaxShared = 2;
constexpr int kFusedSlots = 8 * kMaxTopK + kMaxShared;   // slots of a single-launch call (T <= 8)
constexpr int kFusedPairs = 8 * (kMaxTopK + kMaxShared); // (token, expert) pairs of such a call
constexpr int kRouteWarps = 8;     // experts per router CTA
constexpr int kMaxKSplit = 8;      // router: K splits of the rows (blocks along z)

// Everything a kernel needs to know about a layer (passed by value).
struct DevLayer {
    int H, E, k, I, S, Is, normalize;
    float routed_scale;
    int max_tokens, max_slots, max_pairs, Imax;
    const float *router_w;          // [E,H]
    const float *router_b;          // [E] or null
    const uint8_t *w13r;            // repacked, E experts
    const uint8_t *w2r;
    const float *gs13;              // [E,2]
    const float *gs2;               // [E]
    const uint8_t *sw13r;           // repacked, S shared experts
    const uint8_t *sw2r;
    const float *sgs13;             // [S,2]
    const float *sgs2;              // [S]
    const float4 *gsp;              // [E+S] per expert: gate gs, up gs, down gs, router bias
                                    //   (routed experts first, then the shared ones; bias 0 for those)
    size_t e13_stride, e2_stride;   // bytes per routed expert
    size_t s13_stride, s2_stride;   // bytes per shared expert
    // workspace (device)
    float *logits;                  // [Tm, E]
    float *lpart;                   // [kMaxKSplit, Tm, E] router partial sums by K range
    unsigned *xmaxb;                // [Tm] router: max |x| bits per token (zero between calls)
    int *ids;                       // [Tm, k]
    float *wsel;                    // [Tm, k]
    int *xexp;                      // [Tm]  power-of-two prescale of x rows
    int *nslots;                    // [1]
    int *slot_expert;               // [max_slots]  >=0 routed id, <0 -(shared+1)
    int *slot_m;                    // [max_slots]  tokens on the slot
    int *slot_p0;                   // [max_slots]  first pair of the slot
    int *pair_tok;                  // [max_pairs]
    float *pair_w;                  // [max_pairs]
    int *pair_of;                   // [Tm, k+S]
    unsigned *hmax;                 // [max_pairs]  max |h| bits per pair
    __nv_bfloat16 *h_ws;            // [max_pairs, Imax]
    float *y_ws;                    // [max_pairs, H]
    unsigned *ticket;               // [1]
    unsigned *down_cnt;             // [H/16] arrivals per down row group
    int *err;                       // [1] sticky device error word
    // single-launch path: values exchanged between blocks carry the call's
    // tag (calls finished + 1) in their upper 32 bits, so a reader polls the
    // words themselves instead of waiting at a grid barrier
    unsigned long long *logit_tag;  // [8, E] (tag << 32) | FP32 logit bits
    unsigned long long *h_tag;      // [8 * (k + S), Imax / 2] (tag << 32) | two BF16 of h (even index low)
    unsigned *calls;                // [grid size] calls each block has finished
    int grouped_min;                // slots with >= this many tokens use the grouped kernels (0: none)
    int debug_stall;                // single launch: added to the tag its logit wait expects (test hook)
    int *nhot;                      // [1] number of such slots
    int *hot_slots;                 // [max_slots] their slot indices, ascending
    int tick16;                     // grouped down kernel: combine tickets per 16-row tile (beside the
                                    //   wave down kernel) instead of per 128-row group; set per launch
    int nsm;                        // SMs (the grouped kernels' blocks)
    int tau_max;                    // highest grouped threshold the router may raise to (>= grouped_min)
    int *ncold;                     // [1] routed slots below the grouped threshold (steps of > 8 tokens)
    int *cold_slots;                // [max_slots] their slot indices, ascending
    unsigned *tg_ticket;            // [max_tokens] router: arrivals per token group
    unsigned long long *emask;      // [E] router: tokens that selected each expert (bit t)
    unsigned *wave_ctr;             // [2] chain gate/up wave kernel: next unit to hand out (reset by the router)
    unsigned long long *trace;      // traced build only: phase timestamps
    int trace_blocks;
    int score_func;                 // 0 sigmoid per expert, 1 softmax over all experts
    int f8e, f8s;                   // routed / shared experts stored as F8 chunks
    int w4a4;                       // activations quantised (Four-Over-Six NVFP4) before each GEMM
    __nv_bfloat16 *xq;              // [Tm, H] W4A4: the tokens' dequantised e2m1 * e4m3 values
    float *gsx;                     // [Tm] W4A4: their global scales
    float *gsh;                     // [max_pairs] W4A4: the h rows' global scales
    uint8_t *xq4, *xsf;             // [Tm, H/2], [Tm, H/16] W4A4: the tokens' E2M1 codes (element 2j in
                                    //   the low nibble) and E4M3 block scale codes
    uint8_t *hq4, *hsf;             // [max_pairs, Imax/2], [max_pairs, Imax/16] the same for the h rows
};

// Chunks per tile row of K elements, in the NVFP4 or the F8 chunk layout.
__host__ __device__ inline int chunks_of(int K, bool f8) { return f8 ? K / kChunkK8 : K / kChunkK; }

// ---------------------------------------------------------------------------
// Host-side launchers (defined in the .cu files).
// ---------------------------------------------------------------------------
cudaError_t launch_route(const DevLayer &d, const __nv_bfloat16 *x, int T, int *ids_out,
                         float *w_out, int sm_count, cudaStream_t s);
// gate/up: one wave of 16-warp blocks (one per SM) for steps of at most 8
// tokens where the shape allows it, else the per-slot GEMV kernel
cudaError_t launch_gate_up(const DevLayer &d, const __nv_bfloat16 *x, int T, int sm_count, int optin_smem,
                           cudaStream_t s);
cudaError_t launch_down(const DevLayer &d, int T, __nv_bfloat16 *out, int sm_count, int optin_smem,
                        cudaStream_t s);
bool down_tile_tickets(const DevLayer &d, int T, int sm_count, int optin_smem);
int cold_threshold_max(const DevLayer &d, int sm_count, int optin_smem);
bool grouped_supported(const DevLayer &d, int sm_count);
cudaError_t launch_grouped_gate_up(const DevLayer &d, const __nv_bfloat16 *x, int T, int sm_count, cudaStream_t s);
cudaError_t launch_grouped_down(const DevLayer &d, int T, __nv_bfloat16 *out, int sm_count, cudaStream_t s);
cudaError_t prepare_grouped_kernels(int optin_bytes);
cudaError_t prepare_kernels();   // per device, once: shared-memory limits
bool fused_eligible(const DevLayer &d, int T, int sm_count, size_t optin_smem);
// x_sys: x is the device alias of pinned host memory (read by plain loads)
cudaError_t launch_fused(const DevLayer &d, const __nv_bfloat16 *x, int T, __nv_bfloat16 *out, int *ids,
                         float *w, int sm_count, bool coop, cudaStream_t s, bool x_sys = false);
int fused_blocks_per_sm(const DevLayer &d, int T);
cudaError_t launch_repack(const uint8_t *codes, const uint8_t *sf, int n_mats, int rows, int cols,
                          bool gate_up, uint8_t *dst, cudaStream_t s);
cudaError_t launch_pack_scales(const DevLayer &d, cudaStream_t s);
cudaError_t launch_dequant(const uint8_t *rep, float gs_a, float gs_b, int rows, int cols,
                           bool gate_up, float *dst, cudaStream_t s);
// F8 chunks from E4M3 codes [n, rows, cols] and their scales: fmt 2 = FP32
// per 128 x 128 block ([n, ceil(rows/128), ceil(cols/128)]), 3 = E8M0 per
// 32 elements ([n, rows, cols/32]).
cudaError_t launch_repack_f8(const uint8_t *codes, const void *sf, int fmt, int n_mats, int rows, int cols,
                             bool gate_up, uint8_t *dst, cudaStream_t s);
cudaError_t launch_dequant_f8(const uint8_t *rep, int rows, int cols, bool gate_up, float *dst, cudaStream_t s);
// Four-Over-Six NVFP4 quantisation of activation rows (quant.cu): rows of
// `stride` elements, the first n_short of length len_short, the rest len_long;
// writes the dequantised e2m1 * e4m3 values (BF16, exact) to dst (may be
// src), the global scales, and (optional) the f16 prescale exponent and the
// max |value| bits of each row.  wait_late: only right after the router's
// launch (which releases its dependents once its own dependency wait has
// returned), for rows the router reads as well: the rows are read at once
// and the dependency wait comes last.
cudaError_t launch_fos(const __nv_bfloat16 *src, __nv_bfloat16 *dst, int nrows, int stride, int len_long,
                       int n_short, int len_short, float *gs, int *exp_out, unsigned *max_out, uint8_t *codes,
                       uint8_t *sfc, int code_stride, int sf_stride, cudaStream_t s, bool wait_late = false);
// MXFP4 scales: per (matrix, half) the smallest and largest E8M0 code and
// whether a NaN code (255) occurs -> mm[(mat * 2 + half) * 3 + {0,1,2}]
// (half 1 only for gate/up: its up rows).
cudaError_t launch_mx_scale_range(const uint8_t *sf, int n_mats, int rows, int cols, bool gate_up, int *mm,
                                  cudaStream_t s);
// MXFP4 scales -> the NVFP4 scales of the same weights: E8M0 code c of 32
// elements -> the E4M3 code of 2^(c - 127 - off) for both of its 16-element
// blocks, off = offs[mat * 2 + half] (the tensor scale becomes 2^off).
cudaError_t launch_mx_to_nv_scales(const uint8_t *sf, const int *offs, int n_mats, int rows, int cols,
                                   bool gate_up, uint8_t *dst, cudaStream_t s);

// Let `fn` use all the shared memory a block may opt in to, minus its static part.
template <class F>
inline cudaError_t allow_max_dynamic_smem(F fn, int optin_bytes) {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, fn);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin_bytes - (int)a.sharedSizeBytes);
}

// Chunk geometry.
__host__ __device__ inline size_t repacked_bytes(int rows, int cols, bool f8 = false) {
    return (size_t)(rows / 16) * (size_t)chunks_of(cols, f8) * kChunkBytes;
}

// ---------------------------------------------------------------------------
// Device helpers (inline PTX).
// ---------------------------------------------------------------------------
#if defined(__CUDACC__)

// Phase tracing, compiled only into the traced build (-DMOE_TRACE): one
// thread of each block (thread 0 unless named) stores %globaltimer, the SM
// cycle counter or a count at numbered points into the buffer that
// moe_trace_attach() installed in DevLayer ([kernel slot][block][16] u64).
// In the regular build every trace point is empty.
#ifdef MOE_TRACE
#define MOE_TRACE_STORE_(kid, i, tid, val)                                                       \
    do {                                                                                         \
        if (threadIdx.x == (tid) && d.trace) {                                                   \
            const int b_ = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;       \
            if (b_ < d.trace_blocks)                                                             \
                d.trace[((size_t)(kid) * d.trace_blocks + b_) * 16 + (i)] = (unsigned long long)(val); \
        }                                                                                        \
    } while (0)
__device__ __forceinline__ unsigned long long moe_globaltimer_() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
#define MOE_TRACE_POINT_AT(kid, i, tid) MOE_TRACE_STORE_(kid, i, tid, moe_globaltimer_())
#define MOE_TRACE_CLOCK_AT(kid, i, tid) MOE_TRACE_STORE_(kid, i, tid, clock64())
#define MOE_TRACE_VALUE_AT(kid, i, tid, v) MOE_TRACE_STORE_(kid, i, tid, v)
#else
#define MOE_TRACE_POINT_AT(kid, i, tid) \
    do {                                \
    } while (0)
#define MOE_TRACE_CLOCK_AT(kid, i, tid) \
    do {                                \
    } while (0)
#define MOE_TRACE_VALUE_AT(kid, i, tid, v) \
    do {                                   \
    } while (0)
#endif
#define MOE_TRACE_POINT(kid, i) MOE_TRACE_POINT_AT(kid, i, 0)
#define MOE_TRACE_CLOCK(kid, i) MOE_TRACE_CLOCK_AT(kid, i, 0)
#define MOE_TRACE_VALUE(kid, i, v) MOE_TRACE_VALUE_AT(kid, i, 0, v)

__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Streaming loads of weights: read-only, not kept in L1, and first in line
// for eviction from L2 (the weights are read once per call; code, activations
// and the workspace should stay in L2 instead).
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint4 ld_stream_v4(const void *p, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void *p, uint64_t pol) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;\n"
                 : "=r"(r.x), "=r"(r.y) : "l"(p), "l"(pol));
    return r;
}
__device__ __forceinline__ float4 ld_f4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}

// Four E2M1 pairs (one byte each) -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t &h0, uint32_t &h1,
                                                uint32_t &h2, uint32_t &h3) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}\n"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3) : "r"(w));
}

// Two E4M3 bytes (low 16 bits of v) -> f16x2 (low byte -> low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}\n" : "=r"(r) : "r"(v));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// D[16x8] += A[16x16] * B[16x8], f16 inputs, FP32 accumulators.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 r;
    uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}

// Loads that must be issued where they stand (e.g. before a
// griddepcontrol.wait): volatile asm keeps the compiler from sinking them.
__device__ __forceinline__ float2 ld_nc_f2(const float *p) {
    float2 r;
    asm volatile("ld.global.nc.v2.f32 {%0,%1}, [%2];\n" : "=f"(r.x), "=f"(r.y) : "l"(p));
    return r;
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int exp_for_f16(float maxabs) {
    // power of two 2^e such that maxabs * 2^-e lies in [2^14, 2^15) when
    // maxabs > 0: f16 then holds every BF16 value of the row exactly except
    // those below maxabs * 2^-31 (8 significant bits need an f16 exponent of
    // at least -17).  Callers clamp e at -100 so that 2^-e stays a normal
    // FP32 number.
    return (maxabs > 0.f && isfinite(maxabs)) ? ilogbf(maxabs) - 14 : 0;
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// One 576-byte chunk for one lane: 16 code bytes and the 8 scale bytes of its
// row group.
__device__ __forceinline__ void load_chunk(const uint8_t *tbase, int c, int lane, uint4 &cw,
                                           uint2 &sw, uint64_t pol) {
    const uint8_t *ch = tbase + (size_t)c * kChunkBytes;
    cw = ld_stream_v4(ch + 16 * lane, pol);
    sw = ld_stream_v2(ch + kCodeBytes + 8 * (lane >> 2), pol);
}

// ---- mbarrier + bulk async copy (TMA, 1-D) ----
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *b, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_u32(b)), "r"(parity) : "memory");
    return ok != 0;
}
// global -> shared bulk copy completing on mbarrier `b` (bytes % 16 == 0,
// both addresses 16-byte aligned), with an L2 cache policy
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *b,
                                         uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;\n" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(b)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// The router's sigmoid score in FP32: exp to ~2 ulp, then an approximate
// reciprocal (~1 ulp; 0 once 1 + exp(-z) passes 2^126, where the score is
// below 2^-126 anyway) -- branch-free, a few ulp from the correctly rounded
// score.
__device__ __forceinline__ float sigmoid_score(float z) { return __fdividef(1.0f, 1.0f + expf(-z)); }

// The ranking key of an expert: its FP32 logit mapped to an unsigned integer
// of the same order (sigmoid is strictly increasing, so this is the order of
// the scores).  -0 and +0 share one key; a NaN logit gets 0, below every
// number (the smallest key of a number, that of -inf, is 0x007FFFFF).
__device__ __forceinline__ unsigned logit_key(float z) {
    unsigned u = __float_as_uint(z);
    if (u == 0x80000000u) u = 0u;
    return isnan(z) ? 0u : (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The FP32 logit a key encodes (NaN for key 0).
__device__ __forceinline__ float key_logit(unsigned key) {
    const float z = __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
    return key ? z : __int_as_float(0x7fc00000);
}

// The weight of a chosen expert: the sigmoid of the logit its key encodes
// (NaN for key 0).
__device__ __forceinline__ float key_score(unsigned key) {
    const float z = __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
    return key ? sigmoid_score(z) : __int_as_float(0x7fc00000);
}

// c[i] >= c[j] afterwards
__device__ __forceinline__ void key_cx(unsigned long long &a, unsigned long long &b) {
    const bool sw = b > a;
    const unsigned long long x = sw ? b : a, y = sw ? a : b;
    a = x;
    b = y;
}

// Descending sort of M = 1, 2, 4 or 8 keys: Batcher's odd-even merge sort
// network (for 8: 19 comparators in 6 levels).
template <int M>
__device__ __forceinline__ void sort_keys_desc(unsigned long long (&c)[M]) {
    if constexpr (M == 2) {
        key_cx(c[0], c[1]);
    } else if constexpr (M == 4) {
        key_cx(c[0], c[1]); key_cx(c[2], c[3]);
        key_cx(c[0], c[2]); key_cx(c[1], c[3]);
        key_cx(c[1], c[2]);
    } else if constexpr (M == 8) {
        key_cx(c[0], c[1]); key_cx(c[2], c[3]); key_cx(c[4], c[5]); key_cx(c[6], c[7]);
        key_cx(c[0], c[2]); key_cx(c[1], c[3]); key_cx(c[4], c[6]); key_cx(c[5], c[7]);
        key_cx(c[1], c[2]); key_cx(c[5], c[6]);
        key_cx(c[0], c[4]); key_cx(c[1], c[5]); key_cx(c[2], c[6]); key_cx(c[3], c[7]);
        key_cx(c[2], c[4]); key_cx(c[3], c[5]);
        key_cx(c[1], c[2]); key_cx(c[3], c[4]); key_cx(c[5], c[6]);
    } else {
        static_assert(M == 1, "1, 2, 4 or 8 keys per lane");
    }
}

// Warp-wide top-k over 64-bit sort keys, M per lane (M a power of two up to
// 16; all keys distinct; 0 marks an empty place and is never chosen while
// k <= the number of real keys).  Every round the warp takes the largest of
// the lanes' largest keys (its high word, then among the lanes holding that,
// its low word) and the lane that held it drops it.  Lane j < k ends with
// the j-th choice.
// Tree form: a round takes each lane's largest by a pairwise tree and the
// winner clears it in place (c ends with the chosen keys zeroed, the rest
// where they were).  Short code: it runs once per call, from a cold
// instruction cache.
template <int M>
__device__ __forceinline__ unsigned long long warp_topk_tree(unsigned long long (&c)[M], int K, int lane) {
    unsigned long long mine = 0ull;
#pragma unroll 1
    for (int j = 0; j < K; ++j) {
        unsigned long long t[M];
#pragma unroll
        for (int i = 0; i < M; ++i) t[i] = c[i];
#pragma unroll
        for (int w = M / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) t[i] = t[i + w] > t[i] ? t[i + w] : t[i];
        const unsigned hi = (unsigned)(t[0] >> 32), lo = (unsigned)t[0];
        const unsigned mx = __reduce_max_sync(0xffffffffu, hi);
        const unsigned ml = __reduce_max_sync(0xffffffffu, hi == mx ? lo : 0u);
        if (lane == j) mine = ((unsigned long long)mx << 32) | ml;
        if (hi == mx && lo == ml) {
#pragma unroll
            for (int i = 0; i < M; ++i) c[i] = c[i] == t[0] ? 0ull : c[i];
        }
    }
    return mine;
}

// Sorted form (M <= 8): each lane first sorts its keys, largest first, so
// that a round's candidate is its first key and dropping it moves the
// others up by one (shorter rounds, a longer prologue); c ends with the
// lane's keys not chosen, largest first.
template <int M>
__device__ __forceinline__ unsigned long long warp_topk_sorted(unsigned long long (&c)[M], int K, int lane) {
    sort_keys_desc<M>(c);
    unsigned long long mine = 0ull;
#pragma unroll 1
    for (int j = 0; j < K; ++j) {
        const unsigned hi = (unsigned)(c[0] >> 32), lo = (unsigned)c[0];
        const unsigned mx = __reduce_max_sync(0xffffffffu, hi);
        const unsigned ml = __reduce_max_sync(0xffffffffu, hi == mx ? lo : 0u);
        if (lane == j) mine = ((unsigned long long)mx << 32) | ml;
        const bool won = hi == mx && lo == ml;
#pragma unroll
        for (int i = 0; i + 1 < M; ++i) c[i] = won ? c[i + 1] : c[i];
        c[M - 1] = won ? 0ull : c[M - 1];
    }
    return mine;
}

// Routing-weighted combine of output rows [row0, row0 + nrows) for all T
// tokens: out[t, m] = bf16(sum_j w[t, j] * y[pair(t, j), m] + sum_s y[pair(t,
// k + s), m]), FP32 in a fixed order (routed slots in selection order, then
// the shared ones).  Run by threads tid = 0..nthr-1 of the calling block;
// `sync` synchronises exactly those threads.  s_pair/s_pw: shared scratch of
// T * (k + S) entries each.
template <class Sync>
__device__ __forceinline__ void combine_rows(const DevLayer &d, int T, __nv_bfloat16 *out, int row0, int nrows,
                                             int *s_pair, float *s_pw, int tid, int nthr, Sync sync) {
    const int K = d.k, P = d.k + d.S;
    for (int i = tid; i < T * P; i += nthr) {
        const int p = __ldcg(d.pair_of + i);
        s_pair[i] = p;
        s_pw[i] = (i % P) < K ? __ldcg(d.pair_w + p) : 1.0f;
    }
    sync();
    const int nq = nrows / 4;
    for (int it = tid; it < T * nq; it += nthr) {
        const int t = it / nq, m4 = row0 / 4 + (it - t * nq);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < P; ++j) {
            const float w = s_pw[t * P + j];
            const float4 y = __ldcg(reinterpret_cast<const float4 *>(d.y_ws + (size_t)s_pair[t * P + j] * d.H) + m4);
            a.x = fmaf(w, y.x, a.x);
            a.y = fmaf(w, y.y, a.y);
            a.z = fmaf(w, y.z, a.z);
            a.w = fmaf(w, y.w, a.w);
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t *>(&lo);
        v.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(out + (size_t)t * d.H + 4 * m4) = v;
    }
}

// Decode one chunk's A fragments for one lane: 4 blocks x 4 registers.
// a[i][b] = exact f16 products e2m1 * e4m3 (<= 6 significant bits, in range).
__device__ __forceinline__ void decode_chunk(const uint4 &cw, const uint2 &sw,
                                             uint32_t (&a)[4][4]) {
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t sp = (i < 2) ? (sw.x >> (16 * i)) : (sw.y >> (16 * (i - 2)));
        uint32_t s2 = e4m3x2_to_f16x2(sp & 0xFFFFu);     // {s(row g), s(row g+8)}
        uint32_t sg, sg8;                                // {s_g, s_g}, {s_g8, s_g8}
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tmov.b32 %0, {lo, lo};\n\t"
            "mov.b32 %1, {hi, hi};\n\t}\n"
            : "=r"(sg), "=r"(sg8) : "r"(s2));
        uint32_t h0, h1, h2, h3;
        e2m1x8_to_f16x2(words[i], h0, h1, h2, h3);
        a[i][0] = hmul2(h0, sg);
        a[i][1] = hmul2(h1, sg8);
        a[i][2] = hmul2(h2, sg);
        a[i][3] = hmul2(h3, sg8);
    }
}

// Decode one F8 chunk's A fragments for one lane: 2 blocks x 4 registers of
// exact f16 E4M3 values (every E4M3 value is an f16 value).
__device__ __forceinline__ void decode_chunk_f8(const uint4 &cw, uint32_t (&a)[2][4]) {
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        a[w >> 1][2 * (w & 1)] = e4m3x2_to_f16x2(words[w] & 0xFFFFu);
        a[w >> 1][2 * (w & 1) + 1] = e4m3x2_to_f16x2(words[w] >> 16);
    }
}

// One F8 chunk against B (b: the lane's B fragments of the chunk's two K
// blocks): both MMAs into a fresh accumulator, then FP32 scaling of rows g
// (sw.x) and g+8 (sw.y) into acc.
__device__ __forceinline__ void chunk_mma_f8(const uint4 &cw, const uint2 &sw, const uint4 &b, float (&acc)[4]) {
    uint32_t a[2][4];
    decode_chunk_f8(cw, a);
    float t[4] = {0.f, 0.f, 0.f, 0.f};
    mma_16816(t, a[0][0], a[0][1], a[0][2], a[0][3], b.x, b.y);
    mma_16816(t, a[1][0], a[1][1], a[1][2], a[1][3], b.z, b.w);
    const float sg = __uint_as_float(sw.x), sg8 = __uint_as_float(sw.y);
    acc[0] = fmaf(sg, t[0], acc[0]);
    acc[1] = fmaf(sg, t[1], acc[1]);
    acc[2] = fmaf(sg8, t[2], acc[2]);
    acc[3] = fmaf(sg8, t[3], acc[3]);
}

// Offset of the B fragments of chunk c (format chunks along K) in an operand
// row laid out per 64 elements (128 bytes, lane q at 32q): an NVFP4 chunk is
// one such group, an F8 chunk half of one (its K blocks 2(c%2), 2(c%2)+1).
__device__ __forceinline__ int b_offset(int c, bool f8) { return f8 ? (c >> 1) * 128 + (c & 1) * 16 : c * 128; }

#endif  // __CUDACC__

}  // namespace moe
