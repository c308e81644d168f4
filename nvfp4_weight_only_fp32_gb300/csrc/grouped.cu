// grouped.cu -- row a6: the experts that many tokens selected (and the shared
// experts) as dense tensor-core contractions, for steps with more than 8
// tokens.
//
// Sources: "vLLM Day-0 support for Recursive's Flint", "Optimisation strategy"
// (the GEMV kernels are the small-batch path; above it the MoE layer runs as
// grouped GEMMs over the tokens each expert received); "Inkling 2 Small on
// vLLM: Day-0 Support", "vLLM integration and optimisation" (SwiGLU between
// gate/up and down; NVFP4 weights with 16-element E4M3 block scales).
//
// A work item is (hot slot, M-tile of 128 weight rows = 8 repacked 16-row
// tiles); blocks loop over items.  Per stage of two 64-wide K chunks:
//   warps 0-7   each decode one 16-row tile's two 576-byte chunks (E2M1 x
//               E4M3, exact in f16) straight into the A stage, laid out as
//               the tensor core's K-major operand without swizzle: 8x8 core
//               matrices of 128 contiguous bytes, K-adjacent ones 128 bytes
//               apart (LBO), row-adjacent ones 2048 bytes apart (SBO: 16 K
//               groups per row group);
//   warps 8-11  stage the slot's m tokens (gate/up: x rows times 2^-xexp;
//               down: h rows times 2^-hexp, both exact in f16) as the B
//               operand in the same layout, rows >= m zero;
//   warp 12     lane 0 issues eight tcgen05.mma kind::f16 (M=128, N=m
//               rounded up to 16, K=16) into a TMEM accumulator and commits
//               them to the stage's "empty" mbarrier; after the last stage a
//               commit to the accumulator barrier.
// Three stages ring between producers and the MMA issuer (an odd chunk count
// leaves the last stage half full).  Warps 0-7 then
// read the accumulator (tcgen05.ld, warp w owns TMEM lanes 32(w%4).. and
// half of the columns) and run the epilogue:
//   gate/up  rows 16j+r (r < 8) are gate, 16j+r+8 the matching up rows
//            (the repacked tile order), so SwiGLU pairs lanes L and L+8;
//            h = bf16(silu(g) * u) goes to the workspace with the per-pair
//            max |h|, as in the GEMV path;
//   down     y = gs * 2^hexp * acc into the FP32 workspace; the block that
//            completes a 128-row group last (shared ticket with the GEMV
//            down kernel) runs the routing-weighted combine for those rows.
// Every mbarrier wait gives up after about a second (sticky error word and a
// shared abort flag that releases the other roles); the TMEM columns are
// released on every exit path.
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kDecW = 8;                          // decode / epilogue warps
constexpr int kStgW = 4;                          // B staging warps
constexpr int kMmaW = kDecW + kStgW;              // MMA-issuing warp
constexpr int kGW = kMmaW + 1;
constexpr int kGT = 32 * kGW;
constexpr int kCPS = 2;                           // 64-wide K chunks per pipeline stage
constexpr int kNS = 3;                            // pipeline stages
constexpr int kLA = 2;                            // B-operand chunks in flight (raw copies)
constexpr int kMT = 128;                          // weight rows per item (8 tiles)
constexpr int kNmax = kMaxTokens;                 // tokens per slot
constexpr uint32_t kLBO = 128;                    // K-adjacent core matrices
constexpr int kScratch = kMaxTokens * (kMaxTopK + kMaxShared) * 8;   // combine's pair table
constexpr int kCHA = 4;                           // chunks per raw-weight segment
constexpr int kRWA = 3;                           // raw-weight segments per decode warp
static_assert((kLA & (kLA - 1)) == 0, "kLA is a power of two");
constexpr int kMaxItems = 128;                    // work items per block
constexpr unsigned long long kWaitNs = 1000000000ull;

// Shared-memory and TMEM geometry.  f16 operands (W4A16): a 64-wide K chunk
// of a row is 128 bytes, 8 core matrices.  E2M1 operands (W4A4, block-scaled
// MMA): 32 bytes, 2 core matrices, plus one 32-bit word of four E4M3 scales
// per row and chunk, staged in shared memory on the way to TMEM.
template <bool FP4>
struct Geo {
    static constexpr int kRowB = FP4 ? 32 : kChunkK * 2;       // bytes of one row of a chunk
    static constexpr uint32_t kSBO = kCPS * kRowB / 16 * 128;   // row-adjacent core matrices
    static constexpr int kAStage = kMT * kRowB * kCPS;          // f16 32 KB, E2M1 8 KB
    static constexpr int kBStage = kNmax * kRowB * kCPS;        // f16 16 KB, E2M1 4 KB
    static constexpr int kSfStage = FP4 ? kCPS * kMT * 4 : 0;   // the A scale words of a stage
    static constexpr int kScrOff = kNS * (kAStage + kBStage + kSfStage);
    static constexpr int kRawOff = kScrOff + kScratch;
    static constexpr int kBRawOff = kRawOff + kDecW * kRWA * kCHA * kChunkBytes;
    // one chunk of the slot's token rows as stored: f16 path the BF16 rows
    // (8 KB); E2M1 path the codes (2 KB, [K group][token][16 bytes]) and each
    // B warp's own copy of the 64 tokens' scale words
    static constexpr int kBRawStage = FP4 ? kNmax * 32 + kStgW * kNmax * 4 : kNmax * kChunkK * 2;
    static constexpr int kSmem = kBRawOff + kLA * kBRawStage;
    // TMEM: accumulator columns 0..63 (N <= 64); E2M1 path: per (stage,
    // chunk) four columns of A scales from kSfaCol and four of B scales
    // from kSfbCol (block-scaled MMAs take scale addresses that are
    // multiples of four columns: row r at lane r % 32, column r / 32)
    static constexpr uint32_t kSfaCol = 64, kSfbCol = kSfaCol + 4 * kNS * kCPS;
    static constexpr uint32_t kTmemCols = FP4 ? 128 : 64;        // a power of two >= 32
    static_assert(!FP4 || kSfbCol + 4 * kNS * kCPS <= kTmemCols, "scale columns fit the allocation");
};

__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// No-swizzle K-major shared-memory operand descriptor (tcgen05): start
// address, leading (K) and stride (row) byte offsets, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(kLBO >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46);
}

// Instruction descriptor: kind::f16, A = B = f16, D = f32, both K-major.
__device__ __forceinline__ uint32_t instr_desc(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor: kind::mxf4nvf4 block-scaled, A = B = E2M1, scales
// E4M3 (one per 16 elements: scale_vec::4X), D = f32, both K-major.
__device__ __forceinline__ uint32_t instr_desc_fp4(int M, int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 7) << 27);
}

// Byte `b` of each of four words, in order.
__device__ __forceinline__ uint32_t gather4(uint32_t a, uint32_t b0, uint32_t c, uint32_t d, uint32_t b) {
    const uint32_t sel = b | ((b + 4) << 4);
    return __byte_perm(__byte_perm(a, b0, sel), __byte_perm(c, d, sel), 0x5410);
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// 32 lanes (this warp's quadrant) x 2 consecutive TMEM columns.
__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint32_t v0, uint32_t v1) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};\n" ::"r"(taddr), "r"(v0), "r"(v1)
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// 16-byte asynchronous copy global -> shared (L2 only), and its groups.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(b)) : "memory");
}

// Bounded wait; gives up (error word, abort flag) after kWaitNs or as soon
// as another role has given up.
__device__ __forceinline__ bool gwait(uint64_t *b, unsigned parity, volatile int *abort, int *err) {
    if (mbar_try_wait(b, parity)) return true;
    const unsigned long long t0 = gtimer();
    while (!mbar_try_wait(b, parity)) {
        if (*abort) return false;
        if (gtimer() - t0 > kWaitNs) {
            *abort = 1;
            atomicExch(err, 1);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

// 16 consecutive accumulator columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ int hexp_of(unsigned bits) {
    // exact power-of-two prescale of an h row from its max |h| (also upward)
    return max(-100, exp_for_f16(__uint_as_float(bits)));
}

// MODE 0 gate/up + SwiGLU, 1 down + combine; FP4: W4A4 layers, whose
// activations are E2M1 codes with E4M3 block scales, multiplied by
// tcgen05.mma kind::mxf4nvf4 (no decode: the weights' codes are only
// rearranged into the operand layout, their scales go to TMEM).
template <int MODE, bool FP4>
__global__ void __launch_bounds__(kGT, 1) grouped_kernel(DevLayer d, const __nv_bfloat16 *__restrict__ x, int T,
                                                         __nv_bfloat16 *__restrict__ out) {
    using G = Geo<FP4>;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_full[kNS], s_empty[kNS], s_accf, s_acce;
    __shared__ __align__(8) uint64_t s_rbar[kDecW][kRWA];
    __shared__ uint32_t s_taddr;
    __shared__ int s_abort;
    __shared__ int s_last;
    __shared__ int s_t16[kMT / 16];   // down: the 16-row tiles this item completed last
    // this block's items: first byte of tile 8mt (warp w adds w tiles), K
    // chunks, tokens, first pair, expert (< 0: shared), M-tile
    __shared__ const uint8_t *s_it_base[kMaxItems];
    __shared__ int s_it_nc[kMaxItems], s_it_m[kMaxItems], s_it_p0[kMaxItems], s_it_e[kMaxItems], s_it_mt[kMaxItems];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    uint8_t *sA = smem;
    uint8_t *sB = smem + kNS * G::kAStage;
    uint32_t *sSF = reinterpret_cast<uint32_t *>(smem + kNS * (G::kAStage + G::kBStage));   // FP4 only
    int *s_pair = reinterpret_cast<int *>(smem + G::kScrOff);
    float *s_pw = reinterpret_cast<float *>(smem + G::kScrOff + kScratch / 2);
    uint8_t *rraw = smem + G::kRawOff + (size_t)(warp < kDecW ? warp : 0) * kRWA * kCHA * kChunkBytes;
    volatile int *abort = &s_abort;
    const uint64_t pol = evict_first_policy();

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&s_full[i], kDecW + kStgW);
            mbar_init(&s_empty[i], 1);
        }
        mbar_init(&s_accf, 1);
        mbar_init(&s_acce, kDecW);
        for (int w = 0; w < kDecW; ++w)
            for (int i = 0; i < kRWA; ++i) mbar_init(&s_rbar[w][i], 1);
        s_abort = 0;
        fence_proxy_async();
    }
    if (warp == kMmaW) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&s_taddr)),
                     "r"(G::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    MOE_TRACE_POINT(3 + MODE, 0);
    // The router's tables are final when this kernel starts (the GEMV kernel
    // before it released it only after its own dependency wait), and what
    // this kernel reads besides them is x (gate/up) or h (down: complete
    // before the GEMV down kernel released it).  So it starts at once; it
    // waits on its predecessor only at the end, which keeps the chain's
    // completion order.
    pdl_trigger();
    const int nhot = __ldcg(d.nhot);
    const int ns = __ldcg(d.nslots);
    const int MTper = MODE == 0 ? d.I / 64 : d.H / kMT;   // M-tiles of a routed slot
    const int MTs = MODE == 0 ? d.Is / 64 : d.H / kMT;    // of a shared slot
    // items: hot slots in slot order (shared ones first), each with its M-tiles
    int sh = 0;
    if (MODE == 0)
        for (int h = 0; h < nhot && h < d.S; ++h) sh += __ldcg(d.hot_slots + h) < d.S;
    const int nitems = MODE == 0 ? sh * MTs + (nhot - sh) * MTper : nhot * MTper;
    const int nmy = blockIdx.x < nitems ? min(kMaxItems, (nitems - blockIdx.x + gridDim.x - 1) / gridDim.x) : 0;
    if (threadIdx.x < nmy) {
        const int it = blockIdx.x + threadIdx.x * gridDim.x;
        int h, mt;
        if (MODE == 0 && it < sh * MTs) {
            h = it / MTs;
            mt = it - h * MTs;
        } else {
            const int i2 = MODE == 0 ? it - sh * MTs : it;
            h = (MODE == 0 ? sh : 0) + i2 / MTper;
            mt = i2 % MTper;
        }
        const int slot = __ldcg(d.hot_slots + h);
        const int e = __ldcg(d.slot_expert + slot);
        const bool shared = e < 0;
        const int NC = MODE == 0 ? d.H / kChunkK : (shared ? d.Is : d.I) / kChunkK;
        const uint8_t *wbase = MODE == 0 ? (shared ? d.sw13r + (size_t)(-e - 1) * d.s13_stride
                                                   : d.w13r + (size_t)e * d.e13_stride)
                                         : (shared ? d.sw2r + (size_t)(-e - 1) * d.s2_stride
                                                   : d.w2r + (size_t)e * d.e2_stride);
        s_it_base[threadIdx.x] = wbase + (size_t)(8 * mt) * NC * kChunkBytes;
        s_it_nc[threadIdx.x] = NC;
        s_it_m[threadIdx.x] = __ldcg(d.slot_m + slot);
        s_it_p0[threadIdx.x] = __ldcg(d.slot_p0 + slot);
        s_it_e[threadIdx.x] = e;
        s_it_mt[threadIdx.x] = mt;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = s_taddr;
    MOE_TRACE_POINT(3 + MODE, 1);

    // ---- raw weight ring of a decode warp: its tile's chunks of every item,
    // in segments of <= kCHA chunks, issued ahead across items (lane 0) ----
    uint64_t *rbar = s_rbar[warp < kDecW ? warp : 0];
    int ip = 0, cp = 0, n_iss = 0, n_done = 0;
    auto rissue = [&](int limit) {
        if (lane != 0) return;
        while (n_iss < limit && ip < nmy) {
            const int nc = s_it_nc[ip], n = min(kCHA, nc - cp), sl = n_iss % kRWA;
            const uint8_t *src = s_it_base[ip] + ((size_t)warp * nc + cp) * kChunkBytes;
            fence_proxy_async();
            mbar_expect_tx(rbar + sl, (unsigned)(n * kChunkBytes));
            bulk_g2s(rraw + (size_t)sl * kCHA * kChunkBytes, src, (unsigned)(n * kChunkBytes), rbar + sl, pol);
            ++n_iss;
            cp += n;
            if (cp == nc) {
                cp = 0;
                ++ip;
            }
        }
    };
    if (warp < kDecW) rissue(kRWA);

    int gc = 0;        // stages (kCPS chunks each) through the A/B ring so far
    int jc = 0;        // raw segments consumed (decode warps)
#pragma unroll 1
    for (int li = 0; li < nmy; ++li) {
        // (every role runs every item, so that the epilogue warps' named
        // barriers stay matched; after an abort the waits return at once)
        const int NC = s_it_nc[li], m = s_it_m[li], p0 = s_it_p0[li], e = s_it_e[li], mt = s_it_mt[li];
        const int N = FP4 ? kNmax : (m + 15) & ~15;   // E2M1 path: always the shape its layout was checked on
        const bool shared = e < 0;
        float gs0, gs1;
        if (MODE == 0) {
            gs0 = shared ? d.sgs13[2 * (-e - 1)] : d.gs13[2 * e];
            gs1 = shared ? d.sgs13[2 * (-e - 1) + 1] : d.gs13[2 * e + 1];
        } else {
            gs0 = shared ? d.sgs2[-e - 1] : d.gs2[e];
            gs1 = 0.f;
        }

        // The epilogue's per-column factor, loaded now so that its round trip
        // overlaps the main loop: lane i of a decode warp holds the one of
        // column 32 * half + i (gate/up: 2^xexp of the column's token; down:
        // 2^hexp of the pair).  The router's tables, x's exponents and h's
        // maxima are all final when this kernel starts.
        float col_un = 0.f;
        if (warp < kDecW) {
            const int col = 32 * (warp >> 2) + lane;
            if (col < m) {
                // (W4A4: times the row's global scale; the E2M1 operands
                // carry no power-of-two prescale)
                if (MODE == 0) {
                    const int tok = shared ? col : __ldcg(d.pair_tok + p0 + col);
                    col_un = FP4 ? __ldcg(d.gsx + tok)
                                 : pow2f(__ldcg(d.xexp + tok)) * (d.w4a4 ? __ldcg(d.gsx + tok) : 1.f);
                } else {
                    col_un = FP4 ? __ldcg(d.gsh + p0 + col)
                                 : pow2f(hexp_of(__ldcg(d.hmax + p0 + col))) *
                                       (d.w4a4 ? __ldcg(d.gsh + p0 + col) : 1.f);
                }
            }
        }

        if (warp < kDecW) {
            // ---- A producer: tile 8mt + warp, from the raw ring ----
            int oc = 0, cseg = 0;
#pragma unroll 1
            for (int c0 = 0; c0 < NC; c0 += kCPS) {
                const int gcc = gc + c0 / kCPS, st = gcc % kNS, nch = min(kCPS, NC - c0);
                const bool go = gwait(&s_empty[st], ((unsigned)(gcc / kNS) & 1u) ^ 1u, abort, d.err);
#pragma unroll 1
                for (int h = 0; h < nch; ++h) {
                    if (oc == 0 && !*abort) {
                        if (gwait(rbar + jc % kRWA, (unsigned)((jc / kRWA) & 1), abort, d.err)) n_done = jc + 1;
                    }
                    if (go) {
                        const uint8_t *ch = rraw + ((size_t)(jc % kRWA) * kCHA + oc) * kChunkBytes;
                        uint2 sw;
                        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n"
                                     : "=r"(sw.x), "=r"(sw.y) : "r"(smem_u32(ch + kCodeBytes + 8 * g)));
                        if constexpr (FP4) {
                            // The quad's 64 bytes hold rows g and g + 8 of the
                            // tile (lane 4g + p: bytes 16p..; its word i, byte
                            // b: row g + 8(b & 1), K byte 8i + p + 4(b >> 1)).
                            // Lane q writes row g + 8(q & 1), K bytes
                            // 16(q >> 1) .. + 15: one core-matrix row.
                            const uint8_t *qb = ch + 64 * g;
                            const uint4 u0 = lds128(qb), u1 = lds128(qb + 16), u2 = lds128(qb + 32),
                                        u3 = lds128(qb + 48);
                            const uint32_t rb = q & 1, kb = q >> 1;
                            const uint32_t a0 = kb ? u0.z : u0.x, a1 = kb ? u1.z : u1.x, a2 = kb ? u2.z : u2.x,
                                           a3 = kb ? u3.z : u3.x;
                            const uint32_t b0 = kb ? u0.w : u0.y, b1 = kb ? u1.w : u1.y, b2 = kb ? u2.w : u2.y,
                                           b3 = kb ? u3.w : u3.y;
                            uint4 o;
                            o.x = gather4(a0, a1, a2, a3, rb);
                            o.y = gather4(a0, a1, a2, a3, 2 | rb);
                            o.z = gather4(b0, b1, b2, b3, rb);
                            o.w = gather4(b0, b1, b2, b3, 2 | rb);
                            *reinterpret_cast<uint4 *>(sA + (size_t)st * G::kAStage + (2 * warp + rb) * G::kSBO +
                                                       (2 * h + kb) * kLBO + g * 16) = o;
                            // the four K-block scales of rows g (lane q = 0)
                            // and g + 8 (q = 1), byte j = K block j
                            if (q < 2)
                                sSF[(st * kCPS + h) * kMT + 16 * warp + g + 8 * q] =
                                    __byte_perm(sw.x, sw.y, q ? 0x7531 : 0x6420);
                        } else {
                            const uint4 cw = lds128(ch + 16 * lane);
                            uint32_t a[4][4];
                            decode_chunk(cw, sw, a);
                            // chunk h of the stage: K groups 8h .. 8h + 7.
                            // a[i][b] is the MMA fragment of an 8x8 block (rows
                            // + 8(b & 1), K group 2i + (b >> 1)): one stmatrix
                            // per i stores four of them, lane t giving row t % 8
                            // of block b = t / 8 (each block one 128-byte core
                            // matrix).
                            const int bt = lane >> 3;
                            const uint32_t As = smem_u32(sA + (size_t)st * G::kAStage +
                                                         (2 * warp + (bt & 1)) * G::kSBO +
                                                         (8 * h + (bt >> 1)) * kLBO + (lane & 7) * 16);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                asm volatile(
                                    "stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(
                                        As + 2 * i * kLBO),
                                    "r"(a[i][0]), "r"(a[i][1]), "r"(a[i][2]), "r"(a[i][3])
                                    : "memory");
                        }
                    }
                    if (++oc == min(kCHA, NC - cseg)) {
                        cseg += oc;
                        oc = 0;
                        ++jc;
                        if (!*abort) rissue(jc + kRWA);
                    }
                }
                if constexpr (FP4) {
                    // the stage's A scales to TMEM, in every lane quadrant:
                    // quadrant warp % 4 gets columns 2(warp / 4), +1 (rows
                    // 64(warp / 4) .. + 63) from the words all eight decode
                    // warps staged (every decode warp passes this barrier
                    // once per stage, aborted or not)
                    asm volatile("bar.sync 2, %0;\n" ::"r"(32 * kDecW) : "memory");
                    if (__all_sync(0xffffffffu, go)) {
                        const int j0 = 2 * (warp >> 2);
                        for (int h = 0; h < nch; ++h) {
                            const uint32_t *w = sSF + (st * kCPS + h) * kMT;
                            tmem_st2(taddr + ((uint32_t)(32 * (warp & 3)) << 16) + G::kSfaCol + 4 * (st * kCPS + h) +
                                         j0,
                                     w[32 * j0 + lane], w[32 * (j0 + 1) + lane]);
                        }
                        tmem_st_wait();
                    }
                    tc_fence_before();
                }
                if (go) fence_proxy_async();
                __syncwarp();
                if (go && lane == 0) mbar_arrive(&s_full[st]);
                if (li == 0 && c0 == 0) MOE_TRACE_POINT(3 + MODE, 3);
            }
        } else if (warp < kMmaW) {
            // ---- B producer: the slot's m tokens (rows >= m zero).  Each
            // thread copies its own pieces of chunk c + kLA - 1 ahead
            // (cp.async into a raw ring; a thread reads back only what it
            // copied itself, so its own group waits order it) and converts
            // chunk c into the stage ----
            if constexpr (FP4) {
                // E2M1 path: thread tb copies K group kb = tb / 64 (16
                // bytes) of token n = tb % 64 of each chunk, kLA - 1 chunks
                // ahead, into the raw ring ([K group][token][16 bytes]) and
                // from there into the stage (rows >= m zero); each B warp
                // also copies the 64 tokens' scale words of the chunk (lane
                // L: tokens L and L + 32) and writes them to TMEM in its own
                // lane quadrant (columns: tokens 0-31, 32-63).
                const int tb = threadIdx.x - 32 * kDecW;      // 0..127
                const int n = tb & 63, kb = tb >> 6, wq = tb >> 5;
                const uint8_t *csrc = nullptr;
                const uint8_t *ssrc[2] = {nullptr, nullptr};
                if (n < m) {
                    if (MODE == 0) {
                        const int tok = shared ? n : __ldcg(d.pair_tok + p0 + n);
                        csrc = d.xq4 + (size_t)tok * (d.H / 2) + 16 * kb;
                    } else {
                        csrc = d.hq4 + (size_t)(p0 + n) * (d.Imax / 2) + 16 * kb;
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int nn = lane + 32 * u;
                    if (nn < m) {
                        if (MODE == 0) {
                            const int tok = shared ? nn : __ldcg(d.pair_tok + p0 + nn);
                            ssrc[u] = d.xsf + (size_t)tok * (d.H / 16);
                        } else {
                            ssrc[u] = d.hsf + (size_t)(p0 + nn) * (d.Imax / 16);
                        }
                    }
                }
                uint8_t *braw = smem + G::kBRawOff;
                auto bissue = [&](int c) {
                    if (c < NC) {
                        uint8_t *slot = braw + (size_t)(c & (kLA - 1)) * G::kBRawStage;
                        if (csrc) cp_async16(slot + kb * (kNmax * 16) + n * 16, csrc + 32 * c);
#pragma unroll
                        for (int u = 0; u < 2; ++u)
                            if (ssrc[u])
                                cp_async4(slot + kNmax * 32 + wq * (kNmax * 4) + (lane + 32 * u) * 4, ssrc[u] + 4 * c);
                    }
                    cp_async_commit();
                };
#pragma unroll
                for (int j = 0; j < kLA; ++j) bissue(j);
#pragma unroll 1
                for (int c0 = 0; c0 < NC; c0 += kCPS) {
                    const int gcc = gc + c0 / kCPS, st = gcc % kNS, nch = min(kCPS, NC - c0);
                    const bool go = gwait(&s_empty[st], ((unsigned)(gcc / kNS) & 1u) ^ 1u, abort, d.err);
                    const bool gw = __all_sync(0xffffffffu, go);
#pragma unroll 1
                    for (int h = 0; h < nch; ++h) {
                        const int c = c0 + h;
                        cp_async_wait<kLA - 1>();
                        const uint8_t *slot = braw + (size_t)(c & (kLA - 1)) * G::kBRawStage;
                        if (go) {
                            const uint4 v = csrc ? lds128(slot + kb * (kNmax * 16) + n * 16) : make_uint4(0u, 0u, 0u, 0u);
                            *reinterpret_cast<uint4 *>(sB + (size_t)st * G::kBStage + (n >> 3) * G::kSBO +
                                                       (2 * h + kb) * kLBO + (n & 7) * 16) = v;
                        }
                        if (gw) {
                            const uint32_t *sf = reinterpret_cast<const uint32_t *>(slot + kNmax * 32 + wq * (kNmax * 4));
                            tmem_st2(taddr + ((uint32_t)(32 * wq) << 16) + G::kSfbCol + 4 * (st * kCPS + h),
                                     ssrc[0] ? sf[lane] : 0u, ssrc[1] ? sf[lane + 32] : 0u);
                        }
                        bissue(c + kLA);
                    }
                    if (gw) tmem_st_wait();
                    tc_fence_before();
                    if (go) fence_proxy_async();
                    __syncwarp();
                    if (go && lane == 0) mbar_arrive(&s_full[st]);
                    if (li == 0 && c0 == 0) MOE_TRACE_POINT_AT(3 + MODE, 6, 32 * kDecW);
                }
                if (li == 0) MOE_TRACE_POINT_AT(3 + MODE, 7, 32 * kDecW);
            } else {
                // Thread tb takes K group kg of tokens nlo + 8 * nhi + 16 * u:
                // the eight lanes of a quarter warp (one 16-byte store phase)
                // write eight different token rows of one core matrix, so
                // their stores hit eight different bank groups.
                const int tb = threadIdx.x - 32 * kDecW;      // 0..127
                const int nlo = tb & 7, kg = (tb >> 3) & 7, nhi = tb >> 6;
                const uint4 *src[4];
                float sc[4];
    #pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int n = nlo + 8 * nhi + 16 * u;
                    src[u] = nullptr;
                    sc[u] = 0.f;
                    if (n < m) {
                        if (MODE == 0) {
                            const int tok = shared ? n : __ldcg(d.pair_tok + p0 + n);
                            src[u] = reinterpret_cast<const uint4 *>(x + (size_t)tok * d.H);
                            sc[u] = pow2f(-__ldcg(d.xexp + tok));
                        } else {
                            src[u] = reinterpret_cast<const uint4 *>(d.h_ws + (size_t)(p0 + n) * d.Imax);
                            sc[u] = pow2f(-hexp_of(__ldcg(d.hmax + p0 + n)));
                        }
                    }
                }
                // raw ring: token row n of a chunk is 128 bytes, its K groups
                // XOR-swizzled by n % 8 (= nlo) so that a quarter warp's pieces
                // fall in different bank groups here too
                uint8_t *braw = smem + G::kBRawOff + ((kg ^ nlo) << 4);
                // one commit group per chunk index (empty past the end), so that
                // "chunk c landed" is always "at most kLA - 1 groups pending"
                auto bissue = [&](int c) {
                    if (c < NC) {
    #pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int n = nlo + 8 * nhi + 16 * u;
                            if (src[u])
                                cp_async16(braw + (size_t)((c & (kLA - 1)) * kNmax + n) * 128, src[u] + c * 8 + kg);
                        }
                    }
                    cp_async_commit();
                };
    #pragma unroll
                for (int j = 0; j < kLA; ++j) bissue(j);
    #pragma unroll 1
                for (int c0 = 0; c0 < NC; c0 += kCPS) {
                    const int gcc = gc + c0 / kCPS, st = gcc % kNS, nch = min(kCPS, NC - c0);
                    const bool go = gwait(&s_empty[st], ((unsigned)(gcc / kNS) & 1u) ^ 1u, abort, d.err);
    #pragma unroll 1
                    for (int h = 0; h < nch; ++h) {
                        const int c = c0 + h;
                        cp_async_wait<kLA - 1>();
                        if (go) {
                            // chunk h of the stage: K groups 8h .. 8h + 7
                            uint8_t *Bs = sB + (size_t)st * G::kBStage + 8 * h * kLBO;
    #pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int n = nlo + 8 * nhi + 16 * u;
                                if (n < N) {
                                    uint4 o = make_uint4(0u, 0u, 0u, 0u);
                                    if (src[u]) {
                                        const uint4 v = lds128(braw + (size_t)((c & (kLA - 1)) * kNmax + n) * 128);
                                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                                        uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
    #pragma unroll
                                        for (int i = 0; i < 4; ++i)
                                            ow[i] = pack_f16x2(__uint_as_float(w4[i] << 16) * sc[u],
                                                               __uint_as_float(w4[i] & 0xFFFF0000u) * sc[u]);
                                    }
                                    *reinterpret_cast<uint4 *>(Bs + (n >> 3) * G::kSBO + kg * kLBO + (n & 7) * 16) = o;
                                }
                            }
                        }
                        bissue(c + kLA);
                    }
                    if (go) fence_proxy_async();
                    __syncwarp();
                    if (go && lane == 0) mbar_arrive(&s_full[st]);
                    if (li == 0 && c0 == 0) MOE_TRACE_POINT_AT(3 + MODE, 6, 32 * kDecW);
                }
                if (li == 0) MOE_TRACE_POINT_AT(3 + MODE, 7, 32 * kDecW);
            }
        } else if (lane == 0) {
            // ---- MMA issuer ----
            const uint32_t idesc = FP4 ? instr_desc_fp4(kMT, N) : instr_desc(kMT, N);
            bool go = gwait(&s_acce, ((unsigned)li & 1u) ^ 1u, abort, d.err);   // accumulator read out
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < NC && go; c0 += kCPS) {
                const int gcc = gc + c0 / kCPS, st = gcc % kNS, nch = min(kCPS, NC - c0);
                if (!gwait(&s_full[st], (unsigned)(gcc / kNS) & 1u, abort, d.err)) {
                    go = false;
                    break;
                }
                tc_fence_after();
                if (li == 0 && c0 == 0) MOE_TRACE_POINT_AT(3 + MODE, 4, 32 * kMmaW);
                const uint32_t a0 = smem_u32(sA + (size_t)st * G::kAStage),
                               b0 = smem_u32(sB + (size_t)st * G::kBStage);
                if constexpr (FP4) {
                    // one K=64 MMA per chunk, its scales at the stage's columns
#pragma unroll
                    for (int h = 0; h < kCPS; ++h) {
                        if (h >= nch) break;
                        const uint64_t da = smem_desc(a0 + h * 2 * kLBO, G::kSBO),
                                       db = smem_desc(b0 + h * 2 * kLBO, G::kSBO);
                        const uint32_t acc = (c0 > 0 || h > 0) ? 1u : 0u;
                        const uint32_t col = 4 * (st * kCPS + h);
                        asm volatile(
                            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
                            "[%4], [%5], p;\n\t}\n" ::"r"(taddr),
                            "l"(da), "l"(db), "r"(idesc), "r"(taddr + G::kSfaCol + col), "r"(taddr + G::kSfbCol + col),
                            "r"(acc)
                            : "memory");
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < 4 * kCPS; ++ks) {
                        if (ks >= 4 * nch) break;
                        const uint64_t da = smem_desc(a0 + ks * 2 * kLBO, G::kSBO),
                                       db = smem_desc(b0 + ks * 2 * kLBO, G::kSBO);
                        const uint32_t acc = (c0 > 0 || ks > 0) ? 1u : 0u;
                        asm volatile(
                            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(taddr),
                            "l"(da), "l"(db), "r"(idesc), "r"(acc)
                            : "memory");
                    }
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                                 smem_u32(&s_empty[st]))
                             : "memory");
            }
            if (go)
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                                 smem_u32(&s_accf))
                             : "memory");
            if (li == 0) MOE_TRACE_POINT_AT(3 + MODE, 5, 32 * kMmaW);
        }
        gc += (NC + kCPS - 1) / kCPS;
        if (li == 0) MOE_TRACE_POINT(3 + MODE, 2);

        // ---- epilogue: warps 0-7 ----
        if (warp < kDecW) {
            const bool ok = gwait(&s_accf, (unsigned)li & 1u, abort, d.err);
            tc_fence_after();
            if (li == 0) MOE_TRACE_POINT(3 + MODE, 10);
            const int qd = warp & 3, half = warp >> 2;
            float v[32];
            if (ok) {
                const uint32_t ta = taddr + ((uint32_t)(32 * qd) << 16) + (uint32_t)(32 * half);
                if (32 * half < N) {
                    float t16[16];
                    tmem_ld16(ta, t16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = t16[i];
                    if (32 * half + 16 < N) {
                        tmem_ld16(ta + 16, t16);
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[16 + i] = t16[i];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_acce);
            if (ok && 32 * half < N) {
                const int row = 32 * qd + lane;            // row of the M-tile
                if (MODE == 0) {
                    // Two columns per step: lanes rr < 8 hold gate rows and
                    // take column i (up from lane + 8), lanes rr >= 8 hold the
                    // matching up rows and take column i + 1 (gate from
                    // lane - 8), so every lane evaluates one SwiGLU.
                    const int j = row >> 4, rr = row & 15;
                    const bool hi = rr >= 8;
                    const int n_int = 8 * (8 * mt + j) + (rr & 7);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const float from_hi = __shfl_down_sync(0xffffffffu, v[i], 8);
                        const float from_lo = __shfl_up_sync(0xffffffffu, v[i + 1], 8);
                        const float graw = hi ? from_lo : v[i], uraw = hi ? v[i + 1] : from_hi;
                        const int ci = i + (hi ? 1 : 0);
                        const int col = 32 * half + ci;
                        const float un = __shfl_sync(0xffffffffu, col_un, ci);
                        float habs = 0.f;
                        if (col < m) {
                            const int p = p0 + col;
                            const float gt = graw * gs0 * un, uv = uraw * gs1 * un;
                            const __nv_bfloat16 hb = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * uv);
                            d.h_ws[(size_t)p * d.Imax + n_int] = hb;
                            habs = fabsf(__bfloat162float(hb));
                        }
                        // max over the 16 rows of each column: lanes 0-7 and
                        // 16-23 hold column i, lanes 8-15 and 24-31 column i + 1
                        habs = fmaxf(habs, __shfl_xor_sync(0xffffffffu, habs, 1));
                        habs = fmaxf(habs, __shfl_xor_sync(0xffffffffu, habs, 2));
                        habs = fmaxf(habs, __shfl_xor_sync(0xffffffffu, habs, 4));
                        habs = fmaxf(habs, __shfl_xor_sync(0xffffffffu, habs, 16));
                        if (col < m && (lane & 23) == 0) atomicMax(d.hmax + p0 + col, __float_as_uint(habs));
                    }
                } else {
                    const int orow = kMT * mt + row;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int col = 32 * half + i;
                        const float un = __shfl_sync(0xffffffffu, col_un, i);
                        if (col < m) d.y_ws[(size_t)(p0 + col) * d.H + orow] = v[i] * gs0 * un;
                    }
                }
            }
            if (MODE == 1 && !d.tick16) {
                // ticket shared with the per-slot GEMV down kernel: ns
                // arrivals per 128-row group; the last one combines those rows
                asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory");
                if (threadIdx.x == 0) {
                    __threadfence();
                    s_last = !*abort && atomicAdd(d.down_cnt + mt, 1u) == (unsigned)(ns - 1);
                }
                asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory");
                if (s_last) {
                    __threadfence();
                    combine_rows(d, T, out, kMT * mt, kMT, s_pair, s_pw, threadIdx.x, 32 * kDecW,
                                 [] { asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory"); });
                    if (threadIdx.x == 0) d.down_cnt[mt] = 0u;
                }
                asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory");
            } else if (MODE == 1) {
                // tickets shared with the wave down kernel: ns arrivals per
                // 16-row tile; the last one combines that tile's rows
                asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory");
                if (threadIdx.x < kMT / 16) {
                    __threadfence();
                    const bool last = !*abort && atomicAdd(d.down_cnt + (kMT / 16) * mt + threadIdx.x, 1u) ==
                                                     (unsigned)(ns - 1);
                    s_t16[threadIdx.x] = last;
                }
                asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory");
                unsigned lm = 0u;
#pragma unroll
                for (int t16 = 0; t16 < kMT / 16; ++t16) lm |= (s_t16[t16] ? 1u : 0u) << t16;
                asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory");
                if (lm) __threadfence();
                while (lm) {
                    // one combine per run of consecutive tiles (usually all
                    // eight: this kernel runs after the GEMV down kernel)
                    const int t0 = __ffs(lm) - 1;
                    int t1 = t0;
                    while (t1 + 1 < kMT / 16 && ((lm >> (t1 + 1)) & 1u)) ++t1;
                    lm &= ~(((2u << t1) - 1u) & ~((1u << t0) - 1u));
                    combine_rows(d, T, out, kMT * mt + 16 * t0, 16 * (t1 - t0 + 1), s_pair, s_pw, threadIdx.x,
                                 32 * kDecW,
                                 [] { asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory"); });
                    asm volatile("bar.sync 1, %0;\n" ::"r"(32 * kDecW) : "memory");
                    if (threadIdx.x <= t1 - t0) d.down_cnt[(kMT / 16) * mt + t0 + threadIdx.x] = 0u;
                }
            }
        }
    }
    MOE_TRACE_POINT(3 + MODE, 8);
    MOE_TRACE_VALUE(3 + MODE, 12, nmy);
    // the issuer's last commit covers all of its MMAs: wait for it before
    // the columns are released; decode warps wait for raw copies never used
    if (warp == kMmaW && lane == 0 && nmy > 0 && !*abort) gwait(&s_accf, (unsigned)(nmy - 1) & 1u, abort, d.err);
    if (warp >= kDecW && warp < kMmaW) cp_async_wait_all();   // B copies (all landed or empty)
    if (warp < kDecW && lane == 0) {
        for (int j = n_done; j < n_iss; ++j) {
            const unsigned long long t0 = gtimer();
            while (!mbar_try_wait(rbar + j % kRWA, (unsigned)((j / kRWA) & 1)) && gtimer() - t0 < kWaitNs) {
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaW)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(G::kTmemCols)
                     : "memory");
    // completion order of the chain: this kernel ends after its predecessor
    pdl_wait();
    MOE_TRACE_POINT(3 + MODE, 9);
}

template <int MODE>
cudaError_t launch_g(const DevLayer &d, const __nv_bfloat16 *x, int T, __nv_bfloat16 *out, int sm_count,
                     cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count);
    cfg.blockDim = dim3(kGT);
    cfg.dynamicSmemBytes = d.w4a4 ? Geo<true>::kSmem : Geo<false>::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return d.w4a4 ? cudaLaunchKernelEx(&cfg, grouped_kernel<MODE, true>, d, x, T, out)
                  : cudaLaunchKernelEx(&cfg, grouped_kernel<MODE, false>, d, x, T, out);
}

}  // namespace

// Shapes the grouped kernels take: 128-row M-tiles of every matrix (I, Is
// multiples of 64 for gate/up's interleaved tiles, H of 128 for down).
bool grouped_supported(const DevLayer &d, int sm_count) {
    if (!(d.H % kMT == 0 && d.I % 64 == 0 && (d.S == 0 || d.Is % 64 == 0) && d.max_tokens <= kNmax)) return false;
    // every block's items must fit its item table
    const int mt = std::max(std::max(d.I / 64, d.S > 0 ? d.Is / 64 : 0), d.H / kMT);
    const long items = (long)d.max_slots * mt;
    return (items + sm_count - 1) / sm_count <= kMaxItems;
}

cudaError_t launch_grouped_gate_up(const DevLayer &d, const __nv_bfloat16 *x, int T, int sm_count, cudaStream_t s) {
    return launch_g<0>(d, x, T, nullptr, sm_count, s);
}

cudaError_t launch_grouped_down(const DevLayer &d, int T, __nv_bfloat16 *out, int sm_count, cudaStream_t s) {
    return launch_g<1>(d, nullptr, T, out, sm_count, s);
}

cudaError_t prepare_grouped_kernels(int optin_bytes) {
    (void)optin_bytes;
    const int s0 = Geo<false>::kSmem, s1 = Geo<true>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(grouped_kernel<0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, s0);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, s0);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s1);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(grouped_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s1);
    return e;
}

}  // namespace moe
