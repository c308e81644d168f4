// gemv.cu -- rows a3, a4 and a5: NVFP4 weight-only GEMVs over the selected
// experts and the shared experts, and the routing-weighted combine.
//
// Sources: "vLLM Day-0 support for Recursive's Flint", "Optimisation strategy"
// (small-batch MoE kernels: the expert GEMVs read only the selected experts'
// weights; the low-latency path folds the expert combine into the adjacent
// GEMV); "Inkling 2 Small on vLLM: Day-0 Support", "vLLM integration and
// optimisation" (SwiGLU between the gate/up and the down projection; kernels
// chained with programmatic dependent launch so that each one's prologue
// overlaps the previous one's tail).
//
// Work decomposition.  A CTA (8 warps) owns one expert slot (blockIdx.y) and a
// group of 16-row weight tiles (blockIdx.x).  With T <= 8, `ksplit` warps share
// one tile by splitting K and add their partial sums in shared memory in a
// fixed order (deterministic).  Each warp streams its chunks (576 B: one
// 16-byte code load and one 8-byte scale load per lane) through a register
// ring PD chunks deep (8 for gate/up, 12 for down at up to 8 tokens),
// decodes E2M1 x E4M3 exactly into f16 A fragments
// (cvt.rn.f16x2.e2m1x2, cvt.rn.f16x2.e4m3x2, one f16x2 multiply) and issues
// mma.m16n8k16 with FP32 accumulators against the activations of the slot's
// tokens (B, staged once per CTA in shared memory, f16 after an exact
// power-of-two prescale).  The tensor core here only takes the multiply-adds
// off the CUDA cores so that decoding keeps up with HBM; the kernel is bound
// by the weight stream.
//
// Gate/up at up to 8 tokens runs, where the shape allows it, as one wave of
// 16-warp blocks that stage the step's activations once per SM and stream
// units from every slot (gemv_up_wave_kernel below); the per-slot grid ran a
// little over three waves of blocks, each staging the activations anew.
//
// Prefetch before the programmatic-launch wait: gate/up streams the shared
// experts' weights (they do not depend on routing); down streams every slot's
// weights, because by the time it starts the router has finished (the gate/up
// kernel released it only after waiting for the router), so only h is awaited.
//
// gate/up epilogue: tile rows 0..7 are gate rows and 8..15 the matching up
// rows, so lane (g, q) holds gate and up of intermediate row 8r+g for its two
// token columns: h = bf16(silu(gate) * up) is written to the workspace, and
// the row max |h| of each (expert, token) pair is published for the down
// kernel's prescale.
// down epilogue: y = gs * acc (FP32) per (pair, output row) into the
// workspace; the CTA that finishes last among the slots of a row group (atomic
// ticket, no spinning) sums sum_j w_j y_j + y_shared for those rows in a fixed
// order and writes BF16 `out`.
#include <algorithm>
#include <type_traits>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kThreads = 32 * kGemvWarps;
constexpr int kStageBudget = 96 * 1024;   // B staging budget when a slot has > 8 tokens
constexpr int kMaxRows = 64;              // staged B rows (tokens of one slot)

__device__ __forceinline__ int hexp_of(unsigned bits) {
    // exact power-of-two prescale of an h row from its max |h| (also upward)
    return max(-100, exp_for_f16(__uint_as_float(bits)));
}


template <int PD>
__device__ __forceinline__ void prefetch_ring(const uint8_t *tbase, int c_begin, int c_end, int lane,
                                              uint4 (&cb)[PD], uint2 (&sb)[PD], uint64_t pol) {
#pragma unroll
    for (int i = 0; i < PD; ++i)
        if (c_begin + i < c_end) load_chunk(tbase, c_begin + i, lane, cb[i], sb[i], pol);
}

// Stage chunks [kc0, kc0+nch) of the slot's m real B rows into shared memory
// as f16, permuted within each 64-element chunk so that lane (g, q) reads its B
// fragments of four blocks with two 16-byte loads: element kk = 16kb + 8h +
// 2q + e of a chunk sits at half index 16q + 4kb + 2h + e.  Row j comes from
// s_src[j] scaled by s_scale[j] (an exact power of two).  Loads are issued four
// at a time before any store.
template <int NTHR = kThreads>   // threads of the block taking part
__device__ __forceinline__ void stage_rows(int m, int kc0, int nch, uint8_t *bsm, int row_stride,
                                           const uint4 *const *s_src, const float *s_scale) {
    const int per_row = nch * 8;
    const int items = m * per_row;
    for (int base = threadIdx.x; base < items; base += 4 * NTHR) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int it = base + u * NTHR;
            if (it < items) {
                const int j = it / per_row, rem = it - j * per_row;
                v[u] = __ldcg(s_src[j] + (size_t)kc0 * 8 + rem);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int it = base + u * NTHR;
            if (it < items) {
                const int j = it / per_row, rem = it - j * per_row;
                const int cc = rem >> 3, part = rem & 7;
                uint32_t *dst = reinterpret_cast<uint32_t *>(bsm + (size_t)j * row_stride + cc * 128 +
                                                             (part >> 1) * 8 + (part & 1) * 4);
                const float sc = s_scale[j];
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const float lo = __uint_as_float(w[qq] << 16) * sc;
                    const float hi = __uint_as_float(w[qq] & 0xFFFF0000u) * sc;
                    dst[qq * 8] = pack_f16x2(lo, hi);
                }
            }
        }
    }
}

template <int MODE, int GMAX, int PD>
__global__ void __launch_bounds__(kThreads) gemv_kernel(DevLayer d, const __nv_bfloat16 *__restrict__ x,
                                                        int T, int ksplit, __nv_bfloat16 *__restrict__ out) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ const uint4 *s_src[kMaxRows];
    __shared__ float s_scale[kMaxRows];
    __shared__ float s_unscale[kMaxRows];
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int s = blockIdx.y;
    const int tpc = kGemvWarps / ksplit;
    const int tl = warp / ksplit, ks = warp - tl * ksplit;
    const int r = blockIdx.x * tpc + tl;
    const bool shared = s < d.S;
    const uint64_t pol = evict_first_policy();

    int m = 0, p0 = 0, NT = 0, NC = 0, NC64 = 0, ns = 0;
    bool f8 = false;                 // the slot's expert is stored as F8 chunks
    float gsa = 0.f, gsb = 0.f;
    const uint8_t *wbase = nullptr;
    uint4 cb[PD];
    uint2 sb[PD];

    MOE_TRACE_POINT(1 + MODE, 0);
    // NC: the slot's weight chunks per tile (in its format); NC64: 64-element
    // groups of K (the granularity of the B staging)
    auto slot_geometry = [&](int e) {
        f8 = e < 0 ? d.f8s : d.f8e;
        if (MODE == 0) {
            NT = (e < 0 ? d.Is : d.I) / 8;
            NC64 = d.H / kChunkK;
            NC = chunks_of(d.H, f8);
            if (e < 0) {
                const int si = -e - 1;
                gsa = d.sgs13[2 * si];
                gsb = d.sgs13[2 * si + 1];
                wbase = d.sw13r + (size_t)si * d.s13_stride;
            } else {
                gsa = d.gs13[2 * e];
                gsb = d.gs13[2 * e + 1];
                wbase = d.w13r + (size_t)e * d.e13_stride;
            }
        } else {
            NT = d.H / 16;
            NC64 = (e < 0 ? d.Is : d.I) / kChunkK;
            NC = chunks_of(e < 0 ? d.Is : d.I, f8);
            if (e < 0) {
                const int si = -e - 1;
                gsa = d.sgs2[si];
                wbase = d.sw2r + (size_t)si * d.s2_stride;
            } else {
                gsa = d.gs2[e];
                wbase = d.w2r + (size_t)e * d.e2_stride;
            }
        }
    };

    if (MODE == 0) {
        if (shared && T > 8 && d.grouped_min > 0 && T >= d.grouped_min) {   // grouped kernel's
            // every block waits before it leaves, so that "all blocks of this
            // kernel released the next one" implies the router has finished
            pdl_wait();
            pdl_trigger();
            return;
        }
        if (shared) {
            // Shared experts do not depend on routing: stream them now.
            m = T;
            p0 = s * T;
            slot_geometry(-(s + 1));
            if (r < NT)
                prefetch_ring<PD>(wbase + (size_t)r * NC * kChunkBytes, ks * NC / ksplit,
                                  (ks + 1) * NC / ksplit, lane, cb, sb, pol);
        }
        pdl_wait();
        if (!shared) {
            ns = __ldcg(d.nslots);
            if (s >= ns) {
                pdl_trigger();
                return;
            }
            m = __ldcg(d.slot_m + s);
            if (T > 8 && d.grouped_min > 0 && m >= d.grouped_min) {   // grouped kernel's
                pdl_trigger();
                return;
            }
            p0 = __ldcg(d.slot_p0 + s);
            slot_geometry(__ldcg(d.slot_expert + s));
            if (r < NT)
                prefetch_ring<PD>(wbase + (size_t)r * NC * kChunkBytes, ks * NC / ksplit,
                                  (ks + 1) * NC / ksplit, lane, cb, sb, pol);
        }
    } else {
        // The router has completed before this kernel could start: its slot
        // tables are final.  Stream this slot's weights, then wait for h.
        ns = __ldcg(d.nslots);
        if (s >= ns) {
            pdl_wait();
            pdl_trigger();
            return;
        }
        m = __ldcg(d.slot_m + s);
        if (T > 8 && d.grouped_min > 0 && m >= d.grouped_min) {   // grouped kernel's (and its ticket)
            pdl_wait();   // as above: h is complete once every block has released the next kernel
            pdl_trigger();
            return;
        }
        p0 = __ldcg(d.slot_p0 + s);
        slot_geometry(__ldcg(d.slot_expert + s));
        if (r < NT)
            prefetch_ring<PD>(wbase + (size_t)r * NC * kChunkBytes, ks * NC / ksplit,
                              (ks + 1) * NC / ksplit, lane, cb, sb, pol);
        pdl_wait();
    }
    pdl_trigger();
    MOE_TRACE_POINT(1 + MODE, 1);
    if (blockIdx.x * tpc >= NT) return;   // whole CTA beyond this slot's tiles (gate/up only)

    const bool active = r < NT;
    const uint8_t *tbase = wbase + (size_t)(active ? r : 0) * NC * kChunkBytes;
    const int c_begin = ks * NC / ksplit, c_end = (ks + 1) * NC / ksplit;
    const int mpad = (m + 7) & ~7;
    const int G = mpad >> 3;
    int ncst = NC64;                 // 64-element groups staged at a time
    if (GMAX > 1) {
        const int lim = (kStageBudget / mpad - 16) / 128;
        if (lim < NC64) ncst = max(PD, (lim / PD) * PD);
    }
    const int mult = f8 ? 2 : 1;     // weight chunks per 64-element group
    const int row_stride = ncst * 128 + 16;
    float *red = reinterpret_cast<float *>(smem + (size_t)mpad * row_stride);

    // Per-row source pointers and exact power-of-two scales.
    if (threadIdx.x < m) {
        const int j = threadIdx.x;
        int ex;
        float gq = 1.f;    // W4A4: the row's global scale
        const __nv_bfloat16 *row;
        if (MODE == 0) {
            const int tok = shared ? j : __ldcg(d.pair_tok + p0 + j);
            row = x + (size_t)tok * d.H;
            ex = __ldcg(d.xexp + tok);
            if (d.w4a4) gq = __ldcg(d.gsx + tok);
        } else {
            row = d.h_ws + (size_t)(p0 + j) * d.Imax;
            ex = hexp_of(__ldcg(d.hmax + p0 + j));
            if (d.w4a4) gq = __ldcg(d.gsh + p0 + j);
        }
        s_src[j] = reinterpret_cast<const uint4 *>(row);
        s_scale[j] = pow2f(-ex);
        s_unscale[j] = pow2f(ex) * gq;
    }
    // Zero the padding rows once; no stage writes them.
    for (int i = threadIdx.x; i < (mpad - m) * (row_stride / 16); i += kThreads)
        reinterpret_cast<uint4 *>(smem + (size_t)m * row_stride)[i] = make_uint4(0u, 0u, 0u, 0u);

    float acc[GMAX][4];
    float acc1[4] = {0.f, 0.f, 0.f, 0.f};   // one token group: blocks 1 and 3 (a chain half as long)
#pragma unroll
    for (int G2 = 0; G2 < GMAX; ++G2)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[G2][v] = 0.f;

    // The chunk loop of one stage, one instance per chunk format (the
    // format is uniform over a CTA's slot), so the NVFP4 loop carries no F8
    // code.
    auto run_chunks = [&](auto f8c, int lo, int hi, const uint8_t *brow, int cst0) {
        constexpr bool F8 = decltype(f8c)::value;
        for (int cc = lo; cc < hi; cc += PD) {
#pragma unroll
            for (int i = 0; i < PD; ++i) {
                const int c = cc + i;
                if (c < hi) {
                    const uint8_t *bp0 = brow + b_offset(c - cst0, F8);
                    if constexpr (F8) {
#pragma unroll
                        for (int G2 = 0; G2 < GMAX; ++G2)
                            if (G2 < G) chunk_mma_f8(cb[i], sb[i], lds128(bp0 + (size_t)G2 * 8 * row_stride), acc[G2]);
                    } else {
                        uint32_t a[4][4];
                        decode_chunk(cb[i], sb[i], a);
#pragma unroll
                        for (int G2 = 0; G2 < GMAX; ++G2) {
                            if (G2 < G) {
                                const uint8_t *bp = bp0 + (size_t)G2 * 8 * row_stride;
                                const uint4 b01 = lds128(bp);
                                const uint4 b23 = lds128(bp + 16);
                                float(&ac1)[4] = GMAX == 1 ? acc1 : acc[G2];
                                mma_16816(acc[G2], a[0][0], a[0][1], a[0][2], a[0][3], b01.x, b01.y);
                                mma_16816(ac1, a[1][0], a[1][1], a[1][2], a[1][3], b01.z, b01.w);
                                mma_16816(acc[G2], a[2][0], a[2][1], a[2][2], a[2][3], b23.x, b23.y);
                                mma_16816(ac1, a[3][0], a[3][1], a[3][2], a[3][3], b23.z, b23.w);
                            }
                        }
                    }
                    const int cn = c + PD;
                    if (cn < c_end) load_chunk(tbase, cn, lane, cb[i], sb[i], pol);
                }
            }
        }
    };
    for (int st0 = 0; st0 < NC64; st0 += ncst) {
        const int st1 = min(NC64, st0 + ncst);
        __syncthreads();
        stage_rows(m, st0, st1 - st0, smem, row_stride, s_src, s_scale);
        __syncthreads();
        MOE_TRACE_POINT(1 + MODE, 2);
        if (active) {
            const int lo = max(st0 * mult, c_begin), hi = min(st1 * mult, c_end);
            const uint8_t *brow = smem + (size_t)g * row_stride + q * 32;
            if (f8) run_chunks(std::true_type{}, lo, hi, brow, st0 * mult);
            else run_chunks(std::false_type{}, lo, hi, brow, st0 * mult);
        }
    }

    MOE_TRACE_POINT(1 + MODE, 3);
    if (GMAX == 1) {
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[0][v] += acc1[v];
    }
    if (ksplit > 1) {
        // Fixed-order K reduction across the warps sharing a tile.
        if (ks > 0) {
            float *rp = red + (size_t)((tl * (ksplit - 1) + (ks - 1)) * 4) * 32;
#pragma unroll
            for (int v = 0; v < 4; ++v) rp[v * 32 + lane] = acc[0][v];
        }
        __syncthreads();
        if (ks == 0) {
            for (int k2 = 1; k2 < ksplit; ++k2) {
                const float *rp = red + (size_t)((tl * (ksplit - 1) + (k2 - 1)) * 4) * 32;
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[0][v] += rp[v * 32 + lane];
            }
        }
    }
    const bool writer = ks == 0 && active;
    MOE_TRACE_POINT(1 + MODE, 4);

    if (MODE == 0) {
        if (!writer) return;
        const int n = 8 * r + g;
#pragma unroll
        for (int G2 = 0; G2 < GMAX; ++G2) {
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int col = 8 * G2 + 2 * q + e2;
                const bool ok = G2 < G && col < m;
                float habs = 0.f;
                if (ok) {
                    const int p = p0 + col;
                    const float sc = s_unscale[col];
                    const float gt = acc[G2][e2] * gsa * sc;
                    const float up = acc[G2][2 + e2] * gsb * sc;
                    const float hv = gt / (1.0f + expf(-gt)) * up;
                    const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                    d.h_ws[(size_t)p * d.Imax + n] = hb;
                    habs = fabsf(__bfloat162float(hb));
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1)
                    habs = fmaxf(habs, __shfl_xor_sync(0xffffffffu, habs, off));
                if (ok && g == 0) atomicMax(d.hmax + p0 + col, __float_as_uint(habs));
            }
        }
        return;
    }

    // ---- down: write y, then the last slot CTA of this row group combines ----
    if (writer) {
#pragma unroll
        for (int G2 = 0; G2 < GMAX; ++G2) {
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int col = 8 * G2 + 2 * q + e2;
                if (G2 < G && col < m) {
                    const int p = p0 + col;
                    const float sc = s_unscale[col] * gsa;
                    float *yp = d.y_ws + (size_t)p * d.H + 16 * r + g;
                    yp[0] = acc[G2][e2] * sc;
                    yp[8] = acc[G2][2 + e2] * sc;
                }
            }
        }
    }
    __syncthreads();
    MOE_TRACE_POINT(2, 5);
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(d.down_cnt + blockIdx.x, 1u) == (unsigned)(ns - 1);
    }
    __syncthreads();
    MOE_TRACE_POINT(2, 6);
    if (!s_last) return;
    __threadfence();

    int *s_pair = reinterpret_cast<int *>(smem);                       // [T, P]
    float *s_pw = reinterpret_cast<float *>(smem + (size_t)kMaxTokens * 16 * sizeof(int));
    const int row0 = blockIdx.x * tpc * 16;
    combine_rows(d, T, out, row0, min(d.H, row0 + tpc * 16) - row0, s_pair, s_pw, threadIdx.x, kThreads,
                 [] { __syncthreads(); });
    if (threadIdx.x == 0) d.down_cnt[blockIdx.x] = 0u;
    MOE_TRACE_POINT(2, 7);
}

// ---------------------------------------------------------------------------
// Gate/up for steps of at most 8 tokens, as one wave: one block of 16 warps
// per SM stages the step's x rows once (all T tokens: the MMA's N = 8
// columns are the tokens, so every slot uses the same B operand and picks
// its own tokens' columns in the epilogue), then its warps stream gate/up
// units -- (slot, 16-row tile, K part), shared slots first -- handed out by
// an atomic counter as they ask, through an 8-deep register ring that runs
// on from one unit into the next.  Groups of 2^lks warps split a
// tile's K range and add their partial sums in shared memory in a fixed
// order.  Epilogue per unit: SwiGLU of the slot's tokens, h (BF16) and the
// per-pair max |h| as in the per-slot kernel.
// ---------------------------------------------------------------------------
constexpr int kUW = 16;                 // warps per block
constexpr int kUT = 32 * kUW;
constexpr int kUPD = 8;                 // ring depth (a unit's chunks are a multiple of it)
constexpr int kUMax = 32;               // units per warp

constexpr int kWaveSlots = 8 * kMaxTopK + kMaxShared;   // slots of a step of <= 8 tokens

template <bool F8>
__global__ void __launch_bounds__(kUT, 1) gemv_up_wave_kernel(DevLayer d, const __nv_bfloat16 *__restrict__ x,
                                                              int T, int lks, int pre) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ const uint8_t *s_sb[kWaveSlots];   // the slot's gate/up weights
    __shared__ int s_se[kWaveSlots];              // its expert (< 0: shared)
    __shared__ int s_q[kUW][2];                   // a warp group's next units
    __shared__ const uint4 *s_src[8];
    __shared__ float s_scale[8];
    __shared__ float s_unscale[8];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int H = d.H, S = d.S;
    const int ks = 1 << lks, kw = warp & (ks - 1), gj = warp >> lks;
    const bool leader = kw == 0 && lane == 0;
    const int NC64 = H / kChunkK, row_stride = NC64 * 128 + 16;
    float *red = reinterpret_cast<float *>(smem + (size_t)(T + 1) * row_stride);   // [kUW][4][32]
    const uint64_t pol = evict_first_policy();
    // a group's barrier (its K split), or the warp's own for a group of one
    auto gsync = [&] {
        if (ks > 1) asm volatile("bar.sync %0, %1;\n" ::"r"(1 + gj), "r"(32 * ks) : "memory");
        else __syncwarp();
    };

    MOE_TRACE_POINT(1, 0);
    for (int i = threadIdx.x; i < row_stride / 16; i += kUT)
        reinterpret_cast<uint4 *>(smem + (size_t)T * row_stride)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (pre) {
        // x is final before the dependency wait: this kernel starts only once
        // the router has passed its own wait on the kernel that wrote x (L2
        // loads).  Stage it now, with each row's exact power-of-two prescale
        // from its maximum (the router's rule, on the same maximum).
        __shared__ unsigned s_rmax[8];
        uint4 *xraw = reinterpret_cast<uint4 *>(smem + (size_t)(T + 1) * row_stride + (size_t)kUW * 4 * 32 * sizeof(float));
        if (threadIdx.x < 8) s_rmax[threadIdx.x] = 0u;
        __syncthreads();
        const int per_row = H / 8, items = T * per_row;
        for (int base = threadIdx.x; base < items; base += 4 * kUT) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int it = base + u * kUT;
                if (it < items) v[u] = __ldcg(reinterpret_cast<const uint4 *>(x) + it);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int it = base + u * kUT;
                float m = 0.f;
                if (it < items) {
                    xraw[it] = v[u];
                    const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
                        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[qq] << 16)), fabsf(__uint_as_float(w4[qq] & 0xFFFF0000u))));
                    // (non-negative: its bits order as unsigned integers)
                    atomicMax(&s_rmax[it / per_row], __float_as_uint(m));
                }
            }
        }
        __syncthreads();
        if (threadIdx.x < T) {
            const int ex = max(-100, exp_for_f16(__uint_as_float(s_rmax[threadIdx.x])));
            s_scale[threadIdx.x] = pow2f(-ex);
            s_unscale[threadIdx.x] = pow2f(ex);
        }
        __syncthreads();
        // into the MMA's B layout (as stage_rows): half index 16q + 4kb + 2h + e
        for (int it = threadIdx.x; it < items; it += kUT) {
            const int j = it / per_row, rem = it - j * per_row;
            const int cc = rem >> 3, part = rem & 7;
            uint32_t *dst = reinterpret_cast<uint32_t *>(smem + (size_t)j * row_stride + cc * 128 + (part >> 1) * 8 +
                                                         (part & 1) * 4);
            const uint4 v = xraw[it];
            const float sc = s_scale[j];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
                dst[qq * 8] = pack_f16x2(__uint_as_float(w[qq] << 16) * sc, __uint_as_float(w[qq] & 0xFFFF0000u) * sc);
        }
    }
    pdl_wait();     // the router's slot tables, x's exponents (W4A4: and scales), the zeroed h maxima and unit counter
    pdl_trigger();
    MOE_TRACE_POINT(1, 1);
    const int ns = __ldcg(d.nslots);
    const int NTs = d.Is / 8, NT13 = d.I / 8;
    const int units = S * NTs + (ns - S) * NT13;
    // Units -- (slot, 16-row tile), shared slots first -- are handed out in
    // order by an atomic counter as each warp group asks for its next one, so
    // that groups on SMs that stream faster take more of them.  A group
    // knows its next unit one unit ahead (the ring reaches into it) and asks
    // for the one after at the start of each unit.
    if (leader) {
        const int u0 = (int)atomicAdd(d.wave_ctr, 1u);
        s_q[gj][0] = u0;
        s_q[gj][1] = u0 < units ? (int)atomicAdd(d.wave_ctr, 1u) : units;
    }
    for (int sl = threadIdx.x; sl < ns; sl += kUT) {
        const int e = __ldcg(d.slot_expert + sl);
        s_se[sl] = e;
        s_sb[sl] = e < 0 ? d.sw13r + (size_t)(-e - 1) * d.s13_stride : d.w13r + (size_t)e * d.e13_stride;
    }
    if (!pre && threadIdx.x < T) {
        const int t = threadIdx.x;
        const int ex = __ldcg(d.xexp + t);
        s_src[t] = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
        s_scale[t] = pow2f(-ex);
        s_unscale[t] = pow2f(ex) * (d.w4a4 ? __ldcg(d.gsx + t) : 1.f);
    }
    __syncthreads();
    int cur = s_q[gj][0], nxt = s_q[gj][1];
    // unit -> slot, tile, and the first chunk of this warp's K part
    auto decode = [&](int u, int &sl, int &r, int &cpw, const uint8_t *&base, bool &f8) {
        if (u < S * NTs) {
            sl = u / NTs;
            r = u - sl * NTs;
        } else {
            const int v = u - S * NTs;
            sl = S + v / NT13;
            r = v - (sl - S) * NT13;
        }
        const int e = s_se[sl];
        f8 = F8 && (e < 0 ? d.f8s : d.f8e);
        const int nc = chunks_of(H, f8);
        cpw = nc >> lks;
        base = s_sb[sl] + ((size_t)r * nc + kw * cpw) * kChunkBytes;
    };
    int sl = 0, r = 0, cpw = 0, nsl = 0, nr = 0, ncpw = 0;
    bool f8 = false, nf8 = false;
    const uint8_t *base = nullptr, *nbase = nullptr;
    uint4 cb[kUPD];
    uint2 sb[kUPD];
    if (cur < units) {
        decode(cur, sl, r, cpw, base, f8);
#pragma unroll
        for (int i = 0; i < kUPD; ++i) load_chunk(base, i, lane, cb[i], sb[i], pol);
    }
    if (!pre) stage_rows<kUT>(T, 0, NC64, smem, row_stride, s_src, s_scale);
    __syncthreads();
    MOE_TRACE_POINT(1, 2);

    const uint8_t *xb = smem + (size_t)(g < T ? g : T) * row_stride + q * 32;
#pragma unroll 1
    for (int it = 0; cur < units; ++it) {
        if (nxt < units) decode(nxt, nsl, nr, ncpw, nbase, nf8);
        // the unit after next, asked for now, published at this unit's end
        unsigned grab = (unsigned)units;
        if (leader && nxt < units) grab = atomicAdd(d.wave_ctr, 1u);
        const int kc0 = kw * cpw;
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
        int lc = kUPD;     // next chunk to load (of this unit while < cpw, then of the next)
#pragma unroll 1
        for (int cc = 0; cc < cpw; cc += kUPD) {
#pragma unroll
            for (int i = 0; i < kUPD; ++i) {
                const uint8_t *bp = xb + b_offset(kc0 + cc + i, f8);
                if (F8 && f8) {
                    chunk_mma_f8(cb[i], sb[i], lds128(bp), (i & 1) ? a1 : a0);
                } else {
                    uint32_t a[4][4];
                    decode_chunk(cb[i], sb[i], a);
                    const uint4 b01 = lds128(bp), b23 = lds128(bp + 16);
                    mma_16816(a0, a[0][0], a[0][1], a[0][2], a[0][3], b01.x, b01.y);
                    mma_16816(a1, a[1][0], a[1][1], a[1][2], a[1][3], b01.z, b01.w);
                    mma_16816(a0, a[2][0], a[2][1], a[2][2], a[2][3], b23.x, b23.y);
                    mma_16816(a1, a[3][0], a[3][1], a[3][2], a[3][3], b23.z, b23.w);
                }
                // refill this slot with the chunk kUPD ahead (possibly of the next unit)
                if (lc < cpw) load_chunk(base, lc, lane, cb[i], sb[i], pol);
                else if (nxt < units) load_chunk(nbase, lc - cpw, lane, cb[i], sb[i], pol);
                ++lc;
            }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) a0[v] += a1[v];
        if (leader && ks > 1) s_q[gj][it & 1] = (int)grab;
        if (ks > 1) {
            // fixed-order K reduction within the group (named barrier 1 + group)
            if (kw > 0) {
#pragma unroll
                for (int v = 0; v < 4; ++v) red[(warp * 4 + v) * 32 + lane] = a0[v];
            }
            gsync();
            if (kw == 0) {
#pragma unroll 1
                for (int w = 1; w < ks; ++w)
#pragma unroll
                    for (int v = 0; v < 4; ++v) a0[v] += red[((warp + w) * 4 + v) * 32 + lane];
            }
            gsync();
        }
        const int n2 = ks > 1 ? s_q[gj][it & 1] : (int)__shfl_sync(0xffffffffu, grab, 0);
        if (kw == 0) {
            // SwiGLU: tile rows 0..7 gate, 8..15 up of intermediate row 8r + g;
            // columns are tokens, a slot's pairs are its tokens in ascending order
            const int e = s_se[sl];
            const int m = __ldcg(d.slot_m + sl), p0 = __ldcg(d.slot_p0 + sl);
            unsigned msk = 0u;
            if (lane < m) msk = 1u << __ldcg(d.pair_tok + p0 + lane);
            msk = __reduce_or_sync(0xffffffffu, msk);
            float gsa, gsb;
            if (e < 0) {
                gsa = d.sgs13[2 * (-e - 1)];
                gsb = d.sgs13[2 * (-e - 1) + 1];
            } else {
                gsa = d.gs13[2 * e];
                gsb = d.gs13[2 * e + 1];
            }
            const int n = 8 * r + g;
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int t = 2 * q + e2;
                const bool on = t < T && ((msk >> t) & 1u);
                const int p = p0 + __popc(msk & ((1u << t) - 1u));
                float habs = 0.f;
                if (on) {
                    const float sc = s_unscale[t];
                    const float gt = a0[e2] * gsa * sc;
                    const float up = a0[2 + e2] * gsb * sc;
                    const __nv_bfloat16 hb = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
                    d.h_ws[(size_t)p * d.Imax + n] = hb;
                    habs = fabsf(__bfloat162float(hb));
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) habs = fmaxf(habs, __shfl_xor_sync(0xffffffffu, habs, off));
                if (on && g == 0) atomicMax(d.hmax + p, __float_as_uint(habs));
            }
        }
        cur = nxt;
        sl = nsl;
        r = nr;
        cpw = ncpw;
        base = nbase;
        f8 = nf8;
        nxt = n2;
    }
    MOE_TRACE_POINT(1, 3);
}

// ---------------------------------------------------------------------------
// Wave kernels over a list of slots, each slot with its own B operand: down +
// combine (MODE 1) for steps of at most 8 tokens (every slot) and, above 8
// tokens, gate/up + SwiGLU (MODE 0) and down + combine over the routed slots
// that the grouped kernels leave (fewer than grouped_min_tokens <= 8 tokens).
// One block of 16 warps per SM takes a contiguous, slot-major range of
// (slot, 16-row tile) units -- a range spans few slots, whose B rows (a
// slot's tokens' x rows, or its pairs' h rows, at most 8) it stages once --
// and its warp groups take the range's units as they ask (a shared counter),
// streaming them through a PD-deep register ring that runs on from one unit
// into the next.  Groups of 2^lks warps split a unit's K range (fixed-order
// reduction).  Gate/up epilogue: SwiGLU into h with the per-pair max |h|, as
// the per-slot kernel.  Down epilogue: y = gs * acc into the workspace; after
// its last unit a warp takes the per-tile tickets of its units (no spinning),
// and the unit that completed a tile last among the slots combines that
// tile's 16 rows for all tokens.
// ---------------------------------------------------------------------------
constexpr int kDMaxSlots = 12;          // slots one block's units may span

template <int MODE, bool F8, int PD, int NG>
__global__ void __launch_bounds__(kUT, 1) gemv_slot_wave_kernel(DevLayer d, const __nv_bfloat16 *__restrict__ x,
                                                                int T, int lks, int cold,
                                                                __nv_bfloat16 *__restrict__ out) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int RB = 8 * NG;                     // staged B rows per slot
    __shared__ const uint4 *s_src[kDMaxSlots][RB];
    __shared__ float s_scale[kDMaxSlots][RB], s_un[kDMaxSlots][RB];
    __shared__ int s_off[kDMaxSlots], s_rs[kDMaxSlots], s_m[kDMaxSlots], s_p0[kDMaxSlots], s_e[kDMaxSlots];
    __shared__ const uint8_t *s_wb[kDMaxSlots];
    __shared__ int s_pair[MODE == 1 ? kMaxTokens * (kMaxTopK + kMaxShared) : 1];
    __shared__ float s_pw[MODE == 1 ? kMaxTokens * (kMaxTopK + kMaxShared) : 1];
    __shared__ int s_ctr;                          // the block's next unit
    __shared__ int s_q[kUW][2];                    // a warp group's next units
    __shared__ short s_dr[kUW][kUMax];             // tiles whose y a warp wrote, tickets pending

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int H = d.H, K = d.k, P = d.k + d.S;
    const int ks = 1 << lks, kw = warp & (ks - 1), gj = warp >> lks;
    const bool leader = kw == 0 && lane == 0;
    const int NT = MODE == 0 ? d.I / 8 : H / 16;   // units per slot (gate/up: routed slots only)
    float *red = reinterpret_cast<float *>(smem);   // [kUW][4][32]
    uint8_t *stage = smem + (size_t)kUW * 4 * 32 * sizeof(float);
    const uint64_t pol = evict_first_policy();
    auto gsync = [&] {
        if (ks > 1) asm volatile("bar.sync %0, %1;\n" ::"r"(1 + gj), "r"(32 * ks) : "memory");
        else __syncwarp();
    };

    MOE_TRACE_POINT(1 + MODE, 0);
    // Down: the router has completed before this kernel could start (the
    // gate/up kernels released it only after their own waits), so the slot
    // and pair tables are final: stream the weights, wait for h after.
    // Gate/up: the router's tables come from the kernel before: wait first.
    if (MODE == 0) {
        pdl_wait();
        pdl_trigger();
    }
    const int ns = __ldcg(d.nslots);
    const int nlist = cold ? __ldcg(d.ncold) : ns;
    const long U = (long)nlist * NT;
    const int ub0 = (int)(U * blockIdx.x / gridDim.x), ub1 = (int)(U * (blockIdx.x + 1) / gridDim.x);
    const int nu = ub1 - ub0;
    const int ci_lo = ub0 / NT, nsb = nu > 0 ? (ub1 - 1) / NT - ci_lo + 1 : 0;
    if (threadIdx.x == 0) s_ctr = 0;
    // the staged slots' geometry (RB rows each, rows >= m zero) and weights,
    // and the combine's pair table
    if (threadIdx.x < nsb) {
        const int ci = ci_lo + threadIdx.x;
        const int sl = cold ? __ldcg(d.cold_slots + ci) : ci;
        const int e = __ldcg(d.slot_expert + sl);
        s_e[threadIdx.x] = e;
        if (MODE == 0) {
            s_wb[threadIdx.x] = e < 0 ? d.sw13r + (size_t)(-e - 1) * d.s13_stride : d.w13r + (size_t)e * d.e13_stride;
            s_rs[threadIdx.x] = (H / kChunkK) * 128 + 16;
        } else {
            s_wb[threadIdx.x] = e < 0 ? d.sw2r + (size_t)(-e - 1) * d.s2_stride : d.w2r + (size_t)e * d.e2_stride;
            s_rs[threadIdx.x] = ((e < 0 ? d.Is : d.I) / kChunkK) * 128 + 16;
        }
        s_m[threadIdx.x] = __ldcg(d.slot_m + sl);
        s_p0[threadIdx.x] = __ldcg(d.slot_p0 + sl);
    }
    if (MODE == 1) {
        for (int i = threadIdx.x; i < T * P; i += kUT) {
            const int p = __ldcg(d.pair_of + i);
            s_pair[i] = p;
            s_pw[i] = (i % P) < K ? __ldcg(d.pair_w + p) : 1.0f;
        }
    }
    __syncthreads();
    // The block's units are handed out by a shared counter as each warp
    // group asks (one unit ahead, for the ring), so that its warps finish
    // together.
    if (leader) {
        const int u0 = atomicAdd(&s_ctr, 1);
        s_q[gj][0] = u0;
        s_q[gj][1] = u0 < nu ? atomicAdd(&s_ctr, 1) : nu;
    }
    if (threadIdx.x == 0) {
        int off = 0;
        for (int j = 0; j < nsb; ++j) {
            s_off[j] = off;
            off += RB * s_rs[j];
        }
    }
    __syncthreads();
    int cur = s_q[gj][0], nxt = s_q[gj][1];
    // unit -> staged slot, tile, and the first chunk of this warp's K part
    auto decode = [&](int u, int &sj, int &r, int &cpw, const uint8_t *&base, bool &f8) {
        const int tu = ub0 + u;
        const int ci = tu / NT;
        r = tu - ci * NT;
        sj = ci - ci_lo;
        const int e = s_e[sj];
        f8 = F8 && (e < 0 ? d.f8s : d.f8e);
        const int nc = MODE == 0 ? chunks_of(H, f8) : chunks_of(e < 0 ? d.Is : d.I, f8);
        cpw = nc >> lks;
        base = s_wb[sj] + ((size_t)r * nc + kw * cpw) * kChunkBytes;
    };
    int sj = 0, r = 0, cpw = 0, nsj = 0, nr = 0, ncpw = 0;
    bool f8 = false, nf8 = false;
    const uint8_t *base = nullptr, *nbase = nullptr;
    uint4 cb[PD];
    uint2 sb[PD];
    if (cur < nu) {
        decode(cur, sj, r, cpw, base, f8);
#pragma unroll
        for (int i = 0; i < PD; ++i) load_chunk(base, i, lane, cb[i], sb[i], pol);
    }
    if (MODE == 1) {
        pdl_wait();     // h and its maxima
        pdl_trigger();
    }
    MOE_TRACE_POINT(1 + MODE, 1);
    if (threadIdx.x < RB * nsb) {
        const int j = threadIdx.x / RB, c = threadIdx.x % RB;
        if (c < s_m[j]) {
            const int p = s_p0[j] + c;
            if (MODE == 0) {
                const int tok = __ldcg(d.pair_tok + p);
                const int ex = __ldcg(d.xexp + tok);
                s_src[j][c] = reinterpret_cast<const uint4 *>(x + (size_t)tok * H);
                s_scale[j][c] = pow2f(-ex);
                s_un[j][c] = pow2f(ex) * (d.w4a4 ? __ldcg(d.gsx + tok) : 1.f);
            } else {
                const int ex = hexp_of(__ldcg(d.hmax + p));
                s_src[j][c] = reinterpret_cast<const uint4 *>(d.h_ws + (size_t)p * d.Imax);
                s_scale[j][c] = pow2f(-ex);
                s_un[j][c] = pow2f(ex) * (d.w4a4 ? __ldcg(d.gsh + p) : 1.f);
            }
        }
    }
    __syncthreads();
    for (int j = 0; j < nsb; ++j) {
        const int m = s_m[j], rs = s_rs[j];
        uint8_t *reg = stage + s_off[j];
        for (int i = threadIdx.x; i < (RB - m) * (rs / 16); i += kUT)
            reinterpret_cast<uint4 *>(reg + (size_t)m * rs)[i] = make_uint4(0u, 0u, 0u, 0u);
        stage_rows<kUT>(m, 0, (rs - 16) / 128, reg, rs, s_src[j], s_scale[j]);
    }
    __syncthreads();
    MOE_TRACE_POINT(1 + MODE, 2);

    // Down: tickets of the tiles in the warp's pending list.  After the
    // warp's barrier every lane fences (ordering all of the warp's y stores
    // before its tickets), then lane i takes the ticket of entry i; the warp
    // combines the tiles it completed last among the slots.  Taken after the
    // warp's last unit, not after each (a fence and an atomic round trip per
    // unit would stall the ring), or when the list is full.
    int nd = 0;
    auto tickets = [&]() {
        __syncwarp();
        __threadfence();
        const bool lastu = lane < nd && atomicAdd(d.down_cnt + s_dr[warp][lane], 1u) == (unsigned)(ns - 1);
        unsigned lm = __ballot_sync(0xffffffffu, lastu);
        if (lm) __threadfence();
        while (lm) {
            const int i = __ffs(lm) - 1;
            lm &= lm - 1;
            const int rr = s_dr[warp][i];
            // every slot's y of this tile is written: out rows 16rr .. 16rr + 15
            for (int it = lane; it < 4 * T; it += 32) {
                const int t = it >> 2, m4 = 4 * rr + (it & 3);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int j = 0; j < P; ++j) {
                    const float w = s_pw[t * P + j];
                    const float4 y = __ldcg(reinterpret_cast<const float4 *>(d.y_ws + (size_t)s_pair[t * P + j] * H) + m4);
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
                *reinterpret_cast<uint2 *>(out + (size_t)t * H + 4 * m4) = v;
            }
            if (lane == 0) d.down_cnt[rr] = 0u;
        }
        __syncwarp();
        nd = 0;
    };

#pragma unroll 1
    for (int it = 0; cur < nu; ++it) {
        if (nxt < nu) decode(nxt, nsj, nr, ncpw, nbase, nf8);
        // the unit after next, asked for now, published at this unit's end
        int grab = nu;
        if (leader && nxt < nu) grab = atomicAdd(&s_ctr, 1);
        const int kc0 = kw * cpw;
        const uint8_t *xb = stage + s_off[sj] + (size_t)g * s_rs[sj] + q * 32;
        const size_t gstr = (size_t)8 * s_rs[sj];   // the second token group's B rows
        const bool two = NG > 1 && s_m[sj] > 8;
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        int lc = PD;       // next chunk to load (of this unit while < cpw, then of the next)
#pragma unroll 1
        for (int cc = 0; cc < cpw; cc += PD) {
#pragma unroll
            for (int i = 0; i < PD; ++i) {
                const uint8_t *bp = xb + b_offset(kc0 + cc + i, f8);
                if (F8 && f8) {
                    chunk_mma_f8(cb[i], sb[i], lds128(bp), (i & 1) ? a1 : a0);
                } else {
                    uint32_t a[4][4];
                    decode_chunk(cb[i], sb[i], a);
                    const uint4 b01 = lds128(bp), b23 = lds128(bp + 16);
                    mma_16816(a0, a[0][0], a[0][1], a[0][2], a[0][3], b01.x, b01.y);
                    mma_16816(a1, a[1][0], a[1][1], a[1][2], a[1][3], b01.z, b01.w);
                    mma_16816(a0, a[2][0], a[2][1], a[2][2], a[2][3], b23.x, b23.y);
                    mma_16816(a1, a[3][0], a[3][1], a[3][2], a[3][3], b23.z, b23.w);
                    if (NG > 1 && two) {
                        const uint4 c01 = lds128(bp + gstr), c23 = lds128(bp + gstr + 16);
                        mma_16816(c1, a[0][0], a[0][1], a[0][2], a[0][3], c01.x, c01.y);
                        mma_16816(c1, a[1][0], a[1][1], a[1][2], a[1][3], c01.z, c01.w);
                        mma_16816(c1, a[2][0], a[2][1], a[2][2], a[2][3], c23.x, c23.y);
                        mma_16816(c1, a[3][0], a[3][1], a[3][2], a[3][3], c23.z, c23.w);
                    }
                }
                // refill this slot with the chunk PD ahead (possibly of the next unit)
                if (lc < cpw) load_chunk(base, lc, lane, cb[i], sb[i], pol);
                else if (nxt < nu) load_chunk(nbase, lc - cpw, lane, cb[i], sb[i], pol);
                ++lc;
            }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) a0[v] += a1[v];
        if (leader && ks > 1) s_q[gj][it & 1] = grab;
        if (ks > 1) {
            // fixed-order K reduction within the group (named barrier 1 + group)
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) {
                float *av = gg == 0 ? a0 : c1;
                if (kw > 0) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) red[(warp * 4 + v) * 32 + lane] = av[v];
                }
                gsync();
                if (kw == 0) {
#pragma unroll 1
                    for (int w = 1; w < ks; ++w)
#pragma unroll
                        for (int v = 0; v < 4; ++v) av[v] += red[((warp + w) * 4 + v) * 32 + lane];
                }
                gsync();
            }
        }
        const int n2 = ks > 1 ? s_q[gj][it & 1] : __shfl_sync(0xffffffffu, grab, 0);
        if (kw == 0) {
            const int e = s_e[sj], m = s_m[sj], p0 = s_p0[sj];
            if (MODE == 0) {
                // SwiGLU: tile rows 0..7 gate, 8..15 up of intermediate row
                // 8r + g; columns are the slot's pairs
                const float gsa = e < 0 ? d.sgs13[2 * (-e - 1)] : d.gs13[2 * e];
                const float gsb = e < 0 ? d.sgs13[2 * (-e - 1) + 1] : d.gs13[2 * e + 1];
                const int n = 8 * r + g;
#pragma unroll
                for (int e4 = 0; e4 < 2 * NG; ++e4) {
                    const int e2 = e4 & 1, gg = e4 >> 1;
                    const float *av = gg == 0 ? a0 : c1;
                    const int col = 8 * gg + 2 * q + e2;
                    const bool on = col < m;
                    float habs = 0.f;
                    if (on) {
                        const float sc = s_un[sj][col];
                        const float gt = av[e2] * gsa * sc;
                        const float up = av[2 + e2] * gsb * sc;
                        const __nv_bfloat16 hb = __float2bfloat16_rn(gt / (1.0f + expf(-gt)) * up);
                        d.h_ws[(size_t)(p0 + col) * d.Imax + n] = hb;
                        habs = fabsf(__bfloat162float(hb));
                    }
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) habs = fmaxf(habs, __shfl_xor_sync(0xffffffffu, habs, off));
                    if (on && g == 0) atomicMax(d.hmax + p0 + col, __float_as_uint(habs));
                }
            } else {
                // y = gs * 2^hexp * acc for the slot's pairs (columns), rows 16r + g, + 8
                const float gs = e < 0 ? d.sgs2[-e - 1] : d.gs2[e];
#pragma unroll
                for (int e4 = 0; e4 < 2 * NG; ++e4) {
                    const int e2 = e4 & 1, gg = e4 >> 1;
                    const float *av = gg == 0 ? a0 : c1;
                    const int col = 8 * gg + 2 * q + e2;
                    if (col < m) {
                        const float sc = s_un[sj][col] * gs;
                        float *yp = d.y_ws + (size_t)(p0 + col) * H + 16 * r + g;
                        yp[0] = av[e2] * sc;
                        yp[8] = av[2 + e2] * sc;
                    }
                }
                if (lane == 0) s_dr[warp][nd] = (short)r;
                ++nd;
                if (nd == kUMax) tickets();
            }
        }
        cur = nxt;
        sj = nsj;
        r = nr;
        cpw = ncpw;
        base = nbase;
        f8 = nf8;
        nxt = n2;
    }
    if (MODE == 1 && kw == 0 && nd > 0) tickets();
    MOE_TRACE_POINT(1 + MODE, 3);
}

// The slot wave kernel's geometry, or lks = -1 where it does not apply:
// down (MODE 1) at up to 8 tokens over every slot; above 8 tokens (cold =
// 1), gate/up and down over the routed slots below grouped_min_tokens, when
// that threshold is at most 8 (their B rows fit the 8 staged rows).  A
// block's range must span at most kDMaxSlots slots whose staged rows fit
// its shared memory, and a unit's chunks must be whole turns of an 8- or
// 6-deep ring; among the K splits 2^l <= 4, the fewest (chunks + a
// reduction) per group at an even share of the units.
struct SlotWave {
    int lks = -1, pd = 0, cold = 0, ng = 1;
    size_t smem = 0;
};

SlotWave slot_wave(const DevLayer &d, int MODE, int T, int sm_count, size_t optin) {
    SlotWave w;
    if (T > 8) {
        // the cold slots hold fewer than 16 tokens: two groups of 8 B rows
        if (!(d.grouped_min > 0 && d.grouped_min <= 16) || d.f8e || d.f8s) return w;
        w.cold = 1;
        w.ng = 2;
    } else if (MODE == 0) {
        return w;
    }
    const int slots = std::min(d.E, T * d.k) + (w.cold ? 0 : d.S);
    const int NT = MODE == 0 ? d.I / 8 : d.H / 16;
    const long U = (long)slots * NT;
    const long perb = (U + sm_count - 1) / sm_count;
    const long span = perb / NT + 2;
    if (span > kDMaxSlots) return w;
    const int rowb = MODE == 0 ? (d.H / kChunkK) * 128 + 16
                               : ((!w.cold && d.S > 0 ? std::max(d.I, d.Is) : d.I) / kChunkK) * 128 + 16;
    const size_t smem = (size_t)kUW * 4 * 32 * sizeof(float) + (size_t)span * 8 * w.ng * rowb;
    if (smem + 16 * 1024 > optin) return w;
    // chunk counts per tile of the formats present
    int nc[2] = {MODE == 0 ? chunks_of(d.H, d.f8e) : chunks_of(d.I, d.f8e), 0};
    const bool two = !w.cold && d.S > 0;
    if (two) nc[1] = MODE == 0 ? chunks_of(d.H, d.f8s) : chunks_of(d.Is, d.f8s);
    long bestc = 0;
    for (int pd = 8; pd >= 6; pd -= 2) {
        for (int l = 0; l <= 2; ++l) {
            bool fits = true;
            for (int f = 0; f < (two ? 2 : 1) && fits; ++f)
                fits = nc[f] % (1 << l) == 0 && (nc[f] >> l) % pd == 0;
            if (!fits) continue;
            const long per = (perb + (kUW >> l) - 1) / (kUW >> l);
            const long cost = per * ((nc[0] >> l) + (l > 0 ? 2 : 0));
            if (w.lks < 0 || cost < bestc) {
                w.lks = l;
                w.pd = pd;
                bestc = cost;
            }
        }
        if (w.lks >= 0) break;   // the deeper ring where it fits
    }
    w.smem = smem;
    return w;
}

template <int MODE, bool F8, int PD, int NG>
cudaError_t launch_slot_wave(const DevLayer &d, const __nv_bfloat16 *x, int T, const SlotWave &w,
                             __nv_bfloat16 *out, int sm_count, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count);
    cfg.blockDim = dim3(kUT);
    cfg.dynamicSmemBytes = w.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_slot_wave_kernel<MODE, F8, PD, NG>, d, x, T, w.lks, w.cold, out);
}

// (instances: down at up to 8 tokens in both chunk families, one token
// group; the cold slots above 8 tokens NVFP4 only -- the grouped kernels,
// hence the cold slots, exist only for NVFP4 layers -- two token groups)
cudaError_t launch_slot_wave_any(int MODE, const DevLayer &d, const __nv_bfloat16 *x, int T, const SlotWave &w,
                                 __nv_bfloat16 *out, int sm_count, cudaStream_t s) {
    const bool f8 = d.f8e || d.f8s;
    if (w.ng == 2) {
        if (MODE == 0)
            return w.pd == 8 ? launch_slot_wave<0, false, 8, 2>(d, x, T, w, out, sm_count, s)
                             : launch_slot_wave<0, false, 6, 2>(d, x, T, w, out, sm_count, s);
        return w.pd == 8 ? launch_slot_wave<1, false, 8, 2>(d, x, T, w, out, sm_count, s)
                         : launch_slot_wave<1, false, 6, 2>(d, x, T, w, out, sm_count, s);
    }
    if (w.pd == 8)
        return f8 ? launch_slot_wave<1, true, 8, 1>(d, x, T, w, out, sm_count, s)
                  : launch_slot_wave<1, false, 8, 1>(d, x, T, w, out, sm_count, s);
    return f8 ? launch_slot_wave<1, true, 6, 1>(d, x, T, w, out, sm_count, s)
              : launch_slot_wave<1, false, 6, 1>(d, x, T, w, out, sm_count, s);
}

template <int MODE, bool F8, int PD, int NG>
cudaError_t allow_slot_wave(int optin) {
    return allow_max_dynamic_smem(gemv_slot_wave_kernel<MODE, F8, PD, NG>, optin);
}

// The K split of the wave kernel: among 2^l <= 4 whose chunks per unit are a
// whole number of ring turns, the one with the fewest (chunks + a reduction)
// per group at an even share of the units.  -1: the kernel does not apply.
int wave_lks(const DevLayer &d, int T, int sm_count) {
    if (T > 8) return -1;
    // (routed and shared experts may differ in chunk format: an F8 tile has
    // twice the chunks, which the units handed out on demand absorb)
    const int slots = std::min(d.E, T * d.k);
    const long units = (long)d.S * (d.Is / 8) + (long)slots * (d.I / 8);
    int best = -1;
    long bestc = 0;
    if (slots + d.S > kWaveSlots) return -1;
    for (int l = 0; l <= 2; ++l) {
        const long groups = (long)sm_count * (kUW >> l);
        const long per = (units + groups - 1) / groups;
        bool fits = true;
        for (int f = 0; f < 2 && fits; ++f) {
            const bool f8 = f == 0 ? d.f8e : (d.S > 0 && d.f8s);
            const int nc = chunks_of(d.H, f8);
            fits = nc % (1 << l) == 0 && (nc >> l) % kUPD == 0;
        }
        if (!fits) continue;
        const long cost = per * ((chunks_of(d.H, d.f8e) >> l) + (l > 0 ? 2 : 0));
        if (best < 0 || cost < bestc) {
            best = l;
            bestc = cost;
        }
    }
    return best;
}

size_t wave_smem(const DevLayer &d, int T, bool pre) {
    // B rows (+ a zero row), the K reduction, and (staged before the
    // dependency wait) x as loaded
    return (size_t)(T + 1) * ((d.H / kChunkK) * 128 + 16) + (size_t)kUW * 4 * 32 * sizeof(float) +
           (pre ? (size_t)T * d.H * 2 : 0);
}

template <int MODE, int GMAX, int PD>
cudaError_t launch_one(const DevLayer &d, const __nv_bfloat16 *x, int T, int ksplit, dim3 grid,
                       size_t smem, __nv_bfloat16 *out, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<MODE, GMAX, PD>, d, x, T, ksplit, out);
}

template <int MODE>
cudaError_t launch_stage(const DevLayer &d, const __nv_bfloat16 *x, int T, __nv_bfloat16 *out,
                         cudaStream_t s) {
    const int slots = min(d.E, T * d.k) + d.S;
    const int Iall = d.S > 0 ? max(d.I, d.Is) : d.I;
    const int Imin = d.S > 0 ? min(d.I, d.Is) : d.I;
    const int NT = MODE == 0 ? Iall / 8 : d.H / 16;
    const int NCmax = MODE == 0 ? d.H / kChunkK : Iall / kChunkK;
    const int NCmin = MODE == 0 ? d.H / kChunkK : Imin / kChunkK;
    // the combine (down) needs room for the [T, k+S] pair table
    const size_t combine_smem = (size_t)kMaxTokens * 16 * (sizeof(int) + sizeof(float));
    // at most 8 tokens per slot here: up to 8 tokens in all, or the grouped
    // kernels take every slot with at least grouped_min <= 8 of them -- one
    // token group, the 8-deep register ring
    if (T <= 8 || (d.grouped_min > 0 && d.grouped_min <= 8)) {
        const long tiles = (long)slots * NT;
        int ksplit = 1;
        while (ksplit < 4 && tiles * ksplit < 2048 && NCmin >= 4 * ksplit) ksplit *= 2;
        const int tpc = kGemvWarps / ksplit;
        dim3 grid((NT + tpc - 1) / tpc, slots);
        size_t smem = (size_t)8 * (NCmax * 128 + 16) + (size_t)tpc * (ksplit - 1) * 4 * 32 * sizeof(float);
        if (MODE == 1 && smem < combine_smem) smem = combine_smem;
        // down: a 12-deep ring (measured faster on the ML4- and
        // Inkling-shaped layers, the same occupancy); gate/up: 8 deep
        if constexpr (MODE == 1) return launch_one<1, 1, 12>(d, x, T, ksplit, grid, smem, out, s);
        else return launch_one<0, 1, 8>(d, x, T, ksplit, grid, smem, out, s);
    }
    dim3 grid((NT + kGemvWarps - 1) / kGemvWarps, slots);
    return launch_one<MODE, 8, 4>(d, x, T, 1, grid, (size_t)kStageBudget, out, s);
}

template <int MODE, int GMAX, int PD>
cudaError_t allow_smem(int optin) {
    return allow_max_dynamic_smem(gemv_kernel<MODE, GMAX, PD>, optin);
}

}  // namespace

cudaError_t prepare_route_kernel(int optin_bytes);
cudaError_t prepare_fused_kernel(int optin_bytes);

cudaError_t prepare_kernels() {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = allow_smem<0, 1, 8>(optin);
    if (e == cudaSuccess) e = allow_smem<1, 1, 12>(optin);
    if (e == cudaSuccess) e = allow_smem<0, 8, 4>(optin);
    if (e == cudaSuccess) e = allow_max_dynamic_smem(gemv_up_wave_kernel<false>, optin);
    if (e == cudaSuccess) e = allow_max_dynamic_smem(gemv_up_wave_kernel<true>, optin);
    if (e == cudaSuccess) e = allow_slot_wave<0, false, 8, 2>(optin);
    if (e == cudaSuccess) e = allow_slot_wave<0, false, 6, 2>(optin);
    if (e == cudaSuccess) e = allow_slot_wave<1, false, 8, 2>(optin);
    if (e == cudaSuccess) e = allow_slot_wave<1, false, 6, 2>(optin);
    if (e == cudaSuccess) e = allow_slot_wave<1, false, 8, 1>(optin);
    if (e == cudaSuccess) e = allow_slot_wave<1, true, 8, 1>(optin);
    if (e == cudaSuccess) e = allow_slot_wave<1, false, 6, 1>(optin);
    if (e == cudaSuccess) e = allow_slot_wave<1, true, 6, 1>(optin);
    if (e == cudaSuccess) e = allow_smem<1, 8, 4>(optin);
    if (e == cudaSuccess) e = prepare_route_kernel(optin);
    if (e == cudaSuccess) e = prepare_fused_kernel(optin);
    if (e == cudaSuccess) e = prepare_grouped_kernels(optin);
    return e;
}

cudaError_t launch_gate_up(const DevLayer &d, const __nv_bfloat16 *x, int T, int sm_count, int optin_smem,
                           cudaStream_t s) {
    const int sms = sm_count;
    const int lks = wave_lks(d, T, sms);
    // x staged before the dependency wait where it is final then (not W4A4:
    // the quantiser writes it) and its raw copy is at most 64 KB (measured:
    // Inkling-shaped 209.4 -> 205.5 us with 64 KB; ML4-shaped, 96 KB, 146.2
    // -> 152.7 us, so not there)
    const bool pre = !d.w4a4 && (size_t)T * d.H * 2 <= 64 * 1024 &&
                     wave_smem(d, T, true) + 4 * 1024 <= (size_t)optin_smem;
    const size_t smem = wave_smem(d, T, pre);
    if (lks >= 0 && smem + 4 * 1024 <= (size_t)optin_smem) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(sms);
        cfg.blockDim = dim3(kUT);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return (d.f8e || d.f8s) ? cudaLaunchKernelEx(&cfg, gemv_up_wave_kernel<true>, d, x, T, lks, (int)pre)
                                : cudaLaunchKernelEx(&cfg, gemv_up_wave_kernel<false>, d, x, T, lks, (int)pre);
    }
    const SlotWave w = slot_wave(d, 0, T, sms, (size_t)optin_smem);
    if (w.lks >= 0) return launch_slot_wave_any(0, d, x, T, w, nullptr, sms, s);
    return launch_stage<0>(d, x, T, nullptr, s);
}

cudaError_t launch_down(const DevLayer &d, int T, __nv_bfloat16 *out, int sm_count, int optin_smem,
                        cudaStream_t s) {
    const SlotWave w = slot_wave(d, 1, T, sm_count, (size_t)optin_smem);
    if (w.lks >= 0) return launch_slot_wave_any(1, d, nullptr, T, w, out, sm_count, s);
    return launch_stage<1>(d, nullptr, T, out, s);
}

bool down_tile_tickets(const DevLayer &d, int T, int sm_count, int optin_smem) {
    return slot_wave(d, 1, T, sm_count, (size_t)optin_smem).lks >= 0;
}

// Above 8 tokens both wave kernels take cold slots of up to 15 tokens (at
// max_tokens, hence at every smaller step): the router may then raise the
// grouped threshold up to 16 so that the grouped kernels' items fit one per
// block.  Otherwise the threshold stays grouped_min_tokens.
int cold_threshold_max(const DevLayer &d, int sm_count, int optin_smem) {
    if (d.max_tokens <= 8 || d.grouped_min <= 0) return d.grouped_min;
    const bool ok = slot_wave(d, 0, d.max_tokens, sm_count, (size_t)optin_smem).lks >= 0 &&
                    slot_wave(d, 1, d.max_tokens, sm_count, (size_t)optin_smem).lks >= 0;
    return ok ? std::max(d.grouped_min, 16) : d.grouped_min;
}

}  // namespace moe
