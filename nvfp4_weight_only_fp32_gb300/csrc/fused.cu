// fused.cu -- the whole decode step of one layer (rows a1..a5) in ONE launch,
// for T <= 8 tokens.
//
// Sources: "vLLM Day-0 support for Recursive's Flint", "Optimisation strategy"
// (for up to 8 requests a low-latency path folds routing and the expert
// combine into the neighbouring GEMVs; small-batch MoE kernels read only the
// selected experts' weights); "Day 0 support for Mistral Large 4 on vLLM",
// "Specialized decode" (one persistent launch per MoE layer, all blocks
// resident, in-kernel waits that give up after a bound and set a sticky error
// word -- section "Fail-stop").
//
// One block per SM (grid = SM count), at most half an SM each, so the next
// layer's launch (programmatic dependent launch) becomes resident beside it and
// runs its prologue early.  Phases:
//   A  before griddepcontrol.wait: bulk-prefetch into L2 this block's router
//      rows and its first shared-expert tiles (static weights).
//   B  stage x (T rows) once as f16 with an exact per-row power-of-two
//      prescale, compute this block's experts' FP32 logits, publish them and
//      ARRIVE at grid barrier 1.
//   C  pass 0: this block's shared-expert gate/up tiles (no routing needed)
//      while the grid arrives; WAIT on barrier 1; pass 1: every block reads
//      all logits and runs the same deterministic top-k and slot/pair
//      numbering, then gate/up + SwiGLU over the selected experts' tiles,
//      spread over all warps of all blocks.  h goes to the workspace with a
//      per-pair max |h|.  Grid barrier 2.
//   D  each block owns 16-row output tiles for ALL selected experts: stage h
//      of a group of experts, down GEMV per (warp, expert), multiply by the
//      routing weight and accumulate per token, reduce the warps in a fixed
//      order and write BF16 out.  No further exchange.
// The token index is the MMA's N coordinate throughout (T <= 8 = N), so B
// fragments of x are shared by every expert and per-token results land in the
// lane that owns the token.  The code is kept small on purpose: each phase
// runs once per layer, so instruction fetch is on the critical path.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kFT = 256;
constexpr int kFW = 8;
constexpr int kTF = 8;             // tokens (MMA N)
constexpr int kRE = 2;             // router experts per block
constexpr int kPD = 8;             // gate/up register ring depth (chunks)
constexpr int kPD2 = 4;            // down register ring depth (chunks)
constexpr int kSlotsF = kTF * kMaxTopK + kMaxShared;   // slots of a call with T <= 8
constexpr unsigned kSpinLimit = 1u << 22;               // x ~256 ns: about a second

struct FusedArgs {
    const __nv_bfloat16 *x;
    int T;
    __nv_bfloat16 *out;
    int *ids_out;
    float *w_out;
};

struct FusedSmem {
    size_t xrow, logit_off, red_off, oacc_off, total;
};

// [xs: 8 permuted f16 rows][logits T*E][red][oacc].  Phase D stages h over
// [0, red_off).
__host__ __device__ inline FusedSmem fused_smem_layout(int H, int E, int T) {
    FusedSmem L;
    L.xrow = (size_t)H * 2 + 16;
    L.logit_off = (kTF * L.xrow + 15) & ~(size_t)15;
    L.red_off = L.logit_off + (((size_t)T * E * 4 + 15) & ~(size_t)15);
    L.oacc_off = L.red_off + (size_t)kFW * 4 * 32 * 4;
    L.total = L.oacc_off + (size_t)kFW * 4 * 32 * 4;
    return L;
}

// Grid barrier in two halves so that work can run between arriving and
// waiting.  Sense by generation: the last block to arrive resets the counter
// and bumps the generation.  Waits are bounded; on give-up the sticky error
// word is set and false is returned.
__device__ __forceinline__ unsigned gbar_arrive(unsigned *count, unsigned *gen, unsigned nblocks) {
    unsigned my = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
        my = ld_acquire_gpu(gen);
        __threadfence();
        if (atomicAdd(count, 1u) == nblocks - 1) {
            *count = 0u;
            __threadfence();
            atomicAdd(gen, 1u);
        }
    }
    return my;
}

__device__ __forceinline__ bool gbar_wait(unsigned *gen, unsigned my, int *err) {
    __shared__ int s_ok;
    if (threadIdx.x == 0) {
        int ok = 1;
        unsigned it = 0;
        while (ld_acquire_gpu(gen) == my) {
            if (++it > kSpinLimit) {
                atomicExch(err, 1);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// Elements of piece j (16 bytes, positions 8j..8j+7) of a permuted 64-element
// chunk come in four pairs of consecutive elements starting at piece_pair(j, i).
__device__ __forceinline__ int piece_pair(int j, int i) {
    const int q = j >> 1, kb = 2 * (j & 1) + (i >> 1);
    return 16 * kb + 8 * (i & 1) + 2 * q;
}

__device__ __forceinline__ float2 h2f(uint32_t v) {
    return __half22float2(*reinterpret_cast<__half2 *>(&v));
}

__device__ __forceinline__ bool ranks_before(float s, int e, float bs, int be) {
    return s > bs || (s == bs && e < be);
}

// decode + 4 MMAs of one chunk against the B row of this lane's column
__device__ __forceinline__ void chunk_mma(const uint4 &cw, const uint2 &sw, const uint8_t *bp,
                                          float (&acc)[4]) {
    uint32_t a[4][4];
    decode_chunk(cw, sw, a);
    const uint4 b01 = lds128(bp);
    const uint4 b23 = lds128(bp + 16);
    mma_16816(acc, a[0][0], a[0][1], a[0][2], a[0][3], b01.x, b01.y);
    mma_16816(acc, a[1][0], a[1][1], a[1][2], a[1][3], b01.z, b01.w);
    mma_16816(acc, a[2][0], a[2][1], a[2][2], a[2][3], b23.x, b23.y);
    mma_16816(acc, a[3][0], a[3][1], a[3][2], a[3][3], b23.z, b23.w);
}

__device__ __forceinline__ float silu_fast(float v) { return v * __fdividef(1.0f, 1.0f + __expf(-v)); }

__device__ __forceinline__ void hmax_publish(unsigned long long *hm, int p, unsigned epoch, float v) {
    atomicMax(hm + p, ((unsigned long long)epoch << 32) | (unsigned long long)__float_as_uint(v));
}

__device__ __forceinline__ float hmax_read(const unsigned long long *hm, int p, unsigned epoch) {
    const unsigned long long v = __ldcg(hm + p);
    return (unsigned)(v >> 32) == epoch ? __uint_as_float((unsigned)v) : 0.f;
}

template <int XP>
__global__ void __launch_bounds__(kFT, 2) fused_kernel(DevLayer d, FusedArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float s_tmax[kFW][kTF];
    __shared__ int s_xexp[kTF];
    __shared__ unsigned s_epoch;
    __shared__ int s_ids[kTF][kMaxTopK];
    __shared__ float s_w[kTF][kMaxTopK];
    __shared__ __align__(4) unsigned char s_tokmask[kMaxExperts];
    __shared__ int s_slot_e[kSlotsF];
    __shared__ int s_slot_mask[kSlotsF];
    __shared__ int s_slot_p0[kSlotsF];
    __shared__ float s_pw[kTF * (kMaxTopK + kMaxShared)];
    __shared__ int s_wsum[kFW][2];
    __shared__ int s_nslots;
    __shared__ int s_grp[kSlotsF + 1];
    __shared__ int s_ngrp;
    __shared__ int s_rowidx[kFW][kTF];
    __shared__ float s_rowunscale[64];

    const int T = a.T, H = d.H, E = d.E, K = d.k, S = d.S;
    const int G = gridDim.x, c = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const FusedSmem SL = fused_smem_layout(H, E, T);
    uint8_t *xs = smem;
    float *s_logit = reinterpret_cast<float *>(smem + SL.logit_off);
    float *red = reinterpret_cast<float *>(smem + SL.red_off);
    float *oacc = reinterpret_cast<float *>(smem + SL.oacc_off);
    const int npieces = H / 8;               // 16-byte pieces per activation row
    const int NC13 = H / kChunkK;            // gate/up chunks per tile
    const int NTs = d.Is / 8, NT13 = d.I / 8, NRT = H / 16;

    MOE_TRACE_POINT(0, 0);
    const uint64_t pol = evict_first_policy();
    // ---------------- A: bulk L2 prefetch of static weights ----------------
    if (threadIdx.x < kRE) {
        const int e = c + threadIdx.x * G;
        if (e < E) prefetch_l2(d.router_w + (size_t)e * H, (unsigned)H * 4);
    } else if (threadIdx.x == 32 && S > 0 && c < S * NTs) {
        prefetch_l2(d.sw13r + (size_t)(c / NTs) * d.s13_stride + (size_t)(c % NTs) * NC13 * kChunkBytes,
                    (unsigned)(NC13 * kChunkBytes));
    } else if (threadIdx.x == 64 && S > 0 && c < NRT) {
        prefetch_l2(d.sw2r + (size_t)c * (d.Is / kChunkK) * kChunkBytes, (unsigned)(d.Is / kChunkK * kChunkBytes));
    }
    pdl_wait();
    pdl_trigger();
    MOE_TRACE_POINT(0, 1);

    // ---------------- B: x, logits ----------------
    // router rows of this block's experts: the four element pairs of each of
    // this thread's pieces (served from L2 by the prefetch above)
    float2 wr[kRE][XP][4];
#pragma unroll
    for (int re = 0; re < kRE; ++re) {
        const int e = c + re * G;
#pragma unroll
        for (int xp = 0; xp < XP; ++xp) {
            const int P = threadIdx.x + xp * kFT;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                wr[re][xp][i] = (e < E && P < npieces)
                                    ? ld_nc_f2(d.router_w + (size_t)e * H + (P >> 3) * kChunkK + piece_pair(P & 7, i))
                                    : make_float2(0.f, 0.f);
        }
    }
    if (threadIdx.x == 0) s_epoch = __ldcg(d.epoch);
    if (threadIdx.x < S) {
        s_slot_e[threadIdx.x] = -(threadIdx.x + 1);
        s_slot_mask[threadIdx.x] = (1 << T) - 1;
        s_slot_p0[threadIdx.x] = threadIdx.x * T;
    }
    {
        // x rows -> registers, per-token max |x| -> exact power-of-two prescale
        uint4 xv[kTF][XP];
#pragma unroll
        for (int t = 0; t < kTF; ++t)
#pragma unroll
            for (int xp = 0; xp < XP; ++xp) {
                const int P = threadIdx.x + xp * kFT;
                xv[t][xp] = (t < T && P < npieces)
                                ? __ldcg(reinterpret_cast<const uint4 *>(a.x + (size_t)t * H) + P)
                                : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
        for (int t = 0; t < kTF; ++t) {
            float m = 0.f;
#pragma unroll
            for (int xp = 0; xp < XP; ++xp) {
                const uint32_t w4[4] = {xv[t][xp].x, xv[t][xp].y, xv[t][xp].z, xv[t][xp].w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[u] << 16)), fabsf(__uint_as_float(w4[u] & 0xFFFF0000u))));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0) s_tmax[warp][t] = m;
        }
        __syncthreads();
        if (threadIdx.x < kTF) {
            float m = 0.f;
            for (int w = 0; w < kFW; ++w) m = fmaxf(m, s_tmax[w][threadIdx.x]);
            s_xexp[threadIdx.x] = max(-100, exp_for_f16(m));
        }
        __syncthreads();
        // x' = x * 2^-xexp as f16, permuted within each 64-element chunk
        // (element 16kb + 8h + 2q + e at half 16q + 4kb + 2h + e); rows >= T zero
#pragma unroll
        for (int t = 0; t < kTF; ++t) {
            const float sc = pow2f(-s_xexp[t]);
#pragma unroll
            for (int xp = 0; xp < XP; ++xp) {
                const int P = threadIdx.x + xp * kFT;
                if (P < npieces) {
                    uint32_t *dst = reinterpret_cast<uint32_t *>(xs + (size_t)t * SL.xrow + (P >> 3) * 128 +
                                                                 ((P & 7) >> 1) * 8 + (P & 1) * 4);
                    const uint32_t w4[4] = {xv[t][xp].x, xv[t][xp].y, xv[t][xp].z, xv[t][xp].w};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[u * 8] = pack_f16x2(__uint_as_float(w4[u] << 16) * sc,
                                                __uint_as_float(w4[u] & 0xFFFF0000u) * sc);
                }
            }
        }
    }
    __syncthreads();
    MOE_TRACE_POINT(0, 2);
    // logits: this thread's permuted pieces against the matching router pairs
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
        float acc[kRE];
#pragma unroll
        for (int re = 0; re < kRE; ++re) acc[re] = 0.f;
#pragma unroll
        for (int xp = 0; xp < XP; ++xp) {
            const int P = threadIdx.x + xp * kFT;
            if (P < npieces) {
                const uint4 v = lds128(xs + (size_t)t * SL.xrow + (P >> 3) * 128 + (P & 7) * 16);
                const float2 x0 = h2f(v.x), x1 = h2f(v.y), x2 = h2f(v.z), x3 = h2f(v.w);
#pragma unroll
                for (int re = 0; re < kRE; ++re) {
                    float s = acc[re];
                    s = fmaf(x0.x, wr[re][xp][0].x, s);
                    s = fmaf(x0.y, wr[re][xp][0].y, s);
                    s = fmaf(x1.x, wr[re][xp][1].x, s);
                    s = fmaf(x1.y, wr[re][xp][1].y, s);
                    s = fmaf(x2.x, wr[re][xp][2].x, s);
                    s = fmaf(x2.y, wr[re][xp][2].y, s);
                    s = fmaf(x3.x, wr[re][xp][3].x, s);
                    s = fmaf(x3.y, wr[re][xp][3].y, s);
                    acc[re] = s;
                }
            }
        }
#pragma unroll
        for (int re = 0; re < kRE; ++re) {
            float v = acc[re];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) red[(warp * kRE + re) * kTF + t] = v;
        }
    }
    __syncthreads();
    if (threadIdx.x < kRE * kTF) {
        const int re = threadIdx.x / kTF, t = threadIdx.x % kTF;
        const int e = c + re * G;
        if (e < E && t < T) {
            float v = 0.f;
            for (int w = 0; w < kFW; ++w) v += red[(w * kRE + re) * kTF + t];
            v *= pow2f(s_xexp[t]);             // exact: undoes the prescale
            if (d.router_b) v += d.router_b[e];
            d.logits[(size_t)t * E + e] = v;
        }
    }
    const unsigned bar1 = gbar_arrive(d.bar_count, d.bar_gen, G);
    MOE_TRACE_POINT(0, 3);

    // ---------------- C: gate/up, pass 0 shared experts, pass 1 routed ----------------
    uint4 cb[kPD];
    uint2 sb[kPD];
    int nslots = S;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        if (pass == 1) {
            MOE_TRACE_POINT(0, 4);
            if (!gbar_wait(d.bar_gen, bar1, d.err)) return;
            MOE_TRACE_POINT(0, 5);
            // routing, identical in every block
            for (int i = threadIdx.x; i < T * E; i += kFT) s_logit[i] = __ldcg(d.logits + i);
            for (int i = threadIdx.x; i < E; i += kFT) s_tokmask[i] = 0;
            __syncthreads();
            if (warp < T) {
                const int t = warp;
                float sc[kMaxExperts / 32];
#pragma unroll
                for (int m = 0; m < kMaxExperts / 32; ++m) {
                    const int ee = lane + 32 * m;
                    float s = -INFINITY;
                    if (ee < E) {
                        const float z = s_logit[t * E + ee];
                        s = isnan(z) ? -INFINITY : __fdividef(1.0f, 1.0f + __expf(-z));
                    }
                    sc[m] = s;
                }
                unsigned taken = 0u;
                float sel_s = 0.f;
                int sel_e = 0;
#pragma unroll 1
                for (int j = 0; j < K; ++j) {
                    float bs = -INFINITY;
                    int be = 0x7fffffff;
#pragma unroll
                    for (int m = 0; m < kMaxExperts / 32; ++m) {
                        const int ee = lane + 32 * m;
                        if (ee < E && !(taken & (1u << m)) && ranks_before(sc[m], ee, bs, be)) {
                            bs = sc[m];
                            be = ee;
                        }
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const float os = __shfl_xor_sync(0xffffffffu, bs, off);
                        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                        if (ranks_before(os, oe, bs, be)) {
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
                float sum = 0.f;
                for (int j = 0; j < K; ++j) sum += __shfl_sync(0xffffffffu, sel_s, j);
                if (lane < K) {
                    const float w = (d.normalize ? sel_s / sum : sel_s) * d.routed_scale;
                    s_ids[t][lane] = sel_e;
                    s_w[t][lane] = w;
                    atomicOr(reinterpret_cast<unsigned *>(s_tokmask) + (sel_e >> 2), 1u << (8 * (sel_e & 3) + t));
                    if (c == 0) {
                        if (a.ids_out) a.ids_out[t * K + lane] = sel_e;
                        if (a.w_out) a.w_out[t * K + lane] = w;
                    }
                }
            }
            __syncthreads();
            // slots: shared first, then routed experts in ascending id; an
            // expert's pairs are contiguous, tokens ascending
            {
                const int per = (E + kFT - 1) / kFT;
                const int e0 = threadIdx.x * per;
                int fsum = 0, csum = 0;
                for (int i = 0; i < per; ++i)
                    if (e0 + i < E) {
                        const int cnt = __popc(s_tokmask[e0 + i]);
                        fsum += cnt > 0;
                        csum += cnt;
                    }
                int finc = fsum, cinc = csum;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int x1 = __shfl_up_sync(0xffffffffu, finc, off);
                    const int x2 = __shfl_up_sync(0xffffffffu, cinc, off);
                    if (lane >= off) {
                        finc += x1;
                        cinc += x2;
                    }
                }
                if (lane == 31) {
                    s_wsum[warp][0] = finc;
                    s_wsum[warp][1] = cinc;
                }
                __syncthreads();
                int fb = finc - fsum, cbse = cinc - csum;
                for (int w = 0; w < warp; ++w) {
                    fb += s_wsum[w][0];
                    cbse += s_wsum[w][1];
                }
                for (int i = 0; i < per; ++i)
                    if (e0 + i < E && s_tokmask[e0 + i]) {
                        const int msk = s_tokmask[e0 + i];
                        s_slot_e[S + fb] = e0 + i;
                        s_slot_mask[S + fb] = msk;
                        s_slot_p0[S + fb] = S * T + cbse;
                        fb += 1;
                        cbse += __popc(msk);
                    }
                if (threadIdx.x == kFT - 1) s_nslots = S + fb;
                __syncthreads();
                for (int it = threadIdx.x; it < T * K; it += kFT) {
                    const int t = it / K, j = it % K, e = s_ids[t][j];
                    int slot = S;
                    while (s_slot_e[slot] != e) ++slot;     // <= T*k slots
                    s_pw[s_slot_p0[slot] + __popc(s_slot_mask[slot] & ((1 << t) - 1))] = s_w[t][j];
                }
                for (int it = threadIdx.x; it < T * S; it += kFT) s_pw[it] = 1.0f;
                __syncthreads();
            }
            nslots = s_nslots;
            MOE_TRACE_POINT(0, 6);
        }
        // units (slot, 16-row tile) of this pass; ks warps split a unit's K
        const int slot_lo = pass == 0 ? 0 : S;
        const int NT = pass == 0 ? NTs : NT13;
        const int units = (pass == 0 ? S : nslots - S) * NT;
        int ks = 1;
        while (ks < kFW && NC13 % (2 * ks) == 0 && units * 2 * ks <= G * kFW) ks *= 2;
        const int ngrp = kFW / ks, gi = warp / ks, kw = warp % ks;
        const int cpw = NC13 / ks, cb0 = kw * cpw;
        int R = cpw < kPD ? cpw : kPD;           // ring depth: divides cpw
        while (cpw % R) --R;
        const int stride = G * ngrp, u0 = c * ngrp + gi;
        const int my_units = u0 < units ? (units - u0 + stride - 1) / stride : 0;
        auto unit_base = [&](int ui) -> const uint8_t * {
            const int uu = u0 + ui * stride;
            const int e = s_slot_e[slot_lo + uu / NT], r = uu % NT;
            const uint8_t *b = e < 0 ? d.sw13r + (size_t)(-e - 1) * d.s13_stride : d.w13r + (size_t)e * d.e13_stride;
            return b + (size_t)r * NC13 * kChunkBytes;
        };
        if (my_units > 0) {
            const uint8_t *b0 = unit_base(0);
#pragma unroll
            for (int i = 0; i < kPD; ++i)
                if (i < R) load_chunk(b0, cb0 + i, lane, cb[i], sb[i], pol);
        }
        const uint8_t *brow = xs + (size_t)g * SL.xrow + q * 32;
        // every warp of a group has the same unit count, so the group's named
        // barrier (id 1 + gi) is reached by all of its warps together
#pragma unroll 1
        for (int ui = 0; ui < my_units; ++ui) {
            const uint8_t *cur = unit_base(ui);
            const uint8_t *nxt = ui + 1 < my_units ? unit_base(ui + 1) : nullptr;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int c0 = 0; c0 < cpw; c0 += R) {
#pragma unroll
                for (int i = 0; i < kPD; ++i) {
                    if (i < R) {
                        const int cc = c0 + i;
                        chunk_mma(cb[i], sb[i], brow + (cb0 + cc) * 128, acc);
                        const int cn = cc + R;
                        if (cn < cpw) load_chunk(cur, cb0 + cn, lane, cb[i], sb[i], pol);
                        else if (nxt) load_chunk(nxt, cb0 + cn - cpw, lane, cb[i], sb[i], pol);
                    }
                }
            }
            const int uu = u0 + ui * stride;
            const int slot = slot_lo + uu / NT, r = uu % NT;
            if (ks > 1) {
#pragma unroll
                for (int v = 0; v < 4; ++v) red[(warp * 4 + v) * 32 + lane] = acc[v];
                asm volatile("bar.sync %0, %1;\n" ::"r"(1 + gi), "r"(32 * ks) : "memory");
                if (kw == 0)
                    for (int w = 1; w < ks; ++w)
#pragma unroll
                        for (int v = 0; v < 4; ++v) acc[v] += red[((warp + w) * 4 + v) * 32 + lane];
                asm volatile("bar.sync %0, %1;\n" ::"r"(1 + gi), "r"(32 * ks) : "memory");
            }
            if (kw == 0) {
                // SwiGLU: tile rows 0..7 gate, 8..15 up of intermediate row 8r+g
                const int e = s_slot_e[slot];
                const int msk = s_slot_mask[slot], p0 = s_slot_p0[slot];
                const float gsa = e < 0 ? d.sgs13[2 * (-e - 1)] : d.gs13[2 * e];
                const float gsb = e < 0 ? d.sgs13[2 * (-e - 1) + 1] : d.gs13[2 * e + 1];
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int t = 2 * q + e2;
                    const bool on = t < T && ((msk >> t) & 1);
                    const int p = p0 + __popc(msk & ((1 << t) - 1));
                    float habs = 0.f;
                    if (on) {
                        const float un = pow2f(s_xexp[t]);
                        const float gt = acc[e2] * gsa * un, up = acc[2 + e2] * gsb * un;
                        const __nv_bfloat16 hb = __float2bfloat16_rn(silu_fast(gt) * up);
                        d.h_ws[(size_t)p * d.Imax + 8 * r + g] = hb;
                        habs = fabsf(__bfloat162float(hb));
                    }
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1)
                        habs = fmaxf(habs, __shfl_xor_sync(0xffffffffu, habs, off));
                    if (g == 0 && on) hmax_publish(d.hmax64, p, s_epoch, habs);
                }
            }
        }
    }
    MOE_TRACE_POINT(0, 7);

    // ---------------- D plan: groups of experts whose h rows fit in smem ----------------
    const size_t hrow = (size_t)d.Imax * 2 + 16;
    const int rows_cap = (int)(SL.red_off / hrow) - 1;       // last row: zeros
    if (threadIdx.x == 0) {
        int ng = 0, s0 = 0;
        while (s0 < nslots) {
            int s1 = s0, rows = 0;
            while (s1 < nslots && s1 - s0 < kFW && rows + __popc(s_slot_mask[s1]) <= rows_cap) {
                rows += __popc(s_slot_mask[s1]);
                ++s1;
            }
            s_grp[ng++] = s0;
            s0 = s1;
        }
        s_grp[ng] = nslots;
        s_ngrp = ng;
    }
    const unsigned bar2 = gbar_arrive(d.bar_count, d.bar_gen, G);
    if (!gbar_wait(d.bar_gen, bar2, d.err)) return;
    MOE_TRACE_POINT(0, 8);

    // ---------------- D: down + combine, 16 output rows per tile ----------------
    const int ngroups = s_ngrp;
    uint8_t *hs = smem;
    uint4 db[kPD2];
    uint2 dsb[kPD2];
#pragma unroll 1
    for (int rt = c; rt < NRT; rt += G) {
        float oa[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = threadIdx.x; i < (int)(hrow / 16); i += kFT)
            reinterpret_cast<uint4 *>(hs + (size_t)rows_cap * hrow)[i] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
        for (int gk = 0; gk < ngroups; ++gk) {
            const int sa = s_grp[gk], sbnd = s_grp[gk + 1];
            const int myslot = sa + warp < sbnd ? sa + warp : -1;
            // this warp's weights do not depend on h: start them first
            const uint8_t *src = nullptr;
            int nc = 0;
            if (myslot >= 0) {
                const int e = s_slot_e[myslot];
                const int I = e < 0 ? d.Is : d.I;
                nc = I / kChunkK;
                src = (e < 0 ? d.sw2r + (size_t)(-e - 1) * d.s2_stride : d.w2r + (size_t)e * d.e2_stride) +
                      (size_t)rt * nc * kChunkBytes;
#pragma unroll
                for (int i = 0; i < kPD2; ++i)
                    if (i < nc) load_chunk(src, i, lane, db[i], dsb[i], pol);
            }
            __syncthreads();
            // row table: slot (sa + w), token column n -> staged row or the zero row
            int nrows = 0;
            for (int s2 = sa; s2 < sbnd; ++s2) nrows += __popc(s_slot_mask[s2]);
            if (threadIdx.x < kFW * kTF) {
                const int w = threadIdx.x / kTF, n = threadIdx.x % kTF;
                int row = rows_cap;
                if (sa + w < sbnd) {
                    int base = 0;
                    for (int s2 = sa; s2 < sa + w; ++s2) base += __popc(s_slot_mask[s2]);
                    const int msk = s_slot_mask[sa + w];
                    if (n < T && ((msk >> n) & 1)) row = base + __popc(msk & ((1 << n) - 1));
                }
                s_rowidx[w][n] = row;
            }
            const int p_first = s_slot_p0[sa];
            if (threadIdx.x < nrows)
                s_rowunscale[threadIdx.x] = pow2f(max(-100, exp_for_f16(hmax_read(d.hmax64, p_first + threadIdx.x, s_epoch))));
            __syncthreads();
            // stage the group's h rows (pairs p_first.. are contiguous) as f16
            {
                const int pieces = d.Imax / 8;
                const int items = nrows * pieces;
#pragma unroll 1
                for (int base = threadIdx.x; base < items; base += 2 * kFT) {
                    uint4 v[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int it = base + u * kFT;
                        if (it < items) {
                            const int j = it / pieces;
                            v[u] = __ldcg(reinterpret_cast<const uint4 *>(d.h_ws + (size_t)(p_first + j) * d.Imax) +
                                          (it - j * pieces));
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int it = base + u * kFT;
                        if (it < items) {
                            const int j = it / pieces, P = it - j * pieces;
                            uint32_t *dst = reinterpret_cast<uint32_t *>(hs + (size_t)j * hrow + (P >> 3) * 128 +
                                                                         ((P & 7) >> 1) * 8 + (P & 1) * 4);
                            const float sc = __fdividef(1.0f, s_rowunscale[j]);   // exact: a power of two
                            const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                            for (int uu = 0; uu < 4; ++uu)
                                dst[uu * 8] = pack_f16x2(__uint_as_float(w4[uu] << 16) * sc,
                                                         __uint_as_float(w4[uu] & 0xFFFF0000u) * sc);
                        }
                    }
                }
            }
            __syncthreads();
            if (myslot >= 0) {
                const uint8_t *bp = hs + (size_t)s_rowidx[warp][g] * hrow + q * 32;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                for (int c0 = 0; c0 < nc; c0 += kPD2) {
#pragma unroll
                    for (int i = 0; i < kPD2; ++i) {
                        const int cc = c0 + i;
                        if (cc < nc) {
                            chunk_mma(db[i], dsb[i], bp + cc * 128, acc);
                            if (cc + kPD2 < nc) load_chunk(src, cc + kPD2, lane, db[i], dsb[i], pol);
                        }
                    }
                }
                // y = gs * 2^hexp * acc, weighted into the per-token accumulator
                const int e = s_slot_e[myslot];
                const float gs = e < 0 ? d.sgs2[-e - 1] : d.gs2[e];
                const int msk = s_slot_mask[myslot], p0 = s_slot_p0[myslot];
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int t = 2 * q + e2;
                    if (t < T && ((msk >> t) & 1)) {
                        const float wgt = s_pw[p0 + __popc(msk & ((1 << t) - 1))] * gs * s_rowunscale[s_rowidx[warp][t]];
                        oa[e2] = fmaf(wgt, acc[e2], oa[e2]);
                        oa[2 + e2] = fmaf(wgt, acc[2 + e2], oa[2 + e2]);
                    }
                }
            }
        }
        // fixed-order reduction over warps, BF16 out
#pragma unroll
        for (int v = 0; v < 4; ++v) oacc[(warp * 4 + v) * 32 + lane] = oa[v];
        __syncthreads();
        if (warp == 0) {
            float o[4] = {0.f, 0.f, 0.f, 0.f};
            for (int w = 0; w < kFW; ++w)
#pragma unroll
                for (int v = 0; v < 4; ++v) o[v] += oacc[(w * 4 + v) * 32 + lane];
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int t = 2 * q + e2;
                if (t < T) {
                    a.out[(size_t)t * H + 16 * rt + g] = __float2bfloat16_rn(o[e2]);
                    a.out[(size_t)t * H + 16 * rt + g + 8] = __float2bfloat16_rn(o[2 + e2]);
                }
            }
        }
    }
    MOE_TRACE_POINT(0, 9);
    if (c == 0 && threadIdx.x == 0) *d.epoch = s_epoch + 1u;
}

}  // namespace

// Largest T for which moe_decode_forward picks the single launch: above it the
// three-kernel chain streams the weights faster (more warps per SM).
constexpr int kFusedMaxT = 1;

bool fused_eligible(const DevLayer &d, int T, int sm_count, size_t optin_smem) {
    if (T < 1 || T > kFusedMaxT) return false;
    if (d.E > kRE * sm_count) return false;
    if (d.H / 8 > 2 * kFT) return false;                    // x pieces: at most two per thread
    if (d.k * T + d.S > kSlotsF) return false;
    const FusedSmem L = fused_smem_layout(d.H, d.E, T);
    const size_t hrow = (size_t)d.Imax * 2 + 16;
    if ((int)(L.red_off / hrow) - 1 < kTF) return false;    // one expert's 8 rows + the zero row
    if (L.total + 8 * 1024 > optin_smem / 2) return false;  // two blocks per SM
    return true;
}

cudaError_t launch_fused(const DevLayer &d, const __nv_bfloat16 *x, int T, __nv_bfloat16 *out, int *ids,
                         float *w, int sm_count, cudaStream_t s) {
    const FusedSmem L = fused_smem_layout(d.H, d.E, T);
    FusedArgs a{x, T, out, ids, w};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sm_count);
    cfg.blockDim = dim3(kFT);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (d.H / 8 > kFT) return cudaLaunchKernelEx(&cfg, fused_kernel<2>, d, a);
    return cudaLaunchKernelEx(&cfg, fused_kernel<1>, d, a);
}

cudaError_t prepare_fused_kernel(int optin_bytes) {
    cudaError_t e = allow_max_dynamic_smem(fused_kernel<1>, optin_bytes / 2);
    if (e == cudaSuccess) e = allow_max_dynamic_smem(fused_kernel<2>, optin_bytes / 2);
    return e;
}

int fused_blocks_per_sm(const DevLayer &d, int T) {
    const FusedSmem L = fused_smem_layout(d.H, d.E, T);
    int n = 0;
    cudaError_t e = d.H / 8 > kFT
                        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fused_kernel<2>, kFT, L.total)
                        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fused_kernel<1>, kFT, L.total);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace moe
