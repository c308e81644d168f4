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
// One block of 16 warps per SM (grid = SM count, all resident).  Weights move
// from HBM to shared memory by bulk asynchronous copies (cp.async.bulk, the
// 1-D TMA): every warp owns a ring of RW segments of up to CH 576-byte chunks,
// one mbarrier per segment.  Lane 0 issues the copies; the warp decodes and
// multiplies from shared memory.  A warp's segments form one list -- its
// shared-expert gate/up units, then its routed gate/up units, then its down
// pieces -- and lane 0 keeps the ring full along that list, across phase
// boundaries: the down weights do not depend on h, so their copies are in
// flight while gate/up still runs (for one token, a block's whole share of
// the layer's selected weights fits in its rings and is requested right
// after routing).
//
// Phases (no grid barrier: values that cross blocks travel as words tagged
// with the call number and are polled by their readers):
//   A  before griddepcontrol.wait: copy this block's router rows and the
//      packed global scales into shared memory; start the rings of the
//      shared-expert pass; L2-prefetch this block's rows of the shared down
//      weights.
//   B  x (T rows) arrives by each thread's own asynchronous copies of the
//      quads it reads (plain loads from pinned host memory when x lives
//      there); one pass over it gives the
//      per-token max |x| and this block's experts' FP32 logits, published as
//      tagged words; the shared-expert warps stage x as the f16 MMA operand
//      (exact per-row power-of-two prescale).
//   C  pass 0: one warp per token polls all logits and takes the top-k (the
//      same in every block) while, for one or two tokens, the shared-expert
//      warps run their gate/up units (for more tokens those wait for pass 1,
//      where they run first); pass 1: the routed gate/up units.  SwiGLU in
//      the epilogue; h is published as tagged words.
//   D  h is gathered from the tagged words as f16 (an exact power-of-two
//      prescale per piece); each block owns 16-row output tiles for all
//      slots: down GEMV per (slot, K part) and warp, routing weight, a
//      fixed-order warp reduction, BF16 out.
// The token index is the MMA's N coordinate throughout (T <= 8 = N), so the
// B fragments of x are shared by every expert and per-token results land in
// the lane that owns the token.
//
// Everything between the weight streams is a short serial step executed once
// per layer, from a cold instruction cache, so the work split is planned on
// the host (tables indexed by the slot count) and the code of those steps is
// kept short (one kernel instance per token-count class).
#include <algorithm>

#include "moe_internal.cuh"

namespace moe {

namespace {

// Phase point i of the traced build: %globaltimer under kernel slot 0 (for
// the order across blocks) and the SM clock under slot 3 (cycle-exact within
// a block).
#define FUSED_TRACE(i)           \
    do {                         \
        MOE_TRACE_POINT(0, (i)); \
        MOE_TRACE_CLOCK(3, (i)); \
    } while (0)

constexpr int kFW = 16;                                  // warps per block
constexpr int kFT = 32 * kFW;
constexpr int kTF = 8;                                   // tokens (MMA N)
constexpr int kPW = 8;                                   // warps of the shared-expert pass (see pass0_index)
constexpr int kStageBar = 15;                            // named barrier of the x staging (the kPW pass-0 warps)
constexpr int kGroupBar1 = 1;                            // split-K groups of the routed pass: ids 1..8
constexpr int kGroupBar0 = 9;                            // of the shared-expert pass: ids 9..12
static_assert(kGroupBar1 + kFW / 2 <= kGroupBar0 && kGroupBar0 + kPW / 2 <= kStageBar, "named barrier ids overlap");
constexpr int kREmax = 4;                                // router experts per block
static_assert(kTF * kREmax == 32, "the logit reduction gives each lane one (token, expert) value");
static_assert(kTF + kPW <= kFW, "routing warps and shared-expert warps are distinct");
constexpr int kCHmax = 8;                                // chunks per ring segment
constexpr int kCHmin = 4;
constexpr int kRWmax = 6;                                // ring segments per warp
constexpr int kSlotsF = kFusedSlots;                     // slots of a call with T <= 8
constexpr int kPairsF = kFusedPairs;                     // pairs of a call with T <= 8
constexpr int kM1max = 8;                                // experts per lane in the top-k (E <= 256)
constexpr int kTabMax = 32;                              // copy-list items per warp
constexpr int kHU = 8;                                   // tagged h pieces in flight per lane
constexpr int kHU2 = 6;                                  // per task when two tasks share a poll
constexpr unsigned long long kWaitNs = 1000000000ull;    // in-kernel waits give up after ~1 s

struct FusedArgs {
    const __nv_bfloat16 *x;
    int T;
    __nv_bfloat16 *out;
    int *ids_out;
    float *w_out;
    int x_sys;   // x is the device alias of pinned host memory: read by plain loads
};

// Launch geometry and host-planned work split.
// Dynamic shared memory: [phase-local region | rings].  The phase-local
// region holds x as the f16 MMA operand (T+1 rows, the last one zero), the
// router rows and x as copied (BF16) during phases
// B/C, and the staged h rows (all pairs + a zero row) during phase D; then
// the packed per-expert global scales and router biases for the whole call.
struct FusedGeom {
    int kRE, RW, CH;
    int xrow, hrow;
    int router_off, xraw_off, hs_off, gs_off, ring_off, total;
    int m1p;                                // top-k: experts per lane (1, 2, 4, 8)
    int lks0;                               // log2 of the pass-0 K split
    unsigned char lks1[kSlotsF + 1];        // log2 of the pass-1 K split, by slot count
    unsigned char lksd[kSlotsF + 1];        // log2 of the down K split, by slot count
};

inline size_t up16(size_t v) { return (v + 15) & ~(size_t)15; }

// Groups of ks warps share a gate/up unit by splitting K; ks minimises the
// chunks of the busiest warp plus one chunk's worth per unit (the epilogue)
// and, when K is split, two more per unit: the group's named barrier (where
// its warps wait for the one whose data came last) and the reduction.
int choose_lks(int units, int NC, int G, int nw) {
    int best = 0, bestc = 0x7fffffff;
    for (int l = 0; (1 << l) <= nw && NC % (1 << l) == 0; ++l) {
        const int groups = G * (nw >> l);
        const int cost = (units + groups - 1) / groups * (NC / (1 << l) + 1 + (l > 0 ? 2 : 0));
        if (cost < bestc) {
            bestc = cost;
            best = l;
        }
    }
    return best;
}

bool fused_geometry(const DevLayer &d, int T, int G, int dyn_max, FusedGeom &g) {
    g.kRE = (d.E + G - 1) / G;
    g.xrow = d.H * 2 + 16;
    g.hrow = d.Imax * 2 + 16;
    g.m1p = 1;
    while (32 * g.m1p < d.E) g.m1p *= 2;
    if (g.m1p > kM1max) return false;
    const size_t xs = (size_t)(T + 1) * g.xrow;
    g.router_off = (int)up16(xs);
    g.xraw_off = g.router_off + (int)up16((size_t)g.kRE * d.H * 4);
    const size_t pB = (size_t)g.xraw_off + (size_t)T * d.H * 2;
    const size_t pD = (size_t)(T * (d.k + d.S) + 1) * g.hrow;
    // the staged h rows of phase D: for T <= 2 behind x (over the router rows
    // and the copied x, both dead by then), so that a warp may gather and
    // use its h while other warps still read x; else over x as well
    g.hs_off = T <= 2 ? g.router_off : 0;
    g.gs_off = (int)((std::max(pB, (size_t)g.hs_off + pD) + 15) & ~(size_t)15);
    const size_t P = ((size_t)g.gs_off + (size_t)(d.E + d.S) * 16 + 127) & ~(size_t)127;
    g.ring_off = (int)P;
    if ((long)dyn_max <= (long)P) return false;
    const size_t per_warp = ((size_t)dyn_max - P) / kFW;
    g.CH = (int)std::min<size_t>(kCHmax, per_warp / (2 * kChunkBytes));
    if (g.CH < kCHmin) return false;
    g.RW = (int)std::min<size_t>(kRWmax, per_warp / ((size_t)g.CH * kChunkBytes));
    g.total = (int)(P + (size_t)kFW * g.RW * g.CH * kChunkBytes);
    if (g.RW < 2) return false;
    const int NTs = d.Is / 8, NT13 = d.I / 8;
    const int NC13s = chunks_of(d.H, d.f8s), NC13r = chunks_of(d.H, d.f8e);
    const int ncr = d.I / kChunkK, ncs = d.S > 0 ? d.Is / kChunkK : ncr;
    g.lks0 = choose_lks(d.S * NTs, NC13s, G, kPW);
    for (int n = 0; n <= kSlotsF; ++n) {
        g.lks1[n] = (unsigned char)choose_lks(std::max(0, n - d.S) * NT13, NC13r, G, kFW);
        int l = 0;
        while (n * (2 << l) <= kFW && ncr % (2 << l) == 0 && ncs % (2 << l) == 0 && ncr / (2 << l) >= 2 &&
               ncs / (2 << l) >= 2)
            ++l;
        g.lksd[n] = (unsigned char)l;
    }
    // every warp's copy list (units of both passes + down pieces) must fit
    // its table, whatever the number of distinct experts
    const int NRT = d.H / 16, nrt = (NRT + G - 1) / G;
    const int my0 = (d.S * NTs + G * (kPW >> g.lks0) - 1) / (G * (kPW >> g.lks0));
    for (int n = d.S + 1; n <= d.S + std::min(d.E, T * d.k); ++n) {
        const int my1 = ((n - d.S) * NT13 + G * (kFW >> g.lks1[n]) - 1) / (G * (kFW >> g.lks1[n]));
        const int perw = ((n << g.lksd[n]) + kFW - 1) / kFW;
        if (my0 + my1 + nrt * perw > kTabMax) return false;
    }
    return true;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Warp roles while the block routes (one routing warp per token).  Warp w
// runs on SM sub-partition w % 4.  For one or two tokens (TT <= 2) token t's
// warp is 4t, on sub-partition 0, and the shared-expert pass runs on the
// warps of sub-partitions 2 and 3, so that its issue-bound decode does not
// share a scheduler with the latency-bound routing.  For more tokens the
// routing's compare-and-select work is the larger cost and is spread over all
// four sub-partitions: token t on warp t, the pass on warps 8..15.
template <int TT>
__device__ __forceinline__ int routed_token_of(int w) {
    if (TT <= 2) return (w & 3) == 0 ? (w >> 2) : -1;
    return w < kPW ? w : -1;
}
// Index of warp w among the kPW warps of the shared-expert pass (kFW if none).
template <int TT>
__device__ __forceinline__ int pass0_index(int w) {
    if (TT <= 2) return (w & 3) >= 2 ? 2 * (w >> 2) + (w & 3) - 2 : kFW;
    return w >= kFW - kPW ? w - (kFW - kPW) : kFW;
}

// Wait for phase `parity` of an mbarrier; gives up after kWaitNs, setting the
// sticky error word.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, unsigned parity, int *err) {
    if (mbar_try_wait(b, parity)) return true;
    const unsigned long long t0 = gtimer();
    while (!mbar_try_wait(b, parity)) {
        if (gtimer() - t0 > kWaitNs) {
            atomicExch(err, 1);
            return false;
        }
    }
    return true;
}

// Words exchanged between the blocks of one call: (tag << 32) | payload,
// written and read with relaxed gpu-scope accesses (each 64-bit word is
// single-copy atomic).  The tag is the number of calls every block has
// finished, plus one, so a word from an earlier call (or zeroed memory) never
// matches and a reader simply polls the words it needs.
// 8-byte asynchronous copy global -> shared
__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(dst)), "l"(__cvta_generic_to_global(src))
                 : "memory");
}

__device__ __forceinline__ void st_tagged(unsigned long long *p, unsigned tag, unsigned payload) {
    const unsigned long long v = ((unsigned long long)tag << 32) | payload;
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_tagged(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void ld_tagged2(const unsigned long long *p, unsigned long long &a,
                                           unsigned long long &b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];\n" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ bool tag_is(unsigned long long v, unsigned tag) { return (unsigned)(v >> 32) == tag; }

__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float silu_fast(float v) { return v * __fdividef(1.0f, 1.0f + __expf(-v)); }

// On give-up: wait (bounded) for the copies a warp still has in flight
// (segments n_done .. n_iss-1: issued, never waited for; lane 0 knows n_iss).
__device__ __forceinline__ void drain_ring(uint64_t *bar, int RW, int n_done, int n_iss, int lane) {
    if (lane != 0) return;
    for (int j = n_done; j < n_iss; ++j) {
        const unsigned long long t0 = gtimer();
        while (!mbar_try_wait(bar + j % RW, (unsigned)((j / RW) & 1)) && gtimer() - t0 < kWaitNs) {
        }
    }
}

// decode + 4 MMAs of one chunk held in shared memory, against the B row of
// this lane's column; blocks 0/2 and 1/3 go to two accumulators so that the
// MMA dependency chain is half as long.
__device__ __forceinline__ void chunk_mma_smem(const uint8_t *ch, int lane, const uint8_t *bp, bool bon,
                                               float (&a0)[4], float (&a1)[4]) {
    const uint4 cw = lds128(ch + 16 * lane);
    uint2 sw;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n"
                 : "=r"(sw.x), "=r"(sw.y) : "r"(smem_u32(ch + kCodeBytes + 8 * (lane >> 2))));
    uint32_t a[4][4];
    decode_chunk(cw, sw, a);
    const uint4 b01 = bon ? lds128(bp) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 b23 = bon ? lds128(bp + 16) : make_uint4(0u, 0u, 0u, 0u);
    mma_16816(a0, a[0][0], a[0][1], a[0][2], a[0][3], b01.x, b01.y);
    mma_16816(a1, a[1][0], a[1][1], a[1][2], a[1][3], b01.z, b01.w);
    mma_16816(a0, a[2][0], a[2][1], a[2][2], a[2][3], b23.x, b23.y);
    mma_16816(a1, a[3][0], a[3][1], a[3][2], a[3][3], b23.z, b23.w);
}

// Top-k of token t from the tagged logits (polled until they carry `tag`):
// lane L holds experts i * 32 + L, i < M; lane j < K ends with the j-th
// choice's sort key.  With `full_den` (softmax scores without normalisation
// over the chosen) every lane also gets sum_e exp(z_e - z_max) over all
// experts: the experts left after the top-k, then the chosen ones, each lane's
// terms in index order, summed across the warp by a butterfly.
template <int M, bool SORTED>
__device__ __forceinline__ bool route_token(const DevLayer &d, const unsigned long long *lt, int t, int E, int K,
                                            unsigned tag, int lane, int *err, unsigned long long &sel, int &passes,
                                            bool full_den, float &den) {
    unsigned long long v[M];
    bool ok = true;
    unsigned pend = 0u;
#pragma unroll
    for (int i = 0; i < M; ++i)
        if (i * 32 + lane < E) pend |= 1u << i;
    // every pass re-reads all pending words at once: one round trip each
    const unsigned long long t0 = gtimer();
    while (__any_sync(0xffffffffu, pend != 0u)) {
        ++passes;
#pragma unroll
        for (int i = 0; i < M; ++i)
            if ((pend >> i) & 1u) v[i] = ld_tagged(lt + (size_t)t * E + i * 32 + lane);
#pragma unroll
        for (int i = 0; i < M; ++i)
            if (((pend >> i) & 1u) && tag_is(v[i], tag)) pend &= ~(1u << i);
        if (pend && gtimer() - t0 > kWaitNs) {
            atomicExch(err, 1);
            ok = false;
            pend = 0u;
        }
    }
    MOE_TRACE_CLOCK_AT(4, 0, 0);
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const int e = i * 32 + lane;
        v[i] = e < E ? ((unsigned long long)logit_key(__uint_as_float((unsigned)v[i])) << 32) | (unsigned)~e : 0ull;
    }
    MOE_TRACE_CLOCK_AT(4, 1, 0);
    // the sorted top-k: for one or two tokens on a copy, so that v keeps the
    // index order (a lane's chosen keys are larger than every key it has
    // left, rest[0]); for more tokens in place (v ends with the keys not
    // chosen, largest first)
    unsigned long long rest[M];
    if constexpr (SORTED) {
#pragma unroll
        for (int i = 0; i < M; ++i) rest[i] = v[i];
        sel = warp_topk_sorted<M>(rest, K, lane);
    } else {
        sel = warp_topk_sorted<M>(v, K, lane);
    }
    den = 1.f;
    if (full_den) {
        const float zmax = key_logit(__shfl_sync(0xffffffffu, (unsigned)(sel >> 32), 0));
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < M; ++i) {
            bool left = v[i] != 0ull;
            if constexpr (SORTED) left = left && v[i] <= rest[0];
            if (left) acc += expf(key_logit((unsigned)(v[i] >> 32)) - zmax);
        }
        if (lane < K) acc += expf(key_logit((unsigned)(sel >> 32)) - zmax);
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
        den = acc;
    }
    return ok;
}

// Per-warp copy list: the warp's items (gate/up units of pass 0, of pass 1,
// then down pieces) as (first byte, chunk count), filled by the warp's lanes
// in parallel; lane 0 walks it, cutting items into segments of <= CH chunks.

// TT: 1, 2 or 8, the token count the code is specialised for (T == TT for 1
// and 2, 3 <= T <= 8 for 8) -- a step that runs once per call runs from a
// cold instruction cache, so the loops over tokens are only as long as T
// needs.
// F8: the layer has experts in F8 chunks (the instance without it carries
// no F8 code).
template <int TT, bool F8>
__global__ void __launch_bounds__(kFT, 1) fused_kernel(DevLayer d, FusedArgs a, FusedGeom fg) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t s_bar[kFW][kRWmax];
    __shared__ __align__(8) uint64_t s_rbar;   // router rows
    __shared__ const uint8_t *s_tab_src[kFW][kTabMax];
    __shared__ int s_tab_n[kFW][kTabMax];
    __shared__ float s_tmax[kFW][kTF];
    __shared__ int s_xexp[kTF];
    __shared__ unsigned s_tag;
    __shared__ int s_ids[kTF][kMaxTopK];
    __shared__ float s_w[kTF][kMaxTopK];
    __shared__ __align__(4) unsigned char s_tokmask[kMaxExperts];
    __shared__ short s_eslot[kMaxExperts];
    __shared__ int s_slot_e[kSlotsF];
    __shared__ int s_slot_mask[kSlotsF];
    __shared__ int s_slot_p0[kSlotsF];
    __shared__ float s_pw[kPairsF];
    __shared__ signed char s_hx[kPairsF][8];                 // h prescale exponents by pair and K part
    __shared__ __align__(16) int s_wsum[2][kFW];
    __shared__ int s_nslots;
    __shared__ float s_lpart[kFW][kTF * kREmax];
    __shared__ __align__(16) float s_red[kFW][4][32];

    const int T = a.T, H = d.H, E = d.E, K = d.k, S = d.S;
    const int G = gridDim.x, c = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int RW = fg.RW, CH = fg.CH, kRE = fg.kRE;
    uint8_t *xs = smem;
    const float *s_router = reinterpret_cast<const float *>(smem + fg.router_off);
    const uint8_t *xraw = smem + fg.xraw_off;
    const float4 *s_gsp = reinterpret_cast<const float4 *>(smem + fg.gs_off);  // copy of d.gsp
    uint8_t *ring = smem + fg.ring_off + (size_t)warp * RW * CH * kChunkBytes;
    uint64_t *bar = s_bar[warp];
    const int NTs = d.Is / 8, NT13 = d.I / 8, NRT = H / 16;
    const uint64_t pol = evict_first_policy();

    // ---- the copy issuer (lane 0's registers; the other lanes' copies idle) ----
    int n_iss = 0, it = 0, n_known = 0, left = 0, sl_p = 0;
#ifdef MOE_TRACE
    bool trc = false;
#else
    constexpr bool trc = false;
#endif
    const uint8_t *src = nullptr;
    // No proxy fence before a refill: every shared-memory read of a slot
    // being refilled has returned its data before the __syncwarp that
    // precedes the call (the values fed MMAs issued before it), so the bulk
    // copy's write cannot overtake a read -- the write-after-read order that
    // mbarrier-synchronised bulk-copy pipelines rely on as well.
    auto pump = [&](int limit) {
        if (lane != 0) return;
        if (trc) MOE_TRACE_CLOCK(4, 7);
        while (n_iss < limit) {
            if (left == 0) {
                if (it >= n_known) break;
                src = s_tab_src[warp][it];
                left = s_tab_n[warp][it];
                ++it;
            }
            const int n = min(CH, left);
            mbar_expect_tx(bar + sl_p, (unsigned)(n * kChunkBytes));
            bulk_g2s(ring + (size_t)sl_p * CH * kChunkBytes, src, (unsigned)(n * kChunkBytes), bar + sl_p, pol);
            src += (size_t)n * kChunkBytes;
            left -= n;
            sl_p = sl_p + 1 == RW ? 0 : sl_p + 1;
            ++n_iss;
        }
    };
    // gate/up plan of one pass: groups of 2^lks warps share a unit (slot lo +
    // uu / NT, tile uu % NT) by splitting its K range; the warp with index vw
    // among the pass's nw warps takes units uu = u0 + i * stride, i < my, and
    // the K range [cb0, cb0 + cpw).  With more units than groups, unit uu
    // goes to group uu / G of block uu % G (modulo the stride), so every
    // block gets the floor or the ceiling of units / G (the decode rate of
    // an SM is shared by its warps); with fewer, a block's groups take
    // consecutive units (measured slightly faster at one token).
    // nc: the pass's chunks per gate/up tile (H/64 NVFP4 chunks or H/32 F8
    // chunks), f8: its experts' format
    struct Pass {
        int lks, cpw, cb0, stride, u0, my, NT, lo, nc;
        bool f8;
    };
    auto plan = [&](int units, int lks, int NT, int lo, int nw, int vw, bool f8) {
        Pass p;
        const int ngrp = nw >> lks;
        p.f8 = f8;
        p.nc = chunks_of(H, f8);
        p.lks = lks;
        p.cpw = p.nc >> lks;
        p.cb0 = (vw & ((1 << lks) - 1)) * p.cpw;
        p.stride = G * ngrp;
        p.u0 = units > p.stride ? (vw >> lks) * G + c : c * ngrp + (vw >> lks);
        p.my = vw < nw && p.u0 < units ? (units - p.u0 + p.stride - 1) / p.stride : 0;
        p.NT = NT;
        p.lo = lo;
        return p;
    };
    // lanes fill table entries [base, base + p.my) with the units of pass p
    auto fill_units = [&](const Pass &p, int base) {
        for (int i = lane; i < p.my; i += 32) {
            const int uu = p.u0 + i * p.stride;
            const int s = uu / p.NT, r = uu - s * p.NT;
            const int e = s_slot_e[p.lo + s];
            const uint8_t *b = e < 0 ? d.sw13r + (size_t)(-e - 1) * d.s13_stride : d.w13r + (size_t)e * d.e13_stride;
            s_tab_src[warp][base + i] = b + ((size_t)r * p.nc + p.cb0) * kChunkBytes;
            s_tab_n[warp][base + i] = p.cpw;
        }
    };

    FUSED_TRACE(0);
    MOE_TRACE_CLOCK(1, 0);
    // ---------------- A: static data before the dependency wait ----------------
    if (threadIdx.x < S) {
        const int si = threadIdx.x;
        s_slot_e[si] = -(si + 1);
        s_slot_mask[si] = (1 << T) - 1;
        s_slot_p0[si] = si * T;
    }
    if (threadIdx.x < S * T) s_pw[threadIdx.x] = 1.0f;
    if (threadIdx.x < E) s_tokmask[threadIdx.x] = 0;
    if (threadIdx.x == 0) {
        mbar_init(&s_rbar, 1);
    }
    if (lane == 0) {
        for (int i = 0; i < RW; ++i) mbar_init(bar + i, 1);
        fence_proxy_async();
    }
    const int v0 = pass0_index<TT>(warp), tok = routed_token_of<TT>(warp);
    const Pass p0 = plan(S * NTs, fg.lks0, NTs, 0, kPW, v0, F8 && d.f8s);
    __syncthreads();
    fill_units(p0, 0);
    __syncwarp();
    n_known = p0.my;
    if (threadIdx.x == 0) {
        // static data: this block's router rows; the packed global scales
        // and router biases of all experts
        const int nre = min(kRE, (E - c + G - 1) / G);
        mbar_expect_tx(&s_rbar, (unsigned)(nre * H * 4 + (E + S) * 16));
        bulk_g2s(smem + fg.gs_off, d.gsp, (unsigned)((E + S) * 16), &s_rbar, pol);
#pragma unroll 1
        for (int re = 0; re < nre; ++re)
            bulk_g2s(smem + fg.router_off + (size_t)re * H * 4, d.router_w + (size_t)(c + re * G) * H,
                     (unsigned)(H * 4), &s_rbar, pol);
    } else if (threadIdx.x >= 32 && threadIdx.x < 32 + S && c < NRT) {
        const int si = threadIdx.x - 32, ncs = chunks_of(d.Is, F8 && d.f8s);
        prefetch_l2(d.sw2r + (size_t)si * d.s2_stride + (size_t)c * ncs * kChunkBytes, (unsigned)(ncs * kChunkBytes));
    }
    pump(RW);
    pdl_wait();
    pdl_trigger();
    FUSED_TRACE(1);

    // ---------------- B: x, logits ----------------
    bool ok = true;
    const int nq = H / 4;                    // 4-element quads of an activation row
    if (threadIdx.x == 0) s_tag = __ldcg(d.calls + c) + 1u;
    // x: each thread copies the quads it reads in the pass below (quads
    // threadIdx.x + i * kFT of every token) with 8-byte asynchronous copies,
    // so that only its own copies stand between it and its first use (a
    // single bulk copy of all rows took longer to land)
    if (TT <= 2 && a.x_sys) {
        // x in pinned host memory, through its device alias: plain loads
        // (taken for one or two tokens only; the instance for more carries
        // none of this code)
#pragma unroll 1
        for (int P = threadIdx.x; P < nq; P += kFT) {
            uint2 v[TT];
#pragma unroll
            for (int t = 0; t < TT; ++t)
                if (t < T) v[t] = *reinterpret_cast<const uint2 *>(a.x + (size_t)t * H + 4 * P);
#pragma unroll
            for (int t = 0; t < TT; ++t)
                if (t < T) *reinterpret_cast<uint2 *>(smem + fg.xraw_off + ((size_t)t * H + 4 * P) * 2) = v[t];
        }
    } else {
#pragma unroll 1
        for (int P = threadIdx.x; P < nq; P += kFT)
#pragma unroll
            for (int t = 0; t < TT; ++t)
                if (t < T) cp_async8(smem + fg.xraw_off + ((size_t)t * H + 4 * P) * 2, a.x + (size_t)t * H + 4 * P);
        asm volatile("cp.async.wait_all;\n" ::: "memory");
    }
    if (!mbar_wait(&s_rbar, 0u, d.err)) ok = false;
    MOE_TRACE_CLOCK(2, 12);
    // One pass over x for all tokens: this thread's max |x| per token and its
    // partial FP32 logits (token t, expert c + re * G) from the exact FP32
    // values of x; each router quad is read once for all tokens.
    {
        float mx[TT], acc[TT * kREmax];
#pragma unroll
        for (int t = 0; t < TT; ++t) mx[t] = 0.f;
#pragma unroll
        for (int i = 0; i < TT * kREmax; ++i) acc[i] = 0.f;
#pragma unroll 1
        for (int P = threadIdx.x; P < nq; P += kFT) {
            float4 w4[kREmax];
#pragma unroll
            for (int re = 0; re < kREmax; ++re)
                if (re < kRE) w4[re] = *reinterpret_cast<const float4 *>(s_router + (size_t)re * H + 4 * P);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                if (t < T) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(xraw + ((size_t)t * H + 4 * P) * 2);
                    const float x0 = __uint_as_float(v.x << 16), x1 = __uint_as_float(v.x & 0xFFFF0000u);
                    const float x2 = __uint_as_float(v.y << 16), x3 = __uint_as_float(v.y & 0xFFFF0000u);
                    mx[t] = fmaxf(mx[t], fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))));
#pragma unroll
                    for (int re = 0; re < kREmax; ++re)
                        if (re < kRE)
                            acc[t * kREmax + re] = fmaf(x3, w4[re].w, fmaf(x2, w4[re].z, fmaf(x1, w4[re].y,
                                                        fmaf(x0, w4[re].x, acc[t * kREmax + re]))));
                }
            }
        }
        MOE_TRACE_CLOCK(4, 9);
        // warp maxima per token (mx >= 0 and not NaN -- fmaxf drops NaN --
        // so its bits order as unsigned)
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            if (t < T) {
                const float m = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx[t])));
                if (lane == 0) s_tmax[warp][t] = m;
            }
        }
        MOE_TRACE_CLOCK(4, 10);
        if constexpr (TT <= 2) {
            // few values: a butterfly sum of each (the same pairing order)
#pragma unroll
            for (int i = 0; i < TT * kREmax; ++i) {
                if (i < T * kREmax) {
                    float v = acc[i];
#pragma unroll
                    for (int w = 16; w >= 1; w >>= 1) v += __shfl_xor_sync(0xffffffffu, v, w);
                    if (lane == 0) s_lpart[warp][i] = v;
                }
            }
        } else {
            // warp sums of the 32 partial logits by a transposing butterfly:
            // at the step of distance w every lane keeps the half of its
            // values selected by bit w of its lane index and adds the
            // partner's copy of that half; lane L ends with value L (token L /
            // kREmax, expert L % kREmax)
#pragma unroll
            for (int w = 16; w >= 1; w >>= 1) {
#pragma unroll
                for (int i = 0; i < w; ++i) {
                    const bool up = (lane & w) != 0;
                    const float send = up ? acc[i] : acc[i + w];
                    const float keep = up ? acc[i + w] : acc[i];
                    acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
                }
            }
            s_lpart[warp][lane] = acc[0];
        }
    }
    MOE_TRACE_CLOCK(2, 13);
    __syncthreads();
    MOE_TRACE_CLOCK(2, 9);
    if constexpr (TT <= 2) {
        // Across the warps, two warps side by side: warp 0 the tokens'
        // maxima, warp 1 the logits.  Lane l takes value l % NV (NV values, a
        // power of two) over warps l / NV, l / NV + 32 / NV, ... in ascending
        // order, then the lanes of one value combine by a butterfly: a fixed
        // order, shorter than one thread walking all sixteen warps (measured
        // faster for one token; no better for eight, which keep the walk).
        if (warp == 0) {
            constexpr int NV = TT;
            const int t = lane % NV;
            float m = 0.f;
#pragma unroll
            for (int w = lane / NV; w < kFW; w += 32 / NV) m = fmaxf(m, s_tmax[w][t]);
#pragma unroll
            for (int o = NV; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane < T) s_xexp[lane] = max(-100, exp_for_f16(m));
        } else if (warp == 1) {
            // logits plus the router bias: value i = (token i / kREmax,
            // expert c + (i % kREmax) G)
            constexpr int NV = TT * kREmax;
            const int i = lane % NV;
            float v = 0.f;
#pragma unroll
            for (int w = lane / NV; w < kFW; w += 32 / NV) v += s_lpart[w][i];
#pragma unroll
            for (int o = NV; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            const int t = lane / kREmax, re = lane % kREmax, e = c + re * G;
            if (lane < NV && re < kRE && e < E && t < T)
                st_tagged(d.logit_tag + (size_t)t * E + e, s_tag, __float_as_uint(v + s_gsp[e].w));
        }
    } else {
        if (threadIdx.x < T) {
            float m = 0.f;
#pragma unroll
            for (int w = 0; w < kFW; ++w) m = fmaxf(m, s_tmax[w][threadIdx.x]);
            s_xexp[threadIdx.x] = max(-100, exp_for_f16(m));
        }
        if (threadIdx.x < TT * kREmax) {
            // logits: the warps' sums in a fixed order, plus the router bias
            const int t = threadIdx.x / kREmax, re = threadIdx.x % kREmax, e = c + re * G;
            if (re < kRE && e < E && t < T) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kFW; ++w) v += s_lpart[w][threadIdx.x];
                st_tagged(d.logit_tag + (size_t)t * E + e, s_tag, __float_as_uint(v + s_gsp[e].w));
            }
        }
    }
    MOE_TRACE_CLOCK(4, 12);
    // zero row T (the B column of absent tokens)
    for (int i = threadIdx.x; i < fg.xrow / 16; i += kFT)
        reinterpret_cast<uint4 *>(xs + (size_t)T * fg.xrow)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    FUSED_TRACE(2);
    // x' = x * 2^-xexp as f16, permuted within each 64-element chunk (element
    // 16kb + 8h + 2q + e sits at half 16q + 4kb + 2h + e: quad m of a chunk,
    // elements 4m..4m+3, has kb = m/4, h = (m/2)%2 and q = 2(m%2) for its
    // first pair, q + 1 for its second).  Staged by the warps of the
    // shared-expert pass alone; the routing warps start polling at once (the
    // block barrier at the start of pass 1 orders the staging before their
    // own use of x).
    if (v0 < kPW) {
#pragma unroll 1
        for (int P = 32 * v0 + lane; P < nq; P += 32 * kPW) {
            const int m = P & 15, kb = m >> 2, hh = (m >> 1) & 1, q0 = 2 * (m & 1);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                if (t < T) {
                    const float sc = pow2f(-s_xexp[t]);
                    const uint2 v = *reinterpret_cast<const uint2 *>(xraw + ((size_t)t * H + 4 * P) * 2);
                    const float x0 = __uint_as_float(v.x << 16), x1 = __uint_as_float(v.x & 0xFFFF0000u);
                    const float x2 = __uint_as_float(v.y << 16), x3 = __uint_as_float(v.y & 0xFFFF0000u);
                    uint8_t *row = xs + (size_t)t * fg.xrow + (P >> 4) * 128;
                    *reinterpret_cast<uint32_t *>(row + 32 * q0 + 8 * kb + 4 * hh) = pack_f16x2(x0 * sc, x1 * sc);
                    *reinterpret_cast<uint32_t *>(row + 32 * (q0 + 1) + 8 * kb + 4 * hh) = pack_f16x2(x2 * sc, x3 * sc);
                }
            }
        }
        asm volatile("bar.sync %0, %1;\n" ::"n"(kStageBar), "n"(32 * kPW) : "memory");
        MOE_TRACE_CLOCK_AT(3, 3, 64);
    }

    // ---------------- C: gate/up, pass 0 shared experts, pass 1 routed ----------------
    const uint8_t *xb = xs + (size_t)(g < T ? g : T) * fg.xrow + q * 32;
    int n_con = 0, sl_c = 0;             // segments consumed by this warp; its ring slot
    unsigned par_c = 0u;                 // and the slot's phase parity
    int n_done = 0;                      // segments whose copies have landed (waited for)
    int nslots = S, lksd = 0, perw = 0, nrt = 0, n_list = 0;
    const int nrt0 = c < NRT ? (NRT - c + G - 1) / G : 0;   // this block's output tiles
    // One ring segment of n chunks against the B rows at bp: wait for it,
    // decode and multiply, release the slot and keep the ring full.
    // The segment holds chunks c0 .. c0 + n - 1 of its tile's K range; their
    // B fragments are at bbase + b_offset(c) (F8 chunks: half a 64-element
    // group each, scaled in FP32 after their two MMAs).
    auto segment = [&](int n, const uint8_t *bbase, int c0, bool f8, bool bon, float (&a0)[4], float (&a1)[4]) {
        if (ok) {
            if (mbar_wait(bar + sl_c, par_c, d.err)) n_done = n_con + 1;
            else ok = false;
        }
        if (ok) {
            const uint8_t *ch = ring + (size_t)sl_c * CH * kChunkBytes;
            if (F8 && f8) {
#pragma unroll 2
                for (int i = 0; i < n; ++i) {
                    const uint8_t *ci = ch + (size_t)i * kChunkBytes;
                    const uint4 cw = lds128(ci + 16 * lane);
                    uint2 sw;
                    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n"
                                 : "=r"(sw.x), "=r"(sw.y) : "r"(smem_u32(ci + kCodeBytes + 8 * (lane >> 2))));
                    const uint4 b = bon ? lds128(bbase + b_offset(c0 + i, true)) : make_uint4(0u, 0u, 0u, 0u);
                    chunk_mma_f8(cw, sw, b, (i & 1) ? a1 : a0);
                }
            } else {
#pragma unroll 2
                for (int i = 0; i < n; ++i)
                    chunk_mma_smem(ch + (size_t)i * kChunkBytes, lane, bbase + (c0 + i) * 128, bon, a0, a1);
            }
        }
        __syncwarp();
        ++n_con;
        if (++sl_c == RW) {
            sl_c = 0;
            par_c ^= 1u;
        }
        if (ok) pump(n_con + RW);
    };
    // gate/up units of a pass plan: vw is this warp's index among the pass's
    // warps, tp the pass (0 shared experts, 1 routed), rb + vw the warp's
    // row of the reduction scratch (the physical warp where the two passes
    // may overlap)
    auto run_units = [&](const Pass &pp, int vw, int tp, int rb) {
        const int ks = 1 << pp.lks, gi = vw >> pp.lks, kw = vw & (ks - 1);
        // every warp of a group has the same unit count, so the group's named
        // barrier is reached by all of its warps together: id kGroupBar1 + gi
        // in the routed pass (at most 8 groups), kGroupBar0 + gi in the
        // shared-expert pass (at most 4), which the routed pass may overlap
        const int gb = (tp == 0 ? kGroupBar0 : kGroupBar1) + gi;
#pragma unroll 1
        for (int ui = 0; ui < pp.my; ++ui) {
            float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
            int c0 = pp.cb0;
            int lft = pp.cpw;
#pragma unroll 1
            while (lft > 0) {
                const int n = min(CH, lft);
                if (ui == 0 && lft == pp.cpw) MOE_TRACE_CLOCK_AT(2, 4 * tp, tp == 0 ? 64 : 0);
                segment(n, xb, c0, pp.f8, true, a0, a1);
                c0 += n;
                lft -= n;
            }
            if (ui == 0) MOE_TRACE_CLOCK_AT(2, 4 * tp + 1, tp == 0 ? 64 : 0);
#pragma unroll
            for (int v = 0; v < 4; ++v) a0[v] += a1[v];
            const int uu = pp.u0 + ui * pp.stride;
            const int s = uu / pp.NT, r = uu - s * pp.NT, slot = pp.lo + s;
            if (ks > 1) {
#pragma unroll
                for (int v = 0; v < 4; ++v) s_red[rb + vw][v][lane] = a0[v];
                asm volatile("bar.sync %0, %1;\n" ::"r"(gb), "r"(32 * ks) : "memory");
                if (kw == 0) {
#pragma unroll 1
                    for (int w = 1; w < ks; ++w)
#pragma unroll
                        for (int v = 0; v < 4; ++v) a0[v] += s_red[rb + vw + w][v][lane];
                }
                asm volatile("bar.sync %0, %1;\n" ::"r"(gb), "r"(32 * ks) : "memory");
            }
            if (ui == 0) MOE_TRACE_CLOCK_AT(2, 4 * tp + 2, tp == 0 ? 64 : 0);
            if (kw == 0 && __all_sync(0xffffffffu, ok)) {
                // SwiGLU: tile rows 0..7 gate, 8..15 up of intermediate row
                // 8r+g; lanes g and g+1 publish one tagged word of two BF16
                const int e = s_slot_e[slot], msk = s_slot_mask[slot], p0s = s_slot_p0[slot];
                const float4 gsv = s_gsp[e < 0 ? E - e - 1 : e];
                const float gsa = gsv.x, gsb = gsv.y;
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int t = 2 * q + e2;
                    const bool on = t < T && ((msk >> t) & 1);
                    const int p = p0s + __popc(msk & ((1 << t) - 1));
                    unsigned hbits = 0u;
                    if (on) {
                        const float un = pow2f(s_xexp[t]);
                        const float gt = a0[e2] * gsa * un, upv = a0[2 + e2] * gsb * un;
                        hbits = __bfloat16_as_ushort(__float2bfloat16_rn(silu_fast(gt) * upv));
                    }
                    const unsigned hnext = __shfl_down_sync(0xffffffffu, hbits, 4);
                    if (on && !(g & 1))
                        st_tagged(d.h_tag + ((size_t)p * d.Imax + 8 * r + g) / 2, s_tag, hbits | (hnext << 16));
                }
            }
            MOE_TRACE_CLOCK_AT(2, 4 * tp + 3, tp == 0 ? 64 : 0);
        }
    };
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        Pass pp = p0;
        if (pass == 0 && tok >= 0 && tok < T) {
            // routing, identical in every block, straight from the tagged
            // logits: one warp per token t (routed_token_of), lane L the
            // experts i * 32 + L.  An expert's sort key is
            // logit_key(logit) << 32 | ~id: larger is better, equal logits go
            // to the lower id, all keys differ.
            const int t = tok;
            const unsigned ltag = s_tag + (unsigned)d.debug_stall;
            int lpass = 0;
            unsigned long long sel = 0ull;
            const bool smax = d.score_func == 1, fden = smax && !d.normalize;
            float den = 1.f;
            switch (fg.m1p) {
                case 1: ok = route_token<1, (TT <= 2)>(d, d.logit_tag, t, E, K, ltag, lane, d.err, sel, lpass, fden, den) && ok; break;
                case 2: ok = route_token<2, (TT <= 2)>(d, d.logit_tag, t, E, K, ltag, lane, d.err, sel, lpass, fden, den) && ok; break;
                case 4: ok = route_token<4, (TT <= 2)>(d, d.logit_tag, t, E, K, ltag, lane, d.err, sel, lpass, fden, den) && ok; break;
                default: ok = route_token<8, (TT <= 2)>(d, d.logit_tag, t, E, K, ltag, lane, d.err, sel, lpass, fden, den) && ok; break;
            }
            const unsigned sel_key = (unsigned)(sel >> 32);
            const int sel_e = (int)~(unsigned)sel;
            MOE_TRACE_CLOCK_AT(3, 10, 0);
            MOE_TRACE_VALUE_AT(1, 2, 0, lpass);
            // scores: the sigmoid of the chosen logit, or (softmax routing)
            // exp(z - z_max) over the full-softmax denominator (1 when the
            // weights are normalised over the chosen, where it cancels).
            // Weights are normalised in selection order; for one token the
            // slots follow directly: routed slot S + (rank of the id among
            // the k choices), one pair each
            float sel_s;
            if (smax) {
                const float zs = key_logit(sel_key);
                sel_s = expf(zs - __shfl_sync(0xffffffffu, zs, 0)) / den;
            } else {
                sel_s = key_score(sel_key);
            }
            float sv[kMaxTopK];
            int ev[kMaxTopK];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                sv[j] = __shfl_sync(0xffffffffu, sel_s, j);
                ev[j] = __shfl_sync(0xffffffffu, sel_e, j);
            }
            float sum = 0.f;                 // in selection order
            int rank = 0;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                if (j < K) {
                    sum += sv[j];
                    rank += ev[j] < sel_e;
                }
            }
            if (lane < K) {
                const float w = (d.normalize ? sel_s / sum : sel_s) * d.routed_scale;
                s_ids[t][lane] = sel_e;
                s_w[t][lane] = w;
                if (c == 0) {
                    if (a.ids_out) a.ids_out[t * K + lane] = sel_e;
                    if (a.w_out) a.w_out[t * K + lane] = w;
                }
                if constexpr (TT == 1) {
                    s_slot_e[S + rank] = sel_e;
                    s_slot_mask[S + rank] = 1;
                    s_slot_p0[S + rank] = S + rank;
                    s_pw[S + rank] = w;
                } else {
                    atomicOr(reinterpret_cast<unsigned *>(s_tokmask) + (sel_e >> 2), 1u << (8 * (sel_e & 3) + t));
                }
            }
            if (TT == 1 && lane == 0) s_nslots = S + K;
            MOE_TRACE_CLOCK_AT(3, 5, 0);
        }
        if (pass == 1) {
            FUSED_TRACE(4);
            if (!__syncthreads_and(ok)) {
                ok = false;
                break;
            }
            FUSED_TRACE(11);
            if constexpr (TT > 1) {
                // slots: shared first, then routed experts in ascending id
                // (one expert per thread); an expert's pairs are contiguous,
                // tokens ascending
                const int e = threadIdx.x;
                const int msk = e < E ? s_tokmask[e] : 0;
                const int cnt = __popc(msk);
                const unsigned flags = __ballot_sync(0xffffffffu, msk != 0);
                int cinc = cnt;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, cinc, off);
                    if (lane >= off) cinc += v;
                }
                if (lane == 31) {
                    s_wsum[0][warp] = __popc(flags);
                    s_wsum[1][warp] = cinc;
                }
                __syncthreads();
                int fb = __popc(flags & ((1u << lane) - 1u)), cb = cinc - cnt;
#pragma unroll
                for (int w = 0; w < kFW; ++w)
                    if (w < warp) {
                        fb += s_wsum[0][w];
                        cb += s_wsum[1][w];
                    }
                if (msk) {
                    const int sl = S + fb;
                    s_slot_e[sl] = e;
                    s_slot_mask[sl] = msk;
                    s_slot_p0[sl] = S * T + cb;
                    s_eslot[e] = (short)sl;
                }
                if (threadIdx.x == kFT - 1) s_nslots = S + fb + (msk != 0);
                __syncthreads();
                if (threadIdx.x < T * K) {
                    const int t = threadIdx.x / K, j = threadIdx.x - (threadIdx.x / K) * K, ee = s_ids[t][j];
                    const int sl = s_eslot[ee];
                    s_pw[s_slot_p0[sl] + __popc(s_slot_mask[sl] & ((1 << t) - 1))] = s_w[t][j];
                }
            }
            FUSED_TRACE(12);
            // this warp's routed units and down pieces -> its copy list
            nslots = s_nslots;
            pp = plan((nslots - S) * NT13, fg.lks1[nslots], NT13, S, kFW, warp, F8 && d.f8e);
            MOE_TRACE_CLOCK(4, 3);
            fill_units(pp, p0.my);
            __syncwarp();
            MOE_TRACE_CLOCK(4, 4);
            // the routed units' copies start before the down pieces are listed
            n_known = p0.my + pp.my;
#ifdef MOE_TRACE
            trc = true;
#endif
            if (ok) pump(n_con + RW);
#ifdef MOE_TRACE
            trc = false;
#endif
            MOE_TRACE_CLOCK(4, 5);
            lksd = fg.lksd[nslots];
            perw = warp < (nslots << lksd) ? ((nslots << lksd) - warp + kFW - 1) / kFW : 0;
            nrt = nrt0;
            for (int i = lane; i < nrt * perw; i += 32) {
                const int ri = nrt == 1 ? 0 : i / perw, r2 = i - ri * perw;
                const int rt = c + ri * G, pi = warp + kFW * r2;
                const int e = s_slot_e[pi >> lksd], kp = pi & ((1 << lksd) - 1);
                const int ncd = chunks_of(e < 0 ? d.Is : d.I, F8 && (e < 0 ? d.f8s : d.f8e)), cpk = ncd >> lksd;
                const uint8_t *b = e < 0 ? d.sw2r + (size_t)(-e - 1) * d.s2_stride : d.w2r + (size_t)e * d.e2_stride;
                s_tab_src[warp][p0.my + pp.my + i] = b + ((size_t)rt * ncd + kp * cpk) * kChunkBytes;
                s_tab_n[warp][p0.my + pp.my + i] = cpk;
            }
            __syncwarp();
            MOE_TRACE_CLOCK(2, 14);
            n_list = p0.my + pp.my + nrt * perw;
            n_known = n_list;
            // a warp with routed units requests its down pieces as its ring
            // frees up, so that the routed gate/up weights, on which h and
            // hence every block's phase D wait, come first
            if (ok && pp.my == 0) pump(n_con + RW);
            MOE_TRACE_CLOCK(2, 15);
            __syncwarp();
            FUSED_TRACE(6);
        }
        if constexpr (TT > 2) {
            // more tokens: the shared-expert units wait for the routing (whose
            // compare-and-select work would share schedulers with their
            // decode); their segments were requested first, so they run
            // first in pass 1
            if (pass == 1) {
                run_units(p0, v0, 0, kFW - kPW);   // the pass-0 warps are kFW - kPW .. kFW - 1
                run_units(pp, warp, 1, 0);
            }
        } else {
            run_units(pp, pass == 0 ? v0 : warp, pass, 0);
        }
    }
    FUSED_TRACE(7);
    // a block without output tiles is done.  For more than two tokens every
    // warp must be done with x and its gate/up units before phase D reuses
    // the shared memory; for one or two the h rows have a region of their
    // own, and a warp that failed a wait skips its work but keeps to the
    // block's barriers.
    if constexpr (TT <= 2) {
        if (nrt == 0) {
            drain_ring(bar, RW, n_done, n_iss, lane);
            FUSED_TRACE(9);
            if (threadIdx.x == 0) d.calls[c] = s_tag;
            return;
        }
    } else {
        if (!__syncthreads_and(ok) || nrt == 0) {
            drain_ring(bar, RW, n_done, n_iss, lane);
            FUSED_TRACE(9);
            if (threadIdx.x == 0) d.calls[c] = s_tag;
            return;
        }
    }
    FUSED_TRACE(8);

    // ---------------- D: down + combine, 16 output rows per tile ----------------
    // h comes from the tagged words (polled until they carry this call's tag)
    // into shared memory in the MMA operand order, by tasks (pair p, K part
    // kp): a task's pieces are all in flight at once (one pass for parts of
    // up to 32 * kHU pieces), and its range is rescaled to f16 by an exact
    // power-of-two prescale of its own.  For one or two tokens each warp
    // gathers the tasks of its own down pieces and starts at once; for more
    // tokens (the shared expert's slot alone has T rows) the tasks are spread
    // evenly over the warps and the block waits for all of them.  The B
    // column of a token a slot does not serve is zero.
    uint8_t *hs = smem + fg.hs_off;
    const int npairs = T * (K + S);
    int hpass = 0;
    FUSED_TRACE(14);
    auto gather = [&](int p, int kp) {
        const int cpk = (p < S * T ? d.Is : d.I) / kChunkK >> lksd;
        const int npc = cpk * 16, pc0 = kp * npc;        // 16-byte pieces of the K part; the first
        const unsigned long long *src = d.h_tag + (size_t)p * (d.Imax / 2) + 2 * pc0;
        uint32_t *row = reinterpret_cast<uint32_t *>(hs + (size_t)p * fg.hrow);
        // one batch: the prescale follows from the registers and the words
        // are written once, already as f16; else raw BF16 first, rescaled
        // after the last batch
        const bool one = npc <= 32 * kHU;
        float mx = 0.f, sc = 1.f;
        int hx = 0;
        MOE_TRACE_CLOCK(4, 13);
#pragma unroll 1
        for (int P0 = 0; P0 < npc; P0 += 32 * kHU) {
            unsigned long long v[kHU][2];
            unsigned pend = 0u;          // pieces not yet carrying the tag
#pragma unroll
            for (int u = 0; u < kHU; ++u) {
                v[u][0] = v[u][1] = 0ull;
                if (P0 + lane + 32 * u < npc) pend |= 1u << u;
            }
            // every pass re-reads all pending pieces at once
            const unsigned long long t0 = gtimer();
            while (pend && ok) {
                ++hpass;
#pragma unroll
                for (int u = 0; u < kHU; ++u)
                    if ((pend >> u) & 1u) ld_tagged2(src + 2 * (P0 + lane + 32 * u), v[u][0], v[u][1]);
#pragma unroll
                for (int u = 0; u < kHU; ++u)
                    if (((pend >> u) & 1u) && tag_is(v[u][0], s_tag) && tag_is(v[u][1], s_tag)) pend &= ~(1u << u);
                if (pend && gtimer() - t0 > kWaitNs) {
                    atomicExch(d.err, 1);
                    ok = false;
                }
            }
            MOE_TRACE_CLOCK(4, 14);
            // pieces past the end hold zeros, which leave the maximum alone
#pragma unroll
            for (int u = 0; u < kHU; ++u)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const unsigned wv = (unsigned)v[u][h2];
                    mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(wv << 16)), fabsf(__uint_as_float(wv & 0xFFFF0000u))));
                }
            if (one) {
                // mx >= 0 and not NaN (fmaxf drops NaN): its bits order as unsigned
                mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx)));
                hx = max(-100, exp_for_f16(mx));
                sc = pow2f(-hx);
            }
#pragma unroll
            for (int u = 0; u < kHU; ++u) {
                if (P0 + lane + 32 * u < npc) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const unsigned wv = (unsigned)v[u][h2];
                        // word wi of the row (elements 2wi, 2wi+1) -> its
                        // place in the operand order (as for x)
                        const int wi = 2 * (pc0 + P0 + lane + 32 * u) + h2, l = wi & 31;
                        row[(wi & ~31) + 8 * (l & 3) + 2 * (l >> 3) + ((l >> 2) & 1)] =
                            one ? pack_f16x2(__uint_as_float(wv << 16) * sc, __uint_as_float(wv & 0xFFFF0000u) * sc)
                                : wv;
                    }
                }
            }
        }
        MOE_TRACE_CLOCK(4, 15);
        if (!one) {
            mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx)));
            hx = max(-100, exp_for_f16(mx));
            sc = pow2f(-hx);
            // each lane rescales the words it wrote
#pragma unroll 1
            for (int P = lane; P < npc; P += 32) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int wi = 2 * (pc0 + P) + h2, l = wi & 31;
                    uint32_t *w = row + (wi & ~31) + 8 * (l & 3) + 2 * (l >> 3) + ((l >> 2) & 1);
                    const unsigned wv = *w;
                    *w = pack_f16x2(__uint_as_float(wv << 16) * sc, __uint_as_float(wv & 0xFFFF0000u) * sc);
                }
            }
        }
        if (lane == 0) s_hx[p][kp] = (signed char)hx;
        MOE_TRACE_CLOCK(4, 11);
    };
    // two tasks polled together (one round trip for both) when each has at
    // most 32 * kHU2 pieces; else one after the other
    auto gather2 = [&](int pa, int kpa, int pb, int kpb) {
        const int pp2[2] = {pa, pb}, kk2[2] = {kpa, kpb};
        int npc2[2], pc02[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            npc2[j] = ((pp2[j] < S * T ? d.Is : d.I) / kChunkK >> lksd) * 16;
            pc02[j] = kk2[j] * npc2[j];
        }
        if (npc2[0] > 32 * kHU2 || npc2[1] > 32 * kHU2) {
            gather(pa, kpa);
            gather(pb, kpb);
            return;
        }
        unsigned long long v[2][kHU2][2];
        unsigned pend = 0u;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int u = 0; u < kHU2; ++u) {
                v[j][u][0] = v[j][u][1] = 0ull;
                if (lane + 32 * u < npc2[j]) pend |= 1u << (j * kHU2 + u);
            }
        const unsigned long long t0 = gtimer();
        while (pend && ok) {
            ++hpass;
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int u = 0; u < kHU2; ++u)
                    if ((pend >> (j * kHU2 + u)) & 1u)
                        ld_tagged2(d.h_tag + (size_t)pp2[j] * (d.Imax / 2) + 2 * (pc02[j] + lane + 32 * u), v[j][u][0],
                                   v[j][u][1]);
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int u = 0; u < kHU2; ++u)
                    if (((pend >> (j * kHU2 + u)) & 1u) && tag_is(v[j][u][0], s_tag) && tag_is(v[j][u][1], s_tag))
                        pend &= ~(1u << (j * kHU2 + u));
            if (pend && gtimer() - t0 > kWaitNs) {
                atomicExch(d.err, 1);
                ok = false;
            }
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = 0.f;
#pragma unroll
            for (int u = 0; u < kHU2; ++u)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const unsigned wv = (unsigned)v[j][u][h2];
                    mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(wv << 16)), fabsf(__uint_as_float(wv & 0xFFFF0000u))));
                }
            // mx >= 0 and not NaN (fmaxf drops NaN): its bits order as unsigned
            mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx)));
            const int hx = max(-100, exp_for_f16(mx));
            const float sc = pow2f(-hx);
            uint32_t *row = reinterpret_cast<uint32_t *>(hs + (size_t)pp2[j] * fg.hrow);
#pragma unroll
            for (int u = 0; u < kHU2; ++u) {
                if (lane + 32 * u < npc2[j]) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const unsigned wv = (unsigned)v[j][u][h2];
                        const int wi = 2 * (pc02[j] + lane + 32 * u) + h2, l = wi & 31;
                        row[(wi & ~31) + 8 * (l & 3) + 2 * (l >> 3) + ((l >> 2) & 1)] =
                            pack_f16x2(__uint_as_float(wv << 16) * sc, __uint_as_float(wv & 0xFFFF0000u) * sc);
                    }
                }
            }
            if (lane == 0) s_hx[pp2[j]][kk2[j]] = (signed char)hx;
        }
    };
    if constexpr (TT <= 2) {
#pragma unroll 1
        for (int r2 = 0; r2 < perw; ++r2) {
            const int pi = warp + kFW * r2, slot = pi >> lksd;
            const int ntok = __popc(s_slot_mask[slot]), p0s = s_slot_p0[slot];
#pragma unroll 1
            for (int k = 0; k < ntok; ++k) gather(p0s + k, pi & ((1 << lksd) - 1));
        }
        __syncwarp();
    } else {
#pragma unroll 1
        for (int tk = warp; tk < (npairs << lksd); tk += 2 * kFW) {
            const int tb = tk + kFW;
            if (tb < (npairs << lksd))
                gather2(tk >> lksd, tk & ((1 << lksd) - 1), tb >> lksd, tb & ((1 << lksd) - 1));
            else
                gather(tk >> lksd, tk & ((1 << lksd) - 1));
        }
        if (!__syncthreads_and(ok)) {
            drain_ring(bar, RW, n_done, n_iss, lane);
            FUSED_TRACE(9);
            if (threadIdx.x == 0) d.calls[c] = s_tag;
            return;
        }
    }
    MOE_TRACE_VALUE(1, 3, hpass);
#pragma unroll 1
    for (int ri = 0; ri < nrt; ++ri) {
        const int rt = c + ri * G;
        float oa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int r2 = 0; r2 < perw; ++r2) {
            const int pi = warp + kFW * r2;
            const int slot = pi >> lksd, kp = pi & ((1 << lksd) - 1);
            const int e = s_slot_e[slot];
            const int msk = s_slot_mask[slot], p0s = s_slot_p0[slot];
            const float gs = s_gsp[e < 0 ? E - e - 1 : e].z;
            const bool f8 = F8 && (e < 0 ? d.f8s : d.f8e);
            const int cpk = chunks_of(e < 0 ? d.Is : d.I, f8) >> lksd;
            const bool bon = (msk >> g) & 1;
            const uint8_t *bb = hs + (size_t)(bon ? p0s + __popc(msk & ((1 << g) - 1)) : 0) * fg.hrow + q * 32;
            float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
            int c0 = kp * cpk;
            int lft = cpk;
#pragma unroll 1
            while (lft > 0) {
                const int n = min(CH, lft);
                if (ri == 0 && r2 == 0 && lft == cpk) MOE_TRACE_CLOCK(2, 10);
                segment(n, bb, c0, f8, bon, a0, a1);
                c0 += n;
                lft -= n;
            }
            if (ri == 0) MOE_TRACE_CLOCK(2, 11);
            // y = gs * 2^hexp * acc, weighted into the per-token accumulator
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int t = 2 * q + e2;
                if (t < T && ((msk >> t) & 1)) {
                    const int k = __popc(msk & ((1 << t) - 1));
                    const float wgt = s_pw[p0s + k] * gs * pow2f(s_hx[p0s + k][kp]);
                    oa[e2] = fmaf(wgt, a0[e2] + a1[e2], oa[e2]);
                    oa[2 + e2] = fmaf(wgt, a0[2 + e2] + a1[2 + e2], oa[2 + e2]);
                }
            }
        }
        // fixed-order reduction over warps, BF16 out
#pragma unroll
        for (int v = 0; v < 4; ++v) s_red[warp][v][lane] = oa[v];
        __syncthreads();
        FUSED_TRACE(15);
        if (warp == 0) {
            float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w = 0; w < kFW; ++w)
#pragma unroll
                for (int v = 0; v < 4; ++v) o[v] += s_red[w][v][lane];
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int t = 2 * q + e2;
                if (t < T) {
                    a.out[(size_t)t * H + 16 * rt + g] = __float2bfloat16_rn(o[e2]);
                    a.out[(size_t)t * H + 16 * rt + g + 8] = __float2bfloat16_rn(o[2 + e2]);
                }
            }
        }
        __syncthreads();
    }
    if (!ok) drain_ring(bar, RW, n_done, n_iss, lane);
    FUSED_TRACE(9);
    MOE_TRACE_CLOCK(1, 9);
    if (threadIdx.x == 0) d.calls[c] = s_tag;
}

// coop: launch as a cooperative grid, which the driver starts only when all
// its blocks can be resident at once (the blocks' exchanges then cannot wait
// on a block that kernels of other streams keep off the GPU); the attribute is
// combined with programmatic dependent launch.
template <int TT, bool F8>
cudaError_t launch_tt(const DevLayer &d, const FusedArgs &a, const FusedGeom &fg, int G, bool coop,
                      cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kFT);
    cfg.dynamicSmemBytes = (size_t)fg.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = coop ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, fused_kernel<TT, F8>, d, a, fg);
}

// the kernel instance for T tokens: 0 (TT = 1), 1 (TT = 2), 2 (TT = 8)
int inst_of(int T) { return T == 1 ? 0 : T == 2 ? 1 : 2; }
constexpr int kInst = 3;
int g_dyn_max[kInst];                        // dynamic shared memory a block may use, by instance

template <int TT>
cudaError_t prepare_tt(int optin) {
    cudaFuncAttributes fa, fb;
    cudaError_t e = cudaFuncGetAttributes(&fa, fused_kernel<TT, false>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fb, fused_kernel<TT, true>);
    if (e != cudaSuccess) return e;
    g_dyn_max[inst_of(TT)] = optin - (int)std::max(fa.sharedSizeBytes, fb.sharedSizeBytes);
    e = cudaFuncSetAttribute(fused_kernel<TT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             g_dyn_max[inst_of(TT)]);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fused_kernel<TT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g_dyn_max[inst_of(TT)]);
    return e;
}

}  // namespace

// Largest T for which moe_decode_forward picks the single launch.
constexpr int kFusedMaxT = 8;
constexpr int kMaxFusedH = 8192;             // hidden sizes the single launch takes

bool fused_eligible(const DevLayer &d, int T, int sm_count, size_t optin_smem) {
    (void)optin_smem;
    if (T < 1 || T > kFusedMaxT) return false;
    if (d.E > kREmax * sm_count) return false;
    if (d.H > kMaxFusedH || g_dyn_max[inst_of(T)] <= 0) return false;
    if (d.k * T + d.S > kSlotsF) return false;
    FusedGeom fg;
    return fused_geometry(d, T, sm_count, g_dyn_max[inst_of(T)], fg);
}

cudaError_t launch_fused(const DevLayer &d, const __nv_bfloat16 *x, int T, __nv_bfloat16 *out, int *ids,
                         float *w, int sm_count, bool coop, cudaStream_t s, bool x_sys) {
    FusedGeom fg;
    if (T < 1 || T > kFusedMaxT || d.H > kMaxFusedH || !fused_geometry(d, T, sm_count, g_dyn_max[inst_of(T)], fg))
        return cudaErrorInvalidValue;
    FusedArgs a{x, T, out, ids, w, x_sys ? 1 : 0};
    const bool f8 = d.f8e || d.f8s;
    switch (inst_of(T)) {
        case 0: return f8 ? launch_tt<1, true>(d, a, fg, sm_count, coop, s) : launch_tt<1, false>(d, a, fg, sm_count, coop, s);
        case 1: return f8 ? launch_tt<2, true>(d, a, fg, sm_count, coop, s) : launch_tt<2, false>(d, a, fg, sm_count, coop, s);
        default: return f8 ? launch_tt<8, true>(d, a, fg, sm_count, coop, s) : launch_tt<8, false>(d, a, fg, sm_count, coop, s);
    }
}

cudaError_t prepare_fused_kernel(int optin_bytes) {
    cudaError_t e = prepare_tt<1>(optin_bytes);
    if (e == cudaSuccess) e = prepare_tt<2>(optin_bytes);
    if (e == cudaSuccess) e = prepare_tt<8>(optin_bytes);
    return e;
}

int fused_blocks_per_sm(const DevLayer &d, int T) {
    int sms = 0, dev = 0;
    if (T < 1 || T > kFusedMaxT || d.H > kMaxFusedH || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    FusedGeom fg;
    if (!fused_geometry(d, T, sms, g_dyn_max[inst_of(T)], fg)) return 0;
    int n = 0;
    cudaError_t e;
    const bool f8 = d.f8e || d.f8s;
    switch (inst_of(T)) {
        case 0: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f8 ? fused_kernel<1, true> : fused_kernel<1, false>, kFT, fg.total); break;
        case 1: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f8 ? fused_kernel<2, true> : fused_kernel<2, false>, kFT, fg.total); break;
        default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f8 ? fused_kernel<8, true> : fused_kernel<8, false>, kFT, fg.total); break;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace moe
