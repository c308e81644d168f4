// abi.cu -- the C ABI declared in include/moe_nvfp4.h: validation
// (default-deny), the load-time repack, workspace management and the launch
// sequence of one decode step.
//
// Default-deny start-up follows "Day 0 support for Mistral Large 4 on vLLM",
// "Fail-stop": a configuration the kernels do not cover fails at start-up and
// the error lists every reason, rather than running something unsupported.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "moe_internal.cuh"

using namespace moe;

struct moe_layer {
    moe_config cfg;
    int device;
    int sm_count;
    DevLayer d;
    void *wmem;
    size_t wbytes;
    void *wsmem;
    size_t wsbytes;
    __nv_bfloat16 *x_stage;
    __nv_bfloat16 *out_stage;
    int *ids_stage;
    float *w_stage;
    std::vector<float> gs13_h, gs2_h, sgs13_h, sgs2_h;
    size_t expert_bytes, shared_bytes;
    float *router_b_slot;
    int optin_smem;
    int fused_ok[kMaxTokens + 1];   // single-launch path usable for this T
    int inject_stall = 0;           // moe_debug_inject: for the next single launch only
    unsigned long long fused_calls = 0;   // single launches since the tags were last restarted
};

namespace {

thread_local std::string g_err;

moe_status fail(moe_status st, const std::string &msg) {
    g_err = msg;
    return st;
}

moe_status cuda_fail(cudaError_t e, const char *what) {
    g_err = std::string(what) + ": " + cudaGetErrorString(e);
    cudaGetLastError();   // clear a non-sticky error so later CUDA calls do not report it
    return MOE_ERR_CUDA;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

std::string join(const std::vector<std::string> &v) {
    std::string s;
    for (size_t i = 0; i < v.size(); ++i) {
        if (i) s += "; ";
        s += v[i];
    }
    return s;
}

std::vector<std::string> unsupported_reasons(const moe_config *c) {
    std::vector<std::string> why;
    auto chk = [&](bool ok, const char *msg) {
        if (!ok) why.emplace_back(msg);
    };
    chk(c->hidden >= 64 && c->hidden <= 16384 && c->hidden % 64 == 0,
        "hidden must be a multiple of 64 in [64, 16384]");
    chk(c->inter >= 64 && c->inter <= 16384 && c->inter % 64 == 0,
        "inter must be a multiple of 64 in [64, 16384]");
    chk(c->num_shared >= 0 && c->num_shared <= kMaxShared, "num_shared must be 0, 1 or 2");
    if (c->num_shared > 0)
        chk(c->shared_inter >= 64 && c->shared_inter <= 16384 && c->shared_inter % 64 == 0,
            "shared_inter must be a multiple of 64 in [64, 16384]");
    chk(c->num_experts >= 1 && c->num_experts <= kMaxExperts, "num_experts must be in [1, 512]");
    chk(c->top_k >= 1 && c->top_k <= kMaxTopK, "top_k must be in [1, 8]");
    chk(c->top_k <= c->num_experts, "top_k must not exceed num_experts");
    chk(c->max_tokens >= 1 && c->max_tokens <= kMaxTokens, "max_tokens must be in [1, 64]");
    chk(c->normalize_topk == 0 || c->normalize_topk == 1, "normalize_topk must be 0 or 1");
    chk(std::isfinite(c->routed_scale), "routed_scale must be finite");
    chk(c->score_func == 0 || c->score_func == 1, "score_func must be 0 (sigmoid) or 1 (softmax)");
    chk(c->expert_format >= MOE_FMT_NVFP4 && c->expert_format <= MOE_FMT_MXFP8,
        "expert_format must be 0 (NVFP4), 1 (MXFP4), 2 (FP8 block) or 3 (MXFP8)");
    chk(c->shared_format >= MOE_FMT_NVFP4 && c->shared_format <= MOE_FMT_MXFP8,
        "shared_format must be 0 (NVFP4), 1 (MXFP4), 2 (FP8 block) or 3 (MXFP8)");
    chk(c->w4a4 == 0 || c->w4a4 == 1, "w4a4 must be 0 or 1");
    return why;
}

bool is_device_ptr(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

struct Carver {
    char *base;
    size_t off = 0;
    template <class T>
    T *take(size_t count) {
        off = (off + 255) & ~(size_t)255;
        T *p = reinterpret_cast<T *>(base ? base + off : nullptr);
        off += count * sizeof(T);
        return p;
    }
};

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// Lay out (or measure, when base == nullptr) the weight block.
void carve_weights(moe_layer *L, char *base) {
    const moe_config &c = L->cfg;
    DevLayer &d = L->d;
    Carver cv{base};
    const int E = c.num_experts, H = c.hidden, I = c.inter, S = c.num_shared;
    const int Is = S > 0 ? c.shared_inter : I;
    d.router_w = cv.take<float>((size_t)E * H);
    d.router_b = nullptr;
    L->router_b_slot = cv.take<float>(E);
    d.e13_stride = repacked_bytes(2 * I, H, d.f8e);
    d.e2_stride = repacked_bytes(H, I, d.f8e);
    d.s13_stride = repacked_bytes(2 * Is, H, d.f8s);
    d.s2_stride = repacked_bytes(H, Is, d.f8s);
    d.w13r = cv.take<uint8_t>((size_t)E * d.e13_stride);
    d.w2r = cv.take<uint8_t>((size_t)E * d.e2_stride);
    d.gs13 = cv.take<float>((size_t)E * 2);
    d.gs2 = cv.take<float>(E);
    d.sw13r = cv.take<uint8_t>((size_t)S * d.s13_stride);
    d.sw2r = cv.take<uint8_t>((size_t)S * d.s2_stride);
    d.sgs13 = cv.take<float>((size_t)(S > 0 ? S : 1) * 2);
    d.sgs2 = cv.take<float>(S > 0 ? S : 1);
    d.gsp = cv.take<float4>((size_t)E + S);
    L->wbytes = cv.off;
}

void carve_workspace(moe_layer *L, char *base) {
    const moe_config &c = L->cfg;
    DevLayer &d = L->d;
    Carver cv{base};
    const int Tm = c.max_tokens, E = c.num_experts, K = c.top_k, S = c.num_shared, H = c.hidden;
    d.logits = cv.take<float>((size_t)Tm * E);
    d.lpart = cv.take<float>((size_t)kMaxKSplit * Tm * E);
    d.xmaxb = cv.take<unsigned>(Tm);
    d.ids = cv.take<int>((size_t)Tm * K);
    d.wsel = cv.take<float>((size_t)Tm * K);
    d.xexp = cv.take<int>(Tm);
    d.nslots = cv.take<int>(1);
    d.slot_expert = cv.take<int>(d.max_slots);
    d.slot_m = cv.take<int>(d.max_slots);
    d.slot_p0 = cv.take<int>(d.max_slots);
    d.pair_tok = cv.take<int>(d.max_pairs);
    d.pair_w = cv.take<float>(d.max_pairs);
    d.pair_of = cv.take<int>((size_t)Tm * (K + S));
    d.hmax = cv.take<unsigned>(d.max_pairs);
    d.h_ws = cv.take<__nv_bfloat16>((size_t)d.max_pairs * d.Imax);
    d.y_ws = cv.take<float>((size_t)d.max_pairs * H);
    d.ticket = cv.take<unsigned>(1);
    d.down_cnt = cv.take<unsigned>((size_t)H / 16);
    d.err = cv.take<int>(1);
    const int Tf = std::min(Tm, 8);
    d.logit_tag = cv.take<unsigned long long>((size_t)Tf * E);
    d.h_tag = cv.take<unsigned long long>((size_t)Tf * (K + S) * (d.Imax / 2));
    d.calls = cv.take<unsigned>(L->sm_count);
    d.nhot = cv.take<int>(1);
    d.hot_slots = cv.take<int>(d.max_slots);
    d.ncold = cv.take<int>(1);
    d.cold_slots = cv.take<int>(d.max_slots);
    d.tg_ticket = cv.take<unsigned>(Tm);
    d.emask = cv.take<unsigned long long>(E);
    d.wave_ctr = cv.take<unsigned>(2);
    d.xq = cv.take<__nv_bfloat16>((size_t)Tm * H);
    d.gsx = cv.take<float>(Tm);
    d.gsh = cv.take<float>(d.max_pairs);
    const bool q4 = c.w4a4 != 0;   // the packed codes only for W4A4 layers
    d.xq4 = cv.take<uint8_t>(q4 ? (size_t)Tm * H / 2 : 0);
    d.xsf = cv.take<uint8_t>(q4 ? (size_t)Tm * H / 16 : 0);
    d.hq4 = cv.take<uint8_t>(q4 ? (size_t)d.max_pairs * d.Imax / 2 : 0);
    d.hsf = cv.take<uint8_t>(q4 ? (size_t)d.max_pairs * d.Imax / 16 : 0);
    L->x_stage = cv.take<__nv_bfloat16>((size_t)Tm * H);
    L->out_stage = cv.take<__nv_bfloat16>((size_t)Tm * H);
    L->ids_stage = cv.take<int>((size_t)Tm * K);
    L->w_stage = cv.take<float>((size_t)Tm * K);
    L->wsbytes = cv.off;
}

bool is_f8(int fmt) { return fmt == MOE_FMT_FP8_BLOCK || fmt == MOE_FMT_MXFP8; }

// Repack one expert group (n experts of intermediate size I) from the
// caller's canonical tensors in format `fmt` into the library's chunks, and
// set the group's tensor scales (device gs13 [n,2] / gs2 [n] and their host
// copies): the caller's for NVFP4; 1 for the FP8 formats (their scales live
// in the chunks); for MXFP4 the power of two by which each matrix half's
// E8M0 scales are shifted into E4M3's range, exactly (the repack then is
// NVFP4).  MXFP4 needs the E8M0 codes of one matrix half to span at most 17
// octaves (the powers of two E4M3 holds) and no NaN code; otherwise the
// reasons are appended to `why`.  Synchronises `st` for MXFP4.
cudaError_t repack_group(int fmt, int n, int H, int I, const uint8_t *w13, const uint8_t *w13_sf,
                         const float *w13_gs, const uint8_t *w2, const uint8_t *w2_sf, const float *w2_gs,
                         uint8_t *d13, uint8_t *d2, float *gs13, float *gs2, std::vector<float> &gs13_h,
                         std::vector<float> &gs2_h, const char *what, std::vector<std::string> &why,
                         cudaStream_t st) {
    gs13_h.assign((size_t)n * 2, 1.f);
    gs2_h.assign((size_t)n, 1.f);
    if (n <= 0) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (fmt == MOE_FMT_NVFP4) {
        e = cudaMemcpyAsync(gs13, w13_gs, (size_t)n * 2 * sizeof(float), cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(gs2, w2_gs, (size_t)n * sizeof(float), cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess) e = launch_repack(w13, w13_sf, n, 2 * I, H, true, d13, st);
        if (e == cudaSuccess) e = launch_repack(w2, w2_sf, n, H, I, false, d2, st);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(gs13_h.data(), w13_gs, (size_t)n * 2 * sizeof(float), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(gs2_h.data(), w2_gs, (size_t)n * sizeof(float), cudaMemcpyDeviceToHost, st);
        return e;
    }
    if (is_f8(fmt)) {
        e = cudaMemcpyAsync(gs13, gs13_h.data(), (size_t)n * 2 * sizeof(float), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(gs2, gs2_h.data(), (size_t)n * sizeof(float), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = launch_repack_f8(w13, w13_sf, fmt, n, 2 * I, H, true, d13, st);
        if (e == cudaSuccess) e = launch_repack_f8(w2, w2_sf, fmt, n, H, I, false, d2, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);   // the host ones above are read by the copies
        return e;
    }
    // MXFP4: scale ranges -> offsets -> NVFP4 scales, then the NVFP4 repack
    int *mm = nullptr, *offs = nullptr;
    uint8_t *sf13 = nullptr, *sf2 = nullptr;
    std::vector<int> mm_h((size_t)n * 2 * 3 * 2), offs_h((size_t)n * 2 * 2);
    e = cudaMalloc(&mm, mm_h.size() * sizeof(int));
    if (e == cudaSuccess) e = cudaMalloc(&offs, offs_h.size() * sizeof(int));
    if (e == cudaSuccess) e = cudaMalloc(&sf13, (size_t)n * 2 * I * (H / 16));
    if (e == cudaSuccess) e = cudaMalloc(&sf2, (size_t)n * H * (I / 16));
    if (e == cudaSuccess) e = launch_mx_scale_range(w13_sf, n, 2 * I, H, true, mm, st);
    if (e == cudaSuccess) e = launch_mx_scale_range(w2_sf, n, H, I, false, mm + (size_t)n * 2 * 3, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(mm_h.data(), mm, mm_h.size() * sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    bool bad = false;
    if (e == cudaSuccess) {
        for (int m = 0; m < 2; ++m) {        // 0 gate/up, 1 down
            for (int x = 0; x < n; ++x) {
                for (int h = 0; h < (m == 0 ? 2 : 1); ++h) {
                    const int *r = mm_h.data() + (size_t)m * n * 2 * 3 + ((size_t)x * 2 + h) * 3;
                    const char *mat = m == 0 ? (h == 0 ? "gate" : "up") : "down";
                    if (r[2]) {
                        why.push_back(std::string(what) + " expert " + std::to_string(x) + " " + mat +
                                      ": E8M0 scale code 255 (NaN)");
                        bad = true;
                    } else if (r[1] - r[0] > 17) {
                        why.push_back(std::string(what) + " expert " + std::to_string(x) + " " + mat +
                                      ": E8M0 scales span " + std::to_string(r[1] - r[0]) +
                                      " octaves (at most 17 convert exactly)");
                        bad = true;
                    }
                    // the largest scale maps to 2^8, the largest power of two of E4M3
                    const int off = r[1] - 127 - 8;
                    offs_h[(size_t)m * n * 2 + (size_t)x * 2 + h] = off;
                    const float g = ldexpf(1.f, off);
                    if (m == 0) gs13_h[(size_t)x * 2 + h] = g;
                    else gs2_h[x] = g;
                }
            }
        }
    }
    if (e == cudaSuccess && !bad) {
        e = cudaMemcpyAsync(offs, offs_h.data(), offs_h.size() * sizeof(int), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = launch_mx_to_nv_scales(w13_sf, offs, n, 2 * I, H, true, sf13, st);
        if (e == cudaSuccess) e = launch_mx_to_nv_scales(w2_sf, offs + (size_t)n * 2, n, H, I, false, sf2, st);
        if (e == cudaSuccess) e = launch_repack(w13, sf13, n, 2 * I, H, true, d13, st);
        if (e == cudaSuccess) e = launch_repack(w2, sf2, n, H, I, false, d2, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(gs13, gs13_h.data(), (size_t)n * 2 * sizeof(float), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(gs2, gs2_h.data(), (size_t)n * sizeof(float), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    cudaFree(mm);
    cudaFree(offs);
    cudaFree(sf13);
    cudaFree(sf2);
    return e;
}

// The single launch tags the words its blocks exchange with the call number
// (32 bits): restart the per-block call counters and clear the tagged words,
// enqueued on `st` (stream order puts it after the last call and before the
// next one).
cudaError_t restart_tags(moe_layer *L, cudaStream_t st) {
    const int Tf = std::min(L->cfg.max_tokens, 8);
    cudaError_t e = cudaMemsetAsync(L->d.calls, 0, sizeof(unsigned) * L->sm_count, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L->d.logit_tag, 0, sizeof(unsigned long long) * Tf * L->d.E, st);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(L->d.h_tag, 0, sizeof(unsigned long long) * Tf * (L->d.k + L->d.S) * (L->d.Imax / 2), st);
    L->fused_calls = 0;
    return e;
}

// Restart the tags well before the 32-bit call number could wrap to a value
// that words left from an early call still carry.
constexpr unsigned long long kTagRestart = 1ull << 31;

moe_status check_call(moe_layer *L, int T) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer handle is NULL");
    if (T < 1 || T > L->cfg.max_tokens)
        return fail(MOE_ERR_INVALID_ARG,
                    "T=" + std::to_string(T) + " outside [1, max_tokens=" +
                        std::to_string(L->cfg.max_tokens) + "]");
    return MOE_OK;
}

}  // namespace

namespace moe {
// Lets other translation units report through moe_last_error().
void record_error(const std::string &msg) { g_err = msg; }
}  // namespace moe

extern "C" {

const char *moe_last_error(void) { return g_err.c_str(); }

moe_status moe_init(const moe_config *cfg, const moe_weights *w, void *stream, moe_layer **out) {
    g_err.clear();
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!cfg || !w) return fail(MOE_ERR_INVALID_ARG, "cfg or weights is NULL");
    std::vector<std::string> why = unsupported_reasons(cfg);
    if (!why.empty()) return fail(MOE_ERR_UNSUPPORTED, join(why));

    const int S = cfg->num_shared;
    std::vector<std::string> bad;
    auto need = [&](const void *p, const char *name) {
        if (!p) bad.push_back(std::string(name) + " is NULL");
        else if (!aligned16(p)) bad.push_back(std::string(name) + " is not 16-byte aligned");
        else if (!is_device_ptr(p)) bad.push_back(std::string(name) + " is not a device pointer");
    };
    need(w->router_w, "router_w");
    if (w->router_b) need(w->router_b, "router_b");
    need(w->w13, "w13");
    need(w->w13_sf, "w13_sf");
    need(w->w2, "w2");
    need(w->w2_sf, "w2_sf");
    if (cfg->expert_format == MOE_FMT_NVFP4) {   // tensor scales: NVFP4 only
        need(w->w13_gs, "w13_gs");
        need(w->w2_gs, "w2_gs");
    }
    if (S > 0) {
        need(w->sw13, "sw13");
        need(w->sw13_sf, "sw13_sf");
        need(w->sw2, "sw2");
        need(w->sw2_sf, "sw2_sf");
        if (cfg->shared_format == MOE_FMT_NVFP4) {
            need(w->sw13_gs, "sw13_gs");
            need(w->sw2_gs, "sw2_gs");
        }
    }
    if (!bad.empty()) return fail(MOE_ERR_INVALID_ARG, join(bad));

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    moe_layer *L = new moe_layer();
    L->cfg = *cfg;
    if (L->cfg.grouped_min_tokens == 0) L->cfg.grouped_min_tokens = 8;
    cudaError_t e = cudaGetDevice(&L->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L->sm_count, cudaDevAttrMultiProcessorCount, L->device);
    if (e != cudaSuccess) {
        delete L;
        return cuda_fail(e, "device query");
    }
    const int E = cfg->num_experts, H = cfg->hidden, I = cfg->inter, K = cfg->top_k;
    const int Is = S > 0 ? cfg->shared_inter : I;
    DevLayer &d = L->d;
    d.H = H;
    d.E = E;
    d.k = K;
    d.I = I;
    d.S = S;
    d.Is = Is;
    d.normalize = cfg->normalize_topk;
    d.routed_scale = cfg->routed_scale;
    d.score_func = cfg->score_func;
    d.max_tokens = cfg->max_tokens;
    d.max_slots = std::min(E, cfg->max_tokens * K) + S;
    d.max_pairs = cfg->max_tokens * (K + S);
    d.Imax = std::max(I, Is);
    d.grouped_min = 0;   // set once the shape is known to suit the grouped kernels
    d.debug_stall = 0;
    d.f8e = is_f8(cfg->expert_format);
    d.f8s = S > 0 && is_f8(cfg->shared_format);
    d.w4a4 = cfg->w4a4;

    carve_weights(L, nullptr);
    carve_workspace(L, nullptr);
    e = cudaMalloc(&L->wmem, L->wbytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete L;
        return fail(MOE_ERR_OOM, "cudaMalloc of " + std::to_string(L->wbytes) + " weight bytes failed");
    }
    e = cudaMalloc(&L->wsmem, L->wsbytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFree(L->wmem);
        delete L;
        return fail(MOE_ERR_OOM, "cudaMalloc of workspace failed");
    }
    carve_weights(L, static_cast<char *>(L->wmem));
    carve_workspace(L, static_cast<char *>(L->wsmem));
    L->expert_bytes = d.e13_stride + d.e2_stride;
    L->shared_bytes = d.s13_stride + d.s2_stride;

    auto cp = [&](const void *dst, const void *src, size_t n) {
        if (e == cudaSuccess && n) e = cudaMemcpyAsync(const_cast<void *>(dst), src, n, cudaMemcpyDeviceToDevice, st);
    };
    cp(d.router_w, w->router_w, (size_t)E * H * sizeof(float));
    if (w->router_b) {
        cp(L->router_b_slot, w->router_b, (size_t)E * sizeof(float));
        d.router_b = L->router_b_slot;
    }
    std::vector<std::string> fmt_why;
    if (e == cudaSuccess)
        e = repack_group(cfg->expert_format, E, H, I, w->w13, w->w13_sf, w->w13_gs, w->w2, w->w2_sf, w->w2_gs,
                         const_cast<uint8_t *>(d.w13r), const_cast<uint8_t *>(d.w2r), const_cast<float *>(d.gs13),
                         const_cast<float *>(d.gs2), L->gs13_h, L->gs2_h, "routed", fmt_why, st);
    if (e == cudaSuccess)
        e = repack_group(cfg->shared_format, S, H, Is, w->sw13, w->sw13_sf, w->sw13_gs, w->sw2, w->sw2_sf,
                         w->sw2_gs, const_cast<uint8_t *>(d.sw13r), const_cast<uint8_t *>(d.sw2r),
                         const_cast<float *>(d.sgs13), const_cast<float *>(d.sgs2), L->sgs13_h, L->sgs2_h,
                         "shared", fmt_why, st);
    if (e == cudaSuccess && !fmt_why.empty()) {
        cudaStreamSynchronize(st);
        cudaFree(L->wmem);
        cudaFree(L->wsmem);
        delete L;
        return fail(MOE_ERR_UNSUPPORTED, join(fmt_why));
    }
    if (e == cudaSuccess) e = launch_pack_scales(d, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L->wsmem, 0, L->wsbytes, st);
    if (e == cudaSuccess) e = prepare_kernels();
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&L->optin_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, L->device);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    // the grouped tensor-core kernels decode NVFP4 chunks only
    if (L->cfg.grouped_min_tokens > 0 && !d.f8e && !d.f8s && grouped_supported(d, L->sm_count))
        d.grouped_min = L->cfg.grouped_min_tokens;
    d.nsm = L->sm_count;
    d.tau_max = cold_threshold_max(d, L->sm_count, L->optin_smem);
    for (int T = 0; T <= kMaxTokens; ++T) {
        L->fused_ok[T] = 0;
        if (e == cudaSuccess && cfg->fused >= 0 && !cfg->w4a4 && T >= 1 && T <= cfg->max_tokens &&
            fused_eligible(d, T, L->sm_count, (size_t)L->optin_smem))
            L->fused_ok[T] = fused_blocks_per_sm(d, T) >= 1;
    }
    if (e != cudaSuccess) {
        moe_status rs = cuda_fail(e, "moe_init");
        cudaFree(L->wmem);
        cudaFree(L->wsmem);
        delete L;
        return rs;
    }
    *out = L;
    return MOE_OK;
}

void moe_destroy(moe_layer *L) {
    if (!L) return;
    DeviceGuard g(L->device);
    cudaDeviceSynchronize();
    cudaFree(L->wmem);
    cudaFree(L->wsmem);
    delete L;
}

moe_status moe_stage_route(moe_layer *L, const void *x, int T, int *topk_ids, float *topk_w,
                           void *stream) {
    moe_status rc = check_call(L, T);
    if (rc != MOE_OK) return rc;
    if (!x || !aligned16(x)) return fail(MOE_ERR_INVALID_ARG, "x is NULL or not 16-byte aligned");
    DeviceGuard g(L->device);
    cudaError_t e = launch_route(L->d, static_cast<const __nv_bfloat16 *>(x), T, topk_ids, topk_w, L->sm_count,
                                 reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "router launch");
}

moe_status moe_stage_gate_up(moe_layer *L, const void *x, int T, void *stream) {
    moe_status rc = check_call(L, T);
    if (rc != MOE_OK) return rc;
    if (!x || !aligned16(x)) return fail(MOE_ERR_INVALID_ARG, "x is NULL or not 16-byte aligned");
    DeviceGuard g(L->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const __nv_bfloat16 *xa = static_cast<const __nv_bfloat16 *>(x);
    cudaError_t e = cudaSuccess;
    if (L->d.w4a4) {
        // W4A4: the tokens quantised first (their f16 prescale exponents are
        // the only ones: the router leaves them out); gate/up reads the
        // dequantised rows.  The router's launch comes right before this one
        // (the stages run in order), so the quantiser runs beside it and
        // waits for it at its end.
        const int H = L->cfg.hidden;
        e = launch_fos(xa, L->d.xq, T, H, H, 0, 0, L->d.gsx, L->d.xexp, nullptr, L->d.xq4, L->d.xsf, H / 2, H / 16,
                       st, true);
        xa = L->d.xq;
    }
    if (e == cudaSuccess) e = launch_gate_up(L->d, xa, T, L->sm_count, L->optin_smem, st);
    // above 8 tokens the GEMV kernel leaves the slots with >= grouped_min
    // tokens to the grouped tensor-core kernel
    if (e == cudaSuccess && T > 8 && L->d.grouped_min > 0)
        e = launch_grouped_gate_up(L->d, xa, T, L->sm_count, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "gate/up launch");
}

moe_status moe_stage_down(moe_layer *L, int T, void *out, void *stream) {
    moe_status rc = check_call(L, T);
    if (rc != MOE_OK) return rc;
    if (!out || !aligned16(out)) return fail(MOE_ERR_INVALID_ARG, "out is NULL or not 16-byte aligned");
    DeviceGuard g(L->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (L->d.w4a4) {
        // W4A4: the h rows quantised in place (the shared experts' pairs
        // first, rows of Is; then the routed ones, rows of I); their maxima
        // replace those the SwiGLU epilogue left for the down prescale
        const DevLayer &d = L->d;
        e = launch_fos(d.h_ws, d.h_ws, T * (d.k + d.S), d.Imax, d.I, d.S * T, d.Is, d.gsh, nullptr, d.hmax, d.hq4,
                       d.hsf, d.Imax / 2, d.Imax / 16, st);
    }
    if (e == cudaSuccess) e = launch_down(L->d, T, static_cast<__nv_bfloat16 *>(out), L->sm_count, L->optin_smem, st);
    if (e == cudaSuccess && T > 8 && L->d.grouped_min > 0) {
        DevLayer dd = L->d;
        dd.tick16 = down_tile_tickets(L->d, T, L->sm_count, L->optin_smem) ? 1 : 0;
        e = launch_grouped_down(dd, T, static_cast<__nv_bfloat16 *>(out), L->sm_count, st);
    }
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "down launch");
}

// The single launch for one call (L->fused_ok[T]); x_sys: x is the device
// alias of pinned host memory.
static moe_status forward_fused(moe_layer *L, const void *x, int T, void *out, int *topk_ids, float *topk_w,
                                void *stream, bool x_sys) {
    DeviceGuard g(L->device);
    DevLayer d = L->d;
    d.debug_stall = L->inject_stall;
    L->inject_stall = 0;
    cudaError_t e = cudaSuccess;
    if (++L->fused_calls >= kTagRestart) e = restart_tags(L, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tag restart");
    e = launch_fused(d, static_cast<const __nv_bfloat16 *>(x), T, static_cast<__nv_bfloat16 *>(out), topk_ids, topk_w,
                     L->sm_count, L->cfg.fused > 0, reinterpret_cast<cudaStream_t>(stream), x_sys);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "single-launch layer");
}

moe_status moe_decode_forward(moe_layer *L, const void *x, int T, void *out, int *topk_ids,
                              float *topk_w, void *stream) {
    moe_status rc = check_call(L, T);
    if (rc != MOE_OK) return rc;
    if (!x || !aligned16(x)) return fail(MOE_ERR_INVALID_ARG, "x is NULL or not 16-byte aligned");
    if (!out || !aligned16(out)) return fail(MOE_ERR_INVALID_ARG, "out is NULL or not 16-byte aligned");
    const size_t nb = (size_t)T * L->cfg.hidden * 2;
    const char *xa = static_cast<const char *>(x), *oa = static_cast<const char *>(out);
    if (xa < oa + nb && oa < xa + nb) return fail(MOE_ERR_INVALID_ARG, "out overlaps x");
    if (L->fused_ok[T]) return forward_fused(L, x, T, out, topk_ids, topk_w, stream, false);
    rc = moe_stage_route(L, x, T, topk_ids, topk_w, stream);
    if (rc == MOE_OK) rc = moe_stage_gate_up(L, x, T, stream);
    if (rc == MOE_OK) rc = moe_stage_down(L, T, out, stream);
    return rc;
}

moe_status moe_decode_forward_host(moe_layer *L, const void *x_host, int T, void *out_host,
                                   int *topk_ids_host, float *topk_w_host, void *stream) {
    moe_status rc = check_call(L, T);
    if (rc != MOE_OK) return rc;
    if (!x_host || !out_host) return fail(MOE_ERR_INVALID_ARG, "x_host or out_host is NULL");
    DeviceGuard g(L->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t nb = (size_t)T * L->cfg.hidden * 2;
    const size_t nk = (size_t)T * L->cfg.top_k;
    // pinned (page-locked, mapped) host buffers: their device aliases
    auto alias = [](const void *p) -> void * {
        cudaPointerAttributes pa;
        void *dev = nullptr;
        if (cudaPointerGetAttributes(&pa, p) == cudaSuccess && pa.type == cudaMemoryTypeHost && pa.devicePointer &&
            aligned16(pa.devicePointer))
            dev = pa.devicePointer;
        cudaGetLastError();
        return dev;
    };
    // the kernels store the output straight into a pinned out_host instead of
    // a copy after them; the single launch of one or two tokens also reads a
    // pinned x_host in place (each block reads the rows once), so that no copy
    // stands between two layers' kernels
    void *out_dev = alias(out_host);
    const char *xa = static_cast<const char *>(x_host), *oa = static_cast<const char *>(out_host);
    const bool apart = !(xa < oa + nb && oa < xa + nb);
    const void *x_dev = L->fused_ok[T] && T <= 2 && apart ? alias(x_host) : nullptr;
    if (x_dev) {
        rc = forward_fused(L, x_dev, T, out_dev ? out_dev : L->out_stage, L->ids_stage, L->w_stage, stream, true);
    } else {
        cudaError_t e = cudaMemcpyAsync(L->x_stage, x_host, nb, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return cuda_fail(e, "x upload");
        rc = moe_decode_forward(L, L->x_stage, T, out_dev ? out_dev : L->out_stage, L->ids_stage, L->w_stage, stream);
    }
    if (rc != MOE_OK) return rc;
    cudaError_t e;
    e = out_dev ? cudaSuccess : cudaMemcpyAsync(out_host, L->out_stage, nb, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && topk_ids_host)
        e = cudaMemcpyAsync(topk_ids_host, L->ids_stage, nk * sizeof(int), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && topk_w_host)
        e = cudaMemcpyAsync(topk_w_host, L->w_stage, nk * sizeof(float), cudaMemcpyDeviceToHost, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "result download");
}

moe_status moe_check(moe_layer *L, void *stream) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer handle is NULL");
    DeviceGuard g(L->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int word = 0;
    e = cudaMemcpy(&word, L->d.err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "error word read");
    // restart the single-launch path's call counters and clear the words
    // tagged with them (after a wait that gave up the blocks' counters may
    // disagree; otherwise this bounds the count between checks)
    e = restart_tags(L, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "tag restart");
    if (word == 0) return MOE_OK;
    int zero = 0;
    cudaMemcpy(L->d.err, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (word == 1) return fail(MOE_ERR_TIMEOUT, "an in-kernel wait gave up");
    return fail(MOE_ERR_DEVICE, "device error word " + std::to_string(word));
}

moe_status moe_debug_dequant(moe_layer *L, int which, int expert, float *dst, void *stream) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer handle is NULL");
    if (!dst) return fail(MOE_ERR_INVALID_ARG, "dst is NULL");
    const DevLayer &d = L->d;
    const uint8_t *rep = nullptr;
    int rows = 0, cols = 0;
    float ga = 0.f, gb = 0.f;
    bool gu = false;
    if (which == 0 || which == 1) {
        if (expert < 0 || expert >= d.E) return fail(MOE_ERR_INVALID_ARG, "expert out of range");
        if (which == 0) {
            rep = d.w13r + (size_t)expert * d.e13_stride;
            rows = 2 * d.I;
            cols = d.H;
            ga = L->gs13_h[2 * expert];
            gb = L->gs13_h[2 * expert + 1];
            gu = true;
        } else {
            rep = d.w2r + (size_t)expert * d.e2_stride;
            rows = d.H;
            cols = d.I;
            ga = gb = L->gs2_h[expert];
        }
    } else if (which == 2 || which == 3) {
        if (expert < 0 || expert >= d.S) return fail(MOE_ERR_INVALID_ARG, "shared index out of range");
        if (which == 2) {
            rep = d.sw13r + (size_t)expert * d.s13_stride;
            rows = 2 * d.Is;
            cols = d.H;
            ga = L->sgs13_h[2 * expert];
            gb = L->sgs13_h[2 * expert + 1];
            gu = true;
        } else {
            rep = d.sw2r + (size_t)expert * d.s2_stride;
            rows = d.H;
            cols = d.Is;
            ga = gb = L->sgs2_h[expert];
        }
    } else {
        return fail(MOE_ERR_INVALID_ARG, "which must be 0..3");
    }
    DeviceGuard g(L->device);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool f8 = which < 2 ? d.f8e : d.f8s;
    cudaError_t e = f8 ? launch_dequant_f8(rep, rows, cols, gu, dst, st)
                       : launch_dequant(rep, ga, gb, rows, cols, gu, dst, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "dequant");
}

moe_status moe_trace_attach(moe_layer *L, unsigned long long *buf, int blocks_per_kernel) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer handle is NULL");
#ifdef MOE_TRACE
    L->d.trace = buf;
    L->d.trace_blocks = buf ? blocks_per_kernel : 0;
    return MOE_OK;
#else
    (void)buf;
    (void)blocks_per_kernel;
    return fail(MOE_ERR_UNSUPPORTED, "this library was built without MOE_TRACE");
#endif
}

moe_status moe_debug_inject(moe_layer *L, int what, int value) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer handle is NULL");
    if (what != MOE_INJECT_WAIT_STALL) return fail(MOE_ERR_INVALID_ARG, "unknown injection " + std::to_string(what));
    if (value < 0) return fail(MOE_ERR_INVALID_ARG, "injection value must be >= 0");
    L->inject_stall = value;
    return MOE_OK;
}

moe_status moe_quant_fos(const void *x, int rows, int n, void *deq, float *gs, void *stream) {
    g_err.clear();
    if (rows < 0 || n <= 0 || n % 16 != 0)
        return fail(MOE_ERR_INVALID_ARG, "rows must be >= 0 and n a positive multiple of 16");
    if (rows == 0) return MOE_OK;
    if (!x || !deq || !gs) return fail(MOE_ERR_INVALID_ARG, "x, deq or gs is NULL");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(deq)) % 8 != 0)
        return fail(MOE_ERR_INVALID_ARG, "x and deq must be 8-byte aligned");
    cudaError_t e = launch_fos(static_cast<const __nv_bfloat16 *>(x), static_cast<__nv_bfloat16 *>(deq), rows, n, n,
                               0, 0, gs, nullptr, nullptr, nullptr, nullptr, 0, 0,
                               reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "quantiser launch");
}

moe_status moe_get_info(const moe_layer *L, moe_layer_info *info) {
    if (!L || !info) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    info->weight_bytes = L->wbytes;
    info->workspace_bytes = L->wsbytes;
    info->expert_bytes = L->expert_bytes;
    info->shared_bytes = L->shared_bytes;
    info->max_slots = L->d.max_slots;
    info->sm_count = L->sm_count;
    info->single_launch_max_tokens = 0;
    for (int T = 1; T <= L->cfg.max_tokens; ++T)
        if (L->fused_ok[T]) info->single_launch_max_tokens = T;
    return MOE_OK;
}

}  // extern "C"
