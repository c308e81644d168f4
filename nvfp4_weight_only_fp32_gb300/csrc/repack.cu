// repack.cu -- the load-time, lossless repack of NVFP4 expert weights into the
// streaming chunk layout (described in moe_internal.cuh), and its inverse
// decoder used by moe_debug_dequant.
//
// The Flint page ("vLLM Day-0 support for Recursive's Flint", section "Flint
// model overview") repacks its NVFP4 checkpoint losslessly when loading it; the
// same idea here turns the canonical row-major codes/scales into 576-byte
// chunks so that one warp streams a 16x64 tile with one 16-byte and one 8-byte
// load per lane.
#include "moe_internal.cuh"

namespace moe {

namespace {

// Canonical row of MMA row `rho` of tile `r`.
__device__ __forceinline__ int canon_row(int rho, int r, int rows, bool gate_up) {
    if (!gate_up) return 16 * r + rho;
    int half = rows / 2;  // I: rows < I are gate, rows >= I are up
    return rho < 8 ? 8 * r + rho : half + 8 * r + (rho - 8);
}

__global__ void repack_kernel(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ sf,
                              int n_mats, int rows, int cols, bool gate_up,
                              uint8_t *__restrict__ dst) {
    const int NT = rows / 16, NC = cols / kChunkK;
    const size_t total = (size_t)n_mats * NT * NC * kChunkBytes;
    const size_t code_row = (size_t)cols / 2, sf_row = (size_t)cols / kBlockK;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        size_t chunk = idx / kChunkBytes;
        int off = (int)(idx % kChunkBytes);
        int c = (int)(chunk % NC);
        int r = (int)((chunk / NC) % NT);
        size_t mat = chunk / ((size_t)NC * NT);
        if (off < kCodeBytes) {
            int L = off / 16, i = (off % 16) / 4, b = off % 4;
            int g = L / 4, q = L % 4;
            int rho = (b & 1) ? g + 8 : g;
            int k = kBlockK * (4 * c + i) + 2 * q + ((b & 2) ? 8 : 0);
            int R = canon_row(rho, r, rows, gate_up);
            dst[idx] = codes[(mat * rows + R) * code_row + (size_t)(k / 2)];
        } else {
            int s = off - kCodeBytes;
            int g = s / 8, i = (s % 8) / 2, h = s % 2;
            int R = canon_row(g + 8 * h, r, rows, gate_up);
            dst[idx] = sf[(mat * rows + R) * sf_row + (size_t)(4 * c + i)];
        }
    }
}

// One warp per (tile, chunk): decode with the GEMV kernels' own decoder and
// scatter back to canonical [rows, cols] FP32, value = fl32(e2m1*e4m3*gs).
__global__ void dequant_kernel(const uint8_t *__restrict__ rep, float gs_a, float gs_b,
                               int rows, int cols, bool gate_up, float *__restrict__ dst) {
    const int NT = rows / 16, NC = cols / kChunkK;
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= NT * NC) return;
    const int r = warp / NC, c = warp % NC;
    const uint8_t *chunk = rep + (size_t)warp * kChunkBytes;
    const uint64_t pol = evict_first_policy();
    uint4 cw = ld_stream_v4(chunk + 16 * lane, pol);
    const int g = lane >> 2, q = lane & 3;
    uint2 sw = ld_stream_v2(chunk + kCodeBytes + 8 * g, pol);
    uint32_t a[4][4];
    decode_chunk(cw, sw, a);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            int rho = (b & 1) ? g + 8 : g;
            int k = kBlockK * (4 * c + i) + 2 * q + ((b & 2) ? 8 : 0);
            int R = canon_row(rho, r, rows, gate_up);
            float gs = (gate_up && rho >= 8) ? gs_b : gs_a;
            __half2 h2 = *reinterpret_cast<__half2 *>(&a[i][b]);
            float2 f = __half22float2(h2);
            dst[(size_t)R * cols + k] = __fmul_rn(f.x, gs);
            dst[(size_t)R * cols + k + 1] = __fmul_rn(f.y, gs);
        }
    }
}

// One 16-byte record per expert (routed, then shared): the global scales of
// gate, up and down and the router bias, so that a block fetches them all
// with one bulk copy.
__global__ void pack_scales_kernel(DevLayer d) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= d.E + d.S) return;
    float4 v;
    if (i < d.E) {
        v = make_float4(d.gs13[2 * i], d.gs13[2 * i + 1], d.gs2[i], d.router_b ? d.router_b[i] : 0.f);
    } else {
        const int si = i - d.E;
        v = make_float4(d.sgs13[2 * si], d.sgs13[2 * si + 1], d.sgs2[si], 0.f);
    }
    const_cast<float4 *>(d.gsp)[i] = v;
}

}  // namespace

cudaError_t launch_pack_scales(const DevLayer &d, cudaStream_t s) {
    pack_scales_kernel<<<(d.E + d.S + 255) / 256, 256, 0, s>>>(d);
    return cudaGetLastError();
}

cudaError_t launch_repack(const uint8_t *codes, const uint8_t *sf, int n_mats, int rows, int cols,
                          bool gate_up, uint8_t *dst, cudaStream_t s) {
    if (n_mats <= 0) return cudaSuccess;
    size_t total = (size_t)n_mats * repacked_bytes(rows, cols);
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535u * 32u) blocks = 65535u * 32u;
    repack_kernel<<<(unsigned)blocks, 256, 0, s>>>(codes, sf, n_mats, rows, cols, gate_up, dst);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t *rep, float gs_a, float gs_b, int rows, int cols,
                           bool gate_up, float *dst, cudaStream_t s) {
    int warps = (rows / 16) * (cols / kChunkK);
    int blocks = (warps + 7) / 8;
    dequant_kernel<<<blocks, 256, 0, s>>>(rep, gs_a, gs_b, rows, cols, gate_up, dst);
    return cudaGetLastError();
}

}  // namespace moe
