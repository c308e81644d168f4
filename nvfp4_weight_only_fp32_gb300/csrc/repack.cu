// repack.cu -- the load-time, lossless repack of the expert weights into the
// streaming chunk layouts (described in moe_internal.cuh), and the inverse
// decoders used by moe_debug_dequant.  NVFP4 and MXFP4 experts become NVFP4
// chunks (MXFP4 through an exact change of scale: "Day 0 support for Mistral
// Large 4 on vLLM", "MXFP4 experts at load, one layer at a time": E2M1 values
// with one E8M0 scale per 32); FP8 experts (block-scaled, or MXFP8: "Inkling 2
// Small on vLLM: Day-0 Support", "Mixed-precision MoE and Four-Over-Six
// NVFP4") become F8 chunks.
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

// F8 chunks (layout in moe_internal.cuh) from canonical E4M3 codes and their
// scales: fmt 2 = one FP32 per 128 x 128 block, 3 = one E8M0 per 32 elements
// of a row.  One thread per output byte.
__global__ void repack_f8_kernel(const uint8_t *__restrict__ codes, const void *__restrict__ sfv, int fmt,
                                 int n_mats, int rows, int cols, bool gate_up, uint8_t *__restrict__ dst) {
    const int NT = rows / 16, NC = cols / kChunkK8;
    const size_t total = (size_t)n_mats * NT * NC * kChunkBytes;
    const int nbr = (rows + 127) / 128, nbc = (cols + 127) / 128;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t chunk = idx / kChunkBytes;
        const int off = (int)(idx % kChunkBytes);
        const int c = (int)(chunk % NC);
        const int r = (int)((chunk / NC) % NT);
        const size_t mat = chunk / ((size_t)NC * NT);
        if (off < kCodeBytes) {
            const int L = off / 16, p = off % 16;
            const int g = L / 4, q = L % 4;
            const int kb = p / 8, j = (p % 8) / 2, e = p % 2;
            const int rho = (j & 1) ? g + 8 : g;
            const int k = kChunkK8 * c + 16 * kb + 2 * q + ((j & 2) ? 8 : 0) + e;
            const int R = canon_row(rho, r, rows, gate_up);
            dst[idx] = codes[(mat * rows + R) * (size_t)cols + k];
        } else {
            const int sb = off - kCodeBytes;
            const int g = sb / 8, h = (sb % 8) / 4, byte = sb % 4;
            const int R = canon_row(g + 8 * h, r, rows, gate_up);
            float v;
            if (fmt == 2) {
                v = reinterpret_cast<const float *>(sfv)[(mat * nbr + R / 128) * (size_t)nbc + (kChunkK8 * c) / 128];
            } else {
                const int ec = reinterpret_cast<const uint8_t *>(sfv)[(mat * rows + R) * (size_t)(cols / 32) + c];
                // 2^(ec - 127): normal for ec >= 1, 2^-127 (subnormal) for 0,
                // NaN for 255
                v = ec == 255 ? __int_as_float(0x7fc00000) : ec == 0 ? __int_as_float(0x00400000)
                                                                      : __int_as_float(ec << 23);
            }
            dst[idx] = (uint8_t)(__float_as_uint(v) >> (8 * byte));
        }
    }
}

// One warp per (tile, F8 chunk): decode with the kernels' own F8 decoder and
// scatter back to canonical [rows, cols] FP32, value = fl32(e4m3 * scale).
__global__ void dequant_f8_kernel(const uint8_t *__restrict__ rep, int rows, int cols, bool gate_up,
                                  float *__restrict__ dst) {
    const int NT = rows / 16, NC = cols / kChunkK8;
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= NT * NC) return;
    const int r = warp / NC, c = warp % NC;
    const uint8_t *chunk = rep + (size_t)warp * kChunkBytes;
    const uint64_t pol = evict_first_policy();
    const uint4 cw = ld_stream_v4(chunk + 16 * lane, pol);
    const int g = lane >> 2, q = lane & 3;
    const uint2 sw = ld_stream_v2(chunk + kCodeBytes + 8 * g, pol);
    uint32_t a[2][4];
    decode_chunk_f8(cw, a);
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int rho = (j & 1) ? g + 8 : g;
            const int k = kChunkK8 * c + 16 * kb + 2 * q + ((j & 2) ? 8 : 0);
            const int R = canon_row(rho, r, rows, gate_up);
            const float sc = __uint_as_float((j & 1) ? sw.y : sw.x);
            const float2 f = __half22float2(*reinterpret_cast<__half2 *>(&a[kb][j]));
            dst[(size_t)R * cols + k] = __fmul_rn(f.x, sc);
            dst[(size_t)R * cols + k + 1] = __fmul_rn(f.y, sc);
        }
    }
}

// Smallest and largest E8M0 code (and any NaN code) per (matrix, half): one
// block per (matrix, half).
__global__ void mx_scale_range_kernel(const uint8_t *__restrict__ sf, int rows, int cols, bool gate_up,
                                      int *__restrict__ mm) {
    const int mat = blockIdx.x >> 1, half = blockIdx.x & 1;
    const int nr = gate_up ? rows / 2 : rows, r0 = half * nr;
    const size_t per_row = (size_t)cols / 32;
    __shared__ int s_mn, s_mx, s_nan;
    if (threadIdx.x == 0) {
        s_mn = 255;
        s_mx = 0;
        s_nan = 0;
    }
    __syncthreads();
    int mn = 255, mx = 0, nan = 0;
    if (gate_up || half == 0) {
        const uint8_t *base = sf + ((size_t)mat * rows + r0) * per_row;
        for (size_t i = threadIdx.x; i < (size_t)nr * per_row; i += blockDim.x) {
            const int v = base[i];
            if (v == 255) nan = 1;
            else {
                mn = min(mn, v);
                mx = max(mx, v);
            }
        }
    }
    atomicMin(&s_mn, mn);
    atomicMax(&s_mx, mx);
    atomicMax(&s_nan, nan);
    __syncthreads();
    if (threadIdx.x == 0) {
        mm[blockIdx.x * 3 + 0] = s_mn;
        mm[blockIdx.x * 3 + 1] = s_mx;
        mm[blockIdx.x * 3 + 2] = s_nan;
    }
}

// E4M3 code of 2^j for -9 <= j <= 8 (exact: subnormal below 2^-6).
__device__ __forceinline__ uint8_t e4m3_pow2(int j) {
    return j >= -6 ? (uint8_t)((j + 7) << 3) : (uint8_t)(1 << (j + 9));
}

__global__ void mx_to_nv_kernel(const uint8_t *__restrict__ sf, const int *__restrict__ offs, int n_mats,
                                int rows, int cols, bool gate_up, uint8_t *__restrict__ dst) {
    const size_t per_row = (size_t)cols / 16, total = (size_t)n_mats * rows * per_row;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t row = i / per_row;
        const int b16 = (int)(i % per_row);
        const int mat = (int)(row / rows), R = (int)(row % rows);
        const int half = gate_up && R >= rows / 2;
        const int ec = sf[row * (per_row / 2) + b16 / 2];
        dst[i] = e4m3_pow2(ec - 127 - offs[mat * 2 + half]);
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

cudaError_t launch_repack_f8(const uint8_t *codes, const void *sf, int fmt, int n_mats, int rows, int cols,
                             bool gate_up, uint8_t *dst, cudaStream_t s) {
    if (n_mats <= 0) return cudaSuccess;
    size_t total = (size_t)n_mats * repacked_bytes(rows, cols, true);
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535u * 32u) blocks = 65535u * 32u;
    repack_f8_kernel<<<(unsigned)blocks, 256, 0, s>>>(codes, sf, fmt, n_mats, rows, cols, gate_up, dst);
    return cudaGetLastError();
}

cudaError_t launch_dequant_f8(const uint8_t *rep, int rows, int cols, bool gate_up, float *dst, cudaStream_t s) {
    int warps = (rows / 16) * (cols / kChunkK8);
    dequant_f8_kernel<<<(warps + 7) / 8, 256, 0, s>>>(rep, rows, cols, gate_up, dst);
    return cudaGetLastError();
}

cudaError_t launch_mx_scale_range(const uint8_t *sf, int n_mats, int rows, int cols, bool gate_up, int *mm,
                                  cudaStream_t s) {
    if (n_mats <= 0) return cudaSuccess;
    mx_scale_range_kernel<<<2 * n_mats, 256, 0, s>>>(sf, rows, cols, gate_up, mm);
    return cudaGetLastError();
}

cudaError_t launch_mx_to_nv_scales(const uint8_t *sf, const int *offs, int n_mats, int rows, int cols,
                                   bool gate_up, uint8_t *dst, cudaStream_t s) {
    if (n_mats <= 0) return cudaSuccess;
    size_t total = (size_t)n_mats * rows * (cols / 16);
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535u * 32u) blocks = 65535u * 32u;
    mx_to_nv_kernel<<<(unsigned)blocks, 256, 0, s>>>(sf, offs, n_mats, rows, cols, gate_up, dst);
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
