// simt.cuh -- the block's memory-bound steps as vectorised SIMT kernels:
// the RoPE table, LayerNorm + per-stream modulation, and the Euler update.
#pragma once
#include "sm103.cuh"
#include "../../include/flux3.h"

namespace f3 {

struct SegOffsets {
    int n_seg;
    int off[FLUX3_MAX_SEGMENTS + 1];
};

F3_DEV int segment_of_row(const SegOffsets& s, int r) {
    int g = 0;
#pragma unroll 1
    for (int i = 1; i < s.n_seg; ++i)
        if (r >= s.off[i]) g = i;
    return g;
}

// ---------------------------------------------------------------- RoPE table
// rope[r][p] = (cos, sin)(pos[r][a] * theta^(-2j/32)), p = 16 a + j.  The angle and its
// sine/cosine are taken in fp64 (angles reach thousands of radians) and rounded to fp32.
__global__ void rope_table_kernel(const int* __restrict__ pos, int n_tokens, double log2_theta, float2* __restrict__ rope) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)n_tokens * 64) return;
    const int r = (int)(i >> 6), pr = (int)(i & 63);
    const int axis = pr >> 4, j = pr & 15;
    const double freq = exp2(-(double)(2 * j) / 32.0 * log2_theta);
    const double ang = (double)pos[4 * r + axis] * freq;
    double s, c;
    sincos(ang, &s, &c);
    rope[i] = make_float2((float)c, (float)s);
}

// ---------------------------------------------------------------- LayerNorm + modulation
// One warp per row, the row held in registers (D <= 32 * 8 * kMaxChunks), two-pass
// statistics in fp32, output a = (x - mean) * rstd * (1 + scale_s) + shift_s in bf16.
constexpr int kAdaLnMaxChunks = 16;  // D <= 4096

__global__ void __launch_bounds__(256) adaln_kernel(const __nv_bfloat16* __restrict__ x, int n_rows, int D, float eps,
                                                    const float* __restrict__ mod, const SegOffsets segs, int row_offset,
                                                    __nv_bfloat16* __restrict__ a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + warp;
    if (r >= n_rows) return;
    const int nc = D >> 8;  // chunks of 256 columns: 8 per lane
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * D);
    float v[kAdaLnMaxChunks][8];
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < kAdaLnMaxChunks; ++c) {
        if (c < nc) {
            const uint4 u = __ldg(xr + c * 32 + lane);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
                v[c][2 * e] = __bfloat162float(h.x);
                v[c][2 * e + 1] = __bfloat162float(h.y);
                sum += v[c][2 * e] + v[c][2 * e + 1];
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum / (float)D;
    float sq = 0.f;
#pragma unroll
    for (int c = 0; c < kAdaLnMaxChunks; ++c)
        if (c < nc) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float d = v[c][e] - mean;
                sq = fmaf(d, d, sq);
            }
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    const float rstd = rsqrtf(sq / (float)D + eps);
    const int seg = segment_of_row(segs, r + row_offset);
    const float* shift = mod + (size_t)seg * 3 * D;
    const float* scale = shift + D;
    uint4* ar = reinterpret_cast<uint4*>(a + (size_t)r * D);
#pragma unroll
    for (int c = 0; c < kAdaLnMaxChunks; ++c) {
        if (c < nc) {
            const int col = c * 256 + lane * 8;
            const float4 s0 = __ldg(reinterpret_cast<const float4*>(scale + col));
            const float4 s1 = __ldg(reinterpret_cast<const float4*>(scale + col + 4));
            const float4 h0 = __ldg(reinterpret_cast<const float4*>(shift + col));
            const float4 h1 = __ldg(reinterpret_cast<const float4*>(shift + col + 4));
            const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
            const float sh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = fmaf((v[c][e] - mean) * rstd, 1.f + sc[e], sh[e]);
            ar[c * 32 + lane] = make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
        }
    }
}

// ---------------------------------------------------------------- Euler update
__global__ void euler_kernel(float* __restrict__ latent, const float* __restrict__ vel, long long n, float dt) {
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (; i < n; i += stride) latent[i] = fmaf(dt, vel[i], latent[i]);
}

}  // namespace f3
