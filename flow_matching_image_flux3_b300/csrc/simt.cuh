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
// rope[r][p] = (cos, sin)(pos[r][a] * theta^(-2j/32)), p = 16 a + j.  The angle reaches
// thousands of radians, so it is formed and reduced modulo 2*pi in fp64; the reduced
// angle (|r| <= pi) is rounded to fp32 and passed to sincosf.
struct RopeFreqs {
    double f[16];  // theta^(-2j/32), j = 0..15
};

__global__ void rope_table_kernel(const int* __restrict__ pos, int n_tokens, const RopeFreqs fr, float2* __restrict__ rope) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)n_tokens * 64) return;
    const int r = (int)(i >> 6), pr = (int)(i & 63);
    const int axis = pr >> 4, j = pr & 15;
    const double two_pi = 6.283185307179586476925286766559;
    const double ang = (double)__ldg(pos + 4 * r + axis) * fr.f[j];
    const double red = fma(-rint(ang / two_pi), two_pi, ang);
    float s, c;
    sincosf((float)red, &s, &c);
    rope[i] = make_float2(c, s);
}

// ---------------------------------------------------------------- LayerNorm + modulation
// One warp per row, the row held in registers (NC chunks of 256 columns, 8 per lane),
// two-pass statistics in fp32, output a = (x - mean) * rstd * (1 + scale_s) + shift_s.
constexpr int kAdaLnMaxChunks = 16;  // D <= 4096

template <int NC>
__global__ void __launch_bounds__(256, 2) adaln_kernel(const __nv_bfloat16* __restrict__ x, int n_rows, float eps,
                                                    const float* __restrict__ mod, const SegOffsets segs,
                                                    __nv_bfloat16* __restrict__ a) {
    constexpr int D = NC * 256;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + warp;
    if (r >= n_rows) return;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * D);
    uint4 raw[NC];  // the row stays packed (bf16 is exact); each pass unpacks it
#pragma unroll
    for (int c = 0; c < NC; ++c) raw[c] = __ldg(xr + c * 32 + lane);
    auto unpack = [](const uint4& u, float (&f)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16);
            f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    };
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        float f[8];
        unpack(raw[c], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) sum += f[e];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum * (1.f / D);
    float sq = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        float f[8];
        unpack(raw[c], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float d = f[e] - mean;
            sq = fmaf(d, d, sq);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    const float rstd = rsqrtf(sq * (1.f / D) + eps);
    const int seg = segment_of_row(segs, r);
    const float* shift = mod + (size_t)seg * 3 * D;
    const float* scale = shift + D;
    uint4* ar = reinterpret_cast<uint4*>(a + (size_t)r * D);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int col = c * 256 + lane * 8;
        const float4 s0 = __ldg(reinterpret_cast<const float4*>(scale + col));
        const float4 s1 = __ldg(reinterpret_cast<const float4*>(scale + col + 4));
        const float4 h0 = __ldg(reinterpret_cast<const float4*>(shift + col));
        const float4 h1 = __ldg(reinterpret_cast<const float4*>(shift + col + 4));
        const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
        const float sh[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
        float f[8], o[8];
        unpack(raw[c], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = fmaf((f[e] - mean) * rstd, 1.f + sc[e], sh[e]);
        ar[c * 32 + lane] = make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
    }
}

template <int NC>
void launch_adaln_nc(const __nv_bfloat16* x, int n_rows, float eps, const float* mod, const SegOffsets& segs, __nv_bfloat16* a,
                     cudaStream_t st) {
    adaln_kernel<NC><<<(n_rows + 7) / 8, 256, 0, st>>>(x, n_rows, eps, mod, segs, a);
}

// dispatch on the width (a multiple of 256, at most 4096)
inline bool launch_adaln(int D, const __nv_bfloat16* x, int n_rows, float eps, const float* mod, const SegOffsets& segs,
                         __nv_bfloat16* a, cudaStream_t st) {
    switch (D / 256) {
#define F3_ADALN_CASE(n) \
    case n: launch_adaln_nc<n>(x, n_rows, eps, mod, segs, a, st); return true;
        F3_ADALN_CASE(1) F3_ADALN_CASE(2) F3_ADALN_CASE(3) F3_ADALN_CASE(4) F3_ADALN_CASE(5) F3_ADALN_CASE(6)
        F3_ADALN_CASE(7) F3_ADALN_CASE(8) F3_ADALN_CASE(9) F3_ADALN_CASE(10) F3_ADALN_CASE(11) F3_ADALN_CASE(12)
        F3_ADALN_CASE(13) F3_ADALN_CASE(14) F3_ADALN_CASE(15) F3_ADALN_CASE(16)
#undef F3_ADALN_CASE
        default: return false;
    }
}

// ---------------------------------------------------------------- Euler update
__global__ void euler_kernel(float* __restrict__ latent, const float* __restrict__ vel, long long n, float dt) {
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (; i < n; i += stride) latent[i] = fmaf(dt, vel[i], latent[i]);
}

}  // namespace f3
