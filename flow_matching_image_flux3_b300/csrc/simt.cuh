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
// thousands of radians, so it is reduced in turns without fp64 (slow on this part): the
// frequency in turns, g_j = theta^(-2j/32) / (2 pi), is a pair of floats hi + lo (fitted
// in fp64 on the host); pos * hi is split exactly into its rounded product and the fma
// error, the whole turns are dropped exactly, and the fraction f in [-1/2, 1/2] (rounding
// error <= 2^-25 turns) gives (cos, sin)(2 pi f) through sincospif.
struct RopeFreqs {
    float hi[16], lo[16];  // theta^(-2j/32) / (2 pi) = hi + lo, j = 0..15
};

__global__ void rope_table_kernel(const int* __restrict__ pos, int n_tokens, const RopeFreqs fr, float2* __restrict__ rope) {
    // the lanes of a warp index 16 different frequencies: read them from shared memory
    // (a per-lane index into the parameter bank would serialise)
    __shared__ float s_hi[16], s_lo[16];
    if (threadIdx.x < 16) {
        s_hi[threadIdx.x] = fr.hi[threadIdx.x];
        s_lo[threadIdx.x] = fr.lo[threadIdx.x];
    }
    __syncthreads();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)n_tokens * 64) return;
    const int r = (int)(i >> 6), pr = (int)(i & 63);
    const int axis = pr >> 4, j = pr & 15;
    const float ps = (float)__ldg(pos + 4 * r + axis);  // |pos| < 2^24: exact
    const float hi = s_hi[j], lo = s_lo[j];
    const float prod = ps * hi;
    const float err = fmaf(ps, hi, -prod);               // prod + err == ps * hi exactly
    const float f = (prod - rintf(prod)) + (err + ps * lo);
    float s, c;
    sincospif(2.f * f, &s, &c);
    rope[i] = make_float2(c, s);
}

// ---------------------------------------------------------------- LayerNorm + modulation
// One warp per row, output a = (x - mean) * rstd * (1 + scale_s) + shift_s.  The
// statistics take one pass over the row as sums of (x - c) and (x - c)^2 with c the row's
// first element (so the variance does not cancel catastrophically when the mean is far
// from zero); the output pass reads the row again, from L1/L2 (HBM sees each row once).
// Nothing of the row stays in registers, so 32 warps fit on an SM and a 4,256-row call has
// every row in flight in one wave.  A block's 8 rows nearly always share one segment: its
// shift and scale vectors are then staged once in shared memory (instead of every warp
// streaming 2 D floats through L1 per row).
constexpr int kAdaLnMaxChunks = 16;  // D <= 4096

F3_DEV void unpack_bf16x8(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}

template <int NC>
__global__ void __launch_bounds__(256, 4) adaln_kernel(const __nv_bfloat16* __restrict__ x, int n_rows, float eps,
                                                    const float* __restrict__ mod, const __grid_constant__ SegOffsets segs,
                                                    __nv_bfloat16* __restrict__ a) {
    constexpr int D = NC * 256;
    __shared__ __align__(16) float s_mod[2 * D];  // shift | scale of the block's segment
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r_first = blockIdx.x * 8;
    const int r_last = min(r_first + 7, n_rows - 1);
    const int seg_first = segment_of_row(segs, r_first);
    const bool staged = segment_of_row(segs, r_last) == seg_first;  // uniform over the block
    if (staged) {
        const float4* src = reinterpret_cast<const float4*>(mod + (size_t)seg_first * 3 * D);
        for (int i = threadIdx.x; i < 2 * D / 4; i += blockDim.x) reinterpret_cast<float4*>(s_mod)[i] = __ldg(src + i);
        __syncthreads();
    }
    const int r = r_first + warp;
    if (r >= n_rows) return;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * D);
    const float c0 = __bfloat162float(x[(size_t)r * D]);
    float sum = 0.f, sq = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        float f[8];
        unpack_bf16x8(__ldg(xr + c * 32 + lane), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float d = f[e] - c0;
            sum += d;
            sq = fmaf(d, d, sq);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    const float md = sum * (1.f / D);
    const float mean = c0 + md;
    const float rstd = rsqrtf(fmaxf(sq * (1.f / D) - md * md, 0.f) + eps);
    const float* shift = staged ? s_mod : mod + (size_t)segment_of_row(segs, r) * 3 * D;
    const float* scale = shift + D;
    uint4* ar = reinterpret_cast<uint4*>(a + (size_t)r * D);
#pragma unroll 2
    for (int c = 0; c < NC; ++c) {
        const int col = c * 256 + lane * 8;
        const float4 s0 = *reinterpret_cast<const float4*>(scale + col);
        const float4 s1 = *reinterpret_cast<const float4*>(scale + col + 4);
        const float4 h0 = *reinterpret_cast<const float4*>(shift + col);
        const float4 h1 = *reinterpret_cast<const float4*>(shift + col + 4);
        float f[8];
        unpack_bf16x8(__ldg(xr + c * 32 + lane), f);
        auto mo = [&](float v, float sc, float sh) { return fmaf((v - mean) * rstd, 1.f + sc, sh); };
        ar[c * 32 + lane] = make_uint4(pack_bf16(mo(f[0], s0.x, h0.x), mo(f[1], s0.y, h0.y)),
                                       pack_bf16(mo(f[2], s0.z, h0.z), mo(f[3], s0.w, h0.w)),
                                       pack_bf16(mo(f[4], s1.x, h1.x), mo(f[5], s1.y, h1.y)),
                                       pack_bf16(mo(f[6], s1.z, h1.z), mo(f[7], s1.w, h1.w)));
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
