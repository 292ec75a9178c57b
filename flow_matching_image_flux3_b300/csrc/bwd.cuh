// bwd.cuh -- the element-wise and reduction steps of the joint block's backward pass (the
// chain rule of "How it works" in "Welcome FLUX.3 Image Klein in Diffusers"; the Miles
// page, section 1, fine-tunes the base checkpoint).  The contractions around them run on
// the tcgen05 GEMM (gemm.cuh); these kernels are HBM-bound SIMT passes.
//
// Segment-wise column sums (the modulation vectors' gradients, the biases') accumulate per
// CTA over a run of rows and add into the fp32 outputs with one atomic per column per
// segment the run touches, so the outputs must be zeroed first.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>
#include "simt.cuh"

namespace f3 {

constexpr int BWD_ROWS = 32;  // rows per CTA of the column-sum kernels

// dst[c][r] = src[r][c] for a bf16 [rows, cols] matrix (row strides in elements, even,
// both bases 4-byte aligned): 64 x 64 tiles through shared memory, block (32, 8), each
// thread reading two adjacent columns and writing two adjacent rows (bf16 pairs); a ragged
// edge falls back to single elements.  The tile's row stride of 65 keeps both phases free
// of bank conflicts.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const __nv_bfloat16* __restrict__ src, int rows, int cols,
                                                            int ld_src, __nv_bfloat16* __restrict__ dst, int ld_dst) {
    __shared__ __nv_bfloat16 tile[64][65];
    const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
    const int c = c0 + 2 * threadIdx.x;
    for (int i = threadIdx.y; i < 64; i += 8) {
        const int r = r0 + i;
        __nv_bfloat16 e0 = __float2bfloat16_rn(0.f), e1 = e0;
        if (r < rows) {
            const __nv_bfloat16* sp = src + (size_t)r * ld_src + c;
            if (c + 1 < cols) {
                const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(sp);
                e0 = v.x;
                e1 = v.y;
            } else if (c < cols) {
                e0 = sp[0];
            }
        }
        tile[i][2 * threadIdx.x] = e0;
        tile[i][2 * threadIdx.x + 1] = e1;
    }
    __syncthreads();
    const int r = r0 + 2 * threadIdx.x;
    for (int i = threadIdx.y; i < 64; i += 8) {
        const int cc = c0 + i;
        if (cc >= cols) continue;
        __nv_bfloat16* dp = dst + (size_t)cc * ld_dst + r;
        if (r + 1 < rows) {
            __nv_bfloat162 v;
            v.x = tile[2 * threadIdx.x][i];
            v.y = tile[2 * threadIdx.x + 1][i];
            *reinterpret_cast<__nv_bfloat162*>(dp) = v;
        } else if (r < rows) {
            dp[0] = tile[2 * threadIdx.x][i];
        }
    }
}

// x' = x + gate_s y:  dy = gate_s dxo (bf16, the next GEMM's operand), and per column the
// sums dgate_s += dxo * y over the rows of stream s and db_out += dy over all rows.
// grid (ceil(N / BWD_ROWS), D / 256), block 256; mod [n_seg][3][D].
__global__ void __launch_bounds__(256) bwd_gate_kernel(const float* __restrict__ dxo, const float* __restrict__ y, int N,
                                                      int D, const float* __restrict__ mod, const __grid_constant__ SegOffsets segs,
                                                      __nv_bfloat16* __restrict__ dy, float* __restrict__ dmod,
                                                      float* __restrict__ db_out) {
    const int col = blockIdx.y * 256 + threadIdx.x;
    const int r0 = blockIdx.x * BWD_ROWS, r1 = min(N, r0 + BWD_ROWS);
    int seg = 0;
    while (seg + 1 < segs.n_seg && r0 >= segs.off[seg + 1]) ++seg;
    float acc_g = 0.f, acc_b = 0.f;
    for (int r = r0; r < r1; ++r) {
        while (r >= segs.off[seg + 1]) {  // the run crosses into the next stream
            atomicAdd(dmod + ((size_t)seg * 3 + 2) * D + col, acc_g);
            acc_g = 0.f;
            ++seg;
        }
        const size_t i = (size_t)r * D + col;
        const float g = mod[((size_t)seg * 3 + 2) * D + col];
        const float v = dxo[i];
        const float d = g * v;
        dy[i] = __float2bfloat16_rn(d);
        acc_g = fmaf(v, y[i], acc_g);
        acc_b += d;
    }
    atomicAdd(dmod + ((size_t)seg * 3 + 2) * D + col, acc_g);
    atomicAdd(db_out + col, acc_b);
}

// act = silu(G) U:  dG = dact U silu'(G), dU = dact silu(G), silu'(g) = s (1 + g (1 - s)),
// s = sigmoid(g).  dycat [N, D + F] (dact = columns D..), p [N, 3D + 2F] (G, U = columns
// 3D.., 3D + F..), dp the same layout as p.
__global__ void bwd_swiglu_kernel(const __nv_bfloat16* __restrict__ dycat, const __nv_bfloat16* __restrict__ p, int N,
                                  int D, int F, __nv_bfloat16* __restrict__ dp) {
    const long long total = (long long)N * F;
    const int ldy = D + F, ldp = 3 * D + 2 * F;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(e / F), j = (int)(e - (long long)r * F);
        const float g = __bfloat162float(p[(size_t)r * ldp + 3 * D + j]);
        const float u = __bfloat162float(p[(size_t)r * ldp + 3 * D + F + j]);
        const float da = __bfloat162float(dycat[(size_t)r * ldy + D + j]);
        const float sg = 1.f / (1.f + __expf(-g));
        dp[(size_t)r * ldp + 3 * D + j] = __float2bfloat16_rn(da * u * sg * (1.f + g * (1.f - sg)));
        dp[(size_t)r * ldp + 3 * D + F + j] = __float2bfloat16_rn(da * g * sg);
    }
}

// delta[h][r] = sum_d dO[r][h * 128 + d] O[r][h * 128 + d]: one warp per (row, head), four
// dims per lane.  d_o, o bf16 [N, ld] (the attention columns of d[O | act] and [O | act]).
__global__ void __launch_bounds__(256) attn_delta_kernel(const __nv_bfloat16* __restrict__ d_o,
                                                        const __nv_bfloat16* __restrict__ o, int ld, int N, int H,
                                                        float* __restrict__ delta) {
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < N * H; item += warps) {
        const int r = item / H, h = item - r * H;
        const size_t base = (size_t)r * ld + h * 128 + 4 * lane;
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc = fmaf(__bfloat162float(d_o[base + i]), __bfloat162float(o[base + i]), acc);
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) delta[(size_t)h * N + r] = acc;
    }
}

// The QK-norm + RoPE backward and the V columns: for every (row, head), one warp, each lane
// 4 consecutive dims (two rotation pairs):
//   dn = R(-theta) dq                     (the transpose of the rotation)
//   dP = r (dn g) - P r^3 sum(dn g P) / 128,  r = (mean(P^2) + eps)^(-1/2)   (RMSNorm)
//   dg += dn P r                           (summed over rows and heads)
// q and k alike; dv is copied.  dq, dk, dv fp32 [N, D]; p bf16 [N, 3D + 2F] (the projection
// before normalisation); rope [N][64] (cos, sin); dp bf16, the same layout as p.
__global__ void __launch_bounds__(256) bwd_qk_kernel(const float* __restrict__ dq, const float* __restrict__ dk,
                                                    const float* __restrict__ dv, const __nv_bfloat16* __restrict__ p,
                                                    const float2* __restrict__ rope, const float* __restrict__ gq,
                                                    const float* __restrict__ gk, float eps, int N, int H, int D, int F,
                                                    __nv_bfloat16* __restrict__ dp, float* __restrict__ dgq,
                                                    float* __restrict__ dgk) {
    const int lane = threadIdx.x & 31;
    const int ldp = 3 * D + 2 * F;
    const int warps = gridDim.x * (blockDim.x >> 5);
    float accq[4] = {0.f, 0.f, 0.f, 0.f}, acck[4] = {0.f, 0.f, 0.f, 0.f};
    float g4q[4], g4k[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        g4q[i] = gq[4 * lane + i];
        g4k[i] = gk[4 * lane + i];
    }
    for (int item = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < N * H; item += warps) {
        const int r = item / H, h = item - r * H;
        const float2 cs0 = rope[(size_t)r * 64 + 2 * lane], cs1 = rope[(size_t)r * 64 + 2 * lane + 1];
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const float* src = (which == 0 ? dq : dk) + (size_t)r * D + h * 128 + 4 * lane;
            const float4 d4 = *reinterpret_cast<const float4*>(src);
            // transpose of [[c, -s], [s, c]] on (d0, d1)
            float dn[4] = {d4.x * cs0.x + d4.y * cs0.y, -d4.x * cs0.y + d4.y * cs0.x, d4.z * cs1.x + d4.w * cs1.y,
                           -d4.z * cs1.y + d4.w * cs1.x};
            const __nv_bfloat16* pp = p + (size_t)r * ldp + which * D + h * 128 + 4 * lane;
            float pv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pv[i] = __bfloat162float(pp[i]);
            const float* g = which == 0 ? g4q : g4k;
            float ss = 0.f, sd = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ss = fmaf(pv[i], pv[i], ss);
                sd = fmaf(dn[i] * g[i], pv[i], sd);
            }
            for (int o = 16; o > 0; o >>= 1) {
                ss += __shfl_xor_sync(0xffffffffu, ss, o);
                sd += __shfl_xor_sync(0xffffffffu, sd, o);
            }
            const float rr = rsqrtf(ss * (1.f / 128.f) + eps);
            const float c3 = rr * rr * rr * sd * (1.f / 128.f);
            __nv_bfloat16* out = dp + (size_t)r * ldp + which * D + h * 128 + 4 * lane;
            float* acc = which == 0 ? accq : acck;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                out[i] = __float2bfloat16_rn(rr * dn[i] * g[i] - pv[i] * c3);
                acc[i] = fmaf(dn[i] * pv[i], rr, acc[i]);
            }
        }
        const float4 v4 = *reinterpret_cast<const float4*>(dv + (size_t)r * D + h * 128 + 4 * lane);
        __nv_bfloat16* ov = dp + (size_t)r * ldp + 2 * D + h * 128 + 4 * lane;
        ov[0] = __float2bfloat16_rn(v4.x);
        ov[1] = __float2bfloat16_rn(v4.y);
        ov[2] = __float2bfloat16_rn(v4.z);
        ov[3] = __float2bfloat16_rn(v4.w);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        atomicAdd(dgq + 4 * lane + i, accq[i]);
        atomicAdd(dgk + 4 * lane + i, acck[i]);
    }
}

// out[c] += sum over rows of a bf16 [rows, cols] matrix (row stride ld).  grid
// (ceil(cols / 256), ceil(rows / 64)), block 256.
__global__ void __launch_bounds__(256) colsum_bf16_kernel(const __nv_bfloat16* __restrict__ m, int rows, int cols, int ld,
                                                         float* __restrict__ out) {
    const int c = blockIdx.x * 256 + threadIdx.x;
    if (c >= cols) return;
    const int r0 = blockIdx.y * 64, r1 = min(rows, r0 + 64);
    float acc = 0.f;
    for (int r = r0; r < r1; ++r) acc += __bfloat162float(m[(size_t)r * ld + c]);
    atomicAdd(out + c, acc);
}

// LayerNorm + modulation backward, one warp per row:
//   dln = da (1 + scale_s),  dx = dxo + rstd (dln - mean(dln) - ln mean(dln ln))
// and the row's mean and rstd for the modulation sums.  x bf16 [N, D]; da, dxo, dx fp32.
__global__ void __launch_bounds__(256) bwd_ln_kernel(const float* __restrict__ da, const __nv_bfloat16* __restrict__ x,
                                                    const float* __restrict__ dxo, const float* __restrict__ mod,
                                                    const __grid_constant__ SegOffsets segs, float eps, int N, int D,
                                                    float* __restrict__ dx, float2* __restrict__ stats) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= N) return;
    int seg = 0;
    while (seg + 1 < segs.n_seg && r >= segs.off[seg + 1]) ++seg;
    const __nv_bfloat16* xr = x + (size_t)r * D;
    const float x0 = __bfloat162float(xr[0]);
    float s1 = 0.f, s2 = 0.f;
    for (int j = lane; j < D; j += 32) {
        const float t = __bfloat162float(xr[j]) - x0;
        s1 += t;
        s2 = fmaf(t, t, s2);
    }
    for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    const float mt = s1 / D;
    const float mu = x0 + mt;
    const float rstd = rsqrtf(fmaxf(s2 / D - mt * mt, 0.f) + eps);
    const float* scale = mod + ((size_t)seg * 3 + 1) * D;
    const float* dar = da + (size_t)r * D;
    float a1 = 0.f, a2 = 0.f;
    for (int j = lane; j < D; j += 32) {
        const float dl = dar[j] * (1.f + scale[j]);
        const float ln = (__bfloat162float(xr[j]) - mu) * rstd;
        a1 += dl;
        a2 = fmaf(dl, ln, a2);
    }
    for (int o = 16; o > 0; o >>= 1) {
        a1 += __shfl_xor_sync(0xffffffffu, a1, o);
        a2 += __shfl_xor_sync(0xffffffffu, a2, o);
    }
    const float m1 = a1 / D, m2 = a2 / D;
    for (int j = lane; j < D; j += 32) {
        const float dl = dar[j] * (1.f + scale[j]);
        const float ln = (__bfloat162float(xr[j]) - mu) * rstd;
        dx[(size_t)r * D + j] = dxo[(size_t)r * D + j] + rstd * (dl - m1 - ln * m2);
    }
    if (lane == 0) stats[r] = make_float2(mu, rstd);
}

// The modulation's shift and scale gradients: per column, dshift_s += da and dscale_s +=
// da ln over the rows of stream s (ln from the row statistics).  Launch as bwd_gate_kernel.
__global__ void __launch_bounds__(256) bwd_mod_kernel(const float* __restrict__ da, const __nv_bfloat16* __restrict__ x,
                                                     const float2* __restrict__ stats, int N, int D,
                                                     const __grid_constant__ SegOffsets segs, float* __restrict__ dmod) {
    const int col = blockIdx.y * 256 + threadIdx.x;
    const int r0 = blockIdx.x * BWD_ROWS, r1 = min(N, r0 + BWD_ROWS);
    int seg = 0;
    while (seg + 1 < segs.n_seg && r0 >= segs.off[seg + 1]) ++seg;
    float a0 = 0.f, a1 = 0.f;
    for (int r = r0; r < r1; ++r) {
        while (r >= segs.off[seg + 1]) {
            atomicAdd(dmod + ((size_t)seg * 3 + 0) * D + col, a0);
            atomicAdd(dmod + ((size_t)seg * 3 + 1) * D + col, a1);
            a0 = a1 = 0.f;
            ++seg;
        }
        const size_t i = (size_t)r * D + col;
        const float2 st = stats[r];
        const float v = da[i];
        a0 += v;
        a1 = fmaf(v, (__bfloat162float(x[i]) - st.x) * st.y, a1);
    }
    atomicAdd(dmod + ((size_t)seg * 3 + 0) * D + col, a0);
    atomicAdd(dmod + ((size_t)seg * 3 + 1) * D + col, a1);
}

}  // namespace f3
