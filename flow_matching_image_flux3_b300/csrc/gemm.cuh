// gemm.cuh -- persistent tcgen05 GEMM, D = A B^T, bf16 in / fp32 accumulate in TMEM,
// fed by TMA, with the block's fused epilogues:
//   EPI_QKV_SWIGLU      input projection: per-head QK RMSNorm + 4-axis RoPE -> q, k;
//                       v -> V^T; silu(gate) * up -> y[:, D:]  ("How it works":
//                       attention and SwiGLU run in parallel on the same normalized input)
//   EPI_GATED_RESIDUAL  output projection: x_out = x + gate_s * (acc + b_out)
//   EPI_F32             plain fp32 store (+ bias): the output layer
//   EPI_BF16            plain bf16 store (+ bias): the token embedders
//
// Warp roles (one CTA per SM): warp 0 issues TMA loads, warp 1 issues tcgen05.mma and
// owns the TMEM allocation (both run as converged warps with one elected lane issuing),
// warps 2.. run the epilogue, one accumulator row (TMEM lane) per thread: 4 warps, or 8
// (two per TMEM lane quarter, each taking half of a tile's columns).
// Two TMEM accumulators let the epilogue of one tile overlap the MMAs of the next.
#pragma once
#include <cuda.h>
#include "sm103.cuh"
#include "../../include/flux3.h"

namespace f3 {

constexpr int GEMM_BM = 128;
constexpr int GEMM_BK = 64;  // bf16 elements per 128-byte swizzle row
// Threads of a GEMM CTA with `ew` epilogue warps (4, or 8 for the quantized input
// projections, whose shorter mainloop no longer hides a 4-warp epilogue).
__host__ __device__ constexpr int gemm_threads(int ew) { return 64 + 32 * ew; }

enum EpiKind { EPI_QKV_SWIGLU = 0, EPI_GATED_RESIDUAL = 1, EPI_F32 = 2, EPI_BF16 = 3, EPI_PROB_T = 4, EPI_DS_T = 5 };

struct GemmGroup {
    int row_begin, row_end, tile_begin, wset;
};
struct EpiWeights {
    const float* bias;
    const float* q_norm;
    const float* k_norm;
    const float* w_scale;  // e4m3 / NVFP4 operands: scale of each weight row (output column)
    const uint8_t* w_sf;   // NVFP4 operands: the weight's tiled block scales
};

struct GemmParams {
    CUtensorMap tm_a;                      // A [rows, K]
    CUtensorMap tm_b[FLUX3_MAX_SEGMENTS];  // B per weight set [rows, K]
    EpiWeights ew[FLUX3_MAX_SEGMENTS];
    GemmGroup grp[FLUX3_MAX_SEGMENTS];
    int n_groups;
    int m_tiles, n_tiles, k_blocks;
    const float* a_scale;  // e4m3 / NVFP4 operands: scale of each A row (token)
    const uint8_t* a_sf;   // NVFP4 operands: A's tiled block scales
    int sf_steps;          // NVFP4: 64-element steps per row (K / 64)
    // EPI_QKV_SWIGLU
    int heads, width, ffn, n_tokens, ld_vt, ld_y;
    float rms_eps;
    const float* rope;
    __nv_bfloat16 *q, *k, *vt, *y;
    // EPI_GATED_RESIDUAL
    const __nv_bfloat16* x;
    __nv_bfloat16* x_out;
    const float* mod;
    int n_seg;
    int seg_off[FLUX3_MAX_SEGMENTS + 1];
    // EPI_F32 / EPI_BF16
    float* out;
    __nv_bfloat16* out_bf;
    int ld_out;
    int n_cols;  // columns of the output: a tile's columns at or past it are not stored
    // EPI_PROB_T / EPI_DS_T (attention backward, keys as rows and queries as columns)
    const float* col_vec;        // per column: the query's log2-sum-exp2 / its rowsum(dO O)
    const __nv_bfloat16* aux;    // EPI_DS_T: the probabilities P^T, row stride ld_aux
    int ld_aux;
    float alpha;                 // EPI_PROB_T: log2(e) / sqrt(d);  EPI_DS_T: 1 / sqrt(d)
};

template <int BN>
struct GemmCfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int A_BYTES = GEMM_BM * GEMM_BK * 2;
    static constexpr int B_BYTES = BN * GEMM_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
};

F3_DEV int group_of_tile(const GemmParams& p, int mt) {
    int g = 0;
#pragma unroll 1
    for (int i = 1; i < p.n_groups; ++i)
        if (mt >= p.grp[i].tile_begin) g = i;
    return g;
}

// B rows of output tile n: two 128-row boxes.  For the input projection the SwiGLU
// tiles pair gate rows (3D + 128 j ..) with up rows (3D + F + 128 j ..), so one
// accumulator holds both halves of 128 outputs.
template <int BN, int EPI>
F3_DEV void b_rows(const GemmParams& p, int n, int& r0, int& r1) {
    if (EPI == EPI_QKV_SWIGLU) {
        const int nq = 3 * p.heads / 2;
        if (n < nq) {
            r0 = 256 * n;
            r1 = r0 + 128;
        } else {
            const int j = n - nq;
            r0 = 3 * p.width + 128 * j;
            r1 = r0 + p.ffn;
        }
    } else {
        r0 = BN * n;
        r1 = r0 + 128;
    }
}

F3_DEV void unpack32(const uint32_t (&r)[32], float* v) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// --------------------------------------------------------------------- epilogues
// 32 accumulator columns of this thread's row as floats.  AK = 1 (e4m3 codes) or 2 (NVFP4
// codes, block scales already applied by the MMA): scaled by the token's and the weight
// rows' scales; then the bias (may be null).
template <int AK>
F3_DEV void acc_chunk(uint32_t taddr, float (&v)[32], float sa, const float* wsc, const float* bias) {
    uint32_t t[32];
    tmem_ld32(taddr, t);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(t[i]);
    if (AK) {
        const float4* s4 = reinterpret_cast<const float4*>(wsc);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 sw = __ldg(s4 + i);
            v[4 * i] *= sa * sw.x; v[4 * i + 1] *= sa * sw.y; v[4 * i + 2] *= sa * sw.z; v[4 * i + 3] *= sa * sw.w;
        }
    }
    if (bias) {
        const float4* b4 = reinterpret_cast<const float4*>(bias);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 b = __ldg(b4 + i);
            v[4 * i] += b.x; v[4 * i + 1] += b.y; v[4 * i + 2] += b.z; v[4 * i + 3] += b.w;
        }
    }
}

// part / nparts: this warp's share of the tile when two warps serve one lane quarter (a
// QKV tile's heads, a SwiGLU tile's 32-column chunks, interleaved).  A Q or K head is read
// from TMEM twice, 32 columns at a time: once for the RMS, once to normalise, rotate and
// store, so a thread holds 32 values rather than the whole head.
template <int AK, int NPARTS>
F3_DEV void epi_qkv(const GemmParams& p, const EpiWeights& w, int n, uint32_t tacc, int r, bool valid, int part) {
    const int nq = 3 * p.heads / 2;
    const float sa = AK ? p.a_scale[r] : 1.f;
    if (n < nq) {
#pragma unroll 1
        for (int hh = part; hh < 2; hh += NPARTS) {
            const int hg = 2 * n + hh;  // head index in Q | K | V order
            const int kind = hg / p.heads;
            const int head = hg - kind * p.heads;
            const uint32_t th = tacc + hh * 128;
            const float* wsc = AK ? w.w_scale + hg * 128 : nullptr;
            const float* bias = w.bias ? w.bias + hg * 128 : nullptr;
            if (kind < 2) {
                float ss = 0.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float v[32];
                    acc_chunk<AK>(th + c * 32, v, sa, wsc + (AK ? c * 32 : 0), bias ? bias + c * 32 : nullptr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ss = fmaf(v[i], v[i], ss);
                }
                const float inv = rsqrtf(ss * (1.f / 128.f) + p.rms_eps);
                const float4* g4 = reinterpret_cast<const float4*>(kind == 0 ? w.q_norm : w.k_norm);
                const float4* cs = reinterpret_cast<const float4*>(p.rope + (size_t)r * 128);
                __nv_bfloat16* dst = (kind == 0 ? p.q : p.k) + ((size_t)head * p.n_tokens + r) * 128;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float v[32];
                    acc_chunk<AK>(th + c * 32, v, sa, wsc + (AK ? c * 32 : 0), bias ? bias + c * 32 : nullptr);
                    if (!valid) continue;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 g = __ldg(g4 + c * 8 + i);
                        v[4 * i] *= inv * g.x; v[4 * i + 1] *= inv * g.y; v[4 * i + 2] *= inv * g.z; v[4 * i + 3] *= inv * g.w;
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {  // two pairs per float4: (cos0, sin0, cos1, sin1)
                        const float4 e = __ldg(cs + c * 8 + i);
                        const float a0 = v[4 * i], a1 = v[4 * i + 1], b0 = v[4 * i + 2], b1 = v[4 * i + 3];
                        v[4 * i] = a0 * e.x - a1 * e.y;
                        v[4 * i + 1] = a0 * e.y + a1 * e.x;
                        v[4 * i + 2] = b0 * e.z - b1 * e.w;
                        v[4 * i + 3] = b0 * e.w + b1 * e.z;
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_global_v4(dst + c * 32 + 8 * i, pack_bf16(v[8 * i], v[8 * i + 1]),
                                     pack_bf16(v[8 * i + 2], v[8 * i + 3]), pack_bf16(v[8 * i + 4], v[8 * i + 5]),
                                     pack_bf16(v[8 * i + 6], v[8 * i + 7]));
                }
            } else {
                __nv_bfloat16* dst = p.vt + (size_t)head * 128 * p.ld_vt + r;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float v[32];
                    acc_chunk<AK>(th + c * 32, v, sa, wsc + (AK ? c * 32 : 0), bias ? bias + c * 32 : nullptr);
                    if (!valid) continue;
#pragma unroll
                    for (int i = 0; i < 32; ++i) dst[(size_t)(c * 32 + i) * p.ld_vt] = __float2bfloat16_rn(v[i]);
                }
            }
        }
    } else {
        const int j = n - nq;
        __nv_bfloat16* dst = p.y + (size_t)r * p.ld_y + p.width + 128 * j;
        const float* bg = w.bias ? w.bias + 3 * p.width + 128 * j : nullptr;
        const float* bu = w.bias ? w.bias + 3 * p.width + p.ffn + 128 * j : nullptr;
        const float* sg = AK ? w.w_scale + 3 * p.width + 128 * j : nullptr;
        const float* su = AK ? sg + p.ffn : nullptr;
#pragma unroll 1
        for (int c = part; c < 4; c += NPARTS) {
            float g[32], u[32];
            acc_chunk<AK>(tacc + c * 32, g, sa, AK ? sg + c * 32 : nullptr, bg ? bg + c * 32 : nullptr);
            acc_chunk<AK>(tacc + 128 + c * 32, u, sa, AK ? su + c * 32 : nullptr, bu ? bu + c * 32 : nullptr);
            if (!valid) continue;
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a0 = g[2 * i] / (1.f + __expf(-g[2 * i])) * u[2 * i];
                const float a1 = g[2 * i + 1] / (1.f + __expf(-g[2 * i + 1])) * u[2 * i + 1];
                o[i] = pack_bf16(a0, a1);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) st_global_v4(dst + c * 32 + 8 * i, o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
    }
}

// AK != 0: the operands were quantized codes; the accumulator is scaled by the token's
// and the weight rows' scales first.
template <int BN, int AK>
F3_DEV void epi_gated_residual(const GemmParams& p, const EpiWeights& w, int n, uint32_t tacc, int r, bool valid) {
    const float sa = AK ? p.a_scale[r] : 1.f;
    int seg = 0;
#pragma unroll 1
    for (int s = 1; s < p.n_seg; ++s)
        if (r >= p.seg_off[s]) seg = s;
    const int D = p.width;
    const float* gate = p.mod + ((size_t)seg * 3 + 2) * D;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t t[32];
        tmem_ld32(tacc + c * 32, t);
        tmem_ld_wait();
        if (!valid) continue;
        const int col = n * BN + c * 32;
        float a[32];
        unpack32(t, a);
        if (AK) {
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] *= sa * __ldg(w.w_scale + col + i);
        }
        if (w.bias) {
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] += __ldg(w.bias + col + i);
        }
        const uint4* xs = reinterpret_cast<const uint4*>(p.x + (size_t)r * D + col);
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 xv = *(xs + i);  // x may alias x_out: plain (coherent) load
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&xw[e]);
                const int k = 8 * i + 2 * e;
                const float g0 = __ldg(gate + col + k), g1 = __ldg(gate + col + k + 1);
                o[4 * i + e] = pack_bf16(fmaf(g0, a[k], __bfloat162float(h.x)), fmaf(g1, a[k + 1], __bfloat162float(h.y)));
            }
        }
        __nv_bfloat16* dst = p.x_out + (size_t)r * D + col;
#pragma unroll
        for (int i = 0; i < 4; ++i) st_global_v4(dst + 8 * i, o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
}

template <int BN>
F3_DEV void epi_f32(const GemmParams& p, const EpiWeights& w, int n, uint32_t tacc, int r, bool valid) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t t[32];
        tmem_ld32(tacc + c * 32, t);
        tmem_ld_wait();
        const int col = n * BN + c * 32;
        if (!valid || col >= p.n_cols) continue;
        float a[32];
        unpack32(t, a);
        float* dst = p.out + (size_t)r * p.ld_out + col;
        if (col + 32 <= p.n_cols) {
            if (w.bias) {
#pragma unroll
                for (int i = 0; i < 32; ++i) a[i] += __ldg(w.bias + col + i);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                st_global_v4(dst + 4 * i, __float_as_uint(a[4 * i]), __float_as_uint(a[4 * i + 1]),
                             __float_as_uint(a[4 * i + 2]), __float_as_uint(a[4 * i + 3]));
        } else {  // the ragged last columns
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (col + i < p.n_cols) dst[i] = a[i] + (w.bias ? __ldg(w.bias + col + i) : 0.f);
        }
    }
}

template <int BN>
F3_DEV void epi_bf16(const GemmParams& p, const EpiWeights& w, int n, uint32_t tacc, int r, bool valid) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t t[32];
        tmem_ld32(tacc + c * 32, t);
        tmem_ld_wait();
        const int col = n * BN + c * 32;
        if (!valid || col >= p.n_cols) continue;
        float a[32];
        unpack32(t, a);
        __nv_bfloat16* dst = p.out_bf + (size_t)r * p.ld_out + col;
        if (col + 32 <= p.n_cols) {
            if (w.bias) {
#pragma unroll
                for (int i = 0; i < 32; ++i) a[i] += __ldg(w.bias + col + i);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                st_global_v4(dst + 8 * i, pack_bf16(a[8 * i], a[8 * i + 1]), pack_bf16(a[8 * i + 2], a[8 * i + 3]),
                             pack_bf16(a[8 * i + 4], a[8 * i + 5]), pack_bf16(a[8 * i + 6], a[8 * i + 7]));
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (col + i < p.n_cols) dst[i] = __float2bfloat16_rn(a[i] + (w.bias ? __ldg(w.bias + col + i) : 0.f));
        }
    }
}

// Attention backward with keys as rows and queries as columns.  EPI_PROB_T: the
// accumulator is k q^T; P^T = exp2(alpha acc - lse[query]) in bf16.  EPI_DS_T: the
// accumulator is v dO^T = dP^T; dS^T = alpha P^T (acc - delta[query]) in bf16.
template <int BN, int EPI, int NPARTS>
F3_DEV void epi_attn_t(const GemmParams& p, int n, uint32_t tacc, int r, bool valid, int part) {
#pragma unroll 1
    for (int c = part; c < BN / 32; c += NPARTS) {
        uint32_t t[32];
        tmem_ld32(tacc + c * 32, t);
        tmem_ld_wait();
        const int col = n * BN + c * 32;
        if (!valid || col >= p.n_cols) continue;
        float a[32];
        unpack32(t, a);
        const int lim = p.n_cols - col < 32 ? p.n_cols - col : 32;
        if (EPI == EPI_PROB_T) {
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = i < lim ? exp2f(p.alpha * a[i] - __ldg(p.col_vec + col + i)) : 0.f;
        } else {
            const uint4* pa = reinterpret_cast<const uint4*>(p.aux + (size_t)r * p.ld_aux + col);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = v * 8 < lim ? pa[v] : make_uint4(0, 0, 0, 0);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 8 * v + 2 * e;
                    const float p0 = __uint_as_float(w4[e] << 16), p1 = __uint_as_float(w4[e] & 0xffff0000u);
                    a[i] = i < lim ? p.alpha * p0 * (a[i] - __ldg(p.col_vec + col + i)) : 0.f;
                    a[i + 1] = i + 1 < lim ? p.alpha * p1 * (a[i + 1] - __ldg(p.col_vec + col + i + 1)) : 0.f;
                }
            }
        }
        __nv_bfloat16* dst = p.out_bf + (size_t)r * p.ld_out + col;
        if (lim == 32) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                st_global_v4(dst + 8 * i, pack_bf16(a[8 * i], a[8 * i + 1]), pack_bf16(a[8 * i + 2], a[8 * i + 3]),
                             pack_bf16(a[8 * i + 4], a[8 * i + 5]), pack_bf16(a[8 * i + 6], a[8 * i + 7]));
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < lim) dst[i] = __float2bfloat16_rn(a[i]);
        }
    }
}

// --------------------------------------------------------------------- the kernel
// Tiles are numbered n-major (all m-tiles of one weight tile run together, so each weight
// tile is read from HBM once).  With CL = 2 the kernel runs as clusters of two CTAs that
// take adjacent m-tiles of the same weight tile: each CTA loads its own A tile and one
// 128-row half of the shared B tile, multicast into both CTAs' shared memory, which cuts
// each SM's L2 reads per k-block from 48 KB to 32 KB.  A stage is free only when both CTAs'
// MMAs have read it: every MMA commit arrives on the slot barrier of both CTAs.  Groups of
// the grouped GEMM then start on an even m-tile, so a pair never straddles two weight sets.
// Tasks run n-major: all m-tiles of one weight tile together, so each weight tile is read
// from HBM once (the A operand, re-read by every weight tile, is served from L2).  The ~17
// clusters that share a weight tile run in near lockstep, so each walks the K dimension
// from its own starting k-block (spread by m index): a weight k-block's first read from
// DRAM stalls one cluster rather than all of them.  (An m-major order for the output
// projection, whose A operand Y is larger than its weight, cut its DRAM reads from 447 to
// 368 MB per launch but ran 2-3% slower.)
struct TileInfo {
    int n, g, row0, kb0;
};
F3_DEV TileInfo tile_info(const GemmParams& p, int task, int rank, int cl) {
    const int m_units = p.m_tiles / cl;
    const int n = task / m_units;
    const int mu = task - n * m_units;
    const int mt = mu * cl + rank;
    const int g = group_of_tile(p, mt);
    return {n, g, p.grp[g].row_begin + (mt - p.grp[g].tile_begin) * GEMM_BM, (int)((long long)mu * p.k_blocks / m_units)};
}

// AK: operand kind, 0 = bf16 (64 elements per 128-byte row of a k-block), 1 = e4m3 (128).
// EW: epilogue warps (4, or 8 for the input projection).
template <int BN, int EPI, int CL, int AK = 0, int EW = 4>
__global__ void __launch_bounds__(gemm_threads(EW), 1) gemm_tcgen05_kernel(const __grid_constant__ GemmParams p) {
    static_assert(CL == 1 || (CL == 2 && BN == 256), "clusters of two split a 256-row B tile");
    static_assert(AK == 0 || EPI == EPI_QKV_SWIGLU || EPI == EPI_GATED_RESIDUAL, "e4m3 operands: the projections");
    static_assert(EW == 4 || (EW == 8 && (EPI == EPI_QKV_SWIGLU || EPI == EPI_PROB_T || EPI == EPI_DS_T)),
                  "8 epilogue warps: the input projection and the attention-backward epilogues");
    constexpr int KB_ELEMS = AK ? 128 : GEMM_BK;
    using C = GemmCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * C::STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 4);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const uint32_t smem_base = smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = CL == 2 ? (int)cluster_ctarank() : 0;
    const int unit = blockIdx.x / CL, n_units = gridDim.x / CL;  // cluster index and count
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), CL);  // one MMA commit from each CTA of the cluster
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EW);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_a);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    if (CL > 1) cluster_sync();  // the peer's barriers exist before any multicast reaches them
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int tasks = (p.m_tiles / CL) * p.n_tiles;
    constexpr uint16_t kPair = 0x3;

    if (warp == 0) {
        // ---------------- TMA producer (converged warp, one elected lane issues)
        const bool leader = elect_one();
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        bool ok = true;
        for (int task = unit; task < tasks && ok; task += n_units) {
            const TileInfo ti = tile_info(p, task, rank, CL);
            const CUtensorMap* tb = &p.tm_b[p.grp[ti.g].wset];
            int r0, r1;
            b_rows<BN, EPI>(p, ti.n, r0, r1);
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!mbar_wait_warp(empty_bar(s), ph ^ 1u, abort_flag)) { ok = false; break; }
                if (leader) {
                    const uint32_t sa = smem_base + s * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_BYTES;
                    int kr = ti.kb0 + kb;
                    if (kr >= p.k_blocks) kr -= p.k_blocks;
                    const int kc = kr * KB_ELEMS;
                    mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
                    tma_load_2d(sa, &p.tm_a, full_bar(s), kc, ti.row0);
                    if (CL == 2) {
                        tma_load_2d_multicast(sb + rank * 128 * 128, tb, full_bar(s), kc, rank ? r1 : r0, kPair);
                    } else {
                        tma_load_2d(sb, tb, full_bar(s), kc, r0);
                        if (BN == 256) tma_load_2d(sb + 128 * 128, tb, full_bar(s), kc, r1);
                    }
                }
                __syncwarp();
                ++issued;
                if (++s == C::STAGES) { s = 0; ph ^= 1u; }
            }
        }
        if (!ok && leader) {
            // let the copies already in flight land before the CTA exits
            int back = issued < C::STAGES ? issued : C::STAGES;
            int ss = s;
            uint32_t pp = ph;
            for (int i = 0; i < back; ++i) {
                if (--ss < 0) { ss = C::STAGES - 1; pp ^= 1u; }
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(full_bar(ss), pp) && globaltimer() - t0 < kWaitTimeoutNs) {}
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (converged warp, one elected lane issues)
        const bool leader = elect_one();
        constexpr uint32_t IDESC = AK ? idesc_e4m3_f32(GEMM_BM, BN) : idesc_bf16_f32(GEMM_BM, BN);
        int s = 0;
        uint32_t ph = 0;
        int acc = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int task = unit; task < tasks && ok; task += n_units) {
            if (!mbar_wait_warp(tempty_bar(acc), aph ^ 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem_base + acc * BN;
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!mbar_wait_warp(full_bar(s), ph, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_base + s * C::STAGE_BYTES;
                const uint64_t ad = sdesc_kmajor_sw128(sa);
                const uint64_t bd = sdesc_kmajor_sw128(sa + C::A_BYTES);
#pragma unroll
                for (int k = 0; k < 4; ++k) {  // 32 bytes of each row per instruction
                    if (AK) mma_e4m3_ss_if(leader, d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), IDESC, (kb | k) != 0);
                    else mma_bf16_ss_if(leader, d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), IDESC, (kb | k) != 0);
                }
                if (CL == 2) mma_commit_multicast_if(leader, empty_bar(s), kPair);
                else mma_commit_if(leader, empty_bar(s));
                if (++s == C::STAGES) { s = 0; ph ^= 1u; }
            }
            if (!ok) break;
            mma_commit_if(leader, tfull_bar(acc));
            if (++acc == 2) { acc = 0; aph ^= 1u; }
        }
        // all issued MMAs retire before TMEM is released
        if (leader) {
            mma_commit(drain_bar);
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < kWaitTimeoutNs) {}
        }
        __syncwarp();
    } else {
        // ---------------- epilogue warps 2 .. 2 + EW - 1
        const int sub = warp & 3;  // TMEM lane quarter this warp may access
        const int part = (warp - 2) >> 2;
        int acc = 0;
        uint32_t aph = 0;
        for (int task = unit; task < tasks; task += n_units) {
            const TileInfo ti = tile_info(p, task, rank, CL);
            const int r = ti.row0 + sub * 32 + lane;
            const bool valid = r < p.grp[ti.g].row_end;
            if (!mbar_wait_warp(tfull_bar(acc), aph, abort_flag)) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(sub * 32) << 16) + acc * BN;
            const EpiWeights& w = p.ew[p.grp[ti.g].wset];
            if (EPI == EPI_QKV_SWIGLU) epi_qkv<AK, EW / 4>(p, w, ti.n, tacc, valid ? r : 0, valid, part);
            else if (EPI == EPI_GATED_RESIDUAL) epi_gated_residual<BN, AK>(p, w, ti.n, tacc, valid ? r : 0, valid);
            else if (EPI == EPI_F32) epi_f32<BN>(p, w, ti.n, tacc, valid ? r : 0, valid);
            else if (EPI == EPI_BF16) epi_bf16<BN>(p, w, ti.n, tacc, valid ? r : 0, valid);
            else epi_attn_t<BN, EPI, EW / 4>(p, ti.n, tacc, valid ? r : 0, valid, part);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (++acc == 2) { acc = 0; aph ^= 1u; }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    if (CL > 1) cluster_sync();  // no CTA leaves while its peer may still signal it
}

}  // namespace f3
