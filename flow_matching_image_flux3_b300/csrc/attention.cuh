// attention.cuh -- flash attention for the block: softmax(q k^T / sqrt(128)) v per head,
// bidirectional, no padding mask, optionally restricted to the query's own segment
// ("How it works": stage 1 attends within each stream, stage 2 over all tokens, and the
// text padding is attended).
//
// One CTA per (pair of 128-query tiles, head); both query tiles share every K and V^T
// tile the TMA warp streams into a 4-slot ring.  Warp roles (320 threads):
//   warps 0-3  softmax of query tile 0, warps 4-7 softmax of query tile 1: one query row
//              per thread (TMEM lane), online softmax in the log2 domain;
//   warp 8     TMA producer (Q tiles once, then K_0, V_0, K_1, V_1, ...);
//   warp 9     tcgen05.mma issuer and owner of the 512 TMEM columns.
// TMEM: S_t (tile t's 128 x 128 fp32 scores) at columns 128 t, O_t at 256 + 128 t.  The
// softmax writes P_t as bf16 pairs over the first 64 columns of S_t and the P V MMA
// reads its A operand from there (no shared-memory round trip for P).  The MMA order is
//   O_0 += P_0 V_j, S_0 = Q_0 K_{j+1}^T, O_1 += P_1 V_j, S_1 = Q_1 K_{j+1}^T,
// so while one warpgroup runs its softmax the tensor core works on the other tile.  A
// row keeps a stale running max until the new one exceeds it by 8 (probabilities stay
// below 2^8), so O is rescaled in TMEM only on those rare tiles.
#pragma once
#include <cuda.h>
#include "sm103.cuh"
#include "../../include/flux3.h"

namespace f3 {

constexpr int ATT_THREADS = 320;
constexpr int ATT_SLOTS = 4;
constexpr int ATT_TILE_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 operand tile
constexpr int ATT_SMEM_BYTES = 1024 + (2 + ATT_SLOTS) * ATT_TILE_BYTES + 256;
constexpr float ATT_RESCALE_LOG2 = 8.f;        // stale-max slack, log2 units

struct AttnParams {
    CUtensorMap tm_q, tm_k, tm_v;
    int n_tokens, heads, n_seg;
    int seg_off[FLUX3_MAX_SEGMENTS + 1];
    int pair_begin[FLUX3_MAX_SEGMENTS + 1];  // first query-tile pair of each segment
    __nv_bfloat16* out;
    int ld_out;
    float scale_log2;  // log2(e) / sqrt(128)
    float* lse;        // optional [heads][n_tokens]: each row's log2-sum-exp2 of scale_log2 * scores
};

// ------------------------------------------------------------------ softmax arithmetic
// Packed fp32 pairs (one 64-bit register, low word first) for the sm_100-family f32x2
// instructions, which do two fp32 operations per issue slot.
F3_DEV uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
F3_DEV void f2_split(uint64_t v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
F3_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
F3_DEV uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
F3_DEV uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
F3_DEV float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
F3_DEV uint32_t bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// 2^x for a pair on the FMA pipe instead of the MUFU unit (which alone would need as many
// cycles as the tensor core for this kernel).  Range reduction x = j + f with j the
// nearest integer (adding 1.5 * 2^23 leaves j in the low mantissa bits), f in [-1/2, 1/2];
// 2^f from a cubic fitted for minimax relative error on [-1/2, 1/2] (max relative error
// 7.5e-5, far below the bf16 rounding of P); 2^j is added to the exponent field.  x is
// clamped at -125 so 2^j stays a normal number.
F3_DEV void exp2_poly2(float x0, float x1, float& p0, float& p1) {
    constexpr float kRound = 12582912.f;  // 1.5 * 2^23
    constexpr float c0 = 0.9999280571937561f, c1 = 0.6932608485221863f, c2 = 0.24261115491390228f,
                    c3 = 0.05517221987247467f;
    const uint64_t x = f2(fmaxf(x0, -125.f), fmaxf(x1, -125.f));
    const uint64_t t = f2_add(x, f2(kRound, kRound));
    const uint64_t f = f2_sub(x, f2_sub(t, f2(kRound, kRound)));
    uint64_t q = f2_fma(f2(c3, c3), f, f2(c2, c2));
    q = f2_fma(q, f, f2(c1, c1));
    q = f2_fma(q, f, f2(c0, c0));
    float q0, q1, t0, t1;
    f2_split(q, q0, q1);
    f2_split(t, t0, t1);
    p0 = __int_as_float(__float_as_int(q0) + (__float_as_int(t0) << 23));
    p1 = __int_as_float(__float_as_int(q1) + (__float_as_int(t1) << 23));
}

#ifndef FLUX3_ATT_POLY_EVERY
#define FLUX3_ATT_POLY_EVERY 0
#endif

// P = 2^(s * sc - m) for keys 64 h .. 64 h + 63 of one 128-key row: every POLY-th pair
// goes through exp2_poly2 (0: none), the rest through ex2.approx; P is stored as bf16
// pairs over TMEM columns 32 h .. 32 h + 31 of the row's score tile.  Returns the sum of
// those 64 P values (fp32, before rounding).
template <int POLY>
F3_DEV float softmax_exp_store(const float (&s)[128], int h, float sc, float m, uint32_t tS) {
    const uint64_t sc2 = f2(sc, sc), nm2 = f2(-m, -m);
    uint64_t acc[4] = {0, 0, 0, 0};
    {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int e = 64 * h + 2 * i;
            float x0, x1, p0, p1;
            f2_split(f2_fma(f2(s[e], s[e + 1]), sc2, nm2), x0, x1);
            if (POLY > 0 && (i % (POLY > 0 ? POLY : 1)) == POLY - 1) {
                exp2_poly2(x0, x1, p0, p1);
            } else {
                p0 = ex2(x0);
                p1 = ex2(x1);
            }
            pk[i] = bf16x2(p0, p1);
            acc[i & 3] = f2_add(acc[i & 3], f2(p0, p1));
        }
        tmem_st32(tS + 32 * h, pk);
    }
    float a0, a1;
    f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
    return a0 + a1;
}

__global__ void __launch_bounds__(ATT_THREADS, 1) attn_tcgen05_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto sQ = [&](int t) { return sbase + t * ATT_TILE_BYTES; };
    auto sKV = [&](int slot) { return sbase + (2 + slot) * ATT_TILE_BYTES; };
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (2 + ATT_SLOTS) * ATT_TILE_BYTES);
    const uint32_t b0 = smem_u32(bars);
    auto q_full = [&](int t) { return b0 + 8u * t; };
    auto kv_full = [&](int s) { return b0 + 8u * (2 + s); };
    auto kv_empty = [&](int s) { return b0 + 8u * (2 + ATT_SLOTS + s); };
    auto s_full = [&](int t) { return b0 + 8u * (2 + 2 * ATT_SLOTS + t); };
    auto p_full = [&](int t) { return b0 + 8u * (4 + 2 * ATT_SLOTS + t); };
    auto o_full = [&](int t) { return b0 + 8u * (6 + 2 * ATT_SLOTS + t); };
    const uint32_t drain = b0 + 8u * (8 + 2 * ATT_SLOTS);
    auto p_half = [&](int t) { return b0 + 8u * (9 + 2 * ATT_SLOTS + t); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 11 + 2 * ATT_SLOTS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int head = blockIdx.y;
    const int pr = blockIdx.x;
    int seg = 0;
    for (int s = 1; s < p.n_seg; ++s)
        if (pr >= p.pair_begin[s]) seg = s;
    const int seg_lo = p.seg_off[seg], seg_hi = p.seg_off[seg + 1];
    const int q0 = seg_lo + (pr - p.pair_begin[seg]) * 256;  // query tile t starts at q0 + 128 t
    const bool has_q1 = q0 + 128 < seg_hi;
    const int kv0 = seg_lo & ~7;  // TMA needs the key (innermost V^T) coordinate 16-byte aligned
    const int nkv = (seg_hi - kv0 + 127) / 128;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(q_full(t), 1);
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), 4);
            mbar_init(p_half(t), 4);
            mbar_init(o_full(t), 1);
        }
        for (int s = 0; s < ATT_SLOTS; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 8) {
        // ---------------- TMA producer (converged warp, one elected lane issues)
        const bool leader = elect_one();
        const int nq = has_q1 ? 2 : 1;
        if (leader) {
            for (int t = 0; t < nq; ++t) {
                mbar_arrive_expect_tx(q_full(t), ATT_TILE_BYTES);
                tma_load_3d(sQ(t), &p.tm_q, q_full(t), 0, q0 + 128 * t, head);
                tma_load_3d(sQ(t) + 16384, &p.tm_q, q_full(t), 64, q0 + 128 * t, head);
            }
        }
        int issued = 0;
        bool ok = true;
        for (int j = 0; j < nkv && ok; ++j) {
            const int k0 = kv0 + 128 * j;
            for (int which = 0; which < 2; ++which) {
                const int idx = 2 * j + which;
                const int slot = idx % ATT_SLOTS;
                if (!mbar_wait_warp(kv_empty(slot), ((idx / ATT_SLOTS) & 1) ^ 1, abort_flag)) { ok = false; break; }
                if (leader) {
                    mbar_arrive_expect_tx(kv_full(slot), ATT_TILE_BYTES);
                    if (which == 0) {
                        tma_load_3d(sKV(slot), &p.tm_k, kv_full(slot), 0, k0, head);
                        tma_load_3d(sKV(slot) + 16384, &p.tm_k, kv_full(slot), 64, k0, head);
                    } else {
                        tma_load_3d(sKV(slot), &p.tm_v, kv_full(slot), k0, 0, head);
                        tma_load_3d(sKV(slot) + 16384, &p.tm_v, kv_full(slot), k0 + 64, 0, head);
                    }
                }
                __syncwarp();
                ++issued;
            }
        }
        if (!ok && leader) {
            // let the copies in flight land before the CTA exits
            for (int t = 0; t < nq; ++t) {
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(q_full(t), 0) && globaltimer() - t0 < kWaitTimeoutNs) {}
            }
            for (int idx = issued - 1; idx >= 0 && idx >= issued - ATT_SLOTS; --idx) {
                const unsigned long long t1 = globaltimer();
                while (!mbar_try_wait(kv_full(idx % ATT_SLOTS), (idx / ATT_SLOTS) & 1) &&
                       globaltimer() - t1 < kWaitTimeoutNs) {}
            }
        }
    } else if (warp == 9) {
        // ---------------- MMA issuer (converged warp, one elected lane issues)
        const bool leader = elect_one();
        constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
        const int nq = has_q1 ? 2 : 1;
        // S_t = Q_t K^T for the K tile in `slot`
        auto qk = [&](int t, int slot) {
            const uint64_t qd = sdesc_kmajor_sw128(sQ(t)), kd = sdesc_kmajor_sw128(sKV(slot));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                mma_bf16_ss_if(leader, tmem + t * 128, qd + off, kd + off, IDESC, kk > 0);
            }
            mma_commit_if(leader, s_full(t));
        };
        // O_t += P_t V for the V^T tile in `slot`; P_t is bf16 in columns 0..63 of S_t
        // (keys 64 h .. 64 h + 63: the half in V^T's swizzle atom h, P columns 32 h ..)
        auto pv = [&](int t, int slot, int h, bool acc) {
            const uint64_t vd = sdesc_kmajor_sw128(sKV(slot));
#pragma unroll
            for (int kk = 4 * h; kk < 4 * h + 4; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                mma_bf16_ts_if(leader, tmem + 256 + t * 128, tmem + t * 128 + kk * 8, vd + off, IDESC, acc || kk > 0);
            }
        };
        auto commit = [&](uint32_t bar) { mma_commit_if(leader, bar); };
        bool ok = mbar_wait_warp(q_full(0), 0, abort_flag) && mbar_wait_warp(kv_full(0), 0, abort_flag);
        if (ok) {
            tc_fence_after();
            qk(0, 0);
            if (has_q1) {
                ok = mbar_wait_warp(q_full(1), 0, abort_flag);
                if (ok) {
                    tc_fence_after();
                    qk(1, 0);
                }
            }
            commit(kv_empty(0));
        }
        for (int j = 0; j < nkv && ok; ++j) {
            const int vidx = 2 * j + 1, vslot = vidx % ATT_SLOTS;
            const int kidx = 2 * j + 2, kslot = kidx % ATT_SLOTS;
            const bool more = j + 1 < nkv;
            if (!mbar_wait_warp(kv_full(vslot), (vidx / ATT_SLOTS) & 1, abort_flag)) { ok = false; break; }
            if (more && !mbar_wait_warp(kv_full(kslot), (kidx / ATT_SLOTS) & 1, abort_flag)) { ok = false; break; }
            for (int t = 0; t < nq; ++t) {
                // the first half of P V starts while the softmax still computes the second
                if (!mbar_wait_warp(p_half(t), j & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                pv(t, vslot, 0, j > 0);
                if (!mbar_wait_warp(p_full(t), j & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                pv(t, vslot, 1, true);
                if (more) qk(t, kslot);  // runs after the P V that reads S_t's columns
            }
            if (!ok) break;
            commit(kv_empty(vslot));
            if (more) commit(kv_empty(kslot));
        }
        if (ok) {
            commit(o_full(0));
            if (has_q1) commit(o_full(1));
        }
        commit(drain);
        if (leader) {
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kWaitTimeoutNs) {}
        }
        __syncwarp();
    } else {
        if (warp < 4 || has_q1) {
        // ---------------- softmax of query tile t: one query row per thread
        const int t = warp >> 2;
        const int sub = warp & 3;
        const int row = sub * 32 + lane;
        const uint32_t tS = tmem + ((uint32_t)(sub * 32) << 16) + t * 128;
        const uint32_t tO = tmem + ((uint32_t)(sub * 32) << 16) + 256 + t * 128;
        const float sc = p.scale_log2;
        float m = -INFINITY, l = 0.f;  // running max (log2 units, scaled) and sum
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            if (!mbar_wait_warp(s_full(t), j & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            float s[128];
            {
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tmem_ld32(tS, r0);
                tmem_ld32(tS + 32, r1);
                tmem_ld32(tS + 64, r2);
                tmem_ld32(tS + 96, r3);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    s[i] = __uint_as_float(r0[i]);
                    s[32 + i] = __uint_as_float(r1[i]);
                    s[64 + i] = __uint_as_float(r2[i]);
                    s[96 + i] = __uint_as_float(r3[i]);
                }
            }
            const int k0 = kv0 + 128 * j;
            const bool full = k0 >= seg_lo && k0 + 128 <= seg_hi;
            if (!full) {
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    const int key = k0 + i;
                    if (key < seg_lo || key >= seg_hi) s[i] = -INFINITY;
                }
            }
            // row max: eight independent chains of 3-input max
            float mc[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) mc[c] = max3(s[c], s[8 + 2 * c], s[9 + 2 * c]);
#pragma unroll
            for (int i = 24; i < 128; i += 16)
#pragma unroll
                for (int c = 0; c < 8; ++c) mc[c] = max3(mc[c], s[i + 2 * c], s[i + 2 * c + 1]);
            const float mx = max3(max3(mc[0], mc[1], mc[2]), max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7])) * sc;
            // keep the stale max unless the new one exceeds it by the slack
            const float mnew = (mx > m + ATT_RESCALE_LOG2) ? mx : m;
            if (j > 0 && __any_sync(0xffffffffu, mnew != m)) {
                // S_t's arrival means every earlier MMA, the P V of tile j-1 included, is done
                const float alpha = ex2(m - mnew);
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t o[16];
                    tmem_ld16(tO + c * 16, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st16(tO + c * 16, o);
                }
                l *= alpha;
            }
            m = mnew;
            // P in two halves (keys 0..63, then 64..127), each signalled as soon as it is in
            // TMEM.  Masked tiles hold -inf scores: they take the exact ex2 path throughout.
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                l += full ? softmax_exp_store<FLUX3_ATT_POLY_EVERY>(s, h, sc, m, tS)
                          : softmax_exp_store<0>(s, h, sc, m, tS);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(h == 0 ? p_half(t) : p_full(t));
            }
        }
        if (ok && mbar_wait_warp(o_full(t), 0, abort_flag)) {
            tc_fence_after();
            const int qrow = q0 + 128 * t + row;
            const bool valid = qrow < seg_hi;
            const float inv = 1.f / l;
            if (p.lse && valid) p.lse[(size_t)head * p.n_tokens + qrow] = m + log2f(l);
            __nv_bfloat16* dst = p.out + (size_t)(valid ? qrow : 0) * p.ld_out + head * 128;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_global_v4(dst + c * 32 + 8 * i,
                                     pack_bf16(__uint_as_float(o[8 * i]) * inv, __uint_as_float(o[8 * i + 1]) * inv),
                                     pack_bf16(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv),
                                     pack_bf16(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv),
                                     pack_bf16(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv));
                }
            }
        }
    }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// --------------------------------------------------------------------- fp32 check path
// One warp per query row, fp32 throughout (expf, fp32 accumulation); lane t holds head
// dims 4t .. 4t+3.  Reads V from the transposed layout.  Slow; for checking only.
struct SegTable {
    int n_seg;
    int off[FLUX3_MAX_SEGMENTS + 1];
};

__global__ void __launch_bounds__(128) attn_f32_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                                                       const __nv_bfloat16* __restrict__ vt, int ld_vt, int n_tokens,
                                                       const SegTable segs, float* __restrict__ out, int ld_out,
                                                       float scale) {
    const int head = blockIdx.y;
    const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= n_tokens) return;
    int sg = 0;
    for (int i = 1; i < segs.n_seg; ++i)
        if (r >= segs.off[i]) sg = i;
    const int lo = segs.off[sg], hi = segs.off[sg + 1];
    const __nv_bfloat16* qr = q + ((size_t)head * n_tokens + r) * 128 + 4 * lane;
    float qv[4];
    for (int i = 0; i < 4; ++i) qv[i] = __bfloat162float(qr[i]);
    float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    const __nv_bfloat16* vh = vt + (size_t)head * 128 * ld_vt;
    for (int key = lo; key < hi; ++key) {
        const __nv_bfloat16* kr = k + ((size_t)head * n_tokens + key) * 128 + 4 * lane;
        float d = 0.f;
        for (int i = 0; i < 4; ++i) d = fmaf(qv[i], __bfloat162float(kr[i]), d);
        for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        d *= scale;
        const float mnew = fmaxf(m, d);
        const float a = expf(m - mnew), pr = expf(d - mnew);
        l = l * a + pr;
        for (int i = 0; i < 4; ++i) acc[i] = acc[i] * a + pr * __bfloat162float(vh[(size_t)(4 * lane + i) * ld_vt + key]);
        m = mnew;
    }
    float* dst = out + (size_t)r * ld_out + head * 128 + 4 * lane;
    for (int i = 0; i < 4; ++i) dst[i] = acc[i] / l;
}

}  // namespace f3
