// attention.cuh -- flash attention for the block: softmax(q k^T / sqrt(128)) v per head,
// bidirectional, no padding mask, optionally restricted to the query's own segment
// ("How it works": stage 1 attends within each stream, stage 2 over all tokens, and the
// text padding is attended).
//
// One CTA per (128-query tile, head).  Warp 0 streams K and V^T tiles of 128 keys by TMA
// into a 4-slot ring; warp 1 issues tcgen05.mma: S = Q K^T into one of two TMEM score
// buffers (so QK^T of tile j+1 overlaps the softmax of tile j) and O += P V into a TMEM
// accumulator; warps 2..5 own one query row per thread: online softmax in the log2
// domain, rescaling of O in TMEM when the running max moves, P written as bf16 to
// shared memory in the 128-byte-swizzled K-major layout the MMA reads.
#pragma once
#include <cuda.h>
#include "sm103.cuh"
#include "../../include/flux3.h"

namespace f3 {

constexpr int ATT_THREADS = 192;
constexpr int ATT_SLOTS = 4;
constexpr int ATT_TILE_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 operand tile
constexpr int ATT_SMEM_BYTES = 1024 + (2 + ATT_SLOTS) * ATT_TILE_BYTES + 256;

struct AttnParams {
    CUtensorMap tm_q, tm_k, tm_v;
    int n_tokens, heads, n_seg;
    int seg_off[FLUX3_MAX_SEGMENTS + 1];
    int qt_begin[FLUX3_MAX_SEGMENTS + 1];
    __nv_bfloat16* out;
    int ld_out;
    float scale_log2;  // log2(e) / sqrt(128)
};

// byte offset of 16-byte chunk `c` (0..15, 8 keys each) of row `r` in a 128 x 128 bf16
// K-major tile stored as two 64-wide swizzle atoms of 16 KB
F3_DEV uint32_t sw128_offset(int r, int c) {
    return (uint32_t)((c >> 3) * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(ATT_THREADS, 1) attn_tcgen05_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase;
    const uint32_t sP = sbase + ATT_TILE_BYTES;
    auto sKV = [&](int slot) { return sbase + (2 + slot) * ATT_TILE_BYTES; };
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (2 + ATT_SLOTS) * ATT_TILE_BYTES);
    const uint32_t b0 = smem_u32(bars);
    const uint32_t q_full = b0;
    auto kv_full = [&](int s) { return b0 + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return b0 + 8u * (1 + ATT_SLOTS + s); };
    auto s_full = [&](int b) { return b0 + 8u * (1 + 2 * ATT_SLOTS + b); };
    auto s_free = [&](int b) { return b0 + 8u * (3 + 2 * ATT_SLOTS + b); };
    const uint32_t p_full = b0 + 8u * (5 + 2 * ATT_SLOTS);
    const uint32_t o_ready = b0 + 8u * (6 + 2 * ATT_SLOTS);
    const uint32_t drain = b0 + 8u * (7 + 2 * ATT_SLOTS);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 8 + 2 * ATT_SLOTS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int head = blockIdx.y;
    const int qt = blockIdx.x;
    int seg = 0;
    for (int s = 1; s < p.n_seg; ++s)
        if (qt >= p.qt_begin[s]) seg = s;
    const int seg_lo = p.seg_off[seg], seg_hi = p.seg_off[seg + 1];
    const int q0 = seg_lo + (qt - p.qt_begin[seg]) * 128;
    const int kv0 = seg_lo & ~7;  // TMA needs the key (innermost V^T) coordinate 16-byte aligned
    const int nkv = (seg_hi - kv0 + 127) / 128;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < ATT_SLOTS; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(s_free(b), 4);
        }
        mbar_init(p_full, 4);
        mbar_init(o_ready, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;  // S0: cols 0..127, S1: 128..255, O: 256..383

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: Q once, then K_0, V_0, K_1, V_1, ...
            mbar_arrive_expect_tx(q_full, ATT_TILE_BYTES);
            tma_load_3d(sQ, &p.tm_q, q_full, 0, q0, head);
            tma_load_3d(sQ + 16384, &p.tm_q, q_full, 64, q0, head);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < nkv && ok; ++j) {
                const int k0 = kv0 + 128 * j;
                for (int which = 0; which < 2; ++which) {
                    const int idx = 2 * j + which;
                    const int slot = idx % ATT_SLOTS;
                    if (!mbar_wait(kv_empty(slot), ((idx / ATT_SLOTS) & 1) ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(kv_full(slot), ATT_TILE_BYTES);
                    if (which == 0) {
                        tma_load_3d(sKV(slot), &p.tm_k, kv_full(slot), 0, k0, head);
                        tma_load_3d(sKV(slot) + 16384, &p.tm_k, kv_full(slot), 64, k0, head);
                    } else {
                        tma_load_3d(sKV(slot), &p.tm_v, kv_full(slot), k0, 0, head);
                        tma_load_3d(sKV(slot) + 16384, &p.tm_v, kv_full(slot), k0 + 64, 0, head);
                    }
                    ++issued;
                }
            }
            if (!ok) {
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(q_full, 0) && globaltimer() - t0 < kWaitTimeoutNs) {}
                for (int idx = issued - 1; idx >= 0 && idx >= issued - ATT_SLOTS; --idx) {
                    const unsigned long long t1 = globaltimer();
                    while (!mbar_try_wait(kv_full(idx % ATT_SLOTS), (idx / ATT_SLOTS) & 1) &&
                           globaltimer() - t1 < kWaitTimeoutNs) {}
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t IDESC = idesc_bf16_f32(128, 128);
            bool ok = mbar_wait(q_full, 0, abort_flag);
            auto issue_s = [&](int j) -> bool {
                const int idx = 2 * j, slot = idx % ATT_SLOTS, b = j & 1;
                if (!mbar_wait(kv_full(slot), (idx / ATT_SLOTS) & 1, abort_flag)) return false;
                if (!mbar_wait(s_free(b), ((j >> 1) & 1) ^ 1, abort_flag)) return false;
                tc_fence_after();
                const uint64_t qd = sdesc_kmajor_sw128(sQ), kd = sdesc_kmajor_sw128(sKV(slot));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    mma_bf16_ss(tmem + b * 128, qd + off, kd + off, IDESC, kk > 0);
                }
                mma_commit(s_full(b));
                mma_commit(kv_empty(slot));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; j < nkv && ok; ++j) {
                if (j + 1 < nkv && !(ok = issue_s(j + 1))) break;
                const int idx = 2 * j + 1, slot = idx % ATT_SLOTS;
                if (!mbar_wait(p_full, j & 1, abort_flag)) { ok = false; break; }
                if (!mbar_wait(kv_full(slot), (idx / ATT_SLOTS) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint64_t pd = sdesc_kmajor_sw128(sP), vd = sdesc_kmajor_sw128(sKV(slot));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    mma_bf16_ss(tmem + 256, pd + off, vd + off, IDESC, (j | kk) != 0);
                }
                mma_commit(o_ready);
                mma_commit(kv_empty(slot));
            }
            mma_commit(drain);
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kWaitTimeoutNs) {}
        }
    } else {
        // ---------------- softmax warps: one query row per thread
        const int sub = warp & 3;
        const int row = sub * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(sub * 32) << 16;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        uint8_t* sPgen = smem + ATT_TILE_BYTES;
        for (int j = 0; j < nkv; ++j) {
            const int b = j & 1;
            if (!mbar_wait(s_full(b), (j >> 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            float s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t t[32];
                tmem_ld32(tmem + lane_addr + b * 128 + c * 32, t);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(t[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(b));

            const int k0 = kv0 + 128 * j;
            float mx = -INFINITY;
            if (k0 >= seg_lo && k0 + 128 <= seg_hi) {
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    s[i] *= p.scale_log2;
                    mx = fmaxf(mx, s[i]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    const int key = k0 + i;
                    s[i] = (key >= seg_lo && key < seg_hi) ? s[i] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, s[i]);
                }
            }
            const float mnew = fmaxf(m, mx);
            const float alpha = ex2(m - mnew);  // 0 on the first tile (m = -inf)
            float sum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const float p0 = ex2(s[2 * i] - mnew), p1 = ex2(s[2 * i + 1] - mnew);
                sum += p0 + p1;
                pk[i] = pack_bf16(p0, p1);
            }
            l = l * alpha + sum;
            m = mnew;
            if (j > 0) {
                // PV of the previous tile is done: O is final up to j-1 and P is free
                if (!mbar_wait(o_ready, (j - 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t t[32];
                        tmem_ld32(tmem + lane_addr + 256 + c * 32, t);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) t[i] = __float_as_uint(__uint_as_float(t[i]) * alpha);
                        tmem_st32(tmem + lane_addr + 256 + c * 32, t);
                    }
                    tmem_st_wait();
                }
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint32_t off = sw128_offset(row, c);
                *reinterpret_cast<uint4*>(sPgen + off) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok && mbar_wait(o_ready, (nkv - 1) & 1, abort_flag)) {
            tc_fence_after();
            const int qrow = q0 + row;
            const bool valid = qrow < seg_hi;
            const float inv = 1.f / l;
            __nv_bfloat16* dst = p.out + (size_t)(valid ? qrow : 0) * p.ld_out + head * 128;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t t[32];
                tmem_ld32(tmem + lane_addr + 256 + c * 32, t);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_global_v4(dst + c * 32 + 8 * i,
                                     pack_bf16(__uint_as_float(t[8 * i]) * inv, __uint_as_float(t[8 * i + 1]) * inv),
                                     pack_bf16(__uint_as_float(t[8 * i + 2]) * inv, __uint_as_float(t[8 * i + 3]) * inv),
                                     pack_bf16(__uint_as_float(t[8 * i + 4]) * inv, __uint_as_float(t[8 * i + 5]) * inv),
                                     pack_bf16(__uint_as_float(t[8 * i + 6]) * inv, __uint_as_float(t[8 * i + 7]) * inv));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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
