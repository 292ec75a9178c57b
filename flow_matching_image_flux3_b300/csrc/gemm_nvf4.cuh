// gemm_nvf4.cuh -- the block's projections on NVFP4 operands ("FLUX.3" cookbook, section 3,
// Quantized checkpoints: FP4 (E2M1) values with FP8 block scales on a Blackwell GPU):
//   P = s_a[token] * sum_k (e2m1(a) sb_a)(e2m1(w) sb_w) * s_w[out] + b
// with the block-scaled tcgen05 MMA (kind::mxf4nvf4, one e4m3 scale per 16 elements of K
// for each operand row) and the same fused epilogues as the bf16 projections (EPI:
// EPI_QKV_SWIGLU for the input projection, EPI_GATED_RESIDUAL for the output projection).
//
// The same persistent, warp-specialised structure as gemm_tcgen05_kernel (warp 0 TMA,
// warp 1 MMA, EW epilogue warps from warp 2; clusters of two share the weight tile by
// multicast),
// with two differences:
//  - a stage also carries the tiles' block scales (2 KB for the 128 A rows, 4 KB for the
//    256 B rows of a 256-element k-block, 1-D bulk copies of the tiled scale layout), and
//    the MMA warp copies them into TMEM (tcgen05.cp) right before the k-block's MMAs;
//  - the scales take 48 TMEM columns per stage, so the accumulator is single (256
//    columns + 4 x 48): the next tile's MMAs start once the epilogue has read this one.
// A TMEM scale slot belongs to its shared-memory stage: the MMAs that read it are
// complete before the stage's empty barrier fires, which the producer waits for before
// refilling the stage, which the MMA warp waits for before copying new scales in.
#pragma once
#include "gemm.cuh"

namespace f3 {

struct Nvf4Cfg {
    static constexpr int STAGES = 4;
    static constexpr int A_BYTES = GEMM_BM * 128;      // 128 rows x 256 codes
    static constexpr int B_BYTES = 256 * 128;          // 256 rows x 256 codes
    static constexpr int SFA_BYTES = 4 * 512;          // 128 rows x 16 scales: 4 tiles of 512 B
    static constexpr int SFB_BYTES = 8 * 512;          // 256 rows x 16 scales
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;  // 54 KB
    static constexpr int ACC_COLS = 256;
    static constexpr int SF_COLS = 48;                 // per stage: 4 x 4 (A) + 4 x 8 (B)
    static constexpr int TMEM_COLS = 512;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned for the 128-byte swizzle");
    static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
};

template <int CL, int EW, int EPI>
__global__ void __launch_bounds__(gemm_threads(EW), 1) gemm_nvf4_kernel(const __grid_constant__ GemmParams p) {
    static_assert(CL == 1 || CL == 2, "clusters of one or two");
    static_assert(EPI == EPI_QKV_SWIGLU || EPI == EPI_GATED_RESIDUAL, "the block's projections");
    static_assert(EW == 4 || (EW == 8 && EPI == EPI_QKV_SWIGLU), "8 epilogue warps: input projection only");
    using C = Nvf4Cfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    const uint32_t tfull_bar = bar0 + 8u * (2 * C::STAGES);
    const uint32_t tempty_bar = bar0 + 8u * (2 * C::STAGES + 1);
    const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 2);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const uint32_t smem_base = smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = CL == 2 ? (int)cluster_ctarank() : 0;
    const int unit = blockIdx.x / CL, n_units = gridDim.x / CL;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), CL);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, EW);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&p.tm_a);
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    if (CL > 1) cluster_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int tasks = (p.m_tiles / CL) * p.n_tiles;
    constexpr uint16_t kPair = 0x3;
    const size_t sf_row_tile = (size_t)p.sf_steps * 512;  // bytes of scales per 128 rows

    if (warp == 0) {
        // ---------------- TMA producer
        const bool leader = elect_one();
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        bool ok = true;
        for (int task = unit; task < tasks && ok; task += n_units) {
            const TileInfo ti = tile_info(p, task, rank, CL);
            const int ws = p.grp[ti.g].wset;
            const CUtensorMap* tb = &p.tm_b[ws];
            int r0, r1;
            b_rows<256, EPI>(p, ti.n, r0, r1);
            const uint8_t* sfa = p.a_sf + (size_t)(ti.row0 / GEMM_BM) * sf_row_tile;
            const uint8_t* sfb0 = p.ew[ws].w_sf + (size_t)(r0 / 128) * sf_row_tile;
            const uint8_t* sfb1 = p.ew[ws].w_sf + (size_t)(r1 / 128) * sf_row_tile;
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!mbar_wait_warp(empty_bar(s), ph ^ 1u, abort_flag)) { ok = false; break; }
                if (leader) {
                    const uint32_t sa = smem_base + s * C::STAGE_BYTES;
                    const uint32_t sb = sa + C::A_BYTES;
                    const uint32_t ssa = sb + C::B_BYTES;
                    const uint32_t ssb = ssa + C::SFA_BYTES;
                    int kr = ti.kb0 + kb;
                    if (kr >= p.k_blocks) kr -= p.k_blocks;
                    mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
                    tma_load_2d(sa, &p.tm_a, full_bar(s), kr * 128, ti.row0);
                    if (CL == 2) {
                        tma_load_2d_multicast(sb + rank * 128 * 128, tb, full_bar(s), kr * 128, rank ? r1 : r0, kPair);
                    } else {
                        tma_load_2d(sb, tb, full_bar(s), kr * 128, r0);
                        tma_load_2d(sb + 128 * 128, tb, full_bar(s), kr * 128, r1);
                    }
                    bulk_load(ssa, sfa + (size_t)kr * 2048, 2048, full_bar(s));
                    bulk_load(ssb, sfb0 + (size_t)kr * 2048, 2048, full_bar(s));
                    bulk_load(ssb + 2048, sfb1 + (size_t)kr * 2048, 2048, full_bar(s));
                }
                __syncwarp();
                ++issued;
                if (++s == C::STAGES) { s = 0; ph ^= 1u; }
            }
        }
        if (!ok && leader) {
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
        // ---------------- MMA issuer: per k-block, 12 scale copies into the stage's TMEM
        // slot, then 4 block-scaled MMAs (K = 64 each)
        const bool leader = elect_one();
        constexpr uint32_t IDESC = idesc_nvf4_f32(GEMM_BM, 256);
        int s = 0;
        uint32_t ph = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int task = unit; task < tasks && ok; task += n_units) {
            if (!mbar_wait_warp(tempty_bar, aph ^ 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!mbar_wait_warp(full_bar(s), ph, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_base + s * C::STAGE_BYTES;
                const uint32_t ssa = sa + C::A_BYTES + C::B_BYTES;
                const uint32_t ssb = ssa + C::SFA_BYTES;
                const uint32_t tsf = tmem_base + C::ACC_COLS + s * C::SF_COLS;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    tmem_cp_32x128b_x4_if(leader, tsf + 4 * k, ssa + 512 * k);
                    tmem_cp_32x128b_x4_if(leader, tsf + 16 + 8 * k, ssb + 512 * k);
                    tmem_cp_32x128b_x4_if(leader, tsf + 16 + 8 * k + 4, ssb + 2048 + 512 * k);
                }
                const uint64_t ad = sdesc_kmajor_sw128(sa);
                const uint64_t bd = sdesc_kmajor_sw128(sa + C::A_BYTES);
#pragma unroll
                for (int k = 0; k < 4; ++k)  // 32 bytes of each row per instruction
                    mma_nvf4_ss_if(leader, tmem_base, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), IDESC, tsf + 4 * k,
                                   tsf + 16 + 8 * k, (kb | k) != 0);
                if (CL == 2) mma_commit_multicast_if(leader, empty_bar(s), kPair);
                else mma_commit_if(leader, empty_bar(s));
                if (++s == C::STAGES) { s = 0; ph ^= 1u; }
            }
            if (!ok) break;
            mma_commit_if(leader, tfull_bar);
            aph ^= 1u;
        }
        if (leader) {
            mma_commit(drain_bar);
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < kWaitTimeoutNs) {}
        }
        __syncwarp();
    } else {
        // ---------------- epilogue warps 2 .. 2 + EW - 1
        const int sub = warp & 3;
        const int part = (warp - 2) >> 2;
        uint32_t aph = 0;
        for (int task = unit; task < tasks; task += n_units) {
            const TileInfo ti = tile_info(p, task, rank, CL);
            const int r = ti.row0 + sub * 32 + lane;
            const bool valid = r < p.grp[ti.g].row_end;
            if (!mbar_wait_warp(tfull_bar, aph, abort_flag)) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + ((uint32_t)(sub * 32) << 16);
            if constexpr (EPI == EPI_QKV_SWIGLU)
                epi_qkv<2, EW / 4>(p, p.ew[p.grp[ti.g].wset], ti.n, tacc, valid ? r : 0, valid, part);
            else
                epi_gated_residual<256, 2>(p, p.ew[p.grp[ti.g].wset], ti.n, tacc, valid ? r : 0, valid);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar);
            aph ^= 1u;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    if (CL > 1) cluster_sync();
}

}  // namespace f3
