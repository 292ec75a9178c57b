// flux3.cu -- libflux3.so: the C-ABI entry points of include/flux3.h.  Host-side
// argument checks, TMA tensor-map encoding, workspace carving and kernel launches.
// Every step of the block runs in the kernels of gemm.cuh, attention.cuh and simt.cuh.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/flux3.h"
#include "sm103.cuh"
#include "simt.cuh"
#include "gemm.cuh"
#include "gemm_nvf4.cuh"
#include "attention.cuh"
#include "bwd.cuh"

using namespace f3;

namespace {

constexpr int kMaxTokens = 1 << 22;

// ------------------------------------------------------------------ driver entry point
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool have_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// bf16 row-major [outer, inner] (row stride in bytes), box 64 x box_outer, 128-byte swizzle
bool tmap_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {64, box_outer};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// 8-bit codes (e4m3) row-major [outer, inner], box 128 x box_outer (128 bytes), 128-byte swizzle
bool tmap_2d_u8(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {128, box_outer};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bf16 [d2][d1][d0], strides in bytes, box 64 x 128 x 1, 128-byte swizzle
bool tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2) {
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Raise a kernel's dynamic shared-memory limit once per device (the attribute persists;
// setting it again on every launch is host work, and is not a stream operation a graph
// capture can record).
// (one flag array per kernel: the kernel is the template argument)
template <auto Kernel>
bool smem_attr_once(int bytes) {
    static std::atomic<bool> done[64] = {};  // host threads may launch concurrently
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev].load(std::memory_order_acquire)) return true;
    if (cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    done[dev].store(true, std::memory_order_release);  // setting it twice is harmless
    return true;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// ------------------------------------------------------------------ profiling marks
struct Profiler {
    bool on = false;
    int cap = 0, n = 0;
    std::vector<cudaEvent_t> ev;
    std::vector<int> kind;
} g_prof;

void prof_before(int kind, cudaStream_t st) {
    if (!g_prof.on || g_prof.n >= g_prof.cap) return;
    cudaEventRecord(g_prof.ev[2 * g_prof.n], st);
    g_prof.kind[g_prof.n] = kind;
}
void prof_after(cudaStream_t st) {
    if (!g_prof.on || g_prof.n >= g_prof.cap) return;
    cudaEventRecord(g_prof.ev[2 * g_prof.n + 1], st);
    ++g_prof.n;
}

flux3_status launch_status() { return cudaGetLastError() == cudaSuccess ? FLUX3_OK : FLUX3_ERR_CUDA; }

// ------------------------------------------------------------------ argument checks
bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
size_t up256(size_t b) { return (b + 255) & ~size_t(255); }

flux3_status check_dims(const flux3_dims* d) {
    if (!d) return FLUX3_ERR_INVALID_ARG;
    if (d->heads <= 0 || d->width <= 0 || d->ffn_hidden <= 0 || d->head_dim <= 0) return FLUX3_ERR_INVALID_ARG;
    if (!(d->ln_eps > 0.f) || !(d->rms_eps > 0.f) || !(d->rope_theta > 0.f) || !std::isfinite(d->rope_theta))
        return FLUX3_ERR_INVALID_ARG;
    if ((long long)d->heads * d->head_dim != d->width) return FLUX3_ERR_INVALID_ARG;
    if (d->head_dim != 128) return FLUX3_ERR_UNSUPPORTED;
    if (d->heads % 2 != 0 || d->ffn_hidden % 128 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (d->width > 32 * 8 * kAdaLnMaxChunks) return FLUX3_ERR_UNSUPPORTED;
    if (d->ffn_hidden > 65536) return FLUX3_ERR_UNSUPPORTED;
    return FLUX3_OK;
}

flux3_status check_offsets(const int32_t* off, int n_seg, int n_tokens) {
    if (!off || n_seg < 1 || n_seg > FLUX3_MAX_SEGMENTS) return FLUX3_ERR_INVALID_ARG;
    if (off[0] != 0 || off[n_seg] != n_tokens) return FLUX3_ERR_INVALID_ARG;
    for (int i = 0; i < n_seg; ++i)
        if (off[i + 1] < off[i]) return FLUX3_ERR_INVALID_ARG;
    return FLUX3_OK;
}

flux3_status check_segs(const flux3_segments* s, int n_tokens, bool need_mod) {
    if (!s) return FLUX3_ERR_INVALID_ARG;
    flux3_status st = check_offsets(s->seg_off, s->n_seg, n_tokens);
    if (st != FLUX3_OK) return st;
    if (need_mod && (!s->mod || !al16(s->mod))) return FLUX3_ERR_INVALID_ARG;
    return FLUX3_OK;
}

flux3_status check_weights(const flux3_block_weights* w, int n_w, bool in_proj, bool out_proj) {
    if (!w || n_w < 1 || n_w > FLUX3_MAX_SEGMENTS) return FLUX3_ERR_INVALID_ARG;
    for (int i = 0; i < n_w; ++i) {
        if (in_proj) {
            if (!w[i].w_in || !al16(w[i].w_in) || !w[i].q_norm || !al16(w[i].q_norm) || !w[i].k_norm ||
                !al16(w[i].k_norm) || (w[i].b_in && !al16(w[i].b_in)))
                return FLUX3_ERR_INVALID_ARG;
        }
        if (out_proj) {
            if (!w[i].w_out || !al16(w[i].w_out) || (w[i].b_out && !al16(w[i].b_out))) return FLUX3_ERR_INVALID_ARG;
        }
    }
    return FLUX3_OK;
}

SegOffsets seg_table(const int32_t* off, int n_seg) {
    SegOffsets t;
    std::memset(&t, 0, sizeof t);
    t.n_seg = n_seg;
    for (int i = 0; i <= n_seg; ++i) t.off[i] = off[i];
    return t;
}

// workspace carve-up of one block
struct BlockWs {
    __nv_bfloat16 *a, *q, *k, *vt, *y;
    int ld_vt;
    size_t bytes;
};
BlockWs block_ws_layout(const flux3_dims* d, int N, uint8_t* base) {
    BlockWs w;
    const size_t D = d->width, H = d->heads, F = d->ffn_hidden;
    w.ld_vt = (N + 7) & ~7;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = base ? base + off : nullptr;
        off += up256(bytes);
        return reinterpret_cast<__nv_bfloat16*>(p);
    };
    w.a = take((size_t)N * D * 2);
    w.q = take(H * (size_t)N * 128 * 2);
    w.k = take(H * (size_t)N * 128 * 2);
    w.vt = take(H * 128 * (size_t)w.ld_vt * 2);
    w.y = take((size_t)N * (D + F) * 2);
    w.bytes = off;
    return w;
}

// ------------------------------------------------------------------ launchers (checked args)
flux3_status run_adaln(const flux3_dims* d, const float* mod, const SegOffsets& segs, const void* x, int n_rows, void* a,
                       cudaStream_t st) {
    if (n_rows == 0) return FLUX3_OK;
    prof_before(FLUX3_KERNEL_ADALN, st);
    if (!launch_adaln(d->width, static_cast<const __nv_bfloat16*>(x), n_rows, d->ln_eps, mod, segs,
                      static_cast<__nv_bfloat16*>(a), st))
        return FLUX3_ERR_UNSUPPORTED;
    prof_after(st);
    return launch_status();
}

// Clusters of two CTAs that can be resident at once for a GEMM kernel (SMs are paired
// within a GPC, so this can be below half the SM count); cached per device.
template <auto Kernel>
int max_active_pairs(int smem, int threads, int sms) {
    static std::atomic<int> cache[64] = {};  // host threads may launch concurrently
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int known = cache[dev].load(std::memory_order_acquire);
    if (known > 0) return known;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms & ~1));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, Kernel, &cfg) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_release);
    return n;
}

// A persistent GEMM kernel in clusters of two: one cluster per resident pair, at most one
// per pair of tiles.
template <auto Kernel>
flux3_status launch_pairs(const GemmParams& P, int smem, int threads, cudaStream_t st, int kind) {
    const int tasks = (P.m_tiles / 2) * P.n_tiles;
    if (tasks == 0) return FLUX3_OK;
    if (!smem_attr_once<Kernel>(smem)) return FLUX3_ERR_CUDA;
    const int sms = sm_count();
    if (sms <= 0) return FLUX3_ERR_CUDA;
    const int pairs = max_active_pairs<Kernel>(smem, threads, sms);
    if (pairs <= 0) return FLUX3_ERR_CUDA;
    const int units = tasks < pairs ? tasks : pairs;  // persistent: every cluster resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * units));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_before(kind, st);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, Kernel, P);
    prof_after(st);
    return e == cudaSuccess ? launch_status() : FLUX3_ERR_CUDA;
}

template <int BN, int EPI, int CL, int AK = 0, int EW = 4>
flux3_status launch_gemm(const GemmParams& P, cudaStream_t st, int kind) {
    const int smem = GemmCfg<BN>::SMEM_BYTES;
    if constexpr (CL == 1) {
        const int tasks = P.m_tiles * P.n_tiles;
        if (tasks == 0) return FLUX3_OK;
        if (!smem_attr_once<gemm_tcgen05_kernel<BN, EPI, CL, AK, EW>>(smem)) return FLUX3_ERR_CUDA;
        const int sms = sm_count();
        if (sms <= 0) return FLUX3_ERR_CUDA;
        const int grid = tasks < sms ? tasks : sms;
        prof_before(kind, st);
        gemm_tcgen05_kernel<BN, EPI, CL, AK, EW><<<grid, gemm_threads(EW), smem, st>>>(P);
        prof_after(st);
        return launch_status();
    } else {
        return launch_pairs<gemm_tcgen05_kernel<BN, EPI, 2, AK, EW>>(P, smem, gemm_threads(EW), st, kind);
    }
}

// groups of rows sharing one weight set; m-tiles never straddle a group, and with clusters
// of `cl` CTAs every group starts on a multiple of cl (a cluster's tiles share weights)
void fill_groups(GemmParams& P, const int32_t* off, int n_seg, int n_w, int N, int cl) {
    auto units = [cl](int rows) { return ((rows + GEMM_BM - 1) / GEMM_BM + cl - 1) / cl * cl; };
    int tiles = 0;
    if (n_w == 1) {
        P.n_groups = 1;
        P.grp[0] = {0, N, 0, 0};
        tiles = units(N);
    } else {
        P.n_groups = n_seg;
        for (int s = 0; s < n_seg; ++s) {
            P.grp[s] = {off[s], off[s + 1], tiles, s};
            tiles += units(off[s + 1] - off[s]);
        }
    }
    P.m_tiles = tiles;
}

flux3_status run_in_proj(const flux3_dims* d, const flux3_block_weights* w, int n_w, const flux3_segments* segs, const void* a,
                         int N, const float* rope, void* q, void* k, void* vt, int ld_vt, void* y, cudaStream_t st) {
    if (N == 0) return FLUX3_OK;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    const int D = d->width, F = d->ffn_hidden, H = d->heads;
    const int n_in = 3 * D + 2 * F;
    if (!tmap_2d(&P.tm_a, a, D, N, (uint64_t)D * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    for (int i = 0; i < n_w; ++i) {
        if (!tmap_2d(&P.tm_b[i], w[i].w_in, D, n_in, (uint64_t)D * 2, 128)) return FLUX3_ERR_INVALID_ARG;
        P.ew[i] = {w[i].b_in, w[i].q_norm, w[i].k_norm};
    }
    fill_groups(P, segs->seg_off, segs->n_seg, n_w, N, 2);
    P.n_tiles = 3 * H / 2 + F / 128;
    P.k_blocks = D / GEMM_BK;
    P.heads = H; P.width = D; P.ffn = F; P.n_tokens = N; P.ld_vt = ld_vt; P.ld_y = D + F;
    P.rms_eps = d->rms_eps;
    P.rope = rope;
    P.q = static_cast<__nv_bfloat16*>(q); P.k = static_cast<__nv_bfloat16*>(k);
    P.vt = static_cast<__nv_bfloat16*>(vt); P.y = static_cast<__nv_bfloat16*>(y);
    return launch_gemm<256, EPI_QKV_SWIGLU, 2>(P, st, FLUX3_KERNEL_IN_PROJ);
}

// the input projection on e4m3 operands: a8 [N, D] codes with per-token scales sa, each
// weight set's e4m3 W_in with per-row scales
flux3_status run_in_proj_fp8(const flux3_dims* d, const flux3_block_weights_fp8* w, int n_w, const flux3_segments* segs,
                             const void* a8, const float* sa, int N, const float* rope, void* q, void* k, void* vt,
                             int ld_vt, void* y, cudaStream_t st) {
    if (N == 0) return FLUX3_OK;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    const int D = d->width, F = d->ffn_hidden, H = d->heads;
    const int n_in = 3 * D + 2 * F;
    if (!tmap_2d_u8(&P.tm_a, a8, D, N, (uint64_t)D, 128)) return FLUX3_ERR_INVALID_ARG;
    for (int i = 0; i < n_w; ++i) {
        if (!tmap_2d_u8(&P.tm_b[i], w[i].w_in, D, n_in, (uint64_t)D, 128)) return FLUX3_ERR_INVALID_ARG;
        P.ew[i] = {w[i].b_in, w[i].q_norm, w[i].k_norm, w[i].s_in};
    }
    fill_groups(P, segs->seg_off, segs->n_seg, n_w, N, 2);
    P.n_tiles = 3 * H / 2 + F / 128;
    P.k_blocks = D / 128;
    P.a_scale = sa;
    P.heads = H; P.width = D; P.ffn = F; P.n_tokens = N; P.ld_vt = ld_vt; P.ld_y = D + F;
    P.rms_eps = d->rms_eps;
    P.rope = rope;
    P.q = static_cast<__nv_bfloat16*>(q); P.k = static_cast<__nv_bfloat16*>(k);
    P.vt = static_cast<__nv_bfloat16*>(vt); P.y = static_cast<__nv_bfloat16*>(y);
    return launch_gemm<256, EPI_QKV_SWIGLU, 2, 1, 8>(P, st, FLUX3_KERNEL_IN_PROJ);
}

flux3_status run_quantize_rows(const void* x, int rows, int k, void* q, float* scale, cudaStream_t st) {
    if (rows == 0) return FLUX3_OK;
    prof_before(FLUX3_KERNEL_QUANTIZE, st);
    quantize_rows_e4m3_kernel<<<(rows + 7) / 8, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), rows, k,
                                                             static_cast<uint8_t*>(q), scale);
    prof_after(st);
    return launch_status();
}

// the input projection on NVFP4 operands (one weight set): a4 [N, D / 2] codes, a_sf the
// tiled block scales, sa the per-token scales
flux3_status run_in_proj_nvfp4(const flux3_dims* d, const flux3_block_weights_nvfp4* w, const void* a4, const void* a_sf,
                               const float* sa, int N, const float* rope, void* q, void* k, void* vt, int ld_vt, void* y,
                               cudaStream_t st) {
    if (N == 0) return FLUX3_OK;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    const int D = d->width, F = d->ffn_hidden, H = d->heads;
    const int n_in = 3 * D + 2 * F;
    if (!tmap_2d_u8(&P.tm_a, a4, D / 2, N, (uint64_t)D / 2, 128)) return FLUX3_ERR_INVALID_ARG;
    if (!tmap_2d_u8(&P.tm_b[0], w->w_in, D / 2, n_in, (uint64_t)D / 2, 128)) return FLUX3_ERR_INVALID_ARG;
    P.ew[0] = {w->b_in, w->q_norm, w->k_norm, w->s_in, static_cast<const uint8_t*>(w->w_sf)};
    const int32_t one[2] = {0, N};
    fill_groups(P, one, 1, 1, N, 2);
    P.n_tiles = 3 * H / 2 + F / 128;
    P.k_blocks = D / 256;
    P.sf_steps = D / 64;
    P.a_scale = sa;
    P.a_sf = static_cast<const uint8_t*>(a_sf);
    P.heads = H; P.width = D; P.ffn = F; P.n_tokens = N; P.ld_vt = ld_vt; P.ld_y = D + F;
    P.rms_eps = d->rms_eps;
    P.rope = rope;
    P.q = static_cast<__nv_bfloat16*>(q); P.k = static_cast<__nv_bfloat16*>(k);
    P.vt = static_cast<__nv_bfloat16*>(vt); P.y = static_cast<__nv_bfloat16*>(y);
    return launch_pairs<gemm_nvf4_kernel<2, 8, EPI_QKV_SWIGLU>>(P, Nvf4Cfg::SMEM_BYTES, gemm_threads(8), st,
                                                               FLUX3_KERNEL_IN_PROJ);
}

// rows padded to a pair of 128-row tiles: the scale rows an NVFP4 GEMM may read
int nvfp4_rows_padded(int rows) { return (rows + 255) / 256 * 256; }

flux3_status run_quantize_rows_nvfp4(const void* x, int rows, int k, void* q, void* sf, float* scale, cudaStream_t st) {
    if (rows == 0) return FLUX3_OK;
    const int rp = nvfp4_rows_padded(rows);
    prof_before(FLUX3_KERNEL_QUANTIZE, st);
    quantize_rows_nvfp4_kernel<<<rp / 8, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), rows, rp, k,
                                                       static_cast<uint8_t*>(q), static_cast<uint8_t*>(sf), scale);
    prof_after(st);
    return launch_status();
}

flux3_status run_out_proj(const flux3_dims* d, const flux3_block_weights* w, int n_w, const flux3_segments* segs, const void* y,
                          const void* x, void* x_out, int N, cudaStream_t st) {
    if (N == 0) return FLUX3_OK;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    const int D = d->width, F = d->ffn_hidden;
    const int K = D + F;
    if (!tmap_2d(&P.tm_a, y, K, N, (uint64_t)K * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    for (int i = 0; i < n_w; ++i) {
        if (!tmap_2d(&P.tm_b[i], w[i].w_out, K, D, (uint64_t)K * 2, 128)) return FLUX3_ERR_INVALID_ARG;
        P.ew[i] = {w[i].b_out, nullptr, nullptr};
    }
    fill_groups(P, segs->seg_off, segs->n_seg, n_w, N, 2);
    P.n_tiles = D / 256;
    P.k_blocks = K / GEMM_BK;
    P.width = D;
    P.x = static_cast<const __nv_bfloat16*>(x);
    P.x_out = static_cast<__nv_bfloat16*>(x_out);
    P.mod = segs->mod;
    P.n_seg = segs->n_seg;
    for (int i = 0; i <= segs->n_seg; ++i) P.seg_off[i] = segs->seg_off[i];
    return launch_gemm<256, EPI_GATED_RESIDUAL, 2>(P, st, FLUX3_KERNEL_OUT_PROJ);
}

// the output projection with the gated residual on quantized operands (one weight set):
// y_q [N, K] codes of [attention | SwiGLU] (K = D + F; e4m3: K bytes per row, NVFP4: K / 2
// with tiled block scales y_sf), sy their per-token scales; w_q W_out's codes [D, ...],
// w_sf its block scales (NVFP4), s_w its row scales
flux3_status run_out_proj_quant(const flux3_dims* d, bool nvfp4, const void* w_q, const void* w_sf, const float* s_w,
                                const float* b_out, const flux3_segments* segs, const void* y_q, const void* y_sf,
                                const float* sy, const void* x, void* x_out, int N, cudaStream_t st) {
    if (N == 0) return FLUX3_OK;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    const int D = d->width, F = d->ffn_hidden;
    const int K = D + F;
    const uint64_t row = nvfp4 ? (uint64_t)K / 2 : (uint64_t)K;
    if (!tmap_2d_u8(&P.tm_a, y_q, row, N, row, 128)) return FLUX3_ERR_INVALID_ARG;
    if (!tmap_2d_u8(&P.tm_b[0], w_q, row, D, row, 128)) return FLUX3_ERR_INVALID_ARG;
    P.ew[0] = {b_out, nullptr, nullptr, s_w, static_cast<const uint8_t*>(w_sf)};
    const int32_t one[2] = {0, N};
    fill_groups(P, one, 1, 1, N, 2);
    P.n_tiles = D / 256;
    P.k_blocks = nvfp4 ? K / 256 : K / 128;
    P.sf_steps = K / 64;
    P.a_scale = sy;
    P.a_sf = static_cast<const uint8_t*>(y_sf);
    P.width = D;
    P.x = static_cast<const __nv_bfloat16*>(x);
    P.x_out = static_cast<__nv_bfloat16*>(x_out);
    P.mod = segs->mod;
    P.n_seg = segs->n_seg;
    for (int i = 0; i <= segs->n_seg; ++i) P.seg_off[i] = segs->seg_off[i];
    if (nvfp4)
        return launch_pairs<gemm_nvf4_kernel<2, 4, EPI_GATED_RESIDUAL>>(P, Nvf4Cfg::SMEM_BYTES, gemm_threads(4), st,
                                                                        FLUX3_KERNEL_OUT_PROJ);
    return launch_gemm<256, EPI_GATED_RESIDUAL, 2, 1>(P, st, FLUX3_KERNEL_OUT_PROJ);
}

flux3_status run_attn(const flux3_dims* d, const void* q, const void* k, const void* vt, int ld_vt, int N, const int32_t* off,
                      int n_seg, void* out, int ld_out, bool f32, cudaStream_t st, float* lse = nullptr) {
    if (N == 0) return FLUX3_OK;
    const int H = d->heads;
    if (f32) {
        SegTable t;
        std::memset(&t, 0, sizeof t);
        t.n_seg = n_seg;
        for (int i = 0; i <= n_seg; ++i) t.off[i] = off[i];
        prof_before(FLUX3_KERNEL_ATTN_F32, st);
        attn_f32_kernel<<<dim3((N + 3) / 4, H), 128, 0, st>>>(static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                                                             static_cast<const __nv_bfloat16*>(vt), ld_vt, N, t,
                                                             static_cast<float*>(out), ld_out, 1.0f / sqrtf(128.f));
        prof_after(st);
        return launch_status();
    }
    AttnParams P;
    std::memset(&P, 0, sizeof P);
    if (!tmap_3d(&P.tm_q, q, 128, N, H, 256, (uint64_t)N * 256)) return FLUX3_ERR_INVALID_ARG;
    if (!tmap_3d(&P.tm_k, k, 128, N, H, 256, (uint64_t)N * 256)) return FLUX3_ERR_INVALID_ARG;
    if (!tmap_3d(&P.tm_v, vt, N, 128, H, (uint64_t)ld_vt * 2, (uint64_t)ld_vt * 256)) return FLUX3_ERR_INVALID_ARG;
    P.n_tokens = N;
    P.heads = H;
    P.n_seg = n_seg;
    int pairs = 0;  // one CTA per pair of 128-query tiles of one segment and head
    for (int s = 0; s < n_seg; ++s) {
        P.seg_off[s] = off[s];
        P.pair_begin[s] = pairs;
        pairs += (off[s + 1] - off[s] + 255) / 256;
    }
    P.seg_off[n_seg] = off[n_seg];
    P.pair_begin[n_seg] = pairs;
    P.out = static_cast<__nv_bfloat16*>(out);
    P.ld_out = ld_out;
    P.scale_log2 = (float)(1.4426950408889634 / std::sqrt(128.0));
    P.lse = lse;
    if (pairs == 0) return FLUX3_OK;
    if (!smem_attr_once<attn_tcgen05_kernel>(ATT_SMEM_BYTES)) return FLUX3_ERR_CUDA;
    prof_before(FLUX3_KERNEL_ATTN, st);
    attn_tcgen05_kernel<<<dim3(pairs, H), ATT_THREADS, ATT_SMEM_BYTES, st>>>(P);
    prof_after(st);
    return launch_status();
}

flux3_status run_block(const flux3_dims* d, const flux3_block_weights* w, int n_w, const flux3_segments* segs, const void* x,
                       void* x_out, int N, const float* rope, void* ws, size_t ws_bytes, cudaStream_t st, bool stage1) {
    flux3_status s = check_dims(d);
    if (s != FLUX3_OK) return s;
    if (N < 0 || N > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, N, true)) != FLUX3_OK) return s;
    if ((s = check_weights(w, n_w, true, true)) != FLUX3_OK) return s;
    if (N == 0) return FLUX3_OK;
    if (!x || !x_out || !rope || !al16(x) || !al16(x_out) || !al16(rope)) return FLUX3_ERR_INVALID_ARG;
    const BlockWs need = block_ws_layout(d, N, nullptr);
    if (!ws || !al256(ws) || ws_bytes < need.bytes) return FLUX3_ERR_WORKSPACE;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    const BlockWs b = block_ws_layout(d, N, static_cast<uint8_t*>(ws));
    const int D = d->width, F = d->ffn_hidden;
    const SegOffsets so = seg_table(segs->seg_off, segs->n_seg);
    if ((s = run_adaln(d, segs->mod, so, x, N, b.a, st)) != FLUX3_OK) return s;
    if ((s = run_in_proj(d, w, n_w, segs, b.a, N, rope, b.q, b.k, b.vt, b.ld_vt, b.y, st)) != FLUX3_OK) return s;
    const int32_t full[2] = {0, N};
    if (stage1) s = run_attn(d, b.q, b.k, b.vt, b.ld_vt, N, segs->seg_off, segs->n_seg, b.y, D + F, false, st);
    else s = run_attn(d, b.q, b.k, b.vt, b.ld_vt, N, full, 1, b.y, D + F, false, st);
    if (s != FLUX3_OK) return s;
    return run_out_proj(d, w, n_w, segs, b.y, x, x_out, N, st);
}

flux3_status run_final(const flux3_dims* d, const void* w_final, const float* b_final, int out_ch, const float* mod_final,
                       const void* x, int n_rows, float* out, void* ws, size_t ws_bytes, cudaStream_t st) {
    if (n_rows == 0) return FLUX3_OK;
    const int D = d->width;
    SegOffsets so;
    std::memset(&so, 0, sizeof so);
    so.n_seg = 1;
    so.off[1] = n_rows;
    flux3_status s = run_adaln(d, mod_final, so, x, n_rows, ws, st);
    if (s != FLUX3_OK) return s;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    if (!tmap_2d(&P.tm_a, ws, D, n_rows, (uint64_t)D * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    if (!tmap_2d(&P.tm_b[0], w_final, D, out_ch, (uint64_t)D * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    P.ew[0] = {b_final, nullptr, nullptr};
    P.n_groups = 1;
    P.grp[0] = {0, n_rows, 0, 0};
    P.m_tiles = (n_rows + GEMM_BM - 1) / GEMM_BM;
    P.n_tiles = out_ch / 128;
    P.k_blocks = D / GEMM_BK;
    P.width = D;
    P.out = out;
    P.ld_out = out_ch;
    P.n_cols = out_ch;
    return launch_gemm<128, EPI_F32, 1>(P, st, FLUX3_KERNEL_FINAL);
}

flux3_status run_linear(const flux3_dims* d, const void* x, int rows, int k, const void* w, const float* b, void* out,
                        int ld_out, cudaStream_t st) {
    if (rows == 0) return FLUX3_OK;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    const int D = d->width;
    if (!tmap_2d(&P.tm_a, x, k, rows, (uint64_t)k * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    if (!tmap_2d(&P.tm_b[0], w, k, D, (uint64_t)k * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    P.ew[0] = {b, nullptr, nullptr};
    const int32_t off[2] = {0, rows};
    fill_groups(P, off, 1, 1, rows, 1);
    P.n_tiles = D / 256;
    P.k_blocks = k / GEMM_BK;
    P.width = D;
    P.out_bf = static_cast<__nv_bfloat16*>(out);
    P.ld_out = ld_out;
    P.n_cols = D;
    return launch_gemm<256, EPI_BF16, 1>(P, st, FLUX3_KERNEL_LINEAR);
}

// C[M, N] = A[M, K] B[N, K]^T (+ bias): bf16 K-major operands with row strides in elements
// (multiples of 8), ragged M, N and K (the tensor maps read zeros past K and past the B
// rows; the epilogue stores only the N columns); C fp32 or bf16 with row stride ldc.
flux3_status run_gemm_plain(const void* A, int lda, const void* B, int ldb, int M, int N, int K, const float* bias,
                            void* C, int ldc, bool c_bf16, cudaStream_t st) {
    if (M == 0 || N == 0) return FLUX3_OK;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    if (!tmap_2d(&P.tm_a, A, K, M, (uint64_t)lda * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    if (!tmap_2d(&P.tm_b[0], B, K, N, (uint64_t)ldb * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    P.ew[0] = {bias, nullptr, nullptr};
    const int32_t off[2] = {0, M};
    fill_groups(P, off, 1, 1, M, 1);
    P.k_blocks = (K + GEMM_BK - 1) / GEMM_BK;
    P.n_cols = N;
    P.ld_out = ldc;
    if (c_bf16) P.out_bf = static_cast<__nv_bfloat16*>(C);
    else P.out = static_cast<float*>(C);
    if (N <= 128) {
        P.n_tiles = 1;
        return c_bf16 ? launch_gemm<128, EPI_BF16, 1>(P, st, FLUX3_KERNEL_BWD_GEMM)
                      : launch_gemm<128, EPI_F32, 1>(P, st, FLUX3_KERNEL_BWD_GEMM);
    }
    P.n_tiles = (N + 255) / 256;
    return c_bf16 ? launch_gemm<256, EPI_BF16, 1>(P, st, FLUX3_KERNEL_BWD_GEMM)
                  : launch_gemm<256, EPI_F32, 1>(P, st, FLUX3_KERNEL_BWD_GEMM);
}

// The attention-backward GEMMs with keys as rows and queries as columns (EPI_PROB_T: P^T
// from k q^T and the queries' log2-sum-exp2; EPI_DS_T: dS^T from v dO^T, P^T and the
// queries' rowsum(dO O)); bf16 C [M, N], row stride ldc.
template <int EPI>
flux3_status run_gemm_attn_t(const void* A, int lda, const void* B, int ldb, int M, int N, int K, const float* col_vec,
                             const void* aux, int ld_aux, float alpha, void* C, int ldc, cudaStream_t st) {
    if (M == 0 || N == 0) return FLUX3_OK;
    GemmParams P;
    std::memset(&P, 0, sizeof P);
    if (!tmap_2d(&P.tm_a, A, K, M, (uint64_t)lda * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    if (!tmap_2d(&P.tm_b[0], B, K, N, (uint64_t)ldb * 2, 128)) return FLUX3_ERR_INVALID_ARG;
    const int32_t off[2] = {0, M};
    fill_groups(P, off, 1, 1, M, 1);
    P.k_blocks = (K + GEMM_BK - 1) / GEMM_BK;
    P.n_tiles = (N + 255) / 256;
    P.n_cols = N;
    P.ld_out = ldc;
    P.out_bf = static_cast<__nv_bfloat16*>(C);
    P.col_vec = col_vec;
    P.aux = static_cast<const __nv_bfloat16*>(aux);
    P.ld_aux = ld_aux;
    P.alpha = alpha;
    return launch_gemm<256, EPI, 1, 0, 8>(P, st, FLUX3_KERNEL_BWD_GEMM);
}

// dst [cols, ld_dst] = src [rows, cols]^T (bf16; even strides, 4-byte aligned bases)
flux3_status run_transpose(const void* src, int rows, int cols, int ld_src, void* dst, int ld_dst, cudaStream_t st) {
    if (rows == 0 || cols == 0) return FLUX3_OK;
    if ((ld_src | ld_dst) & 1 || (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 3)
        return FLUX3_ERR_INVALID_ARG;
    prof_before(FLUX3_KERNEL_BWD_ELEM, st);
    transpose_bf16_kernel<<<dim3((unsigned)((cols + 63) / 64), (unsigned)((rows + 63) / 64)), dim3(32, 8), 0, st>>>(
        static_cast<const __nv_bfloat16*>(src), rows, cols, ld_src, static_cast<__nv_bfloat16*>(dst), ld_dst);
    prof_after(st);
    return launch_status();
}

flux3_status run_cfg_euler(float* latent, const float* vp, const float* vn, long long n, float s, float dt,
                           __nv_bfloat16* lat_bf, cudaStream_t st) {
    if (n == 0) return FLUX3_OK;
    const int sms = sm_count();
    if (sms <= 0) return FLUX3_ERR_CUDA;
    long long blocks = (n + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    prof_before(FLUX3_KERNEL_CFG_EULER, st);
    cfg_euler_kernel<<<(unsigned)blocks, 256, 0, st>>>(latent, vp, vn, n, s, dt, lat_bf);
    prof_after(st);
    return launch_status();
}

void sigma_schedule(int n_steps, double alpha, float* out) {
    for (int i = 0; i <= n_steps; ++i) {
        const double x = 1.0 - (double)i / n_steps;
        out[i] = (float)(alpha * x / (1.0 + (alpha - 1.0) * x));
    }
}

// workspace of the sampling loop: tokens | reference+text context (prompt) | context
// (negative prompt, with guidance) | latent in bf16 | velocities | the denoiser's workspace
struct SampleWs {
    __nv_bfloat16 *tokens, *ctx_pos, *ctx_neg, *lat_bf;
    float *v_pos, *v_neg;
    uint8_t* dit;
    size_t dit_bytes, bytes;
};
SampleWs sample_ws_layout(const flux3_dims* d, const flux3_sample_args* a, uint8_t* base) {
    SampleWs w;
    const size_t D = d->width, N = (size_t)a->n_img + a->n_ref + a->n_txt, nc = (size_t)a->n_ref + a->n_txt;
    const bool cfg = a->cfg_scale != 1.f;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = base ? base + off : nullptr;
        off += up256(bytes);
        return p;
    };
    w.tokens = reinterpret_cast<__nv_bfloat16*>(take(N * D * 2));
    w.ctx_pos = reinterpret_cast<__nv_bfloat16*>(take(nc * D * 2));
    w.ctx_neg = cfg ? reinterpret_cast<__nv_bfloat16*>(take(nc * D * 2)) : nullptr;
    w.lat_bf = reinterpret_cast<__nv_bfloat16*>(take((size_t)a->n_img * a->latent_channels * 2));
    w.v_pos = reinterpret_cast<float*>(take((size_t)a->n_img * a->latent_channels * 4));
    w.v_neg = cfg ? reinterpret_cast<float*>(take((size_t)a->n_img * a->latent_channels * 4)) : nullptr;
    w.dit_bytes = flux3_dit_workspace_size(d, a->n_img, a->n_ref, a->n_txt);
    w.dit = take(w.dit_bytes);
    w.bytes = off;
    return w;
}

}  // namespace

// result slot of the bounded-wait diagnostic (flux3_selftest_timeout)
static __device__ int g_selftest_result;

// ---------------------------------------------------------------- static scratch
// Scratch for flux3_block_fwd_static: one file-scope device array.  Host code may not use
// the symbol as an address; the device address is looked up once per device.
static __device__ __align__(256) unsigned char g_static_scratch[FLUX3_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

flux3_status static_scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FLUX3_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FLUX3_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return FLUX3_ERR_CUDA;
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return FLUX3_OK;
}
}  // namespace

// ====================================================================== C-ABI
extern "C" {

const char* flux3_status_string(flux3_status s) {
    switch (s) {
        case FLUX3_OK: return "ok";
        case FLUX3_ERR_INVALID_ARG: return "invalid argument";
        case FLUX3_ERR_UNSUPPORTED: return "unsupported configuration";
        case FLUX3_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case FLUX3_ERR_CUDA: return "CUDA error";
        case FLUX3_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

const char* flux3_version(void) { return "flux3-b300 0.1 (sm_103a, tcgen05)"; }

flux3_status flux3_rope_build(const flux3_dims* dims, const int32_t* pos, int32_t n_tokens, float* rope, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if (n_tokens == 0) return FLUX3_OK;
    if (!pos || !rope || !al16(pos) || !al16(rope)) return FLUX3_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const long long total = (long long)n_tokens * 64;
    prof_before(FLUX3_KERNEL_ROPE, st);
    RopeFreqs fr;
    for (int j = 0; j < 16; ++j) {
        const double g = std::pow((double)dims->rope_theta, -(double)(2 * j) / 32.0) / 6.283185307179586476925286766559;
        fr.hi[j] = (float)g;
        fr.lo[j] = (float)(g - (double)fr.hi[j]);
    }
    rope_table_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(pos, n_tokens, fr, reinterpret_cast<float2*>(rope));
    prof_after(st);
    return launch_status();
}

flux3_status flux3_adaln_fwd(const flux3_dims* dims, const flux3_segments* segs, const void* x, int32_t n_tokens, void* a,
                             flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, n_tokens, true)) != FLUX3_OK) return s;
    if (n_tokens == 0) return FLUX3_OK;
    if (!x || !a || !al16(x) || !al16(a) || x == a) return FLUX3_ERR_INVALID_ARG;
    return run_adaln(dims, segs->mod, seg_table(segs->seg_off, segs->n_seg), x, n_tokens, a,
                     reinterpret_cast<cudaStream_t>(stream));
}

flux3_status flux3_in_proj_fwd(const flux3_dims* dims, const flux3_block_weights* w, int32_t n_w, const flux3_segments* segs,
                               const void* a, int32_t n_tokens, const float* rope, void* q, void* k, void* vt, int32_t ld_vt,
                               void* y, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, n_tokens, false)) != FLUX3_OK) return s;
    if ((s = check_weights(w, n_w, true, false)) != FLUX3_OK) return s;
    if (n_w != 1 && n_w != segs->n_seg) return FLUX3_ERR_INVALID_ARG;
    if (n_tokens == 0) return FLUX3_OK;
    if (!a || !rope || !q || !k || !vt || !y) return FLUX3_ERR_INVALID_ARG;
    if (!al16(a) || !al16(rope) || !al16(q) || !al16(k) || !al16(vt) || !al16(y)) return FLUX3_ERR_INVALID_ARG;
    if (ld_vt < n_tokens || ld_vt % 8 != 0) return FLUX3_ERR_INVALID_ARG;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    return run_in_proj(dims, w, n_w, segs, a, n_tokens, rope, q, k, vt, ld_vt, y, reinterpret_cast<cudaStream_t>(stream));
}

flux3_status flux3_attn_fwd(const flux3_dims* dims, const void* q, const void* k, const void* vt, int32_t ld_vt, int32_t n_tokens,
                            const int32_t* seg_off, int32_t n_seg, void* out, int32_t ld_out, int32_t fp32_debug,
                            flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    const int32_t full[2] = {0, n_tokens};
    if (!seg_off) {
        if (n_seg != 1 && n_seg != 0) return FLUX3_ERR_INVALID_ARG;
        seg_off = full;
        n_seg = 1;
    }
    if ((s = check_offsets(seg_off, n_seg, n_tokens)) != FLUX3_OK) return s;
    if (n_tokens == 0) return FLUX3_OK;
    if (!q || !k || !vt || !out || !al16(q) || !al16(k) || !al16(vt) || !al16(out)) return FLUX3_ERR_INVALID_ARG;
    if (ld_vt < n_tokens || ld_vt % 8 != 0) return FLUX3_ERR_INVALID_ARG;
    if (ld_out < dims->width || ld_out % 8 != 0) return FLUX3_ERR_INVALID_ARG;
    if (!fp32_debug && !have_encode()) return FLUX3_ERR_CUDA;
    return run_attn(dims, q, k, vt, ld_vt, n_tokens, seg_off, n_seg, out, ld_out, fp32_debug != 0,
                    reinterpret_cast<cudaStream_t>(stream));
}

flux3_status flux3_out_proj_fwd(const flux3_dims* dims, const flux3_block_weights* w, int32_t n_w, const flux3_segments* segs,
                                const void* y, const void* x, void* x_out, int32_t n_tokens, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, n_tokens, true)) != FLUX3_OK) return s;
    if ((s = check_weights(w, n_w, false, true)) != FLUX3_OK) return s;
    if (n_w != 1 && n_w != segs->n_seg) return FLUX3_ERR_INVALID_ARG;
    if (n_tokens == 0) return FLUX3_OK;
    if (!y || !x || !x_out || !al16(y) || !al16(x) || !al16(x_out)) return FLUX3_ERR_INVALID_ARG;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    return run_out_proj(dims, w, n_w, segs, y, x, x_out, n_tokens, reinterpret_cast<cudaStream_t>(stream));
}

size_t flux3_block_workspace_size(const flux3_dims* dims, int32_t n_tokens) {
    if (check_dims(dims) != FLUX3_OK || n_tokens < 0 || n_tokens > kMaxTokens) return 0;
    return block_ws_layout(dims, n_tokens, nullptr).bytes;
}

flux3_status flux3_block_fwd(const flux3_dims* dims, const flux3_block_weights* w, const flux3_segments* segs, const void* x,
                             void* x_out, int32_t n_tokens, const float* rope, void* ws, size_t ws_bytes, flux3_stream_t stream) {
    return run_block(dims, w, 1, segs, x, x_out, n_tokens, rope, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), false);
}

flux3_status flux3_stream_block_fwd(const flux3_dims* dims, const flux3_block_weights* w, const flux3_segments* segs,
                                    const void* x, void* x_out, int32_t n_tokens, const float* rope, void* ws, size_t ws_bytes,
                                    flux3_stream_t stream) {
    if (!segs) return FLUX3_ERR_INVALID_ARG;
    return run_block(dims, w, segs->n_seg, segs, x, x_out, n_tokens, rope, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream),
                     true);
}

flux3_status flux3_final_fwd(const flux3_dims* dims, const void* w_final, const float* b_final, int32_t out_channels,
                             const float* mod_final, const void* x, int32_t n_rows, float* out, void* ws, size_t ws_bytes,
                             flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (n_rows < 0 || n_rows > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if (out_channels <= 0 || out_channels > 4096) return FLUX3_ERR_INVALID_ARG;
    if (out_channels % 128 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (n_rows == 0) return FLUX3_OK;
    if (!w_final || !mod_final || !x || !out || !al16(w_final) || !al16(mod_final) || !al16(x) || !al16(out) ||
        (b_final && !al16(b_final)))
        return FLUX3_ERR_INVALID_ARG;
    if (!ws || !al256(ws) || ws_bytes < up256((size_t)n_rows * dims->width * 2)) return FLUX3_ERR_WORKSPACE;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    return run_final(dims, w_final, b_final, out_channels, mod_final, x, n_rows, out, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

namespace {
// Row offsets of the denoiser's streams in the token buffer: image | [reference] | text.
struct DitStreams {
    int n;          // 2 or 3
    int32_t off[4];  // off[i] .. off[i + 1]: the rows of stream i
};
DitStreams dit_streams(int ns, int n_img, int n_ref, int n_txt) {
    DitStreams d;
    d.n = ns;
    d.off[0] = 0;
    d.off[1] = n_img;
    d.off[2] = ns == 3 ? n_img + n_ref : n_img + n_txt;
    d.off[3] = ns == 3 ? n_img + n_ref + n_txt : 0;
    return d;
}

// The denoiser's weights: counts, pointers and the output layer's shape.
flux3_status check_dit(const flux3_dims* d, const flux3_dit_weights* w) {
    (void)d;
    if (w->n_streams < 2 || w->n_streams > 3) return FLUX3_ERR_INVALID_ARG;
    if (w->n_stage1 < 0 || w->n_joint < 0 || (w->n_stage1 > 0 && !w->stage1) || (w->n_joint > 0 && !w->joint))
        return FLUX3_ERR_INVALID_ARG;
    if (w->out_channels <= 0 || w->out_channels > 4096) return FLUX3_ERR_INVALID_ARG;
    if (w->out_channels % 128 != 0) return FLUX3_ERR_UNSUPPORTED;
    flux3_status s;
    for (int i = 0; i < w->n_stage1; ++i)
        if ((s = check_weights(w->stage1 + (size_t)i * w->n_streams, w->n_streams, true, true)) != FLUX3_OK) return s;
    for (int i = 0; i < w->n_joint; ++i)
        if ((s = check_weights(w->joint + i, 1, true, true)) != FLUX3_OK) return s;
    return FLUX3_OK;
}

// Stage 1 (each stream through its own blocks, attention within the stream) for streams
// s0 .. s1-1, whose rows start at x (bf16, updated in place); rope holds the table rows
// of those tokens.  mod_stage1 is the denoiser's [n_stage1][n_streams][3][D] array.
flux3_status dit_stage1(const flux3_dims* d, const flux3_dit_weights* w, const float* mod_stage1, const DitStreams& ds,
                        int s0, int s1, void* x, const float* rope, void* bws, size_t bws_bytes, cudaStream_t st) {
    const int n_seg = s1 - s0, N = ds.off[s1] - ds.off[s0];
    if (n_seg <= 0 || N == 0) return FLUX3_OK;
    int32_t loc[FLUX3_MAX_SEGMENTS + 1];
    for (int i = 0; i <= n_seg; ++i) loc[i] = ds.off[s0 + i] - ds.off[s0];
    const size_t mstride = (size_t)ds.n * 3 * d->width;
    for (int b = 0; b < w->n_stage1; ++b) {
        flux3_segments sg{n_seg, loc, mod_stage1 + b * mstride + (size_t)s0 * 3 * d->width};
        const flux3_status s =
            run_block(d, w->stage1 + (size_t)b * ds.n + s0, n_seg, &sg, x, x, N, rope, bws, bws_bytes, st, true);
        if (s != FLUX3_OK) return s;
    }
    return FLUX3_OK;
}

// Stage 2 (the joint blocks over all tokens) and the output layer on the image rows.
flux3_status dit_stage2(const flux3_dims* d, const flux3_dit_weights* w, const flux3_dit_mod* mod, const DitStreams& ds,
                        void* tokens, const float* rope, float* velocity, void* bws, size_t bws_bytes, cudaStream_t st) {
    const int N = ds.off[ds.n];
    const size_t mstride = (size_t)ds.n * 3 * d->width;
    for (int b = 0; b < w->n_joint; ++b) {
        flux3_segments sg{ds.n, ds.off, mod->joint + b * mstride};
        const flux3_status s = run_block(d, w->joint + b, 1, &sg, tokens, tokens, N, rope, bws, bws_bytes, st, false);
        if (s != FLUX3_OK) return s;
    }
    return run_final(d, w->w_final, w->b_final, w->out_channels, mod->final, tokens, ds.off[1], velocity, bws, bws_bytes,
                     st);
}
}  // namespace

size_t flux3_dit_workspace_size(const flux3_dims* dims, int32_t n_img, int32_t n_ref, int32_t n_txt) {
    if (check_dims(dims) != FLUX3_OK || n_img < 0 || n_ref < 0 || n_txt < 0) return 0;
    const long long N = (long long)n_img + n_ref + n_txt;
    if (N > kMaxTokens) return 0;
    return up256((size_t)N * 128 * 4) + block_ws_layout(dims, (int)N, nullptr).bytes;
}

flux3_status flux3_dit_fwd(const flux3_dims* dims, const flux3_dit_weights* w, const flux3_dit_mod* mod, void* tokens,
                           int32_t n_img, int32_t n_ref, int32_t n_txt, const int32_t* pos, float* velocity, void* ws,
                           size_t ws_bytes, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (!w || !mod || n_img < 0 || n_ref < 0 || n_txt < 0) return FLUX3_ERR_INVALID_ARG;
    const long long NN = (long long)n_img + n_ref + n_txt;
    if (NN > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    const int N = (int)NN;
    if (w->n_streams != (n_ref > 0 ? 3 : 2)) return FLUX3_ERR_INVALID_ARG;
    if ((w->n_stage1 > 0 && !mod->stage1) || (w->n_joint > 0 && !mod->joint)) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_dit(dims, w)) != FLUX3_OK) return s;
    if (N == 0) return FLUX3_OK;
    if (!tokens || !pos || !velocity || !w->w_final || !mod->final) return FLUX3_ERR_INVALID_ARG;
    if (!al16(tokens) || !al16(pos) || !al16(velocity)) return FLUX3_ERR_INVALID_ARG;
    if (!ws || !al256(ws) || ws_bytes < flux3_dit_workspace_size(dims, n_img, n_ref, n_txt)) return FLUX3_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* rope = static_cast<float*>(ws);
    uint8_t* bws = static_cast<uint8_t*>(ws) + up256((size_t)N * 128 * 4);
    const size_t bws_bytes = ws_bytes - up256((size_t)N * 128 * 4);
    if ((s = flux3_rope_build(dims, pos, N, rope, stream)) != FLUX3_OK) return s;
    const DitStreams ds = dit_streams(w->n_streams, n_img, n_ref, n_txt);
    if ((s = dit_stage1(dims, w, mod->stage1, ds, 0, ds.n, tokens, rope, bws, bws_bytes, st)) != FLUX3_OK) return s;
    return dit_stage2(dims, w, mod, ds, tokens, rope, velocity, bws, bws_bytes, st);
}

flux3_status flux3_block_fwd_static(const flux3_dims* dims, const flux3_block_weights* w, const flux3_segments* segs,
                                    const void* x, void* x_out, int32_t n_tokens, const float* rope, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if (block_ws_layout(dims, n_tokens, nullptr).bytes > FLUX3_STATIC_SCRATCH_BYTES) return FLUX3_ERR_WORKSPACE;
    void* ws = nullptr;
    if (n_tokens > 0 && (s = static_scratch_address(&ws)) != FLUX3_OK) return s;
    return run_block(dims, w, 1, segs, x, x_out, n_tokens, rope, ws, FLUX3_STATIC_SCRATCH_BYTES,
                     reinterpret_cast<cudaStream_t>(stream), false);
}

flux3_status flux3_euler_step(float* latent, const float* velocity, int64_t n, float sigma, float sigma_next, flux3_stream_t stream) {
    if (n < 0 || (n > 0 && (!latent || !velocity))) return FLUX3_ERR_INVALID_ARG;
    if (n == 0) return FLUX3_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int sms = sm_count();
    if (sms <= 0) return FLUX3_ERR_CUDA;
    long long blocks = (n + 255) / 256;
    if (blocks > 8LL * sms) blocks = 8LL * sms;
    prof_before(FLUX3_KERNEL_EULER, st);
    euler_kernel<<<(unsigned)blocks, 256, 0, st>>>(latent, velocity, n, sigma_next - sigma);
    prof_after(st);
    return launch_status();
}

flux3_status flux3_sigma_schedule(int32_t n_steps, float alpha, float* sigmas) {
    if (n_steps < 1 || !sigmas || !(alpha > 0.f) || !std::isfinite(alpha)) return FLUX3_ERR_INVALID_ARG;
    sigma_schedule(n_steps, alpha, sigmas);
    return FLUX3_OK;
}

flux3_status flux3_linear_fwd(const flux3_dims* dims, const void* x, int32_t rows, int32_t k, const void* w, const float* b,
                              void* out, int32_t ld_out, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (rows < 0 || rows > kMaxTokens || k <= 0 || k > (1 << 20)) return FLUX3_ERR_INVALID_ARG;
    if (k % GEMM_BK != 0 || dims->width % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (rows == 0) return FLUX3_OK;
    if (!x || !w || !out || !al16(x) || !al16(w) || !al16(out) || (b && !al16(b))) return FLUX3_ERR_INVALID_ARG;
    if (ld_out < dims->width || ld_out % 8 != 0) return FLUX3_ERR_INVALID_ARG;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    return run_linear(dims, x, rows, k, w, b, out, ld_out, reinterpret_cast<cudaStream_t>(stream));
}

flux3_status flux3_cfg_euler_step(float* latent, const float* v_pos, const float* v_neg, int64_t n, float cfg_scale,
                                  float sigma, float sigma_next, void* latent_bf16, flux3_stream_t stream) {
    if (n < 0 || (n > 0 && (!latent || !v_pos))) return FLUX3_ERR_INVALID_ARG;
    if (!std::isfinite(cfg_scale) || !std::isfinite(sigma) || !std::isfinite(sigma_next)) return FLUX3_ERR_INVALID_ARG;
    return run_cfg_euler(latent, v_pos, v_neg, n, cfg_scale, sigma_next - sigma, static_cast<__nv_bfloat16*>(latent_bf16),
                         reinterpret_cast<cudaStream_t>(stream));
}

static flux3_status check_sample_args(const flux3_dims* d, const flux3_sample_args* a) {
    flux3_status s = check_dims(d);
    if (s != FLUX3_OK) return s;
    if (!a || a->n_img < 0 || a->n_ref < 0 || a->n_txt < 0 || a->n_steps < 1 || a->n_steps > 100000) return FLUX3_ERR_INVALID_ARG;
    if ((long long)a->n_img + a->n_ref + a->n_txt > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if (!(a->alpha > 0.f) || !std::isfinite(a->alpha) || !std::isfinite(a->cfg_scale)) return FLUX3_ERR_INVALID_ARG;
    if (a->latent_channels <= 0 || a->text_dim <= 0 || a->text_dim > (1 << 20) || a->latent_channels > 4096)
        return FLUX3_ERR_INVALID_ARG;
    if (a->latent_channels % GEMM_BK != 0 || a->text_dim % GEMM_BK != 0 || d->width % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (!a->w_img || !al16(a->w_img) || (a->b_img && !al16(a->b_img))) return FLUX3_ERR_INVALID_ARG;
    if (a->n_txt > 0 && (!a->w_txt || !al16(a->w_txt) || (a->b_txt && !al16(a->b_txt)) || !a->text_pos ||
                         !al16(a->text_pos)))
        return FLUX3_ERR_INVALID_ARG;
    if (a->n_txt > 0 && a->cfg_scale != 1.f && (!a->text_neg || !al16(a->text_neg))) return FLUX3_ERR_INVALID_ARG;
    if (a->n_ref > 0 && (!a->ref_latent || !al16(a->ref_latent))) return FLUX3_ERR_INVALID_ARG;
    if (!a->pos || !al16(a->pos) || !a->mod) return FLUX3_ERR_INVALID_ARG;
    return FLUX3_OK;
}

size_t flux3_sample_workspace_size(const flux3_dims* dims, const flux3_sample_args* a) {
    if (check_sample_args(dims, a) != FLUX3_OK) return 0;
    return sample_ws_layout(dims, a, nullptr).bytes;
}

flux3_status flux3_sample_fwd(const flux3_dims* dims, const flux3_dit_weights* w, const flux3_sample_args* a, float* latent,
                              void* ws, size_t ws_bytes, flux3_stream_t stream) {
    flux3_status s = check_sample_args(dims, a);
    if (s != FLUX3_OK) return s;
    if (!w || w->out_channels != a->latent_channels) return FLUX3_ERR_INVALID_ARG;
    if (w->n_streams != (a->n_ref > 0 ? 3 : 2)) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_dit(dims, w)) != FLUX3_OK) return s;
    for (int i = 0; i < a->n_steps; ++i)
        if ((w->n_stage1 > 0 && !a->mod[i].stage1) || (w->n_joint > 0 && !a->mod[i].joint) || !a->mod[i].final)
            return FLUX3_ERR_INVALID_ARG;
    if (a->n_img == 0) return FLUX3_OK;
    if (!latent || !al16(latent) || !w->w_final) return FLUX3_ERR_INVALID_ARG;
    const SampleWs need = sample_ws_layout(dims, a, nullptr);
    if (!ws || !al256(ws) || ws_bytes < need.bytes) return FLUX3_ERR_WORKSPACE;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const SampleWs b = sample_ws_layout(dims, a, static_cast<uint8_t*>(ws));
    const int D = dims->width, C = a->latent_channels;
    const bool cfg = a->cfg_scale != 1.f;
    const long long n_lat = (long long)a->n_img * C;
    const size_t ctx_bytes = ((size_t)a->n_ref + a->n_txt) * D * 2;
    std::vector<float> sig(a->n_steps + 1);
    sigma_schedule(a->n_steps, a->alpha, sig.data());
    // the clean context (references, text) is embedded once
    for (int k = 0; k < (cfg ? 2 : 1); ++k) {
        __nv_bfloat16* ctx = k == 0 ? b.ctx_pos : b.ctx_neg;
        if ((s = run_linear(dims, a->ref_latent, a->n_ref, C, a->w_img, a->b_img, ctx, D, st)) != FLUX3_OK) return s;
        if ((s = run_linear(dims, k == 0 ? a->text_pos : a->text_neg, a->n_txt, a->text_dim, a->w_txt, a->b_txt,
                            ctx + (size_t)a->n_ref * D, D, st)) != FLUX3_OK)
            return s;
    }
    prof_before(FLUX3_KERNEL_TO_BF16, st);
    to_bf16_kernel<<<(unsigned)((n_lat + 255) / 256), 256, 0, st>>>(latent, n_lat, b.lat_bf);
    prof_after(st);
    if ((s = launch_status()) != FLUX3_OK) return s;
    const bool cache = a->cache_context != 0 && ctx_bytes > 0 && w->n_stage1 > 0;
    const DitStreams ds = dit_streams(w->n_streams, a->n_img, a->n_ref, a->n_txt);
    const int N = ds.off[ds.n];
    float* rope = reinterpret_cast<float*>(b.dit);
    uint8_t* bws = b.dit + up256((size_t)N * 128 * 4);
    const size_t bws_bytes = b.dit_bytes - up256((size_t)N * 128 * 4);
    if (cache) {
        // The reference and text streams see the same modulation at every step (step 0's)
        // and attend only to themselves in stage 1, so their stage-1 output does not
        // depend on the step: compute it once per prompt, in place in the context buffers.
        if ((s = flux3_rope_build(dims, a->pos, N, rope, stream)) != FLUX3_OK) return s;
        for (int k = 0; k < (cfg ? 2 : 1); ++k)
            if ((s = dit_stage1(dims, w, a->mod[0].stage1, ds, 1, ds.n, k == 0 ? b.ctx_pos : b.ctx_neg,
                                rope + (size_t)a->n_img * 128, bws, bws_bytes, st)) != FLUX3_OK)
                return s;
    }
    for (int i = 0; i < a->n_steps; ++i) {
        for (int k = 0; k < (cfg ? 2 : 1); ++k) {
            // the denoiser overwrites the token buffer: rebuild it for every call
            if ((s = run_linear(dims, b.lat_bf, a->n_img, C, a->w_img, a->b_img, b.tokens, D, st)) != FLUX3_OK) return s;
            if (ctx_bytes > 0 &&
                cudaMemcpyAsync(b.tokens + (size_t)a->n_img * D, k == 0 ? b.ctx_pos : b.ctx_neg, ctx_bytes,
                                cudaMemcpyDeviceToDevice, st) != cudaSuccess)
                return FLUX3_ERR_CUDA;
            float* v = k == 0 ? b.v_pos : b.v_neg;
            if (!cache) {
                if ((s = flux3_dit_fwd(dims, w, &a->mod[i], b.tokens, a->n_img, a->n_ref, a->n_txt, a->pos, v, b.dit,
                                       b.dit_bytes, stream)) != FLUX3_OK)
                    return s;
                continue;
            }
            if ((s = dit_stage1(dims, w, a->mod[i].stage1, ds, 0, 1, b.tokens, rope, bws, bws_bytes, st)) != FLUX3_OK ||
                (s = dit_stage2(dims, w, &a->mod[i], ds, b.tokens, rope, v, bws, bws_bytes, st)) != FLUX3_OK)
                return s;
        }
        if ((s = run_cfg_euler(latent, b.v_pos, cfg ? b.v_neg : nullptr, n_lat, a->cfg_scale, sig[i + 1] - sig[i], b.lat_bf,
                               st)) != FLUX3_OK)
            return s;
    }
    return FLUX3_OK;
}

flux3_status flux3_quantize_rows_fp8(const void* x, int32_t rows, int32_t k, void* q, float* scale, flux3_stream_t stream) {
    if (rows < 0 || rows > kMaxTokens * 16 || k <= 0 || k > (1 << 20)) return FLUX3_ERR_INVALID_ARG;
    if (k % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (rows == 0) return FLUX3_OK;
    if (!x || !q || !scale || !al16(x) || !al16(q)) return FLUX3_ERR_INVALID_ARG;
    return run_quantize_rows(x, rows, k, q, scale, reinterpret_cast<cudaStream_t>(stream));
}

static flux3_status check_weights_fp8(const flux3_block_weights_fp8* w, int n_w) {
    if (!w || n_w < 1 || n_w > FLUX3_MAX_SEGMENTS) return FLUX3_ERR_INVALID_ARG;
    for (int i = 0; i < n_w; ++i)
        if (!w[i].w_in || !al16(w[i].w_in) || !w[i].s_in || !al16(w[i].s_in) || !w[i].q_norm || !al16(w[i].q_norm) ||
            !w[i].k_norm || !al16(w[i].k_norm) || (w[i].b_in && !al16(w[i].b_in)))
            return FLUX3_ERR_INVALID_ARG;
    return FLUX3_OK;
}

flux3_status flux3_in_proj_fp8_fwd(const flux3_dims* dims, const flux3_block_weights_fp8* w, int32_t n_w,
                                   const flux3_segments* segs, const void* a8, const float* sa, int32_t n_tokens,
                                   const float* rope, void* q, void* k, void* vt, int32_t ld_vt, void* y,
                                   flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (dims->width % 128 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, n_tokens, false)) != FLUX3_OK) return s;
    if ((s = check_weights_fp8(w, n_w)) != FLUX3_OK) return s;
    if (n_w != 1 && n_w != segs->n_seg) return FLUX3_ERR_INVALID_ARG;
    if (n_tokens == 0) return FLUX3_OK;
    if (!a8 || !sa || !rope || !q || !k || !vt || !y) return FLUX3_ERR_INVALID_ARG;
    if (!al16(a8) || !al16(rope) || !al16(q) || !al16(k) || !al16(vt) || !al16(y)) return FLUX3_ERR_INVALID_ARG;
    if (ld_vt < n_tokens || ld_vt % 8 != 0) return FLUX3_ERR_INVALID_ARG;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    return run_in_proj_fp8(dims, w, n_w, segs, a8, sa, n_tokens, rope, q, k, vt, ld_vt, y,
                           reinterpret_cast<cudaStream_t>(stream));
}

namespace {
// the quantized block's scratch after the bf16 block's: the input projection's codes,
// block scales (NVFP4) and row scales, then the output projection's
struct QuantWs {
    uint8_t *a_q, *a_sf, *y_q, *y_sf;
    float *sa, *sy;
    size_t bytes;
};
QuantWs quant_ws(const flux3_dims* d, int N, bool nvfp4, uint8_t* base) {
    const int D = d->width, K = d->width + d->ffn_hidden;
    QuantWs w;
    size_t off = block_ws_layout(d, N, nullptr).bytes;
    auto take = [&](size_t bytes) {
        uint8_t* p = base ? base + off : nullptr;
        off += up256(bytes);
        return p;
    };
    const size_t rp = (size_t)nvfp4_rows_padded(N);
    w.a_q = take((size_t)N * (nvfp4 ? D / 2 : D));
    w.a_sf = nvfp4 ? take(rp * (D / 16)) : nullptr;
    w.sa = reinterpret_cast<float*>(take((size_t)N * 4));
    w.y_q = take((size_t)N * (nvfp4 ? K / 2 : K));
    w.y_sf = nvfp4 ? take(rp * (K / 16)) : nullptr;
    w.sy = reinterpret_cast<float*>(take((size_t)N * 4));
    w.bytes = off;
    return w;
}
}  // namespace

size_t flux3_block_fp8_workspace_size(const flux3_dims* dims, int32_t n_tokens) {
    if (check_dims(dims) != FLUX3_OK || n_tokens < 0 || n_tokens > kMaxTokens) return 0;
    return quant_ws(dims, n_tokens, false, nullptr).bytes;
}

flux3_status flux3_block_fp8_fwd(const flux3_dims* dims, const flux3_block_weights_fp8* w, const flux3_segments* segs,
                                 const void* x, void* x_out, int32_t n_tokens, const float* rope, void* ws, size_t ws_bytes,
                                 flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (dims->width % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    const int N = n_tokens;
    if (N < 0 || N > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, N, true)) != FLUX3_OK) return s;
    if ((s = check_weights_fp8(w, 1)) != FLUX3_OK) return s;
    if (w->b_out && !al16(w->b_out)) return FLUX3_ERR_INVALID_ARG;
    if (w->w_out_q ? (!al16(w->w_out_q) || !w->s_out) : (!w->w_out || !al16(w->w_out))) return FLUX3_ERR_INVALID_ARG;
    if ((dims->width + dims->ffn_hidden) % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (N == 0) return FLUX3_OK;
    if (!x || !x_out || !rope || !al16(x) || !al16(x_out) || !al16(rope)) return FLUX3_ERR_INVALID_ARG;
    if (!ws || !al256(ws) || ws_bytes < flux3_block_fp8_workspace_size(dims, N)) return FLUX3_ERR_WORKSPACE;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const BlockWs b = block_ws_layout(dims, N, static_cast<uint8_t*>(ws));
    const QuantWs qw = quant_ws(dims, N, false, static_cast<uint8_t*>(ws));
    const int D = dims->width, F = dims->ffn_hidden;
    if ((s = run_adaln(dims, segs->mod, seg_table(segs->seg_off, segs->n_seg), x, N, b.a, st)) != FLUX3_OK) return s;
    if ((s = run_quantize_rows(b.a, N, D, qw.a_q, qw.sa, st)) != FLUX3_OK) return s;
    if ((s = run_in_proj_fp8(dims, w, 1, segs, qw.a_q, qw.sa, N, rope, b.q, b.k, b.vt, b.ld_vt, b.y, st)) != FLUX3_OK)
        return s;
    const int32_t full[2] = {0, N};
    if ((s = run_attn(dims, b.q, b.k, b.vt, b.ld_vt, N, full, 1, b.y, D + F, false, st)) != FLUX3_OK) return s;
    if (w->w_out_q) {
        if ((s = run_quantize_rows(b.y, N, D + F, qw.y_q, qw.sy, st)) != FLUX3_OK) return s;
        return run_out_proj_quant(dims, false, w->w_out_q, nullptr, w->s_out, w->b_out, segs, qw.y_q, nullptr, qw.sy, x,
                                  x_out, N, st);
    }
    const flux3_block_weights wo{nullptr, nullptr, nullptr, nullptr, w->w_out, w->b_out};
    return run_out_proj(dims, &wo, 1, segs, b.y, x, x_out, N, st);
}

size_t flux3_nvfp4_scale_bytes(int32_t rows, int32_t k) {
    if (rows < 0 || rows > kMaxTokens * 16 || k <= 0 || k > (1 << 20) || k % 64 != 0) return 0;
    return (size_t)nvfp4_rows_padded(rows) * (size_t)(k / 16);
}

flux3_status flux3_quantize_rows_nvfp4(const void* x, int32_t rows, int32_t k, void* q, void* sf, float* scale,
                                       flux3_stream_t stream) {
    if (rows < 0 || rows > kMaxTokens * 16 || k <= 0 || k > (1 << 20)) return FLUX3_ERR_INVALID_ARG;
    if (k % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (rows == 0) return FLUX3_OK;
    if (!x || !q || !sf || !scale || !al16(x) || !al16(q) || !al16(sf)) return FLUX3_ERR_INVALID_ARG;
    return run_quantize_rows_nvfp4(x, rows, k, q, sf, scale, reinterpret_cast<cudaStream_t>(stream));
}

static flux3_status check_weights_nvfp4(const flux3_block_weights_nvfp4* w) {
    if (!w || !w->w_in || !al16(w->w_in) || !w->w_sf || !al16(w->w_sf) || !w->s_in || !w->q_norm || !al16(w->q_norm) ||
        !w->k_norm || !al16(w->k_norm) || (w->b_in && !al16(w->b_in)))
        return FLUX3_ERR_INVALID_ARG;
    return FLUX3_OK;
}

flux3_status flux3_in_proj_nvfp4_fwd(const flux3_dims* dims, const flux3_block_weights_nvfp4* w, const void* a4,
                                     const void* a_sf, const float* sa, int32_t n_tokens, const float* rope, void* q,
                                     void* k, void* vt, int32_t ld_vt, void* y, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (dims->width % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_weights_nvfp4(w)) != FLUX3_OK) return s;
    if (n_tokens == 0) return FLUX3_OK;
    if (!a4 || !a_sf || !sa || !rope || !q || !k || !vt || !y) return FLUX3_ERR_INVALID_ARG;
    if (!al16(a4) || !al16(a_sf) || !al16(rope) || !al16(q) || !al16(k) || !al16(vt) || !al16(y)) return FLUX3_ERR_INVALID_ARG;
    if (ld_vt < n_tokens || ld_vt % 8 != 0) return FLUX3_ERR_INVALID_ARG;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    return run_in_proj_nvfp4(dims, w, a4, a_sf, sa, n_tokens, rope, q, k, vt, ld_vt, y,
                             reinterpret_cast<cudaStream_t>(stream));
}

size_t flux3_block_nvfp4_workspace_size(const flux3_dims* dims, int32_t n_tokens) {
    if (check_dims(dims) != FLUX3_OK || n_tokens < 0 || n_tokens > kMaxTokens) return 0;
    return quant_ws(dims, n_tokens, true, nullptr).bytes;
}

flux3_status flux3_block_nvfp4_fwd(const flux3_dims* dims, const flux3_block_weights_nvfp4* w, const flux3_segments* segs,
                                   const void* x, void* x_out, int32_t n_tokens, const float* rope, void* ws,
                                   size_t ws_bytes, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (dims->width % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    const int N = n_tokens;
    if (N < 0 || N > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, N, true)) != FLUX3_OK) return s;
    if ((s = check_weights_nvfp4(w)) != FLUX3_OK) return s;
    if (w->b_out && !al16(w->b_out)) return FLUX3_ERR_INVALID_ARG;
    if (w->w_out_q ? (!al16(w->w_out_q) || !w->w_out_sf || !al16(w->w_out_sf) || !w->s_out)
                   : (!w->w_out || !al16(w->w_out)))
        return FLUX3_ERR_INVALID_ARG;
    if ((dims->width + dims->ffn_hidden) % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (N == 0) return FLUX3_OK;
    if (!x || !x_out || !rope || !al16(x) || !al16(x_out) || !al16(rope)) return FLUX3_ERR_INVALID_ARG;
    if (!ws || !al256(ws) || ws_bytes < flux3_block_nvfp4_workspace_size(dims, N)) return FLUX3_ERR_WORKSPACE;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const BlockWs b = block_ws_layout(dims, N, static_cast<uint8_t*>(ws));
    const QuantWs qw = quant_ws(dims, N, true, static_cast<uint8_t*>(ws));
    const int D = dims->width, F = dims->ffn_hidden;
    if ((s = run_adaln(dims, segs->mod, seg_table(segs->seg_off, segs->n_seg), x, N, b.a, st)) != FLUX3_OK) return s;
    if ((s = run_quantize_rows_nvfp4(b.a, N, D, qw.a_q, qw.a_sf, qw.sa, st)) != FLUX3_OK) return s;
    if ((s = run_in_proj_nvfp4(dims, w, qw.a_q, qw.a_sf, qw.sa, N, rope, b.q, b.k, b.vt, b.ld_vt, b.y, st)) != FLUX3_OK)
        return s;
    const int32_t full[2] = {0, N};
    if ((s = run_attn(dims, b.q, b.k, b.vt, b.ld_vt, N, full, 1, b.y, D + F, false, st)) != FLUX3_OK) return s;
    if (w->w_out_q) {
        if ((s = run_quantize_rows_nvfp4(b.y, N, D + F, qw.y_q, qw.y_sf, qw.sy, st)) != FLUX3_OK) return s;
        return run_out_proj_quant(dims, true, w->w_out_q, w->w_out_sf, w->s_out, w->b_out, segs, qw.y_q, qw.y_sf, qw.sy, x,
                                  x_out, N, st);
    }
    const flux3_block_weights wo{nullptr, nullptr, nullptr, nullptr, w->w_out, w->b_out};
    return run_out_proj(dims, &wo, 1, segs, b.y, x, x_out, N, st);
}

// ---------------------------------------------------------------- the joint block's backward
namespace {
constexpr int kBwdSlots = 4;  // heads whose attention backward runs concurrently
struct BwdWs {
    BlockWs f;                      // the forward pass recomputed: a, q, k, V^T, [O | act]
    __nv_bfloat16 *p, *dy, *dyT, *woT, *wiT, *dycat, *ycatT, *dp, *dpT, *aT;
    __nv_bfloat16 *pT[kBwdSlots], *dsT[kBwdSlots], *dsn[kBwdSlots], *doT[kBwdSlots], *kT[kBwdSlots], *qT[kBwdSlots];
    float *yout, *lse, *delta, *dq, *dk, *dv, *da;
    float2* stats;
    int ldn;  // row stride of the [., N] buffers (N rounded up to 8)
    size_t bytes;
};
BwdWs bwd_ws_layout(const flux3_dims* d, int N, uint8_t* base) {
    BwdWs w;
    w.f = block_ws_layout(d, N, base);
    const size_t D = d->width, F = d->ffn_hidden, n_in = 3 * D + 2 * F;
    w.ldn = (N + 7) & ~7;
    const size_t ldn = w.ldn;
    size_t off = w.f.bytes;
    auto take = [&](size_t bytes) {
        uint8_t* p = base ? base + off : nullptr;
        off += up256(bytes);
        return p;
    };
    auto bf = [&](size_t elems) { return reinterpret_cast<__nv_bfloat16*>(take(elems * 2)); };
    auto f32 = [&](size_t elems) { return reinterpret_cast<float*>(take(elems * 4)); };
    w.p = bf((size_t)N * n_in);
    w.yout = f32((size_t)N * D);
    w.dy = bf((size_t)N * D);
    w.dyT = bf(D * ldn);
    w.woT = bf((D + F) * D);
    w.wiT = bf(D * n_in);
    w.dycat = bf((size_t)N * (D + F));
    w.ycatT = bf((D + F) * ldn);
    w.lse = f32((size_t)d->heads * N);
    w.delta = f32((size_t)d->heads * N);
    for (int i = 0; i < kBwdSlots; ++i) {
        w.pT[i] = bf((size_t)N * ldn);
        w.dsT[i] = bf((size_t)N * ldn);
        w.dsn[i] = bf((size_t)N * ldn);
        w.doT[i] = bf(128 * ldn);
        w.kT[i] = bf(128 * ldn);
        w.qT[i] = bf(128 * ldn);
    }
    w.dq = f32((size_t)N * D);
    w.dk = f32((size_t)N * D);
    w.dv = f32((size_t)N * D);
    w.dp = bf((size_t)N * n_in);
    w.dpT = bf(n_in * ldn);
    w.aT = bf(D * ldn);
    w.da = f32((size_t)N * D);
    w.stats = reinterpret_cast<float2*>(take((size_t)N * 8));
    w.bytes = off;
    return w;
}
}  // namespace

namespace {
// Library-owned streams of the current device on which the attention backward runs
// several heads at once (created once per device, non-blocking).
bool bwd_streams(cudaStream_t (&out)[kBwdSlots]) {
    static std::mutex mu;
    static cudaStream_t pool[64][kBwdSlots] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < kBwdSlots; ++i) {
        if (!pool[dev][i] && cudaStreamCreateWithFlags(&pool[dev][i], cudaStreamNonBlocking) != cudaSuccess) return false;
        out[i] = pool[dev][i];
    }
    return true;
}
}  // namespace

size_t flux3_block_bwd_workspace_size(const flux3_dims* dims, int32_t n_tokens) {
    if (check_dims(dims) != FLUX3_OK || n_tokens < 0 || n_tokens > kMaxTokens) return 0;
    return bwd_ws_layout(dims, n_tokens, nullptr).bytes;
}

flux3_status flux3_block_bwd(const flux3_dims* dims, const flux3_block_weights* w, const flux3_segments* segs,
                             const void* x, const float* rope, const float* dxo, int32_t n_tokens, float* dx, float* dw_in,
                             float* db_in, float* dq_norm, float* dk_norm, float* dw_out, float* db_out, float* dmod,
                             void* ws, size_t ws_bytes, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    const int N = n_tokens;
    if (N < 0 || N > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, N, true)) != FLUX3_OK) return s;
    if ((s = check_weights(w, 1, true, true)) != FLUX3_OK) return s;
    if (dims->width % 256 != 0) return FLUX3_ERR_UNSUPPORTED;
    if (N == 0) return FLUX3_OK;
    if (!x || !rope || !dxo || !dx || !dw_in || !db_in || !dq_norm || !dk_norm || !dw_out || !db_out || !dmod)
        return FLUX3_ERR_INVALID_ARG;
    if (!al16(x) || !al16(rope) || !al16(dxo) || !al16(dx) || !al16(dw_in) || !al16(dw_out)) return FLUX3_ERR_INVALID_ARG;
    if (!ws || !al256(ws) || ws_bytes < flux3_block_bwd_workspace_size(dims, N)) return FLUX3_ERR_WORKSPACE;
    if (!have_encode()) return FLUX3_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const BwdWs b = bwd_ws_layout(dims, N, static_cast<uint8_t*>(ws));
    const int D = dims->width, F = dims->ffn_hidden, H = dims->heads, n_in = 3 * D + 2 * F, ldy = D + F, ldn = b.ldn;
    const SegOffsets so = seg_table(segs->seg_off, segs->n_seg);
    const int n_seg = segs->n_seg;
    const float sc = (float)(1.0 / std::sqrt(128.0));
    // outputs that accumulate
    if (cudaMemsetAsync(db_in, 0, (size_t)n_in * 4, st) != cudaSuccess || cudaMemsetAsync(dq_norm, 0, 128 * 4, st) != cudaSuccess ||
        cudaMemsetAsync(dk_norm, 0, 128 * 4, st) != cudaSuccess || cudaMemsetAsync(db_out, 0, (size_t)D * 4, st) != cudaSuccess ||
        cudaMemsetAsync(dmod, 0, (size_t)n_seg * 3 * D * 4, st) != cudaSuccess)
        return FLUX3_ERR_CUDA;

    // ---- the forward pass again: a, q, k, V^T, [O | act], the projections P and y
    if ((s = run_adaln(dims, segs->mod, so, x, N, b.f.a, st)) != FLUX3_OK) return s;
    if ((s = run_in_proj(dims, w, 1, segs, b.f.a, N, rope, b.f.q, b.f.k, b.f.vt, b.f.ld_vt, b.f.y, st)) != FLUX3_OK) return s;
    const int32_t full[2] = {0, N};
    if ((s = run_attn(dims, b.f.q, b.f.k, b.f.vt, b.f.ld_vt, N, full, 1, b.f.y, ldy, false, st, b.lse)) != FLUX3_OK) return s;
    if ((s = run_gemm_plain(b.f.a, D, w->w_in, D, N, n_in, D, w->b_in, b.p, n_in, true, st)) != FLUX3_OK) return s;
    if ((s = run_gemm_plain(b.f.y, ldy, w->w_out, ldy, N, D, ldy, w->b_out, b.yout, D, false, st)) != FLUX3_OK) return s;

    // ---- x' = x + gate y
    prof_before(FLUX3_KERNEL_BWD_ELEM, st);
    bwd_gate_kernel<<<dim3((unsigned)((N + BWD_ROWS - 1) / BWD_ROWS), (unsigned)(D / 256)), 256, 0, st>>>(
        dxo, b.yout, N, D, segs->mod, so, b.dy, dmod, db_out);
    prof_after(st);
    if ((s = launch_status()) != FLUX3_OK) return s;
    // ---- y = [O | act] W_out^T + b_out
    if ((s = run_transpose(w->w_out, D, ldy, ldy, b.woT, D, st)) != FLUX3_OK) return s;
    if ((s = run_gemm_plain(b.dy, D, b.woT, D, N, ldy, D, nullptr, b.dycat, ldy, true, st)) != FLUX3_OK) return s;
    if ((s = run_transpose(b.dy, N, D, D, b.dyT, ldn, st)) != FLUX3_OK) return s;
    if ((s = run_transpose(b.f.y, N, ldy, ldy, b.ycatT, ldn, st)) != FLUX3_OK) return s;
    if ((s = run_gemm_plain(b.dyT, ldn, b.ycatT, ldn, D, ldy, N, nullptr, dw_out, ldy, false, st)) != FLUX3_OK) return s;
    // ---- act = silu(G) U
    prof_before(FLUX3_KERNEL_BWD_ELEM, st);
    bwd_swiglu_kernel<<<(unsigned)(8 * sm_count()), 256, 0, st>>>(b.dycat, b.p, N, D, F, b.dp);
    prof_after(st);
    if ((s = launch_status()) != FLUX3_OK) return s;
    // ---- attention, one head at a time, keys as rows: P^T and dS^T come out of the GEMM
    // epilogues (the forward pass's log2-sum-exp2 per query, rowsum(dO O) per query)
    prof_before(FLUX3_KERNEL_BWD_ELEM, st);
    attn_delta_kernel<<<(unsigned)(4 * sm_count()), 256, 0, st>>>(b.dycat, b.f.y, ldy, N, H, b.delta);
    prof_after(st);
    if ((s = launch_status()) != FLUX3_OK) return s;
    const float sc_log2 = (float)(1.4426950408889634 / std::sqrt(128.0));
    // the heads run kBwdSlots at a time on library-owned streams forked from `st` and
    // joined back into it by events (each head writes its own columns of dQ, dK, dV)
    cudaStream_t hs[kBwdSlots];
    if (!bwd_streams(hs)) return FLUX3_ERR_CUDA;
    cudaEvent_t fork = nullptr, join[kBwdSlots] = {};
    auto release = [&]() {
        if (fork) cudaEventDestroy(fork);
        for (int i = 0; i < kBwdSlots; ++i)
            if (join[i]) cudaEventDestroy(join[i]);
    };
    if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess || cudaEventRecord(fork, st) != cudaSuccess) {
        release();
        return FLUX3_ERR_CUDA;
    }
    for (int i = 0; i < kBwdSlots; ++i)
        if (cudaEventCreateWithFlags(&join[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaStreamWaitEvent(hs[i], fork, 0) != cudaSuccess) {
            release();
            return FLUX3_ERR_CUDA;
        }
    for (int h = 0; h < H && s == FLUX3_OK; ++h) {
        const int sl = h % kBwdSlots;
        cudaStream_t hst = hs[sl];
        const __nv_bfloat16* qh = b.f.q + (size_t)h * N * 128;
        const __nv_bfloat16* kh = b.f.k + (size_t)h * N * 128;
        const __nv_bfloat16* doh = b.dycat + (size_t)h * 128;     // row stride ldy
        const __nv_bfloat16* vh = b.p + 2 * D + (size_t)h * 128;  // row stride n_in
        // P^T = exp2(scale_log2 k q^T - lse);  dV = P^T dO
        if ((s = run_gemm_attn_t<EPI_PROB_T>(kh, 128, qh, 128, N, N, 128, b.lse + (size_t)h * N, nullptr, 0, sc_log2,
                                             b.pT[sl], ldn, hst)) != FLUX3_OK ||
            (s = run_transpose(doh, N, 128, ldy, b.doT[sl], ldn, hst)) != FLUX3_OK ||
            (s = run_gemm_plain(b.pT[sl], ldn, b.doT[sl], ldn, N, 128, N, nullptr, b.dv + (size_t)h * 128, D, false, hst)) !=
                FLUX3_OK)
            break;
        // dS^T = scale P^T (v dO^T - delta);  dK = dS^T q
        if ((s = run_gemm_attn_t<EPI_DS_T>(vh, n_in, doh, ldy, N, N, 128, b.delta + (size_t)h * N, b.pT[sl], ldn, sc,
                                           b.dsT[sl], ldn, hst)) != FLUX3_OK ||
            (s = run_transpose(qh, N, 128, 128, b.qT[sl], ldn, hst)) != FLUX3_OK ||
            (s = run_gemm_plain(b.dsT[sl], ldn, b.qT[sl], ldn, N, 128, N, nullptr, b.dk + (size_t)h * 128, D, false, hst)) !=
                FLUX3_OK)
            break;
        // dQ = dS k
        if ((s = run_transpose(b.dsT[sl], N, N, ldn, b.dsn[sl], ldn, hst)) != FLUX3_OK ||
            (s = run_transpose(kh, N, 128, 128, b.kT[sl], ldn, hst)) != FLUX3_OK ||
            (s = run_gemm_plain(b.dsn[sl], ldn, b.kT[sl], ldn, N, 128, N, nullptr, b.dq + (size_t)h * 128, D, false, hst)) !=
                FLUX3_OK)
            break;
    }
    for (int i = 0; i < kBwdSlots; ++i)
        if (cudaEventRecord(join[i], hs[i]) != cudaSuccess || cudaStreamWaitEvent(st, join[i], 0) != cudaSuccess) {
            release();
            return FLUX3_ERR_CUDA;
        }
    release();
    if (s != FLUX3_OK) return s;
    // ---- RoPE, QK RMSNorm and the V columns of dP; then P = a W_in^T + b_in
    prof_before(FLUX3_KERNEL_BWD_ELEM, st);
    bwd_qk_kernel<<<(unsigned)(4 * sm_count()), 256, 0, st>>>(b.dq, b.dk, b.dv, b.p, reinterpret_cast<const float2*>(rope),
                                                             w->q_norm, w->k_norm, dims->rms_eps, N, H, D, F, b.dp, dq_norm,
                                                             dk_norm);
    prof_after(st);
    if ((s = launch_status()) != FLUX3_OK) return s;
    prof_before(FLUX3_KERNEL_BWD_ELEM, st);
    colsum_bf16_kernel<<<dim3((unsigned)((n_in + 255) / 256), (unsigned)((N + 63) / 64)), 256, 0, st>>>(b.dp, N, n_in, n_in,
                                                                                                    db_in);
    prof_after(st);
    if ((s = launch_status()) != FLUX3_OK) return s;
    if ((s = run_transpose(w->w_in, n_in, D, D, b.wiT, n_in, st)) != FLUX3_OK) return s;
    if ((s = run_gemm_plain(b.dp, n_in, b.wiT, n_in, N, D, n_in, nullptr, b.da, D, false, st)) != FLUX3_OK) return s;
    if ((s = run_transpose(b.dp, N, n_in, n_in, b.dpT, ldn, st)) != FLUX3_OK) return s;
    if ((s = run_transpose(b.f.a, N, D, D, b.aT, ldn, st)) != FLUX3_OK) return s;
    if ((s = run_gemm_plain(b.dpT, ldn, b.aT, ldn, n_in, D, N, nullptr, dw_in, D, false, st)) != FLUX3_OK) return s;
    // ---- LayerNorm + modulation
    prof_before(FLUX3_KERNEL_BWD_ELEM, st);
    bwd_ln_kernel<<<(unsigned)((N + 7) / 8), 256, 0, st>>>(b.da, static_cast<const __nv_bfloat16*>(x), dxo, segs->mod, so,
                                                           dims->ln_eps, N, D, dx, b.stats);
    prof_after(st);
    if ((s = launch_status()) != FLUX3_OK) return s;
    prof_before(FLUX3_KERNEL_BWD_ELEM, st);
    bwd_mod_kernel<<<dim3((unsigned)((N + BWD_ROWS - 1) / BWD_ROWS), (unsigned)(D / 256)), 256, 0, st>>>(
        b.da, static_cast<const __nv_bfloat16*>(x), b.stats, N, D, so, dmod);
    prof_after(st);
    return launch_status();
}

size_t flux3_stream_block_bwd_workspace_size(const flux3_dims* dims, const flux3_segments* segs) {
    if (check_dims(dims) != FLUX3_OK || !segs || segs->n_seg < 1 || segs->n_seg > FLUX3_MAX_SEGMENTS || !segs->seg_off)
        return 0;
    size_t need = 0;
    for (int s = 0; s < segs->n_seg; ++s) {
        const int n = segs->seg_off[s + 1] - segs->seg_off[s];
        if (n < 0 || n > kMaxTokens) return 0;
        const size_t b = flux3_block_bwd_workspace_size(dims, n);
        need = b > need ? b : need;
    }
    return need;
}

flux3_status flux3_stream_block_bwd(const flux3_dims* dims, const flux3_block_weights* w, const flux3_segments* segs,
                                    const void* x, const float* rope, const float* dxo, int32_t n_tokens, float* dx,
                                    float* dw_in, float* db_in, float* dq_norm, float* dk_norm, float* dw_out,
                                    float* db_out, float* dmod, void* ws, size_t ws_bytes, flux3_stream_t stream) {
    flux3_status s = check_dims(dims);
    if (s != FLUX3_OK) return s;
    if (n_tokens < 0 || n_tokens > kMaxTokens) return FLUX3_ERR_INVALID_ARG;
    if ((s = check_segs(segs, n_tokens, true)) != FLUX3_OK) return s;
    if ((s = check_weights(w, segs->n_seg, true, true)) != FLUX3_OK) return s;
    if (n_tokens == 0) return FLUX3_OK;
    if (!ws || ws_bytes < flux3_stream_block_bwd_workspace_size(dims, segs)) return FLUX3_ERR_WORKSPACE;
    const size_t D = dims->width, F = dims->ffn_hidden, n_in = 3 * D + 2 * F;
    // stage 1: every stream runs its own block on its own rows and attends only to itself,
    // so the block's backward is the joint block's backward of each stream on its own
    for (int g = 0; g < segs->n_seg; ++g) {
        const int lo = segs->seg_off[g], n = segs->seg_off[g + 1] - lo;
        if (n == 0) {  // an empty stream: its parameters get zero gradients
            cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
            if (cudaMemsetAsync(dw_in + g * n_in * D, 0, n_in * D * 4, st) != cudaSuccess ||
                cudaMemsetAsync(db_in + g * n_in, 0, n_in * 4, st) != cudaSuccess ||
                cudaMemsetAsync(dq_norm + g * 128, 0, 128 * 4, st) != cudaSuccess ||
                cudaMemsetAsync(dk_norm + g * 128, 0, 128 * 4, st) != cudaSuccess ||
                cudaMemsetAsync(dw_out + g * D * (D + F), 0, D * (D + F) * 4, st) != cudaSuccess ||
                cudaMemsetAsync(db_out + g * D, 0, D * 4, st) != cudaSuccess ||
                cudaMemsetAsync(dmod + g * 3 * D, 0, 3 * D * 4, st) != cudaSuccess)
                return FLUX3_ERR_CUDA;
            continue;
        }
        const int32_t one[2] = {0, n};
        const flux3_segments sg{1, one, segs->mod + g * 3 * D};
        s = flux3_block_bwd(dims, w + g, &sg, static_cast<const __nv_bfloat16*>(x) + (size_t)lo * D, rope + (size_t)lo * 128,
                            dxo + (size_t)lo * D, n, dx + (size_t)lo * D, dw_in + g * n_in * D, db_in + g * n_in,
                            dq_norm + g * 128, dk_norm + g * 128, dw_out + g * D * (D + F), db_out + g * D, dmod + g * 3 * D,
                            ws, ws_bytes, stream);
        if (s != FLUX3_OK) return s;
    }
    return FLUX3_OK;
}

flux3_status flux3_device_error(uint32_t* flags, int32_t reset) {
    if (cudaDeviceSynchronize() != cudaSuccess) return FLUX3_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return FLUX3_ERR_CUDA;
    if (reset) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_device_error, &z, sizeof z) != cudaSuccess) return FLUX3_ERR_CUDA;
    }
    if (flags) *flags = v;
    return v ? FLUX3_ERR_TIMEOUT : FLUX3_OK;
}

flux3_status flux3_selftest_timeout(uint32_t timeout_us) {
    if (timeout_us < 1 || timeout_us > 10u * 1000 * 1000) return FLUX3_ERR_INVALID_ARG;
    int* d = nullptr;  // the kernel's one-int result slot: a file-scope device symbol, no allocation
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d), g_selftest_result) != cudaSuccess) return FLUX3_ERR_CUDA;
    int h = -1;
    selftest_wait_kernel<<<1, 32>>>(1000ull * timeout_us, d);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&h, g_selftest_result, sizeof(int));  // synchronises
    if (e != cudaSuccess) return FLUX3_ERR_CUDA;
    return h == 0 ? FLUX3_OK : FLUX3_ERR_CUDA;  // h == 1 would mean the barrier completed
}

flux3_status flux3_profile_begin(int32_t capacity) {
    if (capacity <= 0 || capacity > (1 << 16)) return FLUX3_ERR_INVALID_ARG;
    for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
    g_prof.ev.assign(2 * (size_t)capacity, nullptr);
    for (auto& e : g_prof.ev)
        if (cudaEventCreate(&e) != cudaSuccess) return FLUX3_ERR_CUDA;
    g_prof.kind.assign(capacity, 0);
    g_prof.cap = capacity;
    g_prof.n = 0;
    g_prof.on = true;
    return FLUX3_OK;
}

flux3_status flux3_profile_end(float* ms, int32_t* kinds, int32_t capacity, int32_t* n) {
    if (!g_prof.on) return FLUX3_ERR_INVALID_ARG;
    g_prof.on = false;
    if (cudaDeviceSynchronize() != cudaSuccess) return FLUX3_ERR_CUDA;
    const int cnt = g_prof.n < capacity ? g_prof.n : capacity;
    for (int i = 0; i < cnt; ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) return FLUX3_ERR_CUDA;
        if (ms) ms[i] = t;
        if (kinds) kinds[i] = g_prof.kind[i];
    }
    if (n) *n = cnt;
    return FLUX3_OK;
}

}  // extern "C"
