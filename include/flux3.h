/*
 * flux3.h -- C-ABI of libflux3.so: the FLUX.3 Image Klein transformer block on one
 * B300 (sm_103a).
 *
 * What the block computes is stated on "Welcome FLUX.3 Image Klein in Diffusers",
 * section "How it works": each block runs attention and a SwiGLU MLP in parallel on
 * the same normalized input; scale, shift and gate come from timestep modulation set
 * separately per stream (image at t, text and references at t = 0); RoPE uses four
 * axes (t, h, w, l) of 32 head dims each; stage 1 runs 5 blocks per stream with the
 * stream's own weights and self-only attention, stage 2 runs 28 shared blocks with
 * full attention over the concatenated streams, and the output layers read the image
 * tokens only.  The QK normalisation with a learned scale follows the module names
 * "*.{query,key}_norm.scale" on the Miles page "FLUX 3 Image Klein", section 3
 * ("Family config"), and the absence of a padding mask follows the same table
 * (row "Micro-batch") and "How it works" (the text is padded to a multiple of 80 tokens
 * and the padded tokens are attended, not masked).
 *
 * Conventions for every entry point
 *  - The caller owns all memory.  Pointers marked "device" must point to device
 *    memory of the current CUDA device, 16-byte aligned; "host" pointers are read
 *    during the call only.  The library allocates nothing.
 *  - Work is enqueued on `stream` and runs asynchronously; the return value reports
 *    argument validation and launch errors only.  No entry point synchronises the host
 *    except flux3_device_error and flux3_profile_end.
 *  - Arguments are checked on the host before anything is launched; a failed check
 *    returns FLUX3_ERR_INVALID_ARG / FLUX3_ERR_UNSUPPORTED / FLUX3_ERR_WORKSPACE and
 *    leaves every output untouched.  The library never traps or aborts.
 *  - Activations are bf16 row-major; accumulation is fp32.  Batch is 1: one token
 *    sequence per call, because the model takes no padding mask.
 *  - Device kernels bound every wait; a wait that runs out sets a device flag that
 *    flux3_device_error reports as FLUX3_ERR_TIMEOUT.
 *  - Not thread-safe with respect to flux3_profile_begin / flux3_profile_end.
 */
#ifndef FLUX3_H
#define FLUX3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. NULL is the legacy default stream. */
typedef struct CUstream_st *flux3_stream_t;

typedef enum flux3_status {
    FLUX3_OK = 0,
    FLUX3_ERR_INVALID_ARG = 1, /* NULL / misaligned pointer, bad size or offsets      */
    FLUX3_ERR_UNSUPPORTED = 2, /* valid but not implemented (head_dim != 128, ...)     */
    FLUX3_ERR_WORKSPACE = 3,   /* workspace pointer NULL/misaligned or too small       */
    FLUX3_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed          */
    FLUX3_ERR_TIMEOUT = 5      /* a device-side wait ran out (see flux3_device_error)  */
} flux3_status;

/* At most this many token segments (streams) per call. */
#define FLUX3_MAX_SEGMENTS 16

/* Model dimensions.  FLUX.3 Image Klein: width 3072, 24 heads x 128, SwiGLU hidden
 * 9216 ("How it works" gives the width 3072 and the 128 head dims; the SGLang
 * cookbook, section 4, the 24 heads).  Requirements: head_dim == 128 (else
 * UNSUPPORTED), width == heads * head_dim, heads even, ffn_hidden % 128 == 0,
 * eps > 0, rope_theta > 0.  Defaults used throughout: ln_eps = rms_eps = 1e-6,
 * rope_theta = 10000. */
typedef struct flux3_dims {
    int32_t width;
    int32_t heads;
    int32_t head_dim;
    int32_t ffn_hidden;
    float ln_eps;     /* LayerNorm epsilon (no affine: the modulation replaces it)   */
    float rms_eps;    /* QK RMSNorm epsilon                                          */
    float rope_theta; /* RoPE base                                                    */
} flux3_dims;

/* One block's parameters (all device memory; nn.Linear layout, i.e. [out, in]).
 *  w_in   bf16 [3D + 2F, D]: rows Q | K | V | gate | up, each head's 128 rows
 *         contiguous ("How it works": attention and SwiGLU read the same normalized
 *         input, so one projection produces both).
 *  b_in   fp32 [3D + 2F] or NULL (zero).
 *  q_norm, k_norm  fp32 [128]: learned RMSNorm scales ("*.query_norm.scale",
 *         "*.key_norm.scale" on the Miles page, section 3).
 *  w_out  bf16 [D, D + F]: columns attention-out | SwiGLU-out.
 *  b_out  fp32 [D] or NULL (zero). */
typedef struct flux3_block_weights {
    const void *w_in;
    const float *b_in;
    const float *q_norm;
    const float *k_norm;
    const void *w_out;
    const float *b_out;
} flux3_block_weights;

/* Token segments = streams, contiguous in token order [image | reference | text].
 *  n_seg     1 .. FLUX3_MAX_SEGMENTS.
 *  seg_off   HOST int32 [n_seg + 1], seg_off[0] = 0, non-decreasing, seg_off[n_seg] = N.
 *  mod       DEVICE fp32 [n_seg][3][D]: (shift, scale, gate) of each stream.  The
 *            image stream's vectors come from its timestep t and the text/reference
 *            streams' from t = 0 ("How it works"); the library takes them as inputs. */
typedef struct flux3_segments {
    int32_t n_seg;
    const int32_t *seg_off;
    const float *mod;
} flux3_segments;

const char *flux3_status_string(flux3_status s);
const char *flux3_version(void);

/* ---- a1: RoPE table ("How it works": four axes t, h, w, l, 32 of the 128 dims each).
 * pos   device int32 [N, 4]: (t, h, w, l) per token.
 * rope  device fp32 [N, 64, 2]: (cos, sin) of pair p = 16 a + j (axis a, j = 0..15),
 *       angle pos[a] * theta^(-2 j / 32), reduced modulo 2 pi (in turns, exactly split
 *       in fp32) before sin/cos: error <= pi * 2^-24 plus sincospif's rounding.
 *       Pair p rotates head dims (2p, 2p+1).  N == 0 is a no-op. */
flux3_status flux3_rope_build(const flux3_dims *dims, const int32_t *pos, int32_t n_tokens,
                              float *rope, flux3_stream_t stream);

/* ---- a2 + a3: LayerNorm and per-stream modulation ("How it works": the block's
 * normalized input; scale and shift per stream).
 * a[r] = (x[r] - mean) * rsqrt(var + ln_eps) * (1 + scale_s) + shift_s, s = segment of r.
 * x  device bf16 [N, D];  a  device bf16 [N, D] (may not alias x). */
flux3_status flux3_adaln_fwd(const flux3_dims *dims, const flux3_segments *segs, const void *x,
                             int32_t n_tokens, void *a, flux3_stream_t stream);

/* ---- a4 .. a7: fused input projection with its epilogues.
 * P = a W_in^T + b_in on tcgen05 tensor cores, then per token and head
 *   q = RoPE(RMSNorm(P_q) * q_norm), k = RoPE(RMSNorm(P_k) * k_norm), v = P_v,
 *   act = silu(P_gate) * P_up.
 * w, n_w      host array of 1 weight set (shared by all tokens, stage 2) or of
 *             segs->n_seg sets (segment s uses w[s], stage 1).
 * a           device bf16 [N, D] (output of flux3_adaln_fwd).
 * rope        device fp32 [N, 64, 2] (flux3_rope_build).
 * q, k        device bf16 [H, N, 128].
 * vt          device bf16 [H, 128, ld_vt]: V transposed (token index fastest),
 *             ld_vt >= N and ld_vt % 8 == 0.
 * y           device bf16 [N, D + F]: act is written to columns D .. D+F-1; columns
 *             0 .. D-1 are left for the attention output. */
flux3_status flux3_in_proj_fwd(const flux3_dims *dims, const flux3_block_weights *w, int32_t n_w,
                               const flux3_segments *segs, const void *a, int32_t n_tokens,
                               const float *rope, void *q, void *k, void *vt, int32_t ld_vt,
                               void *y, flux3_stream_t stream);

/* ---- a8: attention, softmax(q k^T / sqrt(128)) v per head, bidirectional, no padding
 * mask ("How it works": the transformer attends to the text padding; stage 1 attends
 * only within each stream, stage 2 over all tokens).
 * seg_off     HOST int32 [n_seg + 1]: a query attends to the keys of its own segment.
 *             n_seg = 1 (or seg_off = NULL) is full attention over the N tokens.
 * q, k        device bf16 [H, N, 128];  vt  device bf16 [H, 128, ld_vt] (as above).
 * out         device [N, ld_out], columns h*128 .. h*128+127 for head h; bf16, or
 *             fp32 when fp32_debug != 0 (a SIMT fp32 path kept for checking; slow). */
flux3_status flux3_attn_fwd(const flux3_dims *dims, const void *q, const void *k, const void *vt,
                            int32_t ld_vt, int32_t n_tokens, const int32_t *seg_off, int32_t n_seg,
                            void *out, int32_t ld_out, int32_t fp32_debug, flux3_stream_t stream);

/* ---- a9: fused output projection with the gated residual ("How it works": gate from
 * the stream's modulation).  x_out = x + gate_s * (y W_out^T + b_out).
 * w, n_w   as for flux3_in_proj_fwd.   y  device bf16 [N, D + F].
 * x        device bf16 [N, D];  x_out  device bf16 [N, D], may alias x. */
flux3_status flux3_out_proj_fwd(const flux3_dims *dims, const flux3_block_weights *w, int32_t n_w,
                                const flux3_segments *segs, const void *y, const void *x,
                                void *x_out, int32_t n_tokens, flux3_stream_t stream);

/* Workspace bytes for flux3_block_fwd / flux3_stream_block_fwd at N tokens. */
size_t flux3_block_workspace_size(const flux3_dims *dims, int32_t n_tokens);

/* ---- one stage-2 joint block ("How it works", "Stage 2": shared weights, full
 * attention over [image | reference | text]).  Runs a2 .. a9 with one weight set.
 * rope   device fp32 [N, 64, 2] from flux3_rope_build.
 * ws     device workspace, 256-byte aligned, >= flux3_block_workspace_size bytes.
 * x_out may alias x. */
flux3_status flux3_block_fwd(const flux3_dims *dims, const flux3_block_weights *w,
                             const flux3_segments *segs, const void *x, void *x_out,
                             int32_t n_tokens, const float *rope, void *ws, size_t ws_bytes,
                             flux3_stream_t stream);

/* ---- one stage-1 block for every stream at once ("How it works", "Stage 1": each
 * stream has its own weights and attends only to itself).  w is a host array of
 * segs->n_seg weight sets; segment s uses w[s].  Other arguments as flux3_block_fwd. */
flux3_status flux3_stream_block_fwd(const flux3_dims *dims, const flux3_block_weights *w,
                                    const flux3_segments *segs, const void *x, void *x_out,
                                    int32_t n_tokens, const float *rope, void *ws,
                                    size_t ws_bytes, flux3_stream_t stream);

/* ---- output layer on image tokens ("How it works": image tokens only go to the
 * output layers).  out = ((LN(x) * (1 + scale) + shift) W_final^T + b_final), fp32.
 * w_final    device bf16 [out_channels, D], out_channels % 128 == 0.
 * b_final    device fp32 [out_channels] or NULL.
 * mod_final  device fp32 [2][D]: shift, scale.
 * x          device bf16 [n_rows, D];  out  device fp32 [n_rows, out_channels].
 * ws         device workspace >= n_rows * D * 2 bytes (rounded up to 256). */
flux3_status flux3_final_fwd(const flux3_dims *dims, const void *w_final, const float *b_final,
                             int32_t out_channels, const float *mod_final, const void *x,
                             int32_t n_rows, float *out, void *ws, size_t ws_bytes,
                             flux3_stream_t stream);

/* The denoiser stack's parameters (host structs pointing at device memory). */
typedef struct flux3_dit_weights {
    int32_t n_streams;                  /* 2 (image, text) or 3 (image, reference, text) */
    int32_t n_stage1;                   /* blocks per stream before concatenation (5)   */
    int32_t n_joint;                    /* shared joint blocks (28)                     */
    const flux3_block_weights *stage1;  /* host [n_stage1][n_streams]                   */
    const flux3_block_weights *joint;   /* host [n_joint]                               */
    const void *w_final;                /* device bf16 [out_channels, D]                */
    const float *b_final;               /* device fp32 [out_channels] or NULL           */
    int32_t out_channels;               /* 128 (one packed latent patch)                */
} flux3_dit_weights;

/* Modulation vectors of every block (device fp32). */
typedef struct flux3_dit_mod {
    const float *stage1;  /* [n_stage1][n_streams][3][D] */
    const float *joint;   /* [n_joint][n_streams][3][D]  */
    const float *final;   /* [2][D]: shift, scale        */
} flux3_dit_mod;

size_t flux3_dit_workspace_size(const flux3_dims *dims, int32_t n_img, int32_t n_ref, int32_t n_txt);

/* ---- the denoiser forward ("How it works": stage 1, concatenation, stage 2, output
 * layers on image tokens).
 * tokens    device bf16 [N, D], N = n_img + n_ref + n_txt, streams contiguous in the
 *           order image | reference | text; overwritten with the last hidden state
 *           (the concatenation of stage 1 is this buffer itself, no copy).
 * pos       device int32 [N, 4].
 * velocity  device fp32 [n_img, out_channels].
 * n_ref == 0 requires n_streams == 2, n_ref > 0 requires n_streams == 3. */
flux3_status flux3_dit_fwd(const flux3_dims *dims, const flux3_dit_weights *w,
                           const flux3_dit_mod *mod, void *tokens, int32_t n_img, int32_t n_ref,
                           int32_t n_txt, const int32_t *pos, float *velocity, void *ws,
                           size_t ws_bytes, flux3_stream_t stream);

/* ---- one Euler step of the flow ODE: latent += (sigma_next - sigma) * velocity.
 * latent, velocity  device fp32 [n]. */
flux3_status flux3_euler_step(float *latent, const float *velocity, int64_t n, float sigma,
                              float sigma_next, flux3_stream_t stream);

/* ---- the base-model sampling loop around the denoiser.  "Welcome FLUX.3 Image Klein in
 * Diffusers", "How it works": image tokens are the 2x2 patches of the 32-channel latents
 * packed into 128 channels; text is a 20,480-dim stack of 8 Qwen3-VL hidden layers
 * projected to the width; references go through the same encoder as the image; the
 * scheduler applies a time shift of 6.93, so 44 of 50 steps run above sigma = 0.5.
 * "What it claims": the base checkpoint runs 50 steps with classifier-free guidance.
 * DiffSynth-Studio FLUX.3 page, pipeline arguments: alpha is the rational-shift
 * coefficient (6.93); cfg_scale 1.0 turns guidance off, the Base examples use 3.5.
 * Readings where the pages are silent: the unshifted grid 1 - i / n_steps; the shift
 * s(x) = alpha x / (1 + (alpha - 1) x); a step x += (sigma_next - sigma) v (velocity
 * from data to noise); guidance v_neg + s (v_pos - v_neg); linear embedders with bias.
 * The timestep -> modulation map is not on the pages: every step's modulation vectors
 * are inputs. */

/* Noise levels of an n_steps run, computed on the host (no GPU needed):
 * sigmas[i] = s(1 - i / n_steps), i = 0..n_steps, so sigmas[0] = 1 and sigmas[n_steps] = 0.
 * sigmas  host fp32 [n_steps + 1].  n_steps >= 1, alpha > 0 and finite. */
flux3_status flux3_sigma_schedule(int32_t n_steps, float alpha, float *sigmas);

/* A token embedder: out[r, 0:D] = x[r, :] W^T + b in bf16 (image: latent_channels -> D,
 * text: text_dim -> D), fp32 accumulation.
 * x    device bf16 [rows, k], k % 64 == 0;  w  device bf16 [D, k];  b  device fp32 [D] or NULL.
 * out  device bf16 rows of stride ld_out elements (ld_out >= D, ld_out % 8 == 0): typically
 *      the rows of a token buffer. */
flux3_status flux3_linear_fwd(const flux3_dims *dims, const void *x, int32_t rows, int32_t k, const void *w,
                              const float *b, void *out, int32_t ld_out, flux3_stream_t stream);

/* One guided Euler step: latent += (sigma_next - sigma) (v_neg + s (v_pos - v_neg)), or
 * latent += (sigma_next - sigma) v_pos when v_neg is NULL (no guidance).
 * latent, v_pos, v_neg  device fp32 [n].  latent_bf16: device bf16 [n] that receives the
 * updated latent rounded to bf16 (the next step's embedder input), or NULL. */
flux3_status flux3_cfg_euler_step(float *latent, const float *v_pos, const float *v_neg, int64_t n, float cfg_scale,
                                  float sigma, float sigma_next, void *latent_bf16, flux3_stream_t stream);

/* The sampling loop's inputs (host struct pointing at device memory). */
typedef struct flux3_sample_args {
    int32_t n_img, n_ref, n_txt;  /* tokens per stream; order image | reference | text          */
    int32_t latent_channels;      /* 128: a packed 2x2 patch of 32-channel latents (% 64 == 0)  */
    int32_t text_dim;             /* 20,480: the stacked text features (% 64 == 0)              */
    const void *w_img;            /* device bf16 [D, latent_channels]: image/reference embedder */
    const float *b_img;           /* device fp32 [D] or NULL                                    */
    const void *w_txt;            /* device bf16 [D, text_dim]: text embedder                   */
    const float *b_txt;           /* device fp32 [D] or NULL                                    */
    const void *ref_latent;       /* device bf16 [n_ref, latent_channels] (clean) or NULL       */
    const void *text_pos;         /* device bf16 [n_txt, text_dim]: the prompt's features       */
    const void *text_neg;         /* device bf16 [n_txt, text_dim]: the negative prompt's;
                                     required when cfg_scale != 1, ignored otherwise            */
    const int32_t *pos;           /* device int32 [N, 4] position ids (N = n_img + n_ref + n_txt) */
    const flux3_dit_mod *mod;     /* host [n_steps]: each step's modulation vectors (device)    */
    int32_t n_steps;              /* >= 1 (50 for the base checkpoint)                          */
    float alpha;                  /* rational time shift (6.93)                                 */
    float cfg_scale;              /* 1 = no guidance (one denoiser call per step), else two     */
    int32_t cache_context;        /* nonzero: run the stage-1 blocks of the reference and text
                                     streams once per prompt instead of once per step (below)  */
} flux3_sample_args;

/* Workspace of flux3_sample_fwd in bytes (0 for invalid arguments). */
size_t flux3_sample_workspace_size(const flux3_dims *dims, const flux3_sample_args *a);

/* The loop: for i = 0..n_steps-1, embed the latent (rounded to bf16) as the image tokens,
 * append the embedded references and text (embedded once per call), run the denoiser
 * for the prompt (and with guidance again for the negative prompt), and take the guided
 * Euler step from sigmas[i] to sigmas[i + 1] (flux3_sigma_schedule).
 * cache_context: the reference and text streams get the modulation vector of timestep 0
 * at every step ("Welcome FLUX.3 Image Klein in Diffusers", section "How it works": text
 * and references are clean inputs), and in stage 1 a stream attends only to itself, so
 * their stage-1 outputs are the same at every step.  With cache_context set the loop
 * runs those streams' stage-1 blocks once per prompt, with the stage-1 modulation of
 * step 0 (mod[0].stage1, the reference and text entries), and reuses the result; the
 * caller asserts that these entries are the same at every step.  The result then equals
 * the uncached loop's up to fp32 summation order inside the stage-1 GEMMs. 
 * latent  device fp32 [n_img, latent_channels], updated in place (in: the initial noise,
 *         out: the sample).  The denoiser's out_channels must equal latent_channels;
 *         n_ref > 0 requires a 3-stream denoiser, n_ref == 0 a 2-stream one. */
flux3_status flux3_sample_fwd(const flux3_dims *dims, const flux3_dit_weights *w, const flux3_sample_args *a,
                              float *latent, void *ws, size_t ws_bytes, flux3_stream_t stream);

/* ---- FP8 (e4m3) row-wise input projection.  The pages run quantized variants of the DiT's
 * projections (SGLang cookbook FLUX.3, section 7: FP8 and NVFP4 checkpoints; the Miles
 * page, section 3: "fp8 rowwise").  Here the input projection multiplies e4m3 codes on
 * the tensor cores (kind::f8f6f4) with fp32 accumulation:
 *   P = s_a[token] * (a_q W_q^T)[token, out] * s_w[out] + b_in
 * then the same epilogues as flux3_in_proj_fwd; the block entry point can run the output
 * projection the same way.  Quantization (flux3_quantize_rows_fp8) is per row: scale = amax / 448, codes =
 * e4m3(x * (448 / amax)) rounded to nearest even, saturated at +-448, all in fp32
 * (an all-zero row: zero codes, scale 0).  NVFP4: below. */

/* Row-wise e4m3 quantization of a bf16 [rows, k] matrix, k % 256 == 0.
 * q      device uint8 [rows, k]: e4m3 codes;  scale  device fp32 [rows]. */
flux3_status flux3_quantize_rows_fp8(const void *x, int32_t rows, int32_t k, void *q, float *scale,
                                     flux3_stream_t stream);

/* One block's parameters with e4m3 projections (device memory).
 *  w_in    uint8 [3D + 2F, D]: e4m3 codes of W_in (rows Q | K | V | gate | up), quantized
 *          per row (flux3_quantize_rows_fp8);  s_in  fp32 [3D + 2F]: their scales.
 *  w_out_q uint8 [D, D + F]: e4m3 codes of W_out, s_out fp32 [D] their row scales; when
 *          set, the block quantizes [attention | SwiGLU] per token and runs the output
 *          projection on e4m3 operands too; when NULL it runs in bf16 on w_out.
 *  Other fields as flux3_block_weights. */
typedef struct flux3_block_weights_fp8 {
    const void *w_in;
    const float *s_in;
    const float *b_in;
    const float *q_norm;
    const float *k_norm;
    const void *w_out;
    const float *b_out;
    const void *w_out_q;
    const float *s_out;
} flux3_block_weights_fp8;

/* flux3_in_proj_fwd on e4m3 operands: a8  device uint8 [N, D] codes of the modulated input,
 * sa  device fp32 [N] their per-token scales; w, n_w as flux3_in_proj_fwd (fp8 weight sets).
 * D % 128 == 0.  Outputs and other arguments as flux3_in_proj_fwd. */
flux3_status flux3_in_proj_fp8_fwd(const flux3_dims *dims, const flux3_block_weights_fp8 *w, int32_t n_w,
                                   const flux3_segments *segs, const void *a8, const float *sa, int32_t n_tokens,
                                   const float *rope, void *q, void *k, void *vt, int32_t ld_vt, void *y,
                                   flux3_stream_t stream);

size_t flux3_block_fp8_workspace_size(const flux3_dims *dims, int32_t n_tokens);

/* The joint block (stage 2) with e4m3 projections: LayerNorm + modulation (bf16), row
 * quantization, FP8 input projection with its epilogues, attention, then (w_out_q set)
 * row quantization of [attention | SwiGLU] and the FP8 output projection, or (w_out_q
 * NULL) the bf16 output projection, with the gated residual.  Arguments as
 * flux3_block_fwd; workspace flux3_block_fp8_workspace_size bytes. */
flux3_status flux3_block_fp8_fwd(const flux3_dims *dims, const flux3_block_weights_fp8 *w, const flux3_segments *segs,
                                 const void *x, void *x_out, int32_t n_tokens, const float *rope, void *ws,
                                 size_t ws_bytes, flux3_stream_t stream);

/* ---- NVFP4 input projection.  The cookbook's NVFP4 checkpoints store FP4 (E2M1) values
 * with FP8 block scales and need a Blackwell GEMM (SGLang cookbook FLUX.3, section 3,
 * Quantized checkpoints).  Here both operands of the input projection are NVFP4 and the
 * product runs on the block-scaled tensor cores (tcgen05 kind::mxf4nvf4):
 *   P = s_a[token] * sum_k (e2m1(a) sb_a)(e2m1(w) sb_w) * s_w[out] + b_in,
 * then the same epilogues as flux3_in_proj_fwd; the block entry point can run the output
 * projection the same way.  Format, per row of a bf16 [rows, k] matrix (k % 256 == 0), every step one fp32 operation
 * rounded to nearest even:
 *   g = 2688 / amax (2688 = 6 x 448; an all-zero row, or one whose g overflows fp32,
 *   gives zero codes and scales), s_row = amax / 2688;
 *   per 16 consecutive elements: sb = e4m3(bmax * g / 6) (saturating), the codes
 *   e2m1(x * (g / sb)) (saturating at 6, the sign kept at zero; 0 where sb = 0).
 * Storage: codes two per byte, the even element in the low nibble ([rows, k / 2] bytes);
 * block scales in the tiled layout the MMA reads: 512 bytes per 128 rows x 64 elements,
 * row r's four scales of 64-element step j at byte
 *   ((r / 128) * (k / 64) + j) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4,
 * rows padded to a multiple of 256 with zero scales (flux3_nvfp4_scale_bytes). */

/* Bytes of the tiled block scales of a [rows, k] matrix (0 for invalid sizes). */
size_t flux3_nvfp4_scale_bytes(int32_t rows, int32_t k);

/* NVFP4 quantization of a bf16 [rows, k] matrix (device), k % 256 == 0.
 * q  uint8 [rows, k / 2] codes;  sf  uint8 [flux3_nvfp4_scale_bytes(rows, k)] block scales;
 * scale  fp32 [rows].  All 16-byte aligned except scale. */
flux3_status flux3_quantize_rows_nvfp4(const void *x, int32_t rows, int32_t k, void *q, void *sf, float *scale,
                                       flux3_stream_t stream);

/* One block's parameters with NVFP4 projections (device memory).
 *  w_in     uint8 [3D + 2F, D / 2]: W_in codes (rows Q | K | V | gate | up), w_sf their tiled
 *           block scales, s_in fp32 [3D + 2F] their row scales (flux3_quantize_rows_nvfp4).
 *  w_out_q  uint8 [D, (D + F) / 2]: W_out codes, w_out_sf their tiled block scales, s_out
 *           fp32 [D] their row scales; when set, the block quantizes [attention | SwiGLU]
 *           per token and runs the output projection on NVFP4 operands too; when NULL it
 *           runs in bf16 on w_out.
 *  Other fields as flux3_block_weights. */
typedef struct flux3_block_weights_nvfp4 {
    const void *w_in;
    const void *w_sf;
    const float *s_in;
    const float *b_in;
    const float *q_norm;
    const float *k_norm;
    const void *w_out;
    const float *b_out;
    const void *w_out_q;
    const void *w_out_sf;
    const float *s_out;
} flux3_block_weights_nvfp4;

/* flux3_in_proj_fwd (one weight set) on NVFP4 operands: a4 uint8 [N, D / 2] codes of the
 * modulated input, a_sf their tiled block scales, sa fp32 [N] their row scales.  D % 256 == 0.
 * Outputs and other arguments as flux3_in_proj_fwd. */
flux3_status flux3_in_proj_nvfp4_fwd(const flux3_dims *dims, const flux3_block_weights_nvfp4 *w, const void *a4,
                                     const void *a_sf, const float *sa, int32_t n_tokens, const float *rope, void *q,
                                     void *k, void *vt, int32_t ld_vt, void *y, flux3_stream_t stream);

size_t flux3_block_nvfp4_workspace_size(const flux3_dims *dims, int32_t n_tokens);

/* The joint block (stage 2) with NVFP4 projections: LayerNorm + modulation (bf16), NVFP4
 * row quantization, the block-scaled input projection with its epilogues, attention, then
 * (w_out_q set) NVFP4 row quantization of [attention | SwiGLU] and the block-scaled output
 * projection, or (w_out_q NULL) the bf16 output projection, with the gated residual.
 * Arguments as flux3_block_fwd; workspace flux3_block_nvfp4_workspace_size bytes. */
flux3_status flux3_block_nvfp4_fwd(const flux3_dims *dims, const flux3_block_weights_nvfp4 *w,
                                   const flux3_segments *segs, const void *x, void *x_out, int32_t n_tokens,
                                   const float *rope, void *ws, size_t ws_bytes, flux3_stream_t stream);

/* ---- the joint block's backward pass (fine-tuning the base checkpoint: "FLUX 3 Image
 * Klein" Miles page, section 1; the block of "Welcome FLUX.3 Image Klein in Diffusers",
 * "How it works").  For a loss whose gradient with respect to the block output x' is dxo,
 * the gradients of the block input and of every parameter of flux3_block_fwd:
 *   dx      fp32 [N, D]          dw_in  fp32 [3D + 2F, D]   db_in  fp32 [3D + 2F]
 *   dq_norm fp32 [128]           dk_norm fp32 [128]         dw_out fp32 [D, D + F]
 *   db_out  fp32 [D]             dmod   fp32 [n_seg][3][D]  (shift, scale, gate, each summed
 *                                                            over its stream's rows)
 * The forward pass is recomputed inside (no saved activations); attention's score and
 * probability matrices are materialized in the workspace one head at a time.  Arguments x,
 * rope, segs, w as flux3_block_fwd (w's biases may be NULL: their gradients are still
 * written); dxo fp32 [N, D].  All outputs are overwritten; workspace
 * flux3_block_bwd_workspace_size bytes (about 2.2 GB at N = 4,256 and width 3072).
 * Attention's backward runs four heads at a time on four library-owned streams of the
 * current device, forked from `stream` and joined back into it with events (so the call
 * stays asynchronous and capturable into a CUDA graph). */
size_t flux3_block_bwd_workspace_size(const flux3_dims *dims, int32_t n_tokens);
flux3_status flux3_block_bwd(const flux3_dims *dims, const flux3_block_weights *w, const flux3_segments *segs,
                             const void *x, const float *rope, const float *dxo, int32_t n_tokens, float *dx,
                             float *dw_in, float *db_in, float *dq_norm, float *dk_norm, float *dw_out, float *db_out,
                             float *dmod, void *ws, size_t ws_bytes, flux3_stream_t stream);

/* The stage-1 (per-stream) block's backward: stream s has its own weights w[s] and
 * attends only to itself ("How it works", stage 1), so its gradients are those of the joint
 * block run on that stream alone.  Arguments as flux3_block_bwd with w [n_seg] and the
 * parameter gradients one set per stream, concatenated: dw_in [n_seg][3D + 2F][D],
 * db_in [n_seg][3D + 2F], dq_norm and dk_norm [n_seg][128], dw_out [n_seg][D][D + F],
 * db_out [n_seg][D], dmod [n_seg][3][D]; an empty stream gets zero gradients.  Workspace
 * flux3_stream_block_bwd_workspace_size bytes (that of the longest stream). */
size_t flux3_stream_block_bwd_workspace_size(const flux3_dims *dims, const flux3_segments *segs);
flux3_status flux3_stream_block_bwd(const flux3_dims *dims, const flux3_block_weights *w, const flux3_segments *segs,
                                    const void *x, const float *rope, const float *dxo, int32_t n_tokens, float *dx,
                                    float *dw_in, float *db_in, float *dq_norm, float *dk_norm, float *dw_out,
                                    float *db_out, float *dmod, void *ws, size_t ws_bytes, flux3_stream_t stream);

/* ---- flux3_block_fwd without a caller-provided workspace.
 * This entry point has no counterpart in the model description; it is a service for
 * callers that cannot allocate device memory: for example a host program that hands all
 * device memory to its own pool at start-up and forbids any other allocation, a
 * real-time loop that cannot afford the implicit device synchronisation cudaMalloc
 * performs, or a small C host linked only against this library with no allocator of
 * its own.  Instead of `ws`, the block's scratch lives in one statically sized device
 * array inside the library (FLUX3_STATIC_SCRATCH_BYTES = 64 MiB); every GPU that loads
 * the library holds that array until the process exits.
 *  - Limit: the call needs flux3_block_workspace_size(dims, n_tokens) bytes of it; a
 *    larger request returns FLUX3_ERR_WORKSPACE before anything runs.  At width 3072
 *    (24 heads, SwiGLU 9216) that is about 48 KB per token, i.e. up to ~1,360 tokens.
 *  - The first call on a device looks up the array's device address (with that device
 *    current); make that first call before any stream capture.
 *  - All calls share the one array and it keeps the previous call's contents: calls
 *    whose work overlaps on the GPU (other streams, other threads) race and corrupt each
 *    other; serialise them.  Nothing in the array needs clearing: every scratch element
 *    the kernels read is written earlier in the same call.
 *  - Allocates nothing (no cudaMalloc / cudaFree, no allocating library routine).
 * Other arguments and errors as flux3_block_fwd (one weight set, joint stage). */
#define FLUX3_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
flux3_status flux3_block_fwd_static(const flux3_dims *dims, const flux3_block_weights *w,
                                    const flux3_segments *segs, const void *x, void *x_out,
                                    int32_t n_tokens, const float *rope, flux3_stream_t stream);

/* Synchronises the device and reads the device error flags (bit 0: a bounded wait ran
 * out).  Returns FLUX3_ERR_TIMEOUT if any bit is set, else FLUX3_OK; flags may be NULL.
 * reset != 0 clears the flags.  Blocking; not for the hot path. */
flux3_status flux3_device_error(uint32_t *flags, int32_t reset);

/* Diagnostic (not part of the model): exercises the bounded-wait path every kernel uses.
 * Launches one warp that waits on a device barrier nothing ever completes; after
 * timeout_us microseconds (1 .. 10,000,000) the wait gives up, sets the device error flag
 * that flux3_device_error reports as FLUX3_ERR_TIMEOUT, and the kernel returns normally:
 * the CUDA context stays usable.  Synchronises; returns FLUX3_OK when the wait timed
 * out as designed (the flag is left set for flux3_device_error to read and reset). */
flux3_status flux3_selftest_timeout(uint32_t timeout_us);

/* Kernel timing for measurement.  Between begin and end, every kernel launch is
 * bracketed by two CUDA events on its stream (at most `capacity` launches are
 * recorded).  flux3_profile_end synchronises, writes each launch's duration in ms and
 * kind (FLUX3_KERNEL_*) into the host arrays and the count into *n. */
enum {
    FLUX3_KERNEL_ROPE = 1, FLUX3_KERNEL_ADALN = 2, FLUX3_KERNEL_IN_PROJ = 3,
    FLUX3_KERNEL_ATTN = 4, FLUX3_KERNEL_OUT_PROJ = 5, FLUX3_KERNEL_FINAL = 6,
    FLUX3_KERNEL_EULER = 7, FLUX3_KERNEL_ATTN_F32 = 8, FLUX3_KERNEL_LINEAR = 9, FLUX3_KERNEL_CFG_EULER = 10,
    FLUX3_KERNEL_TO_BF16 = 11, FLUX3_KERNEL_QUANTIZE = 12, FLUX3_KERNEL_BWD_GEMM = 13, FLUX3_KERNEL_BWD_ELEM = 14
};
flux3_status flux3_profile_begin(int32_t capacity);
flux3_status flux3_profile_end(float *ms, int32_t *kinds, int32_t capacity, int32_t *n);

#ifdef __cplusplus
}
#endif
#endif /* FLUX3_H */
