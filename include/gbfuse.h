/*
 * gbfuse.h -- C ABI of the GB300 (sm_103a) fused GEMM + epilogue library.
 *
 * The operation: a bf16 matrix product whose pointwise ending is applied to
 * each output tile while it is still on-chip, so the product crosses HBM
 * once ("Fusion and Epilogues", bullet "Epilogue fusion, the mechanical
 * form": alpha*AB + beta*C, bias and activation applied in registers on the
 * way to the one memory write; "Kernel fusion" guide, section "Concept":
 * bias, activation, scaling, residual add; "kernel fusion" wiki, the
 * activation-after-matmul case).
 *
 * Conventions shared by every entry point
 *   - Matrices are row-major.  bf16 arguments point at IEEE bfloat16 values;
 *     results are rounded to bf16 round-to-nearest-even from fp32.
 *   - Every pointer is a DEVICE pointer of the current CUDA device, owned by
 *     the caller; the library keeps no reference after the call returns and
 *     never allocates device memory.
 *   - Inputs must not overlap `out`, except `residual == out` (an in-place
 *     residual add), which is allowed.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     GBF_OK means the work was enqueued; a kernel that gives up on a
 *     bounded wait is reported later by gbf_check_device_error().
 *   - Errors are returned, never printed or thrown.  Argument, alignment and
 *     shape errors are detected before anything is launched.
 *   - Alignment: every non-null pointer 16-byte aligned; K % 8 == 0 and
 *     N % 8 == 0 (16-byte row strides for the TMA engine).  M >= 0 is free;
 *     M, N or K == 0 is accepted (an empty output, or with K == 0 an empty
 *     sum, acc = 0).
 *   - Null operands: C == NULL means beta is ignored; bias == NULL and
 *     residual == NULL mean zero.
 *   - Arithmetic: bf16 x bf16 products accumulated in fp32 on the tensor
 *     cores (tcgen05, accumulators in tensor memory), epilogue in fp32,
 *     one rounding to bf16.
 */
#ifndef GBFUSE_H
#define GBFUSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GBF_API __attribute__((visibility("default")))
#else
#define GBF_API
#endif

/* A cudaStream_t (the two types are the same pointer type). */
typedef struct CUstream_st *gbf_stream_t;

/* Activation `act` of the epilogue. */
#define GBF_ACT_IDENTITY 0
#define GBF_ACT_RELU 1      /* max(v, 0) */
#define GBF_ACT_SILU 2      /* v * sigmoid(v)  ("Fusion Thinking", Pattern 2) */
#define GBF_ACT_GELU_TANH 3 /* 0.5 v (1 + tanh(sqrt(2/pi)(v + 0.044715 v^3))) */

/* Layout of the second operand `B` / weights. */
#define GBF_B_KN 0 /* B is K x N, N contiguous: computes A * B          */
#define GBF_B_NK 1 /* W is N x K, K contiguous: computes A * W^T        */

/* Status codes. */
typedef int gbf_status_t;
#define GBF_OK 0
#define GBF_ERR_INVALID_ARG 1       /* null required pointer, bad enum, negative size */
#define GBF_ERR_MISALIGNED 2        /* pointer not 16-byte aligned */
#define GBF_ERR_UNSUPPORTED_SHAPE 3 /* N or K not a multiple of 8, bad group size, too large */
#define GBF_ERR_WORKSPACE 4         /* workspace missing or too small */
#define GBF_ERR_CUDA 5              /* a CUDA runtime/driver call failed */
#define GBF_ERR_TIMEOUT 6           /* a kernel gave up on a bounded wait */
#define GBF_ERR_NO_DEVICE 7         /* no sm_103-class device is current */

/* Operation ids for gbf_workspace_size(). */
#define GBF_OP_GEMM_EPILOGUE 0
#define GBF_OP_SWIGLU 1
#define GBF_OP_W4A16 2
#define GBF_OP_MLP 3 /* gbf_workspace_size(GBF_OP_MLP, M, D, F, fused) */
#define GBF_OP_W8A16_FP8 4
#define GBF_OP_W4A16_NVFP4 5

/*
 * gemm_epilogue -- out[M][N] = bf16( act(alpha * A*B~ + beta*C + bias) + residual )
 *   A         [M][K] bf16, required.
 *   B         b_layout == GBF_B_KN: [K][N] bf16;  GBF_B_NK: W [N][K] bf16
 *             (then B~ = W^T).  Required.
 *   C         [M][N] bf16 or NULL.   bias [N] bf16 or NULL (broadcast over rows).
 *   residual  [M][N] bf16 or NULL, added after the activation; may equal out.
 *   out       [M][N] bf16, required.
 *   workspace unused by the fused kernels (pass NULL, 0).
 * Order of the ending: bias inside the activation, residual outside it
 * ("Fusion and Epilogues", epilogue-fusion bullet; "Kernel fusion" guide,
 * "Check yourself": bias, activation and residual add in one pass).
 */
GBF_API gbf_status_t gemm_epilogue(const void *A, const void *B, int b_layout, const void *C,
                           const void *bias, const void *residual, void *out, int64_t M,
                           int64_t N, int64_t K, float alpha, float beta, int act,
                           void *workspace, size_t workspace_bytes, gbf_stream_t stream);

/*
 * swiglu_dual_gemm -- h[M][N] = bf16( act(alpha*g) * (alpha*u) + beta*C ),
 *   g = x*Wg~, u = x*Wu~ with the same layout rule as gemm_epilogue
 *   ("Fusion Thinking", Pattern 2, level 2: both products from one x tile in
 *   one kernel, SiLU(gate)*up in the epilogue).  act = GBF_ACT_SILU gives
 *   SwiGLU; GELU_TANH / RELU / IDENTITY give the other gated units.
 *   x [M][K]; w_gate, w_up [N][K] (GBF_B_NK) or [K][N] (GBF_B_KN); C [M][N]
 *   or NULL; h [M][N].  Workspace unused (NULL, 0).
 */
GBF_API gbf_status_t swiglu_dual_gemm(const void *x, const void *w_gate, const void *w_up,
                              int w_layout, void *h, int64_t M, int64_t N, int64_t K,
                              float alpha, float beta, const void *C, int act,
                              void *workspace, size_t workspace_bytes, gbf_stream_t stream);

/*
 * w4a16_gemm -- the gemm_epilogue result with B~[k][n] = bf16((q[k][n] - 8) * s[k/G][n]),
 *   dequantised on-chip ("Fusion Thinking", Pattern 3: the kernel loads int4
 *   weights and scales directly, dequantises them on-chip, zero point 8).
 *   Wq     [K][N/2] bytes; byte j of row k holds column 2j in its HIGH nibble
 *          and column 2j+1 in its LOW nibble (interleave(w_hi, w_lo)).
 *   scales [K/group_size][N] bf16.   group_size: a multiple of 64 dividing K.
 *   A [M][K] bf16; C, bias, residual, out as in gemm_epilogue.
 *   Requires N % 32 == 0.  Workspace unused (NULL, 0).
 */
GBF_API gbf_status_t w4a16_gemm(const void *A, const uint8_t *Wq, const void *scales, int group_size,
                        const void *C, const void *bias, const void *residual, void *out,
                        int64_t M, int64_t N, int64_t K, float alpha, float beta, int act,
                        void *workspace, size_t workspace_bytes, gbf_stream_t stream);

/*
 * w8a16_fp8_gemm -- the gemm_epilogue result with
 *   B~[k][n] = bf16( e4m3(Wq[k][n]) * s[k/G][n] ), dequantised on-chip: FP8
 *   weight-only quantisation with bf16 activations ("Fusion Thinking",
 *   Pattern 3 names INT8/FP8-class weight-only formats with BF16 activations;
 *   "Fusion and Epilogues" lists FP8 GEMM paths).
 *   Wq     [K][N] bytes, each an OCP FP8 E4M3 code (bias 7, subnormals,
 *          S.1111.111 = NaN; NaN codes are not valid weights and give an
 *          unspecified result).
 *   scales [K/group_size][N] bf16; group_size a multiple of 64 dividing K
 *          (group_size == K: one scale per output channel).
 *   The one rounding is the product e4m3 * s to bf16 (round to nearest even).
 *   Requires N % 32 == 0.  Workspace unused (NULL, 0).
 *
 * w4a16_nvfp4_gemm -- the gemm_epilogue result with
 *   B~[k][n] = e2m1(q[k][n]) * e4m3(S[k/16][n])   (exact in bf16),
 *   NVFP4 weight-only quantisation with bf16 activations ("Fusion Thinking",
 *   Pattern 3 lists NVFP4 among the weight-only formats used with bf16
 *   activations).
 *   Wq     [K][N/2] bytes of OCP FP4 E2M1 codes, packed like w4a16_gemm's
 *          (column 2j in the HIGH nibble of byte j).
 *   scales [K/16][N] bytes, each an E4M3 factor for 16 consecutive k.
 *   The format's per-tensor factor is alpha (it multiplies the product);
 *   a finite alpha with |alpha| >= 2^100 returns GBF_ERR_INVALID_ARG.
 *   Requires K % 16 == 0 and N % 32 == 0.  Workspace unused (NULL, 0).
 */
GBF_API gbf_status_t w8a16_fp8_gemm(const void *A, const uint8_t *Wq, const void *scales,
                                    int group_size, const void *C, const void *bias,
                                    const void *residual, void *out, int64_t M, int64_t N,
                                    int64_t K, float alpha, float beta, int act, void *workspace,
                                    size_t workspace_bytes, gbf_stream_t stream);
GBF_API gbf_status_t w4a16_nvfp4_gemm(const void *A, const uint8_t *Wq, const uint8_t *scales,
                                      const void *C, const void *bias, const void *residual,
                                      void *out, int64_t M, int64_t N, int64_t K, float alpha,
                                      float beta, int act, void *workspace,
                                      size_t workspace_bytes, gbf_stream_t stream);

/*
 * swiglu_pointwise -- the level-1 fused gated ending on its own:
 *   h[M][N] = bf16( act(alpha*g) * (alpha*u) + beta*C ) from bf16 g, u, C
 *   ("Fusion Thinking", Pattern 2, level 1: one elementwise kernel replaces
 *   the separate sigmoid, multiply and multiply of an eager framework; SiLU
 *   computed in fp32).  Unlike the page's snippet, silu(g) is not rounded to
 *   bf16 before the product (one rounding at the end, as everywhere here).
 *   g, u, C (nullable), h: [M][N] bf16, 16-byte aligned, N % 8 == 0.
 *   HBM-bound: reads g and u (and C) once, writes h once.
 */
GBF_API gbf_status_t swiglu_pointwise(const void *g, const void *u, const void *C, void *h,
                                      int64_t M, int64_t N, float alpha, float beta, int act,
                                      gbf_stream_t stream);

/*
 * add_rmsnorm -- fused residual add + RMSNorm, per row m:
 *   r = a + x (fp32);  out_resid = bf16(r);
 *   out_norm = bf16( r * rsqrt(mean_j(r_j^2) + eps) * weight )
 *   ("Fusion Thinking", Pattern 1, Fused RMSNorm + residual: one pass reads
 *   attn_out and x once, writes the residual for the next add and the
 *   normalised tensor).  The norm uses the unrounded fp32 sum.
 *   a, x: [M][N] bf16; weight: [N] bf16; out_norm, out_resid: [M][N] bf16
 *   (out_resid may be NULL: not written).  N % 8 == 0 and N <= 16384; eps >= 0.
 *   HBM-bound: reads a and x once, writes each result once.
 * add_rmsnorm_unfused -- the same as two kernels: bf16(a + x) written to
 *   out_resid (required), then an RMSNorm kernel that reads it back
 *   ("x = x + a; rmsnorm(x)"); the norm is then taken of the bf16 residual.
 */
GBF_API gbf_status_t add_rmsnorm(const void *a, const void *x, const void *weight, void *out_norm,
                                 void *out_resid, int64_t M, int64_t N, float eps,
                                 gbf_stream_t stream);
GBF_API gbf_status_t add_rmsnorm_unfused(const void *a, const void *x, const void *weight,
                                         void *out_norm, void *out_resid, int64_t M, int64_t N,
                                         float eps, gbf_stream_t stream);

/*
 * mlp_swiglu_down -- one gated MLP block with its residual add:
 *   h   = bf16( silu(x*Wg^T) * (x*Wu^T) )     [M][F]   (the fused gate/up GEMM)
 *   out = bf16( h*Wd^T + residual )            [M][D]   (GEMM with the residual fused)
 *   ("Fusion Thinking", Pattern 2: gate = W_gate x, up = W_up x,
 *   h = silu(gate)*up, out = W_down h; with Pattern 1's "h = mlp(h) + h").
 *   x [M][D]; w_gate, w_up [F][D]; w_down [D][F] (all K-contiguous); residual
 *   [M][D] or NULL (may equal out); out [M][D].  h lives in the workspace
 *   (gbf_workspace_size(GBF_OP_MLP, M, D, F, 1) bytes) and is left there.
 *   Two kernel launches on `stream`, no host synchronisation between them.
 * mlp_swiglu_down_unfused -- the same block the eager way: two GEMMs writing
 *   g and u, the GLU pointwise pass, the down GEMM writing bf16 D, the
 *   residual pointwise pass (workspace: gbf_workspace_size(GBF_OP_MLP, M, D,
 *   F, 0) bytes: g, u, h, D in 256-byte aligned sections).
 */
GBF_API gbf_status_t mlp_swiglu_down(const void *x, const void *w_gate, const void *w_up,
                                     const void *w_down, const void *residual, void *out,
                                     int64_t M, int64_t D, int64_t F, void *workspace,
                                     size_t workspace_bytes, gbf_stream_t stream);
GBF_API gbf_status_t mlp_swiglu_down_unfused(const void *x, const void *w_gate,
                                             const void *w_up, const void *w_down,
                                             const void *residual, void *out, int64_t M,
                                             int64_t D, int64_t F, void *workspace,
                                             size_t workspace_bytes, gbf_stream_t stream);

/*
 * Unfused reference compositions: the same results as above, computed the
 * way an eager framework does it, with the intermediate written to HBM and
 * read back by a second kernel ("kernel fusion" wiki: unfused, the product
 * writes its whole output and a second kernel reads it, applies the
 * activation and writes it again; "Fusion Thinking", Pattern 2 un-fused and
 * Pattern 3 un-fused).  They exist to measure the bytes fusion deletes.
 * The intermediates live in the caller's workspace (256-byte aligned
 * sections, gbf_workspace_size() bytes):
 *   gemm_epilogue_unfused   D = bf16(A*B~) [M][N] at offset 0, then the
 *                           pointwise ending D -> out.
 *   swiglu_dual_gemm_unfused  g = bf16(x*Wg~) [M][N] at 0, u = bf16(x*Wu~)
 *                           [M][N] at align256(2*M*N), then the GLU pass.
 *   w4a16_gemm_unfused      w = bf16((q-8)*s) [K][N] at 0, then a bf16
 *                           GEMM with the fused ending (identical result).
 *   w8a16_fp8_gemm_unfused, w4a16_nvfp4_gemm_unfused   the same with the
 *                           FP8 / NVFP4 weight dequantised into [K][N] bf16.
 * The workspace contents are left in place after the call.
 */
GBF_API gbf_status_t gemm_epilogue_unfused(const void *A, const void *B, int b_layout, const void *C,
                                   const void *bias, const void *residual, void *out,
                                   int64_t M, int64_t N, int64_t K, float alpha, float beta,
                                   int act, void *workspace, size_t workspace_bytes,
                                   gbf_stream_t stream);
GBF_API gbf_status_t swiglu_dual_gemm_unfused(const void *x, const void *w_gate, const void *w_up,
                                      int w_layout, void *h, int64_t M, int64_t N, int64_t K,
                                      float alpha, float beta, const void *C, int act,
                                      void *workspace, size_t workspace_bytes,
                                      gbf_stream_t stream);
GBF_API gbf_status_t w4a16_gemm_unfused(const void *A, const uint8_t *Wq, const void *scales,
                                int group_size, const void *C, const void *bias,
                                const void *residual, void *out, int64_t M, int64_t N,
                                int64_t K, float alpha, float beta, int act, void *workspace,
                                size_t workspace_bytes, gbf_stream_t stream);
GBF_API gbf_status_t w8a16_fp8_gemm_unfused(const void *A, const uint8_t *Wq,
                                            const void *scales, int group_size, const void *C,
                                            const void *bias, const void *residual, void *out,
                                            int64_t M, int64_t N, int64_t K, float alpha,
                                            float beta, int act, void *workspace,
                                            size_t workspace_bytes, gbf_stream_t stream);
GBF_API gbf_status_t w4a16_nvfp4_gemm_unfused(const void *A, const uint8_t *Wq,
                                              const uint8_t *scales, const void *C,
                                              const void *bias, const void *residual, void *out,
                                              int64_t M, int64_t N, int64_t K, float alpha,
                                              float beta, int act, void *workspace,
                                              size_t workspace_bytes, gbf_stream_t stream);

/*
 * gemm_epilogue_unfused_noalloc -- the gemm_epilogue_unfused result for a
 *   caller that cannot allocate device memory: code running inside a host
 *   framework that owns every device allocation, or under a policy that
 *   forbids new allocations once the process has started, so it has no way
 *   to hand over a workspace.  The bf16 intermediate lives in a scratch
 *   array built into the library instead.  The pages have no counterpart to
 *   this entry point; it exists for such callers only.
 *   Arguments are checked as gemm_epilogue_unfused checks them (same status
 *   codes); then sizes with M*N > 4194304 elements (the array holds 8 MiB,
 *   and every GPU that loads the library holds it until the process exits)
 *   return GBF_ERR_WORKSPACE before anything is launched.  The first call on
 *   a device looks up the array's device address, so make it before any
 *   stream capture; a failed lookup returns GBF_ERR_CUDA and is tried again
 *   by the next call.  Every call shares the one array: calls whose work
 *   overlaps on the GPU race on it and must be serialised by the caller.
 *   Allocates nothing.  Other arguments and results as gemm_epilogue.
 */
GBF_API gbf_status_t gemm_epilogue_unfused_noalloc(const void *A, const void *B, int b_layout,
                                                   const void *C, const void *bias,
                                                   const void *residual, void *out, int64_t M,
                                                   int64_t N, int64_t K, float alpha, float beta,
                                                   int act, gbf_stream_t stream);

/* Workspace bytes an entry point needs (0 for the fused ones).  `op` is a
 * GBF_OP_* id; `fused` selects the fused (1) or unfused (0) entry point. */
GBF_API size_t gbf_workspace_size(int op, int64_t M, int64_t N, int64_t K, int fused);

/* Synchronises `stream`, then reads and clears the library's device error
 * word on the current device.  Returns GBF_OK, GBF_ERR_TIMEOUT (a kernel
 * gave up on a bounded wait; its output is undefined) or GBF_ERR_CUDA. */
GBF_API gbf_status_t gbf_check_device_error(gbf_stream_t stream);

/* A static, human-readable name of a status code. */
GBF_API const char *gbf_status_string(gbf_status_t status);

/* Limit, in nanoseconds, of every bounded wait inside the kernels (default
 * 2e9 = 2 s; clamped to [1e6, 6e10]).  Applies to later launches. */
GBF_API gbf_status_t gbf_set_wait_timeout_ns(uint64_t ns);


/* Which kernel family a call with these arguments runs (for tests and the
 * benchmark's roofline attribution).  op: GBF_OP_GEMM_EPILOGUE,
 * GBF_OP_SWIGLU, GBF_OP_W4A16, GBF_OP_W8A16_FP8 or GBF_OP_W4A16_NVFP4.
 * Returns 1 = persistent 128x256-tile kernel, 2 = small-M swapped kernel
 * with cluster split-K (also the gate/up GEMM at M <= 32), 3 = weight-only
 * kernel (int4, FP8, NVFP4), 4 = persistent kernel on CTA pairs (chosen over 1
 * when its 512-row units fill the GPU better), 5 = the persistent kernel's
 * split-K form (two CTAs per tile, chosen when the tiles fill at most half
 * of the SMs), 6 = the CTA-pair kernel with one MMA stream (units of 256
 * rows), 7 = its split-K form (two CTA pairs per 256 x 256 tile, each over
 * half of K, chosen when every tile's cluster fits at once), 0 = no launch
 * (empty output), -1 = the arguments would be rejected.
 * `*splits` (may be NULL) receives the split-K cluster size.
 *
 * Kernels of families 2, 3, 4, 6 and 7 are launched with programmatic stream
 * serialization: they may begin while the previous kernel in the stream is
 * finishing, and read or write nothing in global memory before it has
 * completed (griddepcontrol.wait), so stream order is preserved. */
GBF_API int gbf_kernel_path(int op, int64_t M, int64_t N, int64_t K, int b_layout, int *splits);

/* Library version, e.g. 100 for 1.0.0. */
GBF_API int gbf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBFUSE_H */
