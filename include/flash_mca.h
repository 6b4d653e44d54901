/*
 * flash_mca.h -- C ABI of the FLASH mixed-chunk attention forward core on GB300.
 *
 * The operation (one call = one forward pass of the attention core of a GAU
 * layer, after its U/V/Z projections and before its W_o projection) follows
 * "FLASH: Possibly the Most Interesting Efficient Transformer Design Recently"
 * (kexue.fm archive 8934):
 *
 *   T_k = Z * gamma[k] + beta[k], k = 0..3       section "Weak Attention", eq.
 *                                                relu-att (affine Q, K of Z) and
 *                                                "Mixed Chunk" (four maps: quad_q,
 *                                                quad_k, lin_q, lin_k)
 *   chunks of C tokens, G = n / C                "Mixed Chunk", first paragraph
 *   quad_g = relu(T0_g T1_g^T / C)^2 V_g,        "Mixed Chunk", eq. for V^quad_g;
 *            strict upper triangle masked         masking sentence (decoder)
 *            in causal mode
 *   lin_g  = T2_g (sum_h T3_h^T V_h) / n         "Mixed Chunk", eq. for V^lin_g
 *            over all chunks h (bidirectional)   (non-causal form) and its cumsum
 *            or chunks h < g (causal)            form for a decoder
 *   O_g    = U_g * (quad_g + lin_g)              "Mixed Chunk", eq. for O_g
 *                                                (W_o is not applied here)
 *
 * Readings where the page leaves a choice: the intra-chunk scale is relu(x/C)^2
 * (the appendix scale relu(x/n)^2 of "Weak Attention" applied to a chunk); the
 * global normaliser is 1/n in both modes; the causal sum over chunks is
 * exclusive (h < g), so chunk 0 has no global term; the causal mask keeps the
 * diagonal.
 *
 * Layouts (all row-major, contiguous, last index fastest):
 *   Z[B][n][s], V[B][n][e], U[B][n][e], O[B][n][e]  -- element type `dtype`
 *   gamma[4][s], beta[4][s]                         -- float32, rows in the
 *                                                      order quad_q, quad_k,
 *                                                      lin_q, lin_k
 *
 * Ownership: every pointer is owned by the caller; the library allocates no
 * memory.  Device pointers must stay valid until the work queued on `stream`
 * has finished.
 *
 * Errors: every argument check runs on the host before anything is queued; a
 * call that returns a status other than FMCA_OK has queued nothing, except for
 * FMCA_ERR_CUDA (a launch or copy failed after earlier work was queued).  The
 * kernels never trap: a bounded wait that runs out records FMCA_ERR_TIMEOUT in
 * a device-side status word that flash_mca_device_status() returns.
 */
#ifndef FLASH_MCA_H
#define FLASH_MCA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (the same object as cudaStream_t); NULL is the
 * legacy default stream. */
typedef struct CUstream_st *fmca_stream_t;

typedef int32_t fmca_status;
#define FMCA_OK 0
#define FMCA_ERR_INVALID_ARG 1 /* NULL pointer, non-positive size, bad enum */
#define FMCA_ERR_SHAPE 2       /* C does not divide n, or C > n */
#define FMCA_ERR_UNSUPPORTED 3 /* shape outside what the kernels support */
#define FMCA_ERR_ALIGN 4       /* a device pointer is not 16-byte aligned */
#define FMCA_ERR_WORKSPACE 5   /* workspace NULL or smaller than required */
#define FMCA_ERR_CUDA 6        /* a CUDA launch or copy failed */
#define FMCA_ERR_TIMEOUT 7     /* a bounded device-side wait ran out */

typedef int32_t fmca_dtype;
#define FMCA_F32 0  /* Z, V, U, O are float32; arithmetic in fp32 FMA */
#define FMCA_BF16 1 /* Z, V, U, O are bfloat16; tensor-core products with
                       fp32 accumulation, output rounded to nearest even */

/* Which kernels carry a call. */
typedef int32_t fmca_path;
#define FMCA_PATH_AUTO 0    /* tensor-core path when the shape allows it,
                               else the SIMT path */
#define FMCA_PATH_SIMT 1    /* CUDA-core fp32 kernels, any supported shape */
#define FMCA_PATH_TCGEN05 2 /* tcgen05/TMEM + TMA kernels; FMCA_BF16 only,
                               s == 128, C % 128 == 0, e % 64 == 0
                               (e % 256 == 0 without a global term for
                               C > 256, and for the backward pass) */

/* Supported sizes: B, n, s, e >= 1; 1 <= C <= n with n % C == 0; s <= 256;
 * B * n * max(s, e) < 2^31.  The tensor-core path additionally needs the
 * conditions listed at FMCA_PATH_TCGEN05.
 *
 * Tensor-core coverage of the bf16 shapes: the tcgen05 kernels take s = 128
 * (the pages' attention width), C a multiple of 128 (128, 256, ..., up to
 * C = n for the quadratic-only model) and e a multiple of 64.  Two forms
 * need e a multiple of 256: the quadratic-only model with chunks over 256
 * tokens (FMCA_LIN_NORM_NONE, C > 256), whose relu^2 weights go through the
 * workspace, and the backward pass.  Every other bf16 shape in the
 * supported sizes (s = 16 ... 256 other than 128, C = 64 or any C that is
 * not a multiple of 128, e not a multiple of 64) runs the fp32 CUDA-core
 * kernels: correct, to the fp32 bar, but several times slower.
 * FMCA_PATH_AUTO picks the tensor-core path whenever it applies
 * (flash_mca_auto_path answers for the default options). */

/*
 * Bytes of device workspace one flash_mca_forward call with these arguments
 * needs, whichever path it takes.  SIMT path: the per-chunk linear-attention
 * states and their prefix sums, fp32.  Tensor-core path (whose relu^2 weights
 * never leave the chip): in causal mode the chunks' local state sums (bf16,
 * the sum of the states before each chunk within its segment of the chunk
 * axis), the segment totals that become carries (bf16), the rows T0, T1, T2
 * (bf16) and 256 bytes of counters.
 * Returns 0 for arguments flash_mca_forward would reject.
 */
size_t flash_mca_workspace_bytes(int B, int n, int s, int e, int C, int causal,
                                 fmca_dtype dtype);

/*
 * The forward pass O = U * (quad + lin) described at the top of this file.
 *   Z, V, U, O     device pointers, 16-byte aligned, element type `dtype`;
 *                  O must not overlap Z, V, U or the workspace.
 *   gamma, beta    device pointers to float32 [4][s].
 *   causal         nonzero: decoder form (masked chunk, exclusive chunk sum).
 *   workspace      device buffer of at least flash_mca_workspace_bytes(...)
 *                  bytes, 256-byte aligned; its contents on entry do not
 *                  matter and are undefined on exit.
 *   stream         work is queued on this stream; the call does not wait.
 * Deterministic: fixed shapes and inputs give bit-identical outputs.
 */
fmca_status flash_mca_forward(const void *Z, const void *V, const void *U,
                              const float *gamma, const float *beta, void *O, int B,
                              int n, int s, int e, int C, int causal, fmca_dtype dtype,
                              void *workspace, size_t workspace_bytes,
                              fmca_stream_t stream);

/* flash_mca_forward with an explicit choice of kernels (FMCA_PATH_*).
 * FMCA_PATH_TCGEN05 returns FMCA_ERR_UNSUPPORTED for shapes it does not
 * cover instead of falling back. */
fmca_status flash_mca_forward_path(const void *Z, const void *V, const void *U,
                                   const float *gamma, const float *beta, void *O, int B,
                                   int n, int s, int e, int C, int causal,
                                   fmca_dtype dtype, void *workspace,
                                   size_t workspace_bytes, fmca_path path,
                                   fmca_stream_t stream);

/*
 * Scale and normalisation variants.  The page states some factors in more
 * than one way; flash_mca_forward uses the readings given at the top of this
 * file, flash_mca_forward_ex lets the caller pick:
 *
 *   quad_scale   intra-chunk weights are quad_scale * relu(T0_i . T1_j)^2.
 *                "Mixed Chunk", eq. for V^quad_g, writes 1/(cs) relu^2(Q K^T):
 *                quad_scale = 1/(C s).  The default relu(x/C)^2 (the appendix
 *                scale of "Weak Attention" applied per chunk) is 1/C^2.
 *                Must be finite and >= 0.
 *   lin_norm     the divisor of the global term:
 *     FMCA_LIN_NORM_N         n, in both modes (default; "Mixed Chunk", the
 *                             non-causal eq.'s 1/n).
 *     FMCA_LIN_NORM_SUMMED    the number of tokens the global sum covers: g*C
 *                             for chunk g (counted from 0) in causal mode --
 *                             the decoder eq.'s 1/((g-1)c) with chunks counted
 *                             from 1 -- and n otherwise.  Chunk 0's causal sum
 *                             is empty, so its global term is 0.
 *     FMCA_LIN_NORM_POSITION  t+1 for the token at position t (counted from 0)
 *                             of its sequence ("Extended Thoughts": the sum of
 *                             the first t items should be divided by t).
 *     FMCA_LIN_NORM_NONE      no global term at all.  With C = n this is the
 *                             quadratic-only model FLASH-Quad ("Weak
 *                             Attention": relu(q.k / n)^2 attention over the
 *                             whole sequence, the upper triangle masked for a
 *                             decoder); the kernels then skip the chunk
 *                             states, the scan and the global product.
 */
typedef int32_t fmca_lin_norm;
#define FMCA_LIN_NORM_N 0
#define FMCA_LIN_NORM_SUMMED 1
#define FMCA_LIN_NORM_POSITION 2
#define FMCA_LIN_NORM_NONE 3

typedef struct fmca_options {
  float quad_scale;
  fmca_lin_norm lin_norm;
} fmca_options;

/* Fills *opts with the defaults for chunk length C (quad_scale = 1/C^2,
 * lin_norm = FMCA_LIN_NORM_N).  FMCA_ERR_INVALID_ARG for C <= 0 or NULL. */
fmca_status flash_mca_default_options(int C, fmca_options *opts);

/* flash_mca_forward_path with the variants of `opts` (host pointer, read
 * during the call; NULL means the defaults).  A negative or non-finite
 * quad_scale or an unknown lin_norm returns FMCA_ERR_INVALID_ARG.  Same
 * kernels, workspace and launch count as flash_mca_forward_path. */
fmca_status flash_mca_forward_ex(const void *Z, const void *V, const void *U,
                                 const float *gamma, const float *beta, void *O, int B,
                                 int n, int s, int e, int C, int causal, fmca_dtype dtype,
                                 void *workspace, size_t workspace_bytes, fmca_path path,
                                 const fmca_options *opts, fmca_stream_t stream);

/*
 * One piece of longer causal sequences: the pages' cumsum form of the global
 * term ("Mixed Chunk") carried across calls, so that a long sequence can be
 * split over calls (chunked prefill) or over ranks (each rank one piece).
 *   state_in     NULL, or fp32 device [B][s][e], 16-byte aligned: the sum of
 *                T3_h^T V_h over the sequences' chunks before this piece
 *                (unscaled); every chunk of the piece adds it to its sum.
 *   state_out    NULL, or fp32 device [B][s][e], 16-byte aligned: receives
 *                state_in (or 0) plus the sum over the piece's chunks, the
 *                state_in of the next piece.  It may be state_in itself and
 *                must not overlap the other buffers.
 *   token_offset the piece's first token in its sequences (a multiple of C,
 *                >= 0): positions and chunk indices of the divisors
 *                (FMCA_LIN_NORM_SUMMED, FMCA_LIN_NORM_POSITION) count from
 *                the sequence start.
 *   n_norm       the length the default divisor 1/n uses (the whole
 *                sequence's length); 0 means the piece's n.
 */
typedef struct fmca_seq {
  const float *state_in;
  float *state_out;
  int64_t token_offset;
  int64_t n_norm;
} fmca_seq;

/* flash_mca_forward_ex (path FMCA_PATH_AUTO) on one piece of longer
 * sequences.  Only causal attention on the tensor-core path, with a global
 * term: other arguments return FMCA_ERR_UNSUPPORTED (bidirectional attention
 * needs every piece's total before any output; gather the totals first).
 * seq == NULL is flash_mca_forward_ex.  Splitting a sequence at a chunk
 * boundary and running the pieces in order with state_out of one as state_in
 * of the next gives the output of one call on the whole sequence (within the
 * same error bounds: the sums are rounded at other points).  The workspace is
 * the one flash_mca_workspace_bytes gives for the piece. */
fmca_status flash_mca_forward_seq(const void *Z, const void *V, const void *U,
                                  const float *gamma, const float *beta, void *O, int B, int n,
                                  int s, int e, int C, int causal, fmca_dtype dtype,
                                  void *workspace, size_t workspace_bytes,
                                  const fmca_options *opts, const fmca_seq *seq,
                                  fmca_stream_t stream);

/* flash_mca_forward_ex that also records caller-created CUDA events
 * (cudaEvent_t handles) on `stream` around its kernels: events[0] before the
 * first kernel and events[i] after kernel i (1-based), so `n_events` must be
 * flash_mca_launch_count(...) + 1.  Lets a caller time each kernel on the
 * stream it runs on.  `opts` as for flash_mca_forward_ex (NULL: defaults).
 * Kernel order: tensor-core path -- the segment walkers (local state sums,
 * segment totals and the rows T0, T1, T2); then, for chunks of 256, the
 * row-pair output kernel, which forms the segment carries (bidirectional: the
 * total) itself; for other chunk sizes the segment-carry kernel (only with
 * more than one segment, or bidirectional) and the fused chunk kernel
 * (scores, relu^2 weights, both products and the gate); without a
 * global term (FMCA_LIN_NORM_NONE) the rows T0, T1, then the fused kernel;
 * SIMT path -- chunk states, state scan, chunk output. */
fmca_status flash_mca_forward_timed(const void *Z, const void *V, const void *U,
                                    const float *gamma, const float *beta, void *O, int B,
                                    int n, int s, int e, int C, int causal,
                                    fmca_dtype dtype, void *workspace,
                                    size_t workspace_bytes, fmca_path path,
                                    const fmca_options *opts, void *const *events,
                                    int n_events, fmca_stream_t stream);

/*
 * Autoregressive decoding, one token per call, in the recurrent form of the
 * causal core ("Mixed Chunk": the decoder's masked intra-chunk term and the
 * cumsum form of the global term; the linear-attention recurrence of
 * "大模型训练之加速篇 -attention优化", section 1.4).  For B sequences decoded in
 * lockstep, the token at position t (chunk g = t / C, index i = t % C) gets
 *
 *   o = u * ( sum_{j <= i in chunk g} quad_scale * relu(T0_t . T1_j)^2 v_j
 *           + T2_t . (sum_{h < g} T3_h^T V_h) / d(t) )
 *
 * which is row t of flash_mca_forward(causal = 1) over the sequence decoded so
 * far.  d(t) is n_norm (FMCA_LIN_NORM_N: pass the length n of the sequence
 * whose forward pass the decode must reproduce), g*C (FMCA_LIN_NORM_SUMMED) or
 * t+1 (FMCA_LIN_NORM_POSITION); quad_scale and lin_norm come from `opts`
 * (NULL: the defaults).  The caller-owned device `state` carries the fp32 sum
 * of T3^T V over completed chunks (with FMCA_BF16 also a bf16 copy of it,
 * refreshed at each fold, which the per-token reads use) and the current
 * chunk's Z and V rows:
 *
 *   flash_mca_decode_state_bytes  its size (0 for rejected sizes);
 *   flash_mca_decode_reset        clears it before position 0 (queued on
 *                                 `stream`);
 *   flash_mca_decode_step         one token: z [B][s], v, u, o [B][e] device
 *                                 arrays of `dtype`, 16-byte aligned; calls
 *                                 must come in order t = 0, 1, 2, ... on one
 *                                 stream (the state is not told which
 *                                 positions it has seen).  The last token of a
 *                                 chunk also folds the chunk into the state.
 *
 * Sizes: B, s, e >= 1, s <= 256, 1 <= C <= 1024, t >= 0; n_norm > t for
 * FMCA_LIN_NORM_N (ignored otherwise).  fp32 arithmetic on the CUDA cores.
 */
size_t flash_mca_decode_state_bytes(int B, int s, int e, int C, fmca_dtype dtype);
fmca_status flash_mca_decode_reset(void *state, size_t state_bytes, int B, int s, int e, int C,
                                   fmca_dtype dtype, fmca_stream_t stream);
fmca_status flash_mca_decode_step(const void *z, const void *v, const void *u,
                                  const float *gamma, const float *beta, void *o, int B, int s,
                                  int e, int C, int t, int n_norm, fmca_dtype dtype,
                                  const fmca_options *opts, void *state, size_t state_bytes,
                                  fmca_stream_t stream);

/*
 * Backward pass: gradients of sum(O * dO) for the O that flash_mca_forward_ex
 * computes with the same arguments and options.  The pages define only the
 * forward pass ("Mixed Chunk"); the gradient follows by calculus through the
 * gate, the masked relu^2 chunk attention, the chunk states and their
 * exclusive (causal) or total sum with its divisor, and the four affine maps.
 *   Z, V, U, dO          device arrays of `dtype` (layouts as for the forward)
 *   dZ, dV, dU           device outputs of `dtype` (overwritten)
 *   dgamma, dbeta        device float32 [4][s] outputs (overwritten)
 *   workspace            at least flash_mca_backward_workspace_bytes(...) bytes,
 *                        256-byte aligned
 * bf16 inputs with s == 128, C % 128 == 0 and e % 256 == 0 run on the
 * tensor cores: the forward kernels recompute the
 * ungated output and the relu^2 weights, and batched bf16 products with fp32
 * accumulation form the gradients (intermediates rounded to bf16).  Every
 * other shape, and float32, runs in fp32 on the CUDA cores.  Both use a fixed
 * reduction order (deterministic).  Sizes as for flash_mca_forward (any
 * supported shape, both dtypes); the workspace size depends on which path the
 * shape takes.  The outputs must not overlap the inputs or the workspace.
 */
size_t flash_mca_backward_workspace_bytes(int B, int n, int s, int e, int C, int causal,
                                          fmca_dtype dtype);
fmca_status flash_mca_backward(const void *Z, const void *V, const void *U, const float *gamma,
                               const float *beta, const void *dO, void *dZ, void *dV, void *dU,
                               float *dgamma, float *dbeta, int B, int n, int s, int e, int C,
                               int causal, fmca_dtype dtype, const fmca_options *opts,
                               void *workspace, size_t workspace_bytes, fmca_stream_t stream);

/*
 * flash_mca_backward for training loops that keep the forward pass's
 * intermediates: the same gradients, but the chunk states and their scaled
 * prefix are not recomputed.  `workspace` must hold what an earlier
 * flash_mca_forward (or _ex, FMCA_PATH_AUTO or FMCA_PATH_TCGEN05) left in it,
 * called with the same Z, V, U, gamma, beta, sizes and options and with this
 * workspace (sized by flash_mca_backward_workspace_bytes: the forward pass
 * uses its first flash_mca_workspace_bytes), with nothing written to it
 * since; the library cannot check this.  The relu^2 weights and lin_q rows
 * (which the forward pass keeps on chip) and the output kernel (fed dO, for
 * dU) run again.  FMCA_BF16 with s == 128, C % 128 == 0 and e % 256 == 0
 * only; others return FMCA_ERR_UNSUPPORTED.
 */
/* Number of kernels one flash_mca_backward (saved = 0) or
 * flash_mca_backward_saved (saved = 1) call launches for these arguments (0
 * when they would be rejected). */
int flash_mca_backward_launch_count(int B, int n, int s, int e, int C, int causal,
                                    fmca_dtype dtype, const fmca_options *opts, int saved);
fmca_status flash_mca_backward_saved(const void *Z, const void *V, const void *U,
                                     const float *gamma, const float *beta, const void *dO,
                                     void *dZ, void *dV, void *dU, float *dgamma, float *dbeta,
                                     int B, int n, int s, int e, int C, int causal,
                                     fmca_dtype dtype, const fmca_options *opts, void *workspace,
                                     size_t workspace_bytes, fmca_stream_t stream);

/*
 * The dense projections of a GAU layer around the attention core, on the
 * tensor cores (bf16 in, fp32 accumulation, bf16 out):
 *   flash_mca_gau_project  U = SiLU(X W_u), V = SiLU(X W_v), Z = SiLU(X W_z)
 *                          ("Initial Power": U and V with the Swish activation;
 *                          "Weak Attention": Z = phi(X W_z))
 *   flash_mca_gau_output   Out = Y W_o ("Strong Combination", eq. mix: the
 *                          layer output (U * A V) W_o, Y being the core's O)
 * No biases (the equations have none).  Weights are passed transposed, one
 * row per output feature:
 *   Wt   [2e + s][d]  rows 0..e-1 = columns of W_u, e..2e-1 = W_v, 2e.. = W_z
 *   Wo_t [d][e]       = W_o^T
 * X [M][d], U and V [M][e], Z [M][s], Y [M][e], Out [M][d]: row-major bf16
 * device arrays, 16-byte aligned, outputs not overlapping inputs.  Sizes:
 * M >= 1; d % 8 == 0; e and s multiples of 64 (project); d a multiple of 64
 * (output).  Queued on `stream`, nothing allocated.
 */
fmca_status flash_mca_gau_project(const void *X, const void *Wt, void *U, void *V, void *Z,
                                  int M, int d, int e, int s, fmca_stream_t stream);
fmca_status flash_mca_gau_output(const void *Y, const void *Wo_t, void *Out, int M, int e,
                                 int d, fmca_stream_t stream);

/* Which path FMCA_PATH_AUTO takes for these arguments (FMCA_PATH_SIMT or
 * FMCA_PATH_TCGEN05), or -1 for arguments that would be rejected. */
int flash_mca_auto_path(int B, int n, int s, int e, int C, int causal, fmca_dtype dtype);

/* Number of kernel launches one flash_mca_forward call queues for these
 * arguments (0 when they would be rejected); memsets are not counted. */
int flash_mca_launch_count(int B, int n, int s, int e, int C, int causal,
                           fmca_dtype dtype, fmca_path path);
/* The same for flash_mca_forward_ex with options `opts` (NULL: the defaults):
 * without a global term (FMCA_LIN_NORM_NONE) the tensor-core path launches
 * fewer kernels.  flash_mca_forward_timed takes this count + 1 events. */
int flash_mca_launch_count_ex(int B, int n, int s, int e, int C, int causal,
                              fmca_dtype dtype, fmca_path path, const fmca_options *opts);

/*
 * End-to-end variant on HOST buffers: copies Z, V, U, gamma, beta from host
 * memory into `device_arena`, runs flash_mca_forward on `stream`, copies O
 * back to host memory and waits for the stream before returning, so hO is
 * ready on return.  Host buffers should be page-locked for the copies to run
 * at full speed (pageable memory works, more slowly).  With at least two
 * sequences and 96 MB of inputs and output, the call runs pieces so that
 * copies and passes overlap: up to four pieces of whole sequences, or, with
 * fewer than four causal sequences on the tensor-core path, four (or two)
 * pieces of every sequence's tokens run in order with the chunk-state sum
 * carried between them (flash_mca_forward_seq).  The copies go on two
 * streams of the library's own (created once per device), chained to
 * `stream` by events, the passes on `stream`.  Each piece is a batch of its
 * own, so the output bits can differ from one flash_mca_forward call on the
 * whole batch (within the same error bounds).
 *   device_arena   caller-owned device buffer, 256-byte aligned, of at least
 *                  flash_mca_host_arena_bytes(...) bytes; it holds the device
 *                  copies of the inputs and output, the workspace and the
 *                  carried state of token pieces (fp32 [B][s][e]).
 */
size_t flash_mca_host_arena_bytes(int B, int n, int s, int e, int C, int causal,
                                  fmca_dtype dtype);
fmca_status flash_mca_forward_host(const void *hZ, const void *hV, const void *hU,
                                   const float *hgamma, const float *hbeta, void *hO,
                                   int B, int n, int s, int e, int C, int causal,
                                   fmca_dtype dtype, void *device_arena,
                                   size_t arena_bytes, fmca_stream_t stream);

/*
 * flash_mca_forward without a caller-provided workspace, for callers that
 * cannot allocate device memory: code running inside a host framework that
 * owns all device memory and only lends out the tensors it manages, code that
 * must not call cudaMalloc (an allocation lock held elsewhere, or a hard rule
 * against failing half-way on an out-of-memory error).  The computation has no
 * counterpart on the pages: it is the same forward pass, only the scratch
 * comes from a fixed array inside the library.
 *
 * The scratch is one array of FMCA_NOALLOC_SCRATCH_BYTES compiled into the
 * library; a GPU keeps it until the process exits once this entry point has
 * run there (with eager module loading, CUDA_MODULE_LOADING=EAGER, every GPU
 * the process creates a context on holds it, whichever entry points run).
 * Problems whose tensor-core scratch (in causal mode the bf16 local state
 * sums, 2 B G s e bytes; the bf16 segment totals, 2 B S s e bytes with S the
 * segments of the chunk axis; the bf16 rows T0, T1, T2, 6 B n s bytes; 256
 * bytes of counters) exceeds it are rejected with FMCA_ERR_WORKSPACE: B=2,
 * n=8192, C=256, e=1536 fits (46.4 MB); B=1, n=32768, C=256, e=2048
 * (100.7 MB) must use flash_mca_forward.  Only the tensor-core path is available (FMCA_BF16,
 * s == 128, C % 128 == 0, e % 256 == 0); other shapes return
 * FMCA_ERR_UNSUPPORTED.
 *
 * The first call on a device looks up the array's device address on that
 * device (the current one); make that first call before any CUDA stream
 * capture begins.  The address is looked up again when the device's primary
 * context has changed since (after cudaDeviceReset).  All calls on a device share the array: calls whose work
 * overlaps on the GPU (different streams) race and give wrong results; calls
 * queued on one stream are ordered.  The call allocates nothing, queues its
 * kernels on `stream` and does not wait.  Arguments as for flash_mca_forward.
 */
#define FMCA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20) /* 64 MiB */
fmca_status flash_mca_forward_noalloc(const void *Z, const void *V, const void *U,
                                      const float *gamma, const float *beta, void *O,
                                      int B, int n, int s, int e, int C, int causal,
                                      fmca_dtype dtype, fmca_stream_t stream);

/* Status recorded by the kernels on the current device since the last call of
 * this function (FMCA_OK or FMCA_ERR_TIMEOUT); waits for `stream`, then
 * clears the record.  *where (if not NULL) receives a code naming the wait
 * that ran out (0 when none did). */
fmca_status flash_mca_device_status(fmca_stream_t stream, int32_t *where);

/* Queues one kernel whose single bounded wait can never be satisfied; with a
 * limit of `limit_us` microseconds it gives up, records FMCA_ERR_TIMEOUT and
 * returns, leaving the context usable.  Exercises the timeout path of the
 * kernels' waits without faulting or hanging the GPU. */
fmca_status flash_mca_selftest_timeout(int limit_us, fmca_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *flash_mca_status_string(fmca_status status);

/* Library version, e.g. "0.1.0". */
const char *flash_mca_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLASH_MCA_H */
