/*
 * rg.h -- C ABI of the GB300 (sm_103a) MoE grouped-GEMM library (librg.so).
 *
 * Two operations, after the RapidGEMM README, section "Kernels":
 *
 *   rg_mgemm  M-grouped BF16 GEMM for the forward pass and the input
 *             gradient ("Mgemm": x [M,K], w [E,N,K], cumulative row offsets
 *             with a leading zero, optional transpose of B).
 *   rg_kgemm  K-grouped weight gradient with FP32 output ("Kgemm": grad and
 *             X hold expert-grouped rows; dW[e] = grad[rows of e]^T X[rows of e]).
 *
 * Group boundaries may fall anywhere: they need not be multiples of any tile
 * size, and groups may be empty.  The offsets vector stays on the device and
 * is read only by the kernels, so no call synchronises with the host.
 *
 * Conventions for every entry point:
 *   - All tensors are dense and row-major.  "device" pointers must point to
 *     memory of the current CUDA device; "host" pointers to host memory.
 *   - The caller owns every buffer.  The library allocates no memory and keeps
 *     no pointer after a call returns; a call only enqueues work on `stream`
 *     and returns without waiting for it.
 *   - Return values: RG_OK (0) or a negative RG_ERR_* code.  Argument errors
 *     are detected before anything is enqueued.  Errors that only the GPU can
 *     see (invalid offsets contents, a pipeline wait that ran out) are recorded
 *     in a per-device status word read by rg_get_device_status().
 *   - No C++ exception crosses this interface.
 *   - Thread safety: calls may be made from several host threads, on one or
 *     several streams; calls on different streams are independent (except
 *     rg_kgemm_noalloc, whose calls share one fixed array: see there).
 *   - CUDA graphs: the first call on a device sets up the library's state for
 *     it (kernel attributes, grid sizes); every later call enqueues only
 *     kernel launches (rg_kgemm_ws also a memset of its workspace), so a
 *     sequence of calls may be captured in a CUDA graph and replayed with new
 *     contents in the same buffers.  This note does not cover
 *     rg_kgemm_noalloc.
 */
#ifndef RG_H_
#define RG_H_

#include <stdint.h>
#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

#define RG_OK 0
#define RG_ERR_INVALID_ARG (-1) /* null/misaligned pointer, bad size or stride */
#define RG_ERR_UNSUPPORTED (-2) /* device is not an sm_103 (GB300-class) GPU */
#define RG_ERR_CUDA (-3)        /* a CUDA call failed; see rg_last_cuda_error() */
#define RG_ERR_SCRATCH (-4)     /* rg_kgemm_noalloc: the problem needs more than the library's
                                   fixed scratch holds (RG_KGEMM_NOALLOC_MAX_FLAGS) */

/* Bits of the device status word (rg_get_device_status). */
#define RG_DEV_BAD_OFFSETS 0x1u /* offsets[0] != 0, decreasing, or offsets[E] > M */
#define RG_DEV_TIMEOUT 0x2u     /* a bounded pipeline wait ran out; the kernel stopped */
#define RG_DEV_LAUNCH_CONFIG 0x4u /* shared-memory window misaligned; the kernel did nothing */
#define RG_DEV_BOUNDS 0x8u        /* debug-bounds builds only (RG_DEBUG_BOUNDS=1): a copy or store
                                     coordinate fell outside its operand; that access was skipped */

/* Largest number of experts one call accepts. */
#define RG_MAX_EXPERTS 1024
/* Largest number of experts of rg_kgemm / rg_kgemm_acc / rg_kgemm_ws (the
 * same as every other entry point's; beyond 239 experts their per-expert
 * tables take the room of one of the four stages of the operand ring). */
#define RG_KGEMM_MAX_EXPERTS 1024
/* Largest number of outer groups of rg_mgemm_nested. */
#define RG_MAX_OUTER 65536
/* Hand-over flags in the fixed scratch of rg_kgemm_noalloc (4 bytes each). */
#define RG_KGEMM_NOALLOC_MAX_FLAGS 65536

/*
 * rg_mgemm -- M-grouped GEMM, forward (transpose_B == 0) or input gradient
 * (transpose_B != 0).  RapidGEMM README, "Kernels", Mgemm.
 *
 *   x        device, bf16 [M, K].
 *   w        device, bf16 [E, N, K] when transpose_B == 0:  y = x . w[e]^T
 *                    bf16 [E, K, N] when transpose_B != 0:  y = x . w[e]
 *            (the second form reads a forward weight [E, N_fwd, K_fwd] as B
 *            without transposing it: K = N_fwd, N = K_fwd).
 *   offsets  device, int32 [E+1]; offsets[0] == 0, non-decreasing,
 *            offsets[E] <= M.  Expert e owns rows offsets[e] .. offsets[e+1]-1.
 *   y        device, bf16 [M, N].  Row r of expert e receives
 *            y[r, n] = sum_k x[r, k] * B_e[k, n], accumulated in FP32 by the
 *            tensor cores and rounded to bf16 (nearest even).  Rows
 *            >= offsets[E] are not written.
 *   E        1 .. RG_MAX_EXPERTS.   M  0 .. 2^31-1 (M == 0 enqueues nothing).
 *   N, K     >= 8 and multiples of 8 (16-byte row strides).
 *   x, w, y must be 16-byte aligned; offsets 4-byte aligned.
 *   stream   CUDA stream (0 = legacy default stream).
 *
 * Invalid offsets contents do not fault: every CTA sees them, writes nothing
 * and sets RG_DEV_BAD_OFFSETS.
 */
int rg_mgemm(const void* x, const void* w, const int32_t* offsets, int E, int64_t M,
             int N, int K, int transpose_B, void* y, cudaStream_t stream);

/*
 * rg_mgemm_nested -- nested grouped GEMM, flattened: O outer groups split
 * the columns of x and y, and inside each, L inner groups split the rows
 * (CUTLASS discussion #1452, "Grouped GEMM where each subproblem is another
 * grouped gemm instance": batched LoRA over MoE, and an A matrix [M, 3K]
 * grouped along its columns for the outer problem and along its rows for the
 * inner one; both levels share one row-offset vector, so the problem is
 * flattened into O * L groups served by one launch).
 *
 *   x        device, bf16 [M, O*K]; outer group o reads columns o*K .. o*K+K-1.
 *   w        device, bf16 [O, L, N, K] when transpose_B == 0,
 *                    bf16 [O, L, K, N] when transpose_B != 0.
 *   offsets  device, int32 [L+1], rules as for rg_mgemm with E = L; inner
 *            group l owns rows offsets[l] .. offsets[l+1]-1 in every outer
 *            group.
 *   y        device, bf16 [M, O*N].  Row r of inner group l receives, for
 *            every o and n,
 *              y[r, o*N + n] = sum_k x[r, o*K + k] * B_{o,l}[k, n]
 *            with B_{o,l} = w[o, l]^T (or w[o, l] with transpose_B),
 *            accumulated in FP32 and rounded to bf16 (nearest even).  Rows
 *            >= offsets[L] are not written.
 *   O        1 .. RG_MAX_OUTER (O == 1 is rg_mgemm with E = L).
 *   L        1 .. RG_MAX_EXPERTS.   N, K >= 8, multiples of 8 (K may be a
 *            LoRA rank such as 16).  O*N, O*K and O*L must fit in int32.
 *   Alignment, M and stream as for rg_mgemm.
 * LoRA over MoE (adapter a, expert e) is the case O == 1 with the inner
 * groups ordered (a, e) and w = the stacked [A*E, N, K] adapter weights.
 */
int rg_mgemm_nested(const void* x, const void* w, const int32_t* offsets, int O, int L, int64_t M,
                    int N, int K, int transpose_B, void* y, cudaStream_t stream);

/*
 * rg_mx_blocked_bytes -- size in bytes that rg_mx_scales_blocked may write
 * for R scale rows of KS columns in G groups: (R/128 + G) * ceil(KS/4) * 512
 * (an upper bound of the blocks the groups need).  -1 on bad arguments.
 * Host-only; touches no device.
 */
int64_t rg_mx_blocked_bytes(int64_t R, int KS, int G);

/*
 * rg_mx_scales_blocked -- convert grouped E8M0 block scales to the blocked
 * ("128x4") layout that rg_mgemm_mxfp8 reads: the scale conversion for
 * grouped GEMMs of the torchao MoE-training PR (blocks of 128 rows x 4 scale
 * columns with a per-block swizzle, no block straddling two groups).
 *
 *   scales   device, uint8 [R, KS] row-major: E8M0 codes, KS scales per row
 *            (one per 32 elements of the row's contraction).
 *   offsets  device, int32 [G+1], same rules as rg_mgemm's (offsets[G] <= R).
 *            For an activation: the expert offsets.  For a weight stack
 *            [E, N, K/32]: G = E groups of N rows, offsets[g] = g*N.
 *   out      device, uint8, 16-byte aligned, out_bytes >= rg_mx_blocked_bytes.
 *            Each group is cut into 128-row blocks from its first row; the
 *            blocks of all groups are numbered in order; block b, chunk c
 *            (scale columns 4c..4c+3) is the 512 bytes at (b*ceil(KS/4)+c)*512,
 *            with row i of the block, column j of the chunk at byte
 *            16*(i%32) + 4*(i/32) + j.  Positions past a group's last row or
 *            past column KS-1 are 0x7F (scale 1.0).  Bytes past the last
 *            block are not written.
 *   G        1 .. RG_MAX_EXPERTS.  R 0 .. 2^31-1.  KS >= 1.
 * Invalid offsets contents set RG_DEV_BAD_OFFSETS and write nothing.
 */
int rg_mx_scales_blocked(const uint8_t* scales, const int32_t* offsets, int G, int64_t R, int KS,
                         uint8_t* out, int64_t out_bytes, cudaStream_t stream);

/*
 * rg_mgemm_mxfp8 -- M-grouped MXFP8 GEMM: FP8 E4M3 operands with one E8M0
 * power-of-two scale per 32 consecutive elements along the contraction
 * (the MXFP8 grouped GEMM of the torchao MoE-training PR; the block-scaled
 * FP8 GEMMs of the DeepGEMM issue discussion), forward (transpose_B == 0) or
 * input gradient (transpose_B != 0), over the Mgemm row grouping.
 *
 *   xq          device, uint8 [M, K]: E4M3 codes.
 *   sx_blocked  device: the scales sx [M, K/32] of xq (sx[r, k/32] scales
 *               xq[r, k]) in the blocked layout of rg_mx_scales_blocked with
 *               the same offsets; the buffer holds rg_mx_blocked_bytes(M,
 *               K/32, E) bytes.
 *   wq          device, uint8 E4M3 codes, [E, N, K] when transpose_B == 0,
 *               [E, K, N] when transpose_B != 0.
 *   sw_blocked  device: the scales sw [E, N, K/32] of B (sw[e, n, k/32]
 *               scales B element (k, n) of expert e, in both layouts) in the
 *               blocked layout with G = E groups of N rows; the buffer holds
 *               rg_mx_blocked_bytes(E*N, K/32, E) bytes.
 *   offsets     device, int32 [E+1], as for rg_mgemm.
 *   y           device, bf16 [M, N]: for row r of expert e
 *                 y[r, n] = sum_k xq[r,k] 2^(sx[r,k/32]-127) * B[k,n] 2^(sw[e,n,k/32]-127)
 *               accumulated in FP32 by the tensor cores, rounded to bf16
 *               (nearest even).  Rows >= offsets[E] are not written.
 *   N >= 16, multiple of 16.  K >= 32, multiple of 32.  E 1..RG_MAX_EXPERTS.
 *   xq, wq, the scale buffers and y 16-byte aligned.
 * An E4M3 NaN code or an E8M0 code 0xFF in a valid row or column makes the
 * outputs it reaches NaN.
 */
int rg_mgemm_mxfp8(const void* xq, const void* sx_blocked, const void* wq, const void* sw_blocked,
                   const int32_t* offsets, int E, int64_t M, int N, int K, int transpose_B, void* y,
                   cudaStream_t stream);

/*
 * rg_mx_blocked_k_bytes -- size in bytes that rg_mx_scales_blocked_k may
 * write for R rows of KS scales in G contraction groups:
 * ceil(R/128) * (KS/4 + G) * 512.  -1 on bad arguments.  Host-only.
 */
int64_t rg_mx_blocked_k_bytes(int64_t R, int KS, int G);

/*
 * rg_mx_scales_blocked_k -- blocked ("128x4") layout of E8M0 scales whose
 * groups run along the contraction: the conversion "for groups along K" of
 * the torchao MoE-training PR, which the K-grouped weight gradient reads.
 *
 *   scales   device, uint8 [R, KS]: R rows (an operand's columns, e.g. the N
 *            columns of the output gradient), KS scales along the contraction
 *            (one per 32 rows of the expert-grouped operand).
 *   offsets  device, int32 [G+1]: contraction indices with a leading zero,
 *            non-decreasing, all multiples of 32, offsets[G] <= 32*KS (the
 *            expert row offsets of rg_kgemm_mxfp8).  Group g owns scale
 *            columns offsets[g]/32 .. offsets[g+1]/32 - 1.
 *   out      device, uint8, 16-byte aligned, out_bytes >= rg_mx_blocked_k_bytes.
 *            Each group's scale columns are cut into chunks of 4 from its
 *            first column; the chunks of all groups are numbered in order
 *            (NQ in total); row block rb (rows 128rb ..), chunk q is the 512
 *            bytes at (rb*NQ + q)*512 with row i, column j of the chunk at
 *            byte 16*(i%32) + 4*(i/32) + j.  Positions past row R-1 or past
 *            the group's last column are 0x7F.  Later bytes are not written.
 *   G 1 .. RG_MAX_EXPERTS, R >= 1, KS >= 1.
 * Invalid offsets contents (including a multiple-of-32 violation) set
 * RG_DEV_BAD_OFFSETS and write nothing.
 */
int rg_mx_scales_blocked_k(const uint8_t* scales, const int32_t* offsets, int G, int64_t R, int KS,
                           uint8_t* out, int64_t out_bytes, cudaStream_t stream);

/*
 * rg_kgemm_mxfp8 -- K-grouped MXFP8 weight gradient with FP32 output (the
 * wgrad of MXFP8 MoE training in the torchao PR; the DeepGEMM issue thread
 * asks for FP8 wgrad with per-expert row counts that are not multiples of
 * 128 -- here they need only be multiples of the 32-row scale block).
 *
 *   gq          device, uint8 [M, N]: E4M3 codes of the output gradient.
 *   sg_blocked  device: its scales sg [N, M/32] (sg[n, r/32] scales gq[r, n])
 *               in the layout of rg_mx_scales_blocked_k with these offsets.
 *   xq          device, uint8 [M, K]: E4M3 codes of the layer input.
 *   sx_blocked  device: its scales sx [K, M/32], same layout.
 *   offsets     device, int32 [E+1]: expert row offsets, all multiples of 32.
 *   dW          device, fp32 [E, N, K]:
 *                 dW[e,n,k] (+)= sum over rows r of expert e of
 *                   gq[r,n] 2^(sg[n,r/32]-127) * xq[r,k] 2^(sx[k,r/32]-127)
 *               overwritten (accumulate == 0; an expert without rows gets 0)
 *               or added to (accumulate != 0; experts without rows unchanged).
 *               The rows of an expert are summed in FP32 by the tensor cores in
 *               chunks of at most 4096 rows, added in FP32 in row order.
 *   M multiple of 32; N, K >= 16 and multiples of 16; E 1..RG_MAX_EXPERTS.
 *   Pointers 16-byte aligned.  M == 0 is valid (zeroes dW unless accumulating).
 */
int rg_kgemm_mxfp8(const void* gq, const void* sg_blocked, const void* xq, const void* sx_blocked,
                   const int32_t* offsets, int E, int64_t M, int N, int K, float* dW, int accumulate,
                   cudaStream_t stream);

/*
 * rg_mgemm_swiglu -- M-grouped forward gate-up GEMM with the SwiGLU
 * activation applied in the epilogue (the fused activation named in the
 * DeepGEMM issue discussion of wgrad utilities, "fused with SwiGLU"; the
 * standard SwiGLU is used: h = SiLU(gate) * up, SiLU(z) = z / (1 + e^-z)).
 *
 *   x        device, bf16 [M, K].
 *   w13      device, bf16 [E, 2F, K]: rows 0..F-1 of w13[e] are the gate
 *            projection, rows F..2F-1 the up projection.
 *   offsets  device, int32 [E+1], as for rg_mgemm.
 *   y13      device, bf16 [M, 2F], or NULL.  If given it receives the gate-up
 *            output x . w13[e]^T rounded to bf16 (what rg_mgemm would write),
 *            e.g. for the backward pass.
 *   h        device, bf16 [M, F]: h[r, f] = SiLU(g) * u with g, u the fp32
 *            accumulators of gate column f and up column F+f, rounded to bf16
 *            once.  Rows >= offsets[E] are not written.
 *   F        >= 8, multiple of 8.  Other rules as for rg_mgemm.
 * Returns RG_ERR_UNSUPPORTED in builds without CTA pairs.
 */
int rg_mgemm_swiglu(const void* x, const void* w13, const int32_t* offsets, int E, int64_t M,
                    int F, int K, void* y13, void* h, cudaStream_t stream);

/*
 * rg_mgemm_swiglu_dgrad -- input gradient of the down projection followed by
 * the SwiGLU backward, in one M-grouped GEMM (the activation's backward fused
 * with the GEMM, per the same DeepGEMM issue discussion).
 *
 *   dy       device, bf16 [M, K]: gradient of the down projection's output.
 *   w2       device, bf16 [E, K, F]: the down projection's weight in its
 *            forward layout (rg_mgemm with w2 computes y = h . w2[e]^T).
 *   offsets  device, int32 [E+1], as for rg_mgemm.
 *   y13      device, bf16 [M, 2F]: the gate-up output saved by the forward
 *            pass (rg_mgemm_swiglu's y13).  Must not overlap dy13.
 *   dy13     device, bf16 [M, 2F]: with dh = dy . w2[e] kept in fp32, g, u the
 *            gate and up values of y13 and s = 1 / (1 + e^-g):
 *              dy13[r, f]     = dh[r, f] * u * s * (1 + g * (1 - s))
 *              dy13[r, F + f] = dh[r, f] * g * s
 *            rounded to bf16 once.  Rows >= offsets[E] are not written.
 *   F        >= 8, multiple of 8; K >= 8, multiple of 8.
 */
int rg_mgemm_swiglu_dgrad(const void* dy, const void* w2, const int32_t* offsets, int E, int64_t M,
                          int F, int K, const void* y13, void* dy13, cudaStream_t stream);

/*
 * rg_kgemm -- K-grouped weight gradient with FP32 output.  RapidGEMM README,
 * "Kernels", Kgemm.
 *
 *   grad     device, bf16 [M, N].
 *   X        device, bf16 [M, K].
 *   offsets  device, int32 [E+1], same rules as rg_mgemm (the README's
 *            "cumulative expert row ends" are offsets[1..E]).
 *   dW       device, fp32 [E, N, K], overwritten:
 *            dW[e, n, k] = sum over rows r of expert e of grad[r, n] * X[r, k],
 *            accumulated in FP32 by the tensor cores over chunks of at most
 *            4032 rows, whose partial sums are added in FP32 in row order
 *            (deterministic); an expert with no rows gets dW[e] = 0.
 *            Rows >= offsets[E] are ignored, and no row outside an
 *            expert's range is read for its dW[e]: Inf or NaN in one
 *            expert's rows reaches that expert's dW only.
 *   E 1 .. RG_KGEMM_MAX_EXPERTS; M, N, K, alignment and stream as for
 *   rg_mgemm (dW 16-byte aligned).  M == 0 is valid and zeroes dW.
 */
int rg_kgemm(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M,
             int N, int K, float* dW, cudaStream_t stream);

/*
 * rg_kgemm_acc -- as rg_kgemm, but accumulates into dW instead of
 * overwriting it:  dW[e, n, k] += sum over rows r of expert e of
 * grad[r, n] * X[r, k].  dW must hold the values to add to (for example an
 * FP32 main gradient); experts without rows leave dW[e] unchanged.  The sum of
 * each expert's rows is formed as in rg_kgemm and added to dW in FP32 (round
 * to nearest), chunk by chunk in row order, so results are deterministic.
 * TransformerEngine PR #2045 discussion (fuse_wgrad_accumulation: the weight
 * gradient GEMM accumulating into an FP32 main_grad whose dtype differs from
 * its BF16 inputs).
 */
int rg_kgemm_acc(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M,
                 int N, int K, float* dW, cudaStream_t stream);

/*
 * rg_kgemm_workspace_bytes -- device workspace that rg_kgemm_ws needs for E
 * experts and an [N, K] weight gradient: one 4-byte flag per expert, dW tile
 * (256 x 256) and CTA of a tile's CTA pair,
 * E * ceil(N/256) * ceil(K/256) * 2 * 4 bytes.  -1 on bad arguments.
 * Host-only; touches no device.
 */
int64_t rg_kgemm_workspace_bytes(int E, int N, int K);

/*
 * rg_kgemm_ws -- rg_kgemm (accumulate == 0) or rg_kgemm_acc (accumulate != 0)
 * with a schedule that reads each row of a long expert from DRAM once.  When
 * an expert has more dW tiles (256 x 256) than the GPU runs at once and is
 * longer than one accumulation chunk (4032 rows), rg_kgemm's tiles span
 * several rounds of the persistent grid and, once the expert's rows exceed
 * the L2 cache, read them again in each round.  Here all of its tiles work on
 * one chunk of its rows in the same round instead.  (Otherwise the schedule
 * is rg_kgemm's.)  The chunks of a tile then run on different CTAs,
 * and each chunk's fp32 reduce-add into dW waits for the previous chunk's
 * writes through a flag in `workspace`, so the chunks are still added in row
 * order: results are bit-identical to rg_kgemm's / rg_kgemm_acc's.
 * (RapidGEMM README, "Kernels", Kgemm; the schedule is this library's.)
 *
 *   grad, X, offsets, E, M, N, K, dW  as for rg_kgemm.
 *   workspace        device memory owned by the caller, 4-byte aligned, at
 *                    least rg_kgemm_workspace_bytes(E, N, K) bytes.  When
 *                    an expert has more dW tiles than the grid has CTA
 *                    pairs (half the SMs: 76 on a GB300), the call zeroes
 *                    those bytes on `stream` before the kernel; otherwise
 *                    the kernel cannot take the chunk-major schedule and
 *                    the workspace is not touched.  Two calls that may run
 *                    at the same time need two workspaces.
 *   workspace_bytes  its size.
 * Returns RG_ERR_INVALID_ARG for a null, misaligned or too small workspace,
 * otherwise as rg_kgemm.
 */
int rg_kgemm_ws(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M, int N, int K,
                float* dW, int accumulate, void* workspace, int64_t workspace_bytes, cudaStream_t stream);

/*
 * rg_kgemm_noalloc -- rg_kgemm_ws for callers that cannot allocate device
 * memory.  Nothing in the paper corresponds to it; it exists for this
 * library's users.  Some callers have no way to call cudaMalloc, or must not:
 * a framework or serving runtime that has handed all device memory to its own
 * pool (a cudaMalloc there fails or fragments the pool), a plugin running
 * inside another system that offers it no allocator, a runtime that forbids
 * allocation once it has started.  Such a caller cannot provide
 * rg_kgemm_ws's workspace, so this entry point takes the hand-over flags from
 * a fixed array in the library's device memory: RG_KGEMM_NOALLOC_MAX_FLAGS
 * 4-byte flags (256 KB), held on every GPU that loads the library until the
 * process exits.  It allocates nothing, on the device or the host.
 *
 *   grad, X, offsets, E, M, N, K, dW, accumulate, stream  as for rg_kgemm_ws.
 *
 * Results are those of rg_kgemm_ws (and so of rg_kgemm / rg_kgemm_acc).
 * The call zeroes the flags the problem uses on `stream` (where the kernel
 * may use them, as for rg_kgemm_ws's workspace), then launches the kernel.  Every call on a device shares that one array: two calls whose
 * work overlaps on the GPU (other streams, or graphs replayed concurrently)
 * race on it and may give wrong results or report RG_DEV_TIMEOUT; calls
 * ordered on one stream are safe.  The first call on a device looks up the
 * array's device address (that device must be current, as for every entry
 * point); make that first call before capturing stream work, as with every
 * other first call on a device.
 * Returns RG_ERR_SCRATCH if the problem needs more flags than the array
 * holds, that is if rg_kgemm_workspace_bytes(E, N, K) exceeds
 * 4 * RG_KGEMM_NOALLOC_MAX_FLAGS (for example E = 128, N = 2560, K = 3072
 * needs 30720 flags); otherwise as rg_kgemm_ws.
 */
int rg_kgemm_noalloc(const void* grad, const void* X, const int32_t* offsets, int E, int64_t M, int N, int K,
                     float* dW, int accumulate, cudaStream_t stream);

/*
 * rg_get_device_status -- after the work already queued on `stream`, read
 * and clear, in one atomic step, the RG_DEV_* bits that kernels of this
 * library set on the current device since the previous call; wait for the
 * read (synchronises `stream`) and return the bits (>= 0), or RG_ERR_CUDA /
 * RG_ERR_UNSUPPORTED (< 0).  The status is per device, not per stream: it
 * holds the bits of kernels on every stream of the device that finished
 * before the read, and a bit set concurrently by a kernel on another stream
 * is kept for the next call.  Not for use inside CUDA-graph capture.
 */
int rg_get_device_status(cudaStream_t stream);

/*
 * rg_set_wait_timeout_ns -- bound, in nanoseconds, on any single pipeline
 * wait inside the kernels (default 2e9, at least 1e6).  A wait that runs out
 * sets RG_DEV_TIMEOUT and every role of the kernel stops; issued MMAs and
 * copies are then waited for (those waits have their own fixed bound,
 * independent of this one), tensor memory is freed and the kernel returns.
 * Takes effect for launches made after the call.  Returns RG_ERR_INVALID_ARG
 * for a bound below 1e6 (1 ms).
 */
int rg_set_wait_timeout_ns(uint64_t ns);

/*
 * rg_selftest_wait_timeout -- enqueue one CTA whose warps wait on pipeline
 * barriers which nothing ever signals, one through each form of bounded wait
 * the kernels use (suspending, cluster-scope polling, the epilogues' sleeping
 * poll), each bounded by `ns` nanoseconds, and report through *status (host
 * pointer) the status bits the CTA set: RG_DEV_TIMEOUT when every form gave
 * up by itself, 0 when any of them returned as if its barrier had completed.
 * The self-test reports through a status word of its own, so bits pending
 * for rg_get_device_status are left as they are.  Synchronises `stream`.
 * Exercises the timeout path without a fault or a hang.
 */
int rg_selftest_wait_timeout(uint64_t ns, cudaStream_t stream, uint32_t* status);

/*
 * rg_shutdown -- forget the per-device set-up of every device (the kernels'
 * shared-memory attributes, grid sizes and the device addresses of the
 * status words), so that the next call on a device sets it up again.  The
 * library holds no memory, stream or other resource to release (its status
 * words are module variables of each device context), so this is needed
 * only after a device's context was destroyed (cudaDeviceReset) and before
 * the library is used on it again.  Must not run concurrently with other
 * calls into the library.  Returns RG_OK.
 */
int rg_shutdown(void);

/* CUDA error code (cudaError_t as int) behind the last RG_ERR_CUDA of the
 * calling thread, 0 if none. */
int rg_last_cuda_error(void);

/* 1 if the current device can run the kernels (compute capability 10.3), else 0. */
int rg_device_supported(void);

/* Library version string, static storage. */
const char* rg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RG_H_ */
