/*
 * mx.h -- C ABI of the GB300 (sm_103a) MXFP4 linear-layer library.
 *
 * What the library computes (cited by page title and section):
 *   [36kr] "Neue Studie von AMD durchbricht die bestehende Erkenntnis: Die
 *          Instabilitaet von FP4-Training liegt nicht an unzureichender
 *          Zufaelligkeit" (eu.36kr.com); [htx] its Indonesian rendering
 *          (htx.com); [show] "AMD颠覆认知：FP4不稳定性的真正原因" (showapi.com).
 *   - MXFP4 encoding: blocks of 32 consecutive elements along the contraction
 *     dimension share one E8M0 exponent, the block's largest exponent; each
 *     element is rounded to the nearest FP4 (E2M1: 1 sign, 2 exponent, 1
 *     mantissa bit) value ([36kr] "Was ist MXFP4?", [htx] "Apa itu MXFP4",
 *     [show] 2.2).  Reading of the lost reconstruction formula:
 *     x_hat = 2^s * Q(x / 2^s), s = floor(log2 amax) - 2 (OCP MX, [36kr] "Fazit").
 *   - The three GEMMs of a linear layer, Fprop Y = X W^T, Dgrad dX = dY W,
 *     Wgrad dW = dY^T X, computed from MXFP4 operands on the FP4 tensor cores
 *     with fp32 accumulation ([36kr] "Fehlerdiagnoseexperiment").
 *   - Rotation before quantisation: deterministic block Hadamard (the
 *     stabiliser; "H16" in [36kr] "Ende-zu-Ende-Effizienz" figure caption),
 *     Hadamard with a random sign flip, and stochastic rounding (the two
 *     randomised ablations of [36kr] "Fehlerdiagnoseexperiment").
 *
 * Conventions for every entry point:
 *   - Pointers named d_* are DEVICE pointers; h_* are HOST pointers.  The
 *     caller owns every buffer.  Nothing on the compute path allocates memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All compute entry points are asynchronous on `stream`.
 *   - Argument errors are detected on the host BEFORE anything is launched
 *     and returned as mx_status; nothing is written in that case.
 *   - A device-side wait that exceeds its time limit (a stalled pipeline)
 *     records MX_ERR_TIMEOUT in a per-device status word; the kernel then
 *     returns without faulting.  mx_check_status() reports and clears it.
 *   - bf16 inputs are raw IEEE bfloat16 bit patterns (uint16), row-major.
 *   - Alignment: every device pointer must be 16-byte aligned.  The
 *     contiguous (last) dimension of a bf16 input must be a multiple of 8
 *     elements so that each row starts on a 16-byte boundary (TMA rule).
 */
#ifndef MX_H
#define MX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MX_OK = 0,
    MX_ERR_INVALID_ARG = 1, /* null pointer, bad enum, unsupported rot_block */
    MX_ERR_SHAPE = 2,       /* negative size or contraction length not a multiple of 32
                               (or of rot_block when rotating) */
    MX_ERR_ALIGN = 3,       /* pointer or row pitch not 16-byte aligned */
    MX_ERR_WORKSPACE = 4,   /* workspace smaller than mx_linear_workspace_bytes() */
    MX_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed */
    MX_ERR_TIMEOUT = 6,     /* a device-side bounded wait expired (see mx_check_status) */
    MX_ERR_UNSUPPORTED = 7, /* not an sm_103 device, or arguments the call does not cover */
    MX_ERR_BOUNDS = 8       /* bounds-checked build only (MX_CHECKED=1): a kernel store fell
                               outside its buffer and was skipped (see mx_check_status) */
} mx_status;

typedef enum {
    MX_ROT_NONE = 0,          /* no rotation */
    MX_ROT_HADAMARD_DET = 1,  /* deterministic block Hadamard along the contraction dim */
    MX_ROT_HADAMARD_RAND = 2  /* random sign flip d_t, then block Hadamard */
} mx_rot;

typedef enum {
    MX_ROUND_RNE = 0,  /* round to nearest, ties to the even code */
    MX_ROUND_SR = 1    /* stochastic rounding (zero-mean error) */
} mx_round;

typedef enum {
    MX_CONTRACT_ROWS = 0, /* src[rows, cols]: blocks run down each column (the
                             contraction dim is `rows`); output is transposed to
                             codes[cols][rows/2] so the contraction dim is contiguous */
    MX_CONTRACT_COLS = 1  /* blocks run along each row; codes[rows][cols/2] */
} mx_contract;

typedef enum { MX_OP_FPROP = 0, MX_OP_DGRAD = 1, MX_OP_WGRAD = 2 } mx_op;

/* ------------------------------------------------------------------------ */
/* Encoded operand layout                                                    */
/* ------------------------------------------------------------------------ */
/*
 * An encoded operand has `mn` lines (rows of the GEMM operand) and contraction
 * length `k` (a multiple of 32).
 *
 * Codes: uint8 [mn][k/2], row-major; element 2i of a line in bits [3:0] of
 * byte i, element 2i+1 in bits [7:4].  E2M1 code: bit 3 sign, bits [2:1]
 * exponent (bias 1), bit 0 mantissa; magnitudes 0,.5,1,1.5,2,3,4,6.
 *
 * Scales: one E8M0 byte (2^(byte-127); 0xFF = NaN) per 32-element block,
 * tiled for the tensor cores' scale-factor path.  Lines are padded to
 * MP = 128*ceil(mn/128) and blocks to KB = 8*ceil(k/256).  The byte of line
 * r, block b lives at
 *     ((r/128) * (KB/4) + b/4) * 512 + (r%32)*16 + ((r%128)/32)*4 + (b%4).
 * i.e. 512-byte atoms of 128 lines x 4 blocks; atoms of one 128-line group
 * are contiguous along k.  Padding bytes are zero (mx_quantize writes them).
 */
size_t mx_codes_bytes(int64_t mn, int64_t k);
size_t mx_scales_bytes(int64_t mn, int64_t k);

/*
 * mx_scales_to_canonical -- copy a tiled scale array (the layout above, as
 * written by mx_quantize) into plain row-major bytes d_canon[lines][k/32]
 * (scale of line r, block b at r*(k/32) + b), dropping the padding.  For
 * tests and for handing scales to code that expects the canonical order.
 * k % 32 == 0; lines == 0 or k == 0: MX_OK, nothing launched.  Asynchronous
 * on `stream`; both buffers are device memory owned by the caller.
 */
mx_status mx_scales_to_canonical(const void *d_scales, int64_t lines, int64_t k, void *d_canon,
                                 void *stream);

/*
 * mx_quantize -- rotate and MXFP4-encode a bf16 matrix d_src[rows][cols].
 *   contract   MX_CONTRACT_ROWS: lines = columns, k = rows (needs cols % 8 == 0)
 *              MX_CONTRACT_COLS: lines = rows,    k = cols
 *   rot        mx_rot; rot_block in {16, 32, 64, 128, 256} must divide k
 *              (ignored for MX_ROT_NONE).  The Hadamard is Sylvester-ordered,
 *              normalised by 1/sqrt(rot_block), evaluated in fp32 as butterfly
 *              stages of stride 1, 2, ..., rot_block/2 then one multiply.
 *   rnd        mx_round.  SR draws come from the random stream (seed, 1):
 *              Philox4x32-10 with key (seed low 32 bits, seed high 32 bits)
 *              and counter (n low, n high, tag low, tag high) for block n and
 *              tag 1.  Element e = line*k + position takes the top 24 bits u of
 *              word e%4 of block e/4 and rounds away from the lower grid
 *              neighbour iff u < frac * 2^24.
 *   seed       key of the random sign (stream (seed, 0): bit t%32 of word
 *              (t%128)/32 of block t/128, t = position along k) and of SR.
 *   d_codes    mx_codes_bytes(lines, k) bytes; d_scales mx_scales_bytes(lines, k).
 * rows == 0 or cols == 0: returns MX_OK and launches nothing.
 */
mx_status mx_quantize(const void *d_src, int64_t rows, int64_t cols, int contract, int rot,
                      int rot_block, int rnd, uint64_t seed, void *d_codes, void *d_scales,
                      void *stream);

/*
 * mx_quantize_pair -- encode the two operands of a Wgrad in ONE launch: both
 * d_src0[rows0][cols0] and d_src1[rows1][cols1] are encoded down their rows
 * (MX_CONTRACT_ROWS: contraction length rows0 == rows1) with the same rotation,
 * rounding and seed; SR draws use stream (seed, 1) for operand 0 and (seed, 2)
 * for operand 1 (as mx_linear_wgrad does).  Outputs, layouts and argument rules
 * are those of mx_quantize for each operand.  One launch instead of two lets
 * the two HBM-bound encodes share one pipeline ramp-up and tail.
 */
mx_status mx_quantize_pair(const void *d_src0, int64_t rows0, int64_t cols0, const void *d_src1,
                           int64_t rows1, int64_t cols1, int rot, int rot_block, int rnd,
                           uint64_t seed, void *d_codes0, void *d_scales0, void *d_codes1,
                           void *d_scales1, void *stream);

/*
 * mx_quantize_dual -- one read of the output gradient d_src[T][N] (bf16,
 * row-major) writes both encodings a linear layer's backward pass needs
 * ([36kr] "Fehlerdiagnoseexperiment": dY feeds both Dgrad dX = dY W,
 * contracting N, and Wgrad dW = dY^T X, contracting T):
 *   d_codes_t / d_scales_t  the Wgrad operand: as mx_quantize(d_src, T, N,
 *                           MX_CONTRACT_ROWS, rot, rot_block, rnd, seed)
 *                           (N lines, contraction T, rotated along T);
 *   d_codes_n / d_scales_n  the Dgrad operand: as mx_quantize(d_src, T, N,
 *                           MX_CONTRACT_COLS, MX_ROT_NONE, 32, rnd, seed)
 *                           (T lines, contraction N, no rotation).
 * Both encodings are bit-identical to the two separate calls; SR draws use
 * stream (seed, 1) for both (dY is operand A of both GEMMs), each with its own
 * line*k + position counter.  Argument rules are the union of the two calls
 * (T % 32, T % rot_block, N % 32, N % 8).  T == 0 or N == 0: MX_OK, nothing
 * launched.
 */
mx_status mx_quantize_dual(const void *d_src, int64_t T, int64_t N, int rot, int rot_block,
                           int rnd, uint64_t seed, void *d_codes_t, void *d_scales_t,
                           void *d_codes_n, void *d_scales_n, void *stream);

/*
 * mx_gemm -- C[M][N] (fp32, row-major, overwritten) = A . B^T, where A is an
 * encoded operand with M lines and B one with N lines, both of contraction
 * length K (K % 32 == 0).  Block-scaled FP4 tensor-core contraction with fp32
 * accumulation.  Needs N % 4 == 0 (16-byte output rows).  M, N or K == 0: C is
 * zero-filled (K == 0) or untouched (M or N == 0) and MX_OK is returned.
 */
mx_status mx_gemm(const void *d_Aq, const void *d_As, const void *d_Bq, const void *d_Bs,
                  float *d_C, int64_t M, int64_t N, int64_t K, void *stream);

/* ------------------------------------------------------------------------ */
/* Linear-layer GEMMs ([36kr] "Fehlerdiagnoseexperiment")                     */
/* ------------------------------------------------------------------------ */
/*
 * Workspace (device, caller-owned) for one call of the given op: the two
 * encoded operands, each 256-byte aligned.
 *   FPROP: X[T][K], W[N][K] -> Y[T][N]       contraction K
 *   DGRAD: dY[T][N], W[N][K] -> dX[T][K]     contraction N
 *   WGRAD: dY[T][N], X[T][K] -> dW[N][K]     contraction T
 */
size_t mx_linear_workspace_bytes(int op, int64_t T, int64_t N, int64_t K);

/*
 * mx_linear_wgrad -- dW[N][K] = dY^T X.  Both operands are rotated along T
 * with the same rotation (same sign vector in MX_ROT_HADAMARD_RAND) and
 * encoded along T; operand dY uses SR stream (seed, 1), X uses (seed, 2).
 * T % 32 == 0 (and % rot_block); N, K % 8 == 0.
 */
mx_status mx_linear_wgrad(const void *d_dY, const void *d_X, float *d_dW, int64_t T,
                          int64_t N, int64_t K, int rot, int rot_block, int rnd, uint64_t seed,
                          void *d_ws, size_t ws_bytes, void *stream);

/*
 * mx_linear_wgrad_fused -- mx_linear_wgrad as ONE launch: encoder warps in
 * the GEMM's own CTAs encode dY and X into the workspace chunk by chunk
 * (in the order the GEMM first needs them) while the tensor cores consume
 * what is ready; per (256-line panel, 512-token chunk) counters in the
 * workspace, zeroed by a small memset before the launch, tell the GEMM's
 * producers when a stage's operands are stored.  Same arguments, workspace
 * size and results (the same bits) as mx_linear_wgrad.  Covers
 * round-to-nearest with no rotation or the deterministic Hadamard of 16 or
 * 32, T a multiple of 512 and N, K multiples of 256; other arguments get
 * MX_ERR_UNSUPPORTED (nothing launched).  On GB300 it is SLOWER than
 * mx_linear_wgrad's two launches (the encoder warps and the GEMM compete
 * for the same memory path, and shared memory is full with GEMM stages), so
 * mx_linear_wgrad does not use it.  No counterpart in the pages (the fusion
 * of the encode into the GEMM is a scheduling choice).
 * mx_linear_wgrad_fused_supported() returns 1 for arguments it covers.
 */
mx_status mx_linear_wgrad_fused(const void *d_dY, const void *d_X, float *d_dW, int64_t T,
                                int64_t N, int64_t K, int rot, int rot_block, int rnd,
                                uint64_t seed, void *d_ws, size_t ws_bytes, void *stream);
int mx_linear_wgrad_fused_supported(int64_t T, int64_t N, int64_t K, int rot, int rot_block,
                                    int rnd);

/*
 * MXFP8 comparator -- the FP8 baseline the pages compare MXFP4 against
 * ("Neue Studie von AMD ...", eu.36kr.com, section "Ende-zu-Ende-Effizienz":
 * MXFP4 training against an FP8 baseline; E4M3 is the FP8 layout named in
 * "AMD颠覆认知", showapi.com, section 2.2), run on the same shapes and the
 * same kernels with 8-bit elements.  Read here as OCP MXFP8: blocks of 32
 * along the contraction dimension share one E8M0 exponent,
 * floor(log2 amax) - 8 (E4M3's largest exponent), biased by 127 and clamped
 * to [0, 254] (0xFF: a block holding Inf/NaN, whose codes are zero); each
 * element becomes the nearest E4M3 value of x * 2^-exponent (ties to even,
 * magnitudes beyond 448 saturate to 448, sign kept).  No rotation and no
 * stochastic rounding (the FP8 baseline uses neither).
 *
 * Layouts: codes are one byte per element, row-major [lines][k]
 * (mx_mxfp8_codes_bytes(lines, k) = lines * k); scales use the same tiled
 * layout and size as MXFP4 (mx_scales_bytes).
 *
 * mx_quantize_mxfp8: contraction down the rows of src[rows][cols] (the
 *   Wgrad operands): codes [cols][rows].  rows % 32 == 0, cols % 8 == 0,
 *   16-byte aligned pointers.
 * mx_gemm_mxfp8: C[M][N] = A . B^T (fp32) over MXFP8 operands, contraction
 *   K (K % 32 == 0, N % 4 == 0); the arguments of mx_gemm otherwise.
 * mx_linear_wgrad_mxfp8: dW[N][K] = dY^T X with both operands MXFP8-encoded
 *   along T (one encode launch, one GEMM launch), workspace of
 *   mx_linear_wgrad_mxfp8_workspace_bytes(T, N, K) bytes, 256-byte aligned.
 *   T % 32 == 0; N, K % 8 == 0.
 * Status codes and asynchrony as for the MXFP4 calls.
 */
size_t mx_mxfp8_codes_bytes(int64_t mn, int64_t k);
mx_status mx_quantize_mxfp8(const void *d_src, int64_t rows, int64_t cols, void *d_codes,
                            void *d_scales, void *stream);
mx_status mx_gemm_mxfp8(const void *d_Aq, const void *d_As, const void *d_Bq, const void *d_Bs,
                        float *d_C, int64_t M, int64_t N, int64_t K, void *stream);
size_t mx_linear_wgrad_mxfp8_workspace_bytes(int64_t T, int64_t N, int64_t K);
mx_status mx_linear_wgrad_mxfp8(const void *d_dY, const void *d_X, float *d_dW, int64_t T,
                                int64_t N, int64_t K, void *d_ws, size_t ws_bytes, void *stream);

/*
 * NVFP4 variant -- NVFP4 is named as prior work in "Neue Studie von AMD ..."
 * (eu.36kr.com), introduction; its definition here is NVIDIA's published
 * format: E2M1 elements in blocks of 16 along the contraction dimension, one
 * UE4M3 scale per block and one fp32 encode scale per tensor.
 *   tensor:  amax = largest finite |x| of the (rotated) operand;
 *            s_enc = 2688 / amax (448 * 6, the largest block value), FLT_MAX
 *            if that overflows, 1 if amax == 0;
 *   block:   sf = E4M3 nearest-even of fl(fl(block_amax / 6) * s_enc),
 *            saturating at 448 (0x7F: a block holding Inf/NaN; its codes 0);
 *   element: E2M1 nearest-even of fl(x * min(fl(s_enc / sf), FLT_MAX))
 *            (sf == 0: code 0); it stands for e2m1 * sf / s_enc.
 * The same rotations as MXFP4 with Hadamard blocks of 16 or 32 (others:
 * MX_ERR_UNSUPPORTED); round to nearest only.
 *
 * Layouts: codes as MXFP4 ([lines][k/2], mx_codes_bytes); scales in their
 * own tiled layout of mx_nvfp4_scales_bytes(lines, k) bytes: byte (line r,
 * block b of 16) at ((r/128)*(KB/4) + b/4)*512 + (r%32)*16 + ((r%128)/32)*4
 * + b%4 with KB = 16*ceil(k/256) blocks per line (padding blocks 0).
 *
 * mx_quantize_nvfp4: contraction down the rows of src[rows][cols]; two
 *   launches (the tensor amax, then the encode); *d_amax (device float,
 *   8-byte aligned) receives the tensor amax, which mx_gemm_nvfp4 takes.
 * mx_gemm_nvfp4: C[M][N] = (sum over K of decoded a * b), i.e. the
 *   block-scaled product divided by s_enc(amax_a) * s_enc(amax_b) in the
 *   epilogue; K % 32 == 0, N % 4 == 0.
 * mx_linear_wgrad_nvfp4: dW[N][K] = dY^T X with both operands NVFP4-encoded
 *   along T (three launches and a memset of the two amax words), workspace of
 *   mx_linear_wgrad_nvfp4_workspace_bytes(T, N, K) bytes, 256-byte aligned.
 */
size_t mx_nvfp4_scales_bytes(int64_t mn, int64_t k);
mx_status mx_quantize_nvfp4(const void *d_src, int64_t rows, int64_t cols, int rot, int rot_block,
                            uint64_t seed, void *d_codes, void *d_scales, float *d_amax,
                            void *stream);
mx_status mx_gemm_nvfp4(const void *d_Aq, const void *d_As, const float *d_amax_a,
                        const void *d_Bq, const void *d_Bs, const float *d_amax_b, float *d_C,
                        int64_t M, int64_t N, int64_t K, void *stream);
size_t mx_linear_wgrad_nvfp4_workspace_bytes(int64_t T, int64_t N, int64_t K);
mx_status mx_linear_wgrad_nvfp4(const void *d_dY, const void *d_X, float *d_dW, int64_t T,
                                int64_t N, int64_t K, int rot, int rot_block, uint64_t seed,
                                void *d_ws, size_t ws_bytes, void *stream);

/* mx_linear_fprop -- Y[T][N] = X W^T, contraction K (K % 32 == 0, N % 4 == 0). */
mx_status mx_linear_fprop(const void *d_X, const void *d_W, float *d_Y, int64_t T, int64_t N,
                          int64_t K, int rot, int rot_block, int rnd, uint64_t seed,
                          void *d_ws, size_t ws_bytes, void *stream);

/* mx_linear_dgrad -- dX[T][K] = dY W, contraction N (N % 32 == 0, K % 8 == 0). */
mx_status mx_linear_dgrad(const void *d_dY, const void *d_W, float *d_dX, int64_t T, int64_t N,
                          int64_t K, int rot, int rot_block, int rnd, uint64_t seed,
                          void *d_ws, size_t ws_bytes, void *stream);

/*
 * mx_linear_wgrad_noalloc -- mx_linear_wgrad without a caller workspace.
 * No counterpart in the paper: this is a deployment convenience.
 *
 * For callers that cannot allocate device memory themselves: plugins and
 * custom ops running inside a framework that owns all device memory through
 * its own pool (an allocation behind the pool's back breaks its accounting or
 * fails under a hard memory cap), bare C/Fortran hosts without a device
 * allocator, and hot loops that cannot afford the implicit device-wide
 * synchronisation of cudaMalloc/cudaFree.  The encoded operands go to a fixed
 * scratch area of MX_NOALLOC_SCRATCH_BYTES held by the library's module on
 * every GPU that loads it, until process exit.  The call itself allocates
 * nothing and calls no allocating routine.
 *
 * Limits and behaviour:
 *   - mx_linear_workspace_bytes(MX_OP_WGRAD, T, N, K) must not exceed
 *     MX_NOALLOC_SCRATCH_BYTES (64 MiB; e.g. T = 8192 with N = K = 4096 needs
 *     35.7 MB), else MX_ERR_WORKSPACE is returned and nothing is launched.
 *   - The first call on a device looks up the scratch area's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - Every call on a device shares the one scratch area and leaves its
 *     contents behind (they are fully rewritten by the next call).  Calls that
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on it and give undefined results; serialise them.
 *   - Arguments, layouts and the other status codes are those of
 *     mx_linear_wgrad.
 */
#define MX_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
mx_status mx_linear_wgrad_noalloc(const void *d_dY, const void *d_X, float *d_dW, int64_t T,
                                  int64_t N, int64_t K, int rot, int rot_block, int rnd,
                                  uint64_t seed, void *stream);

/* ------------------------------------------------------------------------ */
/* Status and diagnostics                                                    */
/* ------------------------------------------------------------------------ */
/* Synchronises `stream`, then returns and clears the current device's status
 * word: MX_ERR_TIMEOUT if a bounded device wait expired since the last call,
 * MX_ERR_CUDA if the stream reported an error, else MX_OK. */
mx_status mx_check_status(void *stream);

/* Launches one CTA that waits on a barrier nothing will ever complete; its
 * bounded wait gives up after `limit_us` microseconds and records
 * MX_ERR_TIMEOUT.  Exists to test the timeout path without hanging a GPU. */
mx_status mx_debug_timeout_probe(int64_t limit_us, void *stream);

/*
 * mx_bench_mma -- tensor-core issue-rate microbenchmark (measurement only; no
 * counterpart in the pages, which report no kernel-level figure).  Every SM
 * (one CTA each, or one 2-CTA cluster per SM pair for cta_group = 2) issues
 * `iters` iterations of: `copies_per_iter` scale copies shared -> tensor
 * memory, then `mmas_per_iter` tcgen05.mma of M = 128*cta_group, N = n, on
 * operands resident in shared memory, with fp32 accumulation in tensor memory.
 *   kind        0 mxf4 (E2M1, UE8M0/32, K=64)   1 mxf4nvf4 2X (same scales)
 *               2 mxf4nvf4 4X (UE4M3/16)        3 f8f6f4 E4M3 (K=32)
 *               4 f16 with bf16 inputs (K=16)   5 mxf8f6f4 E4M3, UE8M0/32 (K=32)
 *   copy_shape  0 32x128b.warpx4, 1 128x256b, 2 128x128b
 *   depth       0: no handshake; 1..7: commit every iteration to an mbarrier
 *               and wait for the commit of iteration it - depth (a ring of
 *               `depth` stages in flight, as in a pipelined GEMM)
 *   flags       bit 0: the copies fill the NEXT iteration's scale columns;
 *               bit 1: with depth > 0, commit every iteration but never wait;
 *               bit 2: four more warps keep storing to unused tensor-memory
 *               columns (tcgen05.st) while the MMAs run
 *   d_ns        device int64[256]: per CTA, ns from the first to the last
 *               MMA's completion (0 for the second CTA of a pair; -1 if a
 *               bounded wait expired)
 *   h_ctas      host int: CTAs launched
 * MMA flops per CTA = 2 * 128 * n * K * mmas_per_iter * iters.
 */
mx_status mx_bench_mma(int kind, int cta_group, int n, int mmas_per_iter, int copies_per_iter,
                       int copy_shape, int depth, int flags, int64_t iters, int64_t *d_ns,
                       int *h_ctas, void *stream);

/* Human-readable name of a status code (static storage). */
const char *mx_status_string(int status);

/* Library ABI version (major*100 + minor). */
int mx_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MX_H */
