/*
 * lpfa — MXFP8 block-scaled FlashAttention (forward and backward) for
 * NVIDIA GB300 (sm_103a).  C ABI.
 *
 * Entry points: the MX quantizer (lpfa_mx_quantize, and lpfa_mx_quantize_fmt
 * for the other MX element formats), the attention forward and backward
 * (lpfa_fwd, lpfa_bwd, lpfa_bwd_noalloc) with their workspace queries and
 * lpfa_check, the jagged scale-row offsets (lpfa_varlen_sf_rows), the fused
 * producers of quantized operands (lpfa_rmsnorm_mx_quantize,
 * lpfa_mx_gemm_quantize), the block-scaled GEMM (lpfa_mx_gemm), the
 * tensor-pipe rate microbench (lpfa_mma_peak), the FP6 / FP4 / NVFP4 GEMMs and
 * quantizers, the jagged GEMM-Norm backward pieces, the forward's bounded-wait
 * self-test and the status / version / device queries.
 *
 * Sources of the operations (page title, section):
 *  [P1] "Low Precision Flash Attention 4: End-to-End Block-Scaled Attention
 *       for Blackwell" — paragraph 2 (tcgen05 block-scaled MMA; TMEM budget
 *       for scale factors; online square-block quantization of dS with a
 *       warp max-abs reduction; FP8 outputs with dual scale layouts; jagged
 *       inputs with FP8 data unpadded and 128-aligned scale rows), paragraph
 *       3 (forward softmax in FP32 with P converted to MXFP8 reusing the
 *       softmax max; backward Q, K, dO in square [32, 32] blocks; FP16 dQ
 *       with a static scale).
 *  [P2] "Low-Precision FlashAttention-4: End-to-End Block-Scaled Attention
 *       for NVIDIA Blackwell" — "Understanding OCP MXFP8 Microscaling on
 *       Blackwell" (32-element blocks sharing an E8M0 scale
 *       s = 2^(E8M0-127), E4M3 elements), "Key Algorithmic Innovations"
 *       (both GEMMs block-scaled, FP32 running max/sum with 1/sqrt(d_k)
 *       folded in), "PyTorch Integration & Implementation Example" (BSHD
 *       tensors; q, k, v, their scales, softmax_scale, causal).
 *  [P3] "FlashAttention-4 Adds Low-Precision Blackwell Support" — "Technical
 *       Deep Dive" (TMEM/tcgen05 data flow, selective rescaling), "Hardware
 *       Portability Gate" (datacenter Blackwell only).
 *
 * Conventions for every call
 *  - All pointers named *_dev (or documented as device) are CUDA device
 *    pointers owned by the caller; the library never allocates or frees
 *    memory and keeps no state between calls.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All device work is enqueued asynchronously on it.
 *  - Argument errors are detected on the host before any launch and return
 *    LPFA_ERR_INVALID_ARG / LPFA_ERR_UNSUPPORTED; launch failures return
 *    LPFA_ERR_CUDA.  Kernels never trap: a bounded wait that expires records
 *    an error word in the caller's workspace, which lpfa_check() turns into
 *    LPFA_ERR_TIMEOUT.
 *  - Token-major data layout: a tensor is [T, H, D] with rows (tokens)
 *    contiguous in H*D elements.  Dense BSHD [B, S, H, D] is the special case
 *    T = B*S with B sequences of S tokens (lpfa_seqs with cu_seqlens NULL).
 *  - Scale rows (see lpfa_seqs): scale tensors index tokens in a padded row
 *    space where every sequence starts at a multiple of 128 rows; FP8 data
 *    are never padded ([P1] paragraph 2, jagged module).
 */
#ifndef LPFA_H_
#define LPFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LPFA_VERSION 1

typedef enum lpfa_status {
  LPFA_OK = 0,
  LPFA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape or size  */
  LPFA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head_dim, GPU)   */
  LPFA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed           */
  LPFA_ERR_TIMEOUT = 4       /* a kernel's bounded wait expired (lpfa_check) */
} lpfa_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* lpfa_status_string(lpfa_status s);

/* LPFA_VERSION of the built library. */
int lpfa_version(void);

/* Returns LPFA_OK when the current device is datacenter Blackwell with
 * tensor memory (compute capability 10.x: sm_100/sm_103), else
 * LPFA_ERR_UNSUPPORTED ([P3] "Hardware Portability Gate"; consumer SM120
 * has no TMEM). */
lpfa_status lpfa_device_supported(void);

/* ------------------------------------------------------------------------
 * Sequences.  Dense: nseq sequences of `seqlen` tokens each, cu_seqlens and
 * cu_sf_rows NULL.  Jagged ([P1] paragraph 2): cu_seqlens (device int32,
 * nseq+1 prefix offsets into the packed tokens) and cu_sf_rows (device
 * int32, nseq+1) with cu_sf_rows[s] = sum_{t<s} ceil(L_t/128)*128, the first
 * padded scale row of sequence s (lpfa_varlen_sf_rows computes it);
 * `seqlen` is then the maximum sequence length.
 * total_tokens = T, total_sf_rows = Tp = cu_sf_rows[nseq] (dense:
 * nseq * ceil(seqlen/128) * 128).
 * ---------------------------------------------------------------------- */
typedef struct lpfa_seqs {
  int64_t nseq;
  int64_t seqlen;
  int64_t total_tokens;
  int64_t total_sf_rows;
  const int32_t* cu_seqlens;   /* device, nseq+1, or NULL (dense) */
  const int32_t* cu_sf_rows;   /* device, nseq+1, or NULL (dense) */
} lpfa_seqs;

/* Fill cu_sf_rows[0..nseq] (device int32) from cu_seqlens (device int32):
 * cu_sf_rows[s] = sum_{t<s} ceil((cu_seqlens[t+1]-cu_seqlens[t])/128)*128.
 * One small kernel on `stream`.  nseq in [1, 2^20]. */
lpfa_status lpfa_varlen_sf_rows(const int32_t* cu_seqlens, int64_t nseq,
                                int32_t* cu_sf_rows, void* stream);

/* ------------------------------------------------------------------------
 * MX quantizer ([P2] "Understanding OCP MXFP8 Microscaling on Blackwell";
 * [P1] paragraphs 2-3).
 *
 * x: bf16 [T, heads, head_dim] (device, 16-byte aligned), head_dim in
 * {64, 128}.  Every block of 32 elements (or 32x32) gets
 *   amax = max |x|, e = clamp(floor(log2 amax) - 8, -127, 127),
 *   scale code = e + 127 (E8M0; amax == 0 -> code 0; Inf/NaN -> 0xFF with
 *   payloads 0x7F),
 *   payload = E4M3(x * 2^-e), round to nearest even, saturating to +-448.
 *
 * Block shapes (lpfa_block):
 *  LPFA_BLK_1X32   32 consecutive head_dim channels of one token (forward
 *                  Q and K; backward V).
 *  LPFA_BLK_32X1   32 consecutive tokens of one channel, blocks starting at
 *                  each sequence start, the last one possibly short
 *                  (forward V: the PV product contracts over keys).
 *  LPFA_BLK_32X32  32 tokens x 32 channels, transpose-invariant (backward
 *                  Q, K, dO).
 *
 * Outputs (device, caller-allocated; any of the scale outputs may be NULL):
 *  out_e4m3    uint8 [T, heads, head_dim], same positions as x (unpadded).
 *  out_sf      compact E8M0 scales:
 *                1X32:  [T, heads, head_dim/32]
 *                32X1:  [Tp/32, heads, head_dim]
 *                32X32: [Tp/32, heads, head_dim/32]
 *              (token blocks indexed in the padded scale-row space).
 *  out_sf_mma  tensor-core scale layout for use with the contraction over
 *              head_dim (1X32, 32X32) or over tokens (32X1):
 *              [Tp/128, heads, 512] bytes; in each 512-byte tile operand row
 *              r (token, or channel for 32X1) and contraction block kb sit at
 *              byte (r%32)*16 + (r/32)*4 + kb.
 *  out_sf_mma_t (32X32 only) the same square scales arranged for use with
 *              the contraction over tokens (operand rows = channels):
 *              [Tp/128, heads, 512].  With out_sf_mma this is the pair of
 *              scale layouts of one quantized payload ([P1] paragraph 2).
 * Padding bytes of the scale outputs are written as 0.
 * ---------------------------------------------------------------------- */
typedef enum lpfa_block {
  LPFA_BLK_1X32 = 0,
  LPFA_BLK_32X1 = 1,
  LPFA_BLK_32X32 = 2
} lpfa_block;

lpfa_status lpfa_mx_quantize(const lpfa_seqs* seqs, const void* x,
                             int64_t heads, int64_t head_dim, lpfa_block blk,
                             void* out_e4m3, void* out_sf, void* out_sf_mma,
                             void* out_sf_mma_t, void* stream);

/* ------------------------------------------------------------------------
 * The same quantizer for the other OCP MX element formats ([P2] names
 * MXFP8, MXFP6 and MXFP4 as the block-scaled MMA formats): identical block
 * shapes, outputs and layouts, one element per payload byte in its low bits
 * (sign on top of the element's field).  The scale exponent subtracts the
 * format's emax instead of E4M3's 8:
 *   LPFA_ELEM_E4M3  emax 8,  max 448    (lpfa_mx_quantize)
 *   LPFA_ELEM_E5M2  emax 15, max 57344  (IEEE-like Inf/NaN)
 *   LPFA_ELEM_E3M2  emax 4,  max 28     (FP6, no Inf/NaN)
 *   LPFA_ELEM_E2M3  emax 2,  max 7.5    (FP6, no Inf/NaN)
 *   LPFA_ELEM_E2M1  emax 2,  max 6      (FP4, no Inf/NaN)
 * Elements round to nearest even and saturate to the largest finite
 * magnitude; a block holding Inf or NaN gets scale 0xFF and payload bytes
 * 0x7F (E4M3, E5M2) or the largest positive code (0x1F FP6, 0x07 FP4).
 * Errors: as lpfa_mx_quantize; fmt outside the enum -> INVALID_ARG.
 * ---------------------------------------------------------------------- */
typedef enum lpfa_elem {
  LPFA_ELEM_E4M3 = 0,
  LPFA_ELEM_E5M2 = 1,
  LPFA_ELEM_E3M2 = 2,
  LPFA_ELEM_E2M3 = 3,
  LPFA_ELEM_E2M1 = 4
} lpfa_elem;

lpfa_status lpfa_mx_quantize_fmt(const lpfa_seqs* seqs, const void* x,
                                 int64_t heads, int64_t head_dim,
                                 lpfa_block blk, lpfa_elem fmt, void* out,
                                 void* out_sf, void* out_sf_mma,
                                 void* out_sf_mma_t, void* stream);

/* ------------------------------------------------------------------------
 * Fused RMSNorm + MX quantization ([P1] paragraph 2: fused RMSNorm+Quantize
 * kernels producing FP8 output with dual scale factor layouts in one pass).
 *
 * x: bf16 [T, heads, head_dim] (device, 16-byte aligned), one token row of
 * N = heads * head_dim values per token; weight: bf16 [N] (device, 16-byte
 * aligned); eps > 0.  For every token
 *   y = x / sqrt(mean(x^2) + eps) * weight,
 * formed in fp32 by a fixed sequence of correctly rounded operations: ss =
 * the fp32 sum of the exact squares, 32 partial sums (partial l over the
 * 8-element chunks l, l + 32, ... of the row, element by element) combined
 * pairwise at distance 16, 8, 4, 2, 1; rstd = 1 / sqrt(ss / N + eps);
 * y = (x * rstd) * weight, each product rounded to fp32.  y is then quantized
 * exactly as lpfa_mx_quantize quantizes its input (same rule, same outputs
 * and layouts), with blk = LPFA_BLK_1X32 or LPFA_BLK_32X32 (the square blocks
 * give one payload with the two tensor-core scale arrangements out_sf_mma and
 * out_sf_mma_t); LPFA_BLK_32X1 returns LPFA_ERR_UNSUPPORTED.
 *
 * out_rstd: fp32 [T] (device) or NULL; receives rstd of every token.
 * HBM sees x once: a CTA reads its 32 token rows for the sums of squares and
 * again, from L2, for the payload.
 * Errors: null or misaligned pointers, eps <= 0 or non-finite, heads outside
 * [1, 4096] -> LPFA_ERR_INVALID_ARG; head_dim not 64/128 -> UNSUPPORTED.
 * ---------------------------------------------------------------------- */
lpfa_status lpfa_rmsnorm_mx_quantize(const lpfa_seqs* seqs, const void* x,
                                     const void* weight, int64_t heads,
                                     int64_t head_dim, float eps,
                                     lpfa_block blk, void* out_e4m3,
                                     void* out_sf, void* out_sf_mma,
                                     void* out_sf_mma_t, float* out_rstd,
                                     void* stream);

/* ------------------------------------------------------------------------
 * Block-scaled MXFP8 GEMM (measures the dense MX MMA rate in the same run as
 * the attention kernels; also the tcgen05 block-scale bring-up).
 *   D[M, N] (fp32, row-major, ldd = N) = A[M, K] * B[N, K]^T
 * A, B: e4m3, K contiguous (row-major [M, K] / [N, K]); sfa_mma, sfb_mma:
 * tensor-core scale layout of their 1x32 (along K) scales,
 * [M/128][K/128][512] and [N/128][K/128][512] bytes (tile (i, kt) holds rows
 * 128i.. and contraction blocks 4kt..4kt+3).  N a multiple of 256, K of 128;
 * M any positive value (rows past M read as zeros and are not stored; the A
 * scales then hold ceil(M/128) row tiles).  Persistent kernel on CTA pairs
 * (clusters of two; 256 x 256 output tiles, one CTA pair per two SMs).
 * ---------------------------------------------------------------------- */
lpfa_status lpfa_mx_gemm(const void* a8, const void* sfa_mma, const void* b8,
                         const void* sfb_mma, float* d, int64_t M, int64_t N,
                         int64_t K, void* stream);

/* ------------------------------------------------------------------------
 * The same GEMM on operands of other MX element formats ([P1] paragraph 2:
 * the block-scaled MMA takes MXFP8, MXFP6 and MXFP4 operands): the
 * kind::mxf8f6f4 MMA with the A and B element types a_fmt, b_fmt (any pair
 * of lpfa_elem), 1x32 UE8M0 scales along K in the layout of lpfa_mx_gemm.
 * a, b: [M, K] / [N, K] bytes in the tensor core's operand layout (see
 * lpfa_mx_pack_operand): for E4M3 and E5M2 one code per byte; for FP6 and
 * FP4 every 16 consecutive elements of a row take 16 bytes, their codes
 * packed at the front.
 * Constraints and errors as lpfa_mx_gemm; a format outside the enum ->
 * LPFA_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
lpfa_status lpfa_mx_gemm_fmt(const void* a, const void* sfa_mma, const void* b,
                             const void* sfb_mma, float* d, int64_t M, int64_t N,
                             int64_t K, lpfa_elem a_fmt, lpfa_elem b_fmt, void* stream);

/* Operand bytes for lpfa_mx_gemm_fmt from one-code-per-byte payloads (the
 * output of lpfa_mx_quantize_fmt).  codes, out: [rows, cols] bytes, cols a
 * multiple of 16, 16-byte aligned.  Each group of 16 consecutive codes of a
 * row becomes 16 bytes:
 *   E4M3, E5M2  unchanged (a copy unless codes == out);
 *   E3M2, E2M3  a little-endian 96-bit stream, code e at bits 6e..6e+5, in
 *               bytes 0..11; bytes 12..15 zero;
 *   E2M1        code e in bits 4(e%2).. of byte e/2 (bytes 0..7); bytes 8..15
 *               zero.
 * (The layout kind::mxf8f6f4 MMAs read for 6- and 4-bit operands.)
 * Errors: NULL / misaligned pointers, cols % 16 != 0, a format outside the
 * enum -> LPFA_ERR_INVALID_ARG. */
lpfa_status lpfa_mx_pack_operand(const void* codes, int64_t rows, int64_t cols,
                                 lpfa_elem fmt, void* out, void* stream);

/* ------------------------------------------------------------------------
 * FP4 operands at the dense FP4 MMA rate ([P1] paragraph 2: MXFP4 and NVFP4
 * among the block-scaled MMA formats): D[M, N] (fp32) = A[M, K] * B[N, K]^T
 * with kind::mxf4nvf4 MMAs (K = 64 per instruction).
 *  a, b: dense E2M1 [M, K/2] / [N, K/2] bytes, element 2i in the low nibble
 *        of byte i (lpfa_fp4_pack_dense, or lpfa_nvfp4_quantize's output).
 *  nvfp4 = 0 (MXFP4): 32-element UE8M0 blocks; sfa_mma / sfb_mma in the
 *        layout of lpfa_mx_gemm ([R/128][K/128][512], four blocks per row
 *        per tile), e.g. lpfa_mx_quantize_fmt(LPFA_ELEM_E2M1) out_sf_mma.
 *  nvfp4 = 1 (NVFP4): 16-element UE4M3 blocks; [R/128][K/64][512], row r and
 *        block kb of a tile at byte (r%32)*16 + (r/32)*4 + kb
 *        (lpfa_nvfp4_quantize out_sf_mma).
 * M, N multiples of 128 (N of 256), K a multiple of 256 (else
 * LPFA_ERR_UNSUPPORTED); other errors as lpfa_mx_gemm.
 * ---------------------------------------------------------------------- */
lpfa_status lpfa_mx_gemm_fp4(const void* a, const void* sfa_mma, const void* b,
                             const void* sfb_mma, float* d, int64_t M, int64_t N,
                             int64_t K, int nvfp4, void* stream);

/* One-code-per-byte E2M1 [rows, cols] (cols % 16 == 0, 16-byte aligned) ->
 * dense [rows, cols/2] bytes (8-byte aligned), code 2i in the low nibble of
 * byte i: the operand layout of lpfa_mx_gemm_fp4. */
lpfa_status lpfa_fp4_pack_dense(const void* codes, int64_t rows, int64_t cols,
                                void* out, void* stream);

/* NVFP4 quantization ([P1] paragraph 2 names the format; reading): x bf16
 * [rows, cols] row-major (16-byte aligned, cols % 16 == 0); every 16
 * consecutive elements of a row form a block with
 *   s = E4M3(amax / 6)   (fp32 division; round to nearest even, saturating)
 *   element = E2M1(x / s) (fp32 division; nearest even, saturating at 6),
 * an all-zero block (or one whose scale rounds to 0) gets scale code 0 and
 * zero elements; no per-tensor second-level scale.  Outputs: out dense E2M1
 * [rows, cols/2] (8-byte aligned); out_sf E4M3 codes [rows, cols/16] or
 * NULL; out_sf_mma [rows/128][cols/64][512] (rows % 128 == 0, cols % 64 ==
 * 0) in the layout lpfa_mx_gemm_fp4 reads, or NULL.  Inputs are finite. */
lpfa_status lpfa_nvfp4_quantize(const void* x, int64_t rows, int64_t cols, void* out,
                                void* out_sf, void* out_sf_mma, void* stream);

/* ------------------------------------------------------------------------
 * Grouped block-scaled GEMM: one or two independent MXFP8 GEMMs
 * D_i = A_i B_i^T (E4M3 operands, fp32 output) in one persistent launch, with
 * the arguments, layouts and errors of lpfa_mx_gemm for each problem.  The
 * problem with the longer contraction runs first on every CTA pair and the
 * other's tiles are split so that the pairs finish together (the two
 * backward GEMMs of the GEMM-Norm backward: dW, with a contraction over the
 * tokens, and dX).
 * ---------------------------------------------------------------------- */
typedef struct lpfa_gemm_problem {
  const void* a;          /* E4M3 [M, K] */
  const void* sfa_mma;    /* [ceil(M/128)][K/128][512] */
  const void* b;          /* E4M3 [N, K] */
  const void* sfb_mma;    /* [N/128][K/128][512] */
  float* d;               /* fp32 [M, N] */
  int64_t M, N, K;
} lpfa_gemm_problem;

lpfa_status lpfa_mx_gemm_grouped(const lpfa_gemm_problem* problems, int32_t count, void* stream);

/* ------------------------------------------------------------------------
 * Jagged GEMM-Norm backward ([P1] paragraph 4 reports it for throughput
 * only; [P1] paragraph 2: fused RMSNorm + Quantize with dual scale layouts).
 * Reading: over the T tokens of a jagged batch (rows of X [T, K], sequences
 * concatenated), Y = X W^T (W [N, K]), Z = Y r gamma with
 * r_t = rsqrt(mean_n Y_tn^2 + eps); from dZ [T, N]
 *   c_t = (1/N) sum_n gamma_n dZ_tn Y_tn,  dY = r (gamma dZ - Y r^2 c),
 *   dgamma_n = sum_t dZ_tn Y_tn r_t,  dX = dY W,  dW = dY^T X,
 * with dY, X, W quantized in square 32x32 blocks so that one payload serves
 * the GEMM over N (dX) and the GEMM over T (dW).  The two GEMMs are
 * lpfa_mx_gemm calls on the outputs below (dX: A = dY [T, N] with sf_mma,
 * B = W's transposed payload [K, N] with W's sf_mma_t; dW: A = dY's
 * transposed payload [N, Tp] with sf_mma_t, B = X's transposed payload
 * [K, Tp] with X's sf_mma_t).
 *
 * lpfa_mx_quantize_t: 32x32 MX quantization of x bf16 [rows, cols]
 * (row-major, 16-byte aligned; cols a multiple of 128) with the payload in
 * both orientations.  rows_p = rows rounded up to 128; rows past `rows` are
 * zeros.  Outputs (device, caller-allocated, 16-byte aligned):
 *   out       E4M3 [rows, cols]           out_t  E4M3 [cols, rows_p]
 *   out_sf    compact codes [rows_p/32, cols/32] or NULL
 *   out_sf_mma    rows = rows, blocks along cols: [rows_p/128][cols/128][512]
 *   out_sf_mma_t  rows = cols, blocks along rows: [cols/128][rows_p/128][512]
 *   (either may be NULL; layout of lpfa_mx_gemm's operand scales).
 * lpfa_rmsnorm_bwd_mx_quantize: the same outputs for dY computed from y (the
 * forward's bf16 Y [rows, cols]), dz (bf16 [rows, cols]), gamma (bf16
 * [cols]) and rstd (fp32 [rows]) in fp32, plus dgamma (fp32 [cols]) summed in
 * a fixed order from dgamma_part (fp32 scratch, 16-byte aligned, of
 * (rows_p/32) * cols + rows_p floats: the per-block partials, then c_t).
 * Errors: NULL or misaligned pointers, cols % 128 != 0 -> INVALID_ARG.
 * ---------------------------------------------------------------------- */
lpfa_status lpfa_mx_quantize_t(const void* x, int64_t rows, int64_t cols, void* out,
                               void* out_t, void* out_sf, void* out_sf_mma,
                               void* out_sf_mma_t, void* stream);
lpfa_status lpfa_rmsnorm_bwd_mx_quantize(const void* y, const void* dz, const void* gamma,
                                         const float* rstd, int64_t rows, int64_t cols,
                                         void* out, void* out_t, void* out_sf,
                                         void* out_sf_mma, void* out_sf_mma_t,
                                         float* dgamma_part, float* dgamma, void* stream);

/* ------------------------------------------------------------------------
 * Tensor-pipe rate of block-scaled MXFP8 MMAs, for the roofline of the
 * attention kernels ([P1] paragraph 2: tcgen05.mma.block_scale).  One CTA
 * per SM issues M128 N256 K32 kind::mxf8f6f4 block-scaled MMAs (E4M3
 * operands resident in shared memory, UE8M0 scales in tensor memory) back to
 * back for about 17 ms; *flops_per_s receives 2*M*N*K per MMA times the MMAs
 * of all CTAs over the CUDA-event time of that launch (after a warm-up
 * launch).  Synchronises `stream`.  Allocates no device memory (its error
 * word is a static device variable).  Errors: flops_per_s NULL ->
 * LPFA_ERR_INVALID_ARG; a launch failure -> LPFA_ERR_CUDA; the kernel's
 * bounded wait expired -> LPFA_ERR_TIMEOUT.
 * ---------------------------------------------------------------------- */
lpfa_status lpfa_mma_peak(double* flops_per_s, void* stream);

/* ------------------------------------------------------------------------
 * Block-scaled MXFP8 GEMM with a quantizing epilogue ([P1] paragraph 2:
 * fused GEMM+Quantize kernels producing FP8 output with dual scale factor
 * layouts in one pass).  The fp32 result D = A * B^T (operands and
 * constraints as lpfa_mx_gemm, with M a multiple of 128) is quantized in
 * registers with the quantizer's rule (lpfa_mx_quantize) before it leaves
 * the SM:
 *   blk = LPFA_BLK_1X32   32 consecutive columns of one row;
 *   blk = LPFA_BLK_32X32  32 rows x 32 columns (transpose-invariant payload).
 * Outputs (device, caller-allocated):
 *   out_e4m3      uint8 [M, N] row-major (16-byte aligned).
 *   out_sf        compact codes: [M, N/32] (1X32) or [M/32, N/32] (32X32),
 *                 8-byte aligned, or NULL.
 *   out_sf_mma    the result as a GEMM operand contracting over N (rows = M):
 *                 [M/128][N/128][512], byte (r%32)*16 + (r/32)*4 + kb of
 *                 tile (i, j) for row 128i + r and block 4j + kb; or NULL.
 *   out_sf_mma_t  32X32 only: as an operand contracting over M (rows = N):
 *                 [N/128][M/128][512]; or NULL.
 *   d             fp32 [M, N] as lpfa_mx_gemm, or NULL (not written).
 * The codes are decided on the fp32 accumulator values that d holds.
 * Errors: as lpfa_mx_gemm; blk = LPFA_BLK_32X1 -> LPFA_ERR_UNSUPPORTED.
 * ---------------------------------------------------------------------- */
lpfa_status lpfa_mx_gemm_quantize(const void* a8, const void* sfa_mma,
                                  const void* b8, const void* sfb_mma,
                                  int64_t M, int64_t N, int64_t K,
                                  lpfa_block blk, void* out_e4m3, void* out_sf,
                                  void* out_sf_mma, void* out_sf_mma_t,
                                  float* d, void* stream);

/* ------------------------------------------------------------------------
 * Attention descriptor.
 *  heads_q % heads_kv == 0 (GQA: query head h reads kv head
 *  h / (heads_q/heads_kv)); head_dim in {64, 128}.
 *  softmax_scale c: logits are c * q.k ([P2] "PyTorch Integration" example,
 *  default 1/sqrt(head_dim)).
 *  causal: key j visible to query i iff j <= i within a sequence.
 *  rescale_threshold (log2 units, >= 0): selective rescaling ([P3]
 *  "Technical Deep Dive"): the running reference max of a row moves to a
 *  key tile's max only when that exceeds it by more than the threshold; P
 *  is quantized against the reference max in force ([P1] paragraph 3).
 *  dq_static_scale: power of two multiplying dQ partials before the FP16
 *  accumulation ([P1] paragraph 3); lpfa_bwd divides it out at the end.
 * ---------------------------------------------------------------------- */
typedef struct lpfa_attn_desc {
  lpfa_seqs seqs;
  int64_t heads_q;
  int64_t heads_kv;
  int64_t head_dim;
  float softmax_scale;
  int32_t causal;
  float rescale_threshold;
  float dq_static_scale;
} lpfa_attn_desc;

/* Bytes of device workspace lpfa_fwd / lpfa_bwd need (>= 256; the first 16
 * bytes hold the error word read by lpfa_check). */
size_t lpfa_fwd_workspace_size(const lpfa_attn_desc* desc);
size_t lpfa_bwd_workspace_size(const lpfa_attn_desc* desc);

/* Forward ([P1] paragraphs 2-3, [P2] "Key Algorithmic Innovations" 1-2).
 *  q8 [T, Hq, D], k8 [T, Hkv, D]: e4m3 payloads of 1X32 quantization;
 *  sfq_mma [Tp/128, Hq, 512], sfk_mma [Tp/128, Hkv, 512]: their out_sf_mma.
 *  v8 [T, Hkv, D]: e4m3 payload of 32X1 quantization; sfv_mma
 *  [Tp/128, Hkv, 512]: its out_sf_mma.
 *  o: bf16 [T, Hq, D] = softmax(c q k^T) v (normalised).
 *  lse: fp32 [Hq, T], natural-log sum_j exp(c q_i.k_j).
 *  workspace: >= lpfa_fwd_workspace_size bytes, 256-byte aligned; zeroed
 *  by the call before use.
 * All data pointers 16-byte aligned. */
lpfa_status lpfa_fwd(const lpfa_attn_desc* desc, const void* q8,
                     const void* sfq_mma, const void* k8, const void* sfk_mma,
                     const void* v8, const void* sfv_mma, void* o, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Forward in bf16 ([P1] paragraph 1: the MXFP8 kernels are measured against
 * their bf16 counterparts).  The same algorithm as lpfa_fwd with kind::f16
 * MMAs on bf16 operands and no block scales: S = c q k^T in fp32, the same
 * online softmax (rescale_threshold as in the descriptor) over 64-key tiles,
 * P rounded to bf16 for the PV product, l summed in fp32.  Its kernel keeps
 * two 128-query tiles in flight per CTA (its faster structure).
 *  q [T, Hq, D], k, v [T, Hkv, D]: bf16, token-major, 16-byte aligned.
 *  o, lse, workspace, errors: as lpfa_fwd. */
lpfa_status lpfa_fwd_bf16(const lpfa_attn_desc* desc, const void* q, const void* k,
                          const void* v, void* o, float* lse, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Self-test of the forward's bounded waits (failure detection; the pages
 * have no counterpart).  Runs lpfa_fwd's kernel with every wait bounded by
 * wait_limit_us microseconds (1 .. 2e6) instead of 2 s, and with the copy of
 * each CTA's first key/value tile withheld, so that the MMA warp's wait for
 * that tile expires: the kernel records the error word, raises its abort
 * flag, drains the copies and MMAs it issued, frees its tensor memory and
 * returns.  Arguments and errors as lpfa_fwd; returns LPFA_OK once the
 * launch is queued, after which lpfa_check(workspace, stream) returns
 * LPFA_ERR_TIMEOUT.  o and lse are left undefined; the stream and the
 * context stay usable. */
lpfa_status lpfa_fwd_wait_expiry_selftest(const lpfa_attn_desc* desc, const void* q8,
                                          const void* sfq_mma, const void* k8,
                                          const void* sfk_mma, const void* v8,
                                          const void* sfv_mma, void* o, float* lse,
                                          void* workspace, size_t workspace_bytes,
                                          uint32_t wait_limit_us, void* stream);

/* Backward ([P1] paragraphs 2-3).
 *  q8, k8, do8: e4m3 payloads of 32X32 quantization, with both scale
 *  arrangements (sf*_mma: contraction over head_dim; sf*_mma_t: contraction
 *  over tokens).  v8/sfv_mma: 1X32 quantization of V.
 *  o (bf16 [T, Hq, D]) and dout (bf16 [T, Hq, D]) give D_i = sum_d dO*O;
 *  lse: the forward's fp32 [Hq, T].
 *  dq: fp16 [T, Hq, D] (zeroed and accumulated by the call; holds dQ after
 *  the call, the static scale divided out); dk, dv: bf16 [T, Hkv, D].
 *  workspace: >= lpfa_bwd_workspace_size bytes. */
lpfa_status lpfa_bwd(const lpfa_attn_desc* desc,
                     const void* q8, const void* sfq_mma, const void* sfq_mma_t,
                     const void* k8, const void* sfk_mma, const void* sfk_mma_t,
                     const void* v8, const void* sfv_mma,
                     const void* do8, const void* sfdo_mma,
                     const void* sfdo_mma_t,
                     const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Backward in bf16 ([P1] paragraph 1: the bf16 counterpart the MXFP8 kernels
 * are measured against).  lpfa_bwd's kernel with kind::f16 MMAs on bf16
 * operands and no block scales: P^T and dS^T are rounded to bf16 for their
 * products, dQ is accumulated in FP16 with the static scale as in lpfa_bwd.
 *  q [T, Hq, D], k, v [T, Hkv, D], o, dout [T, Hq, D]: bf16 (dout is both
 *  the dO operand and the D_i input); lse, dq, dk, dv, workspace, errors: as
 *  lpfa_bwd.  head_dim 128 only (64 -> LPFA_ERR_UNSUPPORTED). */
lpfa_status lpfa_bwd_bf16(const lpfa_attn_desc* desc, const void* q, const void* k,
                          const void* v, const void* o, const void* dout, const float* lse,
                          void* dq, void* dk, void* dv, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * lpfa_bwd_noalloc — the backward for callers that cannot allocate device
 * memory.  (The pages have no counterpart; this is a library convenience.)
 *
 * Some callers cannot hand lpfa_bwd a workspace: code embedded in a runtime
 * that owns every device buffer and gives plugins no allocator, or
 * latency-critical code that must not call cudaMalloc because it can
 * synchronise the whole device.  This entry point takes the same inputs and
 * outputs as lpfa_bwd but keeps its scratch (the error word, and the
 * per-row log2-LSE and D_i arrays) in one static device array of
 * LPFA_BWD_NOALLOC_SCRATCH_BYTES bytes that the library holds on every GPU
 * that loads it, until the process exits.  It allocates nothing itself.
 *  - Size limit: needs lpfa_bwd_workspace_size(desc) <= the array size
 *    (256 + 8 * heads_q * total_sf_rows bytes); larger problems return
 *    LPFA_ERR_INVALID_ARG before any device work.
 *  - The first call on a device looks up the array's device address
 *    (with that device current); make that first call before any stream
 *    capture begins.
 *  - All calls share the array.  Each call clears the part it uses before
 *    its kernels run, but two calls whose work overlaps on the GPU (on
 *    different streams, or on different host threads without ordering)
 *    race on it: serialise them.
 *  - Expired kernel waits are recorded in the shared array, which callers
 *    cannot pass to lpfa_check; use lpfa_bwd with a workspace of your own
 *    when that report is needed.
 * Arguments, layouts and the returned gradients are those of lpfa_bwd. */
#define LPFA_BWD_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
lpfa_status lpfa_bwd_noalloc(const lpfa_attn_desc* desc,
                             const void* q8, const void* sfq_mma,
                             const void* sfq_mma_t, const void* k8,
                             const void* sfk_mma, const void* sfk_mma_t,
                             const void* v8, const void* sfv_mma,
                             const void* do8, const void* sfdo_mma,
                             const void* sfdo_mma_t, const void* o,
                             const void* dout, const float* lse, void* dq,
                             void* dk, void* dv, void* stream);

/* Synchronises `stream`, reads the error word of a workspace used by
 * lpfa_fwd / lpfa_bwd and returns LPFA_ERR_TIMEOUT if a kernel recorded an
 * expired wait, LPFA_ERR_CUDA if the stream holds an error, else LPFA_OK. */
lpfa_status lpfa_check(const void* workspace, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* LPFA_H_ */
