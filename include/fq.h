/*
 * fq.h -- C ABI of libfq.so: block-scaled FP4 / FP8 casts of training
 * tensors on GB300 (sm_103a).
 *
 * Formats and operations follow two sources, cited by page title and section:
 *   [MoE-FP4] "Practical FP4 Training for Large-Scale MoE Models on Hopper
 *             GPUs", technical overview, section 2 (Methodology):
 *             item 1 -- MXFP4 = 32-element blocks sharing a power-of-two UE8M0
 *             scale, E2M1 elements; direct bitwise FP4->FP8 conversion without
 *             a BF16 intermediate; hierarchical scale alignment that maps four
 *             32-element MX blocks onto one 128-element E4M3 block by aligning
 *             exponents to the largest of the four scales;
 *             item 2 -- FP4 values packed two per uint8;
 *             item 3 -- kernels BF16ToFP4Row, FP4RowToFP8Row, FP4RowToFP8Col
 *             (transpose fused with the conversion, for Wgrad) and ragged
 *             per-expert token groups handled without padding.
 *   [NVFP4]   "Train models faster with JAX and MaxText using NVFP4 on NVIDIA
 *             Blackwell", section "Receta de pre-entrenamiento NVFP4":
 *             16-element micro-blocks, E4M3 block scales under one FP32
 *             per-tensor scale, 16x16 2D block scaling of weights, stochastic
 *             rounding for gradient quantizers.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor is dense, row-major, contiguous, and lives in device memory
 *   of the current CUDA device; the caller allocates and owns every buffer.
 *   The library allocates nothing and keeps no state between calls.
 * - Every pointer must be 16-byte aligned.  Inputs and outputs must not
 *   overlap.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *   enqueued on it asynchronously; no entry point synchronizes the host.
 *   Every kernel is launched with programmatic dependent launch: it may
 *   be scheduled while the stream's previous kernel is still running, but
 *   touches no global memory before that kernel has completed, so stream
 *   order holds for every buffer.
 * - Arguments are checked on the host before anything is enqueued; a failed
 *   check returns a status other than FQ_OK and enqueues nothing.  A failed
 *   launch returns FQ_ERR_CUDA (the CUDA error code is then available from
 *   fq_last_cuda_error() in the calling thread).
 * - A size of 0 rows is a successful no-op.
 * - BF16 inputs are passed as 16-bit words.  Non-finite inputs are not an
 *   error: MXFP4 marks the block (scale byte 0xFF); for NVFP4 a non-finite
 *   per-tensor amax is a precondition violation that still writes only
 *   inside the outputs.
 *
 * Encodings
 * ---------
 * - E2M1 code (4 bits): sign bit 3, magnitude code 0..7 = {0, 0.5, 1, 1.5,
 *   2, 3, 4, 6}.  Element 2i is the low nibble of byte i, element 2i+1 the
 *   high nibble.  Rounding is to nearest, ties to the even code, saturating
 *   at 6; the sign of a value rounded to zero is kept.
 * - UE8M0 byte e encodes 2^(e-127); 0xFF marks a block with NaN or Inf.
 * - E4M3 ("fn": bias 7, 0x7F = NaN, largest finite 448), round to nearest
 *   even, saturating at 448.
 */
#ifndef FQ_H
#define FQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FQ_OK = 0,
    FQ_ERR_NULL = 1,  /* a required pointer is NULL */
    FQ_ERR_SHAPE = 2, /* a size is negative, too large, or not a multiple of the block */
    FQ_ERR_ALIGN = 3, /* a pointer is not 16-byte aligned */
    FQ_ERR_ARG = 4,   /* another argument is out of range */
    FQ_ERR_CUDA = 5   /* the CUDA runtime reported an error */
} fq_status;

/* Static, human-readable name of a status. */
const char *fq_status_string(int status);

/* cudaError_t of the last FQ_ERR_CUDA returned in the calling thread (0 if none). */
int fq_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int fq_version(void);

/*
 * MXFP4 row quantization of BF16 activations ([MoE-FP4] 2.1 and 2.3,
 * BF16ToFP4Row).
 *   x  : bf16 [M, K]            input
 *   q  : uint8 [M, K/2]         packed E2M1 codes (output)
 *   s  : uint8 [M, K/32]        UE8M0 scale per 32-element block (output)
 * For each block of 32 consecutive elements of a row: amax = max |x|;
 * e = clamp(floor(log2 amax) - 2 + 127, 0, 254) (e = 0 for an all-zero
 * block); each element is rounded as x / 2^(e-127) to E2M1.  A block that
 * holds NaN or Inf gets e = 0xFF and all-zero codes.
 * Requires K > 0, K % 32 == 0, M >= 0.
 */
fq_status mxfp4_quantize_rows(const void *x, int64_t M, int64_t K, uint8_t *q, uint8_t *s,
                              void *stream);

/*
 * Direct FP4 -> FP8 conversion, row layout ([MoE-FP4] 2.1, FP4RowToFP8Row).
 *   q, s : MXFP4 [M, K/2], [M, K/32] as produced by mxfp4_quantize_rows
 *   y    : uint8 [M, K]          E4M3 codes (output)
 *   ys   : float [M, K/128]      FP32 dequantization scale per 128 elements (output)
 * Each 128-element block covers four MX blocks with exponents e0..e3;
 * S = max(e_i).  An element of MX block i with E2M1 value v becomes
 * E4M3(v * 2^(k - (S - e_i))), sign kept; ys = 2^(S - 127 - k), so
 * ys * y == 2^(e_i - 127) * v exactly wherever S - e_i <= k + 8.  If any
 * e_i is 0xFF the block gets ys = NaN (0x7FC00000) and all codes 0x7F.
 * `exp_offset_k` (k) in [0, 6]: 0 is the plain alignment to the largest
 * scale; larger k keeps k more binades exact (6 * 2^6 <= 448).
 * Requires K > 0, K % 128 == 0, M >= 0.
 */
fq_status fp4_to_fp8_rows(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K,
                          int exp_offset_k, uint8_t *y, float *ys, void *stream);

/* Largest number of 128-token blocks fp4_to_fp8_cols can produce for M rows
 * in G groups: ceil(M / 128) + G.  Returns -1 for M < 0 or G < 1. */
int64_t fp4_to_fp8_cols_scale_capacity(int64_t M, int32_t G);

/* Largest group count accepted by fp4_to_fp8_cols. */
#define FQ_COLS_MAX_GROUPS 1024

/* Number of kernels fp4_to_fp8_cols enqueues for feature count K: 1 (one
 * pass that also computes the block scales) when the CUDA driver can encode
 * tensor maps; 0 for a K the conversion rejects, or without that driver
 * support (the conversion then returns FQ_ERR_CUDA, cudaErrorNotSupported).
 * Host only: no kernel is launched (for a valid K it initialises the CUDA
 * runtime on the current device, as the conversion itself would). */
int fp4_to_fp8_cols_launch_count(int64_t K);

/*
 * Direct FP4 -> FP8 conversion fused with the transpose, on ragged
 * per-expert token groups without padding ([MoE-FP4] 2.3, FP4RowToFP8Col;
 * the Wgrad operand layout).
 *   q, s          : MXFP4 [M, K/2], [M, K/32] (M tokens, K features)
 *   group_offsets : int64 [G+1] in DEVICE memory; group g owns tokens
 *                   offsets[g] .. offsets[g+1]-1; offsets[0] = 0,
 *                   non-decreasing, offsets[G] = M (empty groups allowed)
 *   yT            : uint8 [K, M]   E4M3, element (feature k, token t) at k*M + t
 *   yT_scale      : float [cap, K]: row base_g + b holds the FP32 scales of
 *                   block b of group g, feature k at (base_g + b)*K + k,
 *                   base_g = sum_{h<g} ceil(count_h/128) (one row of K
 *                   scales per block, as a GEMM reading the scales of one
 *                   token block wants them); rows past the last block are
 *                   not written
 *   cap           : >= fp4_to_fp8_cols_scale_capacity(M, G)
 *   dev_status    : optional int32 in device memory; if the offsets are
 *                   malformed the kernel clamps them (so nothing is written
 *                   out of bounds) and ORs 1 into *dev_status; 2 is ORed in
 *                   if a shared-memory copy of the single pass did not
 *                   arrive within two seconds (the outputs are then
 *                   incomplete; not expected to happen)
 * Each group is cut into 128-token blocks starting at its first token (the
 * last block of a group may be short).  For a block and a 32-feature MX
 * column, S = max of the tokens' exponents; each element is converted as in
 * fp4_to_fp8_rows with that S.  Requires K % 128 == 0, 1 <= G <=
 * FQ_COLS_MAX_GROUPS, 0 <= M < 2^31, k in [0, 6].
 */
fq_status fp4_to_fp8_cols(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K,
                          const int64_t *group_offsets, int32_t G, int exp_offset_k,
                          uint8_t *yT, float *yT_scale, int64_t cap, int32_t *dev_status,
                          void *stream);

/*
 * The MXFP4 forward cast in one call ([MoE-FP4] 2.1-2.3: BF16ToFP4Row,
 * FP4RowToFP8Row and FP4RowToFP8Col without any BF16 intermediate): every
 * output is byte-for-byte what mxfp4_quantize_rows(x) -> (q, s) followed by
 * fp4_to_fp8_rows(q, s, k) -> (y, ys) and fp4_to_fp8_cols(q, s, offsets, k)
 * -> (yT, yT_scale) produce; dev_status as in fp4_to_fp8_cols.  The BF16
 * tensor is read once: the FP8 rows are made from the codes in registers,
 * and the transposed stage reads q and s back (kept in L2 where they fit).
 *   x : bf16 [M, K];  q, s, y, ys, yT, yT_scale, group_offsets, G, cap :
 *   as in the three calls.  Requires K % 128 == 0, 1 <= G <=
 *   FQ_COLS_MAX_GROUPS, 0 <= M < 2^31, k in [0, 6].  Enqueues two
 *   kernels (the row kernel, then the transposed conversion).
 */
fq_status bf16_to_mxfp4_fp8(const void *x, int64_t M, int64_t K, const int64_t *group_offsets,
                            int32_t G, int exp_offset_k, uint8_t *q, uint8_t *s, uint8_t *y,
                            float *ys, uint8_t *yT, float *yT_scale, int64_t cap,
                            int32_t *dev_status, void *stream);

/*
 * The same call as one kernel: the BF16 tensor is read once and every output
 * is written once from registers and shared memory, q and s are not read
 * back.  Same arguments, outputs (byte for byte) and requirements as
 * bf16_to_mxfp4_fp8; *dev_status also gets bit 2 if a shared-memory copy did
 * not land within the kernel's time limit.  Slower than bf16_to_mxfp4_fp8 on
 * GB300.  Needs the driver's tensor-map encoder: without it the call returns
 * FQ_ERR_CUDA with cudaErrorNotSupported as the CUDA error.
 */
fq_status bf16_to_mxfp4_fp8_single_pass(const void *x, int64_t M, int64_t K,
                                        const int64_t *group_offsets, int32_t G, int exp_offset_k,
                                        uint8_t *q, uint8_t *s, uint8_t *y, float *ys, uint8_t *yT,
                                        float *yT_scale, int64_t cap, int32_t *dev_status,
                                        void *stream);

/*
 * BF16 -> FP8 E4M3 block quantization for the FP8 backward flow ([MoE-FP4]
 * 2.2: gradients stay in standard FP8; 2.1: the Hopper FP8 pipeline is E4M3
 * with 128-element blocks and FP32 block scales).  The pages give the format
 * only; this library's rule, per block, in IEEE binary32:
 *   r = min(448 / amax, FLT_MAX), s = amax / 448 (the dequantization scale),
 *   code = E4M3(x * r), round to nearest even, saturating at 448, sign kept;
 *   a block holding NaN or Inf gets s = NaN (0x7FC00000) and codes 0x7F.
 *   Decode: x ~ s * E4M3(code).
 * fp8_quantize_1x128:   x bf16 [M, K] -> y uint8 [M, K], s float [M, K/128]
 *                       (blocks of 128 consecutive elements of a row);
 *                       K % 128 == 0.
 * fp8_quantize_128x128: w bf16 [N, K] -> y uint8 [N, K], s float [N/128, K/128]
 *                       (128 x 128 tiles); N % 128 == 0, K % 128 == 0.
 */
fq_status fp8_quantize_1x128(const void *x, int64_t M, int64_t K, uint8_t *y, float *s,
                             void *stream);
fq_status fp8_quantize_128x128(const void *w, int64_t N, int64_t K, uint8_t *y, float *s,
                               void *stream);

/*
 * MXFP4 -> BF16 dequantization ([MoE-FP4] 2.1: an element's value is its
 * E2M1 value times 2^(e-127) of its block's UE8M0 scale byte e).
 *   q, s : MXFP4 [M, K/2], [M, K/32];  x : bf16 [M, K] (output)
 * Element = BF16(v * 2^(e-127)): exact, or +-infinity where the product
 * exceeds BF16's range; the code's sign is kept (code 8 gives -0); a block
 * with e = 0xFF gives 0x7FC0 everywhere.  Requires K % 32 == 0.
 */
fq_status mxfp4_dequantize_rows(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K, void *x,
                                void *stream);

/*
 * MXFP4 scales re-laid for a block-scaled MMA operand ([MoE-FP4] 2.1 fixes
 * the UE8M0 scale per 32-element block; the pages fix no layout for a GEMM
 * to read it, so this is the tiled layout that Blackwell's block-scaled MMA
 * operands use for their scale factors, as NVIDIA documents it for its
 * block-scaled GEMMs).
 *   s     : uint8 [M, K/32]  row-major scales, as mxfp4_quantize_rows writes them
 *   s_mma : uint8, mxfp4_scales_mma_bytes(M, K) bytes (output): 512-byte atoms
 *           of 128 rows x 4 scale columns; atom (rb, cb) starts at byte
 *           (rb * (K/128) + cb) * 512; the scale of row 128 rb + 32 i + j,
 *           column 4 cb + l sits at byte 16 j + 4 i + l of its atom; rows
 *           from M up to the next multiple of 128 are 0.
 * Requires K > 0, K % 128 == 0, M >= 0; s and s_mma 16-byte aligned.
 * mxfp4_scales_mma_bytes returns -1 for a rejected shape.
 */
int64_t mxfp4_scales_mma_bytes(int64_t M, int64_t K);
fq_status mxfp4_scales_mma_layout(const uint8_t *s, int64_t M, int64_t K, uint8_t *s_mma,
                                  void *stream);

/*
 * Per-tensor amax for NVFP4's FP32 tensor scale ([NVFP4] "Receta"):
 *   x      : bf16 [n]
 *   amax   : float in device memory (output) = max |x| (NaN if x holds NaN;
 *            0 for n == 0)
 */
fq_status nvfp4_amax(const void *x, int64_t n, float *amax, void *stream);

/*
 * NVFP4 1x16 quantization ([NVFP4] "Receta": 16-element micro-blocks with
 * E4M3 block scales under one FP32 per-tensor scale; stochastic rounding).
 *   x        : bf16 [M, K]
 *   amax     : float in device memory, max |x| of the whole tensor (nvfp4_amax)
 *   q        : uint8 [M, K/2]   packed E2M1 codes (output)
 *   sb       : uint8 [M, K/16]  E4M3 block scales (output)
 *   g        : float in device memory, per-tensor decode scale (output)
 * With all arithmetic in IEEE binary32, one rounding per operation:
 *   g = amax / 2688 (g = 1 if amax == 0), enc = 1 / (6 g);  per block:
 *   t = amax_blk * enc, b = E4M3(t), r = min(1 / (b g), FLT_MAX) (r = 0 if
 *   b == 0), element code = E2M1(|x| * r) with the sign of x.
 *   Decode: x ~ v * b * g.
 * use_sr = 0: round to nearest even.  use_sr = 1: stochastic rounding --
 *   with lo <= y < hi the neighbouring grid points and
 *   F = floor(2^16 (y - lo) / (hi - lo)), round up iff F + R >= 2^16, R a
 *   16-bit random number.  Element j = offset + i (i its row-major index in
 *   this call) takes R from W = output word (j / 4) mod 4 of Philox4x32-10
 *   with key (seed low word, seed high word) and counter (c low word, c high
 *   word, 0, 0), c = j / 16: with P = W[23:16] * 256 + W[7:0] and
 *   Q = W[31:24] * 256 + W[15:8], elements j mod 4 = 0, 1, 2, 3 use P,
 *   bitrev16(P), Q, bitrev16(Q).  Each element's R is uniform over 16 bits,
 *   but the two elements of a pair (j mod 4 in {0, 1} or {2, 3}) draw
 *   bit-reversed copies of one number, so their rounding decisions are not
 *   independent of each other (this is how Blackwell's cvt.rs ... e2m1x4
 *   spreads one 32-bit random word over four values; the NVFP4 page's
 *   "Redondeo estocástico" names only unbiased rounding, native to those
 *   instructions).  `offset` lets row shards of one tensor reproduce the
 *   unsharded stream; it must be a multiple of 16.
 * Requires K > 0, K % 16 == 0, M >= 0.
 */
fq_status nvfp4_quantize(const void *x, int64_t M, int64_t K, const float *amax, int use_sr,
                         uint64_t seed, uint64_t offset, uint8_t *q, uint8_t *sb, float *g,
                         void *stream);

/*
 * Random Hadamard transform for the NVFP4 WGRAD inputs ([NVFP4] "Receta":
 * a random Hadamard transform is applied only to the WGRAD GEMM inputs, to
 * make outliers Gaussian before 4-bit quantization).  The page fixes neither
 * size, order, sign source nor precision; this library reads it as: per 16
 * consecutive elements along the contiguous dimension,
 *     y = 1/4 H16 diag(d) x,   H16[i][j] = (-1)^popcount(i & j),
 * d_i = -1 where bit i of sign_mask (low 16 bits) is set, else +1, computed
 * in IEEE binary32: the signed inputs, then the butterfly stages h = 1, 2, 4,
 * 8 (pair (j, j+h) with bit h of j clear -> (a + b, a - b)), then times 0.25.
 * Pass the operand with its GEMM reduction dimension contiguous.
 *
 * nvfp4_amax_rht: amax (device float) = max |y| over the transformed
 *   tensor x[n], n % 16 == 0 (NaN if a transformed value is NaN; 0 for n == 0).
 * nvfp4_quantize_rht: nvfp4_quantize applied to y instead of x (amax = max |y|,
 *   block amax over |y|, element codes E2M1(|y| r) with the sign of y; the
 *   stochastic-rounding stream and `offset` as in nvfp4_quantize).  The
 *   transformed amax must be finite.
 */
fq_status nvfp4_amax_rht(const void *x, int64_t n, uint32_t sign_mask, float *amax, void *stream);
fq_status nvfp4_quantize_rht(const void *x, int64_t M, int64_t K, const float *amax,
                             uint32_t sign_mask, int use_sr, uint64_t seed, uint64_t offset,
                             uint8_t *q, uint8_t *sb, float *g, void *stream);

/* Largest history window accepted by nvfp4_quantize_delayed. */
#define FQ_AMAX_WINDOW_MAX 4096

/*
 * NVFP4 1x16 quantization with delayed per-tensor scaling from a Max-Window
 * amax history ("Max-Window scale estimation for HiF8 W8A8 QAT", 手法 and
 * 貢献 2: the A_max estimate is the maximum over a 64-step history window,
 * which rules out scale-induced saturation for every step inside it).  One
 * pass over x: no separate amax read.
 *   amax_history : uint64 [window + 1] in device memory, caller-owned,
 *                  zero-initialised once; entry = (step << 32) | binary32
 *                  bits of that step's amax.
 *   window       : W in [1, FQ_AMAX_WINDOW_MAX] (64 in the source);
 *   step         : t, the caller's step counter (32-bit, may wrap).
 * The per-tensor amax A is the largest amax of the entries tagged t-W .. t-1
 * (0 if none, so g = 1 until the history fills); x is quantized exactly as
 * nvfp4_quantize with that A (a tensor larger than its estimate saturates);
 * then entry t mod (W+1) becomes (t << 32) | bits(max |x|), unless it
 * already carries tag t with a larger amax.  Calls sharing one history must
 * be ordered on one stream.  Other arguments as in nvfp4_quantize.
 */
fq_status nvfp4_quantize_delayed(const void *x, int64_t M, int64_t K, uint64_t *amax_history,
                                 int32_t window, uint32_t step, int use_sr, uint64_t seed,
                                 uint64_t offset, uint8_t *q, uint8_t *sb, float *g, void *stream);

/*
 * NVFP4 with 16x16 2D block scaling of weights ([NVFP4] "Escalado de pesos
 * 2D": one scale per 16x16 tile so that FPROP and the transposed DGRAD use
 * the same scales).
 *   w   : bf16 [N, K];  amax: float in device memory, max |w|
 *   q   : uint8 [N, K/2] packed E2M1 codes (output)
 *   sb  : uint8 [N/16, K/16] E4M3 tile scales (output)
 *   g   : float in device memory (output)
 * As nvfp4_quantize with round-to-nearest-even, amax_blk taken over the tile.
 * Requires N % 16 == 0, K % 16 == 0, K > 0, N >= 0.
 */
fq_status nvfp4_quantize_2d(const void *w, int64_t N, int64_t K, const float *amax, uint8_t *q,
                            uint8_t *sb, float *g, void *stream);

/*
 * The 2D weight quantization together with the DGRAD operand ([NVFP4]
 * "Escalado de pesos 2D": FPROP and its transposed DGRAD use the same 16x16
 * scales).  Reading: the DGRAD operand is W^T [K, N] laid out as any 2D
 * quantized tensor, with block (j, i) scaled by sb[i][j] and every code equal
 * to W's code of the same element; it is what nvfp4_quantize_2d gives for the
 * BF16 transpose of w.  One read of w.
 *   w, amax, q, sb, g : as in nvfp4_quantize_2d
 *   qT  : uint8 [K, N/2] packed E2M1 codes of W^T (element (k, n) in nibble
 *         n of row k, element 2i in the low nibble) (output)
 *   sbT : uint8 [K/16, N/16] E4M3 tile scales of W^T, sbT[j][i] = sb[i][j]
 *         (output)
 * Requires N % 16 == 0, K % 16 == 0, K > 0, N >= 0; pointers 16-byte aligned.
 */
fq_status nvfp4_quantize_2d_t(const void *w, int64_t N, int64_t K, const float *amax, uint8_t *q,
                              uint8_t *sb, uint8_t *qT, uint8_t *sbT, float *g, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FQ_H */
