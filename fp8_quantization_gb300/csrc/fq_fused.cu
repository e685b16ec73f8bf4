// One call for the whole MXFP4 forward cast of the MoE recipe: BF16 ->
// MXFP4 (BF16ToFP4Row), the direct FP4 -> FP8 row conversion
// (FP4RowToFP8Row) and the transposed, ragged FP4 -> FP8 conversion
// (FP4RowToFP8Col), with every output byte equal to the three separate
// calls.
//
// Source: "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// technical overview section 2, items 1-3 (the three kernels and the
// no-intermediate principle: FP8 operands are made from the FP4 codes, never
// from a BF16 round trip).
//
// Two stages on the caller's stream: the row stage reads the BF16 tensor
// once and writes the MXFP4 codes and scales together with the FP8 rows made
// from the codes still in registers (the separate FP8 row call would read the
// codes back from memory); the transposed stage then reads the codes and
// scales, which the row stage leaves in L2 with an evict-last policy where
// they fit.
#include "fq_common.cuh"

using namespace fq;

extern "C" fq_status bf16_to_mxfp4_fp8(const void *x, int64_t M, int64_t K,
                                       const int64_t *group_offsets, int32_t G, int exp_offset_k,
                                       uint8_t *q, uint8_t *s, uint8_t *y, float *ys, uint8_t *yT,
                                       float *yT_scale, int64_t cap, int32_t *dev_status,
                                       void *stream)
{
    if (M < 0 || M > INT32_MAX - 512 || K <= 0 || K % 128 != 0)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (((M + 127) / 128) * (K / 128) > INT32_MAX - 4096)  // tile index is 32-bit
        return FQ_ERR_SHAPE;
    if (G < 1 || G > FQ_COLS_MAX_GROUPS || exp_offset_k < 0 || exp_offset_k > 6)
        return FQ_ERR_ARG;
    if (cap < fp4_to_fp8_cols_scale_capacity(M, G))
        return FQ_ERR_ARG;
    if (M == 0)
        return FQ_OK;
    if (!x || !group_offsets || !q || !s || !y || !ys || !yT || !yT_scale)
        return FQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(group_offsets) || !aligned16(q) || !aligned16(s) ||
        !aligned16(y) || !aligned16(ys) || !aligned16(yT) || !aligned16(yT_scale))
        return FQ_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const fq_status rc = launch_mxfp4_rows(x, M, K, q, s, exp_offset_k, y, ys, st);
    if (rc != FQ_OK)
        return rc;
    return launch_fp4_to_fp8_cols(q, s, M, K, group_offsets, G, exp_offset_k, yT, yT_scale, cap,
                                  dev_status, st);
}
