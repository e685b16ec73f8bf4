// MXFP4 row quantization (BF16ToFP4Row) and direct FP4 -> FP8 row conversion
// (FP4RowToFP8Row).
//
// Source: "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// technical overview section 2 -- 32-element MX blocks with a UE8M0 scale and
// E2M1 elements, two values per byte; the bitwise FP4->FP8 conversion that
// aligns the four MX exponents of a 128-element block to their maximum.
//
// Both kernels stream HBM once: 128-bit loads, warp-shuffle block amax, packed
// conversion instructions, coalesced stores; persistent grids sized to the
// SM count.  Rows play no role: with K a multiple of the block, a row-major
// tensor is a flat sequence of blocks.
#include "fq_common.cuh"

namespace fq {

// ---------------------------------------------------------------- a1: BF16 -> MXFP4

// One warp tile = 32 MX blocks = 1024 elements.  Lane l owns the 16-byte
// chunks l, l+32, l+64, l+96 of the tile; chunk c is quarter (c & 3) of MX
// block c >> 2, so the four lanes 4g..4g+3 hold block g + 8i of unroll i and
// a two-step xor shuffle gives the block amax.  Every load and every code
// store of the warp covers 512 / 128 contiguous bytes.
//
// kRows8 fuses the FP8 row conversion of the fresh codes (FP4RowToFP8Row):
// unroll step i of a warp holds two whole 128-element FP8 blocks (lanes 0-15
// and 16-31; lanes 4 and 8 apart hold the other MX blocks of a lane's FP8
// block), so S is a two-shuffle byte max and each lane converts its 8 codes
// with the shift table exactly as the FP8 row kernel does.  x is then read
// and y written with an L2 evict-first policy and q, s written evict-last:
// the transposed conversion that follows reads them back from L2.
template <bool kRows8>
__global__ void __launch_bounds__(kThreads) mxfp4_quantize_rows_kernel(
    const uint16_t *__restrict__ x, int64_t nblk, uint8_t *__restrict__ q,
    uint8_t *__restrict__ s, int k, uint8_t *__restrict__ y, float *__restrict__ ys)
{
    __shared__ __align__(16) uint8_t tab[kRows8 ? kTabRows * 8 : 8];
    uint64_t keep = 0, stream = 0;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t ntiles = (nblk + 31) >> 5;
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    if (kRows8) {
        // the warp's first tile is requested into L2 before the shift table
        // is built, as in the FP8 row kernel
        if (warp < ntiles)
            for (int i = 0; i < 4; i++) {
                const int64_t blk = (warp << 5) + (lane >> 2) + 8 * i;
                if (blk < nblk)
                    prefetch_l2(x + blk * 32 + (lane & 3) * 8);
            }
        build_fp8_table(tab);
        __syncthreads();
        keep = l2_evict_last();
        stream = l2_evict_first();
    }
    griddep_launch_dependents();  // the next kernel may start its set-up

    for (int64_t tile = warp; tile < ntiles; tile += nwarps) {
        const int64_t blk0 = tile << 5;
        uint4 v[4];
        bool ok[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int64_t blk = blk0 + (lane >> 2) + 8 * i;
            ok[i] = blk < nblk;
            const uint16_t *src = x + blk * 32 + (lane & 3) * 8;
            v[i] = ok[i] ? (kRows8 ? ld_nc_v4_hint(src, stream) : ld_nc_v4(src))
                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint32_t m = absmax_bf16x2(absmax_bf16x2(v[i].x & 0x7FFF7FFFu, v[i].y), v[i].z);
            m = absmax_bf16x2(m, v[i].w);
            m = max_u16x2(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = max_u16x2(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const uint32_t amax = hmax_u16x2(m);  // |x| bits of the block max
            // e = max(E - 2, 0) for the block max's exponent field E (BF16
            // subnormals and zero have E = 0); 0xFF if the block has NaN/Inf.
            const bool special = amax >= 0x7F80u;
            const int E = static_cast<int>(amax >> 7);
            const uint32_t e = static_cast<uint32_t>(E > 2 ? E - 2 : 0);  // <= 252
            const float mul = __uint_as_float((254u - e) << 23);             // 2^(127 - e)
            uint32_t codes = cvt_e2m1x8(
                __fmul_rn(bf16_lo(v[i].x), mul), __fmul_rn(bf16_hi(v[i].x), mul),
                __fmul_rn(bf16_lo(v[i].y), mul), __fmul_rn(bf16_hi(v[i].y), mul),
                __fmul_rn(bf16_lo(v[i].z), mul), __fmul_rn(bf16_hi(v[i].z), mul),
                __fmul_rn(bf16_lo(v[i].w), mul), __fmul_rn(bf16_hi(v[i].w), mul));
            if (special)
                codes = 0;
            const uint32_t eb = special ? 0xFFu : e;  // the block's scale byte
            const int64_t blk = blk0 + (lane >> 2) + 8 * i;
            if (kRows8) {
                uint32_t S = max(eb, __shfl_xor_sync(0xffffffffu, eb, 4));
                S = max(S, __shfl_xor_sync(0xffffffffu, S, 8));
                int u = static_cast<int>(S - eb) - k + 6;  // >= 0: S is the max
                u = u < kShiftRows - 1 ? u : kShiftRows - 1;
                const bool nan = S == 0xFFu;
                const uint2 t = *reinterpret_cast<const uint2 *>(tab + 8 * (nan ? kNanRow : u));
                uint32_t lo, hi;
                fp4x8_to_fp8x8(codes, t.x, t.y, lo, hi, nan ? 0u : 0x80808080u);
                if (ok[i]) {
                    st_u32_hint(q + blk * 16 + (lane & 3) * 4, codes, keep);
                    if ((lane & 3) == 0)
                        st_u8_hint(s + blk, eb, keep);
                    __stcs(reinterpret_cast<uint2 *>(y + blk * 32 + (lane & 3) * 8),
                           make_uint2(lo, hi));
                    if ((lane & 15) == 0)
                        reinterpret_cast<uint32_t *>(ys)[blk >> 2] = fp8_block_scale_bits(S, k);
                }
            } else if (ok[i]) {
                *reinterpret_cast<uint32_t *>(q + blk * 16 + (lane & 3) * 4) = codes;
                if ((lane & 3) == 0)
                    s[blk] = static_cast<uint8_t>(eb);
            }
        }
    }
}

// ---------------------------------------------------------------- a2: FP4 -> FP8 rows

// One warp pass = 4 FP8 blocks (128 elements each): lane l converts 16 codes
// (8 bytes of q) of FP8 block (l >> 3), i.e. half of MX block (l & 7) >> 1,
// into 16 E4M3 bytes.  The four scale bytes of an FP8 block are one aligned
// 32-bit word.  Per MX block an 8-entry magnitude table row is fetched from
// shared memory by shift; codes are translated with byte permutes.
constexpr int kRowsUnroll = 8;

__global__ void __launch_bounds__(kThreads) fp4_to_fp8_rows_kernel(
    const uint8_t *__restrict__ q, const uint8_t *__restrict__ s, int64_t nfb, int k,
    uint8_t *__restrict__ y, float *__restrict__ ys)
{
    __shared__ __align__(16) uint8_t tab[kTabRows * 8];
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up

    const int lane = threadIdx.x & 31;
    const int part = lane & 7;  // 8-byte part of the 64-byte FP8 block
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t ntiles = (nfb + 4 * kRowsUnroll - 1) / (4 * kRowsUnroll);
    // the warp's first tile is requested into L2 before the shift table is
    // built, so that its DRAM latency runs under the table and the barrier
    // (16384 x 7168: 30.8 -> 30.2 us alone, 71.7 -> 70.5 us after the row
    // quantizer; building the table before the programmatic-launch wait
    // instead overlaps it with the previous kernel but leaves the first
    // loads behind it)
    if (warp < ntiles && part == 0) {
        const int64_t fb0 = warp * (4 * kRowsUnroll);
        for (int i = 0; i < kRowsUnroll; i++) {
            const int64_t fb = fb0 + 4 * i + (lane >> 3);
            if (fb < nfb) {
                prefetch_l2(q + fb * 64);
                prefetch_l2(s + fb * 4);
            }
        }
    }
    build_fp8_table(tab);
    __syncthreads();

    for (int64_t tile = warp; tile < ntiles; tile += nwarps) {
        const int64_t fb0 = tile * (4 * kRowsUnroll);
        uint2 c[kRowsUnroll];
        uint32_t sw[kRowsUnroll];
#pragma unroll
        for (int i = 0; i < kRowsUnroll; i++) {
            const int64_t fb = fb0 + 4 * i + (lane >> 3);
            if (fb < nfb) {
                c[i] = __ldg(reinterpret_cast<const uint2 *>(q + fb * 64 + part * 8));
                sw[i] = __ldg(reinterpret_cast<const uint32_t *>(s) + fb);
            } else {
                c[i] = make_uint2(0, 0);
                sw[i] = 0;
            }
        }
#pragma unroll
        for (int i = 0; i < kRowsUnroll; i++) {
            const int64_t fb = fb0 + 4 * i + (lane >> 3);
            const uint32_t w = sw[i];
            const uint32_t b0 = w & 0xFFu, b1 = (w >> 8) & 0xFFu, b2 = (w >> 16) & 0xFFu,
                           b3 = w >> 24;
            const uint32_t S = max(max(b0, b1), max(b2, b3));
            const uint32_t e = (w >> (8 * (part >> 1))) & 0xFFu;
            int u = static_cast<int>(S - e) - k + 6;
            u = u < kShiftRows - 1 ? u : kShiftRows - 1;
            const uint2 t = *reinterpret_cast<const uint2 *>(tab + 8 * u);
            uint4 out;
            fp4x8_to_fp8x8(c[i].x, t.x, t.y, out.x, out.y);
            fp4x8_to_fp8x8(c[i].y, t.x, t.y, out.z, out.w);
            if (S == 0xFFu)
                out = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
            if (fb < nfb) {
                __stcs(reinterpret_cast<uint4 *>(y + fb * 128 + part * 16), out);  // evict-first: y is not re-read
                if (part == 0)
                    reinterpret_cast<uint32_t *>(ys)[fb] = fp8_block_scale_bits(S, k);
            }
        }
    }
}

// ---------------------------------------------------------------- MMA scale layout

// MXFP4 scales in the tiled layout that Blackwell block-scaled MMA operands
// use: 512-byte atoms of 128 rows x 4 scale columns, atom (rb, cb) at byte
// (rb * ncb + cb) * 512, and inside an atom the scale of row 32i + j, column
// l at byte 16j + 4i + l.  A CTA takes one (128-row block, chunk of 16 atom
// columns) unit at a time: each thread loads 8 words (half warps read 64
// contiguous bytes of a row; rows past M and columns past the row's end read
// as zero) into shared memory, and after a barrier each warp writes two whole
// atoms, lane j the 16 bytes of rows j, j+32, j+64, j+96 (shared rows are
// padded by one word, so those four reads are free of bank conflicts): one
// 512-byte contiguous store per warp per atom.
constexpr int kMmaRows = 128;    // rows of an atom
constexpr int kMmaChunk = 16;    // atom columns (4-byte words of a row) per unit
constexpr int kMmaRowWords = kMmaChunk + 1;

__global__ void __launch_bounds__(kThreads) mxfp4_scales_mma_kernel(const uint8_t *__restrict__ s,
                                                                    int64_t M, int64_t ncb,
                                                                    int64_t nrb,
                                                                    uint8_t *__restrict__ out)
{
    __shared__ uint32_t rows[kMmaRows * kMmaRowWords];
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint32_t *s32 = reinterpret_cast<const uint32_t *>(s);
    const int64_t nch = (ncb + kMmaChunk - 1) / kMmaChunk;  // chunks per row block
    const int w = tid & 15, i0 = tid >> 4;                  // word, first row of this thread
    for (int64_t u = blockIdx.x; u < nrb * nch; u += gridDim.x) {
        const int64_t rb = u / nch, c0 = (u - rb * nch) * kMmaChunk;
        const bool col_ok = c0 + w < ncb;
        uint32_t v[kMmaRows / 16];
#pragma unroll
        for (int k = 0; k < kMmaRows / 16; k++) {
            const int64_t r = 128 * rb + i0 + 16 * k;
            v[k] = r < M && col_ok ? __ldg(s32 + r * ncb + c0 + w) : 0u;  // ncb words per row
        }
#pragma unroll
        for (int k = 0; k < kMmaRows / 16; k++)
            rows[(i0 + 16 * k) * kMmaRowWords + w] = v[k];
        __syncthreads();
        for (int c = wid; c < kMmaChunk && c0 + c < ncb; c += kThreads / 32) {
            uint4 o;
            o.x = rows[lane * kMmaRowWords + c];
            o.y = rows[(lane + 32) * kMmaRowWords + c];
            o.z = rows[(lane + 64) * kMmaRowWords + c];
            o.w = rows[(lane + 96) * kMmaRowWords + c];
            __stcs(reinterpret_cast<uint4 *>(out + (rb * ncb + c0 + c) * 512 + 16 * lane), o);
        }
        __syncthreads();  // the rows are read before the next unit lands
    }
}

}  // namespace fq

using namespace fq;

namespace fq {

fq_status launch_mxfp4_rows(const void *x, int64_t M, int64_t K, uint8_t *q, uint8_t *s, int k,
                            uint8_t *y, float *ys, cudaStream_t st)
{
    const int64_t nblk = M * (K / 32);
    const int64_t work = (nblk + 32 * (kThreads / 32) - 1) / (32 * (kThreads / 32));
    if (y) {
        const int grid = persistent_grid(mxfp4_quantize_rows_kernel<true>, kThreads, 0, work, 4);
        launch_pdl(mxfp4_quantize_rows_kernel<true>, dim3(grid), dim3(kThreads), 0, st,
                   static_cast<const uint16_t *>(x), nblk, q, s, k, y, ys);
    } else {
        const int grid = persistent_grid(mxfp4_quantize_rows_kernel<false>, kThreads, 0, work, 4);
        launch_pdl(mxfp4_quantize_rows_kernel<false>, dim3(grid), dim3(kThreads), 0, st,
                   static_cast<const uint16_t *>(x), nblk, q, s, 0, static_cast<uint8_t *>(nullptr),
                   static_cast<float *>(nullptr));
    }
    return launch_status();
}

}  // namespace fq

extern "C" fq_status mxfp4_quantize_rows(const void *x, int64_t M, int64_t K, uint8_t *q,
                                         uint8_t *s, void *stream)
{
    if (M < 0 || K <= 0 || K % 32 != 0)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (M == 0)
        return FQ_OK;
    if (!x || !q || !s)
        return FQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s))
        return FQ_ERR_ALIGN;
    return launch_mxfp4_rows(x, M, K, q, s, 0, nullptr, nullptr,
                             static_cast<cudaStream_t>(stream));
}

extern "C" fq_status fp4_to_fp8_rows(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K,
                                     int exp_offset_k, uint8_t *y, float *ys, void *stream)
{
    if (M < 0 || K <= 0 || K % 128 != 0)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (exp_offset_k < 0 || exp_offset_k > 6)
        return FQ_ERR_ARG;
    if (M == 0)
        return FQ_OK;
    if (!q || !s || !y || !ys)
        return FQ_ERR_NULL;
    if (!aligned16(q) || !aligned16(s) || !aligned16(y) || !aligned16(ys))
        return FQ_ERR_ALIGN;
    const int64_t nfb = M * (K / 128);
    const int64_t per_cta = 4 * kRowsUnroll * (kThreads / 32);
    const int grid =
        persistent_grid(fp4_to_fp8_rows_kernel, kThreads, 0, (nfb + per_cta - 1) / per_cta, 4);
    launch_pdl(fp4_to_fp8_rows_kernel, dim3(grid), dim3(kThreads), 0,
               static_cast<cudaStream_t>(stream), q, s, nfb, exp_offset_k, y, ys);
    return launch_status();
}

extern "C" int64_t mxfp4_scales_mma_bytes(int64_t M, int64_t K)
{
    if (M < 0 || K <= 0 || K % 128 != 0 || M > INT64_MAX - 127)
        return -1;
    const int64_t nrb = (M + 127) / 128;
    if (nrb > INT64_MAX / 512 / (K / 128))  // the byte count must fit in int64
        return -1;
    return nrb * (K / 128) * 512;
}

extern "C" fq_status mxfp4_scales_mma_layout(const uint8_t *s, int64_t M, int64_t K,
                                             uint8_t *s_mma, void *stream)
{
    if (mxfp4_scales_mma_bytes(M, K) < 0)
        return FQ_ERR_SHAPE;
    if (M == 0)
        return FQ_OK;
    if (!s || !s_mma)
        return FQ_ERR_NULL;
    if (!aligned16(s) || !aligned16(s_mma))
        return FQ_ERR_ALIGN;
    const int64_t ncb = K / 128;
    const int64_t nrb = (M + 127) / 128;
    const int grid = persistent_grid(mxfp4_scales_mma_kernel, kThreads, 0,
                                     nrb * ((ncb + kMmaChunk - 1) / kMmaChunk));
    launch_pdl(mxfp4_scales_mma_kernel, dim3(grid), dim3(kThreads), 0,
               static_cast<cudaStream_t>(stream), s, M, ncb, nrb, s_mma);
    return launch_status();
}
