// NVFP4 quantization: per-tensor amax, 1x16 micro-blocks (round to nearest
// even or stochastic rounding) and 16x16 2D weight blocks.
//
// Source: "Train models faster with JAX and MaxText using NVFP4 on NVIDIA
// Blackwell", section "Receta de pre-entrenamiento NVFP4": 16-element
// micro-block scaling, E4M3 block scale factors under an FP32 per-tensor
// scale, 2D 16x16 weight scaling, stochastic rounding for gradients (round
// to nearest even for weights and activations).
//
// The scale arithmetic is IEEE binary32 with one rounding per operation
// (explicit __fdiv_rn / __frcp_rn / __fmul_rn), so every code is a function
// of the inputs alone:
//   g = A / 2688 (1 if A == 0); enc = 1 / (6 g); t = amax_blk * enc;
//   b = E4M3(t); r = min(1 / (b g), FLT_MAX) (0 if b == 0);
//   code = E2M1(|x| r), sign of x.
// enc and the 128 possible r values are computed once per CTA.
#include <cfloat>

#include "fq_common.cuh"

namespace fq {

// ---------------------------------------------------------------- amax

__global__ void __launch_bounds__(kThreads, 6) nvfp4_amax_kernel(const uint16_t *__restrict__ x,
                                                              int64_t n,
                                                              uint32_t *__restrict__ out_bits)
{
    __shared__ uint32_t red[kThreads / 32];
    const int64_t nvec = n >> 3;  // 16-byte chunks
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    uint32_t m = 0;
    int64_t i = gtid;
    for (; i + 3 * nthr < nvec; i += 4 * nthr) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; u++)
            v[u] = ld_nc_v4(x + (i + u * nthr) * 8);
#pragma unroll
        for (int u = 0; u < 4; u++) {
            m = absmax_bf16x2(m, v[u].x);
            m = absmax_bf16x2(m, v[u].y);
            m = absmax_bf16x2(m, v[u].z);
            m = absmax_bf16x2(m, v[u].w);
        }
    }
    for (; i < nvec; i += nthr) {
        const uint4 v = ld_nc_v4(x + i * 8);
        m = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(m, v.x), v.y), v.z), v.w);
    }
    for (int64_t t = nvec * 8 + gtid; t < n; t += nthr)
        m = max_u16x2(m, x[t] & 0x7FFFu);
    uint32_t h = hmax_u16x2(m);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        h = max(h, __shfl_xor_sync(0xffffffffu, h, d));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = h;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int w = 0; w < kThreads / 32; w++)
            b = max(b, red[w]);
        // |x| as binary32 bits: non-negative floats order like their bits,
        // and NaN patterns sit above infinity.
        atomicMax(out_bits, b << 16);
    }
}

// ---------------------------------------------------------------- block scale

// Per-tensor set-up, once per CTA: decode scale g, encode factor
// enc = 1 / (6 g), and the table r[b] = min(1 / (b g), FLT_MAX) (r[0] = 0)
// of element multipliers for every E4M3 block-scale byte b.
struct TensorScales {
    float g, enc;
};

__device__ __forceinline__ TensorScales nvfp4_tensor_setup(const float *amax, float *rtab /* [128] */)
{
    const float A = *amax;
    TensorScales ts;
    ts.g = A > 0.0f ? __fdiv_rn(A, 2688.0f) : 1.0f;
    ts.enc = __frcp_rn(__fmul_rn(6.0f, ts.g));
    for (int b = threadIdx.x; b < 128; b += blockDim.x)
        rtab[b] = b ? fminf(__frcp_rn(__fmul_rn(e4m3_value(b), ts.g)), FLT_MAX) : 0.0f;
    __syncthreads();
    return ts;
}

struct BlockScale {
    uint32_t b;  // E4M3 byte
    float r;     // element multiplier
};

__device__ __forceinline__ BlockScale nvfp4_block_scale(uint32_t amax_bits16, float enc,
                                                        const float *rtab)
{
    BlockScale bs;
    bs.b = cvt_e4m3(__fmul_rn(__uint_as_float(amax_bits16 << 16), enc));
    bs.r = rtab[bs.b];
    return bs;
}

// Eight BF16 values (one uint4) times r -> eight E2M1 codes in a word,
// round to nearest even (sign kept, including -0).
__device__ __forceinline__ uint32_t encode8_rne(uint4 v, float r)
{
    float p0, p1, p2, p3, p4, p5, p6, p7;
    fmul2(bf16_lo(v.x), bf16_hi(v.x), r, p0, p1);
    fmul2(bf16_lo(v.y), bf16_hi(v.y), r, p2, p3);
    fmul2(bf16_lo(v.z), bf16_hi(v.z), r, p4, p5);
    fmul2(bf16_lo(v.w), bf16_hi(v.w), r, p6, p7);
    return cvt_e2m1x8(p0, p1, p2, p3, p4, p5, p6, p7);
}

// Eight BF16 values times r -> eight E2M1 codes, stochastic rounding: the
// Blackwell FP4 conversion adds 16 random bits below the kept precision of
// each value and truncates.  Values 0..3 draw on random word w0, 4..7 on w1;
// within a group of four, value i sits in nibble i (first source = nibble 3).
__device__ __forceinline__ uint32_t encode8_sr(uint4 v, float r, uint32_t w0, uint32_t w1)
{
    float p0, p1, p2, p3, p4, p5, p6, p7;
    fmul2(bf16_lo(v.x), bf16_hi(v.x), r, p0, p1);
    fmul2(bf16_lo(v.y), bf16_hi(v.y), r, p2, p3);
    fmul2(bf16_lo(v.z), bf16_hi(v.z), r, p4, p5);
    fmul2(bf16_lo(v.w), bf16_hi(v.w), r, p6, p7);
    uint16_t lo, hi;
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=h"(lo)
        : "f"(p3), "f"(p2), "f"(p1), "f"(p0), "r"(w0));
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=h"(hi)
        : "f"(p7), "f"(p6), "f"(p5), "f"(p4), "r"(w1));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// ---------------------------------------------------------------- 1x16

// One lane per 16-element block (32 bytes of input, 8 bytes of codes), four
// blocks in flight per lane (their Philox chains interleave).  With
// stochastic rounding the block's Philox call (counter = offset/16 + block)
// yields one random word per four values.
constexpr int kNvUnroll = 4;

template <bool kSR>
__global__ void __launch_bounds__(kThreads) nvfp4_quantize_kernel(
    const uint16_t *__restrict__ x, int64_t nblk, const float *__restrict__ amax, uint64_t seed,
    uint64_t offset, uint8_t *__restrict__ q, uint8_t *__restrict__ sb, float *__restrict__ g_out)
{
    __shared__ float rtab[128];
    const TensorScales ts = nvfp4_tensor_setup(amax, rtab);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *g_out = ts.g;
    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    const uint64_t c0 = offset >> 4;

    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;

    for (int64_t b0 = gtid; b0 < nblk; b0 += kNvUnroll * nthr) {
        uint4 v[kNvUnroll][2];
#pragma unroll
        for (int u = 0; u < kNvUnroll; u++) {
            const int64_t blk = b0 + u * nthr;
            if (blk < nblk) {
                v[u][0] = ld_nc_v4(x + blk * 16);
                v[u][1] = ld_nc_v4(x + blk * 16 + 8);
            } else {
                v[u][0] = v[u][1] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < kNvUnroll; u++) {
            const int64_t blk = b0 + u * nthr;
            if (blk >= nblk)
                break;
            uint32_t m = absmax_bf16x2(absmax_bf16x2(v[u][0].x & 0x7FFF7FFFu, v[u][0].y), v[u][0].z);
            m = absmax_bf16x2(absmax_bf16x2(m, v[u][0].w), v[u][1].x);
            m = absmax_bf16x2(absmax_bf16x2(m, v[u][1].y), v[u][1].z);
            m = absmax_bf16x2(m, v[u][1].w);
            const BlockScale bs = nvfp4_block_scale(hmax_u16x2(m), ts.enc, rtab);
            uint2 codes;
            if (kSR) {
                const uint64_t c = c0 + static_cast<uint64_t>(blk);
                const uint4 w = philox4x32_10(
                    make_uint4(static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32), 0u, 0u),
                    k0, k1);
                codes.x = encode8_sr(v[u][0], bs.r, w.x, w.y);
                codes.y = encode8_sr(v[u][1], bs.r, w.z, w.w);
            } else {
                codes.x = encode8_rne(v[u][0], bs.r);
                codes.y = encode8_rne(v[u][1], bs.r);
            }
            __stcs(reinterpret_cast<uint2 *>(q + blk * 8), codes);
            sb[blk] = static_cast<uint8_t>(bs.b);
        }
    }
}

// ---------------------------------------------------------------- 16x16

// A warp owns a 16-row strip x 256 columns: lane l holds columns 8l..8l+7 of
// all 16 rows (lanes 2t, 2t+1 form tile t), so every row load / store of the
// warp is 512 / 128 contiguous bytes.
__global__ void __launch_bounds__(kThreads, 2) nvfp4_quantize_2d_kernel(
    const uint16_t *__restrict__ w, int64_t N, int64_t K, const float *__restrict__ amax,
    uint8_t *__restrict__ q, uint8_t *__restrict__ sb, float *__restrict__ g_out)
{
    __shared__ float rtab[128];
    const TensorScales ts = nvfp4_tensor_setup(amax, rtab);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *g_out = ts.g;

    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t ncg = (K + 255) >> 8;  // 256-column groups
    const int64_t nunits = (N >> 4) * ncg;

    for (int64_t unit = warp; unit < nunits; unit += nwarps) {
        const int64_t strip = unit / ncg;
        const int64_t col = ((unit - strip * ncg) << 8) + 8 * lane;
        const bool ok = col < K;
        const uint16_t *src = w + (strip << 4) * K + col;
        uint4 v[16];
#pragma unroll
        for (int r = 0; r < 16; r++)
            v[r] = ok ? ld_nc_v4(src + r * K) : make_uint4(0, 0, 0, 0);
        uint32_t m = 0;
#pragma unroll
        for (int r = 0; r < 16; r++) {
            m = absmax_bf16x2(m, v[r].x);
            m = absmax_bf16x2(m, v[r].y);
            m = absmax_bf16x2(m, v[r].z);
            m = absmax_bf16x2(m, v[r].w);
        }
        m = max_u16x2(m, __shfl_xor_sync(0xffffffffu, m, 1));
        const BlockScale bs = nvfp4_block_scale(hmax_u16x2(m), ts.enc, rtab);
        if (ok) {
            uint8_t *dst = q + (strip << 4) * (K >> 1) + (col >> 1);
#pragma unroll
            for (int r = 0; r < 16; r++)
                __stcs(reinterpret_cast<unsigned int *>(dst + r * (K >> 1)), encode8_rne(v[r], bs.r));
            if (!(lane & 1))
                sb[strip * (K >> 4) + (col >> 4)] = static_cast<uint8_t>(bs.b);
        }
    }
}

}  // namespace fq

using namespace fq;

extern "C" fq_status nvfp4_amax(const void *x, int64_t n, float *amax, void *stream)
{
    if (n < 0)
        return FQ_ERR_SHAPE;
    if (!amax || (n > 0 && !x))
        return FQ_ERR_NULL;
    if ((n > 0 && !aligned16(x)) || !aligned16(amax))
        return FQ_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(amax, 0, sizeof(float), st) != cudaSuccess)
        return launch_status();
    if (n == 0)
        return FQ_OK;
    const int64_t work = (n / 8 + 4 * kThreads - 1) / (4 * kThreads);
    const int grid = persistent_grid(nvfp4_amax_kernel, kThreads, 0, work < 1 ? 1 : work);
    nvfp4_amax_kernel<<<grid, kThreads, 0, st>>>(static_cast<const uint16_t *>(x), n,
                                                  reinterpret_cast<uint32_t *>(amax));
    return launch_status();
}

extern "C" fq_status nvfp4_quantize(const void *x, int64_t M, int64_t K, const float *amax,
                                    int use_sr, uint64_t seed, uint64_t offset, uint8_t *q,
                                    uint8_t *sb, float *g, void *stream)
{
    if (M < 0 || K <= 0 || K % 16 != 0)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (offset % 16 != 0 || (use_sr != 0 && use_sr != 1))
        return FQ_ERR_ARG;
    if (M == 0)
        return FQ_OK;
    if (!x || !amax || !q || !sb || !g)
        return FQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(amax) || !aligned16(q) || !aligned16(sb) || !aligned16(g))
        return FQ_ERR_ALIGN;
    const int64_t nblk = M * (K / 16);
    const int64_t work = (nblk + kNvUnroll * kThreads - 1) / (kNvUnroll * kThreads);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (use_sr) {
        const int grid = persistent_grid(nvfp4_quantize_kernel<true>, kThreads, 0, work);
        nvfp4_quantize_kernel<true><<<grid, kThreads, 0, st>>>(
            static_cast<const uint16_t *>(x), nblk, amax, seed, offset, q, sb, g);
    } else {
        const int grid = persistent_grid(nvfp4_quantize_kernel<false>, kThreads, 0, work);
        nvfp4_quantize_kernel<false><<<grid, kThreads, 0, st>>>(
            static_cast<const uint16_t *>(x), nblk, amax, seed, offset, q, sb, g);
    }
    return launch_status();
}

extern "C" fq_status nvfp4_quantize_2d(const void *w, int64_t N, int64_t K, const float *amax,
                                       uint8_t *q, uint8_t *sb, float *g, void *stream)
{
    if (N < 0 || K <= 0 || N % 16 != 0 || K % 16 != 0)
        return FQ_ERR_SHAPE;
    if (N > 0 && K > INT64_MAX / N)
        return FQ_ERR_SHAPE;
    if (N == 0)
        return FQ_OK;
    if (!w || !amax || !q || !sb || !g)
        return FQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(amax) || !aligned16(q) || !aligned16(sb) || !aligned16(g))
        return FQ_ERR_ALIGN;
    const int64_t units = (N / 16) * ((K + 255) / 256);
    const int grid =
        persistent_grid(nvfp4_quantize_2d_kernel, kThreads, 0, (units + 7) / 8);
    nvfp4_quantize_2d_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(w), N, K, amax, q, sb, g);
    return launch_status();
}
