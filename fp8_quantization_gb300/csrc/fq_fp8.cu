// BF16 -> FP8 E4M3 block quantization (1x128 row blocks and 128x128 tiles)
// and MXFP4 -> BF16 dequantization.
//
// Source: "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// technical overview section 2: gradients stay in standard FP8 (item 2, the
// asymmetric FP4-forward / FP8-backward flow); the Hopper FP8 pipeline uses
// E4M3 with 128-element blocks and FP32 block scales (item 1); an MXFP4
// element's value is its E2M1 value times the block's power-of-two scale
// (item 1).
//
// Quantizer, per block (binary32, one rounding per operation):
//   r = min(448 / amax, FLT_MAX), s = amax / 448 (the dequantization scale),
//   code = E4M3(x * r) round to nearest even, saturating at 448;
//   a block holding NaN or Inf gets s = NaN and all codes 0x7F.
// Dequantizer: BF16(v * 2^(e - 127)), exact or +-infinity on overflow; a
// block with scale byte 0xFF gives 0x7FC0 everywhere.
#include <cfloat>

#include "fq_common.cuh"

namespace fq {

// Eight FP32 values -> eight E4M3 bytes (two words), round to nearest even
// with saturation; cvt ... e4m3x2 puts its first source in the upper byte.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d)
{
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// r and s of a block from the |x| bits of its max (a BF16 pattern).
__device__ __forceinline__ void fp8_block_factors(uint32_t amax_bits16, float &r, float &s)
{
    const float amax = __uint_as_float(amax_bits16 << 16);
    r = fminf(__fdiv_rn(448.0f, amax), FLT_MAX);
    s = __fdiv_rn(amax, 448.0f);
}

// Eight BF16 values (one uint4) times r -> eight E4M3 bytes.
__device__ __forceinline__ uint2 fp8_encode8(uint4 v, float r)
{
    float p[8];
    fmul2(bf16_lo(v.x), bf16_hi(v.x), r, p[0], p[1]);
    fmul2(bf16_lo(v.y), bf16_hi(v.y), r, p[2], p[3]);
    fmul2(bf16_lo(v.z), bf16_hi(v.z), r, p[4], p[5]);
    fmul2(bf16_lo(v.w), bf16_hi(v.w), r, p[6], p[7]);
    return make_uint2(cvt_e4m3x4(p[0], p[1], p[2], p[3]), cvt_e4m3x4(p[4], p[5], p[6], p[7]));
}

// ---------------------------------------------------------------- 1 x 128

// One warp tile = 8 blocks of 128 elements.  Lane l owns the 16-byte chunks
// l, l+32, l+64, l+96; chunk c belongs to block c / 16, so in unroll step i
// lanes 0-15 hold block 2i and lanes 16-31 block 2i+1: four xor shuffles give
// the block max.  Loads cover 512 contiguous bytes per warp, code stores 256.
__global__ void __launch_bounds__(kThreads) fp8_quantize_1x128_kernel(
    const uint16_t *__restrict__ x, int64_t nblk, uint8_t *__restrict__ y, float *__restrict__ s)
{
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t ntiles = (nblk + 7) >> 3;

    for (int64_t tile = warp; tile < ntiles; tile += nwarps) {
        const int64_t c0 = tile << 7;  // first chunk of the tile
        uint4 v[4];
        bool ok[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int64_t c = c0 + lane + 32 * i;
            ok[i] = (c >> 4) < nblk;
            v[i] = ok[i] ? ld_nc_v4(x + c * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            uint32_t m = absmax_bf16x2(absmax_bf16x2(v[i].x & 0x7FFF7FFFu, v[i].y), v[i].z);
            m = absmax_bf16x2(m, v[i].w);
#pragma unroll
            for (int d = 1; d < 16; d <<= 1)
                m = max_u16x2(m, __shfl_xor_sync(0xffffffffu, m, d));
            const uint32_t amax = hmax_u16x2(m);
            const bool special = amax >= 0x7F80u;
            float r, sc;
            fp8_block_factors(amax, r, sc);
            uint2 codes = fp8_encode8(v[i], r);
            if (special)
                codes = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
            if (ok[i]) {
                const int64_t c = c0 + lane + 32 * i;
                __stcs(reinterpret_cast<uint2 *>(y + c * 8), codes);
                if ((lane & 15) == 0)
                    reinterpret_cast<uint32_t *>(s)[c >> 4] =
                        special ? 0x7FC00000u : __float_as_uint(sc);
            }
        }
    }
}

// ---------------------------------------------------------------- 128 x 128

// One CTA per 128 x 128 tile: thread t holds columns 8 (t % 16) .. +7 of rows
// t / 16 + 16 j, j = 0..7 (every warp load covers two 256-byte row segments);
// the tile max is a warp shuffle reduction plus one shared-memory step.
__global__ void __launch_bounds__(kThreads) fp8_quantize_128x128_kernel(
    const uint16_t *__restrict__ w, int64_t N, int64_t K, uint8_t *__restrict__ y,
    float *__restrict__ s)
{
    __shared__ uint32_t red[kThreads / 32];
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t tcols = K >> 7;
    const int64_t ntiles = (N >> 7) * tcols;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t tr = tile / tcols, tc = tile - tr * tcols;
        const int64_t row0 = (tr << 7) + (tid >> 4);
        const int64_t col = (tc << 7) + 8 * (tid & 15);
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; j++)
            v[j] = ld_nc_v4(w + (row0 + 16 * j) * K + col);
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            m = absmax_bf16x2(m, v[j].x);
            m = absmax_bf16x2(m, v[j].y);
            m = absmax_bf16x2(m, v[j].z);
            m = absmax_bf16x2(m, v[j].w);
        }
        uint32_t h = hmax_u16x2(m);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
            h = max(h, __shfl_xor_sync(0xffffffffu, h, d));
        if (lane == 0)
            red[wid] = h;
        __syncthreads();
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < kThreads / 32; i++)
            amax = max(amax, red[i]);
        __syncthreads();  // red is reused by the next tile
        const bool special = amax >= 0x7F80u;
        float r, sc;
        fp8_block_factors(amax, r, sc);
#pragma unroll
        for (int j = 0; j < 8; j++) {
            uint2 codes = fp8_encode8(v[j], r);
            if (special)
                codes = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
            __stcs(reinterpret_cast<uint2 *>(y + (row0 + 16 * j) * K + col), codes);
        }
        if (tid == 0)
            reinterpret_cast<uint32_t *>(s)[tile] = special ? 0x7FC00000u : __float_as_uint(sc);
    }
}

// ---------------------------------------------------------------- MXFP4 -> BF16

// Per scale byte e a 16-byte table row: the high bytes (8) then the low bytes
// (8) of BF16(v_m * 2^(e - 127)) for the E2M1 magnitudes m = 0..7, built in
// shared memory at kernel start with binary32 products (exact: v_m has at most
// two significant bits, 2^(e - 127) is a binary32 number for every e < 255,
// and an overflowing product is infinity, as its BF16 rounding); row 255 is
// 0x7FC0 throughout.
__device__ __forceinline__ void build_dequant_table(uint8_t *tab /* [256 * 16] */)
{
    for (int i = threadIdx.x; i < 256 * 8; i += blockDim.x) {
        const int e = i >> 3, c = i & 7;
        uint32_t bits;
        if (e == 255) {
            bits = 0x7FC0u;
        } else {
            float v;
            if (c == 0)
                v = 0.0f;
            else if (c == 1)
                v = 0.5f;
            else
                v = __uint_as_float(((126u + (c >> 1)) << 23) | ((c & 1u) << 22));
            const float p2 = __uint_as_float(e ? static_cast<uint32_t>(e) << 23 : 0x00400000u);
            bits = __float_as_uint(__fmul_rn(v, p2)) >> 16;
        }
        tab[16 * e + c] = static_cast<uint8_t>(bits >> 8);
        tab[16 * e + 8 + c] = static_cast<uint8_t>(bits & 0xFFu);
    }
}

// Lane l of a warp step owns 8 codes (4 bytes) and writes their 16 BF16
// bytes: loads cover 128 contiguous bytes per warp, stores 512.
constexpr int kDeqUnroll = 8;

__global__ void __launch_bounds__(kThreads) mxfp4_dequantize_rows_kernel(
    const uint8_t *__restrict__ q, const uint8_t *__restrict__ s, int64_t nw /* code words */,
    uint16_t *__restrict__ out)
{
    __shared__ __align__(16) uint8_t tab[256 * 16];
    build_dequant_table(tab);
    __syncthreads();
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
    const uint32_t *q32 = reinterpret_cast<const uint32_t *>(q);
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t w0 = gtid; w0 < nw; w0 += kDeqUnroll * nthr) {
        uint32_t c[kDeqUnroll], e[kDeqUnroll];
#pragma unroll
        for (int u = 0; u < kDeqUnroll; u++) {
            const int64_t wi = w0 + u * nthr;
            c[u] = wi < nw ? __ldg(q32 + wi) : 0u;
            e[u] = wi < nw ? __ldg(s + (wi >> 2)) : 0u;  // 4 code words per MX block
        }
#pragma unroll
        for (int u = 0; u < kDeqUnroll; u++) {
            const int64_t wi = w0 + u * nthr;
            if (wi >= nw)
                break;
            const uint4 t = *reinterpret_cast<const uint4 *>(tab + 16 * e[u]);
            const uint32_t smask = e[u] == 255u ? 0u : 0x80808080u;
            uint32_t h03, h47, l03, l47;
            // high bytes carry the sign (bit 7), low bytes never do
            fp4x8_to_fp8x8(c[u], t.x, t.y, h03, h47, smask);
            const uint32_t sel = c[u] & 0x77777777u;
            l03 = prmt(t.z, t.w, sel);
            l47 = prmt(t.z, t.w, sel >> 16);
            uint4 o;
            o.x = prmt(l03, h03, 0x5140u);  // elements 0, 1
            o.y = prmt(l03, h03, 0x7362u);  // elements 2, 3
            o.z = prmt(l47, h47, 0x5140u);  // elements 4, 5
            o.w = prmt(l47, h47, 0x7362u);  // elements 6, 7
            __stcs(reinterpret_cast<uint4 *>(out + wi * 8), o);
        }
    }
}

}  // namespace fq

using namespace fq;

extern "C" fq_status fp8_quantize_1x128(const void *x, int64_t M, int64_t K, uint8_t *y, float *s,
                                        void *stream)
{
    if (M < 0 || K <= 0 || K % 128 != 0)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (M == 0)
        return FQ_OK;
    if (!x || !y || !s)
        return FQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(y) || !aligned16(s))
        return FQ_ERR_ALIGN;
    const int64_t nblk = M * (K / 128);
    const int64_t work = (nblk + 8 * (kThreads / 32) - 1) / (8 * (kThreads / 32));
    const int grid = persistent_grid(fp8_quantize_1x128_kernel, kThreads, 0, work, 4);
    launch_pdl(fp8_quantize_1x128_kernel, dim3(grid), dim3(kThreads), 0,
               static_cast<cudaStream_t>(stream), static_cast<const uint16_t *>(x), nblk, y, s);
    return launch_status();
}

extern "C" fq_status fp8_quantize_128x128(const void *w, int64_t N, int64_t K, uint8_t *y, float *s,
                                          void *stream)
{
    if (N < 0 || K <= 0 || N % 128 != 0 || K % 128 != 0)
        return FQ_ERR_SHAPE;
    if (N > 0 && K > INT64_MAX / N)
        return FQ_ERR_SHAPE;
    if (N == 0)
        return FQ_OK;
    if (!w || !y || !s)
        return FQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(y) || !aligned16(s))
        return FQ_ERR_ALIGN;
    const int64_t tiles = (N / 128) * (K / 128);
    const int grid = persistent_grid(fp8_quantize_128x128_kernel, kThreads, 0, tiles, 4);
    launch_pdl(fp8_quantize_128x128_kernel, dim3(grid), dim3(kThreads), 0,
               static_cast<cudaStream_t>(stream), static_cast<const uint16_t *>(w), N, K, y, s);
    return launch_status();
}

extern "C" fq_status mxfp4_dequantize_rows(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K,
                                           void *x, void *stream)
{
    if (M < 0 || K <= 0 || K % 32 != 0)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (M == 0)
        return FQ_OK;
    if (!q || !s || !x)
        return FQ_ERR_NULL;
    if (!aligned16(q) || !aligned16(s) || !aligned16(x))
        return FQ_ERR_ALIGN;
    const int64_t nw = M * (K / 8);
    const int64_t work = (nw + kDeqUnroll * kThreads - 1) / (kDeqUnroll * kThreads);
    const int grid = persistent_grid(mxfp4_dequantize_rows_kernel, kThreads, 0, work, 4);
    launch_pdl(mxfp4_dequantize_rows_kernel, dim3(grid), dim3(kThreads), 0,
               static_cast<cudaStream_t>(stream), q, s, nw, static_cast<uint16_t *>(x));
    return launch_status();
}
