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
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
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

// ---------------------------------------------------------------- random Hadamard transform

// 16-point random Hadamard transform of one block ("Transformada de Hadamard
// Aleatoria" of the recipe, applied to the WGRAD inputs): y = 1/4 H16 diag(d) x
// with H16[i][j] = (-1)^popcount(i & j) and d_i = -1 where bit i of the sign
// mask is set.  The sign flips act on the BF16 words (flip[i] holds the sign
// bits of elements 2i and 2i+1); then the four butterfly stages in binary32
// (pair (j, j + h) with bit h of j clear -> (a + b, a - b), h = 1, 2, 4, 8) and
// the factor 0.25, in that order, so the result is a fixed function of x.
struct RhtFlip {
    uint32_t w[8];
};

__device__ __forceinline__ RhtFlip rht_flip_words(uint32_t sign_mask)
{
    RhtFlip f;
#pragma unroll
    for (int i = 0; i < 8; i++)
        f.w[i] = (((sign_mask >> (2 * i)) & 1u) << 15) | (((sign_mask >> (2 * i + 1)) & 1u) << 31);
    return f;
}

// Packed IEEE binary32 pairs: (a, b) -> (a + b, a - b) element-wise on
// (a0, a1) and (b0, b1), and (a0, a1) * c; one rounding per element, as the
// scalar operations.
__device__ __forceinline__ void addsub2(float &a0, float &a1, float &b0, float &b1)
{
    asm("{\n\t.reg .b64 A, B, S, D;\n\t"
        "mov.b64 A, {%0, %1};\n\t"
        "mov.b64 B, {%2, %3};\n\t"
        "add.rn.f32x2 S, A, B;\n\t"
        "sub.rn.f32x2 D, A, B;\n\t"
        "mov.b64 {%0, %1}, S;\n\t"
        "mov.b64 {%2, %3}, D;\n\t}"
        : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// Butterfly stages h = 2, 4, 8 on pairs (j, j + 1), after stage h = 1.
__device__ __forceinline__ void rht16_stages248(float z[16])
{
#pragma unroll
    for (int h = 2; h < 16; h <<= 1)
#pragma unroll
        for (int j = 0; j < 16; j += 2)
            if (!(j & h))
                addsub2(z[j], z[j + 1], z[j + h], z[j + h + 1]);
}

// The butterflies, without the final factor 0.25 (z = H16 diag(d) x).
__device__ __forceinline__ void rht16_z(const uint4 &a, const uint4 &b, const RhtFlip &f, float z[16])
{
    const uint32_t w[8] = {a.x ^ f.w[0], a.y ^ f.w[1], a.z ^ f.w[2], a.w ^ f.w[3],
                           b.x ^ f.w[4], b.y ^ f.w[5], b.z ^ f.w[6], b.w ^ f.w[7]};
    // stage h = 1 pairs the two halves of a BF16 word
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const float u = bf16_lo(w[i]), v = bf16_hi(w[i]);
        z[2 * i] = __fadd_rn(u, v);
        z[2 * i + 1] = __fsub_rn(u, v);
    }
    rht16_stages248(z);
}

// The same transform with the sign flips as bit 31 of one word per element,
// folded into the BF16 -> binary32 conversions ((w << 16) + 2^31 flips bit
// 31 as an exclusive or would).  The amax kernel takes these words as a
// kernel argument, so they are read from the constant bank instead of being
// held in registers (41.4 -> 40.4 us on 16384 x 7168; the quantizer with the
// same change went from 48 to 68 registers and became slower).
struct RhtFlipBits {
    uint32_t lo[8], hi[8];  // element 2i / 2i+1 flips where bit 31 is set
};

inline RhtFlipBits rht_flip_bits(uint32_t sign_mask)
{
    RhtFlipBits f;
    for (int i = 0; i < 8; i++) {
        f.lo[i] = ((sign_mask >> (2 * i)) & 1u) << 31;
        f.hi[i] = ((sign_mask >> (2 * i + 1)) & 1u) << 31;
    }
    return f;
}

__device__ __forceinline__ void rht16_z(const uint4 &a, const uint4 &b, const RhtFlipBits &f,
                                        float z[16])
{
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const float u = __uint_as_float((w[i] << 16) + f.lo[i]);
        const float v = __uint_as_float((w[i] & 0xFFFF0000u) ^ f.hi[i]);
        z[2 * i] = __fadd_rn(u, v);
        z[2 * i + 1] = __fsub_rn(u, v);
    }
    rht16_stages248(z);
}

__device__ __forceinline__ void rht16(const uint4 &a, const uint4 &b, const RhtFlip &f, float y[16])
{
    rht16_z(a, b, f, y);
#pragma unroll
    for (int i = 0; i < 16; i += 2)
        fmul2(y[i], y[i + 1], 0.25f, y[i], y[i + 1]);
}

// max |y| over the transformed tensor: |y| bits ordered as unsigned integers
// (NaN above infinity above every finite value), one atomicMax per CTA.
__global__ void __launch_bounds__(kThreads) nvfp4_amax_rht_kernel(const uint16_t *__restrict__ x,
                                                                  int64_t nblk, const RhtFlipBits f,
                                                                  uint32_t *__restrict__ out_bits)
{
    __shared__ uint32_t red[kThreads / 32];
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    uint32_t m = 0;
    for (int64_t b0 = gtid; b0 < nblk; b0 += 2 * nthr) {
        uint4 v[2][2];
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const int64_t blk = b0 + u * nthr;
            if (blk < nblk) {
                v[u][0] = ld_nc_v4(x + blk * 16);
                v[u][1] = ld_nc_v4(x + blk * 16 + 8);
            } else {
                v[u][0] = v[u][1] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; u++) {
            float z[16];
            rht16_z(v[u][0], v[u][1], f, z);
#pragma unroll
            for (int i = 0; i < 16; i++)
                m = max(m, __float_as_uint(z[i]) & 0x7FFFFFFFu);
        }
    }
    // max |y| = max |z| * 0.25: rounding is monotone (NaN bit patterns stay NaN)
    {
        const float mz = __uint_as_float(m);
        if (m <= 0x7F800000u)
            m = __float_as_uint(__fmul_rn(mz, 0.25f));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t b = 0;
        for (int w = 0; w < kThreads / 32; w++)
            b = max(b, red[w]);
        atomicMax(out_bits, b);
    }
}

// ---------------------------------------------------------------- block scale

// Per-tensor set-up, once per CTA: decode scale g, encode factor
// enc = 1 / (6 g), and the table r[b] = min(1 / (b g), FLT_MAX) (r[0] = 0)
// of element multipliers for every E4M3 block-scale byte b.
struct TensorScales {
    float g, enc;
};

__device__ __forceinline__ TensorScales nvfp4_tensor_setup_from(float A, float *rtab /* [128] */)
{
    TensorScales ts;
    ts.g = A > 0.0f ? __fdiv_rn(A, 2688.0f) : 1.0f;
    ts.enc = __frcp_rn(__fmul_rn(6.0f, ts.g));
    for (int b = threadIdx.x; b < 128; b += blockDim.x)
        rtab[b] = b ? fminf(__frcp_rn(__fmul_rn(e4m3_value(b), ts.g)), FLT_MAX) : 0.0f;
    __syncthreads();
    return ts;
}

__device__ __forceinline__ TensorScales nvfp4_tensor_setup(const float *amax, float *rtab /* [128] */)
{
    return nvfp4_tensor_setup_from(*amax, rtab);
}

// ---------------------------------------------------------------- Max-Window history

// Delayed per-tensor scaling ("Max-Window scale estimation for HiF8 W8A8
// QAT": the A_max estimate is the maximum over a 64-step history window).
// The history is a ring of W + 1 entries (step tag << 32 | binary32 bits of
// that step's amax).  The estimate at step t is the largest amax tagged
// t-W .. t-1 (unsigned tag arithmetic); entry t mod (W+1) then holds a step
// that has left the window, so the CTAs' updates during the step cannot
// change any CTA's estimate.
__device__ float window_estimate(const uint64_t *__restrict__ hist, int32_t W, uint32_t t,
                                 uint32_t *red /* [kThreads / 32] */)
{
    uint32_t m = 0;  // |amax| bits: NaN above infinity above every finite value
    for (int i = threadIdx.x; i <= W; i += blockDim.x) {
        const uint64_t e = hist[i];
        const uint32_t tag = static_cast<uint32_t>(e >> 32);
        if (t - tag - 1u < static_cast<uint32_t>(W))
            m = max(m, static_cast<uint32_t>(e) & 0x7FFFFFFFu);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = m;
    __syncthreads();
    uint32_t a = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); w++)
        a = max(a, red[w]);
    __syncthreads();
    return __uint_as_float(a);
}

// Entry t mod (W+1) := (t, this CTA's amax) unless it already carries tag t
// with a larger amax.  Each failed compare-and-swap means another CTA's
// update landed, so the loop ends after at most grid-size rounds; the bound
// only guards against misuse (the same history shared by concurrent calls).
__device__ void window_record(uint64_t *hist, int32_t W, uint32_t t, uint32_t amax_bits)
{
    unsigned long long *e = reinterpret_cast<unsigned long long *>(hist + t % static_cast<uint32_t>(W + 1));
    const unsigned long long mine = (static_cast<unsigned long long>(t) << 32) | amax_bits;
    unsigned long long old = *reinterpret_cast<volatile unsigned long long *>(e);
    for (int it = 0; it < (1 << 16); it++) {
        if (static_cast<uint32_t>(old >> 32) == t && static_cast<uint32_t>(old) >= amax_bits)
            return;
        const unsigned long long prev = atomicCAS(e, old, mine);
        if (prev == old)
            return;
        old = prev;
    }
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

// max(|a|, |b|, |c|) in one instruction, NaN if any input is NaN (a block
// holding NaN gets the NaN scale byte, as the integer maximum of the BF16
// paths gives).
__device__ __forceinline__ float absmax3f_nan(float a, float b, float c)
{
    float r;
    asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// The same scale and encoders for binary32 block values (the transformed
// blocks): amax over |y| (NaN propagates), codes from y * r with y's sign.
__device__ __forceinline__ BlockScale nvfp4_block_scale_f(float amax, float enc, const float *rtab)
{
    BlockScale bs;
    bs.b = cvt_e4m3(__fmul_rn(amax, enc));
    bs.r = rtab[bs.b];
    return bs;
}

__device__ __forceinline__ uint32_t encode8f_rne(const float *y, float r)
{
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2)
        fmul2(y[i], y[i + 1], r, p[i], p[i + 1]);
    return cvt_e2m1x8(p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7]);
}

__device__ __forceinline__ uint32_t encode8f_sr(const float *y, float r, uint32_t w0, uint32_t w1)
{
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2)
        fmul2(y[i], y[i + 1], r, p[i], p[i + 1]);
    uint16_t lo, hi;
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=h"(lo)
        : "f"(p[3]), "f"(p[2]), "f"(p[1]), "f"(p[0]), "r"(w0));
    asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
        : "=h"(hi)
        : "f"(p[7]), "f"(p[6]), "f"(p[5]), "f"(p[4]), "r"(w1));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// ---------------------------------------------------------------- 1x16

// One lane per 16-element block (32 bytes of input, 8 bytes of codes), four
// blocks in flight per lane (their Philox chains interleave).  With
// stochastic rounding the block's Philox call (counter = offset/16 + block)
// yields one random word per four values.
constexpr int kNvUnroll = 4;

// kDelayed: the per-tensor amax is the Max-Window estimate from `hist` (W, t)
// instead of *amax, and the tensor's own amax is recorded under tag t.  Left
// free, the compiler gives that instance 78 registers (3 CTAs per SM); the
// bound holds it to 64 (4 CTAs per SM, no spills: 55.1 -> 53.4 us with SR on
// 16384 x 7168).  The other instances keep the compiler's choice (48 / 56).
template <bool kSR, bool kDelayed>
__global__ void __launch_bounds__(kThreads, kDelayed ? 4 : 0) nvfp4_quantize_kernel(
    const uint16_t *__restrict__ x, int64_t nblk, const float *__restrict__ amax, uint64_t seed,
    uint64_t offset, uint8_t *__restrict__ q, uint8_t *__restrict__ sb, float *__restrict__ g_out,
    uint64_t *__restrict__ hist, int32_t W, uint32_t t)
{
    __shared__ float rtab[128];
    __shared__ uint32_t red[kThreads / 32];
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
    // the first grid-stride iteration's blocks are requested into L2 before
    // the per-tensor set-up (the amax load, the division, the scale table and
    // a CTA barrier), so that their DRAM latency runs under it (16384 x 7168
    // alone: 1x16 SR 50.3 -> 50.0 us, 16x16 49.2 -> 48.0 us; neutral or
    // slower for the delayed, Hadamard and transposed-operand kernels, which
    // do not issue it)
    if (!kDelayed) {
        const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        const int64_t n = static_cast<int64_t>(gridDim.x) * blockDim.x;
#pragma unroll
        for (int u = 0; u < kNvUnroll; u++)
            if (b + u * n < nblk)
                prefetch_l2(x + (b + u * n) * 16);
    }
    const TensorScales ts = kDelayed ? nvfp4_tensor_setup_from(window_estimate(hist, W, t, red), rtab)
                                     : nvfp4_tensor_setup(amax, rtab);
    uint32_t own = 0;  // max of this thread's block maxima (BF16 bits)
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
            const uint32_t amax16 = hmax_u16x2(m);
            if (kDelayed)
                own = max(own, amax16);
            const BlockScale bs = nvfp4_block_scale(amax16, ts.enc, rtab);
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
    if (kDelayed) {
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
            own = max(own, __shfl_xor_sync(0xffffffffu, own, d));
        if ((threadIdx.x & 31) == 0)
            red[threadIdx.x >> 5] = own;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t a = 0;
            for (int w = 0; w < kThreads / 32; w++)
                a = max(a, red[w]);
            window_record(hist, W, t, a << 16);
        }
    }
}

// 1x16 quantization of the transformed tensor: one lane per block as above,
// rht_unroll(kSR) blocks in flight (their transforms and Philox chains
// interleave; with stochastic rounding two, as four cost occupancy).
__host__ __device__ constexpr int rht_unroll(bool sr) { return sr ? 2 : 4; }

template <bool kSR>
__global__ void __launch_bounds__(kThreads) nvfp4_quantize_rht_kernel(
    const uint16_t *__restrict__ x, int64_t nblk, const float *__restrict__ amax,
    uint32_t sign_mask, uint64_t seed, uint64_t offset, uint8_t *__restrict__ q,
    uint8_t *__restrict__ sb, float *__restrict__ g_out)
{
    __shared__ float rtab[128];
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
    const TensorScales ts = nvfp4_tensor_setup(amax, rtab);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *g_out = ts.g;
    const RhtFlip f = rht_flip_words(sign_mask);
    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    const uint64_t c0 = offset >> 4;
    constexpr int kU = rht_unroll(kSR);
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;

    for (int64_t b0 = gtid; b0 < nblk; b0 += kU * nthr) {
        uint4 v[kU][2];
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int64_t blk = b0 + u * nthr;
            if (blk < nblk) {
                v[u][0] = ld_nc_v4(x + blk * 16);
                v[u][1] = ld_nc_v4(x + blk * 16 + 8);
            } else {
                v[u][0] = v[u][1] = make_uint4(0, 0, 0, 0);
            }
        }
        if (kSR) {
            // with stochastic rounding the arithmetic below keeps each warp
            // busy long enough that its next loads start late: the next
            // iteration's blocks are requested into L2 now (no registers
            // held; round to nearest is bound by HBM and gains nothing)
#pragma unroll
            for (int u = 0; u < kU; u++) {
                const int64_t nb = b0 + (kU + u) * nthr;
                if (nb < nblk)
                    prefetch_l2(x + nb * 16);
            }
        }
#pragma unroll
        for (int u = 0; u < kU; u++) {
            const int64_t blk = b0 + u * nthr;
            if (blk >= nblk)
                break;
            float y[16];
            rht16(v[u][0], v[u][1], f, y);
            float a = 0.0f;  // max |y|, NaN if the block holds NaN
#pragma unroll
            for (int i = 0; i < 16; i += 2)
                a = absmax3f_nan(a, y[i], y[i + 1]);
            const BlockScale bs = nvfp4_block_scale_f(a, ts.enc, rtab);
            uint2 codes;
            if (kSR) {
                const uint64_t c = c0 + static_cast<uint64_t>(blk);
                const uint4 w = philox4x32_10(
                    make_uint4(static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32), 0u, 0u),
                    k0, k1);
                codes.x = encode8f_sr(y, bs.r, w.x, w.y);
                codes.y = encode8f_sr(y + 8, bs.r, w.z, w.w);
            } else {
                codes.x = encode8f_rne(y, bs.r);
                codes.y = encode8f_rne(y + 8, bs.r);
            }
            __stcs(reinterpret_cast<uint2 *>(q + blk * 8), codes);
            sb[blk] = static_cast<uint8_t>(bs.b);
        }
    }
}

// ---------------------------------------------------------------- 16x16

// One warp's share of the 2D quantization: the 16-row strip `strip` x 256
// columns from `col0`, lane l holding columns col0 + 8l .. + 7 of all 16 rows
// (lanes 2t, 2t+1 form tile t), so every row load / store of the warp is
// 512 / 128 contiguous bytes.  Writes the strip's codes and tile scales and
// returns them (c[r] = the lane's eight codes of row r) for the caller.
__device__ __forceinline__ uint32_t nvfp4_2d_strip(const uint16_t *__restrict__ w, int64_t K,
                                                   int64_t strip, int64_t col, bool ok,
                                                   const TensorScales &ts, const float *rtab,
                                                   uint8_t *__restrict__ q,
                                                   uint8_t *__restrict__ sb, uint32_t c[16])
{
    const int lane = threadIdx.x & 31;
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
        for (int r = 0; r < 16; r++) {
            c[r] = encode8_rne(v[r], bs.r);
            __stcs(reinterpret_cast<unsigned int *>(dst + r * (K >> 1)), c[r]);
        }
        if (!(lane & 1))
            sb[strip * (K >> 4) + (col >> 4)] = static_cast<uint8_t>(bs.b);
    }
    return bs.b;
}

__global__ void __launch_bounds__(kThreads, 2) nvfp4_quantize_2d_kernel(
    const uint16_t *__restrict__ w, int64_t N, int64_t K, const float *__restrict__ amax,
    uint8_t *__restrict__ q, uint8_t *__restrict__ sb, float *__restrict__ g_out)
{
    __shared__ float rtab[128];
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up

    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t ncg = (K + 255) >> 8;  // 256-column groups
    const int64_t nunits = (N >> 4) * ncg;
    if (warp < nunits) {  // the warp's first strip, requested as in the 1x16 kernel
        const int64_t strip = warp / ncg;
        const int64_t col = ((warp - strip * ncg) << 8) + 8 * lane;
        if (col < K)
            for (int r = 0; r < 16; r++)
                prefetch_l2(w + ((strip << 4) + r) * K + col);
    }
    const TensorScales ts = nvfp4_tensor_setup(amax, rtab);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *g_out = ts.g;

    for (int64_t unit = warp; unit < nunits; unit += nwarps) {
        const int64_t strip = unit / ncg;
        const int64_t col = ((unit - strip * ncg) << 8) + 8 * lane;
        uint32_t c[16];
        nvfp4_2d_strip(w, K, strip, col, col < K, ts, rtab, q, sb, c);
    }
}

// Transpose of an 8 x 8 matrix of nibbles held as eight words (A[i] nibble j
// = M[i][j] -> A[j] nibble i = M[i][j]): the off-diagonal 4 x 4 and then 2 x 2
// blocks swap with byte permutes, the 1 x 1 blocks with a masked exchange.
__device__ __forceinline__ void transpose_nibbles8x8(uint32_t A[8])
{
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const uint32_t a = A[i], b = A[i + 4];
        A[i] = prmt(a, b, 0x5410u);
        A[i + 4] = prmt(a, b, 0x7632u);
    }
#pragma unroll
    for (int i = 0; i < 8; i += (i & 1) ? 3 : 1) {  // i = 0, 1, 4, 5
        const uint32_t a = A[i], b = A[i + 2];
        A[i] = prmt(a, b, 0x6240u);
        A[i + 2] = prmt(a, b, 0x7351u);
    }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint32_t t = ((A[i] >> 4) ^ A[i + 1]) & 0x0F0F0F0Fu;
        A[i] ^= t << 4;
        A[i + 1] ^= t;
    }
}

// With the DGRAD operand W^T (the same codes and 16 x 16 scales, transposed).
// A CTA unit is 8 consecutive strips (warp w: strip 8 sg + w) x one 256-column
// group, i.e. a 128 x 256 block of W and a 256 x 128 block of W^T.  Each warp
// quantizes its strip as above, transposes its lane's 16 x 8 codes in
// registers (two 8 x 8 nibble transposes) and leaves the lane's eight W^T rows
// (8 bytes each) in a shared tile of 256 rows x 64 bytes; the CTA then writes
// every W^T row's 64 bytes with four 16-byte stores.  Tile slot (row, strip)
// is stored at 2-word slot strip ^ ((row / 8) & 7), so the eight strips'
// writes of one row phase spread over the banks.
constexpr int kT2Strips = kThreads / 32;  // 8
constexpr int kT2Rows = 256;              // W^T rows (columns of W) per unit

__global__ void __launch_bounds__(kThreads, 2) nvfp4_quantize_2d_t_kernel(
    const uint16_t *__restrict__ w, int64_t N, int64_t K, const float *__restrict__ amax,
    uint8_t *__restrict__ q, uint8_t *__restrict__ sb, uint8_t *__restrict__ qT,
    uint8_t *__restrict__ sbT, float *__restrict__ g_out)
{
    __shared__ float rtab[128];
    __shared__ __align__(16) uint32_t tile[kT2Rows * 2 * kT2Strips];  // 16 KB
    __shared__ uint8_t stile[16 * kT2Strips];  // [tile column][strip]
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the next kernel may start its set-up
    const TensorScales ts = nvfp4_tensor_setup(amax, rtab);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *g_out = ts.g;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t nstrips = N >> 4;
    const int64_t nsg = (nstrips + kT2Strips - 1) / kT2Strips;
    const int64_t ncg = (K + 255) >> 8;
    const int64_t nunits = nsg * ncg;
    const int64_t rowT = N >> 1;  // bytes per W^T row

    for (int64_t unit = blockIdx.x; unit < nunits; unit += gridDim.x) {
        const int64_t sg = unit / ncg, cg = unit - sg * ncg;
        const int64_t strip = sg * kT2Strips + wid;
        const int64_t col = (cg << 8) + 8 * lane;
        const bool ok = strip < nstrips && col < K;
        uint32_t c[16];
        const uint32_t b = nvfp4_2d_strip(w, K, strip, col, ok, ts, rtab, q, sb, c);
        if (ok) {
            transpose_nibbles8x8(c);
            transpose_nibbles8x8(c + 8);
            // W^T row col + j: codes of strip rows 0..7 in the low word, 8..15 high
            const int slot = 2 * (wid ^ (lane & 7));
#pragma unroll
            for (int j = 0; j < 8; j++)
                *reinterpret_cast<uint2 *>(&tile[(8 * lane + j) * 16 + slot]) =
                    make_uint2(c[j], c[8 + j]);
            if (!(lane & 1))
                stile[(lane >> 1) * kT2Strips + wid] = static_cast<uint8_t>(b);
        }
        __syncthreads();
        const int rows = static_cast<int>(min(static_cast<int64_t>(kT2Rows), K - (cg << 8)));
        const int strips = static_cast<int>(min(static_cast<int64_t>(kT2Strips), nstrips - sg * kT2Strips));
        // four threads per W^T row, 16 bytes (strips 2p, 2p + 1) each
        const int p = tid & 3;
#pragma unroll
        for (int i = 0; i < kT2Rows / (kThreads / 4); i++) {
            const int r = (tid >> 2) + i * (kThreads / 4);
            if (r < rows && 2 * p < strips) {
                const int x = (r >> 3) & 7;
                const uint2 lo = *reinterpret_cast<const uint2 *>(&tile[r * 16 + 2 * ((2 * p) ^ x)]);
                uint8_t *dst = qT + ((cg << 8) + r) * rowT + sg * 64 + 16 * p;
                if (2 * p + 1 < strips) {
                    const uint2 hi =
                        *reinterpret_cast<const uint2 *>(&tile[r * 16 + 2 * ((2 * p + 1) ^ x)]);
                    if (!(rowT & 15)) {
                        __stcs(reinterpret_cast<uint4 *>(dst), make_uint4(lo.x, lo.y, hi.x, hi.y));
                    } else {
                        __stcs(reinterpret_cast<uint2 *>(dst), lo);
                        __stcs(reinterpret_cast<uint2 *>(dst + 8), hi);
                    }
                } else {
                    __stcs(reinterpret_cast<uint2 *>(dst), lo);
                }
            }
        }
        // tile scales of W^T: row (16 cg + j) gets the unit's strips
        if (tid < 16 * kT2Strips) {
            const int j = tid / kT2Strips, s2 = tid % kT2Strips;
            if (16 * j < rows && s2 < strips)
                sbT[((cg << 4) + j) * (N >> 4) + sg * kT2Strips + s2] = stile[j * kT2Strips + s2];
        }
        __syncthreads();  // the tile is rewritten by the next unit
    }
}

// The amax word zeroed by one thread, in the chain of programmatically
// dependent launches (the kernel before may still read or write it until
// griddepcontrol.wait returns).
__global__ void zero_word_kernel(uint32_t *__restrict__ w)
{
    griddep_wait();
    griddep_launch_dependents();
    *w = 0u;
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
    if (launch_pdl(zero_word_kernel, dim3(1), dim3(1), 0, st, reinterpret_cast<uint32_t *>(amax)) !=
        cudaSuccess)
        return launch_status();
    if (n == 0)
        return launch_status();
    const int64_t work = (n / 8 + 4 * kThreads - 1) / (4 * kThreads);
    const int grid = persistent_grid(nvfp4_amax_kernel, kThreads, 0, work < 1 ? 1 : work);
    launch_pdl(nvfp4_amax_kernel, dim3(grid), dim3(kThreads), 0, st,
               static_cast<const uint16_t *>(x), n, reinterpret_cast<uint32_t *>(amax));
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
    auto kern = use_sr ? nvfp4_quantize_kernel<true, false> : nvfp4_quantize_kernel<false, false>;
    const int grid = persistent_grid(kern, kThreads, 0, work, 2);
    launch_pdl(kern, dim3(grid), dim3(kThreads), 0, st, static_cast<const uint16_t *>(x), nblk,
               amax, seed, offset, q, sb, g, static_cast<uint64_t *>(nullptr), 0, 0u);
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
        persistent_grid(nvfp4_quantize_2d_kernel, kThreads, 0, (units + 7) / 8, 2);
    launch_pdl(nvfp4_quantize_2d_kernel, dim3(grid), dim3(kThreads), 0,
               static_cast<cudaStream_t>(stream), static_cast<const uint16_t *>(w), N, K, amax, q, sb,
               g);
    return launch_status();
}

extern "C" fq_status nvfp4_quantize_2d_t(const void *w, int64_t N, int64_t K, const float *amax,
                                         uint8_t *q, uint8_t *sb, uint8_t *qT, uint8_t *sbT,
                                         float *g, void *stream)
{
    if (N < 0 || K <= 0 || N % 16 != 0 || K % 16 != 0)
        return FQ_ERR_SHAPE;
    if (N > 0 && K > INT64_MAX / N)
        return FQ_ERR_SHAPE;
    if (N == 0)
        return FQ_OK;
    if (!w || !amax || !q || !sb || !qT || !sbT || !g)
        return FQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(amax) || !aligned16(q) || !aligned16(sb) || !aligned16(qT) ||
        !aligned16(sbT) || !aligned16(g))
        return FQ_ERR_ALIGN;
    const int64_t units = ((N / 16 + kT2Strips - 1) / kT2Strips) * ((K + 255) / 256);
    const int grid = persistent_grid(nvfp4_quantize_2d_t_kernel, kThreads, 0, units, 2);
    launch_pdl(nvfp4_quantize_2d_t_kernel, dim3(grid), dim3(kThreads), 0,
               static_cast<cudaStream_t>(stream), static_cast<const uint16_t *>(w), N, K, amax, q,
               sb, qT, sbT, g);
    return launch_status();
}

extern "C" fq_status nvfp4_amax_rht(const void *x, int64_t n, uint32_t sign_mask, float *amax,
                                    void *stream)
{
    if (n < 0 || n % 16 != 0)
        return FQ_ERR_SHAPE;
    if (!amax || (n > 0 && !x))
        return FQ_ERR_NULL;
    if ((n > 0 && !aligned16(x)) || !aligned16(amax))
        return FQ_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (launch_pdl(zero_word_kernel, dim3(1), dim3(1), 0, st, reinterpret_cast<uint32_t *>(amax)) !=
        cudaSuccess)
        return launch_status();
    if (n == 0)
        return launch_status();
    const int64_t nblk = n / 16;
    const int64_t work = (nblk + 2 * kThreads - 1) / (2 * kThreads);
    const int grid = persistent_grid(nvfp4_amax_rht_kernel, kThreads, 0, work);
    launch_pdl(nvfp4_amax_rht_kernel, dim3(grid), dim3(kThreads), 0, st,
               static_cast<const uint16_t *>(x), nblk, rht_flip_bits(sign_mask & 0xFFFFu),
               reinterpret_cast<uint32_t *>(amax));
    return launch_status();
}

extern "C" fq_status nvfp4_quantize_rht(const void *x, int64_t M, int64_t K, const float *amax,
                                        uint32_t sign_mask, int use_sr, uint64_t seed,
                                        uint64_t offset, uint8_t *q, uint8_t *sb, float *g,
                                        void *stream)
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
    const int u = rht_unroll(use_sr != 0);
    const int64_t work = (nblk + u * kThreads - 1) / (u * kThreads);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint32_t mask = sign_mask & 0xFFFFu;
    if (use_sr) {
        const int grid = persistent_grid(nvfp4_quantize_rht_kernel<true>, kThreads, 0, work, 2);
        launch_pdl(nvfp4_quantize_rht_kernel<true>, dim3(grid), dim3(kThreads), 0, st,
                   static_cast<const uint16_t *>(x), nblk, amax, mask, seed, offset, q, sb, g);
    } else {
        const int grid = persistent_grid(nvfp4_quantize_rht_kernel<false>, kThreads, 0, work, 2);
        launch_pdl(nvfp4_quantize_rht_kernel<false>, dim3(grid), dim3(kThreads), 0, st,
                   static_cast<const uint16_t *>(x), nblk, amax, mask, seed, offset, q, sb, g);
    }
    return launch_status();
}

extern "C" fq_status nvfp4_quantize_delayed(const void *x, int64_t M, int64_t K,
                                            uint64_t *amax_history, int32_t window, uint32_t step,
                                            int use_sr, uint64_t seed, uint64_t offset, uint8_t *q,
                                            uint8_t *sb, float *g, void *stream)
{
    if (M < 0 || K <= 0 || K % 16 != 0)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (window < 1 || window > FQ_AMAX_WINDOW_MAX || offset % 16 != 0 ||
        (use_sr != 0 && use_sr != 1))
        return FQ_ERR_ARG;
    if (M == 0)
        return FQ_OK;
    if (!x || !amax_history || !q || !sb || !g)
        return FQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(amax_history) || !aligned16(q) || !aligned16(sb) ||
        !aligned16(g))
        return FQ_ERR_ALIGN;
    const int64_t nblk = M * (K / 16);
    const int64_t work = (nblk + kNvUnroll * kThreads - 1) / (kNvUnroll * kThreads);
    auto kern = use_sr ? nvfp4_quantize_kernel<true, true> : nvfp4_quantize_kernel<false, true>;
    const int grid = persistent_grid(kern, kThreads, 0, work);
    launch_pdl(kern, dim3(grid), dim3(kThreads), 0, static_cast<cudaStream_t>(stream),
               static_cast<const uint16_t *>(x), nblk, static_cast<const float *>(nullptr), seed,
               offset, q, sb, g, amax_history, window, step);
    return launch_status();
}
