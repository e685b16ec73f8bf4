// Device helpers shared by the cast kernels of libfq.so (sm_103a only).
//
// Conversions use the PTX packed conversion instructions (cvt ... e2m1x2,
// e4m3x2) whose rounding is round-to-nearest-even with saturation to the
// largest finite value; the tests check their outputs against the CPU
// oracle over every input the kernels can feed them.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fq.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libfq.so is written for sm_103a (Blackwell Ultra); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace fq {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- host side

// Records the CUDA error of a failed launch for fq_last_cuda_error().
void set_last_cuda_error(int err);
// SM count of the current device (cached per device).
int sm_count();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline fq_status launch_status()
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_last_cuda_error(static_cast<int>(e));
        return FQ_ERR_CUDA;
    }
    return FQ_OK;
}

// Launch with programmatic stream serialization (the kernel may start while
// the previous one on the stream finishes; it synchronises with griddep_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Grid of `waves` times the CTAs that fill every SM at the kernel's
// occupancy, never more than there is work for.  One wave is a persistent
// grid.  For the grid-stride streaming kernels, two or four waves are faster
// on GB300: each CTA then takes a smaller share, and SM slots are refilled as
// CTAs finish.  With one wave, the warp schedulers favour an SM's oldest CTAs,
// and its last-launched CTAs trail at the end with the SM part empty.
template <typename Kernel>
inline int persistent_grid(Kernel kernel, int threads, size_t smem, int64_t work_ctas,
                           int waves = 1)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    int64_t g = static_cast<int64_t>(sm_count()) * per_sm * waves;
    if (work_ctas < g)
        g = work_ctas;
    return static_cast<int>(g < 1 ? 1 : g);
}

// ---------------------------------------------------------------- device side

// BF16 halves of a 32-bit word as FP32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Element-wise max of two packed u16 pairs.  Applied to BF16 words with the
// sign bits cleared, this is |x| max in which Inf (0x7F80) and NaN (above
// 0x7F80) are the largest values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w)
{
    return max_u16x2(acc, w & 0x7FFF7FFFu);
}

// Larger of the two u16 halves.
__device__ __forceinline__ uint32_t hmax_u16x2(uint32_t w)
{
    uint32_t lo = w & 0xFFFFu, hi = w >> 16;
    return lo > hi ? lo : hi;
}

// Eight FP32 values -> eight E2M1 codes in one word, value i in bits 4i..4i+3.
// cvt ... e2m1x2 puts its first source in the high nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                               float v5, float v6, float v7)
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
    return r;
}

// Non-negative FP32 -> E4M3 byte (round to nearest even, saturating at 448).
__device__ __forceinline__ uint32_t cvt_e4m3(float t)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
    return static_cast<uint32_t>(r) & 0xFFu;
}

// E4M3 magnitude of code b (0..126) as FP32, exact.
__device__ __forceinline__ float e4m3_value(uint32_t b)
{
    uint32_t E = b >> 3, m = b & 7u;
    if (E == 0)
        return __uint2float_rn(m) * 0x1p-9f;
    return __uint_as_float((b + 960u) << 20);  // exponent field E - 7 + 127
}

// Two IEEE binary32 products (round to nearest) in one packed instruction.
__device__ __forceinline__ void fmul2(float a0, float a1, float b, float &r0, float &r1)
{
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %4};\n\t"
        "mul.rn.f32x2 z, x, y;\n\t"
        "mov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b));
}

// Byte permute (prmt.b32): result byte i chosen by selector nibble i from the
// eight bytes {b:a}; a selector with bit 3 set replicates that byte's msb.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Eight E2M1 codes (one word, code i in bits 4i..4i+3) -> eight E4M3 bytes
// through an 8-entry magnitude table {t1:t0}; the sign of each code becomes
// bit 7 of its byte where `sign_mask` is 0x80808080 (0 keeps the table bytes
// as they are, e.g. the all-NaN row).
__device__ __forceinline__ void fp4x8_to_fp8x8(uint32_t w, uint32_t t0, uint32_t t1,
                                               uint32_t &lo, uint32_t &hi,
                                               uint32_t sign_mask = 0x80808080u)
{
    const uint32_t sel = w & 0x77777777u;
    const uint32_t w4 = w << 4;
    const uint32_t mlo = prmt(t0, t1, sel);
    const uint32_t mhi = prmt(t0, t1, sel >> 16);
    const uint32_t slo = prmt(w4, w, 0xD9C8u);  // msb of codes 0..3 replicated
    const uint32_t shi = prmt(w4, w, 0xFBEAu);  // msb of codes 4..7 replicated
    lo = mlo | (slo & sign_mask);
    hi = mhi | (shi & sign_mask);
}

// FP32 bits of the FP8 block scale 2^(S - 127 - k); NaN for S = 0xFF.
__device__ __forceinline__ uint32_t fp8_block_scale_bits(uint32_t S, int k)
{
    if (S == 0xFFu)
        return 0x7FC00000u;
    int ex = static_cast<int>(S) - k;  // biased exponent of the result, >= -6
    if (ex >= 1)
        return static_cast<uint32_t>(ex) << 23;
    return 1u << (ex + 22);  // binary32 subnormal 2^(ex - 127)
}

// Table of E4M3 bytes for E2M1 magnitude code c (0..7) shifted by 2^(6-u),
// u = 0..19 (u = 19 covers every larger shift: all values flush to zero),
// plus row kNanRow of 0x7F (the E4M3 NaN) for blocks whose scale is NaN.
constexpr int kShiftRows = 20;
constexpr int kNanRow = kShiftRows;
constexpr int kTabRows = kShiftRows + 1;
__device__ __forceinline__ void build_fp8_table(uint8_t *tab /* [kTabRows * 8] */)
{
    for (int i = threadIdx.x; i < kTabRows * 8; i += blockDim.x) {
        int u = i >> 3, c = i & 7;
        if (u == kNanRow) {
            tab[i] = 0x7F;
            continue;
        }
        // E2M1 magnitude of c times 2^(6 - u), built exactly from bits
        float v;
        if (c == 0)
            v = 0.0f;
        else if (c == 1)
            v = 0.5f;
        else
            v = __uint_as_float(((126u + (c >> 1)) << 23) | ((c & 1u) << 22));
        v *= __uint_as_float(static_cast<uint32_t>(127 + 6 - u) << 23);
        tab[i] = static_cast<uint8_t>(cvt_e4m3(v));
    }
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream is still
// running; it must read nothing that kernel writes, and write nothing,
// before griddep_wait() returns (a hardware wait for that grid's
// completion; a no-op for a normal launch).  griddep_launch_dependents()
// lets the next such kernel start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- TMA and mbarriers

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes initialised mbarriers visible to the tensor-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::
                     : "memory");
}

// One arrival that also announces `bytes` of tensor-copy data.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Waits for phase `parity` of the barrier to complete; gives up (returns
// false) after about two seconds so that a lost copy cannot hang the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > kWaitLimitNs)
            return false;
    return true;
}

// 2D tiled tensor copy global -> shared, completing on `bar` (x is the
// innermost coordinate in elements; x * element size must be a multiple of
// 16 bytes; rows outside the tensor read as zero).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Asynchronous 4-byte copy global -> shared (cp.async); with `src_bytes` 0
// nothing is read and the 4 bytes are zero-filled.
__device__ __forceinline__ void cp_async_4(void *dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
                 : "memory");
}

// One arrival on `bar` once every cp.async this thread issued so far has
// landed (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Barrier `id` over the first `count` threads of the CTA (a multiple of 32)
// that also ORs a predicate across them.
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
                 : "memory");
    return r != 0;
}

// Host: launchers shared by the entry points (arguments already checked).
// MXFP4 rows; with y != nullptr also the FP8 rows of the fresh codes.
fq_status launch_mxfp4_rows(const void *x, int64_t M, int64_t K, uint8_t *q, uint8_t *s, int k,
                            uint8_t *y, float *ys, cudaStream_t st);
// FP4 -> FP8 transposed conversion on ragged groups.
fq_status launch_fp4_to_fp8_cols(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K,
                                 const int64_t *group_offsets, int32_t G, int k, uint8_t *yT,
                                 float *yT_scale, int64_t cap, int32_t *dev_status,
                                 cudaStream_t st);

// Host: encoder of tensor maps (driver entry point, looked up once).
// Returns false if the driver does not provide it.  promote_l2: fill whole
// 128-byte L2 lines on a miss (for boxes whose neighbouring bytes are read
// soon); otherwise only the 32-byte sectors the box touches are fetched.
bool encode_tensor_map_2d_u8(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                             uint64_t row_pitch, uint32_t box_inner, uint32_t box_rows,
                             bool promote_l2 = true);
// The same for any element type and shared-memory swizzle (inner, box_inner
// in elements; row_pitch in bytes).
bool encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t rows, uint64_t row_pitch, uint32_t box_inner,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle, bool promote_l2);

// Philox4x32-10 (Salmon et al., SC'11).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int i = 0; i < 10; i++) {
        if (i) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// Requests the line holding p into L2 (no registers held, nothing returned).
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 ld_nc_v4(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// ---------------------------------------------------------------- L2 eviction policies

// Lines touched with evict_last stay in L2 ahead of other lines (data the next
// kernel reads back); evict_first lines leave first (streamed data).
__device__ __forceinline__ uint64_t l2_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_nc_v4_hint(const void *p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_u32_hint(void *p, uint32_t v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_u8_hint(void *p, uint32_t v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.b8 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol)
                 : "memory");
}

}  // namespace fq
