// Direct FP4 -> FP8 conversion fused with the transpose, on ragged
// per-expert token groups (FP4RowToFP8Col).
//
// Source: "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// technical overview section 2, item 3 -- layout-aware kernels: the weight
// gradient operand is transposed and converted in one pass without a global
// round trip, the transpose goes through a padded (skewed) shared-memory
// layout to avoid bank conflicts, and ragged expert groups are handled
// without padding.  Scale alignment as in the row conversion (item 1).
//
// Design (GB300): persistent CTAs walk output tiles of 128 features x 128
// tokens.  Tiles are aligned to 128 tokens of the OUTPUT (so every output row
// segment is a full, aligned 128-byte line), not to the groups: a tile may
// cut through several 128-token blocks of several groups, whose scale maxima
// are reduced from a staged window of scale words.  The next tile's codes and
// scale words are prefetched into registers while the current tile is
// written out.
#include <cstddef>

#include "fq_common.cuh"

namespace fq {

constexpr int kTok = 128;                // tokens per tile (output columns)
constexpr int kQuadWords = 132;          // 128 words + 4 pad per 4-token group
constexpr int kStage = 384;              // scale words staged: tokens [W-128, W+256)

struct __align__(16) ColsTileSmem {
    __align__(16) uint32_t tile[(kTok / 4) * kQuadWords];  // FP8 bytes, [token/4][kword][token%4]
    uint32_t sw[kStage];                     // scale words (4 MX columns) of staged tokens
    uint32_t smax[kTok];                     // per block: byte j = max exponent of column j
    int32_t rel[kTok];                       // window token -> block index within the tile
    int32_t bstart[kTok], bend[kTok], bslot[kTok];
    int32_t nblocks;
    __align__(16) uint8_t tab[kShiftRows * 8];
};
static_assert(offsetof(ColsTileSmem, tile) % 16 == 0, "tile is read with 128-bit loads");
static_assert(offsetof(ColsTileSmem, tab) % 16 == 0, "table rows are read with 64-bit loads");

// Largest g in [lo, hi] with off[g] <= t (off non-decreasing, off[lo] <= t).
__device__ __forceinline__ int find_group(const int32_t *off, int lo, int hi, int32_t t)
{
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// In-place inclusive scan (max or sum) of a[0..n) in shared memory by the
// whole CTA; n <= 4 * 1024 + 1 is enough here.
template <bool kMax>
__device__ void cta_scan(int32_t *a, int n, int32_t *warp_tot /* [kThreads/32] */)
{
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = threadIdx.x * per, hi = min(lo + per, n);
    int32_t run = kMax ? INT32_MIN : 0;
    for (int i = lo; i < hi; i++) {
        run = kMax ? max(run, a[i]) : run + a[i];
        a[i] = run;
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int32_t incl = run;
    for (int d = 1; d < 32; d <<= 1) {
        int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d)
            incl = kMax ? max(incl, o) : incl + o;
    }
    if (lane == 31)
        warp_tot[wid] = incl;
    __syncthreads();
    int32_t before = kMax ? INT32_MIN : 0;
    for (int w = 0; w < wid; w++)
        before = kMax ? max(before, warp_tot[w]) : before + warp_tot[w];
    int32_t excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane > 0)
        before = kMax ? max(before, excl) : before + excl;
    for (int i = lo; i < hi; i++)
        a[i] = kMax ? max(before, a[i]) : before + a[i];
    __syncthreads();
}

// 4x4 byte transpose: in = four words (rows), out[r] = byte r of each word.
__device__ __forceinline__ void transpose4x4(uint4 v, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                             uint32_t &r3)
{
    const uint32_t ab_lo = prmt(v.x, v.y, 0x5140u), ab_hi = prmt(v.x, v.y, 0x7362u);
    const uint32_t cd_lo = prmt(v.z, v.w, 0x5140u), cd_hi = prmt(v.z, v.w, 0x7362u);
    r0 = prmt(ab_lo, cd_lo, 0x5410u);
    r1 = prmt(ab_lo, cd_lo, 0x7632u);
    r2 = prmt(ab_hi, cd_hi, 0x5410u);
    r3 = prmt(ab_hi, cd_hi, 0x7632u);
}

template <bool kAligned4>
__global__ void __launch_bounds__(kThreads, 4) fp4_to_fp8_cols_kernel(
    const uint8_t *__restrict__ q, const uint8_t *__restrict__ s, int32_t M, int64_t K,
    const int64_t *__restrict__ offs, int32_t G, int k, uint8_t *__restrict__ yT,
    float *__restrict__ yTs, int64_t cap, int32_t *__restrict__ dev_status)
{
    __shared__ ColsTileSmem sm;
    __shared__ int32_t warp_tot[kThreads / 32];
    extern __shared__ int32_t dyn[];
    int32_t *off = dyn;           // [G+1] clamped, monotone group offsets
    int32_t *base = dyn + G + 1;  // [G+1] first scale slot of each group

    const int tid = threadIdx.x;
    build_fp8_table(sm.tab);

    // ---- group structure (once per CTA): clamp, make monotone, count blocks
    int bad = 0;
    for (int i = tid; i <= G; i += kThreads) {
        const int64_t o = offs[i];
        const int64_t c = o < 0 ? 0 : (o > M ? M : o);
        off[i] = static_cast<int32_t>(c);
        if (c != o || (i == 0 && o != 0) || (i == G && o != M) || (i > 0 && o < offs[i - 1]))
            bad = 1;
    }
    bad = __syncthreads_or(bad);
    if (bad && blockIdx.x == 0 && tid == 0 && dev_status)
        atomicOr(dev_status, 1);
    cta_scan<true>(off, G + 1, warp_tot);
    if (tid == 0) {
        off[0] = 0;
        off[G] = M;
    }
    __syncthreads();
    for (int g = tid; g <= G; g += kThreads)
        base[g] = g == 0 ? 0 : (off[g] - off[g - 1] + kTok - 1) / kTok;
    __syncthreads();
    cta_scan<false>(base, G + 1, warp_tot);  // base[g] = blocks of groups < g

    const int32_t nwin = (M + kTok - 1) / kTok;
    const int32_t nfeat = static_cast<int32_t>(K / 128);
    const int64_t ntiles = static_cast<int64_t>(nwin) * nfeat;
    const int64_t qrow = K / 2, srow = K / 32;

    // prefetch: unit u = tid + 256*r (r = 0, 1): token tl = u & 127, column
    // block j = u >> 7 -> 16 bytes of q; staged scale words tokens W-128+tid
    // and W+128+tid.
    uint4 qv[2];
    uint32_t sv[2];
    auto prefetch = [&](int64_t tau) {
        const int32_t win = static_cast<int32_t>(tau % nwin);
        const int32_t f = static_cast<int32_t>(tau / nwin);
        const int32_t W = win * kTok;
#pragma unroll
        for (int r = 0; r < 2; r++) {
            const int u = tid + kThreads * r;
            const int32_t t = W + (u & 127);
            qv[r] = t < M ? ld_nc_v4(q + t * qrow + f * 64 + 16 * (u >> 7)) : make_uint4(0, 0, 0, 0);
            const int32_t ts = W - 128 + tid + 256 * r;
            sv[r] = (r == 0 || tid < 128) && ts >= 0 && ts < M
                        ? __ldg(reinterpret_cast<const uint32_t *>(s + ts * srow + 4 * f))
                        : 0u;
        }
    };

    int64_t tau = blockIdx.x;
    if (tau < ntiles)
        prefetch(tau);
    for (; tau < ntiles; tau += gridDim.x) {
        const int32_t win = static_cast<int32_t>(tau % nwin);
        const int32_t f = static_cast<int32_t>(tau / nwin);
        const int32_t W = win * kTok;
        const int32_t We = min(W + kTok, M);

        // ---- stage scale words; find the groups at both ends of the window
        sm.sw[tid] = sv[0];
        if (tid < 128)
            sm.sw[256 + tid] = sv[1];
        const int g_first = find_group(off, 0, G - 1, W);
        const int g_last = find_group(off, g_first, G - 1, We - 1);
        const int32_t slot_lo = base[g_first] + (W - off[g_first]) / kTok;
        __syncthreads();

        // ---- every window token: its block; blocks starting here (or at W)
        if (tid < kTok) {
            const int32_t t = W + tid;
            if (t < We) {
                const int g = g_first == g_last ? g_first : find_group(off, g_first, g_last, t);
                const int32_t bl = (t - off[g]) / kTok;
                const int32_t r = base[g] + bl - slot_lo;
                sm.rel[tid] = r;
                const int32_t start = off[g] + bl * kTok;
                if (t == W || t == start) {
                    sm.bstart[r] = start;
                    sm.bend[r] = min(start + kTok, off[g + 1]);
                    sm.bslot[r] = base[g] + bl;
                }
                if (t == We - 1)
                    sm.nblocks = r + 1;
            }
        }
        __syncthreads();

        // ---- per block: byte-wise max of the staged scale words (warp per block)
        {
            const int lane = tid & 31, wid = tid >> 5;
            const int nb = sm.nblocks;
            for (int r = wid; r < nb; r += kThreads / 32) {
                const int32_t a = sm.bstart[r], b = sm.bend[r];
                uint32_t even = 0, odd = 0;  // bytes 0,2 and 1,3 as u16 pairs
                for (int32_t t = a + lane; t < b; t += 32) {
                    const uint32_t w = sm.sw[t - (W - 128)];
                    even = max_u16x2(even, w & 0x00FF00FFu);
                    odd = max_u16x2(odd, (w >> 8) & 0x00FF00FFu);
                }
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) {
                    even = max_u16x2(even, __shfl_xor_sync(0xffffffffu, even, d));
                    odd = max_u16x2(odd, __shfl_xor_sync(0xffffffffu, odd, d));
                }
                if (lane == 0)
                    sm.smax[r] = even | (odd << 8);
            }
        }
        __syncthreads();

        // ---- convert the prefetched codes into the shared FP8 tile
#pragma unroll
        for (int rr = 0; rr < 2; rr++) {
            const int u = tid + kThreads * rr;
            const int tl = u & 127, j = u >> 7;
            if (W + tl < We) {
                const uint32_t Sw = sm.smax[sm.rel[tl]];
                const uint32_t S = (Sw >> (8 * j)) & 0xFFu;
                const uint32_t e = (sm.sw[tl + 128] >> (8 * j)) & 0xFFu;
                int uu = static_cast<int>(S - e) - k + 6;
                uu = uu < kShiftRows - 1 ? uu : kShiftRows - 1;
                const uint2 t = *reinterpret_cast<const uint2 *>(sm.tab + 8 * uu);
                uint32_t o[8];
                fp4x8_to_fp8x8(qv[rr].x, t.x, t.y, o[0], o[1]);
                fp4x8_to_fp8x8(qv[rr].y, t.x, t.y, o[2], o[3]);
                fp4x8_to_fp8x8(qv[rr].z, t.x, t.y, o[4], o[5]);
                fp4x8_to_fp8x8(qv[rr].w, t.x, t.y, o[6], o[7]);
                uint32_t *dst = sm.tile + (tl >> 2) * kQuadWords + 32 * j + (tl & 3);
#pragma unroll
                for (int w = 0; w < 8; w++)
                    dst[4 * w] = S == 0xFFu ? 0x7F7F7F7Fu : o[w];
            }
        }
        __syncthreads();

        // ---- prefetch the next tile, then write this one out
        if (tau + gridDim.x < ntiles)
            prefetch(tau + gridDim.x);
        {
            const int lane = tid & 31, wid = tid >> 5;
            const int32_t t0 = W + 4 * lane;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int m = wid + 8 * i;  // word of 4 features
                const uint4 v = *reinterpret_cast<const uint4 *>(sm.tile + lane * kQuadWords + 4 * m);
                uint32_t r[4];
                transpose4x4(v, r[0], r[1], r[2], r[3]);
#pragma unroll
                for (int rr = 0; rr < 4; rr++) {
                    uint8_t *dst = yT + (static_cast<int64_t>(f) * 128 + 4 * m + rr) * M + t0;
                    if (kAligned4 && t0 + 3 < We) {
                        *reinterpret_cast<uint32_t *>(dst) = r[rr];
                    } else {
#pragma unroll
                        for (int b = 0; b < 4; b++)
                            if (t0 + b < We)
                                dst[b] = static_cast<uint8_t>(r[rr] >> (8 * b));
                    }
                }
            }
        }
        // ---- scales of the blocks that start inside this window
        {
            const int nb = sm.nblocks;
            for (int idx = tid; idx < nb * 128; idx += kThreads) {
                const int r = idx >> 7, kf = idx & 127;
                if (sm.bstart[r] >= W) {
                    const uint32_t S = (sm.smax[r] >> (8 * (kf >> 5))) & 0xFFu;
                    reinterpret_cast<uint32_t *>(yTs)[(static_cast<int64_t>(f) * 128 + kf) * cap +
                                                      sm.bslot[r]] = fp8_block_scale_bits(S, k);
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace fq

using namespace fq;

extern "C" int64_t fp4_to_fp8_cols_scale_capacity(int64_t M, int32_t G)
{
    if (M < 0 || G < 1)
        return -1;
    return (M + 127) / 128 + G;
}

extern "C" fq_status fp4_to_fp8_cols(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K,
                                     const int64_t *group_offsets, int32_t G, int exp_offset_k,
                                     uint8_t *yT, float *yT_scale, int64_t cap,
                                     int32_t *dev_status, void *stream)
{
    if (M < 0 || M > INT32_MAX - 512 || K <= 0 || K % 128 != 0)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (G < 1 || G > FQ_COLS_MAX_GROUPS || exp_offset_k < 0 || exp_offset_k > 6)
        return FQ_ERR_ARG;
    if (cap < fp4_to_fp8_cols_scale_capacity(M, G))
        return FQ_ERR_ARG;
    if (M == 0)
        return FQ_OK;
    if (!q || !s || !group_offsets || !yT || !yT_scale)
        return FQ_ERR_NULL;
    if (!aligned16(q) || !aligned16(s) || !aligned16(group_offsets) || !aligned16(yT) ||
        !aligned16(yT_scale))
        return FQ_ERR_ALIGN;
    const size_t dyn = static_cast<size_t>(G + 1) * 2 * sizeof(int32_t);
    const int64_t ntiles = ((M + 127) / 128) * (K / 128);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M % 4 == 0) {
        const int grid = persistent_grid(fp4_to_fp8_cols_kernel<true>, kThreads, dyn, ntiles);
        fp4_to_fp8_cols_kernel<true><<<grid, kThreads, dyn, st>>>(
            q, s, static_cast<int32_t>(M), K, group_offsets, G, exp_offset_k, yT, yT_scale, cap,
            dev_status);
    } else {
        const int grid = persistent_grid(fp4_to_fp8_cols_kernel<false>, kThreads, dyn, ntiles);
        fp4_to_fp8_cols_kernel<false><<<grid, kThreads, dyn, st>>>(
            q, s, static_cast<int32_t>(M), K, group_offsets, G, exp_offset_k, yT, yT_scale, cap,
            dev_status);
    }
    return launch_status();
}
