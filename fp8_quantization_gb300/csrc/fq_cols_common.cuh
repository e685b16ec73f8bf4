// Device helpers of the transposed FP4 -> FP8 conversion, shared by the
// transposed cast (fq_cols.cu) and the one-pass forward cast (fq_fused.cu):
// the FP8 tile layout in shared memory, 4x4 byte transposes, byte-wise
// maxima, the group structure of the ragged token blocks and the per-unit
// conversion through the shift table.
//
// Source: "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// technical overview section 2, item 3 (transpose fused with the conversion
// through a skewed shared-memory layout; ragged expert groups without
// padding) and item 1 (scale alignment to the largest exponent).
#pragma once

#include "fq_common.cuh"

namespace fq {

constexpr int kTok = 128;  // tokens per block / per tile
// FP8 tile: 32 token-quads x 32 feature-words; the 16-byte slot holding
// (four tokens) x (one feature word) is slot_index(quad, m).  Within a quad
// the slots of an 8-word octet are consecutive (+2 between octets); the quad
// stride 39 = -1 (mod 8) plus quad/4 makes the slot's bank group
// (slot mod 8) = m + 2*(m/8) - quad + quad/4 (mod 8), which is
// conflict-free both for the conversion stores (2 quads x 4 column blocks x
// 4 tokens per warp) and for the 128-bit transposed reads (8 quads 4 apart
// per quarter warp: -3c distinct for c = 0..7).
constexpr int kQuadStride = 39;
// slots of an FP8 tile of nq token quads (the slot index of the last quad's last
// feature word, plus one)
constexpr int tile_slots(int nq) { return (nq - 1) * kQuadStride + (nq - 1) / 4 + 38; }

__device__ __forceinline__ int slot_index(int quad, int m)
{
    return quad * kQuadStride + (quad >> 2) + m + 2 * (m >> 3);
}

// Largest g in [lo, hi] with a[g] <= t (a non-decreasing, a[lo] <= t).
__device__ __forceinline__ int find_last_le(const int32_t *a, int lo, int hi, int32_t t)
{
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (a[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Same search for a warp-uniform t: with n <= 64 one or two ballots over the
// array replace the binary search.
__device__ __forceinline__ int warp_find_last_le(const int32_t *a, int n, int32_t t)
{
    if (n > 64)
        return find_last_le(a, 0, n - 1, t);
    const int lane = threadIdx.x & 31;
    int g = 0;
    for (int b0 = 0; b0 < n; b0 += 32) {
        const int i = b0 + lane;
        const unsigned m = __ballot_sync(0xffffffffu, i < n && a[i] <= t);
        if (m)
            g = b0 + 31 - __clz(m);
        if (m != 0xffffffffu)
            break;
    }
    return g;
}

// In-place inclusive scan (max or sum) of a[0..n) in shared memory by the
// whole CTA.
template <bool kMax>
__device__ inline void cta_scan(int32_t *a, int n, int32_t *warp_tot /* [kThreads/32] */)
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

// Group structure of the offsets, in shared memory (once per CTA): off[0..G]
// clamped into [0, M], non-decreasing, off[0] = 0, off[G] = M; base[g] = the
// first scale slot of group g (number of 128-token blocks of the groups
// before it), base[G] = total blocks.  Returns nonzero if the offsets given
// were malformed.
__device__ inline int load_groups(const int64_t *__restrict__ offs, int32_t G, int32_t M, int32_t *off,
                           int32_t *base, int32_t *warp_tot)
{
    const int tid = threadIdx.x;
    if (G < 64) {
        // one warp, entries 2l and 2l + 1 in lane l (G + 1 <= 64): clamp,
        // max-scan and sum-scan with shuffles, no CTA barrier but the last
        int bad = 0;
        if (tid < 32) {
            const int lane = tid;
            const int i0 = 2 * lane, i1 = i0 + 1;
            const int64_t o0 = i0 <= G ? offs[i0] : M;
            const int64_t o1 = i1 <= G ? offs[i1] : M;
            const int64_t p0 = __shfl_up_sync(0xffffffffu, o1, 1);  // offs[i0 - 1] for lane >= 1
            const int64_t c0 = o0 < 0 ? 0 : (o0 > M ? M : o0);
            const int64_t c1 = o1 < 0 ? 0 : (o1 > M ? M : o1);
            bad = (i0 <= G && (c0 != o0 || (i0 == 0 && o0 != 0) || (i0 == G && o0 != M) ||
                               (i0 > 0 && o0 < p0))) ||
                  (i1 <= G && (c1 != o1 || (i1 == G && o1 != M) || o1 < o0));
            const int32_t m1 = static_cast<int32_t>(c0 > c1 ? c0 : c1);
            int32_t incl = m1;
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t u = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d)
                    incl = max(incl, u);
            }
            int32_t excl = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane == 0)
                excl = 0;
            int32_t v0 = max(excl, static_cast<int32_t>(c0)), v1 = max(excl, m1);
            if (i0 == 0)
                v0 = 0;
            if (i0 == G)
                v0 = M;
            if (i1 == G)
                v1 = M;
            const int32_t vprev = __shfl_up_sync(0xffffffffu, v1, 1);  // entry i0 - 1
            const int32_t nb0 = i0 >= 1 && i0 <= G ? (v0 - vprev + kTok - 1) / kTok : 0;
            const int32_t nb1 = i1 <= G ? (v1 - v0 + kTok - 1) / kTok : 0;
            int32_t sincl = nb0 + nb1;
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t u = __shfl_up_sync(0xffffffffu, sincl, d);
                if (lane >= d)
                    sincl += u;
            }
            int32_t sexcl = __shfl_up_sync(0xffffffffu, sincl, 1);
            if (lane == 0)
                sexcl = 0;
            if (i0 <= G) {
                off[i0] = v0;
                base[i0] = sexcl + nb0;
            }
            if (i1 <= G) {
                off[i1] = v1;
                base[i1] = sexcl + nb0 + nb1;
            }
            bad = __any_sync(0xffffffffu, bad);
        }
        return __syncthreads_or(bad);
    }
    int bad = 0;
    for (int i = tid; i <= G; i += kThreads) {
        const int64_t o = offs[i];
        const int64_t c = o < 0 ? 0 : (o > M ? M : o);
        off[i] = static_cast<int32_t>(c);
        if (c != o || (i == 0 && o != 0) || (i == G && o != M) || (i > 0 && o < offs[i - 1]))
            bad = 1;
    }
    bad = __syncthreads_or(bad);
    cta_scan<true>(off, G + 1, warp_tot);
    if (tid == 0) {
        off[0] = 0;
        off[G] = M;
    }
    __syncthreads();
    for (int g = tid; g <= G; g += kThreads)
        base[g] = g == 0 ? 0 : (off[g] - off[g - 1] + kTok - 1) / kTok;
    __syncthreads();
    cta_scan<false>(base, G + 1, warp_tot);
    return bad;
}

// Word i (0..3, not a compile-time constant) of y, without indexing a
// register array.
__device__ __forceinline__ uint32_t word_sel(const uint32_t y[4], int i)
{
    return (i & 2) ? ((i & 1) ? y[3] : y[2]) : ((i & 1) ? y[1] : y[0]);
}

// Bytes [s, s + 16) of the 32 bytes p ++ x (p first), 0 < s < 16.
__device__ __forceinline__ void bytes_at(const uint32_t p[4], const uint32_t x[4], int s,
                                         uint32_t y[4])
{
    const uint32_t z[8] = {p[0], p[1], p[2], p[3], x[0], x[1], x[2], x[3]};
    const int w0 = s >> 2;
    uint32_t zs[5];
#pragma unroll
    for (int j = 0; j < 5; j++)
        zs[j] = (w0 & 2) ? ((w0 & 1) ? z[3 + j] : z[2 + j]) : ((w0 & 1) ? z[1 + j] : z[j]);
#pragma unroll
    for (int i = 0; i < 4; i++)
        y[i] = __funnelshift_r(zs[i], zs[i + 1], 8 * (s & 3));
}

// Bytes [lo, hi) of the 16-byte block y to blk + lo .. blk + hi - 1 (blk
// 16-byte aligned), as aligned pieces of 8, 4, 2 and 1 bytes.
__device__ __forceinline__ void store_block_range(uint8_t *blk, const uint32_t y[4], int lo,
                                                  int hi)
{
    if (hi == 16) {
        // a suffix [lo, 16): the pieces are the set bits of 16 - lo, smallest first
#pragma unroll
        for (int sz = 1; sz <= 8; sz <<= 1) {
            if (lo & sz) {
                const uint32_t w = word_sel(y, lo >> 2);
                if (sz == 8)
                    __stcs(reinterpret_cast<uint2 *>(blk + lo), make_uint2(w, word_sel(y, (lo >> 2) + 1)));
                else if (sz == 4)
                    __stcs(reinterpret_cast<unsigned int *>(blk + lo), w);
                else if (sz == 2)
                    __stcs(reinterpret_cast<unsigned short *>(blk + lo),
                           static_cast<unsigned short>(w >> (8 * (lo & 2))));
                else
                    blk[lo] = static_cast<uint8_t>(w >> (8 * (lo & 3)));
                lo += sz;
            }
        }
        return;
    }
    if (lo == 0) {
        // a prefix [0, hi): the pieces are the set bits of hi, largest first
#pragma unroll
        for (int sz = 8; sz >= 1; sz >>= 1) {
            if (hi & sz) {
                const int o = hi & ~(2 * sz - 1);
                const uint32_t w = word_sel(y, o >> 2);
                if (sz == 8)
                    __stcs(reinterpret_cast<uint2 *>(blk + o), make_uint2(w, word_sel(y, (o >> 2) + 1)));
                else if (sz == 4)
                    __stcs(reinterpret_cast<unsigned int *>(blk + o), w);
                else if (sz == 2)
                    __stcs(reinterpret_cast<unsigned short *>(blk + o),
                           static_cast<unsigned short>(w >> (8 * (o & 2))));
                else
                    blk[o] = static_cast<uint8_t>(w >> (8 * (o & 3)));
            }
        }
        return;
    }
    int o = lo;
    while (o < hi) {
        const uint32_t w = word_sel(y, o >> 2);
        if (!(o & 7) && o + 8 <= hi) {
            __stcs(reinterpret_cast<uint2 *>(blk + o), make_uint2(w, word_sel(y, (o >> 2) + 1)));
            o += 8;
        } else if (!(o & 3) && o + 4 <= hi) {
            __stcs(reinterpret_cast<unsigned int *>(blk + o), w);
            o += 4;
        } else if (!(o & 1) && o + 2 <= hi) {
            __stcs(reinterpret_cast<unsigned short *>(blk + o),
                   static_cast<unsigned short>(w >> (8 * (o & 2))));
            o += 2;
        } else {
            blk[o] = static_cast<uint8_t>(w >> (8 * (o & 3)));
            o += 1;
        }
    }
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

__device__ __forceinline__ uint32_t bytemax4(uint32_t a, uint32_t b)
{
    const uint32_t e02 = max_u16x2(a & 0x00FF00FFu, b & 0x00FF00FFu);
    const uint32_t e13 = max_u16x2((a >> 8) & 0x00FF00FFu, (b >> 8) & 0x00FF00FFu);
    return e02 | (e13 << 8);
}

// The shift-table rows of four MX columns at once: byte i of the result is
// min(S_i - e_i - k + 6, kShiftRows - 1), or kNanRow where S_i = 0xFF (S is
// the block max, so S_i >= e_i and the byte-wise subtraction never borrows).
__device__ __forceinline__ uint32_t shift_rows4(uint32_t S, uint32_t e, int k)
{
    const uint32_t ones = 0x01010101u;
    const uint32_t d = S - e;
    uint32_t u = __vminu4(d, static_cast<uint32_t>(kShiftRows - 1 - 6 + k) * ones) +
                 static_cast<uint32_t>(6 - k) * ones;
    const uint32_t nan = __vcmpeq4(S, 0xFFFFFFFFu);  // 0xFF in bytes where S = 0xFF
    return (u & ~nan) | (static_cast<uint32_t>(kNanRow) * ones & nan);
}

// One unit from its shift-table row u (as convert_unit with u precomputed).
__device__ __forceinline__ void convert_unit_row(uint32_t *tile, const uint8_t *tab, int tl, int j,
                                                 uint4 qv, uint32_t u)
{
    const uint2 t = *reinterpret_cast<const uint2 *>(tab + 8 * u);
    const uint32_t smask = u == static_cast<uint32_t>(kNanRow) ? 0u : 0x80808080u;
    uint32_t o[8];
    fp4x8_to_fp8x8(qv.x, t.x, t.y, o[0], o[1], smask);
    fp4x8_to_fp8x8(qv.y, t.x, t.y, o[2], o[3], smask);
    fp4x8_to_fp8x8(qv.z, t.x, t.y, o[4], o[5], smask);
    fp4x8_to_fp8x8(qv.w, t.x, t.y, o[6], o[7], smask);
    uint32_t *dst = tile + 4 * slot_index(tl >> 2, 8 * j) + (tl & 3);
#pragma unroll
    for (int w = 0; w < 8; w++)
        dst[4 * w] = o[w];
}

}  // namespace fq
