// The whole MXFP4 forward cast of the MoE recipe in one call: BF16 -> MXFP4
// (BF16ToFP4Row), the direct FP4 -> FP8 row conversion (FP4RowToFP8Row) and
// the transposed, ragged FP4 -> FP8 conversion (FP4RowToFP8Col), every output
// byte equal to the three separate calls.
//
// Source: "Practical FP4 Training for Large-Scale MoE Models on Hopper GPUs",
// technical overview section 2: item 1 (MXFP4; the direct FP4 -> FP8
// conversion with scales aligned to the largest of four, no BF16
// intermediate), item 3 (BF16ToFP4Row, FP4RowToFP8Row, FP4RowToFP8Col; the
// transpose fused with the quantization so that global memory is touched as
// little as possible; ragged expert groups without padding); section 3, items
// 2 and 3.
//
// Two entry points with the same arguments and outputs:
//  * bf16_to_mxfp4_fp8 -- two kernels on the caller's stream.  The row
//    kernel reads the BF16 tensor once and writes the MXFP4 codes and scales
//    together with the FP8 rows made from the codes still in registers; the
//    transposed kernel then reads the codes and scales back (the row kernel
//    leaves them in L2 with an evict-last policy where they fit).  The faster
//    of the two on GB300.
//  * bf16_to_mxfp4_fp8_single_pass -- one kernel, bf16_to_mxfp4_fp8_kernel,
//    that reads the BF16 tensor once and writes every output once from
//    registers and shared memory; no output is read back.
//
// The single-pass kernel's work unit is one 128-token block of the
// transposed conversion (blocks start at each group's first token, the last
// block of a group may be short) times 128 features.  Such a unit holds
// everything its outputs need: the MX blocks of its tokens (four per token),
// the FP8 row blocks (one per token) and the transposed FP8 blocks (one per
// MX column, over the unit's tokens).  Persistent CTAs of 9 warps (three per
// SM) walk the units block fastest (neighbouring CTAs write neighbouring
// token ranges of the same FP8 rows):
//  * the producer warp copies each unit's BF16 tile (128 rows x 2 x 128 B,
//    128-byte swizzled so that the reads below are free of bank conflicts)
//    into one of two shared-memory stages with tensor-memory-access copies;
//  * the eight converting warps take a unit in two phases.  Row phase: each
//    lane owns two (token, MX block) pairs: the block amax, the UE8M0
//    exponent, 32 E2M1 codes, and -- the token's four exponents exchanged
//    over two shuffles -- the FP8 row conversion of its codes with the shift
//    table; it writes the codes, the exponent word, the FP8 bytes and the FP8
//    row scale, and keeps its codes and exponents in registers.  Each warp's
//    byte-wise maximum of its tokens' exponent words goes to shared memory.
//    Transposed phase (after a named barrier, when the stage's BF16 is no
//    longer read): S of each MX column is the maximum of the warps' words;
//    each lane converts its own pairs with their shifts (S - e) into an FP8
//    tile laid out in the same stage, and after a second barrier the tile is
//    read back transposed and written as the FP8 rows of the unit's 128
//    features, each row segment at the block's token offset: full 16-byte
//    pieces by quarter warps, the partial 16-byte pieces at the two ends of
//    a segment that does not start on a 16-byte boundary by one lane per row
//    (aligned 8/4/2/1-byte stores); the unit's 128 FP32 block scales are one
//    512-byte store.  Then the stage goes back to the producer.
// Every mbarrier wait is bounded; a wait that gives up ends the kernel with
// bit 2 of *dev_status set.
#include "fq_cols_common.cuh"

namespace fq {

constexpr int kFusedWarps = 8;                       // converting warps
constexpr int kFusedThreads = 32 * (kFusedWarps + 1);
constexpr int kFusedStages = 2;
constexpr int kFusedHalfBytes = kTok * 128;          // 64 features x 128 tokens of BF16
constexpr int kFusedStageBytes = 2 * kFusedHalfBytes;
constexpr int kFusedQuads = kTok / 4 + 4;            // token columns 0..143 (offset a <= 15)
constexpr int kFusedTileSlots = tile_slots(kFusedQuads);
constexpr int kFusedAlign = 1024;                    // 128-byte swizzled copy destinations
static_assert(kFusedTileSlots * 16 <= kFusedStageBytes, "the FP8 tile fits in a stage");

inline size_t fused_dyn_bytes(int32_t G)
{
    return kFusedAlign + static_cast<size_t>(kFusedStages) * kFusedStageBytes +
           kFusedWarps * sizeof(uint32_t) + static_cast<size_t>(G + 1) * 2 * sizeof(int32_t);
}

// Element-wise max of |a| and |b| for two BF16 pairs (NaN wins; the sign
// bits of the result are to be cleared by the caller).
__device__ __forceinline__ uint32_t amax_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Largest of the four bytes of a word.
__device__ __forceinline__ uint32_t byte_max(uint32_t w)
{
    const uint32_t h = max_u16x2(w & 0x00FF00FFu, (w >> 8) & 0x00FF00FFu);
    return max(h & 0xFFFFu, h >> 16);
}

// Word i4 (0..3, not a compile-time constant) of {w0, w1, w2, w3}: selects
// without indexing a register array.
__device__ __forceinline__ uint32_t word_at(const uint32_t w[4], int i4)
{
    const uint32_t lo = (i4 & 1) ? w[1] : w[0];
    const uint32_t hi = (i4 & 1) ? w[3] : w[2];
    return (i4 & 2) ? hi : lo;
}

// Stores of the `bytes` low bytes (1, 2, 4 or 8) of the 16-byte row {w}
// starting at byte o (aligned to the size) to p + o.
__device__ __forceinline__ void store_aligned(uint8_t *p, const uint32_t w[4], int o, int bytes)
{
    const uint32_t v = word_at(w, o >> 2);
    if (bytes == 8)
        __stcs(reinterpret_cast<uint2 *>(p + o), make_uint2(v, word_at(w, (o >> 2) + 1)));
    else if (bytes == 4)
        __stcs(reinterpret_cast<unsigned int *>(p + o), v);
    else if (bytes == 2)
        __stcs(reinterpret_cast<unsigned short *>(p + o),
               static_cast<unsigned short>(v >> (8 * (o & 2))));
    else
        p[o] = static_cast<uint8_t>(v >> (8 * (o & 3)));
}

// Row rr (0..3) of the four slots (quads 4i .. 4i+3) of feature word m: the
// 16 FP8 bytes of output row 4m + rr for token columns 16i .. 16i+15.
__device__ __forceinline__ void tile_row16(const uint32_t *tile, int i, int m, int rr,
                                           uint32_t w[4])
{
    const uint32_t sel = static_cast<uint32_t>(rr) | (static_cast<uint32_t>(rr + 4) << 4);
#pragma unroll
    for (int qq = 0; qq < 4; qq++) {
        const uint4 v = *reinterpret_cast<const uint4 *>(tile + 4 * slot_index(4 * i + qq, m));
        w[qq] = prmt(prmt(v.x, v.y, sel), prmt(v.z, v.w, sel), 0x5410u);
    }
}

// Write-out of a unit's FP8 tile: tokens t0 .. t0+n-1 sit at token columns
// a .. a+n-1 (a = t0 mod 16 when every output row starts on a 16-byte
// boundary, else 0); chunk i covers columns 16i .. 16i+15 and output bytes
// t0 - a + 16i .. +15 of each row.
//  * full chunks: a quarter warp handles one feature word (four output
//    rows) and chunks c_out, c_out + 8, one 16-byte store per row;
//  * the partial first chunk [a, 16) and last chunk [0, r): one thread per
//    output row (threads 0..127 the first, 128..255 the last), as aligned
//    pieces of 1, 2, 4 and 8 bytes -- the set bits of the piece's length.
// Without 16-byte aligned rows every chunk is written byte by byte.
template <bool kAligned16>
__device__ __forceinline__ void write_block_tile(const uint32_t *tile, uint8_t *__restrict__ yT,
                                                 int32_t M, int32_t t0, int32_t n, int a,
                                                 int64_t feat0, int tid)
{
    const int nch = (a + n + 15) >> 4;  // <= 9
    const int r = (a + n) & 15;         // bytes of the last chunk if partial
    const int wid = tid >> 5, lane = tid & 31;
    const int m_out = 4 * wid + (lane >> 3), c_out = lane & 7;
    uint8_t *const base = yT + (t0 - a);
    if (!kAligned16) {
        // rows of yT not 16-byte aligned (a = 0: the tile's token columns are
        // the unit's tokens).  Row k's segment starts a_k = (its start) mod 16
        // bytes past a 16-byte boundary, so its aligned blocks start at token
        // sft = (16 - a_k) mod 16 and every 16 tokens after: lane c writes
        // block c when it is whole (bytes sft .. 15 of chunk c and 0 .. sft - 1
        // of chunk c + 1); the partial blocks at the segment's two ends are
        // written below, one thread per row and end.  (Single-byte stores
        // made M % 16 != 0 about three times slower than M % 16 == 0.)
        uint32_t cur[4][4], nx[4][4];
#pragma unroll
        for (int qq = 0; qq < 4; qq++) {
            const uint4 v =
                *reinterpret_cast<const uint4 *>(tile + 4 * slot_index(4 * c_out + qq, m_out));
            transpose4x4(v, cur[0][qq], cur[1][qq], cur[2][qq], cur[3][qq]);
            const uint4 u =
                *reinterpret_cast<const uint4 *>(tile + 4 * slot_index(4 * c_out + 4 + qq, m_out));
            transpose4x4(u, nx[0][qq], nx[1][qq], nx[2][qq], nx[3][qq]);
        }
        uint8_t *seg = yT + (feat0 + 4 * m_out) * static_cast<int64_t>(M) + t0;
#pragma unroll
        for (int rr = 0; rr < 4; rr++) {
            const int ar = static_cast<int>(reinterpret_cast<uintptr_t>(seg) & 15);
            const int sft = (16 - ar) & 15;
            const int t_blk = sft + 16 * c_out;
            if (t_blk + 16 <= n) {
                uint32_t y[4];
                if (sft == 0) {
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        y[i] = cur[rr][i];
                } else {
                    bytes_at(cur[rr], nx[rr], sft, y);
                }
                __stcs(reinterpret_cast<uint4 *>(seg + t_blk), make_uint4(y[0], y[1], y[2], y[3]));
            }
            seg += M;
        }
        // the partial blocks: thread tid & 127 owns row tid & 127, threads
        // below 128 its head (tokens 0 .. sft - 1), the others its tail
        const int kr = tid & (kTok - 1);
        uint8_t *row = yT + (feat0 + kr) * static_cast<int64_t>(M) + t0;
        const int ar = static_cast<int>(reinterpret_cast<uintptr_t>(row) & 15);
        const int sft = (16 - ar) & 15;
        const int full = n >= sft ? (n - sft) >> 4 : 0;  // whole blocks
        uint32_t w0[4], w1[4], y[4];
        if (tid < kTok) {
            if (sft > 0) {
                tile_row16(tile, 0, kr >> 2, kr & 3, w0);
                bytes_at(w0, w0, 16 - ar, y);  // y[ar + i] = token i
                store_block_range(row - ar, y, ar, ar + min(sft, n));
            }
        } else {
            const int tt = sft + 16 * full;  // the tail block's first token
            if (n > sft && tt < n) {
                tile_row16(tile, full, kr >> 2, kr & 3, w0);
                if (sft == 0) {
#pragma unroll
                    for (int i = 0; i < 4; i++)
                        y[i] = w0[i];
                } else {
                    tile_row16(tile, full + 1, kr >> 2, kr & 3, w1);
                    bytes_at(w0, w1, sft, y);
                }
                store_block_range(row + tt, y, 0, n - tt);
            }
        }
        return;
    }
    for (int i = c_out; i < nch; i += 8) {
        if ((i == 0 && a != 0) || (i == nch - 1 && r != 0))
            continue;  // a partial chunk, below
        uint32_t rows[4][4];
#pragma unroll
        for (int qq = 0; qq < 4; qq++) {
            const uint4 v =
                *reinterpret_cast<const uint4 *>(tile + 4 * slot_index(4 * i + qq, m_out));
            transpose4x4(v, rows[0][qq], rows[1][qq], rows[2][qq], rows[3][qq]);
        }
        uint8_t *p = base + (feat0 + 4 * m_out) * static_cast<int64_t>(M) + 16 * i;
#pragma unroll
        for (int rr = 0; rr < 4; rr++) {
            __stcs(reinterpret_cast<uint4 *>(p),  // evict-first: yT is not re-read
                   make_uint4(rows[rr][0], rows[rr][1], rows[rr][2], rows[rr][3]));
            p += M;
        }
    }
    // partial chunks: thread tid & 127 owns output row tid & 127
    const bool head = tid < kTok;
    const int i = head ? 0 : nch - 1;
    int lo, len;
    if (head) {
        lo = a;
        len = (nch == 1 ? a + n : 16) - a;
        if (a == 0)
            len = 0;
    } else {
        lo = 0;
        len = (nch == 1 && a != 0) ? 0 : r;  // a single chunk with a > 0 is the head's
    }
    if (len == 0)
        return;
    const int k = tid & (kTok - 1);
    uint32_t w[4];
    tile_row16(tile, i, k >> 2, k & 3, w);
    uint8_t *p = base + (feat0 + k) * static_cast<int64_t>(M) + 16 * i;
    if (lo + len == 16 || lo == 0) {
        // [lo, 16) from the bottom up, or [0, len) from the top down: the
        // piece of size s sits after the smaller (first case) or larger
        // (second case) pieces
        if (lo + len == 16) {
#pragma unroll
            for (int sz = 1; sz <= 8; sz <<= 1)
                if (len & sz)
                    store_aligned(p, w, lo + (len & (sz - 1)), sz);
        } else {
#pragma unroll
            for (int sz = 8; sz >= 1; sz >>= 1)
                if (len & sz)
                    store_aligned(p, w, len & ~(2 * sz - 1), sz);
        }
    } else {
        for (int bb = lo; bb < lo + len; bb++)  // a short block inside one chunk
            p[bb] = static_cast<uint8_t>(word_at(w, bb >> 2) >> (8 * (bb & 3)));
    }
}

template <bool kAligned16>
__global__ void __launch_bounds__(kFusedThreads, 3) bf16_to_mxfp4_fp8_kernel(
    const __grid_constant__ CUtensorMap tm_x, int32_t M, int32_t nchunk,
    const int64_t *__restrict__ offs, int32_t G, int k, uint8_t *__restrict__ q,
    uint8_t *__restrict__ s, uint8_t *__restrict__ y, float *__restrict__ ys,
    uint8_t *__restrict__ yT, float *__restrict__ yTs, int32_t *__restrict__ dev_status)
{
    __shared__ __align__(16) uint8_t tab[kTabRows * 8];
    __shared__ int32_t warp_tot[kFusedThreads / 32];
    __shared__ __align__(8) uint64_t full[kFusedStages];   // a unit's BF16 tile landed
    __shared__ __align__(8) uint64_t empty[kFusedStages];  // unit written out by every warp
    extern __shared__ __align__(16) uint8_t dyn_raw[];
    uint8_t *stages = dyn_raw + ((kFusedAlign - (smem_u32(dyn_raw) & (kFusedAlign - 1))) &
                                 (kFusedAlign - 1));
    uint32_t *part = reinterpret_cast<uint32_t *>(stages + kFusedStages * kFusedStageBytes);
    int32_t *off = reinterpret_cast<int32_t *>(part + kFusedWarps);       // [G + 1]
    int32_t *base = off + G + 1;                                          // [G + 1]

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t K = 128 * static_cast<int64_t>(nchunk);
    if (tid == 0) {
        for (int i = 0; i < kFusedStages; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kFusedWarps);
        }
        mbar_init_fence();
    }
    build_fp8_table(tab);
    griddep_wait();  // x and the offsets may come from the previous kernel
    griddep_launch_dependents();
    const int bad = load_groups(offs, G, M, off, base, warp_tot);  // ends with a CTA barrier
    if (bad && blockIdx.x == 0 && tid == 0 && dev_status)
        atomicOr(dev_status, 1);

    const int32_t NB = base[G];
    const int32_t nunits = NB * nchunk;  // < 2^31, checked on the host
    const int32_t grid = static_cast<int32_t>(gridDim.x);
    const int32_t bx = static_cast<int32_t>(blockIdx.x);
    const int32_t my_units = bx < nunits ? (nunits - bx + grid - 1) / grid : 0;

    // unit m of this CTA: block b (fastest), feature chunk f; the block's
    // first token t0 and length n (warp-uniform, all 32 lanes call it)
    auto unit = [&](int32_t m, int32_t &b, int32_t &f, int32_t &t0, int32_t &n) {
        const int32_t u = bx + m * grid;
        b = u % NB;
        f = u / NB;
        const int g = warp_find_last_le(base, G, b);
        t0 = off[g] + (b - base[g]) * kTok;
        n = min(kTok, off[g + 1] - t0);
    };

    if (wid == kFusedWarps) {
        // ================================================= producer warp
        bool ok = true;
        int32_t issued = 0;
        for (int32_t m = 0; m < my_units; m++) {
            const int st = m % kFusedStages;
            if (m >= kFusedStages) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&empty[st], static_cast<uint32_t>(m / kFusedStages - 1) & 1u));
                if (!ok)
                    break;
            }
            int32_t b, f, t0, n;
            unit(m, b, f, t0, n);
            if (lane == 0) {
                uint8_t *dst = stages + st * kFusedStageBytes;
                mbar_arrive_expect_tx(&full[st], kFusedStageBytes);
                tma_load_2d(dst, &tm_x, 128 * f, t0, &full[st]);
                tma_load_2d(dst + kFusedHalfBytes, &tm_x, 128 * f + 64, t0, &full[st]);
            }
            issued++;
        }
        if (!ok) {
            // report, and wait (bounded) for the copies that may still be in
            // flight before the CTA's shared memory is released
            if (lane == 0 && dev_status)
                atomicOr(dev_status, 2);
            for (int32_t m = max(0, issued - kFusedStages); m < issued; m++)
                mbar_wait(&full[m % kFusedStages], static_cast<uint32_t>(m / kFusedStages) & 1u);
        }
        return;
    }

    // ===================================================== converting warps
    const int jr = lane >> 3;             // the lane's MX block (of four) and MX column
    const int tr = 8 * wid + (lane & 7);  // its tokens tr and tr + 64
    const int64_t qrow = K / 2, srow = K / 32;
    for (int32_t m = 0; m < my_units; m++) {
        const int st = m % kFusedStages;
        uint8_t *stage = stages + st * kFusedStageBytes;
        int32_t b, f, t0, n;
        unit(m, b, f, t0, n);
        const bool ok = mbar_wait(&full[st], static_cast<uint32_t>(m / kFusedStages) & 1u);

        // ---- row phase
        uint32_t c4[2][4], eb[2];
        uint32_t acc = 0;  // byte-wise max of the exponent words of this warp's tokens
        if (ok) {
            const uint8_t *half = stage + (jr >> 1) * kFusedHalfBytes;
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int tl = tr + 64 * h;
                const uint8_t *row = half + tl * 128;
                uint4 v[4];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    v[i] = *reinterpret_cast<const uint4 *>(row +
                                                            16 * ((4 * (jr & 1) + i) ^ (tl & 7)));
                const uint32_t m2a = amax_bf16x2(amax_bf16x2(v[0].x, v[0].y),
                                                 amax_bf16x2(v[0].z, v[0].w));
                const uint32_t m2b = amax_bf16x2(amax_bf16x2(v[1].x, v[1].y),
                                                 amax_bf16x2(v[1].z, v[1].w));
                const uint32_t m2c = amax_bf16x2(amax_bf16x2(v[2].x, v[2].y),
                                                 amax_bf16x2(v[2].z, v[2].w));
                const uint32_t m2d = amax_bf16x2(amax_bf16x2(v[3].x, v[3].y),
                                                 amax_bf16x2(v[3].z, v[3].w));
                const uint32_t mx =
                    amax_bf16x2(amax_bf16x2(m2a, m2b), amax_bf16x2(m2c, m2d)) & 0x7FFF7FFFu;
                const uint32_t amax = hmax_u16x2(mx);  // |x| bits of the block max
                // e = max(E - 2, 0) for the exponent field E of the block max
                // (zero and subnormals have E = 0); 0xFF for NaN or Inf
                const bool special = amax >= 0x7F80u;
                const int Ex = static_cast<int>(amax >> 7);
                const uint32_t e = static_cast<uint32_t>(Ex > 2 ? Ex - 2 : 0);
                const float mul = __uint_as_float((254u - e) << 23);  // 2^(127 - e)
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    float a0, a1, a2, a3, a4, a5, a6, a7;
                    fmul2(bf16_lo(v[i].x), bf16_hi(v[i].x), mul, a0, a1);
                    fmul2(bf16_lo(v[i].y), bf16_hi(v[i].y), mul, a2, a3);
                    fmul2(bf16_lo(v[i].z), bf16_hi(v[i].z), mul, a4, a5);
                    fmul2(bf16_lo(v[i].w), bf16_hi(v[i].w), mul, a6, a7);
                    c4[h][i] = special ? 0u : cvt_e2m1x8(a0, a1, a2, a3, a4, a5, a6, a7);
                }
                eb[h] = special ? 0xFFu : e;
                // the token's four exponents (lanes 8 apart hold its blocks)
                uint32_t word = eb[h] << (8 * jr);
                word |= __shfl_xor_sync(0xffffffffu, word, 8);
                word |= __shfl_xor_sync(0xffffffffu, word, 16);
                const uint32_t S = byte_max(word);
                // FP8 row block of the token: its 32 codes of this MX block
                const bool nan = S == 0xFFu;
                int u = static_cast<int>(S - eb[h]) - k + 6;
                u = u < kShiftRows - 1 ? u : kShiftRows - 1;
                const uint2 t = *reinterpret_cast<const uint2 *>(tab + 8 * (nan ? kNanRow : u));
                const uint32_t smask = nan ? 0u : 0x80808080u;
                uint32_t o[8];
#pragma unroll
                for (int i = 0; i < 4; i++)
                    fp4x8_to_fp8x8(c4[h][i], t.x, t.y, o[2 * i], o[2 * i + 1], smask);
                if (tl < n) {
                    const int64_t tg = t0 + tl;
                    __stcs(reinterpret_cast<uint4 *>(q + tg * qrow + 64 * f + 16 * jr),
                           make_uint4(c4[h][0], c4[h][1], c4[h][2], c4[h][3]));
                    uint4 *yp = reinterpret_cast<uint4 *>(y + tg * K + 128 * f + 32 * jr);
                    __stcs(yp, make_uint4(o[0], o[1], o[2], o[3]));
                    __stcs(yp + 1, make_uint4(o[4], o[5], o[6], o[7]));
                    if (jr == 0) {
                        __stcs(reinterpret_cast<unsigned int *>(s + tg * srow + 4 * f), word);
                        __stcs(reinterpret_cast<unsigned int *>(ys) + tg * nchunk + f,
                               fp8_block_scale_bits(S, k));
                    }
                    acc = bytemax4(acc, word);
                }
            }
        }
        acc = bytemax4(acc, __shfl_xor_sync(0xffffffffu, acc, 1));
        acc = bytemax4(acc, __shfl_xor_sync(0xffffffffu, acc, 2));
        acc = bytemax4(acc, __shfl_xor_sync(0xffffffffu, acc, 4));
        if (lane == 0)
            part[wid] = acc;
        // every warp is done with the stage's BF16 (it now holds the FP8
        // tile) and has published its maxima
        if (named_barrier_or(1, kFusedWarps * 32, !ok)) {
            // a copy did not arrive in time; the producer may be past its
            // last wait, so the converting warps report it themselves
            if (tid == 0 && dev_status)
                atomicOr(dev_status, 2);
            break;
        }

        // ---- transposed phase
        uint32_t *tile = reinterpret_cast<uint32_t *>(stage);
        uint32_t Sw = part[0];
#pragma unroll
        for (int w = 1; w < kFusedWarps; w++)
            Sw = bytemax4(Sw, part[w]);
        const int a = kAligned16 ? (t0 & 15) : 0;
        const uint32_t Sj = (Sw >> (8 * jr)) & 0xFFu;
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int tl = tr + 64 * h;
            if (tl < n) {
                uint32_t u;
                if (Sj == 0xFFu) {
                    u = kNanRow;
                } else {
                    const int d = static_cast<int>(Sj - eb[h]) - k + 6;  // >= 0: Sj is the max
                    u = static_cast<uint32_t>(d < kShiftRows - 1 ? d : kShiftRows - 1);
                }
                convert_unit_row(tile, tab, a + tl, jr,
                                 make_uint4(c4[h][0], c4[h][1], c4[h][2], c4[h][3]), u);
            }
        }
        named_barrier_or(1, kFusedWarps * 32, false);  // the FP8 tile is complete
        if (wid == 0) {
            // block b's FP32 scales of features 128f .. 128f+127: 512 bytes
            const uint32_t v = fp8_block_scale_bits((Sw >> (8 * (lane >> 3))) & 0xFFu, k);
            __stcs(reinterpret_cast<uint4 *>(yTs + static_cast<int64_t>(b) * K + 128 * f) + lane,
                   make_uint4(v, v, v, v));
        }
        write_block_tile<kAligned16>(tile, yT, M, t0, n, a, 128 * static_cast<int64_t>(f), tid);
        // the stage's next contents come from a tensor copy: order this
        // warp's shared-memory accesses before it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);  // this warp is done with the stage
    }
}

}  // namespace fq

using namespace fq;

namespace {

// Shared argument checks of the two entry points (FQ_OK: go on; M == 0 is
// reported as FQ_OK through *empty).
fq_status check_fused_args(const void *x, int64_t M, int64_t K, const int64_t *group_offsets,
                           int32_t G, int exp_offset_k, const uint8_t *q, const uint8_t *s,
                           const uint8_t *y, const float *ys, const uint8_t *yT,
                           const float *yT_scale, int64_t cap, bool *empty)
{
    *empty = false;
    if (M < 0 || M > INT32_MAX - 512 || K <= 0 || K % 128 != 0 || K > INT32_MAX - 256)
        return FQ_ERR_SHAPE;
    if (M > 0 && K > INT64_MAX / M)
        return FQ_ERR_SHAPE;
    if (((M + 127) / 128) * (K / 128) > INT32_MAX - 4096)  // tile index is 32-bit
        return FQ_ERR_SHAPE;
    if ((M / 128 + 1 + static_cast<int64_t>(G)) * (K / 128) > INT32_MAX - 4096)  // unit index
        return FQ_ERR_SHAPE;
    if (G < 1 || G > FQ_COLS_MAX_GROUPS || exp_offset_k < 0 || exp_offset_k > 6)
        return FQ_ERR_ARG;
    if (cap < fp4_to_fp8_cols_scale_capacity(M, G))
        return FQ_ERR_ARG;
    if (M == 0) {
        *empty = true;
        return FQ_OK;
    }
    if (!x || !group_offsets || !q || !s || !y || !ys || !yT || !yT_scale)
        return FQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(group_offsets) || !aligned16(q) || !aligned16(s) ||
        !aligned16(y) || !aligned16(ys) || !aligned16(yT) || !aligned16(yT_scale))
        return FQ_ERR_ALIGN;
    return FQ_OK;
}

}  // namespace

extern "C" fq_status bf16_to_mxfp4_fp8(const void *x, int64_t M, int64_t K,
                                       const int64_t *group_offsets, int32_t G, int exp_offset_k,
                                       uint8_t *q, uint8_t *s, uint8_t *y, float *ys, uint8_t *yT,
                                       float *yT_scale, int64_t cap, int32_t *dev_status,
                                       void *stream)
{
    bool empty;
    const fq_status chk = check_fused_args(x, M, K, group_offsets, G, exp_offset_k, q, s, y, ys,
                                           yT, yT_scale, cap, &empty);
    if (chk != FQ_OK || empty)
        return chk;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const fq_status rc = launch_mxfp4_rows(x, M, K, q, s, exp_offset_k, y, ys, st);
    if (rc != FQ_OK)
        return rc;
    return launch_fp4_to_fp8_cols(q, s, M, K, group_offsets, G, exp_offset_k, yT, yT_scale, cap,
                                  dev_status, st);
}

extern "C" fq_status bf16_to_mxfp4_fp8_single_pass(const void *x, int64_t M, int64_t K,
                                                   const int64_t *group_offsets, int32_t G,
                                                   int exp_offset_k, uint8_t *q, uint8_t *s,
                                                   uint8_t *y, float *ys, uint8_t *yT,
                                                   float *yT_scale, int64_t cap,
                                                   int32_t *dev_status, void *stream)
{
    bool empty;
    const fq_status chk = check_fused_args(x, M, K, group_offsets, G, exp_offset_k, q, s, y, ys,
                                           yT, yT_scale, cap, &empty);
    if (chk != FQ_OK || empty)
        return chk;
    CUtensorMap tm_x;
    if (!encode_tensor_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, static_cast<uint64_t>(K),
                              static_cast<uint64_t>(M), static_cast<uint64_t>(K) * 2, 64, kTok,
                              CU_TENSOR_MAP_SWIZZLE_128B, true)) {
        // no tensor-map encoder in this driver
        set_last_cuda_error(static_cast<int>(cudaErrorNotSupported));
        return FQ_ERR_CUDA;
    }
    const size_t dyn = fused_dyn_bytes(G);
    auto kern = M % 16 == 0 ? bf16_to_mxfp4_fp8_kernel<true> : bf16_to_mxfp4_fp8_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(dyn)) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return launch_status();
    const int64_t max_units = cap * (K / 128);
    const int grid = persistent_grid(kern, kFusedThreads, dyn, max_units);
    launch_pdl(kern, dim3(grid), dim3(kFusedThreads), dyn, static_cast<cudaStream_t>(stream),
               tm_x, static_cast<int32_t>(M), static_cast<int32_t>(K / 128), group_offsets, G,
               exp_offset_k, q, s, y, ys, yT, yT_scale, dev_status);
    return launch_status();
}
