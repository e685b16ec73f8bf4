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
// When K % 512 == 0 (a token's 16-byte exponent row slice then covers a
// super-tile of four 128-feature blocks) one launch does everything:
// fp4_to_fp8_cols_1pass_kernel, warp-specialised, with tensor-memory-access
// copies into shared memory (described at the kernel).  Otherwise two
// launches on the caller's stream:
//  1. fp4_to_fp8_cols_scales_kernel -- one CTA per 128-token block (blocks
//     start at each group's first token): the byte-wise max of the block's
//     UE8M0 exponents for every MX column, written out as the FP32 block
//     scales (an output of the operation).
//  2. fp4_to_fp8_cols_kernel -- persistent CTAs walk output tiles of
//     128 features x 128 tokens aligned to the OUTPUT, so every output row
//     segment is a full, aligned 128-byte line; each token reads its block's
//     aligned exponent back from the scale written by launch 1.  Codes are
//     converted through a shared-memory tile (double buffered, one barrier
//     per tile) and transposed with byte permutes; the next tile's inputs
//     are prefetched into registers while the current one is converted.
#include "fq_cols_common.cuh"

namespace fq {

constexpr int kTileSlots = tile_slots(kTok / 4);  // 1254
constexpr int kTileWords = kTileSlots * 4;

// ---------------------------------------------------------------- launch 1: block scales

// CTA (exponent word w, 32 consecutive blocks): warp i reduces blocks
// 4i..4i+3 of the chunk -- each lane loads the word w of four tokens per
// block (16 loads in flight), then a byte-wise warp max -- and the CTA writes
// the scales of the 128 features of word w (4 MX columns x 32) for its 32
// blocks: 128 consecutive floats per block, one 128-byte line per warp store.
constexpr int kScaleSlots = 32;

__global__ void __launch_bounds__(kThreads) fp4_to_fp8_cols_scales_kernel(
    const uint8_t *__restrict__ s, int32_t M, int64_t K, const int64_t *__restrict__ offs,
    int32_t G, int k, float *__restrict__ yTs, int32_t *__restrict__ dev_status)
{
    __shared__ int32_t warp_tot[kThreads / 32];
    __shared__ uint32_t smax[kScaleSlots];
    extern __shared__ int32_t dyn[];
    int32_t *off = dyn, *base = dyn + G + 1;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    griddep_wait();  // the previous kernel's outputs (PDL launch)
    griddep_launch_dependents();  // the convert pass may start its set-up now
    const int bad = load_groups(offs, G, M, off, base, warp_tot);
    if (bad && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0 && dev_status)
        atomicOr(dev_status, 1);

    const int32_t nblocks = base[G];
    const int32_t J4 = static_cast<int32_t>(K / 128);  // exponent words per token row
    const int32_t word = blockIdx.x;                     // < J4
    const uint32_t *s32 = reinterpret_cast<const uint32_t *>(s);
    uint32_t *out = reinterpret_cast<uint32_t *>(yTs);

    for (int32_t slot0 = blockIdx.y * kScaleSlots; slot0 < nblocks;
         slot0 += gridDim.y * kScaleSlots) {
        // ---- block maxima: warp wid owns slots slot0 + 4*wid .. +3
        uint32_t v[4][4];
        int32_t bs[4], be[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int32_t slot = slot0 + 4 * wid + i;
            bs[i] = be[i] = 0;
            if (slot < nblocks) {
                const int g = find_last_le(base, 0, G - 1, slot);
                bs[i] = off[g] + (slot - base[g]) * kTok;
                be[i] = min(bs[i] + kTok, off[g + 1]);
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int32_t t = bs[i] + lane + 32 * u;
                v[i][u] = t < be[i] ? __ldg(s32 + static_cast<int64_t>(t) * J4 + word) : 0u;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t m = bytemax4(bytemax4(v[i][0], v[i][1]), bytemax4(v[i][2], v[i][3]));
            const uint32_t b0 = __reduce_max_sync(0xffffffffu, m & 0xFFu);
            const uint32_t b1 = __reduce_max_sync(0xffffffffu, (m >> 8) & 0xFFu);
            const uint32_t b2 = __reduce_max_sync(0xffffffffu, (m >> 16) & 0xFFu);
            const uint32_t b3 = __reduce_max_sync(0xffffffffu, m >> 24);
            if (lane == 0)
                smax[4 * wid + i] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
        }
        __syncthreads();
        // ---- scales: feature 128*word + rr (rr = tid % 128) of the chunk's
        // blocks tid / 128, tid / 128 + 2, ...
        const int rr = tid & 127;
        for (int c = tid >> 7; c < kScaleSlots && slot0 + c < nblocks; c += kThreads / 128)
            out[static_cast<int64_t>(slot0 + c) * K + static_cast<int64_t>(word) * 128 + rr] =
                fp8_block_scale_bits((smax[c] >> (8 * (rr >> 5))) & 0xFFu, k);
        __syncthreads();
    }
}

// One unit: the 32 codes of token tl in MX column j (16 bytes) -> 32 E4M3
// bytes into the FP8 tile, for the block's aligned exponent S and the
// token's own exponent e.
__device__ __forceinline__ void convert_unit(uint32_t *tile, const uint8_t *tab, int tl, int j,
                                             uint4 qv, uint32_t S, uint32_t e, int k)
{
    int u = static_cast<int>(S - e) - k + 6;
    u = min(max(u, 0), kShiftRows - 1);  // u >= 0: S is the max over the block
    const bool nan = S == 0xFFu;
    const uint2 t = *reinterpret_cast<const uint2 *>(tab + 8 * (nan ? kNanRow : u));
    const uint32_t smask = nan ? 0u : 0x80808080u;
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

// Write-out of a converted tile (window W, feature block f): warp w handles
// feature words 4w..4w+3 (m_out), lane%8 tokens 16c..16c+15 (c_out); each
// 16-byte store of a quarter warp fills one 128-byte output line.
template <bool kAligned16>
__device__ __forceinline__ void write_tile(const uint32_t *tile, uint8_t *__restrict__ yT,
                                           int32_t M, int32_t W, int32_t f, int m_out, int c_out)
{
    uint32_t rows[4][4];
#pragma unroll
    for (int qq = 0; qq < 4; qq++) {
        const uint4 v =
            *reinterpret_cast<const uint4 *>(tile + 4 * slot_index(4 * c_out + qq, m_out));
        transpose4x4(v, rows[0][qq], rows[1][qq], rows[2][qq], rows[3][qq]);
    }
    const int32_t t0 = W + 16 * c_out;
    uint8_t *p = yT + (static_cast<int64_t>(f) * 128 + 4 * m_out) * M + t0;
    if (kAligned16 && W + kTok <= M) {
#pragma unroll
        for (int rr = 0; rr < 4; rr++) {
            __stcs(reinterpret_cast<uint4 *>(p),  // evict-first: yT is not re-read
                   make_uint4(rows[rr][0], rows[rr][1], rows[rr][2], rows[rr][3]));
            p += M;
        }
    } else {
        const int32_t We = min(W + kTok, M);
#pragma unroll
        for (int rr = 0; rr < 4; rr++) {
            if (kAligned16 && t0 + 16 <= We) {
                __stcs(reinterpret_cast<uint4 *>(p),
                       make_uint4(rows[rr][0], rows[rr][1], rows[rr][2], rows[rr][3]));
            } else {
                for (int b = 0; b < 16; b++)
                    if (t0 + b < We)
                        p[b] = static_cast<uint8_t>(rows[rr][b >> 2] >> (8 * (b & 3)));
            }
            p += M;
        }
    }
}

// ---------------------------------------------------------------- launch 2: convert + transpose

// Tile (W, f): tokens W..W+127 (W a multiple of 128) x features
// 128f..128f+127.  Thread t converts units (token t/4, column block t%4) and
// (token t/4 + 64, column block t%4): each warp load covers eight token rows
// x 64 contiguous bytes.  For the write-out, warp w handles feature words
// 4w..4w+3 (lane/8 picks the word) and lane%8 picks 16 tokens: each 16-byte
// store of a quarter warp fills one 128-byte output line.  A window that is
// full and lies in one group (the common case) takes a path without
// per-token checks; the next tile's inputs are loaded into the other of two
// register sets while the current tile is converted and written.

struct ColsPrefetch {
    uint4 q0, q1;      // 16 bytes of codes of the two units
    uint32_t e0, e1;   // exponent words (4 MX columns) of the two tokens
    uint32_t s0, s1;   // FP32 block scales (column j) of the two tokens
};

template <bool kAligned16>
__global__ void __launch_bounds__(kThreads, 4) fp4_to_fp8_cols_kernel(
    const uint8_t *__restrict__ q, const uint8_t *__restrict__ s, int32_t M, int64_t K,
    const int64_t *__restrict__ offs, int32_t G, int k, uint8_t *__restrict__ yT,
    const float *__restrict__ yTs)
{
    __shared__ __align__(16) uint8_t tab[kTabRows * 8];
    __shared__ int32_t warp_tot[kThreads / 32];
    extern __shared__ __align__(16) uint32_t dyn_words[];
    uint32_t *tiles = dyn_words;  // [2][kTileWords]
    int32_t *off = reinterpret_cast<int32_t *>(dyn_words + 2 * kTileWords);
    int32_t *base = off + G + 1;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    build_fp8_table(tab);
    load_groups(offs, G, M, off, base, warp_tot);
    // everything above reads only kernel arguments; the codes, exponents and
    // block scales below come from earlier kernels on the stream
    griddep_wait();

    const int32_t nwin = (M + kTok - 1) / kTok;
    const int32_t nfeat = static_cast<int32_t>(K / 128);
    const int32_t ntiles = nwin * nfeat;  // < 2^31, checked on the host
    const int64_t qrow = K / 2, srow = K / 32;
    const int j = tid & 3;     // column block of both units
    const int tl0 = tid >> 2;  // token of unit 0 (unit 1: tl0 + 64)
    const uint32_t *ys32 = reinterpret_cast<const uint32_t *>(yTs);
    // loop-invariant parts of the addresses
    const int64_t qoff0 = static_cast<int64_t>(tl0) * qrow + 16 * j;
    const int64_t qoff1 = qoff0 + 64 * qrow;
    const int64_t soff0 = static_cast<int64_t>(tl0) * srow;
    const int64_t soff1 = soff0 + 64 * srow;
    // write-out: feature word m (4 rows) and tokens 16c..16c+15
    const int m_out = 4 * wid + (lane >> 3);
    const int c_out = lane & 7;
    const int32_t step_w = static_cast<int32_t>(gridDim.x) % nwin;
    const int32_t step_f = static_cast<int32_t>(gridDim.x) / nwin;

    auto prefetch = [&](int32_t win, int32_t f, ColsPrefetch &P) {
        const int32_t W = win * kTok;
        const int g0 = warp_find_last_le(off, G, W);
        const int32_t end0 = off[g0 + 1];
        const uint8_t *qb = q + static_cast<int64_t>(W) * qrow + 64 * f;
        const uint8_t *sp = s + static_cast<int64_t>(W) * srow + 4 * f;
        const uint32_t *yc = ys32 + static_cast<int64_t>(f) * 128 + 32 * j;  // + slot * K
        if (W + kTok <= end0) {  // full window inside group g0 (warp-uniform)
            const int32_t t0 = W + tl0 - off[g0];
            P.q0 = ld_nc_v4(qb + qoff0);
            P.q1 = ld_nc_v4(qb + qoff1);
            P.e0 = __ldg(reinterpret_cast<const uint32_t *>(sp + soff0));
            P.e1 = __ldg(reinterpret_cast<const uint32_t *>(sp + soff1));
            P.s0 = yc[static_cast<int64_t>(base[g0] + (t0 >> 7)) * K];
            P.s1 = yc[static_cast<int64_t>(base[g0] + ((t0 + 64) >> 7)) * K];
        } else {  // window crossing groups or past M
            const int32_t tA = W + tl0, tB = tA + 64;
            P.q0 = tA < M ? ld_nc_v4(qb + qoff0) : make_uint4(0, 0, 0, 0);
            P.q1 = tB < M ? ld_nc_v4(qb + qoff1) : make_uint4(0, 0, 0, 0);
            P.e0 = tA < M ? __ldg(reinterpret_cast<const uint32_t *>(sp + soff0)) : 0u;
            P.e1 = tB < M ? __ldg(reinterpret_cast<const uint32_t *>(sp + soff1)) : 0u;
            const int gA = tA < end0 ? g0 : find_last_le(off, g0, G - 1, min(tA, M - 1));
            const int gB = tB < end0 ? g0 : find_last_le(off, g0, G - 1, min(tB, M - 1));
            P.s0 = tA < M ? yc[static_cast<int64_t>(base[gA] + ((tA - off[gA]) >> 7)) * K] : 0u;
            P.s1 = tB < M ? yc[static_cast<int64_t>(base[gB] + ((tB - off[gB]) >> 7)) * K] : 0u;
        }
    };

    auto convert = [&](uint32_t *tile, int tl, uint4 qv, uint32_t ev, uint32_t sv) {
        convert_unit(tile, tab, tl, j, qv, fp8_block_scale_exponent(sv, k), (ev >> (8 * j)) & 0xFFu,
                     k);
    };

    auto process = [&](int32_t win, int32_t f, const ColsPrefetch &P, uint32_t *tile) {
        const int32_t W = win * kTok;
        const bool full = W + kTok <= M;
        if (full) {
            convert(tile, tl0, P.q0, P.e0, P.s0);
            convert(tile, tl0 + 64, P.q1, P.e1, P.s1);
        } else {
            if (W + tl0 < M)
                convert(tile, tl0, P.q0, P.e0, P.s0);
            if (W + tl0 + 64 < M)
                convert(tile, tl0 + 64, P.q1, P.e1, P.s1);
        }
        __syncthreads();
        write_tile<kAligned16>(tile, yT, M, W, f, m_out, c_out);
    };

    int32_t tau = blockIdx.x;
    if (tau >= ntiles)
        return;
    int32_t win = tau % nwin, f = tau / nwin;
    ColsPrefetch PA, PB;
    prefetch(win, f, PA);
    for (;;) {
        // ---- tile in PA (buffer 0), prefetch the next into PB
        int32_t win2 = win + step_w, f2 = f + step_f;
        if (win2 >= nwin) {
            win2 -= nwin;
            f2++;
        }
        const bool more = tau + static_cast<int32_t>(gridDim.x) < ntiles;
        if (more)
            prefetch(win2, f2, PB);
        process(win, f, PA, tiles);
        if (!more)
            break;
        tau += gridDim.x;
        win = win2;
        f = f2;
        // ---- tile in PB (buffer 1), prefetch the next into PA
        win2 = win + step_w;
        f2 = f + step_f;
        if (win2 >= nwin) {
            win2 -= nwin;
            f2++;
        }
        const bool more2 = tau + static_cast<int32_t>(gridDim.x) < ntiles;
        if (more2)
            prefetch(win2, f2, PA);
        process(win, f, PB, tiles + kTileWords);
        if (!more2)
            break;
        tau += gridDim.x;
        win = win2;
        f = f2;
    }
}

// ---------------------------------------------------------------- single pass (K % 512 == 0)

// One launch, no block-scale pass, warp-specialised.  Work unit: the
// super-tile (128-token window W) x (feature blocks 4F .. 4F+3), whose four
// 128 x 128 tiles are converted one after the other.  Persistent CTAs walk
// the super-tiles window fastest when there are at most kWinFastMax windows
// (the FP8 rows of one feature quad are then written in long runs, and one
// pass over the windows of a feature quad, about 100 KB each, stays well
// inside L2, so the next quad finds the rest of each exponent row there);
// beyond that feature quad fastest: the super-tiles in flight then cover a
// few whole windows, and the other 16-byte slices of their tokens' exponent
// rows, and the neighbouring windows' rows, are read by CTAs running at the
// same time (walked window fastest, a tensor much larger than L2 read its
// exponents from DRAM about three times over).  One 16-byte exponent row
// slice per token holds the UE8M0 exponents of all 16 MX columns of a
// super-tile, so its block maxima are found once for four tiles.
//  * The producer warp (warp 8) issues tensor-memory-access copies into
//    shared memory: each tile's 128 x 64-byte codes into a ring of kStages
//    code stages, and each super-tile's exponent rows of tokens
//    W-128 .. W+255 (three 128-row copies; rows outside the tensor read as
//    zero) into a ring of kExps exponent buffers.  Three tiles before a
//    super-tile starts it computes its block maxima: the 128-token blocks
//    meeting the window are numbered consecutively; the byte-wise max of a
//    block's exponent rows (up to 127 tokens beyond the window on either
//    side come from the neighbouring rows) gives S for the 16 MX columns,
//    from which it stores the shift-table row of every (token of the window,
//    MX column) and, for a block whose first token lies in the window,
//    writes the block's FP32 scales of the super-tile's 512 features (2 KB,
//    contiguous in the block-major scale rows).  The first super-tile's
//    maxima are computed by all nine warps at once.
//  * The eight converting warps wait for a tile's codes (and, on a
//    super-tile's first tile, for its maxima), convert into the FP8 tile as
//    in the two-launch path once every warp has written the previous tile
//    out (named barrier), release the code stage (and, after the fourth
//    tile, the shift-row buffer), meet at a second named barrier and write
//    the tile out transposed.
// Every wait is bounded (mbar_wait); a wait that gives up ends the kernel
// with bit 2 of *dev_status set.
constexpr int32_t kWinFastMax = 512;  // windows walked fastest up to this many
constexpr int kExpBufs = 2;     // shift-row buffers (super-tiles in flight)
constexpr int kConvWarps = kThreads / 32;
constexpr int kThreads1p = kThreads + 32;
constexpr int kCodeBytes = kTok * 64;
constexpr int kExpRowBytes = 16;
constexpr int kExpBytes = 3 * kTok * kExpRowBytes;
constexpr int kSmemAlign = 128;  // tensor-copy destinations
static_assert(kCodeBytes % kSmemAlign == 0 && kExpBytes % kSmemAlign == 0, "aligned buffers");

// Two configurations of the single pass (code stages x exponent buffers):
// kStages x kExps = 4 x 2 up to kWinFastMax windows, 2 x 1 beyond (measured:
// at 131072 x 7168 the 2 x 1 kernel is 6 % faster, at 16384 x 7168 7 %
// slower).  Per shift-row buffer: the shift-table rows of every token of a
// super-tile (uint4: one byte per MX column).
inline size_t cols1_dyn_bytes(int32_t G, int stages, int exps)
{
    return kSmemAlign + static_cast<size_t>(stages) * kCodeBytes +
           static_cast<size_t>(exps) * kExpBytes + static_cast<size_t>(kExpBufs) * kTok * sizeof(uint4) +
           kTileWords * sizeof(uint32_t) + static_cast<size_t>(G + 1) * 2 * sizeof(int32_t);
}

template <bool kAligned16, int kStages, int kExps>
__global__ void __launch_bounds__(kThreads1p, 3) fp4_to_fp8_cols_1pass_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_s,
    int32_t M, int32_t nfeat, const int64_t *__restrict__ offs, int32_t G, int k,
    uint8_t *__restrict__ yT, float *__restrict__ yTs, int32_t *__restrict__ dev_status)
{
    __shared__ __align__(16) uint8_t tab[kTabRows * 8];
    __shared__ int32_t warp_tot[kThreads1p / 32];
    __shared__ __align__(8) uint64_t full_c[kStages];    // code copies landed
    __shared__ __align__(8) uint64_t empty_c[kStages];   // code stage read by every converting warp
    __shared__ __align__(8) uint64_t full_e[kExps];      // exponent copies landed
    __shared__ __align__(8) uint64_t sready[kExpBufs];   // block maxima written
    __shared__ __align__(8) uint64_t empty_e[kExpBufs];  // shift-table rows no longer read
    extern __shared__ __align__(16) uint8_t dyn_raw[];
    uint8_t *codes_ring = dyn_raw + ((kSmemAlign - (smem_u32(dyn_raw) & (kSmemAlign - 1))) &
                                     (kSmemAlign - 1));
    uint8_t *exp_ring = codes_ring + kStages * kCodeBytes;
    uint4 *Uring = reinterpret_cast<uint4 *>(exp_ring + kExps * kExpBytes);  // [kExpBufs][kTok]
    uint32_t *tile = reinterpret_cast<uint32_t *>(Uring + kExpBufs * kTok);    // [kTileWords]
    int32_t *off = reinterpret_cast<int32_t *>(tile + kTileWords);             // [G + 1]
    int32_t *base = off + G + 1;                                              // [G + 1]

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int32_t nwin = (M + kTok - 1) / kTok;
    const int32_t nquad = nfeat >> 2;
    const int32_t nsuper = nwin * nquad;  // < 2^29, checked on the host
    const bool wfast = nwin <= kWinFastMax;
    const int32_t grid = static_cast<int32_t>(gridDim.x);
    // super-tiles of this CTA: blockIdx.x + m * grid, m < my_super
    const int32_t my_super = (nsuper - static_cast<int32_t>(blockIdx.x) + grid - 1) / grid;
    const int32_t my_tiles = 4 * my_super;
    if (tid == 0) {
        for (int i = 0; i < kStages; i++) {
            mbar_init(&full_c[i], 1);
            mbar_init(&empty_c[i], kConvWarps);
        }
        for (int i = 0; i < kExps; i++)
            mbar_init(&full_e[i], 1);
        for (int i = 0; i < kExpBufs; i++) {
            mbar_init(&sready[i], 1);
            mbar_init(&empty_e[i], kConvWarps);
        }
        mbar_init_fence();
    }
    auto super_xy = [&](int32_t m, int32_t &W, int32_t &F) {
        const int32_t sg = static_cast<int32_t>(blockIdx.x) + m * grid;
        W = (wfast ? sg % nwin : sg / nquad) * kTok;
        F = wfast ? sg / nwin : sg % nquad;
    };
    auto issue_exps = [&](int32_t m) {  // one thread: super-tile m of this CTA
        int32_t W, F;
        super_xy(m, W, F);
        const int be = m % kExps;
        uint8_t *dst = exp_ring + be * kExpBytes;
        mbar_arrive_expect_tx(&full_e[be], kExpBytes);
#pragma unroll
        for (int h = 0; h < 3; h++)
            tma_load_2d(dst + h * kTok * kExpRowBytes, &tm_s, 16 * F, W + (h - 1) * kTok,
                        &full_e[be]);
    };
    auto issue_codes = [&](int32_t n) {  // one thread: tile n of this CTA
        int32_t W, F;
        super_xy(n >> 2, W, F);
        const int st = n % kStages;
        mbar_arrive_expect_tx(&full_c[st], kCodeBytes);
        tma_load_2d(codes_ring + st * kCodeBytes, &tm_q, 64 * (4 * F + (n & 3)), W, &full_c[st]);
    };

    build_fp8_table(tab);
    __syncthreads();  // the barriers are initialised before the first copy
    griddep_wait();   // offsets, codes and exponents may come from the previous kernel
    // the first copies need only the window, not the groups: issue them now
    // so that they overlap the group set-up
    if (tid == kThreads) {
        issue_exps(0);
        for (int32_t n = 0; n < kStages - 1 && n < my_tiles; n++)
            issue_codes(n);
    }
    const int bad = load_groups(offs, G, M, off, base, warp_tot);  // ends with a CTA barrier
    if (bad && blockIdx.x == 0 && tid == 0 && dev_status)
        atomicOr(dev_status, 1);

    // block maxima of super-tile m: warp w0 takes the blocks w0, w0 + wstep, ...
    // of those meeting the window; each writes the shift-table rows of the
    // block's tokens in the window and, if the block starts in the window, the
    // block's FP32 scales of the super-tile's 512 features: contiguous in the
    // block's row of yTs, four 16-byte stores per lane
    auto maxima = [&](int32_t m, int w0, int wstep) {
        int32_t W, F;
        super_xy(m, W, F);
        const uint4 *ex = reinterpret_cast<const uint4 *>(exp_ring + (m % kExps) * kExpBytes);
        uint4 *U_of = Uring + (m % kExpBufs) * kTok;
        const int32_t We = min(W + kTok, M);
        const int gW = warp_find_last_le(off, G, W);
        const int32_t blkW = base[gW] + ((W - off[gW]) >> 7);
        const int gL = warp_find_last_le(off, G, We - 1);
        const int32_t nbw = base[gL] + ((We - 1 - off[gL]) >> 7) - blkW + 1;  // <= 128
        int g = gW;
        for (int32_t jb = w0; jb < nbw; jb += wstep) {
            const int32_t b = blkW + jb;
            while (base[g + 1] <= b)  // group of block b (skips empty groups)
                g++;
            const int32_t bs = off[g] + ((b - base[g]) << 7);
            const int32_t be = min(bs + kTok, off[g + 1]);  // W-127 <= bs, be <= W+255
            uint4 m4 = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int32_t t = bs + lane + 32 * u;
                if (t < be) {
                    const uint4 v = ex[t - W + kTok];
                    m4.x = bytemax4(m4.x, v.x);
                    m4.y = bytemax4(m4.y, v.y);
                    m4.z = bytemax4(m4.z, v.z);
                    m4.w = bytemax4(m4.w, v.w);
                }
            }
            auto wmax = [](uint32_t w) {
                return __reduce_max_sync(0xffffffffu, w & 0xFFu) |
                       (__reduce_max_sync(0xffffffffu, (w >> 8) & 0xFFu) << 8) |
                       (__reduce_max_sync(0xffffffffu, (w >> 16) & 0xFFu) << 16) |
                       (__reduce_max_sync(0xffffffffu, w >> 24) << 24);
            };
            const uint4 S = make_uint4(wmax(m4.x), wmax(m4.y), wmax(m4.z), wmax(m4.w));
            for (int32_t t = max(bs, W) + lane; t < min(be, We); t += 32) {
                const uint4 e = ex[t - W + kTok];
                U_of[t - W] = make_uint4(shift_rows4(S.x, e.x, k), shift_rows4(S.y, e.y, k),
                                         shift_rows4(S.z, e.z, k), shift_rows4(S.w, e.w, k));
            }
            if (bs >= W) {
                // feature 512F + x, x = 4 lane + 128 c4 .. + 3: MX column x / 32
                const uint32_t Sw[4] = {S.x, S.y, S.z, S.w};
                uint4 *dst = reinterpret_cast<uint4 *>(
                    yTs + static_cast<int64_t>(b) * (128 * static_cast<int64_t>(nfeat)) +
                    512 * static_cast<int64_t>(F) + 4 * lane);
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) {
                    const int c = 4 * c4 + (lane >> 3);  // MX column of x
                    const uint32_t v = fp8_block_scale_bits((Sw[c >> 2] >> (8 * (c & 3))) & 0xFFu, k);
                    dst[32 * c4] = make_uint4(v, v, v, v);
                }
            }
        }
    };
    // ---- super-tile 0: its maxima with every warp
    const bool ok0 = !__syncthreads_or(!mbar_wait(&full_e[0], 0));
    if (ok0)
        maxima(0, wid, kThreads1p / 32);
    __syncthreads();  // every warp is done with exponent buffer 0
    // with one exponent buffer the copy of super-tile 1 follows the first
    // maxima (with two it is issued in the loop below)
    const int32_t pre_e = kExps == 1 && ok0 && my_super > 1 ? 2 : 1;
    if (tid == kThreads && pre_e == 2)
        issue_exps(1);

    if (wid == kConvWarps) {
        // ================================================= producer warp
        bool ok = ok0;
        int32_t issued_c = min(kStages - 1, my_tiles), issued_e = pre_e;  // copies issued
        int32_t waited_e = ok0 ? 1 : 0;  // exponent copies waited for
        if (ok0 && lane == 0)
            mbar_arrive(&sready[0]);
        for (int32_t n = 0; ok && n < my_tiles; n++) {
            // refill: codes of tile n + kStages - 1 into the stage of tile n - 1
            const int32_t nn = n + kStages - 1;
            if (nn < my_tiles) {
                if (n >= 1) {
                    const int32_t p = n - 1;
                    ok = __all_sync(0xffffffffu, mbar_wait(&empty_c[p % kStages],
                                                           static_cast<uint32_t>(p / kStages) & 1u));
                    if (!ok)
                        break;
                }
                if (lane == 0)
                    issue_codes(nn);
                issued_c++;
            }
            // Super-tile m's maxima are computed on the second tile of
            // super-tile m - 1, three tiles before m starts, into the
            // shift-row buffer super-tile m - 2 released.  Two exponent
            // buffers: super-tile m's exponent copy is issued one tile
            // earlier (into the buffer super-tile m - 2's maxima read).  One
            // buffer: the copy of super-tile m + 1 follows super-tile m's
            // maxima (only this warp reads the exponent buffers after the
            // first super-tile).
            if (kExps == 2 && (n & 3) == 0 && (n >> 2) + 1 < my_super) {
                const int32_t m = (n >> 2) + 1;
                const int32_t p = m - kExpBufs;  // last user of the shift-row buffer
                if (p >= 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&empty_e[p % kExpBufs],
                                                           static_cast<uint32_t>(p / kExpBufs) & 1u));
                    if (!ok)
                        break;
                }
                if (lane == 0)
                    issue_exps(m);
                issued_e++;
            }
            if ((n & 3) == 1) {
                const int32_t m = (n >> 2) + 1;
                if (m < my_super) {
                    const int32_t p = m - kExpBufs;
                    if (kExps == 1 && p >= 0) {
                        ok = __all_sync(0xffffffffu, mbar_wait(&empty_e[p % kExpBufs],
                                                               static_cast<uint32_t>(p / kExpBufs) & 1u));
                        if (!ok)
                            break;
                    }
                    ok = __all_sync(0xffffffffu, mbar_wait(&full_e[m % kExps],
                                                           static_cast<uint32_t>(m / kExps) & 1u));
                    if (!ok)
                        break;
                    waited_e = m + 1;
                    maxima(m, 0, 1);
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&sready[m % kExpBufs]);
                        if (kExps == 1 && m + 1 < my_super)
                            issue_exps(m + 1);
                    }
                    if (kExps == 1 && m + 1 < my_super)
                        issued_e++;
                }
            }
        }
        // every code copy issued is waited for by the converting warps and
        // every exponent copy by this warp; if a wait gave up, report and
        // wait (bounded) for the copies still in flight before the CTA's
        // shared memory is released.  A code stage that took a later copy
        // was released first, so only the last kStages copies can be in
        // flight (waiting on an older one would name a phase the stage has
        // since passed, and run into the time limit)
        if (!ok) {
            if (lane == 0 && dev_status)
                atomicOr(dev_status, 2);
            for (int32_t m = waited_e; m < issued_e; m++)
                mbar_wait(&full_e[m % kExps], static_cast<uint32_t>(m / kExps) & 1u);
            for (int32_t n = max(0, issued_c - kStages); n < issued_c; n++)
                mbar_wait(&full_c[n % kStages], static_cast<uint32_t>(n / kStages) & 1u);
        }
        return;
    }

    // ===================================================== converting warps
    if (!ok0)
        return;  // the producer, which reached no refill, reports it
    const int j = tid & 3;     // MX column of both units
    const int tl0 = tid >> 2;  // token of unit 0 (unit 1: tl0 + 64)
    const int m_out = 4 * wid + (lane >> 3);
    const int c_out = lane & 7;
    const int32_t sg0 = blockIdx.x;  // first super-tile
    int32_t win = wfast ? sg0 % nwin : sg0 / nquad, F = wfast ? sg0 / nwin : sg0 % nquad;
    const int32_t step_w = wfast ? grid % nwin : grid / nquad;
    const int32_t step_F = wfast ? grid / nwin : grid % nquad;
    int st = 0, bf = 0;
    uint32_t ph_c = 0, ph_e = 0;
    for (int32_t n = 0; n < my_tiles; n++) {
        const int i = n & 3;  // tile within the super-tile
        const int32_t W = win * kTok, f = 4 * F + i;
        const bool ok = mbar_wait(&full_c[st], ph_c) && (i != 0 || mbar_wait(&sready[bf], ph_e));
        if (n > 0)
            named_barrier_or(1, kThreads, false);  // the previous tile has been written out
        if (ok) {
            const uint4 *codes = reinterpret_cast<const uint4 *>(codes_ring + st * kCodeBytes);
            const uint32_t *U_w = reinterpret_cast<const uint32_t *>(Uring + bf * kTok);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int tl = tl0 + 64 * h;
                if (W + tl < M)
                    convert_unit_row(tile, tab, tl, j, codes[tl * 4 + j],
                                     (U_w[tl * 4 + i] >> (8 * j)) & 0xFFu);
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty_c[st]);  // this warp is done with the code stage
            if (i == 3)
                mbar_arrive(&empty_e[bf]);  // ... and with the super-tile's exponents
        }
        if (named_barrier_or(1, kThreads, !ok)) {
            // a code or maxima wait gave up; the producer may already be past
            // its last wait, so the converting warps report it themselves
            if (tid == 0 && dev_status)
                atomicOr(dev_status, 2);
            break;
        }
        write_tile<kAligned16>(tile, yT, M, W, f, m_out, c_out);

        if (++st == kStages) {
            st = 0;
            ph_c ^= 1;
        }
        if (i == 3) {
            win += step_w;
            F += step_F;
            if (wfast && win >= nwin) {
                win -= nwin;
                F++;
            } else if (!wfast && F >= nquad) {
                F -= nquad;
                win++;
            }
            if (++bf == kExpBufs) {
                bf = 0;
                ph_e ^= 1;
            }
        }
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

namespace {
bool single_pass_ok(int64_t K)
{
    if (K % 512 != 0)
        return false;
    CUtensorMap probe;  // encoding touches no memory: a dummy 16-byte aligned base
    return encode_tensor_map_2d_u8(&probe, reinterpret_cast<const void *>(uintptr_t{256}),
                                   static_cast<uint64_t>(K / 32), 1, static_cast<uint64_t>(K / 32),
                                   kExpRowBytes, kTok);
}
}  // namespace

extern "C" int fp4_to_fp8_cols_launch_count(int64_t K)
{
    if (K <= 0 || K % 128 != 0)
        return 0;
    return single_pass_ok(K) ? 1 : 2;
}

fq_status fq::launch_fp4_to_fp8_cols(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K,
                                     const int64_t *group_offsets, int32_t G, int exp_offset_k,
                                     uint8_t *yT, float *yT_scale, int64_t cap,
                                     int32_t *dev_status, cudaStream_t st)
{
    const size_t groups_bytes = static_cast<size_t>(G + 1) * 2 * sizeof(int32_t);
    const int64_t work_ctas = ((M + 127) / 128) * (K / 128);

    // single pass: exponent rows of K/32 bytes are a multiple of 16 bytes
    CUtensorMap tm_q, tm_s;
    if (K % 512 == 0 &&
        encode_tensor_map_2d_u8(&tm_q, q, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(M),
                                static_cast<uint64_t>(K / 2), 64, kTok, false) &&
        // a super-tile reads 16 of each exponent row's K/32 bytes; the rest of
        // the 128-byte line belongs to super-tiles a whole pass of windows
        // later, so whole-line promotion would fetch it again from DRAM once
        // the tensor outgrows L2
        encode_tensor_map_2d_u8(&tm_s, s, static_cast<uint64_t>(K / 32), static_cast<uint64_t>(M),
                                static_cast<uint64_t>(K / 32), kExpRowBytes, kTok, false)) {
        const bool large = (M + kTok - 1) / kTok > kWinFastMax;
        const size_t dyn = large ? cols1_dyn_bytes(G, 2, 1) : cols1_dyn_bytes(G, 4, 2);
        auto kern = large ? (M % 16 == 0 ? fp4_to_fp8_cols_1pass_kernel<true, 2, 1>
                                         : fp4_to_fp8_cols_1pass_kernel<false, 2, 1>)
                          : (M % 16 == 0 ? fp4_to_fp8_cols_1pass_kernel<true, 4, 2>
                                         : fp4_to_fp8_cols_1pass_kernel<false, 4, 2>);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(dyn)) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return launch_status();
        const int grid = persistent_grid(kern, kThreads1p, dyn, work_ctas / 4);
        if (launch_pdl(kern, dim3(grid), dim3(kThreads1p), dyn, st, tm_q, tm_s,
                       static_cast<int32_t>(M), static_cast<int32_t>(K / 128), group_offsets, G,
                       exp_offset_k, yT, yT_scale, dev_status) != cudaSuccess)
            return launch_status();
        return launch_status();
    }

    // launch 1: block scales, CTA per (exponent word, 32 blocks)
    const int64_t chunks = (cap + kScaleSlots - 1) / kScaleSlots;
    const dim3 grid1(static_cast<unsigned>(K / 128),
                     static_cast<unsigned>(chunks < 65535 ? chunks : 65535));
    launch_pdl(fp4_to_fp8_cols_scales_kernel, grid1, dim3(kThreads), groups_bytes, st, s,
               static_cast<int32_t>(M), K, group_offsets, G, exp_offset_k, yT_scale, dev_status);
    fq_status rc = launch_status();
    if (rc != FQ_OK)
        return rc;

    // launch 2: convert + transpose (two FP8 tiles + the group arrays)
    const size_t dyn = 2 * kTileWords * sizeof(uint32_t) + groups_bytes;
    if (M % 16 == 0) {
        if (cudaFuncSetAttribute(fp4_to_fp8_cols_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(dyn)) != cudaSuccess)
            return launch_status();
        const int grid = persistent_grid(fp4_to_fp8_cols_kernel<true>, kThreads, dyn, work_ctas);
        if (launch_pdl(fp4_to_fp8_cols_kernel<true>, dim3(grid), dim3(kThreads), dyn, st, q, s,
                       static_cast<int32_t>(M), K, group_offsets, G, exp_offset_k, yT,
                       static_cast<const float *>(yT_scale)) != cudaSuccess)
            return launch_status();
    } else {
        if (cudaFuncSetAttribute(fp4_to_fp8_cols_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(dyn)) != cudaSuccess)
            return launch_status();
        const int grid = persistent_grid(fp4_to_fp8_cols_kernel<false>, kThreads, dyn, work_ctas);
        if (launch_pdl(fp4_to_fp8_cols_kernel<false>, dim3(grid), dim3(kThreads), dyn, st, q, s,
                       static_cast<int32_t>(M), K, group_offsets, G, exp_offset_k, yT,
                       static_cast<const float *>(yT_scale)) != cudaSuccess)
            return launch_status();
    }
    return launch_status();
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
    if (((M + 127) / 128) * (K / 128) > INT32_MAX - 4096)  // tile index is 32-bit
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
    return launch_fp4_to_fp8_cols(q, s, M, K, group_offsets, G, exp_offset_k, yT, yT_scale, cap,
                                  dev_status, static_cast<cudaStream_t>(stream));
}
