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
// One launch does everything: fp4_to_fp8_cols_1pass_kernel, warp-specialised,
// with tensor-memory-access copies into shared memory (described at the
// kernel).  When a token's row of exponents (K/32 bytes) is a multiple of 16
// bytes (K % 512 == 0) the exponent rows come by tensor copy; otherwise by
// tensor copies of four-row groups (M >= 4; the last M % 4 rows patched in
// shared memory) or by 4-byte asynchronous copies (M < 4), and the last
// super-tile of a row of 128-feature blocks may be short.
#include "fq_cols_common.cuh"

namespace fq {

// Output-row alignment of an instance: the rows of yT start on 16-byte
// boundaries (M % 16 == 0), on 4-byte boundaries (M % 4 == 0), or anywhere.
// Tile geometry: the instances for the first two convert the window's 128
// tokens; the last ("extended" tiles) also the next window's first 16
// tokens, so that every row segment they write starts on a 16-byte boundary
// (see write_tile).
__host__ __device__ constexpr int code_rows(bool ext) { return ext ? kTok + 16 : kTok; }
constexpr int tile_words(bool ext) { return tile_slots(code_rows(ext) / 4) * 4; }

// Write-out of a converted tile (window W, feature block f): warp w handles
// feature words 4w..4w+3 (m_out), lane%8 tokens 16c..16c+15 (c_out); each
// 16-byte store of a quarter warp fills one 128-byte output line.  When the
// output rows are not 16-byte aligned (M % 16 != 0):
//  * M % 4 == 0: a row's chunks all start a = 4, 8 or 12 bytes past a
//    16-byte boundary (or on it), and each lane stores its chunk as two
//    8-byte or four 4-byte pieces;
//  * otherwise the tile holds the next window's first 16 tokens too, and
//    each row's segment is shifted to start on a 16-byte boundary, so that
//    it is still written as whole aligned 16-byte blocks (pieces only at the
//    tensor's two ends).
// Earlier designs for such M (16384 x 7040 takes 37 us): single-byte stores,
// 16385 x 7040 in 399 us and 16392 x 7168 in 401 us; then for M % 4 != 0
// aligned blocks between shuffled chunks with 1-8-byte pieces at both ends
// of every row segment, 16385 x 7040 in 82 us (the pieces alone cost 27 us:
// five times the L2 write requests of the aligned case); the extended tiles
// take 56 us.  For M % 4 == 0 the pieces take 45 us and extended tiles 51.
template <int kAlign>
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
    if (kAlign == 4) {
        // rows 4-byte aligned: each lane stores its own chunk in aligned
        // pieces of its row's alignment (16, 8 or 4 bytes); the window's
        // token count is a multiple of 4
        const int n = min(kTok, M - W);
#pragma unroll
        for (int rr = 0; rr < 4; rr++) {
            const int a = static_cast<int>(reinterpret_cast<uintptr_t>(p) & 15);
            const int m = min(16, n - 16 * c_out);  // bytes of the chunk in the window
            if (m == 16 && a == 0) {
                __stcs(reinterpret_cast<uint4 *>(p),
                       make_uint4(rows[rr][0], rows[rr][1], rows[rr][2], rows[rr][3]));
            } else if (m == 16 && (a & 7) == 0) {
                __stcs(reinterpret_cast<uint2 *>(p), make_uint2(rows[rr][0], rows[rr][1]));
                __stcs(reinterpret_cast<uint2 *>(p + 8), make_uint2(rows[rr][2], rows[rr][3]));
            } else {
#pragma unroll
                for (int i = 0; i < 4; i++)
                    if (4 * i < m)
                        __stcs(reinterpret_cast<unsigned int *>(p + 4 * i), rows[rr][i]);
            }
            p += M;
        }
    } else if (kAlign == 1) {
        // row k of yT starts a = (k M + W) mod 16 bytes past a 16-byte
        // boundary: this window writes its tokens from sft = (16 - a) mod 16
        // on as eight aligned 16-byte blocks, the last of which reaches sft
        // tokens into the next window (converted in the same tile, chunk 8);
        // the previous window wrote tokens W .. W + sft - 1 the same way.
        // Block c holds tile tokens sft + 16 c .. + 15: bytes sft .. 15 of
        // chunk c and 0 .. sft - 1 of chunk c + 1.
        uint32_t nx[4][4];
#pragma unroll
        for (int qq = 0; qq < 4; qq++) {
            const uint4 v =
                *reinterpret_cast<const uint4 *>(tile + 4 * slot_index(4 * c_out + 4 + qq, m_out));
            transpose4x4(v, nx[0][qq], nx[1][qq], nx[2][qq], nx[3][qq]);
        }
        const int32_t left = M - W;  // tokens from W to the end of the tensor
        uint8_t *seg = yT + (static_cast<int64_t>(f) * 128 + 4 * m_out) * M + W;
#pragma unroll
        for (int rr = 0; rr < 4; rr++) {
            const int a = static_cast<int>(reinterpret_cast<uintptr_t>(seg) & 15);
            const int sft = (16 - a) & 15;
            uint32_t y[4];
            if (sft == 0) {
#pragma unroll
                for (int i = 0; i < 4; i++)
                    y[i] = rows[rr][i];
            } else {
                bytes_at(rows[rr], nx[rr], sft, y);
            }
            const int t_blk = sft + 16 * c_out;  // the block's first token, from W
            const int len = min(16, left - t_blk);
            if (len >= 16)
                __stcs(reinterpret_cast<uint4 *>(seg + t_blk), make_uint4(y[0], y[1], y[2], y[3]));
            else if (len > 0)
                store_block_range(seg + t_blk, y, 0, len);
            if (W == 0 && c_out == 0 && sft != 0) {
                // the row's first tokens 0 .. sft - 1: bytes a .. 15 of the
                // aligned block before the first
                uint32_t yh[4];
                bytes_at(rows[rr], rows[rr], 16 - a, yh);
                store_block_range(seg - a, yh, a, a + min(sft, left));
            }
            seg += M;
        }
    } else if (W + kTok <= M) {
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
            if (t0 + 16 <= We) {
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

// ---------------------------------------------------------------- the single pass

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
//    maxima are computed by all nine warps at once, one (block, 4-column
//    word) item per warp.
//  * The eight converting warps wait for a tile's codes (and, on a
//    super-tile's first tile, for its maxima), convert each (token, MX
//    column) unit into the FP8 tile through its shift-table row once every
//    warp has written the previous tile out (named barrier), release the code stage (and, after the fourth
//    tile, the shift-row buffer), meet at a second named barrier and write
//    the tile out transposed.
// Every wait is bounded (mbar_wait); a wait that gives up ends the kernel
// with bit 2 of *dev_status set.
constexpr int32_t kWinFastMax = 512;  // windows walked fastest up to this many
constexpr int kExpBufs = 2;     // shift-row buffers (super-tiles in flight)
constexpr int kConvWarps = kThreads / 32;
constexpr int kThreads1p = kThreads + 32;
constexpr int kExpRowBytes = 16;
constexpr int kSmemAlign = 128;  // tensor-copy destinations
// exponent rows of a super-tile: tokens W - 128 .. W - 128 + exp_rows - 1, in
// 128-row copies; the blocks of the tile's tokens reach 127 tokens beyond
// its last (W + 255, or W + 271 with the next window's first 16 tokens)
constexpr int exp_rows(bool ext) { return (ext ? 4 : 3) * kTok; }
static_assert((kTok + 16) * 64 % kSmemAlign == 0, "aligned code stages");

// How a super-tile's exponent rows (tokens W-128 .. W+255, or W+383 when
// the tile takes 16 more tokens; the 16 bytes of its 16 MX columns from
// each) reach shared memory:
//  * kExpRows (K % 512 == 0): three (four) tensor copies of 128 rows x 16
//    bytes.
//  * kExpQuads (K % 512 != 0, M >= 4): a row of 4 nfeat exponent bytes is
//    then not a multiple of 16 bytes, which a tensor map's row pitch must
//    be, but a group of four rows is.  The exponents are viewed as
//    floor(M/4) rows of 16 nfeat bytes.  Row j of a group starts 4 nfeat j
//    bytes into it, so its slice [16F, 16F + 16) lies in the 32 bytes from
//    the 16-byte boundary 16F + floor16(4 nfeat j), at offset 4 nfeat j mod
//    16.  One tensor copy per j brings those 32 bytes of the super-tile's 96
//    (128) groups: buffer [j][group][32 bytes].  Bytes past a row's end belong to
//    the next row (or read as zero); they fall in the columns of a short
//    super-tile's missing feature blocks, whose maxima are never used.  When
//    M % 4 != 0 the last M % 4 tokens lie past the view's rows (read as
//    zero); once a copy that reaches them has landed, the producer warp
//    writes their slices into the buffer with 4-byte loads (patch_tail).
//  * kExpAsync (M < 4): 4-byte asynchronous copies of each row's slice.
constexpr int kExpAsync = 0;
constexpr int kExpRows = 1;
constexpr int kExpQuads = 2;
constexpr int quad_rows(bool ext) { return exp_rows(ext) / 4; }  // four-row groups of a super-tile
constexpr int exp_buf_bytes(int mode, bool ext)
{
    return mode == kExpQuads ? 4 * quad_rows(ext) * 32 : exp_rows(ext) * kExpRowBytes;
}
static_assert(exp_buf_bytes(kExpQuads, true) % kSmemAlign == 0 &&
                  exp_buf_bytes(kExpQuads, false) % kSmemAlign == 0 &&
                  exp_buf_bytes(kExpRows, true) % kSmemAlign == 0 &&
                  exp_buf_bytes(kExpRows, false) % kSmemAlign == 0,
              "aligned buffers");

// Two configurations of the single pass (code stages x exponent buffers):
// kStages x kExps = 4 x 2 up to kWinFastMax windows, 2 x 1 beyond (measured:
// at 131072 x 7168 the 2 x 1 kernel is 6 % faster, at 16384 x 7168 7 %
// slower).  Per shift-row buffer: the shift-table rows of every token of a
// super-tile (uint4: one byte per MX column).
inline size_t cols1_dyn_bytes(int32_t G, int stages, int exps, int exp_mode, bool ext)
{
    return kSmemAlign + static_cast<size_t>(stages) * code_rows(ext) * 64 +
           static_cast<size_t>(exps) * exp_buf_bytes(exp_mode, ext) +
           static_cast<size_t>(kExpBufs) * code_rows(ext) * sizeof(uint4) +
           tile_words(ext) * sizeof(uint32_t) + static_cast<size_t>(G + 1) * 2 * sizeof(int32_t);
}

template <int kAlign, int kStages, int kExps, int kExpMode>
__global__ void __launch_bounds__(kThreads1p, 3) fp4_to_fp8_cols_1pass_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_s,
    const uint8_t *__restrict__ s, int32_t M, int32_t nfeat, const int64_t *__restrict__ offs,
    int32_t G, int k, uint8_t *__restrict__ yT, float *__restrict__ yTs,
    int32_t *__restrict__ dev_status)
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
    constexpr bool kExt = kAlign == 1;             // extended tiles
    constexpr int kRows = code_rows(kExt);         // tokens of a tile
    constexpr int kCodeBytes = kRows * 64;
    constexpr int kExpN = exp_rows(kExt);
    constexpr int kQuadRows = quad_rows(kExt);
    uint8_t *exp_ring = codes_ring + kStages * kCodeBytes;
    constexpr int kExpBuf = exp_buf_bytes(kExpMode, kExt);
    uint4 *Uring = reinterpret_cast<uint4 *>(exp_ring + kExps * kExpBuf);  // [kExpBufs][kRows]
    uint32_t *tile = reinterpret_cast<uint32_t *>(Uring + kExpBufs * kRows);  // [tile_words]
    int32_t *off = reinterpret_cast<int32_t *>(tile + tile_words(kExt));  // [G + 1]
    int32_t *base = off + G + 1;                                              // [G + 1]

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int32_t nwin = (M + kTok - 1) / kTok;
    const int32_t nquad = (nfeat + 3) >> 2;  // the last super-tile of a row may be short
    const int32_t nsuper = nwin * nquad;     // < 2^29, checked on the host
    const int64_t srow = 4 * static_cast<int64_t>(nfeat);  // exponent bytes per token
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
            mbar_init(&full_e[i], kExpMode == kExpAsync ? 32 : 1);
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
    // exponent rows of super-tile m (tokens W-128 .. W+255, 16 bytes each;
    // rows outside the tensor read as zero), called by the whole producer
    // warp in the three modes described above; the asynchronous copies (12
    // rows per lane, columns past the last feature block read as zero) are
    // tracked by the same barrier
    auto issue_exps = [&](int32_t m) {
        int32_t W, F;
        super_xy(m, W, F);
        const int be = m % kExps;
        uint8_t *dst = exp_ring + be * kExpBuf;
        if (kExpMode == kExpRows) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&full_e[be], kExpBuf);
#pragma unroll
                for (int h = 0; h < kExpN / kTok; h++)
                    tma_load_2d(dst + h * kTok * kExpRowBytes, &tm_s, 16 * F,
                                W + (h - 1) * kTok, &full_e[be]);
            }
        } else if (kExpMode == kExpQuads) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&full_e[be], kExpBuf);
#pragma unroll
                for (int j = 0; j < 4; j++)
                    tma_load_2d(dst + j * kQuadRows * 32, &tm_s,
                                16 * F + ((j * static_cast<int32_t>(srow)) & ~15),
                                (W - kTok) / 4, &full_e[be]);
            }
        } else {
            // lanes 4r' .. 4r'+3 copy the four words of one row: eight rows
            // (16 contiguous bytes each) per warp instruction
            const int nw = min(4, nfeat - 4 * F);  // exponent words of the super-tile
            const int w = lane & 3;
            for (int r = lane >> 2; r < kExpN; r += 8) {
                const int32_t t = W - kTok + r;
                const bool rd = t >= 0 && t < M && w < nw;
                const uint8_t *src = rd ? s + static_cast<int64_t>(t) * srow + 16 * F + 4 * w : s;
                cp_async_4(dst + kExpRowBytes * r + 4 * w, src, rd ? 4u : 0u);
            }
            cp_async_mbar_arrive(&full_e[be]);
        }
    };
    // code tile n of this CTA (one thread); a tile past the last feature
    // block of a short super-tile is an empty slot: its stage completes
    // without a copy and nothing is converted or written for it
    auto issue_codes = [&](int32_t n) {
        int32_t W, F;
        super_xy(n >> 2, W, F);
        const int st = n % kStages;
        const int32_t f = 4 * F + (n & 3);
        if (f < nfeat) {
            mbar_arrive_expect_tx(&full_c[st], kCodeBytes);
            tma_load_2d(codes_ring + st * kCodeBytes, &tm_q, 64 * f, W, &full_c[st]);
        } else {
            mbar_arrive(&full_c[st]);
        }
    };

    // four-row groups with M % 4 != 0: the slices of the last M % 4 tokens,
    // which the tensor copies read as zero, written into super-tile m's
    // landed exponent buffer by the calling warp (lane 4i + w: word w of
    // tail token i; words past the row's end are left alone), then ordered
    // before the tensor copies that later refill the buffer
    const int32_t Mq = M & ~3;  // tokens the four-row view covers
    auto patch_tail = [&](int32_t m) {
        int32_t W, F;
        super_xy(m, W, F);
        const int ti = lane >> 2, w = lane & 3;
        const int32_t t = Mq + ti;
        const int32_t r = t - W + kTok;  // row of the super-tile's exponent rows
        if (ti < 3 && t < M && w < min(4, nfeat - 4 * F) && r >= 0 && r < kExpN) {
            const int j = r & 3;
            uint32_t *dst = reinterpret_cast<uint32_t *>(
                exp_ring + (m % kExps) * kExpBuf + j * kQuadRows * 32 + (r >> 2) * 32 +
                ((j * static_cast<int32_t>(srow)) & 15));
            dst[w] = *reinterpret_cast<const uint32_t *>(s + static_cast<int64_t>(t) * srow +
                                                         16 * F + 4 * w);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    };
    // does super-tile m's exponent copy reach the tokens past the view?
    auto reaches_tail = [&](int32_t m) {
        int32_t W, F;
        super_xy(m, W, F);
        return kExpMode == kExpQuads && Mq != M && W - kTok + kExpN > Mq;
    };

    build_fp8_table(tab);
    __syncthreads();  // the barriers are initialised before the first copy
    griddep_wait();   // offsets, codes and exponents may come from the previous kernel
    // the first exponent copy and the first code copies need only the
    // window, not the groups: issue them now so that they overlap the group
    // set-up and the first maxima.  Median timer stamps from the first CTA's
    // entry, 16384 x 7168: the wait returns at 1.1 us, the groups are in
    // shared memory at 2.1 us (one warp for up to 63 groups; 2.9 us with
    // CTA-wide scans), the first maxima are done at 3.5 us (split over all
    // warps; 4.5 us with one warp per block) and the first tile is written
    // at 5.3 us (6.4 us).  The code copies are then already in flight (they
    // used to follow the exponent copy's landing).  65536 x 2048: 41.2 ->
    // 40.5 us; one-call forward cast: 97.4 -> 96.5 us.
    if (wid == kConvWarps) {
        issue_exps(0);
        if (lane == 0)
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
        const uint8_t *eb = exp_ring + (m % kExps) * kExpBuf;
        // exponent slice of token W - 128 + r
        auto exp_row = [&](int32_t r) -> uint4 {
            if (kExpMode != kExpQuads)
                return reinterpret_cast<const uint4 *>(eb)[r];
            const int j = r & 3;
            const uint32_t *p = reinterpret_cast<const uint32_t *>(
                eb + j * kQuadRows * 32 + (r >> 2) * 32 + ((j * static_cast<int32_t>(srow)) & 15));
            return make_uint4(p[0], p[1], p[2], p[3]);
        };
        uint4 *U_of = Uring + (m % kExpBufs) * kRows;
        const int32_t We = min(W + kRows, M);  // the tile's tokens end
        const int gW = warp_find_last_le(off, G, W);
        const int32_t blkW = base[gW] + ((W - off[gW]) >> 7);
        const int gL = warp_find_last_le(off, G, We - 1);
        const int32_t nbw = base[gL] + ((We - 1 - off[gL]) >> 7) - blkW + 1;  // <= kRows
        int g = gW;
        for (int32_t jb = w0; jb < nbw; jb += wstep) {
            const int32_t b = blkW + jb;
            while (base[g + 1] <= b)  // group of block b (skips empty groups)
                g++;
            const int32_t bs = off[g] + ((b - base[g]) << 7);
            const int32_t be = min(bs + kTok, off[g + 1]);  // W-127 <= bs, be <= We+127
            uint4 m4 = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int32_t t = bs + lane + 32 * u;
                if (t < be) {
                    const uint4 v = exp_row(t - W + kTok);
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
                const uint4 e = exp_row(t - W + kTok);
                U_of[t - W] = make_uint4(shift_rows4(S.x, e.x, k), shift_rows4(S.y, e.y, k),
                                         shift_rows4(S.z, e.z, k), shift_rows4(S.w, e.w, k));
            }
            if (bs >= W && (!kExt || bs < W + kTok)) {  // the block starts in the window
                // feature 512F + x, x = 4 lane + 128 c4 .. + 3: MX column x / 32
                const uint32_t Sw[4] = {S.x, S.y, S.z, S.w};
                uint4 *dst = reinterpret_cast<uint4 *>(
                    yTs + static_cast<int64_t>(b) * (128 * static_cast<int64_t>(nfeat)) +
                    512 * static_cast<int64_t>(F) + 4 * lane);
#pragma unroll
                for (int c4 = 0; c4 < 4; c4++) {
                    if (4 * F + c4 >= nfeat)
                        break;  // a short super-tile ends early
                    const int c = 4 * c4 + (lane >> 3);  // MX column of x
                    const uint32_t v = fp8_block_scale_bits((Sw[c >> 2] >> (8 * (c & 3))) & 0xFFu, k);
                    dst[32 * c4] = make_uint4(v, v, v, v);
                }
            }
        }
    };
    // the first super-tile's maxima with every warp: one work item per
    // (block, 4-column word), so that the few blocks meeting the window are
    // spread over all nine warps
    auto maxima_split = [&](int32_t m, int w0, int wstep) {
        int32_t W, F;
        super_xy(m, W, F);
        const uint8_t *eb = exp_ring + (m % kExps) * kExpBuf;
        auto exp_word = [&](int32_t r, int cw) -> uint32_t {
            if (kExpMode != kExpQuads)
                return reinterpret_cast<const uint32_t *>(eb)[4 * r + cw];
            const int j = r & 3;
            const uint32_t *p = reinterpret_cast<const uint32_t *>(
                eb + j * kQuadRows * 32 + (r >> 2) * 32 + ((j * static_cast<int32_t>(srow)) & 15));
            return p[cw];
        };
        uint32_t *U32 = reinterpret_cast<uint32_t *>(Uring + (m % kExpBufs) * kRows);
        const int32_t We = min(W + kRows, M);
        const int gW = warp_find_last_le(off, G, W);
        const int32_t blkW = base[gW] + ((W - off[gW]) >> 7);
        const int gL = warp_find_last_le(off, G, We - 1);
        const int32_t nbw = base[gL] + ((We - 1 - off[gL]) >> 7) - blkW + 1;  // <= kRows
        int g = gW;
        for (int32_t it = w0; it < 4 * nbw; it += wstep) {
            const int32_t b = blkW + (it >> 2);
            const int cw = it & 3;
            while (base[g + 1] <= b)  // group of block b (skips empty groups)
                g++;
            const int32_t bs = off[g] + ((b - base[g]) << 7);
            const int32_t be = min(bs + kTok, off[g + 1]);
            uint32_t mx = 0;
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const int32_t t = bs + lane + 32 * u;
                if (t < be)
                    mx = bytemax4(mx, exp_word(t - W + kTok, cw));
            }
            const uint32_t S = __reduce_max_sync(0xffffffffu, mx & 0xFFu) |
                               (__reduce_max_sync(0xffffffffu, (mx >> 8) & 0xFFu) << 8) |
                               (__reduce_max_sync(0xffffffffu, (mx >> 16) & 0xFFu) << 16) |
                               (__reduce_max_sync(0xffffffffu, mx >> 24) << 24);
            for (int32_t t = max(bs, W) + lane; t < min(be, We); t += 32)
                U32[4 * (t - W) + cw] = shift_rows4(S, exp_word(t - W + kTok, cw), k);
            if (bs >= W && (!kExt || bs < W + kTok) && 4 * F + cw < nfeat) {
                // features 512 F + 128 cw + 4 lane .. + 3: MX column 4 cw + lane / 8
                float *dst = yTs + static_cast<int64_t>(b) * (128 * static_cast<int64_t>(nfeat)) +
                             512 * static_cast<int64_t>(F) + 128 * cw + 4 * lane;
                const uint32_t v = fp8_block_scale_bits((S >> (8 * (lane >> 3))) & 0xFFu, k);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(v, v, v, v);
            }
        }
    };
    // ---- super-tile 0: its maxima with every warp
    const bool ok0 = !__syncthreads_or(!mbar_wait(&full_e[0], 0));
    if (ok0 && reaches_tail(0)) {
        if (wid == kConvWarps)
            patch_tail(0);
        __syncthreads();
    }
    if (ok0)
        maxima_split(0, wid, kThreads1p / 32);
    __syncthreads();  // every warp is done with exponent buffer 0
    // with one exponent buffer the copy of super-tile 1 follows the first
    // maxima (with two it is issued in the loop below)
    const int32_t pre_e = kExps == 1 && ok0 && my_super > 1 ? 2 : 1;
    if (wid == kConvWarps && pre_e == 2)
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
                    if (reaches_tail(m)) {
                        patch_tail(m);
                        __syncwarp();
                    }
                    maxima(m, 0, 1);
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&sready[m % kExpBufs]);
                    if (kExps == 1 && m + 1 < my_super) {
                        issue_exps(m + 1);
                        issued_e++;
                    }
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
    const int tl0 = tid >> 2;  // token of unit 0 (unit h: tl0 + 64 h, below kRows)
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
        const bool real = f < nfeat;  // not the empty slot of a short super-tile
        if (ok && real) {
            const uint4 *codes = reinterpret_cast<const uint4 *>(codes_ring + st * kCodeBytes);
            const uint32_t *U_w = reinterpret_cast<const uint32_t *>(Uring + bf * kRows);
#pragma unroll
            for (int h = 0; h < (kRows + 63) / 64; h++) {
                const int tl = tl0 + 64 * h;
                if ((!kExt || tl < kRows) && W + tl < M)
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
        if (real)
            write_tile<kAlign>(tile, yT, M, W, f, m_out, c_out);

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
    CUtensorMap probe;  // encoding touches no memory: a dummy 16-byte aligned base
    return encode_tensor_map_2d_u8(&probe, reinterpret_cast<const void *>(uintptr_t{256}),
                                   static_cast<uint64_t>(K / 2), 1, static_cast<uint64_t>(K / 2),
                                   64, kTok);
}
}  // namespace

extern "C" int fp4_to_fp8_cols_launch_count(int64_t K)
{
    if (K <= 0 || K % 128 != 0)
        return 0;
    return single_pass_ok(K) ? 1 : 0;
}

namespace {
using Cols1Kernel = void (*)(const CUtensorMap, const CUtensorMap, const uint8_t *, int32_t,
                             int32_t, const int64_t *, int32_t, int, uint8_t *, float *,
                             int32_t *);

// The instances: beyond kWinFastMax windows two code stages and one
// exponent buffer (the exponents then come by rows or four-row groups: M
// >= 4); up to it by exponent mode and output-row alignment.  The extended
// tiles (kAlign 1) keep three CTAs per SM with one exponent buffer, and three
// code stages with the four-row groups (two for M < 4).
template <int kAlign>
Cols1Kernel pick_cols1_large(int mode)
{
    return mode == kExpRows ? fp4_to_fp8_cols_1pass_kernel<kAlign, 2, 1, kExpRows>
                            : fp4_to_fp8_cols_1pass_kernel<kAlign, 2, 1, kExpQuads>;
}

Cols1Kernel pick_cols1_small(int align, int mode, int &stages, int &exps)
{
    if (align != 1) {  // M >= 4: no asynchronous exponent copies
        stages = 4;
        exps = mode == kExpQuads ? 1 : 2;
        if (align == 16)
            return mode == kExpRows ? fp4_to_fp8_cols_1pass_kernel<16, 4, 2, kExpRows>
                                    : fp4_to_fp8_cols_1pass_kernel<16, 4, 1, kExpQuads>;
        return mode == kExpRows ? fp4_to_fp8_cols_1pass_kernel<4, 4, 2, kExpRows>
                                : fp4_to_fp8_cols_1pass_kernel<4, 4, 1, kExpQuads>;
    }
    exps = 1;
    stages = mode == kExpRows ? 4 : (mode == kExpQuads ? 3 : 2);
    return mode == kExpRows    ? fp4_to_fp8_cols_1pass_kernel<1, 4, 1, kExpRows>
           : mode == kExpQuads ? fp4_to_fp8_cols_1pass_kernel<1, 3, 1, kExpQuads>
                               : fp4_to_fp8_cols_1pass_kernel<1, 2, 1, kExpAsync>;
}
}  // namespace

fq_status fq::launch_fp4_to_fp8_cols(const uint8_t *q, const uint8_t *s, int64_t M, int64_t K,
                                     const int64_t *group_offsets, int32_t G, int exp_offset_k,
                                     uint8_t *yT, float *yT_scale, int64_t cap,
                                     int32_t *dev_status, cudaStream_t st)
{
    // single pass; the exponent rows come in one of the three modes
    // described at kExpRows
    CUtensorMap tm_q, tm_s;
    const int mode = K % 512 == 0 ? kExpRows : (M >= 4 ? kExpQuads : kExpAsync);
    const int align = M % 16 == 0 ? 16 : (M % 4 == 0 ? 4 : 1);  // of the rows of yT
    const bool ext = align == 1;
    bool maps = encode_tensor_map_2d_u8(&tm_q, q, static_cast<uint64_t>(K / 2),
                                        static_cast<uint64_t>(M), static_cast<uint64_t>(K / 2), 64,
                                        code_rows(ext), false);
    // a super-tile reads 16 (or 32) of each exponent row's bytes; the rest of
    // the 128-byte line belongs to super-tiles a whole pass of windows later,
    // so whole-line promotion would fetch it again from DRAM once the tensor
    // outgrows L2
    if (maps && mode == kExpRows)
        maps = encode_tensor_map_2d_u8(&tm_s, s, static_cast<uint64_t>(K / 32),
                                       static_cast<uint64_t>(M), static_cast<uint64_t>(K / 32),
                                       kExpRowBytes, kTok, false);
    else if (maps && mode == kExpQuads)
        maps = encode_tensor_map_2d_u8(&tm_s, s, static_cast<uint64_t>(K / 8),
                                       static_cast<uint64_t>(M / 4), static_cast<uint64_t>(K / 8),
                                       32, quad_rows(ext), false);
    else
        tm_s = tm_q;  // not read
    if (maps) {
        // four code stages and two exponent buffers up to kWinFastMax
        // windows, two and one beyond; the four-row groups fill twice the
        // exponent buffer, so they keep one (and three CTAs per SM)
        const bool large = (M + kTok - 1) / kTok > kWinFastMax;
        int stages = 2, exps = 1;
        const Cols1Kernel kern =
            large ? (align == 16  ? pick_cols1_large<16>(mode)
                     : align == 4 ? pick_cols1_large<4>(mode)
                                  : pick_cols1_large<1>(mode))
                  : pick_cols1_small(align, mode, stages, exps);
        const size_t dyn = cols1_dyn_bytes(G, stages, exps, mode, ext);
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(dyn)) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return launch_status();
        const int64_t nsuper = ((M + 127) / 128) * ((K / 128 + 3) / 4);
        const int grid = persistent_grid(kern, kThreads1p, dyn, nsuper);
        if (launch_pdl(kern, dim3(grid), dim3(kThreads1p), dyn, st, tm_q, tm_s, s,
                       static_cast<int32_t>(M), static_cast<int32_t>(K / 128), group_offsets, G,
                       exp_offset_k, yT, yT_scale, dev_status) != cudaSuccess)
            return launch_status();
        return launch_status();
    }

    // no tensor-map encoder in this driver
    set_last_cuda_error(static_cast<int>(cudaErrorNotSupported));
    return FQ_ERR_CUDA;
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
