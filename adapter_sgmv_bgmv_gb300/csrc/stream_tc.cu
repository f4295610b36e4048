// Streaming rank-r update of 128-row blocks on the tensor cores, shared by the
// expand of the tile path and by the merge / unmerge mode switch:
//
//   expand:  y[rows, :] = bf16(y + s_k * V . B_k)       V = 128 x r   (per tile)
//   merge:   W[c0:c0+128, :] = bf16(W +/- s_k * A_k[c0:c0+128, :] . B_k)
//
// (BEE-30060, Background: the per-request term x_i A_i B_i; VaLoRA blog, section
// 4.4.1: Delta W = A B computed at run time and added to / subtracted from the
// base weight in one pass -- it never exists in memory, only one 128 x 128 block
// of it at a time in TMEM.)
//
// Every block (a tile of the expand, a 128-row slice of W for the merge) is cut
// into 128-column chunks, and the block-major sequence of all chunks is split
// evenly over one CTA per SM: a CTA streams a contiguous run of chunks that
// crosses a block boundary now and then.  Per CTA:
//   - warp 0 (producer) fills a ring of NS stages by TMA alone: per chunk the
//     128 x 128 y / W tile (two 64-column boxes, 128-byte swizzle) and B_k's r x 128
//     block from the B row matrix (dense.cu: pages as consecutive rows; per 64-column
//     half one to three boxes of 64 / 32 / 16 rows, landing in the MMA's N-major
//     swizzled layout), all counted on the stage's one barrier -- so the producer
//     never waits on its own copies;
//   - warp 1 (MMA) issues M = 128, N = 128, K = r MMAs per chunk into one of two
//     TMEM accumulators, so the MMAs of chunk i + 1 overlap the epilogue of chunk i;
//   - warps 11-14 (left) stage the left operand of each block of the CTA's share --
//     V as the in-order sum of the shrink's fp32 partials (coalesced loads, up to 16
//     in flight per thread) or from the caller's fp32 rows, split into bf16
//     hi = bf16(v) and lo = bf16(v - hi) (about 16 significant bits; the MMAs run on
//     both), or A_k's 128 x r slice (M-major; one thread loads it by TMA from the A
//     row matrix) -- into one of two buffers, so the next block's operand is ready
//     before the current block ends (one buffer when a second would cost a stage);
//     the MMA warp frees a buffer with a commit after the block's last MMA.  The
//     producer holds the first block's third tile until its V is staged (V's loads
//     then do not queue behind a full ring of tile loads), and when its share runs
//     on into another block it fetches that block's partials into L2 as it issues
//     the current block's last chunk;
//   - warps 2-9 (epilogue) per chunk read the accumulator (warp w: TMEM lanes
//     32*(w%4).., one 64-column half; both TMEM loads in flight before one wait),
//     add s * acc to its own row of the tile in shared memory (and store that row
//     itself if it is one of a ragged block's last < 8 rows), then arrive on the
//     stage's "tile ready" barrier -- no barrier among the epilogue warps per chunk;
//   - warp 10 (store) stores each ready tile by TMA -- whole 128-row boxes when
//     every row belongs to the block, else 8-row boxes (one swizzle atom each) --
//     and hands the stage back to the producer as soon as the store has read it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace lora {

namespace {

constexpr int kTM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 480;                 // producer, MMA, 8 epilogue, store, 4 left
constexpr int kEpi = 256;
constexpr int kLeftWarp0 = 11;                // warps 11..14 stage the left operand
constexpr int kLeftThreads = 128;
constexpr uint32_t kBox = kTM * 128;          // one 64-column TMA box of 128 rows
constexpr uint32_t kTile = 2 * kBox;          // 128 x 128 bf16
constexpr int kMaxStages = 4;
constexpr int kGateChunk = 2;                 // chunks of the first block issued before its V
constexpr int kShortShare = 24;               // chunks per CTA up to which two left buffers win

enum Left : int { kLeftVParts = 0, kLeftVRows = 1, kLeftAPages = 2 };

struct StreamArgs {
    CUtensorMap map;                          // y (expand) or W (merge), 128-row boxes
    CUtensorMap map8;                         // the same tensor, 8-row boxes
    CUtensorMap bmap[3];                      // the B row matrix, 64 x 16 / 32 / 64 boxes
    CUtensorMap amap[3];                      // merge: the A row matrix, same boxes
    TileParams p;                             // expand: items; merge: unused fields
    MergeParams m;                            // merge only
    int left;
    int n_blocks;
    int n_chunks;                             // chunks per block
    int ctas;                                 // the chunk sequence is split over these
    int rp_max;                               // padded rank that sizes the layout
    int stages;
    int nbuf;                                 // left-operand buffers (2: next block staged ahead)
};

__host__ __device__ inline int rank_pad16(int r) { return (r + 15) & ~15; }
__host__ __device__ inline int v_atoms(int rp) { return (rp + 63) / 64; }

// Shared memory: [left operand] x nbuf [stage s: B | tile] x NS [barriers]
__host__ __device__ inline uint32_t left_bytes(int left, int rp)
{
    return left == kLeftAPages ? uint32_t(rp) * kTM * 2u               // A: rp x 128, M-major
                               : 2u * uint32_t(v_atoms(rp)) * kBox;    // V hi + lo, K-major
}

__host__ __device__ inline uint32_t stage_bytes(int rp) { return uint32_t(rp) * kBN * 2u + kTile; }

__host__ __device__ inline uint32_t stream_smem_bytes(int left, int rp, int stages, int nbuf)
{
    return 1024u + uint32_t(nbuf) * left_bytes(left, rp) + uint32_t(stages) * stage_bytes(rp) +
           192u;   // + barriers
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// What a chunk needs to know about its block.
struct Block {
    int r, rp, row0, nrows;
    float scale;
    int a_row, b_row;                         // first rows in the A / B row matrices
};

__device__ __forceinline__ Block block_info(const StreamArgs &a, int blk)
{
    Block b;
    if (a.left == kLeftAPages) {
        b.r = a.m.rank;
        b.row0 = blk * kTM;
        b.nrows = min(kTM, a.m.d_in - b.row0);
        b.scale = a.m.scale;
        b.a_row = a.m.a_row;
        b.b_row = a.m.b_row;
    } else {
        const TileItem it = tile_item(a.p, blk);
        b.r = it.rank;
        b.row0 = it.row0;
        b.nrows = it.nrows;
        b.scale = it.scale;
        b.a_row = it.a_row;
        b.b_row = it.b_row;
    }
    b.rp = rank_pad16(b.r);
    return b;
}

// Left operand of block blk from the shrink's K-split partials: V as bf16 hi = bf16(v)
// and lo = bf16(v - hi) in K-major 128-byte-swizzled atoms at `dst`, v the in-order
// sum of the ks shares.  A share's partial is 128 rows x rp floats, row-major: piece
// pc (16 bytes) is columns 4 (pc % (rp/4)) .. + 3 of row pc / (rp/4), half of a
// 16-byte chunk of the operand.  Thread vr (0..127) takes pieces vr, vr + 128, ..., so
// each load instruction of a warp reads 512 contiguous bytes.
__device__ __forceinline__ void store_v_piece(uint8_t *dst, int atoms, int q4, int pc, float4 v)
{
    const int row = pc / q4, col = 4 * (pc - row * q4), c = col >> 3;
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
    const float2 b01 = __bfloat1622float2(h01), b23 = __bfloat1622float2(h23);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - b01.x, v.y - b01.y);
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - b23.x, v.w - b23.y);
    const uint32_t off = tc::sw128(uint32_t(row), uint32_t(c & 7)) + 8u * uint32_t((col >> 2) & 1);
    *reinterpret_cast<uint2 *>(dst + (c >> 3) * kBox + off) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
    *reinterpret_cast<uint2 *>(dst + (atoms + (c >> 3)) * kBox + off) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&l01), *reinterpret_cast<const uint32_t *>(&l23));
}

__device__ __forceinline__ void add4(float4 &a, const float4 &b)
{
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// Up to two shares: eight pieces of each in flight at once, summed in place.
__device__ __forceinline__ void stage_v_parts2(const StreamArgs &a, int blk, int rp, int vr, uint8_t *dst)
{
    const int KS = a.p.ksplit, atoms = v_atoms(rp), q4 = rp / 4;
    const float4 *part =
        reinterpret_cast<const float4 *>(a.p.vparts + size_t(blk) * KS * (kVPartBytes / 4)) + vr;
    for (int j0 = 0; j0 < q4; j0 += 8) {
        float4 t0[8], t1[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            if (j0 + jj < q4) {
                t0[jj] = __ldg(part + 128 * (j0 + jj));
                if (KS == 2)
                    t1[jj] = __ldg(part + kVPartBytes / 16 + 128 * (j0 + jj));
            }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
            if (j0 + jj < q4) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);   // 0 + p0 (+ p1): the shares' order
                add4(v, t0[jj]);
                if (KS == 2)
                    add4(v, t1[jj]);
                store_v_piece(dst, atoms, q4, vr + 128 * (j0 + jj), v);
            }
    }
}

// Any number of shares: four shares x four pieces in flight per batch.
__device__ __forceinline__ void stage_v_parts4(const StreamArgs &a, int blk, int rp, int vr, uint8_t *dst)
{
    const int KS = a.p.ksplit, atoms = v_atoms(rp), q4 = rp / 4;
    const float4 *part =
        reinterpret_cast<const float4 *>(a.p.vparts + size_t(blk) * KS * (kVPartBytes / 4)) + vr;
    for (int j0 = 0; j0 < q4; j0 += 4) {
        float4 acc[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            acc[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int ks0 = 0; ks0 < KS; ks0 += 4) {
            float4 t[4][4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    if (ks0 + q < KS)
                        t[q][jj] = __ldg(part + size_t(ks0 + q) * (kVPartBytes / 16) + 128 * (j0 + jj));
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    if (ks0 + q < KS)
                        add4(acc[jj], t[q][jj]);
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
            store_v_piece(dst, atoms, q4, vr + 128 * (j0 + jj), acc[jj]);
    }
}

// kWide: the K-split has at most two shares and V is staged 16 loads deep per thread
// (stage_v_parts2); otherwise four shares x four pieces (stage_v_parts4).  Two
// instantiations, since one kernel holding both would spill.
template <bool kWide>
__global__ void __launch_bounds__(kThreads) k_stream_tc(const __grid_constant__ StreamArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // This CTA's share [g0, g0 + nch) of the block-major chunk sequence.
    const int64_t total = int64_t(a.n_blocks) * a.n_chunks;
    const int g0 = int(total * blockIdx.x / a.ctas);
    const int nch = int(total * (blockIdx.x + 1) / a.ctas) - g0;

    const bool merge = a.left == kLeftAPages;
    const int d_out = merge ? a.m.d_out : a.p.d_out;
    unsigned *status = merge ? a.m.status : a.p.status;
    const int NS = a.stages, NB = a.nbuf;
    const uint32_t sL = base, LB = left_bytes(a.left, a.rp_max);
    const uint32_t sStage0 = sL + uint32_t(NB) * LB;
    const uint32_t sBar = sStage0 + uint32_t(NS) * stage_bytes(a.rp_max);
    // barriers: full[4], empty[4], tready[4], tfull[2], tempty[2], lfull[2], lempty[2]
    const uint32_t full0 = sBar + 8, empty0 = sBar + 40, tready0 = sBar + 72;
    const uint32_t tfull0 = sBar + 104, tempty0 = sBar + 120;
    const uint32_t tmem_slot = sBar + 136;
    const uint32_t lfull0 = sBar + 144, lempty0 = sBar + 160;
    auto stage_b = [&](int i) { return sStage0 + uint32_t(i % NS) * stage_bytes(a.rp_max); };
    auto stage_t = [&](int i) { return stage_b(i) + uint32_t(a.rp_max) * kBN * 2u; };

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(lfull0 + 8 * b, 1);      // left warps (or their TMA bytes)
            mbar_init(lempty0 + 8 * b, 1);     // MMA commit after a block's last MMA
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);       // producer's expect-tx; tile + B bytes
            mbar_init(empty0 + 8 * s, 1);      // the stage's store has read it
            mbar_init(tready0 + 8 * s, kEpi / 32);   // one arrive per epilogue warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);      // MMA commit
            mbar_init(tempty0 + 8 * b, kEpi / 32);   // one arrive per epilogue warp
        }
        fence_mbar_init();
    }
    if (warp == 1)
        tc::tmem_alloc(tmem_slot, 2 * kBN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));
    // Launched as a programmatic dependent: everything above overlapped the previous
    // kernel; y / W, V and the row matrices may be its to write.  Right after the
    // shrink of the same call (early_tiles) that kernel writes only the partials, and
    // it let this one start only once the kernel before it had completed: the
    // producer's y and B loads and the MMA warp (shared memory and TMEM only) go
    // ahead, and the warps that read the partials or write global memory wait.
    if (!(a.left == kLeftVParts && a.p.early_tiles) || warp >= 2)
        grid_dep_wait();
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // A 64-column half of B that lies wholly right of d_out is not loaded; its
        // accumulator columns are never stored.
        if (lane == 0) {
            int cur_blk = -1;
            Block bk{};
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i % NS, u = i / NS;
                if (u > 0)
                    ok = mbar_wait_bounded(empty0 + 8 * s, uint32_t((u - 1) & 1), status,
                                           kDevTimeoutPipe);
                // Two chunks of the first block go out at once; the rest wait until its
                // V is staged, so that the tiles' loads do not queue ahead of V's.  (Only
                // within the first block: the first V is staged whatever the producer
                // does, so this wait always ends.)
                if (ok && i == kGateChunk && !merge && (g0 + i) / a.n_chunks == g0 / a.n_chunks)
                    ok = mbar_wait_bounded(lfull0, 0u, status, kDevTimeoutLoad);
                if (!ok)
                    break;
                const int g = g0 + i, blk = g / a.n_chunks;
                if (blk != cur_blk) {
                    bk = block_info(a, blk);
                    cur_blk = blk;
                }
                const int n0 = (g - blk * a.n_chunks) * kBN;
                const int halves = n0 + 64 < d_out ? 2 : 1;
                mbar_arrive_expect_tx(full0 + 8 * s,
                                      kTile + uint32_t(halves) * uint32_t(bk.rp) * 128u);
                tc::tma_load_2d(stage_t(i), &a.map, n0, bk.row0, full0 + 8 * s);
                tc::tma_load_2d(stage_t(i) + kBox, &a.map, n0 + 64, bk.row0, full0 + 8 * s);
                const uint32_t sb = stage_b(i);
                const uint32_t lbo_b = uint32_t(bk.rp) * 128u;   // N-atom stride of B
                for (int h = 0; h < halves; ++h)
                    tc::for_row_boxes(bk.rp, [&](int off, int m) {
                        tc::tma_load_2d(sb + uint32_t(h) * lbo_b + uint32_t(off) * 128u,
                                        &a.bmap[m], n0 + 64 * h, bk.b_row + off, full0 + 8 * s);
                    });
                // The block's last chunk, and the share goes on into the next block: the
                // next block's partials (long since evicted from L2 by the tile stream)
                // are fetched into L2 now, so that their staging hits L2.
                if (a.left == kLeftVParts && i + 1 < nch && (g + 1) / a.n_chunks != blk) {
                    const int rpn = rank_pad16(tile_item(a.p, blk + 1).rank);
                    for (int ks = 0; ks < a.p.ksplit; ++ks)
                        tc::prefetch_l2(a.p.vparts + (size_t(blk + 1) * a.p.ksplit + ks) * (kVPartBytes / 4),
                                        uint32_t(kTM * rpn * 4));
                }
            }
            grid_dep_launch();   // every load issued: the next kernel may start its set-up
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kTM, kBN, merge ? 1 : 0, 1);
            const int parts = merge ? 1 : 2;
            int cur_blk = -1, seg = -1;
            uint32_t sLb = sL;
            Block bk{};
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i % NS, b = i & 1;
                const int blk = (g0 + i) / a.n_chunks;
                if (blk != cur_blk) {
                    // The previous block's buffer is free once its MMAs complete; then
                    // wait for the new block's left operand.
                    if (seg >= 0)
                        tc::mma_commit(lempty0 + 8 * (seg % NB));
                    bk = block_info(a, blk);
                    cur_blk = blk;
                    ++seg;
                    sLb = sL + uint32_t(seg % NB) * LB;
                    ok = mbar_wait_bounded(lfull0 + 8 * (seg % NB), uint32_t((seg / NB) & 1), status,
                                           kDevTimeoutLoad);
                }
                if (ok)
                    ok = mbar_wait_bounded(full0 + 8 * s, uint32_t((i / NS) & 1), status,
                                           kDevTimeoutLoad);
                if (ok && i >= 2)
                    ok = mbar_wait_bounded(tempty0 + 8 * b, uint32_t(((i >> 1) - 1) & 1), status,
                                           kDevTimeoutPipe);
                if (!ok)
                    break;
                tc::fence_after_sync();
                const uint32_t sb = stage_b(i);
                const uint32_t d = tmem + uint32_t(b * kBN);
                const uint32_t lbo = uint32_t(bk.rp / 8) * 1024u;
                const int atoms = v_atoms(bk.rp);
                for (int part = 0; part < parts; ++part) {
                    for (int kk = 0; kk < bk.rp / 16; ++kk) {
                        uint64_t dl;
                        if (merge)
                            dl = tc::smem_desc_sw128(sLb + uint32_t(kk) * 2048u, lbo, 1024u);
                        else
                            dl = tc::smem_desc_sw128(sLb + uint32_t(part * atoms + (kk >> 2)) * kBox +
                                                         uint32_t(kk & 3) * 32u,
                                                     16u, 1024u);
                        const uint64_t db = tc::smem_desc_sw128(sb + uint32_t(kk) * 2048u, lbo, 1024u);
                        tc::mma_bf16(d, dl, db, idesc, (part > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                tc::mma_commit(tfull0 + 8 * b);
            }
        }
        __syncwarp();
    } else if (warp >= kLeftWarp0) {
        // ------------------------------------------------------------ left operand
        // One block after another of this CTA's share, into buffer seg % NB once the
        // MMAs of the block that last used it have completed (with two buffers, the
        // next block's operand is ready before the current block's last chunk).
        // Every left thread runs the same sequence of named barriers whatever
        // happens: after a failed wait it skips the work, never the barrier.
        const int vr = tid - 32 * kLeftWarp0;   // 0..127: a row of V, or a lane over V's pieces
        const int blk0 = nch > 0 ? g0 / a.n_chunks : 0;
        const int nseg = nch > 0 ? (g0 + nch - 1) / a.n_chunks - blk0 + 1 : 0;
        for (int seg = 0; seg < nseg; ++seg) {
            const int blk = blk0 + seg, buf = seg % NB;
            const Block bk = block_info(a, blk);
            if (ok && seg >= NB)
                ok = mbar_wait_bounded(lempty0 + 8 * buf, uint32_t((seg / NB - 1) & 1), status,
                                       kDevTimeoutPipe);
            ok = __all_sync(0xffffffffu, ok);
            const uint32_t sLb = sL + uint32_t(buf) * LB;
            if (ok && a.left == kLeftVParts) {
                uint8_t *dst = gbase + (sLb - base);
                if (kWide)
                    stage_v_parts2(a, blk, bk.rp, vr, dst);
                else
                    stage_v_parts4(a, blk, bk.rp, vr, dst);
                tc::fence_proxy_async_smem();
            } else if (ok && !merge) {
                // V row vr from the caller's fp32 rows (row stride ldv), as hi / lo.
                const int atoms = v_atoms(bk.rp), nc = bk.rp / 8;
                for (int c0 = 0; c0 < nc; c0 += 4) {
                    float f[4][8];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = 8 * (c0 + u) + e;
                            f[u][e] = (c0 + u < nc && vr < bk.nrows && j < bk.r)
                                          ? __ldg(a.p.v + int64_t(bk.row0 + vr) * a.p.ldv + j)
                                          : 0.f;
                        }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int c = c0 + u;
                        if (c >= nc)
                            break;
                        float back[8];
                        const uint4 hv = pack8(f[u]);
                        unpack8(hv, back);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            f[u][e] -= back[e];
                        const uint32_t off = tc::sw128(uint32_t(vr), uint32_t(c & 7));
                        *reinterpret_cast<uint4 *>(gbase + (sLb - base) + (c >> 3) * kBox + off) = hv;
                        *reinterpret_cast<uint4 *>(gbase + (sLb - base) + (atoms + (c >> 3)) * kBox + off) =
                            pack8(f[u]);
                    }
                }
                tc::fence_proxy_async_smem();
            }
            named_bar_sync(1, kLeftThreads);
            if (vr == 0) {
                if (ok && merge) {
                    // A_k rows row0..row0+127 (M-major: page j of A_k is row j of the
                    // operand, 64 M values per 128-byte row), one 64-row half at a time;
                    // a half wholly below d_in is not loaded (its rows are not stored).
                    const int halves = bk.row0 + 64 < a.m.d_in ? 2 : 1;
                    const uint32_t lbo_a = uint32_t(bk.rp) * 128u;
                    mbar_arrive_expect_tx(lfull0 + 8 * buf, uint32_t(halves) * uint32_t(bk.rp) * 128u);
                    for (int h = 0; h < halves; ++h)
                        tc::for_row_boxes(bk.rp, [&](int off, int m) {
                            tc::tma_load_2d(sLb + uint32_t(h) * lbo_a + uint32_t(off) * 128u, &a.amap[m],
                                            bk.row0 + 64 * h, bk.a_row + off, lfull0 + 8 * buf);
                        });
                } else {
                    mbar_arrive(lfull0 + 8 * buf);
                }
            }
        }
    } else if (warp == 10) {
        // ------------------------------------------------------------ store
        if (lane == 0) {
            int cur_blk = -1;
            Block bk{};
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i % NS;
                ok = mbar_wait_bounded(tready0 + 8 * s, uint32_t((i / NS) & 1), status,
                                       kDevTimeoutPipe);
                if (!ok)
                    break;
                const int g = g0 + i, blk = g / a.n_chunks;
                if (blk != cur_blk) {
                    bk = block_info(a, blk);
                    cur_blk = blk;
                }
                const int n0 = (g - blk * a.n_chunks) * kBN;
                const bool full_rows = merge || bk.nrows == kTM;
                const int rows8 = full_rows ? kTM : (bk.nrows & ~7);
                const uint32_t st = stage_t(i);
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && n0 + 64 >= d_out)   // a box wholly right of the matrix
                        break;
                    const uint32_t src = st + uint32_t(h) * kBox;
                    if (full_rows)
                        tc::tma_store_2d(&a.map, n0 + 64 * h, bk.row0, src);
                    else
                        for (int r8 = 0; r8 < rows8; r8 += 8)
                            tc::tma_store_2d(&a.map8, n0 + 64 * h, bk.row0 + r8,
                                             src + uint32_t(r8) * 128u);
                }
                tc::bulk_commit();
                tc::bulk_wait_read0();
                mbar_arrive(empty0 + 8 * s);
            }
            tc::bulk_wait0();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;                  // TMEM lanes 32*q4 .. 32*q4+31
        const int half = (warp - 2) >> 2;         // columns 64*half .. 64*half+63
        const int row = 32 * q4 + lane;
        int cur_blk = -1;
        Block bk{};
        for (int i = 0; i < nch; ++i) {
            const int s = i % NS, b = i & 1;
            const int g = g0 + i, blk = g / a.n_chunks;
            if (blk != cur_blk) {
                bk = block_info(a, blk);
                cur_blk = blk;
            }
            if (ok)
                ok = mbar_wait_bounded(tfull0 + 8 * b, uint32_t((i >> 1) & 1), status, kDevTimeoutMma);
            if (ok)
                ok = mbar_wait_bounded(full0 + 8 * s, uint32_t((i / NS) & 1), status, kDevTimeoutLoad);
            ok = __all_sync(0xffffffffu, ok);
            const uint32_t st = stage_t(i);
            uint8_t *box = gbase + (st - base) + half * kBox;   // the 64-column TMA box
            if (ok) {
                tc::fence_after_sync();
                uint32_t acc[2][32];
                const uint32_t ta = tmem + (uint32_t(32 * q4) << 16) + uint32_t(b * kBN + 64 * half);
                tc::tmem_ld32_nowait(ta, acc[0]);
                tc::tmem_ld32_nowait(ta + 32, acc[1]);
                tc::tmem_wait_ld();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(tempty0 + 8 * b);      // accumulator b is free for chunk i + 2
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 *ptr = reinterpret_cast<uint4 *>(
                            box + tc::sw128(uint32_t(row), uint32_t(cc * 4 + q)));
                        float t[8];
                        unpack8(*ptr, t);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            t[e] = fmaf(bk.scale, __uint_as_float(acc[cc][q * 8 + e]), t[e]);
                        *ptr = pack8(t);
                    }
                }
                tc::fence_proxy_async_smem();
                // one of a ragged block's last (< 8) rows: this thread wrote its 64
                // columns of it and stores them (the TMA store covers 8-row boxes)
                if (!merge && bk.nrows < kTM && row >= (bk.nrows & ~7) && row < bk.nrows) {
                    const int col = (g - blk * a.n_chunks) * kBN + 64 * half;
                    for (int c = 0; c < 8 && col + 8 * c + 8 <= d_out; ++c)
                        *reinterpret_cast<uint4 *>(a.p.y + int64_t(bk.row0 + row) * a.p.ldy + col +
                                                   8 * c) =
                            *reinterpret_cast<const uint4 *>(box + tc::sw128(uint32_t(row),
                                                                              uint32_t(c)));
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(tready0 + 8 * s);
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 2 * kBN);
    }
}

// Stages and left-operand buffers: as many stages as fit beside one buffer, and a
// second buffer (the next block's operand staged during the current block) only if
// it costs no stage -- a stage fewer lowered the expand's bandwidth more than the
// prefetch saved at a CTA's one or two block changes.  False if two stages do not fit.
bool pick_layout(int left, int rp, int &stages, int &nbuf)
{
    stages = 0;
    for (int ns = kMaxStages; ns >= 2 && !stages; --ns)
        if (stream_smem_bytes(left, rp, ns, 1) <= 227u * 1024u)
            stages = ns;
    if (!stages)
        return false;
    nbuf = stream_smem_bytes(left, rp, stages, 2) <= 227u * 1024u ? 2 : 1;
    return true;
}

int device_sms()
{
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0)
            sms = 148;
    }
    return sms;
}

cudaError_t launch_stream(StreamArgs &a, const void *tensor, uint64_t inner, uint64_t outer,
                          uint64_t row_bytes, cudaStream_t stream)
{
    if (!pick_layout(a.left, a.rp_max, a.stages, a.nbuf))
        return cudaErrorInvalidValue;
    if (!encode_bf16_2d(&a.map, tensor, inner, outer, row_bytes, 64, kTM, true) ||
        !encode_bf16_2d(&a.map8, tensor, inner, outer, row_bytes, 64, 8, true))
        return cudaErrorInvalidValue;
    // One CTA per SM (the shared memory holds no second one), each with an even
    // share of the chunks but at least two, so the pipeline has something to overlap.
    const int64_t total = int64_t(a.n_blocks) * a.n_chunks;
    a.ctas = int(std::max<int64_t>(1, std::min<int64_t>(device_sms(), total / 2)));
    // Short shares (a few chunks per CTA, so the first V and a block change weigh
    // more than a stage of streaming): two left buffers even at the cost of a stage.
    if (a.left != kLeftAPages && a.nbuf == 1 && total / a.ctas <= kShortShare)
        for (int ns = kMaxStages; ns >= 2; --ns)
            if (stream_smem_bytes(a.left, a.rp_max, ns, 2) <= 227u * 1024u) {
                a.stages = ns;
                a.nbuf = 2;
                break;
            }
    static bool configured = false;
    if (!configured) {
        for (auto *k : {k_stream_tc<false>, k_stream_tc<true>}) {
            cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
            if (e != cudaSuccess)
                return e;
        }
        configured = true;
    }
    const bool wide = a.left == kLeftVParts && a.p.ksplit <= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = stream_smem_bytes(a.left, a.rp_max, a.stages, a.nbuf);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return wide ? cudaLaunchKernelEx(&cfg, k_stream_tc<true>, a) : cudaLaunchKernelEx(&cfg, k_stream_tc<false>, a);
}

}  // namespace

cudaError_t launch_expand_tc(const TileParams &p, cudaStream_t stream)
{
    StreamArgs a{};
    a.p = p;
    a.left = p.vmode == 0 ? kLeftVParts : kLeftVRows;
    a.n_blocks = p.n_items;
    a.n_chunks = (p.d_out + kBN - 1) / kBN;
    a.rp_max = rank_pad16(p.max_tile_rank);
    if (!encode_row_maps(a.bmap, p.b_rows, uint64_t(p.d_out), p.b_nrows, p.b_ld))
        return cudaErrorInvalidValue;
    return launch_stream(a, p.y, uint64_t(p.d_out), uint64_t(p.n_rows), uint64_t(p.ldy) * 2u,
                         stream);
}

bool merge_tc_supported(int d_in, int d_out, int rank)
{
    int ns = 0, nb = 0;
    return rank >= 8 && rank <= 128 && d_in > 0 && d_out > 0 &&
           pick_layout(kLeftAPages, rank_pad16(rank), ns, nb);
}

cudaError_t launch_merge_tc(const MergeParams &p, int /*n_split*/, cudaStream_t stream)
{
    StreamArgs a{};
    a.m = p;
    a.left = kLeftAPages;
    a.n_blocks = (p.d_in + kTM - 1) / kTM;
    a.n_chunks = (p.d_out + kBN - 1) / kBN;
    a.rp_max = rank_pad16(p.rank);
    if (!encode_row_maps(a.bmap, p.b_rows, uint64_t(p.d_out), p.b_nrows, p.b_ld) ||
        !encode_row_maps(a.amap, p.a_rows, uint64_t(p.d_in), p.a_nrows, p.a_ld))
        return cudaErrorInvalidValue;
    return launch_stream(a, p.W, uint64_t(p.d_out), uint64_t(p.d_in), uint64_t(p.ldw) * 2u,
                         stream);
}

}  // namespace lora
