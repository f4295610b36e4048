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
//     block, gathered four pages at a time (tile::gather4) straight into the MMA's
//     N-major swizzled layout, all counted on the stage's one barrier -- so the
//     producer never waits on its own copies;
//   - warp 1 (MMA) issues M = 128, N = 128, K = r MMAs per chunk into one of two
//     TMEM accumulators, so the MMAs of chunk i + 1 overlap the epilogue of chunk i;
//   - warps 2-9 (epilogue) stage the left operand each time the CTA enters a block
//     -- V as the in-order sum of the shrink's fp32 partials or from the caller's
//     fp32 rows, split into bf16 hi = bf16(v) and lo = bf16(v - hi) (about 16
//     significant bits; the MMAs run on both), or A_k's 128 x r slice from the pages
//     (M-major) -- then per chunk read the accumulator (warp w: TMEM lanes
//     32*(w%4).., one 64-column half; both TMEM loads in flight before one wait),
//     add s * acc to the tile in shared memory and store it: whole 128-row boxes by
//     TMA when every row belongs to the block, else 8-row boxes (one swizzle atom
//     each) over the block's rows and the last < 8 rows by the epilogue threads.
//     A stage is released as soon as its store has read shared memory.
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
constexpr int kThreads = 320;                 // producer, MMA, 8 epilogue warps
constexpr int kEpi = 256;
constexpr uint32_t kBox = kTM * 128;          // one 64-column TMA box of 128 rows
constexpr uint32_t kTile = 2 * kBox;          // 128 x 128 bf16
constexpr int kMaxStages = 4;
constexpr int kMaxRank = 128;                 // page-id slots per operand

enum Left : int { kLeftVParts = 0, kLeftVRows = 1, kLeftAPages = 2 };

struct StreamArgs {
    CUtensorMap map;                          // y (expand) or W (merge), 128-row boxes
    CUtensorMap map8;                         // the same tensor, 8-row boxes
    CUtensorMap bmap;                         // the B pool, rows = pages, 64 x 1 boxes
    TileParams p;                             // expand: items; merge: unused fields
    MergeParams m;                            // merge only
    int left;
    int n_blocks;
    int n_chunks;                             // chunks per block
    int ctas;                                 // the chunk sequence is split over these
    int rp_max;                               // padded rank that sizes the layout
    int stages;
};

__host__ __device__ inline int rank_pad16(int r) { return (r + 15) & ~15; }
__host__ __device__ inline int v_atoms(int rp) { return (rp + 63) / 64; }

// Shared memory: [left operand][stage s: B | tile] x NS [barriers][page ids of B, of A]
__host__ __device__ inline uint32_t left_bytes(int left, int rp)
{
    return left == kLeftAPages ? uint32_t(rp) * kTM * 2u               // A: rp x 128, M-major
                               : 2u * uint32_t(v_atoms(rp)) * kBox;    // V hi + lo, K-major
}

__host__ __device__ inline uint32_t stage_bytes(int rp) { return uint32_t(rp) * kBN * 2u + kTile; }

__host__ __device__ inline uint32_t stream_smem_bytes(int left, int rp, int stages)
{
    return 1024u + left_bytes(left, rp) + uint32_t(stages) * stage_bytes(rp) + 128u + 1024u;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// What a chunk needs to know about its block.
struct Block {
    int r, rp, row0, nrows;
    float scale;
    const int32_t *b_pages;
};

__device__ __forceinline__ Block block_info(const StreamArgs &a, int blk)
{
    Block b;
    if (a.left == kLeftAPages) {
        b.r = a.m.rank;
        b.row0 = blk * kTM;
        b.nrows = min(kTM, a.m.d_in - b.row0);
        b.scale = a.m.scale;
        b.b_pages = a.m.b_pages;
    } else {
        const TileItem it = a.p.items[blk];
        b.r = it.rank;
        b.row0 = it.row0;
        b.nrows = it.nrows;
        b.scale = it.scale;
        b.b_pages = a.p.b_pages + size_t(it.adapter) * a.p.max_rank;
    }
    b.rp = rank_pad16(b.r);
    return b;
}

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
    const int NS = a.stages;
    const uint32_t sL = base;
    const uint32_t sStage0 = sL + left_bytes(a.left, a.rp_max);
    const uint32_t sBar = sStage0 + uint32_t(NS) * stage_bytes(a.rp_max);
    // barriers: left, full[4], empty[4], tfull[2], tempty[2]
    const uint32_t bar_left = sBar;
    const uint32_t full0 = sBar + 8, empty0 = sBar + 40;
    const uint32_t tfull0 = sBar + 72, tempty0 = sBar + 88;
    const uint32_t tmem_slot = sBar + 104;
    // The current block's page ids, read once per block: a page id loaded per copy
    // would put a dependent global load in front of every cp.async.
    int32_t *s_bpg = reinterpret_cast<int32_t *>(gbase + (sBar + 128u - base));
    int32_t *s_apg = s_bpg + kMaxRank;
    auto stage_b = [&](int i) { return sStage0 + uint32_t(i % NS) * stage_bytes(a.rp_max); };
    auto stage_t = [&](int i) { return stage_b(i) + uint32_t(a.rp_max) * kBN * 2u; };

    if (tid == 0) {
        mbar_init(bar_left, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);       // producer's expect-tx; tile + B bytes
            mbar_init(empty0 + 8 * s, 1);      // the stage's store has read it
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);      // MMA commit
            mbar_init(tempty0 + 8 * b, kEpi / 32);   // one arrive per epilogue warp
        }
        fence_mbar_init();
    }
    if (merge && tid < a.m.rank)       // one adapter for the whole launch
        s_apg[tid] = a.m.a_pages[tid];
    if (warp == 1)
        tc::tmem_alloc(tmem_slot, 2 * kBN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Rank padding (rows r..rp-1 of B) repeats page 0: it meets zero columns of
        // the left operand.  A 64-column half of B that lies wholly right of d_out
        // is not gathered; its accumulator columns are never stored.
        int cur_blk = -1;
        Block bk{};
        for (int i = 0; i < nch; ++i) {
            const int s = i % NS, u = i / NS;
            if (u > 0)
                ok = mbar_wait_bounded(empty0 + 8 * s, uint32_t((u - 1) & 1), status,
                                       kDevTimeoutPipe) && ok;
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            const int g = g0 + i, blk = g / a.n_chunks;
            if (blk != cur_blk) {
                bk = block_info(a, blk);
                cur_blk = blk;
                // gathers already issued took their page ids when issued
                for (int j = lane; j < bk.rp; j += 32)
                    s_bpg[j] = bk.b_pages[j < bk.r ? j : 0];
                __syncwarp();
            }
            const int n0 = (g - blk * a.n_chunks) * kBN;
            const int halves = n0 + 64 < d_out ? 2 : 1;
            if (lane == 0) {
                mbar_arrive_expect_tx(full0 + 8 * s,
                                      kTile + uint32_t(halves) * uint32_t(bk.rp) * 128u);
                tc::tma_load_2d(stage_t(i), &a.map, n0, bk.row0, full0 + 8 * s);
                tc::tma_load_2d(stage_t(i) + kBox, &a.map, n0 + 64, bk.row0, full0 + 8 * s);
            }
            __syncwarp();
            const uint32_t sb = stage_b(i);
            const uint32_t lbo_b = uint32_t(bk.rp / 8) * 1024u;   // N-atom stride of B
            const int quads = bk.rp / 4;
            for (int q = lane; q < halves * quads; q += 32) {
                const int h = q / quads, j = 4 * (q - h * quads);
                tc::tma_gather4(sb + uint32_t(h) * lbo_b + uint32_t(j >> 3) * 1024u +
                                    uint32_t(j & 7) * 128u,
                                &a.bmap, n0 + 64 * h, s_bpg[j], s_bpg[j + 1], s_bpg[j + 2],
                                s_bpg[j + 3], full0 + 8 * s);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kTM, kBN, merge ? 1 : 0, 1);
            const int parts = merge ? 1 : 2;
            int cur_blk = -1, seg = -1;
            Block bk{};
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i % NS, b = i & 1;
                const int blk = (g0 + i) / a.n_chunks;
                if (blk != cur_blk) {              // wait for the new block's left operand
                    bk = block_info(a, blk);
                    cur_blk = blk;
                    ++seg;
                    ok = mbar_wait_bounded(bar_left, uint32_t(seg & 1), status, kDevTimeoutLoad);
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
                            dl = tc::smem_desc_sw128(sL + uint32_t(kk) * 2048u, lbo, 1024u);
                        else
                            dl = tc::smem_desc_sw128(sL + uint32_t(part * atoms + (kk >> 2)) * kBox +
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
    } else {
        // ------------------------------------------------------------ epilogue
        // Every epilogue thread runs the same sequence of named barriers whatever
        // happens: after a failed (timed-out) wait a warp skips its work, never the
        // barriers, so no other warp is left waiting on it.
        const int et = tid - 64;                 // 0..255
        const int q4 = warp & 3;                  // TMEM lanes 32*q4 .. 32*q4+31
        const int half = (warp - 2) >> 2;         // columns 64*half .. 64*half+63
        const int row = 32 * q4 + lane;
        int cur_blk = -1;
        Block bk{};
        for (int i = 0; i < nch; ++i) {
            const int s = i % NS, b = i & 1;
            const int g = g0 + i, blk = g / a.n_chunks;
            if (blk != cur_blk) {
                // Left operand of the new block.  This thread has seen the commit of
                // every MMA of the previous block, so the buffer is free.
                bk = block_info(a, blk);
                cur_blk = blk;
                if (ok && !merge && et < kTM) {
                    const int vr = et;
                    const int KS = a.left == kLeftVParts ? a.p.ksplit : 1;
                    const int atoms = v_atoms(bk.rp);
                    for (int c = 0; c < bk.rp / 8; ++c) {
                        float f[8], back[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            f[e] = 0.f;
                        if (a.left == kLeftVParts) {
                            for (int ks = 0; ks < KS; ++ks) {
                                const float *src = a.p.vparts +
                                                   (size_t(blk) * KS + ks) * (kVPartBytes / 4) +
                                                   size_t(vr) * bk.rp + 8 * c;
                                const float4 lo4 = *reinterpret_cast<const float4 *>(src);
                                const float4 hi4 = *reinterpret_cast<const float4 *>(src + 4);
                                f[0] += lo4.x; f[1] += lo4.y; f[2] += lo4.z; f[3] += lo4.w;
                                f[4] += hi4.x; f[5] += hi4.y; f[6] += hi4.z; f[7] += hi4.w;
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int j = 8 * c + e;
                                f[e] = (vr < bk.nrows && j < bk.r)
                                           ? a.p.v[int64_t(bk.row0 + vr) * a.p.ldv + j]
                                           : 0.f;
                            }
                        }
                        const uint4 hv = pack8(f);
                        unpack8(hv, back);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            f[e] -= back[e];
                        const uint32_t off = tc::sw128(uint32_t(vr), uint32_t(c & 7));
                        *reinterpret_cast<uint4 *>(gbase + (sL - base) + (c >> 3) * kBox + off) = hv;
                        *reinterpret_cast<uint4 *>(gbase + (sL - base) + (atoms + (c >> 3)) * kBox +
                                                   off) = pack8(f);
                    }
                    tc::fence_proxy_async_smem();
                } else if (ok && merge) {
                    // A_k rows row0..row0+127, column j = page j: M-major, 64-row atoms.
                    const uint32_t lbo_a = uint32_t(bk.rp / 8) * 1024u;
                    for (int q = et; q < bk.rp * 16; q += kEpi) {
                        const int j = q >> 4, c16 = q & 15;
                        const int c = bk.row0 + 8 * c16;
                        const bool valid = j < bk.r && c + 8 <= a.m.d_in;
                        const uint32_t off = uint32_t(c16 >> 3) * lbo_a + uint32_t(j >> 3) * 1024u +
                                             tc::sw128(uint32_t(j & 7), uint32_t(c16 & 7));
                        tc::cp_async16(sL + off,
                                       valid ? a.m.a_pool + int64_t(s_apg[j]) * a.m.a_pw + c
                                             : a.m.a_pool,
                                       valid ? 16u : 0u);
                    }
                    tc::cp_async_commit();
                    tc::cp_async_wait<0>();
                    tc::fence_proxy_async_smem();
                }
                named_bar_sync(1, kEpi);
                if (et == 0)
                    mbar_arrive(bar_left);
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
            }
            named_bar_sync(1, kEpi);
            const int n0 = (g - blk * a.n_chunks) * kBN;
            const bool full_rows = merge || bk.nrows == kTM;
            const int rows8 = full_rows ? kTM : (bk.nrows & ~7);
            if (ok && row >= rows8 && row < bk.nrows) {
                // one of the block's last (< 8) rows: this thread's 64 columns of it
                const int col = n0 + 64 * half;
                for (int c = 0; c < 8 && col + 8 * c + 8 <= d_out; ++c)
                    *reinterpret_cast<uint4 *>(a.p.y + int64_t(bk.row0 + row) * a.p.ldy + col + 8 * c) =
                        *reinterpret_cast<const uint4 *>(box + tc::sw128(uint32_t(row), uint32_t(c)));
            }
            if (et == 0 && ok) {
                for (int h = 0; h < 2; ++h) {
                    if (h == 1 && n0 + 64 >= d_out)   // a box wholly right of the matrix
                        break;
                    const uint32_t src = st + uint32_t(h) * kBox;
                    if (full_rows)
                        tc::tma_store_2d(&a.map, n0 + 64 * h, bk.row0, src);
                    else
                        for (int r8 = 0; r8 < rows8; r8 += 8)
                            tc::tma_store_2d(&a.map8, n0 + 64 * h, bk.row0 + r8, src + uint32_t(r8) * 128u);
                }
                tc::bulk_commit();
            }
            // The stage goes back to the producer once its store has read it (and,
            // in a tile with a ragged end, once the threads storing the last rows
            // have): a stage held longer is one load fewer in flight.
            if (!full_rows && rows8 < bk.nrows)
                named_bar_sync(1, kEpi);
            if (et == 0 && ok) {
                tc::bulk_wait_read0();
                mbar_arrive(empty0 + 8 * s);
            }
        }
        if (et == 0)
            tc::bulk_wait0();
    }
    if (!ok)
        tc::cp_async_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 2 * kBN);
    }
}

int pick_stages(int left, int rp)
{
    for (int ns = kMaxStages; ns >= 2; --ns)
        if (stream_smem_bytes(left, rp, ns) <= 227u * 1024u)
            return ns;
    return 0;
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
                          uint64_t row_bytes, const void *b_pool, int64_t b_pw, int64_t b_pages,
                          cudaStream_t stream)
{
    a.stages = pick_stages(a.left, a.rp_max);
    if (a.stages == 0)
        return cudaErrorInvalidValue;
    if (!encode_bf16_2d(&a.map, tensor, inner, outer, row_bytes, 64, kTM, true) ||
        !encode_bf16_2d(&a.map8, tensor, inner, outer, row_bytes, 64, 8, true) ||
        !encode_bf16_2d(&a.bmap, b_pool, inner, uint64_t(b_pages), uint64_t(b_pw) * 2u, 64, 1, true))
        return cudaErrorInvalidValue;
    // One CTA per SM (the shared memory holds no second one), each with an even
    // share of the chunks but at least two, so the pipeline has something to overlap.
    const int64_t total = int64_t(a.n_blocks) * a.n_chunks;
    a.ctas = int(std::max<int64_t>(1, std::min<int64_t>(device_sms(), total / 2)));
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_stream_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = stream_smem_bytes(a.left, a.rp_max, a.stages);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k_stream_tc, a);
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
    return launch_stream(a, p.y, uint64_t(p.d_out), uint64_t(p.n_rows), uint64_t(p.ldy) * 2u,
                         p.b_pool, p.b_pw, p.b_n_pages, stream);
}

bool merge_tc_supported(int d_in, int d_out, int rank)
{
    return rank >= 8 && rank <= 128 && d_in > 0 && d_out > 0 &&
           pick_stages(kLeftAPages, rank_pad16(rank)) > 0;
}

cudaError_t launch_merge_tc(const MergeParams &p, int /*n_split*/, cudaStream_t stream)
{
    StreamArgs a{};
    a.m = p;
    a.left = kLeftAPages;
    a.n_blocks = (p.d_in + kTM - 1) / kTM;
    a.n_chunks = (p.d_out + kBN - 1) / kBN;
    a.rp_max = rank_pad16(p.rank);
    return launch_stream(a, p.W, uint64_t(p.d_out), uint64_t(p.d_in), uint64_t(p.ldw) * 2u,
                         p.b_pool, p.b_pw, p.b_n_pages, stream);
}

}  // namespace lora
