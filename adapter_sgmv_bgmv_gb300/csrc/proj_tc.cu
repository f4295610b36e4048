// The base projection with the adapter term fused into it, on the tensor cores:
//
//   y[i, :] = bf16( x_i . W + s_k (x_i . A_k) . B_k ),   k = ids[i]
//   y[i, :] = bf16( x_i . W )                           for a released row (id -1)
//
// (S-LoRA article, Batching: the batched base model x W and the separately computed
// x A B, "formula 2"; VaLoRA blog, C2: unmerged inference pays for the adapter term
// beside the base GEMM.  Here the adapter term is more K steps of the same
// accumulator, so y is written once and never read.)
//
// k_proj_prep writes the left operand of every adapter stage before the GEMM runs:
// per chunk (256-row block m, adapter k with rows in it, 64 columns c.. of its
// padded rank) two 256 x 64 bf16 matrices, hi = bf16(s_k v) and lo = bf16(s_k v - hi)
// (v = x A_k, the shrink's fp32 rows; hi + lo carries about 16 significant bits),
// zero in the rows of other adapters, released rows, rows past n and columns past
// the rank.  The GEMM then loads them by TMA like any other operand.
//
// k_proj_tc: persistent kernel over pairs of CTAs (clusters of two on neighbouring
// SMs) that share one tcgen05 MMA of M = 256, N = 256 (cta_group::2): a pair owns
// the tile (256-row block m, 256-column block n); CTA rank c of the pair loads rows
// 128c .. 128c + 127 of the left operand and columns 128c .. 128c + 127 of the right
// one into its own shared memory, and its TMEM holds those 128 rows of the 256 x 256
// fp32 accumulator.  Against one CTA per 128 x 256 tile, every SM fills a third less
// shared memory per MMA flop (32 KB per K block of 64 instead of 48 KB), and the
// ring holds six stages.  Tiles go in groups of 16 row blocks (row blocks fastest
// within a group, so that a 256-column slice of W is fetched once per group and the
// group's x blocks stay in L2).  Per tile the accumulator (two of them, so that one
// tile's epilogue overlaps the next tile's MMAs) takes
//   - the base: d_in / 64 stages of x block (128 x 64 per CTA, K-major, 128-byte
//     swizzle) times W block (64 x 128 per CTA, N-major: two 64-column boxes);
//   - then, for every chunk of block m, two stages (hi, then lo) of K = the chunk's
//     width: the prepared left operand times B_k's rows (N-major boxes from the B
//     row matrix, whose rank-padding rows are zero).
// Warps:
//   0      producer (both CTAs): TMA loads of the CTA's halves of every stage into a
//          ring of 6 (32 KB each); the bytes of both CTAs complete on rank 0's stage
//          barrier, which rank 0's producer arms with the pair's byte count;
//   1      rank 0 only, MMA issuer: tcgen05.mma M = 256, N = 256, K = 16; a commit
//          multicast to both CTAs frees each stage, and another hands each finished
//          accumulator to both CTAs' epilogues;
//   2-5    epilogue (both CTAs): TMEM -> registers -> bf16 -> the warp's 32 x 64
//          slab of y in shared memory (two slabs per warp, in turn) -> one TMA store
//          per slab; the accumulator goes back to rank 0's MMA warp once all eight
//          warps of the pair have read it.  (Per-thread 16-byte stores to 32
//          different rows cost the producer and MMA warps, which share the SM's
//          schedulers with the epilogue warps, ≈ 6 % of the kernel.)
// The producer and the MMA warp read a block's chunk list for the next tile while
// the current tile's base stages run, so that at a tile's end they go straight on.
// Every wait is bounded (1 s); on expiry the status word records it, the stores are
// skipped, and the kernel still ends.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace lora {

namespace {

constexpr int kBM = 128;                            // rows per CTA
constexpr int kPM = 2 * kBM;                        // rows per pair: the MMA's M
constexpr int kBN = 256;                            // columns per tile: the MMA's N
constexpr int kHN = kBN / 2;                        // columns of B in each CTA
constexpr int kBK = 64;
constexpr int kNS = 6;                              // stages in the ring
constexpr uint32_t kAStage = kBM * kBK * 2;         // 16 KB: x block or a prepared half
constexpr uint32_t kBAtom = kBK * 128;              // 8 KB: 64 K rows x 64 columns
constexpr uint32_t kBStage = 2 * kBAtom;            // 16 KB: this CTA's 128 columns
constexpr uint32_t kStage = kAStage + kBStage;      // 32 KB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 2 * kBN;             // two 256-column accumulators
constexpr uint32_t kSlab = 32 * 128;                // 4 KB: 32 rows x 64 columns of y (bf16)
constexpr uint32_t kEpiBytes = 4 * 2 * kSlab;       // two slabs per epilogue warp

struct ProjArgs {
    CUtensorMap xmap;                               // x [n, d_in], 64 x 128 boxes
    CUtensorMap wmap;                               // W [d_in, d_out], 64 x 64 boxes
    CUtensorMap amap;                               // prepared left operands, 64 x 128 boxes
    CUtensorMap ymap;                               // y [n, d_out], 64 x 32 boxes (stores)
    CUtensorMap bmap[3];                            // B row matrix, 64 x 16 / 32 / 64 boxes
    ProjParams p;
};

__host__ __device__ inline uint32_t proj_smem_bytes()
{
    return 1024u + uint32_t(kNS) * kStage + kEpiBytes + 256u;   // + barriers (2 x 6 x 8 B + 5 x 8 B + 4 B)
}

// Tile t of the launch: groups of kGroupM row blocks, each group swept over every
// column block with its row blocks fastest, so that the pairs running at one time
// share a few x blocks and each 256-column slice of W is fetched from DRAM once per
// group (x, W and y stay streaming; W is not assumed to stay in L2).
constexpr int kGroupM = 16;
__device__ __forceinline__ void tile_coords(const ProjParams &p, int t, int &m, int &nb)
{
    const int gsize = kGroupM * p.n_nblk;
    const int g = t / gsize, local = t - g * gsize;
    const int m0 = g * kGroupM;
    const int gm = min(kGroupM, p.n_mblk - m0);
    m = m0 + local % gm;
    nb = local / gm;
}

// The chunks of one row block as far as a warp holds them in registers: the range
// [c0, c1) of the chunk list and its first two chunks (further ones, rare, are read
// when they come).  Filled in two steps -- the range, then (once it has arrived)
// the chunks -- so that the producer and the MMA warp can issue both loads for the
// next tile while the current tile's base stages run.
struct BlockChunks {
    int c0, c1;
    ProjChunk ch[2];
};

__device__ __forceinline__ ProjChunk load_chunk(const ProjParams &p, int i)
{
    const int4 *q = reinterpret_cast<const int4 *>(p.chunks + i);
    const int4 u = __ldg(q), w = __ldg(q + 1);
    return ProjChunk{u.x, u.y, u.z, __int_as_float(u.w), w.x, w.y, w.z, w.w};
}

__device__ __forceinline__ void block_chunks_range(const ProjParams &p, int m, BlockChunks &bc)
{
    bc.c0 = __ldg(p.chunk_off + m);
    bc.c1 = __ldg(p.chunk_off + m + 1);
}

__device__ __forceinline__ void block_chunks_first(const ProjParams &p, BlockChunks &bc)
{
    if (bc.c1 > bc.c0)
        bc.ch[0] = load_chunk(p, bc.c0);
    if (bc.c1 > bc.c0 + 1)
        bc.ch[1] = load_chunk(p, bc.c0 + 1);
}

// The adapter stages of a block: per chunk, hi then lo.  f(chunk index, chunk, half).
template <typename F>
__device__ __forceinline__ void for_chunk_stages(const ProjParams &p, const BlockChunks &bc, F &&f)
{
    for (int i = bc.c0; i < bc.c1; ++i) {
        const ProjChunk ch = i == bc.c0 ? bc.ch[0] : i == bc.c0 + 1 ? bc.ch[1] : load_chunk(p, i);
        for (int half = 0; half < 2; ++half)
            if (!f(i, ch, half))
                return;
    }
}

// ------------------------------------------------------------------ prep

// One CTA per chunk, thread t = row t of the chunk's 256-row block: the row's 64
// values of s_k v[row, c .. c + 64) (zero unless the row is adapter k's and the
// column below its rank) as bf16 hi into row 2 * chunk * 256 + t of the prepared
// matrix and lo into row (2 * chunk + 1) * 256 + t.
__global__ void __launch_bounds__(kPM) k_proj_prep(const __grid_constant__ ProjParams p)
{
    const int i = blockIdx.x, t = threadIdx.x;
    const ProjChunk ch = load_chunk(p, i);
    const int row = ch.m * kPM + t;
    // v is the shrink's: wait for the kernels before.  Then the GEMM may start: before
    // its own wait it reads only x and W, and every kernel before this one has
    // completed by now.
    grid_dep_wait();
    grid_dep_launch();
    const bool mine = row < p.n && __ldg(p.ids + row) == ch.adapter;
    float4 v[16];
    const float *vrow = p.v + int64_t(row) * p.ldv + ch.c;   // ldv: a multiple of 4
#pragma unroll
    for (int q = 0; q < 16; ++q)
        v[q] = (mine && ch.c + 4 * q < ch.rank) ? __ldg(reinterpret_cast<const float4 *>(vrow) + q)
                                                : make_float4(0.f, 0.f, 0.f, 0.f);
    uint4 *hi = reinterpret_cast<uint4 *>(p.a_prep + (int64_t(2 * i) * kPM + t) * kBK);
    uint4 *lo = reinterpret_cast<uint4 *>(p.a_prep + (int64_t(2 * i + 1) * kPM + t) * kBK);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 a = v[2 * q], b = v[2 * q + 1];
        const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            f[e] = (ch.c + 8 * q + e < ch.rank) ? ch.scale * w[e] : 0.f;
        const uint4 h = pack8(f);
        float back[8];
        unpack8(h, back);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            f[e] -= back[e];
        hi[q] = h;
        lo[q] = pack8(f);
    }
}

// ------------------------------------------------------------------ GEMM

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_proj_tc(const __grid_constant__ ProjArgs a)
{
    const ProjParams &p = a.p;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t crank = cluster_ctarank();          // 0 issues the pair's MMAs
    const bool leader = crank == 0;
    const int pair = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);

    const uint32_t sEpi = base + uint32_t(kNS) * kStage;   // the epilogue warps' y slabs
    const uint32_t sBar = sEpi + kEpiBytes;
    // barriers: full[6], empty[6], tfull[2], tempty[2], done; then the TMEM address.
    // full (rank 0's) counts both CTAs' bytes; empty and tfull get rank 0's commits
    // in both CTAs; tempty (rank 0's) one arrival per epilogue warp of the pair.
    const uint32_t full0 = sBar, empty0 = sBar + 8 * kNS;
    const uint32_t tfull0 = sBar + 16 * kNS;
    const uint32_t tempty0 = tfull0 + 16, done = tempty0 + 16, tmem_slot = done + 8;
    auto stage_a = [&](int s) { return base + uint32_t(s) * kStage; };
    auto stage_b = [&](int s) { return base + uint32_t(s) * kStage + kAStage; };
    // rank 0's copy of a barrier of this CTA's layout
    auto at_leader = [&](uint32_t bar) { return map_cluster(bar, 0u); };

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 8);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 1)
        tc::tmem_alloc_pair(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    // Both CTAs' barriers are initialised and their TMEM allocated before anything
    // is addressed across the pair.
    cluster_sync();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));
    // Launched as a programmatic dependent of the prep kernel (early), which lets it
    // start once every kernel before the prep has completed: the base stages' x and W
    // loads and the MMAs (shared memory and TMEM only) go ahead while the prep runs;
    // the producer waits before its first adapter stage (the prepared operands, the
    // B rows), the epilogue before its first store.  Without a prep kernel before
    // it, everything waits here.
    if (!p.early)
        grid_dep_wait();

    const int n_tiles = p.n_mblk * p.n_nblk;
    const int nkb = (p.d_in + kBK - 1) / kBK;
    const int kpre = min(8, nkb - 1);   // base stage at which the next tile's chunks are read
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Boxes that lie past n, d_out or the rank are loaded all the same (zero
        // fill, full byte count), so that both CTAs' byte counts are fixed per stage.
        if (lane == 0) {
            uint32_t g = 0;
            bool waited = !p.early;
            BlockChunks cur{}, nxt{};
            if (pair < n_tiles) {
                int m, nb;
                tile_coords(p, pair, m, nb);
                block_chunks_range(p, m, cur);
                block_chunks_first(p, cur);
            }
            auto next_slot = [&](uint32_t bytes) -> int {
                const int s = int(g % kNS);
                if (g >= kNS)
                    ok = mbar_wait_bounded(empty0 + 8 * s, ((g / kNS) - 1) & 1, p.status,
                                           kDevTimeoutPipe);
                if (ok && leader)
                    mbar_arrive_expect_tx(full0 + 8 * s, 2u * bytes);
                return s;
            };
            for (int tile = pair; tile < n_tiles && ok; tile += npairs) {
                int m, nb;
                tile_coords(p, tile, m, nb);
                const int n0 = nb * kBN + int(crank) * kHN;     // this CTA's columns of B
                const int row0 = m * kPM + int(crank) * kBM;    // this CTA's rows
                const bool more = tile + npairs < n_tiles;
                if (more) {
                    int mn, nbn;
                    tile_coords(p, tile + npairs, mn, nbn);
                    block_chunks_range(p, mn, nxt);
                }
                for (int kb = 0; kb < nkb && ok; ++kb, ++g) {
                    if (kb == kpre && more)
                        block_chunks_first(p, nxt);
                    const int s = next_slot(kStage);
                    if (!ok)
                        break;
                    const uint32_t fb = at_leader(full0 + 8 * s);
                    tc::tma_load_2d_pair(stage_a(s), &a.xmap, kb * kBK, row0, fb);
                    tc::tma_load_2d_pair(stage_b(s), &a.wmap, n0, kb * kBK, fb);
                    tc::tma_load_2d_pair(stage_b(s) + kBAtom, &a.wmap, n0 + 64, kb * kBK, fb);
                }
                for_chunk_stages(p, cur, [&](int i, const ProjChunk &ch, int half) {
                    if (!waited) {
                        grid_dep_wait();
                        waited = true;
                    }
                    const int s = next_slot(kAStage + 2u * uint32_t(ch.kc) * 128u);
                    if (!ok)
                        return false;
                    const uint32_t fb = at_leader(full0 + 8 * s);
                    tc::tma_load_2d_pair(stage_a(s), &a.amap, 0, (2 * i + half) * kPM + int(crank) * kBM, fb);
                    for (int q = 0; q < 2; ++q)
                        tc::for_row_boxes(ch.kc, [&](int off, int mi) {
                            tc::tma_load_2d_pair(stage_b(s) + uint32_t(q) * kBAtom + uint32_t(off) * 128u,
                                                 &a.bmap[mi], n0 + 64 * q, ch.b_row + off, fb);
                        });
                    ++g;
                    return true;
                });
                cur = nxt;
            }
            if (!waited)
                grid_dep_wait();
            grid_dep_launch();   // every load issued: the next kernel may start its set-up
            if (!ok && leader) {
                // Let the loads already issued (both CTAs' bytes complete here) land
                // before the pair can leave.
                for (uint32_t q = g > kNS ? g - kNS : 0; q < g; ++q)
                    mbar_wait_bounded(full0 + 8 * (q % kNS), (q / kNS) & 1, nullptr, 0, 20000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && leader) {
            const uint32_t idesc = tc::idesc_bf16(kPM, kBN, 0, 1);
            uint32_t g = 0;
            int lt = 0;
            BlockChunks cur{}, nxt{};
            if (pair < n_tiles) {
                int m, nb;
                tile_coords(p, pair, m, nb);
                block_chunks_range(p, m, cur);
                block_chunks_first(p, cur);
            }
            for (int tile = pair; tile < n_tiles && ok; tile += npairs, ++lt) {
                const bool more = tile + npairs < n_tiles;
                if (more) {
                    int mn, nbn;
                    tile_coords(p, tile + npairs, mn, nbn);
                    block_chunks_range(p, mn, nxt);
                }
                const int acc = lt & 1;
                if (lt >= 2)
                    ok = mbar_wait_bounded_cluster(tempty0 + 8 * acc, ((lt >> 1) - 1) & 1, p.status,
                                                   kDevTimeoutPipe);
                if (!ok)
                    break;
                tc::fence_after_sync();
                const uint32_t d = tmem + uint32_t(acc * kBN);
                int st = 0;
                auto stage = [&](int kc) -> bool {
                    const int s = int(g % kNS);
                    ok = mbar_wait_bounded(full0 + 8 * s, (g / kNS) & 1, p.status, kDevTimeoutLoad);
                    if (!ok)
                        return false;
                    tc::fence_after_sync();
                    for (int kk = 0; kk < kc / 16; ++kk) {
                        const uint64_t da = tc::smem_desc_sw128(stage_a(s) + 32u * uint32_t(kk), 16u, 1024u);
                        const uint64_t db = tc::smem_desc_sw128(stage_b(s) + 2048u * uint32_t(kk), kBAtom, 1024u);
                        tc::mma_bf16_pair(d, da, db, idesc, (st > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit_pair_both(empty0 + 8 * s);
                    ++st;
                    ++g;
                    return true;
                };
                for (int kb = 0; kb < nkb && ok; ++kb) {
                    if (kb == kpre && more)
                        block_chunks_first(p, nxt);
                    stage(kBK);
                }
                if (ok)
                    for_chunk_stages(p, cur, [&](int, const ProjChunk &ch, int) { return stage(ch.kc); });
                if (!ok)
                    break;
                tc::mma_commit_pair_both(tfull0 + 8 * acc);
                cur = nxt;
            }
            // Every MMA issued so far has completed once this arrives.
            tc::mma_commit_pair(done);
            mbar_wait_bounded(done, 0, nullptr, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;                       // TMEM lanes 32*q4 .. 32*q4+31
        const uint32_t my_slabs = sEpi + uint32_t(warp - 2) * 2u * kSlab;
        int slab_use = 0;
        if (p.early)
            grid_dep_wait();
        int lt = 0;
        for (int tile = pair; tile < n_tiles; tile += npairs, ++lt) {
            int m, nb;
            tile_coords(p, tile, m, nb);
            const int n0 = nb * kBN, row0 = m * kPM + int(crank) * kBM;
            const int acc = lt & 1;
            if (ok)
                ok = mbar_wait_bounded(tfull0 + 8 * acc, (lt >> 1) & 1, p.status, kDevTimeoutMma);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc::fence_after_sync();
            const uint32_t ta = tmem + (uint32_t(32 * q4) << 16) + uint32_t(acc * kBN);
            for (int c0 = 0; c0 < kBN; c0 += 64, ++slab_use) {
                uint32_t v[2][32];
                tc::tmem_ld32_nowait(ta + uint32_t(c0), v[0]);
                tc::tmem_ld32_nowait(ta + uint32_t(c0 + 32), v[1]);
                tc::tmem_wait_ld();
                if (c0 + 64 == kBN) {
                    // the whole accumulator is in registers: it may take the next tile
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader)
                            mbar_arrive(tempty0 + 8 * acc);
                        else
                            mbar_arrive_remote(at_leader(tempty0 + 8 * acc));
                    }
                }
                // Row `lane` of the warp's 32 x 64 slab (128-byte swizzle), once the
                // store issued from it two slabs ago has read it; then one TMA store
                // of the slab (rows past n and columns past d_out are clipped).
                const uint32_t slab = my_slabs + uint32_t(slab_use & 1) * kSlab;
                if (lane == 0)
                    tc::bulk_wait_read1();
                __syncwarp();
                uint8_t *sp = gbase + (slab - base);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            f[e] = __uint_as_float(v[h][8 * u + e]);
                        *reinterpret_cast<uint4 *>(sp + tc::sw128(uint32_t(lane), uint32_t(4 * h + u))) =
                            pack8(f);
                    }
                tc::fence_proxy_async_smem();
                __syncwarp();
                // (a box wholly past n or d_out is not stored at all)
                if (lane == 0) {
                    if (row0 + 32 * q4 < p.n && n0 + c0 < p.d_out)
                        tc::tma_store_2d(&a.ymap, n0 + c0, row0 + 32 * q4, slab);
                    tc::bulk_commit();
                }
            }
        }
        // Every store has finished before the slabs (and the kernel) go away.
        if (lane == 0)
            tc::bulk_wait0();
        __syncwarp();
    }
    tc::fence_before_sync();
    __syncthreads();
    // The pair's MMAs have completed (rank 0 waited for them above) and no arrival or
    // copy is still addressed to the other CTA: TMEM may go, and the CTAs may leave.
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc_pair(tmem, kTmemCols);
    }
}

int device_sms_proj()
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

}  // namespace

cudaError_t launch_proj_prep(const ProjParams &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.n_chunks));
    cfg.blockDim = dim3(kPM);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_proj_prep, p);
}

cudaError_t launch_proj_tc(const ProjParams &p, cudaStream_t stream)
{
    ProjArgs a;
    a.p = p;
    if (!encode_bf16_2d(&a.xmap, p.x, uint64_t(p.d_in), uint64_t(p.n), uint64_t(p.ldx) * 2u, kBK, kBM,
                        true) ||
        !encode_bf16_2d(&a.wmap, p.W, uint64_t(p.d_out), uint64_t(p.d_in), uint64_t(p.ldw) * 2u, 64,
                        kBK, true) ||
        !encode_bf16_2d(&a.ymap, p.y, uint64_t(p.d_out), uint64_t(p.n), uint64_t(p.ldy) * 2u, 64, 32,
                        true))
        return cudaErrorInvalidValue;
    if (p.n_chunks > 0) {
        if (!encode_row_maps(a.bmap, p.b_rows, uint64_t(p.d_out), p.b_nrows, p.b_ld) ||
            !encode_bf16_2d(&a.amap, p.a_prep, uint64_t(kBK), uint64_t(p.n_chunks) * 2u * kPM,
                            uint64_t(kBK) * 2u, kBK, kBM, true))
            return cudaErrorInvalidValue;
    } else {
        for (auto &m : a.bmap)
            m = CUtensorMap{};
        a.amap = CUtensorMap{};
    }
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_proj_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(proj_smem_bytes()));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = proj_smem_bytes();
    cfg.stream = stream;
    // As many pairs as can be resident at once (a pair waits on nothing outside
    // itself, so a larger grid would only run in a second wave).
    static int max_pairs = 0;
    if (!max_pairs) {
        cfg.gridDim = dim3(2u * unsigned(device_sms_proj() / 2));
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, k_proj_tc, &cfg) != cudaSuccess || nc <= 0) {
            cudaGetLastError();
            nc = device_sms_proj() / 2;
        }
        max_pairs = nc;
    }
    const int n_tiles = p.n_mblk * p.n_nblk;
    cfg.gridDim = dim3(2u * unsigned(n_tiles < max_pairs ? n_tiles : max_pairs));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_proj_tc, a);
}

int proj_block_rows() { return kPM; }
int proj_block_cols() { return kBN; }
int proj_chunk_cols() { return kBK; }

}  // namespace lora
