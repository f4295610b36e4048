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
// Persistent kernel, one CTA per SM, over the tiles (128-row block m, 256-column
// block n) in groups of 16 row blocks (row blocks fastest within a group, so that a
// 256-column slice of W is fetched once per group and the group's x blocks stay in
// L2).  Per tile the accumulator (TMEM,
// 128 lanes x 256 fp32 columns, two of them so that one tile's epilogue overlaps the
// next tile's MMAs) takes
//   - the base: d_in / 64 stages of x block (128 x 64, K-major, 128-byte swizzle)
//     times W block (64 x 256, N-major: four 64-column boxes);
//   - then, for every adapter k with rows in block m, its term as stages of K <= 64:
//     the left operand is s_k v (v = x A_k, the shrink's fp32 rows) split into bf16
//     hi = bf16(s v) and lo = bf16(s v - hi) (about 16 significant bits; the MMAs
//     run on both halves), with the rows of other adapters and released rows zero;
//     the right operand is B_k's rows (N-major boxes from the B row matrix, whose
//     rank-padding rows are zero).
// Warps:
//   0      producer: TMA loads of every stage into a ring of 4 (48 KB each), one
//          barrier per stage (two arrivals: the producer's with the bytes, and a
//          second one -- the producer's own for a base stage, the left-operand
//          warps' for an adapter stage);
//   1      MMA issuer: tcgen05.mma M = 128, N = 256, K = 16, frees each stage with
//          tcgen05.commit, and hands each finished accumulator to the epilogue;
//   2-5    epilogue: TMEM -> registers -> bf16 -> y rows (16-byte stores), then the
//          accumulator goes back to the MMA warp;
//   6-9    left operand of the adapter stages (thread = row of the block).
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

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kNS = 4;                              // stages in the ring
constexpr uint32_t kAStage = kBM * kBK * 2;         // 16 KB: x block or one V half
constexpr uint32_t kBAtom = kBK * 128;              // 8 KB: 64 K rows x 64 columns
constexpr uint32_t kBStage = 4 * kBAtom;            // 32 KB: W block or B_k block
constexpr uint32_t kStage = kAStage + kBStage;      // 48 KB
constexpr int kThreads = 320;
constexpr int kEpiWarp0 = 2;
constexpr int kLeftWarp0 = 6;
constexpr uint32_t kTmemCols = 2 * kBN;             // two 256-column accumulators

struct ProjArgs {
    CUtensorMap xmap;                               // x [n, d_in], 64 x 128 boxes
    CUtensorMap wmap;                               // W [d_in, d_out], 64 x 64 boxes
    CUtensorMap bmap[3];                            // B row matrix, 64 x 16 / 32 / 64 boxes
    ProjParams p;
};

__host__ __device__ inline int rank_pad16(int r) { return (r + 15) & ~15; }

__host__ __device__ inline uint32_t proj_smem_bytes()
{
    return 1024u + uint32_t(kNS) * kStage + 256u;   // + barriers (24 x 8 B + 4 x 8 B + 12 B)
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier over `nthreads` threads that also returns the AND of `v` over them,
// so that every one of them takes the same branch afterwards.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Tile t of the launch: groups of kGroupM row blocks, each group swept over every
// column block with its row blocks fastest, so that the CTAs running at one time
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

// The stages of block m's adapter terms: for each term, hi then lo, each in chunks
// of at most 64 of its padded rank.  f(term index, half, first column, K of stage).
template <typename F>
__device__ __forceinline__ void for_term_stages(const ProjParams &p, int m, F &&f)
{
    const int t0 = __ldg(p.term_off + m), t1 = __ldg(p.term_off + m + 1);
    for (int ti = t0; ti < t1; ++ti) {
        const int rp = rank_pad16(p.terms[ti].rank);
        for (int half = 0; half < 2; ++half)
            for (int c = 0; c < rp; c += kBK)
                if (!f(ti, half, c, min(kBK, rp - c)))
                    return;
    }
}

__global__ void __launch_bounds__(kThreads, 1) k_proj_tc(const __grid_constant__ ProjArgs a)
{
    const ProjParams &p = a.p;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const uint32_t sBar = base + uint32_t(kNS) * kStage;
    // barriers: full[4], empty[4], vgo[4], tfull[2], tempty[2], done; then the TMEM
    // address.  vgo[s]: the producer found slot s free for an adapter stage, so the
    // left-operand warps may write its A half.  (They cannot wait on empty[s]
    // themselves: they skip the base stages, and a parity wait more than one phase
    // ahead of the barrier would pass early.)
    const uint32_t full0 = sBar, empty0 = sBar + 8 * kNS, vgo0 = sBar + 16 * kNS;
    const uint32_t tfull0 = sBar + 24 * kNS;
    const uint32_t tempty0 = tfull0 + 16, done = tempty0 + 16, tmem_slot = done + 8;
    auto stage_a = [&](int s) { return base + uint32_t(s) * kStage; };
    auto stage_b = [&](int s) { return base + uint32_t(s) * kStage + kAStage; };

    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(full0 + 8 * s, 2);
            mbar_init(empty0 + 8 * s, 1);
            mbar_init(vgo0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 4);
        }
        mbar_init(done, 1);
        fence_mbar_init();
    }
    if (warp == 1)
        tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(gbase + (tmem_slot - base));
    // Launched as a programmatic dependent of the shrink that wrote v: everything
    // above overlapped its tail.
    grid_dep_wait();

    const int n_tiles = p.n_mblk * p.n_nblk;
    const int nkb = (p.d_in + kBK - 1) / kBK;
    bool ok = true;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t g = 0;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                int m, nb;
                tile_coords(p, tile, m, nb);
                const int n0 = nb * kBN, row0 = m * kBM;
                const int natoms = min(4, (p.d_out - n0 + 63) / 64);   // 64-column boxes inside d_out
                for (int kb = 0; kb < nkb && ok; ++kb, ++g) {
                    const int s = int(g % kNS);
                    if (g >= kNS)
                        ok = mbar_wait_bounded(empty0 + 8 * s, ((g / kNS) - 1) & 1, p.status,
                                               kDevTimeoutPipe);
                    if (!ok)
                        break;
                    mbar_arrive_expect_tx(full0 + 8 * s, kAStage + uint32_t(natoms) * kBAtom);
                    tc::tma_load_2d(stage_a(s), &a.xmap, kb * kBK, row0, full0 + 8 * s);
                    for (int q = 0; q < natoms; ++q)
                        tc::tma_load_2d(stage_b(s) + uint32_t(q) * kBAtom, &a.wmap, n0 + 64 * q, kb * kBK,
                                        full0 + 8 * s);
                    mbar_arrive(full0 + 8 * s);
                }
                for_term_stages(p, m, [&](int ti, int, int c, int kc) {
                    const int s = int(g % kNS);
                    if (g >= kNS)
                        ok = mbar_wait_bounded(empty0 + 8 * s, ((g / kNS) - 1) & 1, p.status,
                                               kDevTimeoutPipe);
                    if (!ok)
                        return false;
                    mbar_arrive(vgo0 + 8 * s);   // the left-operand warps may fill its A half
                    const int brow = p.terms[ti].b_row + c;
                    mbar_arrive_expect_tx(full0 + 8 * s, uint32_t(natoms) * uint32_t(kc) * 128u);
                    for (int q = 0; q < natoms; ++q)
                        tc::for_row_boxes(kc, [&](int off, int mi) {
                            tc::tma_load_2d(stage_b(s) + uint32_t(q) * kBAtom + uint32_t(off) * 128u,
                                            &a.bmap[mi], n0 + 64 * q, brow + off, full0 + 8 * s);
                        });
                    ++g;
                    return true;
                });
            }
            grid_dep_launch();   // every load issued: the next kernel may start its set-up
            if (!ok) {
                // Let the loads already issued land before this CTA can leave.
                for (uint32_t q = g > kNS ? g - kNS : 0; q < g; ++q)
                    mbar_wait_bounded(full0 + 8 * (q % kNS), (q / kNS) & 1, nullptr, 0, 20000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kBM, kBN, 0, 1);
            uint32_t g = 0;
            int lt = 0;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++lt) {
                int m, nb;
                tile_coords(p, tile, m, nb);
                const int acc = lt & 1;
                if (lt >= 2)
                    ok = mbar_wait_bounded(tempty0 + 8 * acc, ((lt >> 1) - 1) & 1, p.status,
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
                        tc::mma_bf16(d, da, db, idesc, (st > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(empty0 + 8 * s);
                    ++st;
                    ++g;
                    return true;
                };
                for (int kb = 0; kb < nkb && ok; ++kb)
                    stage(kBK);
                if (ok)
                    for_term_stages(p, m, [&](int, int, int, int kc) { return stage(kc); });
                if (!ok)
                    break;
                tc::mma_commit(tfull0 + 8 * acc);
            }
            // Every MMA issued so far has completed once this arrives.
            tc::mma_commit(done);
            mbar_wait_bounded(done, 0, nullptr, 0);
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0 && warp < kLeftWarp0) {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;                       // TMEM lanes 32*q4 .. 32*q4+31
        const int r_in = 32 * q4 + lane;               // this thread's row of the tile
        int lt = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++lt) {
            int m, nb;
            tile_coords(p, tile, m, nb);
            const int n0 = nb * kBN, row0 = m * kBM;
            const int acc = lt & 1;
            if (ok)
                ok = mbar_wait_bounded(tfull0 + 8 * acc, (lt >> 1) & 1, p.status, kDevTimeoutMma);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok)
                break;
            tc::fence_after_sync();
            const bool row_ok = row0 + r_in < p.n;
            uint16_t *yrow = p.y + int64_t(row0 + r_in) * p.ldy + n0;
            const uint32_t ta = tmem + (uint32_t(32 * q4) << 16) + uint32_t(acc * kBN);
            for (int c0 = 0; c0 < kBN; c0 += 64) {
                uint32_t v[2][32];
                tc::tmem_ld32_nowait(ta + uint32_t(c0), v[0]);
                tc::tmem_ld32_nowait(ta + uint32_t(c0 + 32), v[1]);
                tc::tmem_wait_ld();
                if (c0 + 64 == kBN) {
                    // the whole accumulator is in registers: it may take the next tile
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(tempty0 + 8 * acc);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int col = c0 + 32 * h + 8 * u;
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            f[e] = __uint_as_float(v[h][8 * u + e]);
                        if (row_ok && n0 + col < p.d_out)
                            *reinterpret_cast<uint4 *>(yrow + col) = pack8(f);
                    }
            }
        }
    } else {
        // ------------------------------------------------------------ left operand
        // Thread vr writes row vr of every adapter stage's A half: s_k v[row, c..c+kc)
        // as bf16 hi or lo (zero for rows of other adapters, released rows and rows
        // past n), in the K-major 128-byte-swizzled layout of the x blocks.
        // The four warps agree on every decision (named_bar_and), so that they all run
        // the same sequence of named barriers whatever happens.
        const int vr = tid - 32 * kLeftWarp0;
        uint32_t g = 0;
        uint32_t uses[kNS] = {0, 0, 0, 0};   // adapter stages this thread has filled, per slot
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
            int m, nb;
            tile_coords(p, tile, m, nb);
            const int row0 = m * kBM;
            const int row = row0 + vr;
            const int id = (p.ids && row < p.n) ? __ldg(p.ids + row) : -1;
            g += uint32_t(nkb);
            for_term_stages(p, m, [&](int ti, int half, int c, int kc) {
                const int s = int(g % kNS);
                // The producer arrives on vgo[s] once per adapter stage in slot s, and
                // the next such arrival needs this stage consumed first: never more
                // than one phase ahead, so the parity of this slot's count is exact.
                uint32_t u = 0;
#pragma unroll
                for (int q = 0; q < kNS; ++q)
                    if (q == s)
                        u = uses[q]++;
                ok = mbar_wait_bounded(vgo0 + 8 * s, u & 1, p.status, kDevTimeoutPipe);
                ok = named_bar_and(1, 128, ok);
                if (ok) {
                    const ProjTerm tm = p.terms[ti];
                    const bool mine = id == tm.adapter;
                    const float* vrow = p.v + int64_t(row) * p.ldv;
                    uint8_t *dst = gbase + (stage_a(s) - base);
                    for (int q = 0; q < kc / 8; ++q) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = c + 8 * q + e;
                            f[e] = (mine && j < tm.rank) ? tm.scale * __ldg(vrow + j) : 0.f;
                        }
                        uint4 out = pack8(f);
                        if (half) {
                            float back[8];
                            unpack8(out, back);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                f[e] -= back[e];
                            out = pack8(f);
                        }
                        *reinterpret_cast<uint4 *>(dst + tc::sw128(uint32_t(vr), uint32_t(q))) = out;
                    }
                    tc::fence_proxy_async_smem();
                    named_bar_sync(2, 128);
                    if (vr == 0)
                        mbar_arrive(full0 + 8 * s);
                }
                ++g;
                return ok;
            });
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
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

cudaError_t launch_proj_tc(const ProjParams &p, cudaStream_t stream)
{
    ProjArgs a;
    a.p = p;
    if (!encode_bf16_2d(&a.xmap, p.x, uint64_t(p.d_in), uint64_t(p.n), uint64_t(p.ldx) * 2u, kBK, kBM,
                        true) ||
        !encode_bf16_2d(&a.wmap, p.W, uint64_t(p.d_out), uint64_t(p.d_in), uint64_t(p.ldw) * 2u, 64,
                        kBK, true))
        return cudaErrorInvalidValue;
    if (p.b_rows) {
        if (!encode_row_maps(a.bmap, p.b_rows, uint64_t(p.d_out), p.b_nrows, p.b_ld))
            return cudaErrorInvalidValue;
    } else {
        for (auto &m : a.bmap)
            m = CUtensorMap{};
    }
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_proj_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(proj_smem_bytes()));
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    const int n_tiles = p.n_mblk * p.n_nblk;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(n_tiles < device_sms_proj() ? n_tiles : device_sms_proj()));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = proj_smem_bytes();
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_proj_tc, a);
}

int proj_block_rows() { return kBM; }
int proj_block_cols() { return kBN; }

}  // namespace lora
