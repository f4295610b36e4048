// Row-gather multi-LoRA kernel (decode / BGMV-like case) on CUDA cores.
//
// One work item = up to `rows_alloc` rows that share adapter k (a slice of one
// segment of the by-adapter permutation).  Each item is handled by a thread-block
// cluster of `cluster` CTAs.  CTA c of the cluster owns the c-th slice of d_in for
// the shrink and the c-th slice of d_out for the expand:
//
//   1. warp 0 issues bulk (TMA) copies: lane i < nrows fetches x row i and y row i,
//      lane j < r reads page j of A_k / B_k from the page table and fetches its
//      slice, so the CTA's whole working set is in flight after one dependent load;
//   2. shrink: partial v[i, j] over the CTA's d_in slice, half a warp per page (all
//      pages of a rank <= 16 at once), 128-bit shared loads and a shuffle reduction,
//      into the CTA's own shared memory;
//   3. every CTA pushes its partial into its C - 1 peers' shared memory with
//      asynchronous remote stores (st.async) that complete bytes on the receiver's
//      own mbarrier, waits on that mbarrier for the C - 1 partials addressed to it,
//      and sums all C in cluster-rank order (all CTAs get an identical v).  The one
//      cluster barrier (arrived at right after the mbarriers are set up, waited on
//      before the first push) only makes every peer's mbarrier valid before anything
//      is stored into it; no CTA leaves before all partials addressed to it have
//      landed, so no barrier is needed at exit;
//   4. expand: y[i, o] = bf16(y[i, o] + s_k * sum_j v[i, j] B_k[j, o]) for the CTA's
//      d_out slice, 128-bit stores straight to the gathered rows.
//
// Released rows (id -1) are in no item, so they cost no CTA and are never touched
// (LoRazor page: the launch follows the active rows).  Modes: shrink-only writes v
// (fp32) and skips 4; expand-only reads v, skips 1-3 for x/A and needs no cluster.
#include <algorithm>

#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxCluster = 16;

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// no_y: a fused launch whose threads read y straight from global memory after the
// dependency wait (see y_late below) has no y rows in shared memory.  b_over_a: a
// fused launch copies B's slice into A's space after the shrink (one region, the
// larger of the two).
__host__ __device__ inline size_t carve(int mode, int si, int so, int rows, int ranks,
                                        int cluster, bool no_y, bool b_over_a, size_t off[8])
{
    size_t o = 0;
    const bool has_in = mode != kExpand, has_out = mode != kShrink;
    const bool over = b_over_a && has_in && has_out;
    const size_t a_sz = has_in ? align16(size_t(ranks) * si * 2) : 0;
    const size_t b_sz = has_out ? align16(size_t(ranks) * so * 2) : 0;
    off[0] = o; o += over ? (a_sz > b_sz ? a_sz : b_sz) : a_sz;             // A slice
    off[1] = o; o += has_in ? align16(size_t(rows) * si * 2) : 0;           // x rows
    off[2] = over ? off[0] : o; o += over ? 0 : b_sz;                       // B slice
    off[3] = o; o += (has_out && !no_y) ? align16(size_t(rows) * so * 2) : 0;   // y rows
    // own partial, then the C partials of the cluster (rank c at c * rows * ranks)
    off[4] = o; o += (has_in && cluster > 1) ? align16(size_t(rows) * ranks * 4) * (1 + cluster) : 0;
    off[5] = o; o += align16(size_t(rows) * ranks * 4);                     // v
    off[6] = o; o += align16(size_t(rows) * 4);                             // the rows' indices
    off[7] = o; o += 32;                                                    // 3 mbarriers
    return o;
}

// Expand of `ROWS` rows starting at i0 for 8 output columns at vector q:
// acc[u][e] = sum_j v[i0+u, j] * B[j, 8q+e].
template <int ROWS>
__device__ __forceinline__ void expand_vec(const uint16_t *sB, int slice_out, const float *vsum,
                                           int RA, int r, int i0, int q, float acc[ROWS][8])
{
#pragma unroll
    for (int u = 0; u < ROWS; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[u][e] = 0.f;
#pragma unroll 4
    for (int j = 0; j < r; ++j) {
        float bf[8];
        unpack8(reinterpret_cast<const uint4 *>(sB + size_t(j) * slice_out)[q], bf);
#pragma unroll
        for (int u = 0; u < ROWS; ++u) {
            const float vv = vsum[(i0 + u) * RA + j];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[u][e] = fmaf(vv, bf[e], acc[u][e]);
        }
    }
}

// DIRECT: the device-resident-ids mode (a kernel of its own, so that its id scan
// costs the host-planned kernels no registers).
template <int MODE, bool DIRECT>
__device__ __forceinline__ void rows_body(const RowsParams &pin, const RowItem *items,
                                          const int32_t *perm)
{
    // A register copy of the parameters: read through the parameter block's
    // address, every field would be loaded again after each asm statement that
    // clobbers memory (barriers, cluster stores).
    const RowsParams p = pin;
    extern __shared__ __align__(128) uint8_t smem[];
    const int C = p.cluster;
    size_t off[8];
    const bool b_late = MODE == kFused && p.b_over_a != 0;
    carve(MODE, p.slice_in, p.slice_out, p.rows_alloc, p.rank_alloc, C, p.no_y_smem != 0, b_late,
          off);
    uint16_t *sA = reinterpret_cast<uint16_t *>(smem + off[0]);
    uint16_t *sX = reinterpret_cast<uint16_t *>(smem + off[1]);
    uint16_t *sB = reinterpret_cast<uint16_t *>(smem + off[2]);
    uint16_t *sY = reinterpret_cast<uint16_t *>(smem + off[3]);
    float *vin = reinterpret_cast<float *>(smem + off[4]);
    float *vsum = reinterpret_cast<float *>(smem + off[5]);
    int32_t *s_rows = reinterpret_cast<int32_t *>(smem + off[6]);   // perm[it.p0 + i]
    const uint32_t bar0 = smem_u32(smem + off[7]);
    const uint32_t bar1 = bar0 + 8;
    const uint32_t xbar = bar0 + 16;              // the cluster's partials have landed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool clustered = (MODE != kExpand) && C > 1;
    const int item_id = blockIdx.x / C;
    const uint32_t crank = clustered ? cluster_ctarank() : uint32_t(blockIdx.x % C);
    constexpr bool direct = DIRECT;
    RowItem it;
    if (direct) {
        // Device-resident ids, one row per cluster: item i is row i, of the adapter
        // the ids give -- read after the wait for the previous kernel, unless early
        // page copies are on (the caller's guarantee then covers the ids too: the
        // kernel just before does not write them).  A released row has nothing to
        // do; a row whose id the table cannot serve is left as it is and flagged.  A
        // cluster shares its row, so all its CTAs leave together, before any barrier.
        if (!p.early_pages)
            grid_dep_wait();
        const int row = item_id;
        const int ka = p.ids_dev[row];
        if (ka == -1)
            return;
        if (ka < -1 || ka >= p.n_adapters || !p.ok[ka]) {
            if (crank == 0 && threadIdx.x == 0)
                raise_status(p.status, kDevBadId);
            return;
        }
        it.adapter = ka;
        it.p0 = row;
        it.nrows = 1;
        it.rank = int16_t(p.rank[ka]);
        it.scale = p.scale[ka];
    } else {
        if (p.n_items_dev) {
            // A device-side plan is the previous kernel's output: wait for it before
            // reading it.  Clusters past its item count have nothing to do (a cluster
            // shares its item, so all its CTAs leave together, before any barrier).
            grid_dep_wait();
            if (item_id >= *p.n_items_dev)
                return;
        }
        it = items[item_id];
    }
    const int k = it.adapter;
    const int r = it.rank;
    const int nrows = it.nrows;
    const float s = it.scale;
    const int RA = p.rank_alloc;

    const int in0 = int(crank) * p.slice_in;
    const int in_len = max(0, min(p.d_in - in0, p.slice_in));
    const int out0 = int(crank) * p.slice_out;
    const int out_len = max(0, min(p.d_out - out0, p.slice_out));

    // The partials exchanged per CTA: nrows x RA floats, sent in 16-byte pieces.
    const int xchunks = (nrows * RA + 3) >> 2;
    // Ahead of the wait for the previous kernel: the adapter pages (early_pages, or
    // early_x, whose guarantee covers the pools too), and with early_x also x, the
    // shrink and the cluster exchange.  A fused call whose every thread has at most one
    // output vector (y_late) then computes its expand term before the wait as well
    // and afterwards only reads its y vectors, adds and stores.  Either way the next
    // kernel may start as soon as this one's copies are out: whatever it reads of y or
    // v waits for this kernel, and this kernel for the one before it.
    const bool pages_early = p.early_pages || p.early_x;
    const bool x_early = p.early_x && MODE != kExpand;
    const int nvo_all = out_len >> 3;
    const int ngroups = nrows == 1 ? 1 : (nrows + 1) >> 1;
    // (no_y_smem: the host found that every CTA of the launch qualifies)
    const bool y_late = x_early && MODE == kFused && (p.no_y_smem || nvo_all * ngroups <= kThreads);
    if (tid == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar1, 1);
        mbar_init(xbar, 1);
        if (clustered)   // the C - 1 peers' partials (its own is copied locally)
            mbar_arrive_expect_tx(xbar, uint32_t(C - 1) * uint32_t(xchunks) * 16u);
        fence_mbar_init();
    }
    __syncthreads();
    if (clustered)
        cluster_arrive_relaxed();   // this CTA's mbarriers are valid (waited on before the pushes)

    // ---- 1. copies.  Page ids come from the table (written once, at registration),
    // so they are read before waiting for the preceding kernel; everything it may
    // have written (x, y, v, the pools) is touched only after the wait.
    const uint32_t in_bytes = uint32_t(in_len) * 2u, out_bytes = uint32_t(out_len) * 2u;
    int32_t pa0 = 0, pa1 = 0, pb0 = 0, pb1 = 0, pr0 = 0, pr1 = 0;
    const int32_t *ap = p.a_pages + size_t(k) * p.max_rank;
    const int32_t *bp = p.b_pages + size_t(k) * p.max_rank;
    if (warp == 0) {
        if (lane < r) {
            if (MODE != kExpand)
                pa0 = ap[lane];
            if (MODE != kShrink)
                pb0 = bp[lane];
        }
        if (lane + 32 < r) {
            if (MODE != kExpand)
                pa1 = ap[lane + 32];
            if (MODE != kShrink)
                pb1 = bp[lane + 32];
        }
        if (lane < nrows)
            pr0 = direct ? it.p0 : perm[it.p0 + lane];
        if (lane + 32 < nrows)
            pr1 = perm[it.p0 + lane + 32];
        for (int q = lane; q < nrows; q += 32)
            s_rows[q] = q < 32 ? pr0 : q < 64 ? pr1 : perm[it.p0 + q];
    }
    // Adapter pages first (by lane j < r), then the rows (lane i < nrows); with
    // early_pages the page copies go out before waiting for the preceding kernel
    // (the pools are not that kernel's to write), overlapping its tail.  With b_late
    // B's pages land in A's space, so they go out once the shrink is done with it.
    auto issue_b = [&]() {
        for (int q = lane; q < r; q += 32) {
            const int32_t qb = q < 32 ? pb0 : q < 64 ? pb1 : (MODE != kShrink ? bp[q] : 0);
            if (MODE != kShrink && out_bytes)
                bulk_g2s(smem_u32(sB + size_t(q) * p.slice_out),
                         p.b_pool + int64_t(qb) * p.b_pw + out0, out_bytes, bar1);
        }
    };
    auto issue_pages = [&]() {
        for (int q = lane; q < r; q += 32) {
            const int32_t qa = q < 32 ? pa0 : q < 64 ? pa1 : (MODE != kExpand ? ap[q] : 0);
            if (MODE != kExpand && in_bytes)
                bulk_g2s(smem_u32(sA + size_t(q) * p.slice_in),
                         p.a_pool + int64_t(qa) * p.a_pw + in0, in_bytes, bar0);
        }
        if (!b_late)
            issue_b();
    };
    // Called by every thread once all reads of A are done (after a block barrier).
    auto issue_b_late = [&]() {
        if (b_late && warp == 0) {
            // the shrink's reads of A (generic proxy) before the copies' writes (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_b();
        }
    };
    auto issue_x = [&]() {
        for (int q = lane; q < nrows; q += 32)
            if (MODE != kExpand && in_bytes)
                bulk_g2s(smem_u32(sX + size_t(q) * p.slice_in),
                         p.x + int64_t(s_rows[q]) * p.ldx + in0, in_bytes, bar0);
    };
    auto issue_y = [&]() {
        for (int q = lane; q < nrows; q += 32)
            if (MODE != kShrink && out_bytes)
                bulk_g2s(smem_u32(sY + size_t(q) * p.slice_out),
                         p.y + int64_t(s_rows[q]) * p.ldy + out0, out_bytes, bar1);
    };
    if (warp == 0) {
        if (lane == 0) {
            if (MODE != kExpand)
                mbar_arrive_expect_tx(bar0, uint32_t(r + nrows) * in_bytes);
            if (MODE != kShrink)
                mbar_arrive_expect_tx(bar1, uint32_t(y_late ? r : r + nrows) * out_bytes);
        }
        __syncwarp();
        if (pages_early)
            issue_pages();
        if (x_early)
            issue_x();
    }
    if (x_early) {
        grid_dep_launch();
    } else {
        grid_dep_wait();
        if (warp == 0) {
            if (!pages_early)
                issue_pages();
            issue_x();
            issue_y();
        }
        grid_dep_launch();
    }

    bool ok = true;

    // ---- 2./3. shrink and cluster exchange
    if (MODE != kExpand) {
        ok = mbar_wait_bounded(bar0, 0, p.status, kDevTimeoutLoad) && ok;
        const int nvec = in_len >> 3;
        // Half a warp per page, all pages of a rank <= 16 at once: thread l16 of
        // the half takes every 16th 8-element vector of the CTA's slice.
        const int l16 = lane & 15;
        const unsigned hmask = 0xffffu << (lane & 16);
        for (int j = tid >> 4; j < r; j += kThreads / 16) {
            const uint4 *a = reinterpret_cast<const uint4 *>(sA + size_t(j) * p.slice_in);
            for (int i0 = 0; i0 < nrows; i0 += 4) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
                const int nr = min(4, nrows - i0);
                for (int q = l16; q < nvec; q += 16) {
                    const uint4 av = a[q];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (u < nr)
                            dot8_bf16(reinterpret_cast<const uint4 *>(sX + size_t(i0 + u) * p.slice_in)[q],
                                      av, acc[u], acc2[u]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (u < nr) {
                        float t = acc[u] + acc2[u];
#pragma unroll
                        for (int o = 8; o > 0; o >>= 1)
                            t += __shfl_xor_sync(hmask, t, o);
                        const int slot = (i0 + u) * RA + j;
                        if (l16 == 0)
                            (clustered ? vin : vsum)[slot] = t;
                    }
                }
            }
        }
        if (clustered) {
            // Push this CTA's partial into every peer of the cluster, at slot crank of
            // their partials, once every peer's mbarrier is valid (and copy it into its
            // own slot); then wait for the C - 1 partials addressed to this CTA and sum
            // all C in cluster-rank order, so that every CTA holds the same v.
            float *vall = vin + align16(size_t(p.rows_alloc) * RA * 4) / 4;
            __syncthreads();                       // vin complete, A read
            issue_b_late();
            cluster_wait_acquire();
            const uint32_t dst0 = smem_u32(vall) + uint32_t(crank) * uint32_t(xchunks) * 16u;
            for (int q = tid; q < C * xchunks; q += kThreads) {
                const int c = q / xchunks, piece = q - c * xchunks;
                const float4 val = reinterpret_cast<const float4 *>(vin)[piece];
                if (c == int(crank))
                    reinterpret_cast<float4 *>(vall)[size_t(c) * xchunks + piece] = val;
                else
                    st_async_v4(map_cluster(dst0 + uint32_t(piece) * 16u, uint32_t(c)), val,
                                map_cluster(xbar, uint32_t(c)));
            }
            ok = mbar_wait_bounded(xbar, 0, p.status, kDevTimeoutLoad) && ok;
            __syncthreads();                       // the local copy too
            for (int q = tid; q < nrows * r; q += kThreads) {
                const int i = q / r, j = q - (q / r) * r;
                float acc = 0.f;
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c)
                    if (c < C)
                        acc += vall[size_t(c) * (xchunks * 4) + i * RA + j];
                vsum[i * RA + j] = acc;
            }
        }
        __syncthreads();
        if (!clustered)
            issue_b_late();
        if (x_early && !y_late) {
            // Everything past here reads y or writes global memory.
            grid_dep_wait();
            if (warp == 0)
                issue_y();
        }
        if (MODE == kShrink && ok && crank == 0) {
            for (int q = tid; q < nrows * r; q += kThreads) {
                const int i = q / r, j = q - (q / r) * r;
                p.v[int64_t(s_rows[i]) * p.ldv + j] = vsum[i * RA + j];
            }
        }
    } else {
        __syncthreads();   // s_rows
        for (int q = tid; q < nrows * r; q += kThreads) {
            const int i = q / r, j = q - (q / r) * r;
            vsum[i * RA + j] = p.v[int64_t(s_rows[i]) * p.ldv + j];
        }
        __syncthreads();
    }

    // ---- 4. expand into the CTA's d_out slice
    if (MODE != kShrink && y_late) {
        // Thread w holds output vector q = w % nvo of rows 2 (w / nvo) and + 1 (one
        // row when nrows == 1): the term is computed from B in shared memory before
        // the wait, y is read straight from global memory after it.
        ok = mbar_wait_bounded(bar1, 0, p.status, kDevTimeoutLoad) && ok;
        const int nvo = nvo_all;
        const int w = tid, q = nvo > 0 ? w % nvo : 0;
        const int i0 = nvo > 0 ? (w / nvo) * 2 : 0;
        const bool act = w < nvo * ngroups;
        const int nr = nrows == 1 ? 1 : min(2, nrows - i0);
        float acc[2][8];
        if (act) {
            if (nr == 2) {
                expand_vec<2>(sB, p.slice_out, vsum, RA, r, i0, q, acc);
            } else {
                float a1[1][8];
                expand_vec<1>(sB, p.slice_out, vsum, RA, r, i0, q, a1);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[0][e] = a1[0][e];
            }
        }
        uint16_t *yp[2];
        if (act) {
            // Bring the y vectors into L2 ahead of the wait (a hint: L2 stays coherent
            // with the previous kernel's writes), so that the read after it hits L2.
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (u < nr) {
                    yp[u] = p.y + int64_t(s_rows[i0 + u]) * p.ldy + out0 + 8 * q;
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(yp[u]));
                }
        }
        grid_dep_wait();
        if (act) {
            uint4 yv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (u < nr)
                    yv[u] = *reinterpret_cast<const uint4 *>(yp[u]);
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (u < nr) {
                    float yf[8];
                    unpack8(yv[u], yf);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        yf[e] = fmaf(s, acc[u][e], yf[e]);
                    if (ok)
                        *reinterpret_cast<uint4 *>(yp[u]) = pack8(yf);
                }
        }
    } else if (MODE != kShrink) {
        ok = mbar_wait_bounded(bar1, 0, p.status, kDevTimeoutLoad) && ok;
        const int nvo = out_len >> 3;
        if (nrows == 1) {
            const int row = s_rows[0];
            for (int q = tid; q < nvo; q += kThreads) {
                float acc[1][8];
                expand_vec<1>(sB, p.slice_out, vsum, RA, r, 0, q, acc);
                float yf[8];
                unpack8(reinterpret_cast<const uint4 *>(sY)[q], yf);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    yf[e] = fmaf(s, acc[0][e], yf[e]);
                if (ok)
                    *reinterpret_cast<uint4 *>(p.y + int64_t(row) * p.ldy + out0 + 8 * q) = pack8(yf);
            }
        } else {
            const int ngroups = (nrows + 1) >> 1;
            for (int w = tid; w < nvo * ngroups; w += kThreads) {
                const int q = w % nvo;
                const int i0 = (w / nvo) * 2;
                float acc[2][8];
                if (i0 + 1 < nrows) {
                    expand_vec<2>(sB, p.slice_out, vsum, RA, r, i0, q, acc);
                } else {
                    float a1[1][8];
                    expand_vec<1>(sB, p.slice_out, vsum, RA, r, i0, q, a1);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        acc[0][e] = a1[0][e];
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (i0 + u < nrows) {
                        float yf[8];
                        unpack8(reinterpret_cast<const uint4 *>(
                                    sY + size_t(i0 + u) * p.slice_out)[q], yf);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            yf[e] = fmaf(s, acc[u][e], yf[e]);
                        const int row = s_rows[i0 + u];
                        if (ok)
                            *reinterpret_cast<uint4 *>(p.y + int64_t(row) * p.ldy + out0 + 8 * q) =
                                pack8(yf);
                    }
                }
            }
        }
    }

    if (!ok) {
        // A copy did not land in time: give the copies in flight one more bounded
        // wait so none of them writes into shared memory after this CTA has left.
        if (MODE != kExpand)
            mbar_wait_bounded(bar0, 0, nullptr, 0);
        if (MODE != kShrink)
            mbar_wait_bounded(bar1, 0, nullptr, 0);
    }
}

// OCC: CTAs per SM the registers must allow.  A launch whose shared memory fits six
// CTAs per SM takes the OCC = 6 instance (40 registers, so that six are resident:
// more of consecutive calls' CTAs overlap); a larger one, which fits fewer CTAs
// anyway, takes the unconstrained instance.
template <int MODE, bool DIRECT, int OCC>
__global__ void __launch_bounds__(kThreads, OCC) k_rows(const __grid_constant__ RowsParams p)
{
    rows_body<MODE, DIRECT>(p, p.items, p.perm);
}

// Same kernel with the plan (items and permutation) in the parameter block.
template <int MODE, typename Inline, int OCC>
__global__ void __launch_bounds__(kThreads, OCC) k_rows_inline(const __grid_constant__ Inline a)
{
    rows_body<MODE, false>(a.p, a.items, a.perm);
}

// Shared memory per SM on sm_100-family GPUs, and what the runtime reserves per CTA.
constexpr size_t kSmemPerSm = 228 * 1024, kSmemReservedPerCta = 1024;

template <typename Kernel>
cudaError_t configure(Kernel k)
{
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         rows_max_smem());
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int MODE, bool INLINE, typename Arg, bool DIRECT, int OCC>
cudaError_t launch_occ(const RowsParams &p, const Arg &arg, size_t smem, cudaStream_t stream)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e;
        if constexpr (INLINE)
            e = configure(k_rows_inline<MODE, Arg, OCC>);
        else
            e = configure(k_rows<MODE, DIRECT, OCC>);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.n_items) * unsigned(p.cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (MODE == kExpand) ? 1u : unsigned(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // May start while the previous kernel of the stream drains (see grid_dep_wait).
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if constexpr (INLINE)
        return cudaLaunchKernelEx(&cfg, k_rows_inline<MODE, Arg, OCC>, arg);
    else
        return cudaLaunchKernelEx(&cfg, k_rows<MODE, DIRECT, OCC>, arg);
}

// The instance a launch takes: the register budget that lets as many CTAs be
// resident as its shared memory allows, from six down to five (fused only); the
// unconstrained instance below that.
int occ_instance(int mode, size_t smem)
{
    const size_t fit = kSmemPerSm / (smem + kSmemReservedPerCta);
    if (fit >= 6)
        return 6;
    if (fit == 5 && mode == kFused)
        return 5;
    return 1;
}

template <int MODE, bool INLINE, typename Arg, bool DIRECT = false>
cudaError_t launch_mode(const RowsParams &p, const Arg &arg, size_t smem, cudaStream_t stream)
{
    const int occ = occ_instance(MODE, smem);
    if (occ == 6)
        return launch_occ<MODE, INLINE, Arg, DIRECT, 6>(p, arg, smem, stream);
    if constexpr (MODE == kFused)
        if (occ == 5)
            return launch_occ<MODE, INLINE, Arg, DIRECT, 5>(p, arg, smem, stream);
    return launch_occ<MODE, INLINE, Arg, DIRECT, 1>(p, arg, smem, stream);
}

}  // namespace

int rows_max_smem() { return 227 * 1024; }
int rows_max_cluster() { return kMaxCluster; }

size_t rows_smem_bytes(int mode, int slice_in, int slice_out, int rows_alloc, int rank_alloc,
                       int cluster, bool no_y, bool b_over_a)
{
    size_t off[8];
    return carve(mode, slice_in, slice_out, rows_alloc, rank_alloc, cluster, no_y, b_over_a, off);
}

int rows_ctas_per_sm(int mode, size_t smem)
{
    // The unconstrained instances take 72 to 82 registers a thread: three CTAs.
    const int fit = int(kSmemPerSm / (smem + kSmemReservedPerCta));
    const int occ = occ_instance(mode, smem);
    return std::min(fit, occ == 1 ? 3 : occ);
}

bool rows_y_late(int mode, bool early_x, int slice_out, int rows_alloc)
{
    const int ngroups = rows_alloc <= 1 ? 1 : (rows_alloc + 1) / 2;
    return early_x && mode == kFused && (slice_out / 8) * ngroups <= kThreads;
}

cudaError_t launch_rows(int mode, const RowsParams &p, size_t smem, cudaStream_t stream)
{
    if (p.ids_dev)   // device-resident ids: fused only
        return launch_mode<kFused, false, RowsParams, true>(p, p, smem, stream);
    switch (mode) {
    case kShrink: return launch_mode<kShrink, false>(p, p, smem, stream);
    case kExpand: return launch_mode<kExpand, false>(p, p, smem, stream);
    default: return launch_mode<kFused, false>(p, p, smem, stream);
    }
}

cudaError_t launch_rows_inline(int mode, const RowsParamsInline &a, size_t smem,
                               cudaStream_t stream)
{
    switch (mode) {
    case kShrink: return launch_mode<kShrink, true>(a.p, a, smem, stream);
    case kExpand: return launch_mode<kExpand, true>(a.p, a, smem, stream);
    default: return launch_mode<kFused, true>(a.p, a, smem, stream);
    }
}

cudaError_t launch_rows_inline_small(int mode, const RowsParamsInlineSmall &a, size_t smem,
                                     cudaStream_t stream)
{
    switch (mode) {
    case kShrink: return launch_mode<kShrink, true>(a.p, a, smem, stream);
    case kExpand: return launch_mode<kExpand, true>(a.p, a, smem, stream);
    default: return launch_mode<kFused, true>(a.p, a, smem, stream);
    }
}

}  // namespace lora
