// Row-gather multi-LoRA kernel (decode / BGMV-like case) on CUDA cores.
//
// One work item = up to `rows_alloc` rows that share adapter k (a slice of one
// segment of the by-adapter permutation).  Each item is handled by a thread-block
// cluster of `cluster` CTAs.  CTA c of the cluster owns the c-th slice of d_in for
// the shrink and the c-th slice of d_out for the expand:
//
//   1. one warp issues bulk (TMA) copies of its slice of every page of A_k and of
//      every gathered x row (barrier 0), then of B_k and of the y rows (barrier 1),
//      so the whole working set of the CTA is in flight at once;
//   2. shrink: partial v[i, j] over the CTA's d_in slice, warp-per-page dot
//      products with 128-bit shared loads and a warp-shuffle reduction;
//   3. the partial sums are combined through distributed shared memory in a fixed
//      rank order (every CTA of the cluster gets identical v);
//   4. expand: y[i, o] = bf16(y[i, o] + s_k * sum_j v[i, j] B_k[j, o]) for the CTA's
//      d_out slice, 128-bit stores straight to the gathered rows.
//
// Released rows (id -1) are in no item, so they cost no CTA and are never touched
// (LoRazor page: the launch follows the active rows).  Modes: shrink-only writes v
// (fp32) and skips 4; expand-only reads v and skips 1-3 for x/A.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

__host__ __device__ inline size_t carve(int mode, int si, int so, int rows, int ranks,
                                        size_t off[7])
{
    size_t o = 0;
    const bool has_in = mode != kExpand, has_out = mode != kShrink;
    off[0] = o; o += has_in ? align16(size_t(ranks) * si * 2) : 0;    // A slice
    off[1] = o; o += has_in ? align16(size_t(rows) * si * 2) : 0;     // x rows
    off[2] = o; o += has_out ? align16(size_t(ranks) * so * 2) : 0;   // B slice
    off[3] = o; o += has_out ? align16(size_t(rows) * so * 2) : 0;   // y rows
    off[4] = o; o += align16(size_t(rows) * ranks * 4);               // partial v
    off[5] = o; o += align16(size_t(rows) * ranks * 4);               // v
    off[6] = o; o += 16;                                              // 2 mbarriers
    return o;
}

template <int MODE>
__device__ __forceinline__ void rows_body(const RowsParams &p, const RowItem *items,
                                          const int32_t *perm)
{
    extern __shared__ __align__(128) uint8_t smem[];
    size_t off[7];
    carve(MODE, p.slice_in, p.slice_out, p.rows_alloc, p.rank_alloc, off);
    uint16_t *sA = reinterpret_cast<uint16_t *>(smem + off[0]);
    uint16_t *sX = reinterpret_cast<uint16_t *>(smem + off[1]);
    uint16_t *sB = reinterpret_cast<uint16_t *>(smem + off[2]);
    uint16_t *sY = reinterpret_cast<uint16_t *>(smem + off[3]);
    float *vpart = reinterpret_cast<float *>(smem + off[4]);
    float *vsum = reinterpret_cast<float *>(smem + off[5]);
    const uint32_t bar0 = smem_u32(smem + off[6]);
    const uint32_t bar1 = bar0 + 8;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = p.cluster;
    const int item_id = blockIdx.x / C;
    const uint32_t crank = (C > 1) ? cluster_ctarank() : 0u;
    const RowItem it = items[item_id];
    const int k = it.adapter;
    const int r = p.rank[k];
    const int nrows = it.nrows;
    const float s = p.scale[k];
    const int RA = p.rank_alloc;

    const int in0 = int(crank) * p.slice_in;
    const int in_len = max(0, min(p.d_in - in0, p.slice_in));
    const int out0 = int(crank) * p.slice_out;
    const int out_len = max(0, min(p.d_out - out0, p.slice_out));

    if (tid == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar1, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // ---- 1. issue every copy this CTA needs
    if (warp == 0) {
        const int32_t *ap = p.a_pages + size_t(k) * p.max_rank;
        const int32_t *bp = p.b_pages + size_t(k) * p.max_rank;
        if (MODE != kExpand) {
            if (lane == 0)
                mbar_arrive_expect_tx(bar0, uint32_t(r + nrows) * uint32_t(in_len) * 2u);
            __syncwarp();
            if (in_len > 0) {
                for (int q = lane; q < r + nrows; q += 32) {
                    const uint16_t *src;
                    uint16_t *dst;
                    if (q < r) {
                        src = p.a_pool + int64_t(ap[q]) * p.a_pw + in0;
                        dst = sA + size_t(q) * p.slice_in;
                    } else {
                        const int row = perm[it.p0 + (q - r)];
                        src = p.x + int64_t(row) * p.ldx + in0;
                        dst = sX + size_t(q - r) * p.slice_in;
                    }
                    bulk_g2s(smem_u32(dst), src, uint32_t(in_len) * 2u, bar0);
                }
            }
        }
        if (MODE != kShrink) {
            if (lane == 0)
                mbar_arrive_expect_tx(bar1, uint32_t(r + nrows) * uint32_t(out_len) * 2u);
            __syncwarp();
            if (out_len > 0) {
                for (int q = lane; q < r + nrows; q += 32) {
                    const uint16_t *src;
                    uint16_t *dst;
                    if (q < r) {
                        src = p.b_pool + int64_t(bp[q]) * p.b_pw + out0;
                        dst = sB + size_t(q) * p.slice_out;
                    } else {
                        const int row = perm[it.p0 + (q - r)];
                        src = p.y + int64_t(row) * p.ldy + out0;
                        dst = sY + size_t(q - r) * p.slice_out;
                    }
                    bulk_g2s(smem_u32(dst), src, uint32_t(out_len) * 2u, bar1);
                }
            }
        }
    }

    bool ok = true;

    // ---- 2./3. shrink and cluster reduction
    if (MODE != kExpand) {
        ok = mbar_wait_bounded(bar0, 0, p.status, kDevTimeoutLoad) && ok;
        const int nvec = in_len >> 3;
        for (int j = warp; j < r; j += kWarps) {
            const uint4 *a = reinterpret_cast<const uint4 *>(sA + size_t(j) * p.slice_in);
            for (int i0 = 0; i0 < nrows; i0 += 4) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                for (int q = lane; q < nvec; q += 32) {
                    float af[8];
                    unpack8(a[q], af);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (i0 + u < nrows) {
                            float xf[8];
                            unpack8(reinterpret_cast<const uint4 *>(
                                        sX + size_t(i0 + u) * p.slice_in)[q], xf);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                acc[u] = fmaf(xf[e], af[e], acc[u]);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float t = warp_sum(acc[u]);
                    if (lane == 0 && i0 + u < nrows)
                        vpart[(i0 + u) * RA + j] = t;
                }
            }
        }
        if (C > 1) {
            cluster_sync();   // partial sums of every CTA are visible cluster-wide
            for (int q = tid; q < nrows * r; q += kThreads) {
                const int i = q / r, j = q - (q / r) * r;
                float acc = 0.f;
                for (int c = 0; c < C; ++c)
                    acc += ld_dsmem_f32(vpart + i * RA + j, uint32_t(c));
                vsum[i * RA + j] = acc;
            }
            cluster_arrive_release();   // peers may leave once everyone has read
        } else {
            __syncthreads();
            for (int q = tid; q < nrows * r; q += kThreads) {
                const int i = q / r, j = q - (q / r) * r;
                vsum[i * RA + j] = vpart[i * RA + j];
            }
        }
        __syncthreads();
        if (MODE == kShrink && ok && crank == 0) {
            for (int q = tid; q < nrows * r; q += kThreads) {
                const int i = q / r, j = q - (q / r) * r;
                const int row = perm[it.p0 + i];
                p.v[int64_t(row) * p.ldv + j] = vsum[i * RA + j];
            }
        }
    } else {
        for (int q = tid; q < nrows * r; q += kThreads) {
            const int i = q / r, j = q - (q / r) * r;
            const int row = perm[it.p0 + i];
            vsum[i * RA + j] = p.v[int64_t(row) * p.ldv + j];
        }
        __syncthreads();
    }

    // ---- 4. expand into the CTA's d_out slice
    if (MODE != kShrink) {
        ok = mbar_wait_bounded(bar1, 0, p.status, kDevTimeoutLoad) && ok;
        const int nvo = out_len >> 3;
        const int ngroups = (nrows + 3) >> 2;
        for (int w = tid; w < nvo * ngroups; w += kThreads) {
            const int q = w % nvo;
            const int i0 = (w / nvo) * 4;
            float acc[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[u][e] = 0.f;
            for (int j = 0; j < r; ++j) {
                float bf[8];
                unpack8(reinterpret_cast<const uint4 *>(sB + size_t(j) * p.slice_out)[q], bf);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float vv = (i0 + u < nrows) ? vsum[(i0 + u) * RA + j] : 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        acc[u][e] = fmaf(vv, bf[e], acc[u][e]);
                }
            }
            if (ok) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (i0 + u < nrows) {
                        float yf[8];
                        unpack8(reinterpret_cast<const uint4 *>(
                                    sY + size_t(i0 + u) * p.slice_out)[q], yf);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            yf[e] = fmaf(s, acc[u][e], yf[e]);
                        const int row = perm[it.p0 + i0 + u];
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
    if (MODE != kExpand && C > 1)
        cluster_wait_acquire();   // keep this CTA's shared memory alive for its peers
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) k_rows(const __grid_constant__ RowsParams p)
{
    rows_body<MODE>(p, p.items, p.perm);
}

// Same kernel with the plan (items and permutation) in the parameter block.
template <int MODE>
__global__ void __launch_bounds__(kThreads) k_rows_inline(const __grid_constant__ RowsParamsInline a)
{
    rows_body<MODE>(a.p, a.items, a.perm);
}

template <typename Kernel>
cudaError_t configure(Kernel k)
{
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         rows_max_smem());
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int MODE, bool INLINE, typename Arg>
cudaError_t launch_mode(const RowsParams &p, const Arg &arg, size_t smem, cudaStream_t stream)
{
    static bool configured = false;
    if (!configured) {
        cudaError_t e = INLINE ? configure(k_rows_inline<MODE>) : configure(k_rows<MODE>);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.n_items) * unsigned(p.cluster), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (INLINE)
        return cudaLaunchKernelEx(&cfg, k_rows_inline<MODE>, arg);
    else
        return cudaLaunchKernelEx(&cfg, k_rows<MODE>, arg);
}

}  // namespace

int rows_max_smem() { return 227 * 1024; }

size_t rows_smem_bytes(int mode, int slice_in, int slice_out, int rows_alloc, int rank_alloc)
{
    size_t off[7];
    return carve(mode, slice_in, slice_out, rows_alloc, rank_alloc, off);
}

cudaError_t launch_rows(int mode, const RowsParams &p, size_t smem, cudaStream_t stream)
{
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

}  // namespace lora
