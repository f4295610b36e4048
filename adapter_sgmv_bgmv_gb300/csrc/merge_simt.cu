// Merge / unmerge on CUDA cores: W[c, o] = bf16(W[c, o] + s * sum_j A[c, j] B[j, o])
// (VaLoRA blog, section 4.4.1: Delta W computed at run time from A and B and
// added to / subtracted from the base weight in one pass).  Each CTA owns a
// 64 x 256 tile of W; A's 64 x r block and B's r x 256 block are staged in shared
// memory, each thread accumulates an 8 x 8 block in fp32.  This is the CUDA-core
// variant; the tensor-core variant lives in tc_merge.cu.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace lora {

namespace {

constexpr int kRowsTile = 64;
constexpr int kColsTile = 256;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) k_merge_simt(const MergeParams p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int r = p.rank;
    float *sA = reinterpret_cast<float *>(smem);                               // [64][r]
    uint16_t *sB = reinterpret_cast<uint16_t *>(smem + size_t(kRowsTile) * r * 4);  // [r][256]
    const int c0 = blockIdx.y * kRowsTile;
    const int o0 = blockIdx.x * kColsTile;
    const int tid = threadIdx.x;
    const int rows = min(kRowsTile, p.d_in - c0);
    const int cols = min(kColsTile, p.d_out - o0);

    // A block: element (c, j) from page j at offset c0 + c (coalesced along c).
    for (int q = tid; q < kRowsTile * r; q += kThreads) {
        const int j = q / kRowsTile, c = q - j * kRowsTile;
        float a = 0.f;
        if (c < rows) {
            const uint16_t h = p.a_pool[int64_t(p.a_pages[j]) * p.a_pw + c0 + c];
            a = __uint_as_float(uint32_t(h) << 16);
        }
        sA[c * r + j] = a;
    }
    // B block: row j, 256 columns, 128-bit loads.
    for (int q = tid; q < r * (kColsTile / 8); q += kThreads) {
        const int j = q / (kColsTile / 8), v = q - j * (kColsTile / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (8 * v < cols)
            val = *reinterpret_cast<const uint4 *>(p.b_pool + int64_t(p.b_pages[j]) * p.b_pw +
                                                   o0 + 8 * v);
        reinterpret_cast<uint4 *>(sB + size_t(j) * kColsTile)[v] = val;
    }
    __syncthreads();

    const int vq = tid & 31;      // 8-column vector within the tile
    const int g = tid >> 5;       // group of 8 rows
    float acc[8][8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[u][e] = 0.f;
    for (int j = 0; j < r; ++j) {
        float bf[8];
        unpack8(reinterpret_cast<const uint4 *>(sB + size_t(j) * kColsTile)[vq], bf);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float a = sA[(g * 8 + u) * r + j];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                acc[u][e] = fmaf(a, bf[e], acc[u][e]);
        }
    }
    if (8 * vq >= cols)
        return;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int c = g * 8 + u;
        if (c >= rows)
            break;
        uint4 *w = reinterpret_cast<uint4 *>(p.W + int64_t(c0 + c) * p.ldw + o0 + 8 * vq);
        float wf[8];
        unpack8(*w, wf);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            wf[e] = fmaf(p.scale, acc[u][e], wf[e]);
        *w = pack8(wf);
    }
}

}  // namespace

cudaError_t launch_merge_simt(const MergeParams &p, cudaStream_t stream)
{
    const size_t smem = size_t(kRowsTile) * p.rank * 4 + size_t(p.rank) * kColsTile * 2;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k_merge_simt,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             200 * 1024);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.d_out + kColsTile - 1) / kColsTile, (p.d_in + kRowsTile - 1) / kRowsTile);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, k_merge_simt, p);
}

}  // namespace lora
