// fattn_fwd_simt.cu -- plain SIMT attention forward (fp32 CUDA cores).
//
// A second GPU implementation of the same operation, deliberately simple: it
// shares no code with the tcgen05 kernel and serves the tests as an
// independent GPU cross-check at sizes where the CPU oracle only samples rows.
// It keeps the online-softmax recurrence of "Triton hand-written kernels:
// vector add -> tiled GEMM -> FlashAttention core", section 4 (running max,
// running sum, rescaled accumulator), tiled over 32 keys at a time, with
// fp32 scores and probabilities (no 16-bit rounding of P).
#include <cuda_bf16.h>
#include <math.h>

#include "fattn_internal.h"

namespace fattn {
namespace {

constexpr int kRowsPerWarp = 2;
constexpr int kWarps = 8;
constexpr int kRows = kRowsPerWarp * kWarps;  // query rows per CTA
constexpr int kKeys = 32;                     // keys per shared-memory tile

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    fwd_simt_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                    const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ o,
                    float *__restrict__ lse, int N, int row_blocks, float scale, int causal)
{
    constexpr int kCols = D / 32;  // output columns owned by one lane
    __shared__ float qs[kRows][D];
    __shared__ float ks[kKeys][D + 1];
    __shared__ float vs[kKeys][D];

    const int bh = blockIdx.x / row_blocks;
    const int row0 = (blockIdx.x % row_blocks) * kRows;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const size_t head = static_cast<size_t>(bh) * N * D;

    for (int idx = threadIdx.x; idx < kRows * D; idx += blockDim.x) {
        const int r = idx / D, c = idx % D;
        qs[r][c] = row0 + r < N ? __bfloat162float(q[head + static_cast<size_t>(row0 + r) * D + c])
                                : 0.f;
    }

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kCols];
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.f;
#pragma unroll
        for (int c = 0; c < kCols; ++c)
            acc[rr][c] = 0.f;
    }

    const int last_row = min(row0 + kRows, N) - 1;
    const int n_keys = causal ? last_row + 1 : N;
    for (int j0 = 0; j0 < n_keys; j0 += kKeys) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < kKeys * D; idx += blockDim.x) {
            const int r = idx / D, c = idx % D;
            const bool in = j0 + r < N;
            const size_t g = head + static_cast<size_t>(j0 + r) * D + c;
            ks[r][c] = in ? __bfloat162float(k[g]) : 0.f;
            vs[r][c] = in ? __bfloat162float(v[g]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int r = warp * kRowsPerWarp + rr;
            const int i = row0 + r;
            const int j = j0 + lane;
            float s = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c)
                s = fmaf(qs[r][c], ks[lane][c], s);
            s *= scale;
            const bool valid = j < N && (!causal || j <= i);
            s = valid ? s : -INFINITY;
            float tile_max = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                tile_max = fmaxf(tile_max, __shfl_xor_sync(0xffffffffu, tile_max, off));
            const float m_new = fmaxf(m[rr], tile_max);
            if (m_new == -INFINITY)  // no visible key in this tile (warp-uniform)
                continue;
            const float alpha = expf(m[rr] - m_new);
            const float p = valid ? expf(s - m_new) : 0.f;
            float psum = p;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l[rr] = l[rr] * alpha + psum;
#pragma unroll
            for (int c = 0; c < kCols; ++c)
                acc[rr][c] *= alpha;
#pragma unroll 4
            for (int jj = 0; jj < kKeys; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
                for (int c = 0; c < kCols; ++c)
                    acc[rr][c] = fmaf(pj, vs[jj][lane + 32 * c], acc[rr][c]);
            }
            m[rr] = m_new;
        }
    }

#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int i = row0 + warp * kRowsPerWarp + rr;
        if (i >= N)
            continue;
        const float inv = 1.f / l[rr];
#pragma unroll
        for (int c = 0; c < kCols; ++c)
            o[head + static_cast<size_t>(i) * D + lane + 32 * c] =
                __float2bfloat16_rn(acc[rr][c] * inv);
        if (lane == 0)
            lse[static_cast<size_t>(bh) * N + i] = m[rr] + logf(l[rr]);
    }
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs &a, cudaStream_t stream)
{
    const int row_blocks = (a.N + kRows - 1) / kRows;
    const long long blocks = static_cast<long long>(a.B) * a.H * row_blocks;
    if (blocks == 0)
        return cudaSuccess;
    if (blocks > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    const auto *q = static_cast<const __nv_bfloat16 *>(a.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(a.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(a.v);
    auto *o = static_cast<__nv_bfloat16 *>(a.o);
    if (a.d == 64)
        fwd_simt_kernel<64><<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(
            q, k, v, o, a.lse, a.N, row_blocks, a.scale, a.causal);
    else if (a.d == 96)
        fwd_simt_kernel<96><<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(
            q, k, v, o, a.lse, a.N, row_blocks, a.scale, a.causal);
    else
        fwd_simt_kernel<128><<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(
            q, k, v, o, a.lse, a.N, row_blocks, a.scale, a.causal);
    return cudaGetLastError();
}

}  // namespace fattn
