// fattn_rowops.cu -- standalone row softmax and row sum (HBM-bound).
//
// The row softmax and row-sum kernels of "CS336 lecture 6: kernels and
// Triton": one program per row, masked loads that pad with -inf for the max
// and 0 for the sum, and for rows longer than one block a loop over column
// tiles.  Its cost note (a fused softmax reads and writes the matrix once,
// against ~5 reads and 3 writes for the unfused chain) is the design target:
//   - rows of up to 16384 elements are read once into registers (16-byte
//     loads), reduced, and written once;
//   - longer rows take two passes: an online pass keeping a running max and
//     a rescaled running sum per thread (the same recurrence as the attention
//     kernel), merged across the block, then a pass that writes the output.
// One CTA of 256 threads per row, rows dealt grid-stride over a grid sized to
// the SM count.  Element types: fp32 or bf16 in and out; fp32 arithmetic.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "fattn_internal.h"

namespace fattn {
namespace {

constexpr int kThreads = 256;
// 16-byte chunks per thread kept in registers: 64 fp32 values either way
// (16 chunks of 4 fp32, 8 chunks of 8 bf16), i.e. rows of up to 16384.
template <typename T> struct MaxChunks {
    static constexpr int value = 64 / (16 / static_cast<int>(sizeof(T)));
};
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Elements per 16-byte chunk and their conversion to / from fp32.
template <typename T> struct Chunk;
template <> struct Chunk<float> {
    static constexpr int kElems = 4;
    __device__ static void load(const float *p, float (&v)[4])
    {
        const float4 f = *reinterpret_cast<const float4 *>(p);
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
    __device__ static void store(float *p, const float (&v)[4])
    {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __device__ static float get(const float *p) { return *p; }
    __device__ static void put(float *p, float v) { *p = v; }
};
template <> struct Chunk<__nv_bfloat16> {
    static constexpr int kElems = 8;
    __device__ static void load(const __nv_bfloat16 *p, float (&v)[8])
    {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void store(__nv_bfloat16 *p, const float (&v)[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ static float get(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    __device__ static void put(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
};

// Block-wide max and sum of one value per thread (all threads get the result).
__device__ __forceinline__ float block_max(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();  // red may still be read by a previous reduction
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x / 32] = v;
    __syncthreads();
    v = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w)
        v = fmaxf(v, red[w]);
    return v;
}
__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x / 32] = v;
    __syncthreads();
    v = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w)
        v += red[w];
    return v;
}

// Chunk c of this thread covers elements [(c*256 + t)*E, +E) of the row; a
// chunk that crosses N is handled element by element (never read past N).
// x and y may be the same buffer (in place): every element is read and then
// written by the same thread, and no thread reads another thread's elements.
// kMaxChunks = 0 selects the two-pass path; otherwise chunks <= kMaxChunks and
// the row stays in registers (instantiated for 1, 2, 4, ... so that short
// rows use few registers and many rows are in flight per SM).
template <typename T, int kMaxChunks>
__global__ void __launch_bounds__(kThreads)
    softmax_rows_kernel(const T *x, T *y, int M, int N, int chunks, int vec_ok)
{
    using Ck = Chunk<T>;
    constexpr int E = Ck::kElems;
    __shared__ float red[kThreads / 32];
    const int t = threadIdx.x;
    for (int row = blockIdx.x; row < M; row += gridDim.x) {
        const T *xr = x + static_cast<size_t>(row) * N;
        T *yr = y + static_cast<size_t>(row) * N;
        if constexpr (kMaxChunks > 0) {
            // One read: the row lives in registers.
            float v[kMaxChunks][E];
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c) {
                if (c >= chunks)
                    break;
                const int e0 = (c * kThreads + t) * E;
                if (vec_ok && e0 + E <= N) {
                    Ck::load(xr + e0, v[c]);
                } else {
#pragma unroll
                    for (int i = 0; i < E; ++i)
                        v[c][i] = e0 + i < N ? Ck::get(xr + e0 + i) : -INFINITY;
                }
#pragma unroll
                for (int i = 0; i < E; ++i)
                    mx = fmaxf(mx, v[c][i]);
            }
            mx = block_max(mx, red);
            const float mb = mx * kLog2e;
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c) {
                if (c >= chunks)
                    break;
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    v[c][i] = ex2f(fmaf(v[c][i], kLog2e, -mb));  // -inf pads give 0
                    sum += v[c][i];
                }
            }
            sum = block_sum(sum, red);
            const float inv = 1.f / sum;
#pragma unroll
            for (int c = 0; c < kMaxChunks; ++c) {
                if (c >= chunks)
                    break;
                const int e0 = (c * kThreads + t) * E;
#pragma unroll
                for (int i = 0; i < E; ++i)
                    v[c][i] *= inv;
                if (vec_ok && e0 + E <= N) {
                    Ck::store(yr + e0, v[c]);
                } else {
#pragma unroll
                    for (int i = 0; i < E; ++i)
                        if (e0 + i < N)
                            Ck::put(yr + e0 + i, v[c][i]);
                }
            }
        } else {
            // Two passes: running (max, rescaled sum) per thread, then write.
            float m = -INFINITY, l = 0.f;
            for (int c = 0; c < chunks; ++c) {
                const int e0 = (c * kThreads + t) * E;
                float v[E];
                if (vec_ok && e0 + E <= N) {
                    Ck::load(xr + e0, v);
                } else {
#pragma unroll
                    for (int i = 0; i < E; ++i)
                        v[i] = e0 + i < N ? Ck::get(xr + e0 + i) : -INFINITY;
                }
                float cm = v[0];
#pragma unroll
                for (int i = 1; i < E; ++i)
                    cm = fmaxf(cm, v[i]);
                const float mn = fmaxf(m, cm);
                if (mn == -INFINITY)
                    continue;
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < E; ++i)
                    s += ex2f((v[i] - mn) * kLog2e);
                l = l * ex2f((m - mn) * kLog2e) + s;
                m = mn;
            }
            const float mrow = block_max(m, red);
            const float lrow = block_sum(m == -INFINITY ? 0.f : l * ex2f((m - mrow) * kLog2e), red);
            const float inv = 1.f / lrow;
            const float mb = mrow * kLog2e;
            for (int c = 0; c < chunks; ++c) {
                const int e0 = (c * kThreads + t) * E;
                float v[E];
                if (vec_ok && e0 + E <= N) {
                    Ck::load(xr + e0, v);
#pragma unroll
                    for (int i = 0; i < E; ++i)
                        v[i] = ex2f(fmaf(v[i], kLog2e, -mb)) * inv;
                    Ck::store(yr + e0, v);
                } else {
#pragma unroll
                    for (int i = 0; i < E; ++i)
                        if (e0 + i < N)
                            Ck::put(yr + e0 + i, ex2f(fmaf(Ck::get(xr + e0 + i), kLog2e, -mb)) * inv);
                }
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    row_sum_kernel(const T *__restrict__ x, float *__restrict__ out, int M, int N, int chunks,
                   int vec_ok)
{
    using Ck = Chunk<T>;
    constexpr int E = Ck::kElems;
    __shared__ float red[kThreads / 32];
    const int t = threadIdx.x;
    for (int row = blockIdx.x; row < M; row += gridDim.x) {
        const T *xr = x + static_cast<size_t>(row) * N;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c = 0; c < chunks; ++c) {
            const int e0 = (c * kThreads + t) * E;
            float v[E];
            if (vec_ok && e0 + E <= N) {
                Ck::load(xr + e0, v);
            } else {
#pragma unroll
                for (int i = 0; i < E; ++i)
                    v[i] = e0 + i < N ? Ck::get(xr + e0 + i) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < E; ++i)
                acc[i & 3] += v[i];
        }
        const float s = block_sum((acc[0] + acc[1]) + (acc[2] + acc[3]), red);
        if (t == 0)
            out[row] = s;
    }
}

// Grid of (resident CTAs per SM) x SMs, rows dealt grid-stride.
template <typename K>
cudaError_t launch_grid(K kernel, int M, int num_sms, int *grid)
{
    int per_sm = 1;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
    if (e != cudaSuccess)
        return e;
    const long long slots = static_cast<long long>(num_sms) * (per_sm > 0 ? per_sm : 1);
    *grid = static_cast<int>(M < slots ? M : slots);
    return cudaSuccess;
}

template <typename T, int C>
cudaError_t launch_softmax(const void *x, void *y, int M, int N, int chunks, int vec_ok,
                           int num_sms, cudaStream_t stream)
{
    int grid = 0;
    const cudaError_t e = launch_grid(softmax_rows_kernel<T, C>, M, num_sms, &grid);
    if (e != cudaSuccess)
        return e;
    softmax_rows_kernel<T, C><<<grid, kThreads, 0, stream>>>(
        static_cast<const T *>(x), static_cast<T *>(y), M, N, chunks, vec_ok);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_rowop(bool softmax, const void *x, void *y, int M, int N, int num_sms,
                         cudaStream_t stream)
{
    constexpr int E = Chunk<T>::kElems;
    const long long per_pass = static_cast<long long>(kThreads) * E;
    const int chunks = static_cast<int>((N + per_pass - 1) / per_pass);
    const int vec_ok = (N % E == 0) && ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) &&
                       (!softmax || (reinterpret_cast<uintptr_t>(y) & 15u) == 0);
    if (!softmax) {
        int grid = 0;
        const cudaError_t e = launch_grid(row_sum_kernel<T>, M, num_sms, &grid);
        if (e != cudaSuccess)
            return e;
        row_sum_kernel<T><<<grid, kThreads, 0, stream>>>(static_cast<const T *>(x),
                                                         static_cast<float *>(y), M, N, chunks,
                                                         vec_ok);
        return cudaGetLastError();
    }
    constexpr int kMax = MaxChunks<T>::value;
    if (chunks <= 1)
        return launch_softmax<T, 1>(x, y, M, N, chunks, vec_ok, num_sms, stream);
    if (chunks <= 2)
        return launch_softmax<T, 2>(x, y, M, N, chunks, vec_ok, num_sms, stream);
    if (chunks <= 4)
        return launch_softmax<T, 4>(x, y, M, N, chunks, vec_ok, num_sms, stream);
    if (chunks <= 8)
        return launch_softmax<T, 8>(x, y, M, N, chunks, vec_ok, num_sms, stream);
    if (chunks <= kMax)
        return launch_softmax<T, kMax>(x, y, M, N, chunks, vec_ok, num_sms, stream);
    return launch_softmax<T, 0>(x, y, M, N, chunks, vec_ok, num_sms, stream);
}

}  // namespace

cudaError_t launch_softmax_rows(const void *x, void *y, int M, int N, int dtype, int num_sms,
                                cudaStream_t stream)
{
    return dtype == 0 ? launch_rowop<float>(true, x, y, M, N, num_sms, stream)
                      : launch_rowop<__nv_bfloat16>(true, x, y, M, N, num_sms, stream);
}

cudaError_t launch_row_sum(const void *x, float *out, int M, int N, int dtype, int num_sms,
                           cudaStream_t stream)
{
    return dtype == 0 ? launch_rowop<float>(false, x, out, M, N, num_sms, stream)
                      : launch_rowop<__nv_bfloat16>(false, x, out, M, N, num_sms, stream);
}

}  // namespace fattn
