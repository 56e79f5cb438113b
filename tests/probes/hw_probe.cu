// Hardware probe for the forward kernel's design numbers on this GPU: the
// throughput of the exponential unit (ex2.approx.ftz.f32, which the softmax
// issues once per score) and of the tcgen05 MMA shapes the kernel issues
// (S = Q K^T from shared memory, P V with P in tensor memory), alone and while
// eight warps stream the softmax's tensor-memory loads and stores.
// Built and run by tests/test_hw_probe_gpu.py; prints one line per figure.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#include "ptx_sm103.cuh"

using namespace fattn::ptx;

namespace {

constexpr int kMufuIters = 4096;
constexpr int kMufuChains = 8;
constexpr uint32_t kBox = 16384;  // one 128-row x 64-column bf16 swizzle box
// A (2 boxes), B (2 boxes) and a 256-row B (from box 4; its second K chunk
// starts one box in and spans two): 8 boxes bound every operand read.
constexpr uint32_t kBoxes = 8;

// Every thread runs kMufuChains independent chains x <- 2^x - 1 (x stays in
// [0, 1)); the block's elapsed SM clocks give exponentials per clock per SM.
__global__ void __launch_bounds__(1024, 1) mufu_kernel(float seed, unsigned long long *cycles,
                                                       float *sink)
{
    float x[kMufuChains];
#pragma unroll
    for (int c = 0; c < kMufuChains; ++c)
        x[c] = seed * static_cast<float>(c + 1) * (1.0f / kMufuChains);
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < kMufuIters; ++it) {
#pragma unroll
        for (int c = 0; c < kMufuChains; ++c)
            x[c] = ex2(x[c]) - 1.0f;
    }
    __syncthreads();
    const long long t1 = clock64();
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < kMufuChains; ++c)
        acc += x[c];
    if (acc == 12345.f)  // never true; keeps the chains alive
        sink[threadIdx.x] = acc;
    if (threadIdx.x == 0)
        cycles[blockIdx.x] = static_cast<unsigned long long>(t1 - t0);
}

// One thread issues `iters` rounds of MMAs of one mode; with `stream_tmem`
// warps 2..9 meanwhile load 128 TMEM columns and store 64 per round, as the
// softmax does.  Modes: 0 S (SS 128x128, K = 128), 1 P V (TS 128x128,
// K = 128), 2 both, 3 SS 128x256, 4 P V with N = 64, 5 P V with N = 80,
// 6 and 7 the same two P V shapes with P read from shared memory (SS; A laid
// out like Q in mode 0, B like V in modes 4 and 5).
__global__ void __launch_bounds__(320, 1) mma_kernel(int mode, int iters, int stream_tmem,
                                                     unsigned long long *cycles)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *tiles = smem_raw + (base - raw);
    for (int i = threadIdx.x; i < static_cast<int>(kBoxes * kBox / 4); i += blockDim.x)
        reinterpret_cast<uint32_t *>(tiles)[i] = 0x3c003c00u;  // small bf16 values
    fence_proxy_async_smem();
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_base;
    __shared__ volatile int stop;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&done), 1);
        fence_barrier_init();
        stop = 0;
    }
    if (threadIdx.x < 32) {
        tmem_alloc(smem_addr(&tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    const int warp = threadIdx.x / 32;
    const uint32_t a = base, b = base + 2 * kBox, b256 = base + 4 * kBox;
    if (warp >= 2 && stream_tmem) {
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t acc = 0;
        for (int round = 0; round < 1000000 && !stop; ++round) {
            uint32_t r[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld32(tmem + lane_off + 384 + (c & 1) * 32, r[c]);
            tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = r[0][i] ^ r[1][i + 16] ^ r[2][i] ^ r[3][i + 8];
            acc ^= pk[5];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_st16(tmem + lane_off + 448 + (c & 1) * 16, pk);
            tmem_wait_st();
        }
        if (acc == 0x9e3779b9u)
            cycles[1000] = acc;
    }
    if (threadIdx.x == 0) {
        const uint32_t id_s = idesc_bf16_f32(128, 128, false);
        const uint32_t id_s256 = idesc_bf16_f32(128, 256, false);
        const uint32_t id_pv = idesc_bf16_f32(128, 128, true);
        const uint32_t id_pv64 = idesc_bf16_f32(128, 64, true);
        const uint32_t id_pv80 = idesc_bf16_f32(128, 80, true);
        const long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
            if (mode == 0 || mode == 2)
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                    mma_ss(tmem, smem_desc(a + off, 16, 1024), smem_desc(b + off, 16, 1024), id_s,
                           kk > 0);
                }
            if (mode == 1 || mode == 2)
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + 256, tmem + 128 + kk * 8, smem_desc(b + kk * 2048, kBox, 1024),
                           id_pv, 1);
            if (mode == 3)
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                    mma_ss(tmem, smem_desc(a + off, 16, 1024), smem_desc(b256 + off, 16, 1024),
                           id_s256, kk > 0);
                }
            if (mode == 4)
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + 256, tmem + 128 + kk * 8, smem_desc(b + kk * 2048, 1024, 1024),
                           id_pv64, 1);
            if (mode == 5)  // N = 80: the second 64-column atom is the next box
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tmem + 256, tmem + 128 + kk * 8, smem_desc(b + kk * 2048, kBox, 1024),
                           id_pv80, 1);
            if (mode == 6 || mode == 7)
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                    mma_ss(tmem + 256, smem_desc(a + off, 16, 1024),
                           smem_desc(b + kk * 2048, mode == 6 ? 1024 : kBox, 1024),
                           mode == 6 ? id_pv64 : id_pv80, 1);
                }
        }
        mma_commit(smem_addr(&done));
        const bool ok = mbar_wait(smem_addr(&done), 0, 2000000000ull, nullptr);
        const long long t1 = clock64();
        cycles[blockIdx.x] = ok ? static_cast<unsigned long long>(t1 - t0) : 0ull;
        stop = 1;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

int main()
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    unsigned long long *cycles = nullptr;
    float *sink = nullptr;
    if (cudaMalloc(&cycles, 1024 * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMalloc(&sink, 1024 * sizeof(float)) != cudaSuccess) {
        printf("error cudaMalloc\n");
        return 1;
    }
    unsigned long long h[1024];
    printf("sms %d\n", sms);

    for (int rep = 0; rep < 2; ++rep) {  // the first launch warms up
        mufu_kernel<<<sms, 1024>>>(0.37f, cycles, sink);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            printf("error %s\n", cudaGetErrorString(e));
            return 1;
        }
    }
    cudaMemcpy(h, cycles, sms * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    unsigned long long worst = 0;
    for (int i = 0; i < sms; ++i)
        worst = h[i] > worst ? h[i] : worst;
    printf("mufu_ex2_per_clk_per_sm %.2f\n",
           1024.0 * kMufuChains * kMufuIters / static_cast<double>(worst));

    const int smem = kBoxes * kBox + 1024;
    cudaFuncSetAttribute(mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const char *names[] = {"s_ss_128x128x16", "pv_ts_128x128x16", "s_and_pv", "s_ss_128x256x16",
                           "pv_ts_128x64x16", "pv_ts_128x80x16", "pv_ss_128x64x16",
                           "pv_ss_128x80x16"};
    const double flops[] = {128.0 * 128 * 32, 128.0 * 128 * 32, 128.0 * 128 * 32,
                            128.0 * 256 * 32, 128.0 * 64 * 32,  128.0 * 80 * 32,
                            128.0 * 64 * 32,  128.0 * 80 * 32};
    for (int stream_tmem = 0; stream_tmem < 2; ++stream_tmem)
        for (int mode = 0; mode < 8; ++mode) {
            if (stream_tmem && mode != 2)
                continue;
            const int iters = 2000;
            mma_kernel<<<sms, 320, smem>>>(mode, iters, stream_tmem, cycles);
            cudaError_t e = cudaDeviceSynchronize();
            if (e != cudaSuccess) {
                printf("error %s\n", cudaGetErrorString(e));
                return 1;
            }
            cudaMemcpy(h, cycles, sms * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
            worst = 0;
            for (int i = 0; i < sms; ++i) {
                if (h[i] == 0) {
                    printf("error mma wait timed out\n");
                    return 1;
                }
                worst = h[i] > worst ? h[i] : worst;
            }
            const double n = iters * (mode == 2 ? 16.0 : 8.0);
            printf("mma_%s%s clk_per_instr %.1f flop_per_clk_per_sm %.0f\n", names[mode],
                   stream_tmem ? "_with_tmem_traffic" : "", worst / n, flops[mode] * n / worst);
        }
    cudaFree(cycles);
    cudaFree(sink);
    return 0;
}
