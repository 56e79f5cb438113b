// fattn_api.cu -- the C ABI of libfattn (see include/fattn.h).
//
// Validation follows the wrapper conventions of "Triton programming
// template" (check device, shape, dtype and layout before launching; return
// early for empty inputs; launch asynchronously on the caller's stream).  All
// checks are synchronous and nothing is enqueued when one fails.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "fattn.h"
#include "fattn_internal.h"

namespace {

thread_local int t_last_cuda_error = 0;

fattn_status_t cuda_fail(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
    return FATTN_ERR_CUDA;
}

// Per-device facts, read once.
struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    int dev = -1;
};
constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

fattn_status_t current_device(int *dev, DeviceInfo *info)
{
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (*dev < 0 || *dev >= kMaxDevices)
        return FATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_dev[*dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess)
            return cuda_fail(e);
        d.supported = (major == 10 && minor == 3);  // the kernels are built for sm_103a only
        d.num_sms = sms;
        d.dev = *dev;
        d.probed = true;
    }
    *info = d;
    return d.supported ? FATTN_OK : FATTN_ERR_UNSUPPORTED;
}

fattn_status_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn)
{
    std::call_once(g_encode_once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
            g_encode_err = cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (g_encode_err != cudaSuccess || g_encode == nullptr)
        return cuda_fail(g_encode_err != cudaSuccess ? g_encode_err : cudaErrorSymbolNotFound);
    *fn = g_encode;
    return FATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Shape and scalar checks that need no device.  Sets *empty when there is no
// work (B*H*N == 0).
fattn_status_t check_shape(int B, int H, int N, int d, float scale, int causal, bool *empty)
{
    if (B < 0 || H < 0 || N < 0)
        return FATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1)
        return FATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale))
        return FATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 96 && d != 128 && d != 256)
        return FATTN_ERR_UNSUPPORTED;
    const long long rows = static_cast<long long>(B) * H * N;
    *empty = rows == 0;
    // Each tensor must stay below 2^40 bytes (tensor-map stride limit) and
    // B*H must fit the tensor map's outer dimension.
    if (static_cast<long long>(B) * H > 0x7fffffffLL)
        return FATTN_ERR_UNSUPPORTED;
    if (!*empty && rows > (1LL << 39) / (2LL * d))
        return FATTN_ERR_UNSUPPORTED;
    return FATTN_OK;
}

// Key-length checks of a call whose keys (Nk) may differ from its queries
// (Nq): Nk >= 0, at least one key when there are queries, Nq <= Nk under the
// causal mask (the queries are the last Nq key positions), and K, V within the
// same size limit as Q.
fattn_status_t check_keys(int B, int H, int Nq, int Nk, int d, int causal)
{
    if (Nk < 0)
        return FATTN_ERR_INVALID_ARG;
    const long long q_rows = static_cast<long long>(B) * H * Nq;
    if (q_rows > 0 && Nk == 0)
        return FATTN_ERR_INVALID_ARG;
    if (causal && Nq > Nk)
        return FATTN_ERR_INVALID_ARG;
    if (q_rows > 0 && static_cast<long long>(B) * H * Nk > (1LL << 39) / (2LL * d))
        return FATTN_ERR_UNSUPPORTED;
    return FATTN_OK;
}

// Pointer checks: non-null, 16-byte aligned, no output overlapping an input or
// the other output.  q_bytes covers q and o, kv_bytes each of k and v.
fattn_status_t check_pointers(const void *q, const void *k, const void *v, const void *o,
                              const float *lse, size_t q_bytes, size_t kv_bytes, size_t lse_bytes)
{
    if (!q || !k || !v || !o || !lse)
        return FATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FATTN_ERR_INVALID_ARG;
    if (overlap(o, q_bytes, q, q_bytes) || overlap(o, q_bytes, k, kv_bytes) ||
        overlap(o, q_bytes, v, kv_bytes) || overlap(o, q_bytes, lse, lse_bytes) ||
        overlap(lse, lse_bytes, q, q_bytes) || overlap(lse, lse_bytes, k, kv_bytes) ||
        overlap(lse, lse_bytes, v, kv_bytes))
        return FATTN_ERR_INVALID_ARG;
    return FATTN_OK;
}

// The buffer must be device (or managed) memory of the current device.
fattn_status_t check_device_buffer(const void *p, int dev)
{
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error state of this query
        return FATTN_ERR_INVALID_ARG;
    }
    if (attr.type == cudaMemoryTypeDevice)
        return attr.device == dev ? FATTN_OK : FATTN_ERR_INVALID_ARG;
    if (attr.type == cudaMemoryTypeManaged)
        return FATTN_OK;
    return FATTN_ERR_INVALID_ARG;
}

fattn_status_t make_map(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *m, const void *ptr,
                        int N, int d, long long BH, bool f16 = false)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    const CUresult r = encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              3, const_cast<void *>(ptr), dims,
                              strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return FATTN_ERR_CUDA;
    }
    return FATTN_OK;
}

// Element strides (batch, head, row) of q, k, v and o; the last dimension
// (d) is contiguous.
struct Layout {
    long long q[3], k[3], v[3], o[3];
};

Layout dense_layout(int H, int N, int Nk, int d)
{
    const long long qn = d, qh = static_cast<long long>(N) * d, qb = qh * H;
    const long long kh = static_cast<long long>(Nk) * d, kb = kh * H;
    return Layout{{qb, qh, qn}, {kb, kh, qn}, {kb, kh, qn}, {qb, qh, qn}};
}

// Bytes from a tensor's base to one past its last element.
size_t span_bytes(const long long st[3], int B, int H, int rows, int d)
{
    return static_cast<size_t>(st[0] * (B - 1) + st[1] * (H - 1) +
                               st[2] * static_cast<long long>(rows - 1) + d) * 2;
}

// 4-D map (d, rows, H, B) of a 16-bit tensor with element strides st
// (batch, head, row), box (64, box_rows, 1, 1), 128-byte swizzle, zero fill
// outside the tensor.  box_rows is 128 (one tile's rows), or 64 for V at
// d = 256, whose kernel copies each V tile as two halves of 64 keys.
fattn_status_t make_map4(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *m,
                         const void *ptr, int rows, int d, int H, int B, const long long st[3],
                         bool f16, unsigned box_rows = 128)
{
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2,
                                   static_cast<cuuint64_t>(st[1]) * 2,
                                   static_cast<cuuint64_t>(st[0]) * 2};
    const cuuint32_t box[4] = {64, box_rows, 1, 1};
    const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
    const CUresult r = encode(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              4, const_cast<void *>(ptr), dims, strides, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return FATTN_ERR_CUDA;
    }
    return FATTN_OK;
}

// Stride rules of a strided call: every stride a positive multiple of 8
// elements (16 bytes, the tensor-map rule; o is written in 16-byte pieces),
// each tensor's span below 2^39 bytes, o's elements all distinct (nested
// strides: sorted by size, each stride at least the span of the smaller
// dimensions), and no output overlapping an input or the other output.
fattn_status_t check_layout(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, int B, int H, int N, int Nk, int d, const Layout &L)
{
    if (!q || !k || !v || !o || !lse)
        return FATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FATTN_ERR_INVALID_ARG;
    const long long *all[4] = {L.q, L.k, L.v, L.o};
    const int rows[4] = {N, Nk, Nk, N};
    size_t span[4];
    for (int t = 0; t < 4; ++t) {
        for (int i = 0; i < 3; ++i)
            if (all[t][i] < 1 || all[t][i] % 8 != 0 || all[t][i] > (1LL << 38))
                return FATTN_ERR_INVALID_ARG;
        const long double far = static_cast<long double>(all[t][0]) * (B - 1) +
                                static_cast<long double>(all[t][1]) * (H - 1) +
                                static_cast<long double>(all[t][2]) * (rows[t] - 1) + d;
        if (far * 2 >= static_cast<long double>(1LL << 39))
            return FATTN_ERR_UNSUPPORTED;
        span[t] = span_bytes(all[t], B, H, rows[t], d);
    }
    // o: nested strides over the dimensions of extent > 1.
    long long st[3] = {L.o[2], L.o[1], L.o[0]};
    long long ext[3] = {N, H, B};
    for (int i = 0; i < 3; ++i)  // sort by stride (3 elements)
        for (int j = i + 1; j < 3; ++j)
            if (st[j] < st[i]) {
                long long t = st[i]; st[i] = st[j]; st[j] = t;
                t = ext[i]; ext[i] = ext[j]; ext[j] = t;
            }
    long long covered = d;
    for (int i = 0; i < 3; ++i) {
        if (ext[i] <= 1)
            continue;
        if (st[i] < covered)
            return FATTN_ERR_INVALID_ARG;
        covered += st[i] * (ext[i] - 1);
    }
    const size_t lb = static_cast<size_t>(B) * H * N * 4;
    if (overlap(o, span[3], q, span[0]) || overlap(o, span[3], k, span[1]) ||
        overlap(o, span[3], v, span[2]) || overlap(o, span[3], lse, lb) ||
        overlap(lse, lb, q, span[0]) || overlap(lse, lb, k, span[1]) ||
        overlap(lse, lb, v, span[2]))
        return FATTN_ERR_INVALID_ARG;
    return FATTN_OK;
}

// kTcgen05: bf16, P in fp16 (V converted on chip); kTcgen05F16: fp16;
// kTcgen05Bf16P: bf16, P in bf16; kSimt: the fp32 cross-check kernel.
enum class Kernel { kTcgen05, kTcgen05F16, kTcgen05Bf16P, kSimt };

// Every check of a forward call with N queries and Nk keys per head.  On
// FATTN_OK, *empty tells whether there is any work, and (when there is)
// *dev / *info describe the current device.
// L == nullptr: contiguous tensors.
fattn_status_t validate(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, int B, int H, int N, int Nk, int d, float scale,
                        int causal, bool *empty, int *dev, DeviceInfo *info,
                        const Layout *L = nullptr)
{
    fattn_status_t s = check_shape(B, H, N, d, scale, causal, empty);
    if (s != FATTN_OK)
        return s;
    if ((s = check_keys(B, H, N, Nk, d, causal)) != FATTN_OK || *empty)
        return s;
    const size_t rows = static_cast<size_t>(B) * H * N;
    const size_t kv_bytes = static_cast<size_t>(B) * H * Nk * d * 2;
    if (L != nullptr)
        s = check_layout(q, k, v, o, lse, B, H, N, Nk, d, *L);
    else
        s = check_pointers(q, k, v, o, lse, rows * d * 2, kv_bytes, rows * 4);
    if (s != FATTN_OK)
        return s;
    if ((s = current_device(dev, info)) != FATTN_OK)
        return s;
    const void *bufs[5] = {q, k, v, o, lse};
    for (const void *p : bufs)
        if ((s = check_device_buffer(p, *dev)) != FATTN_OK)
            return s;
    return FATTN_OK;
}

// ---------------------------------------------------------------- V pre-pass
// For bf16 inputs with P in fp16, V is rounded to fp16 either on chip, per
// work unit, by the forward kernel's converter warps, or once per call by a
// pre-pass into scratch that the forward kernel then reads (the same bits
// either way).  The scratch comes from one stream-ordered memory pool per
// device, created on first use, which keeps freed blocks for the next call
// (release threshold: unlimited), so a steady loop of calls maps no new
// device memory; fattn_trim_scratch returns them.
std::atomic<int> g_v_convert{FATTN_V_CONVERT_AUTO};
std::mutex g_pool_mutex;
cudaMemPool_t g_pool[kMaxDevices] = {};

// FATTN_V_CONVERT_AUTO: the pre-pass where it was measured to pay.  The
// converter warps round each V tile once for every work unit that reads it
// (a pair of 128-row Q tiles, one Q tile at d = 256), on average `visits`
// times: the units per head, halved under the causal mask.  The pre-pass
// costs a fixed 4 bytes of HBM traffic per V element and one more launch.
// On one GB300 (bf16, L2 flushed) it was faster from these visits on and
// slower below them: d = 64 from 24 (16: -0.4 %, 24: +2 %, 256: +4 %);
// d = 96 from 8 (4: -3 % to +1 %, 8: +4.5 %); d = 128 from 16 (12: -1.5 %,
// 16: +0.6 % causal and +3 % not, 32: +3 to +5 %); d = 256 from 12 (8: -1 %
// to -6 %, 12: +13 %, 32: +36 %).
enum class VRoute { kOnChip, kPrepass };

VRoute v_route(int Nq, int d, int causal)
{
    if (Nq <= 0)
        return VRoute::kOnChip;
    const int mode = g_v_convert.load(std::memory_order_relaxed);
    if (mode == FATTN_V_CONVERT_PREPASS)
        return VRoute::kPrepass;
    if (mode == FATTN_V_CONVERT_ON_CHIP)
        return VRoute::kOnChip;
    const long long tiles = (static_cast<long long>(Nq) + 127) / 128;
    const long long units = d == 256 ? tiles : (tiles + 1) / 2;
    const long long visits2 = causal ? units : 2 * units;  // twice the visits
    const long long need2 = d == 64 ? 48 : d == 96 ? 16 : d == 128 ? 32 : 24;
    return visits2 >= need2 ? VRoute::kPrepass : VRoute::kOnChip;
}


// Scratch of `bytes` on `stream`, or nullptr where there is none to be had
// (the stream is being captured into a graph, the pool cannot be created or
// the device is out of memory): the caller then converts on chip.
void *prepass_scratch(int dev, size_t bytes, cudaStream_t stream)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return nullptr;
    }
    cudaMemPool_t pool = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_pool_mutex);
        if (g_pool[dev] == nullptr) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t created = nullptr;
            if (cudaMemPoolCreate(&created, &props) != cudaSuccess) {
                cudaGetLastError();
                return nullptr;
            }
            uint64_t keep = UINT64_MAX;
            cudaMemPoolSetAttribute(created, cudaMemPoolAttrReleaseThreshold, &keep);
            g_pool[dev] = created;
        }
        pool = g_pool[dev];
    }
    void *ptr = nullptr;
    if (cudaMallocFromPoolAsync(&ptr, bytes, pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return ptr;
}

// Enqueue one validated forward call with N queries and Nk keys per head
// (split.splits > 1: key-range split with the caller's scratch).
// may_allocate false: no device memory is taken (V is converted on chip).
fattn_status_t launch(Kernel which, const DeviceInfo &info, const void *q, const void *k,
                      const void *v, void *o, float *lse, int B, int H, int N, int Nk, int d,
                      float scale, int causal, cudaStream_t stream,
                      const fattn::FwdSplit &split = fattn::FwdSplit{1, nullptr, nullptr},
                      const Layout *L = nullptr, bool may_allocate = true)
{
    fattn::FwdArgs a{q, k, v, o, lse, B, H, N, d, scale, causal};
    const bool f16 = which == Kernel::kTcgen05F16;
    a.f16 = f16 ? 1 : 0;
    a.bf16p = which == Kernel::kTcgen05Bf16P ? 1 : 0;
    a.Nk = Nk;
    cudaError_t e;
    if (which == Kernel::kSimt) {
        if (Nk != N || L != nullptr || d > 128)
            return FATTN_ERR_UNSUPPORTED;
        e = fattn::launch_fwd_simt(a, stream);
    } else {
        PFN_cuTensorMapEncodeTiled_v12000 encode;
        fattn_status_t s;
        if ((s = get_encoder(&encode)) != FATTN_OK)
            return s;
        const Layout lay = L != nullptr ? *L : dense_layout(H, N, Nk, d);
        a.o_sb = lay.o[0];
        a.o_sh = lay.o[1];
        a.o_sn = lay.o[2];
        fattn::FwdMaps maps;
        if ((s = make_map4(encode, &maps.q, q, N, d, H, B, lay.q, f16)) != FATTN_OK ||
            (s = make_map4(encode, &maps.k, k, Nk, d, H, B, lay.k, f16)) != FATTN_OK)
            return s;
        void *v16 = nullptr;
        const unsigned v_box_rows = d == 256 ? 64u : 128u;
        if (which == Kernel::kTcgen05 && may_allocate && v_route(N, d, causal) == VRoute::kPrepass)
            v16 = prepass_scratch(info.dev, static_cast<size_t>(B) * H * Nk * d * 2, stream);
        if (v16 != nullptr) {
            const Layout dense = dense_layout(H, N, Nk, d);
            a.v16 = v16;
            a.v_sb = lay.v[0];
            a.v_sh = lay.v[1];
            a.v_sn = lay.v[2];
            s = make_map4(encode, &maps.v, v16, Nk, d, H, B, dense.v, true, v_box_rows);
        } else {
            s = make_map4(encode, &maps.v, v, Nk, d, H, B, lay.v, f16, v_box_rows);
        }
        e = s == FATTN_OK ? fattn::launch_fwd_sm103(a, maps, split, info.num_sms, stream)
                          : cudaSuccess;
        if (v16 != nullptr) {
            const cudaError_t ef = cudaFreeAsync(v16, stream);
            if (e == cudaSuccess)
                e = ef;
        }
        if (s != FATTN_OK)
            return s;
    }
    return e == cudaSuccess ? FATTN_OK : cuda_fail(e);
}

fattn_status_t forward(Kernel which, const void *q, const void *k, const void *v, void *o,
                       float *lse, int B, int H, int N, int d, float scale, int causal,
                       cudaStream_t stream, bool may_allocate = true)
{
    bool empty = false;
    int dev = 0;
    DeviceInfo info;
    fattn_status_t s =
        validate(q, k, v, o, lse, B, H, N, N, d, scale, causal, &empty, &dev, &info);
    if (s != FATTN_OK || empty)
        return s;
    return launch(which, info, q, k, v, o, lse, B, H, N, N, d, scale, causal, stream,
                  fattn::FwdSplit{1, nullptr, nullptr}, nullptr, may_allocate);
}

constexpr int kMaxSplits = 64;
constexpr size_t kWsAlign = 256;


// Scratch layout of a split call: fp32 partial O, then (256-byte aligned) the
// base-2 partial lse pairs.
size_t split_ws_o_bytes(int B, int H, int N, int d, int splits)
{
    return static_cast<size_t>(splits) * B * H * N * d * sizeof(float);
}
size_t split_ws_bytes(int B, int H, int N, int d, int splits)
{
    if (splits <= 1)
        return 0;
    return align_up(split_ws_o_bytes(B, H, N, d, splits), kWsAlign) +
           static_cast<size_t>(splits) * B * H * N * 2 * sizeof(float);
}

// Splits for a grid of fewer work units than SMs: the s (at most one split
// per two key tiles, at most kMaxSplits) that minimises the estimated time in
// key-tile steps: ceil(units * s / SMs) rounds of ceil(KT / s) steps plus
// kUnitCost steps per unit (Q load, pipeline fill, epilogue), plus
// kMergeCost steps for the partial outputs and their merge when s > 1 (both
// measured on one and four splits of 16 pairs x 32 key tiles, d = 64).  Ties
// go to the smaller s.
constexpr long long kUnitCost = 3, kMergeCost = 6;
int choose_splits(int B, int H, int Nq, int Nk, int d, int num_sms)
{
    // A work unit is a pair of 128-row Q tiles, or one Q tile for d = 256.
    const long long q_tiles = (static_cast<long long>(Nq) + 127) / 128;
    const long long pairs = d == 256 ? q_tiles : (q_tiles + 1) / 2;
    const long long units = static_cast<long long>(B) * H * pairs;
    const long long key_tiles = (static_cast<long long>(Nk) + 127) / 128;
    if (units <= 0 || units >= num_sms)
        return 1;
    long long best_s = 1, best = key_tiles + kUnitCost;
    const long long s_max = key_tiles / 2 < kMaxSplits ? key_tiles / 2 : kMaxSplits;
    for (long long s = 2; s <= s_max; ++s) {
        const long long rounds = (units * s + num_sms - 1) / num_sms;
        const long long est = rounds * ((key_tiles + s - 1) / s + kUnitCost) + kMergeCost;
        if (est < best) {
            best = est;
            best_s = s;
        }
    }
    return static_cast<int>(best_s);
}

// The automatic schedule of attn_fwd_kv: stream-K for one Q-tile pair per
// head when whole heads would leave SMs idle, else choose_splits.  Returns
// the partial slots per head (1: no split).
int auto_slots(int B, int H, int Nq, int Nk, int d, int causal, int num_sms, int *streamk)
{
    const fattn::FwdPlan plan = fattn::plan_fwd_streamk(B, H, Nq, Nk, causal, num_sms);
    *streamk = plan.streamk;
    return plan.streamk ? plan.slots : choose_splits(B, H, Nq, Nk, d, num_sms);
}

// num_splits == 0: the automatic schedule for the current device.
// L == nullptr: contiguous tensors.
fattn_status_t forward_split(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int Nk, int d, float scale, int causal,
                             int num_splits, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream, const Layout *L = nullptr,
                             Kernel which = Kernel::kTcgen05, bool may_allocate = true)
{
    if (num_splits < 0 || num_splits > kMaxSplits)
        return FATTN_ERR_INVALID_ARG;
    bool empty = false;
    int dev = 0;
    DeviceInfo info;
    fattn_status_t s =
        validate(q, k, v, o, lse, B, H, N, Nk, d, scale, causal, &empty, &dev, &info, L);
    if (s != FATTN_OK || empty)
        return s;
    int streamk = 0;
    if (num_splits == 0)
        num_splits = auto_slots(B, H, N, Nk, d, causal, info.num_sms, &streamk);
    if (num_splits == 1)
        return launch(which, info, q, k, v, o, lse, B, H, N, Nk, d, scale, causal, stream,
                      fattn::FwdSplit{1, nullptr, nullptr}, L, may_allocate);
    const size_t need = split_ws_bytes(B, H, N, d, num_splits);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return FATTN_ERR_INVALID_ARG;
    const Layout lay = L != nullptr ? *L : dense_layout(H, N, Nk, d);
    const size_t lb = static_cast<size_t>(B) * H * N * 4;
    if (overlap(workspace, need, q, span_bytes(lay.q, B, H, N, d)) ||
        overlap(workspace, need, k, span_bytes(lay.k, B, H, Nk, d)) ||
        overlap(workspace, need, v, span_bytes(lay.v, B, H, Nk, d)) ||
        overlap(workspace, need, o, span_bytes(lay.o, B, H, N, d)) ||
        overlap(workspace, need, lse, lb))
        return FATTN_ERR_INVALID_ARG;
    if ((s = check_device_buffer(workspace, dev)) != FATTN_OK)
        return s;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const fattn::FwdSplit split{
        num_splits, reinterpret_cast<float *>(ws),
        reinterpret_cast<float *>(ws + align_up(split_ws_o_bytes(B, H, N, d, num_splits), kWsAlign)),
        streamk};
    return launch(which, info, q, k, v, o, lse, B, H, N, Nk, d, scale, causal, stream, split, L,
                  may_allocate);
}

// ---------------------------------------------------------------- no-allocation split
// Scratch for attn_fwd_split_noalloc: a fixed device array that lives as long
// as the library is loaded, so that callers that may not allocate device
// memory on their execution path still get the split kernel.  Its device
// address is looked up once per device (cudaGetSymbolAddress, with that device
// current); in host code the array's name is only a host-side stand-in.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

fattn_status_t noalloc_scratch(int dev, void **out)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return FATTN_OK;
}

// attn_fwd_host's copy/compute pipeline: per-device helper streams and
// events, created on first use and kept for the process.  Calls are
// serialised by g_pipe_mutex (each call synchronises before it returns).
constexpr int kHostChunks = 16;

// Head ranges [bounds[c], bounds[c+1]) of that pipeline.  Nothing overlaps
// the first chunk's copy in, nor the last chunk's kernel and copy out, so the
// ends are kept short: chunks of m/4 and m/2 heads first, equal chunks of
// about m = ceil(BH/8) in the middle, m/2 and m/4 last.  No chunk has fewer
// than min_heads heads, the heads that give every SM a work unit: a chunk's
// kernel lasts at least as long as its heaviest unit, so smaller chunks would
// only leave SMs idle.  Shapes too small for the ramps get equal chunks.
// Returns the number of chunks (at most 11).
int host_chunk_plan(long long BH, long long min_heads, long long bounds[kHostChunks + 1])
{
    const long long m = std::max((BH + 7) / 8, min_heads);
    const long long q = std::max(m / 4, min_heads), h = std::max(m / 2, min_heads);
    const long long rest = BH - 2 * (q + h);
    int n = 0;
    bounds[0] = 0;
    if (rest < m) {
        n = static_cast<int>(std::min<long long>((BH + m - 1) / m, 8));
        for (int c = 1; c <= n; ++c)
            bounds[c] = BH * c / n;
        return n;
    }
    const long long k = rest / m;  // middle chunks, 1..7
    for (long long sz : {q, h})
        bounds[n + 1] = bounds[n] + sz, ++n;
    for (long long i = 0; i < k; ++i)
        bounds[n + 1] = bounds[n] + rest / k + (i < rest % k ? 1 : 0), ++n;
    for (long long sz : {h, q})
        bounds[n + 1] = bounds[n] + sz, ++n;
    return n;
}
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t ev_in[kHostChunks] = {}, ev_done[kHostChunks] = {};
};
std::mutex g_pipe_mutex;
HostPipe g_pipe[kMaxDevices];

fattn_status_t host_pipe(int dev, HostPipe **out)
{
    HostPipe &hp = g_pipe[dev];
    if (!hp.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
        for (int c = 0; c < kHostChunks && e == cudaSuccess; ++c) {
            e = cudaEventCreateWithFlags(&hp.ev_in[c], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&hp.ev_done[c], cudaEventDisableTiming);
        }
        if (e != cudaSuccess)
            return cuda_fail(e);
        hp.ready = true;
    }
    *out = &hp;
    return FATTN_OK;
}

}  // namespace

extern "C" {

fattn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                        int H, int N, int d, float scale, int causal, struct CUstream_st *stream)
{
    return forward(Kernel::kTcgen05, q, k, v, o, lse, B, H, N, d, scale, causal, stream);
}

fattn_status_t attn_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, float scale, int causal,
                             struct CUstream_st *stream)
{
    return forward(Kernel::kTcgen05F16, q, k, v, o, lse, B, H, N, d, scale, causal, stream);
}

int attn_fwd_split_count(int B, int H, int N, int d, int causal)
{
    bool empty = false;
    if (check_shape(B, H, N, d, 1.0f, causal, &empty) != FATTN_OK)
        return 0;
    if (empty)
        return 1;
    int dev = 0;
    DeviceInfo info;
    if (current_device(&dev, &info) != FATTN_OK)
        return 0;
    return choose_splits(B, H, N, N, d, info.num_sms);
}

size_t attn_fwd_split_workspace_size(int B, int H, int N, int d, int num_splits)
{
    bool empty = false;
    if (num_splits < 1 || num_splits > kMaxSplits ||
        check_shape(B, H, N, d, 1.0f, 0, &empty) != FATTN_OK || empty)
        return 0;
    return split_ws_bytes(B, H, N, d, num_splits);
}

fattn_status_t attn_fwd_split(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int H, int N, int d, float scale, int causal, int num_splits,
                              void *workspace, size_t workspace_bytes, struct CUstream_st *stream)
{
    if (num_splits < 1)
        return FATTN_ERR_INVALID_ARG;
    return forward_split(q, k, v, o, lse, B, H, N, N, d, scale, causal, num_splits, workspace,
                         workspace_bytes, stream);
}

fattn_status_t attn_fwd_strided(const void *q, const void *k, const void *v, void *o,
                                float *lse, int B, int H, int Nq, int Nk, int d,
                                const long long *q_strides, const long long *k_strides,
                                const long long *v_strides, const long long *o_strides,
                                float scale, int causal, int num_splits, void *workspace,
                                size_t workspace_bytes, int dtype, struct CUstream_st *stream)
{
    if (!q_strides || !k_strides || !v_strides || !o_strides || dtype < 0 || dtype > 2)
        return FATTN_ERR_INVALID_ARG;
    Layout L;
    for (int i = 0; i < 3; ++i) {
        L.q[i] = q_strides[i];
        L.k[i] = k_strides[i];
        L.v[i] = v_strides[i];
        L.o[i] = o_strides[i];
    }
    // A dimension of extent 1 has no meaningful stride: give it the span of
    // the smaller dimensions, as a contiguous tensor would have.
    long long *all[4] = {L.q, L.k, L.v, L.o};
    const int rows[4] = {Nq, Nk, Nk, Nq};
    for (int t = 0; t < 4; ++t) {
        if (rows[t] == 1)
            all[t][2] = (static_cast<long long>(d) + 7) / 8 * 8;
        if (H == 1)
            all[t][1] = all[t][2] * (rows[t] > 0 ? rows[t] : 1);
        if (B == 1)
            all[t][0] = all[t][1] * (H > 0 ? H : 1);
    }
    return forward_split(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, workspace,
                         workspace_bytes, stream, &L,
                         dtype == 1 ? Kernel::kTcgen05F16
                                    : (dtype == 2 ? Kernel::kTcgen05Bf16P : Kernel::kTcgen05));
}

size_t attn_fwd_kv_workspace_size(int B, int H, int Nq, int Nk, int d, int causal,
                                  int num_splits)
{
    bool empty = false;
    if (num_splits < 0 || num_splits > kMaxSplits ||
        check_shape(B, H, Nq, d, 1.0f, causal, &empty) != FATTN_OK ||
        check_keys(B, H, Nq, Nk, d, causal) != FATTN_OK || empty)
        return 0;
    if (num_splits == 0) {
        int dev = 0, streamk = 0;
        DeviceInfo info;
        if (current_device(&dev, &info) != FATTN_OK)
            return 0;
        num_splits = auto_slots(B, H, Nq, Nk, d, causal, info.num_sms, &streamk);
    }
    return split_ws_bytes(B, H, Nq, d, num_splits);
}

fattn_status_t attn_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int H, int Nq, int Nk, int d, float scale, int causal,
                           int num_splits, void *workspace, size_t workspace_bytes,
                           struct CUstream_st *stream)
{
    return forward_split(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, workspace,
                         workspace_bytes, stream);
}

fattn_status_t attn_fwd_split_noalloc(const void *q, const void *k, const void *v, void *o,
                                      float *lse, int B, int H, int N, int d, float scale,
                                      int causal, int num_splits, struct CUstream_st *stream)
{
    if (num_splits < 1 || num_splits > kMaxSplits)
        return FATTN_ERR_INVALID_ARG;
    bool empty = false;
    fattn_status_t s = check_shape(B, H, N, d, scale, causal, &empty);
    if (s != FATTN_OK || empty)
        return s;
    if (num_splits == 1)  // no scratch needed: attn_fwd's result (V converted on chip)
        return forward(Kernel::kTcgen05, q, k, v, o, lse, B, H, N, d, scale, causal, stream,
                       false);
    if (split_ws_bytes(B, H, N, d, num_splits) > kNoAllocScratchBytes)
        return FATTN_ERR_UNSUPPORTED;  // beyond the fixed scratch: use attn_fwd_split
    int dev = 0;
    DeviceInfo info;
    if ((s = current_device(&dev, &info)) != FATTN_OK)
        return s;
    void *scratch = nullptr;
    if ((s = noalloc_scratch(dev, &scratch)) != FATTN_OK)
        return s;
    return forward_split(q, k, v, o, lse, B, H, N, N, d, scale, causal, num_splits, scratch,
                         kNoAllocScratchBytes, stream, nullptr, Kernel::kTcgen05, false);
}

int fattn_set_v_conversion(int mode)
{
    if (mode < FATTN_V_CONVERT_AUTO || mode > FATTN_V_CONVERT_PREPASS)
        return -1;
    return g_v_convert.exchange(mode);
}

int fattn_v_conversion_route(int N, int d, int causal)
{
    if (N < 0 || (d != 64 && d != 96 && d != 128 && d != 256) || (causal != 0 && causal != 1))
        return -1;
    return v_route(N, d, causal) == VRoute::kPrepass ? FATTN_V_CONVERT_PREPASS
                                                     : FATTN_V_CONVERT_ON_CHIP;
}

fattn_status_t fattn_trim_scratch(void)
{
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    for (int dev = 0; dev < kMaxDevices; ++dev) {
        if (g_pool[dev] == nullptr)
            continue;
        const cudaError_t e = cudaMemPoolTrimTo(g_pool[dev], 0);
        if (e != cudaSuccess)
            return cuda_fail(e);
    }
    return FATTN_OK;
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d)
{
    bool empty = false;
    if ((d != 64 && d != 128) || check_shape(B, H, N, d, 1.0f, 0, &empty) != FATTN_OK || empty)
        return 0;
    return static_cast<size_t>(B) * H * N * sizeof(float);
}

fattn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                        int H, int N, int d, float scale, int causal, void *workspace,
                        size_t workspace_bytes, struct CUstream_st *stream)
{
    bool empty = false;
    fattn_status_t s = check_shape(B, H, N, d, scale, causal, &empty);
    if (s != FATTN_OK || empty)
        return s;
    if (d != 64 && d != 128)  // the backward kernels take d = 64 or 128
        return FATTN_ERR_UNSUPPORTED;
    const size_t rows = static_cast<size_t>(B) * H * N;
    const size_t tb = rows * d * 2, lb = rows * 4;
    const void *ins[6] = {q, k, v, o, lse, dout};
    const size_t in_bytes[6] = {tb, tb, tb, tb, lb, tb};
    void *outs[4] = {dq, dk, dv, workspace};
    const size_t out_bytes[4] = {tb, tb, tb, lb};
    for (const void *p : ins)
        if (!p || !aligned16(p))
            return FATTN_ERR_INVALID_ARG;
    for (void *p : outs)
        if (!p || !aligned16(p))
            return FATTN_ERR_INVALID_ARG;
    if (workspace_bytes < lb)
        return FATTN_ERR_INVALID_ARG;
    // Outputs (and the scratch) overlap neither each other nor any input.
    for (int a = 0; a < 4; ++a) {
        for (int i = 0; i < 6; ++i)
            if (overlap(outs[a], out_bytes[a], ins[i], in_bytes[i]))
                return FATTN_ERR_INVALID_ARG;
        for (int c = a + 1; c < 4; ++c)
            if (overlap(outs[a], out_bytes[a], outs[c], out_bytes[c]))
                return FATTN_ERR_INVALID_ARG;
    }
    int dev = 0;
    DeviceInfo info;
    if ((s = current_device(&dev, &info)) != FATTN_OK)
        return s;
    for (const void *p : ins)
        if ((s = check_device_buffer(p, dev)) != FATTN_OK)
            return s;
    for (void *p : outs)
        if ((s = check_device_buffer(p, dev)) != FATTN_OK)
            return s;
    PFN_cuTensorMapEncodeTiled_v12000 encode;
    if ((s = get_encoder(&encode)) != FATTN_OK)
        return s;
    fattn::FwdMaps maps;
    fattn::BwdMaps bmaps;
    const long long BH = static_cast<long long>(B) * H;
    if ((s = make_map(encode, &maps.q, q, N, d, BH)) != FATTN_OK ||
        (s = make_map(encode, &maps.k, k, N, d, BH)) != FATTN_OK ||
        (s = make_map(encode, &maps.v, v, N, d, BH)) != FATTN_OK ||
        (s = make_map(encode, &bmaps.dout, dout, N, d, BH)) != FATTN_OK)
        return s;
    uint32_t *status = nullptr;
    cudaError_t e = fattn::status_word_address(&status);
    if (e != cudaSuccess)
        return cuda_fail(e);
    fattn::BwdArgs a{q, k, v, o, dout, lse, dq, dk, dv, static_cast<float *>(workspace), status,
                     B, H, N, d, scale, causal};
    e = fattn::launch_bwd_sm103(a, maps, bmaps, info.num_sms, stream);
    return e == cudaSuccess ? FATTN_OK : cuda_fail(e);
}

static fattn_status_t rowop(bool softmax, const void *x, void *y, int M, int N, int dtype,
                            cudaStream_t stream)
{
    if (M < 0 || N < 0 || (dtype != 0 && dtype != 1))
        return FATTN_ERR_INVALID_ARG;
    if (M == 0 || (N == 0 && softmax))
        return FATTN_OK;
    if (!y || (!x && N > 0))
        return FATTN_ERR_INVALID_ARG;
    if (N == 0) {  // row sums of empty rows are zero; x is not read
        if (reinterpret_cast<uintptr_t>(y) % 4)
            return FATTN_ERR_INVALID_ARG;
        int dev = 0;
        DeviceInfo info;
        fattn_status_t s = current_device(&dev, &info);
        if (s != FATTN_OK || (s = check_device_buffer(y, dev)) != FATTN_OK)
            return s;
        const cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(M) * 4, stream);
        return e == cudaSuccess ? FATTN_OK : cuda_fail(e);
    }
    const size_t elem = dtype == 0 ? 4 : 2;
    const size_t in_bytes = static_cast<size_t>(M) * N * elem;
    const size_t out_bytes = softmax ? in_bytes : static_cast<size_t>(M) * 4;
    if (reinterpret_cast<uintptr_t>(x) % elem || reinterpret_cast<uintptr_t>(y) % 4 ||
        (softmax && reinterpret_cast<uintptr_t>(y) % elem))
        return FATTN_ERR_INVALID_ARG;
    // The softmax may run in place (y == x) but not on partly overlapping
    // buffers; the row sums must not overlap the input.
    if ((!softmax || x != y) && overlap(x, in_bytes, y, out_bytes))
        return FATTN_ERR_INVALID_ARG;
    int dev = 0;
    DeviceInfo info;
    fattn_status_t s = current_device(&dev, &info);
    if (s != FATTN_OK)
        return s;
    if ((s = check_device_buffer(x, dev)) != FATTN_OK || (s = check_device_buffer(y, dev)) != FATTN_OK)
        return s;
    const cudaError_t e =
        softmax ? fattn::launch_softmax_rows(x, y, M, N, dtype, info.num_sms, stream)
                : fattn::launch_row_sum(x, static_cast<float *>(y), M, N, dtype, info.num_sms, stream);
    return e == cudaSuccess ? FATTN_OK : cuda_fail(e);
}

fattn_status_t fattn_softmax_rows(const void *x, void *y, int M, int N, int dtype,
                                  struct CUstream_st *stream)
{
    return rowop(true, x, y, M, N, dtype, stream);
}

fattn_status_t fattn_row_sum(const void *x, float *out, int M, int N, int dtype,
                             struct CUstream_st *stream)
{
    return rowop(false, x, out, M, N, dtype, stream);
}

fattn_status_t attn_fwd_simt(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, float scale, int causal,
                             struct CUstream_st *stream)
{
    return forward(Kernel::kSimt, q, k, v, o, lse, B, H, N, d, scale, causal, stream);
}

fattn_status_t attn_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                             void *o_host, float *lse_host, void *dq, void *dk, void *dv, void *do_,
                             float *dlse, int B, int H, int N, int d, float scale, int causal,
                             struct CUstream_st *stream)
{
    bool empty = false;
    int dev = 0;
    DeviceInfo info;
    fattn_status_t s = validate(dq, dk, dv, do_, dlse, B, H, N, N, d, scale, causal, &empty, &dev,
                                &info);
    if (s != FATTN_OK || empty)
        return s;
    if (!q_host || !k_host || !v_host || !o_host || !lse_host)
        return FATTN_ERR_INVALID_ARG;
    // Heads are independent, so the copies and the compute are pipelined
    // over chunks of consecutive (b, h) heads: copies in on one helper
    // stream, the kernel on `stream`, copies out on another, ordered by
    // events.  The helper streams first wait for the work already on
    // `stream`; the call returns after everything has completed.
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    HostPipe *hp = nullptr;
    if ((s = host_pipe(dev, &hp)) != FATTN_OK)
        return s;
    const long long BH = static_cast<long long>(B) * H;
    long long bounds[kHostChunks + 1];
    const long long q_tiles = (static_cast<long long>(N) + 127) / 128;
    const long long units = d == 256 ? q_tiles : (q_tiles + 1) / 2;  // work units per head
    const int chunks = host_chunk_plan(BH, (info.num_sms + units - 1) / units, bounds);
    const size_t head_bytes = static_cast<size_t>(N) * d * 2, head_lse = static_cast<size_t>(N) * 4;
    auto at = [](const void *base, size_t off) {
        return static_cast<const uint8_t *>(base) + off;
    };
    auto atw = [](void *base, size_t off) { return static_cast<uint8_t *>(base) + off; };
    cudaError_t e = cudaEventRecord(hp->start, stream);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(hp->in, hp->start, 0);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(hp->out, hp->start, 0);
    for (int c = 0; c < chunks && e == cudaSuccess && s == FATTN_OK; ++c) {
        const long long h0 = bounds[c], h1 = bounds[c + 1];
        const size_t off = static_cast<size_t>(h0) * head_bytes;
        const size_t bytes = static_cast<size_t>(h1 - h0) * head_bytes;
        if ((e = cudaMemcpyAsync(atw(dq, off), at(q_host, off), bytes, cudaMemcpyHostToDevice,
                                 hp->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(atw(dk, off), at(k_host, off), bytes, cudaMemcpyHostToDevice,
                                 hp->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(atw(dv, off), at(v_host, off), bytes, cudaMemcpyHostToDevice,
                                 hp->in)) != cudaSuccess ||
            (e = cudaEventRecord(hp->ev_in[c], hp->in)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(stream, hp->ev_in[c], 0)) != cudaSuccess)
            break;
        float *lse_c = reinterpret_cast<float *>(atw(dlse, static_cast<size_t>(h0) * head_lse));
        if ((s = launch(Kernel::kTcgen05, info, at(dq, off), at(dk, off), at(dv, off),
                        atw(do_, off), lse_c, 1, static_cast<int>(h1 - h0), N, N, d, scale, causal,
                        stream)) != FATTN_OK)
            break;
        if ((e = cudaEventRecord(hp->ev_done[c], stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(hp->out, hp->ev_done[c], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(atw(o_host, off), at(do_, off), bytes, cudaMemcpyDeviceToHost,
                                 hp->out)) != cudaSuccess ||
            (e = cudaMemcpyAsync(atw(lse_host, static_cast<size_t>(h0) * head_lse), lse_c,
                                 static_cast<size_t>(h1 - h0) * head_lse, cudaMemcpyDeviceToHost,
                                 hp->out)) != cudaSuccess)
            break;
    }
    // Drain all three streams whatever happened, so that no copy still
    // touches the caller's buffers after the return.
    const cudaError_t e_in = cudaStreamSynchronize(hp->in);
    const cudaError_t e_st = cudaStreamSynchronize(stream);
    const cudaError_t e_out = cudaStreamSynchronize(hp->out);
    if (s != FATTN_OK)
        return s;
    for (cudaError_t x : {e, e_in, e_st, e_out})
        if (x != cudaSuccess)
            return cuda_fail(x);
    return FATTN_OK;
}

const char *fattn_status_string(fattn_status_t status)
{
    switch (status) {
    case FATTN_OK: return "FATTN_OK";
    case FATTN_ERR_INVALID_ARG: return "FATTN_ERR_INVALID_ARG";
    case FATTN_ERR_UNSUPPORTED: return "FATTN_ERR_UNSUPPORTED";
    case FATTN_ERR_CUDA: return "FATTN_ERR_CUDA";
    case FATTN_ERR_TIMEOUT: return "FATTN_ERR_TIMEOUT";
    case FATTN_ERR_RANGE: return "FATTN_ERR_RANGE";
    }
    return "FATTN_UNKNOWN_STATUS";
}

int fattn_last_cuda_error(void) { return t_last_cuda_error; }

fattn_status_t fattn_get_device_status(int *status, struct CUstream_st *stream)
{
    if (!status)
        return FATTN_ERR_INVALID_ARG;
    uint32_t word = 0;
    const cudaError_t e = fattn::read_and_clear_status(&word, stream);
    if (e != cudaSuccess)
        return cuda_fail(e);
    *status = static_cast<int>(word);
    if (word == 0)
        return FATTN_OK;
    return (word & 0xffu) == FATTN_ERR_RANGE ? FATTN_ERR_RANGE : FATTN_ERR_TIMEOUT;
}

fattn_status_t fattn_selftest_wait_timeout(unsigned int limit_us, struct CUstream_st *stream)
{
    if (limit_us == 0 || limit_us > 2000000u)
        return FATTN_ERR_INVALID_ARG;
    int dev = 0;
    DeviceInfo info;
    fattn_status_t s = current_device(&dev, &info);
    if (s != FATTN_OK)
        return s;
    const cudaError_t e =
        fattn::launch_selftest_wait_timeout(static_cast<uint64_t>(limit_us) * 1000u, stream);
    return e == cudaSuccess ? FATTN_OK : cuda_fail(e);
}

const char *fattn_version(void) { return "libfattn 0.1.0 sm_103a"; }

}  // extern "C"
