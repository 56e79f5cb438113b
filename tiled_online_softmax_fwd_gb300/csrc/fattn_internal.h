// fattn_internal.h -- declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fattn {

// Arguments of one forward call, already validated by the C-ABI layer.
struct FwdArgs {
    const void *q;
    const void *k;
    const void *v;
    void *o;
    float *lse;
    int B, H, N, d;
    float scale;
    int causal;
    int f16 = 0;    // 1: fp16 q, k, v, o (P in fp16); 0: bf16
    int bf16p = 0;  // bf16 only: 0 = P in fp16 (V converted to fp16 on chip),
                    // 1 = P in bf16 (V of any bf16 magnitude)
    int Nk = 0;   // keys per head (N: queries per head); the queries are the
                  // last N key positions under the causal mask
    // Element strides of o for (batch, head, row); all 0 = contiguous.
    long long o_sb = 0, o_sh = 0, o_sn = 0;
    // bf16 with fp16 P only: non-null = V pre-pass.  The caller's V (v,
    // element strides v_sb, v_sh, v_sn, each a multiple of 8) is rounded to
    // fp16 into v16, contiguous [B][H][Nk][d], which FwdMaps::v then reads.
    void *v16 = nullptr;
    long long v_sb = 0, v_sh = 0, v_sn = 0;
};

// Tensor maps over Q, K, V.  The forward kernel takes 4-D maps (d, N or Nk,
// H, B) with the tensors' own row, head and batch strides, box (64, 128, 1,
// 1); the backward takes 3-D maps (d, N, B*H) of contiguous tensors, box
// (64, 128, 1).  128-byte swizzle, zero fill outside the sequence.
struct FwdMaps {
    CUtensorMap q, k, v;
};

// Key-range split of the forward pass: splits > 1 sends fp32 partial O
// ([splits][B*H*N][d]) and base-2 partial lse pairs ([splits][B*H*N] x 2
// floats) to caller-provided scratch, then a combine kernel writes o / lse.
struct FwdSplit {
    int splits;  // stream-K: partial slots per head
    float *ws_o;
    float *ws_l;
    int streamk = 0;  // 1: stream-K schedule (one Q-tile pair per head)
};

// Stream-K plan for N queries against Nk keys per head: when every head has
// one pair of 128-row Q tiles (N <= 256) and whole heads per CTA would leave
// SMs idle, the (head, key tile) steps are dealt evenly over the SMs and the
// partial results merged; slots bounds the partials of one head.  streamk 0:
// no stream-K plan for this shape.
struct FwdPlan {
    int streamk;
    int slots;
};
FwdPlan plan_fwd_streamk(int B, int H, int N, int Nk, int causal, int num_sms);

// Device status word codes (see fattn_get_device_status in fattn.h).
enum DeviceRole : uint32_t {
    kRoleLoad = 1,
    kRoleMma = 2,
    kRoleSoftmax = 3,
    kRoleEpilogue = 4,
    kRoleSelfTest = 5,
    kRoleConvert = 6
};

// tcgen05 / TMA kernel: one persistent CTA per SM.
cudaError_t launch_fwd_sm103(const FwdArgs &a, const FwdMaps &maps, const FwdSplit &split,
                             int num_sms, cudaStream_t stream);
// Failure-path self-test: a wait that nothing satisfies, limited to limit_ns.
cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);
// Reads (and clears) the device status word of the current device.
cudaError_t read_and_clear_status(uint32_t *out, cudaStream_t stream);

// Plain SIMT kernel (fp32 CUDA cores): a second, independent GPU path used by
// the tests as a cross-check.  Not used by attn_fwd.
cudaError_t launch_fwd_simt(const FwdArgs &a, cudaStream_t stream);

// Backward pass (dQ, dK, dV) of the forward above.  dvec is scratch for
// D = rowsum(dO * O) (fp32, B*H*N); status is the device status word.
struct BwdArgs {
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    float *dvec;
    uint32_t *status;
    int B, H, N, d;
    float scale;
    int causal;
};
struct BwdMaps {
    CUtensorMap dout;  // same geometry as FwdMaps
};
cudaError_t launch_bwd_sm103(const BwdArgs &a, const FwdMaps &m, const BwdMaps &mb, int num_sms,
                             cudaStream_t stream);
// Device address of the status word on the current device.
cudaError_t status_word_address(uint32_t **out);

// Row softmax / row sum over a contiguous [M][N] matrix of fp32 (dtype 0) or
// bf16 (dtype 1); the softmax output has the input's type, the sums are fp32.
cudaError_t launch_softmax_rows(const void *x, void *y, int M, int N, int dtype, int num_sms,
                                cudaStream_t stream);
cudaError_t launch_row_sum(const void *x, float *out, int M, int N, int dtype, int num_sms,
                           cudaStream_t stream);

}  // namespace fattn
