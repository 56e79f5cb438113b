/*
 * fattn.h -- C ABI of libfattn, the GB300 (sm_103a) attention forward pass.
 *
 * The operation is the FlashAttention forward pass that the pages build up
 * to: for every head (b, h) and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j( scale * Q[b,h,i,:] . K[b,h,j,:] ) * V[b,h,j,:]
 *     lse[b,h,i] = log( sum_j exp( scale * Q[b,h,i,:] . K[b,h,j,:] ) )
 *
 * with j over all keys, or over j <= i when `causal` is set (the lower
 * triangle including the diagonal).  Sources: "OpenAI Triton: from
 * introduction to model practice", section 3 (the standard attention it
 * replaces: scores scaled by 1/sqrt(head_dim), causal masked_fill, softmax,
 * times V) and section 5 (Figure 5 and Source 2: one fused kernel that keeps
 * a running row max m_i and exp-sum l_i, rescales the accumulator, and writes
 * the output plus lse = m_i + log(l_i) in natural log); "Triton hand-written
 * kernels: vector add -> tiled GEMM -> FlashAttention core", section 4 (the
 * online softmax with m_i, l_i and acc; fp32 accumulation, 16-bit P into the
 * second product).  The N x N score matrix is never written to memory.
 *
 * Conventions shared by every call:
 *   - Tensors q, k, v, o are contiguous bf16 [B][H][N][d]: element (b,h,i,c)
 *     lives at ((b*H + h)*N + i)*d + c.  lse is contiguous fp32 [B][H][N].
 *   - Device pointers must come from the CUDA device that is current on the
 *     calling thread and be 16-byte aligned.  The caller allocates and owns
 *     every buffer; q, k, v are only read; o and lse are fully overwritten
 *     (every row 0..N-1 of every head).  o and lse must not overlap q, k, v
 *     or each other.
 *   - Supported: d in {64, 96, 128, 256} for the forward calls (attn_bwd:
 *     64 or 128; attn_fwd_simt: up to 128); B, H, N >= 0 with B*H < 2^31 and each
 *     tensor under 2^39 bytes; scale finite and > 0; causal in {0, 1}.
 *     Any N works: a ragged last tile is masked (keys past N get weight 0,
 *     rows past N are not written).
 *   - Calls are asynchronous: the work is enqueued on `stream` (NULL = the
 *     legacy default stream) and the call returns; results are valid once
 *     the stream has been synchronised.  Arguments are checked synchronously
 *     and nothing is enqueued when a check fails.  B*H*N == 0 is a no-op that
 *     returns FATTN_OK.
 *   - The caller provides every buffer of a call.  The one memory the
 *     library takes on its own is the scratch of the V pre-pass (see
 *     fattn_set_v_conversion), stream-ordered on the call's stream from a
 *     library-owned pool; attn_fwd_split_noalloc never takes it.
 *   - Calls are thread-safe; concurrent calls on different streams may run
 *     concurrently on the device.
 */
#ifndef FATTN_H
#define FATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t / CUstream */

typedef enum fattn_status {
    FATTN_OK = 0,
    FATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad scale, misalignment, overlap */
    FATTN_ERR_UNSUPPORTED = 2, /* d not supported by the call, tensor too large, device is not sm_103 */
    FATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed; see fattn_last_cuda_error() */
    FATTN_ERR_TIMEOUT = 4,     /* a kernel gave up on a pipeline wait (see fattn_get_device_status) */
    FATTN_ERR_RANGE = 5        /* a non-finite output row, e.g. from |V| >= 65520 (see attn_fwd) */
} fattn_status_t;

/*
 * attn_fwd -- the attention forward pass on device buffers.
 *
 *   q, k, v : device, bf16 [B][H][N][d], read only
 *   o       : device, bf16 [B][H][N][d], written: the normalised output
 *   lse     : device, fp32 [B][H][N], written: natural-log log-sum-exp of
 *             the scaled (and masked) scores of each row
 *   B, H, N : batch, heads, sequence length (queries and keys alike)
 *   d       : head dimension, 64, 96, 128 or 256
 *   scale   : multiplies Q.K before masking and softmax (usually 1/sqrt(d))
 *   causal  : 1 keeps keys j <= i for query i, 0 keeps all keys
 *   stream  : CUDA stream the kernel is enqueued on
 *
 * Precision.  Scores, row max, row sums and the output accumulator are fp32.
 * P, the probabilities that enter the second product, is rounded to fp16 (not
 * to bf16, the inputs' type): with bf16 P the bf16 output misses the stated
 * 1e-2 bound on peaked rows whose |O| is in [2, 4), where one bf16 ulp is
 * 0.0156 and P's rounding moves O across a rounding midpoint.  Both operands
 * of a tensor-core product share one type, so V is rounded to fp16 (on
 * chip, or by a pre-pass: see fattn_set_v_conversion; the bits are the
 * same).  That is exact for |v| < 65520; a V element of larger
 * magnitude becomes infinite in the product.  Any output row that comes out
 * non-finite -- from such a V element, or from non-finite inputs -- makes
 * the kernel record FATTN_ERR_RANGE in the device status word (those rows
 * of o are then not meaningful).  For V beyond that range use
 * attn_fwd_strided with dtype 2 (P in bf16).  O is divided by the fp32 row
 * sum and rounded to bf16 (nearest even).
 *
 * Returns FATTN_OK once the kernel is enqueued, or an error status without
 * enqueuing anything.  A pipeline timeout inside the kernel is not reported
 * here (the call has already returned); it leaves o/lse undefined and sets the
 * device status word read by fattn_get_device_status().
 */
fattn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                        int B, int H, int N, int d, float scale, int causal,
                        struct CUstream_st *stream);

/*
 * attn_fwd_fp16 -- attn_fwd for fp16 q, k, v and o (lse stays fp32): the
 * element type of the page-1 kernel of "Triton hand-written kernels: vector
 * add -> tiled GEMM -> FlashAttention core" (section 4, fp16 inputs and P
 * cast to fp16 before the second product).  P is rounded to fp16 and O is
 * normalised by the fp32 row sum.  Same arguments, rules and errors as
 * attn_fwd.
 */
fattn_status_t attn_fwd_fp16(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, float scale, int causal,
                             struct CUstream_st *stream);

/*
 * attn_fwd_host -- the same operation on HOST buffers, end to end.
 *
 * Copies q_host, k_host, v_host to the caller's device buffers dq, dk, dv,
 * runs attn_fwd into do_ / dlse, and copies the results back to o_host and
 * lse_host; it returns once everything has completed.  The work is
 * pipelined over up to eleven chunks of consecutive (b, h) heads (short ones
 * first and last, so that the parts nothing overlaps are short): the copies
 * in run on a library-owned helper stream, the kernels on `stream`, the
 * copies out on a second helper stream, ordered by events, so copies and
 * compute overlap.  The helper streams first wait for the work already
 * enqueued on `stream`.  Calls are serialised inside the library.  Host
 * buffers should be page-locked (cudaHostAlloc / pinned) for asynchronous
 * full-bandwidth copies; pageable memory works but is slower.  Device
 * buffers follow attn_fwd's rules.  The helper streams and events are
 * created once per device; the V pre-pass scratch is as for attn_fwd.  The return value
 * includes any error raised while the streams drained.
 */
fattn_status_t attn_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                             void *o_host, float *lse_host,
                             void *dq, void *dk, void *dv, void *do_, float *dlse,
                             int B, int H, int N, int d, float scale, int causal,
                             struct CUstream_st *stream);

/*
 * V conversion.  The pages cast P to a 16-bit type before the second product
 * ("Triton hand-written kernels: vector add -> tiled GEMM -> FlashAttention
 * core", section 4); this library takes fp16 for it with bf16 inputs (see
 * attn_fwd), and both operands of a tensor-core product share one type, so
 * for bf16 inputs with P in fp16 (attn_fwd, attn_fwd_split, attn_fwd_kv,
 * attn_fwd_strided with dtype 0, attn_fwd_host) every V element is rounded
 * to fp16 for the P V product, in one of two places:
 *   - on chip: converter warps of the forward kernel round each V tile in
 *     shared memory, once for every work unit that reads it; no memory is
 *     taken;
 *   - by a pre-pass: one more kernel rounds all of V once into device scratch
 *     of B*H*Nk*d*2 bytes (Nk: keys per head), which the forward kernel then
 *     reads instead of v.  The scratch is taken on `stream` from a
 *     library-owned stream-ordered memory pool of the current device and
 *     given back on `stream` after the forward kernel; the pool keeps what is
 *     given back for later calls until fattn_trim_scratch.
 * Both round with the same function, so the outputs are bit for bit the
 * same.  fattn_set_v_conversion chooses for the whole process:
 *   FATTN_V_CONVERT_AUTO (the default): the pre-pass where each V tile
 *     would otherwise be rounded for many work units.  With T = ceil(N/128)
 *     query tiles per head, units U = T for d = 256 and ceil(T/2) otherwise,
 *     and visits = U/2 with the causal mask, U without: the pre-pass from 24
 *     visits at d = 64, 8 at d = 96, 16 at d = 128 and 12 at d = 256 (where
 *     it was measured to be faster on a GB300), on chip below;
 *   FATTN_V_CONVERT_ON_CHIP: never the pre-pass, so no call takes memory;
 *   FATTN_V_CONVERT_PREPASS: the pre-pass for every shape.
 * Whatever the setting, a call converts on chip when `stream` is being
 * captured into a CUDA graph or the scratch cannot be had (out of memory),
 * and attn_fwd_split_noalloc always does.  Each call reads the setting once.
 * Returns the previous setting, or -1 (nothing changed) for an unknown mode.
 *
 * fattn_v_conversion_route: where a call with N queries per head, head
 * dimension d and mask `causal` rounds V under the current setting (scratch
 * permitting): FATTN_V_CONVERT_ON_CHIP or FATTN_V_CONVERT_PREPASS; -1 for an
 * unsupported d, N < 0 or causal not 0 or 1.
 *
 * fattn_trim_scratch gives the pool's unused memory on every device back to
 * the system (memory of calls still in flight stays).  FATTN_OK, or
 * FATTN_ERR_CUDA.  Like all per-device state, the pools do not survive
 * cudaDeviceReset.
 */
#define FATTN_V_CONVERT_AUTO 0
#define FATTN_V_CONVERT_ON_CHIP 1
#define FATTN_V_CONVERT_PREPASS 2
int fattn_set_v_conversion(int mode);
int fattn_v_conversion_route(int N, int d, int causal);
fattn_status_t fattn_trim_scratch(void);

/*
 * Key-range split (split-KV).  When B*H*ceil(N/256) work units are fewer
 * than the device's SMs (few heads, or one long sequence), attn_fwd leaves
 * most SMs idle.  attn_fwd_split divides the keys of every pair of 128-row
 * query tiles into num_splits contiguous ranges processed by different CTAs,
 * each producing a partial output and partial log-sum-exp, and a second
 * kernel merges them exactly: lse = log(sum_s exp(lse_s)) and
 * O = sum_s exp(lse_s - lse) O_s -- the blocked softmax statistics merge
 * ("OpenAI Triton: from introduction to model practice", section 1.1,
 * example 3: per-block max and sum combined into the global max and sum).
 *
 * attn_fwd_split_count: the number of splits the library would use on the
 *   current device for this shape (1 = no split helps), or 0 on invalid
 *   arguments / no usable device.
 * attn_fwd_split_workspace_size: bytes of device scratch attn_fwd_split
 *   needs for num_splits (0 when num_splits == 1 or on invalid arguments):
 *   num_splits * B*H*N * (4*d + 8) bytes plus alignment.
 * attn_fwd_split: attn_fwd's arguments and contract, plus num_splits
 *   (1..64; 1 is exactly attn_fwd and ignores the workspace) and the
 *   caller-owned device workspace (16-byte aligned, at least the size above,
 *   not overlapping q, k, v, o, lse; its contents on entry are ignored and on
 *   exit are undefined).  Two kernels are enqueued on `stream`; calls that
 *   share one workspace must not overlap on the device.
 */
int attn_fwd_split_count(int B, int H, int N, int d, int causal);
size_t attn_fwd_split_workspace_size(int B, int H, int N, int d, int num_splits);
fattn_status_t attn_fwd_split(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int H, int N, int d, float scale, int causal, int num_splits,
                              void *workspace, size_t workspace_bytes,
                              struct CUstream_st *stream);

/*
 * attn_fwd_split_noalloc -- attn_fwd_split for callers that cannot allocate
 * device memory at the point of the call: for example a serving runtime that
 * plans all of its device memory before it starts and forbids allocation on
 * its execution path, or a plugin whose host framework owns every device
 * allocation.  The pages have no counterpart of this call; it exists only for
 * such callers.
 *
 * Same arguments and result as attn_fwd_split without the workspace: the
 * scratch is a fixed 32 MiB array of device memory inside the library
 * (every GPU that loads the library holds it until the process exits).  The
 * call allocates nothing.  Its first call on each device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture.  A shape whose scratch
 * (attn_fwd_split_workspace_size) exceeds 32 MiB returns
 * FATTN_ERR_UNSUPPORTED without enqueuing anything: use attn_fwd_split with
 * your own workspace then.  num_splits == 1 is exactly attn_fwd.  The array
 * keeps the previous call's contents; nothing in it needs to start at zero,
 * because every value the merge reads is written earlier by the same call.
 * All calls in the process share the one array per device, so calls that
 * overlap on the GPU (e.g. on two streams at once) race and corrupt each
 * other's results: serialise them.
 */
fattn_status_t attn_fwd_split_noalloc(const void *q, const void *k, const void *v, void *o,
                                      float *lse, int B, int H, int N, int d, float scale,
                                      int causal, int num_splits, struct CUstream_st *stream);

/*
 * attn_fwd_kv -- queries and keys of different lengths: the decode step of
 * autoregressive generation, where a few new query rows attend to a long,
 * growing cache of keys and values and every step reads the whole cache
 * ("OpenAI Triton: from introduction to model practice", section 4, the note
 * on why attention is the bottleneck: 1 x seq_len scores per generated token,
 * bound by memory bandwidth).
 *
 *   q     : bf16 [B][H][Nq][d]      k, v : bf16 [B][H][Nk][d]
 *   o     : bf16 [B][H][Nq][d]      lse  : fp32 [B][H][Nq]
 * All contiguous, device memory, 16-byte aligned; d in {64, 96, 128, 256}.
 * Without the mask every query sees all Nk keys.  With causal = 1 the Nq
 * queries are the LAST Nq positions of the key sequence: query i sees keys
 * j <= i + (Nk - Nq), so Nq <= Nk is required; Nq == Nk is attn_fwd's causal
 * mask.  Nk >= 1 whenever B*H*Nq > 0; B*H*Nq == 0 enqueues nothing.
 *
 * num_splits: 0 = the library's schedule for the current device; 1..64 =
 * that many equal key ranges per pair of 128-row query tiles, as
 * attn_fwd_split (1: one kernel, the workspace is ignored and may be NULL).
 * The automatic schedule, for Nq <= 256 (one pair of query tiles per head)
 * when whole heads per SM would leave SMs idle, deals the B*H*(key tiles)
 * steps evenly over the SMs in contiguous head-major ranges (a head may be
 * shared by several SMs, each producing a partial result) and merges the
 * partials as attn_fwd_split does; otherwise it is attn_fwd_split_count's
 * choice.  The workspace rules are attn_fwd_split's;
 * attn_fwd_kv_workspace_size gives the bytes for the same (B, H, Nq, Nk, d,
 * causal, num_splits) on the current device (0 when none is needed or on
 * invalid arguments).  Errors: FATTN_ERR_INVALID_ARG for bad
 * shapes, pointers, Nq > Nk under the mask, Nk == 0 with queries, or a
 * workspace that is missing, too small, misaligned or overlapping;
 * FATTN_ERR_UNSUPPORTED for other d or tensors beyond 2^39 bytes; nothing is
 * enqueued on an error.
 */
size_t attn_fwd_kv_workspace_size(int B, int H, int Nq, int Nk, int d, int causal,
                                  int num_splits);

/*
 * attn_fwd_strided -- attn_fwd_kv on tensors with arbitrary strides: the
 * kernel takes the layout's strides explicitly instead of assuming a
 * contiguous one ("Triton programming template", the Python wrapper section;
 * "CS336 lecture 6: kernels and Triton", the matmul + ReLU example's note on
 * strided pointers for non-contiguous layouts).  E.g. q, k, v as views of one
 * packed [B][N][3][H][d] projection output, or o written into a [B][N][H][d]
 * buffer.
 *
 *   x_strides[3] : element strides of (batch, head, row) for x in q, k, v, o;
 *                  the last dimension (d) is contiguous (stride 1).
 * Element (b, h, i, c) of x lives at x + b*s[0] + h*s[1] + i*s[2] + c.
 * Every stride must be a positive multiple of 8 elements (16 bytes) and at
 * most 2^38; the stride of a dimension of extent 1 is ignored.  q, k, v may
 * overlap each other (all are only read); o's elements must be distinct
 * (checked by nesting: its strides sorted by size, each at least the span
 * of the smaller dimensions) and o must not overlap q, k, v or lse (checked
 * over each tensor's address span).  lse stays contiguous fp32 [B][H][Nq].
 * dtype: 0 = bf16 q, k, v, o (P in fp16, as attn_fwd); 1 = fp16 (as
 * attn_fwd_fp16: P rounded to fp16, O normalised by the fp32 sum); 2 = bf16
 * with P rounded to bf16, for V of any bf16 magnitude (O normalised by the row
 * sum of the rounded P, so the rounding of each tile's largest p cancels; its
 * bf16 output can miss the 1e-2 bound by up to one ulp where |O| >= 2);
 * anything else gives FATTN_ERR_INVALID_ARG.
 * Everything else -- shapes, the causal alignment, num_splits, the workspace
 * (attn_fwd_kv_workspace_size) and the errors -- is attn_fwd_kv's.  A
 * stride array that is NULL gives FATTN_ERR_INVALID_ARG.
 */
fattn_status_t attn_fwd_strided(const void *q, const void *k, const void *v, void *o,
                                float *lse, int B, int H, int Nq, int Nk, int d,
                                const long long *q_strides, const long long *k_strides,
                                const long long *v_strides, const long long *o_strides,
                                float scale, int causal, int num_splits, void *workspace,
                                size_t workspace_bytes, int dtype, struct CUstream_st *stream);
fattn_status_t attn_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int H, int Nq, int Nk, int d, float scale, int causal,
                           int num_splits, void *workspace, size_t workspace_bytes,
                           struct CUstream_st *stream);

/*
 * attn_fwd_simt -- the same operation and contract as attn_fwd, computed by a
 * plain fp32 SIMT kernel (no tensor cores, no 16-bit rounding of P).  It is
 * an independent second GPU implementation for cross-checking results at
 * sizes where the CPU reference is too slow; it is far slower than attn_fwd.
 */
fattn_status_t attn_fwd_simt(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, float scale, int causal,
                             struct CUstream_st *stream);

/*
 * attn_bwd -- gradients of attn_fwd: dq, dk, dv (bf16 [B][H][N][d]) for the
 * upstream gradient dout (bf16 [B][H][N][d]), from the forward's inputs and
 * its saved outputs o (bf16) and lse (fp32 [B][H][N]), as the autograd
 * wrapper of "OpenAI Triton: from introduction to model practice", section
 * 6, saves and passes them.  The scores are recomputed from q, k and lse:
 *   P = exp(scale Q K^T - lse) (masked entries 0),  D_i = dO_i . O_i,
 *   dV = P^T dO,  dS = P * (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q.
 * P and dS are rounded to bf16 for the products that use them; accumulation
 * is fp32.  Same B, H, N, d, scale, causal rules as attn_fwd.  workspace is
 * caller-owned device scratch of at least attn_bwd_workspace_size(...) bytes
 * (B*H*N*4; contents ignored on entry, undefined on exit), 16-byte aligned.
 * dq, dk, dv and the workspace must not overlap each other or any input.
 * Three kernels are enqueued on `stream`.  Errors as for attn_fwd.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d);
fattn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                        int H, int N, int d, float scale, int causal, void *workspace,
                        size_t workspace_bytes, struct CUstream_st *stream);

/*
 * Standalone row softmax and row sum (HBM-bound), after the row softmax and
 * row-sum examples of "CS336 lecture 6: kernels and Triton":
 *   fattn_softmax_rows: y[i][j] = exp(x[i][j] - max_k x[i][k]) / sum_k exp(x[i][k] - max_k x[i][k])
 *   fattn_row_sum:      out[i]  = sum_j x[i][j]
 * x is a contiguous row-major [M][N] device matrix of dtype 0 = fp32 or
 * 1 = bf16 (arithmetic in fp32); the softmax writes y with x's shape and type
 * (y may equal x for an in-place softmax, but must not otherwise overlap it);
 * the row sums go to fp32 out[M].  Pointers must be device pointers aligned
 * to their element size.  Rows of up to 16384 elements are read from HBM
 * once; longer rows twice (an online max/sum pass, then the output pass).
 * Empty inputs are no-ops (an empty row sums to 0).  Asynchronous on
 * `stream`; errors as for attn_fwd.
 */
fattn_status_t fattn_softmax_rows(const void *x, void *y, int M, int N, int dtype,
                                  struct CUstream_st *stream);
fattn_status_t fattn_row_sum(const void *x, float *out, int M, int N, int dtype,
                             struct CUstream_st *stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *fattn_status_string(fattn_status_t status);

/* The CUDA error code (cudaError_t value) behind the calling thread's most
 * recent FATTN_ERR_CUDA, or 0. */
int fattn_last_cuda_error(void);

/*
 * fattn_get_device_status -- read and clear the device status word of the
 * current device, after synchronising `stream`.
 *
 * *status receives 0 when no kernel reported a problem since the last read,
 * otherwise the first code recorded: bits 0..7 = FATTN_ERR_TIMEOUT or
 * FATTN_ERR_RANGE, bits 8..15 = the role that reported it (1 load, 2 mma,
 * 3 softmax, 4 epilogue, 5 self-test, 6 V conversion), bits 16..31 = the CTA
 * index.  Returns the status in bits 0..7 (FATTN_ERR_TIMEOUT or
 * FATTN_ERR_RANGE) if *status is nonzero, FATTN_OK if it is zero, or
 * FATTN_ERR_INVALID_ARG / FATTN_ERR_CUDA.
 *
 * The library keeps per-device state for the life of the process (the
 * helper streams of attn_fwd_host, the scratch address of
 * attn_fwd_split_noalloc); it is not valid after cudaDeviceReset.
 */
fattn_status_t fattn_get_device_status(int *status, struct CUstream_st *stream);

/*
 * fattn_selftest_wait_timeout -- exercise the failure path without a fault.
 *
 * Enqueues on `stream` a one-warp kernel that waits, with the same bounded
 * wait the forward kernel's pipeline roles use, on a barrier that nothing
 * ever signals.  After `limit_us` microseconds (1 .. 2,000,000) the wait gives
 * up, the kernel records FATTN_ERR_TIMEOUT with role 5 in the device status
 * word (see fattn_get_device_status) and returns; the CUDA context stays
 * usable.  Returns FATTN_OK once enqueued, FATTN_ERR_INVALID_ARG for a limit
 * out of range, FATTN_ERR_UNSUPPORTED / FATTN_ERR_CUDA for device problems.
 */
fattn_status_t fattn_selftest_wait_timeout(unsigned int limit_us, struct CUstream_st *stream);

/* Library version string, e.g. "libfattn 0.1.0 sm_103a". */
const char *fattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H */
