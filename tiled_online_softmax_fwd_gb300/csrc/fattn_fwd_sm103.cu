// fattn_fwd_sm103.cu -- attention forward pass for GB300 (sm_103a).
//
// The method is the FlashAttention forward pass with an online softmax
// ("Triton hand-written kernels: vector add -> tiled GEMM -> FlashAttention
// core", section 4; "OpenAI Triton: from introduction to model practice",
// section 5, Figure 5 and Source 2): for each tile of query rows, stream the
// key/value tiles, form S = scale * Q K^T, keep a running row max m and
// exp-sum l, rescale the accumulator when m grows, add P V, and at the end
// write O = acc / l and lse = m + ln l.  Scores never leave the chip.
//
// GB300 design (one persistent CTA per SM, 320 threads):
//   warp 8      TMA producer: Q tiles and a ring of K/V tiles in 128-byte
//               swizzled shared memory, completion tracked by mbarriers.
//   warp 9      MMA issuer: S = Q K^T and O += P V as tcgen05 MMAs (bf16 in,
//               fp32 accumulate) into tensor memory (TMEM); the warp runs
//               converged and one elected lane issues.
//   warps 0-7   two softmax warpgroups, one per 128-row Q tile; they
//               alternate (ping-pong) so that one computes exponentials
//               while the tensor core works on the other tile.  Each thread
//               owns one query row: it reads its S row from TMEM, applies
//               the causal / tail mask, updates m and l, writes P (16-bit)
//               back into TMEM over its S row, rescales its O row in TMEM
//               when needed, and finally normalises and stores O and lse.
//   warps 10-11 (bf16 inputs) V converters: each V tile is rewritten in
//               place from bf16 to fp16 before the P V product reads it.
// A work unit is two consecutive 128-row Q tiles of one (batch, head).  The
// units are ordered heaviest first (for the causal mask the work of a Q tile
// grows with its index) and dealt to the CTAs in a serpentine order so that
// no SM is left with a long tail ("wave quantisation").  Under the causal
// mask, key tiles entirely above the diagonal are skipped and only the
// diagonal tile is masked element-wise.
//
// Tensor memory (512 columns x 128 lanes, fp32 words):
//   [0,128)   S of tile 0 (P of tile 0 overwrites its first 64 columns)
//   [128,256) S of tile 1 (likewise)
//   [256,256+D)      O accumulator of tile 0
//   [256+D,256+2D)   O accumulator of tile 1
//
// Softmax details.  Scores are handled in the base-2 domain: x = s * scale *
// log2(e), p = 2^(x - m).  The running max m is only raised when a new row
// maximum exceeds it by more than kRescaleLog2 (so O and l need rescaling
// rarely); until then p may exceed 1 by at most 2^kRescaleLog2.  This is
// exact algebra: O and l always refer to the same m, so O / l and
// lse = ln2 * (m + log2 l) are unchanged.
//
// Precision of P (kPrec).  P is rounded to fp16 for bf16 and for fp16
// inputs, and O is normalised by l, the fp32 sum of the unrounded p: with
// P in bf16 the bf16 output of peaked rows misses a 1e-2 bound where |O| is
// in [2, 4), since P's own rounding moves O across a rounding midpoint.  For
// bf16 inputs V is converted to fp16 on chip (run_convert).  The bf16-P mode
// (kPrecBf16P, for V beyond the fp16 range) keeps a second sum, l_round,
// which normalises O and stands for the sum of the bf16-rounded
// probabilities that enter P V, so that the rounding of a dominant p cancels
// in O / l_round.  With d = 64 it is that sum exactly, formed by the tensor
// cores: V is extended by a constant column of ones (its own 16 KB swizzle
// atom after the K/V ring), so column d of the O accumulator is the row sum
// of the rounded P, summed in fp32 and rescaled together with O (see
// Cfg::kOnes).  Otherwise l_round is l minus the rounding error of the
// largest p of each key tile, which costs one exponential per tile instead
// of a second sum over all 128 keys.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <float.h>
#include <stdint.h>

#include "fattn_internal.h"
#include "ptx_sm103.cuh"

namespace fattn {

// Device status word: 0, or the first timeout code recorded by any CTA.
__device__ uint32_t g_fattn_status;

namespace {

using namespace ptx;

constexpr int kBM = 128;  // query rows per Q tile (= MMA M = TMEM lanes)
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kWarpConv = 10;  // and 11 (kPrecBf16)
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kChunkBytes = kBM * 64 * 2;  // one 128-row x 64-column bf16 box

// Precision modes.  Inputs and output are bf16 or fp16; P, the 16-bit
// probabilities that enter the P V product, is fp16 or bf16.  Both operands
// of one tensor-core product have one type, so for bf16 inputs with fp16 P
// the V tiles are converted to fp16 in shared memory (exactly, for |v| below
// 65520) by two converter warps before the P V product reads them.
constexpr int kPrecBf16 = 0;    // bf16 q, k, v, o; P in fp16 (V converted)
constexpr int kPrecF16 = 1;     // fp16 q, k, v, o; P in fp16
constexpr int kPrecBf16P = 2;   // bf16 q, k, v, o; P in bf16 (V of any bf16 magnitude)
constexpr int kPrecBf16V16 = 3; // bf16 q, k, o; V rounded to fp16 beforehand; P in fp16

template <int D, int kPrec = kPrecBf16>
struct Cfg {
    static constexpr bool kInF16 = kPrec == kPrecF16;    // q, k, v, o in fp16
    static constexpr bool kPF16 = kPrec != kPrecBf16P;   // P (and V in P V) in fp16
    static constexpr bool kConv = kPrec == kPrecBf16;    // converter warps
    // V rounded from bf16 to fp16 (on chip or by v_to_f16_kernel): an
    // infinity from |v| >= 65520 is reported by the epilogue.
    static constexpr bool kVRounded = kConv || kPrec == kPrecBf16V16;
    // Threads: the two-tile kernel has 8 softmax warps, a TMA warp and an
    // MMA warp; the one-tile kernel 4, 1 and 1; both add 2 converter warps.
    static constexpr int kThreads = (D == 256 ? 192 : 320) + (kConv ? 64 : 0);
    // 128-byte swizzle atoms along d.  d = 96 takes two: the tensor map's
    // 64-column box reads columns 96..127 as zeros, which no MMA uses (the
    // S product stops at K = 96, the P V product has N = 96).
    static constexpr int kChunks = (D + 63) / 64;
    static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;
    // d = 256 runs one Q tile per CTA (fwd_single_kernel): a 64 KB Q tile and
    // two 64 KB K/V stages.  Otherwise two Q tiles and a deeper ring.
    static constexpr int kQTiles = D == 256 ? 1 : 2;
    static constexpr int kStages = kChunks == 4 ? 2 : (kChunks == 2 ? 4 : 8);  // K/V ring
    // The one-tile kernel fills and frees each 64 KB stage in two 32 KB
    // halves with barriers of their own (K: d-columns 0-127 and 128-255, the
    // S product's K-steps 0-7 and 8-15; V: keys 0-63 and 64-127, the P V
    // product's K-steps 0-3 and 4-7), so the next copy into a half starts
    // once the products reading that half are done, half a product earlier.
    static constexpr int kHalves = kQTiles == 1 ? 2 : 1;
    static constexpr uint32_t kHalfBytes = kTileBytes / kHalves;
    // Ones column: P V runs with N = D + 16 against V extended by a constant
    // atom whose first column is 1.0, so O column D accumulates l_round.
    // Needs 2 * (128 + D + 16) <= 512 TMEM columns; used for bf16 P, d = 64.
    static constexpr bool kOnes = !kPF16 && D == 64;
    static constexpr uint32_t kOnesOffset = (kQTiles + kStages) * kTileBytes;
    static constexpr uint32_t kTilesBytes = kOnesOffset + (kOnes ? kChunkBytes : 0);
    // Epilogue staging: 4 KB (32 rows x 128 bytes) for each softmax warp (4 in
    // the one-tile kernel, 8 in the two-tile one).
    static constexpr uint32_t kStageOffset = kTilesBytes;
    static constexpr uint32_t kBarsOffset = kStageOffset + (kQTiles == 1 ? 4 : 8) * 4096;
    static constexpr uint32_t kON = D + (kOnes ? 16 : 0);  // O accumulator columns
    // P V in two halves (keys 0-63 as soon as their P is written), so only
    // the second half's product lies between the last P and the next S:
    // faster at d = 64, where the softmax dominates (1101 -> 1148 TFLOP/s on
    // B2 H8 N65536), and at d = 128 since the row maximum comes from the
    // reducing TMEM load (B4 H16 N4096 d128 causal 1277-1282 -> 1324-1334,
    // B8 H16 N2048 d128 causal 1010-1017 -> 1047-1061, the headline level or
    // up to 1 %; with the software max it had been slower there, 1441 ->
    // 1389).  At d = 96 it pays only with converter warps (B8 H16 N2048 d96
    // causal 782-789 -> 809-820, its register spills gone) and cost 0.3-0.8 %
    // with V rounded beforehand.
    static constexpr bool kHalfP = D == 64 || D == 128 || (D == 96 && kConv);
    static constexpr uint32_t kColO0 = 256;
    static constexpr uint32_t kColO1 = 256 + kON;
};

struct Bars {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[8], kv_empty[8];
    uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
    uint64_t p_half[2];  // two-tile kernel: P of the first 64 keys written
    uint64_t drain;
    uint64_t pv_done;  // single-tile kernel: completion of each P V
    uint64_t v_ready[8];  // converter warps: the V tile in this stage is fp16
    uint64_t v_full[8];   // single-tile kernel: a V copy landed (K copies use kv_full)
    uint32_t tmem_base;
    int abort;
    // Stream-K range of this CTA (see cta_unit): first head, its first key
    // tile and partial slot, and the end of the range.
    int sk_h0, sk_j0, sk_slot0;
    long long sk_hi;
};

struct Params {
    void *o;       // bf16 or fp16, element (b, h, i, c) at b*o_sb + h*o_sh + i*o_sn + c
    float *lse;
    float *ws_o;   // split mode: fp32 partial O [splits][B*H*Nq][D]
    float2 *ws_l;  // split mode: base-2 partial lse (of l, of l_round) [splits][B*H*Nq]
    int Nq;        // query rows per head
    int Nk;        // keys per head
    int off;       // Nk - Nq: query i sits at key position i + off (causal mask)
    int extra;     // ceil(off / 128): key tiles past the diagonal (causal mask)
    int BH;        // batch * heads
    int H;         // heads
    long long o_sb, o_sh, o_sn;  // element strides of o (batch, head, row)
    int QT;        // query tiles per head = ceil(Nq / 128)
    int KT;        // key tiles per head = ceil(Nk / 128)
    int pairs;     // Q-tile pairs per head = ceil(QT / 2)
    int splits;    // key-range splits per pair (1: no split, results go to o / lse);
                   // stream-K: partial slots per head
    int units;     // BH * pairs * splits
    int causal;
    int single;    // 1: a work unit has one Q tile (d = 256), "pairs" counts Q tiles
    int streamk;   // 1: one Q-tile pair per head, key tiles dealt evenly over CTAs
    int grid;      // CTAs of the launch (stream-K ranges)
    int F;         // key tiles of the pair (stream-K)
    long long W;   // BH * F: stream-K work in key tiles
    float sl2;     // scale * log2(e)
};

// A work unit: Q tiles qt[0], qt[1] of head bh, over key tiles [j0, j1[t]).
struct Unit {
    int bh;
    int split;
    int qt[2];
    int j0;
    int j1[2];  // j1[t] <= j0: tile t has no work in this unit
    int n[2];   // key tiles of tile t: j1[t] - j0 (or 0)
    int n_max;
};

// Key tiles visited by Q tile qt over the whole key range (0 past the end):
// under the causal mask, up to the tile holding the last visible key of the
// tile's last row, min(128 qt + 127, Nq - 1) + off.  For every tile but the
// last that is tile qt + ceil(off / 128); for the last one it is the last
// key tile, which the min with KT gives.
__host__ __device__ __forceinline__ int key_tiles(int QT, int KT, int extra, int causal, int qt)
{
    if (qt >= QT)
        return 0;
    return causal ? min(qt + 1 + extra, KT) : KT;
}
__device__ __forceinline__ int key_tiles(const Params &p, int qt)
{
    return key_tiles(p.QT, p.KT, p.extra, p.causal, qt);
}

// Q tile t of a unit (pair index, or Q tile index in single-tile mode, where
// the second tile is absent: index QT has no key tiles).
__device__ __forceinline__ int unit_tile(const Params &p, int pair, int t)
{
    return p.single ? (t == 0 ? pair : p.QT) : 2 * pair + t;
}

// Key tiles of a unit: the max over its Q tiles.
__device__ __forceinline__ int unit_tiles(const Params &p, int pair)
{
    return max(key_tiles(p, unit_tile(p, pair, 0)), key_tiles(p, unit_tile(p, pair, 1)));
}

// Tile t of the pair works on key tiles [j0, min(je, its own count)).
__device__ __forceinline__ Unit make_unit(const Params &p, int bh, int split, int pair, int j0,
                                          int je)
{
    Unit u;
    u.bh = bh;
    u.split = split;
    u.j0 = j0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        u.qt[t] = unit_tile(p, pair, t);
        u.j1[t] = min(je, key_tiles(p, u.qt[t]));
        u.n[t] = max(u.j1[t] - u.j0, 0);
    }
    u.n_max = max(u.n[0], u.n[1]);
    return u;
}

// The split s of a pair covers key tiles [s*F/S, (s+1)*F/S) of the pair's
// F = max over its two tiles; the combine kernel uses the same ranges.
__device__ __forceinline__ Unit unit_at(const Params &p, int k)
{
    const int split = k % p.splits;
    const int rest = k / p.splits;
    const int pair = p.pairs - 1 - rest / p.BH;  // heaviest pairs first
    const int fmax = unit_tiles(p, pair);
    return make_unit(p, rest % p.BH, split, pair, split * fmax / p.splits,
                     (split + 1) * fmax / p.splits);
}

// Stream-K (one Q-tile pair per head): the BH * F (head, key tile) steps,
// head-major, are dealt in equal contiguous ranges, CTA c taking
// [c W / G, (c+1) W / G).  A head split over several CTAs gets one partial
// slot per CTA, numbered from the first CTA that covers it.
__host__ __device__ __forceinline__ long long sk_lo(long long W, int G, long long c)
{
    return c * W / G;
}
// The CTA whose range holds step x: the largest c with lo(c) <= x.
__host__ __device__ __forceinline__ int sk_cta(long long W, int G, long long x)
{
    return static_cast<int>(((x + 1) * G - 1) / W);
}

// Serpentine deal: round r gives CTA c the unit r*G + c (r even) or
// r*G + G-1-c (r odd).
__device__ __forceinline__ int unit_index(int round, int cta, int grid)
{
    return round * grid + ((round & 1) ? grid - 1 - cta : cta);
}

// The r-th work unit of this CTA; false past its last.  Under stream-K the
// r-th unit is the r-th head of the CTA's range: every head after the first
// starts inside the range, so this CTA is its first (slot 0).
__device__ __forceinline__ bool cta_unit(const Params &p, const Bars &b, int r, Unit &u)
{
    if (p.streamk) {
        const int h = b.sk_h0 + r;
        const long long base = static_cast<long long>(h) * p.F;
        if (h >= p.BH || base >= b.sk_hi)
            return false;
        const int je = static_cast<int>(min(b.sk_hi - base, static_cast<long long>(p.F)));
        u = make_unit(p, h, r == 0 ? b.sk_slot0 : 0, 0, r == 0 ? b.sk_j0 : 0, je);
        return true;
    }
    const int k = unit_index(r, blockIdx.x, gridDim.x);
    if (k >= p.units)
        return false;
    u = unit_at(p, k);
    return true;
}

__device__ __forceinline__ void record_failure(Bars &b, uint32_t role)
{
    const uint32_t code = 4u /* FATTN_ERR_TIMEOUT */ | (role << 8) | ((blockIdx.x & 0xffffu) << 16);
    atomicCAS(&g_fattn_status, 0u, code);
    *reinterpret_cast<volatile int *>(&b.abort) = 1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two floats rounded to the 16-bit element type (bf16, or fp16 when kF16),
// low half first.
template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (kF16) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    } else {
        return pack_bf16x2(lo, hi);
    }
}

// ------------------------------------------------------------------ producer
// The producer and MMA roles run on a whole converged warp so that their
// address and descriptor arithmetic stays warp-uniform; one elected lane
// issues each TMA copy, MMA and commit.  Waits are done by every lane and
// their outcome is made warp-uniform with a vote.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort)
{
    const bool ok = mbar_wait(bar, parity, kWaitLimitNs, abort);
    return __all_sync(0xffffffffu, ok);
}

template <int D>
__device__ void run_load(const Params &p, Bars &b, uint32_t smem_base, const CUtensorMap *mq,
                         const CUtensorMap *mk, const CUtensorMap *mv)
{
    using C = Cfg<D>;
    const volatile int *abort = &b.abort;
    const bool leader = elect_one();
    uint32_t q_phase[2] = {0, 0};
    uint32_t pos = 0;  // K/V ring position (K_j, V_j alternate)
    bool ok = true;
    int last_q_parity[2] = {-1, -1};
    // Launched behind the V pre-pass (kPrecBf16V16): its writes are visible
    // after this wait.  Without a preceding dependent grid it returns at once.
    grid_dependency_wait();
    for (int r = 0; ok; ++r) {
        Unit u;
        if (!cta_unit(p, b, r, u))
            break;
        const int hh = u.bh % p.H, bb = u.bh / p.H;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!ok || u.n[t] == 0)
                continue;
            const uint32_t full = smem_addr(&b.q_full[t]);
            if (!warp_wait(smem_addr(&b.q_empty[t]), q_phase[t] ^ 1, abort)) {
                ok = false;
                break;
            }
            if (leader) {
                mbar_arrive_expect_tx(full, C::kTileBytes);
                const uint32_t dst = smem_base + t * C::kTileBytes;
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_4d(dst + c * kChunkBytes, mq, full, 64 * c, u.qt[t] * kBM, hh, bb);
            }
            last_q_parity[t] = q_phase[t];
            q_phase[t] ^= 1;
        }
        for (int j = u.j0; ok && j < u.j0 + u.n_max; ++j) {
#pragma unroll
            for (int which = 0; which < 2; ++which, ++pos) {
                const uint32_t stage = pos % C::kStages;
                const uint32_t phase = (pos / C::kStages) & 1;
                if (!warp_wait(smem_addr(&b.kv_empty[stage]), phase ^ 1, abort)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    const uint32_t full = smem_addr(&b.kv_full[stage]);
                    mbar_arrive_expect_tx(full, C::kTileBytes);
                    const uint32_t dst = smem_base + (2 + stage) * C::kTileBytes;
                    const CUtensorMap *m = which == 0 ? mk : mv;
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_4d(dst + c * kChunkBytes, m, full, 64 * c, j * kBN, hh, bb);
                }
            }
        }
    }
    if (!ok) {
        if (leader)
            record_failure(b, kRoleLoad);
        // Let the copies already issued land before the CTA exits.
        const uint32_t issued = pos;
        const uint32_t first = issued > (uint32_t)C::kStages ? issued - C::kStages : 0;
        for (uint32_t q = first; q < issued; ++q)
            mbar_wait(smem_addr(&b.kv_full[q % C::kStages]), (q / C::kStages) & 1,
                      kWaitLimitNs / 8, nullptr);
        for (int t = 0; t < 2; ++t)
            if (last_q_parity[t] >= 0)
                mbar_wait(smem_addr(&b.q_full[t]), last_q_parity[t], kWaitLimitNs / 8, nullptr);
    }
}

// ------------------------------------------------------------------ V conversion
// kPrecBf16: the P V product runs in fp16 (both operands of one product share
// one type), so every V tile is rewritten in place from bf16 to fp16 after its
// copy lands and before the product reads it.  Element order and swizzle are
// unchanged (both types are 2 bytes).  The conversion is exact for |v| <
// 65520 (fp16 has three more significand bits than bf16; the smallest bf16
// magnitudes become fp16 subnormals, off by at most 2^-25); a larger
// magnitude becomes infinite, which makes the rows that weigh it non-finite:
// the epilogue records FATTN_ERR_RANGE for any non-finite output row (see
// epilogue_row).  Three instructions a pair of elements: two to widen the
// bf16 halves to fp32, one to round both to fp16.  Two converter warps share
// each tile.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 w)
{
    return make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z),
                      bf16x2_to_f16x2(w.w));
}

constexpr int kConvThreads = 64;

// Eight 16-byte steps in flight per thread over kVecs consecutive granules.
template <int kVecs>
__device__ __forceinline__ void convert_linear(uint4 *tile, int tid)
{
    constexpr int kBatch = 8;
    static_assert(kVecs % (kConvThreads * kBatch) == 0, "whole batches per thread");
#pragma unroll 1
    for (int base = tid; base < kVecs; base += kConvThreads * kBatch) {
        uint4 w[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            w[i] = tile[base + i * kConvThreads];
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            tile[base + i * kConvThreads] = bf16x8_to_f16x8(w[i]);
    }
}

// A whole tile: its 64-column boxes of 128 rows x 128 bytes.  At d = 96 the
// second box holds columns 64..95 in its logical granules 0-3 (granule g of
// row r sits at g ^ (r % 8)) and the copy's zero fill in 4-7, which no
// product reads: only the used half is converted.  Each 8-lane store phase
// covers rows r and r + 4, whose granules 0-3 land on complementary halves
// of the banks.
template <int D, uint32_t kTileBytes>
__device__ __forceinline__ void convert_tile(uint8_t *tile, int tid)
{
    if constexpr (D % 64 == 0) {
        convert_linear<kTileBytes / 16>(reinterpret_cast<uint4 *>(tile), tid);
    } else {
        static_assert(D == 96 && kTileBytes == 2 * kChunkBytes, "d = 96: two boxes");
        convert_linear<kChunkBytes / 16>(reinterpret_cast<uint4 *>(tile), tid);
        uint8_t *box = tile + kChunkBytes;
        constexpr int kBatch = 8;
#pragma unroll 1
        for (int base = tid; base < kBM * 4; base += kConvThreads * kBatch) {
            uint4 w[kBatch];
            uint4 *at[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                const int x = base + i * kConvThreads, k = x / 8, e = x % 8;
                const int r = (k / 4) * 8 + k % 4 + (e / 4) * 4, g = e % 4;
                at[i] = reinterpret_cast<uint4 *>(box + r * 128 + ((g ^ (r & 7)) << 4));
                w[i] = *at[i];
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                *at[i] = bf16x8_to_f16x8(w[i]);
        }
    }
}

// Converter warp cw (0 or 1); its waits are warp-uniform (warp_wait), so a
// timeout never splits the warp before the __syncwarp in convert.  Visits
// the V tiles in the producer's order:
// the two-tile kernel's ring holds K_j and V_j alternately over an even
// number of stages, so V copies always land on the odd stages, whose
// kv_full phases are all V copies; the one-tile kernel loads K_0, K_1, then
// V_i and K_(i+2) alternately, its V copies completing on v_full (one phase
// bit per stage).  For each V tile it waits for the copy, converts its share,
// makes the writes visible to the tensor cores (async proxy) and arrives on
// v_ready of the stage.
template <int D, int kPrec>
__device__ void run_convert(const Params &p, Bars &b, uint8_t *tiles, int cw)
{
    using C = Cfg<D, kPrec>;
    const volatile int *abort = &b.abort;
    const int lane = threadIdx.x & 31;
    const int tid = cw * 32 + lane;
    uint32_t pos = 0, vbits = 0;
    bool ok = true;
    auto convert = [&](uint32_t stage) {
        convert_tile<D, C::kTileBytes>(tiles + (C::kQTiles + stage) * C::kTileBytes, tid);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&b.v_ready[stage]));
    };
    // One-tile kernel: half h of the V tile in this stage (slot 2 * stage + h).
    auto convert_half = [&](uint32_t stage, int h) {
        convert_linear<C::kHalfBytes / 16>(
            reinterpret_cast<uint4 *>(tiles + (C::kQTiles + stage) * C::kTileBytes +
                                      h * C::kHalfBytes),
            tid);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&b.v_ready[2 * stage + h]));
    };
    for (int r = 0; ok; ++r) {
        Unit u;
        if (!cta_unit(p, b, r, u))
            break;
        if constexpr (C::kQTiles == 2) {
            for (int i = 0; ok && i < u.n_max; ++i) {
                const uint32_t at = pos + 2 * i + 1;
                const uint32_t stage = at % C::kStages;
                ok = warp_wait(smem_addr(&b.kv_full[stage]), (at / C::kStages) & 1, abort);
                if (ok)
                    convert(stage);
            }
            pos += 2 * u.n_max;
        } else {
            const int n = u.n[0];
            if (n == 0)
                continue;
            pos += n > 1 ? 2 : 1;  // K_0 (and K_1)
            for (int i = 0; ok && i < n; ++i) {
                const uint32_t stage = pos % C::kStages;
                const uint32_t parity = (vbits >> stage) & 1u;
                vbits ^= 1u << stage;
                for (int h = 0; ok && h < 2; ++h) {
                    ok = warp_wait(smem_addr(&b.v_full[2 * stage + h]), parity, abort);
                    if (ok)
                        convert_half(stage, h);
                }
                pos += i + 2 < n ? 2 : 1;  // V_i (and K_(i+2))
            }
        }
    }
    if (!ok && lane == 0)
        record_failure(b, kRoleConvert);
}

// ------------------------------------------------------------------ MMA issue
// S = Q K^T: both operands K-major (d contiguous), 128-byte swizzled, 8-row
// groups 1024 bytes apart.  Each K = 16 step moves 32 bytes along d inside a
// 64-column box, or to the next 16 KB box.  The start address occupies the
// low 14 bits of the descriptor's low word and never carries out of them
// (shared memory is below 256 KB), so a step is one 32-bit add.
template <int D, int kPrec, int kK0 = 0, int kK1 = D / 16>
__device__ __forceinline__ void issue_s(uint32_t tmem_d, uint32_t q_smem, uint32_t k_smem)
{
    constexpr uint32_t idesc = idesc_f32acc(kBM, kBN, false, Cfg<D, kPrec>::kInF16);
    constexpr uint32_t hi = smem_desc_hi(1024);
    const uint32_t a_lo = smem_desc_lo(q_smem, 16), b_lo = smem_desc_lo(k_smem, 16);
#pragma unroll
    for (int kk = kK0; kk < kK1; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ss_w(tmem_d, a_lo + off, hi, b_lo + off, hi, idesc, kk > 0 ? 1u : 0u);
    }
}

// V tiles are MN-major (d contiguous) for the P V product: the stride between
// 8-key groups is 1024 bytes (SBO) and the stride between the two 64-column
// halves of d = 128 is one 16 KB box (LBO; with d = 64 there is one half and
// the value is irrelevant, so it is kept inside the tile).  P is read from
// tensor memory, 8 columns (16 keys of bf16 pairs) per K = 16 step.
// With the ones column (Cfg::kOnes, d = 64) N = 80: the MMA's second atom
// along N is the constant ones atom, so LBO is its distance from this stage.
// In the one-tile kernel (Cfg::kHalves = 2) a V tile is two 32 KB halves of
// 64 keys, each four 8 KB boxes of 64 columns: LBO is 8 KB, and K-step kk
// reads half kk / 4.
template <int D, int kPrec, int kK0 = 0, int kK1 = kBN / 16>
__device__ __forceinline__ void issue_pv(uint32_t tmem_d, uint32_t tmem_p, uint32_t v_smem,
                                         uint32_t ones_smem, bool accumulate)
{
    using C = Cfg<D, kPrec>;
    constexpr bool kSplitV = C::kHalves == 2;
    constexpr uint32_t idesc = idesc_f32acc(kBM, C::kON, true, C::kPF16);
    constexpr uint32_t kVLbo = kSplitV ? kChunkBytes / 2 : (D > 64 ? kChunkBytes : 1024);
    constexpr uint32_t hi = smem_desc_hi(1024);
    const uint32_t b_lo = smem_desc_lo(v_smem, C::kOnes ? ones_smem - v_smem : kVLbo);
    const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
    for (int kk = kK0; kk < kK1; ++kk) {
        const uint32_t off = kSplitV ? (kk / 4) * C::kHalfBytes + (kk % 4) * 16 * 128
                                     : kk * 16 * 128;
        mma_ts_w(tmem_d, tmem_p + kk * 8, b_lo + (off >> 4), hi, idesc, kk > 0 ? 1u : acc0);
    }
}

template <int D, int kPrec>
__device__ void run_mma(const Params &p, Bars &b, uint32_t smem_base, uint32_t tmem)
{
    using C = Cfg<D, kPrec>;
    const volatile int *abort = &b.abort;
    const bool leader = elect_one();
    uint32_t q_phase[2] = {0, 0}, p_phase[2] = {0, 0}, ph_phase[2] = {0, 0}, oe_phase[2] = {0, 0};
    uint32_t pos = 0;
    bool ok = true;

    auto kv_stage = [&](uint32_t at) { return at % C::kStages; };
    auto kv_wait = [&](uint32_t at) {
        return warp_wait(smem_addr(&b.kv_full[at % C::kStages]), (at / C::kStages) & 1, abort);
    };
    auto kv_smem = [&](uint32_t at) { return smem_base + (2 + kv_stage(at)) * C::kTileBytes; };
    // A V tile is ready once copied (and, with converter warps, converted);
    // v_ready keeps one phase bit per stage.
    uint32_t vr_bits = 0;
    auto v_wait = [&](uint32_t at) {
        if constexpr (!C::kConv) {
            return kv_wait(at);
        } else {
            const uint32_t st = at % C::kStages;
            const bool r = warp_wait(smem_addr(&b.v_ready[st]), (vr_bits >> st) & 1u, abort);
            vr_bits ^= 1u << st;
            return r;
        }
    };
    auto commit = [&](uint64_t &bar) {
        if (leader)
            mma_commit(smem_addr(&bar));
    };

    for (int r = 0; ok; ++r) {
        Unit u;
        if (!cta_unit(p, b, r, u))
            break;
        const uint32_t base = pos;  // K_(j0+i) at base + 2i, V_(j0+i) at base + 2i + 1
        if (u.n_max == 0)
            continue;
        for (int t = 0; t < 2 && ok; ++t)
            if (u.n[t] > 0) {
                ok = warp_wait(smem_addr(&b.q_full[t]), q_phase[t], abort);
                q_phase[t] ^= 1;
            }
        if (ok)
            ok = kv_wait(base);
        if (!ok)
            break;
        tc_fence_after();
        // First key tile: S for both Q tiles.
        for (int t = 0; t < 2; ++t) {
            if (u.n[t] == 0)
                continue;
            if (leader)
                issue_s<D, kPrec>(tmem + (t == 0 ? 0u : 128u), smem_base + t * C::kTileBytes,
                           kv_smem(base));
            commit(b.s_full[t]);
            if (u.n[t] == 1)
                commit(b.q_empty[t]);
        }
        commit(b.kv_empty[kv_stage(base)]);

        // Key tiles 1..n-1 of the unit: P V of the previous tile, then S of
        // this one (j counts key tiles from j0).
        for (int j = 1; j <= u.n_max && ok; ++j) {
            const uint32_t at_v = base + 2 * (j - 1) + 1;
            const uint32_t at_k = base + 2 * j;
            const bool has_k = j < u.n_max;
            ok = v_wait(at_v) && (!has_k || kv_wait(at_k));
            if (!ok)
                break;
            for (int t = 0; t < 2 && ok; ++t) {
                if (j - 1 >= u.n[t])
                    continue;  // tile t finished earlier (or is absent)
                // With kHalfP, P V in two halves: keys 0-63 as soon as the
                // softmax has written their P, keys 64-127 once all of P is.
                if (C::kHalfP) {
                    ok = warp_wait(smem_addr(&b.p_half[t]), ph_phase[t], abort);
                    ph_phase[t] ^= 1;
                } else {
                    ok = warp_wait(smem_addr(&b.p_full[t]), p_phase[t], abort);
                    p_phase[t] ^= 1;
                }
                if (ok && j - 1 == 0) {  // first P V of the unit overwrites O
                    ok = warp_wait(smem_addr(&b.o_empty[t]), oe_phase[t] ^ 1, abort);
                    oe_phase[t] ^= 1;
                }
                if (!ok)
                    break;
                tc_fence_after();
                const uint32_t col_s = t == 0 ? 0u : 128u;
                const uint32_t col_o = t == 0 ? C::kColO0 : C::kColO1;
                if (C::kHalfP) {
                    if (leader)
                        issue_pv<D, kPrec, 0, kBN / 32>(tmem + col_o, tmem + col_s, kv_smem(at_v),
                                                       smem_base + C::kOnesOffset, j - 1 > 0);
                    ok = warp_wait(smem_addr(&b.p_full[t]), p_phase[t], abort);
                    p_phase[t] ^= 1;
                    if (!ok)
                        break;
                    tc_fence_after();
                    if (leader)
                        issue_pv<D, kPrec, kBN / 32, kBN / 16>(tmem + col_o, tmem + col_s,
                                                              kv_smem(at_v),
                                                              smem_base + C::kOnesOffset, true);
                } else if (leader) {
                    issue_pv<D, kPrec>(tmem + col_o, tmem + col_s, kv_smem(at_v),
                                      smem_base + C::kOnesOffset, j - 1 > 0);
                }
                if (j < u.n[t]) {
                    if (leader)
                        issue_s<D, kPrec>(tmem + col_s, smem_base + t * C::kTileBytes, kv_smem(at_k));
                    commit(b.s_full[t]);
                    if (j == u.n[t] - 1)
                        commit(b.q_empty[t]);
                } else {
                    commit(b.o_full[t]);
                }
            }
            if (!ok)
                break;
            commit(b.kv_empty[kv_stage(at_v)]);
            if (has_k)
                commit(b.kv_empty[kv_stage(at_k)]);
        }
        pos = base + 2 * u.n_max;
    }
    if (!ok && leader)
        record_failure(b, kRoleMma);
    // Wait until every MMA this warp issued has completed.
    commit(b.drain);
    mbar_wait(smem_addr(&b.drain), 0, kWaitLimitNs, nullptr);
}

// ------------------------------------------------------------------ softmax
// One key tile of one row (thread r of the tile's warpgroup), on the S row at
// TMEM address t_s: mask, row max, p = 2^(s*scale*log2e - m), P (16-bit)
// written over the first 64 columns of S, and the row sums.  Returns the
// rescale factor alpha of O and l for the new running max m_new.  pre(alpha)
// runs once alpha is known, before any P is written; mid() runs when P of the
// first 64 keys has been stored.
struct NoHook {
    __device__ __forceinline__ void operator()() const {}
    __device__ __forceinline__ void operator()(float) const {}
};

template <int D, int kPrec, bool kOnes, class Pre = NoHook, class Mid = NoHook>
__device__ __forceinline__ float softmax_tile(const Params &p, uint32_t t_s, int r, int j,
                                              int first_vis, bool first, float m, float &m_new,
                                              float &l, float &l_round, Pre pre = Pre(),
                                              Mid mid = Mid())
{
    // The whole S row: four 32-column loads in flight, one wait.  The
    // loads also reduce: each returns the maximum of its 32 columns, which
    // is the row maximum's input wherever no key is masked.
    uint32_t sraw[kBN / 32][32];
    float cmax[kBN / 32];
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c)
        tmem_ld32_max(t_s + c * 32, sraw[c], cmax[c]);
    tmem_wait_ld();
    float s[kBN];
#pragma unroll
    for (int i = 0; i < kBN; ++i)
        s[i] = __uint_as_float(sraw[i / 32][i % 32]);
    // Mask (only on tiles that cross the diagonal and on the ragged last
    // tile; the branch is uniform across the warp): keys past row position +
    // off and keys past Nk get -inf, i.e. weight exactly 0.  first_vis is
    // the last visible column of row 0 in this key tile.  The row max is
    // then taken over the masked values: four independent chains of 3-input
    // max over s[0..kBN).
    const bool diag = p.causal && first_vis < kBN - 1;
    const bool tail = (j + 1) * kBN > p.Nk;
    static_assert(kBN == 128, "four 32-column loads a row");
    float smax = fmaxf(fmaxf(cmax[0], cmax[1]), fmaxf(cmax[2], cmax[3]));
    if (diag || tail) {
        int limit = diag ? first_vis + r : kBN - 1;
        if (tail)
            limit = min(limit, p.Nk - 1 - j * kBN);
#pragma unroll
        for (int i = 0; i < kBN; ++i)
            s[i] = i > limit ? -INFINITY : s[i];
        float mx[4] = {fmaxf(s[0], s[1]), fmaxf(s[2], s[3]), fmaxf(s[4], s[5]), fmaxf(s[6], s[7])};
#pragma unroll
        for (int i = 8; i < kBN; i += 8) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                mx[c] = fmax3(mx[c], s[i + 2 * c], s[i + 2 * c + 1]);
        }
        smax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    }
    const float cand = smax * p.sl2;
    m_new = (first || cand > m + kRescaleLog2) ? fmaxf(m, cand) : m;
    const float alpha = ex2(m - m_new);  // 0 on the first tile, 1 when m is kept
    pre(alpha);
    // p = 2^(s*scale*log2e - m), two lanes per instruction, and its row sum
    // (two independent packed accumulators, four partials).
    const uint64_t sl2x2 = f2_pack(p.sl2, p.sl2);
    const uint64_t negm = f2_pack(-m_new, -m_new);
    uint64_t sum_exact[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), sl2x2, negm), x0,
                      x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            pk[i] = pack2<Cfg<D, kPrec>::kPF16>(p0, p1);
            sum_exact[i & 1] = f2_add(sum_exact[i & 1], f2_pack(p0, p1));
        }
        tmem_st16(t_s + c * 16, pk);
        if (c == kBN / 64 - 1)
            mid();
    }
    float e0, e1, e2, e3;
    f2_unpack(sum_exact[0], e0, e1);
    f2_unpack(sum_exact[1], e2, e3);
    const float esum = (e0 + e1) + (e2 + e3);
    l = l * alpha + esum;
    if constexpr (!Cfg<D, kPrec>::kPF16 && !kOnes) {
        // The tile's largest p, from the same fused multiply-add and
        // exponential as its P element, and its bf16 rounding error.
        const float pt = ex2(fmaf(smax, p.sl2, -m_new));
        const float pt_round = __uint_as_float(pack2<false>(pt, pt) & 0xffff0000u);
        l_round = l_round * alpha + (esum - (pt - pt_round));
    }
    return alpha;
}

// O row (and with kOnes the l_round column) times alpha, in TMEM.  The
// rescale sits on the softmax's path to P V, and with wide logits a warp
// needs one on a large share of its key tiles (some row's maximum rises past
// the threshold), so the chunks' loads are issued together and waited for
// once: up to 128 columns at a time (D = 256: two batches).
template <int D, bool kOnes>
__device__ __forceinline__ void rescale_o(uint32_t t_o, float alpha)
{
    constexpr int kChunksPerBatch = D <= 128 ? D / 32 : 4;
    const uint64_t alpha2 = f2_pack(alpha, alpha);
    // Two columns per packed multiply.
    auto scale = [&](uint32_t &a, uint32_t &b) {
        float x, y;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(a), __uint_as_float(b)), alpha2), x, y);
        a = __float_as_uint(x);
        b = __float_as_uint(y);
    };
#pragma unroll 1
    for (int c0 = 0; c0 < D / 32; c0 += kChunksPerBatch) {
        uint32_t o[kChunksPerBatch][32];
#pragma unroll
        for (int c = 0; c < kChunksPerBatch; ++c)
            tmem_ld32(t_o + (c0 + c) * 32, o[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kChunksPerBatch; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2)
                scale(o[c][i], o[c][i + 1]);
            tmem_st32(t_o + (c0 + c) * 32, o[c]);
        }
    }
    if constexpr (kOnes) {  // the l_round column and its 15 zero neighbours
        uint32_t o[16];
        tmem_ld16(t_o + D, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; i += 2)
            scale(o[i], o[i + 1]);
        tmem_st16(t_o + D, o);
    }
}

// Staged row stores (both kernels, every d).  The epilogue runs on
// the softmax warps between units, so with short units (a few key tiles per
// Q tile) its store time is a large share of the launch.  Thread r of a warp (row r of the warp's 32) puts a 128-byte piece of its row
// into row r of the warp's staging area, 16-byte granule g at position
// g ^ (r % 8), so the 8 threads of a store phase hit 8 different bank groups;
// then 8 lanes per row copy the pieces out as whole 128-byte lines, 4 rows per
// instruction, instead of 32 rows' 16-byte pieces per instruction.
__device__ __forceinline__ void stage_put(uint8_t *stage, int lane, int g, uint4 v)
{
    reinterpret_cast<uint4 *>(stage + lane * 128)[g ^ (lane & 7)] = v;
}

// The first 64 bytes of each staged row (the last 32 columns of a d = 96
// row): 4 lanes per row, 8 rows per instruction.
__device__ __forceinline__ void stage_flush_half(const uint8_t *stage, int lane, char *dst0,
                                                 long long row_bytes, int live_rows)
{
    __syncwarp();
    const int g = lane % 4;
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
        const int rr = pass * 8 + lane / 4;
        const uint4 x = reinterpret_cast<const uint4 *>(stage + rr * 128)[g ^ (rr & 7)];
        if (rr < live_rows)
            *reinterpret_cast<uint4 *>(dst0 + rr * row_bytes + g * 16) = x;
    }
    __syncwarp();
}

__device__ __forceinline__ void stage_flush(const uint8_t *stage, int lane, char *dst0,
                                            long long row_bytes, int live_rows)
{
    __syncwarp();
    const int g = lane % 8;
#pragma unroll
    for (int pass = 0; pass < 8; ++pass) {
        const int rr = pass * 4 + lane / 8;
        const uint4 x = reinterpret_cast<const uint4 *>(stage + rr * 128)[g ^ (rr & 7)];
        if (rr < live_rows)
            *reinterpret_cast<uint4 *>(dst0 + rr * row_bytes + g * 16) = x;
    }
    __syncwarp();
}

// The epilogue's check for non-finite output (V rounded to fp16): sums a
// chunk of the unnormalised O row into two packed accumulators.  Every
// finite O element is below 2^8 * Nk * 65504 in magnitude (p <= 2^8 with the
// rescale threshold, |v| < 65520), so a finite row sums to a finite value far
// below FLT_MAX, and an infinity or NaN anywhere makes the sum non-finite.
__device__ __forceinline__ void nonfinite_acc(const uint32_t (&o)[32], uint64_t (&acc)[2])
{
#pragma unroll
    for (int i = 0; i < 16; ++i)
        acc[i & 1] = f2_add(acc[i & 1], f2_pack(__uint_as_float(o[2 * i]),
                                                __uint_as_float(o[2 * i + 1])));
}

// Epilogue of one row after the unit's last P V: O / l_round in bf16 (fp16)
// and lse = ln2 * (m + log2 l); in split mode the fp32 partial O and the two
// base-2 partial lse go to the workspace instead, for the combine kernel.  The
// rows leave through the staging area (softmax warp w uses its w-th 4 KB) in
// 128-byte pieces of the row (and a 64-byte last piece of a d = 96 bf16 row).
template <int D, int kPrec, bool kOnes>
__device__ __forceinline__ void epilogue_row(const Params &p, const Unit &u, uint32_t t_o, int row,
                                             float m, float l, float l_round)
{
    static_assert(D % 32 == 0, "staged rows are 64- and 128-byte pieces");
    // fp16 P is rounded 8x more finely than bf16 P: O is normalised by the
    // exact sum there.  With the ones column l_round is O column D.  l is 0
    // only for a split that saw no key of this row.
    if constexpr (kOnes) {
        l_round = __uint_as_float(tmem_ld1(t_o + D));
        tmem_wait_ld();
    }
    constexpr bool kOutF16 = Cfg<D, kPrec>::kInF16;
    const float l_norm = Cfg<D, kPrec>::kPF16 ? l : l_round;
    const float inv_l = l_norm > 0.f ? 1.f / l_norm : 0.f;
    const uint64_t inv2 = f2_pack(inv_l, inv_l);
    const bool live = row < p.Nq;
    const size_t grow = static_cast<size_t>(u.bh) * p.Nq + row;
    // With V converted to fp16 (kPrecBf16, kPrecBf16V16), a V element of
    // magnitude 65520 or more turns into an infinity: a non-finite output row
    // (which non-finite inputs also give) records FATTN_ERR_RANGE.
    uint64_t nf[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
    auto check = [&](const uint32_t (&o)[32]) {
        if constexpr (Cfg<D, kPrec>::kVRounded)
            nonfinite_acc(o, nf);
    };
    // O times 1/l, two columns per packed multiply.
    auto scaled = [&](const uint32_t (&o)[32], int i, float &a, float &b) {
        f2_unpack(f2_mul(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), inv2), a, b);
    };
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t *stage = smem_raw + (((raw + 1023u) & ~1023u) - raw) + Cfg<D, kPrec>::kStageOffset +
                     (threadIdx.x / 32) * 4096;
    const int lane = threadIdx.x & 31;
    const int row0 = row - lane;  // the warp's first row
    const int live_rows = min(32, p.Nq - row0);
    if (p.splits == 1) {  // 64 columns (128 bytes) a piece
        char *dst0 = reinterpret_cast<char *>(
            static_cast<uint16_t *>(p.o) + (u.bh / p.H) * p.o_sb + (u.bh % p.H) * p.o_sh +
            static_cast<long long>(row0) * p.o_sn);
        // One 64-column piece: its two 32-column chunks of O, loaded together
        // (one wait) where the registers allow it, i.e. without converter
        // warps in the kernel, else one chunk per wait.
        constexpr int kLoads = Cfg<D, kPrec>::kConv || D % 64 != 0 ? 1 : 2;
#pragma unroll 1
        for (int c = 0; c < D / 32; c += kLoads) {
            uint32_t o[kLoads][32];
            __syncwarp();
#pragma unroll
            for (int h = 0; h < kLoads; ++h)
                tmem_ld32(t_o + (c + h) * 32, o[h]);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < kLoads; ++h) {
                check(o[h]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float a, b;
                        scaled(o[h], 8 * i + 2 * k, a, b);
                        w[k] = pack2<kOutF16>(a, b);
                    }
                    stage_put(stage, lane, ((c + h) % 2) * 4 + i, make_uint4(w[0], w[1], w[2], w[3]));
                }
            }
            if ((c + kLoads - 1) % 2 == 1)
                stage_flush(stage, lane, dst0 + ((c + kLoads - 1) / 2) * 128, p.o_sn * 2,
                            live_rows);
            else if (c + kLoads == D / 32)  // d = 96: the row's last 64 bytes
                stage_flush_half(stage, lane, dst0 + (c / 2) * 128, p.o_sn * 2, live_rows);
        }
        if (live)
            p.lse[grow] = (m + log2f(l)) * kLn2;
    } else {  // 32 fp32 columns (128 bytes) a piece
        const size_t srow0 = static_cast<size_t>(u.split) * p.BH * p.Nq + grow - lane;
        char *dst0 = reinterpret_cast<char *>(p.ws_o + srow0 * D);
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            __syncwarp();
            tmem_ld32(t_o + c * 32, o);
            tmem_wait_ld();
            check(o);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float a, b, cc, dd;
                scaled(o, 4 * i, a, b);
                scaled(o, 4 * i + 2, cc, dd);
                stage_put(stage, lane, i, make_uint4(__float_as_uint(a), __float_as_uint(b),
                                                     __float_as_uint(cc), __float_as_uint(dd)));
            }
            stage_flush(stage, lane, dst0 + c * 128, static_cast<long long>(D) * 4, live_rows);
        }
        if (live)
            p.ws_l[srow0 + lane] = make_float2(m + log2f(l), m + log2f(l_norm));
    }
    if constexpr (Cfg<D, kPrec>::kVRounded) {
        float e0, e1, e2, e3;
        f2_unpack(nf[0], e0, e1);
        f2_unpack(nf[1], e2, e3);
        const float acc = (e0 + e1) + (e2 + e3);
        if (live && !(fabsf(acc) <= FLT_MAX)) {
            const uint32_t code = 5u /* FATTN_ERR_RANGE */ | (kRoleEpilogue << 8) |
                                  ((blockIdx.x & 0xffffu) << 16);
            atomicCAS(&g_fattn_status, 0u, code);
        }
    }
}

template <int D, int kPrec>
__device__ void run_softmax(const Params &p, Bars &b, uint32_t tmem, int t)
{
    using C = Cfg<D, kPrec>;
    const volatile int *abort = &b.abort;
    const int warp = (threadIdx.x / 32) & 3;
    const int lane = threadIdx.x & 31;
    const int r = warp * 32 + lane;                          // row within the Q tile
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t t_s = tmem + lane_off + (t == 0 ? 0u : 128u);
    const uint32_t t_o = tmem + lane_off + (t == 0 ? C::kColO0 : C::kColO1);
    uint32_t s_phase = 0, of_phase = 0;
    bool ok = true;

    for (int rr = 0; ok; ++rr) {
        Unit u;
        if (!cta_unit(p, b, rr, u))
            break;
        if (u.n[t] == 0)
            continue;
        const int qt = u.qt[t];
        const int row = qt * kBM + r;
        // m starts at -FLT_MAX, not -inf: a row can see no key of a tile
        // only on its last tile (when Nk - Nq is not a multiple of 128), and
        // when that tile is also its first in this unit, m - m_new and the
        // exponents stay -inf or 0 instead of NaN (l = 0, lse = -inf).
        float m = -FLT_MAX, l = 0.f, l_round = 0.f;
        // Last visible column of row 0 in key tile j (causal mask).
        int first_vis = qt * kBM + p.off - u.j0 * kBN;
        for (int j = u.j0; j < u.j1[t]; ++j, first_vis -= kBN) {
            const bool first = j == u.j0;
            ok = mbar_wait(smem_addr(&b.s_full[t]), s_phase, kWaitLimitNs, abort);
            s_phase ^= 1;
            if (!ok)
                break;
            tc_fence_after();
            __syncwarp();
            float m_new;
            if constexpr (C::kHalfP) {
                // P of the first 64 keys goes to the tensor cores as soon as
                // it is written, unless O has to be rescaled first (rare; the
                // warp decides together): then both halves follow the rescale.
                bool rescale = false;
                auto pre = [&](float) { rescale = !first && __any_sync(0xffffffffu, m_new != m); };
                auto mid = [&]() {
                    if (!rescale) {
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(smem_addr(&b.p_half[t]));
                    }
                };
                const float alpha = softmax_tile<D, kPrec, C::kOnes>(
                    p, t_s, r, j, first_vis, first, m, m_new, l, l_round, pre, mid);
                if (rescale)
                    rescale_o<D, C::kOnes>(t_o, alpha);
                m = m_new;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (rescale)
                        mbar_arrive(smem_addr(&b.p_half[t]));
                    mbar_arrive(smem_addr(&b.p_full[t]));
                }
            } else {
                const float alpha = softmax_tile<D, kPrec, C::kOnes>(p, t_s, r, j, first_vis, first,
                                                                    m, m_new, l, l_round);
                if (!first && __any_sync(0xffffffffu, m_new != m))
                    rescale_o<D, C::kOnes>(t_o, alpha);
                m = m_new;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&b.p_full[t]));
            }
        }
        if (!ok)
            break;
        ok = mbar_wait(smem_addr(&b.o_full[t]), of_phase, kWaitLimitNs, abort);
        of_phase ^= 1;
        if (!ok)
            break;
        tc_fence_after();
        epilogue_row<D, kPrec, C::kOnes>(p, u, t_o, row, m, l, l_round);
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&b.o_empty[t]));
    }
    if (!ok)
        record_failure(b, kRoleSoftmax);
}

// ------------------------------------------------------------------ kernel
// The ones atom (Cfg::kOnes): 128 key rows of 128 bytes in the 128-byte
// swizzle (16-byte chunk c of row k stored at chunk c ^ (k % 8)); column 0
// (chunk 0, first element) is bf16 1.0, everything else 0.  Written by all
// threads before the CTA-wide barrier that precedes the first MMA.
__device__ __forceinline__ void init_ones_atom(uint8_t *atom)
{
    uint32_t *ones = reinterpret_cast<uint32_t *>(atom);
    for (int w = threadIdx.x; w < static_cast<int>(kChunkBytes / 4); w += blockDim.x) {
        const int k = w / 32, wr = w % 32;
        ones[w] = wr == (k % 8) * 4 ? 0x3F80u : 0u;  // bf16 1.0 in the low half
    }
    fence_proxy_async_smem();
}

template <int D, int kPrec>
__global__ void __launch_bounds__(Cfg<D, kPrec>::kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
               const __grid_constant__ CUtensorMap mv, const Params p)
{
    using C = Cfg<D, kPrec>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t smem_base = (raw + 1023u) & ~1023u;
    Bars &b = *reinterpret_cast<Bars *>(smem_raw + (smem_base - raw) + C::kBarsOffset);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_addr(&b.q_full[t]), 1);
            mbar_init(smem_addr(&b.q_empty[t]), 1);
            mbar_init(smem_addr(&b.s_full[t]), 1);
            mbar_init(smem_addr(&b.p_full[t]), 4);
            mbar_init(smem_addr(&b.p_half[t]), 4);
            mbar_init(smem_addr(&b.o_full[t]), 1);
            mbar_init(smem_addr(&b.o_empty[t]), 4);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_addr(&b.kv_full[s]), 1);
            mbar_init(smem_addr(&b.kv_empty[s]), 1);
            mbar_init(smem_addr(&b.v_ready[s]), 2);
        }
        mbar_init(smem_addr(&b.drain), 1);
        b.abort = 0;
        if (p.streamk) {
            const long long lo = sk_lo(p.W, p.grid, blockIdx.x);
            const long long h0 = lo / p.F;
            b.sk_h0 = static_cast<int>(h0);
            b.sk_j0 = static_cast<int>(lo - h0 * p.F);
            b.sk_slot0 = static_cast<int>(blockIdx.x) - sk_cta(p.W, p.grid, h0 * p.F);
            b.sk_hi = sk_lo(p.W, p.grid, blockIdx.x + 1);
        }
        fence_barrier_init();
    }
    if constexpr (C::kOnes)
        init_ones_atom(smem_raw + (smem_base - raw) + C::kOnesOffset);
    if (warp == kWarpMma) {
        tmem_alloc(smem_addr(&b.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpLoad && lane == 0) {
        prefetch_tensormap(&mq);
        prefetch_tensormap(&mk);
        prefetch_tensormap(&mv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem_base;

    if (warp < 8) {
        run_softmax<D, kPrec>(p, b, tmem, warp / 4);
    } else if (warp == kWarpLoad) {
        run_load<D>(p, b, smem_base, &mq, &mk, &mv);
    } else if (warp == kWarpMma) {
        run_mma<D, kPrec>(p, b, smem_base, tmem);
    } else if constexpr (C::kConv) {
        run_convert<D, kPrec>(p, b, smem_raw + (smem_base - raw), warp - kWarpConv);
    }
    // The merge kernel of a split call (launched with programmatic stream
    // serialisation) may be scheduled now; it still waits for this grid to
    // finish before it reads the partials.
    grid_launch_dependents();

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ single tile
// d = 256: a 128-row Q tile and its 256-column O accumulator leave TMEM room
// for one Q tile per CTA, so the overlap comes from two S buffers instead of
// two Q tiles: S(j+1) is computed into the other buffer while the softmax
// works on S(j), and the tensor cores run P V(j) and S(j+2) once P(j) is
// written.  TMEM: S buffers at columns 0 and 128, O at 256..511.  Roles: warps
// 0-3 softmax (thread r owns row r), warp 4 TMA, warp 5 MMA.  K/V ring of two
// 64 KB stages, filled in the order the MMAs consume it: K0, K1, then V(i)
// and K(i+2) alternately, each stage in two 32 KB halves (Cfg::kHalves).
constexpr int kSingleWarpLoad = 4;
constexpr int kSingleWarpMma = 5;
constexpr int kSingleWarpConv = 6;  // and 7 (kPrecBf16)

template <int D>
__device__ void run_load_single(const Params &p, Bars &b, uint32_t smem_base,
                                const CUtensorMap *mq, const CUtensorMap *mk,
                                const CUtensorMap *mv)
{
    using C = Cfg<D>;
    const volatile int *abort = &b.abort;
    const bool leader = elect_one();
    uint32_t q_phase = 0, pos = 0;
    int last_q_parity = -1;
    bool ok = true;
    // K and V share the two stages irregularly (K_0, K_1, then V_i and
    // K_(i+2) alternately), so K copies complete on kv_full and V copies on
    // v_full: each barrier then sees only its own tiles, in order, and the
    // next phase's parity is kept per half-stage slot (2 * stage + half) and
    // barrier.  A K half is two of the tile's 128-row boxes (d-columns
    // 128h..128h+127); a V half is four 64-row boxes (keys 64h..64h+63, the
    // V tensor map's box is 64 rows) stored 8 KB apart.
    static_assert(C::kHalves == 2 && C::kChunks == 4, "one-tile kernel: d = 256");
    uint32_t kbits = 0, vbits = 0, last_v = 0, used = 0;
    grid_dependency_wait();  // see run_load
    auto load_tile = [&](const CUtensorMap *m, int row, int hh, int bb, bool is_v) {
        const uint32_t stage = pos % C::kStages;
        const uint32_t dst = smem_base + (C::kQTiles + stage) * C::kTileBytes;
        for (int h = 0; h < 2; ++h) {
            const uint32_t slot = 2 * stage + h;
            ok = warp_wait(smem_addr(&b.kv_empty[slot]), ((pos / C::kStages) & 1) ^ 1, abort);
            if (!ok)
                return;
            if (leader) {
                const uint32_t full = smem_addr(is_v ? &b.v_full[slot] : &b.kv_full[slot]);
                mbar_arrive_expect_tx(full, C::kHalfBytes);
                if (is_v) {
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_4d(dst + h * C::kHalfBytes + c * (kChunkBytes / 2), m, full,
                                    64 * c, row + 64 * h, hh, bb);
                } else {
#pragma unroll
                    for (int c = 2 * h; c < 2 * h + 2; ++c)
                        tma_load_4d(dst + c * kChunkBytes, m, full, 64 * c, row, hh, bb);
                }
            }
            const uint32_t bit = 1u << slot;
            if (is_v) {
                vbits ^= bit;
                last_v |= bit;
            } else {
                kbits ^= bit;
                last_v &= ~bit;
            }
            used |= bit;
        }
        ++pos;
    };
    for (int r = 0; ok; ++r) {
        Unit u;
        if (!cta_unit(p, b, r, u))
            break;
        const int n = u.n[0];
        if (n == 0)
            continue;
        const int hh = u.bh % p.H, bb = u.bh / p.H;
        if (!warp_wait(smem_addr(&b.q_empty[0]), q_phase ^ 1, abort)) {
            ok = false;
            break;
        }
        if (leader) {
            const uint32_t full = smem_addr(&b.q_full[0]);
            mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_4d(smem_base + c * kChunkBytes, mq, full, 64 * c, u.qt[0] * kBM, hh, bb);
        }
        last_q_parity = q_phase;
        q_phase ^= 1;
        load_tile(mk, u.j0 * kBN, hh, bb, false);
        if (ok && n > 1)
            load_tile(mk, (u.j0 + 1) * kBN, hh, bb, false);
        for (int i = 0; ok && i < n; ++i) {
            load_tile(mv, (u.j0 + i) * kBN, hh, bb, true);
            if (ok && i + 2 < n)
                load_tile(mk, (u.j0 + i + 2) * kBN, hh, bb, false);
        }
    }
    if (!ok) {
        if (leader)
            record_failure(b, kRoleLoad);
        // Let the copies already issued land before the CTA exits: only the
        // last copy into each half-stage slot can still be in flight.
        for (int st = 0; st < 2 * C::kStages; ++st) {
            const uint32_t bit = 1u << st;
            if (!(used & bit))
                continue;
            if (last_v & bit)
                mbar_wait(smem_addr(&b.v_full[st]), ((vbits & bit) ? 0u : 1u), kWaitLimitNs / 8,
                          nullptr);
            else
                mbar_wait(smem_addr(&b.kv_full[st]), ((kbits & bit) ? 0u : 1u), kWaitLimitNs / 8,
                          nullptr);
        }
        if (last_q_parity >= 0)
            mbar_wait(smem_addr(&b.q_full[0]), last_q_parity, kWaitLimitNs / 8, nullptr);
    }
}

template <int D, int kPrec>
__device__ void run_mma_single(const Params &p, Bars &b, uint32_t smem_base, uint32_t tmem)
{
    using C = Cfg<D, kPrec>;
    const volatile int *abort = &b.abort;
    const bool leader = elect_one();
    uint32_t q_phase = 0, oe_phase = 0, p_phase[2] = {0, 0}, pos = 0;
    bool ok = true;
    auto commit = [&](uint64_t &bar) {
        if (leader)
            mma_commit(smem_addr(&bar));
    };
    // The next ring position: its stage and shared-memory address, and the
    // parity of its fill.  Its two halves complete separately (see
    // run_load_single): K halves on kv_full, V halves on v_full, or with
    // converter warps on v_ready once converted; both halves of a stage
    // share one phase bit per barrier kind.
    uint32_t kbits = 0, vbits = 0;
    uint32_t fill_parity = 0;
    bool fill_v = false;
    auto next_tile = [&](uint32_t &addr, bool is_v = false) {
        const uint32_t stage = pos % C::kStages;
        const uint32_t bit = 1u << stage;
        fill_v = is_v;
        if (is_v) {
            fill_parity = (vbits & bit) ? 1u : 0u;
            vbits ^= bit;
        } else {
            fill_parity = (kbits & bit) ? 1u : 0u;
            kbits ^= bit;
        }
        addr = smem_base + (C::kQTiles + stage) * C::kTileBytes;
        return stage;
    };
    // Waits for half h of the position next_tile returned last.
    auto wait_half = [&](uint32_t stage, int h) {
        const uint32_t slot = 2 * stage + h;
        const uint32_t bar = smem_addr(!fill_v ? &b.kv_full[slot]
                                               : (C::kConv ? &b.v_ready[slot] : &b.v_full[slot]));
        ok = warp_wait(bar, fill_parity, abort);
        return ok;
    };
    for (int r = 0; ok; ++r) {
        Unit u;
        if (!cta_unit(p, b, r, u))
            break;
        const int n = u.n[0];
        if (n == 0)
            continue;
        ok = warp_wait(smem_addr(&b.q_full[0]), q_phase, abort);
        q_phase ^= 1;
        if (!ok)
            break;
        // S over one K tile into S buffer buf, a half of the tile at a time:
        // each half of the stage is freed once the products reading it are
        // done.
        auto s_product = [&](uint32_t buf, uint32_t k_addr, uint32_t stage) {
            if (!wait_half(stage, 0))
                return;
            tc_fence_after();
            if (leader)
                issue_s<D, kPrec, 0, D / 32>(tmem + buf * 128u, smem_base, k_addr);
            commit(b.kv_empty[2 * stage]);
            if (!wait_half(stage, 1))
                return;
            tc_fence_after();
            if (leader)
                issue_s<D, kPrec, D / 32, D / 16>(tmem + buf * 128u, smem_base, k_addr);
            commit(b.s_full[buf]);
            commit(b.kv_empty[2 * stage + 1]);
        };
        // S(0) and S(1) into the two buffers.
        for (int i = 0; i < 2 && i < n && ok; ++i) {
            uint32_t k_addr;
            const uint32_t stage = next_tile(k_addr);
            s_product(i, k_addr, stage);
            if (!ok)
                break;
            ++pos;
            if (i == n - 1)
                commit(b.q_empty[0]);
        }
        for (int i = 0; i < n && ok; ++i) {
            const int buf = i & 1;
            ok = warp_wait(smem_addr(&b.p_full[buf]), p_phase[buf], abort);
            p_phase[buf] ^= 1;
            if (ok && i == 0) {  // the first P V of the unit overwrites O
                ok = warp_wait(smem_addr(&b.o_empty[0]), oe_phase ^ 1, abort);
                oe_phase ^= 1;
            }
            if (!ok)
                break;
            uint32_t v_addr = 0;
            const uint32_t stage = next_tile(v_addr, true);
            // P V(i), keys 0-63 then 64-127, each half of V freed after its
            // products.
            if (!wait_half(stage, 0))
                break;
            tc_fence_after();
            if (leader)
                issue_pv<D, kPrec, 0, kBN / 32>(tmem + C::kColO0, tmem + buf * 128u, v_addr,
                                                smem_base + C::kOnesOffset, i > 0);
            commit(b.kv_empty[2 * stage]);
            if (!wait_half(stage, 1))
                break;
            tc_fence_after();
            if (leader)
                issue_pv<D, kPrec, kBN / 32, kBN / 16>(tmem + C::kColO0, tmem + buf * 128u,
                                                      v_addr, smem_base + C::kOnesOffset, true);
            commit(b.pv_done);
            commit(b.kv_empty[2 * stage + 1]);
            ++pos;
            if (i + 2 < n) {  // S(i+2) into the buffer P V(i) has just read
                uint32_t k_addr;
                const uint32_t ks = next_tile(k_addr);
                s_product(buf, k_addr, ks);
                if (!ok)
                    break;
                ++pos;
                if (i + 2 == n - 1)
                    commit(b.q_empty[0]);
            }
        }
        if (ok)
            commit(b.o_full[0]);
    }
    if (!ok && leader)
        record_failure(b, kRoleMma);
    // Wait until every MMA this warp issued has completed.
    commit(b.drain);
    mbar_wait(smem_addr(&b.drain), 0, kWaitLimitNs, nullptr);
}

template <int D, int kPrec>
__device__ void run_softmax_single(const Params &p, Bars &b, uint32_t tmem)
{
    using C = Cfg<D, kPrec>;
    const volatile int *abort = &b.abort;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int r = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t t_o = tmem + lane_off + C::kColO0;
    uint32_t s_phase[2] = {0, 0}, of_phase = 0, pv_count = 0;
    bool ok = true;

    for (int rr = 0; ok; ++rr) {
        Unit u;
        if (!cta_unit(p, b, rr, u))
            break;
        if (u.n[0] == 0)
            continue;
        const int qt = u.qt[0];
        const int row = qt * kBM + r;
        float m = -FLT_MAX, l = 0.f, l_round = 0.f;  // -FLT_MAX: see run_softmax
        int first_vis = qt * kBM + p.off - u.j0 * kBN;
        for (int j = u.j0; j < u.j1[0]; ++j, first_vis -= kBN) {
            const bool first = j == u.j0;
            const int buf = (j - u.j0) & 1;
            ok = mbar_wait(smem_addr(&b.s_full[buf]), s_phase[buf], kWaitLimitNs, abort);
            s_phase[buf] ^= 1;
            if (!ok)
                break;
            tc_fence_after();
            __syncwarp();
            float m_new;
            const float alpha = softmax_tile<D, kPrec, C::kOnes>(p, tmem + lane_off + buf * 128u, r,
                                                                j, first_vis, first, m, m_new, l,
                                                                l_round);
            if (!first && __any_sync(0xffffffffu, m_new != m)) {
                // O may still be receiving P V of the previous key tile: wait
                // for that product (the pv_count-th P V of this CTA) first.
                ok = mbar_wait(smem_addr(&b.pv_done), (pv_count - 1) & 1, kWaitLimitNs, abort);
                if (!ok)
                    break;
                tc_fence_after();
                rescale_o<D, C::kOnes>(t_o, alpha);
            }
            m = m_new;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&b.p_full[buf]));
            ++pv_count;
        }
        if (!ok)
            break;
        ok = mbar_wait(smem_addr(&b.o_full[0]), of_phase, kWaitLimitNs, abort);
        of_phase ^= 1;
        if (!ok)
            break;
        tc_fence_after();
        epilogue_row<D, kPrec, C::kOnes>(p, u, t_o, row, m, l, l_round);
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&b.o_empty[0]));
    }
    if (!ok)
        record_failure(b, kRoleSoftmax);
}

template <int D, int kPrec>
__global__ void __launch_bounds__(Cfg<D, kPrec>::kThreads, 1)
    fwd_single_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv, const Params p)
{
    using C = Cfg<D, kPrec>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t smem_base = (raw + 1023u) & ~1023u;
    Bars &b = *reinterpret_cast<Bars *>(smem_raw + (smem_base - raw) + C::kBarsOffset);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_addr(&b.q_full[t]), 1);
            mbar_init(smem_addr(&b.q_empty[t]), 1);
            mbar_init(smem_addr(&b.s_full[t]), 1);
            mbar_init(smem_addr(&b.p_full[t]), 4);
            mbar_init(smem_addr(&b.o_full[t]), 1);
            mbar_init(smem_addr(&b.o_empty[t]), 4);
        }
        for (int s = 0; s < 2 * C::kStages; ++s) {  // two half-stage slots a stage
            mbar_init(smem_addr(&b.kv_full[s]), 1);
            mbar_init(smem_addr(&b.kv_empty[s]), 1);
            mbar_init(smem_addr(&b.v_ready[s]), 2);
            mbar_init(smem_addr(&b.v_full[s]), 1);
        }
        mbar_init(smem_addr(&b.drain), 1);
        mbar_init(smem_addr(&b.pv_done), 1);
        b.abort = 0;
        if (p.streamk) {
            const long long lo = sk_lo(p.W, p.grid, blockIdx.x);
            const long long h0 = lo / p.F;
            b.sk_h0 = static_cast<int>(h0);
            b.sk_j0 = static_cast<int>(lo - h0 * p.F);
            b.sk_slot0 = static_cast<int>(blockIdx.x) - sk_cta(p.W, p.grid, h0 * p.F);
            b.sk_hi = sk_lo(p.W, p.grid, blockIdx.x + 1);
        }
        fence_barrier_init();
    }
    if constexpr (C::kOnes)
        init_ones_atom(smem_raw + (smem_base - raw) + C::kOnesOffset);
    if (warp == kSingleWarpMma) {
        tmem_alloc(smem_addr(&b.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kSingleWarpLoad && lane == 0) {
        prefetch_tensormap(&mq);
        prefetch_tensormap(&mk);
        prefetch_tensormap(&mv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem_base;

    if (warp < 4)
        run_softmax_single<D, kPrec>(p, b, tmem);
    else if (warp == kSingleWarpLoad)
        run_load_single<D>(p, b, smem_base, &mq, &mk, &mv);
    else if (warp == kSingleWarpMma)
        run_mma_single<D, kPrec>(p, b, smem_base, tmem);
    else if constexpr (C::kConv)
        run_convert<D, kPrec>(p, b, smem_raw + (smem_base - raw), warp - kSingleWarpConv);
    grid_launch_dependents();  // see fwd_kernel

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kSingleWarpMma) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ combine
// Merge of the key-range splits of each row (the blocked softmax statistics
// merge: per-block maxima and sums combined into the global ones).  With
// base-2 partial log-sum-exps le_s (of the exact sums l) and lr_s (of the
// normalisers l_round) and partial outputs O_s = acc_s / l_round_s:
//   lse = ln2 * log2(sum_s 2^le_s)
//   O   = sum_s w_s O_s,  w_s = 2^lr_s / sum_s' 2^lr_s'
// Slots with no key tile for the row's Q tile are skipped (the same ranges
// as unit_at / cta_unit).  One warp per row; lane l owns D/32 consecutive
// columns.  Blocks of four rows: with the registers a batch of eight slots
// needs, 128-thread blocks fill the SMs' warp slots where 256-thread ones
// left a partial second wave.
//
// Key-tile range [j0, je) of partial slot sp of head bh's pair (false: no
// such slot).
__device__ __forceinline__ bool slot_range(const Params &p, int bh, int fmax, int sp, int &j0,
                                           int &je)
{
    if (!p.streamk) {
        j0 = sp * fmax / p.splits;
        je = (sp + 1) * fmax / p.splits;
        return sp < p.splits;
    }
    const long long x = static_cast<long long>(bh) * p.F;
    const long long c = sk_cta(p.W, p.grid, x) + sp;
    if (c >= p.grid)
        return false;
    const long long lo = sk_lo(p.W, p.grid, c);
    if (lo >= x + p.F)
        return false;
    j0 = static_cast<int>(max(lo - x, 0LL));
    je = static_cast<int>(min(sk_lo(p.W, p.grid, c + 1) - x, static_cast<long long>(p.F)));
    return true;
}

template <int D, int kPrec>
__global__ void __launch_bounds__(128)
    combine_kernel(const float *__restrict__ ws_o, const float2 *__restrict__ ws_l, const Params p)
{
    constexpr int kCols = D / 32;
    constexpr bool kOutF16 = Cfg<D, kPrec>::kInF16;
    const long long row = static_cast<long long>(blockIdx.x) * 4 + threadIdx.x / 32;
    const long long rows = static_cast<long long>(p.BH) * p.Nq;
    if (row >= rows)
        return;
    const int lane = threadIdx.x & 31;
    int bh, i;
    if (rows <= 0x7fffffffLL) {  // 32-bit division
        const uint32_t r32 = static_cast<uint32_t>(row), nq = static_cast<uint32_t>(p.Nq);
        bh = static_cast<int>(r32 / nq);
        i = static_cast<int>(r32 - static_cast<uint32_t>(bh) * nq);
    } else {
        bh = static_cast<int>(row / p.Nq);
        i = static_cast<int>(row % p.Nq);
    }
    const int qt = i / kBM, pair = p.single ? qt : qt / 2;
    const int fmax = unit_tiles(p, pair), fown = key_tiles(p, qt);
    // Launched as a programmatic dependent of the forward grid: wait for it
    // to finish (and its partials to be visible) before reading them.
    grid_dependency_wait();
    // Online merge over the slots in slot order.  The slots' key ranges depend
    // only on the row's Q tile: each lane works out one slot of a group of 32,
    // and a ballot gives the group's slots that hold keys of this row; only
    // those are read, kBatch loads issued before any of them is used.  A slot
    // whose range held no key of this row (l = 0, partial lse -inf, possible
    // in the decode shape) contributes nothing.
    constexpr int kBatch = 8;
    float mx_e = -INFINITY, mx_r = -INFINITY, se = 0.f, sr = 0.f;
    float acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c)
        acc[c] = 0.f;
    for (int sg = 0;; sg += 32) {
        int j0 = 0, je = 0;
        const bool exists = slot_range(p, bh, fmax, sg + lane, j0, je);
        unsigned live = __ballot_sync(0xffffffffu, exists && min(je, fown) > j0);
        // Slots exist up to a count, so a group with a missing slot is the last.
        const bool last = __ballot_sync(0xffffffffu, exists) != 0xffffffffu;
        while (live != 0) {
            float2 ll[kBatch];
            float o[kBatch][kCols];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                ll[u] = make_float2(-INFINITY, -INFINITY);
                if (live != 0) {
                    const int sp = sg + __ffs(live) - 1;
                    live &= live - 1;
                    const size_t srow = static_cast<size_t>(sp) * rows + row;
                    ll[u] = ws_l[srow];
                    const float *src = ws_o + srow * D + lane * kCols;
#pragma unroll
                    for (int c = 0; c < kCols; ++c)
                        o[u][c] = src[c];
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (ll[u].x == -INFINITY)
                    continue;
                const float ne = fmaxf(mx_e, ll[u].x), nr = fmaxf(mx_r, ll[u].y);
                se = se * ex2(mx_e - ne) + ex2(ll[u].x - ne);
                const float a = ex2(mx_r - nr), w = ex2(ll[u].y - nr);
                sr = sr * a + w;
#pragma unroll
                for (int c = 0; c < kCols; ++c)
                    acc[c] = fmaf(w, o[u][c], acc[c] * a);
                mx_e = ne;
                mx_r = nr;
            }
        }
        if (last)
            break;
    }
    const float inv = 1.f / sr;
    uint16_t *dst = static_cast<uint16_t *>(p.o) + (bh / p.H) * p.o_sb + (bh % p.H) * p.o_sh +
                    static_cast<long long>(i) * p.o_sn + lane * kCols;
    if constexpr (kCols % 2 == 0) {
#pragma unroll
        for (int c = 0; c < kCols; c += 2)
            *reinterpret_cast<uint32_t *>(dst + c) = pack2<kOutF16>(acc[c] * inv, acc[c + 1] * inv);
    } else {  // d = 96: three columns per lane, stored one by one
#pragma unroll
        for (int c = 0; c < kCols; ++c)
            dst[c] = static_cast<uint16_t>(pack2<kOutF16>(acc[c] * inv, 0.f) & 0xffffu);
    }
    if (lane == 0)
        p.lse[row] = (mx_e + log2f(se)) * kLn2;
}

// ------------------------------------------------------------------ V pre-pass
// kPrecBf16V16: V rounded from bf16 to fp16 once, into a contiguous
// [B][H][Nk][d] buffer that the forward grid's V tensor map reads, instead of
// once per work unit in shared memory.  The rounding is bf16x2_to_f16x2, the
// converter warps' own, so both routes give the same bits.  One 16-byte
// granule (8 elements) per step and kVBatch steps in flight per thread, over
// a single wave of CTAs; the grid lets the forward grid launch at once
// (programmatic dependent launch), whose load warp waits for these writes in
// griddepcontrol.wait before its first copy.
struct VConv {
    const uint4 *src;  // the caller's V
    uint4 *dst;        // fp16 copy, contiguous
    long long granules;          // B * H * Nk * d / 8
    long long sb, sh, sn;        // strides of src (batch, head, row) in granules
    int gpr;                     // granules per row, d / 8
    int H, Nk;
    int dense;                   // 1: src is contiguous as well
};
constexpr int kVBatch = 8;
constexpr int kVThreads = 256;
constexpr int kVBlocksPerSm = 2;

__device__ __forceinline__ long long v_src_index(const VConv &c, long long g)
{
    if (c.dense)
        return g;
    const long long row = g / c.gpr;
    const long long col = g - row * c.gpr;
    const long long bh = row / c.Nk;
    const long long n = row - bh * c.Nk;
    const long long b = bh / c.H;
    return b * c.sb + (bh - b * c.H) * c.sh + n * c.sn + col;
}

__global__ void __launch_bounds__(kVThreads) v_to_f16_kernel(VConv c)
{
    grid_launch_dependents();
    const long long stride = static_cast<long long>(gridDim.x) * kVThreads;
    for (long long base = static_cast<long long>(blockIdx.x) * kVThreads + threadIdx.x;
         base < c.granules; base += stride * kVBatch) {
        uint4 w[kVBatch];
#pragma unroll
        for (int i = 0; i < kVBatch; ++i) {
            const long long g = base + i * stride;
            if (g < c.granules)
                w[i] = __ldcs(c.src + v_src_index(c, g));
        }
#pragma unroll
        for (int i = 0; i < kVBatch; ++i) {
            const long long g = base + i * stride;
            if (g < c.granules)
                c.dst[g] = bf16x8_to_f16x8(w[i]);
        }
    }
}

template <int D, int kPrec>
cudaError_t launch(const FwdArgs &a, const FwdMaps &maps, const FwdSplit &split, int num_sms,
                   cudaStream_t stream)
{
    using C = Cfg<D, kPrec>;
    Params p;
    p.o = a.o;
    p.lse = a.lse;
    p.ws_o = split.ws_o;
    p.ws_l = reinterpret_cast<float2 *>(split.ws_l);
    p.Nq = a.N;
    p.Nk = a.Nk;
    p.off = a.Nk - a.N;
    p.extra = p.off > 0 ? (p.off + kBN - 1) / kBN : 0;
    p.BH = a.B * a.H;
    p.H = a.H;
    const bool dense_o = a.o_sb == 0 && a.o_sh == 0 && a.o_sn == 0;
    p.o_sn = dense_o ? D : a.o_sn;
    p.o_sh = dense_o ? static_cast<long long>(a.N) * D : a.o_sh;
    p.o_sb = dense_o ? static_cast<long long>(a.H) * a.N * D : a.o_sb;
    p.QT = (a.N + kBM - 1) / kBM;
    p.KT = (a.Nk + kBN - 1) / kBN;
    p.single = D == 256 ? 1 : 0;
    p.pairs = p.single ? p.QT : (p.QT + 1) / 2;
    p.splits = split.splits < 1 ? 1 : split.splits;
    p.causal = a.causal;
    p.streamk = split.streamk;
    long long units = static_cast<long long>(p.BH) * p.pairs * p.splits;
    if (p.streamk) {
        if (p.pairs != 1 || p.splits < 2)
            return cudaErrorInvalidValue;
        p.F = max(key_tiles(p.QT, p.KT, p.extra, p.causal, 0),
                  key_tiles(p.QT, p.KT, p.extra, p.causal, 1));
        p.W = static_cast<long long>(p.BH) * p.F;
        units = p.W;
    }
    if (units == 0)
        return cudaSuccess;
    if (!p.streamk && units > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    p.units = static_cast<int>(min(units, 0x7fffffffLL));
    p.sl2 = a.scale * kLog2e;
    const size_t smem = C::kBarsOffset + sizeof(Bars) + 1024;
    cudaError_t e;
    if constexpr (D == 256)
        e = cudaFuncSetAttribute(fwd_single_kernel<D, kPrec>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
    else
        e = cudaFuncSetAttribute(fwd_kernel<D, kPrec>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    const int grid = static_cast<int>(units < num_sms ? units : num_sms);
    p.grid = grid;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    if constexpr (kPrec == kPrecBf16V16) {
        VConv c;
        c.src = static_cast<const uint4 *>(a.v);
        c.dst = static_cast<uint4 *>(a.v16);
        c.gpr = D / 8;
        c.granules = static_cast<long long>(p.BH) * a.Nk * c.gpr;
        c.H = a.H;
        c.Nk = a.Nk;
        c.sb = a.v_sb / 8;
        c.sh = a.v_sh / 8;
        c.sn = a.v_sn / 8;
        c.dense = a.v_sn == D && a.v_sh == static_cast<long long>(a.Nk) * D &&
                  (a.B == 1 || a.v_sb == static_cast<long long>(a.H) * a.Nk * D);
        const long long want = (c.granules + kVThreads - 1) / kVThreads;
        const long long cap = static_cast<long long>(num_sms) * kVBlocksPerSm;
        v_to_f16_kernel<<<static_cast<unsigned>(want < cap ? want : cap), kVThreads, 0,
                          stream>>>(c);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    cudaLaunchConfig_t fcfg = {};
    fcfg.gridDim = dim3(static_cast<unsigned>(grid));
    fcfg.blockDim = dim3(C::kThreads);
    fcfg.dynamicSmemBytes = smem;
    fcfg.stream = stream;
    fcfg.attrs = pdl;
    fcfg.numAttrs = kPrec == kPrecBf16V16 ? 1 : 0;
    if constexpr (D == 256)
        e = cudaLaunchKernelEx(&fcfg, fwd_single_kernel<D, kPrec>, maps.q, maps.k, maps.v, p);
    else
        e = cudaLaunchKernelEx(&fcfg, fwd_kernel<D, kPrec>, maps.q, maps.k, maps.v, p);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess || p.splits == 1)
        return e;
    const long long rows = static_cast<long long>(p.BH) * p.Nq;
    const long long blocks = (rows + 3) / 4;
    if (blocks > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    // Programmatic dependent launch: the merge grid is set up while the
    // forward grid drains and waits for it in griddepcontrol.wait.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel<D, kPrec>, static_cast<const float *>(p.ws_o),
                              static_cast<const float2 *>(p.ws_l), p);
}

}  // namespace

FwdPlan plan_fwd_streamk(int B, int H, int N, int Nk, int causal, int num_sms)
{
    const FwdPlan none{0, 0};
    // Only for one 128-row Q tile per head: with two, the pair's work per key
    // tile is twice the tensor work and the partial outputs, their merge and
    // the extra unit boundaries cost more than the idle SMs (measured: 256
    // queries x 16K keys x 128 heads, 1173 TFLOP/s stream-K against 1304
    // with whole heads).
    const int QT = (N + kBM - 1) / kBM, KT = (Nk + kBN - 1) / kBN;
    if (QT != 1 || num_sms < 1)
        return none;
    const int off = Nk - N;
    const int extra = off > 0 ? (off + kBN - 1) / kBN : 0;
    const long long F = max(key_tiles(QT, KT, extra, causal, 0), key_tiles(QT, KT, extra, causal, 1));
    const long long BH = static_cast<long long>(B) * H;
    const long long W = BH * F;
    // Whole heads per CTA already fill the SMs to within 3 %, or there are
    // fewer than two key tiles per SM: no stream-K.
    const long long rounds = (BH + num_sms - 1) / num_sms;
    if (BH * 100 >= rounds * num_sms * 97 || W < 2LL * num_sms)
        return none;
    // A head's F steps meet at most ceil(F / shortest range) + 1 ranges.
    const long long shortest = W / num_sms;
    const long long slots = (F + shortest - 1) / shortest + 1;
    return FwdPlan{1, static_cast<int>(slots)};
}

template <int D>
cudaError_t launch_prec(const FwdArgs &a, const FwdMaps &maps, const FwdSplit &split, int num_sms,
                        cudaStream_t stream)
{
    if (a.f16)
        return launch<D, kPrecF16>(a, maps, split, num_sms, stream);
    if (a.bf16p)
        return launch<D, kPrecBf16P>(a, maps, split, num_sms, stream);
    if (a.v16)
        return launch<D, kPrecBf16V16>(a, maps, split, num_sms, stream);
    return launch<D, kPrecBf16>(a, maps, split, num_sms, stream);
}

cudaError_t launch_fwd_sm103(const FwdArgs &a, const FwdMaps &maps, const FwdSplit &split,
                             int num_sms, cudaStream_t stream)
{
    switch (a.d) {
    case 64:
        return launch_prec<64>(a, maps, split, num_sms, stream);
    case 96:
        return launch_prec<96>(a, maps, split, num_sms, stream);
    case 128:
        return launch_prec<128>(a, maps, split, num_sms, stream);
    case 256:
        return launch_prec<256>(a, maps, split, num_sms, stream);
    }
    return cudaErrorInvalidValue;
}

namespace {

// Self-test of the failure path: one warp waits on an mbarrier that nothing
// ever arrives on, with the same bounded wait as the pipeline roles; when the
// limit passes it records a timeout in the status word and returns.
__global__ void selftest_wait_timeout_kernel(uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(smem_addr(&bar), 0, limit_ns, &abort_flag);
    if (!ok && threadIdx.x == 0) {
        const uint32_t code = 4u | (static_cast<uint32_t>(kRoleSelfTest) << 8) |
                              ((blockIdx.x & 0xffffu) << 16);
        atomicCAS(&g_fattn_status, 0u, code);
    }
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream)
{
    selftest_wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t status_word_address(uint32_t **out)
{
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_fattn_status);
    *out = static_cast<uint32_t *>(ptr);
    return e;
}

cudaError_t read_and_clear_status(uint32_t *out, cudaStream_t stream)
{
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fattn_status, sizeof(uint32_t), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess)
        return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return e;
    if (*out != 0) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbolAsync(g_fattn_status, &zero, sizeof(uint32_t), 0,
                                    cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace fattn
