// fattn_bwd_sm103.cu -- gradients of the attention forward pass on GB300.
//
// The backward that "OpenAI Triton: from introduction to model practice"
// (section 6) wraps around the forward, from the saved q, k, v, o and lse:
// the scores are recomputed, never stored.  With P = exp(scale*Q K^T - lse)
// (masked entries 0) and D_i = dO_i . O_i:
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,
//   dK = scale dS^T Q.
// Three kernels:
//   prep_kernel    D_i = dO_i . O_i into the caller's scratch (fp32).
//   dkdv_kernel    one CTA per 128-row key tile j (persistent, heaviest
//                  first): for every query tile i it computes S^T = K_j Q_i^T
//                  and dP^T = V_j dO_i^T on the tensor cores (keys on TMEM
//                  lanes); the elementwise threads form P^T in bf16 over S^T,
//                  then dS^T over dP^T, and the tensor cores accumulate
//                  dV_j += P^T dO_i and dK_j += dS^T Q_i in TMEM.
//   dq_kernel      one CTA per 128-row query tile i: for every key tile j,
//                  S = Q_i K_j^T and dP = dO_i V_j^T, one thread per query
//                  row forms dS in bf16, and dQ_i += dS K_j.
// S and dP are computed twice (once per kernel) so that neither kernel needs
// atomics or an fp32 dQ accumulator in memory.  The roles are those of the
// forward kernel: a TMA producer warp, a warp-converged MMA warp with one
// elected issuing lane, and two warpgroups for the elementwise work (thread r
// of warpgroup h owns TMEM lane r and columns 64h..64h+63: the pass has no
// row reduction, so the halves are independent), with every wait bounded.
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

#include "fattn_internal.h"
#include "ptx_sm103.cuh"

namespace fattn {
namespace {

using namespace ptx;

constexpr int kTile = 128;
constexpr int kThreads = 320;  // warps 0-7 elementwise, 8 producer, 9 MMA
constexpr int kElemWarps = 8;   // two warpgroups, one per half of the 128 columns
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kChunkBytes = kTile * 64 * 2;
constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256;

template <int D, bool kDkDv = true>
struct BCfg {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;  // one [128][D] bf16 tile
    // smem: two resident tiles, then
    //   dK/dV: a ring of two stages, each a (Q, dO) pair;
    //   dQ:    a ring of three K tiles and a separate ring of two V tiles
    //          (V is released as soon as dP has read it, K only after dQ).
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr uint32_t kKRing = 2 * kTileBytes;
    static constexpr uint32_t kVRing = kKRing + kKStages * kTileBytes;
    static constexpr uint32_t kTilesBytes =
        kDkDv ? 6 * kTileBytes : kVRing + kVStages * kTileBytes;
    static constexpr uint32_t kBarsBytes = 256;  // BBars, rounded up
    static constexpr uint32_t kColAcc1 = kColAcc0 + D;
    // dq kernel: a second S buffer in the columns after the dQ accumulator,
    // so that S of the next key tile is computed while the elementwise pass
    // works on this one.
    static constexpr uint32_t kColS1 = kColAcc0 + D;
};

// dq kernel: the S buffer of the i-th key tile of a unit.
template <int D>
__device__ __forceinline__ uint32_t dq_s_col(int i)
{
    return (i & 1) ? BCfg<D>::kColS1 : kColS;
}

struct BBars {
    uint64_t res_full, res_empty;  // the CTA's resident pair (K_j,V_j or Q_i,dO_i)
    uint64_t st_full[3], st_empty[3];  // dK/dV: Q stages; dQ: K stages
    uint64_t v_full[2], v_empty[2];    // dK/dV: dO stages; dQ: V stages
    uint64_t s_full, p_full, o_full, o_empty;
    // dkdv: P^T of the tile written (p_full then means dS^T written), and
    // dP^T of the tile computed (s_full then means S^T computed).
    uint64_t p1_full, dp_full;
    uint64_t dp_free;  // dq: the elementwise pass holds dP in registers
    // dq: dS of the CTA's n-th key tile written (all eight warps), on
    // dq_full[n % 2].  dP is released early (dp_free), so a warp can finish
    // tile n and write dS of tile n + 1 while another still writes dS of
    // tile n; one barrier would then complete tile n's phase with arrivals
    // of tile n + 1.  The skew is at most one tile (tile n + 2 needs dP of
    // n + 1 released by every warp), so two barriers keep the tiles apart.
    uint64_t dq_full[2];
    // dkdv: per warpgroup, its four warps have stored lse and D of the tile
    // (a bounded wait, unlike a hardware barrier, cannot hang if a warp has
    // left the loop after a timed-out wait).
    uint64_t grp[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

static_assert(sizeof(BBars) <= 256, "BBars outgrew its shared-memory slot");

// dK/dV kernel only (after BBars): -lse * log2(e) and -D of the current query
// tile's 128 rows, double-buffered.
struct BXch {
    float lse2[2][kTile];
    float dd[2][kTile];
};

struct BParams {
    const __nv_bfloat16 *o, *dout;
    const float *lse;
    float *dvec;  // D = rowsum(dO * O), fp32 [B*H*N]
    __nv_bfloat16 *g0, *g1;  // dkdv: dK, dV   dq: dQ, unused
    uint32_t *status;
    int N, BH, T;  // T = tiles per head
    int units;
    int causal;
    float scale, sl2;
};

__device__ __forceinline__ void fail(const BParams &p, BBars &b, uint32_t role)
{
    const uint32_t code = 4u | (role << 8) | ((blockIdx.x & 0xffffu) << 16);
    atomicCAS(p.status, 0u, code);
    *reinterpret_cast<volatile int *>(&b.abort) = 1;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort)
{
    const bool ok = mbar_wait(bar, parity, kWaitLimitNs, abort);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ int deal(int round, int cta, int grid)
{
    return round * grid + ((round & 1) ? grid - 1 - cta : cta);
}

// Tiles that interact with resident tile `own` (the loop range of the CTA):
// dkdv (key tile own): query tiles [causal ? own : 0, T); dq (query tile own):
// key tiles [0, causal ? own + 1 : T).
template <bool kDkDv>
__device__ __forceinline__ void loop_range(const BParams &p, int own, int &lo, int &hi)
{
    if (kDkDv) {
        lo = p.causal ? own : 0;
        hi = p.T;
    } else {
        lo = 0;
        hi = p.causal ? own + 1 : p.T;
    }
}

// Unit k -> (head, resident tile), heaviest first.
template <bool kDkDv>
__device__ __forceinline__ void unit_of(const BParams &p, int k, int &bh, int &own)
{
    bh = k % p.BH;
    own = kDkDv ? k / p.BH : p.T - 1 - k / p.BH;
}

// ------------------------------------------------------------------ MMA helpers
// [128 x D] x [128 x D]^T, both K-major 128-byte-swizzled tiles, into 128
// fp32 TMEM columns.
template <int D>
__device__ __forceinline__ void mma_nt(uint32_t tmem_d, uint32_t a_smem, uint32_t b_smem)
{
    constexpr uint32_t idesc = idesc_bf16_f32(kTile, kTile, false);
    constexpr uint32_t hi = smem_desc_hi(1024);
    const uint32_t a_lo = smem_desc_lo(a_smem, 16), b_lo = smem_desc_lo(b_smem, 16);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ss_w(tmem_d, a_lo + off, hi, b_lo + off, hi, idesc, kk > 0 ? 1u : 0u);
    }
}

// TMEM [128 x 128] (bf16 pairs) x smem tile [128 x D] (D contiguous, i.e.
// MN-major B) into D fp32 TMEM columns, with A in the interleaved TMEM layout
// of the elementwise pass: each 32-column chunk of the S (S^T) region holds
// 16 columns of one operand (part 0: P^T, or dS in the dQ kernel) then 16 of
// another (part 16: dS^T), i.e. K = 16 step kk of A sits at column
// 32*(kk/2) + part + 8*(kk%2).
template <int D>
__device__ __forceinline__ void mma_tn_il(uint32_t tmem_d, uint32_t tmem_a, uint32_t part,
                                          uint32_t b_smem, bool accumulate)
{
    constexpr uint32_t idesc = idesc_bf16_f32(kTile, D, true);
    constexpr uint32_t lbo = D == 128 ? kChunkBytes : 1024;
    constexpr uint32_t hi = smem_desc_hi(1024);
    const uint32_t b_lo = smem_desc_lo(b_smem, lbo);
    const uint32_t acc0 = accumulate ? 1u : 0u;
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
        mma_ts_w(tmem_d, tmem_a + 32 * (kk >> 1) + part + 8 * (kk & 1),
                 b_lo + ((kk * 16 * 128) >> 4), hi, idesc, kk > 0 ? 1u : acc0);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ------------------------------------------------------------------ roles
// Producer: the resident pair (A0, A1) once per unit, then the streamed pairs
// (B0, B1) of every tile of the loop range into a two-stage ring.
template <int D, bool kDkDv>
__device__ void bwd_load(const BParams &p, BBars &b, uint32_t smem, const CUtensorMap *ra0,
                         const CUtensorMap *ra1, const CUtensorMap *sb0, const CUtensorMap *sb1)
{
    using C = BCfg<D, kDkDv>;
    const volatile int *abort = &b.abort;
    const bool leader = elect_one();
    uint32_t res_phase = 0, kpos = 0, vpos = 0;
    bool ok = true;
    int res_issued = 0;
    for (int r = 0; ok; ++r) {
        const int k = deal(r, blockIdx.x, gridDim.x);
        if (k >= p.units)
            break;
        int bh, own, lo, hi;
        unit_of<kDkDv>(p, k, bh, own);
        loop_range<kDkDv>(p, own, lo, hi);
        if (!warp_wait(smem_addr(&b.res_empty), res_phase ^ 1, abort)) {
            ok = false;
            break;
        }
        res_phase ^= 1;
        if (leader) {
            const uint32_t full = smem_addr(&b.res_full);
            mbar_arrive_expect_tx(full, 2 * C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(smem + c * kChunkBytes, ra0, full, 64 * c, own * kTile, bh);
                tma_load_3d(smem + C::kTileBytes + c * kChunkBytes, ra1, full, 64 * c, own * kTile,
                            bh);
            }
        }
        ++res_issued;
        if constexpr (!kDkDv) {
            // K(t) into the three-stage K ring, V(t) into the two-stage V ring.
            for (int t = lo; ok && t < hi; ++t) {
                const uint32_t ks = kpos % C::kKStages, kph = (kpos / C::kKStages) & 1;
                const uint32_t vs = vpos % C::kVStages, vph = (vpos / C::kVStages) & 1;
                if (!warp_wait(smem_addr(&b.st_empty[ks]), kph ^ 1, abort)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    const uint32_t full = smem_addr(&b.st_full[ks]);
                    const uint32_t dst = smem + C::kKRing + ks * C::kTileBytes;
                    mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(dst + c * kChunkBytes, sb0, full, 64 * c, t * kTile, bh);
                }
                ++kpos;
                if (!warp_wait(smem_addr(&b.v_empty[vs]), vph ^ 1, abort)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    const uint32_t full = smem_addr(&b.v_full[vs]);
                    const uint32_t dst = smem + C::kVRing + vs * C::kTileBytes;
                    mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(dst + c * kChunkBytes, sb1, full, 64 * c, t * kTile, bh);
                }
                ++vpos;
            }
        } else {
            // Q(t) and dO(t) share a stage of the two-stage ring but are
            // released separately: dO after dV(t), Q after dK(t).  kpos and
            // vpos count the Q and dO tiles issued.
            for (int t = lo; ok && t < hi; ++t) {
                const uint32_t stage = kpos & 1, phase = (kpos >> 1) & 1;
                const uint32_t dst = smem + (2 + 2 * stage) * C::kTileBytes;
                // dO first: its slot is released (after dV) before Q's (after dK).
                if (!warp_wait(smem_addr(&b.v_empty[stage]), phase ^ 1, abort)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    const uint32_t full = smem_addr(&b.v_full[stage]);
                    mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(dst + C::kTileBytes + c * kChunkBytes, sb1, full, 64 * c,
                                    t * kTile, bh);
                }
                ++vpos;
                if (!warp_wait(smem_addr(&b.st_empty[stage]), phase ^ 1, abort)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    const uint32_t full = smem_addr(&b.st_full[stage]);
                    mbar_arrive_expect_tx(full, C::kTileBytes);
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(dst + c * kChunkBytes, sb0, full, 64 * c, t * kTile, bh);
                }
                ++kpos;
            }
        }
    }
    if (!ok) {
        if (leader)
            fail(p, b, kRoleLoad);
        // Let the copies already issued land before the CTA exits.
        if constexpr (kDkDv) {
            for (uint32_t q = kpos > 2 ? kpos - 2 : 0; q < kpos; ++q)
                mbar_wait(smem_addr(&b.st_full[q & 1]), (q >> 1) & 1, kWaitLimitNs / 8, nullptr);
            for (uint32_t q = vpos > 2 ? vpos - 2 : 0; q < vpos; ++q)
                mbar_wait(smem_addr(&b.v_full[q & 1]), (q >> 1) & 1, kWaitLimitNs / 8, nullptr);
        } else {
            for (uint32_t q = kpos > 3 ? kpos - 3 : 0; q < kpos; ++q)
                mbar_wait(smem_addr(&b.st_full[q % 3]), (q / 3) & 1, kWaitLimitNs / 8, nullptr);
            for (uint32_t q = vpos > 2 ? vpos - 2 : 0; q < vpos; ++q)
                mbar_wait(smem_addr(&b.v_full[q & 1]), (q >> 1) & 1, kWaitLimitNs / 8, nullptr);
        }
        if (res_issued > 0)
            mbar_wait(smem_addr(&b.res_full), res_phase ^ 1, kWaitLimitNs / 8, nullptr);
    }
}

// MMA issuer.  dkdv: S^T = K Q^T (cols 0-127), dP^T = V dO^T (128-255); then
// dV += P^T dO (acc0), dK += dS^T Q (acc1).  dq: S = Q K^T, dP = dO V^T; then
// dQ += dS K (acc0).
template <int D, bool kDkDv>
__device__ void bwd_mma(const BParams &p, BBars &b, uint32_t smem, uint32_t tmem)
{
    using C = BCfg<D, kDkDv>;
    const volatile int *abort = &b.abort;
    const bool leader = elect_one();
    uint32_t res_phase = 0, s_phase = 0, oe_phase = 0, dp_phase = 0, pos = 0;
    uint32_t n_tile = 0;  // dq: key tiles of this CTA so far (dq_full[n % 2])
    bool ok = true;
    auto commit = [&](uint64_t &bar) {
        if (leader)
            mma_commit(smem_addr(&bar));
    };
    const uint32_t a0 = smem, a1 = smem + C::kTileBytes;  // resident pair
    auto stage_smem = [&](uint32_t at) { return smem + (2 + 2 * (at & 1)) * C::kTileBytes; };
    for (int r = 0; ok; ++r) {
        const int k = deal(r, blockIdx.x, gridDim.x);
        if (k >= p.units)
            break;
        int bh, own, lo, hi;
        unit_of<kDkDv>(p, k, bh, own);
        loop_range<kDkDv>(p, own, lo, hi);
        ok = warp_wait(smem_addr(&b.res_full), res_phase, abort);
        res_phase ^= 1;
        if (ok)
            ok = warp_wait(smem_addr(&b.o_empty), oe_phase ^ 1, abort);
        oe_phase ^= 1;
        if (!ok)
            break;
        if constexpr (!kDkDv) {
            // dq: S(t+1) goes into the other S buffer before dS(t) is ready,
            // and dP(t+1) follows as soon as the elementwise pass of t holds
            // dP(t) in registers (dp_free); dQ += dS(t) K_t once dS(t) is
            // written.  K(t) sits in the
            // three-stage K ring until dQ(t), V(t) in the two-stage V ring
            // until dP(t).  Position pos is tile lo in both rings.
            if (hi <= lo)
                continue;
            auto k_tile = [&](int t) {
                const uint32_t at = pos + (t - lo);
                return smem + C::kKRing + (at % C::kKStages) * C::kTileBytes;
            };
            auto v_tile = [&](int t) {
                const uint32_t at = pos + (t - lo);
                return smem + C::kVRing + (at % C::kVStages) * C::kTileBytes;
            };
            auto wait_k = [&](int t) {
                const uint32_t at = pos + (t - lo);
                return warp_wait(smem_addr(&b.st_full[at % C::kKStages]), (at / C::kKStages) & 1,
                                 abort);
            };
            auto wait_v = [&](int t) {
                const uint32_t at = pos + (t - lo);
                return warp_wait(smem_addr(&b.v_full[at % C::kVStages]), (at / C::kVStages) & 1,
                                 abort);
            };
            auto release_v = [&](int t) { commit(b.v_empty[(pos + (t - lo)) % C::kVStages]); };
            ok = wait_k(lo) && wait_v(lo);
            if (!ok)
                break;
            tc_fence_after();
            if (leader) {
                mma_nt<D>(tmem + dq_s_col<D>(0), a0, k_tile(lo));  // S = Q K^T
                mma_nt<D>(tmem + kColDP, a1, v_tile(lo));          // dP = dO V^T
            }
            commit(b.s_full);
            release_v(lo);
            if (lo == hi - 1)
                commit(b.res_empty);
            for (int t = lo; ok && t < hi; ++t) {
                const bool next = t + 1 < hi;
                if (next) {
                    ok = wait_k(t + 1);
                    if (!ok)
                        break;
                    tc_fence_after();
                    if (leader)
                        mma_nt<D>(tmem + dq_s_col<D>(t + 1 - lo), a0, k_tile(t + 1));
                }
                if (next) {
                    ok = warp_wait(smem_addr(&b.dp_free), dp_phase, abort);
                    dp_phase ^= 1;
                }
                if (ok && next)
                    ok = wait_v(t + 1);
                if (!ok)
                    break;
                tc_fence_after();
                if (next) {
                    if (leader)
                        mma_nt<D>(tmem + kColDP, a1, v_tile(t + 1));
                    commit(b.s_full);
                    release_v(t + 1);
                    if (t + 1 == hi - 1)
                        commit(b.res_empty);  // resident pair no longer read
                }
                ok = warp_wait(smem_addr(&b.dq_full[n_tile & 1]), (n_tile >> 1) & 1, abort);
                ++n_tile;
                if (!ok)
                    break;
                tc_fence_after();
                if (leader)  // dQ += dS K (dS in the first 16 columns of each chunk)
                    mma_tn_il<D>(tmem + kColAcc0, tmem + dq_s_col<D>(t - lo), 0u, k_tile(t),
                                 t > lo);
                commit(b.st_empty[(pos + (t - lo)) % C::kKStages]);
                if (t == hi - 1)
                    commit(b.o_full);
            }
            pos += hi - lo;
        } else {
            // dkdv: the elementwise pass writes P^T(t) over the S^T columns
            // and then dS^T(t) over the dP^T columns (the first 16 of every
            // 32), so S^T(t+1) follows dV(t) and dP^T(t+1) follows dK(t): the
            // pass forms P^T of the next tile while dK(t) and dP^T(t+1) run.
            // dO(t) is released after dV(t), Q(t) after dK(t).
            if (hi <= lo)
                continue;
            auto wait_q = [&](int t) {
                const uint32_t at = pos + (t - lo);
                return warp_wait(smem_addr(&b.st_full[at & 1]), (at >> 1) & 1, abort);
            };
            auto wait_do = [&](int t) {
                const uint32_t at = pos + (t - lo);
                return warp_wait(smem_addr(&b.v_full[at & 1]), (at >> 1) & 1, abort);
            };
            ok = wait_q(lo);
            if (!ok)
                break;
            tc_fence_after();
            if (leader)
                mma_nt<D>(tmem + kColS, a0, stage_smem(pos));  // S^T = K Q^T
            commit(b.s_full);
            ok = wait_do(lo);
            if (!ok)
                break;
            tc_fence_after();
            if (leader)
                mma_nt<D>(tmem + kColDP, a1, stage_smem(pos) + C::kTileBytes);  // dP^T = V dO^T
            commit(b.dp_full);
            if (lo == hi - 1)
                commit(b.res_empty);
            for (int t = lo; ok && t < hi; ++t) {
                const uint32_t at = pos + (t - lo);
                const bool next = t + 1 < hi;
                const uint32_t q_t = stage_smem(at), do_t = q_t + C::kTileBytes;
                ok = warp_wait(smem_addr(&b.p1_full), dp_phase, abort);
                dp_phase ^= 1;
                if (!ok)
                    break;
                tc_fence_after();
                if (leader)  // dV += P^T dO
                    mma_tn_il<D>(tmem + kColAcc0, tmem + kColS, 0u, do_t, t > lo);
                commit(b.v_empty[at & 1]);
                if (next) {
                    ok = wait_q(t + 1);
                    if (!ok)
                        break;
                    tc_fence_after();
                    if (leader)
                        mma_nt<D>(tmem + kColS, a0, stage_smem(at + 1));  // S^T(t+1)
                    commit(b.s_full);
                }
                ok = warp_wait(smem_addr(&b.p_full), s_phase, abort);
                s_phase ^= 1;
                if (!ok)
                    break;
                tc_fence_after();
                if (leader)  // dK += dS^T Q
                    mma_tn_il<D>(tmem + C::kColAcc1, tmem + kColDP, 0u, q_t, t > lo);
                commit(b.st_empty[at & 1]);
                if (next) {
                    ok = wait_do(t + 1);
                    if (!ok)
                        break;
                    tc_fence_after();
                    if (leader)
                        mma_nt<D>(tmem + kColDP, a1, stage_smem(at + 1) + C::kTileBytes);
                    commit(b.dp_full);
                    if (t + 1 == hi - 1)
                        commit(b.res_empty);  // resident pair no longer read
                }
                if (t == hi - 1)
                    commit(b.o_full);
            }
            pos += hi - lo;
        }
    }
    if (!ok && leader)
        fail(p, b, kRoleMma);
    commit(b.drain);
    mbar_wait(smem_addr(&b.drain), 0, kWaitLimitNs, nullptr);
}

// Elementwise warpgroups: thread r of either owns TMEM lane r = row
// `own*128 + r` of the resident tile (a key in dkdv, a query in dq); warpgroup
// h handles columns 64h..64h+63 of that row (two 32-column chunks), and each
// chunk's results go back into that chunk's own columns.
template <int D, bool kDkDv>
__device__ void bwd_elem(const BParams &p, BBars &b, BXch &x, uint32_t tmem)
{
    using C = BCfg<D>;
    const volatile int *abort = &b.abort;
    const int warp = (threadIdx.x / 32) & 3, lane = threadIdx.x & 31;
    const int half = threadIdx.x / 128;  // this warpgroup's 64 columns
    const int r = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    constexpr int kHalfChunks = kTile / 64;  // 32-column chunks per half
    uint32_t s_phase = 0, of_phase = 0, dp_phase = 0, grp_phase = 0;
    uint32_t n_tile = 0;  // dq: key tiles of this CTA so far (dq_full[n % 2])
    int xbuf = 0;
    bool ok = true;
    for (int rr = 0; ok; ++rr) {
        const int k = deal(rr, blockIdx.x, gridDim.x);
        if (k >= p.units)
            break;
        int bh, own, lo, hi;
        unit_of<kDkDv>(p, k, bh, own);
        loop_range<kDkDv>(p, own, lo, hi);
        const int row = own * kTile + r;                    // this thread's row
        const size_t head = static_cast<size_t>(bh) * p.N;
        float my_lse2 = 0.f, my_d = 0.f;
        if (!kDkDv && row < p.N) {
            my_lse2 = p.lse[head + row] * kLog2e;
            my_d = p.dvec[head + row];
        }
        // dkdv: lse and D of this warpgroup's 64 queries of a tile (threads
        // 0-63 take lse, 64-127 take D), fetched one tile ahead so that the
        // global loads are in flight while the previous tile runs (nothing
        // uses the loaded value until the next tile: no arithmetic on it
        // here, which would wait for the load at once).
        const int xq = half * 64 + (r & 63);
        const float *xsrc = (r < 64 ? p.lse : p.dvec) + head;
        auto fetch = [&](int tt) {
            const int qrow = tt * kTile + xq;
            return qrow < p.N ? xsrc[qrow] : 0.f;
        };
        float xnext = (kDkDv && lo < hi) ? fetch(lo) : 0.f;
        for (int t = lo; ok && t < hi; ++t) {
            if (kDkDv) {
                // Shared through smem as -lse*log2e and -D (double-buffered;
                // an mbarrier of the warpgroup alone publishes them, so the
                // two warpgroups never wait for each other here).
                if (r < 64)
                    x.lse2[xbuf][xq] = -xnext * kLog2e;
                else
                    x.dd[xbuf][xq] = -xnext;
                if (t + 1 < hi)
                    xnext = fetch(t + 1);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&b.grp[half]));
                ok = mbar_wait(smem_addr(&b.grp[half]), grp_phase, kWaitLimitNs, abort);
                grp_phase ^= 1;
                if (!ok)
                    break;
            }
            ok = mbar_wait(smem_addr(&b.s_full), s_phase, kWaitLimitNs, abort);
            s_phase ^= 1;
            if (!ok)
                break;
            tc_fence_after();
            // Column c of this row pairs row `row` of the resident tile with
            // row t*128+c of the streamed one.  Valid: inside N and, under the
            // causal mask, query >= key.
            const int col0 = t * kTile;
            int c_lo = 0, c_hi = kTile - 1;  // valid columns [c_lo, c_hi]
            if (kDkDv) {
                if (p.causal && t == own)
                    c_lo = r;  // query t*128+c >= key own*128+r
            } else {
                if (p.causal && t == own)
                    c_hi = r;  // key t*128+c <= query own*128+r
            }
            c_hi = min(c_hi, p.N - 1 - col0);
            const uint32_t col_s = kDkDv ? kColS : dq_s_col<D>(t - lo);
            // Element mask only on the diagonal tile and the ragged last one
            // (the branch is uniform across the warp).
            const bool masked = (p.causal && t == own) || col0 + kTile > p.N;
            const uint64_t sl2x2 = f2_pack(p.sl2, p.sl2);
            const uint64_t row_nl2 = f2_pack(-my_lse2, -my_lse2), row_nd = f2_pack(-my_d, -my_d);
            // dq: 16 column pairs of one 32-column chunk: p = 2^(s*scale*log2e -
            // lse*log2e) and dS = p (dP - D) of this thread's query row, two
            // columns per packed instruction; returns dS packed to bf16 pairs
            // (and P, unused there).
            auto pairs = [&](int ch, const uint32_t *sr, const uint32_t *dr, uint32_t *pk,
                             uint32_t *dk, auto masked_tag) {
                constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = ch * 32 + 2 * i;
                    const uint64_t nl2 = row_nl2, nd = row_nd;
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])),
                                     sl2x2, nl2),
                              x0, x1);
                    float p0 = ex2(x0), p1 = ex2(x1);
                    if constexpr (kMasked) {
                        p0 = (c >= c_lo && c <= c_hi) ? p0 : 0.f;
                        p1 = (c + 1 >= c_lo && c + 1 <= c_hi) ? p1 : 0.f;
                    }
                    const uint64_t pp = f2_pack(p0, p1);
                    float d0, d1;
                    f2_unpack(f2_mul(pp, f2_add(f2_pack(__uint_as_float(dr[2 * i]),
                                                        __uint_as_float(dr[2 * i + 1])),
                                                nd)),
                              d0, d1);
                    pk[i] = pack2(p0, p1);
                    dk[i] = pack2(d0, d1);
                }
            };
            // The dK/dV kernel's two phases over one chunk: probs forms p (kept
            // as fp32) and P packed; grads forms dS = p (dP - D) packed.
            auto probs = [&](int ch, const uint32_t *sr, float *pf, uint32_t *pk,
                             auto masked_tag) {
                constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = ch * 32 + 2 * i;
                    const uint64_t nl2 = *reinterpret_cast<const uint64_t *>(&x.lse2[xbuf][c]);
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])),
                                     sl2x2, nl2),
                              x0, x1);
                    float p0 = ex2(x0), p1 = ex2(x1);
                    if constexpr (kMasked) {
                        p0 = (c >= c_lo && c <= c_hi) ? p0 : 0.f;
                        p1 = (c + 1 >= c_lo && c + 1 <= c_hi) ? p1 : 0.f;
                    }
                    pf[2 * i] = p0;
                    pf[2 * i + 1] = p1;
                    pk[i] = pack2(p0, p1);
                }
            };
            auto grads = [&](int ch, const float *pf, const uint32_t *dr, uint32_t *dk) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = ch * 32 + 2 * i;
                    const uint64_t nd = *reinterpret_cast<const uint64_t *>(&x.dd[xbuf][c]);
                    float d0, d1;
                    f2_unpack(f2_mul(f2_pack(pf[2 * i], pf[2 * i + 1]),
                                     f2_add(f2_pack(__uint_as_float(dr[2 * i]),
                                                    __uint_as_float(dr[2 * i + 1])),
                                            nd)),
                              d0, d1);
                    dk[i] = pack2(d0, d1);
                }
            };
            if constexpr (kDkDv) {
                // Phase 1: P^T of this half's chunks, kept in registers and
                // written over the first 16 columns of each S^T chunk; then
                // dV and S^T of the next tile may run.
                float pr[kHalfChunks][32];
#pragma unroll
                for (int hc = 0; hc < kHalfChunks; ++hc) {
                    const int ch = half * kHalfChunks + hc;
                    uint32_t sr[32], pk[16];
                    __syncwarp();
                    tmem_ld32(tmem + lane_off + kColS + ch * 32, sr);
                    tmem_wait_ld();
                    if (masked)
                        probs(ch, sr, pr[hc], pk, std::true_type{});
                    else
                        probs(ch, sr, pr[hc], pk, std::false_type{});
                    tmem_st16(tmem + lane_off + kColS + ch * 32, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&b.p1_full));
                // Phase 2: dS^T = P^T (dP^T - D) over the first 16 columns of
                // each of this half's dP^T chunks.
                ok = mbar_wait(smem_addr(&b.dp_full), dp_phase, kWaitLimitNs, abort);
                dp_phase ^= 1;
                if (!ok)
                    break;
                tc_fence_after();
#pragma unroll
                for (int hc = 0; hc < kHalfChunks; ++hc) {
                    const int ch = half * kHalfChunks + hc;
                    uint32_t dr[32], dk[16];
                    __syncwarp();
                    tmem_ld32(tmem + lane_off + kColDP + ch * 32, dr);
                    tmem_wait_ld();
                    grads(ch, pr[hc], dr, dk);
                    tmem_st16(tmem + lane_off + kColDP + ch * 32, dk);
                }
            } else {
                // This half of the dP row into registers first, so that dP of
                // the next key tile is computed meanwhile.
                uint32_t dr[kHalfChunks][32];
#pragma unroll
                for (int hc = 0; hc < kHalfChunks; ++hc)
                    tmem_ld32(tmem + lane_off + kColDP + (half * kHalfChunks + hc) * 32, dr[hc]);
                tmem_wait_ld();
                if (t + 1 < hi) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_addr(&b.dp_free));
                }
#pragma unroll
                for (int hc = 0; hc < kHalfChunks; ++hc) {
                    const int ch = half * kHalfChunks + hc;
                    uint32_t sr[32], pk[16], dk[16];
                    __syncwarp();
                    tmem_ld32(tmem + lane_off + col_s + ch * 32, sr);
                    tmem_wait_ld();
                    if (masked)
                        pairs(ch, sr, dr[hc], pk, dk, std::true_type{});
                    else
                        pairs(ch, sr, dr[hc], pk, dk, std::false_type{});
                    // dS over the first half of its own chunk of S (the
                    // other warpgroup may still be reading its chunks).
                    tmem_st16(tmem + lane_off + col_s + ch * 32, dk);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(kDkDv ? &b.p_full : &b.dq_full[n_tile & 1]));
            ++n_tile;
            xbuf ^= 1;
        }
        if (!ok)
            break;
        // Epilogue: the accumulators -> bf16 rows (dK and dQ times scale).
        ok = mbar_wait(smem_addr(&b.o_full), of_phase, kWaitLimitNs, abort);
        of_phase ^= 1;
        if (!ok)
            break;
        tc_fence_after();
        const bool live = row < p.N;
        {
            // dkdv: warpgroup 0 writes dV (acc0, unscaled) -> g1, warpgroup 1
            // dK (acc1) -> g0; dq: each warpgroup half of the columns of dQ.
            const int which = kDkDv ? half : 1;
            const uint32_t col = which == 0 ? kColAcc0 : (kDkDv ? C::kColAcc1 : kColAcc0);
            const float f = (kDkDv && which == 0) ? 1.f : p.scale;
            __nv_bfloat16 *dst = ((kDkDv && which == 0) ? p.g1 : p.g0) + (head + row) * D;
            const int c_begin = kDkDv ? 0 : half * (D / 64);
            const int c_end = kDkDv ? D / 32 : (half + 1) * (D / 64);
#pragma unroll 1
            for (int c = c_begin; c < c_end; ++c) {
                uint32_t o[32];
                __syncwarp();
                tmem_ld32(tmem + lane_off + col + c * 32, o);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack2(__uint_as_float(o[2 * i]) * f, __uint_as_float(o[2 * i + 1]) * f);
                if (live) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&b.o_empty));
    }
    if (!ok)
        fail(p, b, kRoleSoftmax);
}

template <int D, bool kDkDv>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap ra0, const __grid_constant__ CUtensorMap ra1,
               const __grid_constant__ CUtensorMap sb0, const __grid_constant__ CUtensorMap sb1,
               const BParams p)
{
    using C = BCfg<D, kDkDv>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t smem = (raw + 1023u) & ~1023u;
    BBars &b = *reinterpret_cast<BBars *>(smem_raw + (smem - raw) + C::kTilesBytes);
    BXch &xch = *reinterpret_cast<BXch *>(smem_raw + (smem - raw) + C::kTilesBytes +
                                          C::kBarsBytes);
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&b.res_full), 1);
        mbar_init(smem_addr(&b.res_empty), 1);
        for (int s = 0; s < 3; ++s) {
            mbar_init(smem_addr(&b.st_full[s]), 1);
            mbar_init(smem_addr(&b.st_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_addr(&b.v_full[s]), 1);
            mbar_init(smem_addr(&b.v_empty[s]), 1);
        }
        mbar_init(smem_addr(&b.s_full), 1);
        mbar_init(smem_addr(&b.p_full), kElemWarps);
        mbar_init(smem_addr(&b.o_full), 1);
        mbar_init(smem_addr(&b.o_empty), kElemWarps);
        mbar_init(smem_addr(&b.p1_full), kElemWarps);
        mbar_init(smem_addr(&b.dp_full), 1);
        mbar_init(smem_addr(&b.dp_free), kElemWarps);
        mbar_init(smem_addr(&b.dq_full[0]), kElemWarps);
        mbar_init(smem_addr(&b.dq_full[1]), kElemWarps);
        mbar_init(smem_addr(&b.grp[0]), kElemWarps / 2);
        mbar_init(smem_addr(&b.grp[1]), kElemWarps / 2);
        mbar_init(smem_addr(&b.drain), 1);
        b.abort = 0;
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_addr(&b.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem_base;
    if (warp < kElemWarps)
        bwd_elem<D, kDkDv>(p, b, xch, tmem);
    else if (warp == kWarpLoad)
        bwd_load<D, kDkDv>(p, b, smem, &ra0, &ra1, &sb0, &sb1);
    else
        bwd_mma<D, kDkDv>(p, b, smem, tmem);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// D_i = dO_i . O_i (fp32).  Eight bf16 per lane per 16-byte load: a row of
// D elements takes D/8 lanes, so one warp covers 256/D rows.
template <int D>
__global__ void __launch_bounds__(256)
    prep_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
                float *__restrict__ dvec, long long rows)
{
    constexpr int kLanes = D / 8;            // lanes per row
    constexpr int kRowsPerWarp = 32 / kLanes;
    const int lane = threadIdx.x & 31;
    const long long row = (static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32) * kRowsPerWarp +
                          lane / kLanes;
    const int part = lane % kLanes;
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = *reinterpret_cast<const uint4 *>(o + row * D + part * 8);
        const uint4 c = *reinterpret_cast<const uint4 *>(dout + row * D + part * 8);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&av[i]));
            const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&cv[i]));
            acc = fmaf(x.x, y.x, acc);
            acc = fmaf(x.y, y.y, acc);
        }
    }
#pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0)
        dvec[row] = acc;
}

template <int D, bool kDkDv>
cudaError_t launch_one(const CUtensorMap &ra0, const CUtensorMap &ra1, const CUtensorMap &sb0,
                       const CUtensorMap &sb1, const BParams &p, int num_sms, cudaStream_t stream)
{
    using C = BCfg<D, kDkDv>;
    const size_t smem = C::kTilesBytes + C::kBarsBytes + (kDkDv ? sizeof(BXch) : 0) + 1024;
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D, kDkDv>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    const int grid = p.units < num_sms ? p.units : num_sms;
    bwd_kernel<D, kDkDv><<<grid, kThreads, smem, stream>>>(ra0, ra1, sb0, sb1, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd(const BwdArgs &a, const FwdMaps &m, const BwdMaps &mb, int num_sms,
                       cudaStream_t stream)
{
    BParams p;
    p.o = static_cast<const __nv_bfloat16 *>(a.o);
    p.dout = static_cast<const __nv_bfloat16 *>(a.dout);
    p.lse = a.lse;
    p.dvec = a.dvec;
    p.status = a.status;
    p.N = a.N;
    p.BH = a.B * a.H;
    p.T = (a.N + kTile - 1) / kTile;
    const long long units = static_cast<long long>(p.BH) * p.T;
    if (units == 0)
        return cudaSuccess;
    if (units > 0x7fffffffLL)
        return cudaErrorInvalidConfiguration;
    p.units = static_cast<int>(units);
    p.causal = a.causal;
    p.scale = a.scale;
    p.sl2 = a.scale * kLog2e;
    const long long rows = static_cast<long long>(p.BH) * p.N;
    const long long rows_per_block = 8LL * (256 / D);  // 8 warps of 256/D rows
    prep_kernel<D><<<static_cast<unsigned>((rows + rows_per_block - 1) / rows_per_block), 256, 0,
                     stream>>>(p.o, p.dout, p.dvec, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    // dK, dV: resident (K, V), streamed (Q, dO).
    p.g0 = static_cast<__nv_bfloat16 *>(a.dk);
    p.g1 = static_cast<__nv_bfloat16 *>(a.dv);
    if ((e = launch_one<D, true>(m.k, m.v, m.q, mb.dout, p, num_sms, stream)) != cudaSuccess)
        return e;
    // dQ: resident (Q, dO), streamed (K, V).
    p.g0 = static_cast<__nv_bfloat16 *>(a.dq);
    p.g1 = nullptr;
    return launch_one<D, false>(m.q, mb.dout, m.k, m.v, p, num_sms, stream);
}

}  // namespace

cudaError_t launch_bwd_sm103(const BwdArgs &a, const FwdMaps &m, const BwdMaps &mb, int num_sms,
                             cudaStream_t stream)
{
    return a.d == 64 ? launch_bwd<64>(a, m, mb, num_sms, stream)
                     : launch_bwd<128>(a, m, mb, num_sms, stream);
}

}  // namespace fattn
