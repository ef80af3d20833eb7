// Tensor-core GEMM for prefill-sized ubatches on sm_103a (tcgen05 + TMEM + TMA):
//   out[t][n] = sum_k A[t][k] W[n][k]
// with A the f16 activations [T][K] (RMS-normed input, attention output or SwiGLU output) and W a
// Q4_0 / Q8_0 matrix dequantised to f16 on load, f32 accumulation in tensor memory, and the
// shared epilogues (RoPE + KV append, residual add, SwiGLU, logits + argmax).
//
// Prefill is where the work is compute-bound (KV-cache section of the article: prefill loads the
// compute units), so the contraction runs on the 5th-generation tensor cores. One CTA computes MT
// (1 or 2) 128-row weight tiles (adjacent rows, or gate chunks and their up chunks) against BN
// tokens (64, 128 or 256), optionally a share of the K steps (split K):
//   warp 0      TMA producer: one box per stage holds the quants and scales of the weight tiles
//               (64 row quads of the quad-interleaved layout; issued before the grid-dependency
//               wait: the weights do not depend on the previous kernel);
//   warp 1      allocates the TMEM accumulator and issues tcgen05.mma from one lane -- W A_hi and
//               W A_lo (with BN <= 128 as one MMA over both parts' rows, N = 2 BN, the epilogue
//               adding the two halves; with BN = 256 into the same accumulator), so the
//               activations keep about 22 bits and only the f16 rounding of the dequantised
//               weights remains; each stage's tcgen05.commit frees its shared-memory slots.
//               With 64 tokens and two tiles the operands swap (the activations' 128 rows as M,
//               both weight tiles as N = 256) and the epilogue transposes the sums first;
//   warps 2..9  dequantise the raw blocks (with two weight tiles warps 2..5 tile 0, warps 6..9
//               tile 1) into the K-major SWIZZLE_128B f16 tile the MMA reads ((q - 8) or q is
//               exact in f16, then one f16 multiply by the block scale); then run the epilogue
//               from TMEM with tcgen05.ld, its operands (RoPE rows, residual rows, other splits'
//               partial sums) staged with cp.async in the ring space the main loop has freed;
//   warp 10     loads the activation tiles [BN][64] f16 (high and low parts) with TMA into the
//               SWIZZLE_128B layout, as many steps ahead as the activation ring holds. The CTAs of
//               a cluster (CL consecutive weight tiles, one token tile) share every activation
//               tile: each loads 1/CL of its rows, multicast to all of them, and a slot is reused
//               once every CTA's MMAs of the cluster have released it (their commits arrive on
//               all the cluster's barriers). The activations, 4 bytes per element and re-read by
//               every weight tile, thus cross L2 once per cluster, and no dequantising warp waits
//               on an activation load.
// All mbarrier waits are bounded; a timeout sets the context's error word and the CTA finishes
// without further work.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/lcx.h"
#include "epilogue.cuh"
#include "tc_common.cuh"

namespace lcx {
namespace tc {

constexpr int BM = 128;   // weight rows per MMA (tensor-memory lanes)
constexpr int BK = 64;    // k per stage: 128 bytes of f16
// The 8 dequantising / epilogue warps (256 threads) on named barrier 1.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// true for all 256 threads if `pred` holds in every one of them
__device__ __forceinline__ bool epi_all(bool pred) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, 1, 256, q;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(r) : "r"((uint32_t)pred) : "memory");
    return r != 0;
}
// Shared memory: three rings. The dequantised f16 weight tiles (SA slots, the largest part of a
// step); the activation tiles (SB slots, freed by the MMAs of every CTA of the cluster that read
// them); the raw weight boxes (SR slots, freed by the dequantising warps as soon as they have read
// them -- not by the MMA, so the next boxes stream in while the tensor pipe works). With SA = 3 the
// dequantisation of step j waits only for the MMAs of step j - 3, so it overlaps the MMAs of steps
// j - 2 and j - 1.
// MT weight tiles of 128 rows per CTA (1 or 2) share each activation tile of BN tokens.
template <int QT, int BN, int MT>
struct Cfg {
    static constexpr int QB = QT == Q8 ? 32 : 16;          // quant bytes per 32-element block
    static constexpr int A_BYTES = MT * BM * BK * 2;      // f16 weight tiles (one slot of the A ring)
    static constexpr int B_BYTES = 2 * BN * BK * 2;       // f16 activation tiles: high and low parts
    static constexpr int PB = 8 * QB + 16;                // one block pair of a row quad (QMat)
    static constexpr int RQ_BYTES = MT * (BM / 4) * PB;   // raw tiles: 32 quads per tile x one block pair
    static constexpr int RQ_SLOT = ((RQ_BYTES + 1023) / 1024) * 1024;
    static constexpr int SA = (MT == 2 && QT == Q4 && BN == 64) ? 3 : 2;
    static constexpr int SR = (MT == 2 && QT == Q8 && BN == 128) ? 2 : 3;
    static constexpr int SB_FIT = (220 * 1024 - SA * A_BYTES - SR * RQ_SLOT) / B_BYTES;
    static constexpr int SB = SB_FIT < 6 ? SB_FIT : 6;
    static constexpr int DB = SB - 1;   // activation prefetch distance (the loader runs a ring ahead)
    static_assert(SB >= 2, "the activation prefetch needs at least two slots");
    static constexpr int SMEM = SA * A_BYTES + SB * B_BYTES + SR * RQ_SLOT + 1024 /* align */ + 512 /* barriers */;
    // the A and B rings, reused by the epilogue for its staged operands
    static constexpr int STAGE = SA * A_BYTES + SB * B_BYTES;
    static_assert(16 * BN + BN * 128 * 4 <= STAGE, "positions, cells and RoPE rows of the tile's tokens");
    static_assert(BN * MT * BM * 4 <= STAGE, "residual rows of the tile");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
    // Per weight tile one accumulator. With BN <= 128 the high and low activation rows form one
    // B operand of 2 BN rows (the ring slot holds them contiguously), so one MMA of N = 2 BN
    // computes W A_hi into the accumulator's first BN columns and W A_lo into the next BN, and the
    // epilogue adds the two; an MMA of N = 256 keeps the tensor pipe far busier than two of N = 128
    // (each instruction has a fixed cost, and the N = 256 form reads the weight tile once for
    // twice the products). With BN = 256 the two parts are accumulated into the same BN columns.
    static constexpr bool STACK = BN <= 128;
    static constexpr int ACC_COLS = STACK ? 2 * BN : BN;   // TMEM columns per weight tile
    // 64 tokens x 2 tiles: the operands swap -- the activation tile's 128 rows (64 high, 64 low)
    // are the MMA's M and both weight tiles (256 rows, contiguous in the A ring) its N, so a K
    // step takes 4 MMAs of N = 256 instead of 8 of N = 128; TMEM lanes are then activation rows
    // and columns weight rows, and the epilogue transposes the sums through shared memory
    static constexpr bool SWAP = BN == 64 && MT == 2;
    static constexpr int TMEM_NEED = SWAP ? MT * BM : MT * ACC_COLS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    static_assert(TMEM_NEED <= 512, "tensor memory holds 512 columns");
    static_assert(BN <= 256, "one MMA covers at most 256 columns");
    // SWAP: the transposed sums [MT * BM rows][BN + 1] f32 (a row padded by one float, so that
    // the threads of a warp, one weight row each, read different banks) at the end of the
    // staging space
    static constexpr int T_LD = BN + 1;
    static constexpr int T_OFF = (STAGE - MT * BM * T_LD * 4) / 16 * 16;
    static_assert(!SWAP || (16 * BN + BN * 128 * 4 <= T_OFF && BN * MT * BM * 4 <= T_OFF),
                  "staged operands and the transposed sums side by side");
};

struct GemmParams {
    int N;          // logical rows (outputs) of W
    int T;          // tokens
    int nk;         // K / 64: steps of the whole contraction
    int ks;         // splits of the K steps (gridDim.z); 1: the CTA applies the epilogue itself
    int N_pad;      // rows of the partial sums' layout
    float *part;    // ks > 1: partial sums [ks][T][N_pad] f32
    int32_t *cnt;   // ks > 1: arrival counter per output tile (zero between launches)
};

// Dequantise blocks b0 .. b0 + NBLK - 1 (of the step's block pair) of row `row` (0..127) of one
// raw tile -- 32 row quads x one block pair, as stored (QMat) -- into the swizzled f16 tile.
template <int QT, int NBLK>
__device__ __forceinline__ void dequant_row(const uint8_t *rq, uint8_t *atile, int row, int b0) {
    constexpr int QB = QT == Q8 ? 32 : 16, PB = 8 * QB + 16;
    const uint8_t *q = rq + (row >> 2) * PB + (row & 3) * 2 * QB;
    const __half *sc = reinterpret_cast<const __half *>(rq + (row >> 2) * PB + 8 * QB);
    uint8_t *dst = atile + row * 128;
#pragma unroll
    for (int bb = 0; bb < NBLK; ++bb) {
        const int blk = b0 + bb;
        const __half2 d2 = __half2half2(sc[blk * 4 + (row & 3)]);
        if (QT == Q4) {
            const uint4 w = *reinterpret_cast<const uint4 *>(q + blk * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            const __half2 off = __float2half2_rn(1032.f);
            const __half2 sixteenth = __float2half2_rn(0.0625f), m72 = __float2half2_rn(-72.f);
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // bytes 0..7 (h = 0) or 8..15 (h = 1)
                uint32_t lo[4], hi[4];
#pragma unroll
                for (int wi = 0; wi < 2; ++wi) {
                    const uint32_t t0 = __byte_perm(ws[2 * h + wi], 0u, 0x4140u);   // [b0, 0, b1, 0]
                    const uint32_t t1 = __byte_perm(ws[2 * h + wi], 0u, 0x4342u);   // [b2, 0, b3, 0]
                    // low nibbles as f16 1024 + q, high nibbles as 1024 + 16 q (no shift needed)
                    lo[2 * wi] = (t0 & 0x000F000Fu) | 0x64006400u;
                    lo[2 * wi + 1] = (t1 & 0x000F000Fu) | 0x64006400u;
                    hi[2 * wi] = (t0 & 0x00F000F0u) | 0x64006400u;
                    hi[2 * wi + 1] = (t1 & 0x00F000F0u) | 0x64006400u;
                }
                uint32_t olo[4], ohi[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __half2 a = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&lo[e]), off), d2);
                    // (1024 + 16 q) / 16 - 72 = q - 8, exact in one fused multiply-add
                    __half2 b = __hmul2(__hfma2(*reinterpret_cast<__half2 *>(&hi[e]), sixteenth, m72), d2);
                    olo[e] = *reinterpret_cast<uint32_t *>(&a);
                    ohi[e] = *reinterpret_cast<uint32_t *>(&b);
                }
                const int c_lo = blk * 4 + h;       // elements 8h .. 8h+7 of the block
                const int c_hi = blk * 4 + 2 + h;   // elements 16+8h ..
                *reinterpret_cast<uint4 *>(dst + ((c_lo ^ (row & 7)) << 4)) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
                *reinterpret_cast<uint4 *>(dst + ((c_hi ^ (row & 7)) << 4)) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
            }
        } else {
            const __half2 off = __float2half2_rn(1152.f);
#pragma unroll
            for (int c = 0; c < 4; ++c) {           // chunk c of the block: bytes 8c .. 8c+7
                const uint2 w = *reinterpret_cast<const uint2 *>(q + blk * 32 + c * 8);
                const uint32_t ws[2] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u};
                uint32_t o[4];
#pragma unroll
                for (int wi = 0; wi < 2; ++wi) {
                    uint32_t p0 = __byte_perm(ws[wi], 0x64646464u, 0x4140u);   // (1024 + q0 + 128, 1024 + q1 + 128)
                    uint32_t p1 = __byte_perm(ws[wi], 0x64646464u, 0x4342u);
                    __half2 a = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&p0), off), d2);
                    __half2 b = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&p1), off), d2);
                    o[2 * wi] = *reinterpret_cast<uint32_t *>(&a);
                    o[2 * wi + 1] = *reinterpret_cast<uint32_t *>(&b);
                }
                const int cc = blk * 4 + c;
                *reinterpret_cast<uint4 *>(dst + ((cc ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

template <int QT, int BN, int MT, int EPI>
__global__ void __launch_bounds__(352, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tm_ahi, const __grid_constant__ CUtensorMap tm_alo,
              const __grid_constant__ CUtensorMap tm_w, const GemmParams p, const FwdArgs a, const int layer) {
    using C = Cfg<QT, BN, MT>;
    constexpr int SA = C::SA, SB = C::SB, SR = C::SR;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *act_ring = smem + SA * C::A_BYTES;
    uint8_t *raw_ring = act_ring + SB * C::B_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(raw_ring + SR * C::RQ_SLOT);
    // full_w / empty_w: a raw weight box landed / read by the dequantising warps; full_b / empty_b:
    // an activation tile landed / read by the MMAs; full_a / empty_a: a dequantised tile written /
    // read by the MMAs
    uint64_t *full_w = bars, *empty_w = full_w + SR, *full_b = empty_w + SR, *empty_b = full_b + SB,
             *full_a = empty_b + SB, *empty_a = full_a + SA, *acc_bar = empty_a + SA;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x, tok0 = blockIdx.y * BN;
    // the cluster: CL CTAs of consecutive weight tiles sharing this token tile
    const int CL = (int)cluster_size(), crank = (int)cluster_rank();
    const uint16_t cmask = (uint16_t)((1u << CL) - 1u);
    // this CTA's K steps: split blockIdx.z of p.ks (equal runs; the last may be short)
    const int nk_per = (p.nk + p.ks - 1) / p.ks;
    const int kb = blockIdx.z * nk_per;
    const int nk = max(0, min(p.nk, kb + nk_per) - kb);
    // first weight row of each M tile: MT adjacent 128-row tiles (for gate/up each holds 16
    // gate quads interleaved with their 16 up quads)
    int row0[MT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) row0[mt] = (m_tile * MT + mt) * BM;
    auto a_tile = [&](int aslot, int mt) { return smem + aslot * C::A_BYTES + mt * BM * BK * 2; };
    auto b_tile = [&](int slot) { return act_ring + slot * C::B_BYTES; };
    auto rq_tile = [&](int slot, int mt) { return raw_ring + slot * C::RQ_SLOT + mt * (BM / 4) * C::PB; };

    if (threadIdx.x == 0) {
        for (int i = 0; i < SR; ++i) {
            mbar_init(&full_w[i], 1);
            mbar_init(&empty_w[i], 8);   // one arrival per dequantising warp
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(&full_b[i], 1);     // the loader's expect_tx; the bytes come from every CTA's share
            mbar_init(&empty_b[i], CL);   // one MMA commit from each CTA of the cluster
        }
        for (int i = 0; i < SA; ++i) {
            mbar_init(&full_a[i], 8);   // one arrival per dequantising warp
            mbar_init(&empty_a[i], 1);
        }
        mbar_init(acc_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {   // tensor-memory accumulators: MT x BN f32 columns, 128 lanes
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(saddr(tmem_slot)), "r"((uint32_t)C::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    // every CTA's barriers are initialised before any peer multicasts into this one or arrives here
    if (CL > 1) cluster_sync_all();

    if (warp == 10) {
        // ---------------------------------------------------------------- activation loader
        if (lane == 0) {
            bool ok = true;
            constexpr int PART_ROWS_MAX = BN;
            const int prow = BN / CL;             // this CTA's share of the tile's rows
            const uint32_t part_bytes = (uint32_t)prow * BK * 2;
            LCX_PDL_WAIT();   // the activations are the previous kernel's output
            int issued = 0;
            for (int j = 0; j < nk && ok; ++j) {
                const int slot = j % SB;
                if (j >= SB && !(ok = mbar_wait(&empty_b[slot], ((j / SB) - 1) & 1))) break;
                mbar_expect_tx(&full_b[slot], (uint32_t)C::B_BYTES);
                uint8_t *bt = b_tile(slot);
                const int x = (kb + j) * BK, y = tok0 + crank * prow;
                if (CL > 1) {
                    tma_2d_mc(bt + crank * prow * 128, &tm_ahi, x, y, &full_b[slot], cmask);
                    tma_2d_mc(bt + BN * BK * 2 + crank * prow * 128, &tm_alo, x, y, &full_b[slot], cmask);
                } else {
                    tma_2d(bt, &tm_ahi, x, y, &full_b[slot]);
                    tma_2d(bt + BN * BK * 2, &tm_alo, x, y, &full_b[slot]);
                }
                issued = j + 1;
                (void)part_bytes;
                (void)PART_ROWS_MAX;
            }
            if (!ok) atomicExch(a.err, 1);
            // every step issued has landed in this CTA before it ends (each CTA waits for its own copy)
            for (int j = (issued > SB ? issued - SB : 0); j < issued; ++j) mbar_wait(&full_b[j % SB], (j / SB) & 1);
        }
    } else if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            bool ok = true;
            auto issue_w = [&](int j) {   // quants and scales of the 32 MT quads of the tiles: one box
                const int slot = j % SR;
                mbar_expect_tx(&full_w[slot], C::RQ_BYTES);
                tma_2d(rq_tile(slot, 0), &tm_w, (kb + j) * (C::PB / 4), row0[0] / 4, &full_w[slot]);
            };
            const int pre = nk < SR ? nk : SR;
            for (int j = 0; j < pre; ++j) issue_w(j);
            LCX_PDL_TRIGGER();
            int issued = pre;
            for (int j = SR; j < nk && ok; ++j) {
                if (!(ok = mbar_wait(&empty_w[j % SR], ((j / SR) - 1) & 1))) break;
                issue_w(j);
                issued = j + 1;
            }
            if (!ok) atomicExch(a.err, 1);
            // every copy issued must land before the CTA exits
            for (int j = (issued > SR ? issued - SR : 0); j < issued; ++j) mbar_wait(&full_w[j % SR], (j / SR) & 1);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr int NP = C::STACK ? 1 : 2;                      // MMAs per weight tile and k
            constexpr uint32_t idesc = C::SWAP ? idesc_f16(2 * BN, MT * BM) : idesc_f16(BM, C::STACK ? 2 * BN : BN);
            bool ok = true;
            for (int j = 0; j < nk; ++j) {
                const int slot = j % SB, aslot = j % SA;
                if (!(ok = mbar_wait(&full_a[aslot], (j / SA) & 1) && mbar_wait(&full_b[slot], (j / SB) & 1))) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t bbase = saddr(b_tile(slot));
                // stacked: one MMA over the high and low rows together (2 BN rows of B, 2 BN
                // accumulator columns); otherwise W A_hi then W A_lo into the same BN columns. The
                // weight tiles alternate so consecutive MMAs use different accumulators.
                if (C::SWAP) {
                    // D[act row][weight row] += A_act (128 rows: high then low) x W^T (256 rows)
                    const uint32_t wbase = saddr(a_tile(aslot, 0));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(tmem, sw128_desc(bbase + kk * 32), sw128_desc(wbase + kk * 32), idesc,
                                (j > 0 || kk > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
                        for (int hl = 0; hl < NP; ++hl) {
#pragma unroll
                            for (int mt = 0; mt < MT; ++mt) {
                                const uint32_t abase = saddr(a_tile(aslot, mt));
                                mma_f16(tmem + mt * C::ACC_COLS, sw128_desc(abase + kk * 32),
                                        sw128_desc(bbase + hl * BN * BK * 2 + kk * 32), idesc,
                                        (j > 0 || kk > 0 || hl > 0) ? 1u : 0u);
                            }
                        }
                    }
                }
                // the activation slot is free once these MMAs (in every CTA of the cluster) have read
                // it, and so is the A slot
                if (CL > 1) mma_commit_mc(&empty_b[slot], cmask);
                else mma_commit(&empty_b[slot]);
                mma_commit(&empty_a[aslot]);
            }
            if (!ok) atomicExch(a.err, 1);
            mma_commit(acc_bar);
        }
    } else {
        // ---------------------------------------------------------------- activations, dequant, epilogue
        // 8 warps. Dequantisation: with two weight tiles, warps 2..5 own tile 0 and warps 6..9
        // tile 1, a row per thread; with one, two threads per row, a block each. All 8 run the
        // epilogue (see below).
        const int wt = threadIdx.x - 64;           // 0..255
        const int my_mt = MT == 2 ? wt >> 7 : 0;
        const int drow = MT == 2 ? wt & 127 : wt >> 1, dblk = MT == 2 ? 0 : wt & 1;
        bool ok = true;
        LCX_PDL_WAIT();   // the epilogue reads the previous kernels' output
        LCX_PDL_TRIGGER();
        for (int j = 0; j < nk; ++j) {
            const int rslot = j % SR, aslot = j % SA;
            ok = __all_sync(0xffffffffu, mbar_wait(&full_w[rslot], (j / SR) & 1));   // warp-uniform
            // the A slot is free once the MMAs of step j - SA are done
            if (ok && j >= SA) ok = __all_sync(0xffffffffu, mbar_wait(&empty_a[aslot], ((j / SA) - 1) & 1));
            if (!ok) break;
            dequant_row<QT, MT>(rq_tile(rslot, my_mt), a_tile(aslot, my_mt), drow, dblk);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor-core reads
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&full_a[aslot]);
                mbar_arrive(&empty_w[rslot]);   // this warp's rows of the raw box are read
            }
        }
        if (!ok) atomicExch(a.err, 1);
        const bool acc_ok = __all_sync(0xffffffffu, ok && mbar_wait(acc_bar, 0));
        // one answer for the 8 warps, so every named barrier below is reached by all of them
        const bool cta_ok = epi_all(acc_ok);
        if (acc_ok) asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        else if (ok) atomicExch(a.err, 1);
        // a warp reads the TMEM lanes of its quarter (warp % 4); with two tiles warps 2..5 take
        // tile 0 and 6..9 tile 1, all BN columns; with one tile the two warps of a quarter take
        // half of the columns each
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int lrow = q * 32 + lane;         // row within the tile
        const int r = row0[my_mt] + lrow;       // weight row
        const int rc = my_mt * BM + lrow;       // row within the CTA's MT tiles
        constexpr int RW = MT * BM;             // rows of the CTA
        const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + my_mt * C::ACC_COLS;
        // the sums of 32 tokens (chunk cb) of this thread's row: W (A_hi + A_lo); both halves'
        // loads are in flight before the one wait
        float *s_t = reinterpret_cast<float *>(smem + C::T_OFF);   // SWAP: [RW rows][T_LD]
        auto acc_ld = [&](int cb, uint32_t (&vv)[32]) {
            if (C::SWAP) {
#pragma unroll
                for (int i = 0; i < 32; ++i) vv[i] = __float_as_uint(s_t[rc * C::T_LD + cb * 32 + i]);
            } else if (C::STACK) {
                uint32_t lo[32];
                tmem_ld32_issue(tq + cb * 32, vv);
                tmem_ld32_issue(tq + BN + cb * 32, lo);
                tmem_ld_wait(vv);
                regs_ready(lo);
#pragma unroll
                for (int i = 0; i < 32; ++i) vv[i] = __float_as_uint(__uint_as_float(vv[i]) + __uint_as_float(lo[i]));
            } else {
                tmem_ld32_issue(tq + cb * 32, vv);
                tmem_ld_wait(vv);
            }
        };
        const int cb0 = MT == 2 ? 0 : (wt >> 7) * (BN / 64), cb1 = MT == 2 ? BN / 32 : cb0 + BN / 64;

        if (C::SWAP) {
            // TMEM lane = activation row (lanes 0..63 the tokens' high parts, 64..127 their low
            // parts), column = weight row. The low rows' warps store theirs transposed, then the
            // high rows' warps add theirs: s_t[weight row][token] = W (A_hi + A_lo). A warp pair
            // of a lane quarter takes half of the 256 columns each.
            const int arow = q * 32 + lane;           // activation row of this thread's lane
            const int col0 = (wt >> 7) * 128;         // this warp's half of the weight rows
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {
                const bool mine = pass == 0 ? arow >= BN : arow < BN;   // warp-uniform
                if (cta_ok && mine)
                    for (int c = 0; c < 128; c += 64) {   // two 32-column loads before one wait
                        uint32_t v0[32], v1[32];
                        tmem_ld32_issue(tmem + ((uint32_t)(q * 32) << 16) + col0 + c, v0);
                        tmem_ld32_issue(tmem + ((uint32_t)(q * 32) << 16) + col0 + c + 32, v1);
                        tmem_ld_wait(v0);
                        regs_ready(v1);
                        const int tok = arow & (BN - 1);
                        float *d0 = s_t + (col0 + c) * C::T_LD + tok;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float *a0 = d0 + i * C::T_LD, *a1 = d0 + (32 + i) * C::T_LD;
                            if (pass == 0) {
                                *a0 = __uint_as_float(v0[i]);
                                *a1 = __uint_as_float(v1[i]);
                            } else {
                                *a0 += __uint_as_float(v0[i]);
                                *a1 += __uint_as_float(v1[i]);
                            }
                        }
                    }
                epi_sync();
            }
        }

        // Operands of the epilogue staged in shared memory: once the accumulator is complete every
        // activation and weight tile has been consumed and no copy is in flight, so the A and B
        // rings (contiguous from the base) are free. All 256 threads copy with cp.async, every
        // copy in flight before one wait:
        //   QKV    the tokens' positions and cells, then the RoPE (cos, sin) rows of their positions;
        //   RESID  the residual rows x[t][rows of the CTA] of the CTA's tokens.
        const int qw = a.H * a.hd, kw = a.KV * a.hd;
        // s_coff: a token's cache cell as an element offset within (layer, kv head) of the cache
        // [L][n_pages][KV][kPage][hd]: page * KV * kPage * hd + slot * hd
        long long *s_coff = reinterpret_cast<long long *>(smem);
        int *s_pos = reinterpret_cast<int *>(smem + 8 * BN);
        float2 *s_rope = reinterpret_cast<float2 *>(smem + 16 * BN);
        float *s_x = reinterpret_cast<float *>(smem);
        const bool any_rot = EPI == EPI_QKV && row0[0] < qw + kw;
        if (EPI == EPI_QKV) {
            if (cta_ok)
                for (int i = wt; i < BN; i += 256) {
                    const int t = min(tok0 + i, p.T - 1);
                    s_pos[i] = __ldg(a.ub.pos + t);
                    const int cell = __ldg(a.ub.cell + t);
                    s_coff[i] = ((long long)(cell / kPage) * a.KV * kPage + cell % kPage) * a.hd;
                }
            epi_sync();
            if (cta_ok && any_rot) {
                const int chunks = a.hd / 4;   // 16-byte pieces of a row of hd / 2 pairs
                for (int i = wt; i < BN * chunks; i += 256) {
                    const int tt = i / chunks, c = i - tt * chunks;
                    cp_async16(saddr(s_rope) + (uint32_t)i * 16, a.rope + (size_t)s_pos[tt] * (a.hd / 2) + c * 2);
                }
                cp_async_wait_all();
            }
            epi_sync();
        }
        // x rows of the CTA's tokens [first, first + n) into s_x[t - first][RW] (rows past N and
        // tokens past T are not read)
        auto stage_x = [&](int first, int n, float *dst) {
            constexpr int CPR = RW / 4;   // 16-byte pieces a token
            for (int i = wt; i < n * CPR; i += 256) {
                const int tt = i / CPR, c = i - tt * CPR;
                const int t = tok0 + first + tt, rr = row0[0] + 4 * c;
                if (t < p.T && rr < p.N) cp_async16(saddr(dst) + (uint32_t)i * 16, a.x + (size_t)t * a.d + rr);
            }
        };
        if (EPI == EPI_RESID && p.ks == 1) {
            if (cta_ok) {
                stage_x(0, BN, s_x);
                cp_async_wait_all();
            }
            epi_sync();
        }

        // the fused epilogue of 32 tokens (chunk cb) of this thread's row, from their sums vv;
        // sx: the staged residual rows of those tokens (RESID)
        auto epilogue = [&](int cb, uint32_t (&vv)[32], const float *sx) {
            if (EPI == EPI_SWIGLU) {
                // rows 8f'..8f'+3 gate, 8f'+4..8f'+7 up of features 4f'..: the gate lane takes the
                // chunk's first 16 tokens and its up partner (lane + 4) the last 16, each sending
                // the other the half it needs
                const int f = (r >> 3) * 4 + (lrow & 3);
                const bool gate = (lane & 7) < 4;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float lo_half = __uint_as_float(vv[i]), hi_half = __uint_as_float(vv[16 + i]);
                    const float mine = gate ? lo_half : hi_half;
                    const float other = __shfl_xor_sync(0xffffffffu, gate ? hi_half : lo_half, 4);
                    const float g = gate ? mine : other, u = gate ? other : mine;
                    const int t = tok0 + cb * 32 + (gate ? i : 16 + i);
                    if (t < p.T && f < a.F) store_split(a.h16, a.h16_lo, (size_t)t * a.F_pad + f, silu_f(g) * u);
                }
            } else if (EPI == EPI_RESID) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = tok0 + cb * 32 + i;
                    if (t < p.T && r < p.N) a.x[(size_t)t * a.d + r] = sx[i * RW + rc] + __uint_as_float(vv[i]);
                }
            } else if (EPI == EPI_LOGITS) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = tok0 + cb * 32 + i;
                    const float v = __uint_as_float(vv[i]);
                    unsigned long long key = 0ull;
                    if (t < p.T && r < p.N) {
                        a.logits[(size_t)t * a.V + r] = v;
                        key = argmax_key(v, r);
                        if (!isfinite(v)) note_nonfinite(a);
                    }
#pragma unroll
                    for (int o = 16; o; o >>= 1) {
                        const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
                        key = other > key ? other : key;
                    }
                    if (lane == 0 && key) atomicMax(&a.amax_key[t], key);
                }
            } else {   // EPI_QKV: rotate (q, k) pairs of adjacent rows, store q f32 and k, v f16
                // Every lane stores its own row, so no branch diverges within a warp: a rotated
                // pair (even row e, odd row e + 1) is y_e = v_e cos - v_o sin and y_o = v_o cos +
                // v_e sin, i.e. y = v cos + s v_partner sin with s = -1 on the even lane and +1 on
                // the odd one; V rows keep v (a select, so the compiler can issue every token's
                // shared-memory load and shuffle ahead of the predicated stores).
                const bool isq = r < qw, rot = r < qw + kw;
                const bool store_row = r < qw + 2 * kw;
                const float sgn = (lane & 1) ? 1.f : -1.f;
                const int dim = (isq ? r : r - qw) & (a.hd - 1);   // hd is 64 or 128
                const int rr = isq ? 0 : (rot ? r - qw : r - qw - kw);
                const int sh = __ffs(a.hd) - 1, hd2 = a.hd / 2;
                float *qdst = a.q + r;
                __half *kvdst = (rot ? a.kc : a.vc) +
                                (((size_t)layer * a.n_pages * a.KV + (rr >> sh)) * kPage) * a.hd + dim;
                const float2 *rope = s_rope + dim / 2;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int tt = cb * 32 + i, t = tok0 + tt;
                    const float v = __uint_as_float(vv[i]);
                    const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
                    const float2 cs = rope[tt * hd2];
                    const float z = fmaf(sgn * partner, cs.y, v * cs.x);
                    const float y = rot ? z : v;
                    if (store_row && t < p.T) {
                        if (isq) qdst[(size_t)t * qw] = y;
                        else kvdst[s_coff[tt]] = __float2half_rn(y);
                    }
                }
            }
        };
        if (p.ks == 1) {
            if (cta_ok)
                for (int cb = cb0; cb < cb1; ++cb) {
                    uint32_t vv[32];
                    acc_ld(cb, vv);
                    epilogue(cb, vv, s_x + cb * 32 * RW);
                }
        } else {
            // split K: every CTA of an output tile stores its partial sums; the last of them to
            // arrive adds the ks partials in split order (its own from tensor memory, the others
            // staged in shared memory) and applies the epilogue. The counter is bumped even after
            // a failed wait, so it always returns to zero.
            __shared__ int s_last;
            if (cta_ok)
                for (int cb = cb0; cb < cb1; ++cb) {
                    uint32_t vv[32];
                    acc_ld(cb, vv);
                    float *dst = p.part + ((size_t)blockIdx.z * p.T) * p.N_pad + r;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int t = tok0 + cb * 32 + i;
                        if (t < p.T && r < p.N_pad) __stcg(dst + (size_t)t * p.N_pad, __uint_as_float(vv[i]));
                    }
                }
            epi_sync();   // the 8 epilogue warps' stores are done
            if (wt == 0) {
                __threadfence();
                const int prev = atomicAdd(p.cnt + blockIdx.x * gridDim.y + blockIdx.y, 1);
                s_last = prev == p.ks - 1;
            }
            epi_sync();
            if (s_last) {
                __threadfence();
                // token groups of G tokens (a multiple of 32): the other splits' partials of the
                // group and, for RESID, its residual rows, staged together
                const int n_in = p.ks - 1 + (EPI == EPI_RESID ? 1 : 0);
                // the staging space ends where the transposed sums begin (SWAP: they are the own
                // split's sums, read while the others' are added)
                const int stage_end = C::SWAP ? C::T_OFF : C::STAGE;
                const int stage_bytes = stage_end - (EPI == EPI_QKV ? 16 * BN + BN * 128 * 4 : 0);
                const int per_chunk = n_in * 32 * RW * 4;
                int G = (stage_bytes / per_chunk) * 32;
                G = G > BN ? BN : G;
                uint8_t *sbase = smem + (EPI == EPI_QKV ? stage_end - stage_bytes : 0);
                if (G >= 32) {
                    for (int g0 = 0; g0 < BN; g0 += G) {
                        float *sp = reinterpret_cast<float *>(sbase);   // [n_in][G][RW]
                        const int gn = min(G, BN - g0);                  // tokens of this group
                        if (cta_ok) {
                            int slot = 0;
                            for (int z = 0; z < p.ks; ++z) {
                                if (z == (int)blockIdx.z) continue;
                                float *d = sp + (size_t)slot * G * RW;
                                constexpr int CPR = RW / 4;
                                for (int i = wt; i < gn * CPR; i += 256) {
                                    const int tt = i / CPR, c = i - tt * CPR;
                                    const int t = tok0 + g0 + tt, rr = row0[0] + 4 * c;
                                    if (t < p.T && rr < p.N_pad)
                                        cp_async16(saddr(d) + (uint32_t)i * 16,
                                                   p.part + ((size_t)z * p.T + t) * p.N_pad + rr);
                                }
                                ++slot;
                            }
                            if (EPI == EPI_RESID) stage_x(g0, gn, sp + (size_t)slot * G * RW);
                            cp_async_wait_all();
                        }
                        epi_sync();
                        if (cta_ok)
                            for (int cb = max(cb0, g0 / 32); cb < min(cb1, (g0 + G) / 32); ++cb) {
                                uint32_t own[32];
                                acc_ld(cb, own);
                                const int tb = cb * 32 - g0;   // first token of the chunk in the group
                                float sum[32];
#pragma unroll
                                for (int i = 0; i < 32; ++i) sum[i] = 0.f;
                                int slot = 0;
                                for (int z = 0; z < p.ks; ++z) {
                                    if (z == (int)blockIdx.z) {
#pragma unroll
                                        for (int i = 0; i < 32; ++i) sum[i] += __uint_as_float(own[i]);
                                    } else {
                                        const float *src = sp + ((size_t)slot * G + tb) * RW + rc;
#pragma unroll
                                        for (int i = 0; i < 32; ++i) sum[i] += src[i * RW];
                                        ++slot;
                                    }
                                }
                                uint32_t vv[32];
#pragma unroll
                                for (int i = 0; i < 32; ++i) vv[i] = __float_as_uint(sum[i]);
                                epilogue(cb, vv, sp + ((size_t)(p.ks - 1) * G + tb) * RW);
                            }
                        epi_sync();   // the group's staging space is reused by the next group
                    }
                } else if (stage_bytes / (32 * RW * 4) >= 1 + (EPI == EPI_RESID ? 1 : 0)) {
                    // too many splits to stage all of one 32-token chunk: per chunk, the other
                    // splits' partials in batches of as many as fit (in split order, added into
                    // registers), the residual rows (RESID) in the last slot from the first batch
                    constexpr int CB = 32 * RW * 4;                     // bytes of a staged chunk
                    const int xs = EPI == EPI_RESID ? 1 : 0;
                    const int per_batch = stage_bytes / CB - xs;
                    float *sp = reinterpret_cast<float *>(sbase);     // [slot][32][RW]
                    float *sxc = sp + (size_t)per_batch * 32 * RW;    // RESID: the chunk's x rows
                    for (int cb = 0; cb < BN / 32; ++cb) {
                        const bool mine = cta_ok && cb >= cb0 && cb < cb1;   // warp-uniform
                        uint32_t own[32];
                        if (mine) acc_ld(cb, own);
                        float sum[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) sum[i] = 0.f;
                        for (int z = 0; z < p.ks;) {
                            // the batch: splits z .. ze - 1, at most per_batch of them other than ours
                            int ze = z, n_other = 0;
                            while (ze < p.ks && (ze == (int)blockIdx.z || n_other < per_batch)) {
                                if (ze != (int)blockIdx.z) ++n_other;
                                ++ze;
                            }
                            if (cta_ok) {
                                constexpr int CPR = RW / 4;
                                int slot = 0;
                                for (int zz = z; zz < ze; ++zz) {
                                    if (zz == (int)blockIdx.z) continue;
                                    float *d = sp + (size_t)slot * 32 * RW;
                                    for (int i = wt; i < 32 * CPR; i += 256) {
                                        const int tt = i / CPR, c = i - tt * CPR;
                                        const int t = tok0 + cb * 32 + tt, rr = row0[0] + 4 * c;
                                        if (t < p.T && rr < p.N_pad)
                                            cp_async16(saddr(d) + (uint32_t)i * 16,
                                                       p.part + ((size_t)zz * p.T + t) * p.N_pad + rr);
                                    }
                                    ++slot;
                                }
                                if (EPI == EPI_RESID && z == 0) stage_x(cb * 32, 32, sxc);
                                cp_async_wait_all();
                            }
                            epi_sync();
                            if (mine) {
                                int slot = 0;
                                for (int zz = z; zz < ze; ++zz) {
                                    if (zz == (int)blockIdx.z) {
#pragma unroll
                                        for (int i = 0; i < 32; ++i) sum[i] += __uint_as_float(own[i]);
                                    } else {
                                        const float *src = sp + (size_t)slot * 32 * RW + rc;
#pragma unroll
                                        for (int i = 0; i < 32; ++i) sum[i] += src[i * RW];
                                        ++slot;
                                    }
                                }
                            }
                            epi_sync();   // the slots are restaged by the next batch
                            z = ze;
                        }
                        if (mine) {
                            uint32_t vv[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) vv[i] = __float_as_uint(sum[i]);
                            epilogue(cb, vv, sxc);
                        }
                        epi_sync();   // the x slot is restaged for the next chunk
                    }
                } else if (cta_ok) {
                    // too many splits to stage one chunk: the partials straight from L2
                    for (int cb = cb0; cb < cb1; ++cb) {
                        float sum[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) sum[i] = 0.f;
                        for (int z = 0; z < p.ks; ++z) {
                            const float *src = p.part + ((size_t)z * p.T) * p.N_pad + r;
                            float v[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int t = min(tok0 + cb * 32 + i, p.T - 1);
                                v[i] = r < p.N_pad ? __ldcg(src + (size_t)t * p.N_pad) : 0.f;
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) sum[i] += v[i];
                        }
                        uint32_t vv[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) vv[i] = __float_as_uint(sum[i]);
                        if (EPI == EPI_RESID) {
                            float xo[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int t = tok0 + cb * 32 + i;
                                xo[i] = t < p.T && r < p.N ? __ldcg(a.x + (size_t)t * a.d + r) : 0.f;
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int t = tok0 + cb * 32 + i;
                                if (t < p.T && r < p.N) a.x[(size_t)t * a.d + r] = xo[i] + sum[i];
                            }
                        } else {
                            epilogue(cb, vv, nullptr);
                        }
                    }
                }
                if (wt == 0) p.cnt[blockIdx.x * gridDim.y + blockIdx.y] = 0;
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    // no CTA leaves while a peer's commit may still arrive on its barriers or a peer's copy land in
    // its shared memory (every CTA is past its accumulator wait and its loader's last landing here)
    if (CL > 1) cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)C::TMEM_COLS));
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    });
    return fn;
}

// 2D map over a row-major byte/half matrix: inner extent `inner` elements, `outer` rows.
bool make_map_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t inner, uint64_t outer,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return false;
    (void)esize;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int QT, int BN, int MT, int EPI>
cudaError_t run(const QMat &W, int T, int ks, const __half *A, const __half *A_lo, const FwdArgs &a, int layer,
                cudaStream_t s) {
    using C = Cfg<QT, BN, MT>;
    auto kern = k_gemm_tc<QT, BN, MT, EPI>;
    cudaError_t e = func_attr_once((const void *)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (!W.tm_ready) return cudaErrorInvalidValue;
    GemmParams p{W.N, T, W.K / BK, ks, W.N_pad, a.gemm_part, a.gemm_cnt};
    const int m_tiles = (W.N_pad + MT * BM - 1) / (MT * BM);   // rows past N_pad read as zeros
    // clusters of CL = 2 consecutive weight tiles share each activation tile (a CTA loads BN / 2
    // rows of it for both); the grid is padded to whole clusters (an extra tile reads zero rows).
    // Pairs, not fours: a cluster's CTAs must fit one GPC together, and with 220 KB of shared memory
    // each, larger clusters would leave a GPC's odd SMs idle.
    const int CL = m_tiles >= 2 ? 2 : 1;
    // activation maps: [T][K] f16 row-major; box 64 elements (128 bytes) x BN / CL rows, 128-byte
    // swizzle (the K-major layout the MMA reads); rows past T read as zeros
    alignas(64) CUtensorMap tm_hi, tm_lo;
    if (!make_map_2d(&tm_hi, A, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)W.K, (uint64_t)T, (uint64_t)W.K * 2, BK,
                     (uint32_t)(BN / CL), CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tm_lo, A_lo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)W.K, (uint64_t)T, (uint64_t)W.K * 2, BK,
                     (uint32_t)(BN / CL), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((m_tiles + CL - 1) / CL * CL, (T + BN - 1) / BN, ks);
    cfg.blockDim = dim3(352);
    cfg.dynamicSmemBytes = (size_t)C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    prefer_max_shared(kern);
    return cudaLaunchKernelEx(&cfg, kern, tm_hi, tm_lo, *reinterpret_cast<const CUtensorMap *>(MT == 2 ? W.tm_w : W.tm_w1),
                              p, a, layer);
}

template <int QT, int BN, int MT>
cudaError_t dispatch(const QMat &W, Epi epi, int T, int ks, const __half *A, const __half *A_lo, const FwdArgs &a,
                     int layer, cudaStream_t s) {
    switch (epi) {
        case EPI_QKV: return run<QT, BN, MT, EPI_QKV>(W, T, ks, A, A_lo, a, layer, s);
        case EPI_RESID: return run<QT, BN, MT, EPI_RESID>(W, T, ks, A, A_lo, a, layer, s);
        case EPI_SWIGLU: return run<QT, BN, MT, EPI_SWIGLU>(W, T, ks, A, A_lo, a, layer, s);
        case EPI_LOGITS: return run<QT, BN, MT, EPI_LOGITS>(W, T, ks, A, A_lo, a, layer, s);
    }
    return cudaErrorInvalidValue;
}

template <int QT>
cudaError_t dispatch_shape(const GemmShape &g, const QMat &W, Epi epi, int T, const __half *A, const __half *A_lo,
                           const FwdArgs &a, int layer, cudaStream_t s) {
    if (g.bn == 64 && g.mt == 1) return dispatch<QT, 64, 1>(W, epi, T, g.ks, A, A_lo, a, layer, s);
    if (g.bn == 64) return dispatch<QT, 64, 2>(W, epi, T, g.ks, A, A_lo, a, layer, s);
    if (g.bn == 128 && g.mt == 1) return dispatch<QT, 128, 1>(W, epi, T, g.ks, A, A_lo, a, layer, s);
    if (g.bn == 128) return dispatch<QT, 128, 2>(W, epi, T, g.ks, A, A_lo, a, layer, s);
    return dispatch<QT, 256, 1>(W, epi, T, g.ks, A, A_lo, a, layer, s);
}

}  // namespace tc

bool make_weight_maps(QMat &W) {
    // the storage as [N_pad / 4 quads][quad_bytes] in 4-byte units; a box is one block pair
    // (quants and scales) of 64 quads (two 128-row tiles of a CTA) or of 32 (one tile)
    const int pb = W.pair_bytes();
    W.tm_ready = tc::make_map_2d(reinterpret_cast<CUtensorMap *>(W.tm_w), W.w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4,
                                 W.quad_bytes() / 4, (uint64_t)W.N_pad / 4, W.quad_bytes(), (uint32_t)(pb / 4),
                                 (uint32_t)(tc::BM / 2), CU_TENSOR_MAP_SWIZZLE_NONE) &&
                 tc::make_map_2d(reinterpret_cast<CUtensorMap *>(W.tm_w1), W.w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4,
                                 W.quad_bytes() / 4, (uint64_t)W.N_pad / 4, W.quad_bytes(), (uint32_t)(pb / 4),
                                 (uint32_t)(tc::BM / 4), CU_TENSOR_MAP_SWIZZLE_NONE);
    return W.tm_ready;
}

// Tile shape of a launch: BN tokens x MT 128-row weight tiles per CTA, and the K steps split
// over ks CTAs, from a cost model per K step (cycles of one SM): the MMAs take 4 BN MT (128 x BN x
// 16 per MMA, hi and lo parts, four per 64-wide step, about 4096 multiply-adds a cycle), the
// dequantisation of MT tiles about 435 MT, given a 30% margin since it must also hide its waits,
// and the activation tile's L2 round trip over the shape's prefetch distance;
// the launch takes as many of those steps as each CTA runs, times its waves of CTAs. A split adds
// the partial sums' round trip (the last CTA of a tile reads ks partial tiles from L2; about
// 25000 + 16 BN MT ks cycles, measured, so a split is taken only where the CTAs would otherwise
// leave many SMs idle: on the 8B shape, the 64-token ubatches' QKV, O and down projections and the
// 512-token ubatch's down projection). Ties go to
// fewer CTAs (less activation traffic). Splits need room in the context's partial-sum scratch.
GemmShape gemm_shape(int type, int N_pad, int T, int nk, int n_sm, size_t part_bytes, int max_tiles) {
    static const int cand[5][2] = {{64, 1}, {64, 2}, {128, 1}, {128, 2}, {256, 1}};
    // activation prefetch distance of each shape (its ring depths), Q4_0 and Q8_0
    static const int db[2][5] = {{tc::Cfg<Q4, 64, 1>::DB, tc::Cfg<Q4, 64, 2>::DB, tc::Cfg<Q4, 128, 1>::DB,
                                  tc::Cfg<Q4, 128, 2>::DB, tc::Cfg<Q4, 256, 1>::DB},
                                 {tc::Cfg<Q8, 64, 1>::DB, tc::Cfg<Q8, 64, 2>::DB, tc::Cfg<Q8, 128, 1>::DB,
                                  tc::Cfg<Q8, 128, 2>::DB, tc::Cfg<Q8, 256, 1>::DB}};
    GemmShape best{64, 2, 1};
    long best_cost = -1, best_ctas = 0;
    for (int ci = 0; ci < 5; ++ci) {
        const int *c = cand[ci];
        const long tiles = (long)((N_pad + c[1] * 128 - 1) / (c[1] * 128)) * ((T + c[0] - 1) / c[0]);
        // a step also waits for its activation tile, loaded DB steps ahead from L2 (about 4000
        // cycles under load, measured: 64-step launches of each shape on the 8B 512-token ubatch)
        const long step = std::max<long>(std::max<long>(4L * c[0] * c[1], 566L * c[1]), 4000L / db[type == Q8][ci]);
        for (int ks = 1; ks <= 8; ++ks) {
            if (ks > 1 && (nk / ks < 4 || tiles * ks > 2L * n_sm || tiles > max_tiles ||
                           (size_t)ks * T * N_pad * 4 > part_bytes))
                break;
            if ((long)(ks - 1) * ((nk + ks - 1) / ks) >= nk) continue;   // every split gets K steps
            const long ctas = tiles * ks;
            const long waves = (ctas + n_sm - 1) / n_sm;
            const long cost = waves * ((nk + ks - 1) / ks) * step + (ks > 1 ? 25000L + ks * 16L * c[0] * c[1] : 0L);
            if (best_cost < 0 || cost < best_cost || (cost == best_cost && ctas < best_ctas)) {
                best_cost = cost;
                best_ctas = ctas;
                best = GemmShape{c[0], c[1], ks};
            }
        }
    }
    return best;
}

// a forced tile shape (lcx_set_gemm_tile): bn | mt << 12 | ks << 16, 0 for none
static std::atomic<int> g_forced_tile{0};

cudaError_t launch_gemm_tc(const QMat &W, Epi epi, int T, const __half *A, const __half *A_lo, const FwdArgs &a,
                           int layer, cudaStream_t s, int64_t &launches, int64_t *wide) {
    ++launches;
    const int nk = W.K / tc::BK;
    const size_t part_bytes = a.gemm_part ? a.gemm_part_bytes : 0;
    const int max_tiles = a.gemm_cnt ? kGemmMaxTiles : 0;
    GemmShape g;
    if (const int f = g_forced_tile.load(std::memory_order_relaxed)) {
        g = GemmShape{f & 0xFFF, (f >> 12) & 0xF, f >> 16};
        const long tiles = (long)((W.N_pad + g.mt * 128 - 1) / (g.mt * 128)) * ((T + g.bn - 1) / g.bn);
        if (g.ks > 1 && (nk / g.ks < 4 || tiles > max_tiles || (size_t)g.ks * T * W.N_pad * 4 > part_bytes ||
                         (long)(g.ks - 1) * ((nk + g.ks - 1) / g.ks) >= nk))
            g.ks = 1;
    } else {
        g = gemm_shape(W.type, W.N_pad, T, nk, device_sm_count(), part_bytes, max_tiles);
    }
    if (g.bn >= 128 && wide) ++*wide;
    if (W.type == Q4) return tc::dispatch_shape<Q4>(g, W, epi, T, A, A_lo, a, layer, s);
    if (W.type == Q8) return tc::dispatch_shape<Q8>(g, W, epi, T, A, A_lo, a, layer, s);
    return cudaErrorInvalidValue;
}

}  // namespace lcx

extern "C" int32_t lcx_set_gemm_tile(int32_t bn, int32_t mt, int32_t ks) {
    if (bn == 0) {
        lcx::g_forced_tile.store(0);
        return LCX_OK;
    }
    const bool ok = ((bn == 64 || bn == 128) && (mt == 1 || mt == 2)) || (bn == 256 && mt == 1);
    if (!ok || ks < 1 || ks > 8) return LCX_INVALID;
    lcx::g_forced_tile.store(bn | mt << 12 | ks << 16);
    return LCX_OK;
}
