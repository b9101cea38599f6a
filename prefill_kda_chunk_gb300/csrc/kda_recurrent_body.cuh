// The per-chunk step of the 16-token recurrent kernels, shared by the
// recurrent kernel and the fused kernel's chains: the record of one chunk in
// shared memory (stg, at shared address sw), this warp's 16 value channels
// vw .. vw + 15 of the stage's Ut^T slice, and the S^T fragments acc:
//
//   U   = Ut - W S                                   (16 x 16 values)
//   o_r = (q_r * exp(G_r))^T S + sum_{i<=r} P[r,i] U_i  (scale is in the record)
//   S  <- Diag(exp(G_last)) S + (K * exp(G_last - G))^T U
//
// Step order follows the chunk-to-chunk dependency chain (S -> U -> S): the
// U product first, the decay of S while it drains, S^T Qg^T to keep the
// tensor pipe busy, then the state update, and only after it the output
// branch (P U, store), which nothing later depends on.
#pragma once

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kStages = 4;

template <int BV>
struct RecurLayout {
    static constexpr int kWarps = BV / 16;          // consumer warps
    static constexpr int kSlices = kDim / BV;
    static constexpr int kStageBytes = kRecUt + BV * 32;  // W, Qg, Kd, P, gamma + Ut^T slice
    static constexpr int kOStage = kStages * kStageBytes;   // per-warp o staging, 512 B each
    static constexpr int kBars = kOStage + kWarps * 512;
    static constexpr int kSmem = kBars + 2 * kStages * 8;
};

// S^T fragments of this warp (value channels v0 .. v0 + 15, all 128 keys)
// from a [128 keys][128 values] fp32 state, or zero (S0 == nullptr).
__device__ __forceinline__ void recur_load_state(float (&acc)[16][4], const float *S0, int v0) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    if (S0 != nullptr) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int key = 8 * j + 2 * tig;
            acc[j][0] = S0[key * kDim + v0 + gid];
            acc[j][1] = S0[(key + 1) * kDim + v0 + gid];
            acc[j][2] = S0[key * kDim + v0 + gid + 8];
            acc[j][3] = S0[(key + 1) * kDim + v0 + gid + 8];
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    }
}

__device__ __forceinline__ void recur_store_state(const float (&acc)[16][4], float *SF, int v0) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int key = 8 * j + 2 * tig;
        SF[key * kDim + v0 + gid] = acc[j][0];
        SF[(key + 1) * kDim + v0 + gid] = acc[j][1];
        SF[key * kDim + v0 + gid + 8] = acc[j][2];
        SF[(key + 1) * kDim + v0 + gid + 8] = acc[j][3];
    }
}

// One chunk. virt: the columns are those of a segment's transition map (no
// Ut term). so: this warp's 512-byte o staging; orow: o of the chunk's first
// token at this warp's first value channel (token stride H * 128); L: tokens
// of the chunk. peek() is called once the state update is issued; its result
// is returned (the caller's look at the next stage's barrier).
template <bool OUT, typename Peek>
__device__ __forceinline__ bool recur_step(float (&acc)[16][4], const uint8_t *stg, uint32_t sw,
                                           int vw, bool virt, uint8_t *so, __nv_bfloat16 *orow,
                                           int L, int H, Peek &&peek) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3, quad = lane >> 3;
    // S^T as bf16 A fragments, one per 16-key step
    uint32_t aS[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        aS[kk][0] = pack_bf16(acc[2 * kk][0], acc[2 * kk][1]);
        aS[kk][1] = pack_bf16(acc[2 * kk][2], acc[2 * kk][3]);
        aS[kk][2] = pack_bf16(acc[2 * kk + 1][0], acc[2 * kk + 1][1]);
        aS[kk][3] = pack_bf16(acc[2 * kk + 1][2], acc[2 * kk + 1][3]);
    }

    // U^T = Ut^T - S^T W^T first (it gates the state update), two partial sums
    float uT[2][2][4], oT[2][2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int tk = 8 * nt + 2 * tig;
        // (a column of the map M has no input term)
        const float2 u01 = virt ? make_float2(0.f, 0.f) : unpack_bf16(
            *reinterpret_cast<const uint32_t *>(stg + kRecUt + ((vw + gid) * 16 + tk) * 2));
        const float2 u23 = virt ? make_float2(0.f, 0.f) : unpack_bf16(*reinterpret_cast<const uint32_t *>(
            stg + kRecUt + ((vw + gid + 8) * 16 + tk) * 2));
        uT[nt][0][0] = u01.x; uT[nt][0][1] = u01.y; uT[nt][0][2] = u23.x; uT[nt][0][3] = u23.y;
#pragma unroll
        for (int e = 0; e < 4; ++e) { uT[nt][1][e] = 0.f; oT[nt][0][e] = 0.f; oT[nt][1][e] = 0.f; }
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t bw[4];
        const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
        ldsm_x4(sw + kRecW + swz(rb, cb), bw[0], bw[1], bw[2], bw[3]);
        mma_r(uT[0][kk & 1], aS[kk], bw[0], bw[1]);
        mma_r(uT[1][kk & 1], aS[kk], bw[2], bw[3]);
    }
    // decay of the state, while the U products drain
    const float *gam = reinterpret_cast<const float *>(stg + kRecGamma);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float2 gm = *reinterpret_cast<const float2 *>(gam + 8 * j + 2 * tig);
        mul2(acc[j][0], acc[j][1], gm.x, gm.y);
        mul2(acc[j][2], acc[j][3], gm.x, gm.y);
    }
    // (Q e^G S)^T = S^T Qg^T keeps the tensor pipe busy meanwhile
    if constexpr (OUT) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t bq[4];
            const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
            ldsm_x4(sw + kRecQg + swz(rb, cb), bq[0], bq[1], bq[2], bq[3]);
            mma_r(oT[0][kk & 1], aS[kk], bq[0], bq[1]);
            mma_r(oT[1][kk & 1], aS[kk], bq[2], bq[3]);
        }
    }
    uint32_t aU[4];
    {
        float u[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) u[nt][e] = uT[nt][0][e] + uT[nt][1][e];
        aU[0] = pack_bf16(u[0][0], u[0][1]);
        aU[1] = pack_bf16(u[0][2], u[0][3]);
        aU[2] = pack_bf16(u[1][0], u[1][1]);
        aU[3] = pack_bf16(u[1][2], u[1][3]);
    }
    // S^T <- S^T Diag(gamma) + U^T Kd
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
        uint32_t b[4];
        const int rk = (quad & 1) * 8 + (lane & 7), ck = 16 * jp + (quad >> 1) * 8;
        ldsm_x4_t(sw + kRecKd + swz(rk, ck), b[0], b[1], b[2], b[3]);
        mma_r(acc[2 * jp], aU, b[0], b[1]);
        mma_r(acc[2 * jp + 1], aU, b[2], b[3]);
    }
    // look at the next stage's barrier now; its latency hides behind the MMAs
    const bool ready = peek();
    if constexpr (OUT) {
        // o^T = (Q e^G S)^T + U^T P^T (scale is in the record), off the chain
        float o[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[nt][e] = oT[nt][0][e] + oT[nt][1][e];
        {
            uint32_t bp[4];
            const int rp = (quad >> 1) * 8 + (lane & 7);
            ldsm_x4(sw + kRecP + rp * 32 + (quad & 1) * 16, bp[0], bp[1], bp[2], bp[3]);
            mma_r(o[0], aU, bp[0], bp[1]);
            mma_r(o[1], aU, bp[2], bp[3]);
        }
        {
            const int j = lane >> 3, r = lane & 7;
            stsm_x4_t(smem_u32(so) + ((j >> 1) * 8 + r) * 32 + (j & 1) * 16,
                      pack_bf16(o[0][0], o[0][1]), pack_bf16(o[0][2], o[0][3]),
                      pack_bf16(o[1][0], o[1][1]), pack_bf16(o[1][2], o[1][3]));
        }
        __syncwarp();
        {
            const int tok = lane >> 1, hf = lane & 1;
            if (tok < L) {
                const uint4 val = *reinterpret_cast<const uint4 *>(so + tok * 32 + hf * 16);
                *reinterpret_cast<uint4 *>(orow + tok * static_cast<int64_t>(H) * kDim + hf * 8) =
                    val;
            }
        }
    }
    return ready;
}

}  // namespace

}  // namespace kda
