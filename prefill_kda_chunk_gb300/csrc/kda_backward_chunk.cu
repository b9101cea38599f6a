// Gradients of KDA prefill in the chunked form (16-token chunks).
//
// The pages say that K3 trains with KDA layers ("Kimi K3 開源基礎設施";
// "Kimi K3 的三個系統設計": 69 KDA layers of 93). The forward is the chunk
// algebra of the prefill ("Kimi K3 的三個系統設計", section
// "為什麼 FlashKDA 選擇 16-token chunks"): per chunk, with S the state
// entering it and the record's quantities (W, Ut, Qg, Kd, P, gamma),
//
//   U = Ut - W S,  O = Qg S + P U,  S_next = Diag(gamma) S + Kd^T U.
//
// Its reverse, given dO and dS_next (= dL/dS_next):
//
//   dU = P^T dO + Kd dS_next
//   dS = Diag(gamma) dS_next + Qg^T dO - W^T dU          (to the chunk before)
//   dQg = dO S^T, dP = tril(dO U^T), dKd = U dS_next^T, dW = -dU S^T, dUt = dU
//   dgamma = rowsum(dS_next o S)
//
// and then back through the WY construction of the record (A, P, T = (I +
// A)^-1, W = T diag(beta) K e^G, Ut = T diag(beta) V, Qg = scale Q e^G,
// Kd = K e^(G_last - G), gamma = e^(G_last)) to dq, dk, dv, dbeta and dG, and
// dg as the reverse cumulative sum of dG within the chunk.
//
// Two launches after the forward's intra-chunk kernels (which build the
// records and T = (I + A)^-1 per chunk-head):
//   kda_bwd_chains_kernel: the forward chain again without outputs, keeping
//     every chunk's entry state S^T in bf16, and the reverse chain over the
//     chunks (the forward step with roles swapped), keeping every chunk's
//     dS_next^T in bf16 and writing dL/d(initial state); both roles in one
//     launch, neither waiting on the other;
//   kda_bwd_grad_kernel: chunk-parallel, one CTA per (chunk, head) at a time,
//     for everything else.
// The WY reverse factors the gated products like the forward (about the chunk
// start, or about the middle of the chunk's decay range) and takes exact
// per-pair exponentials exp(G_r - G_i) (r >= i) beyond those ranges, so it
// holds for any decay.

#include <cuda.h>

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_intra_body.cuh"
#include "kda_recurrent_body.cuh"

namespace kda {

namespace {

// ---------------------------------------------------------------------------
// The two chains. Each CTA owns (sequence, head, 64-value slice), 4 consumer
// warps holding 16 value rows x 128 keys of an fp32 state in MMA fragments
// and one producer warp streaming the records into a ring of stages. Every
// chunk, each consumer warp writes its rows of the state, in bf16, to the
// [record index][H][128 v][128 k] array of the gradient kernel: stmatrix into
// a shared staging half-pair ([16][64] x 2, 128-byte swizzle, double
// buffered) and two TMA tensor stores, so the chain issues 8 shared stores
// and 2 copies a step instead of 32 scattered global stores a thread.
constexpr int kCBV = 64;                   // value channels per chain CTA
constexpr int kCWarps = kCBV / 16;
constexpr int kStageOff = kCWarps * 2 * 4096;            // after the staging buffers
constexpr int kChainStageBytes = kRecUt + 2048;          // W, Qg, Kd, P, gamma (no Ut), then dO
                                                         //   [16 t][64 v] bf16, 128-byte swizzle
constexpr int kStatesStageBytes = kRecUt + kCBV * 32;    // ... and the slice of Ut^T
static_assert(kChainStageBytes == kStatesStageBytes, "one stage size for both chains");
constexpr int kChainSmem = kStageOff + kStages * kChainStageBytes + 2 * kStages * 8;

struct ChainMaps {
    CUtensorMap ckpt;      // S^T per chunk: [items][128 v][128 k] bf16, boxes of 16 v x 64 k
    CUtensorMap dsn;       // dS_next^T per chunk, the same
    CUtensorMap dout;      // dO [tokens][H][128] bf16, boxes of 16 tokens x 1 head x 64 v
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void stsm_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(r0),
                 "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// The warp's 16 x 128 slice of the state fragments (rows v0 .. v0 + 15) to
// row z's entry of the bf16 state array. Lane 0 owns the bulk groups: the
// buffer written now was last read by the store of two chunks ago.
__device__ __forceinline__ void store_state_slice(const float (&acc)[16][4], uint32_t stage_buf,
                                                  const CUtensorMap *map, int v0, int z, int lane) {
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    __syncwarp();
    const int m = lane >> 3, rr = (m & 1) * 8 + (lane & 7);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        const int c = 8 * (j + (m >> 1));   // key column of this lane's row address
        const uint32_t addr = stage_buf + ((c >> 6) << 11) + rr * 128 + ((((c >> 3) & 7) ^ (rr & 7)) << 4);
        stsm_x4(addr, pack_bf16(acc[j][0], acc[j][1]), pack_bf16(acc[j][2], acc[j][3]),
                pack_bf16(acc[j + 1][0], acc[j + 1][1]), pack_bf16(acc[j + 1][2], acc[j + 1][3]));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(map, stage_buf, 0, v0, z);
        tma_store_3d(map, stage_buf + 2048, 64, v0, z);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}

// The chunks of unit n: tokens [tb, te), records from chunk0, nck chunks.
__device__ __forceinline__ void chain_unit(const ChunkGeometry &geo, int n, int64_t &tb, int64_t &te,
                                           int64_t &chunk0, int &nck) {
    if (geo.cu == nullptr) {
        tb = static_cast<int64_t>(n) * geo.seq_len;
        te = tb + geo.seq_len;
        chunk0 = static_cast<int64_t>(n) * geo.chunks_per_seq;
        nck = geo.chunks_per_seq;
    } else {
        tb = geo.cu[n];
        te = geo.cu[n + 1];
        chunk0 = geo.chunk_off[n];
        nck = static_cast<int>((te - tb + 15) / 16);
    }
}

// ---------------------------------------------------------------------------
// Forward chain keeping the states: the recurrent step without outputs, the
// state entering every chunk stored as S^T. unit = (sequence, head, slice).
__device__ __forceinline__ void states_cta(const BwdChunkParams &p, const CUtensorMap *out, int unit,
                                           uint8_t *smem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    constexpr int kSlices = kDim / kCBV;
    const int s = unit % kSlices;
    const int h = (unit / kSlices) % H;
    const int n = unit / (kSlices * H);
    const uint32_t sb = smem_u32(smem);
    const uint32_t stage0 = sb + kStageOff;
    const uint32_t bar_full = stage0 + kStages * kStatesStageBytes;
    const uint32_t bar_empty = bar_full + kStages * 8;
    if (sb & 1023u) {   // the swizzled staging halves need 1024-byte alignment
        if (threadIdx.x == 0) atomicOr(p.err, kErrTimeout);
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, kCWarps * 32);
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (geo.cu != nullptr && (*geo.call_flags & kErrBadCu)) return;
    int64_t tb, te, chunk0;
    int nck;
    chain_unit(geo, n, tb, te, chunk0, nck);
    const uint8_t *rec0 = p.rec + (chunk0 * H + h) * static_cast<int64_t>(kRecBytes);

    if (warp == kCWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < nck; ++i) {
                const int st = i % kStages;
                if (i >= kStages && !mbar_wait(bar_empty + 8 * st, ((i / kStages) - 1) & 1)) {
                    atomicOr(p.err, kErrTimeout);
                    break;
                }
                const uint8_t *src = rec0 + static_cast<int64_t>(i) * H * kRecBytes;
                const uint32_t dst = stage0 + st * kStatesStageBytes;
                mbar_arrive_expect_tx(bar_full + 8 * st, kStatesStageBytes);
                bulk_g2s(dst, src, kRecUt, bar_full + 8 * st);
                bulk_g2s(dst + kRecUt, src + kRecUt + s * kCBV * 32, kCBV * 32, bar_full + 8 * st);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int vw = 16 * warp;
    const int v0 = s * kCBV + vw;
    float acc[16][4];   // S^T fragments: rows = value, cols = key
    recur_load_state(acc, p.s0 != nullptr ? p.s0 + (static_cast<int64_t>(n) * H + h) * kDim * kDim : nullptr, v0);
    const uint32_t buf0 = sb + warp * 8192;
    bool ready = false;
    for (int i = 0; i < nck; ++i) {
        const int st = i % kStages;
        store_state_slice(acc, buf0 + (i & 1) * 4096, out, v0, static_cast<int>((chunk0 + i) * H + h), lane);
        if (!ready && !mbar_wait(bar_full + 8 * st, (i / kStages) & 1)) {
            atomicOr(p.err, kErrTimeout);
            break;
        }
        const int64_t t0 = tb + 16 * static_cast<int64_t>(i);
        ready = recur_step<false>(acc, smem + kStageOff + st * kStatesStageBytes, stage0 + st * kStatesStageBytes,
                                  vw, false, nullptr, nullptr, static_cast<int>(te - t0 < 16 ? te - t0 : 16), H,
                                  [&] {
                                      return i + 1 < nck &&
                                             mbar_test(bar_full + 8 * ((i + 1) % kStages), ((i + 1) / kStages) & 1);
                                  });
        mbar_arrive(bar_empty + 8 * st);
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Reverse chain: the records last chunk first, each with its 16 rows of dO
// for the CTA's 64 values, dS^T in the fragments, dS_next^T of every chunk
// stored, dL/d(initial state) at the end.
__device__ __forceinline__ void chain_cta(const BwdChunkParams &p, const CUtensorMap *out,
                                          const CUtensorMap *dout_map, int unit, uint8_t *smem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tig = lane & 3, quad = lane >> 3;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    constexpr int kSlices = kDim / kCBV;
    const int s = unit % kSlices;
    const int h = (unit / kSlices) % H;
    const int n = unit / (kSlices * H);
    const uint32_t sb = smem_u32(smem);
    const uint32_t stage0 = sb + kStageOff;
    const uint32_t bar_full = stage0 + kStages * kChainStageBytes;
    const uint32_t bar_empty = bar_full + kStages * 8;
    if (sb & 1023u) {
        if (threadIdx.x == 0) atomicOr(p.err, kErrTimeout);
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, kCWarps * 32);
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (geo.cu != nullptr && (*geo.call_flags & kErrBadCu)) return;
    int64_t tb, te, chunk0;
    int nck;
    chain_unit(geo, n, tb, te, chunk0, nck);
    const uint8_t *rec0 = p.rec + (chunk0 * H + h) * static_cast<int64_t>(kRecBytes);

    if (warp == kCWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < nck; ++i) {
                const int st = i % kStages;
                if (i >= kStages && !mbar_wait(bar_empty + 8 * st, ((i / kStages) - 1) & 1)) {
                    atomicOr(p.err, kErrTimeout);
                    break;
                }
                mbar_arrive_expect_tx(bar_full + 8 * st, kChainStageBytes);
                bulk_g2s(stage0 + st * kChainStageBytes,
                         rec0 + static_cast<int64_t>(nck - 1 - i) * H * kRecBytes, kRecUt,
                         bar_full + 8 * st);
                tma_load_3d(stage0 + st * kChainStageBytes + kRecUt, dout_map, s * kCBV, h,
                            static_cast<int>(tb + 16 * static_cast<int64_t>(nck - 1 - i)), bar_full + 8 * st);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int vw = 16 * warp;
    const int v0 = s * kCBV + vw;
    const int64_t sbase = (static_cast<int64_t>(n) * H + h) * kDim * kDim;
    float acc[16][4];   // dS^T fragments: rows = value, cols = key
    recur_load_state(acc, p.dsf != nullptr ? p.dsf + sbase : nullptr, v0);
    const uint32_t buf0 = sb + warp * 8192;

    for (int i = 0; i < nck; ++i) {
        const int c = nck - 1 - i;                   // chunk of the sequence
        const int st = i % kStages;
        // dS_next^T of this chunk (bf16, [v][k]) for the gradient kernel
        store_state_slice(acc, buf0 + (i & 1) * 4096, out, v0, static_cast<int>((chunk0 + c) * H + h), lane);
        if (!mbar_wait(bar_full + 8 * st, (i / kStages) & 1)) {
            atomicOr(p.err, kErrTimeout);
            break;
        }
        const uint8_t *stg = smem + kStageOff + st * kChainStageBytes;
        const uint32_t sw = stage0 + st * kChainStageBytes;
        // dO^T as the A operand (rows vw + gid (+ 8), tokens 2 tig (+ 1), + 8) from
        // the [t][v] tile; tokens past the end of the sequence are zero
        uint32_t aO[4];
        {
            const int m = lane >> 3, t = (m >> 1) * 8 + (lane & 7), vc = vw + (m & 1) * 8;
            ldsm_x4_t(sw + kRecUt + t * 128 + ((((vc >> 3) & 7) ^ (t & 7)) << 4), aO[0], aO[1], aO[2], aO[3]);
            const int64_t t0 = tb + 16 * static_cast<int64_t>(c);
            const int L = static_cast<int>(te - t0 < 16 ? te - t0 : 16);
            if (L < 16) {
                const int ta = 2 * tig;
                const uint32_t lo = (ta < L ? 0x0000ffffu : 0u) | (ta + 1 < L ? 0xffff0000u : 0u);
                const uint32_t hi = (ta + 8 < L ? 0x0000ffffu : 0u) | (ta + 9 < L ? 0xffff0000u : 0u);
                aO[0] &= lo;
                aO[1] &= lo;
                aO[2] &= hi;
                aO[3] &= hi;
            }
        }

        // dS_next^T as bf16 A fragments, one per 16-key step
        uint32_t aD[8][4];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            aD[kk][0] = pack_bf16(acc[2 * kk][0], acc[2 * kk][1]);
            aD[kk][1] = pack_bf16(acc[2 * kk][2], acc[2 * kk][3]);
            aD[kk][2] = pack_bf16(acc[2 * kk + 1][0], acc[2 * kk + 1][1]);
            aD[kk][3] = pack_bf16(acc[2 * kk + 1][2], acc[2 * kk + 1][3]);
        }
        // dU^T = dS_next^T Kd^T + dO^T P (16 values x 16 tokens, two partial sums)
        float uT[2][2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) uT[nt][0][e] = uT[nt][1][e] = 0.f;
        {
            // P as B (k = row r, n = token t): 8x8 blocks (r 0-7 | 8-15) x (t 0-7 | 8-15), transposed
            uint32_t bp[4];
            const int m = lane >> 3;
            ldsm_x4_t(sw + kRecP + (((m & 1) * 8 + (lane & 7)) * 16 + (m >> 1) * 8) * 2, bp[0], bp[1],
                      bp[2], bp[3]);
            mma_r(uT[0][1], aO, bp[0], bp[1]);
            mma_r(uT[1][1], aO, bp[2], bp[3]);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t b[4];
            const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
            ldsm_x4(sw + kRecKd + swz(rb, cb), b[0], b[1], b[2], b[3]);
            mma_r(uT[0][kk & 1], aD[kk], b[0], b[1]);
            mma_r(uT[1][kk & 1], aD[kk], b[2], b[3]);
        }
        // dS^T <- dS_next^T Diag(gamma) + dO^T Qg + dU^T (-W)
        const float *gam = reinterpret_cast<const float *>(stg + kRecGamma);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 gm = *reinterpret_cast<const float2 *>(gam + 8 * j + 2 * tig);
            mul2(acc[j][0], acc[j][1], gm.x, gm.y);
            mul2(acc[j][2], acc[j][3], gm.x, gm.y);
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
#pragma unroll
        for (int jp = 0; jp < 8; ++jp) {
            uint32_t b[4];
            const int rk = (quad & 1) * 8 + (lane & 7), ck = 16 * jp + (quad >> 1) * 8;
            ldsm_x4_t(sw + kRecQg + swz(rk, ck), b[0], b[1], b[2], b[3]);
            mma_r(acc[2 * jp], aO, b[0], b[1]);
            mma_r(acc[2 * jp + 1], aO, b[2], b[3]);
            ldsm_x4_t(sw + kRecW + swz(rk, ck), b[0], b[1], b[2], b[3]);
            mma_r(acc[2 * jp], aU, b[0], b[1]);
            mma_r(acc[2 * jp + 1], aU, b[2], b[3]);
        }
        mbar_arrive(bar_empty + 8 * st);
    }
    if (p.ds0 != nullptr) recur_store_state(acc, p.ds0 + sbase, v0);
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Both chains in one launch: CTAs [0, units) keep the forward states, the
// rest run the reverse chain. Neither waits on the other, so they need not be
// resident together; sharing the launch lets them share the SMs.
__global__ void __launch_bounds__((kCWarps + 1) * 32)
kda_bwd_chains_kernel(const __grid_constant__ BwdChunkParams p, const __grid_constant__ ChainMaps tm,
                      int units) {
    extern __shared__ __align__(1024) uint8_t smem[];
    if (static_cast<int>(blockIdx.x) < units)
        states_cta(p, &tm.ckpt, blockIdx.x, smem);
    else
        chain_cta(p, &tm.dsn, &tm.dout, blockIdx.x - units, smem);
}

// ---------------------------------------------------------------------------
// Chunk-parallel gradients: one 128-thread CTA per (chunk, head) at a time
// (persistent, two CTAs per SM). Shared memory:
constexpr int kGOffST = 0;                  // S^T bf16 [128 v][128 k] as two 64-key halves
                                            //   (128-byte swizzle, by TMA); later fp32
                                            //   [16][kFS] tiles Z, dKd, T1
constexpr int kGOffDT = 32768;              // dS_next^T bf16, the same; later small fp32
                                            //   tiles and the Yc tile
constexpr int kGOffRec = 65536;             // the chunk's record
constexpr int kTStride = 20;                // floats per row of T in shared memory
constexpr int kGOffT = kGOffRec + kRecBytes;             // T = (I + A)^{-1} fp32 [16][20]
constexpr int kGOffV = kGOffT + 16 * kTStride * 4;       // V bf16 [16 t][128 v], swizzled
constexpr int kGOffKg = kGOffV + 4096;      // K e^G bf16 [16 t][128 k], swizzled
constexpr int kGOffKn = kGOffKg + 4096;     // K e^-G bf16 [16 t][128 k], swizzled; in phase 1
                                            //   first k as loaded (bf16 [16][128], row-major)
constexpr int kGOffDO = kGOffKn + 4096;     // dO bf16 [16 t][128 v], swizzled; later dW bf16
constexpr int kGOffUB = kGOffDO + 4096;     // U bf16 [16 t][128 v], swizzled; in phase 1, with
                                            //   the next 4 KiB, g fp32 [16][128] row-major
constexpr int kGOffDUB = kGOffUB + 4096;    // dU bf16 [16 t][128 v], swizzled
constexpr int kGOffQn = kGOffDUB + 4096;    // q as loaded (bf16 [16][128], row-major), then, for
                                            //   chunks factored about the middle of their
                                            //   range, scale Q e^(G - G_ref) bf16, swizzled
constexpr int kGOffMisc = kGOffQn + 4096;   // beta [16], dbeta from M [16], dbeta parts [4][16],
                                            //   the copy barrier, range partials [4][2]
constexpr int kGBar = kGOffMisc + 384;       // the item's g and k (and q)
constexpr int kGBarQ = kGOffMisc + 392;      // a late copy of q
constexpr int kGRed = kGOffMisc + 400;      // range partials [4][2]
constexpr int kGBarS = kGOffMisc + 432;     // the item's S^T, record and T
constexpr int kGBarD = kGOffMisc + 440;     // the item's dS_next^T
constexpr int kGSmem = kGOffMisc + 512;
constexpr uint32_t kGTxBytes = 8192 + 4096;                   // g and k, q aside
constexpr uint32_t kGTxBytesS = 32768 + kRecBytes + 16 * kTStride * 4;   // S^T, record, T
constexpr uint32_t kGTxBytesD = 32768;                        // dS_next^T
static_assert(kGOffT % 16 == 0 && kGOffV % 16 == 0 && kGOffDO % 16 == 0 && kGOffQn % 128 == 0 &&
                  kGOffUB % 128 == 0 && kGOffKn % 128 == 0, "alignment");
// fp32 [16 rows][128 channels] tiles, rows kFS floats apart: the fragment
// stores of eight rows then fall on distinct banks in two wavefronts
constexpr int kFS = 136;
constexpr int kFT = 16 * kFS * 4;
constexpr int kGZ = kGOffST, kGK = kGZ + kFT, kGT1 = kGK + kFT;
// small tiles in the dS_next^T region once it is read
constexpr int kSdP = kGOffDT;               // dP (w.r.t. the record's scale P) [16][16]
constexpr int kSdG = kSdP + 1024;           // dgamma [128] (2 KB kept)
constexpr int kSdMp = kSdG + 2048;          // dM parts [4 warps][16][16]
constexpr int kSdM = kSdMp + 4096;          // dM [16][16]
constexpr int kSdT = kSdM + 1024;           // dT = dM diag(beta)
constexpr int kSY = kSdT + 1024;            // Y = T^T dT
constexpr int kSdA = kSY + 1024;            // dA, strict lower
constexpr int kGYc = kSdA + 1024;           // Yc fp32 [16][kFS]
constexpr int kGGt = kGYc + kFT;            // G - G_ref fp32 [16][128] (for phase 4f's layout)
constexpr int kGTot = kGGt + 8192;          // phase 4f's row-block totals, fp32 [2][4][128]
static_assert(kGT1 + kFT <= kGOffDT && kGTot + 4096 <= kGOffRec, "tiles overlap");
constexpr int kGThreads = 128;

// Byte offset of (row, col) in a [128][128] bf16 tile stored as two
// [128][64] halves, 16-byte chunks swizzled within each 128-byte row (the
// layout of a TMA box with 128-byte swizzling)
__device__ __forceinline__ int sw2(int row, int col) {
    return ((col >> 6) << 14) + row * 128 + ((((col >> 3) & 7) ^ (row & 7)) << 4) + ((col & 7) << 1);
}

struct GradMaps {
    CUtensorMap st, dst;   // S^T and dS_next^T: [items][128 v][128 k] bf16, boxes of 128 v x 64 k
    CUtensorMap g, k, q;   // g fp32, k and q bf16: [tokens][H][128], boxes of 16 tokens x 1 head x 128
};

constexpr float kLog2eG = 1.4426950408889634f;

// D += A * B, m16n8k8, tf32 operands, fp32 accumulate.
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2g(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The A fragment (m16n8k16, row-major 16 x 16) of the matrix el(m, k).
template <typename F>
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], int gid, int tig, F el) {
    const int c0 = 2 * tig, c1 = c0 + 8;
    a[0] = pack_bf16(el(gid, c0), el(gid, c0 + 1));
    a[1] = pack_bf16(el(gid + 8, c0), el(gid + 8, c0 + 1));
    a[2] = pack_bf16(el(gid, c1), el(gid, c1 + 1));
    a[3] = pack_bf16(el(gid + 8, c1), el(gid + 8, c1 + 1));
}

// Per item: phase 1 copies in S^T, dS_next^T, the record, T, V and dO and
// builds K e^G and K e^-G; phase 2 forms U and dU; phase 3 the contractions
// over the values (dW, dQg, dKd, dP, dgamma); phase 4 the WY reverse (dM, dT,
// dbeta, dA), the gated products as MMAs and the per-channel combination.
//
// In the factored range (|G| <= 80 in every channel of the chunk, the same
// test as the forward) the gated products of the reverse factor like the
// forward's: with dY = scale dP, Kn = K e^-G, Qg = scale Q e^G, Kg = K e^G,
//   dq = e^G o (dY Kn + scale dQg)
//   dk = e^G o beta (dA Kn + T^T dW) + e^-G o (dP^T Qg + (diag(beta) dA)^T Kg)
//        + e^(G_last - G) o dKd
// and dG picks the same terms times q or k (with signs + for e^G, - for
// e^-G and e^(G_last - G)). The diagonal of P (exp(0) = 1) stays out of the
// products: its dq and dk terms are added directly and its two dG terms,
// equal and opposite, are left out. Outside the factored range the A and P
// terms take exact per-pair exponentials, one channel per thread.
// The kernel's items. kMid = false compiles out the form factored about the
// middle of a chunk's range (its chunks then take the exact form): the kernel
// takes it for calls whose intra-chunk kernel saw no chunk out of the
// start-referenced range, where carrying that form measured 3 % slower.
template <bool kMid>
__device__ __forceinline__ void grad_items(const BwdChunkParams &p, const GradMaps &tm, uint8_t *smem) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3, quad = lane >> 3;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    if (geo.cu != nullptr && (*geo.call_flags & kErrBadCu)) return;
    const uint32_t sb = smem_u32(smem);
    if (sb & 1023u) {   // the swizzled TMA boxes need 1024-byte alignment
        if (tid == 0) atomicOr(p.err, kErrTimeout);
        return;
    }
    const uint32_t bar = sb + kGBar, bar_q = sb + kGBarQ, bar_s = sb + kGBarS, bar_d = sb + kGBarD;
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(bar_q, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_d, 1);
        mbar_fence_init();
    }
    __syncthreads();
    uint32_t parity = 0, parity_q = 0;
    // q is needed only by chunks factored about the middle of their range; it
    // comes with an item's copies when the CTA's previous item needed it (the
    // decay of a workload changes little from chunk to chunk), else late
    bool want_q = false;
    const uint32_t sST = sb + kGOffST, sDT = sb + kGOffDT, sRec = sb + kGOffRec, sDO = sb + kGOffDO,
                   sUB = sb + kGOffUB, sDUB = sb + kGOffDUB, sT = sb + kGOffT, sV = sb + kGOffV,
                   sKg = sb + kGOffKg, sKn = sb + kGOffKn;
    const int64_t rowe = static_cast<int64_t>(H) * kDim;
    const float scale = p.ip.scale;
    const int64_t items = p.max_chunks * H;
    float *sBeta = reinterpret_cast<float *>(smem + kGOffMisc);
    float *sBM = sBeta + 16, *sPB = sBeta + 32;
    const float *T = reinterpret_cast<const float *>(smem + kGOffT);   // T[r * kTStride + i]
    float *gZ = reinterpret_cast<float *>(smem + kGZ);
    float *gK = reinterpret_cast<float *>(smem + kGK);
    float *gT1 = reinterpret_cast<float *>(smem + kGT1);
    float *gYc = reinterpret_cast<float *>(smem + kGYc);
    float *gP = reinterpret_cast<float *>(smem + kSdP);
    float *sdG = reinterpret_cast<float *>(smem + kSdG);
    float *sdMp = reinterpret_cast<float *>(smem + kSdMp);
    float *sdM = reinterpret_cast<float *>(smem + kSdM);
    float *sdT = reinterpret_cast<float *>(smem + kSdT);
    float *sY = reinterpret_cast<float *>(smem + kSY);
    float *sdA = reinterpret_cast<float *>(smem + kSdA);

    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t c = item / H;
        const int h = static_cast<int>(item - c * H);
        int n, L;
        int64_t t0, rec_idx;
        if (!locate_chunk(geo, c, n, t0, L, rec_idx)) continue;
        (void)n;
        __syncthreads();   // the previous item is done with every tile
        const int64_t qoff = (t0 * H + h) * kDim;

        // ---- phase 1: g, k and q (TMA boxes) first; then S^T (TMA boxes), the
        //      record and T (bulk copies) on a second barrier and dS_next^T on
        //      a third, and V and dO (16-byte copies, rows past the end zero);
        //      thread = channel for G (kept in registers) and the K e^G and
        //      K e^-G tiles, built while the rest is still arriving
        bool exact, middle;
        float Gc[16];       // this channel's G in base-2 units, less G_ref
        float gref = 0.f;   // G_ref in base-2 units
        float eref = 1.f;   // exp(G_ref)
        {
            const int64_t ri = rec_idx * H + h;
            if (warp == 0) {
                if (lane == 0) {
                    // the previous item wrote these tiles through the generic proxy
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive_expect_tx(bar, kGTxBytes + (kMid && want_q ? 4096u : 0u));
                    mbar_arrive_expect_tx(bar_s, kGTxBytesS);
                    mbar_arrive_expect_tx(bar_d, kGTxBytesD);
                }
                __syncwarp();
                if (lane == 0) {
                    const int z = static_cast<int>(ri);
                    tma_load_3d(sUB, &tm.g, 0, h, static_cast<int>(t0), bar);
                    tma_load_3d(sKn, &tm.k, 0, h, static_cast<int>(t0), bar);
                    if (kMid && want_q) tma_load_3d(sb + kGOffQn, &tm.q, 0, h, static_cast<int>(t0), bar);
                    tma_load_3d(sST, &tm.st, 0, 0, z, bar_s);
                    tma_load_3d(sST + 16384, &tm.st, 64, 0, z, bar_s);
                    bulk_g2s(sRec, p.rec + ri * static_cast<int64_t>(kRecBytes), kRecBytes, bar_s);
                    bulk_g2s(sT, p.ip.tinv + ri * (16 * kTStride), 16 * kTStride * 4, bar_s);
                    tma_load_3d(sDT, &tm.dst, 0, 0, z, bar_d);
                    tma_load_3d(sDT + 16384, &tm.dst, 64, 0, z, bar_d);
                }
            }
            const __nv_bfloat16 *dop = static_cast<const __nv_bfloat16 *>(p.dout) + qoff;
            const __nv_bfloat16 *vp = static_cast<const __nv_bfloat16 *>(p.ip.v) + qoff;
            for (int i = tid; i < 256; i += kGThreads) {
                const int r = i >> 4, cc = i & 15;
                const bool ok = r < L;
                const uint32_t dst = r * 256 + ((cc ^ (r & 7)) << 4);
                cp_async16(sDO + dst, dop + (ok ? r : 0) * rowe + cc * 8, ok ? 16u : 0u);
                cp_async16(sV + dst, vp + (ok ? r : 0) * rowe + cc * 8, ok ? 16u : 0u);
            }
            cp_async_commit();
            if (tid < 16) sBeta[tid] = tid < L ? __ldg(p.ip.beta + (t0 + tid) * H + h) : 0.f;
            const bool got = mbar_wait(bar, parity);
            if (__syncthreads_or(!got)) {
                // give the copies in flight another bounded wait, then stop
                if (tid == 0) atomicOr(p.err, kErrTimeout);
                if (!got) mbar_wait(bar, parity);
                mbar_wait(bar_s, parity);
                mbar_wait(bar_d, parity);
                cp_async_wait_all();
                break;
            }
            // G = running sum of g (rows past the end: zero): its largest |G|, its
            // range from the chunk start on and its largest rise (nats)
            const float *gs = reinterpret_cast<const float *>(smem + kGOffUB) + tid;
            const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(smem + kGOffKn) + tid;
            float run = 0.f, gmax = 0.f, kr[16], hi = 0.f, low = 0.f, rise = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const bool ok = r < L;
                run += ok ? gs[r * kDim] : 0.f;
                gmax = fmaxf(gmax, fabsf(run));
                if constexpr (kMid) {
                    rise = fmaxf(rise, run - low);
                    low = fminf(low, run);
                    hi = fmaxf(hi, run);
                }
                kr[r] = ok ? __bfloat162float(ks[r * kDim]) : 0.f;
                Gc[r] = run * kLog2eG;
            }
            // The chunk's form, as in the forward: the gated products factor about
            // G_ref = 0 while |G| <= 80, else about the middle of G's range while
            // that range is at most 160 and G rises by at most 80; beyond, exact
            exact = false;
            middle = false;
            if constexpr (!kMid) {
                exact = __syncthreads_or(!(gmax <= 80.f)) != 0;   // (also: k as loaded is read)
            } else {
                if (__syncthreads_or(!(gmax <= 80.f))) {   // (also: k as loaded is read)
                    float *red = reinterpret_cast<float *>(smem + kGRed);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
                        low = fminf(low, __shfl_xor_sync(0xffffffffu, low, o));
                    }
                    if (lane == 0) { red[2 * warp] = hi; red[2 * warp + 1] = low; }
                    const bool big_rise = __syncthreads_or(!(rise <= 80.f)) != 0;
                    hi = fmaxf(fmaxf(red[0], red[2]), fmaxf(red[4], red[6]));
                    low = fminf(fminf(red[1], red[3]), fminf(red[5], red[7]));
                    exact = big_rise || !(hi - low <= 160.f);
                    middle = !exact;
                }
                if (middle && !want_q) {
                    // q was not among the item's copies: fetch it now
                    if (tid == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        mbar_arrive_expect_tx(bar_q, 4096u);
                        tma_load_3d(sb + kGOffQn, &tm.q, 0, h, static_cast<int>(t0), bar_q);
                    }
                    const bool got_q = mbar_wait(bar_q, parity_q);
                    parity_q ^= 1u;
                    if (__syncthreads_or(!got_q)) {
                        if (tid == 0) atomicOr(p.err, kErrTimeout);
                        if (!got_q) mbar_wait(bar_q, parity_q ^ 1u);
                        mbar_wait(bar_s, parity);
                        mbar_wait(bar_d, parity);
                        cp_async_wait_all();
                        break;
                    }
                }
                want_q = middle;
                if (middle) {
                    // G now holds G - G_ref; this channel's column of scale Q e^(G - G_ref)
                    gref = 0.5f * (hi + low) * kLog2eG;
                    eref = ex2g(gref);
                    const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(smem + kGOffQn) + tid;
                    float qr[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        Gc[r] -= gref;
                        qr[r] = r < L ? __bfloat162float(qs[r * kDim]) : 0.f;
                    }
                    __syncthreads();   // q as loaded is read; its space takes the tile
#pragma unroll
                    for (int r = 0; r < 16; ++r)
                        *reinterpret_cast<__nv_bfloat16 *>(smem + kGOffQn + swz(r, tid)) =
                            __float2bfloat16_rn(scale * qr[r] * ex2g(Gc[r]));
                }
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                *reinterpret_cast<__nv_bfloat16 *>(smem + kGOffKg + swz(r, tid)) =
                    __float2bfloat16_rn(kr[r] * ex2g(Gc[r]));
                *reinterpret_cast<__nv_bfloat16 *>(smem + kGOffKn + swz(r, tid)) =
                    __float2bfloat16_rn(kr[r] * ex2g(-Gc[r]));
            }
            // S^T, the record and T, and V and dO
            cp_async_wait_all();
            const bool got_s = mbar_wait(bar_s, parity);
            if (__syncthreads_or(!got_s)) {
                if (tid == 0) atomicOr(p.err, kErrTimeout);
                if (!got_s) mbar_wait(bar_s, parity);
                mbar_wait(bar_d, parity);
                break;
            }
        }
        // scale Q e^(G - G_ref): the record's scale Q e^G when G_ref = 0
        const uint32_t sQs = kMid && middle ? sb + kGOffQn : sRec + kRecQg;

        // ---- phase 2: U^T = Ut^T + S^T (-W)^T, value rows 32 warp + 16 mt, all 16
        //      tokens; then, once dS_next^T is in, dU^T = dS_next^T Kd^T + dO^T P
        const int m2 = lane >> 3;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const int vb = 32 * warp + 16 * mt;
            float uT[2][2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tk = 8 * nt + 2 * tig;
                const float2 u01 = unpack_bf16(*reinterpret_cast<const uint32_t *>(
                    smem + kGOffRec + kRecUt + ((vb + gid) * 16 + tk) * 2));
                const float2 u23 = unpack_bf16(*reinterpret_cast<const uint32_t *>(
                    smem + kGOffRec + kRecUt + ((vb + gid + 8) * 16 + tk) * 2));
                uT[nt][0][0] = u01.x; uT[nt][0][1] = u01.y; uT[nt][0][2] = u23.x; uT[nt][0][3] = u23.y;
#pragma unroll
                for (int e = 0; e < 4; ++e) uT[nt][1][e] = 0.f;
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t aS[4], bw[4];
                const int ra = vb + (lane & 7) + 8 * ((lane >> 3) & 1), ca = 16 * kk + 8 * (lane >> 4);
                ldsm_x4(sST + sw2(ra, ca), aS[0], aS[1], aS[2], aS[3]);
                const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
                ldsm_x4(sRec + kRecW + swz(rb, cb), bw[0], bw[1], bw[2], bw[3]);
                mma_r(uT[0][kk & 1], aS, bw[0], bw[1]);
                mma_r(uT[1][kk & 1], aS, bw[2], bw[3]);
            }
            float u[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) u[nt][e] = uT[nt][0][e] + uT[nt][1][e];
            // U to its [t][v] tile (bf16), transposed by stmatrix
            stsm_x4_t(sUB + swz(8 * (m2 >> 1) + (lane & 7), vb + 8 * (m2 & 1)), pack_bf16(u[0][0], u[0][1]),
                      pack_bf16(u[0][2], u[0][3]), pack_bf16(u[1][0], u[1][1]), pack_bf16(u[1][2], u[1][3]));
        }
        {
            const bool got_d = mbar_wait(bar_d, parity);
            parity ^= 1u;
            if (__syncthreads_or(!got_d)) {
                if (tid == 0) atomicOr(p.err, kErrTimeout);
                if (!got_d) mbar_wait(bar_d, parity ^ 1u);
                break;
            }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const int vb = 32 * warp + 16 * mt;
            float dT[2][2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) { dT[nt][0][e] = 0.f; dT[nt][1][e] = 0.f; }
            {
                // dO^T (v x t) from the [t][v] tile, transposed; P as B (r x t), transposed
                uint32_t aO[4], bp[4];
                ldsm_x4_t(sDO + swz((lane & 7) + 8 * (m2 >> 1), vb + 8 * (m2 & 1)), aO[0], aO[1], aO[2], aO[3]);
                ldsm_x4_t(sRec + kRecP + (((m2 & 1) * 8 + (lane & 7)) * 16 + (m2 >> 1) * 8) * 2, bp[0], bp[1],
                          bp[2], bp[3]);
                mma_r(dT[0][1], aO, bp[0], bp[1]);
                mma_r(dT[1][1], aO, bp[2], bp[3]);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t aD[4], bk[4];
                const int ra = vb + (lane & 7) + 8 * ((lane >> 3) & 1), ca = 16 * kk + 8 * (lane >> 4);
                ldsm_x4(sDT + sw2(ra, ca), aD[0], aD[1], aD[2], aD[3]);
                const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
                ldsm_x4(sRec + kRecKd + swz(rb, cb), bk[0], bk[1], bk[2], bk[3]);
                mma_r(dT[0][kk & 1], aD, bk[0], bk[1]);
                mma_r(dT[1][kk & 1], aD, bk[2], bk[3]);
            }
            float du[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) du[nt][e] = dT[nt][0][e] + dT[nt][1][e];
            stsm_x4_t(sDUB + swz(8 * (m2 >> 1) + (lane & 7), vb + 8 * (m2 & 1)), pack_bf16(du[0][0], du[0][1]),
                      pack_bf16(du[0][2], du[0][3]), pack_bf16(du[1][0], du[1][1]), pack_bf16(du[1][2], du[1][3]));
        }
        __syncthreads();

        // ---- phase 3: contractions over the 128 values. Warp w: keys 32 w .. + 31.
        //      dW = -dU S^T, dQg = dO S^T, dKd = U dS_next^T; warp 0 also dP = dO U^T;
        //      dgamma = rowsum(dS_next o S) as the diagonal of the 16 x 16 blocks
        //      S dS_next^T of the warp's keys (the S^T fragments loaded as B serve
        //      as A: both hold two consecutive values of one key)
        float cW[4][4], cQ[4][4], cK[4][4], cP[2][4], cG[2][2][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) cW[j][e] = cQ[j][e] = cK[j][e] = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) cP[j][e] = cG[j][0][e] = cG[j][1][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t aU_[4], aO_[4], aDU[4];
            const int ra = (lane & 7) + 8 * ((lane >> 3) & 1), ca = 16 * kk + 8 * (lane >> 4);
            ldsm_x4(sDUB + swz(ra, ca), aDU[0], aDU[1], aDU[2], aDU[3]);
            ldsm_x4(sDO + swz(ra, ca), aO_[0], aO_[1], aO_[2], aO_[3]);
            ldsm_x4(sUB + swz(ra, ca), aU_[0], aU_[1], aU_[2], aU_[3]);
#pragma unroll
            for (int jp = 0; jp < 2; ++jp) {
                uint32_t bs[4], bd[4];
                const int rk = 16 * kk + (quad & 1) * 8 + (lane & 7), ck = 32 * warp + 16 * jp + (quad >> 1) * 8;
                ldsm_x4_t(sST + sw2(rk, ck), bs[0], bs[1], bs[2], bs[3]);
                ldsm_x4_t(sDT + sw2(rk, ck), bd[0], bd[1], bd[2], bd[3]);
                mma_r(cW[2 * jp], aDU, bs[0], bs[1]);
                mma_r(cW[2 * jp + 1], aDU, bs[2], bs[3]);
                mma_r(cQ[2 * jp], aO_, bs[0], bs[1]);
                mma_r(cQ[2 * jp + 1], aO_, bs[2], bs[3]);
                mma_r(cK[2 * jp], aU_, bd[0], bd[1]);
                mma_r(cK[2 * jp + 1], aU_, bd[2], bd[3]);
                const uint32_t aS[4] = {bs[0], bs[2], bs[1], bs[3]};   // S: 16 keys x 16 values
                mma_r(cG[jp][0], aS, bd[0], bd[1]);
                mma_r(cG[jp][1], aS, bd[2], bd[3]);
            }
            if (warp == 0) {
                uint32_t bu[4];
                const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
                ldsm_x4(sUB + swz(rb, cb), bu[0], bu[1], bu[2], bu[3]);
                mma_r(cP[0], aO_, bu[0], bu[1]);
                mma_r(cP[1], aO_, bu[2], bu[3]);
            }
        }
        __syncthreads();
        // results: dQg, dKd fp32 over S^T; dW bf16 over dO; dP and dgamma over
        // dS_next^T
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int key = 32 * warp + 8 * j + 2 * tig;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int t = gid + 8 * hf;
                *reinterpret_cast<float2 *>(gZ + t * kFS + key) = make_float2(cQ[j][2 * hf], cQ[j][2 * hf + 1]);
                *reinterpret_cast<float2 *>(gK + t * kFS + key) = make_float2(cK[j][2 * hf], cK[j][2 * hf + 1]);
                *reinterpret_cast<uint32_t *>(smem + kGOffDO + swz(t, key)) =
                    pack_bf16(-cW[j][2 * hf], -cW[j][2 * hf + 1]);
            }
        }
        if (warp == 0) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int r = gid + 8 * hf, i = 8 * nt + 2 * tig;
                    gP[r * 16 + i] = i <= r ? cP[nt][2 * hf] : 0.f;
                    gP[r * 16 + i + 1] = i + 1 <= r ? cP[nt][2 * hf + 1] : 0.f;
                }
        }
        if (tig == (gid >> 1)) {
            // the diagonal: row gid of the first n-tile, row gid + 8 of the second
            const bool odd = gid & 1;
#pragma unroll
            for (int jp = 0; jp < 2; ++jp) {
                const int kb = 32 * warp + 16 * jp;
                sdG[kb + gid] = odd ? cG[jp][0][1] : cG[jp][0][0];
                sdG[kb + 8 + gid] = odd ? cG[jp][1][3] : cG[jp][1][2];
            }
        }
        __syncthreads();

        // ---- phase 4a: dM = dU V^T + dW Kg^T (16 x 16), warp w over channels 32 w .. + 31
        //      (the tile holds K e^(G - G_ref): its product is scaled by exp(G_ref))
        {
            float m2[2][4] = {}, m3[2][4] = {};
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const int kk = 2 * warp + q2;
                uint32_t aD[4], aW[4], bv[4], bg[4];
                const int ra = (lane & 7) + 8 * ((lane >> 3) & 1), ca = 16 * kk + 8 * (lane >> 4);
                ldsm_x4(sDUB + swz(ra, ca), aD[0], aD[1], aD[2], aD[3]);
                ldsm_x4(sDO + swz(ra, ca), aW[0], aW[1], aW[2], aW[3]);   // dW
                const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
                ldsm_x4(sV + swz(rb, cb), bv[0], bv[1], bv[2], bv[3]);
                ldsm_x4(sKg + swz(rb, cb), bg[0], bg[1], bg[2], bg[3]);
                mma_r(m2[0], aD, bv[0], bv[1]);
                mma_r(m2[1], aD, bv[2], bv[3]);
                if constexpr (kMid) {
                    mma_r(m3[0], aW, bg[0], bg[1]);
                    mma_r(m3[1], aW, bg[2], bg[3]);
                } else {
                    mma_r(m2[0], aW, bg[0], bg[1]);
                    mma_r(m2[1], aW, bg[2], bg[3]);
                }
            }
            if constexpr (kMid) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) m2[nt][e] = fmaf(eref, m3[nt][e], m2[nt][e]);
            }
            float *part = sdMp + warp * 256;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int r = gid + 8 * hf, i = 8 * nt + 2 * tig;
                    *reinterpret_cast<float2 *>(part + r * 16 + i) = make_float2(m2[nt][2 * hf], m2[nt][2 * hf + 1]);
                }
        }
        __syncthreads();
        // ---- phase 4b: dM and dT = dM diag(beta) (M = T diag(beta)); two entries per thread
#pragma unroll
        for (int e = tid; e < 256; e += kGThreads) {
            const float m = sdMp[e] + sdMp[256 + e] + sdMp[512 + e] + sdMp[768 + e];
            sdM[e] = m;
            sdT[e] = m * sBeta[e & 15];
        }
        __syncthreads();
        // ---- phase 4c (warp 0): Y = T^T dT and dA = -(Y T^T) on the strict lower
        //      triangle, as tf32 MMAs (m16n8k8); dbeta_j (from M) = sum_r dM[r][j] T[r][j]
        if (warp == 0) {
            auto tf = [](float x) {
                uint32_t r;
                asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
                return r;
            };
            float y[2][4] = {};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int a = 8 * ks + tig;
                const uint32_t a0 = tf(T[a * kTStride + gid]), a1 = tf(T[a * kTStride + gid + 8]);
                const uint32_t a2 = tf(T[(a + 4) * kTStride + gid]), a3 = tf(T[(a + 4) * kTStride + gid + 8]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    mma_tf32(y[nt], a0, a1, a2, a3, tf(sdT[a * 16 + 8 * nt + gid]),
                             tf(sdT[(a + 4) * 16 + 8 * nt + gid]));
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                *reinterpret_cast<float2 *>(sY + gid * 16 + 8 * nt + 2 * tig) = make_float2(y[nt][0], y[nt][1]);
                *reinterpret_cast<float2 *>(sY + (gid + 8) * 16 + 8 * nt + 2 * tig) = make_float2(y[nt][2], y[nt][3]);
            }
            __syncwarp();
            float da[2][4] = {};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int b = 8 * ks + tig;
                const uint32_t a0 = tf(sY[gid * 16 + b]), a1 = tf(sY[(gid + 8) * 16 + b]);
                const uint32_t a2 = tf(sY[gid * 16 + b + 4]), a3 = tf(sY[(gid + 8) * 16 + b + 4]);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
                    mma_tf32(da[nt], a0, a1, a2, a3, tf(T[(8 * nt + gid) * kTStride + b]),
                             tf(T[(8 * nt + gid) * kTStride + b + 4]));
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int r = gid + 8 * hf, i = 8 * nt + 2 * tig;
                    *reinterpret_cast<float2 *>(sdA + r * 16 + i) =
                        make_float2(i < r ? -da[nt][2 * hf] : 0.f, i + 1 < r ? -da[nt][2 * hf + 1] : 0.f);
                }
            if (lane < 16) {
                float sbj = 0.f;
#pragma unroll
                for (int r = 0; r < 16; ++r) sbj = fmaf(sdM[r * 16 + lane], T[r * kTStride + lane], sbj);
                sBM[lane] = sbj;
            }
        }
        __syncthreads();

        // ---- phase 4e: the products over the chunk's tokens, warp w: channels 32 w .. + 31
        {
            // (this channel's G for phase 4f, whose threads hold other channels)
            float *sGt = reinterpret_cast<float *>(smem + kGGt);
#pragma unroll
            for (int r = 0; r < 16; ++r) sGt[r * kDim + tid] = Gc[r];
            uint32_t aTt[4];
            frag_a(aTt, gid, tig, [&](int m, int k) { return T[k * kTStride + m]; });
            float zc[4][4], xc[4][4], dc[4][4], uc[4][4], yc[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) zc[j][e] = xc[j][e] = dc[j][e] = uc[j][e] = yc[j][e] = 0.f;
            const int rk = (quad & 1) * 8 + (lane & 7);
#pragma unroll
            for (int jp = 0; jp < 2; ++jp) {
                const int ck = 32 * warp + 16 * jp + (quad >> 1) * 8;
                uint32_t b[4];
                ldsm_x4_t(sDO + swz(rk, ck), b[0], b[1], b[2], b[3]);    // dW
                mma_r(dc[2 * jp], aTt, b[0], b[1]);
                mma_r(dc[2 * jp + 1], aTt, b[2], b[3]);
                ldsm_x4_t(sDUB + swz(rk, ck), b[0], b[1], b[2], b[3]);   // dU
                mma_r(uc[2 * jp], aTt, b[0], b[1]);
                mma_r(uc[2 * jp + 1], aTt, b[2], b[3]);
            }
            if (!exact) {
                uint32_t aY[4], aA[4], aYt[4], aAt[4];
                // the diagonal of P (exp(0) = 1) is left to the combination below
                frag_a(aY, gid, tig, [&](int m, int k) { return m == k ? 0.f : scale * gP[m * 16 + k]; });
                frag_a(aA, gid, tig, [&](int m, int k) { return sdA[m * 16 + k]; });
                frag_a(aYt, gid, tig, [&](int m, int k) { return m == k ? 0.f : gP[k * 16 + m]; });
                frag_a(aAt, gid, tig, [&](int m, int k) { return sBeta[k] * sdA[k * 16 + m]; });
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    const int ck = 32 * warp + 16 * jp + (quad >> 1) * 8;
                    uint32_t b[4];
                    ldsm_x4_t(sKn + swz(rk, ck), b[0], b[1], b[2], b[3]);
                    mma_r(zc[2 * jp], aY, b[0], b[1]);
                    mma_r(zc[2 * jp + 1], aY, b[2], b[3]);
                    mma_r(xc[2 * jp], aA, b[0], b[1]);
                    mma_r(xc[2 * jp + 1], aA, b[2], b[3]);
                    ldsm_x4_t(sQs + swz(rk, ck), b[0], b[1], b[2], b[3]);
                    mma_r(yc[2 * jp], aYt, b[0], b[1]);
                    mma_r(yc[2 * jp + 1], aYt, b[2], b[3]);
                    ldsm_x4_t(sKg + swz(rk, ck), b[0], b[1], b[2], b[3]);
                    mma_r(yc[2 * jp], aAt, b[0], b[1]);
                    mma_r(yc[2 * jp + 1], aAt, b[2], b[3]);
                }
            }
            // epilogue: Z = dY Kn + exp(G_ref) scale dQg, T1 = beta (dA Kn +
            // exp(G_ref) T^T dW), Yc, dv = beta T^T dU; dbeta parts sum_c Kg (dA Kn)
            // (Kn, Kg about G_ref: the terms that carry e^G itself are brought to
            // e^(G - G_ref) here; exp(G_ref) = 1 for chunks factored about the start)
            const float sref = scale * eref;
            float pb0 = 0.f, pb1 = 0.f;
            const float b0 = sBeta[gid], b1 = sBeta[gid + 8];
            float *dvp = p.dv + qoff;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = 32 * warp + 8 * j + 2 * tig;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int r = gid + 8 * hf;
                    const float br = hf ? b1 : b0;
                    const float x0 = xc[j][2 * hf], x1 = xc[j][2 * hf + 1];
                    float2 *zp = reinterpret_cast<float2 *>(gZ + r * kFS + col);
                    const float2 q2 = *zp;
                    *zp = make_float2(fmaf(sref, q2.x, zc[j][2 * hf]), fmaf(sref, q2.y, zc[j][2 * hf + 1]));
                    *reinterpret_cast<float2 *>(gT1 + r * kFS + col) =
                        make_float2(br * fmaf(eref, dc[j][2 * hf], x0), br * fmaf(eref, dc[j][2 * hf + 1], x1));
                    *reinterpret_cast<float2 *>(gYc + r * kFS + col) = make_float2(yc[j][2 * hf], yc[j][2 * hf + 1]);
                    const float2 kg = unpack_bf16(*reinterpret_cast<const uint32_t *>(smem + kGOffKg + swz(r, col)));
                    const float pb = fmaf(kg.x, x0, kg.y * x1);
                    if (hf) pb1 += pb; else pb0 += pb;
                    if (r < L)
                        *reinterpret_cast<float2 *>(dvp + r * rowe + col) =
                            make_float2(br * uc[j][2 * hf], br * uc[j][2 * hf + 1]);
                }
            }
            if (!exact) {
#pragma unroll
                for (int o = 1; o < 4; o <<= 1) {
                    pb0 += __shfl_xor_sync(0xffffffffu, pb0, o);
                    pb1 += __shfl_xor_sync(0xffffffffu, pb1, o);
                }
                if (tig == 0) {
                    sPB[warp * 16 + gid] = pb0;
                    sPB[warp * 16 + gid + 8] = pb1;
                }
            }
        }
        __syncthreads();

        // ---- phase 4f: the combination. Factored forms: warp w takes rows 4 w .. + 3,
        //      lane l channels 4 l .. + 3 (128- and 64-bit shared loads, 16-byte
        //      stores); the exact form: thread = channel, all 16 rows
        if (!exact) {
            const int c0 = 4 * lane, rb = 4 * warp;
            const float *sGt = reinterpret_cast<const float *>(smem + kGGt);
            float *sTot = reinterpret_cast<float *>(smem + kGTot);   // [0]: dG sums, [1]: kdv sums
            // q and k enter through the tiles scale Q e^(G - G_ref), K e^(G - G_ref),
            // K e^(G_ref - G) and the record's K e^(G_last - G); G here is less G_ref
            const float inv_scale = scale != 0.f ? 1.f / scale : 0.f;
            const float4 gl4 = *reinterpret_cast<const float4 *>(sGt + 15 * kDim + c0);
            const float gL[4] = {gl4.x, gl4.y, gl4.z, gl4.w};
            // e^(G_last - G) = e^(G_last - G_ref) e^(G_ref - G): both within e^+-80 here
            float eLr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) eLr[e] = ex2g(gL[e]);
            float dG[4][4];    // dG less the K e^(G_last - G) terms
            float kdv[4][4];   // those terms: k e^(G_last - G) dKd
            auto bf4 = [](uint2 u, float (&f)[4]) {
                const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y);
                f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
            };
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = rb + i;
                const float4 g4 = *reinterpret_cast<const float4 *>(sGt + r * kDim + c0);
                const float4 z4 = *reinterpret_cast<const float4 *>(gZ + r * kFS + c0);
                const float4 t4 = *reinterpret_cast<const float4 *>(gT1 + r * kFS + c0);
                const float4 y4 = *reinterpret_cast<const float4 *>(gYc + r * kFS + c0);
                const float4 d4 = *reinterpret_cast<const float4 *>(gK + r * kFS + c0);
                const int o16 = swz(r, c0);   // channels c0 .. c0 + 3: 8 bytes of one 16-byte chunk
                float qs[4], kd[4], kgv[4], knv[4];
                bf4(*reinterpret_cast<const uint2 *>(smem + (sQs - sb) + o16), qs);
                bf4(*reinterpret_cast<const uint2 *>(smem + kGOffRec + kRecKd + o16), kd);
                bf4(*reinterpret_cast<const uint2 *>(smem + kGOffKg + o16), kgv);
                bf4(*reinterpret_cast<const uint2 *>(smem + kGOffKn + o16), knv);
                const float G[4] = {g4.x, g4.y, g4.z, g4.w}, z[4] = {z4.x, z4.y, z4.z, z4.w};
                const float t1[4] = {t4.x, t4.y, t4.z, t4.w}, yc[4] = {y4.x, y4.y, y4.z, y4.w};
                const float dkd[4] = {d4.x, d4.y, d4.z, d4.w};
                const float yd = scale * gP[r * 17];   // the diagonal pair: its dG terms cancel
                float dq[4], dk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float eG = ex2g(G[e]), eN = ex2g(-G[e]), eD = eLr[e] * eN;
                    const float qgs = qs[e] * inv_scale;
                    // q dq = (q e^G) Z, k a = (k e^G) T1, k b = (k e^-G) Yc, k d = Kd dKd
                    // (each e^G here is e^(G - G_ref), e^-G is e^(G_ref - G))
                    kdv[i][e] = kd[e] * dkd[e];
                    dG[i][e] = fmaf(qgs, z[e], fmaf(kgv[e], t1[e], -knv[e] * yc[e]));
                    dq[e] = fmaf(yd, knv[e] * eG, eG * z[e]);
                    dk[e] = fmaf(yd, qgs * eN, fmaf(eG, t1[e], fmaf(eN, yc[e], eD * dkd[e])));
                }
                if (r < L) {
                    const int64_t o = qoff + r * rowe + c0;
                    *reinterpret_cast<float4 *>(p.dq + o) = make_float4(dq[0], dq[1], dq[2], dq[3]);
                    *reinterpret_cast<float4 *>(p.dk + o) = make_float4(dk[0], dk[1], dk[2], dk[3]);
                }
            }
            if (warp == 3) {
                // the last row also takes dgamma e^(G_last)
#pragma unroll
                for (int e = 0; e < 4; ++e) dG[3][e] = fmaf(sdG[c0 + e], ex2g(gL[e] + gref), dG[3][e]);
            }
            // dg_u = sum_{r >= u} dG_r + sum_{r < u} kdv_r (see the exact form below):
            // within the block, then the other blocks' totals
            float sfx[4][4], pfx[4][4], tS[4], tK[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float a = 0.f, b = 0.f;
#pragma unroll
                for (int i = 3; i >= 0; --i) { a += dG[i][e]; sfx[i][e] = a; }
#pragma unroll
                for (int i = 0; i < 4; ++i) { pfx[i][e] = b; b += kdv[i][e]; }
                tS[e] = a;
                tK[e] = b;
            }
            *reinterpret_cast<float4 *>(sTot + warp * kDim + c0) = make_float4(tS[0], tS[1], tS[2], tS[3]);
            *reinterpret_cast<float4 *>(sTot + 4 * kDim + warp * kDim + c0) = make_float4(tK[0], tK[1], tK[2], tK[3]);
            __syncthreads();
            float addS[4] = {0.f, 0.f, 0.f, 0.f}, addK[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int w2 = 0; w2 < 4; ++w2) {
                if (w2 > warp) {
                    const float4 v = *reinterpret_cast<const float4 *>(sTot + w2 * kDim + c0);
                    addS[0] += v.x; addS[1] += v.y; addS[2] += v.z; addS[3] += v.w;
                } else if (w2 < warp) {
                    const float4 v = *reinterpret_cast<const float4 *>(sTot + 4 * kDim + w2 * kDim + c0);
                    addK[0] += v.x; addK[1] += v.y; addK[2] += v.z; addK[3] += v.w;
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = rb + i;
                if (r < L)
                    *reinterpret_cast<float4 *>(p.dg + qoff + r * rowe + c0) =
                        make_float4(sfx[i][0] + addS[0] + (pfx[i][0] + addK[0]),
                                    sfx[i][1] + addS[1] + (pfx[i][1] + addK[1]),
                                    sfx[i][2] + addS[2] + (pfx[i][2] + addK[2]),
                                    sfx[i][3] + addS[3] + (pfx[i][3] + addK[3]));
            }
        } else {
            const int ch = tid;
            const int64_t base = qoff + ch;
            float dG[16];    // dG less the K e^(G_last - G) terms
            float kdv[16];   // those terms: k e^(G_last - G) dKd per row
            const float G2L = Gc[15];
            float dGL = sdG[ch] * ex2g(G2L + gref);
            {
                // exact per-pair exponentials for the P and A terms
                const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.ip.q);
                const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(p.ip.k);
                float kk_[16], qq[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const bool ok = r < L;
                    kk_[r] = ok ? __bfloat162float(kg[base + r * rowe]) : 0.f;
                    qq[r] = ok ? __bfloat162float(qg[base + r * rowe]) : 0.f;
                }
                float dk[16], dq[16], pb[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) { dk[r] = 0.f; dq[r] = 0.f; dG[r] = 0.f; pb[r] = 0.f; }
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const float br = sBeta[r];
#pragma unroll
                    for (int i = 0; i <= r; ++i) {
                        const float E = ex2g(Gc[r] - Gc[i]);
                        const float wP = scale * gP[r * 16 + i] * E;
                        dq[r] = fmaf(wP, kk_[i], dq[r]);
                        dk[i] = fmaf(wP, qq[r], dk[i]);
                        if (i < r) {
                            // (the diagonal pair's two dG terms cancel: left out)
                            const float tP = wP * qq[r] * kk_[i];
                            dG[r] += tP;
                            dG[i] -= tP;
                            const float dAr = sdA[r * 16 + i];
                            const float kkE = kk_[r] * kk_[i] * E;
                            pb[r] = fmaf(dAr, kkE, pb[r]);
                            const float wA = br * dAr * E;
                            dk[r] = fmaf(wA, kk_[i], dk[r]);
                            dk[i] = fmaf(wA, kk_[r], dk[i]);
                            const float tA = br * dAr * kkE;
                            dG[r] += tA;
                            dG[i] -= tA;
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const float eG = ex2g(Gc[r]), eD = ex2g(G2L - Gc[r]);
                    const float q1 = eG * gZ[r * kFS + ch];
                    const float a = eG * gT1[r * kFS + ch];
                    const float d = eD * gK[r * kFS + ch];
                    dG[r] = fmaf(qq[r], q1, fmaf(kk_[r], a, dG[r]));
                    kdv[r] = kk_[r] * d;
                    if (r < L) {
                        const int64_t o = base + r * rowe;
                        p.dq[o] = dq[r] + q1;
                        p.dk[o] = dk[r] + a + d;
                    }
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float x = pb[r];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                    if (lane == 0) sPB[warp * 16 + r] = x;
                }
            }
            dG[15] += dGL;
            // dg = reverse cumulative sum of the full dG over the rows. Each row's
            // K e^(G_last - G) term enters its own row with - and the last row with
            // + (through G_last), so it cancels in dg_u for u at or before its row;
            // summed as dg_u = sum_{r >= u} dG_r + sum_{r < u} kdv_r it cancels
            // exactly (under strong decay dg is far below those terms)
            float kpre = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float x = kdv[r];
                kdv[r] = kpre;
                kpre += x;
            }
            float acc = 0.f;
#pragma unroll
            for (int r = 15; r >= 0; --r) {
                acc += dG[r];
                if (r < L) p.dg[base + r * rowe] = acc + kdv[r];
            }
        }
        __syncthreads();
        if (tid < 16 && tid < L)
            p.dbeta[(t0 + tid) * H + h] = sBM[tid] + sPB[tid] + sPB[16 + tid] + sPB[32 + tid] + sPB[48 + tid];
    }
}

__global__ void __launch_bounds__(kGThreads, 2)
kda_bwd_grad_kernel(const __grid_constant__ BwdChunkParams p, const __grid_constant__ GradMaps tm) {
    extern __shared__ __align__(1024) uint8_t smem[];
    // p.wide[0]: raised by this call's intra-chunk kernel for a chunk out of the
    // start-referenced range (a stale raise costs time only: the other form
    // handles every chunk too)
    if (p.wide != nullptr && __ldcg(p.wide) != 0)
        grad_items<true>(p, tm, smem);
    else
        grad_items<false>(p, tm, smem);
    if (p.wide != nullptr) {
        // the last CTA to finish lowers the flag and its own counter for the next call
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(p.wide + 1, 1) == static_cast<int>(gridDim.x) - 1) {
                p.wide[0] = 0;
                p.wide[1] = 0;
                __threadfence();
            }
        }
    }
}

}  // namespace

namespace {

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// [items][128 v][128 k] bf16 with boxes of `rows` values x 64 keys, 128-byte swizzle
bool encode_states(EncodeFn enc, CUtensorMap *m, const void *base, int64_t items, uint32_t rows) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(kDim),
                                static_cast<cuuint64_t>(items)};
    const cuuint64_t strides[2] = {kDim * 2, kDim * kDim * 2};
    const cuuint32_t box[3] = {64, rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [tokens][H][128] rows with boxes of 16 tokens x 1 head x `width` channels: 128
// without swizzle, or 64 bf16 (128 bytes) with 128-byte swizzle
bool encode_rows16(EncodeFn enc, CUtensorMap *m, const void *base, bool f32, int64_t H, int64_t tokens,
                   uint32_t width = 128) {
    const cuuint64_t es = f32 ? 4 : 2;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[2] = {kDim * es, static_cast<cuuint64_t>(H) * kDim * es};
    const cuuint32_t box[3] = {width, 1, 16};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               width == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t configure_backward_chunk() {
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_chains_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kChainSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kda_bwd_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
}

cudaError_t launch_bwd_chains(const BwdChunkParams &p, cudaStream_t stream) {
    const int64_t units = static_cast<int64_t>(p.geo.n_seqs) * p.geo.n_heads * (kDim / kCBV);
    if (units <= 0) return cudaSuccess;
    const EncodeFn enc = reinterpret_cast<EncodeFn>(tensor_map_encoder());
    if (enc == nullptr) return cudaErrorNotSupported;
    ChainMaps tm;
    const int64_t items = p.max_chunks * p.geo.n_heads;
    const int64_t tokens =
        p.geo.cu != nullptr ? p.geo.seq_len : static_cast<int64_t>(p.geo.n_seqs) * p.geo.seq_len;
    if (!encode_states(enc, &tm.ckpt, p.ckpt, items, 16) || !encode_states(enc, &tm.dsn, p.dsn, items, 16) ||
        !encode_rows16(enc, &tm.dout, p.dout, false, p.geo.n_heads, tokens, 64))
        return cudaErrorInvalidValue;
    kda_bwd_chains_kernel<<<static_cast<unsigned>(2 * units), (kCWarps + 1) * 32, kChainSmem, stream>>>(
        p, tm, static_cast<int>(units));
    return cudaGetLastError();
}

cudaError_t launch_bwd_grad(const BwdChunkParams &p, cudaStream_t stream) {
    const int64_t items = p.max_chunks * p.geo.n_heads;
    if (items <= 0) return cudaSuccess;
    const EncodeFn enc = reinterpret_cast<EncodeFn>(tensor_map_encoder());
    if (enc == nullptr) return cudaErrorNotSupported;
    const int64_t tokens =
        p.geo.cu != nullptr ? p.geo.seq_len : static_cast<int64_t>(p.geo.n_seqs) * p.geo.seq_len;
    GradMaps tm;
    if (!encode_states(enc, &tm.st, p.ckpt, items, 128) || !encode_states(enc, &tm.dst, p.dsn, items, 128) ||
        !encode_rows16(enc, &tm.g, p.ip.g, true, p.geo.n_heads, tokens) ||
        !encode_rows16(enc, &tm.k, p.ip.k, false, p.geo.n_heads, tokens) ||
        !encode_rows16(enc, &tm.q, p.ip.q, false, p.geo.n_heads, tokens))
        return cudaErrorInvalidValue;
    int dev = 0, sms = 0, nb = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kda_bwd_grad_kernel, kGThreads, kGSmem);
    int64_t grid = static_cast<int64_t>(sms > 0 ? sms : 152) * (nb > 0 ? nb : 1);
    if (grid > items) grid = items;
    kda_bwd_grad_kernel<<<static_cast<unsigned>(grid), kGThreads, kGSmem, stream>>>(p, tm);
    return cudaGetLastError();
}

}  // namespace kda
