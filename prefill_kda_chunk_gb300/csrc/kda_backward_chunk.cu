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
// Three launches after the forward's intra-chunk kernels (which build the
// records): the forward chain again without outputs, keeping every chunk's
// entry state S^T in bf16; kda_bwd_chain_kernel, the reverse chain over
// the chunks (the forward step with roles swapped), keeping every chunk's
// dS_next^T in bf16 and writing dL/d(initial state); and kda_bwd_grad_kernel,
// chunk-parallel, one CTA per (chunk, head), for everything else. The WY
// reverse takes exact per-pair exponentials exp(G_r - G_i) (r >= i), so it
// holds for any decay; the record it starts from is rebuilt by the
// forward's own per-chunk code, factored or exact form as the forward chose.

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_intra_body.cuh"
#include "kda_recurrent_body.cuh"

namespace kda {

namespace {

constexpr int kChainStageBytes = kRecUt;   // W, Qg, Kd, P, gamma (the reverse needs no Ut)
constexpr int kCBV = 64;                   // value channels per reverse-chain CTA
constexpr int kCWarps = kCBV / 16;
constexpr int kChainSmem = kStages * kChainStageBytes + 2 * kStages * 8;

// ---------------------------------------------------------------------------
// Reverse chain: one CTA per (sequence, head, 64-value slice), 4 consumer
// warps holding dS^T fragments (16 values x 128 keys each, fp32) and one
// producer warp streaming the records (last chunk first) into a ring of
// shared-memory stages.
__global__ void __launch_bounds__((kCWarps + 1) * 32) kda_bwd_chain_kernel(BwdChunkParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3, quad = lane >> 3;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    constexpr int kSlices = kDim / kCBV;
    const int s = blockIdx.x % kSlices;
    const int h = (blockIdx.x / kSlices) % H;
    const int n = blockIdx.x / (kSlices * H);
    const uint32_t stage0 = smem_u32(smem);
    const uint32_t bar_full = stage0 + kStages * kChainStageBytes;
    const uint32_t bar_empty = bar_full + kStages * 8;
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
                         rec0 + static_cast<int64_t>(nck - 1 - i) * H * kRecBytes, kChainStageBytes,
                         bar_full + 8 * st);
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
    const __nv_bfloat16 *dout = static_cast<const __nv_bfloat16 *>(p.dout);
    const int64_t rowe = static_cast<int64_t>(H) * kDim;

    for (int i = 0; i < nck; ++i) {
        const int c = nck - 1 - i;                   // chunk of the sequence
        const int st = i % kStages;
        const int64_t t0 = tb + 16 * static_cast<int64_t>(c);
        const int L = static_cast<int>(te - t0 < 16 ? te - t0 : 16);
        // dO^T as the A operand: rows v0 + gid (+ 8), tokens 2 tig (+ 1), + 8
        uint32_t aO[4];
        {
            auto ld = [&](int t, int v) -> float {
                return t < L ? __bfloat162float(dout[(t0 + t) * rowe + h * kDim + v]) : 0.f;
            };
            const int va = v0 + gid, vb = va + 8, ta = 2 * tig, tc = ta + 8;
            aO[0] = pack_bf16(ld(ta, va), ld(ta + 1, va));
            aO[1] = pack_bf16(ld(ta, vb), ld(ta + 1, vb));
            aO[2] = pack_bf16(ld(tc, va), ld(tc + 1, va));
            aO[3] = pack_bf16(ld(tc, vb), ld(tc + 1, vb));
        }
        // dS_next^T of this chunk (bf16, [v][k]) for the gradient kernel
        {
            __nv_bfloat16 *dp = static_cast<__nv_bfloat16 *>(p.dsn) +
                                ((chunk0 + c) * H + h) * static_cast<int64_t>(kDim * kDim) +
                                static_cast<int64_t>(v0 + gid) * kDim + 2 * tig;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                *reinterpret_cast<uint32_t *>(dp + 8 * j) = pack_bf16(acc[j][0], acc[j][1]);
                *reinterpret_cast<uint32_t *>(dp + 8 * kDim + 8 * j) = pack_bf16(acc[j][2], acc[j][3]);
            }
        }
        if (!mbar_wait(bar_full + 8 * st, (i / kStages) & 1)) {
            atomicOr(p.err, kErrTimeout);
            break;
        }
        const uint8_t *stg = smem + st * kChainStageBytes;
        const uint32_t sw = stage0 + st * kChainStageBytes;

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
}

// ---------------------------------------------------------------------------
// Chunk-parallel gradients: one 128-thread CTA per (chunk, head) at a time
// (persistent, two CTAs per SM). Shared memory:
constexpr int kGOffST = 0;                  // S^T bf16 [128 v][128 k], swizzled; later
                                            //   dW, dQg, dKd, dU fp32 [16][128] each
constexpr int kGOffDT = 32768;              // dS_next^T bf16, swizzled; later small fp32
                                            //   tiles: dP, dgamma, dM, dA, Y, dbeta parts
constexpr int kGOffRec = 65536;             // the chunk's record, rebuilt
constexpr int kGOffWS = kGOffRec + kRecBytes;            // warp 0's per-chunk scratch
constexpr int kGOffDO = kGOffWS + static_cast<int>(sizeof(IntraWarpSmem));   // dO bf16
                                            //   [16 t][128 v], swizzled; later dW bf16
constexpr int kGOffUB = kGOffDO + 4096;     // U bf16 [16 t][128 v], swizzled
constexpr int kGOffDUB = kGOffUB + 4096;    // dU bf16 [16 t][128 v], swizzled
constexpr int kGSmem = kGOffDUB + 4096;
static_assert(kGOffWS % 16 == 0 && kGOffDO % 16 == 0, "alignment");
// small tiles in the dS_next^T region once it is read
constexpr int kSdP = kGOffDT, kSdG = kSdP + 1024, kSdM = kSdG + 512, kSdA = kSdM + 1024,
              kSY = kSdA + 1024, kSdB = kSY + 1024;
constexpr int kGThreads = 128;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2eG = 1.4426950408889634f;

__device__ __forceinline__ float ex2g(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kGThreads, 2) kda_bwd_grad_kernel(BwdChunkParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3, quad = lane >> 3;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    if (geo.cu != nullptr && (*geo.call_flags & kErrBadCu)) return;
    const uint32_t sb = smem_u32(smem);
    const uint32_t sST = sb + kGOffST, sDT = sb + kGOffDT, sRec = sb + kGOffRec, sDO = sb + kGOffDO,
                   sUB = sb + kGOffUB, sDUB = sb + kGOffDUB;
    IntraWarpSmem &ws = *reinterpret_cast<IntraWarpSmem *>(smem + kGOffWS);
    const int64_t rowe = static_cast<int64_t>(H) * kDim;
    const float scale = p.ip.scale;
    const int64_t items = p.max_chunks * H;

    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t c = item / H;
        const int h = static_cast<int>(item - c * H);
        int n, L;
        int64_t t0, rec_idx;
        if (!locate_chunk(geo, c, n, t0, L, rec_idx)) continue;
        (void)n;
        __syncthreads();   // the previous item is done with every tile

        // ---- phase 1: warp 0 rebuilds the record (and T, K e^G, V in its
        //      scratch); warps 1-3 stage S^T, dS_next^T and dO
        if (warp == 0) {
            uint8_t *rec = smem + kGOffRec;
            if (intra_item<false, true>(p.ip, ws, t0, L, h, rec))
                intra_exact_item<false, true>(p.ip, ws, t0, L, h, rec);
        } else {
            const int64_t off = (rec_idx * H + h) * static_cast<int64_t>(kDim * kDim);
            const __nv_bfloat16 *cs = static_cast<const __nv_bfloat16 *>(p.ckpt) + off;
            const __nv_bfloat16 *ds = static_cast<const __nv_bfloat16 *>(p.dsn) + off;
            for (int i = tid - 32; i < 2048; i += 96) {
                const int r = i >> 4, cc = i & 15;
                const uint32_t dst = r * 256 + ((cc ^ (r & 7)) << 4);
                cp_async16(sST + dst, cs + r * kDim + cc * 8, 16u);
                cp_async16(sDT + dst, ds + r * kDim + cc * 8, 16u);
            }
            const __nv_bfloat16 *dop = static_cast<const __nv_bfloat16 *>(p.dout) + (t0 * H + h) * kDim;
            for (int i = tid - 32; i < 256; i += 96) {
                const int r = i >> 4, cc = i & 15;
                const bool ok = r < L;
                cp_async16(sDO + r * 256 + ((cc ^ (r & 7)) << 4), dop + (ok ? r : 0) * rowe + cc * 8,
                           ok ? 16u : 0u);
            }
            cp_async_commit();
            cp_async_wait_all();
        }
        __syncthreads();

        // ---- phase 2: U^T = Ut^T + S^T (-W)^T and dU^T = dS_next^T Kd^T + dO^T P,
        //      value rows 32 warp + 16 mt, all 16 tokens
        float dUf[2][2][4];   // dU^T fragments kept in fp32
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const int vb = 32 * warp + 16 * mt;
            float uT[2][2][4], dT[2][2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tk = 8 * nt + 2 * tig;
                const float2 u01 = unpack_bf16(*reinterpret_cast<const uint32_t *>(
                    smem + kGOffRec + kRecUt + ((vb + gid) * 16 + tk) * 2));
                const float2 u23 = unpack_bf16(*reinterpret_cast<const uint32_t *>(
                    smem + kGOffRec + kRecUt + ((vb + gid + 8) * 16 + tk) * 2));
                uT[nt][0][0] = u01.x; uT[nt][0][1] = u01.y; uT[nt][0][2] = u23.x; uT[nt][0][3] = u23.y;
#pragma unroll
                for (int e = 0; e < 4; ++e) { uT[nt][1][e] = 0.f; dT[nt][0][e] = 0.f; dT[nt][1][e] = 0.f; }
            }
            {
                // dO^T (v x t) from the [t][v] tile, transposed; P as B (r x t), transposed
                uint32_t aO[4], bp[4];
                const int m = lane >> 3;
                ldsm_x4_t(sDO + swz((lane & 7) + 8 * (m >> 1), vb + 8 * (m & 1)), aO[0], aO[1], aO[2], aO[3]);
                ldsm_x4_t(sRec + kRecP + (((m & 1) * 8 + (lane & 7)) * 16 + (m >> 1) * 8) * 2, bp[0], bp[1],
                          bp[2], bp[3]);
                mma_r(dT[0][1], aO, bp[0], bp[1]);
                mma_r(dT[1][1], aO, bp[2], bp[3]);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t aS[4], aD[4], bw[4], bk[4];
                const int ra = vb + (lane & 7) + 8 * ((lane >> 3) & 1), ca = 16 * kk + 8 * (lane >> 4);
                ldsm_x4(sST + swz(ra, ca), aS[0], aS[1], aS[2], aS[3]);
                ldsm_x4(sDT + swz(ra, ca), aD[0], aD[1], aD[2], aD[3]);
                const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
                ldsm_x4(sRec + kRecW + swz(rb, cb), bw[0], bw[1], bw[2], bw[3]);
                ldsm_x4(sRec + kRecKd + swz(rb, cb), bk[0], bk[1], bk[2], bk[3]);
                mma_r(uT[0][kk & 1], aS, bw[0], bw[1]);
                mma_r(uT[1][kk & 1], aS, bw[2], bw[3]);
                mma_r(dT[0][kk & 1], aD, bk[0], bk[1]);
                mma_r(dT[1][kk & 1], aD, bk[2], bk[3]);
            }
            float u[2][4], du[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    u[nt][e] = uT[nt][0][e] + uT[nt][1][e];
                    du[nt][e] = dT[nt][0][e] + dT[nt][1][e];
                    dUf[mt][nt][e] = du[nt][e];
                }
            // U and dU to their [t][v] tiles (bf16), transposed by stmatrix
            const int m = lane >> 3;
            const uint32_t so = swz(8 * (m >> 1) + (lane & 7), vb + 8 * (m & 1));
            stsm_x4_t(sUB + so, pack_bf16(u[0][0], u[0][1]), pack_bf16(u[0][2], u[0][3]),
                      pack_bf16(u[1][0], u[1][1]), pack_bf16(u[1][2], u[1][3]));
            stsm_x4_t(sDUB + so, pack_bf16(du[0][0], du[0][1]), pack_bf16(du[0][2], du[0][3]),
                      pack_bf16(du[1][0], du[1][1]), pack_bf16(du[1][2], du[1][3]));
        }
        __syncthreads();

        // ---- phase 3: contractions over the 128 values. Warp w: keys 32 w .. + 31.
        //      dW = -dU S^T, dQg = dO S^T, dKd = U dS_next^T; warp 0 also dP = dO U^T;
        //      thread = key for dgamma = rowsum(dS_next o S)
        float cW[4][4], cQ[4][4], cK[4][4], cP[2][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) cW[j][e] = cQ[j][e] = cK[j][e] = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) cP[j][e] = 0.f;
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
                ldsm_x4_t(sST + swz(rk, ck), bs[0], bs[1], bs[2], bs[3]);
                ldsm_x4_t(sDT + swz(rk, ck), bd[0], bd[1], bd[2], bd[3]);
                mma_r(cW[2 * jp], aDU, bs[0], bs[1]);
                mma_r(cW[2 * jp + 1], aDU, bs[2], bs[3]);
                mma_r(cQ[2 * jp], aO_, bs[0], bs[1]);
                mma_r(cQ[2 * jp + 1], aO_, bs[2], bs[3]);
                mma_r(cK[2 * jp], aU_, bd[0], bd[1]);
                mma_r(cK[2 * jp + 1], aU_, bd[2], bd[3]);
            }
            if (warp == 0) {
                uint32_t bu[4];
                const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
                ldsm_x4(sUB + swz(rb, cb), bu[0], bu[1], bu[2], bu[3]);
                mma_r(cP[0], aO_, bu[0], bu[1]);
                mma_r(cP[1], aO_, bu[2], bu[3]);
            }
        }
        float dgam = 0.f;
        {
            const int k = tid;
            for (int v = 0; v < kDim; ++v) {
                const uint32_t o = v * 256 + ((((k >> 3) ^ (v & 7))) << 4) + (k & 7) * 2;
                dgam = fmaf(__bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(smem + kGOffST + o)),
                            __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(smem + kGOffDT + o)),
                            dgam);
            }
        }
        __syncthreads();
        // results: dW, dQg, dKd, dU fp32 [16][128] over S^T; dW bf16 over dO;
        // dP, dgamma over dS_next^T
        float *gW = reinterpret_cast<float *>(smem + kGOffST);
        float *gQ = gW + 16 * kDim, *gK = gQ + 16 * kDim, *gU = gK + 16 * kDim;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int key = 32 * warp + 8 * j + 2 * tig;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int t = gid + 8 * hf;
                *reinterpret_cast<float2 *>(gW + t * kDim + key) = make_float2(-cW[j][2 * hf], -cW[j][2 * hf + 1]);
                *reinterpret_cast<float2 *>(gQ + t * kDim + key) = make_float2(cQ[j][2 * hf], cQ[j][2 * hf + 1]);
                *reinterpret_cast<float2 *>(gK + t * kDim + key) = make_float2(cK[j][2 * hf], cK[j][2 * hf + 1]);
                *reinterpret_cast<uint32_t *>(smem + kGOffDO + swz(t, key)) =
                    pack_bf16(-cW[j][2 * hf], -cW[j][2 * hf + 1]);
            }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int v = 32 * warp + 16 * mt + gid, t = 8 * nt + 2 * tig;
                gU[t * kDim + v] = dUf[mt][nt][0];
                gU[(t + 1) * kDim + v] = dUf[mt][nt][1];
                gU[t * kDim + v + 8] = dUf[mt][nt][2];
                gU[(t + 1) * kDim + v + 8] = dUf[mt][nt][3];
            }
        float *gP = reinterpret_cast<float *>(smem + kSdP);
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
        reinterpret_cast<float *>(smem + kSdG)[tid] = dgam;
        __syncthreads();

        // ---- phase 4a (warp 0): dM = dU V^T + dW Kg^T (16 x 16), then dT = dM diag(beta),
        //      dbeta from M = T diag(beta), dA = -(T^T dT T^T) on the strict lower triangle
        float *sM = reinterpret_cast<float *>(smem + kSdM);
        float *sA = reinterpret_cast<float *>(smem + kSdA);
        float *sY = reinterpret_cast<float *>(smem + kSY);
        float *sB = reinterpret_cast<float *>(smem + kSdB);   // [0,16): dbeta from dM; [16,80): parts
        if (warp == 0) {
            float m2[2][4] = {};
            const uint32_t sV = smem_u32(ws.v), sKg = smem_u32(ws.kg);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t aD[4], aW[4], bv[4], bg[4];
                const int ra = (lane & 7) + 8 * ((lane >> 3) & 1), ca = 16 * kk + 8 * (lane >> 4);
                ldsm_x4(sDUB + swz(ra, ca), aD[0], aD[1], aD[2], aD[3]);
                ldsm_x4(sDO + swz(ra, ca), aW[0], aW[1], aW[2], aW[3]);   // dW
                const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
                ldsm_x4(sV + swz(rb, cb), bv[0], bv[1], bv[2], bv[3]);
                ldsm_x4(sKg + swz(rb, cb), bg[0], bg[1], bg[2], bg[3]);
                mma_r(m2[0], aD, bv[0], bv[1]);
                mma_r(m2[1], aD, bv[2], bv[3]);
                mma_r(m2[0], aW, bg[0], bg[1]);
                mma_r(m2[1], aW, bg[2], bg[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int r = gid + 8 * hf, i = 8 * nt + 2 * tig;
                    sM[r * 16 + i] = m2[nt][2 * hf];
                    sM[r * 16 + i + 1] = m2[nt][2 * hf + 1];
                }
            __syncwarp();
            const float *T = ws.t;   // T[r * 17 + i]
            const float *bet = p.ip.beta;
            // lane j < 16: dbeta_j (from M) = sum_r dM[r][j] T[r][j]; dT[r][j] = dM[r][j] beta_j
            if (lane < 16) {
                const float bj = lane < L ? __ldg(bet + (t0 + lane) * H + h) : 0.f;
                float sbj = 0.f;
                for (int r = 0; r < 16; ++r) {
                    sbj = fmaf(sM[r * 16 + lane], T[r * 17 + lane], sbj);
                    sM[r * 16 + lane] *= bj;                  // now dT
                }
                sB[lane] = sbj;
            }
            __syncwarp();
            // Y = T^T dT: Y[r][b] = sum_a T[a][r] dT[a][b]; lane: 8 entries
            for (int e = lane; e < 256; e += 32) {
                const int r = e >> 4, b = e & 15;
                float y = 0.f;
                for (int a = 0; a < 16; ++a) y = fmaf(T[a * 17 + r], sM[a * 16 + b], y);
                sY[e] = y;
            }
            __syncwarp();
            // dA[r][i] = -sum_b Y[r][b] T[i][b], strict lower
            for (int e = lane; e < 256; e += 32) {
                const int r = e >> 4, i = e & 15;
                float a = 0.f;
                for (int b = 0; b < 16; ++b) a = fmaf(sY[r * 16 + b], T[i * 17 + b], a);
                sA[e] = i < r ? -a : 0.f;
            }
        }
        __syncthreads();

        // ---- phase 4b: thread = channel ch, all 16 rows
        {
            const int ch = tid;
            const int64_t base = (t0 * H + h) * kDim + ch;
            const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.ip.q);
            const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(p.ip.k);
            float kk_[16], qq[16], G2[16], bet[16];
            float run = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const bool ok = r < L;
                kk_[r] = ok ? __bfloat162float(kg[base + r * rowe]) : 0.f;
                qq[r] = ok ? __bfloat162float(qg[base + r * rowe]) : 0.f;
                run += ok ? __ldg(p.ip.g + base + r * rowe) * kLog2eG : 0.f;
                G2[r] = run;
                bet[r] = ok ? __ldg(p.ip.beta + (t0 + r) * H + h) : 0.f;
            }
            const float *T = ws.t;
            float dk[16], dq[16], dG[16], pb[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) { dk[r] = 0.f; dq[r] = 0.f; dG[r] = 0.f; pb[r] = 0.f; }
            // the gated Gram products, exact per-pair exponentials
#pragma unroll
            for (int r = 0; r < 16; ++r) {
#pragma unroll
                for (int i = 0; i <= r; ++i) {
                    const float E = ex2g(G2[r] - G2[i]);
                    const float dY = scale * gP[r * 16 + i];
                    const float wP = dY * E;
                    dq[r] = fmaf(wP, kk_[i], dq[r]);
                    dk[i] = fmaf(wP, qq[r], dk[i]);
                    const float tP = wP * qq[r] * kk_[i];
                    dG[r] += tP;
                    dG[i] -= tP;
                    if (i < r) {
                        const float dAr = sA[r * 16 + i];
                        const float kkE = kk_[r] * kk_[i] * E;
                        pb[r] = fmaf(dAr, kkE, pb[r]);
                        const float wA = bet[r] * dAr * E;
                        dk[r] = fmaf(wA, kk_[i], dk[r]);
                        dk[i] = fmaf(wA, kk_[r], dk[i]);
                        const float tA = bet[r] * dAr * kkE;
                        dG[r] += tA;
                        dG[i] -= tA;
                    }
                }
            }
            // Qg = scale q e^G, Kd = k e^(G_last - G), gamma = e^(G_last), Kg = k e^G
            const float G2L = G2[15];
            float dGL = reinterpret_cast<const float *>(smem + kSdG)[ch] * ex2g(G2L);
            float dv[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float eG = ex2g(G2[r]);
                const float dQg = gQ[r * kDim + ch];
                dq[r] = fmaf(scale * dQg, eG, dq[r]);
                dG[r] = fmaf(dQg, scale * qq[r] * eG, dG[r]);
                const float eD = ex2g(G2L - G2[r]);
                const float dKd = gK[r * kDim + ch];
                dk[r] = fmaf(dKd, eD, dk[r]);
                const float kdv = dKd * kk_[r] * eD;
                dG[r] -= kdv;
                dGL += kdv;
                // dKg = M^T dW and dv = M^T dUt, M[u][r] = T[u][r] beta_r
                float sW = 0.f, sU = 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float tr = T[u * 17 + r];
                    sW = fmaf(tr, gW[u * kDim + ch], sW);
                    sU = fmaf(tr, gU[u * kDim + ch], sU);
                }
                const float dKg = bet[r] * sW;
                dv[r] = bet[r] * sU;
                dk[r] = fmaf(dKg, eG, dk[r]);
                dG[r] = fmaf(dKg, kk_[r] * eG, dG[r]);
            }
            dG[15] += dGL;
            // dbeta partials of this channel (A part), summed over the channels below
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float x = pb[r];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                if (lane == 0) sB[16 + warp * 16 + r] = x;
            }
            // dg = reverse cumulative sum of dG; outputs for rows < L
            float acc = 0.f;
#pragma unroll
            for (int r = 15; r >= 0; --r) {
                acc += dG[r];
                if (r < L) {
                    const int64_t o = base + r * rowe;
                    p.dq[o] = dq[r];
                    p.dk[o] = dk[r];
                    p.dv[o] = dv[r];
                    p.dg[o] = acc;
                }
            }
        }
        __syncthreads();
        if (tid < 16 && tid < L) {
            const float bA = sB[16 + tid] + sB[32 + tid] + sB[48 + tid] + sB[64 + tid];
            p.dbeta[(t0 + tid) * H + h] = sB[tid] + bA;
        }
    }
    (void)kLn2;
}

}  // namespace

cudaError_t configure_backward_chunk() {
    cudaError_t e = cudaFuncSetAttribute(kda_bwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kChainSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kda_bwd_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
}

cudaError_t launch_bwd_chain(const BwdChunkParams &p, cudaStream_t stream) {
    const int64_t ctas = static_cast<int64_t>(p.geo.n_seqs) * p.geo.n_heads * (kDim / kCBV);
    if (ctas <= 0) return cudaSuccess;
    kda_bwd_chain_kernel<<<static_cast<unsigned>(ctas), (kCWarps + 1) * 32, kChainSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_grad(const BwdChunkParams &p, cudaStream_t stream) {
    const int64_t items = p.max_chunks * p.geo.n_heads;
    if (items <= 0) return cudaSuccess;
    int dev = 0, sms = 0, nb = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kda_bwd_grad_kernel, kGThreads, kGSmem);
    int64_t grid = static_cast<int64_t>(sms > 0 ? sms : 152) * (nb > 0 ? nb : 1);
    if (grid > items) grid = items;
    kda_bwd_grad_kernel<<<static_cast<unsigned>(grid), kGThreads, kGSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
