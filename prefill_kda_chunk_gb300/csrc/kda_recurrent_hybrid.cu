// Recurrent half of chunked KDA prefill, hybrid form: the chunk-to-chunk
// chain on warp-level MMAs, the output product on the 5th-generation tensor
// core (tcgen05, tensor memory).
//
// Per chunk, with S (K x V, fp32) the state entering it ("Kimi K3 的三個系統設計",
// section "為什麼 FlashKDA 選擇 16-token chunks": the recurrent-propagation kernel):
//
//   U   = Ut - W S                                   (16 x BV)
//   o   = Qg S + P U          (the record's Qg and P carry the output scale)
//   S  <- Diag(exp(G_last)) S + (K * exp(G_last - G))^T U
//
// Only U and the state update lie on the dependency chain S -> U -> S. One
// CTA per (sequence, head, 64 value channels):
//
//  * four chain warps (16 value channels each) hold S^T in registers as
//    mma.sync fragments and do U^T = Ut^T - S^T W^T, the decay and
//    S^T += U^T Kd. Each step they also write the bf16 S^T they used into
//    tensor memory with tcgen05.st.16x256b, whose register layout is the
//    mma.sync accumulator fragment: value row r of the CTA lands in TMEM lane
//    32 (r / 16) + r % 16, the layout of the M = 64 operand;
//  * one thread issues the output product o^T = S^T Qg^T as eight
//    tcgen05.mma (M = 64 values, N = 16 tokens, K = 16 keys each; A from
//    TMEM, B = Qg from the shared-memory stage, fp32 accumulate in TMEM);
//  * the chain warps read o^T back in fragment layout, add U^T P^T with two
//    warp MMAs and store o.
//
// The tensor core reads Qg once per CTA, where warp MMAs would read it once
// per warp, and the state hand-off goes to tensor memory, so shared-memory
// traffic and warp MMA issue both drop by about a third. Tensor memory: two A
// buffers (64 columns each, bf16 pairs) and two D buffers (16 fp32 columns),
// alternating by chunk parity.
//
// Within each 16-key block the TMEM columns hold key pairs in the order the
// fragments put them: column m holds the pair (m >> 1) + 4 (m & 1). The
// intra-chunk kernel writes the record's Qg in the matching K-major layout
// (core matrices of 8 tokens x 8 keys, 128 B each; 128 B between key groups,
// 2048 B between token groups).
//
// Every wait is bounded; a timeout is recorded in the device error word and
// the CTA winds down (tensor memory is always released).

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_tcgen05.cuh"

namespace kda {

namespace {

constexpr int kHStages = 4;
constexpr int kHBV = 64;                             // value channels per CTA
constexpr int kHSlices = kDim / kHBV;
constexpr int kHWarps = kHBV / 16;                   // chain warps
constexpr int kHProd = kHWarps, kHMma = kHWarps + 1; // warp indices
constexpr int kHThreads = (kHWarps + 2) * 32;
constexpr int kHStageBytes = kRecUt + kHBV * 32;     // W, Qg, Kd, P, gamma + Ut^T slice
constexpr int kHOStage = kHStages * kHStageBytes;    // o staging, 512 B per chain warp
constexpr int kHMisc = kHOStage + kHWarps * 512;     // TMEM base address
constexpr int kHBars = kHMisc + 16;
constexpr int kBFull = 0, kBEmpty = kHStages, kBAReady = 2 * kHStages, kBODone = kBAReady + 2,
              kHNumBars = kBODone + 2;
constexpr int kHSmem = kHBars + kHNumBars * 8;

constexpr uint32_t kTA = 0;     // S^T as bf16 pairs, 2 x 64 columns
constexpr uint32_t kTD = 128;   // o^T partial, fp32, 2 x 16 columns
constexpr uint32_t kHTCols = 256;

__global__ void __launch_bounds__(kHThreads)
kda_recurrent_hybrid_kernel(RecurParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3, quad = lane >> 3;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    const int s = blockIdx.x % kHSlices;
    const int h = (blockIdx.x / kHSlices) % H;
    const int n = blockIdx.x / (kHSlices * H);

    const uint32_t bar0 = smem_u32(smem + kHBars);
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kHMisc);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kHStages; ++i) {
            mbar_init(bar(kBFull + i), 1);
            mbar_init(bar(kBEmpty + i), kHWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBAReady + i), kHWarps);
            mbar_init(bar(kBODone + i), 1);
        }
        mbar_fence_init();
    }
    if (warp == kHMma) {
        tc::alloc(smem_u32(tslot), kHTCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;

    // A bad cu_seqlens leaves nothing to do, but every warp still reaches the
    // final barrier so that tensor memory is released.
    int64_t tb = 0, te = 0, chunk0 = 0;
    int nck = 0;
    const bool bad_cu = geo.cu != nullptr && (*geo.call_flags & kErrBadCu);
    if (geo.cu == nullptr) {
        tb = static_cast<int64_t>(n) * geo.seq_len + 16 * static_cast<int64_t>(geo.pos_begin);
        te = static_cast<int64_t>(n) * geo.seq_len + geo.seq_len;
        chunk0 = static_cast<int64_t>(n) * geo.slot_stride;
        const int64_t left = te > tb ? (te - tb + 15) / 16 : 0;
        nck = static_cast<int>(left < geo.seg_len ? left : geo.seg_len);
    } else if (!bad_cu) {
        tb = geo.cu[n];
        te = geo.cu[n + 1];
        chunk0 = geo.chunk_off[n];
        nck = static_cast<int>((te - tb + 15) / 16);
    }
    const uint8_t *rec0 = p.rec + (chunk0 * H + h) * static_cast<int64_t>(kRecBytes);
    const uint32_t stage0 = smem_u32(smem);

    if (warp == kHProd) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < nck; ++i) {
                const int st = i % kHStages;
                if (i >= kHStages &&
                    !mbar_wait(bar(kBEmpty + st), ((i / kHStages) - 1) & 1)) {
                    atomicOr(p.err, kErrTimeout);
                    break;
                }
                const uint8_t *src = rec0 + static_cast<int64_t>(i) * H * kRecBytes;
                const uint32_t dst = stage0 + st * kHStageBytes;
                mbar_arrive_expect_tx(bar(kBFull + st), kHStageBytes);
                bulk_g2s(dst, src, kRecUt, bar(kBFull + st));
                bulk_g2s(dst + kRecUt, src + kRecUt + s * kHBV * 32, kHBV * 32, bar(kBFull + st));
            }
        }
    } else if (warp == kHMma) {
        // ------------------------------------------------------ o^T = S^T Qg^T
        if (lane == 0) {
            for (int i = 0; i < nck; ++i) {
                const int st = i % kHStages, b = i & 1;
                if (!mbar_wait(bar(kBFull + st), (i / kHStages) & 1) ||
                    !mbar_wait(bar(kBAReady + b), (i >> 1) & 1)) {
                    atomicOr(p.err, kErrTimeout);
                    break;
                }
                tc::fence_after();
                const uint32_t qg = stage0 + st * kHStageBytes + kRecQg;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16_ts(tmem + kTD + 16 * b, tmem + kTA + 64 * b + 8 * kk,
                                    tc::sdesc(qg + 256 * kk, 128, 2048), tc::idesc(64, 16, 1),
                                    kk > 0);
                tc::commit(bar(kBODone + b));
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ chain warps
        const int vw = 16 * warp;          // first value channel of this warp within the slice
        const int v0 = s * kHBV + vw;      // ... within the head
        const uint32_t tlane = static_cast<uint32_t>(32 * warp) << 16;
        float acc[16][4];                  // S^T fragments: rows = value, cols = key
        const int64_t sbase = (static_cast<int64_t>(n) * H + h) * kDim * kDim;
        if (p.s0 != nullptr) {
            const float *S0 = p.s0 + sbase;
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

        uint8_t *so = smem + kHOStage + warp * 512;   // [16 tok][16 val] bf16
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.out) + (tb * H + h) * kDim + v0;
        const int64_t ostep = 16 * static_cast<int64_t>(H) * kDim;
        bool ready = false, failed = false;
        uint32_t aU_prev[4] = {0u, 0u, 0u, 0u};
        // o of chunk j: o^T = (Qg S)^T from tensor memory + U^T P^T, then the
        // store and the release of chunk j's stage
        auto o_branch = [&](int j, const uint32_t (&aUj)[4]) -> bool {
            const int stj = j % kHStages, bj = j & 1;
            if (!mbar_wait(bar(kBODone + bj), (j >> 1) & 1)) {
                atomicOr(p.err, kErrTimeout);
                failed = true;
                return false;
            }
            tc::fence_after();
            float o[2][4];
            {
                uint32_t d[2][4];
                tc::ld_16x256b(tmem + tlane + kTD + 16 * bj, d[0][0], d[0][1], d[0][2], d[0][3]);
                tc::ld_16x256b(tmem + tlane + kTD + 16 * bj + 8, d[1][0], d[1][1], d[1][2],
                               d[1][3]);
                tc::ld_wait();
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[nt][e] = __uint_as_float(d[nt][e]);
            }
            {
                uint32_t bp[4];
                const int rp = (quad >> 1) * 8 + (lane & 7);
                ldsm_x4(stage0 + stj * kHStageBytes + kRecP + rp * 32 + (quad & 1) * 16, bp[0],
                        bp[1], bp[2], bp[3]);
                mma_r(o[0], aUj, bp[0], bp[1]);
                mma_r(o[1], aUj, bp[2], bp[3]);
            }
            const int64_t t0 = tb + 16 * static_cast<int64_t>(j);
            const int L = static_cast<int>((te - t0) < 16 ? (te - t0) : 16);
            {
                const int q8 = lane >> 3, r = lane & 7;
                stsm_x4_t(smem_u32(so) + ((q8 >> 1) * 8 + r) * 32 + (q8 & 1) * 16,
                          pack_bf16(o[0][0], o[0][1]), pack_bf16(o[0][2], o[0][3]),
                          pack_bf16(o[1][0], o[1][1]), pack_bf16(o[1][2], o[1][3]));
            }
            __syncwarp();
            {
                const int tok = lane >> 1, hf = lane & 1;
                if (tok < L) {
                    const uint4 val = *reinterpret_cast<const uint4 *>(so + tok * 32 + hf * 16);
                    *reinterpret_cast<uint4 *>(orow + tok * static_cast<int64_t>(H) * kDim +
                                               hf * 8) = val;
                }
            }
            orow += ostep;
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBEmpty + stj));
            return true;
        };
        for (int i = 0; i < nck; ++i) {
            const int st = i % kHStages, b = i & 1;
            if (!ready && !mbar_wait(bar(kBFull + st), (i / kHStages) & 1)) {
                atomicOr(p.err, kErrTimeout);
                failed = true;
                break;
            }
            const uint8_t *stg = smem + st * kHStageBytes;
            const uint32_t sw = stage0 + st * kHStageBytes;

            // S^T as bf16 A fragments, one per 16-key step
            uint32_t aS[8][4];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                aS[kk][0] = pack_bf16(acc[2 * kk][0], acc[2 * kk][1]);
                aS[kk][1] = pack_bf16(acc[2 * kk][2], acc[2 * kk][3]);
                aS[kk][2] = pack_bf16(acc[2 * kk + 1][0], acc[2 * kk + 1][1]);
                aS[kk][3] = pack_bf16(acc[2 * kk + 1][2], acc[2 * kk + 1][3]);
            }

            // start handing the rounded S^T to the tensor core (buffer b was
            // read by the product of chunk i - 2, which this warp has waited
            // for); the stores complete in the background
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc::st_16x256b(tmem + tlane + kTA + 64 * b + 8 * kk, aS[kk][0], aS[kk][2],
                               aS[kk][1], aS[kk][3]);

            // U^T = Ut^T - S^T W^T, two partial sums
            float uT[2][2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tk = 8 * nt + 2 * tig;
                const float2 u01 = unpack_bf16(*reinterpret_cast<const uint32_t *>(
                    stg + kRecUt + ((vw + gid) * 16 + tk) * 2));
                const float2 u23 = unpack_bf16(*reinterpret_cast<const uint32_t *>(
                    stg + kRecUt + ((vw + gid + 8) * 16 + tk) * 2));
                uT[nt][0][0] = u01.x; uT[nt][0][1] = u01.y;
                uT[nt][0][2] = u23.x; uT[nt][0][3] = u23.y;
#pragma unroll
                for (int e = 0; e < 4; ++e) uT[nt][1][e] = 0.f;
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t bw[4];
                const int rb = (quad >> 1) * 8 + (lane & 7), cb = 16 * kk + (quad & 1) * 8;
                ldsm_x4(sw + kRecW + swz(rb, cb), bw[0], bw[1], bw[2], bw[3]);
                mma_r(uT[0][kk & 1], aS[kk], bw[0], bw[1]);
                mma_r(uT[1][kk & 1], aS[kk], bw[2], bw[3]);
            }

            // decay of the state while the U products drain
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
            // S^T <- S^T Diag(gamma) + U^T Kd
#pragma unroll
            for (int jp = 0; jp < 8; ++jp) {
                uint32_t bk[4];
                const int rk = (quad & 1) * 8 + (lane & 7), ck = 16 * jp + (quad >> 1) * 8;
                ldsm_x4_t(sw + kRecKd + swz(rk, ck), bk[0], bk[1], bk[2], bk[3]);
                mma_r(acc[2 * jp], aU, bk[0], bk[1]);
                mma_r(acc[2 * jp + 1], aU, bk[2], bk[3]);
            }
            // the hand-off is complete: let the tensor core start o^T of chunk i
            tc::st_wait();
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBAReady + b));
            if (i + 1 < nck)
                ready = mbar_test(bar(kBFull + (i + 1) % kHStages), ((i + 1) / kHStages) & 1);

            // output of the previous chunk: its tensor-core product has had a
            // whole step to finish
            if (i > 0 && !o_branch(i - 1, aU_prev)) break;
#pragma unroll
            for (int e = 0; e < 4; ++e) aU_prev[e] = aU[e];
        }
        if (nck > 0 && !failed) o_branch(nck - 1, aU_prev);

        if (p.s_final != nullptr && !bad_cu) {
            float *SF = p.s_final + sbase;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int key = 8 * j + 2 * tig;
                SF[key * kDim + v0 + gid] = acc[j][0];
                SF[(key + 1) * kDim + v0 + gid] = acc[j][1];
                SF[key * kDim + v0 + gid + 8] = acc[j][2];
                SF[(key + 1) * kDim + v0 + gid + 8] = acc[j][3];
            }
        }
    }

    // every tensor-memory access of this CTA is complete before the release
    tc::fence_before();
    __syncthreads();
    if (warp == kHMma) {
        tc::fence_after();
        tc::dealloc(tmem, kHTCols);
    }
}

}  // namespace

cudaError_t configure_recurrent_hybrid() {
    return cudaFuncSetAttribute(kda_recurrent_hybrid_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kHSmem);
}

cudaError_t launch_recurrent_hybrid(const RecurParams &p, cudaStream_t stream) {
    const int64_t ctas = static_cast<int64_t>(p.geo.n_seqs) * p.geo.n_heads * kHSlices;
    if (ctas <= 0) return cudaSuccess;
    kda_recurrent_hybrid_kernel<<<static_cast<unsigned>(ctas), kHThreads, kHSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
