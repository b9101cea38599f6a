// Recurrent half of chunked KDA prefill: the inter-chunk kernel.
//
// For one (sequence, head, slice of BV value channels) a CTA walks the
// sequence's chunks in order ("Kimi K3 的三個系統設計", section
// "為什麼 FlashKDA 選擇 16-token chunks": the recurrent-propagation kernel),
// with S (K x V, fp32) the state entering the chunk:
//
//   U   = Ut - W S                                   (16 x BV)
//   o_r = scale ( (q_r * exp(G_r))^T S + sum_{i<=r} P[r,i] U_i )
//   S  <- Diag(exp(G_last)) S + (K * exp(G_last - G))^T U
//
// (scale already multiplies the record's Q*exp(G) and P tiles.)
//
// The state lives in registers as S^T fragments of the warp MMA (each
// consumer warp owns 16 value channels x all 128 key channels), which is at
// the same time the A operand of S^T W^T (the transposed U product) and the
// accumulator of the state update. A producer warp streams each chunk's
// record into a ring of shared-memory stages with bulk async copies,
// completion tracked by mbarriers; every wait is bounded and a timeout is
// recorded in the device error word instead of hanging.
//
// Step order follows the chunk-to-chunk dependency chain (S -> U -> S): the
// U product first, the decay of S while it drains, S^T Qg^T to keep the
// tensor pipe busy, then the state update, and only after it the output
// branch (P U, store), which nothing later depends on. The next
// stage's barrier is tested right after the update MMAs are issued so that
// its latency overlaps them.

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

// OUT = false carries only the state (no output products, no o stores).
template <int BV, bool OUT>
__global__ void __launch_bounds__((BV / 16 + 1) * 32)
kda_recurrent_kernel(RecurParams p) {
    using Lay = RecurLayout<BV>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3, quad = lane >> 3;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    const int s = blockIdx.x % Lay::kSlices;
    const int h = (blockIdx.x / Lay::kSlices) % H;
    const int n = blockIdx.x / (Lay::kSlices * H);   // unit: sequence, or (half, sequence)

    const uint32_t bar_full = smem_u32(smem + Lay::kBars);
    const uint32_t bar_empty = bar_full + kStages * 8;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, Lay::kWarps * 32);
        }
        mbar_fence_init();
    }
    __syncthreads();
    if (geo.cu != nullptr && (*geo.call_flags & kErrBadCu)) return;

    int64_t tb, te, chunk0;
    int nck;
    int seq = n;                       // the sequence whose states this CTA reads and writes
    const float *s_in = p.s0;
    float *s_out = p.s_final;
    if (geo.cu == nullptr && p.split_chunks > 0) {
        // split replay: half 0 = chunks [0, c) from s0, half 1 = [c, end) from s_mid
        const int half = n / geo.n_seqs;
        seq = n % geo.n_seqs;
        const int64_t c = p.split_chunks;
        const int64_t base = static_cast<int64_t>(seq) * geo.seq_len;
        tb = base + (half ? 16 * c : 0);
        te = half ? base + geo.seq_len : base + 16 * c;
        chunk0 = static_cast<int64_t>(seq) * geo.slot_stride + (half ? c : 0);
        nck = static_cast<int>(half ? (geo.seq_len + 15) / 16 - c : c);
        s_in = half ? p.s_mid : p.s0;
        s_out = half ? p.s_final : nullptr;
    } else if (geo.cu == nullptr) {
        tb = static_cast<int64_t>(n) * geo.seq_len + 16 * static_cast<int64_t>(geo.pos_begin);
        te = static_cast<int64_t>(n) * geo.seq_len + geo.seq_len;
        chunk0 = static_cast<int64_t>(n) * geo.slot_stride;
        const int64_t left = te > tb ? (te - tb + 15) / 16 : 0;
        nck = static_cast<int>(left < geo.seg_len ? left : geo.seg_len);
    } else {
        tb = geo.cu[n];
        te = geo.cu[n + 1];
        chunk0 = geo.chunk_off[n];
        nck = static_cast<int>((te - tb + 15) / 16);
    }
    const uint8_t *rec0 = p.rec + (chunk0 * H + h) * static_cast<int64_t>(kRecBytes);
    const uint32_t stage0 = smem_u32(smem);

    if (warp == Lay::kWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < nck; ++i) {
                const int st = i % kStages;
                if (i >= kStages &&
                    !mbar_wait(bar_empty + 8 * st, ((i / kStages) - 1) & 1)) {
                    atomicOr(p.err, kErrTimeout);
                    break;
                }
                const uint8_t *src = rec0 + static_cast<int64_t>(i) * H * kRecBytes;
                const uint32_t dst = stage0 + st * Lay::kStageBytes;
                mbar_arrive_expect_tx(bar_full + 8 * st, Lay::kStageBytes);
                bulk_g2s(dst, src, kRecUt, bar_full + 8 * st);
                bulk_g2s(dst + kRecUt, src + kRecUt + s * BV * 32, BV * 32, bar_full + 8 * st);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int vw = 16 * warp;          // first value channel of this warp within the slice
    const int v0 = s * BV + vw;        // ... within the head
    float acc[16][4];                  // S^T fragments: rows = value, cols = key
    const int64_t sbase = (static_cast<int64_t>(seq) * H + h) * kDim * kDim;
    if (s_in != nullptr) {
        const float *S0 = s_in + sbase;
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

    uint8_t *so = smem + Lay::kOStage + warp * 512;   // [16 tok][16 val] bf16
    __nv_bfloat16 *outp = static_cast<__nv_bfloat16 *>(p.out);

    bool ready = false;
    __nv_bfloat16 *orow = outp + (tb * H + h) * kDim + v0;   // row 0 of the chunk's o tile
    const int64_t ostep = 16 * static_cast<int64_t>(H) * kDim;
    for (int i = 0; i < nck; ++i) {
        const int st = i % kStages;
        if (!ready && !mbar_wait(bar_full + 8 * st, (i / kStages) & 1)) {
            atomicOr(p.err, kErrTimeout);
            break;
        }
        const uint8_t *stg = smem + st * Lay::kStageBytes;
        const uint32_t sw = stage0 + st * Lay::kStageBytes;

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
            const float2 u01 = unpack_bf16(
                *reinterpret_cast<const uint32_t *>(stg + kRecUt + ((vw + gid) * 16 + tk) * 2));
            const float2 u23 = unpack_bf16(*reinterpret_cast<const uint32_t *>(
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
        if (i + 1 < nck)
            ready = mbar_test(bar_full + 8 * ((i + 1) % kStages), ((i + 1) / kStages) & 1);
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
            const int64_t t0 = tb + 16 * i;
            const int L = static_cast<int>((te - t0) < 16 ? (te - t0) : 16);
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
            orow += ostep;
        }
        mbar_arrive(bar_empty + 8 * st);
    }

    if (s_out != nullptr) {
        float *SF = s_out + sbase;
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

constexpr int kBV = 64;

template <bool OUT>
cudaError_t launch(const RecurParams &p, cudaStream_t stream) {
    using Lay = RecurLayout<kBV>;
    const int64_t units = static_cast<int64_t>(p.geo.n_seqs) * (p.split_chunks > 0 ? 2 : 1);
    const int64_t ctas = units * p.geo.n_heads * Lay::kSlices;
    if (ctas <= 0) return cudaSuccess;
    kda_recurrent_kernel<kBV, OUT><<<static_cast<unsigned>(ctas), (Lay::kWarps + 1) * 32,
                                     Lay::kSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t configure_recurrent() {
    cudaError_t e = cudaFuncSetAttribute(kda_recurrent_kernel<kBV, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         RecurLayout<kBV>::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kda_recurrent_kernel<kBV, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                RecurLayout<kBV>::kSmem);
}

cudaError_t launch_recurrent(const RecurParams &p, cudaStream_t stream) {
    return launch<true>(p, stream);
}

cudaError_t launch_recurrent_state_only(const RecurParams &p, cudaStream_t stream) {
    return launch<false>(p, stream);
}

}  // namespace kda
