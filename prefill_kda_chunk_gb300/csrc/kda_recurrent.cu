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
#include "kda_recurrent_body.cuh"

namespace kda {

namespace {

// OUT = false carries only the state (no output products, no o stores): the
// maps launch of the segment-parallel scan.
template <int BV, bool OUT>
__global__ void __launch_bounds__((BV / 16 + 1) * 32)
kda_recurrent_kernel(RecurParams p) {
    using Lay = RecurLayout<BV>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    const bool scan = geo.cu == nullptr && p.scan_segs >= 2;
    // slices per unit: 2 (value columns), or 4 in the maps launch (value
    // columns, then the columns of the segment's transition map)
    const int nsl = scan && !OUT ? 2 * Lay::kSlices : Lay::kSlices;
    const int sl = blockIdx.x % nsl;
    const int s = sl % Lay::kSlices;
    const bool virt = sl >= Lay::kSlices;   // a column slice of the map M
    const int h = (blockIdx.x / nsl) % H;
    const int n = blockIdx.x / (nsl * H);   // unit: sequence, or (sequence, segment)

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
    if (scan) {
        // segment j of sequence seq: chunks [j L, min((j + 1) L, chunks))
        const int P = p.scan_segs;
        const int per = OUT ? P : P - 1;   // segments of a sequence in this launch
        const int j = n % per;
        seq = n / per;
        if (virt && j == 0) return;        // the first segment starts from s0: no map
        const int64_t L = p.scan_len, cps = (geo.seq_len + 15) / 16;
        const int64_t c0 = j * L, c1 = (j + 1) * L < cps ? (j + 1) * L : cps;
        const int64_t base = static_cast<int64_t>(seq) * geo.seq_len;
        tb = base + 16 * c0;
        te = base + (16 * c1 < geo.seq_len ? 16 * c1 : geo.seq_len);
        chunk0 = static_cast<int64_t>(seq) * geo.slot_stride + c0;
        nck = static_cast<int>(c1 - c0);
        const int64_t plane = static_cast<int64_t>(geo.n_seqs) * H * kDim * kDim;
        if (OUT) {
            s_in = j == 0 ? p.s0 : p.seg_entry + (j - 1) * plane;
            s_out = j == P - 1 ? p.s_final : nullptr;
        } else {
            s_in = j == 0 ? p.s0 : nullptr;
            s_out = j == 0 ? p.seg_entry : (virt ? p.seg_m : p.seg_c) + (j - 1) * plane;
        }
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
    const unsigned long long wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;

    if (warp == Lay::kWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            for (int i = 0; i < nck; ++i) {
                if (i == p.stall_chunk) break;   // test hook: the consumers' wait runs out
                const int st = i % kStages;
                if (i >= kStages &&
                    !mbar_wait(bar_empty + 8 * st, ((i / kStages) - 1) & 1, wait_ns)) {
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
    if (virt) {
        // the identity: column v0 + gid (+ 8) of M starts as the unit vector
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int key = 8 * j + 2 * tig, c = v0 + gid;
            acc[j][0] = key == c ? 1.f : 0.f;
            acc[j][1] = key + 1 == c ? 1.f : 0.f;
            acc[j][2] = key == c + 8 ? 1.f : 0.f;
            acc[j][3] = key + 1 == c + 8 ? 1.f : 0.f;
        }
    } else {
        recur_load_state(acc, s_in != nullptr ? s_in + sbase : nullptr, v0);
    }

    uint8_t *so = smem + Lay::kOStage + warp * 512;   // [16 tok][16 val] bf16
    __nv_bfloat16 *outp = static_cast<__nv_bfloat16 *>(p.out);

    bool ready = false;
    __nv_bfloat16 *orow = outp + (tb * H + h) * kDim + v0;   // row 0 of the chunk's o tile
    const int64_t ostep = 16 * static_cast<int64_t>(H) * kDim;
    for (int i = 0; i < nck; ++i) {
        const int st = i % kStages;
        if (!ready && !mbar_wait(bar_full + 8 * st, (i / kStages) & 1, wait_ns)) {
            atomicOr(p.err, kErrTimeout);
            break;
        }
        const uint8_t *stg = smem + st * Lay::kStageBytes;
        const uint32_t sw = stage0 + st * Lay::kStageBytes;
        ready = recur_step<OUT>(acc, stg, sw, vw, virt, so, orow,
                                static_cast<int>((te - (tb + 16 * i)) < 16 ? (te - (tb + 16 * i)) : 16), H,
                                [&] {
                                    return i + 1 < nck &&
                                           mbar_test(bar_full + 8 * ((i + 1) % kStages), ((i + 1) / kStages) & 1);
                                });
        if constexpr (OUT) orow += ostep;
        mbar_arrive(bar_empty + 8 * st);
    }

    if (s_out != nullptr) recur_store_state(acc, s_out + sbase, v0);
}

// Serial combine of the segment-parallel scan, one CTA per (sequence, head,
// block of 32 value columns): E_{j+1} = M_j E_j + c_j in fp32 for the entry
// states E of segments 2 .. P-1, the column block of E kept in shared memory
// and M_j staged there whole.
constexpr int kCombineCols = 32;
constexpr int kCombineSmem = (kDim * kDim + 2 * kDim * kCombineCols) * 4;

__global__ void __launch_bounds__(256) kda_scan_combine_kernel(RecurParams p) {
    extern __shared__ __align__(16) float csm[];
    float *Ms = csm;                              // [128][128]
    float *E = csm + kDim * kDim;                 // [2][128][32]
    const int tid = threadIdx.x;
    const int nblk = kDim / kCombineCols;
    const int cb = blockIdx.x % nblk;
    const int64_t unit = blockIdx.x / nblk;       // sequence * H + head
    const int64_t plane = static_cast<int64_t>(p.geo.n_seqs) * p.geo.n_heads * kDim * kDim;
    const int64_t ub = unit * kDim * kDim;
    // thread: row r = tid / 2, columns 16 (tid % 2) .. + 15 of the block
    const int r = tid >> 1, c0 = 16 * (tid & 1);
    for (int i = tid; i < kDim * kCombineCols; i += 256)
        E[i] = p.seg_entry[ub + (i / kCombineCols) * kDim + cb * kCombineCols + i % kCombineCols];
    for (int j = 1; j + 1 < p.scan_segs; ++j) {
        const float *Mg = p.seg_m + (j - 1) * plane + ub;
        const float *Cg = p.seg_c + (j - 1) * plane + ub;
        float *Eo = p.seg_entry + j * plane + ub;
        const float *Ein = E + ((j - 1) & 1) * kDim * kCombineCols;
        float *Eout = E + (j & 1) * kDim * kCombineCols;
        __syncthreads();   // the previous step's E is complete and Ms is free
        for (int i = tid; i < kDim * kDim / 4; i += 256)
            reinterpret_cast<float4 *>(Ms)[i] = reinterpret_cast<const float4 *>(Mg)[i];
        __syncthreads();
        float acc[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[c] = Cg[r * kDim + cb * kCombineCols + c0 + c];
        for (int m = 0; m < kDim; ++m) {
            const float a = Ms[r * kDim + m];
            const float4 *e4 = reinterpret_cast<const float4 *>(Ein + m * kCombineCols + c0);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 e = e4[q4];
                acc[4 * q4] = fmaf(a, e.x, acc[4 * q4]);
                acc[4 * q4 + 1] = fmaf(a, e.y, acc[4 * q4 + 1]);
                acc[4 * q4 + 2] = fmaf(a, e.z, acc[4 * q4 + 2]);
                acc[4 * q4 + 3] = fmaf(a, e.w, acc[4 * q4 + 3]);
            }
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            Eout[r * kCombineCols + c0 + c] = acc[c];
            Eo[r * kDim + cb * kCombineCols + c0 + c] = acc[c];
        }
    }
}

constexpr int kBV = 64;

template <bool OUT>
cudaError_t launch(const RecurParams &p, cudaStream_t stream) {
    using Lay = RecurLayout<kBV>;
    const bool scan = p.geo.cu == nullptr && p.scan_segs >= 2;
    const int64_t per = scan ? (OUT ? p.scan_segs : p.scan_segs - 1) : 1;
    const int64_t units = static_cast<int64_t>(p.geo.n_seqs) * per;
    const int64_t ctas = units * p.geo.n_heads * Lay::kSlices * (scan && !OUT ? 2 : 1);
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
    e = cudaFuncSetAttribute(kda_recurrent_kernel<kBV, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, RecurLayout<kBV>::kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kda_scan_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kCombineSmem);
}

cudaError_t launch_recurrent(const RecurParams &p, cudaStream_t stream) {
    return launch<true>(p, stream);
}

cudaError_t launch_recurrent_scan_maps(const RecurParams &p, cudaStream_t stream) {
    return launch<false>(p, stream);
}

cudaError_t launch_scan_combine(const RecurParams &p, cudaStream_t stream) {
    if (p.scan_segs <= 2) return cudaSuccess;
    const int64_t ctas = static_cast<int64_t>(p.geo.n_seqs) * p.geo.n_heads * (kDim / kCombineCols);
    if (ctas <= 0) return cudaSuccess;
    kda_scan_combine_kernel<<<static_cast<unsigned>(ctas), 256, kCombineSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
