// Recurrent half of chunked KDA prefill on the 5th-generation tensor core
// (tcgen05, tensor memory), one CTA per (sequence, head).
//
// The method (the recurrent-propagation kernel of "Kimi K3 的三個系統設計",
// section "為什麼 FlashKDA 選擇 16-token chunks") with S_n (K x V) the state
// entering chunk n:
//
//   U_n     = Ut_n - W_n S_n
//   o_n     = Qg_n S_n + P_n U_n                    (the record's Qg and P carry scale)
//   S_{n+1} = Diag(gamma_n) S_n + Kd_n^T U_n
//
// State in tensor memory, decay carried lazily. TMEM holds Shat = Diag(c)^-1 S
// in fp32, with c_n the per-key product of the decays since the key's last
// renormalisation (c_0 = 1). Then
//
//   W_n S_n = (W_n Diag(c_n)) Shat_n,   Qg_n S_n = (Qg_n Diag(c_n)) Shat_n,
//   Shat_{n+1} = Shat_n + Diag(c_{n+1})^-1 Kd_n^T U_n,   c_{n+1} = c_n gamma_n,
//
// so a step never rescales the 128 x 128 state: the products read Shat straight
// from TMEM as the tf32 A operand, and the decay goes into the small B
// operands, which four "prep" warps build ahead of the tensor core from the
// chunk record (W and Qg times c as tf32, Kd over c_{n+1} as bf16). Before a
// step whose c_n gamma_n would fall below 1e-30 for some key, that key's
// column of Shat is multiplied back by its c and c is reset to 1 (a
// renormalisation pass over TMEM, rare unless decay is extreme). A chunk
// decay gamma below 1e-30 is raised to 1e-30 (see the prep warps), so c stays
// in [1e-30, 1] and every operand inside the fp32 / bf16 range.
//
// Warp roles (320 threads): warps 0-3 epilogue (thread v <-> TMEM lane v <->
// value channel v), warps 4-7 prep, warp 8 producer (bulk async copies of the
// chunk records into a 3-stage ring), warp 9 MMA issue (one thread) and TMEM
// owner. All hand-offs are mbarriers; every wait is bounded, and a timeout or
// a raised abort flag ends the CTA cleanly with the error word set.

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_tcgen05.cuh"

namespace kda {

namespace {

constexpr int kTcStages = 3;
constexpr int kTcThreads = 320;
constexpr int kProdWarp = 8, kMmaWarp = 9;

// B operands of one step, K-major, no swizzle (core matrix = 8 rows x 16 B)
constexpr int kB1 = 0;               // [-W c ; Qg c] tf32: N = 32 rows, K = 128 keys
constexpr int kB2 = 16384;           // Kd / c_next bf16: N = 128 keys, K = 16 tokens
constexpr int kB3 = kB2 + 4096;      // P bf16: N = 16 rows r, K = 16 tokens i
constexpr int kPrepBytes = kB3 + 512;

constexpr int kOffPrep = kTcStages * kRecBytes;
constexpr int kOffCn = kOffPrep + 2 * kPrepBytes;  // c used by B1 [2][128] f32
constexpr int kOffFac = kOffCn + 1024;             // renormalisation factors [2][128]
constexpr int kOffCfin = kOffFac + 1024;           // c after the last chunk [128]
constexpr int kOffFlag = kOffCfin + 512;           // renormalisation votes [2][4] int
constexpr int kOffMisc = kOffFlag + 32;            // TMEM base (u32), abort flag (int)
constexpr int kOffBar = kOffMisc + 32;
// barriers
constexpr int kBarFull = 0, kBarEmpty = 3, kBarPrepDone = 6, kBarMma1 = 8, kBarMma2 = 10,
              kBarUReady = 12, kBarRenorm = 13, kBarPrepSync = 14, kBarTeardown = 16,
              kNumBars = 17;
constexpr int kTcSmem = kOffBar + kNumBars * 8;

// TMEM columns
constexpr uint32_t kTS = 0;     // Shat^T fp32, 128 columns (keys)
constexpr uint32_t kTD = 128;   // two 32-column result tiles: [U part | o part]
constexpr uint32_t kTU = 192;   // U^T as bf16 pairs, 8 columns (tokens)
constexpr uint32_t kTCols = 256;

// Bounded wait that also gives up when another warp has raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag, int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1)
kda_recurrent_tc_kernel(RecurParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    const int h = blockIdx.x % H;
    const int n = blockIdx.x / H;

    const uint32_t bar0 = smem_u32(smem + kOffBar);
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
    if (tid == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(bar(kBarFull + i), 1);
            mbar_init(bar(kBarEmpty + i), 8);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(kBarPrepDone + i), 4);
            mbar_init(bar(kBarMma1 + i), 1);
            mbar_init(bar(kBarMma2 + i), 1);
            mbar_init(bar(kBarPrepSync + i), 4);
        }
        mbar_init(bar(kBarUReady), 4);
        mbar_init(bar(kBarRenorm), 4);
        mbar_init(bar(kBarTeardown), kTcThreads / 32);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) {
        tc::alloc(smem_u32(tmem_slot), kTCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = geo.cu != nullptr && (*geo.call_flags & kErrBadCu);

    int64_t tb = 0, te = 0, chunk0 = 0;
    int nck = 0;
    if (!skip) {
        if (geo.cu == nullptr) {
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
    }
    const uint8_t *rec0 = p.rec + (chunk0 * H + h) * static_cast<int64_t>(kRecBytes);
    const uint32_t sbase_u32 = smem_u32(smem);
    const int64_t sbase = (static_cast<int64_t>(n) * H + h) * kDim * kDim;

    if (skip) {
        // nothing to do; fall through to the teardown
    } else if (warp < 4) {
        // ============================================================ epilogue
        const int v = tid;                                 // value channel, TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
        const uint32_t tS = tmem + lane_off + kTS;
        // initial state, column v of S (zeros if none)
        for (int c0 = 0; c0 < kDim; c0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
                r[c] = __float_as_uint(p.s0 ? p.s0[sbase + (c0 + c) * kDim + v] : 0.f);
            tc::st16(tS + c0, r);
        }
        tc::st_wait();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarRenorm));   // "renormalisation" phase 0 = init
        int renorms = 1;
        const float *cn_fac = reinterpret_cast<const float *>(smem + kOffFac);
        const int *flags = reinterpret_cast<const int *>(smem + kOffFlag);
        __nv_bfloat16 *outp = static_cast<__nv_bfloat16 *>(p.out);
        bool ok = true;
        for (int i = 0; i < nck && ok; ++i) {
            const int s = i % kTcStages, b = i & 1;
            const uint32_t tD = tmem + lane_off + kTD + 32 * b;
            if (!wait_or_abort(bar(kBarFull + s), (i / kTcStages) & 1, abort_flag, p.err)) break;
            const uint8_t *stg = smem + s * kRecBytes;
            float ut[16];
            {
                const uint4 u0 = *reinterpret_cast<const uint4 *>(stg + kRecUt + v * 32);
                const uint4 u1 = *reinterpret_cast<const uint4 *>(stg + kRecUt + v * 32 + 16);
                const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float2 f = unpack_bf16(w[c]);
                    ut[2 * c] = f.x;
                    ut[2 * c + 1] = f.y;
                }
            }
            if (!wait_or_abort(bar(kBarPrepDone + b), (i >> 1) & 1, abort_flag, p.err)) break;
            if (flags[4 * b] | flags[4 * b + 1] | flags[4 * b + 2] | flags[4 * b + 3]) {
                // renormalise the flagged keys' columns before this step's products
                tc::fence_after();
                const float *fac = cn_fac + 128 * b;
                for (int c0 = 0; c0 < kDim; c0 += 16) {
                    uint32_t r[16];
                    tc::ld16(tS + c0, r);
                    tc::ld_wait();
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        r[c] = __float_as_uint(__uint_as_float(r[c]) * fac[c0 + c]);
                    tc::st16(tS + c0, r);
                }
                tc::st_wait();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kBarRenorm));
                ++renorms;
            }
            // U^T row v = Ut^T row v + (-(W c) Shat)^T row v
            if (!wait_or_abort(bar(kBarMma1 + b), (i >> 1) & 1, abort_flag, p.err)) break;
            tc::fence_after();
            {
                uint32_t r[16];
                tc::ld16(tD, r);
                tc::ld_wait();
                uint32_t pk[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    pk[c] = pack_bf16(ut[2 * c] + __uint_as_float(r[2 * c]),
                                      ut[2 * c + 1] + __uint_as_float(r[2 * c + 1]));
                tc::st8(tmem + lane_off + kTU, pk);
                tc::st_wait();
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarUReady));
            // o row tokens of column v
            if (!wait_or_abort(bar(kBarMma2 + b), (i >> 1) & 1, abort_flag, p.err)) break;
            tc::fence_after();
            {
                uint32_t r[16];
                tc::ld16(tD + 16, r);
                tc::ld_wait();
                const int64_t t0 = tb + 16 * static_cast<int64_t>(i);
                const int L = static_cast<int>((te - t0) < 16 ? (te - t0) : 16);
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    if (c < L)
                        outp[((t0 + c) * H + h) * kDim + v] =
                            __float2bfloat16_rn(__uint_as_float(r[c]));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarEmpty + s));
            (void)renorms;
        }
        // final state: S = Diag(c) Shat, column v
        if (!*abort_flag && p.s_final != nullptr) {
            tc::fence_after();
            const float *cfin = reinterpret_cast<const float *>(smem + kOffCfin);
            for (int c0 = 0; c0 < kDim; c0 += 16) {
                uint32_t r[16];
                tc::ld16(tS + c0, r);
                tc::ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    p.s_final[sbase + (c0 + c) * kDim + v] =
                        __uint_as_float(r[c]) * (nck > 0 ? cfin[c0 + c] : 1.f);
            }
        }
    } else if (warp < 8) {
        // ================================================================ prep
        const int pt = tid - 128;   // 0..127: owns key pt's running c
        const int pw = warp - 4;
        float c = 1.f;
        float *cn = reinterpret_cast<float *>(smem + kOffCn);
        float *fac = reinterpret_cast<float *>(smem + kOffFac);
        int *flags = reinterpret_cast<int *>(smem + kOffFlag);
        for (int i = 0; i < nck; ++i) {
            const int s = i % kTcStages, b = i & 1;
            if (!wait_or_abort(bar(kBarFull + s), (i / kTcStages) & 1, abort_flag, p.err)) break;
            if (i >= 2 &&
                !wait_or_abort(bar(kBarMma2 + b), ((i - 2) >> 1) & 1, abort_flag, p.err))
                break;
            const uint8_t *stg = smem + s * kRecBytes;
            uint8_t *buf = smem + kOffPrep + b * kPrepBytes;
            // decay bookkeeping for key pt
            // a decay below 1e-30 (down to 0: a key that forgets at once) is
            // taken as 1e-30, so 1 / c stays finite; the state row then keeps
            // 1e-30 of its old value, far below fp32 resolution of the new one
            const float g = fmaxf(reinterpret_cast<const float *>(stg + kRecGamma)[pt], 1e-30f);
            const bool ren = c * g < 1e-30f;
            fac[128 * b + pt] = ren ? c : 1.f;
            const float cu = ren ? 1.f : c;
            cn[128 * b + pt] = cu;
            c = cu * g;
            const int vote = __any_sync(0xffffffffu, ren) ? 1 : 0;
            if (lane == 0) flags[4 * b + pw] = vote;
            if (i == nck - 1) reinterpret_cast<float *>(smem + kOffCfin)[pt] = c;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPrepSync + b));
            if (!wait_or_abort(bar(kBarPrepSync + b), (i >> 1) & 1, abort_flag, p.err)) break;
            __syncwarp();
            // B1: row r (0-15: -W, 16-31: Qg) times c, keys [32 kq, 32 kq + 32), tf32
            {
                const int r = pt >> 2, kq = pt & 3;
                const uint8_t *tile = stg + (r < 16 ? kRecW : kRecQg);
                const int rr = r & 15;
                const float *cu4 = cn + 128 * b;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int key = 32 * kq + 4 * j;
                    const uint2 w = *reinterpret_cast<const uint2 *>(tile + swz(rr, key));
                    const float4 cc = *reinterpret_cast<const float4 *>(cu4 + key);
                    const float2 w01 = unpack_bf16(w.x), w23 = unpack_bf16(w.y);
                    *reinterpret_cast<float4 *>(buf + kB1 + (r >> 3) * 4096 + (key >> 2) * 128 +
                                                (r & 7) * 16) =
                        make_float4(w01.x * cc.x, w01.y * cc.y, w23.x * cc.z, w23.y * cc.w);
                }
            }
            // B2: key pt, 16 tokens of Kd / c_next, bf16
            {
                const float inv = 1.f / c;
                uint32_t pk[8];
#pragma unroll
                for (int t = 0; t < 16; t += 2) {
                    const float k0 = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16 *>(stg + kRecKd + swz(t, pt)));
                    const float k1 = __bfloat162float(
                        *reinterpret_cast<const __nv_bfloat16 *>(stg + kRecKd + swz(t + 1, pt)));
                    pk[t >> 1] = pack_bf16(k0 * inv, k1 * inv);
                }
                uint8_t *dst = buf + kB2 + (pt >> 3) * 256 + (pt & 7) * 16;
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(dst + 128) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            // B3: P in core-matrix order (one warp)
            if (pw == 0) {
                const int r = lane >> 1, hf = lane & 1;
                const uint4 pv = *reinterpret_cast<const uint4 *>(stg + kRecP + r * 32 + hf * 16);
                *reinterpret_cast<uint4 *>(buf + kB3 + (r >> 3) * 256 + hf * 128 + (r & 7) * 16) = pv;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(kBarPrepDone + b));
                mbar_arrive(bar(kBarEmpty + s));
            }
        }
    } else if (warp == kProdWarp) {
        // ============================================================ producer
        if (lane == 0) {
            for (int i = 0; i < nck; ++i) {
                const int s = i % kTcStages;
                if (i >= kTcStages &&
                    !wait_or_abort(bar(kBarEmpty + s), ((i / kTcStages) - 1) & 1, abort_flag,
                                   p.err))
                    break;
                const uint8_t *src = rec0 + static_cast<int64_t>(i) * H * kRecBytes;
                mbar_arrive_expect_tx(bar(kBarFull + s), kRecBytes);
                bulk_g2s(sbase_u32 + s * kRecBytes, src, kRecBytes, bar(kBarFull + s));
            }
        }
    } else {
        // ============================================================ MMA issue
        if (lane == 0) {
            const uint32_t tS = tmem + kTS, tU = tmem + kTU;
            const int *flags = reinterpret_cast<const int *>(smem + kOffFlag);
            int renorms = 0;
            bool ok = wait_or_abort(bar(kBarRenorm), 0, abort_flag, p.err);   // initial state in
            renorms = 1;
            for (int i = 0; i < nck && ok; ++i) {
                const int b = i & 1;
                const uint32_t tD = tmem + kTD + 32 * b;
                const uint32_t buf = sbase_u32 + kOffPrep + b * kPrepBytes;
                if (!wait_or_abort(bar(kBarPrepDone + b), (i >> 1) & 1, abort_flag, p.err)) break;
                if (flags[4 * b] | flags[4 * b + 1] | flags[4 * b + 2] | flags[4 * b + 3]) {
                    if (!wait_or_abort(bar(kBarRenorm), renorms & 1, abort_flag, p.err)) break;
                    ++renorms;
                }
                tc::fence_after();
                // U part: D[:, 0:16] = Shat^T (-(W c))^T
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    tc::mma_tf32_ts(tD, tS + 8 * kk, tc::sdesc(buf + kB1 + kk * 256, 128, 4096),
                                    tc::idesc(128, 16, 2), kk > 0);
                tc::commit(bar(kBarMma1 + b));
                // o part: D[:, 16:32] = Shat^T (Qg c)^T
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    tc::mma_tf32_ts(tD + 16, tS + 8 * kk,
                                    tc::sdesc(buf + kB1 + 2 * 4096 + kk * 256, 128, 4096),
                                    tc::idesc(128, 16, 2), kk > 0);
                if (!wait_or_abort(bar(kBarUReady), i & 1, abort_flag, p.err)) break;
                tc::fence_after();
                // Shat += U^T (Kd / c_next)^T ;  o part += U^T P^T
                tc::mma_bf16_ts(tS, tU, tc::sdesc(buf + kB2, 128, 256), tc::idesc(128, 128, 1), 1);
                tc::mma_bf16_ts(tD + 16, tU, tc::sdesc(buf + kB3, 128, 256), tc::idesc(128, 16, 1),
                                1);
                tc::commit(bar(kBarMma2 + b));
            }
        }
    }

    // ============================================================ teardown
    tc::fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarTeardown));
    if (warp == kMmaWarp) {
        wait_or_abort(bar(kBarTeardown), 0, abort_flag, p.err);
        tc::fence_after();
        tc::dealloc(tmem, kTCols);
    }
}

}  // namespace

cudaError_t configure_recurrent_tc() {
    return cudaFuncSetAttribute(kda_recurrent_tc_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
}

cudaError_t launch_recurrent_tc(const RecurParams &p, cudaStream_t stream) {
    const int64_t ctas = static_cast<int64_t>(p.geo.n_seqs) * p.geo.n_heads;
    if (ctas <= 0) return cudaSuccess;
    kda_recurrent_tc_kernel<<<static_cast<unsigned>(ctas), kTcThreads, kTcSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
