// The per-warp work of the 16-token intra-chunk kernels (the intra-chunk
// kernel, its exact-form companion and the fused kernel's record builders):
// for every 16-token chunk of every head and independently of every other
// chunk ("Kimi K3 的三個系統設計", section "為什麼 FlashKDA 選擇 16-token
// chunks": the token-parallel kernel, the 16x16 inversion, the MMA-shaped
// tiles), with G_r = sum_{u<=r} g_u the chunk-local cumulative log decay
// (per key channel):
//
//   A[r,i] = beta_r sum_c k_rc k_ic exp(G_rc - G_ic)   (i < r), as the MMA
//            (K * exp(G)) (K * exp(-G))^T, then masked and row-scaled by beta
//   P[r,i] = sum_c q_rc k_ic exp(G_rc - G_ic)           (i <= r), likewise
//   Tm     = (I + A)^{-1} by forward substitution (unit lower triangular)
//   W      = Tm diag(beta) (K * exp(G)),   Ut = Tm diag(beta) V
//
// stored per (chunk, head) as the record the recurrent kernel consumes: -W,
// scale*Q*exp(G), K*exp(G_last - G), scale*P, exp(G_last) and Ut^T (the
// output scale rides on the two output operands). Rows past the end of a
// sequence are zero (their k, v, q, beta and g are taken as 0).
//
// KEEP = false stores records evict-first (st.global.cs: the separate
// recurrent kernel reads them back long after they leave L2); KEEP = true
// stores them normally (the fused kernel's ring is read from L2 a few chunks
// later).
#pragma once

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

template <bool KEEP, typename T>
__device__ __forceinline__ void st_rec(T *ptr, T v) {
    if constexpr (KEEP) *ptr = v;
    else __stcs(ptr, v);
}

constexpr int kIntraWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the special-function unit. The factored form keeps inputs within
// +-116; the exact form of strongly decaying chunks can go far below, where
// the result flushes to 0 (its true value is below fp32's normal range)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The same, but never merged with an earlier 2^x of the same input (which
// would keep that value alive in a register all the while)
__device__ __forceinline__ float ex2_again(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// two fp32 products in one packed instruction
__device__ __forceinline__ float2 mul2v(float2 a, float2 b) {
    float2 d;
    asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
        " mul.rn.f32x2 z, x, y;\n mov.b64 {%0, %1}, z;\n}\n"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

struct IntraWarpSmem {
    uint8_t kg[4096];   // K as loaded, then K*exp(G); swizzled
    uint8_t kn[4096];   // K*exp(-G), swizzled; later stages -W
    uint8_t qg[4096];   // Q as loaded, then scale*Q*exp(G); swizzled
    uint8_t v[4096];    // V, swizzled
    float a[16 * 17];   // masked, beta-scaled A
    float t[16 * 17];   // (I + A)^{-1}
};

__device__ __forceinline__ bool locate_chunk(const ChunkGeometry &geo, int64_t c, int &n,
                                             int64_t &t0, int &L, int64_t &rec_idx) {
    if (geo.cu == nullptr) {
        const int64_t per = geo.seg_len;
        n = static_cast<int>(c / per);
        if (n >= geo.n_seqs) return false;
        const int64_t il = c - static_cast<int64_t>(n) * per;
        const int64_t i = geo.pos_begin + il;
        t0 = static_cast<int64_t>(n) * geo.seq_len + 16 * i;
        const int64_t rem = geo.seq_len - 16 * i;
        if (rem <= 0) return false;
        L = static_cast<int>(rem < 16 ? rem : 16);
        rec_idx = static_cast<int64_t>(n) * geo.slot_stride + il;
        return true;
    }
    const int32_t *off = geo.chunk_off;
    if (c >= off[geo.n_seqs]) return false;
    int lo = 0, hi = geo.n_seqs;  // off[lo] <= c < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= c) lo = mid; else hi = mid;
    }
    n = lo;
    t0 = static_cast<int64_t>(geo.cu[n]) + 16 * (c - off[n]);
    const int64_t rem = static_cast<int64_t>(geo.cu[n + 1]) - t0;
    L = static_cast<int>(rem < 16 ? rem : 16);
    rec_idx = c;
    return true;
}

// Queues the chunk's q, k, v rows as 16-byte async copies into their swizzled
// tiles; rows at or past L are zero-filled without a read.
__device__ __forceinline__ void load_chunk(const IntraParams &p, IntraWarpSmem &sm, int64_t t0,
                                           int L, int h, int lane) {
    const int H = p.geo.n_heads;
    const int64_t rowe = static_cast<int64_t>(H) * kDim;
    const int64_t base = (t0 * H + h) * kDim;
    const __nv_bfloat16 *qp = static_cast<const __nv_bfloat16 *>(p.q) + base;
    const __nv_bfloat16 *kp = static_cast<const __nv_bfloat16 *>(p.k) + base;
    const __nv_bfloat16 *vp = static_cast<const __nv_bfloat16 *>(p.v) + base;
    const uint32_t sq = smem_u32(sm.qg), sk = smem_u32(sm.kg), sv = smem_u32(sm.v);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int idx = lane + 32 * j, r = idx >> 4, c = idx & 15;
        const uint32_t dst = r * 256 + ((c ^ (r & 7)) << 4);
        const int rr = r < L ? r : 0;
        const uint32_t nb = r < L ? 16u : 0u;
        cp_async16(sq + dst, qp + rr * rowe + c * 8, nb);
        cp_async16(sk + dst, kp + rr * rowe + c * 8, nb);
        cp_async16(sv + dst, vp + rr * rowe + c * 8, nb);
    }
    cp_async_commit();
}

// The chunk's gating, A and P without factoring exp(G_r - G_i) as
// exp(G_r) exp(-G_i) about the chunk start, for chunks whose cumulative log
// decay leaves [-80, 80] in some channel (strong decay: exp(-G) would
// overflow and exp(G) underflow).
//
// Every pair i < r of the chunk lies in exactly one block of the binary
// split of its 16 rows: for half-block size s = 8, 4, 2, 1, the rows r with
// bit s set against the rows i of the same 2s-block with it clear. Within a
// block, factoring about its boundary row m (the last of the lower half),
//
//   exp(G_r - G_i) = exp(G_r - G_m) exp(G_m - G_i),   i <= m < r,
//
// both factors are at most 1 under decay (G non-increasing), and each is at
// least the product, so nothing overflows and a factor underflows only where
// the exact value is below fp32's range too. One level is one 16x8 tensor-core
// product over the 128 channels: rows (K, Q of the 8 upper-half tokens, each
// times exp(G_r - G_m)) against columns (K of the 8 lower-half tokens, each
// times exp(G_m - G_i)); entries that pair different blocks are dropped. The
// diagonal of P (exp(0) = 1) is one plain Q K^T product. Growth above exp(80)
// between two points of the chunk (positive gates) still sets kErrGate.
//
// Same outputs as the factored code: sm.kg = K e^G (bf16, swizzled), sm.a =
// the masked, beta-scaled A, and the record's scale Q e^G, K e^(G_last - G),
// scale P and exp(G_last). Reads the raw q, k tiles (dividing q and k by their
// L2 norms first when pre asks). Scratch while it runs: the level's row tile
// in sm.kg, its column tile in sm.a / sm.t (2 KB of their 2176 B).
template <bool KEEP>
__device__ __forceinline__ void intra_exact_chunk(const float *gp, int64_t rowe, int L, int pre,
                                               float scale, float beta_l,
                                               IntraWarpSmem *smp, uint8_t *rec, int *err) {
    IntraWarpSmem &sm = *smp;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3, quad = lane >> 3;

    // cumulative log decay (base-2 units) of this lane's channels 4 lane..+3,
    // and the largest rise of G over the chunk (from 0 before the first row)
    float G[16][4];
    {
        float run[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f}, rise = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float4 gg = (r < L) ? __ldg(reinterpret_cast<const float4 *>(gp + r * rowe))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            if ((pre & kPreGateLogits) && r < L) {
                gg.x = log_sigmoid(gg.x); gg.y = log_sigmoid(gg.y);
                gg.z = log_sigmoid(gg.z); gg.w = log_sigmoid(gg.w);
            }
            run[0] += gg.x; run[1] += gg.y; run[2] += gg.z; run[3] += gg.w;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                rise = fmaxf(rise, run[e] - lo[e]);
                lo[e] = fminf(lo[e], run[e]);
                G[r][e] = run[e] * kLog2e;
            }
        }
        if (__any_sync(0xffffffffu, !(rise <= 80.f)) && lane == 0) atomicOr(err, kErrGate);
    }

    // ---- per row: (normalised) q to sm.qg and k to sm.kn as bf16; scale
    //      Q e^G and K e^(G_last - G) to the record
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int off = swz(r, 4 * lane);
        const uint2 qq = *reinterpret_cast<const uint2 *>(sm.qg + off);
        const uint2 kk = *reinterpret_cast<const uint2 *>(sm.kg + off);
        const float2 q01 = unpack_bf16(qq.x), q23 = unpack_bf16(qq.y);
        const float2 k01 = unpack_bf16(kk.x), k23 = unpack_bf16(kk.y);
        float q[4] = {q01.x, q01.y, q23.x, q23.y}, k[4] = {k01.x, k01.y, k23.x, k23.y};
        if (pre & kPreNormQK) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) { sq = fmaf(q[e], q[e], sq); sk = fmaf(k[e], k[e], sk); }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            const float rq = rsqrtf(sq + kNormEps), rk = rsqrtf(sk + kNormEps);
#pragma unroll
            for (int e = 0; e < 4; ++e) { q[e] *= rq; k[e] *= rk; }
            *reinterpret_cast<uint2 *>(sm.qg + off) =
                make_uint2(pack_bf16(q[0], q[1]), pack_bf16(q[2], q[3]));
        }
        *reinterpret_cast<uint2 *>(sm.kn + off) =
            make_uint2(pack_bf16(k[0], k[1]), pack_bf16(k[2], k[3]));
        float qg[4], kd[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qg[e] = q[e] * scale * ex2(G[r][e]);
            kd[e] = k[e] * ex2(G[15][e] - G[r][e]);
        }
        const uint2 uqg = make_uint2(pack_bf16(qg[0], qg[1]), pack_bf16(qg[2], qg[3]));
        st_rec<KEEP>(reinterpret_cast<uint2 *>(rec + kRecQg + off), uqg);
        st_rec<KEEP>(reinterpret_cast<uint2 *>(rec + kRecKd + off),
               make_uint2(pack_bf16(kd[0], kd[1]), pack_bf16(kd[2], kd[3])));
    }
    st_rec<KEEP>(reinterpret_cast<float4 *>(rec + kRecGamma + 16 * lane),
           make_float4(ex2(G[15][0]), ex2(G[15][1]), ex2(G[15][2]), ex2(G[15][3])));
    __syncwarp();

    // ---- the four levels of the split, then the diagonal of P
    const uint32_t s_row = smem_u32(sm.kg), s_col = smem_u32(sm.a);
    const uint32_t s_q = smem_u32(sm.qg), s_k = smem_u32(sm.kn);
    uint8_t *const col_tile = reinterpret_cast<uint8_t *>(sm.a);
    float acc[4][4] = {};
#pragma unroll
    for (int lv = 0; lv < 4; ++lv) {
        const int sz = 8 >> lv;   // half-block size s
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            // a-th upper-half token r and a-th lower-half token i, with the
            // boundary rows of their blocks
            const int r = 2 * sz * (a / sz) + sz + a % sz, mr = r - a % sz - 1;
            const int i = 2 * sz * (a / sz) + a % sz, mi = i - a % sz + sz - 1;
            const uint2 kr2 = *reinterpret_cast<const uint2 *>(sm.kn + swz(r, 4 * lane));
            const uint2 qr2 = *reinterpret_cast<const uint2 *>(sm.qg + swz(r, 4 * lane));
            const uint2 ki2 = *reinterpret_cast<const uint2 *>(sm.kn + swz(i, 4 * lane));
            const float2 kr01 = unpack_bf16(kr2.x), kr23 = unpack_bf16(kr2.y);
            const float2 qr01 = unpack_bf16(qr2.x), qr23 = unpack_bf16(qr2.y);
            const float2 ki01 = unpack_bf16(ki2.x), ki23 = unpack_bf16(ki2.y);
            const float kr[4] = {kr01.x, kr01.y, kr23.x, kr23.y};
            const float qr[4] = {qr01.x, qr01.y, qr23.x, qr23.y};
            const float ki[4] = {ki01.x, ki01.y, ki23.x, ki23.y};
            float fr[4], fi[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                fr[e] = ex2(G[r][e] - G[mr][e]);
                fi[e] = (mi == i) ? 1.f : ex2(G[mi][e] - G[i][e]);
            }
            *reinterpret_cast<uint2 *>(sm.kg + swz(a, 4 * lane)) =
                make_uint2(pack_bf16(kr[0] * fr[0], kr[1] * fr[1]),
                           pack_bf16(kr[2] * fr[2], kr[3] * fr[3]));
            *reinterpret_cast<uint2 *>(sm.kg + swz(a + 8, 4 * lane)) =
                make_uint2(pack_bf16(qr[0] * fr[0], qr[1] * fr[1]),
                           pack_bf16(qr[2] * fr[2], qr[3] * fr[3]));
            *reinterpret_cast<uint2 *>(col_tile + swz(a, 4 * lane)) =
                make_uint2(pack_bf16(ki[0] * fi[0], ki[1] * fi[1]),
                           pack_bf16(ki[2] * fi[2], ki[3] * fi[3]));
            // one token pair at a time: keeps the live registers within the
            // kernel's budget
            asm volatile("" ::: "memory");
        }
        __syncwarp();
#pragma unroll
        for (int kk = 0; kk < 8; kk += 2) {
            uint32_t b[4];
            ldsm_x4(s_col + swz(lane & 7, (2 * kk + quad) * 8), b[0], b[1], b[2], b[3]);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t af[4];
                const int ra = (quad & 1) * 8 + (lane & 7), ca = (2 * (kk + h2) + (quad >> 1)) * 8;
                ldsm_x4(s_row + swz(ra, ca), af[0], af[1], af[2], af[3]);
                mma16816(acc[lv], af, b[2 * h2], b[2 * h2 + 1]);
            }
        }
        __syncwarp();
    }
    // K e^G for W, into sm.kg (free again; the last use of G)
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int off = swz(r, 4 * lane);
        const uint2 kk = *reinterpret_cast<const uint2 *>(sm.kn + off);
        const float2 k01 = unpack_bf16(kk.x), k23 = unpack_bf16(kk.y);
        *reinterpret_cast<uint2 *>(sm.kg + off) =
            make_uint2(pack_bf16(k01.x * ex2_again(G[r][0]), k01.y * ex2_again(G[r][1])),
                       pack_bf16(k23.x * ex2_again(G[r][2]), k23.y * ex2_again(G[r][3])));
    }
    float accd[2][4] = {};   // Q K^T, for its diagonal
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t aq[4], b[4];
        const int ra = (quad & 1) * 8 + (lane & 7), ca = (2 * kk + (quad >> 1)) * 8;
        ldsm_x4(s_q + swz(ra, ca), aq[0], aq[1], aq[2], aq[3]);
        const int rb = (quad >> 1) * 8 + (lane & 7), cb = (2 * kk + (quad & 1)) * 8;
        ldsm_x4(s_k + swz(rb, cb), b[0], b[1], b[2], b[3]);
        mma16816(accd[0], aq, b[0], b[1]);
        mma16816(accd[1], aq, b[2], b[3]);
    }

    // ---- scatter: A (beta-scaled) to sm.a, scale P to sm.t, zeros elsewhere
    for (int x = lane; x < 16 * 17; x += 32) { sm.a[x] = 0.f; sm.t[x] = 0.f; }
    __syncwarp();
#pragma unroll
    for (int lv = 0; lv < 4; ++lv) {
        const int sz = 8 >> lv;
        // fragment row gid: K of upper token a = gid (an A entry); row gid + 8:
        // Q of the same token (a P entry); columns: lower tokens b = 2 tig, +1
        const int a = gid, r = 2 * sz * (a / sz) + sz + a % sz;
        const float beta_r = __shfl_sync(0xffffffffu, beta_l, r);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int b = 2 * tig + cc, i = 2 * sz * (b / sz) + b % sz;
            if (a / sz == b / sz) {
                sm.a[r * 17 + i] = beta_r * acc[lv][cc];
                sm.t[r * 17 + i] = scale * acc[lv][2 + cc];
            }
        }
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        if (2 * tig + cc == gid) {
            sm.t[gid * 17 + gid] = scale * accd[0][cc];
            sm.t[(gid + 8) * 17 + gid + 8] = scale * accd[1][2 + cc];
        }
    }
    __syncwarp();
    // scale P to the record: 128 words of two bf16, four per lane
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int w = lane + 32 * it, r = w >> 3, i = 2 * (w & 7);
        st_rec<KEEP>(reinterpret_cast<unsigned int *>(rec + kRecP) + w,
               pack_bf16(sm.t[r * 17 + i], sm.t[r * 17 + i + 1]));
    }
    __syncwarp();
}

// The part of an item common to both forms: Tm = (I + A)^{-1} from sm.a,
// then W = Tm diag(beta) (K e^G) from sm.kg and Ut^T = (Tm diag(beta) V)^T
// from sm.v, both to the record; Tm itself to tout ([16] rows of 20 fp32, the
// last 4 zero) when TOUT and tout is not null.
template <bool KEEP, bool TOUT = true>
__device__ __forceinline__ void intra_tail(IntraWarpSmem &sm, uint8_t *rec, float *tout,
                                           float beta_l, int lane, float wscale = 1.f) {
    const int gid = lane >> 2, tig = lane & 3, quad = lane >> 3;
    const uint32_t s_kg = smem_u32(sm.kg), s_v = smem_u32(sm.v);

    // ---- Tm = (I + A)^{-1}: lane j (< 16) solves column j by forward substitution
    {
        const int j = lane & 15;
        float tc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float s = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) s = fmaf(-sm.a[r * 17 + i], tc[i], s);
            tc[r] = s;
        }
        if (lane < 16) {
#pragma unroll
            for (int r = 0; r < 16; ++r) sm.t[r * 17 + j] = tc[r];
        }
    }
    __syncwarp();
    if (TOUT && tout != nullptr) {
        // whole rows, the 4 pad columns as zeros: every 32-byte sector of the
        // item is written in full (no read of partly written sectors)
#pragma unroll
        for (int it = 0; it < 10; ++it) {
            const int e = lane + 32 * it, r = e / 20, col = e - 20 * r;
            __stcs(tout + e, col < 16 ? sm.t[r * 17 + col] : 0.f);
        }
    }

    // ---- A fragments of Tm diag(beta) (bf16)
    uint32_t aT[4];
    {
        const int c0 = 2 * tig, c1 = 2 * tig + 8;
        const float b0 = __shfl_sync(0xffffffffu, beta_l, c0);
        const float b1 = __shfl_sync(0xffffffffu, beta_l, c0 + 1);
        const float b2 = __shfl_sync(0xffffffffu, beta_l, c1);
        const float b3 = __shfl_sync(0xffffffffu, beta_l, c1 + 1);
        aT[0] = pack_bf16(sm.t[gid * 17 + c0] * b0, sm.t[gid * 17 + c0 + 1] * b1);
        aT[1] = pack_bf16(sm.t[(gid + 8) * 17 + c0] * b0, sm.t[(gid + 8) * 17 + c0 + 1] * b1);
        aT[2] = pack_bf16(sm.t[gid * 17 + c1] * b2, sm.t[gid * 17 + c1 + 1] * b3);
        aT[3] = pack_bf16(sm.t[(gid + 8) * 17 + c1] * b2, sm.t[(gid + 8) * 17 + c1 + 1] * b3);
    }

    // ---- W = Tm diag(beta) (K e^G): stage -W (bf16, swizzled) in sm.kn
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
        uint32_t b[4];
        const int rk = (quad & 1) * 8 + (lane & 7), ck = (2 * jp + (quad >> 1)) * 8;
        ldsm_x4_t(s_kg + swz(rk, ck), b[0], b[1], b[2], b[3]);
        float w0[4] = {}, w1[4] = {};
        mma16816(w0, aT, b[0], b[1]);
        mma16816(w1, aT, b[2], b[3]);
        const int c0 = 16 * jp + 2 * tig, c1 = c0 + 8;
        if (wscale != 1.f) {
#pragma unroll
            for (int e = 0; e < 4; ++e) { w0[e] *= wscale; w1[e] *= wscale; }
        }
        *reinterpret_cast<uint32_t *>(sm.kn + swz(gid, c0)) = pack_bf16(-w0[0], -w0[1]);
        *reinterpret_cast<uint32_t *>(sm.kn + swz(gid + 8, c0)) = pack_bf16(-w0[2], -w0[3]);
        *reinterpret_cast<uint32_t *>(sm.kn + swz(gid, c1)) = pack_bf16(-w1[0], -w1[1]);
        *reinterpret_cast<uint32_t *>(sm.kn + swz(gid + 8, c1)) = pack_bf16(-w1[2], -w1[3]);
    }

    // ---- Ut^T = V^T (Tm diag(beta))^T, M = value channel, N = token
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4];
        const int ri = (quad >> 1) * 8 + (lane & 7), cv = 16 * mt + (quad & 1) * 8;
        ldsm_x4_t(s_v + swz(ri, cv), a[0], a[1], a[2], a[3]);
        float u0[4] = {}, u1[4] = {};
        mma16816(u0, a, aT[0], aT[2]);  // tokens 0..7
        mma16816(u1, a, aT[1], aT[3]);  // tokens 8..15
        const int vr = 16 * mt + gid, tk = 2 * tig;
        unsigned int *ut = reinterpret_cast<unsigned int *>(rec + kRecUt);
        st_rec<KEEP>(ut + (vr * 16 + tk) / 2, pack_bf16(u0[0], u0[1]));
        st_rec<KEEP>(ut + ((vr + 8) * 16 + tk) / 2, pack_bf16(u0[2], u0[3]));
        st_rec<KEEP>(ut + (vr * 16 + tk + 8) / 2, pack_bf16(u1[0], u1[1]));
        st_rec<KEEP>(ut + ((vr + 8) * 16 + tk + 8) / 2, pack_bf16(u1[2], u1[3]));
    }
    __syncwarp();

    // ---- copy the staged -W tile out (same swizzled layout), 16 B per lane
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int idx = (it * 32 + lane) * 16;
        st_rec<KEEP>(reinterpret_cast<uint4 *>(rec + kRecW + idx), *reinterpret_cast<const uint4 *>(sm.kn + idx));
    }
    __syncwarp();
}
// One (chunk, head) item in the factored form, by one warp: sm is the warp's
// shared memory, rec its record, tout where (I + A)^{-1} goes (or null),
// rows [t0, t0 + L) of head h its tokens.
// A chunk outside both factored ranges (see below) gets wrong numbers in its
// record until intra_exact_item rewrites it: its item index (list_item) goes
// on p.exact_list.
template <bool PRE, bool KEEP, bool GRAD = false>
__device__ __forceinline__ void intra_item(const IntraParams &p, IntraWarpSmem &sm, int64_t t0,
                                           int L, int h, uint8_t *rec, float *tout,
                                           int32_t list_item) {
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3, quad = lane >> 3;
    const int H = p.geo.n_heads;
    load_chunk(p, sm, t0, L, h, lane);
    const float beta_l = (lane < L) ? __ldg(p.beta + (t0 + lane) * H + h) : 0.f;

    // ---- chunk-local cumulative log decay; lane owns channels 4*lane..+3
    float4 graw[16];
    {
        const float *gp = p.g + (t0 * H + h) * kDim + 4 * lane;
        const int64_t rowe = static_cast<int64_t>(H) * kDim;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            graw[r] = (r < L) ? __ldcs(reinterpret_cast<const float4 *>(gp + r * rowe))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float G[16][4];   // cumulative log decay in base 2 (g log2 e summed), then about G_ref
    float run[4] = {0.f, 0.f, 0.f, 0.f};
    float gmax = 0.f;   // largest |G| (base 2)
    const bool gate_logits = PRE && (p.pre & kPreGateLogits) != 0;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        float4 gg = graw[r];
        if (gate_logits && r < L) {   // rows past the end keep g = 0
            gg.x = log_sigmoid(gg.x); gg.y = log_sigmoid(gg.y);
            gg.z = log_sigmoid(gg.z); gg.w = log_sigmoid(gg.w);
        }
        run[0] = fmaf(gg.x, kLog2e, run[0]); run[1] = fmaf(gg.y, kLog2e, run[1]);
        run[2] = fmaf(gg.z, kLog2e, run[2]); run[3] = fmaf(gg.w, kLog2e, run[3]);
        G[r][0] = run[0]; G[r][1] = run[1]; G[r][2] = run[2]; G[r][3] = run[3];
        gmax = fmaxf(gmax, fmaxf(fmaxf(fabsf(run[0]), fabsf(run[1])),
                                 fmaxf(fabsf(run[2]), fabsf(run[3]))));
    }
    // The gated products factor about a reference G_ref: exp(G_r - G_i) =
    // exp(G_r - G_ref) exp(G_ref - G_i). G_ref = 0 (the chunk start) while
    // |G| <= 80 everywhere; otherwise the middle of the chunk's range of G,
    // which keeps both factors within exp(+-80) as long as that range is at
    // most 160 and G rises by at most 80 anywhere (the record's exp(G) and
    // exp(G_last - G) stay representable). In base 2: 80 nats = 115.42,
    // 160 nats = 230.84 (with room for the rounding of the sums).
    float gref = 0.f;   // G_ref in base 2
    float eref = 1.f;   // exp(G_ref): rescales the record's gamma, scale Q e^G and W
    bool exact = false;
    const bool wide = __any_sync(0xffffffffu, !(gmax <= 115.42f));
    // (a loop of opaque trip count keeps this a branch: written as an if, it
    //  measured 4 % slower on chunks that never need it)
#pragma unroll 1
    for (int once = 0, n = opaque_trips(wide); once < n; ++once) {
        if constexpr (GRAD) {
            if (lane == 0) *p.wide_flag = 1;   // (only in the gradient call's instantiation)
        }
        // range of G from the chunk start (0) on, and its largest rise
        float hi = 0.f, low = 0.f, rise = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float m = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                rise = fmaxf(rise, G[r][e] - m);
                m = fminf(m, G[r][e]);
                hi = fmaxf(hi, G[r][e]);
            }
            low = fminf(low, m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
            low = fminf(low, __shfl_xor_sync(0xffffffffu, low, o));
        }
        exact = !(hi - low <= 230.84f) || __any_sync(0xffffffffu, !(rise <= 115.42f));
        if (exact && lane == 0) p.exact_list[atomicAdd(p.exact_ctr, 1)] = list_item;
        if (!exact) {
            gref = 0.5f * (hi + low);
            eref = ex2(gref);
#pragma unroll
            for (int r = 0; r < 16; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e) G[r][e] -= gref;
        }
    }
    float eL[4];       // exp(G_last - G_ref): K e^(G_last - G) = (K e^(G_ref - G)) eL; gamma = eL eref
#pragma unroll
    for (int e = 0; e < 4; ++e) eL[e] = ex2(G[15][e]);
    cp_async_wait_all();
    __syncwarp();

    // ---- gated operand tiles (in place for K e^G and scale Q e^G)
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const int off = swz(r, 4 * lane);
        const uint2 qq = *reinterpret_cast<const uint2 *>(sm.qg + off);
        const uint2 kk = *reinterpret_cast<const uint2 *>(sm.kg + off);
        float2 q01 = unpack_bf16(qq.x), q23 = unpack_bf16(qq.y);
        float2 k01 = unpack_bf16(kk.x), k23 = unpack_bf16(kk.y);
        if (PRE && (p.pre & kPreNormQK)) {
            // L2 norms of this row's q and k over the 128 channels of the warp
            float sq = q01.x * q01.x + q01.y * q01.y + q23.x * q23.x + q23.y * q23.y;
            float sk = k01.x * k01.x + k01.y * k01.y + k23.x * k23.x + k23.y * k23.y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            const float rq = rsqrtf(sq + kNormEps), rk = rsqrtf(sk + kNormEps);
            q01.x *= rq; q01.y *= rq; q23.x *= rq; q23.y *= rq;
            k01.x *= rk; k01.y *= rk; k23.x *= rk; k23.y *= rk;
        }
        float2 eg[2], en[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            eg[e] = make_float2(ex2(G[r][2 * e]), ex2(G[r][2 * e + 1]));
            en[e] = make_float2(ex2(-G[r][2 * e]), ex2(-G[r][2 * e + 1]));
        }
        const float2 eL01 = make_float2(eL[0], eL[1]), eL23 = make_float2(eL[2], eL[3]);
        const float2 sc2 = make_float2(p.scale, p.scale);
        const float2 kg01 = mul2v(k01, eg[0]), kg23 = mul2v(k23, eg[1]);
        const float2 qg01 = mul2v(q01, mul2v(eg[0], sc2)), qg23 = mul2v(q23, mul2v(eg[1], sc2));
        const float2 kn01 = mul2v(k01, en[0]), kn23 = mul2v(k23, en[1]);
        const float2 kd01 = mul2v(kn01, eL01), kd23 = mul2v(kn23, eL23);
        const float kg[4] = {kg01.x, kg01.y, kg23.x, kg23.y};
        const float kn[4] = {kn01.x, kn01.y, kn23.x, kn23.y};
        const float qg[4] = {qg01.x, qg01.y, qg23.x, qg23.y};
        const float kd[4] = {kd01.x, kd01.y, kd23.x, kd23.y};
        const uint2 ukg = make_uint2(pack_bf16(kg[0], kg[1]), pack_bf16(kg[2], kg[3]));
        const uint2 ukn = make_uint2(pack_bf16(kn[0], kn[1]), pack_bf16(kn[2], kn[3]));
        const uint2 uqg = make_uint2(pack_bf16(qg[0], qg[1]), pack_bf16(qg[2], qg[3]));
        const uint2 ukd = make_uint2(pack_bf16(kd[0], kd[1]), pack_bf16(kd[2], kd[3]));
        *reinterpret_cast<uint2 *>(sm.kg + off) = ukg;
        *reinterpret_cast<uint2 *>(sm.kn + off) = ukn;
        *reinterpret_cast<uint2 *>(sm.qg + off) = uqg;
        st_rec<KEEP>(reinterpret_cast<uint2 *>(rec + kRecQg + off), uqg);
        st_rec<KEEP>(reinterpret_cast<uint2 *>(rec + kRecKd + off), ukd);
    }
    st_rec<KEEP>(reinterpret_cast<float4 *>(rec + kRecGamma + 16 * lane),
           make_float4(eL[0] * eref, eL[1] * eref, eL[2] * eref, eL[3] * eref));
    if (!exact && eref != 1.f) {
        // the record's scale Q e^G = (scale Q e^(G - G_ref)) exp(G_ref), from the tile
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int off = swz(r, 4 * lane);
            const uint2 qq = *reinterpret_cast<const uint2 *>(sm.qg + off);
            const float2 a = unpack_bf16(qq.x), b = unpack_bf16(qq.y);
            st_rec<KEEP>(reinterpret_cast<uint2 *>(rec + kRecQg + off),
                         make_uint2(pack_bf16(a.x * eref, a.y * eref), pack_bf16(b.x * eref, b.y * eref)));
        }
    }
    __syncwarp();

    // ---- A_raw = (K e^G)(K e^-G)^T and P_raw = scale (Q e^G)(K e^-G)^T, 16x16 each
    const uint32_t s_kg = smem_u32(sm.kg), s_kn = smem_u32(sm.kn), s_qg = smem_u32(sm.qg);
    float accA[2][4] = {}, accP[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t aK[4], aQ[4], b[4];
        const int ra = (quad & 1) * 8 + (lane & 7), ca = (2 * kk + (quad >> 1)) * 8;
        ldsm_x4(s_kg + swz(ra, ca), aK[0], aK[1], aK[2], aK[3]);
        ldsm_x4(s_qg + swz(ra, ca), aQ[0], aQ[1], aQ[2], aQ[3]);
        const int rb = (quad >> 1) * 8 + (lane & 7), cb = (2 * kk + (quad & 1)) * 8;
        ldsm_x4(s_kn + swz(rb, cb), b[0], b[1], b[2], b[3]);
        mma16816(accA[0], aK, b[0], b[1]);
        mma16816(accA[1], aK, b[2], b[3]);
        mma16816(accP[0], aQ, b[0], b[1]);
        mma16816(accP[1], aQ, b[2], b[3]);
    }

    // ---- masks, beta rows; P goes to the record, A to shared memory
    const float beta_r0 = __shfl_sync(0xffffffffu, beta_l, gid);
    const float beta_r1 = __shfl_sync(0xffffffffu, beta_l, gid + 8);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int r = gid + 8 * hf;
            const int i = 8 * nt + 2 * tig;
            const float br = hf ? beta_r1 : beta_r0;
            const float a0 = (i < r) ? br * accA[nt][2 * hf] : 0.f;
            const float a1 = (i + 1 < r) ? br * accA[nt][2 * hf + 1] : 0.f;
            sm.a[r * 17 + i] = a0;
            sm.a[r * 17 + i + 1] = a1;
            const float p0 = (i <= r) ? accP[nt][2 * hf] : 0.f;
            const float p1 = (i + 1 <= r) ? accP[nt][2 * hf + 1] : 0.f;
            st_rec<KEEP>(reinterpret_cast<unsigned int *>(rec + kRecP + (r * 16 + i) * 2),
                   pack_bf16(p0, p1));
        }
    }
    __syncwarp();
    intra_tail<KEEP, GRAD>(sm, rec, tout, beta_l, lane, eref);
}

// The same item in the exact per-pair form (the whole record rewritten).
template <bool PRE, bool KEEP>
__device__ __forceinline__ void intra_exact_item(const IntraParams &p, IntraWarpSmem &sm, int64_t t0,
                                                 int L, int h, uint8_t *rec, float *tout) {
    const int lane = threadIdx.x & 31;
    const int H = p.geo.n_heads;
    load_chunk(p, sm, t0, L, h, lane);
    const float beta_l = (lane < L) ? __ldg(p.beta + (t0 + lane) * H + h) : 0.f;
    cp_async_wait_all();
    __syncwarp();
    intra_exact_chunk<KEEP>(p.g + (t0 * H + h) * kDim + 4 * lane, static_cast<int64_t>(H) * kDim, L,
                            PRE ? p.pre : 0, p.scale, beta_l, &sm, rec, p.err);
    __syncwarp();
    intra_tail<KEEP>(sm, rec, tout, beta_l, lane);
}

}  // namespace

}  // namespace kda
