// Gradients of KDA prefill (training), one CTA per (sequence, head).
//
// The pages say that K3 trains with KDA ("Kimi K3 開源基礎設施"); the
// forward map is the token recurrence of the prefill ("Kimi K3 的三個系統設計",
// section 第一個設計): with a_t = exp(g_t) per key channel,
//
//   S' = Diag(a_t) S_{t-1},  w = v_t - S'^T k_t,  S_t = S' + beta_t k_t w^T,
//   o_t = scale S_t^T q_t.
//
// Walking a sequence backwards with dS = dL/dS_t (seeded with dL/d(final
// state), or 0):
//
//   dS   += scale q_t dO_t^T;   dq_t = scale S_t dO_t
//   x     = dS^T k_t;           dv_t = beta_t x;     dbeta_t = w . x
//   dk_t  = beta_t (dS w - S' x)
//   dS'   = dS - beta_t k_t x^T;  dg_t = a_t * rowsum(dS' o S_{t-1})
//   dS    = Diag(a_t) dS'       (then dL/dS_{t-1})
//
// and dL/d(initial state) is the last dS.
//
// The states S_{t-1} come from a forward pass that keeps one checkpoint
// every 16 tokens (64 KiB each, in the workspace); each 16-token segment,
// last first, is recomputed from its checkpoint into a per-CTA ring of 16
// states and then walked backwards. The state, its gradient and the ring
// live in the layout of the decode kernel: 256 threads, thread t holding
// columns 4 (t % 32) .. +3 of rows t / 32 + 8 m, m = 0..15, so every warp
// access is one contiguous 512-byte row; column sums (S'^T k, dS^T k) go
// through shared memory and row sums (four per row) through warp
// reduce-scatters (31 shuffles per 32 sums).
// All arithmetic is fp32; q, k, v and dO are read as bf16.
//
// This is the first, token-serial form: its time is the serial chain of
// 3 T token steps per (sequence, head), not memory traffic.

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kBwdThreads = 256;
constexpr int kRing = 16;            // tokens per segment
constexpr int64_t kStateF4 = 4096;   // float4 in one 128 x 128 fp32 state

struct BwdSmem {
    float k[kDim], v[kDim], a[kDim], q[kDim], dout[kDim], w[kDim], x[kDim];
    float red[8][kDim];              // per-warp column partial sums
    float rowq[4][kDim];             // per-row sums: S_t dO, dS w, S' x, dS' o S_{t-1}
    float dbeta_part[4];
    float beta;
};

__device__ __forceinline__ float4 f4_zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Token t's k, v and a = exp(g) (and beta) into shared memory.
__device__ __forceinline__ void load_kva(const BackParams &p, BwdSmem &sm, int64_t row,
                                         int64_t bidx) {
    const int t = threadIdx.x;
    if (t < kDim) {
        sm.k[t] = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.k)[row + t]);
        sm.v[t] = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.v)[row + t]);
        sm.a[t] = __expf(p.g[row + t]);
    }
    if (t == 0) sm.beta = p.beta[bidx];
}

// w = v - (Diag(a) S)^T k into sm.w (S = the state before the token).
__device__ __forceinline__ void compute_w(BwdSmem &sm, const float4 (&S)[16], int warp, int lane) {
    float4 pu = f4_zero();
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int i = warp + 8 * m;
        const float ka = sm.k[i] * sm.a[i];
        pu.x = fmaf(ka, S[m].x, pu.x); pu.y = fmaf(ka, S[m].y, pu.y);
        pu.z = fmaf(ka, S[m].z, pu.z); pu.w = fmaf(ka, S[m].w, pu.w);
    }
    reinterpret_cast<float4 *>(sm.red[warp])[lane] = pu;
    __syncthreads();
    const int t = threadIdx.x;
    if (t < kDim) {
        float u = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) u += sm.red[r][t];
        sm.w[t] = sm.v[t] - u;
    }
    __syncthreads();
}

// One forward token step of the state held in S (row layout above).
__device__ __forceinline__ void forward_step(const BackParams &p, BwdSmem &sm, float4 (&S)[16],
                                             int64_t row, int64_t bidx, int warp, int lane) {
    __syncthreads();   // the previous step's readers of shared memory are done
    load_kva(p, sm, row, bidx);
    __syncthreads();
    compute_w(sm, S, warp, lane);
    const float b = sm.beta;
    const float4 w4 = reinterpret_cast<const float4 *>(sm.w)[lane];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int i = warp + 8 * m;
        const float a = sm.a[i], kb = b * sm.k[i];
        S[m].x = fmaf(a, S[m].x, kb * w4.x); S[m].y = fmaf(a, S[m].y, kb * w4.y);
        S[m].z = fmaf(a, S[m].z, kb * w4.z); S[m].w = fmaf(a, S[m].w, kb * w4.w);
    }
}

__global__ void __launch_bounds__(kBwdThreads, 1)
kda_backward_kernel(BackParams p, int64_t units) {
    __shared__ BwdSmem sm;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    if (geo.cu != nullptr && (*geo.call_flags & kErrBadCu)) return;
    // persistent: this CTA takes units blockIdx.x, + gridDim.x, ... and owns
    // ring blockIdx.x for all of them
    float4 *ring = reinterpret_cast<float4 *>(p.ring) +
                   static_cast<int64_t>(blockIdx.x) * kRing * kStateF4;
    for (int64_t unit = blockIdx.x; unit < units; unit += gridDim.x) {
    const int n = static_cast<int>(unit / H), h = static_cast<int>(unit % H);
    int64_t t0, L, coff;
    if (geo.cu == nullptr) {
        t0 = static_cast<int64_t>(n) * geo.seq_len;
        L = geo.seq_len;
        coff = static_cast<int64_t>(n) * geo.chunks_per_seq;
    } else {
        t0 = geo.cu[n];
        L = geo.cu[n + 1] - t0;
        coff = geo.chunk_off[n];
    }
    const int64_t nck = (L + kRing - 1) / kRing;
    // checkpoint c of this unit: state index (coff + c) * H + h
    float4 *ckpt = reinterpret_cast<float4 *>(p.ckpt) + (coff * H + h) * kStateF4;
    const int64_t ck_stride = static_cast<int64_t>(H) * kStateF4;
    const int64_t me = static_cast<int64_t>(warp) * 32 + lane;   // + 256 m: this thread's float4

    // ---- forward pass, a checkpoint before every 16th token
    float4 S[16];
    if (p.s0 != nullptr) {
        const float4 *S0 = reinterpret_cast<const float4 *>(p.s0) + unit * kStateF4;
#pragma unroll
        for (int m = 0; m < 16; ++m) S[m] = S0[me + 256 * m];
    } else {
#pragma unroll
        for (int m = 0; m < 16; ++m) S[m] = f4_zero();
    }
    for (int64_t j = 0; j < L; ++j) {
        if (j % kRing == 0) {
            float4 *c = ckpt + (j / kRing) * ck_stride;
#pragma unroll
            for (int m = 0; m < 16; ++m) c[me + 256 * m] = S[m];
        }
        const int64_t tok = t0 + j;
        forward_step(p, sm, S, (tok * H + h) * kDim, tok * H + h, warp, lane);
    }

    // ---- reverse pass
    float4 dS[16];
    if (p.dsf != nullptr) {
        const float4 *D = reinterpret_cast<const float4 *>(p.dsf) + unit * kStateF4;
#pragma unroll
        for (int m = 0; m < 16; ++m) dS[m] = D[me + 256 * m];
    } else {
#pragma unroll
        for (int m = 0; m < 16; ++m) dS[m] = f4_zero();
    }
    const float scale = p.scale;
    for (int64_t c = nck - 1; c >= 0; --c) {
        const int64_t j0 = c * kRing, j1 = (j0 + kRing < L) ? j0 + kRing : L;
        // states before tokens j0 .. j1-1 into the ring
        const float4 *cp = ckpt + c * ck_stride;
#pragma unroll
        for (int m = 0; m < 16; ++m) S[m] = cp[me + 256 * m];
        for (int64_t j = j0; j < j1; ++j) {
            float4 *r = ring + (j - j0) * kStateF4;
#pragma unroll
            for (int m = 0; m < 16; ++m) r[me + 256 * m] = S[m];
            if (j + 1 < j1) {
                const int64_t tok = t0 + j;
                forward_step(p, sm, S, (tok * H + h) * kDim, tok * H + h, warp, lane);
            }
        }
        for (int64_t j = j1 - 1; j >= j0; --j) {
            const int64_t tok = t0 + j, row = (tok * H + h) * kDim, bidx = tok * H + h;
            // S := S_{t-1}
            const float4 *r = ring + (j - j0) * kStateF4;
#pragma unroll
            for (int m = 0; m < 16; ++m) S[m] = r[me + 256 * m];
            __syncthreads();
            load_kva(p, sm, row, bidx);
            if (t < kDim) {
                sm.q[t] = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.q)[row + t]);
                sm.dout[t] = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.dout)[row + t]);
            }
            __syncthreads();
            compute_w(sm, S, warp, lane);
            const float b = sm.beta;
            // dS += scale q dO^T; then x = dS^T k
            const float4 do4 = reinterpret_cast<const float4 *>(sm.dout)[lane];
            float4 px = f4_zero();
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int i = warp + 8 * m;
                const float sq = scale * sm.q[i], ki = sm.k[i];
                dS[m].x = fmaf(sq, do4.x, dS[m].x); dS[m].y = fmaf(sq, do4.y, dS[m].y);
                dS[m].z = fmaf(sq, do4.z, dS[m].z); dS[m].w = fmaf(sq, do4.w, dS[m].w);
                px.x = fmaf(ki, dS[m].x, px.x); px.y = fmaf(ki, dS[m].y, px.y);
                px.z = fmaf(ki, dS[m].z, px.z); px.w = fmaf(ki, dS[m].w, px.w);
            }
            reinterpret_cast<float4 *>(sm.red[warp])[lane] = px;
            __syncthreads();
            if (t < kDim) {
                float xs = 0.f;
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) xs += sm.red[rr][t];
                sm.x[t] = xs;
                p.dv[row + t] = b * xs;
                const float db = warp_sum(sm.w[t] * xs);
                if (lane == 0) sm.dbeta_part[warp] = db;
            }
            __syncthreads();
            // row sums: S_t dO, dS w, S' x (before the erase), dS' o S_{t-1}.
            // Per half of this thread's rows, the 32 partials (4 sums x 8 rows)
            // reduce over the warp in one butterfly reduce-scatter of 31
            // shuffles; lane l then holds sum l / 8 of row 8 hf + l % 8.
            const float4 w4 = reinterpret_cast<const float4 *>(sm.w)[lane];
            const float4 x4 = reinterpret_cast<const float4 *>(sm.x)[lane];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float v[32];
#pragma unroll
                for (int mm = 0; mm < 8; ++mm) {
                    const int m = 8 * hf + mm, i = warp + 8 * m;
                    const float a = sm.a[i], kb = b * sm.k[i];
                    float4 st;
                    st.x = fmaf(a, S[m].x, kb * w4.x); st.y = fmaf(a, S[m].y, kb * w4.y);
                    st.z = fmaf(a, S[m].z, kb * w4.z); st.w = fmaf(a, S[m].w, kb * w4.w);
                    v[mm] = dot4(st, do4);
                    v[8 + mm] = dot4(dS[m], w4);
                    v[16 + mm] = a * dot4(S[m], x4);
                    dS[m].x = fmaf(-kb, x4.x, dS[m].x); dS[m].y = fmaf(-kb, x4.y, dS[m].y);
                    dS[m].z = fmaf(-kb, x4.z, dS[m].z); dS[m].w = fmaf(-kb, x4.w, dS[m].w);
                    v[24 + mm] = dot4(dS[m], S[m]);
                    dS[m].x *= a; dS[m].y *= a; dS[m].z *= a; dS[m].w *= a;
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int jj = 0; jj < o; ++jj) {
                        const float send = up ? v[jj] : v[jj + o];
                        const float keep = up ? v[jj + o] : v[jj];
                        v[jj] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
                const int qi = lane >> 3, i = warp + 8 * (8 * hf + (lane & 7));
                sm.rowq[qi][i] = (qi == 0) ? scale * v[0] : v[0];
            }
            __syncthreads();
            if (t < kDim) {
                p.dq[row + t] = sm.rowq[0][t];
                p.dk[row + t] = b * (sm.rowq[1][t] - sm.rowq[2][t]);
                p.dg[row + t] = sm.a[t] * sm.rowq[3][t];
            }
            if (t == 0)
                p.dbeta[bidx] = sm.dbeta_part[0] + sm.dbeta_part[1] + sm.dbeta_part[2] +
                                sm.dbeta_part[3];
        }
    }
    if (p.ds0 != nullptr) {
        float4 *D = reinterpret_cast<float4 *>(p.ds0) + unit * kStateF4;
#pragma unroll
        for (int m = 0; m < 16; ++m) D[me + 256 * m] = dS[m];
    }
    }  // units
}

}  // namespace

static int64_t backward_grid(int64_t units) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_backward_kernel, kBwdThreads,
                                                      0) != cudaSuccess)
        return 0;
    int64_t grid = static_cast<int64_t>(sms) * (per_sm > 0 ? per_sm : 1);
    if (grid > kBackwardMaxRings) grid = kBackwardMaxRings;
    return units < grid ? units : grid;
}

cudaError_t launch_backward(const BackParams &p, int64_t units, cudaStream_t stream) {
    if (units <= 0) return cudaSuccess;
    const int64_t grid = backward_grid(units);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    kda_backward_kernel<<<static_cast<unsigned>(grid), kBwdThreads, 0, stream>>>(p, units);
    return cudaGetLastError();
}

}  // namespace kda
