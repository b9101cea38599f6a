// One-token step of the KDA recurrence for a batch of sequences (decode).
//
// The pages describe KDA as keeping a fixed-size state that is updated for
// every new token ("Kimi K3 的三個系統設計", section 第一個設計). For one
// (sequence, head), with alpha = exp(g) per key channel and S the state
// (K x V, rows = key channels):
//
//   S' = Diag(alpha) S
//   u  = k^T S'                                (1 x V)
//   S <- S' + beta k (v - u)^T                 = (I - beta k k^T) Diag(alpha) S + beta k v^T
//   o  = scale S^T q = scale ( (q * alpha)^T S_old + (q . k) beta (v - u) )
//
// so a step needs two column reductions of the old state (weights k*alpha and
// q*alpha) and one rank-1 update. One CTA per (sequence, head) holds the
// 128 x 128 fp32 state in registers (256 threads x 64 values): thread t owns
// columns 4 (t % 32) .. +3 of rows t / 32 + 8 m, m = 0..15, so every warp
// load and store is one contiguous 512-byte row. The state is read once and
// written once: the kernel is bound by HBM bandwidth (131,072 + 1,540 B per
// (sequence, head)). Exponentials are taken per channel exactly, so any
// finite log decay is fine. With the preprocessing flags, q and k are
// divided by their L2 norms (a block reduction) and g is read as gate logits.

#include "kda_device.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

constexpr int kDecThreads = 256;

__global__ void __launch_bounds__(kDecThreads, 2)
kda_decode_kernel(DecodeParams p) {
    __shared__ float s_k[kDim], s_ka[kDim], s_qa[kDim], s_a[kDim], s_v[kDim], s_d[kDim];
    __shared__ float s_red[2][8][kDim];
    __shared__ float s_dot[3][4];   // per-warp partial q.q, k.k, q.k
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t unit = blockIdx.x;   // sequence * H + head
    const int64_t row = unit * kDim;

    // the old state, all loads in flight before anything waits on them
    float4 s[16];
    if (p.s_in != nullptr) {
        const float4 *S0 = reinterpret_cast<const float4 *>(p.s_in + unit * kDim * kDim);
#pragma unroll
        for (int m = 0; m < 16; ++m) s[m] = __ldcs(S0 + (warp + 8 * m) * (kDim / 4) + lane);
    } else {
#pragma unroll
        for (int m = 0; m < 16; ++m) s[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // this token's vectors (threads 0..127 own channel t)
    float qv = 0.f, kv = 0.f, a = 0.f;
    if (t < kDim) {
        const __nv_bfloat16 *qp = static_cast<const __nv_bfloat16 *>(p.q);
        const __nv_bfloat16 *kp = static_cast<const __nv_bfloat16 *>(p.k);
        const __nv_bfloat16 *vp = static_cast<const __nv_bfloat16 *>(p.v);
        qv = __bfloat162float(qp[row + t]);
        kv = __bfloat162float(kp[row + t]);
        const float gl = p.g[row + t];
        a = __expf((p.pre & kPreGateLogits) ? log_sigmoid(gl) : gl);
        s_v[t] = __bfloat162float(vp[row + t]);
        float d3[3] = {qv * qv, kv * kv, qv * kv};
#pragma unroll
        for (int c = 0; c < 3; ++c) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d3[c] += __shfl_xor_sync(0xffffffffu, d3[c], o);
            if (lane == 0) s_dot[c][warp] = d3[c];
        }
    }
    __syncthreads();
    // q.k, with q and k divided by their L2 norms when asked to
    float rq = 1.f, rk = 1.f;
    if (p.pre & kPreNormQK) {
        rq = rsqrtf(s_dot[0][0] + s_dot[0][1] + s_dot[0][2] + s_dot[0][3] + kNormEps);
        rk = rsqrtf(s_dot[1][0] + s_dot[1][1] + s_dot[1][2] + s_dot[1][3] + kNormEps);
    }
    const float qk_all = (s_dot[2][0] + s_dot[2][1] + s_dot[2][2] + s_dot[2][3]) * rq * rk;
    if (t < kDim) {
        qv *= rq;
        kv *= rk;
        s_k[t] = kv;
        s_ka[t] = kv * a;
        s_qa[t] = qv * a;
        s_a[t] = a;
    }
    __syncthreads();

    // partial column reductions over this thread's 16 rows
    float4 pu = make_float4(0.f, 0.f, 0.f, 0.f), pw = pu;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int i = warp + 8 * m;
        const float ka = s_ka[i], qa = s_qa[i];
        pu.x = fmaf(ka, s[m].x, pu.x); pu.y = fmaf(ka, s[m].y, pu.y);
        pu.z = fmaf(ka, s[m].z, pu.z); pu.w = fmaf(ka, s[m].w, pu.w);
        pw.x = fmaf(qa, s[m].x, pw.x); pw.y = fmaf(qa, s[m].y, pw.y);
        pw.z = fmaf(qa, s[m].z, pw.z); pw.w = fmaf(qa, s[m].w, pw.w);
    }
    reinterpret_cast<float4 *>(s_red[0][warp])[lane] = pu;
    reinterpret_cast<float4 *>(s_red[1][warp])[lane] = pw;
    __syncthreads();

    // column totals; threads 0..127 own column j = t
    if (t < kDim) {
        float u = 0.f, w = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            u += s_red[0][r][t];
            w += s_red[1][r][t];
        }
        const float beta = p.beta[unit];
        const float d = beta * (s_v[t] - u);
        s_d[t] = d;
        static_cast<__nv_bfloat16 *>(p.out)[row + t] =
            __float2bfloat16_rn(p.scale * (w + qk_all * d));
    }
    __syncthreads();

    // S <- Diag(alpha) S + k d^T
    const float4 d4 = reinterpret_cast<const float4 *>(s_d)[lane];
    float4 *S1 = reinterpret_cast<float4 *>(p.s_out + unit * kDim * kDim);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int i = warp + 8 * m;
        const float ai = s_a[i], ki = s_k[i];
        float4 r;
        r.x = fmaf(ai, s[m].x, ki * d4.x);
        r.y = fmaf(ai, s[m].y, ki * d4.y);
        r.z = fmaf(ai, s[m].z, ki * d4.z);
        r.w = fmaf(ai, s[m].w, ki * d4.w);
        S1[(warp + 8 * m) * (kDim / 4) + lane] = r;
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, int64_t units, cudaStream_t stream) {
    if (units <= 0) return cudaSuccess;
    kda_decode_kernel<<<static_cast<unsigned>(units), kDecThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
