// Chunked KDA prefill with 64-token chunks on the 5th-generation tensor core.
//
// The two kernels of different parallelism that the pages describe ("Kimi K3
// 的三個系統設計", section "為什麼 FlashKDA 選擇 16-token chunks": a
// token-parallel intra-chunk kernel and a recurrent inter-chunk kernel), with
// the chunk widened from 16 to 64 tokens so that every product of the
// recurrent step is a tcgen05 MMA with M = 128:
//
//   intra-chunk, per (64-token chunk, head), G_r = sum_{u<=r} g_u per channel:
//     A  = strict_lower( (beta K e^G) (K e^-G)^T )      Gram, one tcgen05 MMA group
//     P  = scale lower( (Q e^G) (K e^-G)^T )             (same MMA, rows 64..127)
//     T  = (I + A)^-1                                    blocked forward substitution:
//          16 x 16 diagonal blocks in fp32, off-diagonal blocks by tf32 warp MMAs
//     W  = T (beta K e^G),  Ut = T (beta V)              tcgen05 MMAs
//   recurrent, per (sequence, head), state S^T (V x K, fp32) in tensor memory:
//     U^T = Ut^T - S^T W^T,  o^T = S^T (scale Qg)^T + U^T (scale P)^T
//     S^T <- S^T Diag(gamma) + U^T Kd
//
// The inputs are staged by TMA tensor-map loads (cp.async.bulk.tensor), the
// records by bulk copies. Chunks whose cumulative log decay leaves [-80, 80]
// in some channel (strong decay) get A and P from exact per-pair
// exponentials instead of the factored form; everything else is shared.
//
// Launch forms: the intra-chunk kernel over all chunk-heads followed by the
// recurrent kernel (records in the workspace), or one cooperative kernel in
// which some CTAs run the recurrent chains while the others build the records
// into a small ring that stays in L2 (ring_depth slots per head, ready and
// consumed counters in global memory, every wait bounded).

#include <cuda.h>

#include "kda_c64.cuh"
#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_tcgen05.cuh"

namespace kda {
namespace c64 {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
// |G| bound of the factored exponentials (natural-log units)
constexpr float kFactorRange = 80.f;

// ------------------------------------------------------------------ shared memory
// recurrent role
constexpr int kCStages = 3;
constexpr int kCOffMisc = kCStages * kRecBytes;   // tmem base, abort flag
constexpr int kCOffBar = kCOffMisc + 64;
enum {
    kCBFull = 0, kCBEmpty = 3, kCBSop = 6, kCBUdone = 8, kCBUop = 9, kCBSdone = 10,
    kCBOdone = 11, kCBOfree = 12, kCBTear = 13, kCBDrain = 14, kCNumBars = 15
};
constexpr int kCSmem = kCOffBar + kCNumBars * 8;
// intra-chunk role (a three-stage pipeline over items, see intra_role)
constexpr int kIOffG = 0;                         // G (base-2 cumulative log decay), fp32,
                                                  //   4 swizzled panels of 64 rows x 32 channels
constexpr int kIOffBeta = 32768;                  // fp32 [64]
constexpr int kIOffGA = 33792;                    // [beta K e^G ; scale Q e^G] 128 x 128 keys
                                                  //   (exact form: A and P staging, fp32 [128][64])
constexpr int kIOffGB = kIOffGA + 32768;          // K e^-G: 64 x 128 keys (norm partials first)
constexpr int kIOffWB = kIOffGB + 16384;          // (beta K e^G)^T x2: 128 keys x 64 tokens
constexpr int kIOffUA = kIOffWB + 2 * 16384;      // (beta V)^T x2: 128 v x 64 tokens
constexpr int kIOffTA = kIOffUA + 2 * 16384;      // T: 64 x 64 tokens, bf16
constexpr int kIOffAT = kIOffTA + 8192;           // A^T (strict upper) and T (lower), fp32 [64][68]
constexpr int kATStride = 68;
constexpr int kIOffScr = kIOffAT + 64 * kATStride * 4;   // inversion scratch, 4 x 16 x 17 fp32
constexpr int kIOffTot = kIOffScr + 4352;         // half sums [2][128] fp32
constexpr int kIOffRed = kIOffTot + 1024;         // [8] per-warp range flags
constexpr int kIOffMisc = kIOffRed + 64;          // tmem base, abort flag
constexpr int kIOffQKV = 180224;                  // q, k, v tiles (TMA, 128-byte swizzled),
                                                  //   16 KiB each: panels of 64 rows x 64 channels
constexpr int kIOffBar = kIOffQKV + 3 * 16384;
enum {
    kIBGram = 0, kIBCdone = 2, kIBWU = 4, kIBFdone = 6, kIBTear = 8, kIBDrain = 9, kIBIn = 10,
    kINumBars = 11
};
static_assert(kIOffMisc + 64 <= kIOffQKV, "intra shared memory layout");
constexpr int kISmem = kIOffBar + kINumBars * 8;
constexpr int kIThreads = 512;                    // 16 warps
constexpr int kSmem = kCSmem > kISmem ? kCSmem : kISmem;
static_assert(kSmem <= 227 * 1024, "shared memory");

// tensor memory columns
constexpr uint32_t kCTmemCols = 512;   // S^T [0,128), O^T [128,192), U^T [192,256),
                                       // bf16 S^T x2 [256,384), bf16 U^T [384,416)
constexpr uint32_t kITmemCols = 512;   // Gram x2 [0,128); per buffer b: W [128+192b, +128),
                                       // Ut^T [256+192b, +64)

constexpr uint32_t kIdFull = tc::idesc(128, 64, 1);    // M=128, N=64
constexpr uint32_t kIdW = tc::idesc(64, 128, 1);       // M=64, N=128

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads:
// every thread gets the same answer (used to leave a loop together).
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %3, 0;\n"
        " bar.red.or.pred q, %1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(id), "r"(n), "r"(pred ? 1u : 0u)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void st_global_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// D += A * B, m16n8k8, tf32 operands, fp32 accumulate
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 32 lanes x 32 bits, 32 or 64 consecutive columns (thread i <-> lane i)
__device__ __forceinline__ void tld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tst32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Bounded mbarrier wait that also gives up once another warp raised the abort flag.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int *err) {
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

__device__ __forceinline__ long long ld_acquire(const long long *p) {
    long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(long long *p, long long v) {
    asm volatile("st.release.gpu.global.b64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}

// Bounded wait for a global counter written by another CTA of the same
// (cooperative) launch to reach `target`.
__device__ __forceinline__ bool wait_counter(const long long *p, long long target,
                                             volatile int *abort_flag, int *err) {
    if (ld_acquire(p) >= target) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 16; ++i) {
            __nanosleep(64);
            if (ld_acquire(p) >= target) return true;
        }
        if (*abort_flag) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(err, kErrTimeout);
            *abort_flag = 1;
            return false;
        }
    }
}

}  // namespace

// ------------------------------------------------------------------ parameters
struct Params {
    CUtensorMap tm_q, tm_k, tm_v, tm_g;   // (128 channels, H, tokens), swizzled 128-byte boxes
    const void *q, *k, *v;                // bf16 [tokens, H, 128]
    const float *g;                       // [tokens, H, 128]
    const float *beta;                    // [tokens, H]
    const float *s0;                      // [N, H, 128, 128] or nullptr
    void *out;                            // bf16 [tokens, H, 128]
    float *s_final;                       // [N, H, 128, 128] or nullptr
    uint8_t *rec;                         // records
    int *err;                             // sticky device error word
    const int32_t *cu;                    // packed: cu_seqlens [N+1]
    const int32_t *chunk_off;             // packed: first 64-token chunk of each sequence [N+1]
    const int *call_flags;                // packed: per-call flags (bad cu_seqlens)
    int64_t seq_len;                      // fixed: tokens per sequence; packed: total tokens
    int64_t max_chunks;                   // chunks of the call (upper bound when packed)
    int32_t n_seqs, n_heads, cps;         // cps: chunks per sequence (fixed)
    float scale;
    int pre;                              // kPreNormQK | kPreGateLogits
    // ring form (one cooperative launch)
    int ring_depth;                       // 0: record of (chunk c, head h) at c * H + h
    int n_chain;                          // CTAs [0, n_chain) run chains (head = blockIdx.x)
    long long *ready;                     // [ring_depth * H]: chunk index + 1 of the slot's record
    long long *consumed;                  // [H]: chunks of head h copied out by its chain
    int *exit_ctr;                        // CTAs finished (the last one clears the counters)
};

// Where chunk c is: sequence n, first token t0, length L. False past the end.
__device__ __forceinline__ bool locate(const Params &p, int64_t c, int &n, int64_t &t0, int &L) {
    if (p.cu == nullptr) {
        if (c >= static_cast<int64_t>(p.n_seqs) * p.cps) return false;
        n = static_cast<int>(c / p.cps);
        const int64_t i = c - static_cast<int64_t>(n) * p.cps;
        t0 = static_cast<int64_t>(n) * p.seq_len + kC * i;
        const int64_t rem = p.seq_len - kC * i;
        L = static_cast<int>(rem < kC ? rem : kC);
        return true;
    }
    const int32_t *off = p.chunk_off;
    if (c >= off[p.n_seqs]) return false;
    int lo = 0, hi = p.n_seqs;   // off[lo] <= c < off[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= c) lo = mid; else hi = mid;
    }
    n = lo;
    t0 = static_cast<int64_t>(p.cu[n]) + kC * (c - off[n]);
    const int64_t rem = static_cast<int64_t>(p.cu[n + 1]) - t0;
    L = static_cast<int>(rem < kC ? rem : kC);
    return true;
}

__device__ __forceinline__ uint8_t *record_of(const Params &p, int64_t c, int h) {
    const int64_t H = p.n_heads;
    const int64_t slot = p.ring_depth > 0 ? (c % p.ring_depth) : c;
    return p.rec + (slot * H + h) * static_cast<int64_t>(kRecBytes);
}

// ============================================================================
// Intra-chunk role: warps 0-7 compute, warp 8 issues the TMA loads and MMAs.
// Items (chunk c, head h) = c * H + h, taken with a stride of `nworkers`.
// ============================================================================
namespace {

// Input tiles as the TMA writes them with 128-byte swizzling: panels of 64
// token rows x 128 bytes (64 bf16 or 32 fp32 channels), the 16-byte chunk c
// of row r stored at chunk c ^ (r % 8). Byte offset of (row r, channel ch):
__device__ __forceinline__ uint32_t sw_bf16(int r, int ch) {
    return static_cast<uint32_t>((ch >> 6) * 8192 + r * 128 + ((((ch & 63) >> 3) ^ (r & 7)) << 4) +
                                 (ch & 7) * 2);
}
__device__ __forceinline__ uint32_t sw_f32(int r, int ch) {
    return static_cast<uint32_t>((ch >> 5) * 8192 + r * 128 + ((((ch & 31) >> 2) ^ (r & 7)) << 4) +
                                 (ch & 3) * 4);
}

// Fragment of an 8 x 8 bf16 tile (thread i: row i / 4, columns 2 (i % 4) and
// +1) transposed across the warp.
__device__ __forceinline__ uint32_t movt(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void ldsm_x4_addr(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void stsm_x4_addr(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                             uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}
__device__ __forceinline__ void stsm_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                              uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ void st_global_u32(void *ptr, uint32_t v) {
    asm volatile("st.global.b32 [%0], %1;\n" ::"l"(ptr), "r"(v) : "memory");
}

__device__ __forceinline__ void tma_load_3d_e(uint32_t dst, const CUtensorMap *map, int x, int y,
                                              int z, uint32_t bar) {
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n}\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_ss_e(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                         uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void commit_e(uint32_t bar) {
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
            bar)
        : "memory");
}
__device__ __forceinline__ void arrive_tx_e(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n}\n" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

// bf16 T (64 x 64, K-major core matrices) for the MMAs: element (r, i)
__device__ __forceinline__ void ta_put(uint8_t *ta, int r, int i, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(ta + kmaj(r, i, 64)) = __float2bfloat16_rn(x);
}

// The fp32 A / T buffer (64 x 64, row stride kATStride): A (strictly lower)
// is stored transposed in the strict upper triangle, A[R][C] at [C][R]; T
// (unit lower triangular) in place in the lower triangle incl. the diagonal.
// Element (r, c) of 16 x 16 block (I, J):
__device__ __forceinline__ float a_blk(const float *at, int I, int J, int r, int c) {
    return at[(16 * J + c) * kATStride + 16 * I + r];
}
__device__ __forceinline__ float t_blk(const float *at, int I, int J, int r, int c) {
    return (I > J || r >= c) ? at[(16 * I + r) * kATStride + 16 * J + c] : 0.f;
}

// Forward substitution of one 16 x 16 diagonal block (warp w, lanes 0-15
// each solve one column): T to the lower part of the block and in bf16 to TA.
__device__ __forceinline__ void invert_diag(float *at, uint8_t *ta, int w, int lane) {
    const int j = lane & 15, b = 16 * w;
    float t[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        // four independent partial sums keep the dependent chain short
        float s4[4] = {(r == j) ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < r; ++i)
            s4[i & 3] = fmaf(-at[(b + i) * kATStride + b + r], t[i], s4[i & 3]);
        t[r] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    }
    __syncwarp();
    if (lane < 16) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            if (r >= j) at[(b + r) * kATStride + b + j] = t[r];
            ta_put(ta, b + r, b + j, t[r]);
        }
    }
    __syncwarp();
}

// acc (16 x 16, two m16n8 fragments) += A(I,K) * T(K,J)
__device__ __forceinline__ void blk_mma(float (&acc)[2][4], const float *at, int I, int K, int J,
                                        int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kk = 0; kk < 16; kk += 8) {
        const uint32_t a0 = tf32(a_blk(at, I, K, g, kk + t));
        const uint32_t a1 = tf32(a_blk(at, I, K, g + 8, kk + t));
        const uint32_t a2 = tf32(a_blk(at, I, K, g, kk + t + 4));
        const uint32_t a3 = tf32(a_blk(at, I, K, g + 8, kk + t + 4));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b0 = tf32(t_blk(at, K, J, kk + t, 8 * nt + g));
            const uint32_t b1 = tf32(t_blk(at, K, J, kk + t + 4, 8 * nt + g));
            mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
        }
    }
}

// T(I,J) = -T(I,I) * X where X (16 x 16, fragments) is staged in scratch; to
// the lower part of the fp32 buffer and in bf16 to TA.
__device__ __forceinline__ void finish_blk(float *at, uint8_t *ta, float *scratch,
                                           const float (&x)[2][4], int I, int J, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        scratch[g * 17 + 8 * nt + 2 * t] = x[nt][0];
        scratch[g * 17 + 8 * nt + 2 * t + 1] = x[nt][1];
        scratch[(g + 8) * 17 + 8 * nt + 2 * t] = x[nt][2];
        scratch[(g + 8) * 17 + 8 * nt + 2 * t + 1] = x[nt][3];
    }
    __syncwarp();
    float acc[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 16; kk += 8) {
        const uint32_t a0 = tf32(t_blk(at, I, I, g, kk + t));
        const uint32_t a1 = tf32(t_blk(at, I, I, g + 8, kk + t));
        const uint32_t a2 = tf32(t_blk(at, I, I, g, kk + t + 4));
        const uint32_t a3 = tf32(t_blk(at, I, I, g + 8, kk + t + 4));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b0 = tf32(scratch[(kk + t) * 17 + 8 * nt + g]);
            const uint32_t b1 = tf32(scratch[(kk + t + 4) * 17 + 8 * nt + g]);
            mma_tf32(acc[nt], a0, a1, a2, a3, b0, b1);
        }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int c0 = 8 * nt + 2 * t;
        float *row0 = at + (16 * I + g) * kATStride + 16 * J + c0;
        float *row1 = at + (16 * I + g + 8) * kATStride + 16 * J + c0;
        row0[0] = -acc[nt][0];
        row0[1] = -acc[nt][1];
        row1[0] = -acc[nt][2];
        row1[1] = -acc[nt][3];
        *reinterpret_cast<uint32_t *>(ta + kmaj(16 * I + g, 16 * J + c0, 64)) =
            pack_bf16(-acc[nt][0], -acc[nt][1]);
        *reinterpret_cast<uint32_t *>(ta + kmaj(16 * I + g + 8, 16 * J + c0, 64)) =
            pack_bf16(-acc[nt][2], -acc[nt][3]);
    }
    __syncwarp();
}

// T = (I + A)^{-1} for the 64 x 64 strictly lower A held transposed in `at`
// (four warps; named barrier `bar_id` over their 128 threads; the caller
// synchronises them before and after). T goes to the lower part of `at`
// (fp32) and to TA (bf16; the blocks above the diagonal are zero).
__device__ __forceinline__ void invert64(float *at, uint8_t *ta, float *scratch, int w, int lane,
                                         int bar_id) {
    for (int x = 32 * w + lane; x < 6 * 32; x += 128) {
        const int blk = x >> 5, piece = x & 31;           // 32 pieces of 16 bytes per block
        const int I = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
        const int J = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        const int r = 16 * I + (piece >> 1), c8 = 16 * J + 8 * (piece & 1);
        *reinterpret_cast<uint4 *>(ta + kmaj(r, c8, 64)) = make_uint4(0, 0, 0, 0);
    }
    invert_diag(at, ta, w, lane);
    named_sync(bar_id, 128);
    // level 1: T(I, I-1) for I = 1..3 on warps 0..2
    if (w < 3) {
        const int I = w + 1;
        float x[2][4] = {};
        blk_mma(x, at, I, I - 1, I - 1, lane);
        finish_blk(at, ta, scratch + w * 16 * 17, x, I, I - 1, lane);
    }
    named_sync(bar_id, 128);
    // level 2: T(I, I-2) for I = 2, 3 on warps 0, 1
    if (w < 2) {
        const int I = w + 2;
        float x[2][4] = {};
        blk_mma(x, at, I, I - 2, I - 2, lane);
        blk_mma(x, at, I, I - 1, I - 2, lane);
        finish_blk(at, ta, scratch + w * 16 * 17, x, I, I - 2, lane);
    }
    named_sync(bar_id, 128);
    // level 3: T(3, 0) on warp 0
    if (w == 0) {
        float x[2][4] = {};
        blk_mma(x, at, 3, 0, 0, lane);
        blk_mma(x, at, 3, 1, 0, lane);
        blk_mma(x, at, 3, 2, 0, lane);
        finish_blk(at, ta, scratch, x, 3, 0, lane);
    }
}

__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}


// Intra-chunk role, a three-stage pipeline over this CTA's items (16 warps):
//   warps 0-7  (builders): cumulative log decay and the gated operand tiles of
//              item n + 1 (inputs read from L2, prefetched by TMA one item
//              ahead), the record's Q e^G, Kd, gamma, then the Gram MMA; the
//              exact per-pair A and P of strongly decaying chunks instead go
//              straight to the Gram's tensor memory;
//   warps 8-11 (solvers): A and P of item n out of tensor memory, P to the
//              record, T = (I + A)^{-1}, then the W and Ut MMAs; TMEM owner;
//   warps 12-15 (writers): Ut^T and -W of item n - 1 to the record.
// Double-buffered (by item parity): the Gram's tensor memory, the W / Ut
// accumulators and the WB / UA operand tiles. One elected lane of warp 0
// (Gram) and of warp 8 (W, Ut) issues the MMAs.
template <bool PRE>
__device__ void intra_role(const Params &p, uint8_t *smem, int worker, int nworkers) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.n_heads;
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + kIOffBar;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kIOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kIOffMisc + 4);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(kIBGram + b), 1);
            mbar_init(bar(kIBCdone + b), 4);
            mbar_init(bar(kIBWU + b), 1);
            mbar_init(bar(kIBFdone + b), 4);
        }
        mbar_init(bar(kIBTear), blockDim.x / 32);
        mbar_init(bar(kIBDrain), 2);
        mbar_init(bar(kIBIn), 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 8) {
        tc::alloc(smem_u32(tmem_slot), kITmemCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = p.cu != nullptr && (*p.call_flags & kErrBadCu);
    const int64_t items = skip ? 0 : p.max_chunks * H;
    const int64_t rowe = static_cast<int64_t>(H) * 128;   // elements between tokens

    // next item of this worker at or after `item` that holds a real chunk
    auto next_real = [&](int64_t item) {
        while (item < items) {
            int n, L;
            int64_t t0;
            if (locate(p, item / H, n, t0, L)) break;
            item += nworkers;
        }
        return item;
    };
    // per-buffer barrier parity of item m (phases complete every second item)
    auto pb = [](int m) { return static_cast<uint32_t>((m >> 1) & 1); };

    // TMA prefetch of an item's gate boxes into L2 (one lane)
    auto prefetch = [&](int64_t itm) {
        if (itm >= items) return;
        int n, L;
        int64_t t0;
        const int64_t c = itm / H;
        const int h = static_cast<int>(itm - c * H);
        locate(p, c, n, t0, L);
        const int z = static_cast<int>(t0);
#pragma unroll
        for (int x = 0; x < 4; ++x) tma_prefetch_3d(&p.tm_g, 32 * x, h, z);
    };

    if (warp < 8) {
        // ================================================ builders (256 threads)
        const int ct = tid;                 // 0..255
        const int gq = lane >> 2, tq = lane & 3;   // fragment row / column pair
        float *tot = reinterpret_cast<float *>(smem + kIOffTot);   // [2][128] half sums
        int *red = reinterpret_cast<int *>(smem + kIOffRed);
        float *betas = reinterpret_cast<float *>(smem + kIOffBeta);
        float *gs = reinterpret_cast<float *>(smem + kIOffG);
        const __nv_bfloat16 *qg_ = static_cast<const __nv_bfloat16 *>(p.q);
        const __nv_bfloat16 *kg_ = static_cast<const __nv_bfloat16 *>(p.k);
        int it = 0, issued = 0;   // issued: input loads started (warp 0)
        if (warp == 0) {
            const int64_t first = next_real(worker);
            if (first < items) {
                int n2, L2;
                int64_t t02;
                const int64_t c2 = first / H;
                const int h2 = static_cast<int>(first - c2 * H);
                locate(p, c2, n2, t02, L2);
                arrive_tx_e(bar(kIBIn), 3 * 16384);
                const int z = static_cast<int>(t02);
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    tma_load_3d_e(sb + kIOffQKV + 8192 * x, &p.tm_q, 64 * x, h2, z, bar(kIBIn));
                    tma_load_3d_e(sb + kIOffQKV + 16384 + 8192 * x, &p.tm_k, 64 * x, h2, z, bar(kIBIn));
                    tma_load_3d_e(sb + kIOffQKV + 32768 + 8192 * x, &p.tm_v, 64 * x, h2, z, bar(kIBIn));
                }
                ++issued;
            }
        }
        for (int64_t item = next_real(worker); item < items; item = next_real(item + nworkers), ++it) {
            const int b = it & 1;
            const int64_t c = item / H;
            const int h = static_cast<int>(item - c * H);
            int n, L;
            int64_t t0;
            locate(p, c, n, t0, L);
            (void)n;
            uint8_t *rec = record_of(p, c, h);
            const int64_t base = t0 * rowe + static_cast<int64_t>(h) * 128;   // element of (t0, h, 0)
            if (ct == 0) {
                if (it == 0) prefetch(item);
                prefetch(next_real(item + nworkers));
            }
            // ring form: the slot's previous record must have been copied out
            if (p.ring_depth > 0 && ct == 0 && c >= p.ring_depth)
                wait_counter(p.consumed + h, c - p.ring_depth + 1, abort_flag, p.err);
            if (ct < kC) betas[ct] = ct < L ? __ldg(p.beta + (t0 + ct) * H + h) : 0.f;

            // ---- q, k, v fragments (thread (gq, tq) of warp w: rows 8 tb + gq, channels
            //      16 w + 8 cw + 2 tq and + 1) from the TMA tiles; the tiles are then
            //      free for the next item's loads
            uint32_t qf[8][2], kf[8][2], vf[8][2];
            wait_bar(bar(kIBIn), it & 1, abort_flag, p.err);
            {
                // ldmatrix x4: matrices (tb, cw) for tb = 2 tbp + (lane >> 4), cw = (lane >> 3) & 1
                const uint32_t lm = sb + kIOffQKV + sw_bf16(lane & 7, 16 * warp + 8 * ((lane >> 3) & 1)) +
                                    1024 * (lane >> 4);
#pragma unroll
                for (int tbp = 0; tbp < 4; ++tbp) {
                    uint32_t r[4];
                    ldsm_x4_addr(lm + 2048 * tbp, r);
                    qf[2 * tbp][0] = r[0]; qf[2 * tbp][1] = r[1];
                    qf[2 * tbp + 1][0] = r[2]; qf[2 * tbp + 1][1] = r[3];
                    ldsm_x4_addr(lm + 16384 + 2048 * tbp, r);
                    kf[2 * tbp][0] = r[0]; kf[2 * tbp][1] = r[1];
                    kf[2 * tbp + 1][0] = r[2]; kf[2 * tbp + 1][1] = r[3];
                    ldsm_x4_addr(lm + 32768 + 2048 * tbp, r);
                    vf[2 * tbp][0] = r[0]; vf[2 * tbp][1] = r[1];
                    vf[2 * tbp + 1][0] = r[2]; vf[2 * tbp + 1][1] = r[3];
                }
                // rows past the sequence end count as zero
#pragma unroll
                for (int tb = 0; tb < 8; ++tb)
                    if (8 * tb + gq >= L) {
                        qf[tb][0] = qf[tb][1] = kf[tb][0] = kf[tb][1] = vf[tb][0] = vf[tb][1] = 0u;
                    }
            }
            named_sync(1, 256);
            if (warp == 0) {
                const int64_t nxt = next_real(item + nworkers);
                if (nxt < items) {
                    int n2, L2;
                    int64_t t02;
                    const int64_t c2 = nxt / H;
                    const int h2 = static_cast<int>(nxt - c2 * H);
                    locate(p, c2, n2, t02, L2);
                    arrive_tx_e(bar(kIBIn), 3 * 16384);
                    const int z = static_cast<int>(t02);
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        tma_load_3d_e(sb + kIOffQKV + 8192 * x, &p.tm_q, 64 * x, h2, z, bar(kIBIn));
                        tma_load_3d_e(sb + kIOffQKV + 16384 + 8192 * x, &p.tm_k, 64 * x, h2, z, bar(kIBIn));
                        tma_load_3d_e(sb + kIOffQKV + 32768 + 8192 * x, &p.tm_v, 64 * x, h2, z, bar(kIBIn));
                    }
                    ++issued;
                }
            }

            // ---- cumulative log decay (base 2) into the G tile: thread = channel
            //      ct % 128, tokens [32 half, 32 half + 32); the second half adds the
            //      first half's sum
            float gmax = 0.f;
            bool anypos = false;
            {
                const int ch = ct & 127, th = ct >> 7;
                const uint32_t o0 = sw_f32(32 * th, ch);
                float x[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const int t = 32 * th + r;
                    x[r] = t < L ? __ldg(p.g + base + t * rowe + ch) : 0.f;
                }
                float run = 0.f;
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const int t = 32 * th + r;
                    float xv = x[r];
                    if (PRE && (p.pre & kPreGateLogits) && t < L) xv = log_sigmoid(xv);
                    anypos |= xv > 0.f;
                    run = fmaf(xv, kLog2e, run);
                    x[r] = run;
                }
                tot[th * 128 + ch] = run;
                if (named_sync_or(1, 256, *abort_flag != 0)) break;
                const float carry = th ? tot[ch] : 0.f;
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const uint32_t o = o0 + (r >> 3) * 1024 + (r & 7) * 128 +
                                       ((((ch & 31) >> 2) ^ (r & 7)) - ((ch & 31) >> 2)) * 16;
                    const float v = x[r] + carry;
                    *reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(gs) + o) = v;
                    gmax = fmaxf(gmax, fabsf(v));
                }
                // the factored form holds while |G| <= 80 (natural log); with
                // positive gates in the chunk while |G| <= 40, so that no
                // lower-triangle product exp(G_r - G_i) exceeds exp(80) either
                const bool pos = __any_sync(0xffffffffu, anypos);
                const float lim = pos ? 0.5f * kFactorRange * kLog2e : kFactorRange * kLog2e;
                const unsigned any_bad = __ballot_sync(0xffffffffu, !(gmax <= lim));
                if (lane == 0) red[warp] = any_bad != 0;
            }
            // the operand tiles are free: GA / GB once the Gram of item it - 1 is
            // done, WB / UA of buffer b once the W / Ut MMAs of item it - 2 are
            if (it >= 1) wait_bar(bar(kIBGram + (b ^ 1)), pb(it - 1), abort_flag, p.err);
            if (it >= 2) wait_bar(bar(kIBWU + b), pb(it - 2), abort_flag, p.err);
            tc::fence_after();
            named_sync(1, 256);
            bool exact = false;
#pragma unroll
            for (int w = 0; w < 8; ++w) exact |= red[w] != 0;

            // ---- gated operand tiles and the record's Qg, Kd, gamma
            const bool norm = PRE && (p.pre & kPreNormQK);
            float glast[2][2], egl[2][2];
#pragma unroll
            for (int cw = 0; cw < 2; ++cw)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int ch = 16 * warp + 8 * cw + 2 * tq + e;
                    glast[cw][e] = tot[ch] + tot[128 + ch];
                    egl[cw][e] = ex2f(glast[cw][e]);
                }
            if (gq == 0) {
#pragma unroll
                for (int cw = 0; cw < 2; ++cw) {
                    const int ch = 16 * warp + 8 * cw + 2 * tq;
                    *reinterpret_cast<float2 *>(rec + kRecGam + ch * 4) = make_float2(egl[cw][0], egl[cw][1]);
                }
            }
            float rq[8], rk[8];
#pragma unroll
            for (int tb = 0; tb < 8; ++tb) { rq[tb] = 1.f; rk[tb] = 1.f; }
            if (norm) {
                // row norms over the 128 channels: each warp's 16-channel partial
                // sums meet in the GB tile (written only after this)
                float *part = reinterpret_cast<float *>(smem + kIOffGB);   // [2][64][8]
#pragma unroll
                for (int tb = 0; tb < 8; ++tb) {
                    float sq = 0.f, sk = 0.f;
#pragma unroll
                    for (int cw = 0; cw < 2; ++cw) {
                        const float2 q2 = unpack_bf16(qf[tb][cw]), k2 = unpack_bf16(kf[tb][cw]);
                        sq = fmaf(q2.x, q2.x, fmaf(q2.y, q2.y, sq));
                        sk = fmaf(k2.x, k2.x, fmaf(k2.y, k2.y, sk));
                    }
                    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
                    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
                    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
                    sk += __shfl_xor_sync(0xffffffffu, sk, 2);
                    if (tq == 0) {
                        part[(8 * tb + gq) * 8 + warp] = sq;
                        part[(64 + 8 * tb + gq) * 8 + warp] = sk;
                    }
                }
                named_sync(1, 256);
#pragma unroll
                for (int tb = 0; tb < 8; ++tb) {
                    const int r = 8 * tb + gq;
                    float sq = 0.f, sk = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        sq += part[r * 8 + w];
                        sk += part[(64 + r) * 8 + w];
                    }
                    rq[tb] = rsqrtf(sq + kNormEps);
                    rk[tb] = rsqrtf(sk + kNormEps);
                }
                named_sync(1, 256);
            }
            // loop-invariant parts of the addresses: row 8 tb + gq of the G tile sits
            // tb * 1024 bytes after row gq (the swizzle depends on the row mod 8)
            const uint32_t g_off0 = sw_f32(gq, 16 * warp + 2 * tq);
            const uint32_t g_off1 = sw_f32(gq, 16 * warp + 8 + 2 * tq);
            const uint32_t o_tk0 = kmaj(0, 16 * warp, 128) + gq * 16 + tq * 4;   // + tb 2048 + cw 128
            const uint32_t o_kt0 = kmaj(16 * warp, 0, 64) + gq * 16 + tq * 4;    // + cw 1024 + tb 128
            uint8_t *const gB1 = rec + kRecB1 + o_tk0, *const gB2 = rec + kRecB2 + o_kt0;
            const float *const beta_r = betas + gq;
            const float sc = p.scale;
            // stmatrix row addresses: matrix m = lane >> 3 of a group of four is
            // (tb = 2 tbp + (m >> 1), cw = m & 1), row j = lane & 7
            const int mq = lane >> 3, jr = lane & 7;
            const uint32_t st_tk = sb + kmaj(0, 16 * warp, 128) + 2048 * (mq >> 1) + 128 * (mq & 1) + 16 * jr;
            const uint32_t st_kt = sb + kmaj(16 * warp, 0, 64) + 128 * (mq >> 1) + 1024 * (mq & 1) + 16 * jr;
#pragma unroll
            for (int tbp = 0; tbp < 4; ++tbp) {
                uint32_t ukb4[4], uqg4[4], ukn4[4], ubv4[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int tb = 2 * tbp + (m >> 1), cw = m & 1;
                    const float2 g2 = *reinterpret_cast<const float2 *>(
                        reinterpret_cast<const uint8_t *>(gs) + (cw ? g_off1 : g_off0) + 1024 * tb);
                    const float br = beta_r[8 * tb];
                    float2 q2 = unpack_bf16(qf[tb][cw]), k2 = unpack_bf16(kf[tb][cw]);
                    float2 v2 = unpack_bf16(vf[tb][cw]);
                    if (norm) {
                        q2.x *= rq[tb]; q2.y *= rq[tb];
                        k2.x *= rk[tb]; k2.y *= rk[tb];
                    }
                    const float e0 = ex2f(g2.x), e1 = ex2f(g2.y);
                    float2 qg = q2, kb = k2, kn = k2, kd, bv = v2;
                    mul2(qg.x, qg.y, e0 * sc, e1 * sc);
                    mul2(kb.x, kb.y, e0 * br, e1 * br);
                    if (!exact) {
                        mul2(kn.x, kn.y, ex2f(-g2.x), ex2f(-g2.y));
                        kd = kn;
                        mul2(kd.x, kd.y, egl[cw][0], egl[cw][1]);
                    } else {
                        kn = make_float2(0.f, 0.f);
                        kd = make_float2(k2.x * ex2f(glast[cw][0] - g2.x), k2.y * ex2f(glast[cw][1] - g2.y));
                    }
                    mul2(bv.x, bv.y, br, br);
                    uqg4[m] = pack_bf16(qg.x, qg.y);
                    ukb4[m] = pack_bf16(kb.x, kb.y);
                    ukn4[m] = pack_bf16(kn.x, kn.y);
                    ubv4[m] = pack_bf16(bv.x, bv.y);
                    const uint32_t ukd = pack_bf16(kd.x, kd.y);
                    // record B1 rows 0-63 (scale Q e^G) and B2 (Kd^T), straight from the fragments
                    st_global_u32(gB1 + 2048 * tb + 128 * cw, uqg4[m]);
                    st_global_u32(gB2 + 1024 * cw + 128 * tb, movt(ukd));
                }
                // [tok][key] core matrices: GA rows 0-63 (beta K e^G) and 64-127
                // (scale Q e^G), GB (K e^-G); transposed: WB, UA
                stsm_x4_addr(st_tk + kIOffGA + 4096 * tbp, ukb4[0], ukb4[1], ukb4[2], ukb4[3]);
                stsm_x4_addr(st_tk + kIOffGA + 16384 + 4096 * tbp, uqg4[0], uqg4[1], uqg4[2], uqg4[3]);
                stsm_x4_addr(st_tk + kIOffGB + 4096 * tbp, ukn4[0], ukn4[1], ukn4[2], ukn4[3]);
                stsm_x4_trans(st_kt + kIOffWB + 16384 * b + 256 * tbp, ukb4[0], ukb4[1], ukb4[2], ukb4[3]);
                stsm_x4_trans(st_kt + kIOffUA + 16384 * b + 256 * tbp, ubv4[0], ubv4[1], ubv4[2], ubv4[3]);
            }
            if (exact) {
                // exact per-pair exponentials into the fp32 staging (the GA tile,
                // [128][64]: rows 0-63 A, 64-127 P), then into the Gram's tensor
                // memory (buffer b, free once the solvers read item it - 2)
                named_sync(1, 256);
                float *stg = reinterpret_cast<float *>(smem + kIOffGA);
                float *rn = tot;   // inverse row norms: q 0..63, k 64..127
                if (ct < 128) {
                    float x = 1.f;
                    if (norm) {
                        const __nv_bfloat16 *src = (ct < 64 ? qg_ : kg_) + base + (ct & 63) * rowe;
                        float ss = 0.f;
                        if ((ct & 63) < L) {
                            for (int c8 = 0; c8 < 16; ++c8) {
                                const uint4 u = __ldg(reinterpret_cast<const uint4 *>(src + 8 * c8));
                                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 f = unpack_bf16(w4[e]);
                                    ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
                                }
                            }
                        }
                        x = rsqrtf(ss + kNormEps);
                    }
                    rn[ct] = x;
                }
                named_sync(1, 256);
                const int rp = ct >> 3, sub = ct & 7;
                bool overflow = false;
                for (int side = 0; side < 2; ++side) {
                    const int r = side == 0 ? rp : 63 - rp;
                    for (int i = sub; i <= r; i += 8) {
                        float sa = 0.f, sp = 0.f;
                        if (r < L) {
                            for (int c8 = 0; c8 < 16; ++c8) {
                                const uint4 kr = __ldg(reinterpret_cast<const uint4 *>(kg_ + base + r * rowe + 8 * c8));
                                const uint4 qr = __ldg(reinterpret_cast<const uint4 *>(qg_ + base + r * rowe + 8 * c8));
                                const uint4 ki = __ldg(reinterpret_cast<const uint4 *>(kg_ + base + i * rowe + 8 * c8));
                                const uint32_t krw[4] = {kr.x, kr.y, kr.z, kr.w};
                                const uint32_t qrw[4] = {qr.x, qr.y, qr.z, qr.w};
                                const uint32_t kiw[4] = {ki.x, ki.y, ki.z, ki.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 a = unpack_bf16(krw[e]), bq = unpack_bf16(qrw[e]),
                                                 cc = unpack_bf16(kiw[e]);
                                    const int ch = 8 * c8 + 2 * e;
                                    const float2 gr = *reinterpret_cast<const float2 *>(
                                        reinterpret_cast<const uint8_t *>(gs) + sw_f32(r, ch));
                                    const float2 gi = *reinterpret_cast<const float2 *>(
                                        reinterpret_cast<const uint8_t *>(gs) + sw_f32(i, ch));
                                    const float x0 = gr.x - gi.x, x1 = gr.y - gi.y;
                                    overflow |= x0 > kFactorRange * kLog2e || x1 > kFactorRange * kLog2e;
                                    const float e0 = ex2f(x0), e1 = ex2f(x1);
                                    sa = fmaf(a.x * cc.x, e0, sa);
                                    sa = fmaf(a.y * cc.y, e1, sa);
                                    sp = fmaf(bq.x * cc.x, e0, sp);
                                    sp = fmaf(bq.y * cc.y, e1, sp);
                                }
                            }
                        }
                        const bool real = r < L && i < L;
                        const float rki = rn[64 + i];
                        stg[r * 64 + i] = (i < r && real) ? betas[r] * rn[64 + r] * rki * sa : 0.f;
                        stg[(64 + r) * 64 + i] = real ? p.scale * rn[r] * rki * sp : 0.f;
                    }
                }
                if (overflow) atomicOr(p.err, kErrGate);
                if (it >= 2) wait_bar(bar(kIBCdone + b), pb(it - 2), abort_flag, p.err);
                named_sync(1, 256);
                tc::fence_after();
                {
                    // thread: Gram row 32 (warp % 4) + lane, columns [32 (warp / 4), +32);
                    // entries above the row's range are never read
                    const int q4 = warp & 3, half = warp >> 2, R = 32 * q4 + lane;
                    uint32_t d[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int i = 32 * half + j;
                        const bool keep = R < 64 ? (i < R) : (i <= R - 64);
                        d[j] = __float_as_uint(keep ? stg[R * 64 + i] : 0.f);
                    }
                    tst32(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 64 * b + 32 * half, d);
                    tc::st_wait();
                }
            }
            fence_async_smem();
            tc::fence_before();
            const bool stop = named_sync_or(1, 256, *abort_flag != 0);
            if (warp == 0) {
                // the Gram (or, for the exact form, the tensor-memory stores above)
                if (!exact && it >= 2) wait_bar(bar(kIBCdone + b), pb(it - 2), abort_flag, p.err);
                __syncwarp();
                tc::fence_after();
                if (!exact && !stop) {
                    const uint64_t dGA = tc::sdesc(sb + kIOffGA, 128, 2048);
                    const uint64_t dGB = tc::sdesc(sb + kIOffGB, 128, 2048);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss_e(tmem + 64 * b, dGA + 16 * kk, dGB + 16 * kk, kIdFull, kk > 0);
                }
                commit_e(bar(kIBGram + b));
            }
            if (stop) break;
        }
        if (warp == 0) {
            // no input load of this CTA is in flight when it exits (early exit
            // after an abort); every MMA this warp issued completes before the
            // teardown
            if (issued > 0) wait_bar(bar(kIBIn), (issued - 1) & 1, abort_flag, p.err);
            commit_e(bar(kIBDrain));
        }
    } else if (warp < 12) {
        // ================================================ solvers (warps 8-11)
        const int w = warp - 8, q4 = warp & 3;
        float *at = reinterpret_cast<float *>(smem + kIOffAT);
        uint8_t *ta = smem + kIOffTA;
        float *scratch = reinterpret_cast<float *>(smem + kIOffScr);
        int it = 0;
        for (int64_t item = next_real(worker); item < items; item = next_real(item + nworkers), ++it) {
            const int b = it & 1;
            const int64_t c = item / H;
            const int h = static_cast<int>(item - c * H);
            uint8_t *rec = record_of(p, c, h);
            wait_bar(bar(kIBGram + b), pb(it), abort_flag, p.err);
            // TA is free once the W / Ut MMAs of item it - 1 are done
            if (it >= 1) wait_bar(bar(kIBWU + (b ^ 1)), pb(it - 1), abort_flag, p.err);
            tc::fence_after();
            {
                // Gram row R = 32 q4 + lane: 0-63 A (to A^T in the strict upper
                // triangle), 64-127 P (to the record)
                const int R = 32 * q4 + lane;
                uint32_t d0[32], d1[32];
                tld32(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 64 * b, d0);
                tld32(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 64 * b + 32, d1);
                tc::ld_wait();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kIBCdone + b));
                if (R < 64) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i < R) at[i * kATStride + R] = __uint_as_float(d0[i]);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (32 + i < R) at[(32 + i) * kATStride + R] = __uint_as_float(d1[i]);
                } else {
                    const int r = R - 64;
#pragma unroll
                    for (int g8 = 0; g8 < 8; ++g8) {
                        uint32_t w4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i0 = 8 * g8 + 2 * e;
                            const uint32_t x0 = g8 < 4 ? d0[i0] : d1[i0 - 32];
                            const uint32_t x1 = g8 < 4 ? d0[i0 + 1] : d1[i0 + 1 - 32];
                            w4[e] = pack_bf16(i0 <= r ? __uint_as_float(x0) : 0.f,
                                              i0 + 1 <= r ? __uint_as_float(x1) : 0.f);
                        }
                        st_global_v4(rec + kRecB3 + kmaj(r, 8 * g8, 64),
                                     make_uint4(w4[0], w4[1], w4[2], w4[3]));
                    }
                }
            }
            if (named_sync_or(2, 128, *abort_flag != 0)) break;
            invert64(at, ta, scratch, w, lane, 2);
            fence_async_smem();
            tc::fence_before();
            named_sync(2, 128);
            if (w == 0) {
                // W and Ut^T into buffer b once the writers have read item it - 2's
                if (it >= 2) wait_bar(bar(kIBFdone + b), pb(it - 2), abort_flag, p.err);
                __syncwarp();
                tc::fence_after();
                const uint64_t dTA = tc::sdesc(sb + kIOffTA, 128, 1024);
                const uint64_t dWB = tc::sdesc(sb + kIOffWB + 16384 * b, 128, 1024);
                const uint64_t dUA = tc::sdesc(sb + kIOffUA + 16384 * b, 128, 1024);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)   // W = T (beta K e^G): M = 64, N = 128 keys, K = 64
                    mma_ss_e(tmem + 128 + 192 * b, dTA + 16 * kk, dWB + 16 * kk, kIdW, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)   // Ut^T = (beta V)^T T^T: M = 128 v, N = 64, K = 64
                    mma_ss_e(tmem + 256 + 192 * b, dUA + 16 * kk, dTA + 16 * kk, kIdFull, kk > 0);
                commit_e(bar(kIBWU + b));
            }
        }
        if (w == 0) commit_e(bar(kIBDrain));
    } else if (warp < 16) {
        // ================================================ writers (warps 12-15)
        const int q4 = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        const int gq = lane >> 2, tq = lane & 3;
        int it = 0;
        for (int64_t item = next_real(worker); item < items; item = next_real(item + nworkers), ++it) {
            const int b = it & 1;
            const int64_t c = item / H;
            const int h = static_cast<int>(item - c * H);
            uint8_t *rec = record_of(p, c, h);
            wait_bar(bar(kIBWU + b), pb(it), abort_flag, p.err);
            tc::fence_after();
            // Ut^T row v = 32 q4 + lane, 32 tokens at a time, then W (M = 64): rows
            // 16 q4 + (0..15), thread (gq, tq) rows gq, gq + 8 and the column pair
            // 2 tq of each 8-column block, 64 keys at a time (one half of the
            // tensor-memory data in registers at once)
            const int v = 32 * q4 + lane;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t d[32];
                tld32(tmem + lane_base + 256 + 192 * b + 32 * hf, d);
                tc::ld_wait();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t *dd = d + 8 * j;
                    st_global_v4(rec + kRecUt + ut_off(v, 4 * hf + j),
                                 make_uint4(pack_bf16(__uint_as_float(dd[0]), __uint_as_float(dd[1])),
                                            pack_bf16(__uint_as_float(dd[2]), __uint_as_float(dd[3])),
                                            pack_bf16(__uint_as_float(dd[4]), __uint_as_float(dd[5])),
                                            pack_bf16(__uint_as_float(dd[6]), __uint_as_float(dd[7]))));
                }
            }
            const int r0 = 16 * q4 + gq;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t wr[8][4];
#pragma unroll
                for (int b8 = 0; b8 < 8; ++b8)
                    tc::ld_16x256b(tmem + lane_base + 128 + 192 * b + 8 * (8 * hf + b8), wr[b8][0],
                                   wr[b8][1], wr[b8][2], wr[b8][3]);
                tc::ld_wait();
                if (hf == 1) {
                    // the accumulators of buffer b are read: release them
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kIBFdone + b));
                }
#pragma unroll
                for (int b8 = 0; b8 < 8; ++b8) {
                    const int key = 8 * (8 * hf + b8) + 2 * tq;
                    st_global_u32(rec + kRecB1 + kmaj(64 + r0, key, 128),
                                  pack_bf16(-__uint_as_float(wr[b8][0]), -__uint_as_float(wr[b8][1])));
                    st_global_u32(rec + kRecB1 + kmaj(64 + r0 + 8, key, 128),
                                  pack_bf16(-__uint_as_float(wr[b8][2]), -__uint_as_float(wr[b8][3])));
                }
            }
            // the whole record is written once the writers are done (the builders'
            // and solvers' parts came earlier in the item's chain of barriers)
            const bool stop = named_sync_or(3, 128, *abort_flag != 0);
            if (p.ring_depth > 0 && warp == 12 && lane == 0 && !stop) {
                __threadfence();
                st_release(p.ready + (c % p.ring_depth) * H + h, c + 1);
            }
            if (stop) break;
        }
    }

    // ---- teardown: every warp, then TMEM is freed by warp 8 once every MMA
    //      of the two issuing warps has completed
    tc::fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kIBTear));
    if (warp == 8) {
        wait_bar(bar(kIBTear), 0, abort_flag, p.err);
        wait_bar(bar(kIBDrain), 0, abort_flag, p.err);
        tc::fence_after();
        tc::dealloc(tmem, kITmemCols);
    }
}

// ============================================================================
// Recurrent role: one (sequence, head) chain at a time, 448 threads.
// warps 0-7 state and U epilogues (lane quadrant warp % 4, key / token half
// warp / 4), warp 8 record copies, warp 9 MMA issue (one elected lane) and
// TMEM, warps 10-13 the o epilogue.
// Tensor memory: S^T [0,128), O^T [128,192), U^T [192,256) in fp32, and the
// bf16 operands S^T (two buffers, [256,320) and [320,384)) and U^T
// [384,416), two values per column. Per step, in issue order:
//   MMA-U: U = S^T (-W)^T          (N = 64, K = 128 keys; the first half of
//                                   the keys as soon as the state epilogue has them)
//   MMA-B: [S | O] += U^T [Kd^T ; scale P]^T   (N = 192, K = 64 tokens: one
//                                   group, since O sits between S and U)
//   MMA-O: O += S^T (scale Qg)^T   (N = 64, after the state is ready again)
// The o warps read O and set it back to zero before MMA-B of the next step.
// ============================================================================
constexpr int kChainThreads = 448;

constexpr uint32_t kIdA = tc::idesc(128, 64, 1);       // MMA-A halves: M=128, N=64
constexpr uint32_t kIdB = tc::idesc(128, 192, 1);      // MMA-B: M=128, N=192
constexpr uint32_t kTAs = 256, kTAu = 384;             // bf16 operand columns

__device__ __forceinline__ void mma_ts_e(uint32_t d, uint32_t a, uint64_t b, uint32_t id,
                                         uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

__device__ void chain_role(const Params &p, uint8_t *smem, int h, int n_first, int n_step) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.n_heads;
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + kCOffBar;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kCOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kCOffMisc + 4);
    if (tid == 0) {
        for (int s = 0; s < kCStages; ++s) {
            mbar_init(bar(kCBFull + s), 1);
            mbar_init(bar(kCBEmpty + s), 9);
        }
        mbar_init(bar(kCBSop), 8);
        mbar_init(bar(kCBSop + 1), 8);
        mbar_init(bar(kCBUdone), 1);
        mbar_init(bar(kCBUop), 8);
        mbar_init(bar(kCBSdone), 1);
        mbar_init(bar(kCBOdone), 1);
        mbar_init(bar(kCBOfree), 4);
        mbar_init(bar(kCBTear), blockDim.x / 32);
        mbar_init(bar(kCBDrain), 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) {
        tc::alloc(smem_u32(tmem_slot), kCTmemCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = p.cu != nullptr && (*p.call_flags & kErrBadCu);

    // chunks of sequence n: first global chunk index and count, token range
    auto seq_chunks = [&](int n, int64_t &c0, int &nck, int64_t &tb, int64_t &te) {
        if (p.cu == nullptr) {
            c0 = static_cast<int64_t>(n) * p.cps;
            nck = p.cps;
            tb = static_cast<int64_t>(n) * p.seq_len;
            te = tb + p.seq_len;
        } else {
            c0 = p.chunk_off[n];
            nck = p.chunk_off[n + 1] - p.chunk_off[n];
            tb = p.cu[n];
            te = p.cu[n + 1];
        }
    };

    if (skip) {
        // nothing
    } else if (warp < 8) {
        // ===================================================== state and U epilogues
        // A failed (bounded) wait raises the abort flag and the warp goes on;
        // the eight warps leave together at the next OR-reducing barrier.
        const int q4 = warp & 3, half = warp >> 2;
        const int v = 32 * q4 + lane;                      // value channel, TMEM lane
        const uint32_t tS = tmem + (static_cast<uint32_t>(32 * q4) << 16);
        int64_t gi = 0;                                    // global step counter
        bool stop = false;
        for (int n = n_first; n < p.n_seqs && !stop; n += n_step) {
            int64_t c0, tb, te;
            int nck;
            seq_chunks(n, c0, nck, tb, te);
            const int64_t sbase = (static_cast<int64_t>(n) * H + h) * 128 * 128;
            // initial state into S^T: keys [64 half, 64 half + 64), lane v
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int key = 64 * half + 32 * c2 + j;
                    r[j] = __float_as_uint(p.s0 ? p.s0[sbase + key * 128 + v] : 0.f);
                }
                tst32(tS + 64 * half + 32 * c2, r);
            }
            tc::st_wait();
            for (int i = 0; i < nck; ++i, ++gi) {
                const int s = static_cast<int>(gi % kCStages);
                const uint8_t *stg = smem + s * kRecBytes;
                wait_bar(bar(kCBFull + s), (gi / kCStages) & 1, abort_flag, p.err);
                if (i > 0) wait_bar(bar(kCBSdone), (gi - 1) & 1, abort_flag, p.err);
                tc::fence_after();
                // ---- state: S^T (keys of this half) -> bf16 operand in TMEM (buffer
                //      gi % 2); keys [64 half + 32 c2, +32) signal barrier sop + c2; the
                //      decayed state goes back to TMEM after both signals
                const float *gam = reinterpret_cast<const float *>(stg + kRecGam) + 64 * half;
                const uint32_t tAs = tS + kTAs + 64 * static_cast<uint32_t>(gi & 1) + 32 * half;
                uint32_t r0[32], r1[32];
                tld32(tS + 64 * half, r0);
                tld32(tS + 64 * half + 32, r1);
                tc::ld_wait();
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const uint32_t (&r)[32] = c2 ? r1 : r0;
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        pk[j] = pack_bf16(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                    tc::st16(tAs + 16 * c2, pk);
                    tc::st_wait();
                    tc::fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kCBSop + c2));
                }
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    uint32_t (&r)[32] = c2 ? r1 : r0;
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 gg = *reinterpret_cast<const float4 *>(gam + 32 * c2 + j);
                        float a0 = __uint_as_float(r[j]), a1 = __uint_as_float(r[j + 1]);
                        float a2 = __uint_as_float(r[j + 2]), a3 = __uint_as_float(r[j + 3]);
                        mul2(a0, a1, gg.x, gg.y);
                        mul2(a2, a3, gg.z, gg.w);
                        r[j] = __float_as_uint(a0);
                        r[j + 1] = __float_as_uint(a1);
                        r[j + 2] = __float_as_uint(a2);
                        r[j + 3] = __float_as_uint(a3);
                    }
                    tst32(tS + 64 * half + 32 * c2, r);
                }
                // ---- U^T = Ut^T + (-W S)^T (tokens of this half) -> bf16 operand in TMEM
                wait_bar(bar(kCBUdone), gi & 1, abort_flag, p.err);
                tc::fence_after();
                {
                    uint32_t d[32];
                    tld32(tS + 192 + 32 * half, d);
                    uint4 u4[4];
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4)
                        u4[j4] = *reinterpret_cast<const uint4 *>(stg + kRecUt + ut_off(v, 4 * half + j4));
                    tc::ld_wait();
                    uint32_t pk[16];
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const uint32_t uw[4] = {u4[j4].x, u4[j4].y, u4[j4].z, u4[j4].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_bf16(uw[e]);
                            pk[4 * j4 + e] = pack_bf16(f.x + __uint_as_float(d[8 * j4 + 2 * e]),
                                                       f.y + __uint_as_float(d[8 * j4 + 2 * e + 1]));
                        }
                    }
                    tc::st16(tS + kTAu + 16 * half, pk);
                    tc::st_wait();
                }
                tc::fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(kCBUop));
                    mbar_arrive(bar(kCBEmpty + s));
                }
                if (named_sync_or(3, 256, *abort_flag != 0)) { stop = true; break; }
            }
            if (stop) break;
            if (nck > 0) {
                wait_bar(bar(kCBSdone), (gi - 1) & 1, abort_flag, p.err);
                tc::fence_after();
            }
            if (named_sync_or(3, 256, *abort_flag != 0)) break;
            if (p.s_final != nullptr) {
                uint32_t r0[32], r1[32];
                tld32(tS + 64 * half, r0);
                tld32(tS + 64 * half + 32, r1);
                tc::ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    p.s_final[sbase + (64 * half + j) * 128 + v] = __uint_as_float(r0[j]);
                    p.s_final[sbase + (64 * half + 32 + j) * 128 + v] = __uint_as_float(r1[j]);
                }
            }
            tc::fence_before();
        }
    } else if (warp >= 10 && warp < 14) {
        // ===================================================== o epilogue
        // O accumulates U^T P^T (MMA-B) and S^T Qg^T (MMA-O) from zero: these
        // warps clear it once at the start and again after each read
        const int q4 = warp & 3;
        const int v = 32 * q4 + lane;
        const uint32_t tO = tmem + (static_cast<uint32_t>(32 * q4) << 16) + 128;
        __nv_bfloat16 *outp = static_cast<__nv_bfloat16 *>(p.out);
        uint32_t zero[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) zero[j] = 0u;
        tst32(tO, zero);
        tst32(tO + 32, zero);
        tc::st_wait();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kCBOfree));
        int64_t gi = 0;
        bool ok = true;
        for (int n = n_first; n < p.n_seqs && ok; n += n_step) {
            int64_t c0, tb, te;
            int nck;
            seq_chunks(n, c0, nck, tb, te);
            for (int i = 0; i < nck; ++i, ++gi) {
                if (!wait_bar(bar(kCBOdone), gi & 1, abort_flag, p.err)) { ok = false; break; }
                tc::fence_after();
                uint32_t d0[32], d1[32];
                tld32(tO, d0);
                tld32(tO + 32, d1);
                tc::ld_wait();
                tst32(tO, zero);
                tst32(tO + 32, zero);
                tc::st_wait();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kCBOfree));
                const int64_t t0 = tb + static_cast<int64_t>(kC) * i;
                const int L = static_cast<int>(te - t0 < kC ? te - t0 : kC);
                __nv_bfloat16 *op = outp + (t0 * H + h) * 128 + v;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < L) op[static_cast<int64_t>(j) * H * 128] = __float2bfloat16_rn(__uint_as_float(d0[j]));
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (32 + j < L)
                        op[static_cast<int64_t>(32 + j) * H * 128] = __float2bfloat16_rn(__uint_as_float(d1[j]));
            }
        }
    } else if (warp == 8) {
        // ===================================================== record copies
        if (lane == 0) {
            int64_t gi = 0, issued = 0;
            int64_t pend_c = -1, pend_gi = 0;   // ring form: copy whose completion is unpublished
            bool ok = true;
            for (int n = n_first; n < p.n_seqs && ok; n += n_step) {
                int64_t c0, tb, te;
                int nck;
                seq_chunks(n, c0, nck, tb, te);
                for (int i = 0; i < nck; ++i, ++gi) {
                    const int s = static_cast<int>(gi % kCStages);
                    const int64_t c = c0 + i;
                    if (gi >= kCStages &&
                        !wait_bar(bar(kCBEmpty + s), ((gi / kCStages) - 1) & 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    if (p.ring_depth > 0) {
                        if (!wait_counter(p.ready + (c % p.ring_depth) * H + h, c + 1, abort_flag,
                                          p.err)) {
                            ok = false;
                            break;
                        }
                        asm volatile("fence.proxy.async.global;\n" ::: "memory");
                    }
                    const uint8_t *src = record_of(p, c, h);
                    mbar_arrive_expect_tx(bar(kCBFull + s), kRecBytes);
#pragma unroll
                    for (int part = 0; part < 4; ++part)
                        bulk_g2s(sb + s * kRecBytes + part * (kRecBytes / 4), src + part * (kRecBytes / 4),
                                 kRecBytes / 4, bar(kCBFull + s));
                    issued = gi + 1;
                    if (p.ring_depth > 0) {
                        if (pend_c >= 0) {
                            const int ps = static_cast<int>(pend_gi % kCStages);
                            if (!wait_bar(bar(kCBFull + ps), (pend_gi / kCStages) & 1, abort_flag, p.err)) {
                                ok = false;
                                break;
                            }
                            st_release(p.consumed + h, pend_c + 1);
                        }
                        pend_c = c;
                        pend_gi = gi;
                    }
                }
            }
            if (ok && p.ring_depth > 0 && pend_c >= 0) {
                const int ps = static_cast<int>(pend_gi % kCStages);
                if (wait_bar(bar(kCBFull + ps), (pend_gi / kCStages) & 1, abort_flag, p.err))
                    st_release(p.consumed + h, pend_c + 1);
            }
            // drain: no copy of this CTA is still in flight when it exits
            for (int64_t g2 = issued - kCStages; g2 < issued; ++g2) {
                if (g2 < 0) continue;
                const int ps = static_cast<int>(g2 % kCStages);
                mbar_wait(bar(kCBFull + ps), (g2 / kCStages) & 1);
            }
        }
    } else if (warp == 9) {
        // ===================================================== MMA issue (warp 9, one elected lane)
        int64_t gi = 0;
        bool ok = true;
        for (int n = n_first; n < p.n_seqs && ok; n += n_step) {
            int64_t c0, tb, te;
            int nck;
            seq_chunks(n, c0, nck, tb, te);
            for (int i = 0; i < nck; ++i, ++gi) {
                const int s = static_cast<int>(gi % kCStages);
                const uint32_t stg = sb + s * kRecBytes;
                const uint32_t tAs = tmem + kTAs + 64 * static_cast<uint32_t>(gi & 1);
                const uint64_t dQ = tc::sdesc(stg + kRecB1, 128, 2048);           // rows 0-63: Qg
                const uint64_t dW = tc::sdesc(stg + kRecB1 + 16384, 128, 2048);   // rows 64-127: -W
                const uint64_t dB2 = tc::sdesc(stg + kRecB2, 128, 1024);
                if (!wait_bar(bar(kCBFull + s), (gi / kCStages) & 1, abort_flag, p.err)) { ok = false; break; }
                // U = S^T (-W)^T, the key blocks (16 keys) of each state chunk once it is in
                // (chunk c2 of the two key halves h: blocks 4 h + 2 c2 and 4 h + 2 c2 + 1)
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    if (!wait_bar(bar(kCBSop + c2), gi & 1, abort_flag, p.err)) { ok = false; break; }
                    __syncwarp();
                    tc::fence_after();
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const int k16 = 4 * (x >> 1) + 2 * c2 + (x & 1);
                        mma_ts_e(tmem + 192, tAs + 8 * k16, dW + 16 * k16, kIdA,
                                 (c2 > 0 || x > 0) ? 1u : 0u);
                    }
                }
                if (!ok) break;
                commit_e(bar(kCBUdone));
                // [S | O] += U^T [Kd^T ; scale P]^T, once U^T is in and O was read and cleared
                if (!wait_bar(bar(kCBUop), gi & 1, abort_flag, p.err) ||
                    !wait_bar(bar(kCBOfree), gi & 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                tc::fence_after();
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16)
                    mma_ts_e(tmem, tmem + kTAu + 8 * k16, dB2 + 16 * k16, kIdB, 1);
                commit_e(bar(kCBSdone));
                // O += S^T (scale Qg)^T
#pragma unroll
                for (int k16 = 0; k16 < 8; ++k16)
                    mma_ts_e(tmem + 128, tAs + 8 * k16, dQ + 16 * k16, kIdA, 1);
                commit_e(bar(kCBOdone));
                commit_e(bar(kCBEmpty + s));
            }
        }
        // every MMA this warp issued has completed before the teardown
        commit_e(bar(kCBDrain));
        wait_bar(bar(kCBDrain), 0, abort_flag, p.err);
    }

    // ---- teardown
    tc::fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kCBTear));
    if (warp == 9) {
        wait_bar(bar(kCBTear), 0, abort_flag, p.err);
        tc::fence_after();
        tc::dealloc(tmem, kCTmemCols);
    }
}

// ------------------------------------------------------------------ kernels
template <bool PRE>
__global__ void __launch_bounds__(kIThreads, 1) kda_c64_intra_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    intra_role<PRE>(p, smem, blockIdx.x, gridDim.x);
}

__global__ void __launch_bounds__(kChainThreads, 1) kda_c64_chain_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int H = p.n_heads;
    chain_role(p, smem, blockIdx.x % H, blockIdx.x / H, p.n_seqs);
}

// One cooperative launch: CTAs [0, n_chain) run head blockIdx.x's chains over
// all sequences, the others build the records into the ring. The last CTA to
// finish clears the ring counters for the next call.
template <bool PRE>
__global__ void __launch_bounds__(kIThreads, 1) kda_c64_fused_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    if (static_cast<int>(blockIdx.x) < p.n_chain)
        chain_role(p, smem, blockIdx.x, 0, 1);
    else
        intra_role<PRE>(p, smem, blockIdx.x - p.n_chain, gridDim.x - p.n_chain);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.exit_ctr, 1) == static_cast<int>(gridDim.x) - 1) {
            const int nr = p.ring_depth * p.n_heads;
            for (int i = 0; i < nr; ++i) p.ready[i] = 0;
            for (int i = 0; i < p.n_heads; ++i) p.consumed[i] = 0;
            *p.exit_ctr = 0;
            __threadfence();
        }
    }
}

}  // namespace
}  // namespace c64
}  // namespace kda

// ============================================================================
// Host side
// ============================================================================
namespace kda {

void *tensor_map_encoder() {
    static void *fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<void *>(nullptr);
        }
        return f;
    }();
    return fn;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() { return reinterpret_cast<EncodeTiledFn>(tensor_map_encoder()); }

// [tokens, H, 128] row-major as a 3D tiled map (channel, head, token); a box
// is 64 tokens x 1 head x 128 bytes of channels (64 bf16 or 32 fp32), stored
// with 128-byte swizzling; rows past the end read as zero.
bool encode_rows(CUtensorMap *m, const void *base, bool f32, int64_t H, int64_t tokens) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t es = f32 ? 4 : 2;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[2] = {128 * es, static_cast<cuuint64_t>(H) * 128 * es};
    const cuuint32_t box[3] = {f32 ? 32u : 64u, 1, static_cast<cuuint32_t>(c64::kC)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_params(const C64Args &a, c64::Params *p) {
    *p = c64::Params{};
    if (!encode_rows(&p->tm_q, a.q, false, a.n_heads, a.tokens) ||
        !encode_rows(&p->tm_k, a.k, false, a.n_heads, a.tokens) ||
        !encode_rows(&p->tm_v, a.v, false, a.n_heads, a.tokens) ||
        !encode_rows(&p->tm_g, a.g, true, a.n_heads, a.tokens))
        return false;
    p->q = a.q;
    p->k = a.k;
    p->v = a.v;
    p->g = a.g;
    p->beta = a.beta;
    p->s0 = a.s0;
    p->out = a.out;
    p->s_final = a.s_final;
    p->rec = a.rec;
    p->err = a.err;
    p->cu = a.cu;
    p->chunk_off = a.chunk_off;
    p->call_flags = a.call_flags;
    p->seq_len = a.seq_len;
    p->max_chunks = a.max_chunks;
    p->n_seqs = a.n_seqs;
    p->n_heads = a.n_heads;
    p->cps = a.cps;
    p->scale = a.scale;
    p->pre = a.pre;
    p->ring_depth = a.ring_depth;
    p->n_chain = a.n_chain;
    p->ready = a.ready;
    p->consumed = a.consumed;
    p->exit_ctr = a.exit_ctr;
    return true;
}

}  // namespace

cudaError_t configure_c64() {
    const void *fns[] = {reinterpret_cast<const void *>(c64::kda_c64_intra_kernel<false>),
                         reinterpret_cast<const void *>(c64::kda_c64_intra_kernel<true>),
                         reinterpret_cast<const void *>(c64::kda_c64_chain_kernel),
                         reinterpret_cast<const void *>(c64::kda_c64_fused_kernel<false>),
                         reinterpret_cast<const void *>(c64::kda_c64_fused_kernel<true>)};
    for (const void *f : fns) {
        const cudaError_t e =
            cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, c64::kSmem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_c64_intra(const C64Args &a, int intra_ctas, cudaStream_t stream) {
    if (a.tokens <= 0) return cudaSuccess;
    c64::Params p;
    if (!make_params(a, &p)) return cudaErrorInvalidValue;
    p.ring_depth = 0;
    p.n_chain = 0;
    const int64_t items = a.max_chunks * a.n_heads;
    int64_t grid = intra_ctas < items ? intra_ctas : items;
    if (grid < 1) grid = 1;
    if (a.pre != 0)
        c64::kda_c64_intra_kernel<true><<<static_cast<unsigned>(grid), c64::kIThreads, c64::kSmem,
                                          stream>>>(p);
    else
        c64::kda_c64_intra_kernel<false><<<static_cast<unsigned>(grid), c64::kIThreads, c64::kSmem,
                                           stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_c64_chain(const C64Args &a, cudaStream_t stream) {
    const int64_t units = static_cast<int64_t>(a.n_seqs) * a.n_heads;
    if (units <= 0) return cudaSuccess;
    c64::Params p;
    if (a.tokens > 0) {
        if (!make_params(a, &p)) return cudaErrorInvalidValue;
    } else {
        // no tokens: the chains only carry the initial states to the final ones
        p = c64::Params{};
        p.s0 = a.s0;
        p.s_final = a.s_final;
        p.err = a.err;
        p.cu = a.cu;
        p.chunk_off = a.chunk_off;
        p.call_flags = a.call_flags;
        p.n_seqs = a.n_seqs;
        p.n_heads = a.n_heads;
    }
    p.ring_depth = 0;
    p.n_chain = 0;
    c64::kda_c64_chain_kernel<<<static_cast<unsigned>(units), c64::kChainThreads, c64::kSmem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_c64_fused(const C64Args &a, int grid, cudaStream_t stream) {
    if (a.tokens <= 0) return cudaSuccess;
    c64::Params p;
    if (!make_params(a, &p)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(c64::kIThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(c64::kSmem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return a.pre != 0 ? cudaLaunchKernelEx(&cfg, c64::kda_c64_fused_kernel<true>, p)
                      : cudaLaunchKernelEx(&cfg, c64::kda_c64_fused_kernel<false>, p);
}

}  // namespace kda
