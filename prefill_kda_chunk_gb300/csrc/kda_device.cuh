// Device-side building blocks shared by the KDA prefill kernels: the
// chunk-record layout that the intra-chunk kernel writes and the recurrent
// kernel reads, the shared-memory swizzle, and thin inline-PTX wrappers
// (warp MMA, ldmatrix, mbarrier, bulk async copy, bounded waits).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {

constexpr int kChunk = 16;   // tokens per chunk
constexpr int kDim = 128;    // K = V

// One record per (chunk, head), written by the intra-chunk kernel and read
// whole by the recurrent kernel with bulk copies. 16x128 bf16 tiles are
// stored with the 16-byte granule index XOR-ed by (row & 7) so that eight
// consecutive rows of one granule column fall in distinct shared-memory
// banks (ldmatrix reads them without conflicts).
constexpr int kRecW = 0;          // -W = -(T diag(beta)) (K * exp(G))   [16 tok][128 key], swizzled
constexpr int kRecQg = 4096;      // scale * Q * exp(G)                  [16 tok][128 key], swizzled
constexpr int kRecKd = 8192;      // K * exp(G_last - G)                 [16 tok][128 key], swizzled
constexpr int kRecP = 12288;      // scale * P, lower triangle incl. diag [16 r][16 i] bf16
constexpr int kRecGamma = 12800;  // exp(G_last)                         [128] fp32
constexpr int kRecUt = 13312;     // (T diag(beta) V)^T                  [128 val][16 tok] bf16
constexpr int kRecBytes = 17408;

// Input preprocessing done inside the kernels (the flags of the C ABI):
// q and k divided by their L2 norm per (token, head), and g given as gate
// logits x with the log decay taken as logsigmoid(x).
enum : int { kPreNormQK = 1, kPreGateLogits = 2 };
constexpr float kNormEps = 1e-6f;

__device__ __forceinline__ float log_sigmoid(float x) {
    // log(1 / (1 + e^-x)) = min(x, 0) - log(1 + e^-|x|)
    return fminf(x, 0.f) - __logf(1.f + __expf(-fabsf(x)));
}

// Error bits. kErrBadCu lives in the per-call flag word and the sticky
// per-device word; the others only in the sticky word.
enum : int { kErrBadCu = 1, kErrTimeout = 2, kErrGate = 4 };

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// 1 if c else 0, through an instruction the compiler does not look into: a
// loop of that many trips stays a branch. Work written as an if can be
// predicated into the straight-line code around it, and then costs every
// thread that does not need it.
__device__ __forceinline__ int opaque_trips(bool c) {
    int t;
    asm volatile("mov.b32 %0, %1;" : "=r"(t) : "r"(static_cast<int>(c)));
    return t;
}

__device__ __forceinline__ int swz(int row, int col) {
    return row * 256 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A * B, m16n8k16, bf16 operands, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same MMA as a register-only asm (not volatile: the compiler may move it
// around other work; use it where nothing else orders it).
__device__ __forceinline__ void mma_r(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                      uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (a, b) *= (x, y) as one packed fp32x2 multiply
__device__ __forceinline__ void mul2(float &a, float &b, float x, float y) {
    asm("{\n .reg .b64 t, u;\n mov.b64 t, {%0, %1};\n mov.b64 u, {%2, %3};\n"
        " mul.rn.f32x2 t, t, u;\n mov.b64 {%0, %1}, t;\n}\n"
        : "+f"(a), "+f"(b) : "f"(x), "f"(y));
}
// Non-blocking look at an mbarrier phase (acquire on success).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Four 8x8 b16 matrices from registers to shared memory, transposed.
__device__ __forceinline__ void stsm_x4_t(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false after
// kWaitLimitNs without completion (the caller records a timeout).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// Bulk (non-tensor) async copy global -> shared, completion counted in
// bytes on an mbarrier. Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// 16-byte async copy global -> shared (L1 bypassed); src_bytes < 16 zero-fills
// the rest of the destination (0 reads nothing).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;\n" ::: "memory");
}

}  // namespace kda
