// Token-parallel half of chunked KDA prefill: the packed-batch prologue, the
// intra-chunk kernel and its exact-form companion. The per-chunk work (A, P,
// (I + A)^{-1}, W, Ut and the record) is in kda_intra_body.cuh.
//
// Record stores are evict-first (st.global.cs): the records are read back by
// the recurrent kernel long after they leave L2, so keeping them there only
// pushes out input rows. No L2 prefetch of later chunks either: on GB300 it
// raised DRAM reads and cost time.

#include "kda_device.cuh"
#include "kda_internal.h"
#include "kda_intra_body.cuh"

namespace kda {

namespace {

// Per device: SM count and resident CTAs per SM of the intra-chunk kernel.
constexpr int kMaxDev = 128;
int g_sm_count[kMaxDev] = {};
int g_blocks_per_sm[kMaxDev] = {};
int g_exact_blocks_per_sm[kMaxDev] = {};

// Persistent: each warp walks (chunk, head) items with a grid-wide stride,
// items ordered chunk-major so the warps of a CTA share a chunk's rows.
// PRE = false compiles no preprocessing code at all (p.pre must be 0);
// PRE = true reads the preprocessing flags from p.pre. GRAD = true is the
// gradient call's instantiation: it also writes (I + A)^{-1} to p.tinv and
// raises p.wide_flag for chunks out of the start-referenced range (the
// forward's instantiation carries no code for either).
template <bool PRE, bool GRAD = false>
__global__ void __launch_bounds__(kIntraWarps * 32, 3)
kda_intra_chunk_kernel(IntraParams p, int64_t max_chunks) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    // let the exact-form kernel, launched next as a programmatic dependent, be
    // scheduled now: its CTAs start as these exit and then wait for the grid
    asm volatile("griddepcontrol.launch_dependents;");
    if (geo.cu != nullptr && (*geo.call_flags & kErrBadCu)) return;
    IntraWarpSmem &sm = reinterpret_cast<IntraWarpSmem *>(smem_raw)[warp];
    const int64_t items = max_chunks * H;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kIntraWarps;

    for (int64_t item = static_cast<int64_t>(blockIdx.x) * kIntraWarps + warp; item < items;
         item += stride) {
    const int64_t chunk = item / H;
    const int h = static_cast<int>(item - chunk * H);
    int n, L;
    int64_t t0, rec_idx;
    if (!locate_chunk(geo, chunk, n, t0, L, rec_idx)) continue;
    (void)n;
    const int64_t ri = rec_idx * H + h;
    uint8_t *rec = p.rec + ri * kRecBytes;
    intra_item<PRE, false, GRAD>(p, sm, t0, L, h, rec, p.tinv != nullptr ? p.tinv + ri * 320 : nullptr,
                                 static_cast<int32_t>(item));
    }  // items
}

// The exact form over the chunk-heads the intra-chunk kernel listed (it runs
// right after it on the same stream and rewrites their whole records): one
// item per warp at a time, warps strided over the list. With an empty list it
// only reads the count. Otherwise the last CTA to finish zeroes the count (and
// its own finish counter), so the next call starts from an empty list.
// Two CTAs per SM: with the registers that frees it spills nothing, which
// measured 2 % faster than three CTAs with spills.
template <bool PRE>
__global__ void __launch_bounds__(kIntraWarps * 32, 2)
kda_intra_exact_kernel(IntraParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5;
    const ChunkGeometry &geo = p.geo;
    const int H = geo.n_heads;
    IntraWarpSmem &sm = reinterpret_cast<IntraWarpSmem *>(smem_raw)[warp];
    // launched as a programmatic dependent of the intra-chunk kernel: wait for
    // all of it (and its memory) before reading the list
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int count = __ldcg(p.exact_ctr);
    const int64_t wstride = static_cast<int64_t>(gridDim.x) * kIntraWarps;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kIntraWarps + warp; j < count;
         j += wstride) {
        const int64_t item = __ldcg(p.exact_list + j);
        const int64_t chunk = item / H;
        const int h = static_cast<int>(item - chunk * H);
        int n, L;
        int64_t t0, rec_idx;
        if (!locate_chunk(geo, chunk, n, t0, L, rec_idx)) continue;
        (void)n;
        const int64_t ri = rec_idx * H + h;
        intra_exact_item<PRE, false>(p, sm, t0, L, h, p.rec + ri * kRecBytes,
                                     p.tinv != nullptr ? p.tinv + ri * 320 : nullptr);
    }
    if (count == 0) return;   // the same count in every CTA: nothing to reset
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.exact_ctr + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            p.exact_ctr[0] = 0;
            p.exact_ctr[1] = 0;
            __threadfence();
        }
    }
}

// Validates cu_seqlens and writes each sequence's first chunk index
// (exclusive prefix sum of ceil(len / 2^shift): 16- or 64-token chunks). One
// CTA of 1024 threads.
__global__ void __launch_bounds__(1024)
kda_varlen_prologue_kernel(const int32_t *cu, int32_t n_seqs, int64_t total, int32_t *chunk_off,
                           int *call_flags, int *err, int shift) {
    __shared__ int warp_sums[32];
    __shared__ int s_bad;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) { s_bad = 0; chunk_off[0] = 0; }
    __syncthreads();
    int running = 0;
    for (int base = 0; base < n_seqs; base += 1024) {
        const int i = base + tid;
        int cnt = 0;
        if (i < n_seqs) {
            const int64_t a = cu[i], b = cu[i + 1];
            bool bad = (b < a) || (i == 0 && a != 0) || (i == n_seqs - 1 && b != total);
            if (bad) s_bad = 1;
            else cnt = static_cast<int>((b - a + (int64_t(1) << shift) - 1) >> shift);
        }
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int incl = x + (wid > 0 ? warp_sums[wid - 1] : 0);
        if (i < n_seqs) chunk_off[i + 1] = running + incl;
        running += warp_sums[31];
        __syncthreads();
    }
    if (tid == 0) {
        *call_flags = s_bad ? kErrBadCu : 0;
        if (s_bad) atomicOr(err, kErrBadCu);
    }
}

}  // namespace

cudaError_t launch_varlen_prologue(const int32_t *cu, int32_t n_seqs, int64_t total_tokens,
                                   int32_t *chunk_off, int *call_flags, int *err,
                                   cudaStream_t stream, int chunk_shift) {
    kda_varlen_prologue_kernel<<<1, 1024, 0, stream>>>(cu, n_seqs, total_tokens, chunk_off,
                                                       call_flags, err, chunk_shift);
    return cudaGetLastError();
}

cudaError_t configure_intra() {
    const int smem = kIntraWarps * static_cast<int>(sizeof(IntraWarpSmem));
    cudaError_t e = cudaFuncSetAttribute(kda_intra_chunk_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_intra_chunk_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_intra_chunk_kernel<false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_intra_exact_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kda_intra_exact_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, nb = 0, nbx = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kda_intra_chunk_kernel<false>,
                                                           kIntraWarps * 32, smem)) != cudaSuccess)
        return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nbx, kda_intra_exact_kernel<false>,
                                                           kIntraWarps * 32, smem)) != cudaSuccess)
        return e;
    g_sm_count[dev] = sms;
    g_blocks_per_sm[dev] = nb > 0 ? nb : 1;
    g_exact_blocks_per_sm[dev] = nbx > 0 ? nbx : 1;
    return cudaSuccess;
}

cudaError_t launch_intra_chunk(const IntraParams &p, int64_t max_chunks, cudaStream_t stream) {
    if (max_chunks <= 0) return cudaSuccess;
    const int smem = kIntraWarps * static_cast<int>(sizeof(IntraWarpSmem));
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t items = max_chunks * p.geo.n_heads;
    int64_t blocks = (items + kIntraWarps - 1) / kIntraWarps;
    if (dev >= 0 && dev < kMaxDev && g_sm_count[dev] > 0) {
        const int64_t resident = static_cast<int64_t>(g_sm_count[dev]) * g_blocks_per_sm[dev];
        if (blocks > resident) blocks = resident;
    }
    if (p.pre != 0)
        kda_intra_chunk_kernel<true><<<static_cast<unsigned>(blocks), kIntraWarps * 32, smem,
                                       stream>>>(p, max_chunks);
    else if (p.tinv != nullptr)   // a gradient call (p.wide_flag set too)
        kda_intra_chunk_kernel<false, true><<<static_cast<unsigned>(blocks), kIntraWarps * 32, smem,
                                              stream>>>(p, max_chunks);
    else
        kda_intra_chunk_kernel<false><<<static_cast<unsigned>(blocks), kIntraWarps * 32, smem,
                                        stream>>>(p, max_chunks);
    return cudaGetLastError();
}

cudaError_t launch_intra_exact(const IntraParams &p, cudaStream_t stream) {
    const int smem = kIntraWarps * static_cast<int>(sizeof(IntraWarpSmem));
    int dev = 0;
    cudaGetDevice(&dev);
    // every resident CTA: the list may hold every chunk-head of the call
    int64_t blocks = 1;
    if (dev >= 0 && dev < kMaxDev && g_sm_count[dev] > 0)
        blocks = static_cast<int64_t>(g_sm_count[dev]) * g_exact_blocks_per_sm[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kIntraWarps * 32);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return p.pre != 0 ? cudaLaunchKernelEx(&cfg, kda_intra_exact_kernel<true>, p)
                      : cudaLaunchKernelEx(&cfg, kda_intra_exact_kernel<false>, p);
}

}  // namespace kda
