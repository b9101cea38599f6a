// kda_chunk_prefill_noalloc: the same prefill for callers that may not
// allocate device memory themselves or through this library.
//
// Who needs it: code that runs where cudaMalloc / cudaMallocAsync is not
// allowed or not wanted on the hot path, e.g. a host framework that owns
// every device allocation through its own allocator, a real-time serving
// loop that must never enter the driver's allocator (it may synchronise the
// device or fail under memory pressure), or a plug-in sandbox that forbids
// allocations. Those callers still pass every input and output; the
// scratch that the kernels need between the intra-chunk and the recurrent
// kernel comes from one fixed-size array in device memory that this file
// declares, instead of the per-stream workspace of kda_chunk_prefill.
//
// Costs and limits, stated for the user of this entry point:
//   - Every GPU that loads this library holds kNoAllocScratchBytes (64 MiB)
//     of device memory for that array until the process exits.
//   - A call whose scratch need exceeds that size is rejected with
//     KDA_ERR_SCRATCH_LIMIT before anything is enqueued. The need is what
//     this entry point holds at once: a 256-byte flag block, the chunk-offset
//     table of a packed batch, every chunk record of the call (17,408 B per
//     16-token chunk per head) and one 4-byte exact-form list entry per
//     chunk-head, each part rounded up to 256 bytes (noalloc_scratch_need).
//   - All calls share the one array, so calls whose GPU work overlaps (for
//     example on two streams) race on it and give wrong results; serialise
//     them.
//   - The first call on a device does a one-time set-up with that device
//     current (architecture check, kernel attributes, the array's device
//     address, zeroing its flag block); make that first call before any
//     stream capture. A first call made while its stream is capturing is
//     refused with KDA_ERR_CAPTURE.
//   - Device-side errors of this entry point (bad cu_seqlens contents, a
//     bounded wait that ran out, a log decay rising by more than 80 within a
//     chunk) are recorded in the array's error word; kda_last_device_error()
//     reads and clears it together with the library's own error word.

#include <cuda_runtime.h>

#include <mutex>

#include "kda.h"
#include "kda_device.cuh"
#include "kda_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;

// Layout: [0, 256) flag block (call flags at byte 0, error word at byte 4),
// then the chunk-offset table and the chunk records, as in the workspace of
// kda_chunk_prefill.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_na_mu;
bool g_na_ready[kMaxDevices] = {};
uint8_t *g_na_base[kMaxDevices] = {};

kda_status noalloc_setup(int dev) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (major != 10 || minor != 3) return KDA_ERR_NO_DEVICE_SUPPORT;
    if (kda::configure_intra() != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::configure_recurrent() != cudaSuccess) return KDA_ERR_CUDA;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
        return KDA_ERR_CUDA;
    if (cudaMemset(ptr, 0, 256) != cudaSuccess) return KDA_ERR_CUDA;
    g_na_base[dev] = static_cast<uint8_t *>(ptr);
    g_na_ready[dev] = true;
    return KDA_OK;
}

// Bytes of the fixed array one call needs: flag block, chunk offsets (packed
// batches), all chunk records at once and the exact-form list.
int64_t noalloc_scratch_need(int64_t B, int64_t T, int64_t H, int64_t N, bool packed) {
    const int64_t off = packed ? (((N + 1) * 4 + 255) & ~int64_t(255)) : 0;
    const int64_t chunks = packed ? (T + 15 * N) / 16 : B * ((T + 15) / 16);
    const int64_t list = ((chunks * H * 4) + 255) & ~int64_t(255);
    return 256 + off + chunks * H * kda::kRecBytes + list;
}

bool na_misaligned(const void *p, uintptr_t a) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) != 0;
}

bool na_overlap(const void *a, int64_t na, const void *b, int64_t nb) {
    if (a == nullptr || b == nullptr || na <= 0 || nb <= 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

}  // namespace

bool kda::noalloc_take_error(int dev, int *word) {
    *word = 0;
    if (dev < 0 || dev >= kMaxDevices) return true;
    uint8_t *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_na_mu);
        if (!g_na_ready[dev]) return true;
        base = g_na_base[dev];
    }
    int *err = reinterpret_cast<int *>(base + 4);
    if (cudaMemcpy(word, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return false;
    if (*word != 0 && cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return false;
    return true;
}

extern "C" kda_status kda_chunk_prefill_noalloc(
    const void *q, const void *k, const void *v, const float *g, const float *beta,
    const float *initial_state, const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
    int64_t K, int64_t V, int64_t N, float scale, void *out, float *final_state, void *stream_) {
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_DIM;
    const bool packed = cu_seqlens != nullptr;
    if (kda_workspace_bytes(B, T, H, N, packed ? 1 : 0) <= 0) return KDA_ERR_BAD_SHAPE;
    // this entry point never splits a call into segments: every chunk record
    // of the call is in the array at once
    const int64_t need = noalloc_scratch_need(B, T, H, N, packed);
    if (static_cast<size_t>(need) > kNoAllocScratchBytes) return KDA_ERR_SCRATCH_LIMIT;
    const int64_t tokens = packed ? T : B * T;
    if (tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL_ARG;
    if (na_misaligned(q, 16) || na_misaligned(k, 16) || na_misaligned(v, 16) ||
        na_misaligned(g, 16) || na_misaligned(out, 16) || na_misaligned(initial_state, 16) ||
        na_misaligned(final_state, 16) || na_misaligned(beta, 4) || na_misaligned(cu_seqlens, 4))
        return KDA_ERR_MISALIGNED;
    const int64_t nqkv = tokens * H * 128 * 2, ng = tokens * H * 128 * 4, nb = tokens * H * 4;
    const int64_t ns = N * H * 128 * 128 * 4, ncu = packed ? (N + 1) * 4 : 0;
    const void *ins[] = {q, k, v, g, beta, cu_seqlens};
    const int64_t nins[] = {nqkv, nqkv, nqkv, ng, nb, ncu};
    for (int i = 0; i < 6; ++i)
        if (na_overlap(out, nqkv, ins[i], nins[i]) || na_overlap(final_state, ns, ins[i], nins[i]))
            return KDA_ERR_ALIAS;
    if (na_overlap(out, nqkv, initial_state, ns) || na_overlap(out, nqkv, final_state, ns))
        return KDA_ERR_ALIAS;
    if (final_state != initial_state && na_overlap(final_state, ns, initial_state, ns))
        return KDA_ERR_ALIAS;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return KDA_ERR_CUDA;
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    uint8_t *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_na_mu);
        if (!g_na_ready[dev]) {
            // the set-up makes synchronous calls, which would end a capture
            if (capturing) return KDA_ERR_CAPTURE;
            const kda_status rc = noalloc_setup(dev);
            if (rc != KDA_OK) return rc;
        }
        base = g_na_base[dev];
    }
    // the same device checks as kda_chunk_prefill (they allocate nothing);
    // pointer queries are not stream work, so a capturing call skips them
    if (stream != nullptr && !capturing) {
        int sdev = -1;
        if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return KDA_ERR_CUDA;
        if (sdev != dev) return KDA_ERR_WRONG_DEVICE;
    }
    if (!capturing) {
        const void *ptrs[] = {q, k, v, g, beta, initial_state, cu_seqlens, out, final_state};
        for (const void *ptr : ptrs) {
            const int rc = kda::pointer_device_status(ptr, dev);
            if (rc != KDA_OK) return static_cast<kda_status>(rc);
        }
    }
    const int64_t off_bytes = packed ? (((N + 1) * 4 + 255) & ~int64_t(255)) : 0;
    const int64_t max_chunks = packed ? (T + 15 * N) / 16 : B * ((T + 15) / 16);
    int *call_flags = reinterpret_cast<int *>(base);
    int *err = reinterpret_cast<int *>(base + 4);

    kda::ChunkGeometry geo{};
    geo.cu = cu_seqlens;
    geo.chunk_off = packed ? reinterpret_cast<const int32_t *>(base + 256) : nullptr;
    geo.call_flags = call_flags;
    geo.seq_len = packed ? tokens : T;
    geo.n_seqs = static_cast<int32_t>(N);
    geo.n_heads = static_cast<int32_t>(H);
    geo.chunks_per_seq = static_cast<int32_t>((T + 15) / 16);
    geo.pos_begin = 0;
    geo.seg_len = geo.chunks_per_seq;
    geo.slot_stride = geo.chunks_per_seq;
    if (packed && kda::launch_varlen_prologue(cu_seqlens, geo.n_seqs, tokens,
                                              reinterpret_cast<int32_t *>(base + 256), call_flags,
                                              err, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    uint8_t *rec = base + 256 + off_bytes;
    // the exact-form list after the records, its counters in the flag block
    int32_t *exact_list = reinterpret_cast<int32_t *>(rec + max_chunks * H * kda::kRecBytes);
    int *exact_ctr = reinterpret_cast<int *>(base + 64);
    kda::IntraParams ip{q, k, v, g, beta, rec, scale, 0, err, geo, exact_list, exact_ctr};
    if (kda::launch_intra_chunk(ip, max_chunks, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::launch_intra_exact(ip, stream) != cudaSuccess) return KDA_ERR_CUDA;
    kda::RecurParams rp{rec, initial_state, out, final_state, err, geo};
    if (kda::launch_recurrent(rp, stream) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}
