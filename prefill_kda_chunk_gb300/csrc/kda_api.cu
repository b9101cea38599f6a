// C ABI of the chunked KDA prefill library (declared in include/kda.h):
// argument validation, per-device error word, per-stream workspace, and
// the launch sequence prologue -> intra-chunk kernel -> recurrent kernel.

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <vector>

#include "kda.h"
#include "kda_device.cuh"
#include "kda_internal.h"

namespace {

struct StreamWorkspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};

struct DeviceState {
    bool ready = false;
    int *err = nullptr;  // sticky error word (device memory, 256 B)
    std::map<cudaStream_t, StreamWorkspace> ws;
};

std::mutex g_mu;
std::map<int, DeviceState> g_devices;
struct StageTiming {
    std::vector<cudaEvent_t> ev;  // 3 per call
    int used = 0;
};
thread_local StageTiming t_timing;

constexpr int64_t kMaxElems = int64_t(1) << 40;

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

struct Plan {
    int64_t tokens = 0;      // total tokens
    int64_t max_chunks = 0;  // chunk records needed (upper bound when packed)
    int64_t off_bytes = 0;   // chunk offset table
    int64_t ws_bytes = 0;
};

bool misaligned(const void *p, uintptr_t a) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) != 0;
}

bool overlap(const void *a, int64_t na, const void *b, int64_t nb) {
    if (a == nullptr || b == nullptr || na <= 0 || nb <= 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

kda_status plan_sizes(int64_t B, int64_t T, int64_t H, int64_t N, bool packed, Plan *pl) {
    if (H < 1 || T < 0 || B < 1 || N < 1) return KDA_ERR_BAD_SHAPE;
    if (H > 65535 * 4) return KDA_ERR_BAD_SHAPE;
    if (packed) {
        if (B != 1) return KDA_ERR_BAD_SHAPE;
        if (N > (int64_t(1) << 30)) return KDA_ERR_BAD_SHAPE;
        pl->tokens = T;
        pl->max_chunks = (T + 15 * N) / 16;
    } else {
        if (N != B) return KDA_ERR_BAD_SHAPE;
        if (T > kMaxElems || B > kMaxElems / (T > 0 ? T : 1)) return KDA_ERR_BAD_SHAPE;
        pl->tokens = B * T;
        pl->max_chunks = B * ((T + 15) / 16);
    }
    if (pl->tokens > kMaxElems / (H * kda::kDim)) return KDA_ERR_BAD_SHAPE;
    if (pl->max_chunks >= (int64_t(1) << 31)) return KDA_ERR_BAD_SHAPE;
    if (N * H * 2 >= (int64_t(1) << 31)) return KDA_ERR_BAD_SHAPE;
    pl->off_bytes = packed ? align256((N + 1) * 4) : 0;
    pl->ws_bytes = 256 + pl->off_bytes + pl->max_chunks * H * kda::kRecBytes;
    return KDA_OK;
}

kda_status init_device(int dev, DeviceState &st) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (major != 10 || minor != 3) return KDA_ERR_NO_DEVICE_SUPPORT;
    if (cudaMalloc(&st.err, 256) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaMemset(st.err, 0, 256) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::configure_intra() != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::configure_recurrent() != cudaSuccess) return KDA_ERR_CUDA;
    st.ready = true;
    return KDA_OK;
}

kda_status check_pointer_device(const void *p, int dev) {
    if (p == nullptr) return KDA_OK;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_NOT_DEVICE_MEMORY;
    }
    if (at.type == cudaMemoryTypeManaged) return KDA_OK;
    if (at.type != cudaMemoryTypeDevice) return KDA_ERR_NOT_DEVICE_MEMORY;
    if (at.device != dev) return KDA_ERR_WRONG_DEVICE;
    return KDA_OK;
}

}  // namespace

extern "C" {

const char *kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_NULL_ARG: return "a required pointer is NULL";
        case KDA_ERR_BAD_SHAPE: return "sizes are inconsistent or out of range";
        case KDA_ERR_UNSUPPORTED_DIM: return "only K = V = 128 is supported";
        case KDA_ERR_MISALIGNED: return "a pointer is not aligned as required";
        case KDA_ERR_BAD_CU_SEQLENS: return "cu_seqlens must start at 0, end at T and not decrease";
        case KDA_ERR_CUDA: return "a CUDA runtime call failed";
        case KDA_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel timed out";
        case KDA_ERR_NO_DEVICE_SUPPORT: return "the current device is not sm_103";
        case KDA_ERR_ALIAS: return "an output overlaps an input";
        case KDA_ERR_GATE_RANGE: return "a chunk's cumulative log decay left [-80, 80]";
        case KDA_ERR_CAPTURE: return "workspace cannot grow while the stream is capturing";
        case KDA_ERR_WRONG_DEVICE: return "a buffer or the stream belongs to another device";
        case KDA_ERR_NOT_DEVICE_MEMORY: return "a pointer is not CUDA device memory";
        case KDA_ERR_SCRATCH_LIMIT:
            return "the call needs more scratch than the fixed 64 MiB array of "
                   "kda_chunk_prefill_noalloc";
    }
    return "unknown status";
}

const char *kda_build_info(void) {
    return "prefill_kda_chunk_gb300 0.1 (sm_103a; intra-chunk mma.sync + recurrent mma.sync, "
           "bulk-async staged)";
}

int64_t kda_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t N, int has_cu_seqlens) {
    Plan pl;
    if (plan_sizes(B, T, H, N, has_cu_seqlens != 0, &pl) != KDA_OK) return 0;
    return pl.ws_bytes;
}

kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *initial_state,
                             const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
                             int64_t K, int64_t V, int64_t N, float scale, void *out,
                             float *final_state, void *stream_) {
    // ---- checks that need no GPU
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_DIM;
    Plan pl;
    kda_status rc = plan_sizes(B, T, H, N, cu_seqlens != nullptr, &pl);
    if (rc != KDA_OK) return rc;
    if (pl.tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL_ARG;
    if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(g, 16) ||
        misaligned(out, 16) || misaligned(initial_state, 16) || misaligned(final_state, 16) ||
        misaligned(beta, 4) || misaligned(cu_seqlens, 4))
        return KDA_ERR_MISALIGNED;
    const int64_t nqkv = pl.tokens * H * 128 * 2, ng = pl.tokens * H * 128 * 4;
    const int64_t nb = pl.tokens * H * 4, ns = N * H * 128 * 128 * 4;
    const int64_t ncu = cu_seqlens ? (N + 1) * 4 : 0;
    const void *ins[] = {q, k, v, g, beta, cu_seqlens};
    const int64_t nins[] = {nqkv, nqkv, nqkv, ng, nb, ncu};
    for (int i = 0; i < 6; ++i) {
        if (overlap(out, nqkv, ins[i], nins[i])) return KDA_ERR_ALIAS;
        if (overlap(final_state, ns, ins[i], nins[i])) return KDA_ERR_ALIAS;
    }
    if (overlap(out, nqkv, initial_state, ns) || overlap(out, nqkv, final_state, ns))
        return KDA_ERR_ALIAS;
    if (final_state != initial_state && overlap(final_state, ns, initial_state, ns))
        return KDA_ERR_ALIAS;

    // ---- device checks
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &st = g_devices[dev];
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return KDA_ERR_CUDA;
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    if (!st.ready) {
        if (capturing) return KDA_ERR_CAPTURE;
        rc = init_device(dev, st);
        if (rc != KDA_OK) return rc;
    }
    if (stream != nullptr && !capturing) {
        int sdev = -1;
        if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return KDA_ERR_CUDA;
        if (sdev != dev) return KDA_ERR_WRONG_DEVICE;
    }
    const void *ptrs[] = {q, k, v, g, beta, initial_state, cu_seqlens, out, final_state};
    for (const void *p : ptrs) {
        if (capturing) break;  // pointer queries are not stream work; checked on uncaptured calls
        rc = check_pointer_device(p, dev);
        if (rc != KDA_OK) return rc;
    }

    StreamWorkspace &ws = st.ws[stream];
    if (ws.bytes < static_cast<size_t>(pl.ws_bytes)) {
        if (capturing) return KDA_ERR_CAPTURE;
        if (ws.ptr != nullptr && cudaFreeAsync(ws.ptr, stream) != cudaSuccess) return KDA_ERR_CUDA;
        ws.ptr = nullptr;
        ws.bytes = 0;
        if (cudaMallocAsync(&ws.ptr, pl.ws_bytes, stream) != cudaSuccess) {
            ws.ptr = nullptr;
            return KDA_ERR_CUDA;
        }
        ws.bytes = pl.ws_bytes;
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws.ptr);

    kda::ChunkGeometry geo{};
    geo.cu = cu_seqlens;
    geo.chunk_off = cu_seqlens ? reinterpret_cast<const int32_t *>(wsb + 256) : nullptr;
    geo.call_flags = reinterpret_cast<const int *>(wsb);
    geo.seq_len = cu_seqlens ? pl.tokens : T;
    geo.n_seqs = static_cast<int32_t>(N);
    geo.n_heads = static_cast<int32_t>(H);
    geo.chunks_per_seq = static_cast<int32_t>((T + 15) / 16);

    if (cu_seqlens != nullptr) {
        if (kda::launch_varlen_prologue(cu_seqlens, geo.n_seqs, pl.tokens,
                                        reinterpret_cast<int32_t *>(wsb + 256),
                                        reinterpret_cast<int *>(wsb), st.err, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    uint8_t *rec = wsb + 256 + pl.off_bytes;
    cudaEvent_t *tev = nullptr;
    if (static_cast<size_t>(3 * (t_timing.used + 1)) <= t_timing.ev.size())
        tev = &t_timing.ev[3 * t_timing.used++];
    if (tev && cudaEventRecord(tev[0], stream) != cudaSuccess) return KDA_ERR_CUDA;
    kda::IntraParams ip{q, k, v, g, beta, rec, st.err, geo};
    if (kda::launch_intra_chunk(ip, pl.max_chunks, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (tev && cudaEventRecord(tev[1], stream) != cudaSuccess) return KDA_ERR_CUDA;
    kda::RecurParams rp{rec, initial_state, out, final_state, scale, st.err, geo};
    if (kda::launch_recurrent(rp, stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (tev && cudaEventRecord(tev[2], stream) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

static void free_timing() {
    for (cudaEvent_t e : t_timing.ev) cudaEventDestroy(e);
    t_timing.ev.clear();
    t_timing.used = 0;
}

kda_status kda_stage_timing_begin(int max_calls) {
    if (max_calls < 1) return KDA_ERR_BAD_SHAPE;
    free_timing();
    t_timing.ev.resize(3 * static_cast<size_t>(max_calls), nullptr);
    for (auto &e : t_timing.ev)
        if (cudaEventCreate(&e) != cudaSuccess) {
            e = nullptr;
            free_timing();
            return KDA_ERR_CUDA;
        }
    return KDA_OK;
}

kda_status kda_stage_timing_end(double *intra_ms, double *recurrent_ms, int *calls) {
    const int n = t_timing.used;
    double a = 0.0, b = 0.0;
    kda_status rc = KDA_OK;
    if (n > 0 && cudaEventSynchronize(t_timing.ev[3 * n - 1]) != cudaSuccess) rc = KDA_ERR_CUDA;
    for (int i = 0; i < n && rc == KDA_OK; ++i) {
        float x = 0.f, y = 0.f;
        if (cudaEventElapsedTime(&x, t_timing.ev[3 * i], t_timing.ev[3 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&y, t_timing.ev[3 * i + 1], t_timing.ev[3 * i + 2]) != cudaSuccess)
            rc = KDA_ERR_CUDA;
        a += x;
        b += y;
    }
    free_timing();
    if (rc != KDA_OK) return rc;
    if (intra_ms) *intra_ms = n ? a / n : 0.0;
    if (recurrent_ms) *recurrent_ms = n ? b / n : 0.0;
    if (calls) *calls = n;
    return KDA_OK;
}

kda_status kda_last_device_error(void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
    int *err = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_devices.find(dev);
        if (it == g_devices.end() || !it->second.ready) return KDA_OK;
        err = it->second.err;
    }
    int word = 0;
    if (cudaMemcpy(&word, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
    if (word != 0 && cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    if (word & kda::kErrBadCu) return KDA_ERR_BAD_CU_SEQLENS;
    if (word & kda::kErrTimeout) return KDA_ERR_DEVICE_TIMEOUT;
    if (word & kda::kErrGate) return KDA_ERR_GATE_RANGE;
    return KDA_OK;
}

kda_status kda_workspace_release(void) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_devices.find(dev);
    if (it == g_devices.end()) return KDA_OK;
    for (auto &kv : it->second.ws)
        if (kv.second.ptr != nullptr && cudaFree(kv.second.ptr) != cudaSuccess) return KDA_ERR_CUDA;
    it->second.ws.clear();
    return KDA_OK;
}

}  // extern "C"
