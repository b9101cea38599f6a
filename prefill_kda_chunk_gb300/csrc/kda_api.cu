// C ABI of the chunked KDA prefill library (declared in include/kda.h):
// argument validation, per-device error word, per-stream workspace, and
// the launch sequence prologue -> intra-chunk kernel -> recurrent kernel.

#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <vector>

#include "kda.h"
#include "kda_device.cuh"
#include "kda_internal.h"

namespace {

// Per caller stream: the scratch buffer.
struct StreamWorkspace {
    void *ptr = nullptr;
    size_t bytes = 0;
    // bytes at offset 256 known to hold zeros for the fused launch's ring
    // counters (a fused launch leaves its own counters zero and writes past
    // them; any other use of the buffer may overwrite them)
    int64_t ring_clean = 0;
};

struct DeviceState {
    bool ready = false;
    int *err = nullptr;  // sticky error word (device memory, 256 B)
    std::map<cudaStream_t, StreamWorkspace> ws;
};

std::mutex g_mu;
std::map<int, DeviceState> g_devices;
// Measurement hook state (per host thread): event pairs around every launch
// of the two kernels during the timed calls.
struct StageTiming {
    int max_calls = 0, calls = 0;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> intra, recur;
};
thread_local StageTiming t_timing;

// Path: 1 = 16-token chunks (intra-chunk kernel, then the warp-MMA recurrent
// kernel); 3 = 64-token chunks on tcgen05, intra-chunk kernel then recurrent
// kernel; 4 = 64-token chunks, both in one cooperative launch with the
// records in an L2-resident ring (3 when the heads leave too few SMs for the
// record builders).
std::atomic<int> g_recur_impl{1};
constexpr int kImplC16 = 1, kImplC64Split = 3, kImplC64Fused = 4;
constexpr int64_t kC64Ring = 4;          // ring slots per head (fused launch)
constexpr int kC64MinBuilders = 16;      // SMs left for record builders in a fused launch

constexpr int64_t kMaxElems = int64_t(1) << 40;

// Segment-parallel scan (fixed-length calls, 16-token path). A recurrent
// step is a serial chain, so with few (sequence, head) units most SMs idle
// through T/16 steps. Cutting every sequence into P segments, the maps launch
// builds each segment's affine state map (M, c) in parallel (the first
// segment's end state directly), a short serial combine gives the entry
// states, and one launch replays all segments side by side: about
// (P - 1)/P light + 1/P full chain lengths instead of one full one.
// A CTA's chain step costs about the same SM time whether it runs alone on an
// SM or beside others (T=131072, H=32 on GB300: 1.1 k cycles alone, 2.7 k
// with 2.5 CTAs per SM), so the scan pays only while the plain chains (2 N H
// CTAs) leave more than half of the SMs idle; then P fills about three replay
// CTAs per SM (measured there: P = 1, 2, 6, 8 -> 4.25, 3.78, 3.36, 3.42 ms).
// kda_set_scan_segments forces P.
constexpr int64_t kScanMinChunks = 64;     // per sequence
constexpr int64_t kScanMinSegChunks = 16;  // per segment
constexpr int64_t kScanMaxSegs = 16;
constexpr int64_t kScanSpareSms = 4;
std::atomic<int> g_scan_segs{0};           // 0: automatic, 1: off, >= 2: forced
std::atomic<int> g_bwd_impl{0};            // gradients: 0 chunked, 1 token-serial
// test hook of the recurrent kernel (kda_test_stall_recurrent)
std::atomic<int> g_stall_chunk{-1};
std::atomic<long long> g_stall_wait_ns{0};

int64_t scan_segments(int64_t NH, int64_t cps, int sm_count) {
    const int forced = g_scan_segs.load();
    int64_t P;
    if (forced == 1) return 1;
    if (forced >= 2) {
        P = forced;
    } else {
        if (cps < kScanMinChunks || 4 * NH > sm_count - kScanSpareSms) return 1;
        P = 3 * (sm_count - kScanSpareSms) / (2 * NH);
        if (P > kScanMaxSegs) P = kScanMaxSegs;
        if (P > cps / kScanMinSegChunks) P = cps / kScanMinSegChunks;
    }
    if (P > cps) P = cps;
    return P >= 2 ? P : 1;
}

// SM count of the current device; the sizing-only entry point kda_workspace_bytes
// may run without a device, and then sizes for GB300's 152 SMs.
int current_sm_count() {
    int dev = -1, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0) {
        cudaGetLastError();
        return 152;
    }
    return sms;
}

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

struct Plan {
    int impl = 1;            // recurrent kernel / path actually used (see g_recur_impl)
    int64_t c64_chunks = 0;  // 64-token paths: chunks of the call (upper bound when packed)
    int64_t c64_sync = 0;    // fused 64-token path: bytes of the ring counters after the flag block
    int64_t tokens = 0;      // total tokens
    int64_t max_chunks = 0;  // chunk records of one launch (upper bound when packed)
    int64_t off_bytes = 0;   // chunk offset table
    int64_t ws_bytes = 0;
    int64_t seg_len = 0;     // fixed-length: chunks per sequence
    // Segment-parallel scan of fixed-length sequences (see kScan*): scan_segs
    // segments of scan_len chunks; scan_bytes of entry states (P - 1), offsets
    // and maps (P - 2 each): planes of N H 128 x 128 fp32 after the records.
    int64_t scan_segs = 1;
    int64_t scan_len = 0;
    int64_t scan_bytes = 0;
    // list of chunk-heads for the exact form (one int32 per item of a launch)
    // at the end of the workspace; its two counters sit in the flag block
    int64_t list_bytes = 0;
};

// flag block (the first 256 bytes of a workspace): per-call flag word at 0,
// the exact-form list counters at kExactCtrOff
constexpr int64_t kExactCtrOff = 64;
// ... and, in a gradient call, the out-of-range flag and the gradient kernel's
// finish count at kWideOff (both reset by that kernel)
constexpr int64_t kWideOff = 128;

bool misaligned(const void *p, uintptr_t a) {
    return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) != 0;
}

bool overlap(const void *a, int64_t na, const void *b, int64_t nb) {
    if (a == nullptr || b == nullptr || na <= 0 || nb <= 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

kda_status plan_sizes(int64_t B, int64_t T, int64_t H, int64_t N, bool packed, int sm_count,
                      int impl, Plan *pl) {
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
    pl->seg_len = (T + 15) / 16;
    if (!packed) {
        pl->scan_segs = scan_segments(N * H, pl->seg_len, sm_count);
        if (pl->scan_segs >= 2) {
            pl->scan_len = (pl->seg_len + pl->scan_segs - 1) / pl->scan_segs;
            pl->scan_segs = (pl->seg_len + pl->scan_len - 1) / pl->scan_len;   // none empty
        }
        if (pl->scan_segs >= 2) {
            pl->scan_bytes = (3 * pl->scan_segs - 5) * align256(N * H * 128 * 128 * 4);
            pl->ws_bytes += pl->scan_bytes;
        }
    }
    pl->list_bytes = align256(pl->max_chunks * H * 4);
    pl->ws_bytes += pl->list_bytes;
    pl->impl = impl;
    if (impl >= kImplC64Split) {
        // 64-token chunks: flag block, 64-token chunk offsets (packed), then the
        // records of every chunk-head (split) or a ring of kC64Ring per head and
        // its counters (fused). TMA coordinates are 32-bit.
        if (pl->tokens >= (int64_t(1) << 31)) return KDA_ERR_BAD_SHAPE;
        pl->c64_chunks = packed ? (T + 63 * N) / 64 : B * ((T + 63) / 64);
        if (impl == kImplC64Fused && H + kC64MinBuilders > sm_count) pl->impl = kImplC64Split;
        pl->scan_segs = 1;
        pl->scan_bytes = 0;
        pl->list_bytes = 0;
        if (pl->impl == kImplC64Split) {
            pl->ws_bytes = 256 + pl->off_bytes + pl->c64_chunks * H * kda::kC64RecBytes;
        } else {
            // the ring counters sit right after the flag block, whatever H is
            pl->c64_sync = align256((kC64Ring * H + H) * 8 + 64);
            pl->ws_bytes = 256 + pl->c64_sync + pl->off_bytes + kC64Ring * H * kda::kC64RecBytes;
        }
    }
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
    if (kda::configure_c64() != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::configure_backward_chunk() != cudaSuccess) return KDA_ERR_CUDA;
    st.ready = true;
    return KDA_OK;
}

kda_status check_pointer_device(const void *p, int dev) {
    return static_cast<kda_status>(kda::pointer_device_status(p, dev));
}

}  // namespace

int kda::pointer_device_status(const void *p, int dev) {
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
        case KDA_ERR_GATE_RANGE: return "log decay rose by more than 80 within a chunk (exp leaves fp32)";
        case KDA_ERR_CAPTURE: return "workspace cannot grow while the stream is capturing";
        case KDA_ERR_WRONG_DEVICE: return "a buffer or the stream belongs to another device";
        case KDA_ERR_NOT_DEVICE_MEMORY: return "a pointer is not CUDA device memory";
        case KDA_ERR_SCRATCH_LIMIT:
            return "the call needs more scratch than the fixed 64 MiB array of "
                   "kda_chunk_prefill_noalloc";
        case KDA_ERR_BAD_FLAGS: return "an unknown preprocessing flag bit is set";
    }
    return "unknown status";
}

kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const float *state_in, float *state_out, int64_t N,
                           int64_t H, int64_t K, int64_t V, float scale, int flags, void *out,
                           void *stream_) {
    // ---- checks that need no GPU
    if ((flags & ~(KDA_PRE_NORM_QK | KDA_PRE_GATE_LOGITS)) != 0) return KDA_ERR_BAD_FLAGS;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_DIM;
    if (N < 0 || H < 1 || H > (int64_t(1) << 24) || N > ((int64_t(1) << 31) - 1) / H)
        return KDA_ERR_BAD_SHAPE;
    const int64_t units = N * H;
    if (units > 0 && (!q || !k || !v || !g || !beta || !out || !state_out))
        return KDA_ERR_NULL_ARG;
    if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(g, 16) ||
        misaligned(out, 16) || misaligned(state_in, 16) || misaligned(state_out, 16) ||
        misaligned(beta, 4))
        return KDA_ERR_MISALIGNED;
    const int64_t nqkv = units * 128 * 2, ng = units * 128 * 4, nb = units * 4;
    const int64_t ns = units * 128 * 128 * 4;
    const void *ins[] = {q, k, v, g, beta};
    const int64_t nins[] = {nqkv, nqkv, nqkv, ng, nb};
    for (int i = 0; i < 5; ++i) {
        if (overlap(out, nqkv, ins[i], nins[i])) return KDA_ERR_ALIAS;
        if (overlap(state_out, ns, ins[i], nins[i])) return KDA_ERR_ALIAS;
    }
    if (overlap(out, nqkv, state_in, ns) || overlap(out, nqkv, state_out, ns))
        return KDA_ERR_ALIAS;
    if (state_out != state_in && overlap(state_out, ns, state_in, ns)) return KDA_ERR_ALIAS;
    if (units == 0) return KDA_OK;   // an empty batch enqueues nothing

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
        const kda_status rc = init_device(dev, st);
        if (rc != KDA_OK) return rc;
    }
    if (stream != nullptr && !capturing) {
        int sdev = -1;
        if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return KDA_ERR_CUDA;
        if (sdev != dev) return KDA_ERR_WRONG_DEVICE;
    }
    const void *ptrs[] = {q, k, v, g, beta, state_in, state_out, out};
    for (const void *ptr : ptrs) {
        if (capturing) break;  // pointer queries are not stream work
        const kda_status rc = check_pointer_device(ptr, dev);
        if (rc != KDA_OK) return rc;
    }
    const kda::DecodeParams p{q, k, v, g, beta, state_in, state_out, out, scale, flags};
    return kda::launch_decode(p, units, stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

const char *kda_build_info(void) {
    return "prefill_kda_chunk_gb300 0.4 (sm_103a; 16-token chunks: intra-chunk mma.sync with an "
           "exact form for strong decay, recurrent warp-MMA chain with bulk-async staged records "
           "and a segment-parallel scan for long sequences; 64-token chunks on tcgen05 opt-in; decode step; in-kernel q/k "
           "normalisation and gate logits; token-serial gradients)";
}

int64_t kda_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t N, int has_cu_seqlens) {
    Plan pl;
    if (plan_sizes(B, T, H, N, has_cu_seqlens != 0, current_sm_count(), g_recur_impl.load(), &pl) !=
        KDA_OK)
        return 0;
    return pl.ws_bytes;
}

kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *initial_state,
                             const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
                             int64_t K, int64_t V, int64_t N, float scale, void *out,
                             float *final_state, void *stream) {
    return kda_chunk_prefill_ex(q, k, v, g, beta, initial_state, cu_seqlens, B, T, H, K, V, N,
                                scale, 0, out, final_state, stream);
}

kda_status kda_chunk_prefill_ex(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, const float *initial_state,
                                const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H,
                                int64_t K, int64_t V, int64_t N, float scale, int flags,
                                void *out, float *final_state, void *stream_) {
    // ---- checks that need no GPU
    if ((flags & ~(KDA_PRE_NORM_QK | KDA_PRE_GATE_LOGITS)) != 0) return KDA_ERR_BAD_FLAGS;
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_DIM;
    // one read of the kernel choice per call: the record layout depends on it
    const int impl = g_recur_impl.load();
    Plan pl;
    const int sm_count = current_sm_count();
    kda_status rc = plan_sizes(B, T, H, N, cu_seqlens != nullptr, sm_count, impl, &pl);
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
        ws.ring_clean = 0;
        // the flag block starts zeroed (the exact-form list counters above all)
        if (cudaMemsetAsync(ws.ptr, 0, 256, stream) != cudaSuccess) return KDA_ERR_CUDA;
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws.ptr);

    const bool timed = t_timing.calls < t_timing.max_calls;
    if (timed) ++t_timing.calls;
    auto timed_launch = [&](bool intra, cudaStream_t s, auto &&launch) -> kda_status {
        cudaEvent_t e0 = nullptr, e1 = nullptr;
        if (timed) {
            if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
                return KDA_ERR_CUDA;
            (intra ? t_timing.intra : t_timing.recur).emplace_back(e0, e1);
            if (cudaEventRecord(e0, s) != cudaSuccess) return KDA_ERR_CUDA;
        }
        if (launch() != cudaSuccess) return KDA_ERR_CUDA;
        if (timed && cudaEventRecord(e1, s) != cudaSuccess) return KDA_ERR_CUDA;
        return KDA_OK;
    };

    if (pl.impl >= kImplC64Split) {
        // ---- 64-token chunks on tcgen05
        const bool fused = pl.impl == kImplC64Fused;
        if (!fused) ws.ring_clean = 0;
        // fused: [flags | ring counters | chunk offsets | ring]; split: [flags | offsets | records]
        const int64_t off_at = 256 + (fused ? pl.c64_sync : 0);
        if (cu_seqlens != nullptr &&
            kda::launch_varlen_prologue(cu_seqlens, static_cast<int32_t>(N), pl.tokens,
                                        reinterpret_cast<int32_t *>(wsb + off_at),
                                        reinterpret_cast<int *>(wsb), st.err, stream,
                                        6) != cudaSuccess)
            return KDA_ERR_CUDA;
        kda::C64Args a{};
        a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.s0 = initial_state;
        a.out = out; a.s_final = final_state;
        a.cu = cu_seqlens;
        a.chunk_off = cu_seqlens ? reinterpret_cast<const int32_t *>(wsb + off_at) : nullptr;
        a.call_flags = reinterpret_cast<const int *>(wsb);
        a.err = st.err;
        a.tokens = pl.tokens;
        a.seq_len = cu_seqlens ? pl.tokens : T;
        a.max_chunks = pl.c64_chunks;
        a.n_seqs = static_cast<int32_t>(N);
        a.n_heads = static_cast<int32_t>(H);
        a.cps = static_cast<int32_t>((T + 63) / 64);
        a.scale = scale;
        a.pre = flags;
        a.rec = wsb + off_at + pl.off_bytes;
        if (!fused) {
            rc = timed_launch(true, stream, [&] { return kda::launch_c64_intra(a, sm_count, stream); });
            if (rc != KDA_OK) return rc;
            return timed_launch(false, stream, [&] { return kda::launch_c64_chain(a, stream); });
        }
        if (pl.tokens == 0)   // nothing for the builders: the chains alone carry the states
            return timed_launch(false, stream, [&] { return kda::launch_c64_chain(a, stream); });
        long long *sync = reinterpret_cast<long long *>(wsb + 256);
        if (ws.ring_clean < pl.c64_sync &&
            cudaMemsetAsync(sync, 0, pl.c64_sync, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        // the launch leaves its own counters zero again; what lies past them
        // (chunk offsets, ring) is not, whatever a larger layout needs there
        ws.ring_clean = pl.c64_sync;
        a.ring_depth = static_cast<int>(kC64Ring);
        a.n_chain = static_cast<int>(H);
        a.ready = sync;
        a.consumed = sync + kC64Ring * H;
        a.exit_ctr = reinterpret_cast<int *>(sync + kC64Ring * H + H);
        return timed_launch(false, stream, [&] { return kda::launch_c64_fused(a, sm_count, stream); });
    }
    ws.ring_clean = 0;

    kda::ChunkGeometry geo{};
    geo.cu = cu_seqlens;
    geo.chunk_off = cu_seqlens ? reinterpret_cast<const int32_t *>(wsb + 256) : nullptr;
    geo.call_flags = reinterpret_cast<const int *>(wsb);
    geo.seq_len = cu_seqlens ? pl.tokens : T;
    geo.n_seqs = static_cast<int32_t>(N);
    geo.n_heads = static_cast<int32_t>(H);
    geo.chunks_per_seq = static_cast<int32_t>((T + 15) / 16);
    geo.pos_begin = 0;
    geo.seg_len = geo.chunks_per_seq;
    geo.slot_stride = geo.chunks_per_seq;

    if (cu_seqlens != nullptr) {
        if (kda::launch_varlen_prologue(cu_seqlens, geo.n_seqs, pl.tokens,
                                        reinterpret_cast<int32_t *>(wsb + 256),
                                        reinterpret_cast<int *>(wsb), st.err, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    uint8_t *rec = wsb + 256 + pl.off_bytes;
    int32_t *exact_list = reinterpret_cast<int32_t *>(wsb + pl.ws_bytes - pl.list_bytes);
    int *exact_ctr = reinterpret_cast<int *>(wsb + kExactCtrOff);
    // the intra-chunk kernel, then the exact form of what it listed
    auto intra = [&](const kda::IntraParams &ip, int64_t items, cudaStream_t s) {
        const cudaError_t e = kda::launch_intra_chunk(ip, items, s);
        return e != cudaSuccess ? e : kda::launch_intra_exact(ip, s);
    };

    kda::IntraParams ip{q, k, v, g, beta, rec, scale, flags, st.err, geo, exact_list, exact_ctr};
    rc = timed_launch(true, stream, [&] { return intra(ip, pl.max_chunks, stream); });
    if (rc != KDA_OK) return rc;
    kda::RecurParams rp{rec, initial_state, out, final_state, st.err, geo};
    rp.stall_chunk = g_stall_chunk.load();
    rp.wait_ns = static_cast<unsigned long long>(g_stall_wait_ns.load());
    // (an in-place state would be read by the first segment while the last
    // one writes it)
    if (pl.scan_segs >= 2 && (initial_state == nullptr || initial_state != final_state)) {
        // segment maps, their serial combine, then every segment at once
        const int64_t plane = align256(N * H * 128 * 128 * 4);
        uint8_t *sc = rec + pl.max_chunks * H * kda::kRecBytes;
        rp.scan_segs = static_cast<int32_t>(pl.scan_segs);
        rp.scan_len = static_cast<int32_t>(pl.scan_len);
        rp.seg_entry = reinterpret_cast<float *>(sc);
        rp.seg_c = reinterpret_cast<float *>(sc + (pl.scan_segs - 1) * plane);
        rp.seg_m = reinterpret_cast<float *>(sc + (2 * pl.scan_segs - 3) * plane);
        return timed_launch(false, stream, [&] {
            cudaError_t e = kda::launch_recurrent_scan_maps(rp, stream);
            if (e == cudaSuccess) e = kda::launch_scan_combine(rp, stream);
            return e != cudaSuccess ? e : kda::launch_recurrent(rp, stream);
        });
    }
    return timed_launch(false, stream, [&] { return kda::launch_recurrent(rp, stream); });
}

// Gradient workspace: flag block, chunk offsets (packed), one checkpoint state
// per 16 tokens per head, and a ring of 16 states per CTA of the persistent
// gradient kernel (at most kBackwardMaxRings).
static int64_t backward_ckpt_bytes(int64_t B, int64_t T, int64_t H, int64_t N, bool packed,
                                   const Plan &pl) {
    const int64_t chunks = packed ? (pl.tokens + 15 * N) / 16 : B * ((T + 15) / 16);
    return chunks * H * 128 * 128 * 4;
}

// Chunked gradients: flag block, chunk offsets (packed), the records, the
// exact-form list, (I + A)^{-1} of every chunk-head (fp32), then S^T and
// dS_next^T of every chunk-head in bf16.
static int64_t backward_chunk_ws_bytes(int64_t H, const Plan &pl) {
    const int64_t ch = pl.max_chunks * H;
    return 256 + pl.off_bytes + ch * kda::kRecBytes + align256(ch * 4) + ch * 1280 +
           2 * ch * kda::kDim * kda::kDim * 2;
}

static int64_t backward_ws_bytes(int64_t B, int64_t T, int64_t H, int64_t N, bool packed,
                                 const Plan &pl) {
    if (g_bwd_impl.load() == 0) return backward_chunk_ws_bytes(H, pl);
    const int64_t rings = N * H < kda::kBackwardMaxRings ? N * H : kda::kBackwardMaxRings;
    return 256 + pl.off_bytes + backward_ckpt_bytes(B, T, H, N, packed, pl) +
           rings * 16 * 128 * 128 * 4;
}

int64_t kda_backward_workspace_bytes(int64_t B, int64_t T, int64_t H, int64_t N,
                                     int has_cu_seqlens) {
    Plan pl;
    if (plan_sizes(B, T, H, N, has_cu_seqlens != 0, current_sm_count(), 1, &pl) != KDA_OK) return 0;
    if (N * H > (int64_t(1) << 31) - 1) return 0;
    return backward_ws_bytes(B, T, H, N, has_cu_seqlens != 0, pl);
}

kda_status kda_chunk_prefill_backward(const void *q, const void *k, const void *v,
                                      const float *g, const float *beta,
                                      const float *initial_state, const int32_t *cu_seqlens,
                                      int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                                      int64_t N, float scale, const void *d_out,
                                      const float *d_final_state, float *dq, float *dk,
                                      float *dv, float *dg, float *dbeta,
                                      float *d_initial_state, void *stream_) {
    // ---- checks that need no GPU
    if (K != 128 || V != 128) return KDA_ERR_UNSUPPORTED_DIM;
    Plan pl;
    kda_status rc = plan_sizes(B, T, H, N, cu_seqlens != nullptr, current_sm_count(), 1, &pl);
    if (rc != KDA_OK) return rc;
    if (N * H > (int64_t(1) << 31) - 1) return KDA_ERR_BAD_SHAPE;
    if (pl.tokens > 0 && (!q || !k || !v || !g || !beta || !d_out || !dq || !dk || !dv || !dg ||
                          !dbeta))
        return KDA_ERR_NULL_ARG;
    if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(g, 16) ||
        misaligned(d_out, 16) || misaligned(initial_state, 16) ||
        misaligned(d_final_state, 16) || misaligned(dq, 16) || misaligned(dk, 16) ||
        misaligned(dv, 16) || misaligned(dg, 16) || misaligned(d_initial_state, 16) ||
        misaligned(beta, 4) || misaligned(dbeta, 4) || misaligned(cu_seqlens, 4))
        return KDA_ERR_MISALIGNED;
    const int64_t nqkv = pl.tokens * H * 128 * 2, nf = pl.tokens * H * 128 * 4;
    const int64_t nb = pl.tokens * H * 4, ns = N * H * 128 * 128 * 4;
    const int64_t ncu = cu_seqlens ? (N + 1) * 4 : 0;
    const void *ins[] = {q, k, v, g, beta, initial_state, cu_seqlens, d_out, d_final_state};
    const int64_t nins[] = {nqkv, nqkv, nqkv, nf, nb, ns, ncu, nqkv, ns};
    void *outs[] = {dq, dk, dv, dg, dbeta, d_initial_state};
    const int64_t nouts[] = {nf, nf, nf, nf, nb, ns};
    for (int o = 0; o < 6; ++o) {
        for (int i = 0; i < 9; ++i)
            if (overlap(outs[o], nouts[o], ins[i], nins[i])) return KDA_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 6; ++o2)
            if (overlap(outs[o], nouts[o], outs[o2], nouts[o2])) return KDA_ERR_ALIAS;
    }

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
    const void *ptrs[] = {q, k, v, g, beta, initial_state, cu_seqlens, d_out, d_final_state,
                          dq, dk, dv, dg, dbeta, d_initial_state};
    for (const void *p : ptrs) {
        if (capturing) break;  // pointer queries are not stream work
        rc = check_pointer_device(p, dev);
        if (rc != KDA_OK) return rc;
    }

    const int64_t ckpt_bytes = backward_ckpt_bytes(B, T, H, N, cu_seqlens != nullptr, pl);
    const int64_t need = backward_ws_bytes(B, T, H, N, cu_seqlens != nullptr, pl);
    StreamWorkspace &ws = st.ws[stream];
    if (ws.bytes < static_cast<size_t>(need)) {
        if (capturing) return KDA_ERR_CAPTURE;
        if (ws.ptr != nullptr && cudaFreeAsync(ws.ptr, stream) != cudaSuccess) return KDA_ERR_CUDA;
        ws.ptr = nullptr;
        ws.bytes = 0;
        if (cudaMallocAsync(&ws.ptr, need, stream) != cudaSuccess) {
            ws.ptr = nullptr;
            return KDA_ERR_CUDA;
        }
        ws.bytes = need;
        if (cudaMemsetAsync(ws.ptr, 0, 256, stream) != cudaSuccess) return KDA_ERR_CUDA;
    }
    uint8_t *wsb = static_cast<uint8_t *>(ws.ptr);
    ws.ring_clean = 0;   // this call overwrites the area of the 64-token ring counters

    kda::ChunkGeometry geo{};
    geo.cu = cu_seqlens;
    geo.chunk_off = cu_seqlens ? reinterpret_cast<const int32_t *>(wsb + 256) : nullptr;
    geo.call_flags = reinterpret_cast<const int *>(wsb);
    geo.seq_len = cu_seqlens ? pl.tokens : T;
    geo.n_seqs = static_cast<int32_t>(N);
    geo.n_heads = static_cast<int32_t>(H);
    geo.chunks_per_seq = static_cast<int32_t>((T + 15) / 16);
    geo.pos_begin = 0;
    geo.seg_len = geo.chunks_per_seq;
    geo.slot_stride = geo.chunks_per_seq;
    if (cu_seqlens != nullptr &&
        kda::launch_varlen_prologue(cu_seqlens, geo.n_seqs, pl.tokens,
                                    reinterpret_cast<int32_t *>(wsb + 256),
                                    reinterpret_cast<int *>(wsb), st.err, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (g_bwd_impl.load() == 0) {
        // chunked: records, the forward chain keeping chunk-entry states, the
        // reverse chain keeping dS_next, then the chunk-parallel gradients
        if (pl.tokens == 0) {
            // no chunks: dL/d(initial state) = dL/d(final state)
            if (d_initial_state != nullptr) {
                const size_t ns = static_cast<size_t>(N * H) * 128 * 128 * 4;
                const cudaError_t e = d_final_state != nullptr
                    ? cudaMemcpyAsync(d_initial_state, d_final_state, ns, cudaMemcpyDeviceToDevice, stream)
                    : cudaMemsetAsync(d_initial_state, 0, ns, stream);
                if (e != cudaSuccess) return KDA_ERR_CUDA;
            }
            return KDA_OK;
        }
        const int64_t ch = pl.max_chunks * H;
        uint8_t *rec = wsb + 256 + pl.off_bytes;
        int32_t *exact_list = reinterpret_cast<int32_t *>(rec + ch * kda::kRecBytes);
        float *tinv = reinterpret_cast<float *>(rec + ch * kda::kRecBytes + align256(ch * 4));
        uint8_t *ck = reinterpret_cast<uint8_t *>(tinv + ch * 320);
        uint8_t *dsn = ck + ch * kda::kDim * kda::kDim * 2;
        int *exact_ctr = reinterpret_cast<int *>(wsb + kExactCtrOff);
        int *wide = reinterpret_cast<int *>(wsb + kWideOff);
        const kda::IntraParams ip{q, k, v, g, beta, rec, scale, 0, st.err, geo, exact_list, exact_ctr, tinv, wide};
        if (kda::launch_intra_chunk(ip, pl.max_chunks, stream) != cudaSuccess ||
            kda::launch_intra_exact(ip, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        kda::BwdChunkParams bp{};
        bp.ip = ip;
        bp.rec = rec;
        bp.s0 = initial_state;
        bp.dout = d_out;
        bp.dsf = d_final_state;
        bp.ds0 = d_initial_state;
        bp.ckpt = ck;
        bp.dsn = dsn;
        bp.dq = dq; bp.dk = dk; bp.dv = dv; bp.dg = dg; bp.dbeta = dbeta;
        bp.err = st.err;
        bp.geo = geo;
        bp.max_chunks = pl.max_chunks;
        bp.wide = wide;
        if (kda::launch_bwd_chains(bp, stream) != cudaSuccess) return KDA_ERR_CUDA;
        return kda::launch_bwd_grad(bp, stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    float *ckpt = reinterpret_cast<float *>(wsb + 256 + pl.off_bytes);
    float *ring = reinterpret_cast<float *>(wsb + 256 + pl.off_bytes + ckpt_bytes);
    const kda::BackParams p{q, k, v, g, beta, initial_state, d_out, d_final_state, scale,
                            dq, dk, dv, dg, dbeta, d_initial_state, ckpt, ring, geo};
    return kda::launch_backward(p, N * H, stream) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_set_backward_impl(int impl) {
    if (impl != 0 && impl != 1) return KDA_ERR_BAD_SHAPE;
    g_bwd_impl.store(impl);
    return KDA_OK;
}

static void free_timing() {
    for (auto *v : {&t_timing.intra, &t_timing.recur}) {
        for (auto &pr : *v) {
            if (pr.first) cudaEventDestroy(pr.first);
            if (pr.second) cudaEventDestroy(pr.second);
        }
        v->clear();
    }
    t_timing.max_calls = t_timing.calls = 0;
}

kda_status kda_stage_timing_begin(int max_calls) {
    if (max_calls < 1) return KDA_ERR_BAD_SHAPE;
    free_timing();
    t_timing.max_calls = max_calls;
    return KDA_OK;
}

kda_status kda_stage_timing_end(double *intra_ms, double *recurrent_ms, int *calls) {
    const int n = t_timing.calls;
    double sum[2] = {0.0, 0.0};
    kda_status rc = KDA_OK;
    int which = 0;
    for (auto *v : {&t_timing.intra, &t_timing.recur}) {
        for (auto &pr : *v) {
            float ms = 0.f;
            if (cudaEventSynchronize(pr.second) != cudaSuccess ||
                cudaEventElapsedTime(&ms, pr.first, pr.second) != cudaSuccess) {
                rc = KDA_ERR_CUDA;
                break;
            }
            sum[which] += ms;
        }
        ++which;
    }
    free_timing();
    if (rc != KDA_OK) return rc;
    if (intra_ms) *intra_ms = n ? sum[0] / n : 0.0;
    if (recurrent_ms) *recurrent_ms = n ? sum[1] / n : 0.0;
    if (calls) *calls = n;
    return KDA_OK;
}

kda_status kda_test_stall_recurrent(int chunk, int64_t wait_ns) {
    if (chunk < -1 || wait_ns < 0) return KDA_ERR_BAD_SHAPE;
    g_stall_chunk.store(chunk);
    g_stall_wait_ns.store(chunk < 0 ? 0 : wait_ns);
    return KDA_OK;
}

kda_status kda_set_scan_segments(int segments) {
    if (segments < 0 || segments > 4096) return KDA_ERR_BAD_SHAPE;
    g_scan_segs.store(segments);
    return KDA_OK;
}

kda_status kda_set_recurrent_impl(int impl) {
    if (impl != kImplC16 && impl != kImplC64Split && impl != kImplC64Fused) return KDA_ERR_BAD_SHAPE;
    g_recur_impl.store(impl);
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
        if (it != g_devices.end() && it->second.ready) err = it->second.err;
    }
    int word = 0;
    if (err != nullptr) {
        if (cudaMemcpy(&word, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (word != 0 && cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    }
    // the allocation-free entry point records its device errors in its own array
    int na_word = 0;
    if (!kda::noalloc_take_error(dev, &na_word)) return KDA_ERR_CUDA;
    word |= na_word;
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
    for (auto &kv : it->second.ws) {
        StreamWorkspace &w = kv.second;
        if (w.ptr != nullptr && cudaFree(w.ptr) != cudaSuccess) return KDA_ERR_CUDA;
    }
    it->second.ws.clear();
    return KDA_OK;
}

}  // extern "C"
