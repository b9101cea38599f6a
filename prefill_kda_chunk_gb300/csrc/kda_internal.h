// Host-side interface between the C ABI (kda_api.cu) and the kernel
// translation units. Nothing here is exported from the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Where each sequence's tokens and chunks are. Fixed-length batches
// (cu == nullptr) hold N sequences of `seq_len` tokens each; packed batches
// use cu_seqlens and the per-sequence chunk offsets the prologue writes.
struct ChunkGeometry {
    const int32_t *cu;         // [N+1] or nullptr
    const int32_t *chunk_off;  // [N+1] (packed) or nullptr
    const int *call_flags;     // per-call flag word (packed only)
    int64_t seq_len;           // fixed: tokens per sequence; packed: total tokens
    int32_t n_seqs;
    int32_t n_heads;
    int32_t chunks_per_seq;    // fixed only: chunks of one whole sequence
    // Fixed-length only: one launch covers chunk positions
    // [pos_begin, pos_begin + seg_len) of every sequence, and the record of
    // (sequence n, position pos_begin + i, head h) sits at index
    // (n * slot_stride + i) * H + h. The first position of a segment is
    // treated as the start of a sequence by the intra-chunk kernel (no
    // look-ahead terms), so each segment's recurrent launch starts afresh
    // from the state the previous one left.
    int32_t pos_begin;
    int32_t seg_len;
    int32_t slot_stride;
};

struct IntraParams {
    const void *q, *k, *v;     // bf16 [tokens, H, 128]
    const float *g;            // [tokens, H, 128]
    const float *beta;         // [tokens, H]
    uint8_t *rec;              // chunk records [chunks, H, kRecBytes]
    float scale;               // output scale, folded into the record's Q e^G and P
    int pre;                   // kPreNormQK | kPreGateLogits (input preprocessing)
    int *err;                  // sticky per-device error word
    ChunkGeometry geo;
    // Chunk-heads outside the range of the factored exponentials: the
    // intra-chunk kernel appends their item index (chunk * H + head) to
    // exact_list, counting in exact_ctr[0]; the exact kernel consumes the list
    // and zeroes both counters (exact_ctr[1] counts its finished CTAs). Both
    // counters are 0 between calls; exact_list holds one entry per item.
    int32_t *exact_list = nullptr;
    int *exact_ctr = nullptr;
    // When not null, (I + A)^{-1} of every chunk-head, fp32, 16 rows of 20
    // floats (the last 4 unused) at item index (record index * H + head) * 320
    // (the gradient kernel copies one item's 1280 bytes in one piece)
    float *tinv = nullptr;
    // When not null, set to 1 by any chunk-head whose |G| passes 80 (the
    // gradient kernel compiles the form for such chunks in only when it is set)
    int *wide_flag = nullptr;
};

struct RecurParams {
    const uint8_t *rec;
    const float *s0;           // [N, H, 128, 128] or nullptr
    void *out;                 // bf16 [tokens, H, 128]
    float *s_final;            // [N, H, 128, 128] or nullptr
    int *err;
    ChunkGeometry geo;
    // Segment-parallel scan of fixed-length sequences (cu == nullptr): with
    // scan_segs = P >= 2 every sequence's chunks are cut into segments of
    // scan_len chunks (the last one takes the rest). Over a segment the state
    // map is affine, S_end = M S_begin + c, and M (K x K) evolves like the
    // state with Ut taken as zero, starting from the identity.
    //   maps launch (launch_recurrent_scan_maps): units (sequence, segment
    //     j < P-1) x 4 slices of 64 columns; slices 0-1 carry the state
    //     columns (from s0 for j = 0, else from zero), slices 2-3 the columns
    //     of M (j > 0 only). j = 0 writes its end state to seg_entry[0], j > 0
    //     writes c to seg_c[j-1] and M to seg_m[j-1].
    //   replay launch (launch_recurrent): units (sequence, segment), segment
    //     j > 0 starting from seg_entry[j-1]; only the last one writes s_final.
    int32_t scan_segs = 0;
    int32_t scan_len = 0;
    float *seg_entry = nullptr;    // [P-1][N][H][128][128]: entry states of segments 1..P-1
    float *seg_c = nullptr;        // [P-2][N][H][128][128]
    float *seg_m = nullptr;        // [P-2][N][H][128][128]
    // Test hook (kda_test_stall_recurrent): the record producer of every CTA
    // issues no copy for chunk stall_chunk and later ones (-1: off), and both
    // roles give up a wait after wait_ns (0: the default limit). A copy that
    // was issued is always waited for, so none is in flight at exit.
    int32_t stall_chunk = -1;
    unsigned long long wait_ns = 0;
};

// One-token decode step for N*H independent (sequence, head) units.
struct DecodeParams {
    const void *q, *k, *v;     // bf16 [N, H, 128]
    const float *g;            // [N, H, 128] per-token log decay
    const float *beta;         // [N, H]
    const float *s_in;         // [N, H, 128, 128] or nullptr (zero state)
    float *s_out;              // [N, H, 128, 128]; may be s_in itself
    void *out;                 // bf16 [N, H, 128]
    float scale;
    int pre;                   // kPreNormQK | kPreGateLogits (input preprocessing)
};

// Gradients of the prefill for N*H independent (sequence, head) units; see
// kda_backward.cu. The geometry's cu / chunk_off / call_flags / seq_len /
// chunks_per_seq / n_heads are used as in the prefill.
struct BackParams {
    const void *q, *k, *v;     // bf16 [tokens, H, 128]
    const float *g;            // [tokens, H, 128] per-token log decay
    const float *beta;         // [tokens, H]
    const float *s0;           // [N, H, 128, 128] or nullptr (zero state)
    const void *dout;          // bf16 [tokens, H, 128]: dL/do
    const float *dsf;          // [N, H, 128, 128] or nullptr: dL/d(final state)
    float scale;
    float *dq, *dk, *dv, *dg;  // fp32 [tokens, H, 128]
    float *dbeta;              // fp32 [tokens, H]
    float *ds0;                // fp32 [N, H, 128, 128] or nullptr: dL/d(initial state)
    float *ckpt;               // workspace: one state per 16 tokens per head
    float *ring;               // workspace: 16 states per CTA of the launch
    ChunkGeometry geo;
};

// Chunked gradients (kda_backward_chunk.cu). ip carries the inputs (q, k,
// v, g, beta, scale; pre = 0) and the geometry; rec holds the forward's
// records, ckpt the forward chain's chunk-entry states S^T and dsn the
// reverse chain's dS_next^T, both bf16 [record index][H][128 v][128 k].
struct BwdChunkParams {
    IntraParams ip;
    const uint8_t *rec;
    const float *s0;           // [N, H, 128, 128] or nullptr (zero initial state)
    const void *dout;          // bf16 [tokens, H, 128]: dL/do
    const float *dsf;          // [N, H, 128, 128] or nullptr: dL/d(final state)
    float *ds0;                // [N, H, 128, 128] or nullptr: dL/d(initial state)
    void *ckpt;
    void *dsn;
    float *dq, *dk, *dv, *dg;  // fp32 [tokens, H, 128]
    float *dbeta;              // fp32 [tokens, H]
    int *err;
    ChunkGeometry geo;
    int64_t max_chunks;
    // [0]: the intra-chunk kernel's wide_flag; [1]: the gradient kernel's finish
    // count (both 0 between calls; the gradient kernel's last CTA resets them)
    int *wide = nullptr;
};
// cuTensorMapEncodeTiled from the driver (cast to its signature), or null.
void *tensor_map_encoder();

cudaError_t configure_backward_chunk();
// the forward chain keeping chunk-entry states and the reverse chain, one launch
cudaError_t launch_bwd_chains(const BwdChunkParams &p, cudaStream_t stream);
cudaError_t launch_bwd_grad(const BwdChunkParams &p, cudaStream_t stream);

// Per-device, once: raise the dynamic shared-memory limits of the kernels.
cudaError_t configure_intra();
cudaError_t configure_recurrent();

// chunk_off[n] = first chunk of sequence n for chunks of 2^chunk_shift tokens
cudaError_t launch_varlen_prologue(const int32_t *cu, int32_t n_seqs, int64_t total_tokens,
                                   int32_t *chunk_off, int *call_flags, int *err,
                                   cudaStream_t stream, int chunk_shift = 4);
cudaError_t launch_intra_chunk(const IntraParams &p, int64_t max_chunks, cudaStream_t stream);
// the exact form over the chunk-heads the intra-chunk kernel listed; launch
// after every launch_intra_chunk, on the same stream
cudaError_t launch_intra_exact(const IntraParams &p, cudaStream_t stream);
cudaError_t launch_recurrent(const RecurParams &p, cudaStream_t stream);     // warp MMA
// the maps launch of the segment-parallel scan (RecurParams::scan_segs >= 2)
cudaError_t launch_recurrent_scan_maps(const RecurParams &p, cudaStream_t stream);
// its serial combine: seg_entry[j] = seg_m[j-1] seg_entry[j-1] + seg_c[j-1]
// for j = 1 .. P-2, per (sequence, head); a no-op for P = 2
cudaError_t launch_scan_combine(const RecurParams &p, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams &p, int64_t units, cudaStream_t stream);
// The gradient kernel is persistent: at most one CTA per resident slot and
// never more than kBackwardMaxRings, each owning one 16-state ring of the
// workspace (BackParams::ring holds min(units, kBackwardMaxRings) rings).
constexpr int64_t kBackwardMaxRings = 1024;
cudaError_t launch_backward(const BackParams &p, int64_t units, cudaStream_t stream);

// The 64-token chunk path on the 5th-generation tensor core (kda_c64.cu).
struct C64Args {
    const void *q, *k, *v;      // bf16 [tokens, H, 128]
    const float *g, *beta;      // [tokens, H, 128], [tokens, H]
    const float *s0;            // [N, H, 128, 128] or nullptr
    void *out;                  // bf16 [tokens, H, 128]
    float *s_final;             // [N, H, 128, 128] or nullptr
    const int32_t *cu;          // packed: cu_seqlens [N+1]; fixed: nullptr
    const int32_t *chunk_off;   // packed: first 64-token chunk of each sequence [N+1]
    const int *call_flags;      // packed: per-call flags of the prologue
    int *err;                   // sticky per-device error word
    int64_t tokens;             // rows of q
    int64_t seq_len;            // fixed: tokens per sequence; packed: total tokens
    int64_t max_chunks;         // 64-token chunks (upper bound when packed)
    int32_t n_seqs, n_heads, cps;   // cps: chunks per sequence (fixed)
    float scale;
    int pre;                    // kPreNormQK | kPreGateLogits
    uint8_t *rec;               // records: max_chunks * H (split) or ring_depth * H (fused)
    int ring_depth;             // fused: ring slots per head
    int n_chain;                // fused: chain CTAs (one per head)
    long long *ready;           // fused: [ring_depth * H], zero between calls
    long long *consumed;        // fused: [H], zero between calls
    int *exit_ctr;              // fused: zero between calls
};
constexpr int64_t kC64RecBytes = 74240;   // bytes of one (64-token chunk, head) record
cudaError_t configure_c64();
// the intra-chunk kernel over every chunk-head (persistent, intra_ctas CTAs)
cudaError_t launch_c64_intra(const C64Args &a, int intra_ctas, cudaStream_t stream);
// one recurrent CTA per (sequence, head), records from the intra-chunk kernel
cudaError_t launch_c64_chain(const C64Args &a, cudaStream_t stream);
// one cooperative kernel of `grid` CTAs: a.n_chain = H chain CTAs (each over
// all sequences of its head) and grid - H record builders feeding the ring
cudaError_t launch_c64_fused(const C64Args &a, int grid, cudaStream_t stream);

// Host-side checks shared by the entry points (kda_api.cu): 0 when `p` is
// NULL, device memory of device `dev` or managed memory; otherwise the
// kda_status the entry point returns (not device memory / wrong device).
int pointer_device_status(const void *p, int dev);

// The error word of the allocation-free entry point's fixed scratch array on
// device `dev` (kda_noalloc.cu): read and cleared with a synchronous copy,
// 0 when that array has not been set up on the device. Returns false if a
// CUDA call failed.
bool noalloc_take_error(int dev, int *word);

}  // namespace kda
