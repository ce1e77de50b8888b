// Internal host-side interface between the C ABI layer (smla_api.cu) and the
// kernel translation units. Not installed; not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/sparse_mla.h"

namespace smla {

// Everything a forward launch needs, already validated by the ABI layer.
struct FwdArgs {
    const void *q;          // bf16 [T, H, D_qk]
    const void *kv;         // [num_slots, D_qk] bf16 or E4M3
    const float *kv_scale;  // device scalar (fp8) or nullptr
    const int32_t *indices; // [T, topk]
    void *out;              // bf16 [T, H, D_v]
    float *lse;             // [T, H] or nullptr
    uint16_t *part_o16;     // [T, S, H, D_v] binary16 split partials (S > kClusterMaxSplits)
    float *part_lse;        // [T, S, H]        (S > kClusterMaxSplits)
    int *tickets;           // [T, H / 16]      (S > kClusterMaxSplits)
    uint8_t *q8;            // [T, H, 512] E4M3 codes of q's first 512 columns (128-head kernel)
    uint8_t *q8_rope;       // [T, H/128] blocks of 8 KB: the last 64 columns, core-matrix order
    float *q_scale;         // [T, H] per-(row, head) q scales (128-head kernel)
    int64_t num_slots;
    int T, H, D_qk, D_v, topk;
    int S;                  // splits of the top-k list
    int keys_per_split;     // multiple of the key tile
    float scale;
    bool kv_fp8;            // E4M3 cache with fp8 QK dots
    const float *sinks;     // [H] per-head sink logits (natural-log units), or nullptr
    bool bf16_dots;         // E4M3 cache with bf16 q . dequantized K dots (warp-MMA kernel)
    bool q_fp8_in;          // q holds E4M3 codes [T, H, D_qk] with one per-tensor scale
    const float *q_scale_in; // that scale (device scalar), or nullptr
    // 128-head kernel: pairs of CTAs the (row, key tile) sequence is cut into
    // (rows = T * H / 128 gives one row per pair), and for rows a pair shares
    // with its neighbour the partial outputs [2 * pairs][2 halves][16 head
    // groups][256 dims][8 heads] (binary16, in units of the cache's codes), their lse
    // [2 * pairs][2][128], and per (row, half) merge flags [rows][2] (in the
    // counter region)
    int wide_pairs;
    uint16_t *wide_part;
    float *wide_part_lse;
    int *wide_tickets;
    // 16-head kernel, cp.async copies: first find the split's last valid index
    // and skip the tiles after it (set by its launcher for pools in L2)
    bool trim_tail;
};

// Key tile of the warp-MMA kernel (keys per pipeline stage).
constexpr int kMmaTileKeys = 32;
// Key tile of the tcgen05 16-head kernel (the M of its QK MMA).
constexpr int kUmma16TileKeys = 64;

// Up to this many splits of a row's top-k list run as one thread-block
// cluster and merge their partial results through distributed shared memory
// (no workspace; the automatic plan stays within it). More splits (very small
// T, explicit split counts up to kMaxSplits) merge through the workspace.
constexpr int kClusterMaxSplits = 8;
constexpr int kMaxSplits = 128;

// The workspace opens with a fixed-size region of merge counters, so the
// counters of any call land in memory that is zero between calls: each call
// returns the counters it used to zero, and partial results never overlap
// the region, whatever the shapes of earlier calls.
constexpr int kTicketSlots = 16384;

// Workspace layout (byte offsets, 256-byte aligned): a region of merge
// counters that every call leaves zero, then, for S > kClusterMaxSplits, the
// split partials in binary16 and their lse, or, for the 128-head kernel, the quantized q and
// its scales (and the partials of rows its CTA pairs share).
struct WorkspaceLayout {
    size_t tickets, part_lse, part_o16, q8, q8_rope, q_scale, wide_part_lse, wide_part, total;
};
// wide_pairs: the 128-head kernel's pairs when they are fewer than its rows
// (rows shared between pairs need partial slots), else 0
WorkspaceLayout workspace_layout(int T, int H, int D_qk, int D_v, int S, bool wide, int wide_pairs = 0);

// The plan of one forward call (see plan_forward in smla_api.cu).
struct FwdPlan {
    int path;            // the kernel that serves the call
    int S;               // splits of each row's top-k list
    bool bf16_dots;      // E4M3 cache with bf16 dots
    bool uses_tickets;   // the workspace's merge counters take part (S > kClusterMaxSplits, or shared rows)
    int wide_pairs;      // 128-head kernel: CTA pairs of the launch
    WorkspaceLayout layout;
};
// Plans a call whose arguments are valid; returns SMLA_OK or the status that
// rejects it (SMLA_ERR_UNSUPPORTED, or SMLA_ERR_CUDA for a failed device query).
smla_status plan_forward(int T, int H, int D_qk, int D_v, int topk, int kv_dtype, int dot_precision,
                         int num_splits, int kernel, FwdPlan *out);

cudaError_t launch_fwd_mma(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_fwd_wide(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_fwd_umma16(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_fwd_lean16(const FwdArgs &a, cudaStream_t stream);
// The 128-head kernels' q pass: per (row, head) E4M3 codes and scales of q
// (or the pre-quantized codes rearranged) into the workspace.
cudaError_t launch_quantize_q_wide(const FwdArgs &a, cudaStream_t stream);
// cuTensorMapEncodeTiled from the driver (resolved once; nullptr if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// First error code recorded by a bounded device-side wait that gave up (0 = none).
cudaError_t read_umma_error(int *out, bool reset);
cudaError_t read_wide_error(int *out, bool reset);
cudaError_t read_lean_error(int *out, bool reset);

// The fused producer step (RoPE + q concat + cache write), validated by the ABI layer.
struct FusedProducerArgs {
    const void *ql_nope;            // bf16 [T, H, 512], element strides (t, h), rows 16-byte aligned
    int64_t ql_stride_t, ql_stride_h;
    const void *q_pe;               // bf16 [T, H, 64], element strides (t, h), rows 4-byte aligned
    int64_t qpe_stride_t, qpe_stride_h;
    const void *kv_c;               // bf16 [T, 512], row stride, rows 16-byte aligned
    int64_t kvc_stride_t;
    const void *k_pe;               // bf16 [T, 64], row stride, rows 4-byte aligned
    int64_t kpe_stride_t;
    const int64_t *positions;       // [T]
    const float *cos_sin_cache;     // [max_position, 64]: 32 cosines, then 32 sines
    int64_t max_position;
    const int64_t *slot_mapping;    // [T], negative = no cache row
    void *kv_cache;                 // [num_slots, 576] bf16 or E4M3
    int64_t num_slots;
    const float *kv_scale;          // device scalar (E4M3 cache)
    void *q_out;                    // [T, H, 576] bf16 or E4M3, contiguous
    const float *q_scale;           // device scalar (E4M3 q_out)
    int T, H;
    bool is_neox, q_out_fp8, cache_fp8;
};
cudaError_t launch_fused_producer(const FusedProducerArgs &a, cudaStream_t stream);
cudaError_t read_producer_error(int *out, bool reset);

// Measurement kernels: a pure indexed-row copy at the forward kernels' gather
// pattern, and an L2 -> SM streaming read.
cudaError_t launch_gather_probe(const void *pool, int64_t num_rows, int row_bytes, const int32_t *indices,
                                int64_t n_indices, int ctas_per_sm, int stages, int hold_ns, int pair_mode,
                                int issue_warps, int copy_mode, uint32_t *checksum, int sm_count,
                                cudaStream_t stream);
cudaError_t launch_l2_read_probe(const void *buf, int64_t bytes, int reps, uint32_t *checksum, int blocks,
                                 cudaStream_t stream);
cudaError_t read_probe_error(int *out, bool reset);

cudaError_t launch_fp8_scale(const void *x, int64_t n, float *scale_out, int sm_count,
                             cudaStream_t stream);
cudaError_t launch_fp8_cache_write(const void *src, const int64_t *slot_mapping, int64_t N, int D,
                                   const float *kv_scale, void *cache, int64_t num_slots,
                                   cudaStream_t stream);
cudaError_t launch_validate_indices(const int32_t *indices, int64_t n, int64_t num_slots,
                                    int *bad_count, int sm_count, cudaStream_t stream);

} // namespace smla
