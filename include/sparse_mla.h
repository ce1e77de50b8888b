/*
 * sparse_mla.h — C ABI of libsparse_mla.so, a GB300 (sm_103a) sparse MLA
 * attention forward and its companion fp8 cache writer.
 *
 * Sources (by page title and section):
 *   [P1] "[ROCm][Perf][GLM-5.3-Flash] Enable AITER sparse MLA on gfx942,
 *        including FP8 KV" (vLLM PR 60583): Overview, Claims, Details
 *        ("FP8 KV on gfx942": q quantized per tile inside the kernel, fp8 dots;
 *        the optional dot_precision argument; "Numerics").
 *   [P3] "[ROCm][DSv4.1][Perf] Route gfx942 sparse MLA prefill to AITER
 *        pa_prefill_sparse" (vLLM PR 60102): What changed (one KV pool, output
 *        of q's dtype), Gating and the jin-amd A/B (split-K decode vs no split).
 *   [P4] "[ROCm][MLA][Perf] Fuse decode QK-RoPE + Q-concat + KV-concat +
 *        KV-cache write for sparse MLA" (vLLM PR 47757): Test plan (cache row =
 *        concat(latent, rope); fp8 storage = x / scale, scaled_fp8_quant
 *        convention), "Why positions is a real argument" (graph safety), and the
 *        non-contiguous-input hazard.
 *
 * Conventions shared by every entry point:
 *   - Pointers marked "device" are CUDA device pointers on the current device.
 *     The caller owns every buffer; the library never allocates, frees or
 *     synchronizes, so every call may be captured into a CUDA graph.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *   - Arguments are checked on the host before anything is launched. A failed
 *     check returns its status and writes nothing. SMLA_ERR_CUDA reports a
 *     CUDA runtime error seen at launch.
 *   - Tensors are dense and row-major (contiguous). Strided views are not
 *     accepted: a strided input once produced silently wrong results [P4].
 *   - bf16 is IEEE binary32's upper half; fp8 is OCP E4M3 ("e4m3fn": max 448,
 *     S.1111.111 = NaN, no infinities).
 */
#ifndef SPARSE_MLA_H
#define SPARSE_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SMLA_API __attribute__((visibility("default")))
#else
#define SMLA_API
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *smla_stream_t;

typedef enum {
    SMLA_OK = 0,
    SMLA_ERR_NULL_POINTER = 1,        /* a required pointer is NULL                   */
    SMLA_ERR_BAD_SHAPE = 2,           /* a size is negative or inconsistent            */
    SMLA_ERR_BAD_DTYPE = 3,           /* unknown dtype / precision, or a bad pairing    */
    SMLA_ERR_MISALIGNED = 4,          /* a pointer lacks the alignment stated below    */
    SMLA_ERR_UNSUPPORTED = 5,         /* valid arguments the library has no kernel for */
    SMLA_ERR_WORKSPACE_TOO_SMALL = 6, /* workspace_bytes below the required size       */
    SMLA_ERR_CUDA = 7                 /* CUDA runtime error (device query or launch)   */
} smla_status;

typedef enum {
    SMLA_KV_BF16 = 0,
    SMLA_KV_FP8_E4M3 = 1
} smla_kv_dtype;

/* Precision of the QK dot products [P1 Details: optional dot_precision; when
 * omitted the precision follows q's dtype, which is bf16 here].
 *   AUTO = BF16.
 *   BF16: bf16 q . K, with K the bf16 cache or the fp8 cache's values
 *         code * kv_scale.
 *   FP8 : q quantized inside the kernel per (row, head) tile to E4M3 with
 *         s_q = amax|q[t,h,:]| / 448 (1.0 if amax == 0), q8 = RNE_sat(q / s_q),
 *         dotted with the E4M3 cache; requires an fp8 cache.
 * The PV product always runs on 16-bit operands with fp32 accumulation. */
typedef enum {
    SMLA_DOT_AUTO = 0,
    SMLA_DOT_BF16 = 1,
    SMLA_DOT_FP8 = 2
} smla_dot_precision;

/* Which kernel serves a forward call (smla_fwd_params.kernel).
 *   AUTO     : the library's choice (described under sparse_mla_fwd).
 *   WARP_MMA : the warp-level mma.sync kernel, for every supported shape and
 *              precision (a comparison path: slower, same results within the
 *              stated tolerances).
 *   TCGEN05_BASIC : the first tcgen05 kernels, whose CTAs take a whole SM:
 *              for 16 heads over an E4M3 cache one CTA per SM (AUTO runs two
 *              lean ones per SM); otherwise as AUTO. */
typedef enum {
    SMLA_KERNEL_AUTO = 0,
    SMLA_KERNEL_WARP_MMA = 1,
    SMLA_KERNEL_TCGEN05_BASIC = 2
} smla_kernel_choice;

/* Human-readable name of a status. Never NULL. */
SMLA_API const char *smla_status_string(int status);

/* ABI version, (major << 16) | minor. */
SMLA_API int smla_version(void);

/* Text of the last CUDA runtime error behind an SMLA_ERR_CUDA returned to the
 * calling thread ("no CUDA error" if there was none). Never NULL. */
SMLA_API const char *smla_last_error_string(void);

/* Number of splits of the top-k list ("split-K", [P3] jin-amd A/B: decode-sized
 * calls need it) that sparse_mla_fwd uses when num_splits == 0, for a device
 * with `sm_count` SMs. Host-only arithmetic; returns >= 1, or 0 for invalid
 * arguments. A caller that runs independent calls concurrently (each on its
 * own stream with its own buffers) can pass the SMs one call will get, e.g.
 * half the device's with two or more in flight, and give the result as the
 * calls' num_splits. */
SMLA_API int smla_plan_num_splits(int T, int H, int D_qk, int topk, int kv_dtype,
                                  int sm_count);

/* Bytes of workspace sparse_mla_fwd needs with `num_splits` splits
 * (num_splits == 0: the automatic plan for the current device, which queries
 * the device), for any dot precision the cache allows (the largest of their
 * needs). 0 means no workspace is needed. Returns (size_t)-1 on invalid
 * arguments or a failed device query. (The boundary's first sketch took
 * (T, H, D_v, topk, sm_count); D_qk and kv_dtype are needed because the
 * 128-head E4M3 kernel keeps its quantized q in the workspace, and
 * num_splits because an explicit split count decides the merge path.) */
SMLA_API size_t sparse_mla_fwd_workspace_size(int T, int H, int D_qk, int D_v, int topk,
                                              int kv_dtype, int num_splits);

/*
 * Sparse MLA attention forward ([P1] Overview and Details, [P3] per-call
 * benchmark shapes, [P4] cache layout).
 *
 * For each query row t in [0, T) and head h in [0, H):
 *   I      = { indices[t, i] : indices[t, i] != -1 }            (order free,
 *            duplicates count; entries < -1 or >= num_slots are masked and
 *            never dereferenced — smla_validate_indices reports them)
 *   K(j)   = dequant(kv_cache[j, 0:D_qk]),  V(j) = dequant(kv_cache[j, 0:D_v])
 *            (MLA: one latent row serves as key and value; for D_qk = 576 the
 *            last 64 columns are the rope part, used by QK only)
 *   s_i    = scale * q[t, h, :] . K(I_i)
 *   out[t, h, :] = sum_i softmax(s)_i V(I_i)      (bf16, round to nearest even)
 *   lse[t, h]    = ln sum_i exp(s_i)              (natural log; scale included)
 *   An empty I gives out = 0 and lse = -inf.
 *
 * q            device, bf16 [T, H, D_qk], 16-byte aligned (q and out may be
 *              NULL when T == 0).
 * kv_cache     device, [num_slots, D_qk] of bf16 or E4M3 (kv_dtype): the paged
 *              pool with its blocks flattened (slot = block * block_size +
 *              offset), 16-byte aligned.
 * kv_dtype     smla_kv_dtype.
 * kv_scale     device pointer to one float (dequant = code * kv_scale);
 *              required for SMLA_KV_FP8_E4M3, ignored (may be NULL) for bf16.
 *              Read on the device, so a graph replays the current value.
 * indices      device, int32 [T, topk], 4-byte aligned (may be NULL when topk == 0).
 * T, H, D_qk, D_v, num_slots, topk
 *              supported: H a multiple of 16, D_v = 512, D_qk in {512, 576}.
 *              T = 0 is a no-op. topk = 0 gives empty rows.
 * scale        softmax scale (e.g. 1/sqrt(D_qk)).
 * dot_precision smla_dot_precision (FP8 needs an fp8 cache). AUTO or BF16
 *              with an fp8 cache keeps q in bf16 and dots it with the cache
 *              values code * kv_scale ([P1 Details, "Numerics": the BF16-dots
 *              option]); this runs on the warp-MMA kernel, with at most 8
 *              automatic splits.
 * out          device, bf16 [T, H, D_v], 16-byte aligned, written.
 * lse          device, float [T, H], or NULL to skip.
 * workspace    device, >= sparse_mla_fwd_workspace_size(...) bytes, 256-byte
 *              aligned; may be NULL when that size is 0, which is the case for
 *              up to 8 splits with 16 heads: the splits of a row form one
 *              thread-block cluster and merge through distributed shared
 *              memory. The workspace opens with a fixed region of merge
 *              counters, which must be zero-filled before the buffer's first
 *              use; every call leaves that region zero, so one buffer serves
 *              later calls of any shape on the same stream. With more than 8
 *              splits, after the region, every split writes its partial output
 *              in binary16 (T*H*S*D_v*2 bytes in all) and its lse, then takes a
 *              counter ticket; the split that takes a row's last ticket merges
 *              the row's partials (no split waits for another). The binary16
 *              partials hold averages of value rows: a bf16 cache with values
 *              beyond +-65504 is not supported with more than 8 splits.
 *              The 128-head E4M3 kernel (below) also needs a workspace, after
 *              that region: q quantized per (row, head), T*H*D_qk bytes, and
 *              its T*H scales.
 *              Calls that overlap in time must not share a workspace.
 * Kernels: 16 heads with D_qk = D_v = 512 run on tcgen05 kernels (keys on
 *              the MMA's M axis, accumulators in tensor memory, TMA row
 *              gathers): a bf16 cache on one that takes a whole SM per CTA,
 *              an E4M3 cache with fp8 dots on a lean one that runs two CTAs
 *              per SM (its splits fill twice as many CTAs); H a multiple of
 *              128 with D_qk = 576, D_v = 512 and an E4M3 cache runs, when the
 *              call does not ask for more than one split, on a tcgen05 kernel
 *              with heads on M (two CTAs per row, each owning half of the
 *              value dims; a first pass quantizes q into the workspace); every
 *              other supported shape runs on a warp-MMA (mma.sync) kernel
 *              (sparse_mla_fwd_ex can ask for it for any shape: its `kernel`
 *              field).
 * num_splits   0 = automatic (smla_plan_num_splits for the current device);
 *              otherwise the number of top-k splits to use, 1..128. More than 8
 *              splits need T * H / 16 <= 16384 (else SMLA_ERR_UNSUPPORTED).
 *              For 128 heads over an E4M3 cache with fp8 dots the automatic
 *              plan (0) also spreads the rows' key tiles evenly over pairs of
 *              SMs when the rows outnumber the pairs (a row cut between two
 *              pairs is merged through the workspace); 1 keeps one pair of
 *              CTAs per row.
 * stream       CUDA stream.
 */
SMLA_API smla_status sparse_mla_fwd(const void *q, const void *kv_cache, int kv_dtype,
                                    const float *kv_scale, const int32_t *indices,
                                    int T, int H, int D_qk, int D_v, int64_t num_slots,
                                    int topk, float scale, int dot_precision,
                                    void *out, float *lse,
                                    void *workspace, size_t workspace_bytes,
                                    int num_splits, smla_stream_t stream);

/*
 * The forward with every option in one versioned structure (set `size` to
 * sizeof(smla_fwd_params)); the fields mean what sparse_mla_fwd's arguments
 * mean, plus:
 *   q_scale  NULL for a bf16 q; else q holds E4M3 codes [T, H, D_qk] with this
 *            per-tensor scale (as sparse_mla_fwd_q8: an E4M3 cache, fp8 dots;
 *            dot_precision AUTO or FP8, else SMLA_ERR_BAD_DTYPE).
 *   sinks    NULL, or device float [H], 4-byte aligned: per-head attention
 *            sink logits [P1 Limitations: sinks are passed through], in the
 *            units of scale * q.k. The sink joins each row's softmax
 *            denominator and has no value row:
 *              out = sum_i e^{s_i} v_i / (e^{sink_h} + sum_j e^{s_j}),
 *              lse = log(e^{sink_h} + sum_j e^{s_j});
 *            a row with no valid index gives out = 0 and lse = sink_h.
 */
typedef struct smla_fwd_params {
    size_t size;
    const void *q;
    const float *q_scale;
    const void *kv_cache;
    int kv_dtype;
    const float *kv_scale;
    const int32_t *indices;
    int T, H, D_qk, D_v;
    int64_t num_slots;
    int topk;
    float scale;
    int dot_precision;
    const float *sinks;
    void *out;
    float *lse;
    void *workspace;
    size_t workspace_bytes;
    int num_splits;
    smla_stream_t stream;
    int kernel;          /* smla_kernel_choice (ABI 1.1; a structure of the 1.0
                            size, without this field, means AUTO) */
} smla_fwd_params;

SMLA_API smla_status sparse_mla_fwd_ex(const smla_fwd_params *params);

/* The exact workspace bytes the call described by `params` needs (its dot
 * precision, q form, kernel choice and split count; pointers are not read).
 * 0 = none. Returns (size_t)-1 for arguments sparse_mla_fwd_ex would reject
 * or a failed device query. */
SMLA_API size_t sparse_mla_fwd_ex_workspace_size(const smla_fwd_params *params);

/*
 * The same forward with a pre-quantized q [P1 Details, "FP8 KV on gfx942":
 * gfx950 keeps the pre-quantized q]: q8 holds E4M3 codes [T, H, D_qk] (as
 * written, for example, by smla_fused_qk_rope_cache with an E4M3 q_out) and
 * *q_scale is their per-tensor scale, so q enters the dots as code * q_scale.
 * The cache must be E4M3 (kv_scale as above); the dots run in fp8, as with
 * SMLA_DOT_FP8, without quantizing q again. Every other argument, the
 * workspace and the kernels are as for sparse_mla_fwd.
 * q8       device, uint8 [T, H, D_qk], 16-byte aligned.
 * q_scale  device, one float, 4-byte aligned.
 */
SMLA_API smla_status sparse_mla_fwd_q8(const void *q8, const float *q_scale, const void *kv_cache,
                                       const float *kv_scale, const int32_t *indices, int T, int H, int D_qk,
                                       int D_v, int64_t num_slots, int topk, float scale, void *out, float *lse,
                                       void *workspace, size_t workspace_bytes, int num_splits,
                                       smla_stream_t stream);


/*
 * Maximum workspace bytes sparse_mla_fwd_no_alloc can serve from its static
 * device array (8 MiB): every GPU that loads the library holds this much.
 */
#define SMLA_NO_ALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * sparse_mla_fwd without a caller-provided workspace (the pages have no
 * counterpart; it exists for callers of this library that cannot allocate
 * device memory: a serving engine that reserved nearly all of HBM for its
 * KV-cache pool up front, or a host framework that only lets a plug-in use
 * the buffers it hands over).
 *
 * Arguments and results are those of sparse_mla_fwd; q, kv_cache, indices,
 * out and lse remain the caller's. When the call's own plan needs a workspace
 * the library uses a static device array of SMLA_NO_ALLOC_SCRATCH_BYTES
 * instead, and returns SMLA_ERR_WORKSPACE_TOO_SMALL (nothing launched) when
 * the call would need more. Two kinds of call need it:
 *   - more than 8 splits of a row (merge counters, then T * S * H * 1 KB of
 *     binary16 partial results);
 *   - the 128-head E4M3 kernel with fp8 dots (H a multiple of 128, D_qk = 576,
 *     one split), at any split plan: its quantized q, T * H * 580 bytes after
 *     a 64 KB counter region. When its automatic plan spreads the rows over
 *     CTA pairs (more rows than pairs) it also keeps partials of shared rows;
 *     if those do not fit, this entry point runs the call with one CTA pair
 *     per row, which needs the quantized q only. T * H must stay below about
 *     14,300: 128 rows of 128 heads (9.5 MB) do not fit and are rejected.
 * Calls with bf16 dots or a bf16 cache and at most 8 splits use no workspace
 * and never touch the array. Nothing is allocated or freed. Each call looks
 * the array's device address up (cudaGetSymbolAddress) with its device
 * current; make a device's first call before any stream capture, since that
 * lookup may load the module. A call that merges through the counters clears
 * them on `stream` before launching. All calls share the one array: calls
 * that can run at the same time on the GPU (unordered streams) race on it and
 * must not overlap.
 */
SMLA_API smla_status sparse_mla_fwd_no_alloc(const void *q, const void *kv_cache, int kv_dtype,
                                             const float *kv_scale, const int32_t *indices,
                                             int T, int H, int D_qk, int D_v, int64_t num_slots,
                                             int topk, float scale, int dot_precision,
                                             void *out, float *lse, int num_splits,
                                             smla_stream_t stream);

/*
 * Error word of the device-side checks (0 = none). The tcgen05 kernels wait on
 * the tensor core and on their own warps with a time limit (about 2 s); a wait
 * that gives up sets a bit here (1 = an awaited barrier never completed,
 * 2 = the copies or MMAs in flight did not drain), abandons the call's
 * arithmetic, frees its tensor memory and returns, leaving the context usable.
 * smla_fused_qk_rope_cache sets 4 for a position outside [0, max_position) and
 * 8 for a slot >= num_slots. Synchronous (copies the word from the device):
 * unlike every other entry point it waits for the device, since the word is
 * read on the host. reset != 0 clears it.
 */
SMLA_API smla_status smla_device_error(int *code, int reset);

/*
 * Per-tensor fp8 scale of a bf16 tensor [P4 Test plan: scaled_fp8_quant with a
 * per-tensor scale]: *scale_out = amax(|x|) / 448 in binary32, or 1.0 when
 * amax == 0. NaN elements are ignored.
 * x          device, bf16 [n], 16-byte aligned (may be NULL when n == 0).
 * scale_out  device, one float, 4-byte aligned; used as the reduction cell
 *            during the call.
 */
SMLA_API smla_status smla_compute_fp8_scale(const void *x, int64_t n, float *scale_out,
                                            smla_stream_t stream);

/*
 * Quantizing cache write [P4 Summary and Test plan: concat_and_cache_mla into
 * an fp8 cache]: for n in [0, N) with slot = slot_mapping[n] in [0, num_slots):
 *   kv_cache[slot, d] = E4M3_RNE_satfinite(src[n, d] / *kv_scale)   (binary32
 *   division), d in [0, D). slot == -1 skips the row, as does any slot outside
 *   [0, num_slots) (a contract violation).
 * src          device, bf16 [N, D], 16-byte aligned, D a multiple of 8.
 * slot_mapping device, int64 [N].
 * kv_scale     device, one float.
 * kv_cache     device, uint8 [num_slots, D], 8-byte aligned.
 */
SMLA_API smla_status smla_fp8_cache_write(const void *src, const int64_t *slot_mapping,
                                          int64_t N, int D, const float *kv_scale,
                                          void *kv_cache, int64_t num_slots,
                                          smla_stream_t stream);

/*
 * The fused producer step of sparse MLA decode [P4 Summary: main RoPE on
 * q_pe/k_pe, the query concat, the KV concat and the fp8 KV-cache write in one
 * kernel; Test plan: parity with the split chain]. For each token t, with
 * p = positions[t] and R = the rotation below:
 *   q_out[t, h, :]  = concat(ql_nope[t, h, 0:512], R_p(q_pe[t, h, 0:64]))   h in [0, H)
 *   kv_cache[slot_mapping[t], :] = concat(kv_c[t, 0:512], R_p(k_pe[t, 0:64]))
 * stored as bf16, or (q_out_dtype / kv_dtype = SMLA_KV_FP8_E4M3) as the codes
 * E4M3_RNE_satfinite(x / *q_scale) resp. (x / *kv_scale), binary32 division of
 * the bf16 value x (the scaled_fp8_quant convention).
 * R_p rotates each pair (a, b) to (a cos - b sin, b cos + a sin) with
 * cos = cos_sin_cache[p, i], sin = cos_sin_cache[p, 32 + i] for pair i: in
 * binary32, each product and the difference or sum rounded (no fused
 * multiply-add), then rounded to bf16 before any quantization, as the split
 * chain stores it. is_neox != 0 pairs element i with i + 32, else 2i with
 * 2i + 1.
 *
 * ql_nope        device, bf16 [T, H, 512], element strides (ql_stride_t,
 *                ql_stride_h), the last dimension contiguous; strides
 *                multiples of 8, pointer 16-byte aligned (a transposed
 *                [H, T, 512] buffer is stride_t = 512, stride_h = T * 512).
 * q_pe           device, bf16 [T, H, 64] pre-RoPE, strides (qpe_stride_t,
 *                qpe_stride_h), even, pointer 4-byte aligned.
 * kv_c           device, bf16 [T, 512], row stride kvc_stride_t (multiple of
 *                8), 16-byte aligned.
 * k_pe           device, bf16 [T, 64] pre-RoPE, row stride kpe_stride_t (even),
 *                4-byte aligned.
 * positions      device, int64 [T].
 * cos_sin_cache  device, float [max_position, 64]: 32 cosines then 32 sines.
 * slot_mapping   device, int64 [T]; a negative slot writes no cache row.
 * kv_cache       device, [num_slots, 576] bf16 or E4M3 (kv_dtype), 16-byte aligned.
 * kv_scale       device, one float; required for an E4M3 cache.
 * q_out          device, [T, H, 576] bf16 or E4M3 (q_out_dtype), contiguous,
 *                16-byte aligned; must not overlap the inputs.
 * q_scale        device, one float; required for E4M3 q_out.
 * H may be 0 (cache rows only; the q pointers may then be NULL); H above
 * 524279 is SMLA_ERR_BAD_SHAPE.
 * A token whose position is outside [0, max_position) gets neither its q rows
 * nor its cache row, and sets bit 4 of smla_device_error; a slot >= num_slots
 * writes no row and sets bit 8. Asynchronous on `stream`.
 */
SMLA_API smla_status smla_fused_qk_rope_cache(const void *ql_nope, int64_t ql_stride_t, int64_t ql_stride_h,
                                              const void *q_pe, int64_t qpe_stride_t, int64_t qpe_stride_h,
                                              const void *kv_c, int64_t kvc_stride_t, const void *k_pe,
                                              int64_t kpe_stride_t, const int64_t *positions,
                                              const float *cos_sin_cache, int64_t max_position, int is_neox,
                                              const int64_t *slot_mapping, void *kv_cache, int kv_dtype,
                                              int64_t num_slots, const float *kv_scale, void *q_out,
                                              int q_out_dtype, const float *q_scale, int T, int H,
                                              smla_stream_t stream);

/*
 * Measurement kernels (not part of the forward; bench.py reports them beside
 * the forward's rate as the ceilings it is held against).
 *
 * smla_gather_probe: a pure indexed-row copy at the forward kernels' gather
 * pattern. The n_indices entries of `indices` are taken as consecutive tiles
 * of 64 rows, split evenly over ctas_per_sm CTAs on each SM; each CTA copies
 * its tiles' rows [idx, 0:row_bytes) of the pool [num_rows, row_bytes]
 * (row_bytes a multiple of 16, at most 1024) into a ring of `stages` tiles in
 * shared memory (128-byte column blocks, 128-byte swizzle): copy_mode 0 by TMA
 * tile::gather4 (128-byte boxes), copy_mode 1 by 16-byte cp.async copies from
 * eight warps (pair_mode and issue_warps 0, else SMLA_ERR_UNSUPPORTED). -1
 * and out-of-range entries are zero-filled without a read. A consumer folds
 * the first 4 bytes of each row into checksum[cta] (XOR, written; device
 * uint32 [sm_count * ctas_per_sm]) and holds each tile hold_ns nanoseconds
 * before releasing it. SMLA_ERR_UNSUPPORTED when `stages` tiles do not fit
 * ctas_per_sm CTAs on one SM; ctas_per_sm in 1..4, stages in 1..8.
 * pair_mode (with ctas_per_sm = 1): 0 = single CTAs; 1 or 2 = CTAs in pairs,
 * each pair a thread-block cluster of two that takes the tiles one CTA would:
 * each CTA gathers half of every tile's rows (so every row is read once) and
 * delivers it to both CTAs, by cluster multicast of its gathers (1) or by a
 * bulk copy of its landed half into the peer's ring (2); a stage is refilled
 * once both consumers released it (the patterns of a pair that shares its key
 * rows). Only the first CTA of a pair writes its checksum (the second writes
 * 0). 3 = single CTAs launched in clusters of two (a control for 1 and 2).
 * issue_warps: 0 = copy c of a tile (c < 16 * boxes per row, boxes =
 * row_bytes / 128 rounded up; half that in pair modes 1 and 2) is issued by
 * producer thread c of four warps; 1..8 = the copies are spread evenly over
 * that many warps, ceil(copies / issue_warps) lanes each, which must not
 * exceed 32 (else SMLA_ERR_BAD_SHAPE).
 *
 * smla_l2_read_probe: `blocks` blocks of 512 threads read the first `bytes`
 * of `buf` (a multiple of 16, 16-byte aligned) `reps` times with 16-byte
 * loads that bypass L1, and write one word per block to checksum[block]. With
 * a buffer smaller than L2 its rate is the L2 -> SM read bandwidth.
 */
SMLA_API smla_status smla_gather_probe(const void *pool, int64_t num_rows, int row_bytes,
                                       const int32_t *indices, int64_t n_indices, int ctas_per_sm,
                                       int stages, int hold_ns, int pair_mode, int issue_warps, int copy_mode,
                                       uint32_t *checksum, smla_stream_t stream);
SMLA_API smla_status smla_l2_read_probe(const void *buf, int64_t bytes, int reps, uint32_t *checksum,
                                        int blocks, smla_stream_t stream);

/*
 * Counts the entries of indices [T, topk] that are neither -1 nor inside
 * [0, num_slots) and stores the count in *bad_count (device int, overwritten).
 */
SMLA_API smla_status smla_validate_indices(const int32_t *indices, int T, int topk,
                                           int64_t num_slots, int *bad_count,
                                           smla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MLA_H */
