// C ABI of libsparse_mla.so: argument checks on the host, the split plan, and
// dispatch to the kernels. Declared and documented in include/sparse_mla.h.
#include "../../include/sparse_mla.h"
#include "smla_internal.h"

#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

namespace {

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

// Record a CUDA error for smla_last_error_string and map it to a status.
smla_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess)
        return SMLA_OK;
    t_last_cuda_error = e;
    return SMLA_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

// SM count of the current device (cached per device).
cudaError_t current_sm_count(int *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < kMaxDevices) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) {
            *out = cached;
            return cudaSuccess;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= 0 && dev < kMaxDevices)
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return cudaSuccess;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Which kernel serves a call.
enum class Path { Mma, Umma16, Wide, Lean16 };

// 16 heads with D_qk = D_v = 512: an E4M3 cache with fp8 dots runs on the
// lean tcgen05 16-head kernel (two CTAs per SM: its random 512-byte row
// gathers complete faster with more CTAs per SM), a bf16 cache, or an E4M3
// cache with bf16 dots, on the tcgen05 16-head kernel that takes a whole SM
// per CTA (its 1 KB row gathers reach the DRAM bound already; with bf16 dots
// it expands the gathered E4M3 rows to binary16 in shared memory); a
// multiple of 128 heads with D_qk = 576, D_v = 512 and an E4M3 cache with
// fp8 dots: the tcgen05 128-head kernel (no split of the top-k list); every
// other shape or precision: the warp-MMA kernel. `kernel`
// (smla_kernel_choice) can ask for the warp-MMA kernel, or for the first
// tcgen05 kernels (whole SM per CTA, nothing shared).
Path choose_path(int H, int D_qk, int D_v, bool kv_fp8, bool fp8_dots, int kernel)
{
    if (kernel == SMLA_KERNEL_WARP_MMA)
        return Path::Mma;
    if (H == 16 && D_qk == 512 && D_v == 512)
        return kv_fp8 && fp8_dots && kernel != SMLA_KERNEL_TCGEN05_BASIC ? Path::Lean16 : Path::Umma16;
    if (kv_fp8 && !fp8_dots)
        return Path::Mma;
    if (H % 128 == 0 && D_qk == 576 && D_v == 512 && kv_fp8)
        return Path::Wide;
    return Path::Mma;
}

int ctas_per_sm(Path p) { return (p == Path::Mma || p == Path::Lean16) ? 2 : 1; }
int tile_keys(Path p)
{
    return (p == Path::Umma16 || p == Path::Lean16) ? smla::kUmma16TileKeys : smla::kMmaTileKeys;
}

// Split plan, from the per-call sweep (rows {2..16K} x fan-out {128, 512,
// 2048}, 16 heads, bf16): a split keeps at least two key tiles (128 keys);
// the automatic plan stays within one cluster merge (up to 8 splits: the
// workspace merge of more splits cost up to 2x at 2 rows x 2048 keys); and
// 8-CTA clusters, fast when few (2 rows), were slower than 6-CTA ones once
// rows x splits passed 64 (16 rows: 28 us at 8 splits, 17.6 us at 6).
constexpr int kMinKeysPerSplit = 128;
using smla::kClusterMaxSplits;
constexpr int kWideClusterSplits = 6;
constexpr int64_t kWideClusterRowSplits = 64;
using smla::kMaxSplits;
using smla::kTicketSlots;

int plan_splits(int T, int H, int topk, int sm_count, Path path)
{
    if (T <= 0 || H <= 0 || topk <= 0 || sm_count <= 0 || path == Path::Wide)
        return 1;
    const int64_t units = (int64_t)T * (H / 16);
    const int64_t slots = (int64_t)sm_count * ctas_per_sm(path);
    int64_t S = units >= slots ? 1 : slots / units;
    const int64_t by_keys = topk / kMinKeysPerSplit;
    if (S > by_keys)
        S = by_keys;
    if (S > kClusterMaxSplits)
        S = kClusterMaxSplits;
    if (S > kWideClusterSplits && units * S > kWideClusterRowSplits)
        S = kWideClusterSplits;
    return S < 1 ? 1 : (int)S;
}

int keys_per_split(int topk, int S, int tile)
{
    const int per = (topk + S - 1) / S;
    return ((per + tile - 1) / tile) * tile;
}

bool shape_supported(int H, int D_qk, int D_v)
{
    return H > 0 && H % 16 == 0 && D_v == 512 && (D_qk == 512 || D_qk == 576);
}

} // namespace

namespace smla {

// The plan of one forward call whose arguments have passed the checks: the
// kernel, the split count and the workspace layout. Queries the device's SM
// count only for the automatic split plan (num_splits == 0).
smla_status plan_forward(int T, int H, int D_qk, int D_v, int topk, int kv_dtype, int dot_precision,
                         int num_splits, int kernel, FwdPlan *out)
{
    const bool kv_fp8 = kv_dtype == SMLA_KV_FP8_E4M3;
    const bool bf16_dots = kv_fp8 && dot_precision != SMLA_DOT_FP8; // bf16 q . dequantized K
    Path path = choose_path(H, D_qk, D_v, kv_fp8, !bf16_dots, kernel);
    if ((path == Path::Wide) && num_splits > 1)
        path = Path::Mma; // the 128-head kernels do not split the top-k list
    int S = num_splits;
    if (S == 0) {
        int sms = 0;
        if (const cudaError_t e = current_sm_count(&sms); e != cudaSuccess)
            return cuda_status(e);
        S = plan_splits(T, H, topk, sms, path);
        if (bf16_dots && S > kClusterMaxSplits)
            S = kClusterMaxSplits;
    }
    if (S > kClusterMaxSplits && (int64_t)T * (H / 16) > kTicketSlots)
        return SMLA_ERR_UNSUPPORTED;
    // 128 heads: in the automatic plan the rows' (row, key tile) sequence is
    // spread over pairs of CTAs, one pair per two SMs when the rows outnumber
    // them (shared rows merge through the workspace's tickets; a CTA's tiles
    // stay below 2^30); with an explicit single split, the first kernels, or
    // no keys, one pair per row
    int pairs = 0;
    bool shared_rows = false;
    if (path == Path::Wide) {
        const int64_t rows = (int64_t)T * (H / 128);
        const int64_t ntiles = (topk + 63) / 64;
        pairs = (int)rows;
        int sms = 0;
        if (num_splits == 0 && kernel != SMLA_KERNEL_TCGEN05_BASIC && topk > 0 && rows * 2 <= kTicketSlots) {
            if (const cudaError_t e = current_sm_count(&sms); e != cudaSuccess)
                return cuda_status(e);
            // (128 rows on 76 pairs: 104 us spread against 107 us with one
            // pair per row and its second wave 68% full)
            const int64_t P = sms / 2;
            if (P > 0 && rows > P && rows * ntiles / P + ntiles < (int64_t(1) << 30)) {
                pairs = (int)P;
                shared_rows = rows % pairs != 0;
            }
        }
    }
    out->path = static_cast<int>(path);
    out->S = S;
    out->bf16_dots = bf16_dots;
    out->wide_pairs = pairs;
    out->layout = workspace_layout(T, H, D_qk, D_v, S, path == Path::Wide, shared_rows ? pairs : 0);
    out->uses_tickets = S > kClusterMaxSplits || shared_rows;
    return SMLA_OK;
}

} // namespace smla

namespace smla {

WorkspaceLayout workspace_layout(int T, int H, int D_qk, int D_v, int S, bool wide, int wide_pairs)
{
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    WorkspaceLayout w{};
    if (wide) {
        // after the merge-counter region, which must stay zero between calls
        w.q8 = up((size_t)kTicketSlots * sizeof(int));
        w.q8_rope = up(w.q8 + (size_t)T * H * 512);
        w.q_scale = up(w.q8_rope + (size_t)T * H * (D_qk - 512));
        w.total = up(w.q_scale + (size_t)T * H * sizeof(float));
        if (wide_pairs > 0) {
            // two partial slots per pair and value half: 256 dims x 128 heads binary16 and 128 lse
            w.wide_part_lse = w.total;
            w.wide_part = up(w.wide_part_lse + (size_t)wide_pairs * 2 * 2 * 128 * sizeof(float));
            w.total = up(w.wide_part + (size_t)wide_pairs * 2 * 2 * 128 * 256 * sizeof(uint16_t));
        }
        return w;
    }
    if (S <= kClusterMaxSplits)
        return w;
    w.tickets = 0;
    w.part_lse = up((size_t)kTicketSlots * sizeof(int));
    w.part_o16 = up(w.part_lse + (size_t)T * S * H * sizeof(float));
    w.total = up(w.part_o16 + (size_t)T * S * H * D_v * sizeof(uint16_t));
    return w;
}

} // namespace smla

extern "C" {

SMLA_API const char *smla_status_string(int status)
{
    switch (status) {
    case SMLA_OK:
        return "SMLA_OK";
    case SMLA_ERR_NULL_POINTER:
        return "SMLA_ERR_NULL_POINTER: a required pointer is NULL";
    case SMLA_ERR_BAD_SHAPE:
        return "SMLA_ERR_BAD_SHAPE: a size is negative or inconsistent";
    case SMLA_ERR_BAD_DTYPE:
        return "SMLA_ERR_BAD_DTYPE: unknown dtype or precision, or an invalid pairing";
    case SMLA_ERR_MISALIGNED:
        return "SMLA_ERR_MISALIGNED: a pointer lacks the required alignment";
    case SMLA_ERR_UNSUPPORTED:
        return "SMLA_ERR_UNSUPPORTED: no kernel for this shape / precision";
    case SMLA_ERR_WORKSPACE_TOO_SMALL:
        return "SMLA_ERR_WORKSPACE_TOO_SMALL: workspace below sparse_mla_fwd_workspace_size()";
    case SMLA_ERR_CUDA:
        return "SMLA_ERR_CUDA: CUDA runtime error";
    default:
        return "SMLA_ERR_UNKNOWN";
    }
}

SMLA_API int smla_version(void) { return (1 << 16) | 1; }

SMLA_API const char *smla_last_error_string(void)
{
    return t_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(t_last_cuda_error);
}

SMLA_API int smla_plan_num_splits(int T, int H, int D_qk, int topk, int kv_dtype, int sm_count)
{
    (void)D_qk;
    (void)kv_dtype;
    if (T < 0 || H <= 0 || H % 16 != 0 || topk < 0 || sm_count <= 0)
        return 0;
    const bool fp8 = kv_dtype == SMLA_KV_FP8_E4M3;
    return plan_splits(T, H, topk, sm_count, choose_path(H, D_qk, 512, fp8, fp8, SMLA_KERNEL_AUTO));
}

SMLA_API size_t sparse_mla_fwd_workspace_size(int T, int H, int D_qk, int D_v, int topk, int kv_dtype,
                                              int num_splits)
{
    if (T < 0 || topk < 0 || num_splits < 0 || num_splits > kMaxSplits || !shape_supported(H, D_qk, D_v) ||
        (kv_dtype != SMLA_KV_BF16 && kv_dtype != SMLA_KV_FP8_E4M3))
        return (size_t)-1;
    // the most any dot precision valid for this cache needs
    size_t most = 0;
    const int dots[3] = {SMLA_DOT_AUTO, SMLA_DOT_BF16, SMLA_DOT_FP8};
    for (int dp : dots) {
        if (dp == SMLA_DOT_FP8 && kv_dtype != SMLA_KV_FP8_E4M3)
            continue;
        smla::FwdPlan pl;
        if (smla::plan_forward(T, H, D_qk, D_v, topk, kv_dtype, dp, num_splits, SMLA_KERNEL_AUTO, &pl) != SMLA_OK)
            return (size_t)-1;
        if (pl.layout.total > most)
            most = pl.layout.total;
    }
    return most;
}

SMLA_API size_t sparse_mla_fwd_ex_workspace_size(const smla_fwd_params *p)
{
    if (p == nullptr || p->size < offsetof(smla_fwd_params, kernel))
        return (size_t)-1;
    const int kernel = p->size >= sizeof(smla_fwd_params) ? p->kernel : SMLA_KERNEL_AUTO;
    const bool q8 = p->q_scale != nullptr;
    const int dot = q8 ? SMLA_DOT_FP8 : p->dot_precision;
    if (p->T < 0 || p->topk < 0 || p->num_splits < 0 || p->num_splits > kMaxSplits ||
        !shape_supported(p->H, p->D_qk, p->D_v) ||
        (p->kv_dtype != SMLA_KV_BF16 && p->kv_dtype != SMLA_KV_FP8_E4M3) ||
        (dot != SMLA_DOT_AUTO && dot != SMLA_DOT_BF16 && dot != SMLA_DOT_FP8) ||
        (dot == SMLA_DOT_FP8 && p->kv_dtype != SMLA_KV_FP8_E4M3) ||
        (kernel != SMLA_KERNEL_AUTO && kernel != SMLA_KERNEL_WARP_MMA && kernel != SMLA_KERNEL_TCGEN05_BASIC))
        return (size_t)-1;
    if (p->T == 0)
        return 0;
    smla::FwdPlan pl;
    if (smla::plan_forward(p->T, p->H, p->D_qk, p->D_v, p->topk, p->kv_dtype, dot, p->num_splits, kernel, &pl) !=
        SMLA_OK)
        return (size_t)-1;
    return pl.layout.total;
}

// The forward for a bf16 q, or (q_fp8_in) for E4M3 codes of q with one
// per-tensor scale q_scale_in.
static smla_status fwd_impl(const void *q, bool q_fp8_in, const float *q_scale_in, const void *kv_cache,
                            int kv_dtype, const float *kv_scale, const int32_t *indices, int T, int H, int D_qk,
                            int D_v, int64_t num_slots, int topk, float scale, int dot_precision, void *out,
                            float *lse, void *workspace, size_t workspace_bytes, int num_splits,
                            smla_stream_t stream, const float *sinks = nullptr, int kernel = SMLA_KERNEL_AUTO)
{
    // 1. pointers
    if (kv_cache == nullptr || ((q == nullptr || out == nullptr) && T > 0) ||
        (indices == nullptr && (int64_t)T * topk > 0) || (q_fp8_in && q_scale_in == nullptr))
        return SMLA_ERR_NULL_POINTER;
    if (kv_dtype == SMLA_KV_FP8_E4M3 && kv_scale == nullptr)
        return SMLA_ERR_NULL_POINTER;
    // 2. sizes
    if (T < 0 || H <= 0 || D_qk <= 0 || D_v <= 0 || D_v > D_qk || num_slots < 0 || topk < 0 ||
        num_splits < 0)
        return SMLA_ERR_BAD_SHAPE;
    // 3. dtypes and their pairing
    if (kv_dtype != SMLA_KV_BF16 && kv_dtype != SMLA_KV_FP8_E4M3)
        return SMLA_ERR_BAD_DTYPE;
    if (dot_precision != SMLA_DOT_AUTO && dot_precision != SMLA_DOT_BF16 && dot_precision != SMLA_DOT_FP8)
        return SMLA_ERR_BAD_DTYPE;
    const bool fp8_dots = dot_precision == SMLA_DOT_FP8;
    if (fp8_dots && kv_dtype != SMLA_KV_FP8_E4M3)
        return SMLA_ERR_BAD_DTYPE;
    // 4. the shapes the library has kernels for
    if (!shape_supported(H, D_qk, D_v))
        return SMLA_ERR_UNSUPPORTED;
    if (num_splits > kMaxSplits)
        return SMLA_ERR_UNSUPPORTED;
    if (kernel != SMLA_KERNEL_AUTO && kernel != SMLA_KERNEL_WARP_MMA && kernel != SMLA_KERNEL_TCGEN05_BASIC)
        return SMLA_ERR_BAD_SHAPE;
    // 5. alignment
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(indices, 4) ||
        (lse != nullptr && !aligned(lse, 4)) || (kv_scale != nullptr && !aligned(kv_scale, 4)) ||
        (q_scale_in != nullptr && !aligned(q_scale_in, 4)) || (sinks != nullptr && !aligned(sinks, 4)))
        return SMLA_ERR_MISALIGNED;
    if (T == 0)
        return SMLA_OK;
    // 6. split plan and workspace
    smla::FwdPlan plan;
    if (const smla_status st = smla::plan_forward(T, H, D_qk, D_v, topk, kv_dtype, dot_precision, num_splits,
                                                  kernel, &plan);
        st != SMLA_OK)
        return st;
    const Path path = static_cast<Path>(plan.path);
    const int S = plan.S;
    const bool bf16_dots = plan.bf16_dots;
    const smla::WorkspaceLayout wl = plan.layout;
    if (wl.total > 0) {
        if (workspace == nullptr)
            return SMLA_ERR_NULL_POINTER;
        if (workspace_bytes < wl.total)
            return SMLA_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(workspace, 256))
            return SMLA_ERR_MISALIGNED;
    }

    const bool wide = path == Path::Wide;
    smla::FwdArgs a{};
    a.q = q;
    a.kv = kv_cache;
    a.kv_scale = kv_scale;
    a.indices = indices;
    a.out = out;
    a.lse = lse;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const bool split_merge = S > kClusterMaxSplits && !wide;
    a.part_o16 = split_merge ? reinterpret_cast<uint16_t *>(ws + wl.part_o16) : nullptr;
    a.part_lse = split_merge ? reinterpret_cast<float *>(ws + wl.part_lse) : nullptr;
    a.tickets = split_merge ? reinterpret_cast<int *>(ws + wl.tickets) : nullptr;
    a.q8 = wide ? ws + wl.q8 : nullptr;
    a.q8_rope = wide ? ws + wl.q8_rope : nullptr;
    a.q_scale = wide ? reinterpret_cast<float *>(ws + wl.q_scale) : nullptr;
    a.num_slots = num_slots;
    a.T = T;
    a.H = H;
    a.D_qk = D_qk;
    a.D_v = D_v;
    a.topk = topk;
    a.S = S;
    a.keys_per_split = topk > 0 ? keys_per_split(topk, S, tile_keys(path)) : tile_keys(path);
    a.scale = scale;
    a.kv_fp8 = kv_dtype == SMLA_KV_FP8_E4M3;
    a.bf16_dots = bf16_dots;
    a.sinks = sinks;
    a.q_fp8_in = q_fp8_in;
    a.q_scale_in = q_scale_in;
    a.wide_pairs = plan.wide_pairs;
    a.wide_part = wl.wide_part ? reinterpret_cast<uint16_t *>(ws + wl.wide_part) : nullptr;
    a.wide_part_lse = wl.wide_part ? reinterpret_cast<float *>(ws + wl.wide_part_lse) : nullptr;
    a.wide_tickets = wl.wide_part ? reinterpret_cast<int *>(ws) : nullptr;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (path) {
    case Path::Umma16:
        return cuda_status(smla::launch_fwd_umma16(a, st));
    case Path::Lean16:
        return cuda_status(smla::launch_fwd_lean16(a, st));
    case Path::Wide:
        return cuda_status(smla::launch_fwd_wide(a, st));
    default:
        return cuda_status(smla::launch_fwd_mma(a, st));
    }
}

SMLA_API smla_status sparse_mla_fwd(const void *q, const void *kv_cache, int kv_dtype, const float *kv_scale,
                                    const int32_t *indices, int T, int H, int D_qk, int D_v, int64_t num_slots,
                                    int topk, float scale, int dot_precision, void *out, float *lse,
                                    void *workspace, size_t workspace_bytes, int num_splits,
                                    smla_stream_t stream)
{
    return fwd_impl(q, false, nullptr, kv_cache, kv_dtype, kv_scale, indices, T, H, D_qk, D_v, num_slots, topk,
                    scale, dot_precision, out, lse, workspace, workspace_bytes, num_splits, stream);
}

SMLA_API smla_status sparse_mla_fwd_ex(const smla_fwd_params *p)
{
    if (p == nullptr)
        return SMLA_ERR_NULL_POINTER;
    // callers built against ABI 1.0 pass the structure without `kernel`
    if (p->size < offsetof(smla_fwd_params, kernel))
        return SMLA_ERR_BAD_SHAPE; // a caller built against a different layout
    const int kernel = p->size >= sizeof(smla_fwd_params) ? p->kernel : SMLA_KERNEL_AUTO;
    const bool q8 = p->q_scale != nullptr;
    if (q8 && (p->kv_dtype != SMLA_KV_FP8_E4M3 ||
               (p->dot_precision != SMLA_DOT_AUTO && p->dot_precision != SMLA_DOT_FP8)))
        return SMLA_ERR_BAD_DTYPE; // E4M3 q codes are dotted in fp8 with an E4M3 cache
    return fwd_impl(p->q, q8, p->q_scale, p->kv_cache, p->kv_dtype, p->kv_scale, p->indices, p->T, p->H, p->D_qk,
                    p->D_v, p->num_slots, p->topk, p->scale, q8 ? SMLA_DOT_FP8 : p->dot_precision, p->out, p->lse,
                    p->workspace, p->workspace_bytes, p->num_splits, p->stream, p->sinks, kernel);
}

SMLA_API smla_status sparse_mla_fwd_q8(const void *q8, const float *q_scale, const void *kv_cache,
                                       const float *kv_scale, const int32_t *indices, int T, int H, int D_qk,
                                       int D_v, int64_t num_slots, int topk, float scale, void *out, float *lse,
                                       void *workspace, size_t workspace_bytes, int num_splits,
                                       smla_stream_t stream)
{
    return fwd_impl(q8, true, q_scale, kv_cache, SMLA_KV_FP8_E4M3, kv_scale, indices, T, H, D_qk, D_v, num_slots,
                    topk, scale, SMLA_DOT_FP8, out, lse, workspace, workspace_bytes, num_splits, stream);
}

SMLA_API smla_status smla_device_error(int *code, int reset)
{
    if (code == nullptr)
        return SMLA_ERR_NULL_POINTER;
    int c16 = 0, cw = 0, cp = 0, cg = 0, cl = 0;
    if (const cudaError_t e = smla::read_umma_error(&c16, reset != 0); e != cudaSuccess)
        return cuda_status(e);
    if (const cudaError_t e = smla::read_lean_error(&cl, reset != 0); e != cudaSuccess)
        return cuda_status(e);
    if (const cudaError_t e = smla::read_probe_error(&cg, reset != 0); e != cudaSuccess)
        return cuda_status(e);
    if (const cudaError_t e = smla::read_wide_error(&cw, reset != 0); e != cudaSuccess)
        return cuda_status(e);
    if (const cudaError_t e = smla::read_producer_error(&cp, reset != 0); e != cudaSuccess)
        return cuda_status(e);
    *code = c16 | cw | cp | cg | cl;
    return SMLA_OK;
}

SMLA_API smla_status smla_fused_qk_rope_cache(const void *ql_nope, int64_t ql_stride_t, int64_t ql_stride_h,
                                              const void *q_pe, int64_t qpe_stride_t, int64_t qpe_stride_h,
                                              const void *kv_c, int64_t kvc_stride_t, const void *k_pe,
                                              int64_t kpe_stride_t, const int64_t *positions,
                                              const float *cos_sin_cache, int64_t max_position, int is_neox,
                                              const int64_t *slot_mapping, void *kv_cache, int kv_dtype,
                                              int64_t num_slots, const float *kv_scale, void *q_out,
                                              int q_out_dtype, const float *q_scale, int T, int H,
                                              smla_stream_t stream)
{
    // a token's H + 1 rows run as blocks of 8 along the grid's y (at most 65535)
    constexpr int kMaxProducerHeads = 65535 * 8 - 1;
    if (T < 0 || H < 0 || num_slots < 0 || max_position < 0 || ql_stride_t < 0 || ql_stride_h < 0 ||
        qpe_stride_t < 0 || qpe_stride_h < 0 || kvc_stride_t < 0 || kpe_stride_t < 0)
        return SMLA_ERR_BAD_SHAPE;
    if ((kv_dtype != SMLA_KV_BF16 && kv_dtype != SMLA_KV_FP8_E4M3) ||
        (q_out_dtype != SMLA_KV_BF16 && q_out_dtype != SMLA_KV_FP8_E4M3))
        return SMLA_ERR_BAD_DTYPE;
    if (T == 0)
        return SMLA_OK;
    const bool qrows = H > 0;
    if ((qrows && (ql_nope == nullptr || q_pe == nullptr || q_out == nullptr)) || kv_c == nullptr ||
        k_pe == nullptr || positions == nullptr || cos_sin_cache == nullptr || slot_mapping == nullptr ||
        kv_cache == nullptr || (kv_dtype == SMLA_KV_FP8_E4M3 && kv_scale == nullptr) ||
        (qrows && q_out_dtype == SMLA_KV_FP8_E4M3 && q_scale == nullptr))
        return SMLA_ERR_NULL_POINTER;
    if (max_position == 0 || H > kMaxProducerHeads)
        return SMLA_ERR_BAD_SHAPE;
    // latent rows move as 16-byte vectors, rope pairs as 4-byte words
    if (ql_stride_t % 8 != 0 || ql_stride_h % 8 != 0 || kvc_stride_t % 8 != 0 || qpe_stride_t % 2 != 0 ||
        qpe_stride_h % 2 != 0 || kpe_stride_t % 2 != 0)
        return SMLA_ERR_MISALIGNED;
    if ((qrows && (!aligned(ql_nope, 16) || !aligned(q_pe, 4) || !aligned(q_out, 16))) || !aligned(kv_c, 16) ||
        !aligned(k_pe, 4) || !aligned(kv_cache, 16) || !aligned(positions, 8) || !aligned(slot_mapping, 8) ||
        !aligned(cos_sin_cache, 4) || (kv_scale != nullptr && !aligned(kv_scale, 4)) ||
        (q_scale != nullptr && !aligned(q_scale, 4)))
        return SMLA_ERR_MISALIGNED;
    smla::FusedProducerArgs a;
    a.ql_nope = ql_nope;
    a.ql_stride_t = ql_stride_t;
    a.ql_stride_h = ql_stride_h;
    a.q_pe = q_pe;
    a.qpe_stride_t = qpe_stride_t;
    a.qpe_stride_h = qpe_stride_h;
    a.kv_c = kv_c;
    a.kvc_stride_t = kvc_stride_t;
    a.k_pe = k_pe;
    a.kpe_stride_t = kpe_stride_t;
    a.positions = positions;
    a.cos_sin_cache = cos_sin_cache;
    a.max_position = max_position;
    a.slot_mapping = slot_mapping;
    a.kv_cache = kv_cache;
    a.num_slots = num_slots;
    a.kv_scale = kv_scale;
    a.q_out = q_out;
    a.q_scale = q_scale;
    a.T = T;
    a.H = H;
    a.is_neox = is_neox != 0;
    a.q_out_fp8 = q_out_dtype == SMLA_KV_FP8_E4M3;
    a.cache_fp8 = kv_dtype == SMLA_KV_FP8_E4M3;
    return cuda_status(smla::launch_fused_producer(a, reinterpret_cast<cudaStream_t>(stream)));
}

SMLA_API smla_status smla_compute_fp8_scale(const void *x, int64_t n, float *scale_out, smla_stream_t stream)
{
    if ((x == nullptr && n > 0) || scale_out == nullptr)
        return SMLA_ERR_NULL_POINTER;
    if (n < 0)
        return SMLA_ERR_BAD_SHAPE;
    if (!aligned(x, 16) || !aligned(scale_out, 4))
        return SMLA_ERR_MISALIGNED;
    int sms = 0;
    if (const cudaError_t e = current_sm_count(&sms); e != cudaSuccess)
        return cuda_status(e);
    return cuda_status(smla::launch_fp8_scale(x, n, scale_out, sms, reinterpret_cast<cudaStream_t>(stream)));
}

SMLA_API smla_status smla_fp8_cache_write(const void *src, const int64_t *slot_mapping, int64_t N, int D,
                                          const float *kv_scale, void *kv_cache, int64_t num_slots,
                                          smla_stream_t stream)
{
    if (src == nullptr || slot_mapping == nullptr || kv_scale == nullptr || kv_cache == nullptr)
        return SMLA_ERR_NULL_POINTER;
    if (N < 0 || D <= 0 || D % 8 != 0 || num_slots < 0)
        return SMLA_ERR_BAD_SHAPE;
    if (!aligned(src, 16) || !aligned(kv_cache, 8) || !aligned(slot_mapping, 8) || !aligned(kv_scale, 4))
        return SMLA_ERR_MISALIGNED;
    return cuda_status(smla::launch_fp8_cache_write(src, slot_mapping, N, D, kv_scale, kv_cache, num_slots,
                                                    reinterpret_cast<cudaStream_t>(stream)));
}

SMLA_API smla_status smla_gather_probe(const void *pool, int64_t num_rows, int row_bytes, const int32_t *indices,
                                       int64_t n_indices, int ctas_per_sm, int stages, int hold_ns, int pair_mode,
                                       int issue_warps, int copy_mode, uint32_t *checksum, smla_stream_t stream)
{
    if (pool == nullptr || checksum == nullptr || (indices == nullptr && n_indices > 0))
        return SMLA_ERR_NULL_POINTER;
    if (num_rows < 0 || n_indices < 0 || row_bytes < 16 || row_bytes > 1024 || row_bytes % 16 != 0 ||
        ctas_per_sm < 1 || ctas_per_sm > 4 || stages < 1 || stages > 8 || hold_ns < 0 ||
        pair_mode < 0 || pair_mode > 3 || issue_warps < 0 || issue_warps > 8 || copy_mode < 0 || copy_mode > 1)
        return SMLA_ERR_BAD_SHAPE;
    const int copies = (pair_mode == 1 || pair_mode == 2 ? 8 : 16) * ((row_bytes + 127) / 128);
    if (issue_warps > 0 && (copies + issue_warps - 1) / issue_warps > 32)
        return SMLA_ERR_BAD_SHAPE;
    if ((pair_mode && ctas_per_sm != 1) || (copy_mode == 1 && (pair_mode != 0 || issue_warps != 0)))
        return SMLA_ERR_UNSUPPORTED;
    if (!aligned(pool, 16) || !aligned(indices, 4) || !aligned(checksum, 4))
        return SMLA_ERR_MISALIGNED;
    int sms = 0;
    if (const cudaError_t e = current_sm_count(&sms); e != cudaSuccess)
        return cuda_status(e);
    const cudaError_t e = smla::launch_gather_probe(pool, num_rows, row_bytes, indices, n_indices, ctas_per_sm,
                                                    stages, hold_ns, pair_mode, issue_warps, copy_mode, checksum, sms,
                                                    reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue)
        return SMLA_ERR_UNSUPPORTED; // the stages do not fit ctas_per_sm CTAs on an SM
    return cuda_status(e);
}

SMLA_API smla_status smla_l2_read_probe(const void *buf, int64_t bytes, int reps, uint32_t *checksum, int blocks,
                                        smla_stream_t stream)
{
    if (buf == nullptr || checksum == nullptr)
        return SMLA_ERR_NULL_POINTER;
    if (bytes < 16 || bytes % 16 != 0 || reps < 1 || blocks < 1)
        return SMLA_ERR_BAD_SHAPE;
    if (!aligned(buf, 16) || !aligned(checksum, 4))
        return SMLA_ERR_MISALIGNED;
    return cuda_status(smla::launch_l2_read_probe(buf, bytes, reps, checksum, blocks,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

SMLA_API smla_status smla_validate_indices(const int32_t *indices, int T, int topk, int64_t num_slots,
                                           int *bad_count, smla_stream_t stream)
{
    if ((indices == nullptr && (int64_t)T * topk > 0) || bad_count == nullptr)
        return SMLA_ERR_NULL_POINTER;
    if (T < 0 || topk < 0 || num_slots < 0)
        return SMLA_ERR_BAD_SHAPE;
    if (!aligned(indices, 4) || !aligned(bad_count, 4))
        return SMLA_ERR_MISALIGNED;
    int sms = 0;
    if (const cudaError_t e = current_sm_count(&sms); e != cudaSuccess)
        return cuda_status(e);
    return cuda_status(smla::launch_validate_indices(indices, (int64_t)T * topk, num_slots, bad_count, sms,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

} // extern "C"
