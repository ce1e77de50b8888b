// sparse_mla_fwd_no_alloc: the sparse MLA forward for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: a serving engine that has
// reserved nearly all of HBM for its KV-cache pool up front has nothing left
// to cudaMalloc from, and a host framework that loads this library as a
// plug-in may only let it use the buffers it hands over. For them the
// workspace that sparse_mla_fwd needs (the merge counters and partial results
// when a row's top-k list is split more than 8 ways, or the quantized q of the
// 128-head E4M3 kernel) lives in a fixed array inside the library instead.
//
// The array is a file-scope device variable: every GPU that loads the library
// holds it until the process exits. Host code cannot use its name as an
// address (it is a host-side stand-in), so every call looks the device address
// up with cudaGetSymbolAddress, with the call's device current (a lookup
// cached across calls could outlive a context reset that moves the module).
// The call's workspace need comes from the same plan the forward itself
// makes (its dot precision and split count included), so a call that needs no
// workspace never touches the array. A call that merges through the array's
// counters clears them on its stream first. All calls share the array, so
// calls that overlap on the GPU (different streams, no ordering between them)
// race on it.
#include "../../include/sparse_mla.h"
#include "smla_internal.h"

#include <cuda_runtime.h>

namespace {

constexpr size_t kScratchBytes = SMLA_NO_ALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_no_alloc_scratch[kScratchBytes];

} // namespace

extern "C" SMLA_API smla_status sparse_mla_fwd_no_alloc(const void *q, const void *kv_cache, int kv_dtype,
                                                        const float *kv_scale, const int32_t *indices, int T, int H,
                                                        int D_qk, int D_v, int64_t num_slots, int topk, float scale,
                                                        int dot_precision, void *out, float *lse, int num_splits,
                                                        smla_stream_t stream)
{
    smla_fwd_params p{};
    p.size = sizeof(smla_fwd_params);
    p.q = q;
    p.kv_cache = kv_cache;
    p.kv_dtype = kv_dtype;
    p.kv_scale = kv_scale;
    p.indices = indices;
    p.T = T;
    p.H = H;
    p.D_qk = D_qk;
    p.D_v = D_v;
    p.num_slots = num_slots;
    p.topk = topk;
    p.scale = scale;
    p.dot_precision = dot_precision;
    p.out = out;
    p.lse = lse;
    p.num_splits = num_splits;
    p.stream = stream;
    p.kernel = SMLA_KERNEL_AUTO;
    size_t need = sparse_mla_fwd_ex_workspace_size(&p);
    if (need == (size_t)-1 || need == 0) // invalid (the full checks report why), or no workspace needed
        return sparse_mla_fwd_ex(&p);
    smla::FwdPlan plan;
    if (const smla_status st = smla::plan_forward(T, H, D_qk, D_v, topk, kv_dtype, dot_precision, num_splits,
                                                  SMLA_KERNEL_AUTO, &plan);
        st != SMLA_OK)
        return st;
    if (need > kScratchBytes && plan.wide_pairs > 0 && num_splits == 0) {
        // the 128-head kernel's automatic plan spreads rows over CTA pairs and
        // keeps partials of the rows they share; one pair per row needs only
        // the quantized q, so run that plan when it fits
        p.kernel = SMLA_KERNEL_TCGEN05_BASIC;
        need = sparse_mla_fwd_ex_workspace_size(&p);
        if (const smla_status st = smla::plan_forward(T, H, D_qk, D_v, topk, kv_dtype, dot_precision, num_splits,
                                                      p.kernel, &plan);
            st != SMLA_OK)
            return st;
    }
    if (need > kScratchBytes)
        return SMLA_ERR_WORKSPACE_TOO_SMALL;
    void *ws = nullptr;
    if (cudaGetSymbolAddress(&ws, g_no_alloc_scratch) != cudaSuccess)
        return SMLA_ERR_CUDA;
    // merge counters must start at zero whatever an earlier call left there
    if (plan.uses_tickets &&
        cudaMemsetAsync(ws, 0, (size_t)smla::kTicketSlots * sizeof(int), reinterpret_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
        return SMLA_ERR_CUDA;
    p.workspace = ws;
    p.workspace_bytes = kScratchBytes;
    return sparse_mla_fwd_ex(&p);
}
