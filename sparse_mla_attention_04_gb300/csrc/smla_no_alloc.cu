// sparse_mla_fwd_no_alloc: the sparse MLA forward for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: a serving engine that has
// reserved nearly all of HBM for its KV-cache pool up front has nothing left
// to cudaMalloc from, and a host framework that loads this library as a
// plug-in may only let it use the buffers it hands over. For them the
// workspace that sparse_mla_fwd needs when a row's top-k list is split more
// than 8 ways lives in a fixed array inside the library instead.
//
// The array is a file-scope device variable: every GPU that loads the library
// holds it until the process exits. Host code cannot use its name as an
// address (it is a host-side stand-in), so the device address is looked up
// once per device with cudaGetSymbolAddress on the first call made with that
// device current. Each call clears the merge counters at the start of the
// array before launching; all calls share the array, so calls that overlap
// on the GPU (different streams, no ordering between them) race on it.
#include "../../include/sparse_mla.h"
#include "smla_internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr size_t kScratchBytes = SMLA_NO_ALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_no_alloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

} // namespace

extern "C" SMLA_API smla_status sparse_mla_fwd_no_alloc(const void *q, const void *kv_cache, int kv_dtype,
                                                        const float *kv_scale, const int32_t *indices, int T, int H,
                                                        int D_qk, int D_v, int64_t num_slots, int topk, float scale,
                                                        int dot_precision, void *out, float *lse, int num_splits,
                                                        smla_stream_t stream)
{
    if (T == 0 || num_splits < 0)
        return sparse_mla_fwd(q, kv_cache, kv_dtype, kv_scale, indices, T, H, D_qk, D_v, num_slots, topk, scale,
                              dot_precision, out, lse, nullptr, 0, num_splits, stream);
    const size_t need = sparse_mla_fwd_workspace_size(T, H, D_qk, D_v, topk, kv_dtype, num_splits);
    if (need == (size_t)-1) // invalid shape or plan: let the full checks report why
        return sparse_mla_fwd(q, kv_cache, kv_dtype, kv_scale, indices, T, H, D_qk, D_v, num_slots, topk, scale,
                              dot_precision, out, lse, nullptr, 0, num_splits, stream);
    if (need > kScratchBytes)
        return SMLA_ERR_WORKSPACE_TOO_SMALL;
    void *ws = nullptr;
    if (need > 0) {
        if (scratch_address(&ws) != cudaSuccess)
            return SMLA_ERR_CUDA;
        // the merge counters must start at zero whatever an earlier call left
        if (cudaMemsetAsync(ws, 0, (size_t)smla::kTicketSlots * sizeof(int),
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
            return SMLA_ERR_CUDA;
    }
    return sparse_mla_fwd(q, kv_cache, kv_dtype, kv_scale, indices, T, H, D_qk, D_v, num_slots, topk, scale,
                          dot_precision, out, lse, ws, need > 0 ? kScratchBytes : 0, num_splits, stream);
}
