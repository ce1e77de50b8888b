// Companion kernels of the sparse MLA forward (sm_103a):
//   - per-tensor fp8 scale: amax(|x|) / 448 over a bf16 tensor,
//   - the quantizing cache write: cache[slot] = E4M3(x / scale),
//   - an index validator that counts entries outside {-1} U [0, num_slots).
//
// Source: "Fuse decode QK-RoPE + Q-concat + KV-concat + KV-cache write for
// sparse MLA" (vLLM PR 47757), Summary and Test plan — the fp8 KV-cache write
// (concat_and_cache_mla) and the scaled_fp8_quant convention it is checked
// against (stored = x / scale, tested with a non-unit scale).
// All three kernels are HBM-streaming: 16-byte vector loads, grid-stride
// loops sized to the SM count.
#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

// amax over bf16 values as the bit pattern of a non-negative float; the bit
// patterns of non-negative floats order like the values, so an integer
// atomicMax reduces them. NaN is skipped (fmaxf ignores a NaN operand).
__global__ void __launch_bounds__(256) amax_bf16_kernel(const __nv_bfloat16 *__restrict__ x, int64_t n,
                                                        unsigned int *__restrict__ cell)
{
    float m = 0.f;
    const int64_t nvec = n / 8;
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const uint4 u = __ldcs(xv + i);
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(b[e]);
            m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    for (int64_t i = nvec * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        m = fmaxf(m, fabsf(__bfloat162float(x[i])));
    m = warp_max(m);
    __shared__ float wm[8];
    if ((threadIdx.x & 31) == 0)
        wm[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = wm[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            b = fmaxf(b, wm[w]);
        atomicMax(cell, __float_as_uint(b));
    }
}

// cell holds amax bits; replace them with the scale amax / 448 (1.0 if 0).
__global__ void amax_to_scale_kernel(float *cell)
{
    const float amax = __uint_as_float(*reinterpret_cast<unsigned int *>(cell));
    *cell = (amax == 0.f) ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// One warp per source row; each lane converts 8 values (16 B in, 8 B out).
__global__ void __launch_bounds__(256) fp8_cache_write_kernel(const __nv_bfloat16 *__restrict__ src,
                                                              const int64_t *__restrict__ slot_mapping, int64_t N,
                                                              int D, const float *__restrict__ kv_scale,
                                                              uint8_t *__restrict__ cache, int64_t num_slots)
{
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= N)
        return;
    const int64_t slot = slot_mapping[row];
    if (slot < 0 || slot >= num_slots)
        return;
    const float s = *kv_scale;
    const E4m3Recip inv = e4m3_recip(s);
    const uint4 *in = reinterpret_cast<const uint4 *>(src + row * D);
    uint2 *outp = reinterpret_cast<uint2 *>(cache + slot * D);
    for (int v = lane; v < D / 8; v += 32) {
        const uint4 u = in[v];
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
        const float2 f0 = __bfloat1622float2(b[0]), f1 = __bfloat1622float2(b[1]);
        const float2 f2 = __bfloat1622float2(b[2]), f3 = __bfloat1622float2(b[3]);
        uint2 r;
        r.x = quant4_e4m3(f0.x, f0.y, f1.x, f1.y, s, inv);
        r.y = quant4_e4m3(f2.x, f2.y, f3.x, f3.y, s, inv);
        outp[v] = r;
    }
}

__global__ void __launch_bounds__(256) validate_indices_kernel(const int32_t *__restrict__ idx, int64_t n,
                                                               int64_t num_slots, int *__restrict__ bad)
{
    int cnt = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int32_t v = idx[i];
        cnt += (v != -1) && (v < 0 || (int64_t)v >= num_slots);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if ((threadIdx.x & 31) == 0 && cnt)
        atomicAdd(bad, cnt);
}

int grid_for(int64_t work_items, int threads, int sm_count, int per_sm)
{
    int64_t b = (work_items + threads - 1) / threads;
    const int64_t cap = (int64_t)(sm_count > 0 ? sm_count : 1) * per_sm;
    if (b > cap)
        b = cap;
    return (int)(b > 0 ? b : 1);
}

} // namespace

cudaError_t launch_fp8_scale(const void *x, int64_t n, float *scale_out, int sm_count, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(scale_out, 0, sizeof(float), stream);
    if (e != cudaSuccess)
        return e;
    if (n > 0) {
        const int grid = grid_for((n + 7) / 8, 256, sm_count, 8);
        amax_bf16_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x), n,
                                                   reinterpret_cast<unsigned int *>(scale_out));
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    amax_to_scale_kernel<<<1, 1, 0, stream>>>(scale_out);
    return cudaGetLastError();
}

cudaError_t launch_fp8_cache_write(const void *src, const int64_t *slot_mapping, int64_t N, int D,
                                   const float *kv_scale, void *cache, int64_t num_slots, cudaStream_t stream)
{
    if (N == 0)
        return cudaSuccess;
    const int64_t blocks = (N * 32 + 255) / 256;
    fp8_cache_write_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(src),
                                                                 slot_mapping, N, D, kv_scale,
                                                                 static_cast<uint8_t *>(cache), num_slots);
    return cudaGetLastError();
}

cudaError_t launch_validate_indices(const int32_t *indices, int64_t n, int64_t num_slots, int *bad_count,
                                    int sm_count, cudaStream_t stream)
{
    cudaError_t e = cudaMemsetAsync(bad_count, 0, sizeof(int), stream);
    if (e != cudaSuccess || n == 0)
        return e;
    const int grid = grid_for(n, 256, sm_count, 8);
    validate_indices_kernel<<<grid, 256, 0, stream>>>(indices, n, num_slots, bad_count);
    return cudaGetLastError();
}

} // namespace smla
