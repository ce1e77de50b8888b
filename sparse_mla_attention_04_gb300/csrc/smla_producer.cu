// The fused producer step of sparse MLA decode: RoPE on the pre-RoPE q_pe and
// k_pe at each token's position, q_out = concat(ql_nope, RoPE(q_pe)) (bf16, or
// E4M3 codes of / q_scale), and the cache row concat(kv_c, RoPE(k_pe)) (bf16,
// or E4M3 codes of / kv_scale), in one pass over the inputs. sm_103a.
//
// Source: "[ROCm][MLA][Perf] Fuse decode QK-RoPE + Q-concat + KV-concat +
// KV-cache write for sparse MLA" — Summary (one kernel for main RoPE on
// q_pe/k_pe, the query concat, the KV concat and the fp8 cache write) and
// Test plan (parity with the split chain: bf16 q_out, scaled_fp8_quant of q
// with a per-tensor q_scale, concat_and_cache_mla of the rotated k_pe).
//
// The rotation of a pair (a, b) by theta is (a cos - b sin, b cos + a sin),
// in binary32 with each product and the difference or sum rounded (no fused
// multiply-add), then rounded to bf16: the split chain stores the rotated
// values as bf16 before quantizing them. neox pairs element i with i + 32,
// GPT-J pairs 2i with 2i + 1; the cos/sin cache row of a position holds the 32
// cosines, then the 32 sines, in binary32.
//
// Work: one warp per output row, i.e. per (token, head) of q_out plus one per
// token for its cache row; a block holds 8 rows of one token (blockIdx.x is
// the token, blockIdx.y the group of 8 rows), so no index is divided. A warp
// issues all its loads whose addresses do not depend on a loaded value before
// using any. The 512 latent columns move as
// 16-byte vectors (two per lane); the 64 rope columns as one rotary pair per
// lane. Per q row 1,152 bytes are read and 1,152 (bf16) or 576 (E4M3) written.
#include "smla_device.cuh"
#include "smla_internal.h"

#include <climits>

namespace smla {

__device__ int g_producer_error = 0; // bit 4: a position out of range; bit 8: a slot out of range

namespace {

constexpr int kDn = 512;  // latent columns
constexpr int kDr = 64;   // rope columns
constexpr int kD = kDn + kDr;
constexpr int kWarpsPerBlock = 8;

struct ProducerArgs {
    const __nv_bfloat16 *ql_nope;
    int64_t ql_st, ql_sh;
    const __nv_bfloat16 *q_pe;
    int64_t qp_st, qp_sh;
    const __nv_bfloat16 *kv_c;
    int64_t kc_st;
    const __nv_bfloat16 *k_pe;
    int64_t kp_st;
    const int64_t *positions;
    const float *cos_sin;
    int64_t max_position;
    const int64_t *slot_mapping;
    void *kv_cache;
    int64_t num_slots;
    const float *kv_scale;
    void *q_out;
    const float *q_scale;
    int T, H;
    bool neox, q_fp8, cache_fp8;
};

__device__ __forceinline__ float rot_a(float a, float b, float c, float s)
{
    return __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s));
}
__device__ __forceinline__ float rot_b(float a, float b, float c, float s)
{
    return __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, s));
}

// Eight bf16 values (a 16-byte vector) as eight E4M3 codes of x / s (inv = e4m3_recip(s)).
__device__ __forceinline__ uint2 quant8(const uint4 v, float s, const E4m3Recip &inv)
{
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&v);
    const float2 f0 = __bfloat1622float2(p[0]), f1 = __bfloat1622float2(p[1]);
    const float2 f2 = __bfloat1622float2(p[2]), f3 = __bfloat1622float2(p[3]);
    uint2 o;
    o.x = quant4_e4m3(f0.x, f0.y, f1.x, f1.y, s, inv);
    o.y = quant4_e4m3(f2.x, f2.y, f3.x, f3.y, s, inv);
    return o;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32, 8) fused_qk_rope_cache_kernel(const ProducerArgs a)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    const int j = blockIdx.y * kWarpsPerBlock + (threadIdx.x >> 5); // j < H: q row of head j; j == H: the cache row
    if (j > a.H)
        return;
    const bool qrow = j < a.H;
    // every load whose address does not depend on a loaded value is issued
    // before any is used: the row's latent vectors, its rope pair, the position
    // and (cache row) the slot
    const __nv_bfloat16 *nope = qrow ? a.ql_nope + t * a.ql_st + j * a.ql_sh : a.kv_c + t * a.kc_st;
    const __nv_bfloat16 *pe = qrow ? a.q_pe + t * a.qp_st + j * a.qp_sh : a.k_pe + t * a.kp_st;
    const uint4 *src4 = reinterpret_cast<const uint4 *>(nope);
    const uint4 v0 = __ldg(src4 + lane), v1 = __ldg(src4 + lane + 32);
    const int ia = a.neox ? lane : 2 * lane;
    const int ib = a.neox ? lane + kDr / 2 : 2 * lane + 1;
    float xa, xb;
    if (a.neox) {
        xa = __bfloat162float(pe[ia]);
        xb = __bfloat162float(pe[ib]);
    } else {
        const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162 *>(pe + ia);
        xa = __low2float(p2);
        xb = __high2float(p2);
    }
    const int64_t pos = __ldg(a.positions + t);
    const int64_t slot = qrow ? 0 : __ldg(a.slot_mapping + t);
    if (pos < 0 || pos >= a.max_position) {
        if (j == 0 && lane == 0)
            atomicOr(&g_producer_error, 4);
        return;
    }
    void *dst;
    bool fp8;
    const float *scale_p;
    if (qrow) {
        const int64_t r = (int64_t)t * a.H + j;
        fp8 = a.q_fp8;
        dst = fp8 ? static_cast<void *>(static_cast<uint8_t *>(a.q_out) + r * kD)
                  : static_cast<void *>(static_cast<__nv_bfloat16 *>(a.q_out) + r * kD);
        scale_p = a.q_scale;
    } else {
        if (slot < 0)
            return;
        if (slot >= a.num_slots) {
            if (lane == 0)
                atomicOr(&g_producer_error, 8);
            return;
        }
        fp8 = a.cache_fp8;
        dst = fp8 ? static_cast<void *>(static_cast<uint8_t *>(a.kv_cache) + slot * kD)
                  : static_cast<void *>(static_cast<__nv_bfloat16 *>(a.kv_cache) + slot * kD);
        scale_p = a.kv_scale;
    }
    const float s = fp8 ? __ldg(scale_p) : 1.0f;
    const float *row = a.cos_sin + pos * kDr;
    const float c = __ldg(row + lane), sn = __ldg(row + kDr / 2 + lane);
    const __nv_bfloat16 ra = __float2bfloat16_rn(rot_a(xa, xb, c, sn));
    const __nv_bfloat16 rb = __float2bfloat16_rn(rot_b(xa, xb, c, sn));

    if (!fp8) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        d4[lane] = v0;
        d4[lane + 32] = v1;
        __nv_bfloat16 *dr = static_cast<__nv_bfloat16 *>(dst) + kDn;
        if (a.neox) {
            dr[ia] = ra;
            dr[ib] = rb;
        } else {
            *reinterpret_cast<__nv_bfloat162 *>(dr + ia) = __halves2bfloat162(ra, rb);
        }
    } else {
        const E4m3Recip inv = e4m3_recip(s);
        uint2 *d2 = reinterpret_cast<uint2 *>(dst);
        d2[lane] = quant8(v0, s, inv);
        d2[lane + 32] = quant8(v1, s, inv);
        uint8_t *dr = static_cast<uint8_t *>(dst) + kDn;
        const uint16_t cab = (uint16_t)quant2_e4m3(__bfloat162float(ra), __bfloat162float(rb), s, inv);
        if (a.neox) {
            dr[ia] = (uint8_t)(cab & 0xFFu);
            dr[ib] = (uint8_t)(cab >> 8);
        } else {
            *reinterpret_cast<uint16_t *>(dr + ia) = cab;
        }
    }
}

} // namespace

cudaError_t launch_fused_producer(const FusedProducerArgs &f, cudaStream_t stream)
{
    ProducerArgs a;
    a.ql_nope = static_cast<const __nv_bfloat16 *>(f.ql_nope);
    a.ql_st = f.ql_stride_t;
    a.ql_sh = f.ql_stride_h;
    a.q_pe = static_cast<const __nv_bfloat16 *>(f.q_pe);
    a.qp_st = f.qpe_stride_t;
    a.qp_sh = f.qpe_stride_h;
    a.kv_c = static_cast<const __nv_bfloat16 *>(f.kv_c);
    a.kc_st = f.kvc_stride_t;
    a.k_pe = static_cast<const __nv_bfloat16 *>(f.k_pe);
    a.kp_st = f.kpe_stride_t;
    a.positions = f.positions;
    a.cos_sin = f.cos_sin_cache;
    a.max_position = f.max_position;
    a.slot_mapping = f.slot_mapping;
    a.kv_cache = f.kv_cache;
    a.num_slots = f.num_slots;
    a.kv_scale = f.kv_scale;
    a.q_out = f.q_out;
    a.q_scale = f.q_scale;
    a.T = f.T;
    a.H = f.H;
    a.neox = f.is_neox;
    a.q_fp8 = f.q_out_fp8;
    a.cache_fp8 = f.cache_fp8;
    if (f.T == 0)
        return cudaSuccess;
    const int64_t groups = ((int64_t)f.H + 1 + kWarpsPerBlock - 1) / kWarpsPerBlock; // rows of a token, in blocks
    if (groups > 65535)
        return cudaErrorInvalidValue;
    fused_qk_rope_cache_kernel<<<dim3((unsigned)f.T, (unsigned)groups), dim3(kWarpsPerBlock * 32), 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t read_producer_error(int *out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_producer_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_producer_error, &zero, sizeof(int));
    }
    return e;
}

} // namespace smla
