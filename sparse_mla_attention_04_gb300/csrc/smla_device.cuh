// Device-side helpers shared by the kernels of libsparse_mla.so (sm_103a).
// Thin inline-PTX wrappers: asynchronous 16-byte copies into shared memory,
// ldmatrix fragment loads and warp-level mma.sync tensor-core products.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace smla {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy that bypasses L1. src_bytes = 0 writes zeros
// and reads nothing (the source address is then only required to be valid).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
    return v;
}

// Four 8 x 8 matrices of 16-bit elements, transposed on the way: lane l gives
// the address of row l % 8 of matrix l / 8 (16 contiguous bytes); lane l gets
// in d[m] element l / 4 of rows 2 (l % 4) (low half) and 2 (l % 4) + 1 (high
// half) of matrix m.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&d)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr)
                 : "memory");
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A(16x16, row) * B(16x8, col), fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A(16x32, row) * B(32x8, col), E4M3 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two E4M3 codes (byte `b` of wa -> low half, byte `b` of wb -> high half) as
// an f16x2 holding each code's value times 2^-8. Exact: an E4M3 code
// s.eeee.mmm placed at bits [14:7] of a binary16 (with bit 14 clear) has the
// binary16 exponent field 0eeee and mantissa mmm0000000, i.e. the value
// 2^(e-15)(1 + m/8) for e > 0 and m/8 * 2^-14 for e = 0, which is the E4M3
// value (bias 7) scaled by 2^-8. The NaN code is not produced by the
// quantizer for finite input.
template <int B>
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t wa, uint32_t wb)
{
    constexpr uint32_t sel = B | (B << 4) | ((B + 4) << 8) | ((B + 4) << 12);
    const uint32_t y = __byte_perm(wa, wb, sel); // code(a) at bits 15:8, code(b) at 31:24
    return (y & 0x80008000u) | ((y >> 1) & 0x3F803F80u);
}

// The two reciprocals quant2_e4m3 multiplies by: 1/s rounded to binary32 and
// scaled by (1 -+ 2^-21), each rounded again; `ok` is false for a reciprocal that is
// zero, infinite or NaN (then every element is divided).
struct E4m3Recip {
    float lo, hi;
    bool ok;
};
__device__ __forceinline__ E4m3Recip e4m3_recip(float s)
{
    const float inv = __fdiv_rn(1.0f, s);
    E4m3Recip r;
    r.lo = __fmul_rn(inv, 1.0f - 0x1p-21f);
    r.hi = __fmul_rn(inv, 1.0f + 0x1p-21f);
    r.ok = fabsf(inv) <= 3.4028234663852886e38f && inv != 0.0f; // finite, nonzero (false for NaN)
    return r;
}

// E4M3 codes (round to nearest even, saturating) of x0 / s and x1 / s in
// IEEE binary32 division, first value in the low byte.
//
// The codes are those of the correctly rounded quotients, found without a
// division for almost every element. x * r.lo and x * r.hi bracket x / s with
// a relative margin of 2^-21 on each side, while the rounding of 1/s, of the
// factor (1 -+ 2^-21), of the product and of the quotient itself move a value
// by at most 2^-24 relative each: the correctly rounded quotient lies between
// the two products. Rounding onto the E4M3 grid is monotone, so when both
// products give the same code, so does the quotient; otherwise (they straddle
// a rounding midpoint, about one element in 10^5) the element is divided.
__device__ __forceinline__ uint32_t quant2_e4m3(float x0, float x1, float s, const E4m3Recip &r)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x0, r.lo), __fmul_rn(x1, r.lo)),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x0, r.hi), __fmul_rn(x1, r.hi)),
                                                 __NV_SATFINITE, __NV_E4M3);
    if (r.ok && ((lo ^ hi) & 0xFFFFu) == 0)
        return lo & 0xFFFFu;
    const float2 d = make_float2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
    return __nv_cvt_float2_to_fp8x2(d, __NV_SATFINITE, __NV_E4M3) & 0xFFFFu;
}

// Four floats divided by `s` (IEEE binary32 division) and rounded to E4M3
// with saturation, packed lowest index in the lowest byte; r = e4m3_recip(s).
// The same bracketing as quant2_e4m3, with one comparison for the four codes.
__device__ __forceinline__ uint32_t quant4_e4m3(float x0, float x1, float x2, float x3, float s, const E4m3Recip &r)
{
    const uint32_t lo01 = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x0, r.lo), __fmul_rn(x1, r.lo)),
                                                   __NV_SATFINITE, __NV_E4M3);
    const uint32_t lo23 = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x2, r.lo), __fmul_rn(x3, r.lo)),
                                                   __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi01 = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x0, r.hi), __fmul_rn(x1, r.hi)),
                                                   __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi23 = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(x2, r.hi), __fmul_rn(x3, r.hi)),
                                                   __NV_SATFINITE, __NV_E4M3);
    const uint32_t lo = __byte_perm(lo01, lo23, 0x5410), hi = __byte_perm(hi01, hi23, 0x5410);
    if (r.ok && lo == hi)
        return lo;
    const uint32_t d01 = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x0, s), __fdiv_rn(x1, s)), __NV_SATFINITE,
                                                  __NV_E4M3);
    const uint32_t d23 = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x2, s), __fdiv_rn(x3, s)), __NV_SATFINITE,
                                                  __NV_E4M3);
    return __byte_perm(d01, d23, 0x5410);
}

__device__ __forceinline__ uint32_t quant4_e4m3(float x0, float x1, float x2, float x3, float s)
{
    return quant4_e4m3(x0, x1, x2, x3, s, e4m3_recip(s));
}

// Four E4M3 codes (lowest byte first) as two f16x2 words holding their
// values exactly (every E4M3 value, subnormals included, is a normal
// binary16), by the hardware conversion.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    asm("{\n.reg .b16 a, b;\nmov.b32 {a, b}, %2;\n"
        "cvt.rn.f16x2.e4m3x2 %0, a;\ncvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// 2^x by the hardware approximation (relative error about 2^-22, far below
// the 16-bit rounding the softmax weights get next); -inf gives 0.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

} // namespace smla
