// Sparse MLA forward, warp-MMA kernel for groups of 16 heads (sm_103a).
//
// One CTA = (query row t, 16-head group, split s of the top-k list). It
// streams the split's key rows through a multi-stage shared-memory ring with
// 16-byte cp.async gathers (zero-filled for masked entries, which are never
// dereferenced), computes S = q K^T and O += P V with mma.sync, and keeps an
// online softmax in registers. A row's splits (at most 8) form one
// thread-block cluster: each split stages its normalised partial (o_j, lse_j)
// in shared memory, and after a cluster barrier every split merges a slice of
// the output from all partials through distributed shared memory with LSE
// weights. With more splits (very small T) the partials go to the workspace
// and the split that draws the last ticket (one atomic, no spinning) merges.
//
// Method sources (page titles and sections):
//   "Enable AITER sparse MLA on gfx942, including FP8 KV" — Overview, Details
//     ("FP8 KV on gfx942": the kernel quantizes q per tile, dots in fp8).
//   "Route gfx942 sparse MLA prefill to AITER pa_prefill_sparse" — the
//     jin-amd A/B: without a split of the top-k list decode-sized calls are
//     ~9x slower; hence split-K plus an LSE merge for small T.
//   "Fuse decode QK-RoPE + ... KV-cache write for sparse MLA" — Test plan:
//     the cache row is concat(latent, rope); only the first D_v columns are V.
//
// Work split inside a CTA (4 warps, 16 heads = the MMA's M):
//   QK: warp w owns a quarter of the D_qk reduction and produces a partial
//       S[16 x 32 keys]; the four partials are summed through shared memory
//       (each warp reduces 8 keys), so every warp ends with the full S tile.
//   PV: warp w owns 128 of the 512 value columns; O[16 x 128] stays in
//       registers (fp32) for the whole split.
//   bf16 cache: QK and PV in bf16 (K via ldmatrix, V via ldmatrix.trans).
//   fp8 cache : QK in E4M3 (m16n8k32) with q quantized in the kernel,
//       s_q = amax|q[t,h,:]| / 448 per (row, head); PV in fp16 with P in fp16
//       and V = code * 2^-8 formed exactly from the code bits in registers
//       (the 2^8 and kv_scale fold into the epilogue).
//   fp8 cache with bf16 dots ("Enable AITER sparse MLA on gfx942, including
//       FP8 KV", Details, "Numerics": the BF16-dots option): q stays bf16; each
//       register of four key codes (k = 4c..4c+3) becomes two bf16 pairs
//       code * 2^-8 (exact) feeding two bf16 m16n8k16 MMAs, with q's fragments
//       loaded in the same order of k; the 2^8 * kv_scale folds into the
//       logit factor. PV as for the fp8 cache.
#include "smla_device.cuh"
#include "smla_epilogue.cuh"
#include "smla_internal.h"

#include <atomic>
#include <cfloat>
#include <cmath>

namespace smla {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 128;
constexpr int kHeads = 16; // heads per CTA
constexpr int kTile = kMmaTileKeys;
constexpr int kDv = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <bool FP8, int DQK>
struct Cfg {
    static constexpr int EB = FP8 ? 1 : 2;                // bytes per cache element
    static constexpr int ROW = DQK * EB;                  // bytes per cache row
    static constexpr int PITCH = ROW + 16;                // padded smem row: conflict-free 8-row accesses
    static constexpr int CHUNKS = ROW / 16;               // 16-byte chunks per row
    static constexpr int CPT = CHUNKS / 4;                // chunks per thread per tile (4 threads per row)
    static constexpr int KDIM = FP8 ? 32 : 16;            // reduction depth of one QK mma
    static constexpr int KS = DQK / KDIM;                 // QK k-steps over D_qk
    static constexpr int KS_MAX = (KS + kWarps - 1) / kWarps;
    static constexpr int STAGE_BYTES = kTile * PITCH;
    static constexpr int STAGES = (!FP8 && DQK == 512) ? 3 : (!FP8 ? 2 : (DQK == 512 ? 6 : 5));
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    // after the ring: partial S [4 warps][4 n-blocks][32 lanes] float4, summed S [4][32] float4,
    // tile indices [STAGES][kTile] int, q scales [16], row lse [16], ticket flag
    static constexpr int OFF_RED = RING_BYTES;
    static constexpr int OFF_SUM = OFF_RED + kWarps * 4 * 32 * 16;
    static constexpr int OFF_IDX = OFF_SUM + 4 * 32 * 16;
    static constexpr int OFF_SQ = OFF_IDX + STAGES * kTile * 4;
    static constexpr int OFF_LSE = OFF_SQ + kHeads * 4;
    static constexpr int OFF_FLAG = OFF_LSE + kHeads * 4;
    static constexpr int SMEM = OFF_FLAG + 16;
    static_assert(CHUNKS % 4 == 0, "row must split into 4 equal parts");
    static_assert(RING_BYTES >= kHeads * kDv * 4, "epilogue staging must fit in the ring");
    static_assert(kWarps * 4 * 32 * 16 >= 128 * kHeads * 4, "merge weights must fit");
};

// Four E4M3 codes (k = 4c..4c+3 of one key) as two bf16x2 words holding
// code * 2^-8 exactly: (k0, k1) and (k2, k3), the lower k in the low half.
__device__ __forceinline__ void e4m3x4_to_bf16x4_scaled(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    // binary16 code * 2^-8: the sign to bit 15, exponent and mantissa to bits 14..7
    const uint32_t h01 = ((w & 0x80u) << 8) | ((w & 0x7Fu) << 7) | ((w & 0x8000u) << 16) | ((w & 0x7F00u) << 15);
    const uint32_t h23 = ((w & 0x800000u) >> 8) | ((w & 0x7F0000u) >> 9) | (w & 0x80000000u) | ((w & 0x7F000000u) >> 1);
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&h23));
    lo = pack_bf16x2(f01.x, f01.y);
    hi = pack_bf16x2(f23.x, f23.y);
}

// q fragments (A operand) for this warp's share of the QK reduction.
template <bool FP8, int DQK, bool BD = false>
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[Cfg<FP8, DQK>::KS_MAX][BD ? 8 : 4],
                                             const __nv_bfloat16 *__restrict__ q0, // head (group base + g)
                                             const uint8_t *__restrict__ c0, // pre-quantized codes of that head, or null
                                             const float *sq, int g, int c, int ks0, int ks1)
{
    using C = Cfg<FP8, DQK>;
    const __nv_bfloat16 *q8 = q0 + 8 * DQK; // head + 8
#pragma unroll
    for (int i = 0; i < C::KS_MAX; ++i) {
        const int ks = ks0 + i;
        if (ks < ks1) {
            if constexpr (BD) {
                // bf16 q against an E4M3 key tile: for the k32 step, MMA 0 takes
                // k = 4c..4c+3 and MMA 1 k = 16 + 4c..16 + 4c+3, in the order the
                // key registers are split (slot 2c, 2c+1 <- 4c, 4c+1; slot 8+2c,
                // 9+2c <- 4c+2, 4c+3)
#pragma unroll
                for (int mm = 0; mm < 2; ++mm) {
                    const int d = ks * 32 + mm * 16 + 4 * c;
                    const uint2 u0 = *reinterpret_cast<const uint2 *>(q0 + d);
                    const uint2 u1 = *reinterpret_cast<const uint2 *>(q8 + d);
                    qa[i][4 * mm + 0] = u0.x;
                    qa[i][4 * mm + 1] = u1.x;
                    qa[i][4 * mm + 2] = u0.y;
                    qa[i][4 * mm + 3] = u1.y;
                }
            } else if (FP8 && c0 != nullptr) {
                // pre-quantized q: the m16n8k32 A fragment takes 4 consecutive codes per register
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int d = ks * 32 + half * 16 + 4 * c;
                    qa[i][2 * half + 0] = *reinterpret_cast<const uint32_t *>(c0 + d);
                    qa[i][2 * half + 1] = *reinterpret_cast<const uint32_t *>(c0 + 8 * DQK + d);
                }
            } else if constexpr (!FP8) {
                const int d = ks * 16 + 2 * c;
                qa[i][0] = *reinterpret_cast<const uint32_t *>(q0 + d);
                qa[i][1] = *reinterpret_cast<const uint32_t *>(q8 + d);
                qa[i][2] = *reinterpret_cast<const uint32_t *>(q0 + d + 8);
                qa[i][3] = *reinterpret_cast<const uint32_t *>(q8 + d + 8);
            } else {
                const float s0 = sq[g], s1 = sq[g + 8];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int d = ks * 32 + half * 16 + 4 * c;
                    const uint2 u0 = *reinterpret_cast<const uint2 *>(q0 + d);
                    const uint2 u1 = *reinterpret_cast<const uint2 *>(q8 + d);
                    const __nv_bfloat162 *b0 = reinterpret_cast<const __nv_bfloat162 *>(&u0);
                    const __nv_bfloat162 *b1 = reinterpret_cast<const __nv_bfloat162 *>(&u1);
                    const float2 x0 = __bfloat1622float2(b0[0]), x1 = __bfloat1622float2(b0[1]);
                    const float2 y0 = __bfloat1622float2(b1[0]), y1 = __bfloat1622float2(b1[1]);
                    qa[i][2 * half + 0] = quant4_e4m3(x0.x, x0.y, x1.x, x1.y, s0);
                    qa[i][2 * half + 1] = quant4_e4m3(y0.x, y0.y, y1.x, y1.y, s1);
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < (BD ? 8 : 4); ++r)
                qa[i][r] = 0u;
        }
    }
}

template <bool FP8, int DQK, bool BD = false>
__global__ void __launch_bounds__(kThreads, 2) sparse_mla_fwd_mma_kernel(const FwdArgs a)
{
    using C = Cfg<FP8, DQK>;
    extern __shared__ __align__(128) uint8_t smem[];
    float4 *red = reinterpret_cast<float4 *>(smem + C::OFF_RED);
    float4 *sum = reinterpret_cast<float4 *>(smem + C::OFF_SUM);
    int *idx_s = reinterpret_cast<int *>(smem + C::OFF_IDX);
    float *sq = reinterpret_cast<float *>(smem + C::OFF_SQ);
    float *lse_s = reinterpret_cast<float *>(smem + C::OFF_LSE);
    int *flag_s = reinterpret_cast<int *>(smem + C::OFF_FLAG);
    const uint32_t ring = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int G = a.H / kHeads;
    int bid = blockIdx.x;
    const int s = bid % a.S;
    bid /= a.S;
    const int hg = bid % G;
    const int t = bid / G;

    const int kb = s * a.keys_per_split;
    const int ke = min(a.topk, kb + a.keys_per_split);
    const int ntiles = ke > kb ? (ke - kb + kTile - 1) / kTile : 0;
    const int32_t *__restrict__ row_idx = a.indices + (int64_t)t * a.topk;
    const uint8_t *__restrict__ kv = static_cast<const uint8_t *>(a.kv);
    const __nv_bfloat16 *__restrict__ qg =
        static_cast<const __nv_bfloat16 *>(a.q) + ((int64_t)t * a.H + hg * kHeads) * DQK;

    float kvs = 1.0f;
    if constexpr (FP8)
        kvs = *a.kv_scale;

    // ---- gather issue: thread -> (key r, quarter sub) of each tile ---------
    const int my_key = tid >> 2, my_sub = tid & 3;
    auto fetch_idx = [&](int tile) -> int {
        const int p = kb + tile * kTile + my_key;
        int v = -1;
        if (tile < ntiles && p < ke) {
            v = __ldg(row_idx + p);
            if (v < 0 || (int64_t)v >= a.num_slots)
                v = -1; // masked, or outside the pool: never dereferenced
        }
        return v;
    };
    auto issue = [&](int tile, int idx) {
        const int st = tile % C::STAGES;
        if (my_sub == 0)
            idx_s[st * kTile + my_key] = idx;
        const uint32_t dst = ring + st * C::STAGE_BYTES + my_key * C::PITCH + my_sub * 16;
        const uint8_t *src = kv + (idx >= 0 ? (int64_t)idx * C::ROW : 0) + my_sub * 16;
        const uint32_t nbytes = idx >= 0 ? 16u : 0u;
#pragma unroll
        for (int j = 0; j < C::CPT; ++j)
            cp_async_16(dst + j * 64, src + j * 64, nbytes);
    };

    // ---- q: per-head fp8 scales, then this warp's A fragments ---------------
    if constexpr (BD) {
        // q stays bf16: no q scales
    } else if (FP8 && a.q_fp8_in) {
        if (tid < kHeads) // one per-tensor scale for every head
            sq[tid] = *a.q_scale_in;
    } else if constexpr (FP8) {
#pragma unroll
        for (int hh = 0; hh < kHeads / kWarps; ++hh) {
            const int h = warp * (kHeads / kWarps) + hh;
            const __nv_bfloat16 *qr = qg + (int64_t)h * DQK;
            float m = 0.f;
            for (int d = lane * 8; d < DQK; d += 32 * 8) {
                const uint4 u = *reinterpret_cast<const uint4 *>(qr + d);
                const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(b[e]);
                    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
            }
            m = warp_max(m);
            if (lane == 0)
                sq[h] = (m == 0.f) ? 1.0f : __fdiv_rn(m, 448.0f);
        }
    }

    // prologue: indices for the first STAGES-1 tiles, then their gathers
    int pre[C::STAGES];
#pragma unroll
    for (int j = 0; j < C::STAGES; ++j)
        pre[j] = fetch_idx(j);
    __syncthreads(); // sq visible
    const int ks0 = warp * C::KS / kWarps, ks1 = (warp + 1) * C::KS / kWarps;
    uint32_t qa[C::KS_MAX][BD ? 8 : 4];
    const uint8_t *cg = a.q_fp8_in ? static_cast<const uint8_t *>(a.q) + (qg - static_cast<const __nv_bfloat16 *>(a.q))
                                   : nullptr; // the same row and head offset, in codes
    load_q_frags<FP8, DQK, BD>(qa, qg + (int64_t)g * DQK, cg ? cg + (int64_t)g * DQK : nullptr, sq, g, c, ks0, ks1);
#pragma unroll
    for (int j = 0; j < C::STAGES - 1; ++j) {
        if (j < ntiles)
            issue(j, pre[j]);
        cp_async_commit();
    }
    int idx_next = pre[C::STAGES - 1];

    float qk_fac0 = a.scale * kLog2e, qk_fac1 = qk_fac0;
    if constexpr (BD) {
        qk_fac0 *= 256.0f * kvs; // keys entered the dots as code * 2^-8
        qk_fac1 = qk_fac0;
    } else if constexpr (FP8) {
        qk_fac0 *= sq[g] * kvs;
        qk_fac1 *= sq[g + 8] * kvs;
    }

    float o[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    cp_async_wait<C::STAGES - 2>();
    __syncthreads();

    for (int it = 0; it < ntiles; ++it) {
        const int st = it % C::STAGES;
        const uint32_t sbase = ring + st * C::STAGE_BYTES;
        const bool any = __any_sync(0xffffffffu, idx_s[st * kTile + lane] >= 0);

        // ---- partial S over this warp's share of D_qk ----
        if (any) {
            float sacc[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
            const int mtx = lane >> 3;
#pragma unroll
            for (int i = 0; i < C::KS_MAX; ++i) {
                const int ks = ks0 + i;
                if (ks < ks1) {
#pragma unroll
                    for (int nbp = 0; nbp < 2; ++nbp) {
                        const int row = nbp * 16 + (mtx >> 1) * 8 + (lane & 7);
                        const int chunk = 2 * ks + (mtx & 1);
                        uint32_t b[4];
                        ldmatrix_x4(b, sbase + row * C::PITCH + chunk * 16);
                        if constexpr (BD) {
#pragma unroll
                            for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
                                for (int mm = 0; mm < 2; ++mm) {
                                    uint32_t lo, hi;
                                    e4m3x4_to_bf16x4_scaled(b[2 * nb + mm], lo, hi);
                                    const uint32_t(&aq)[4] = *reinterpret_cast<const uint32_t(*)[4]>(&qa[i][4 * mm]);
                                    mma_bf16_16816(sacc[2 * nbp + nb], aq, lo, hi);
                                }
                            }
                        } else if constexpr (FP8) {
                            mma_e4m3_16832(sacc[2 * nbp], qa[i], b[0], b[1]);
                            mma_e4m3_16832(sacc[2 * nbp + 1], qa[i], b[2], b[3]);
                        } else {
                            mma_bf16_16816(sacc[2 * nbp], qa[i], b[0], b[1]);
                            mma_bf16_16816(sacc[2 * nbp + 1], qa[i], b[2], b[3]);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                red[(warp * 4 + j) * 32 + lane] = make_float4(sacc[j][0], sacc[j][1], sacc[j][2], sacc[j][3]);
        }
        __syncthreads(); // (A) partials written; everyone is past the previous tile

        // refill the stage the previous tile used
        {
            const int nt = it + C::STAGES - 1;
            if (nt < ntiles) {
                issue(nt, idx_next);
                idx_next = fetch_idx(nt + 1);
            }
            cp_async_commit();
        }

        if (any) {
            // this warp sums key block `warp` (8 keys) over the four partials
            float4 v = red[(0 * 4 + warp) * 32 + lane];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) {
                const float4 u = red[(w * 4 + warp) * 32 + lane];
                v.x += u.x;
                v.y += u.y;
                v.z += u.z;
                v.w += u.w;
            }
            const int k0 = warp * 8 + 2 * c;
            const bool ok0 = idx_s[st * kTile + k0] >= 0, ok1 = idx_s[st * kTile + k0 + 1] >= 0;
            v.x = ok0 ? v.x * qk_fac0 : -INFINITY;
            v.y = ok1 ? v.y * qk_fac0 : -INFINITY;
            v.z = ok0 ? v.z * qk_fac1 : -INFINITY;
            v.w = ok1 ? v.w * qk_fac1 : -INFINITY;
            sum[warp * 32 + lane] = v;
        }
        cp_async_wait<C::STAGES - 2>(); // own copies of the next tile have landed
        __syncthreads();                // (B) summed S and the next tile visible

        if (!any)
            continue;

        // ---- online softmax on the full 16 x 32 tile (base-2 logits) ----
        float sv[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 u = sum[j * 32 + lane];
            sv[j][0] = u.x;
            sv[j][1] = u.y;
            sv[j][2] = u.z;
            sv[j][3] = u.w;
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            mx0 = fmaxf(mx0, fmaxf(sv[j][0], sv[j][1]));
            mx1 = fmaxf(mx1, fmaxf(sv[j][2], sv[j][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sv[j][0] = exp2f(sv[j][0] - mu0);
            sv[j][1] = exp2f(sv[j][1] - mu0);
            sv[j][2] = exp2f(sv[j][2] - mu1);
            sv[j][3] = exp2f(sv[j][3] - mu1);
            ps0 += sv[j][0] + sv[j][1];
            ps1 += sv[j][2] + sv[j][3];
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            o[j][0] *= al0;
            o[j][1] *= al0;
            o[j][2] *= al1;
            o[j][3] *= al1;
        }
        uint32_t pa[2][4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            if constexpr (FP8) {
                pa[kk][0] = pack_f16x2(sv[2 * kk][0], sv[2 * kk][1]);
                pa[kk][1] = pack_f16x2(sv[2 * kk][2], sv[2 * kk][3]);
                pa[kk][2] = pack_f16x2(sv[2 * kk + 1][0], sv[2 * kk + 1][1]);
                pa[kk][3] = pack_f16x2(sv[2 * kk + 1][2], sv[2 * kk + 1][3]);
            } else {
                pa[kk][0] = pack_bf16x2(sv[2 * kk][0], sv[2 * kk][1]);
                pa[kk][1] = pack_bf16x2(sv[2 * kk][2], sv[2 * kk][3]);
                pa[kk][2] = pack_bf16x2(sv[2 * kk + 1][0], sv[2 * kk + 1][1]);
                pa[kk][3] = pack_bf16x2(sv[2 * kk + 1][2], sv[2 * kk + 1][3]);
            }
        }

        // ---- O[16 x 128] += P[16 x 32] V[32 x 128] for this warp's columns ----
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            if constexpr (!FP8) {
                const int mtx = lane >> 3;
                const int row = kk * 16 + (mtx & 1) * 8 + (lane & 7);
#pragma unroll
                for (int jp = 0; jp < 8; ++jp) {
                    const int chunk = warp * 16 + 2 * jp + (mtx >> 1);
                    uint32_t b[4];
                    ldmatrix_x4_trans(b, sbase + row * C::PITCH + chunk * 16);
                    mma_bf16_16816(o[2 * jp], pa[kk], b[0], b[1]);
                    mma_bf16_16816(o[2 * jp + 1], pa[kk], b[2], b[3]);
                }
            } else {
                // column permutation inside each 32-byte group: logical n-block 4q+b,
                // column n=g  <->  value column 128*warp + 32q + 4g + b
                const uint32_t r0 = sbase + (kk * 16 + 2 * c) * C::PITCH;
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    const uint32_t off = warp * 128 + qd * 32 + 4 * g;
                    const uint32_t w0 = lds32(r0 + off);
                    const uint32_t w1 = lds32(r0 + C::PITCH + off);
                    const uint32_t w2 = lds32(r0 + 8 * C::PITCH + off);
                    const uint32_t w3 = lds32(r0 + 9 * C::PITCH + off);
                    mma_f16_16816(o[4 * qd + 0], pa[kk], e4m3x2_to_f16x2_scaled<0>(w0, w1),
                                  e4m3x2_to_f16x2_scaled<0>(w2, w3));
                    mma_f16_16816(o[4 * qd + 1], pa[kk], e4m3x2_to_f16x2_scaled<1>(w0, w1),
                                  e4m3x2_to_f16x2_scaled<1>(w2, w3));
                    mma_f16_16816(o[4 * qd + 2], pa[kk], e4m3x2_to_f16x2_scaled<2>(w0, w1),
                                  e4m3x2_to_f16x2_scaled<2>(w2, w3));
                    mma_f16_16816(o[4 * qd + 3], pa[kk], e4m3x2_to_f16x2_scaled<3>(w0, w1),
                                  e4m3x2_to_f16x2_scaled<3>(w2, w3));
                }
            }
        }
    }
    cp_async_wait<0>();

    // ---- epilogue: normalise, stage [16][512] fp32 in the ring ----
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float vfac = FP8 ? kvs * 256.0f : 1.0f;
    const float i0 = l0 > 0.f ? vfac / l0 : 0.f;
    const float i1 = l1 > 0.f ? vfac / l1 : 0.f;
    __syncthreads(); // every warp is done with the ring
    float *ost = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if constexpr (!FP8) {
            const int d = warp * 128 + j * 8 + 2 * c;
            *reinterpret_cast<float2 *>(ost + g * kDv + d) = make_float2(o[j][0] * i0, o[j][1] * i0);
            *reinterpret_cast<float2 *>(ost + (g + 8) * kDv + d) = make_float2(o[j][2] * i1, o[j][3] * i1);
        } else {
            const int qd = j >> 2, b = j & 3;
            const int d0 = warp * 128 + qd * 32 + 4 * (2 * c) + b;
            const int d1 = d0 + 4;
            ost[g * kDv + d0] = o[j][0] * i0;
            ost[g * kDv + d1] = o[j][1] * i0;
            ost[(g + 8) * kDv + d0] = o[j][2] * i1;
            ost[(g + 8) * kDv + d1] = o[j][3] * i1;
        }
    }
    if (warp == 0 && c == 0) {
        lse_s[g] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
        lse_s[g + 8] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
    }
    __syncthreads();

    finish_tile<kThreads>(a, ost, lse_s, reinterpret_cast<float *>(smem + C::OFF_RED), flag_s, t, hg, s, tid);
}

template <bool FP8, int DQK, bool BD = false>
cudaError_t launch_one(const FwdArgs &a, cudaStream_t stream)
{
    using C = Cfg<FP8, DQK>;
    auto kern = sparse_mla_fwd_mma_kernel<FP8, DQK, BD>;
    // The shared-memory opt-in is per function and per device: set it on the
    // first launch on each device (before any stream capture of that device).
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess)
            return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    const int64_t blocks = (int64_t)a.T * (a.H / kHeads) * a.S;
    if (blocks == 0)
        return cudaSuccess;
    if (a.S > 1 && a.S <= kClusterMaxSplits) {
        // the S splits of a (row, head group) are consecutive blocks: one cluster
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = C::SMEM;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)a.S;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kern, a);
    }
    kern<<<dim3((unsigned)blocks), dim3(kThreads), C::SMEM, stream>>>(a);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_fwd_mma(const FwdArgs &a, cudaStream_t stream)
{
    if (a.kv_fp8 && a.bf16_dots)
        return a.D_qk == 512 ? launch_one<true, 512, true>(a, stream) : launch_one<true, 576, true>(a, stream);
    if (a.kv_fp8)
        return a.D_qk == 512 ? launch_one<true, 512>(a, stream) : launch_one<true, 576>(a, stream);
    return a.D_qk == 512 ? launch_one<false, 512>(a, stream) : launch_one<false, 576>(a, stream);
}

} // namespace smla
