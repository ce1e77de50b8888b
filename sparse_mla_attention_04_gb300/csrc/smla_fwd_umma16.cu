// Sparse MLA forward for 16 heads on the 5th-generation tensor cores
// (tcgen05 + tensor memory), sm_103a.
//
// One CTA = (query row t, split s of its top-k list). With only 16 heads per
// row the contraction is computed transposed, keys on the MMA's M axis:
//   S^T [64 keys x 16 heads] = KV_tile [64 x 512] . q^T          (QK, M=64, N=16)
//   O^T [512 dims x 16 heads] += V^T [512 x 64 keys] . P^T       (PV, 4 x M=128, N=16)
// Both accumulators live in tensor memory (S^T double-buffered, O^T in 64
// columns). One shared-memory tile of gathered rows serves as the K-major A
// operand of QK and, read MN-major, as V^T of PV.
//
// Warp roles, handing tiles over through mbarriers:
//   producers (warps 5..): gather the split's key rows, 64 per tile, with
//     16-byte global loads into registers and store them into a 3-stage
//     shared-memory ring in the tensor core's core-matrix layout (masked or
//     out-of-range indices are never read; their rows are zeros), then arrive
//     on the stage's "full" barrier. Loads through registers keep many more
//     bytes in flight per SM than cp.async for scattered 1 KB rows. A stage is
//     refilled once the PV that read it has completed ("empty").
//   MMA issuer (warp 4, one thread): QK(i) as soon as tile i has landed, then
//     PV(i-1) as soon as the softmax has written P(i-1); commits signal the
//     softmax (S full), the producers (stage empty), the P buffers and O.
//   softmax (warps 0-3, one key per thread of lanes 0-15): reads the key's 16
//     logits from TMEM, masks, and exponentiates against a running reference
//     max; the max is recomputed over the tile (and O^T rescaled in TMEM) only
//     when some logit exceeds the reference by more than 2^8, so the common
//     tile needs no cross-thread reduction; writes one row of P^T.
// Every barrier completes once per use of the resource it guards, so no
// waiter can fall two phases behind; every wait gives up after about 2 s
// (the call then records an error and finishes without further waiting).
//
// Method sources (page titles and sections):
//   "Enable AITER sparse MLA on gfx942, including FP8 KV" — Overview, Details.
//   "Route gfx942 sparse MLA prefill to AITER pa_prefill_sparse" — jin-amd
//     A/B: split-K for decode-sized calls.
#include "smla_device.cuh"
#include "smla_epilogue.cuh"
#include "smla_internal.h"
#include "smla_umma.cuh"

#include <atomic>
#include <cmath>

namespace smla {

__device__ int g_umma_error = 0; // set when a bounded wait gives up

namespace {

#ifndef SMLA_UMMA16_PRODUCER_WARPS
#define SMLA_UMMA16_PRODUCER_WARPS 8
#endif
constexpr int kSoftmaxWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kProducerWarp0 = 5;
constexpr int kProducerThreads = 32 * SMLA_UMMA16_PRODUCER_WARPS;
constexpr int kThreads = (kProducerWarp0 * 32) + kProducerThreads;
constexpr int kGroupSets = kProducerThreads / 128;   // producer sets, one per column of key groups
constexpr int kGroupsPerThread = 8 / kGroupSets;     // 8-key groups each producer moves per tile
static_assert(kProducerThreads % 128 == 0 && 8 % kGroupSets == 0, "producer mapping");
constexpr int kKeys = kUmma16TileKeys; // keys per tile (M of QK)
constexpr int kHeads = 16;
constexpr int kDv = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f; // log2 units: p <= 2^8 between rescales

struct U16 {
    static constexpr int ROW = 1024;              // bytes per cache row (bf16, D = 512)
    static constexpr int CPR = ROW / 16;          // core-matrix columns per row (64)
    static constexpr int KGRP = CPR * 128;        // one 8-key group (8 KB)
    static constexpr int TILE = 8 * KGRP;         // 64 keys (64 KB)
    static constexpr int STAGES = 3;
    static constexpr int OFF_Q = STAGES * TILE;   // q [16 x 512] bf16 in core matrices (16 KB)
    static constexpr int OFF_P = OFF_Q + 16 * ROW;// P^T [64 keys x 16 heads] bf16, 2 buffers x 2 KB
    static constexpr int OFF_EX = OFF_P + 2 * 2048; // [2][4] exceed flags
    static constexpr int OFF_WMAX = OFF_EX + 32;
    static constexpr int OFF_LRED = OFF_WMAX + 4 * 16 * 4;
    static constexpr int OFF_LSE = OFF_LRED + 4 * 16 * 4;
    static constexpr int OFF_ALPHA = OFF_LSE + 16 * 4;
    static constexpr int OFF_MISC = OFF_ALPHA + 16 * 4; // flag, tmem address, abort
    static constexpr int OFF_MBAR = OFF_MISC + 16;
    // full[3], empty[3], s_full[2], p_full[2], p_empty[2], o_done
    static constexpr int NBAR = 13;
    static constexpr int SMEM = OFF_MBAR + NBAR * 8;
    static_assert(STAGES * TILE >= kHeads * kDv * 4, "epilogue staging fits in the ring");
    static_assert(16 * ROW >= 128 * kHeads * 4, "merge weights fit in the q area");
    static_assert(OFF_MBAR % 8 == 0, "mbarrier alignment");
};

// QK: A = KV tile (K-major), B = q (K-major), M = 64 keys, N = 16 heads, bf16
constexpr uint32_t kIdescQK = umma::idesc(64, 16, 1, 1, 0, 0);
// PV: A = V^T (MN-major over the same tile), B = P^T (MN-major), M = 128 dims, N = 16
constexpr uint32_t kIdescPV = umma::idesc(128, 16, 1, 1, 1, 1);

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_fwd_umma16_kernel(const FwdArgs a)
{
    using C = U16;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    const uint32_t ring = sbase, q_s = sbase + C::OFF_Q, p_s = sbase + C::OFF_P;
    int *ex_s = reinterpret_cast<int *>(smem + C::OFF_EX);
    float *wmax_s = reinterpret_cast<float *>(smem + C::OFF_WMAX);
    float *lred_s = reinterpret_cast<float *>(smem + C::OFF_LRED);
    float *lse_s = reinterpret_cast<float *>(smem + C::OFF_LSE);
    float *alpha_s = reinterpret_cast<float *>(smem + C::OFF_ALPHA);
    int *flag_s = reinterpret_cast<int *>(smem + C::OFF_MISC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC + 4);
    int *abort_s = reinterpret_cast<int *>(smem + C::OFF_MISC + 8);
    const uint32_t bar0 = sbase + C::OFF_MBAR;
    auto full = [&](int st) { return bar0 + 8 * st; };
    auto empty = [&](int st) { return bar0 + 8 * (3 + st); };
    auto s_full = [&](int b) { return bar0 + 8 * (6 + b); };
    auto p_full = [&](int b) { return bar0 + 8 * (8 + b); };
    auto p_empty = [&](int b) { return bar0 + 8 * (10 + b); };
    const uint32_t o_done = bar0 + 8 * 12;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x % a.S;
    const int t = blockIdx.x / a.S;
    const int kb = s * a.keys_per_split;
    const int ke = min(a.topk, kb + a.keys_per_split);
    const int ntiles = ke > kb ? (ke - kb + kKeys - 1) / kKeys : 0;
    const int32_t *__restrict__ row_idx = a.indices + (int64_t)t * a.topk;

    if (tid == 0) {
        for (int st = 0; st < C::STAGES; ++st) {
            umma::mbar_init(full(st), kProducerThreads);
            umma::mbar_init(empty(st), 1);
        }
        for (int b = 0; b < 2; ++b) {
            umma::mbar_init(s_full(b), 1);
            umma::mbar_init(p_full(b), kSoftmaxWarps * 32);
            umma::mbar_init(p_empty(b), 1);
        }
        umma::mbar_init(o_done, 1);
        umma::mbar_init_fence();
        *abort_s = 0;
    }
    if (warp == 0)
        umma::alloc(smem_u32(tmem_slot), 128);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    auto wait_bar = [&](uint32_t mbar, uint32_t parity) {
        if (*(volatile int *)abort_s)
            return;
        if (!umma::mbar_wait(mbar, parity)) {
            atomicOr(&g_umma_error, 1);
            *(volatile int *)abort_s = 1;
        }
    };

    if (warp >= kProducerWarp0) {
        // ======================= producers =======================
        const int ptid = tid - kProducerWarp0 * 32;
        const uint8_t *__restrict__ kv = static_cast<const uint8_t *>(a.kv);
        const __nv_bfloat16 *__restrict__ qg =
            static_cast<const __nv_bfloat16 *>(a.q) + (int64_t)t * kHeads * 512;
        // q [16 x 512] -> core matrices (8 heads x 16 B): LBO 128 (K), SBO 8 KB
        // (heads); published with tile 0
        for (int e = ptid; e < kHeads * C::CPR; e += kProducerThreads) {
            const int h = e / C::CPR, c = e % C::CPR;
            cp_async_16(q_s + (h >> 3) * C::KGRP + c * 128 + (h & 7) * 16, qg + h * 512 + c * 8, 16);
        }
        cp_async_commit();
        cp_async_wait<0>();
        // The thread moves chunks 16*c4 + kc (c4 = 0..3) of key 8*g + kr for its
        // key groups g; each warp-wide store fills four whole core matrices.
        const int kr = ptid & 7, kc = (ptid >> 3) & 15, gs = ptid >> 7;
        int raw[kGroupsPerThread];
        auto fetch = [&](int tile) {
#pragma unroll
            for (int u = 0; u < kGroupsPerThread; ++u) {
                const int p = kb + tile * kKeys + 8 * (gs * kGroupsPerThread + u) + kr;
                raw[u] = (tile < ntiles && p < ke) ? __ldg(row_idx + p) : -1;
            }
        };
        fetch(0);
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % C::STAGES;
            uint4 v[kGroupsPerThread * 4];
#pragma unroll
            for (int u = 0; u < kGroupsPerThread; ++u) {
                const int r = raw[u];
                const bool ok = r >= 0 && (int64_t)r < a.num_slots;
                const uint4 *src = reinterpret_cast<const uint4 *>(kv + (int64_t)(ok ? r : 0) * C::ROW) + kc;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    v[4 * u + c4] = ok ? __ldcs(src + 16 * c4) : make_uint4(0u, 0u, 0u, 0u);
            }
            fetch(j + 1);
            if (j >= C::STAGES)
                wait_bar(empty(st), (uint32_t)((j / C::STAGES - 1) & 1));
            const uint32_t base = ring + st * C::TILE;
#pragma unroll
            for (int u = 0; u < kGroupsPerThread; ++u) {
                const uint32_t dst = base + (gs * kGroupsPerThread + u) * C::KGRP + kc * 128 + kr * 16;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const uint4 x = v[4 * u + c4];
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst + c4 * 16 * 128), "r"(x.x),
                                 "r"(x.y), "r"(x.z), "r"(x.w)
                                 : "memory");
                }
            }
            umma::fence_async_smem();
            umma::mbar_arrive(full(st));
        }
    } else if (warp == kMmaWarp) {
        // ======================= MMA issuer =======================
        if (lane == 0) {
            const uint64_t qdesc = umma::desc(q_s, 128, C::KGRP);
            auto issue_pv = [&](int i) {
                const int b = i & 1, st = i % C::STAGES;
                wait_bar(p_full(b), (uint32_t)((i >> 1) & 1));
                umma::fence_after_sync();
                const uint64_t ad = umma::desc(ring + st * C::TILE, C::KGRP, 128);
                const uint64_t bd = umma::desc(p_s + b * 2048, 256, 128);
#pragma unroll
                for (int blk = 0; blk < 4; ++blk)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma::mma_f16(tmem + 16 * blk, ad + (uint64_t)(blk * 128 + kk * 1024), bd + (uint64_t)(kk * 32),
                                      kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                umma::commit(empty(st));
                umma::commit(p_empty(b));
                umma::commit(o_done);
            };
            for (int i = 0; i < ntiles; ++i) {
                const int b = i & 1, st = i % C::STAGES;
                wait_bar(full(st), (uint32_t)((i / C::STAGES) & 1));
                umma::fence_async_smem();
                umma::fence_after_sync();
                const uint64_t ad = umma::desc(ring + st * C::TILE, 128, C::KGRP);
#pragma unroll 8
                for (int ks = 0; ks < 32; ++ks)
                    umma::mma_f16(tmem + 64 + 16 * b, ad + (uint64_t)(ks * 16), qdesc + (uint64_t)(ks * 16), kIdescQK,
                                  ks > 0);
                umma::commit(s_full(b));
                if (i >= 1)
                    issue_pv(i - 1);
            }
            if (ntiles > 0)
                issue_pv(ntiles - 1);
        }
        __syncwarp();
    } else {
        // ======================= softmax =======================
        const uint32_t tm_lane = (uint32_t)(warp * 32) << 16;
        const float fac = a.scale * kLog2e;
        const int key = warp * 16 + lane; // meaningful for lane < 16
        float m_ref[16], l_part[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
            m_ref[h] = -INFINITY;
            l_part[h] = 0.f;
        }
        auto load_idx = [&](int tile) {
            const int p = kb + tile * kKeys + key;
            return (lane < 16 && tile < ntiles && p < ke) ? __ldg(row_idx + p) : -1;
        };
        int my_idx = load_idx(0);
        for (int i = 0; i < ntiles; ++i) {
            const int b = i & 1;
            const bool kvalid = my_idx >= 0 && (int64_t)my_idx < a.num_slots;
            my_idx = load_idx(i + 1);
            wait_bar(s_full(b), (uint32_t)((i >> 1) & 1));
            umma::fence_after_sync();
            float sv[16];
            umma::ld16(tmem + 64 + 16 * b + tm_lane, reinterpret_cast<uint32_t(&)[16]>(sv));
            umma::wait_ld();
            bool exceed = false;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                sv[h] = kvalid ? sv[h] * fac : -INFINITY;
                exceed |= sv[h] > m_ref[h] + kRescaleThreshold;
            }
            exceed = __any_sync(0xffffffffu, exceed);
            if (lane == 0)
                ex_s[b * 4 + warp] = exceed;
            umma::named_bar(1, kSoftmaxWarps * 32);
            if (ex_s[b * 4] | ex_s[b * 4 + 1] | ex_s[b * 4 + 2] | ex_s[b * 4 + 3]) {
                // new reference max across the tile's 64 keys (one head at a time)
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    float mx = sv[h];
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1)
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    if (lane == 0)
                        wmax_s[warp * 16 + h] = mx;
                }
                umma::named_bar(1, kSoftmaxWarps * 32);
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const float tmx = fmaxf(fmaxf(wmax_s[h], wmax_s[16 + h]), fmaxf(wmax_s[32 + h], wmax_s[48 + h]));
                    const float mn = fmaxf(m_ref[h], tmx);
                    const float al = (m_ref[h] == -INFINITY) ? 0.f : exp2f(m_ref[h] - mn);
                    m_ref[h] = mn;
                    l_part[h] *= al;
                    if (tid == 0)
                        alpha_s[h] = al;
                }
                umma::named_bar(1, kSoftmaxWarps * 32);
                if (i >= 1) {
                    // O^T holds PV(0..i-1): let PV(i-1) finish, then rescale each head (column)
                    wait_bar(o_done, (uint32_t)((i - 1) & 1));
                    umma::fence_after_sync();
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk) {
                        uint32_t o[16];
                        umma::ld16(tmem + 16 * blk + tm_lane, o);
                        umma::wait_ld();
#pragma unroll
                        for (int h = 0; h < 16; ++h)
                            o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha_s[h]);
                        umma::st16(tmem + 16 * blk + tm_lane, o);
                    }
                    umma::wait_st();
                }
            }
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const float mu = (m_ref[h] == -INFINITY) ? 0.f : m_ref[h];
                sv[h] = exp2f(sv[h] - mu);
                l_part[h] += sv[h];
            }
            if (i >= 2)
                wait_bar(p_empty(b), (uint32_t)(((i - 2) >> 1) & 1)); // PV(i-2) is done with this P buffer
            if (lane < 16) {
                const uint32_t prow = p_s + b * 2048 + (key >> 3) * 256 + (key & 7) * 16;
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow), "r"(pack_bf16x2(sv[0], sv[1])),
                             "r"(pack_bf16x2(sv[2], sv[3])), "r"(pack_bf16x2(sv[4], sv[5])),
                             "r"(pack_bf16x2(sv[6], sv[7])));
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + 128),
                             "r"(pack_bf16x2(sv[8], sv[9])), "r"(pack_bf16x2(sv[10], sv[11])),
                             "r"(pack_bf16x2(sv[12], sv[13])), "r"(pack_bf16x2(sv[14], sv[15])));
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            umma::mbar_arrive(p_full(b));
        }
        // ---- epilogue part 1: l per head, normalised O^T -> staging [16][512] fp32 ----
        if (ntiles > 0)
            wait_bar(o_done, (uint32_t)((ntiles - 1) & 1)); // the last PV (and every MMA) is done
        umma::fence_after_sync();
#pragma unroll
        for (int h = 0; h < 16; ++h) {
#pragma unroll
            for (int o = 8; o > 0; o >>= 1)
                l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < 16; ++h)
                lred_s[warp * 16 + h] = l_part[h];
        }
        umma::named_bar(1, kSoftmaxWarps * 32);
#pragma unroll
        for (int h = 0; h < 16; ++h) {
            if (tid == h) {
                const float l = lred_s[h] + lred_s[16 + h] + lred_s[32 + h] + lred_s[48 + h];
                lse_s[h] = l > 0.f ? (m_ref[h] + log2f(l)) * kLn2 : -INFINITY;
                alpha_s[h] = l > 0.f ? 1.0f / l : 0.f; // reused: 1 / l per head
            }
        }
        umma::named_bar(1, kSoftmaxWarps * 32);
        float *ost = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            uint32_t o[16];
            umma::ld16(tmem + 16 * blk + tm_lane, o);
            umma::wait_ld();
            const int d = blk * 128 + warp * 32 + lane;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const float iv = alpha_s[h];
                ost[h * kDv + d] = iv > 0.f ? __uint_as_float(o[h]) * iv : 0.f;
            }
        }
        umma::fence_before_sync();
    }
    __syncthreads();
    if (warp == 0)
        umma::dealloc(tmem, 128);
    finish_tile<kThreads>(a, reinterpret_cast<float *>(smem), lse_s, reinterpret_cast<float *>(smem + C::OFF_Q),
                          flag_s, t, 0, s, tid);
}

} // namespace

cudaError_t launch_fwd_umma16(const FwdArgs &a, cudaStream_t stream)
{
    auto kern = sparse_mla_fwd_umma16_kernel;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, U16::SMEM);
        if (e != cudaSuccess)
            return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    const int64_t blocks = (int64_t)a.T * a.S;
    if (blocks == 0)
        return cudaSuccess;
    if (a.S > 1 && a.S <= kClusterMaxSplits) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = U16::SMEM;
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
    kern<<<dim3((unsigned)blocks), dim3(kThreads), U16::SMEM, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t read_umma_error(int *out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_umma_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_umma_error, &zero, sizeof(int));
    }
    return e;
}

} // namespace smla
