// Sparse MLA forward for 128 heads with an E4M3 cache (D_qk = 576: 512
// latent + 64 rope columns, D_v = 512) on the 5th-generation tensor cores
// (tcgen05 + tensor memory) with TMA row gathers, sm_103a.
//
// With 128 heads QK runs head-major and PV dims-major:
//   S   [128 heads x 64 keys]  = q8 [128 x 576] . K_tile^T          (E4M3, 18 MMAs, M=128 N=64)
//   O^T [256 dims x 128 heads] += V^T[half] [256 x 64] . P^T        (fp16, 8 MMAs, 2 x M=128 N=128)
// The fp32 output for 128 heads x 512 dims alone would fill an SM's tensor
// memory (256 KB), so each query row runs as two CTAs, each owning one half
// of the value dims; both compute the full QK and softmax (identical inputs,
// identical P).
//
// Tensor memory (512 columns): O^T in 0..255 (two M-blocks of 128 dims x 128
// heads), S in 256 + 64 b (double-buffered), V^T in 384 + 64 b (binary16,
// two keys per column, double-buffered; the A operand of PV). Shared memory:
// q8 (4 swizzled blocks of [128 heads x 128 B] for the latent part plus an
// 8 KB core-matrix block for the rope part), a 3-stage ring of 40 KB tiles,
// and P^T (fp16, [128 heads x 64 keys] K-major, double-buffered; the B
// operand of PV).
//
// q is quantized per (row, head) by a separate pass over all rows (one warp
// per head: s_q = amax|q[t,h,:]| / 448, 1 if zero; q8 = RNE_satfinite(q /
// s_q)) into the workspace, the rope part already in core-matrix order; the
// CTA copies its 128 heads with four TMA tile loads and one bulk copy.
//
// Warp roles, handing tiles over through mbarriers (every wait bounded):
//   producers (warps 5-8): per 64-key tile 80 TMA tile::gather4 copies (16
//     key quads x 5 column blocks of 128 B; the last block reaches past
//     column 576 and is zero filled). Masked and out-of-range indices are
//     passed as row -1 (zero fill, no memory read).
//   QK issuer (warp 4): S(i) once tile i has landed and the softmax has read
//     S(i-2).
//   softmax (warps 0-3, thread = head, whole S row in the thread): masks,
//     scales by scale * s_q[h] * kv_scale, exponentiates base 2 against a
//     running reference max that moves (all heads agree per tile, then the
//     O^T columns are rescaled in tensor memory) only when a logit exceeds
//     it by more than 2^8, and then to 2^8 above the tile max; writes its
//     row of P^T (fp16).
//   converters (warps 10-13, one per quarter of the TMEM lanes): the tile's
//     half of the value columns, E4M3 -> binary16 (exact), as V^T into
//     tensor memory (4x4 byte transposes within lane quads).
//   PV issuer (warp 9): O^T += V^T(i) . P^T(i) once both are written.
//
// Method sources (page titles and sections):
//   "Enable AITER sparse MLA on gfx942, including FP8 KV" — Overview, Details
//     ("FP8 KV on gfx942": the kernel quantizes q per tile, dots in fp8).
//   "[ROCm][MLA][Perf] Fuse decode QK-RoPE + Q-concat + KV-concat + KV-cache
//     write for sparse MLA" — Summary (the cache row is the latent part
//     followed by the rope part, written as fp8).
#include "smla_device.cuh"
#include "smla_internal.h"
#include "smla_umma.cuh"

#include <atomic>
#include <climits>
#include <cmath>

namespace smla {

__device__ int g_wide_error = 0; // set when a bounded wait gives up

namespace {

constexpr int kHeads = 128;    // heads per CTA (M of QK, N of PV)
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kDvHalf = 256;   // value dims per CTA
constexpr int kKeys = 64;      // keys per tile (N of QK)
constexpr int kQkSteps = kDqk / 32;   // 18 E4M3 k-steps of 32
constexpr int kCB = 5;                // 128-byte column blocks per cache row (the last half used)
constexpr int kStages = 3;
constexpr int kCopies = 16 * kCB;     // gather4 copies per tile
constexpr int kIdxAhead = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f; // log2 units a logit may exceed the reference by
constexpr float kHeadroom = 8.0f;         // a moved reference sits this far above the tile max

// warps 0-3: softmax
constexpr int kQkWarp = 4;
constexpr int kProducerWarp0 = 5;     // warps 5-8
constexpr int kPvWarp = 9;
constexpr int kConverterWarp0 = 10;   // warps 10-13
constexpr int kThreads = 14 * 32;
constexpr int kProducerThreads = 128;
constexpr int kConverterThreads = 128;

// shared memory (bytes from a 1 KB-aligned base)
constexpr int kQBlk = kHeads * 128;           // one swizzled column block of q8 (16 KB)
constexpr int kOffQ8 = 0;                     // 4 blocks: columns 0..511
constexpr int kQRope = kHeads * 64;           // rope part in core matrices (8 KB)
constexpr int kOffQRope = kOffQ8 + 4 * kQBlk;
constexpr int kKBlk = kKeys * 128;            // one column block of a tile (8 KB)
constexpr int kTile = kCB * kKBlk;            // 40 KB
constexpr int kOffRing = kOffQRope + kQRope;
constexpr int kPT = kHeads * 128;             // P^T: 128 heads x 64 keys fp16 (16 KB)
constexpr int kOffPT = kOffRing + kStages * kTile;
constexpr int kOffAlpha = kOffPT + 2 * kPT;   // [128] per-head factors (rescale, then 1/l)
constexpr int kOffEx = kOffAlpha + kHeads * 4;// [2][4] exceed flags
constexpr int kOffMisc = kOffEx + 32;         // tmem address, abort, go[2]
constexpr int kOffMbar = kOffMisc + 32;
// full[3], empty[3], s_full[2], p_full[2], p_empty[2], v_full[2], q_full, drain
constexpr int kNBar = 16;
constexpr int kSmem = kOffMbar + kNBar * 8;
constexpr int kSmemAlloc = kSmem + 1024;
static_assert(kOffRing % 1024 == 0 && kOffPT % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kSmemAlloc <= 227 * 1024, "shared memory budget");

// tensor memory columns
constexpr int kTmemCols = 512;
constexpr int kSCol = 256;
constexpr int kVCol = 384;

// QK: A = q8 (K-major), B = K tile (K-major), M = 128 heads, N = 64 keys, E4M3
constexpr uint32_t kIdescQK = umma::idesc(128, 64, 0, 0, 0, 0);
// PV: A = V^T in tensor memory (fp16), B = P^T (K-major), M = 128 dims, N = 128 heads
constexpr uint32_t kIdescPV = umma::idesc(128, 128, 0, 0, 0, 0);

// q [rows x 576] bf16 (rows = T * H) -> E4M3 codes: columns 0..511 to q8
// [rows x 512], columns 512..575 to q8_rope in the core-matrix order the QK
// reads (per (row t, group of 128 heads) an 8 KB block: 8-head groups of 4
// chunks of 8 heads x 16 B), and the per-row scale. One warp per row; lanes
// 0-23 hold 24 elements each.
//
// With a pre-quantized q (codes [rows x 576] and one per-tensor scale) the
// codes are only rearranged and the scale copied to every row.
__global__ void __launch_bounds__(128) quantize_q_e4m3_kernel(const __nv_bfloat16 *__restrict__ q, int64_t rows, int H,
                                                             uint8_t *__restrict__ q8, uint8_t *__restrict__ q8_rope,
                                                             float *__restrict__ scale,
                                                             const uint8_t *__restrict__ codes_in,
                                                             const float *__restrict__ scale_in)
{
    const int64_t r = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows)
        return;
    if (codes_in != nullptr) {
        if (lane == 0)
            scale[r] = *scale_in;
        if (lane < 24) {
            const int64_t t = r / H;
            const int h = (int)(r % H), hg = h / kHeads, hl = h % kHeads;
            uint8_t *rope = q8_rope + (t * (H / kHeads) + hg) * kQRope;
#pragma unroll
            for (int u = 0; u < 3; ++u) {
                const int e0 = 24 * lane + 8 * u;
                const uint2 o = __ldg(reinterpret_cast<const uint2 *>(codes_in + r * kDqk + e0));
                if (e0 < 512) {
                    *reinterpret_cast<uint2 *>(q8 + r * 512 + e0) = o;
                } else {
                    const int d = e0 - 512;
                    *reinterpret_cast<uint2 *>(rope + ((hl >> 3) * 4 + (d >> 4)) * 128 + (hl & 7) * 16 + (d & 15)) = o;
                }
            }
        }
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(q + r * kDqk);
    uint4 v[3];
    float m = 0.f;
    if (lane < 24) {
#pragma unroll
        for (int u = 0; u < 3; ++u)
            v[u] = __ldg(src + 3 * lane + u);
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&v[u]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(b2[e]);
                m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    }
    m = warp_max(m);
    const float s = (m == 0.f) ? 1.0f : __fdiv_rn(m, 448.0f);
    const E4m3Recip inv = e4m3_recip(s);
    if (lane == 0)
        scale[r] = s;
    if (lane < 24) {
        const int64_t t = r / H;
        const int h = (int)(r % H), hg = h / kHeads, hl = h % kHeads;
        uint8_t *rope = q8_rope + (t * (H / kHeads) + hg) * kQRope;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
            const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&v[u]);
            const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
            const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
            uint2 o;
            o.x = quant4_e4m3(f0.x, f0.y, f1.x, f1.y, s, inv);
            o.y = quant4_e4m3(f2.x, f2.y, f3.x, f3.y, s, inv);
            const int e0 = 24 * lane + 8 * u; // first column of these 8 codes
            if (e0 < 512) {
                *reinterpret_cast<uint2 *>(q8 + r * 512 + e0) = o;
            } else {
                const int d = e0 - 512;
                *reinterpret_cast<uint2 *>(rope + ((hl >> 3) * 4 + (d >> 4)) * 128 + (hl & 7) * 16 + (d & 15)) = o;
            }
        }
    }
}

__global__ void __launch_bounds__(512, 1)
    sparse_mla_fwd_wide_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap kv_map,
                               const __grid_constant__ CUtensorMap q8_map)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    const uint32_t q8_s = sbase + kOffQ8, qrope_s = sbase + kOffQRope, ring = sbase + kOffRing,
                   pt_s = sbase + kOffPT;
    float *alpha_s = reinterpret_cast<float *>(smem + kOffAlpha);
    int *ex_s = reinterpret_cast<int *>(smem + kOffEx);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    int *abort_s = reinterpret_cast<int *>(smem + kOffMisc + 4);
    volatile int *go_s = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    const uint32_t bar0 = sbase + kOffMbar;
    auto full = [&](int st) { return bar0 + 8 * st; };
    auto empty = [&](int st) { return bar0 + 8 * (3 + st); };
    auto s_full = [&](int b) { return bar0 + 8 * (6 + b); };
    auto p_full = [&](int b) { return bar0 + 8 * (8 + b); };
    auto p_empty = [&](int b) { return bar0 + 8 * (10 + b); };
    auto v_full = [&](int b) { return bar0 + 8 * (12 + b); };
    const uint32_t q_full = bar0 + 8 * 14;
    const uint32_t drain = bar0 + 8 * 15;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.H / kHeads;
    const int half = blockIdx.x & 1;
    const int hg = (blockIdx.x >> 1) % G;
    const int t = (blockIdx.x >> 1) / G;
    const int ntiles = (a.topk + kKeys - 1) / kKeys;
    const int32_t *__restrict__ row_idx = a.indices + (int64_t)t * a.topk;

    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            umma::mbar_init(full(st), 1);
            umma::mbar_init(empty(st), 1 + kConverterThreads); // QK commit + converters
        }
        for (int b = 0; b < 2; ++b) {
            umma::mbar_init(s_full(b), 1);
            umma::mbar_init(p_full(b), 128);
            umma::mbar_init(p_empty(b), 1); // PV(i) done: P^T(b) and V^T(b) free, O^T holds PV(0..i)
            umma::mbar_init(v_full(b), kConverterThreads);
        }
        umma::mbar_init(q_full, 1);
        umma::mbar_init(drain, 2);
        umma::mbar_init_fence();
        *abort_s = 0;
    }
    if (warp == kQkWarp)
        umma::alloc(smem_u32(tmem_slot), kTmemCols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // the prologue above touches no global memory: from here on the previous
    // kernel in the stream (which may produce this call's inputs, or still
    // read this call's outputs) must be complete; the next one may start its
    // own prologue on free SMs meanwhile
    umma::grid_launch_dependents();
    umma::grid_wait();

    // ---- q8 of this CTA's 128 heads: four TMA tile loads and one bulk copy ----
    if (tid == 0) {
        umma::mbar_arrive_expect_tx(q_full, 4 * kQBlk + kQRope);
        const int qrow = t * a.H + hg * kHeads;
        for (int cb = 0; cb < 4; ++cb)
            umma::tma_load_2d(q8_s + cb * kQBlk, &q8_map, 128 * cb, qrow, q_full);
        umma::bulk_copy_g2s(qrope_s, a.q8_rope + ((int64_t)t * G + hg) * kQRope, kQRope, q_full);
    }

    auto wait_bar = [&](uint32_t mbar, uint32_t parity) {
        if (*(volatile int *)abort_s)
            return;
        if (!umma::mbar_wait(mbar, parity)) {
            atomicOr(&g_wide_error, 1);
            *(volatile int *)abort_s = 1;
        }
    };
    auto wait_issued = [&](uint32_t mbar, uint32_t parity) {
        if (!umma::mbar_wait(mbar, parity))
            atomicOr(&g_wide_error, 2);
    };

    if (warp >= kProducerWarp0 && warp < kProducerWarp0 + 4) {
        // ======================= producers =======================
        const int pt = tid - kProducerWarp0 * 32;
        // copy cid (20 per warp): key quad qd, column block cb
        const bool copier = (pt & 31) < kCopies / 4;
        const int cid = (pt >> 5) * (kCopies / 4) + (pt & 31);
        const int qd = cid / kCB, cb = cid % kCB;
        auto fetch = [&](int tile, int (&r)[4]) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = tile * kKeys + 4 * qd + u;
                r[u] = (copier && tile < ntiles && p < a.topk) ? __ldg(row_idx + p) : -1;
            }
        };
        auto row = [&](int x) { return (x >= 0 && (int64_t)x < a.num_slots) ? x : -1; };
        int r0[4], r1[4], r2[4], r3[4];
        static_assert(kIdxAhead == 4, "one register slot per tile of look-ahead");
        fetch(0, r0);
        fetch(1, r1);
        fetch(2, r2);
        fetch(3, r3);
        int issued = 0;
        bool stop = false;
        auto step = [&](int j, int(&r)[4]) {
            if (stop || j >= ntiles) {
                stop = true;
                return;
            }
            const int st = j % kStages;
            if (pt == 0) {
                if (j >= kStages)
                    wait_bar(empty(st), (uint32_t)((j / kStages - 1) & 1));
                const int go = !*(volatile int *)abort_s;
                if (go)
                    umma::mbar_arrive_expect_tx(full(st), kTile);
                go_s[j & 1] = go;
            }
            umma::named_bar(2, kProducerThreads);
            if (!go_s[j & 1]) {
                stop = true;
                return;
            }
            if (copier)
                umma::tma_gather4(ring + st * kTile + cb * kKBlk + qd * 512, &kv_map, 128 * cb, row(r[0]),
                                  row(r[1]), row(r[2]), row(r[3]), full(st));
            issued = j + 1;
            fetch(j + kIdxAhead, r);
        };
        for (int j0 = 0; !stop; j0 += kIdxAhead) {
            step(j0, r0);
            step(j0 + 1, r1);
            step(j0 + 2, r2);
            step(j0 + 3, r3);
        }
        if (pt == 0) {
            wait_issued(q_full, 0); // the q8 copies have landed (also after an abort)
            for (int j = max(0, issued - kStages); j < issued; ++j)
                wait_issued(full(j % kStages), (uint32_t)((j / kStages) & 1));
        }
    } else if (warp == kQkWarp) {
        // ======================= QK issuer =======================
        if (lane == 0) {
            wait_bar(q_full, 0);
            for (int i = 0; i < ntiles; ++i) {
                const int b = i & 1, st = i % kStages;
                wait_bar(full(st), (uint32_t)((i / kStages) & 1));
                if (i >= 2) // the softmax has read S(i-2)
                    wait_bar(p_full(b), (uint32_t)(((i - 2) >> 1) & 1));
                if (*(volatile int *)abort_s)
                    break;
                umma::fence_after_sync();
                const uint64_t ad = umma::desc_sw128(q8_s, 16, 1024);
                const uint64_t rd = umma::desc(qrope_s, 128, 512); // core matrices: K 128 B, M 512 B apart
                const uint64_t bd = umma::desc_sw128(ring + st * kTile, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < kQkSteps; ++ks) {
                    const uint64_t ak = ks < 16 ? ad + (uint64_t)(((ks >> 2) * kQBlk + (ks & 3) * 32) >> 4)
                                                : rd + (uint64_t)(((ks - 16) * 256) >> 4);
                    umma::mma_f8(tmem + kSCol + 64 * b, ak,
                                 bd + (uint64_t)(((ks >> 2) * kKBlk + (ks & 3) * 32) >> 4), kIdescQK, ks > 0);
                }
                umma::commit(s_full(b));
                umma::commit(empty(st));
            }
            umma::commit(drain);
            wait_issued(drain, 0);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ======================= PV issuer =======================
        if (lane == 0) {
            for (int i = 0; i < ntiles; ++i) {
                const int b = i & 1;
                wait_bar(p_full(b), (uint32_t)((i >> 1) & 1));
                wait_bar(v_full(b), (uint32_t)((i >> 1) & 1));
                if (*(volatile int *)abort_s)
                    break;
                umma::fence_after_sync();
                // P^T(b): K-major, 8-head atoms 1 KB apart; k-step kk starts 32 B into the rows
                const uint64_t bd = umma::desc_sw128(pt_s + b * kPT, 16, 1024);
#pragma unroll
                for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma::mma_f16_ts(tmem + 128 * mb, tmem + kVCol + 64 * b + 32 * mb + 8 * kk,
                                         bd + (uint64_t)((kk * 32) >> 4), kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                umma::commit(p_empty(b));
            }
            umma::commit(drain);
            wait_issued(drain, 0);
        }
        __syncwarp();
    } else if (warp >= kConverterWarp0) {
        // ======================= converters =======================
        // lane quad (g, ii): member ii loads 4 dims (4g..4g+3 of this warp's 32)
        // of key 4kq+ii; after the transpose it holds dim 4g+ii of keys 4kq..4kq+3
        const int q4 = warp & 3, g = lane >> 2, ii = lane & 3;
        const uint32_t selA = ii < 2 ? 0x5410u : 0x3276u; // keep / take 16-bit halves (xor 2)
        const uint32_t selB = ii & 1 ? 0x3715u : 0x6240u; // interleave bytes (xor 1)
        const uint32_t tlane = (uint32_t)(32 * q4) << 16;
        for (int i = 0; i < ntiles; ++i) {
            const int st = i % kStages, vb = i & 1;
            wait_bar(full(st), (uint32_t)((i / kStages) & 1));
            if (i >= 2) // PV(i-2) has read V^T buffer vb
                wait_bar(p_empty(vb), (uint32_t)(((i - 2) >> 1) & 1));
            const uint32_t src0 = ring + st * kTile;
#pragma unroll 1
            for (int mb = 0; mb < 2; ++mb) {
                const uint32_t blk = src0 + (2 * half + mb) * kKBlk; // E4M3 block: dims 256 half + 128 mb + ...
                uint32_t col[32];
#pragma unroll
                for (int kq = 0; kq < 16; ++kq) {
                    const int key = 4 * kq + ii;
                    const uint32_t w = lds32(blk + key * 128 + (((2 * q4 + (g >> 2)) ^ (key & 7)) << 4) + (g & 3) * 4);
                    const uint32_t x = __byte_perm(w, __shfl_xor_sync(0xffffffffu, w, 2), selA);
                    const uint32_t y = __byte_perm(x, __shfl_xor_sync(0xffffffffu, x, 1), selB);
                    e4m3x4_to_f16x4(y, col[2 * kq], col[2 * kq + 1]);
                }
                umma::st32(tmem + tlane + kVCol + 64 * vb + 32 * mb, col);
            }
            umma::wait_st();
            umma::fence_before_sync();
            umma::mbar_arrive(v_full(vb));
            umma::mbar_arrive(empty(st));
        }
    } else {
        // ======================= softmax (thread = head) =======================
        const int h = tid; // 0..127
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        const float kvs = *a.kv_scale;
        const float fac = a.scale * kLog2e * a.q_scale[(int64_t)t * a.H + hg * kHeads + h] * kvs;
        float m_ref = -INFINITY, l = 0.f;
        // validity of the tile's 64 keys (the same for every head): lane j
        // checks keys j and j + 32, a ballot gathers the mask
        auto load_idx = [&](int tile, int off) {
            const int p = tile * kKeys + off + lane;
            return (tile < ntiles && p < a.topk) ? __ldg(row_idx + p) : -1;
        };
        int xa0 = load_idx(0, 0), xb0 = load_idx(0, 32), xa1 = load_idx(1, 0), xb1 = load_idx(1, 32);
        int xa2 = load_idx(2, 0), xb2 = load_idx(2, 32), xa3 = load_idx(3, 0), xb3 = load_idx(3, 32);
        auto ok = [&](int x) { return x >= 0 && (int64_t)x < a.num_slots; };
        auto step = [&](int i, int &xa, int &xb) {
            if (i >= ntiles)
                return;
            const int b = i & 1;
            const uint32_t m_lo = __ballot_sync(0xffffffffu, ok(xa));
            const uint32_t m_hi = __ballot_sync(0xffffffffu, ok(xb));
            xa = load_idx(i + kIdxAhead, 0);
            xb = load_idx(i + kIdxAhead, 32);
            wait_bar(s_full(b), (uint32_t)((i >> 1) & 1));
            umma::fence_after_sync();
            float sv[64];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                umma::ld16(tl + kSCol + 64 * b + 16 * c, reinterpret_cast<uint32_t(&)[16]>(sv[16 * c]));
            umma::wait_ld();
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const bool v = ((j < 32 ? m_lo >> j : m_hi >> (j - 32)) & 1u) != 0;
                sv[j] = v ? sv[j] * fac : -INFINITY;
                mt = fmaxf(mt, sv[j]);
            }
            // move the reference max: every head's O^T column spans all four warps'
            // lanes, so the four softmax warps agree on it per tile
            const bool exceed = mt > m_ref + kRescaleThreshold;
            const bool wx = __any_sync(0xffffffffu, exceed);
            if (lane == 0)
                ex_s[b * 4 + warp] = wx;
            umma::named_bar(1, 128);
            if (ex_s[b * 4] | ex_s[b * 4 + 1] | ex_s[b * 4 + 2] | ex_s[b * 4 + 3]) {
                const float mn = exceed ? mt + kHeadroom : m_ref;
                const float al = !exceed ? 1.f : (m_ref == -INFINITY ? 0.f : exp2f(m_ref - mn));
                m_ref = mn;
                l *= al;
                alpha_s[h] = al;
                umma::named_bar(1, 128);
                if (i >= 1) {
                    // O^T holds PV(0..i-1): let PV(i-1) finish, then scale each head column
                    wait_bar(p_empty((i - 1) & 1), (uint32_t)(((i - 1) >> 1) & 1));
                    umma::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < 2 * kHeads; c += 16) {
                        uint32_t o[16];
                        umma::ld16(tl + c, o);
                        umma::wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha_s[(c + e) & (kHeads - 1)]);
                        umma::st16(tl + c, o);
                    }
                    umma::wait_st();
                }
                umma::named_bar(1, 128); // alpha_s is read by all before the next tile writes it
            }
            const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
            uint32_t pw[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = ex2_approx(sv[2 * c] - mu), p1 = ex2_approx(sv[2 * c + 1] - mu);
                l += p0 + p1;
                pw[c] = pack_f16x2(p0, p1);
            }
            if (i >= 2) // PV(i-2) has read P^T(b)
                wait_bar(p_empty(b), (uint32_t)(((i - 2) >> 1) & 1));
            // this head's row of P^T: 64 keys x fp16 = one 128-byte swizzled row
            const uint32_t prow = pt_s + b * kPT + h * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + ((c ^ (h & 7)) << 4)),
                             "r"(pw[4 * c]), "r"(pw[4 * c + 1]), "r"(pw[4 * c + 2]), "r"(pw[4 * c + 3])
                             : "memory");
            umma::fence_async_smem();
            umma::fence_before_sync();
            umma::mbar_arrive(p_full(b));
        };
        for (int i0 = 0; i0 < ntiles; i0 += kIdxAhead) {
            step(i0, xa0, xb0);
            step(i0 + 1, xa1, xb1);
            step(i0 + 2, xa2, xb2);
            step(i0 + 3, xa3, xb3);
        }
        // ---- epilogue: O^T / l -> out, lse ----
        if (ntiles > 0) // the last PV (and every earlier one) is done
            wait_bar(p_empty((ntiles - 1) & 1), (uint32_t)(((ntiles - 1) >> 1) & 1));
        umma::fence_after_sync();
        {
            // output factor and lse per head; a sink logit (base-2 units sk) joins the
            // denominator: l 2^m_ref + 2^sk, taken relative to M = max(m_ref, sk)
            const float sk = a.sinks != nullptr ? a.sinks[hg * kHeads + h] * kLog2e : -INFINITY;
            float f = 0.f, lse_h = -INFINITY;
            if (l > 0.f) {
                const float M = fmaxf(m_ref, sk);
                const float lt = l * exp2f(m_ref - M) + (sk == -INFINITY ? 0.f : exp2f(sk - M));
                f = kvs * exp2f(m_ref - M) / lt;
                lse_h = (M + log2f(lt)) * kLn2;
            } else if (sk != -INFINITY) {
                lse_h = sk * kLn2; // no valid key: the sink alone
            }
            alpha_s[h] = f; // output factor per head
            if (half == 0 && a.lse != nullptr)
                a.lse[(int64_t)t * a.H + hg * kHeads + h] = lse_h;
        }
        umma::named_bar(1, 128);
        // thread = value dim 128 mb + 32 warp + lane; columns = heads
        __nv_bfloat16 *obase = static_cast<__nv_bfloat16 *>(a.out) + ((int64_t)t * a.H + hg * kHeads) * kDv +
                               half * kDvHalf + warp * 32 + lane;
#pragma unroll 1
        for (int mb = 0; mb < 2; ++mb) {
#pragma unroll 1
            for (int c = 0; c < kHeads; c += 16) {
                uint32_t o[16];
                umma::ld16(tl + 128 * mb + c, o);
                umma::wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float f = alpha_s[c + e];
                    obase[(int64_t)(c + e) * kDv + 128 * mb] = __float2bfloat16_rn(f > 0.f ? __uint_as_float(o[e]) * f : 0.f);
                }
            }
        }
        umma::fence_before_sync();
    }
    __syncthreads();
    if (warp == kQkWarp)
        umma::dealloc(tmem, kTmemCols);
}

} // namespace

cudaError_t launch_quantize_q_wide(const FwdArgs &a, cudaStream_t stream)
{
    const int64_t qrows = (int64_t)a.T * a.H;
    if (qrows == 0)
        return cudaSuccess;
    quantize_q_e4m3_kernel<<<dim3((unsigned)((qrows + 3) / 4)), dim3(128), 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(a.q), qrows, a.H, a.q8, a.q8_rope, a.q_scale,
        a.q_fp8_in ? static_cast<const uint8_t *>(a.q) : nullptr, a.q_scale_in);
    return cudaGetLastError();
}

cudaError_t launch_fwd_wide(const FwdArgs &a, cudaStream_t stream)
{
    auto kern = sparse_mla_fwd_wide_kernel;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess)
            return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    const int64_t blocks = (int64_t)a.T * (a.H / kHeads) * 2;
    if (blocks == 0)
        return cudaSuccess;
    // The cache as a 2-D tensor [rows x 576] bytes, read in boxes of 128 bytes
    // x 1 row with the 128-byte swizzle (the fifth box of a row reaches past
    // column 576 and is zero filled).
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr)
        return cudaErrorNotSupported;
    CUtensorMap kv_map;
    const int64_t rows = a.num_slots < 1 ? 1 : (a.num_slots > INT_MAX ? (int64_t)INT_MAX : a.num_slots);
    cuuint64_t gdim[2] = {(cuuint64_t)kDqk, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)kDqk};
    cuuint32_t box[2] = {128, 1};
    cuuint32_t estride[2] = {1, 1};
    if (encode(&kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(a.kv), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // q8 (latent part) as a 2-D tensor [T*H rows x 512] bytes, copied in boxes
    // of 128 B x 128 rows with the 128-byte swizzle
    CUtensorMap q8_map;
    cuuint64_t qdim[2] = {512, (cuuint64_t)a.T * a.H};
    cuuint64_t qstride[1] = {512};
    cuuint32_t qbox[2] = {128, (cuuint32_t)kHeads};
    if (encode(&q8_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.q8, qdim, qstride, qbox, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (const cudaError_t qe = launch_quantize_q_wide(a, stream); qe != cudaSuccess)
        return qe;
    // programmatic dependent launch: the kernel's prologue overlaps the q pass's
    // tail; it waits for it in grid_wait before reading q8
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a, kv_map, q8_map);
}

cudaError_t read_wide_error(int *out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_wide_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_wide_error, &zero, sizeof(int));
    }
    return e;
}

} // namespace smla
