// Sparse MLA forward for 16 heads over an E4M3 cache with fp8 dots, in lean
// CTAs that run two to an SM (tcgen05 + tensor memory, TMA row gathers,
// sm_103a).
//
// The row gather is the bound of this path, and the rate at which a CTA's
// gathers complete is limited per CTA: random 512-byte rows arrive about
// twice as fast with two or three CTAs per SM as with one (measured with the
// gather probe). So each CTA here stays within half an SM: at most 113 KB of
// shared memory, 256 columns of tensor memory and 448 threads (72 registers
// each; the softmax keeps its per-head reference max in shared memory to fit).
//
// One CTA = (query row t, split s of its top-k list). As in the 16-head
// kernel the contraction runs transposed, keys on the MMA's M axis:
//   S^T [64 keys x 16 heads] = KV_tile [64 x 512] . q8^T         (QK, E4M3, M=64, N=16)
//   O^T [512 dims x 16 heads] += V^T [512 x 64 keys] . P^T       (PV, fp16, 4 x M=128, N=16)
// Tensor memory: O^T in columns 0..63, S^T in 64 + 16 b (two buffers), and
// V^T (binary16, two keys per column; the A operand of PV) in two half
// buffers of 256 dims each at 128 + 64 h. The conversion of a tile's first
// half waits only for the previous tile's PV over that half.
//
// Warp roles, handing tiles over through mbarriers (every wait bounded):
//   softmax (warps 0-3, one key per thread of lanes 0-15): as in the 16-head
//     kernel (lazy reference max, rescale of O^T in tensor memory only when
//     a logit passes the reference by more than 2^8), writes P^T (fp16). The
//     reference max per head, the same in every softmax thread, lives in
//     shared memory (two buffers: the new one is written while the old one
//     is read).
//   QK issuer (warp 4), PV issuer (warp 5): one thread each.
//   producers (warps 6-9): one gather4 copy per thread of lanes 0-15 per tile
//     (16 key quads x 4 column blocks of 128 codes; a warp issues its lanes'
//     copies one after another, so four warps issue a tile in half the time
//     of two) into a 3-stage ring; -1 and out-of-range indices go to the TMA
//     as row -1 (zero fill, no read).
//   converters (warps 10-13, one per quarter of the TMEM lanes): first q,
//     quantized per (row, head) straight from global memory (s_q =
//     amax/448, q8 = RNE_satfinite(q / s_q)), or the pre-quantized codes;
//     then per tile each half of the values, E4M3 -> binary16 (exact), as
//     V^T into tensor memory (transposing ldmatrix of 8 keys x 16 bytes, a
//     byte permute, 16x256b stores; the lane and K orders this gives are
//     kVLaneDim and kPRow below).
// Splits of a row merge as in the 16-head kernel (a cluster of up to 8 CTAs
// through distributed shared memory, or the workspace ticket merge).
//
// Method sources (page titles and sections):
//   "Enable AITER sparse MLA on gfx942, including FP8 KV" — Details ("FP8 KV
//     on gfx942": q quantized per tile in the kernel, dots in fp8).
//   "Route gfx942 sparse MLA prefill to AITER pa_prefill_sparse" — jin-amd
//     A/B: split-K for decode-sized calls.
#include "smla_device.cuh"
#include "smla_epilogue.cuh"
#include "smla_internal.h"
#include "smla_umma.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>

namespace smla {

__device__ int g_lean_error = 0; // set when a bounded wait gives up

namespace {

constexpr int kSoftmaxWarps = 4;
constexpr int kQkWarp = 4;
constexpr int kPvWarp = 5;
constexpr int kProducerWarp0 = 6;
constexpr int kProducerThreads = 128;
constexpr int kConverterWarp0 = 10;
constexpr int kConverterThreads = 128;
constexpr int kThreads = 14 * 32;
constexpr int kKeys = kUmma16TileKeys; // keys per tile (M of QK)
constexpr int kHeads = 16;
constexpr int kD = 512;
constexpr int kNcb = 4;                 // 128-code column blocks per row
constexpr int kBlk = kKeys * 128;       // one column block of a tile (8 KB)
constexpr int kTile = kNcb * kBlk;      // 32 KB
constexpr int kStages = 3;
constexpr int kQkMmas = kD / 32;        // E4M3 k-steps per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kHeadroom = 8.0f;
constexpr int kIdxAhead = 4;

// shared memory (bytes from a 1 KB-aligned base)
constexpr int kOffQ = kStages * kTile;            // q8 [16 x 512] in core matrices (8 KB)
constexpr int kQGrp = 8 * kD;                     // 8 heads x 512 codes
constexpr int kOffP = kOffQ + 2 * kQGrp;          // P^T [64 keys x 16 heads] fp16, 2 x 2 KB
constexpr int kOffSq = kOffP + 2 * 2048;          // [16] per-head q scales
constexpr int kOffFac = kOffSq + 16 * 4;          // [16] per-head logit factors
constexpr int kOffEx = kOffFac + 16 * 4;          // [2][4] exceed flags
constexpr int kOffGo = kOffEx + 32;               // [2] producer issue decisions
constexpr int kOffWmax = kOffGo + 8;
constexpr int kOffLred = kOffWmax + 4 * 16 * 4;
constexpr int kOffLse = kOffLred + 4 * 16 * 4;
constexpr int kOffAlpha = kOffLse + 16 * 4;
constexpr int kOffMisc = kOffAlpha + 16 * 4;      // flag, tmem address, abort
constexpr int kOffMref = kOffMisc + 16;            // [2][16] reference max per head (double-buffered)
constexpr int kOffMbar = (kOffMref + 128 + 7) & ~7;
// full[3], empty[3], s_full[2], p_full[2], p_empty[2], q_full, drain, v_full[2], v_free[2]
constexpr int kNBar = 2 * kStages + 6 + 2 + 4;
constexpr int kSmem = kOffMbar + kNBar * 8;
constexpr int kSmemAlloc = kSmem + 1024;
static_assert(kSmemAlloc <= 113 * 1024, "two CTAs per SM");
static_assert(kStages * kTile >= kHeads * kD * 4, "epilogue staging fits in the ring");
static_assert(2 * kQGrp >= 128 * kHeads * 4, "merge weights fit in the q area");

// tensor memory columns
constexpr int kTmemCols = 256;
constexpr int kSCol = 64;
constexpr int kVCol = 128;

// V^T layout in tensor memory (as the converters write it): lane 32w + l of a
// 128-dim block holds dim 32w + kVLaneDim(l); within a 16-key group the K
// order of the PV contraction is keys 0,1,8,9, 2,3,10,11, 4,5,12,13, 6,7,14,15,
// so key k's P^T row is kPRow(k)
__device__ __forceinline__ int kVLaneDim(int l)
{
    const int r = l & 15;
    return (l & 16) + (r < 8 ? 2 * r : 2 * r - 15);
}
__device__ __forceinline__ int kPRow(int key)
{
    const int s = key & 15;
    return (key & ~15) + 4 * ((s >> 1) & 3) + 2 * (s >> 3) + (s & 1);
}

constexpr uint32_t kIdescQK = umma::idesc(64, 16, 0, 0, 0, 0);        // E4M3 x E4M3, K-major
constexpr uint32_t kIdescPV = umma::idesc(128, 16, 0, 0, 0, 1);       // fp16: A in TMEM, B = P^T MN-major

__global__ void __launch_bounds__(kThreads, 2)
    sparse_mla_fwd_lean16_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap kv_map)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    const uint32_t ring = sbase, q_s = sbase + kOffQ, p_s = sbase + kOffP;
    float *sq_s = reinterpret_cast<float *>(smem + kOffSq);
    float *fac_s = reinterpret_cast<float *>(smem + kOffFac);
    int *ex_s = reinterpret_cast<int *>(smem + kOffEx);
    volatile int *go_s = reinterpret_cast<volatile int *>(smem + kOffGo);
    float *wmax_s = reinterpret_cast<float *>(smem + kOffWmax);
    float *lred_s = reinterpret_cast<float *>(smem + kOffLred);
    float *lse_s = reinterpret_cast<float *>(smem + kOffLse);
    float *alpha_s = reinterpret_cast<float *>(smem + kOffAlpha);
    int *flag_s = reinterpret_cast<int *>(smem + kOffMisc);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc + 4);
    int *abort_s = reinterpret_cast<int *>(smem + kOffMisc + 8);
    const uint32_t bar0 = sbase + kOffMbar;
    auto full = [&](int st) { return bar0 + 8 * st; };
    auto empty = [&](int st) { return bar0 + 8 * (kStages + st); };
    auto s_full = [&](int b) { return bar0 + 8 * (2 * kStages + b); };
    auto p_full = [&](int b) { return bar0 + 8 * (2 * kStages + 2 + b); };
    auto p_empty = [&](int b) { return bar0 + 8 * (2 * kStages + 4 + b); };
    const uint32_t q_full = bar0 + 8 * (2 * kStages + 6);
    const uint32_t drain = bar0 + 8 * (2 * kStages + 7);
    auto v_full = [&](int h) { return bar0 + 8 * (2 * kStages + 8 + h); };
    auto v_free = [&](int h) { return bar0 + 8 * (2 * kStages + 10 + h); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x % a.S;
    const int t = blockIdx.x / a.S;
    const int kb = s * a.keys_per_split;
    const int ke = min(a.topk, kb + a.keys_per_split);
    const int ntiles = ke > kb ? (ke - kb + kKeys - 1) / kKeys : 0;
    const int32_t *__restrict__ row_idx = a.indices + (int64_t)t * a.topk;

    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            umma::mbar_init(full(st), 1);
            umma::mbar_init(empty(st), 1 + kConverterThreads); // the QK commit + every converter
        }
        for (int b = 0; b < 2; ++b) {
            umma::mbar_init(s_full(b), 1);
            umma::mbar_init(p_full(b), kSoftmaxWarps * 32);
            umma::mbar_init(p_empty(b), 1);
            umma::mbar_init(v_full(b), kConverterThreads);
            umma::mbar_init(v_free(b), 1);
        }
        umma::mbar_init(q_full, kConverterThreads);
        umma::mbar_init(drain, 2);
        umma::mbar_init_fence();
        *abort_s = 0;
    }
    if (warp == 0)
        umma::alloc(smem_u32(tmem_slot), kTmemCols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // the prologue above touches no global memory: from here on the previous
    // kernel in the stream must be complete; the next one may start its own
    // prologue meanwhile (on a free half of an SM)
    umma::grid_launch_dependents();
    umma::grid_wait();

    auto wait_bar = [&](uint32_t mbar, uint32_t parity) {
        if (*(volatile int *)abort_s)
            return;
        if (!umma::mbar_wait(mbar, parity)) {
            atomicOr(&g_lean_error, 1);
            *(volatile int *)abort_s = 1;
        }
    };
    auto wait_issued = [&](uint32_t mbar, uint32_t parity) {
        if (!umma::mbar_wait(mbar, parity))
            atomicOr(&g_lean_error, 2);
    };

    if (warp >= kProducerWarp0 && warp < kConverterWarp0) {
        // ======================= producers =======================
        const int pt = tid - kProducerWarp0 * 32;
        const bool copier = (pt & 31) < 16; // copy cid: key quad cid / 4, column block cid % 4
        const int cid = (pt >> 5) * 16 + (pt & 15);
        const int qd = cid / kNcb, cb = cid % kNcb;
        auto fetch = [&](int tile, int (&r)[4]) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = kb + tile * kKeys + 4 * qd + u;
                r[u] = (copier && tile < ntiles && p < ke) ? __ldg(row_idx + p) : -1;
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
            // all or none of a tile's copies are issued, so a stage's barrier
            // always completes once its copies are in flight
            umma::named_bar(2, kProducerThreads);
            if (!go_s[j & 1]) {
                stop = true;
                return;
            }
            if (copier)
                umma::tma_gather4(ring + st * kTile + cb * kBlk + qd * 512, &kv_map, 128 * cb, row(r[0]), row(r[1]),
                                  row(r[2]), row(r[3]), full(st));
            issued = j + 1;
            fetch(j + kIdxAhead, r);
        };
        for (int j0 = 0; !stop; j0 += kIdxAhead) {
            step(j0, r0);
            step(j0 + 1, r1);
            step(j0 + 2, r2);
            step(j0 + 3, r3);
        }
        // every copy issued has landed before the CTA can finish (also after an abort)
        if (pt == 0) {
            for (int j = max(0, issued - kStages); j < issued; ++j)
                wait_issued(full(j % kStages), (uint32_t)((j / kStages) & 1));
        }
    } else if (warp == kQkWarp) {
        // ======================= QK issuer =======================
        if (lane == 0) {
            wait_bar(q_full, 0);
            const uint64_t qdesc = umma::desc(q_s, 128, kQGrp);
            for (int i = 0; i < ntiles; ++i) {
                const int b = i & 1, st = i % kStages;
                wait_bar(full(st), (uint32_t)((i / kStages) & 1));
                if (i >= 2) // the softmax has read S buffer b for tile i-2
                    wait_bar(p_full(b), (uint32_t)(((i - 2) >> 1) & 1));
                if (*(volatile int *)abort_s)
                    break;
                umma::fence_after_sync();
                // KV tile: K-major, 8-key atoms 1 KB apart; k-step ks reads column
                // block ks/4, starting 32 B * (ks%4) into its 128-byte rows
                const uint64_t ad = umma::desc_sw128(ring + st * kTile, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < kQkMmas; ++ks) {
                    const uint64_t ak = ad + (uint64_t)(((ks >> 2) * kBlk + (ks & 3) * 32) >> 4);
                    const uint64_t bk = qdesc + (uint64_t)(ks * 16); // 2 core matrices of q per k-step
                    umma::mma_f8(tmem + kSCol + 16 * b, ak, bk, kIdescQK, ks > 0);
                }
                umma::commit(s_full(b));
                umma::commit(empty(st)); // QK(i) no longer reads the stage
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
                const uint64_t bd = umma::desc(p_s + b * 2048, 256, 128);
                for (int h = 0; h < 2; ++h) {
                    wait_bar(v_full(h), (uint32_t)(i & 1)); // V^T half h holds tile i
                    if (*(volatile int *)abort_s)
                        break;
                    umma::fence_after_sync();
                    // M-block 2h + m: V^T half h at +32 m, 16 keys = 8 columns
                    const uint32_t va = tmem + kVCol + 64 * h;
#pragma unroll
                    for (int m = 0; m < 2; ++m)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma::mma_f16_ts(tmem + 16 * (2 * h + m), va + 32 * m + 8 * kk, bd + (uint64_t)(kk * 32),
                                             kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                    umma::commit(v_free(h));
                }
                if (*(volatile int *)abort_s)
                    break;
                // p_empty(b) also tells the softmax that O^T holds PV(0..i)
                umma::commit(p_empty(b));
            }
            umma::commit(drain);
            wait_issued(drain, 0);
        }
        __syncwarp();
    } else if (warp >= kConverterWarp0) {
        // ======================= converters =======================
        const int ct = tid - kConverterWarp0 * 32;
        {
            // q: thread ct handles 64 columns of head ct/8 (the 8 threads of a
            // head are adjacent lanes), into core matrices (8 heads x 16 B)
            const int h = ct >> 3, c0 = (ct & 7) * 64;
            if (a.q_fp8_in) {
                const uint8_t *q8g = static_cast<const uint8_t *>(a.q) + ((int64_t)t * kHeads + h) * kD + c0;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(q8g) + u);
                    const int c = (c0 >> 4) + u; // 16-code column of the head's row
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(q_s + (h >> 3) * kQGrp + c * 128 +
                                                                                 (h & 7) * 16),
                                 "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                                 : "memory");
                }
                if (ct < kHeads) // one per-tensor scale for every head
                    sq_s[ct] = *a.q_scale_in;
            } else {
                const uint4 *qg = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q) +
                                                                  ((int64_t)t * kHeads + h) * kD + c0);
                uint4 qraw[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    qraw[u] = __ldg(qg + u);
                float m = 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&qraw[u]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(b2[e]);
                        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
                    }
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                const float sq = (m == 0.f) ? 1.0f : __fdiv_rn(m, 448.0f);
                if ((ct & 7) == 0)
                    sq_s[h] = sq;
                const E4m3Recip inv = e4m3_recip(sq);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t w[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&qraw[2 * cc + v / 2]);
                        const float2 f0 = __bfloat1622float2(b2[2 * (v & 1)]);
                        const float2 f1 = __bfloat1622float2(b2[2 * (v & 1) + 1]);
                        w[v] = quant4_e4m3(f0.x, f0.y, f1.x, f1.y, sq, inv);
                    }
                    const int c = (c0 >> 4) + cc;
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(q_s + (h >> 3) * kQGrp + c * 128 +
                                                                                 (h & 7) * 16),
                                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
            }
            umma::fence_async_smem();
            umma::mbar_arrive(q_full);
        }
        // values: this warp's 32 dims of each 128-dim block are two 16-dim
        // chunks (16 bytes of every key row). A transposing ldmatrix of 8 keys x
        // 16 bytes hands lane (c, j) = (lane / 4, lane % 4) dims 2c, 2c+1 of keys
        // 2j, 2j+1; one byte permute pairs the two keys of each dim, and the
        // 16x256b store puts dim 2c at TMEM lane c and dim 2c+1 at lane c + 8 of
        // the chunk's 16 lanes (kVLaneDim; the softmax reads O^T back that way),
        // keys 16G + 2j, +1 at column 8G + 2j and keys 16G + 8 + 2j, +1 at column
        // 8G + 2j + 1 (kPRow orders P^T's rows the same way)
        const int q4 = warp & 3;
        for (int i = 0; i < ntiles; ++i) {
            const int st = i % kStages;
            wait_bar(full(st), (uint32_t)((i / kStages) & 1));
            const uint32_t src0 = ring + st * kTile;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                if (i >= 1) // PV(i-1) has read V^T half h
                    wait_bar(v_free(h), (uint32_t)((i - 1) & 1));
#pragma unroll 1
                for (int m = 0; m < 2; ++m) {
                    const int mb = 2 * h + m;
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int cl = 2 * q4 + u; // the chunk's 16-byte slot in its line, before the swizzle
                        uint32_t col[16];
#pragma unroll
                        for (int g2 = 0; g2 < 2; ++g2) {
                            // matrix mm = lane / 8: keys 32 g2 + 8 mm .. +7, i.e. key group
                            // G = 2 g2 + mm / 2, its first (mm even) or second 8 keys
                            const int key = 32 * g2 + 8 * (lane >> 3) + (lane & 7);
                            uint32_t d[4];
                            ldsm_x4_trans(src0 + mb * kBlk + key * 128 + ((cl ^ (lane & 7)) << 4), d);
#pragma unroll
                            for (int mm = 0; mm < 4; ++mm) {
                                const int G = 2 * g2 + (mm >> 1), ab = mm & 1;
                                // bytes (key 2j: dim 2c, 2c+1), (key 2j+1: dim 2c, 2c+1) -> per dim
                                e4m3x4_to_f16x4(__byte_perm(d[mm], 0u, 0x3120u), col[4 * G + ab], col[4 * G + 2 + ab]);
                            }
                        }
                        umma::st16x256b_x4(tmem + ((uint32_t)(32 * q4 + 16 * u) << 16) + kVCol + 64 * h + 32 * m, col);
                    }
                }
                umma::wait_st();
                umma::fence_before_sync();
                umma::mbar_arrive(v_full(h));
            }
            umma::mbar_arrive(empty(st)); // done reading the stage
        }
    } else {
        // ======================= softmax =======================
        const uint32_t tm_lane = (uint32_t)(warp * 32) << 16;
        const int key = warp * 16 + lane; // meaningful for lane < 16
        const float kvs = *a.kv_scale;
        wait_bar(q_full, 0); // the per-head q scales
        float *mref_s = reinterpret_cast<float *>(smem + kOffMref);
        int mcur = 0;
        if (tid < 16) {
            fac_s[tid] = a.scale * kLog2e * sq_s[tid] * kvs;
            mref_s[tid] = -INFINITY;
        }
        umma::named_bar(1, kSoftmaxWarps * 32);
        float l_part[16];
#pragma unroll
        for (int h = 0; h < 16; ++h)
            l_part[h] = 0.f;
        auto load_idx = [&](int tile) {
            const int p = kb + tile * kKeys + key;
            return (lane < 16 && tile < ntiles && p < ke) ? __ldg(row_idx + p) : -1;
        };
        int x0 = load_idx(0), x1 = load_idx(1), x2 = load_idx(2), x3 = load_idx(3);
        auto step = [&](int i, int &my_idx) {
            if (i >= ntiles)
                return;
            const int b = i & 1;
            const bool kvalid = my_idx >= 0 && (int64_t)my_idx < a.num_slots;
            my_idx = load_idx(i + kIdxAhead);
            wait_bar(s_full(b), (uint32_t)((i >> 1) & 1));
            umma::fence_after_sync();
            float sv[16];
            umma::ld16(tmem + kSCol + 16 * b + tm_lane, reinterpret_cast<uint32_t(&)[16]>(sv));
            umma::wait_ld();
            bool exceed = false;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                sv[h] = kvalid ? sv[h] * fac_s[h] : -INFINITY;
                exceed |= sv[h] > mref_s[mcur * 16 + h] + kRescaleThreshold;
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
                    const float mo = mref_s[mcur * 16 + h];
                    const float mn = fmaxf(mo, tmx + kHeadroom);
                    const float al = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
                    l_part[h] *= al;
                    if (tid == 0) {
                        alpha_s[h] = al;
                        mref_s[(mcur ^ 1) * 16 + h] = mn;
                    }
                }
                umma::named_bar(1, kSoftmaxWarps * 32);
                mcur ^= 1;
                if (i >= 1) {
                    // O^T holds PV(0..i-1): let PV(i-1) finish (its P buffer's barrier; this
                    // thread already waited there for PV(i-3), so the phase cannot alias),
                    // then rescale each head (column)
                    wait_bar(p_empty((i - 1) & 1), (uint32_t)(((i - 1) >> 1) & 1));
                    umma::fence_after_sync();
                    // eight columns at a time: the live registers stay within two CTAs per SM
#pragma unroll 1
                    for (int c = 0; c < 64; c += 8) {
                        uint32_t o[8];
                        umma::ld8(tmem + c + tm_lane, o);
                        umma::wait_ld();
#pragma unroll
                        for (int h = 0; h < 8; ++h)
                            o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha_s[(c & 15) + h]);
                        umma::st8(tmem + c + tm_lane, o);
                    }
                    umma::wait_st();
                }
            }
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const float mr = mref_s[mcur * 16 + h];
                const float mu = (mr == -INFINITY) ? 0.f : mr;
                sv[h] = ex2_approx(sv[h] - mu);
                l_part[h] += sv[h];
            }
            if (i >= 2)
                wait_bar(p_empty(b), (uint32_t)(((i - 2) >> 1) & 1)); // PV(i-2) is done with this P buffer
            if (lane < 16) {
                const int pk = kPRow(key);
                const uint32_t prow = p_s + b * 2048 + (pk >> 3) * 256 + (pk & 7) * 16;
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow), "r"(pack_f16x2(sv[0], sv[1])),
                             "r"(pack_f16x2(sv[2], sv[3])), "r"(pack_f16x2(sv[4], sv[5])), "r"(pack_f16x2(sv[6], sv[7])));
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + 128), "r"(pack_f16x2(sv[8], sv[9])),
                             "r"(pack_f16x2(sv[10], sv[11])), "r"(pack_f16x2(sv[12], sv[13])),
                             "r"(pack_f16x2(sv[14], sv[15])));
            }
            umma::fence_async_smem();
            umma::fence_before_sync();
            umma::mbar_arrive(p_full(b));
        };
        for (int i0 = 0; i0 < ntiles; i0 += kIdxAhead) {
            step(i0, x0);
            step(i0 + 1, x1);
            step(i0 + 2, x2);
            step(i0 + 3, x3);
        }
        // ---- epilogue part 1: l per head, normalised O^T -> staging [16][512] fp32 ----
        if (ntiles > 0) // the last PV is done (and with it every earlier PV)
            wait_bar(p_empty((ntiles - 1) & 1), (uint32_t)(((ntiles - 1) >> 1) & 1));
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
        if (tid < 16) { // thread h finishes head h
            const float mh = mref_s[mcur * 16 + tid];
            const float l = lred_s[tid] + lred_s[16 + tid] + lred_s[32 + tid] + lred_s[48 + tid];
            lse_s[tid] = l > 0.f ? (mh + log2f(l)) * kLn2 : -INFINITY;
            alpha_s[tid] = l > 0.f ? kvs / l : 0.f; // reused: output factor per head
        }
        umma::named_bar(1, kSoftmaxWarps * 32);
        float *ost = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t o[2][16];
#pragma unroll
            for (int u = 0; u < 2; ++u)
                umma::ld16(tmem + 16 * (2 * half + u) + tm_lane, o[u]);
            umma::wait_ld();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int d = (2 * half + u) * 128 + warp * 32 + kVLaneDim(lane);
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const float iv = alpha_s[h];
                    ost[h * kD + d] = iv > 0.f ? __uint_as_float(o[u][h]) * iv : 0.f;
                }
            }
        }
        umma::fence_before_sync();
    }
    __syncthreads();
    if (warp == 0)
        umma::dealloc(tmem, kTmemCols);
    finish_tile<kThreads>(a, reinterpret_cast<float *>(smem), lse_s, reinterpret_cast<float *>(smem + kOffQ), flag_s,
                          t, 0, s, tid);
}

} // namespace

cudaError_t launch_fwd_lean16(const FwdArgs &a, cudaStream_t stream)
{
    auto kern = sparse_mla_fwd_lean16_kernel;
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
    const int64_t blocks = (int64_t)a.T * a.S;
    if (blocks == 0)
        return cudaSuccess;
    // The cache as a 2-D tensor [rows x 512] codes, read in boxes of 128 codes
    // x 1 row with the 128-byte swizzle; rows past the int32 index range are
    // unreachable, so the row count is clamped there.
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr)
        return cudaErrorNotSupported;
    CUtensorMap kv_map;
    const int64_t rows = a.num_slots < 1 ? 1 : (a.num_slots > INT_MAX ? (int64_t)INT_MAX : a.num_slots);
    cuuint64_t gdim[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)kD};
    cuuint32_t box[2] = {128, 1};
    cuuint32_t estride[2] = {1, 1};
    if (encode(&kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(a.kv), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.S > 1 && a.S <= kClusterMaxSplits) {
        // the S splits of a (row, head group) are consecutive blocks: one cluster
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)a.S;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, kern, a, kv_map);
}

cudaError_t read_lean_error(int *out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_lean_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_lean_error, &zero, sizeof(int));
    }
    return e;
}

} // namespace smla
