// Sparse MLA forward for 16 heads on the 5th-generation tensor cores
// (tcgen05 + tensor memory) with TMA row gathers, sm_103a. Two variants: a
// bf16 cache, and an E4M3 cache with a per-tensor scale and fp8 QK dots.
//
// One CTA = (query row t, split s of its top-k list). With only 16 heads per
// row the contraction is computed transposed, keys on the MMA's M axis:
//   S^T [64 keys x 16 heads] = KV_tile [64 x 512] . q^T          (QK, M=64, N=16)
//   O^T [512 dims x 16 heads] += V^T [512 x 64 keys] . P^T       (PV, 4 x M=128, N=16)
// Both accumulators live in tensor memory (O^T in 64 columns; S^T double-
// buffered, each buffer as two partial sums over halves of the 512
// columns).
//
// The tile is gathered by the TMA engine: a 2-D tensor map over the cache
// ([num_slots rows x 512] elements, boxes of 128 bytes x 1 row, 128-byte
// swizzle) and tile::gather4 copies, each moving a 128-byte column block of
// 4 named rows. A 64-key tile is 16 key quads x (8 bf16 | 4 E4M3) column
// blocks, landing as blocks of [64 keys x 128 B] in exactly the swizzled
// layout the MMA reads. Masked (-1) and out-of-range indices are passed as
// row -1, which the TMA fills with zeros without reading memory. A tile's
// copies are issued from four warps: the TMA engine accepts copies from
// several warps in parallel, and one warp alone cannot issue random rows
// fast enough to keep up with HBM.
//
// bf16 cache: the tile is the K-major A operand of QK and, read MN-major,
// V^T of PV.
// E4M3 cache: q is quantized in the kernel per (row, head), s_q =
// amax|q[t,h,:]| / 448 (1 if zero), q8 = RNE_satfinite(q / s_q); QK runs in
// E4M3 (kind::f8f6f4) on the gathered tile and the logits are scaled by
// scale * s_q * kv_scale. PV needs 16-bit operands of one type, so four
// converter warps turn each tile's values into binary16 (exact) and write
// V^T straight into tensor memory (three buffers), where PV reads its A
// operand; P is kept in fp16 and kv_scale is applied with 1/l. Keeping V^T
// out of shared memory matters: a binary16 copy there costs 128 KB of
// shared-memory traffic per 32 KB tile, more than the rest of the tile.
//
// Warp roles, handing tiles over through mbarriers:
//   producers (warps 5-12 for a bf16 cache, 5-8 for E4M3): q into shared
//     memory once (quantized for E4M3); then the rows of each tile. bf16
//     rows are copied by 16-byte cp.async: each of the 256 producer threads
//     issues 16 per tile (a warp instruction reads 512 contiguous bytes of a
//     row) straight into the 128-byte swizzled layout, and the stage's
//     "full" barrier counts every producer thread once its copies have
//     landed; the MMA issuers fence the generic proxy's writes before their
//     MMAs read the stage. E4M3 rows come by TMA gather4, one per thread,
//     completing "full" by transaction bytes. A stage is refilled once
//     everything that reads it is done ("empty"). The TMA gathers of bf16
//     rows were slower both from DRAM (decode 34.6 against 32.6 us) and from
//     L2 (prefill 2.44 against 2.24 ms): a warp issues its lanes' gather
//     copies one after another. For a pool that fits in L2 the CTA first
//     finds its split's last valid index and runs only the tiles up to it
//     (a row shorter than top-k is padded at its end: prefill 2.01 ms).
//   MMA issuers (one thread each in warps 4, 13, 14 and 15 for bf16): QK(i)
//     as soon as tile i has landed (and the softmax is done with the S
//     buffer), in two halves for bf16; PV(i) as soon as the softmax has
//     written P(i), two threads each taking half of the value dims. A single
//     thread issues small MMAs at about one per 26 ns; threads issue in
//     parallel, so splitting a tile's MMAs across issuers shortens the time
//     each stage is held and the chain of the last tile. Commits signal the
//     softmax (S full), the producers (stage empty) and the P buffers.
//   converters (E4M3 only, warps 11-14, one per quarter of the TMEM lanes):
//     tile i -> V^T in tensor memory buffer i%3 once PV(i-3) has read it
//     (three buffers: the conversion of a tile overlaps the PV of the two
//     before it, so neither waits on the other in steady state);
//     lane d of M-block b holds dim 128b + d, two keys per column. Each
//     thread loads 4-byte words (4 dims of one key), transposes 4x4 bytes
//     within its lane quad by two shuffles, converts, and stores 32 columns.
//   softmax (warps 0-3, one key per thread of lanes 0-15): reads the key's 16
//     logits (two partial sums) from TMEM, masks, and exponentiates against a
//     running reference max; the max is recomputed over the tile (and O^T
//     rescaled in TMEM) only when some logit exceeds the reference by more
//     than 2^8, and the reference then moves to 2^8 above the tile max (p
//     stays <= 1; O/l does not depend on the reference), so the common tile
//     needs no cross-thread reduction beyond one flag exchange; writes one
//     row of P^T. The reference max per head, the same in every softmax
//     thread, lives in shared memory (two buffers: thread 0 writes the new
//     one while the others read the old), not in 16 registers a thread.
// Every barrier completes once per use of the resource it guards, so no
// waiter can fall two phases behind; every wait gives up after about 2 s
// (the call then records an error, stops issuing, waits with a bound for the
// copies and MMAs already issued, and finishes).
//
// Method sources (page titles and sections):
//   "Enable AITER sparse MLA on gfx942, including FP8 KV" — Overview, Details
//     ("FP8 KV on gfx942": the kernel quantizes q per tile, dots in fp8).
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
#include <mutex>

namespace smla {

__device__ int g_umma_error = 0; // set when a bounded wait gives up

namespace {

constexpr int kSoftmaxWarps = 4;
constexpr int kMmaWarp = 4;       // QK, first half of the columns
constexpr int kProducerWarp0 = 5; // 4 producer warps (8 for a bf16 pool held in L2), then more MMA issuers
constexpr int kConverterThreads = 128;
// tensor memory columns: O^T 0..63, S^T partial p of buffer b at kSCol + 32 p + 16 b
constexpr int kSCol = 64;
constexpr int kKeys = kUmma16TileKeys; // keys per tile (M of QK)
constexpr int kHeads = 16;
constexpr int kD = 512;                // D_qk = D_v
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f; // log2 units a logit may exceed the reference by
constexpr float kHeadroom = 8.0f;         // a moved reference sits this far above the tile max
constexpr int kIdxAhead = 4;              // tiles of index look-ahead

// The three variants: a bf16 cache; an E4M3 cache with fp8 dots; an E4M3
// cache with bf16 dots (q . code * kv_scale with q unquantized), run as the
// bf16 variant on binary16 operands that converter warps expand exactly from
// the gathered E4M3 tile.
// A fourth: a bf16 cache whose pool fits in L2 (e.g. prefill over one
// sequence's keys), where the gathers come from L2 and eight producer warps
// issue them faster than four; from DRAM eight are slower than four.
// bf16 cache rows are copied by cp.async (kBf16Async); E4M3 rows by TMA gathers
enum Mode : int { kFp8 = 1, kBf16Dots = 2, kBf16Async = 4 };

template <int MODE>
struct Cfg {
    static constexpr bool FP8 = MODE == kFp8;
    static constexpr bool BD = MODE == kBf16Dots;
    static constexpr bool G8 = FP8 || BD;         // the gathered cache rows are E4M3
    static constexpr int EB = G8 ? 1 : 2;         // bytes per cache element
    static constexpr int ROW = kD * EB;           // bytes per cache row
    static constexpr int NCB = ROW / 128;         // 128-byte column blocks per row (8 | 4)
    static constexpr int BOXW = 128 / EB;         // elements per gather box
    static constexpr int BLK = kKeys * 128;       // one column block of a tile (8 KB)
    static constexpr int TILE = NCB * BLK;        // 64 keys (64 KB | 32 KB)
    static constexpr int COPIES = 16 * NCB;       // gather4 copies per tile (128 | 64)
    // bf16 rows are copied by 16-byte cp.async from eight producer warps
    static constexpr bool ASYNC = MODE == kBf16Async;
    static constexpr int PWARPS = ASYNC ? 8 : 4; // producer warps
    static constexpr int PTHREADS = 32 * PWARPS;
    static constexpr int COPY_LANES = COPIES / PWARPS;          // copies a producer warp issues per tile
    static constexpr int MMA_WARP2 = kProducerWarp0 + PWARPS;   // further MMA issuers from here
    static constexpr int STAGES = FP8 ? 5 : (BD ? 2 : 3);
    // bf16 dots: binary16 stages [64 keys x 512] in the layout of the bf16
    // variant's tile, each written by the converters and read by QK and PV
    static constexpr int FSTAGES = BD ? 2 : 0;
    static constexpr int FTILE = 8 * BLK;         // 64 KB
    static constexpr int OFF_FRING = STAGES * TILE;
    static constexpr int KSTEP = FP8 ? 32 : 16;   // reduction depth of one QK MMA
    static constexpr int QK_MMAS = kD / KSTEP;    // per tile (32 | 16)
    static constexpr int QK_ISSUERS = FP8 ? 1 : 2; // threads issuing QK (S partial sums)
    static constexpr int PV_ISSUERS = 2;           // threads issuing PV (halves of the 512 dims)
    // E4M3 / bf16 dots: bf16 q staged for the quantizer (16 KB); with bf16 dots
    // inside the second binary16 stage, which is first written after q is done
    static constexpr int OFF_QSTG = BD ? OFF_FRING + FTILE : OFF_FRING;
    static constexpr int OFF_Q = OFF_FRING + FSTAGES * FTILE + (FP8 ? kHeads * kD * 2 : 0); // q in core matrices
    static constexpr int QROW = kD * (FP8 ? 1 : 2); // bytes of one head's q
    static constexpr int QGRP = 8 * QROW;         // q: 8 heads x 512 elements
    static constexpr int OFF_P = OFF_Q + 2 * QGRP;// P^T [64 keys x 16 heads] 16-bit, 2 buffers x 2 KB
    static constexpr int OFF_SQ = OFF_P + 2 * 2048; // [16] per-head q scales (E4M3, bf16 dots)
    static constexpr int OFF_FAC = OFF_SQ + 16 * 4; // [16] per-head logit factors
    static constexpr int OFF_EX = OFF_FAC + 16 * 4; // [2][4] exceed flags
    static constexpr int OFF_GO = OFF_EX + 32;    // [2] producer issue decisions
    static constexpr int OFF_WMAX = OFF_GO + 8;
    static constexpr int OFF_LRED = OFF_WMAX + 4 * 16 * 4;
    static constexpr int OFF_LSE = OFF_LRED + 4 * 16 * 4;
    static constexpr int OFF_ALPHA = OFF_LSE + 16 * 4;
    static constexpr int OFF_MISC = OFF_ALPHA + 16 * 4; // flag, tmem address, abort
    static constexpr int OFF_MREF = OFF_MISC + 16;  // [2][16] reference max per head (double-buffered)
    static constexpr int OFF_MBAR = (OFF_MREF + 128 + 7) & ~7;
    // full[S], empty[S], s_full[2] (a commit per QK issuer), p_full[2], p_empty[2] (a
    // commit per PV issuer), q_full, drain (a commit per MMA issuer), v_full[3] (E4M3:
    // V^T buffer written), v_free[3] (E4M3: a commit per PV issuer, V^T buffer read),
    // f_full[2] (bf16 dots: binary16 stage written), f_free[2] (a commit per PV issuer)
    static constexpr int VBUFS = 3;
    static constexpr int NBAR = 2 * STAGES + 8 + 2 * VBUFS + 2 * 2;
    // tensor memory: O^T 0..63, S^T 64..127; E4M3: V^T buffers at 128 + 128 v
    static constexpr int TMEM_COLS = FP8 ? 512 : 128;
    static constexpr int VCOL = 128;
    static_assert(!FP8 || VCOL + VBUFS * 128 <= TMEM_COLS, "the V^T buffers fit in tensor memory");
    static constexpr int SMEM = OFF_MBAR + NBAR * 8;
    static constexpr int SMEM_ALLOC = SMEM + 1024; // the base is aligned up to 1 KB in the kernel
    // MMA issuers in warps 4 and MMA_WARP2.. (bf16, bf16 dots: 2 QK + 2 PV; E4M3: 1 + 2)
    static constexpr int MMA_WARPS2 = QK_ISSUERS + PV_ISSUERS - 1;
    static constexpr int CONVERTER_WARP0 = MMA_WARP2 + MMA_WARPS2; // E4M3, bf16 dots
    static constexpr int THREADS = 32 * (G8 ? CONVERTER_WARP0 + 4 : MMA_WARP2 + MMA_WARPS2);
    // 15 or 16 warps share the register file, so at most 128 registers a thread
    static constexpr int BOUND_THREADS = G8 ? 512 : THREADS;
    static_assert(THREADS <= 512 && COPY_LANES <= 32 && COPIES % PWARPS == 0, "the warp layout fits");
    // stage "empty" arrivals: the PV commits (bf16), the QK commits and every
    // converter thread (E4M3: PV reads V^T from tensor memory, not the stage),
    // every converter thread (bf16 dots: QK and PV read the binary16 stage)
    static constexpr int EMPTY_COUNT = FP8 ? QK_ISSUERS + kConverterThreads : (BD ? kConverterThreads : PV_ISSUERS);
    static_assert(STAGES * TILE >= kHeads * kD * 4, "epilogue staging fits in the ring");
    static_assert(2 * QGRP >= 128 * kHeads * 4, "merge weights fit in the q area");
    static_assert(COPIES <= PTHREADS, "one copy per producer thread at most");
    static_assert(!BD || OFF_QSTG + kHeads * kD * 2 <= OFF_FRING + FSTAGES * FTILE, "q staging fits in a stage");
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// QK: A = KV tile (K-major, 128-byte swizzle), B = q (K-major), M = 64 keys, N = 16 heads
constexpr uint32_t kIdescQKbf16 = umma::idesc(64, 16, 1, 1, 0, 0);
constexpr uint32_t kIdescQKe4m3 = umma::idesc(64, 16, 0, 0, 0, 0);
// PV: A = V^T (MN-major), B = P^T (MN-major), M = 128 dims, N = 16; bf16 or fp16
constexpr uint32_t kIdescPVbf16 = umma::idesc(128, 16, 1, 1, 1, 1);
// bf16 dots: the same two contractions on binary16 operands
constexpr uint32_t kIdescQKf16 = umma::idesc(64, 16, 0, 0, 0, 0);
constexpr uint32_t kIdescPVf16 = umma::idesc(128, 16, 0, 0, 1, 1);
// E4M3: A = V^T in tensor memory (binary16), B = P^T fp16 (MN-major)
constexpr uint32_t kIdescPVf16ts = umma::idesc(128, 16, 0, 0, 0, 1);

template <int MODE>
__global__ void __launch_bounds__(Cfg<MODE>::BOUND_THREADS, 1)
    sparse_mla_fwd_umma16_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap kv_map)
{
    using C = Cfg<MODE>;
    constexpr bool FP8 = C::FP8, BD = C::BD, G8 = C::G8;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u; // swizzle atoms need 1 KB alignment
    uint8_t *smem = smem_raw + (sbase - raw_base);
    const uint32_t ring = sbase, q_s = sbase + C::OFF_Q, p_s = sbase + C::OFF_P;
    float *sq_s = reinterpret_cast<float *>(smem + C::OFF_SQ);
    float *fac_s = reinterpret_cast<float *>(smem + C::OFF_FAC);
    int *ex_s = reinterpret_cast<int *>(smem + C::OFF_EX);
    volatile int *go_s = reinterpret_cast<volatile int *>(smem + C::OFF_GO);
    float *wmax_s = reinterpret_cast<float *>(smem + C::OFF_WMAX);
    float *lred_s = reinterpret_cast<float *>(smem + C::OFF_LRED);
    float *lse_s = reinterpret_cast<float *>(smem + C::OFF_LSE);
    float *alpha_s = reinterpret_cast<float *>(smem + C::OFF_ALPHA);
    int *flag_s = reinterpret_cast<int *>(smem + C::OFF_MISC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC + 4);
    int *abort_s = reinterpret_cast<int *>(smem + C::OFF_MISC + 8);
    int *last_s = reinterpret_cast<int *>(smem + C::OFF_MISC + 12); // the split's last valid position
    const uint32_t bar0 = sbase + C::OFF_MBAR;
    constexpr int S_ = C::STAGES;
    auto full = [&](int st) { return bar0 + 8 * st; };
    auto empty = [&](int st) { return bar0 + 8 * (S_ + st); };
    auto s_full = [&](int b) { return bar0 + 8 * (2 * S_ + b); };
    auto p_full = [&](int b) { return bar0 + 8 * (2 * S_ + 2 + b); };
    auto p_empty = [&](int b) { return bar0 + 8 * (2 * S_ + 4 + b); };
    const uint32_t q_full = bar0 + 8 * (2 * S_ + 6);
    const uint32_t drain = bar0 + 8 * (2 * S_ + 7);
    auto v_full = [&](int vb) { return bar0 + 8 * (2 * S_ + 8 + vb); };
    auto v_free = [&](int vb) { return bar0 + 8 * (2 * S_ + 8 + C::VBUFS + vb); };
    auto f_full = [&](int fs) { return bar0 + 8 * (2 * S_ + 8 + 2 * C::VBUFS + fs); };
    auto f_free = [&](int fs) { return bar0 + 8 * (2 * S_ + 8 + 2 * C::VBUFS + 2 + fs); };
    const uint32_t fring = sbase + C::OFF_FRING;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x % a.S;
    const int t = blockIdx.x / a.S;
    const int kb = s * a.keys_per_split;
    const int ke = min(a.topk, kb + a.keys_per_split);
    int ntiles = ke > kb ? (ke - kb + kKeys - 1) / kKeys : 0; // (a pool in L2: trimmed below)
    const int32_t *__restrict__ row_idx = a.indices + (int64_t)t * a.topk;

    if (tid == 0) {
        for (int st = 0; st < S_; ++st) {
            // TMA: one arrival with the tile's bytes; cp.async: every producer thread
            umma::mbar_init(full(st), C::ASYNC ? C::PTHREADS : 1);
            umma::mbar_init(empty(st), C::EMPTY_COUNT);
        }
        for (int b = 0; b < 2; ++b) {
            umma::mbar_init(s_full(b), C::QK_ISSUERS);
            umma::mbar_init(p_full(b), kSoftmaxWarps * 32);
            umma::mbar_init(p_empty(b), C::PV_ISSUERS);
        }
        umma::mbar_init(q_full, C::PTHREADS);
        umma::mbar_init(drain, C::QK_ISSUERS + C::PV_ISSUERS);
        for (int vb = 0; vb < C::VBUFS; ++vb) {
            umma::mbar_init(v_full(vb), kConverterThreads);
            umma::mbar_init(v_free(vb), C::PV_ISSUERS);
        }
        for (int fs = 0; fs < 2; ++fs) {
            umma::mbar_init(f_full(fs), kConverterThreads);
            umma::mbar_init(f_free(fs), C::PV_ISSUERS);
        }
        umma::mbar_init_fence();
        *abort_s = 0;
        *last_s = -1;
    }
    if (warp == 0)
        umma::alloc(smem_u32(tmem_slot), C::TMEM_COLS);
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
    if (C::ASYNC && a.trim_tail) {
        // tiles after the split's last valid index hold only masked keys (a row
        // shorter than top-k is padded at its end): find that index (one load
        // per thread and round from L2) and run only the tiles up to it
        int last = -1;
        for (int p = kb + tid; p < ke; p += C::THREADS) {
            const int x = __ldg(row_idx + p);
            if (x >= 0 && (int64_t)x < a.num_slots)
                last = p;
        }
        last = __reduce_max_sync(0xffffffffu, last);
        if (lane == 0 && last >= 0)
            atomicMax(last_s, last);
        __syncthreads();
        const int lv = *(volatile int *)last_s;
        ntiles = lv < kb ? 0 : (lv - kb) / kKeys + 1;
    }

    auto wait_bar = [&](uint32_t mbar, uint32_t parity) {
        if (*(volatile int *)abort_s)
            return;
        if (!umma::mbar_wait(mbar, parity)) {
            atomicOr(&g_umma_error, 1);
            *(volatile int *)abort_s = 1;
        }
    };
    // a wait that runs even after an abort (for work already issued), still bounded
    auto wait_issued = [&](uint32_t mbar, uint32_t parity) {
        if (!umma::mbar_wait(mbar, parity))
            atomicOr(&g_umma_error, 2);
    };

    if (warp >= kProducerWarp0 && warp < kProducerWarp0 + C::PWARPS) {
        // ======================= producers =======================
        const int pt = tid - kProducerWarp0 * 32;
        const __nv_bfloat16 *__restrict__ qg =
            static_cast<const __nv_bfloat16 *>(a.q) + (int64_t)t * kHeads * kD;
        // this thread's copy (the first COPY_LANES lanes of each producer warp:
        // all 32 for bf16 rows from four warps, 16 otherwise): key quad qd (keys
        // 4qd..4qd+3), column block cb
        const int cid = (pt >> 5) * C::COPY_LANES + (pt & 31);
        const bool copier = (pt & 31) < C::COPY_LANES;
        const int qd = cid / C::NCB, cb = cid % C::NCB;
        // raw indices only: checking them here would wait for the loads
        auto fetch = [&](int tile, int (&r)[4]) {
            if constexpr (C::ASYNC) {
                // cp.async: lane k < 8 of producer warp pw holds the index of key 8 pw + k
                const int p = kb + tile * kKeys + 8 * (pt >> 5) + (pt & 7);
                r[0] = ((pt & 31) < 8 && tile < ntiles && p < ke) ? __ldg(row_idx + p) : -1;
                r[1] = r[2] = r[3] = -1;
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int p = kb + tile * kKeys + 4 * qd + u;
                    r[u] = (copier && tile < ntiles && p < ke) ? __ldg(row_idx + p) : -1;
                }
            }
        };
        auto row = [&](int x) { return (x >= 0 && (int64_t)x < a.num_slots) ? x : -1; };
        // Indices are loaded kIdxAhead tiles before their copies are issued
        // (a load from HBM under full load takes longer than a tile), in
        // register slots fixed at compile time by unrolling over the slots.
        int r0[4], r1[4], r2[4], r3[4];
        static_assert(kIdxAhead == 4, "one register slot per tile of look-ahead");
        fetch(0, r0);
        fetch(1, r1);
        fetch(2, r2);
        fetch(3, r3);
        // q [16 x 512] -> core matrices (8 heads x 16 B): LBO 128 (K), SBO = 8 heads;
        // published once the first tile's copies are in flight, so both latencies overlap
        auto issue_q = [&] {
            if constexpr (!G8) {
                for (int e = pt; e < kHeads * 64; e += C::PTHREADS) {
                    const int h = e >> 6, c = e & 63;
                    cp_async_16(q_s + (h >> 3) * C::QGRP + c * 128 + (h & 7) * 16, qg + h * kD + c * 8, 16);
                }
            } else if (FP8 && a.q_fp8_in) {
                // pre-quantized q: each head's 512 codes straight into core matrices
                // (a core-matrix row holds 16 codes)
                const uint8_t *q8g = static_cast<const uint8_t *>(a.q) + (int64_t)t * kHeads * kD;
                for (int e = pt; e < kHeads * (kD / 16); e += C::PTHREADS) {
                    const int h = e / (kD / 16), c = e % (kD / 16);
                    cp_async_16(q_s + (h >> 3) * C::QGRP + c * 128 + (h & 7) * 16, q8g + h * kD + c * 16, 16);
                }
            } else {
                // bf16 q staged row-major: this thread's 64 elements of head pt/8,
                // the ones it quantizes (E4M3) or rescales to binary16 (bf16 dots)
                const int h = pt >> 3, e0 = h * kD + (pt & 7) * 64;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    cp_async_16(sbase + C::OFF_QSTG + (e0 + 8 * u) * 2, qg + e0 + 8 * u, 16);
            }
            cp_async_commit();
        };
        issue_q();
        bool q_pending = true;
        auto publish_q = [&] {
            cp_async_wait<0>();
            if (FP8 && a.q_fp8_in) {
                if (pt < kHeads) // one per-tensor scale for every head
                    sq_s[pt] = *a.q_scale_in;
            } else if constexpr (FP8) {
                // thread pt quantizes the 64 elements of head pt/8 it staged
                const int h = pt >> 3;
                uint4 qraw[8];
                const uint4 *src = reinterpret_cast<const uint4 *>(smem + C::OFF_QSTG + (h * kD + (pt & 7) * 64) * 2);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    qraw[u] = src[u];
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
                for (int o = 1; o < 8; o <<= 1) // the 8 threads of a head are adjacent lanes
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                const float sq = (m == 0.f) ? 1.0f : __fdiv_rn(m, 448.0f);
                if ((pt & 7) == 0)
                    sq_s[h] = sq;
                // 64 codes = 4 core-matrix rows of 16 B
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t w[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&qraw[2 * cc + v / 2]);
                        const float2 f0 = __bfloat1622float2(b2[2 * (v & 1)]);
                        const float2 f1 = __bfloat1622float2(b2[2 * (v & 1) + 1]);
                        w[v] = quant4_e4m3(f0.x, f0.y, f1.x, f1.y, sq);
                    }
                    const int c = (pt & 7) * 4 + cc; // 16-byte column of the head's row
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(q_s + (h >> 3) * C::QGRP + c * 128 +
                                                                                 (h & 7) * 16),
                                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
            }
            if constexpr (BD) {
                // thread pt rescales the 64 elements of head pt/8 by 2^e, e chosen so
                // that the head's amax lands in [2^14, 2^15): every bf16 value of q
                // at least 2^-29 of the amax is exactly a binary16 normal (the
                // smaller ones, worth less than 2^-29 of the largest term, round as
                // binary16 subnormals), and 2^-e goes into the logits' factor
                const int h = pt >> 3;
                uint4 qraw[8];
                const uint4 *src = reinterpret_cast<const uint4 *>(smem + C::OFF_QSTG + (h * kD + (pt & 7) * 64) * 2);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    qraw[u] = src[u];
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
                for (int o = 1; o < 8; o <<= 1) // the 8 threads of a head are adjacent lanes
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                // the amax's binary exponent from its bits (q is finite); a zero head keeps 2^0
                const int ex = m > 0.f ? (int)((__float_as_uint(m) >> 23) & 0xff) - 127 : 14;
                const int e = max(-126, min(126, 14 - ex));
                const float up = __uint_as_float((uint32_t)(127 + e) << 23), down = __uint_as_float((uint32_t)(127 - e) << 23);
                if ((pt & 7) == 0)
                    sq_s[h] = down;
                // 64 binary16 values = 8 core-matrix rows of 16 B
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&qraw[u]);
                    uint32_t w[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const float2 f = __bfloat1622float2(b2[v]);
                        w[v] = pack_f16x2(f.x * up, f.y * up);
                    }
                    const int c = (pt & 7) * 8 + u; // 16-byte column of the head's row
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(q_s + (h >> 3) * C::QGRP + c * 128 +
                                                                                 (h & 7) * 16),
                                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
            }
            umma::fence_async_smem();
            umma::mbar_arrive(q_full);
            q_pending = false;
        };
        int issued = 0;
        bool stop = false;
        auto step = [&](int j, int(&r)[4]) {
            if (stop || j >= ntiles) {
                stop = true;
                return;
            }
            const int st = j % S_;
            if (pt == 0) {
                if (j >= S_)
                    wait_bar(empty(st), (uint32_t)((j / S_ - 1) & 1));
                const int go = !*(volatile int *)abort_s;
                if (go && !C::ASYNC)
                    umma::mbar_arrive_expect_tx(full(st), C::TILE);
                go_s[j & 1] = go;
            }
            // all or none of a tile's copies are issued, so a stage's barrier
            // always completes once its copies are in flight
            umma::named_bar(2, C::PTHREADS);
            if (!go_s[j & 1]) {
                stop = true;
                return;
            }
            if constexpr (C::ASYNC) {
                // producer warp pw copies keys 8 pw .. 8 pw + 7: per key two rounds of
                // 32 lanes x 16 bytes (512 contiguous bytes of the row each), into the
                // 128-byte swizzled layout the TMA would write (16-byte chunk c of the
                // row: column block c / 8, chunk (c % 8) ^ (key % 8)); a masked key's
                // chunks are zero-filled without a read. The stage's barrier counts
                // each thread once its copies have landed.
                const uint8_t *kvb = static_cast<const uint8_t *>(a.kv);
                const int l = pt & 31;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int x = row(__shfl_sync(0xffffffffu, r[0], k));
                    const int key = 8 * (pt >> 5) + k;
                    const uint8_t *src = kvb + (int64_t)(x < 0 ? 0 : x) * C::ROW;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int c = 32 * i + l;
                        cp_async_16(ring + st * C::TILE + (c >> 3) * C::BLK + key * 128 + (((c & 7) ^ (key & 7)) << 4),
                                    src + c * 16, x < 0 ? 0u : 16u);
                    }
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(full(st)) : "memory");
            } else if (copier) {
                umma::tma_gather4(ring + st * C::TILE + cb * C::BLK + qd * 512, &kv_map, C::BOXW * cb, row(r[0]),
                                  row(r[1]), row(r[2]), row(r[3]), full(st));
            }
            issued = j + 1;
            fetch(j + kIdxAhead, r);
            if (q_pending)
                publish_q();
        };
        for (int j0 = 0; !stop; j0 += kIdxAhead) {
            step(j0, r0);
            step(j0 + 1, r1);
            step(j0 + 2, r2);
            step(j0 + 3, r3);
        }
        if (q_pending)
            publish_q();
        // every copy issued has landed before the CTA can finish (also after an abort)
        if (pt == 0) {
            for (int j = max(0, issued - S_); j < issued; ++j)
                wait_issued(full(j % S_), (uint32_t)((j / S_) & 1));
        }
    } else if (warp == kMmaWarp || (warp >= C::MMA_WARP2 && warp < C::MMA_WARP2 + C::MMA_WARPS2)) {
        // ======================= MMA issuers =======================
        if (lane == 0) {
            // roles 0 .. QK_ISSUERS-1: parts of QK; the next PV_ISSUERS: PV over
            // halves of the value dims (M-blocks 2 v, 2 v + 1 for PV issuer v)
            const int role = warp == kMmaWarp ? 0 : 1 + warp - C::MMA_WARP2;
            const bool is_pv = role >= C::QK_ISSUERS;
            if (role < C::QK_ISSUERS) {
                wait_bar(q_full, 0);
                const uint64_t qdesc = umma::desc(q_s, 128, C::QGRP);
                constexpr int kHalf = C::QK_MMAS / C::QK_ISSUERS;
                const int ks0 = kHalf * role;
                for (int i = 0; i < ntiles; ++i) {
                    const int b = i & 1, st = i % S_, fs = i & 1;
                    if constexpr (BD) // the binary16 stage holds tile i
                        wait_bar(f_full(fs), (uint32_t)((i >> 1) & 1));
                    else
                        wait_bar(full(st), (uint32_t)((i / S_) & 1));
                    if (i >= 2) // the softmax has read S buffer b for tile i-2
                        wait_bar(p_full(b), (uint32_t)(((i - 2) >> 1) & 1));
                    if (*(volatile int *)abort_s)
                        break;
                    umma::fence_after_sync();
                    if constexpr (C::ASYNC) // the stage was written by cp.async (generic proxy)
                        umma::fence_async_smem();
                    // KV tile: K-major, 8-key atoms 1 KB apart; k-step ks reads column
                    // block ks/4, starting 32 B * (ks%4) into its 128-byte rows
                    const uint64_t ad = umma::desc_sw128(BD ? fring + fs * C::FTILE : ring + st * C::TILE, 16, 1024);
#pragma unroll
                    for (int ks = ks0; ks < ks0 + kHalf; ++ks) {
                        const uint64_t ak = ad + (uint64_t)(((ks >> 2) * C::BLK + (ks & 3) * 32) >> 4);
                        const uint64_t bk = qdesc + (uint64_t)(ks * 16); // 2 core matrices of q per k-step
                        if constexpr (FP8)
                            umma::mma_f8(tmem + kSCol + 32 * role + 16 * b, ak, bk, kIdescQKe4m3, ks > ks0);
                        else
                            umma::mma_f16(tmem + kSCol + 32 * role + 16 * b, ak, bk, BD ? kIdescQKf16 : kIdescQKbf16,
                                          ks > ks0);
                    }
                    umma::commit(s_full(b));
                    if constexpr (FP8)
                        umma::commit(empty(st)); // this half of QK(i) no longer reads the stage
                }
            } else if (is_pv) {
                const int blk0 = 2 * (role - C::QK_ISSUERS), blk1 = blk0 + 2;
                for (int i = 0; i < ntiles; ++i) {
                    const int b = i & 1, st = i % S_;
                    wait_bar(p_full(b), (uint32_t)((i >> 1) & 1));
                    const int vb = i % C::VBUFS;
                    if constexpr (FP8) // V^T buffer vb holds tile i
                        wait_bar(v_full(vb), (uint32_t)((i / C::VBUFS) & 1));
                    if (*(volatile int *)abort_s)
                        break;
                    umma::fence_after_sync();
                    if constexpr (C::ASYNC)
                        umma::fence_async_smem();
                    const uint64_t bd = umma::desc(p_s + b * 2048, 256, 128);
                    if constexpr (FP8) {
                        // V^T in tensor memory: M-block blk at +32 blk, 16 keys = 8 columns
                        const uint32_t va = tmem + C::VCOL + 128 * vb;
                        for (int blk = blk0; blk < blk1; ++blk)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                umma::mma_f16_ts(tmem + 16 * blk, va + 32 * blk + 8 * kk, bd + (uint64_t)(kk * 32),
                                                 kIdescPVf16ts, (i > 0 || kk > 0) ? 1u : 0u);
                    } else {
                        // V^T: MN-major, 64-column atoms 8 KB apart (LBO), 8-key atoms 1 KB apart (SBO)
                        const uint64_t ad =
                            umma::desc_sw128(BD ? fring + (i & 1) * C::FTILE : ring + st * C::TILE, C::BLK, 1024);
                        for (int blk = blk0; blk < blk1; ++blk)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                umma::mma_f16(tmem + 16 * blk, ad + (uint64_t)((blk * 2 * C::BLK + kk * 2048) >> 4),
                                              bd + (uint64_t)(kk * 32), BD ? kIdescPVf16 : kIdescPVbf16,
                                              (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    // PV(i) follows the softmax's read of S(i), so QK(i) is complete too.
                    // p_empty(b) also tells the softmax (and the converters) that O^T holds
                    // PV(0..i): each issuer's commit covers all its earlier MMAs.
                    if constexpr (FP8)
                        umma::commit(v_free(vb));
                    else if constexpr (BD)
                        umma::commit(f_free(i & 1)); // this half of PV(i) no longer reads the binary16 stage
                    else
                        umma::commit(empty(st)); // this half of PV(i) no longer reads the stage
                    umma::commit(p_empty(b));
                }
            }
            // every MMA issued has completed before TMEM is released
            if (role < C::QK_ISSUERS || is_pv) {
                umma::commit(drain);
                wait_issued(drain, 0);
            }
        }
        __syncwarp();
    } else if (G8 && warp >= C::CONVERTER_WARP0) {
        // ======================= converters (E4M3) =======================
        if constexpr (BD) {
            // tile i (E4M3, 4 swizzled column blocks) -> binary16 stage i%2 (8
            // swizzled column blocks, the bf16 variant's layout), once PV(i-2) has
            // read that stage. Item w of 2048: key r = w % 64 (a warp's lanes take
            // consecutive keys, so each 16-byte access spreads over all banks),
            // E4M3 16-byte chunk c = w / 64 of the row, i.e. codes 16c..16c+15,
            // which become binary16 chunks 2(c%4), 2(c%4)+1 of column block c/4*...
            const int ct = tid - C::CONVERTER_WARP0 * 32;
            wait_bar(q_full, 0); // the q staging (inside binary16 stage 1) has been read
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % S_, fs = i & 1;
                wait_bar(full(st), (uint32_t)((i / S_) & 1));
                if (i >= 2) // PV(i-2) has read binary16 stage fs
                    wait_bar(f_free(fs), (uint32_t)(((i >> 1) - 1) & 1));
                const uint32_t src0 = ring + st * C::TILE, dst0 = fring + fs * C::FTILE;
#pragma unroll 4
                for (int w = ct; w < kKeys * 32; w += kConverterThreads) {
                    const int r = w & (kKeys - 1), c = w >> 6; // c = 8 cb + c16
                    const int cb = c >> 3, c16 = c & 7;
                    uint4 v;
                    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                 : "r"(src0 + cb * C::BLK + r * 128 + ((c16 ^ (r & 7)) << 4)));
                    uint32_t h[8];
                    e4m3x4_to_f16x4(v.x, h[0], h[1]);
                    e4m3x4_to_f16x4(v.y, h[2], h[3]);
                    e4m3x4_to_f16x4(v.z, h[4], h[5]);
                    e4m3x4_to_f16x4(v.w, h[6], h[7]);
                    // codes 128 cb + 16 c16 .. +15 = binary16 columns of block 2 cb + c16 / 4,
                    // 16-byte chunks 2 (c16 % 4) and 2 (c16 % 4) + 1 of its row
                    const int fb = 2 * cb + (c16 >> 2), f0 = 2 * (c16 & 3);
                    const uint32_t drow = dst0 + fb * C::BLK + r * 128;
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(drow + ((f0 ^ (r & 7)) << 4)),
                                 "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                                 : "memory");
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(drow + (((f0 + 1) ^ (r & 7)) << 4)),
                                 "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                                 : "memory");
                }
                umma::fence_async_smem(); // the MMAs read what these threads wrote
                umma::mbar_arrive(f_full(fs));
                umma::mbar_arrive(empty(st)); // done reading the E4M3 stage
            }
        } else if constexpr (FP8) {
            // lane quad (g, ii): member ii loads 4 dims (4g..4g+3 of this warp's 32)
            // of key 4kq+ii; after the transpose it holds dim 4g+ii of keys 4kq..4kq+3
            const int q4 = warp & 3, g = lane >> 2, ii = lane & 3;
            const uint32_t selA = ii < 2 ? 0x5410u : 0x3276u; // keep / take 16-bit halves (xor 2)
            const uint32_t selB = ii & 1 ? 0x3715u : 0x6240u; // interleave bytes (xor 1)
            const uint32_t tlane = (uint32_t)(32 * q4) << 16;
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % S_, vb = i % C::VBUFS;
                wait_bar(full(st), (uint32_t)((i / S_) & 1));
                if (i >= C::VBUFS) // PV(i-3) has read V^T buffer vb
                    wait_bar(v_free(vb), (uint32_t)((i / C::VBUFS - 1) & 1));
                const uint32_t src0 = ring + st * C::TILE;
#pragma unroll 1
                for (int mb = 0; mb < 4; ++mb) {
                    uint32_t col[32];
#pragma unroll
                    for (int kq = 0; kq < 16; ++kq) {
                        const int key = 4 * kq + ii;
                        const uint32_t w = lds32(src0 + mb * C::BLK + key * 128 +
                                                 (((2 * q4 + (g >> 2)) ^ (key & 7)) << 4) + (g & 3) * 4);
                        const uint32_t x = __byte_perm(w, __shfl_xor_sync(0xffffffffu, w, 2), selA);
                        const uint32_t y = __byte_perm(x, __shfl_xor_sync(0xffffffffu, x, 1), selB);
                        e4m3x4_to_f16x4(y, col[2 * kq], col[2 * kq + 1]);
                    }
                    umma::st32(tmem + tlane + C::VCOL + 128 * vb + 32 * mb, col);
                }
                umma::wait_st();
                umma::fence_before_sync();
                umma::mbar_arrive(v_full(vb));
                umma::mbar_arrive(empty(st)); // done reading the stage
            }
        }
    } else {
        // ======================= softmax =======================
        const uint32_t tm_lane = (uint32_t)(warp * 32) << 16;
        const int key = warp * 16 + lane; // meaningful for lane < 16
        // log2-domain logit factor: per head for an E4M3 cache (the q scale, or the
        // power of two that brought q into binary16; in shared memory), one for bf16
        float ovs = 1.0f; // output factor besides 1/l
        if constexpr (G8) {
            const float kvs = *a.kv_scale;
            ovs = kvs;
            wait_bar(q_full, 0); // the per-head q scales
            if (tid < 16)
                fac_s[tid] = a.scale * kLog2e * sq_s[tid] * kvs;
            umma::named_bar(1, kSoftmaxWarps * 32);
        }
        auto fac = [&](int h) { return G8 ? fac_s[h] : a.scale * kLog2e; };
        float *mref_s = reinterpret_cast<float *>(smem + C::OFF_MREF);
        int mcur = 0;
        if (tid < 16)
            mref_s[tid] = -INFINITY;
        umma::named_bar(1, kSoftmaxWarps * 32);
        float l_part[16];
#pragma unroll
        for (int h = 0; h < 16; ++h)
            l_part[h] = 0.f;
        auto load_idx = [&](int tile) {
            const int p = kb + tile * kKeys + key;
            return (lane < 16 && tile < ntiles && p < ke) ? __ldg(row_idx + p) : -1;
        };
        // the key's index, loaded kIdxAhead tiles ahead in fixed register slots
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
            if constexpr (C::QK_ISSUERS == 2) {
                float s2[16];
                umma::ld16(tmem + kSCol + 32 + 16 * b + tm_lane, reinterpret_cast<uint32_t(&)[16]>(s2));
                umma::wait_ld();
#pragma unroll
                for (int h = 0; h < 16; ++h)
                    sv[h] += s2[h];
            } else {
                umma::wait_ld();
            }
            bool exceed = false;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                sv[h] = kvalid ? sv[h] * fac(h) : -INFINITY;
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
                const float mr = mref_s[mcur * 16 + h];
                const float mu = (mr == -INFINITY) ? 0.f : mr;
                sv[h] = ex2_approx(sv[h] - mu);
                l_part[h] += sv[h];
            }
            if (i >= 2)
                wait_bar(p_empty(b), (uint32_t)(((i - 2) >> 1) & 1)); // PV(i-2) is done with this P buffer
            if (lane < 16) {
                auto pk = [&](float x, float y) { return G8 ? pack_f16x2(x, y) : pack_bf16x2(x, y); };
                const uint32_t prow = p_s + b * 2048 + (key >> 3) * 256 + (key & 7) * 16;
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow), "r"(pk(sv[0], sv[1])),
                             "r"(pk(sv[2], sv[3])), "r"(pk(sv[4], sv[5])), "r"(pk(sv[6], sv[7])));
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + 128), "r"(pk(sv[8], sv[9])),
                             "r"(pk(sv[10], sv[11])), "r"(pk(sv[12], sv[13])), "r"(pk(sv[14], sv[15])));
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
        if (tid < 16) { // thread h finishes head h (all heads at once)
            const float mh = mref_s[mcur * 16 + tid];
            const float l = lred_s[tid] + lred_s[16 + tid] + lred_s[32 + tid] + lred_s[48 + tid];
            lse_s[tid] = l > 0.f ? (mh + log2f(l)) * kLn2 : -INFINITY;
            alpha_s[tid] = l > 0.f ? ovs / l : 0.f; // reused: output factor per head
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
                const int d = (2 * half + u) * 128 + warp * 32 + lane;
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
        umma::dealloc(tmem, C::TMEM_COLS);
    finish_tile<C::THREADS>(a, reinterpret_cast<float *>(smem), lse_s, reinterpret_cast<float *>(smem + C::OFF_Q),
                            flag_s, t, 0, s, tid);
}


template <int MODE>
cudaError_t launch(const FwdArgs &a, cudaStream_t stream)
{
    using C = Cfg<MODE>;
    auto kern = sparse_mla_fwd_umma16_kernel<MODE>;
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_ALLOC);
        if (e != cudaSuccess)
            return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    const int64_t blocks = (int64_t)a.T * a.S;
    if (blocks == 0)
        return cudaSuccess;

    // The cache as a 2-D tensor [rows x 512] (row pitch 1 KB bf16 | 512 B E4M3),
    // read in boxes of 128 bytes x 1 row with the 128-byte swizzle. Rows beyond
    // the int32 index range are unreachable, so the row count is clamped there.
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr)
        return cudaErrorNotSupported;
    CUtensorMap kv_map;
    const int64_t rows = a.num_slots < 1 ? 1 : (a.num_slots > INT_MAX ? (int64_t)INT_MAX : a.num_slots);
    cuuint64_t gdim[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)C::ROW};
    cuuint32_t box[2] = {(cuuint32_t)C::BOXW, 1};
    cuuint32_t estride[2] = {1, 1};
    if (encode(&kv_map, C::G8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(a.kv), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    // programmatic dependent launch (the kernel waits for its predecessor in
    // grid_wait after a prologue that reads no global memory)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_ALLOC;
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

} // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

cudaError_t launch_fwd_umma16(const FwdArgs &a, cudaStream_t stream)
{
    if (!a.kv_fp8) {
        // bf16 rows by cp.async; a pool that fits in a quarter of L2 also skips
        // the padded tail of short rows
        static std::atomic<int> l2_bytes[64];
        int dev = 0;
        if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess)
            return e;
        int l2 = l2_bytes[dev & 63].load(std::memory_order_relaxed);
        if (l2 == 0) {
            if (const cudaError_t e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev); e != cudaSuccess)
                return e;
            l2_bytes[dev & 63].store(l2, std::memory_order_relaxed);
        }
        const bool in_l2 = a.num_slots * (int64_t)(kD * 2) * 4 <= (int64_t)l2;
        FwdArgs b = a;
        b.trim_tail = in_l2; // one more round of loads pays off only from L2
        return launch<kBf16Async>(b, stream);
    }
    return a.bf16_dots ? launch<kBf16Dots>(a, stream) : launch<kFp8>(a, stream);
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
