// Sparse MLA forward for 128 heads with an E4M3 cache (D_qk = 576: 512
// latent + 64 rope columns, D_v = 512) on the 5th-generation tensor cores
// (tcgen05 + tensor memory) with TMA row gathers, sm_103a.
//
// With 128 heads QK runs head-major and PV dims-major:
//   S   [128 heads x 64 keys]  = q8 [128 x 576] . K_tile^T          (E4M3, 18 MMAs, M=128 N=64)
//   O^T [256 dims x 128 heads] += V^T[half] [256 x 64] . P^T        (fp16, 8 MMAs, 2 x M=128 N=128)
// The fp32 output for 128 heads x 512 dims alone would fill an SM's tensor
// memory (256 KB), so each query row runs on a pair of CTAs, each owning one
// half of the value dims; both compute the full QK and softmax (identical
// inputs, identical P), and the second gather of each key row mostly hits L2.
//
// Work is spread over the pairs stream-K style: the sequence of (row, 64-key
// tile) units is cut into as many contiguous ranges as there are pairs (one
// pair per two SMs when the rows outnumber them), so no SM idles in a second
// wave. A range of at least a row's length holds whole rows and at most two
// pieces of rows it shares with a neighbouring pair: the end of its first row
// (run first) and the beginning of its last (run last). A piece of a shared
// row that finds the other piece finished merges at once, its own half
// straight from tensor memory and the other from the workspace; otherwise it
// stores a normalised partial (binary16, in units of the cache's codes) with
// its lse and marks itself finished, and whichever of the two sees the other
// finished merges (one atomic per piece, no spinning).
// At each new piece a CTA reloads that row's q8 and starts a fresh
// accumulation in tensor memory once the previous piece has been read out.
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
//   producers (warps 6-11): per 64-key tile 80 TMA tile::gather4 copies (16
//     key quads x 5 column blocks of 128 B; the last block reaches past
//     column 576 and is zero filled), 13 or 14 from each warp: the copies of
//     one warp are issued one after another, so six warps start a tile's
//     gathers well over twice as soon as two and a half would. Each warp adds
//     its own bytes to the stage's barrier. (Six, not eight: with 16 warps an
//     SM sub-partition holds four, which leaves 128 registers a thread.)
//     Masked and out-of-range indices are passed as row -1 (zero fill, no
//     memory read).
//   QK issuer (warp 4): S(i) once tile i has landed and the softmax has read
//     S(i-2).
//   softmax (warps 0-3, thread = head, whole S row in the thread): masks,
//     scales by scale * s_q[h] * kv_scale, exponentiates base 2 against a
//     running reference max that moves (all heads agree per tile, then the
//     O^T columns are rescaled in tensor memory) only when a logit exceeds
//     it by more than 2^8, and then to 2^8 above the tile max; writes its
//     row of P^T (fp16).
//   converters (warps 12-15, one per quarter of the TMEM lanes): the tile's
//     half of the value columns, E4M3 -> binary16 (exact), as V^T into
//     tensor memory (4x4 byte transposes within lane quads).
//   PV issuer (warp 5): O^T += V^T(i) . P^T(i) once both are written.
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
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f; // log2 units a logit may exceed the reference by
constexpr float kHeadroom = 8.0f;         // a moved reference sits this far above the tile max

// warps 0-3: softmax
constexpr int kQkWarp = 4;
constexpr int kPvWarp = 5;
constexpr int kProducerWarp0 = 6;     // warps 6-11
constexpr int kProducerWarps = 6;
constexpr int kCopies = 16 * kCB;     // gather4 copies per tile
constexpr int kCopiesPerWarp = (kCopies + kProducerWarps - 1) / kProducerWarps; // 14 (the last warp 10)
constexpr int kConverterWarp0 = kProducerWarp0 + kProducerWarps; // warps 12-15
constexpr int kThreads = (kConverterWarp0 + 4) * 32;
constexpr int kConverterThreads = 128;
constexpr int kIdxAhead = 4;          // tiles of index look-ahead in the producers

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
constexpr int kOffWts = kOffEx + 32;          // [2][128] merge weights of a shared row
constexpr int kOffMisc = kOffWts + 2 * kHeads * 4; // tmem address, abort, last
constexpr int kOffSeg = kOffMisc + 32;        // the CTA's work segments
constexpr int kOffMbar = kOffSeg + 64;
// full[3], empty[3], s_full[2], p_full[2], p_empty[2], v_full[2], q_full, drain, q_free, o_free
constexpr int kNBar = 18;
constexpr int kSmem = kOffMbar + kNBar * 8;
constexpr int kSmemAlloc = kSmem + 1024;
static_assert(kOffRing % 1024 == 0 && kOffPT % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kSmemAlloc <= 227 * 1024, "shared memory budget");
static_assert(kCopies * 512 == kTile && kCopiesPerWarp <= 32, "the producer warps fill a tile");

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
    // launched as a programmatic dependent of the previous kernel in the stream:
    // its blocks may be resident early, but nothing is read or written before
    // that kernel (which may produce q, or still read this workspace) completes
    umma::grid_wait();
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

// A CTA's work: up to three segments of consecutive (row, key tile) units,
// run in this order: the end of the first row of its range, the whole rows
// between (a segment may run over many rows), then the beginning of the last
// row. The neighbour that holds the other piece of a shared row runs that
// piece first, so it has usually finished by the time this CTA reaches the
// row's beginning, which then merges straight from tensor memory.
struct SegTab {
    int64_t t[3];
    int hg[3], k[3], len[3];
    int n;
};
static_assert(sizeof(SegTab) <= 64, "segment table fits its shared-memory slot");

// A walk over the segments: the current unit (row t, head group hg, key tile
// k), the units left in its segment, and whether a piece (a run of one row's
// tiles) starts here.
struct Cur {
    int64_t t;
    int hg, k, left, seg;
    bool begin;
};

__device__ __forceinline__ void cur_load(Cur &c, const SegTab &s, int i)
{
    c.seg = i;
    c.left = 0;
    if (i < s.n) {
        c.t = s.t[i];
        c.hg = s.hg[i];
        c.k = s.k[i];
        c.left = s.len[i];
        c.begin = true;
    }
}

__device__ __forceinline__ void cur_next(Cur &c, const SegTab &s, int ntiles, int G)
{
    if (--c.left > 0) {
        c.begin = false;
        if (++c.k == ntiles) {
            c.k = 0;
            c.begin = true;
            if (++c.hg == G) {
                c.hg = 0;
                ++c.t;
            }
        }
    } else {
        cur_load(c, s, c.seg + 1);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
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
    volatile int *last_s = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);
    float *wts_s = reinterpret_cast<float *>(smem + kOffWts); // [2][128] merge weights
    SegTab &sg = *reinterpret_cast<SegTab *>(smem + kOffSeg);
    const uint32_t bar0 = sbase + kOffMbar;
    auto full = [&](int st) { return bar0 + 8 * st; };
    auto empty = [&](int st) { return bar0 + 8 * (3 + st); };
    auto s_full = [&](int b) { return bar0 + 8 * (6 + b); };
    auto p_full = [&](int b) { return bar0 + 8 * (8 + b); };
    auto p_empty = [&](int b) { return bar0 + 8 * (10 + b); };
    auto v_full = [&](int b) { return bar0 + 8 * (12 + b); };
    const uint32_t q_full = bar0 + 8 * 14;
    const uint32_t drain = bar0 + 8 * 15;
    const uint32_t q_free = bar0 + 8 * 16; // the QK MMAs of a finished piece no longer read q8
    const uint32_t o_free = bar0 + 8 * 17; // a finished piece's O^T has been read out

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = a.H / kHeads;
    const int half = blockIdx.x & 1;
    const int64_t pair = blockIdx.x >> 1;
    const int ntiles = (a.topk + kKeys - 1) / kKeys;

    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            umma::mbar_init(full(st), kProducerWarps);      // each producer warp: its bytes
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
        umma::mbar_init(q_free, 1);
        umma::mbar_init(o_free, 128);
        umma::mbar_init_fence();
        *abort_s = 0;
        // this pair's range [u0, u1) of the (row, key tile) sequence and its segments
        const int64_t rows = (int64_t)a.T * G, P = a.wide_pairs;
        int64_t u0 = 0, u1 = 0;
        if (P == rows) {
            u0 = pair * ntiles;
            u1 = u0 + ntiles;
        } else {
            const int64_t U = rows * ntiles;
            u0 = pair * U / P;
            u1 = (pair + 1) * U / P;
        }
        sg.n = 0;
        auto add = [&](int64_t r, int k, int64_t len) {
            if (len <= 0)
                return;
            sg.t[sg.n] = r / G;
            sg.hg[sg.n] = (int)(r % G);
            sg.k[sg.n] = k;
            sg.len[sg.n] = (int)len;
            ++sg.n;
        };
        if (u1 > u0) {
            const int64_t rf = u0 / ntiles, rl = (u1 - 1) / ntiles;
            const int kf = (int)(u0 % ntiles), kl = (int)((u1 - 1) % ntiles);
            if (rf == rl) {
                add(rf, kf, u1 - u0);
            } else {
                if (kf != 0)
                    add(rf, kf, ntiles - kf); // the end of the first row
                const int64_t w0 = kf != 0 ? rf + 1 : rf, w1 = kl != ntiles - 1 ? rl - 1 : rl;
                if (w1 >= w0)
                    add(w0, 0, (w1 - w0 + 1) * ntiles);
                if (kl != ntiles - 1)
                    add(rl, 0, kl + 1);       // the beginning of the last
            }
        }
    }
    if (warp == kQkWarp)
        umma::alloc(smem_u32(tmem_slot), kTmemCols);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    int n = 0; // tiles of this CTA
    for (int i = 0; i < sg.n; ++i)
        n += sg.len[i];
    // the prologue above touches no global memory: from here on the previous
    // kernel in the stream (which may produce this call's inputs, or still
    // read this call's outputs) must be complete; the next one may start its
    // own prologue on free SMs meanwhile
    umma::grid_launch_dependents();
    umma::grid_wait();

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

    if (ntiles == 0) {
        // no keys (topk = 0): one pair per row; the softmax threads write the
        // row's half of zeros and its lse (the sink alone, or -inf)
        if (warp < 4) {
            const int64_t t = pair / G;
            const int hg = (int)(pair % G), h = tid;
            uint4 *o = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.out) +
                                                 ((t * a.H + hg * kHeads + h) * kDv + half * kDvHalf));
#pragma unroll 4
            for (int i = 0; i < kDvHalf / 8; ++i)
                o[i] = make_uint4(0u, 0u, 0u, 0u);
            if (half == 0 && a.lse != nullptr)
                a.lse[t * a.H + hg * kHeads + h] = a.sinks != nullptr ? a.sinks[hg * kHeads + h] : -INFINITY;
        }
    } else if (warp >= kProducerWarp0 && warp < kProducerWarp0 + kProducerWarps) {
        // ======================= producers =======================
        // warp pw issues copies 14 pw .. 14 pw + 13 of every tile (fewer in the
        // last warp): copy c = key quad c / 5, column block c % 5; each copier
        // lane loads its quad's four indices, kIdxAhead tiles ahead
        const int pw = warp - kProducerWarp0;
        const int cid = pw * kCopiesPerWarp + lane;
        const bool copier = lane < kCopiesPerWarp && cid < kCopies;
        const int quad = cid / kCB, cb = cid % kCB;
        const int warp_copies = min(kCopiesPerWarp, kCopies - pw * kCopiesPerWarp);
        Cur cf;
        cur_load(cf, sg, 0);
        auto fetch = [&](int (&r)[4]) {
            const bool live = cf.seg < sg.n;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = cf.k * kKeys + 4 * quad + u;
                r[u] = (live && copier && p < a.topk) ? __ldg(a.indices + cf.t * (int64_t)a.topk + p) : -1;
            }
            if (live)
                cur_next(cf, sg, ntiles, G);
        };
        auto row = [&](int x) { return (x >= 0 && (int64_t)x < a.num_slots) ? x : -1; };
        static_assert(kIdxAhead == 4, "one register slot per tile of look-ahead");
        int r0[4], r1[4], r2[4], r3[4];
        fetch(r0);
        fetch(r1);
        fetch(r2);
        fetch(r3);
        int issued = 0;
        bool stop = false;
        auto step = [&](int j, int (&r)[4]) {
            if (stop || j >= n) {
                stop = true;
                return;
            }
            const int st = j % kStages;
            int go = 0;
            if (lane == 0) {
                if (j >= kStages)
                    wait_bar(empty(st), (uint32_t)((j / kStages - 1) & 1));
                go = !*(volatile int *)abort_s;
                if (go)
                    umma::mbar_arrive_expect_tx(full(st), (uint32_t)(warp_copies * 512));
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!go) {
                stop = true;
                return;
            }
            if (copier)
                umma::tma_gather4(ring + st * kTile + cb * kKBlk + quad * 512, &kv_map, 128 * cb, row(r[0]),
                                  row(r[1]), row(r[2]), row(r[3]), full(st));
            issued = j + 1;
            fetch(r);
        };
        for (int j0 = 0; !stop; j0 += kIdxAhead) {
            step(j0, r0);
            step(j0 + 1, r1);
            step(j0 + 2, r2);
            step(j0 + 3, r3);
        }
        // this warp's copies in flight have landed (also after an abort)
        if (lane == 0) {
            for (int j = max(0, issued - kStages); j < issued; ++j)
                wait_issued(full(j % kStages), (uint32_t)((j / kStages) & 1));
        }
        __syncwarp();
    } else if (warp == kQkWarp) {
        // ======================= QK issuer =======================
        if (lane == 0) {
            Cur cu;
            cur_load(cu, sg, 0);
            int piece = -1; // the piece whose q8 was loaded last
            for (int j = 0; j < n; ++j) {
                const int b = j & 1, st = j % kStages;
                if (cu.begin) {
                    // this piece's row: its q8 (once the previous piece's QK MMAs are done with q8)
                    if (piece >= 0) {
                        umma::commit(q_free);
                        wait_bar(q_free, (uint32_t)(piece & 1));
                    }
                    if (*(volatile int *)abort_s)
                        break;
                    ++piece;
                    umma::mbar_arrive_expect_tx(q_full, 4 * kQBlk + kQRope);
                    const int qrow = (int)(cu.t * a.H + cu.hg * kHeads);
                    for (int c = 0; c < 4; ++c)
                        umma::tma_load_2d(q8_s + c * kQBlk, &q8_map, 128 * c, qrow, q_full);
                    umma::bulk_copy_g2s(qrope_s, a.q8_rope + (cu.t * G + cu.hg) * kQRope, kQRope, q_full);
                    // the next piece's q8 into L2 meanwhile: the next row of this
                    // segment, or the next segment's first
                    int64_t nt = -1;
                    int nhg = 0;
                    if (cu.left > ntiles - cu.k) {
                        nt = cu.t + (cu.hg + 1 == G ? 1 : 0);
                        nhg = cu.hg + 1 == G ? 0 : cu.hg + 1;
                    } else if (cu.seg + 1 < sg.n) {
                        nt = sg.t[cu.seg + 1];
                        nhg = sg.hg[cu.seg + 1];
                    }
                    if (nt >= 0) {
                        umma::prefetch_l2(a.q8 + (nt * a.H + nhg * kHeads) * 512, kHeads * 512);
                        umma::prefetch_l2(a.q8_rope + (nt * G + nhg) * kQRope, kQRope);
                    }
                    wait_bar(q_full, (uint32_t)(piece & 1));
                }
                wait_bar(full(st), (uint32_t)((j / kStages) & 1));
                if (j >= 2) // the softmax has read S(j-2)
                    wait_bar(p_full(b), (uint32_t)(((j - 2) >> 1) & 1));
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
                cur_next(cu, sg, ntiles, G);
            }
            // the q8 copies in flight have landed (also after an abort)
            if (piece >= 0)
                wait_issued(q_full, (uint32_t)(piece & 1));
            umma::commit(drain);
            wait_issued(drain, 0);
        }
        __syncwarp();
    } else if (warp == kPvWarp) {
        // ======================= PV issuer =======================
        if (lane == 0) {
            Cur cu;
            cur_load(cu, sg, 0);
            int piece = -1;
            bool first = false; // the piece's first PV overwrites O^T
            for (int j = 0; j < n; ++j) {
                const int b = j & 1;
                if (cu.begin) {
                    // O^T is overwritten by this piece: the previous piece's O^T has been read out
                    if (piece >= 0)
                        wait_bar(o_free, (uint32_t)(piece & 1));
                    ++piece;
                    first = true;
                }
                wait_bar(p_full(b), (uint32_t)((j >> 1) & 1));
                wait_bar(v_full(b), (uint32_t)((j >> 1) & 1));
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
                                         bd + (uint64_t)((kk * 32) >> 4), kIdescPV, (!first || kk > 0) ? 1u : 0u);
                first = false;
                umma::commit(p_empty(b));
                cur_next(cu, sg, ntiles, G);
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
        for (int i = 0; i < n; ++i) {
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
    } else if (warp < 4) {
        // ======================= softmax (thread = head) =======================
        const int h = tid; // 0..127
        const int d0 = warp * 32 + lane; // this thread's O^T lane: value dim d0 (+128) of the half
        const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
        const float kvs = *a.kv_scale;
        float m_ref = -INFINITY, l = 0.f, fac = 0.f;
        int kp = 0, jp = 0; // the current piece's first key tile and its tile index
        Cur cu;
        cur_load(cu, sg, 0);
        // validity of a tile's 64 keys (the same for every head): lane j checks
        // keys j and j + 32, a ballot gathers the mask; the indices are loaded
        // four tiles ahead (cursor cf), since under the gathers' traffic a load
        // can take longer than a tile
        Cur cf;
        cur_load(cf, sg, 0);
        auto load_idx = [&](int off) {
            if (cf.seg >= sg.n)
                return -1;
            const int p = cf.k * kKeys + off + lane;
            return p < a.topk ? __ldg(a.indices + cf.t * (int64_t)a.topk + p) : -1;
        };
        auto ok = [&](int x) { return x >= 0 && (int64_t)x < a.num_slots; };
        int xa0 = load_idx(0), xb0 = load_idx(32);
        if (cf.seg < sg.n)
            cur_next(cf, sg, ntiles, G);
        int xa1 = load_idx(0), xb1 = load_idx(32);
        if (cf.seg < sg.n)
            cur_next(cf, sg, ntiles, G);
        int xa2 = load_idx(0), xb2 = load_idx(32);
        if (cf.seg < sg.n)
            cur_next(cf, sg, ntiles, G);
        int xa3 = load_idx(0), xb3 = load_idx(32);
        if (cf.seg < sg.n)
            cur_next(cf, sg, ntiles, G);
        __nv_bfloat16 *const out_b = static_cast<__nv_bfloat16 *>(a.out);
        // output staging: [64 heads][256 dims] bf16 of this half in the P^T
        // buffers (free while a piece finishes: its last PV is done, and the
        // next piece's P^T comes from these threads), then written out with
        // 16-byte stores, a head's 512 bytes contiguous
        __nv_bfloat16 *const stage = reinterpret_cast<__nv_bfloat16 *>(smem + kOffPT);
        static_assert(2 * kPT == 64 * kDvHalf * 2, "the staging block fills the P^T buffers");
        auto flush_stage = [&](int64_t t, int hg, int c0) {
            umma::named_bar(1, 128); // the block is staged
            __nv_bfloat16 *orow = out_b + (t * a.H + hg * kHeads + c0) * kDv + half * kDvHalf;
            const uint4 *src = reinterpret_cast<const uint4 *>(stage);
#pragma unroll 4
            for (int i = h; i < 64 * (kDvHalf / 8); i += 128)
                *reinterpret_cast<uint4 *>(orow + (int64_t)(i >> 5) * kDv + (i & 31) * 8) = src[i];
            umma::named_bar(1, 128); // the block may be restaged
        };

        // ---- the end of a piece: O^T / l -> out (a whole row), or a partial to
        // the workspace and, for the second piece of a shared row, the merge ----
        auto finish_piece = [&](int j) {
            const int64_t t = cu.t;
            const int hg = cu.hg;
            const bool whole = kp == 0 && cu.k == ntiles - 1;
            wait_bar(p_empty(j & 1), (uint32_t)((j >> 1) & 1)); // the piece's last PV (and every earlier one)
            umma::fence_after_sync();
            const float sk = a.sinks != nullptr ? a.sinks[hg * kHeads + h] * kLog2e : -INFINITY;
            // the piece's output factor and lse (natural log; with the sink for a whole row)
            float f = 0.f, lse_p = -INFINITY;
            if (whole) {
                // a sink logit (base-2 units sk) joins the denominator: l 2^m_ref + 2^sk,
                // taken relative to M = max(m_ref, sk)
                if (l > 0.f) {
                    const float M = fmaxf(m_ref, sk);
                    const float lt = l * exp2f(m_ref - M) + (sk == -INFINITY ? 0.f : exp2f(sk - M));
                    f = kvs * exp2f(m_ref - M) / lt;
                    lse_p = (M + log2f(lt)) * kLn2;
                } else if (sk != -INFINITY) {
                    lse_p = sk * kLn2; // no valid key: the sink alone
                }
                if (half == 0 && a.lse != nullptr)
                    a.lse[t * a.H + hg * kHeads + h] = lse_p;
            } else if (l > 0.f) {
                f = 1.0f / l; // a partial stays in units of the cache's codes
                lse_p = (m_ref + log2f(l)) * kLn2;
            }
            alpha_s[h] = f; // output factor per head
            umma::named_bar(1, 128);
            if (whole) {
                // thread = value dims 128 mb + d0; columns = heads; each store
                // instruction writes 32 consecutive dims of one head (direct
                // stores measured faster than staging the block through
                // shared memory)
                __nv_bfloat16 *const obase = out_b + (t * a.H + hg * kHeads) * kDv + half * kDvHalf + d0;
#pragma unroll 1
                for (int mb = 0; mb < 2; ++mb) {
#pragma unroll 1
                    for (int c = 0; c < kHeads; c += 32) {
                        uint32_t o[32];
                        umma::ld32(tl + 128 * mb + c, o);
                        umma::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float fe = alpha_s[c + e];
                            obase[(int64_t)(c + e) * kDv + 128 * mb] =
                                __float2bfloat16_rn(fe > 0.f ? __uint_as_float(o[e]) * fe : 0.f);
                        }
                    }
                }
                umma::fence_before_sync();
                umma::mbar_arrive(o_free);
                return;
            }
            // a piece of a shared row: the end of the pair's first row (slot
            // 2 pair) or the beginning of its last (slot 2 pair + 1). The row's
            // flag word holds bit 1 once the end piece's partial is visible and
            // bit 2 once the beginning piece's is.
            const bool beginning = kp == 0;
            const int64_t slot = 2 * pair + (beginning ? 1 : 0);
            const int my_bit = beginning ? 2 : 1, other_bit = 3 - my_bit;
            int *flag = a.wide_tickets + (t * G + hg) * 2 + half;
            if (h == 0)
                *last_s = (atomicOr(flag, 0) & other_bit) != 0; // the other piece has finished
            umma::named_bar(1, 128);
            if (!*last_s) {
                // store this piece (binary16 of this half) as 16-byte granules of 8
                // heads, [head group][256 dims][8 heads], so that a warp's lanes
                // (consecutive dims) store, and the merge later loads, contiguous
                // 512 bytes; and its 128 lse
                uint4 *po = reinterpret_cast<uint4 *>(a.wide_part + (slot * 2 + half) * (int64_t)(kDvHalf * kHeads));
#pragma unroll 1
                for (int mb = 0; mb < 2; ++mb) {
                    uint4 *pd = po + 128 * mb + d0;
#pragma unroll 1
                    for (int c = 0; c < kHeads; c += 32) {
                        uint32_t o[32];
                        umma::ld32(tl + 128 * mb + c, o);
                        umma::wait_ld();
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float f0 = alpha_s[c + 2 * e], f1 = alpha_s[c + 2 * e + 1];
                            w[e] = pack_f16x2(f0 > 0.f ? __uint_as_float(o[2 * e]) * f0 : 0.f,
                                              f1 > 0.f ? __uint_as_float(o[2 * e + 1]) * f1 : 0.f);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            __stcg(pd + (c / 8 + q) * kDvHalf, make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
                    }
                }
                __stcg(a.wide_part_lse + (slot * 2 + half) * kHeads + h, lse_p);
                __threadfence();
                umma::named_bar(1, 128);
                if (h == 0)
                    *last_s = (atomicOr(flag, my_bit) & other_bit) != 0;
                umma::named_bar(1, 128);
                if (!*last_s) {
                    umma::fence_before_sync();
                    umma::mbar_arrive(o_free);
                    return;
                }
            }
            if (h == 0)
                *flag = 0; // both pieces are in: ready for the next call
            __threadfence();
            // ---- the merge: the row's beginning piece and its end piece, in that
            // order; this CTA's own piece comes from tensor memory, rounded to
            // binary16 exactly as it was stored, the other from the workspace ----
            const int64_t other = beginning ? 2 * (pair + 1) : 2 * (pair - 1) + 1;
            const float lo = __ldcg(a.wide_part_lse + (other * 2 + half) * kHeads + h) * kLog2e;
            const float lm = lse_p * kLog2e;
            const float lb = beginning ? lm : lo, le = beginning ? lo : lm;
            const float mx = fmaxf(sk, fmaxf(lb, le));
            const float eb = mx == -INFINITY ? 0.f : exp2f(lb - mx), ee = mx == -INFINITY ? 0.f : exp2f(le - mx);
            const float tot = eb + ee + ((mx == -INFINITY || sk == -INFINITY) ? 0.f : exp2f(sk - mx)); // the sink: no output
            if (half == 0 && a.lse != nullptr)
                a.lse[t * a.H + hg * kHeads + h] = mx == -INFINITY ? -INFINITY : (mx + log2f(tot)) * kLn2;
            wts_s[h] = tot > 0.f ? kvs * (eb / tot) : 0.f;
            wts_s[kHeads + h] = tot > 0.f ? kvs * (ee / tot) : 0.f;
            umma::named_bar(1, 128);
            const uint4 *ps = reinterpret_cast<const uint4 *>(a.wide_part + (other * 2 + half) * (int64_t)(kDvHalf * kHeads));
#pragma unroll 1
            for (int c0 = 0; c0 < kHeads; c0 += 64) {
                uint4 v[2][8]; // the other piece's 64 heads of this thread's two dims, loaded together
#pragma unroll
                for (int mb = 0; mb < 2; ++mb)
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        v[mb][u] = __ldcg(ps + (c0 / 8 + u) * kDvHalf + 128 * mb + d0);
#pragma unroll
                for (int mb = 0; mb < 2; ++mb) {
#pragma unroll
                    for (int cc = 0; cc < 64; cc += 16) {
                        const int c = c0 + cc;
                        uint32_t o[16];
                        umma::ld16(tl + 128 * mb + c, o);
                        umma::wait_ld();
                        const uint32_t wv[8] = {v[mb][cc / 8].x,     v[mb][cc / 8].y,     v[mb][cc / 8].z,
                                                v[mb][cc / 8].w,     v[mb][cc / 8 + 1].x, v[mb][cc / 8 + 1].y,
                                                v[mb][cc / 8 + 1].z, v[mb][cc / 8 + 1].w};
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            const float f0 = alpha_s[c + e], f1 = alpha_s[c + e + 1];
                            const uint32_t own = pack_f16x2(f0 > 0.f ? __uint_as_float(o[e]) * f0 : 0.f,
                                                            f1 > 0.f ? __uint_as_float(o[e + 1]) * f1 : 0.f);
                            const float2 pm = __half22float2(*reinterpret_cast<const __half2 *>(&own));
                            const float2 px = __half22float2(*reinterpret_cast<const __half2 *>(&wv[e / 2]));
                            const float2 pb = beginning ? pm : px, pe = beginning ? px : pm;
                            stage[(cc + e) * kDvHalf + 128 * mb + d0] =
                                __float2bfloat16_rn(wts_s[c + e] * pb.x + wts_s[kHeads + c + e] * pe.x);
                            stage[(cc + e + 1) * kDvHalf + 128 * mb + d0] =
                                __float2bfloat16_rn(wts_s[c + e + 1] * pb.y + wts_s[kHeads + c + e + 1] * pe.y);
                        }
                    }
                }
                flush_stage(t, hg, c0);
            }
            umma::fence_before_sync();
            umma::mbar_arrive(o_free);
        };

#pragma unroll 1
        for (int j = 0; j < n; ++j) {
            const int b = j & 1;
            if (cu.begin) {
                jp = j;
                kp = cu.k;
                m_ref = -INFINITY;
                l = 0.f;
                fac = a.scale * kLog2e * a.q_scale[cu.t * a.H + cu.hg * kHeads + h] * kvs;
            }
            const uint32_t m_lo = __ballot_sync(0xffffffffu, ok(xa0));
            const uint32_t m_hi = __ballot_sync(0xffffffffu, ok(xb0));
            xa0 = xa1;
            xb0 = xb1;
            xa1 = xa2;
            xb1 = xb2;
            xa2 = xa3;
            xb2 = xb3;
            xa3 = load_idx(0); // tile j + 4
            xb3 = load_idx(32);
            if (cf.seg < sg.n)
                cur_next(cf, sg, ntiles, G);
            wait_bar(s_full(b), (uint32_t)((j >> 1) & 1));
            umma::fence_after_sync();
            float sv[64];
            umma::ld32(tl + kSCol + 64 * b, reinterpret_cast<uint32_t(&)[32]>(sv[0]));
            umma::ld32(tl + kSCol + 64 * b + 32, reinterpret_cast<uint32_t(&)[32]>(sv[32]));
            umma::wait_ld();
            // the tile max in four independent chains; a tile whose 64 keys are all
            // valid (the common case) skips the masking
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if ((m_lo & m_hi) == 0xffffffffu) {
#pragma unroll
                for (int q = 0; q < 64; ++q) {
                    sv[q] *= fac;
                    mx[q & 3] = fmaxf(mx[q & 3], sv[q]);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 64; ++q) {
                    const bool v = ((q < 32 ? m_lo >> q : m_hi >> (q - 32)) & 1u) != 0;
                    sv[q] = v ? sv[q] * fac : -INFINITY;
                    mx[q & 3] = fmaxf(mx[q & 3], sv[q]);
                }
            }
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
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
                if (j > jp) {
                    // O^T holds PV(jp..j-1): let PV(j-1) finish, then scale each head column
                    wait_bar(p_empty((j - 1) & 1), (uint32_t)(((j - 1) >> 1) & 1));
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
            if (j >= 2) // PV(j-2) has read P^T(b)
                wait_bar(p_empty(b), (uint32_t)(((j - 2) >> 1) & 1));
            // this head's row of P^T: 64 keys x fp16 = one 128-byte swizzled row,
            // written 16 bytes (8 keys) at a time
            const uint32_t prow = pt_s + b * kPT + h * 128;
            float ls[4] = {0.f, 0.f, 0.f, 0.f}; // the tile's sum in four independent chains
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = ex2_approx(sv[8 * c8 + 2 * e] - mu), p1 = ex2_approx(sv[8 * c8 + 2 * e + 1] - mu);
                    ls[e] += p0 + p1;
                    w[e] = pack_f16x2(p0, p1);
                }
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + ((c8 ^ (h & 7)) << 4)), "r"(w[0]),
                             "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            umma::fence_async_smem();
            umma::fence_before_sync();
            umma::mbar_arrive(p_full(b));
            if (cu.left == 1 || cu.k == ntiles - 1)
                finish_piece(j);
            cur_next(cu, sg, ntiles, G);
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((qrows + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_q_e4m3_kernel, static_cast<const __nv_bfloat16 *>(a.q), qrows, a.H,
                              a.q8, a.q8_rope, a.q_scale,
                              a.q_fp8_in ? static_cast<const uint8_t *>(a.q) : nullptr, a.q_scale_in);
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
    const int64_t blocks = (int64_t)a.wide_pairs * 2;
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
