// Sparse MLA forward for 128 heads over an E4M3 cache (D_qk = 576: 512
// latent + 64 rope columns, D_v = 512) with each key row gathered once per
// query row: a pair of CTAs in one thread-block cluster (tcgen05 + tensor
// memory, TMA row gathers with cluster multicast, sm_103a).
//
// The two CTAs of a query row each own half of the value dims (the fp32
// output for 128 heads x 512 dims would fill an SM's tensor memory), so each
// needs every key's 576 columns for QK and its half of the values for PV.
// Gathering every key in both CTAs makes the row gather, which bounds this
// path, twice as long. Here each CTA gathers half of every 64-key tile (32
// keys, all five 128-byte column blocks) and delivers it to both CTAs' shared
// memory with one multicast copy, so each row leaves HBM once. A stage is
// refilled only after both CTAs are done with it: the QK issuer of each CTA
// commits to the "empty" barrier of both, and so does one converter thread.
//
// Per CTA (as in the 128-head kernel without the pair):
//   S   [128 heads x 64 keys]  = q8 [128 x 576] . K_tile^T          (E4M3, 18 MMAs, M=128 N=64)
//   O^T [256 dims x 128 heads] += V^T[half] [256 x 64] . P^T        (fp16, 8 MMAs, 2 x M=128 N=128)
// Tensor memory (512 columns): O^T in 0..255, S in 256 + 64 b, V^T in
// 384 + 64 b (binary16, two keys per column). Shared memory: q8 (4 swizzled
// blocks [128 heads x 128 B] + an 8 KB core-matrix block for the rope part),
// a 3-stage ring of 40 KB tiles, P^T (fp16 [128 heads x 64 keys], K-major,
// double-buffered).
//
// Warp roles (every wait bounded):
//   softmax (warps 0-7): thread = (head 32 (w % 4) + lane, key half w / 4),
//     32 logits each; masks, scales by scale * s_q[h] * kv_scale,
//     exponentiates base 2 against a running reference max that moves (all
//     heads agree per tile, then the O^T columns are rescaled in tensor
//     memory) only when a logit passes it by more than 2^8, and then to 2^8
//     above the tile max; writes its half of the head's P^T row (fp16).
//   QK issuer (warp 8), PV issuer (warp 9): one thread each.
//   producers (warps 10-11): 40 multicast gather4 copies per tile (this
//     CTA's 8 key quads x 5 column blocks; the fifth block reaches past
//     column 576 and is zero filled); -1 and out-of-range indices go to the
//     TMA as row -1 (zero fill, no read).
//   converters (warps 12-15): this CTA's half of the value columns, E4M3 ->
//     binary16 (exact), as V^T into tensor memory.
// q is quantized by the same pre-pass as the 128-head kernel (per (row,
// head): s_q = amax/448, q8 = RNE_satfinite(q / s_q)).
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

__device__ int g_wide2_error = 0; // set when a bounded wait gives up

namespace {

constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kDvHalf = 256;
constexpr int kKeys = 64;             // keys per tile (N of QK), 32 gathered by each CTA
constexpr int kQkSteps = kDqk / 32;
constexpr int kCB = 5;
constexpr int kStages = 3;
constexpr int kCopies = 8 * kCB;      // this CTA's gather4 copies per tile
constexpr int kIdxAhead = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kHeadroom = 8.0f;

constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kQkWarp = 8;
constexpr int kPvWarp = 9;
constexpr int kProducerWarp0 = 10;    // warps 10-11
constexpr int kProducerThreads = 64;
constexpr int kConverterWarp0 = 12;   // warps 12-15
constexpr int kConverterThreads = 128;
constexpr int kThreads = 16 * 32;

// shared memory (bytes from a 1 KB-aligned base)
constexpr int kQBlk = kHeads * 128;
constexpr int kOffQ8 = 0;
constexpr int kQRope = kHeads * 64;
constexpr int kOffQRope = kOffQ8 + 4 * kQBlk;
constexpr int kKBlk = kKeys * 128;
constexpr int kTile = kCB * kKBlk;    // 40 KB
constexpr int kOffRing = kOffQRope + kQRope;
constexpr int kPT = kHeads * 128;
constexpr int kOffPT = kOffRing + kStages * kTile;
constexpr int kOffAlpha = kOffPT + 2 * kPT;     // [128] per-head factors
constexpr int kOffHmax = kOffAlpha + kHeads * 4; // [2][128] half-tile maxima, then the two l halves
constexpr int kOffEx = kOffHmax + 2 * kHeads * 4;
constexpr int kOffMisc = kOffEx + 2 * kSoftmaxWarps * 4; // tmem address, abort, go[2]
constexpr int kOffMbar = kOffMisc + 32;
// full[3], empty[3], s_full[2], p_full[2], p_empty[2], v_full[2], q_full, drain
constexpr int kNBar = 16;
constexpr int kSmem = kOffMbar + kNBar * 8;
constexpr int kSmemAlloc = kSmem + 1024;
static_assert(kOffRing % 1024 == 0 && kOffPT % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kSmemAlloc <= 227 * 1024, "shared memory budget");

constexpr int kTmemCols = 512;
constexpr int kSCol = 256;
constexpr int kVCol = 384;

constexpr uint32_t kIdescQK = umma::idesc(128, 64, 0, 0, 0, 0);
constexpr uint32_t kIdescPV = umma::idesc(128, 128, 0, 0, 0, 0);

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_fwd_wide2_kernel(const FwdArgs a, const __grid_constant__ CUtensorMap kv_map,
                                const __grid_constant__ CUtensorMap q8_map)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    const uint32_t q8_s = sbase + kOffQ8, qrope_s = sbase + kOffQRope, ring = sbase + kOffRing,
                   pt_s = sbase + kOffPT;
    float *alpha_s = reinterpret_cast<float *>(smem + kOffAlpha);
    float *hmax_s = reinterpret_cast<float *>(smem + kOffHmax);
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
    const uint32_t rank = umma::cluster_rank(); // == blockIdx.x & 1: the value half this CTA owns
    const uint32_t peer = rank ^ 1u;
    const int half = (int)rank;
    const int hg = (blockIdx.x >> 1) % G;
    const int t = (blockIdx.x >> 1) / G;
    const int ntiles = (a.topk + kKeys - 1) / kKeys;
    const int32_t *__restrict__ row_idx = a.indices + (int64_t)t * a.topk;

    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) {
            umma::mbar_init(full(st), 1);
            umma::mbar_init(empty(st), 4); // each CTA's QK commit and each CTA's converters
        }
        for (int b = 0; b < 2; ++b) {
            umma::mbar_init(s_full(b), 1);
            umma::mbar_init(p_full(b), kSoftmaxThreads);
            umma::mbar_init(p_empty(b), 1);
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
    // both CTAs' barriers are initialised before either sends to the other
    umma::cluster_barrier();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    umma::grid_launch_dependents();
    umma::grid_wait();

    // ---- q8 of this row's 128 heads: four TMA tile loads and one bulk copy ----
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
            atomicOr(&g_wide2_error, 1);
            *(volatile int *)abort_s = 1;
        }
    };
    auto wait_issued = [&](uint32_t mbar, uint32_t parity) {
        if (!umma::mbar_wait(mbar, parity))
            atomicOr(&g_wide2_error, 2);
    };

    if (warp >= kProducerWarp0 && warp < kConverterWarp0) {
        // ======================= producers =======================
        // copy cid: this CTA's key quad cid / 5 (tile keys 32 rank + 4 qd ..), column block cid % 5
        const int pt = tid - kProducerWarp0 * 32;
        const int cid = (pt >> 5) * (kCopies / 2) + (pt & 31);
        const bool copier = (pt & 31) < kCopies / 2;
        const int qd = cid / kCB, cb = cid % kCB;
        const int kq = 8 * half + qd; // the quad's position among the tile's 16
        auto fetch = [&](int tile, int (&r)[4]) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int p = tile * kKeys + 4 * kq + u;
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
                if (j >= kStages) // both CTAs are done with the stage's previous tile
                    wait_bar(empty(st), (uint32_t)((j / kStages - 1) & 1));
                const int go = !*(volatile int *)abort_s;
                if (go) // this CTA's stage receives the whole tile: its own half and the peer's
                    umma::mbar_arrive_expect_tx(full(st), kTile);
                go_s[j & 1] = go;
            }
            umma::named_bar(2, kProducerThreads);
            if (!go_s[j & 1]) {
                stop = true;
                return;
            }
            if (copier)
                umma::tma_gather4_multicast(ring + st * kTile + cb * kKBlk + kq * 512, &kv_map, 128 * cb, row(r[0]),
                                            row(r[1]), row(r[2]), row(r[3]), full(st), (uint16_t)3);
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
            // this CTA's stages: every copy into them (its own and the peer's) has landed
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
                const uint64_t rd = umma::desc(qrope_s, 128, 512);
                const uint64_t bd = umma::desc_sw128(ring + st * kTile, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < kQkSteps; ++ks) {
                    const uint64_t ak = ks < 16 ? ad + (uint64_t)(((ks >> 2) * kQBlk + (ks & 3) * 32) >> 4)
                                                : rd + (uint64_t)(((ks - 16) * 256) >> 4);
                    umma::mma_f8(tmem + kSCol + 64 * b, ak,
                                 bd + (uint64_t)(((ks >> 2) * kKBlk + (ks & 3) * 32) >> 4), kIdescQK, ks > 0);
                }
                umma::commit(s_full(b));
                umma::commit_multicast(empty(st), (uint16_t)3); // this CTA's QK no longer reads the stage
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
        const int q4 = warp & 3, g = lane >> 2, ii = lane & 3;
        const uint32_t selA = ii < 2 ? 0x5410u : 0x3276u;
        const uint32_t selB = ii & 1 ? 0x3715u : 0x6240u;
        const uint32_t tlane = (uint32_t)(32 * q4) << 16;
        for (int i = 0; i < ntiles; ++i) {
            const int st = i % kStages, vb = i & 1;
            wait_bar(full(st), (uint32_t)((i / kStages) & 1));
            if (i >= 2) // PV(i-2) has read V^T buffer vb
                wait_bar(p_empty(vb), (uint32_t)(((i - 2) >> 1) & 1));
            const uint32_t src0 = ring + st * kTile;
#pragma unroll 1
            for (int mb = 0; mb < 2; ++mb) {
                const uint32_t blk = src0 + (2 * half + mb) * kKBlk;
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
            // done reading the stage: one arrival on each CTA's "empty" barrier
            umma::named_bar(3, kConverterThreads);
            if (warp == kConverterWarp0 && lane == 0) {
                umma::mbar_arrive_cluster(empty(st), rank);
                umma::mbar_arrive_cluster(empty(st), peer);
            }
        }
    } else {
        // ======================= softmax =======================
        const int h = 32 * (warp & 3) + lane; // head (TMEM lane)
        const int kh = warp >> 2;             // key half of the tile: keys 32 kh .. 32 kh + 31
        const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const float kvs = *a.kv_scale;
        const float fac = a.scale * kLog2e * a.q_scale[(int64_t)t * a.H + hg * kHeads + h] * kvs;
        float m_ref = -INFINITY, l = 0.f;
        auto load_idx = [&](int tile) {
            const int p = tile * kKeys + 32 * kh + lane;
            return (tile < ntiles && p < a.topk) ? __ldg(row_idx + p) : -1;
        };
        int x0 = load_idx(0), x1 = load_idx(1), x2 = load_idx(2), x3 = load_idx(3);
        auto ok = [&](int x) { return x >= 0 && (int64_t)x < a.num_slots; };
        auto step = [&](int i, int &x) {
            if (i >= ntiles)
                return;
            const int b = i & 1;
            const uint32_t mask = __ballot_sync(0xffffffffu, ok(x)); // validity of this half's 32 keys
            x = load_idx(i + kIdxAhead);
            wait_bar(s_full(b), (uint32_t)((i >> 1) & 1));
            umma::fence_after_sync();
            float sv[32];
            umma::ld16(tl + kSCol + 64 * b + 32 * kh, reinterpret_cast<uint32_t(&)[16]>(sv[0]));
            umma::ld16(tl + kSCol + 64 * b + 32 * kh + 16, reinterpret_cast<uint32_t(&)[16]>(sv[16]));
            umma::wait_ld();
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                sv[j] = ((mask >> j) & 1u) ? sv[j] * fac : -INFINITY;
                mt = fmaxf(mt, sv[j]);
            }
            hmax_s[kh * kHeads + h] = mt;
            const bool wx = __any_sync(0xffffffffu, mt > m_ref + kRescaleThreshold);
            if (lane == 0)
                ex_s[b * kSoftmaxWarps + warp] = wx;
            umma::named_bar(1, kSoftmaxThreads);
            int any = 0;
#pragma unroll
            for (int w = 0; w < kSoftmaxWarps; ++w)
                any |= ex_s[b * kSoftmaxWarps + w];
            if (any) {
                // the head's tile max over both halves decides, the same in both threads
                const float tmx = fmaxf(hmax_s[h], hmax_s[kHeads + h]);
                const bool exceed = tmx > m_ref + kRescaleThreshold;
                const float mn = exceed ? tmx + kHeadroom : m_ref;
                const float al = !exceed ? 1.f : (m_ref == -INFINITY ? 0.f : exp2f(m_ref - mn));
                m_ref = mn;
                l *= al;
                if (kh == 0)
                    alpha_s[h] = al;
                umma::named_bar(1, kSoftmaxThreads);
                if (i >= 1) {
                    // O^T holds PV(0..i-1): let PV(i-1) finish, then scale each head column;
                    // warps 0-3 take M-block 0, warps 4-7 M-block 1
                    wait_bar(p_empty((i - 1) & 1), (uint32_t)(((i - 1) >> 1) & 1));
                    umma::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < kHeads; c += 16) {
                        uint32_t o[16];
                        umma::ld16(tl + 128 * kh + c, o);
                        umma::wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha_s[c + e]);
                        umma::st16(tl + 128 * kh + c, o);
                    }
                    umma::wait_st();
                }
                // every thread has read the tile's maxima and factors before the next tile writes them
                umma::named_bar(1, kSoftmaxThreads);
            }
            const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;
            uint32_t pw[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float p0 = ex2_approx(sv[2 * c] - mu), p1 = ex2_approx(sv[2 * c + 1] - mu);
                l += p0 + p1;
                pw[c] = pack_f16x2(p0, p1);
            }
            if (i >= 2) // PV(i-2) has read P^T(b)
                wait_bar(p_empty(b), (uint32_t)(((i - 2) >> 1) & 1));
            // this thread's half of the head's P^T row: 32 keys x fp16 = chunks 4 kh .. 4 kh + 3
            const uint32_t prow = pt_s + b * kPT + h * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + (((4 * kh + c) ^ (h & 7)) << 4)),
                             "r"(pw[4 * c]), "r"(pw[4 * c + 1]), "r"(pw[4 * c + 2]), "r"(pw[4 * c + 3])
                             : "memory");
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
        // ---- epilogue: O^T / l -> out, lse ----
        if (ntiles > 0) // the last PV (and every earlier one) is done
            wait_bar(p_empty((ntiles - 1) & 1), (uint32_t)(((ntiles - 1) >> 1) & 1));
        umma::fence_after_sync();
        hmax_s[kh * kHeads + h] = l; // the two halves' sums of the head
        umma::named_bar(1, kSoftmaxThreads);
        if (kh == 0) {
            // output factor and lse per head; a sink logit (base-2 units sk) joins the
            // denominator: l 2^m_ref + 2^sk, taken relative to M = max(m_ref, sk)
            const float lt0 = hmax_s[h] + hmax_s[kHeads + h];
            const float sk = a.sinks != nullptr ? a.sinks[hg * kHeads + h] * kLog2e : -INFINITY;
            float f = 0.f, lse_h = -INFINITY;
            if (lt0 > 0.f) {
                const float M = fmaxf(m_ref, sk);
                const float lt = lt0 * exp2f(m_ref - M) + (sk == -INFINITY ? 0.f : exp2f(sk - M));
                f = kvs * exp2f(m_ref - M) / lt;
                lse_h = (M + log2f(lt)) * kLn2;
            } else if (sk != -INFINITY) {
                lse_h = sk * kLn2; // no valid key: the sink alone
            }
            alpha_s[h] = f; // output factor per head
            if (half == 0 && a.lse != nullptr)
                a.lse[(int64_t)t * a.H + hg * kHeads + h] = lse_h;
        }
        umma::named_bar(1, kSoftmaxThreads);
        // thread = value dim 128 kh + 32 (warp % 4) + lane of this CTA's half; columns = heads
        __nv_bfloat16 *obase = static_cast<__nv_bfloat16 *>(a.out) + ((int64_t)t * a.H + hg * kHeads) * kDv +
                               half * kDvHalf + 128 * kh + 32 * (warp & 3) + lane;
#pragma unroll 1
        for (int c = 0; c < kHeads; c += 16) {
            uint32_t o[16];
            umma::ld16(tl + 128 * kh + c, o);
            umma::wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float f = alpha_s[c + e];
                obase[(int64_t)(c + e) * kDv] = __float2bfloat16_rn(f > 0.f ? __uint_as_float(o[e]) * f : 0.f);
            }
        }
        umma::fence_before_sync();
    }
    __syncthreads();
    if (warp == kQkWarp)
        umma::dealloc(tmem, kTmemCols);
    // the peer may still send to this CTA's barriers and ring: leave together
    umma::cluster_barrier();
}

} // namespace

cudaError_t launch_fwd_wide2(const FwdArgs &a, cudaStream_t stream)
{
    auto kern = sparse_mla_fwd_wide2_kernel;
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
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr)
        return cudaErrorNotSupported;
    // the cache as [rows x 576] bytes, boxes of 128 B x 1 row, 128-byte swizzle
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
    // q8 (latent part) as [T*H rows x 512] bytes, boxes of 128 B x 128 rows
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a, kv_map, q8_map);
}

cudaError_t read_wide2_error(int *out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_wide2_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_wide2_error, &zero, sizeof(int));
    }
    return e;
}

} // namespace smla
