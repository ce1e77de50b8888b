// Measurement kernels: the ceilings the forward kernels are held against.
//
// smla_gather_probe_kernel: a pure indexed-row copy. It moves the rows named
// by an index list from a row pool into a shared-memory ring exactly as the
// forward kernels do, and does nothing with them but fold the first word of
// each row into a checksum. Two copy methods fill the same ring layout (64
// rows per tile, 128-byte column blocks of 128-byte-swizzled rows): TMA
// tile::gather4 copies through a 2-D tensor map over the pool (boxes of 128
// bytes x 1 row, issued by the lanes of up to eight producer warps; -1 passed
// as row -1 so the engine fills zeros and reads nothing), or 16-byte cp.async
// copies from eight warps, a warp per 8 rows, that zero-fill a masked row
// without reading it. Its rate is the most a kernel that gathers the same
// rows this way can reach; the consumer may hold each tile for a while, as
// a stand-in for the arithmetic a real kernel does on it.
//
// smla_l2_read_probe_kernel: every block streams through an L2-resident
// buffer with 16-byte loads that bypass L1, many times over; its rate is the
// L2 -> SM bandwidth a kernel whose data sits in L2 is bound by.
#include "smla_device.cuh"
#include "smla_internal.h"
#include "smla_umma.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>

namespace smla {

__device__ int g_probe_error = 0; // set when a bounded wait gives up

namespace {

constexpr int kRows = 64;            // rows per tile
constexpr int kProducerWarps = 8;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr int kThreads = kProducerThreads + 64; // + a consumer warp and a relay warp
constexpr int kMaxStages = 8;

struct ProbeArgs {
    const uint8_t *pool; // read by the cp.async copies (the TMA copies go through the tensor map)
    const int32_t *indices;
    int64_t n_indices;
    int64_t num_rows;
    uint32_t *checksum; // [gridDim.x]
    int boxes;          // 128-byte boxes per row (1..8)
    int stages;
    int hold_ns;
    int pair_mode;      // 0: single CTAs; CTA pairs in clusters, each gathering half of every tile and
                        // delivering it to both: 1 by TMA multicast, 2 by a bulk copy into the peer;
                        // 3: single CTAs launched in clusters of two
    int issue_warps;    // 0: copy c issued by producer thread c; k (1..8): the copies spread evenly
                        // over warps 0..k-1, ceil(copies / k) lanes each
    int row_bytes;
    int copy_mode;      // 0: TMA tile::gather4; 1: 16-byte cp.async (pair_mode 0, issue_warps 0)
};

__global__ void __launch_bounds__(kThreads) smla_gather_probe_kernel(const ProbeArgs a,
                                                                   const __grid_constant__ CUtensorMap map)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t sbase = (raw_base + 1023u) & ~1023u;
    const int tile_bytes = kRows * 128 * a.boxes;
    const uint32_t ring = sbase;
    const uint32_t bar0 = sbase + a.stages * tile_bytes;
    uint8_t *smem = smem_raw + (sbase - raw_base);
    volatile int *go_s = reinterpret_cast<volatile int *>(smem + a.stages * tile_bytes + 24 * kMaxStages);
    int *abort_s = const_cast<int *>(go_s) + 2;
    auto full = [&](int st) { return bar0 + 8 * st; };                   // this CTA's gathers
    auto empty = [&](int st) { return bar0 + 8 * (kMaxStages + st); };
    auto xfull = [&](int st) { return bar0 + 8 * (2 * kMaxStages + st); }; // the peer's half (pair_mode 2)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // pair_mode 3: independent CTAs, launched in clusters of two (a control)
    const bool mc = a.pair_mode == 1 || a.pair_mode == 2, xc = a.pair_mode == 2;
    const bool async = a.copy_mode == 1;
    const uint32_t rank = mc ? umma::cluster_rank() : 0u;
    const int half_bytes = tile_bytes / 2;
    // tiles are split over CTAs, or over CTA pairs in the multicast mode
    const int64_t units = mc ? gridDim.x / 2 : gridDim.x, unit = mc ? blockIdx.x / 2 : blockIdx.x;
    const int64_t ntiles_all = (a.n_indices + kRows - 1) / kRows;
    const int64_t j0 = ntiles_all * unit / units;
    const int64_t j1 = ntiles_all * (unit + 1) / units;
    const int ntiles = (int)(j1 - j0);

    if (tid == 0) {
        for (int st = 0; st < a.stages; ++st) {
            // cp.async: every producer thread arrives once its own copies of the tile land
            umma::mbar_init(full(st), async ? kProducerThreads : 1);
            umma::mbar_init(empty(st), mc ? 2 : 1); // a pair's stage is refilled once both consumers are done
            umma::mbar_init(xfull(st), 1);
        }
        umma::mbar_init_fence();
        *abort_s = 0;
    }
    __syncthreads();
    if (mc) // both CTAs' barriers are initialised before either sends to the other
        umma::cluster_barrier();

    auto wait_bar = [&](uint32_t mbar, uint32_t parity) {
        if (*(volatile int *)abort_s)
            return;
        if (!umma::mbar_wait(mbar, parity)) {
            atomicOr(&g_probe_error, 1);
            *(volatile int *)abort_s = 1;
        }
    };

    if (warp < kProducerWarps) {
        // copy `tid`: key quad qd (rows 4qd..4qd+3 of the tile), box cb; in the
        // multicast mode each CTA of the pair issues half of the 16 quads
        const int copies = (mc ? 8 : 16) * a.boxes;
        const int per_warp = a.issue_warps > 0 ? (copies + a.issue_warps - 1) / a.issue_warps : 32;
        const int cid = a.issue_warps > 0 ? warp * per_warp + lane : tid;
        const bool copier = (a.issue_warps == 0 || (warp < a.issue_warps && lane < per_warp)) && cid < copies;
        const int qd = (mc ? 8 * (int)rank : 0) + cid / a.boxes, cb = cid % a.boxes;
        auto fetch = [&](int j, int (&r)[4]) {
            if (async) { // lane k < 8 holds row 8 warp + k of the tile
                const int64_t p = (j0 + j) * kRows + 8 * warp + lane;
                r[0] = (lane < 8 && j < ntiles && p < a.n_indices) ? __ldg(a.indices + p) : -1;
                return;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t p = (j0 + j) * kRows + 4 * qd + u;
                r[u] = (copier && j < ntiles && p < a.n_indices) ? __ldg(a.indices + p) : -1;
            }
        };
        auto row = [&](int x) { return (x >= 0 && (int64_t)x < a.num_rows) ? x : -1; };
        int r0[4], r1[4];
        fetch(0, r0);
        fetch(1, r1);
        int issued = 0;
        bool stop = false;
        auto step = [&](int j, int (&r)[4]) {
            if (stop || j >= ntiles) {
                stop = true;
                return;
            }
            const int st = j % a.stages;
            if (tid == 0) {
                if (j >= a.stages)
                    wait_bar(empty(st), (uint32_t)((j / a.stages - 1) & 1));
                const int go = !*(volatile int *)abort_s;
                if (go && !async) // the whole tile, or (pair_mode 2) this CTA's half
                    umma::mbar_arrive_expect_tx(full(st), (uint32_t)(xc ? half_bytes : tile_bytes));
                go_s[j & 1] = go;
            }
            umma::named_bar(1, kProducerThreads);
            if (!go_s[j & 1]) {
                stop = true;
                return;
            }
            if (async) {
                // row `key`: chunk c (16 bytes) to column block c / 8, swizzled chunk (c % 8) ^ (key % 8)
                const uint32_t dst = ring + st * tile_bytes;
                for (int k = 0; k < 8; ++k) {
                    const int x = row(__shfl_sync(0xffffffffu, r[0], k));
                    const int key = 8 * warp + k;
                    const uint8_t *src = a.pool + (int64_t)(x < 0 ? 0 : x) * a.row_bytes;
                    for (int c = lane; c < a.row_bytes / 16; c += 32)
                        cp_async_16(dst + (c >> 3) * (kRows * 128) + key * 128 + (((c & 7) ^ (key & 7)) << 4),
                                    src + c * 16, x < 0 ? 0u : 16u);
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(full(st)) : "memory");
            } else if (copier && mc && !xc)
                umma::tma_gather4_multicast(ring + st * tile_bytes + cb * (kRows * 128) + qd * 512, &map, 128 * cb,
                                            row(r[0]), row(r[1]), row(r[2]), row(r[3]), full(st), (uint16_t)3);
            else if (copier)
                umma::tma_gather4(ring + st * tile_bytes + cb * (kRows * 128) + qd * 512, &map, 128 * cb,
                                  row(r[0]), row(r[1]), row(r[2]), row(r[3]), full(st));
            issued = j + 1;
            fetch(j + 2, r);
        };
        for (int j = 0; !stop; j += 2) {
            step(j, r0);
            step(j + 1, r1);
        }
        // every copy issued has landed before the CTA finishes (also after an abort)
        if (async)
            asm volatile("cp.async.wait_all;\n" ::: "memory");
        if (tid == 0) {
            for (int j = max(0, issued - a.stages); j < issued; ++j)
                if (!umma::mbar_wait(full(j % a.stages), (uint32_t)((j / a.stages) & 1)))
                    atomicOr(&g_probe_error, 2);
        }
    } else if (warp == kProducerWarps + 1) {
        // relay (pair_mode 2): once this CTA's half of a tile has landed, copy it
        // into the same place of the peer's ring (one bulk copy per 128-byte
        // column block: 8 key quads x 512 B), counted on the peer's xfull; the
        // peer's stage is free once both consumers released the tile before
        if (xc && lane == 0) {
            const uint32_t peer = rank ^ 1u;
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % a.stages;
                if (j >= a.stages)
                    wait_bar(empty(st), (uint32_t)((j / a.stages - 1) & 1));
                if (*(volatile int *)abort_s)
                    break;
                umma::mbar_arrive_expect_tx(xfull(st), (uint32_t)half_bytes); // the peer's half, into this CTA
                wait_bar(full(st), (uint32_t)((j / a.stages) & 1));
                if (*(volatile int *)abort_s)
                    break;
                for (int cb = 0; cb < a.boxes; ++cb) {
                    const uint32_t off = ring + st * tile_bytes + cb * (kRows * 128) + rank * 8 * 512;
                    umma::bulk_copy_s2peer(off, off, 8 * 512, xfull(st), peer);
                }
            }
        }
    } else if (lane == 0) {
        // consumer: fold word 0 of every row (box 0; row r's first 16-byte chunk
        // sits at chunk r & 7 of its 128-byte swizzled line), hold, release
        uint32_t x = 0;
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % a.stages;
            wait_bar(full(st), (uint32_t)((j / a.stages) & 1));
            if (xc)
                wait_bar(xfull(st), (uint32_t)((j / a.stages) & 1));
            if (*(volatile int *)abort_s)
                break;
            const uint32_t base = ring + st * tile_bytes;
            const uint64_t t_land = umma::globaltimer();
            for (int r = 0; r < kRows; ++r)
                x ^= lds32(base + r * 128 + ((r & 7) << 4));
            if (a.hold_ns > 0)
                while (umma::globaltimer() - t_land < (uint64_t)a.hold_ns) {
                }
            if (mc) {
                umma::mbar_arrive_cluster(empty(st), rank);
                umma::mbar_arrive_cluster(empty(st), rank ^ 1u);
            } else {
                umma::mbar_arrive(empty(st));
            }
        }
        a.checksum[blockIdx.x] = rank == 0 ? x : 0u; // a pair's two CTAs see the same rows
    }
    __syncthreads();
    if (mc) // the peer may still send to this CTA's ring and barriers
        umma::cluster_barrier();
}

// Streams `n16` 16-byte words `reps` times; each block starts at its own
// offset so the blocks spread over the buffer.
__global__ void __launch_bounds__(512) smla_l2_read_probe_kernel(const uint4 *__restrict__ buf, int64_t n16, int reps,
                                                                uint32_t *checksum)
{
    uint32_t x = 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int r = 0; r < reps; ++r) {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
            const uint4 v = __ldcg(buf + i);
            x = ((x << 1) | (x >> 31)) ^ (v.x + v.y + v.z + v.w);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x ^= __shfl_xor_sync(0xffffffffu, x, o);
    __shared__ uint32_t red[16];
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t y = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
            y ^= red[w];
        checksum[blockIdx.x] = y;
    }
}

} // namespace

// Shared memory of one SM and the part each resident CTA reserves.
constexpr int kSmPerSmBytes = 233472;
constexpr int kCtaReservedBytes = 1024;

int gather_probe_smem(int boxes, int stages)
{
    return 1024 + stages * kRows * 128 * boxes + 24 * kMaxStages + 64;
}

cudaError_t launch_gather_probe(const void *pool, int64_t num_rows, int row_bytes, const int32_t *indices,
                                int64_t n_indices, int ctas_per_sm, int stages, int hold_ns, int pair_mode,
                                int issue_warps, int copy_mode, uint32_t *checksum, int sm_count,
                                cudaStream_t stream)
{
    if ((pair_mode && ctas_per_sm != 1) || copy_mode < 0 || copy_mode > 1 ||
        (copy_mode == 1 && (pair_mode != 0 || issue_warps != 0)))
        return cudaErrorInvalidValue;
    const int boxes = (row_bytes + 127) / 128;
    if (issue_warps > 0 && ((pair_mode == 1 || pair_mode == 2 ? 8 : 16) * boxes + issue_warps - 1) / issue_warps > 32)
        return cudaErrorInvalidValue;
    const int need = gather_probe_smem(boxes, stages);
    // pad each CTA so that no more than ctas_per_sm fit on an SM
    const int pad = kSmPerSmBytes / (ctas_per_sm + 1) - kCtaReservedBytes + 1;
    const int smem = need > pad ? need : pad;
    if ((int64_t)ctas_per_sm * (smem + kCtaReservedBytes) > kSmPerSmBytes || smem > 227 * 1024)
        return cudaErrorInvalidValue;
    // the attribute is raised to the largest size once per device (outside any
    // graph capture: the first call on a device must not be captured)
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    if (const cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess)
        return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
        const cudaError_t e =
            cudaFuncSetAttribute(smla_gather_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess)
            return e;
        attr_done.fetch_or(bit, std::memory_order_release);
    }
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode == nullptr)
        return cudaErrorNotSupported;
    CUtensorMap map;
    const int64_t rows = num_rows < 1 ? 1 : (num_rows > INT_MAX ? (int64_t)INT_MAX : num_rows);
    cuuint64_t gdim[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128, 1};
    cuuint32_t estride[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    ProbeArgs a;
    a.pool = static_cast<const uint8_t *>(pool);
    a.indices = indices;
    a.n_indices = n_indices;
    a.num_rows = num_rows;
    a.checksum = checksum;
    a.boxes = boxes;
    a.stages = stages;
    a.hold_ns = hold_ns;
    a.pair_mode = pair_mode;
    a.issue_warps = issue_warps;
    a.row_bytes = row_bytes;
    a.copy_mode = copy_mode;
    const int grid = pair_mode ? (sm_count / 2) * 2 : sm_count * ctas_per_sm;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pair_mode ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, smla_gather_probe_kernel, a, map);
}

cudaError_t launch_l2_read_probe(const void *buf, int64_t bytes, int reps, uint32_t *checksum, int blocks,
                                 cudaStream_t stream)
{
    smla_l2_read_probe_kernel<<<blocks, 512, 0, stream>>>(static_cast<const uint4 *>(buf), bytes / 16, reps,
                                                          checksum);
    return cudaGetLastError();
}

cudaError_t read_probe_error(int *out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_probe_error, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_probe_error, &zero, sizeof(int));
    }
    return e;
}

} // namespace smla
