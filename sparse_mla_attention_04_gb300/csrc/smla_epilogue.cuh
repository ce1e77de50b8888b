// Epilogue shared by the sparse MLA forward kernels: a CTA that owns one
// (row t, 16-head group, split s) has staged its normalised partial output
// o_s [16 heads][512] (fp32) and lse_s [16] in shared memory; this writes the
// final bf16 out and lse. With one split it stores directly. With up to
// kClusterMaxSplits splits the row's CTAs form one thread-block cluster and
// each merges a slice of the tile from every split's staging through
// distributed shared memory (LSE weights). With more splits the partials go
// to the workspace in binary16 and the split that draws the last ticket (one
// atomic; no spinning) merges them, summing the splits in index order from
// the same binary16 values whichever split that is.
//
// Attention sinks: a per-head sink logit (natural-log units, like the lse)
// joins the softmax denominator once per row: with one split the staged
// output is scaled by 1 / (1 + e^{sink - lse}) and the lse becomes
// log(e^lse + e^sink); with several, the sink enters the merge's total as a
// partial with no output.
#pragma once

#include "smla_device.cuh"
#include "smla_internal.h"

#include <cooperative_groups.h>

namespace smla {

template <int kThreads>
__device__ __forceinline__ void finish_tile(const FwdArgs &a, float *ost, const float *lse_s, float *wts,
                                            int *flag_s, int t, int hg, int s, int tid)
{
    namespace cg = cooperative_groups;
    constexpr int kHeads = 16;
    constexpr int kDv = 512;
    const int G = a.H / kHeads;
    const int hbase = hg * kHeads;
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((int64_t)t * a.H + hbase) * kDv;
    // the row's sink logit of head `h` of this group (-inf: none)
    auto sink = [&](int h) { return a.sinks != nullptr ? a.sinks[hbase + h] : -INFINITY; };
    if (a.S == 1) {
        if (a.sinks != nullptr) {
            if (tid < kHeads) {
                const float l = lse_s[tid], sk = sink(tid);
                const float M = fmaxf(l, sk);
                // e^lse / (e^lse + e^sink), and the lse with the sink
                const float el = l == -INFINITY ? 0.f : expf(l - M), es = sk == -INFINITY ? 0.f : expf(sk - M);
                wts[tid] = el + es > 0.f ? el / (el + es) : 0.f;
                if (a.lse != nullptr)
                    a.lse[(int64_t)t * a.H + hbase + tid] = M == -INFINITY ? -INFINITY : M + logf(el + es);
            }
            __syncthreads();
        }
        for (int e = tid; e < kHeads * kDv / 8; e += kThreads) {
            const int h = e / (kDv / 8), d = (e % (kDv / 8)) * 8;
            const float f = a.sinks != nullptr ? wts[h] : 1.0f;
            const float4 x = *reinterpret_cast<const float4 *>(ost + h * kDv + d);
            const float4 y = *reinterpret_cast<const float4 *>(ost + h * kDv + d + 4);
            uint4 u;
            u.x = pack_bf16x2(x.x * f, x.y * f);
            u.y = pack_bf16x2(x.z * f, x.w * f);
            u.z = pack_bf16x2(y.x * f, y.y * f);
            u.w = pack_bf16x2(y.z * f, y.w * f);
            *reinterpret_cast<uint4 *>(out + (int64_t)h * kDv + d) = u;
        }
        if (a.sinks == nullptr && a.lse != nullptr && tid < kHeads)
            a.lse[(int64_t)t * a.H + hbase + tid] = lse_s[tid];
        return;
    }

    if (a.S <= kClusterMaxSplits) {
        // ---- the row's S splits form one cluster: merge through DSMEM ----
        cg::cluster_group cluster = cg::this_cluster();
        const int rank = (int)cluster.block_rank(); // == s
        cluster.sync(); // every split's staged o and lse are visible cluster-wide
        if (tid < kHeads) {
            // every split's lse in one round of remote loads
            float lj[kClusterMaxSplits];
#pragma unroll
            for (int j = 0; j < kClusterMaxSplits; ++j)
                lj[j] = j < a.S ? *cluster.map_shared_rank(lse_s + tid, j) : -INFINITY;
            const float sk = sink(tid);
            float mx = sk;
#pragma unroll
            for (int j = 0; j < kClusterMaxSplits; ++j)
                mx = fmaxf(mx, lj[j]);
            float tot = (mx == -INFINITY || sk == -INFINITY) ? 0.f : expf(sk - mx); // the sink: no output
#pragma unroll
            for (int j = 0; j < kClusterMaxSplits; ++j) {
                lj[j] = (mx == -INFINITY || j >= a.S) ? 0.f : expf(lj[j] - mx);
                tot += lj[j];
            }
            const float inv = tot > 0.f ? 1.0f / tot : 0.f;
#pragma unroll
            for (int j = 0; j < kClusterMaxSplits; ++j)
                if (j < a.S)
                    wts[j * kHeads + tid] = lj[j] * inv;
            if (rank == 0 && a.lse != nullptr)
                a.lse[(int64_t)t * a.H + hbase + tid] = (mx == -INFINITY) ? -INFINITY : mx + logf(tot);
        }
        __syncthreads();
        // this CTA writes a contiguous share of the 16 x 512 tile; each thread
        // takes kU float4 elements and issues their remote loads together
        constexpr int E4 = kHeads * kDv / 4;
        constexpr int kU = 4;
        const int chunk = (E4 + a.S - 1) / a.S;
        const int e_beg = rank * chunk, e_end = min(E4, (rank + 1) * chunk);
        for (int e0 = e_beg + tid; e0 < e_end; e0 += kU * kThreads) {
            float4 acc[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u)
                acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < a.S; ++j) {
                // this CTA's own partial from its shared memory, the others' through DSMEM
                const float4 *src = j == rank ? reinterpret_cast<const float4 *>(ost)
                                              : cluster.map_shared_rank(reinterpret_cast<const float4 *>(ost), j);
                float4 x[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int e = e0 + u * kThreads;
                    x[u] = e < e_end ? src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int e = e0 + u * kThreads;
                    const float w = wts[j * kHeads + min(e, E4 - 1) / (kDv / 4)];
                    acc[u].x += w * x[u].x;
                    acc[u].y += w * x[u].y;
                    acc[u].z += w * x[u].z;
                    acc[u].w += w * x[u].w;
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int e = e0 + u * kThreads;
                if (e < e_end) {
                    uint2 v;
                    v.x = pack_bf16x2(acc[u].x, acc[u].y);
                    v.y = pack_bf16x2(acc[u].z, acc[u].w);
                    *reinterpret_cast<uint2 *>(out + (int64_t)e * 4) = v;
                }
            }
        }
        cluster.sync(); // keep this CTA's staging alive until every peer has read it
        return;
    }

    // ---- many splits: (o_s, lse_s) to the workspace (o_s in binary16), then
    // take a ticket; the split that draws the row's last ticket merges (no
    // split waits for another: more splits than a cluster holds need not be
    // co-resident).
    const int64_t rowbase = (int64_t)t * a.S;
    uint4 *po = reinterpret_cast<uint4 *>(a.part_o16 + ((rowbase + s) * a.H + hbase) * kDv);
    for (int e = tid; e < kHeads * kDv / 8; e += kThreads) {
        const float4 x = reinterpret_cast<const float4 *>(ost)[2 * e];
        const float4 y = reinterpret_cast<const float4 *>(ost)[2 * e + 1];
        uint4 u;
        u.x = pack_f16x2(x.x, x.y);
        u.y = pack_f16x2(x.z, x.w);
        u.z = pack_f16x2(y.x, y.y);
        u.w = pack_f16x2(y.z, y.w);
        __stcg(po + e, u);
    }
    if (tid < kHeads)
        __stcg(a.part_lse + (rowbase + s) * a.H + hbase + tid, lse_s[tid]);
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int *tk = a.tickets + (int64_t)t * G + hg;
        const int ticket = atomicAdd(tk, 1);
        const int last = (ticket == a.S - 1);
        if (last)
            *tk = 0; // every split of this row has arrived: reset for the next call
        *flag_s = last;
    }
    __syncthreads();
    if (!*flag_s)
        return;
    __threadfence();

    // ---- last split of the row: LSE merge of the S partials ----
    // every split's lse (loaded in parallel), then the weights per (split, head)
    for (int i = tid; i < a.S * kHeads; i += kThreads)
        wts[i] = __ldcg(a.part_lse + (rowbase + i / kHeads) * a.H + hbase + i % kHeads);
    __syncthreads();
    if (tid < kHeads) {
        const float sk = sink(tid);
        float mx = sk;
        for (int j = 0; j < a.S; ++j)
            mx = fmaxf(mx, wts[j * kHeads + tid]);
        float tot = (mx == -INFINITY || sk == -INFINITY) ? 0.f : expf(sk - mx); // the sink: no output
        for (int j = 0; j < a.S; ++j) {
            const float e = (mx == -INFINITY) ? 0.f : expf(wts[j * kHeads + tid] - mx);
            wts[j * kHeads + tid] = e;
            tot += e;
        }
        const float inv = tot > 0.f ? 1.0f / tot : 0.f;
        for (int j = 0; j < a.S; ++j)
            wts[j * kHeads + tid] *= inv;
        if (a.lse != nullptr)
            a.lse[(int64_t)t * a.H + hbase + tid] = (mx == -INFINITY) ? -INFINITY : mx + logf(tot);
    }
    __syncthreads();
    // groups of 8 values; a thread takes kU groups and, two splits at a time,
    // issues all their loads before accumulating. This split's own partial is
    // rounded to binary16 from shared memory, exactly as the others stored
    // theirs, and the splits are summed in index order: whichever split merges,
    // the result is the same bits.
    constexpr int E8 = kHeads * kDv / 8;
    constexpr int kU = 4;
    const uint4 *pall = reinterpret_cast<const uint4 *>(a.part_o16 + (rowbase * a.H + hbase) * kDv);
    const int64_t split_stride = (int64_t)a.H * kDv / 8; // uint4 per split
    auto own16 = [&](int e) {
        const float4 x = reinterpret_cast<const float4 *>(ost)[2 * e];
        const float4 y = reinterpret_cast<const float4 *>(ost)[2 * e + 1];
        return make_uint4(pack_f16x2(x.x, x.y), pack_f16x2(x.z, x.w), pack_f16x2(y.x, y.y), pack_f16x2(y.z, y.w));
    };
    for (int e0 = tid; e0 < E8; e0 += kU * kThreads) {
        float acc[kU][8];
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
            for (int c = 0; c < 8; ++c)
                acc[u][c] = 0.f;
        for (int j0 = 0; j0 < a.S; j0 += 2) {
            uint4 raw[2][kU];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = j0 + jj;
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int e = e0 + u * kThreads;
                    raw[jj][u] = (j >= a.S || e >= E8) ? make_uint4(0u, 0u, 0u, 0u)
                                 : (j == s)              ? own16(e)
                                                         : __ldcg(pall + j * split_stride + e);
                }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int j = j0 + jj;
                if (j >= a.S)
                    continue;
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int e = min(e0 + u * kThreads, E8 - 1);
                    const float w = wts[j * kHeads + e / (kDv / 8)];
                    const uint32_t q[4] = {raw[jj][u].x, raw[jj][u].y, raw[jj][u].z, raw[jj][u].w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&q[c]));
                        acc[u][2 * c] += w * f.x;
                        acc[u][2 * c + 1] += w * f.y;
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int e = e0 + u * kThreads;
            if (e < E8) {
                uint4 v;
                v.x = pack_bf16x2(acc[u][0], acc[u][1]);
                v.y = pack_bf16x2(acc[u][2], acc[u][3]);
                v.z = pack_bf16x2(acc[u][4], acc[u][5]);
                v.w = pack_bf16x2(acc[u][6], acc[u][7]);
                *reinterpret_cast<uint4 *>(out + (int64_t)e * 8) = v;
            }
        }
    }
}


} // namespace smla
