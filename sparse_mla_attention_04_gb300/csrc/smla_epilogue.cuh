// Epilogue shared by the sparse MLA forward kernels: a CTA that owns one
// (row t, 16-head group, split s) has staged its normalised partial output
// o_s [16 heads][512] (fp32) and lse_s [16] in shared memory; this writes the
// final bf16 out and lse. With one split it stores directly. With up to
// kClusterMaxSplits splits the row's CTAs form one thread-block cluster and
// each merges a slice of the tile from every split's staging through
// distributed shared memory (LSE weights). With more splits the partials go
// to the workspace and the split that draws the last ticket (one atomic; no
// spinning) merges them.
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

    // ---- many splits: (o_j, lse_j) to the workspace, then take a ticket ----
    float *po = a.part_o + (((int64_t)t * a.S + s) * a.H + hbase) * kDv;
    for (int e = tid; e < kHeads * kDv / 4; e += kThreads)
        __stcg(reinterpret_cast<float4 *>(po) + e, reinterpret_cast<const float4 *>(ost)[e]);
    if (tid < kHeads)
        __stcg(a.part_lse + ((int64_t)t * a.S + s) * a.H + hbase + tid, lse_s[tid]);
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

    // ---- last CTA of the row: LSE merge of the S partials ----
    if (tid < kHeads) {
        const float sk = sink(tid);
        float mx = sk;
        for (int j = 0; j < a.S; ++j)
            mx = fmaxf(mx, __ldcg(a.part_lse + ((int64_t)t * a.S + j) * a.H + hbase + tid));
        float tot = (mx == -INFINITY || sk == -INFINITY) ? 0.f : expf(sk - mx); // the sink: no output
        for (int j = 0; j < a.S; ++j) {
            const float lj = __ldcg(a.part_lse + ((int64_t)t * a.S + j) * a.H + hbase + tid);
            const float e = (mx == -INFINITY) ? 0.f : expf(lj - mx);
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
    for (int e = tid; e < kHeads * kDv / 4; e += kThreads) {
        const int h = e / (kDv / 4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < a.S; ++j) {
            const float w = wts[j * kHeads + h];
            const float4 x = (j == s) ? reinterpret_cast<const float4 *>(ost)[e]
                                      : __ldcg(reinterpret_cast<const float4 *>(
                                                   a.part_o + (((int64_t)t * a.S + j) * a.H + hbase) * kDv) +
                                               e);
            acc.x += w * x.x;
            acc.y += w * x.y;
            acc.z += w * x.z;
            acc.w += w * x.w;
        }
        uint2 u;
        u.x = pack_bf16x2(acc.x, acc.y);
        u.y = pack_bf16x2(acc.z, acc.w);
        *reinterpret_cast<uint2 *>(out + (int64_t)e * 4) = u;
    }
}


} // namespace smla
