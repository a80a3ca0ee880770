// S4: token -> expert permutation (histogram, exclusive prefix sum, stable
// scatter), deterministic: inside one expert the pairs p = t*k + j keep their
// order, which is token order because a token picks an expert at most once.
//
// A pair the route-tail skip dropped has expert -1: it gets no position
// (inv = -1) and is left out of the counts.
//
// Small calls (P <= 1024 pairs, every decode batch): one CTA does all of it.
// Large calls: per-chunk histograms (1024 pairs per CTA, shared-memory
// atomics), one CTA turns them into expert offsets and per-chunk bases (for
// long chunk lists through sums over groups of chunks, so that no thread runs
// down a whole column), then each chunk scatters its pairs with warp
// match/popc ranks in pair order, from a shared-memory copy of its expert ids.
// No global atomics decide any position.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Exclusive scan over the 1024 threads of a block; also returns the total.
__device__ int block_exclusive_scan_1024(int v, int& total) {
    __shared__ int warp_off[32];
    __shared__ int grand;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_off[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int t = warp_off[lane];
        int ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += n;
        }
        warp_off[lane] = ti - t;
        if (lane == 31) grand = ti;
    }
    __syncthreads();
    const int excl = incl - v + warp_off[warp];
    total = grand;
    __syncthreads();
    return excl;
}

// Writes counts/offsets/active from per-expert totals held one per thread.
__device__ void finish_offsets(int e, int E, int total_e, int32_t* counts, int32_t* offsets,
                               int32_t* active, uint32_t* scal, int& off_e) {
    int all;
    off_e = block_exclusive_scan_1024(e < E ? total_e : 0, all);
    int nact;
    const int apos = block_exclusive_scan_1024(e < E && total_e > 0 ? 1 : 0, nact);
    if (e < E) {
        counts[e] = total_e;
        offsets[e] = off_e;
        if (total_e > 0) active[apos] = e;
    }
    if (threadIdx.x == 0) {
        offsets[E] = all;
        scal[kScalActive] = (uint32_t)nact;
    }
}

// Scatter pairs [p0, p1) in order; run[e] holds the next free position of e.
// idx holds the experts of pairs p0 .. p1 - 1 (idx[0] is pair p0's).  With
// wperm, each position also gets its pair's router weight (w[0] is pair p0's).
__device__ void warp_scatter(const int32_t* idx, int p0, int p1, int* run,
                             int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                             const float* w, float* __restrict__ wperm) {
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    for (int base = p0; base < p1; base += 32) {
        const int p = base + lane;
        const int e = p < p1 ? idx[p - p0] : -1;
        const float wp = wperm && p < p1 ? w[p - p0] : 0.0f;
        const uint32_t same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lt);
        int pos = 0;
        if (e >= 0) pos = run[e] + rank;
        __syncwarp();
        if (e >= 0 && rank == 0) run[e] += __popc(same);
        __syncwarp();
        if (e >= 0) {
            perm[pos] = p;
            inv[p] = pos;
            if (wperm) wperm[pos] = wp;
        } else if (p < p1) {
            inv[p] = -1;
        }
    }
}

__global__ void __launch_bounds__(1024) k_perm_small(const int32_t* __restrict__ idx, int P, int E,
                                                     int32_t* counts, int32_t* offsets,
                                                     int32_t* active, uint32_t* scal,
                                                     int32_t* perm, int32_t* inv,
                                                     const float* w, float* wperm) {
    __shared__ int cnt[1024];
    const int e = threadIdx.x;
    cnt[e] = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int ep = idx[p];
        if (ep >= 0) atomicAdd(&cnt[ep], 1);
    }
    __syncthreads();
    const int tot = e < E ? cnt[e] : 0;
    int off_e;
    finish_offsets(e, E, tot, counts, offsets, active, scal, off_e);
    __syncthreads();
    if (e < E) cnt[e] = off_e;
    __syncthreads();
    if (threadIdx.x < 32) warp_scatter(idx, 0, P, cnt, perm, inv, w, wperm);
}

__global__ void __launch_bounds__(256) k_perm_count(const int32_t* __restrict__ idx, int P, int E,
                                                    int32_t* __restrict__ chunk_cnt) {
    __shared__ int hist[1024];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int p0 = blockIdx.x * kPermChunk, p1 = min(P, p0 + kPermChunk);
    for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const int ep = idx[p];
        if (ep >= 0) atomicAdd(&hist[ep], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_cnt[(size_t)blockIdx.x * E + e] = hist[e];
}

// Group sums: group_cnt[g][e] = sum of chunk_cnt[c][e] over the chunks c of
// group g (one CTA per group).
__global__ void __launch_bounds__(256) k_perm_group_sum(int nchunks, int E, const int32_t* __restrict__ chunk_cnt,
                                                        int32_t* __restrict__ group_cnt) {
    const int c0 = blockIdx.x * kPermGroup, c1 = min(nchunks, c0 + kPermGroup);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int n[kPermGroup];
#pragma unroll
        for (int u = 0; u < kPermGroup; ++u) n[u] = c0 + u < c1 ? chunk_cnt[(size_t)(c0 + u) * E + e] : 0;
        int tot = 0;
#pragma unroll
        for (int u = 0; u < kPermGroup; ++u) tot += n[u];
        group_cnt[(size_t)blockIdx.x * E + e] = tot;
    }
}

// Chunk bases from the group bases: chunk c of group g starts expert e at
// group_cnt[g][e] plus the counts of the group's earlier chunks.
__global__ void __launch_bounds__(256) k_perm_group_base(int nchunks, int E, int32_t* __restrict__ chunk_cnt,
                                                         const int32_t* __restrict__ group_cnt) {
    const int c0 = blockIdx.x * kPermGroup, c1 = min(nchunks, c0 + kPermGroup);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int n[kPermGroup];
#pragma unroll
        for (int u = 0; u < kPermGroup; ++u) n[u] = c0 + u < c1 ? chunk_cnt[(size_t)(c0 + u) * E + e] : 0;
        int run = group_cnt[(size_t)blockIdx.x * E + e];
#pragma unroll
        for (int u = 0; u < kPermGroup; ++u) {
            if (c0 + u < c1) chunk_cnt[(size_t)(c0 + u) * E + e] = run;
            run += n[u];
        }
    }
}

// Expert totals and offsets from the rows of cnt ([nrows][E]: the chunks'
// histograms, or the groups' sums), then each row turned into its exclusive
// base (expert offset plus the earlier rows' counts).
__global__ void __launch_bounds__(1024) k_perm_scan(int nchunks, int E, int32_t* chunk_cnt,
                                                    int32_t* counts, int32_t* offsets,
                                                    int32_t* active, uint32_t* scal) {
    const int e = threadIdx.x;
    int tot = 0;
    if (e < E) {
#pragma unroll 8
        for (int c = 0; c < nchunks; ++c) tot += chunk_cnt[(size_t)c * E + e];
    }
    int off_e;
    finish_offsets(e, E, tot, counts, offsets, active, scal, off_e);
    if (e < E) {
        // exclusive running sum down the column, eight loads in flight at a
        // time so the chain of dependent adds does not wait on each load
        int run = off_e;
        int c = 0;
        for (; c + 8 <= nchunks; c += 8) {
            int n[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) n[u] = chunk_cnt[(size_t)(c + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                chunk_cnt[(size_t)(c + u) * E + e] = run;
                run += n[u];
            }
        }
        for (; c < nchunks; ++c) {
            const int n = chunk_cnt[(size_t)c * E + e];
            chunk_cnt[(size_t)c * E + e] = run;
            run += n;
        }
    }
}

__global__ void __launch_bounds__(32) k_perm_scatter(const int32_t* __restrict__ idx, int P, int E,
                                                     const int32_t* __restrict__ chunk_base,
                                                     int32_t* __restrict__ perm,
                                                     int32_t* __restrict__ inv,
                                                     const float* __restrict__ w,
                                                     float* __restrict__ wperm) {
    __shared__ int run[1024];
    __shared__ __align__(16) int32_t sidx[kPermChunk];
    __shared__ __align__(16) float sw[kPermChunk];
    const int p0 = blockIdx.x * kPermChunk, p1 = min(P, p0 + kPermChunk);
    // the chunk's expert ids (and router weights) first, all loads in flight
    // at once (16-byte loads where the chunk is whole and idx, w 16-byte aligned)
    const bool vec = p1 - p0 == kPermChunk && (reinterpret_cast<uintptr_t>(idx) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(w) & 15u) == 0;
    if (vec) {
        const int4* src = reinterpret_cast<const int4*>(idx + p0);
        const float4* wsrc = reinterpret_cast<const float4*>(w + p0);
#pragma unroll
        for (int i = 0; i < kPermChunk / 128; ++i) {
            reinterpret_cast<int4*>(sidx)[threadIdx.x + 32 * i] = src[threadIdx.x + 32 * i];
            if (wperm) reinterpret_cast<float4*>(sw)[threadIdx.x + 32 * i] = wsrc[threadIdx.x + 32 * i];
        }
    } else {
        for (int p = p0 + threadIdx.x; p < p1; p += 32) {
            sidx[p - p0] = idx[p];
            if (wperm) sw[p - p0] = w[p];
        }
    }
    for (int e = threadIdx.x; e < E; e += 32) run[e] = chunk_base[(size_t)blockIdx.x * E + e];
    __syncwarp();
    warp_scatter(sidx, p0, p1, run, perm, inv, sw, wperm);
}

}  // namespace

cudaError_t launch_permute(const int32_t* idx, int T, const Shape& s, const Workspace& ws,
                           cudaStream_t st) {
    const int P = T * s.k;
    if (P <= kPermChunk) {
        k_perm_small<<<1, 1024, 0, st>>>(idx, P, s.E, ws.counts, ws.offsets, ws.active, ws.scal,
                                         ws.perm, ws.inv, ws.w, ws.wperm);
        count_launches(1);
        return cudaGetLastError();
    }
    const int nchunks = (P + kPermChunk - 1) / kPermChunk;
    const int ngroups = perm_groups(nchunks);
    if (ngroups > 0 && ws.group_cnt == nullptr) return cudaErrorInvalidValue;
    k_perm_count<<<nchunks, 256, 0, st>>>(idx, P, s.E, ws.chunk_cnt);
    if (ngroups > 0) {
        k_perm_group_sum<<<ngroups, 256, 0, st>>>(nchunks, s.E, ws.chunk_cnt, ws.group_cnt);
        k_perm_scan<<<1, 1024, 0, st>>>(ngroups, s.E, ws.group_cnt, ws.counts, ws.offsets, ws.active,
                                        ws.scal);
        k_perm_group_base<<<ngroups, 256, 0, st>>>(nchunks, s.E, ws.chunk_cnt, ws.group_cnt);
    } else {
        k_perm_scan<<<1, 1024, 0, st>>>(nchunks, s.E, ws.chunk_cnt, ws.counts, ws.offsets, ws.active,
                                        ws.scal);
    }
    k_perm_scatter<<<nchunks, 32, 0, st>>>(idx, P, s.E, ws.chunk_cnt, ws.perm, ws.inv, ws.w, ws.wperm);
    count_launches(ngroups > 0 ? 5 : 3);
    return cudaGetLastError();
}

}  // namespace moe
