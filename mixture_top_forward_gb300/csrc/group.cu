// Grouping queries by expert: a counting sort on the routes.
//
// The pages process queries grouped by expert so that every query of one
// routed expert shares the same gathered keys and values
// ("NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), end of section
// "MiTA：用少量地标查询，同时完成压缩与专家构造"; Algorithm 1 caption of
// "And attention is also FFN? …" (en.roboind.com)).
//
//  1. the routing kernel has already counted queries per (head, expert);
//  2. offsets_kernel (one CTA per head): exclusive scan of the counts gives
//     each expert's segment of `perm`; it also cuts every segment into work
//     items (expert, start, length <= qtile, head) for the attention kernel,
//     appended to one flat list: each head reserves its range with one global
//     atomic, and keeps its items in expert order inside it;
//  3. scatter_kernel (one CTA per 4096 queries of a head): counts its queries
//     per expert in shared memory, reserves a range of each expert's segment
//     with one global atomic per (CTA, expert), and writes the query indices
//     there (each expert's queries of the CTA land contiguously).
// The order of queries inside a segment depends on CTA timing; it does not
// affect any result, because every query's attention is computed on its own.
#include "mita_internal.cuh"

namespace mita {

namespace {

constexpr int GT = 1024;  // threads of the offsets kernel (>= MITA_MAX_M_INTERNAL)
constexpr int SCT = 1024;  // threads per scatter CTA
constexpr int SQT = 4;     // queries per scatter thread

__global__ void __launch_bounds__(GT) offsets_kernel(int m, int64_t N, int qtile, int* __restrict__ counts,
                                                     int* __restrict__ expoff, int* __restrict__ cursor,
                                                     int4* __restrict__ items, int* __restrict__ nitems) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    __shared__ int sc[GT];
    __shared__ int st[GT];
    __shared__ int base;
    const int64_t bh = blockIdx.x;
    const int e = threadIdx.x;
    const int c = e < m ? counts[bh * m + e] : 0;
    const int tiles = (c + qtile - 1) / qtile;
    sc[e] = c;
    st[e] = tiles;
    __syncthreads();
    for (int o = 1; o < GT; o <<= 1) {  // inclusive Hillis-Steele scans
        const int a = e >= o ? sc[e - o] : 0;
        const int b = e >= o ? st[e - o] : 0;
        __syncthreads();
        sc[e] += a;
        st[e] += b;
        __syncthreads();
    }
    if (e == m - 1) {
        expoff[bh * (m + 1) + m] = sc[e];
        base = atomicAdd(nitems, st[e]);
    }
    __syncthreads();
    if (e < m) {
        const int off = sc[e] - c;
        expoff[bh * (m + 1) + e] = off;
        cursor[bh * m + e] = off;
        counts[bh * m + e] = 0;  // ready for the next call
        const int ib = base + st[e] - tiles;
        for (int t = 0; t < tiles; ++t) {
            const int start = t * qtile;
            items[ib + t] = make_int4(e, off + start, min(qtile, c - start), static_cast<int>(bh));
        }
    }
}

__global__ void __launch_bounds__(SCT) scatter_kernel(const int32_t* __restrict__ route, int64_t N, int m, int s,
                                                      int j, int64_t nblocks, int* __restrict__ cursor,
                                                      int* __restrict__ perm) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    __shared__ int sh[MITA_MAX_M_INTERNAL];
    const int64_t blk = blockIdx.x % nblocks;
    const int64_t bh = blockIdx.x / nblocks;
    for (int e = threadIdx.x; e < m; e += SCT) sh[e] = 0;
    __syncthreads();
    // query n0 + u * SCT (u < SQT): consecutive threads read consecutive routes
    const int64_t n0 = blk * (SCT * SQT) + threadIdx.x;
    int e[SQT], rank[SQT];
#pragma unroll
    for (int u = 0; u < SQT; ++u) e[u] = n0 + u * SCT < N ? route[(bh * N + n0 + u * SCT) * s + j] : -1;
#pragma unroll
    for (int u = 0; u < SQT; ++u) rank[u] = e[u] >= 0 ? atomicAdd(&sh[e[u]], 1) : 0;
    __syncthreads();
    for (int x = threadIdx.x; x < m; x += SCT)
        if (sh[x]) sh[x] = atomicAdd(&cursor[bh * m + x], sh[x]);
    __syncthreads();
#pragma unroll
    for (int u = 0; u < SQT; ++u)
        if (e[u] >= 0) perm[bh * N + sh[e[u]] + rank[u]] = static_cast<int>(n0 + u * SCT);
}

}  // namespace

// Groups the queries by the j-th entry of their routes (route is [BH][N][s];
// s = 1, j = 0 for one expert per query) into plane j of perm and items.
cudaError_t launch_group(const Plan& p, const Work& w, const int32_t* route, int j, cudaStream_t st) {
    const size_t mrows = static_cast<size_t>(p.s.BH) * p.s.m;
    int* perm = w.perm + static_cast<size_t>(j) * p.s.BH * p.s.N;
    int4* items = w.items + static_cast<size_t>(j) * p.s.BH * p.max_items;
    cudaError_t e = launch_dep(offsets_kernel, dim3(static_cast<unsigned>(p.s.BH)), dim3(GT), 0, st, p.s.m, p.s.N,
                               p.qtile, w.counts + j * mrows, w.expoff, w.cursor, items, w.nitems + j);
    if (e != cudaSuccess) return e;
    const int64_t nblocks = (p.s.N + SCT * SQT - 1) / (SCT * SQT);
    return launch_dep(scatter_kernel, dim3(static_cast<unsigned>(p.s.BH * nblocks)), dim3(SCT), 0, st, route, p.s.N,
                      p.s.m, p.s.s_route, j, nblocks, w.cursor, perm);
}

}  // namespace mita
