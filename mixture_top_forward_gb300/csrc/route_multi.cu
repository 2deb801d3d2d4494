// Stage 3 with s routed experts per query (s > 1), CUDA-core version.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), end of section
// "MiTA：用少量地标查询，同时完成压缩与专家构造": the pages run what they call the
// s = 1 configuration (one routed expert per query) and leave the general
// form undescribed. Here a query takes the s landmarks with the highest
// logits tau <q_n, Lq_i>, highest first, ties to the lower landmark index
// (s = 1 is the argmax of the one-expert routing kernels).
//
// One thread per query, 256 queries per CTA; the landmark queries stream
// through shared memory in tiles of 32 rows (fp32, read as broadcasts). The
// s best (logit, landmark) pairs stay in registers as a list sorted by
// descending logit. Each CTA counts its queries per (rank j, expert) in
// shared memory and adds the counts to the per-rank expert counts that the
// grouping of rank j consumes.
#include "mita_internal.cuh"

namespace mita {

namespace {

constexpr int RT = 256;    // queries (threads) per CTA
constexpr int LTILE = 32;  // landmark rows per staged tile

__global__ void __launch_bounds__(RT) route_multi_kernel(const __nv_bfloat16* __restrict__ Q, int64_t N, int m,
                                                         int s, int64_t nblocks, int64_t BH,
                                                         const float* __restrict__ lq32, int32_t* __restrict__ route,
                                                         int* __restrict__ counts) {
    __shared__ __align__(16) float Ls[LTILE][D];
    __shared__ int sh[MITA_MAX_S][MITA_MAX_M_INTERNAL];
    const int64_t blk = blockIdx.x % nblocks;
    const int64_t bh = blockIdx.x / nblocks;
    const int64_t n = blk * RT + threadIdx.x;
    const bool valid = n < N;
    for (int x = threadIdx.x; x < s * m; x += RT) sh[x / m][x % m] = 0;

    float q[D];
    {
        const __nv_bfloat16* qr = Q + (bh * N + (valid ? n : 0)) * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) unpack_bf16x8(ldg_nc_v4(qr + c), q + c);
    }
    // bv/bi: the best s so far, by descending logit; the placeholder indices
    // are distinct so that the result stays a valid set whatever the logits
    float bv[MITA_MAX_S];
    int bi[MITA_MAX_S];
#pragma unroll
    for (int u = 0; u < MITA_MAX_S; ++u) {
        bv[u] = -INFINITY;
        bi[u] = u;
    }
    float thr = -INFINITY;  // the s-th best logit so far
    for (int i0 = 0; i0 < m; i0 += LTILE) {
        const int nt = min(LTILE, m - i0);
        __syncthreads();
        for (int t = threadIdx.x; t < nt * D; t += RT) Ls[t / D][t % D] = lq32[(bh * m + i0) * D + t];
        __syncthreads();
        for (int ii = 0; ii < nt; ++ii) {
            const float4* lr = reinterpret_cast<const float4*>(Ls[ii]);
            float dot = 0.f;
#pragma unroll
            for (int c4 = 0; c4 < D / 4; ++c4) {
                const float4 a = lr[c4];
                dot = fmaf(q[4 * c4], a.x, dot);
                dot = fmaf(q[4 * c4 + 1], a.y, dot);
                dot = fmaf(q[4 * c4 + 2], a.z, dot);
                dot = fmaf(q[4 * c4 + 3], a.w, dot);
            }
            const float t = dot * 0.125f;
            if (t > thr) {
                // insert before the first strictly smaller entry (landmarks
                // arrive in index order, so equal logits keep the lower index
                // first), shifting the rest down by one
                float cv = t;
                int ci = i0 + ii;
                bool moved = false;
#pragma unroll
                for (int u = 0; u < MITA_MAX_S; ++u) {
                    if (u < s && (moved || cv > bv[u])) {
                        const float tv = bv[u];
                        const int ti = bi[u];
                        bv[u] = cv;
                        bi[u] = ci;
                        cv = tv;
                        ci = ti;
                        moved = true;
                    }
                }
#pragma unroll
                for (int u = 0; u < MITA_MAX_S; ++u)
                    if (u == s - 1) thr = bv[u];
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int u = 0; u < MITA_MAX_S; ++u) {
            if (u < s) {
                const int r = min(max(bi[u], 0), m - 1);
                route[(bh * N + n) * s + u] = r;
                atomicAdd(&sh[u][r], 1);
            }
        }
    }
    __syncthreads();
    for (int x = threadIdx.x; x < s * m; x += RT) {
        const int j = x / m, e = x % m;
        if (sh[j][e]) atomicAdd(&counts[(j * BH + bh) * m + e], sh[j][e]);
    }
}

}  // namespace

cudaError_t launch_route_multi(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route,
                               cudaStream_t st) {
    const int64_t nblocks = (p.s.N + RT - 1) / RT;
    const unsigned grid = static_cast<unsigned>(p.s.BH * nblocks);
    route_multi_kernel<<<grid, RT, 0, st>>>(Q, p.s.N, p.s.m, p.s.s_route, nblocks, p.s.BH, w.lq32, route, w.counts);
    return cudaGetLastError();
}

}  // namespace mita
