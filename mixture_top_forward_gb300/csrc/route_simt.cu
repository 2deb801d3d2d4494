// Stage 3: routing, CUDA-core version.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造": each query picks the expert of
// the landmark query it matches best (one expert per query, s = 1), reusing
// the query-to-landmark logits: e(n) = argmax_i tau <q_n, Lq_i>, ties to the
// lowest i.
//
// One thread per query, 256 queries per CTA; the landmark queries stream
// through shared memory in tiles of 128 (fp32, read as broadcasts). The CTA
// also counts its queries per expert in shared memory and adds the counts to
// the per-head histogram used by the grouping step.
#include "mita_internal.cuh"

namespace mita {

namespace {

constexpr int RT = 256;  // queries (threads) per CTA
constexpr int LTILE = 128;

__global__ void __launch_bounds__(RT) route_simt_kernel(const __nv_bfloat16* __restrict__ Q, int64_t N, int m,
                                                        int64_t nblocks, const float* __restrict__ lq32,
                                                        int32_t* __restrict__ route, int* __restrict__ counts) {
    __shared__ __align__(16) float Ls[LTILE][D];
    __shared__ int sh[MITA_MAX_M_INTERNAL];
    const int64_t blk = blockIdx.x % nblocks;
    const int64_t bh = blockIdx.x / nblocks;
    const int64_t n = blk * RT + threadIdx.x;
    const bool valid = n < N;
    for (int e = threadIdx.x; e < m; e += RT) sh[e] = 0;

    float q[D];
    {
        const __nv_bfloat16* qr = Q + (bh * N + (valid ? n : 0)) * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) unpack_bf16x8(ldg_nc_v4(qr + c), q + c);
    }
    float best = -INFINITY;
    int arg = 0;
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
            if (t > best) {
                best = t;
                arg = i0 + ii;
            }
        }
    }
    if (valid) {
        route[bh * N + n] = arg;
        atomicAdd(&sh[arg], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < m; e += RT)
        if (sh[e]) atomicAdd(&counts[bh * m + e], sh[e]);
}

}  // namespace

cudaError_t launch_route_simt(const Plan& p, const Work& w, const __nv_bfloat16* Q, int32_t* route, cudaStream_t st) {
    const int64_t nblocks = (p.s.N + RT - 1) / RT;
    const unsigned grid = static_cast<unsigned>(p.s.BH * nblocks);
    route_simt_kernel<<<grid, RT, 0, st>>>(Q, p.s.N, p.s.m, nblocks, w.lq32, route, w.counts);
    return cudaGetLastError();
}

}  // namespace mita
