// Stage 2: the landmark scan, CUDA-core version.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造": every landmark query is matched
// against all keys; its k best keys form its routed expert, and the same
// landmark's cross-attention over the whole context gives its shared-expert
// value. One pass over K and V serves both: s = tau <Lq_i, K_j> feeds an
// online softmax (max, sum, sum p V) and the streaming top-k filter of
// topk.cuh.
//
// Grid: one CTA per (head, key chunk, tile of 32 landmarks), landmark tile
// fastest so CTAs of one chunk run together and share K/V through L2.
// 8 warps x 4 landmarks each. Per 32-key step the CTA stages K (transposed)
// and V in fp32 shared memory; lane j scores key j, lane l accumulates
// output dims 2l, 2l+1. Scores use the fp32 landmark queries, so they are
// exact up to fp32 accumulation. Each (head, chunk, landmark) leaves a
// softmax partial (max, sum, o[64]) and a candidate buffer; select.cu merges
// them.
#include "topk.cuh"

namespace mita {

namespace {

constexpr int SW = 8;             // warps per CTA
constexpr int LPW = 4;            // landmarks per warp
constexpr int LT = SW * LPW;      // landmarks per CTA
constexpr int KT = 32;            // keys per step

__global__ void __launch_bounds__(SW * 32) scan_simt_kernel(
    const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V, int64_t N, int m, int k,
    int chunks, int64_t chunk_len, int cap, int ltiles, const float* __restrict__ lq32, float* __restrict__ part,
    uint64_t* __restrict__ cand, int* __restrict__ ccount) {
    __shared__ float Ls[LT][D];
    __shared__ float Kt[D][KT + 1];
    __shared__ __align__(16) float Vs[KT][D];
    __shared__ unsigned hist[SW][256];

    const int lt = static_cast<int>(blockIdx.x % static_cast<unsigned>(ltiles));
    const int64_t rest = blockIdx.x / static_cast<unsigned>(ltiles);
    const int c = static_cast<int>(rest % chunks);
    const int64_t bh = rest / chunks;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t k0 = static_cast<int64_t>(c) * chunk_len;
    const int64_t k1 = min(N, k0 + chunk_len);
    const float tau = 0.125f;  // 1/sqrt(64)

    for (int t = threadIdx.x; t < LT * D; t += blockDim.x) {
        const int li = lt * LT + t / D;
        Ls[t / D][t % D] = li < m ? lq32[(bh * m + li) * D + t % D] : 0.f;
    }

    float mx[LPW], l[LPW], o0[LPW], o1[LPW];
    uint64_t theta[LPW];
    int cnt[LPW];
#pragma unroll
    for (int r = 0; r < LPW; ++r) {
        mx[r] = -INFINITY;
        l[r] = 0.f;
        o0[r] = o1[r] = 0.f;
        theta[r] = 0;
        cnt[r] = 0;
    }
    const __nv_bfloat16* Kh = K + bh * N * D;
    const __nv_bfloat16* Vh = V + bh * N * D;

    for (int64_t j0 = k0; j0 < k1; j0 += KT) {
        __syncthreads();
        {
            const int row = threadIdx.x >> 3, col = (threadIdx.x & 7) * 8;
            const int64_t j = j0 + row;
            float fk[8], fv[8];
            if (j < k1) {
                unpack_bf16x8(ldg_nc_v4(Kh + j * D + col), fk);
                unpack_bf16x8(ldg_nc_v4(Vh + j * D + col), fv);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) fk[t] = fv[t] = 0.f;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                Kt[col + t][row] = fk[t];
                Vs[row][col + t] = fv[t];
            }
        }
        __syncthreads();
        const int64_t j = j0 + lane;
        const bool valid = j < k1;
#pragma unroll
        for (int r = 0; r < LPW; ++r) {
            const int lr = warp * LPW + r;
            const int li = lt * LT + lr;
            if (li >= m) break;  // warp-uniform
            float dot = 0.f;
#pragma unroll 16
            for (int cc = 0; cc < D; ++cc) dot = fmaf(Ls[lr][cc], Kt[cc][lane], dot);
            const float s = valid ? dot * tau : -INFINITY;
            // online softmax over this chunk
            const float nm = fmaxf(mx[r], warp_max(s));
            const float sc = exp2f((mx[r] - nm) * kLog2e);
            const float pj = valid ? exp2f((s - nm) * kLog2e) : 0.f;
            l[r] = l[r] * sc + warp_sum(pj);
            float a0 = o0[r] * sc, a1 = o1[r] * sc;
#pragma unroll 8
            for (int jj = 0; jj < KT; ++jj) {
                const float pv = __shfl_sync(0xffffffffu, pj, jj);
                const float2 vv = *reinterpret_cast<const float2*>(&Vs[jj][2 * lane]);
                a0 = fmaf(pv, vv.x, a0);
                a1 = fmaf(pv, vv.y, a1);
            }
            o0[r] = a0;
            o1[r] = a1;
            mx[r] = nm;
            // routed-expert candidates
            uint64_t* buf = cand + ((bh * chunks + c) * m + li) * static_cast<int64_t>(cap);
            warp_offer(buf, cnt[r], theta[r], cap, k, valid, topk_key(s, static_cast<uint32_t>(j)), hist[warp]);
        }
    }
#pragma unroll
    for (int r = 0; r < LPW; ++r) {
        const int li = lt * LT + warp * LPW + r;
        if (li >= m) break;
        const int64_t slot = (bh * chunks + c) * m + li;
        float* pp = part + slot * 68;
        if (lane == 0) {
            pp[0] = mx[r];
            pp[1] = l[r];
            ccount[slot] = cnt[r];
        }
        pp[4 + 2 * lane] = o0[r];
        pp[5 + 2 * lane] = o1[r];
    }
}

}  // namespace

cudaError_t launch_scan(const Plan& p, const Work& w, const __nv_bfloat16* K, const __nv_bfloat16* V,
                        cudaStream_t st) {
    const int ltiles = (p.s.m + LT - 1) / LT;
    const ScanLevel& L = p.lev[0];
    const unsigned grid = static_cast<unsigned>(p.s.BH * L.chunks * ltiles);
    scan_simt_kernel<<<grid, SW * 32, 0, st>>>(K, V, p.s.N, p.s.m, p.s.k, L.chunks, L.chunk_len, L.cap, ltiles,
                                               w.lq32, w.part, w.cand, w.ccount);
    return cudaGetLastError();
}

}  // namespace mita
