// Stage 4: query-expert attention, CUDA-core version.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造", and Figure 3 of
// "And attention is also FFN? …" (en.roboind.com): a query routed to expert e
// attends to the m shared pairs (keys Lq_i, values LV_i) and the k routed
// pairs (K_j, V_j for j in E_e) under ONE softmax over all m+k logits.
// Algorithm 1 of the same page combines the parts by online softmax, which
// is what the key loop below does: the m+k pairs stream through shared memory
// in blocks of 32, with a running max and rescaled accumulators.
//
// One CTA per work item (expert, start, <= 128 queries, head) of the flat
// item list, one thread per query; key/value rows are read from shared
// memory as broadcasts. Used where experts hold few queries.
#include "mita_internal.cuh"

namespace mita {

namespace {

constexpr int ET = 128;  // queries (threads) per work item
constexpr int EB = 32;   // keys per staged block

__global__ void __launch_bounds__(ET) expert_simt_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
    int64_t N, int m, int ms, int k, const int4* __restrict__ items, const int* __restrict__ nitems,
    const int* __restrict__ perm, const int32_t* __restrict__ expert_idx, const float* __restrict__ lq32,
    const float* __restrict__ lv32, __nv_bfloat16* __restrict__ out) {
    __shared__ __align__(16) float Ks[EB][D];
    __shared__ __align__(16) float Vs[EB][D];
    if (static_cast<int>(blockIdx.x) >= *nitems) return;
    const int4 item = items[blockIdx.x];
    const int e = item.x, start = item.y, len = item.z;
    const int64_t bh = item.w;
    const int t = threadIdx.x;
    const bool valid = t < len;
    const int n = valid ? perm[bh * N + start + t] : 0;

    float q[D], o[D];
    {
        const __nv_bfloat16* qr = Q + (bh * N + n) * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) unpack_bf16x8(ldg_nc_v4(qr + c), q + c);
    }
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] = 0.f;
    float mx = -INFINITY, l = 0.f;
    const int total = ms + k;  // ms = m shared pairs, or 0 (routing-only)
    const int32_t* sel = expert_idx + (bh * m + e) * static_cast<int64_t>(k);

    for (int j0 = 0; j0 < total; j0 += EB) {
        const int nb = min(EB, total - j0);
        __syncthreads();
        {   // stage 32 key rows and 32 value rows: 4 threads per row, 16 dims each
            const int r = t >> 2, c0 = (t & 3) * 16;
            const int j = j0 + r;
            if (r < nb) {
                if (j < ms) {
                    const float* kr = lq32 + (bh * m + j) * D + c0;
                    const float* vr = lv32 + (bh * m + j) * D + c0;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        Ks[r][c0 + c] = kr[c];
                        Vs[r][c0 + c] = vr[c];
                    }
                } else {
                    const int64_t row = bh * N + sel[j - ms];
                    unpack_bf16x8(ldg_nc_v4(K + row * D + c0), &Ks[r][c0]);
                    unpack_bf16x8(ldg_nc_v4(K + row * D + c0 + 8), &Ks[r][c0 + 8]);
                    unpack_bf16x8(ldg_nc_v4(V + row * D + c0), &Vs[r][c0]);
                    unpack_bf16x8(ldg_nc_v4(V + row * D + c0 + 8), &Vs[r][c0 + 8]);
                }
            }
        }
        __syncthreads();
        float s[EB];
        float bm = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < EB; ++jj) {
            if (jj < nb) {
                const float4* kr = reinterpret_cast<const float4*>(Ks[jj]);
                float dot = 0.f;
#pragma unroll
                for (int c4 = 0; c4 < D / 4; ++c4) {
                    const float4 a = kr[c4];
                    dot = fmaf(q[4 * c4], a.x, dot);
                    dot = fmaf(q[4 * c4 + 1], a.y, dot);
                    dot = fmaf(q[4 * c4 + 2], a.z, dot);
                    dot = fmaf(q[4 * c4 + 3], a.w, dot);
                }
                s[jj] = dot * 0.125f;
                bm = fmaxf(bm, s[jj]);
            } else {
                s[jj] = -INFINITY;
            }
        }
        const float nm = fmaxf(mx, bm);
        const float sc = exp2f((mx - nm) * kLog2e);
        l *= sc;
#pragma unroll
        for (int c = 0; c < D; ++c) o[c] *= sc;
#pragma unroll
        for (int jj = 0; jj < EB; ++jj) {
            if (jj < nb) {
                const float pj = exp2f((s[jj] - nm) * kLog2e);
                l += pj;
                const float4* vr = reinterpret_cast<const float4*>(Vs[jj]);
#pragma unroll
                for (int c4 = 0; c4 < D / 4; ++c4) {
                    const float4 b = vr[c4];
                    o[4 * c4] = fmaf(pj, b.x, o[4 * c4]);
                    o[4 * c4 + 1] = fmaf(pj, b.y, o[4 * c4 + 1]);
                    o[4 * c4 + 2] = fmaf(pj, b.z, o[4 * c4 + 2]);
                    o[4 * c4 + 3] = fmaf(pj, b.w, o[4 * c4 + 3]);
                }
            }
        }
        mx = nm;
    }
    if (valid) {
        const float inv = 1.f / l;
        uint4* dst = reinterpret_cast<uint4*>(out + (bh * N + n) * D);
#pragma unroll
        for (int c = 0; c < D; c += 8) {
            uint4 pk;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
            for (int u = 0; u < 4; ++u) h[u] = __floats2bfloat162_rn(o[c + 2 * u] * inv, o[c + 2 * u + 1] * inv);
            dst[c / 8] = pk;
        }
    }
}

}  // namespace

cudaError_t launch_expert_simt(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                          const __nv_bfloat16* V, const int32_t* expert_idx, __nv_bfloat16* out, cudaStream_t st) {
    const unsigned grid = static_cast<unsigned>(p.s.BH * p.max_items);
    expert_simt_kernel<<<grid, ET, 0, st>>>(Q, K, V, p.s.N, p.s.m, p.shared ? p.s.m : 0, p.s.k, w.items, w.nitems,
                                            w.perm,
                                            expert_idx, w.lq32, w.lv32, out);
    return cudaGetLastError();
}

}  // namespace mita
