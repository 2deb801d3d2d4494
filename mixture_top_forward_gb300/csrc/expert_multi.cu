// Stage 4 with s routed experts per query (s > 1): one pass per rank j.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造": a query attends to the m shared
// pairs (Lq_i, LV_i) and to its routed keys under ONE softmax. With s routed
// experts the routed keys are the union of the s experts' key sets, each key
// once. Algorithm 1 of "And attention is also FFN? …" (en.roboind.com)
// combines the parts of that softmax by online softmax; here the parts are
// the ranks j = 0 .. s-1 of the query's routes:
//   pass j groups the queries by their j-th expert e (the grouping step of
//   rank j) and streams e's k pairs (pass 0 also the m shared pairs) through
//   the running max / sum / accumulator of each query. A key that one of the
//   query's earlier-ranked experts also holds was already counted, so its
//   logit is set to -inf: expert key lists are ascending, so each query walks
//   one pointer per earlier expert alongside the keys (at most k steps each).
//   Passes 0 .. s-2 leave (accumulator, max, sum) in an fp32 state row per
//   query; pass s-1 writes the normalised bf16 output.
//
// One CTA per work item (expert, start, <= 128 queries, head), one thread
// per query; key/value rows are read from shared memory as broadcasts.
#include <climits>

#include "mita_internal.cuh"

namespace mita {

namespace {

constexpr int ET = 128;  // queries (threads) per work item
constexpr int EB = 32;   // keys per staged block
constexpr int SW = 68;   // floats per state row: accumulator[64], max, sum, 2 unused

__global__ void __launch_bounds__(ET) expert_multi_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
    int64_t N, int m, int k, int s, int j, const int4* __restrict__ items, const int* __restrict__ nitems,
    const int* __restrict__ perm, const int32_t* __restrict__ expert_idx, const int32_t* __restrict__ route,
    const float* __restrict__ lq32, const float* __restrict__ lv32, float* __restrict__ state,
    __nv_bfloat16* __restrict__ out) {
    __shared__ __align__(16) float Ks[EB][D];
    __shared__ __align__(16) float Vs[EB][D];
    __shared__ int Kix[EB];  // key index of each staged row (-1: a shared pair)
    if (static_cast<int>(blockIdx.x) >= *nitems) return;
    const int4 item = items[blockIdx.x];
    const int e = item.x, start = item.y, len = item.z;
    const int64_t bh = item.w;
    const int t = threadIdx.x;
    const bool valid = t < len;
    const int n = valid ? perm[bh * N + start + t] : 0;
    const int64_t qrow = bh * N + n;

    float q[D], o[D];
    {
        const __nv_bfloat16* qr = Q + qrow * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) unpack_bf16x8(ldg_nc_v4(qr + c), q + c);
    }
    float mx = -INFINITY, l = 0.f;
    if (j > 0 && valid) {
        const float4* sr = reinterpret_cast<const float4*>(state + qrow * SW);
#pragma unroll
        for (int c4 = 0; c4 < D / 4; ++c4) {
            const float4 x = sr[c4];
            o[4 * c4] = x.x;
            o[4 * c4 + 1] = x.y;
            o[4 * c4 + 2] = x.z;
            o[4 * c4 + 3] = x.w;
        }
        const float4 ml = sr[D / 4];
        mx = ml.x;
        l = ml.y;
    } else {
#pragma unroll
        for (int c = 0; c < D; ++c) o[c] = 0.f;
    }
    // the key lists of the query's earlier-ranked experts, walked alongside
    const int32_t* prev[MITA_MAX_S - 1];
    int ptr[MITA_MAX_S - 1], cur[MITA_MAX_S - 1];
#pragma unroll
    for (int i = 0; i < MITA_MAX_S - 1; ++i) {
        if (i < j && valid) {
            const int ei = route[qrow * s + i];
            prev[i] = expert_idx + (bh * m + ei) * static_cast<int64_t>(k);
            ptr[i] = 0;
            cur[i] = prev[i][0];
        } else {
            prev[i] = nullptr;
            ptr[i] = k;
            cur[i] = INT_MAX;
        }
    }
    const int ms = j == 0 ? m : 0;  // the shared pairs enter in pass 0 only
    const int total = ms + k;
    const int32_t* sel = expert_idx + (bh * m + e) * static_cast<int64_t>(k);

    for (int j0 = 0; j0 < total; j0 += EB) {
        const int nb = min(EB, total - j0);
        __syncthreads();
        {   // stage 32 key rows and 32 value rows: 4 threads per row, 16 dims each
            const int r = t >> 2, c0 = (t & 3) * 16;
            const int jj = j0 + r;
            if (r < nb) {
                if (jj < ms) {
                    const float* kr = lq32 + (bh * m + jj) * D + c0;
                    const float* vr = lv32 + (bh * m + jj) * D + c0;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        Ks[r][c0 + c] = kr[c];
                        Vs[r][c0 + c] = vr[c];
                    }
                    if (c0 == 0) Kix[r] = -1;
                } else {
                    const int key = sel[jj - ms];
                    const int64_t row = bh * N + key;
                    unpack_bf16x8(ldg_nc_v4(K + row * D + c0), &Ks[r][c0]);
                    unpack_bf16x8(ldg_nc_v4(K + row * D + c0 + 8), &Ks[r][c0 + 8]);
                    unpack_bf16x8(ldg_nc_v4(V + row * D + c0), &Vs[r][c0]);
                    unpack_bf16x8(ldg_nc_v4(V + row * D + c0 + 8), &Vs[r][c0 + 8]);
                    if (c0 == 0) Kix[r] = key;
                }
            }
        }
        __syncthreads();
        float sv[EB];
        float bm = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < EB; ++jj) {
            sv[jj] = -INFINITY;
            if (jj < nb) {
                const int key = Kix[jj];
                bool dup = false;
                if (key >= 0) {
#pragma unroll
                    for (int i = 0; i < MITA_MAX_S - 1; ++i) {
                        if (i < j) {
                            while (cur[i] < key) {
                                ++ptr[i];
                                cur[i] = ptr[i] < k ? prev[i][ptr[i]] : INT_MAX;
                            }
                            dup = dup || cur[i] == key;
                        }
                    }
                }
                if (!dup) {
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
                    sv[jj] = dot * 0.125f;
                    bm = fmaxf(bm, sv[jj]);
                }
            }
        }
        if (bm == -INFINITY) continue;  // every key of the block was counted before
        const float nm = fmaxf(mx, bm);
        const float sc = exp2f((mx - nm) * kLog2e);  // mx = -inf: 0 (nothing accumulated yet)
        l *= sc;
#pragma unroll
        for (int c = 0; c < D; ++c) o[c] *= sc;
#pragma unroll
        for (int jj = 0; jj < EB; ++jj) {
            if (sv[jj] != -INFINITY) {
                const float pj = exp2f((sv[jj] - nm) * kLog2e);
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
    if (!valid) return;
    if (j == s - 1) {
        const float inv = 1.f / l;
        uint4* dst = reinterpret_cast<uint4*>(out + qrow * D);
#pragma unroll
        for (int c = 0; c < D; c += 8) {
            uint4 pk;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
            for (int u = 0; u < 4; ++u) h[u] = __floats2bfloat162_rn(o[c + 2 * u] * inv, o[c + 2 * u + 1] * inv);
            dst[c / 8] = pk;
        }
    } else {
        float4* sr = reinterpret_cast<float4*>(state + qrow * SW);
#pragma unroll
        for (int c4 = 0; c4 < D / 4; ++c4)
            sr[c4] = make_float4(o[4 * c4], o[4 * c4 + 1], o[4 * c4 + 2], o[4 * c4 + 3]);
        sr[D / 4] = make_float4(mx, l, 0.f, 0.f);
    }
}

}  // namespace

size_t expert_multi_state_bytes(const Plan& p) {
    return p.s.s_route > 1 ? static_cast<size_t>(p.s.BH) * p.s.N * SW * sizeof(float) : 0;
}

cudaError_t launch_expert_multi(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                                const __nv_bfloat16* V, const int32_t* expert_idx, const int32_t* route, int j,
                                __nv_bfloat16* out, cudaStream_t st) {
    const unsigned grid = static_cast<unsigned>(p.s.BH * p.max_items);
    expert_multi_kernel<<<grid, ET, 0, st>>>(Q, K, V, p.s.N, p.s.m, p.s.k, p.s.s_route, j,
                                             w.items + static_cast<size_t>(j) * p.s.BH * p.max_items, w.nitems + j,
                                             w.perm + static_cast<size_t>(j) * p.s.BH * p.s.N, expert_idx, route,
                                             w.lq32, w.lv32, w.state, out);
    return cudaGetLastError();
}

}  // namespace mita
