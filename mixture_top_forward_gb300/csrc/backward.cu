// Backward pass of MiTA: gradients of the forward output with respect to Q, K
// and V, with each landmark's top-k key set and each query's route held fixed
// (both are piecewise constant in the inputs; the pages train MiTA models --
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), results section -- but
// do not describe the backward pass, so this is the derivative of the
// forward pass as written in that page's section
// "MiTA：用少量地标查询，同时完成压缩与专家构造").
//
// Per head, tau = 1/sqrt(d), with the forward pass
//   Lq = W Q (local average pooling),  A = softmax(tau Lq K^T),  LV = A V,
//   out_n = sum_i p_ni LV_i + sum_{j in E} p_nj V_j,
//   p_n = softmax over [tau q_n Lq_i (i < m), tau q_n K_j (j in E)],
// and Delta_n = dO_n . out_n, dS = p (dO . value - Delta):
//   dq_n  = tau sum ds_nj key_j                        (expert attention)
//   dLq_i += tau sum_n ds_ni q_n,   dLV_i += sum_n p_ni dO_n
//   dK_j  += tau sum_n ds_nj q_n,   dV_j  += sum_n p_nj dO_n   (routed keys)
//   dt_ij = A_ij (dLV_i . V_j - dLV_i . LV_i)          (landmark attention)
//   dK_j  += tau sum_i dt_ij Lq_i,  dV_j += sum_i A_ij dLV_i,
//   dLq_i += tau sum_j dt_ij K_j
//   dQ_n  += sum over the windows i holding n of dLq_i / |window i|.
// Everything runs in fp32 on the CUDA cores from the bf16 inputs (a first
// version: every kernel is a plain loop over staged rows).
#include <algorithm>
#include <climits>

#include "mita_internal.cuh"
#include "pool_grad.cuh"

namespace mita {

namespace {

constexpr float kTau = 0.125f;  // 1/sqrt(64)
constexpr int BT = 128;         // threads per CTA
constexpr int KBLK = 32;        // staged key rows
constexpr int LD = D + 1;       // padded row stride of per-thread rows in shared memory

__device__ __forceinline__ void flag_bad(int* status) { atomicCAS(status, 0, MITA_ERR_INVALID_ARG); }

// 16 dims of a bf16 row, widened to fp32 (the staging loops give each of 4
// threads 16 dims of a row).
__device__ __forceinline__ void stage_bf16_row(const __nv_bfloat16* src, float* dst) {
    unpack_bf16x8(ldg_nc_v4(src), dst);
    unpack_bf16x8(ldg_nc_v4(src + 8), dst + 8);
}

// ---- landmark statistics: LV_i and log-sum-exp_i over all keys ----
// One thread per landmark, one CTA per (head, 128 landmarks, key chunk).
__global__ void __launch_bounds__(BT) lm_stats_kernel(const __nv_bfloat16* __restrict__ K,
                                                      const __nv_bfloat16* __restrict__ V, int64_t N, int m,
                                                      int ltiles, int chunks, int64_t chunk_len,
                                                      const float* __restrict__ lq32, float* __restrict__ part) {
    __shared__ __align__(16) float Ks[KBLK][D];
    __shared__ __align__(16) float Vs[KBLK][D];
    const int c = static_cast<int>(blockIdx.x % chunks);
    const int64_t rest = blockIdx.x / chunks;
    const int lt = static_cast<int>(rest % ltiles);
    const int64_t bh = rest / ltiles;
    const int t = threadIdx.x;
    const int i = lt * BT + t;
    const bool valid = i < m;
    float lq[D], o[D];
#pragma unroll
    for (int x = 0; x < D; ++x) {
        lq[x] = valid ? lq32[(bh * m + i) * D + x] : 0.f;
        o[x] = 0.f;
    }
    float mx = -INFINITY, l = 0.f;
    const int64_t k0 = c * chunk_len, k1 = min(N, k0 + chunk_len);
    for (int64_t j0 = k0; j0 < k1; j0 += KBLK) {
        const int nb = static_cast<int>(k1 - j0 < KBLK ? k1 - j0 : KBLK);
        __syncthreads();
        {
            const int r = t >> 2, c0 = (t & 3) * 16;
            if (r < nb) {
                const int64_t row = bh * N + j0 + r;
                stage_bf16_row(K + row * D + c0, &Ks[r][c0]);
                stage_bf16_row(V + row * D + c0, &Vs[r][c0]);
            }
        }
        __syncthreads();
        float sv[KBLK];
        float bm = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < KBLK; ++jj) {
            float dot = 0.f;
            if (jj < nb) {
#pragma unroll
                for (int x = 0; x < D; ++x) dot = fmaf(lq[x], Ks[jj][x], dot);
            }
            sv[jj] = jj < nb ? dot * kTau : -INFINITY;
            bm = fmaxf(bm, sv[jj]);
        }
        const float nm = fmaxf(mx, bm);
        const float sc = expf(mx - nm);  // mx = -inf: 0
        l *= sc;
#pragma unroll
        for (int x = 0; x < D; ++x) o[x] *= sc;
#pragma unroll
        for (int jj = 0; jj < KBLK; ++jj) {
            if (jj < nb) {
                const float p = expf(sv[jj] - nm);
                l += p;
#pragma unroll
                for (int x = 0; x < D; ++x) o[x] = fmaf(p, Vs[jj][x], o[x]);
            }
        }
        mx = nm;
    }
    if (valid) {
        float* dst = part + ((bh * chunks + c) * m + i) * 68;
#pragma unroll
        for (int x = 0; x < D; ++x) dst[x] = o[x];
        dst[D] = mx;
        dst[D + 1] = l;
    }
}

// Merges the chunks: LV_i (fp32) and lse_i = max + log(sum).
__global__ void __launch_bounds__(BT) lm_merge_kernel(int64_t BH, int m, int chunks, const float* __restrict__ part,
                                                      float* __restrict__ lv, float* __restrict__ lse) {
    const int64_t x = static_cast<int64_t>(blockIdx.x) * BT + threadIdx.x;
    if (x >= BH * m) return;
    const int64_t bh = x / m;
    const int i = static_cast<int>(x % m);
    float M = -INFINITY;
    for (int c = 0; c < chunks; ++c) M = fmaxf(M, part[((bh * chunks + c) * m + i) * 68 + D]);
    float S = 0.f, acc[D];
#pragma unroll
    for (int y = 0; y < D; ++y) acc[y] = 0.f;
    for (int c = 0; c < chunks; ++c) {
        const float* pr = part + ((bh * chunks + c) * m + i) * 68;
        if (pr[D + 1] == 0.f) continue;  // an empty chunk
        const float f = expf(pr[D] - M);
        S = fmaf(pr[D + 1], f, S);
#pragma unroll
        for (int y = 0; y < D; ++y) acc[y] = fmaf(pr[y], f, acc[y]);
    }
    const float inv = 1.f / S;
#pragma unroll
    for (int y = 0; y < D; ++y) lv[x * D + y] = acc[y] * inv;
    lse[x] = M + logf(S);
}

// ---- routes: checked copy and per-expert counts for the grouping ----
__global__ void __launch_bounds__(256) route_count_kernel(const int32_t* __restrict__ route, int64_t N, int m,
                                                          int64_t nblocks, int32_t* __restrict__ route_ok,
                                                          int* __restrict__ counts, int* __restrict__ status) {
    __shared__ int sh[MITA_MAX_M_INTERNAL];
    const int64_t blk = blockIdx.x % nblocks, bh = blockIdx.x / nblocks;
    for (int e = threadIdx.x; e < m; e += 256) sh[e] = 0;
    __syncthreads();
    const int64_t n = blk * 256 + threadIdx.x;
    if (n < N) {
        int e = route[bh * N + n];
        if (e < 0 || e >= m) {  // not a route of this problem: counted as expert 0, and reported
            flag_bad(status);
            e = 0;
        }
        route_ok[bh * N + n] = e;
        atomicAdd(&sh[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < m; e += 256)
        if (sh[e]) atomicAdd(&counts[bh * m + e], sh[e]);
}

// ---- expert attention backward: one CTA per work item (<= 128 queries of one expert) ----
struct ExpSmem {
    float q[BT][LD];     // the item's query rows
    float dO[BT][LD];    // their output gradients
    float k[KBLK][D];    // staged key rows
    float v[KBLK][D];    // staged value rows
    float p[KBLK][BT + 1];   // softmax weights of the block, per query
    float ds[KBLK][BT + 1];  // dS of the block, per query
    int kix[KBLK];       // key index (>= 0), shared pair -1 - i, or INT_MIN (invalid, masked)
};

__global__ void __launch_bounds__(BT) exp_bwd_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K, const __nv_bfloat16* __restrict__ V,
    const __nv_bfloat16* __restrict__ dO, int64_t N, int m, int k, const int4* __restrict__ items,
    const int* __restrict__ nitems, const int* __restrict__ perm, const int32_t* __restrict__ expert_idx,
    const float* __restrict__ lq32, const float* __restrict__ lv, float* __restrict__ dQ, float* __restrict__ dK,
    float* __restrict__ dV, float* __restrict__ dlq, float* __restrict__ dlv, int* __restrict__ status) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    ExpSmem& S = *reinterpret_cast<ExpSmem*>(smem_raw);
    if (static_cast<int>(blockIdx.x) >= *nitems) return;
    const int4 item = items[blockIdx.x];
    const int e = item.x, start = item.y, len = item.z;
    const int64_t bh = item.w;
    const int t = threadIdx.x;
    const bool valid = t < len;
    const int n = valid ? perm[bh * N + start + t] : 0;
    float q[D];
    {
        float g[D];
        const __nv_bfloat16* qr = Q + (bh * N + n) * D;
        const __nv_bfloat16* gr = dO + (bh * N + n) * D;
#pragma unroll
        for (int c = 0; c < D; c += 8) {
            unpack_bf16x8(ldg_nc_v4(qr + c), q + c);
            unpack_bf16x8(ldg_nc_v4(gr + c), g + c);
        }
#pragma unroll
        for (int c = 0; c < D; ++c) {
            if (!valid) q[c] = g[c] = 0.f;
            S.q[t][c] = q[c];
            S.dO[t][c] = g[c];
        }
    }
    const int total = m + k;
    const int32_t* sel = expert_idx + (bh * m + e) * static_cast<int64_t>(k);
    auto stage = [&](int j0, int nb) {
        const int r = t >> 2, c0 = (t & 3) * 16;
        if (r < nb) {
            const int jj = j0 + r;
            int kix;
            if (jj < m) {
                const float* kr = lq32 + (bh * m + jj) * D + c0;
                const float* vr = lv + (bh * m + jj) * D + c0;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    S.k[r][c0 + c] = kr[c];
                    S.v[r][c0 + c] = vr[c];
                }
                kix = -1 - jj;
            } else {
                const int key = sel[jj - m];
                if (key < 0 || key >= N) {  // not a key index: masked, and reported
                    if (c0 == 0) flag_bad(status);
#pragma unroll
                    for (int c = 0; c < 16; ++c) S.k[r][c0 + c] = S.v[r][c0 + c] = 0.f;
                    kix = INT_MIN;
                } else {
                    const int64_t row = bh * N + key;
                    stage_bf16_row(K + row * D + c0, &S.k[r][c0]);
                    stage_bf16_row(V + row * D + c0, &S.v[r][c0]);
                    kix = key;
                }
            }
            if (c0 == 0) S.kix[r] = kix;
        }
    };
    // pass A: the query's log-sum-exp and Delta = dO . out (as sum p (dO . value))
    float mx = -INFINITY, l = 0.f, dl = 0.f;
    for (int j0 = 0; j0 < total; j0 += KBLK) {
        const int nb = min(KBLK, total - j0);
        __syncthreads();
        stage(j0, nb);
        __syncthreads();
        float sv[KBLK];
        float bm = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < KBLK; ++jj) {
            float dot = 0.f;
            const bool use = jj < nb && S.kix[jj] != INT_MIN;
            if (use) {
#pragma unroll
                for (int c = 0; c < D; ++c) dot = fmaf(q[c], S.k[jj][c], dot);
            }
            sv[jj] = use ? dot * kTau : -INFINITY;
            bm = fmaxf(bm, sv[jj]);
        }
        if (bm == -INFINITY) continue;
        const float nm = fmaxf(mx, bm);
        const float sc = expf(mx - nm);
        l *= sc;
        dl *= sc;
#pragma unroll
        for (int jj = 0; jj < KBLK; ++jj) {
            if (sv[jj] != -INFINITY) {
                const float p = expf(sv[jj] - nm);
                float dpv = 0.f;
#pragma unroll
                for (int c = 0; c < D; ++c) dpv = fmaf(S.dO[t][c], S.v[jj][c], dpv);
                l += p;
                dl = fmaf(p, dpv, dl);
            }
        }
        mx = nm;
    }
    const float lse = mx + logf(l);
    const float delta = dl / l;
    // pass B: dq, and the block's p and dS for the key-side sums
    float dq[D];
#pragma unroll
    for (int c = 0; c < D; ++c) dq[c] = 0.f;
    for (int j0 = 0; j0 < total; j0 += KBLK) {
        const int nb = min(KBLK, total - j0);
        __syncthreads();
        stage(j0, nb);
        __syncthreads();
        for (int jj = 0; jj < nb; ++jj) {
            float p = 0.f, ds = 0.f;
            if (S.kix[jj] != INT_MIN) {
                float dot = 0.f, dpv = 0.f;
#pragma unroll
                for (int c = 0; c < D; ++c) {
                    dot = fmaf(q[c], S.k[jj][c], dot);
                    dpv = fmaf(S.dO[t][c], S.v[jj][c], dpv);
                }
                p = expf(dot * kTau - lse);
                ds = p * (dpv - delta);
                const float f = ds * kTau;
#pragma unroll
                for (int c = 0; c < D; ++c) dq[c] = fmaf(f, S.k[jj][c], dq[c]);
            }
            S.p[jj][t] = valid ? p : 0.f;
            S.ds[jj][t] = valid ? ds : 0.f;
        }
        __syncthreads();
        {   // key-side sums over the item's queries: thread -> (key row r, 16 dims)
            const int r = t >> 2, c0 = (t & 3) * 16;
            if (r < nb && S.kix[r] != INT_MIN) {
                float gk[16], gv[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) gk[c] = gv[c] = 0.f;
                for (int u = 0; u < BT; ++u) {
                    const float ds = S.ds[r][u], p = S.p[r][u];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        gk[c] = fmaf(ds, S.q[u][c0 + c], gk[c]);
                        gv[c] = fmaf(p, S.dO[u][c0 + c], gv[c]);
                    }
                }
                const int kix = S.kix[r];
                float* tk = kix >= 0 ? dK + (bh * N + kix) * D : dlq + (bh * m + (-1 - kix)) * D;
                float* tv = kix >= 0 ? dV + (bh * N + kix) * D : dlv + (bh * m + (-1 - kix)) * D;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    atomicAdd(tk + c0 + c, gk[c] * kTau);
                    atomicAdd(tv + c0 + c, gv[c]);
                }
            }
        }
    }
    if (valid) {
        float4* dst = reinterpret_cast<float4*>(dQ + (bh * N + n) * D);
#pragma unroll
        for (int c = 0; c < D; c += 4) dst[c / 4] = make_float4(dq[c], dq[c + 1], dq[c + 2], dq[c + 3]);
    }
}

// Tensor-core path, per landmark: Delta'_i = dLV_i . LV_i, the log-sum-exp
// in log2 units, and dLV_i rounded to bf16 (an MMA operand).
__global__ void __launch_bounds__(BT) lm_prep_kernel(int64_t rows, const float* __restrict__ dlv,
                                                     const float* __restrict__ lv, const float* __restrict__ lse,
                                                     float* __restrict__ dlt, float* __restrict__ lse2,
                                                     __nv_bfloat16* __restrict__ dlvb) {
    const int64_t x = static_cast<int64_t>(blockIdx.x) * BT + threadIdx.x;
    if (x >= rows) return;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < D; ++c) {
        s = fmaf(dlv[x * D + c], lv[x * D + c], s);
        dlvb[x * D + c] = __float2bfloat16_rn(dlv[x * D + c]);
    }
    dlt[x] = s;
    lse2[x] = lse[x] * kLog2e;
}

// Delta'_i = dLV_i . LV_i
__global__ void __launch_bounds__(BT) lm_delta_kernel(int64_t rows, const float* __restrict__ dlv,
                                                      const float* __restrict__ lv, float* __restrict__ dlt) {
    const int64_t x = static_cast<int64_t>(blockIdx.x) * BT + threadIdx.x;
    if (x >= rows) return;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < D; ++c) s = fmaf(dlv[x * D + c], lv[x * D + c], s);
    dlt[x] = s;
}

// ---- landmark attention backward, key side: one thread per key ----
constexpr int LT = 16;  // staged landmarks
struct KeySmem {
    float k[BT][LD];
    float v[BT][LD];
    float lq[LT][D];
    float dlv[LT][D];
    float lse[LT], dlt[LT];
};

__global__ void __launch_bounds__(BT) lm_bwd_key_kernel(const __nv_bfloat16* __restrict__ K,
                                                        const __nv_bfloat16* __restrict__ V, int64_t N, int m,
                                                        int64_t nblocks, const float* __restrict__ lq32,
                                                        const float* __restrict__ dlv, const float* __restrict__ lse,
                                                        const float* __restrict__ dlt, float* __restrict__ dK,
                                                        float* __restrict__ dV) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    KeySmem& S = *reinterpret_cast<KeySmem*>(smem_raw);
    const int64_t blk = blockIdx.x % nblocks, bh = blockIdx.x / nblocks;
    const int t = threadIdx.x;
    const int64_t j = blk * BT + t;
    const bool valid = j < N;
    {
        float a[D], b[D];
        const int64_t row = bh * N + (valid ? j : 0);
#pragma unroll
        for (int c = 0; c < D; c += 8) {
            unpack_bf16x8(ldg_nc_v4(K + row * D + c), a + c);
            unpack_bf16x8(ldg_nc_v4(V + row * D + c), b + c);
        }
#pragma unroll
        for (int c = 0; c < D; ++c) {
            S.k[t][c] = a[c];
            S.v[t][c] = b[c];
        }
    }
    float gk[D], gv[D];
#pragma unroll
    for (int c = 0; c < D; ++c) gk[c] = gv[c] = 0.f;
    for (int i0 = 0; i0 < m; i0 += LT) {
        const int nt = min(LT, m - i0);
        __syncthreads();
        for (int x = t; x < nt * D; x += BT) {
            const int ii = x / D, c = x % D;
            S.lq[ii][c] = lq32[(bh * m + i0 + ii) * D + c];
            S.dlv[ii][c] = dlv[(bh * m + i0 + ii) * D + c];
        }
        if (t < nt) {
            S.lse[t] = lse[bh * m + i0 + t];
            S.dlt[t] = dlt[bh * m + i0 + t];
        }
        __syncthreads();
        for (int ii = 0; ii < nt; ++ii) {
            float dot = 0.f, da = 0.f;
#pragma unroll
            for (int c = 0; c < D; ++c) {
                dot = fmaf(S.lq[ii][c], S.k[t][c], dot);
                da = fmaf(S.dlv[ii][c], S.v[t][c], da);
            }
            const float a = expf(dot * kTau - S.lse[ii]);
            const float f = a * (da - S.dlt[ii]) * kTau;
#pragma unroll
            for (int c = 0; c < D; ++c) {
                gk[c] = fmaf(f, S.lq[ii][c], gk[c]);
                gv[c] = fmaf(a, S.dlv[ii][c], gv[c]);
            }
        }
    }
    if (valid) {
        float* tk = dK + (bh * N + j) * D;
        float* tv = dV + (bh * N + j) * D;
#pragma unroll
        for (int c = 0; c < D; ++c) {
            tk[c] += gk[c];
            tv[c] += gv[c];
        }
    }
}

// ---- landmark attention backward, landmark side: dLq over key chunks ----
struct LmSmem {
    float lq[BT][LD];
    float dlv[BT][LD];
    float k[KBLK][D];
    float v[KBLK][D];
};

__global__ void __launch_bounds__(BT) lm_bwd_lq_kernel(const __nv_bfloat16* __restrict__ K,
                                                       const __nv_bfloat16* __restrict__ V, int64_t N, int m,
                                                       int ltiles, int chunks, int64_t chunk_len,
                                                       const float* __restrict__ lq32, const float* __restrict__ dlv,
                                                       const float* __restrict__ lse, const float* __restrict__ dlt,
                                                       float* __restrict__ dlq) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    LmSmem& S = *reinterpret_cast<LmSmem*>(smem_raw);
    const int c = static_cast<int>(blockIdx.x % chunks);
    const int64_t rest = blockIdx.x / chunks;
    const int lt = static_cast<int>(rest % ltiles);
    const int64_t bh = rest / ltiles;
    const int t = threadIdx.x;
    const int i = lt * BT + t;
    const bool valid = i < m;
#pragma unroll
    for (int x = 0; x < D; ++x) {
        S.lq[t][x] = valid ? lq32[(bh * m + i) * D + x] : 0.f;
        S.dlv[t][x] = valid ? dlv[(bh * m + i) * D + x] : 0.f;
    }
    const float lsei = valid ? lse[bh * m + i] : 0.f, dlti = valid ? dlt[bh * m + i] : 0.f;
    float g[D];
#pragma unroll
    for (int x = 0; x < D; ++x) g[x] = 0.f;
    const int64_t k0 = c * chunk_len, k1 = min(N, k0 + chunk_len);
    for (int64_t j0 = k0; j0 < k1; j0 += KBLK) {
        const int nb = static_cast<int>(k1 - j0 < KBLK ? k1 - j0 : KBLK);
        __syncthreads();
        {
            const int r = t >> 2, c0 = (t & 3) * 16;
            if (r < nb) {
                const int64_t row = bh * N + j0 + r;
                stage_bf16_row(K + row * D + c0, &S.k[r][c0]);
                stage_bf16_row(V + row * D + c0, &S.v[r][c0]);
            }
        }
        __syncthreads();
        for (int jj = 0; jj < nb; ++jj) {
            float dot = 0.f, da = 0.f;
#pragma unroll
            for (int x = 0; x < D; ++x) {
                dot = fmaf(S.lq[t][x], S.k[jj][x], dot);
                da = fmaf(S.dlv[t][x], S.v[jj][x], da);
            }
            const float a = expf(dot * kTau - lsei);
            const float f = a * (da - dlti) * kTau;
#pragma unroll
            for (int x = 0; x < D; ++x) g[x] = fmaf(f, S.k[jj][x], g[x]);
        }
    }
    if (valid) {
        float* dst = dlq + (bh * m + i) * D;
#pragma unroll
        for (int x = 0; x < D; ++x) atomicAdd(dst + x, g[x]);
    }
}

// ---- pooling backward: dQ_n += dLq_i / |window i| for every window holding n ----
__global__ void __launch_bounds__(256) pool_bwd_kernel(int64_t BH, int64_t N, int gh, int gw, int p, int m,
                                                       const float* __restrict__ dlq, float* __restrict__ dQ) {
    const int64_t x = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    if (x >= BH * N) return;
    const int64_t bh = x / N, n = x % N;
    float g[D];
#pragma unroll
    for (int c = 0; c < D; ++c) g[c] = 0.f;
    pool_windows_of(N, gh, gw, p, m, n, [&](int i, float w) {
        const float4* s = reinterpret_cast<const float4*>(dlq + (bh * m + i) * D);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) {
            const float4 v = s[c];
            g[4 * c] = fmaf(v.x, w, g[4 * c]);
            g[4 * c + 1] = fmaf(v.y, w, g[4 * c + 1]);
            g[4 * c + 2] = fmaf(v.z, w, g[4 * c + 2]);
            g[4 * c + 3] = fmaf(v.w, w, g[4 * c + 3]);
        }
    });
    float4* dst = reinterpret_cast<float4*>(dQ + x * D);
#pragma unroll
    for (int c = 0; c < D / 4; ++c) {
        float4 v = dst[c];
        v.x += g[4 * c];
        v.y += g[4 * c + 1];
        v.z += g[4 * c + 2];
        v.w += g[4 * c + 3];
        dst[c] = v;
    }
}

int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

// Rows of Q and dO in grouped order: row p of head h is query perm[h][p]
// (16 bytes a thread).
static __global__ void group_rows_kernel(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ dO,
                                  const int* __restrict__ perm, int64_t rows, int64_t N, __nv_bfloat16* __restrict__ qg,
                                  __nv_bfloat16* __restrict__ dog) {
    const int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (x >= rows * 8) return;
    const int64_t r = x >> 3, c = x & 7;
    const int64_t src = (r / N) * N + perm[r];
    reinterpret_cast<uint4*>(qg)[r * 8 + c] = __ldg(reinterpret_cast<const uint4*>(Q) + src * 8 + c);
    reinterpret_cast<uint4*>(dog)[r * 8 + c] = __ldg(reinterpret_cast<const uint4*>(dO) + src * 8 + c);
}

BwdLayout backward_layout(const Plan& p) {
    BwdLayout L{};
    const int64_t BH = p.s.BH, N = p.s.N, m = p.s.m;
    L.ltiles = static_cast<int>(cdiv64(m, BT));
    const int sms = device_sms();
    int64_t chunks = cdiv64(4LL * sms, BH * L.ltiles);
    chunks = std::max<int64_t>(1, std::min<int64_t>(chunks, cdiv64(N, 256)));
    L.chunk_len = cdiv64(N, chunks);
    L.chunks = static_cast<int>(cdiv64(N, L.chunk_len));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) / 256 * 256;
        return o;
    };
    L.off_lv = take(BH * m * D * sizeof(float));
    L.off_lse = take(BH * m * sizeof(float));
    L.off_part = take(static_cast<size_t>(BH) * L.chunks * m * 68 * sizeof(float));
    L.off_dlq = take(BH * m * D * sizeof(float));
    L.off_dlv = take(BH * m * D * sizeof(float));
    L.off_dlt = take(BH * m * sizeof(float));
    L.off_route = take(BH * N * sizeof(int32_t));
    const bool tc = backward_tc_supported(p);
    L.off_qlse = take(tc ? BH * N * sizeof(float) : 0);
    L.off_qdelta = take(tc ? BH * N * sizeof(float) : 0);
    L.off_eidx = take(tc ? BH * m * static_cast<size_t>(p.s.k) * sizeof(int32_t) : 0);
    L.off_lse2 = take(tc ? BH * m * sizeof(float) : 0);
    L.off_dlvb = take(tc ? BH * m * D * 2 : 0);
    L.off_qg = take(tc ? BH * N * D * 2 : 0);
    L.off_dog = take(tc ? BH * N * D * 2 : 0);
    L.total = off;
    return L;
}

cudaError_t launch_backward(const Plan& p, const Work& w, const BwdLayout& L, void* bbase, const __nv_bfloat16* Q,
                            const __nv_bfloat16* K, const __nv_bfloat16* V, const __nv_bfloat16* dO,
                            const int32_t* expert_idx, const int32_t* route, float* dQ, float* dK, float* dV,
                            cudaStream_t st) {
    char* b = static_cast<char*>(bbase);
    float* lv = reinterpret_cast<float*>(b + L.off_lv);
    float* lse = reinterpret_cast<float*>(b + L.off_lse);
    float* part = reinterpret_cast<float*>(b + L.off_part);
    float* dlq = reinterpret_cast<float*>(b + L.off_dlq);
    float* dlv = reinterpret_cast<float*>(b + L.off_dlv);
    float* dlt = reinterpret_cast<float*>(b + L.off_dlt);
    int32_t* route_ok = reinterpret_cast<int32_t*>(b + L.off_route);
    const int64_t BH = p.s.BH, N = p.s.N;
    const int m = p.s.m, k = p.s.k;
    const size_t rows = static_cast<size_t>(BH) * N, mrows = static_cast<size_t>(BH) * m;
    cudaError_t e;
    if ((e = cudaMemsetAsync(dK, 0, rows * D * sizeof(float), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dV, 0, rows * D * sizeof(float), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dlq, 0, mrows * D * sizeof(float), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dlv, 0, mrows * D * sizeof(float), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(w.counts, 0, mrows * sizeof(int), st)) != cudaSuccess ||
        (e = cudaMemsetAsync(w.nitems, 0, sizeof(int), st)) != cudaSuccess)
        return e;
    if ((e = launch_pool(p, w, Q, st)) != cudaSuccess) return e;
    if (backward_tc_supported(p) && expert_tc_supported(p) && p.scan_tc && !p.split) {
        // Tensor-core path. Landmark statistics: the forward pass's scan and
        // merge (LV in fp32 and bf16, each landmark's log-sum-exp); the expert
        // sets it selects go to scratch (the caller's are the ones used).
        int32_t* eidx = reinterpret_cast<int32_t*>(b + L.off_eidx);
        float* qlse = reinterpret_cast<float*>(b + L.off_qlse);
        float* qdelta = reinterpret_cast<float*>(b + L.off_qdelta);
        float* lse2 = reinterpret_cast<float*>(b + L.off_lse2);
        __nv_bfloat16* dlvb = reinterpret_cast<__nv_bfloat16*>(b + L.off_dlvb);
        if (p.nlev > 1 && (e = cudaMemsetAsync(w.theta, 0, mrows * sizeof(uint64_t), st)) != cudaSuccess) return e;
        for (int l = 0; l + 1 < p.nlev; ++l) {
            if ((e = launch_scan_tc(p, w, K, V, l, st)) != cudaSuccess) return e;
            if ((e = launch_pilot_select(p, w, l, st)) != cudaSuccess) return e;
        }
        if ((e = launch_scan_tc(p, w, K, V, p.nlev - 1, st)) != cudaSuccess) return e;
        if (p.spec_j && (e = launch_scan_verify(p, w, K, st)) != cudaSuccess) return e;
        if ((e = launch_select(p, w, eidx, st, lse)) != cudaSuccess) return e;
        // routes (checked) and grouping, then each query's statistics
        const int64_t rb = cdiv64(N, 256);
        route_count_kernel<<<static_cast<unsigned>(BH * rb), 256, 0, st>>>(route, N, m, rb, route_ok, w.counts,
                                                                             w.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_group(p, w, route_ok, 0, st)) != cudaSuccess) return e;
        if ((e = launch_expert_stats(p, w, Q, K, V, expert_idx, dO, qlse, qdelta, st)) != cudaSuccess) return e;
        // expert attention, key side: dK, dV of the routed keys, dLq, dLV of the
        // shared ones; its row tiles from copies of Q and dO in grouped order
        __nv_bfloat16* qg = reinterpret_cast<__nv_bfloat16*>(b + L.off_qg);
        __nv_bfloat16* dog = reinterpret_cast<__nv_bfloat16*>(b + L.off_dog);
        group_rows_kernel<<<static_cast<unsigned>(cdiv64(static_cast<int64_t>(rows) * 8, 256)), 256, 0, st>>>(
            Q, dO, w.perm, static_cast<int64_t>(rows), N, qg, dog);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_backward_tc_expert_keys(p, w, qg, K, V, dog, expert_idx, qlse, qdelta, dK, dV, dlq, dlv,
                                                st)) != cudaSuccess)
            return e;
        // landmark attention: dK, dV, dLq
        lm_prep_kernel<<<static_cast<unsigned>(cdiv64(BH * m, BT)), BT, 0, st>>>(BH * m, dlv, w.lv32, lse, dlt, lse2,
                                                                                 dlvb);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = launch_backward_tc_landmark(p, w, K, V, dlvb, lse2, dlt, dK, dV, dlq, st)) != cudaSuccess) return e;
        // expert attention, row side, and the pooling: dQ
        return launch_backward_tc_expert_rows(p, w, qg, K, V, dog, expert_idx, qlse, qdelta, dlq, dQ, st);
    }
    const unsigned g1 = static_cast<unsigned>(BH * L.ltiles * L.chunks);
    lm_stats_kernel<<<g1, BT, 0, st>>>(K, V, N, m, L.ltiles, L.chunks, L.chunk_len, w.lq32, part);
    lm_merge_kernel<<<static_cast<unsigned>(cdiv64(BH * m, BT)), BT, 0, st>>>(BH, m, L.chunks, part, lv, lse);
    const int64_t rb = cdiv64(N, 256);
    route_count_kernel<<<static_cast<unsigned>(BH * rb), 256, 0, st>>>(route, N, m, rb, route_ok, w.counts,
                                                                         w.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_group(p, w, route_ok, 0, st)) != cudaSuccess) return e;
    const int sm_exp = static_cast<int>(sizeof(ExpSmem));
    if ((e = cudaFuncSetAttribute(exp_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sm_exp)) != cudaSuccess)
        return e;
    exp_bwd_kernel<<<static_cast<unsigned>(BH * p.max_items), BT, sm_exp, st>>>(
        Q, K, V, dO, N, m, k, w.items, w.nitems, w.perm, expert_idx, w.lq32, lv, dQ, dK, dV, dlq, dlv, w.status);
    lm_delta_kernel<<<static_cast<unsigned>(cdiv64(BH * m, BT)), BT, 0, st>>>(BH * m, dlv, lv, dlt);
    const int sm_key = static_cast<int>(sizeof(KeySmem));
    if ((e = cudaFuncSetAttribute(lm_bwd_key_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sm_key)) !=
        cudaSuccess)
        return e;
    const int64_t kb = cdiv64(N, BT);
    lm_bwd_key_kernel<<<static_cast<unsigned>(BH * kb), BT, sm_key, st>>>(K, V, N, m, kb, w.lq32, dlv, lse, dlt, dK,
                                                                          dV);
    const int sm_lm = static_cast<int>(sizeof(LmSmem));
    if ((e = cudaFuncSetAttribute(lm_bwd_lq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sm_lm)) !=
        cudaSuccess)
        return e;
    lm_bwd_lq_kernel<<<g1, BT, sm_lm, st>>>(K, V, N, m, L.ltiles, L.chunks, L.chunk_len, w.lq32, dlv, lse, dlt, dlq);
    pool_bwd_kernel<<<static_cast<unsigned>(cdiv64(BH * N, 256)), 256, 0, st>>>(BH, N, p.s.gh, p.s.gw, p.s.p, m, dlq,
                                                                                 dQ);
    return cudaGetLastError();
}

}  // namespace mita
