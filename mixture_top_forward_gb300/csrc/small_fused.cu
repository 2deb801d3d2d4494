// The whole MiTA forward pass of a short head in one kernel (one CTA per
// head), for heads whose queries, keys and values fit in shared memory
// (N <= 256 tokens, m <= 32 landmarks): the ViT shapes of the pages' image
// experiments ("NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), results
// section: DeiT-S on 14 x 14 patch grids).
//
// The stages are those of section "MiTA：用少量地标查询，同时完成压缩与专家构造"
// of the same page, in its order, on the CUDA cores in fp32:
//   1. landmarks Lq_i = mean of Q over window i (1-D windows or 2-D adaptive
//      pooling of the token grid, as pool.cu);
//   2. landmark scan: raw_ij = <Lq_i, K_j>; the shared-expert value LV_i =
//      softmax_j(tau raw_ij) V (one warp per landmark, the row in registers);
//      the routed expert E_i = the k keys with the largest tau raw_ij, ties
//      to the lower index, written in ascending index order;
//   3. routing: e(n) = argmax_i <q_n, Lq_i>, ties to the lowest i;
//   4. expert attention: one softmax over the m shared pairs (Lq_i, LV_i) and
//      the k routed pairs (K_j, V_j), j in E_e(n), by online softmax.
// At these sizes the general path spends its time on launches, short rows
// and work items of a few queries each; here every operand is read from HBM
// once and the head's rows stay in shared memory throughout.
//
// Shared memory: Q, K, V rows of the head, bf16, 128 bytes a row (16-byte
// chunk c of row r at chunk position c ^ (r & 7): a warp reading one chunk
// of 32 consecutive rows, or one whole row, hits every bank equally); Lq and
// LV, fp32 [m][64]; the experts E, one byte an index [m][k]. The products
// run as packed fp32 pairs (fma.rn.f32x2), the top-k on registers.
#include "mita_internal.cuh"
#include "umma.cuh"

namespace mita {

namespace {

constexpr int SF_THREADS = 512;  // 16 warps; two threads per query (N <= 256)
constexpr int SF_WARPS = SF_THREADS / 32;
static_assert(SF_THREADS == 2 * 256, "two threads per query of up to 256");
constexpr int SF_MAX_N = 256;
constexpr int SF_MAX_M = 32;
constexpr float kTauSF = 0.125f;  // 1 / sqrt(64)

struct SFArgs {
    const __nv_bfloat16* Q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    __nv_bfloat16* out;
    int32_t* expert_idx;  // [BH][m][k]
    int32_t* route;       // [BH][N]
    float* lq_out;        // [BH][m][64] or null
    float* lv_out;        // [BH][m][64] or null
    int N, m, k, gh, gw, p;
};

struct SFLayout {
    size_t q, kk, v, lq, lv, e, total;
};

__host__ __device__ inline SFLayout sf_layout(int N, int m, int k) {
    SFLayout L;
    L.q = 0;
    L.kk = static_cast<size_t>(N) * 128;
    L.v = L.kk + static_cast<size_t>(N) * 128;
    L.lq = L.v + static_cast<size_t>(N) * 128;
    L.lv = L.lq + static_cast<size_t>(m) * 64 * 4;
    L.e = L.lv + static_cast<size_t>(m) * 64 * 4;
    L.total = L.e + static_cast<size_t>(m) * k;
    return L;
}

// byte offset of 16-byte chunk c of bf16 row r (128 bytes a row)
__device__ __forceinline__ uint32_t sf_chunk(int r, int c) {
    return static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>(c ^ (r & 7)) << 4);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// element c of bf16 row r
__device__ __forceinline__ float sf_elem(const uint8_t* rows, int r, int c) {
    const uint16_t h = *reinterpret_cast<const uint16_t*>(rows + sf_chunk(r, c >> 3) + (c & 7) * 2);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ float2 lo2(const float4& v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(const float4& v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float sum2(const float2& v) { return v.x + v.y; }

__device__ __forceinline__ float2 bf2(uint32_t w) { return make_float2(bf_lo(w), bf_hi(w)); }
// Half h (columns 32 h .. 32 h + 31) of <x, bf16 row r>; x holds those 32
// columns as 16 pairs
__device__ __forceinline__ float sf_half_dot(const float2* x, const uint8_t* rows, int r, int h) {
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(rows + sf_chunk(r, 4 * h + c));
        a0 = __ffma2_rn(x[4 * c], bf2(w.x), a0);
        a1 = __ffma2_rn(x[4 * c + 1], bf2(w.y), a1);
        a0 = __ffma2_rn(x[4 * c + 2], bf2(w.z), a0);
        a1 = __ffma2_rn(x[4 * c + 3], bf2(w.w), a1);
    }
    return sum2(a0) + sum2(a1);
}
// Half h of <x, y>, y fp32 [64] in shared memory (broadcast reads)
__device__ __forceinline__ float sf_half_dot_f32(const float2* x, const float* y, int h) {
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float4 w = reinterpret_cast<const float4*>(y + 32 * h)[c];
        a0 = __ffma2_rn(x[2 * c], lo2(w), a0);
        a1 = __ffma2_rn(x[2 * c + 1], hi2(w), a1);
    }
    return sum2(a0) + sum2(a1);
}
// order key of a logit: larger tau * raw first (the score bits of topk_key)
__device__ __forceinline__ uint32_t sf_key(float raw) {
    return static_cast<uint32_t>(topk_key(raw * kTauSF, 0u) >> 32);
}

__global__ void __launch_bounds__(SF_THREADS, 1) small_fused_kernel(SFArgs a) {
    extern __shared__ __align__(16) uint8_t sm[];
    const SFLayout Ly = sf_layout(a.N, a.m, a.k);
    uint8_t* Qs = sm + Ly.q;
    uint8_t* Ks = sm + Ly.kk;
    uint8_t* Vs = sm + Ly.v;
    float* Lq = reinterpret_cast<float*>(sm + Ly.lq);
    float* LV = reinterpret_cast<float*>(sm + Ly.lv);
    uint8_t* E = sm + Ly.e;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = a.N, m = a.m, k = a.k;
    const int64_t bh = blockIdx.x;
    const int64_t row0 = bh * N;

    // ---- the head's Q, K, V rows into shared memory (16-byte copies) ----
    {
        const __nv_bfloat16* src[3] = {a.Q + row0 * 64, a.K + row0 * 64, a.V + row0 * 64};
        uint8_t* dst[3] = {Qs, Ks, Vs};
#pragma unroll
        for (int t = 0; t < 3; ++t)
            for (int x = tid; x < N * 8; x += SF_THREADS) {
                const int r = x >> 3, c = x & 7;
                umma::cp_async16(umma::smem_u32(dst[t] + sf_chunk(r, c)), src[t] + static_cast<int64_t>(r) * 64 + c * 8);
            }
        umma::cp_async_wait_all();
    }
    __syncthreads();

    // ---- 1. landmarks: window means of Q ----
    // (windows as pool.cu: [floor(i L / w), ceil((i + 1) L / w)); all
    // products here stay below 2^16)
    for (int o = tid; o < m * 64; o += SF_THREADS) {
        const int i = o >> 6, c = o & 63;
        float sum = 0.f;
        int cnt;
        if (a.p == 0) {
            const int w0 = (i * N) / m, w1 = ((i + 1) * N + m - 1) / m;
            for (int n = w0; n < w1; ++n) sum += sf_elem(Qs, n, c);
            cnt = w1 - w0;
        } else {
            const int r = i / a.p, cc = i % a.p;
            const int ya = (r * a.gh) / a.p, yb = ((r + 1) * a.gh + a.p - 1) / a.p;
            const int xa = (cc * a.gw) / a.p, xb = ((cc + 1) * a.gw + a.p - 1) / a.p;
            for (int y = ya; y < yb; ++y)
                for (int x = xa; x < xb; ++x) sum += sf_elem(Qs, y * a.gw + x, c);
            cnt = (yb - ya) * (xb - xa);
        }
        const float v = sum / static_cast<float>(cnt);
        Lq[o] = v;
        if (a.lq_out) a.lq_out[bh * m * 64 + o] = v;
    }
    __syncthreads();

    // ---- 2. landmark scan: LV_i and E_i, one warp per landmark; lane l
    //      holds keys j = 32 t + l ----
    constexpr int T = SF_MAX_N / 32;
    for (int i = warp; i < m; i += SF_WARPS) {
        const float* lqi = Lq + i * 64;
        float2 acc[T];
#pragma unroll
        for (int t = 0; t < T; ++t) acc[t] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // columns 8c .. 8c + 7
            const float4 la = reinterpret_cast<const float4*>(lqi)[2 * c];
            const float4 lb = reinterpret_cast<const float4*>(lqi)[2 * c + 1];
#pragma unroll
            for (int t = 0; t < T; ++t) {
                const int j = 32 * t + lane;
                if (32 * t < N) {  // (warp-uniform)
                    const uint4 w = *reinterpret_cast<const uint4*>(Ks + sf_chunk(j < N ? j : 0, c));
                    acc[t] = __ffma2_rn(lo2(la), bf2(w.x), acc[t]);
                    acc[t] = __ffma2_rn(hi2(la), bf2(w.y), acc[t]);
                    acc[t] = __ffma2_rn(lo2(lb), bf2(w.z), acc[t]);
                    acc[t] = __ffma2_rn(hi2(lb), bf2(w.w), acc[t]);
                }
            }
        }
        float raw[T], mx = -INFINITY;
#pragma unroll
        for (int t = 0; t < T; ++t) {
            raw[t] = 32 * t + lane < N ? sum2(acc[t]) : -INFINITY;
            mx = fmaxf(mx, raw[t] * kTauSF);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float pr[T], sum = 0.f;
#pragma unroll
        for (int t = 0; t < T; ++t) {
            pr[t] = 32 * t + lane < N ? __expf(raw[t] * kTauSF - mx) : 0.f;
            sum += pr[t];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        // LV_i: lane l sums columns 2l, 2l + 1 over the keys (weights by shuffle)
        float2 lv0 = make_float2(0.f, 0.f), lv1 = lv0;
        const uint32_t woff = static_cast<uint32_t>(lane & 3) * 4;  // word `lane` of a row: columns 2 lane, 2 lane + 1
#pragma unroll
        for (int t = 0; t < T; ++t) {
            if (32 * t >= N) break;  // (warp-uniform)
#pragma unroll
            for (int s2 = 0; s2 < 32; s2 += 2) {
                const int j = 32 * t + s2;
                const float p0 = __shfl_sync(0xffffffffu, pr[t], s2), p1 = __shfl_sync(0xffffffffu, pr[t], s2 + 1);
                const float2 v0 = bf2(*reinterpret_cast<const uint32_t*>(Vs + sf_chunk(j < N ? j : 0, lane >> 2) + woff));
                const float2 v1 =
                    bf2(*reinterpret_cast<const uint32_t*>(Vs + sf_chunk(j + 1 < N ? j + 1 : 0, lane >> 2) + woff));
                lv0 = __ffma2_rn(make_float2(p0, p0), v0, lv0);
                lv1 = __ffma2_rn(make_float2(p1, p1), v1, lv1);
            }
        }
        const float inv = 1.f / sum;
        const float2 lv2 = make_float2((lv0.x + lv1.x) * inv, (lv0.y + lv1.y) * inv);
        reinterpret_cast<float2*>(LV + i * 64)[lane] = lv2;
        if (a.lv_out) reinterpret_cast<float2*>(a.lv_out + (bh * m + i) * 64)[lane] = lv2;
        // E_i: the k largest keys. Their threshold (the k-th largest key) bit
        // by bit from the top: the largest value with at least k keys at or
        // above it. Then every key above it and, of the keys equal to it, the
        // lowest indices, in ascending index order.
        uint32_t kk[T];
#pragma unroll
        for (int t = 0; t < T; ++t) kk[t] = 32 * t + lane < N ? sf_key(raw[t]) : 0u;  // real keys are > 0
        uint32_t thr = 0;
        for (int b = 31; b >= 0; --b) {
            const uint32_t cand = thr | (1u << b);
            unsigned c = 0;
#pragma unroll
            for (int t = 0; t < T; ++t) c += kk[t] >= cand ? 1u : 0u;
            if (__reduce_add_sync(0xffffffffu, c) >= static_cast<unsigned>(k)) thr = cand;
        }
        unsigned above = 0;
#pragma unroll
        for (int t = 0; t < T; ++t) above += kk[t] > thr ? 1u : 0u;
        const unsigned remaining = static_cast<unsigned>(k) - __reduce_add_sync(0xffffffffu, above);
        int32_t* dst = a.expert_idx + (bh * m + i) * static_cast<int64_t>(k);
        uint8_t* ei = E + i * k;
        const unsigned below = (1u << lane) - 1u;
        unsigned taken = 0, eq_seen = 0;
#pragma unroll
        for (int t = 0; t < T; ++t) {
            if (32 * t >= N) break;  // (warp-uniform)
            const bool eq = kk[t] == thr && kk[t] != 0u;
            const unsigned eqb = __ballot_sync(0xffffffffu, eq);
            const bool sel = kk[t] > thr || (eq && eq_seen + __popc(eqb & below) < remaining);
            const unsigned sb = __ballot_sync(0xffffffffu, sel);
            if (sel) {
                const int r = static_cast<int>(taken + __popc(sb & below));
                dst[r] = 32 * t + lane;
                ei[r] = static_cast<uint8_t>(32 * t + lane);
            }
            taken += __popc(sb);
            eq_seen += __popc(eqb);
        }
    }
    __syncthreads();

    // ---- 3. routing and 4. expert attention: two threads per query ----
    // (lanes 2t and 2t + 1 of a warp: each holds half of q and of the output;
    // a logit is the sum of the two halves' dot products, formed the same way
    // in both threads)
    const int n = tid >> 1, h = tid & 1;
    const unsigned act = __ballot_sync(0xffffffffu, n < N);
    if (n < N) {
        float2 q[16];  // columns 32 h .. 32 h + 31
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 w = *reinterpret_cast<const uint4*>(Qs + sf_chunk(n, 4 * h + c));
            q[4 * c] = make_float2(bf_lo(w.x), bf_hi(w.x));
            q[4 * c + 1] = make_float2(bf_lo(w.y), bf_hi(w.y));
            q[4 * c + 2] = make_float2(bf_lo(w.z), bf_hi(w.z));
            q[4 * c + 3] = make_float2(bf_lo(w.w), bf_hi(w.w));
        }
        auto both = [&](float part) { return part + __shfl_xor_sync(act, part, 1); };
        // e(n) = argmax_i <q_n, Lq_i>; a strict comparison in ascending i keeps
        // the lowest i on ties (eight independent dot products at a time)
        float best = -INFINITY;
        int e = 0;
        for (int i0 = 0; i0 < m; i0 += 8) {
            float l[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) l[u] = i0 + u < m ? both(sf_half_dot_f32(q, Lq + (i0 + u) * 64, h)) : -INFINITY;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (l[u] > best) {
                    best = l[u];
                    e = i0 + u;
                }
        }
        if (h == 0) a.route[row0 + n] = e;
        // one online softmax over the shared pairs, then the routed ones, eight
        // keys at a time: their logits, one rescale for the block's maximum,
        // their weights and values
        float M = -INFINITY, L = 0.f;
        float2 o[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) o[c] = make_float2(0.f, 0.f);
        auto fold = [&](float* sv) {  // sv[8]: logits (-inf: no key); on return, weights
            float bm = sv[0];
#pragma unroll
            for (int u = 1; u < 8; ++u) bm = fmaxf(bm, sv[u]);
            if (bm > M) {  // a new running maximum: rescale what was summed so far
                const float f = __expf(M - bm);
                L *= f;
#pragma unroll
                for (int c = 0; c < 16; ++c) o[c] = __fmul2_rn(o[c], make_float2(f, f));
                M = bm;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                sv[u] = __expf(sv[u] - M);
                L += sv[u];
            }
        };
        for (int i0 = 0; i0 < m; i0 += 8) {
            float sv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                sv[u] = i0 + u < m ? kTauSF * both(sf_half_dot_f32(q, Lq + (i0 + u) * 64, h)) : -INFINITY;
            fold(sv);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (i0 + u >= m) break;
                const float4* lv4 = reinterpret_cast<const float4*>(LV + (i0 + u) * 64 + 32 * h);
                const float2 p2 = make_float2(sv[u], sv[u]);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 v = lv4[c];
                    o[2 * c] = __ffma2_rn(p2, lo2(v), o[2 * c]);
                    o[2 * c + 1] = __ffma2_rn(p2, hi2(v), o[2 * c + 1]);
                }
            }
        }
        const uint8_t* ee = E + e * k;
        for (int j0 = 0; j0 < k; j0 += 8) {
            float sv[8];
            int rr[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                rr[u] = j0 + u < k ? ee[j0 + u] : 0;
                sv[u] = j0 + u < k ? kTauSF * both(sf_half_dot(q, Ks, rr[u], h)) : -INFINITY;
            }
            fold(sv);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (j0 + u >= k) break;
                const float2 p2 = make_float2(sv[u], sv[u]);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4*>(Vs + sf_chunk(rr[u], 4 * h + c));
                    o[4 * c] = __ffma2_rn(p2, bf2(w.x), o[4 * c]);
                    o[4 * c + 1] = __ffma2_rn(p2, bf2(w.y), o[4 * c + 1]);
                    o[4 * c + 2] = __ffma2_rn(p2, bf2(w.z), o[4 * c + 2]);
                    o[4 * c + 3] = __ffma2_rn(p2, bf2(w.w), o[4 * c + 3]);
                }
            }
        }
        const float inv = 1.f / L;
        uint4* dst = reinterpret_cast<uint4*>(a.out + (row0 + n) * 64 + 32 * h);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                __nv_bfloat162 b2 = __floats2bfloat162_rn(o[4 * c + u].x * inv, o[4 * c + u].y * inv);
                w[u] = *reinterpret_cast<uint32_t*>(&b2);
            }
            dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

}  // namespace

bool small_fused_applies(const Plan& p) {
    return p.shared && !p.split && p.s.s_route == 1 && p.s.N <= SF_MAX_N && p.s.m <= SF_MAX_M && p.s.k <= p.s.N &&
           p.s.BH < (int64_t(1) << 31) && sf_layout(static_cast<int>(p.s.N), p.s.m, p.s.k).total <= 232448;
}

cudaError_t launch_small_fused(const Plan& p, const __nv_bfloat16* Q, const __nv_bfloat16* K, const __nv_bfloat16* V,
                               __nv_bfloat16* out, int32_t* expert_idx, int32_t* route, float* lq_out, float* lv_out,
                               cudaStream_t st) {
    SFArgs a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.out = out;
    a.expert_idx = expert_idx;
    a.route = route;
    a.lq_out = lq_out;
    a.lv_out = lv_out;
    a.N = static_cast<int>(p.s.N);
    a.m = p.s.m;
    a.k = p.s.k;
    a.gh = p.s.gh;
    a.gw = p.s.gw;
    a.p = p.s.p;
    const size_t smem = sf_layout(a.N, a.m, a.k).total;
    cudaError_t e =
        cudaFuncSetAttribute(small_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    small_fused_kernel<<<static_cast<unsigned>(p.s.BH), SF_THREADS, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mita
