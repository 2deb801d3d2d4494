// Stage 4: query-expert attention on the tensor cores (tcgen05, TMEM).
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造", and Figure 3 / Algorithm 1 of
// "And attention is also FFN? …" (en.roboind.com): a query routed to expert e
// attends to the m shared pairs (keys Lq_i, values LV_i) and the k routed pairs
// (K_j, V_j, j in E_e) under one softmax over all m+k logits; the page's
// implementation groups queries by expert and combines by online softmax.
//
// Work: persistent CTAs walk a contiguous range of the flat, expert-ordered
// item list (<= 128 queries of one expert per item). Whenever the expert
// changes, the CTA stages the expert's key list [Lq_0..Lq_{m-1}, K_e] and
// value list [LV_0..LV_{m-1}, V_e] (bf16, 128-byte swizzled rows, zero padded
// to whole 128-row blocks) in shared memory with cp.async gathers. NWG
// warpgroups each take one item of a round (consecutive items of the same
// expert) and run it on their own:
//   Q rows (gathered by the grouping permutation) -> shared memory;
//   for each 128-key block j: S = Q . keys_j^T into TMEM (4 MMAs, K = 64);
//   each thread owns one query row: it loads its 128 logits, updates the
//   running max (kept while it grows by < 2^8, so O rarely needs rescaling),
//   forms p = 2^(s tau log2e - max) in registers and writes P (bf16) to
//   shared memory; O += P . values_j into TMEM (8 MMAs, N = 64).
//   The next block's S MMA is issued as soon as every thread has read S.
//   Epilogue: O / rowsum -> bf16 -> the query's output row.
// MMAs are issued by one thread of the warpgroup and tracked with tcgen05
// commits on mbarriers; every wait is bounded (umma.cuh), and its outcome is
// made uniform over the warpgroup before anyone acts on it, so a timeout ends
// the item in every thread and the kernel still reaches its TMEM release.
#include "umma.cuh"

namespace mita {

namespace {

using namespace umma;

constexpr float kC = 0.125f * kLog2e;  // tau * log2(e), tau = 1/sqrt(64)
constexpr float kLazy = 8.0f;          // keep the running max while the new one is within 2^8
constexpr uint32_t kIdescS = idesc_bf16(128, 128, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, true);

struct Args {
    const __nv_bfloat16* Q;
    const __nv_bfloat16* K;
    const __nv_bfloat16* V;
    const __nv_bfloat16* lqhi;
    const __nv_bfloat16* lvbf;
    const int4* items;
    const int* nitems;
    const int* perm;
    const int32_t* expert_idx;
    __nv_bfloat16* out;
    int* status;
    int64_t N;
    int m, k, nblk;
};

__device__ __forceinline__ void zero16(uint8_t* p) { *reinterpret_cast<uint4*>(p) = make_uint4(0, 0, 0, 0); }

// Stages the key and value lists of expert (bh, e); all NT threads call it.
template <int NT>
__device__ void stage_expert(const Args& a, int64_t bh, int e, uint8_t* keys, uint8_t* vals) {
    const int rows = a.nblk * 128;
    const int32_t* sel = a.expert_idx + (bh * a.m + e) * static_cast<int64_t>(a.k);
    const uint32_t kb = smem_u32(keys), vb = smem_u32(vals);
    for (int x = threadIdx.x; x < rows * 8; x += NT) {
        const int row = x >> 3, c = x & 7;
        const uint32_t off = swz128(row, c);
        if (row < a.m) {
            const int64_t src = (bh * a.m + row) * D + c * 8;
            cp_async16(kb + off, a.lqhi + src);
            cp_async16(vb + off, a.lvbf + src);
        } else if (row < a.m + a.k) {
            const int64_t src = (bh * a.N + sel[row - a.m]) * D + c * 8;
            cp_async16(kb + off, a.K + src);
            cp_async16(vb + off, a.V + src);
        } else {
            zero16(keys + off);
            zero16(vals + off);
        }
    }
    cp_async_wait_all();
    fence_proxy_async();
}

// One work item on warpgroup `wg` (thread t = its query row).
__device__ void run_item(const Args& a, int4 it, int wg, int t, uint8_t* keys, uint8_t* vals, uint8_t* qb,
                         uint8_t* pb, uint64_t* barS, uint64_t* barO, uint32_t tS, uint32_t tO, uint32_t& ps,
                         uint32_t& po) {
    const int e = it.x, start = it.y, len = it.z;
    const int64_t bh = it.w;
    (void)e;
    const uint32_t lane_off = static_cast<uint32_t>((t >> 5) * 32) << 16;
    const uint32_t qa = smem_u32(qb), pa = smem_u32(pb), ka = smem_u32(keys), va = smem_u32(vals);
    const int nkeys = a.m + a.k;
    int n = 0;
    if (t < len) {
        n = a.perm[bh * a.N + start + t];
        const __nv_bfloat16* src = a.Q + (bh * a.N + n) * D;
#pragma unroll
        for (int c = 0; c < 8; ++c) cp_async16(qa + swz128(t, c), src + c * 8);
    } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) zero16(qb + swz128(t, c));
    }
    cp_async_wait_all();
    fence_proxy_async();
    named_bar(1 + wg, 128);

    auto issue_s = [&](int j) {
#pragma unroll
        for (int s = 0; s < 4; ++s)
            mma_ss(tS, sdesc_sw128(qa + s * 32), sdesc_sw128(ka + j * 16384 + s * 32), kIdescS, s > 0);
        mma_commit(barS);
    };
    auto issue_pv = [&](int j) {
#pragma unroll
        for (int s = 0; s < 8; ++s)
            mma_ss(tO, sdesc_sw128(pa + (s >> 2) * 16384 + (s & 3) * 32), sdesc_sw128(va + j * 16384 + s * 2048),
                   kIdescPV, (j > 0 || s > 0) ? 1u : 0u);
        mma_commit(barO);
    };

    if (t == 0) {
        tc_fence_after();
        issue_s(0);
    }
    float mrun = -INFINITY, lrun = 0.f;
    for (int j = 0; j < a.nblk; ++j) {
        if (!named_bar_and(1 + wg, 128, mbar_wait(barS, ps, a.status))) return;
        ps ^= 1;
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + lane_off + q * 32, s + q * 32);
        tmem_ld_wait();
        tc_fence_before();
        named_bar(1 + wg, 128);
        if (t == 0 && j + 1 < a.nblk) {
            tc_fence_after();
            issue_s(j + 1);
        }
        const int valid = min(128, nkeys - j * 128);
        float bmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
            s[c] = c < valid ? s[c] * kC : -INFINITY;
            bmax = fmaxf(bmax, s[c]);
        }
        const float mnew = (bmax > mrun + kLazy) ? bmax : mrun;
        const float alpha = exp2f(mrun - mnew);  // 0 on the first block, 1 when the max is kept
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
            s[c] = exp2f(s[c] - mnew);
            sum += s[c];
        }
        lrun = lrun * alpha + sum;
        if (j > 0) {
            if (!named_bar_and(1 + wg, 128, mbar_wait(barO, po, a.status))) return;
            po ^= 1;
            tc_fence_after();
            if (__any_sync(0xffffffffu, alpha != 1.f)) {  // rescale this warp's rows of O
                float o[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    tmem_ld32(tO + lane_off + h * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] *= alpha;
                    tmem_st32(tO + lane_off + h * 32, o);
                }
                tmem_st_wait();
            }
        }
#pragma unroll
        for (int g = 0; g < 16; ++g) {
            uint4 pk;
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
            for (int u = 0; u < 4; ++u) h2[u] = __floats2bfloat162_rn(s[8 * g + 2 * u], s[8 * g + 2 * u + 1]);
            *reinterpret_cast<uint4*>(pb + (g >> 3) * 16384 + swz128(t, g & 7)) = pk;
        }
        fence_proxy_async();
        tc_fence_before();
        named_bar(1 + wg, 128);
        if (t == 0) {
            tc_fence_after();
            issue_pv(j);
        }
        mrun = mnew;
    }
    if (!named_bar_and(1 + wg, 128, mbar_wait(barO, po, a.status))) return;
    po ^= 1;
    tc_fence_after();
    float o[64];
    tmem_ld32(tO + lane_off, o);
    tmem_ld32(tO + lane_off + 32, o + 32);
    tmem_ld_wait();
    tc_fence_before();
    if (t < len) {
        const float inv = 1.f / lrun;
        uint4* dst = reinterpret_cast<uint4*>(a.out + (bh * a.N + n) * D);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 pk;
            __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                h2[u] = __floats2bfloat162_rn(o[8 * c + 2 * u] * inv, o[8 * c + 2 * u + 1] * inv);
            dst[c] = pk;
        }
    }
}

template <int NWG>
__global__ void __launch_bounds__(NWG * 128) expert_tc_kernel(Args a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t barS[NWG], barO[NWG];
    __shared__ uint32_t tmem_base;
    constexpr int NT = NWG * 128;
    constexpr uint32_t kCols = NWG == 2 ? 512 : 256;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* keys = base;
    uint8_t* vals = keys + a.nblk * 16384;
    uint8_t* qbuf = vals + a.nblk * 16384;
    uint8_t* pbuf = qbuf + NWG * 16384;

    const int tid = threadIdx.x, wg = tid >> 7, t = tid & 127;
    if (tid == 0) {
        for (int w = 0; w < NWG; ++w) {
            mbar_init(&barS[w], 1);
            mbar_init(&barO[w], 1);
        }
        fence_barrier_init();
    }
    if (tid < 32) tmem_alloc(&tmem_base, kCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = tmem_base + wg * 256, tO = tS + 128;

    const int total = *a.nitems;
    const int i0 = static_cast<int>(static_cast<int64_t>(total) * blockIdx.x / gridDim.x);
    const int i1 = static_cast<int>(static_cast<int64_t>(total) * (blockIdx.x + 1) / gridDim.x);
    int staged_bh = -1, staged_e = -1;
    uint32_t ps = 0, po = 0;
    for (int r = i0; r < i1;) {
        const int4 it0 = a.items[r];
        int cnt = 1;
        int4 it1 = it0;
        if (NWG == 2 && r + 1 < i1) {
            it1 = a.items[r + 1];
            if (it1.x == it0.x && it1.w == it0.w) cnt = 2;
        }
        if (it0.w != staged_bh || it0.x != staged_e) {
            __syncthreads();  // every warpgroup is done with the previous expert
            stage_expert<NT>(a, it0.w, it0.x, keys, vals);
            __syncthreads();
            staged_bh = it0.w;
            staged_e = it0.x;
        }
        if (wg < cnt)
            run_item(a, wg == 0 ? it0 : it1, wg, t, keys, vals, qbuf + wg * 16384, pbuf + wg * 32768, &barS[wg],
                     &barO[wg], tS, tO, ps, po);
        r += cnt;
    }
    tc_fence_before();
    __syncthreads();
    if (tid < 32) tmem_free(tmem_base, kCols);
}

template <int NWG>
size_t smem_bytes(int nblk) {
    return 1024 + static_cast<size_t>(nblk) * 32768 + NWG * (16384 + 32768);
}

}  // namespace

bool expert_tc_supported(const Plan& p) {
    const int nkeys = p.s.m + p.s.k;
    return nkeys <= 512 && smem_bytes<2>((nkeys + 127) / 128) <= 232448;
}

cudaError_t launch_expert_tc(const Plan& p, const Work& w, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                             const __nv_bfloat16* V, const int32_t* expert_idx, __nv_bfloat16* out,
                             cudaStream_t st) {
    Args a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.lqhi = w.lqhi;
    a.lvbf = w.lvbf;
    a.items = w.items;
    a.nitems = w.nitems;
    a.perm = w.perm;
    a.expert_idx = expert_idx;
    a.out = out;
    a.status = w.status;
    a.N = p.s.N;
    a.m = p.s.m;
    a.k = p.s.k;
    a.nblk = (p.s.m + p.s.k + 127) / 128;
    const int sms = device_sms();
    cudaError_t e;
    if (a.nblk <= 2) {  // small key lists: one warpgroup per CTA, two CTAs per SM
        const size_t sm = smem_bytes<1>(a.nblk);
        if ((e = cudaFuncSetAttribute(expert_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(sm))) != cudaSuccess)
            return e;
        expert_tc_kernel<1><<<2 * sms, 128, sm, st>>>(a);
    } else {
        const size_t sm = smem_bytes<2>(a.nblk);
        if ((e = cudaFuncSetAttribute(expert_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(sm))) != cudaSuccess)
            return e;
        expert_tc_kernel<2><<<sms, 256, sm, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace mita
