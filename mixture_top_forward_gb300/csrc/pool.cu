// Stage 1: landmark queries by local average pooling.
//
// "NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), section
// "MiTA：用少量地标查询，同时完成压缩与专家构造": the m landmark queries are
// obtained by simple local average pooling of the queries. Windows: 1-D
// contiguous [floor(i N/m), ceil((i+1) N/m)); 2-D adaptive pooling of the
// token grid onto a p x p landmark grid (m = p^2), rows
// [floor(r gh/p), ceil((r+1) gh/p)), columns likewise.
//
// One CTA per (head, landmark), flattened into blockIdx.x. 256 threads: 8 threads cover one 128-byte
// query row with 16-byte loads, 32 rows are in flight per step. Sums are kept
// in fp32 registers and reduced through shared memory in a fixed order, so the
// result is deterministic. Outputs: Lq in fp32 and as a bf16 hi/lo pair
// (hi = bf16(Lq), lo = bf16(Lq - hi)) for the tensor-core consumers.
#include "mita_internal.cuh"

namespace mita {

namespace {

__global__ void __launch_bounds__(256) pool_kernel(const __nv_bfloat16* __restrict__ Q, int64_t N, int gh, int gw,
                                                   int p, int m, float* __restrict__ lq32,
                                                   __nv_bfloat16* __restrict__ lqhi,
                                                   __nv_bfloat16* __restrict__ lqlo) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    __shared__ float red[32][D + 4];
    const int i = static_cast<int>(blockIdx.x % static_cast<unsigned>(m));
    const int64_t bh = blockIdx.x / static_cast<unsigned>(m);
    int64_t t0, cnt;
    int64_t y0 = 0, x0 = 0, wdt = 1;
    if (p == 0) {
        t0 = (static_cast<int64_t>(i) * N) / m;
        int64_t t1 = (static_cast<int64_t>(i + 1) * N + m - 1) / m;
        cnt = t1 - t0;
    } else {
        const int r = i / p, c = i % p;
        y0 = (static_cast<int64_t>(r) * gh) / p;
        const int64_t y1 = (static_cast<int64_t>(r + 1) * gh + p - 1) / p;
        x0 = (static_cast<int64_t>(c) * gw) / p;
        const int64_t x1 = (static_cast<int64_t>(c + 1) * gw + p - 1) / p;
        wdt = x1 - x0;
        cnt = (y1 - y0) * wdt;
        t0 = 0;
    }
    const __nv_bfloat16* Qh = Q + bh * N * D;
    const int col = (threadIdx.x & 7) * 8;
    const int slot = threadIdx.x >> 3;
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
    auto token = [&](int64_t t) -> int64_t {
        return p == 0 ? t0 + t : (y0 + t / wdt) * gw + x0 + t % wdt;
    };
    int64_t t = slot;
    for (; t + 96 < cnt; t += 128) {  // 4 rows per thread in flight
        uint4 r0 = ldg_nc_v4(Qh + token(t) * D + col);
        uint4 r1 = ldg_nc_v4(Qh + token(t + 32) * D + col);
        uint4 r2 = ldg_nc_v4(Qh + token(t + 64) * D + col);
        uint4 r3 = ldg_nc_v4(Qh + token(t + 96) * D + col);
        float f[8];
        unpack_bf16x8(r0, f);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += f[c];
        unpack_bf16x8(r1, f);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += f[c];
        unpack_bf16x8(r2, f);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += f[c];
        unpack_bf16x8(r3, f);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += f[c];
    }
    for (; t < cnt; t += 32) {
        float f[8];
        unpack_bf16x8(ldg_nc_v4(Qh + token(t) * D + col), f);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += f[c];
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) red[slot][col + c] = acc[c];
    __syncthreads();
    if (threadIdx.x < D) {
        const int c = threadIdx.x;
        float s = 0.f;
#pragma unroll 8
        for (int r = 0; r < 32; ++r) s += red[r][c];
        const float mean = s / static_cast<float>(cnt);
        const int64_t o = (bh * m + i) * D + c;
        lq32[o] = mean;
        const __nv_bfloat16 hi = __float2bfloat16_rn(mean);
        lqhi[o] = hi;
        lqlo[o] = __float2bfloat16_rn(mean - __bfloat162float(hi));
    }
}

// Small windows (at most 128 tokens): one warp per landmark, 8 landmarks
// per CTA. Lanes 8s .. 8s + 7 cover one query row with 16-byte
// loads (4 rows per step, all of a window's loads in flight), the 4 row
// slots are summed by two shuffles in a fixed order.
__global__ void __launch_bounds__(256) pool_warp_kernel(const __nv_bfloat16* __restrict__ Q, int64_t N, int gh, int gw,
                                                        int p, int m, int64_t rows, float* __restrict__ lq32,
                                                        __nv_bfloat16* __restrict__ lqhi,
                                                        __nv_bfloat16* __restrict__ lqlo) {
    dep_entry();  // (launched by launch_dep: the kernel before may still be finishing)
    const int lane = threadIdx.x & 31;
    const int64_t wg = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (wg >= rows) return;  // (warp-uniform; no block-wide barrier)
    const int i = static_cast<int>(wg % m);
    const int64_t bh = wg / m;
    int64_t t0 = 0, cnt, y0 = 0, x0 = 0, wdt = 1;
    if (p == 0) {
        t0 = (static_cast<int64_t>(i) * N) / m;
        cnt = (static_cast<int64_t>(i + 1) * N + m - 1) / m - t0;
    } else {
        const int r = i / p, c = i % p;
        y0 = (static_cast<int64_t>(r) * gh) / p;
        const int64_t y1 = (static_cast<int64_t>(r + 1) * gh + p - 1) / p;
        x0 = (static_cast<int64_t>(c) * gw) / p;
        wdt = (static_cast<int64_t>(c + 1) * gw + p - 1) / p - x0;
        cnt = (y1 - y0) * wdt;
    }
    const __nv_bfloat16* Qh = Q + bh * N * D;
    const int col = (lane & 7) * 8, slot = lane >> 3;
    auto token = [&](int64_t t) -> int64_t { return p == 0 ? t0 + t : (y0 + t / wdt) * gw + x0 + t % wdt; };
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.f;
    // eight 16-byte loads per lane in flight (a 64-token window: two rounds)
    int64_t t = slot;
    for (; t + 28 < cnt; t += 32) {
        uint4 raw[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) raw[u] = ldg_nc_v4(Qh + token(t + 4 * u) * D + col);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float f[8];
            unpack_bf16x8(raw[u], f);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] += f[c];
        }
    }
    for (; t < cnt; t += 4) {
        float f[8];
        unpack_bf16x8(ldg_nc_v4(Qh + token(t) * D + col), f);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += f[c];
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 8);
        acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 16);
    }
    if (slot == 0) {
        float v[8];
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = acc[c] / static_cast<float>(cnt);
#pragma unroll
        for (int c = 0; c < 8; c += 2) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[c], v[c + 1]);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(v[c] - __low2float(h2), v[c + 1] - __high2float(h2));
            hw[c >> 1] = *reinterpret_cast<const uint32_t*>(&h2);
            lw[c >> 1] = *reinterpret_cast<const uint32_t*>(&l2);
        }
        const int64_t o = (bh * m + i) * D + col;
        reinterpret_cast<float4*>(lq32 + o)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(lq32 + o)[1] = make_float4(v[4], v[5], v[6], v[7]);
        *reinterpret_cast<uint4*>(lqhi + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(lqlo + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
}

}  // namespace

cudaError_t launch_pool(const Plan& p, const Work& w, const __nv_bfloat16* Q, cudaStream_t st) {
    // the largest window: 1-D ceil(N / m) + 1 tokens; 2-D (ceil(gh / p) + 1) (ceil(gw / p) + 1);
    // long windows keep a whole CTA per landmark
    const int64_t win = p.s.p == 0 ? (p.s.N + p.s.m - 1) / p.s.m + 1
                                   : ((p.s.gh + p.s.p - 1) / p.s.p + 1) * ((p.s.gw + p.s.p - 1) / p.s.p + 1);
    const int64_t rows = p.s.BH * p.s.m;
    if (win <= 128) {
        return launch_dep(pool_warp_kernel, dim3(static_cast<unsigned>((rows + 7) / 8)), dim3(256), 0, st, Q, p.s.N,
                          p.s.gh, p.s.gw, p.s.p, p.s.m, rows, w.lq32, w.lqhi, w.lqlo);
    }
    const unsigned grid = static_cast<unsigned>(rows);
    return launch_dep(pool_kernel, dim3(grid), dim3(256), 0, st, Q, p.s.N, p.s.gh, p.s.gw, p.s.p, p.s.m, w.lq32,
                      w.lqhi, w.lqlo);
}

}  // namespace mita
