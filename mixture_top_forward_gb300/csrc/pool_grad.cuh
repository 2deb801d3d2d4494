// The pooling's share of dQ: token n of a head receives dLq_i / |window i|
// from every landmark window i that holds it (windows as in pool.cu: 1-D
// [floor(i N/m), ceil((i+1) N/m)), 2-D adaptive pooling of the token grid onto
// a p x p landmark grid; neighbouring windows overlap by at most one token or
// grid line, so only the windows around the token's own need checking).
#pragma once

#include "mita_internal.cuh"

namespace mita {

__device__ __forceinline__ void pool_window(int64_t N, int m, int i, int64_t& a, int64_t& b) {
    a = (static_cast<int64_t>(i) * N) / m;
    b = (static_cast<int64_t>(i + 1) * N + m - 1) / m;
}

// Calls f(i, 1 / |window i|) for each landmark window i of the head holding token n.
template <class F>
__device__ __forceinline__ void pool_windows_of(int64_t N, int gh, int gw, int p, int m, int64_t n, F&& f) {
    if (p == 0) {
        const int i0 = static_cast<int>((n * m) / N);
        for (int i = max(0, i0 - 2); i <= min(m - 1, i0 + 2); ++i) {
            int64_t a, b;
            pool_window(N, m, i, a, b);
            if (a <= n && n < b) f(i, 1.f / static_cast<float>(b - a));
        }
    } else {
        const int64_t y = n / gw, xx = n % gw;
        const int r0 = static_cast<int>((y * p) / gh), c0 = static_cast<int>((xx * p) / gw);
        for (int r = max(0, r0 - 2); r <= min(p - 1, r0 + 2); ++r) {
            int64_t ya, yb;
            pool_window(gh, p, r, ya, yb);
            if (!(ya <= y && y < yb)) continue;
            for (int cc = max(0, c0 - 2); cc <= min(p - 1, c0 + 2); ++cc) {
                int64_t xa, xb;
                pool_window(gw, p, cc, xa, xb);
                if (xa <= xx && xx < xb) f(r * p + cc, 1.f / static_cast<float>((yb - ya) * (xb - xa)));
            }
        }
    }
}

}  // namespace mita
