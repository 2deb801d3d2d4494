// MiTA forward-pass oracle: plain, slow, fp64 CPU code.
//
// TEST INFRASTRUCTURE ONLY. It is called by the tests, by __graft_entry__.smoke()
// and by the CPU-baseline leg of bench.py; the library under
// mixture_top_forward_gb300/ never calls, links or loads it. It shares no code
// with the CUDA path.
//
// Sources (the method is described in prose; the formulas on the pages were lost
// in extraction, so each step below is the plain reading of that prose):
//  [P1] "NeurIPS'26：注意力也是FFN？从快权重出发，重新理解高效注意力"
//       (pro-axy-igame.com), section "用少量地标查询，同时构造全局概括与细节专家"
//  [P2] "NeurIPS 2026 | Mixture-of-Top-k 注意力：从快权重统一高效注意力…"
//       (shuwu5.cn), section "MiTA：用少量地标查询，同时完成压缩与专家构造"
//  [P3] "And attention is also FFN? …" (en.roboind.com), Figure 3 and
//       Algorithm 1 captions
//  [P4] "不止提速，还能兼容预训练模型：聊聊MiTA高效注意力" (ai.yesky.com),
//       section "跳出选择困境：把压缩和路由真正结合起来"
//
// Notation, per head (b,h): Q,K,V are N x d (bf16 inputs, widened exactly to
// double), tau = 1/sqrt(d) scales every logit, m landmarks, k keys per routed
// expert. Everything is computed in double; nothing is rounded to bf16.
//
// Readings taken where the prose is silent (the readings below):
//  * landmark windows: 1-D contiguous [floor(i N/m), ceil((i+1) N/m));
//    2-D adaptive pooling over a p x p landmark grid (m = p^2), rows
//    [floor(r gh/p), ceil((r+1) gh/p)), columns likewise with gw, landmarks and
//    tokens row-major;
//  * top-k ties go to the lower key index; the set is reported in ascending
//    key order;
//  * routing ties go to the lowest landmark index;
//  * the query-expert softmax is one softmax over the m shared logits and the
//    k routed logits together.
//
// Parity pins: every function here is checked in tests/test_oracle_pins.py
// against facts that do not come from this file (brute-force ranking, closed
// forms, invariants, a hand-worked example in tests/golden/).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

double widen(uint16_t h) {
    uint32_t u = static_cast<uint32_t>(h) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return static_cast<double>(f);
}

double dot_bf16(const double* a, const uint16_t* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * widen(b[c]);
    return s;
}

double dot_f64(const double* a, const double* b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

int isqrt_exact(int m) {
    int p = static_cast<int>(std::lround(std::sqrt(static_cast<double>(m))));
    while (p * p > m) --p;
    while ((p + 1) * (p + 1) <= m) ++p;
    return p * p == m ? p : -1;
}

int64_t floor_div(int64_t a, int64_t b) { return a / b; }           // a, b >= 0
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }  // a >= 0, b > 0

bool valid_shape(int64_t N, int d, int gh, int gw, int m) {
    if (N < 1 || d < 1 || m < 1 || m > N) return false;
    if (gh == 0 && gw == 0) return true;
    if (gh < 1 || gw < 1 || static_cast<int64_t>(gh) * gw != N) return false;
    int p = isqrt_exact(m);
    return p > 0 && p <= gh && p <= gw;
}

}  // namespace

extern "C" {

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

// Tokens pooled into landmark i ([P1], [P2]: landmarks are local average
// pools of the queries). Writes the token indices (row-major) when `tokens` is
// non-null and returns their count, or -1 for an invalid shape.
int64_t oracle_window(int64_t N, int gh, int gw, int m, int i, int64_t* tokens) {
    if (!valid_shape(N, 1, gh, gw, m) || i < 0 || i >= m) return -1;
    if (gh == 0) {
        int64_t a = floor_div(static_cast<int64_t>(i) * N, m);
        int64_t b = ceil_div(static_cast<int64_t>(i + 1) * N, m);
        if (tokens)
            for (int64_t t = a; t < b; ++t) tokens[t - a] = t;
        return b - a;
    }
    int p = isqrt_exact(m);
    int r = i / p, c = i % p;
    int64_t y0 = floor_div(static_cast<int64_t>(r) * gh, p), y1 = ceil_div(static_cast<int64_t>(r + 1) * gh, p);
    int64_t x0 = floor_div(static_cast<int64_t>(c) * gw, p), x1 = ceil_div(static_cast<int64_t>(c + 1) * gw, p);
    int64_t n = 0;
    for (int64_t y = y0; y < y1; ++y)
        for (int64_t x = x0; x < x1; ++x) {
            if (tokens) tokens[n] = y * gw + x;
            ++n;
        }
    return n;
}

// Stage 1, landmarks ([P1], [P2]): Lq_i = mean of the query rows in window i.
// q: [BH][N][d] bf16; lq: [BH][m][d] double.
int oracle_landmarks(const uint16_t* q, int64_t BH, int64_t N, int d, int gh, int gw, int m, double* lq) {
    if (!valid_shape(N, d, gh, gw, m)) return -1;
#pragma omp parallel for schedule(dynamic)
    for (int64_t li = 0; li < BH * m; ++li) {
        int64_t bh = li / m;
        int i = static_cast<int>(li % m);
        int64_t cnt = oracle_window(N, gh, gw, m, i, nullptr);
        std::vector<int64_t> tok(cnt);
        oracle_window(N, gh, gw, m, i, tok.data());
        double* out = lq + li * d;
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        for (int64_t t : tok) {
            const uint16_t* row = q + (bh * N + t) * d;
            for (int c = 0; c < d; ++c) out[c] += widen(row[c]);
        }
        for (int c = 0; c < d; ++c) out[c] /= static_cast<double>(cnt);
    }
    return 0;
}

// Landmark-to-key logits s_j = tau <Lq_i, K_j> for j = 0..N-1 of head bh.
int oracle_scores(const double* lq, const uint16_t* k, int64_t BH, int64_t N, int d, int m, int64_t bh, int i,
                  double* s) {
    if (bh < 0 || bh >= BH || i < 0 || i >= m) return -1;
    const double tau = 1.0 / std::sqrt(static_cast<double>(d));
    const double* a = lq + (bh * m + i) * d;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j) s[j] = tau * dot_bf16(a, k + (bh * N + j) * d, d);
    return 0;
}

// Stage 2, the landmark scan ([P2]; [P1]; [P3] Figure 3), for the landmarks
// listed in `which` (global ids bh*m + i; all BH*m when null):
//  * shared expert value LV_i = sum_j softmax_j(s) V_j, s_j = tau <Lq_i, K_j>
//    (landmark cross-attention over the whole sequence);
//  * routed expert E_i = the kk keys with the largest s_j (ties to the lower
//    key index), reported in ascending key order;
//  * gap_i = s_(kk) - s_(kk+1) in that order (+inf when kk = N), used by the
//    tests to tell exact ties from separable choices.
// Any of lv / eidx / gap may be null to skip that part.
int oracle_scan(const double* lq, const uint16_t* k, const uint16_t* v, int64_t BH, int64_t N, int d, int m, int kk,
                const int64_t* which, int64_t n_which, double* lv, int32_t* eidx, double* gap) {
    if (N < 1 || d < 1 || m < 1 || kk < 1 || kk > N) return -1;
    const int64_t n_items = which ? n_which : BH * m;
    const double tau = 1.0 / std::sqrt(static_cast<double>(d));
#pragma omp parallel for schedule(dynamic)
    for (int64_t it = 0; it < n_items; ++it) {
        const int64_t li = which ? which[it] : it;
        const int64_t bh = li / m;
        const double* a = lq + li * d;
        std::vector<double> s(N);
        for (int64_t j = 0; j < N; ++j) s[j] = tau * dot_bf16(a, k + (bh * N + j) * d, d);
        if (lv) {
            double mx = -std::numeric_limits<double>::infinity();
            for (int64_t j = 0; j < N; ++j) mx = std::max(mx, s[j]);
            std::vector<double> acc(d, 0.0);
            double z = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double w = std::exp(s[j] - mx);
                z += w;
                const uint16_t* row = v + (bh * N + j) * d;
                for (int c = 0; c < d; ++c) acc[c] += w * widen(row[c]);
            }
            for (int c = 0; c < d; ++c) lv[it * d + c] = acc[c] / z;
        }
        if (eidx || gap) {
            std::vector<int64_t> ord(N);
            for (int64_t j = 0; j < N; ++j) ord[j] = j;
            auto before = [&](int64_t x, int64_t y) { return s[x] > s[y] || (s[x] == s[y] && x < y); };
            const int64_t take = std::min<int64_t>(N, static_cast<int64_t>(kk) + 1);
            std::partial_sort(ord.begin(), ord.begin() + take, ord.end(), before);
            if (gap) gap[it] = (kk < N) ? s[ord[kk - 1]] - s[ord[kk]] : std::numeric_limits<double>::infinity();
            if (eidx) {
                std::vector<int64_t> sel(kk);
                for (int t = 0; t < kk; ++t) sel[t] = ord[t];
                std::sort(sel.begin(), sel.end());
                for (int t = 0; t < kk; ++t) eidx[it * kk + t] = static_cast<int32_t>(sel[t]);
            }
        }
    }
    return 0;
}

// Stage 3, routing ([P2]; [P1]): query n goes to the expert of the landmark it
// matches best, e = argmax_i tau <q_n, Lq_i> (first index on ties); rgap_n is
// the margin to the runner-up (+inf when m = 1). `which` lists global query
// ids bh*N + n (all BH*N when null); outputs are indexed like `which`.
int oracle_route(const uint16_t* q, const double* lq, int64_t BH, int64_t N, int d, int m, const int64_t* which,
                 int64_t n_which, int32_t* route, double* rgap) {
    if (N < 1 || d < 1 || m < 1) return -1;
    const int64_t n_items = which ? n_which : BH * N;
    const double tau = 1.0 / std::sqrt(static_cast<double>(d));
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t it = 0; it < n_items; ++it) {
        const int64_t qi = which ? which[it] : it;
        const int64_t bh = qi / N;
        std::vector<double> qd(d);
        for (int c = 0; c < d; ++c) qd[c] = widen(q[qi * d + c]);
        int best = 0;
        double bv = -std::numeric_limits<double>::infinity(), second = -std::numeric_limits<double>::infinity();
        for (int i = 0; i < m; ++i) {
            const double* a = lq + (bh * m + i) * d;
            double t = 0.0;
            for (int c = 0; c < d; ++c) t += qd[c] * a[c];
            t *= tau;
            if (t > bv) {
                second = bv;
                bv = t;
                best = i;
            } else if (t > second) {
                second = t;
            }
        }
        if (route) route[it] = best;
        if (rgap) rgap[it] = (m > 1) ? bv - second : std::numeric_limits<double>::infinity();
    }
    return 0;
}

// Stage 4, query-expert attention ([P2]; [P1]; [P3] Figure 3 and
// Algorithm 1): the shared expert's m pairs (keys Lq_i, values LV_i) and the
// routed expert's k pairs (keys K_j, values V_j, j in E_e, e = route of the
// query) are concatenated and weighted by ONE softmax over all m+k logits
// tau <q, key>. `route` is the full [BH][N] route array and `eidx` the full
// [BH][m][kk] expert array the output is conditioned on; `lv` is [BH][m][d].
// out[it][:] is the attention output of query which[it]; wsum[it] the sum of its
// m+k softmax weights (1 up to rounding). Null `which` means every query.
// shared = 0 gives the routing-only ablation the pages compare MiTA with
// ([P2] results section; [P3] Figure 4): no shared pairs, one softmax over
// the k routed logits alone.
int oracle_attend(const uint16_t* q, const double* lq, const double* lv, const uint16_t* k, const uint16_t* v,
                  const int32_t* eidx, const int32_t* route, int64_t BH, int64_t N, int d, int m, int kk,
                  const int64_t* which, int64_t n_which, int shared, double* out, double* wsum) {
    if (N < 1 || d < 1 || m < 1 || kk < 1 || kk > N) return -1;
    const int64_t n_items = which ? n_which : BH * N;
    const double tau = 1.0 / std::sqrt(static_cast<double>(d));
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(| : bad)
    for (int64_t it = 0; it < n_items; ++it) {
        const int64_t qi = which ? which[it] : it;
        const int64_t bh = qi / N;
        const int e = route[qi];
        if (e < 0 || e >= m) {
            bad |= 1;
            continue;
        }
        const int32_t* sel = eidx + (bh * m + e) * static_cast<int64_t>(kk);
        const int ms = shared ? m : 0;  // shared pairs taken
        std::vector<double> qd(d), logit(ms + kk);
        for (int c = 0; c < d; ++c) qd[c] = widen(q[qi * d + c]);
        for (int i = 0; i < ms; ++i) {
            const double* a = lq + (bh * m + i) * d;
            double t = 0.0;
            for (int c = 0; c < d; ++c) t += qd[c] * a[c];
            logit[i] = tau * t;
        }
        for (int j = 0; j < kk; ++j) {
            if (sel[j] < 0 || sel[j] >= N) {
                bad |= 1;
                logit[ms + j] = 0.0;
                continue;
            }
            const uint16_t* row = k + (bh * N + sel[j]) * d;
            double t = 0.0;
            for (int c = 0; c < d; ++c) t += qd[c] * widen(row[c]);
            logit[ms + j] = tau * t;
        }
        double mx = -std::numeric_limits<double>::infinity();
        for (double t : logit) mx = std::max(mx, t);
        std::vector<double> acc(d, 0.0);
        double z = 0.0;
        for (int i = 0; i < ms; ++i) {
            double w = std::exp(logit[i] - mx);
            z += w;
            const double* val = lv + (bh * m + i) * d;
            for (int c = 0; c < d; ++c) acc[c] += w * val[c];
        }
        for (int j = 0; j < kk; ++j) {
            double w = std::exp(logit[ms + j] - mx);
            z += w;
            int64_t jj = (sel[j] >= 0 && sel[j] < N) ? sel[j] : 0;
            const uint16_t* row = v + (bh * N + jj) * d;
            for (int c = 0; c < d; ++c) acc[c] += w * widen(row[c]);
        }
        for (int c = 0; c < d; ++c) out[it * d + c] = acc[c] / z;
        if (wsum) {
            double ws = 0.0;
            for (double t : logit) ws += std::exp(t - mx) / z;
            wsum[it] = ws;
        }
    }
    return bad ? -1 : 0;
}

// Stage 3 with s experts per query. The pages use one routed expert per
// query and call that "the s = 1 configuration" ([P2], end of section
// "MiTA：…"), which names the general form without describing it. Reading
// taken: a query takes the s landmarks with the highest logits tau <q, Lq_i>,
// listed highest first, ties to the lower landmark index (s = 1 is
// oracle_route). route is [n_items][s]; rgap[it] is the s-th highest logit
// minus the (s+1)-th (+inf when s = m), the margin that decides the set.
int oracle_route_multi(const uint16_t* q, const double* lq, int64_t BH, int64_t N, int d, int m, int s,
                       const int64_t* which, int64_t n_which, int32_t* route, double* rgap) {
    if (N < 1 || d < 1 || m < 1 || s < 1 || s > m) return -1;
    const int64_t n_items = which ? n_which : BH * N;
    const double tau = 1.0 / std::sqrt(static_cast<double>(d));
#pragma omp parallel for schedule(dynamic, 256)
    for (int64_t it = 0; it < n_items; ++it) {
        const int64_t qi = which ? which[it] : it;
        const int64_t bh = qi / N;
        std::vector<double> qd(d), sc(m);
        for (int c = 0; c < d; ++c) qd[c] = widen(q[qi * d + c]);
        for (int i = 0; i < m; ++i) sc[i] = tau * dot_f64(lq + (bh * m + i) * d, qd.data(), d);
        std::vector<int> order(m);
        for (int i = 0; i < m; ++i) order[i] = i;
        // highest logit first; a stable sort keeps equal logits in index order
        std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return sc[x] > sc[y]; });
        for (int u = 0; u < s; ++u) route[it * s + u] = order[u];
        if (rgap) rgap[it] = s < m ? sc[order[s - 1]] - sc[order[s]] : std::numeric_limits<double>::infinity();
    }
    return 0;
}

// Stage 4 with s experts per query: the m shared pairs and the keys of the s
// routed experts under ONE softmax, as for s = 1 ([P2] "MiTA：…", unified
// softmax). Reading taken: the routed part is the UNION of the s experts' key
// sets, so a key that two of the chosen experts hold enters once (attention
// over a set of keys; counting it twice would weight it twice). route is the
// full [BH][N][s] array; everything else as in oracle_attend (shared = 1).
int oracle_attend_multi(const uint16_t* q, const double* lq, const double* lv, const uint16_t* k, const uint16_t* v,
                        const int32_t* eidx, const int32_t* route, int64_t BH, int64_t N, int d, int m, int kk, int s,
                        const int64_t* which, int64_t n_which, double* out, double* wsum) {
    if (N < 1 || d < 1 || m < 1 || kk < 1 || kk > N || s < 1 || s > m) return -1;
    const int64_t n_items = which ? n_which : BH * N;
    const double tau = 1.0 / std::sqrt(static_cast<double>(d));
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(| : bad)
    for (int64_t it = 0; it < n_items; ++it) {
        const int64_t qi = which ? which[it] : it;
        const int64_t bh = qi / N;
        std::vector<int32_t> keys;
        for (int u = 0; u < s; ++u) {
            const int e = route[qi * s + u];
            if (e < 0 || e >= m) {
                bad |= 1;
                continue;
            }
            const int64_t row0 = (bh * m + e) * static_cast<int64_t>(kk);  // expert e's kk key indices
            for (int j = 0; j < kk; ++j) {
                if (eidx[row0 + j] < 0 || eidx[row0 + j] >= N)
                    bad |= 1;
                else
                    keys.push_back(eidx[row0 + j]);
            }
        }
        std::sort(keys.begin(), keys.end());
        keys.erase(std::unique(keys.begin(), keys.end()), keys.end());
        const int64_t nk = static_cast<int64_t>(keys.size());
        std::vector<double> qd(d), logit(m + nk);
        for (int c = 0; c < d; ++c) qd[c] = widen(q[qi * d + c]);
        for (int i = 0; i < m; ++i) logit[i] = tau * dot_f64(lq + (bh * m + i) * d, qd.data(), d);
        for (int64_t j = 0; j < nk; ++j) {
            const uint16_t* row = k + (bh * N + keys[j]) * d;
            double t = 0.0;
            for (int c = 0; c < d; ++c) t += qd[c] * widen(row[c]);
            logit[m + j] = tau * t;
        }
        double mx = -std::numeric_limits<double>::infinity();
        for (double t : logit) mx = std::max(mx, t);
        std::vector<double> acc(d, 0.0);
        double z = 0.0;
        for (int64_t j = 0; j < m + nk; ++j) {  // shared pairs first, then the union's keys
            const double p = std::exp(logit[j] - mx);
            z += p;
            if (j < m) {
                const double* lvj = lv + (bh * m + j) * d;
                for (int c = 0; c < d; ++c) acc[c] += p * lvj[c];
            } else {
                const uint16_t* vrow = v + (bh * N + keys[j - m]) * d;
                for (int c = 0; c < d; ++c) acc[c] += p * widen(vrow[c]);
            }
        }
        for (int c = 0; c < d; ++c) out[it * d + c] = acc[c] / z;
        if (wsum) {
            double ws = 0.0;
            for (double t : logit) ws += std::exp(t - mx) / z;
            wsum[it] = ws;
        }
    }
    return bad ? -1 : 0;
}

// The whole forward pass, stages 1-4 in order, with the oracle's own routes
// and experts. Buffers: out [BH][N][d], eidx [BH][m][kk], route [BH][N],
// lq/lv [BH][m][d], gap [BH][m], rgap [BH][N], wsum [BH][N]; the last five
// may be null. shared = 0: the routing-only ablation (see oracle_attend).
int oracle_forward(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t B, int64_t H, int64_t N, int d,
                   int gh, int gw, int m, int kk, int shared, double* out, int32_t* eidx, int32_t* route,
                   double* lq_out, double* lv_out, double* gap, double* rgap, double* wsum) {
    if (B < 0 || H < 0) return -1;
    const int64_t BH = B * H;
    if (BH == 0) return 0;
    if (!valid_shape(N, d, gh, gw, m) || kk < 1 || kk > N) return -1;
    std::vector<double> lq(lq_out ? 0 : BH * m * d), lv(lv_out ? 0 : BH * m * d);
    double* L = lq_out ? lq_out : lq.data();
    double* LV = lv_out ? lv_out : lv.data();
    if (oracle_landmarks(q, BH, N, d, gh, gw, m, L)) return -1;
    if (oracle_scan(L, k, v, BH, N, d, m, kk, nullptr, 0, LV, eidx, gap)) return -1;
    if (oracle_route(q, L, BH, N, d, m, nullptr, 0, route, rgap)) return -1;
    return oracle_attend(q, L, LV, k, v, eidx, route, BH, N, d, m, kk, nullptr, 0, shared, out, wsum);
}

}  // extern "C"
