"""GPU-vs-oracle parity checks (the acceptance rule of the MiTA forward pass).

* Expert index sets: identical to the oracle's wherever the oracle's gap
  between the k-th and (k+1)-th landmark-key logit is >= 1e-3. Below that the
  GPU set must still be a valid top-k: k distinct ascending indices whose
  smallest oracle logit is within 1e-3 of the largest logit left out.
* Routes: identical wherever the oracle's top-2 margin is >= 1e-3; otherwise
  the GPU's landmark must score within 1e-3 of the best. With s routed
  experts per query: s distinct landmarks, the same set as the oracle's
  wherever its s-th/(s+1)-th margin is >= 1e-3 (else every chosen landmark
  within 1e-3 of every one left out), in descending order up to 1e-3, and in
  the oracle's exact order wherever all its margins are >= 1e-3.
* Outputs: compared with the oracle conditioned on the GPU's own routes and
  expert sets (so legal near-tie choices cost nothing): max-abs <= 2e-2 and
  mean-abs <= 2e-3 over all compared elements.
* Lq and LV (diagnostic): within 1e-4 and 1e-2 of the oracle. LV's bound
  comes from the tensor-core P.V product: the softmax weights enter it as
  bf16 (relative rounding 2^-9 each), so |LV error| <= max|V| * 2^-8 or so,
  about 1e-2 for unit-normal values.
All gaps and logits are tau-scaled, tau = 1/sqrt(d).
"""
from __future__ import annotations

import numpy as np

import synth

GAP = 1e-3
OUT_MAX, OUT_MEAN = 2e-2, 2e-3
LQ_TOL, LV_TOL = 1e-4, 1e-2


def to_device(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def out_rows(out_dev, rows):
    """float64 copy of the given flattened rows of a device bf16 [..., d] tensor."""
    import torch

    d = out_dev.shape[-1]
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=out_dev.device)
    sel = out_dev.reshape(-1, d).index_select(0, idx)
    return synth.bf16_to_f64(sel.view(torch.int16).cpu().numpy().view(np.uint16))


def run_gpu(q, k, v, gh, gw, m, kk, full_out=True, shared=True):
    """Runs the library on device copies. Small results come back as numpy;
    `out` stays on the device unless full_out (then float64 numpy).
    shared=False runs the routing-only ablation, which returns no Lq or LV."""
    import torch

    import mixture_top_forward_gb300 as M

    Q, K, V = to_device(q), to_device(k), to_device(v)
    if shared:
        out, eidx, route, lq, lv = M.mita_forward_aux(Q, K, V, gh, gw, m, kk)
    else:
        out, eidx, route = M.mita_forward_routed(Q, K, V, gh, gw, m, kk)
        lq = lv = None
    torch.cuda.synchronize()
    assert M.mita_sync_status() == 0
    del Q, K, V
    if full_out:
        out = synth.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    res = dict(out=out, expert_idx=eidx.cpu().numpy(), route=route.cpu().numpy(), lq=None, lv=None)
    if shared:
        res.update(lq=lq.cpu().numpy().astype(np.float64), lv=lv.cpu().numpy().astype(np.float64))
    return res


def check_experts(orc, lq_o, k, gpu_e, ora_e, gap, report):
    """gpu_e / ora_e: [BH, m, kk]; gap: [BH, m]; lq_o, k flattened per head."""
    BH, m, kk = gpu_e.shape
    N = k.shape[-2]
    exact = near = 0
    for bh in range(BH):
        for i in range(m):
            g = gpu_e[bh, i]
            assert np.all(np.diff(g) > 0), f"expert ({bh},{i}) not strictly ascending"
            assert g[0] >= 0 and g[-1] < N, f"expert ({bh},{i}) index out of range"
            if gap[bh, i] >= GAP:
                assert np.array_equal(g, ora_e[bh, i]), f"expert ({bh},{i}) differs (gap {gap[bh, i]:.3g})"
                exact += 1
            else:
                s = orc.scores(lq_o, k, bh, i)
                mask = np.zeros(N, bool)
                mask[g] = True
                worst_in = s[mask].min()
                best_out = s[~mask].max() if kk < N else -np.inf
                assert worst_in >= best_out - GAP, f"expert ({bh},{i}) not a 1e-3 top-k"
                near += 1
    report["experts_exact"] = report.get("experts_exact", 0) + exact
    report["experts_near_tie"] = report.get("experts_near_tie", 0) + near


def check_routes(q, lq_o, gpu_r, ora_r, rgap, which, report):
    """gpu_r/ora_r/rgap indexed like `which` (global query ids)."""
    d = q.shape[-1]
    qf = q.reshape(-1, d)
    m = lq_o.shape[-2]
    lqf = lq_o.reshape(-1, m, d)
    N = q.shape[-2]
    far = rgap >= GAP
    bad = np.nonzero(far & (gpu_r != ora_r))[0]
    assert bad.size == 0, f"{bad.size} routes differ outside near-ties, first query {which[bad[0]]}"
    idx = np.nonzero(~far)[0]
    for t in idx:
        n = which[t]
        logits = lqf[n // N] @ synth.bf16_to_f64(qf[n]) / np.sqrt(d)
        assert logits[gpu_r[t]] >= logits.max() - GAP, f"route of query {n} is not a 1e-3 argmax"
    report["routes_exact"] = report.get("routes_exact", 0) + int(far.sum())
    report["routes_near_tie"] = report.get("routes_near_tie", 0) + int((~far).sum())


def check_outputs(gpu_out, cond_out, report):
    err = np.abs(gpu_out - cond_out)
    mx, mean = float(err.max()), float(err.mean())
    report["out_max_abs"] = max(report.get("out_max_abs", 0.0), mx)
    report["out_mean_abs"] = mean
    assert mx <= OUT_MAX, f"max-abs output error {mx:.3g} > {OUT_MAX}"
    assert mean <= OUT_MEAN, f"mean-abs output error {mean:.3g} > {OUT_MEAN}"


def full_parity(orc, q, k, v, gh, gw, m, kk, gpu=None, shared=True):
    """Every element against the full oracle (small problems). shared=False:
    the routing-only ablation (no Lq/LV diagnostics: that path returns none)."""
    B, H, N, d = q.shape
    gpu = gpu or run_gpu(q, k, v, gh, gw, m, kk, shared=shared)
    ora = orc.forward(q, k, v, gh, gw, m, kk, shared=shared)
    rep = {}
    BH = B * H
    lq_o = ora["lq"].reshape(BH, m, d)
    if shared:
        assert np.max(np.abs(gpu["lq"].reshape(BH, m, d) - lq_o)) <= LQ_TOL, "Lq differs"
        rep["lv_max_abs"] = float(np.max(np.abs(gpu["lv"].reshape(BH, m, d) - ora["lv"].reshape(BH, m, d))))
        assert rep["lv_max_abs"] <= LV_TOL, f"LV differs by {rep['lv_max_abs']:.3g}"
    kf = k.reshape(BH, N, d)
    check_experts(orc, lq_o, kf, gpu["expert_idx"].reshape(BH, m, kk), ora["expert_idx"].reshape(BH, m, kk),
                  ora["gap"].reshape(BH, m), rep)
    which = np.arange(BH * N)
    check_routes(q, lq_o, gpu["route"].reshape(-1), ora["route"].reshape(-1), ora["rgap"].reshape(-1), which, rep)
    cond, ws = orc.attend(q, ora["lq"], ora["lv"], k, v, gpu["expert_idx"], gpu["route"], shared=shared)
    assert np.max(np.abs(ws - 1.0)) < 1e-9
    check_outputs(gpu["out"].reshape(BH, N, d), cond.reshape(BH, N, d), rep)
    rep["out_max_abs_unconditioned"] = float(np.max(np.abs(gpu["out"] - ora["out"])))
    return rep


def sampled_parity(orc, q, k, v, gh, gw, m, kk, gpu, heads, queries_per_head, seed=0, shared=True):
    """Full checks on a few heads; routes and outputs on sampled queries.
    shared=False: the routing-only ablation (no Lq/LV diagnostics)."""
    B, H, N, d = q.shape
    BH = B * H
    rng = np.random.default_rng(seed)
    rep = {"heads": list(map(int, heads))}
    qf, kf, vf = q.reshape(BH, N, d), k.reshape(BH, N, d), v.reshape(BH, N, d)
    for bh in heads:
        qs, ks, vs = qf[bh:bh + 1][None], kf[bh:bh + 1][None], vf[bh:bh + 1][None]
        lq_o = orc.landmarks(qs, gh, gw, m)  # [1,1,m,d]
        lv_o, e_o, gap = orc.scan(lq_o, ks, vs, kk)
        if shared:
            assert np.max(np.abs(gpu["lq"].reshape(BH, m, d)[bh] - lq_o[0, 0])) <= LQ_TOL, f"Lq differs in head {bh}"
            lv_err = float(np.max(np.abs(gpu["lv"].reshape(BH, m, d)[bh] - lv_o[0])))
            rep["lv_max_abs"] = max(rep.get("lv_max_abs", 0.0), lv_err)
            assert lv_err <= LV_TOL, f"LV differs by {lv_err:.3g} in head {bh}"
        g_e = gpu["expert_idx"].reshape(BH, m, kk)[bh:bh + 1]
        check_experts(orc, lq_o.reshape(1, m, d), ks.reshape(1, N, d), g_e, e_o, gap, rep)
        n_s = min(N, queries_per_head)
        which = np.sort(rng.choice(N, size=n_s, replace=False)) if n_s < N else np.arange(N)
        r_o, rg = orc.route(qs, lq_o, which=which)
        g_r = gpu["route"].reshape(BH, N)[bh]
        check_routes(qs, lq_o, g_r[which], r_o, rg, which, rep)
        cond, ws = orc.attend(qs, lq_o, lv_o.reshape(1, 1, m, d), ks, vs, g_e.reshape(1, 1, m, kk),
                              g_r.reshape(1, 1, N), which=which, shared=shared)
        check_outputs(out_rows(gpu["out"], bh * N + which), cond, rep)
    return rep


# ---------------------------------------------------------------------------
# s routed experts per query
# ---------------------------------------------------------------------------
def run_gpu_multi(q, k, v, gh, gw, m, kk, s, full_out=True):
    import torch

    import mixture_top_forward_gb300 as M

    Q, K, V = to_device(q), to_device(k), to_device(v)
    out, eidx, route = M.mita_forward_multi(Q, K, V, gh, gw, m, kk, s)
    torch.cuda.synchronize()
    assert M.mita_sync_status() == 0
    del Q, K, V
    if full_out:
        out = synth.bf16_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))
    return dict(out=out, expert_idx=eidx.cpu().numpy(), route=route.cpu().numpy())


def check_routes_multi(q, lq_o, gpu_r, ora_r, rgap, which, report):
    """gpu_r/ora_r [n, s] and rgap [n] indexed like `which` (global query ids)."""
    d = q.shape[-1]
    N = q.shape[-2]
    qf = q.reshape(-1, d)
    m = lq_o.shape[-2]
    lqf = lq_o.reshape(-1, m, d)
    n, s = gpu_r.shape
    exact = near = 0
    for t in range(n):
        g, o = gpu_r[t], ora_r[t]
        qi = which[t]
        assert np.all((g >= 0) & (g < m)) and len(set(g.tolist())) == s, f"routes of query {qi} not {s} distinct"
        lg = lqf[qi // N] @ synth.bf16_to_f64(qf[qi]) / np.sqrt(d)
        assert np.all(np.diff(lg[g]) <= GAP), f"routes of query {qi} not in descending order"
        if rgap[t] >= GAP:
            assert set(g.tolist()) == set(o.tolist()), f"route set of query {qi} differs (margin {rgap[t]:.3g})"
            if np.all(-np.diff(lg[o]) >= GAP):
                assert np.array_equal(g, o), f"route order of query {qi} differs"
            exact += 1
        else:
            out_mask = np.ones(m, bool)
            out_mask[g] = False
            best_out = lg[out_mask].max() if s < m else -np.inf
            assert lg[g].min() >= best_out - GAP, f"routes of query {qi} are not a 1e-3 top-{s}"
            near += 1
    report["routes_exact"] = report.get("routes_exact", 0) + exact
    report["routes_near_tie"] = report.get("routes_near_tie", 0) + near


def full_parity_multi(orc, q, k, v, gh, gw, m, kk, s, gpu=None):
    """Every element against the oracle's s-expert forward (small problems)."""
    B, H, N, d = q.shape
    BH = B * H
    gpu = gpu or run_gpu_multi(q, k, v, gh, gw, m, kk, s)
    ora = orc.forward_multi(q, k, v, gh, gw, m, kk, s)
    rep = {}
    lq_o = ora["lq"].reshape(BH, m, d)
    check_experts(orc, lq_o, k.reshape(BH, N, d), gpu["expert_idx"].reshape(BH, m, kk),
                  ora["expert_idx"].reshape(BH, m, kk), ora["gap"].reshape(BH, m), rep)
    check_routes_multi(q, lq_o, gpu["route"].reshape(-1, s), ora["route"].reshape(-1, s), ora["rgap"].reshape(-1),
                       np.arange(BH * N), rep)
    cond, ws = orc.attend_multi(q, ora["lq"], ora["lv"], k, v, gpu["expert_idx"], gpu["route"])
    assert np.max(np.abs(ws - 1.0)) < 1e-9
    check_outputs(gpu["out"].reshape(BH, N, d), cond.reshape(BH, N, d), rep)
    return rep


def sampled_parity_multi(orc, q, k, v, gh, gw, m, kk, s, gpu, heads, queries_per_head, seed=0):
    """Experts of a few heads in full; routes and outputs of sampled queries."""
    B, H, N, d = q.shape
    BH = B * H
    rng = np.random.default_rng(seed)
    rep = {"heads": list(map(int, heads))}
    qf, kf, vf = q.reshape(BH, N, d), k.reshape(BH, N, d), v.reshape(BH, N, d)
    for bh in heads:
        qs, ks, vs = qf[bh:bh + 1][None], kf[bh:bh + 1][None], vf[bh:bh + 1][None]
        lq_o = orc.landmarks(qs, gh, gw, m)
        lv_o, e_o, gap = orc.scan(lq_o, ks, vs, kk)
        g_e = gpu["expert_idx"].reshape(BH, m, kk)[bh:bh + 1]
        check_experts(orc, lq_o.reshape(1, m, d), ks.reshape(1, N, d), g_e, e_o, gap, rep)
        n_s = min(N, queries_per_head)
        which = np.sort(rng.choice(N, size=n_s, replace=False)) if n_s < N else np.arange(N)
        r_o, rg = orc.route_multi(qs, lq_o, s, which=which)
        g_r = gpu["route"].reshape(BH, N, s)[bh]
        check_routes_multi(qs, lq_o, g_r[which], r_o, rg, which, rep)
        cond, ws = orc.attend_multi(qs, lq_o, lv_o.reshape(1, 1, m, d), ks, vs, g_e.reshape(1, 1, m, kk),
                                    g_r.reshape(1, 1, N, s), which=which)
        check_outputs(out_rows(gpu["out"], bh * N + which), cond, rep)
    return rep
