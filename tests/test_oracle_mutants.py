"""Plant a plausible mistake in a copy of the oracle and check that at least
one pin fails on it: evidence that the pins would catch such a mistake in the
real oracle. The copies are built in a temporary directory; the oracle's own
source is never modified."""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mita_oracle.cpp")

# (name, text in mita_oracle.cpp, replacement)
MUTANTS = [
    ("scan drops tau", "s[j] = tau * dot_bf16(a, k + (bh * N + j) * d, d);\n        if (lv)",
     "s[j] = dot_bf16(a, k + (bh * N + j) * d, d);\n        if (lv)"),
    ("top-k keeps smallest", "return s[x] > s[y] ||", "return s[x] < s[y] ||"),
    ("top-k ties to higher index", "(s[x] == s[y] && x < y)", "(s[x] == s[y] && x > y)"),
    ("1-D window end floored", "int64_t b = ceil_div(static_cast<int64_t>(i + 1) * N, m);",
     "int64_t b = floor_div(static_cast<int64_t>(i + 1) * N, m);"),
    ("2-D rows and columns swapped", "int r = i / p, c = i % p;", "int r = i % p, c = i / p;"),
    ("mean over count+1", "out[c] /= static_cast<double>(cnt);", "out[c] /= static_cast<double>(cnt + 1);"),
    ("LV softmax sign", "double w = std::exp(s[j] - mx);", "double w = std::exp(mx - s[j]);"),
    ("LV reads head 0 values", "const uint16_t* row = v + (bh * N + j) * d;\n                for (int c = 0; c < d; ++c) acc[c] += w * widen(row[c]);\n            }\n            for (int c = 0; c < d; ++c) lv[",
     "const uint16_t* row = v + (j) * d;\n                for (int c = 0; c < d; ++c) acc[c] += w * widen(row[c]);\n            }\n            for (int c = 0; c < d; ++c) lv["),
    ("route ties to last", "if (t > bv) {", "if (t >= bv) {"),
    ("shared branch dropped", "double w = std::exp(logit[i] - mx);", "double w = 0.0 * std::exp(logit[i] - mx);"),
    ("shared values are Lq", "const double* val = lv + (bh * m + i) * d;", "const double* val = lq + (bh * m + i) * d;"),
    ("expert of landmark 0", "eidx + (bh * m + e) * static_cast<int64_t>(kk);", "eidx + (bh * m + 0) * static_cast<int64_t>(kk);"),
    ("attend drops tau on routed logits", "logit[ms + j] = tau * t;", "logit[ms + j] = t;"),
    ("routing-only keeps the shared pairs", "const int ms = shared ? m : 0;", "const int ms = m;"),
    ("s experts: union keeps duplicates", "keys.erase(std::unique(keys.begin(), keys.end()), keys.end());",
     "(void)0;"),
    ("s experts: lowest logits taken", "return sc[x] > sc[y]; });", "return sc[x] < sc[y]; });"),
    ("s experts: ties to the higher landmark", "return sc[x] > sc[y]; });",
     "return sc[x] > sc[y] || (sc[x] == sc[y] && x > y); });"),
    ("s experts: only the first expert attended", "for (int u = 0; u < s; ++u) {\n            const int e",
     "for (int u = 0; u < 1; ++u) {\n            const int e"),
]


def _build(tmp, idx, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/not found: {old!r}"
    path = os.path.join(tmp, f"m{idx}.cpp")
    open(path, "w").write(src.replace(old, new))
    lib = os.path.join(tmp, f"libm{idx}.so")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-fopenmp", "-shared", "-fPIC", path, "-o", lib])
    return lib


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("mutants"))
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        futs = [ex.submit(_build, tmp, i, old, new) for i, (_, old, new) in enumerate(MUTANTS)]
        return [f.result() for f in futs]


@pytest.mark.parametrize("idx", range(len(MUTANTS)), ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(mutant_libs, idx):
    o = oracle.Oracle(mutant_libs[idx])
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {MUTANTS[idx][0]!r}"


GRAD_MUTANTS = [
    ("landmark values detached", "lv = torch.softmax(tau * (lq @ k.T), dim=-1) @ v",
     "lv = (torch.softmax(tau * (lq @ k.T), dim=-1) @ v).detach()"),
    ("landmarks detached", "lq = W @ q", "lq = (W @ q).detach()"),
    ("routed keys detached", "qi @ k[sel].T", "qi @ k[sel].detach().T"),
    ("shared values dropped from the gradient", "vals.append(p[:, :m] @ lv + p[:, m:] @ v[sel])",
     "vals.append(p[:, :m] @ lv.detach() + p[:, m:] @ v[sel])"),
]


@pytest.mark.parametrize("idx", range(len(GRAD_MUTANTS)), ids=[g[0] for g in GRAD_MUTANTS])
def test_grad_pin_catches_mutant(idx):
    """A copy of the gradient oracle with one dependence cut must fail the
    finite-difference pin (its values are unchanged, its gradients are not)."""
    import types

    import torch

    from oracle import mita_grad

    _, old, new = GRAD_MUTANTS[idx]
    src = open(mita_grad.__file__).read()
    assert src.count(old) == 1, f"mutation anchor not unique/not found: {old!r}"
    mod = types.ModuleType("mita_grad_mutant")
    exec(compile(src.replace(old, new), "mita_grad_mutant", "exec"), mod.__dict__)
    rng = np.random.default_rng(3)
    N, d, m, kk = 12, 4, 3, 5
    W = mita_grad.pooling_matrix(oracle.Oracle(), N, 0, 0, m)
    eidx = np.sort(np.stack([rng.choice(N, kk, replace=False) for _ in range(m)]), axis=1)[None]
    route = (np.arange(N) % m)[None]
    Q, K, V = (torch.from_numpy(rng.standard_normal((1, N, d))).requires_grad_(True) for _ in range(3))
    ok = torch.autograd.gradcheck(lambda a, b, c: mod.forward_fixed(W, a, b, c, eidx, route), (Q, K, V), eps=1e-6,
                                  atol=1e-7, rtol=1e-6, raise_exception=False)
    assert not ok, "the finite-difference pin did not catch the mutant"
