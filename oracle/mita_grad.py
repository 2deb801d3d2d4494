"""Gradients of the MiTA forward pass, fp64 on the CPU -- TEST INFRASTRUCTURE ONLY.

Only tests/ and bench.py's CPU legs import this module; the CUDA library never
uses it and shares no code with it.

The pages train MiTA models (the Long Range Arena training times in
"NeurIPS 2026 | Mixture-of-Top-k 注意力" (shuwu5.cn), results section) but do
not describe the backward pass. Reading taken: the gradient of the forward
pass with respect to Q, K and V with the discrete choices held fixed -- each
landmark's top-k key set and each query's route. Both are piecewise constant
in the inputs, so their derivative is zero almost everywhere.

The forward pass is restated with plain torch float64 ops and differentiated
by autograd (per head; tau = 1/sqrt(d)):
  Lq = W Q            W: the pooling matrix, row i = 1/|window i| on the
                      tokens of window i (windows from the C++ oracle);
  A  = softmax(tau Lq K^T) over all N keys,  LV = A V;
  out_n = softmax([tau q_n Lq^T, tau q_n K_E^T]) [LV; V_E],  E the key set
          of the query's routed expert (the shared pairs and the routed
          pairs under one softmax).
Pins (tests/oracle_pins.py): this forward equals the C++ oracle's, and
torch.autograd.gradcheck compares its gradients with finite differences.
"""
from __future__ import annotations

import numpy as np
import torch


def _widen(a):
    """bf16 bit patterns (uint16) -> float64 torch tensor."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    f = (a.astype(np.uint32) << 16).view(np.float32)
    return torch.from_numpy(f.astype(np.float64))


def pooling_matrix(orc, N: int, grid_h: int, grid_w: int, m: int) -> torch.Tensor:
    W = torch.zeros((m, N), dtype=torch.float64)
    for i in range(m):
        idx = torch.from_numpy(orc.window(N, grid_h, grid_w, m, i))
        W[i, idx] = 1.0 / len(idx)
    return W


def forward_fixed(W, Q, K, V, eidx, route):
    """The forward pass with fixed experts and routes, differentiable in Q, K, V.

    W [m,N]; Q, K, V [BH,N,d] float64; eidx [BH,m,kk], route [BH,N] int arrays.
    Returns out [BH,N,d].
    """
    BH, N, d = Q.shape
    m = W.shape[0]
    tau = 1.0 / np.sqrt(d)
    outs = []
    for bh in range(BH):
        q, k, v = Q[bh], K[bh], V[bh]
        lq = W @ q
        lv = torch.softmax(tau * (lq @ k.T), dim=-1) @ v
        rows, vals = [], []
        r = np.asarray(route[bh])
        for e in range(m):
            idx = np.nonzero(r == e)[0]
            if idx.size == 0:
                continue
            sel = torch.from_numpy(np.asarray(eidx[bh, e], dtype=np.int64))
            qi = q[torch.from_numpy(idx)]
            logits = tau * torch.cat([qi @ lq.T, qi @ k[sel].T], dim=1)
            p = torch.softmax(logits, dim=1)
            vals.append(p[:, :m] @ lv + p[:, m:] @ v[sel])
            rows.append(torch.from_numpy(idx))
        order = torch.cat(rows)
        out = torch.zeros((N, d), dtype=torch.float64).index_copy(0, order, torch.cat(vals))
        outs.append(out)
    return torch.stack(outs)


def grads(orc, q, k, v, dout, grid_h: int, grid_w: int, m: int, eidx, route):
    """dQ, dK, dV (float64 numpy, the shape of q) of sum(out * dout), with
    the experts eidx [B,H,m,kk] and routes route [B,H,N] held fixed. q, k, v
    are bf16 bit patterns; dout is bf16 bit patterns or float."""
    B, H, N, d = q.shape
    BH = B * H
    W = pooling_matrix(orc, N, grid_h, grid_w, m)
    Q, K, V = (_widen(x).reshape(BH, N, d).requires_grad_(True) for x in (q, k, v))
    dO = _widen(dout) if np.asarray(dout).dtype == np.uint16 else torch.from_numpy(np.asarray(dout, np.float64))
    out = forward_fixed(W, Q, K, V, np.asarray(eidx).reshape(BH, m, -1), np.asarray(route).reshape(BH, N))
    out.backward(dO.reshape(BH, N, d))
    return tuple(t.grad.numpy().reshape(B, H, N, d) for t in (Q, K, V))


def forward(orc, q, k, v, grid_h: int, grid_w: int, m: int, eidx, route):
    """out (float64 numpy [B,H,N,d]) of the restated forward pass."""
    B, H, N, d = q.shape
    BH = B * H
    W = pooling_matrix(orc, N, grid_h, grid_w, m)
    Q, K, V = (_widen(x).reshape(BH, N, d) for x in (q, k, v))
    with torch.no_grad():
        out = forward_fixed(W, Q, K, V, np.asarray(eidx).reshape(BH, m, -1), np.asarray(route).reshape(BH, N))
    return out.numpy().reshape(B, H, N, d)
