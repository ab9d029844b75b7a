"""fp64 CPU reference of the MiTA backward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` may import this module (it imports nothing from the product).

The pages train MiTA models end to end (LRA, MiTA tutorial ch. 7 table 5; the
bit.fan article's LRA section) but give no gradient through the selections.
Reading taken (the plainest one): the selections -- every landmark's top-k key
set and every query's top-s landmarks -- are held constant (top-k and argmax are
piecewise constant), and the rounding of q~ to the input dtype passes the
gradient straight through.  The backward is then the gradient of this
composition, per (batch, head), written as plain fp64 torch ops in the pages'
order and differentiated by autograd:

  q~ = pool(Q)                                  (tutorial ch. 4 step 1, eq. 5)
  A  = softmax(q~ K^T / sqrt(d)),  v~ = A V     (steps 2-3, eq. 6-9)
  l_n = [q_n . q~_i * c_sh]_i ++ [q_n . k_j / sqrt(d)]_{j in the s experts}
  out_n = softmax(l_n) . ([v~_i]_i ++ [v_j]_j)  (steps 5-6, eq. 11-12)

c_sh = 1/sqrt(d), or 1/d for the official code's shared temperature (tutorial
ch. 8 caveat 3); branches="routed" drops the shared pairs.
"""
from __future__ import annotations

import math

import torch

from . import landmark as _landmark, pool as _pool, route as _route


def _windows(n_in: int, n_out: int):
    """Adaptive windows [floor(i*in/out), ceil((i+1)*in/out)) along one axis."""
    return [((i * n_in) // n_out, -((-(i + 1) * n_in) // n_out)) for i in range(n_out)]


def pool_matrix(grid_h: int, grid_w: int, m: int, landmark_grid=None) -> torch.Tensor:
    """[m, N] float64 matrix whose row i averages landmark i's window."""
    if landmark_grid is not None:
        mh, mw = landmark_grid
    elif grid_h == 1:
        mh, mw = 1, m
    else:
        mh = mw = int(round(math.sqrt(m)))
    N = grid_h * grid_w
    P = torch.zeros((m, N), dtype=torch.float64)
    rows, cols = _windows(grid_h, mh), _windows(grid_w, mw)
    for i in range(m):
        r0, r1 = rows[i // mw]
        c0, c1 = cols[i % mw]
        idx = [r * grid_w + c for r in range(r0, r1) for c in range(c0, c1)]
        P[i, idx] = 1.0 / len(idx)
    return P


def forward_fixed(q, k, v, q_tilde_rounded, topk_idx, route_idx, grid_h, grid_w, m,
                  landmark_grid=None, shared_temperature="sqrt_d", branches="both"):
    """The forward with the selections given (fp64 tensors with autograd).
    ``q_tilde_rounded`` = None uses the exact window means (fp64 inputs)."""
    B, H, N, d = q.shape
    P = pool_matrix(grid_h, grid_w, m, landmark_grid)
    c = 1.0 / math.sqrt(d)
    c_sh = c if shared_temperature == "sqrt_d" else 1.0 / d
    outs = []
    for b in range(B):
        hs = []
        for h in range(H):
            Q, K, V = q[b, h], k[b, h], v[b, h]
            qt = P @ Q
            if q_tilde_rounded is not None:
                # the forward's value is the rounded mean; its gradient is the exact mean's
                qt = qt + (q_tilde_rounded[b, h] - qt).detach()
            A = torch.softmax((qt @ K.T) * c, dim=-1)
            vt = A @ V
            rows = topk_idx[b, h].long()[route_idx[b, h].long()].reshape(N, -1)   # [N, s*k]
            Kr, Vr = K[rows], V[rows]                                            # [N, s*k, d]
            raw = torch.einsum("nd,nrd->nr", Q, Kr) * c
            if branches == "routed":
                p = torch.softmax(raw, dim=-1)
                hs.append(torch.einsum("nr,nrd->nd", p, Vr))
            else:
                sh = (Q @ qt.T) * c_sh
                p = torch.softmax(torch.cat([sh, raw], dim=-1), dim=-1)
                hs.append(p[:, :m] @ vt + torch.einsum("nr,nrd->nd", p[:, m:], Vr))
        outs.append(torch.stack(hs))
    return torch.stack(outs)


def selections(q, k, v, grid_h, grid_w, m, topk, s, landmark_grid=None):
    """The forward's selections and rounded q~, from the C oracle."""
    qt = _pool(q, grid_h, grid_w, m, landmark_grid)
    ti, _, _ = _landmark(qt, k, v, topk)
    r, _ = _route(q, qt, s)
    return qt, ti, r


def backward(q, k, v, dout, grid_h, grid_w, m, topk, s=1, landmark_grid=None,
             shared_temperature="sqrt_d", branches="both"):
    """(dq, dk, dv) float64 for upstream gradient ``dout`` (all [B,H,N,d])."""
    qt, ti, r = selections(q, k, v, grid_h, grid_w, m, topk, s, landmark_grid)
    qd = q.detach().double().requires_grad_(True)
    kd = k.detach().double().requires_grad_(True)
    vd = v.detach().double().requires_grad_(True)
    out = forward_fixed(qd, kd, vd, qt, ti, r, grid_h, grid_w, m, landmark_grid,
                        shared_temperature, branches)
    return torch.autograd.grad(out, (qd, kd, vd), dout.double())
