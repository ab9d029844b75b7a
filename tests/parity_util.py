"""Shared comparison rules of the GPU-vs-oracle parity tests.

Rules (applied element by element on the same seeded inputs):
  * index outputs (top-k sets, routes, buckets) match bit-exactly, except a
    row whose oracle score gap at the selection boundary is below 1e-6
    relative to that row's largest |score| (then either choice is correct);
    such a tolerated row must still be a valid answer under the oracle's fp64
    scores: every selected score at least every unselected score minus
    1e-6 * max|score| (and, for routes, the same at every rank);
  * the library re-scores every undecided selection exactly (error-free
    products and sums), so its index outputs are held to the tighter
    EXACT_GAP_TOL: a row may differ from the oracle only where the fp64
    oracle's own rounding could decide the order (gap below 1e-12 relative),
    and it must then be valid within that same margin;
  * float outputs: fp32 inputs -> max-abs error <= 1e-4; bf16 inputs ->
    max-abs error <= 2e-2 and relative L2 error <= 5e-3.
"""
import math

import torch

GAP_TOL = 1e-6
EXACT_GAP_TOL = 1e-12
F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3


def landmark_scores(q_tilde, k, rows):
    """fp64 scores q~_i . k_j / sqrt(d) of the given flat landmark rows (bh*m + i)
    against every key of their head: [len(rows), N] (harness-side, for judging
    near ties)."""
    B, H, m, d = q_tilde.shape
    N = k.shape[2]
    rows = torch.as_tensor(rows, dtype=torch.int64)
    qt = q_tilde.reshape(-1, d)[rows].double()
    kk = k.reshape(B * H, N, d)
    out = torch.empty((rows.numel(), N), dtype=torch.float64)
    for t, r in enumerate(rows.tolist()):
        out[t] = kk[r // m].double() @ qt[t]
    return out / math.sqrt(d)


def assert_valid_topk(sel, scores, tol, what="top-k"):
    """sel: [R, k] GPU index lists; scores: [R, N] fp64.  Each list must hold k
    distinct in-range keys, and its lowest score must be at least the highest
    unselected score minus tol * max|score| of the row."""
    sel = sel.to(torch.int64)
    R, k = sel.shape
    N = scores.shape[1]
    assert bool(((sel >= 0) & (sel < N)).all()), f"{what}: index out of range"
    for r in range(R):
        assert torch.unique(sel[r]).numel() == k, f"{what}: repeated index in row {r}"
        mask = torch.zeros(N, dtype=torch.bool)
        mask[sel[r]] = True
        amax = scores[r].abs().max().item()
        lo = scores[r][mask].min().item()
        hi = scores[r][~mask].max().item() if k < N else -math.inf
        assert lo >= hi - tol * amax, (f"{what}: row {r} is not a valid top-{k}: selected "
                                       f"min {lo!r} < unselected max {hi!r} beyond {tol:g}")


def assert_index_sets_match(gpu, ora, gap, what="top-k", exact=False, scores=None):
    """gpu/ora: [..., k] int index lists (ascending), gap: [...] oracle gaps.

    Rows that differ must lie below the gap tolerance (GAP_TOL, or EXACT_GAP_TOL
    with ``exact``); when ``scores`` is given (a callable: flat row ids -> fp64
    scores [R, N]) each such row must also be a valid selection under them."""
    g = gpu.to("cpu").to(torch.int64).reshape(-1, gpu.shape[-1])
    o = ora.to("cpu").to(torch.int64).reshape(-1, ora.shape[-1])
    gp = gap.to("cpu").reshape(-1)
    tol = EXACT_GAP_TOL if exact else GAP_TOL
    diff = (g != o).any(-1)
    bad = diff & (gp >= tol)
    nbad = int(bad.sum())
    assert nbad == 0, (f"{what}: {nbad} rows differ with oracle gap >= {tol} "
                       f"(first row {int(bad.nonzero()[0])})")
    rows = diff.nonzero().flatten()
    if rows.numel() and scores is not None:
        assert_valid_topk(g[rows], scores(rows), tol, what)
    return int(diff.sum())


def assert_close(gpu, ora, dtype, what="output", scale=1.0):
    """``scale``: the magnitude of the values (the bounds are for O(1) data; a
    workload drawn at scale x has its max-abs bounds multiplied by x)."""
    g = gpu.to("cpu").double()
    o = ora.to("cpu").double()
    err = (g - o).abs()
    mx = err.max().item() if err.numel() else 0.0
    if dtype == torch.float32:
        assert mx <= F32_MAX_ABS * scale, f"{what}: max-abs {mx:.3e} > {F32_MAX_ABS * scale}"
    else:
        rel = (torch.linalg.vector_norm(g - o) / torch.linalg.vector_norm(o).clamp_min(1e-30)).item()
        assert mx <= BF16_MAX_ABS * scale, f"{what}: max-abs {mx:.3e} > {BF16_MAX_ABS * scale}"
        assert rel <= BF16_REL_L2, f"{what}: rel-L2 {rel:.3e} > {BF16_REL_L2}"
    return mx


def route_scores(q, q_tilde, rows):
    """fp64 scores q_n . q~_i of the given flat query rows against their head's
    landmarks: [len(rows), m] (harness-side, for judging near ties)."""
    B, H, N, d = q.shape
    m = q_tilde.shape[2]
    rows = torch.as_tensor(rows, dtype=torch.int64)
    qr = q.reshape(-1, d)[rows].double()
    lt = q_tilde.reshape(B * H, m, d)[rows // N].double()
    return torch.einsum("rd,rmd->rm", qr, lt)


def assert_routes_match(gpu, ora, gap, q, q_tilde, rows=None, what="route", exact=True):
    """s = 1 routes: bit-exact except where the oracle's gap is below the
    tolerance; a differing route must then score within that margin of the best
    (a valid argmax).  ``rows``: flat query ids of the compared entries."""
    g = gpu.to("cpu").to(torch.int64).reshape(-1, gpu.shape[-1])
    if rows is None:
        rows = torch.arange(g.shape[0])
    rows = torch.as_tensor(rows, dtype=torch.int64)

    def sc(r):
        return route_scores(q, q_tilde, rows[r])

    return assert_index_sets_match(g, ora, gap, what, exact=exact, scores=sc)


def assert_ranked_routes_match(gpu, ora, q, q_tilde, rows=None, what="route", exact=True):
    """Top-s lists, best first: equal, or every position's oracle score within
    the tolerance (EXACT_GAP_TOL by default, GAP_TOL without ``exact``) times
    max|score| of the other list's (a near tie, either order correct); the list
    must also hold s distinct landmarks."""
    g = gpu.to("cpu").to(torch.int64).reshape(-1, gpu.shape[-1])
    o = ora.to("cpu").to(torch.int64).reshape(-1, ora.shape[-1])
    tol = EXACT_GAP_TOL if exact else GAP_TOL
    if rows is None:
        rows = torch.arange(g.shape[0])
    diff = (g != o).any(-1).nonzero().flatten()
    if diff.numel():
        sc = route_scores(q, q_tilde, torch.as_tensor(rows)[diff])
        amax = sc.abs().amax(-1, keepdim=True)
        sg = sc.gather(1, g[diff])
        so = sc.gather(1, o[diff])
        bad = ((sg - so).abs() > tol * amax).any(-1)
        assert not bool(bad.any()), (f"{what}: {int(bad.sum())} rows differ beyond a near tie "
                                     f"(first row {int(torch.as_tensor(rows)[diff][bad][0])})")
        for r in range(diff.numel()):
            assert torch.unique(g[diff[r]]).numel() == g.shape[1], f"{what}: repeated landmark"
    return int(diff.numel())
