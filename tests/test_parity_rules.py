"""The parity checker itself, on the CPU: mistakes are planted in oracle-side
data (never on the GPU) and must be caught, while the alternatives the rules
allow must pass."""
import pytest
import torch

import oracle
from parity_util import (assert_index_sets_match, assert_ranked_routes_match,
                         assert_routes_match, landmark_scores)
from sparse_top_landmark_gb300 import workloads as W


def _landmark_case():
    w = W.custom("rules", 1, 2, 300, 16, "bf16", 1, 300, 6, 9, index=500)
    q, k, v = W.make_qkv(w, 0)
    qt = oracle.pool(q, 1, 300, 6)
    ti, vt, gap = oracle.landmark(qt, k, v, 9)
    return qt, k, ti, gap


def test_identical_index_sets_pass():
    qt, k, ti, gap = _landmark_case()
    assert assert_index_sets_match(ti.clone(), ti, gap, exact=True,
                                   scores=lambda r: landmark_scores(qt, k, r)) == 0


def test_a_swapped_member_is_caught():
    qt, k, ti, gap = _landmark_case()
    bad = ti.clone()
    row = bad[0, 0, 1]                            # flat landmark row 1
    # replace the row's member with the lowest score by the best non-member
    sc = landmark_scores(qt, k, [1])[0]
    mem = set(row.tolist())
    worst = min(mem, key=lambda j: sc[j].item())
    out = max((j for j in range(sc.numel()) if j not in mem), key=lambda j: sc[j].item())
    # the swap is wrong by the row's gap, which is far above both tolerances here
    assert gap[0, 0, 1].item() > 1e-6
    bad[0, 0, 1] = torch.tensor(sorted((mem - {worst}) | {out}), dtype=torch.int32)
    with pytest.raises(AssertionError):
        assert_index_sets_match(bad, ti, gap, exact=True,
                                scores=lambda r: landmark_scores(qt, k, r))
    with pytest.raises(AssertionError):
        assert_index_sets_match(bad, ti, gap)


def test_a_tied_row_needs_a_valid_set():
    """A row whose boundary is an exact tie tolerates the other tied key, but not
    a key from below the boundary."""
    N, d = 12, 4
    base = torch.randn((1, 1, 3, d), generator=torch.Generator().manual_seed(3))
    k = base[:, :, torch.tensor([0, 1, 2, 1, 0, 2, 0, 1, 2, 1, 0, 2])].contiguous()
    qt = torch.randn((1, 1, 1, d), generator=torch.Generator().manual_seed(4)).double()
    ti, _, gap = oracle.landmark(qt, k, k, 2)
    assert gap.item() == 0.0                      # the 2nd and 3rd best keys are equal
    sc = landmark_scores(qt, k, [0])[0]
    best = torch.argsort(-sc, stable=True)
    tied = [j for j in range(N) if sc[j] == sc[best[1]] and j not in ti[0, 0, 0].tolist()]
    ok = ti.clone()
    ok[0, 0] = torch.tensor(sorted([best[0].item(), tied[0]]), dtype=torch.int32)
    assert_index_sets_match(ok, ti, gap, exact=True, scores=lambda r: landmark_scores(qt, k, r))
    low = min(range(N), key=lambda j: sc[j].item())
    wrong = ti.clone()
    wrong[0, 0] = torch.tensor(sorted([best[0].item(), low]), dtype=torch.int32)
    with pytest.raises(AssertionError):
        assert_index_sets_match(wrong, ti, gap, exact=True,
                                scores=lambda r: landmark_scores(qt, k, r))


def test_route_rules():
    w = W.custom("rules_r", 1, 1, 200, 16, "f32", 1, 200, 8, 4, index=501)
    q, _, _ = W.make_qkv(w, 0)
    qt = oracle.pool(q, 1, 200, 8)
    r, gap = oracle.route(q, qt, 1)
    assert assert_routes_match(r.clone(), r, gap, q, qt) == 0
    bad = r.clone()
    n = int(torch.argmax(gap.view(-1)))           # the clearest route
    bad.view(-1)[n] = (bad.view(-1)[n] + 1) % 8
    with pytest.raises(AssertionError):
        assert_routes_match(bad, r, gap, q, qt)
    r2, _ = oracle.route(q, qt, 2)
    bad2 = r2.clone()
    bad2.view(-1, 2)[n] = bad2.view(-1, 2)[n].flip(0)   # best and second swapped
    with pytest.raises(AssertionError):
        assert_ranked_routes_match(bad2, r2, q, qt)
