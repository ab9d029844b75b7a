"""Pins for the fp64 oracle: each check comes from something other than the
oracle itself -- a value the pages print, a textbook/library routine the step
reduces to, a brute-force sort on tiny inputs, or an invariant of the maths.

Sources: MiTA tutorial (iwxt.cn), ch. 1 (softmax example), ch. 4 (step list,
paper Sec. 3.2 eq. 5-12, merge identity), ch. 5 quiz (unselected KV still
contributes), ch. 8 caveat 2 (Appendix A counterexample); bit.fan article
(Algorithm 1: group queries by expert).
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from sparse_top_landmark_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(None, 1)
            vals[key] = float(val)
    return vals


def _bruteforce_topk(scores, k):
    """Full sort of one row by (score desc, index asc); returns the k indices."""
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))
    return np.sort(order[:k]), order


def _rand(shape, dtype, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float64) * scale).to(dtype)


# ----------------------------------------------------------------------------
# Worked values printed on the pages
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("d", [1, 16])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float64])
def test_appendix_a_counterexample(d, dtype):
    """Tutorial ch. 8 caveat 2: m = k = N gives 0.5577646447, dense gives 0.5."""
    gold = _golden("appendix_a_counterexample.txt")
    q = torch.zeros((1, 1, 2, d), dtype=torch.float64)
    k = torch.zeros_like(q)
    v = torch.zeros_like(q)
    q[0, 0, 1, 0] = 1.0 if d == 1 else 4.0   # q1 . k1 / sqrt(d) = 1
    k[0, 0, 1, 0] = 1.0
    v[0, 0, 1, :] = 1.0
    q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
    res = oracle.forward(q, k, v, grid_h=1, grid_w=2, m=2, topk=2, s=1)
    # shared values [0.5, sigmoid(1)] printed on the page
    assert abs(res["v_tilde"][0, 0, 0, 0].item() - 0.5) < 1e-15
    assert abs(res["v_tilde"][0, 0, 1, 0].item() - 1 / (1 + math.exp(-1))) < 1e-15
    out0 = res["out"][0, 0, 0, 0].item()
    tol = 0.5 * 10 ** (-int(gold["digits"]))
    assert abs(out0 - gold["mita_output"]) <= tol
    # dense attention of q = 0 over the same KV (textbook softmax)
    dense = torch.softmax(torch.zeros(2, dtype=torch.float64), 0) @ v[0, 0, :, 0].double()
    assert abs(dense.item() - gold["dense_output"]) < 1e-15
    assert abs(out0 - dense.item()) > 0.05
    # the official code's shared temperature (q . q~ / d): query 0 has q = 0, so all four
    # logits stay 0 and the printed value is unchanged
    res_d = oracle.forward(q, k, v, grid_h=1, grid_w=2, m=2, topk=2, s=1,
                           shared_temperature="d")
    assert abs(res_d["out"][0, 0, 0, 0].item() - gold["mita_output"]) <= tol


@pytest.mark.parametrize("temp", ["sqrt_d", "d"])
def test_counterexample_second_query_closed_form(temp):
    """Query 1 of the same example at d = 16: q1 = 4 e0, k1 = e0, q~ = q.  Raw logits
    q1 . k / 4 = [0, 1]; shared logits q1 . q~ / 4 = [0, 4] (every logit / sqrt(d)) or
    q1 . q~ / 16 = [0, 1] (shared logits / d); values [0.5, sigmoid(1)] then [0, 1]."""
    d = 16
    q = torch.zeros((1, 1, 2, d), dtype=torch.float64)
    k = torch.zeros_like(q)
    v = torch.zeros_like(q)
    q[0, 0, 1, 0] = 4.0
    k[0, 0, 1, 0] = 1.0
    v[0, 0, 1, :] = 1.0
    res = oracle.forward(q, k, v, grid_h=1, grid_w=2, m=2, topk=2, s=1, shared_temperature=temp)
    sh = 4.0 if temp == "sqrt_d" else 1.0
    sig1 = 1 / (1 + math.exp(-1))
    want = (0.5 + math.exp(sh) * sig1 + math.exp(1.0)) / (2 + math.exp(sh) + math.exp(1.0))
    assert abs(res["out"][0, 0, 1, 0].item() - want) < 1e-14


def test_two_equal_scores_average():
    """Tutorial ch. 1: two scores of 0 give weights 1/2; values 0 and 2 give 1."""
    q = torch.zeros((1, 1, 2, 1), dtype=torch.float64)
    k = torch.tensor([0.3, -1.7], dtype=torch.float64).view(1, 1, 2, 1)
    v = torch.tensor([0.0, 2.0], dtype=torch.float64).view(1, 1, 2, 1)
    qt = oracle.pool(q, 1, 2, 1)
    assert qt.abs().max().item() == 0.0
    _, vt, _ = oracle.landmark(qt, k, v, 1)
    assert vt.item() == 1.0


# ----------------------------------------------------------------------------
# Step 1: pooling
# ----------------------------------------------------------------------------
def _check_rounded_mean(qt, mean, dtype):
    """qt must be the dtype value nearest to the fp64 mean."""
    assert torch.equal(qt.to(dtype).double(), qt)          # representable
    err = (qt - mean).abs()
    mant = 8 if dtype == torch.bfloat16 else 24
    ulp = torch.exp2(torch.floor(torch.log2(mean.abs().clamp_min(1e-30))) - (mant - 1))
    assert bool((err <= 0.5 * ulp * (1 + 1e-12)).all())
    # equal to the library rounding nearly everywhere (the library rounds
    # through float32 first, which can differ only next to exact midpoints)
    lib = mean.to(dtype).double()
    assert (lib == qt).double().mean().item() > 0.999


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_pool_1d_closed_form(dtype):
    B, H, N, d, m = 2, 3, 96, 16, 8
    q = _rand((B, H, N, d), dtype, 1)
    qt = oracle.pool(q, 1, N, m)
    mean = q.double().view(B, H, m, N // m, d).mean(3)
    _check_rounded_mean(qt, mean, dtype)


@pytest.mark.parametrize("gh,gw,m", [(14, 14, 25), (32, 32, 49), (2, 4, 4), (6, 10, 9), (5, 7, 16)])
def test_pool_2d_matches_adaptive_avg_pool(gh, gw, m):
    B, H, d = 2, 2, 8
    dtype = torch.bfloat16
    q = _rand((B, H, gh * gw, d), dtype, 2)
    qt = oracle.pool(q, gh, gw, m)
    r = int(round(math.sqrt(m)))
    img = q.double().view(B * H, gh, gw, d).permute(0, 3, 1, 2)
    ref = F.adaptive_avg_pool2d(img, (r, r)).permute(0, 2, 3, 1).reshape(B, H, m, d)
    _check_rounded_mean(qt, ref, dtype)


@pytest.mark.parametrize("gh,gw,mh,mw", [(14, 14, 3, 5), (32, 32, 4, 8), (6, 10, 2, 5),
                                        (5, 7, 5, 1), (9, 4, 1, 4)])
def test_pool_2d_nonsquare_landmark_grid_matches_adaptive_avg_pool(gh, gw, mh, mw):
    B, H, d = 2, 2, 8
    dtype = torch.bfloat16
    q = _rand((B, H, gh * gw, d), dtype, 3)
    qt = oracle.pool(q, gh, gw, mh * mw, landmark_grid=(mh, mw))
    img = q.double().view(B * H, gh, gw, d).permute(0, 3, 1, 2)
    ref = F.adaptive_avg_pool2d(img, (mh, mw)).permute(0, 2, 3, 1).reshape(B, H, mh * mw, d)
    _check_rounded_mean(qt, ref, dtype)


def test_pool_1d_uneven_windows():
    """1D with m not dividing N uses the adaptive window rule (1 x N grid)."""
    B, H, N, d, m = 1, 2, 50, 4, 7
    q = _rand((B, H, N, d), torch.float32, 3)
    qt = oracle.pool(q, 1, N, m)
    img = q.double().view(B * H, 1, N, d).permute(0, 3, 1, 2)
    ref = F.adaptive_avg_pool2d(img, (1, m)).permute(0, 2, 3, 1).reshape(B, H, m, d)
    _check_rounded_mean(qt, ref, torch.float32)


# ----------------------------------------------------------------------------
# Steps 2-3: top-k experts and shared values
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("seed,N,d,m,k", [(0, 64, 16, 4, 4), (1, 200, 8, 5, 17),
                                           (2, 256, 64, 9, 64), (3, 33, 4, 3, 33)])
def test_topk_matches_full_sort(seed, N, d, m, k):
    B, H = 2, 2
    kk = _rand((B, H, N, d), torch.bfloat16, seed)
    vv = _rand((B, H, N, d), torch.bfloat16, seed + 50)
    qt = _rand((B, H, m, d), torch.bfloat16, seed + 99).double()
    idx, vt, gap = oracle.landmark(qt, kk, vv, k)
    S = (qt @ kk.double().transpose(-1, -2)).numpy() / math.sqrt(d)
    for b in range(B):
        for h in range(H):
            for i in range(m):
                ref, order = _bruteforce_topk(S[b, h, i], k)
                assert np.array_equal(idx[b, h, i].numpy(), ref)
                if k < N:
                    amax = np.abs(S[b, h, i]).max()
                    g = (S[b, h, i][order[k - 1]] - S[b, h, i][order[k]]) / amax
                    assert abs(gap[b, h, i].item() - g) < 1e-15
                else:
                    assert gap[b, h, i].item() > 1e299


def test_topk_ties_go_to_lowest_index():
    B, H, N, d, m, k = 1, 1, 40, 8, 3, 6
    base = _rand((1, 1, 4, d), torch.float32, 7)
    # every key is one of 4 rows -> groups of 10 equal scores in every row
    kk = base[:, :, torch.arange(N) % 4, :].contiguous()
    vv = _rand((B, H, N, d), torch.float32, 8)
    qt = _rand((B, H, m, d), torch.float32, 9).double()
    idx, _, gap = oracle.landmark(qt, kk, vv, k)
    S = (qt @ kk.double().transpose(-1, -2)).numpy()
    for i in range(m):
        best = int(np.argmax(S[0, 0, i]))          # first index of the best group
        expect = np.sort(np.lexsort((np.arange(N), -S[0, 0, i]))[:k])
        assert np.array_equal(idx[0, 0, i].numpy(), expect)
        assert idx[0, 0, i, 0].item() == best % 4
        assert gap[0, 0, i].item() == 0.0           # k = 6 splits a group of 10


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_shared_value_is_dense_attention_of_landmark(dtype):
    """Tutorial ch. 4 step 3: v~_i is full attention of q~_i over all N pairs."""
    B, H, N, d, m = 2, 2, 300, 32, 6
    kk = _rand((B, H, N, d), dtype, 11)
    vv = _rand((B, H, N, d), dtype, 12)
    qt = _rand((B, H, m, d), dtype, 13).double()
    _, vt, _ = oracle.landmark(qt, kk, vv, 5)
    ref = F.scaled_dot_product_attention(qt, kk.double(), vv.double())
    assert torch.allclose(vt, ref, rtol=0, atol=1e-13)


def test_landmark_rows_subset_matches_full():
    w = W.custom("t", 1, 2, 128, 16, "bf16", 1, 128, 8, 10)
    q, k, v = W.make_qkv(w, 0)
    qt = oracle.pool(q, 1, 128, 8)
    idx, vt, gap = oracle.landmark(qt, k, v, 10)
    rows = [0, 5, 9, 15]
    i2, v2, g2 = oracle.landmark(qt, k, v, 10, rows=rows)
    assert torch.equal(i2, idx.view(-1, 10)[rows])
    assert torch.equal(v2, vt.view(-1, 16)[rows])
    assert torch.equal(g2, gap.view(-1)[rows])


# ----------------------------------------------------------------------------
# Steps 4-5: routing and grouping
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("s", [1, 2, 3])
def test_route_matches_full_sort(s):
    B, H, N, d, m = 2, 2, 77, 16, 9
    q = _rand((B, H, N, d), torch.bfloat16, 21)
    qt = _rand((B, H, m, d), torch.bfloat16, 22).double()
    r, gap = oracle.route(q, qt, s)
    S = (q.double() @ qt.transpose(-1, -2)).numpy()
    for b in range(B):
        for h in range(H):
            for n in range(N):
                order = np.lexsort((np.arange(m), -S[b, h, n]))
                assert np.array_equal(r[b, h, n].numpy(), order[:s])
                # the boundary gap: s-th minus (s+1)-th best logit over max |logit|
                amax = np.abs(S[b, h, n]).max()
                g = (S[b, h, n][order[s - 1]] - S[b, h, n][order[s]]) / amax
                assert abs(gap[b, h, n].item() - g) < 1e-15
    # sampled queries give the same routes and gaps as the full run
    sel = torch.tensor([0, 5, N + 3, 4 * N - 1])
    r2, g2 = oracle.route(q, qt, s, queries=sel)
    assert torch.equal(r2, r.view(-1, s)[sel])
    assert torch.equal(g2, gap.view(-1)[sel])


def test_route_gap_when_every_landmark_is_chosen():
    """s = m: there is no boundary, the gap is reported as +inf-like (1e300)."""
    q = _rand((1, 1, 5, 8), torch.float32, 25)
    qt = _rand((1, 1, 3, 8), torch.float32, 26).double()
    r, gap = oracle.route(q, qt, 3)
    assert bool((gap > 1e299).all())
    S = (q.double() @ qt.transpose(-1, -2))[0, 0]
    for n in range(5):
        order = np.lexsort((np.arange(3), -S[n].numpy()))
        assert np.array_equal(r[0, 0, n].numpy(), order)


def test_route_ties_go_to_lowest_landmark():
    B, H, N, d, m = 1, 1, 10, 4, 6
    q = _rand((B, H, N, d), torch.float32, 23)
    base = _rand((B, H, 2, d), torch.float32, 24).double()
    qt = base[:, :, [0, 1, 0, 1, 1, 0], :].contiguous()   # duplicated landmarks
    r, gap = oracle.route(q, qt, 1)
    S = (q.double() @ base.transpose(-1, -2))[0, 0]
    for n in range(N):
        assert r[0, 0, n, 0].item() == (0 if S[n, 0] >= S[n, 1] else 1)
        assert gap[0, 0, n].item() == 0.0


@pytest.mark.parametrize("s", [1, 2])
def test_bucket_is_stable_counting_sort(s):
    B, H, N, m = 2, 3, 500, 13
    g = torch.Generator().manual_seed(5)
    r = torch.randint(0, m, (B, H, N, s), generator=g, dtype=torch.int32)
    off, qidx = oracle.bucket(r, m)
    for b in range(B):
        for h in range(H):
            flat = r[b, h].reshape(-1).numpy()
            cnt = np.bincount(flat, minlength=m)
            assert np.array_equal(off[b, h].numpy(), np.concatenate([[0], np.cumsum(cnt)]))
            order = np.argsort(flat, kind="stable") // s
            assert np.array_equal(qidx[b, h].numpy(), order)


# ----------------------------------------------------------------------------
# Step 6: joint attention
# ----------------------------------------------------------------------------
def _setup(seed=0, B=2, H=2, N=256, d=16, m=8, k=12, s=1, dtype="bf16", temp="sqrt_d"):
    w = W.custom("t", B, H, N, d, dtype, 1, N, m, k, s, index=seed)
    q, kk, vv = W.make_qkv(w, seed)
    return q, kk, vv, oracle.forward(q, kk, vv, 1, N, m, k, s, shared_temperature=temp)


@pytest.mark.parametrize("s,temp", [(1, "sqrt_d"), (2, "sqrt_d"), (1, "d"), (3, "d")])
def test_joint_softmax_equals_branch_merge(s, temp):
    """Tutorial ch. 4: (Z1 o1 + Z2 o2) / (Z1 + Z2) is the joint softmax; o1 + o2 is not.
    With temp = "d" the shared branch's logits are q . q~ / d (raw ones stay / sqrt(d))."""
    q, k, v, res = _setup(seed=1, s=s, temp=temp)
    B, H, N, d = q.shape
    qd, kd, vd = q.double(), k.double(), v.double()
    sq = math.sqrt(d)
    sh = sq if temp == "sqrt_d" else float(d)
    naive_err = 0.0
    for b in range(B):
        for h in range(H):
            ls = qd[b, h] @ res["q_tilde"][b, h].T / sh                   # [N, m]
            lse1 = torch.logsumexp(ls, -1)
            o1 = torch.softmax(ls, -1) @ res["v_tilde"][b, h]
            for n in range(0, N, 7):
                rows = torch.cat([res["topk_idx"][b, h, e].long() for e in res["route"][b, h, n]])
                lr = kd[b, h, rows] @ qd[b, h, n] / sq
                lse2 = torch.logsumexp(lr, 0)
                o2 = torch.softmax(lr, 0) @ vd[b, h, rows]
                z1, z2 = torch.exp(lse1[n]), torch.exp(lse2)
                merged = (z1 * o1[n] + z2 * o2) / (z1 + z2)
                got = res["out"][b, h, n]
                assert torch.allclose(got, merged, rtol=0, atol=1e-12)
                naive_err = max(naive_err, (o1[n] + o2 - got).abs().max().item())
    assert naive_err > 1e-2


def test_output_is_convex_combination():
    q, k, v, res = _setup(seed=2, N=300, m=10, k=20)
    B, H, N, d = q.shape
    vd = v.double()
    for b in range(B):
        for h in range(H):
            for n in range(N):
                e = res["route"][b, h, n, 0].item()
                vals = torch.cat([res["v_tilde"][b, h], vd[b, h, res["topk_idx"][b, h, e].long()]])
                o = res["out"][b, h, n]
                assert bool((o <= vals.max(0).values + 1e-12).all())
                assert bool((o >= vals.min(0).values - 1e-12).all())


@pytest.mark.parametrize("temp", ["sqrt_d", "d"])
def test_single_landmark_full_topk_reduces_to_dense_plus_one_shared_pair(temp):
    """m = 1, k = N: the routed expert is every KV row, so the output is the
    textbook dense attention merged with the one shared pair (q~_0, v~_0), whose
    logit is q . q~_0 / sqrt(d) or, with the official code's temperature, / d."""
    B, H, N, d = 1, 2, 64, 16
    q, k, v, res = _setup(seed=3, B=B, H=H, N=N, d=d, m=1, k=N, temp=temp)
    qd, kd, vd = q.double(), k.double(), v.double()
    sq = math.sqrt(d)
    dense = F.scaled_dot_product_attention(qd, kd, vd)
    lse_dense = torch.logsumexp(qd @ kd.transpose(-1, -2) / sq, -1)
    l_sh = (qd @ res["q_tilde"].transpose(-1, -2) / (sq if temp == "sqrt_d" else d))[..., 0]
    w_sh = torch.sigmoid(l_sh - lse_dense).unsqueeze(-1)
    ref = w_sh * res["v_tilde"][:, :, 0:1, :] + (1 - w_sh) * dense
    assert torch.allclose(res["out"], ref, rtol=0, atol=1e-12)


def test_permuting_kv_rows_relabels_experts_only():
    B, H, N, d, m, k = 1, 2, 128, 16, 4, 9
    q, kk, vv, res = _setup(seed=4, B=B, H=H, N=N, d=d, m=m, k=k)
    g = torch.Generator().manual_seed(11)
    perm = torch.randperm(N, generator=g)
    res2 = oracle.forward(q, kk[:, :, perm].contiguous(), vv[:, :, perm].contiguous(), 1, N, m, k, 1)
    assert torch.allclose(res2["out"], res["out"], rtol=0, atol=1e-12)
    assert torch.allclose(res2["v_tilde"], res["v_tilde"], rtol=0, atol=1e-12)
    mapped = perm[res2["topk_idx"].long()].sort(-1).values
    assert bool((res["topk_gap"] > 1e-9).all())     # tie-free, so sets are unique
    assert torch.equal(mapped.int(), res["topk_idx"])


def test_unselected_kv_still_contributes_through_shared_values():
    """Tutorial ch. 5 quiz: a KV row outside every top-k still reaches the
    output through v~.  Changing such a V row changes the output."""
    B, H, N, d, m, k = 1, 1, 64, 8, 2, 3
    q, kk, vv, res = _setup(seed=5, B=B, H=H, N=N, d=d, m=m, k=k, dtype="f32")
    used = set(res["topk_idx"].view(-1).tolist())
    j = next(i for i in range(N) if i not in used)
    vv2 = vv.clone()
    vv2[0, 0, j] += 10.0
    res2 = oracle.forward(q, kk, vv2, 1, N, m, k, 1)
    assert (res2["out"] - res["out"]).abs().max().item() > 1e-6
    assert torch.equal(res2["topk_idx"], res["topk_idx"])


def test_entry_count_is_m_plus_sk():
    """Each query attends m + s*k entries (tutorial ch. 4 step 5): with all
    logits equal the output is the plain mean over exactly those entries."""
    B, H, N, d, m, k, s = 1, 1, 16, 4, 4, 3, 2
    q = torch.zeros((B, H, N, d), dtype=torch.float64)
    kk = torch.zeros_like(q)
    vv = _rand((B, H, N, d), torch.float64, 31)
    res = oracle.forward(q, kk, vv, 1, N, m, k, s)
    vt = vv.mean(2)                                    # uniform softmax over all N
    for n in range(N):
        rows = torch.cat([res["topk_idx"][0, 0, e].long() for e in res["route"][0, 0, n]])
        ref = (m * vt[0, 0] + vv[0, 0, rows].sum(0)) / (m + s * k)
        assert torch.allclose(res["out"][0, 0, n], ref, rtol=0, atol=1e-14)


def test_tiny_workload_runs():
    w = W.WORKLOADS["tiny_1d"]
    q, k, v = W.make_qkv(w, 0)
    res = oracle.forward(q, k, v, w.grid_h, w.grid_w, w.m, w.topk, w.s)
    assert res["out"].shape == (1, 1, 64, 16)
    assert bool(torch.isfinite(res["out"]).all())
    assert res["bucket_off"][0, 0, -1].item() == 64


# ----------------------------------------------------------------------------
# Dense attention and the routing-only ablation
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_dense_matches_library_attention(dtype):
    """The dense baseline is the textbook softmax(Q K^T / sqrt(d)) V."""
    B, H, N, d = 2, 3, 200, 16
    q, k, v = (_rand((B, H, N, d), dtype, s) for s in (11, 12, 13))
    out = oracle.dense(q, k, v)
    ref = F.scaled_dot_product_attention(q.double(), k.double(), v.double())
    assert torch.allclose(out, ref, rtol=0, atol=1e-12)
    sel = torch.tensor([0, 5, N - 1, N, B * H * N - 1])
    assert torch.allclose(oracle.dense(q, k, v, queries=sel), ref.reshape(-1, d)[sel],
                          rtol=0, atol=1e-12)


def test_routed_only_single_expert_of_all_keys_is_dense():
    """Routing only, m = 1, k = N: the one expert holds every key, so the output is
    dense attention (no shared pair)."""
    B, H, N, d = 1, 2, 96, 16
    q, k, v, res = _setup(seed=14, B=B, H=H, N=N, d=d, m=1, k=N)
    out = oracle.attend(q, k, v, res["q_tilde"], res["v_tilde"], res["topk_idx"], res["route"],
                        branches="routed")
    ref = F.scaled_dot_product_attention(q.double(), k.double(), v.double())
    assert torch.allclose(out, ref, rtol=0, atol=1e-12)
    # with the shared branch the same call differs (one more pair in the softmax)
    assert (res["out"] - ref).abs().max().item() > 1e-3


@pytest.mark.parametrize("s", [1, 2])
def test_routed_only_is_softmax_over_the_routed_rows(s):
    q, k, v, res = _setup(seed=15, s=s)
    B, H, N, d = q.shape
    out = oracle.attend(q, k, v, res["q_tilde"], res["v_tilde"], res["topk_idx"], res["route"],
                        branches="routed")
    qd, kd, vd = q.double(), k.double(), v.double()
    for b in range(B):
        for h in range(H):
            for n in range(0, N, 5):
                rows = torch.cat([res["topk_idx"][b, h, e].long() for e in res["route"][b, h, n]])
                p = torch.softmax(kd[b, h, rows] @ qd[b, h, n] / math.sqrt(d), 0)
                assert torch.allclose(out[b, h, n], p @ vd[b, h, rows], rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# Backward (selections held constant)
# ----------------------------------------------------------------------------
from oracle import backward as OB  # noqa: E402


@pytest.mark.parametrize("s,temp,branches,grid", [
    (1, "sqrt_d", "both", None), (2, "d", "both", None), (1, "sqrt_d", "routed", None),
    (1, "sqrt_d", "both", (6, 8, (2, 3)))])
def test_backward_forward_matches_c_oracle(s, temp, branches, grid):
    """The torch restatement the backward differentiates gives the C oracle's output."""
    if grid is None:
        B, H, N, d, m, k, gh, gw, lg = 2, 2, 96, 16, 6, 10, 1, 96, None
    else:
        gh, gw, lg = grid
        B, H, N, d, m, k = 2, 2, gh * gw, 16, lg[0] * lg[1], 9
    w = W.custom("bw", B, H, N, d, "bf16", gh, gw, m, k, s, index=90)
    q, kk, vv = W.make_qkv(w, 0)
    ref = oracle.forward(q, kk, vv, gh, gw, m, k, s, shared_temperature=temp, landmark_grid=lg,
                         branches=branches)
    out = OB.forward_fixed(q.double(), kk.double(), vv.double(), ref["q_tilde"],
                           ref["topk_idx"], ref["route"], gh, gw, m, lg, temp, branches)
    assert torch.allclose(out, ref["out"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("s,temp,branches", [(1, "sqrt_d", "both"), (2, "d", "both"),
                                             (2, "sqrt_d", "routed")])
def test_backward_matches_finite_differences(s, temp, branches):
    """gradcheck: autograd's gradient of the fixed-selection forward against central
    differences, on fp64 inputs (q~ rounding is then the identity)."""
    B, H, N, d, m, k = 1, 2, 12, 4, 3, 5
    g = torch.Generator().manual_seed(21)
    q, kk, vv = (torch.randn((B, H, N, d), generator=g, dtype=torch.float64) for _ in range(3))
    qt = oracle.pool(q, 1, N, m)
    ti, _, _ = oracle.landmark(qt, kk, vv, k)
    r, _ = oracle.route(q, qt, s)

    def f(a, b_, c_):
        return OB.forward_fixed(a, b_, c_, None, ti, r, 1, N, m, None, temp, branches)

    assert torch.autograd.gradcheck(f, (q.requires_grad_(), kk.requires_grad_(),
                                        vv.requires_grad_()), eps=1e-6, atol=1e-7)


def test_backward_routed_single_expert_is_dense_attention_gradient():
    """Routing only, m = 1, k = N is dense attention, so its gradient is the library
    attention's gradient."""
    B, H, N, d = 1, 2, 40, 8
    g = torch.Generator().manual_seed(22)
    q, kk, vv, do = (torch.randn((B, H, N, d), generator=g, dtype=torch.float64)
                     for _ in range(4))
    got = OB.backward(q, kk, vv, do, 1, N, 1, N, 1, branches="routed")
    qr, kr, vr = (t.clone().requires_grad_(True) for t in (q, kk, vv))
    ref = torch.autograd.grad(F.scaled_dot_product_attention(qr, kr, vr), (qr, kr, vr), do)
    for a, b in zip(got, ref):
        assert torch.allclose(a, b, rtol=0, atol=1e-12)
