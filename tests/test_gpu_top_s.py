"""Top-s routing (s > 1) on the GPU against the fp64 oracle.

With s > 1 every query keeps its s best landmarks (best first), sits in s
buckets, and attends over m + s*k entries: the shared pairs plus the raw pairs
of all s experts, rows two experts share counted twice (the literal
concatenation).  Same comparison rules as the s = 1 parity tests: stage tests
feed the oracle's upstream outputs into each GPU stage; routes match except
at near ties (1e-6 relative), buckets bit-exactly, outputs within the dtype's
tolerance.
"""
import functools

import pytest
import torch

import oracle
from parity_util import assert_close, assert_ranked_routes_match
from sparse_top_landmark_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_f32_s2": (W.WORKLOADS["tiny_1d"], 2),
    "tiny_f32_s_eq_m": (W.WORKLOADS["tiny_1d"], 4),
    "vit_bf16_s3": (W.WORKLOADS["vit_s_14x14"], 3),
    "seg_bf16_s8": (W.WORKLOADS["seg_32x32"], 8),
    "ragged_f32_d32_s3": (W.custom("ragged_f32", 2, 3, 1000, 32, "f32", 1, 1000, 10, 37,
                                   index=31), 3),
    "d128_bf16_s2": (W.custom("d128_bf16", 1, 2, 2048, 128, "bf16", 1, 2048, 16, 64,
                              index=32), 2),
    # bf16, d = 64, s = 2: the tensor-core route (m <= 256) and expert partials
    "vit_bf16_s2": (W.WORKLOADS["vit_s_14x14"], 2),
    "seg_bf16_s2": (W.WORKLOADS["seg_32x32"], 2),
    "ragged_bf16_m200_s2": (W.custom("ragged_bf16", 2, 2, 3000, 64, "bf16", 1, 3000, 200, 40,
                                     index=34), 2),
    "m256_bf16_s2": (W.custom("m256_bf16", 1, 2, 4096, 64, "bf16", 1, 4096, 256, 24,
                              index=35), 2),
    # m > 256: the SIMT route, then the tensor-core expert partials
    "m300_bf16_s2": (W.custom("m300_bf16", 1, 1, 3000, 64, "bf16", 1, 3000, 300, 20,
                              index=36), 2),
}
NAMES = list(CASES)


def M():
    from sparse_top_landmark_gb300 import build, mita
    build.build()
    return mita


def dev(t):
    return t.cuda().contiguous()


@functools.lru_cache(maxsize=None)
def inputs(name):
    w, s = CASES[name]
    q, k, v = W.make_qkv(w, 0)
    qt = oracle.pool(q, w.grid_h, w.grid_w, w.m)
    oti, ovt, _ = oracle.landmark(qt, k, v, w.topk)
    orr, _ = oracle.route(q, qt, s)
    return w, s, q, k, v, qt, oti, ovt, orr


@pytest.mark.parametrize("name", NAMES)
def test_route_top_s(name):
    mita = M()
    w, s, q, k, v, qt, oti, ovt, orr = inputs(name)
    dq, dqt, dvt = dev(q), dev(qt.to(w.torch_dtype)), dev(ovt.float())
    r, lse, so = mita.mita_route(dq, dqt, dvt, s=s, shared=True)
    assert r.shape == (w.B, w.H, w.N, s)
    assert_ranked_routes_match(r.cpu(), orr, q, qt)
    # the s chosen landmarks are distinct
    rs = r.cpu().sort(-1).values
    assert bool((rs[..., 1:] != rs[..., :-1]).all())
    # the shared partial does not depend on s: bit for bit where s = 1 also runs the SIMT
    # route kernel; bf16 with d = 64 routes s = 1 on the tensor cores (P and v~ in bf16), so
    # there the two agree to the bf16 output tolerance
    _, lse1, so1 = mita.mita_route(dq, dqt, dvt, s=1, shared=True)
    if w.dtype == "bf16" and w.d == 64:
        assert (lse.cpu() - lse1.cpu()).abs().max().item() <= 1e-4 * max(1.0, lse.abs().max().item())
        assert_close(so1.cpu(), so.cpu().double(), torch.bfloat16, "shared o, s = 1 vs s")
    else:
        assert torch.equal(lse.cpu(), lse1.cpu()) and torch.equal(so.cpu(), so1.cpu())
    assert mita.get_last_device_error() == 0


@pytest.mark.parametrize("name", NAMES)
def test_bucket_top_s_bit_exact(name):
    mita = M()
    w, s, q, k, v, qt, oti, ovt, orr = inputs(name)
    off, qidx = mita.mita_bucket(dev(orr), w.m)
    ooff, oqidx = oracle.bucket(orr, w.m)
    assert qidx.shape == (w.B, w.H, w.N * s)
    assert torch.equal(off.cpu(), ooff)
    assert torch.equal(qidx.cpu(), oqidx)
    # skewed routes: 70 % of the queries pick the same s experts, the rest s random distinct ones
    g = torch.Generator().manual_seed(11)
    perm = torch.argsort(torch.rand((w.B, w.H, w.N, w.m), generator=g), dim=-1)[..., :s]
    hot = torch.rand((w.B, w.H, w.N, 1), generator=g) < 0.7
    fixed = torch.arange(s).flip(0).expand(w.B, w.H, w.N, s)
    r = torch.where(hot, fixed, perm).to(torch.int32).contiguous()
    off, qidx = mita.mita_bucket(dev(r), w.m)
    ooff, oqidx = oracle.bucket(r, w.m)
    assert torch.equal(off.cpu(), ooff)
    assert torch.equal(qidx.cpu(), oqidx)
    off2, qidx2 = mita.mita_bucket_noalloc(dev(r), w.m, torch.empty_like(off),
                                           torch.empty_like(qidx))
    assert torch.equal(off2.cpu(), ooff) and torch.equal(qidx2.cpu(), oqidx)
    assert mita.get_last_device_error() == 0


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("carried", [False, True])
def test_expert_top_s(name, carried):
    mita = M()
    w, s, q, k, v, qt, oti, ovt, orr = inputs(name)
    ooff, oqidx = oracle.bucket(orr, w.m)
    dq, dk, dv = dev(q), dev(k), dev(v)
    dqt, dvt = dev(qt.to(w.torch_dtype)), dev(ovt.float())
    lse = so = None
    if carried:
        _, lse, so = mita.mita_route(dq, dqt, dvt, s=1, shared=True)
    out = mita.mita_expert_attn(dq, dk, dv, dqt, dvt, dev(oti), dev(ooff), dev(oqidx), lse, so,
                                s=s)
    ref = oracle.attend(q, k, v, qt, ovt, oti, orr)
    assert_close(out.cpu(), ref, w.torch_dtype)
    assert mita.get_last_device_error() == 0


@pytest.mark.parametrize("name", NAMES)
def test_forward_top_s(name):
    mita = M()
    w, s, q, k, v, qt, oti, ovt, orr = inputs(name)
    out = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, s)
    assert mita.get_last_device_error() == 0
    ref = oracle.attend(q, k, v, qt, ovt, oti, orr)
    assert_close(out.cpu(), ref, w.torch_dtype)
    # s = 1 and s > 1 differ (the extra experts' rows enter the softmax)
    out1 = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, 1)
    assert not torch.equal(out.cpu(), out1.cpu())


def test_forward_top_s_is_deterministic():
    """Partial slots are taken with atomics; the merge orders them by bucket
    position, so repeated runs agree bit for bit."""
    mita = M()
    w, s, q, k, v, *_ = inputs("seg_bf16_s8")
    dq, dk, dv = dev(q), dev(k), dev(v)
    a = mita.mita_forward(dq, dk, dv, w.grid_h, w.grid_w, w.m, w.topk, s)
    b = mita.mita_forward(dq, dk, dv, w.grid_h, w.grid_w, w.m, w.topk, s)
    assert torch.equal(a, b)


def test_route_top_s_equal_landmarks_take_lowest_index():
    """Landmarks 2j and 2j+1 are equal: every near tie is an exact tie, which
    the oracle and the GPU both break towards the lower index."""
    mita = M()
    w = W.custom("dup_lm", 2, 2, 512, 64, "bf16", 1, 512, 32, 16, index=33)
    q, _, _ = W.make_qkv(w, 0)
    qt = oracle.pool(q, 1, 512, 32).to(torch.bfloat16)
    qt = qt[:, :, ::2].repeat_interleave(2, dim=2).contiguous()
    for s in (2, 3, 5):
        r = mita.mita_route(dev(q), dev(qt), s=s)
        orr, _ = oracle.route(q, qt, s)
        assert torch.equal(r.cpu(), orr)
    # with the shared partial, s = 2 routes on the tensor cores (ties go to the exact fix-up)
    vt = torch.randn((w.B, w.H, w.m, w.d), generator=torch.Generator().manual_seed(3))
    r, _, _ = mita.mita_route(dev(q), dev(qt), dev(vt), s=2, shared=True)
    orr, _ = oracle.route(q, qt, 2)
    assert torch.equal(r.cpu(), orr)
    assert mita.get_last_device_error() == 0


def test_forward_top_s_long_64k_sampled():
    """The 64K sequence at s = 2, in the launch configuration of the s = 1
    benchmark, on sampled queries the oracle computes one by one."""
    mita = M()
    w = W.WORKLOADS["long_64k"]
    s = 2
    q, k, v = W.make_qkv(w, 0)
    out = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, s)
    assert mita.get_last_device_error() == 0
    g = torch.Generator().manual_seed(5)
    total = w.B * w.H * w.N
    sel = torch.unique(torch.cat([torch.tensor([0, w.N - 1, total - 1]),
                                  torch.randint(0, total, (1024,), generator=g)]))
    heads = torch.unique(sel // w.N)
    qt = oracle.pool(q, w.grid_h, w.grid_w, w.m)
    rows = (heads[:, None] * w.m + torch.arange(w.m)[None]).flatten()
    ti_r, vt_r, _ = oracle.landmark(qt, k, v, w.topk, rows=rows)
    ti = torch.zeros((w.B * w.H * w.m, w.topk), dtype=torch.int32)
    vt = torch.zeros((w.B * w.H * w.m, w.d), dtype=torch.float64)
    ti[rows], vt[rows] = ti_r, vt_r
    ti = ti.view(w.B, w.H, w.m, w.topk)
    vt = vt.view(w.B, w.H, w.m, w.d)
    orr, _ = oracle.route(q, qt, s, queries=sel)
    r = mita.mita_route(dev(q), dev(qt.to(w.torch_dtype)), s=s)
    assert_ranked_routes_match(r.view(-1, s).cpu()[sel], orr, q, qt, rows=sel)
    ref = oracle.attend(q, k, v, qt, vt, ti, orr, queries=sel)
    assert_close(out.view(-1, w.d).cpu()[sel], ref, w.torch_dtype)
