"""GPU (libmita.so, through the C ABI) against the fp64 oracle.

Stage tests feed the oracle's upstream outputs into each GPU stage, so a
tolerated index difference upstream cannot cascade.  End-to-end tests run
mita_forward exactly as bench.py times it.  Small workloads are compared on
every element; the 64K and 1M workloads on sampled rows/queries the oracle
computes one by one (landmark rows for all heads involved, since every
query's output needs all of its head's shared values).
"""
import functools

import pytest
import torch

import oracle
from parity_util import (assert_close, assert_index_sets_match, assert_routes_match,
                         landmark_scores)
from sparse_top_landmark_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SMALL = ["tiny_1d", "vit_s_14x14", "seg_32x32"]
LARGE = ["long_64k", "long_1m"]


def M():
    from sparse_top_landmark_gb300 import build, mita
    build.build()
    return mita


@functools.lru_cache(maxsize=None)
def inputs(name):
    w = W.WORKLOADS[name]
    return (w,) + W.make_qkv(w, 0)


@functools.lru_cache(maxsize=None)
def oracle_pool(name):
    w, q, k, v = inputs(name)
    return oracle.pool(q, w.grid_h, w.grid_w, w.m)


@functools.lru_cache(maxsize=None)
def oracle_landmark(name):
    w, q, k, v = inputs(name)
    return oracle.landmark(oracle_pool(name), k, v, w.topk)


def dev(t):
    return t.cuda().contiguous()


def sample_queries(w, n=2048, seed=1):
    g = torch.Generator().manual_seed(seed)
    total = w.B * w.H * w.N
    picks = torch.randint(0, total, (n,), generator=g)
    edge = torch.tensor([0, w.N - 1, total - 1, total - w.N])
    return torch.unique(torch.cat([edge, picks]))


# ----------------------------------------------------------------------------
@pytest.mark.parametrize("name", SMALL + LARGE)
def test_pool_bit_exact(name):
    mita = M()
    w, q, k, v = inputs(name)
    qt = mita.mita_pool(dev(q), w.grid_h, w.grid_w, w.m)
    ref = oracle_pool(name)
    got = qt.cpu().double()
    assert torch.equal(got, ref), f"{int((got != ref).sum())} landmark elements differ"


@pytest.mark.parametrize("name", SMALL + ["long_64k"])
def test_landmark_stage(name):
    mita = M()
    w, q, k, v = inputs(name)
    qt = oracle_pool(name).to(w.torch_dtype)
    ti, vt = mita.mita_landmark_topk_shared(dev(qt), dev(k), dev(v), w.topk)
    oti, ovt, gap = oracle_landmark(name)
    assert_index_sets_match(ti.cpu(), oti, gap, exact=True,
                            scores=lambda r: landmark_scores(qt, k, r))
    assert_close(vt.cpu(), ovt, w.torch_dtype, "v_tilde")
    assert mita.get_last_device_error() == 0


def test_landmark_stage_1m_all_rows():
    """Every one of the 1,024 landmark rows of the 1M workload (the oracle's rows
    are the ones the end-to-end test uses)."""
    mita = M()
    name = "long_1m"
    w, q, k, v = inputs(name)
    qt = oracle_pool(name)
    ti, vt = mita.mita_landmark_topk_shared(dev(qt.to(w.torch_dtype)), dev(k), dev(v), w.topk)
    oti, ovt, gap = oracle_landmark(name)
    assert_index_sets_match(ti.cpu(), oti, gap, exact=True,
                            scores=lambda r: landmark_scores(qt, k, r))
    assert_close(vt.cpu(), ovt, w.torch_dtype, "v_tilde")
    assert mita.get_last_device_error() == 0


@pytest.mark.parametrize("name", SMALL + LARGE)
def test_route_stage(name):
    mita = M()
    w, q, k, v = inputs(name)
    qt = oracle_pool(name)
    r = mita.mita_route(dev(q), dev(qt.to(w.torch_dtype)))
    if name in SMALL:
        orr, gap = oracle.route(q, qt, 1)
        assert_routes_match(r.cpu(), orr, gap, q, qt)
    else:
        sel = sample_queries(w, 8192)
        orr, gap = oracle.route(q, qt, 1, queries=sel)
        assert_routes_match(r.view(-1, 1).cpu()[sel], orr, gap, q, qt, rows=sel)


@pytest.mark.parametrize("name", SMALL + LARGE)
def test_bucket_stage_bit_exact(name):
    mita = M()
    w = W.WORKLOADS[name]
    g = torch.Generator().manual_seed(7)
    # skewed synthetic routing: half the queries go to 3 experts
    r = torch.randint(0, w.m, (w.B, w.H, w.N, 1), generator=g, dtype=torch.int32)
    hot = torch.rand((w.B, w.H, w.N, 1), generator=g) < 0.5
    r = torch.where(hot, r % min(3, w.m), r).to(torch.int32).contiguous()
    off, qidx = mita.mita_bucket(dev(r), w.m)
    ooff, oqidx = oracle.bucket(r, w.m)
    assert torch.equal(off.cpu(), ooff)
    assert torch.equal(qidx.cpu(), oqidx)
    assert mita.get_last_device_error() == 0


@pytest.mark.parametrize("name", SMALL + ["long_64k"])
@pytest.mark.parametrize("carried", [False, True])
def test_expert_stage(name, carried):
    mita = M()
    w, q, k, v = inputs(name)
    qt = oracle_pool(name)
    oti, ovt, _ = oracle_landmark(name)
    orr, _ = oracle.route(q, qt, 1)
    ooff, oqidx = oracle.bucket(orr, w.m)
    dq, dk, dv = dev(q), dev(k), dev(v)
    dqt = dev(qt.to(w.torch_dtype))
    dvt = dev(ovt.float())
    lse = so = None
    if carried:
        _, lse, so = mita.mita_route(dq, dqt, dvt, shared=True)
    out = mita.mita_expert_attn(dq, dk, dv, dqt, dvt, dev(oti), dev(ooff), dev(oqidx), lse, so)
    if name in SMALL:
        ref = oracle.attend(q, k, v, qt, ovt, oti, orr)
        assert_close(out.cpu(), ref, w.torch_dtype)
    else:
        sel = sample_queries(w)
        ref = oracle.attend(q, k, v, qt, ovt, oti, orr.view(-1, 1)[sel], queries=sel)
        assert_close(out.view(-1, w.d).cpu()[sel], ref, w.torch_dtype)
    assert mita.get_last_device_error() == 0


@pytest.mark.parametrize("name", SMALL + LARGE)
def test_forward_end_to_end(name):
    mita = M()
    w, q, k, v = inputs(name)
    out = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, w.s)
    assert mita.get_last_device_error() == 0
    qt = oracle_pool(name)
    oti, ovt, _ = oracle_landmark(name)
    if name in SMALL:
        orr, _ = oracle.route(q, qt, 1)
        ref = oracle.attend(q, k, v, qt, ovt, oti, orr)
        assert_close(out.cpu(), ref, w.torch_dtype)
    else:
        sel = sample_queries(w)
        orr, _ = oracle.route(q, qt, 1, queries=sel)
        ref = oracle.attend(q, k, v, qt, ovt, oti, orr, queries=sel)
        assert_close(out.view(-1, w.d).cpu()[sel], ref, w.torch_dtype)


def _host_reference(name):
    w, q, k, v = inputs(name)
    qt = oracle_pool(name)
    oti, ovt, _ = oracle_landmark(name)
    orr, _ = oracle.route(q, qt, 1)
    return oracle.attend(q, k, v, qt, ovt, oti, orr)


# The host-buffer forward pipelines groups of heads (copies of one group overlap the forward of
# another), and each group runs as its own batch: some launch plans (e.g. the landmark stage's
# key splits) depend on the batch's head count, so results may differ from the one-shot device
# forward in the last bits.  Both must meet the oracle tolerance.
def test_forward_host_buffers_match_device_path():
    mita = M()
    w, q, k, v = inputs("seg_32x32")
    dout = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    hout = mita.mita_forward(hq, hk, hv, w.grid_h, w.grid_w, w.m, w.topk)
    assert not hout.is_cuda
    ref = _host_reference("seg_32x32")
    assert_close(hout, ref, w.torch_dtype)
    assert_close(dout.cpu(), ref, w.torch_dtype)
    # a single head runs as one group: identical to the device path
    h1 = mita.mita_forward(hq[:1, :1].contiguous().pin_memory(), hk[:1, :1].contiguous().pin_memory(),
                           hv[:1, :1].contiguous().pin_memory(), w.grid_h, w.grid_w, w.m, w.topk)
    d1 = mita.mita_forward(dev(q[:1, :1]), dev(k[:1, :1]), dev(v[:1, :1]), w.grid_h, w.grid_w,
                           w.m, w.topk)
    assert torch.equal(h1, d1.cpu())


def test_forward_host_pageable_buffers_match_device_path():
    mita = M()
    w, q, k, v = inputs("seg_32x32")
    hout = torch.empty_like(q)                    # pageable, caller-owned
    r = mita.mita_forward(q.contiguous(), k.contiguous(), v.contiguous(), w.grid_h, w.grid_w,
                          w.m, w.topk, out=hout)
    assert r is hout
    assert_close(hout, _host_reference("seg_32x32"), w.torch_dtype)
    pinned = mita.mita_forward(q.pin_memory(), k.pin_memory(), v.pin_memory(), w.grid_h,
                               w.grid_w, w.m, w.topk)
    assert torch.equal(hout, pinned)


@pytest.mark.parametrize("name", ["seg_32x32", "long_64k"])
def test_forward_replays_from_a_cuda_graph(name):
    """mita_forward queues its launches without host synchronisation, so it can be
    captured into a CUDA graph (after one call of the same size has grown the
    stream's workspace) and replayed with the same result."""
    mita = M()
    w, q, k, v = inputs(name)
    dq, dk, dv = dev(q), dev(k), dev(v)
    s = torch.cuda.Stream()
    out = torch.empty_like(dq)
    with torch.cuda.stream(s):
        mita.mita_forward(dq, dk, dv, w.grid_h, w.grid_w, w.m, w.topk, out=out, stream=s)
    s.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        mita.mita_forward(dq, dk, dv, w.grid_h, w.grid_w, w.m, w.topk, out=out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


def test_forward_is_deterministic():
    mita = M()
    w, q, k, v = inputs("long_64k")
    n0 = mita.kernel_launches()
    a = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk)
    n1 = mita.kernel_launches()
    b = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk)
    n2 = mita.kernel_launches()
    assert torch.equal(a, b)
    # the library's own kernels run the forward, the same set each time
    assert n1 - n0 == n2 - n1 >= 10


# ----------------------------------------------------------------------------
# Edge cases: ragged tails, odd sizes, degenerate settings, forced ties
# ----------------------------------------------------------------------------
EDGE = [
    # name,            B, H,    N,   d, dtype,  gh,  gw,   m, topk
    ("ragged_1d",      2, 3, 1000,  64, "bf16",   1, 1000,  37,   45),
    ("uneven_windows", 1, 2,  777,  32, "f32",    1,  777,  10,   13),
    ("grid_2d_rect",   2, 2,  300,  64, "bf16",  12,   25,  16,   20),
    ("k_equals_n",     1, 2,   96,  16, "f32",    1,   96,   4,   96),
    ("k_one",          2, 1,  500,  64, "bf16",   1,  500,   9,    1),
    ("m_one",          1, 3,  300, 128, "bf16",   1,  300,   1,   40),
    ("m_equals_n",     1, 1,   64,  16, "f32",    1,   64,  64,    8),
    ("n_one",          3, 2,    1,  16, "f32",    1,    1,   1,    1),
    ("d128_big_k",     1, 2, 5000, 128, "bf16",   1, 5000,  20,  700),
    ("many_heads",    40, 8,   50,  32, "bf16",   5,   10,   4,    5),
]


@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
def test_edge_case_end_to_end_and_stages(case):
    mita = M()
    name, B, H, N, d, dt, gh, gw, m, topk = case
    w = W.custom(name, B, H, N, d, dt, gh, gw, m, topk, index=200 + EDGE.index(case))
    q, k, v = W.make_qkv(w, 0)
    res = oracle.forward(q, k, v, gh, gw, m, topk, 1)
    dq, dk, dv = dev(q), dev(k), dev(v)
    qt = mita.mita_pool(dq, gh, gw, m)
    assert torch.equal(qt.cpu().double(), res["q_tilde"])
    ti, vt = mita.mita_landmark_topk_shared(dev(res["q_tilde"].to(w.torch_dtype)), dk, dv, topk)
    assert_index_sets_match(ti.cpu(), res["topk_idx"], res["topk_gap"], exact=True,
                            scores=lambda r: landmark_scores(res["q_tilde"], k, r))
    assert_close(vt.cpu(), res["v_tilde"], w.torch_dtype, "v_tilde")
    r = mita.mita_route(dq, dev(res["q_tilde"].to(w.torch_dtype)))
    assert_routes_match(r.cpu(), res["route"], res["route_gap"], q, res["q_tilde"])
    out = mita.mita_forward(dq, dk, dv, gh, gw, m, topk, 1)
    assert_close(out.cpu(), res["out"], w.torch_dtype)
    assert mita.get_last_device_error() == 0


@pytest.mark.parametrize("pattern", ["duplicated_keys", "all_equal_keys", "sorted_keys",
                                     "zero_landmark"])
@pytest.mark.parametrize("N,topk", [(32768, 300), (65536, 64)], ids=["heap_path", "tc_path"])
def test_forced_ties_and_adversarial_order(pattern, N, topk):
    """Mass ties and a key order that puts every top-k member in one split
    drive the exact fallback; the result must still be the lowest-index set.
    (65536, 64) runs the two-pass tensor-core selection, (32768, 300) the
    per-split candidate heaps."""
    mita = M()
    B, H, d, m = 1, 2, 64, 8
    w = W.custom(pattern, B, H, N, d, "bf16", 1, N, m, topk, index=300)
    q, k, v = W.make_qkv(w, 0)
    if pattern == "duplicated_keys":
        k = k[:, :, torch.arange(N) % 5].contiguous()
    elif pattern == "all_equal_keys":
        k = k[:, :, :1].expand(B, H, N, d).contiguous()
    elif pattern == "sorted_keys":
        qt0 = oracle.pool(q, 1, N, m)[:, :, 0]
        s = torch.einsum("bhnd,bhd->bhn", k.double(), qt0)
        order = torch.argsort(s, dim=-1)              # ascending: best keys at the end
        k = torch.gather(k, 2, order.unsqueeze(-1).expand(B, H, N, d)).contiguous()
    elif pattern == "zero_landmark":
        q = q.clone()
        q[:, :, : N // m] = 0                          # landmark 0 pools to exactly 0
    res = oracle.forward(q, k, v, 1, N, m, topk, 1)
    ti, vt = mita.mita_landmark_topk_shared(dev(res["q_tilde"].to(torch.bfloat16)), dev(k), dev(v), topk)
    ti = ti.cpu()
    if pattern == "all_equal_keys":
        # every score of a row is equal: the k lowest indices, in every row
        assert torch.equal(ti, torch.arange(topk, dtype=torch.int32).expand_as(ti))
    if pattern == "zero_landmark":
        # landmark 0 scores every key exactly 0: its k lowest indices
        assert torch.equal(ti[:, :, 0], torch.arange(topk, dtype=torch.int32).expand(B, H, topk))
    if pattern in ("duplicated_keys", "all_equal_keys", "zero_landmark"):
        # exact ties everywhere at the boundary: the lowest-index rule decides every row
        assert torch.equal(ti, res["topk_idx"]), f"{int((ti != res['topk_idx']).any(-1).sum())} rows differ"
    assert_index_sets_match(ti, res["topk_idx"], res["topk_gap"], exact=True,
                            scores=lambda r: landmark_scores(res["q_tilde"], k, r))
    assert_close(vt.cpu(), res["v_tilde"], torch.bfloat16, "v_tilde")
    out = mita.mita_forward(dev(q), dev(k), dev(v), 1, N, m, topk, 1)
    assert_close(out.cpu(), res["out"], torch.bfloat16)


def test_bad_route_values_are_flagged_not_dereferenced():
    mita = M()
    B, H, N, m = 1, 2, 5000, 16
    r = torch.randint(0, m, (B, H, N, 1), dtype=torch.int32)
    r[0, 1, 17, 0] = m + 3
    r[0, 0, 4000, 0] = -1
    off, qidx = mita.mita_bucket(dev(r), m)
    bits = mita.get_last_device_error()
    assert bits & 4
    assert off[0, 0, -1].item() == N - 1
    assert mita.get_last_device_error() == 0         # cleared by the read


def test_bad_expert_index_is_flagged_not_dereferenced():
    mita = M()
    w = W.custom("bad_idx", 1, 1, 256, 64, "bf16", 1, 256, 4, 8, index=400)
    q, k, v = W.make_qkv(w, 0)
    res = oracle.forward(q, k, v, 1, 256, 4, 8, 1)
    ti = res["topk_idx"].clone()
    ti[0, 0, 1, 3] = 10 ** 6
    out = mita.mita_expert_attn(dev(q), dev(k), dev(v), dev(res["q_tilde"].to(torch.bfloat16)),
                                dev(res["v_tilde"].float()), dev(ti), dev(res["bucket_off"]),
                                dev(res["bucket_qidx"]))
    assert mita.get_last_device_error() & 1
    assert bool(torch.isfinite(out.float()).all())


@pytest.mark.parametrize("scale_log2", [17, -20], ids=["values_1e5", "values_1e-6"])
def test_values_outside_fp16_range(scale_log2):
    """Values far beyond fp16's range (|V| ~ 1e5, above 65504) or far below its normal
    range: the shared values v~ and the softmax weights stay in bf16 (fp32's exponent
    range) on the tensor cores, so nothing overflows or flushes.  Head 0's V is scaled by
    a power of two (exact in bf16), head 1's is not; each head must meet the bf16
    tolerance at its own scale."""
    mita = M()
    w = W.custom("scaled_v", 1, 2, 8192, 64, "bf16", 1, 8192, 32, 64, index=410)
    q, k, v = W.make_qkv(w, 0)
    v = v.clone()
    scale = 2.0 ** scale_log2
    v[:, 0] = (v[:, 0].double() * scale).to(torch.bfloat16)
    res = oracle.forward(q, k, v, 1, w.N, w.m, w.topk, 1)
    out = mita.mita_forward(dev(q), dev(k), dev(v), 1, w.N, w.m, w.topk, 1)
    assert mita.get_last_device_error() == 0
    out = out.cpu()
    assert bool(torch.isfinite(out.float()).all())
    assert_close(out[:, 0], res["out"][:, 0], torch.bfloat16, "scaled head", scale=scale)
    assert_close(out[:, 1], res["out"][:, 1], torch.bfloat16, "unscaled head")


@pytest.mark.parametrize("name", ["vit_s_14x14", "seg_32x32", "long_64k"])
def test_route_with_shared_partial(name):
    """mita_route with both shared outputs requested: the tensor-core kernel reuses the
    routing logits q . q~_i as the shared logits (tutorial ch. 6: one dot product for both)
    and emits each query's route, the natural log-sum-exp of the scaled shared logits and
    the normalised shared output.  Routes are exact; lse and o are compared with fp64
    values formed from the oracle's q~ and v~ (o to the bf16 tolerance: P and v~ enter the
    tensor cores in bf16)."""
    mita = M()
    w, q, k, v = inputs(name)
    qt = oracle_pool(name)
    _, ovt, _ = oracle_landmark(name)
    r, lse, so = mita.mita_route(dev(q), dev(qt.to(w.torch_dtype)), dev(ovt.float()), shared=True)
    assert mita.get_last_device_error() == 0
    sel = sample_queries(w, 4096) if name == "long_64k" else torch.arange(w.B * w.H * w.N)
    orr, gap = oracle.route(q, qt, 1, queries=sel)
    assert_routes_match(r.view(-1, 1).cpu()[sel], orr, gap, q, qt, rows=sel)
    qd = q.reshape(-1, w.d)[sel].double()
    lt = qt.reshape(w.B * w.H, w.m, w.d)[sel // w.N]
    vt = ovt.reshape(w.B * w.H, w.m, w.d)[sel // w.N]
    logits = torch.einsum("rd,rmd->rm", qd, lt) / w.d ** 0.5
    ref_lse = torch.logsumexp(logits, -1)
    ref_o = torch.einsum("rm,rmd->rd", torch.softmax(logits, -1), vt)
    got_lse = lse.view(-1).cpu()[sel].double()
    assert (got_lse - ref_lse).abs().max().item() <= 1e-4 * max(1.0, ref_lse.abs().max().item())
    assert_close(so.view(-1, w.d).cpu()[sel], ref_o, torch.bfloat16, "shared o")
