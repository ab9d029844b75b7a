"""Dense attention and the routing-only ablation on the GPU against the fp64 oracle.

* mita_dense_attn: softmax(q k^T / sqrt(d)) v over all keys, the baseline of the
  long-sequence throughput comparison (tutorial ch. 7 figure 5).
* mita_forward_ex(branches="routed"): the model without the shared branch that
  the bit.fan article's LRA ablation compares against.
"""
import pytest
import torch

import oracle
from parity_util import assert_close
from sparse_top_landmark_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def M():
    from sparse_top_landmark_gb300 import build, mita
    build.build()
    return mita


def dev(t):
    return t.cuda().contiguous()


DENSE = [
    # name, B, H, N, d, dtype  (bf16 d = 64: tensor cores; the rest SIMT)
    ("tc_1000", 2, 2, 1000, 64, "bf16"),
    ("tc_ragged_300", 3, 1, 300, 64, "bf16"),
    ("tc_one_key", 2, 2, 1, 64, "bf16"),
    ("simt_f32_d32", 2, 2, 500, 32, "f32"),
    ("simt_bf16_d128", 1, 2, 700, 128, "bf16"),
]


@pytest.mark.parametrize("case", DENSE, ids=[c[0] for c in DENSE])
def test_dense_attention(case):
    mita = M()
    name, B, H, N, d, dt = case
    w = W.custom(name, B, H, N, d, dt, 1, N, 1, 1, index=60 + DENSE.index(case))
    q, k, v = W.make_qkv(w, 0)
    out = mita.mita_dense_attn(dev(q), dev(k), dev(v))
    assert mita.get_last_device_error() == 0
    assert_close(out.cpu(), oracle.dense(q, k, v), w.torch_dtype)


def test_dense_attention_64k_sampled():
    """A 64K-token sequence (the throughput comparison's size), sampled queries."""
    mita = M()
    w = W.custom("dense_64k", 1, 2, 65536, 64, "bf16", 1, 65536, 1, 1, clusters=64, index=66)
    q, k, v = W.make_qkv(w, 0)
    out = mita.mita_dense_attn(dev(q), dev(k), dev(v))
    assert mita.get_last_device_error() == 0
    g = torch.Generator().manual_seed(3)
    sel = torch.unique(torch.cat([torch.tensor([0, 65535, 65536, 2 * 65536 - 1]),
                                  torch.randint(0, 2 * 65536, (256,), generator=g)]))
    ref = oracle.dense(q, k, v, queries=sel)
    assert_close(out.view(-1, 64).cpu()[sel], ref, w.torch_dtype)


ROUTED = {
    # name: (workload, s)
    "tiny_f32": (W.WORKLOADS["tiny_1d"], 1),
    "vit_bf16_tc": (W.WORKLOADS["vit_s_14x14"], 1),
    "seg_bf16_tc": (W.WORKLOADS["seg_32x32"], 1),
    # the equal-entry setting: topk = m + k of the MiTA model it is compared with
    "equal_entries_bf16_tc": (W.custom("eq_entries", 4, 2, 4096, 64, "bf16", 1, 4096, 32, 64,
                                       index=67), 1),
    "seg_bf16_s2": (W.WORKLOADS["seg_32x32"], 2),
    "d32_f32_s3": (W.custom("routed_d32", 2, 2, 1500, 32, "f32", 1, 1500, 15, 40, index=68), 3),
}


@pytest.mark.parametrize("name", list(ROUTED))
def test_routing_only_forward(name):
    mita = M()
    w, s = ROUTED[name]
    q, k, v = W.make_qkv(w, 0)
    out = mita.mita_forward_ex(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, s,
                               branches="routed")
    assert mita.get_last_device_error() == 0
    ref = oracle.forward(q, k, v, w.grid_h, w.grid_w, w.m, w.topk, s, branches="routed")["out"]
    assert_close(out.cpu(), ref, w.torch_dtype)
    both = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, s)
    assert not torch.equal(both, out)


def test_routing_only_single_expert_of_all_keys_is_dense():
    """m = 1, k = N without the shared branch is dense attention (oracle pin); the GPU's
    two paths agree with it."""
    mita = M()
    w = W.custom("one_expert", 2, 2, 1024, 64, "bf16", 1, 1024, 1, 1024, index=69)
    q, k, v = W.make_qkv(w, 0)
    routed = mita.mita_forward_ex(dev(q), dev(k), dev(v), 1, w.N, 1, w.N, 1, branches="routed")
    dense = mita.mita_dense_attn(dev(q), dev(k), dev(v))
    ref = oracle.dense(q, k, v)
    assert_close(routed.cpu(), ref, w.torch_dtype)
    assert_close(dense.cpu(), ref, w.torch_dtype)


def test_routing_only_long_64k_sampled():
    mita = M()
    w = W.WORKLOADS["long_64k"]
    q, k, v = W.make_qkv(w, 0)
    out = mita.mita_forward_ex(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, 1,
                               branches="routed")
    assert mita.get_last_device_error() == 0
    g = torch.Generator().manual_seed(13)
    total = w.B * w.H * w.N
    sel = torch.unique(torch.randint(0, total, (1024,), generator=g))
    heads = torch.unique(sel // w.N)
    qt = oracle.pool(q, w.grid_h, w.grid_w, w.m)
    rows = (heads[:, None] * w.m + torch.arange(w.m)[None]).flatten()
    ti_r, vt_r, _ = oracle.landmark(qt, k, v, w.topk, rows=rows)
    ti = torch.zeros((w.B * w.H * w.m, w.topk), dtype=torch.int32)
    vt = torch.zeros((w.B * w.H * w.m, w.d), dtype=torch.float64)
    ti[rows], vt[rows] = ti_r, vt_r
    orr, _ = oracle.route(q, qt, 1, queries=sel)
    ref = oracle.attend(q, k, v, qt, vt.view(w.B, w.H, w.m, w.d), ti.view(w.B, w.H, w.m, w.topk),
                        orr, queries=sel, branches="routed")
    assert_close(out.view(-1, w.d).cpu()[sel], ref, w.torch_dtype)
