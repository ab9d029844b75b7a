"""mita_forward_ex options on the GPU against the fp64 oracle.

* The official code's shared temperature (MiTA tutorial ch. 8 caveat 3): the
  m shared logits are q . q~ / d while the raw logits stay q . k / sqrt(d).
* 2D pooling onto an explicit (possibly non-square) landmark grid.

Same rules as the other parity tests: q~ bit-exact, outputs within the dtype's
tolerance, the long workload on sampled queries in the benchmark's launch
configuration.
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


TEMP_CASES = {
    # name: (workload, s) -- bf16 d = 64 runs the tensor-core expert kernel, the rest SIMT
    "tiny_f32": (W.WORKLOADS["tiny_1d"], 1),
    "vit_bf16_tc": (W.WORKLOADS["vit_s_14x14"], 1),
    "seg_bf16_tc": (W.WORKLOADS["seg_32x32"], 1),
    "d32_bf16_simt": (W.custom("d32_bf16", 2, 3, 2000, 32, "bf16", 1, 2000, 20, 50,
                               index=41), 1),
    "seg_bf16_s2": (W.WORKLOADS["seg_32x32"], 2),
    "ragged_f32_s3": (W.custom("ragged_f32_t", 2, 2, 999, 64, "f32", 1, 999, 12, 40,
                               index=42), 3),
}


@pytest.mark.parametrize("name", list(TEMP_CASES))
def test_forward_shared_temperature_d(name):
    mita = M()
    w, s = TEMP_CASES[name]
    q, k, v = W.make_qkv(w, 0)
    out = mita.mita_forward_ex(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, s,
                               shared_temperature="d")
    assert mita.get_last_device_error() == 0
    ref = oracle.forward(q, k, v, w.grid_h, w.grid_w, w.m, w.topk, s,
                         shared_temperature="d")["out"]
    assert_close(out.cpu(), ref, w.torch_dtype)
    # the default temperature through the same entry point is mita_forward, bit for bit
    a = mita.mita_forward_ex(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, s)
    b = mita.mita_forward(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, s)
    assert torch.equal(a, b)
    assert not torch.equal(a, out)


def test_forward_shared_temperature_d_long_64k_sampled():
    mita = M()
    w = W.WORKLOADS["long_64k"]
    q, k, v = W.make_qkv(w, 0)
    out = mita.mita_forward_ex(dev(q), dev(k), dev(v), w.grid_h, w.grid_w, w.m, w.topk, 1,
                               shared_temperature="d")
    assert mita.get_last_device_error() == 0
    g = torch.Generator().manual_seed(9)
    total = w.B * w.H * w.N
    sel = torch.unique(torch.cat([torch.tensor([0, total - 1]),
                                  torch.randint(0, total, (1024,), generator=g)]))
    heads = torch.unique(sel // w.N)
    qt = oracle.pool(q, w.grid_h, w.grid_w, w.m)
    rows = (heads[:, None] * w.m + torch.arange(w.m)[None]).flatten()
    ti_r, vt_r, _ = oracle.landmark(qt, k, v, w.topk, rows=rows)
    ti = torch.zeros((w.B * w.H * w.m, w.topk), dtype=torch.int32)
    vt = torch.zeros((w.B * w.H * w.m, w.d), dtype=torch.float64)
    ti[rows], vt[rows] = ti_r, vt_r
    orr, _ = oracle.route(q, qt, 1, queries=sel)
    ref = oracle.attend(q, k, v, qt, vt.view(w.B, w.H, w.m, w.d),
                        ti.view(w.B, w.H, w.m, w.topk), orr, queries=sel,
                        shared_temperature="d")
    assert_close(out.view(-1, w.d).cpu()[sel], ref, w.torch_dtype)


GRID_CASES = [
    # name, B, H, gh, gw, d, dtype, mh, mw, topk
    ("vit_3x5", 8, 2, 14, 14, 64, "bf16", 3, 5, 25),
    ("seg_4x8", 4, 2, 32, 32, 64, "bf16", 4, 8, 49),
    ("rect_2x5_f32", 2, 3, 6, 10, 32, "f32", 2, 5, 12),
    ("tall_7x1", 2, 2, 21, 9, 16, "f32", 7, 1, 30),
]


@pytest.mark.parametrize("case", GRID_CASES, ids=[c[0] for c in GRID_CASES])
def test_nonsquare_landmark_grid(case):
    mita = M()
    name, B, H, gh, gw, d, dt, mh, mw, topk = case
    m = mh * mw
    w = W.custom(name, B, H, gh * gw, d, dt, gh, gw, m, topk, index=50 + GRID_CASES.index(case))
    q, k, v = W.make_qkv(w, 0)
    qt = mita.mita_pool_grid(dev(q), gh, gw, mh, mw)
    oqt = oracle.pool(q, gh, gw, m, landmark_grid=(mh, mw))
    assert torch.equal(qt.cpu().double(), oqt)
    out = mita.mita_forward_ex(dev(q), dev(k), dev(v), gh, gw, m, topk, 1,
                               landmark_grid=(mh, mw))
    assert mita.get_last_device_error() == 0
    ref = oracle.forward(q, k, v, gh, gw, m, topk, 1, landmark_grid=(mh, mw))["out"]
    assert_close(out.cpu(), ref, w.torch_dtype)
    # both options together
    out2 = mita.mita_forward_ex(dev(q), dev(k), dev(v), gh, gw, m, topk, 2,
                                shared_temperature="d", landmark_grid=(mh, mw))
    ref2 = oracle.forward(q, k, v, gh, gw, m, topk, 2, shared_temperature="d",
                          landmark_grid=(mh, mw))["out"]
    assert_close(out2.cpu(), ref2, w.torch_dtype)
