"""mita_backward on the GPU against the fp64 oracle's backward.

Reading (the pages give no gradient through the selections): top-k key sets and
routes held constant, q~'s rounding passed straight through; the oracle is the
autograd gradient of a plain fp64 restatement of the forward, pinned by finite
differences.  The GPU computes every gradient in fp32 from the same inputs:
fp32 inputs must agree to rel-L2 1e-5; bf16 inputs use the forward's bf16 output
tolerance on the relative L2 error (5e-3), since the recomputed v~ may come from
the tensor-core landmark path with bf16 softmax weights.  Element by element,
every gradient entry must also lie within the forward's max-abs bound (1e-4 for
fp32, 2e-2 for bf16) scaled by the gradient's own largest magnitude: gradients
are sums over many queries, so their scale is not the O(1) scale of the outputs.
"""
import pytest
import torch

from oracle import backward as OB
from sparse_top_landmark_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    # name: (workload, s, options)
    "tiny_f32": (W.WORKLOADS["tiny_1d"], 1, {}),
    "f32_d32_s1": (W.custom("b1", 2, 2, 300, 32, "f32", 1, 300, 6, 10, index=71), 1, {}),
    "f32_d64_s2": (W.custom("b2", 1, 2, 256, 64, "f32", 1, 256, 8, 12, index=72), 2, {}),
    "f32_routed": (W.custom("b3", 2, 1, 200, 16, "f32", 1, 200, 5, 9, index=73), 1,
                   {"branches": "routed"}),
    "f32_temp_d_grid": (W.custom("b4", 1, 2, 120, 32, "f32", 10, 12, 6, 8, index=74), 1,
                        {"shared_temperature": "d", "landmark_grid": (2, 3)}),
    "bf16_d64_s1": (W.custom("b5", 2, 2, 512, 64, "bf16", 1, 512, 16, 24, index=75), 1, {}),
    "bf16_d64_s3": (W.custom("b6", 1, 2, 400, 64, "bf16", 1, 400, 10, 16, index=76), 3, {}),
    "bf16_d128": (W.custom("b7", 1, 2, 256, 128, "bf16", 1, 256, 4, 20, index=77), 1, {}),
    "bf16_vit_2d": (W.custom("b8", 2, 2, 196, 64, "bf16", 14, 14, 25, 25, index=78), 1, {}),
    # several 64-row chunks per CTA, and streams split over CTAs (shared and v~ passes)
    "bf16_multi_chunk": (W.custom("b10", 1, 2, 4096, 64, "bf16", 1, 4096, 64, 256, index=80), 1,
                         {}),
    # top-k and buckets longer than one CTA's stream (the raw pass split both ways), s = 2
    "bf16_long_lists_s2": (W.custom("b11", 1, 1, 3000, 64, "bf16", 1, 3000, 3, 1100, index=81), 2,
                           {}),
    "bf16_routed_d64": (W.custom("b12", 1, 2, 2048, 64, "bf16", 1, 2048, 32, 96, index=82), 1,
                        {"branches": "routed"}),
    # more than 1 024 landmarks: the v~ pass splits its landmark stream (dk, dv are added)
    "bf16_many_landmarks": (W.custom("b14", 1, 1, 2048, 64, "bf16", 1, 2048, 1100, 8, index=84),
                            1, {}),
    # s = 1 with top-k lists over 1 024 rows: the routed dq launch is split (dq is added)
    "bf16_s1_long_topk": (W.custom("b15", 1, 2, 2048, 64, "bf16", 1, 2048, 2, 1100, index=85), 1,
                          {}),
}


def M():
    from sparse_top_landmark_gb300 import build, mita
    build.build()
    return mita


def _rel(a, b):
    return (torch.linalg.vector_norm(a.double() - b) / torch.linalg.vector_norm(b)).item()


def _max_abs(a, b):
    """(max |a - b|, max |b|) over all entries."""
    return (a.double() - b).abs().max().item(), b.abs().max().item()


@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name):
    mita = M()
    w, s, opt = CASES[name]
    q, k, v = W.make_qkv(w, 0)
    g = torch.Generator().manual_seed(5)
    dout = torch.randn(q.shape, generator=g).to(q.dtype)
    dq, dk, dv = mita.mita_backward(q.cuda(), k.cuda(), v.cuda(), dout.cuda(), w.grid_h, w.grid_w,
                                    w.m, w.topk, s, **opt)
    assert mita.get_last_device_error() == 0
    ref = OB.backward(q, k, v, dout, w.grid_h, w.grid_w, w.m, w.topk, s, **opt)
    tol = 1e-5 if w.dtype == "f32" else 5e-3
    atol = 1e-4 if w.dtype == "f32" else 2e-2
    for got, want, nm in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        err = _rel(got.cpu(), want)
        assert err <= tol, f"{name} {nm}: rel-L2 {err:.3e} > {tol}"
        mx, scale = _max_abs(got.cpu(), want)
        assert mx <= atol * max(scale, 1.0), (f"{name} {nm}: max-abs {mx:.3e} > {atol} x "
                                              f"max(|grad|, 1) = {atol * max(scale, 1.0):.3e}")


def test_autograd_function_trains_like_the_oracle():
    """loss = sum(out * w): gradients through MiTAFunction equal the oracle's for dout = w."""
    mita = M()
    w = W.custom("b9", 2, 2, 256, 32, "f32", 1, 256, 8, 16, index=79)
    q, k, v = W.make_qkv(w, 0)
    wt = torch.randn(q.shape, generator=torch.Generator().manual_seed(6))
    qc, kc, vc = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out = mita.MiTAFunction.apply(qc, kc, vc, 1, w.N, w.m, w.topk, 2)
    (out * wt.cuda()).sum().backward()
    ref = OB.backward(q, k, v, wt, 1, w.N, w.m, w.topk, 2)
    for got, want in zip((qc.grad, kc.grad, vc.grad), ref):
        assert _rel(got.cpu(), want) <= 1e-5
        mx, scale = _max_abs(got.cpu(), want)
        assert mx <= 1e-4 * max(scale, 1.0)



@pytest.mark.parametrize("offset", [1, 2])
def test_backward_rejects_unaligned_gradient_buffers(offset):
    """Gradient buffers offset by 4 or 8 bytes are refused on the host (invalid argument,
    the 16-byte atomic adds need aligned rows) before anything is written to them."""
    import ctypes
    mita = M()
    w = W.custom("b13", 1, 2, 1024, 64, "bf16", 32, 32, 16, 48, index=83)
    q, k, v = (t.cuda() for t in W.make_qkv(w, 0))
    dout = torch.randn(q.shape, generator=torch.Generator().manual_seed(7)).to(q.dtype).cuda()
    n = q.numel()
    bufs = [torch.full((n + 4,), 7.0, dtype=torch.float32, device="cuda") for _ in range(3)]
    views = [b[offset:offset + n].view(q.shape) for b in bufs]
    B, H, N, d = q.shape
    opt = mita._options("sqrt_d", None, "both")
    rc = mita._fn("mita_backward", q.dtype)(
        mita._ptr(q), mita._ptr(k), mita._ptr(v), mita._ptr(dout), B, H, N, d, w.grid_h,
        w.grid_w, w.m, w.topk, 1, ctypes.byref(opt), mita._ptr(views[0]), mita._ptr(views[1]),
        mita._ptr(views[2]), mita._stream(None, q.device))
    assert rc == 1, rc   # MITA_ERR_INVALID_ARG
    assert "16-byte aligned" in mita.load().mita_last_error_message().decode()
    torch.cuda.synchronize()
    assert all(torch.all(b == 7.0).item() for b in bufs)
