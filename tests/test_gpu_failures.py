"""Failure paths on the GPU, made on the host: an allocation that fails (the workspace cap
injects it before the allocator runs), with no kernel launched and the library usable after."""
import pytest
import torch

from sparse_top_landmark_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MITA_ERR_OOM = 4


def M():
    from sparse_top_landmark_gb300 import build, mita
    build.build()
    return mita


def test_failed_workspace_allocation_returns_oom_and_recovers():
    mita = M()
    w = W.custom("oom", 2, 2, 4096, 64, "bf16", 1, 4096, 32, 64, index=95)
    q, k, v = (t.cuda() for t in W.make_qkv(w, 0))
    mita.workspace_release()                  # the next call must grow the cache
    n0 = mita.kernel_launches()
    prev = mita.workspace_set_limit(1 << 16)
    try:
        with pytest.raises(mita.MitaError) as err:
            mita.mita_forward(q, k, v, 1, w.N, w.m, w.topk)
        assert err.value.status == MITA_ERR_OOM
        assert "workspace limit" in str(err.value)
        assert mita.kernel_launches() == n0   # refused before any launch
    finally:
        mita.workspace_set_limit(prev)
    out = mita.mita_forward(q, k, v, 1, w.N, w.m, w.topk)
    ref = mita.mita_forward(q, k, v, 1, w.N, w.m, w.topk)
    assert mita.get_last_device_error() == 0
    assert torch.equal(out, ref)


def test_bounded_waits_give_up_flag_timeout_and_leave_the_context_usable():
    """A kernel waits on an mbarrier nothing arrives on, with the same whole-warp and
    single-thread wait routines the library's kernels use: both give up after about a
    second, the timeout bit (8) reaches the status word, and a forward runs after it."""
    import time
    mita = M()
    assert mita.get_last_device_error() == 0
    t0 = time.time()
    gave_up = mita.check_bounded_wait()
    bits = mita.get_last_device_error()          # synchronises: the probe has returned
    dt = time.time() - t0
    assert gave_up.cpu().tolist() == [1, 1]
    assert bits == 8
    assert dt < 30, f"the probe took {dt:.1f} s"
    assert mita.get_last_device_error() == 0     # cleared by the read
    w = W.custom("after_timeout", 1, 2, 2048, 64, "bf16", 1, 2048, 16, 32, index=96)
    q, k, v = (t.cuda() for t in W.make_qkv(w, 0))
    out = mita.mita_forward(q, k, v, 1, w.N, w.m, w.topk)
    assert mita.get_last_device_error() == 0
    assert bool(torch.isfinite(out.float()).all())
