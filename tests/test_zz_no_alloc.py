"""mita_bucket_noalloc: the bucket step for callers that cannot allocate.

Callers that hand all device memory to their own allocator, or that forbid
allocation once they are running, cannot let the library grow its workspace
cache.  mita_bucket_noalloc keeps its counters in a fixed 4 MiB device array
inside the library instead.  These tests call it through the C ABI (ctypes)
and check it against the fp64 oracle's grouping and against mita_bucket on two
calls in a row; the second call sees the scratch the first one left behind,
so it also checks that each call clears what it uses.  The cases cover the
per-chunk counters (m <= 2048), the global-counter path (m > 2048) and two
routes per query (N*s entries).  While the no-allocation calls run, the
library's workspace cache is released and capped at one byte, so any call that
tried to allocate would fail.  This file sorts last so that a run stopping at
the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
from sparse_top_landmark_gb300 import build, mita

MITA_OK, MITA_ERR_INVALID_ARG, MITA_ERR_UNSUPPORTED = 0, 1, 2


def _lib():
    build.build()
    return mita.load()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib()
    g = ctypes.c_void_p(1 << 20)     # never dereferenced: the size check fails first
    # 4 * 8 heads * 256 chunks of 4096 queries * 512 experts > 1048576 counters
    rc = lib.mita_bucket_noalloc(g, 4, 8, 1 << 20, 512, 1, g, g, None)
    assert rc == MITA_ERR_UNSUPPORTED
    assert b"static scratch" in lib.mita_last_error_message()
    assert lib.mita_bucket_noalloc(g, 1, 1, 100, 16, 9, g, g, None) == MITA_ERR_UNSUPPORTED
    assert lib.mita_bucket_noalloc(None, 1, 1, 100, 4, 1, g, g, None) == MITA_ERR_INVALID_ARG


# B, H, N, m, s, seed: per-chunk counters; the global-counter path (m > 2048); two routes
SHAPES = [(2, 3, 20000, 77, 1, 11), (1, 2, 9000, 40, 1, 12), (1, 1, 20000, 3000, 1, 13),
          (1, 2, 9000, 40, 2, 14)]


def _routes(B, H, N, m, s, seed):
    g = torch.Generator().manual_seed(seed)
    if s == 1:
        r = torch.randint(0, m, (B, H, N, 1), generator=g, dtype=torch.int32)
        skew = torch.rand((B, H, N, 1), generator=g) < 0.4
        return torch.where(skew, r % 3, r).to(torch.int32).contiguous()
    # s distinct landmarks per query
    return torch.argsort(torch.rand((B, H, N, m), generator=g), dim=-1)[..., :s].to(
        torch.int32).contiguous()


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_mita_bucket_on_two_calls_in_a_row():
    lib = _lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    cases = []
    for B, H, N, m, s, seed in SHAPES:
        r = _routes(B, H, N, m, s, seed)
        ooff, oqidx = oracle.bucket(r, m)
        dr = r.to(dev)
        ref_off, ref_qidx = mita.mita_bucket(dr, m)
        cases.append((B, H, N, m, s, dr, ooff, oqidx, ref_off, ref_qidx))
    torch.cuda.synchronize()
    mita.workspace_release()
    prev = mita.workspace_set_limit(1)
    try:
        for _ in range(2):
            for B, H, N, m, s, dr, ooff, oqidx, ref_off, ref_qidx in cases:
                off = torch.full((B, H, m + 1), -7, dtype=torch.int32, device=dev)
                qidx = torch.full((B, H, N * s), -7, dtype=torch.int32, device=dev)
                rc = lib.mita_bucket_noalloc(ctypes.c_void_p(dr.data_ptr()), B, H, N, m, s,
                                             ctypes.c_void_p(off.data_ptr()),
                                             ctypes.c_void_p(qidx.data_ptr()),
                                             ctypes.c_void_p(stream.cuda_stream))
                assert rc == MITA_OK, lib.mita_last_error_message()
                stream.synchronize()
                assert torch.equal(off.cpu(), ooff), (B, H, N, m, s)
                assert torch.equal(qidx.cpu(), oqidx), (B, H, N, m, s)
                assert torch.equal(off, ref_off)
                assert torch.equal(qidx, ref_qidx)
    finally:
        mita.workspace_set_limit(prev)
