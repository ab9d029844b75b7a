"""mita_bucket_noalloc: the bucket step for callers that cannot allocate.

Callers that hand all device memory to their own allocator, or that forbid
allocation once they are running, cannot let the library grow its workspace
cache.  mita_bucket_noalloc keeps its counters in a fixed 4 MiB device array
inside the library instead.  These tests call it through the C ABI (ctypes)
and check it against mita_bucket on two calls in a row; the second call sees
the scratch the first one left behind, so it also checks that each call
clears what it uses.  This file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

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


@pytest.mark.gpu
def test_noalloc_matches_mita_bucket_on_two_calls_in_a_row():
    lib = _lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    shapes = [(2, 3, 20000, 77, 11), (1, 2, 9000, 40, 12)]   # B, H, N, m, seed
    for B, H, N, m, seed in shapes:
        g = torch.Generator().manual_seed(seed)
        r = torch.randint(0, m, (B, H, N, 1), generator=g, dtype=torch.int32)
        skew = torch.rand((B, H, N, 1), generator=g) < 0.4
        r = torch.where(skew, r % 3, r).to(torch.int32).to(dev).contiguous()
        ref_off, ref_qidx = mita.mita_bucket(r, m)
        off = torch.full((B, H, m + 1), -7, dtype=torch.int32, device=dev)
        qidx = torch.full((B, H, N), -7, dtype=torch.int32, device=dev)
        rc = lib.mita_bucket_noalloc(ctypes.c_void_p(r.data_ptr()), B, H, N, m, 1,
                                     ctypes.c_void_p(off.data_ptr()),
                                     ctypes.c_void_p(qidx.data_ptr()),
                                     ctypes.c_void_p(stream.cuda_stream))
        assert rc == MITA_OK, lib.mita_last_error_message()
        stream.synchronize()
        assert torch.equal(off, ref_off)
        assert torch.equal(qidx, ref_qidx)
