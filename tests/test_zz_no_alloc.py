"""hspz_compact_noalloc against hspz_compact.

The no-allocation compaction is for callers that cannot allocate device
memory while they run (their device memory belongs to another allocator, or
they cannot afford the device synchronization an allocation may cause).  It
keeps its scratch in one fixed array inside the library that every call
reuses, so this test makes two calls in a row -- a large one and then a
smaller one -- and checks each against the allocating entry point exactly:
nothing left over from the first call may leak into the second.  It lives in
a file of its own, collected last.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_noalloc_compaction_matches_allocating_compaction_on_two_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from seed_hits_ungapped_gb300 import hspz
    lib = hspz.load_library()
    rng = np.random.default_rng(2024)
    for n, p, base in ((3_000_011, 0.02, 77), (100_003, 0.4, 5)):
        flags = torch.from_numpy((rng.random(n) < p).astype(np.uint8)).cuda()
        want_ids = torch.empty(n, dtype=torch.int32, device="cuda")
        got_ids = torch.full((n,), -1, dtype=torch.int32, device="cuda")
        k_want = hspz.hspz_compact(flags, n, base, want_ids)
        k_got = hspz.hspz_compact_noalloc(flags, n, base, got_ids)
        assert k_got == k_want > 0
        assert torch.equal(got_ids[:k_got], want_ids[:k_want])
    # beyond the fixed scratch: refused before any device access
    out = ctypes.c_uint64(0)
    limit = lib.hspz_compact_noalloc_max_flags()
    assert limit == 1 << 28
    one = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = lib.hspz_compact_noalloc(ctypes.c_void_p(one.data_ptr()), limit + 1, 0, None, 0, ctypes.byref(out), None)
    assert rc == hspz.HSPZ_E_INVAL
    assert b"2^28" in lib.hspz_last_error()
