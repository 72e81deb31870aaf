"""hspz_compact_noalloc against hspz_compact and the oracle's compaction.

The no-allocation compaction is for callers that cannot allocate device
memory while they run: their device memory was handed to another allocator
at start-up, or they cannot afford the device synchronization an allocation
may cause.  It keeps its scratch in one fixed array inside the library that
every call reuses, so this test makes two calls in a row -- a large one and
then a smaller one -- and checks each, exactly, against the allocating entry
point and against the oracle: nothing left over from the first call may leak
into the second.  It also checks the property the call exists for: after one
call with no flags on the device (which loads the library's code and array
there), a call leaves the device's free memory unchanged.  The test lives in
a file of its own, collected last, and passes alone or after the others.
"""
import ctypes

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


def test_noalloc_compaction_matches_allocating_compaction_on_two_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from seed_hits_ungapped_gb300 import hspz
    lib = hspz.load_library()
    rng = np.random.default_rng(2024)
    cases = []
    for n, p, base in ((3_000_011, 0.02, 77), (100_003, 0.4, 5)):
        h = (rng.random(n) < p).astype(np.uint8)
        cases.append((h, base, torch.from_numpy(h).cuda(), torch.empty(n, dtype=torch.int32, device="cuda"),
                      torch.full((n,), -1, dtype=torch.int32, device="cuda")))
    # the first call on this device loads the code and the fixed array (n = 0 does only that)
    out = ctypes.c_uint64(7)
    assert lib.hspz_compact_noalloc(None, 0, 0, None, 0, ctypes.byref(out), None) == hspz.HSPZ_OK
    assert out.value == 0
    torch.cuda.synchronize()
    for h, base, flags, want_ids, got_ids in cases:
        n = h.size
        k_want = hspz.hspz_compact(flags, n, base, want_ids)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        k_got = hspz.hspz_compact_noalloc(flags, n, base, got_ids)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before  # no device memory taken
        assert k_got == k_want > 0
        assert torch.equal(got_ids[:k_got], want_ids[:k_want])
        assert np.array_equal(got_ids[:k_got].cpu().numpy().view(np.uint32), oracle.compact(h, base))
    # beyond the fixed scratch: refused before any device access
    limit = lib.hspz_compact_noalloc_max_flags()
    assert limit == 1 << 28
    one = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = lib.hspz_compact_noalloc(ctypes.c_void_p(one.data_ptr()), limit + 1, 0, None, 0, ctypes.byref(out), None)
    assert rc == hspz.HSPZ_E_INVAL
    assert b"2^28" in lib.hspz_last_error()
