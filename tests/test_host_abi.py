"""Host-side checks that need no GPU: the C ABI loads and exports every entry
point declared in include/hspz.h, and its host logic (keep threshold, MAX_HITS
chunk walk, argument checks) agrees with the oracle."""
import os
import re

import numpy as np
import pytest

import oracle
from seed_hits_ungapped_gb300 import _build, hspz

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(hspz.LIB_PATH):
        _build.build()
    return hspz.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "hspz.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hspz_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(hspz.EXPORTS) == names
    assert lib.hspz_abi_version() == 1


def test_keep_threshold_matches_oracle(lib):
    rng = np.random.default_rng(3)
    Ks = [1, 2, 3000, 2 ** 24 - 1, 2 ** 24, 2 ** 24 + 1, 2 ** 25 + 3, 2 ** 30 - 1, 2 ** 30] + \
        rng.integers(1, 2 ** 30, 200).tolist()
    for K in Ks:
        assert hspz.hspz_keep_threshold(K) == oracle.keep_threshold(K), K
    for bad in (0, -5, 2 ** 30 + 1):
        with pytest.raises(hspz.HspzError):
            hspz.hspz_keep_threshold(bad)


@pytest.mark.parametrize("seed", range(8))
def test_chunk_walk_host_matches_oracle(lib, seed):
    rng = np.random.default_rng(seed)
    S = int(rng.integers(1, 3000))
    cnt = rng.integers(0, 40, S).astype(np.uint32)
    cnt[rng.random(S) < 0.5] = 0
    if seed % 3 == 0:
        cnt[int(rng.integers(0, S))] = 5000  # one seed bucket far above the cap
    if seed % 2 == 0:
        cnt[-300:] = 0
    P, total, rc = oracle.inclusive_prefix(cnt)
    assert rc == 0
    for cap in [0, 1, 7, 64, 255, 256, 257, 1000, max(1, total // 5), total, total + 1]:
        want = oracle.chunk_walk(P, cap)
        for blocks in (True, False):
            got = hspz.hspz_chunk_walk_host(P, cap, use_block_sums=blocks)
            assert np.array_equal(got, want), (cap, blocks)


def test_chunk_walk_host_empty(lib):
    assert hspz.hspz_chunk_walk_host(np.zeros(0, np.uint32), 5).shape == (0, 4)


def test_argument_checks_without_gpu(lib):
    import ctypes
    h = ctypes.c_void_p(0)
    for pat in (b"", b"0110", b"11x1", b"1" * 13, b"1" + b"0" * 40 + b"1"):
        assert lib.hspz_build_index(None, 0, pat, ctypes.byref(h), None) == hspz.HSPZ_E_INVAL
    assert lib.hspz_find_hits(None, None, 0, 0, 0, ctypes.byref(h), None, None) == hspz.HSPZ_E_INVAL
    out = ctypes.c_uint64(7)
    assert lib.hspz_compact(None, 0, 0, None, 0, ctypes.byref(out), None) == hspz.HSPZ_OK and out.value == 0
    assert lib.hspz_compact(None, 5, 0, None, 0, ctypes.byref(out), None) == hspz.HSPZ_E_INVAL
    assert lib.hspz_materialize_plan(None, None, None, 0, 0, None, 0, None, None, None, None) == hspz.HSPZ_E_INVAL
    # the raw-sequence gate and materializer check their arguments before any CUDA call
    params = hspz.score_params(np.eye(5, dtype=np.int32), 10, 3)
    P = ctypes.byref(params)
    assert lib.hspz_score_gate(None, 0, None, 0, None, 0, None, None, None) == hspz.HSPZ_E_INVAL  # no params
    assert lib.hspz_score_gate(None, 0, None, 0, None, 0, P, None, None) == hspz.HSPZ_OK  # nothing to gate
    assert lib.hspz_score_gate(None, 5, None, 0, None, 0, P, None, None) == hspz.HSPZ_E_INVAL  # no anchors
    assert lib.hspz_score_gate(None, 0, None, 10, None, 0, P, None, None) == hspz.HSPZ_E_INVAL  # no reference
    assert lib.hspz_materialize(None, 0, 0, None, 0, None, 0, None, 0, None, None, None, None) == hspz.HSPZ_E_INVAL
    assert lib.hspz_materialize(None, 0, 0, None, 0, None, 0, None, 0, P, None, None, None) == hspz.HSPZ_OK
    assert lib.hspz_materialize(None, 0, 0, None, 3, None, 0, None, 0, P, None, None, None) == hspz.HSPZ_E_INVAL
    bad = hspz.score_params(np.eye(5, dtype=np.int32), -1, 3)  # negative X-drop
    assert lib.hspz_score_gate(None, 0, None, 0, None, 0, ctypes.byref(bad), None, None) == hspz.HSPZ_E_INVAL
    assert lib.hspz_strerror(hspz.HSPZ_E_HIT_OVERFLOW).decode().startswith("total hits")
