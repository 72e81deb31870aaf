"""The reference index tables the library builds on the GPU ("C. Hit
discovery", C.1: inclusive cumulative bucket ends; C.5: each bucket's
reference ends, ascending), exported by hspz_index_tables, against the
oracle's index: idx and pos equal element by element."""
import numpy as np
import pytest

import oracle
from seed_hits_ungapped_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from seed_hits_ungapped_gb300 import hspz
    hspz.load_library()
    return torch


def _references():
    rng = np.random.default_rng(12)
    low = rng.choice(np.array([0, 1], np.uint8), size=30_000, p=[0.7, 0.3])
    low[rng.random(low.size) < 0.01] = 4
    return [("tiny", synth.make("tiny").ref), ("mid_0.05", synth.make("mid", scale=0.05).ref),
            ("chunking_0.02", synth.make("chunking", scale=0.02).ref), ("low_complexity", low),
            ("all_A", np.zeros(5_000, np.uint8)), ("shorter_than_span", np.arange(10, dtype=np.uint8) % 4),
            ("all_N", np.full(3_000, 4, np.uint8))]


@pytest.mark.parametrize("pattern", [oracle.SEED_PATTERN, "11011", "1"])
def test_index_tables_equal_oracle_index(torch_cuda, pattern):
    from seed_hits_ungapped_gb300 import hspz
    torch = torch_cuda
    for name, ref in _references():
        index = hspz.hspz_build_index(torch.from_numpy(ref).cuda(), pattern)
        idx, pos = index.tables()
        want_idx, want_pos = oracle.build_index(ref, pattern)
        assert index.n_positions == want_pos.size, name
        assert np.array_equal(idx.cpu().numpy().view(np.uint32), want_idx), name
        assert np.array_equal(pos.cpu().numpy().view(np.uint32), want_pos), name
        index.close()
