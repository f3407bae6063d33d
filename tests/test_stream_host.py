"""The library's host-side subset schedule of the streaming codebook
synchronisation (mapl_stream_subset, C) equals the oracle's independent
implementation of the same published generator and shuffle.  CPU only."""
import numpy as np
import pytest

import oracle
import pipeline_activation_compression_gb300 as mapl


@pytest.fixture(scope="module")
def lib():
    mapl.build()
    return mapl.load_library()


@pytest.mark.parametrize("total,per,seed", [(2048, 410, 0), (2048, 8, 12345),
                                            (97, 20, 5), (1, 1, 3), (4096, 4096, 2**63 + 7)])
def test_subset_matches_oracle(lib, total, per, seed):
    n_sub = -(-total // per)
    for step in list(range(min(n_sub, 6))) + [n_sub, n_sub + 1, 3 * n_sub + 2]:
        got = mapl.mapl_stream_subset(total, per, seed, step)
        want = oracle.stream_subset(total, per, seed, step)
        assert np.array_equal(got, want), (total, per, seed, step)


def test_subset_arguments(lib):
    for args in [(0, 1, 0, 0), (10, 0, 0, 0), (10, 11, 0, 0), (10, 5, 0, -1)]:
        with pytest.raises(mapl.MaplError):
            mapl.mapl_stream_subset(*args)
