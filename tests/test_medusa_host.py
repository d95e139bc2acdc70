"""spec_medusa_topology (host-only C code) against the oracle's pruned Cartesian topology."""

import numpy as np
import pytest

import oracle
import tree_speculative_decoding_split_gb300 as st


@pytest.mark.parametrize("topk,n", [((3, 3, 2), 31), ((3, 3, 2, 2, 1), 63), ((4, 4, 3, 2, 2), 127),
                                    ((6, 5, 4, 3, 3), 255), ((1, 1, 1), 4), ((10,), 11), ((2, 2), 7), ((5,), 1)])
def test_topology_matches_oracle(topk, n):
    p, r = st.medusa_topology(topk, n)
    po, ro = oracle.pruned_topology(topk, n)
    assert (p == po).all() and (r == ro).all()


def test_topology_random_shapes():
    rng = np.random.default_rng(1)
    for _ in range(40):
        K = int(rng.integers(1, 7))
        topk = [int(x) for x in rng.integers(1, 6, size=K)]
        total = sum(int(np.prod(topk[:d])) for d in range(1, K + 1))
        n = int(rng.integers(1, min(255, 1 + total) + 1))
        p, r = st.medusa_topology(topk, n)
        po, ro = oracle.pruned_topology(topk, n)
        assert (p == po).all() and (r == ro).all(), (topk, n)


def test_topology_errors():
    with pytest.raises(st.SpecError) as e:
        st.medusa_topology((3, 3, 2), 32)  # 31 nodes at most
    assert e.value.code == 1
    with pytest.raises(st.SpecError) as e:
        st.medusa_topology((9, 9, 9), 256)
    assert e.value.code == 2
    with pytest.raises(st.SpecError) as e:
        st.medusa_topology((3, 0), 3)
    assert e.value.code == 1
