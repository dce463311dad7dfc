"""The CPU oracle against its pins (no GPU).  See tests/pins.py for what each
pin ties the oracle to."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.OracleLib(oracle.build())


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


def test_invariant_checker_rejects_bad_results(orc):
    """The invariant checker itself must reject a wrong but plausible result."""
    import numpy as np
    ids = np.array([[2, 0], [1, 2], [2, 3], [0, 2]], np.int32)
    good = orc.permute(ids, 4)
    pins.check_routing_invariants(ids, 4, good)
    bad = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in good.items()}
    p = bad["permuted_idx"]
    p[3], p[4] = p[4], p[3]  # swap two rows inside expert 2's segment
    bad["inv_permuted_idx"][p[3]], bad["inv_permuted_idx"][p[4]] = 3, 4
    with pytest.raises(AssertionError):
        pins.check_routing_invariants(ids, 4, bad)
