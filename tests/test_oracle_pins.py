"""The FP64 oracle against facts fixed outside it (closed forms, brute force, the
pages' merge identity, invariants, finite differences, autograd)."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())


def test_rejects_bad_arguments():
    import numpy as np

    q = np.zeros((4, 2))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, np.zeros((4, 3)), np.zeros((4, 3)), False, 1.0)
    with pytest.raises(RuntimeError):          # causal needs at least as many keys as queries
        oracle.attn_fwd(q, np.zeros((3, 2)), np.zeros((3, 2)), True, 1.0)
    with pytest.raises(RuntimeError):
        oracle.attn_bwd(q, np.zeros((3, 2)), np.zeros((3, 2)), q, True, 1.0)
    with pytest.raises(RuntimeError):          # sampled row out of range
        oracle.attn_fwd(q, q, q, False, 1.0, rows=[4])
