"""The CPU oracle against what the MoE pages and the mathematics fix (no GPU)."""
import inspect
import re

import pytest

import oracle.moe_oracle as M
import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check()


def test_every_oracle_function_is_called_by_a_pin():
    """Each public function of the oracle is called by name in at least one
    pin, so none of them is trusted only through itself."""
    src = inspect.getsource(oracle_pins)
    public = [n for n, f in vars(M).items()
              if inspect.isfunction(f) and f.__module__ == M.__name__ and not n.startswith("_")]
    assert public
    missing = [n for n in public if not re.search(r"\bO\.%s\(" % n, src)]
    assert not missing, f"oracle functions no pin calls: {missing}"
