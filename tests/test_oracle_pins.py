"""The FP64 oracle against hand tables, closed forms, library routines on special
cases, invariants and finite differences (CPU only)."""
import pytest

import pins

ALL_PINS = [name for name in dir(pins) if name.startswith("pin_")]


@pytest.mark.parametrize("name", ALL_PINS)
def test_oracle_pin(name):
    getattr(pins, name)()


def test_pack_rejects_negative():
    import oracle
    with pytest.raises(ValueError):
        oracle.pack([(1, 2, 3), (-1, 2, 2)])
