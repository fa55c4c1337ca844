"""The oracle against its pins (CPU only)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    check(orc)


def test_tiny_case_digests():
    """The oracle reproduces the digests stored by tests/golden/make_golden.py."""
    import os
    import sys
    sys.path.insert(0, os.path.join(os.path.dirname(__file__), "golden"))
    import make_golden
    stored = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            k, v = line.split()
            stored[k] = v
    got = {k: str(v) for k, v in make_golden.digests().items()}
    assert got == stored
