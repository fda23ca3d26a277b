"""The committed oracle regression fixture still matches the oracle bit for bit."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_oracle_regression_fixture(oracle_mod):
    with open(os.path.join(HERE, "golden", "oracle_regression.txt")) as fh:
        stored = fh.read()
    assert make_golden.render() == stored
