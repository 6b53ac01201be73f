"""The oracle still reproduces its committed regression fixture bit for bit.

The fixtures (tests/golden/oracle_small.txt, and oracle_nvfp4_small.txt for the NVFP4
routines) were written by
tests/golden/make_oracle_fixtures.py, which calls only the oracle; see that script for the
closed-form input.  The scheme's pages print no worked example to compare against.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_reproduces_fixture(oracle):
    sys.path.insert(0, os.path.join(HERE, "golden"))
    import make_oracle_fixtures as mk
    with open(os.path.join(HERE, "golden", "oracle_small.txt")) as f:
        stored = f.read()
    assert mk.render() == stored


def test_oracle_reproduces_nvfp4_fixture(oracle):
    sys.path.insert(0, os.path.join(HERE, "golden"))
    import make_oracle_fixtures as mk
    with open(os.path.join(HERE, "golden", "oracle_nvfp4_small.txt")) as f:
        stored = f.read()
    assert mk.render_nvfp4() == stored
