"""The oracle still produces the stored results of tests/golden/ (written by
tests/golden/make_golden.py, which calls only the oracle)."""

import json
import os

from tests.golden.make_golden import tiny_decode_record

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_decode_oracle_unchanged():
    with open(os.path.join(HERE, "tiny_decode_oracle.json")) as f:
        stored = json.load(f)
    assert tiny_decode_record() == stored
