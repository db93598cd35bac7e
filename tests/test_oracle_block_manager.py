"""Pins of the block manager oracle (CPU): the pages' worked examples (48 tokens -> 3 blocks,
the 4-token block that fills before the next one opens, 100 requests sharing a 2000-token
prompt, the window's bounded block count), brute-force enumerations over random traces, and the
worker-side table writes and zero fill."""
import pytest

from oracle import block_manager as bmo

from .bm_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_block_manager_oracle_pin(pin):
    pin(bmo)
