"""Plant plausible mistakes in copies of the block manager oracle (on the CPU) and check that a
pin fails for each: the pins would notice the oracle itself going wrong in these ways."""
import importlib.util
import os

import pytest

from .bm_pins import ALL_PINS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "block_manager.py")

MUTANTS = {
    "blocks_floor": ("return (num_tokens + block_size - 1) // block_size",
                     "return num_tokens // block_size"),
    "release_one_late": ("if last_pos > first_query - self.window:",
                         "if last_pos >= first_query - self.window:"),
    "release_one_early": ("if last_pos > first_query - self.window:",
                          "if last_pos > first_query - self.window + 1:"),
    "share_without_count": ("            self.ref[b] += 1\n", "            pass\n"),
    "drop_loses_block": ("            self.free_pool.append(b)\n", "            pass\n"),
    "partial_allocation": ("if missing > len(self.free_pool):", "if missing > len(self.free_pool) + 1:"),
    "zero_fills_shared": ("            self.rows[dst].append(b)\n",
                          "            self.rows[dst].append(b)\n            self.fresh.add(b)\n"),
    "zero_fills_returned": ("if self.ref[b] > 0) if self.zero_fill", "if True) if self.zero_fill"),
    "release_not_staged": ("                self.staged[(row, j)] = -1\n", ""),
    "free_keeps_tokens": ("        self.rows[row] = []\n        self.tokens[row] = 0\n",
                          "        self.rows[row] = []\n"),
    "staged_column_shift": ("self.staged[(row, len(self.rows[row]) - 1)] = b",
                            "self.staged[(row, len(self.rows[row]) % 64)] = b"),
    "apply_rejects_release": ("not (-1 <= v < num_blocks)", "not (0 <= v < num_blocks)"),
    "apply_zeroes_one_cache": ("        for cache in caches:\n", "        for cache in caches[:1]:\n"),
    "share_from_released": ("        if any(b < 0 for b in prefix):\n            return INVALID_ARG\n", ""),
}


def load_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site of {name} not found"
    path = tmp_path / f"bm_{name}.py"
    path.write_text(text.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location(f"bm_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_a_pin_catches_mutant(name, tmp_path):
    mod = load_mutant(name, tmp_path)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception:  # an assertion or a crash: the pin noticed
            failed.append(pin.__name__)
            break
    assert failed, f"no pin fails for the planted mistake {name}"
