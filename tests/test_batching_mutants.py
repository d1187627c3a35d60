"""The pins of the batch-construction oracle catch plausible mistakes: each
mutant below is one textual change to a copy of oracle/batching.py (the
oracle itself is not touched), loaded as a module of its own; at least one
pin must fail on it."""
import importlib.util
import os

import pytest

from tests.test_batching import pin_min_max_split, pin_stochastic_length

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "batching.py")

MUTANTS = {
    "window start modulus off by one": ("% (len(seq) - max_seq + 1)", "% (len(seq) - max_seq)"),
    "window one token short": ("seq[start:start + max_seq]", "seq[start:start + max_seq - 1]"),
    "window taken from the end": ("seq = seq[start:start + max_seq]", "seq = seq[len(seq) - max_seq:]"),
    "RealTime tokens dropped": ("gid[t] >= 2]", "gid[t] >= 3]"),
    "User tokens dropped": ("if gid[t] == 0]", "if gid[t] == 0 and False]"),
    "groups reordered": ("keep += user + seq + rest", "keep += user + rest + seq"),
    "offsets count the input": ("new_offsets.append(len(keep))", "new_offsets.append(s1)"),
    "no empty ranks": ("combinations_with_replacement(", "combinations("),
    "smallest group instead of largest": ("worst = max(", "worst = min("),
    "largest cut instead of smallest": ("min(best, worst)", "max(best, worst)"),
}


def _mutant(name, old, new, tmp_path):
    text = open(SRC, encoding="utf-8").read()
    assert text.count(old) == 1, name
    path = tmp_path / "batching_mutant.py"
    path.write_text(text.replace(old, new), encoding="utf-8")
    spec = importlib.util.spec_from_file_location("batching_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_batching_mutant(name, tmp_path):
    mod = _mutant(name, *MUTANTS[name], tmp_path)
    caught = False
    for pin in (pin_stochastic_length, pin_min_max_split):
        try:
            pin(mod)
        except Exception:  # an AssertionError, or a crash the mistake causes
            caught = True
    assert caught, f"no pin fails on the mutant '{name}'"
