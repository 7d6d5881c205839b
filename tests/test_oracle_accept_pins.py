"""The acceptance / commit oracle against its pins, and planted mistakes in a
copy of it against the same pins (CPU only)."""
import importlib.util
import inspect
import os

import pytest

import oracle.accept as acc
import oracle_accept_pins as pins


def _run(pin, module, orc):
    params = inspect.signature(pin).parameters
    if "oracle_c" in params:
        return pin(module, orc)
    return pin(module)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=[p.__name__ for p in pins.ALL_PINS])
def test_accept_oracle_pin(pin, oracle):
    _run(pin, acc, oracle)


MUTANTS = {
    "compares_with_own_target": ("draft[i] == target[p]", "draft[i] == target[i]"),
    "ignores_parent_verdict": ("accepted[p] and draft[i]", "draft[i]"),
    "tie_goes_to_highest_index": ("depth[i] > depth[best]", "depth[i] >= depth[best]"),
    "path_left_reversed": ("    path.reverse()\n", "\n"),
    "bonus_from_root": ("int(target[best])", "int(target[path[0]])"),
    "only_node_zero_is_a_root": ("accepted[i] = True", "accepted[i] = i == 0"),
    "commit_at_node_position": ("pg, off = slot(b, L + k)", "pg, off = slot(b, L + j)"),
    "commit_without_prefix_offset": ("pg, off = slot(b, L + k)", "pg, off = slot(b, k)"),
    "length_not_updated": ("np.asarray(seq_lens, dtype=np.int64) + np.asarray(accept_len",
                           "np.asarray(seq_lens, dtype=np.int64) + 0 * np.asarray(accept_len"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_accept_mutant_is_caught(name, tmp_path, oracle):
    before, after = MUTANTS[name]
    src = open(acc.__file__).read()
    assert before in src, name
    path = os.path.join(tmp_path, "accept_mutant.py")
    with open(path, "w") as f:
        f.write(src.replace(before, after))
    spec = importlib.util.spec_from_file_location("accept_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            _run(pin, mod, oracle)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
