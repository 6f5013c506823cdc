"""Plant plausible mistakes in a copy of the block-manager reference model (CPU only) and check
that the pins in test_block_pool_pins.py catch each one: a pin that cannot tell a wrong model
from the right one pins nothing."""
import importlib.util
import inspect
import sys

import pytest

import test_block_pool_pins as PINS
from oracle import block_pool as BP

SRC = inspect.getsourcefile(BP)

# (name, exact text in the model, replacement)
MUTANTS = [
    ("unhashed_blocks_to_the_back", "                    self.queue.insert(0, i)",
     "                    self.queue.append(i)"),
    ("hashed_blocks_to_the_front", "                else:\n                    self.queue.append(i)",
     "                else:\n                    self.queue.insert(0, i)"),
    ("free_head_first", "self._free(list(reversed(r.blocks)))", "self._free(list(r.blocks))"),
    ("eager_eviction", "                else:\n                    self.queue.append(i)",
     "                else:\n                    lst = self.cache[b.key]\n                    lst.remove(b.id)\n"
     "                    if not lst:\n                        del self.cache[b.key]\n                    b.key = None\n"
     "                    self.queue.append(i)"),
    ("prompt_may_hit_in_full", "min(n_full, (len(tokens) - 1) // bs)", "n_full"),
    ("salt_on_every_block", 'extra = salt if k == 0 else b""', "extra = salt"),
    ("no_copy_on_write", "if last.ref > 1:  # shared, partly filled: copy on write", "if False:"),
    ("null_block_handed_out", "self.null = self.queue.pop(0)", "self.null = -1"),
    ("hashes_not_chained", "parent = block_hash(parent, tokens", "parent = block_hash(self.root, tokens"),
]


def _pins():
    return [f for n, f in sorted(vars(PINS).items()) if n.startswith("test_") and callable(f)]


def _load_variant(tmp_path, text, repl, tag):
    src = open(SRC).read()
    assert src.count(text) >= 1, f"mutation anchor not found: {text!r}"
    path = tmp_path / f"block_pool_{tag}.py"
    path.write_text(src.replace(text, repl, 1))
    name = f"block_pool_mutant_{tag}"
    spec = importlib.util.spec_from_file_location(name, str(path))
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod  # dataclasses look their module up while the class is made
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.modules.pop(name, None)
    return mod


def _failures(monkeypatch, mod):
    monkeypatch.setattr(PINS, "BP", mod)
    failed = []
    for f in _pins():
        try:
            f()
        except (Exception, pytest.fail.Exception):  # a failed assert, raise or pytest.raises
            failed.append(f.__name__)
    return failed


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    mod = _load_variant(tmp_path, "BLOCK = 16", "BLOCK = 16", "identity")
    assert _failures(monkeypatch, mod) == []


@pytest.mark.parametrize("name,text,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, monkeypatch, name, text, repl):
    mod = _load_variant(tmp_path, text, repl, name)
    assert _failures(monkeypatch, mod), f"no pin caught the planted mistake {name}"
