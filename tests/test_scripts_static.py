"""Static check of the repository's scripts: every name a function reads from the global
scope exists at module level or among the builtins.  bench.py and __graft_entry__.py run
only on a GPU, so a misspelt name in a rarely taken branch would otherwise surface there
first."""
import builtins
import os
import symtable

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _undefined_globals(path):
    src = open(path).read()
    top = symtable.symtable(src, path, "exec")
    defined = {s.get_name() for s in top.get_symbols()
               if s.is_assigned() or s.is_imported() or s.is_namespace()}
    defined |= set(dir(builtins))
    bad = []

    def walk(t):
        for s in t.get_symbols():
            if s.is_referenced() and s.is_global() and s.get_name() not in defined:
                bad.append(f"{t.get_name()}: {s.get_name()}")
        for c in t.get_children():
            walk(c)

    for c in top.get_children():
        walk(c)
    return bad


@pytest.mark.parametrize("script", ["bench.py", "__graft_entry__.py"])
def test_no_undefined_globals(script):
    assert _undefined_globals(os.path.join(ROOT, script)) == []
