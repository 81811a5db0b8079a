"""pytest plugin used by test_oracle_mutants.py (TEST INFRASTRUCTURE ONLY).

With ORACLE_MUTANT = JSON [module, old, new] in the environment, it replaces
oracle.<module> by a copy of its source in which the text ``old`` (which must
occur exactly once) is replaced by ``new``, before any test module is imported,
and points the other oracle modules that hold the original at the copy.
"""
import importlib
import json
import os
import sys
import types


def pytest_configure(config):
    spec = os.environ.get("ORACLE_MUTANT")
    if not spec:
        return
    name, old, new = json.loads(spec)
    import oracle
    orig = importlib.import_module(f"oracle.{name}")
    src = open(orig.__file__).read()
    if src.count(old) != 1:
        raise RuntimeError(f"mutant pattern occurs {src.count(old)} times in oracle/{name}.py: {old!r}")
    mod = types.ModuleType(orig.__name__)
    mod.__file__ = orig.__file__
    mod.__package__ = "oracle"
    sys.modules[orig.__name__] = mod
    exec(compile(src.replace(old, new), orig.__file__, "exec"), mod.__dict__)
    setattr(oracle, name, mod)
    for other_name, other in list(sys.modules.items()):
        if other_name.startswith("oracle.") and other is not mod:
            for attr, value in list(vars(other).items()):
                if value is orig:
                    setattr(other, attr, mod)
