"""Every global name a function loads exists (CPU): paths that only run on a
GPU, or only in the full benchmark, cannot hide an undefined helper."""
import builtins
import dis
import importlib
import types

import pytest

MODULES = ["bench", "zero_sharded_mixed_gb300.binding", "zero_sharded_mixed_gb300.step",
           "zero_sharded_mixed_gb300.engine", "zero_sharded_mixed_gb300.config",
           "zero_sharded_mixed_gb300.checkpoint", "zero_sharded_mixed_gb300.inputs",
           "zero_sharded_mixed_gb300.build"]


def _global_loads(code):
    for ins in dis.get_instructions(code):
        if ins.opname in ("LOAD_GLOBAL", "LOAD_NAME"):
            yield ins.argval
    for const in code.co_consts:
        if isinstance(const, types.CodeType):
            yield from _global_loads(const)


@pytest.mark.parametrize("name", MODULES)
def test_every_loaded_global_exists(name):
    mod = importlib.import_module(name)
    missing = set()
    for obj in list(vars(mod).values()):
        funcs = []
        if isinstance(obj, types.FunctionType) and obj.__module__ == mod.__name__:
            funcs.append(obj)
        elif isinstance(obj, type) and obj.__module__ == mod.__name__:
            funcs += [f for f in vars(obj).values() if isinstance(f, types.FunctionType)]
            funcs += [f.fget for f in vars(obj).values() if isinstance(f, property) and f.fget]
            funcs += [f.__func__ for f in vars(obj).values() if isinstance(f, (classmethod, staticmethod))]
        for f in funcs:
            if f.__globals__ is not vars(mod):        # generated elsewhere (dataclass methods)
                continue
            for g in _global_loads(f.__code__):
                if g not in vars(mod) and not hasattr(builtins, g):
                    missing.add(f"{f.__qualname__}: {g}")
    assert not missing, sorted(missing)
