import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def orc(tmp_path_factory):
    import oracle
    src = os.environ.get("CLEF_ORACLE_MUTANT")
    if src:
        # a copy of the oracle with one planted mistake (see
        # test_oracle_mutants.py): the same bindings over a build of that source
        import importlib.util
        spec = importlib.util.spec_from_file_location("oracle_mutant", oracle.__file__)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod._SRC = src
        mod._BUILD = str(tmp_path_factory.mktemp("oracle_mutant"))
        mod._LIB = os.path.join(mod._BUILD, "libclef_oracle.so")
        mod.lib()
        return mod
    oracle.lib()
    return oracle
