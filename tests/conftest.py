import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.get()


class FnormEnv:
    """Sets FNORM_* tuning switches for one test. The library reads them once
    per process, so every change is followed by fnorm_tuning_reload()."""

    def __init__(self, mp):
        self.mp = mp

    def setenv(self, name, value):
        import normalization_reduction_gb300 as fn
        self.mp.setenv(name, value)
        fn.fnorm_tuning_reload()

    def delenv(self, name, raising=True):
        import normalization_reduction_gb300 as fn
        self.mp.delenv(name, raising=raising)
        fn.fnorm_tuning_reload()

    def force_timeout(self, on):
        import normalization_reduction_gb300 as fn
        fn.fnorm_debug_force_timeout(on)


@pytest.fixture
def fnorm_env(monkeypatch):
    """FNORM_* switches and the forced-timeout hook, restored after the test."""
    import normalization_reduction_gb300 as fn
    yield FnormEnv(monkeypatch)
    monkeypatch.undo()
    fn.fnorm_tuning_reload()
    fn.fnorm_debug_force_timeout(False)
