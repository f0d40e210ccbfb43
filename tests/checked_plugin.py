"""pytest plugin of the checked-build runs (test_gpu_checked_build.py): makes
sure the child process really loaded libgemm_gather_checked.so, and that no
test left a report in the library's status word (a check that fired where the
arguments were valid would land there when a launch had no status word)."""
import pytest


def pytest_sessionstart(session):
    import gemm_gather_gb300 as gg
    if not gg.checked_build():
        raise pytest.UsageError("checked_plugin: the checked build is not loaded "
                                "(set GEMM_GATHER_CHECKED=1)")


@pytest.fixture(autouse=True)
def _library_word_stays_clear(request):
    if request.node.get_closest_marker("gpu") is None or "checked_table" in request.node.nodeid:
        yield
        return
    import gemm_gather_gb300 as gg
    gg.clear_device_status()
    yield
    assert gg.device_status() == 0, "a device-side check fired on valid arguments"
