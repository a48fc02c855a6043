"""The in-tree build: concurrent builds of the CUDA library are serialised (they
share the object files in the build folder).  The compile step is replaced by a
stub here, so nothing is compiled and no GPU is needed."""
import threading
import time

from combine_moe_route_02_gb300 import _build


def test_concurrent_builds_are_serialised(monkeypatch):
    state = {"active": 0, "calls": 0, "overlaps": 0}
    guard = threading.Lock()

    def fake_build(verbose_ptxas):
        with guard:
            state["active"] += 1
            state["calls"] += 1
            state["overlaps"] += state["active"] > 1
        time.sleep(0.2)
        with guard:
            state["active"] -= 1
        return _build.LIB_PATH

    monkeypatch.setattr(_build, "_build_locked", fake_build)
    # force: every caller builds, so all three go through the lock
    threads = [threading.Thread(target=_build.build, kwargs={"force": True}) for _ in range(3)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert state["calls"] == 3
    assert state["overlaps"] == 0
