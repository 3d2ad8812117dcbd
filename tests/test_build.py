"""The in-tree build (CPU only): builds of one folder never overlap, a caller that waited for
another's build of the default library does not build it again (both with the compile step
stubbed out), and two processes building one folder at once leave a library that loads."""
import os
import threading
import time

from combine_moe_route_gb300 import build as bld


def test_builds_of_one_folder_do_not_overlap(tmp_path, monkeypatch):
    spans = []

    def fake(out_dir, ptxas_info, verbose, defines):
        t0 = time.monotonic()
        time.sleep(0.2)
        spans.append((t0, time.monotonic()))
        return os.path.join(out_dir, bld.LIB_NAME)

    monkeypatch.setattr(bld, "_compile_and_link", fake)
    # a build with defines into its own folder is always redone, so each thread builds
    ths = [threading.Thread(target=bld.build, kwargs=dict(out_dir=str(tmp_path), defines=("X",)))
           for _ in range(3)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    spans.sort()
    assert len(spans) == 3
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))


def test_a_waiting_default_build_reuses_the_first(monkeypatch):
    state = {"built": False, "calls": 0}

    def fake(out_dir, ptxas_info, verbose, defines):
        time.sleep(0.2)
        state["calls"] += 1
        state["built"] = True
        return bld.library_path()

    monkeypatch.setattr(bld, "up_to_date", lambda: state["built"])
    monkeypatch.setattr(bld, "_compile_and_link", fake)
    paths = []
    ths = [threading.Thread(target=lambda: paths.append(bld.build())) for _ in range(2)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    assert state["calls"] == 1 and paths == [bld.library_path()] * 2


def test_two_processes_building_one_folder_leave_a_loadable_library(tmp_path):
    import ctypes
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = f"from combine_moe_route_gb300 import build; build.build(out_dir={str(tmp_path)!r}, force=True)"
    procs = [subprocess.Popen([sys.executable, "-c", code], cwd=root) for _ in range(2)]
    assert all(p.wait(timeout=600) == 0 for p in procs)
    lib = ctypes.CDLL(os.path.join(str(tmp_path), bld.LIB_NAME))
    assert lib.moe_abi_version() == 1
