"""Host side of the phase-trace tool (CPU only): how raw stamp slots become phase times."""
import pytest

trace = pytest.importorskip("combine_moe_route_gb300.trace")


def test_phases_are_relative_to_the_first_stamp():
    raw = [trace.UNSET if i % 2 == 0 else 0 for i in range(trace.SLOTS)]
    # histogram block starts at t = 1000 ns (first) .. 1500 ns (last); scan done 5000 .. 7000 ns
    raw[12], raw[13] = 1_000, 1_500
    raw[26], raw[27] = 5_000, 7_000
    got = trace._phases(raw, trace.DISPATCH_PHASES)
    assert got == {"histogram block starts": (0.0, 0.5), "scan block done": (4.0, 6.0)}


def test_unset_slots_are_left_out():
    raw = [trace.UNSET if i % 2 == 0 else 0 for i in range(trace.SLOTS)]
    assert trace._phases(raw, trace.COMBINE_PHASES) == {}
    raw[0], raw[1] = 10, 20
    assert trace._phases(raw, trace.COMBINE_PHASES) == {"combine block starts": (0.0, 0.01)}


def test_phase_slots_match_the_device_enum():
    # slot numbers are those of TraceSlot in csrc/trace.cuh (even = first, odd = last stamp)
    import os
    import re
    src = open(os.path.join(os.path.dirname(trace.__file__), "csrc", "trace.cuh")).read()
    slots = {name: int(v) for name, v in re.findall(r"(kTr\w+) = (\d+),", src)}
    assert all(v % 2 == 0 and v + 1 < trace.SLOTS for v in slots.values())
    dispatch = {k: v for k, v in slots.items() if not k.startswith("kTrCombine")}
    assert sorted(dispatch.values()) == sorted(trace.DISPATCH_PHASES)
    assert sorted(v for k, v in slots.items() if k.startswith("kTrCombine")) == sorted(trace.COMBINE_PHASES)
    assert int(re.search(r"kTraceSlots = (\d+);", src).group(1)) == trace.SLOTS
